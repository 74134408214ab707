#!/usr/bin/env python3
"""Benchmark of the sharded MLP block's forward + backward on one GB300.

One step = the whole hot path over one batch of synthetic input:
  forward:  column GEMM + bias + GELU-tanh (all T shards), row GEMM with the
            shard sum folded into the split-K accumulator (b2 once);
  backward: dZ GEMM with the act' epilogue, dW2 GEMM, dW1 GEMM, dX GEMM with
            the shard sum folded into split-K.
Workload: N = 8192 tokens (B=4, L=2048), D = 8192, F = 28672, T = 8, bf16
storage, fp32 accumulation, no bias, seeded synthetic inputs (X, dY ~ N(0,1),
W ~ N(0, 0.02)).

The JSON line also carries: the dominant kernel's roofline (CUDA-event
durations measured live during the timed region), the float64 CPU oracle timed
on a bounded sample of the same workload, an end-to-end number through the
public API with host buffers, SM clocks sampled during the timed region, and
secondary measurements (the PARTIALS variant with its block-end reduce
kernel, and the vocab-parallel cross-entropy kernel).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
"""

import argparse
import json
import os
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from workloads.configs import MLP_CONFIGS, CE_CONFIGS  # noqa: E402
from workloads.gen import gen_mlp_inputs  # noqa: E402

WORKLOAD = "mlp_bf16_gelu_n8192_d8192_f28672_t8_fwdbwd"
METRIC = "sharded-MLP fwd+bwd TFLOP/s (% BF16 peak); reduce & CE HBM GB/s (% peak)"
BAD_REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown")


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    # defaults time the power-capped steady state: a 20-step timed region after
    # 3 warm-ups read about 2.5% higher than 100 steps after 20
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--mode", choices=["splitk", "partials"], default="splitk")
    ap.add_argument("--no-secondary", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--shape", default=None,
                    help="N,D,F,T override of the fwd+bwd workload (small cases for profiling)")
    ap.add_argument("--only-embedding", action="store_true",
                    help="time only the vocab embedding gather (32000 x 8192 bf16, T=4, 8192 ids)")
    ap.add_argument("--only-ce", type=int, default=0, metavar="TOKENS",
                    help="time only the vocab CE forward and backward (V=128000, T=8) on TOKENS "
                         "tokens (small cases for profiling)")
    return ap.parse_args()


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "source": "fallback"}


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 50 ms."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.f = None

    def start(self):
        try:
            self.f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"]}
        time.sleep(0.3)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.flush()
        rows = []
        for line in open(self.f.name):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append({"sm": float(parts[1]), "max": float(parts[2]),
                             "power": float(parts[3]) if parts[3] not in ("[N/A]", "") else None,
                             "hw": parts[5], "hwt": parts[6], "swt": parts[7], "pcap": parts[8]})
            except ValueError:
                continue
        os.unlink(self.f.name)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        load = [r for r in rows if r["power"] is not None and r["power"] > 300] or rows
        reasons = set()
        for r in load:
            if r["hw"] == "Active":
                reasons.add("hw_slowdown")
            if r["hwt"] == "Active":
                reasons.add("hw_thermal_slowdown")
            if r["swt"] == "Active":
                reasons.add("sw_thermal_slowdown")
            if r["pcap"] == "Active":
                reasons.add("sw_power_cap")
        return {"sm_mhz": float(np.median([r["sm"] for r in load])),
                "sm_max_mhz": float(max(r["max"] for r in rows)),
                "samples": len(rows), "samples_under_load": len(load),
                "reasons": sorted(reasons)}


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------

class Block:
    """Device-resident inputs, outputs and workspace of one fwd+bwd step."""

    def __init__(self, cfg, mode, dev, with_dy=True):
        import tensor_transformer_mlp_columnparallel_gb300 as tp
        self.tp = tp
        self.cfg, self.mode, self.dev = cfg, mode, dev
        inp = gen_mlp_inputs(cfg, with_dy=with_dy)
        self.host = inp
        self.X = inp.X.to(dev)
        self.dY = inp.dY.to(dev) if with_dy else None
        self.W1 = [w.to(dev) for w in inp.W1_shards()]
        self.W2 = [w.contiguous().to(dev) for w in inp.W2_shards()]
        self.b1 = None if inp.b1 is None else [b.contiguous().to(dev) for b in inp.b1_shards()]
        self.b2 = None if inp.b2 is None else inp.b2.to(dev)
        N, D, Fs, T = cfg.N, cfg.D, cfg.Fs, cfg.T
        dt = self.X.dtype
        e = lambda *s: torch.empty(s, dtype=dt, device=dev)
        self.Y = e(N, D)
        self.H = [e(N, Fs) for _ in range(T)]
        self.Z = [e(N, Fs) for _ in range(T)]
        if with_dy:
            self.dX = e(N, D)
            self.dW1 = [e(D, Fs) for _ in range(T)]
            self.dW2 = [e(Fs, D) for _ in range(T)]
        # the balanced size also holds the few-token GEMMs' stream-K scratch
        wf = tp.tpmlp_workspace_bytes_balanced(0, dt, N, D, cfg.F, T, mode)
        wb = tp.tpmlp_workspace_bytes_balanced(1, dt, N, D, cfg.F, T, mode) if with_dy else 0
        self.ws = torch.empty(max(wf, wb, 256), dtype=torch.uint8, device=dev)

    def set_mode(self, mode):
        tp = self.tp
        cfg = self.cfg
        self.mode = mode
        wsb = tp.tpmlp_workspace_bytes_balanced
        need = max(wsb(0, self.X.dtype, cfg.N, cfg.D, cfg.F, cfg.T, mode),
                   wsb(1, self.X.dtype, cfg.N, cfg.D, cfg.F, cfg.T, mode), 256)
        if self.ws.numel() < need:
            self.ws = torch.empty(need, dtype=torch.uint8, device=self.dev)

    def forward(self):
        self.tp.tpmlp_forward(self.X, self.W1, self.b1, self.W2, self.b2, self.Y, self.H, self.Z,
                              self.cfg.act, self.mode, self.ws)

    def step(self):
        tp = self.tp
        tp.tpmlp_forward(self.X, self.W1, self.b1, self.W2, self.b2, self.Y, self.H, self.Z,
                         self.cfg.act, self.mode, self.ws)
        tp.tpmlp_backward(self.X, self.W1, self.W2, self.H, self.Z, self.dY, self.dX, self.dW1,
                          self.dW2, None, None, self.cfg.act, self.mode, self.ws)


def workload_config(args):
    cfg = MLP_CONFIGS[WORKLOAD]
    if args.shape:
        import dataclasses
        N, D, F, T = (int(x) for x in args.shape.split(","))
        cfg = dataclasses.replace(cfg, name=f"{WORKLOAD}_shape_{N}_{D}_{F}_{T}", B=1, L=N, D=D,
                                  F=F, T=T)
    return cfg


def barrier(world):
    if world > 1:
        torch.distributed.barrier()


def max_over_ranks(x, world, dev):
    if world == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def timed(fn, steps, warmup, world, dev, stream, reset=None):
    """Device time (ms) of `steps` calls of fn after `warmup` untimed ones;
    `reset` (e.g. the library's kernel-timing reset) runs between the two so
    per-kernel tables cover the timed calls only."""
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    if reset is not None:
        reset()
    barrier(world)
    torch.cuda.synchronize()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(steps):
        fn()
    b.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    return a.elapsed_time(b)


def kernel_table(t, total_ms):
    out = {}
    for name, v in sorted(t.items(), key=lambda kv: -kv[1]["total_ms"]):
        out[name] = {"launches": v["launches"], "ms_per_launch": v["total_ms"] / max(v["launches"], 1),
                     "share": v["total_ms"] / total_ms if total_ms > 0 else None}
    return out


KERNEL_FAMILIES = {
    # kernel timing name prefix -> CUDA sources that define that kernel
    "gemm": ("gemm_tc.cu", "ptx.cuh", "act.cuh", "tpmlp_internal.h"),
    "hbm": ("hbm_kernels.cu", "ptx.cuh", "act.cuh", "tpmlp_internal.h"),
}


def kernel_family(kernel):
    return "gemm" if "gemm" in kernel else "hbm"


def kernel_source_hash(family="gemm"):
    """sha256 over the CUDA sources of one kernel family: file names and the
    code with `//` comments, trailing blanks and empty lines removed, so that
    editing a comment does not invalidate a capture of the same code."""
    import hashlib
    h = hashlib.sha256()
    d = os.path.join(ROOT, "tensor_transformer_mlp_columnparallel_gb300", "csrc")
    for f in KERNEL_FAMILIES[family]:
        h.update(f.encode())
        for line in open(os.path.join(d, f), encoding="utf-8"):
            code = line.split("//", 1)[0].rstrip()
            if code:
                h.update(code.encode() + b"\n")
    return h.hexdigest()


def load_traffic(kernel):
    """DRAM bytes per launch of `kernel` from the committed ncu summary
    (profiles/traffic.json), or None when that summary was taken on other
    sources of the kernel's family than the ones built now."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    try:
        d = json.load(open(p))
        fam = kernel_family(kernel)
        if d.get("source_hash", {}).get(fam) != kernel_source_hash(fam):
            return None
        return d["kernels"].get(kernel, {}).get("dram_bytes_per_launch")
    except Exception:
        return None


def cpu_baseline_mlp(cfg, tokens=96):
    """Float64 oracle fwd+bwd on `tokens` rows of the same workload, all
    host cores (numpy / OpenBLAS default threading). The per-token work of
    fwd+bwd is 12 D F FLOP (two forward GEMM rows, four backward)."""
    import oracle
    inp = gen_mlp_inputs(cfg, N=tokens)
    W1 = oracle.mlp.as_f64(inp.W1)
    W2 = oracle.mlp.as_f64(inp.W2)
    t0 = time.perf_counter()
    oracle.mlp.forward(inp.X, W1, None, W2, None, cfg.act)
    oracle.mlp.backward(inp.X, W1, None, W2, inp.dY, cfg.act)
    dt = time.perf_counter() - t0
    flops = 12.0 * tokens * cfg.D * cfg.F
    cores = len(os.sched_getaffinity(0))
    return {"value": flops / dt / 1e12, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
            "sample": f"{tokens} of {cfg.N} tokens, fwd+bwd, float64 numpy (OpenBLAS threads = "
                      f"host cores), {dt:.1f} s"}


def measure_embedding(dev, steps, pk):
    """Vocab-parallel embedding: table 32000 x 8192 bf16 over T = 4 (the
    textbook page's row-parallel embedding), 8192 tokens; L2 flushed by a read
    before every launch. Returns the record of the secondary measurements."""
    import tensor_transformer_mlp_columnparallel_gb300 as tp
    Ve, He, Te, Ne = 32000, 8192, 4, 8192
    ge = torch.Generator(device=dev)
    ge.manual_seed(0)
    shards = [(torch.randn(Ve // Te, He, generator=ge, device=dev) * 0.02).to(torch.bfloat16)
              for _ in range(Te)]
    ids = torch.randint(0, Ve, (Ne,), generator=ge, device=dev)
    emb = torch.empty(Ne, He, dtype=torch.bfloat16, device=dev)
    # L2 flush by READING a buffer twice the L2 size: L2 then holds clean lines,
    # so no write-back of flush data (or of the previous output, which the
    # flush evicts) lands inside the timed launch
    flush = torch.ones(256 << 20, dtype=torch.uint8, device=dev)
    tp.tpmlp_timing_reset()
    for i in range(3 + steps):
        flush.max()
        if i == 3:
            tp.tpmlp_timing_enable(True)
        tp.tpmlp_vocab_embedding(ids, shards, emb)
    torch.cuda.synchronize()
    tp.tpmlp_timing_enable(False)
    k = tp.tpmlp_timing_read()["vocab_embedding"]
    ms = k["total_ms"] / k["launches"]
    e_bytes = 2.0 * Ne * He * 2 + Ne * 8
    gbs = e_bytes / (ms * 1e-3) / 1e9
    return {
        "kernel": "vocab_embedding", "ms_per_launch": ms, "GB/s": gbs,
        "l2": "flushed before each launch by reading a 256 MB buffer",
        "roofline": {"bound": "hbm", "achieved": gbs, "peak": pk["hbm_gbs"], "unit": "GB/s",
                     "frac": gbs / pk["hbm_gbs"], "algorithmic_bytes_per_launch": e_bytes,
                     "traffic": load_traffic("vocab_embedding")}}


def secondary(dev, stream, steps, pk, ce_tokens=0):
    import dataclasses
    import tensor_transformer_mlp_columnparallel_gb300 as tp
    out = {}
    # vocab-parallel CE, N = 8192, V = 128000, T = 8: logits drawn on the device
    ce = CE_CONFIGS["vocab_ce_n8192_v128000_t8"]
    if ce_tokens:
        ce = dataclasses.replace(ce, N=ce_tokens)
    g = torch.Generator(device=dev)
    g.manual_seed(0)
    logits = torch.randn((ce.N, ce.V), generator=g, device=dev) * ce.logit_std
    targets = torch.randint(0, ce.V, (ce.N,), generator=g, device=dev)
    loss = torch.empty(ce.N, device=dev)
    mean = torch.empty(1, device=dev)
    amax = torch.empty(ce.N, dtype=torch.int32, device=dev)
    own = torch.empty(ce.N, dtype=torch.int32, device=dev)
    fn = lambda: tp.tpmlp_vocab_ce(logits, targets, ce.T, loss, mean, amax, own)
    tp.tpmlp_timing_reset()
    tp.tpmlp_timing_enable(True)
    timed(fn, steps, 3, 1, dev, stream, reset=tp.tpmlp_timing_reset)
    tp.tpmlp_timing_enable(False)
    t = tp.tpmlp_timing_read()
    k = t["vocab_ce_fwd"]
    ms = k["total_ms"] / k["launches"]
    gbs = ce.algorithmic_bytes() / (ms * 1e-3) / 1e9
    out["vocab_ce_n8192_v128000_t8"] = {
        "kernel": "vocab_ce_fwd", "ms_per_launch": ms, "GB/s": gbs,
        "roofline": {"bound": "hbm", "achieved": gbs, "peak": pk["hbm_gbs"], "unit": "GB/s",
                     "frac": gbs / pk["hbm_gbs"],
                     # the committed traffic is per full-size launch
                     "traffic": None if ce_tokens else load_traffic("vocab_ce_fwd")}}
    # backward of the same cross-entropy (mean reduction): read z, write dz
    dlog = torch.empty_like(logits)
    fnb = lambda: tp.tpmlp_vocab_ce_backward(logits, targets, ce.T, loss, 1.0 / ce.N, dlog)
    tp.tpmlp_timing_reset()
    tp.tpmlp_timing_enable(True)
    timed(fnb, steps, 3, 1, dev, stream, reset=tp.tpmlp_timing_reset)
    tp.tpmlp_timing_enable(False)
    t = tp.tpmlp_timing_read()
    k = t["vocab_ce_bwd"]
    ms = k["total_ms"] / k["launches"]
    bwd_bytes = 8.0 * ce.N * ce.V + 12.0 * ce.N
    gbs = bwd_bytes / (ms * 1e-3) / 1e9
    out["vocab_ce_backward_n8192_v128000_t8"] = {
        "kernel": "vocab_ce_bwd", "ms_per_launch": ms, "GB/s": gbs,
        "roofline": {"bound": "hbm", "achieved": gbs, "peak": pk["hbm_gbs"], "unit": "GB/s",
                     "frac": gbs / pk["hbm_gbs"],
                     "traffic": None if ce_tokens else load_traffic("vocab_ce_bwd"),
                     "algorithmic_bytes_per_launch": bwd_bytes}}
    del logits, dlog
    torch.cuda.empty_cache()
    if ce_tokens:
        return out
    # block end as a reduce-scatter (T = 8 fp32 partials of [8192, 8192] -> 8 bf16
    # row blocks of [1024, 8192]); the partials exceed L2
    Tn, Nn, Dn = 8, 8192, 8192
    parts = [torch.randn(Nn, Dn, device=dev) for _ in range(Tn)]
    rows_out = [torch.empty(Nn // Tn, Dn, dtype=torch.bfloat16, device=dev) for _ in range(Tn)]
    b2 = torch.zeros(Dn, dtype=torch.bfloat16, device=dev)
    fn = lambda: tp.tpmlp_block_reduce_scatter(parts, b2, rows_out)
    tp.tpmlp_timing_reset()
    tp.tpmlp_timing_enable(True)
    timed(fn, steps, 3, 1, dev, stream, reset=tp.tpmlp_timing_reset)
    tp.tpmlp_timing_enable(False)
    k = tp.tpmlp_timing_read()["block_reduce_scatter_bias"]
    ms = k["total_ms"] / k["launches"]
    rs_bytes = Tn * Nn * Dn * 4 + Nn * Dn * 2 + Dn * 2
    gbs = rs_bytes / (ms * 1e-3) / 1e9
    out["block_reduce_scatter_t8_n8192_d8192"] = {
        "kernel": "block_reduce_scatter_bias", "ms_per_launch": ms, "GB/s": gbs,
        "roofline": {"bound": "hbm", "achieved": gbs, "peak": pk["hbm_gbs"], "unit": "GB/s",
                     "frac": gbs / pk["hbm_gbs"], "algorithmic_bytes_per_launch": rs_bytes,
                     "traffic": load_traffic("block_reduce_scatter_bias")}}
    del parts, rows_out
    torch.cuda.empty_cache()
    out["vocab_embedding_v32000_h8192_t4_n8192"] = measure_embedding(dev, steps, pk)
    torch.cuda.empty_cache()
    # forward-only workloads: N=4096 D=4096 F=16384 T=4 (tensor-bound) and
    # N=16 D=12288 F=49152 T=8 (weight streaming, HBM-bound)
    for name in ("mlp_bf16_gelu_n4096_d4096_f16384_t4", "mlp_bf16_gelu_n16_d12288_f49152_t8"):
        fc = MLP_CONFIGS[name]
        fb = Block(fc, "splitk", dev, with_dy=False)
        for mode in ("splitk", "partials"):
            fb.set_mode(mode)
            tp.tpmlp_timing_reset()
            tp.tpmlp_timing_enable(True)
            ms_f = timed(fb.forward, steps, 3, 1, dev, stream, reset=tp.tpmlp_timing_reset)
            tp.tpmlp_timing_enable(False)
            t = tp.tpmlp_timing_read()
            flops = fc.fwd_flops()
            wbytes = 2.0 * fc.D * fc.F * 2 + fc.F * 2 + fc.D * 2      # W1, W2, b1, b2 (bf16)
            abytes = wbytes + 2.0 * fc.N * fc.D * 2 + 2.0 * fc.N * fc.F * 2   # + X, Y, H, Z
            rec = {"mode": mode, "ms_per_forward": ms_f / steps,
                   "TFLOP/s": flops * steps / (ms_f * 1e-3) / 1e12,
                   "GB/s": abytes * steps / (ms_f * 1e-3) / 1e9,
                   "kernels": kernel_table(t, ms_f)}
            if fc.N <= 64:
                rec["roofline"] = {"bound": "hbm", "achieved": rec["GB/s"], "peak": pk["hbm_gbs"],
                                   "unit": "GB/s", "frac": rec["GB/s"] / pk["hbm_gbs"],
                                   "algorithmic_bytes_per_forward": abytes}
            else:
                rec["roofline"] = {"bound": "tensor", "achieved": rec["TFLOP/s"],
                                   "peak": pk["bf16_tflops_sustained"], "unit": "TFLOP/s",
                                   "frac": rec["TFLOP/s"] / pk["bf16_tflops_sustained"]}
            out[f"{name}_{mode}"] = rec
        del fb
        torch.cuda.empty_cache()
    # the exact-fp32 block, N=64 D=256 F=1024 T=2 (ReLU, biases): latency-bound
    # (67 MFLOP forward), so time per call, eager and replayed from a CUDA graph
    fc = MLP_CONFIGS["mlp_f32_relu_n64_d256_f1024_t2"]
    fb = Block(fc, "splitk", dev)
    rec = {"note": "latency-bound; time reported, no roofline claim"}
    for label, fn in (("forward", fb.forward), ("forward+backward", fb.step)):
        ms_e = timed(fn, steps, 3, 1, dev, stream) / steps
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            for _ in range(10):
                fn()
        graph.replay()
        torch.cuda.synchronize()
        ms_g = timed(graph.replay, max(1, steps // 10), 1, 1, dev, stream) / (10 * max(1, steps // 10))
        rec[label] = {"us_per_call_eager": ms_e * 1e3, "us_per_call_graph": ms_g * 1e3}
    out["mlp_f32_relu_n64_d256_f1024_t2_latency"] = rec
    del fb
    torch.cuda.empty_cache()
    # gated (SwiGLU) block, N=4096 D=4096 F=16384 T=4: gate and up as one dual
    # GEMM per shard, then the split-K down projection
    Ns, Ds, Fg, Tg = 4096, 4096, 16384, 4
    gs = torch.Generator(device=dev)
    gs.manual_seed(0)
    Xg = torch.randn(Ns, Ds, generator=gs, device=dev).to(torch.bfloat16)
    mk = lambda r, c: (torch.randn(r, c, generator=gs, device=dev) * 0.02).to(torch.bfloat16)
    Wg = [mk(Ds, Fg // Tg) for _ in range(Tg)]
    Wu = [mk(Ds, Fg // Tg) for _ in range(Tg)]
    Wd = [mk(Fg // Tg, Ds) for _ in range(Tg)]
    Yg = torch.empty(Ns, Ds, dtype=torch.bfloat16, device=dev)
    Hg = [torch.empty(Ns, Fg // Tg, dtype=torch.bfloat16, device=dev) for _ in range(Tg)]
    fn = lambda: tp.tpmlp_swiglu_forward(Xg, Wg, Wu, Wd, Yg, Hg, None, None, "splitk", None)
    tp.tpmlp_timing_reset()
    tp.tpmlp_timing_enable(True)
    ms_s = timed(fn, steps, 3, 1, dev, stream, reset=tp.tpmlp_timing_reset)
    tp.tpmlp_timing_enable(False)
    t = tp.tpmlp_timing_read()
    sflops = 6.0 * Ns * Ds * Fg
    out["swiglu_bf16_n4096_d4096_f16384_t4_splitk"] = {
        "TFLOP/s": sflops * steps / (ms_s * 1e-3) / 1e12, "ms_per_forward": ms_s / steps,
        "kernels": kernel_table(t, ms_s),
        "roofline": {"bound": "tensor", "achieved": sflops * steps / (ms_s * 1e-3) / 1e12,
                     "peak": pk["bf16_tflops_sustained"], "unit": "TFLOP/s",
                     "frac": sflops * steps / (ms_s * 1e-3) / 1e12 / pk["bf16_tflops_sustained"]}}
    del Xg, Wg, Wu, Wd, Yg, Hg
    torch.cuda.empty_cache()
    # the PARTIALS variant of the same fwd+bwd step: T fp32 partials + block reduce
    cfg = MLP_CONFIGS[WORKLOAD]
    blk = Block(cfg, "partials", dev)
    tp.tpmlp_timing_reset()
    tp.tpmlp_timing_enable(True)
    ms_total = timed(blk.step, max(3, steps // 2), 3, 1, dev, stream, reset=tp.tpmlp_timing_reset)
    tp.tpmlp_timing_enable(False)
    t = tp.tpmlp_timing_read()
    nsteps = max(3, steps // 2)
    flops = (cfg.fwd_flops() + cfg.bwd_flops()) * nsteps
    red_bytes = cfg.T * cfg.N * cfg.D * 4 + cfg.N * cfg.D * 2   # read T fp32 partials, write bf16
    rk = {}
    for name in ("block_reduce_bias", "block_reduce_dx"):
        if name in t:
            ms = t[name]["total_ms"] / t[name]["launches"]
            gbs = red_bytes / (ms * 1e-3) / 1e9
            rk[name] = {"ms_per_launch": ms, "GB/s": gbs,
                        "roofline": {"bound": "hbm", "achieved": gbs, "peak": pk["hbm_gbs"],
                                     "unit": "GB/s", "frac": gbs / pk["hbm_gbs"],
                                     "traffic": load_traffic(name)}}
    out["partials_variant_" + WORKLOAD] = {
        "TFLOP/s": flops / (ms_total * 1e-3) / 1e12, "ms_per_step": ms_total / nsteps,
        "reduce_kernels": rk, "kernels": kernel_table(t, ms_total)}
    return out


def e2e_measure(blk, steps, stream):
    """The same step through the public API with host buffers. Every step
    copies that step's batch (X, dY) from pinned host memory to the device and
    its activation results (Y, dX) back to pinned host memory; the weights and
    their gradients are resident model state and stay on the device. The
    copy-in of step i+1 and the read-back of step i-1 run on two copy streams
    (one per link direction) while step i computes, with double-buffered
    device batches and results; all of it is inside the timed region."""
    import tensor_transformer_mlp_columnparallel_gb300 as tp
    cfg, dev = blk.cfg, blk.dev
    h = blk.host
    hX = [h.X.contiguous().pin_memory() for _ in range(2)]
    hdY = [h.dY.contiguous().pin_memory() for _ in range(2)]
    oY = [torch.empty_like(hX[0]).pin_memory() for _ in range(2)]
    odX = [torch.empty_like(hX[0]).pin_memory() for _ in range(2)]
    dX_in = [blk.X, torch.empty_like(blk.X)]
    dY_in = [blk.dY, torch.empty_like(blk.dY)]
    Y_out = [blk.Y, torch.empty_like(blk.Y)]
    dX_out = [blk.dX, torch.empty_like(blk.dX)]
    h2d = 2 * h.X.numel() * h.X.element_size()
    d2h = 2 * h.X.numel() * h.X.element_size()
    cin, cout = torch.cuda.Stream(dev), torch.cuda.Stream(dev)   # both link directions at once
    ready = [torch.cuda.Event() for _ in range(2)]      # batch i copied in
    done = [torch.cuda.Event() for _ in range(2)]       # step i computed
    drained = [torch.cuda.Event() for _ in range(2)]    # results of step i copied out

    def compute(i):
        b = i % 2
        stream.wait_event(ready[b])
        if i >= 2:
            stream.wait_event(drained[b])
        tp.tpmlp_forward(dX_in[b], blk.W1, blk.b1, blk.W2, blk.b2, Y_out[b], blk.H, blk.Z,
                         cfg.act, blk.mode, blk.ws)
        tp.tpmlp_backward(dX_in[b], blk.W1, blk.W2, blk.H, blk.Z, dY_in[b], dX_out[b], blk.dW1,
                          blk.dW2, None, None, cfg.act, blk.mode, blk.ws)
        done[b].record(stream)

    def copy_in(i):
        b = i % 2
        with torch.cuda.stream(cin):
            if i >= 2:
                cin.wait_event(done[b])       # the batch buffer of step i-2 is free
            dX_in[b].copy_(hX[b], non_blocking=True)
            dY_in[b].copy_(hdY[b], non_blocking=True)
            ready[b].record(cin)

    def copy_out(i):
        b = i % 2
        with torch.cuda.stream(cout):
            cout.wait_event(done[b])
            oY[b].copy_(Y_out[b], non_blocking=True)
            odX[b].copy_(dX_out[b], non_blocking=True)
            drained[b].record(cout)

    def run(n):
        copy_in(0)
        for i in range(n):
            if i + 1 < n:
                copy_in(i + 1)
            compute(i)
            copy_out(i)
        stream.wait_stream(cin)
        stream.wait_stream(cout)

    run(2)
    torch.cuda.synchronize()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record(stream)
    run(steps)
    b.record(stream)
    torch.cuda.synchronize()
    ms = a.elapsed_time(b)
    # the results of the last step reached the host: check one value against the device
    assert torch.equal(oY[(steps - 1) % 2][0, :8], Y_out[(steps - 1) % 2][0, :8].cpu())
    return ms, h2d, d2h


def run_ours(args):
    rank, world, local = dist_env()
    if world > 1:
        torch.distributed.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    import __graft_entry__
    __graft_entry__.build()
    import tensor_transformer_mlp_columnparallel_gb300 as tp

    cfg = workload_config(args)
    pk = peaks()
    blk = Block(cfg, args.mode, dev)
    stream = torch.cuda.current_stream(dev)
    for _ in range(args.warmup):
        blk.step()
    torch.cuda.synchronize()
    assert tp.tpmlp_check_device_error() == 0

    clocks = ClockSampler(local)
    clocks.start()
    tp.tpmlp_timing_reset()
    tp.tpmlp_timing_enable(True)
    launches0 = tp.tpmlp_launch_count()
    ms = timed(blk.step, args.steps, 0, world, dev, stream)
    launches = tp.tpmlp_launch_count() - launches0
    tp.tpmlp_timing_enable(False)
    clk = clocks.stop()
    kt = tp.tpmlp_timing_read()
    status = tp.tpmlp_check_device_error()
    if status != 0:
        raise RuntimeError(f"device error word {status} after the timed region")

    ms_max = max_over_ranks(ms, world, dev)
    flops_step = cfg.fwd_flops() + cfg.bwd_flops()
    value = flops_step * args.steps * world / (ms_max * 1e-3) / 1e12
    ktab = kernel_table(kt, ms)
    dom = max(kt.items(), key=lambda kv: kv[1]["total_ms"])[0]
    dom_ms = kt[dom]["total_ms"] / kt[dom]["launches"]
    gemm_flops = 2.0 * cfg.N * cfg.D * cfg.F      # every GEMM of the step has this size
    achieved = gemm_flops / (dom_ms * 1e-3) / 1e12
    peak = pk["bf16_tflops_sustained"]
    roof = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
            "frac": achieved / peak, "traffic": load_traffic(dom), "kernel": dom,
            "peak_source": f"{pk['source']} bf16_tflops_sustained (kernel timed inside a "
                           f"back-to-back step loop)",
            "algorithmic_flops_per_launch": gemm_flops}

    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_max / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded; X, dY ~ N(0,1), W ~ N(0,0.02))",
        "config": {"workload": cfg.name, "N": cfg.N, "B": cfg.B, "L": cfg.L, "D": cfg.D,
                   "F": cfg.F, "T": cfg.T, "act": cfg.act, "bias": False,
                   "reduce_mode": args.mode, "pass": "forward+backward",
                   "l2": "inputs larger than L2 (weights 0.94 GB, activations 1.1 GB per step)",
                   "parallelism": f"replicas x{world} (T logical shards per GPU)"},
        "frac_of_peak_step": value / world / peak,
        "roofline": roof,
        "gpu_launches": launches,
        "clocks": clk,
        "kernels": ktab,
    }
    if rank == 0 and not args.no_e2e:
        n_e = args.steps
        e_ms, h2d, d2h = e2e_measure(blk, n_e, stream)
        line["e2e"] = {"value": flops_step * n_e / (e_ms * 1e-3) / 1e12, "unit": "TFLOP/s",
                       "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                       "ms_per_step": e_ms / n_e, "steps": n_e,
                       "copies": "batch X, dY in and results Y, dX out every step, pinned host "
                                 "memory, overlapped with compute on two copy streams; weights and "
                                 "their gradients resident"}
    del blk
    torch.cuda.empty_cache()
    if rank == 0 and not args.no_secondary:
        line["secondary"] = secondary(dev, stream, args.steps, pk)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline_mlp(cfg)
    if rank == 0:
        print(json.dumps(line))
    if world > 1:
        torch.distributed.destroy_process_group()


# ---------------------------------------------------------------------------
# reference arm: the float64 oracle on the host cores
# ---------------------------------------------------------------------------

def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    import oracle
    cfg = MLP_CONFIGS[WORKLOAD]
    tokens = 32
    inp = gen_mlp_inputs(cfg, N=tokens)
    W1 = oracle.mlp.as_f64(inp.W1)
    W2 = oracle.mlp.as_f64(inp.W2)

    def step():
        oracle.mlp.forward(inp.X, W1, None, W2, None, cfg.act)
        oracle.mlp.backward(inp.X, W1, None, W2, inp.dY, cfg.act)
    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    dt = time.perf_counter() - t0
    flops = 12.0 * tokens * cfg.D * cfg.F * args.steps
    value = flops / dt / 1e12
    cores = len(os.sched_getaffinity(0))
    sample = (f"{tokens} of {cfg.N} tokens per step, fwd+bwd, float64 numpy (OpenBLAS threads = "
              f"host cores)")
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": dt * 1e3 / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded)",
        "config": {"workload": cfg.name, "N": cfg.N, "D": cfg.D, "F": cfg.F, "T": cfg.T,
                   "act": cfg.act, "pass": "forward+backward"},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }))


def run_only_ce(args):
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    import __graft_entry__
    __graft_entry__.build()
    out = secondary(dev, torch.cuda.current_stream(dev), args.steps, peaks(), args.only_ce)
    print(json.dumps({"only": "vocab_ce", "tokens": args.only_ce, "results": out}))


def run_only_embedding(args):
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    import __graft_entry__
    __graft_entry__.build()
    print(json.dumps({"only": "vocab_embedding",
                      "results": measure_embedding(dev, args.steps, peaks())}))


def main():
    args = parse()
    if args.only_ce:
        run_only_ce(args)
        return
    if args.only_embedding:
        run_only_embedding(args)
        return
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
