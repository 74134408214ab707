"""Bit-exact parity at long reduction lengths, through every launch form of
the GEMMs, against the float64 oracle.

Inputs are sparse integers in {-1, 0, 1} (workloads.gen.gen_sparse_integer_mlp)
under ReLU. Every value the path stores (Z, H, Y, dZ, dX, dW1, dW2) is then an
integer of magnitude at most 256, which bf16 holds exactly, and every fp32
accumulation of such terms is exact, so the sharded GPU result must equal the
unsharded definition bit for bit whatever the order of the additions (page
"一层 MLP 太宽而放不下时怎样切？", §10: integer matrices checked against the
full-matrix answer, outputs, input gradients and weight gradients alike). A
dropped, repeated or misplaced k-block, tile, shard or split partial shows up
as a mismatch that the 2e-2 tolerance of the random-input tests could hide.
Each case first checks its own premise (magnitudes within 256) on the oracle.

Forms, asked of the library's own plan where the choice depends on the device:
- CTA pair with 128-deep K stages (more than 128 token rows), ragged in every
  dimension, reduction lengths 4104-4160, over several waves and bands of
  tiles: whole tiles of odd waves take their k-blocks from the last down
  (across the shard boundary of a folded K) and odd bands walk their tiles
  in reverse; the same block again with the plain ascending orders
  (TPMLP_ALT_ORDER=0, in a fresh process); the reduce-scatter forward's
  row-block epilogue over several waves and bands; the bias-gradient
  column sums in two passes and in one;
- single-CTA 128-row tiles (65-128 token rows, 64-deep stages);
- the cluster K split of 2, 3 and 4 CTAs (at most 64 token rows, no scratch);
- stream-K (at most 64 token rows, with the scratch), and the part-wave
  stream-K of larger GEMMs (CTA pairs or single CTAs: whole tiles for the
  full waves, the last wave's k-blocks dealt out);
- the fp32 GEMM's cluster K split (up to 8 CTAs per tile).
"""

import os
import subprocess
import sys

import numpy as np
import pytest
import torch

import oracle
import tensor_transformer_mlp_columnparallel_gb300 as tp
from tensor_transformer_mlp_columnparallel_gb300 import _binding
from workloads.gen import gen_sparse_integer_mlp

pytestmark = pytest.mark.gpu

MODES = ["splitk", "partials"]
BF16_EXACT = 256.0


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)
    yield
    assert tp.tpmlp_check_device_error() == 0


def dev():
    return torch.device("cuda:0")


def f64(t):
    return t.detach().double().cpu().numpy()


def expected(inp, bias_grads):
    """The oracle's forward and backward, after checking that every stored
    value is an integer bf16 holds exactly."""
    f = oracle.mlp.forward(inp.X, inp.W1, inp.b1, inp.W2, inp.b2, "relu")
    g = oracle.mlp.backward(inp.X, inp.W1, inp.b1, inp.W2, inp.dY, "relu")
    names = ["Z", "H", "Y"], ["dZ", "dX", "dW1", "dW2"] + (["db1", "db2"] if bias_grads else [])
    for src, keys in ((f, names[0]), (g, names[1])):
        for k in keys:
            v = src[k]
            assert np.all(v == np.round(v)), k
            if inp.dtype == "bf16":
                assert np.max(np.abs(v)) <= BF16_EXACT, (k, np.max(np.abs(v)))
    # many outputs are non-zero, so the comparison has something to catch
    assert np.mean(f["Y"] != 0) > 0.5 and np.mean(g["dW1"] != 0) > 0.05
    return f, g


def run_block(inp, mode, balanced, bias_grads):
    d = dev()
    N, D, F, T = inp.N, inp.D, inp.F, inp.T
    X = inp.X.to(d)
    dY = inp.dY.to(d)
    W1 = [w.to(d) for w in inp.W1_shards()]
    W2 = [w.contiguous().to(d) for w in inp.W2_shards()]
    b1 = None if inp.b1 is None else [b.contiguous().to(d) for b in inp.b1_shards()]
    b2 = None if inp.b2 is None else inp.b2.to(d)
    size = tp.tpmlp_workspace_bytes_balanced if balanced else tp.tpmlp_workspace_bytes
    ws = [torch.empty(max(size(op, X.dtype, N, D, F, T, mode), 256), dtype=torch.uint8, device=d)
          for op in (_binding.OP_FORWARD, _binding.OP_BACKWARD)]
    Y, H, Z = tp.mlp_forward(X, W1, W2, b1, b2, act="relu", mode=mode, workspace=ws[0])
    dX, dW1, dW2, db1, db2 = tp.mlp_backward(X, W1, W2, H, Z, dY, act="relu", mode=mode,
                                             bias_grads=bias_grads, workspace=ws[1])
    torch.cuda.synchronize()
    cat1 = lambda ts: torch.cat([t.float() for t in ts], dim=1)
    out = {"Y": Y, "H": cat1(H), "Z": cat1(Z), "dX": dX, "dW1": cat1(dW1),
           "dW2": torch.cat([t.float() for t in dW2], dim=0)}
    if bias_grads:
        out["db1"] = torch.cat([t.float() for t in db1])
        out["db2"] = db2
    return out


def assert_exact(inp, out, f, g, tag):
    for k in ("Y", "H", "Z"):
        np.testing.assert_array_equal(f64(out[k]), f[k], err_msg=f"{k} {tag}")
    for k in [k for k in ("dX", "dW1", "dW2", "db1", "db2") if k in out]:
        np.testing.assert_array_equal(f64(out[k]), g[k], err_msg=f"{k} {tag}")


# ---------------------------------------------------------------------------
# tensor-core GEMMs: CTA pair and single CTA
# ---------------------------------------------------------------------------

PAIR_CANDIDATES = [(4160, 4104, 2312), (4128, 4168, 2312), (4352, 4104, 2056),
                   (4096, 4104, 2056)]


def pair_shape(T=2):
    """The first (N, D, F/T), ragged against the 256-row pair tile and the
    64-wide box where possible, whose column GEMM (and dZ GEMM, the same
    problem), folded row GEMM (and dX GEMM) and dW2 GEMM all run as CTA pairs
    on this device (the plan weighs waves, so ragged shapes may prefer single
    CTAs)."""
    for N, D, Fs in PAIR_CANDIDATES:
        if all(tp.tpmlp_gemm_plan(M, Nn, K, T, fold=f)[1] == 2
               for M, Nn, K, f in ((N, Fs, D, False), (N, D, Fs, True), (Fs, D, N, False))):
            return N, D, Fs
    raise AssertionError("no candidate shape runs every GEMM as a CTA pair")


def test_cta_pair_128_deep_ring_long_k_ragged():
    """About 4100-4350 tokens, D about 4100, F/T = 2056-2312, ragged against the
    256-row pair tile, the 256-wide tile and the 64-wide box: the column, dZ
    and dX GEMMs reduce over D or F, the dW GEMMs over the tokens, all more
    than 4096 deep, in 128-deep stages of a 3-stage ring."""
    T = 2
    N, D, Fs = pair_shape(T)
    # premise: more than two waves of pair tiles and more than one band of
    # 12 tile rows in the column GEMM and the folded row GEMM
    pairs = torch.cuda.get_device_properties(0).multi_processor_count // 2
    m_tiles = -(-N // 256)
    for n_tiles in (T * -(-Fs // 256), -(-D // 256)):
        assert m_tiles * n_tiles > 2 * pairs and m_tiles > 12
    inp = gen_sparse_integer_mlp(N=N, D=D, F=T * Fs, T=T, dtype="bf16", seed=301)
    f, g = expected(inp, bias_grads=False)
    for mode in MODES:
        assert_exact(inp, run_block(inp, mode, True, False), f, g, f"pair {mode}")


def test_cta_pair_plain_orders_bit_exact():
    """The CTA-pair case with every tile's K loop ascending and every band
    walked forwards (the library reads TPMLP_ALT_ORDER once per process)."""
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = dict(os.environ, TPMLP_ALT_ORDER="0")
    r = subprocess.run([sys.executable, "-m", "pytest", os.path.abspath(__file__), "-q",
                        "-p", "no:cacheprovider", "-m", "gpu",
                        "-k", "test_cta_pair_128_deep_ring_long_k_ragged"],
                       env=env, cwd=root, capture_output=True, text=True, timeout=900)
    assert r.returncode == 0 and "1 passed" in r.stdout, r.stdout[-3000:] + r.stderr[-2000:]


def test_forward_reduce_scatter_over_waves_and_bands_bit_exact():
    """The row GEMM's row-block epilogue (rank r's token rows written to its
    own output buffer) over several waves and bands of pair tiles, where the
    alternating K and band orders apply: each rank's rows equal the
    unsharded definition's bit for bit, in both block-end modes (the
    reduce-scatter block end, page 1 §04)."""
    T = 4
    N, D, Fs = 4096, 4104, 2056
    bn, ctas, ks = tp.tpmlp_gemm_plan(N, D, Fs, T, fold=True, balanced=True)
    pairs = torch.cuda.get_device_properties(0).multi_processor_count // 2
    assert ctas == 2 and -(-N // 256) * -(-D // bn) > 2 * pairs and -(-N // 256) > 12
    inp = gen_sparse_integer_mlp(N=N, D=D, F=T * Fs, T=T, dtype="bf16", seed=350, bias=True)
    f, _ = expected(inp, bias_grads=False)
    d = dev()
    X = inp.X.to(d)
    W1 = [w.to(d) for w in inp.W1_shards()]
    W2 = [w.contiguous().to(d) for w in inp.W2_shards()]
    b1 = [b.contiguous().to(d) for b in inp.b1_shards()]
    b2 = inp.b2.to(d)
    Ns = N // T
    for mode in MODES:
        Y_rows, _, _ = tp.mlp_forward_reduce_scatter(X, W1, W2, b1, b2, act="relu", mode=mode)
        torch.cuda.synchronize()
        for r in range(T):
            np.testing.assert_array_equal(f64(Y_rows[r]), f["Y"][r * Ns:(r + 1) * Ns],
                                          err_msg=f"rank {r} rows, {mode}")


def test_bias_gradient_column_sums_bit_exact():
    """db1 = sum_n dZ^(r) and db2 = sum_n dY over 1100 token rows, with dZ
    shard rows and dY rows of 4104 columns: with the balanced workspace the
    two passes through the scratch (two column ranges per row, the second
    8 columns wide, and 17 uneven row chunks), with the plain workspace the
    one-pass strips; both equal to the oracle bit for bit."""
    T, N, D, Fs = 2, 1100, 4104, 4104
    inp = gen_sparse_integer_mlp(N=N, D=D, F=T * Fs, T=T, dtype="bf16", seed=360,
                                 density=(0.1, 0.02, 0.02, 0.05), bias=True)
    f, g = expected(inp, bias_grads=True)
    assert np.mean(g["db1"] != 0) > 0.5 and np.mean(g["db2"] != 0) > 0.5
    for mode in MODES:
        for balanced in (True, False):
            assert_exact(inp, run_block(inp, mode, balanced, True), f, g,
                         f"bias grads {mode} bal={balanced}")


def test_single_cta_tiles_long_k_with_biases():
    """100 token rows: the column, row, dZ and dX GEMMs run single-CTA
    128-row tiles over 64-deep stages (K = 4096 and 4 x 1024); biases and
    their gradients are integers too."""
    N, D, Fs, T = 100, 4096, 1024, 4
    assert tp.tpmlp_gemm_plan(N, Fs, D, T)[1] == 1
    inp = gen_sparse_integer_mlp(N=N, D=D, F=T * Fs, T=T, dtype="bf16", seed=302,
                                 density=(0.25, 0.02, 0.02, 0.25), bias=True)
    f, g = expected(inp, bias_grads=True)
    for mode in MODES:
        assert_exact(inp, run_block(inp, mode, True, True), f, g, f"single {mode}")


def part_wave_shapes(T=2):
    """Blocks whose folded row GEMM (more than 64 token rows) the plan runs
    with a part wave dealt out (stream-K after the full waves), one with CTA
    pairs and one with single-CTA tiles if the device's plans have them."""
    found = {}
    for N, D, Fs in ((4096, 4096, 2048), (2048, 4096, 1024), (4160, 4104, 2056), (1024, 2048, 2048),
                     (100, 4096, 1024), (120, 2048, 2048), (96, 8192, 1024)):
        bn, ctas, ks = tp.tpmlp_gemm_plan(N, D, Fs, T, fold=True, balanced=True)
        if ks == 0:
            found.setdefault(ctas, (N, D, Fs))
    return found


def test_part_wave_stream_k_bit_exact():
    """The whole tiles of the full waves, then the part wave's k-blocks dealt
    out to every unit, partial accumulators summed through the scratch in
    unit order: equal to the oracle bit for bit, with and without the scratch
    (the form without it runs the part wave as whole tiles)."""
    T = 2
    found = part_wave_shapes(T)
    assert 2 in found, found
    for ctas, (N, D, Fs) in sorted(found.items()):
        dens = (0.1, 0.02, 0.02, 0.04) if N > 1000 else (0.25, 0.02, 0.02, 0.25)
        inp = gen_sparse_integer_mlp(N=N, D=D, F=T * Fs, T=T, dtype="bf16", seed=340 + ctas,
                                     density=dens, bias=True)
        bias_grads = N <= 1000
        f, g = expected(inp, bias_grads=bias_grads)
        for mode in MODES:
            for balanced in (True, False):
                out = run_block(inp, mode, balanced, bias_grads)
                assert_exact(inp, out, f, g, f"part wave ctas={ctas} N={N} {mode} bal={balanced}")


# ---------------------------------------------------------------------------
# few token rows: cluster K split and stream-K
# ---------------------------------------------------------------------------

FS_FEW = 1096      # 17 full 64-deep k-blocks and a ragged one per shard
T_FEW = 4          # the folded K is 4 x 1096 = 4384


def few_density(D):
    """Densities for a few token rows: X and dY thinned in proportion above
    D = 4096, so that sums over D keep the same size at every width."""
    p = 0.25 * min(1.0, 4096.0 / D)
    return (p, 0.02, 0.02, p)


def split_shapes(rows):
    """Model widths D for which the folded row GEMM (and the dX GEMM, the
    same problem) is planned without the scratch with each (tile columns,
    K-split factor) that occurs."""
    found = {}
    for D in range(128, 160 * 128 + 1, 128):
        bn, _, ks = tp.tpmlp_gemm_plan(rows, D, FS_FEW, T_FEW, fold=True)
        found.setdefault((bn, ks), D)
    return found


@pytest.mark.parametrize("rows", [17, 64])
def test_cluster_k_split_every_factor_bit_exact(rows):
    found = split_shapes(rows)
    factors = sorted({ks for (_, ks) in found if ks > 1})
    assert len(factors) >= 2, sorted(found)
    for (bn, ks), D in sorted(found.items()):
        if ks <= 1:
            continue
        inp = gen_sparse_integer_mlp(N=rows, D=D, F=T_FEW * FS_FEW, T=T_FEW, dtype="bf16",
                                     seed=310 + ks, density=few_density(D), bias=True)
        f, g = expected(inp, bias_grads=True)
        for mode in MODES:
            out = run_block(inp, mode, balanced=False, bias_grads=True)
            assert_exact(inp, out, f, g, f"rows={rows} D={D} bn={bn} ks={ks} {mode}")


def stream_k_shapes():
    """(rows, D, T) whose column GEMM (K = D >= 4096) the plan runs as
    stream-K given the scratch."""
    out = []
    for rows in (1, 16, 33, 64):
        for D, T in ((4096, 2), (4104, 3), (4096, 4), (6144, 2), (8192, 2)):
            if tp.tpmlp_gemm_plan(rows, 1000, D, T, balanced=True)[2] == 0:
                out.append((rows, D, T))
                break
    return out


def test_stream_k_bit_exact():
    shapes = stream_k_shapes()
    assert len(shapes) >= 2, shapes
    for i, (rows, D, T) in enumerate(shapes):
        inp = gen_sparse_integer_mlp(N=rows, D=D, F=T * 1000, T=T, dtype="bf16", seed=320 + i,
                                     density=few_density(D), bias=True)
        f, g = expected(inp, bias_grads=True)
        for mode in MODES:
            out = run_block(inp, mode, balanced=True, bias_grads=True)
            assert_exact(inp, out, f, g, f"stream-K rows={rows} D={D} T={T} {mode}")


# ---------------------------------------------------------------------------
# the fp32 GEMM's cluster K split
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("N,D,F,T", [(64, 4096, 2 * 128, 2),    # column GEMM: 4 tiles, 8-CTA split, K = 4096
                                     (64, 256, 4 * 1024, 4),    # row GEMM: 4 tiles, 8-CTA split, K = 4 x 1024
                                     (40, 4104, 3 * 136, 3)])   # ragged tiles and K chunks
def test_fp32_cluster_split_bit_exact(N, D, F, T):
    inp = gen_sparse_integer_mlp(N=N, D=D, F=F, T=T, dtype="f32", seed=330 + T,
                                 density=(0.25, 0.02, 0.02, 0.25), bias=True)
    f, g = expected(inp, bias_grads=True)
    for mode in MODES:
        assert_exact(inp, run_block(inp, mode, False, True), f, g, f"fp32 {mode}")
