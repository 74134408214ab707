"""Parity of the CUDA path (called through the C-ABI) with the float64 oracle,
element by element on the same seeded inputs.

Tolerances (normwise max relative error, per output tensor): 1e-5 on the
fp32 path, 2e-2 on the bf16 path (bf16 storage, fp32 accumulation). Integer
inputs and the pages' worked example are compared bit for bit. The
cross-entropy's argmax and target-owner outputs are compared exactly.
"""

import json
import os

import numpy as np
import pytest
import torch

import oracle
import tensor_transformer_mlp_columnparallel_gb300 as tp
from tensor_transformer_mlp_columnparallel_gb300 import _binding
from tests.gpu_helpers import to_gpu, run_forward, run_backward, cat_cols, cat_rows, dev
from tests.tolerance import assert_close, normwise_rel_err, TOL
from workloads.configs import MLP_CONFIGS, CE_CONFIGS
from workloads.gen import gen_random_mlp, gen_integer_mlp, gen_mlp_inputs, gen_ce_inputs, MLPInputs

pytestmark = pytest.mark.gpu

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
MODES = ["partials", "splitk"]


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)
    yield
    assert tp.tpmlp_check_device_error() == 0


def f64(t):
    return t.detach().double().cpu().numpy()


def check_forward(inp, Y, H, Z, tol_dtype):
    f = oracle.mlp.forward(inp.X, inp.W1, inp.b1, inp.W2, inp.b2, inp.act)
    assert_close(Y, f["Y"], tol_dtype, "Y")
    assert_close(cat_cols(H), f["H"], tol_dtype, "H")
    if Z is not None:
        assert_close(cat_cols(Z), f["Z"], tol_dtype, "Z")
    return f


def check_backward(inp, grads, tol_dtype):
    dX, dW1, dW2, db1, db2 = grads
    g = oracle.mlp.backward(inp.X, inp.W1, inp.b1, inp.W2, inp.dY, inp.act)
    assert_close(dX, g["dX"], tol_dtype, "dX")
    assert_close(cat_cols(dW1), g["dW1"], tol_dtype, "dW1")
    assert_close(cat_rows(dW2), g["dW2"], tol_dtype, "dW2")
    if db1 is not None:
        assert_close(torch.cat([b.float() for b in db1]), g["db1"], tol_dtype, "db1")
        assert_close(db2, g["db2"], tol_dtype, "db2")
    return g


# ---------------------------------------------------------------------------
# the pages' worked example, bit for bit
# ---------------------------------------------------------------------------

def _worked_example(dtype, pad):
    """The 2 -> 4 -> 2 example; on the bf16 path (row pitches must be
    multiples of 8 elements) it is embedded in D = 8, F = 16 with zeros:
    shard 0's hidden units 0, 1 and shard 1's units 8, 9 carry the page's
    four units, the rest are zero and contribute nothing."""
    g = json.load(open(os.path.join(GOLDEN, "worked_example.json")))
    gb = json.load(open(os.path.join(GOLDEN, "worked_example_backward.json")))
    st = torch.float32 if dtype == "f32" else torch.bfloat16
    x, W1, W2 = torch.tensor(g["x"]), torch.tensor(g["W1"]), torch.tensor(g["W2"])
    dY = torch.tensor(gb["dY"])
    if pad:
        D, Fs = 8, 8
        Xp = torch.zeros(1, D); Xp[:, :2] = x
        W1p = torch.zeros(D, 2 * Fs); W1p[:2, 0:2] = W1[:, 0:2]; W1p[:2, Fs:Fs + 2] = W1[:, 2:4]
        W2p = torch.zeros(2 * Fs, D); W2p[0:2, :2] = W2[0:2]; W2p[Fs:Fs + 2, :2] = W2[2:4]
        dYp = torch.zeros(1, D); dYp[:, :2] = dY
        x, W1, W2, dY = Xp, W1p, W2p, dYp
    return g, gb, MLPInputs(X=x.to(st), W1=W1.to(st), W2=W2.to(st), b1=None, b2=None,
                            dY=dY.to(st), T=2, act="relu", dtype=dtype)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_worked_example_bit_exact(dtype):
    pad = dtype == "bf16"
    g, gb, inp = _worked_example(dtype, pad)
    e, eb = g["expected"], gb["expected"]
    gp = to_gpu(inp)
    Fs = inp.Fs
    # PARTIALS: shard activations and partial sums are visible
    N, D = inp.N, inp.D
    ws_bytes = tp.tpmlp_workspace_bytes(0, gp["X"].dtype, N, D, inp.F, 2, "partials")
    ws = torch.zeros(ws_bytes, dtype=torch.uint8, device=dev())
    Y, H, Z = tp.mlp_forward(gp["X"], gp["W1"], gp["W2"], None, None, act="relu", mode="partials",
                             workspace=ws)
    torch.cuda.synchronize()
    stride = ((N * D * 4 + 255) // 256) * 256
    for r in range(2):
        np.testing.assert_array_equal(f64(H[r])[:, :2], np.array(e["shard_H"][r], dtype=float))
        part = ws[r * stride:r * stride + N * D * 4].view(torch.float32).view(N, D)
        np.testing.assert_array_equal(f64(part)[:, :2], np.array(e["partials"][r], dtype=float))
    np.testing.assert_array_equal(f64(Y)[:, :2], np.array(e["Y"], dtype=float))
    if pad:
        assert np.all(f64(Y)[:, 2:] == 0)
    # SPLITK
    Y2, H2, Z2 = tp.mlp_forward(gp["X"], gp["W1"], gp["W2"], None, None, act="relu", mode="splitk")
    np.testing.assert_array_equal(f64(Y2)[:, :2], np.array(e["Y"], dtype=float))
    # backward, both modes
    for mode in MODES:
        dX, dW1, dW2, _, _ = tp.mlp_backward(gp["X"], gp["W1"], gp["W2"], H2, Z2, gp["dY"],
                                             act="relu", mode=mode)
        np.testing.assert_array_equal(f64(dX)[:, :2], np.array(eb["dX"], dtype=float))
        for r in range(2):
            np.testing.assert_array_equal(f64(dW2[r])[:2, :2], np.array(eb["dW2_shards"][r], dtype=float))
            np.testing.assert_array_equal(f64(dW1[r])[:2, :2], np.array(eb["dW1_shards"][r], dtype=float))


# ---------------------------------------------------------------------------
# integer inputs: sharded GPU result equals the unsharded definition exactly
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("T", [1, 2, 4, 8])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("mode", MODES)
def test_integer_inputs_bit_exact(T, dtype, mode):
    inp = gen_integer_mlp(N=150, D=16, F=8 * 8, T=T, dtype=dtype, bias=True, seed=21)
    f = oracle.mlp.forward(inp.X, inp.W1, inp.b1, inp.W2, inp.b2, "relu")
    assert np.max(np.abs(f["Y"])) <= 256
    gp = to_gpu(inp)
    Y, H, Z = run_forward(gp, "relu", mode)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(f64(Y), f["Y"])
    np.testing.assert_array_equal(f64(cat_cols(H)), f["H"])
    np.testing.assert_array_equal(f64(cat_cols(Z)), f["Z"])


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_bias_added_once_and_the_per_shard_mistake_is_detected(dtype):
    T = 4
    inp = gen_integer_mlp(N=64, D=16, F=64, T=T, dtype=dtype, bias=True, seed=33)
    gp = to_gpu(inp)
    for mode in MODES:
        Y, _, _ = run_forward(gp, "relu", mode)
        torch.cuda.synchronize()
        right = oracle.sharded.forward(inp.X, inp.W1, inp.b1, inp.W2, inp.b2, "relu", T)["Y"]
        wrong = oracle.sharded.forward(inp.X, inp.W1, inp.b1, inp.W2, inp.b2, "relu", T,
                                       bias_per_shard=True)["Y"]
        np.testing.assert_array_equal(f64(Y), right)
        assert normwise_rel_err(Y, wrong) > TOL["bf16"]


# ---------------------------------------------------------------------------
# random inputs, tolerances
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("mode", MODES)
def test_small_fp32_relu_block_forward_backward(mode):
    """N=64 (B=2, L=32), D=256, F=1024, T=2, fp32, ReLU, biases; X ~ N(0,1),
    W ~ N(0, 1/sqrt(fan_in)), b ~ U(-0.1, 0.1), seed 0."""
    cfg = MLP_CONFIGS["mlp_f32_relu_n64_d256_f1024_t2"]
    inp = gen_mlp_inputs(cfg, with_dy=True)
    gp = to_gpu(inp)
    Y, H, Z = run_forward(gp, "relu", mode)
    grads = run_backward(gp, H, Z, "relu", mode, bias_grads=True)
    torch.cuda.synchronize()
    check_forward(inp, Y, H, Z, "f32")
    check_backward(inp, grads, "f32")


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("act", ["relu", "gelu_tanh"])
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_ragged_shapes_forward_backward(mode, act, dtype):
    """Several tiles in every dimension plus a ragged tail: N = 300 (3 row
    tiles of 128, last one partial), D = 520, F/T = 264 (partial 256-wide
    column tile and partial 64-deep K block)."""
    inp = gen_random_mlp(N=300, D=520, F=2 * 264, T=2, dtype=dtype, act=act, bias=True, seed=5)
    gp = to_gpu(inp)
    Y, H, Z = run_forward(gp, act, mode)
    grads = run_backward(gp, H, Z, act, mode, bias_grads=True)
    torch.cuda.synchronize()
    check_forward(inp, Y, H, Z, dtype)
    check_backward(inp, grads, dtype)


@pytest.mark.parametrize("T", [1, 2, 4, 8, 16])
@pytest.mark.parametrize("mode", MODES)
def test_shard_count_sweep_bf16(T, mode):
    inp = gen_random_mlp(N=256, D=512, F=2048, T=T, dtype="bf16", act="gelu_tanh", bias=True, seed=T)
    gp = to_gpu(inp)
    Y, H, Z = run_forward(gp, "gelu_tanh", mode)
    grads = run_backward(gp, H, Z, "gelu_tanh", mode, bias_grads=True)
    torch.cuda.synchronize()
    check_forward(inp, Y, H, Z, "bf16")
    check_backward(inp, grads, "bf16")


def test_result_does_not_depend_on_t():
    """Same weights sliced for T = 1, 2, 4, 8: the GPU outputs agree (the
    shard sum equals the unsharded product)."""
    base = gen_random_mlp(N=128, D=256, F=1024, T=1, dtype="bf16", act="gelu_tanh", bias=True, seed=4)
    outs = []
    for T in (1, 2, 4, 8):
        inp = MLPInputs(X=base.X, W1=base.W1, W2=base.W2, b1=base.b1, b2=base.b2, dY=base.dY, T=T,
                        act="gelu_tanh", dtype="bf16")
        Y, _, _ = run_forward(to_gpu(inp), "gelu_tanh", "splitk")
        outs.append(f64(Y))
    for o in outs[1:]:
        assert normwise_rel_err(o, outs[0]) < 1e-2


def test_block_reduce_standalone():
    g = torch.Generator().manual_seed(7)
    for D, dt in [(40, torch.float32), (40, torch.bfloat16), (41, torch.float32), (41, torch.bfloat16)]:
        parts = [torch.randn(37, D, generator=g) for _ in range(3)]
        b2 = (torch.randn(D, generator=g) * 0.1).to(dt)
        Y = tp.block_reduce([p.to(dev()) for p in parts], b2.to(dev()), dt)
        torch.cuda.synchronize()
        ref = oracle.sharded.block_reduce(parts, b2)
        assert_close(Y, ref, "f32" if dt == torch.float32 else "bf16", f"block_reduce D={D}")
        if dt == torch.float32:
            assert normwise_rel_err(Y, ref) < 1e-6


# ---------------------------------------------------------------------------
# the named workloads at full size (sampled outputs where the oracle is slow)
# ---------------------------------------------------------------------------

def _rows(n, k, seed):
    rng = np.random.default_rng(seed)
    return np.unique(np.concatenate([[0, n - 1], rng.choice(n, size=min(k, n), replace=False)]))


@pytest.mark.parametrize("mode", MODES)
def test_d4096_f16384_t4_forward_full_size_sampled(mode):
    cfg = MLP_CONFIGS["mlp_bf16_gelu_n4096_d4096_f16384_t4"]
    inp = gen_mlp_inputs(cfg)
    gp = to_gpu(inp)
    Y, H, Z = run_forward(gp, cfg.act, mode)
    torch.cuda.synchronize()
    rows = _rows(inp.N, 64, 1)
    f = oracle.mlp.forward_rows(inp.X, inp.W1, inp.b1, inp.W2, inp.b2, cfg.act, rows)
    assert_close(Y[rows], f["Y"], "bf16", "Y rows")
    assert_close(cat_cols([h[rows] for h in H]), f["H"], "bf16", "H rows")


@pytest.mark.parametrize("mode", MODES)
def test_d8192_f28672_t8_forward_backward_full_size_sampled(mode):
    """The fwd+bwd workload in both block-end modes (split-K shard sum: the
    launch configuration the benchmark's headline times; T fp32 partials and
    the reduce: its PARTIALS figure), no bias: sampled rows of Y and dX,
    sampled hidden units of dW1 (columns) and dW2 (rows)."""
    cfg = MLP_CONFIGS["mlp_bf16_gelu_n8192_d8192_f28672_t8_fwdbwd"]
    inp = gen_mlp_inputs(cfg)
    gp = to_gpu(inp)
    Y, H, Z = run_forward(gp, cfg.act, mode)
    dX, dW1, dW2, _, _ = run_backward(gp, H, Z, cfg.act, mode, bias_grads=False)
    torch.cuda.synchronize()
    rows = _rows(inp.N, 48, 2)
    f = oracle.mlp.forward_rows(inp.X, inp.W1, None, inp.W2, None, cfg.act, rows)
    assert_close(Y[rows], f["Y"], "bf16", "Y rows")
    dx = oracle.mlp.backward_rows_dx(inp.X, inp.W1, None, inp.W2, inp.dY, cfg.act, rows)
    assert_close(dX[rows], dx, "bf16", "dX rows")
    fidx = _rows(cfg.F, 24, 3)
    hu = oracle.mlp.backward_hidden_units(inp.X, inp.W1, None, inp.W2, inp.dY, cfg.act, fidx)
    Fs = cfg.Fs
    got_dw1 = torch.stack([dW1[f // Fs][:, f % Fs].float() for f in fidx], dim=1)
    got_dw2 = torch.stack([dW2[f // Fs][f % Fs, :].float() for f in fidx], dim=0)
    assert_close(got_dw1, hu["dW1"], "bf16", "dW1 columns")
    assert_close(got_dw2, hu["dW2"], "bf16", "dW2 rows")


@pytest.mark.parametrize("mode", MODES)
def test_n16_weight_streaming_forward_full_size(mode):
    cfg = MLP_CONFIGS["mlp_bf16_gelu_n16_d12288_f49152_t8"]
    inp = gen_mlp_inputs(cfg)
    gp = to_gpu(inp)
    Y, H, Z = run_forward(gp, cfg.act, mode)
    torch.cuda.synchronize()
    check_forward(inp, Y, H, Z, "bf16")


# ---------------------------------------------------------------------------
# vocab-parallel cross-entropy
# ---------------------------------------------------------------------------

def _ce_check(logits, targets, T, rows=None):
    loss, mean, amax, owner = tp.vocab_ce(logits.to(dev()), targets.to(dev()), T)
    torch.cuda.synchronize()
    o = oracle.ce.vocab_ce(logits, targets, T)
    assert_close(loss, o["loss"], "f32", "loss")
    assert abs(float(mean.item()) - o["mean"]) <= 1e-5 * max(abs(o["mean"]), 1.0)
    np.testing.assert_array_equal(amax.cpu().numpy(), o["argmax"])
    np.testing.assert_array_equal(owner.cpu().numpy(), o["owner"])


def test_vocab_ce_full_size():
    cfg = CE_CONFIGS["vocab_ce_n8192_v128000_t8"]
    inp = gen_ce_inputs(cfg)
    _ce_check(inp.logits, inp.targets, cfg.T)


@pytest.mark.parametrize("N,V,T", [(1, 8, 1), (33, 1000, 8), (17, 1001, 7), (5, 16, 16),
                                   (64, 4096, 2), (3, 12, 3)])
def test_vocab_ce_shapes(N, V, T):
    """Vector path (V/T % 4 == 0) and scalar path (odd shard widths),
    one-element shards, a single shard."""
    cfg = CE_CONFIGS["vocab_ce_n8192_v128000_t8"]
    inp = gen_ce_inputs(cfg, N=N, V=V, T=T)
    _ce_check(inp.logits, inp.targets, T)


def test_vocab_ce_ties_take_lowest_index_and_uniform_rows_give_log_v():
    V, T = 64, 8
    logits = torch.zeros(4, V)
    logits[1, 10] = logits[1, 50] = 3.0
    logits[2, 63] = logits[2, 0] = 5.0
    logits[3] = 1.5
    targets = torch.tensor([0, 50, 63, 7])
    _ce_check(logits, targets, T)
    loss, _, amax, _ = tp.vocab_ce(logits.to(dev()), targets.to(dev()), T)
    assert abs(float(loss[3]) - np.log(V)) < 1e-5
    assert amax.cpu().tolist() == [0, 10, 0, 0]


def test_vocab_ce_bad_target_sets_device_error_and_nan():
    logits = torch.randn(4, 32)
    targets = torch.tensor([1, 32, 5, -1])
    loss, _, _, owner = tp.vocab_ce(logits.to(dev()), targets.to(dev()), 4)
    assert tp.tpmlp_check_device_error() == _binding.ERR_ARG
    l = loss.cpu()
    assert torch.isnan(l[1]) and torch.isnan(l[3]) and torch.isfinite(l[0]) and torch.isfinite(l[2])
    assert tp.tpmlp_check_device_error() == 0


# ---------------------------------------------------------------------------
# edge cases and failure detection
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_empty_token_batch(dtype):
    D, F, T = 16, 32, 2
    X = torch.empty(0, D, dtype=dtype, device=dev())
    W1 = [torch.randn(D, F // T, device=dev()).to(dtype) for _ in range(T)]
    W2 = [torch.randn(F // T, D, device=dev()).to(dtype) for _ in range(T)]
    Y, H, Z = tp.mlp_forward(X, W1, W2, act="relu", mode="partials")
    dX, dW1, dW2, db1, db2 = tp.mlp_backward(X, W1, W2, H, Z, torch.empty(0, D, dtype=dtype, device=dev()),
                                             act="relu", mode="partials", bias_grads=True)
    torch.cuda.synchronize()
    assert Y.shape == (0, D)
    for t in dW1 + dW2 + db1 + [db2]:
        assert torch.count_nonzero(t) == 0
    loss, mean, amax, owner = tp.vocab_ce(torch.empty(0, 8, device=dev()),
                                          torch.empty(0, dtype=torch.int64, device=dev()), 2)
    torch.cuda.synchronize()
    assert torch.isnan(mean).all()


def test_single_token_and_single_shard():
    inp = gen_random_mlp(N=1, D=8, F=8, T=1, dtype="bf16", act="gelu_tanh", bias=True, seed=8)
    gp = to_gpu(inp)
    for mode in MODES:
        Y, H, Z = run_forward(gp, "gelu_tanh", mode)
        grads = run_backward(gp, H, Z, "gelu_tanh", mode, bias_grads=True)
        torch.cuda.synchronize()
        check_forward(inp, Y, H, Z, "bf16")
        check_backward(inp, grads, "bf16")


def test_rejected_arguments_launch_nothing():
    D, Fs, T = 16, 8, 2
    X = torch.randn(4, D, device=dev()).bfloat16()
    W1 = [torch.randn(D, Fs, device=dev()).bfloat16() for _ in range(T)]
    W2 = [torch.randn(Fs, D, device=dev()).bfloat16() for _ in range(T)]
    Y = torch.empty(4, D, device=dev()).bfloat16()
    H = [torch.empty(4, Fs, device=dev()).bfloat16() for _ in range(T)]
    before = tp.tpmlp_launch_count()
    # misaligned X (offset by one element)
    Xbig = torch.randn(4 * D + 1, device=dev()).bfloat16()
    Xmis = Xbig[1:].view(4, D)
    with pytest.raises(tp.TpmlpError) as e:
        tp.tpmlp_forward(Xmis, W1, None, W2, None, Y, H, None, "relu", "splitk")
    assert e.value.status == _binding.ERR_ALIGN
    # PARTIALS without a workspace
    with pytest.raises(tp.TpmlpError) as e:
        tp.tpmlp_forward(X, W1, None, W2, None, Y, H, None, "relu", "partials", None)
    assert e.value.status == _binding.ERR_WORKSPACE
    # bf16 path with a row pitch that is not a multiple of 8 elements
    X6 = torch.randn(4, 6, device=dev()).bfloat16()
    W16 = [torch.randn(6, Fs, device=dev()).bfloat16() for _ in range(T)]
    W26 = [torch.randn(Fs, 6, device=dev()).bfloat16() for _ in range(T)]
    with pytest.raises(tp.TpmlpError) as e:
        tp.tpmlp_forward(X6, W16, None, W26, None, torch.empty(4, 6, device=dev()).bfloat16(), H,
                         None, "relu", "splitk")
    assert e.value.status == _binding.ERR_ALIGN
    # mixed element types (fp32 weights with a bf16 input) are refused by the binding
    with pytest.raises(TypeError):
        tp.tpmlp_forward(X, [w.float() for w in W1], None, W2, None, Y, H, None, "relu", "splitk")
    assert tp.tpmlp_launch_count() == before


def test_bounded_wait_times_out_and_the_context_survives():
    tp.tpmlp_selftest_wait_timeout(20_000_000)  # 20 ms
    assert tp.tpmlp_check_device_error() == _binding.ERR_TIMEOUT
    assert tp.tpmlp_check_device_error() == 0
    # the context is still usable: a normal call works and is exact
    test_integer_inputs_bit_exact(2, "bf16", "splitk")


def test_timing_records_every_kernel_kind():
    inp = gen_random_mlp(N=128, D=128, F=512, T=4, dtype="bf16", act="gelu_tanh", bias=True, seed=9)
    gp = to_gpu(inp)
    tp.tpmlp_timing_reset()
    tp.tpmlp_timing_enable(True)
    try:
        before = tp.tpmlp_launch_count()
        Y, H, Z = run_forward(gp, "gelu_tanh", "partials")
        run_backward(gp, H, Z, "gelu_tanh", "partials", bias_grads=True)
        t = tp.tpmlp_timing_read()
    finally:
        tp.tpmlp_timing_enable(False)
    names = set(t)
    assert {"col_gemm_bias_act", "row_gemm_partials", "block_reduce_bias", "bwd_dz_gemm_dact",
            "bwd_dw2_gemm", "bwd_dw1_gemm", "bwd_dx_gemm_partials", "block_reduce_dx",
            "bias_grad_colsum"} <= names
    assert tp.tpmlp_launch_count() - before == sum(v["launches"] for v in t.values())
    assert all(v["total_ms"] > 0 for v in t.values())


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("mode", MODES)
def test_inference_forward_without_saved_z(dtype, mode):
    inp = gen_random_mlp(N=200, D=264, F=4 * 136, T=4, dtype=dtype, act="gelu_tanh", bias=True,
                         seed=12, with_dy=False)
    gp = to_gpu(inp)
    Y, H, Z = run_forward(gp, "gelu_tanh", mode, save_z=False)
    torch.cuda.synchronize()
    assert Z is None
    check_forward(inp, Y, H, None, dtype)


def test_max_shard_count_and_beyond():
    """T = 16 (the library's maximum) runs; T = 17 is rejected before launch."""
    inp = gen_random_mlp(N=256, D=256, F=16 * 64, T=16, dtype="bf16", act="relu", bias=True, seed=16)
    gp = to_gpu(inp)
    Y, H, Z = run_forward(gp, "relu", "splitk")
    grads = run_backward(gp, H, Z, "relu", "splitk", bias_grads=True)
    torch.cuda.synchronize()
    check_forward(inp, Y, H, Z, "bf16")
    check_backward(inp, grads, "bf16")
    W1 = gp["W1"] + [gp["W1"][0]]
    W2 = gp["W2"] + [gp["W2"][0]]
    H17 = H + [H[0]]
    with pytest.raises(tp.TpmlpError) as e:
        tp.tpmlp_forward(gp["X"], W1, None, W2, None, Y, H17, None, "relu", "splitk")
    assert e.value.status == _binding.ERR_SHAPE
