"""Reduce-scatter block end and vocab-parallel embedding on the GPU against
the float64 oracle."""

import numpy as np
import pytest
import torch

import oracle
import tensor_transformer_mlp_columnparallel_gb300 as tp
from tensor_transformer_mlp_columnparallel_gb300 import _binding
from tests.gpu_helpers import to_gpu
from tests.tolerance import assert_close
from workloads.gen import gen_random_mlp, gen_integer_mlp

pytestmark = pytest.mark.gpu
MODES = ["partials", "splitk"]


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


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("T", [2, 4, 8])
def test_forward_reduce_scatter_matches_all_reduce_and_oracle(mode, dtype, T):
    inp = gen_random_mlp(N=64 * T, D=264, F=T * 136, T=T, dtype=dtype, act="gelu_tanh", bias=True,
                         seed=40 + T, with_dy=False)
    g = to_gpu(inp)
    Y_rows, H, Z = tp.mlp_forward_reduce_scatter(g["X"], g["W1"], g["W2"], g["b1"], g["b2"],
                                                 act="gelu_tanh", mode=mode)
    Y, _, _ = tp.mlp_forward(g["X"], g["W1"], g["W2"], g["b1"], g["b2"], act="gelu_tanh", mode=mode)
    torch.cuda.synchronize()
    assert len(Y_rows) == T and all(y.shape == (inp.N // T, inp.D) for y in Y_rows)
    # same arithmetic as the all-reduce form, only the rows land in T buffers
    assert torch.equal(torch.cat(Y_rows, 0), Y)
    f = oracle.mlp.forward(inp.X, inp.W1, inp.b1, inp.W2, inp.b2, "gelu_tanh")
    Ns = inp.N // T
    for r in range(T):
        assert_close(Y_rows[r], f["Y"][r * Ns:(r + 1) * Ns], dtype, f"rank {r} rows")


@pytest.mark.parametrize("N,T", [(32, 2), (64, 4), (16, 8)])
def test_forward_reduce_scatter_through_the_k_split(N, T):
    """A few tokens: the split-K row GEMM shares each tile's k-blocks across a
    CTA cluster, and the leader's epilogue writes rank r's rows into Y_rows[r]
    after adding the peers' partials (with b2 once)."""
    D, Fs = 1024, 512
    assert tp.tpmlp_gemm_plan(N, D, Fs, T, fold=True)[2] > 1
    inp = gen_random_mlp(N=N, D=D, F=T * Fs, T=T, dtype="bf16", act="gelu_tanh", bias=True,
                         seed=90 + T, with_dy=False)
    g = to_gpu(inp)
    Y_rows, _, _ = tp.mlp_forward_reduce_scatter(g["X"], g["W1"], g["W2"], g["b1"], g["b2"],
                                                 act="gelu_tanh", mode="splitk")
    Y, _, _ = tp.mlp_forward(g["X"], g["W1"], g["W2"], g["b1"], g["b2"], act="gelu_tanh",
                             mode="splitk")
    torch.cuda.synchronize()
    assert torch.equal(torch.cat(Y_rows, 0), Y)
    f = oracle.mlp.forward(inp.X, inp.W1, inp.b1, inp.W2, inp.b2, "gelu_tanh")
    Ns = N // T
    for r in range(T):
        assert_close(Y_rows[r], f["Y"][r * Ns:(r + 1) * Ns], "bf16", f"rank {r} rows")


def test_forward_reduce_scatter_integer_inputs_bit_exact():
    T = 4
    inp = gen_integer_mlp(N=128, D=16, F=64, T=T, dtype="bf16", bias=True, seed=8, with_dy=False)
    g = to_gpu(inp)
    for mode in MODES:
        Y_rows, _, _ = tp.mlp_forward_reduce_scatter(g["X"], g["W1"], g["W2"], g["b1"], g["b2"],
                                                     act="relu", mode=mode)
        torch.cuda.synchronize()
        sh = oracle.sharded.forward(inp.X, inp.W1, inp.b1, inp.W2, inp.b2, "relu", T)
        blocks = oracle.sharded.block_reduce_scatter(sh["P"], inp.b2, T)
        for r in range(T):
            np.testing.assert_array_equal(f64(Y_rows[r]), blocks[r])


@pytest.mark.parametrize("D", [40, 41])
def test_block_reduce_scatter_standalone(D):
    g = torch.Generator().manual_seed(D)
    T, N = 3, 36
    parts = [torch.randn(N, D, generator=g) for _ in range(T)]
    b2 = torch.randn(D, generator=g) * 0.1
    out = [torch.empty(N // T, D, device=dev()) for _ in range(T)]
    tp.tpmlp_block_reduce_scatter([p.to(dev()) for p in parts], b2.to(dev()), out)
    torch.cuda.synchronize()
    ref = oracle.sharded.block_reduce_scatter(parts, b2, T)
    for r in range(T):
        assert_close(out[r], ref[r], "f32", f"block {r}")


def test_reduce_scatter_rejects_ragged_token_count():
    inp = gen_random_mlp(N=30, D=16, F=32, T=4, dtype="bf16", act="relu", bias=False, seed=1,
                         with_dy=False)
    g = to_gpu(inp)
    Y_rows = [torch.empty(8, 16, dtype=torch.bfloat16, device=dev()) for _ in range(4)]
    H = [torch.empty(30, 8, dtype=torch.bfloat16, device=dev()) for _ in range(4)]
    with pytest.raises(tp.TpmlpError) as e:
        tp.tpmlp_forward_reduce_scatter(g["X"], g["W1"], None, g["W2"], None, Y_rows, H, None,
                                        "relu", "splitk")
    assert e.value.status == _binding.ERR_SHAPE


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_vocab_embedding_textbook_shape(dtype):
    """Table 32000 x 8192 split over T = 4 (textbook §4.2.3), 4096 tokens."""
    V, Hd, T, N = 32000, 8192, 4, 4096
    g = torch.Generator().manual_seed(3)
    E = (torch.randn(V, Hd, generator=g) * 0.02).to(dtype)
    ids = torch.randint(0, V, (N,), generator=g)
    shards = [E[k * V // T:(k + 1) * V // T].contiguous().to(dev()) for k in range(T)]
    out = tp.vocab_embedding(ids.to(dev()), shards)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(f64(out), oracle.embedding.vocab_embedding(ids, E))


def test_vocab_embedding_odd_width_and_bad_ids():
    V, Hd, T = 12, 3, 3                 # 6-byte bf16 rows: the byte-wise path
    E = torch.arange(V * Hd, dtype=torch.float32).reshape(V, Hd).to(torch.bfloat16)
    ids = torch.tensor([0, 11, 12, -3, 5, 4])
    shards = [E[k * 4:(k + 1) * 4].contiguous().to(dev()) for k in range(T)]
    out = tp.vocab_embedding(ids.to(dev()), shards)
    assert tp.tpmlp_check_device_error() == _binding.ERR_ARG
    np.testing.assert_array_equal(f64(out), oracle.embedding.vocab_embedding(ids, E))
    np.testing.assert_array_equal(f64(out), oracle.sharded.vocab_embedding_sharded(ids, E, T))


@pytest.mark.parametrize("Hd", [8, 8192, 8200, 20480])
def test_vocab_embedding_bulk_path_rows_chunks_and_bad_ids(Hd):
    """16-byte aligned rows take the bulk-copy path: rows of one chunk, of
    exactly one 16 KB chunk, of a chunk plus a 16-byte tail, and of several
    chunks; bad ids (outside [0, V)) give zero rows and TPMLP_ERR_ARG."""
    V, T = 40, 4
    g = torch.Generator().manual_seed(Hd)
    E = torch.randn(V, Hd, generator=g).to(torch.bfloat16)
    ids = torch.randint(0, V, (300,), generator=g)
    ids[7], ids[150], ids[299] = -1, V, 10 * V
    shards = [E[k * (V // T):(k + 1) * (V // T)].contiguous().to(dev()) for k in range(T)]
    out = tp.vocab_embedding(ids.to(dev()), shards)
    assert tp.tpmlp_check_device_error() == _binding.ERR_ARG
    np.testing.assert_array_equal(f64(out), oracle.embedding.vocab_embedding(ids, E))
    good = ids[(ids >= 0) & (ids < V)][:64]
    out2 = tp.vocab_embedding(good.to(dev()), shards)
    assert tp.tpmlp_check_device_error() == 0
    np.testing.assert_array_equal(f64(out2), oracle.embedding.vocab_embedding(good, E))
