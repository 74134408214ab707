"""The exact-fp32 GEMM with its K range split across a CTA cluster.

When the 64 x 64 tiles of an fp32 GEMM are fewer than the SMs, up to 8 CTAs
of a cluster share each tile's K chunks and the leader adds the peers'
partial tiles in rank order. The small fp32 blocks below all take that path
(a few tiles each); they must match the float64 oracle within the fp32
bound, forward and backward, in both block-end modes, and repeated runs must
be bit-identical (the sum order is fixed by the ranks, not by timing).
"""

import pytest
import torch

import oracle
import tensor_transformer_mlp_columnparallel_gb300 as tp
from tests.gpu_helpers import to_gpu, run_forward, run_backward, cat_cols, cat_rows
from tests.tolerance import assert_close
from workloads.gen import gen_random_mlp

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)
    yield
    assert tp.tpmlp_check_device_error() == 0


SHAPES = [(64, 256, 1024, 2), (1, 512, 2048, 4), (33, 1000, 3000, 3), (17, 136, 8 * 200, 8)]


@pytest.mark.parametrize("mode", ["splitk", "partials"])
@pytest.mark.parametrize("N,D,F,T", SHAPES)
def test_f32_split_k_matches_oracle_and_repeats_bit_for_bit(N, D, F, T, mode):
    inp = gen_random_mlp(N=N, D=D, F=F, T=T, dtype="f32", act="relu", bias=True, seed=N + D)
    gp = to_gpu(inp)
    outs = []
    for _ in range(2):
        Y, H, Z = run_forward(gp, "relu", mode)
        dX, dW1, dW2, db1, db2 = run_backward(gp, H, Z, "relu", mode, bias_grads=True)
        torch.cuda.synchronize()
        outs.append([Y, cat_cols(H), dX, cat_cols(dW1), cat_rows(dW2)])
    for a, b in zip(outs[0], outs[1]):
        assert torch.equal(a, b)
    Y, H, dX, dW1, dW2 = outs[0]
    f = oracle.mlp.forward(inp.X, inp.W1, inp.b1, inp.W2, inp.b2, "relu")
    g = oracle.mlp.backward(inp.X, inp.W1, inp.b1, inp.W2, inp.dY, "relu")
    assert_close(Y, f["Y"], "f32", "Y")
    assert_close(H, f["H"], "f32", "H")
    assert_close(dX, g["dX"], "f32", "dX")
    assert_close(dW1, g["dW1"], "f32", "dW1")
    assert_close(dW2, g["dW2"], "f32", "dW2")
