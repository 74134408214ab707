"""Back-to-back launches with programmatic dependent launch.

Every tensor-core GEMM and block-end reduce is launched so that it may start
while the previous kernel on the stream winds down, and waits
(griddepcontrol.wait) before reading anything an earlier kernel wrote or
writing anything; the reduce lets the next kernel start its set-up while it
streams. These tests queue many calls
without synchronising, each writing fresh outputs, and require every result
to equal the first bit for bit (a read before the producer finished, or a
write while the consumer still reads, would show as a difference) and to
match the float64 oracle.
"""

import pytest
import torch

import oracle
import tensor_transformer_mlp_columnparallel_gb300 as tp
from tests.gpu_helpers import to_gpu, cat_cols, cat_rows
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


@pytest.mark.parametrize("mode", ["splitk", "partials"])
def test_weight_streaming_forwards_back_to_back(mode):
    """16 tokens, D = 4096, F = 8 x 2048 (the weight-streaming GEMM forms):
    24 forwards queued at once."""
    inp = gen_random_mlp(N=16, D=4096, F=8 * 2048, T=8, dtype="bf16", act="gelu_tanh", bias=True,
                         seed=601, with_dy=False)
    g = to_gpu(inp)
    outs = [tp.mlp_forward(g["X"], g["W1"], g["W2"], g["b1"], g["b2"], act="gelu_tanh",
                           mode=mode) for _ in range(24)]
    torch.cuda.synchronize()
    Y0, H0, _ = outs[0]
    for Y, H, _ in outs[1:]:
        assert torch.equal(Y, Y0)
        assert torch.equal(cat_cols(H), cat_cols(H0))
    f = oracle.mlp.forward(inp.X, inp.W1, inp.b1, inp.W2, inp.b2, "gelu_tanh")
    assert_close(Y0, f["Y"], "bf16", "Y")


@pytest.mark.parametrize("mode", ["splitk", "partials"])
def test_forward_backward_steps_back_to_back(mode):
    """Eight fwd+bwd steps queued at once on one shape that uses CTA pairs,
    the reduce (PARTIALS) and the backward chain (dZ read by dW1 and dX)."""
    inp = gen_random_mlp(N=512, D=1024, F=4 * 1024, T=4, dtype="bf16", act="gelu_tanh",
                         bias=True, seed=602)
    g = to_gpu(inp)
    res = []
    for _ in range(8):
        Y, H, Z = tp.mlp_forward(g["X"], g["W1"], g["W2"], g["b1"], g["b2"], act="gelu_tanh",
                                 mode=mode)
        dX, dW1, dW2, db1, db2 = tp.mlp_backward(g["X"], g["W1"], g["W2"], H, Z, g["dY"],
                                                 act="gelu_tanh", mode=mode, bias_grads=True)
        res.append([Y, dX, cat_cols(dW1), cat_rows(dW2), torch.cat(db1), db2])
    torch.cuda.synchronize()
    for r in res[1:]:
        for a, b in zip(r, res[0]):
            assert torch.equal(a, b)
    f = oracle.mlp.forward(inp.X, inp.W1, inp.b1, inp.W2, inp.b2, "gelu_tanh")
    b = oracle.mlp.backward(inp.X, inp.W1, inp.b1, inp.W2, inp.dY, "gelu_tanh")
    Y, dX, dW1, dW2, db1, db2 = res[0]
    assert_close(Y, f["Y"], "bf16", "Y")
    assert_close(dX, b["dX"], "bf16", "dX")
    assert_close(dW1, b["dW1"], "bf16", "dW1")
    assert_close(dW2, b["dW2"], "bf16", "dW2")


def test_fp32_blocks_back_to_back():
    inp = gen_random_mlp(N=64, D=256, F=1024, T=2, dtype="f32", act="relu", bias=True, seed=603)
    g = to_gpu(inp)
    outs = []
    for _ in range(16):
        Y, H, Z = tp.mlp_forward(g["X"], g["W1"], g["W2"], g["b1"], g["b2"], act="relu",
                                 mode="partials")
        dX = tp.mlp_backward(g["X"], g["W1"], g["W2"], H, Z, g["dY"], act="relu",
                             mode="partials")[0]
        outs.append((Y, dX))
    torch.cuda.synchronize()
    for Y, dX in outs[1:]:
        assert torch.equal(Y, outs[0][0]) and torch.equal(dX, outs[0][1])
    f = oracle.mlp.forward(inp.X, inp.W1, inp.b1, inp.W2, inp.b2, "relu")
    assert_close(outs[0][0], f["Y"], "f32", "Y")
