"""Seeded sweep over shapes, forward + backward against the float64 oracle.

24 shapes drawn once from a fixed seed: token counts from 1 to 700 (so the
few-token K-split, single-CTA and CTA-pair tile forms all occur), model and
shard widths that are multiples of 8 but rarely of the tile sizes, T in
{1, 2, 3, 4, 8}, both activations, both block-end modes, with and without
biases, mostly bf16 with some fp32. Tolerances as everywhere: normwise
2e-2 (bf16 storage) and 1e-5 (fp32).
"""

import numpy as np
import pytest
import torch

import oracle
import tensor_transformer_mlp_columnparallel_gb300 as tp
from tests.gpu_helpers import to_gpu, run_forward, run_backward, cat_cols, cat_rows
from tests.tolerance import assert_close
from workloads.gen import gen_random_mlp

pytestmark = pytest.mark.gpu


def _shapes():
    rng = np.random.default_rng(2024)
    out = []
    for i in range(24):
        T = int(rng.choice([1, 2, 3, 4, 8]))
        N = int(rng.choice([1, 7, 16, 33, 64, 65, 130, 257, 400, 700]))
        D = 8 * int(rng.integers(1, 129))           # 8 .. 1024
        Fs = 8 * int(rng.integers(1, 97))           # 8 .. 768 per shard
        dtype = "f32" if i % 6 == 5 else "bf16"
        act = "relu" if rng.random() < 0.3 else "gelu_tanh"
        mode = "partials" if rng.random() < 0.4 else "splitk"
        bias = bool(rng.random() < 0.5)
        out.append((N, D, T * Fs, T, dtype, act, mode, bias, 100 + i))
    return out


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)
    yield
    assert tp.tpmlp_check_device_error() == 0


@pytest.mark.parametrize("N,D,F,T,dtype,act,mode,bias,seed", _shapes())
def test_shape_sweep_forward_backward(N, D, F, T, dtype, act, mode, bias, seed):
    inp = gen_random_mlp(N=N, D=D, F=F, T=T, dtype=dtype, act=act, bias=bias, seed=seed)
    gp = to_gpu(inp)
    Y, H, Z = run_forward(gp, act, mode)
    dX, dW1, dW2, db1, db2 = run_backward(gp, H, Z, act, mode, bias_grads=bias)
    torch.cuda.synchronize()
    assert tp.tpmlp_check_device_error() == 0
    f = oracle.mlp.forward(inp.X, inp.W1, inp.b1, inp.W2, inp.b2, act)
    g = oracle.mlp.backward(inp.X, inp.W1, inp.b1, inp.W2, inp.dY, act)
    assert_close(Y, f["Y"], dtype, "Y")
    assert_close(cat_cols(H), f["H"], dtype, "H")
    assert_close(dX, g["dX"], dtype, "dX")
    assert_close(cat_cols(dW1), g["dW1"], dtype, "dW1")
    assert_close(cat_rows(dW2), g["dW2"], dtype, "dW2")
    if bias:
        assert_close(torch.cat([b.float() for b in db1]), g["db1"], dtype, "db1")
        assert_close(db2, g["db2"], dtype, "db2")
