"""Activation epilogues element by element over a wide range of pre-activations.

With X = I (N = D = 128) the column GEMM returns Z = W1 exactly, so the saved
H is act(W1) entry by entry; with dY = e_0 rows and W2[:, 0] = 1 the hidden
gradient dH is 1 everywhere, so dZ = act'(Z) and dW1 = X^T dZ = act'(W1).
W1 holds 32768 bf16 values spread over [-12, 12], which covers both tails of
GELU (tanh and erf forms) and the zero of GELU'. The oracle evaluates act and
act' in float64 on the same (bf16-rounded) values.

Bounds (derived from the arithmetic, not fitted):
- bf16 path: round-to-nearest bf16 of the fp32 result moves it by at most
  2^-8 of its magnitude; the fp32 evaluation (sigmoid forms with __expf and
  __fdividef, relative error below 1e-5) adds a few percent of that, plus an
  absolute 2e-6 for the cancellation in act' near its zero (z ~ -0.75).
- fp32 path (tanhf): relative 1e-5 plus an absolute 3e-6, the worst case of
  0.5 z (1 - t^2) u'(z) with t = tanhf(u) carrying a couple of ulps near 1.
- the erf form (erff, a couple of ulps, on both paths) stays inside the same
  bounds: its one cancellation, 1 + erf(z / sqrt(2)) in the negative tail,
  costs at most ~1e-7 absolute after the factor z / 2.
"""

import numpy as np
import pytest
import torch

import oracle
import tensor_transformer_mlp_columnparallel_gb300 as tp

pytestmark = pytest.mark.gpu

N = D = 128
T = 2
F = 256


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)
    yield
    assert tp.tpmlp_check_device_error() == 0


def dev():
    return torch.device("cuda:0")


def z_grid():
    """[D, F] pre-activations in [-12, 12], rounded to bf16 (exact in fp32)."""
    z = torch.linspace(-12.0, 12.0, D * F, dtype=torch.float64).reshape(D, F)
    return z.to(torch.bfloat16).to(torch.float32)


def bound(o, dtype):
    o = np.abs(o)
    if dtype == "bf16":
        return 2.0 ** -8 * 1.05 * o + 2e-6
    return 1e-5 * o + 3e-6


def assert_elementwise(got, want, dtype, what):
    got = got.detach().double().cpu().numpy()
    err = np.abs(got - want)
    lim = bound(want, dtype)
    bad = err > lim
    assert not bad.any(), (
        f"{what}: {bad.sum()} entries outside the bound; worst at z-index "
        f"{np.unravel_index(np.argmax(err - lim), err.shape)}: got "
        f"{got.flat[np.argmax(err - lim)]}, want {want.flat[np.argmax(err - lim)]}")


def shards_cols(W, st):
    Fs = W.shape[1] // T
    return [W[:, r * Fs:(r + 1) * Fs].contiguous().to(st).to(dev()) for r in range(T)]


def shards_rows(W, st):
    Fs = W.shape[0] // T
    return [W[r * Fs:(r + 1) * Fs].contiguous().to(st).to(dev()) for r in range(T)]


@pytest.mark.parametrize("mode", ["splitk", "partials"])
@pytest.mark.parametrize("act", ["gelu_tanh", "relu", "gelu_erf", "gelu_sigmoid"])
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_act_and_act_grad_elementwise_over_both_tails(dtype, act, mode):
    st = torch.bfloat16 if dtype == "bf16" else torch.float32
    Zv = z_grid()
    X = torch.eye(N, D)
    W2 = torch.zeros(F, D)
    W2[:, 0] = 1.0
    dY = torch.zeros(N, D)
    dY[:, 0] = 1.0
    gX = X.to(st).to(dev())
    gW1 = shards_cols(Zv, st)
    gW2 = shards_rows(W2, st)
    Y, H, Zs = tp.mlp_forward(gX, gW1, gW2, act=act, mode=mode)
    dX, dW1, dW2, _, _ = tp.mlp_backward(gX, gW1, gW2, H, Zs, dY.to(st).to(dev()), act=act,
                                         mode=mode)
    torch.cuda.synchronize()
    z = Zv.double().numpy()
    # Z is X W1 = W1 exactly (one nonzero product per entry)
    assert torch.equal(torch.cat([t.float() for t in Zs], dim=1).cpu(), Zv)
    kind = act
    assert_elementwise(torch.cat([h.float() for h in H], dim=1), oracle.mlp.act(z, kind), dtype,
                       f"{act}(z)")
    assert_elementwise(torch.cat([g.float() for g in dW1], dim=1), oracle.mlp.act_grad(z, kind),
                       dtype, f"{act}'(z)")


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_silu_elementwise_over_both_tails(dtype):
    """Gated block with X = I and the up projection all ones: H = SiLU(z)."""
    st = torch.bfloat16 if dtype == "bf16" else torch.float32
    Zv = z_grid()
    X = torch.eye(N, D)
    Wu = torch.ones(D, F)
    Wd = torch.zeros(F, D)
    Wd[:, 0] = 1.0
    Y, H, G, U = tp.swiglu_forward(X.to(st).to(dev()), shards_cols(Zv, st), shards_cols(Wu, st),
                                   shards_rows(Wd, st), mode="partials", save_gate_up=True)
    torch.cuda.synchronize()
    assert torch.equal(torch.cat([g.float() for g in G], dim=1).cpu(), Zv)
    assert_elementwise(torch.cat([h.float() for h in H], dim=1),
                       oracle.mlp.silu(Zv.double().numpy()), dtype, "SiLU(z)")


@pytest.mark.parametrize("mode", ["splitk", "partials"])
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("act", ["gelu_erf", "gelu_sigmoid"])
def test_other_gelu_forms_block_forward_backward(dtype, mode, act):
    """The pages' exact (erf) GELU and the interview page's sigmoid GELU
    through a whole block, ragged shapes."""
    from tests.gpu_helpers import to_gpu, run_forward, run_backward, cat_cols, cat_rows
    from tests.tolerance import assert_close
    from workloads.gen import gen_random_mlp
    inp = gen_random_mlp(N=200, D=264, F=2 * 520, T=2, dtype=dtype, act=act, bias=True,
                         seed=77)
    gp = to_gpu(inp)
    Y, H, Z = run_forward(gp, act, mode)
    dX, dW1, dW2, db1, db2 = run_backward(gp, H, Z, act, mode, bias_grads=True)
    torch.cuda.synchronize()
    f = oracle.mlp.forward(inp.X, inp.W1, inp.b1, inp.W2, inp.b2, act)
    g = oracle.mlp.backward(inp.X, inp.W1, inp.b1, inp.W2, inp.dY, act)
    assert_close(Y, f["Y"], dtype, "Y")
    assert_close(cat_cols(H), f["H"], dtype, "H")
    assert_close(dX, g["dX"], dtype, "dX")
    assert_close(cat_cols(dW1), g["dW1"], dtype, "dW1")
    assert_close(cat_rows(dW2), g["dW2"], dtype, "dW2")
    assert_close(torch.cat([b.float() for b in db1]), g["db1"], dtype, "db1")
    assert_close(db2, g["db2"], dtype, "db2")
