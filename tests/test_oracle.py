"""Pins of the float64 oracle against values and facts that do not come from
the oracle itself: the pages' worked examples, hand derivations, closed
forms, finite differences and library routines (torch autograd, torch's
tanh-GELU, torch.logsumexp). CPU only."""

import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from oracle import mlp as omlp
from oracle import sharded as osh
from oracle import ce as oce
from workloads.gen import gen_random_mlp, gen_integer_mlp, gen_sparse_integer_mlp
from tests.tolerance import normwise_rel_err, TOL

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def load(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def arr(x):
    return np.asarray(x, dtype=np.float64)


# ---------------------------------------------------------------------------
# The pages' 2 -> 4 -> 2 worked example
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("storage", [torch.float32, torch.bfloat16])
def test_worked_example_forward(storage):
    g = load("worked_example.json")
    x = torch.tensor(g["x"], dtype=storage)
    W1 = torch.tensor(g["W1"], dtype=storage)
    W2 = torch.tensor(g["W2"], dtype=storage)
    out = omlp.forward(x, W1, None, W2, None, g["act"])
    np.testing.assert_array_equal(out["Y"], arr(g["expected"]["Y"]))
    sh = osh.forward(x, W1, None, W2, None, g["act"], g["T"])
    for r in range(g["T"]):
        np.testing.assert_array_equal(sh["H"][r], arr(g["expected"]["shard_H"][r]))
        np.testing.assert_array_equal(sh["P"][r], arr(g["expected"]["partials"][r]))
    np.testing.assert_array_equal(sh["Y"], arr(g["expected"]["Y"]))
    # pre-activations of the two shards (the page prints x @ W1 per rank)
    for r, zr in enumerate(g["expected"]["shard_Z"]):
        np.testing.assert_array_equal(out["Z"][:, 2 * r:2 * r + 2], arr(zr))


def test_worked_example_backward_hand_derived():
    g = load("worked_example.json")
    b = load("worked_example_backward.json")
    x, W1, W2, dY = arr(g["x"]), arr(g["W1"]), arr(g["W2"]), arr(b["dY"])
    out = omlp.backward(x, W1, None, W2, dY, "relu")
    e = b["expected"]
    np.testing.assert_array_equal(out["dZ"], arr(e["dZ"]))
    np.testing.assert_array_equal(out["dX"], arr(e["dX"]))
    for r in range(2):
        np.testing.assert_array_equal(out["dW2"][2 * r:2 * r + 2, :], arr(e["dW2_shards"][r]))
        np.testing.assert_array_equal(out["dW1"][:, 2 * r:2 * r + 2], arr(e["dW1_shards"][r]))
    parts = osh.backward_dx(x, W1, None, W2, dY, "relu", 2)
    for r in range(2):
        np.testing.assert_array_equal(parts["parts"][r], arr(e["dX_parts"][r]))
    np.testing.assert_array_equal(parts["dX"], arr(e["dX"]))
    # Jacobian dY_j / dx_i: backward with dY = e_j gives row j
    J = np.stack([omlp.backward(x, W1, None, W2, np.eye(2)[j:j + 1], "relu")["dX"][0]
                  for j in range(2)], axis=1)
    np.testing.assert_array_equal(J, arr(e["jacobian_dYj_dxi"]))


def test_relu_grad_at_zero_convention_is_observable(monkeypatch):
    """A planted change of convention (ReLU'(0) = 1) must break the pin."""
    g = load("worked_example.json")
    b = load("worked_example_backward.json")
    x, W1, W2 = arr(g["x"]), arr(g["W1"]), arr(g["W2"])
    real = omlp.act_grad

    def mutant(z, kind):
        if kind == "relu":
            return np.where(np.asarray(z) >= 0.0, 1.0, 0.0)
        return real(z, kind)
    monkeypatch.setattr(omlp, "act_grad", mutant)
    J = np.stack([omlp.backward(x, W1, None, W2, np.eye(2)[j:j + 1], "relu")["dX"][0]
                  for j in range(2)], axis=1)
    np.testing.assert_array_equal(J, arr(b["expected"]["jacobian_if_relu_grad_at_0_were_1"]))
    assert not np.array_equal(J, arr(b["expected"]["jacobian_dYj_dxi"]))


def test_column_dx_example():
    """Linear column-parallel backward of the interview page: run it through
    the MLP oracle with W2 = I and ReLU on a strictly positive Z (so act' = 1
    and dZ = dY)."""
    g = load("column_dx_example.json")
    X, A, dY = arr(g["X"]), arr(g["A"]), arr(g["dY"])
    Z = X @ A
    assert np.all(Z > 0)
    out = omlp.backward(X, A, None, np.eye(2), dY, "relu")
    np.testing.assert_array_equal(out["dX"], arr(g["expected"]["dX"]))
    parts = osh.backward_dx(X, A, None, np.eye(2), dY, "relu", g["T"])
    for r in range(g["T"]):
        np.testing.assert_array_equal(parts["parts"][r], arr(g["expected"]["dX_parts"][r]))
    # the sum, not the concatenation
    assert parts["dX"].shape == (1, 2)


# ---------------------------------------------------------------------------
# Sharding invariance, bias once, the row-first counter-example
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("T", [1, 2, 4, 8])
@pytest.mark.parametrize("kind", ["relu", "gelu_tanh", "gelu_erf", "gelu_sigmoid"])
@pytest.mark.parametrize("bias", [False, True])
def test_shard_sum_equals_unsharded(T, kind, bias):
    inp = gen_random_mlp(N=24, D=32, F=64, T=T, dtype="f32", act=kind, bias=bias, seed=3)
    full = omlp.forward(inp.X, inp.W1, inp.b1, inp.W2, inp.b2, kind)
    sh = osh.forward(inp.X, inp.W1, inp.b1, inp.W2, inp.b2, kind, T)
    assert normwise_rel_err(sh["Y"], full["Y"]) <= 1e-12
    # the concatenated shard activations are the full H
    np.testing.assert_allclose(np.concatenate(sh["H"], axis=1), full["H"], rtol=0, atol=1e-12)
    dxs = osh.backward_dx(inp.X, inp.W1, inp.b1, inp.W2, inp.dY, kind, T)
    dfull = omlp.backward(inp.X, inp.W1, inp.b1, inp.W2, inp.dY, kind)
    assert normwise_rel_err(dxs["dX"], dfull["dX"]) <= 1e-12


@pytest.mark.parametrize("T", [1, 2, 4, 8])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_shard_sum_integer_inputs_bit_exact(T, dtype):
    inp = gen_integer_mlp(N=16, D=64, F=128, T=T, dtype=dtype, bias=True, seed=5)
    full = omlp.forward(inp.X, inp.W1, inp.b1, inp.W2, inp.b2, "relu")
    sh = osh.forward(inp.X, inp.W1, inp.b1, inp.W2, inp.b2, "relu", T)
    np.testing.assert_array_equal(sh["Y"], full["Y"])
    assert np.all(np.abs(full["Y"]) < 256) and np.all(full["Y"] == np.round(full["Y"]))


@pytest.mark.parametrize("T", [2, 4])
def test_sparse_integer_inputs_long_k_shard_sum_bit_exact(T):
    """The sparse {-1, 0, 1} inputs of the GPU's long-K bit-exact tests: at a
    reduction length of 4104 every stored value stays an integer within bf16's
    exact range, most outputs are non-zero, and the shard sum (forward) and the
    column-shard dX sum (backward) equal the unsharded definition exactly."""
    inp = gen_sparse_integer_mlp(N=48, D=4104, F=T * 1032, T=T, dtype="bf16", seed=7,
                                 density=(0.25, 0.02, 0.02, 0.25), bias=True)
    X = omlp.as_f64(inp.X)
    assert set(np.unique(X)) <= {-1.0, 0.0, 1.0}
    assert 0.2 < np.mean(X != 0) < 0.3 and 0.015 < np.mean(omlp.as_f64(inp.W1) != 0) < 0.025
    full = omlp.forward(inp.X, inp.W1, inp.b1, inp.W2, inp.b2, "relu")
    sh = osh.forward(inp.X, inp.W1, inp.b1, inp.W2, inp.b2, "relu", T)
    np.testing.assert_array_equal(sh["Y"], full["Y"])
    g = omlp.backward(inp.X, inp.W1, inp.b1, inp.W2, inp.dY, "relu")
    gs = osh.backward_dx(inp.X, inp.W1, inp.b1, inp.W2, inp.dY, "relu", T)
    np.testing.assert_array_equal(gs["dX"], g["dX"])
    for v in (full["Z"], full["Y"], g["dZ"], g["dX"], g["dW1"], g["dW2"], g["db1"]):
        assert np.all(v == np.round(v)) and np.max(np.abs(v)) <= 256
    assert np.mean(full["Y"] != 0) > 0.5


@pytest.mark.parametrize("T", [2, 4, 8])
def test_bias_added_per_shard_gives_y_plus_t_b2_and_is_detected(T):
    inp = gen_integer_mlp(N=8, D=32, F=64, T=T, dtype="f32", bias=True, seed=11)
    b2 = arr(inp.b2)
    assert np.any(b2 != 0)
    right = osh.forward(inp.X, inp.W1, inp.b1, inp.W2, inp.b2, "relu", T)["Y"]
    wrong = osh.forward(inp.X, inp.W1, inp.b1, inp.W2, inp.b2, "relu", T, bias_per_shard=True)["Y"]
    no_bias = osh.forward(inp.X, inp.W1, inp.b1, inp.W2, None, "relu", T)["Y"]
    # page's closed form: sum_r (P^(r) + b2) = Y_without_b2 + T b2
    np.testing.assert_array_equal(wrong, no_bias + T * b2[None, :])
    np.testing.assert_array_equal(wrong - right, (T - 1) * np.broadcast_to(b2, right.shape))
    # and the parity metric flags it, in both precisions
    assert normwise_rel_err(wrong, right) > TOL["bf16"]


def test_block_reduce_worked_example_and_bias_once():
    g = load("worked_example.json")
    parts = [arr(p) for p in g["expected"]["partials"]]
    np.testing.assert_array_equal(osh.block_reduce(parts, None), arr(g["expected"]["Y"]))
    b2 = np.array([0.5, -2.0])
    np.testing.assert_array_equal(osh.block_reduce(parts, b2), arr(g["expected"]["Y"]) + b2)


@pytest.mark.parametrize("kind", ["relu", "gelu_tanh", "gelu_erf", "gelu_sigmoid"])
def test_row_first_split_is_wrong(kind):
    rng = np.random.default_rng(0)
    X = rng.standard_normal((4, 8))
    W1 = rng.standard_normal((8, 32))
    good = omlp.act(X @ W1, kind)
    bad = osh.row_first_forward(X, W1, kind, 2)
    assert not np.allclose(bad, good)
    # degenerate case: with one shard nothing is split
    np.testing.assert_allclose(osh.row_first_forward(X, W1, kind, 1), good, rtol=0, atol=1e-12)


# ---------------------------------------------------------------------------
# Gradients: finite differences and torch autograd
# ---------------------------------------------------------------------------

def _fd_case(kind, seed):
    rng = np.random.default_rng(seed)
    while True:
        X = rng.standard_normal((3, 4))
        W1 = rng.standard_normal((4, 8)) * 0.7
        b1 = rng.standard_normal(8) * 0.3
        W2 = rng.standard_normal((8, 4)) * 0.5
        b2 = rng.standard_normal(4) * 0.3
        dY = rng.standard_normal((3, 4))
        if kind != "relu" or np.min(np.abs(X @ W1 + b1)) > 1e-3:
            return X, W1, b1, W2, b2, dY


@pytest.mark.parametrize("kind", ["relu", "gelu_tanh", "gelu_erf", "gelu_sigmoid"])
def test_backward_matches_central_finite_differences(kind):
    X, W1, b1, W2, b2, dY = _fd_case(kind, 7)
    h = 1e-6
    g = omlp.backward(X, W1, b1, W2, dY, kind)
    params = {"dX": X, "dW1": W1, "db1": b1, "dW2": W2, "db2": b2}

    def loss():
        return float(np.sum(dY * omlp.forward(X, W1, b1, W2, b2, kind)["Y"]))
    for name, p in params.items():
        num = np.zeros_like(p)
        it = np.nditer(p, flags=["multi_index"])
        for _ in it:
            i = it.multi_index
            old = p[i]
            p[i] = old + h
            lp = loss()
            p[i] = old - h
            lm = loss()
            p[i] = old
            num[i] = (lp - lm) / (2 * h)
        assert normwise_rel_err(g[name], num) <= 1e-6, name


@pytest.mark.parametrize("kind", ["relu", "gelu_tanh", "gelu_erf", "gelu_sigmoid"])
@pytest.mark.parametrize("bias", [False, True])
def test_backward_matches_torch_autograd(kind, bias):
    inp = gen_random_mlp(N=10, D=12, F=16, T=2, dtype="f32", act=kind, bias=bias, seed=2)
    t = {k: (None if v is None else v.double().clone().requires_grad_(True))
         for k, v in dict(X=inp.X, W1=inp.W1, b1=inp.b1, W2=inp.W2, b2=inp.b2).items()}
    Z = t["X"] @ t["W1"] + (t["b1"] if bias else 0.0)
    if kind == "relu":
        H = torch.relu(Z)
    elif kind == "gelu_sigmoid":
        H = torch.nn.functional.silu(1.702 * Z) / 1.702
    else:
        H = torch.nn.functional.gelu(Z, approximate="tanh" if kind == "gelu_tanh" else "none")
    Y = H @ t["W2"] + (t["b2"] if bias else 0.0)
    dY = inp.dY.double()
    (Y * dY).sum().backward()
    g = omlp.backward(inp.X, inp.W1, inp.b1, inp.W2, inp.dY, kind)
    f = omlp.forward(inp.X, inp.W1, inp.b1, inp.W2, inp.b2, kind)
    np.testing.assert_allclose(f["Y"], Y.detach().numpy(), rtol=1e-12, atol=1e-12)
    for ours, theirs in [("dX", "X"), ("dW1", "W1"), ("dW2", "W2")] + (
            [("db1", "b1"), ("db2", "b2")] if bias else []):
        np.testing.assert_allclose(g[ours], t[theirs].grad.numpy(), rtol=1e-12, atol=1e-12)


def test_gelu_tanh_matches_torch():
    z = torch.linspace(-8, 8, 4001, dtype=torch.float64, requires_grad=True)
    y = torch.nn.functional.gelu(z, approximate="tanh")
    y.sum().backward()
    zn = z.detach().numpy()
    np.testing.assert_allclose(omlp.act(zn, "gelu_tanh"), y.detach().numpy(), rtol=0, atol=1e-12)
    np.testing.assert_allclose(omlp.act_grad(zn, "gelu_tanh"), z.grad.numpy(), rtol=0, atol=1e-12)
    # closed-form values: act(0) = 0, act'(0) = 1/2, act(z) -> z for large z
    assert omlp.act(0.0, "gelu_tanh") == 0.0
    assert omlp.act_grad(0.0, "gelu_tanh") == 0.5
    assert abs(omlp.act(10.0, "gelu_tanh") - 10.0) < 1e-12


def test_gelu_erf_matches_torch_and_closed_forms():
    """The pages' exact GELU: torch's gelu(approximate='none') and its
    autograd in float64; GELU(0) = 0, GELU'(0) = 1/2, GELU(z) - GELU(-z) = z
    (Phi(z) + Phi(-z) = 1), GELU(z) -> z for large z."""
    z = torch.linspace(-8, 8, 4001, dtype=torch.float64, requires_grad=True)
    y = torch.nn.functional.gelu(z, approximate="none")
    y.sum().backward()
    zn = z.detach().numpy()
    np.testing.assert_allclose(omlp.act(zn, "gelu_erf"), y.detach().numpy(), rtol=0, atol=1e-12)
    np.testing.assert_allclose(omlp.act_grad(zn, "gelu_erf"), z.grad.numpy(), rtol=0, atol=1e-12)
    assert omlp.act(0.0, "gelu_erf") == 0.0
    assert omlp.act_grad(0.0, "gelu_erf") == 0.5
    np.testing.assert_allclose(omlp.act(zn, "gelu_erf") - omlp.act(-zn, "gelu_erf"), zn,
                               rtol=0, atol=1e-12)
    assert abs(omlp.act(10.0, "gelu_erf") - 10.0) < 1e-12
    # the erf and tanh forms are different functions (up to ~1e-3 apart)
    assert np.max(np.abs(omlp.act(zn, "gelu_erf") - omlp.act(zn, "gelu_tanh"))) > 1e-4


def test_gelu_sigmoid_matches_scaled_silu_and_approximates_gelu():
    """The interview page's sigmoid GELU equals SiLU(1.702 z) / 1.702 (torch's
    silu and autograd in float64); act(0) = 0, act'(0) = 1/2; it stays within
    0.021 of the exact GELU (the known accuracy of that approximation)."""
    z = torch.linspace(-10, 10, 4001, dtype=torch.float64, requires_grad=True)
    y = torch.nn.functional.silu(1.702 * z) / 1.702
    y.sum().backward()
    zn = z.detach().numpy()
    np.testing.assert_allclose(omlp.act(zn, "gelu_sigmoid"), y.detach().numpy(), rtol=0, atol=1e-12)
    np.testing.assert_allclose(omlp.act_grad(zn, "gelu_sigmoid"), z.grad.numpy(), rtol=0, atol=1e-12)
    assert omlp.act(0.0, "gelu_sigmoid") == 0.0
    assert omlp.act_grad(0.0, "gelu_sigmoid") == 0.5
    gap = np.max(np.abs(omlp.act(zn, "gelu_sigmoid") - omlp.act(zn, "gelu_erf")))
    assert 0.01 < gap < 0.021


def test_gelu_constant_mutation_is_detected(monkeypatch):
    monkeypatch.setattr(omlp, "GELU_CUBIC", 0.045)
    z = torch.linspace(-4, 4, 101, dtype=torch.float64)
    ref = torch.nn.functional.gelu(z, approximate="tanh").numpy()
    assert np.max(np.abs(omlp.act(z.numpy(), "gelu_tanh") - ref)) > 1e-6


def test_sampled_helpers_equal_full_computation():
    inp = gen_random_mlp(N=40, D=24, F=48, T=4, dtype="f32", act="gelu_tanh", bias=True, seed=9)
    f = omlp.forward(inp.X, inp.W1, inp.b1, inp.W2, inp.b2, "gelu_tanh")
    g = omlp.backward(inp.X, inp.W1, inp.b1, inp.W2, inp.dY, "gelu_tanh")
    rows = [0, 7, 39, 12]
    fidx = [0, 5, 47, 23]
    np.testing.assert_allclose(omlp.forward_rows(inp.X, inp.W1, inp.b1, inp.W2, inp.b2,
                                                 "gelu_tanh", rows)["Y"], f["Y"][rows],
                               rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(omlp.backward_rows_dx(inp.X, inp.W1, inp.b1, inp.W2, inp.dY,
                                                     "gelu_tanh", rows), g["dX"][rows],
                               rtol=1e-13, atol=1e-13)
    hu = omlp.backward_hidden_units(inp.X, inp.W1, inp.b1, inp.W2, inp.dY, "gelu_tanh", fidx)
    np.testing.assert_allclose(hu["dW1"], g["dW1"][:, fidx], rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(hu["dW2"], g["dW2"][fidx, :], rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(hu["db1"], g["db1"][fidx], rtol=1e-13, atol=1e-13)


# ---------------------------------------------------------------------------
# Vocab-parallel cross-entropy
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("V,T", [(16, 4), (1000, 8), (7, 7)])
def test_ce_uniform_logits_gives_log_v(V, T):
    z = np.full((5, V), 3.25)
    t = np.arange(5) % V
    out = oce.vocab_ce(z, t, T)
    np.testing.assert_allclose(out["loss"], math.log(V), rtol=0, atol=1e-14)
    np.testing.assert_array_equal(out["argmax"], np.zeros(5))   # ties -> lowest index
    np.testing.assert_array_equal(out["owner"], t // (V // T))


def test_ce_matches_torch_logsumexp_and_cross_entropy():
    g = torch.Generator().manual_seed(1)
    z = torch.randn(37, 96, generator=g, dtype=torch.float64) * 2.0
    t = torch.randint(0, 96, (37,), generator=g)
    out = oce.vocab_ce(z, t, 8)
    ref = torch.logsumexp(z, dim=1) - z[torch.arange(37), t]
    np.testing.assert_allclose(out["loss"], ref.numpy(), rtol=1e-13, atol=1e-13)
    ref_mean = torch.nn.functional.cross_entropy(z, t).item()
    assert abs(out["mean"] - ref_mean) < 1e-13
    np.testing.assert_array_equal(out["argmax"], torch.argmax(z, dim=1).numpy())


@pytest.mark.parametrize("T", [1, 2, 8])
def test_ce_shard_combine_equals_one_shot(T):
    g = torch.Generator().manual_seed(4)
    z = torch.randn(9, 64, generator=g, dtype=torch.float64) * 3.0
    t = torch.randint(0, 64, (9,), generator=g)
    one = oce.vocab_ce(z, t, T)
    sh = osh.vocab_ce_sharded(z.numpy(), t.numpy(), T)
    np.testing.assert_allclose(sh["loss"], one["loss"], rtol=1e-13, atol=1e-13)
    np.testing.assert_array_equal(sh["owner"], one["owner"])


def test_ce_one_element_per_shard_is_plain_softmax():
    z = np.array([[0.5, -1.0, 2.0, 0.0]])
    out = oce.vocab_ce(z, np.array([2]), 4)
    p = np.exp(z) / np.exp(z).sum()
    assert abs(out["loss"][0] + math.log(p[0, 2])) < 1e-14
    assert out["owner"][0] == 2


def test_ce_argmax_tie_break_lowest_index():
    z = np.array([[1.0, 5.0, 5.0, 2.0, 5.0, 0.0]])
    out = oce.vocab_ce(z, np.array([0]), 3)
    assert out["argmax"][0] == 1


def test_oracle_package_does_not_import_the_product():
    import sys
    assert "tensor_transformer_mlp_columnparallel_gb300" not in oracle.__dict__
    for mod in (oracle.mlp, oracle.ce, oracle.sharded):
        src = open(mod.__file__).read()
        assert "tensor_transformer_mlp_columnparallel_gb300" not in src
    del sys


# ---------------------------------------------------------------------------
# Vocab-parallel cross-entropy backward
# ---------------------------------------------------------------------------

def test_ce_backward_matches_torch_autograd():
    g = torch.Generator().manual_seed(5)
    z = (torch.randn(13, 40, generator=g, dtype=torch.float64) * 2.0).requires_grad_(True)
    t = torch.randint(0, 40, (13,), generator=g)
    torch.nn.functional.cross_entropy(z, t).backward()      # mean over tokens
    ours = oce.vocab_ce_backward(z.detach(), t, 1.0 / 13)
    np.testing.assert_allclose(ours, z.grad.numpy(), rtol=1e-12, atol=1e-14)


def test_ce_backward_matches_finite_differences_of_the_forward():
    rng = np.random.default_rng(3)
    z = rng.standard_normal((3, 10)) * 1.5
    t = np.array([2, 9, 0])
    h = 1e-6
    num = np.zeros_like(z)
    for i in range(z.shape[0]):
        for j in range(z.shape[1]):
            zp, zm = z.copy(), z.copy()
            zp[i, j] += h
            zm[i, j] -= h
            num[i, j] = (oce.vocab_ce(zp, t, 2)["loss"].sum() - oce.vocab_ce(zm, t, 2)["loss"].sum()) / (2 * h)
    np.testing.assert_allclose(oce.vocab_ce_backward(z, t, 1.0), num, rtol=1e-6, atol=1e-8)


def test_ce_backward_closed_forms_and_invariants():
    V = 64
    z = np.full((4, V), -0.75)
    t = np.array([0, 5, 63, 17])
    d = oce.vocab_ce_backward(z, t, 0.5)
    expect = np.full((4, V), 0.5 / V)
    expect[np.arange(4), t] -= 0.5
    np.testing.assert_allclose(d, expect, rtol=0, atol=1e-15)
    rng = np.random.default_rng(1)
    z = rng.standard_normal((20, 33)) * 3
    t = rng.integers(0, 33, 20)
    d = oce.vocab_ce_backward(z, t, 1.0)
    np.testing.assert_allclose(d.sum(axis=1), 0.0, atol=1e-13)       # rows of softmax - onehot sum to 0
    assert np.all(d[np.arange(20), t] < 0) and np.all(np.delete(d.ravel(), t + 33 * np.arange(20)) > 0)


@pytest.mark.parametrize("T", [1, 4, 11])
def test_ce_backward_sharded_equals_one_shot(T):
    rng = np.random.default_rng(T)
    z = rng.standard_normal((7, 44)) * 2
    t = rng.integers(0, 44, 7)
    np.testing.assert_allclose(osh.vocab_ce_backward_sharded(z, t, T, 0.25),
                               oce.vocab_ce_backward(z, t, 0.25), rtol=1e-13, atol=1e-15)


# ---------------------------------------------------------------------------
# Reduce-scatter block end and vocab-parallel embedding
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("T", [1, 2, 4])
def test_reduce_scatter_blocks_concatenate_to_the_all_reduce(T):
    inp = gen_integer_mlp(N=8 * T, D=16, F=32, T=T, dtype="f32", bias=True, seed=19)
    sh = osh.forward(inp.X, inp.W1, inp.b1, inp.W2, inp.b2, "relu", T)
    blocks = osh.block_reduce_scatter(sh["P"], inp.b2, T)
    assert len(blocks) == T and all(b.shape == (8, 16) for b in blocks)
    np.testing.assert_array_equal(np.concatenate(blocks, axis=0), sh["Y"])
    full = omlp.forward(inp.X, inp.W1, inp.b1, inp.W2, inp.b2, "relu")["Y"]
    np.testing.assert_array_equal(np.concatenate(blocks, axis=0), full)


def test_reduce_scatter_rejects_ragged_token_counts():
    with pytest.raises(ValueError):
        osh.block_reduce_scatter([np.zeros((5, 4))], None, 2)


@pytest.mark.parametrize("T", [1, 2, 4, 8])
def test_embedding_sharded_equals_gather(T):
    from oracle import embedding as oemb
    rng = np.random.default_rng(T)
    E = rng.standard_normal((64, 12))
    ids = rng.integers(0, 64, 40)
    out = oemb.vocab_embedding(ids, E)
    np.testing.assert_array_equal(out, E[ids])                  # the definition, by brute force
    np.testing.assert_array_equal(osh.vocab_embedding_sharded(ids, E, T), out)


def test_embedding_out_of_range_ids_give_zero_rows():
    from oracle import embedding as oemb
    E = np.arange(24, dtype=float).reshape(8, 3) + 1
    ids = np.array([0, 8, -1, 7])
    out = oemb.vocab_embedding(ids, E)
    np.testing.assert_array_equal(out[[1, 2]], 0.0)
    np.testing.assert_array_equal(out[[0, 3]], E[[0, 7]])
    np.testing.assert_array_equal(osh.vocab_embedding_sharded(ids, E, 4), out)


# ---------------------------------------------------------------------------
# SwiGLU gated MLP
# ---------------------------------------------------------------------------

def test_swiglu_matches_torch():
    g = torch.Generator().manual_seed(6)
    X = torch.randn(9, 12, generator=g, dtype=torch.float64)
    Wg, Wu = (torch.randn(12, 20, generator=g, dtype=torch.float64) * 0.5 for _ in range(2))
    Wd = torch.randn(20, 12, generator=g, dtype=torch.float64) * 0.5
    ref = (torch.nn.functional.silu(X @ Wg) * (X @ Wu)) @ Wd
    out = omlp.swiglu_forward(X, Wg, Wu, Wd)
    np.testing.assert_allclose(out["Y"], ref.numpy(), rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(omlp.silu(np.array([0.0, 1.0])), [0.0, 1.0 / (1.0 + np.exp(-1.0))],
                               rtol=0, atol=1e-15)


@pytest.mark.parametrize("T", [1, 2, 4])
def test_swiglu_same_column_split_equals_unsharded(T):
    rng = np.random.default_rng(T)
    X = rng.standard_normal((6, 8))
    Wg, Wu = rng.standard_normal((8, 16)), rng.standard_normal((8, 16))
    Wd = rng.standard_normal((16, 8))
    full = omlp.swiglu_forward(X, Wg, Wu, Wd)
    sh = osh.swiglu_forward_sharded(X, Wg, Wu, Wd, T)
    assert normwise_rel_err(sh["Y"], full["Y"]) <= 1e-12
    np.testing.assert_allclose(np.concatenate(sh["H"], axis=1), full["H"], rtol=0, atol=1e-12)


def test_swiglu_channel_tags_detect_misaligned_up_shards():
    """Channel tags (page §10: give gate/up recognisable channel numbers): with
    x = [1] and Wg[0, c] = Wu[0, c] = c + 1, channel c of H is SiLU(c + 1) (c + 1).
    Swapping the order of the up shards keeps every shape valid but moves the
    tags, and the result no longer equals the unsharded one."""
    F, T = 8, 2
    X = np.ones((1, 1))
    tags = np.arange(1, F + 1, dtype=float)[None, :]
    Wd = np.eye(F)[:, :1] + 0.1              # any row-shardable down projection
    full = omlp.swiglu_forward(X, tags, tags, Wd)
    np.testing.assert_allclose(full["H"][0], omlp.silu(tags[0]) * tags[0], rtol=1e-15)
    good = osh.swiglu_forward_sharded(X, tags, tags, Wd, T)
    np.testing.assert_allclose(np.concatenate(good["H"], axis=1), full["H"], rtol=1e-15)
    bad = osh.swiglu_forward_sharded(X, tags, tags, Wd, T, up_shard_order=[1, 0])
    assert not np.allclose(np.concatenate(bad["H"], axis=1), full["H"])
    assert normwise_rel_err(bad["Y"], full["Y"]) > TOL["bf16"]
