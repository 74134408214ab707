"""Vocab-parallel cross-entropy backward on the GPU against the float64
oracle (normwise max relative error per tensor, fp32 bar 1e-5)."""

import numpy as np
import pytest
import torch

import oracle
import tensor_transformer_mlp_columnparallel_gb300 as tp
from tensor_transformer_mlp_columnparallel_gb300 import _binding
from tests.tolerance import assert_close
from workloads.configs import CE_CONFIGS
from workloads.gen import gen_ce_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)
    yield
    assert tp.tpmlp_check_device_error() == 0


def dev():
    return torch.device("cuda:0")


def _run(inp, T, scale, in_place=False):
    z = inp.logits.to(dev())
    t = inp.targets.to(dev())
    loss, _, _, _ = tp.vocab_ce(z, t, T, want_argmax=False)
    d = tp.vocab_ce_backward(z, t, T, loss, scale, in_place=in_place)
    torch.cuda.synchronize()
    return d


def test_ce_backward_full_size_sampled_rows():
    """N=8192, V=128000, T=8, mean reduction (grad_scale 1/N)."""
    cfg = CE_CONFIGS["vocab_ce_n8192_v128000_t8"]
    inp = gen_ce_inputs(cfg)
    scale = 1.0 / cfg.N
    d = _run(inp, cfg.T, scale)
    rng = np.random.default_rng(0)
    rows = np.unique(np.concatenate([[0, cfg.N - 1], rng.choice(cfg.N, 192, replace=False)]))
    ref = oracle.ce.vocab_ce_backward(inp.logits[rows], inp.targets[rows], scale)
    assert_close(d[rows], ref, "f32", "dlogits rows")


@pytest.mark.parametrize("N,V,T", [(1, 8, 1), (33, 1000, 8), (17, 1001, 7), (5, 16, 16),
                                   (64, 4096, 2)])
def test_ce_backward_shapes(N, V, T):
    cfg = CE_CONFIGS["vocab_ce_n8192_v128000_t8"]
    inp = gen_ce_inputs(cfg, N=N, V=V, T=T)
    d = _run(inp, T, 1.0)
    assert_close(d, oracle.ce.vocab_ce_backward(inp.logits, inp.targets, 1.0), "f32", "dlogits")


def test_ce_backward_in_place_and_row_sums():
    cfg = CE_CONFIGS["vocab_ce_n8192_v128000_t8"]
    inp = gen_ce_inputs(cfg, N=48, V=3200, T=8)
    d = _run(inp, 8, 0.5, in_place=True)
    assert_close(d, oracle.ce.vocab_ce_backward(inp.logits, inp.targets, 0.5), "f32", "in place")
    # softmax - onehot: every row sums to zero
    assert float(d.double().sum(dim=1).abs().max()) < 1e-5


def test_ce_backward_bad_target_gives_nan_row_and_device_error():
    z = torch.randn(3, 32, device=dev())
    t = torch.tensor([1, 40, 2], device=dev())
    loss = torch.zeros(3, device=dev())
    d = torch.empty_like(z)
    tp.tpmlp_vocab_ce_backward(z, t, 4, loss, 1.0, d)
    assert tp.tpmlp_check_device_error() == _binding.ERR_ARG
    assert torch.isnan(d[1]).all() and torch.isfinite(d[0]).all() and torch.isfinite(d[2]).all()
