"""Gated (SwiGLU) block on the GPU against the float64 oracle."""

import numpy as np
import pytest
import torch

import oracle
import tensor_transformer_mlp_columnparallel_gb300 as tp
from tests.tolerance import assert_close

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


def make(N, D, F, T, dtype, seed):
    g = torch.Generator().manual_seed(seed)
    st = torch.bfloat16 if dtype == "bf16" else torch.float32
    X = torch.randn(N, D, generator=g).to(st)
    Wg = (torch.randn(D, F, generator=g) / D ** 0.5).to(st)
    Wu = (torch.randn(D, F, generator=g) / D ** 0.5).to(st)
    Wd = (torch.randn(F, D, generator=g) / F ** 0.5).to(st)
    Fs = F // T
    cols = lambda W: [W[:, r * Fs:(r + 1) * Fs].contiguous().to(dev()) for r in range(T)]
    return X, Wg, Wu, Wd, X.to(dev()), cols(Wg), cols(Wu), [Wd[r * Fs:(r + 1) * Fs].contiguous().to(dev()) for r in range(T)]


def cat(ts):
    return torch.cat([t.float() for t in ts], dim=1)


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_swiglu_ragged_shapes(mode, dtype):
    X, Wg, Wu, Wd, gX, gWg, gWu, gWd = make(300, 520, 2 * 264, 2, dtype, 11)
    Y, H, G, U = tp.swiglu_forward(gX, gWg, gWu, gWd, mode=mode, save_gate_up=True)
    torch.cuda.synchronize()
    o = oracle.mlp.swiglu_forward(X, Wg, Wu, Wd)
    assert_close(Y, o["Y"], dtype, "Y")
    assert_close(cat(H), o["H"], dtype, "H")
    assert_close(cat(G), o["G"], dtype, "G")
    assert_close(cat(U), o["U"], dtype, "U")


@pytest.mark.parametrize("T", [1, 2, 4, 8])
def test_swiglu_shard_sweep(T):
    X, Wg, Wu, Wd, gX, gWg, gWu, gWd = make(256, 512, 2048, T, "bf16", 20 + T)
    Y, H, _, _ = tp.swiglu_forward(gX, gWg, gWu, gWd, mode="splitk")
    torch.cuda.synchronize()
    o = oracle.mlp.swiglu_forward(X, Wg, Wu, Wd)
    assert_close(Y, o["Y"], "bf16", "Y")
    assert_close(cat(H), o["H"], "bf16", "H")


def test_swiglu_llama_like_shape_sampled_rows():
    """N=4096, D=4096, F=11008, T=4 (F/T = 2752): sampled token rows."""
    X, Wg, Wu, Wd, gX, gWg, gWu, gWd = make(4096, 4096, 11008, 4, "bf16", 5)
    Y, H, _, _ = tp.swiglu_forward(gX, gWg, gWu, gWd, mode="splitk")
    torch.cuda.synchronize()
    rows = np.unique(np.concatenate([[0, 4095], np.random.default_rng(0).choice(4096, 48, replace=False)]))
    o = oracle.mlp.swiglu_forward(X[rows], Wg, Wu, Wd)
    assert_close(Y[rows], o["Y"], "bf16", "Y rows")
    assert_close(cat([h[rows] for h in H]), o["H"], "bf16", "H rows")


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_swiglu_channel_tags_stay_aligned(dtype):
    """Channel tags (page §10): x = e_0 and Wg[0, c] = Wu[0, c] = tag_c make
    channel c of H equal SiLU(tag_c) tag_c; every shard must pair the gate and
    up columns of the same channel."""
    T, D, F, N = 4, 16, 256, 8
    st = torch.bfloat16 if dtype == "bf16" else torch.float32
    tags = (torch.arange(F, dtype=torch.float32) % 17 - 8) / 4          # exact in bf16
    X = torch.zeros(N, D)
    X[:, 0] = 1
    Wg = torch.zeros(D, F)
    Wg[0] = tags
    Wu = torch.zeros(D, F)
    Wu[0] = tags
    Wd = torch.zeros(F, D)
    Wd[:, 0] = 1
    Fs = F // T
    gX = X.to(st).to(dev())
    gWg = [Wg[:, r * Fs:(r + 1) * Fs].contiguous().to(st).to(dev()) for r in range(T)]
    gWu = [Wu[:, r * Fs:(r + 1) * Fs].contiguous().to(st).to(dev()) for r in range(T)]
    gWd = [Wd[r * Fs:(r + 1) * Fs].contiguous().to(st).to(dev()) for r in range(T)]
    Y, H, _, _ = tp.swiglu_forward(gX, gWg, gWu, gWd, mode="partials")
    torch.cuda.synchronize()
    want = oracle.mlp.silu(tags.double().numpy()) * tags.double().numpy()
    assert_close(cat(H)[0], want, dtype, "tagged channels")
    assert_close(Y[:, 0], np.full(N, want.sum()), dtype, "Y")
