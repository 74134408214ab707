"""The tensor-core GEMM's own failure detection, in every launch form.

Page "一层 MLP 太宽而放不下时怎样切？" §11 lists a collective that waits forever
among the usual faults; on one GPU the equivalent is a wait inside a kernel
that never completes. Every wait in the GEMM is bounded: when one runs out
the kernel records TPMLP_ERR_TIMEOUT in the device error word, raises its
abort flag, and every role leaves through one exit that first waits for the
copies and MMAs it already issued, then frees tensor memory, with the CTAs
of a cluster leaving together.

tpmlp_selftest_gemm_stall makes one role of every CTA (epilogue, MMA issuer
or TMA producer) wait on a barrier that nothing completes, with a short
limit, so that wait runs out on purpose. For each launch form (single CTA,
CTA pair, cluster K split, stream-K of a few tokens, CTA pairs with the part
wave dealt out) and each role the test checks that the
forward returns promptly, that the device error word reads
TPMLP_ERR_TIMEOUT (and is clear after reading), and that the next normal call
on the same context gives exactly the result it gave before.
"""

import time

import pytest
import torch

import tensor_transformer_mlp_columnparallel_gb300 as tp
from tensor_transformer_mlp_columnparallel_gb300 import _binding
from workloads.gen import gen_random_mlp

pytestmark = pytest.mark.gpu

LIMIT_NS = 20_000_000          # 20 ms: far above any copy or MMA latency
DEFAULT_NS = 2_000_000_000
ROLES = {1: "epilogue", 2: "mma", 3: "producer"}


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)
    yield
    tp.tpmlp_selftest_gemm_stall(0)
    tp.tpmlp_set_wait_timeout_ns(DEFAULT_NS)
    assert tp.tpmlp_check_device_error() == 0


def dev():
    return torch.device("cuda:0")


def ksplit_width(rows, fs, T):
    for D in range(128, 160 * 128 + 1, 128):
        if tp.tpmlp_gemm_plan(rows, D, fs, T, fold=True)[2] > 1:
            return D
    raise AssertionError("no shape with a cluster K split")


def forms():
    """(name, N, D, F/T, T, balanced) of one block per launch form; the plan
    is checked to take that form for one of the block's GEMMs."""
    out = []
    assert tp.tpmlp_gemm_plan(2048, 2048, 2048, 2)[1] == 2
    out.append(("pair", 2048, 2048, 2048, 2, True))
    assert tp.tpmlp_gemm_plan(100, 1024, 1024, 2)[1] == 1
    out.append(("single", 100, 1024, 1024, 2, True))
    D = ksplit_width(17, 1000, 2)
    out.append(("ksplit", 17, D, 1000, 2, False))
    assert tp.tpmlp_gemm_plan(16, 1000, 1024, 2, balanced=True)[2] == 0
    out.append(("streamk", 16, 1024, 1000, 2, True))
    # CTA pairs with the part wave cut into K chunks (16 x 8 x 2 pair tiles
    # of the column GEMM: 3 full waves of 76 and 28 tiles in 2 chunks each)
    assert tp.tpmlp_gemm_plan(4096, 2048, 4096, 2, balanced=True)[1:] == (2, 0)
    out.append(("pair-streamk", 4096, 4096, 2048, 2, True))
    return out


def forward(g, mode, balanced):
    X, W1, W2 = g["X"], g["W1"], g["W2"]
    N, D = X.shape
    T, Fs = len(W1), W1[0].shape[1]
    size = tp.tpmlp_workspace_bytes_balanced if balanced else tp.tpmlp_workspace_bytes
    ws = torch.empty(max(size(_binding.OP_FORWARD, X.dtype, N, D, Fs * T, T, mode), 256),
                     dtype=torch.uint8, device=dev())
    Y, H, Z = tp.mlp_forward(X, W1, W2, g["b1"], g["b2"], act="gelu_tanh", mode=mode, workspace=ws)
    return Y, H


@pytest.mark.parametrize("role", sorted(ROLES))
@pytest.mark.parametrize("form", ["pair", "single", "ksplit", "streamk", "pair-streamk"])
def test_stalled_role_times_out_and_the_context_survives(form, role):
    name, N, D, Fs, T, balanced = next(f for f in forms() if f[0] == form)
    inp = gen_random_mlp(N=N, D=D, F=T * Fs, T=T, dtype="bf16", act="gelu_tanh", bias=True,
                         seed=500 + role, with_dy=False)
    g = {"X": inp.X.to(dev()), "W1": [w.to(dev()) for w in inp.W1_shards()],
         "W2": [w.contiguous().to(dev()) for w in inp.W2_shards()],
         "b1": [b.contiguous().to(dev()) for b in inp.b1_shards()], "b2": inp.b2.to(dev())}
    Y0, H0 = forward(g, "splitk", balanced)
    torch.cuda.synchronize()
    assert tp.tpmlp_check_device_error() == 0
    tp.tpmlp_set_wait_timeout_ns(LIMIT_NS)
    tp.tpmlp_selftest_gemm_stall(role)
    try:
        t0 = time.perf_counter()
        forward(g, "splitk", balanced)
        torch.cuda.synchronize()
        elapsed = time.perf_counter() - t0
    finally:
        tp.tpmlp_selftest_gemm_stall(0)
        tp.tpmlp_set_wait_timeout_ns(DEFAULT_NS)
    assert elapsed < 5.0, f"{form}/{ROLES[role]}: {elapsed:.2f} s"
    assert tp.tpmlp_check_device_error() == _binding.ERR_TIMEOUT, f"{form}/{ROLES[role]}"
    assert tp.tpmlp_check_device_error() == 0
    Y1, H1 = forward(g, "splitk", balanced)
    torch.cuda.synchronize()
    assert tp.tpmlp_check_device_error() == 0
    assert torch.equal(Y1, Y0)
    for a, b in zip(H1, H0):
        assert torch.equal(a, b)
