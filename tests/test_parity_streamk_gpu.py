"""Few-token GEMMs in the stream-K form, against the float64 oracle.

Given the optional scratch of tpmlp_workspace_bytes_balanced, a GEMM whose M
is a token count <= 64 deals its (tile, k-block) units out evenly to all SMs;
a tile whose K range several CTAs share is summed through the scratch by the
last CTA to finish it, in CTA order. The tests ask the library's plan which
GEMMs take that form, run the block's forward and backward on such shapes
(F/T = 1000: every shard ends in a ragged k-block, and with few units per
CTA one tile is shared by up to ten CTAs), compare with the oracle, check
that repeated runs are bit-identical (the sum order does not depend on which
CTA finishes last), and that the same call without the scratch (cluster
split or unsplit) agrees within the tolerance.
"""

import pytest
import torch

import oracle
import tensor_transformer_mlp_columnparallel_gb300 as tp
from tensor_transformer_mlp_columnparallel_gb300 import _binding
from tests.tolerance import assert_close, normwise_rel_err

pytestmark = pytest.mark.gpu

FS = 1000


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)
    yield
    assert tp.tpmlp_check_device_error() == 0


def dev():
    return torch.device("cuda:0")


def col_plan(N, D, T, balanced=True):
    return tp.tpmlp_gemm_plan(N, FS, D, T, balanced=balanced)


def test_plans_take_stream_k_only_with_the_scratch_and_few_rows():
    # the weight-streaming forward of N=16, D=12288, F=49152, T=8 (measured):
    # whole 192-column tiles for the column GEMM (256 tiles, 1.7 waves, started
    # together on the same weight rows), a K split over 2-CTA clusters of
    # 192-column tiles for the folded row GEMM (128 CTAs in two lockstep
    # fronts), whole 256-column tiles for the grouped partial-sum GEMM;
    # stream-K for none
    assert tp.tpmlp_gemm_plan(16, 6144, 12288, 8, balanced=True) == (192, 1, 1)
    assert tp.tpmlp_gemm_plan(16, 12288, 6144, 8, fold=True, balanced=True) == (192, 1, 2)
    assert tp.tpmlp_gemm_plan(16, 12288, 6144, 8, balanced=True) == (256, 1, 1)
    # 192-column tiles only for a few token rows
    assert tp.tpmlp_gemm_plan(65, 12288, 6144, 8, fold=True)[0] != 192
    # a few tiles of a small block take it (the shapes below)
    assert tp.tpmlp_gemm_plan(16, FS, 1024, 2, balanced=True)[2] == 0
    assert tp.tpmlp_gemm_plan(16, FS, 1024, 2, balanced=False)[2] != 0
    # the gated dual GEMM never takes it
    assert tp.tpmlp_gemm_plan(16, 6144, 12288, 8, dual=True, balanced=True)[2] != 0
    assert tp.tpmlp_gemm_plan(4096, 4096, 4096, 4, dual=True, balanced=True)[2] != 0
    # more than 64 rows: only the part wave's tiles are cut into K chunks, so
    # a GEMM whose pair tiles fill whole waves runs whole tiles (19 x 4 on 76
    # pairs), one with a small part wave takes it (16 x 16 x 4 = 1024 pair
    # tiles: 13 waves and 36 tiles in 2 chunks), and without the scratch none
    units = 76 if tp.tpmlp_gemm_plan(19 * 256, 1024, 4096, 1, balanced=False)[1] == 2 else 0
    if units:
        assert tp.tpmlp_gemm_plan(19 * 256, 1024, 4096, 1, balanced=True)[2] == 1
    assert tp.tpmlp_gemm_plan(4096, 4096, 4096, 4, balanced=True) == (256, 2, 0)
    assert tp.tpmlp_gemm_plan(4096, 4096, 4096, 4, balanced=False) == (256, 2, 1)


def shapes():
    """(N, D, T) whose column GEMM the plan runs as stream-K."""
    out = []
    for N in (1, 16, 33, 64):
        for D, T in ((1024, 2), (2048, 4), (1536, 3)):
            if col_plan(N, D, T)[2] == 0:
                out.append((N, D, T))
                break
    return out


def inputs(N, D, T, seed, fs=FS):
    g = torch.Generator().manual_seed(seed)
    F = T * fs
    X = torch.randn(N, D, generator=g).to(torch.bfloat16)
    W1 = (torch.randn(D, F, generator=g) / D ** 0.5).to(torch.bfloat16)
    W2 = (torch.randn(F, D, generator=g) / F ** 0.5).to(torch.bfloat16)
    b1 = (torch.randn(F, generator=g) * 0.1).to(torch.bfloat16)
    b2 = (torch.randn(D, generator=g) * 0.1).to(torch.bfloat16)
    dY = torch.randn(N, D, generator=g).to(torch.bfloat16)
    return X, W1, W2, b1, b2, dY


def run(X, W1, W2, b1, b2, dY, T, mode, balanced):
    N, D = X.shape
    F = W1.shape[1]
    fs = F // T
    gW1 = [W1[:, r * fs:(r + 1) * fs].contiguous().to(dev()) for r in range(T)]
    gW2 = [W2[r * fs:(r + 1) * fs].contiguous().to(dev()) for r in range(T)]
    gb1 = [b1[r * fs:(r + 1) * fs].contiguous().to(dev()) for r in range(T)]
    size = tp.tpmlp_workspace_bytes_balanced if balanced else tp.tpmlp_workspace_bytes
    wsf = torch.empty(max(size(_binding.OP_FORWARD, X.dtype, N, D, F, T, mode), 256),
                      dtype=torch.uint8, device=dev())
    wsb = torch.empty(max(size(_binding.OP_BACKWARD, X.dtype, N, D, F, T, mode), 256),
                      dtype=torch.uint8, device=dev())
    gX = X.to(dev())
    Y, H, Z = tp.mlp_forward(gX, gW1, gW2, gb1, b2.to(dev()), act="gelu_tanh", mode=mode,
                             workspace=wsf)
    dX, dW1, dW2, _, _ = tp.mlp_backward(gX, gW1, gW2, H, Z, dY.to(dev()), act="gelu_tanh",
                                         mode=mode, workspace=wsb)
    torch.cuda.synchronize()
    return (Y, torch.cat([h.float() for h in H], dim=1), dX,
            torch.cat([w.float() for w in dW1], dim=1), torch.cat([w.float() for w in dW2], dim=0))


def test_shapes_found():
    assert len(shapes()) >= 3, shapes()


@pytest.mark.parametrize("mode", ["splitk", "partials"])
def test_stream_k_forward_backward_against_oracle(mode):
    for i, (N, D, T) in enumerate(shapes()):
        X, W1, W2, b1, b2, dY = inputs(N, D, T, seed=40 + i)
        Y, H, dX, dW1, dW2 = run(X, W1, W2, b1, b2, dY, T, mode, balanced=True)
        f = oracle.mlp.forward(X, W1, b1, W2, b2, "gelu_tanh")
        b = oracle.mlp.backward(X, W1, b1, W2, dY, "gelu_tanh")
        tag = f"N={N} D={D} T={T} {mode}"
        assert_close(Y, f["Y"], "bf16", "Y " + tag)
        assert_close(H, f["H"], "bf16", "H " + tag)
        assert_close(dX, b["dX"], "bf16", "dX " + tag)
        assert_close(dW1, b["dW1"], "bf16", "dW1 " + tag)
        assert_close(dW2, b["dW2"], "bf16", "dW2 " + tag)


@pytest.mark.parametrize("mode", ["splitk", "partials"])
def test_few_token_block_with_more_tiles_than_sms(mode):
    """8 x 21 = 168 column tiles of 128 (88 of 256) for 152 SMs, in whatever
    form the plan takes with the scratch. F/T = 2600 ends every shard in a
    ragged k-block and a ragged tile."""
    N, D, T, fs = 16, 4096, 8, 2600
    X, W1, W2, b1, b2, dY = inputs(N, D, T, seed=99, fs=fs)
    Y, H, dX, dW1, dW2 = run(X, W1, W2, b1, b2, dY, T, mode, balanced=True)
    f = oracle.mlp.forward(X, W1, b1, W2, b2, "gelu_tanh")
    b = oracle.mlp.backward(X, W1, b1, W2, dY, "gelu_tanh")
    assert_close(Y, f["Y"], "bf16", "Y")
    assert_close(H, f["H"], "bf16", "H")
    assert_close(dX, b["dX"], "bf16", "dX")
    assert_close(dW1, b["dW1"], "bf16", "dW1")
    assert_close(dW2, b["dW2"], "bf16", "dW2")


def test_stream_k_is_deterministic_and_agrees_with_the_unbalanced_form():
    N, D, T = shapes()[1]
    X, W1, W2, b1, b2, dY = inputs(N, D, T, seed=7)
    first = run(X, W1, W2, b1, b2, dY, T, "splitk", balanced=True)
    for _ in range(3):
        again = run(X, W1, W2, b1, b2, dY, T, "splitk", balanced=True)
        for a, b in zip(first, again):
            assert torch.equal(a, b)
    other = run(X, W1, W2, b1, b2, dY, T, "splitk", balanced=False)
    for a, b, name in zip(first, other, ["Y", "H", "dX", "dW1", "dW2"]):
        assert normwise_rel_err(a, b) < 1e-2, name
