"""Weight-streaming GEMMs (<= 64 token rows) whose K range is split across a
cluster of CTAs, against the float64 oracle.

For a few token rows the tiles are fewer than the SMs, so the library splits
each tile's k-blocks across 2, 3 or 4 CTAs of a cluster and adds the peers'
partial accumulators in the leader before the epilogue. Which split a shape
gets depends on the device's co-resident cluster counts, so the test asks the
library's own plan (tpmlp_gemm_plan) for a shape per split factor, checks
that at least two distinct factors occur, and runs the block's forward and
backward on each such shape in both block-end modes. The shard width
F/T = 1000 is not a multiple of the 64-wide k-block, so every shard ends in a
ragged k-block and the split boundaries fall at different places inside the
shards.
"""

import numpy as np
import pytest
import torch

import oracle
import tensor_transformer_mlp_columnparallel_gb300 as tp
from tests.tolerance import assert_close

pytestmark = pytest.mark.gpu

T = 2
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


def shapes_by_split(rows):
    """Model widths D for which the split-K row GEMM (M = rows, N = D,
    K = F/T folded over T shards) is planned with each (tile columns,
    K-split factor)."""
    found = {}
    for D in range(128, 160 * 128 + 1, 128):
        bn, _, ks = tp.tpmlp_gemm_plan(rows, D, FS, T, fold=True)
        found.setdefault((bn, ks), D)
    return found


def test_plans_use_several_split_factors():
    found = shapes_by_split(17)
    splits = sorted({ks for (_, ks) in found if ks > 1})
    assert len(splits) >= 2, f"plans found: {sorted(found)}"
    # a pair never splits K, and wide row counts never split
    assert tp.tpmlp_gemm_plan(4096, 4096, 4096, 4, fold=True)[2] == 1
    assert tp.tpmlp_gemm_plan(65, 1024, 8192, 2, fold=True)[2] == 1


def run_block(rows, D, mode, seed):
    g = torch.Generator().manual_seed(seed)
    X = torch.randn(rows, D, generator=g).to(torch.bfloat16)
    W1 = (torch.randn(D, T * FS, generator=g) / D ** 0.5).to(torch.bfloat16)
    W2 = (torch.randn(T * FS, D, generator=g) / (T * FS) ** 0.5).to(torch.bfloat16)
    dY = torch.randn(rows, D, generator=g).to(torch.bfloat16)
    gW1 = [W1[:, r * FS:(r + 1) * FS].contiguous().to(dev()) for r in range(T)]
    gW2 = [W2[r * FS:(r + 1) * FS].contiguous().to(dev()) for r in range(T)]
    gX = X.to(dev())
    # workspaces of the required size only: without the stream-K scratch the
    # few-token GEMMs take the cluster split that the plan above reports
    F = T * FS
    ws = [torch.empty(max(tp.tpmlp_workspace_bytes(op, torch.bfloat16, rows, D, F, T, mode), 256),
                      dtype=torch.uint8, device=dev()) for op in (0, 1)]
    Y, H, Z = tp.mlp_forward(gX, gW1, gW2, act="gelu_tanh", mode=mode, workspace=ws[0])
    dX, dW1, dW2, _, _ = tp.mlp_backward(gX, gW1, gW2, H, Z, dY.to(dev()), act="gelu_tanh", mode=mode,
                                         workspace=ws[1])
    torch.cuda.synchronize()
    f = oracle.mlp.forward(X, W1, None, W2, None, "gelu_tanh")
    b = oracle.mlp.backward(X, W1, None, W2, dY, "gelu_tanh")
    assert_close(Y, f["Y"], "bf16", "Y")
    assert_close(torch.cat([h.float() for h in H], dim=1), f["H"], "bf16", "H")
    assert_close(dX, b["dX"], "bf16", "dX")
    assert_close(torch.cat([w.float() for w in dW1], dim=1), b["dW1"], "bf16", "dW1")
    assert_close(torch.cat([w.float() for w in dW2], dim=0), b["dW2"], "bf16", "dW2")


@pytest.mark.parametrize("mode", ["splitk", "partials"])
@pytest.mark.parametrize("rows", [1, 17, 64])
def test_split_k_block_matches_oracle(rows, mode):
    found = shapes_by_split(rows)
    for (bn, ks), D in sorted(found.items()):
        if ks == 1:
            continue
        run_block(rows, D, mode, seed=1000 * rows + 10 * ks + bn // 128)
