"""Column->row tensor-parallel MLP block and vocab-parallel cross-entropy,
T logical shards resident on one GB300 (sm_103a).

The computation lives in libtpmlp.so (C-ABI: include/tpmlp.h), built by
``build.build()``. This package is its Python binding: ``_binding`` has the
C calls under the same names; the helpers below only allocate outputs and
workspace with torch (device memory and streams) and call them.
"""

from typing import List, Optional, Sequence

import torch

from . import _binding
from ._binding import (  # noqa: F401
    TpmlpError,
    tpmlp_backward,
    tpmlp_block_reduce,
    tpmlp_block_reduce_scatter,
    tpmlp_check_device_error,
    tpmlp_forward,
    tpmlp_forward_noalloc,
    tpmlp_forward_reduce_scatter,
    tpmlp_gemm_plan,
    tpmlp_launch_count,
    tpmlp_selftest_gemm_stall,
    tpmlp_selftest_wait_timeout,
    tpmlp_set_wait_timeout_ns,
    tpmlp_swiglu_forward,
    tpmlp_timing_enable,
    tpmlp_timing_read,
    tpmlp_timing_reset,
    tpmlp_vocab_ce,
    tpmlp_vocab_ce_backward,
    tpmlp_vocab_embedding,
    tpmlp_workspace_bytes,
    tpmlp_workspace_bytes_balanced,
)


def _workspace(nbytes: int, device) -> Optional[torch.Tensor]:
    if nbytes <= 0:
        return None
    return torch.empty(nbytes, dtype=torch.uint8, device=device)


def mlp_forward(X: torch.Tensor, W1: Sequence[torch.Tensor], W2: Sequence[torch.Tensor],
                b1: Optional[Sequence[torch.Tensor]] = None, b2: Optional[torch.Tensor] = None,
                act: str = "gelu_tanh", mode: str = "splitk", save_z: bool = True,
                workspace: Optional[torch.Tensor] = None):
    """Forward of the block. Returns (Y [N, D], H list of T [N, F/T],
    Z list or None)."""
    T = len(W1)
    N, D = X.shape
    Fs = W1[0].shape[1]
    dev, dt = X.device, X.dtype
    Y = torch.empty((N, D), dtype=dt, device=dev)
    H = [torch.empty((N, Fs), dtype=dt, device=dev) for _ in range(T)]
    Z = [torch.empty((N, Fs), dtype=dt, device=dev) for _ in range(T)] if save_z else None
    if workspace is None:
        workspace = _workspace(
            tpmlp_workspace_bytes_balanced(_binding.OP_FORWARD, dt, N, D, Fs * T, T, mode), dev)
    tpmlp_forward(X, list(W1), list(b1) if b1 is not None else None, list(W2), b2, Y, H, Z,
                  act, mode, workspace)
    return Y, H, Z


def mlp_backward(X, W1, W2, H, Z, dY, act: str = "gelu_tanh", mode: str = "splitk",
                 bias_grads: bool = False, workspace: Optional[torch.Tensor] = None):
    """Backward of the block. Returns (dX, dW1 list, dW2 list, db1 list or
    None, db2 or None)."""
    T = len(W1)
    N, D = X.shape
    Fs = W1[0].shape[1]
    dev, dt = X.device, X.dtype
    dX = torch.empty((N, D), dtype=dt, device=dev)
    dW1 = [torch.empty((D, Fs), dtype=dt, device=dev) for _ in range(T)]
    dW2 = [torch.empty((Fs, D), dtype=dt, device=dev) for _ in range(T)]
    db1 = [torch.empty((Fs,), dtype=dt, device=dev) for _ in range(T)] if bias_grads else None
    db2 = torch.empty((D,), dtype=dt, device=dev) if bias_grads else None
    if workspace is None:
        workspace = _workspace(
            tpmlp_workspace_bytes_balanced(_binding.OP_BACKWARD, dt, N, D, Fs * T, T, mode), dev)
    tpmlp_backward(X, list(W1), list(W2), list(H), list(Z), dY, dX, dW1, dW2, db1, db2, act, mode,
                   workspace)
    return dX, dW1, dW2, db1, db2


def vocab_ce(logits: torch.Tensor, targets: torch.Tensor, T: int, want_argmax: bool = True):
    """Returns (loss_per_token [N], loss_mean [1], argmax [N] int32 or None,
    target_owner [N] int32 or None)."""
    N = logits.shape[0]
    dev = logits.device
    loss = torch.empty((N,), dtype=torch.float32, device=dev)
    mean = torch.empty((1,), dtype=torch.float32, device=dev)
    amax = torch.empty((N,), dtype=torch.int32, device=dev) if want_argmax else None
    owner = torch.empty((N,), dtype=torch.int32, device=dev) if want_argmax else None
    tpmlp_vocab_ce(logits, targets, T, loss, mean, amax, owner)
    return loss, mean, amax, owner


def block_reduce(partials: List[torch.Tensor], b2: Optional[torch.Tensor], out_dtype: torch.dtype):
    N, D = partials[0].shape
    Y = torch.empty((N, D), dtype=out_dtype, device=partials[0].device)
    tpmlp_block_reduce(partials, b2, Y)
    return Y


def vocab_ce_backward(logits: torch.Tensor, targets: torch.Tensor, T: int,
                      loss_per_token: torch.Tensor, grad_scale: float, in_place: bool = False):
    """Gradient of grad_scale * sum_n loss_n with respect to the logits."""
    d = logits if in_place else torch.empty_like(logits)
    tpmlp_vocab_ce_backward(logits, targets, T, loss_per_token, grad_scale, d)
    return d


def mlp_forward_reduce_scatter(X, W1, W2, b1=None, b2=None, act: str = "gelu_tanh",
                               mode: str = "splitk", save_z: bool = True):
    """Forward whose block end is a reduce-scatter: returns (Y_rows list of T
    [N/T, D], H, Z)."""
    T = len(W1)
    N, D = X.shape
    Fs = W1[0].shape[1]
    dev, dt = X.device, X.dtype
    Y_rows = [torch.empty((N // T, D), dtype=dt, device=dev) for _ in range(T)]
    H = [torch.empty((N, Fs), dtype=dt, device=dev) for _ in range(T)]
    Z = [torch.empty((N, Fs), dtype=dt, device=dev) for _ in range(T)] if save_z else None
    ws = _workspace(tpmlp_workspace_bytes_balanced(_binding.OP_FORWARD, dt, N, D, Fs * T, T, mode), dev)
    tpmlp_forward_reduce_scatter(X, list(W1), list(b1) if b1 is not None else None, list(W2), b2,
                                 Y_rows, H, Z, act, mode, ws)
    return Y_rows, H, Z


def vocab_embedding(ids: torch.Tensor, table: Sequence[torch.Tensor]):
    """Embedding rows of `ids` from a table split by rows into len(table) shards."""
    out = torch.empty((ids.shape[0], table[0].shape[1]), dtype=table[0].dtype, device=ids.device)
    tpmlp_vocab_embedding(ids, list(table), out)
    return out


def swiglu_forward(X, Wg, Wu, Wd, mode: str = "splitk", save_gate_up: bool = False):
    """Gated MLP forward; returns (Y, H list, G list or None, U list or None)."""
    T = len(Wg)
    N, D = X.shape
    Fs = Wg[0].shape[1]
    dev, dt = X.device, X.dtype
    Y = torch.empty((N, D), dtype=dt, device=dev)
    H = [torch.empty((N, Fs), dtype=dt, device=dev) for _ in range(T)]
    G = [torch.empty((N, Fs), dtype=dt, device=dev) for _ in range(T)] if save_gate_up else None
    U = [torch.empty((N, Fs), dtype=dt, device=dev) for _ in range(T)] if save_gate_up else None
    ws = _workspace(tpmlp_workspace_bytes_balanced(_binding.OP_FORWARD, dt, N, D, Fs * T, T, mode), dev)
    tpmlp_swiglu_forward(X, list(Wg), list(Wu), list(Wd), Y, H, G, U, mode, ws)
    return Y, H, G, U
