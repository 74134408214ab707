"""Vocab cross-entropy in float64: the plain definition.

Source: page "unpurerationalist ... 3.4 TP for Embedding" (LM-head bullets:
global max m, S = sum exp(z - m), the loss from the target's logit, and the
shard that holds the target) and the Megatron TP chapter §7.8. The sharded
combine is algebraically the same log-sum-exp; here it is taken over the
whole vocabulary at once.

loss_n = max_v z[n, v] + log(sum_v exp(z[n, v] - max_v z[n, v])) - z[n, t_n]
mean   = (1/N) sum_n loss_n
argmax = lowest index v with z[n, v] = max_v z[n, v]
owner  = t_n // (V / T)  (shards are contiguous vocab ranges)

Backward (same course notes, §3.6.4, first step; each shard computes its own
slice with the forward's global m and S, no exchange of logits):
dz[n, v] = g * (exp(z[n, v] - lse_n) - 1(v = t_n)),  lse_n = m_n + ln S_n,
with g the upstream gradient of each token's loss (1/N for the mean).
"""

import numpy as np

from .mlp import as_f64


def vocab_ce(logits, targets, T, row_chunk=256):
    z_all = logits
    t = np.asarray(targets.cpu() if hasattr(targets, "cpu") else targets, dtype=np.int64)
    N, V = z_all.shape
    if V % T != 0:
        raise ValueError("V must be divisible by T")
    Vs = V // T
    loss = np.empty(N, dtype=np.float64)
    amax = np.empty(N, dtype=np.int64)
    for n0 in range(0, N, row_chunk):
        z = as_f64(z_all[n0:n0 + row_chunk])
        m = z.max(axis=1)
        S = np.exp(z - m[:, None]).sum(axis=1)
        rows = np.arange(z.shape[0])
        loss[n0:n0 + z.shape[0]] = m + np.log(S) - z[rows, t[n0:n0 + z.shape[0]]]
        amax[n0:n0 + z.shape[0]] = np.argmax(z, axis=1)
    return {"loss": loss, "mean": float(loss.mean()) if N else float("nan"),
            "argmax": amax, "owner": t // Vs}


def vocab_ce_backward(logits, targets, grad_scale, row_chunk=256):
    """dL/dz for L = grad_scale * sum_n loss_n: grad_scale * (softmax - onehot)."""
    t = np.asarray(targets.cpu() if hasattr(targets, "cpu") else targets, dtype=np.int64)
    N, V = logits.shape
    out = np.empty((N, V), dtype=np.float64)
    for n0 in range(0, N, row_chunk):
        z = as_f64(logits[n0:n0 + row_chunk])
        m = z.max(axis=1, keepdims=True)
        e = np.exp(z - m)
        p = e / e.sum(axis=1, keepdims=True)
        rows = np.arange(z.shape[0])
        p[rows, t[n0:n0 + z.shape[0]]] -= 1.0
        out[n0:n0 + z.shape[0]] = grad_scale * p
    return out
