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
