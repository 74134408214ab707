"""The per-shard algorithm in float64, used ONLY by the oracle's pins.

It restates the method's steps so the tests can show, on the CPU, that the
sharded computation equals the unsharded definition in ``oracle.mlp``:

- column shard r: Z^(r) = X W1^(r) + b1^(r), H^(r) = act(Z^(r)) with
  W1^(r) = W1[:, r*Fs:(r+1)*Fs] (page "一层 MLP 太宽而放不下时怎样切？", §02
  column equation);
- row shard r: P^(r) = H^(r) W2^(r), a full-shape [N, D] partial with
  W2^(r) = W2[r*Fs:(r+1)*Fs, :] (§02 row equation);
- block end: Y = sum_r P^(r) + b2, b2 added once (§04, §05);
- backward: dX = sum_r dZ^(r) W1^(r)^T (§06 equation).

``bias_per_shard=True`` plants the mistake of §05 (every shard adds the whole
b2 before the sum), which yields Y + T b2.
"""

import numpy as np

from .mlp import act, act_grad, as_f64


def split_columns(W1, T):
    W1 = as_f64(W1)
    Fs = W1.shape[1] // T
    return [W1[:, r * Fs:(r + 1) * Fs] for r in range(T)]


def split_rows(W2, T):
    W2 = as_f64(W2)
    Fs = W2.shape[0] // T
    return [W2[r * Fs:(r + 1) * Fs, :] for r in range(T)]


def forward(X, W1, b1, W2, b2, kind, T, bias_per_shard=False):
    X = as_f64(X)
    F = as_f64(W1).shape[1]
    if F % T != 0:
        raise ValueError("F must be divisible by T")
    Fs = F // T
    W1s, W2s = split_columns(W1, T), split_rows(W2, T)
    b1f = None if b1 is None else as_f64(b1)
    b2f = None if b2 is None else as_f64(b2)
    H, P = [], []
    for r in range(T):
        Zr = X @ W1s[r]
        if b1f is not None:
            Zr = Zr + b1f[r * Fs:(r + 1) * Fs][None, :]
        Hr = act(Zr, kind)
        Pr = Hr @ W2s[r]
        if bias_per_shard and b2f is not None:
            Pr = Pr + b2f[None, :]
        H.append(Hr)
        P.append(Pr)
    Y = P[0].copy()
    for r in range(1, T):
        Y = Y + P[r]
    if (not bias_per_shard) and b2f is not None:
        Y = Y + b2f[None, :]
    return {"H": H, "P": P, "Y": Y}


def block_reduce(partials, b2):
    """Block-end sum of full-shape partials, b2 added once (§04-§05):
    Y = sum_r P^(r) + b2, summed in float64."""
    out = as_f64(partials[0]).copy()
    for p in partials[1:]:
        out = out + as_f64(p)
    if b2 is not None:
        out = out + as_f64(b2)[None, :]
    return out


def block_reduce_scatter(partials, b2, T):
    """Reduce-scatter form of the block end (page "一层 MLP 太宽而放不下时怎样切？",
    §04): the sum of the full-shape partials is split by tokens, rank r keeping
    rows [r N/T, (r+1) N/T). Returns the T row blocks."""
    Y = block_reduce(partials, b2)
    N = Y.shape[0]
    if N % T != 0:
        raise ValueError("N must be divisible by T")
    Ns = N // T
    return [Y[r * Ns:(r + 1) * Ns] for r in range(T)]


def vocab_embedding_sharded(ids, table, T):
    """Row-split embedding (textbook page §4.2.3; course notes §3.4): shard k
    holds rows [k V/T, (k+1) V/T); for every token it returns its local row, or
    zeros when the id lies outside its range; the T results are summed."""
    E = as_f64(table)
    ids = np.asarray(ids, dtype=np.int64)
    V, Hd = E.shape
    Vs = V // T
    out = np.zeros((ids.shape[0], Hd))
    for k in range(T):
        local = ids - k * Vs
        mine = (local >= 0) & (local < Vs)
        part = np.zeros_like(out)
        part[mine] = E[k * Vs:(k + 1) * Vs][local[mine]]
        out = out + part
    return out


def backward_dx(X, W1, b1, W2, dY, kind, T):
    """Per-shard dX contributions dZ^(r) W1^(r)^T and their sum."""
    X, dY = as_f64(X), as_f64(dY)
    F = as_f64(W1).shape[1]
    Fs = F // T
    W1s, W2s = split_columns(W1, T), split_rows(W2, T)
    b1f = None if b1 is None else as_f64(b1)
    parts = []
    for r in range(T):
        Zr = X @ W1s[r]
        if b1f is not None:
            Zr = Zr + b1f[r * Fs:(r + 1) * Fs][None, :]
        dZr = (dY @ W2s[r].T) * act_grad(Zr, kind)
        parts.append(dZr @ W1s[r].T)
    total = parts[0].copy()
    for r in range(1, T):
        total = total + parts[r]
    return {"parts": parts, "dX": total}


def row_first_forward(X, W1, kind, T):
    """The wrong split of page "TP: Column / Row Parallel Linear 怎么切?"
    (the counter-example): split X by columns and W1 by rows, apply the
    activation to each partial, then sum. Differs from act(X W1) for any
    non-linear activation."""
    X, W1 = as_f64(X), as_f64(W1)
    D = X.shape[1]
    Ds = D // T
    out = None
    for r in range(T):
        part = act(X[:, r * Ds:(r + 1) * Ds] @ W1[r * Ds:(r + 1) * Ds, :], kind)
        out = part if out is None else out + part
    return out


def vocab_ce_sharded(logits, targets, T):
    """Per-shard (m_k, s_k) with s_k = sum_{v in k} exp(z - m_k), combined as
    m = max_k m_k, S = sum_k s_k exp(m_k - m); loss = m + log S - z[t]."""
    z = as_f64(logits)
    t = np.asarray(targets, dtype=np.int64)
    N, V = z.shape
    Vs = V // T
    m_k = np.stack([z[:, k * Vs:(k + 1) * Vs].max(axis=1) for k in range(T)], axis=1)
    s_k = np.stack([np.exp(z[:, k * Vs:(k + 1) * Vs] - m_k[:, k:k + 1]).sum(axis=1)
                    for k in range(T)], axis=1)
    m = m_k.max(axis=1)
    S = (s_k * np.exp(m_k - m[:, None])).sum(axis=1)
    owner = t // Vs
    zt = np.array([z[n, k * Vs + (t[n] - k * Vs)] for n, k in enumerate(owner)])
    return {"m_k": m_k, "s_k": s_k, "loss": m + np.log(S) - zt, "owner": owner}


def vocab_ce_backward_sharded(logits, targets, T, grad_scale):
    """Shard k computes its own slice from the global (m, S) of the forward:
    dz_k = g * (exp(z_k - m) / S - 1(v = t)), then the slices are concatenated."""
    z = as_f64(logits)
    t = np.asarray(targets, dtype=np.int64)
    N, V = z.shape
    Vs = V // T
    fwd = vocab_ce_sharded(z, t, T)
    m = fwd["m_k"].max(axis=1)
    S = (fwd["s_k"] * np.exp(fwd["m_k"] - m[:, None])).sum(axis=1)
    parts = []
    for k in range(T):
        zk = z[:, k * Vs:(k + 1) * Vs]
        dk = np.exp(zk - m[:, None]) / S[:, None]
        for n in range(N):
            if k * Vs <= t[n] < (k + 1) * Vs:
                dk[n, t[n] - k * Vs] -= 1.0
        parts.append(grad_scale * dk)
    return np.concatenate(parts, axis=1)


def swiglu_forward_sharded(X, Wg, Wu, Wd, T, up_shard_order=None):
    """Gate and up split by the SAME columns (§08): shard r computes
    H^(r) = SiLU(X Wg^(r)) * (X Wu^(r)) and P^(r) = H^(r) Wd^(r); Y = sum_r P^(r).
    `up_shard_order` plants the mistake the page warns about (up shards in a
    different order than gate shards): shapes stay valid, channels misalign."""
    from .mlp import silu
    X = as_f64(X)
    Wgs, Wus, Wds = split_columns(Wg, T), split_columns(Wu, T), split_rows(Wd, T)
    order = list(range(T)) if up_shard_order is None else list(up_shard_order)
    H, P = [], []
    for r in range(T):
        Hr = silu(X @ Wgs[r]) * (X @ Wus[order[r]])
        H.append(Hr)
        P.append(Hr @ Wds[r])
    Y = P[0].copy()
    for r in range(1, T):
        Y = Y + P[r]
    return {"H": H, "P": P, "Y": Y}
