"""Vocab-parallel embedding lookup in float64: the plain definition.

Source: textbook page (5688vip.com ... 04.html) §4.2.3 row-parallel
embedding; course notes (unpurerationalist) §3.4 "TP for Embedding": the
table [V, H] is split by rows over T ranks, every rank looks up its own rows
(zeros for ids it does not own) and an all-reduce SUM yields the embeddings.
The definition that sharded computation must reproduce is the gather

    out[n, :] = E[ids[n], :]

with an id outside [0, V) giving a zero row (no rank owns it).
"""

import numpy as np

from .mlp import as_f64


def vocab_embedding(ids, table):
    E = as_f64(table)
    ids = np.asarray(ids.cpu() if hasattr(ids, "cpu") else ids, dtype=np.int64)
    V, Hd = E.shape
    out = np.zeros((ids.shape[0], Hd))
    ok = (ids >= 0) & (ids < V)
    out[ok] = E[ids[ok]]
    return out
