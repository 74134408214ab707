"""CPU float64 oracle for the column->row sharded MLP block and the
vocab-parallel cross-entropy.

TEST INFRASTRUCTURE ONLY. Only the tests, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import it.
The product path (the CUDA library and its Python binding) never imports,
links or calls anything here, and this package never imports the product.

What it computes (plain definitions, no blocking, fusion or reordering):

- ``mlp.forward``: Z = X W1 + b1, H = act(Z), Y = H W2 + b2 with the FULL,
  unsharded W1 [D, F] and W2 [F, D] (page "一层 MLP 太宽而放不下时怎样切？",
  §01 and §02 equations; §05 for the single b2).
- ``mlp.backward``: dH = dY W2^T, dZ = dH * act'(Z), dW2 = H^T dY,
  dW1 = X^T dZ, dX = dZ W1^T, db1 = sum_n dZ, db2 = sum_n dY (same page,
  §06 and its dX equation).
- ``ce.vocab_ce``: per-token NLL = logsumexp_v z[n, v] - z[n, t_n], mean
  over tokens, argmax per token and the shard that owns each target
  (page "unpurerationalist ... 3.4 TP for Embedding", LM head bullets;
  Megatron TP chapter §7.8).
- ``mlp.swiglu_forward``: G = X Wg, U = X Wu, H = SiLU(G) * U, Y = H Wd
  (same page, §08 gated MLP).
- ``ce.vocab_ce_backward``: grad_scale * (softmax(z) - onehot(t)) (course
  notes §3.6.4).
- ``embedding.vocab_embedding``: out[n] = E[ids[n]] (textbook §4.2.3, course
  notes §3.4 "TP for Embedding").
- ``sharded``: the per-shard algorithm (column shard -> local activation ->
  row shard partial -> sum), used ONLY to pin the claim that sharding leaves
  the result unchanged. The unsharded functions above are the oracle.

Pins (tests/test_oracle.py, run with ``-m "not gpu"``): the pages' 2->4->2
worked example, a hand-derived backward of the same example, the pages'
column-backward dX example, shard-sum invariance (bit-exact on integer
inputs), bias-once versus the x T mistake, the row-first negative example,
central finite differences for every gradient, torch autograd in float64 for
the backward, torch's tanh-GELU for the activation, and closed forms /
torch.logsumexp for the cross-entropy. Every function here has at least one
pin; none is "parity unpinned".
"""

from . import mlp, ce, sharded, embedding  # noqa: F401
