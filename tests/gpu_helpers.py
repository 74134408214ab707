"""Runs the CUDA path (through the C-ABI binding) on seeded inputs, for the
parity tests. Test glue only: it moves tensors to the GPU and concatenates
shard outputs for comparison with the unsharded oracle."""

import torch

import tensor_transformer_mlp_columnparallel_gb300 as tp


def dev():
    return torch.device("cuda:0")


def to_gpu(inp):
    d = dev()
    g = {
        "X": inp.X.to(d),
        "W1": [w.to(d) for w in inp.W1_shards()],
        "W2": [w.contiguous().to(d) for w in inp.W2_shards()],
        "b1": None if inp.b1 is None else [b.contiguous().to(d) for b in inp.b1_shards()],
        "b2": None if inp.b2 is None else inp.b2.to(d),
        "dY": None if inp.dY is None else inp.dY.to(d),
    }
    return g


def run_forward(g, act, mode, save_z=True):
    return tp.mlp_forward(g["X"], g["W1"], g["W2"], g["b1"], g["b2"], act=act, mode=mode,
                          save_z=save_z)


def run_backward(g, H, Z, act, mode, bias_grads):
    return tp.mlp_backward(g["X"], g["W1"], g["W2"], H, Z, g["dY"], act=act, mode=mode,
                           bias_grads=bias_grads)


def cat_cols(ts):
    return torch.cat([t.float() for t in ts], dim=1)


def cat_rows(ts):
    return torch.cat([t.float() for t in ts], dim=0)
