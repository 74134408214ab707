"""Seeded input generators.

Weights are drawn as ONE full matrix and then sliced into shards, so that the
global function does not depend on T (page "一层 MLP 太宽而放不下时怎样切？",
§09: slicing a fixed full weight beats per-shard seeds, because local shapes
change the order in which random numbers are consumed).

Every tensor gets its own generator, seeded from (config seed, tensor index),
so one tensor's values never depend on another tensor's size. Values are
drawn in float32 and then stored in the workload's dtype (bf16 rounding is
round-to-nearest-even, done by torch). The oracle receives exactly the stored
values, promoted to float64.

Nothing here computes any part of the MLP or the loss.
"""

from dataclasses import dataclass, field
from typing import List, Optional

import torch

from .configs import MLPConfig, CEConfig

_TENSOR_INDEX = {"X": 0, "W1": 1, "b1": 2, "W2": 3, "b2": 4, "dY": 5,
                 "logits": 6, "targets": 7}


def _gen(seed: int, name: str) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed) * 1000003 + _TENSOR_INDEX[name])
    return g


def _storage(dtype: str) -> torch.dtype:
    if dtype == "f32":
        return torch.float32
    if dtype == "bf16":
        return torch.bfloat16
    raise ValueError(dtype)


@dataclass
class MLPInputs:
    """One block's inputs. W1 is [D, F] and W2 is [F, D] (math orientation:
    Y = act(X W1 + b1) W2 + b2). Shard r owns W1[:, r*Fs:(r+1)*Fs],
    b1[r*Fs:(r+1)*Fs] and W2[r*Fs:(r+1)*Fs, :]."""
    X: torch.Tensor                     # [N, D]
    W1: torch.Tensor                    # [D, F]
    W2: torch.Tensor                    # [F, D]
    b1: Optional[torch.Tensor]          # [F] or None
    b2: Optional[torch.Tensor]          # [D] or None
    dY: Optional[torch.Tensor]          # [N, D] or None
    T: int
    act: str
    dtype: str
    _w1_shards: List[torch.Tensor] = field(default_factory=list, repr=False)

    @property
    def N(self) -> int:
        return self.X.shape[0]

    @property
    def D(self) -> int:
        return self.X.shape[1]

    @property
    def F(self) -> int:
        return self.W1.shape[1]

    @property
    def Fs(self) -> int:
        return self.F // self.T

    def W1_shards(self) -> List[torch.Tensor]:
        """Contiguous [D, Fs] column blocks of W1 (one buffer per shard)."""
        if not self._w1_shards:
            self._w1_shards = [self.W1[:, r * self.Fs:(r + 1) * self.Fs].contiguous()
                               for r in range(self.T)]
        return self._w1_shards

    def W2_shards(self) -> List[torch.Tensor]:
        """[Fs, D] row blocks of W2 (contiguous views)."""
        return [self.W2[r * self.Fs:(r + 1) * self.Fs, :] for r in range(self.T)]

    def b1_shards(self) -> Optional[List[torch.Tensor]]:
        if self.b1 is None:
            return None
        return [self.b1[r * self.Fs:(r + 1) * self.Fs] for r in range(self.T)]


def _normal(shape, std, seed, name, dtype):
    g = _gen(seed, name)
    t = torch.empty(shape, dtype=torch.float32)
    t.normal_(0.0, float(std), generator=g)
    return t.to(_storage(dtype))


def _uniform(shape, lo, hi, seed, name, dtype):
    g = _gen(seed, name)
    t = torch.empty(shape, dtype=torch.float32)
    t.uniform_(float(lo), float(hi), generator=g)
    return t.to(_storage(dtype))


def _weight(shape, fan_in, cfg, name):
    if cfg.w_init == "fan_in":
        std = 1.0 / (fan_in ** 0.5)
    elif cfg.w_init == "normal002":
        std = 0.02
    else:
        raise ValueError(cfg.w_init)
    return _normal(shape, std, cfg.seed, name, cfg.dtype)


def _bias(n, cfg, name):
    if not cfg.bias or cfg.b_init == "none":
        return None
    if cfg.b_init == "uniform01":
        return _uniform((n,), -0.1, 0.1, cfg.seed, name, cfg.dtype)
    if cfg.b_init == "normal002":
        return _normal((n,), 0.02, cfg.seed, name, cfg.dtype)
    raise ValueError(cfg.b_init)


def gen_mlp_inputs(cfg: MLPConfig, N: Optional[int] = None, with_dy: Optional[bool] = None,
                   T: Optional[int] = None) -> MLPInputs:
    """Inputs of an MLP workload. `N` overrides the token count (rows of X and
    dY are drawn from the same stream, so a smaller N gives the leading rows of
    the full-size X); `T` overrides the shard count (weights do not change)."""
    N = cfg.N if N is None else int(N)
    T = cfg.T if T is None else int(T)
    with_dy = cfg.backward if with_dy is None else with_dy
    D, F = cfg.D, cfg.F
    if F % T != 0:
        raise ValueError(f"F={F} is not divisible by T={T}")
    X = _normal((N, D), cfg.x_std, cfg.seed, "X", cfg.dtype)
    W1 = _weight((D, F), D, cfg, "W1")
    b1 = _bias(F, cfg, "b1")
    W2 = _weight((F, D), F, cfg, "W2")
    b2 = _bias(D, cfg, "b2")
    dY = _normal((N, D), 1.0, cfg.seed, "dY", cfg.dtype) if with_dy else None
    return MLPInputs(X=X, W1=W1, W2=W2, b1=b1, b2=b2, dY=dY, T=T, act=cfg.act, dtype=cfg.dtype)


def gen_random_mlp(N: int, D: int, F: int, T: int, dtype: str, act: str, bias: bool,
                   seed: int, with_dy: bool = True, w_std: Optional[float] = None) -> MLPInputs:
    """Free-shape variant for ragged and edge-case tests (same recipe as the
    named workloads: X, dY ~ N(0,1); W ~ N(0, 1/sqrt(fan_in)) unless `w_std`;
    b ~ U(-0.1, 0.1))."""
    cfg = MLPConfig(name="adhoc", B=1, L=N, D=D, F=F, T=T, dtype=dtype, act=act, bias=bias,
                    backward=with_dy, x_std=1.0, w_init="fan_in",
                    b_init="uniform01" if bias else "none", seed=seed)
    if w_std is None:
        return gen_mlp_inputs(cfg)
    X = _normal((N, D), 1.0, seed, "X", dtype)
    W1 = _normal((D, F), w_std, seed, "W1", dtype)
    W2 = _normal((F, D), w_std, seed, "W2", dtype)
    b1 = _uniform((F,), -0.1, 0.1, seed, "b1", dtype) if bias else None
    b2 = _uniform((D,), -0.1, 0.1, seed, "b2", dtype) if bias else None
    dY = _normal((N, D), 1.0, seed, "dY", dtype) if with_dy else None
    return MLPInputs(X=X, W1=W1, W2=W2, b1=b1, b2=b2, dY=dY, T=T, act=act, dtype=dtype)


def gen_integer_mlp(N: int, D: int, F: int, T: int, dtype: str, bias: bool, seed: int,
                    with_dy: bool = True) -> MLPInputs:
    """Entries drawn from {-1, 0, 1} (biases from {-2..2}): every partial sum
    is a small integer, exactly representable in fp32 and bf16 while |value|
    stays below 256, so sharded and unsharded results can be compared
    bit-for-bit under ReLU."""
    def ints(shape, name, lo, hi):
        g = _gen(seed, name)
        return torch.randint(lo, hi + 1, shape, generator=g).to(_storage(dtype))
    X = ints((N, D), "X", -1, 1)
    W1 = ints((D, F), "W1", -1, 1)
    W2 = ints((F, D), "W2", -1, 1)
    b1 = ints((F,), "b1", -2, 2) if bias else None
    b2 = ints((D,), "b2", -2, 2) if bias else None
    dY = ints((N, D), "dY", -1, 1) if with_dy else None
    return MLPInputs(X=X, W1=W1, W2=W2, b1=b1, b2=b2, dY=dY, T=T, act="relu", dtype=dtype)


def gen_sparse_integer_mlp(N: int, D: int, F: int, T: int, dtype: str, seed: int,
                           density=(0.1, 0.02, 0.02, 0.04), bias: bool = False,
                           with_dy: bool = True) -> MLPInputs:
    """Sparse entries in {-1, 0, 1}: each entry of X, W1, W2 and dY (in that
    order of `density`) is non-zero with the given probability, with sign +1
    or -1 equally likely; biases, if any, from {-2..2}. At long reduction
    lengths (thousands) the sparsity keeps every sum a small integer, so
    sharded and unsharded results stay comparable bit for bit while most
    outputs are non-zero. The caller checks the magnitudes it relies on."""
    pX, pW1, pW2, pdY = density

    def sparse(shape, name, p):
        g = _gen(seed, name)
        keep = torch.rand(shape, generator=g) < p
        sign = torch.randint(0, 2, shape, generator=g) * 2 - 1
        return (keep.to(torch.int64) * sign).to(_storage(dtype))

    def ints(shape, name, lo, hi):
        return torch.randint(lo, hi + 1, shape, generator=_gen(seed, name)).to(_storage(dtype))
    X = sparse((N, D), "X", pX)
    W1 = sparse((D, F), "W1", pW1)
    W2 = sparse((F, D), "W2", pW2)
    b1 = ints((F,), "b1", -2, 2) if bias else None
    b2 = ints((D,), "b2", -2, 2) if bias else None
    dY = sparse((N, D), "dY", pdY) if with_dy else None
    return MLPInputs(X=X, W1=W1, W2=W2, b1=b1, b2=b2, dY=dY, T=T, act="relu", dtype=dtype)


@dataclass
class CEInputs:
    logits: torch.Tensor    # [N, V] float32
    targets: torch.Tensor   # [N] int64 in [0, V)
    T: int

    @property
    def N(self) -> int:
        return self.logits.shape[0]

    @property
    def V(self) -> int:
        return self.logits.shape[1]


def gen_ce_inputs(cfg: CEConfig, N: Optional[int] = None, V: Optional[int] = None,
                  T: Optional[int] = None) -> CEInputs:
    N = cfg.N if N is None else int(N)
    V = cfg.V if V is None else int(V)
    T = cfg.T if T is None else int(T)
    logits = torch.empty((N, V), dtype=torch.float32)
    logits.normal_(0.0, float(cfg.logit_std), generator=_gen(cfg.seed, "logits"))
    targets = torch.randint(0, V, (N,), generator=_gen(cfg.seed, "targets"), dtype=torch.int64)
    return CEInputs(logits=logits, targets=targets, T=T)
