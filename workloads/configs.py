"""Workload shapes, written out from the pages' own examples.

Notation (page "一层 MLP 太宽而放不下时怎样切？", §01-§02): N = B*L tokens,
D model width, F hidden (ffn) width, T tensor-parallel shards, F_s = F/T.

Shapes:
- tiny fp32 ReLU block (N=64, D=256, F=1024, T=2), the small case used for
  exhaustive parity;
- D=4096, F=16384, T=4: the 8-way exercise shape of the same page (§14)
  run at T=4, B=4, L=1024;
- D=8192, F=28672, T=8: the Llama-3-70B FFN matrix quoted on the Megatron
  TP chapter (§7.1), B=4, L=2048, forward and backward;
- N=16, D=12288, F=49152, T=8: the 12288->49152 MLP of the textbook page
  (§4.1.3) at decode-like token counts (weight streaming);
- vocab-parallel cross-entropy over V=128000 (the Llama-3 vocab of the
  Megatron TP chapter, §7.8), T=8 contiguous shards.
"""

from dataclasses import dataclass


@dataclass(frozen=True)
class MLPConfig:
    name: str
    B: int
    L: int
    D: int
    F: int
    T: int
    dtype: str          # "f32" or "bf16": storage type of X, W, b, H, Z, Y, grads
    act: str            # "relu", "gelu_tanh", "gelu_erf" or "gelu_sigmoid"
    bias: bool
    backward: bool
    x_std: float
    w_init: str         # "fan_in": std 1/sqrt(fan_in); "normal002": std 0.02
    b_init: str         # "uniform01": U(-0.1, 0.1); "normal002": N(0, 0.02); "none"
    seed: int = 0

    @property
    def N(self) -> int:
        return self.B * self.L

    @property
    def Fs(self) -> int:
        return self.F // self.T

    def fwd_flops(self) -> float:
        # two GEMMs of 2*N*D*F each
        return 4.0 * self.N * self.D * self.F

    def bwd_flops(self) -> float:
        # dH, dW2, dW1, dX: four GEMMs of 2*N*D*F each
        return 8.0 * self.N * self.D * self.F


@dataclass(frozen=True)
class CEConfig:
    name: str
    N: int
    V: int
    T: int
    logit_std: float
    seed: int = 0

    @property
    def Vs(self) -> int:
        return self.V // self.T

    def algorithmic_bytes(self) -> float:
        # logits read once, int64 targets read once, fp32 loss + int32 argmax
        # + int32 owner written once
        return 4.0 * self.N * self.V + 8.0 * self.N + 12.0 * self.N + 4.0


MLP_CONFIGS = {
    "mlp_f32_relu_n64_d256_f1024_t2": MLPConfig(
        name="mlp_f32_relu_n64_d256_f1024_t2", B=2, L=32, D=256, F=1024, T=2,
        dtype="f32", act="relu", bias=True, backward=False, x_std=1.0,
        w_init="fan_in", b_init="uniform01"),
    "mlp_bf16_gelu_n4096_d4096_f16384_t4": MLPConfig(
        name="mlp_bf16_gelu_n4096_d4096_f16384_t4", B=4, L=1024, D=4096, F=16384, T=4,
        dtype="bf16", act="gelu_tanh", bias=True, backward=False, x_std=1.0,
        w_init="normal002", b_init="normal002"),
    "mlp_bf16_gelu_n8192_d8192_f28672_t8_fwdbwd": MLPConfig(
        name="mlp_bf16_gelu_n8192_d8192_f28672_t8_fwdbwd", B=4, L=2048, D=8192, F=28672, T=8,
        dtype="bf16", act="gelu_tanh", bias=False, backward=True, x_std=1.0,
        w_init="normal002", b_init="none"),
    "mlp_bf16_gelu_n16_d12288_f49152_t8": MLPConfig(
        name="mlp_bf16_gelu_n16_d12288_f49152_t8", B=1, L=16, D=12288, F=49152, T=8,
        dtype="bf16", act="gelu_tanh", bias=True, backward=False, x_std=1.0,
        w_init="normal002", b_init="normal002"),
}

CE_CONFIGS = {
    "vocab_ce_n8192_v128000_t8": CEConfig(
        name="vocab_ce_n8192_v128000_t8", N=8192, V=128000, T=8, logit_std=2.0),
}


def config_by_name(name: str):
    if name in MLP_CONFIGS:
        return MLP_CONFIGS[name]
    if name in CE_CONFIGS:
        return CE_CONFIGS[name]
    raise KeyError(name)
