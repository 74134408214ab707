// Elementwise activations of the block and their derivatives (device side).
// ReLU: act'(0) = 0. GELU, tanh form (Hendrycks & Gimpel 2016):
//   act(z)  = 0.5 z (1 + tanh(u)),  u = sqrt(2/pi) (z + 0.044715 z^3)
//   act'(z) = 0.5 (1 + tanh(u)) + 0.5 z (1 - tanh(u)^2) sqrt(2/pi) (1 + 3 * 0.044715 z^2)
// tanh comes from CUDA's tanhf on the fp32 path; the bf16 tensor-core
// epilogue uses the equivalent sigmoid forms below.
#pragma once
#include <cuda_bf16.h>

#include "tpmlp.h"

namespace tpmlp {

// Exact GELU (the pages' nn.GELU): z Phi(z), Phi(z) = (1 + erf(z / sqrt(2))) / 2,
// derivative Phi(z) + z phi(z), phi(z) = exp(-z^2 / 2) / sqrt(2 pi); erf and
// exp from CUDA's erff / expf (fp32 path) or erff / __expf (bf16 epilogue).
__device__ __forceinline__ float gelu_erf_fwd(float z) {
    return 0.5f * z * (1.f + erff(z * 0.7071067811865476f));
}

// Sigmoid approximation of GELU (interview page): z s, s = sigmoid(1.702 z),
// derivative s (1 + 1.702 z (1 - s)) = s (1 + 1.702 z e s), e = exp(-1.702 z);
// exponent clamped at 80 as in the forms below.
constexpr float GELU_SIGMOID_SCALE = 1.702f;

__device__ __forceinline__ float act_fwd(int act, float z) {
    if (act == TPMLP_ACT_RELU) return z > 0.f ? z : 0.f;
    if (act == TPMLP_ACT_GELU_ERF) return gelu_erf_fwd(z);
    if (act == TPMLP_ACT_GELU_SIGMOID) return z / (1.f + expf(fminf(-GELU_SIGMOID_SCALE * z, 80.f)));
    const float c = 0.7978845608028654f;   // sqrt(2/pi)
    const float u = c * fmaf(0.044715f * z, z * z, z);
    return 0.5f * z * (1.f + tanhf(u));
}

__device__ __forceinline__ float act_grad(int act, float z) {
    if (act == TPMLP_ACT_RELU) return z > 0.f ? 1.f : 0.f;
    if (act == TPMLP_ACT_GELU_ERF)
        return fmaf(z * 0.3989422804014327f, expf(-0.5f * z * z), 0.5f * (1.f + erff(z * 0.7071067811865476f)));
    if (act == TPMLP_ACT_GELU_SIGMOID) {
        const float e = expf(fminf(-GELU_SIGMOID_SCALE * z, 80.f));
        const float sg = 1.f / (1.f + e);
        return sg * fmaf(GELU_SIGMOID_SCALE * z * e, sg, 1.f);
    }
    const float c = 0.7978845608028654f;
    const float z2 = z * z;
    const float t = tanhf(c * fmaf(0.044715f * z, z2, z));
    const float du = c * fmaf(3.f * 0.044715f, z2, 1.f);
    return fmaf(0.5f * z * (1.f - t * t), du, 0.5f * (1.f + t));
}

// SiLU(z) = z / (1 + exp(-z)), the gate nonlinearity of the gated MLP.
__device__ __forceinline__ float silu_f(float z) { return z / (1.f + expf(-z)); }

// Forms for the tensor-core epilogue, whose outputs are rounded to bf16
// (relative step 2^-8). They cut the epilogue's instruction count, which
// matters because the epilogue warps share issue slots with the TMA and MMA
// threads, and stay relatively accurate in both tails:
//   0.5 z (1 + tanh(u)) = z s,            s = sigmoid(2u) = 1 / (1 + e), e = exp(-2u)
//   act'(z) = s + 2 z s (1 - s) u'(z) = s (1 + 2 z u'(z) e s)     (1 - s = e s)
//   SiLU(z) = z / (1 + exp(-z))
// with CUDA's __expf and __fdividef. The exponent is clamped at 80 so that
// e, 1 + e and e s stay finite (for 2u < -80 the outputs are below 1e-33 in
// magnitude either way). The fp32 path keeps the tanhf / expf forms above.
__device__ __forceinline__ float act_fwd_bf16(int act, float z) {
    if (act == TPMLP_ACT_RELU) return z > 0.f ? z : 0.f;
    if (act == TPMLP_ACT_GELU_ERF) return gelu_erf_fwd(z);
    if (act == TPMLP_ACT_GELU_SIGMOID) return __fdividef(z, 1.f + __expf(fminf(-GELU_SIGMOID_SCALE * z, 80.f)));
    const float c = 0.7978845608028654f;
    const float u = c * fmaf(0.044715f * z, z * z, z);
    const float e = __expf(fminf(-2.f * u, 80.f));
    return __fdividef(z, 1.f + e);
}

__device__ __forceinline__ float act_grad_bf16(int act, float z) {
    if (act == TPMLP_ACT_RELU) return z > 0.f ? 1.f : 0.f;
    if (act == TPMLP_ACT_GELU_ERF)
        return fmaf(z * 0.3989422804014327f, __expf(-0.5f * z * z), 0.5f * (1.f + erff(z * 0.7071067811865476f)));
    if (act == TPMLP_ACT_GELU_SIGMOID) {
        const float e = __expf(fminf(-GELU_SIGMOID_SCALE * z, 80.f));
        const float sg = __fdividef(1.f, 1.f + e);
        return sg * fmaf(GELU_SIGMOID_SCALE * z * e, sg, 1.f);
    }
    const float c = 0.7978845608028654f;
    const float z2 = z * z;
    const float u = c * fmaf(0.044715f * z, z2, z);
    const float du = c * fmaf(3.f * 0.044715f, z2, 1.f);
    const float e = __expf(fminf(-2.f * u, 80.f));
    const float s = __fdividef(1.f, 1.f + e);
    return s * fmaf(2.f * z * du, e * s, 1.f);
}

__device__ __forceinline__ float silu_bf16(float z) {
    return __fdividef(z, 1.f + __expf(fminf(-z, 80.f)));
}

__device__ __forceinline__ float bf2f(__nv_bfloat16 v) { return __bfloat162float(v); }

__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
}

__device__ __forceinline__ void unpack_bf16x2(uint32_t w, float& a, float& b) {
    __nv_bfloat162 h = *reinterpret_cast<__nv_bfloat162*>(&w);
    a = __low2float(h);
    b = __high2float(h);
}

}  // namespace tpmlp
