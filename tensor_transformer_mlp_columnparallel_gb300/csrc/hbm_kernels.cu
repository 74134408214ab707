// HBM-bound kernels of the block and of the vocab-parallel cross-entropy.
//
// block_reduce: Y = sum_{r=0}^{T-1} P^(r) + b2 over T full-shape fp32 partial
//   sums (the single-GPU form of the block-end all-reduce SUM and of the
//   "bias once" rule, page "一层 MLP 太宽而放不下时怎样切？", §04-§05). 128-bit
//   streaming loads, 8 outputs per thread per step, shards summed in order
//   r = 0..T-1 in fp32, then b2, then one rounding to the output type.
// colsum: bias gradients db1^(r) = sum_n dZ^(r)[n, :], db2 = sum_n dY[n, :].
// vocab_ce: one CTA per token row. For each vocab shard k (contiguous
//   columns [k V/T, (k+1) V/T)) every thread keeps an online (max, sum of
//   exp) pair and the index of its first maximum; warp shuffles and a
//   shared-memory pass give the shard's (m_k, s_k, argmax_k); the shards are
//   then combined as m = max_k m_k, S = sum_k s_k exp(m_k - m), and the loss
//   is m + ln S - z[t] (page "unpurerationalist ... 3.4 TP for Embedding",
//   LM-head bullets; Megatron TP chapter §7.8). One pass over the logits.
#include <cuda_bf16.h>

#include <atomic>
#include <cmath>

#include "act.cuh"
#include "ptx.cuh"
#include "tpmlp_internal.h"

namespace tpmlp {
namespace {

// ---------------------------------------------------------------- reduce --

struct ReduceParams {
    const float* P[kMaxG];
    int T;
    int64_t N, D;
    const void* bias;
    void* Y;
    void* Yr[kMaxG];      // reduce-scatter: row block i of Y goes to Yr[i]
    int64_t rows_per;     // rows per block (0: plain reduce into Y)
};

// Destination element offset (in elements of OutT) of flat output index e.
template <typename OutT>
__device__ __forceinline__ OutT* reduce_dst(const ReduceParams& p, int64_t e) {
    if (p.rows_per == 0) return static_cast<OutT*>(p.Y) + e;
    const int64_t row = e / p.D;
    const int64_t blk = row / p.rows_per;
    return static_cast<OutT*>(p.Yr[blk]) + (e - blk * p.rows_per * p.D);
}

template <typename OutT>
__device__ __forceinline__ float load_out(const void* p, int64_t i) {
    if constexpr (sizeof(OutT) == 4) {
        return static_cast<const float*>(p)[i];
    } else {
        return __bfloat162float(static_cast<const __nv_bfloat16*>(p)[i]);
    }
}

template <typename OutT, int NT>
__global__ void __launch_bounds__(256) block_reduce_vec_kernel(const ReduceParams p) {
    // launched with programmatic stream serialization after the GEMM that
    // writes the partials: wait for it before the first load; the next
    // kernel (a GEMM) may do its set-up while this one streams
    pdl_launch_dependents();
    pdl_wait();
    const int64_t total8 = p.N * p.D / 8;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total8; i += stride) {
        float acc[8];
        {
            const float4* src = reinterpret_cast<const float4*>(p.P[0]) + 2 * i;
            const float4 a = __ldcs(src), b = __ldcs(src + 1);
            acc[0] = a.x; acc[1] = a.y; acc[2] = a.z; acc[3] = a.w;
            acc[4] = b.x; acc[5] = b.y; acc[6] = b.z; acc[7] = b.w;
        }
        constexpr int kLoop = NT > 0 ? NT : kMaxG;
#pragma unroll
        for (int r = 1; r < kLoop; ++r) {
            if (NT == 0 && r >= p.T) break;
            const float4* src = reinterpret_cast<const float4*>(p.P[r]) + 2 * i;
            const float4 a = __ldcs(src), b = __ldcs(src + 1);
            acc[0] += a.x; acc[1] += a.y; acc[2] += a.z; acc[3] += a.w;
            acc[4] += b.x; acc[5] += b.y; acc[6] += b.z; acc[7] += b.w;
        }
        if (p.bias != nullptr) {
            const int64_t col = (8 * i) % p.D;
            if constexpr (sizeof(OutT) == 4) {
                const float4* bb = reinterpret_cast<const float4*>(static_cast<const float*>(p.bias) + col);
                const float4 a = __ldg(bb), b = __ldg(bb + 1);
                acc[0] += a.x; acc[1] += a.y; acc[2] += a.z; acc[3] += a.w;
                acc[4] += b.x; acc[5] += b.y; acc[6] += b.z; acc[7] += b.w;
            } else {
                const uint4 w = __ldg(reinterpret_cast<const uint4*>(
                    static_cast<const __nv_bfloat16*>(p.bias) + col));
                const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                for (int h = 0; h < 4; ++h) {
                    float lo, hi;
                    unpack_bf16x2(ws[h], lo, hi);
                    acc[2 * h] += lo;
                    acc[2 * h + 1] += hi;
                }
            }
        }
        // D % 8 == 0 on this path, so the 8 outputs share one row (and one block)
        OutT* dst0 = reduce_dst<OutT>(p, 8 * i);
        if constexpr (sizeof(OutT) == 4) {
            float4* dst = reinterpret_cast<float4*>(dst0);
            __stcs(dst, make_float4(acc[0], acc[1], acc[2], acc[3]));
            __stcs(dst + 1, make_float4(acc[4], acc[5], acc[6], acc[7]));
        } else {
            uint4 w;
            w.x = pack_bf16x2(acc[0], acc[1]);
            w.y = pack_bf16x2(acc[2], acc[3]);
            w.z = pack_bf16x2(acc[4], acc[5]);
            w.w = pack_bf16x2(acc[6], acc[7]);
            __stcs(reinterpret_cast<uint4*>(dst0), w);
        }
    }
}

template <typename OutT>
__global__ void __launch_bounds__(256) block_reduce_scalar_kernel(const ReduceParams p) {
    pdl_launch_dependents();
    pdl_wait();
    const int64_t total = p.N * p.D;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += stride) {
        float acc = p.P[0][i];
        for (int r = 1; r < p.T; ++r) acc += p.P[r][i];
        if (p.bias != nullptr) acc += load_out<OutT>(p.bias, i % p.D);
        if constexpr (sizeof(OutT) == 4) {
            *reduce_dst<float>(p, i) = acc;
        } else {
            *reduce_dst<__nv_bfloat16>(p, i) = __float2bfloat16_rn(acc);
        }
    }
}

template <typename OutT>
cudaError_t launch_reduce(const ReduceParams& kp, bool vec, int grid, cudaStream_t s) {
    // programmatic dependent launch: the reduce may start its CTAs while the
    // GEMM that writes the partials finishes; the kernel waits for it first
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = pdl_enabled() ? 1 : 0;
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(256);
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (!vec) return cudaLaunchKernelEx(&cfg, block_reduce_scalar_kernel<OutT>, kp);
    switch (kp.T) {
        case 1: return cudaLaunchKernelEx(&cfg, block_reduce_vec_kernel<OutT, 1>, kp);
        case 2: return cudaLaunchKernelEx(&cfg, block_reduce_vec_kernel<OutT, 2>, kp);
        case 4: return cudaLaunchKernelEx(&cfg, block_reduce_vec_kernel<OutT, 4>, kp);
        case 8: return cudaLaunchKernelEx(&cfg, block_reduce_vec_kernel<OutT, 8>, kp);
        default: return cudaLaunchKernelEx(&cfg, block_reduce_vec_kernel<OutT, 0>, kp);
    }
}

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// ---------------------------------------------------------------- colsum --

struct ColsumParams {
    const void* in[kMaxColsumG];
    void* out[kMaxColsumG];
    int64_t cols[kMaxColsumG], ld[kMaxColsumG];
    int64_t colbase[kMaxColsumG];   // two-pass form: the group's first column in the scratch rows
    int rng0[kMaxColsumG + 1];      // two-pass form: the group's first column range (grid x)
    int64_t rows, total_cols;
    int G, S;                       // two-pass form: row chunks (grid y)
    float* scratch;                 // two-pass form: S rows of total_cols partial sums
};

template <typename T>
__global__ void __launch_bounds__(256) colsum_kernel(const ColsumParams p) {
    __shared__ float red[8][33];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int g = blockIdx.y;
    const int64_t c = (int64_t)blockIdx.x * 32 + lane;
    const int64_t cols = p.cols[g], ld = p.ld[g];
    float s = 0.f;
    if (c < cols) {
        const T* in = static_cast<const T*>(p.in[g]);
        for (int64_t r = warp; r < p.rows; r += 8) {
            if constexpr (sizeof(T) == 4)
                s += in[r * ld + c];
            else
                s += __bfloat162float(in[r * ld + c]);
        }
    }
    red[warp][lane] = s;
    __syncthreads();
    if (warp == 0 && c < cols) {
        float t = 0.f;
#pragma unroll
        for (int w = 0; w < 8; ++w) t += red[w][lane];
        if constexpr (sizeof(T) == 4)
            static_cast<float*>(p.out[g])[c] = t;
        else
            static_cast<__nv_bfloat16*>(p.out[g])[c] = __float2bfloat16_rn(t);
    }
}

// Single-pass form for 16-byte aligned rows (the bf16 path without scratch
// space, fp32 when the columns and pitch allow): each CTA owns a strip of
// CS_COLS columns of one group (grid x: strip, y: group) and all its rows. A
// lane reads one 16-byte vector (VEC columns) of a row, the lanes of a warp
// cover RPW rows at once, the 8 warps PHASES rows, and each thread keeps
// UNROLL such loads in flight before adding them: 8 when the strips fill the
// GPU twice over, else 16 (dY's), so that the resident CTAs keep more bytes
// moving. (Splitting rows across a CTA cluster instead measured slower.)
// Every column's sum is formed in a fixed order (each thread's rows in
// increasing order, then the row phases in turn), so results do not depend
// on timing.
constexpr int CS_THREADS = 256;
constexpr int CS_COLS = 32;      // columns per strip

template <typename T, int UNROLL>
__global__ void __launch_bounds__(CS_THREADS) colsum_vec_kernel(const ColsumParams p) {
    constexpr int VEC = 16 / (int)sizeof(T);         // columns per 16-byte vector
    constexpr int LPR = CS_COLS / VEC;               // lanes per row
    constexpr int RPW = 32 / LPR;                    // rows per warp load
    constexpr int PHASES = (CS_THREADS / 32) * RPW;  // rows covered by one load of every thread
    __shared__ float part[PHASES][CS_COLS + 1];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int slot = lane % LPR;                     // which vector of the strip
    const int phase = warp * RPW + lane / LPR;       // this thread's first row
    const int g = blockIdx.y;
    const int strip = blockIdx.x;
    const int64_t cols = p.cols[g], ld = p.ld[g];
    const int64_t c0 = (int64_t)strip * CS_COLS + slot * VEC;
    float acc[VEC];
#pragma unroll
    for (int v = 0; v < VEC; ++v) acc[v] = 0.f;
    if (c0 < cols) {
        const T* in = static_cast<const T*>(p.in[g]) + c0;
        for (int64_t base = phase; base < p.rows; base += (int64_t)PHASES * UNROLL) {
            uint4 w[UNROLL];
#pragma unroll
            for (int u = 0; u < UNROLL; ++u) {
                const int64_t r = base + (int64_t)u * PHASES;
                w[u] = r < p.rows ? __ldcs(reinterpret_cast<const uint4*>(in + r * ld))
                                  : make_uint4(0u, 0u, 0u, 0u);
            }
#pragma unroll
            for (int u = 0; u < UNROLL; ++u) {
                if constexpr (sizeof(T) == 4) {
                    acc[0] += __uint_as_float(w[u].x);
                    acc[1] += __uint_as_float(w[u].y);
                    acc[2] += __uint_as_float(w[u].z);
                    acc[3] += __uint_as_float(w[u].w);
                } else {
                    const uint32_t ws[4] = {w[u].x, w[u].y, w[u].z, w[u].w};
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        acc[2 * q] += __uint_as_float(ws[q] << 16);
                        acc[2 * q + 1] += __uint_as_float(ws[q] & 0xffff0000u);
                    }
                }
            }
        }
    }
#pragma unroll
    for (int v = 0; v < VEC; ++v) part[phase][slot * VEC + v] = acc[v];
    __syncthreads();
    if (threadIdx.x < CS_COLS) {
        const int64_t c = (int64_t)strip * CS_COLS + threadIdx.x;
        if (c < cols) {
            float t = 0.f;
            for (int ph = 0; ph < PHASES; ++ph) t += part[ph][threadIdx.x];
            if constexpr (sizeof(T) == 4)
                static_cast<float*>(p.out[g])[c] = t;
            else
                static_cast<__nv_bfloat16*>(p.out[g])[c] = __float2bfloat16_rn(t);
        }
    }
}

// Two-pass form (bf16, with scratch space). Pass 1: CTA (x, y) sums row chunk
// y (a contiguous 1/S of the rows) of column range x, up to CP_COLS columns
// of one group: thread t owns the 16-byte vectors t and t + 256 of each row,
// so the CTA reads a contiguous stretch of up to 8 KB of every row (a dZ
// shard's whole row: one contiguous block over its rows), CP_UNROLL rows in
// flight; each thread writes its column sums to row y of the scratch.
// (Reading narrow strips down all rows instead, one 64-byte piece of every
// row per CTA, left DRAM at about 3 TB/s; this form reaches about 4.)
// Pass 2: one thread per column adds the S chunk sums in chunk order. Fixed
// order throughout, so results do not depend on timing.
constexpr int CP_THREADS = 256;
constexpr int CP_VPT = 2;                          // 16-byte vectors per thread and row
constexpr int CP_COLS = CP_THREADS * 8 * CP_VPT;   // bf16 columns per range
constexpr int CP_UNROLL = 2;

__global__ void __launch_bounds__(CP_THREADS) colsum_part_kernel(const ColsumParams p) {
    int g = 0;
    while (g + 1 < p.G && (int)blockIdx.x >= p.rng0[g + 1]) ++g;
    const int64_t c_start = (int64_t)((int)blockIdx.x - p.rng0[g]) * CP_COLS;
    const int64_t cols = p.cols[g], ld = p.ld[g];
    const int chunk = blockIdx.y;
    const int64_t r_lo = p.rows * chunk / p.S, r_hi = p.rows * (chunk + 1) / p.S;
    const __nv_bfloat16* in = static_cast<const __nv_bfloat16*>(p.in[g]);
    bool on[CP_VPT];
    int64_t c[CP_VPT];
#pragma unroll
    for (int k = 0; k < CP_VPT; ++k) {
        c[k] = c_start + (int64_t)(threadIdx.x + CP_THREADS * k) * 8;
        on[k] = c[k] < cols;
    }
    if (!on[0]) return;   // no barrier follows
    float acc[CP_VPT][8];
#pragma unroll
    for (int k = 0; k < CP_VPT; ++k)
#pragma unroll
        for (int v = 0; v < 8; ++v) acc[k][v] = 0.f;
    for (int64_t base = r_lo; base < r_hi; base += CP_UNROLL) {
        uint4 w[CP_UNROLL][CP_VPT];
#pragma unroll
        for (int u = 0; u < CP_UNROLL; ++u)
#pragma unroll
            for (int k = 0; k < CP_VPT; ++k) {
                const int64_t r = base + u;
                w[u][k] = (r < r_hi && on[k])
                              ? __ldcs(reinterpret_cast<const uint4*>(in + r * ld + c[k]))
                              : make_uint4(0u, 0u, 0u, 0u);
            }
#pragma unroll
        for (int u = 0; u < CP_UNROLL; ++u)
#pragma unroll
            for (int k = 0; k < CP_VPT; ++k) {
                const uint32_t ws[4] = {w[u][k].x, w[u][k].y, w[u][k].z, w[u][k].w};
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    acc[k][2 * q] += __uint_as_float(ws[q] << 16);
                    acc[k][2 * q + 1] += __uint_as_float(ws[q] & 0xffff0000u);
                }
            }
    }
#pragma unroll
    for (int k = 0; k < CP_VPT; ++k) {
        if (!on[k]) continue;
        float4* dst = reinterpret_cast<float4*>(p.scratch + chunk * p.total_cols + p.colbase[g] + c[k]);
        dst[0] = make_float4(acc[k][0], acc[k][1], acc[k][2], acc[k][3]);
        dst[1] = make_float4(acc[k][4], acc[k][5], acc[k][6], acc[k][7]);
    }
}

__global__ void __launch_bounds__(256) colsum_final_kernel(const ColsumParams p) {
    const int64_t col = (int64_t)blockIdx.x * 256 + threadIdx.x;
    if (col >= p.total_cols) return;
    int g = 0;
    while (g + 1 < p.G && col >= p.colbase[g + 1]) ++g;
    float t = 0.f;
    for (int chunk = 0; chunk < p.S; ++chunk) t += p.scratch[chunk * p.total_cols + col];
    static_cast<__nv_bfloat16*>(p.out[g])[col - p.colbase[g]] = __float2bfloat16_rn(t);
}

// -------------------------------------------------------------- vocab CE --

constexpr int CE_THREADS = 256;
constexpr int CE_WARPS = CE_THREADS / 32;
constexpr int CE_MAX_UNITS = 16;     // max over T <= 16 of T * ceil(CE_WARPS / T)
constexpr int CE_UNROLL = 8;         // independent 16-byte loads in flight per lane
constexpr float LOG2E = 1.4426950408889634f;

struct CEParams {
    const float* logits;
    const int64_t* targets;
    float* loss;
    int32_t* argmax;
    int32_t* owner;
    int64_t N, V, Vs;
    int T;
    int parts;       // each shard is cut into `parts` contiguous pieces, one per warp
    int vec;
    int* err;
};

// Online (max, sum exp(z - max), first argmax) state of one thread.
struct LseState {
    float m;
    float s;
    int64_t a;
};

__device__ __forceinline__ void lse_push(LseState& st, float x, int64_t idx) {
    if (x > st.m) {
        st.s = st.s * exp2f((st.m - x) * LOG2E) + 1.f;
        st.m = x;
        st.a = idx;
    } else {
        st.s += exp2f((x - st.m) * LOG2E);
    }
}

// Four consecutive elements idx..idx+3; the first of equal maxima wins.
__device__ __forceinline__ void lse_push4(LseState& st, float4 x, int64_t idx) {
    const float mx = fmaxf(fmaxf(x.x, x.y), fmaxf(x.z, x.w));
    if (mx > st.m) {
        st.s *= exp2f((st.m - mx) * LOG2E);
        st.m = mx;
        st.a = idx + (x.x == mx ? 0 : (x.y == mx ? 1 : (x.z == mx ? 2 : 3)));
    }
    const float mL = st.m * LOG2E;
    st.s += (exp2f(fmaf(x.x, LOG2E, -mL)) + exp2f(fmaf(x.y, LOG2E, -mL))) +
            (exp2f(fmaf(x.z, LOG2E, -mL)) + exp2f(fmaf(x.w, LOG2E, -mL)));
}

// Merge two states: the larger max wins; on equal maxima the lower index.
__device__ __forceinline__ void lse_merge(LseState& st, float m2, float s2, int64_t a2) {
    if (m2 == -INFINITY) return;
    if (st.m == -INFINITY) {
        st.m = m2; st.s = s2; st.a = a2;
        return;
    }
    const float M = fmaxf(st.m, m2);
    st.s = st.s * exp2f((st.m - M) * LOG2E) + s2 * exp2f((m2 - M) * LOG2E);
    if (m2 > st.m || (m2 == st.m && a2 < st.a)) st.a = a2;
    st.m = M;
}

// One CTA per token row. Unit u = (shard k = u / parts, piece u % parts) is a
// contiguous range of shard k; warp w streams units w, w + CE_WARPS, ... with
// coalesced 16-byte loads and reduces each unit with shuffles; one shared-
// memory pass then combines the pieces of each shard and the shards.
__global__ void __launch_bounds__(CE_THREADS) vocab_ce_kernel(const CEParams p) {
    __shared__ float sm_m[CE_MAX_UNITS];
    __shared__ float sm_s[CE_MAX_UNITS];
    __shared__ long long sm_a[CE_MAX_UNITS];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int64_t row = blockIdx.x;
    const float* z = p.logits + row * p.V;
    const int units = p.T * p.parts;

    for (int u = warp; u < units; u += CE_WARPS) {
        const int k = u / p.parts, piece = u - k * p.parts;
        LseState st{-INFINITY, 0.f, 0x7fffffffffffffffLL};
        const int64_t base = (int64_t)k * p.Vs;
        if (p.vec) {
            const int64_t n4 = p.Vs / 4;
            const int64_t lo = n4 * piece / p.parts, hi = n4 * (piece + 1) / p.parts;
            const float4* zv = reinterpret_cast<const float4*>(z + base);
            int64_t i = lo + lane;
            for (; i + 32 * (CE_UNROLL - 1) < hi; i += 32 * CE_UNROLL) {
                float4 x[CE_UNROLL];
#pragma unroll
                for (int j = 0; j < CE_UNROLL; ++j) x[j] = __ldcs(zv + i + 32 * j);
#pragma unroll
                for (int j = 0; j < CE_UNROLL; ++j) lse_push4(st, x[j], base + 4 * (i + 32 * j));
            }
            for (; i < hi; i += 32) lse_push4(st, __ldcs(zv + i), base + 4 * i);
        } else {
            const int64_t lo = p.Vs * piece / p.parts, hi = p.Vs * (piece + 1) / p.parts;
            for (int64_t i = lo + lane; i < hi; i += 32) lse_push(st, z[base + i], base + i);
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            const float m2 = __shfl_xor_sync(0xffffffffu, st.m, off);
            const float s2 = __shfl_xor_sync(0xffffffffu, st.s, off);
            const long long a2 = __shfl_xor_sync(0xffffffffu, (long long)st.a, off);
            lse_merge(st, m2, s2, a2);
        }
        if (lane == 0) {
            sm_m[u] = st.m;
            sm_s[u] = st.s;
            sm_a[u] = st.a;
        }
    }
    __syncthreads();
    if (warp != 0) return;
    // lane k < T: merge the pieces of shard k -> (m_k, s_k, argmax_k)
    LseState sh{-INFINITY, 0.f, 0x7fffffffffffffffLL};
    if (lane < p.T) {
        for (int q = 0; q < p.parts; ++q) {
            const int u = lane * p.parts + q;
            lse_merge(sh, sm_m[u], sm_s[u], sm_a[u]);
        }
    }
    // combine the shards: m = max_k m_k, S = sum_k s_k exp(m_k - m)
    float m = sh.m;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
    float term = (lane < p.T && sh.m != -INFINITY) ? sh.s * exp2f((sh.m - m) * LOG2E) : 0.f;
    // lowest index among shards whose max equals the global max
    long long a = (lane < p.T && sh.m == m) ? (long long)sh.a : 0x7fffffffffffffffLL;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        term += __shfl_xor_sync(0xffffffffu, term, off);
        const long long a2 = __shfl_xor_sync(0xffffffffu, a, off);
        a = a2 < a ? a2 : a;
    }
    if (lane == 0) {
        const int64_t t = p.targets[row];
        float loss;
        if (t < 0 || t >= p.V) {
            loss = __int_as_float(0x7fc00000);   // NaN
            atomicCAS(p.err, 0, (int)TPMLP_ERR_ARG);
            if (p.owner) p.owner[row] = -1;
        } else {
            const int64_t own = t / p.Vs;
            // the owning shard reads its local logit t - own * Vs
            const float zt = z[own * p.Vs + (t - own * p.Vs)];
            loss = m + logf(term) - zt;
            if (p.owner) p.owner[row] = (int32_t)own;
        }
        p.loss[row] = loss;
        if (p.argmax) p.argmax[row] = (int32_t)a;
    }
}

// CE backward: dz[n, v] = g * (exp(z[n, v] - lse_n) - 1(v = t_n)), computed by
// every vocab shard on its own columns from the forward's per-token result;
// lse_n = loss_n + z[n, t_n] recovers m_n + ln S_n from the forward's loss.
// One CTA per row; 16-byte streaming loads and stores; may run in place.
struct CEBwdParams {
    const float* logits;
    const int64_t* targets;
    const float* loss;
    float* dlogits;
    int64_t N, V;
    float scale;
    int vec;
    int* err;
};

__device__ __forceinline__ float ce_grad(float z, float lseL, float g, bool is_t) {
    return g * (exp2f(fmaf(z, LOG2E, -lseL)) - (is_t ? 1.f : 0.f));
}

__global__ void __launch_bounds__(256) vocab_ce_bwd_kernel(const CEBwdParams p) {
    __shared__ float s_lse;
    __shared__ long long s_t;
    const int64_t row = blockIdx.x;
    const float* z = p.logits + row * p.V;
    float* dz = p.dlogits + row * p.V;
    if (threadIdx.x == 0) {
        const int64_t t = p.targets[row];
        if (t < 0 || t >= p.V) {
            atomicCAS(p.err, 0, (int)TPMLP_ERR_ARG);
            s_lse = __int_as_float(0x7fc00000);
            s_t = -1;
        } else {
            s_lse = p.loss[row] + z[t];
            s_t = t;
        }
    }
    __syncthreads();   // z[t] is read before any thread overwrites the row
    const float lseL = s_lse * LOG2E;
    const int64_t t = s_t;
    const float g = p.scale;
    if (p.vec) {
        const float4* zv = reinterpret_cast<const float4*>(z);
        float4* dv = reinterpret_cast<float4*>(dz);
        const int64_t n4 = p.V / 4;
        int64_t i = threadIdx.x;
        for (; i + 3 * 256 < n4; i += 4 * 256) {
            float4 x[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) x[u] = __ldcs(zv + i + u * 256);
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int64_t e = 4 * (i + u * 256);
                float4 d;
                d.x = ce_grad(x[u].x, lseL, g, e == t);
                d.y = ce_grad(x[u].y, lseL, g, e + 1 == t);
                d.z = ce_grad(x[u].z, lseL, g, e + 2 == t);
                d.w = ce_grad(x[u].w, lseL, g, e + 3 == t);
                __stcs(dv + i + u * 256, d);
            }
        }
        for (; i < n4; i += 256) {
            const float4 x = __ldcs(zv + i);
            const int64_t e = 4 * i;
            float4 d;
            d.x = ce_grad(x.x, lseL, g, e == t);
            d.y = ce_grad(x.y, lseL, g, e + 1 == t);
            d.z = ce_grad(x.z, lseL, g, e + 2 == t);
            d.w = ce_grad(x.w, lseL, g, e + 3 == t);
            __stcs(dv + i, d);
        }
    } else {
        for (int64_t i = threadIdx.x; i < p.V; i += 256) dz[i] = ce_grad(z[i], lseL, g, i == t);
    }
}

// mean of the per-token losses, one CTA, fixed summation order, fp64 accumulator
__global__ void __launch_bounds__(1024) mean_kernel(const float* loss, int64_t N, float* out) {
    __shared__ double red[1024];
    double s = 0.0;
    for (int64_t i = threadIdx.x; i < N; i += 1024) s += (double)loss[i];
    red[threadIdx.x] = s;
    __syncthreads();
    for (int w = 512; w > 0; w >>= 1) {
        if ((int)threadIdx.x < w) red[threadIdx.x] += red[threadIdx.x + w];
        __syncthreads();
    }
    if (threadIdx.x == 0) *out = N > 0 ? (float)(red[0] / (double)N) : __int_as_float(0x7fc00000);
}

// ------------------------------------------------------ vocab embedding --
// Row-split table: shard k holds rows [k Vs, (k+1) Vs). Each shard would
// return its own row for ids in its range and zeros otherwise, and the sum
// over shards leaves exactly the owner's row; so every token's row is copied
// from the owning shard. One warp per token, 16-byte chunks.

struct EmbParams {
    const int64_t* ids;
    const void* table[kMaxG];
    void* out;
    int64_t N, V, Vs, row_bytes;
    int vec;
    int* err;
};

__global__ void __launch_bounds__(256) vocab_embedding_kernel(const EmbParams p) {
    const int lane = threadIdx.x & 31;
    const int64_t warp_global = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
    for (int64_t n = warp_global; n < p.N; n += nwarps) {
        const int64_t id = p.ids[n];
        char* dst = static_cast<char*>(p.out) + n * p.row_bytes;
        const bool valid = id >= 0 && id < p.V;
        if (!valid && lane == 0) atomicCAS(p.err, 0, (int)TPMLP_ERR_ARG);
        const int64_t k = valid ? id / p.Vs : 0;
        const char* src = valid ? static_cast<const char*>(p.table[k]) + (id - k * p.Vs) * p.row_bytes
                                : nullptr;
        if (p.vec) {
            const int64_t chunks = p.row_bytes / 16;
            const uint4* sv = reinterpret_cast<const uint4*>(src);
            uint4* dv = reinterpret_cast<uint4*>(dst);
            const uint4 zero = make_uint4(0, 0, 0, 0);
            int64_t c = lane;
            // four independent 16-byte loads in flight per lane
            for (; c + 96 < chunks; c += 128) {
                uint4 v[4];
#pragma unroll
                for (int u = 0; u < 4; ++u) v[u] = valid ? __ldg(sv + c + 32 * u) : zero;
#pragma unroll
                for (int u = 0; u < 4; ++u) __stcs(dv + c + 32 * u, v[u]);
            }
            for (; c < chunks; c += 32) __stcs(dv + c, valid ? __ldg(sv + c) : zero);
        } else {
            for (int64_t c = lane; c < p.row_bytes; c += 32) dst[c] = valid ? src[c] : 0;
        }
    }
}

// Bulk-copy form (16-byte aligned rows whose size is a multiple of 16 bytes):
// one thread per CTA streams row chunks global -> shared -> global with
// cp.async.bulk, EMB_BUFS chunks deep, so each SM keeps several 16 KB chunks
// in flight with almost no instructions issued. An id outside [0, V) gives a
// zero row (written with plain stores) and TPMLP_ERR_ARG.
constexpr int EMB_BUFS = 4;
constexpr int EMB_CHUNK = 16384;
constexpr int EMB_SMEM = EMB_BUFS * EMB_CHUNK;

__global__ void __launch_bounds__(32) vocab_embedding_bulk_kernel(const EmbParams p, uint64_t timeout_ns) {
    extern __shared__ __align__(128) uint8_t ebuf[];
    __shared__ __align__(8) uint64_t bars[EMB_BUFS];
    __shared__ int abort_flag;
    if (threadIdx.x != 0) return;
    for (int b = 0; b < EMB_BUFS; ++b) mbar_init(smem_u32(&bars[b]), 1);
    abort_flag = 0;
    fence_mbar_init();
    const int64_t cpr = (p.row_bytes + EMB_CHUNK - 1) / EMB_CHUNK;   // chunks per row
    const int64_t items = p.N * cpr;
    const int64_t first = blockIdx.x, step = gridDim.x;
    const int64_t count = items > first ? (items - 1 - first) / step + 1 : 0;
    // item j of this CTA: token n, chunk c; returns false for an invalid id
    auto locate = [&](int64_t j, const char*& src, char*& dst, uint32_t& bytes) -> bool {
        const int64_t it = first + j * step;
        const int64_t n = it / cpr, c = it - n * cpr;
        const int64_t off = c * EMB_CHUNK;
        const int64_t rem = p.row_bytes - off;
        bytes = (uint32_t)(rem < EMB_CHUNK ? rem : EMB_CHUNK);
        dst = static_cast<char*>(p.out) + n * p.row_bytes + off;
        const int64_t id = p.ids[n];
        if (id < 0 || id >= p.V) {
            src = nullptr;
            return false;
        }
        const int64_t k = id / p.Vs;
        src = static_cast<const char*>(p.table[k]) + (id - k * p.Vs) * p.row_bytes + off;
        return true;
    };
    auto issue = [&](int64_t j) {
        const uint32_t bar = smem_u32(&bars[j % EMB_BUFS]);
        const char* src;
        char* dst;
        uint32_t bytes;
        if (locate(j, src, dst, bytes)) {
            mbar_arrive_expect_tx(bar, bytes);
            bulk_load_g2s(smem_u32(ebuf) + (uint32_t)(j % EMB_BUFS) * EMB_CHUNK, src, bytes, bar);
        } else {
            mbar_arrive(bar);   // keeps the buffer's phase count in step
        }
    };
    int64_t issued = 0;
    for (; issued < count && issued < EMB_BUFS; ++issued) issue(issued);
    int64_t i = 0;
    for (; i < count; ++i) {
        const int b = (int)(i % EMB_BUFS);
        const uint32_t parity = (uint32_t)((i / EMB_BUFS) & 1);
        if (!wait_bounded(smem_u32(&bars[b]), parity, &abort_flag, p.err, timeout_ns, false)) break;
        const char* src;
        char* dst;
        uint32_t bytes;
        if (locate(i, src, dst, bytes)) {
            bulk_store_s2g(dst, smem_u32(ebuf) + (uint32_t)b * EMB_CHUNK, bytes);
            bulk_commit();
            bulk_wait_read_all();   // buffer b may be refilled once its store has read it
        } else {
            atomicCAS(p.err, 0, (int)TPMLP_ERR_ARG);
            for (uint32_t q = 0; q < bytes; q += 16)
                *reinterpret_cast<uint4*>(dst + q) = make_uint4(0, 0, 0, 0);
        }
        if (issued < count) issue(issued++);
    }
    // after a timeout: wait (bounded) for the loads still in flight
    for (; i < issued; ++i)
        wait_bounded(smem_u32(&bars[i % EMB_BUFS]), (uint32_t)((i / EMB_BUFS) & 1), &abort_flag, p.err,
                     timeout_ns, false);
    bulk_wait_all();
}

// ------------------------------------------------------------- self test --

__global__ void selftest_wait_kernel(int* err, uint64_t timeout_ns) {
    __shared__ __align__(8) uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&bar), 1);
        abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        // nothing arrives on this barrier: the bounded wait has to run out
        wait_bounded(smem_u32(&bar), 0, &abort_flag, err, timeout_ns, true);
    }
}

}  // namespace

tpmlp_status run_block_reduce(int out_f32, int64_t N, int64_t D, int T, const float* const* P,
                              const void* bias, void* Y, cudaStream_t s, const char* name,
                              void* const* Y_rows) {
    if (N == 0) return TPMLP_OK;
    ReduceParams kp{};
    bool vec = (D % 8 == 0) && (bias == nullptr || aligned16(bias));
    if (Y_rows != nullptr) {
        kp.rows_per = N / T;
        for (int r = 0; r < T; ++r) {
            kp.Yr[r] = Y_rows[r];
            vec = vec && aligned16(Y_rows[r]);
        }
    } else {
        vec = vec && aligned16(Y);
    }
    for (int r = 0; r < T; ++r) {
        kp.P[r] = P[r];
        vec = vec && aligned16(P[r]);
    }
    kp.T = T;
    kp.N = N;
    kp.D = D;
    kp.bias = bias;
    kp.Y = Y;
    const int64_t work = vec ? N * D / 8 : N * D;
    const int64_t max_grid = (int64_t)device_sm_count() * 8;
    int64_t grid = (work + 255) / 256;
    if (grid > max_grid) grid = max_grid;
    if (grid < 1) grid = 1;
    cudaError_t e;
    {
        LaunchScope ls(name, s);
        e = out_f32 ? launch_reduce<float>(kp, vec, (int)grid, s)
                    : launch_reduce<__nv_bfloat16>(kp, vec, (int)grid, s);
    }
    return e == cudaSuccess ? TPMLP_OK : TPMLP_ERR_CUDA;
}

tpmlp_status run_colsum(int f32, int64_t rows, int G, const int64_t* cols, const int64_t* ld,
                        const void* const* in, void* const* out, cudaStream_t s, float* scratch,
                        size_t scratch_bytes) {
    if (G <= 0) return TPMLP_OK;
    if (G > kMaxColsumG) return TPMLP_ERR_SHAPE;
    ColsumParams kp{};
    kp.rows = rows;
    kp.G = G;
    // the vector forms need every row's vectors 16-byte aligned
    const int vec = f32 ? 4 : 8;
    bool vec_ok = true;
    int64_t max_cols = 0, total = 0, ranges = 0;
    for (int g = 0; g < G; ++g) {
        kp.in[g] = in[g];
        kp.out[g] = out[g];
        kp.cols[g] = cols[g];
        kp.ld[g] = ld[g];
        kp.colbase[g] = total;
        kp.rng0[g] = (int)ranges;
        total += cols[g];
        ranges += (cols[g] + CP_COLS - 1) / CP_COLS;
        max_cols = cols[g] > max_cols ? cols[g] : max_cols;
        vec_ok = vec_ok && cols[g] % vec == 0 && ld[g] % vec == 0 && aligned16(in[g]);
    }
    kp.rng0[G] = (int)ranges;
    kp.total_cols = total;
    if (max_cols == 0) return TPMLP_OK;
    // two-pass form: row chunks for about 8 CTAs per SM in pass 1 (at most
    // 64 chunks, each at least 64 rows, the partials within the scratch). On
    // the fwd+bwd shape's sums (10 ranges) 64 chunks took 0.155 ms, 60 took
    // 0.165, 30 took 0.29; 1 to 4 rows in flight per thread were within 2%,
    // 8 or 16 took 0.29.
    int S = 0;
    if (!f32 && vec_ok && scratch != nullptr && aligned16(scratch) && rows >= 64 && ranges > 0) {
        int64_t sc = 8 * (int64_t)device_sm_count() / ranges;
        sc = sc < 1 ? 1 : (sc > 64 ? 64 : sc);
        if (sc > rows / 64) sc = rows / 64;
        while (sc > 0 && (size_t)sc * (size_t)total * sizeof(float) > scratch_bytes) --sc;
        S = (int)sc;
    }
    {
        LaunchScope ls("bias_grad_colsum", s);
        if (S >= 1) {
            kp.S = S;
            kp.scratch = scratch;
            colsum_part_kernel<<<dim3((unsigned)ranges, (unsigned)S), CP_THREADS, 0, s>>>(kp);
            colsum_final_kernel<<<(unsigned)((total + 255) / 256), 256, 0, s>>>(kp);
        } else if (vec_ok) {
            // deeper per-thread load queues when the strips are few (under
            // two per SM), so the resident CTAs still keep HBM busy
            const int64_t strips = (max_cols + CS_COLS - 1) / CS_COLS;
            const bool few = strips * G < 2 * (int64_t)device_sm_count();
            const dim3 grid((unsigned)strips, (unsigned)G);
            if (f32) {
                if (few)
                    colsum_vec_kernel<float, 16><<<grid, CS_THREADS, 0, s>>>(kp);
                else
                    colsum_vec_kernel<float, 8><<<grid, CS_THREADS, 0, s>>>(kp);
            } else {
                if (few)
                    colsum_vec_kernel<__nv_bfloat16, 16><<<grid, CS_THREADS, 0, s>>>(kp);
                else
                    colsum_vec_kernel<__nv_bfloat16, 8><<<grid, CS_THREADS, 0, s>>>(kp);
            }
        } else {
            dim3 grid((unsigned)((max_cols + 31) / 32), (unsigned)G);
            if (f32)
                colsum_kernel<float><<<grid, 256, 0, s>>>(kp);
            else
                colsum_kernel<__nv_bfloat16><<<grid, 256, 0, s>>>(kp);
        }
    }
    return cudaGetLastError() == cudaSuccess ? TPMLP_OK : TPMLP_ERR_CUDA;
}

tpmlp_status run_vocab_ce(int64_t N, int64_t V, int T, const float* logits,
                          const int64_t* targets, float* loss, float* loss_mean, int32_t* argmax,
                          int32_t* owner, cudaStream_t s) {
    if (N > 0) {
        CEParams kp{};
        kp.logits = logits;
        kp.targets = targets;
        kp.loss = loss;
        kp.argmax = argmax;
        kp.owner = owner;
        kp.N = N;
        kp.V = V;
        kp.Vs = V / T;
        kp.T = T;
        kp.parts = (CE_WARPS + T - 1) / T;
        kp.vec = (kp.Vs % 4 == 0) && aligned16(logits);
        kp.err = device_error_word();
        if (kp.err == nullptr) return TPMLP_ERR_CUDA;
        if (N > 0x7fffffffLL) return TPMLP_ERR_SHAPE;
        LaunchScope ls("vocab_ce_fwd", s);
        vocab_ce_kernel<<<(unsigned)N, CE_THREADS, 0, s>>>(kp);
    }
    if (cudaGetLastError() != cudaSuccess) return TPMLP_ERR_CUDA;
    if (loss_mean != nullptr) {
        LaunchScope ls("vocab_ce_mean", s);
        mean_kernel<<<1, 1024, 0, s>>>(loss, N, loss_mean);
    }
    return cudaGetLastError() == cudaSuccess ? TPMLP_OK : TPMLP_ERR_CUDA;
}

tpmlp_status run_vocab_ce_backward(int64_t N, int64_t V, const float* logits,
                                   const int64_t* targets, const float* loss, float grad_scale,
                                   float* dlogits, cudaStream_t s) {
    if (N == 0) return TPMLP_OK;
    CEBwdParams kp{};
    kp.logits = logits;
    kp.targets = targets;
    kp.loss = loss;
    kp.dlogits = dlogits;
    kp.N = N;
    kp.V = V;
    kp.scale = grad_scale;
    kp.vec = (V % 4 == 0) && aligned16(logits) && aligned16(dlogits);
    kp.err = device_error_word();
    if (kp.err == nullptr) return TPMLP_ERR_CUDA;
    {
        LaunchScope ls("vocab_ce_bwd", s);
        vocab_ce_bwd_kernel<<<(unsigned)N, 256, 0, s>>>(kp);
    }
    return cudaGetLastError() == cudaSuccess ? TPMLP_OK : TPMLP_ERR_CUDA;
}

tpmlp_status run_vocab_embedding(int f32, int64_t N, int64_t V, int64_t H, int T,
                                 const int64_t* ids, const void* const* table, void* out,
                                 cudaStream_t s) {
    if (N == 0) return TPMLP_OK;
    EmbParams kp{};
    kp.ids = ids;
    kp.out = out;
    kp.N = N;
    kp.V = V;
    kp.Vs = V / T;
    kp.row_bytes = H * (f32 ? 4 : 2);
    bool vec = kp.row_bytes % 16 == 0 && aligned16(out);
    for (int k = 0; k < T; ++k) {
        kp.table[k] = table[k];
        vec = vec && aligned16(table[k]);
    }
    kp.vec = vec;
    kp.err = device_error_word();
    if (kp.err == nullptr) return TPMLP_ERR_CUDA;
    if (vec) {
        // bulk copies: three 64 KB CTAs per SM
        static std::atomic<bool> attr_set[64] = {};
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return TPMLP_ERR_CUDA;
        if (!attr_set[dev].load()) {
            // idempotent, so concurrent first calls may both set it
            if (cudaFuncSetAttribute(vocab_embedding_bulk_kernel,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize, EMB_SMEM) != cudaSuccess)
                return TPMLP_ERR_CUDA;
            attr_set[dev].store(true);
        }
        const int64_t items = N * ((kp.row_bytes + EMB_CHUNK - 1) / EMB_CHUNK);
        const int64_t max_grid = (int64_t)device_sm_count() * 3;
        const int64_t grid = items < max_grid ? items : max_grid;
        LaunchScope ls("vocab_embedding", s);
        vocab_embedding_bulk_kernel<<<(unsigned)grid, 32, EMB_SMEM, s>>>(kp, wait_timeout_ns());
    } else {
        const int64_t max_grid = (int64_t)device_sm_count() * 8;
        int64_t grid = (N + 7) / 8;            // 8 warps per CTA, one token each
        if (grid > max_grid) grid = max_grid;
        LaunchScope ls("vocab_embedding", s);
        vocab_embedding_kernel<<<(unsigned)grid, 256, 0, s>>>(kp);
    }
    return cudaGetLastError() == cudaSuccess ? TPMLP_OK : TPMLP_ERR_CUDA;
}

tpmlp_status run_selftest_wait(uint64_t timeout_ns, cudaStream_t s) {
    int* err = device_error_word();
    if (err == nullptr) return TPMLP_ERR_CUDA;
    {
        LaunchScope ls("selftest_wait", s);
        selftest_wait_kernel<<<1, 32, 0, s>>>(err, timeout_ns);
    }
    return cudaGetLastError() == cudaSuccess ? TPMLP_OK : TPMLP_ERR_CUDA;
}

}  // namespace tpmlp
