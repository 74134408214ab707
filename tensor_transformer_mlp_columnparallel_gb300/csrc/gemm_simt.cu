// fp32 grouped / shard-folded GEMM on CUDA cores: the exact-fp32 mode of the
// block (fmaf in fp32, no TF32 tensor cores, whose 10-bit mantissa would not
// meet a 1e-5 relative bound). 64 x 64 output tile per CTA, 256 threads,
// 4 x 4 adjacent outputs per thread, K staged through shared memory 32 at a time with
// the next chunk's loads in flight in registers.
// When the tiles are fewer than the SMs (the small blocks this mode is for),
// a cluster of up to 8 CTAs shares one tile's K chunks; the leader adds the
// peers' partial tiles from their shared memory in rank order (so the result
// does not depend on timing) and runs the epilogue.
// Same problem description and epilogue semantics as the tensor-core GEMM.
#include "act.cuh"
#include "ptx.cuh"
#include "tpmlp_internal.h"

namespace tpmlp {
namespace {

constexpr int TM = 64, TN = 64, TK = 32;

// 16-byte load from another CTA's shared memory (a shared::cluster address
// from mapa_shared).
__device__ __forceinline__ float4 ld_cluster_v4(uint32_t addr) {
    float4 v;
    asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "r"(addr)
                 : "memory");
    return v;
}
constexpr int MAX_KS = 8;   // CTAs of a K-split cluster (the portable cluster limit)

struct SimtParams {
    const float* A[kMaxG];
    const float* B[kMaxG];
    const float* B2[kMaxG];   // DUAL: the up projection
    int64_t lda, ldb;
    int M, N, K, G, fold;
    int ks;   // CTAs per tile (a cluster along z) sharing its K chunks
    EpiArgs epi;
};

__device__ __forceinline__ void epi_scalar(const EpiArgs& e, int g, int m, int n, float v) {
    if (e.bias[g] != nullptr) v += static_cast<const float*>(e.bias[g])[n];
    if (e.kind == EPI_ACT) {
        if (e.aux[g] != nullptr) static_cast<float*>(e.aux[g])[(int64_t)m * e.ldaux + n] = v;
        v = act_fwd(e.act, v);
    } else if (e.kind == EPI_DACT) {
        v *= act_grad(e.act, static_cast<const float*>(e.aux[g])[(int64_t)m * e.ldaux + n]);
    }
    int cg = g;
    int64_t crow = m;
    if (e.row_shard > 0) {
        cg = (int)(m / e.row_shard);
        crow = m - (int64_t)cg * e.row_shard;
    }
    static_cast<float*>(e.C[cg])[crow * e.ldc + n] = v;
}

__device__ __forceinline__ void epi_swiglu_scalar(const EpiArgs& e, int g, int m, int n, float gv,
                                                  float uv) {
    if (e.aux[g] != nullptr) static_cast<float*>(e.aux[g])[(int64_t)m * e.ldaux + n] = gv;
    if (e.aux2[g] != nullptr) static_cast<float*>(e.aux2[g])[(int64_t)m * e.ldaux + n] = uv;
    static_cast<float*>(e.C[g])[(int64_t)m * e.ldc + n] = silu_f(gv) * uv;
}

template <bool A_MN, bool B_MN, bool DUAL>
__global__ void __launch_bounds__(256) simt_gemm_kernel(const SimtParams p) {
    // A and B stages; after the K loop the first 16 KB hold this CTA's
    // partial tile for a K split
    __shared__ __align__(16) float stage[2 * TK * (TM + 4)];
    __shared__ __align__(16) float Bs2[DUAL ? TK : 1][TN + 4];
    float (*As)[TM + 4] = reinterpret_cast<float (*)[TM + 4]>(stage);
    float (*Bs)[TN + 4] = reinterpret_cast<float (*)[TN + 4]>(stage + TK * (TM + 4));
    static_assert(2 * TK * (TM + 4) >= TM * TN, "partial tile fits in the stages");
    const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
    const int n0 = blockIdx.x * TN, m0 = blockIdx.y * TM;
    const int kr = (int)blockIdx.z % p.ks;    // rank in the K-split cluster
    const int gz = (int)blockIdx.z / p.ks;    // group (non-folded)

    float acc[4][4], acc2[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = acc2[i][j] = 0.f;

    // The K loop (over (shard, k) when folded) walks chunks of TK; the global
    // loads of chunk c + 1 go to registers while chunk c is computed from
    // shared memory, so a CTA waits for memory once, not once per chunk.
    const int ngroups = p.fold ? p.G : 1;
    const int kchunks = (p.K + TK - 1) / TK;
    const int nchunks = ngroups * kchunks;
    // this CTA's chunks [c_lo, c_hi) (all of them unless K is split)
    const int c_lo = (int)((int64_t)nchunks * kr / p.ks);
    const int c_hi = (int)((int64_t)nchunks * (kr + 1) / p.ks);
    constexpr int PER = TM * TK / 256;   // A (and B) elements each thread stages
    static_assert(TM * TK == 256 * PER && TN * TK == 256 * PER, "staging split");
    float ra[PER], rb[PER], rb2[PER];
    auto fetch = [&](int c) {
        const int gi = c / kchunks;
        const int k0 = (c - gi * kchunks) * TK;
        const int g = p.fold ? gi : gz;
        const float* A = p.A[g];
        const float* B = p.B[g];
        const float* B2 = p.B2[g];
#pragma unroll
        for (int u = 0; u < PER; ++u) {
            const int i = threadIdx.x + 256 * u;
            const int mm = A_MN ? i % TM : i / TK;
            const int ka = A_MN ? i / TM : i % TK;
            const int m = m0 + mm, k = k0 + ka;
            ra[u] = (m < p.M && k < p.K) ? (A_MN ? A[(int64_t)k * p.lda + m] : A[(int64_t)m * p.lda + k])
                                         : 0.f;
            const int nn = B_MN ? i % TN : i / TK;
            const int kb = B_MN ? i / TN : i % TK;
            const int n = n0 + nn, kq = k0 + kb;
            const bool in = n < p.N && kq < p.K;
            rb[u] = in ? (B_MN ? B[(int64_t)kq * p.ldb + n] : B[(int64_t)n * p.ldb + kq]) : 0.f;
            if (DUAL)
                rb2[u] = in ? (B_MN ? B2[(int64_t)kq * p.ldb + n] : B2[(int64_t)n * p.ldb + kq]) : 0.f;
        }
    };
    auto stash = [&]() {
#pragma unroll
        for (int u = 0; u < PER; ++u) {
            const int i = threadIdx.x + 256 * u;
            As[A_MN ? i / TM : i % TK][A_MN ? i % TM : i / TK] = ra[u];
            const int nn = B_MN ? i % TN : i / TK;
            const int kb = B_MN ? i / TN : i % TK;
            Bs[kb][nn] = rb[u];
            if (DUAL) Bs2[kb][nn] = rb2[u];
        }
    };
    if (c_lo < c_hi) {
        fetch(c_lo);
        stash();
    }
    __syncthreads();
    for (int c = c_lo; c < c_hi; ++c) {
        if (c + 1 < c_hi) fetch(c + 1);
#pragma unroll
        for (int kk = 0; kk < TK; ++kk) {
            // rows 4 ty .. 4 ty + 3 and columns 4 tx .. 4 tx + 3: one 16-byte
            // shared load each (a warp reads 2 A and 16 B vectors)
            const float4 av = *reinterpret_cast<const float4*>(&As[kk][4 * ty]);
            const float4 bv = *reinterpret_cast<const float4*>(&Bs[kk][4 * tx]);
            const float a[4] = {av.x, av.y, av.z, av.w};
            const float b[4] = {bv.x, bv.y, bv.z, bv.w};
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
            if (DUAL) {
                const float4 b2v = *reinterpret_cast<const float4*>(&Bs2[kk][4 * tx]);
                const float b2[4] = {b2v.x, b2v.y, b2v.z, b2v.w};
#pragma unroll
                for (int i = 0; i < 4; ++i)
#pragma unroll
                    for (int j = 0; j < 4; ++j) acc2[i][j] = fmaf(a[i], b2[j], acc2[i][j]);
            }
        }
        __syncthreads();
        if (c + 1 < c_hi) {
            stash();
            __syncthreads();
        }
    }
    if (!DUAL && p.ks > 1) {
        // peers publish their partial tile in their own shared memory; the
        // leader adds them in rank order; every CTA stays until the leader
        // has read it
        float4* red = reinterpret_cast<float4*>(stage);
        if (kr != 0) {
#pragma unroll
            for (int i = 0; i < 4; ++i)
                red[i * 256 + threadIdx.x] = make_float4(acc[i][0], acc[i][1], acc[i][2], acc[i][3]);
        }
        cluster_sync();
        if (kr == 0) {
            for (int r = 1; r < p.ks; ++r) {
                const uint32_t peer = mapa_shared(smem_u32(red), (uint32_t)r);
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const float4 v = ld_cluster_v4(peer + (uint32_t)(i * 256 + threadIdx.x) * 16u);
                    acc[i][0] += v.x;
                    acc[i][1] += v.y;
                    acc[i][2] += v.z;
                    acc[i][3] += v.w;
                }
            }
        }
        cluster_sync();
        if (kr != 0) return;
    }
    const int g_out = p.fold ? 0 : gz;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int m = m0 + 4 * ty + i;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int n = n0 + 4 * tx + j;
            if (m < p.M && n < p.N) {
                if (DUAL)
                    epi_swiglu_scalar(p.epi, g_out, m, n, acc[i][j], acc2[i][j]);
                else
                    epi_scalar(p.epi, g_out, m, n, acc[i][j]);
            }
        }
    }
}

}  // namespace

tpmlp_status run_gemm_simt(const GemmProblem& pr, cudaStream_t s) {
    if (pr.M <= 0 || pr.N <= 0) return TPMLP_OK;
    if (pr.K <= 0 || pr.G < 1 || pr.G > kMaxG) return TPMLP_ERR_SHAPE;
    SimtParams kp{};
    for (int g = 0; g < pr.G; ++g) {
        kp.A[g] = static_cast<const float*>(pr.A[g]);
        kp.B[g] = static_cast<const float*>(pr.B[g]);
        kp.B2[g] = static_cast<const float*>(pr.B2[g]);
    }
    kp.lda = pr.lda;
    kp.ldb = pr.ldb;
    kp.M = pr.M;
    kp.N = pr.N;
    kp.K = pr.K;
    kp.G = pr.G;
    kp.fold = pr.fold;
    kp.epi = pr.epi;
    const unsigned gy = (unsigned)((pr.M + TM - 1) / TM);
    if (gy > 65535u) return TPMLP_ERR_SHAPE;
    const int64_t gx = (pr.N + TN - 1) / TN;
    const int gz = pr.fold ? 1 : pr.G;
    // K split: as many CTAs per tile as fill the SMs once, at most MAX_KS and
    // at most one per K chunk
    int ks = 1;
    if (!pr.dual) {
        const int64_t ctas = gx * (int64_t)gy * gz;
        const int64_t nchunks = (int64_t)(pr.fold ? pr.G : 1) * ((pr.K + TK - 1) / TK);
        int64_t k = device_sm_count() / (ctas > 0 ? ctas : 1);
        if (k > MAX_KS) k = MAX_KS;
        if (k > nchunks) k = nchunks;
        ks = k > 1 ? (int)k : 1;
    }
    kp.ks = ks;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    cfg.gridDim = dim3((unsigned)gx, gy, (unsigned)(gz * ks));
    cfg.blockDim = dim3(256);
    cfg.stream = s;
    if (ks > 1) {
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 1;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = (unsigned)ks;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
    }
    cudaError_t e;
    {
        LaunchScope ls(pr.name, s);
        if (pr.dual) {
            if (pr.a_mn || !pr.b_mn || pr.fold) return TPMLP_ERR_ARG;   // the gated MLP's column GEMM only
            e = cudaLaunchKernelEx(&cfg, simt_gemm_kernel<false, true, true>, kp);
        } else if (pr.a_mn && pr.b_mn) {
            e = cudaLaunchKernelEx(&cfg, simt_gemm_kernel<true, true, false>, kp);
        } else if (pr.a_mn) {
            e = cudaLaunchKernelEx(&cfg, simt_gemm_kernel<true, false, false>, kp);
        } else if (pr.b_mn) {
            e = cudaLaunchKernelEx(&cfg, simt_gemm_kernel<false, true, false>, kp);
        } else {
            e = cudaLaunchKernelEx(&cfg, simt_gemm_kernel<false, false, false>, kp);
        }
    }
    if (e != cudaSuccess) return TPMLP_ERR_CUDA;
    return cudaGetLastError() == cudaSuccess ? TPMLP_OK : TPMLP_ERR_CUDA;
}

}  // namespace tpmlp
