// Grouped / shard-folded bf16 GEMM on the 5th-generation tensor cores.
//
// One persistent CTA per SM, 6 warps with fixed roles:
//   warp 0      TMA producer: streams A and B k-blocks into a STAGES-deep
//               shared-memory ring (128-byte swizzled boxes), one mbarrier
//               pair (full / empty) per stage; a stage is 64 deep in K, or
//               128 (two 64-wide boxes per operand) for CTA pairs;
//   warp 1      tensor-memory owner and MMA issuer: one thread issues
//               tcgen05.mma (M = 128, N = BN, K = 16) into a TMEM accumulator
//               and releases each stage with tcgen05.commit;
//   warps 2..5  epilogue: tcgen05.ld of the accumulator (lane = output row),
//               fused bias / activation / activation-derivative, global stores.
// Two TMEM accumulators (2 x BN columns) let the epilogue of tile i overlap
// the main loop of tile i + 1.
//
// Four launch forms, chosen per GEMM by run_gemm_tc:
//   - CTA pair (cluster of 2, M > 128): cta_group::2 MMAs of M = 256; each
//     CTA stages its own 128 A rows and half of the B rows;
//   - single CTA, 128 x 256 or 128 x 128 tiles (and 128 x 192 for GEMMs that
//     stream weights for a few token rows);
//   - K split (folded GEMMs with M <= 64): a cluster of 2-4 CTAs shares one
//     tile's k-blocks; the peers send their partial accumulator rows to the
//     leader's freed stage memory over DSMEM and the leader adds them before
//     its epilogue (one tile per cluster);
//   - stream-K (M <= 64, given scratch in the caller's workspace): every CTA
//     takes an equal contiguous share of the (tile, k-block) units; tiles
//     shared by several CTAs are summed through the scratch by the last
//     warp to count in, in CTA order.
//
// The problem is a batch of G same-shape GEMMs (one per shard r: the column
// GEMM X W1^(r), the row GEMM H^(r) W2^(r), and the backward products) or,
// with `fold`, ONE output whose K loop runs over (r, k): the row GEMM's shard
// sum Y = sum_r H^(r) W2^(r) then happens inside the fp32 accumulator (the
// block-end reduction of page "一层 MLP 太宽而放不下时怎样切？", §04, done
// without writing partial sums).
//
// Every mbarrier wait is bounded in time (%globaltimer); a wait that runs out
// records TPMLP_ERR_TIMEOUT, raises a CTA-wide abort flag, and every role
// leaves its loop. The producer then waits for its own loads in flight, the
// MMA thread for its own MMAs, and the TMEM owner frees the accumulator.
#include <cuda_bf16.h>
#include <cudaTypedefs.h>

#include <cstdio>
#include <mutex>

#include "act.cuh"
#include "ptx.cuh"
#include "tpmlp_internal.h"

namespace tpmlp {
namespace {

constexpr int BM = 128;           // MMA M (rows of A / TMEM lanes)
constexpr int BKB = 64;           // K extent of a K-major box: one 128-byte swizzle row of bf16
constexpr int UMMA_K = 16;        // K of one kind::f16 MMA
constexpr int NUM_THREADS = 192;
constexpr int ACC_BUFS = 2;
constexpr int BOX_MN = 64;        // MN extent of an MN-major box (128 bytes)
constexpr int GROUP_M = 12;       // raster band height, in M tiles
constexpr int KSPLIT_ROWS = 64;   // rows a K-split cluster exchanges (M <= 64)

// BN: accumulator columns (MMA N). PAIR: a CTA pair (cluster of 2) issues
// cta_group::2 MMAs of M = 256; each CTA stages its own 128 rows of A and its
// own BN/2 rows of B, which halves the B bytes each SM pulls from L2.
template <int BN, bool PAIR>
struct Cfg {
    static constexpr int CTAS = PAIR ? 2 : 1;
    static constexpr int TILE_M = BM * CTAS;
    static constexpr int B_ROWS = BN / CTAS;                 // B rows (N) staged per CTA
    // K depth of one stage. A pair stages 128 (two 64-wide boxes per K-major
    // operand, 3 stages of 64 KB) instead of 64 (7 of 32 KB): half the stage
    // hand-offs per FLOP. On the power-capped fwd+bwd step (~1500 MHz) that
    // took 2-3% fewer cycles; at 2070 MHz (zero data, uncapped) the shallower
    // ring costs ~6% more. Single CTAs (few-token GEMMs) stage 64.
    static constexpr int BK = PAIR ? 2 * BKB : BKB;
    static constexpr int A_SUB = BM * BKB * 2;               // one K-major A box
    static constexpr int B_SUB = B_ROWS * BKB * 2;           // one K-major B box
    static constexpr int MN_BOX_BYTES = BOX_MN * BK * 2;     // one 64-wide MN chunk of a stage
    static constexpr int A_BYTES = BM * BK * 2;
    static constexpr int B_BYTES = B_ROWS * BK * 2;
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;    // per CTA
    // as many stages as fit in 227 KB next to the barriers and the 1 KB alignment slack
    static constexpr int SMEM_LIMIT = 232448;
    static constexpr int STAGES_FIT = (SMEM_LIMIT - 1024 - 256) / STAGE_BYTES;
    static constexpr int STAGES = STAGES_FIT > 8 ? 8 : STAGES_FIT;
    // two accumulators of BN columns, allocated as a power of two
    static constexpr int TMEM_COLS = ACC_BUFS * BN <= 256 ? 256 : 512;
    static constexpr int NUM_BARS_BASE = 2 * STAGES + 2 * ACC_BUFS + 5;
    // Output staging for tensor stores: per epilogue warp two 4 KB buffers
    // (one 32 x 32 chunk of fp32, or of bf16 C and bf16 Z), where the ring
    // leaves room (not for 128-column tiles, whose 7th stage takes it).
    static constexpr int OUT_BUF = 4096;
    static constexpr int OUT_BYTES = 4 * 2 * OUT_BUF;
    static constexpr bool TMA_OUT = SMEM_LIMIT - (1024 + STAGES * STAGE_BYTES + 256) >= OUT_BYTES;
    static constexpr int SMEM_BYTES = 1024 + STAGES * STAGE_BYTES + (TMA_OUT ? OUT_BYTES : 0) + 256;
    // with staging, two barriers per epilogue warp for the act' epilogue's Z loads
    static constexpr int NUM_BARS = NUM_BARS_BASE + (TMA_OUT ? 8 : 0);
    // barriers, then the TMEM address, the abort flag and the pair's load count
    static_assert(NUM_BARS * 8 + 12 <= 256, "barrier area");
    static_assert(SMEM_BYTES <= SMEM_LIMIT, "shared memory");
    static_assert(TMEM_COLS == 256 || TMEM_COLS == 512, "TMEM columns");
    static_assert(B_ROWS % BOX_MN == 0, "MN-major B boxes");
    // K split across a cluster (single-CTA tiles, M <= KSPLIT_ROWS): each peer's
    // partial accumulator rows land in the leader's freed stage memory
    static constexpr int RED_SLOT_BYTES = KSPLIT_ROWS * BN * 4;
    static constexpr int MAX_KSPLIT = PAIR ? 1 : 1 + (STAGES * STAGE_BYTES) / RED_SLOT_BYTES;
};

struct TcParams {
    CUtensorMap tmA[kMaxG];
    CUtensorMap tmB[kMaxG];
    CUtensorMap tmB2[kMaxG];   // dual: the second B (up projection)
    CUtensorMap tmC[kMaxG];    // tma_out: the output of each group (box 32 x 32)
    CUtensorMap tmAux[kMaxG];  // tma_out, EPI_ACT with Z saved: Z of each group
    int M, N, K;
    int G, fold;
    int a_mn, b_mn;
    int a_3d, b_3d;   // MN-major operand read as ONE 3-D box {64, BK, rows/64} per stage
    int m_tiles, n_tiles, k_blocks;
    int num_tiles;
    int dual;         // tile = BN/2 outputs of A B (accumulator columns [0, BN/2)) and of
                      // A B2 (columns [BN/2, BN)); N counts outputs
    int raster;       // tile order, see decode_tile
    int band;         // band width in tiles
    int ksplit;       // CTAs of a cluster sharing one tile's K range (single-CTA
                      // tiles, M <= KSPLIT_ROWS, one tile per cluster); 1 = off
    int sk;           // 1: stream-K phase after the whole tiles (see Work)
    int sk_dp_tiles;  // tiles [0, sk_dp_tiles) run whole before the stream-K phase
    int sk_units;     // U = stream-K tiles x k-blocks
    int sk_parts;     // units taking part in the stream-K phase (the first sk_parts)
    int sk_rows;      // rows per CTA of a scratch slot (32, 64 or 128)
    float* sk_part;   // P x 2 x CTAS slots of sk_rows x BN fp32 partial accumulators
    int* sk_cnt;      // 4 x CTAS counters per stream-K tile (one per 32-row warp), zero at launch
    EpiArgs epi;
    int* err;
    uint64_t timeout_ns;
    uint64_t drain_ns;   // limit of the waits for copies and MMAs already in flight
    int inject;          // failure-detection self test: the role that stalls (0: none)
    int tma_out;         // 1: the epilogue writes C (and Z) through staging and tensor stores
    int alt;             // bit 0: whole tiles of odd waves walk their K range from the top
                         // down; bit 1: odd bands walk their tiles in reverse (decode_tile)
};

// Shared-memory matrix descriptor, 128-byte swizzle (tcgen05 format: start
// address, leading- and stride-dimension byte offsets in 16-byte units,
// descriptor version 1 at bit 46, swizzle mode 2 at bit 61).
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    uint64_t d = (uint64_t)((saddr & 0x3FFFFu) >> 4);
    d |= (uint64_t)((lbo & 0x3FFFFu) >> 4) << 16;
    d |= (uint64_t)((sbo & 0x3FFFFu) >> 4) << 32;
    d |= 1ull << 46;
    d |= 2ull << 61;
    return d;
}

// Instruction descriptor of kind::f16: fp32 accumulator (bits 4-5 = 1), bf16
// A and B (bits 7-9, 10-12 = 1), operand majorness (bits 15, 16: 1 = MN-major),
// N >> 3 at bit 17, M >> 4 at bit 24.
__host__ __device__ constexpr uint32_t instr_desc(int M, int N, int a_mn, int b_mn) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)a_mn << 15) | ((uint32_t)b_mn << 16) |
           ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// Tile order. Consecutive tile indices run on CTAs that are resident at the
// same time, so the order decides what L2 can reuse.
//   raster 0: group by group; inside a group, bands of `band` M-tiles with
//             the M index fastest (the fold GEMMs use this with G = 1);
//   raster 1: A is the same matrix for every group (X, dY): bands of `band`
//             M-tiles with every group's N-tiles inside the band, so the band's
//             A panel is read from HBM once for all groups;
//   raster 2: B is the same matrix for every group: the same with the roles
//             of M and N swapped.
// With p.alt bit 1, odd bands walk their tiles in reverse, so the wave that
// crosses from one band to the next works on the same B (raster 2: A) panels
// on both sides of the boundary.
template <int BN, int TILE_M>
__device__ __forceinline__ void decode_tile(const TcParams& p, int t, int& g, int& m0, int& n0) {
    int mt, nt;
    if (p.raster == 0) {
        const int per_group = p.m_tiles * p.n_tiles;
        g = p.fold ? 0 : t / per_group;
        const int local = t - g * per_group;
        const int band = local / (p.band * p.n_tiles);
        const int first_m = band * p.band;
        const int band_m = min(p.m_tiles - first_m, p.band);
        const int in_band = local - band * p.band * p.n_tiles;
        mt = first_m + in_band % band_m;
        nt = in_band / band_m;
        if ((p.alt & 2) && (band & 1)) nt = p.n_tiles - 1 - nt;
    } else if (p.raster == 1) {
        const int band = t / (p.band * p.n_tiles * p.G);
        const int first_m = band * p.band;
        const int band_m = min(p.m_tiles - first_m, p.band);
        const int in_band = t - band * p.band * p.n_tiles * p.G;
        mt = first_m + in_band % band_m;
        int rest = in_band / band_m;
        if ((p.alt & 2) && (band & 1)) rest = p.n_tiles * p.G - 1 - rest;
        g = rest / p.n_tiles;
        nt = rest - g * p.n_tiles;
    } else {
        const int band = t / (p.band * p.m_tiles * p.G);
        const int first_n = band * p.band;
        const int band_n = min(p.n_tiles - first_n, p.band);
        const int in_band = t - band * p.band * p.m_tiles * p.G;
        nt = first_n + in_band % band_n;
        int rest = in_band / band_n;
        if ((p.alt & 2) && (band & 1)) rest = p.m_tiles * p.G - 1 - rest;
        g = rest / p.m_tiles;
        mt = rest - g * p.m_tiles;
    }
    m0 = mt * TILE_M;
    n0 = nt * BN;
}

// The work items of one unit (a CTA, or a CTA pair / K-split cluster): tiles
// first_tile, first_tile + step, ... (step = the number of units) with the
// k-block range [kb_lo, kb_hi) each. With stream-K the whole tiles stop at
// sk_dp_tiles (full waves: every unit has the same number), and unit i < P
// (P = sk_parts) then takes its contiguous share [i U / P, (i+1) U / P) of
// the U = remaining tiles x k-blocks, cut at tile boundaries. (The few-token
// GEMMs have no whole tiles and P = all units; larger GEMMs cut each
// remaining tile into P / tiles equal K chunks.) Every role walks the same
// sequence.
struct Work {
    int t, kb0, kb1;   // current item: tile, k-blocks [kb0, kb1)
    int u, u_end;      // stream-K: next unit (counted from the first stream-K tile), end
    int kb_total, step, dp_tiles;
    bool sk, has_sk;
    __device__ __forceinline__ Work(const TcParams& p, int first_tile, int tile_step, int kb_lo,
                                    int kb_hi, int kbt)
        : t(first_tile), kb0(kb_lo), kb1(kb_hi), u(0), u_end(0), kb_total(kbt), step(tile_step),
          dp_tiles(p.sk ? p.sk_dp_tiles : p.num_tiles), sk(false), has_sk(p.sk != 0) {
        if (has_sk && first_tile < p.sk_parts) {
            u = (int)((int64_t)first_tile * p.sk_units / p.sk_parts);
            u_end = (int)((int64_t)(first_tile + 1) * p.sk_units / p.sk_parts);
        }
        if (t >= dp_tiles) enter_sk();
    }
    __device__ __forceinline__ void enter_sk() {
        sk = has_sk;
        if (sk) load();
    }
    __device__ __forceinline__ void load() {
        if (u < u_end) {
            const int tl = u / kb_total;
            t = dp_tiles + tl;
            kb0 = u - tl * kb_total;
            kb1 = min(kb_total, kb0 + (u_end - u));
        }
    }
    __device__ __forceinline__ bool valid() const { return sk ? u < u_end : t < dp_tiles; }
    __device__ __forceinline__ void next() {
        if (sk) {
            u += kb1 - kb0;
            load();
        } else {
            t += step;
            if (t >= dp_tiles) enter_sk();
        }
    }
    // a stream-K item that covers only part of its tile's K range
    __device__ __forceinline__ bool partial() const { return sk && (kb0 > 0 || kb1 < kb_total); }
};

// stream-K: the unit whose range holds k-block unit x, and the stream-K tile
// (counted from the first) of unit c's first k-block unit
__device__ __forceinline__ int sk_cta_of(int64_t x, int64_t U, int P) {
    return (int)(((x + 1) * P - 1) / U);
}
__device__ __forceinline__ int sk_first_tile(int c, int64_t U, int P, int kb_total) {
    return (int)((int64_t)c * U / P / kb_total);
}

// act / act' over one 32-column chunk with the activation fixed at compile
// time, so the per-element code carries no activation branches
template <int ACT>
__device__ __forceinline__ void act_chunk(float (&v)[32]) {
#pragma unroll
    for (int j = 0; j < 32; ++j) v[j] = act_fwd_bf16(ACT, v[j]);
}

template <int ACT>
__device__ __forceinline__ void dact_chunk(float (&v)[32], const float (&z)[32]) {
#pragma unroll
    for (int j = 0; j < 32; ++j) v[j] *= act_grad_bf16(ACT, z[j]);
}

// Epilogue arithmetic of one thread, in two steps: 32 consecutive columns
// [col0, col0 + 32) of output row `row`. epilogue_bias: v = acc (+ bias)
// from the accumulator values in r[] (for EPI_ACT this is the pre-activation
// Z); epilogue_act: v = act(v) (EPI_ACT) or v = v * act'(aux) (EPI_DACT).
// Rows >= M (outside the output) read no auxiliary input.
__device__ __forceinline__ void epilogue_bias(const EpiArgs& e, int g, int col0, int N,
                                              const uint32_t (&r)[32], float (&v)[32]) {
#pragma unroll
    for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r[j]);
    const bool full = (col0 + 32 <= N);
    if (e.bias[g] != nullptr) {
        const __nv_bfloat16* b = static_cast<const __nv_bfloat16*>(e.bias[g]) + col0;
        if (full) {
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const uint4 w = __ldg(reinterpret_cast<const uint4*>(b) + q);
                const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                for (int h = 0; h < 4; ++h) {
                    float lo, hi;
                    unpack_bf16x2(ws[h], lo, hi);
                    v[q * 8 + 2 * h] += lo;
                    v[q * 8 + 2 * h + 1] += hi;
                }
            }
        } else {
#pragma unroll
            for (int j = 0; j < 32; ++j)
                if (col0 + j < N) v[j] += bf2f(b[j]);
        }
    }
}

__device__ __forceinline__ void epilogue_act(const EpiArgs& e, int g, int row, int col0, int M,
                                             int N, float (&v)[32]) {
    const bool full = (col0 + 32 <= N);
    if (e.kind == EPI_ACT) {
        switch (e.act) {   // one dispatch per chunk, a tight loop per activation
            case TPMLP_ACT_RELU: act_chunk<TPMLP_ACT_RELU>(v); break;
            case TPMLP_ACT_GELU_ERF: act_chunk<TPMLP_ACT_GELU_ERF>(v); break;
            case TPMLP_ACT_GELU_SIGMOID: act_chunk<TPMLP_ACT_GELU_SIGMOID>(v); break;
            default: act_chunk<TPMLP_ACT_GELU_TANH>(v); break;
        }
    } else if (e.kind == EPI_DACT) {
        float zv[32];
        if (row >= M) {
#pragma unroll
            for (int j = 0; j < 32; ++j) zv[j] = 0.f;
        } else {
            const __nv_bfloat16* za =
                static_cast<const __nv_bfloat16*>(e.aux[g]) + (int64_t)row * e.ldaux + col0;
            if (full) {
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const uint4 w = *(reinterpret_cast<const uint4*>(za) + q);
                    unpack_bf16x2(w.x, zv[q * 8 + 0], zv[q * 8 + 1]);
                    unpack_bf16x2(w.y, zv[q * 8 + 2], zv[q * 8 + 3]);
                    unpack_bf16x2(w.z, zv[q * 8 + 4], zv[q * 8 + 5]);
                    unpack_bf16x2(w.w, zv[q * 8 + 6], zv[q * 8 + 7]);
                }
            } else {
#pragma unroll
                for (int j = 0; j < 32; ++j) zv[j] = col0 + j < N ? bf2f(za[j]) : 0.f;
            }
        }
        switch (e.act) {
            case TPMLP_ACT_RELU: dact_chunk<TPMLP_ACT_RELU>(v, zv); break;
            case TPMLP_ACT_GELU_ERF: dact_chunk<TPMLP_ACT_GELU_ERF>(v, zv); break;
            case TPMLP_ACT_GELU_SIGMOID: dact_chunk<TPMLP_ACT_GELU_SIGMOID>(v, zv); break;
            default: dact_chunk<TPMLP_ACT_GELU_TANH>(v, zv); break;
        }
    }
}

// 32 bf16 values of one row as four 16-byte words
__device__ __forceinline__ void pack_row_bf16(const float (&v)[32], uint4 (&w)[4]) {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        w[q].x = pack_bf16x2(v[q * 8 + 0], v[q * 8 + 1]);
        w[q].y = pack_bf16x2(v[q * 8 + 2], v[q * 8 + 3]);
        w[q].z = pack_bf16x2(v[q * 8 + 4], v[q * 8 + 5]);
        w[q].w = pack_bf16x2(v[q * 8 + 6], v[q * 8 + 7]);
    }
}

// Per-thread global stores of one row chunk (the form without staging):
// Z (bf16, EPI_ACT with aux) and C (bf16 or fp32; by row blocks for the
// reduce-scatter).
__device__ __forceinline__ void store_z_thread(const EpiArgs& e, int g, int row, int col0, int M,
                                               int N, const float (&z)[32]) {
    if (row >= M) return;
    __nv_bfloat16* za = static_cast<__nv_bfloat16*>(e.aux[g]) + (int64_t)row * e.ldaux + col0;
    if (col0 + 32 <= N) {
        uint4 w[4];
        pack_row_bf16(z, w);
#pragma unroll
        for (int q = 0; q < 4; ++q) reinterpret_cast<uint4*>(za)[q] = w[q];
    } else {
#pragma unroll
        for (int j = 0; j < 32; ++j)
            if (col0 + j < N) za[j] = __float2bfloat16_rn(z[j]);
    }
}

__device__ __forceinline__ void store_c_thread(const EpiArgs& e, int g, int row, int col0, int M,
                                               int N, const float (&v)[32]) {
    if (row >= M) return;
    const bool full = (col0 + 32 <= N);
    int cg = g;
    int64_t crow = row;
    if (e.row_shard > 0) {          // reduce-scatter output: row block i -> C[i]
        cg = (int)(row / e.row_shard);
        crow = row - (int64_t)cg * e.row_shard;
    }
    if (e.out_f32) {
        float* c = static_cast<float*>(e.C[cg]) + crow * e.ldc + col0;
        if (full) {
#pragma unroll
            for (int q = 0; q < 8; ++q)
                reinterpret_cast<float4*>(c)[q] =
                    make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
        } else {
#pragma unroll
            for (int j = 0; j < 32; ++j)
                if (col0 + j < N) c[j] = v[j];
        }
    } else {
        __nv_bfloat16* c = static_cast<__nv_bfloat16*>(e.C[cg]) + crow * e.ldc + col0;
        if (full) {
            uint4 w[4];
            pack_row_bf16(v, w);
#pragma unroll
            for (int q = 0; q < 4; ++q) reinterpret_cast<uint4*>(c)[q] = w[q];
        } else {
#pragma unroll
            for (int j = 0; j < 32; ++j)
                if (col0 + j < N) c[j] = __float2bfloat16_rn(v[j]);
        }
    }
}

// Row r of a 32 x 32 bf16 chunk loaded by a tensor load into a 64-byte
// swizzled buffer (the layout stage_row writes), as 32 floats.
__device__ __forceinline__ void load_row_bf16_smem(uint32_t buf, int r, float (&z)[32]) {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        uint32_t w0, w1, w2, w3;
        asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                     : "=r"(w0), "=r"(w1), "=r"(w2), "=r"(w3)
                     : "r"(buf + (uint32_t)r * 64u + (uint32_t)((j ^ ((r >> 1) & 3)) << 4))
                     : "memory");
        unpack_bf16x2(w0, z[j * 8 + 0], z[j * 8 + 1]);
        unpack_bf16x2(w1, z[j * 8 + 2], z[j * 8 + 3]);
        unpack_bf16x2(w2, z[j * 8 + 4], z[j * 8 + 5]);
        unpack_bf16x2(w3, z[j * 8 + 6], z[j * 8 + 7]);
    }
}

// v *= act'(z) over one chunk
__device__ __forceinline__ void dact_apply(int act, float (&v)[32], const float (&z)[32]) {
    switch (act) {
        case TPMLP_ACT_RELU: dact_chunk<TPMLP_ACT_RELU>(v, z); break;
        case TPMLP_ACT_GELU_ERF: dact_chunk<TPMLP_ACT_GELU_ERF>(v, z); break;
        case TPMLP_ACT_GELU_SIGMOID: dact_chunk<TPMLP_ACT_GELU_SIGMOID>(v, z); break;
        default: dact_chunk<TPMLP_ACT_GELU_TANH>(v, z); break;
    }
}

// One row of a 32 x 32 output chunk into the warp's staging buffer, in the
// layout of the output tensor map's swizzle: bf16 rows are 64 bytes with
// 64-byte swizzle (16-byte word j of row r at word j ^ ((r >> 1) & 3)), fp32
// rows 128 bytes with 128-byte swizzle (word j at j ^ (r & 7)), so the
// warp's 16-byte stores of one word index hit distinct banks.
__device__ __forceinline__ void stage_row(uint32_t buf, int r, bool f32, const float (&v)[32]) {
    if (f32) {
#pragma unroll
        for (int j = 0; j < 8; ++j)
            st_shared_v4(buf + (uint32_t)r * 128u + (uint32_t)((j ^ (r & 7)) << 4),
                         __float_as_uint(v[4 * j]), __float_as_uint(v[4 * j + 1]),
                         __float_as_uint(v[4 * j + 2]), __float_as_uint(v[4 * j + 3]));
    } else {
        uint4 w[4];
        pack_row_bf16(v, w);
#pragma unroll
        for (int j = 0; j < 4; ++j)
            st_shared_v4(buf + (uint32_t)r * 64u + (uint32_t)((j ^ ((r >> 1) & 3)) << 4), w[j].x,
                         w[j].y, w[j].z, w[j].w);
    }
}

// Gated-MLP epilogue of one thread: 32 outputs [col0, col0 + 32) of row
// `row` from the gate accumulators rg[] and the up accumulators ru[].
__device__ __forceinline__ void epilogue_swiglu_chunk(const EpiArgs& e, int g, int row, int col0,
                                                      int M, int N, const uint32_t (&rg)[32],
                                                      const uint32_t (&ru)[32]) {
    if (row >= M) return;
    float gv[32], uv[32], h[32];
#pragma unroll
    for (int j = 0; j < 32; ++j) {
        gv[j] = __uint_as_float(rg[j]);
        uv[j] = __uint_as_float(ru[j]);
        h[j] = silu_bf16(gv[j]) * uv[j];
    }
    const bool full = (col0 + 32 <= N);
    const float* srcs[3] = {gv, uv, h};
    void* dsts[3] = {e.aux[g], e.aux2[g], e.C[g]};
    const int64_t lds[3] = {e.ldaux, e.ldaux, e.ldc};
#pragma unroll
    for (int o = 0; o < 3; ++o) {
        if (dsts[o] == nullptr) continue;
        __nv_bfloat16* d = static_cast<__nv_bfloat16*>(dsts[o]) + (int64_t)row * lds[o] + col0;
        const float* v = srcs[o];
        if (full) {
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                uint4 w;
                w.x = pack_bf16x2(v[q * 8 + 0], v[q * 8 + 1]);
                w.y = pack_bf16x2(v[q * 8 + 2], v[q * 8 + 3]);
                w.z = pack_bf16x2(v[q * 8 + 4], v[q * 8 + 5]);
                w.w = pack_bf16x2(v[q * 8 + 6], v[q * 8 + 7]);
                reinterpret_cast<uint4*>(d)[q] = w;
            }
        } else {
#pragma unroll
            for (int j = 0; j < 32; ++j)
                if (col0 + j < N) d[j] = __float2bfloat16_rn(v[j]);
        }
    }
}

template <int BN, bool PAIR>
__global__ void __launch_bounds__(NUM_THREADS, 1) tc_gemm_kernel(const __grid_constant__ TcParams p) {
    using C = Cfg<BN, PAIR>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~static_cast<uintptr_t>(1023));
    const uint32_t sA0 = smem_u32(smem);
    const uint32_t sB0 = sA0 + C::STAGES * C::A_BYTES;
    // staging for the epilogue's tensor stores (1024-byte aligned), then the barriers
    const uint32_t sOut = sA0 + C::STAGES * C::STAGE_BYTES;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::STAGES * C::STAGE_BYTES +
                                                 (C::TMA_OUT ? C::OUT_BYTES : 0));
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + C::NUM_BARS);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    // the odd CTA of a pair writes the number of loads it issued here (even CTA)
    volatile uint32_t* peer_issued = reinterpret_cast<volatile uint32_t*>(tmem_slot + 2);
    const uint32_t bar0 = smem_u32(bars);
    // barrier indices; STALL is never completed (the self test's stall waits on
    // it), XCNT carries the odd CTA's load count to the even CTA
    const int FULL = 0, EMPTY = C::STAGES, TFULL = 2 * C::STAGES, TEMPTY = TFULL + ACC_BUFS,
              DRAIN = TEMPTY + ACC_BUFS, RFREE = DRAIN + 1, RFULL = DRAIN + 2, STALL = DRAIN + 3,
              XCNT = DRAIN + 4, ZLD = DRAIN + 5;   // ZLD + 2 * quarter + set: Z chunk loads
    auto bar = [&](int i) -> uint32_t { return bar0 + 8u * (uint32_t)i; };

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = PAIR ? cluster_ctarank() : 0u;      // CTA within the pair
    const bool leader = rank == 0;
    // K split: CTA `krank` of a cluster of `ks` accumulates its share of the
    // tile's k-blocks; the peers hand their partial rows to CTA 0
    const int ks = PAIR ? 1 : p.ksplit;
    const uint32_t krank = ks > 1 ? cluster_ctarank() : 0u;
    const bool clustered = PAIR || ks > 1;
    const int first_tile = clustered ? (int)cluster_id_x() : (int)blockIdx.x;
    const int tile_step = clustered ? (int)num_clusters_x() : (int)gridDim.x;
    // epilogue warps holding rows that a K split exchanges (rows < min(M, 64))
    const int red_warps = (min(p.M, KSPLIT_ROWS) + 31) / 32;

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::STAGES; ++s) {
            mbar_init(bar(FULL + s), 1);
            mbar_init(bar(EMPTY + s), 1);
        }
        for (int a = 0; a < ACC_BUFS; ++a) {
            mbar_init(bar(TFULL + a), 1);
            mbar_init(bar(TEMPTY + a), 4 * C::CTAS);   // every epilogue warp of the pair
        }
        mbar_init(bar(DRAIN), 1);
        mbar_init(bar(RFREE), 1);                                  // leader: stages free
        mbar_init(bar(RFULL), ks > 1 ? (ks - 1) * red_warps * 32 : 1);   // every peer lane
        mbar_init(bar(STALL), 1);
        mbar_init(bar(XCNT), 1);
        if constexpr (C::TMA_OUT)
            for (int z = 0; z < 8; ++z) mbar_init(bar(ZLD + z), 1);
        *abort_flag = 0;
        fence_mbar_init();
        fence_proxy_async_smem();
    }
    if (warp == 0 && lane == 0) {
        for (int g = 0; g < p.G; ++g) {
            prefetch_tmap(&p.tmA[g]);
            prefetch_tmap(&p.tmB[g]);
            if (p.dual) prefetch_tmap(&p.tmB2[g]);
        }
    }
    if (warp == 1) {
        if constexpr (PAIR) {
            tmem_alloc_pair(smem_u32(tmem_slot), C::TMEM_COLS);
            tmem_relinquish_pair();
        } else {
            tmem_alloc(smem_u32(tmem_slot), C::TMEM_COLS);
            tmem_relinquish();
        }
    }
    tc_fence_before();
    __syncthreads();
    if (clustered) cluster_sync();   // peer barriers initialised before any remote signal
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    // Launched with programmatic stream serialization: the CTAs may start
    // while the previous kernel on the stream winds down; nothing that kernel
    // writes is touched before this wait. (The GEMM does not trigger its own
    // dependents early: CTAs of the next kernel starting on SMs this grid
    // frees, while its last wave still streams, measured slower.)
    if (warp != 0 || lane != 0) pdl_wait();

    const int kb_per_group = p.k_blocks;
    const int kb_total = p.fold ? p.G * kb_per_group : kb_per_group;
    // this CTA's k-blocks of each tile (all of them unless K is split)
    const int kb_lo = (int)((int64_t)kb_total * krank / ks);
    const int kb_hi = (int)((int64_t)kb_total * (krank + 1) / ks);

    if (warp == 0) {
        if (lane == 0) {
            // ---------------- TMA producer (each CTA loads its own rows) ----------------
            // The issue loop is on the critical path (the TMA unit drains its
            // queue quickly), so it carries its shard and K offset as counters
            // instead of dividing the k-block index.
            // the pair's stage is complete when BOTH CTAs' bytes landed on the
            // even CTA's full barrier
            const uint32_t full0 = PAIR ? mapa_shared(bar(FULL), 0) : bar(FULL);
            const int k_group = kb_per_group * C::BK;   // K extent of one shard
            // Loads of one k-block into stage st: the A and B boxes of shard gk
            // at K offset k0, completing on the stage's full barrier.
            auto issue = [&](int st, int gk, int k0, int am0, int bn0, int n0) {
                const uint32_t fb = full0 + 8u * (uint32_t)st;
                const uint32_t a_dst = sA0 + st * C::A_BYTES;
                const uint32_t b_dst = sB0 + st * C::B_BYTES;
                auto load = [&](uint32_t dst, const CUtensorMap* m, int x, int y) {
                    if constexpr (PAIR)
                        tma_load_2d_pair(dst, m, fb, x, y);
                    else
                        tma_load_2d(dst, m, fb, x, y);
                };
                auto load3 = [&](uint32_t dst, const CUtensorMap* m, int x, int y, int z) {
                    if constexpr (PAIR)
                        tma_load_3d_pair(dst, m, fb, x, y, z);
                    else
                        tma_load_3d(dst, m, fb, x, y, z);
                };
                if (!p.a_mn) {
#pragma unroll
                    for (int h = 0; h < C::BK / BKB; ++h)
                        load(a_dst + h * C::A_SUB, &p.tmA[gk], k0 + h * BKB, am0);
                } else if (p.a_3d) {
                    load3(a_dst, &p.tmA[gk], 0, k0, am0 / BOX_MN);
                } else {
#pragma unroll
                    for (int j = 0; j < BM / BOX_MN; ++j)
                        load(a_dst + j * C::MN_BOX_BYTES, &p.tmA[gk], am0 + j * BOX_MN, k0);
                }
                // `rows` B rows (N index) starting at n_start from map m into dst
                auto load_b = [&](uint32_t dst, const CUtensorMap* m, int n_start, int rows) {
                    if (!p.b_mn) {
#pragma unroll
                        for (int h = 0; h < C::BK / BKB; ++h)
                            load(dst + h * C::B_SUB, m, k0 + h * BKB, n_start);
                    } else if (p.b_3d) {
                        load3(dst, m, 0, k0, n_start / BOX_MN);
                    } else {
                        for (int j = 0; j < rows / BOX_MN; ++j)
                            load(dst + j * C::MN_BOX_BYTES, m, n_start + j * BOX_MN, k0);
                    }
                };
                if (!p.dual) {
                    load_b(b_dst, &p.tmB[gk], bn0, C::B_ROWS);
                } else if constexpr (PAIR) {
                    // the even CTA stages the gate rows, the odd CTA the up rows
                    load_b(b_dst, rank == 0 ? &p.tmB[gk] : &p.tmB2[gk], n0 / 2, BN / 2);
                } else {
                    load_b(b_dst, &p.tmB[gk], n0 / 2, BN / 2);
                    load_b(b_dst + (BN / 2) * (p.b_mn ? C::BK : BKB) * 2, &p.tmB2[gk], n0 / 2, BN / 2);
                }
            };
            int s = 0;
            uint32_t ph = 0;
            uint32_t issued = 0;
            bool ok = p.inject != 3 || wait_bounded(bar(STALL), 0, abort_flag, p.err, p.timeout_ns, true);
            pdl_wait();
            for (Work w(p, first_tile, tile_step, kb_lo, kb_hi, kb_total); ok && w.valid(); w.next()) {
                const int t = w.t;
                int g, m0, n0;
                decode_tile<BN, C::TILE_M>(p, t, g, m0, n0);
                const int am0 = m0 + (int)rank * BM;          // this CTA's A rows
                const int bn0 = n0 + (int)rank * C::B_ROWS;   // this CTA's B rows (N)
                // Whole tiles of every other wave (the CTA's tiles t, t + step,
                // ... are one per wave) take their k-blocks from the last down:
                // such a wave starts on the K slices of the panels it shares with
                // the wave before, which that wave read last and which are the
                // likeliest to be still in L2. The MMA issuer counts k-blocks
                // only, so the order is the producer's alone.
                const bool down = (p.alt & 1) && !w.sk && ((w.t / w.step) & 1);
                const int kb_first = down ? w.kb1 - 1 : w.kb0;
                // shard of the first k-block and its K offset inside the shard
                int gk = p.fold ? kb_first / kb_per_group : g;
                int k0 = (p.fold ? kb_first - (kb_first / kb_per_group) * kb_per_group : kb_first) * C::BK;
                for (int kb = w.kb0; kb < w.kb1; ++kb) {
                    if (!wait_fast(bar(EMPTY + s), ph ^ 1u, abort_flag, p.err, p.timeout_ns, true)) {
                        ok = false;
                        break;
                    }
                    if (leader) mbar_arrive_expect_tx(bar(FULL + s), C::CTAS * C::STAGE_BYTES);
                    issue(s, gk, k0, am0, bn0, n0);
                    ++issued;
                    if (++s == C::STAGES) {
                        s = 0;
                        ph ^= 1u;
                    }
                    // next k-block's shard and offset (folded K: shards in turn)
                    if (down) {
                        k0 -= C::BK;
                        if (k0 < 0) {
                            k0 = k_group - C::BK;
                            --gk;
                        }
                    } else {
                        k0 += C::BK;
                        if (k0 == k_group) {
                            k0 = 0;
                            ++gk;
                        }
                    }
                }
            }
            // Drain: no TMA write may still be in flight into either CTA's
            // shared memory when the CTA (pair) leaves. Load j of a CTA went to
            // stage j % STAGES and completes phase j / STAGES of its full
            // barrier; the phases before the last STAGES loads completed before
            // those loads could be issued. In a pair both CTAs' bytes complete
            // on the even CTA's barrier, and after an abort the two CTAs may
            // have issued different numbers of loads, so the odd CTA reports
            // its count and the even CTA settles every phase either of them
            // issued into: it arms the phases only the odd CTA issued (for the
            // odd CTA's bytes) and marks as done the bytes of the phases only
            // it issued, then waits for each phase. The final cluster barrier
            // holds the odd CTA until then.
            uint32_t issued_peer = issued;
            if constexpr (PAIR) {
                if (!leader) {
                    st_cluster_u32(mapa_shared(smem_u32(const_cast<uint32_t*>(peer_issued)), 0u), issued);
                    mbar_arrive_cluster(mapa_shared(bar(XCNT), 0u));   // release: the count
                } else if (wait_bounded(bar(XCNT), 0, abort_flag, p.err, p.timeout_ns + p.drain_ns, false) &&
                           mbar_try_wait_cluster(bar(XCNT), 0)) {
                    issued_peer = *peer_issued;
                }
            }
            if (leader) {
                const uint32_t hi = issued > issued_peer ? issued : issued_peer;
                const uint32_t lo = hi > (uint32_t)C::STAGES ? hi - (uint32_t)C::STAGES : 0u;
                for (uint32_t j = lo; j < hi; ++j) {
                    const int sj = (int)(j % (uint32_t)C::STAGES);
                    if (PAIR && j >= issued) mbar_arrive_expect_tx(bar(FULL + sj), C::STAGE_BYTES);
                    if (PAIR && j >= issued_peer) mbar_complete_tx(bar(FULL + sj), C::STAGE_BYTES);
                    wait_bounded(bar(FULL + sj), (j / (uint32_t)C::STAGES) & 1u, abort_flag, p.err,
                                 p.drain_ns, false);
                }
            }
        }
    } else if (warp == 1) {
        if (lane == 0 && leader) {
            // ---------------- MMA issuer (even CTA of the pair) ----------------
            const uint32_t idesc = instr_desc(C::TILE_M, BN, p.a_mn, p.b_mn);
            // operand descriptors: K-major boxes advance 32 bytes per K=16 step,
            // MN-major boxes advance 16 rows of 128 bytes
            const uint32_t a_lbo = p.a_mn ? C::MN_BOX_BYTES : 16;
            const uint32_t b_lbo = p.b_mn ? C::MN_BOX_BYTES : 16;
            const uint32_t a_kstep = p.a_mn ? UMMA_K * 128 : UMMA_K * 2;
            const uint32_t b_kstep = p.b_mn ? UMMA_K * 128 : UMMA_K * 2;
            // every 4 K steps: the next 64-wide K-major box (MN-major: 16 rows on)
            const uint32_t a_sub = p.a_mn ? 4 * a_kstep : C::A_SUB;
            const uint32_t b_sub = p.b_mn ? 4 * b_kstep : C::B_SUB;
            const uint64_t a_desc0 = smem_desc(sA0, a_lbo, 1024);
            const uint64_t b_desc0 = smem_desc(sB0, b_lbo, 1024);
            int s = 0;
            uint32_t ph = 0;
            int acc = 0;
            uint32_t aph = 0;
            bool ok = p.inject != 2 || wait_bounded(bar(STALL), 0, abort_flag, p.err, p.timeout_ns, true);
            for (Work w(p, first_tile, tile_step, kb_lo, kb_hi, kb_total); ok && w.valid(); w.next()) {
                if (!wait_fast(bar(TEMPTY + acc), aph ^ 1u, abort_flag, p.err, p.timeout_ns, true)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN);
                for (int kb = w.kb0; kb < w.kb1; ++kb) {
                    if (!wait_fast(bar(FULL + s), ph, abort_flag, p.err, p.timeout_ns, true)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    // the start-address field is the low 14 bits (16-byte units): one
                    // add per K step, the rest of the descriptor is fixed
                    const uint64_t ad0 = a_desc0 + (uint64_t)((s * C::A_BYTES) >> 4);
                    const uint64_t bd0 = b_desc0 + (uint64_t)((s * C::B_BYTES) >> 4);
#pragma unroll
                    for (int k = 0; k < C::BK / UMMA_K; ++k) {
                        const uint64_t ad = ad0 + (uint64_t)(((k >> 2) * a_sub + (k & 3) * a_kstep) >> 4);
                        const uint64_t bd = bd0 + (uint64_t)(((k >> 2) * b_sub + (k & 3) * b_kstep) >> 4);
                        const uint32_t accum = ((kb - w.kb0) | k) != 0 ? 1u : 0u;
                        if constexpr (PAIR)
                            tc_mma_f16_pair(d_tmem, ad, bd, idesc, accum);
                        else
                            tc_mma_f16(d_tmem, ad, bd, idesc, accum);
                    }
                    // frees stage s in both CTAs once these MMAs have read it
                    if constexpr (PAIR)
                        tc_commit_pair_multicast(bar(EMPTY + s), 0x3);
                    else
                        tc_commit(bar(EMPTY + s));
                    if (++s == C::STAGES) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
                if (!ok) break;
                if constexpr (PAIR)
                    tc_commit_pair_multicast(bar(TFULL + acc), 0x3);
                else
                    tc_commit(bar(TFULL + acc));
                if (++acc == ACC_BUFS) {
                    acc = 0;
                    aph ^= 1u;
                }
            }
            // every MMA this thread issued has completed before TMEM is freed
            if constexpr (PAIR)
                tc_commit_pair(bar(DRAIN));
            else
                tc_commit(bar(DRAIN));
            wait_bounded(bar(DRAIN), 0, abort_flag, p.err, p.drain_ns, false);
        }
    } else {
        // ---------------- epilogue (warps 2..5 of each CTA) ----------------
        const int quarter = warp & 3;            // TMEM lanes [32*quarter, 32*quarter + 32)
        // the even CTA's TMEM-empty barrier counts the epilogue warps of both CTAs
        const uint32_t tempty0 = PAIR ? mapa_shared(bar(TEMPTY), 0) : bar(TEMPTY);
        int acc = 0;
        uint32_t aph = 0;
        uint32_t rph = 0;   // K split: phase of the exchange barriers
        int live = 1;
        if (p.inject == 1) {
            if (lane == 0) live = wait_bounded(bar(STALL), 0, abort_flag, p.err, p.timeout_ns, true);
            live = __shfl_sync(0xffffffffu, live, 0);
        }
        // Emits one 32-column chunk of the warp's 32 rows (`row` is this
        // lane's, row0 the warp's first). With tensor stores the warp stages
        // the chunk (C, and Z for EPI_ACT) in one of its two buffers and lane
        // 0 writes it with one store per output; a buffer is written again
        // once the stores issued from it two chunks earlier have read it.
        uint32_t oset = 0;
        const uint32_t obuf0 = sOut + (uint32_t)quarter * 2u * (uint32_t)C::OUT_BUF;
        // act' epilogue with staging: each chunk's Z arrives by a tensor load
        // into the Z half of the chunk's staging set (issued one chunk ahead,
        // or at the start of a tile before its accumulator is ready), on one
        // of the warp's two barriers; zpend / zph hold each set's pending
        // load and barrier phase
        const bool zin = C::TMA_OUT && p.tma_out && p.epi.kind == EPI_DACT;
        uint32_t zpend = 0, zph = 0;
        auto zbar = [&](uint32_t set) { return bar(ZLD + 2 * quarter + (int)set); };
        auto zload = [&](uint32_t set, int g, int col0, int row0) {
            if (lane == 0) {
                mbar_arrive_expect_tx(zbar(set), 2048u);
                tma_load_2d(obuf0 + set * (uint32_t)C::OUT_BUF + 2048u, &p.tmAux[g], zbar(set), col0, row0);
            }
            zpend |= 1u << set;
        };
        // next_col0: the next chunk this warp emits for the same rows, or -1
        auto emit = [&](int g, int row, int row0, int col0, const uint32_t (&r)[32], int next_col0) {
            float v[32];
            epilogue_bias(p.epi, g, col0, p.N, r, v);
            const bool z_out = p.epi.kind == EPI_ACT && p.epi.aux[g] != nullptr;
            if (C::TMA_OUT && p.tma_out) {
                const uint32_t buf = obuf0 + oset * (uint32_t)C::OUT_BUF;
                if (zin) {
                    if (!((zpend >> oset) & 1u)) zload(oset, g, col0, row0);
                    if (next_col0 >= 0) zload(oset ^ 1u, g, next_col0, row0);
                }
                if (lane == 0) bulk_wait_read_all_but_one();
                __syncwarp();
                if (z_out) stage_row(buf + 2048u, lane, false, v);   // Z, before the activation
                if (zin) {
                    const uint32_t par = (zph >> oset) & 1u;
                    int okz = 1;
                    if (lane == 0) okz = wait_fast(zbar(oset), par, abort_flag, p.err, p.timeout_ns, true);
                    okz = __shfl_sync(0xffffffffu, okz, 0);
                    if (okz) {
                        mbar_try_wait(zbar(oset), par);   // each lane acquires the completed load
                        zpend &= ~(1u << oset);
                        zph ^= 1u << oset;
                    }
                    float zv[32];
                    load_row_bf16_smem(buf + 2048u, lane, zv);
                    dact_apply(p.epi.act, v, zv);
                } else {
                    epilogue_act(p.epi, g, row, col0, p.M, p.N, v);
                }
                stage_row(buf, lane, p.epi.out_f32 != 0, v);
                fence_proxy_async_smem();   // the staged rows, to the tensor-store proxy
                __syncwarp();
                if (lane == 0) {
                    tma_store_2d(&p.tmC[g], buf, col0, row0);
                    if (z_out) tma_store_2d(&p.tmAux[g], buf + 2048u, col0, row0);
                    bulk_commit();
                }
                oset ^= 1u;
            } else {
                if (z_out) store_z_thread(p.epi, g, row, col0, p.M, p.N, v);
                epilogue_act(p.epi, g, row, col0, p.M, p.N, v);
                store_c_thread(p.epi, g, row, col0, p.M, p.N, v);
            }
        };
        // the next chunk a warp emits after column c of a tile starting at n0
        auto next_of = [&](int n0, int c) { return (c + 32 < BN && n0 + c + 32 < p.N) ? n0 + c + 32 : -1; };
        for (Work w(p, first_tile, tile_step, kb_lo, kb_hi, kb_total); live && w.valid(); w.next()) {
            const int t = w.t;
            int g, m0, n0;
            decode_tile<BN, C::TILE_M>(p, t, g, m0, n0);
            // act' epilogue: the tile's first Z chunk loads while the accumulator fills
            if (zin && !w.partial() && !p.dual && ks == 1 && !((zpend >> oset) & 1u))
                zload(oset, g, n0, m0 + (int)rank * BM + quarter * 32);
            // one lane waits; the warp stays converged for the .sync.aligned TMEM loads
            int ok = 1;
            // (sleeping 1 us between polls: 0.4-1.4% fewer cycles for the GEMM)
            if (lane == 0) ok = wait_sleepy(bar(TFULL + acc), aph, abort_flag, p.err, p.timeout_ns, 1000);
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) break;
            tc_fence_after();
            const int row = m0 + (int)rank * BM + quarter * 32 + lane;
            bool released = false;   // this warp's TEMPTY arrival for the item is done
            const uint32_t tbase =
                tmem_base + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(acc * BN);
            if (ks > 1) {
                // K split. The leader's stage memory is free once its own MMAs
                // are done (TFULL); it tells the peers, each peer stores its
                // partial rows there (slot krank - 1, column groups of 4 x 64
                // rows, 16 bytes per lane and store) and every storing lane
                // arrives on the leader's RFULL with release; the leader's
                // lanes acquire RFULL, add the slots to their own accumulator
                // and run the epilogue.
                const bool xfer = quarter < red_warps;           // warp holds rows < 64
                const uint32_t rrow = (uint32_t)(quarter * 32 + lane);
                const bool has_k = w.kb1 > w.kb0;
                if (krank == 0) {
                    if (warp == 2 && lane == 0)
                        for (int j = 1; j < ks; ++j) mbar_arrive_cluster(mapa_shared(bar(RFREE), (uint32_t)j));
                    int okr = 1;
                    if (xfer) okr = wait_acquire_cluster(bar(RFULL), rph, abort_flag, p.err, p.timeout_ns);
                    if (!__all_sync(0xffffffffu, okr)) break;
                    for (int c = 0; c < BN; c += 32) {
                        if (n0 + c >= p.N) break;
                        uint32_t r[32];
                        __syncwarp();
                        tmem_ld_32cols(tbase + (uint32_t)c, r);
                        tmem_ld_wait();
                        if (!has_k) {
#pragma unroll
                            for (int j = 0; j < 32; ++j) r[j] = 0u;
                        }
                        if (xfer) {
                            for (int j = 0; j < ks - 1; ++j) {
                                const uint32_t slot = sA0 + (uint32_t)(j * C::RED_SLOT_BYTES);
#pragma unroll
                                for (int q = 0; q < 8; ++q) {
                                    const float4 v = ld_shared_v4(
                                        slot + ((uint32_t)(c / 4 + q) * KSPLIT_ROWS + rrow) * 16u);
                                    r[4 * q + 0] = __float_as_uint(__uint_as_float(r[4 * q + 0]) + v.x);
                                    r[4 * q + 1] = __float_as_uint(__uint_as_float(r[4 * q + 1]) + v.y);
                                    r[4 * q + 2] = __float_as_uint(__uint_as_float(r[4 * q + 2]) + v.z);
                                    r[4 * q + 3] = __float_as_uint(__uint_as_float(r[4 * q + 3]) + v.w);
                                }
                            }
                        }
                        emit(g, row, row - lane, n0 + c, r, next_of(n0, c));
                    }
                } else if (xfer) {
                    int okf = 1;
                    if (lane == 0) okf = wait_fast(bar(RFREE), rph, abort_flag, p.err, p.timeout_ns, true);
                    if (!__shfl_sync(0xffffffffu, okf, 0)) break;
                    const uint32_t dst0 =
                        mapa_shared(sA0 + (krank - 1u) * (uint32_t)C::RED_SLOT_BYTES, 0u);
                    for (int c = 0; c < BN; c += 32) {
                        if (n0 + c >= p.N) break;
                        uint32_t r[32];
                        __syncwarp();
                        tmem_ld_32cols(tbase + (uint32_t)c, r);
                        tmem_ld_wait();
                        if (!has_k) {
#pragma unroll
                            for (int j = 0; j < 32; ++j) r[j] = 0u;
                        }
#pragma unroll
                        for (int q = 0; q < 8; ++q)
                            st_cluster_v4(dst0 + ((uint32_t)(c / 4 + q) * KSPLIT_ROWS + rrow) * 16u,
                                          __uint_as_float(r[4 * q + 0]), __uint_as_float(r[4 * q + 1]),
                                          __uint_as_float(r[4 * q + 2]), __uint_as_float(r[4 * q + 3]));
                    }
                    mbar_arrive_cluster(mapa_shared(bar(RFULL), 0u));   // release: this lane's stores
                }
                rph ^= 1u;
            } else if (w.partial()) {
                // Stream-K: this unit accumulated k-blocks [kb0, kb1) of the
                // tile. Each warp holding live rows stores its partial rows in
                // the unit's scratch slot for the tile (one for its first tile,
                // one for its last; per CTA of a pair) and counts itself in on
                // the tile's counter for those rows; the warp that arrives last
                // sums the slots of all units sharing the tile in unit order
                // (the same order whichever warp is last, so the result does
                // not depend on timing) and runs the epilogue. Nothing waits.
                if (quarter < p.sk_rows / 32) {
                    const int P = p.sk_parts;
                    const int64_t U = p.sk_units;
                    const int rrow = quarter * 32 + lane;
                    const int tl = t - p.sk_dp_tiles;   // stream-K tile index
                    // the units c_first .. c_first + n_contrib - 1 share the tile
                    const int c_first = sk_cta_of((int64_t)tl * kb_total, U, P);
                    const int n_contrib = sk_cta_of((int64_t)(tl + 1) * kb_total - 1, U, P) - c_first + 1;
                    auto slot = [&](int k) -> float4* {
                        const int unit = c_first + k;
                        const int which = sk_first_tile(unit, U, P, kb_total) == tl ? 0 : 1;
                        const size_t idx = (size_t)(2 * unit + which) * C::CTAS + rank;
                        return reinterpret_cast<float4*>(p.sk_part + idx * p.sk_rows * BN);
                    };
                    float4* mine = slot(first_tile - c_first);
                    for (int c = 0; c < BN; c += 32) {
                        if (n0 + c >= p.N) break;
                        uint32_t r[32];
                        __syncwarp();
                        tmem_ld_32cols(tbase + (uint32_t)c, r);
                        tmem_ld_wait();
#pragma unroll
                        for (int q = 0; q < 8; ++q)
                            mine[(c / 4 + q) * p.sk_rows + rrow] =
                                make_float4(__uint_as_float(r[4 * q + 0]), __uint_as_float(r[4 * q + 1]),
                                            __uint_as_float(r[4 * q + 2]), __uint_as_float(r[4 * q + 3]));
                    }
                    // the accumulator is read: hand it back to the MMA before
                    // the count and the sum (global memory only from here)
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) {
                        if constexpr (PAIR)
                            mbar_arrive_cluster(tempty0 + 8u * (uint32_t)acc);
                        else
                            mbar_arrive(bar(TEMPTY + acc));
                    }
                    released = true;
                    // release: every lane's partial rows before the count
                    __threadfence();
                    __syncwarp();
                    int last = 0;
                    if (lane == 0) {
                        __threadfence();
                        int* cnt = p.sk_cnt + ((size_t)tl * C::CTAS + rank) * 4 + quarter;
                        last = atomicAdd(cnt, 1) == n_contrib - 1;
                        if (last) __threadfence();   // acquire: the other partials
                    }
                    last = __shfl_sync(0xffffffffu, last, 0);
                    __syncwarp();
                    if (last) {
                        for (int c = 0; c < BN; c += 32) {
                            if (n0 + c >= p.N) break;
                            float v[32];
#pragma unroll
                            for (int j = 0; j < 32; ++j) v[j] = 0.f;
                            // four slots' loads in flight at a time; the sum
                            // still adds the slots in order k = 0, 1, ...
                            int k = 0;
                            for (; k + 4 <= n_contrib; k += 4) {
                                const float4* s0 = slot(k);
                                const float4* s1 = slot(k + 1);
                                const float4* s2 = slot(k + 2);
                                const float4* s3 = slot(k + 3);
#pragma unroll
                                for (int q = 0; q < 8; ++q) {
                                    const int o = (c / 4 + q) * p.sk_rows + rrow;
                                    const float4 x0 = __ldcg(s0 + o), x1 = __ldcg(s1 + o);
                                    const float4 x2 = __ldcg(s2 + o), x3 = __ldcg(s3 + o);
                                    v[4 * q + 0] = (((v[4 * q + 0] + x0.x) + x1.x) + x2.x) + x3.x;
                                    v[4 * q + 1] = (((v[4 * q + 1] + x0.y) + x1.y) + x2.y) + x3.y;
                                    v[4 * q + 2] = (((v[4 * q + 2] + x0.z) + x1.z) + x2.z) + x3.z;
                                    v[4 * q + 3] = (((v[4 * q + 3] + x0.w) + x1.w) + x2.w) + x3.w;
                                }
                            }
                            for (; k < n_contrib; ++k) {
                                const float4* sl = slot(k);
#pragma unroll
                                for (int q = 0; q < 8; ++q) {
                                    const float4 x = __ldcg(sl + (c / 4 + q) * p.sk_rows + rrow);
                                    v[4 * q + 0] += x.x;
                                    v[4 * q + 1] += x.y;
                                    v[4 * q + 2] += x.z;
                                    v[4 * q + 3] += x.w;
                                }
                            }
                            uint32_t r[32];
#pragma unroll
                            for (int j = 0; j < 32; ++j) r[j] = __float_as_uint(v[j]);
                            emit(g, row, row - lane, n0 + c, r, next_of(n0, c));
                        }
                    }
                }
            } else if (!p.dual) {
                for (int c = 0; c < BN; c += 32) {
                    if (n0 + c >= p.N) break;
                    uint32_t r[32];
                    __syncwarp();
                    tmem_ld_32cols(tbase + (uint32_t)c, r);
                    tmem_ld_wait();
                    emit(g, row, row - lane, n0 + c, r, next_of(n0, c));
                }
            } else {
                const int n0o = n0 / 2;
                for (int c = 0; c < BN / 2; c += 32) {
                    if (n0o + c >= p.N) break;
                    uint32_t rg[32], ru[32];
                    __syncwarp();
                    tmem_ld_32cols(tbase + (uint32_t)c, rg);
                    tmem_ld_32cols(tbase + (uint32_t)(BN / 2 + c), ru);
                    tmem_ld_wait();
                    epilogue_swiglu_chunk(p.epi, g, row, n0o + c, p.M, p.N, rg, ru);
                }
            }
            if (!released) {
                tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    if constexpr (PAIR)
                        mbar_arrive_cluster(tempty0 + 8u * (uint32_t)acc);
                    else
                        mbar_arrive(bar(TEMPTY + acc));
                }
            }
            if (++acc == ACC_BUFS) {
                acc = 0;
                aph ^= 1u;
            }
        }
        // every tensor store of this warp has completed (its staging buffers
        // stay valid until then, and the outputs are written when the grid is),
        // and no Z load this warp issued is still in flight
        if (C::TMA_OUT && p.tma_out && lane == 0) {
            bulk_wait_all();
            for (uint32_t set = 0; set < 2; ++set)
                if ((zpend >> set) & 1u)
                    wait_bounded(zbar(set), (zph >> set) & 1u, abort_flag, p.err, p.drain_ns, false);
        }
    }

    __syncwarp();
    tc_fence_before();
    __syncthreads();
    if (clustered) cluster_sync();   // the cluster's MMAs, loads and exchanges are done
    tc_fence_after();
    if (warp == 1) {
        if constexpr (PAIR)
            tmem_dealloc_pair(tmem_base, C::TMEM_COLS);
        else
            tmem_dealloc(tmem_base, C::TMEM_COLS);
    }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    });
    return fn;
}

// Row-major bf16 matrix of `outer` rows x `inner` elements, row pitch `ld`
// elements, read in boxes of box_inner x box_outer with 128-byte swizzle.
bool make_map(CUtensorMap* m, const void* base, int64_t inner, int64_t outer, int64_t ld,
              int box_inner, int box_outer) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {(cuuint64_t)inner, (cuuint64_t)outer};
    cuuint64_t strides[1] = {(cuuint64_t)(ld * 2)};
    cuuint32_t box[2] = {(cuuint32_t)box_inner, (cuuint32_t)box_outer};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides,
                    box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// Output map of the epilogue's tensor stores: `rows` x `cols` elements (bf16,
// or fp32 with f32), row pitch ld elements, boxes of 32 x 32 with the swizzle
// that matches the 64-byte (bf16) or 128-byte (fp32) staged rows.
bool make_map_out(CUtensorMap* m, const void* base, int64_t cols, int64_t rows, int64_t ld,
                  bool f32) {
    auto fn = encode_fn();
    if (!fn) return false;
    const int esz = f32 ? 4 : 2;
    cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)(ld * esz)};
    cuuint32_t box[2] = {32, 32};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(m, f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                    const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    f32 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
                    CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// An MN-major operand ([K rows] x [mn columns], row pitch ld, mn % 64 == 0)
// seen as 64-wide column chunks: dims {64, K, mn/64} with strides {ld*2, 128}
// bytes. A box {64, bk, rows/64} lands in shared memory chunk by chunk, each
// chunk bk rows of 128 bytes: the same layout as rows/64 separate 2-D boxes,
// in one copy.
bool make_map_mn_chunks(CUtensorMap* m, const void* base, int64_t mn, int64_t k, int64_t ld,
                        int rows, int bk) {
    auto fn = encode_fn();
    if (!fn || mn % BOX_MN != 0) return false;
    cuuint64_t dims[3] = {(cuuint64_t)BOX_MN, (cuuint64_t)k, (cuuint64_t)(mn / BOX_MN)};
    cuuint64_t strides[2] = {(cuuint64_t)(ld * 2), (cuuint64_t)(BOX_MN * 2)};
    cuuint32_t box[3] = {(cuuint32_t)BOX_MN, (cuuint32_t)bk, (cuuint32_t)(rows / BOX_MN)};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides,
                    box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// Co-resident CTAs (cl = 1) or clusters of cl CTAs of one kernel instance on
// the current device; 0 when the queries fail. Cached per device and cl.
template <int BN, bool PAIR>
int resident_units(int cl) {
    using C = Cfg<BN, PAIR>;
    static int units[64][9] = {};
    static bool attr_set[64] = {};
    static std::mutex mu;   // first calls may come from several host threads
    std::lock_guard<std::mutex> lock(mu);
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64 || cl < 1 || cl > 8) return 0;
    if (units[dev][cl] > 0) return units[dev][cl];
    if (!attr_set[dev]) {
        if (cudaFuncSetAttribute(tc_gemm_kernel<BN, PAIR>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 C::SMEM_BYTES) != cudaSuccess)
            return 0;
        attr_set[dev] = true;
    }
    int n = device_sm_count();
    if (cl > 1) {
        cudaLaunchConfig_t cfg = {};
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = (unsigned)cl;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        cfg.blockDim = dim3(NUM_THREADS);
        cfg.dynamicSmemBytes = C::SMEM_BYTES;
        cfg.gridDim = dim3((unsigned)(cl * (n / cl)));
        n = 0;
        if (cudaOccupancyMaxActiveClusters(&n, tc_gemm_kernel<BN, PAIR>, &cfg) != cudaSuccess) return 0;
    }
    units[dev][cl] = n > 0 ? n : 0;
    return units[dev][cl];
}

// The stream-K form of a launch with BN-column tiles (PAIR: CTA-pair tiles).
// Few-token GEMMs (M <= KSPLIT_ROWS, single CTAs): every (tile, k-block) unit
// is dealt out, to every co-resident CTA (at most kSkMaxCtas, at most one per
// unit). Other GEMMs: the tiles of the full waves run whole, one per unit (CTA
// or pair) at a time, and each of the r remaining tiles (the part wave) is cut
// into s = units / r equal K chunks run by r s units side by side. Chunk c of
// every remaining tile runs at the same K offsets at the same time, so the
// tiles sharing an operand panel read it together, as whole tiles do (a
// contiguous deal of the k-blocks puts every unit at a different K offset:
// measured slower, the part wave then streams its operands from HBM). `ok`
// is false when the form does not apply (dual B, no scratch, no part wave,
// fewer than two chunks) or the scratch is too small.
struct SkShape {
    int units = 0;          // CTAs, or CTA pairs
    int parts = 0;          // units taking part in the stream-K phase
    int dp_tiles = 0;       // tiles run whole before the stream-K phase
    int64_t sk_units = 0;   // k-block units of the stream-K phase
    int64_t sk_tiles = 0;   // tiles of the stream-K phase
    int rows = 0;           // rows per CTA of a partial slot
    bool ok = false;
};

template <int BN, bool PAIR>
SkShape sk_shape(const GemmProblem& pr, int64_t tiles, int64_t kb_total) {
    SkShape r;
    if (pr.sk_part == nullptr || pr.sk_cnt == nullptr || pr.dual) return r;
    if (pr.M <= KSPLIT_ROWS) {
        if (PAIR) return r;
        int64_t P = resident_units<BN, false>(1);
        const int64_t U = tiles * kb_total;
        if (P > kSkMaxCtas) P = kSkMaxCtas;
        if (P > U) P = U;
        r.units = (int)P;
        r.parts = (int)P;
        r.sk_units = U;
        r.sk_tiles = tiles;
        r.rows = 32 * ((pr.M + 31) / 32);
    } else {
        const int64_t P = resident_units<BN, PAIR>(PAIR ? 2 : 1);
        if (P < 1 || tiles % P == 0) return r;
        r.units = (int)P;
        r.sk_tiles = tiles % P;
        int64_t chunks = P / r.sk_tiles;
        if (chunks > kb_total) chunks = kb_total;
        if (chunks < 2) return SkShape();
        r.parts = (int)(r.sk_tiles * chunks);
        r.dp_tiles = (int)(tiles - r.sk_tiles);
        r.sk_units = r.sk_tiles * kb_total;
        r.rows = BM;
    }
    const int ctas = PAIR ? 2 : 1;
    // every unit gets at least one k-block: the CTAs sharing a tile are then
    // consecutive units, which the partial sums count on
    if (r.units < 1 || r.parts < 1 || r.sk_units < r.parts || r.sk_units > 0x7fffffff ||
        r.sk_tiles * 4 * ctas > pr.sk_cnt_cap ||
        (size_t)r.parts * 2 * ctas * r.rows * BN * 4 > pr.sk_part_bytes)
        return SkShape();
    r.ok = true;
    return r;
}

// ks > 1: split each tile's K range across a cluster of ks CTAs (single-CTA
// tiles, M <= KSPLIT_ROWS, no dual B; one tile per cluster).
// ks == 0: stream-K (see sk_shape; no dual B): k-blocks are dealt out evenly
// to all units and tiles split between
// CTAs are summed through the problem's scratch.
template <int BN, bool PAIR>
tpmlp_status launch(const GemmProblem& pr, cudaStream_t s, int ks = 1) {
    using C = Cfg<BN, PAIR>;
    static TcParams kp;   // large; filled per call under the lock below
    static std::mutex mu;
    std::lock_guard<std::mutex> lock(mu);
    memset(&kp, 0, sizeof(kp));
    const int G = pr.G;
    // MN-major operands whose MN extent is a multiple of 64 use one 3-D box per
    // stage; if the driver refuses that map, the 2-D boxes are used instead
    // B rows staged per map: half the tile's N for a dual GEMM
    const int b_rows = pr.dual ? BN / 2 : C::B_ROWS;
    kp.a_3d = pr.a_mn && pr.M % BOX_MN == 0;
    kp.b_3d = pr.b_mn && pr.N % BOX_MN == 0;
    for (int g = 0; g < G && kp.a_3d; ++g)
        kp.a_3d = make_map_mn_chunks(&kp.tmA[g], pr.A[g], pr.M, pr.K, pr.lda, BM, C::BK);
    for (int g = 0; g < G && kp.b_3d; ++g) {
        kp.b_3d = make_map_mn_chunks(&kp.tmB[g], pr.B[g], pr.N, pr.K, pr.ldb, b_rows, C::BK);
        if (kp.b_3d && pr.dual)
            kp.b_3d = make_map_mn_chunks(&kp.tmB2[g], pr.B2[g], pr.N, pr.K, pr.ldb, b_rows, C::BK);
    }
    for (int g = 0; g < G; ++g) {
        bool ok = true;
        if (!pr.a_mn)
            ok = make_map(&kp.tmA[g], pr.A[g], pr.K, pr.M, pr.lda, BKB, BM);
        else if (!kp.a_3d)
            ok = make_map(&kp.tmA[g], pr.A[g], pr.M, pr.K, pr.lda, BOX_MN, C::BK);
        for (int d = 0; d < (pr.dual ? 2 : 1); ++d) {
            CUtensorMap* m = d == 0 ? &kp.tmB[g] : &kp.tmB2[g];
            const void* b = d == 0 ? pr.B[g] : pr.B2[g];
            if (!pr.b_mn)
                ok = ok && make_map(m, b, pr.K, pr.N, pr.ldb, BKB, b_rows);
            else if (!kp.b_3d)
                ok = ok && make_map(m, b, pr.N, pr.K, pr.ldb, BOX_MN, C::BK);
        }
        if (!ok) return TPMLP_ERR_CUDA;
    }
    kp.M = pr.M;
    kp.N = pr.N;
    kp.K = pr.K;
    kp.G = G;
    kp.fold = pr.fold;
    kp.a_mn = pr.a_mn;
    kp.b_mn = pr.b_mn;
    kp.m_tiles = (pr.M + C::TILE_M - 1) / C::TILE_M;
    kp.dual = pr.dual;
    kp.n_tiles = pr.dual ? (pr.N + BN / 2 - 1) / (BN / 2) : (pr.N + BN - 1) / BN;
    kp.k_blocks = (pr.K + C::BK - 1) / C::BK;
    kp.num_tiles = (pr.fold ? 1 : G) * kp.m_tiles * kp.n_tiles;
    {
        bool shared_a = !pr.fold && G > 1, shared_b = !pr.fold && G > 1;
        for (int g = 1; g < G; ++g) {
            shared_a = shared_a && pr.A[g] == pr.A[0];
            shared_b = shared_b && pr.B[g] == pr.B[0];
        }
        // bands of 12 tiles: with the alternating orders a sweep of 4..24 on
        // the fwd+bwd GEMMs read the least from DRAM at 12 (the folded ones
        // 9% less than at 8, the rest equal) and ran the step as fast as any
        kp.raster = shared_a ? 1 : (shared_b ? 2 : 0);
        kp.band = GROUP_M;
    }
    const bool sk = ks == 0;
    if (sk) ks = 1;
    kp.ksplit = ks;
    if (ks > 1 && (PAIR || pr.dual || pr.M > KSPLIT_ROWS || ks > C::MAX_KSPLIT || ks > 8 ||
                   ks > (pr.fold ? G : 1) * kp.k_blocks))
        return TPMLP_ERR_SHAPE;
    int sk_grid = 0;
    size_t sk_cnt_bytes = 0;
    if (sk) {
        const SkShape sh = sk_shape<BN, PAIR>(pr, kp.num_tiles, (int64_t)(pr.fold ? G : 1) * kp.k_blocks);
        if (!sh.ok) return TPMLP_ERR_SHAPE;
        sk_grid = sh.units;
        kp.sk = 1;
        kp.sk_dp_tiles = sh.dp_tiles;
        kp.sk_units = (int)sh.sk_units;
        kp.sk_parts = sh.parts;
        kp.sk_rows = sh.rows;
        kp.sk_part = pr.sk_part;
        kp.sk_cnt = pr.sk_cnt;
        sk_cnt_bytes = (size_t)sh.sk_tiles * 4 * C::CTAS * sizeof(int);
    }
    kp.epi = pr.epi;
    // alternating orders for the tiles of more than one wave; the few-token
    // forms stream each operand once and keep the plain order
    kp.alt = pr.M > KSPLIT_ROWS && alternate_orders() ? 3 : 0;
    // the epilogue writes through staging and tensor stores where the tile
    // configuration has room for the staging and every output has a map (not
    // the gated epilogue, nor the reduce-scatter's row blocks)
    kp.tma_out = 0;
    if (C::TMA_OUT && !pr.dual && pr.epi.kind != EPI_SWIGLU && pr.epi.row_shard == 0) {
        bool ok = true;
        for (int g = 0; g < (pr.fold ? 1 : G) && ok; ++g) {
            ok = make_map_out(&kp.tmC[g], pr.epi.C[g], pr.N, pr.M, pr.epi.ldc, pr.epi.out_f32 != 0);
            if (ok && (pr.epi.kind == EPI_ACT || pr.epi.kind == EPI_DACT) && pr.epi.aux[g] != nullptr)
                ok = make_map_out(&kp.tmAux[g], pr.epi.aux[g], pr.N, pr.M, pr.epi.ldaux, false);
        }
        kp.tma_out = ok ? 1 : 0;
    }
    kp.err = device_error_word();
    kp.timeout_ns = wait_timeout_ns();
    // copies and MMAs already issued complete in microseconds; their waits
    // get at least 100 ms whatever the limit for waiting on other roles
    kp.drain_ns = kp.timeout_ns > 100000000ull ? kp.timeout_ns : 100000000ull;
    kp.inject = gemm_stall_role();
    if (kp.err == nullptr) return TPMLP_ERR_CUDA;

    const int cl = PAIR ? 2 : ks;   // CTAs per cluster
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[2];
    cfg.blockDim = dim3(NUM_THREADS);
    cfg.dynamicSmemBytes = C::SMEM_BYTES;
    cfg.stream = s;
    cfg.attrs = attr;
    // programmatic dependent launch: the kernel may start while the previous
    // kernel on the stream finishes (it waits for it before using its data)
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = pdl_enabled() ? 1 : 0;
    cfg.numAttrs = 1;
    if (cl > 1) {
        attr[1].id = cudaLaunchAttributeClusterDimension;
        attr[1].val.clusterDim.x = (unsigned)cl;
        attr[1].val.clusterDim.y = 1;
        attr[1].val.clusterDim.z = 1;
        cfg.numAttrs = 2;
    }
    const int max_units = resident_units<BN, PAIR>(PAIR ? 2 : 1);
    if (max_units < 1) return TPMLP_ERR_CUDA;
    // persistent units, one cluster per tile when K is split, or the
    // stream-K CTAs
    const int units = sk ? sk_grid
                         : ks > 1 ? kp.num_tiles
                                  : (kp.num_tiles < max_units ? kp.num_tiles : max_units);
    cfg.gridDim = dim3((unsigned)(units * cl));
    cudaError_t e;
    {
        LaunchScope ls(pr.name, s);
        // the arrival counters start at zero (a memset node inside a graph)
        e = sk ? cudaMemsetAsync(pr.sk_cnt, 0, sk_cnt_bytes, s) : cudaSuccess;
        if (e == cudaSuccess) e = cudaLaunchKernelEx(&cfg, tc_gemm_kernel<BN, PAIR>, kp);
    }
    if (e != cudaSuccess) return TPMLP_ERR_CUDA;
    return cudaGetLastError() == cudaSuccess ? TPMLP_OK : TPMLP_ERR_CUDA;
}

}  // namespace

namespace {

struct Plan {
    int bn;
    bool pair;
    int ks;
    bool ok;
};

Plan choose_plan(const GemmProblem& pr) {
    // Tile choice by estimated time.
    // M > 64 (tensor-bound): waves x per-tile MMA work over the relative rate
    // measured for the tile shape; a wave is one tile per CTA or CTA pair.
    // M <= 64 (weight streaming, HBM-bound): a wave of n CTAs that each
    // stream b weight bytes takes max(n b / kHbm, b / r_cta): together they
    // cannot beat HBM, and one CTA cannot stream faster than r_cta, so a
    // wave of few CTAs leaves HBM idle (fitted on the N = 16, D = 12288,
    // F = 24576 and 49152, T = 8 forward; every GEMM there within 6% of it).
    // Candidates: whole tiles on persistent CTAs; for folded GEMMs a K split
    // across a cluster of ks CTAs (one tile per cluster, a start per wave:
    // on grouped GEMMs, which have T times the tiles, it measured slower);
    // with the scratch, stream-K, whose CTAs read unrelated K ranges and
    // reach kSkEff of the HBM rate of whole tiles started together on the
    // same weight rows. For M > 64 stream-K cuts only the part wave's tiles
    // into K chunks (the full waves run whole tiles): its cost is the full
    // waves plus one chunk and a pipeline fill of kSkFillKb k-blocks, at
    // kSkSlow of the whole-tile rate (partial-row stores and sums).
    struct Cand {
        int bn;
        bool pair;
        int ks;
        double rate;
    };
    // ks = 0: stream-K (with the scratch)
    // 192-column tiles only stream weights (M <= 64): 64 of them cover the
    // N = 12288 row GEMM, which a 2-CTA K split then runs on 128 SMs
    const Cand cands[] = {{256, true, 1, 1.08}, {256, false, 1, 1.0}, {128, false, 1, 0.85},
                          {256, true, 0, 1.08},  {256, false, 0, 1.0},  {128, false, 0, 0.85},
                          {256, false, 2, 1.0},  {256, false, 3, 1.0}, {256, false, 4, 1.0},
                          {128, false, 2, 0.85}, {128, false, 3, 0.85}, {128, false, 4, 0.85},
                          {192, false, 1, 0.95}, {192, false, 0, 0.95}, {192, false, 2, 0.95},
                          {192, false, 3, 0.95}, {192, false, 4, 0.95}};
    const int ncand = (int)(sizeof(cands) / sizeof(cands[0]));
    const int groups = pr.fold ? 1 : pr.G;
    const int64_t kb_total = (int64_t)(pr.fold ? pr.G : 1) * ((pr.K + BKB - 1) / BKB);
    constexpr double kHbm = 6.6e12;     // B/s
    constexpr double kSkEff = 0.87;
    constexpr double kStart = 5e-6;     // s: launch, set-up and pipeline fill
    constexpr double kSkFix = 2e-6;     // s: counter reset and partial-tile sums
    constexpr double kSkFillKb = 4.0;   // M > 64: pipeline fill of a stream-K item, k-blocks
    constexpr double kSkSlow = 1.05;
    double best = 1e300;
    int pick = 1;
    for (int i = 0; i < ncand; ++i) {
        const Cand& c = cands[i];
        if (c.pair && pr.M <= 128) continue;   // a pair covers 256 rows
        if (c.bn == 192 && (pr.M > KSPLIT_ROWS || pr.dual)) continue;
        if (c.ks > 1 && (!pr.fold || pr.M > KSPLIT_ROWS || pr.dual || c.ks > kb_total)) continue;
        const int64_t tile_m = c.pair ? 256 : 128;
        const int64_t n_out = pr.dual ? c.bn / 2 : c.bn;   // outputs per tile along N
        const int64_t tiles = (int64_t)groups * ((pr.M + tile_m - 1) / tile_m) *
                              ((pr.N + n_out - 1) / n_out);
        // one CTA's streaming rate with BN-column tiles, and the weight bytes
        // of a tile (all its k-blocks of BN columns, both halves if dual)
        const double r_cta = c.bn == 128 ? 54e9 : c.bn == 192 ? 60e9 : 66e9;
        const double tile_bytes = (double)c.bn * (double)kb_total * BKB * 2.0;
        auto wave = [&](double ctas, double bytes) {
            const double hbm = ctas * bytes / kHbm, one = bytes / r_cta;
            return hbm > one ? hbm : one;
        };
        double cost;
        if (c.ks == 0) {
            // the candidate's own k-block depth (128 for a pair, else 64)
            const int64_t kbt = c.pair ? (int64_t)(pr.fold ? pr.G : 1) * ((pr.K + 2 * BKB - 1) / (2 * BKB))
                                       : kb_total;
            const SkShape sh = c.pair ? sk_shape<256, true>(pr, tiles, kbt)
                               : c.bn == 128 ? sk_shape<128, false>(pr, tiles, kbt)
                               : c.bn == 192 ? sk_shape<192, false>(pr, tiles, kbt)
                                             : sk_shape<256, false>(pr, tiles, kbt);
            if (!sh.ok) continue;
            if (pr.M > KSPLIT_ROWS) {
                // full waves, then one K chunk of a part-wave tile per unit
                const double part = ((double)sh.sk_units / sh.parts + kSkFillKb) / (double)kbt * kSkSlow;
                cost = ((double)(tiles / sh.units) + part) * 128.0 * c.bn / c.rate;
            } else {
                const int64_t P = sh.units;
                const double b = (double)((sh.sk_units + P - 1) / P) * c.bn * BKB * 2.0;
                const double hbm = (double)P * b / (kHbm * kSkEff), one = b / r_cta;
                cost = kStart + kSkFix + (hbm > one ? hbm : one);
            }
        } else {
            int64_t units = 0;
            if (c.bn == 128) units = resident_units<128, false>(c.ks);
            else if (c.bn == 192) units = resident_units<192, false>(c.ks);
            else if (c.pair) units = resident_units<256, true>(2);
            else units = resident_units<256, false>(c.ks);
            if (units < 1) continue;
            const int64_t full = tiles / units, rem = tiles % units;
            if (pr.M > 64) {
                cost = (double)(full + (rem ? 1 : 0)) * 128.0 * c.bn / c.rate;
            } else if (c.ks == 1) {
                cost = kStart + (double)full * wave((double)units, tile_bytes) +
                       (rem ? wave((double)rem, tile_bytes) : 0.0);
            } else {
                const double per_cta = tile_bytes / c.ks;
                cost = (double)full * (kStart + wave((double)(units * c.ks), per_cta)) +
                       (rem ? kStart + wave((double)(rem * c.ks), per_cta) : 0.0);
            }
        }
        if (cost < best) {
            best = cost;
            pick = i;
        }
    }
    return Plan{cands[pick].bn, cands[pick].pair, cands[pick].ks, best < 1e299};
}

}  // namespace

tpmlp_status plan_gemm_tc(const GemmProblem& pr, int* bn, int* mma_ctas, int* ksplit) {
    if (pr.M <= 0 || pr.N <= 0 || pr.K <= 0 || pr.G < 1 || pr.G > kMaxG) return TPMLP_ERR_SHAPE;
    const Plan c = choose_plan(pr);
    if (!c.ok) return TPMLP_ERR_CUDA;
    *bn = c.bn;
    *mma_ctas = c.pair ? 2 : 1;
    *ksplit = c.ks;
    return TPMLP_OK;
}

tpmlp_status run_gemm_tc(const GemmProblem& pr, cudaStream_t s) {
    if (pr.M <= 0 || pr.N <= 0) return TPMLP_OK;
    if (pr.K <= 0 || pr.G < 1 || pr.G > kMaxG) return TPMLP_ERR_SHAPE;
    const Plan c = choose_plan(pr);
    if (!c.ok) return TPMLP_ERR_CUDA;
    if (c.bn == 128) return launch<128, false>(pr, s, c.ks);
    if (c.bn == 192) return launch<192, false>(pr, s, c.ks);
    if (c.pair) return launch<256, true>(pr, s, c.ks);
    return launch<256, false>(pr, s, c.ks);
}

}  // namespace tpmlp
