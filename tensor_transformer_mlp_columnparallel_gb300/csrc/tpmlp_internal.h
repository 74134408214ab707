// Host-side interfaces shared by the library's translation units (not part of
// the public C-ABI in include/tpmlp.h).
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <cstdint>

#include "tpmlp.h"

namespace tpmlp {

constexpr int kMaxG = TPMLP_MAX_SHARDS;

// What the GEMM epilogue does with each fp32 accumulator value v at (m, n):
//   EPI_STORE: C = v (+ bias[n])
//   EPI_ACT:   z = v (+ bias[n]); aux = z (if aux != NULL); C = act(z)
//   EPI_DACT:  C = v * act'(aux[m, n])
//   EPI_SWIGLU (dual GEMMs): g, u = the two accumulators at (m, n);
//              aux = g, aux2 = u (each if not NULL); C = SiLU(g) * u
enum EpiKind { EPI_STORE = 0, EPI_ACT = 1, EPI_DACT = 2, EPI_SWIGLU = 3 };

struct EpiArgs {
    int kind;
    int act;                   // tpmlp_act
    int out_f32;               // 1: C is fp32; 0: C has the compute element type
    int64_t ldc;               // row pitch of C, elements
    int64_t ldaux;             // row pitch of aux, elements
    void* C[kMaxG];            // per group (FOLD: group 0 only)
    const void* bias[kMaxG];   // per output column, compute element type; NULL: none
    void* aux[kMaxG];          // Z (compute element type), see EpiKind
    void* aux2[kMaxG];         // U of EPI_SWIGLU
    // > 0: C is split by rows into blocks of row_shard rows, block i at C[i]
    // (the reduce-scatter output of the block end); 0: C[g] as above
    int64_t row_shard;
};

// A batch of G GEMMs of identical shape, C_g[M, N] = A_g[M, K] B_g[K, N], or,
// with fold = 1, ONE output C[M, N] = sum_g A_g B_g whose K loop runs over
// (g, k) in order g = 0..G-1.
// Operand addressing (elements):
//   A(m, k) = a_mn ? A[g][k * lda + m] : A[g][m * lda + k]
//   B(k, n) = b_mn ? B[g][k * ldb + n] : B[g][n * ldb + k]
// ("K-major" = the K index is contiguous; "MN-major" = M or N is contiguous.)
struct GemmProblem {
    int M, N, K;
    int G;
    int fold;
    const void* A[kMaxG];
    int64_t lda;
    int a_mn;
    const void* B[kMaxG];
    int64_t ldb;
    int b_mn;
    // dual = 1: a second B (B2, same layout as B) and two products per output,
    // A B and A B2, for the gated MLP's gate and up projections
    int dual;
    const void* B2[kMaxG];
    EpiArgs epi;
    const char* name;          // kernel kind, for the timing records
    // Scratch for work-balanced few-token GEMMs (stream-K, M <= 64): partial
    // accumulator slots and per-tile arrival counters; NULL = not available.
    float* sk_part;
    size_t sk_part_bytes;
    int* sk_cnt;
    int64_t sk_cnt_cap;        // counters available
};

// Stream-K scratch: at most this many CTAs share the (tile, k-block) units,
// each with two slots of up to 64 rows x kSkMaxBn fp32 accumulators, and two
// counters per tile (one per 32-row warp).
constexpr int kSkMaxCtas = 256;
constexpr int kSkMaxBn = 256;

// bf16 inputs on tcgen05 tensor cores (TMA + mbarrier pipeline + TMEM).
tpmlp_status run_gemm_tc(const GemmProblem& p, cudaStream_t s);
// The tile configuration run_gemm_tc launches for p (accumulator columns,
// CTAs per MMA, K-split cluster size); nothing is launched.
tpmlp_status plan_gemm_tc(const GemmProblem& p, int* bn, int* mma_ctas, int* ksplit);
// fp32 inputs on CUDA cores (exact fp32 FMA, no TF32).
tpmlp_status run_gemm_simt(const GemmProblem& p, cudaStream_t s);

// Y = sum_r P[r] + bias, fp32 sum in shard order, output fp32 or bf16. With
// Y_rows != NULL the result is scattered by rows: rows [i*N/T, (i+1)*N/T) to
// Y_rows[i] (reduce-scatter); otherwise it goes to Y.
tpmlp_status run_block_reduce(int out_f32, int64_t N, int64_t D, int T, const float* const* P,
                              const void* bias, void* Y, cudaStream_t s, const char* name,
                              void* const* Y_rows = nullptr);
tpmlp_status run_vocab_embedding(int f32, int64_t N, int64_t V, int64_t H, int T,
                                 const int64_t* ids, const void* const* table, void* out,
                                 cudaStream_t s);
// out_g[c] = sum_r in_g[r * ld_g + c], c < cols_g, for G <= kMaxColsumG groups
// of `rows` rows each (bias gradients: the T dZ shards and dY). With fp32
// scratch space (scratch_bytes, 16-byte aligned; bf16 only) the sums stream
// whole rows in two passes through it, else one pass per column strip.
constexpr int kMaxColsumG = kMaxG + 1;
tpmlp_status run_colsum(int f32, int64_t rows, int G, const int64_t* cols, const int64_t* ld,
                        const void* const* in, void* const* out, cudaStream_t s,
                        float* scratch = nullptr, size_t scratch_bytes = 0);
tpmlp_status run_vocab_ce(int64_t N, int64_t V, int T, const float* logits,
                          const int64_t* targets, float* loss, float* loss_mean, int32_t* argmax,
                          int32_t* owner, cudaStream_t s);
tpmlp_status run_vocab_ce_backward(int64_t N, int64_t V, const float* logits,
                                   const int64_t* targets, const float* loss, float grad_scale,
                                   float* dlogits, cudaStream_t s);
tpmlp_status run_selftest_wait(uint64_t timeout_ns, cudaStream_t s);

// ---- services of the API translation unit --------------------------------
int* device_error_word();          // per current device; NULL on failure
uint64_t wait_timeout_ns();
int gemm_stall_role();             // failure-detection self test of the GEMM (0: off)
bool pdl_enabled();                // programmatic dependent launch (TPMLP_PDL != 0)
bool alternate_orders();           // odd waves walk K down, odd bands their tiles back (TPMLP_ALT_ORDER != 0)
int device_sm_count();

// Counts the launch and, when timing is on, brackets it with CUDA events
// recorded on the launch stream.
class LaunchScope {
  public:
    LaunchScope(const char* name, cudaStream_t s);
    ~LaunchScope();

  private:
    const char* name_;
    cudaStream_t s_;
    cudaEvent_t start_;
    cudaEvent_t stop_;
};

}  // namespace tpmlp
