// The C-ABI of include/tpmlp.h: argument checks, workspace layout, and the
// order in which the steps of the block run on the caller's stream.
//
// Forward (page "一层 MLP 太宽而放不下时怎样切？", §02-§05), T logical shards:
//   1. column GEMM, all shards in one grouped launch:
//        Z^(r) = X W1^(r) + b1^(r), H^(r) = act(Z^(r))       (fused epilogue)
//   2a. PARTIALS: row GEMM P^(r) = H^(r) W2^(r) into T fp32 buffers, then
//       block_reduce Y = sum_r P^(r) + b2                       (b2 once)
//   2b. SPLITK:   row GEMM with the shard sum in the K loop, Y = acc + b2
// Backward (§06):
//   1. dZ^(r) = (dY W2^(r)^T) * act'(Z^(r))                     (fused epilogue)
//   2. dW2^(r) = H^(r)^T dY;  3. dW1^(r) = X^T dZ^(r)
//   4. dX = sum_r dZ^(r) W1^(r)^T   (PARTIALS + block_reduce, or SPLITK)
//   5. db1^(r) = sum_n dZ^(r), db2 = sum_n dY                   (if requested)
#include <cuda_runtime.h>

#include <atomic>
#include <cstdlib>
#include <cstring>
#include <map>
#include <mutex>
#include <string>
#include <vector>

#include "tpmlp_internal.h"

namespace tpmlp {

// ---------------------------------------------------------------------------
// per-device services
// ---------------------------------------------------------------------------

__device__ int g_device_error;   // TPMLP_OK, or the first error a kernel recorded

namespace {
constexpr int kMaxDevices = 64;
std::mutex g_dev_mu;
int* g_err_ptr[kMaxDevices] = {};
int g_sms[kMaxDevices] = {};
std::atomic<uint64_t> g_timeout_ns{2000000000ull};
std::atomic<int> g_gemm_stall{0};
std::atomic<int64_t> g_launches{0};

int current_device() {
    int d = 0;
    if (cudaGetDevice(&d) != cudaSuccess) return -1;
    return d;
}
}  // namespace

int* device_error_word() {
    const int d = current_device();
    if (d < 0 || d >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lk(g_dev_mu);
    if (g_err_ptr[d] == nullptr) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_device_error) != cudaSuccess) return nullptr;
        g_err_ptr[d] = static_cast<int*>(p);
    }
    return g_err_ptr[d];
}

uint64_t wait_timeout_ns() { return g_timeout_ns.load(); }

int gemm_stall_role() { return g_gemm_stall.load(); }

bool pdl_enabled() {
    // TPMLP_PDL=0 in the environment launches every kernel fully serialized
    // after the previous one (for A/B timing, or tools that need it)
    static const bool on = [] {
        const char* v = getenv("TPMLP_PDL");
        return v == nullptr || strcmp(v, "0") != 0;
    }();
    return on;
}

bool alternate_orders() {
    // TPMLP_ALT_ORDER=0 in the environment keeps every GEMM's tiles and K
    // loops in plain ascending order (for A/B timing and traffic counts)
    static const bool on = [] {
        const char* v = getenv("TPMLP_ALT_ORDER");
        return v == nullptr || strcmp(v, "0") != 0;
    }();
    return on;
}

int device_sm_count() {
    const int d = current_device();
    if (d < 0 || d >= kMaxDevices) return 1;
    std::lock_guard<std::mutex> lk(g_dev_mu);
    if (g_sms[d] == 0) {
        int n = 0;
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, d);
        g_sms[d] = n > 0 ? n : 1;
    }
    return g_sms[d];
}

// ---------------------------------------------------------------------------
// launch counting and event timing
// ---------------------------------------------------------------------------

namespace {
struct TimingRec {
    std::string name;
    cudaEvent_t start, stop;
};
struct TimingAgg {
    int64_t launches = 0;
    double ms = 0.0;
};
std::mutex g_t_mu;
bool g_timing = false;
std::vector<TimingRec> g_pending;
std::vector<cudaEvent_t> g_event_pool;
std::map<std::string, TimingAgg> g_agg;

cudaEvent_t take_event() {
    if (!g_event_pool.empty()) {
        cudaEvent_t e = g_event_pool.back();
        g_event_pool.pop_back();
        return e;
    }
    cudaEvent_t e = nullptr;
    if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
    return e;
}
}  // namespace

LaunchScope::LaunchScope(const char* name, cudaStream_t s)
    : name_(name ? name : "?"), s_(s), start_(nullptr), stop_(nullptr) {
    g_launches.fetch_add(1);
    std::lock_guard<std::mutex> lk(g_t_mu);
    if (!g_timing) return;
    start_ = take_event();
    stop_ = take_event();
    if (start_ == nullptr || stop_ == nullptr) {
        start_ = stop_ = nullptr;
        return;
    }
    cudaEventRecord(start_, s_);
}

LaunchScope::~LaunchScope() {
    if (start_ == nullptr) return;
    std::lock_guard<std::mutex> lk(g_t_mu);
    cudaEventRecord(stop_, s_);
    g_pending.push_back(TimingRec{name_, start_, stop_});
}

// ---------------------------------------------------------------------------
// argument checks
// ---------------------------------------------------------------------------

namespace {

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline size_t round256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

tpmlp_status check_dims(tpmlp_dtype dt, int64_t N, int64_t D, int64_t F, int T, tpmlp_act act) {
    if (dt != TPMLP_F32 && dt != TPMLP_BF16) return TPMLP_ERR_DTYPE;
    if (act != TPMLP_ACT_RELU && act != TPMLP_ACT_GELU_TANH && act != TPMLP_ACT_GELU_ERF &&
        act != TPMLP_ACT_GELU_SIGMOID)
        return TPMLP_ERR_ARG;
    if (N < 0) return TPMLP_ERR_ARG;
    if (D <= 0 || F <= 0 || T < 1 || T > TPMLP_MAX_SHARDS) return TPMLP_ERR_SHAPE;
    if (F % T != 0) return TPMLP_ERR_SHAPE;
    if (N > 0x7fffffffLL || D > 0x7fffffffLL || F > 0x7fffffffLL) return TPMLP_ERR_SHAPE;
    if (dt == TPMLP_BF16 && (D % 8 != 0 || (F / T) % 8 != 0)) return TPMLP_ERR_ALIGN;
    return TPMLP_OK;
}

// every entry of a shard-pointer array present (and 16-byte aligned on the bf16 path)
tpmlp_status check_shards(const void* const* a, int T, bool bf16) {
    if (a == nullptr) return TPMLP_ERR_ARG;
    for (int r = 0; r < T; ++r) {
        if (a[r] == nullptr) return TPMLP_ERR_ARG;
        if (bf16 && !aligned16(a[r])) return TPMLP_ERR_ALIGN;
    }
    return TPMLP_OK;
}

tpmlp_status check_ptr(const void* p, bool bf16) {
    if (p == nullptr) return TPMLP_ERR_ARG;
    if (bf16 && !aligned16(p)) return TPMLP_ERR_ALIGN;
    return TPMLP_OK;
}

#define TPMLP_TRY(expr)                      \
    do {                                     \
        const tpmlp_status _s = (expr);      \
        if (_s != TPMLP_OK) return _s;       \
    } while (0)

size_t partials_bytes(int64_t N, int64_t D, int T) { return (size_t)T * round256((size_t)N * D * 4); }
size_t dz_bytes(tpmlp_dtype dt, int64_t N, int64_t Fs, int T) {
    return (size_t)T * round256((size_t)N * Fs * (dt == TPMLP_BF16 ? 2 : 4));
}

// Optional scratch of the bf16 GEMMs' stream-K form
// (tpmlp_workspace_bytes_balanced): per-tile arrival counters, then fp32
// partial-accumulator slots, two per CTA.
// - N <= 64 (few tokens; every (tile, k-block) unit is dealt out): 4
//   counters per tile for the most tiles any GEMM of the block has (T groups
//   of up to max(F/T, D) columns in 128-column tiles), slots of
//   round_up(N, 32) rows for as many CTAs as the GEMMs have units, at most
//   kSkMaxCtas. Every GEMM with M = N of the block has T x (N-columns / 128
//   tiles) x (K / 64 k-blocks) units with {N-columns, K} = {F/T, D}, folded
//   or grouped alike.
// - N > 64 (only the part wave's tiles are dealt out, fewer tiles than
//   units): 8 counters (4 per CTA of a pair) for up to kSkMaxCtas tiles, slots
//   of 128 rows for kSkMaxCtas CTAs (64 MiB).
size_t sk_part_bytes_for(int64_t M, int64_t units) {
    if (M > 64) return (size_t)kSkMaxCtas * 2 * 128 * kSkMaxBn * 4;
    const int64_t rows = M < 64 ? ((M + 31) / 32) * 32 : 64;
    const int64_t ctas = units < kSkMaxCtas ? units : kSkMaxCtas;
    return (size_t)ctas * 2 * (size_t)rows * kSkMaxBn * 4;
}
size_t sk_cnt_bytes(int64_t N, int64_t D, int64_t Fs, int T) {
    if (N > 64) return round256((size_t)kSkMaxCtas * 8 * sizeof(int));
    const int64_t cols = Fs > D ? Fs : D;
    return round256((size_t)4 * T * ((cols + 127) / 128) * sizeof(int));
}
int64_t sk_units_bound(int64_t D, int64_t Fs, int T) {
    const int64_t a = ((Fs + 127) / 128) * ((D + 63) / 64);
    const int64_t b = ((D + 127) / 128) * ((Fs + 63) / 64);
    return (int64_t)T * (a > b ? a : b);
}
size_t sk_bytes(tpmlp_dtype dt, int64_t N, int64_t D, int64_t F, int T) {
    if (dt != TPMLP_BF16 || N < 1) return 0;
    return sk_cnt_bytes(N, D, F / T, T) + sk_part_bytes_for(N, sk_units_bound(D, F / T, T));
}

struct SkArea {
    float* part = nullptr;
    size_t part_bytes = 0;
    int* cnt = nullptr;
    int64_t cnt_cap = 0;
};

// The stream-K scratch at round256(base) bytes into the workspace, if the
// caller's workspace is that large (see tpmlp_workspace_bytes_balanced).
SkArea sk_area(void* ws, size_t ws_bytes, size_t base, tpmlp_dtype dt, int64_t N, int64_t D,
               int64_t F, int T) {
    SkArea a;
    const size_t need = sk_bytes(dt, N, D, F, T);
    const size_t off = round256(base);
    if (need == 0 || ws == nullptr || !aligned16(ws) || ws_bytes < off + need) return a;
    char* p = static_cast<char*>(ws) + off;
    const size_t cb = sk_cnt_bytes(N, D, F / T, T);
    a.cnt = reinterpret_cast<int*>(p);
    a.cnt_cap = (int64_t)(cb / sizeof(int));
    a.part = reinterpret_cast<float*>(p + cb);
    a.part_bytes = need - cb;
    return a;
}

tpmlp_status run_gemm(tpmlp_dtype dt, GemmProblem p, cudaStream_t s, const SkArea& sk = SkArea()) {
    p.sk_part = sk.part;
    p.sk_part_bytes = sk.part_bytes;
    p.sk_cnt = sk.cnt;
    p.sk_cnt_cap = sk.cnt_cap;
    return dt == TPMLP_BF16 ? run_gemm_tc(p, s) : run_gemm_simt(p, s);
}

GemmProblem problem(int M, int N, int K, int G, int fold, int64_t lda, int a_mn, int64_t ldb,
                    int b_mn, const char* name) {
    GemmProblem p;
    memset(&p, 0, sizeof(p));
    p.M = M;
    p.N = N;
    p.K = K;
    p.G = G;
    p.fold = fold;
    p.lda = lda;
    p.a_mn = a_mn;
    p.ldb = ldb;
    p.b_mn = b_mn;
    p.name = name;
    return p;
}

}  // namespace
}  // namespace tpmlp

using namespace tpmlp;

extern "C" {

size_t tpmlp_workspace_bytes(tpmlp_op op, tpmlp_dtype dt, int64_t N, int64_t D, int64_t F, int T,
                             tpmlp_reduce_mode mode) {
    if (check_dims(dt, N, D, F, T, TPMLP_ACT_RELU) == TPMLP_ERR_SHAPE || N < 0 || T < 1)
        return (size_t)-1;
    if (dt != TPMLP_F32 && dt != TPMLP_BF16) return (size_t)-1;
    const size_t part = mode == TPMLP_REDUCE_PARTIALS ? partials_bytes(N, D, T) : 0;
    if (op == TPMLP_OP_FORWARD) return part;
    if (op == TPMLP_OP_BACKWARD) return dz_bytes(dt, N, F / T, T) + part;
    return (size_t)-1;
}

size_t tpmlp_workspace_bytes_balanced(tpmlp_op op, tpmlp_dtype dt, int64_t N, int64_t D, int64_t F,
                                      int T, tpmlp_reduce_mode mode) {
    const size_t base = tpmlp_workspace_bytes(op, dt, N, D, F, T, mode);
    if (base == (size_t)-1) return base;
    const size_t sk = sk_bytes(dt, N, D, F, T);
    return sk == 0 ? base : round256(base) + sk;
}

// Row shards and the block-end sum (§02-§05): Y = sum_r H^(r) W2^(r) + b2, into
// Y or, with Y_rows, row block r of Y into Y_rows[r].
static tpmlp_status block_end(tpmlp_dtype dt, int64_t N, int64_t D, int T, int Fs,
                              const void* const* H, const void* const* W2, const void* b2,
                              void* Y, void* const* Y_rows, tpmlp_reduce_mode mode,
                              void* workspace, cudaStream_t s, const SkArea& sk) {
    const int f32 = dt == TPMLP_BF16 ? 0 : 1;
    if (mode == TPMLP_REDUCE_PARTIALS) {
        const size_t stride = round256((size_t)N * D * 4);
        const float* parts[kMaxG];
        GemmProblem row = problem((int)N, (int)D, Fs, T, 0, Fs, 0, D, 1, "row_gemm_partials");
        row.epi.kind = EPI_STORE;
        row.epi.out_f32 = 1;
        row.epi.ldc = D;
        for (int r = 0; r < T; ++r) {
            float* pr = reinterpret_cast<float*>(static_cast<char*>(workspace) + r * stride);
            row.A[r] = H[r];
            row.B[r] = W2[r];
            row.epi.C[r] = pr;
            parts[r] = pr;
        }
        TPMLP_TRY(run_gemm(dt, row, s, sk));
        TPMLP_TRY(run_block_reduce(f32, N, D, T, parts, b2, Y, s,
                                   Y_rows ? "block_reduce_scatter_bias" : "block_reduce_bias",
                                   Y_rows));
    } else {
        GemmProblem row = problem((int)N, (int)D, Fs, T, 1, Fs, 0, D, 1,
                                  Y_rows ? "row_gemm_splitk_bias_scatter" : "row_gemm_splitk_bias");
        row.epi.kind = EPI_STORE;
        row.epi.out_f32 = f32;
        row.epi.ldc = D;
        row.epi.bias[0] = b2;
        if (Y_rows != nullptr) {
            row.epi.row_shard = N / T;
            for (int r = 0; r < T; ++r) row.epi.C[r] = Y_rows[r];
        } else {
            row.epi.C[0] = Y;
        }
        for (int r = 0; r < T; ++r) {
            row.A[r] = H[r];
            row.B[r] = W2[r];
        }
        TPMLP_TRY(run_gemm(dt, row, s, sk));
    }
    return TPMLP_OK;
}

// The forward's steps; the block end writes Y, or, with Y_rows, row block r
// of Y to Y_rows[r] (reduce-scatter).
static tpmlp_status forward_impl(tpmlp_dtype dt, int64_t N, int64_t D, int64_t F, int T,
                                 tpmlp_act act, const void* X, const void* const* W1,
                                 const void* const* b1, const void* const* W2, const void* b2,
                                 void* Y, void* const* Y_rows, void* const* H, void* const* Z,
                                 tpmlp_reduce_mode mode, void* workspace, size_t workspace_bytes,
                                 void* stream) {
    TPMLP_TRY(check_dims(dt, N, D, F, T, act));
    if (mode != TPMLP_REDUCE_PARTIALS && mode != TPMLP_REDUCE_SPLITK) return TPMLP_ERR_ARG;
    if (N == 0) return TPMLP_OK;   // every output is empty
    const bool bf = dt == TPMLP_BF16;
    TPMLP_TRY(check_ptr(X, bf));
    if (Y_rows != nullptr) {
        if (N % T != 0) return TPMLP_ERR_SHAPE;
        TPMLP_TRY(check_shards(reinterpret_cast<const void* const*>(Y_rows), T, bf));
    } else {
        TPMLP_TRY(check_ptr(Y, bf));
    }
    TPMLP_TRY(check_shards(W1, T, bf));
    TPMLP_TRY(check_shards(W2, T, bf));
    TPMLP_TRY(check_shards(reinterpret_cast<const void* const*>(H), T, bf));
    if (b1 != nullptr) TPMLP_TRY(check_shards(b1, T, bf));
    if (Z != nullptr) TPMLP_TRY(check_shards(reinterpret_cast<const void* const*>(Z), T, bf));
    if (b2 != nullptr) TPMLP_TRY(check_ptr(b2, bf));
    const size_t need = tpmlp_workspace_bytes(TPMLP_OP_FORWARD, dt, N, D, F, T, mode);
    if (need > 0) {
        if (workspace == nullptr || workspace_bytes < need) return TPMLP_ERR_WORKSPACE;
        if (!aligned16(workspace)) return TPMLP_ERR_ALIGN;
    }
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int Fs = (int)(F / T);
    const int f32 = bf ? 0 : 1;

    // 1. column shards: H^(r) = act(X W1^(r) + b1^(r)), Z^(r) saved
    GemmProblem col = problem((int)N, Fs, (int)D, T, 0, D, 0, Fs, 1, "col_gemm_bias_act");
    col.epi.kind = EPI_ACT;
    col.epi.act = act;
    col.epi.out_f32 = f32;
    col.epi.ldc = Fs;
    col.epi.ldaux = Fs;
    for (int r = 0; r < T; ++r) {
        col.A[r] = X;
        col.B[r] = W1[r];
        col.epi.C[r] = H[r];
        col.epi.bias[r] = b1 ? b1[r] : nullptr;
        col.epi.aux[r] = Z ? Z[r] : nullptr;
    }
    const SkArea sk = sk_area(workspace, workspace_bytes, need, dt, N, D, F, T);
    TPMLP_TRY(run_gemm(dt, col, s, sk));

    // 2. row shards and the block-end sum
    return block_end(dt, N, D, T, Fs, reinterpret_cast<const void* const*>(H), W2, b2, Y, Y_rows,
                     mode, workspace, s, sk);
}

tpmlp_status tpmlp_forward(tpmlp_dtype dt, int64_t N, int64_t D, int64_t F, int T, tpmlp_act act,
                           const void* X, const void* const* W1, const void* const* b1,
                           const void* const* W2, const void* b2, void* Y, void* const* H,
                           void* const* Z, tpmlp_reduce_mode mode, void* workspace,
                           size_t workspace_bytes, void* stream) {
    return forward_impl(dt, N, D, F, T, act, X, W1, b1, W2, b2, Y, nullptr, H, Z, mode, workspace,
                        workspace_bytes, stream);
}

tpmlp_status tpmlp_forward_reduce_scatter(tpmlp_dtype dt, int64_t N, int64_t D, int64_t F, int T,
                                          tpmlp_act act, const void* X, const void* const* W1,
                                          const void* const* b1, const void* const* W2,
                                          const void* b2, void* const* Y_rows, void* const* H,
                                          void* const* Z, tpmlp_reduce_mode mode, void* workspace,
                                          size_t workspace_bytes, void* stream) {
    if (Y_rows == nullptr) return TPMLP_ERR_ARG;
    return forward_impl(dt, N, D, F, T, act, X, W1, b1, W2, b2, nullptr, Y_rows, H, Z, mode,
                        workspace, workspace_bytes, stream);
}

tpmlp_status tpmlp_swiglu_forward(tpmlp_dtype dt, int64_t N, int64_t D, int64_t F, int T,
                                  const void* X, const void* const* Wg, const void* const* Wu,
                                  const void* const* Wd, void* Y, void* const* H, void* const* G,
                                  void* const* U, tpmlp_reduce_mode mode, void* workspace,
                                  size_t workspace_bytes, void* stream) {
    TPMLP_TRY(check_dims(dt, N, D, F, T, TPMLP_ACT_RELU));
    if (mode != TPMLP_REDUCE_PARTIALS && mode != TPMLP_REDUCE_SPLITK) return TPMLP_ERR_ARG;
    if (N == 0) return TPMLP_OK;
    const bool bf = dt == TPMLP_BF16;
    TPMLP_TRY(check_ptr(X, bf));
    TPMLP_TRY(check_ptr(Y, bf));
    TPMLP_TRY(check_shards(Wg, T, bf));
    TPMLP_TRY(check_shards(Wu, T, bf));
    TPMLP_TRY(check_shards(Wd, T, bf));
    TPMLP_TRY(check_shards(reinterpret_cast<const void* const*>(H), T, bf));
    if (G != nullptr) TPMLP_TRY(check_shards(reinterpret_cast<const void* const*>(G), T, bf));
    if (U != nullptr) TPMLP_TRY(check_shards(reinterpret_cast<const void* const*>(U), T, bf));
    const size_t need = tpmlp_workspace_bytes(TPMLP_OP_FORWARD, dt, N, D, F, T, mode);
    if (need > 0) {
        if (workspace == nullptr || workspace_bytes < need) return TPMLP_ERR_WORKSPACE;
        if (!aligned16(workspace)) return TPMLP_ERR_ALIGN;
    }
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int Fs = (int)(F / T);
    // 1. gate and up of shard r over the SAME columns, one dual GEMM:
    //    G^(r) = X Wg^(r), U^(r) = X Wu^(r), H^(r) = SiLU(G^(r)) * U^(r)
    GemmProblem col = problem((int)N, Fs, (int)D, T, 0, D, 0, Fs, 1, "col_gemm_swiglu");
    col.dual = 1;
    col.epi.kind = EPI_SWIGLU;
    col.epi.out_f32 = bf ? 0 : 1;
    col.epi.ldc = Fs;
    col.epi.ldaux = Fs;
    for (int r = 0; r < T; ++r) {
        col.A[r] = X;
        col.B[r] = Wg[r];
        col.B2[r] = Wu[r];
        col.epi.C[r] = H[r];
        col.epi.aux[r] = G ? G[r] : nullptr;
        col.epi.aux2[r] = U ? U[r] : nullptr;
    }
    const SkArea sk = sk_area(workspace, workspace_bytes, need, dt, N, D, F, T);
    TPMLP_TRY(run_gemm(dt, col, s, sk));
    // 2. the down projection's row shards and the block-end sum, as in the plain block
    return block_end(dt, N, D, T, Fs, reinterpret_cast<const void* const*>(H), Wd, nullptr, Y,
                     nullptr, mode, workspace, s, sk);
}

tpmlp_status tpmlp_backward(tpmlp_dtype dt, int64_t N, int64_t D, int64_t F, int T, tpmlp_act act,
                            const void* X, const void* const* W1, const void* const* W2,
                            const void* const* H, const void* const* Z, const void* dY, void* dX,
                            void* const* dW1, void* const* dW2, void* const* db1, void* db2,
                            tpmlp_reduce_mode mode, void* workspace, size_t workspace_bytes,
                            void* stream) {
    TPMLP_TRY(check_dims(dt, N, D, F, T, act));
    if (mode != TPMLP_REDUCE_PARTIALS && mode != TPMLP_REDUCE_SPLITK) return TPMLP_ERR_ARG;
    const bool bf = dt == TPMLP_BF16;
    TPMLP_TRY(check_shards(reinterpret_cast<const void* const*>(dW1), T, bf));
    TPMLP_TRY(check_shards(reinterpret_cast<const void* const*>(dW2), T, bf));
    if (db1 != nullptr) TPMLP_TRY(check_shards(reinterpret_cast<const void* const*>(db1), T, bf));
    if (db2 != nullptr) TPMLP_TRY(check_ptr(db2, bf));
    if (N > 0) {   // with no tokens, X, H, Z, dY, dX and the workspace are empty
        TPMLP_TRY(check_ptr(X, bf));
        TPMLP_TRY(check_ptr(dY, bf));
        TPMLP_TRY(check_ptr(dX, bf));
        TPMLP_TRY(check_shards(W1, T, bf));
        TPMLP_TRY(check_shards(W2, T, bf));
        TPMLP_TRY(check_shards(H, T, bf));
        TPMLP_TRY(check_shards(Z, T, bf));
        const size_t need = tpmlp_workspace_bytes(TPMLP_OP_BACKWARD, dt, N, D, F, T, mode);
        if (workspace == nullptr || workspace_bytes < need) return TPMLP_ERR_WORKSPACE;
        if (!aligned16(workspace)) return TPMLP_ERR_ALIGN;
    }
    const SkArea sk =
        N > 0 ? sk_area(workspace, workspace_bytes,
                        tpmlp_workspace_bytes(TPMLP_OP_BACKWARD, dt, N, D, F, T, mode), dt, N, D, F, T)
              : SkArea();
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int Fs = (int)(F / T);
    const int f32 = bf ? 0 : 1;
    const size_t esz = bf ? 2 : 4;

    if (N == 0) {
        // sums over an empty token set
        for (int r = 0; r < T; ++r) {
            if (cudaMemsetAsync(dW1[r], 0, (size_t)D * Fs * esz, s) != cudaSuccess ||
                cudaMemsetAsync(dW2[r], 0, (size_t)Fs * D * esz, s) != cudaSuccess)
                return TPMLP_ERR_CUDA;
            if (db1 && cudaMemsetAsync(db1[r], 0, (size_t)Fs * esz, s) != cudaSuccess)
                return TPMLP_ERR_CUDA;
        }
        if (db2 && cudaMemsetAsync(db2, 0, (size_t)D * esz, s) != cudaSuccess) return TPMLP_ERR_CUDA;
        return TPMLP_OK;
    }

    const size_t dz_stride = round256((size_t)N * Fs * esz);
    void* dZ[kMaxG];
    for (int r = 0; r < T; ++r) dZ[r] = static_cast<char*>(workspace) + r * dz_stride;

    // 1. dZ^(r) = (dY W2^(r)^T) * act'(Z^(r)); B(k, n) = W2^(r)[n, k]: K-major
    GemmProblem g1 = problem((int)N, Fs, (int)D, T, 0, D, 0, D, 0, "bwd_dz_gemm_dact");
    g1.epi.kind = EPI_DACT;
    g1.epi.act = act;
    g1.epi.out_f32 = f32;
    g1.epi.ldc = Fs;
    g1.epi.ldaux = Fs;
    for (int r = 0; r < T; ++r) {
        g1.A[r] = dY;
        g1.B[r] = W2[r];
        g1.epi.C[r] = dZ[r];
        g1.epi.aux[r] = const_cast<void*>(Z[r]);
    }
    TPMLP_TRY(run_gemm(dt, g1, s, sk));

    // 2. dW2^(r) = H^(r)^T dY: A(m, k) = H^(r)[k, m] (MN-major), B(k, n) = dY[k, n]
    GemmProblem g2 = problem(Fs, (int)D, (int)N, T, 0, Fs, 1, D, 1, "bwd_dw2_gemm");
    g2.epi.kind = EPI_STORE;
    g2.epi.out_f32 = f32;
    g2.epi.ldc = D;
    for (int r = 0; r < T; ++r) {
        g2.A[r] = H[r];
        g2.B[r] = dY;
        g2.epi.C[r] = dW2[r];
    }
    TPMLP_TRY(run_gemm(dt, g2, s, sk));

    // 3. dW1^(r) = X^T dZ^(r): A(m, k) = X[k, m] (MN-major), B(k, n) = dZ^(r)[k, n]
    GemmProblem g3 = problem((int)D, Fs, (int)N, T, 0, D, 1, Fs, 1, "bwd_dw1_gemm");
    g3.epi.kind = EPI_STORE;
    g3.epi.out_f32 = f32;
    g3.epi.ldc = Fs;
    for (int r = 0; r < T; ++r) {
        g3.A[r] = X;
        g3.B[r] = dZ[r];
        g3.epi.C[r] = dW1[r];
    }
    TPMLP_TRY(run_gemm(dt, g3, s, sk));

    // 4. dX = sum_r dZ^(r) W1^(r)^T: A = dZ^(r) (K-major), B(k, n) = W1^(r)[n, k] (K-major)
    if (mode == TPMLP_REDUCE_PARTIALS) {
        const size_t pstride = round256((size_t)N * D * 4);
        char* pbase = static_cast<char*>(workspace) + T * dz_stride;
        const float* parts[kMaxG];
        GemmProblem g4 = problem((int)N, (int)D, Fs, T, 0, Fs, 0, Fs, 0, "bwd_dx_gemm_partials");
        g4.epi.kind = EPI_STORE;
        g4.epi.out_f32 = 1;
        g4.epi.ldc = D;
        for (int r = 0; r < T; ++r) {
            float* pr = reinterpret_cast<float*>(pbase + r * pstride);
            g4.A[r] = dZ[r];
            g4.B[r] = W1[r];
            g4.epi.C[r] = pr;
            parts[r] = pr;
        }
        TPMLP_TRY(run_gemm(dt, g4, s, sk));
        TPMLP_TRY(run_block_reduce(f32, N, D, T, parts, nullptr, dX, s, "block_reduce_dx"));
    } else {
        GemmProblem g4 = problem((int)N, (int)D, Fs, T, 1, Fs, 0, Fs, 0, "bwd_dx_gemm_splitk");
        g4.epi.kind = EPI_STORE;
        g4.epi.out_f32 = f32;
        g4.epi.ldc = D;
        g4.epi.C[0] = dX;
        for (int r = 0; r < T; ++r) {
            g4.A[r] = dZ[r];
            g4.B[r] = W1[r];
        }
        TPMLP_TRY(run_gemm(dt, g4, s, sk));
    }

    // 5. bias gradients: the column sums of the T dZ shards (db1) and of dY
    // (db2). With the stream-K scratch of a balanced workspace (free once the
    // GEMMs above are done: same stream) they stream whole rows in two
    // passes through it, all groups at once; without it one pass per column
    // strip, dZ's shards and dY in separate launches.
    {
        const void* in[kMaxColsumG];
        void* out[kMaxColsumG];
        int64_t cols[kMaxColsumG], ld[kMaxColsumG];
        int G = 0;
        if (db1 != nullptr)
            for (int r = 0; r < T; ++r, ++G) {
                in[G] = dZ[r];
                out[G] = db1[r];
                cols[G] = ld[G] = Fs;
            }
        if (db2 != nullptr) {
            in[G] = dY;
            out[G] = db2;
            cols[G] = ld[G] = D;
            ++G;
        }
        if (G > 0 && sk.part != nullptr && !f32) {
            TPMLP_TRY(run_colsum(f32, N, G, cols, ld, in, out, s, sk.part, sk.part_bytes));
        } else {
            const int Gz = db1 != nullptr ? T : 0;
            if (Gz > 0) TPMLP_TRY(run_colsum(f32, N, Gz, cols, ld, in, out, s));
            if (db2 != nullptr) TPMLP_TRY(run_colsum(f32, N, 1, cols + Gz, ld + Gz, in + Gz, out + Gz, s));
        }
    }
    return TPMLP_OK;
}

tpmlp_status tpmlp_block_reduce(tpmlp_dtype dt, int64_t N, int64_t D, int T,
                                const float* const* partials, const void* b2, void* Y,
                                void* stream) {
    if (dt != TPMLP_F32 && dt != TPMLP_BF16) return TPMLP_ERR_DTYPE;
    if (N < 0) return TPMLP_ERR_ARG;
    if (D <= 0 || T < 1 || T > TPMLP_MAX_SHARDS) return TPMLP_ERR_SHAPE;
    if (partials == nullptr || Y == nullptr) return TPMLP_ERR_ARG;
    for (int r = 0; r < T; ++r)
        if (partials[r] == nullptr) return TPMLP_ERR_ARG;
    return run_block_reduce(dt == TPMLP_F32, N, D, T, partials, b2, Y,
                            static_cast<cudaStream_t>(stream), "block_reduce_bias");
}

tpmlp_status tpmlp_block_reduce_scatter(tpmlp_dtype dt, int64_t N, int64_t D, int T,
                                        const float* const* partials, const void* b2,
                                        void* const* Y_rows, void* stream) {
    if (dt != TPMLP_F32 && dt != TPMLP_BF16) return TPMLP_ERR_DTYPE;
    if (N < 0) return TPMLP_ERR_ARG;
    if (D <= 0 || T < 1 || T > TPMLP_MAX_SHARDS || N % T != 0) return TPMLP_ERR_SHAPE;
    if (partials == nullptr || Y_rows == nullptr) return TPMLP_ERR_ARG;
    for (int r = 0; r < T; ++r)
        if (partials[r] == nullptr || Y_rows[r] == nullptr) return TPMLP_ERR_ARG;
    return run_block_reduce(dt == TPMLP_F32, N, D, T, partials, b2, nullptr,
                            static_cast<cudaStream_t>(stream), "block_reduce_scatter_bias", Y_rows);
}

tpmlp_status tpmlp_vocab_embedding(tpmlp_dtype dt, int64_t N, int64_t V, int64_t Hd, int T,
                                   const int64_t* ids, const void* const* table, void* out,
                                   void* stream) {
    if (dt != TPMLP_F32 && dt != TPMLP_BF16) return TPMLP_ERR_DTYPE;
    if (N < 0) return TPMLP_ERR_ARG;
    if (V <= 0 || Hd <= 0 || T < 1 || T > TPMLP_MAX_SHARDS || V % T != 0) return TPMLP_ERR_SHAPE;
    if (N > 0 && (ids == nullptr || out == nullptr || table == nullptr)) return TPMLP_ERR_ARG;
    if (table != nullptr)
        for (int k = 0; k < T; ++k)
            if (table[k] == nullptr) return TPMLP_ERR_ARG;
    return run_vocab_embedding(dt == TPMLP_F32, N, V, Hd, T, ids, table, out,
                               static_cast<cudaStream_t>(stream));
}

tpmlp_status tpmlp_vocab_ce(int64_t N, int64_t V, int T, const float* logits,
                            const int64_t* targets, float* loss_per_token, float* loss_mean,
                            int32_t* argmax, int32_t* target_owner, void* stream) {
    if (N < 0) return TPMLP_ERR_ARG;
    if (V <= 0 || T < 1 || T > TPMLP_MAX_SHARDS || V % T != 0) return TPMLP_ERR_SHAPE;
    if (N > 0 && (logits == nullptr || targets == nullptr || loss_per_token == nullptr))
        return TPMLP_ERR_ARG;
    if (V > 0x7fffffffLL || N > 0x7fffffffLL) return TPMLP_ERR_SHAPE;
    return run_vocab_ce(N, V, T, logits, targets, loss_per_token, loss_mean, argmax, target_owner,
                        static_cast<cudaStream_t>(stream));
}

tpmlp_status tpmlp_vocab_ce_backward(int64_t N, int64_t V, int T, const float* logits,
                                     const int64_t* targets, const float* loss_per_token,
                                     float grad_scale, float* dlogits, void* stream) {
    if (N < 0) return TPMLP_ERR_ARG;
    if (V <= 0 || T < 1 || T > TPMLP_MAX_SHARDS || V % T != 0) return TPMLP_ERR_SHAPE;
    if (V > 0x7fffffffLL || N > 0x7fffffffLL) return TPMLP_ERR_SHAPE;
    if (N > 0 && (logits == nullptr || targets == nullptr || loss_per_token == nullptr ||
                  dlogits == nullptr))
        return TPMLP_ERR_ARG;
    return run_vocab_ce_backward(N, V, logits, targets, loss_per_token, grad_scale, dlogits,
                                 static_cast<cudaStream_t>(stream));
}

tpmlp_status tpmlp_gemm_plan(int64_t M, int64_t N, int64_t K, int G, int fold, int dual,
                             int balanced, int* bn, int* mma_ctas, int* ksplit) {
    if (bn == nullptr || mma_ctas == nullptr || ksplit == nullptr) return TPMLP_ERR_ARG;
    const int64_t lim = 2147483647;
    if (M < 1 || N < 1 || K < 1 || M > lim || N > lim || K > lim || G < 1 || G > TPMLP_MAX_SHARDS)
        return TPMLP_ERR_SHAPE;
    GemmProblem p = problem((int)M, (int)N, (int)K, G, fold ? 1 : 0, K, 0, K, 0, "plan");
    p.dual = dual ? 1 : 0;
    if (balanced) {
        // a scratch as large as the block's workspace would provide (never
        // dereferenced: the plan launches nothing)
        static float part_dummy;
        static int cnt_dummy;
        p.sk_part = &part_dummy;
        p.sk_part_bytes = sk_part_bytes_for(M, kSkMaxCtas);
        p.sk_cnt = &cnt_dummy;
        p.sk_cnt_cap = M > 64 ? (int64_t)kSkMaxCtas * 8 : (int64_t)4 * G * ((N + 127) / 128);
    }
    return plan_gemm_tc(p, bn, mma_ctas, ksplit);
}

const char* tpmlp_status_str(tpmlp_status s) {
    switch (s) {
        case TPMLP_OK: return "TPMLP_OK";
        case TPMLP_ERR_ARG: return "TPMLP_ERR_ARG: invalid argument";
        case TPMLP_ERR_SHAPE: return "TPMLP_ERR_SHAPE: invalid shape (F % T, V % T, T range, zero width)";
        case TPMLP_ERR_ALIGN: return "TPMLP_ERR_ALIGN: pointer or row pitch not 16-byte aligned";
        case TPMLP_ERR_DTYPE: return "TPMLP_ERR_DTYPE: unknown element type";
        case TPMLP_ERR_CUDA: return "TPMLP_ERR_CUDA: CUDA call failed";
        case TPMLP_ERR_TIMEOUT: return "TPMLP_ERR_TIMEOUT: a bounded device wait expired";
        case TPMLP_ERR_WORKSPACE: return "TPMLP_ERR_WORKSPACE: workspace missing or too small";
    }
    return "unknown tpmlp status";
}

tpmlp_status tpmlp_check_device_error(void* stream) {
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return TPMLP_ERR_CUDA;
    int* p = device_error_word();
    if (p == nullptr) return TPMLP_ERR_CUDA;
    int v = 0;
    if (cudaMemcpy(&v, p, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return TPMLP_ERR_CUDA;
    const int zero = 0;
    if (cudaMemcpy(p, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess) return TPMLP_ERR_CUDA;
    return static_cast<tpmlp_status>(v);
}

void tpmlp_set_wait_timeout_ns(uint64_t ns) { g_timeout_ns.store(ns > 0 ? ns : 1); }

tpmlp_status tpmlp_selftest_wait_timeout(uint64_t timeout_ns, void* stream) {
    return run_selftest_wait(timeout_ns, static_cast<cudaStream_t>(stream));
}

tpmlp_status tpmlp_selftest_gemm_stall(int role) {
    if (role < 0 || role > 3) return TPMLP_ERR_ARG;
    g_gemm_stall.store(role);
    return TPMLP_OK;
}

int64_t tpmlp_launch_count(void) { return g_launches.load(); }

void tpmlp_timing_enable(int on) {
    std::lock_guard<std::mutex> lk(g_t_mu);
    g_timing = on != 0;
}

int tpmlp_timing_read(tpmlp_kernel_timing* out, int max_entries) {
    std::lock_guard<std::mutex> lk(g_t_mu);
    int rc = 0;
    for (auto& r : g_pending) {
        float ms = 0.f;
        if (cudaEventSynchronize(r.stop) != cudaSuccess ||
            cudaEventElapsedTime(&ms, r.start, r.stop) != cudaSuccess)
            rc = -1;
        TimingAgg& a = g_agg[r.name];
        a.launches += 1;
        a.ms += ms;
        g_event_pool.push_back(r.start);
        g_event_pool.push_back(r.stop);
    }
    g_pending.clear();
    if (rc < 0) return -1;
    int n = 0;
    for (auto& kv : g_agg) {
        if (n >= max_entries || out == nullptr) break;
        memset(&out[n], 0, sizeof(out[n]));
        strncpy(out[n].name, kv.first.c_str(), sizeof(out[n].name) - 1);
        out[n].launches = kv.second.launches;
        out[n].total_ms = kv.second.ms;
        ++n;
    }
    return n;
}

void tpmlp_timing_reset(void) {
    std::lock_guard<std::mutex> lk(g_t_mu);
    for (auto& r : g_pending) {
        cudaEventSynchronize(r.stop);
        g_event_pool.push_back(r.start);
        g_event_pool.push_back(r.stop);
    }
    g_pending.clear();
    g_agg.clear();
}

}  // extern "C"
