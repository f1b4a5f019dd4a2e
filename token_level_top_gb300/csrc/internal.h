// internal.h -- declarations shared by the libmoe translation units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/moe.h"

namespace moe {

constexpr int kChunk = 256;        // tokens per routing chunk (one route block)
constexpr int kPrefLen = 16;       // preference-order prefix staged per token by the dispatch
constexpr int kBM = 128;           // GEMM tile rows (tokens / slots)
constexpr int kBK = 64;            // GEMM K per pipeline stage (128 bytes of bf16)
constexpr int kExpertBN = 256;     // expert GEMM tile columns
constexpr int kGemmThreads = 192;  // 6 warps: TMA, MMA, 4 x epilogue
constexpr long long kSpinBudget = 2000000000LL;  // ~1 s of SM clock per bounded wait

enum GemmKind : int { GK_ROUTER = 0, GK_GATEUP = 1, GK_DOWN_SLOTS = 3 };

// Byte offsets of every scratch region inside the caller's workspace.
struct WsLayout {
    int nchunks = 0;   // ceil(T / kChunk)
    int splits = 0;    // router GEMM K-splits
    int epad = 0;      // router N tile (E rounded up to 16, at least 16)
    size_t status = 0, ctrl = 0, part = 0, scores = 0, ids = 0, prefs = 0, crank = 0, hist = 0,
           base = 0, ppart = 0, assign = 0, slot = 0, flags = 0, counts = 0, offsets = 0,
           perm = 0, cw = 0, xg = 0, act = 0, y_slots = 0, h_stage = 0, out_stage = 0;
    // MOE_FLAG_FP8: e4m3 activation rows of the down GEMM and the row scales
    // of both GEMMs' activations (the gate-up codes reuse the xg region)
    size_t act_q = 0, x_scale = 0, act_scale = 0, act_amax = 0;
    // MOE_FLAG_NVFP4: e2m1 codes, block scales and row scales of the token rows
    // (gate-up input) and of the activation rows (down input)
    size_t x4 = 0, x4_sf = 0, x4_scale = 0, a4 = 0, a4_sf = 0, a4_scale = 0;
    size_t xn = 0;     // router input after normalisation [T, d] bf16 (router_norm != 0)
    size_t bwd = 0;    // backward scratch (MOE_FLAG_BACKWARD)
    size_t gu = 0;     // g and u of the kept rows, kept by the forward for the backward [T*k, 2F] fp32
    size_t zr = 0;     // two-layer router logits [T, E] fp32 (router_hidden > 0)
    int nr = 0;        // router GEMM output columns: E, or the hidden width H
    size_t total = 0;
};

// ctrl block (int32 words)
enum CtrlWord : int { CTRL_Q1 = 0, CTRL_NRE = 1, CTRL_NDROP = 2, CTRL_WORDS = 64 };

// Bytes per token of the stored preference order: all E experts, padded to 16.
__host__ __device__ inline int pref_stride(int E) { return E <= kPrefLen ? kPrefLen : (E + 15) / 16 * 16; }

// The dispatch's rank-base table [k*nchunks][E] int32, followed by the
// replay's fallback storage for each tail entry's expert (T*k bytes, at
// dispatch_asg_offset) when its staging does not fit in shared memory.
inline size_t dispatch_asg_offset(size_t k, size_t nch, size_t E) { return k * nch * E * 4; }
inline size_t dispatch_base_bytes(size_t T, size_t k, size_t nch, size_t E)
{
    return dispatch_asg_offset(k, nch, E) + T * k;
}

bool layout_for(const moe_config_t& c, WsLayout* L);
// A process-unique id of the current CUDA context (0 if none or unknown):
// host-side set-up that belongs to a context (function attributes, symbol
// addresses) is done again in a new one -- another device, or after a reset.
unsigned long long context_id();
// Raises fn's dynamic shared-memory limit to `bytes` once per context.
cudaError_t ensure_smem_limit(const void* fn, int bytes);
int router_splits(int T, int d, int E);
int router_ctas_per_sm(int E);   // router GEMM CTAs resident per SM (shared memory bound)
int num_sms();

template <class T>
inline T* ws_at(void* ws, size_t off)
{
    return reinterpret_cast<T*>(static_cast<char*>(ws) + off);
}

// ---- launchers (all asynchronous on `stream`) ----
struct RouteArgs {
    int T, E, k, d, splits, epad, nchunks;
    const float* part;       // [splits][T][E] router GEMM partial sums, or NULL
    const float* logits_in;  // [T][E], or NULL
    const float* bias;       // [E] or NULL (added to GEMM partial sums only)
    const float* usage;      // [E] or NULL
    float lambda;
    float tau;               // temperature: s = z / tau - lambda*usage (0 or 1: none)
    float* logits_out;       // [T][E] or NULL
    float* scores_user;      // [T][E] or NULL
    float* scores_ws;        // [T][E] (always)
    int32_t* ids_user;       // [T][k] or NULL
    float* topk_w;           // [T][k] or NULL
    int32_t* ids_ws;         // [T][k]
    uint8_t* prefs;          // [T][pref_stride(E)] full preference order
    int32_t* crank;          // [T][k]
    int32_t* hist;           // [k*nchunks][E]
    float* ppart;            // [nchunks][E]
    int* status;
};
cudaError_t launch_route(const RouteArgs& a, cudaStream_t s);

struct StatsArgs {
    int T, E, k, nchunks;
    const int32_t* hist;
    const float* ppart;
    int32_t* counts_pre;  // or NULL
    float* f;             // or NULL
    float* P;             // or NULL
};
cudaError_t launch_route_stats(const StatsArgs& a, cudaStream_t s);

struct DispatchArgs {
    int T, E, k, nchunks;
    int64_t C;
    const float* scores;
    const int32_t* ids;
    const uint8_t* prefs;    // [T][pref_stride(E)]
    const int32_t* crank;
    const int32_t* hist;
    int32_t* base;
    int32_t* ctrl;
    int32_t* assign;
    int32_t* slot;
    uint8_t* flags;
    int32_t* counts;
    int32_t* offsets;
    int32_t* perm;
    float* cw;
    int32_t* n_rerouted;  // or NULL
    int32_t* n_dropped;   // or NULL
    int* status;
};
cudaError_t launch_dispatch(const DispatchArgs& a, cudaStream_t s);
// Route and dispatch of a batch of one chunk (T <= kChunk, nchunks == 1) in a
// single block: same results as launch_route followed by launch_dispatch.
cudaError_t launch_route_dispatch_small(const RouteArgs& ra, const DispatchArgs& a, cudaStream_t s);

struct GemmLaunch {
    int kind;
    int E, T, topk, d, F;
    const void* a_ptr;  // router: h [T,d]; gate-up: x_perm [T*k, d]; down: act [T*k, F]
    const void* b_ptr;  // router: W_r [E,d]; gate-up: W13 [E,2F,d]; down: W2 [E,d,F]
    const int32_t* offsets;
    const int32_t* perm;
    void* act;
    void* y_slots;
    float* router_part;
    int splits, epad;
    long long rows_cap;  // most rows an expert can hold (the capacity C), or 0 if unknown
    int fp8;                 // expert GEMMs: a_ptr and b_ptr hold e4m3 rows, each with
    const float* a_scale;    //   its scale: a_scale per activation row (slot order),
    const float* b_scale;    //   b_scale per weight row (W13: [E*2F], W2: [E*d])
    float* act_amax;         // gate-up: if set, atomically maxed with each act row's max |bf16 value|
    void* gu_save;           // gate-up (bf16 weights): if set, g and u of each kept row [T*k, 2F] fp32
    int* status;
    long long budget;
};
cudaError_t launch_gemm(const GemmLaunch& g, cudaStream_t s);
// NVFP4 (nvfp4.cu): e2m1 codes packed two per byte, e4m3 scales per 16
// consecutive elements (rows of them padded to nvfp4_sf_stride bytes), an fp32
// scale per row.  launch_quantize_nvfp4 quantises rows [0, rows) of a bf16
// matrix [.., cols]: row r reads source row perm[r] / k (perm given), or the
// W13 row that the 128-row packing puts at r (w13_F = d_ff > 0), or r; rows
// from *nrows on are skipped; amax_in gives each row's max |value|;
// zero_rows, when given, gets 0 at each quantised row.  cols <= 16384, a
// multiple of 32.
int nvfp4_sf_stride(int cols);
cudaError_t launch_quantize_nvfp4(long long rows, int cols, const void* w, const int32_t* perm, int k,
                                  int w13_F, const int32_t* nrows, const float* amax_in, void* codes,
                                  void* bscale, float* scales, float* zero_rows, cudaStream_t s);
struct F4Launch {
    int kind;                 // GK_GATEUP or GK_DOWN_SLOTS
    int E, T, topk, d, F;
    const void* a_codes;      // gate-up: token rows [T*k, d/2]; down: activation rows [T*k, F/2]
    const void* a_sf;         // their block scales [T*k, nvfp4_sf_stride(K)]
    const float* a_scale;     // their row scales [T*k]
    const void* b_codes;      // W13 [E*2F, d/2] (128-row packing) or W2 [E*d, F/2]
    const void* b_sf;
    const float* b_scale;
    const int32_t* offsets;
    void* act;                // gate-up output [T*k, F] bf16
    float* act_amax;          // gate-up: atomically maxed with each act row's max |bf16 value|
    void* y_slots;            // down output [T*k, d] bf16
    long long rows_cap;       // most rows an expert can hold (the capacity C), or 0 if unknown
    int* status;
    long long budget;
};
cudaError_t launch_gemm_nvfp4(const F4Launch& g, cudaStream_t s);

// Tensor map of a row-major bf16 matrix [rows, cols]: boxes of box_rows x 64
// columns (128 bytes), 128-byte swizzle; zero fill outside the matrix.
bool encode_bf16_map(CUtensorMap* tm, const void* ptr, uint64_t rows, uint64_t cols, uint32_t box_rows);

// The backward pass's per-expert products (bwd_gemm.cu) over row blocks that
// hold each expert's kept rows padded with zero rows to a multiple of 128.
enum BwdGemmMode : int { BG_DGRAD = 0, BG_WGRAD = 1 };
struct BwdGemmLaunch {
    int mode, E;
    long long rows;        // rows of the row-block buffers (room for every expert's padded block)
    long long kept;        // most kept rows (T*k): BG_DGRAD pairs CTAs when experts average 2+ row tiles
    int K;                 // BG_DGRAD: inner dimension (the row block's width, the weights' rows per expert)
    int N;                 // output columns
    int Mw;                // BG_WGRAD: output rows per expert (the A row block's width)
    const void* a;         // BG_DGRAD: row block [rows, K]; BG_WGRAD: row block [rows, Mw]
    const void* b;         // BG_DGRAD: weights [E*K, N]; BG_WGRAD: row block [rows, N]
    const int32_t* offsets;  // [E + 1] kept slots per expert (the padded blocks follow from them)
    float* out;            // BG_DGRAD: [rows, N]; BG_WGRAD: [E, Mw, N]
    int* status;
    long long budget;
};
cudaError_t launch_bwd_gemm(const BwdGemmLaunch& g, cudaStream_t s);

cudaError_t launch_pack_w13(int E, int F, int d, const void* w1, const void* w3, void* w13,
                            cudaStream_t s);
// x_perm[j] = h[perm[j] / k] for the offsets[E] kept rows.
cudaError_t launch_gather_rows(int T, int d, int k, int E, const void* h, const int32_t* perm,
                               const int32_t* offsets, void* x_perm, cudaStream_t s);
cudaError_t launch_combine(int T, int d, int k, const void* y_slots, const int32_t* assign,
                           const int32_t* slot, const int32_t* offsets, const float* cw, void* out,
                           cudaStream_t s);
// Per-row e4m3 quantisation of rows [0, rows) (bf16 [.., cols] -> codes + scales);
// row r reads source row perm[r] / k when perm is not NULL; rows from *nrows
// on are skipped when nrows is not NULL.  amax_in, when given, holds each
// row's max |value| already (one pass over the row instead of two);
// zero_rows, when given, gets 0 written at each quantised row's index.
cudaError_t launch_quantize_fp8(long long rows, int cols, const void* w, const int32_t* perm, int k,
                                const int32_t* nrows, void* q, float* scales, cudaStream_t s,
                                const float* amax_in = nullptr, float* zero_rows = nullptr);
// Router front end.  x = LayerNorm(h) (mode 1; gamma, beta [d] or NULL) or
// h / max(||h||, eps) (mode 2), bf16 [T, d]; d <= 16384.
cudaError_t launch_router_norm(int T, int d, int mode, float eps, const void* h, const float* gamma,
                               const float* beta, void* x, cudaStream_t s);
// z [T, E] = silu(sum of the splits x [T, H] partials) . W2^T (+ bias), W2 [E, H]
// bf16; H <= kMaxRouterHidden and E * H <= kMaxRouterWeights2.
constexpr int kMaxRouterHidden = 256;
constexpr int kMaxRouterWeights2 = 16384;
cudaError_t launch_router_head(int T, int E, int H, int splits, const float* part, const void* w2,
                               const float* bias, float* z, cudaStream_t s);
// z [T, E] = the sum of the splits x [T, E] partials (split order) + bias.
cudaError_t launch_router_sum(int T, int E, int splits, const float* part, const float* bias, float* z,
                              cudaStream_t s);
// The backward pass (backward.cu).  Reads the forward's routing state (scores, perm,
// offsets, cw) and writes the gradients; scratch holds backward_bytes(...) bytes.
struct BackwardArgs {
    int T, E, k, d, F;
    long long R;             // rows of the row blocks: room for every expert's kept rows rounded up to 128
    float tau;               // 0 or 1: none
    const float* scores;     // [T, E] the forward's penalised scores
    const int32_t* perm;     // kept slots in slot order: t*k + r
    const int32_t* offsets;  // [E + 1]
    const float* cw;         // [T, k] combine weights
    const void* h;           // [T, d] bf16
    const void* w_router;    // [E, d] bf16
    const void* w13;         // [E, 2F, d] bf16
    const void* w2;          // [E, d, F] bf16
    const void* dout;        // [T, d] bf16
    const float* gu;         // [T*k, 2F] fp32: the forward's g and u of each kept slot
    const float* dP;         // [E] or NULL
    float* dh;               // [T, d]
    float* dw_router;        // [E, d] or NULL
    float* dbias;            // [E] or NULL
    float* dw13;             // [E, 2F, d]
    float* dw2;              // [E, d, F]
    void* scratch;
    int* status;             // device status word
    long long budget;        // bounded waits
};
size_t backward_bytes(long long T, int d, int E, int k, int F, long long R);
// R for backward_bytes: at most sum over experts of (kept rows rounded up to 128).
long long backward_block_rows(long long T, int E, int k, long long C);
cudaError_t run_backward(const BackwardArgs& a, cudaStream_t s);

cudaError_t launch_timeout_probe(int* status, long long budget, cudaStream_t s);

}  // namespace moe
