// api.cu -- the C ABI of libmoe: argument checks, workspace layout and the
// ordering of the kernels on the caller's stream.  No allocation, no
// synchronisation on the forward path (moe_layer_forward_host and
// moe_get_device_status are the documented synchronous exceptions).
#include <math.h>

#include <algorithm>
#include <map>
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace moe {

namespace {
constexpr int kMaxE = 255;  // expert ids are kept in bytes; 255 marks "none"
constexpr int kMaxK = 8;

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

moe_status_t cuda_status(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

// Shape checks shared by every entry point; `need_ff` adds the expert-FFN ones.
moe_status_t check_config(const moe_config_t* c, bool need_ff)
{
    if (!c) return MOE_ERR_INVALID_ARG;
    if ((c->flags & ~(MOE_FLAG_FP8 | MOE_FLAG_BACKWARD | MOE_FLAG_NVFP4)) != 0) return MOE_ERR_INVALID_ARG;
    if (c->T < 0 || c->E <= 0 || c->k <= 0) return MOE_ERR_INVALID_ARG;
    if (c->k > c->E) return MOE_ERR_INVALID_ARG;
    if (c->capacity < 0) return MOE_ERR_INVALID_ARG;
    if (c->capacity == 0 && !(c->cf > 0.0 && c->cf <= 100.0)) return MOE_ERR_INVALID_ARG;
    if (!isfinite(c->lambda)) return MOE_ERR_INVALID_ARG;
    if (!(c->tau == 0.0f || (c->tau > 0.0f && isfinite(c->tau)))) return MOE_ERR_INVALID_ARG;
    if (c->router_norm > MOE_ROUTER_NORM_L2 || !(c->norm_eps >= 0.0f && isfinite(c->norm_eps)))
        return MOE_ERR_INVALID_ARG;
    if (c->router_hidden < 0) return MOE_ERR_INVALID_ARG;
    if (c->router_hidden > kMaxRouterHidden ||
        static_cast<long long>(c->router_hidden) * c->E > kMaxRouterWeights2)
        return MOE_ERR_UNSUPPORTED;
    if (c->router_norm != MOE_ROUTER_NORM_NONE && c->d_model > 16384) return MOE_ERR_UNSUPPORTED;
    if (c->E > kMaxE || c->k > kMaxK) return MOE_ERR_UNSUPPORTED;
    if (c->d_model <= 0 || c->d_model % 64 != 0) return MOE_ERR_UNSUPPORTED;
    if (need_ff && (c->d_ff <= 0 || c->d_ff % 128 != 0)) return MOE_ERR_UNSUPPORTED;
    if (static_cast<long long>(c->T) * c->k > (1LL << 30)) return MOE_ERR_UNSUPPORTED;
    return MOE_OK;
}

moe_status_t check_ws(const moe_config_t* c, void* ws, size_t ws_bytes, WsLayout* L)
{
    if (!ws) return MOE_ERR_INVALID_ARG;
    if (!aligned(ws, 256)) return MOE_ERR_MISALIGNED;
    if (!layout_for(*c, L)) return MOE_ERR_INVALID_ARG;
    if (ws_bytes < L->total) return MOE_ERR_WORKSPACE;
    return MOE_OK;
}

int64_t capacity_of(const moe_config_t& c)
{
    return moe_capacity(c.T, c.k, c.E, c.cf, c.capacity);
}

// Rows of the backward pass's row blocks (each expert's kept rows rounded up to
// 128): an expert holds at most C slots, and at most one per token.
long long backward_rows(const moe_config_t& c)
{
    return backward_block_rows(std::max(c.T, 0), c.E, c.k, capacity_of(c));
}

struct Ev {
    void* const* ev;
    cudaStream_t s;
    void mark(int i) const
    {
        if (ev && ev[i]) cudaEventRecord(static_cast<cudaEvent_t>(ev[i]), s);
    }
};

}  // namespace

namespace {
using PfnCtxGetCurrent = CUresult (*)(CUcontext*);
using PfnCtxGetId = CUresult (*)(CUcontext, unsigned long long*);

template <class Fn>
Fn driver_fn(const char* name)
{
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion(name, &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
        return nullptr;
    return reinterpret_cast<Fn>(p);
}
}  // namespace

unsigned long long context_id()
{
    static const PfnCtxGetCurrent get_cur = driver_fn<PfnCtxGetCurrent>("cuCtxGetCurrent");
    static const PfnCtxGetId get_id = driver_fn<PfnCtxGetId>("cuCtxGetId");
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    if (!get_cur || !get_id || get_cur(&ctx) != CUDA_SUCCESS || !ctx || get_id(ctx, &id) != CUDA_SUCCESS)
        return 0;
    return id + 1;
}

cudaError_t ensure_smem_limit(const void* fn, int bytes)
{
    static std::mutex mu;
    static std::map<std::pair<unsigned long long, const void*>, int> done;
    const unsigned long long ctx = context_id();   // 0: no context yet; set it every call until there is one
    std::lock_guard<std::mutex> lock(mu);
    auto it = done.find({ctx, fn});
    if (ctx != 0 && it != done.end() && it->second >= bytes) return cudaSuccess;
    const cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess && ctx != 0) done[{ctx, fn}] = bytes;
    return e;
}

int num_sms()
{
    static int cache[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
    if (cache[dev] == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
            n = 148;
        cache[dev] = n;
    }
    return cache[dev];
}

int router_splits(int T, int d, int E)
{
    const int mt = (T + kBM - 1) / kBM;
    const int kb = d / kBK;
    // as many splits as fill one resident wave of router CTAs (a second,
    // partial wave would double the makespan), at least 4 K steps each
    int S = router_ctas_per_sm(E) * num_sms() / std::max(mt, 1);
    S = std::max(1, std::min(S, std::max(1, kb / 4)));
    // no empty split: (S - 1) * ceil(kb / S) < kb
    while (S > 1 && (S - 1) * ((kb + S - 1) / S) >= kb) --S;
    return S;
}

bool layout_for(const moe_config_t& c, WsLayout* L)
{
    const size_t T = static_cast<size_t>(std::max(c.T, 0));
    const size_t E = static_cast<size_t>(c.E), k = static_cast<size_t>(c.k);
    const size_t d = static_cast<size_t>(c.d_model), F = static_cast<size_t>(std::max(c.d_ff, 0));
    WsLayout w;
    w.nchunks = static_cast<int>((T + kChunk - 1) / kChunk);
    // the router GEMM's output columns: the experts, or the two-layer router's hidden units
    w.nr = c.router_hidden > 0 ? c.router_hidden : c.E;
    const size_t NR = static_cast<size_t>(w.nr);
    w.splits = router_splits(static_cast<int>(T), static_cast<int>(d), w.nr);
    w.epad = static_cast<int>(std::max<size_t>(32, round_up(NR, 32)));
    size_t off = 0;
    auto take = [&](size_t bytes) {
        const size_t o = off;
        off += round_up(std::max<size_t>(bytes, 1), 256);
        return o;
    };
    const size_t nch = static_cast<size_t>(w.nchunks);
    w.status = take(256);
    w.ctrl = take(CTRL_WORDS * 4);
    w.part = take(static_cast<size_t>(w.splits) * T * NR * 4);
    w.scores = take(T * E * 4);
    w.ids = take(T * k * 4);
    w.prefs = take(T * static_cast<size_t>(pref_stride(c.E)));
    w.crank = take(T * k * 4);
    w.hist = take(k * nch * E * 4);
    w.base = take(dispatch_base_bytes(T, k, nch, E));
    w.ppart = take(nch * E * 4);
    w.assign = take(T * k * 4);
    w.slot = take(T * k * 4);
    w.flags = take(T * k);
    w.counts = take(E * 4);
    w.offsets = take((E + 1) * 4);
    w.perm = take(T * k * 4);
    w.cw = take(T * k * 4);
    w.xg = take(T * k * d * 2);
    w.act = take(T * k * F * 2);
    w.y_slots = take(T * k * d * 2);
    if (c.flags & MOE_FLAG_FP8) {
        w.act_q = take(T * k * F);
        w.x_scale = take(T * k * 4);
        w.act_scale = take(T * k * 4);
    }
    if (c.flags & (MOE_FLAG_FP8 | MOE_FLAG_NVFP4)) w.act_amax = take(T * k * 4);
    if (c.flags & MOE_FLAG_NVFP4) {
        w.x4 = take(T * k * d / 2);
        w.x4_sf = take(T * k * static_cast<size_t>(nvfp4_sf_stride(static_cast<int>(d))));
        w.x4_scale = take(T * k * 4);
        w.a4 = take(T * k * F / 2);
        w.a4_sf = take(T * k * static_cast<size_t>(nvfp4_sf_stride(static_cast<int>(F))));
        w.a4_scale = take(T * k * 4);
    }
    if (c.router_norm != MOE_ROUTER_NORM_NONE) w.xn = take(T * d * 2);
    if (c.router_hidden > 0) w.zr = take(T * E * 4);
    if (c.flags & MOE_FLAG_BACKWARD) w.gu = take(T * k * 2 * F * 4);
    if (c.flags & MOE_FLAG_BACKWARD)
        w.bwd = take(backward_bytes(static_cast<long long>(T), c.d_model, c.E, c.k, c.d_ff, backward_rows(c)));
    w.h_stage = take(T * d * 2);
    w.out_stage = take(T * d * 2);
    w.total = off;
    *L = w;
    return true;
}

namespace {

// The router GEMM (skipped when logits are given): h . W^T over L.nr output
// columns (the experts, or the two-layer router's hidden units).
moe_status_t run_router_gemm(const moe_config_t& c, const WsLayout& L, const void* h,
                             const void* wr, void* ws, cudaStream_t s)
{
    GemmLaunch g{};
    g.kind = GK_ROUTER;
    g.E = L.nr;
    g.T = c.T;
    g.topk = c.k;
    g.d = c.d_model;
    g.F = c.d_ff;
    g.a_ptr = h;
    g.b_ptr = wr;
    g.router_part = ws_at<float>(ws, L.part);
    g.splits = L.splits;
    g.epad = L.epad;
    g.status = ws_at<int>(ws, L.status);
    g.budget = kSpinBudget;
    return cuda_status(launch_gemm(g, s));
}

// The router weights of any variant (moe_router_t without the C type).
struct RouterWeights {
    const void* w;        // [E, d], or W1 [H, d]
    const void* w2;       // [E, H] or NULL
    const float* bias;    // [E] or NULL
    const float* gamma;   // [d] or NULL
    const float* beta;    // [d] or NULL
};

bool router_args_ok(const moe_config_t& c, const RouterWeights& R)
{
    if (!R.w || (c.router_hidden > 0) != (R.w2 != nullptr)) return false;
    if (c.router_norm != MOE_ROUTER_NORM_LAYER && (R.gamma || R.beta)) return false;
    return true;
}

bool router_aligned(const RouterWeights& R)
{
    return aligned(R.w, 16) && (!R.w2 || aligned(R.w2, 16)) && (!R.gamma || aligned(R.gamma, 16)) &&
           (!R.beta || aligned(R.beta, 16));
}

// The router front end up to the logits: the normalisation (into L.xn), the
// router GEMM on h or on it, and for the two-layer router the head that
// writes z (with the bias) into L.zr.  Returns in *logits where the route
// step finds the logits (L.zr), or NULL when it sums the GEMM partials itself
// (and adds the bias).
moe_status_t run_router_front(const moe_config_t& c, const WsLayout& L, const void* h,
                              const RouterWeights& R, void* ws, cudaStream_t s, const float** logits)
{
    const void* x = h;
    if (c.router_norm != MOE_ROUTER_NORM_NONE) {
        const float eps = c.norm_eps;
        if (launch_router_norm(c.T, c.d_model, static_cast<int>(c.router_norm), eps, h, R.gamma, R.beta,
                               ws_at<void>(ws, L.xn), s) != cudaSuccess)
            return MOE_ERR_CUDA;
        x = ws_at<void>(ws, L.xn);
    }
    moe_status_t st = run_router_gemm(c, L, x, R.w, ws, s);
    if (st != MOE_OK) return st;
    *logits = nullptr;
    if (c.router_hidden > 0) {
        float* z = ws_at<float>(ws, L.zr);
        if (launch_router_head(c.T, c.E, c.router_hidden, L.splits, ws_at<float>(ws, L.part), R.w2, R.bias,
                               z, s) != cudaSuccess)
            return MOE_ERR_CUDA;
        *logits = z;
    }
    return MOE_OK;
}

RouteArgs route_args(const moe_config_t& c, const WsLayout& L, const float* bias,
                     const float* usage, const float* logits_in, float* logits_out,
                     float* scores_out, int32_t* ids_user, float* topk_w, void* ws)
{
    RouteArgs a{};
    a.T = c.T;
    a.E = c.E;
    a.k = c.k;
    a.d = c.d_model;
    a.splits = L.splits;
    a.epad = L.epad;
    a.nchunks = L.nchunks;
    a.part = logits_in ? nullptr : ws_at<float>(ws, L.part);
    a.logits_in = logits_in;
    a.bias = logits_in ? nullptr : bias;
    a.usage = usage;
    a.lambda = c.lambda;
    a.tau = c.tau;
    a.logits_out = logits_out;
    a.scores_user = scores_out;
    a.scores_ws = ws_at<float>(ws, L.scores);
    a.ids_user = ids_user;
    a.topk_w = topk_w;
    a.ids_ws = ws_at<int32_t>(ws, L.ids);
    a.prefs = ws_at<uint8_t>(ws, L.prefs);
    a.crank = ws_at<int32_t>(ws, L.crank);
    a.hist = ws_at<int32_t>(ws, L.hist);
    a.ppart = ws_at<float>(ws, L.ppart);
    a.status = ws_at<int>(ws, L.status);
    return a;
}

moe_status_t run_route(const moe_config_t& c, const WsLayout& L, const void* h, const void* wr,
                       const float* bias, const float* usage, const float* logits_in,
                       float* logits_out, float* scores_out, int32_t* ids_user, float* topk_w,
                       void* ws, cudaStream_t s)
{
    if (!logits_in) {
        moe_status_t st = run_router_gemm(c, L, h, wr, ws, s);
        if (st != MOE_OK) return st;
    }
    return cuda_status(launch_route(route_args(c, L, bias, usage, logits_in, logits_out,
                                               scores_out, ids_user, topk_w, ws),
                                    s));
}

moe_status_t run_stats(const moe_config_t& c, const WsLayout& L, int32_t* counts_pre, float* f,
                       float* P, void* ws, cudaStream_t s)
{
    if (!counts_pre && !f && !P) return MOE_OK;
    StatsArgs a{};
    a.T = c.T;
    a.E = c.E;
    a.k = c.k;
    a.nchunks = L.nchunks;
    a.hist = ws_at<int32_t>(ws, L.hist);
    a.ppart = ws_at<float>(ws, L.ppart);
    a.counts_pre = counts_pre;
    a.f = f;
    a.P = P;
    return cuda_status(launch_route_stats(a, s));
}

struct DispatchOut {
    int32_t *assign, *slot, *counts, *offsets, *perm;
    uint8_t* flags;
    float* cw;
    int32_t *n_rerouted, *n_dropped;
};

DispatchArgs dispatch_args(const moe_config_t& c, const WsLayout& L, const float* scores,
                           const DispatchOut& o, void* ws)
{
    DispatchArgs a{};
    a.T = c.T;
    a.E = c.E;
    a.k = c.k;
    a.nchunks = L.nchunks;
    a.C = capacity_of(c);
    a.scores = scores;
    a.ids = ws_at<int32_t>(ws, L.ids);
    a.prefs = ws_at<uint8_t>(ws, L.prefs);
    a.crank = ws_at<int32_t>(ws, L.crank);
    a.hist = ws_at<int32_t>(ws, L.hist);
    a.base = ws_at<int32_t>(ws, L.base);
    a.ctrl = ws_at<int32_t>(ws, L.ctrl);
    a.assign = o.assign;
    a.slot = o.slot;
    a.flags = o.flags;
    a.counts = o.counts;
    a.offsets = o.offsets;
    a.perm = o.perm;
    a.cw = o.cw;
    a.n_rerouted = o.n_rerouted;
    a.n_dropped = o.n_dropped;
    a.status = ws_at<int>(ws, L.status);
    return a;
}

moe_status_t run_dispatch(const moe_config_t& c, const WsLayout& L, const float* scores,
                          const DispatchOut& o, void* ws, cudaStream_t s)
{
    return cuda_status(launch_dispatch(dispatch_args(c, L, scores, o, ws), s));
}

GemmLaunch expert_gemm(const moe_config_t& c, const WsLayout& L, int kind, void* ws)
{
    GemmLaunch g{};
    g.kind = kind;
    g.E = c.E;
    g.T = c.T;
    g.topk = c.k;
    g.d = c.d_model;
    g.F = c.d_ff;
    g.status = ws_at<int>(ws, L.status);
    g.budget = kSpinBudget;
    g.rows_cap = capacity_of(c);
    return g;
}

}  // namespace
}  // namespace moe

namespace moe {
namespace {

// Expert weights: bf16, e4m3 with one fp32 scale per weight row (s13, s2
// non-NULL), or NVFP4 (b13, b2 non-NULL too: e2m1 codes with e4m3 scales per
// 16 elements and an fp32 scale per row; W13 in the 128-row packing).
struct ExpertWeights {
    const void* w13;
    const void* w2;
    const float* s13;
    const float* s2;
    const void* b13 = nullptr;
    const void* b2 = nullptr;
    bool fp8() const { return s13 != nullptr && b13 == nullptr; }
    bool fp4() const { return b13 != nullptr; }
    void apply(GemmLaunch& g, bool gate_up) const
    {
        g.b_ptr = gate_up ? w13 : w2;
        g.fp8 = fp8() ? 1 : 0;
        g.b_scale = gate_up ? s13 : s2;
    }
};

// NVFP4 weights: every pointer given, the workspace sized for them, and the
// shapes the 4-bit GEMM takes (d a multiple of 128, rows of at most 16384).
moe_status_t check_fp4(const moe_config_t& c, const ExpertWeights& W)
{
    if (!W.fp4()) return MOE_OK;
    if (!W.s13 || !W.s2 || !W.b2 || !(c.flags & MOE_FLAG_NVFP4)) return MOE_ERR_INVALID_ARG;
    if (!aligned(W.b13, 16) || !aligned(W.b2, 16)) return MOE_ERR_MISALIGNED;
    if (c.d_model % 128 != 0 || c.d_model > 16384 || c.d_ff > 16384) return MOE_ERR_UNSUPPORTED;
    return MOE_OK;
}

// The two expert GEMMs over the kept slots: gather (and, with e4m3 weights,
// quantise per row) the token rows, gate-up + SwiGLU into act, (quantise act
// per row,) down into y_slots.  Stage marks after the gather and after gate-up.
moe_status_t run_experts(const moe_config_t& c, const WsLayout& L, const void* h, const int32_t* perm,
                         const int32_t* offsets, const ExpertWeights& W, void* y_slots, void* ws,
                         cudaStream_t s, const Ev* ev)
{
    const size_t rows = static_cast<size_t>(c.T) * c.k;
    void* xg = ws_at<void>(ws, L.xg);
    void* act = ws_at<void>(ws, L.act);
    const int32_t* kept = offsets + c.E;   // device count of kept rows
    if (W.fp4()) {
        // token rows of the kept slots quantised per row; gate-up + SwiGLU; the
        // activation rows quantised per row (their maxima from the gate-up); down
        float* amax = ws_at<float>(ws, L.act_amax);
        if (launch_quantize_nvfp4(static_cast<long long>(rows), c.d_model, h, perm, c.k, 0, kept, nullptr,
                                  ws_at<void>(ws, L.x4), ws_at<void>(ws, L.x4_sf), ws_at<float>(ws, L.x4_scale),
                                  amax, s) != cudaSuccess)
            return MOE_ERR_CUDA;
        if (ev) ev->mark(3);
        F4Launch g{};
        g.kind = GK_GATEUP;
        g.E = c.E;
        g.T = c.T;
        g.topk = c.k;
        g.d = c.d_model;
        g.F = c.d_ff;
        g.a_codes = ws_at<void>(ws, L.x4);
        g.a_sf = ws_at<void>(ws, L.x4_sf);
        g.a_scale = ws_at<float>(ws, L.x4_scale);
        g.b_codes = W.w13;
        g.b_sf = W.b13;
        g.b_scale = W.s13;
        g.offsets = offsets;
        g.act = act;
        g.act_amax = amax;
        g.status = ws_at<int>(ws, L.status);
        g.budget = kSpinBudget;
        g.rows_cap = capacity_of(c);
        if (launch_gemm_nvfp4(g, s) != cudaSuccess) return MOE_ERR_CUDA;
        if (ev) ev->mark(4);
        if (launch_quantize_nvfp4(static_cast<long long>(rows), c.d_ff, act, nullptr, 1, 0, kept, amax,
                                  ws_at<void>(ws, L.a4), ws_at<void>(ws, L.a4_sf), ws_at<float>(ws, L.a4_scale),
                                  nullptr, s) != cudaSuccess)
            return MOE_ERR_CUDA;
        g.kind = GK_DOWN_SLOTS;
        g.a_codes = ws_at<void>(ws, L.a4);
        g.a_sf = ws_at<void>(ws, L.a4_sf);
        g.a_scale = ws_at<float>(ws, L.a4_scale);
        g.b_codes = W.w2;
        g.b_sf = W.b2;
        g.b_scale = W.s2;
        g.act = nullptr;
        g.act_amax = nullptr;
        g.y_slots = y_slots;
        return cuda_status(launch_gemm_nvfp4(g, s));
    }
    if (W.fp8()) {
        if (launch_quantize_fp8(static_cast<long long>(rows), c.d_model, h, perm, c.k, kept, xg,
                                ws_at<float>(ws, L.x_scale), s, nullptr, ws_at<float>(ws, L.act_amax)) !=
            cudaSuccess)
            return MOE_ERR_CUDA;
    } else if (launch_gather_rows(c.T, c.d_model, c.k, c.E, h, perm, offsets, xg, s) != cudaSuccess) {
        return MOE_ERR_CUDA;
    }
    if (ev) ev->mark(3);
    GemmLaunch g = expert_gemm(c, L, GK_GATEUP, ws);
    g.a_ptr = xg;
    W.apply(g, true);
    g.a_scale = W.fp8() ? ws_at<float>(ws, L.x_scale) : nullptr;
    g.act_amax = W.fp8() ? ws_at<float>(ws, L.act_amax) : nullptr;   // zeroed by the pass above
    g.offsets = offsets;
    g.perm = perm;
    g.act = act;
    if (c.flags & MOE_FLAG_BACKWARD) g.gu_save = ws_at<void>(ws, L.gu);   // kept for moe_layer_backward
    if (launch_gemm(g, s) != cudaSuccess) return MOE_ERR_CUDA;
    if (ev) ev->mark(4);
    GemmLaunch g2 = expert_gemm(c, L, GK_DOWN_SLOTS, ws);
    g2.a_ptr = act;
    W.apply(g2, false);
    if (W.fp8()) {
        void* act_q = ws_at<void>(ws, L.act_q);
        if (launch_quantize_fp8(static_cast<long long>(rows), c.d_ff, act, nullptr, 1, kept, act_q,
                                ws_at<float>(ws, L.act_scale), s, ws_at<float>(ws, L.act_amax)) != cudaSuccess)
            return MOE_ERR_CUDA;
        g2.a_ptr = act_q;
        g2.a_scale = ws_at<float>(ws, L.act_scale);
    }
    g2.offsets = offsets;
    g2.perm = perm;
    g2.y_slots = y_slots;
    return cuda_status(launch_gemm(g2, s));
}

moe_status_t expert_ffn_impl(const moe_config_t* cfg, const void* h, const int32_t* perm,
                             const int32_t* offsets, const ExpertWeights& W, void* y_slots, void* ws,
                             size_t ws_bytes, void* stream)
{
    moe_status_t st = check_config(cfg, true);
    if (st != MOE_OK) return st;
    const void* w13 = W.w13;
    const void* w2 = W.w2;
    if (!h || !perm || !offsets || !w13 || !w2 || !y_slots) return MOE_ERR_INVALID_ARG;
    if (W.fp8() && (!W.s2 || !(cfg->flags & MOE_FLAG_FP8) || cfg->d_model % 128 != 0))
        return W.s2 && (cfg->flags & MOE_FLAG_FP8) ? MOE_ERR_UNSUPPORTED : MOE_ERR_INVALID_ARG;
    st = check_fp4(*cfg, W);
    if (st != MOE_OK) return st;
    if (!aligned(h, 16) || !aligned(w13, 16) || !aligned(w2, 16) || !aligned(y_slots, 16))
        return MOE_ERR_MISALIGNED;
    WsLayout L;
    st = check_ws(cfg, ws, ws_bytes, &L);
    if (st != MOE_OK) return st;
    if (cfg->T == 0) return MOE_OK;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    return run_experts(*cfg, L, h, perm, offsets, W, y_slots, ws, s, nullptr);
}

moe_status_t layer_forward_impl(const moe_config_t* cfg, const void* h, const RouterWeights& R,
                                const float* usage, const ExpertWeights& W, void* out,
                                float* logits_out, int32_t* assign, int32_t* slot, uint8_t* flags,
                                int32_t* counts, float* f, float* P, void* const* stage_events, void* ws,
                                size_t ws_bytes, void* stream)
{
    const void* w13 = W.w13;
    const void* w2 = W.w2;
    moe_status_t st = check_config(cfg, true);
    if (st != MOE_OK) return st;
    if (W.fp8() && (!(cfg->flags & MOE_FLAG_FP8) || cfg->d_model % 128 != 0))
        return (cfg->flags & MOE_FLAG_FP8) ? MOE_ERR_UNSUPPORTED : MOE_ERR_INVALID_ARG;
    st = check_fp4(*cfg, W);
    if (st != MOE_OK) return st;
    if (!h || !w13 || !w2 || !out || !router_args_ok(*cfg, R)) return MOE_ERR_INVALID_ARG;
    if (!aligned(h, 16) || !router_aligned(R) || !aligned(w13, 16) || !aligned(w2, 16) || !aligned(out, 16))
        return MOE_ERR_MISALIGNED;
    WsLayout L;
    st = check_ws(cfg, ws, ws_bytes, &L);
    if (st != MOE_OK) return st;
    if (cfg->T == 0) return MOE_OK;
    const moe_config_t& c = *cfg;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    Ev ev{stage_events, s};

    ev.mark(0);
    const float* zr = nullptr;
    st = run_router_front(c, L, h, R, ws, s, &zr);
    if (st != MOE_OK) return st;
    const RouteArgs ra =
        route_args(c, L, R.bias, usage, zr, logits_out, nullptr, nullptr, nullptr, ws);
    // a batch of one chunk routes and dispatches in one kernel (the route stage
    // then holds only the router GEMM, the dispatch stage both)
    const bool small = L.nchunks == 1;
    if (!small && launch_route(ra, s) != cudaSuccess) return MOE_ERR_CUDA;
    ev.mark(1);
    DispatchOut o;
    o.assign = assign ? assign : ws_at<int32_t>(ws, L.assign);
    o.slot = slot ? slot : ws_at<int32_t>(ws, L.slot);
    o.flags = flags ? flags : ws_at<uint8_t>(ws, L.flags);
    o.counts = counts ? counts : ws_at<int32_t>(ws, L.counts);
    o.offsets = ws_at<int32_t>(ws, L.offsets);
    o.perm = ws_at<int32_t>(ws, L.perm);
    o.cw = ws_at<float>(ws, L.cw);
    o.n_rerouted = nullptr;
    o.n_dropped = nullptr;
    const DispatchArgs da = dispatch_args(c, L, ws_at<float>(ws, L.scores), o, ws);
    if (cudaError_t e = small ? launch_route_dispatch_small(ra, da, s) : launch_dispatch(da, s);
        e != cudaSuccess)
        return MOE_ERR_CUDA;
    st = run_stats(c, L, nullptr, f, P, ws, s);
    if (st != MOE_OK) return st;
    ev.mark(2);
    st = run_experts(c, L, h, o.perm, o.offsets, W, ws_at<void>(ws, L.y_slots), ws, s, &ev);
    if (st != MOE_OK) return st;
    ev.mark(5);
    if (launch_combine(c.T, c.d_model, c.k, ws_at<void>(ws, L.y_slots), o.assign, o.slot, o.offsets, o.cw,
                       out, s) != cudaSuccess)
        return MOE_ERR_CUDA;
    ev.mark(6);
    return MOE_OK;
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" {

int64_t moe_capacity(int64_t T, int32_t k, int32_t E, double cf, int32_t explicit_cap)
{
    if (explicit_cap > 0) return explicit_cap;
    if (T <= 0 || k <= 0 || E <= 0 || !(cf > 0.0) || cf > 100.0) return 0;
    const long long cf_micro = llround(cf * 1e6);  // cf as a decimal, 6 fractional digits
    const long long num = static_cast<long long>(T) * k * cf_micro;
    const long long den = static_cast<long long>(E) * 1000000LL;
    return (num + den - 1) / den;
}

size_t moe_workspace_size(const moe_config_t* cfg)
{
    if (check_config(cfg, cfg && cfg->d_ff > 0) != MOE_OK) return 0;
    WsLayout L;
    if (!layout_for(*cfg, &L)) return 0;
    return L.total;
}

moe_status_t moe_workspace_init(void* ws, size_t ws_bytes, void* stream)
{
    if (!ws || ws_bytes < 256) return MOE_ERR_INVALID_ARG;
    if (!aligned(ws, 256)) return MOE_ERR_MISALIGNED;
    return cuda_status(cudaMemsetAsync(ws, 0, 256, static_cast<cudaStream_t>(stream)));
}

moe_status_t moe_get_device_status(void* ws, void* stream)
{
    if (!ws) return MOE_ERR_INVALID_ARG;
    if (!aligned(ws, 256)) return MOE_ERR_MISALIGNED;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int host = 0;
    if (cudaMemcpyAsync(&host, ws, sizeof(int), cudaMemcpyDeviceToHost, s) != cudaSuccess)
        return MOE_ERR_CUDA;
    if (cudaMemsetAsync(ws, 0, sizeof(int), s) != cudaSuccess) return MOE_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return MOE_ERR_CUDA;
    return static_cast<moe_status_t>(host);
}

const char* moe_status_string(moe_status_t st)
{
    switch (st) {
        case MOE_OK: return "ok";
        case MOE_ERR_INVALID_ARG: return "invalid argument";
        case MOE_ERR_UNSUPPORTED: return "unsupported shape";
        case MOE_ERR_MISALIGNED: return "misaligned pointer";
        case MOE_ERR_WORKSPACE: return "workspace too small";
        case MOE_ERR_NONFINITE: return "non-finite (NaN) score";
        case MOE_ERR_TIMEOUT: return "bounded device wait timed out";
        case MOE_ERR_CUDA: return "CUDA runtime error";
    }
    return "unknown status";
}

moe_status_t moe_pack_w13(int32_t E, int32_t F, int32_t d, const void* w1, const void* w3,
                          void* w13, void* stream)
{
    if (E <= 0 || F <= 0 || d <= 0 || !w1 || !w3 || !w13) return MOE_ERR_INVALID_ARG;
    if (F % 128 != 0 || d % 64 != 0 || E > kMaxE) return MOE_ERR_UNSUPPORTED;
    if (!aligned(w1, 16) || !aligned(w3, 16) || !aligned(w13, 16)) return MOE_ERR_MISALIGNED;
    return cuda_status(launch_pack_w13(E, F, d, w1, w3, w13, static_cast<cudaStream_t>(stream)));
}

moe_status_t moe_route(const moe_config_t* cfg, const void* h, const void* w_router,
                       const float* bias, const float* usage, const float* logits_in,
                       float* logits_out, float* scores_out, int32_t* topk_ids, float* topk_w,
                       int32_t* counts_pre, float* f, float* P, void* ws, size_t ws_bytes,
                       void* stream)
{
    moe_status_t st = check_config(cfg, false);
    if (st != MOE_OK) return st;
    if (!topk_ids) return MOE_ERR_INVALID_ARG;
    if (!logits_in && (!h || !w_router)) return MOE_ERR_INVALID_ARG;
    if (!logits_in && (cfg->router_norm != MOE_ROUTER_NORM_NONE || cfg->router_hidden != 0))
        return MOE_ERR_INVALID_ARG;   // those routers' logits come from moe_router_logits
    if (!logits_in && (!aligned(h, 16) || !aligned(w_router, 16))) return MOE_ERR_MISALIGNED;
    WsLayout L;
    st = check_ws(cfg, ws, ws_bytes, &L);
    if (st != MOE_OK) return st;
    if (cfg->T == 0) return MOE_OK;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    st = run_route(*cfg, L, h, w_router, bias, usage, logits_in, logits_out, scores_out, topk_ids,
                   topk_w, ws, s);
    if (st != MOE_OK) return st;
    return run_stats(*cfg, L, counts_pre, f, P, ws, s);
}

moe_status_t moe_dispatch(const moe_config_t* cfg, const float* scores, int32_t* assign,
                          int32_t* slot, uint8_t* flags, int32_t* counts, int32_t* offsets,
                          int32_t* perm, float* combine_w, int32_t* n_rerouted,
                          int32_t* n_dropped, void* ws, size_t ws_bytes, void* stream)
{
    moe_status_t st = check_config(cfg, false);
    if (st != MOE_OK) return st;
    if (!scores || !assign || !slot || !flags || !counts || !offsets || !perm || !combine_w ||
        !n_rerouted || !n_dropped)
        return MOE_ERR_INVALID_ARG;
    WsLayout L;
    st = check_ws(cfg, ws, ws_bytes, &L);
    if (st != MOE_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cfg->T == 0) {
        // nothing to place: zero counts/offsets and the two totals
        if (cudaMemsetAsync(counts, 0, sizeof(int32_t) * cfg->E, s) != cudaSuccess ||
            cudaMemsetAsync(offsets, 0, sizeof(int32_t) * (cfg->E + 1), s) != cudaSuccess ||
            cudaMemsetAsync(n_rerouted, 0, sizeof(int32_t), s) != cudaSuccess ||
            cudaMemsetAsync(n_dropped, 0, sizeof(int32_t), s) != cudaSuccess)
            return MOE_ERR_CUDA;
        return MOE_OK;
    }
    // preference prefixes, chunk histograms and ranks of the given scores
    RouteArgs a{};
    a.T = cfg->T;
    a.E = cfg->E;
    a.k = cfg->k;
    a.d = cfg->d_model;
    a.splits = L.splits;
    a.epad = L.epad;
    a.nchunks = L.nchunks;
    a.logits_in = scores;
    a.ids_ws = ws_at<int32_t>(ws, L.ids);
    a.prefs = ws_at<uint8_t>(ws, L.prefs);
    a.crank = ws_at<int32_t>(ws, L.crank);
    a.hist = ws_at<int32_t>(ws, L.hist);
    a.ppart = ws_at<float>(ws, L.ppart);
    a.status = ws_at<int>(ws, L.status);
    DispatchOut o{assign, slot, counts, offsets, perm, flags, combine_w, n_rerouted, n_dropped};
    if (L.nchunks == 1)
        return cuda_status(
            launch_route_dispatch_small(a, dispatch_args(*cfg, L, scores, o, ws), s));
    if (launch_route(a, s) != cudaSuccess) return MOE_ERR_CUDA;
    return run_dispatch(*cfg, L, scores, o, ws, s);
}


moe_status_t moe_expert_ffn(const moe_config_t* cfg, const void* h, const int32_t* perm,
                            const int32_t* offsets, const void* w13, const void* w2,
                            void* y_slots, void* ws, size_t ws_bytes, void* stream)
{
    return expert_ffn_impl(cfg, h, perm, offsets, ExpertWeights{w13, w2, nullptr, nullptr}, y_slots, ws,
                           ws_bytes, stream);
}

moe_status_t moe_expert_ffn_fp8(const moe_config_t* cfg, const void* h, const int32_t* perm,
                                const int32_t* offsets, const void* w13_q, const float* w13_scale,
                                const void* w2_q, const float* w2_scale, void* y_slots, void* ws,
                                size_t ws_bytes, void* stream)
{
    if (!w13_scale || !w2_scale) return MOE_ERR_INVALID_ARG;
    return expert_ffn_impl(cfg, h, perm, offsets, ExpertWeights{w13_q, w2_q, w13_scale, w2_scale}, y_slots,
                           ws, ws_bytes, stream);
}

moe_status_t moe_quantize_fp8(int64_t rows, int32_t cols, const void* w, void* q, float* scales,
                              void* stream)
{
    if (rows < 0 || cols <= 0 || cols % 8 != 0) return MOE_ERR_INVALID_ARG;
    if (rows == 0) return MOE_OK;
    if (!w || !q || !scales) return MOE_ERR_INVALID_ARG;
    if (!aligned(w, 16) || !aligned(q, 8)) return MOE_ERR_MISALIGNED;
    return cuda_status(
        launch_quantize_fp8(rows, cols, w, nullptr, 1, nullptr, q, scales, static_cast<cudaStream_t>(stream)));
}

int32_t moe_nvfp4_sf_stride(int32_t cols) { return cols > 0 ? nvfp4_sf_stride(cols) : 0; }

moe_status_t moe_quantize_nvfp4(int64_t rows, int32_t cols, const void* w, void* codes, void* bscale,
                                float* scales, void* stream)
{
    if (rows < 0 || cols <= 0 || cols % 32 != 0) return MOE_ERR_INVALID_ARG;
    if (cols > 16384) return MOE_ERR_UNSUPPORTED;
    if (rows == 0) return MOE_OK;
    if (!w || !codes || !bscale || !scales) return MOE_ERR_INVALID_ARG;
    if (!aligned(w, 16) || !aligned(codes, 16) || !aligned(bscale, 16)) return MOE_ERR_MISALIGNED;
    return cuda_status(launch_quantize_nvfp4(rows, cols, w, nullptr, 1, 0, nullptr, nullptr, codes, bscale, scales,
                                             nullptr, static_cast<cudaStream_t>(stream)));
}

moe_status_t moe_quantize_w13_nvfp4(int32_t E, int32_t d_ff, int32_t d_model, const void* w13, void* codes,
                                    void* bscale, float* scales, void* stream)
{
    if (E <= 0 || d_ff <= 0 || d_ff % 128 != 0 || d_model <= 0 || d_model % 32 != 0) return MOE_ERR_INVALID_ARG;
    if (d_model > 16384) return MOE_ERR_UNSUPPORTED;
    if (!w13 || !codes || !bscale || !scales) return MOE_ERR_INVALID_ARG;
    if (!aligned(w13, 16) || !aligned(codes, 16) || !aligned(bscale, 16)) return MOE_ERR_MISALIGNED;
    return cuda_status(launch_quantize_nvfp4(static_cast<long long>(E) * 2 * d_ff, d_model, w13, nullptr, 1, d_ff,
                                             nullptr, nullptr, codes, bscale, scales, nullptr,
                                             static_cast<cudaStream_t>(stream)));
}

moe_status_t moe_expert_ffn_nvfp4(const moe_config_t* cfg, const void* h, const int32_t* perm,
                                  const int32_t* offsets, const void* w13_q, const void* w13_bscale,
                                  const float* w13_scale, const void* w2_q, const void* w2_bscale,
                                  const float* w2_scale, void* y_slots, void* ws, size_t ws_bytes, void* stream)
{
    if (!w13_scale || !w2_scale || !w13_bscale || !w2_bscale) return MOE_ERR_INVALID_ARG;
    return expert_ffn_impl(cfg, h, perm, offsets,
                           ExpertWeights{w13_q, w2_q, w13_scale, w2_scale, w13_bscale, w2_bscale}, y_slots, ws,
                           ws_bytes, stream);
}

moe_status_t moe_layer_forward_nvfp4(const moe_config_t* cfg, const void* h, const void* w_router,
                                     const float* bias, const float* usage, const void* w13_q,
                                     const void* w13_bscale, const float* w13_scale, const void* w2_q,
                                     const void* w2_bscale, const float* w2_scale, void* out, float* logits_out,
                                     int32_t* assign, int32_t* slot, uint8_t* flags, int32_t* counts, float* f,
                                     float* P, void* const* stage_events, void* ws, size_t ws_bytes, void* stream)
{
    if (!w13_scale || !w2_scale || !w13_bscale || !w2_bscale) return MOE_ERR_INVALID_ARG;
    if (cfg && (cfg->router_norm != MOE_ROUTER_NORM_NONE || cfg->router_hidden != 0))
        return MOE_ERR_INVALID_ARG;
    return layer_forward_impl(cfg, h, RouterWeights{w_router, nullptr, bias, nullptr, nullptr}, usage,
                              ExpertWeights{w13_q, w2_q, w13_scale, w2_scale, w13_bscale, w2_bscale}, out,
                              logits_out, assign, slot, flags, counts, f, P, stage_events, ws, ws_bytes, stream);
}

moe_status_t moe_combine(const moe_config_t* cfg, const void* y_slots, const int32_t* assign,
                         const int32_t* slot, const int32_t* offsets, const float* combine_w,
                         void* out, void* stream)
{
    moe_status_t st = check_config(cfg, false);
    if (st != MOE_OK) return st;
    if (!y_slots || !assign || !slot || !offsets || !combine_w || !out) return MOE_ERR_INVALID_ARG;
    if (!aligned(y_slots, 16) || !aligned(out, 16)) return MOE_ERR_MISALIGNED;
    if (cfg->T == 0) return MOE_OK;
    return cuda_status(launch_combine(cfg->T, cfg->d_model, cfg->k, y_slots, assign, slot, offsets,
                                      combine_w, out, static_cast<cudaStream_t>(stream)));
}

moe_status_t moe_layer_forward(const moe_config_t* cfg, const void* h, const void* w_router,
                               const float* bias, const float* usage, const void* w13,
                               const void* w2, void* out, float* logits_out, int32_t* assign,
                               int32_t* slot, uint8_t* flags, int32_t* counts, float* f, float* P,
                               void* const* stage_events, void* ws, size_t ws_bytes, void* stream)
{
    if (cfg && (cfg->router_norm != MOE_ROUTER_NORM_NONE || cfg->router_hidden != 0))
        return MOE_ERR_INVALID_ARG;
    return layer_forward_impl(cfg, h, RouterWeights{w_router, nullptr, bias, nullptr, nullptr}, usage,
                              ExpertWeights{w13, w2, nullptr, nullptr}, out, logits_out, assign, slot, flags,
                              counts, f, P, stage_events, ws, ws_bytes, stream);
}

moe_status_t moe_layer_forward_fp8(const moe_config_t* cfg, const void* h, const void* w_router,
                                   const float* bias, const float* usage, const void* w13_q,
                                   const float* w13_scale, const void* w2_q, const float* w2_scale,
                                   void* out, float* logits_out, int32_t* assign, int32_t* slot,
                                   uint8_t* flags, int32_t* counts, float* f, float* P,
                                   void* const* stage_events, void* ws, size_t ws_bytes, void* stream)
{
    if (!w13_scale || !w2_scale) return MOE_ERR_INVALID_ARG;
    if (cfg && (cfg->router_norm != MOE_ROUTER_NORM_NONE || cfg->router_hidden != 0))
        return MOE_ERR_INVALID_ARG;
    return layer_forward_impl(cfg, h, RouterWeights{w_router, nullptr, bias, nullptr, nullptr}, usage,
                              ExpertWeights{w13_q, w2_q, w13_scale, w2_scale}, out, logits_out, assign, slot,
                              flags, counts, f, P, stage_events, ws, ws_bytes, stream);
}

moe_status_t moe_router_logits(const moe_config_t* cfg, const void* h, const moe_router_t* router,
                               float* logits, void* ws, size_t ws_bytes, void* stream)
{
    moe_status_t st = check_config(cfg, false);
    if (st != MOE_OK) return st;
    if (!h || !router || !logits) return MOE_ERR_INVALID_ARG;
    const RouterWeights R{router->w, router->w2, router->bias, router->norm_gamma, router->norm_beta};
    if (!router_args_ok(*cfg, R)) return MOE_ERR_INVALID_ARG;
    if (!aligned(h, 16) || !router_aligned(R)) return MOE_ERR_MISALIGNED;
    WsLayout L;
    st = check_ws(cfg, ws, ws_bytes, &L);
    if (st != MOE_OK) return st;
    if (cfg->T == 0) return MOE_OK;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const float* zr = nullptr;
    st = run_router_front(*cfg, L, h, R, ws, s, &zr);
    if (st != MOE_OK) return st;
    if (zr)
        return cuda_status(cudaMemcpyAsync(logits, zr, sizeof(float) * cfg->T * cfg->E,
                                           cudaMemcpyDeviceToDevice, s));
    return cuda_status(launch_router_sum(cfg->T, cfg->E, L.splits, ws_at<float>(ws, L.part), R.bias, logits, s));
}

moe_status_t moe_layer_forward_router(const moe_config_t* cfg, const void* h, const moe_router_t* router,
                                      const float* usage, const void* w13, const float* w13_scale,
                                      const void* w2, const float* w2_scale, void* out, float* logits_out,
                                      int32_t* assign, int32_t* slot, uint8_t* flags, int32_t* counts,
                                      float* f, float* P, void* const* stage_events, void* ws,
                                      size_t ws_bytes, void* stream)
{
    if (!router || (w13_scale == nullptr) != (w2_scale == nullptr)) return MOE_ERR_INVALID_ARG;
    return layer_forward_impl(cfg, h,
                              RouterWeights{router->w, router->w2, router->bias, router->norm_gamma,
                                            router->norm_beta},
                              usage, ExpertWeights{w13, w2, w13_scale, w2_scale}, out, logits_out, assign, slot,
                              flags, counts, f, P, stage_events, ws, ws_bytes, stream);
}

moe_status_t moe_layer_forward_host(const moe_config_t* cfg, const void* h_host,
                                    const void* w_router, const float* bias, const float* usage,
                                    const void* w13, const void* w2, void* out_host, void* ws,
                                    size_t ws_bytes, void* stream)
{
    moe_status_t st = moe_layer_forward_host_async(cfg, h_host, w_router, bias, usage, w13, w2, out_host, ws,
                                                   ws_bytes, stream);
    if (st != MOE_OK || !cfg || cfg->T == 0) return st;
    return cuda_status(cudaStreamSynchronize(static_cast<cudaStream_t>(stream)));
}

moe_status_t moe_layer_forward_host_async(const moe_config_t* cfg, const void* h_host,
                                          const void* w_router, const float* bias, const float* usage,
                                          const void* w13, const void* w2, void* out_host, void* ws,
                                          size_t ws_bytes, void* stream)
{
    moe_status_t st = check_config(cfg, true);
    if (st != MOE_OK) return st;
    if (!h_host || !out_host) return MOE_ERR_INVALID_ARG;
    WsLayout L;
    st = check_ws(cfg, ws, ws_bytes, &L);
    if (st != MOE_OK) return st;
    if (cfg->T == 0) return MOE_OK;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const size_t bytes = static_cast<size_t>(cfg->T) * cfg->d_model * 2;
    void* h_dev = ws_at<void>(ws, L.h_stage);
    void* out_dev = ws_at<void>(ws, L.out_stage);
    if (cudaMemcpyAsync(h_dev, h_host, bytes, cudaMemcpyHostToDevice, s) != cudaSuccess)
        return MOE_ERR_CUDA;
    st = moe_layer_forward(cfg, h_dev, w_router, bias, usage, w13, w2, out_dev, nullptr, nullptr,
                           nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, ws, ws_bytes, stream);
    if (st != MOE_OK) return st;
    return cuda_status(cudaMemcpyAsync(out_host, out_dev, bytes, cudaMemcpyDeviceToHost, s));
}

moe_status_t moe_layer_backward(const moe_config_t* cfg, const void* h, const void* w_router, const void* w13,
                                const void* w2, const void* dout, const float* dP, float* dh, float* dw_router,
                                float* dbias, float* dw13, float* dw2, void* ws, size_t ws_bytes, void* stream)
{
    moe_status_t st = check_config(cfg, true);
    if (st != MOE_OK) return st;
    if (!(cfg->flags & MOE_FLAG_BACKWARD)) return MOE_ERR_INVALID_ARG;
    if (cfg->router_norm != MOE_ROUTER_NORM_NONE || cfg->router_hidden != 0) return MOE_ERR_UNSUPPORTED;
    const bool any = cfg->T > 0;   // with no tokens only the weight gradients (zeros) are written
    if (!w_router || !w13 || !w2 || !dw13 || !dw2 || (any && (!h || !dout || !dh))) return MOE_ERR_INVALID_ARG;
    if (!aligned(w_router, 16) || !aligned(w13, 16) || !aligned(w2, 16) || !aligned(dw13, 16) || !aligned(dw2, 16) ||
        (any && (!aligned(h, 16) || !aligned(dout, 16) || !aligned(dh, 16))))
        return MOE_ERR_MISALIGNED;
    WsLayout L;
    st = check_ws(cfg, ws, ws_bytes, &L);
    if (st != MOE_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const moe_config_t& c = *cfg;
    if (!any) {   // no tokens: every gradient is zero
        const size_t wbytes = static_cast<size_t>(c.E) * c.d_ff * c.d_model * 4;
        if (cudaMemsetAsync(dw13, 0, 2 * wbytes, s) != cudaSuccess || cudaMemsetAsync(dw2, 0, wbytes, s) != cudaSuccess ||
            (dw_router && cudaMemsetAsync(dw_router, 0, sizeof(float) * c.E * c.d_model, s) != cudaSuccess) ||
            (dbias && cudaMemsetAsync(dbias, 0, sizeof(float) * c.E, s) != cudaSuccess))
            return MOE_ERR_CUDA;
        return MOE_OK;
    }
    BackwardArgs a{};
    a.T = c.T;
    a.E = c.E;
    a.k = c.k;
    a.d = c.d_model;
    a.F = c.d_ff;
    a.R = backward_rows(c);
    a.tau = c.tau;
    a.scores = ws_at<float>(ws, L.scores);
    a.perm = ws_at<int32_t>(ws, L.perm);
    a.offsets = ws_at<int32_t>(ws, L.offsets);
    a.cw = ws_at<float>(ws, L.cw);
    a.h = h;
    a.w_router = w_router;
    a.w13 = w13;
    a.w2 = w2;
    a.dout = dout;
    a.gu = ws_at<float>(ws, L.gu);
    a.dP = dP;
    a.dh = dh;
    a.dw_router = dw_router;
    a.dbias = dbias;
    a.dw13 = dw13;
    a.dw2 = dw2;
    a.scratch = ws_at<void>(ws, L.bwd);
    a.status = ws_at<int>(ws, L.status);
    a.budget = kSpinBudget;
    return cuda_status(run_backward(a, s));
}

moe_status_t moe_debug_timeout_probe(void* ws, size_t ws_bytes, int64_t budget_cycles, void* stream)
{
    if (!ws || ws_bytes < 256 || budget_cycles <= 0) return MOE_ERR_INVALID_ARG;
    if (!aligned(ws, 256)) return MOE_ERR_MISALIGNED;
    return cuda_status(
        launch_timeout_probe(static_cast<int*>(ws), budget_cycles, static_cast<cudaStream_t>(stream)));
}

}  // extern "C"
