/*
 * moe.h -- C ABI of the GB300 (sm_103a) MoE-layer forward library, libmoe.so.
 *
 * One sparsely activated Mixture-of-Experts FFN layer, forward only, on one
 * GPU with every expert resident in HBM:
 *
 *   router GEMM -> load penalty -> softmax + top-k -> capacity-capped
 *   dispatch with reroute/drop -> grouped SwiGLU experts -> weighted combine
 *
 * Pages that state the method (cited below by their bracketed key):
 *   [mhpn]     "GPT-4稀疏激活真相：万亿参数模型的MoE工程落地实践"
 *              (www.mhpn.cn/news/895310)
 *   [coreui]   "MoE架构揭秘：逐Token路由与活跃参数量的工程真相"
 *              (www.coreui.cn/article/2635427.html)
 *   [cnnetsun] "MoE稀疏激活原理与工程实践：从2%激活率到高效推理"
 *              (cnnetsun.cn/a/3071834)
 *   [csdn]     untitled page, adg.csdn.net/6a3116e610ee7a33f27ddf1c.html
 *   [2kiu]     MoE page at www.2kiu.com/news/5042631/
 *
 * Conventions for every entry point
 *   - Pointers named *_dev are DEVICE pointers owned by the caller; the
 *     library never allocates or frees device memory, and never synchronises
 *     on the forward or backward path (the lesson of the per-expert
 *     cudaMallocAsync leak on [cnnetsun] §5.2).
 *     All scratch lives in the caller's workspace `ws` (size from
 *     moe_workspace_size, 256-byte aligned, initialised once with
 *     moe_workspace_init).
 *   - `stream` is a cudaStream_t (NULL = legacy default stream).  Calls are
 *     asynchronous and stream-ordered; they enqueue kernels and small memset
 *     nodes only.
 *   - Argument, shape, alignment and workspace errors are returned
 *     synchronously, before anything is enqueued.  Errors detected on the
 *     device (NaN scores, a bounded wait that ran out) set a status word in
 *     the workspace, read with moe_get_device_status.  Kernels never trap.
 *   - bf16 tensors are IEEE bfloat16, row-major, 16-byte aligned.
 *   - Supported: 1 <= k <= 8, k <= E <= 255, d_model % 64 == 0,
 *     d_ff % 128 == 0, T >= 1 (T = 0 is a no-op).
 */
#ifndef MOE_GB300_H
#define MOE_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    MOE_OK = 0,
    MOE_ERR_INVALID_ARG = 1,   /* null required pointer, bad shape or value */
    MOE_ERR_UNSUPPORTED = 2,   /* shape outside the supported set above */
    MOE_ERR_MISALIGNED = 3,    /* a pointer is not 16-byte (ws: 256-byte) aligned */
    MOE_ERR_WORKSPACE = 4,     /* ws_bytes < moe_workspace_size(cfg) */
    MOE_ERR_NONFINITE = 5,     /* device: a score was NaN */
    MOE_ERR_TIMEOUT = 6,       /* device: a bounded wait ran out */
    MOE_ERR_CUDA = 7           /* a CUDA runtime call failed */
} moe_status_t;

/* moe_config_t.flags: size the workspace for the FP8 entry points too (adds
 * T*k*(d_ff + 12) bytes for the e4m3 activation rows, their scales and row
 * maxima). */
#define MOE_FLAG_FP8 1u
/* moe_config_t.flags: size the workspace for moe_layer_backward too (adds
 * about R*(8d + 10F) + T*k*(8F + 8) + 4T*E + 128*E*d bytes, R = min(E*C',
 * T*k + 127E) with C' = min(C, T) rounded up to 128); moe_layer_forward then
 * also keeps each kept row's g and u (fp32) there for the backward. */
#define MOE_FLAG_BACKWARD 2u
/* moe_config_t.flags: size the workspace for the NVFP4 entry points too (adds
 * about T*k*(d/2 + F/2 + d/16 + F/16 + 12) bytes for the 4-bit token and
 * activation rows, their block scales, row scales and row maxima). */
#define MOE_FLAG_NVFP4 4u

/* Layer shape.  Capacity C = ceil(T*k*cf/E) unless capacity > 0. */
typedef struct {
    int32_t T;        /* tokens in the batch */
    int32_t d_model;  /* hidden size d */
    int32_t E;        /* number of experts */
    int32_t k;        /* experts per token (top-k) */
    int32_t d_ff;     /* expert intermediate size F */
    double cf;        /* capacity factor, read as a decimal with 6 fractional digits */
    int32_t capacity; /* > 0: explicit per-expert capacity, overrides cf */
    float lambda;     /* load-penalty weight (0 = no penalty) */
    uint32_t flags;   /* 0, or any of MOE_FLAG_FP8, MOE_FLAG_BACKWARD, MOE_FLAG_NVFP4 */
    /* Router variants (all zero: the plain linear router, no temperature). */
    float tau;              /* temperature, 0 (= 1) or finite > 0: s = z / tau - lambda*usage */
    uint32_t router_norm;   /* MOE_ROUTER_NORM_*: normalisation of h before the router */
    float norm_eps;         /* epsilon of that normalisation, finite >= 0 */
    int32_t router_hidden;  /* 0: linear router; H in [1, 256]: the two-layer router */
} moe_config_t;

/* moe_config_t.router_norm ([2kiu] §5.2: a LayerNorm before the router, or
 * L2-normalised inputs; [mhpn] §3.1: a router that begins with a LayerNorm).
 * Needs d_model <= 16384. */
#define MOE_ROUTER_NORM_NONE 0u
#define MOE_ROUTER_NORM_LAYER 1u   /* (h - mean) / sqrt(var + eps) * gamma + beta, over d */
#define MOE_ROUTER_NORM_L2 2u      /* h / max(||h||_2, eps) */

/* Router weights for the router variants (moe_router_logits,
 * moe_layer_forward_router).  All device pointers, 16-byte aligned.
 *   w           [E, d] bf16, row e = expert e's gate vector; with
 *               router_hidden = H > 0, W1 [H, d] (row j = hidden unit j)
 *   w2          [E, H] bf16 when router_hidden > 0 (else NULL): the two-layer
 *               router z = silu(x . W1^T) . W2^T ([cnnetsun] §3.1 step 2: W1
 *               d x 2E, W2 2E x E); E * H <= 16384
 *   bias        [E] fp32 added to z, or NULL
 *   norm_gamma, norm_beta  [d] fp32 LayerNorm scale and shift, or NULL (1, 0) */
typedef struct {
    const void* w;
    const void* w2;
    const float* bias;
    const float* norm_gamma;
    const float* norm_beta;
} moe_router_t;

/* Number of stage boundaries recorded by moe_layer_forward's stage_events. */
#define MOE_NUM_STAGES 6

/* Expert capacity C = ceil(T*k*cf/E), exact, with cf read as a decimal with
 * six fractional digits ([coreui] §5.2: ceil(batch*top_k/num_experts*1.3);
 * [coreui] §3.3: Capacity = (Batch*K)/N*alpha).  explicit_cap > 0 is
 * returned as is.  Returns 0 for non-positive inputs. */
int64_t moe_capacity(int64_t T, int32_t k, int32_t E, double cf, int32_t explicit_cap);

/* Bytes of workspace that every call with this config needs (0 on a bad
 * config).  The workspace is reusable across calls with the same or a
 * smaller config; calls that share one workspace must not overlap. */
size_t moe_workspace_size(const moe_config_t* cfg);

/* Clears the workspace's device status word.  Call once after allocating a
 * workspace (enqueued on `stream`). */
moe_status_t moe_workspace_init(void* ws_dev, size_t ws_bytes, void* stream);

/* Synchronises `stream`, returns the device status word recorded in `ws`
 * since the last read (MOE_OK if none) and clears it. */
moe_status_t moe_get_device_status(void* ws_dev, void* stream);

/* Human-readable name of a status code (static string). */
const char* moe_status_string(moe_status_t st);

/* Re-lays out the gate and up projections into the fused gate-up operand.
 *   w1_dev, w3_dev  [E, F, d] bf16 (nn.Linear out x in: W1 = gate, W3 = up)
 *   w13_dev         [E, 2F, d] bf16 out.  For each expert, block j of 256
 *                   rows holds W1 rows [128j, 128j+128) followed by W3 rows
 *                   [128j, 128j+128), so one 256-row tile carries matching
 *                   gate and up columns ([mhpn] §3.1, [2kiu] §1: the
 *                   W1/W2/W3 SwiGLU expert).
 * Requires F % 128 == 0, d % 64 == 0. */
moe_status_t moe_pack_w13(int32_t E, int32_t F, int32_t d, const void* w1_dev,
                          const void* w3_dev, void* w13_dev, void* stream);

/* Router: logits, penalised scores, top-k picks and load statistics.
 *   z = h . W_r^T (+ b)                       [coreui] §3.1, [csdn] §3.1
 *   s_i = z_i / tau - lambda * usage_i        [mhpn] §2.3 (second check),
 *     (fp32, the division and the product     [cnnetsun] §3.1 steps 3-4 (tau,
 *     each rounded, no FMA; tau = cfg->tau)    then the penalty, before top-k)
 *   p = softmax(s); picks = the k best s, ties to the lower expert index
 *   f_i = (#picks of i)/T, P_i = mean_t p_i   [cnnetsun] §4.2, [coreui] §3.1
 * Inputs:
 *   h_dev        [T, d] bf16 (ignored when logits_in_dev != NULL)
 *   w_router_dev [E, d] bf16 (row e = expert e's gate vector)
 *   bias_dev     [E] fp32 or NULL        usage_dev [E] fp32 or NULL
 *   logits_in_dev[T, E] fp32 or NULL: final logits given (no GEMM, no bias)
 * Outputs (each may be NULL unless noted):
 *   logits_out_dev [T, E] fp32; scores_out_dev [T, E] fp32 (penalised);
 *   topk_ids_dev [T, k] int32 (required); topk_w_dev [T, k] fp32 (softmax
 *   probability of each pick); counts_pre_dev [E] int32 (picks per expert
 *   before capacity); f_dev [E], P_dev [E] fp32.
 * NaN scores set MOE_ERR_NONFINITE on the device (NaN then ranks last).
 * The plain linear router only: a config with router_norm or router_hidden
 * set returns MOE_ERR_INVALID_ARG unless logits_in_dev is given (use
 * moe_router_logits for those routers' logits). */
moe_status_t moe_route(const moe_config_t* cfg, const void* h_dev, const void* w_router_dev,
                       const float* bias_dev, const float* usage_dev,
                       const float* logits_in_dev, float* logits_out_dev, float* scores_out_dev,
                       int32_t* topk_ids_dev, float* topk_w_dev, int32_t* counts_pre_dev,
                       float* f_dev, float* P_dev, void* ws_dev, size_t ws_bytes, void* stream);

/* Capacity-capped dispatch on penalised scores ([mhpn] §2.3, third check;
 * [2kiu] §2; [coreui] §3.3).  Slots fill in entry order (rank, token): every
 * rank-0 pick before any rank-1 pick, tokens in index order.  An entry takes
 * the first expert of its preference order that is not full and not already
 * serving the token; when none is left it is dropped.
 *   scores_dev [T, E] fp32 (penalised scores, e.g. moe_route's scores_out)
 * Outputs (all required):
 *   assign_dev [T, k] int32 expert used (-1 = dropped); slot_dev [T, k] int32
 *   position in the expert's slot list (-1 = dropped); flags_dev [T, k] u8
 *   (bit0 rerouted, bit1 dropped); counts_dev [E] int32; offsets_dev [E+1]
 *   int32 (exclusive scan of counts); perm_dev [T*k] int32: slot order, entry
 *   perm[offsets[e] + slot] = t*k + r, entries past offsets[E] untouched;
 *   combine_w_dev [T, k] fp32: p of the expert used, renormalised over the
 *   token's kept experts ([mhpn] §4.3), 0 when dropped; n_rerouted_dev [1],
 *   n_dropped_dev [1] int32. */
moe_status_t moe_dispatch(const moe_config_t* cfg, const float* scores_dev, int32_t* assign_dev,
                          int32_t* slot_dev, uint8_t* flags_dev, int32_t* counts_dev,
                          int32_t* offsets_dev, int32_t* perm_dev, float* combine_w_dev,
                          int32_t* n_rerouted_dev, int32_t* n_dropped_dev,
                          void* ws_dev, size_t ws_bytes, void* stream);

/* Grouped SwiGLU experts over the dispatched slots ([mhpn] §3.1; [2kiu] §1;
 * [cnnetsun] §3.2 step 1, tokens grouped into E sub-batches):
 *   for slot i of expert e (offsets[e] <= i < offsets[e+1]), t = perm[i]/k:
 *   y_slots[i] = W2_e (silu(W1_e h_t) * (W3_e h_t))
 *   h_dev [T, d] bf16; perm_dev, offsets_dev as from moe_dispatch;
 *   w13_dev [E, 2F, d] bf16 from moe_pack_w13; w2_dev [E, d, F] bf16;
 *   y_slots_dev [T*k, d] bf16 out (rows past offsets[E] untouched).
 * The intermediate silu(g)*u is rounded to bf16 between the two GEMMs. */
moe_status_t moe_expert_ffn(const moe_config_t* cfg, const void* h_dev, const int32_t* perm_dev,
                            const int32_t* offsets_dev, const void* w13_dev, const void* w2_dev,
                            void* y_slots_dev, void* ws_dev, size_t ws_bytes, void* stream);

/* FP8 expert path.  The pages quantise expert weights to cut the bytes moved
 * ([2kiu] §5.1: INT4/INT6 per expert; [cnnetsun] §3.2: INT8, where a
 * dequantisation step ate the gain -- the bottleneck is moving data).  This
 * library's form runs the expert GEMMs in e4m3 on the tensor cores, with no
 * dequantisation pass: weights are quantised once per row (output channel),
 * token rows and activation rows per row on the fly, the products accumulate
 * in fp32 and the two row scales multiply the result.
 *
 * Per-row quantisation of a bf16 matrix w_dev [rows, cols] (row-major, cols a
 * multiple of 8; w_dev 16-byte aligned, q_dev 8-byte aligned):
 *   scales_dev[r] = max_c |w[r,c]| / 448 (1 for an all-zero row),
 *   q_dev[r,c] = e4m3(w[r,c] / scales[r]), round to nearest even, saturating.
 * Quantise W13 after moe_pack_w13 (rows E*2F, cols d) and W2 (rows E*d,
 * cols F).  Errors: MOE_ERR_INVALID_ARG (rows < 0, cols not a positive
 * multiple of 8, NULL), MOE_ERR_MISALIGNED. */
moe_status_t moe_quantize_fp8(int64_t rows, int32_t cols, const void* w_dev, void* q_dev,
                              float* scales_dev, void* stream);

/* moe_expert_ffn in e4m3: w13_q_dev [E, 2F, d] and w2_q_dev [E, d, F] from
 * moe_quantize_fp8 with w13_scale_dev [E*2F] and w2_scale_dev [E*d] (weight =
 * code * row scale).  Each kept slot's token row is quantised per row the same
 * way, as is each activation row silu(g)*u (after rounding to bf16); both
 * GEMMs multiply e4m3 codes (tcgen05.mma.kind::f8f6f4, fp32 accumulate) and
 * scale by the activation row's and the weight row's scales.  Needs
 * cfg->flags & MOE_FLAG_FP8 (MOE_ERR_INVALID_ARG otherwise) and d a multiple
 * of 128 (MOE_ERR_UNSUPPORTED otherwise); y_slots as moe_expert_ffn. */
moe_status_t moe_expert_ffn_fp8(const moe_config_t* cfg, const void* h_dev, const int32_t* perm_dev,
                                const int32_t* offsets_dev, const void* w13_q_dev,
                                const float* w13_scale_dev, const void* w2_q_dev,
                                const float* w2_scale_dev, void* y_slots_dev, void* ws_dev,
                                size_t ws_bytes, void* stream);

/* Probability-weighted combine back to token order ([mhpn] §4.3; [2kiu] §3
 * step 5): out[t] = sum over kept r, in rank order, of combine_w[t,r] *
 * y_slots[offsets[assign[t,r]] + slot[t,r]]; tokens with nothing kept get 0.
 * Accumulates in fp32, stores bf16.  out_dev [T, d] bf16. */
moe_status_t moe_combine(const moe_config_t* cfg, const void* y_slots_dev,
                         const int32_t* assign_dev, const int32_t* slot_dev,
                         const int32_t* offsets_dev, const float* combine_w_dev, void* out_dev,
                         void* stream);

/* The whole layer in one call, no host synchronisation: router GEMM, route,
 * dispatch, the token rows gathered into slot order, the gate-up GEMM with the
 * SwiGLU in its epilogue, the down GEMM writing each kept entry's output row
 * (bf16) in slot order, and the combine: out[t] = sum over t's kept ranks, in
 * rank order, of combine weight * output row (fp32), rounded to bf16 once.
 *   h_dev [T, d] bf16; w_router_dev [E, d]; bias_dev, usage_dev as in
 *   moe_route; w13_dev [E, 2F, d]; w2_dev [E, d, F]; out_dev [T, d] bf16.
 * Optional outputs (NULL to skip): logits_out [T,E], assign/slot [T,k] int32,
 *   flags [T,k] u8, counts [E] int32, f/P [E] fp32.
 * stage_events: NULL, or MOE_NUM_STAGES+1 cudaEvent_t recorded on `stream`
 *   at the boundaries route | dispatch | prep (gather the token rows in slot
 *   order) | gate-up | down | combine.  For T <= 256 route and dispatch run
 *   as one kernel: the route stage then holds the router GEMM only.
 * The linear router with cfg->tau; router_norm and router_hidden must be 0
 * (MOE_ERR_INVALID_ARG otherwise; moe_layer_forward_router takes those). */
moe_status_t moe_layer_forward(const moe_config_t* cfg, const void* h_dev,
                               const void* w_router_dev, const float* bias_dev,
                               const float* usage_dev, const void* w13_dev, const void* w2_dev,
                               void* out_dev, float* logits_out_dev, int32_t* assign_dev,
                               int32_t* slot_dev, uint8_t* flags_dev, int32_t* counts_dev,
                               float* f_dev, float* P_dev, void* const* stage_events,
                               void* ws_dev, size_t ws_bytes, void* stream);

/* moe_layer_forward with the expert GEMMs in e4m3 (as moe_expert_ffn_fp8);
 * routing, dispatch and the combine are unchanged (the router GEMM stays
 * bf16).  Stage events as moe_layer_forward; the down stage includes the
 * activation quantisation. */
moe_status_t moe_layer_forward_fp8(const moe_config_t* cfg, const void* h_dev,
                                   const void* w_router_dev, const float* bias_dev,
                                   const float* usage_dev, const void* w13_q_dev,
                                   const float* w13_scale_dev, const void* w2_q_dev,
                                   const float* w2_scale_dev, void* out_dev,
                                   float* logits_out_dev, int32_t* assign_dev, int32_t* slot_dev,
                                   uint8_t* flags_dev, int32_t* counts_dev, float* f_dev,
                                   float* P_dev, void* const* stage_events, void* ws_dev,
                                   size_t ws_bytes, void* stream);

/* NVFP4 expert path: 4-bit weights and activations.  A row x[0..n) is held
 * as e2m1 codes (values 0, 0.5, 1, 1.5, 2, 3, 4, 6 with a sign; two per byte,
 * element 2m in the low nibble), one e4m3 scale per 16 consecutive elements
 * (a byte; the scales of a row padded to moe_nvfp4_sf_stride(n) bytes) and
 * one fp32 scale per row, quantised in fp32 steps:
 *   scale = max|x| / 2688 (= 6 * 448; 1 for an all-zero row);
 *   per block: b = e4m3(fl(fl(max|x_i| / scale) / 6)), den = fl(value(b) * scale),
 *   code_i = e2m1(fl(x_i / den)) (nearest, ties to even, saturating; 0 if den = 0);
 *   x_i ~ e2m1(code_i) * value(b) * scale.
 * The pages quantise experts to 4-6 bits ([2kiu] §5.1) to move fewer bytes;
 * the GEMMs multiply the codes on the tensor cores
 * (tcgen05.mma.kind::mxf4nvf4.block_scale, the block scales applied by the
 * MMA, fp32 accumulate) and the epilogue applies the two row scales.
 * moe_nvfp4_sf_stride(cols): bytes per row of block scales (cols/16 rounded up
 * to a multiple of 16). */
int32_t moe_nvfp4_sf_stride(int32_t cols);

/* NVFP4 quantisation of a bf16 matrix w_dev [rows, cols] (row-major; cols a
 * multiple of 32, at most 16384): codes_dev [rows, cols/2] bytes, bscale_dev
 * [rows, moe_nvfp4_sf_stride(cols)] bytes, scales_dev [rows] fp32.  Use it for
 * W2 (rows E*d, cols F).  Pointers 16-byte aligned.  Errors:
 * MOE_ERR_INVALID_ARG, MOE_ERR_UNSUPPORTED (cols > 16384), MOE_ERR_MISALIGNED. */
moe_status_t moe_quantize_nvfp4(int64_t rows, int32_t cols, const void* w_dev, void* codes_dev,
                                void* bscale_dev, float* scales_dev, void* stream);

/* NVFP4 quantisation of W13 [E, 2F, d] in the moe_pack_w13 layout into this
 * path's own packing: per expert, 128-row block j holds W1 rows 64j..64j+63 and
 * then the matching W3 rows, so that one 128-column tile of the 4-bit gate-up
 * GEMM holds matching gate and up columns.  Outputs as moe_quantize_nvfp4 with
 * rows E*2F, cols d (row r of the outputs is row r of the new packing). */
moe_status_t moe_quantize_w13_nvfp4(int32_t E, int32_t d_ff, int32_t d_model, const void* w13_dev,
                                    void* codes_dev, void* bscale_dev, float* scales_dev, void* stream);

/* moe_expert_ffn with NVFP4 weights (w13 from moe_quantize_w13_nvfp4, w2 from
 * moe_quantize_nvfp4): each kept slot's token row and each activation row
 * silu(g)*u (after rounding to bf16) are quantised the same way on the fly,
 * both GEMMs multiply e2m1 codes with their block scales on the tensor cores
 * and scale the result by the two row scales.  Needs cfg->flags &
 * MOE_FLAG_NVFP4 (MOE_ERR_INVALID_ARG otherwise), d a multiple of 128 and d,
 * F at most 16384 (MOE_ERR_UNSUPPORTED otherwise); y_slots as moe_expert_ffn. */
moe_status_t moe_expert_ffn_nvfp4(const moe_config_t* cfg, const void* h_dev, const int32_t* perm_dev,
                                  const int32_t* offsets_dev, const void* w13_q_dev, const void* w13_bscale_dev,
                                  const float* w13_scale_dev, const void* w2_q_dev, const void* w2_bscale_dev,
                                  const float* w2_scale_dev, void* y_slots_dev, void* ws_dev, size_t ws_bytes,
                                  void* stream);

/* moe_layer_forward with the expert GEMMs in NVFP4 (as moe_expert_ffn_nvfp4);
 * routing, dispatch, the combine and the bf16 router GEMM are unchanged.
 * Stage events as moe_layer_forward: the prep stage is the token rows'
 * quantisation, the down stage includes the activation rows'. */
moe_status_t moe_layer_forward_nvfp4(const moe_config_t* cfg, const void* h_dev, const void* w_router_dev,
                                     const float* bias_dev, const float* usage_dev, const void* w13_q_dev,
                                     const void* w13_bscale_dev, const float* w13_scale_dev,
                                     const void* w2_q_dev, const void* w2_bscale_dev, const float* w2_scale_dev,
                                     void* out_dev, float* logits_out_dev, int32_t* assign_dev,
                                     int32_t* slot_dev, uint8_t* flags_dev, int32_t* counts_dev, float* f_dev,
                                     float* P_dev, void* const* stage_events, void* ws_dev, size_t ws_bytes,
                                     void* stream);

/* The router variants' logits: z = front end of cfg applied to h, for the
 * router in `router` (see moe_router_t): normalisation of each token row
 * (cfg->router_norm, cfg->norm_eps; the normalised rows are rounded to bf16
 * for the router GEMM), then the linear router or, with router_hidden = H,
 * the two-layer router (fp32 hidden units, silu, W2 in fp32 accumulation),
 * plus the bias.  logits_dev [T, E] fp32 out.  Feed them to moe_route as
 * logits_in_dev for the route step. */
moe_status_t moe_router_logits(const moe_config_t* cfg, const void* h_dev, const moe_router_t* router,
                               float* logits_dev, void* ws_dev, size_t ws_bytes, void* stream);

/* The whole layer (as moe_layer_forward) with any router variant of cfg
 * (temperature, normalisation, two-layer router) and bf16 or e4m3 experts:
 * w13_scale_dev and w2_scale_dev NULL for bf16 weights, or the row scales of
 * e4m3 weights (as moe_layer_forward_fp8, which needs MOE_FLAG_FP8).  The
 * route stage holds the router front end.  logits_out_dev receives z (before
 * the temperature and the penalty). */
moe_status_t moe_layer_forward_router(const moe_config_t* cfg, const void* h_dev,
                                      const moe_router_t* router, const float* usage_dev,
                                      const void* w13_dev, const float* w13_scale_dev,
                                      const void* w2_dev, const float* w2_scale_dev, void* out_dev,
                                      float* logits_out_dev, int32_t* assign_dev, int32_t* slot_dev,
                                      uint8_t* flags_dev, int32_t* counts_dev, float* f_dev,
                                      float* P_dev, void* const* stage_events, void* ws_dev,
                                      size_t ws_bytes, void* stream);

/* The same layer from host memory, end to end: copies h (pinned host,
 * [T,d] bf16) to the workspace, runs moe_layer_forward and copies the output
 * back to out_host ([T,d] bf16), all on `stream`; returns after the stream
 * has finished.  Weights stay resident on the device. */
moe_status_t moe_layer_forward_host(const moe_config_t* cfg, const void* h_host,
                                    const void* w_router_dev, const float* bias_dev,
                                    const float* usage_dev, const void* w13_dev,
                                    const void* w2_dev, void* out_host,
                                    void* ws_dev, size_t ws_bytes, void* stream);

/* Backward pass of moe_layer_forward (training; not on the forward path).
 * The routing decisions of the forward are held fixed (top-k and capacity are
 * piecewise constant); gradients flow through the experts and through the
 * combine weights cw[t,r] = p[t,e_r] / sum over t's kept ranks of p ([mhpn]
 * §4.3) into the softmax, the temperature and the router GEMM ([coreui] §3.1).
 *   ws_dev    the workspace of the moe_layer_forward call (bf16 experts, the
 *             linear router) whose gradients these are, sized with
 *             MOE_FLAG_BACKWARD, untouched by any other call since: the
 *             forward's scores, kept-slot order, combine weights and the
 *             gate and up projections g, u of each kept row are read from it.
 *   h_dev, w_router_dev, w13_dev, w2_dev   the forward's inputs (bf16)
 *   dout_dev  [T, d] bf16: dL/dout
 *   dP_dev    [E] fp32 or NULL: dL/dP for a load-balancing loss written from
 *             the mean probabilities P_i = mean_t p[t,i] ([coreui] §3.1; e.g.
 *             2*alpha*P_i for alpha * sum_i P_i^2); adds dP_i / T to dL/dp[t,i]
 * Outputs (fp32, overwritten): dh_dev [T, d]; dw_router_dev [E, d] and
 * dbias_dev [E] (each may be NULL); dw13_dev [E, 2F, d] in the packed W13
 * layout (moe_pack_w13); dw2_dev [E, d, F].
 * Each expert's kept rows are gathered into a row block padded with zero
 * rows to a multiple of 128; the four per-expert products (W2^T dL/dout,
 * dL/dx, dW2, dW13) run on this library's tcgen05 GEMM over those blocks and
 * everything else in its other kernels (no library GEMM, no allocation).
 * Requires
 * MOE_FLAG_BACKWARD (MOE_ERR_INVALID_ARG otherwise), router_norm = 0 and
 * router_hidden = 0 (MOE_ERR_UNSUPPORTED otherwise). */
moe_status_t moe_layer_backward(const moe_config_t* cfg, const void* h_dev, const void* w_router_dev,
                                const void* w13_dev, const void* w2_dev, const void* dout_dev,
                                const float* dP_dev, float* dh_dev, float* dw_router_dev,
                                float* dbias_dev, float* dw13_dev, float* dw2_dev, void* ws_dev,
                                size_t ws_bytes, void* stream);

/* moe_layer_forward_host without its final synchronisation: enqueues the copy
 * of h_host into the workspace, the layer, and the copy of the output to
 * out_host on `stream`, and returns.  h_host and out_host are pinned host
 * memory; the caller synchronises the stream (or an event recorded after the
 * call) before reading out_host or changing h_host, and uses ws_dev for no
 * other call until then.  Two workspaces on two streams let one batch's copies
 * overlap another batch's kernels. */
moe_status_t moe_layer_forward_host_async(const moe_config_t* cfg, const void* h_host,
                                          const void* w_router_dev, const float* bias_dev,
                                          const float* usage_dev, const void* w13_dev,
                                          const void* w2_dev, void* out_host, void* ws_dev,
                                          size_t ws_bytes, void* stream);

/* Failure-path check: launches one kernel whose bounded wait has nothing to
 * wait for; after `budget_cycles` SM clock cycles it records MOE_ERR_TIMEOUT
 * in the workspace status word and returns.  Used by the tests. */
moe_status_t moe_debug_timeout_probe(void* ws_dev, size_t ws_bytes, int64_t budget_cycles,
                                     void* stream);

/* Size of the fixed device array that moe_dispatch_static uses for scratch. */
#define MOE_STATIC_SCRATCH_BYTES (4u << 20)

/* moe_dispatch without a workspace, for callers that cannot allocate device
 * memory: a plugin that only receives its input and output buffers from the
 * engine that owns all allocations, or a loop whose rules forbid allocating
 * after start-up.  The pages have no counterpart to this entry point; it
 * exists for those callers only.
 *
 * Arguments and outputs are those of moe_dispatch (d_model and d_ff are not
 * used; with T = 0 the per-token arrays may be NULL); status_dev (NULL or one int32 on the device) receives the device
 * status of this call (MOE_OK, or MOE_ERR_NONFINITE for a NaN score).
 * Scratch lives in one file-scope device array of MOE_STATIC_SCRATCH_BYTES,
 * held by every GPU that loads the library until the process exits.  Its
 * device address is looked up with cudaGetSymbolAddress during the first call
 * in each CUDA context -- on each device, and again on a device after a reset
 * has recreated its context -- and kept for that context (make that first call
 * before any stream capture).  A config
 * whose scratch does not fit (max(16, E rounded up to 16) + 9k bytes per token
 * plus (8k+4)*E bytes per 256 tokens; about 48k tokens at E=64, k=2) returns
 * MOE_ERR_UNSUPPORTED before anything is enqueued.  The call performs no
 * allocation of any kind.  Every call shares the array and finds the previous
 * call's contents in it (the status word is cleared per call); calls that
 * overlap on the GPU race. */
moe_status_t moe_dispatch_static(const moe_config_t* cfg, const float* scores_dev,
                                 int32_t* assign_dev, int32_t* slot_dev, uint8_t* flags_dev,
                                 int32_t* counts_dev, int32_t* offsets_dev, int32_t* perm_dev,
                                 float* combine_w_dev, int32_t* n_rerouted_dev,
                                 int32_t* n_dropped_dev, int32_t* status_dev, void* stream);

#ifdef __cplusplus
}
#endif
#endif
