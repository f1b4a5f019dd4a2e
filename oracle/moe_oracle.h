/*
 * moe_oracle.h -- plain, slow, single-threaded CPU reference for the forward
 * pass of one sparsely activated Mixture-of-Experts FFN layer.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may include, link,
 * load or call this code: only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg use it.  It shares no code, header, table or
 * helper with the CUDA library under token_level_top_gb300/csrc.
 *
 * Pages cited (the method's only description):
 *   [mhpn]     "GPT-4稀疏激活真相：万亿参数模型的MoE工程落地实践"
 *              (www.mhpn.cn/news/895310)
 *   [coreui]   "MoE架构揭秘：逐Token路由与活跃参数量的工程真相"
 *              (www.coreui.cn/article/2635427.html)
 *   [cnnetsun] "MoE稀疏激活原理与工程实践：从2%激活率到高效推理"
 *              (cnnetsun.cn/a/3071834)
 *   [csdn]     untitled page, adg.csdn.net/6a3116e610ee7a33f27ddf1c.html
 *   [2kiu]     MoE page at www.2kiu.com/news/5042631/
 *
 * Precision: bf16 inputs are widened exactly to fp32.  Dot products, the
 * softmax, combine weights and the expert FFN are evaluated in double and
 * rounded once to fp32 where an fp32 output is defined.  The two values that
 * decide integers -- the logits z and the penalised scores s -- are fp32, as
 * the router is kept in fp32 ([coreui] §5.2, router_dtype=float32), and s is
 * formed with separately rounded fp32 operations (no fused multiply-add).
 *
 * Status codes match the library's meaning: 0 ok, 1 invalid argument,
 * 5 non-finite (NaN) score.
 */
#ifndef MOE_ORACLE_H
#define MOE_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Expert capacity C = ceil(T*k*cf/E), computed exactly with cf read as a
 * decimal with six fractional digits ([coreui] §5.2 writes
 * expert_capacity = ceil(batch_size*top_k/num_experts*1.3); §3.3 gives the
 * factor alpha in 1.2..1.5).  explicit_cap > 0 overrides the formula. */
int64_t oracle_capacity(int64_t T, int k, int E, double cf, int64_t explicit_cap);

/* Router: logits, penalised scores, top-k ids and probabilities, and the
 * load statistics f and P.
 *   h        [T,d] bf16 bits (ignored when logits_in != NULL)
 *   wr       [E,d] bf16 bits, row e is expert e's gate vector
 *   bias     [E] fp32 or NULL (added to the GEMM output)
 *   usage    [E] fp32 or NULL; lambda the penalty weight
 *   tau      temperature, > 0: s = z / tau - lambda * usage ([cnnetsun] §3.1
 *            steps 3-4: the scores are divided by tau, then the penalty is
 *            taken off, before softmax and top-k; [2kiu] §2, third measure)
 *   logits_in[T,E] fp32 or NULL: final logits given directly (bias not added)
 * Outputs (all required): logits [T,E], scores [T,E], ids [T,k],
 * topk_p [T,k] (softmax probability of each pick), counts_pre [E], f [E], P [E].
 * Returns 0, 1 on a bad argument, or 5 if any score is NaN (outputs then
 * undefined). */
int oracle_route(int T, int d, int E, int k, const uint16_t* h, const uint16_t* wr,
                 const float* bias, const float* usage, float lambda, float tau,
                 const float* logits_in, float* logits, float* scores, int32_t* ids,
                 float* topk_p, int32_t* counts_pre, float* f, float* P);

/* Router front ends that produce the logits z ([cnnetsun] §3.1 steps 1-2;
 * [2kiu] §5.2; [mhpn] §3.1 lists a router of Embedding -> LayerNorm ->
 * Linear -> activation -> Linear):
 *   x_t = h_t                                       norm 0
 *   x_t = (h_t - mean) / sqrt(var + eps) * g + b    norm 1 (LayerNorm over d;
 *         var the mean squared deviation; g, b = gamma, beta, NULL = 1, 0)
 *   x_t = h_t / max(||h_t||_2, eps)                 norm 2 (L2 normalisation)
 *   z_t = x_t . W^T + bias                          hidden 0, W [E,d]
 *   z_t = silu(x_t . W1^T) . W2^T + bias            hidden H > 0 (the two-layer
 *         router: W1 [H,d] with H = 2E on the page, W2 [E,H]; silu(u) =
 *         u / (1 + exp(-u)))
 * All in double from the bf16 inputs, each z rounded once to fp32.
 *   h [T,d], w [E,d] or [H,d], w2 [E,H] (hidden > 0, else NULL): bf16 bits;
 *   gamma, beta [d] fp32 or NULL; bias [E] fp32 or NULL; logits [T,E] out.
 * Returns 0 or 1 (bad argument). */
int oracle_router_logits(int T, int d, int E, int hidden, int norm, float eps,
                         const uint16_t* h, const float* gamma, const float* beta,
                         const uint16_t* w, const uint16_t* w2, const float* bias,
                         float* logits);

/* The preference order of one token: experts sorted by score, descending,
 * ties to the lower index.  order[E] out.  Returns 0, or 5 on NaN. */
int oracle_preference(int E, const float* s_row, int32_t* order);

/* Capacity-capped dispatch, literal sequential form: all rank-0 choices in
 * token order, then all rank-1 choices, ...  Outputs: assign [T,k] (-1 =
 * dropped), slot [T,k] (-1 when dropped), flags [T,k] (bit0 rerouted, bit1
 * dropped), counts [E], offsets [E+1], perm [sum counts] (= t*k+r in slot
 * order), cw [T,k] combine weights, n_rerouted, n_dropped.
 * Returns 0, 1 (bad args) or 5 (NaN score). */
int oracle_dispatch(int T, int E, int k, int64_t C, const float* scores,
                    int32_t* assign, int32_t* slot, uint8_t* flags, int32_t* counts,
                    int32_t* offsets, int32_t* perm, float* cw,
                    int32_t* n_rerouted, int32_t* n_dropped);

/* One expert on one token: y = W2_e (silu(W1_e x) * (W3_e x)), in double.
 *   x [d] bf16 bits; w1, w3 [F,d] and w2 [d,F] bf16 bits of expert e. */
void oracle_expert_row(int d, int F, const uint16_t* x, const uint16_t* w1,
                       const uint16_t* w3, const uint16_t* w2, double* y);

/* Expert FFN + probability-weighted combine for a list of tokens:
 * out_rows[i] = sum over kept ranks r (rank order) of cw[t,r] * y(t, assign[t,r]),
 * t = tokens[i]; a token with no kept rank gets 0.
 *   h [T,d], w1/w3 [E,F,d], w2 [E,d,F] bf16 bits; out_rows [ntok,d] fp32. */
int oracle_combine_rows(int T, int d, int E, int k, int F, const uint16_t* h,
                        const uint16_t* w1, const uint16_t* w3, const uint16_t* w2,
                        const int32_t* assign, const float* cw,
                        const int32_t* tokens, int ntok, float* out_rows);

/* Expert outputs per slot, in slot order: y_slots[i] = y(t, e) for the kept
 * entry perm[i] = t*k+r with e = assign[t,r], for slots i in [row0, row1). */
int oracle_expert_slots(int T, int d, int E, int k, int F, const uint16_t* h,
                        const uint16_t* w1, const uint16_t* w3, const uint16_t* w2,
                        const int32_t* assign, const int32_t* perm,
                        int row0, int row1, float* y_slots);

/* The value of an e4m3 code (sign, 4-bit exponent with bias 7, 3-bit
 * mantissa, subnormals at exponent 0, 0x7F/0xFF NaN, no infinity). */
double oracle_e4m3_value(uint8_t b);

/* The e4m3 code nearest to v (ties to even), saturating at +-448. */
uint8_t oracle_e4m3_encode(float v);

/* Row quantisation: scale = max|x| / 448 (fp32; 1 for a zero row), codes[i] =
 * e4m3(x[i] / scale). */
void oracle_quantize_row(int n, const float* x, uint8_t* codes, float* scale);

/* oracle_combine_rows / oracle_expert_slots with 8-bit expert weights: W1, W3
 * as e4m3 codes q1, q3 [E][F][d] with row scales s1, s3 [E][F]; W2 as q2
 * [E][d][F] with s2 [E][d]; weight = code value * row scale.  quant_act != 0:
 * each token row x and each activation row silu(W1 x) * (W3 x) (rounded to
 * bf16 first) also enters its GEMM as row-quantised e4m3 codes times scale. */
int oracle_combine_rows_q8(int T, int d, int E, int k, int F, const uint16_t* h,
                           const uint8_t* q1, const float* s1, const uint8_t* q3, const float* s3,
                           const uint8_t* q2, const float* s2, int quant_act, const int32_t* assign,
                           const float* cw, const int32_t* tokens, int ntok, float* out_rows);
int oracle_expert_slots_q8(int T, int d, int E, int k, int F, const uint16_t* h,
                           const uint8_t* q1, const float* s1, const uint8_t* q3, const float* s3,
                           const uint8_t* q2, const float* s2, int quant_act, const int32_t* assign,
                           const int32_t* perm, int row0, int row1, float* y_slots);

/* e2m1 (the 4-bit element of NVFP4): bit 3 sign, bits 2..1 exponent with
 * bias 1, bit 0 mantissa; exponent 0 holds the subnormal 0.5 * mantissa.  The
 * magnitudes are 0, 0.5, 1, 1.5, 2, 3, 4, 6 (no infinity, no NaN).  Only the
 * low 4 bits of `code` are read. */
double oracle_e2m1_value(uint8_t code);

/* The e2m1 code nearest to v, ties to the code with mantissa bit 0 (even),
 * magnitudes above 6 saturating to +-6; NaN gives 0. */
uint8_t oracle_e2m1_encode(float v);

/* NVFP4 row quantisation of x[0..n) (n a multiple of 16), in fp32 steps:
 *   scale = max|x| / 2688 (= 6 * 448; 1 for an all-zero row);
 *   block j (x[16j..16j+16)): b_j = e4m3(fl(fl(max|x_i| / scale) / 6)), a
 *   non-negative e4m3 code (saturating at 448); den_j = fl(value(b_j) * scale);
 *   code_i = e2m1(fl(x_i / den_j)) (0 for every i when den_j = 0).
 * x_i is then represented as e2m1(code_i) * value(b_j) * scale.  codes holds
 * two per byte, element 2m in the low nibble of byte m; bscale[n/16]. */
void oracle_quantize_row_nvfp4(int n, const float* x, uint8_t* codes, uint8_t* bscale, float* scale);

/* Fill the e2m1 and e4m3 value tables the quantised expert functions read
 * (each also fills them on first use).  Call it once before calling those
 * functions from several threads at a time: every other function here keeps
 * its state on the stack or in its own allocations. */
void oracle_init_tables(void);

/* oracle_combine_rows / oracle_expert_slots with NVFP4 expert weights: W1,
 * W3 [E][F][d] and W2 [E][d][F] as packed e2m1 codes (q1, q3, q2), e4m3 block
 * scales per 16 consecutive elements of a row (b1, b3 [E][F][d/16], b2
 * [E][d][F/16]) and fp32 row scales (s1, s3 [E][F], s2 [E][d]); weight =
 * e2m1(code) * value(block scale) * row scale.  quant_act != 0: each token
 * row x and each activation row silu(W1 x) * (W3 x) (rounded to bf16 first)
 * enters its GEMM NVFP4-quantised per row (oracle_quantize_row_nvfp4). */
int oracle_combine_rows_q4(int T, int d, int E, int k, int F, const uint16_t* h,
                           const uint8_t* q1, const uint8_t* b1, const float* s1,
                           const uint8_t* q3, const uint8_t* b3, const float* s3,
                           const uint8_t* q2, const uint8_t* b2, const float* s2, int quant_act,
                           const int32_t* assign, const float* cw, const int32_t* tokens, int ntok,
                           float* out_rows);
int oracle_expert_slots_q4(int T, int d, int E, int k, int F, const uint16_t* h,
                           const uint8_t* q1, const uint8_t* b1, const float* s1,
                           const uint8_t* q3, const uint8_t* b3, const float* s3,
                           const uint8_t* q2, const uint8_t* b2, const float* s2, int quant_act,
                           const int32_t* assign, const int32_t* perm, int row0, int row1,
                           float* y_slots);

/* Backward pass of the layer for one dispatch (training; not on the forward
 * path).  The forward is out[t] = sum over t's kept ranks r of
 * cw[t,r] * y_e(h_t) with e = assign[t,r], y_e(x) = W2_e (silu(W1_e x) * W3_e x),
 * cw[t,r] = p[t,e] / sum over t's kept ranks r' of p[t,assign[t,r']] (the
 * renormalised weights, [mhpn] §4.3), p = softmax(s) over the experts, s =
 * z / tau - lambda * usage, z = h W_r^T + bias ([coreui] §3.1, [cnnetsun]
 * §3.1).  The routing decisions (assign) are held fixed: the top-k choice and
 * the capacity are piecewise constant, so gradients flow through the combine
 * weights and the experts only.  The load-balancing loss of the pages comes in
 * through its gradient with respect to the mean probabilities P_i = mean_t
 * p[t,i] ([coreui] §3.1 writes it from the per-batch mean probabilities;
 * [2kiu] §2 and [mhpn] §3 give other forms of the same sum of squared loads):
 * dP [E] (NULL = none) adds dP_i / T to every dL/dp[t,i].
 * Inputs: h [T,d], wr [E,d], w1, w3 [E,F,d], w2 [E,d,F] bf16 bits; scores
 * [T,E] the forward's penalised scores s (fp32); assign [T,k] (-1 =
 * dropped); dout [T,d] = dL/dout (fp32).
 * Outputs (double, all required, overwritten): dh [T,d], dwr [E,d], dbias [E],
 * dw1, dw3 [E,F,d], dw2 [E,d,F].  Returns 0 or 1 (bad argument). */
int oracle_layer_backward(int T, int d, int E, int k, int F, float tau, const uint16_t* h,
                          const uint16_t* wr, const uint16_t* w1, const uint16_t* w3,
                          const uint16_t* w2, const float* scores, const int32_t* assign,
                          const float* dout, const float* dP, double* dh, double* dwr,
                          double* dbias, double* dw1, double* dw3, double* dw2);

#ifdef __cplusplus
}
#endif

#endif
