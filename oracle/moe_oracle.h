/*
 * moe_oracle.h -- plain, slow, fp64 CPU oracle of the deterministic MoE layer
 * forward with router replay.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path (the CUDA library and
 * its Python binding) may include, link, load or call this code.  Only the
 * test suite, the smoke check and the CPU-baseline leg of the benchmark use it.
 * It shares no code, header, table or helper with the CUDA path.
 *
 * What it follows (sources are the pages this project is built from):
 *   [TR]  Composer 2 Technical Report (zh-TW and ja renderings, English
 *         summary page):
 *           §6.2 "RL infrastructure", paragraph on inference and weight
 *           sync: router replay -- the inference engine returns the chosen
 *           expert indices per token per MoE layer; the trainer forward
 *           overrides the router's assignment with them; the router still
 *           computes gate scores.
 *           §6.1 "Training infrastructure", Kernels paragraph and Fig. 10:
 *           grouped expert GEMMs, token dispatch/combine (combine kept in
 *           BF16), MXFP8 = E4M3 values with one E8M0 scale per 32 elements.
 *   [TD]  "1TB 权重 60 秒跨洋同步：Cursor 训练 Composer 2 的分布式 RL 工程"
 *         (Training Data No. 94 write-up), section
 *         "浮点数不守规矩，MoE 火上浇油": one gate per layer picks 8 of 384
 *         experts from the hidden state; float addition order decides
 *         rounding; fixed-order ("batch-invariant") accumulation; replay
 *         sends one integer per chosen expert.
 *   [CH]  "「模型會作弊」：Cursor 訓練 Composer 2 的五大工程挑戰", section
 *         "浮點數的陷阱：A+B+C ≠ C+B+A": the same facts.
 *
 * The layer's plain definition (the fixed accumulation order of the GPU
 * changes rounding only, never the mathematics), per token t:
 *   logits   l_e = sum_j x[t][j] * Wr[e][j] + b[e]                (fp64)
 *   own mode ids = the k largest l_e, descending, ties -> lower e
 *   replay   ids = the caller's recorded ids, in the caller's slot order
 *   gates    w_s = exp(l_{i_s} - m) / sum_{s'} exp(l_{i_s'} - m),
 *            m = max over the k chosen logits (softmax over all E, then
 *            renormalised over the chosen set, written in its restricted form)
 *   expert   y_e(x) = sum_f silu(x.Wg_e[f]) * (x.Wu_e[f]) * Wd_e[:, f]
 *   output   out_t = sum_{s=0..k-1} w_s * y_{i_s}(x_t) + sum_shared y_sh(x_t)
 * Every product of two bf16 values is exact in fp64; sums round at 2^-53.
 * No intermediate value is rounded to bf16 or fp32.
 */
#ifndef MOE_ORACLE_H
#define MOE_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Weight storage formats the oracle reads. */
enum { ORACLE_W_BF16 = 0, ORACLE_W_MXFP8 = 1, ORACLE_W_NVFP4 = 2, ORACLE_W_MXFP8_ACT = 3 };

/* One weight matrix [rows][K], rows contiguous along K (K-major).
 * bf16: values = uint16 bf16 bit patterns, scales = NULL.
 * mxfp8: values = E4M3 (fn) bytes, scales = E8M0 bytes [rows][K/32].
 * mxfp8_act: stored as mxfp8; the expert FFN also quantises its activations
 *        (oracle_mx_qdq_rows: each x row along d, each bf16-rounded h row
 *        along F), the MXFP8 expert compute of [TR] §6.1.
 * nvfp4: values = E2M1 codes packed two per byte [rows][K/2] (element 2j in the
 *        low nibble), scales = E4M3 bytes [rows][K/16], tscale = the matrix's
 *        FP32 scale; element = e2m1 * e4m3 * tscale. */
typedef struct {
    int fmt;
    const void *values;
    const uint8_t *scales;
    float tscale;
} oracle_matrix;

/* Exact decoders (bit pattern -> fp64). */
double oracle_bf16_to_f64(uint16_t h);
double oracle_e4m3_to_f64(uint8_t b);
double oracle_e8m0_to_f64(uint8_t s);
/* Element (r, c) of a weight matrix with K columns, dequantised exactly. */
double oracle_matrix_elem(const oracle_matrix *m, int64_t K, int64_t r, int64_t c);

/* ---- NVFP4 with per-token scales ([TR] §6.1, Kernels paragraph) ----------
 * The MoE forward quantises BF16 values to FP4 E2M1 with one E4M3 scale per
 * 16 consecutive values and one FP32 scale per token (per row), using IEEE
 * division.  Readings (the pages name the format, not the arithmetic):
 *   s    = amax(row) / (6 * 448)                       fp32, IEEE division
 *   S_b  = E4M3_RNE(amax(block b) / 6 / s)             fp32 divisions, saturating
 *   q_i  = E2M1_RNE(x_i / (S_b * s))                   fp32 product, IEEE division
 * and the value the GEMM uses is e2m1(q_i) * e4m3(S_b) * s.  An all-zero row
 * has s = 0 and all codes and block scales 0; a block whose S_b rounds to 0
 * has all codes 0.  Zero is always encoded +0 (code 0).  Inputs are finite. */

/* Value of a 4-bit E2M1 code: sign bit 3, exponent bits 2..1 (bias 1),
 * mantissa bit 0; exponent 0 is subnormal (0 or 0.5). */
double oracle_e2m1_to_f64(uint8_t code);
/* E2M1 code of v, rounded to nearest (ties to the even code), magnitudes above
 * 6 saturate to 6. */
uint8_t oracle_e2m1_round(float v);
/* E4M3 (fn) byte of v >= 0, rounded to nearest even, saturating at 448. */
uint8_t oracle_e4m3_round(float v);
/* Quantise R rows of K values (K % 16 == 0; bf16 values given as fp32):
 * codes [R][K] (one code per byte), bscale [R][K/16], rscale [R]. */
void oracle_nvfp4_quantize_rows(const float *x, int64_t R, int64_t K, uint8_t *codes,
                                uint8_t *bscale, float *rscale);
/* Round a double to the nearest bf16 value (ties to even), as a double. */
double oracle_round_bf16(double v);

/* ---- MXFP8 (OCP Microscaling Formats v1.0, E4M3 elements) -----------------
 * [TR] §6.1 (Kernels): MXFP8 = E4M3 values with one E8M0 scale per block of
 * 32 elements.  Per block: X = floor(log2(max |v|)) - 8 (8 = the exponent of
 * E4M3's largest normal), within [-127, 127], -127 for an all-zero block;
 * each value becomes E4M3(v / 2^X) * 2^X, nearest even, clamped to +-448.
 * Quantise-dequantise R rows of K values (K % 32 == 0) along the rows, in ->
 * out (may alias); inputs are values that fp32 holds exactly (bf16 values). */
void oracle_mx_qdq_rows(const double *in, int64_t R, int64_t K, double *out);

/* Router logits for T tokens: logits[t][e] = sum_j x[t][j]*wr[e][j] + bias[e].
 * x [T][d] bf16, wr [E][d] bf16, bias [E] fp32 or NULL. */
void oracle_router_logits(const uint16_t *x, const uint16_t *wr, const float *bias,
                          int64_t T, int64_t d, int64_t E, double *logits);

/* Own-mode selection: ids[t][0..k) = the k largest logits of row t, in
 * descending order, equal logits resolved towards the lower expert id. */
void oracle_select_topk(const double *logits, int64_t T, int64_t E, int64_t k,
                        int32_t *ids);

/* Replay-id validity per token: 1 if every id lies in [0, E) and no id repeats
 * within the token, else 0.  valid [T]. Returns the number of invalid tokens. */
int64_t oracle_check_ids(const int32_t *ids, int64_t T, int64_t E, int64_t k,
                         uint8_t *valid);

/* Replay plausibility filter ([TR] §6.2: replayed experts whose gate score is
 * below a plausibility threshold derived from the router's own top-k are
 * dropped and replaced by the router's candidates).  Reading: with the router's
 * own top-k o_0..o_{k-1} (descending), replayed id e is kept iff its softmax
 * score is at least tau times that of o_{k-1}, i.e. l_e >= l_{o_{k-1}} + ln(tau)
 * (tau = 0 keeps everything); each dropped slot, in ascending slot order, takes
 * the next own candidate (in own order) that is not already among the token's
 * ids.  ids_in must be valid (oracle_check_ids).  Writes ids_out [T][k] and,
 * per token, the number of replaced slots (n_replaced [T], may be NULL). */
void oracle_filter_replay(const double *logits, const int32_t *ids_in, int64_t T,
                          int64_t E, int64_t k, double tau, int32_t *ids_out,
                          int32_t *n_replaced);

/* Gate weights over the given ids (own or replayed): softmax of the chosen
 * logits, i.e. softmax over all E renormalised over the chosen set. */
void oracle_gate_weights(const double *logits, const int32_t *ids, int64_t T,
                         int64_t E, int64_t k, double *gates);

/* Stable counting sort of the (token, slot) pairs by expert id.
 * Pairs are numbered i = t*k + s over n_pairs = T*k entries of ids.
 * cnt[e] = number of pairs routed to e; off[0..E] = exclusive prefix sum;
 * perm[dst] = i for dst = off[e] + (rank of i among earlier pairs with id e);
 * inv[i] = dst.  Every id must be in [0, E). */
void oracle_counting_sort(const int32_t *ids, int64_t n_pairs, int64_t E,
                          int32_t *cnt, int32_t *off, int32_t *perm, int32_t *inv);

/* SwiGLU expert FFN applied to n token rows.
 * x [n][d] bf16 rows; wg, wu: [F][d]; wd: [d][F]; y [n][d] fp64.
 * With NVFP4 weights the FFN is the NVFP4 forward: each x row is quantised as
 * above, h = silu(x.Wg) * (x.Wu) is rounded to bf16 and each h row quantised
 * again before the down projection; everything else is exact fp64. */
void oracle_expert_ffn(const uint16_t *x, int64_t n, int64_t d, int64_t F,
                       const oracle_matrix *wg, const oracle_matrix *wu,
                       const oracle_matrix *wd, double *y);

/* Fixed-slot-order combine for T tokens:
 * out[t][:] = sum_{s<k} gates[t][s] * y_slots[t][s][:] + y_shared[t][:].
 * y_slots [T][k][d]; y_shared [T][d] or NULL; valid [T] or NULL (a token with
 * valid[t] == 0 gets an all-zero row). */
void oracle_combine(const double *y_slots, const double *gates,
                    const double *y_shared, const uint8_t *valid, int64_t T,
                    int64_t k, int64_t d, double *out);

/* Threads the oracle may use (OpenMP); returns the count actually in effect. */
int oracle_set_threads(int n);
int oracle_get_threads(void);

#ifdef __cplusplus
}
#endif
#endif /* MOE_ORACLE_H */
