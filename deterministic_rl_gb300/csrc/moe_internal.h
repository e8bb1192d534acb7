// moe_internal.h -- parameters and launchers shared between the C-ABI layer
// (api.cu) and the kernels.  Not part of the public interface.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <cstdint>

namespace moe {

// Tile shape of the tcgen05 GEMMs: 128 weight rows (M) x BN token rows (N)
// x 64 along K per pipeline stage.  One schedule for every group size, so the
// reduction order of each output element depends on K alone.
constexpr int BM = 128;
constexpr int BN = 128;         // token tile of the one-SM GEMM (gemm.cu)
constexpr int BN_EXPERT = 256;  // token tile of the SM-pair expert GEMMs (gemm_pair.cu)
// Batches of at most this many tokens run the expert GEMMs on the one-SM kernel
// (weight streaming); larger ones on SM pairs.  Both kernels compute every
// output element with the same bf16 MMAs in the same K order (tested bitwise).
constexpr int64_t kOneSmMaxTokens = 128;
constexpr int BK = 64;
// In the SM-pair gate/up tile with MXFP8 weights each CTA's 128 converted
// weight rows alternate in blocks: 16 gate rows, then the same 16 rows of the
// up projection, four times, so that each epilogue warp's 32 accumulator lanes
// hold both halves of 16 rows.
constexpr int kSwigluBlock = 16;
// SwiGLU of one gate/up pair of pre-activations: silu(g) * u = g / (1 + e^-g) * u,
// in fp32 with the fast exponential and division.  Neither branches, so an
// epilogue keeps many of them in flight; their errors (a few ulp) vanish in
// the bf16 rounding of the result.  Every forward kernel computes SwiGLU with
// this one routine, so the kernel families produce the same bits.
__device__ __forceinline__ float swiglu(float g, float u) {
    return __fdividef(g, 1.0f + __expf(-g)) * u;
}

// Expert weight storage formats (the values of the ABI's moe_wfmt).
constexpr int WFMT_BF16 = 0;
constexpr int WFMT_MXFP8 = 1;
constexpr int WFMT_NVFP4 = 2;

// Device status word bits (ws status[0]); status[1] = id of the kernel whose
// wait ran out, status[2] = number of tokens with rejected replay ids.
constexpr int STATUS_BAD_IDS = 1;
constexpr int STATUS_TIMEOUT = 2;

enum GemmMode : int { GEMM_ROUTER = 0, GEMM_SWIGLU = 1, GEMM_DOWN = 2 };

// Weight rows per CTA of an SM-pair tile: the gate/up GEMM's 128-row MMA half
// holds 64 gate rows and the 64 matching up rows.
__host__ __device__ constexpr int gemm_rows(int mode) { return mode == GEMM_SWIGLU ? 64 : BM; }

// Grouped GEMM  D[g] = A[g] . B[g]^T  over groups g of token rows.
// A: weight rows (K-major), B: token rows (K-major), both bf16 via TMA.
// Routed group g < G has cnt[g] token rows starting at B row off[g] and uses
// weight rows [g*M, g*M + M) of a0 (and a1); the optional shared group has
// shared_rows token rows from B row shared_b_off and uses as0 (and as1).
// For the router (cnt == nullptr) there is one group of n_single rows at 0.
struct GemmParams {
    CUtensorMap a0, a1, as0, as1, b;
    CUtensorMap b32;    // same tensor as b with a 32-row box (partial token tiles)
    int32_t partial_b;  // 1: load only the 32-row boxes a tile's tokens occupy
    const int32_t* cnt;
    const int32_t* off;
    int32_t G;
    int32_t has_shared;
    int32_t n_single;
    int32_t shared_rows;
    int32_t shared_b_off;
    int32_t M;      // weight rows per group
    int32_t MT;     // ceil(M / gemm_rows(mode))
    int32_t KB;     // K / BK
    void* out;        // router: fp32 logits [T][ldo]; swiglu: bf16 H [rows][ldo]; down: bf16 Y
    void* out_shared; // down: fp32 Ysh [T][ldo]
    int32_t ldo;
    const float* bias;  // router only
    CUtensorMap sa0, sa1;  // MXFP8: E8M0 scale maps matching a0, a1 (16-byte boxes)
    int32_t* status;
    uint64_t timeout_ns;
    int32_t stall_test;  // test hook: the producers issue nothing, so waits run out
    int32_t ksplit;      // one-SM kernel: K split into this many fixed parts (0/1: none);
                         // part s goes to out + s * split_stride (no bias)
    int64_t split_stride;
    // NVFP4: fp32 scale of each token row of B (applied to its output column),
    // and the per-group fp32 scales of the weight matrices (a0 and a1).
    const float* row_scale;
    const float* wscale0;
    const float* wscale1;
    // SM-pair kernel: tiles are handed out in order by this counter (zeroed
    // before the launch); which pair computes a tile never changes how.
    int32_t* tile_counter;
    // gate/up: SwiGLU output row = token row of B + out_row_off (the shared
    // expert run on its own reads x directly and writes after the routed rows)
    int32_t out_row_off;
    // SM-pair bf16 gate/up: if not null, also store the fp32 pre-activations
    // (gate and up projections) of each H element, same indexing as H.
    float* save_a;
    float* save_b;
    // SM-pair down (MODE 2): 1 = fp32 output rows; with out_shared null the
    // shared group's rows are stored like routed rows (at its B rows).  The
    // block-scaled MXFP8 down GEMM takes it too (its shared group, has_shared,
    // always stores like routed rows).
    int32_t out_f32;
    // SM-pair bf16 gate/up: a0 (and as0) map the packed gate/up weights
    // (64 gate rows then the same 64 up rows per block; 128-row boxes); the
    // CTA's 128 operand rows are one box at packed row 2 * arow.
    int32_t a_packed;
    // Block-scaled GEMMs (gemm_bs.cu): the token rows' block scales (E8M0 per
    // 32 for MXFP8, E4M3 per 16 for NVFP4), [rows][K/32 or K/16] bytes.
    CUtensorMap sb_scale;
    // Block-scaled GEMMs: 1 = load scale groups ahead of the weights (large
    // batches; 0 keeps them with their K block, better for weight streaming).
    int32_t sc_ahead;
};

size_t gemm_smem_bytes(int mode, int n_groups_total);
cudaError_t launch_grouped_gemm(int mode, const GemmParams& p, int grid, cudaStream_t s);
// The expert GEMMs (GEMM_SWIGLU, GEMM_DOWN) on 2-CTA clusters (cta_group::2):
// `clusters` pairs of SMs; M is split in tiles of 2 * gemm_rows(mode) rows.
// wfmt WFMT_MXFP8: a0/a1 are E4M3 weight maps (64-byte boxes) with scale maps
// sa0/sa1; the kernel dequantises them exactly to bf16 in shared memory.
// small != 0 (MXFP8 weights, batches of at most kOneSmMaxTokens): the
// weight-streaming variant with 64-token tiles and a deeper weight ring.
cudaError_t launch_pair_gemm(int mode, const GemmParams& p, int clusters, cudaStream_t s,
                             int wfmt = 0, int small = 0);

// The expert GEMMs on the block-scaled tensor-core MMA (gemm_bs.cu), both
// operands narrow.  fmt BS_MXFP8: E4M3 weights and token rows with E8M0 scales
// per 32; fmt BS_NVFP4: packed E2M1 weights and token rows (two per byte) with
// E4M3 scales per 16, each output then scaled by row_scale of its token times
// the group's wscale0 (gate, down) or wscale1 (up).  a0/a1 (gate, up) or a0
// (down) map the weights with 128-byte boxes and the 128-byte swizzle (64 or
// 128 rows), sa0/sa1 their scales; b and b32 the gathered token rows (128-byte
// boxes of bs_big_box(fmt) and of 32 rows, swizzled) and sb_scale their scales
// (128-row boxes).  Scale boxes are bs_scale_box(fmt) bytes wide.  K runs in
// blocks of 128 bytes (KB a multiple of bs_scale_kb(fmt)); tiles of at most
// bs_tile_tokens(fmt) tokens; no shared expert.
constexpr int BS_MXFP8 = 0;
constexpr int BS_NVFP4 = 1;
cudaError_t launch_bs_gemm(int fmt, int mode, const GemmParams& p, int clusters, cudaStream_t s);
int bs_tile_tokens(int fmt);
int bs_big_box(int fmt);
int bs_scale_box(int fmt);
int bs_scale_kb(int fmt);
// MXFP8 quantisation of R rows of K bf16 values (K % 256 == 0) in blocks of 32
// along the row: E4M3 codes to codes [R][K] and E8M0 scale bytes to scales
// [R][K/32] (OCP MX v1.0: X = floor(log2 max|v|) - 8, codes E4M3(v / 2^X)
// nearest even, saturating; scale byte X + 127).  With inv (R token rows,
// k <= 8): each row's codes and scales also go to its k gathered rows
// inv[r * k + j] of codes_p, scales_p (the gather, fused).
cudaError_t launch_mx_rows_fp8(const uint16_t* src, uint8_t* codes, uint8_t* scales, int64_t R,
                               int K, int sms, cudaStream_t s, const int32_t* inv = nullptr,
                               int k = 0, uint8_t* codes_p = nullptr, uint8_t* scales_p = nullptr);

// Routing: top-k selection (own mode) or replay validation, then gate weights.
cudaError_t launch_topk_gates(const float* logits, int64_t T, int E, int k,
                              const int32_t* ids_in, int32_t* ids_out, float* gates_out,
                              int32_t* valid, int32_t* status, cudaStream_t s);
// Same, from nsplit partial logits (part s at parts + s * stride, summed in
// order s = 0, 1, ..., then + bias; the final logits are stored to logits_out),
// or, with nsplit == 1, from the finished logits in logits_out.  filter != 0
// (replay only) applies the replay plausibility filter with threshold
// ln(tau) = log_tau below the router's own k-th logit.
cudaError_t launch_topk_gates_split(const float* parts, int nsplit, int64_t stride,
                                    const float* bias, float* logits_out, int64_t T, int E,
                                    int k, const int32_t* ids_in, int32_t* ids_out,
                                    float* gates_out, int32_t* valid, int32_t* status,
                                    cudaStream_t s, int filter = 0, float log_tau = 0.0f);

// Dispatch: stable counting sort of the T*k pairs by expert, then the gather
// of token rows into expert order (plus the shared-expert copy of x).
size_t dispatch_scratch_bytes(int64_t n_pairs, int E);
cudaError_t launch_dispatch(const int32_t* ids, int64_t T, int k, int E, int32_t* cnt,
                            int32_t* off, int32_t* perm, int32_t* inv, int32_t* scratch,
                            cudaStream_t s);
// Rows in expert order: xp[inv[t*k + s]] = x[t], and xp[T*k + t] = x[t] for
// the shared expert (n_shared).  scale_in/scale_out (NVFP4): also copy each
// token's fp32 scale to its rows.
cudaError_t launch_gather(const uint16_t* x, const int32_t* inv, int64_t T, int k, int d,
                          int n_shared, uint16_t* xp, cudaStream_t s,
                          const float* scale_in = nullptr, float* scale_out = nullptr);

// NVFP4 quantisation of R rows of K bf16 values (K % 16 == 0), per row: codes
// [R][K/2] bytes (two E2M1 codes, element 2j in the low nibble), bscale
// [R][K/16] E4M3 block scales, rscale [R] the fp32 row scale (nvfp4.cu).
// With inv (R token rows, k <= 8): each row's codes, block scales and row
// scale also go to its k gathered rows inv[r * k + j] of codes_p, bscale_p,
// rscale_p (the gather of the quantised rows, fused).
cudaError_t launch_nvfp4_codes(const uint16_t* src, uint8_t* codes, uint8_t* bscale, float* rscale,
                               int64_t R, int K, int sms, cudaStream_t s,
                               const int32_t* inv = nullptr, int k = 0, uint8_t* codes_p = nullptr,
                               uint8_t* bscale_p = nullptr, float* rscale_p = nullptr);
// ---- backward (backward.cu, wgrad.cu) ----

// Grouped weight-gradient GEMM: for group g, out[g][n][m] = sum over the
// group's K-blocks of A[m][k] * B[n][k] (a: [M][Kpad], b: [N][Kpad] bf16 maps
// with 64 x wgrad_box_rows() boxes), K range [poff[g], poff[g+1]) (multiples
// of 64, zero-padded).  Rows n < n_split go to out0 (routed groups, group g at
// + g * gstride) or sout0 (groups >= G_routed), rows n >= n_split (minus
// n_split) to out1 / sout1.  Row stride M floats.
struct WgradParams {
    CUtensorMap a, b;
    const int32_t* poff;
    int32_t G, G_routed;
    int32_t M, N, MT, NT, n_split;
    float* out0;
    float* out1;
    float* sout0;
    float* sout1;
    int64_t gstride;
    int32_t* status;
    uint64_t timeout_ns;
    int32_t stall_test;
};
constexpr int kMaxWgradGroups = 1024;
// clusters: CTA pairs (the kernel runs on SM pairs, tcgen05 cta_group::2)
cudaError_t launch_wgrad(const WgradParams& p, int clusters, cudaStream_t s);
int wgrad_tile_m();    // A rows per tile (both CTAs)
int wgrad_tile_n();    // B rows per tile (both CTAs)
int wgrad_box_rows();  // rows of the a and b maps' boxes (one CTA's half)

// Padded segment offsets of the G = E (+1 shared) groups: poff[g + 1] =
// poff[g] + round_up(n_g, 64); then, at poff + G + 1, the group of each of the
// ntiles 64-row tiles (-1 past poff[G]).
cudaError_t launch_seg_offsets(const int32_t* cnt, int E, int G, int shared_rows, int32_t* poff,
                               int64_t ntiles, cudaStream_t s);
// Transposed MXFP8 quantisation (blocks of 32 along the input's rows).
struct SegDyArgs {
    const uint16_t* dout;
    const float* gates;
    const int32_t* perm;
    const int32_t* valid;
    int k;
    int64_t Tk;
    const int32_t* inv;  // dispatch position of each (token, slot) pair
    int64_t T;
    int n_shared;
};
// Segment mode: out[c][poff[g] + i] = Q(row i of group g)[c] for bf16 rows
// (src, row stride src_ld), groups padded with zeros to their poff extent;
// out row stride kpad.
cudaError_t launch_tq_segments(const uint16_t* src, int64_t src_ld, int C, const int32_t* cnt,
                               const int32_t* off, const int32_t* poff, int E, int G,
                               int64_t shared_row0, int shared_rows, int64_t kpad, uint16_t* out,
                               int sms, cudaStream_t s);
// dY (gate(t,s) * dout[t] for the routed row of pair t*k + s, dout[t] for shared
// row Tk + t; zero for rejected tokens), quantised along d into E4M3 codes dyc
// [rows][d] with E8M0 scale bytes dys [rows][d / 32], and along each expert's
// tokens into dyt [d][kpad] (bf16 values).
cudaError_t launch_dy_dual(const SegDyArgs& dy, int d, const int32_t* cnt, const int32_t* off,
                           const int32_t* poff, int E, int G, int shared_rows, int64_t kpad,
                           uint8_t* dyc, uint8_t* dys, uint16_t* dyt, int sms, cudaStream_t s);
// SwiGLU backward from dH and the fp32 pre-activations, quantised along F into
// codes dabc [rows][2F] = [dA | dB] with scale bytes dabs [rows][2F / 32], and
// along each expert's tokens into dabt [2F][kpad] = [dA ; dB] (bf16 values).
cudaError_t launch_swiglu_dual(const float* dh, const float* a_pre, const float* b_pre, int F,
                               const int32_t* cnt, const int32_t* off, const int32_t* poff, int E,
                               int G, int64_t shared_row0, int shared_rows, int64_t kpad,
                               uint8_t* dabc, uint8_t* dabs, uint16_t* dabt, int sms,
                               cudaStream_t s);
// Batch mode: nb matrices [R][C] bf16 -> E4M3 codes at codes[b * out_bstride +
// c * out_ld + out_off + r], quantised along r, and the E8M0 scale byte of each
// block of 32 at scales[that offset / 32].
cudaError_t launch_tq_batch(const uint16_t* src, int nb, int R, int C, uint8_t* codes,
                            uint8_t* scales, int64_t out_bstride, int64_t out_ld, int64_t out_off,
                            int sms, cudaStream_t s);
// Gate gradients, softmax backward and the router's part of dx (written to dx).
cudaError_t launch_gate_bwd(const uint16_t* dout, const uint16_t* y, const int32_t* inv,
                            const int32_t* ids, const float* gates, const int32_t* valid,
                            const uint16_t* wr, float* dg, float* dl, float* dx, int64_t T, int k,
                            int d, int sms, cudaStream_t s);
cudaError_t launch_router_wgrad(const uint16_t* xp, const int32_t* perm, const int32_t* cnt,
                                const int32_t* off, const float* dl, float* d_router, int E, int d,
                                int sms, cudaStream_t s);
// dx[t] = (sum_s dxp[inv[t k + s]] + dxp[Tk + t]) + dx[t].
cudaError_t launch_dx_assemble(const float* dxp, const int32_t* inv, float* dx, int64_t T, int k,
                               int d, int n_shared, int sms, cudaStream_t s);


// Packed gate/up weights: G matrices pairs [F][d] (gate, up) -> [G][F/64][128][d]
// (64 gate rows, then the same 64 up rows).  gate[g], up[g] are the g-th
// matrices of the two lists given (routed experts, then the shared expert).
cudaError_t launch_pack_gate_up(const uint16_t* gate, const uint16_t* up, int64_t nmat, int F,
                                int d, uint16_t* packed, cudaStream_t s);

// Fixed-order combine of each token's k expert rows and the shared row.
cudaError_t launch_combine(const uint16_t* y, const float* ysh, const int32_t* inv,
                           const float* gates, const int32_t* valid, int64_t T, int k, int d,
                           int out_fp32, void* out, cudaStream_t s);

}  // namespace moe
