/*
 * moe_det.h -- C ABI of libmoedet: a deterministic, batch-invariant
 * Mixture-of-Experts layer forward with router replay, for GB300 (sm_103a).
 *
 * Sources the operations follow:
 *   [TR] Composer 2 Technical Report, §6.2 "RL infrastructure", paragraph on
 *        inference and weight sync (router replay: the inference engine
 *        returns the chosen expert indices for every token at every MoE
 *        layer; the trainer forward overrides the router's assignment with
 *        them; the router still computes gate scores), and §6.1 "Training
 *        infrastructure", Kernels paragraph and Fig. 10 (grouped expert
 *        GEMMs, dispatch/combine with the combine in BF16, MXFP8 = E4M3
 *        values with an E8M0 scale per 32-element block).
 *   [TD] "1TB 权重 60 秒跨洋同步：Cursor 训练 Composer 2 的分布式 RL 工程",
 *        section "浮点数不守规矩，MoE 火上浇油": a gate per layer picks 8 of
 *        384 experts from the hidden state; batch-invariant kernels force
 *        every accumulation into a fixed order; replay sends one integer per
 *        chosen expert.
 *   [CH] "「模型會作弊」：Cursor 訓練 Composer 2 的五大工程挑戰", section
 *        "浮點數的陷阱：A+B+C ≠ C+B+A": the same facts.
 *
 * Conventions shared by every entry point
 *   - Pointers.  Every tensor argument is a DEVICE pointer unless stated
 *     otherwise; all are row-major and rows are contiguous along the
 *     reduction dimension K ("K-major").  bf16 means IEEE bfloat16 bit
 *     patterns.  The caller allocates and owns every buffer, including the
 *     workspace; the library allocates and frees nothing and keeps no state
 *     between calls.
 *   - Streams.  `stream` is a cudaStream_t (NULL = legacy default stream).
 *     All work is enqueued on it in order; no call synchronises except
 *     moe_get_status.  Calls on different streams need different workspaces.
 *   - Host errors.  Null pointers, bad shapes, misalignment and a short
 *     workspace are rejected before anything is launched, with the status
 *     codes below; nothing is written in that case.
 *   - Device errors.  Replayed ids outside [0, E) or repeated within a token
 *     and bounded waits that run out are recorded in a status word inside
 *     the workspace (read it with moe_get_status); kernels never trap.  A
 *     token whose replayed ids are invalid gets an all-zero output row, zero
 *     gate weights, and ids_out row {0, 1, ..., k-1}.
 *   - Determinism.  For fixed inputs the outputs are bitwise identical run
 *     to run, and the output row of a token depends only on that token's
 *     hidden state, ids and the weights -- never on the other tokens of the
 *     batch or on T.  Expert outputs of a token are added in ascending slot
 *     order, then the shared expert, with fp32 accumulation ([TD], [CH]).
 *   - Limits of this version.  k == 8; 8 <= E <= 512; d and F multiples of
 *     64 (and of 512 for MXFP8 / NVFP4 weights), 64 <= d, F <= 16384; n_shared
 *     in {0, 1} (0 with MXFP8 / NVFP4 weights: MOE_ERR_UNSUPPORTED otherwise);
 *     1 <= T <= 2^20 (T == 0 is a no-op that returns MOE_OK).
 *     Device pointers must be 16-byte aligned.
 */
#ifndef MOE_DET_H
#define MOE_DET_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t, declared here so that the header needs no CUDA
 * include. */
struct CUstream_st;
typedef struct CUstream_st *moe_stream_t;

typedef enum {
    MOE_OK = 0,
    MOE_ERR_ARG = 1,          /* null pointer or invalid enum value          */
    MOE_ERR_SHAPE = 2,        /* dimension outside the limits above          */
    MOE_ERR_ALIGN = 3,        /* pointer not 16-byte aligned                 */
    MOE_ERR_WORKSPACE = 4,    /* ws_bytes < moe_workspace_size(dims)         */
    MOE_ERR_BAD_IDS = 5,      /* (device) replayed id out of range/repeated  */
    MOE_ERR_TIMEOUT = 6,      /* (device) a bounded wait ran out             */
    MOE_ERR_CUDA = 7,         /* a CUDA runtime/driver call failed           */
    MOE_ERR_UNSUPPORTED = 8   /* valid request this build does not serve     */
} moe_status;

typedef enum {
    MOE_W_BF16 = 0,   /* expert weights stored as bf16                        */
    MOE_W_MXFP8 = 1,  /* expert weights E4M3 + one E8M0 scale per 32 along K
                         ([TR] §6.1: the MXFP8 format); router and shared
                         expert stay bf16                                     */
    MOE_W_NVFP4 = 2,  /* the NVFP4 forward ([TR] §6.1, Kernels): expert
                         weights E2M1 (two per byte) + one E4M3 scale per 16
                         along K + one fp32 scale per matrix; the token rows
                         entering each expert GEMM (x, and the SwiGLU
                         activations h in bf16) are quantised to E2M1 with an
                         E4M3 scale per 16 and an fp32 scale per token, with
                         IEEE division.  Router stays bf16; no shared expert */
    MOE_W_MXFP8_ACT = 3 /* MXFP8 expert compute ([TR] §6.1: tokens go out in
                         MXFP8, the experts compute in MXFP8): weights as
                         MOE_W_MXFP8, and the token rows entering each expert
                         GEMM (x along d; the SwiGLU activations h, stored in
                         bf16, along F) quantised to MXFP8 (OCP MX v1.0: per
                         32 values X = floor(log2 max|v|) - 8, E4M3(v / 2^X)
                         nearest even, clamped to +-448).  No shared expert */
} moe_wfmt;

/* Layer shape.  T tokens, hidden size d, E routed experts, k experts per
 * token, expert FFN width F, n_shared always-on shared experts (weight 1). */
typedef struct {
    int64_t T;
    int32_t d;
    int32_t E;
    int32_t k;
    int32_t F;
    int32_t n_shared;
    int32_t wfmt;      /* moe_wfmt                                            */
    int32_t out_fp32;  /* 1: `out` is fp32; 0: `out` is bf16 (round to nearest
                          even of the same fp32 sum)                          */
} moe_dims;

/* Layer weights (all device pointers).
 *   w_router  [E][d] bf16          router (gate) weights; logits = x . w_router^T
 *   router_bias [E] fp32 or NULL   added to the logits before selection and
 *                                  before the gate softmax
 *   w_gate, w_up [E][F][d]         SwiGLU gate / up projections
 *   w_down    [E][d][F]            down projection
 *     bf16 for MOE_W_BF16; E4M3 bytes for MOE_W_MXFP8 with
 *   s_gate, s_up [E][F][d/32], s_down [E][d][F/32]  E8M0 scale bytes
 *     (NULL for MOE_W_BF16);
 *     for MOE_W_NVFP4 w_gate, w_up [E][F][d/2], w_down [E][d][F/2] bytes of
 *     two E2M1 codes (element 2j in the low nibble of byte j) with
 *   s_gate, s_up [E][F][d/16], s_down [E][d][F/16]  E4M3 scale bytes and
 *   gs_gate, gs_up, gs_down [E] fp32  one scale per expert matrix
 *     (NULL unless MOE_W_NVFP4); element = e2m1 * e4m3 * gs
 *   ws_gate, ws_up [F][d], ws_down [d][F]  bf16 shared expert (NULL when
 *     n_shared == 0)
 *   w_gate_up  optional (NULL = not used): the gate and up projections of the
 *     routed experts and then of the shared expert, packed by
 *     moe_pack_weights from the w_gate/w_up/ws_gate/ws_up given here
 *     (bf16 only).  When set, the SM-pair gate/up GEMM of moe_forward /
 *     moe_forward_replay(_filtered) reads each weight tile from it with one
 *     copy instead of two; results are bitwise the same.  The caller repacks
 *     after changing the weights; nothing checks that the copy is current. */
typedef struct {
    const void *w_router;
    const float *router_bias;
    const void *w_gate;
    const void *w_up;
    const void *w_down;
    const uint8_t *s_gate;
    const uint8_t *s_up;
    const uint8_t *s_down;
    const void *ws_gate;
    const void *ws_up;
    const void *ws_down;
    const float *gs_gate;
    const float *gs_up;
    const float *gs_down;
    const void *w_gate_up;
} moe_weights;

/* Byte offsets of the intermediate buffers inside the workspace, for
 * inspection after a call (all int32 unless noted; pairs i = t*k + s):
 *   status   int32[4]      [0] device status bits, [1] where a wait ran out,
 *                          [2] tokens with rejected replay ids, [3] slots replaced
 *                          by the replay filter
 *   logits   fp32 [T][E]   router logits (+ bias)
 *   valid    int32[T]      1 = token's ids valid, 0 = replayed ids rejected
 *   cnt      [E]           pairs routed to each expert (histogram)
 *   off      [E+1]         exclusive prefix sum of cnt
 *   perm     [T*k]         perm[dst] = i, expert-major and stable in i
 *   inv      [T*k]         inv[i] = dst
 *   xp       bf16 [T*k + T*n_shared][d]  gathered token rows (expert order),
 *                                        then the shared-expert rows
 *   h        bf16 [T*k + T*n_shared][F]  SwiGLU activations
 *   y        bf16 [T*k][d]               routed expert outputs (dst order)
 *   ysh      fp32 [T][d]                 shared expert output
 *   MOE_W_NVFP4 only (else empty): the NVFP4 activations as packed E2M1
 *   codes (element 2j in the low nibble of byte j) and E4M3 block scales:
 *   xq       u8 [T][d/2] codes, then u8 [T][d/16] scales of each token row of x
 *   sx       fp32 [T]      each token row's fp32 scale
 *   xp       u8 [T*k][d/2] codes, then u8 [T*k][d/16] scales: the gathered rows
 *   sxp      fp32 [T*k]    the scale of each gathered row of xp
 *   hq       u8 [T*k][F/2] codes, then u8 [T*k][F/16] scales of each row of h
 *            (h keeps the bf16 SwiGLU output)
 *   sh       fp32 [T*k]    the scale of each row of h
 *   MOE_W_MXFP8_ACT: the MXFP8 activations as E4M3 codes and E8M0 scales:
 *   xq       u8 [T][d] codes, then u8 [T][d/32] scales of each token row of x
 *   xp       u8 [T*k][d] codes, then u8 [T*k][d/32] scales: the gathered rows
 *   hq       u8 [T*k][F] codes, then u8 [T*k][F/32] scales of each row of h
 * Offsets are 256-byte aligned; `total` equals moe_workspace_size(dims). */
typedef struct {
    size_t status, logits, valid, cnt, off, perm, inv, xp, h, y, ysh;
    size_t xq, sx, sxp, sh;
    size_t hq;
    size_t total;
} moe_ws_layout;

/* Workspace bytes a call with these dims needs (0 if dims are invalid). */
size_t moe_workspace_size(const moe_dims *dims);

/* Fill *layout for dims.  MOE_ERR_ARG / MOE_ERR_SHAPE on bad input. */
moe_status moe_workspace_layout(const moe_dims *dims, moe_ws_layout *layout);

/* Bytes of the packed gate/up weights for dims (bf16 weights; 0 otherwise):
 * (E + n_shared) * 2 * F * d * 2. */
size_t moe_packed_weights_size(const moe_dims *dims);

/* Pack w->w_gate, w->w_up (and ws_gate, ws_up) into `packed` (device,
 * caller-owned, 16-byte aligned, moe_packed_weights_size bytes): per expert
 * (routed ones, then the shared one), per block of 64 rows of F, the 64 gate
 * rows and then the same 64 up rows, each row d bf16 values.  Set
 * w->w_gate_up = packed afterwards to use it.  A pure copy; stream-ordered.
 * MOE_ERR_UNSUPPORTED for non-bf16 weights. */
moe_status moe_pack_weights(const moe_dims *dims, const moe_weights *w, void *packed,
                            size_t packed_bytes, moe_stream_t stream);

/* Routing only -- the side that records ids at inference ([TR] §6.2:
 * "the engine returns the selected expert indices").  Computes the router
 * logits of x [T][d] bf16, picks the k largest per token (descending logit,
 * equal logits -> lower expert id; [TD]: 8 of 384), and their gate weights
 * (softmax over all E renormalised over the chosen k).
 * Out: ids_out [T][k] int32, gates_out [T][k] fp32. */
moe_status moe_route(const moe_dims *dims, const void *x, const moe_weights *w,
                     int32_t *ids_out, float *gates_out, void *ws,
                     size_t ws_bytes, moe_stream_t stream);

/* Full layer forward with the router's own selection -- the MoE layer of
 * [TD] (section "浮点数不守规矩，MoE 火上浇油": the gate picks 8 of 384
 * experts per token, and the experts' outputs are added in a fixed order so
 * that results do not depend on the batch), with the grouped expert GEMMs and
 * the dispatch/combine of [TR] §6.1 "Training infrastructure" (Fig. 10):
 *   out[t] = sum_{s<k} gates[t][s] * expert_{ids[t][s]}(x[t]) + shared(x[t]),
 * expert(x) = W_down . (silu(W_gate . x) * (W_up . x)), the k routed terms
 * added in ascending slot order in fp32, then the shared expert's, rounded
 * once.  Out: out [T][d] (bf16 or fp32 per dims->out_fp32), ids_out,
 * gates_out as in moe_route. */
moe_status moe_forward(const moe_dims *dims, const void *x, const moe_weights *w,
                       void *out, int32_t *ids_out, float *gates_out, void *ws,
                       size_t ws_bytes, moe_stream_t stream);

/* Full layer forward with router replay ([TR] §6.2; [TD]/[CH]: the trainer
 * activates the recorded experts instead of its own gate's choice).
 * ids_in [T][k] int32 (device) replaces the selection, slot order kept; the
 * router still computes the gate weights over those ids.  Replaying the ids
 * that moe_forward chose reproduces its output bitwise.  ids_out receives
 * the ids actually used. */
moe_status moe_forward_replay(const moe_dims *dims, const void *x,
                              const moe_weights *w, const int32_t *ids_in,
                              void *out, int32_t *ids_out, float *gates_out,
                              void *ws, size_t ws_bytes, moe_stream_t stream);

/* Router replay with the plausibility filter of [TR] §6.2 (replayed experts
 * whose gate score falls below a threshold derived from the router's own
 * top-k are dropped and replaced by the router's candidates).  The threshold is
 * not given on the pages; this library reads it as a fraction tau of the own
 * k-th expert's softmax score: replayed expert e is kept iff
 *   logit_e >= logit_(own k-th) + ln(tau),   0 <= tau <= 1
 * (tau = 0 keeps every replayed id and equals moe_forward_replay).  Dropped
 * slots, in ascending slot order, take the router's own top-k experts, in its
 * own order, that are not already among the token's ids; gate weights are the
 * softmax over the final ids.  Arguments and outputs as moe_forward_replay;
 * ids_out receives the ids actually used.  The total number of replaced slots
 * of the call is added to status word 3 of the workspace (moe_ws_layout.status
 * + 12 bytes, int32).  tau outside [0, 1] or NaN: MOE_ERR_ARG. */
moe_status moe_forward_replay_filtered(const moe_dims *dims, const void *x,
                                       const moe_weights *w, const int32_t *ids_in,
                                       float tau, void *out, int32_t *ids_out,
                                       float *gates_out, void *ws, size_t ws_bytes,
                                       moe_stream_t stream);

/* Synchronise `stream` and return the device status of the last call that
 * used this workspace: MOE_OK, MOE_ERR_BAD_IDS or MOE_ERR_TIMEOUT (the
 * latter wins when both happened), or MOE_ERR_CUDA if reading it failed. */
moe_status moe_get_status(const void *ws, moe_stream_t stream);

/* Static, human-readable name of a status code. */
const char *moe_status_str(moe_status s);

/* Stages of one layer call, in launch order. */
typedef enum {
    MOE_STAGE_ROUTER_GEMM = 0,  /* logits = x . w_router^T + bias             */
    MOE_STAGE_TOPK = 1,         /* selection or replay check, gate weights    */
    MOE_STAGE_DISPATCH = 2,     /* histogram, offsets, stable permutation     */
    MOE_STAGE_GATHER = 3,       /* token rows into expert order               */
    MOE_STAGE_GATE_UP = 4,      /* grouped gate/up GEMM with SwiGLU           */
    MOE_STAGE_DOWN = 5,         /* grouped down GEMM                          */
    MOE_STAGE_COMBINE = 6,      /* fixed-order weighted sum per token         */
    MOE_NUM_STAGES = 7
} moe_stage;

/* Optional per-stage timing for profiling.  `events` points to
 * 2 * MOE_NUM_STAGES cudaEvent_t handles created by the caller (or is NULL to
 * switch timing off).  While set, every call from the calling host thread
 * records events[2*j] on its stream just before stage j and events[2*j+1]
 * just after it (moe_route records only its two stages).  The setting is per
 * host thread; the library does not own or destroy the events.  Returns
 * MOE_OK. */
moe_status moe_set_stage_events(void *const *events);

/* Routing that allocates nothing -- the pages have no counterpart of this
 * call; it is a convenience of this library.
 *
 * Same computation and outputs as moe_route, bit for bit (ids_out [T][k]
 * int32 and gates_out [T][k] fp32, device pointers the caller owns): it runs
 * the same launch sequence, with the router GEMM's K split into the same
 * fixed parts summed in the same order.  The scratch memory moe_route takes
 * from the caller's workspace (status word, per-token flags, fp32 logits and
 * the router's partial logits) lives in a static device array of 4 MiB inside
 * this library, which every GPU that loads the library holds until the
 * process exits.  It is meant for callers that cannot allocate device memory:
 * an inference engine recording routing decisions inside its decode loop,
 * where all device memory belongs to the engine's own pool and a cudaMalloc
 * would synchronise the device or fail, or a plugin whose host framework
 * hands it only input and output buffers.  The call itself makes no
 * cudaMalloc, cudaFree or other allocating call.
 *
 * Limit: with P = 4 partial-logit buffers when d/64 is a multiple of 4 (else
 * P = 0), 256 + round_up(4*T, 256) + round_up(4*T*E, 256) + P*4*T*E <= 4 MiB
 * (T <= 545 at E = 384, d = 7168); larger requests return MOE_ERR_WORKSPACE
 * before any launch.  Shape, null and alignment errors are reported as for
 * moe_route.
 * Set-up: the first call on a device looks up the array's device address
 * (cudaGetSymbolAddress) with that device current; make that first call before
 * any stream capture begins.
 * Sharing: every call uses the same array, which keeps the last call's
 * contents; the call clears its status word itself.  Calls that overlap on the
 * GPU (other streams, other host threads) race on the array and must be
 * serialised by the caller.  The device status word is not readable through
 * this entry point. */
moe_status moe_route_static(const moe_dims *dims, const void *x, const moe_weights *w,
                            int32_t *ids_out, float *gates_out, moe_stream_t stream);

/* ---- Backward ------------------------------------------------------------
 *
 * The gradient of the layer above for an upstream gradient dout, with the
 * expert ids held fixed (the ids the forward used: its ids_out, own or
 * replayed).  [TR] §6.1, Kernels paragraph: the MoE backward runs its grouped
 * GEMMs in standard MXFP8 -- E4M3 values with one E8M0 scale per block of 32
 * elements (OCP Microscaling Formats v1.0: shared exponent
 * X = floor(log2 max|v|) - 8, elements E4M3(v / 2^X), nearest even, clamped
 * to +-448).  Each grouped-GEMM operand is quantised along that GEMM's
 * contraction axis:
 *     dH  = Q_d(dY) . Q_d(Wd)                    dY = gate * dout (routed rows)
 *     dXp = Q_F(dA) . Q_F(Wg) + Q_F(dB) . Q_F(Wu) dA, dB: SwiGLU backward of dH
 *     dWd = Q_tok(dY)^T . Q_tok(H)
 *     dWg = Q_tok(dA)^T . Q_tok(Xp),  dWu = Q_tok(dB)^T . Q_tok(Xp)
 * where along tokens an expert's blocks start at its first row in dispatch
 * order (pairs t*k + s ascending), the last block zero-padded.  The products
 * are exact and accumulate in fp32 (tcgen05, TMEM): dH and dXp on the
 * block-scaled MXFP8 MMA (E4M3 codes and E8M0 scales of both operands), the
 * weight gradients on bf16 MMAs of the exact MXFP8 values.  The gate and router
 * gradients are not grouped GEMMs and are taken in fp32 from the forward's
 * values: dg_s = dout . Y_s (Y the forward's bf16 expert output),
 * dl_s = w_s (dg_s - sum_s' w_s' dg_s'), d_router[e] = sum over e's rows of
 * dl * x, and dx gets sum_s dl_s Wr[ids_s].  The router bias is an input, not
 * a parameter: it has no gradient.  A token whose replayed ids are rejected
 * has a zero forward row and contributes nothing.
 *
 * dx [T][d] fp32 = (sum_s dXp[slot s] + dXp_shared) + router part, slots
 * ascending; its row for a token depends only on that token (batch
 * invariant).  Weight gradients are fp32 and are written, not accumulated
 * into; each element is one CTA's fixed-order K loop (bitwise repeatable).
 *
 * Limits: bf16 expert weights (MOE_ERR_UNSUPPORTED otherwise); d a multiple of
 * 512 and F of 256 (MOE_ERR_SHAPE otherwise: the block-scaled GEMMs take K in
 * steps of 512); the other limits of the forward.
 */
typedef struct {
    float *d_router;                  /* [E][d]                                  */
    float *d_gate, *d_up;             /* [E][F][d]                               */
    float *d_down;                    /* [E][d][F]                               */
    float *ds_gate, *ds_up, *ds_down; /* shared expert: [F][d], [F][d], [d][F];  */
                                      /* NULL when n_shared == 0                 */
} moe_grads;

/* Bytes of the backward's weight copies (see moe_backward_prepare_weights);
 * 0 for dims the backward does not serve. */
size_t moe_backward_weights_size(const moe_dims *dims);

/* The expert weights quantised along the backward's contraction axes and
 * transposed, into wt (device, caller-owned, moe_backward_weights_size bytes,
 * 16-byte aligned), G = E + n_shared groups (the shared expert is group E),
 * each region starting on a 256-byte boundary: E4M3 codes of Q_d(Wd)^T
 * [G][F][d]; their E8M0 scale bytes [G][F][d/32]; codes of
 * [Q_F(Wg)^T | Q_F(Wu)^T] [G][d][2F]; their scale bytes [G][d][2F/32].
 * Depends on the weights only: call it once per weight update and pass wt to
 * every moe_backward with those weights. */
moe_status moe_backward_prepare_weights(const moe_dims *dims, const moe_weights *w, void *wt,
                                        size_t wt_bytes, moe_stream_t stream);

/* Workspace bytes of moe_backward (0 for dims it does not serve). */
size_t moe_backward_workspace_size(const moe_dims *dims);

/* Offsets (bytes into the backward workspace) of its regions; the first ones
 * are those of the forward workspace (moe_ws_layout), so moe_get_status reads
 * a backward workspace too.  Regions after a call: ids/gates the routing
 * used, poff [E+S+1] int32 padded token offsets per expert (followed by
 * [kpad/64] int32: the group of each 64-row tile, -1 past the last), a/b [rows][F]
 * fp32 gate/up pre-activations, dg/dl [T][k] fp32 gate and logit gradients,
 * dyq: Q_d(dY) as E4M3 codes [rows][d] then E8M0 scale bytes [rows][d/32],
 * dh [rows][F] fp32, dabq: [Q_F(dA) | Q_F(dB)] as codes [rows][2F] then scale
 * bytes [rows][2F/32],
 * dxp [rows][d] fp32, and the token-major operands xpt, dyt [d][kpad],
 * ht [F][kpad], dabt [2F][kpad] (bf16), rows = T*k + T*n_shared. */
typedef struct {
    size_t status, logits, valid, cnt, off, perm, inv, xp, h, y;
    size_t ids, gates, poff, a, b, dg, dl, dyq, dh, dabq, dxp, xpt, dyt, ht, dabt;
    size_t kpad; /* elements per row of the token-major operands */
    size_t total;
} moe_bwd_ws_layout;
moe_status moe_backward_workspace_layout(const moe_dims *dims, moe_bwd_ws_layout *layout);

/* Stages of the backward, in launch order (moe_backward_prepare_weights
 * records only MOE_BWD_STAGE_PREPARE). */
typedef enum {
    MOE_BWD_STAGE_PREPARE = 0,        /* weight copies quantised along the backward's K */
    MOE_BWD_STAGE_ROUTE = 1,          /* router GEMM, replay check, gate weights        */
    MOE_BWD_STAGE_DISPATCH = 2,       /* counting sort, padded offsets, gather          */
    MOE_BWD_STAGE_GATE_UP = 3,        /* forward recompute: gate/up (H, pre-activations)*/
    MOE_BWD_STAGE_DOWN = 4,           /* forward recompute: routed expert outputs Y     */
    MOE_BWD_STAGE_GATE = 5,           /* gate/logit gradients, router part of dx, dWr   */
    MOE_BWD_STAGE_DY = 6,             /* dY quantised along d and along tokens          */
    MOE_BWD_STAGE_DH = 7,             /* dH = Q(dY) Q(Wd)                               */
    MOE_BWD_STAGE_SWIGLU = 8,         /* SwiGLU backward, [dA | dB] quantised along F   */
    MOE_BWD_STAGE_DXP = 9,            /* dXp = Q(dA) Q(Wg) + Q(dB) Q(Wu)                */
    MOE_BWD_STAGE_DX = 10,            /* fixed-order sum into dx                        */
    MOE_BWD_STAGE_TRANSPOSE = 11,     /* token-major Xp and H quantised along tokens    */
    MOE_BWD_STAGE_WGRAD_DOWN = 12,    /* dWd                                            */
    MOE_BWD_STAGE_WGRAD_GATE_UP = 13, /* dWg, dWu                                       */
    MOE_BWD_NUM_STAGES = 14
} moe_bwd_stage;

/* Per-stage timing of the backward, as moe_set_stage_events for the forward:
 * `events` holds 2 * MOE_BWD_NUM_STAGES cudaEvent_t handles (or is NULL to
 * switch it off); events[2*j] / events[2*j+1] are recorded on the call's
 * stream just before / after stage j.  Per host thread.  Returns MOE_OK. */
moe_status moe_set_backward_stage_events(void *const *events);

/* The backward.  x [T][d] bf16, w (bf16 experts), wt (prepared from w), ids
 * [T][k] int32 (the forward's ids), dout [T][d] bf16 -> dx [T][d] fp32 and the
 * weight gradients in *grads (all device pointers).  Replayed ids are checked
 * as in moe_forward_replay (moe_get_status reports MOE_ERR_BAD_IDS).
 * Stream-ordered; no synchronisation. */
moe_status moe_backward(const moe_dims *dims, const void *x, const moe_weights *w,
                        const void *wt, const int32_t *ids, const void *dout, float *dx,
                        const moe_grads *grads, void *ws, size_t ws_bytes, moe_stream_t stream);

/* Training without the forward recompute: moe_forward_train is the layer
 * forward (own routing when ids_in is NULL, replay otherwise -- same outputs,
 * bitwise, as moe_forward / moe_forward_replay) run in a BACKWARD workspace
 * (moe_backward_workspace_size), where it leaves what the backward reads: the
 * routing, the gathered rows, H, the fp32 gate/up pre-activations and the
 * routed expert outputs.  moe_backward_saved then computes exactly what
 * moe_backward computes for the same x, weights, ids and dout (bitwise), from
 * that workspace, without routing, dispatch or the forward's expert GEMMs.
 * The caller keeps the workspace untouched in between and passes the same
 * dims and weights to both calls; nothing checks that it did. */
moe_status moe_forward_train(const moe_dims *dims, const void *x, const moe_weights *w,
                             const int32_t *ids_in, void *out, int32_t *ids_out,
                             float *gates_out, void *ws, size_t ws_bytes, moe_stream_t stream);
moe_status moe_backward_saved(const moe_dims *dims, const moe_weights *w, const void *wt,
                              const void *dout, float *dx, const moe_grads *grads, void *ws,
                              size_t ws_bytes, moe_stream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* MOE_DET_H */
