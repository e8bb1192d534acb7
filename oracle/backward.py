"""fp64 CPU oracle of the MoE layer backward, with MXFP8 expert GEMMs.

TEST INFRASTRUCTURE ONLY.  The product path (the CUDA library under
``deterministic_rl_gb300/`` and its binding) never imports or calls anything
here; only ``tests/``, ``__graft_entry__.smoke()`` and the CPU legs of
``bench.py`` do.  It shares no code with the CUDA path.

What it computes -- the gradient of the layer forward (router logits, gate
weights = softmax over the chosen experts' logits, SwiGLU experts, the
always-on shared expert with weight 1, fixed-order combine) for a given
upstream gradient ``dout``, with the expert ids held fixed (the ids the forward
used, own or replayed):

* Composer 2 Technical Report, §6.1 "Training infrastructure" (Kernels): the
  MoE backward runs its grouped GEMMs in the standard MXFP8 format, FP8 E4M3
  values with one FP8 E8M0 scale per block of 32 elements; the forward's
  per-expert grouped GEMMs (Fig. 10) are the ones differentiated here.
* MXFP8 as the OCP Microscaling Formats (MX) v1.0 specification defines it:
  per block, shared exponent X = floor(log2(max |v|)) - 8 (8 = the exponent of
  E4M3's largest normal, 448 = 1.75 * 2^8), E8M0 byte X + 127, elements
  E4M3(v / 2^X) rounded to nearest even and clamped to +-448.
* §6.2 "RL infrastructure": with router replay the router still computes the
  gate scores, so gradients reach the router through the gate weights.

Readings where the pages are silent (each one is a step below):
  1. Each grouped-GEMM operand is quantised along that GEMM's contraction
     axis (blocks never straddle two experts): dH = Q_d(dY) Q_d(Wd);
     dXp = Q_F(dA) Q_F(Wg) + Q_F(dB) Q_F(Wu); dWd = Q_tok(dY)^T Q_tok(H);
     dWg = Q_tok(dA)^T Q_tok(Xp); dWu = Q_tok(dB)^T Q_tok(Xp).
  2. Along tokens, an expert's blocks start at its first row in dispatch
     order (pairs t*k + s ascending); a partial last block holds fewer values
     (equivalently: padded with zeros, which never change a block maximum).
  3. The gate and router gradients are not grouped GEMMs: they are taken in
     full precision from the forward's values.
  4. The forward's stored tensors are used as the forward stores them: H and
     the routed expert outputs Y rounded to bf16 (round_storage=True).
  5. The router bias is a fixed input, not a parameter: it has no gradient.
  6. Tokens whose replayed ids were invalid have a zero forward row, hence a
     zero gradient everywhere.
With quant=False and round_storage=False every step is exact and the result
is the exact gradient of the forward below, which tests/test_oracle_pins.py
checks against central finite differences, and whose forward it checks
against the C oracle.  The quantiser is pinned separately (golden blocks,
the float8_e4m3fn cast, closed forms, a planted-outlier test of the axis).
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import Callable, Dict, List, Optional, Sequence

import numpy as np

E4M3_MAX = 448.0
E4M3_EMAX = 8          # exponent of the largest normal E4M3 value
MX_BLOCK = 32


# ---- MXFP8 quantisation -------------------------------------------------------

def round_e4m3(v: np.ndarray) -> np.ndarray:
    """E4M3 (OCP FP8, 4 exponent bits, bias 7, 3 mantissa bits, no infinities)
    of fp64 values: nearest, ties to even, clamped to +-448.  Normal values
    above 2^-6 have 3 fraction bits; below, the quantum is the subnormal step
    2^-9."""
    v = np.asarray(v, np.float64)
    a = np.abs(v)
    with np.errstate(divide="ignore"):
        e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    # log2 of an exact power of two is exact; guard values just below one
    e = np.where(np.ldexp(1.0, e.astype(np.int64)) > a, e - 1, e)
    e = np.where(np.ldexp(1.0, (e + 1).astype(np.int64)) <= a, e + 1, e)
    e = np.maximum(e, -6.0)
    quantum = np.ldexp(1.0, (e - 3).astype(np.int64))
    q = np.rint(a / quantum) * quantum          # a / quantum is exact
    q = np.minimum(q, E4M3_MAX)
    return np.copysign(q, v) * (a > 0)


def mx_exponent(amax: np.ndarray) -> np.ndarray:
    """Shared exponent X of a block with largest magnitude amax (OCP MX v1.0):
    floor(log2 amax) - 8, within the E8M0 range [-127, 127]; -127 (E8M0 byte
    0) for an all-zero block."""
    amax = np.asarray(amax, np.float64)
    pos = amax > 0
    with np.errstate(divide="ignore"):
        e = np.floor(np.log2(np.where(pos, amax, 1.0)))
    e = np.where(np.ldexp(1.0, e.astype(np.int64)) > amax, e - 1, e)
    e = np.where(np.ldexp(1.0, (e + 1).astype(np.int64)) <= amax, e + 1, e)
    x = np.where(pos, e - E4M3_EMAX, -127.0)
    return np.clip(x, -127, 127).astype(np.int64)


def mx_quantize(v: np.ndarray, axis: int) -> np.ndarray:
    """MXFP8 quantise-dequantise of v along `axis` in blocks of 32 consecutive
    values (the axis length is padded with zeros to a multiple of 32, which
    changes no block maximum): returns E4M3(v / 2^X) * 2^X per block, fp64."""
    v = np.asarray(v, np.float64)
    v = np.moveaxis(v, axis, -1)
    n = v.shape[-1]
    pad = (-n) % MX_BLOCK
    if pad:
        v = np.concatenate([v, np.zeros(v.shape[:-1] + (pad,))], axis=-1)
    blocks = v.reshape(v.shape[:-1] + (-1, MX_BLOCK))
    X = mx_exponent(np.abs(blocks).max(axis=-1))[..., None]
    q = round_e4m3(np.ldexp(blocks, -X)) * np.ldexp(1.0, X)
    q = q.reshape(v.shape)[..., :n]
    return np.moveaxis(q, -1, axis)


def qmatmul_nt(a: np.ndarray, b: np.ndarray, quant: bool) -> np.ndarray:
    """C[i][j] = sum_k Q(a)[i][k] * Q(b)[j][k], both operands quantised along
    the contraction axis k (their last axis) when quant is set."""
    if quant:
        a = mx_quantize(a, -1)
        b = mx_quantize(b, -1)
    return a @ b.T


# ---- the forward, on fp64 values (for the pins; the C oracle is the reference) --

def bf16_round(v: np.ndarray) -> np.ndarray:
    """Round fp64 values to bf16 (8 significant bits), nearest, ties to even.
    Values below bf16's normal range (2^-126) are outside what the layer
    produces and are not treated specially."""
    v = np.asarray(v, np.float64)
    m, e = np.frexp(np.abs(v))                 # |v| = m * 2^e, m in [0.5, 1)
    q = np.ldexp(np.rint(np.ldexp(m, 8)), e - 8)
    return np.copysign(q, v)


def silu(a: np.ndarray) -> np.ndarray:
    return a / (1.0 + np.exp(-a))


def dsilu(a: np.ndarray) -> np.ndarray:
    # d/da [a * sigmoid(a)] = sigmoid(a) * (1 + a * (1 - sigmoid(a)))
    sg = 1.0 / (1.0 + np.exp(-a))
    return sg * (1.0 + a * (1.0 - sg))


@dataclass
class ExpertValues:
    """One expert's weights as fp64 values: w_gate, w_up [F][d]; w_down [d][F]."""
    w_gate: np.ndarray
    w_up: np.ndarray
    w_down: np.ndarray


def gates_from_logits(logits: np.ndarray, ids: np.ndarray) -> np.ndarray:
    """w_s = exp(l_s - m) / sum_s' exp(l_s' - m) over the chosen ids, m their max."""
    lg = np.take_along_axis(logits, ids.astype(np.int64), axis=1)
    m = lg.max(axis=1, keepdims=True)
    e = np.exp(lg - m)
    return e / e.sum(axis=1, keepdims=True)


def dispatch_rows(ids: np.ndarray, E: int) -> List[np.ndarray]:
    """Per expert, the pairs i = t*k + s routed to it, ascending (the stable
    counting-sort order of the dispatch)."""
    flat = ids.reshape(-1)
    return [np.nonzero(flat == e)[0] for e in range(E)]


def layer_forward_values(x: np.ndarray, wr: np.ndarray, bias: Optional[np.ndarray],
                         experts: Sequence[ExpertValues], shared: Sequence[ExpertValues],
                         ids: np.ndarray, valid: Optional[np.ndarray] = None) -> np.ndarray:
    """The layer output for fixed ids, exactly (fp64, no storage rounding):
    out_t = sum_s w_s * expert_{ids[t,s]}(x_t) + sum over shared experts."""
    T, k = ids.shape
    logits = x @ wr.T + (0.0 if bias is None else bias[None, :])
    w = gates_from_logits(logits, ids)
    out = np.zeros((T, x.shape[1]))
    for e, pairs in enumerate(dispatch_rows(ids, len(experts))):
        if pairs.size == 0:
            continue
        ex = experts[e]
        xt = x[pairs // k]
        h = silu(xt @ ex.w_gate.T) * (xt @ ex.w_up.T)
        y = h @ ex.w_down.T
        np.add.at(out, pairs // k, w.reshape(-1)[pairs, None] * y)
    for ex in shared:
        h = silu(x @ ex.w_gate.T) * (x @ ex.w_up.T)
        out += h @ ex.w_down.T
    if valid is not None:
        out = out * (valid != 0)[:, None]
    return out


# ---- the backward -------------------------------------------------------------

@dataclass
class ExpertGrads:
    d_gate: np.ndarray   # [F][d]
    d_up: np.ndarray     # [F][d]
    d_down: np.ndarray   # [d][F]


@dataclass
class BackwardResult:
    dx: np.ndarray                    # [T][d]
    d_router: np.ndarray              # [E][d]
    experts: Dict[int, ExpertGrads]   # routed experts asked for (all by default)
    shared: List[ExpertGrads]
    dgates: np.ndarray                # [T][k]  dL/dw_s
    dlogits: np.ndarray               # [T][k]  dL/dl_{ids[t,s]}
    dx_router: np.ndarray             # [T][d]  the router's part of dx


def expert_backward(xt: np.ndarray, dy: np.ndarray, ex: ExpertValues, quant: bool,
                    round_storage: bool, want_dx: bool = True, want_dw: bool = True):
    """One expert over its rows (in dispatch order): xt [n][d] its input rows,
    dy [n][d] the gradient of its output rows (gate weight applied).  Returns
    (dXp [n][d] or None, ExpertGrads or None)."""
    a = xt @ ex.w_gate.T                       # [n][F]
    b = xt @ ex.w_up.T
    h = silu(a) * b
    if round_storage:
        h = bf16_round(h)
    # dH = dY Wd: contraction over d; Wd [d][F] is read along its first axis
    dh = qmatmul_nt(dy, ex.w_down.T, quant)    # [n][F]
    da = dh * b * dsilu(a)
    db = dh * silu(a)
    dxp = None
    if want_dx:
        # dXp = dA Wg + dB Wu: contraction over F (Wg, Wu [F][d] read along F)
        dxp = qmatmul_nt(da, ex.w_gate.T, quant) + qmatmul_nt(db, ex.w_up.T, quant)
    grads = None
    if want_dw:
        # contraction over the expert's tokens: operands quantised along axis 0
        grads = ExpertGrads(
            d_gate=qmatmul_nt(da.T, xt.T, quant),   # [F][d]
            d_up=qmatmul_nt(db.T, xt.T, quant),
            d_down=qmatmul_nt(dy.T, h.T, quant))    # [d][F]
    return dxp, grads


def layer_backward(x: np.ndarray, wr: np.ndarray, bias: Optional[np.ndarray],
                   get_expert: Callable[[int], ExpertValues], shared: Sequence[ExpertValues],
                   ids: np.ndarray, dout: np.ndarray, valid: Optional[np.ndarray] = None,
                   quant: bool = True, round_storage: bool = True,
                   grad_experts: Optional[Sequence[int]] = None,
                   tokens: Optional[Sequence[int]] = None,
                   grad_shared: bool = True) -> BackwardResult:
    """Gradient of sum(dout * out) w.r.t. x, the router weights and the
    experts' weights, for the layer of layer_forward_values with ids fixed.

    x [T][d], wr [E][d], dout [T][d]: fp64 values (bf16 values in practice).
    get_expert(e) gives expert e's weights (called at most once per expert,
    ascending).  The limits below only skip work; a value that is formed does
    not depend on them:
      tokens        tokens whose dx row, gate gradients and logit gradients
                    are formed (None: all; other rows stay zero).  Row e of
                    d_router sums over the formed tokens routed to e, so it is
                    complete when every token routed to e is formed.
      grad_experts  routed experts whose weight gradients are formed (None:
                    every expert with tokens).
      grad_shared   whether the shared experts' weight gradients are formed.
    """
    T, k = ids.shape
    d = x.shape[1]
    E = wr.shape[0]
    ids = np.asarray(ids).astype(np.int64)
    ok = np.ones(T, bool) if valid is None else (np.asarray(valid) != 0)
    dout = dout * ok[:, None]
    logits = x @ wr.T + (0.0 if bias is None else bias[None, :])
    w = gates_from_logits(logits, ids)
    want_tok = np.zeros(T, bool)
    if tokens is None:
        want_tok[:] = True
    else:
        want_tok[np.asarray(tokens, np.int64)] = True
    dw_set = None if grad_experts is None else set(int(e) for e in grad_experts)

    dgates = np.zeros((T, k))
    dxp_slots = np.zeros((T, k, d))
    eg: Dict[int, ExpertGrads] = {}
    for e, pairs in enumerate(dispatch_rows(ids, E)):
        if pairs.size == 0:
            continue
        need_dw = dw_set is None or e in dw_set
        sel = want_tok[pairs // k]
        if not need_dw and not sel.any():
            continue
        ex = get_expert(e)
        rows = pairs if need_dw else pairs[sel]   # dispatch order kept
        rt = rows // k
        xt = x[rt]
        # the forward's expert output, for the gate gradient: Y = H Wd^T
        h = silu(xt @ ex.w_gate.T) * (xt @ ex.w_up.T)
        if round_storage:
            h = bf16_round(h)
        y = h @ ex.w_down.T
        if round_storage:
            y = bf16_round(y)
        dgates.reshape(-1)[rows] = np.einsum("nd,nd->n", dout[rt], y)
        dy = w.reshape(-1)[rows, None] * dout[rt]
        dxp, grads = expert_backward(xt, dy, ex, quant, round_storage, want_dx=True,
                                     want_dw=need_dw)
        dxp_slots.reshape(T * k, d)[rows] = dxp
        if grads is not None:
            eg[e] = grads
    # the gate weights are a softmax over the chosen logits:
    # dL/dl_s = w_s * (dL/dw_s - sum_s' w_s' dL/dw_s')
    dlog = w * (dgates - (w * dgates).sum(axis=1, keepdims=True))
    dlog = dlog * (ok & want_tok)[:, None]
    # logits = x Wr^T + b
    d_router = np.zeros((E, d))
    np.add.at(d_router, ids.reshape(-1), dlog.reshape(-1, 1) * np.repeat(x, k, axis=0))
    dx_router = np.einsum("ts,tsd->td", dlog, wr[ids])
    dx_sh = np.zeros((T, d))
    sg: List[ExpertGrads] = []
    for ex in shared:
        if grad_shared:
            dxs, grads = expert_backward(x, dout, ex, quant, round_storage)
            dx_sh += dxs
            sg.append(grads)
        else:
            tw = np.nonzero(want_tok)[0]
            dxs, _ = expert_backward(x[tw], dout[tw], ex, quant, round_storage, want_dw=False)
            dx_sh[tw] += dxs
    dx = dxp_slots.sum(axis=1) + dx_sh + dx_router
    dx[~want_tok] = 0.0
    return BackwardResult(dx=dx, d_router=d_router, experts=eg, shared=sg, dgates=dgates,
                          dlogits=dlog, dx_router=dx_router)
