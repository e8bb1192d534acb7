"""fp64 CPU oracle of the deterministic MoE layer forward with router replay.

TEST INFRASTRUCTURE ONLY.  The product path (the CUDA library under
``deterministic_rl_gb300/`` and its binding) never imports, links or calls
anything here; only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline
leg of ``bench.py`` do.  The oracle shares no code with the CUDA path: the
arithmetic lives in ``moe_oracle.c`` (plain C, fp64); this module only builds
it, marshals numpy arrays into it and sequences its per-token steps.

Sources (see ``moe_oracle.h`` for the full statement of the definition):
  * Composer 2 Technical Report, §6.2 "RL infrastructure" (router replay:
    recorded expert indices override the router's selection, the router still
    computes the gate scores) and §6.1 "Training infrastructure" (grouped
    expert GEMMs, dispatch/combine, MXFP8 format, and the NVFP4 forward with
    per-token scales and IEEE division in the quantiser).
  * Training Data No. 94 write-up, section "浮点数不守规矩，MoE 火上浇油", and
    the "五大工程挑戰" write-up, section "浮點數的陷阱": 8 of 384 experts per
    token, fixed-order accumulation.

Every function here is pinned by ``tests/test_oracle_pins.py`` to closed
forms, library routines and brute force; none is "parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import platform
import subprocess
import threading
from dataclasses import dataclass
from typing import Callable, Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_LIB_PATH = os.path.join(_HERE, f"liboracle.{platform.machine()}.so")
_lib = None
_lock = threading.Lock()

W_BF16 = 0
W_MXFP8 = 1
W_NVFP4 = 2
W_MXFP8_ACT = 3


def build(force: bool = False) -> str:
    """Compile moe_oracle.c into liboracle.so next to it (gcc, OpenMP)."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= max(os.path.getmtime(_SRC),
                                                   os.path.getmtime(os.path.join(_HERE, "moe_oracle.h")))):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared", "-fopenmp", "-Wall",
           "-o", tmp, _SRC, "-lm"]
    subprocess.check_call(cmd)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


class _Matrix(ctypes.Structure):
    _fields_ = [("fmt", ctypes.c_int), ("values", ctypes.c_void_p),
                ("scales", ctypes.c_void_p), ("tscale", ctypes.c_float)]


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        build()
        lib = ctypes.CDLL(_LIB_PATH)
        P = ctypes.c_void_p
        I = ctypes.c_int64
        lib.oracle_bf16_to_f64.restype = ctypes.c_double
        lib.oracle_bf16_to_f64.argtypes = [ctypes.c_uint16]
        lib.oracle_e4m3_to_f64.restype = ctypes.c_double
        lib.oracle_e4m3_to_f64.argtypes = [ctypes.c_uint8]
        lib.oracle_e8m0_to_f64.restype = ctypes.c_double
        lib.oracle_e8m0_to_f64.argtypes = [ctypes.c_uint8]
        lib.oracle_e2m1_to_f64.restype = ctypes.c_double
        lib.oracle_e2m1_to_f64.argtypes = [ctypes.c_uint8]
        lib.oracle_e2m1_round.restype = ctypes.c_uint8
        lib.oracle_e2m1_round.argtypes = [ctypes.c_float]
        lib.oracle_e4m3_round.restype = ctypes.c_uint8
        lib.oracle_e4m3_round.argtypes = [ctypes.c_float]
        lib.oracle_round_bf16.restype = ctypes.c_double
        lib.oracle_round_bf16.argtypes = [ctypes.c_double]
        lib.oracle_nvfp4_quantize_rows.restype = None
        lib.oracle_nvfp4_quantize_rows.argtypes = [P, I, I, P, P, P]
        lib.oracle_mx_qdq_rows.restype = None
        lib.oracle_mx_qdq_rows.argtypes = [P, I, I, P]
        lib.oracle_matrix_elem.restype = ctypes.c_double
        lib.oracle_matrix_elem.argtypes = [ctypes.POINTER(_Matrix), I, I, I]
        lib.oracle_router_logits.restype = None
        lib.oracle_router_logits.argtypes = [P, P, P, I, I, I, P]
        lib.oracle_select_topk.restype = None
        lib.oracle_select_topk.argtypes = [P, I, I, I, P]
        lib.oracle_check_ids.restype = ctypes.c_int64
        lib.oracle_check_ids.argtypes = [P, I, I, I, P]
        lib.oracle_filter_replay.restype = None
        lib.oracle_filter_replay.argtypes = [P, P, I, I, I, ctypes.c_double, P, P]
        lib.oracle_gate_weights.restype = None
        lib.oracle_gate_weights.argtypes = [P, P, I, I, I, P]
        lib.oracle_counting_sort.restype = None
        lib.oracle_counting_sort.argtypes = [P, I, I, P, P, P, P]
        lib.oracle_expert_ffn.restype = None
        lib.oracle_expert_ffn.argtypes = [P, I, I, I, ctypes.POINTER(_Matrix),
                                          ctypes.POINTER(_Matrix), ctypes.POINTER(_Matrix), P]
        lib.oracle_combine.restype = None
        lib.oracle_combine.argtypes = [P, P, P, P, I, I, I, P]
        lib.oracle_set_threads.restype = ctypes.c_int
        lib.oracle_set_threads.argtypes = [ctypes.c_int]
        lib.oracle_get_threads.restype = ctypes.c_int
        lib.oracle_get_threads.argtypes = []
        _lib = lib
        return lib


def _ptr(a: Optional[np.ndarray]):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


# ---- scalar decoders -------------------------------------------------------

def bf16_to_f64(h: int) -> float:
    return _load().oracle_bf16_to_f64(int(h) & 0xFFFF)


def e4m3_to_f64(b: int) -> float:
    return _load().oracle_e4m3_to_f64(int(b) & 0xFF)


def e8m0_to_f64(s: int) -> float:
    return _load().oracle_e8m0_to_f64(int(s) & 0xFF)


def e2m1_to_f64(code: int) -> float:
    return _load().oracle_e2m1_to_f64(int(code) & 0xF)


def e2m1_round(v: float) -> int:
    return int(_load().oracle_e2m1_round(float(v)))


def e4m3_round(v: float) -> int:
    return int(_load().oracle_e4m3_round(float(v)))


def round_bf16(v: float) -> float:
    return _load().oracle_round_bf16(float(v))


def nvfp4_quantize_rows(x: np.ndarray):
    """NVFP4 with per-row (per-token) scales, the quantiser of the NVFP4
    forward: x [R][K] fp32 (bf16 values) -> (codes uint8 [R][K], block scales
    uint8 E4M3 [R][K/16], row scales float32 [R])."""
    x = _c(x, np.float32)
    R, K = x.shape
    assert K % 16 == 0
    codes = np.empty((R, K), np.uint8)
    bs = np.empty((R, K // 16), np.uint8)
    rs = np.empty(R, np.float32)
    _load().oracle_nvfp4_quantize_rows(_ptr(x), R, K, _ptr(codes), _ptr(bs), _ptr(rs))
    return codes, bs, rs


def mx_qdq_rows(x: np.ndarray) -> np.ndarray:
    """MXFP8 quantise-dequantise of each row of x [R][K] (K % 32 == 0) in blocks
    of 32 along the row (OCP MX v1.0, E4M3 elements); fp64 in and out."""
    x = _c(x, np.float64)
    R, K = x.shape
    assert K % 32 == 0
    out = np.empty((R, K), np.float64)
    _load().oracle_mx_qdq_rows(_ptr(x), R, K, _ptr(out))
    return out


# ---- weights ----------------------------------------------------------------

@dataclass
class Matrix:
    """One weight matrix [rows][K] as raw storage: bf16 bit patterns (uint16);
    or E4M3 bytes (uint8) plus E8M0 scale bytes [rows][K//32]; or (NVFP4, when
    tscale is given) E2M1 codes packed two per byte [rows][K//2] plus E4M3
    scale bytes [rows][K//16] and the matrix's fp32 scale."""
    values: np.ndarray
    scales: Optional[np.ndarray] = None
    tscale: Optional[float] = None
    act_mx: bool = False  # MXFP8 weights whose expert FFN quantises its activations too

    @property
    def fmt(self) -> int:
        if self.tscale is not None:
            return W_NVFP4
        if self.scales is None:
            return W_BF16
        return W_MXFP8_ACT if self.act_mx else W_MXFP8

    @property
    def K(self) -> int:
        return self.values.shape[-1] * (2 if self.fmt == W_NVFP4 else 1)

    def _struct(self) -> _Matrix:
        if self.fmt == W_BF16:
            assert self.values.dtype == np.uint16
        else:
            assert self.values.dtype == np.uint8 and self.scales.dtype == np.uint8
        return _Matrix(self.fmt, _ptr(self.values), _ptr(self.scales),
                       float(self.tscale) if self.tscale is not None else 0.0)

    def elem(self, r: int, c: int) -> float:
        K = self.K
        st = self._struct()
        return _load().oracle_matrix_elem(ctypes.byref(st), K, r, c)


@dataclass
class Expert:
    w_gate: Matrix   # [F][d]
    w_up: Matrix     # [F][d]
    w_down: Matrix   # [d][F]


# ---- the steps of the layer -------------------------------------------------

def router_logits(x: np.ndarray, w_router: np.ndarray,
                  bias: Optional[np.ndarray]) -> np.ndarray:
    """x [T][d] uint16 (bf16 bits), w_router [E][d] uint16, bias [E] fp32."""
    x = _c(x, np.uint16)
    wr = _c(w_router, np.uint16)
    T, d = x.shape
    E = wr.shape[0]
    assert wr.shape[1] == d
    b = None if bias is None else _c(bias, np.float32)
    out = np.empty((T, E), np.float64)
    _load().oracle_router_logits(_ptr(x), _ptr(wr), _ptr(b), T, d, E, _ptr(out))
    return out


def select_topk(logits: np.ndarray, k: int) -> np.ndarray:
    lg = _c(logits, np.float64)
    T, E = lg.shape
    assert 1 <= k <= E
    ids = np.empty((T, k), np.int32)
    _load().oracle_select_topk(_ptr(lg), T, E, k, _ptr(ids))
    return ids


def check_ids(ids: np.ndarray, E: int) -> np.ndarray:
    ids = _c(ids, np.int32)
    T, k = ids.shape
    valid = np.empty(T, np.uint8)
    _load().oracle_check_ids(_ptr(ids), T, E, k, _ptr(valid))
    return valid


def filter_replay(logits: np.ndarray, ids: np.ndarray, tau: float):
    """Replay plausibility filter: returns (ids [T][k] int32, replaced [T] int32)."""
    lg = _c(logits, np.float64)
    ids = _c(ids, np.int32)
    T, E = lg.shape
    k = ids.shape[1]
    out = np.empty((T, k), np.int32)
    rep = np.empty(T, np.int32)
    _load().oracle_filter_replay(_ptr(lg), _ptr(ids), T, E, k, float(tau), _ptr(out), _ptr(rep))
    return out, rep


def gate_weights(logits: np.ndarray, ids: np.ndarray) -> np.ndarray:
    lg = _c(logits, np.float64)
    ids = _c(ids, np.int32)
    T, E = lg.shape
    k = ids.shape[1]
    g = np.empty((T, k), np.float64)
    _load().oracle_gate_weights(_ptr(lg), _ptr(ids), T, E, k, _ptr(g))
    return g


def counting_sort(ids: np.ndarray, E: int):
    """Returns (cnt[E], off[E+1], perm[n], inv[n]) as int32 for the pairs
    i = t*k + s of ids (flattened row-major)."""
    flat = _c(ids, np.int32).reshape(-1)
    n = flat.shape[0]
    assert n == 0 or (flat.min() >= 0 and flat.max() < E)
    cnt = np.empty(E, np.int32)
    off = np.empty(E + 1, np.int32)
    perm = np.empty(n, np.int32)
    inv = np.empty(n, np.int32)
    _load().oracle_counting_sort(_ptr(flat), n, E, _ptr(cnt), _ptr(off), _ptr(perm), _ptr(inv))
    return cnt, off, perm, inv


def expert_ffn(x: np.ndarray, ex: Expert) -> np.ndarray:
    """x [n][d] uint16 bf16 bits -> y [n][d] fp64."""
    x = _c(x, np.uint16)
    n, d = x.shape
    F = ex.w_gate.values.shape[0]
    assert ex.w_gate.K == d and ex.w_up.K == d and ex.w_up.values.shape[0] == F
    assert ex.w_down.values.shape[0] == d and ex.w_down.K == F
    assert len({ex.w_gate.fmt, ex.w_up.fmt, ex.w_down.fmt}) == 1
    y = np.empty((n, d), np.float64)
    if n == 0:
        return y
    g, u, dn = ex.w_gate._struct(), ex.w_up._struct(), ex.w_down._struct()
    _load().oracle_expert_ffn(_ptr(x), n, d, F, ctypes.byref(g), ctypes.byref(u),
                              ctypes.byref(dn), _ptr(y))
    return y


def combine(y_slots: np.ndarray, gates: np.ndarray, y_shared: Optional[np.ndarray],
            valid: Optional[np.ndarray]) -> np.ndarray:
    ys = _c(y_slots, np.float64)
    T, k, d = ys.shape
    g = _c(gates, np.float64)
    sh = None if y_shared is None else _c(y_shared, np.float64)
    v = None if valid is None else _c(valid, np.uint8)
    out = np.empty((T, d), np.float64)
    _load().oracle_combine(_ptr(ys), _ptr(g), _ptr(sh), _ptr(v), T, k, d, _ptr(out))
    return out


def set_threads(n: int) -> int:
    return _load().oracle_set_threads(int(n))


def get_threads() -> int:
    return _load().oracle_get_threads()


# ---- the layer, step by step ------------------------------------------------

@dataclass
class LayerResult:
    out: np.ndarray      # [T][d] fp64
    ids: np.ndarray      # [T][k] int32 (ids used; sanitised rows for invalid replay tokens)
    gates: np.ndarray    # [T][k] fp64
    logits: np.ndarray   # [T][E] fp64
    valid: np.ndarray    # [T] uint8


def layer_forward(x: np.ndarray, w_router: np.ndarray, bias: Optional[np.ndarray],
                  get_expert: Callable[[int], Expert], shared: Sequence[Expert],
                  k: int, replay_ids: Optional[np.ndarray] = None,
                  filter_tau: Optional[float] = None) -> LayerResult:
    """The MoE layer for the tokens in x, in the order the definition reads:
    logits -> selection (own) or recorded ids (replay) -> gate weights ->
    each chosen expert's FFN on the token -> fixed-order combine.

    get_expert(e) returns expert e's weights; it is called once per distinct
    expert the tokens use, in ascending e, so that large layers can be fed
    one expert at a time.  Replay tokens with invalid ids produce a zero row.
    With filter_tau, the replayed ids of valid tokens first pass the replay
    plausibility filter.
    """
    x = _c(x, np.uint16)
    T, d = x.shape
    E = w_router.shape[0]
    logits = router_logits(x, w_router, bias)
    if replay_ids is None:
        ids = select_topk(logits, k)
        valid = np.ones(T, np.uint8)
    else:
        ids = _c(replay_ids, np.int32).copy()
        assert ids.shape == (T, k)
        valid = check_ids(ids, E)
        ids[valid == 0] = np.arange(k, dtype=np.int32)
        if filter_tau is not None:
            ids, _ = filter_replay(logits, ids, filter_tau)
            ids[valid == 0] = np.arange(k, dtype=np.int32)
    gates = gate_weights(logits, ids)
    gates[valid == 0] = 0.0
    y_slots = np.zeros((T, k, d), np.float64)
    flat = ids.reshape(-1)
    for e in np.unique(flat):
        pairs = np.nonzero(flat == e)[0]
        toks = pairs // k
        y = expert_ffn(x[toks], get_expert(int(e)))
        y_slots.reshape(T * k, d)[pairs] = y
    y_sh = None
    for ex in shared:
        ys = expert_ffn(x, ex)
        y_sh = ys if y_sh is None else _sum_shared(y_sh, ys)
    out = combine(y_slots, gates, y_sh, valid)
    return LayerResult(out=out, ids=ids, gates=gates, logits=logits, valid=valid)


def _sum_shared(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    # More than one shared expert: outputs added in shared-expert order.
    return a + b
