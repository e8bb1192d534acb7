"""Pins of the fp64 oracle to things other than itself: exact decoders checked
against torch's dtype conversions, brute force on tiny inputs, library routines
(numpy/scipy/torch fp64), closed forms and a hand-worked layer
(tests/golden/hand_worked_layer.json).  CPU only."""
import json
import math
import os

import numpy as np
import pytest
import scipy.special
import torch

import oracle
from oracle import Expert, Matrix

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def bf16(a) -> np.ndarray:
    """float array -> bf16 bit patterns (round to nearest even, via torch)."""
    t = torch.as_tensor(np.asarray(a, np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def f64(bits: np.ndarray) -> np.ndarray:
    return torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).double().numpy()


def rand_bf16(rng, shape, std=1.0):
    return bf16(rng.standard_normal(shape) * std)


# ---- decoders ----------------------------------------------------------------

def test_bf16_decode_all_patterns():
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    ref = f64(bits)
    lib = oracle._load()
    got = np.array([lib.oracle_bf16_to_f64(int(b)) for b in bits[::7]])
    r = ref[::7]
    nan = np.isnan(r)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], r[~nan])


def test_e4m3_decode_all_bytes():
    b = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = b.view(torch.float8_e4m3fn).double().numpy()
    got = np.array([oracle.e4m3_to_f64(i) for i in range(256)])
    nan = np.isnan(ref)
    assert nan.sum() == 2
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


def test_e8m0_decode_all_bytes():
    if not hasattr(torch, "float8_e8m0fnu"):
        pytest.skip("torch without float8_e8m0fnu")
    b = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = b.view(torch.float8_e8m0fnu).double().numpy()
    got = np.array([oracle.e8m0_to_f64(i) for i in range(256)])
    assert math.isnan(got[255]) and math.isnan(ref[255])
    assert np.array_equal(got[:255], ref[:255])


# ---- routing -------------------------------------------------------------------

def test_router_logits_match_numpy_matmul():
    rng = np.random.default_rng(1)
    T, d, E = 9, 96, 24
    x = rand_bf16(rng, (T, d))
    wr = rand_bf16(rng, (E, d), 1 / math.sqrt(d))
    b = rng.standard_normal(E).astype(np.float32)
    got = oracle.router_logits(x, wr, b)
    ref = f64(x) @ f64(wr).T + b.astype(np.float64)
    np.testing.assert_allclose(got, ref, rtol=1e-13, atol=1e-13)
    got0 = oracle.router_logits(x, wr, None)
    np.testing.assert_allclose(got0, f64(x) @ f64(wr).T, rtol=1e-13, atol=1e-13)


@pytest.mark.parametrize("k", [1, 2, 5, 8, 16])
def test_topk_matches_brute_force_sort(k):
    rng = np.random.default_rng(k)
    T, E = 200, 16
    # small integers force many exact ties
    lg = rng.integers(-3, 4, size=(T, E)).astype(np.float64)
    lg[::3] += rng.standard_normal((len(lg[::3]), E))
    got = oracle.select_topk(lg, k)
    for t in range(T):
        ref = sorted(range(E), key=lambda e: (-lg[t, e], e))[:k]
        assert list(got[t]) == ref


def test_gates_equal_softmax_over_all_then_renormalised():
    rng = np.random.default_rng(2)
    T, E, k = 50, 64, 8
    lg = rng.standard_normal((T, E)) * 3
    ids = oracle.select_topk(lg, k)
    got = oracle.gate_weights(lg, ids)
    p = scipy.special.softmax(lg, axis=1)
    chosen = np.take_along_axis(p, ids.astype(np.int64), axis=1)
    ref = chosen / chosen.sum(axis=1, keepdims=True)
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=0)
    # replayed (arbitrary, unordered) ids: same renormalised softmax
    rids = np.stack([rng.choice(E, k, replace=False) for _ in range(T)]).astype(np.int32)
    got_r = oracle.gate_weights(lg, rids)
    ch = np.take_along_axis(p, rids.astype(np.int64), axis=1)
    np.testing.assert_allclose(got_r, ch / ch.sum(axis=1, keepdims=True), rtol=1e-12)


def test_gates_closed_forms():
    lg = np.array([[math.log(3.0), 0.0, -50.0]])
    g = oracle.gate_weights(lg, np.array([[0, 1]], np.int32))
    np.testing.assert_allclose(g[0], [0.75, 0.25], rtol=1e-15)
    # all-equal logits -> exactly 1/k
    lg = np.full((3, 16), 0.37)
    ids = oracle.select_topk(lg, 8)
    assert (ids == np.arange(8)).all()
    assert (oracle.gate_weights(lg, ids) == 1 / 8).all()
    # own mode: non-increasing in slot order, sum to one
    rng = np.random.default_rng(3)
    lg = rng.standard_normal((100, 40))
    ids = oracle.select_topk(lg, 8)
    g = oracle.gate_weights(lg, ids)
    assert (np.diff(g, axis=1) <= 0).all()
    np.testing.assert_allclose(g.sum(1), 1.0, rtol=1e-15)


def test_check_ids():
    ids = np.array([[0, 1], [1, 1], [3, 0], [-1, 2], [2, 4]], np.int32)
    assert list(oracle.check_ids(ids, 4)) == [1, 0, 1, 0, 0]


# ---- dispatch -------------------------------------------------------------------

@pytest.mark.parametrize("E,T,k", [(16, 1000, 8), (384, 64, 8), (7, 1, 3), (5, 0, 2)])
def test_counting_sort_is_stable_argsort(E, T, k):
    rng = np.random.default_rng(E + T)
    ids = rng.integers(0, E, size=(T, k)).astype(np.int32)
    cnt, off, perm, inv = oracle.counting_sort(ids, E)
    flat = ids.reshape(-1)
    assert np.array_equal(cnt, np.bincount(flat, minlength=E))
    assert off[0] == 0 and np.array_equal(np.diff(off), cnt) and off[-1] == T * k
    assert np.array_equal(perm, np.argsort(flat, kind="stable"))
    assert np.array_equal(inv[perm], np.arange(T * k))


# ---- expert FFN ------------------------------------------------------------------

def _expert(rng, d, F, std=0.1):
    return Expert(Matrix(rand_bf16(rng, (F, d), std)), Matrix(rand_bf16(rng, (F, d), std)),
                  Matrix(rand_bf16(rng, (d, F), std)))


def test_expert_ffn_matches_torch_swiglu_fp64():
    # E = 1, k = 1 reduces the layer to one dense SwiGLU FFN.
    rng = np.random.default_rng(4)
    n, d, F = 5, 64, 32
    x = rand_bf16(rng, (n, d))
    ex = _expert(rng, d, F, 0.3)
    got = oracle.expert_ffn(x, ex)
    X = torch.from_numpy(f64(x))
    Wg, Wu, Wd = (torch.from_numpy(f64(m.values)) for m in (ex.w_gate, ex.w_up, ex.w_down))
    ref = (torch.nn.functional.silu(X @ Wg.T) * (X @ Wu.T)) @ Wd.T
    np.testing.assert_allclose(got, ref.numpy(), rtol=1e-12, atol=1e-12)


def test_expert_ffn_closed_forms():
    d, F = 6, 2
    x = np.zeros((1, d), np.float32)
    x[0, 2] = 1.0
    wg = np.zeros((F, d), np.float32)
    wu = np.zeros((F, d), np.float32)
    wd = np.zeros((d, F), np.float32)
    wg[0, 2], wu[0, 2] = 64.0, 0.5       # silu(64) = 64 exactly in fp64, h0 = 32
    wg[1, 2], wu[1, 2] = -64.0, 1.0      # silu(-64) = -64/(1+e^64), h1 ~ -1e-26
    wd[:, 0] = [1, 2, 3, -4, 0.5, 0]
    wd[:, 1] = [1e3, 1e3, 1e3, 1e3, 1e3, 1e3]
    ex = Expert(Matrix(bf16(wg)), Matrix(bf16(wu)), Matrix(bf16(wd)))
    y = oracle.expert_ffn(bf16(x), ex)[0]
    h1 = -64.0 / (1.0 + math.exp(64.0))
    ref = 32.0 * np.array([1, 2, 3, -4, 0.5, 0]) + h1 * 1e3
    np.testing.assert_allclose(y, ref, rtol=1e-15, atol=1e-30)
    # zero pre-activation gives zero output whatever the up projection
    x0 = np.zeros((1, d), np.float32)
    assert (oracle.expert_ffn(bf16(x0), ex) == 0).all()


# ---- the layer ---------------------------------------------------------------------

def _layer(rng, T=24, d=64, E=16, F=32, shared=True, bias=True):
    x = rand_bf16(rng, (T, d))
    wr = rand_bf16(rng, (E, d), 1 / math.sqrt(d))
    b = (rng.standard_normal(E) * 0.3).astype(np.float32) if bias else None
    ex = [_expert(rng, d, F) for _ in range(E)]
    sh = [_expert(rng, d, F)] if shared else []
    return x, wr, b, ex, sh


def test_golden_hand_worked_layer():
    with open(os.path.join(GOLDEN, "hand_worked_layer.json")) as f:
        g = json.load(f)
    x = bf16([g["x"]])
    wr = bf16(g["w_router"])
    ex = [Expert(Matrix(bf16(e["w_gate"])), Matrix(bf16(e["w_up"])), Matrix(bf16(e["w_down"])))
          for e in g["experts"]]
    tol = g["tolerance"]
    own = oracle.layer_forward(x, wr, None, lambda e: ex[e], [], g["k"])
    assert list(own.ids[0]) == g["own"]["ids"]
    np.testing.assert_allclose(own.gates[0], g["own"]["gates"], rtol=tol["rel"])
    np.testing.assert_allclose(own.out[0], g["own"]["out"], rtol=tol["rel"], atol=tol["abs"])
    rep = oracle.layer_forward(x, wr, None, lambda e: ex[e], [], g["k"],
                               replay_ids=np.array([g["replay"]["ids"]], np.int32))
    assert list(rep.ids[0]) == g["replay"]["ids"]
    np.testing.assert_allclose(rep.gates[0], g["replay"]["gates"], rtol=tol["rel"])
    np.testing.assert_allclose(rep.out[0], g["replay"]["out"], rtol=tol["rel"], atol=tol["abs"])


def test_replaying_own_ids_reproduces_own_output_exactly():
    rng = np.random.default_rng(5)
    x, wr, b, ex, sh = _layer(rng)
    own = oracle.layer_forward(x, wr, b, lambda e: ex[e], sh, 8)
    rep = oracle.layer_forward(x, wr, b, lambda e: ex[e], sh, 8, replay_ids=own.ids)
    assert np.array_equal(own.out, rep.out) and np.array_equal(own.gates, rep.gates)


def test_identical_experts_give_expert_output_plus_shared():
    rng = np.random.default_rng(6)
    x, wr, b, ex, sh = _layer(rng)
    same = ex[0]
    res = oracle.layer_forward(x, wr, b, lambda e: same, sh, 8)
    ref = oracle.expert_ffn(x, same) + oracle.expert_ffn(x, sh[0])
    np.testing.assert_allclose(res.out, ref, rtol=1e-13, atol=1e-13)


def test_k_equals_E_is_the_dense_softmax_mixture():
    rng = np.random.default_rng(7)
    x, wr, b, ex, _ = _layer(rng, T=6, E=8, shared=False)
    res = oracle.layer_forward(x, wr, b, lambda e: ex[e], [], 8)
    lg = f64(x) @ f64(wr).T + b
    p = scipy.special.softmax(lg, axis=1)
    ys = np.stack([oracle.expert_ffn(x, ex[e]) for e in range(8)], axis=1)  # [T][E][d]
    ref = np.einsum("te,ted->td", p, ys)
    np.testing.assert_allclose(res.out, ref, rtol=1e-12, atol=1e-12)


def test_scaling_w_down_by_two_doubles_output_exactly():
    rng = np.random.default_rng(8)
    x, wr, b, ex, sh = _layer(rng)
    a = oracle.layer_forward(x, wr, b, lambda e: ex[e], sh, 8)

    def dbl(m):
        return Expert(m.w_gate, m.w_up, Matrix(bf16(f64(m.w_down.values) * 2)))
    ex2 = [dbl(m) for m in ex]
    b2 = oracle.layer_forward(x, wr, b, lambda e: ex2[e], [dbl(sh[0])], 8)
    assert np.array_equal(b2.out, 2 * a.out)


def test_invalid_replay_tokens_get_zero_rows():
    rng = np.random.default_rng(9)
    x, wr, b, ex, sh = _layer(rng, T=4)
    ids = np.array([[0, 1, 2, 3, 4, 5, 6, 7], [0, 0, 2, 3, 4, 5, 6, 7],
                    [15, 14, 13, 12, 11, 10, 9, 8], [0, 1, 2, 3, 4, 5, 6, 16]], np.int32)
    res = oracle.layer_forward(x, wr, b, lambda e: ex[e], sh, 8, replay_ids=ids)
    assert list(res.valid) == [1, 0, 1, 0]
    assert (res.out[[1, 3]] == 0).all() and (res.gates[[1, 3]] == 0).all()
    assert (res.ids[1] == np.arange(8)).all()
    assert (res.out[[0, 2]] != 0).any()


def test_tokens_are_independent():
    # The definition is per token: any split of the batch gives the same rows.
    rng = np.random.default_rng(10)
    x, wr, b, ex, sh = _layer(rng, T=10)
    full = oracle.layer_forward(x, wr, b, lambda e: ex[e], sh, 8)
    part = oracle.layer_forward(x[3:7], wr, b, lambda e: ex[e], sh, 8)
    assert np.array_equal(full.out[3:7], part.out)
    assert np.array_equal(full.ids[3:7], part.ids)


# ---- MXFP8 weights ---------------------------------------------------------------------

def test_mxfp8_weight_decode_matches_torch_and_bounds():
    from deterministic_rl_gb300.synthetic import quantize_mxfp8
    g = torch.Generator().manual_seed(0)
    w = torch.randn((8, 128), generator=g) * 0.02
    q, s = quantize_mxfp8(w)
    m = Matrix(q.numpy(), s.numpy())
    deq = np.array([[m.elem(r, c) for c in range(128)] for r in range(8)])
    ref = (q.view(torch.float8_e4m3fn).double()
           * torch.pow(2.0, s.double() - 127).repeat_interleave(32, dim=1)).numpy()
    assert np.array_equal(deq, ref)
    # E4M3 round-to-nearest: relative error <= 2^-4 for normal-range values
    wd = w.double().numpy()
    scale = np.repeat(np.exp2(s.numpy().astype(np.float64) - 127), 32, axis=1)
    sat = np.abs(wd) / scale > 448          # the MX shared exponent lets the block
    assert (np.abs(deq[sat]) == 448 * scale[sat]).all()   # max exceed 448: it saturates
    big = (np.abs(deq) >= scale * 2.0 ** -6) & ~sat
    rel = np.abs(deq - wd)[big] / np.abs(wd)[big]
    assert rel.max() <= 2.0 ** -4 / (1 - 2.0 ** -4)
    # the largest magnitude of each block lands in [256, 448] before scaling
    blk = np.abs(q.view(torch.float8_e4m3fn).double().numpy()).reshape(8, 4, 32).max(-1)
    assert ((blk >= 256) & (blk <= 448)).all()


def test_mxfp8_layer_equals_bf16_layer_on_dequantised_weights():
    # Dequantised MXFP8 values are exact in bf16, so the layer on MXFP8 weights
    # equals the layer on their bf16 dequantisation.
    from deterministic_rl_gb300.synthetic import quantize_mxfp8
    rng = np.random.default_rng(11)
    d, F, E, T = 64, 64, 8, 5
    x = rand_bf16(rng, (T, d))
    wr = rand_bf16(rng, (E, d), 1 / math.sqrt(d))
    exq, exb = [], []
    for _ in range(E):
        mats_q, mats_b = [], []
        for shape in ((F, d), (F, d), (d, F)):
            q, s = quantize_mxfp8(torch.from_numpy(rng.standard_normal(shape).astype(np.float32) * 0.02))
            deq = (q.view(torch.float8_e4m3fn).float()
                   * torch.pow(2.0, s.float() - 127).repeat_interleave(32, dim=1))
            assert torch.equal(deq.to(torch.bfloat16).float(), deq)
            mats_q.append(Matrix(q.numpy(), s.numpy()))
            mats_b.append(Matrix(bf16(deq.numpy())))
        exq.append(Expert(*mats_q))
        exb.append(Expert(*mats_b))
    a = oracle.layer_forward(x, wr, None, lambda e: exq[e], [], 8)
    b = oracle.layer_forward(x, wr, None, lambda e: exb[e], [], 8)
    assert np.array_equal(a.out, b.out)


# ---- replay plausibility filter ------------------------------------------------

def test_replay_filter_hand_worked_cases():
    with open(os.path.join(GOLDEN, "replay_filter_cases.json")) as f:
        g = json.load(f)
    lg = np.array([g["logits"]], np.float64)
    for c in g["cases"]:
        out, rep = oracle.filter_replay(lg, np.array([c["replay"]], np.int32), c["tau"])
        assert list(out[0]) == c["expect"], c
        assert int(rep[0]) == c["replaced"], c


def test_replay_filter_properties():
    rng = np.random.default_rng(12)
    T, E, k = 400, 24, 8
    lg = rng.standard_normal((T, E))
    own = oracle.select_topk(lg, k)
    rids = np.stack([rng.choice(E, k, replace=False) for _ in range(T)]).astype(np.int32)
    # tau = 0 keeps everything; replaying the router's own choice is never filtered
    out0, rep0 = oracle.filter_replay(lg, rids, 0.0)
    assert np.array_equal(out0, rids) and (rep0 == 0).all()
    for tau in (0.1, 0.5, 1.0):
        o, r = oracle.filter_replay(lg, own, tau)
        assert np.array_equal(o, own) and (r == 0).all()
    prev = np.zeros(T, np.int32)
    for tau in (0.01, 0.1, 0.3, 0.7, 1.0):
        out, rep = oracle.filter_replay(lg, rids, tau)
        assert (rep >= prev).all()            # a higher threshold drops more
        prev = rep
        kth = np.take_along_axis(lg, own[:, -1:].astype(np.int64), 1)[:, 0]
        for t in range(T):
            assert len(set(out[t].tolist())) == k
            for s in range(k):
                if out[t, s] == rids[t, s]:
                    assert lg[t, rids[t, s]] >= kth[t] + math.log(tau) - 1e-12
                else:                          # replaced by an own candidate
                    assert lg[t, rids[t, s]] < kth[t] + math.log(tau)
                    assert out[t, s] in set(own[t].tolist())
    # tau = 1 with replayed experts all outside the own top-k: the own top-k set
    far = np.argsort(-lg, axis=1, kind="stable")[:, k:2 * k].astype(np.int32)
    out, rep = oracle.filter_replay(lg, far, 1.0)
    assert (rep == k).all()
    assert np.array_equal(out, own)


# ---- NVFP4 with per-token scales ----------------------------------------------
# The format of the Composer 2 Technical Report, section 6.1 (Kernels): FP4 E2M1
# values, an FP8 E4M3 scale per 16 values, an FP32 scale per token, IEEE
# division in the quantiser.

E2M1_MAGNITUDES = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]  # the published E2M1 value set


def test_e2m1_decode_is_the_published_value_set():
    got = [oracle.e2m1_to_f64(c) for c in range(16)]
    assert got[:8] == E2M1_MAGNITUDES
    assert got[8:] == [-m for m in E2M1_MAGNITUDES]


@pytest.mark.parametrize("v,code", [
    (0.0, 0), (0.25, 0), (0.2500001, 1), (0.5, 1), (0.75, 2), (1.25, 2), (1.5, 3),
    (1.75, 4), (2.5, 4), (2.51, 5), (3.5, 6), (5.0, 6), (5.0001, 7), (6.0, 7), (1e30, 7),
    (-0.2, 0), (-0.3, 9), (-0.75, 10), (-3.5, 14), (-100.0, 15)])
def test_e2m1_rounding_ties_to_even_and_saturates(v, code):
    assert oracle.e2m1_round(v) == code


def test_e4m3_rounding_matches_torch_float8_conversion():
    rng = np.random.default_rng(0)
    # random values over the whole range, every representable value, and the
    # exact midpoints between neighbours (ties)
    grid = np.array([oracle.e4m3_to_f64(b) for b in range(0x7F)], np.float64)
    mids = (grid[1:] + grid[:-1]) / 2
    v = np.concatenate([rng.uniform(0, 463.9, 4000), np.exp(rng.uniform(-12, 6, 4000)), grid, mids])
    v = v[v < 464].astype(np.float32)   # torch turns 464 and above into NaN
    ref = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([oracle.e4m3_round(x) for x in v], np.uint8)
    assert np.array_equal(got, ref)
    # the quantiser's scales saturate at the largest finite value, 448
    for x in (464.0, 500.0, 1e30):
        assert oracle.e4m3_round(x) == 0x7E


def test_round_bf16_matches_torch_on_fp32_inputs():
    rng = np.random.default_rng(1)
    v = np.concatenate([rng.standard_normal(3000) * 10.0 ** rng.integers(-30, 30, 3000),
                        np.ldexp(1.0 + rng.integers(0, 256, 500) / 256 + 1 / 512, 3)])
    v = v.astype(np.float32)
    ref = torch.from_numpy(v).to(torch.bfloat16).double().numpy()
    got = np.array([oracle.round_bf16(float(x)) for x in v])
    assert np.array_equal(got, ref)


def test_nvfp4_golden_hand_worked_rows():
    with open(os.path.join(GOLDEN, "nvfp4_rows.json")) as f:
        g = json.load(f)
    for case in g["cases"]:
        row = np.array(case["row"], np.float32)[None]
        codes, bs, rs = oracle.nvfp4_quantize_rows(row)
        assert float(rs[0]) == case["row_scale"], case["name"]
        assert bs[0].tolist() == case["block_scales"], case["name"]
        assert codes[0].tolist() == case["codes"], case["name"]


def _dequant(codes, bs, rs):
    tab = np.array([oracle.e2m1_to_f64(c) for c in range(16)])
    sc = np.array([oracle.e4m3_to_f64(b) for b in range(256)])
    return tab[codes] * np.repeat(sc[bs], 16, axis=1) * rs.astype(np.float64)[:, None]


def test_nvfp4_quantiser_properties():
    rng = np.random.default_rng(2)
    R, K = 64, 256
    mag = 10.0 ** rng.uniform(-6, 3, (R, 1))
    x = f64(rand_bf16(rng, (R, K))) * mag
    x = f64(bf16(x)).astype(np.float32)
    x[5, 16:32] = 0.0                        # an all-zero block
    codes, bs, rs = oracle.nvfp4_quantize_rows(x)
    xq = _dequant(codes, bs, rs)
    denom = np.repeat(np.array([[oracle.e4m3_to_f64(b) for b in r] for r in bs]), 16, 1) * rs[:, None]
    # where the block scale is a normal E4M3 value, every value is within half
    # an E2M1 step (at most 1 unit of its block's scale, the step between 4 and
    # 6 being 2) of its input, up to the fp32 rounding of the quotient the
    # code is decided on; a block's largest value overshoots 6 units by at
    # most the scale's rounding, 1/16
    normal_el = np.repeat(bs >= 8, 16, axis=1)
    assert np.all((np.abs(xq - x) <= (1.0 + 1e-6) * denom)[normal_el])
    assert normal_el.mean() > 0.9
    # a block's largest magnitude becomes +-6 (E4M3 rounding of the block scale
    # moves it by at most 1/16 relative, which stays nearest to 6)
    blocks = np.abs(x).reshape(R, K // 16, 16)
    arg = blocks.argmax(-1)
    top = np.take_along_axis(codes.reshape(R, K // 16, 16), arg[..., None], -1)[..., 0]
    normal = (bs >= 8) & (bs < 0x7E)
    assert np.all((top[normal] & 7) == 7)
    # the zero block has scale 0 and codes 0
    assert bs[5, 1] == 0 and not codes[5, 16:32].any()
    # rows are independent: a row quantised alone gives the same bytes
    c1, b1, r1 = oracle.nvfp4_quantize_rows(x[7:8])
    assert np.array_equal(c1[0], codes[7]) and np.array_equal(b1[0], bs[7]) and r1[0] == rs[7]
    # scaling a row by a power of two scales only the row scale (exactly)
    c2, b2, r2 = oracle.nvfp4_quantize_rows(np.ldexp(x, -3))
    assert np.array_equal(c2, codes) and np.array_equal(b2, bs)
    assert np.array_equal(r2, np.ldexp(rs, -3))


def _nvfp4_matrix(w):
    from deterministic_rl_gb300.synthetic import quantize_nvfp4
    q, s, ts = quantize_nvfp4(torch.from_numpy(w.astype(np.float32)))
    return Matrix(q.numpy(), s.numpy(), float(ts))


def test_nvfp4_weight_decode_is_code_times_scales():
    rng = np.random.default_rng(3)
    m = _nvfp4_matrix(rng.standard_normal((8, 64)) * 0.02)
    K = 64
    for r, c in [(0, 0), (1, 1), (3, 17), (7, 63)]:
        byte = m.values[r, c // 2]
        code = (byte >> 4) if c & 1 else (byte & 15)
        want = E2M1_MAGNITUDES[code & 7] * (-1 if code & 8 else 1) * \
            float(torch.tensor([m.scales[r, c // 16]], dtype=torch.uint8).view(torch.float8_e4m3fn).double()) * \
            float(np.float32(m.tscale))
        assert m.elem(r, c) == want
    assert m.K == K


def test_nvfp4_expert_ffn_matches_torch_fp64_pipeline():
    """The NVFP4 expert FFN: quantise the token rows (pinned above), the GEMMs
    and SwiGLU in torch float64 on the quantised values, round h to bf16
    (pinned above), quantise h, the down GEMM in torch float64."""
    rng = np.random.default_rng(4)
    n, d, F = 5, 64, 48
    wg, wu, wd = (_nvfp4_matrix(rng.standard_normal(s) * 0.05) for s in ((F, d), (F, d), (d, F)))
    ex = Expert(wg, wu, wd)
    xb = rand_bf16(rng, (n, d))
    got = oracle.expert_ffn(xb, ex)

    def dense(m, rows, K):
        return torch.tensor([[m.elem(r, c) for c in range(K)] for r in range(rows)], dtype=torch.float64)

    G, U, D = dense(wg, F, d), dense(wu, F, d), dense(wd, d, F)
    xq = torch.from_numpy(_dequant(*oracle.nvfp4_quantize_rows(f64(xb).astype(np.float32))))
    g = xq @ G.T
    u = xq @ U.T
    h = torch.nn.functional.silu(g) * u
    hb = np.array([[oracle.round_bf16(float(v)) for v in row] for row in h.numpy()], np.float32)
    hq = torch.from_numpy(_dequant(*oracle.nvfp4_quantize_rows(hb)))
    want = (hq @ D.T).numpy()
    np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-15)
