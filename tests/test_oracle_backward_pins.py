"""Pins of the backward oracle (oracle/backward.py) to things other than itself:
hand-worked MXFP8 blocks, torch's float8_e4m3fn conversion and the C oracle's
pinned E4M3 rounding, closed forms of the block exponent, a planted outlier
that tells the quantisation axis apart, the C forward oracle (for the numpy
forward the gradients are taken of), and central finite differences of that
forward (for every gradient the backward returns)."""
from __future__ import annotations

import json
import os

import numpy as np
import pytest
import torch

import oracle
from oracle import Expert, Matrix
from oracle import backward as B

HERE = os.path.dirname(os.path.abspath(__file__))


def _bf16_bits(a: np.ndarray) -> np.ndarray:
    return torch.from_numpy(np.ascontiguousarray(a, np.float32)).to(torch.bfloat16).view(
        torch.uint16).numpy()


def _bf16_vals(bits: np.ndarray) -> np.ndarray:
    return torch.from_numpy(bits).view(torch.bfloat16).to(torch.float64).numpy()


# ---- the quantiser -------------------------------------------------------------

def _golden_blocks():
    with open(os.path.join(HERE, "golden", "mxfp8_blocks.json")) as f:
        return json.load(f)["blocks"]


def _expand(d):
    v = np.zeros(32)
    for key, h in d.items():
        if key == "all":
            v[:] = float.fromhex(h)
        else:
            v[int(key)] = float.fromhex(h)
    return v


@pytest.mark.parametrize("i", range(len(_golden_blocks())))
def test_mx_golden_blocks(i):
    b = _golden_blocks()[i]
    v = _expand(b["values"])
    assert int(B.mx_exponent(np.abs(v).max())) == b["X"]
    np.testing.assert_array_equal(B.mx_quantize(v[None, :], 1)[0], _expand(b["dequant"]))
    # reversed block order along the other axis: same values, same result
    np.testing.assert_array_equal(B.mx_quantize(v[:, None], 0)[:, 0], _expand(b["dequant"]))


def test_round_e4m3_matches_torch_float8_and_the_c_oracle():
    rng = np.random.default_rng(11)
    mag = np.ldexp(rng.uniform(1, 2, 20000), rng.integers(-12, 10, 20000))
    v = mag * rng.choice([-1.0, 1.0], 20000)
    # every E4M3 value and every midpoint between neighbours (ties)
    vals = np.array(sorted({oracle.e4m3_to_f64(b) for b in range(256)
                            if np.isfinite(oracle.e4m3_to_f64(b))}))
    mids = (vals[1:] + vals[:-1]) / 2
    v = np.concatenate([v, vals, mids, -mids, [500.0, -1000.0, 464.0, 463.9]])
    ours = B.round_e4m3(v)
    # torch's conversion is nearest-even with NaN above the range: clamp first
    # (448 is representable, so clamping and rounding commute)
    ref = torch.from_numpy(np.clip(v, -448, 448)).to(torch.float32).to(
        torch.float8_e4m3fn).to(torch.float64).numpy()
    np.testing.assert_array_equal(ours, ref)
    # the C oracle's rounding (of scales) takes magnitudes
    sample = np.abs(v[::50])
    c = np.array([oracle.e4m3_to_f64(oracle.e4m3_round(x)) for x in sample])
    np.testing.assert_array_equal(B.round_e4m3(sample), c)


def test_mx_exponent_closed_forms():
    for n in range(-100, 100, 7):
        assert B.mx_exponent(np.ldexp(1.0, n)) == n - 8
        assert B.mx_exponent(np.ldexp(1.999999, n)) == n - 8
        assert B.mx_exponent(np.ldexp(0.999999, n)) == n - 9
    assert B.mx_exponent(0.0) == -127
    assert B.mx_exponent(np.ldexp(1.0, -300)) == -127
    assert B.mx_exponent(np.ldexp(1.0, 200)) == 127


def test_mx_quantize_properties():
    rng = np.random.default_rng(12)
    v = rng.standard_normal((64, 96)) * np.ldexp(1.0, rng.integers(-20, 20, (64, 1)))
    q = B.mx_quantize(v, 1)
    # idempotent: a quantised block quantises to itself
    np.testing.assert_array_equal(B.mx_quantize(q, 1), q)
    # each element is an E4M3 value times its block's power of two
    blocks = v.reshape(64, 3, 32)
    X = B.mx_exponent(np.abs(blocks).max(axis=2))
    el = q.reshape(64, 3, 32) / np.ldexp(1.0, X)[..., None]
    np.testing.assert_array_equal(B.round_e4m3(el), el)
    assert np.abs(el).max() <= 448
    # relative error at most 2^-4 for elements in E4M3's normal range that
    # are not clamped (a block's largest scaled magnitude is in [256, 512))
    sv = blocks / np.ldexp(1.0, X)[..., None]
    normal = (np.abs(sv) >= 2.0 ** -6) & (np.abs(sv) <= 448)
    rel = np.abs(q.reshape(64, 3, 32) - blocks)[normal] / np.abs(blocks)[normal]
    assert rel.max() <= 2.0 ** -4
    # blocks are independent: changing one block leaves the others
    w = v.copy()
    w[:, 32:64] *= 1000.0
    q2 = B.mx_quantize(w, 1)
    np.testing.assert_array_equal(q2[:, :32], q[:, :32])
    np.testing.assert_array_equal(q2[:, 64:], q[:, 64:])
    # a ragged axis is quantised as if padded with zeros
    r = v[:, :80]
    np.testing.assert_array_equal(B.mx_quantize(r, 1),
                                  B.mx_quantize(np.pad(r, ((0, 0), (0, 16))), 1)[:, :80])


def test_qmatmul_quantises_along_the_contraction_axis():
    # Row 0 of a holds 2^20 and 31 halves in its first K-block: scaled by
    # 2^-(20-8) the halves become 2^-13, below half the smallest E4M3
    # subnormal, so they vanish; its second K-block (32 halves) is exact.
    a = np.full((2, 64), 0.5)
    a[0, 0] = 2.0 ** 20
    b = np.ones((1, 64))
    c = B.qmatmul_nt(a, b, quant=True)
    assert c[0, 0] == 2.0 ** 20 + 16.0
    assert c[1, 0] == 32.0          # row 1 has no outlier: exact
    exact = B.qmatmul_nt(a, b, quant=False)
    assert exact[0, 0] == 2.0 ** 20 + 31.5
    # quantising along the other axis would have changed row 1 instead
    wrong = B.mx_quantize(a, 0) @ b.T
    assert wrong[1, 0] == 31.5 and wrong[0, 0] == 2.0 ** 20 + 31.5


def test_bf16_round_matches_torch():
    rng = np.random.default_rng(13)
    v = rng.standard_normal(50000).astype(np.float32).astype(np.float64)
    v = np.concatenate([v, [1 + 2 ** -8, 1 + 3 * 2 ** -8, -(1 + 2 ** -8)]])  # ties
    ref = torch.from_numpy(v).to(torch.float32).to(torch.bfloat16).to(torch.float64).numpy()
    np.testing.assert_array_equal(B.bf16_round(v), ref)


# ---- the layer -----------------------------------------------------------------

def _values_layer(rng, T=6, d=64, E=5, k=2, F=32, S=1, scale=0.3):
    x = rng.standard_normal((T, d))
    wr = rng.standard_normal((E, d)) * scale
    bias = rng.standard_normal(E) * 0.5
    experts = [B.ExpertValues(rng.standard_normal((F, d)) * scale,
                              rng.standard_normal((F, d)) * scale,
                              rng.standard_normal((d, F)) * scale) for _ in range(E)]
    shared = [B.ExpertValues(rng.standard_normal((F, d)) * scale,
                             rng.standard_normal((F, d)) * scale,
                             rng.standard_normal((d, F)) * scale) for _ in range(S)]
    ids = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    dout = rng.standard_normal((T, d))
    return x, wr, bias, experts, shared, ids, dout


def test_numpy_forward_matches_the_c_oracle():
    rng = np.random.default_rng(14)
    T, d, E, k, F = 10, 64, 6, 3, 32
    xb = _bf16_bits(rng.standard_normal((T, d)))
    wrb = _bf16_bits(rng.standard_normal((E, d)) * 0.2)
    bias = (rng.standard_normal(E) * 0.3).astype(np.float32)
    eb = [[_bf16_bits(rng.standard_normal(s) * 0.2) for s in ((F, d), (F, d), (d, F))]
          for _ in range(E)]
    sb = [_bf16_bits(rng.standard_normal(s) * 0.2) for s in ((F, d), (F, d), (d, F))]
    ids = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    ref = oracle.layer_forward(xb, wrb, bias, lambda e: Expert(*[Matrix(m) for m in eb[e]]),
                               [Expert(*[Matrix(m) for m in sb])], k, replay_ids=ids)
    out = B.layer_forward_values(_bf16_vals(xb), _bf16_vals(wrb), bias.astype(np.float64),
                                 [B.ExpertValues(*[_bf16_vals(m) for m in ex]) for ex in eb],
                                 [B.ExpertValues(*[_bf16_vals(m) for m in sb])], ids)
    np.testing.assert_allclose(out, ref.out, rtol=1e-12, atol=1e-12)


def _loss(x, wr, bias, experts, shared, ids, dout):
    return float((B.layer_forward_values(x, wr, bias, experts, shared, ids) * dout).sum())


def _fd_check(f, grad, p, rng, eps=1e-6):
    v = rng.standard_normal(p.shape)
    p0 = p.copy()
    p[...] = p0 + eps * v
    lp = f()
    p[...] = p0 - eps * v
    lm = f()
    p[...] = p0
    fd = (lp - lm) / (2 * eps)
    an = float((grad * v).sum())
    assert abs(fd - an) <= 1e-6 * max(1.0, abs(fd)), (fd, an)


def test_exact_backward_matches_finite_differences():
    rng = np.random.default_rng(15)
    x, wr, bias, experts, shared, ids, dout = _values_layer(rng)
    r = B.layer_backward(x, wr, bias, lambda e: experts[e], shared, ids, dout,
                         quant=False, round_storage=False)
    f = lambda: _loss(x, wr, bias, experts, shared, ids, dout)  # noqa: E731
    _fd_check(f, r.dx, x, rng)
    _fd_check(f, r.d_router, wr, rng)
    used = sorted(set(ids.reshape(-1).tolist()))
    for e in used:
        _fd_check(f, r.experts[e].d_gate, experts[e].w_gate, rng)
        _fd_check(f, r.experts[e].d_up, experts[e].w_up, rng)
        _fd_check(f, r.experts[e].d_down, experts[e].w_down, rng)
    _fd_check(f, r.shared[0].d_gate, shared[0].w_gate, rng)
    _fd_check(f, r.shared[0].d_up, shared[0].w_up, rng)
    _fd_check(f, r.shared[0].d_down, shared[0].w_down, rng)
    # the gate gradient: d/dw_s of sum(dout * out) = dout . y_s
    for t in range(2):
        for s in range(ids.shape[1]):
            ex = experts[ids[t, s]]
            h = B.silu(x[t] @ ex.w_gate.T) * (x[t] @ ex.w_up.T)
            assert np.isclose(r.dgates[t, s], dout[t] @ (ex.w_down @ h), rtol=1e-12)


def test_quantised_backward_is_close_to_exact_and_not_equal():
    rng = np.random.default_rng(16)
    x, wr, bias, experts, shared, ids, dout = _values_layer(rng, T=40, d=96, E=4, F=64)
    get = lambda e: experts[e]  # noqa: E731
    ex = B.layer_backward(x, wr, bias, get, shared, ids, dout, quant=False, round_storage=False)
    q = B.layer_backward(x, wr, bias, get, shared, ids, dout)
    pairs = [(q.dx, ex.dx), (q.d_router, ex.d_router),
             (q.shared[0].d_gate, ex.shared[0].d_gate), (q.shared[0].d_down, ex.shared[0].d_down)]
    pairs += [(q.experts[e].d_up, ex.experts[e].d_up) for e in q.experts]
    for a, b in pairs:
        rel = np.linalg.norm(a - b) / np.linalg.norm(b)
        # MXFP8 operands carry at most 2^-4 relative error each
        assert 1e-5 < rel < 0.1, rel


def test_limits_only_skip_work():
    rng = np.random.default_rng(17)
    x, wr, bias, experts, shared, ids, dout = _values_layer(rng, T=30, d=64, E=6, k=2, F=32)
    get = lambda e: experts[e]  # noqa: E731
    full = B.layer_backward(x, wr, bias, get, shared, ids, dout)
    toks = [3, 17, 29]
    part = B.layer_backward(x, wr, bias, get, shared, ids, dout, tokens=toks,
                            grad_experts=[int(ids[5, 0])], grad_shared=False)
    np.testing.assert_array_equal(part.dx[toks], full.dx[toks])
    np.testing.assert_array_equal(part.dlogits[toks], full.dlogits[toks])
    e = int(ids[5, 0])
    for name in ("d_gate", "d_up", "d_down"):
        np.testing.assert_array_equal(getattr(part.experts[e], name),
                                      getattr(full.experts[e], name))
    assert set(part.experts) == {e}
    # a router row is complete when all of its expert's tokens are formed
    e2 = int(ids[0, 1])
    toks2 = sorted(set((np.nonzero((ids == e2).any(axis=1))[0]).tolist()))
    part2 = B.layer_backward(x, wr, bias, get, shared, ids, dout, tokens=toks2, grad_experts=[],
                             grad_shared=False)
    np.testing.assert_allclose(part2.d_router[e2], full.d_router[e2], rtol=1e-13, atol=1e-13)


def test_invalid_tokens_contribute_nothing():
    rng = np.random.default_rng(18)
    x, wr, bias, experts, shared, ids, dout = _values_layer(rng, T=20, d=64, E=5, k=2, F=32)
    get = lambda e: experts[e]  # noqa: E731
    valid = np.ones(20, np.uint8)
    valid[[2, 9]] = 0
    a = B.layer_backward(x, wr, bias, get, shared, ids, dout, valid=valid)
    d0 = dout.copy()
    d0[[2, 9]] = 0.0
    b = B.layer_backward(x, wr, bias, get, shared, ids, d0)
    np.testing.assert_array_equal(a.dx, b.dx)
    np.testing.assert_array_equal(a.d_router, b.d_router)
    assert not a.dx[[2, 9]].any()
    for e in a.experts:
        np.testing.assert_array_equal(a.experts[e].d_down, b.experts[e].d_down)


# ---- the C oracle's MXFP8 row quantiser (MXFP8 activations in the forward) -------

def test_c_mx_quantiser_equals_the_numpy_one_and_the_golden_blocks():
    rng = np.random.default_rng(19)
    x = rng.standard_normal((64, 256)) * np.ldexp(1.0, rng.integers(-30, 30, (64, 1)))
    x = _bf16_vals(_bf16_bits(x))                      # bf16 values, as the layer has
    np.testing.assert_array_equal(oracle.mx_qdq_rows(x), B.mx_quantize(x, 1))
    for b in _golden_blocks():
        v = _expand(b["values"])
        np.testing.assert_array_equal(oracle.mx_qdq_rows(v[None, :])[0], _expand(b["dequant"]))


def test_mxfp8_activation_expert_ffn_is_the_quantised_pipeline():
    """The expert FFN with MXFP8 activations equals, on the decoded MXFP8
    weights, x quantised along d -> SwiGLU in fp64 -> h rounded to bf16 and
    quantised along F -> down projection (each step a pinned function)."""
    import torch as _t
    from deterministic_rl_gb300.synthetic import quantize_mxfp8
    rng = np.random.default_rng(20)
    n, d, F = 5, 64, 96
    x = _bf16_bits(rng.standard_normal((n, d)))
    mats = []
    for shape in ((F, d), (F, d), (d, F)):
        q, sc = quantize_mxfp8(_t.from_numpy(rng.standard_normal(shape).astype(np.float32) * 0.3))
        mats.append((q.numpy(), sc.numpy()))
    ex = Expert(*[Matrix(q, sc, act_mx=True) for q, sc in mats])
    y = oracle.expert_ffn(x, ex)

    def dec(q, sc):
        vals = np.array([oracle.e4m3_to_f64(b) for b in range(256)])[q.astype(np.int64)]
        return vals * np.repeat(np.ldexp(1.0, sc.astype(np.int64) - 127), 32, axis=1)
    wg, wu, wd = (dec(q, sc) for q, sc in mats)
    xq = B.mx_quantize(_bf16_vals(x), 1)
    h = B.silu(xq @ wg.T) * (xq @ wu.T)
    hq = B.mx_quantize(B.bf16_round(h), 1)
    np.testing.assert_allclose(y, hq @ wd.T, rtol=1e-12, atol=1e-12)
    # and it differs from the bf16-activation FFN on the same weights
    y_plain = oracle.expert_ffn(x, Expert(*[Matrix(q, sc) for q, sc in mats]))
    assert not np.allclose(y, y_plain, rtol=1e-6, atol=0)
