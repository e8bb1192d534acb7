"""Shared helpers of the GPU tests: feeding device-resident layer inputs to the
fp64 oracle (one expert at a time), and the comparison rules.

Comparison rules (fp32 arithmetic on the GPU against the exact oracle):
  * ids: the set must equal the oracle's wherever the oracle's fp64 gap between
    the 8th and 9th logit exceeds 1e-3; the slot order must match too where
    every adjacent gap among the top 8 exceeds 1e-4.  Elsewhere the GPU's set
    must be a valid top-8 within 1e-3 of the oracle's logits.
  * logits: |l_gpu - l_oracle| <= 1e-5 * max(1, max|l|).
  * gates: |w_gpu - w_oracle| <= 1e-6 + (2e-5 + 1e-6) * w_oracle (softmax of
    logits that are each within 1e-5).
  * output (the fp32 combine result): relative Frobenius error <= 5e-3 and
    max-abs error <= 3e-2; the bf16 output equals the fp32 result rounded to
    nearest even.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
from oracle import Expert, Matrix
from deterministic_rl_gb300.synthetic import bf16_bits, u8

# fp32 logit error bound: d <= 16384 bf16 products of magnitude ~ |x||w| summed
# in fp32 stay within 1e-5 of the exact value for logits of order 1.
LOGIT_ERR = 1e-5
ID_SET_MARGIN = 1e-3
ID_ORDER_MARGIN = 1e-4
REL_FRO = 5e-3
MAX_ABS = 3e-2


def _mat(w: torch.Tensor, s, gs=None, act_mx=False) -> Matrix:
    if w.dtype == torch.bfloat16:
        return Matrix(bf16_bits(w))
    if gs is not None:  # NVFP4: packed E2M1, E4M3 scales per 16, fp32 matrix scale
        return Matrix(u8(w), u8(s), float(gs))
    return Matrix(u8(w), u8(s), act_mx=act_mx)


def expert_getter(inp):
    def get(e: int) -> Expert:
        sg = inp.s_gate[e] if inp.s_gate is not None else None
        su = inp.s_up[e] if inp.s_up is not None else None
        sd = inp.s_down[e] if inp.s_down is not None else None
        nv = inp.gs_gate is not None
        am = inp.cfg.act_mx
        return Expert(_mat(inp.w_gate[e], sg, inp.gs_gate[e] if nv else None, am),
                      _mat(inp.w_up[e], su, inp.gs_up[e] if nv else None, am),
                      _mat(inp.w_down[e], sd, inp.gs_down[e] if nv else None, am))
    return get


def shared_experts(inp):
    if inp.ws_gate is None:
        return []
    return [Expert(Matrix(bf16_bits(inp.ws_gate)), Matrix(bf16_bits(inp.ws_up)),
                   Matrix(bf16_bits(inp.ws_down)))]


def router_host(inp):
    bias = None if inp.router_bias is None else inp.router_bias.detach().cpu().numpy()
    return bf16_bits(inp.w_router), bias


def oracle_layer(inp, tokens=None, replay_ids=None, x=None):
    """Oracle layer output for the given token indices (default: all)."""
    xt = inp.x if x is None else x
    if tokens is not None:
        xt = xt[torch.as_tensor(tokens, device=xt.device)]
    wr, bias = router_host(inp)
    return oracle.layer_forward(bf16_bits(xt), wr, bias, expert_getter(inp), shared_experts(inp),
                                inp.cfg.k, replay_ids=replay_ids)


def oracle_replay_ids(inp, tokens=None):
    """Recorded ids: the oracle's own routing of the perturbed hidden states."""
    xs = inp.x_replay_src
    if tokens is not None:
        xs = xs[torch.as_tensor(tokens, device=xs.device)]
    wr, bias = router_host(inp)
    lg = oracle.router_logits(bf16_bits(xs), wr, bias)
    return oracle.select_topk(lg, inp.cfg.k)


def check_ids(gpu_ids: np.ndarray, logits: np.ndarray, k: int):
    """Apply the id rules; returns the mask of tokens whose GPU ids equal the
    oracle's own selection exactly (set and order)."""
    T, E = logits.shape
    order = np.argsort(-logits, axis=1, kind="stable")
    srt = np.take_along_axis(logits, order, axis=1)
    gap8 = srt[:, k - 1] - srt[:, k]
    gaps = srt[:, :k - 1] - srt[:, 1:k]
    ref = oracle.select_topk(logits, k)
    same = np.all(gpu_ids == ref, axis=1)
    for t in range(T):
        g = gpu_ids[t]
        assert len(set(g.tolist())) == k and g.min() >= 0 and g.max() < E, (t, g)
        if gap8[t] > ID_SET_MARGIN:
            assert set(g.tolist()) == set(ref[t].tolist()), (t, g, ref[t], gap8[t])
            if gaps[t].min() > ID_ORDER_MARGIN:
                assert (g == ref[t]).all(), (t, g, ref[t])
        else:
            chosen = logits[t, g]
            others = np.delete(logits[t], g)
            assert chosen.min() >= others.max() - ID_SET_MARGIN, (t, g)
            # within the chosen set, slots stay in descending order up to fp32 error
            assert (np.diff(chosen) <= ID_ORDER_MARGIN).all(), (t, chosen)
    return same


def check_logits(gpu_logits: np.ndarray, ref_logits: np.ndarray):
    """fp32 router logits (bf16 products, fp32 accumulation over d) against fp64."""
    err = np.abs(gpu_logits.astype(np.float64) - ref_logits)
    scale = max(1.0, float(np.abs(ref_logits).max()))
    assert err.max() <= LOGIT_ERR * scale, float(err.max())
    return float(err.max())


def check_gates(gpu_gates: np.ndarray, ref_gates: np.ndarray):
    """A gate weight is a softmax of k logits, so a logit error of at most
    LOGIT_ERR moves it by at most 2 * LOGIT_ERR * w; fp32 exp and division add
    a few ulp (< 1e-6 * w), and 1e-6 absolute covers the tiny weights."""
    err = np.abs(gpu_gates.astype(np.float64) - ref_gates)
    bound = 1e-6 + (2 * LOGIT_ERR + 1e-6) * np.abs(ref_gates)
    assert (err <= bound).all(), float((err - bound).max())


def check_out(gpu_out32: np.ndarray, ref: np.ndarray):
    diff = gpu_out32.astype(np.float64) - ref
    den = np.linalg.norm(ref)
    rel = np.linalg.norm(diff) / den if den > 0 else np.linalg.norm(diff)
    mx = np.abs(diff).max() if diff.size else 0.0
    assert rel <= REL_FRO, f"relative Frobenius error {rel:.3e} > {REL_FRO}"
    assert mx <= MAX_ABS, f"max-abs error {mx:.3e} > {MAX_ABS}"
    return rel, mx


def bf16_of(t32: torch.Tensor) -> torch.Tensor:
    return t32.to(torch.bfloat16)


def make_near_ties(inp, frac: float, seed: int, margin: float = 1e-4):
    """Adversarial near-tie tokens (workload 5): for a seeded `frac` of the
    tokens, nudge single bf16 coordinates of x until the 8th and 9th largest
    router logits (exact arithmetic on the stored bf16 values) are within
    `margin`.  Returns the modified x (device bf16), the chosen token indices,
    and a fresh perturbed copy of x for recording replay ids.  Input
    construction only; the layer's own arithmetic is not involved."""
    k = inp.cfg.k
    T = inp.x.shape[0]
    rng = np.random.default_rng(seed)
    idx = np.sort(rng.choice(T, int(round(frac * T)), replace=False))
    wr = torch.from_numpy(bf16_bits(inp.w_router).view(np.int16)).view(torch.bfloat16).double().numpy()
    bias = 0.0 if inp.router_bias is None else inp.router_bias.double().cpu().numpy()
    xs = inp.x[torch.as_tensor(idx, device=inp.x.device)].double().cpu().numpy()
    done = 0
    for n in range(len(idx)):
        x = xs[n]
        for _ in range(12):
            lg = wr @ x + bias
            order = np.argsort(-lg, kind="stable")
            a, b = order[k - 1], order[k]
            gap = lg[a] - lg[b]
            if gap < margin:
                done += 1
                break
            c = wr[a] - wr[b]
            cand = np.argsort(-np.abs(c))[:256]
            target = x[cand] - gap / c[cand]
            new = torch.from_numpy(target).to(torch.bfloat16).double().numpy()
            resid = np.abs(gap + (new - x[cand]) * c[cand])
            resid[np.abs(new) > 4.0] = np.inf
            j = cand[int(np.argmin(resid))]
            x[j] = torch.tensor(float(new[cand.tolist().index(j)])).to(torch.bfloat16).double().item()
        xs[n] = x
    x_new = inp.x.clone()
    x_new[torch.as_tensor(idx, device=inp.x.device)] = torch.from_numpy(xs).to(
        device=inp.x.device, dtype=torch.float32).to(torch.bfloat16)
    g = torch.Generator(device=inp.x.device).manual_seed(seed + 7)
    noise = torch.randn(x_new.shape, generator=g, device=inp.x.device) * inp.cfg.replay_noise
    x_rep = (x_new.float() + noise).to(torch.bfloat16)
    return x_new, idx, x_rep, done


# ---- backward -------------------------------------------------------------------

def _f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().to(torch.float64).cpu().numpy()


def expert_values_getter(inp):
    from oracle.backward import ExpertValues

    def get(e: int):
        return ExpertValues(_f64(inp.w_gate[e]), _f64(inp.w_up[e]), _f64(inp.w_down[e]))
    return get


def shared_values(inp):
    from oracle.backward import ExpertValues
    if inp.ws_gate is None:
        return []
    return [ExpertValues(_f64(inp.ws_gate), _f64(inp.ws_up), _f64(inp.ws_down))]


def oracle_backward(inp, ids, dout, valid=None, **limits):
    """The fp64 backward oracle on the layer's (bf16) inputs, ids [T][k] and
    dout [T][d] (device or host tensors)."""
    from oracle import backward
    bias = None if inp.router_bias is None else _f64(inp.router_bias)
    ids_np = ids.cpu().numpy() if isinstance(ids, torch.Tensor) else np.asarray(ids)
    return backward.layer_backward(_f64(inp.x), _f64(inp.w_router), bias,
                                   expert_values_getter(inp), shared_values(inp), ids_np,
                                   _f64(dout), valid=valid, **limits)


# Gradient comparison: relative Frobenius error <= 5e-3 (as for the forward
# output) and every element within 3e-2 of the tensor's largest magnitude.
# The GPU multiplies the same MXFP8 values as the oracle, so the difference is
# fp32 accumulation order plus rare E4M3 code flips where an fp32 operand lies
# within its rounding error of a rounding boundary (one E4M3 step, <= 2^-3 of
# one operand element, in a few elements).
GRAD_REL_FRO = 5e-3
GRAD_MAX_ABS_REL = 3e-2


def check_grad(name: str, gpu, ref: np.ndarray):
    g = gpu.detach().to(torch.float64).cpu().numpy() if isinstance(gpu, torch.Tensor) else gpu
    assert g.shape == ref.shape, (name, g.shape, ref.shape)
    assert np.isfinite(g).all(), name
    scale = float(np.abs(ref).max())
    if scale == 0.0:
        assert not g.any(), f"{name}: expected all zeros"
        return
    rel = float(np.linalg.norm(g - ref) / np.linalg.norm(ref))
    mx = float(np.abs(g - ref).max())
    assert rel <= GRAD_REL_FRO, f"{name}: relative Frobenius error {rel:.3e}"
    assert mx <= GRAD_MAX_ABS_REL * scale, f"{name}: max-abs error {mx:.3e} (scale {scale:.3e})"


# ---- whole-batch routing checks and sampled outputs at full size ----------------

def boundary_tokens(cnt: np.ndarray, off: np.ndarray, perm: np.ndarray, k: int,
                    tile: int = 256) -> list:
    """Tokens at the edges the expert GEMMs' tiling creates: for one expert of
    every class (no token tile larger than 64, 128, 192 or 256 rows; several
    token tiles, with the last one full or ragged; the busiest and the least
    busy expert), the tokens at rows 0, 31/32, 63/64, 127/128, 255/256,
    511/512 and the last row of its segment in dispatch order."""
    chosen = {}
    nz = np.nonzero(cnt)[0]
    for e in nz:
        n = int(cnt[e])
        cls = ("cold", (n + 63) // 64) if n <= tile else ("hot", min(n // tile, 3), n % tile == 0)
        chosen.setdefault(cls, int(e))
    if len(nz):
        chosen["max"] = int(nz[np.argmax(cnt[nz])])
        chosen["min"] = int(nz[np.argmin(cnt[nz])])
    toks = set()
    for e in chosen.values():
        n = int(cnt[e])
        for pos in (0, 31, 32, 63, 64, 127, 128, 255, 256, 511, 512, n - 1):
            if 0 <= pos < n:
                toks.add(int(perm[off[e] + pos]) // k)
    return sorted(toks)


def check_batch_routing(inp, x, layer, ids, gates, replay_ids=None):
    """Whole-batch checks of one GPU call against the oracle: fp32 logits of
    every token; ids by the id rules (own mode) or equal to the recorded ids
    (replay); every token's gate weights against the oracle's gate weights over
    the ids the GPU used (the oracle in replay mode with those ids); and the
    counting sort (cnt, off, perm, inv) of those ids, bit for bit.  Returns
    (oracle logits, GPU ids, mask of tokens whose GPU ids equal the oracle's
    own selection, intermediates)."""
    T, k, E = x.shape[0], inp.cfg.k, inp.cfg.E
    wr, bias = router_host(inp)
    ref_logits = oracle.router_logits(bf16_bits(x), wr, bias)
    im = layer.intermediates(T)
    check_logits(im["logits"].cpu().numpy(), ref_logits)
    g_ids = ids.cpu().numpy()
    if replay_ids is None:
        same = check_ids(g_ids, ref_logits, k)
    else:
        assert np.array_equal(g_ids, replay_ids)
        same = np.all(g_ids == oracle.select_topk(ref_logits, k), axis=1)
    check_gates(gates.cpu().numpy(), oracle.gate_weights(ref_logits, g_ids))
    cnt, off, perm, inv = oracle.counting_sort(g_ids, E)
    assert np.array_equal(im["cnt"].cpu().numpy(), cnt)
    assert np.array_equal(im["off"].cpu().numpy(), off)
    assert np.array_equal(im["perm"].cpu().numpy(), perm)
    assert np.array_equal(im["inv"].cpu().numpy(), inv)
    return ref_logits, g_ids, same, (cnt, off, perm)


def check_sampled_outputs(inp, x, out32, g_ids, tokens):
    """Layer outputs of the sampled tokens against the oracle run in replay
    mode with the ids the GPU used (for tokens whose ids equal the oracle's own
    selection this is the own-mode oracle)."""
    tk = np.asarray(sorted(set(int(t) for t in tokens)))
    ref = oracle_layer(inp, tokens=tk, replay_ids=g_ids[tk], x=x)
    return check_out(out32.cpu().numpy()[tk], ref.out)
