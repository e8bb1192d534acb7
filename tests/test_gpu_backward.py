"""The MoE layer backward (MXFP8 expert GEMMs) through the C ABI against the
fp64 backward oracle, on seeded inputs: every gradient element by element on
small layers (ragged expert runs, unused experts, the shared expert, rejected
replay ids), the quantised operand buffers bit for bit where their inputs are
the layer's own, run-to-run determinism, batch invariance of dx, and sampled
outputs on the 32k-token layer (d=7168, E=384, F=2048, shared expert)."""
import numpy as np
import pytest
import torch

import oracle
from oracle import backward as OB
from deterministic_rl_gb300 import build, MoELayer
from deterministic_rl_gb300.synthetic import CONFIGS, make_layer, make_dout, make_replay_ids
import moe_cases as mc

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    build.build()
    oracle.build()


def small_cfg(T, d=512, E=16, F=256, shared=1, seed=21, zipf=0.0):
    return CONFIGS["c1_tiny"].with_(name=f"bwd_T{T}_E{E}_S{shared}", seed=seed, T=T, d=d, E=E,
                                    F=F, n_shared=shared, zipf=zipf)


def run_backward(inp, ids=None, dout=None):
    """The backward with recorded ids (seeded, host-drawn) and a seeded dout."""
    layer = MoELayer.from_inputs(inp)
    if ids is None:
        ids = make_replay_ids(inp.cfg, device="cuda")
    if dout is None:
        dout = make_dout(inp.cfg, device="cuda")
    dx, g = layer.backward(inp.x, ids, dout)
    torch.cuda.synchronize()
    return layer, ids, dout, dx, g


def compare_all(inp, ids, dout, dx, g, valid=None):
    ref = mc.oracle_backward(inp, ids, dout, valid=valid)
    mc.check_grad("dx", dx, ref.dx)
    mc.check_grad("d_router", g["d_router"], ref.d_router)
    E = inp.cfg.E
    for e in range(E):
        if e in ref.experts:
            r = ref.experts[e]
            mc.check_grad(f"d_gate[{e}]", g["d_gate"][e], r.d_gate)
            mc.check_grad(f"d_up[{e}]", g["d_up"][e], r.d_up)
            mc.check_grad(f"d_down[{e}]", g["d_down"][e], r.d_down)
        else:  # an expert without tokens has zero gradients
            assert not g["d_gate"][e].any() and not g["d_up"][e].any() and not g["d_down"][e].any()
    if inp.cfg.n_shared:
        mc.check_grad("ds_gate", g["ds_gate"], ref.shared[0].d_gate)
        mc.check_grad("ds_up", g["ds_up"], ref.shared[0].d_up)
        mc.check_grad("ds_down", g["ds_down"], ref.shared[0].d_down)
    return ref


CASES = [CONFIGS["c1_tiny"].with_(n_shared=1, name="c1_tiny_shared"), CONFIGS["c1_tiny"],
         small_cfg(37, shared=0), small_cfg(300, zipf=1.0), small_cfg(1)]


@pytest.mark.parametrize("cfg", CASES, ids=lambda c: c.name)
def test_backward_matches_oracle(cfg):
    inp = make_layer(cfg, "cuda")
    layer, ids, dout, dx, g = run_backward(inp)
    assert layer.backward_status() == 0
    ref = compare_all(inp, ids, dout, dx, g)
    inter = layer.backward_intermediates(cfg.T)
    mc.check_grad("dgates", inter["dg"], ref.dgates)
    mc.check_grad("dlogits", inter["dl"], ref.dlogits)


def test_unused_experts_and_ragged_runs():
    cfg = small_cfg(200, E=16)
    inp = make_layer(cfg, "cuda")
    gen = torch.Generator().manual_seed(5)
    # only experts 0..11 are used, with uneven counts (runs of 1 .. 300 tokens)
    ids = torch.stack([torch.randperm(12, generator=gen)[:8] for _ in range(cfg.T)]).to(torch.int32)
    ids[:40] = torch.arange(8, dtype=torch.int32)  # experts 0..7 get 40 more tokens
    layer, ids, dout, dx, g = run_backward(inp, ids=ids.cuda())
    compare_all(inp, ids, dout, dx, g)
    for e in range(12, 16):
        assert not g["d_router"][e].any()


def test_rejected_replay_ids_contribute_nothing():
    cfg = small_cfg(64)
    inp = make_layer(cfg, "cuda")
    ids = make_replay_ids(cfg)
    bad = ids.clone()
    bad[3, 1] = bad[3, 0]      # repeated id
    bad[10, 7] = cfg.E + 5     # out of range
    layer, _, dout, dx, g = run_backward(inp, ids=bad.cuda())
    from deterministic_rl_gb300 import binding as B
    assert layer.backward_status() == B.MOE_ERR_BAD_IDS
    assert not dx[3].any() and not dx[10].any()
    # rejected rows are replaced by ids 0 .. k-1 with zero weight (the ABI's rule)
    used = bad.clone()
    used[[3, 10]] = torch.arange(cfg.k, dtype=torch.int32)
    assert torch.equal(layer.backward_intermediates(cfg.T)["ids"].cpu(), used)
    valid = np.ones(cfg.T, np.uint8)
    valid[[3, 10]] = 0
    compare_all(inp, used, dout, dx, g, valid=valid)


def mx_values(codes, scales):
    """fp64 values of E4M3 codes [..., n] with E8M0 scale bytes [..., n / 32]."""
    v = codes.cpu().view(torch.float8_e4m3fn).to(torch.float64).numpy()
    x = np.exp2(scales.cpu().numpy().astype(np.float64) - 127.0)
    return v * np.repeat(x, 32, axis=-1)


def test_weight_copies_are_the_oracle_quantisation_bit_for_bit():
    """The block-scaled operands of dH and dXp: codes and scale bytes of the
    transposed weights, routed experts then the shared one (group E)."""
    cfg = small_cfg(16, d=512, E=8, F=256)
    inp = make_layer(cfg, "cuda")
    layer = MoELayer.from_inputs(inp)
    wt = layer.prepare_backward()
    torch.cuda.synchronize()
    E, d, F = cfg.E, cfg.d, cfg.F
    G = E + 1
    n = G * F * d
    align = lambda b: (b + 255) // 256 * 256  # noqa: E731
    o_wds = align(n)
    o_w2 = o_wds + align(n // 32)
    o_w2s = o_w2 + align(2 * n)
    assert wt.numel() >= o_w2s + 2 * n // 32
    wd = mx_values(wt[:n].view(G, F, d), wt[o_wds:o_wds + n // 32].view(G, F, d // 32))
    w2 = mx_values(wt[o_w2:o_w2 + 2 * n].view(G, d, 2 * F),
                   wt[o_w2s:o_w2s + 2 * n // 32].view(G, d, 2 * F // 32))
    f64 = lambda t: t.to(torch.float64).cpu().numpy()  # noqa: E731
    mats = [(inp.w_gate[e], inp.w_up[e], inp.w_down[e]) for e in range(E)]
    mats.append((inp.ws_gate, inp.ws_up, inp.ws_down))
    for g, (wg, wu, wdn) in enumerate(mats):
        np.testing.assert_array_equal(wd[g], OB.mx_quantize(f64(wdn), 0).T)
        np.testing.assert_array_equal(w2[g][:, :F], OB.mx_quantize(f64(wg), 0).T)
        np.testing.assert_array_equal(w2[g][:, F:], OB.mx_quantize(f64(wu), 0).T)


def test_row_operands_are_the_oracle_quantisation_bit_for_bit():
    """Q_d(dY) rows (codes and scale bytes) of the dH GEMM: gate(t, s) * dout[t]
    at the pair's dispatch row, dout[t] at shared row T k + t."""
    cfg = small_cfg(150, E=16, zipf=1.0)
    inp = make_layer(cfg, "cuda")
    layer, ids, dout, dx, g = run_backward(inp)
    inter = layer.backward_intermediates(cfg.T)
    T, k, d = cfg.T, cfg.k, cfg.d
    dyq = mx_values(inter["dyq"], inter["dyq_scales"])
    gates = inter["gates"].cpu().numpy().astype(np.float64)
    do = dout.to(torch.float64).cpu().numpy()
    perm = inter["perm"].cpu().numpy()
    rows = np.empty((T * k + T, d))
    for r in range(T * k):
        pair = perm[r]
        # the product in fp32, as the kernel forms it before quantising
        rows[r] = gates.reshape(-1)[pair].astype(np.float32) * do[pair // k].astype(np.float32)
    rows[T * k:] = do
    np.testing.assert_array_equal(dyq, OB.mx_quantize(rows, 1))


def test_token_major_inputs_are_the_oracle_quantisation_bit_for_bit():
    cfg = small_cfg(150, E=16, zipf=1.0)
    inp = make_layer(cfg, "cuda")
    layer, ids, dout, dx, g = run_backward(inp)
    inter = layer.backward_intermediates(cfg.T)
    ids_np = ids.cpu().numpy()
    k, E, T = cfg.k, cfg.E, cfg.T
    x = inp.x.to(torch.float64).cpu().numpy()
    xpt = inter["xpt"].to(torch.float64).cpu().numpy()
    poff = inter["poff"].cpu().numpy()
    # the oracle's dispatch order and padded offsets
    runs = OB.dispatch_rows(ids_np, E) + [np.arange(T) * k]   # shared: every token
    p = 0
    for gi, pairs in enumerate(runs):
        n = len(pairs)
        assert poff[gi] == p
        pad = (n + 63) // 64 * 64
        rows = x[pairs // k]
        q = OB.mx_quantize(np.pad(rows, ((0, pad - n), (0, 0))), 0)
        np.testing.assert_array_equal(xpt[:, p:p + pad], q.T)
        p += pad
    assert poff[len(runs)] == p


def test_backward_is_deterministic_and_dx_batch_invariant():
    cfg = small_cfg(300, E=16, zipf=1.0)
    inp = make_layer(cfg, "cuda")
    layer, ids, dout, dx1, g1 = run_backward(inp)
    dx1 = dx1.clone()
    g1 = {k: v.clone() for k, v in g1.items()}
    dx2, g2 = layer.backward(inp.x, ids, dout)
    torch.cuda.synchronize()
    assert torch.equal(dx1, dx2)
    for k in g1:
        assert torch.equal(g1[k], g2[k]), k
    # a token's dx row does not depend on the rest of the batch
    for n in (1, 77, 256):
        sub = MoELayer.from_inputs(inp)
        dxs, _ = sub.backward(inp.x[:n].contiguous(), ids[:n].contiguous(), dout[:n].contiguous())
        torch.cuda.synchronize()
        assert torch.equal(dxs, dx1[:n]), n


def test_full_size_layer_sampled():
    """The 32k-token layer (d=7168, E=384, F=2048, shared expert) on the launch
    configuration the benchmark times: dx and the gate/logit gradients of
    sampled tokens, and every weight gradient of the experts with the fewest
    and the most tokens, against the oracle."""
    cfg = CONFIGS["c4_train_32k"]
    inp = make_layer(cfg, "cuda")
    layer, ids, dout, dx, g = run_backward(inp)
    assert layer.backward_status() == 0
    inter = layer.backward_intermediates(cfg.T)
    cnt = inter["cnt"].cpu().numpy()
    e_lo, e_hi = int(cnt.argmin()), int(cnt.argmax())
    toks = [0, 1, 12345, cfg.T - 1]
    ref = mc.oracle_backward(inp, ids, dout, tokens=toks, grad_experts=[e_lo, e_hi],
                             grad_shared=False)
    for t in toks:
        mc.check_grad(f"dx[{t}]", dx[t], ref.dx[t])
        mc.check_grad(f"dgates[{t}]", inter["dg"][t], ref.dgates[t])
        mc.check_grad(f"dlogits[{t}]", inter["dl"][t], ref.dlogits[t])
    for e in (e_lo, e_hi):
        r = ref.experts[e]
        mc.check_grad(f"d_gate[{e}]", g["d_gate"][e], r.d_gate)
        mc.check_grad(f"d_up[{e}]", g["d_up"][e], r.d_up)
        mc.check_grad(f"d_down[{e}]", g["d_down"][e], r.d_down)
    assert torch.isfinite(g["ds_gate"]).all() and torch.isfinite(g["d_router"]).all()


@pytest.mark.parametrize("cfg", [CONFIGS["c1_tiny"].with_(n_shared=1, name="c1_tiny_shared"),
                                 small_cfg(300, zipf=1.0), small_cfg(37, shared=0)],
                         ids=lambda c: c.name)
def test_training_forward_and_saved_backward_match_the_separate_calls(cfg):
    inp = make_layer(cfg, "cuda")
    ref_layer = MoELayer.from_inputs(inp, out_fp32=True)
    layer = MoELayer.from_inputs(inp, out_fp32=True)
    dout = make_dout(cfg, device="cuda")
    rid = make_replay_ids(cfg, device="cuda")
    for replay in (None, rid):
        out0, ids0, g0 = ref_layer.forward(inp.x, replay_ids=replay)
        out1, ids1, g1 = layer.forward_train(inp.x, replay_ids=replay)
        torch.cuda.synchronize()
        assert torch.equal(out0, out1) and torch.equal(ids0, ids1) and torch.equal(g0, g1)
        dx0, gr0 = ref_layer.backward(inp.x, ids0, dout)
        dx0 = dx0.clone()
        gr0 = {k: v.clone() for k, v in gr0.items()}
        for _ in range(2):  # twice on one training forward
            dx1, gr1 = layer.backward_saved(dout)
            torch.cuda.synchronize()
            assert torch.equal(dx0, dx1)
            for k in gr0:
                assert torch.equal(gr0[k], gr1[k]), k
    assert layer.backward_status() == 0
