"""GPU path (through the C ABI) against the fp64 oracle on seeded inputs.

Small cases (the tiny layer and ragged shapes) are compared element by
element; the decode-like replay layer (T=64, d=7168, E=384, F=2048, shared
expert) is compared on every token at full size."""
import numpy as np
import pytest
import torch

import oracle
from deterministic_rl_gb300 import build, MoELayer
from deterministic_rl_gb300.synthetic import CONFIGS, make_layer, bf16_bits
import moe_cases as mc

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    build.build()
    oracle.build()


def run_both(inp, layer32, layer16, replay=None):
    out32, ids32, g32 = layer32.forward(inp.x, replay_ids=replay)
    out16, ids16, g16 = layer16.forward(inp.x, replay_ids=replay)
    torch.cuda.synchronize()
    assert torch.equal(ids32, ids16) and torch.equal(g32, g16)
    # bf16 output is the fp32 result rounded once to nearest even
    assert torch.equal(out16, out32.to(torch.bfloat16))
    return out32, ids32, g32


def small_cfg(T, d=256, E=32, F=128, shared=0, seed=11, zipf=0.0):
    return CONFIGS["c1_tiny"].with_(name=f"small_T{T}", seed=seed, T=T, d=d, E=E, F=F,
                                    n_shared=shared, zipf=zipf)


CASES = [CONFIGS["c1_tiny"], small_cfg(1), small_cfg(37, shared=1), small_cfg(300, shared=1, zipf=1.0),
         small_cfg(129, d=192, E=72, F=320, shared=1, seed=5)]


@pytest.mark.parametrize("cfg", CASES, ids=lambda c: c.name)
def test_own_routing_matches_oracle(cfg):
    inp = make_layer(cfg, "cuda")
    l32, l16 = MoELayer.from_inputs(inp, out_fp32=True), MoELayer.from_inputs(inp)
    out32, ids, gates = run_both(inp, l32, l16)
    assert l32.status() == 0
    ref = mc.oracle_layer(inp)
    same = mc.check_ids(ids.cpu().numpy(), ref.logits, cfg.k)
    assert same.mean() > 0.95
    # logits themselves
    mc.check_logits(l32.intermediates(cfg.T)["logits"].cpu().numpy(), ref.logits)
    g_ids = ids.cpu().numpy()
    # every token's gates over the ids the GPU chose (the oracle in replay mode)
    mc.check_gates(gates.cpu().numpy(), oracle.gate_weights(ref.logits, g_ids))
    mc.check_out(out32.cpu().numpy()[same], ref.out[same])
    # tokens whose GPU ids differ (near ties): the oracle replaying those ids
    if not same.all():
        mc.check_sampled_outputs(inp, inp.x, out32, g_ids, np.nonzero(~same)[0])


@pytest.mark.parametrize("cfg", CASES, ids=lambda c: c.name)
def test_replay_matches_oracle(cfg):
    inp = make_layer(cfg, "cuda")
    rid = mc.oracle_replay_ids(inp)
    l32, l16 = MoELayer.from_inputs(inp, out_fp32=True), MoELayer.from_inputs(inp)
    out32, ids, gates = run_both(inp, l32, l16, replay=torch.from_numpy(rid).cuda())
    assert l32.status() == 0
    assert np.array_equal(ids.cpu().numpy(), rid)
    ref = mc.oracle_layer(inp, replay_ids=rid)
    mc.check_gates(gates.cpu().numpy(), ref.gates)
    mc.check_out(out32.cpu().numpy(), ref.out)


@pytest.mark.parametrize("cfg", CASES[:3] + [small_cfg(1000, E=40), small_cfg(3000, E=384, d=256)],
                         ids=lambda c: c.name)
def test_dispatch_is_the_oracle_counting_sort(cfg):
    inp = make_layer(cfg, "cuda")
    layer = MoELayer.from_inputs(inp, out_fp32=True)
    out, ids, _ = layer.forward(inp.x)
    torch.cuda.synchronize()
    im = layer.intermediates(cfg.T)
    cnt, off, perm, inv = oracle.counting_sort(ids.cpu().numpy(), cfg.E)
    assert np.array_equal(im["cnt"].cpu().numpy(), cnt)
    assert np.array_equal(im["off"].cpu().numpy(), off)
    assert np.array_equal(im["perm"].cpu().numpy(), perm)
    assert np.array_equal(im["inv"].cpu().numpy(), inv)
    # gathered rows are the tokens' hidden states in expert order (rows are
    # gathered into the workspace for batches of at most 128 tokens)
    if cfg.T <= 128:
        xp = im["xp"]
        src = torch.from_numpy(perm // cfg.k).long().cuda()
        assert torch.equal(xp[: cfg.T * cfg.k], inp.x[src])


def test_replay_of_own_ids_is_bitwise_own():
    inp = make_layer(CONFIGS["c1_tiny"], "cuda")
    layer = MoELayer.from_inputs(inp, out_fp32=True)
    out_a, ids_a, g_a = layer.forward(inp.x)
    out_a, ids_a, g_a = out_a.clone(), ids_a.clone(), g_a.clone()
    out_b, ids_b, g_b = layer.forward(inp.x, replay_ids=ids_a)
    torch.cuda.synchronize()
    assert torch.equal(ids_a, ids_b) and torch.equal(g_a, g_b) and torch.equal(out_a, out_b)


def test_decode_replay_full_size_matches_oracle():
    cfg = CONFIGS["c2_decode_replay"]
    inp = make_layer(cfg, "cuda")
    rid = mc.oracle_replay_ids(inp)
    layer = MoELayer.from_inputs(inp, out_fp32=True)
    out32, ids, gates = layer.forward(inp.x, replay_ids=torch.from_numpy(rid).cuda())
    assert layer.status() == 0
    ref = mc.oracle_layer(inp, replay_ids=rid)
    lerr = mc.check_logits(layer.intermediates(cfg.T)["logits"].cpu().numpy(), ref.logits)
    mc.check_gates(gates.cpu().numpy(), ref.gates)
    rel, mx = mc.check_out(out32.cpu().numpy(), ref.out)
    print(f"c2 replay: max logit error {lerr:.3e}")
    print(f"c2 replay: rel Frobenius {rel:.3e}, max-abs {mx:.3e}")
    # own routing agrees with the recorded ids except near ties
    own = MoELayer.from_inputs(inp, out_fp32=True)
    _, ids_own, _ = own.forward(inp.x)
    mc.check_ids(ids_own.cpu().numpy(), ref.logits, cfg.k)
