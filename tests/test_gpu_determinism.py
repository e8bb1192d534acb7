"""Determinism and batch invariance of the GPU path (the property the Training
Data No. 94 write-up, section "浮点数不守规矩，MoE 火上浇油", asks of fixed-order
kernels), replay-id validation, and sampled parity at full size for the
prefill-like and 32k-token layers."""
import numpy as np
import pytest
import torch

import oracle
from deterministic_rl_gb300 import build, MoELayer
from deterministic_rl_gb300 import binding as B
from deterministic_rl_gb300.synthetic import CONFIGS, make_layer
import moe_cases as mc

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    build.build()
    oracle.build()


def small(T, **kw):
    base = dict(name=f"det_T{T}", seed=21, T=T, d=256, E=48, F=192, n_shared=1)
    base.update(kw)
    return CONFIGS["c1_tiny"].with_(**base)


def test_repeated_runs_are_bitwise_identical():
    inp = make_layer(small(300), "cuda")
    layer = MoELayer.from_inputs(inp, out_fp32=True)
    first = [t.clone() for t in layer.forward(inp.x)]
    for _ in range(10):
        again = layer.forward(inp.x)
        for a, b in zip(first, again):
            assert torch.equal(a, b)


def test_token_order_permutes_output_bitwise():
    inp = make_layer(small(257), "cuda")
    layer = MoELayer.from_inputs(inp, out_fp32=True)
    out, ids, gates = [t.clone() for t in layer.forward(inp.x)]
    g = torch.Generator(device="cpu").manual_seed(3)
    perm = torch.randperm(257, generator=g).cuda()
    out_p, ids_p, gates_p = layer.forward(inp.x[perm].contiguous())
    assert torch.equal(ids_p, ids[perm]) and torch.equal(gates_p, gates[perm])
    assert torch.equal(out_p, out[perm])


def test_scaling_w_down_by_two_doubles_output_exactly():
    inp = make_layer(small(200), "cuda")
    a = MoELayer.from_inputs(inp, out_fp32=True).forward(inp.x)[0].clone()
    inp.w_down = inp.w_down * 2
    inp.ws_down = inp.ws_down * 2
    b = MoELayer.from_inputs(inp, out_fp32=True).forward(inp.x)[0]
    assert torch.equal(b, 2 * a)


@pytest.mark.parametrize("T_full,T_part", [(1000, 1), (1000, 130), (4096, 512)])
def test_batch_invariance_small(T_full, T_part):
    inp = make_layer(small(T_full), "cuda")
    layer = MoELayer.from_inputs(inp, out_fp32=True)
    full = [t.clone() for t in layer.forward(inp.x)]
    part = layer.forward(inp.x[:T_part].contiguous())
    for a, b in zip(full, part):
        assert torch.equal(a[:T_part], b)
    # a suffix too: positions inside the batch do not matter
    tail = layer.forward(inp.x[T_full - T_part:].contiguous())
    for a, b in zip(full, tail):
        assert torch.equal(a[T_full - T_part:], b)


def test_invalid_replay_ids_are_reported_and_zeroed():
    cfg = small(16)
    inp = make_layer(cfg, "cuda")
    layer = MoELayer.from_inputs(inp, out_fp32=True)
    rid = mc.oracle_replay_ids(inp)
    good = layer.forward(inp.x, replay_ids=torch.from_numpy(rid).cuda())
    good = [t.clone() for t in good]
    assert layer.status() == B.MOE_OK
    bad = rid.copy()
    bad[3, 2] = cfg.E          # out of range
    bad[7, 5] = bad[7, 1]      # repeated
    bad[9, 0] = -1             # negative
    out, ids, gates = layer.forward(inp.x, replay_ids=torch.from_numpy(bad).cuda())
    assert layer.status() == B.MOE_ERR_BAD_IDS
    assert int(layer.intermediates(cfg.T)["status"][2]) == 3
    rows = [3, 7, 9]
    keep = [t for t in range(cfg.T) if t not in rows]
    assert (out[rows] == 0).all() and (gates[rows] == 0).all()
    assert (ids[rows].cpu() == torch.arange(8, dtype=torch.int32)).all()
    assert torch.equal(out[keep], good[0][keep])
    # the next valid call clears the status
    layer.forward(inp.x, replay_ids=torch.from_numpy(rid).cuda())
    assert layer.status() == B.MOE_OK


def _sampled_parity(inp, layer, tokens, replay):
    out, ids, gates = layer.forward(inp.x, replay_ids=replay)
    torch.cuda.synchronize()
    assert layer.status() == 0
    tk = np.asarray(tokens)
    rid = None if replay is None else replay.cpu().numpy()[tk]
    ref = mc.oracle_layer(inp, tokens=tk, replay_ids=rid)
    lg = layer.intermediates(inp.cfg.T)["logits"].cpu().numpy()[tk]
    mc.check_logits(lg, ref.logits)
    g_ids = ids.cpu().numpy()[tk]
    if replay is None:
        same = mc.check_ids(g_ids, ref.logits, inp.cfg.k)
    else:
        assert np.array_equal(g_ids, rid)
        same = np.ones(len(tk), bool)
    mc.check_gates(gates.cpu().numpy()[tk], oracle.gate_weights(ref.logits, g_ids))
    rel_mx = mc.check_out(out.cpu().numpy()[tk][same], ref.out[same])
    # tokens whose GPU ids differ from the oracle's own choice (near ties):
    # the oracle replaying the GPU's ids
    if not same.all():
        mc.check_sampled_outputs(inp, inp.x, out, ids.cpu().numpy(), tk[~same])
    return rel_mx


@pytest.mark.slow
def test_prefill_zipf_full_size_sampled_parity():
    cfg = CONFIGS["c3_prefill_zipf"]
    inp = make_layer(cfg, "cuda")
    layer = MoELayer.from_inputs(inp, out_fp32=True)
    tokens = [0, 1, 2, 127, 128, 1000, 2047, 2048, 3333, 4094, 4095]
    _sampled_parity(inp, layer, tokens, None)
    rid = mc.oracle_replay_ids(inp)  # the whole batch's recorded ids
    _sampled_parity(inp, layer, tokens, torch.from_numpy(rid).cuda())


@pytest.mark.slow
@pytest.mark.parametrize("zipf", [0.0, 1.2])
def test_train_32k_batch_invariance_and_sampled_parity(zipf):
    cfg = CONFIGS["c4_train_32k"].with_(zipf=zipf)
    inp = make_layer(cfg, "cuda")
    layer = MoELayer.from_inputs(inp, out_fp32=True)
    full = [t.clone() for t in layer.forward(inp.x)]
    part = MoELayer.from_inputs(inp, out_fp32=True).forward(inp.x[:512].contiguous())
    for a, b in zip(full, part):
        assert torch.equal(a[:512], b), "first 512 tokens differ between T=512 and T=32768"
    tokens = [0, 5, 511, 512, 20000, 32767]
    _sampled_parity(inp, layer, tokens, None)
