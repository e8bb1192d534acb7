"""MXFP8 expert weights (E4M3 values, one E8M0 scale per 32 elements along K;
the format of the Composer 2 Technical Report, §6.1) on the GPU path.

The kernel dequantises inside the GEMM; since the dequantised values are exact
in bf16 the layer must equal the bf16 layer on those values bitwise, and the
oracle (which decodes the bytes exactly) within the usual tolerance.  The
full-size workload adds 10 % adversarial near-tie tokens (8th and 9th logit
within 1e-4) to stress replay and determinism."""
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


def small_mx(T=300, E=32, seed=41):
    return CONFIGS["c5_mxfp8"].with_(name=f"mx_T{T}", seed=seed, T=T, d=512, E=E, F=512)


def dequantised(inp):
    """bf16 copies of the MXFP8 weights (exact), for the equivalence check."""
    def deq(q, s):
        v = q.view(torch.float8_e4m3fn).float()
        sc = torch.pow(2.0, s.float() - 127).repeat_interleave(32, dim=-1)
        out = (v * sc).to(torch.bfloat16)
        assert torch.equal(out.float(), v * sc)
        return out
    return deq(inp.w_gate, inp.s_gate), deq(inp.w_up, inp.s_up), deq(inp.w_down, inp.s_down)


@pytest.mark.parametrize("T", [1, 64, 128, 300])  # small-batch variant up to 128 tokens
def test_mxfp8_equals_bf16_on_dequantised_weights_bitwise(T):
    inp = make_layer(small_mx(T), "cuda")
    mx = MoELayer.from_inputs(inp, out_fp32=True)
    assert mx.wfmt == B.MOE_W_MXFP8
    g, u, d = dequantised(inp)
    bf = MoELayer(inp.w_router, g, u, d, router_bias=inp.router_bias, out_fp32=True)
    a = mx.forward(inp.x)
    b = bf.forward(inp.x)
    for x, y in zip(a, b):
        assert torch.equal(x, y)


def test_mxfp8_every_byte_pattern_and_float_route_scales_bitwise():
    """Weight bytes drawn uniformly from every non-NaN E4M3 pattern (one in
    sixteen is zero or subnormal, which the converters send down the exact
    float route), scale bytes 3..6 (also the float route) or 112..121 (the
    integer route): the layer must still equal the bf16 layer on the
    dequantised weights bitwise."""
    inp = make_layer(small_mx(T=300, seed=43), "cuda")
    gen = torch.Generator(device="cuda")
    gen.manual_seed(5)
    pats = torch.tensor([b for b in range(256) if (b & 0x7F) != 0x7F], dtype=torch.uint8,
                        device="cuda")
    for w, sc in ((inp.w_gate, inp.s_gate), (inp.w_up, inp.s_up), (inp.w_down, inp.s_down)):
        w.copy_(pats[torch.randint(0, len(pats), w.shape, generator=gen, device="cuda")])
        slow = torch.rand(sc.shape, generator=gen, device="cuda") < 0.3
        lo = torch.randint(3, 7, sc.shape, generator=gen, device="cuda")
        mid = torch.randint(112, 122, sc.shape, generator=gen, device="cuda")
        sc.copy_(torch.where(slow, lo, mid).to(torch.uint8))
    mx = MoELayer.from_inputs(inp, out_fp32=True)
    g, u, d = dequantised(inp)
    bf = MoELayer(inp.w_router, g, u, d, router_bias=inp.router_bias, out_fp32=True)
    a = mx.forward(inp.x)
    b = bf.forward(inp.x)
    assert torch.isfinite(a[0]).all()
    for x, y in zip(a, b):
        assert torch.equal(x, y)


def test_mxfp8_small_layer_matches_oracle():
    inp = make_layer(small_mx(), "cuda")
    layer = MoELayer.from_inputs(inp, out_fp32=True)
    out, ids, gates = layer.forward(inp.x)
    assert layer.status() == 0
    ref = mc.oracle_layer(inp)
    same = mc.check_ids(ids.cpu().numpy(), ref.logits, 8)
    mc.check_out(out.cpu().numpy()[same], ref.out[same])
    rid = mc.oracle_replay_ids(inp)
    out_r, ids_r, gates_r = layer.forward(inp.x, replay_ids=torch.from_numpy(rid).cuda())
    ref_r = mc.oracle_layer(inp, replay_ids=rid)
    mc.check_gates(gates_r.cpu().numpy(), ref_r.gates)
    mc.check_out(out_r.cpu().numpy(), ref_r.out)


def test_mxfp8_with_shared_expert_is_unsupported():
    inp = make_layer(small_mx(16), "cuda")
    w = inp.w_router
    sh = torch.zeros((512, 512), dtype=torch.bfloat16, device="cuda")
    layer = MoELayer(w, inp.w_gate, inp.w_up, inp.w_down, s_gate=inp.s_gate, s_up=inp.s_up,
                     s_down=inp.s_down, ws_gate=sh, ws_up=sh, ws_down=sh)
    out, ids, gates = layer.outputs(16)
    rc = B.moe_forward(layer.dims(16), inp.x, layer.weights, out, ids, gates, layer.workspace(16),
                       check=False)
    assert rc == B.MOE_ERR_UNSUPPORTED


@pytest.mark.slow
def test_mxfp8_full_size_near_ties():
    cfg = CONFIGS["c5_mxfp8"]
    inp = make_layer(cfg, "cuda")
    x, tie_idx, x_rep, done = mc.make_near_ties(inp, cfg.near_tie_frac, seed=cfg.seed)
    assert done == len(tie_idx) == int(round(0.1 * cfg.T))
    inp.x, inp.x_replay_src = x, x_rep
    layer = MoELayer.from_inputs(inp, out_fp32=True)
    out, ids, gates = [t.clone() for t in layer.forward(x)]
    # determinism on near ties: a second run and a sub-batch give the same bits
    again = layer.forward(x)
    for a, b in zip((out, ids, gates), again):
        assert torch.equal(a, b)
    sub = torch.as_tensor(tie_idx[:700], device="cuda")
    part = MoELayer.from_inputs(inp, out_fp32=True).forward(x[sub].contiguous())
    for a, b in zip((out, ids, gates), part):
        assert torch.equal(a[sub], b)
    # sampled parity: own mode on plain and near-tie tokens, replay with recorded ids
    tokens = [0, 1, 2, 8191, 16383] + tie_idx[:5].tolist()
    tk = np.asarray(tokens)
    ref = mc.oracle_layer(inp, tokens=tk)
    mc.check_logits(layer.intermediates(cfg.T)["logits"].cpu().numpy()[tk], ref.logits)
    same = mc.check_ids(ids.cpu().numpy()[tk], ref.logits, 8)
    mc.check_out(out.cpu().numpy()[tk][same], ref.out[same])
    rid = mc.oracle_replay_ids(inp)
    out_r, ids_r, gates_r = layer.forward(x, replay_ids=torch.from_numpy(rid).cuda())
    assert layer.status() == 0
    ref_r = mc.oracle_layer(inp, tokens=tk, replay_ids=rid[tk])
    mc.check_gates(gates_r.cpu().numpy()[tk], ref_r.gates)
    mc.check_out(out_r.cpu().numpy()[tk], ref_r.out)


def test_mxfp8_rows_equal_across_the_small_batch_variant():
    """Batches of at most 128 tokens run the weight-streaming variant (64-token
    tiles); larger ones the regular SM-pair kernel.  A token's bits do not
    depend on which one ran."""
    inp = make_layer(small_mx(T=600, seed=47), "cuda")
    layer = MoELayer.from_inputs(inp, out_fp32=True)
    full = [t.clone() for t in layer.forward(inp.x)]
    for lo, hi in ((0, 1), (0, 64), (100, 228), (300, 429)):
        part = layer.forward(inp.x[lo:hi].contiguous())
        for a, b in zip(full, part):
            assert torch.equal(a[lo:hi], b)
