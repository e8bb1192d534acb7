"""MXFP8 expert compute (MXFP8 weights and MXFP8 activations: each token row
quantised along d before the gate/up GEMM, each bf16 row of the SwiGLU output
along F before the down GEMM; the pages' MXFP8 format) on the GPU path, where
both expert GEMMs run on the block-scaled tensor-core MMA.

The quantised activations (E4M3 codes and E8M0 scales) decode bitwise to the
oracle's quantisation of the same rows; the layer matches the oracle within
the usual tolerance and keeps batch invariance (across every tile width) and
run-to-run determinism."""
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


def _decoded(codes, scales):
    """E4M3 codes times 2^(E8M0 scale - 127), one scale per 32 codes (fp64)."""
    v = codes.contiguous().view(torch.float8_e4m3fn).to(torch.float64).cpu().numpy()
    e = (scales.to(torch.int64) - 127).repeat_interleave(32, dim=-1).cpu().numpy()
    return np.ldexp(v, e)  # exact (a power-of-two multiply on the host)


def small_mxa(T=300, E=32, seed=43):
    return CONFIGS["c5_mxfp8_act"].with_(name=f"mxa_T{T}", seed=seed, T=T, d=512, E=E, F=512)


@pytest.mark.parametrize("T", [1, 37, 300])
def test_mxfp8_activations_match_oracle(T):
    inp = make_layer(small_mxa(T), "cuda")
    layer = MoELayer.from_inputs(inp, out_fp32=True)
    assert layer.wfmt == B.MOE_W_MXFP8_ACT
    out, ids, gates = layer.forward(inp.x)
    assert layer.status() == 0
    ref = mc.oracle_layer(inp)
    same = mc.check_ids(ids.cpu().numpy(), ref.logits, 8)
    mc.check_out(out.cpu().numpy()[same], ref.out[same])
    rid = mc.oracle_replay_ids(inp)
    out_r, _, gates_r = layer.forward(inp.x, replay_ids=torch.from_numpy(rid).cuda())
    ref_r = mc.oracle_layer(inp, replay_ids=rid)
    mc.check_gates(gates_r.cpu().numpy(), ref_r.gates)
    mc.check_out(out_r.cpu().numpy(), ref_r.out)
    # the token rows entering the experts: the oracle's quantisation, bitwise
    im = layer.intermediates(T)
    np.testing.assert_array_equal(_decoded(im["x8"], im["xs"]),
                                  oracle.mx_qdq_rows(inp.x.to(torch.float64).cpu().numpy()))
    # and the rows of h entering the down GEMM: h8 / hs are h's quantisation
    h = im["h"][: T * 8].to(torch.float64).cpu().numpy()
    np.testing.assert_array_equal(_decoded(im["h8"], im["hs"]), oracle.mx_qdq_rows(h))


def test_quantised_rows_feed_the_mxfp8_weight_layer():
    """With activation quantisation only on x (H quantisation is inside the
    layer) the first GEMM's input equals the MXFP8-weight layer's input on the
    quantised x: their routing and gates agree bitwise (the router reads the
    unquantised x in both)."""
    inp = make_layer(small_mxa(200), "cuda")
    a = MoELayer.from_inputs(inp, out_fp32=True)
    out_a, ids_a, g_a = [t.clone() for t in a.forward(inp.x)]
    plain = MoELayer(inp.w_router, inp.w_gate, inp.w_up, inp.w_down, s_gate=inp.s_gate,
                     s_up=inp.s_up, s_down=inp.s_down, router_bias=inp.router_bias,
                     out_fp32=True)
    out_p, ids_p, g_p = plain.forward(inp.x)
    assert torch.equal(ids_a, ids_p) and torch.equal(g_a, g_p)
    assert not torch.equal(out_a, out_p)   # the activations really are quantised
    rel = (out_a - out_p).norm() / out_p.norm()
    assert rel < 0.1


def test_mxfp8_activations_deterministic_and_batch_invariant():
    inp = make_layer(small_mxa(T=600, seed=49), "cuda")
    layer = MoELayer.from_inputs(inp, out_fp32=True)
    full = [t.clone() for t in layer.forward(inp.x)]
    again = layer.forward(inp.x)
    for a, b in zip(full, again):
        assert torch.equal(a, b)
    # sub-batches, including ones small enough for the weight-streaming variant
    for lo, hi in ((0, 1), (0, 64), (100, 228), (300, 429)):
        part = layer.forward(inp.x[lo:hi].contiguous())
        for a, b in zip(full, part):
            assert torch.equal(a[lo:hi], b)


def test_mxfp8_activations_full_size_sampled():
    cfg = CONFIGS["c5_mxfp8_act"]
    inp = make_layer(cfg, "cuda")
    layer = MoELayer.from_inputs(inp, out_fp32=True)
    out, ids, gates = layer.forward(inp.x)
    assert layer.status() == 0
    tokens = np.asarray([0, 1, 2, 8191, 16383])
    ref = mc.oracle_layer(inp, tokens=tokens)
    same = mc.check_ids(ids.cpu().numpy()[tokens], ref.logits, 8)
    mc.check_out(out.cpu().numpy()[tokens][same], ref.out[same])
    im = layer.intermediates(cfg.T)
    tk = torch.as_tensor(tokens, device="cuda")
    np.testing.assert_array_equal(
        _decoded(im["x8"][tk], im["xs"][tk]),
        oracle.mx_qdq_rows(inp.x[tk].to(torch.float64).cpu().numpy()))
