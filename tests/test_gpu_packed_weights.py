"""Packed gate/up weights (moe_pack_weights): the layout is the documented
interleave (per expert and 64-row block of F: 64 gate rows, then the same 64
up rows), and the forward reading it gives bitwise the outputs of the forward
reading w_gate / w_up, for the SM-pair family (with the shared expert on its
own stream or without one) and the one-SM family (which ignores it)."""
import pytest
import torch

from deterministic_rl_gb300 import build, MoELayer
from deterministic_rl_gb300.synthetic import CONFIGS, make_layer, make_replay_ids

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    build.build()


def _cfg(T, shared, seed):
    return CONFIGS["c1_tiny"].with_(name=f"pk_T{T}_S{shared}", seed=seed, T=T, d=512, E=24,
                                    F=384, n_shared=shared)


def test_packed_layout():
    inp = make_layer(_cfg(16, 1, 71), "cuda")
    layer = MoELayer.from_inputs(inp)
    pk = layer.pack_weights().view(torch.bfloat16)
    torch.cuda.synchronize()
    E, F, d = inp.cfg.E, inp.cfg.F, inp.cfg.d
    g = torch.cat([inp.w_gate, inp.ws_gate[None]]).view(E + 1, F // 64, 64, d)
    u = torch.cat([inp.w_up, inp.ws_up[None]]).view(E + 1, F // 64, 64, d)
    ref = torch.cat([g, u], dim=2).reshape(-1)
    assert torch.equal(pk.view(-1), ref)


@pytest.mark.parametrize("T,shared", [(300, 1), (700, 0), (64, 1)])
def test_packed_forward_is_bitwise_the_unpacked_one(T, shared):
    cfg = _cfg(T, shared, 72 + T)
    inp = make_layer(cfg, "cuda")
    plain = MoELayer.from_inputs(inp, out_fp32=True)
    packed = MoELayer.from_inputs(inp, out_fp32=True)
    packed.pack_weights()
    rid = make_replay_ids(cfg, device="cuda")
    for replay in (None, rid):
        a = [t.clone() for t in plain.forward(inp.x, replay_ids=replay)]
        b = packed.forward(inp.x, replay_ids=replay)
        torch.cuda.synchronize()
        assert plain.status() == 0 and packed.status() == 0
        for x, y in zip(a, b):
            assert torch.equal(x, y)
