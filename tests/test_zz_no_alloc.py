"""moe_route_static -- routing for callers that cannot allocate device memory
(for example an inference engine whose device memory all belongs to its own
pool, recording routing decisions inside its decode loop): the scratch lives in
a static device array of the library instead of a caller workspace.

Checked through the C ABI against moe_route (which takes a workspace) on the
same inputs, on two calls in a row: ids and gate weights must be bitwise equal,
since both calls run the same launch sequence (the same router GEMM with the
same fixed K split).  Cases: the tiny layer, the 384-expert decode shape, the
largest batch the static array serves at E = 384, a batch with adversarial
near-tied 8th/9th logits, and a layer whose K is not split.  This file sorts
last so that a run stopping at the first failure has already run every other
test; it also passes on its own in a fresh process (the static array's address
is set up by its first call)."""
import pytest
import torch

from deterministic_rl_gb300 import build, MoELayer
from deterministic_rl_gb300 import binding as B
from deterministic_rl_gb300.synthetic import CONFIGS, make_layer
import moe_cases as mc

pytestmark = pytest.mark.gpu

# largest T the 4 MiB array serves at E = 384 with the router's 4-way K split
T_MAX_E384 = 545


@pytest.fixture(scope="module", autouse=True)
def _built():
    build.build()


def _compare(inp, x=None):
    x = inp.x if x is None else x
    layer = MoELayer.from_inputs(inp)
    ref_ids, ref_gates = layer.route(x)
    torch.cuda.synchronize()
    dims = layer.dims(x.shape[0])
    for _ in range(2):  # two calls in a row share the static scratch
        ids = torch.full_like(ref_ids, -7)
        gates = torch.full_like(ref_gates, -1.0)
        B.moe_route_static(dims, x, layer.weights, ids, gates)
        torch.cuda.synchronize()
        assert torch.equal(ids, ref_ids)
        assert torch.equal(gates.view(torch.int32), ref_gates.view(torch.int32))


CASES = [CONFIGS["c1_tiny"],
         CONFIGS["c2_decode_replay"].with_(n_shared=0, F=64, name="decode_E384_T64"),
         CONFIGS["c2_decode_replay"].with_(T=T_MAX_E384, n_shared=0, F=64,
                                           name="decode_E384_Tmax"),
         CONFIGS["c1_tiny"].with_(T=1000, d=192, zipf=1.0, name="unsplit_d192_T1000")]


@pytest.mark.parametrize("cfg", CASES, ids=lambda c: c.name)
def test_static_routing_matches_workspace_routing(cfg):
    _compare(make_layer(cfg, "cuda"))


def test_static_routing_near_ties():
    # 8th and 9th logits within 1e-4 (exact arithmetic) on a quarter of the tokens
    cfg = CONFIGS["c2_decode_replay"].with_(T=256, n_shared=0, F=64, name="near_ties")
    inp = make_layer(cfg, "cuda")
    x_nt, idx, _, done = mc.make_near_ties(inp, 0.25, seed=11)
    assert done >= len(idx) // 2
    _compare(inp, x_nt)


def test_static_routing_rejects_too_many_tokens():
    cfg = CONFIGS["c1_tiny"].with_(T=T_MAX_E384 + 1, d=7168, E=384, F=64, name="too_big")
    inp = make_layer(cfg.with_(T=1), "cuda")
    x = torch.zeros((cfg.T, cfg.d), dtype=torch.bfloat16, device="cuda")
    layer = MoELayer.from_inputs(inp)
    ids = torch.empty((cfg.T, 8), dtype=torch.int32, device="cuda")
    gates = torch.empty((cfg.T, 8), dtype=torch.float32, device="cuda")
    rc = B.moe_route_static(layer.dims(cfg.T), x, layer.weights, ids, gates, check=False)
    assert rc == B.MOE_ERR_WORKSPACE
    # the largest size that fits is served
    rc = B.moe_route_static(layer.dims(T_MAX_E384), x[:T_MAX_E384], layer.weights, ids, gates,
                            check=False)
    torch.cuda.synchronize()
    assert rc == B.MOE_OK
