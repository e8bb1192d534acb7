"""moe_route_static -- routing for callers that cannot allocate device memory
(for example an inference engine whose device memory all belongs to its own
pool, recording routing decisions inside its decode loop): the scratch lives in
a static device array of the library instead of a caller workspace.

Checked through the C ABI against moe_route (which takes a workspace) on the
same inputs, on two calls in a row, with the same rules the other tests use:
ids equal, gate weights within the gate tolerance.  This file sorts last so
that a run stopping at the first failure has already run every other test; it
also passes on its own in a fresh process (the static array's address is set
up by its first call)."""
import numpy as np
import pytest
import torch

from deterministic_rl_gb300 import build, MoELayer
from deterministic_rl_gb300 import binding as B
from deterministic_rl_gb300.synthetic import CONFIGS, make_layer
import moe_cases as mc

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    build.build()


@pytest.mark.parametrize("cfg", [CONFIGS["c1_tiny"],
                                 CONFIGS["c2_decode_replay"].with_(E=64, name="decode_E64"),
                                 CONFIGS["c1_tiny"].with_(T=1000, zipf=1.0, name="tiny_T1000")],
                         ids=lambda c: c.name)
def test_static_routing_matches_workspace_routing(cfg):
    inp = make_layer(cfg, "cuda")
    layer = MoELayer.from_inputs(inp)
    ref_ids, ref_gates = layer.route(inp.x)
    torch.cuda.synchronize()
    dims = layer.dims(cfg.T)
    for _ in range(2):  # two calls in a row share the static scratch
        ids = torch.full_like(ref_ids, -7)
        gates = torch.full_like(ref_gates, -1.0)
        B.moe_route_static(dims, inp.x, layer.weights, ids, gates)
        torch.cuda.synchronize()
        assert torch.equal(ids, ref_ids)
        mc.check_gates(gates.cpu().numpy(), ref_gates.cpu().numpy().astype(np.float64))


def test_static_routing_rejects_too_many_tokens():
    cfg = CONFIGS["c1_tiny"].with_(T=2724, d=256, E=384, F=128, name="too_big")
    inp = make_layer(cfg.with_(T=1), "cuda")
    x = torch.zeros((cfg.T, cfg.d), dtype=torch.bfloat16, device="cuda")
    layer = MoELayer.from_inputs(inp)
    ids = torch.empty((cfg.T, 8), dtype=torch.int32, device="cuda")
    gates = torch.empty((cfg.T, 8), dtype=torch.float32, device="cuda")
    rc = B.moe_route_static(layer.dims(cfg.T), x, layer.weights, ids, gates, check=False)
    assert rc == B.MOE_ERR_WORKSPACE
    # the largest size that fits is served
    rc = B.moe_route_static(layer.dims(2723), x[:2723], layer.weights, ids, gates, check=False)
    torch.cuda.synchronize()
    assert rc == B.MOE_OK
