"""Parity of the full-size d=7168 layers against the fp64 oracle.

For the prefill-like layer (Zipf routing), the 32k-token layer (uniform and
Zipf s=1.2 routing) and the MXFP8 layer with 10 % adversarial near-tie tokens,
every token's router logits, ids, gate weights and the whole counting sort
(cnt, off, perm, inv) are checked against the oracle over the whole batch,
in own mode and (prefill, MXFP8) replay mode.  Layer outputs are compared on a
sample: the first 256 tokens, the tokens at the expert GEMMs' tile edges for
one expert of every size class (see moe_cases.boundary_tokens), tokens whose
GPU ids differ from the oracle's own choice (near ties), and near-tie tokens;
every sampled token is checked against the oracle in replay mode with the ids
the GPU used, so no token is dropped from the comparison."""
import numpy as np
import pytest
import torch

import oracle
from deterministic_rl_gb300 import build, MoELayer
from deterministic_rl_gb300.synthetic import CONFIGS, make_layer
import moe_cases as mc

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


@pytest.fixture(scope="module", autouse=True)
def _built():
    build.build()
    oracle.build()


FULL = [CONFIGS["c3_prefill_zipf"], CONFIGS["c4_train_32k"],
        CONFIGS["c4_train_32k"].with_(zipf=1.2, name="c4_train_32k_zipf1.2"),
        CONFIGS["c5_mxfp8"]]


def _inputs(cfg):
    inp = make_layer(cfg, "cuda")
    ties = np.zeros(0, np.int64)
    if cfg.near_tie_frac:
        x, ties, x_rep, done = mc.make_near_ties(inp, cfg.near_tie_frac, seed=cfg.seed)
        assert done == len(ties)
        inp.x, inp.x_replay_src = x, x_rep
    return inp, ties


def _sample(cfg, g_ids, same, sort, ties):
    cnt, off, perm = sort
    toks = set(range(min(256, cfg.T)))
    toks |= set(mc.boundary_tokens(cnt, off, perm, cfg.k))
    toks |= set(np.nonzero(~same)[0][:16].tolist())
    toks |= set(ties[:16].tolist())
    return sorted(toks)


@pytest.mark.parametrize("cfg", FULL, ids=lambda c: c.name)
def test_full_size_own_mode(cfg):
    inp, ties = _inputs(cfg)
    layer = MoELayer.from_inputs(inp, out_fp32=True)
    out, ids, gates = layer.forward(inp.x)
    torch.cuda.synchronize()
    assert layer.status() == 0
    _, g_ids, same, sort = mc.check_batch_routing(inp, inp.x, layer, ids, gates)
    assert same.mean() > 0.98 if not len(ties) else same.mean() > 0.85
    tokens = _sample(cfg, g_ids, same, sort, ties)
    rel, mx = mc.check_sampled_outputs(inp, inp.x, out, g_ids, tokens)
    print(f"{cfg.name} own: {cfg.T} tokens routed; ids equal to the oracle's own choice on "
          f"{same.mean():.4f}; {len(tokens)} sampled outputs rel Frobenius {rel:.2e} "
          f"max-abs {mx:.2e}")


@pytest.mark.parametrize("cfg", [FULL[0], FULL[3]], ids=lambda c: c.name)
def test_full_size_replay_mode(cfg):
    inp, ties = _inputs(cfg)
    rid = mc.oracle_replay_ids(inp)  # the oracle's routing of the perturbed copy
    layer = MoELayer.from_inputs(inp, out_fp32=True)
    out, ids, gates = layer.forward(inp.x, replay_ids=torch.from_numpy(rid).cuda())
    torch.cuda.synchronize()
    assert layer.status() == 0
    _, g_ids, same, sort = mc.check_batch_routing(inp, inp.x, layer, ids, gates, replay_ids=rid)
    tokens = _sample(cfg, g_ids, same, sort, ties)
    rel, mx = mc.check_sampled_outputs(inp, inp.x, out, g_ids, tokens)
    print(f"{cfg.name} replay: recorded ids equal the own choice on {same.mean():.4f}; "
          f"{len(tokens)} sampled outputs rel Frobenius {rel:.2e} max-abs {mx:.2e}")
