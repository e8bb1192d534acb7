"""The expert GEMMs run on the one-SM kernel for small batches and on SM pairs
for large ones.  Batch invariance across that switch needs the two kernel
families to produce the same bits for the same token: both put weights on the
MMA's M side and tokens on N and accumulate bf16 K=16 MMAs in K order into fp32
TMEM.  These tests check it on hardware, directly (a small sub-batch against
the same rows inside a large batch) and with each family forced for the whole
layer (MOE_EXPERT_KERNEL, read once per process, so each run is a subprocess)."""
import os
import subprocess
import sys

import pytest
import torch

from deterministic_rl_gb300 import build, MoELayer
from deterministic_rl_gb300.synthetic import CONFIGS, make_layer

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def _built():
    build.build()


def _cfg(T, **kw):
    base = dict(name=f"fam_T{T}", seed=31, T=T, d=512, E=48, F=384, n_shared=1)
    base.update(kw)
    return CONFIGS["c1_tiny"].with_(**base)


@pytest.mark.parametrize("T_full,T_part", [(1000, 100), (1000, 128), (4096, 64), (300, 1)])
def test_small_sub_batch_equals_rows_of_large_batch(T_full, T_part):
    inp = make_layer(_cfg(T_full), "cuda")
    layer = MoELayer.from_inputs(inp, out_fp32=True)
    full = [t.clone() for t in layer.forward(inp.x)]          # SM-pair kernels
    part = layer.forward(inp.x[:T_part].contiguous())         # one-SM kernels
    for a, b in zip(full, part):
        assert torch.equal(a[:T_part], b)


def test_decode_layer_rows_match_inside_prefill_batch():
    cfg = CONFIGS["c2_decode_replay"].with_(T=1024, E=96, name="decode_in_prefill")
    inp = make_layer(cfg, "cuda")
    layer = MoELayer.from_inputs(inp, out_fp32=True)
    full = [t.clone() for t in layer.forward(inp.x)]
    part = layer.forward(inp.x[-64:].contiguous())
    for a, b in zip(full, part):
        assert torch.equal(a[-64:], b)


_SCRIPT = r"""
import sys, torch
sys.path.insert(0, {root!r})
from deterministic_rl_gb300 import MoELayer
from deterministic_rl_gb300.synthetic import CONFIGS, make_layer
cfg = CONFIGS["c1_tiny"].with_(name="x", seed={seed}, T={T}, d=512, E=48, F=384, n_shared={S}, zipf={zipf})
inp = make_layer(cfg, "cuda")
out, ids, gates = MoELayer.from_inputs(inp, out_fp32=True).forward(inp.x)
torch.save([out.cpu(), ids.cpu(), gates.cpu()], {path!r})
"""


@pytest.mark.parametrize("T,S,zipf", [(64, 1, 0.0), (700, 0, 1.0), (2000, 1, 0.0)])
def test_forced_kernel_families_agree_bitwise(tmp_path, T, S, zipf):
    res = {}
    for fam in ("one_sm", "pair"):
        path = str(tmp_path / f"{fam}.pt")
        env = dict(os.environ, MOE_EXPERT_KERNEL=fam)
        code = _SCRIPT.format(root=ROOT, seed=7 + T, T=T, S=S, zipf=zipf, path=path)
        subprocess.run([sys.executable, "-c", code], env=env, check=True, timeout=300)
        res[fam] = torch.load(path)
    for a, b in zip(res["one_sm"], res["pair"]):
        assert torch.equal(a, b)


@pytest.mark.parametrize("c", [1, 63, 64, 65, 128, 129, 192, 193, 255, 256, 257])
def test_pair_tile_width_does_not_change_a_token(c):
    """The SM-pair kernel issues a tile's MMAs with N = its token count rounded
    up to 64.  Expert 0 gets the first c tokens (its tile N runs through 64,
    128, 192, 256 and a second tile); every other expert's group is the same in
    all runs.  Token 0's output and every other token's routed outputs must not
    change with c."""
    T = 300
    inp = make_layer(_cfg(T, name="width", seed=13), "cuda")
    layer = MoELayer.from_inputs(inp, out_fp32=True)
    ids = torch.empty((T, 8), dtype=torch.int32)
    ids[:, 1:] = torch.arange(1, 8, dtype=torch.int32)
    ids[:, 0] = 8 + torch.arange(T, dtype=torch.int32) % 40
    base = [t.clone() for t in layer.forward(inp.x, replay_ids=ids.cuda())]
    ids[:c, 0] = 0
    out, _, _ = layer.forward(inp.x, replay_ids=ids.cuda())
    # tokens c.. route exactly as in the base run except that their slot-0
    # groups lost tokens 0..c-1: still the same columns-independent results
    assert torch.equal(out[c:], base[0][c:])
    ids2 = ids.clone()
    ids2[1:, 0] = 8 + torch.arange(1, T, dtype=torch.int32) % 40
    single, _, _ = layer.forward(inp.x, replay_ids=ids2.cuda())   # expert 0: token 0 alone
    assert torch.equal(out[0], single[0])
