"""The NVFP4 forward with per-token scales (Composer 2 Technical Report, §6.1,
Kernels: BF16 values quantised to FP4 E2M1 with an FP8 E4M3 scale per 16 and
an FP32 scale per token, IEEE division in the quantiser; block-scaled
tensor-core matmul) on the GPU:
  * the token-row quantiser, bitwise against the oracle's (both take their
    rounding decisions on the same fp32 quotients): codes, block scales and
    row scales, of x and of h;
  * the layer against the oracle (which quantises its own h, rounded to bf16,
    the same way);
  * batch invariance, bitwise: a token's scales depend on that token only."""
import numpy as np
import pytest
import torch

import oracle
from deterministic_rl_gb300 import build, MoELayer
from deterministic_rl_gb300 import binding as B
from deterministic_rl_gb300.synthetic import CONFIGS, bf16_bits, make_layer
import moe_cases as mc

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    build.build()
    oracle.build()


def small_nv(T=300, E=32, seed=51):
    return CONFIGS["c6_nvfp4"].with_(name=f"nv_T{T}", seed=seed, T=T, d=512, E=E, F=512)


def _expect_quantised(x_bf16: torch.Tensor):
    """The oracle's quantisation of bf16 rows: (codes [R][K] 0..15, E4M3 block
    scales [R][K/16], fp32 row scales [R])."""
    xf = torch.from_numpy(bf16_bits(x_bf16).view(np.int16)).view(torch.bfloat16).float().numpy()
    return oracle.nvfp4_quantize_rows(xf)


def _unpack(packed: torch.Tensor) -> np.ndarray:
    """Packed bytes [R][K/2] -> codes [R][K] (element 2j in the low nibble)."""
    b = packed.cpu().numpy()
    out = np.empty((b.shape[0], 2 * b.shape[1]), np.uint8)
    out[:, 0::2] = b & 15
    out[:, 1::2] = b >> 4
    return out


@pytest.mark.parametrize("T", [1, 37, 300])
def test_token_quantiser_bitwise_against_oracle(T):
    inp = make_layer(small_nv(T), "cuda")
    # rows of very different magnitudes, an all-zero row, a row with an all-zero block
    x = inp.x.float() * torch.logspace(-4, 4, T, device="cuda").unsqueeze(1)
    if T > 1:
        x[0, :] = 0
    if T > 2:
        x[2, 32:48] = 0
    x = x.to(torch.bfloat16).contiguous()
    layer = MoELayer.from_inputs(inp, out_fp32=True)
    layer.forward(x)
    assert layer.status() == B.MOE_OK
    im = layer.intermediates(T)
    codes, bs, rs = _expect_quantised(x)
    assert np.array_equal(_unpack(im["x4"]), codes)
    assert np.array_equal(im["xb"].cpu().numpy(), bs)
    assert np.array_equal(im["sx"].cpu().numpy(), rs)


def test_gathered_rows_carry_their_token_scale():
    inp = make_layer(small_nv(200), "cuda")
    layer = MoELayer.from_inputs(inp, out_fp32=True)
    _, ids, _ = layer.forward(inp.x)
    im = layer.intermediates(200)
    perm = im["perm"].long()
    tok = perm // 8
    assert torch.equal(im["sxp"], im["sx"][tok])
    assert torch.equal(im["xp4"], im["x4"][tok])
    assert torch.equal(im["xpb"], im["xb"][tok])


def test_activation_rows_quantised_like_the_oracle():
    """Each row of h (the bf16 SwiGLU output) is quantised like the oracle
    quantises it: codes, block scales and row scales bitwise."""
    inp = make_layer(small_nv(64), "cuda")
    layer = MoELayer.from_inputs(inp, out_fp32=True)
    layer.forward(inp.x)
    im = layer.intermediates(64)
    codes, bs, rs = _expect_quantised(im["h"])
    assert np.array_equal(_unpack(im["h4"]), codes)
    assert np.array_equal(im["hb"].cpu().numpy(), bs)
    assert np.array_equal(im["sh"].cpu().numpy(), rs)
    assert (rs > 0).mean() > 0.99


@pytest.mark.parametrize("T,E", [(1, 16), (130, 32), (300, 32)])
def test_nvfp4_layer_matches_oracle(T, E):
    inp = make_layer(small_nv(T, E), "cuda")
    layer = MoELayer.from_inputs(inp, out_fp32=True)
    out, ids, gates = layer.forward(inp.x)
    assert layer.status() == B.MOE_OK
    ref = mc.oracle_layer(inp)
    g_ids = ids.cpu().numpy()
    ok = mc.check_ids(g_ids, ref.logits, 8)
    ref_r = mc.oracle_layer(inp, replay_ids=g_ids) if not ok.all() else ref
    mc.check_gates(gates.cpu().numpy(), ref_r.gates)
    mc.check_out(out.cpu().numpy(), ref_r.out)


def test_nvfp4_batch_invariance_and_determinism():
    inp = make_layer(small_nv(1000, seed=53), "cuda")
    layer = MoELayer.from_inputs(inp, out_fp32=True)
    full = [t.clone() for t in layer.forward(inp.x)]
    again = layer.forward(inp.x)
    for a, b in zip(full, again):
        assert torch.equal(a, b)
    for lo, hi in ((0, 1), (0, 130), (500, 1000), (17, 40)):
        part = layer.forward(inp.x[lo:hi].contiguous())
        for a, b in zip(full, part):
            assert torch.equal(a[lo:hi], b)


def test_nvfp4_rejects_shared_expert_and_missing_scales():
    inp = make_layer(small_nv(8), "cuda")
    layer = MoELayer.from_inputs(inp)
    out, ids, gates = layer.outputs(8)
    dims = layer.dims(8)
    dims.n_shared = 1
    sh = torch.zeros((512, 512), dtype=torch.bfloat16, device="cuda")
    w = B.make_weights(inp.w_router, None, inp.w_gate, inp.w_up, inp.w_down, inp.s_gate,
                       inp.s_up, inp.s_down, sh, sh, sh, inp.gs_gate, inp.gs_up, inp.gs_down)
    ws = torch.empty(B.moe_workspace_size(dims), dtype=torch.uint8, device="cuda")
    assert B.moe_forward(dims, inp.x, w, out, ids, gates, ws, check=False) == B.MOE_ERR_UNSUPPORTED
    w2 = B.make_weights(inp.w_router, None, inp.w_gate, inp.w_up, inp.w_down, inp.s_gate,
                        inp.s_up, inp.s_down)
    assert B.moe_forward(layer.dims(8), inp.x, w2, out, ids, gates, layer.workspace(8),
                         check=False) == B.MOE_ERR_ARG


def test_nvfp4_full_size_sampled_parity_and_invariance():
    """The 16,384-token NVFP4 layer (d=7168, E=384, F=2048): a 512-token
    sub-batch gives its rows bitwise, the token quantiser matches the oracle
    on sampled rows bitwise, and sampled tokens match the oracle layer."""
    cfg = CONFIGS["c6_nvfp4"]
    inp = make_layer(cfg, "cuda")
    layer = MoELayer.from_inputs(inp, out_fp32=True)
    out, ids, gates = [t.clone() for t in layer.forward(inp.x)]
    assert layer.status() == B.MOE_OK
    im = layer.intermediates(cfg.T)
    tk = np.array([0, 1, 777, 8191, 16383])
    sel = torch.as_tensor(tk, device="cuda")
    codes, bs, rs = _expect_quantised(inp.x[sel])
    assert np.array_equal(_unpack(im["x4"][sel]), codes)
    assert np.array_equal(im["xb"][sel].cpu().numpy(), bs)
    assert np.array_equal(im["sx"].cpu().numpy()[tk], rs)
    part = MoELayer.from_inputs(inp, out_fp32=True).forward(inp.x[:512].contiguous())
    for a, b in zip((out, ids, gates), part):
        assert torch.equal(a[:512], b)
    ref = mc.oracle_layer(inp, tokens=tk)
    same = mc.check_ids(ids.cpu().numpy()[tk], ref.logits, 8)
    mc.check_out(out.cpu().numpy()[tk][same], ref.out[same])
