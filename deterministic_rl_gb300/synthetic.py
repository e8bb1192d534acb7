"""Seeded synthetic inputs for the MoE layer (the workloads' shapes and value
distributions).  This module draws random numbers and encodes them into the
storage formats the layer reads (bf16 rounding, MXFP8 block quantisation of
the weights); it holds none of the layer's arithmetic -- no logits, no
selection, no expert FFN, no combine.  Both the CUDA path's tests and the
oracle consume the bytes it produces.  NVFP4 is the forward format of the
Composer 2 Technical Report, §6.1 (E2M1 values, E4M3 scale per 16, fp32 scale).

Workloads (hidden size, expert count, top-k, expert width, shared expert, value
distributions, seeds):
  c1_tiny          T=128,   d=512,  E=64,  k=8, F=256,  no shared expert
  c2_decode_replay T=64,    d=7168, E=384, k=8, F=2048, 1 shared expert
  c3_prefill_zipf  T=4096,  same layer, router bias -1.0*ln(rank_e)
  c4_train_32k     T=32768, same layer, uniform or Zipf (s=1.2) routing
  c5_mxfp8         T=16384, expert weights MXFP8 (E4M3 + E8M0 per 32 along K),
                   no shared expert, 10 % of tokens near-tied at ranks 8/9
  c6_nvfp4         T=16384, expert weights NVFP4 (E2M1 + E4M3 per 16 along K +
                   an fp32 scale per matrix), no shared expert
Hidden states ~N(0,1); router ~N(0, variance 1/d); expert weights
~N(0, std 0.02); replay ids are recorded from a copy of the hidden states
perturbed by N(0, std 1e-3).  The 384-choose-8 gate is from the Training Data
No. 94 write-up, section "浮点数不守规矩，MoE 火上浇油"; MXFP8 is the format of
the Composer 2 Technical Report, §6.1 (E4M3 values, E8M0 scale per 32).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, replace
from typing import Optional

import torch


@dataclass(frozen=True)
class MoEConfig:
    name: str
    seed: int
    T: int
    d: int
    E: int
    k: int
    F: int
    n_shared: int
    wfmt: str = "bf16"            # "bf16" | "mxfp8" | "nvfp4"
    zipf: float = 0.0             # bias = -zipf * ln(rank_e); 0 = no bias
    near_tie_frac: float = 0.0    # fraction of tokens to near-tie (built in tests)
    replay_noise: float = 1e-3    # std of the perturbation replay ids come from
    w_std: float = 0.02
    act_mx: bool = False          # MXFP8 weights: activations quantised to MXFP8 too

    def with_(self, **kw) -> "MoEConfig":
        return replace(self, **kw)


CONFIGS = {
    "c1_tiny": MoEConfig("c1_tiny", 0, 128, 512, 64, 8, 256, 0),
    "c2_decode_replay": MoEConfig("c2_decode_replay", 1, 64, 7168, 384, 8, 2048, 1),
    "c3_prefill_zipf": MoEConfig("c3_prefill_zipf", 2, 4096, 7168, 384, 8, 2048, 1, zipf=1.0),
    "c4_train_32k": MoEConfig("c4_train_32k", 3, 32768, 7168, 384, 8, 2048, 1),
    "c5_mxfp8": MoEConfig("c5_mxfp8", 4, 16384, 7168, 384, 8, 2048, 0, wfmt="mxfp8",
                          near_tie_frac=0.1),
    "c6_nvfp4": MoEConfig("c6_nvfp4", 5, 16384, 7168, 384, 8, 2048, 0, wfmt="nvfp4"),
    # the MXFP8 layer with MXFP8 activations as well (same seed, same weights)
    "c5_mxfp8_act": MoEConfig("c5_mxfp8_act", 4, 16384, 7168, 384, 8, 2048, 0, wfmt="mxfp8",
                              near_tie_frac=0.1, act_mx=True),
}


@dataclass
class LayerInputs:
    cfg: MoEConfig
    x: torch.Tensor                      # [T][d] bf16
    x_replay_src: torch.Tensor           # [T][d] bf16, x + N(0, noise) rounded
    w_router: torch.Tensor               # [E][d] bf16
    router_bias: Optional[torch.Tensor]  # [E] fp32
    w_gate: torch.Tensor                 # [E][F][d] bf16 | uint8 (E4M3) | [E][F][d/2] uint8 (E2M1 x2)
    w_up: torch.Tensor                   # [E][F][d]
    w_down: torch.Tensor                 # [E][d][F]
    s_gate: Optional[torch.Tensor]       # [E][F][d/32] uint8 (E8M0) | [E][F][d/16] (E4M3) | None
    s_up: Optional[torch.Tensor]
    s_down: Optional[torch.Tensor]       # [E][d][F/32] | [E][d][F/16]
    ws_gate: Optional[torch.Tensor]      # [F][d] bf16 shared expert
    ws_up: Optional[torch.Tensor]
    ws_down: Optional[torch.Tensor]      # [d][F]
    gs_gate: Optional[torch.Tensor] = None   # NVFP4: [E] fp32 scale per matrix
    gs_up: Optional[torch.Tensor] = None
    gs_down: Optional[torch.Tensor] = None


def _randn(shape, std, gen, device) -> torch.Tensor:
    return torch.randn(shape, generator=gen, device=device, dtype=torch.float32) * std


def quantize_mxfp8(w: torch.Tensor):
    """Encode fp32 [rows][K] as MXFP8 (OCP MX v1.0 reading): per 32-element
    block along K, shared exponent e = floor(log2(max|v|)) - 8 (E4M3's largest
    exponent), scale byte e + 127, element byte = E4M3(v * 2^-e) with round to
    nearest even after saturation to +-448.  An all-zero block gets scale 2^0.
    Returns (values uint8 [rows][K], scales uint8 [rows][K/32])."""
    rows, K = w.shape
    assert K % 32 == 0
    blocks = w.reshape(rows, K // 32, 32)
    amax = blocks.abs().amax(dim=-1)
    _, ex = torch.frexp(amax)                     # amax = m * 2^ex, m in [0.5, 1)
    e = (ex.to(torch.int32) - 1) - 8
    e = torch.where(amax == 0, torch.zeros_like(e), e).clamp(-127, 127)
    scaled = torch.ldexp(blocks, (-e).to(torch.float32).unsqueeze(-1))
    q = scaled.clamp(-448.0, 448.0).to(torch.float8_e4m3fn).view(torch.uint8)
    s = (e + 127).to(torch.uint8)
    return q.reshape(rows, K).contiguous(), s.contiguous()


def quantize_nvfp4(w: torch.Tensor):
    """Encode fp32 [rows][K] as NVFP4 weights: one fp32 scale for the matrix,
    ts = amax / (6 * 448); per 16-element block along K an E4M3 scale
    S = E4M3(amax_b / 6 / ts) (nearest even, saturating); values
    E2M1(w / (S * ts)) rounded to nearest with ties to the even code, packed two
    per byte (element 2j in the low nibble).  Returns (packed uint8
    [rows][K/2], scales uint8 [rows][K/16], ts as a 0-d float32 tensor)."""
    rows, K = w.shape
    assert K % 16 == 0
    w = w.float()
    ts = w.abs().max() / 2688.0
    blocks = w.reshape(rows, K // 16, 16)
    bmax = blocks.abs().amax(dim=-1)
    if float(ts) > 0:
        S = ((bmax / 6.0) / ts).to(torch.float8_e4m3fn)
    else:
        S = torch.zeros_like(bmax).to(torch.float8_e4m3fn)
    denom = (S.float() * ts).unsqueeze(-1)
    v = torch.where(denom > 0, blocks / torch.where(denom > 0, denom, torch.ones_like(denom)),
                    torch.zeros_like(blocks))
    a = v.abs()
    m = ((a > 0.25).int() + (a >= 0.75).int() + (a > 1.25).int() + (a >= 1.75).int()
         + (a > 2.5).int() + (a >= 3.5).int() + (a > 5.0).int())
    code = m | (((v < 0) & (m > 0)).int() << 3)
    code = code.reshape(rows, K).to(torch.uint8)
    packed = (code[:, 0::2] | (code[:, 1::2] << 4)).contiguous()
    return packed, S.view(torch.uint8).contiguous(), ts.to(torch.float32)


def make_layer(cfg: MoEConfig, device="cpu") -> LayerInputs:
    """Draw every tensor of the layer from one generator seeded with cfg.seed,
    in a fixed order: x, router, per expert (gate, up, down), shared expert,
    bias rank permutation, replay noise."""
    device = torch.device(device)
    gen = torch.Generator(device=device)
    gen.manual_seed(cfg.seed)
    T, d, E, F = cfg.T, cfg.d, cfg.E, cfg.F
    bf = torch.bfloat16

    x = _randn((T, d), 1.0, gen, device).to(bf)
    w_router = _randn((E, d), 1.0 / math.sqrt(d), gen, device).to(bf)

    mx = cfg.wfmt == "mxfp8"
    nv = cfg.wfmt == "nvfp4"
    u8 = torch.uint8
    if nv:
        w_gate = torch.empty((E, F, d // 2), dtype=u8, device=device)
        w_up = torch.empty((E, F, d // 2), dtype=u8, device=device)
        w_down = torch.empty((E, d, F // 2), dtype=u8, device=device)
        s_gate = torch.empty((E, F, d // 16), dtype=u8, device=device)
        s_up = torch.empty((E, F, d // 16), dtype=u8, device=device)
        s_down = torch.empty((E, d, F // 16), dtype=u8, device=device)
        gs = [torch.empty(E, dtype=torch.float32, device=device) for _ in range(3)]
    else:
        wdt = u8 if mx else bf
        w_gate = torch.empty((E, F, d), dtype=wdt, device=device)
        w_up = torch.empty((E, F, d), dtype=wdt, device=device)
        w_down = torch.empty((E, d, F), dtype=wdt, device=device)
        s_gate = torch.empty((E, F, d // 32), dtype=u8, device=device) if mx else None
        s_up = torch.empty((E, F, d // 32), dtype=u8, device=device) if mx else None
        s_down = torch.empty((E, d, F // 32), dtype=u8, device=device) if mx else None
        gs = [None, None, None]
    for e in range(E):
        for j, (dst, sdst, shape) in enumerate(((w_gate, s_gate, (F, d)), (w_up, s_up, (F, d)),
                                                (w_down, s_down, (d, F)))):
            w = _randn(shape, cfg.w_std, gen, device)
            if mx:
                q, s = quantize_mxfp8(w)
                dst[e].copy_(q)
                sdst[e].copy_(s)
            elif nv:
                q, s, ts = quantize_nvfp4(w)
                dst[e].copy_(q)
                sdst[e].copy_(s)
                gs[j][e] = ts
            else:
                dst[e].copy_(w.to(bf))

    ws_gate = ws_up = ws_down = None
    if cfg.n_shared:
        assert cfg.n_shared == 1
        ws_gate = _randn((F, d), cfg.w_std, gen, device).to(bf)
        ws_up = _randn((F, d), cfg.w_std, gen, device).to(bf)
        ws_down = _randn((d, F), cfg.w_std, gen, device).to(bf)

    bias = None
    if cfg.zipf:
        rank = torch.randperm(E, generator=gen, device=device).to(torch.float64) + 1.0
        bias = (-cfg.zipf * torch.log(rank)).to(torch.float32)

    noise = _randn((T, d), cfg.replay_noise, gen, device)
    x_replay_src = (x.float() + noise).to(bf)

    return LayerInputs(cfg, x, x_replay_src, w_router, bias, w_gate, w_up, w_down,
                       s_gate, s_up, s_down, ws_gate, ws_up, ws_down, gs[0], gs[1], gs[2])


def make_dout(cfg: MoEConfig, T: Optional[int] = None, device="cpu") -> torch.Tensor:
    """The upstream gradient of the layer output for the backward: N(0, 1)
    rounded to bf16, [T][d], from its own generator (seed cfg.seed + 7919)."""
    device = torch.device(device)
    gen = torch.Generator(device=device)
    gen.manual_seed(cfg.seed + 7919)
    T = cfg.T if T is None else T
    return _randn((T, cfg.d), 1.0, gen, device).to(torch.bfloat16)


def make_replay_ids(cfg: MoEConfig, T: Optional[int] = None, device="cpu") -> torch.Tensor:
    """Recorded expert ids for replay: per token k distinct experts drawn
    without replacement, with probability proportional to (e + 1)^-zipf
    (uniform when cfg.zipf == 0), [T][k] int32, from their own generator
    (seed cfg.seed + 104729)."""
    gen = torch.Generator()
    gen.manual_seed(cfg.seed + 104729)
    T = cfg.T if T is None else T
    p = (torch.arange(cfg.E, dtype=torch.float64) + 1.0) ** (-cfg.zipf)
    ids = torch.multinomial(p.expand(T, cfg.E), cfg.k, replacement=False, generator=gen)
    return ids.to(torch.int32).to(device)


def bf16_bits(t: torch.Tensor):
    """bf16 tensor -> numpy uint16 bit patterns (host copy)."""
    import numpy as np
    assert t.dtype == torch.bfloat16
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def u8(t: torch.Tensor):
    return t.detach().contiguous().cpu().numpy()
