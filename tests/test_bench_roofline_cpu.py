"""The roofline arithmetic bench.py reports, against closed forms written out
independently here.

Layer FLOPs are T (2 d E + 6 d F (k + S)): the router GEMM plus the three
expert projections of k routed slots and S shared experts. The bytes are the
touched experts' weights read once plus the router, x, out and the ids/gates
traffic. Expert weight bytes are 3 d F per value: 2 B in bf16, 1 + 1/32 in
MXFP8 (E4M3 plus an E8M0 scale per 32). The kernel launch counts per call are
those of the launch lists under profiles/."""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from deterministic_rl_gb300.synthetic import CONFIGS  # noqa: E402

D, F, E, K = 7168, 2048, 384, 8


def test_expert_weight_bytes():
    bf16 = bench.weight_bytes_per_value(CONFIGS["c4_train_32k"]) * 3 * D * F
    mx = bench.weight_bytes_per_value(CONFIGS["c5_mxfp8"]) * 3 * D * F
    assert bf16 == 88_080_384                  # 3 * 7168 * 2048 * 2
    assert mx == pytest.approx(45_416_448)     # 3 * 7168 * 2048 * (1 + 1/32)


@pytest.mark.parametrize("name,T,S,tflop", [
    # each workload's FLOPs to three or four significant digits
    ("c2_decode_replay", 64, 1, 0.0511),
    ("c3_prefill_zipf", 4096, 1, 3.27),
    ("c4_train_32k", 32768, 1, 26.16),
    ("c5_mxfp8", 16384, 0, 11.64),
])
def test_layer_flops(name, T, S, tflop):
    router = 2 * D * E          # per token
    experts = 3 * 2 * D * F     # per token and expert: gate, up, down
    flops, _ = bench.layer_work(CONFIGS[name], E)
    assert flops == T * (router + experts * (K + S))
    assert flops == pytest.approx(tflop * 1e12, rel=2e-3)


def test_layer_bytes_32k_all_touched():
    cfg = CONFIGS["c4_train_32k"]
    T = cfg.T
    expected = (E + 1) * 3 * D * F * 2 + E * D * 2 + 2 * T * D * 2 + T * K * 12
    _, nbytes = bench.layer_work(cfg, E)
    assert nbytes == expected == 34_859_122_688


def test_roofline_bound_switches_with_the_batch():
    """At the measured peaks the decode layer is HBM-bound and the 32k layer
    tensor-bound (ridge point ~290 FLOP per byte)."""
    tensor, hbm = 1958.8e12, 6761.6e9
    for name, bound in (("c2_decode_replay", "hbm"), ("c4_train_32k", "tensor")):
        flops, nbytes = bench.layer_work(CONFIGS[name], E)
        assert ("tensor" if flops / tensor > nbytes / hbm else "hbm") == bound


@pytest.mark.parametrize("name,launches", [
    ("c1_tiny", 7),            # one-kernel dispatch (<= 4096 pairs), one-SM GEMMs
    ("c2_decode_replay", 7),
    ("c3_prefill_zipf", 10),   # histogram, scan, scatter; shared gate/up on its own stream
    ("c4_train_32k", 10),
    ("c5_mxfp8", 9),           # no shared expert
    ("c5_mxfp8_act", 10),      # quantise-and-gather for x, + the quantiser of h
    ("c6_nvfp4", 10),
])
def test_forward_launches_per_call(name, launches):
    assert bench.launches_per_step(CONFIGS[name]) == launches


def test_backward_launches_per_call():
    cfg = CONFIGS["c4_train_32k"]
    assert bench.backward_launches(cfg) == 28
    assert bench.backward_launches(cfg, train=True) == 29


def test_block_scaled_peaks_and_row_bytes():
    """The expert GEMMs' tensor peak follows their operand type (the measured
    bf16 peak times the nominal dense ratio: fp8 2x, fp4 6x; MXFP8 weights with
    bf16 activations are dequantised and run at the bf16 rate), and the token
    rows they read are counted at their stored size."""
    bf = 1958.8
    assert bench.mma_peak(CONFIGS["c4_train_32k"], bf)[0] == bf
    assert bench.mma_peak(CONFIGS["c5_mxfp8"], bf)[0] == bf
    assert bench.mma_peak(CONFIGS["c5_mxfp8_act"], bf)[0] == 2 * bf
    assert bench.mma_peak(CONFIGS["c6_nvfp4"], bf)[0] == 6 * bf
    assert bench.act_bytes_per_value(CONFIGS["c5_mxfp8"]) == 2.0
    assert bench.act_bytes_per_value(CONFIGS["c5_mxfp8_act"]) == 1 + 1 / 32
    assert bench.act_bytes_per_value(CONFIGS["c6_nvfp4"]) == 0.5 + 1 / 16
    # gate/up bytes of the NVFP4 layer: 384 experts' E2M1 + E4M3 weights, the
    # gathered narrow rows, the bf16 h written
    cfg = CONFIGS["c6_nvfp4"]
    T, d, F, k = cfg.T, cfg.d, cfg.F, cfg.k
    want = 384 * 2 * F * d * (0.5 + 1 / 16) + T * k * d * (0.5 + 1 / 16) + T * k * F * 2
    assert abs(bench.gate_up_bytes(cfg, 384) - want) < 1.0


def test_backward_roofline_takes_each_gemm_at_its_own_peak():
    """dH and dXp run on the block-scaled MXFP8 MMA and are measured against the
    fp8 peak (2x the measured bf16 figure); the weight-gradient GEMMs and the
    forward recompute against bf16; the layer's tensor time sums the grouped
    GEMMs at their peaks plus the router and gate work at bf16."""
    cfg = CONFIGS["c4_train_32k"]
    T, d, k, F, S = cfg.T, cfg.d, cfg.k, cfg.F, cfg.n_shared
    rows = T * k + T * S
    pk = {"hbm_gbs": 6761.6, "bf16_tflops": 1958.8, "bf16_tflops_sustained": 1730.0}
    ms = {"gate_up": 11.97, "down": 5.13, "dh": 3.82, "dxp": 7.98, "wgrad_down": 7.21,
          "wgrad_gate_up": 13.73}
    kernels, roof, layer = bench.backward_roofline(cfg, ms, 70.3, pk, "measured")
    bf, f8 = 1958.8, 2 * 1958.8
    assert kernels["dh"]["peak_tflops"] == f8 and kernels["dxp"]["peak_tflops"] == f8
    for n in ("gate_up", "down", "wgrad_down", "wgrad_gate_up"):
        assert kernels[n]["peak_tflops"] == bf
    assert kernels["dh"]["frac"] == pytest.approx(2 * d * F * rows / 3.82e-3 / 1e12 / f8)
    assert kernels["dxp"]["frac"] == pytest.approx(4 * d * F * rows / 7.98e-3 / 1e12 / f8)
    # the dominant kernel is the longest stage: dWg/dWu, at the bf16 peak
    assert roof["kernel"].startswith("wgrad_kernel (dWg") and roof["peak"] == bf
    assert roof["frac"] == pytest.approx(4 * d * F * rows / 13.73e-3 / 1e12 / bf)
    flops, _ = bench.backward_work(cfg)
    kf = bench.backward_kernel_flops(cfg)
    t = (sum(kf.values()) - kf["dh"] - kf["dxp"]) / bf + (kf["dh"] + kf["dxp"]) / f8
    t += (flops - sum(kf.values())) / bf
    assert layer["bound"] == "tensor"
    assert layer["roofline_ms"] == pytest.approx(t / 1e9)
    assert layer["frac"] == pytest.approx(t / 1e9 / 70.3)
    # a block-scaled stage that dominates is quoted against the fp8 peak
    _, roof2, _ = bench.backward_roofline(cfg, dict(ms, dxp=20.0), 80.0, pk, "measured")
    assert roof2["peak"] == f8 and "x 2" in roof2["peak_source"]
