"""The layer call is stream-ordered: it can be captured in a CUDA graph and
replayed, and calls on different streams run concurrently, with the same bits
as plain eager calls (including the SM-pair path whose shared expert runs on
the library's second stream)."""
import pytest
import torch

from deterministic_rl_gb300 import build, MoELayer
from deterministic_rl_gb300.synthetic import CONFIGS, make_layer

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    build.build()


def _cfg(T, seed):
    return CONFIGS["c1_tiny"].with_(name=f"sg_T{T}", seed=seed, T=T, d=512, E=48, F=384, n_shared=1)


@pytest.mark.parametrize("T", [64, 700])
def test_graph_capture_replays_bitwise(T):
    inp = make_layer(_cfg(T, 61), "cuda")
    layer = MoELayer.from_inputs(inp, out_fp32=True)
    ref = [t.clone() for t in layer.forward(inp.x)]
    x_static = inp.x.clone()
    outs = layer.outputs(T)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):  # warm-up on the capture stream
        layer.forward(x_static, outputs=outs, stream=s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        layer.forward(x_static, outputs=outs, stream=s)
    for o in outs:
        o.zero_()
    g.replay()
    torch.cuda.synchronize()
    for a, b in zip(ref, outs):
        assert torch.equal(a, b)
    # new inputs through the same graph
    x2 = make_layer(_cfg(T, 62), "cuda").x
    x_static.copy_(x2)
    g.replay()
    torch.cuda.synchronize()
    eager = layer.forward(x2)
    for a, b in zip(eager, outs):
        assert torch.equal(a, b)


def test_concurrent_calls_on_two_streams_match_eager():
    a_in = make_layer(_cfg(700, 63), "cuda")
    b_in = make_layer(_cfg(300, 64), "cuda")
    la = MoELayer.from_inputs(a_in, out_fp32=True)
    lb = MoELayer.from_inputs(b_in, out_fp32=True)
    ra = [t.clone() for t in la.forward(a_in.x)]
    rb = [t.clone() for t in lb.forward(b_in.x)]
    sa, sb = torch.cuda.Stream(), torch.cuda.Stream()
    oa, ob = la.outputs(700), lb.outputs(300)
    torch.cuda.synchronize()
    for _ in range(3):
        la.forward(a_in.x, outputs=oa, stream=sa)
        lb.forward(b_in.x, outputs=ob, stream=sb)
    torch.cuda.synchronize()
    for x, y in zip(ra, oa):
        assert torch.equal(x, y)
    for x, y in zip(rb, ob):
        assert torch.equal(x, y)


def test_training_step_graph_capture_replays_bitwise():
    """Weight copies + training forward + saved backward captured once and
    replayed: the same bits as the eager calls, also for new inputs."""
    from deterministic_rl_gb300.synthetic import make_dout, make_replay_ids
    cfg = _cfg(300, 65).with_(d=512, F=256)
    inp = make_layer(cfg, "cuda")
    layer = MoELayer.from_inputs(inp, out_fp32=True)
    ids = make_replay_ids(cfg, device="cuda")
    dout = make_dout(cfg, device="cuda")
    T = cfg.T
    out_e, _, _ = layer.forward_train(inp.x, replay_ids=ids)
    out_e = out_e.clone()
    dx_e, g_e = layer.backward_saved(dout)
    dx_e = dx_e.clone()
    g_e = {k: v.clone() for k, v in g_e.items()}
    x_s, ids_s, dout_s = inp.x.clone(), ids.clone(), dout.clone()
    outs = layer.outputs(T)
    grads = layer.alloc_grads()
    dx = torch.empty((T, cfg.d), dtype=torch.float32, device="cuda")
    s = torch.cuda.Stream()

    def step():
        layer.prepare_backward(stream=s)
        layer.forward_train(x_s, replay_ids=ids_s, outputs=outs, stream=s)
        layer.backward_saved(dout_s, grads=grads, dx=dx, stream=s)

    with torch.cuda.stream(s):
        step()  # warm-up on the capture stream
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        step()
    dx.zero_()
    outs[0].zero_()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(outs[0], out_e) and torch.equal(dx, dx_e)
    for k in g_e:
        assert torch.equal(grads[k], g_e[k]), k
    # new dout through the same graph
    dout2 = make_dout(cfg.with_(seed=cfg.seed + 1), device="cuda")
    dout_s.copy_(dout2)
    g.replay()
    torch.cuda.synchronize()
    layer.forward_train(inp.x, replay_ids=ids)
    dx2, g2 = layer.backward_saved(dout2)
    torch.cuda.synchronize()
    assert torch.equal(dx, dx2)
    for k in g2:
        assert torch.equal(grads[k], g2[k]), k
