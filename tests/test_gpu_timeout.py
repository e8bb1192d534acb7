"""Failure detection without a GPU fault: a bounded wait that runs out.

With MOE_TEST_STALL_CALLS=1 the gate/up GEMM of the first forward call issues
no loads, so its MMA waits on a barrier that nothing fills; the wait gives up
after 1 s, the kernel returns, and moe_get_status reports MOE_ERR_TIMEOUT.  The
context stays usable: the next call in the same process succeeds and matches a
clean run bitwise.  Both GEMM families are covered (T <= 128 one-SM, T > 128 SM
pairs).  The environment variable is read once per process, hence subprocesses."""
import os
import subprocess
import sys

import pytest
import torch

from deterministic_rl_gb300 import build, MoELayer
from deterministic_rl_gb300 import binding as B
from deterministic_rl_gb300.synthetic import CONFIGS, make_layer

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

_SCRIPT = r"""
import sys, time, torch
sys.path.insert(0, {root!r})
from deterministic_rl_gb300 import MoELayer
from deterministic_rl_gb300 import binding as B
from deterministic_rl_gb300.synthetic import CONFIGS, make_layer
cfg = CONFIGS["c1_tiny"].with_(name="stall", seed=5, T={T}, n_shared=1)
inp = make_layer(cfg, "cuda")
layer = MoELayer.from_inputs(inp, out_fp32=True)
t0 = time.time()
layer.forward(inp.x)
first = layer.status()
dt = time.time() - t0
out = [t.clone() for t in layer.forward(inp.x)]
second = layer.status()
torch.save([first, second, dt] + [t.cpu() for t in out], {path!r})
"""


@pytest.fixture(scope="module", autouse=True)
def _built():
    build.build()


@pytest.mark.parametrize("T", [64, 300])
def test_wait_that_runs_out_reports_timeout_and_context_survives(tmp_path, T):
    path = str(tmp_path / "r.pt")
    env = dict(os.environ, MOE_TEST_STALL_CALLS="1")
    subprocess.run([sys.executable, "-c", _SCRIPT.format(root=ROOT, T=T, path=path)], env=env,
                   check=True, timeout=300)
    first, second, dt, *out = torch.load(path)
    assert first == B.MOE_ERR_TIMEOUT
    assert second == B.MOE_OK
    assert dt < 30  # bounded: the waits give up after about a second each
    cfg = CONFIGS["c1_tiny"].with_(name="stall", seed=5, T=T, n_shared=1)
    inp = make_layer(cfg, "cuda")
    ref = MoELayer.from_inputs(inp, out_fp32=True).forward(inp.x)
    for a, b in zip(out, ref):
        assert torch.equal(a, b.cpu())


_BWD_SCRIPT = r"""
import sys, time, torch
sys.path.insert(0, {root!r})
from deterministic_rl_gb300 import MoELayer
from deterministic_rl_gb300.synthetic import CONFIGS, make_layer, make_dout, make_replay_ids
cfg = CONFIGS["c1_tiny"].with_(name="stall_bwd", seed=6, T=300, n_shared=1)
inp = make_layer(cfg, "cuda")
layer = MoELayer.from_inputs(inp)
ids = make_replay_ids(cfg, device="cuda")
dout = make_dout(cfg, device="cuda")
t0 = time.time()
layer.backward(inp.x, ids, dout)
first = layer.backward_status()
dt = time.time() - t0
dx, g = layer.backward(inp.x, ids, dout)
second = layer.backward_status()
torch.save([first, second, dt, dx.cpu()] + [g[k].cpu() for k in sorted(g)], {path!r})
"""


def test_backward_wait_that_runs_out_reports_timeout_and_context_survives(tmp_path):
    """MOE_TEST_STALL_BWD_CALLS=1: the weight-gradient GEMM of the first backward
    issues no loads; its waits run out, the call reports MOE_ERR_TIMEOUT, and the
    next backward in the same process succeeds and matches a clean run bitwise."""
    from deterministic_rl_gb300.synthetic import make_dout, make_replay_ids
    path = str(tmp_path / "b.pt")
    env = dict(os.environ, MOE_TEST_STALL_BWD_CALLS="1")
    subprocess.run([sys.executable, "-c", _BWD_SCRIPT.format(root=ROOT, path=path)], env=env,
                   check=True, timeout=300)
    first, second, dt, dx, *grads = torch.load(path)
    assert first == B.MOE_ERR_TIMEOUT
    assert second == B.MOE_OK
    assert dt < 30
    cfg = CONFIGS["c1_tiny"].with_(name="stall_bwd", seed=6, T=300, n_shared=1)
    inp = make_layer(cfg, "cuda")
    layer = MoELayer.from_inputs(inp)
    rdx, rg = layer.backward(inp.x, make_replay_ids(cfg, device="cuda"), make_dout(cfg, device="cuda"))
    torch.cuda.synchronize()
    assert torch.equal(dx, rdx.cpu())
    for a, k in zip(grads, sorted(rg)):
        assert torch.equal(a, rg[k].cpu()), k
