"""The C-ABI library loads and exports every function include/*.h declares, and
its host-side validation rejects bad arguments before launching anything.
CPU only: no call here reaches the GPU (fake pointers are never dereferenced
because each call fails validation first)."""
import ctypes
import glob
import os
import re

import pytest

from deterministic_rl_gb300 import binding as B
from deterministic_rl_gb300 import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return B.load()


def declared_functions():
    names = []
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        src = open(h).read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        src = re.sub(r"//[^\n]*", "", src)
        names += re.findall(r"\b(moe_[a-z_]+)\s*\([^;{]*\)\s*;", src)
    return sorted(set(names))


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert set(names) == set(B.EXPORTED), names
    for n in names:
        assert hasattr(lib, n), n


def good_dims(**kw):
    d = dict(T=64, d=7168, E=384, k=8, F=2048, n_shared=1)
    d.update(kw)
    return B.Dims(**d)


def test_workspace_size_and_layout(lib):
    d = good_dims()
    n = B.moe_workspace_size(d)
    L = B.moe_workspace_layout(d)
    assert L.total == n > 0
    offs = [L.status, L.logits, L.valid, L.cnt, L.off, L.perm, L.inv, L.xp, L.h, L.y, L.ysh]
    assert offs == sorted(offs) and all(o % 256 == 0 for o in offs)
    assert L.logits - L.status >= 16
    assert L.valid - L.logits >= 64 * 384 * 4
    assert L.h - L.xp >= (64 * 8 + 64) * 7168 * 2
    assert n - L.ysh >= 64 * 7168 * 4
    # the workspace grows linearly in T (no hidden per-call allocation)
    assert B.moe_workspace_size(good_dims(T=128)) > n


@pytest.mark.parametrize("bad", [dict(k=4), dict(E=4), dict(E=1024), dict(d=100), dict(F=96),
                                 dict(n_shared=2), dict(T=-1), dict(T=(1 << 20) + 1),
                                 dict(wfmt=7), dict(out_fp32=2), dict(wfmt=1, d=192)])
def test_bad_dims_rejected(lib, bad):
    d = good_dims(**bad)
    assert B.moe_workspace_size(d) == 0
    with pytest.raises(B.MoEError) as ei:
        B.moe_workspace_layout(d)
    assert ei.value.code == B.MOE_ERR_SHAPE


class _Fake:
    """Stands in for a tensor: an address that validation never dereferences."""
    def __init__(self, addr, nbytes=16):
        self.addr, self.nbytes = addr, nbytes

    def data_ptr(self):
        return self.addr

    def numel(self):
        return self.nbytes

    def element_size(self):
        return 1


_DEFAULT_WS = _Fake(0x10000)


def _call(lib, fn, dims, x, w, *ptrs, ws=_DEFAULT_WS, ws_bytes=None):
    nbytes = ws_bytes if ws_bytes is not None else (B.moe_workspace_size(dims) or 1)
    cargs = [ctypes.c_void_p(p.data_ptr() if p is not None else None) for p in ptrs]
    f = getattr(lib, fn)
    return f(ctypes.byref(dims.c()), ctypes.c_void_p(x.data_ptr() if x else None),
             ctypes.byref(w), *cargs, ctypes.c_void_p(ws.data_ptr() if ws else None),
             nbytes, ctypes.c_void_p(None))


def _weights(**override):
    base = dict(w_router=_Fake(0x20000), router_bias=None, w_gate=_Fake(0x30000),
                w_up=_Fake(0x40000), w_down=_Fake(0x50000), ws_gate=_Fake(0x60000),
                ws_up=_Fake(0x70000), ws_down=_Fake(0x80000))
    base.update(override)
    return B.make_weights(**base)


def test_host_validation_codes(lib):
    d = good_dims()
    x, out, ids, g = _Fake(0x1000), _Fake(0x2000), _Fake(0x3000), _Fake(0x4000)
    fwd = lambda w=_weights(), **kw: _call(lib, "moe_forward", kw.pop("dims", d), kw.pop("x", x), w,
                                           kw.pop("out", out), kw.pop("ids", ids),
                                           kw.pop("g", g), **kw)
    # T == 0 is a no-op
    assert fwd(dims=good_dims(T=0)) == B.MOE_OK
    # null pointers
    assert fwd(x=None) == B.MOE_ERR_ARG
    assert fwd(out=None) == B.MOE_ERR_ARG
    assert fwd(w=_weights(w_gate=None)) == B.MOE_ERR_ARG
    assert fwd(w=_weights(ws_down=None)) == B.MOE_ERR_ARG
    assert fwd(ws=None) == B.MOE_ERR_ARG
    # misaligned pointers
    assert fwd(x=_Fake(0x1004)) == B.MOE_ERR_ALIGN
    assert fwd(w=_weights(w_up=_Fake(0x40008))) == B.MOE_ERR_ALIGN
    assert fwd(g=_Fake(0x4002)) == B.MOE_ERR_ALIGN
    # short workspace
    assert fwd(ws_bytes=B.moe_workspace_size(d) - 1) == B.MOE_ERR_WORKSPACE
    # bad shapes
    assert fwd(dims=good_dims(E=3)) == B.MOE_ERR_SHAPE
    # MXFP8 weights without their scales
    assert fwd(dims=good_dims(wfmt=1)) == B.MOE_ERR_ARG
    # replay needs its ids
    rc = _call(lib, "moe_forward_replay", d, x, _weights(), None, out, ids, g)
    assert rc == B.MOE_ERR_ARG
    # routing only: outputs required
    assert _call(lib, "moe_route", d, x, _weights(), None, g) == B.MOE_ERR_ARG
    assert lib.moe_get_status(None, None) == B.MOE_ERR_ARG


def test_status_strings(lib):
    for code in range(9):
        s = B.moe_status_str(code)
        assert s.startswith("MOE_")
    assert "unknown" in B.moe_status_str(99)


# ---- backward ----------------------------------------------------------------

def test_backward_sizes_and_layout(lib):
    d = good_dims(T=4096)
    n = B.moe_backward_workspace_size(d)
    L = B.moe_backward_workspace_layout(d)
    assert L.total == n > B.moe_workspace_size(d)
    offs = [L.status, L.logits, L.valid, L.cnt, L.off, L.perm, L.inv, L.xp, L.h, L.y, L.ids,
            L.gates, L.poff, L.a, L.b, L.dg, L.dl, L.dyq, L.dh, L.dabq, L.dxp, L.xpt, L.dyt,
            L.ht, L.dabt]
    assert offs == sorted(offs) and all(o % 256 == 0 for o in offs)
    rows = 4096 * 9
    assert L.kpad % 64 == 0 and L.kpad >= rows + 63 * 385
    assert L.xpt - L.dxp >= rows * 7168 * 4
    assert n - L.dabt >= 2 * 2048 * L.kpad * 2
    # the forward's status word sits at the same place
    assert L.status == B.moe_workspace_layout(d).status
    # E4M3 codes and one E8M0 byte per 32 of three matrices per expert, shared one included
    G, FD = 385, 2048 * 7168
    assert B.moe_backward_weights_size(d) >= 3 * G * FD * 33 // 32
    assert B.moe_backward_weights_size(d) < 3 * G * FD * 33 // 32 + 4 * 256
    assert B.moe_backward_weights_size(good_dims(n_shared=0)) < B.moe_backward_weights_size(d)
    # Q(dY) and [Q(dA) | Q(dB)]: codes then scale bytes
    assert L.dh - L.dyq >= rows * 7168 * 33 // 32
    assert L.dxp - L.dabq >= rows * 2 * 2048 * 33 // 32


@pytest.mark.parametrize("bad", [dict(d=7168 - 64), dict(d=7168 - 256), dict(F=2048 + 64),
                                 dict(k=4), dict(wfmt=1), dict(wfmt=2)])
def test_backward_unserved_dims(lib, bad):
    d = good_dims(**bad)
    assert B.moe_backward_workspace_size(d) == 0
    assert B.moe_backward_weights_size(d) == 0
    with pytest.raises(B.MoEError):
        B.moe_backward_workspace_layout(d)


def _bwd(lib, dims=None, x=_Fake(0x1000), w=None, wt=_Fake(0x90000), ids=_Fake(0x3000),
         dout=_Fake(0x5000), dx=_Fake(0x6000), grads=None, ws=_DEFAULT_WS, ws_bytes=None):
    dims = dims or good_dims()
    w = w or _weights()
    grads = grads or B.moe_grads(0xA000, 0xB000, 0xC000, 0xD000, 0xE000, 0xF000, 0x11000)
    nbytes = ws_bytes if ws_bytes is not None else (B.moe_backward_workspace_size(dims) or 1)
    v = lambda p: ctypes.c_void_p(p.data_ptr() if p is not None else None)  # noqa: E731
    return lib.moe_backward(ctypes.byref(dims.c()), v(x), ctypes.byref(w), v(wt), v(ids), v(dout),
                            v(dx), ctypes.byref(grads), v(ws), nbytes, ctypes.c_void_p(None))


def test_backward_host_validation_codes(lib):
    assert _bwd(lib, dims=good_dims(T=0)) == B.MOE_OK
    assert _bwd(lib, x=None) == B.MOE_ERR_ARG
    assert _bwd(lib, wt=None) == B.MOE_ERR_ARG
    assert _bwd(lib, ids=None) == B.MOE_ERR_ARG
    assert _bwd(lib, dout=None) == B.MOE_ERR_ARG
    assert _bwd(lib, dx=None) == B.MOE_ERR_ARG
    assert _bwd(lib, ws=None) == B.MOE_ERR_ARG
    assert _bwd(lib, w=_weights(w_down=None)) == B.MOE_ERR_ARG
    assert _bwd(lib, grads=B.moe_grads(0xA000, 0xB000, 0xC000, 0xD000, None, None, None)) == B.MOE_ERR_ARG
    assert _bwd(lib, dims=good_dims(n_shared=0),
                grads=B.moe_grads(0xA000, 0xB000, 0xC000, 0xD000, None, None, None),
                ws_bytes=1) == B.MOE_ERR_WORKSPACE
    assert _bwd(lib, dout=_Fake(0x5008)) == B.MOE_ERR_ALIGN
    assert _bwd(lib, grads=B.moe_grads(0xA004, 0xB000, 0xC000, 0xD000, 0xE000, 0xF000, 0x11000)) == B.MOE_ERR_ALIGN
    assert _bwd(lib, ws_bytes=B.moe_backward_workspace_size(good_dims()) - 1) == B.MOE_ERR_WORKSPACE
    assert _bwd(lib, dims=good_dims(wfmt=1)) == B.MOE_ERR_UNSUPPORTED
    assert _bwd(lib, dims=good_dims(d=7168 - 64)) == B.MOE_ERR_SHAPE
    # preparing the weight copies: short buffer, null weights
    d = good_dims()
    assert lib.moe_backward_prepare_weights(ctypes.byref(d.c()), ctypes.byref(_weights()),
                                            ctypes.c_void_p(0x90000), 16, None) == B.MOE_ERR_WORKSPACE
    assert lib.moe_backward_prepare_weights(ctypes.byref(d.c()), ctypes.byref(_weights(w_up=None)),
                                            ctypes.c_void_p(0x90000), 1 << 40, None) == B.MOE_ERR_ARG


def test_training_entry_points_validate(lib):
    d = good_dims()
    ws = _DEFAULT_WS
    nb = B.moe_backward_workspace_size(d)
    v = lambda a: ctypes.c_void_p(a)  # noqa: E731
    W = _weights()
    f = lambda **kw: lib.moe_forward_train(  # noqa: E731
        ctypes.byref(kw.get("dims", d).c()), v(kw.get("x", 0x1000)), ctypes.byref(kw.get("w", W)),
        v(kw.get("ids", None)), v(kw.get("out", 0x2000)), v(kw.get("ids_out", 0x3000)),
        v(kw.get("g", 0x4000)), v(0x10000), kw.get("nb", nb), v(None))
    assert f(dims=good_dims(T=0)) == B.MOE_OK
    assert f(x=None) == B.MOE_ERR_ARG
    assert f(out=None) == B.MOE_ERR_ARG
    assert f(g=0x4004) == B.MOE_ERR_ALIGN
    assert f(nb=nb - 1) == B.MOE_ERR_WORKSPACE
    assert f(dims=good_dims(wfmt=1)) == B.MOE_ERR_UNSUPPORTED
    grads = B.moe_grads(0xA000, 0xB000, 0xC000, 0xD000, 0xE000, 0xF000, 0x11000)
    sb = lambda **kw: lib.moe_backward_saved(  # noqa: E731
        ctypes.byref(d.c()), ctypes.byref(W), v(kw.get("wt", 0x90000)), v(kw.get("dout", 0x5000)),
        v(kw.get("dx", 0x6000)), ctypes.byref(grads), v(0x10000), kw.get("nb", nb), v(None))
    assert sb(wt=None) == B.MOE_ERR_ARG
    assert sb(dout=None) == B.MOE_ERR_ARG
    assert sb(dx=0x6008) == B.MOE_ERR_ALIGN
    assert sb(nb=16) == B.MOE_ERR_WORKSPACE


def test_pack_weights_validation(lib):
    d = good_dims()
    assert B.moe_packed_weights_size(d) == (384 + 1) * 2 * 2048 * 7168 * 2
    assert B.moe_packed_weights_size(good_dims(wfmt=1)) == 0
    v = ctypes.c_void_p
    pk = lambda dims, w, ptr, n: lib.moe_pack_weights(  # noqa: E731
        ctypes.byref(dims.c()), ctypes.byref(w), v(ptr), n, v(None))
    n = B.moe_packed_weights_size(d)
    assert pk(good_dims(wfmt=1), _weights(), 0x90000, n) == B.MOE_ERR_UNSUPPORTED
    assert pk(d, _weights(), None, n) == B.MOE_ERR_ARG
    assert pk(d, _weights(w_up=None), 0x90000, n) == B.MOE_ERR_ARG
    assert pk(d, _weights(), 0x90008, n) == B.MOE_ERR_ALIGN
    assert pk(d, _weights(), 0x90000, n - 1) == B.MOE_ERR_WORKSPACE
    # a packed pointer with non-bf16 weights is refused by the forward
    x, out, ids, g = _Fake(0x1000), _Fake(0x2000), _Fake(0x3000), _Fake(0x4000)
    w = _weights(w_gate_up=_Fake(0x90000))
    rc = _call(lib, "moe_forward", good_dims(wfmt=1, n_shared=0), x, w, out, ids, g)
    assert rc in (B.MOE_ERR_ARG, B.MOE_ERR_UNSUPPORTED)
    assert _call(lib, "moe_forward", d, x, _weights(w_gate_up=_Fake(0x90004)), out, ids, g) == B.MOE_ERR_ALIGN


@pytest.mark.parametrize("wfmt", [2, 3])  # NVFP4, MXFP8 weights and activations
def test_narrow_activation_regions_fit(lib, wfmt):
    """The regions the block-scaled layers write hold what they must: the codes
    and block scales of x ([T][d/2] + [T][d/16] for NVFP4, [T][d] + [T][d/32]
    for MXFP8), of the gathered rows (in the xp region) and of h (hq); NVFP4's
    fp32 row scales of x, of the gathered rows and of h."""
    T, d, F, k = 300, 7168, 2048, 8
    dims = good_dims(T=T, n_shared=0, wfmt=wfmt)
    L = B.moe_workspace_layout(dims)
    nv = wfmt == 2
    per = (lambda K: K // 2 + K // 16) if nv else (lambda K: K + K // 32)
    regions = sorted([(L.xp, L.h), (L.xq, L.sx), (L.hq, L.total)])
    assert L.h - L.xp >= T * k * per(d)
    assert L.sx - L.xq >= T * per(d)
    assert L.total - L.hq >= T * k * per(F)
    if nv:
        assert L.sxp - L.sx >= T * 4 and L.sh - L.sxp >= T * k * 4 and L.hq - L.sh >= T * k * 4
    assert all(a % 256 == 0 for a, _ in regions)
