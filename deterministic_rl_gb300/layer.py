"""MoELayer: holds the layer's device weights and a workspace and calls the C
ABI through the binding, allocating output tensors with torch.  Marshalling
only -- every computation happens in libmoedet."""
from __future__ import annotations

from typing import Optional

import torch

from . import binding as B


class MoELayer:
    def __init__(self, w_router, w_gate, w_up, w_down, *, k: int = 8, router_bias=None,
                 s_gate=None, s_up=None, s_down=None, ws_gate=None, ws_up=None, ws_down=None,
                 gs_gate=None, gs_up=None, gs_down=None, out_fp32: bool = False,
                 act_mx: bool = False):
        """Weight formats: bf16 (s_* None); MXFP8 (s_* E8M0 scales; with act_mx
        the activations are quantised to MXFP8 too); NVFP4 (gs_* per-matrix
        fp32 scales given; w_* packed E2M1, s_* E4M3)."""
        self.E, self.d = w_router.shape
        self.F = w_gate.shape[1]
        self.k = k
        self.n_shared = 1 if ws_gate is not None else 0
        if gs_gate is not None:
            self.wfmt = B.MOE_W_NVFP4
        elif s_gate is not None:
            self.wfmt = B.MOE_W_MXFP8_ACT if act_mx else B.MOE_W_MXFP8
        else:
            if act_mx:
                raise ValueError("MXFP8 activations need MXFP8 weights")
            self.wfmt = B.MOE_W_BF16
        self.out_fp32 = bool(out_fp32)
        self.device = w_router.device
        # keep references so the pointers stay valid
        self._tensors = (w_router, router_bias, w_gate, w_up, w_down, s_gate, s_up, s_down,
                         ws_gate, ws_up, ws_down, gs_gate, gs_up, gs_down)
        self.weights = B.make_weights(*self._tensors)
        self._ws = None
        self._ws_T = -1
        self._wt = None      # the backward's weight copies (prepare_backward)
        self._bws = None
        self._bws_T = -1

    @classmethod
    def from_inputs(cls, inp, out_fp32: bool = False) -> "MoELayer":
        return cls(inp.w_router, inp.w_gate, inp.w_up, inp.w_down, k=inp.cfg.k,
                   router_bias=inp.router_bias, s_gate=inp.s_gate, s_up=inp.s_up,
                   s_down=inp.s_down, ws_gate=inp.ws_gate, ws_up=inp.ws_up,
                   ws_down=inp.ws_down, gs_gate=inp.gs_gate, gs_up=inp.gs_up,
                   gs_down=inp.gs_down, out_fp32=out_fp32, act_mx=inp.cfg.act_mx)

    def pack_weights(self, stream=None) -> torch.Tensor:
        """Pack the gate/up weights (bf16) for the SM-pair forward GEMM (one copy
        per weight tile instead of two; same results).  Call again after the
        weights change."""
        n = B.moe_packed_weights_size(self.dims(1))
        if n == 0:
            raise B.MoEError(B.MOE_ERR_UNSUPPORTED, "moe_packed_weights_size")
        self._packed = torch.empty(n, dtype=torch.uint8, device=self.device)
        self.weights.w_gate_up = None
        B.moe_pack_weights(self.dims(1), self.weights, self._packed, stream)
        self.weights.w_gate_up = self._packed.data_ptr()
        return self._packed

    def unpack_weights(self) -> None:
        self.weights.w_gate_up = None
        self._packed = None

    def dims(self, T: int) -> B.Dims:
        return B.Dims(T, self.d, self.E, self.k, self.F, self.n_shared, self.wfmt,
                      int(self.out_fp32))

    def workspace(self, T: int) -> torch.Tensor:
        """A workspace for T tokens (reused while T does not grow)."""
        if self._ws is None or T > self._ws_T:
            n = B.moe_workspace_size(self.dims(T))
            if n == 0:
                raise B.MoEError(B.MOE_ERR_SHAPE, "moe_workspace_size")
            self._ws = torch.empty(n, dtype=torch.uint8, device=self.device)
            self._ws_T = T
        return self._ws

    def outputs(self, T: int):
        odt = torch.float32 if self.out_fp32 else torch.bfloat16
        out = torch.empty((T, self.d), dtype=odt, device=self.device)
        ids = torch.empty((T, self.k), dtype=torch.int32, device=self.device)
        gates = torch.empty((T, self.k), dtype=torch.float32, device=self.device)
        return out, ids, gates

    def route(self, x: torch.Tensor, stream=None):
        T = x.shape[0]
        ids = torch.empty((T, self.k), dtype=torch.int32, device=self.device)
        gates = torch.empty((T, self.k), dtype=torch.float32, device=self.device)
        B.moe_route(self.dims(T), x, self.weights, ids, gates, self.workspace(T), stream)
        return ids, gates

    def forward(self, x: torch.Tensor, replay_ids: Optional[torch.Tensor] = None, stream=None,
                outputs=None, filter_tau: Optional[float] = None):
        T = x.shape[0]
        out, ids, gates = outputs if outputs is not None else self.outputs(T)
        ws = self.workspace(T)
        if replay_ids is not None and filter_tau is not None:
            B.moe_forward_replay_filtered(self.dims(T), x, self.weights, replay_ids, filter_tau,
                                          out, ids, gates, ws, stream)
        elif replay_ids is None:
            B.moe_forward(self.dims(T), x, self.weights, out, ids, gates, ws, stream)
        else:
            B.moe_forward_replay(self.dims(T), x, self.weights, replay_ids, out, ids, gates, ws,
                                 stream)
        return out, ids, gates

    def status(self, stream=None) -> int:
        return B.moe_get_status(self._ws, stream)

    def intermediates(self, T: int) -> dict:
        """Views of the workspace's intermediate buffers after a call with T tokens."""
        L = B.moe_workspace_layout(self.dims(T))
        ws = self.workspace(T)
        k, E, d, F = self.k, self.E, self.d, self.F
        rows = T * k + T * self.n_shared

        def view(off, n, dt):
            nbytes = n * torch.tensor([], dtype=dt).element_size()
            return ws[off:off + nbytes].view(dt)

        r = {
            "status": view(L.status, 4, torch.int32),
            "logits": view(L.logits, T * E, torch.float32).view(T, E),
            "valid": view(L.valid, T, torch.int32),
            "cnt": view(L.cnt, E, torch.int32),
            "off": view(L.off, E + 1, torch.int32),
            "perm": view(L.perm, T * k, torch.int32),
            "inv": view(L.inv, T * k, torch.int32),
            "xp": view(L.xp, rows * d, torch.bfloat16).view(rows, d),
            "h": view(L.h, rows * F, torch.bfloat16).view(rows, F),
            "y": view(L.y, T * k * d, torch.bfloat16).view(T * k, d),
        }
        if self.n_shared:
            r["ysh"] = view(L.ysh, T * d, torch.float32).view(T, d)
        if self.wfmt == B.MOE_W_MXFP8_ACT:
            # E4M3 codes and E8M0 scales of the quantised token rows and of h
            r["x8"] = view(L.xq, T * d, torch.uint8).view(T, d)
            r["xs"] = ws[L.xq + T * d:L.xq + T * d + T * d // 32].view(T, d // 32)
            r["xp8"] = view(L.xp, T * k * d, torch.uint8).view(T * k, d)
            r["h8"] = view(L.hq, T * k * F, torch.uint8).view(T * k, F)
            r["hs"] = ws[L.hq + T * k * F:L.hq + T * k * F + T * k * F // 32].view(T * k, F // 32)
        if self.wfmt == B.MOE_W_NVFP4:
            # packed E2M1 codes (element 2j in the low nibble of byte j), E4M3
            # block scales per 16 and fp32 row scales of x, the gathered rows
            # and h
            tk = T * k
            r["x4"] = view(L.xq, T * d // 2, torch.uint8).view(T, d // 2)
            r["xb"] = ws[L.xq + T * d // 2:L.xq + T * d // 2 + T * d // 16].view(T, d // 16)
            r["xp4"] = view(L.xp, tk * d // 2, torch.uint8).view(tk, d // 2)
            r["xpb"] = ws[L.xp + tk * d // 2:L.xp + tk * d // 2 + tk * d // 16].view(tk, d // 16)
            r["h4"] = view(L.hq, tk * F // 2, torch.uint8).view(tk, F // 2)
            r["hb"] = ws[L.hq + tk * F // 2:L.hq + tk * F // 2 + tk * F // 16].view(tk, F // 16)
            r["sx"] = view(L.sx, T, torch.float32)
            r["sxp"] = view(L.sxp, T * k, torch.float32)
            r["sh"] = view(L.sh, T * k, torch.float32)
        return r

    # ---- backward -------------------------------------------------------------

    def prepare_backward(self, stream=None) -> torch.Tensor:
        """The weight copies the backward reads (quantised along its contraction
        axes, transposed); call again after the weights change."""
        n = B.moe_backward_weights_size(self.dims(1))
        if n == 0:
            raise B.MoEError(B.MOE_ERR_UNSUPPORTED, "moe_backward_weights_size")
        if self._wt is None or self._wt.numel() < n:
            self._wt = torch.empty(n, dtype=torch.uint8, device=self.device)
        B.moe_backward_prepare_weights(self.dims(1), self.weights, self._wt, stream)
        return self._wt

    def backward_workspace(self, T: int) -> torch.Tensor:
        if self._bws is None or T > self._bws_T:
            n = B.moe_backward_workspace_size(self.dims(T))
            if n == 0:
                raise B.MoEError(B.MOE_ERR_SHAPE, "moe_backward_workspace_size")
            self._bws = torch.empty(n, dtype=torch.uint8, device=self.device)
            self._bws_T = T
        return self._bws

    def alloc_grads(self) -> dict:
        E, d, F = self.E, self.d, self.F
        f32 = dict(dtype=torch.float32, device=self.device)
        g = {"d_router": torch.empty((E, d), **f32), "d_gate": torch.empty((E, F, d), **f32),
             "d_up": torch.empty((E, F, d), **f32), "d_down": torch.empty((E, d, F), **f32)}
        if self.n_shared:
            g.update(ds_gate=torch.empty((F, d), **f32), ds_up=torch.empty((F, d), **f32),
                     ds_down=torch.empty((d, F), **f32))
        return g

    def backward(self, x: torch.Tensor, ids: torch.Tensor, dout: torch.Tensor, stream=None,
                 grads: Optional[dict] = None, dx: Optional[torch.Tensor] = None):
        """Gradients for upstream gradient dout [T][d] bf16 with the forward's
        ids [T][k]: returns (dx [T][d] fp32, dict of fp32 weight gradients).
        Prepares the weight copies on first use."""
        T = x.shape[0]
        if self._wt is None:
            self.prepare_backward(stream)
        g = grads if grads is not None else self.alloc_grads()
        if dx is None:
            dx = torch.empty((T, self.d), dtype=torch.float32, device=self.device)
        cg = B.make_grads(g["d_router"], g["d_gate"], g["d_up"], g["d_down"], g.get("ds_gate"),
                          g.get("ds_up"), g.get("ds_down"))
        B.moe_backward(self.dims(T), x, self.weights, self._wt, ids, dout, dx, cg,
                       self.backward_workspace(T), stream)
        return dx, g

    def forward_train(self, x: torch.Tensor, replay_ids: Optional[torch.Tensor] = None,
                      stream=None, outputs=None):
        """The forward (own routing, or replay of replay_ids), keeping in the
        backward workspace what backward_saved reads; same outputs as forward()."""
        T = x.shape[0]
        out, ids, gates = outputs if outputs is not None else self.outputs(T)
        B.moe_forward_train(self.dims(T), x, self.weights, replay_ids, out, ids, gates,
                            self.backward_workspace(T), stream)
        self._saved_T = T
        return out, ids, gates

    def backward_saved(self, dout: torch.Tensor, stream=None, grads: Optional[dict] = None,
                       dx: Optional[torch.Tensor] = None):
        """The backward of the last forward_train (same results as backward()
        on its x and ids, without recomputing the forward)."""
        T = dout.shape[0]
        if getattr(self, "_saved_T", None) != T:
            raise ValueError("backward_saved needs a forward_train of the same batch first")
        if self._wt is None:
            self.prepare_backward(stream)
        g = grads if grads is not None else self.alloc_grads()
        if dx is None:
            dx = torch.empty((T, self.d), dtype=torch.float32, device=self.device)
        cg = B.make_grads(g["d_router"], g["d_gate"], g["d_up"], g["d_down"], g.get("ds_gate"),
                          g.get("ds_up"), g.get("ds_down"))
        B.moe_backward_saved(self.dims(T), self.weights, self._wt, dout, dx, cg,
                             self.backward_workspace(T), stream)
        return dx, g

    def backward_status(self, stream=None) -> int:
        return B.moe_get_status(self._bws, stream)

    def backward_intermediates(self, T: int) -> dict:
        """Views of the backward workspace's buffers after a backward of T tokens."""
        L = B.moe_backward_workspace_layout(self.dims(T))
        ws = self.backward_workspace(T)
        k, E, d, F = self.k, self.E, self.d, self.F
        rows = T * k + T * self.n_shared
        kp = int(L.kpad)

        def view(off, n, dt):
            nbytes = n * torch.tensor([], dtype=dt).element_size()
            return ws[off:off + nbytes].view(dt)

        return {
            "status": view(L.status, 4, torch.int32),
            "valid": view(L.valid, T, torch.int32),
            "cnt": view(L.cnt, E, torch.int32),
            "off": view(L.off, E + 1, torch.int32),
            "perm": view(L.perm, T * k, torch.int32),
            "ids": view(L.ids, T * k, torch.int32).view(T, k),
            "gates": view(L.gates, T * k, torch.float32).view(T, k),
            "poff": view(L.poff, E + self.n_shared + 1, torch.int32),
            "a": view(L.a, rows * F, torch.float32).view(rows, F),
            "b": view(L.b, rows * F, torch.float32).view(rows, F),
            "h": view(L.h, rows * F, torch.bfloat16).view(rows, F),
            "y": view(L.y, T * k * d, torch.bfloat16).view(T * k, d),
            "dg": view(L.dg, T * k, torch.float32).view(T, k),
            "dl": view(L.dl, T * k, torch.float32).view(T, k),
            # E4M3 codes and E8M0 scale bytes of the dH and dXp GEMMs' token rows
            "dyq": view(L.dyq, rows * d, torch.uint8).view(rows, d),
            "dyq_scales": view(L.dyq + rows * d, rows * d // 32, torch.uint8).view(rows, d // 32),
            "dh": view(L.dh, rows * F, torch.float32).view(rows, F),
            "dabq": view(L.dabq, rows * 2 * F, torch.uint8).view(rows, 2 * F),
            "dabq_scales": view(L.dabq + rows * 2 * F, rows * 2 * F // 32,
                                torch.uint8).view(rows, 2 * F // 32),
            "dxp": view(L.dxp, rows * d, torch.float32).view(rows, d),
            "xpt": view(L.xpt, d * kp, torch.bfloat16).view(d, kp),
            "dyt": view(L.dyt, d * kp, torch.bfloat16).view(d, kp),
            "ht": view(L.ht, F * kp, torch.bfloat16).view(F, kp),
            "dabt": view(L.dabt, 2 * F * kp, torch.bfloat16).view(2 * F, kp),
        }

