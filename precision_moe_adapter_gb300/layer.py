"""A device-resident MoE layer driven through the C ABI.

Holds the frozen quantized experts, the router and the adapter as torch
device tensors (torch is only the allocator here), the routing buffers and
the workspaces, and runs one step of the layer:

    moe_route -> moe_permute -> moe_chunked_forward -> moe_backward_data

Every computation happens in libpmoe's kernels; this module only allocates
and passes pointers.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np
import torch

from . import pmoe
from .inputs import LayerConfig


def _dev(a, device) -> torch.Tensor:
    if isinstance(a, torch.Tensor):   # already a tensor (e.g. drawn on the device)
        return a.to(device)
    t = torch.from_numpy(np.ascontiguousarray(a))
    if t.dtype == torch.uint16:
        t = t.view(torch.int16)
    return t.to(device)


@dataclass
class Routing:
    idx: torch.Tensor
    w: torch.Tensor
    counts: torch.Tensor
    offsets: torch.Tensor
    perm: torch.Tensor
    inv_perm: torch.Tensor
    active: torch.Tensor
    num_active: torch.Tensor

    def c(self) -> pmoe.Routing:
        return pmoe.routing(self.idx, self.w, self.counts, self.offsets, self.perm, self.inv_perm,
                            self.active, self.num_active)


class DeviceLayer:
    """Frozen experts + router + adapter of one layer on a CUDA device.

    ``S_up`` / ``S_down`` (f32 [n_sets, dim/b, b, b], n_sets = E or 1) are
    the adapter's skew parameters; the rotations R = Cayley(S) are computed
    on the device by ``adapter_cayley``.  ``R_up`` / ``R_down`` (BF16 bits)
    may be given instead.  Passing neither disables the adapter."""

    def __init__(self, cfg: LayerConfig, w13, s13, w2, s2, Wr=None, bias=None, S_up=None,
                 S_down=None, R_up=None, R_down=None, device="cuda"):
        self.cfg = cfg
        self.device = torch.device(device)
        self.dims = pmoe.dims(cfg.T, cfg.d, cfg.E, cfg.k, cfg.I, cfg.b)
        self.w13, self.s13 = _dev(w13, self.device), _dev(s13, self.device)
        self.w2, self.s2 = _dev(w2, self.device), _dev(s2, self.device)
        self.wts = pmoe.weights(cfg.fmt, self.w13, self.s13, self.w2, self.s2)
        self.Wr = None if Wr is None else _dev(Wr, self.device)
        self.bias = None if bias is None else _dev(bias, self.device)
        self.R_up = self.R_down = None
        self.S_up = self.S_down = None
        self.Rf_up = self.Rf_down = None
        if S_up is not None:
            self.S_up = _dev(S_up, self.device)
            self.R_up, self.Rf_up = self._cayley(self.S_up)
        elif R_up is not None:
            self.R_up = _dev(R_up, self.device)
        if S_down is not None:
            self.S_down = _dev(S_down, self.device)
            self.R_down, self.Rf_down = self._cayley(self.S_down)
        elif R_down is not None:
            self.R_down = _dev(R_down, self.device)
        self.adp = None
        if self.R_up is not None:
            su = 0 if self.R_up.shape[0] == 1 else cfg.d * cfg.b
            sd = 0 if (self.R_down is None or self.R_down.shape[0] == 1) else cfg.I * cfg.b
            self.adp = pmoe.adapter(self.R_up, self.R_down, su, sd)
        self._ws = {}

    def _cayley(self, S):
        b = self.cfg.b
        nblk = S.numel() // (b * b)
        Rb = torch.empty(S.shape, dtype=torch.int16, device=self.device)
        Rf = torch.empty(S.shape, dtype=torch.float32, device=self.device)
        pmoe.adapter_cayley(nblk, b, S, Rb, Rf)
        return Rb, Rf

    def workspace(self, op, C=1, mode=pmoe.MODE_FUSED) -> torch.Tensor:
        key = (op, C, mode)
        if key not in self._ws:
            n = pmoe.moe_workspace_bytes(self.dims, op, C, mode)
            self._ws[key] = torch.zeros(max(n, 256), dtype=torch.uint8, device=self.device)
        return self._ws[key]

    def new_routing(self) -> Routing:
        cfg, dev = self.cfg, self.device
        i32 = dict(dtype=torch.int32, device=dev)
        return Routing(idx=torch.zeros((cfg.T, cfg.k), **i32),
                       w=torch.zeros((cfg.T, cfg.k), dtype=torch.float32, device=dev),
                       counts=torch.zeros(cfg.E, **i32), offsets=torch.zeros(cfg.E + 1, **i32),
                       perm=torch.zeros(cfg.P, **i32), inv_perm=torch.zeros(cfg.P, **i32),
                       active=torch.zeros(cfg.E, **i32), num_active=torch.zeros(1, **i32))

    # -------------------------------------------------------------- steps
    def route(self, X: torch.Tensor, rt: Routing, logits: torch.Tensor | None = None,
              mode: int = pmoe.ROUTE_FAST):
        ws = self.workspace(pmoe.OP_PERMUTE)
        pmoe.moe_route(self.dims, X, self.Wr, self.bias, logits, rt.idx, rt.w, ws, mode=mode)

    def permute(self, rt: Routing):
        pmoe.moe_permute(self.dims, rt.idx, rt.c(), self.workspace(pmoe.OP_PERMUTE))

    def new_ctx(self) -> torch.Tensor:
        """The forward's saved context for the backward (moe_ctx_bytes)."""
        return torch.empty(max(pmoe.moe_ctx_bytes(self.dims), 16), dtype=torch.uint8,
                           device=self.device)

    def forward(self, X, rt: Routing, Y, C=None, mode=pmoe.MODE_FUSED, ctx=None):
        C = C or self.cfg.C
        ws = self.workspace(pmoe.OP_FORWARD, C, mode)
        pmoe.moe_chunked_forward(self.dims, self.wts, self.adp, rt.c(), X, C, mode, Y, ctx, ws)

    def backward(self, X, dY, ctx, rt: Routing, dX, d_topk_w=None, dR_up=None, dR_down=None,
                 C=None):
        C = C or self.cfg.C
        ws = self.workspace(pmoe.OP_BACKWARD, C)
        pmoe.moe_backward_data(self.dims, self.wts, self.adp, rt.c(), X, dY, ctx, C, dX,
                               d_topk_w, dR_up, dR_down, ws)

    def grads(self):
        """Fresh (dR_up, dR_down) buffers shaped like the rotations."""
        dru = None if self.R_up is None else torch.zeros(self.R_up.shape, dtype=torch.float32,
                                                         device=self.device)
        drd = None if self.R_down is None else torch.zeros(self.R_down.shape,
                                                           dtype=torch.float32, device=self.device)
        return dru, drd

    def status(self) -> int:
        """OR of the device error words of every workspace used so far."""
        s = 0
        for ws in self._ws.values():
            s = s or pmoe.moe_query_status(ws)
        return s
