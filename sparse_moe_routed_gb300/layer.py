"""One routed-expert MoE layer driven through the C ABI.

``MoELayer`` owns the device buffers a layer call needs (allocated once with
torch, sized for ``T_max`` tokens) and issues the five boundary calls on one
stream:

    moe_route -> moe_permute (+ row gather) -> moe_expert_gateup ->
    moe_expert_down -> moe_combine

Every step runs in the CUDA library; this class only owns memory.
"""
from __future__ import annotations

import torch

from . import _lib


class MoELayer:
    def __init__(self, w_router, bias, w_gateup, w_down, k: int, T_max: int):
        assert w_router.is_cuda and w_router.dtype == torch.bfloat16
        self.E, self.H = w_router.shape
        self.I = w_gateup.shape[1] // 2
        assert w_gateup.shape == (self.E, 2 * self.I, self.H)
        assert w_down.shape == (self.E, self.H, self.I)
        self.k = k
        self.T_max = T_max
        self.w_router, self.bias, self.w_gateup, self.w_down = w_router, bias, w_gateup, w_down
        dev = w_router.device
        R = T_max * k
        E, H, I = self.E, self.H, self.I
        self.ids = torch.empty((T_max, k), dtype=torch.int32, device=dev)
        self.w = torch.empty((T_max, k), dtype=torch.float32, device=dev)
        self.gap = torch.empty((T_max,), dtype=torch.float32, device=dev)
        ws = _lib.route_workspace_size(T_max, E)
        self.ws = torch.empty((max(ws, 256),), dtype=torch.uint8, device=dev)
        self.counts = torch.empty((E,), dtype=torch.int32, device=dev)
        self.offsets = torch.empty((E + 1,), dtype=torch.int32, device=dev)
        self.perm = torch.empty((R,), dtype=torch.int32, device=dev)
        self.inv = torch.empty((R,), dtype=torch.int32, device=dev)
        self.x_perm = torch.empty((R, H), dtype=torch.bfloat16, device=dev)
        self.h = torch.empty((R, I), dtype=torch.bfloat16, device=dev)
        self.y_perm = torch.empty((R, H), dtype=torch.float32, device=dev)
        self.out = torch.empty((T_max, H), dtype=torch.bfloat16, device=dev)
        self.status = torch.zeros((1,), dtype=torch.int32, device=dev)

    # -- the five calls, exposed one by one so callers can time each --------
    def route(self, x, stream=None):
        T = x.shape[0]
        _lib.moe_route(x, self.w_router, self.bias, self.k, self.ids[:T], self.w[:T], self.gap[:T], self.ws,
                       stream)

    def permute(self, x, stream=None):
        T = x.shape[0]
        R = T * self.k
        _lib.moe_permute(self.ids[:T], self.E, x, self.counts, self.offsets, self.perm[:R], self.inv[:R],
                         self.x_perm[:R], self.status, stream)

    def gateup(self, T, stream=None):
        R = T * self.k
        _lib.moe_expert_gateup(self.x_perm[:R], self.offsets, self.E, self.H, self.I, self.w_gateup, self.h[:R],
                               self.status, stream=stream)

    def down(self, T, stream=None):
        R = T * self.k
        _lib.moe_expert_down(self.h[:R], self.offsets, self.E, self.H, self.I, self.w_down, self.y_perm[:R],
                             self.status, stream=stream)

    def combine(self, T, out=None, stream=None):
        R = T * self.k
        out = self.out[:T] if out is None else out
        _lib.moe_combine(self.y_perm[:R], self.inv[:R], self.w[:T], None, out, None, self.status, stream)
        return out

    def forward(self, x, out=None, stream=None):
        """out[T,H] bf16 = MoE(x) for x [T,H] bf16 on the GPU (asynchronous)."""
        T = x.shape[0]
        assert T <= self.T_max and x.shape[1] == self.H
        if T == 0:
            return self.out[:0] if out is None else out
        self.route(x, stream)
        self.permute(x, stream)
        self.gateup(T, stream)
        self.down(T, stream)
        return self.combine(T, out, stream)

    def forward_host(self, x_host, out_host, x_dev=None, stream=None):
        """Host in, host out: pinned x_host [T,H] bf16 -> out_host [T,H] bf16.

        Copies x to the device, runs the layer, copies the result back, all on
        one stream; returns after the result is in out_host.
        """
        s = torch.cuda.current_stream() if stream is None else stream
        T = x_host.shape[0]
        xd = self.x_dev_buf(T) if x_dev is None else x_dev
        with torch.cuda.stream(s):
            xd.copy_(x_host, non_blocking=True)
            out = self.forward(xd, stream=s)
            out_host.copy_(out, non_blocking=True)
        s.synchronize()
        return out_host

    def x_dev_buf(self, T):
        if not hasattr(self, "_xdev") or self._xdev.shape[0] < T:
            self._xdev = torch.empty((self.T_max, self.H), dtype=torch.bfloat16, device=self.w_router.device)
        return self._xdev[:T]

    def read_status(self) -> int:
        return int(self.status.item())

    def clear_status(self):
        self.status.zero_()
