"""One routed-expert MoE layer driven through the C ABI.

``MoELayer`` owns the device buffers a layer call needs (allocated once with
torch, sized for ``T_max`` tokens) and issues the boundary calls on one
stream.  With plain or int4 records:

    moe_route -> moe_permute (+ row gather) -> moe_expert_gateup ->
    moe_expert_down -> moe_combine

With tile-packed bf16 records gate/up and down run as one persistent launch,
which for a decode-sized block also gathers the token rows itself:

    moe_route -> moe_permute (+ row gather unless few rows) ->
    moe_expert_swiglu_fused -> moe_combine

(`ROUTE_PERMUTE_ONE_LAUNCH` switches a decode block to moe_route_permute,
which routes and groups in one launch.)

``CachedMoELayer`` keeps the expert records in pinned host memory behind an
HBM slot cache and adds moe_cache_plan (and, copy-first, moe_cache_fetch)
before moe_expert_swiglu_cached.

Every step runs in the CUDA library; this class only owns memory.
"""
from __future__ import annotations

import ctypes as C

import torch

from . import _lib


class MoELayer:
    """Buffers and calls of one layer.

    bf16 weights: w_gateup [E,2I,H] bf16, w_down [E,H,I] bf16.
    packed weights (fmt=MOE_W_BF16_TILED or MOE_W_INT4_G64_TILED): the uint8
    buffers moe_pack_experts wrote for the gate/up and down components (pass I).
    """

    GATHER_IN_FUSED_MAX_ROWS = 4096
    ROUTE_PERMUTE_ONE_LAUNCH = False
    # fused launches of more routes than this store the expert outputs as
    # bf16 rows already multiplied by their route weights (half the bytes of
    # fp32 rows, written once and read once by the combine)
    WEIGHTED_Y_MIN_ROWS = 4097
    # from this many routes the grouping runs in chunks on many CTAs
    # (moe_permute_ws); below it one CTA does it in one launch
    PERMUTE_CHUNKED_MIN_ROWS = 8192
    WEIGHTED_Y = True

    def __init__(self, w_router, bias, w_gateup, w_down, k: int, T_max: int, fmt: int = _lib.MOE_W_BF16,
                 I: int = None):
        assert w_router.is_cuda and w_router.dtype == torch.bfloat16
        self.E, self.H = w_router.shape
        self.fmt = fmt
        if fmt == _lib.MOE_W_BF16:
            self.I = w_gateup.shape[1] // 2
            assert w_gateup.shape == (self.E, 2 * self.I, self.H)
            assert w_down.shape == (self.E, self.H, self.I)
        else:
            assert fmt in (_lib.MOE_W_BF16_TILED, _lib.MOE_W_INT4_G64_TILED) and I is not None
            self.I = I
            src = _lib.MOE_W_BF16 if fmt == _lib.MOE_W_BF16_TILED else _lib.MOE_W_INT4_G64
            assert w_gateup.numel() * w_gateup.element_size() == _lib.pack_size(src, self.E, self.H, I, 0)
            assert w_down.numel() * w_down.element_size() == _lib.pack_size(src, self.E, self.H, I, 1)
        self.k = k
        self.T_max = T_max
        self.w_router, self.bias, self.w_gateup, self.w_down = w_router, bias, w_gateup, w_down
        dev = w_router.device
        R = T_max * k
        E, H, I = self.E, self.H, self.I
        self.ids = torch.empty((T_max, k), dtype=torch.int32, device=dev)
        self.w = torch.empty((T_max, k), dtype=torch.float32, device=dev)
        self.gap = torch.empty((T_max,), dtype=torch.float32, device=dev)
        # one workspace for the router's logits and, later in the chain, the
        # chunked grouping's per-chunk counts
        ws = max(_lib.route_workspace_size(T_max, E), _lib.moe_permute_workspace_size(T_max, k, E))
        self.ws = torch.empty((max(ws, 256),), dtype=torch.uint8, device=dev)
        self.counts = torch.empty((E,), dtype=torch.int32, device=dev)
        self.offsets = torch.empty((E + 1,), dtype=torch.int32, device=dev)
        self.perm = torch.empty((R,), dtype=torch.int32, device=dev)
        self.inv = torch.empty((R,), dtype=torch.int32, device=dev)
        self.x_perm = torch.empty((R, H), dtype=torch.bfloat16, device=dev)
        self.h = torch.empty((R, I), dtype=torch.bfloat16, device=dev)
        self.y_perm = torch.empty((R, H), dtype=torch.float32, device=dev)
        # the weighted bf16 rows share y_perm's storage (its first R*H*2 bytes)
        self.yw_perm = self.y_perm.view(-1).view(torch.bfloat16)[:R * H].view(R, H)
        self.out = torch.empty((T_max, H), dtype=torch.bfloat16, device=dev)
        self.status = torch.zeros((1,), dtype=torch.int32, device=dev)
        self.fused = (fmt == _lib.MOE_W_BF16_TILED)
        self.sync_ws = torch.zeros((E + 3,), dtype=torch.int32, device=dev)
        self._bound = {}

    # -- the five boundary calls, bound once per (T, x, out, stream) ---------
    def bound_calls(self, x, T=None, out=None, stream=None, residual=None, out_f32=None, route=True):
        """[(name, fn, args)] of the C-ABI calls for this input.

        Pointers and sizes are converted to ctypes once and cached, so issuing
        a layer costs five foreign calls and nothing else on the host.  With
        residual/out_f32 the combine adds the fp32 residual and writes fp32
        (the residual stream of a stack); route=False leaves out moe_route
        (the caller filled self.ids / self.w).
        """
        T = x.shape[0] if T is None else T
        s = torch.cuda.current_stream() if stream is None else stream
        if out_f32 is None:
            out = self.out[:T] if out is None else out
        key = (T, x.data_ptr(), None if out is None else out.data_ptr(), s.cuda_stream,
               None if residual is None else residual.data_ptr(), None if out_f32 is None else out_f32.data_ptr(),
               route)
        calls = self._bound.get(key)
        if calls is not None:
            return calls
        if len(self._bound) > 64:
            self._bound.clear()
        lib = _lib.load()
        P = _lib._ptr
        st = C.c_void_p(s.cuda_stream)
        R = T * self.k
        E, H, I, k = self.E, self.H, self.I, self.k
        ws_bytes = self.ws.numel()
        calls = []
        # moe_route_permute (route + grouping in one 16-CTA cluster launch) is
        # slower on GB300 than the logits -> top-k -> grouping chain here: a
        # single cluster pulls the router matrix through 16 SMs.  Kept off.
        route_and_group = route and T <= 16 and self.ROUTE_PERMUTE_ONE_LAUNCH
        if route_and_group:
            calls.append(("moe_route_permute", lib.moe_route_permute,
                          (P(x), P(self.w_router), P(self.bias), T, H, E, k, P(self.ids), P(self.w), P(self.gap),
                           P(self.counts), P(self.offsets), P(self.perm), P(self.inv), P(self.status), st)))
        elif route:
            calls.append(("moe_route", lib.moe_route,
                          (P(x), P(self.w_router), P(self.bias), T, H, E, k, P(self.ids), P(self.w), P(self.gap),
                           P(self.ws), ws_bytes, st)))
        # the fused launch gathers the token rows itself when there are few
        # (a decode block); for many rows moe_permute's gather runs at full
        # occupancy instead
        gather_in_fused = self.fused and R <= self.GATHER_IN_FUSED_MAX_ROWS
        if not route_and_group and R >= self.PERMUTE_CHUNKED_MIN_ROWS:
            calls.append(("moe_permute_ws", lib.moe_permute_ws,
                          (P(self.ids), T, k, E, None if gather_in_fused else P(x), H, P(self.counts),
                           P(self.offsets), P(self.perm), P(self.inv),
                           None if gather_in_fused else P(self.x_perm), P(self.ws), ws_bytes, P(self.status), st)))
        elif not route_and_group:
            calls.append(("moe_permute", lib.moe_permute,
                          (P(self.ids), T, k, E, None if gather_in_fused else P(x), H, P(self.counts),
                           P(self.offsets), P(self.perm), P(self.inv),
                           None if gather_in_fused else P(self.x_perm), P(self.status), st)))
        elif not gather_in_fused:
            # grouped already; gather the rows separately
            calls.append(("moe_permute_gather", lib.moe_permute,
                          (P(self.ids), T, k, E, P(x), H, P(self.counts), P(self.offsets), P(self.perm),
                           P(self.inv), P(self.x_perm), P(self.status), st)))
        weighted = self.fused and self.WEIGHTED_Y and R >= self.WEIGHTED_Y_MIN_ROWS
        if weighted:
            calls.append(("moe_expert_swiglu_fused_weighted", lib.moe_expert_swiglu_fused_weighted,
                          (P(x if gather_in_fused else None), k, P(self.perm), P(self.x_perm), P(self.offsets), R,
                           E, H, I, self.fmt, P(self.w_gateup), P(self.w_down), P(self.w), P(self.h),
                           P(self.yw_perm), P(self.sync_ws), P(self.status), st)))
        elif self.fused:
            calls += self._expert_calls(lib, P, x if gather_in_fused else None, R, st)
        else:
            calls += self._two_launch_expert_calls(lib, P, R, st)
        if weighted:
            calls.append(("moe_combine_weighted", lib.moe_combine_weighted,
                          (P(self.yw_perm), P(self.inv), T, k, H, P(residual), P(out), P(out_f32), P(self.status),
                           st)))
        else:
            calls.append(("moe_combine", lib.moe_combine,
                          (P(self.y_perm), P(self.inv), P(self.w), T, k, H, P(residual), P(out), P(out_f32),
                           P(self.status), st)))
        self._bound[key] = calls
        return calls

    def _two_launch_expert_calls(self, lib, P, R, st):
        E, H, I = self.E, self.H, self.I
        return [
            ("moe_expert_gateup", lib.moe_expert_gateup,
             (P(self.x_perm), P(self.offsets), R, E, H, I, self.fmt, P(self.w_gateup), None, P(self.h),
              P(self.status), st)),
            ("moe_expert_down", lib.moe_expert_down,
             (P(self.h), P(self.offsets), R, E, H, I, self.fmt, P(self.w_down), None, P(self.y_perm),
              P(self.status), st)),
        ]

    def _expert_calls(self, lib, P, x_gather, R, st):
        return [("moe_expert_swiglu_fused", lib.moe_expert_swiglu_fused,
                 (P(x_gather), self.k, P(self.perm), P(self.x_perm), P(self.offsets), R, self.E, self.H, self.I,
                  self.fmt, P(self.w_gateup), P(self.w_down), P(self.h), P(self.y_perm), P(self.sync_ws),
                  P(self.status), st))]

    @staticmethod
    def issue(call):
        name, fn, args = call
        st = fn(*args)
        if st != 0:
            raise _lib.MoEError(name, st, _lib.status_str(st))

    def forward(self, x, out=None, stream=None):
        """out[T,H] bf16 = MoE(x) for x [T,H] bf16 on the GPU (asynchronous)."""
        T = x.shape[0]
        assert T <= self.T_max and x.shape[1] == self.H and x.dtype == torch.bfloat16
        if T == 0:
            return self.out[:0] if out is None else out
        for call in self.bound_calls(x, T, out, stream):
            self.issue(call)
        return self.out[:T] if out is None else out

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

    def forward_host_graph(self, x_host, out_host):
        """forward_host replayed from a CUDA graph.

        The host-to-device copy of x, the layer's launches and the copy of the
        result back are captured once per (x_host, out_host) pair and then
        replayed: one graph launch per call instead of seven API calls.  The
        graph reads x_host and writes out_host by address, so the caller
        refills the same pinned buffers between calls.  Returns after the
        result is in out_host.
        """
        MoELayer.wait(self.forward_host_submit(x_host, out_host))
        return out_host

    def forward_host_submit(self, x_host, out_host):
        """forward_host_graph without the wait: enqueues the graph (input copy,
        the layer's launches, result copy) on the current stream and returns
        an event that completes once out_host holds the result.  Until then
        the caller leaves x_host and out_host alone; calls queued on the same
        stream run in order, so a caller may queue the next call (with other
        host buffers) before it waits for this one."""
        key = (x_host.data_ptr(), out_host.data_ptr(), x_host.shape[0])
        graphs = self.__dict__.setdefault("_graphs", {})
        graph = graphs.get(key)
        if graph is None:
            T = x_host.shape[0]
            xd = self.x_dev_buf(T)
            s = torch.cuda.Stream(device=xd.device)
            s.wait_stream(torch.cuda.current_stream())

            def body():
                xd.copy_(x_host, non_blocking=True)
                out = self.forward(xd, stream=s)
                out_host.copy_(out, non_blocking=True)

            with torch.cuda.stream(s):  # one eager pass: first-call set-up stays out of the capture
                body()
            s.synchronize()
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph, stream=s):
                body()
            graphs[key] = graph
        graph.replay()
        done = torch.cuda.Event()
        done.record()
        return done

    def forward_host_pipelined(self, x_host, out_host):
        """forward_host_submit with the two copies off the compute stream.

        The host-to-device copy of x runs on a copy stream into one of two
        device input buffers, the layer's launches (a CUDA graph per buffer
        pair, captured once) on the current stream after that copy, and the
        copy of the result back on a second copy stream, so that a call's
        input copy overlaps the previous call's compute and its result copy
        the next call's.  Returns an event that completes once out_host holds
        the result; until then the caller leaves x_host and out_host alone.
        Calls run their layer work in order on the current stream.
        """
        T = x_host.shape[0]
        st = self.__dict__.get("_pipe")
        if st is None or st["T"] != T:
            dev = self.w_router.device
            st = {"T": T, "n": 0,
                  "h2d": torch.cuda.Stream(device=dev), "d2h": torch.cuda.Stream(device=dev),
                  # zero-filled: the first call's eager pass (before the capture) reads them
                  "x": [torch.zeros((T, self.H), dtype=torch.bfloat16, device=dev) for _ in range(2)],
                  "out": [torch.empty((T, self.H), dtype=torch.bfloat16, device=dev) for _ in range(2)],
                  "x_ready": [torch.cuda.Event() for _ in range(2)],
                  "layer_done": [torch.cuda.Event() for _ in range(2)],
                  "out_free": [torch.cuda.Event() for _ in range(2)],
                  "graphs": [None, None]}
            for b in range(2):
                st["layer_done"][b].record()
                st["out_free"][b].record()
            self._pipe = st
        b = st["n"] & 1
        st["n"] += 1
        cur = torch.cuda.current_stream()
        if st["graphs"][b] is None:
            s = torch.cuda.Stream(device=cur.device)
            s.wait_stream(cur)
            with torch.cuda.stream(s):  # one eager pass: first-call set-up stays out of the capture
                self.forward(st["x"][b], out=st["out"][b], stream=s)
            s.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=s):
                self.forward(st["x"][b], out=st["out"][b], stream=s)
            st["graphs"][b] = g
        # input copy, once the layer that last read this buffer is done
        h2d = st["h2d"]
        h2d.wait_event(st["layer_done"][b])
        with torch.cuda.stream(h2d):
            st["x"][b].copy_(x_host, non_blocking=True)
        st["x_ready"][b].record(h2d)
        # the layer, once its input has landed and its output buffer is free
        cur.wait_event(st["x_ready"][b])
        cur.wait_event(st["out_free"][b])
        st["graphs"][b].replay()
        st["layer_done"][b].record(cur)
        # the result copy
        d2h = st["d2h"]
        d2h.wait_event(st["layer_done"][b])
        with torch.cuda.stream(d2h):
            out_host.copy_(st["out"][b], non_blocking=True)
        done = torch.cuda.Event()
        done.record(d2h)
        st["out_free"][b].record(d2h)
        return done

    @staticmethod
    def wait(done):
        """Block until a call returned by forward_host_submit has finished."""
        done.synchronize()

    def x_dev_buf(self, T):
        if not hasattr(self, "_xdev") or self._xdev.shape[0] < T:
            self._xdev = torch.empty((self.T_max, self.H), dtype=torch.bfloat16, device=self.w_router.device)
        return self._xdev[:T]

    def read_status(self) -> int:
        return int(self.status.item())

    def clear_status(self):
        """Zero the device status word (and the fused launch's sync words,
        which a launch that gave up on a wait may have left non-zero)."""
        self.status.zero_()
        self.sync_ws.zero_()


class CachedMoELayer(MoELayer):
    """A layer whose expert records live in host memory behind an HBM cache.

    host_gateup / host_down: the tile-packed records (moe_pack_experts
    output, MOE_W_BF16_TILED or MOE_W_INT4_G64_TILED) of all E experts in
    pinned host memory, which the GPU reads directly over the CPU-GPU link.
    S slots of HBM hold recently used experts.  Each call plans hits and
    misses on the device (moe_cache_plan) and then either fetches the misses
    in the expert launch itself, in waves of `wave` experts while the
    resident experts compute (fetch="wave"), or copies them first with
    moe_cache_fetch and computes after (fetch="barrier").  int4 records move
    2,611,200 B per miss at the Qwen4Exp shape against 9,830,400 B in bf16;
    their in-launch fetch is done by the gate/up launch for both components.
    Outputs are bit-identical to MoELayer over the same records in HBM.

        moe_route -> moe_permute -> moe_cache_plan [-> moe_cache_fetch] ->
        moe_expert_swiglu_cached (bf16) | moe_expert_int4_fetch or
        moe_expert_int4_slots, then moe_expert_int4_slots (int4) -> moe_combine

    stats [4] int32 on the device: {hits, misses} of the last call and their
    running totals.  policy: "fifo", "lru" or "score" (moe_cache_plan), decay
    the score policy's use-rate factor.
    """

    WEIGHTED_Y = False  # the cached launches keep fp32 expert outputs

    POLICIES = {"fifo": _lib.MOE_CACHE_FIFO, "lru": _lib.MOE_CACHE_LRU, "score": _lib.MOE_CACHE_SCORE}

    def __init__(self, w_router, bias, host_gateup, host_down, k: int, T_max: int, I: int, S: int,
                 wave: int = 1 << 20, fetch: str = "wave", policy: str = "fifo", decay: float = 0.9,
                 fmt: int = _lib.MOE_W_BF16_TILED):
        assert not host_gateup.is_cuda and host_gateup.is_pinned() and host_down.is_pinned()
        assert fetch in ("wave", "barrier") and policy in self.POLICIES
        assert fmt in (_lib.MOE_W_BF16_TILED, _lib.MOE_W_INT4_G64_TILED)
        self.policy, self.decay = self.POLICIES[policy], float(decay)
        super().__init__(w_router, bias, host_gateup, host_down, k, T_max, fmt=fmt, I=I)
        E, H = self.E, self.H
        dev = w_router.device
        self.S, self.wave, self.fetch = S, wave, fetch
        self.rec_gu = host_gateup.numel() * host_gateup.element_size() // E
        self.rec_dn = host_down.numel() * host_down.element_size() // E
        self.pool_gu = torch.empty((S * self.rec_gu,), dtype=torch.uint8, device=dev)
        self.pool_dn = torch.empty((S * self.rec_dn,), dtype=torch.uint8, device=dev)
        self.slot_of = torch.full((E,), -1, dtype=torch.int32, device=dev)
        self.expert_of = torch.full((S,), -1, dtype=torch.int32, device=dev)
        self.hand = torch.zeros((2,), dtype=torch.int32, device=dev)
        self.score = torch.zeros((E,), dtype=torch.float32, device=dev)
        self.last_use = torch.full((S,), -1, dtype=torch.int32, device=dev)
        self.miss_list = torch.zeros((S,), dtype=torch.int32, device=dev)
        self.miss_slot = torch.zeros((S,), dtype=torch.int32, device=dev)
        self.stats = torch.zeros((4,), dtype=torch.int32, device=dev)
        self.sync_ws = torch.zeros((E * (1 + self.I // 64 + H // 128) + 4,), dtype=torch.int32, device=dev)

    def reset_cache(self):
        """Empty the cache and zero the running totals."""
        self.slot_of.fill_(-1)
        self.expert_of.fill_(-1)
        self.hand.zero_()
        self.score.zero_()
        self.last_use.fill_(-1)
        self.stats.zero_()

    def _two_launch_expert_calls(self, lib, P, R, st):
        # int4 records: plan, then either the gate/up launch fetches the
        # misses of both components while the resident experts compute
        # (wave), or the misses are copied first (barrier); the int4
        # contraction reads every expert from its slot
        E, H, I, S = self.E, self.H, self.I, self.S
        wave = self.fetch == "wave"
        calls = self._plan_calls(lib, P, st, fetch_first=not wave)
        if wave:
            calls.append(("moe_expert_int4_fetch", lib.moe_expert_int4_fetch,
                          (P(self.x_perm), P(self.offsets), R, E, H, I, P(self.pool_gu), P(self.pool_dn), S,
                           P(self.slot_of), P(self.w_gateup), P(self.w_down), P(self.miss_list), P(self.miss_slot),
                           P(self.stats), P(self.h), P(self.sync_ws), P(self.status), st)))
        else:
            calls.append(("moe_expert_int4_slots", lib.moe_expert_int4_slots,
                          (0, P(self.x_perm), P(self.offsets), R, E, H, I, P(self.pool_gu), S, P(self.slot_of),
                           P(self.h), P(self.status), st)))
        calls.append(("moe_expert_int4_slots", lib.moe_expert_int4_slots,
                      (1, P(self.h), P(self.offsets), R, E, H, I, P(self.pool_dn), S, P(self.slot_of), P(self.y_perm),
                       P(self.status), st)))
        return calls

    def _plan_calls(self, lib, P, st, fetch_first):
        E, S = self.E, self.S
        calls = [("moe_cache_plan", lib.moe_cache_plan,
                  (P(self.counts), E, P(self.slot_of), P(self.expert_of), S, P(self.hand), self.policy,
                   C.c_float(self.decay), P(self.score), P(self.last_use), P(self.miss_list), P(self.miss_slot),
                   P(self.stats), P(self.status), st))]
        if fetch_first:
            calls.append(("moe_cache_fetch", lib.moe_cache_fetch,
                          (P(self.w_gateup), P(self.w_down), self.rec_gu, self.rec_dn, P(self.miss_list),
                           P(self.miss_slot), P(self.stats), P(self.pool_gu), P(self.pool_dn), st)))
        return calls

    def _expert_calls(self, lib, P, x_gather, R, st):
        E, H, I, S = self.E, self.H, self.I, self.S
        wave = self.fetch == "wave"
        calls = self._plan_calls(lib, P, st, fetch_first=not wave)
        calls.append(("moe_expert_swiglu_cached", lib.moe_expert_swiglu_cached,
                      (P(x_gather), self.k, P(self.perm), P(self.x_perm), P(self.offsets), R, E, H, I, self.fmt,
                       P(self.pool_gu), P(self.pool_dn), S, P(self.slot_of),
                       P(self.w_gateup) if wave else None, P(self.w_down) if wave else None,
                       P(self.miss_list), P(self.miss_slot), P(self.stats), self.wave, P(self.h), P(self.y_perm),
                       P(self.sync_ws), P(self.status), st)))
        return calls


class MoEStack:
    """A residual stack of MoE layers: x <- x + MoE_l(RMSNorm(x)), l = 0..L-1.

    x is an fp32 residual stream [T,H] updated in place; each layer runs
    moe_rmsnorm (fp32 -> bf16, zero-centred gain 1 + gamma) and the five layer
    calls, the combine adding the residual and writing fp32 back into x.
    """

    def __init__(self, layers, T_max: int, eps: float = 1e-6, gammas=None):
        self.layers = list(layers)
        self.eps = eps
        self.gammas = gammas
        H = self.layers[0].H
        dev = self.layers[0].w_router.device
        self.T_max = T_max
        self.n = torch.empty((T_max, H), dtype=torch.bfloat16, device=dev)
        self._norm_bound = {}

    def _norm_call(self, x, l, s, raw=None):
        key = (x.data_ptr(), x.shape[0], l, s.cuda_stream, None if raw is None else raw.data_ptr())
        c = self._norm_bound.get(key)
        if c is None:
            lib = _lib.load()
            P = _lib._ptr
            g = None if self.gammas is None else self.gammas[l]
            T, H = x.shape
            c = ("moe_rmsnorm", lib.moe_rmsnorm,
                 (P(x), P(g), C.c_float(self.eps), T, H, P(self.n), P(raw), C.c_void_p(s.cuda_stream)))
            if len(self._norm_bound) > 4096:
                self._norm_bound.clear()
            self._norm_bound[key] = c
        return c

    def layer_calls(self, x, l, stream=None, route=True, raw=None):
        """Calls of layer l on the residual stream x; raw (optional, [T,H]
        bf16) receives x rounded to bf16 before normalisation."""
        s = torch.cuda.current_stream() if stream is None else stream
        T = x.shape[0]
        L = self.layers[l]
        return [self._norm_call(x, l, s, raw)] + L.bound_calls(self.n[:T], T, stream=s, residual=x, out_f32=x,
                                                              route=route)

    def forward(self, x, stream=None, layers=None):
        """x [T,H] fp32 on the GPU, updated in place through the layers."""
        assert x.dtype == torch.float32 and x.is_contiguous()
        for l in (range(len(self.layers)) if layers is None else layers):
            for call in self.layer_calls(x, l, stream):
                MoELayer.issue(call)
        return x


class PrefillRing:
    """Macro prefill with every layer's records in host memory.

    A prefill tile routes to most experts of a layer, so the layer's records
    are streamed whole (moe_layer_stream, copy engines) into a two-layer HBM
    ring: layer l + 1 lands in one ring slot while layer l computes from the
    other, and the copy into a slot waits until the layer that last used it
    is done (AFN-019, section "Hypothesis H5: prefill and decode need
    different streaming modes").  The residual stack is MoEStack's:
    x <- x + MoE_l(RMSNorm(x)); the output is bit-identical to MoEStack over
    the same records resident in HBM.

    routers: [(w_router [E,H] bf16, bias or None)] per layer (device);
    host_records: [(gate/up, down)] per layer, the pinned uint8 buffers of
    moe_pack_experts (MOE_W_BF16_TILED layout), same sizes for all layers.
    """

    def __init__(self, routers, host_records, k: int, T_max: int, I: int, eps: float = 1e-6, gammas=None):
        assert len(routers) == len(host_records) >= 1
        dev = routers[0][0].device
        gu0, dn0 = host_records[0]
        for gu, dn in host_records:
            assert gu.is_pinned() and dn.is_pinned() and gu.numel() == gu0.numel() and dn.numel() == dn0.numel()
        self.ring = [(torch.empty(gu0.shape, dtype=torch.uint8, device=dev),
                      torch.empty(dn0.shape, dtype=torch.uint8, device=dev)) for _ in range(2)]
        layers = [MoELayer(wr, b, *self.ring[l % 2], k, T_max, fmt=_lib.MOE_W_BF16_TILED, I=I)
                  for l, (wr, b) in enumerate(routers)]
        self.stack = MoEStack(layers, T_max, eps, gammas)
        self.host = list(host_records)
        self.copy_stream = torch.cuda.Stream(device=dev)

    def forward(self, x, stream=None):
        """x [T,H] fp32 residual stream on the GPU, updated in place."""
        s = torch.cuda.current_stream() if stream is None else stream
        cs = self.copy_stream
        L = len(self.host)
        copied = [torch.cuda.Event() for _ in range(L)]
        done = [torch.cuda.Event() for _ in range(L)]
        cs.wait_stream(s)  # the ring is free once earlier work on s is done

        def fill(l):
            if l >= 2:
                cs.wait_event(done[l - 2])
            _lib.moe_layer_stream(*self.host[l], *self.ring[l % 2], stream=cs)
            copied[l].record(cs)

        fill(0)
        if L > 1:
            fill(1)
        for l in range(L):
            s.wait_event(copied[l])
            for call in self.stack.layer_calls(x, l, stream=s):
                MoELayer.issue(call)
            done[l].record(s)
            if l + 2 < L:
                fill(l + 2)
        return x


def pack_layer_experts(w_gateup, w_down, fmt_in, E, H, I, s_gateup=None, s_down=None, stream=None):
    """(packed gate/up, packed down) uint8 device tensors for MoELayer."""
    gu = _lib.moe_pack_experts(fmt_in, w_gateup, s_gateup, E, H, I, 0, stream=stream)
    dn = _lib.moe_pack_experts(fmt_in, w_down, s_down, E, H, I, 1, stream=stream)
    return gu, dn

