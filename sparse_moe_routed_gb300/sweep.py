"""Route-prediction and deduplication sweep over a residual MoE stack.

For every layer l of the stack, on all tokens at once:
  * the native route: moe_route on bf16(RMSNorm(x_l)) (the layer's own call);
  * a pre-attention linear predictor: moe_route on bf16(x_l), the
    representation before normalisation, with the predictor weights Wp_l;
  * two zero-training controls of AFN-019 "Hide SSD misses before the router
    knows they exist", section "Hypothesis H2": the native router applied to
    the earlier representation bf16(x_l), and the previous token's
    same-layer route;
  * moe_route_recall of each against the native route;
then route_block_dedup of the native routes over blocks of B consecutive
tokens: unique experts per (layer, block) and the exact routed bytes a block
needs at 2 and 4 bits (AFN-019, sections "Why overlap alone cannot defeat
the byte roofline" and "Hypothesis H7").

Everything runs in the CUDA library; this module only sequences the calls
and moves the per-layer results into stacked tensors.
"""
from __future__ import annotations

import torch

from . import _lib
from .layer import MoELayer, MoEStack


def route_sweep(stack: MoEStack, x0: torch.Tensor, predictors, blocks=(1, 4, 16, 64), stream=None) -> dict:
    """Run the stack on x0 [T,H] fp32 (a copy; x0 is not modified) and score
    route predictors.  predictors[l] is an [E,H] bf16 matrix for layer l.

    Returns device tensors: native/pred/early ids [L,T,k], hits_pred,
    hits_early [L,T], hits_prev [L,T-1], and per block size B: mask, U [L,nb],
    bytes2, bytes4 [nb]; plus host summary statistics under "summary".
    """
    s = torch.cuda.current_stream() if stream is None else stream
    L = len(stack.layers)
    T, H = x0.shape
    first = stack.layers[0]
    E, k, I = first.E, first.k, first.I
    dev = x0.device
    x = x0.clone()
    raw = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
    native = torch.empty((L, T, k), dtype=torch.int32, device=dev)
    pred = torch.empty((L, T, k), dtype=torch.int32, device=dev)
    early = torch.empty((L, T, k), dtype=torch.int32, device=dev)
    hits_pred = torch.empty((L, T), dtype=torch.int32, device=dev)
    hits_early = torch.empty((L, T), dtype=torch.int32, device=dev)
    hits_prev = torch.empty((L, max(T - 1, 0)), dtype=torch.int32, device=dev)
    pw = torch.empty((T, k), dtype=torch.float32, device=dev)
    ws = torch.empty((max(_lib.route_workspace_size(T, E), 256),), dtype=torch.uint8, device=dev)
    with torch.cuda.stream(s):
        for l in range(L):
            for call in stack.layer_calls(x, l, stream=s, raw=raw):
                MoELayer.issue(call)
            native[l].copy_(stack.layers[l].ids[:T])
            _lib.moe_route(raw, predictors[l], None, k, pred[l], pw, None, ws, stream=s)
            _lib.moe_route(raw, stack.layers[l].w_router, None, k, early[l], pw, None, ws, stream=s)
            _lib.moe_route_recall(pred[l], native[l], hits_pred[l], stream=s)
            _lib.moe_route_recall(early[l], native[l], hits_early[l], stream=s)
            if T > 1:
                _lib.moe_route_recall(native[l, :-1], native[l, 1:], hits_prev[l], stream=s)
        status = torch.zeros((1,), dtype=torch.int32, device=dev)
        dedup = {}
        W = (E + 31) // 32
        for B in blocks:
            nb = (T + B - 1) // B
            mask = torch.empty((L, nb, W), dtype=torch.int32, device=dev)
            U = torch.empty((L, nb), dtype=torch.int32, device=dev)
            b2 = torch.empty((nb,), dtype=torch.int64, device=dev)
            b4 = torch.empty((nb,), dtype=torch.int64, device=dev)
            _lib.route_block_dedup(native, E, B, H, I, mask, U, b2, b4, status, stream=s)
            dedup[B] = {"mask": mask, "U": U, "bytes2": b2, "bytes4": b4}
    s.synchronize()
    out = {"native": native, "pred": pred, "early": early, "hits_pred": hits_pred, "hits_early": hits_early,
           "hits_prev": hits_prev, "dedup": dedup, "x_final": x, "status": int(status.item())}
    out["summary"] = summarize(out, k, T, L)
    return out


def summarize(res, k, T, L) -> dict:
    """Host-side means of the sweep's device results (reporting only)."""
    def rate(h):
        return float(h.float().mean().item()) / k if h.numel() else 0.0

    def exact(h):
        return float((h == k).float().mean().item()) if h.numel() else 0.0

    summ = {
        "recall_linear_predictor": rate(res["hits_pred"]),
        "recall_native_router_on_prenorm": rate(res["hits_early"]),
        "recall_previous_token": rate(res["hits_prev"]),
        "exact10_linear_predictor": exact(res["hits_pred"]),
        "exact10_native_router_on_prenorm": exact(res["hits_early"]),
        "exact10_previous_token": exact(res["hits_prev"]),
        "blocks": {},
    }
    for B, d in res["dedup"].items():
        U = d["U"].float()
        nb = U.shape[1]
        summ["blocks"][B] = {
            "mean_U_per_layer": float(U.mean().item()),
            "break_even_ratio_U_over_10B": float((U / (k * B)).mean().item()),
            "unique_layer_expert_per_block": float(U.sum(0).mean().item()),
            "bytes2_per_token": float(d["bytes2"].double().mean().item()) / B,
            "bytes4_per_token": float(d["bytes4"].double().mean().item()) / B,
            "blocks": nb,
        }
    return summ
