"""Host-side checks of the C ABI that need no GPU.

The library must load, export every function include/moe.h declares, and
reject bad arguments on the host before anything is enqueued.  The rejection
cases here use placeholder addresses, so every one of them must be refused by
host admission before any device work; they run only where no GPU is visible.
"""
import ctypes as C

import pytest
import torch

from sparse_moe_routed_gb300 import _lib

pytestmark = pytest.mark.skipif(torch.cuda.is_available(), reason="placeholder pointers: CPU-only host checks")

P = C.c_void_p(1 << 20)      # 16-byte aligned placeholder address
PM = C.c_void_p((1 << 20) + 2)  # misaligned placeholder address
NUL = None


def lib():
    return _lib.load()


def test_library_loads_and_exports_every_declared_symbol():
    L = lib()
    names = _lib.declared_functions()
    assert len(names) == 31
    for n in names:
        assert hasattr(L, n), n
    assert L.moe_abi_version() == 104
    assert L.moe_status_str(0).decode() == "MOE_OK"
    assert L.moe_status_str(5).decode().startswith("MOE_ENOTSUP")


def test_exports_match_header_exactly():
    import subprocess
    out = subprocess.run(["nm", "-D", "--defined-only", _lib._build.LIB], capture_output=True, text=True).stdout
    exported = sorted(l.split()[-1] for l in out.splitlines() if " T " in l)
    assert exported == _lib.declared_functions()


def test_workspace_size():
    L = lib()
    assert L.moe_route_workspace_size(16, 512) == 16 * 512 * 4
    assert L.moe_route_workspace_size(3, 7) == 256
    assert L.moe_route_workspace_size(0, 512) == 0


def _route(**kw):
    a = dict(x=P, wr=P, bias=NUL, T=16, H=2560, E=512, k=10, ids=P, w=P, gap=NUL, ws=P,
             wsb=16 * 512 * 4, st=NUL)
    a.update(kw)
    return lib().moe_route(a["x"], a["wr"], a["bias"], a["T"], a["H"], a["E"], a["k"], a["ids"], a["w"],
                           a["gap"], a["ws"], a["wsb"], a["st"])


@pytest.mark.parametrize("kw,code", [
    (dict(x=NUL), _lib.MOE_EINVAL),
    (dict(wr=NUL), _lib.MOE_EINVAL),
    (dict(ids=NUL), _lib.MOE_EINVAL),
    (dict(w=NUL), _lib.MOE_EINVAL),
    (dict(x=PM), _lib.MOE_EINVAL),
    (dict(T=-1), _lib.MOE_ESHAPE),
    (dict(H=0), _lib.MOE_ESHAPE),
    (dict(H=2500), _lib.MOE_ENOTSUP),
    (dict(k=0), _lib.MOE_ESHAPE),
    (dict(k=33), _lib.MOE_ENOTSUP),
    (dict(E=8, k=10), _lib.MOE_ENOTSUP),
    (dict(E=1025), _lib.MOE_ENOTSUP),
    (dict(ws=NUL), _lib.MOE_EWORKSPACE),
    (dict(wsb=16 * 512 * 4 - 1), _lib.MOE_EWORKSPACE),
])
def test_route_rejections(kw, code):
    assert _route(**kw) == code


@pytest.mark.parametrize("kw", [dict(k=32), dict(E=1024), dict(E=1024, k=32, wsb=16 * 1024 * 4),
                                dict(E=32, k=32)])
def test_route_last_accepted_shapes_are_admitted(kw):
    """The largest accepted k and E pass host admission (and reach the
    device, absent here)."""
    if "wsb" not in kw and kw.get("E", 512) * 16 * 4 > 16 * 512 * 4:
        kw["wsb"] = kw["E"] * 16 * 4
    assert _route(**kw) == _lib.MOE_ECUDA


def test_permute_last_accepted_expert_count_is_admitted():
    assert _permute(E=1024) == _lib.MOE_ECUDA
    assert _permute(E=1025) == _lib.MOE_ENOTSUP


def test_route_zero_tokens_is_noop():
    assert _route(T=0, ws=NUL, wsb=0) == _lib.MOE_OK


def _permute(**kw):
    a = dict(ids=P, T=16, k=10, E=512, x=P, H=2560, counts=P, offsets=P, perm=P, inv=P, xp=P, st=P)
    a.update(kw)
    return lib().moe_permute(a["ids"], a["T"], a["k"], a["E"], a["x"], a["H"], a["counts"], a["offsets"],
                             a["perm"], a["inv"], a["xp"], a["st"], NUL)


@pytest.mark.parametrize("kw,code", [
    (dict(ids=NUL), _lib.MOE_EINVAL),
    (dict(st=NUL), _lib.MOE_EINVAL),
    (dict(x=NUL), _lib.MOE_EINVAL),
    (dict(xp=PM), _lib.MOE_EINVAL),
    (dict(T=-3), _lib.MOE_ESHAPE),
    (dict(k=11, E=10), _lib.MOE_ENOTSUP),
    (dict(H=100), _lib.MOE_ENOTSUP),
    (dict(E=2048), _lib.MOE_ENOTSUP),
    (dict(T=1 << 28, k=10), _lib.MOE_ENOTSUP),
])
def test_permute_rejections(kw, code):
    assert _permute(**kw) == code


def _permute_ws(**kw):
    a = dict(ids=P, T=4096, k=10, E=512, x=P, H=2560, counts=P, offsets=P, perm=P, inv=P, xp=P, ws=P,
             wsb=1 << 20, st=P)
    a.update(kw)
    return lib().moe_permute_ws(a["ids"], a["T"], a["k"], a["E"], a["x"], a["H"], a["counts"], a["offsets"],
                                a["perm"], a["inv"], a["xp"], a["ws"], a["wsb"], a["st"], NUL)


def test_permute_workspace_size():
    L = lib()
    # 20 chunks of 2,048 routes: [20][512] counts, 20 flags, one abort word
    assert L.moe_permute_workspace_size(4096, 10, 512) == (20 * 512 + 20 + 1) * 4 // 256 * 256 + 256
    assert L.moe_permute_workspace_size(1, 1, 1) == 256
    assert L.moe_permute_workspace_size(0, 10, 512) == 0


@pytest.mark.parametrize("kw,code", [
    (dict(ids=NUL), _lib.MOE_EINVAL),
    (dict(st=NUL), _lib.MOE_EINVAL),
    (dict(x=NUL), _lib.MOE_EINVAL),
    (dict(xp=PM), _lib.MOE_EINVAL),
    (dict(ws=NUL), _lib.MOE_EWORKSPACE),
    (dict(ws=PM), _lib.MOE_EINVAL),
    (dict(wsb=1024), _lib.MOE_EWORKSPACE),
    (dict(T=-3), _lib.MOE_ESHAPE),
    (dict(k=11, E=10), _lib.MOE_ENOTSUP),
    (dict(H=100), _lib.MOE_ENOTSUP),
    (dict(E=2048), _lib.MOE_ENOTSUP),
    (dict(T=1 << 28, k=10), _lib.MOE_ENOTSUP),
])
def test_permute_ws_rejections(kw, code):
    assert _permute_ws(**kw) == code


def test_permute_ws_zero_tokens_is_noop():
    assert _permute_ws(T=0, ws=NUL, wsb=0) == _lib.MOE_OK


def _gateup(**kw):
    a = dict(xp=P, off=P, R=160, E=512, H=2560, I=640, fmt=0, w=P, s=NUL, h=P, st=P)
    a.update(kw)
    return lib().moe_expert_gateup(a["xp"], a["off"], a["R"], a["E"], a["H"], a["I"], a["fmt"], a["w"], a["s"],
                                   a["h"], a["st"], NUL)


@pytest.mark.parametrize("kw,code", [
    (dict(xp=NUL), _lib.MOE_EINVAL),
    (dict(off=NUL), _lib.MOE_EINVAL),
    (dict(h=PM), _lib.MOE_EINVAL),
    (dict(fmt=7), _lib.MOE_EINVAL),
    (dict(s=P), _lib.MOE_EINVAL),
    (dict(R=-1), _lib.MOE_ESHAPE),
    (dict(I=600), _lib.MOE_ENOTSUP),
    (dict(H=2496), _lib.MOE_ENOTSUP),
])
def test_gateup_rejections(kw, code):
    assert _gateup(**kw) == code


def test_expert_zero_rows_is_noop():
    assert _gateup(R=0) == _lib.MOE_OK


def test_combine_rejections():
    L = lib()
    assert L.moe_combine(P, P, P, 16, 10, 2560, NUL, NUL, NUL, NUL, NUL) == _lib.MOE_EINVAL
    assert L.moe_combine(PM, P, P, 16, 10, 2560, NUL, P, NUL, NUL, NUL) == _lib.MOE_EINVAL
    assert L.moe_combine(P, P, P, 16, 40, 2560, NUL, P, NUL, NUL, NUL) == _lib.MOE_ENOTSUP
    assert L.moe_combine(P, P, P, 0, 10, 2560, NUL, P, NUL, NUL, NUL) == _lib.MOE_OK


def test_dedup_rejections():
    L = lib()
    assert L.route_block_dedup(P, 48, 512, 10, 512, 0, 2560, 640, P, P, P, P, P, NUL) == _lib.MOE_ESHAPE
    assert L.route_block_dedup(NUL, 48, 512, 10, 512, 4, 2560, 640, P, P, P, P, P, NUL) == _lib.MOE_EINVAL
    assert L.route_block_dedup(P, 48, 512, 10, 512, 4, 2560, 640, P, P, C.c_void_p((1 << 20) + 4), P, P,
                               NUL) == _lib.MOE_EINVAL
    assert L.route_block_dedup(P, 48, 512, 10, 4096, 4, 2560, 640, P, P, P, P, P, NUL) == _lib.MOE_ENOTSUP


def test_rmsnorm_rejections():
    L = lib()
    assert L.moe_rmsnorm(P, NUL, C.c_float(-1.0), 4, 2560, P, NUL, NUL) == _lib.MOE_EINVAL
    assert L.moe_rmsnorm(P, NUL, C.c_float(1e-6), 4, 2500, P, NUL, NUL) == _lib.MOE_ENOTSUP
    assert L.moe_rmsnorm(NUL, NUL, C.c_float(1e-6), 4, 2560, P, NUL, NUL) == _lib.MOE_EINVAL
    assert L.moe_rmsnorm(P, NUL, C.c_float(1e-6), 4, 2560, P, PM, NUL) == _lib.MOE_EINVAL


def test_recall_rejections():
    L = lib()
    assert L.moe_route_recall(P, NUL, 4, 10, P, NUL) == _lib.MOE_EINVAL
    assert L.moe_route_recall(P, P, 4, 33, P, NUL) == _lib.MOE_ENOTSUP
    assert L.moe_route_recall(P, P, -1, 10, P, NUL) == _lib.MOE_ESHAPE
    assert L.moe_route_recall(P, P, 0, 10, P, NUL) == _lib.MOE_OK


def test_no_device_gives_cuda_error_not_a_crash():
    """Past admission, a machine without a GPU gets MOE_ECUDA back."""
    assert lib().moe_device_sm_count() == -1


def test_pack_rejections_and_sizes():
    L = lib()
    assert L.moe_pack_size(0, 512, 2560, 640, 0) == 512 * 10 * 40 * 16384
    assert L.moe_pack_size(1, 512, 2560, 640, 1) == 512 * 20 * 10 * 4352
    assert L.moe_pack_size(2, 512, 2560, 640, 0) == 0  # packed formats are outputs, not inputs
    n = L.moe_pack_size(0, 64, 256, 64, 0)
    assert L.moe_pack_experts(0, P, NUL, 64, 256, 64, 0, P, n - 1, NUL) == _lib.MOE_EWORKSPACE
    assert L.moe_pack_experts(1, P, NUL, 64, 256, 64, 0, P, n, NUL) == _lib.MOE_EINVAL  # int4 needs scales
    assert L.moe_pack_experts(0, P, P, 64, 256, 64, 0, P, n, NUL) == _lib.MOE_EINVAL   # bf16 takes none
    assert L.moe_pack_experts(0, P, NUL, 64, 256, 64, 2, P, n, NUL) == _lib.MOE_EINVAL
    assert L.moe_pack_experts(0, P, NUL, 64, 250, 64, 0, P, n, NUL) == _lib.MOE_ENOTSUP
    assert _gateup(fmt=1) == _lib.MOE_ENOTSUP  # plain int4 must be packed first



def test_swiglu_fused_rejections():
    L = lib()
    # x, k, perm, x_perm, offsets, R, E, H, I, fmt, w_gateup, w_down, h, y_perm, sync_ws, dev_status, stream
    base = [NUL, 0, NUL, P, P, 160, 512, 2560, 640, _lib.MOE_W_BF16_TILED, P, P, P, P, P, P, NUL]

    def call(**kw):
        a = list(base)
        names = ["x", "k", "perm", "xp", "off", "R", "E", "H", "I", "fmt", "wgu", "wd", "h", "y", "sync", "st"]
        for n, v in kw.items():
            a[names.index(n)] = v
        return L.moe_expert_swiglu_fused(*a)

    assert call(fmt=_lib.MOE_W_BF16) == _lib.MOE_ENOTSUP          # packed bf16 records only
    assert call(fmt=_lib.MOE_W_INT4_G64_TILED) == _lib.MOE_ENOTSUP
    assert call(sync=NUL) == _lib.MOE_EWORKSPACE
    assert call(xp=NUL) == _lib.MOE_EINVAL
    assert call(st=NUL) == _lib.MOE_EINVAL
    assert call(y=PM) == _lib.MOE_EINVAL
    assert call(I=600) == _lib.MOE_ENOTSUP
    assert call(R=-1) == _lib.MOE_ESHAPE
    # with the gather: perm and a k that divides R are required
    assert call(x=P, k=10, perm=NUL) == _lib.MOE_EINVAL
    assert call(x=P, k=0, perm=P) == _lib.MOE_ESHAPE
    assert call(x=P, k=7, perm=P) == _lib.MOE_ESHAPE             # 160 % 7 != 0
    assert call(x=P, k=40, perm=P) == _lib.MOE_ENOTSUP
    assert call(x=PM, k=10, perm=P) == _lib.MOE_EINVAL
    assert call(R=0) == _lib.MOE_OK
    assert call(R=0, x=P, k=10, perm=P) == _lib.MOE_OK


def test_swiglu_fused_weighted_rejections():
    L = lib()
    # x, k, perm, x_perm, offsets, R, E, H, I, fmt, w_gateup, w_down, topk_w, h, yw_perm, sync_ws, dev_status,
    # stream
    base = [NUL, 10, P, P, P, 40960, 512, 2560, 640, _lib.MOE_W_BF16_TILED, P, P, P, P, P, P, P, NUL]
    names = ["x", "k", "perm", "xp", "off", "R", "E", "H", "I", "fmt", "wgu", "wd", "w", "h", "yw", "sync", "st"]

    def call(**kw):
        a = list(base)
        for n, v in kw.items():
            a[names.index(n)] = v
        return L.moe_expert_swiglu_fused_weighted(*a)

    assert call(perm=NUL) == _lib.MOE_EINVAL       # the route of each slot is needed for its weight
    assert call(w=NUL) == _lib.MOE_EINVAL
    assert call(w=PM) == _lib.MOE_EINVAL
    assert call(yw=PM) == _lib.MOE_EINVAL
    assert call(k=0) == _lib.MOE_ESHAPE
    assert call(k=7) == _lib.MOE_ESHAPE            # 40960 % 7 != 0
    assert call(k=40) == _lib.MOE_ENOTSUP
    assert call(fmt=_lib.MOE_W_BF16) == _lib.MOE_ENOTSUP
    assert call(sync=NUL) == _lib.MOE_EWORKSPACE
    assert call(R=0) == _lib.MOE_OK


def test_combine_weighted_rejections():
    L = lib()
    assert L.moe_combine_weighted(P, P, 16, 10, 2560, NUL, NUL, NUL, NUL, NUL) == _lib.MOE_EINVAL
    assert L.moe_combine_weighted(PM, P, 16, 10, 2560, NUL, P, NUL, NUL, NUL) == _lib.MOE_EINVAL
    assert L.moe_combine_weighted(NUL, P, 16, 10, 2560, NUL, P, NUL, NUL, NUL) == _lib.MOE_EINVAL
    assert L.moe_combine_weighted(P, P, 16, 40, 2560, NUL, P, NUL, NUL, NUL) == _lib.MOE_ENOTSUP
    assert L.moe_combine_weighted(P, P, 16, 10, 2500, NUL, P, NUL, NUL, NUL) == _lib.MOE_ENOTSUP
    assert L.moe_combine_weighted(P, P, -1, 10, 2560, NUL, P, NUL, NUL, NUL) == _lib.MOE_ESHAPE
    assert L.moe_combine_weighted(P, P, 0, 10, 2560, NUL, P, NUL, NUL, NUL) == _lib.MOE_OK


def test_int4_slots_rejections():
    L = lib()
    # kind, rows, offsets, R, E, H, I, pool, S, slot_of, out, dev_status, stream
    base = [0, P, P, 160, 512, 2560, 640, P, 192, P, P, P, NUL]
    names = ["kind", "rows", "off", "R", "E", "H", "I", "pool", "S", "slot", "out", "st"]

    def call(**kw):
        a = list(base)
        for n, v in kw.items():
            a[names.index(n)] = v
        return L.moe_expert_int4_slots(*a)

    assert call(kind=2) == _lib.MOE_EINVAL
    assert call(slot=NUL) == _lib.MOE_EINVAL
    assert call(pool=PM) == _lib.MOE_EINVAL
    assert call(st=NUL) == _lib.MOE_EINVAL
    assert call(S=0) == _lib.MOE_ESHAPE
    assert call(S=2048) == _lib.MOE_ENOTSUP
    assert call(I=600) == _lib.MOE_ENOTSUP
    assert call(R=0) == _lib.MOE_OK
    # a prefill-sized launch is not the decode GEMV's: rejected before any launch
    assert call(R=40960) == _lib.MOE_ENOTSUP


def test_int4_fetch_rejections():
    L = lib()
    # x_perm, offsets, R, E, H, I, pool_gu, pool_dn, S, slot_of, host_gu, host_dn, miss_list, miss_slot, stats,
    # h, sync_ws, dev_status, stream
    base = [P, P, 160, 512, 2560, 640, P, P, 160, P, P, P, P, P, P, P, P, P, NUL]
    names = ["xp", "off", "R", "E", "H", "I", "pgu", "pdn", "S", "slot", "hgu", "hdn", "ml", "ms", "stats", "h",
             "sync", "st"]

    def call(**kw):
        a = list(base)
        for n, v in kw.items():
            a[names.index(n)] = v
        return L.moe_expert_int4_fetch(*a)

    assert call(hgu=NUL) == _lib.MOE_EINVAL
    assert call(hdn=PM) == _lib.MOE_EINVAL
    assert call(ml=NUL) == _lib.MOE_EINVAL
    assert call(sync=NUL) == _lib.MOE_EWORKSPACE
    assert call(S=0) == _lib.MOE_ESHAPE
    assert call(S=2048) == _lib.MOE_ENOTSUP
    assert call(R=40960) == _lib.MOE_ENOTSUP      # decode-sized launches only
    assert call(R=0) == _lib.MOE_OK


def test_route_permute_rejections():
    L = lib()
    # x, wr, bias, T, H, E, k, ids, w, gap, counts, offsets, perm, inv, status, stream
    base = [P, P, NUL, 16, 2560, 512, 10, P, P, NUL, P, P, P, P, P, NUL]

    def call(i, v):
        a = list(base)
        a[i] = v
        return L.moe_route_permute(*a)

    assert call(3, 17) == _lib.MOE_ENOTSUP        # one cluster holds at most 16 tokens
    assert call(3, -1) == _lib.MOE_ESHAPE
    assert call(3, 0) == _lib.MOE_OK
    assert call(0, NUL) == _lib.MOE_EINVAL
    assert call(14, NUL) == _lib.MOE_EINVAL       # status word required
    assert call(0, PM) == _lib.MOE_EINVAL
    assert call(6, 40) == _lib.MOE_ENOTSUP        # k > 32
    assert call(4, 2500) == _lib.MOE_ENOTSUP      # H % 128


def test_cache_plan_and_fetch_rejections():
    L = lib()
    # counts, E, slot_of, expert_of, S, hand, policy, decay, score, last_use, miss_list, miss_slot, stats,
    # status, stream
    base = [P, 512, P, P, 256, P, 0, C.c_float(0.9), NUL, NUL, P, P, P, P, NUL]

    def plan(i, v):
        a = list(base)
        a[i] = v
        return L.moe_cache_plan(*a)

    assert plan(4, 0) == _lib.MOE_ESHAPE
    assert plan(1, 0) == _lib.MOE_ESHAPE
    assert plan(4, 1025) == _lib.MOE_ENOTSUP     # one CTA plans at most 1024 slots
    assert plan(1, 1025) == _lib.MOE_ENOTSUP
    for i in (0, 2, 3, 5, 10, 11, 12, 13):
        assert plan(i, NUL) == _lib.MOE_EINVAL, i
    assert plan(2, PM) == _lib.MOE_EINVAL
    assert plan(6, 3) == _lib.MOE_EINVAL          # unknown policy
    assert plan(6, 1) == _lib.MOE_EINVAL          # LRU needs last_use
    assert plan(6, 2) == _lib.MOE_EINVAL          # SCORE needs score
    b2 = list(base)
    b2[6], b2[8] = 2, P
    b2[7] = C.c_float(1.0)
    assert L.moe_cache_plan(*b2) == _lib.MOE_ERANGE   # decay must be < 1
    b2[7] = C.c_float(-0.5)
    assert L.moe_cache_plan(*b2) == _lib.MOE_ERANGE
    b2[7] = C.c_float(0.5)
    assert L.moe_cache_plan(*b2) == _lib.MOE_ECUDA
    b3 = list(base)
    b3[6], b3[9] = 1, P
    assert L.moe_cache_plan(*b3) == _lib.MOE_ECUDA
    assert plan(4, 256) == _lib.MOE_ECUDA         # admitted; no device here

    # host_gu, host_dn, rec_gu, rec_dn, miss_list, miss_slot, stats, pool_gu, pool_dn, stream
    fbase = [P, P, 6553600, 3276800, P, P, P, P, P, NUL]

    def fetch(i, v):
        a = list(fbase)
        a[i] = v
        return L.moe_cache_fetch(*a)

    assert fetch(2, 0) == _lib.MOE_ESHAPE
    assert fetch(3, 8) == _lib.MOE_ESHAPE           # records are whole 16-byte units
    for i in (0, 1, 4, 5, 6, 7, 8):
        assert fetch(i, NUL) == _lib.MOE_EINVAL, i
    assert fetch(0, PM) == _lib.MOE_EINVAL


def test_swiglu_cached_rejections():
    L = lib()
    names = ["x", "k", "perm", "xp", "off", "R", "E", "H", "I", "fmt", "pgu", "pdn", "S", "slot", "hgu", "hdn",
             "ml", "ms", "stats", "wave", "h", "y", "sync", "st"]
    base = [NUL, 0, NUL, P, P, 160, 512, 2560, 640, _lib.MOE_W_BF16_TILED, P, P, 256, P, P, P, P, P, P, 4, P, P,
            P, P, NUL]

    def call(**kw):
        a = list(base)
        for n, v in kw.items():
            a[names.index(n)] = v
        return L.moe_expert_swiglu_cached(*a)

    assert call(fmt=_lib.MOE_W_INT4_G64_TILED) == _lib.MOE_ENOTSUP
    assert call(S=0) == _lib.MOE_ESHAPE
    assert call(S=2000) == _lib.MOE_ENOTSUP
    assert call(slot=NUL) == _lib.MOE_EINVAL
    assert call(slot=PM) == _lib.MOE_EINVAL
    assert call(wave=0) == _lib.MOE_ESHAPE
    assert call(hgu=NUL, wave=0) == _lib.MOE_ECUDA   # no fetch: wave unused; admitted
    for n in ("hdn", "ml", "ms", "stats"):
        assert call(**{n: NUL}) == _lib.MOE_EINVAL, n
    assert call(hgu=PM) == _lib.MOE_EINVAL
    assert call(I=704) == _lib.MOE_ENOTSUP          # I/64 odd: the cached kernel steps K in pairs
    assert call(hgu=NUL, I=704) == _lib.MOE_ENOTSUP
    assert call(sync=NUL) == _lib.MOE_EWORKSPACE
    assert call(R=0) == _lib.MOE_OK


def test_layer_stream_rejections():
    L = lib()
    # host_gu, host_dn, bytes_gu, bytes_dn, dev_gu, dev_dn, stream
    assert L.moe_layer_stream(NUL, NUL, 0, 0, NUL, NUL, NUL) == _lib.MOE_OK       # nothing to copy
    assert L.moe_layer_stream(P, P, 8, 16, P, P, NUL) == _lib.MOE_ESHAPE
    assert L.moe_layer_stream(NUL, P, 16, 16, P, P, NUL) == _lib.MOE_EINVAL
    assert L.moe_layer_stream(P, P, 16, 16, P, NUL, NUL) == _lib.MOE_EINVAL
    assert L.moe_layer_stream(PM, P, 16, 16, P, P, NUL) == _lib.MOE_EINVAL
    assert L.moe_layer_stream(P, P, 16, 16, P, P, NUL) == _lib.MOE_ECUDA         # admitted; no device here


def test_stream_mode_crossover():
    """Selected records win for few distinct records, the whole layer once
    the unique-record fraction passes the measured crossover; the switch
    happens once as U grows, where the two times cross."""
    E, rec = 512, 9830400.0
    modes = [_lib.stream_mode(U, E, rec, 200.0, 211.0, 10.0) for U in range(E + 1)]
    m = [x[0] for x in modes]
    assert m[0] == _lib.MOE_STREAM_SELECTED and modes[0][1] == 0.0
    assert m[16] == _lib.MOE_STREAM_SELECTED and m[E] == _lib.MOE_STREAM_LAYER
    flip = m.index(_lib.MOE_STREAM_LAYER)
    assert all(v == _lib.MOE_STREAM_LAYER for v in m[flip:])
    ts_flip, tl = modes[flip][1], modes[flip][2]
    assert modes[flip - 1][1] <= tl < ts_flip
    # t_layer = E * rec / 211 GB/s, in microseconds
    assert abs(tl - E * rec / 211e3) < 1e-6 * tl
    # equal rates and no overhead: selected never loses
    assert all(_lib.stream_mode(U, E, rec, 211.0, 211.0, 0.0)[0] == _lib.MOE_STREAM_SELECTED for U in (1, 256, 512))
    with pytest.raises(ValueError):
        _lib.stream_mode(E + 1, E, rec, 200.0, 211.0)
    with pytest.raises(ValueError):
        _lib.stream_mode(4, E, rec, 0.0, 211.0)


def test_sidecar_rejections():
    L = lib()
    # w_head, emb, E, r, L, head_bias, stream
    assert L.moe_sidecar_prepare(P, P, 512, 256, 48, P, NUL) == _lib.MOE_ECUDA
    assert L.moe_sidecar_prepare(P, P, 512, 250, 48, P, NUL) == _lib.MOE_ENOTSUP   # r % 8
    assert L.moe_sidecar_prepare(P, P, 2048, 256, 48, P, NUL) == _lib.MOE_ENOTSUP
    assert L.moe_sidecar_prepare(P, P, 0, 256, 48, P, NUL) == _lib.MOE_ESHAPE
    assert L.moe_sidecar_prepare(NUL, P, 512, 256, 48, P, NUL) == _lib.MOE_EINVAL
    assert L.moe_sidecar_prepare(PM, P, 512, 256, 48, P, NUL) == _lib.MOE_EINVAL
    # feat, trunk, head, head_bias, T, F, r, E, L, N, z, cand, score, status, stream
    base = [P, P, P, P, 16, 2560, 256, 512, 48, 16, P, P, P, P, NUL]

    def fwd(i, v):
        a = list(base)
        a[i] = v
        return L.moe_sidecar_forward(*a)

    assert fwd(4, 0) == _lib.MOE_OK
    assert fwd(4, -1) == _lib.MOE_ESHAPE
    assert fwd(5, 2500) == _lib.MOE_ENOTSUP      # F % 128
    assert fwd(9, 33) == _lib.MOE_ENOTSUP        # N <= 32
    assert fwd(7, 8) == _lib.MOE_ENOTSUP         # N <= E
    assert fwd(6, 1032) == _lib.MOE_ENOTSUP      # r <= 1024
    for i in (0, 1, 2, 3, 10, 11, 12, 13):
        assert fwd(i, NUL) == _lib.MOE_EINVAL, i
    assert fwd(0, PM) == _lib.MOE_EINVAL
    assert fwd(4, 16) == _lib.MOE_ECUDA
