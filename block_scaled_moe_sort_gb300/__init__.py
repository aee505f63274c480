"""GB300 (sm_103a) block-scaled fused MoE layer: Python binding.

Argument marshalling only: every function forwards to the entry point of the
same name in ``libmoe_mx.so`` (declared in ``include/moe_mx.h``); all work
runs in that library's CUDA kernels. PyTorch supplies device memory and the
current stream. There is no fallback: if the library is missing, or a tensor
is not on a CUDA device, the call raises.
"""
from __future__ import annotations

import ctypes
import os
import re
from typing import Optional

import torch

from . import build as _build

__all__ = [
    "lib", "MoeError", "moe_sort", "moe_sort_max_padded", "moe_quant_act_mx", "moe_router_topk",
    "moe_prepack_scales_mx", "moe_prepack_weights_mx", "fused_moe_workspace_bytes", "fused_moe_workspace_layout",
    "fused_moe_a8w4", "fused_moe_a16w4", "MoeLayer", "HEADER", "declared_functions",
    "moe_profile_enable", "moe_profile_collect", "PROFILE_SLOTS", "fused_moe_a8w4_noalloc",
    "moe_noalloc_status", "fused_moe_gated", "shared_expert_pieces", "with_shared_expert",
    "moe_prepack_weights_a16w4", "moe_dequant_a16w4",
]

HEADER = os.path.join(_build.ROOT, "include", "moe_mx.h")

_c_void_p = ctypes.c_void_p
_c_int = ctypes.c_int
_c_size_t = ctypes.c_size_t
_c_int64 = ctypes.c_int64


class MoeWsLayout(ctypes.Structure):
    _fields_ = [("block_m", ctypes.c_int32), ("_pad", ctypes.c_int32), ("p_max", _c_int64),
                ("status_off", _c_int64), ("expert_off_off", _c_int64),
                ("sorted_route_off", _c_int64), ("sorted_w_off", _c_int64),
                ("block_expert_off", _c_int64), ("route_pos_off", _c_int64),
                ("sort_scratch_off", _c_int64),
                ("act_off", _c_int64), ("act_sf_off", _c_int64), ("inter_off", _c_int64),
                ("inter_sf_off", _c_int64), ("acc_off", _c_int64), ("split_part_off", _c_int64),
                ("split_cnt_off", _c_int64), ("total_bytes", _c_int64)]


class MoeCallConfig(ctypes.Structure):
    _fields_ = [("block_m", ctypes.c_int32), ("prefetch1", ctypes.c_int32),
                ("prefetch2", ctypes.c_int32), ("split", ctypes.c_int32)]


_SIGS = {
    "moe_status_string": (ctypes.c_char_p, [_c_int]),
    "moe_sort_max_padded": (_c_int64, [_c_int, _c_int, _c_int, _c_int]),
    "moe_sort_workspace_bytes": (_c_size_t, [_c_int, _c_int, _c_int, _c_int]),
    "moe_sort": (_c_int, [_c_void_p, _c_void_p, _c_int, _c_int, _c_int, _c_int, _c_void_p,
                          _c_void_p, _c_void_p, _c_void_p, _c_void_p, _c_void_p, _c_void_p,
                          _c_size_t, _c_void_p]),
    "moe_quant_act_mx": (_c_int, [_c_void_p, _c_int, _c_int, _c_int, _c_void_p, _c_void_p,
                                  _c_void_p]),
    "moe_router_topk": (_c_int, [_c_void_p, _c_int, _c_int, _c_int, _c_int, _c_int, _c_int,
                                 _c_void_p, _c_void_p, _c_void_p]),
    "moe_prepacked_scale_bytes": (_c_size_t, [_c_int, _c_int, _c_int]),
    "moe_prepacked_weight_bytes": (_c_size_t, [_c_int, _c_int, _c_int]),
    "moe_prepack_weights_mx": (_c_int, [_c_void_p, _c_int, _c_int, _c_int, _c_void_p,
                                        _c_void_p]),
    "moe_prepack_scales_mx": (_c_int, [_c_void_p, _c_int, _c_int, _c_int, _c_void_p, _c_void_p]),
    "moe_prepack_weights_a16w4": (_c_int, [_c_void_p, _c_int, _c_int, _c_int, _c_void_p,
                                           _c_void_p]),
    "moe_dequant_a16w4": (_c_int, [_c_void_p, _c_void_p, _c_int, _c_int, _c_int, _c_void_p,
                                   _c_void_p]),
    "fused_moe_workspace_bytes": (_c_size_t, [_c_int] * 6),
    "fused_moe_workspace_layout": (_c_int, [_c_int] * 6 + [ctypes.POINTER(MoeWsLayout)]),
    "fused_moe_a8w4": (_c_int, [_c_void_p, _c_void_p, _c_void_p, _c_int, _c_int, _c_int,
                                _c_void_p, _c_void_p, _c_void_p, _c_void_p, _c_int, _c_int,
                                _c_void_p, _c_void_p, _c_size_t, _c_void_p]),
    "fused_moe_a16w4": (_c_int, [_c_void_p, _c_void_p, _c_void_p, _c_int, _c_int, _c_int,
                                 _c_void_p, _c_void_p, _c_void_p, _c_void_p, _c_int, _c_int,
                                 _c_void_p, _c_void_p, _c_size_t, _c_void_p]),
    "fused_moe_workspace_bytes_bm": (_c_size_t, [_c_int] * 7),
    "fused_moe_workspace_layout_bm": (_c_int, [_c_int] * 7 + [ctypes.POINTER(MoeWsLayout)]),
    "fused_moe_a8w4_bm": (_c_int, [_c_void_p, _c_void_p, _c_void_p, _c_int, _c_int, _c_int,
                                   _c_void_p, _c_void_p, _c_void_p, _c_void_p, _c_int, _c_int,
                                   _c_void_p, _c_void_p, _c_size_t, _c_int, _c_void_p]),
    "fused_moe_a16w4_bm": (_c_int, [_c_void_p, _c_void_p, _c_void_p, _c_int, _c_int, _c_int,
                                    _c_void_p, _c_void_p, _c_void_p, _c_void_p, _c_int, _c_int,
                                    _c_void_p, _c_void_p, _c_size_t, _c_int, _c_void_p]),
    "fused_moe_a8w4_cfg": (_c_int, [_c_void_p, _c_void_p, _c_void_p, _c_int, _c_int, _c_int,
                                    _c_void_p, _c_void_p, _c_void_p, _c_void_p, _c_int, _c_int,
                                    _c_void_p, _c_void_p, _c_size_t,
                                    ctypes.POINTER(MoeCallConfig), _c_void_p]),
    "fused_moe_a16w4_cfg": (_c_int, [_c_void_p, _c_void_p, _c_void_p, _c_int, _c_int, _c_int,
                                     _c_void_p, _c_void_p, _c_void_p, _c_void_p, _c_int, _c_int,
                                     _c_void_p, _c_void_p, _c_size_t,
                                     ctypes.POINTER(MoeCallConfig), _c_void_p]),
    "moe_decode_device_status": (_c_int, [ctypes.c_int32]),
    "moe_debug_wait_selftest": (_c_int, [_c_void_p, _c_int, _c_void_p]),
    "fused_moe_a8w4_noalloc": (_c_int, [_c_void_p, _c_void_p, _c_void_p, _c_int, _c_int, _c_int,
                                        _c_void_p, _c_void_p, _c_void_p, _c_void_p, _c_int,
                                        _c_int, _c_void_p, _c_void_p]),
    "moe_noalloc_status": (_c_int, [_c_void_p, _c_void_p]),
    "fused_moe_a8w4_gated": (_c_int, [_c_void_p, _c_void_p] + [_c_int] * 7 + [_c_void_p] * 4 +
                               [_c_int, _c_int] + [_c_void_p] * 4 + [_c_size_t, _c_void_p]),
    "fused_moe_a16w4_gated": (_c_int, [_c_void_p, _c_void_p] + [_c_int] * 7 + [_c_void_p] * 4 +
                               [_c_int, _c_int] + [_c_void_p] * 4 + [_c_size_t, _c_void_p]),
    "moe_profile_enable": (_c_int, [_c_int]),
    "moe_profile_collect": (_c_int, [ctypes.POINTER(ctypes.c_double),
                                     ctypes.POINTER(ctypes.c_int32)]),
}

PROFILE_SLOTS = ("sort", "gather_quant", "stage1_gemm", "stage2_gemm", "finalize")

_LIB = None


def lib() -> ctypes.CDLL:
    """The loaded C library (raises if it has not been built)."""
    global _LIB
    if _LIB is None:
        if not os.path.exists(_build.LIB):
            raise RuntimeError(
                f"{_build.LIB} is missing: build it with __graft_entry__.build() or "
                "`python -m block_scaled_moe_sort_gb300.build`")
        L = ctypes.CDLL(_build.LIB)
        for name, (res, args) in _SIGS.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _LIB = L
    return _LIB


def declared_functions() -> list:
    """Names of the functions include/moe_mx.h declares."""
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\*?\s+\**(\w+)\s*\(", text, flags=re.M)))


class MoeError(RuntimeError):
    def __init__(self, fn: str, code: int):
        msg = lib().moe_status_string(code).decode()
        super().__init__(f"{fn}: {msg} (status {code})")
        self.code = code


def _check(fn: str, code: int):
    if code != 0:
        raise MoeError(fn, code)


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("tensor must be on a CUDA device")
    if not t.is_contiguous():
        raise ValueError("tensor must be contiguous")
    return t.data_ptr() if t.numel() > 0 else None


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


# ----------------------------------------------------------------- sort

def moe_sort_max_padded(M: int, topk: int, E: int, block_m: int) -> int:
    return int(lib().moe_sort_max_padded(M, topk, E, block_m))


def moe_sort(topk_ids: torch.Tensor, topk_weights: torch.Tensor, E: int, block_m: int,
             stream=None) -> dict:
    """Sorted route lists of ``topk_ids`` [M, topk] (see moe_mx.h)."""
    M, topk = topk_ids.shape
    assert topk_ids.dtype == torch.int32 and topk_weights.dtype == torch.float32
    pm = moe_sort_max_padded(M, topk, E, block_m)
    if pm < 0:
        raise ValueError("unsupported sort shape")
    dev = topk_ids.device
    out = dict(
        sorted_route=torch.empty(pm, dtype=torch.int32, device=dev),
        sorted_w=torch.empty(pm, dtype=torch.float32, device=dev),
        block_expert=torch.empty(pm // block_m, dtype=torch.int32, device=dev),
        expert_off=torch.empty(E + 1, dtype=torch.int32, device=dev),
        num_padded=torch.empty(1, dtype=torch.int32, device=dev),
        route_pos=torch.empty(M * topk, dtype=torch.int32, device=dev),
    )
    nws = int(lib().moe_sort_workspace_bytes(M, topk, E, block_m))
    ws = torch.empty(nws, dtype=torch.uint8, device=dev) if nws else None
    code = lib().moe_sort(_ptr(topk_ids), _ptr(topk_weights), M, topk, E, block_m,
                          out["sorted_route"].data_ptr(), out["sorted_w"].data_ptr(),
                          out["block_expert"].data_ptr() if pm else None,
                          out["expert_off"].data_ptr(), out["num_padded"].data_ptr(),
                          _ptr(out["route_pos"]), _ptr(ws), nws, _stream(stream))
    _check("moe_sort", code)
    return out


# ------------------------------------------------------ failure reporting

def moe_debug_wait_selftest(timeout_us: int = 1000, device="cuda", stream=None):
    """Run the bounded-wait self-test (a wait on a barrier nothing completes)
    and return (decoded status, returned marker): (MOE_ERR_TIMEOUT = 6, 1)
    when the wait gave up and the kernel returned. Synchronises."""
    st = torch.zeros(2, dtype=torch.int32, device=device)
    _check("moe_debug_wait_selftest",
           lib().moe_debug_wait_selftest(_ptr(st), timeout_us, _stream(stream)))
    torch.cuda.synchronize(st.device)
    word, returned = st.cpu().tolist()
    return int(lib().moe_decode_device_status(word)), int(returned)


# ---------------------------------------------------------------- gating

def moe_router_topk(logits: torch.Tensor, topk: int, shared_id: Optional[int] = None,
                    stream=None, n_shared: int = 1):
    """Router logits float32 [M, E] -> (topk_ids int32 [M, k'], topk_weights
    float32 [M, k']), k' = topk (+ n_shared shared-expert columns of weight 1,
    ids shared_id, shared_id + 1, ...)."""
    assert logits.dtype == torch.float32 and logits.dim() == 2 and logits.stride(1) == 1
    M, E = logits.shape
    kout = topk + (n_shared if shared_id is not None else 0)
    ids = torch.empty(M, kout, dtype=torch.int32, device=logits.device)
    w = torch.empty(M, kout, dtype=torch.float32, device=logits.device)
    _check("moe_router_topk", lib().moe_router_topk(
        _ptr(logits), M, E, logits.stride(0), topk, -1 if shared_id is None else shared_id,
        n_shared, _ptr(ids), _ptr(w), _stream(stream)))
    return ids, w


# ---------------------------------------------------------------- quant

def moe_quant_act_mx(x: torch.Tensor, stream=None):
    """BF16 [M, K] -> (E4M3 codes uint8 [M, K], E8M0 scales uint8 [M, K/32])."""
    assert x.dtype == torch.bfloat16 and x.dim() == 2
    M, K = x.shape
    q = torch.empty(M, K, dtype=torch.uint8, device=x.device)
    s = torch.empty(M, K // 32, dtype=torch.uint8, device=x.device)
    _check("moe_quant_act_mx", lib().moe_quant_act_mx(_ptr(x), M, K, K, _ptr(q), _ptr(s),
                                                      _stream(stream)))
    return q, s


def _prepack_weights(fn: str, w: torch.Tensor, stream) -> torch.Tensor:
    assert w.dtype == torch.uint8 and w.dim() == 3
    E, N, KH = w.shape
    K = KH * 2
    nbytes = int(lib().moe_prepacked_weight_bytes(E, N, K))
    if nbytes == 0:
        raise ValueError("unsupported weight shape (N and K must be multiples of 128)")
    out = torch.empty(nbytes, dtype=torch.uint8, device=w.device)
    _check(fn, getattr(lib(), fn)(_ptr(w), E, N, K, _ptr(out), _stream(stream)))
    return out


def moe_prepack_weights_mx(w: torch.Tensor, stream=None) -> torch.Tensor:
    """Row-major packed E2M1 codes [E, N, K/2] -> 8 KB weight tiles (a8w4)."""
    return _prepack_weights("moe_prepack_weights_mx", w, stream)


def moe_prepack_weights_a16w4(w: torch.Tensor, stream=None) -> torch.Tensor:
    """Row-major packed E2M1 codes [E, N, K/2] -> the a16w4 weight tiles
    (the same tiles, each 32-bit word in the a16w4 bit order)."""
    return _prepack_weights("moe_prepack_weights_a16w4", w, stream)


def moe_dequant_a16w4(w_packed: torch.Tensor, scale_packed: torch.Tensor, E: int, N: int, K: int,
                      stream=None) -> torch.Tensor:
    """Diagnostic: the a16w4 GEMMs' dequantisation of prepacked experts ->
    BF16 [E, N, K]."""
    out = torch.empty(E, N, K, dtype=torch.bfloat16, device=w_packed.device)
    _check("moe_dequant_a16w4", lib().moe_dequant_a16w4(_ptr(w_packed), _ptr(scale_packed), E, N,
                                                        K, _ptr(out), _stream(stream)))
    return out


def moe_prepack_scales_mx(scale: torch.Tensor, stream=None) -> torch.Tensor:
    """Row-major E8M0 weight scales [E, N, K/32] -> MMA scale atoms."""
    assert scale.dtype == torch.uint8 and scale.dim() == 3
    E, N, KB = scale.shape
    K = KB * 32
    nbytes = int(lib().moe_prepacked_scale_bytes(E, N, K))
    if nbytes == 0:
        raise ValueError("unsupported scale shape (N and K must be multiples of 128)")
    out = torch.empty(nbytes, dtype=torch.uint8, device=scale.device)
    _check("moe_prepack_scales_mx", lib().moe_prepack_scales_mx(_ptr(scale), E, N, K, _ptr(out),
                                                                _stream(stream)))
    return out


# ---------------------------------------------------------- fused layer

def fused_moe_workspace_bytes(M: int, H: int, Ip: int, E: int, topk: int, a16: bool,
                              block_m: int = 0) -> int:
    """Workspace size; block_m 0 = the library's rule, else the route block
    asked for (fused_moe_workspace_bytes_bm)."""
    if block_m:
        return int(lib().fused_moe_workspace_bytes_bm(M, H, Ip, E, topk, int(a16), block_m))
    return int(lib().fused_moe_workspace_bytes(M, H, Ip, E, topk, int(a16)))


def fused_moe_workspace_layout(M: int, H: int, Ip: int, E: int, topk: int, a16: bool,
                               block_m: int = 0) -> dict:
    L = MoeWsLayout()
    if block_m:
        _check("fused_moe_workspace_layout_bm",
               lib().fused_moe_workspace_layout_bm(M, H, Ip, E, topk, int(a16), block_m,
                                                   ctypes.byref(L)))
    else:
        _check("fused_moe_workspace_layout",
               lib().fused_moe_workspace_layout(M, H, Ip, E, topk, int(a16), ctypes.byref(L)))
    return {f: getattr(L, f) for f, _ in MoeWsLayout._fields_ if f != "_pad"}


def _fused(fn_name, x, topk_ids, topk_weights, w1, w1_scale_packed, w2, w2_scale_packed,
           E, Ip, out=None, ws=None, stream=None, block_m=0, prefetch=None, split=0):
    M, H = x.shape
    topk = topk_ids.shape[1]
    a16 = fn_name == "fused_moe_a16w4"
    assert x.dtype == torch.bfloat16 and topk_ids.dtype == torch.int32
    assert topk_weights.dtype == torch.float32 and w1.dtype == torch.uint8
    assert w1.numel() == E * 2 * Ip * H // 2 and w2.numel() == E * H * Ip // 2
    if out is None:
        out = torch.empty(M, H, dtype=torch.bfloat16, device=x.device)
    if ws is None:
        ws = torch.empty(max(fused_moe_workspace_bytes(M, H, Ip, E, topk, a16, block_m), 1),
                         dtype=torch.uint8, device=x.device)
    args = [_ptr(x), _ptr(topk_ids), _ptr(topk_weights), M, H, topk, _ptr(w1),
            _ptr(w1_scale_packed), _ptr(w2), _ptr(w2_scale_packed), E, Ip, _ptr(out), _ptr(ws),
            ws.numel()]
    if (prefetch and any(prefetch)) or split:
        fn_name = fn_name + "_cfg"
        pf = prefetch or (0, 0)
        cfg = MoeCallConfig(int(block_m), int(pf[0]), int(pf[1]), int(split))
        args.append(ctypes.byref(cfg))
    elif block_m:
        fn_name = fn_name + "_bm"
        args.append(block_m)
    code = getattr(lib(), fn_name)(*args, _stream(stream))
    _check(fn_name, code)
    return out


def fused_moe_a8w4(x, topk_ids, topk_weights, w1_packed, w1_scale_packed, w2_packed,
                   w2_scale_packed, E, Ip, out=None, ws=None, stream=None,
                   block_m: int = 0, prefetch=None, split: int = 0) -> torch.Tensor:
    """FP8-activation x MXFP4-weight fused MoE on prepacked weights; returns
    BF16 [M, H]. block_m 0 = the library's route block rule; prefetch
    (stage-1, stage-2 weight L2 prefetch lead in weight tiles, 0 = default)
    and split (the GEMMs' split walk: 0 = the library's choice, 1 = the
    walk, 2 = whole tiles only) go through fused_moe_a8w4_cfg."""
    return _fused("fused_moe_a8w4", x, topk_ids, topk_weights, w1_packed, w1_scale_packed,
                  w2_packed, w2_scale_packed, E, Ip, out, ws, stream, block_m, prefetch, split)


def fused_moe_a16w4(x, topk_ids, topk_weights, w1_packed, w1_scale_packed, w2_packed,
                    w2_scale_packed, E, Ip, out=None, ws=None, stream=None,
                    block_m: int = 0, prefetch=None, split: int = 0) -> torch.Tensor:
    """BF16-activation x MXFP4-weight fused MoE on weights prepacked by
    moe_prepack_weights_a16w4; returns BF16 [M, H]. block_m 0 = the
    library's route block rule; prefetch and split as for fused_moe_a8w4."""
    return _fused("fused_moe_a16w4", x, topk_ids, topk_weights, w1_packed, w1_scale_packed,
                  w2_packed, w2_scale_packed, E, Ip, out, ws, stream, block_m, prefetch, split)


def fused_moe_gated(x, router_logits, topk, w1_packed, w1_scale_packed, w2_packed,
                    w2_scale_packed, E, Ip, a16=False, shared_id=None, out=None, ws=None,
                    topk_ids=None, topk_weights=None, stream=None, n_shared: int = 1):
    """The fused call with the gating in front: router logits float32
    [M, E_route] -> (out BF16 [M, H], topk_ids int32 [M, k'], topk_weights
    float32 [M, k']), k' = topk (+ n_shared shared-expert columns)."""
    M, H = x.shape
    assert router_logits.dtype == torch.float32 and router_logits.stride(1) == 1
    E_route = router_logits.shape[1]
    kout = topk + (n_shared if shared_id is not None else 0)
    dev = x.device
    if out is None:
        out = torch.empty(M, H, dtype=torch.bfloat16, device=dev)
    if topk_ids is None:
        topk_ids = torch.empty(M, kout, dtype=torch.int32, device=dev)
    if topk_weights is None:
        topk_weights = torch.empty(M, kout, dtype=torch.float32, device=dev)
    if ws is None:
        ws = torch.empty(max(fused_moe_workspace_bytes(M, H, Ip, E, kout, a16), 1),
                         dtype=torch.uint8, device=dev)
    fn = "fused_moe_a16w4_gated" if a16 else "fused_moe_a8w4_gated"
    code = getattr(lib(), fn)(
        _ptr(x), _ptr(router_logits), router_logits.stride(0), E_route, topk,
        -1 if shared_id is None else shared_id, n_shared, M, H, _ptr(w1_packed),
        _ptr(w1_scale_packed),
        _ptr(w2_packed), _ptr(w2_scale_packed), E, Ip, _ptr(out), _ptr(topk_ids),
        _ptr(topk_weights), _ptr(ws), ws.numel(), _stream(stream))
    _check(fn, code)
    return out, topk_ids, topk_weights


NOALLOC_WORKSPACE_BYTES = 16 << 20


def fused_moe_a8w4_noalloc(x, topk_ids, topk_weights, w1, w1_scale_packed, w2,
                           w2_scale_packed, E, Ip, out=None, stream=None) -> torch.Tensor:
    """fused_moe_a8w4 without a caller workspace: the library's own static
    scratch of NOALLOC_WORKSPACE_BYTES is used instead (see moe_mx.h for who
    needs this, the size limit and why overlapping calls must be avoided)."""
    M, H = x.shape
    topk = topk_ids.shape[1]
    assert x.dtype == torch.bfloat16 and topk_ids.dtype == torch.int32
    assert topk_weights.dtype == torch.float32 and w1.dtype == torch.uint8
    if out is None:
        out = torch.empty(M, H, dtype=torch.bfloat16, device=x.device)
    code = lib().fused_moe_a8w4_noalloc(
        _ptr(x), _ptr(topk_ids), _ptr(topk_weights), M, H, topk, _ptr(w1), _ptr(w1_scale_packed),
        _ptr(w2), _ptr(w2_scale_packed), E, Ip, _ptr(out), _stream(stream))
    _check("fused_moe_a8w4_noalloc", code)
    return out


def moe_noalloc_status(device="cuda", stream=None) -> tuple:
    """(decoded device status, padded route count) of the last
    fused_moe_a8w4_noalloc call on `device`, read through
    moe_noalloc_status (synchronises the stream)."""
    st = torch.zeros(4, dtype=torch.int32, device=device)
    _check("moe_noalloc_status", lib().moe_noalloc_status(_ptr(st), _stream(stream)))
    torch.cuda.synchronize(st.device)
    word, padded = st.cpu().tolist()[:2]
    return int(lib().moe_decode_device_status(word)), int(padded)


def moe_profile_enable(enable: bool = True) -> None:
    _check("moe_profile_enable", lib().moe_profile_enable(int(enable)))


def moe_profile_collect() -> tuple:
    """Summed milliseconds per kernel slot of the calls since the last
    collect, and the number of calls (see moe_mx.h)."""
    ms = (ctypes.c_double * len(PROFILE_SLOTS))()
    n = ctypes.c_int32(0)
    _check("moe_profile_collect", lib().moe_profile_collect(ms, ctypes.byref(n)))
    return dict(zip(PROFILE_SLOTS, list(ms))), int(n.value)


def shared_expert_pieces(shared, Ip: int):
    """One shared expert (w1 [2*Is, H/2], w1_scale [2*Is, H/32], w2 [H, Is/2],
    w2_scale [H, Is/32], or the same with a leading dimension of 1) as
    ceil(Is / Ip) experts of the routed intermediate size Ip: piece j holds
    intermediate indices [j*Ip, (j+1)*Ip) - gate/up rows of w1 and columns of
    w2 - zero-padded at the end. SiLU(gate)*up acts on each intermediate index
    alone and the down projection sums over them, so running the pieces as
    experts of weight 1 and adding them gives the shared MLP (Ip is a multiple
    of 32: no 1x32 block of the intermediate straddles two pieces).
    Load-time data preparation; returns [n, ...] tensors."""
    w1, s1, w2, s2 = (t[0] if t.dim() == 3 else t for t in shared)
    Is = w2.shape[1] * 2
    if Is % 32 or w1.shape[0] != 2 * Is or s1.shape[0] != 2 * Is or s2.shape[1] * 32 != Is:
        raise ValueError(f"inconsistent shared expert shapes for intermediate size {Is}")
    n = -(-Is // Ip)
    p1 = torch.zeros(n, 2 * Ip, w1.shape[1], dtype=torch.uint8)
    q1 = torch.zeros(n, 2 * Ip, s1.shape[1], dtype=torch.uint8)
    p2 = torch.zeros(n, w2.shape[0], Ip // 2, dtype=torch.uint8)
    q2 = torch.zeros(n, w2.shape[0], Ip // 32, dtype=torch.uint8)
    for j in range(n):
        lo, hi = j * Ip, min((j + 1) * Ip, Is)
        p1[j, :2 * (hi - lo)] = w1[2 * lo:2 * hi].cpu()
        q1[j, :2 * (hi - lo)] = s1[2 * lo:2 * hi].cpu()
        p2[j, :, :(hi - lo) // 2] = w2[:, lo // 2:hi // 2].cpu()
        q2[j, :, :(hi - lo) // 32] = s2[:, lo // 32:hi // 32].cpu()
    return p1, q1, p2, q2


def with_shared_expert(w1, w1_scale, w2, w2_scale, shared):
    """Routed expert tensors [E, ...] plus one separate shared expert of any
    intermediate size -> the same tensors with the shared expert's pieces
    (shared_expert_pieces) appended as experts E, E+1, ..., and the number of
    pieces (load-time data preparation before the one-time prepack)."""
    Ip = w2.shape[2] * 2
    pieces = shared_expert_pieces(shared, Ip)
    out = []
    for routed, sh in zip((w1, w1_scale, w2, w2_scale), pieces):
        if sh.shape[1:] != routed.shape[1:]:
            raise ValueError(f"shared expert piece of shape {tuple(sh.shape)} does not match "
                             f"routed experts {tuple(routed.shape)}")
        out.append(torch.cat([routed, sh.to(routed.device, routed.dtype)], dim=0))
    return (*out, pieces[0].shape[0])


def shipped_block_m_rows(H: int, Ip: int, E: int, a16: bool) -> dict:
    """The shipped GB300 tuning rows of one geometry: topk -> sorted
    [(max_tokens, block_m[, prefetch1, prefetch2[, split]]), ...] (the
    prefetch leads and the split walk where a tuned row sets them; empty for
    a geometry that was not tuned)."""
    from . import tune
    by_topk = {}
    for r in tune.read_table(tune.PACKAGED_TABLE):
        if (r["H"], r["Ip"], r["E"], r["a16"]) == (H, Ip, E, int(a16)):
            row = (r["max_tokens"], r["block_m"])
            if r["prefetch1"] or r["prefetch2"] or r["split"]:
                row += (r["prefetch1"], r["prefetch2"])
            if r["split"]:
                row += (r["split"],)
            by_topk.setdefault(r["topk"], []).append(row)
    for rows in by_topk.values():
        rows.sort()
    return by_topk


class MoeLayer:
    """Device-resident MXFP4 expert weights with prepacked scales.

    block_m_table: rows (max_tokens, block_m[, prefetch1, prefetch2[, split]])
    sorted by max_tokens (see block_scaled_moe_sort_gb300.tune): a call with M
    tokens uses the route block (weight prefetch leads, split walk) of the first row
    with M <= max_tokens; beyond the last row, or without a table, the
    library's own choices apply. "gb300" takes the rows of this geometry
    from the table shipped with the package.

    shared_expert: (w1, w1_scale, w2, w2_scale) of one separate shared
    expert that every token uses with weight 1 (the shared-first layouts of
    the pages: the 385-expert top-7 case), MXFP4 like the routed experts,
    of any intermediate size Is (a multiple of 32). It is appended as
    ceil(Is / Ip) experts E, E+1, ... (its pieces, shared_expert_pieces) and
    runs inside the same grouped GEMMs as the routed experts; the tile walk
    schedules the last experts' route blocks first, so the shared expert's
    tiles lead both stages. ``route`` and ``forward_gated`` produce ids and
    weights with its columns, which the call takes as they are."""

    def __init__(self, w1, w1_scale, w2, w2_scale, a16: bool = False, device="cuda",
                 block_m_table=None, shared_expert=None):
        self.a16 = a16
        self.E_routed = w1.shape[0]
        self.shared_id = None
        self.n_shared = 0
        if shared_expert is not None:
            w1, w1_scale, w2, w2_scale, self.n_shared = with_shared_expert(
                w1, w1_scale, w2, w2_scale, shared_expert)
            self.shared_id = self.E_routed
        self.E = w1.shape[0]
        self.H = w2.shape[1]
        self.Ip = w2.shape[2] * 2
        self._bm_by_topk = None          # shipped rows of this geometry, per topk
        if isinstance(block_m_table, str):
            if block_m_table != "gb300":
                raise ValueError("block_m_table: rows, None or 'gb300'")
            self._bm_by_topk = shipped_block_m_rows(self.H, self.Ip, self.E, a16)
            block_m_table = None
        self.block_m_table = sorted(block_m_table) if block_m_table else []
        prepack = moe_prepack_weights_a16w4 if a16 else moe_prepack_weights_mx
        self.w1 = prepack(w1.to(device).contiguous())
        self.w2 = prepack(w2.to(device).contiguous())
        self.w1_scale = moe_prepack_scales_mx(w1_scale.to(device).contiguous())
        self.w2_scale = moe_prepack_scales_mx(w2_scale.to(device).contiguous())

    def route(self, logits: torch.Tensor, topk: int, stream=None):
        """Router logits float32 [M, E_routed] -> (topk_ids, topk_weights) for
        this layer, with the shared expert's column when it has one."""
        assert logits.shape[1] == self.E_routed
        return moe_router_topk(logits, topk, shared_id=self.shared_id, stream=stream,
                               n_shared=max(self.n_shared, 1))

    def forward_gated(self, x, router_logits, topk: int, out=None, ws=None, stream=None):
        """Gating + fused call in one (fused_moe_*_gated): router logits
        float32 [M, E_route] -> (out, topk_ids, topk_weights); the shared
        expert's column is added when the layer has one. An expert-parallel
        shard passes the global logits (ids outside its experts are
        dropped)."""
        return fused_moe_gated(x, router_logits, topk, self.w1, self.w1_scale, self.w2,
                               self.w2_scale, self.E, self.Ip, a16=self.a16,
                               shared_id=self.shared_id, out=out, ws=ws, stream=stream,
                               n_shared=max(self.n_shared, 1))

    def _row_for(self, M: int, topk: Optional[int]):
        table = self.block_m_table
        by_topk = getattr(self, "_bm_by_topk", None)
        if by_topk is not None:
            table = by_topk.get(topk, [])
        for row in table:
            if M <= row[0]:
                return row
        return None

    def block_m_for(self, M: int, topk: Optional[int] = None) -> int:
        """Route block for an M-token call (0 = the library's rule)."""
        row = MoeLayer._row_for(self, M, topk)
        return int(row[1]) if row else 0

    def prefetch_for(self, M: int, topk: Optional[int] = None):
        """(stage-1, stage-2) weight prefetch leads for an M-token call
        ((0, 0) = the library's defaults)."""
        row = MoeLayer._row_for(self, M, topk)
        return (int(row[2]), int(row[3])) if row and len(row) >= 4 else (0, 0)

    def split_for(self, M: int, topk: Optional[int] = None) -> int:
        """Split walk for an M-token call (0 = the library's choice)."""
        row = MoeLayer._row_for(self, M, topk)
        return int(row[4]) if row and len(row) >= 5 else 0

    def workspace_bytes(self, M: int, topk: int) -> int:
        return fused_moe_workspace_bytes(M, self.H, self.Ip, self.E, topk, self.a16,
                                         self.block_m_for(M, topk))

    def workspace_layout(self, M: int, topk: int) -> dict:
        return fused_moe_workspace_layout(M, self.H, self.Ip, self.E, topk, self.a16,
                                          self.block_m_for(M, topk))

    def __call__(self, x, topk_ids, topk_weights, out=None, ws=None, stream=None, block_m=None,
                 prefetch=None, split=None):
        fn = fused_moe_a16w4 if self.a16 else fused_moe_a8w4
        M, k = x.shape[0], topk_ids.shape[1]
        bm = self.block_m_for(M, k) if block_m is None else block_m
        pf = self.prefetch_for(M, k) if prefetch is None else prefetch
        sp = self.split_for(M, k) if split is None else split
        return fn(x, topk_ids, topk_weights, self.w1, self.w1_scale, self.w2, self.w2_scale,
                  self.E, self.Ip, out=out, ws=ws, stream=stream, block_m=bm, prefetch=pf,
                  split=sp)
