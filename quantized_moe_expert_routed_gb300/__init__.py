"""GB300 (sm_103a) routed-expert MoE layer: Python binding of libmnw_moe.so.

Argument marshalling only: every step runs in the library's CUDA kernels.
The function names are those of the C ABI in include/mnw_moe.h.  Tensors are
torch CUDA tensors; the current torch stream is used unless ``stream`` is given.
If the library is missing it is built with nvcc on first import; if that
fails, importing this package fails (there is no fallback path).
"""
from __future__ import annotations

import ctypes
import os

import torch

from . import build as _build

_HERE = os.path.dirname(os.path.abspath(__file__))

MNW_OK = 0
FMT_BF16, FMT_INT8_G128, FMT_INT4_G128, FMT_NVFP4_G16 = 0, 1, 2, 3
ACT_BF16, ACT_INT8_G128, ACT_NVFP4_G16, ACT_F16_ROWS = 0, 1, 2, 3
KIND_GATE_UP, KIND_DOWN, KIND_GATE, KIND_UP = 0, 1, 2, 3
DEVERR_BAD_EXPERT_ID, DEVERR_TIMEOUT = 0x1, 0x2
PATH_AUTO, PATH_TCGEN05, PATH_WARP_MMA, PATH_ROWS = 0, 1, 2, 3

# Symbols of include/mnw_moe.h, with their ctypes signatures.
_P, _I, _SZ, _U32P = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t, ctypes.c_void_p
SIGNATURES = {
    "mnw_status_string": (ctypes.c_char_p, [_I]),
    "mnw_moe_layer_init": (_I, [_P, _P, _SZ, ctypes.POINTER(_P)]),
    "mnw_moe_layer_destroy": (None, [_P]),
    "mnw_moe_layer_info": (_I, [_P, _P, _P, _P, _P]),
    "mnw_moe_permute": (_I, [_P, _I, _I, _I, _P, _P, _P, _P, _I, _P, _U32P, _P]),
    "mnw_moe_quantize_act": (_I, [_I, _P, _I, _I, _P, _I, _P, _P, _P, _P]),
    "mnw_moe_permute_host": (_I, [_P, _I, _I, _I, _P, _P, _P, _U32P]),
    "mnw_moe_route_scratch_size": (_SZ, [_I, _I]),
    "mnw_moe_route": (_I, [_P, _P, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _SZ, _U32P, _P]),
    "mnw_moe_workspace_size_routed": (_SZ, [_P, _I, _I, _I]),
    "mnw_moe_forward_routed": (_I, [_P, _I, _P, _P, _I, _I, _P, _P, _P, _P, _SZ, _P]),
    "mnw_moe_grouped_gemm_bf16": (_I, [_P, _I, _P, _P, _I, _P, _U32P, _P]),
    "mnw_moe_grouped_gemm_w8a16": (_I, [_P, _I, _P, _P, _I, _P, _U32P, _P]),
    "mnw_moe_grouped_gemm_w4a16": (_I, [_P, _I, _P, _P, _I, _P, _U32P, _P]),
    "mnw_moe_grouped_gemm_w8a16_f16rows": (_I, [_P, _I, _P, _P, _P, _I, _P, _U32P, _P]),
    "mnw_moe_grouped_gemm_w4a16_f16rows": (_I, [_P, _I, _P, _P, _P, _I, _P, _U32P, _P]),
    "mnw_moe_grouped_gemm_w8a8": (_I, [_P, _I, _P, _P, _P, _I, _P, _P, _U32P, _P]),
    "mnw_moe_grouped_gemm_w4a8": (_I, [_P, _I, _P, _P, _P, _I, _P, _P, _U32P, _P]),
    "mnw_moe_grouped_gemm_nvfp4": (_I, [_P, _I, _P, _P, _P, _P, _I, _P, _U32P, _P]),
    "mnw_moe_combine": (_I, [_P, _P, _P, _I, _I, _I, _P, _P]),
    "mnw_moe_workspace_size": (_SZ, [_P, _I, _I, _I]),
    "mnw_moe_forward": (_I, [_P, _I, _P, _P, _P, _I, _I, _P, _P, _SZ, _P]),
    "mnw_moe_workspace_error_word": (_P, [_P]),
    "mnw_moe_workspace_size_host": (_SZ, [_P, _I, _I, _I]),
    "mnw_moe_forward_host": (_I, [_P, _I, _P, _P, _P, _I, _I, _P, _P, _SZ, _P]),
    "mnw_moe_read_error": (_I, [_P, _P, _P]),
    "mnw_moe_set_gemm_path": (_I, [_I]),
    "mnw_moe_set_fused_activation": (_I, [_I]),
    "mnw_moe_set_host_routing": (_I, [_I]),
    "mnw_moe_silu_mul": (_I, [_P, _P, _SZ, _P, _P]),
    "mnw_moe_launch_count": (ctypes.c_uint64, []),
    "mnw_moe_forward_static": (_I, [_P, _I, _P, _P, _P, _I, _I, _P, _U32P, _P]),
    "mnw_moe_selftest_wait_timeout": (_I, [ctypes.c_uint32, _U32P, _U32P, _P]),
    "mnw_moe_selftest_counter_timeout": (_I, [ctypes.c_uint32, _U32P, ctypes.c_uint32, _U32P, _P]),
    "mnw_attn_workspace_size": (_SZ, [_I, _I, _I, _I]),
    "mnw_attn_prefill": (_I, [_P, _P, _P, _I, _I, _I, _I, _I, _I, ctypes.c_float, _P, _P, _SZ, _U32P, _P]),
}

_lib = None


def lib_path() -> str:
    return _build.LIB


def load() -> ctypes.CDLL:
    """Load (building first if needed) libmnw_moe.so."""
    global _lib
    if _lib is None:
        path = _build.build()
        lib = ctypes.CDLL(path)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib


class MnwError(RuntimeError):
    pass


def _check(rc: int, what: str):
    if rc != MNW_OK:
        msg = load().mnw_status_string(rc).decode()
        raise MnwError(f"{what}: {msg} (status {rc})")


def _ptr(t):
    if t is None:
        return None
    if not t.is_cuda:
        raise MnwError("expected a CUDA tensor")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


class Layer:
    """An expert blob (device uint8 tensor) described to the library.  The
    blob tensor is kept alive by this object."""

    def __init__(self, blob: torch.Tensor, header: bytes):
        self.blob = blob
        self.header = bytes(header)
        h = ctypes.create_string_buffer(self.header, len(self.header))
        out = ctypes.c_void_p()
        _check(load().mnw_moe_layer_init(h, _ptr(blob), blob.numel(), ctypes.byref(out)), "mnw_moe_layer_init")
        self.handle = out
        fmt, E, H, I = (ctypes.c_int() for _ in range(4))
        _check(load().mnw_moe_layer_info(self.handle, ctypes.byref(fmt), ctypes.byref(E), ctypes.byref(H),
                                         ctypes.byref(I)), "mnw_moe_layer_info")
        self.wfmt, self.E, self.H, self.I = fmt.value, E.value, H.value, I.value

    def __del__(self):
        if getattr(self, "handle", None) and _lib is not None:
            _lib.mnw_moe_layer_destroy(self.handle)
            self.handle = None


def mnw_moe_permute(ids, E, x=None, stream=None, err=None):
    """Returns (expert_offsets [E+1], sorted_assign [P], assign_pos [P], x_perm or None)."""
    T, k = ids.shape
    P = T * k
    dev = ids.device
    offsets = torch.empty(E + 1, dtype=torch.int32, device=dev)
    sorted_assign = torch.empty(P, dtype=torch.int32, device=dev)
    assign_pos = torch.empty(P, dtype=torch.int32, device=dev)
    x_perm = None
    H = 0
    if x is not None:
        H = x.shape[1]
        x_perm = torch.empty((P, H), dtype=x.dtype, device=dev)
    _check(load().mnw_moe_permute(_ptr(ids), T, k, E, _ptr(offsets), _ptr(sorted_assign), _ptr(assign_pos),
                                  _ptr(x), H, _ptr(x_perm), _ptr(err), _stream(stream)), "mnw_moe_permute")
    return offsets, sorted_assign, assign_pos, x_perm


def mnw_moe_route(x, w_router, k, scratch=None, stream=None, err=None):
    """GPU routing fused with the permutation (see include/mnw_moe.h).
    x: bf16 [T, H]; w_router: bf16 [E, H].  Returns (ids int32 [T,k], w f32
    [T,k], expert_offsets, sorted_assign, assign_pos, logits f32 [T,E]).
    scratch: a uint8 device tensor reused across calls (zero-filled when new)."""
    T, H = x.shape
    E = w_router.shape[0]
    dev = x.device
    need = load().mnw_moe_route_scratch_size(T, E)
    if scratch is None:
        scratch = torch.zeros(need + 256, dtype=torch.uint8, device=dev)
    base = (-scratch.data_ptr()) % 256
    view = scratch[base:base + need]
    ids = torch.empty((T, k), dtype=torch.int32, device=dev)
    w = torch.empty((T, k), dtype=torch.float32, device=dev)
    off = torch.empty(E + 1, dtype=torch.int32, device=dev)
    sa = torch.empty(T * k, dtype=torch.int32, device=dev)
    pos = torch.empty(T * k, dtype=torch.int32, device=dev)
    _check(load().mnw_moe_route(_ptr(x), _ptr(w_router), T, H, E, k, _ptr(ids), _ptr(w), _ptr(off), _ptr(sa),
                                _ptr(pos), _ptr(view), need, _ptr(err), _stream(stream)), "mnw_moe_route")
    cb = (((1 + (T + 15) // 16) * 4 + 255) // 256) * 256  # the counters come first
    logits = view[cb:cb + T * E * 4].view(torch.float32).view(T, E)
    return ids, w, off, sa, pos, logits


def mnw_moe_workspace_size_routed(layer, act, T, k) -> int:
    return load().mnw_moe_workspace_size_routed(layer.handle, act, T, k)


def mnw_moe_forward_routed(layer, act, x, w_router, k, ws=None, out=None, stream=None):
    """The layer with GPU routing; returns (out bf16 [T,H], ids int32 [T,k], w f32 [T,k])."""
    T = x.shape[0]
    if ws is None:
        n = mnw_moe_workspace_size_routed(layer, act, T, k)
        ws = torch.empty(n + 256, dtype=torch.uint8, device=x.device)
    base = (-ws.data_ptr()) % 256
    ids = torch.empty((T, k), dtype=torch.int32, device=x.device)
    w = torch.empty((T, k), dtype=torch.float32, device=x.device)
    if out is None:
        out = torch.empty((T, layer.H), dtype=torch.bfloat16, device=x.device)
    _check(load().mnw_moe_forward_routed(layer.handle, act, _ptr(x), _ptr(w_router), T, k, _ptr(ids), _ptr(w),
                                         _ptr(out), ctypes.c_void_p(ws.data_ptr() + base), ws.numel() - base,
                                         _stream(stream)), "mnw_moe_forward_routed")
    return out, ids, w


def mnw_moe_permute_host(ids, E):
    """Host-side permutation (numpy int32 [T, k] in): (offsets, sorted_assign,
    assign_pos, dropped) as numpy arrays, the same as mnw_moe_permute's."""
    import numpy as np
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    T, k = ids.shape
    P = T * k
    off = np.zeros(E + 1, np.int32)
    sa = np.zeros(P, np.int32)
    pos = np.zeros(P, np.int32)
    dropped = ctypes.c_uint32()
    p = lambda a: a.ctypes.data_as(ctypes.c_void_p)
    _check(load().mnw_moe_permute_host(p(ids), T, k, E, p(off), p(sa), p(pos), ctypes.byref(dropped)),
           "mnw_moe_permute_host")
    return off, sa, pos, int(dropped.value)


def mnw_moe_quantize_act(act, x, row_index=None, index_div=1, rows=None, stream=None):
    """INT8_G128 -> (codes int8 [R,K], scales f32 [R,K/128]);
    NVFP4_G16 -> (codes u8 [R,K/2], sf u8 [R,K/16], outer f32 [R]);
    F16_ROWS -> (codes fp16 [R,K], factor f32 [R])."""
    R = rows if rows is not None else (row_index.numel() if row_index is not None else x.shape[0])
    K = x.shape[1]
    dev = x.device
    if act == ACT_F16_ROWS:
        codes = torch.empty((R, K), dtype=torch.float16, device=dev)
        outer = torch.empty((R,), dtype=torch.float32, device=dev)
        _check(load().mnw_moe_quantize_act(act, _ptr(x), R, K, _ptr(row_index), index_div, _ptr(codes), None,
                                           _ptr(outer), _stream(stream)), "mnw_moe_quantize_act")
        return codes, outer
    if act == ACT_INT8_G128:
        codes = torch.empty((R, K), dtype=torch.int8, device=dev)
        scales = torch.empty((R, K // 128), dtype=torch.float32, device=dev)
        outer = None
    else:
        codes = torch.empty((R, K // 2), dtype=torch.uint8, device=dev)
        scales = torch.empty((R, K // 16), dtype=torch.uint8, device=dev)
        outer = torch.empty((R,), dtype=torch.float32, device=dev)
    _check(load().mnw_moe_quantize_act(act, _ptr(x), R, K, _ptr(row_index), index_div, _ptr(codes), _ptr(scales),
                                       _ptr(outer), _stream(stream)), "mnw_moe_quantize_act")
    return (codes, scales) if act == ACT_INT8_G128 else (codes, scales, outer)


def mnw_moe_set_fused_activation(fused: bool) -> None:
    _check(load().mnw_moe_set_fused_activation(1 if fused else 0), "mnw_moe_set_fused_activation")


def mnw_moe_set_host_routing(on: bool) -> None:
    _check(load().mnw_moe_set_host_routing(1 if on else 0), "mnw_moe_set_host_routing")


def mnw_moe_silu_mul(g, u, stream=None):
    """bf16(SiLU(g) * u) of two bf16 tensors of the same shape."""
    h = torch.empty_like(g)
    _check(load().mnw_moe_silu_mul(_ptr(g), _ptr(u), g.numel(), _ptr(h), _stream(stream)), "mnw_moe_silu_mul")
    return h


def mnw_attn_prefill(q, k, v, blk: int, scale: float, out=None, ws=None, err=None, stream=None):
    """Block attention of bf16 q [B, T, Hq, d] over k, v [B, T, Hkv, d]; key j
    is allowed for token t when j // blk <= t // blk.  Returns out [B, T, Hq, d]."""
    B, T, Hq, d = q.shape
    Hkv = k.shape[2]
    L = load()
    if out is None:
        out = torch.empty_like(q)
    if ws is None:
        ws = torch.empty((max(1, L.mnw_attn_workspace_size(B, T, Hkv, d)),), dtype=torch.uint8, device=q.device)
    _check(L.mnw_attn_prefill(_ptr(q), _ptr(k), _ptr(v), B, T, Hq, Hkv, d, int(blk), float(scale), _ptr(out),
                              _ptr(ws), ws.numel(), _ptr(err), _stream(stream)), "mnw_attn_prefill")
    return out


def _gemm_out(layer, kind, P, dev):
    N = layer.H if kind == KIND_DOWN else layer.I
    return torch.empty((P, N), dtype=torch.bfloat16, device=dev)


def _gemm_a16(name, layer, kind, a, expert_offsets, err=None, stream=None):
    P = a.shape[0]
    out = _gemm_out(layer, kind, P, a.device)
    fn = getattr(load(), name)
    _check(fn(layer.handle, kind, _ptr(a), _ptr(expert_offsets), P, _ptr(out), _ptr(err), _stream(stream)), name)
    return out


def mnw_moe_grouped_gemm_bf16(layer, kind, a, expert_offsets, err=None, stream=None):
    return _gemm_a16("mnw_moe_grouped_gemm_bf16", layer, kind, a, expert_offsets, err, stream)


def mnw_moe_grouped_gemm_w8a16(layer, kind, a, expert_offsets, err=None, stream=None):
    return _gemm_a16("mnw_moe_grouped_gemm_w8a16", layer, kind, a, expert_offsets, err, stream)


def mnw_moe_grouped_gemm_w4a16(layer, kind, a, expert_offsets, err=None, stream=None):
    return _gemm_a16("mnw_moe_grouped_gemm_w4a16", layer, kind, a, expert_offsets, err, stream)


def _gemm_f16rows(name, layer, kind, a, row_outer, expert_offsets, err=None, stream=None):
    P = a.shape[0]
    out = _gemm_out(layer, kind, P, a.device)
    fn = getattr(load(), name)
    _check(fn(layer.handle, kind, _ptr(a), _ptr(row_outer), _ptr(expert_offsets), P, _ptr(out), _ptr(err),
              _stream(stream)), name)
    return out


def mnw_moe_grouped_gemm_w8a16_f16rows(layer, kind, a, row_outer, expert_offsets, err=None, stream=None):
    return _gemm_f16rows("mnw_moe_grouped_gemm_w8a16_f16rows", layer, kind, a, row_outer, expert_offsets, err,
                         stream)


def mnw_moe_grouped_gemm_w4a16_f16rows(layer, kind, a, row_outer, expert_offsets, err=None, stream=None):
    return _gemm_f16rows("mnw_moe_grouped_gemm_w4a16_f16rows", layer, kind, a, row_outer, expert_offsets, err,
                         stream)


def _gemm_a8(name, layer, kind, a_codes, a_scales, expert_offsets, want_dots=False, err=None, stream=None):
    P, K = a_codes.shape
    out = _gemm_out(layer, kind, P, a_codes.device)
    dots = None
    if want_dots:
        C = (2 * layer.I) if kind == KIND_GATE_UP else (layer.H if kind == KIND_DOWN else layer.I)
        dots = torch.zeros((P, C, K // 128), dtype=torch.int32, device=a_codes.device)
    fn = getattr(load(), name)
    _check(fn(layer.handle, kind, _ptr(a_codes), _ptr(a_scales), _ptr(expert_offsets), P, _ptr(out), _ptr(dots),
              _ptr(err), _stream(stream)), name)
    return (out, dots) if want_dots else out


def mnw_moe_grouped_gemm_w8a8(layer, kind, a_codes, a_scales, expert_offsets, want_dots=False, err=None, stream=None):
    return _gemm_a8("mnw_moe_grouped_gemm_w8a8", layer, kind, a_codes, a_scales, expert_offsets, want_dots, err,
                    stream)


def mnw_moe_grouped_gemm_w4a8(layer, kind, a_codes, a_scales, expert_offsets, want_dots=False, err=None, stream=None):
    return _gemm_a8("mnw_moe_grouped_gemm_w4a8", layer, kind, a_codes, a_scales, expert_offsets, want_dots, err,
                    stream)


def mnw_moe_grouped_gemm_nvfp4(layer, kind, a_codes, a_sf, a_outer, expert_offsets, err=None, stream=None):
    P = a_codes.shape[0]
    out = _gemm_out(layer, kind, P, a_codes.device)
    _check(load().mnw_moe_grouped_gemm_nvfp4(layer.handle, kind, _ptr(a_codes), _ptr(a_sf), _ptr(a_outer),
                                             _ptr(expert_offsets), P, _ptr(out), _ptr(err), _stream(stream)),
           "mnw_moe_grouped_gemm_nvfp4")
    return out


def mnw_moe_combine(y, assign_pos, w, stream=None, out=None):
    T, k = w.shape
    H = y.shape[1]
    if out is None:
        out = torch.empty((T, H), dtype=torch.bfloat16, device=y.device)
    _check(load().mnw_moe_combine(_ptr(y), _ptr(assign_pos), _ptr(w), T, k, H, _ptr(out), _stream(stream)),
           "mnw_moe_combine")
    return out


def mnw_moe_workspace_size(layer, act, T, k) -> int:
    return int(load().mnw_moe_workspace_size(layer.handle, act, T, k))


def mnw_moe_workspace_size_host(layer, act, T, k) -> int:
    return int(load().mnw_moe_workspace_size_host(layer.handle, act, T, k))


def workspace(layer, act, T, k, host=False, device=None) -> torch.Tensor:
    n = mnw_moe_workspace_size_host(layer, act, T, k) if host else mnw_moe_workspace_size(layer, act, T, k)
    return torch.empty(max(n, 256), dtype=torch.uint8, device=device or layer.blob.device)


def mnw_moe_forward(layer, act, x, ids, w, ws=None, out=None, stream=None):
    T, k = ids.shape
    if ws is None:
        ws = workspace(layer, act, T, k, device=x.device)
    if out is None:
        out = torch.empty((T, layer.H), dtype=torch.bfloat16, device=x.device)
    _check(load().mnw_moe_forward(layer.handle, act, _ptr(x), _ptr(ids), _ptr(w), T, k, _ptr(out), _ptr(ws),
                                  ws.numel(), _stream(stream)), "mnw_moe_forward")
    return out


def mnw_moe_forward_host(layer, act, x_host, ids_host, w_host, ws, out_host, stream=None):
    """Host tensors in and out (pinned memory gives overlap); synchronises."""
    T, k = ids_host.shape
    _check(load().mnw_moe_forward_host(layer.handle, act, ctypes.c_void_p(x_host.data_ptr()),
                                       ctypes.c_void_p(ids_host.data_ptr()), ctypes.c_void_p(w_host.data_ptr()),
                                       T, k, ctypes.c_void_p(out_host.data_ptr()), _ptr(ws), ws.numel(),
                                       _stream(stream)), "mnw_moe_forward_host")
    return out_host


def workspace_error_word(ws):
    """The forward's device error word as an int32 view of ws[0:4]."""
    return ws[:4].view(torch.int32)


def mnw_moe_read_error(err, stream=None) -> int:
    out = ctypes.c_uint32()
    _check(load().mnw_moe_read_error(_ptr(err), ctypes.byref(out), _stream(stream)), "mnw_moe_read_error")
    return out.value


def mnw_moe_launch_count() -> int:
    """Kernels this library has enqueued since it was loaded (host-side count)."""
    return int(load().mnw_moe_launch_count())


def mnw_moe_set_gemm_path(path: int) -> None:
    """Process-wide grouped-GEMM kernel choice (PATH_AUTO, PATH_TCGEN05, PATH_WARP_MMA)."""
    _check(load().mnw_moe_set_gemm_path(path), "mnw_moe_set_gemm_path")


STATIC_WS_BYTES = 32 * 1024 * 1024


def mnw_moe_forward_static(layer, act, x, ids, w, out=None, err=None, stream=None):
    """The whole layer with the library's built-in scratch array: no workspace
    and no device allocation by the library (see include/mnw_moe.h)."""
    T, k = ids.shape
    if out is None:
        out = torch.empty((T, layer.H), dtype=torch.bfloat16, device=x.device)
    _check(load().mnw_moe_forward_static(layer.handle, act, _ptr(x), _ptr(ids), _ptr(w), T, k, _ptr(out), _ptr(err),
                                         _stream(stream)), "mnw_moe_forward_static")
    return out


def mnw_moe_selftest_wait_timeout(limit_us, err, left_early, stream=None):
    """Launch the bounded-wait self-test (see include/mnw_moe.h); err and
    left_early are zeroed int32 device tensors of one element."""
    _check(load().mnw_moe_selftest_wait_timeout(limit_us, _ptr(err), _ptr(left_early), _stream(stream)),
           "mnw_moe_selftest_wait_timeout")


def mnw_moe_selftest_counter_timeout(limit_us, counter, need, err, stream=None):
    """Launch the token-tile counter wait self-test (see include/mnw_moe.h);
    counter and err are int32 device tensors of one element."""
    _check(load().mnw_moe_selftest_counter_timeout(limit_us, _ptr(counter), need, _ptr(err), _stream(stream)),
           "mnw_moe_selftest_counter_timeout")
