"""CPU oracle of the routed-expert MoE layer -- TEST INFRASTRUCTURE ONLY.

Loads ``moe_oracle.c`` (plain single-threaded C, FP64 accumulation) through
ctypes, compiling it with gcc on first use.  Only ``tests/``,
``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg may import this
package; the CUDA product path never does.

The arrays passed in and out are numpy arrays; BF16 tensors travel as their
uint16 bit patterns.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_HDR = os.path.join(_HERE, "moe_oracle.h")
_BUILD = os.path.join(_HERE, "_build")
_SO = os.path.join(_BUILD, "libmnw_moe_oracle.so")
_lock = threading.Lock()
_lib = None

FMT_BF16, FMT_INT8_G128, FMT_INT4_G128, FMT_NVFP4_G16 = 0, 1, 2, 3
ACT_BF16, ACT_INT8_G128, ACT_NVFP4_G16 = 0, 1, 2
ACT_F16_ROWS = 3  # FP16 rows with a power-of-two row factor (see encode_f16_rows)
KIND_GATE_UP, KIND_DOWN, KIND_GATE, KIND_UP = 0, 1, 2, 3


def build(force: bool = False) -> str:
    """Compile the oracle into ``oracle/_build`` (gcc, -O2, no FMA contraction)."""
    os.makedirs(_BUILD, exist_ok=True)
    newest = max(os.path.getmtime(_SRC), os.path.getmtime(_HDR))
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < newest:
        tmp = _SO + f".{os.getpid()}.tmp"
        cmd = ["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
               "-shared", "-Wall", "-Wextra", "-Wno-unused-parameter", "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _SO)
    return _SO


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        i32, u8, u16, f32, f64 = ctypes.c_int, ctypes.c_uint8, ctypes.c_uint16, ctypes.c_float, ctypes.c_double
        sig = {
            "mnwo_bf16_to_double": (f64, [u16]),
            "mnwo_fp16_to_double": (i32, [u16, P]),
            "mnwo_int4_value": (i32, [u8]),
            "mnwo_int8_value": (i32, [u8]),
            "mnwo_e2m1_to_double": (f64, [u8]),
            "mnwo_e4m3_to_double": (i32, [u8, P]),
            "mnwo_bf16_from_double": (u16, [f64]),
            "mnwo_fp16_from_double": (u16, [f64]),
            "mnwo_e4m3_rn_satfinite": (u8, [f32]),
            "mnwo_e2m1_rn_satfinite": (u8, [f32]),
            "mnwo_quant_int8_g128": (i32, [P, i32, i32, P, P]),
            "mnwo_quant_nvfp4_g16": (i32, [P, i32, i32, P, P, P]),
            "mnwo_encode_f16_rows": (i32, [P, i32, i32, P, P]),
            "mnwo_permute": (i32, [P, i32, i32, i32, P, P, P]),
            "mnwo_route": (i32, [P, P, i32, i32, i32, i32, P, P, P]),
            "mnwo_silu_mul": (None, [P, P, ctypes.c_size_t, P]),
            "mnwo_gemm_a16": (i32, [P, ctypes.c_size_t, i32, P, P, i32, P]),
            "mnwo_gemm_a8": (i32, [P, ctypes.c_size_t, i32, P, P, P, i32, P, P]),
            "mnwo_gemm_a4": (i32, [P, ctypes.c_size_t, i32, P, P, P, P, i32, P]),
            "mnwo_gemm_f16rows": (i32, [P, ctypes.c_size_t, i32, P, P, P, i32, P]),
            "mnwo_combine": (None, [P, P, P, i32, i32, i32, P]),
            "mnwo_moe_forward": (i32, [P, ctypes.c_size_t, i32, P, P, P, i32, i32, P, i32, P]),
            "mnwo_attention": (i32, [P, P, P, i32, i32, i32, i32, i32, i32, f64, P, i32, P]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
        return lib


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def _check(rc, what):
    if rc != 0:
        raise ValueError(f"oracle {what} failed with code {rc}")


# ---- scalar helpers ---------------------------------------------------------

def bf16_to_double(bits: int) -> float:
    return _load().mnwo_bf16_to_double(bits)


def fp16_to_double(bits: int) -> float:
    out = ctypes.c_double()
    _check(_load().mnwo_fp16_to_double(bits, ctypes.byref(out)), "fp16 decode")
    return out.value


def int4_value(nibble: int) -> int:
    return _load().mnwo_int4_value(nibble)


def int8_value(byte: int) -> int:
    return _load().mnwo_int8_value(byte)


def e2m1_to_double(nibble: int) -> float:
    return _load().mnwo_e2m1_to_double(nibble)


def e4m3_to_double(byte: int) -> float:
    out = ctypes.c_double()
    _check(_load().mnwo_e4m3_to_double(byte, ctypes.byref(out)), "e4m3 decode")
    return out.value


def bf16_from_double(v: float) -> int:
    return _load().mnwo_bf16_from_double(v)


def fp16_from_double(v: float) -> int:
    return _load().mnwo_fp16_from_double(v)


def e4m3_rn_satfinite(v: float) -> int:
    return _load().mnwo_e4m3_rn_satfinite(v)


def e2m1_rn_satfinite(v: float) -> int:
    return _load().mnwo_e2m1_rn_satfinite(v)


# ---- array functions ----------------------------------------------------------

def quant_int8_g128(x_bf16: np.ndarray):
    x = _c(x_bf16, np.uint16)
    R, K = x.shape
    codes = np.zeros((R, K), np.int8)
    scales = np.zeros((R, K // 128), np.float32)
    _check(_load().mnwo_quant_int8_g128(_p(x), R, K, _p(codes), _p(scales)), "quant_int8_g128")
    return codes, scales


def quant_nvfp4_g16(x_bf16: np.ndarray):
    x = _c(x_bf16, np.uint16)
    R, K = x.shape
    codes = np.zeros((R, K // 2), np.uint8)
    sf = np.zeros((R, K // 16), np.uint8)
    outer = np.zeros((R,), np.float32)
    _check(_load().mnwo_quant_nvfp4_g16(_p(x), R, K, _p(codes), _p(sf), _p(outer)), "quant_nvfp4_g16")
    return codes, sf, outer


def encode_f16_rows(x_bf16: np.ndarray):
    """FP16 codes (uint16 bits) and power-of-two row factors of BF16 rows."""
    x = _c(x_bf16, np.uint16)
    R, K = x.shape
    codes = np.zeros((R, K), np.uint16)
    factor = np.zeros((R,), np.float32)
    _check(_load().mnwo_encode_f16_rows(_p(x), R, K, _p(codes), _p(factor)), "encode_f16_rows")
    return codes, factor


def route(x_bf16: np.ndarray, wr_bf16: np.ndarray, k: int):
    """Router of the GPU-routing path: (ids int32 [T,k], w float32 [T,k],
    logits float64 [T,E]); see mnwo_route for the reading of the pages."""
    x = _c(x_bf16, np.uint16)
    wr = _c(wr_bf16, np.uint16)
    T, H = x.shape
    E = wr.shape[0]
    ids = np.zeros((T, k), np.int32)
    w = np.zeros((T, k), np.float32)
    logits = np.zeros((T, E), np.float64)
    _check(_load().mnwo_route(_p(x), _p(wr), T, H, E, k, _p(ids), _p(w), _p(logits)), "route")
    return ids, w, logits


def permute(ids: np.ndarray, E: int):
    ids = _c(ids, np.int32)
    T, k = ids.shape
    P = T * k
    offsets = np.zeros((E + 1,), np.int32)
    sorted_assign = np.zeros((P,), np.int32)
    assign_pos = np.zeros((P,), np.int32)
    dropped = _load().mnwo_permute(_p(ids), T, k, E, _p(offsets), _p(sorted_assign), _p(assign_pos))
    if dropped < 0:
        raise ValueError("oracle permute: bad arguments")
    return offsets, sorted_assign, assign_pos, dropped


def _dims(blob: np.ndarray):
    hdr = blob[:32].view(np.uint32)
    return int(hdr[3]), int(hdr[4]), int(hdr[5])  # E, H, I


def gemm_a16(blob: np.ndarray, kind: int, a_bf16: np.ndarray, offsets: np.ndarray):
    blob = _c(blob, np.uint8)
    a = _c(a_bf16, np.uint16)
    off = _c(offsets, np.int32)
    E, H, I = _dims(blob)
    P = a.shape[0]
    out = np.zeros((P, H if kind == KIND_DOWN else I), np.uint16)
    _check(_load().mnwo_gemm_a16(_p(blob), blob.nbytes, kind, _p(a), _p(off), P, _p(out)), "gemm_a16")
    return out


def gemm_a8(blob: np.ndarray, kind: int, a_codes, a_scales, offsets, want_dots: bool = False):
    blob = _c(blob, np.uint8)
    q = _c(a_codes, np.int8)
    s = _c(a_scales, np.float32)
    off = _c(offsets, np.int32)
    E, H, I = _dims(blob)
    P, K = q.shape
    N = H if kind == KIND_DOWN else I
    out = np.zeros((P, N), np.uint16)
    dots = np.zeros((P, (2 if kind == KIND_GATE_UP else 1) * N, K // 128), np.int32) if want_dots else None
    _check(_load().mnwo_gemm_a8(_p(blob), blob.nbytes, kind, _p(q), _p(s), _p(off), P, _p(out), _p(dots)),
           "gemm_a8")
    return (out, dots) if want_dots else out


def gemm_a4(blob: np.ndarray, kind: int, a_codes, a_sf, a_outer, offsets):
    blob = _c(blob, np.uint8)
    c = _c(a_codes, np.uint8)
    sf = _c(a_sf, np.uint8)
    o = _c(a_outer, np.float32)
    off = _c(offsets, np.int32)
    E, H, I = _dims(blob)
    P = c.shape[0]
    out = np.zeros((P, H if kind == KIND_DOWN else I), np.uint16)
    _check(_load().mnwo_gemm_a4(_p(blob), blob.nbytes, kind, _p(c), _p(sf), _p(o), _p(off), P, _p(out)),
           "gemm_a4")
    return out


def gemm_f16rows(blob: np.ndarray, kind: int, a_f16: np.ndarray, factor, offsets):
    blob = _c(blob, np.uint8)
    a = _c(a_f16, np.uint16)
    f = _c(factor, np.float32)
    off = _c(offsets, np.int32)
    E, H, I = _dims(blob)
    P = a.shape[0]
    out = np.zeros((P, H if kind == KIND_DOWN else I), np.uint16)
    _check(_load().mnwo_gemm_f16rows(_p(blob), blob.nbytes, kind, _p(a), _p(f), _p(off), P, _p(out)),
           "gemm_f16rows")
    return out


def silu_mul(g_bf16, u_bf16):
    """bf16(SiLU(g) * u) of BF16 g and u (the unfused activation), FP64 inside."""
    g = _c(g_bf16, np.uint16)
    u = _c(u_bf16, np.uint16)
    assert g.shape == u.shape
    out = np.zeros(g.shape, np.uint16)
    _load().mnwo_silu_mul(_p(g), _p(u), g.size, _p(out))
    return out


def combine(y_bf16, assign_pos, w, T: int, k: int):
    y = _c(y_bf16, np.uint16)
    pos = _c(assign_pos, np.int32)
    ww = _c(w, np.float32)
    H = y.shape[1]
    out = np.zeros((T, H), np.uint16)
    _load().mnwo_combine(_p(y), _p(pos), _p(ww), T, k, H, _p(out))
    return out


def moe_forward(blob, act: int, x_bf16, ids, w, rows=None):
    blob = _c(blob, np.uint8)
    x = _c(x_bf16, np.uint16)
    i = _c(ids, np.int32)
    ww = _c(w, np.float32)
    T, k = i.shape
    H = x.shape[1]
    r = None if rows is None else _c(rows, np.int32)
    n = T if r is None else r.shape[0]
    out = np.zeros((n, H), np.uint16)
    _check(_load().mnwo_moe_forward(_p(blob), blob.nbytes, act, _p(x), _p(i), _p(ww), T, k, _p(r), n, _p(out)),
           "moe_forward")
    return out


def attention(q_bf16, k_bf16, v_bf16, blk: int, scale: float, rows=None):
    """Block attention (FP64) of BF16 q [B, T, Hq, d] with k, v [B, T, Hkv, d]:
    key j is allowed for token t when j / blk <= t / blk.  Returns FP64
    [B, T, Hq, d], or [len(rows), Hq, d] for the flat token indices in rows."""
    q = _c(q_bf16, np.uint16)
    k = _c(k_bf16, np.uint16)
    v = _c(v_bf16, np.uint16)
    B, T, Hq, d = q.shape
    Hkv = k.shape[2]
    assert k.shape == (B, T, Hkv, d) and v.shape == k.shape
    r = None if rows is None else _c(rows, np.int32)
    n = B * T if r is None else r.size
    out = np.zeros((n, Hq, d), np.float64)
    _check(_load().mnwo_attention(_p(q), _p(k), _p(v), B, T, Hq, Hkv, d, int(blk), float(scale), _p(r),
                                  0 if r is None else n, _p(out)), "attention")
    return out.reshape(B, T, Hq, d) if r is None else out
