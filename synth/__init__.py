"""Seeded synthetic inputs for the routed-expert MoE layer.

This module serves both the CUDA path and the CPU oracle, and holds none of
the layer's arithmetic.  It draws:

* BF16 activations ~N(0, 1), optionally with sparse x20 outliers;
* top-k expert ids (uniform, Zipf-skewed or hot/cold) and routing weights
  (softmax of k N(0, 1) logits, float32);
* expert-weight blobs in the four storage formats.  INT8/INT4 weights are
  N(0, sigma) values quantised with one FP16 absmax scale per 128 along K (the
  workload recipe; the pages give no converter rule).  NVFP4 weights are drawn
  directly as E2M1 codes, E4M3 block-scale bytes and an FP32 outer scale, so
  that no FP4/FP8 rounding lives here.

Every random number comes from a counter-based 32-bit hash of
(seed, stream, index) computed with integer tensor ops only; normals come from
a fixed table of N(0, 1) quantiles indexed by 16 hash bits, so activations,
uniform routing and weight codes are the same bits on CPU and GPU.  The few
floating steps (softmax weights, Zipf keys) may differ in the last ulp between
devices: a comparison draws its inputs once, on one device, and copies them.

The blob layout written here is documented in ``include/mnw_moe.h``.
"""
from __future__ import annotations

import math
import statistics
import struct
import zlib
from dataclasses import dataclass, field

import torch

FMT_BF16, FMT_INT8_G128, FMT_INT4_G128, FMT_NVFP4_G16 = 0, 1, 2, 3
ACT_BF16, ACT_INT8_G128, ACT_NVFP4_G16 = 0, 1, 2
GATE, UP, DOWN = 0, 1, 2
_M32 = 0xFFFFFFFF

# ---------------------------------------------------------------------------
# counter-based bits
# ---------------------------------------------------------------------------


def _mul32(x: torch.Tensor, c: int) -> torch.Tensor:
    """(x * c) mod 2^32 for 0 <= x < 2^32 without int64 overflow."""
    lo, hi = c & 0xFFFF, c >> 16
    return (x * lo + (((x * hi) & 0xFFFF) << 16)) & _M32


def _mix32(x: torch.Tensor) -> torch.Tensor:
    """A 32-bit integer finaliser (xorshift-multiply rounds)."""
    x = x ^ (x >> 16)
    x = _mul32(x, 0x7FEB352D)
    x = x ^ (x >> 15)
    x = _mul32(x, 0x846CA68B)
    x = x ^ (x >> 16)
    return x


def _key(seed: int, stream: int, salt: int) -> int:
    t = torch.tensor([(seed * 0x9E3779B1 + stream * 0x85EBCA77 + salt * 0xC2B2AE3D) & _M32], dtype=torch.int64)
    return int(_mix32(_mix32(t))[0])


def bits32(seed: int, stream: int, idx: torch.Tensor) -> torch.Tensor:
    """Uniform 32-bit values (int64 tensor) for counters ``idx``."""
    k1, k2 = _key(seed, stream, 1), _key(seed, stream, 2)
    lo = idx & _M32
    hi = idx >> 32
    h = _mix32(lo ^ k1)
    return _mix32(h ^ hi ^ k2)


def _counters(n: int, device, start: int = 0) -> torch.Tensor:
    return torch.arange(start, start + n, dtype=torch.int64, device=device)


_QTABLE = {}


def _normal_table(device) -> torch.Tensor:
    """N(0,1) quantiles at (i + 0.5) / 65536, float64 (computed once on the host)."""
    key = str(device)
    if key not in _QTABLE:
        nd = statistics.NormalDist()
        vals = [nd.inv_cdf((i + 0.5) / 65536.0) for i in range(65536)]
        _QTABLE[key] = torch.tensor(vals, dtype=torch.float64, device=device)
    return _QTABLE[key]


def normal_f64(seed: int, stream: int, n: int, device, start: int = 0) -> torch.Tensor:
    """n draws ~N(0,1) (quantile table, 16 bits each) as float64."""
    b = bits32(seed, stream, _counters(n, device, start))
    return _normal_table(device)[b & 0xFFFF]


def to_bf16_bits(v: torch.Tensor) -> torch.Tensor:
    """BF16 (round to nearest even) of a float tensor, as int16 bit patterns."""
    return v.to(torch.float32).to(torch.bfloat16).view(torch.int16)


# ---------------------------------------------------------------------------
# activations and routing
# ---------------------------------------------------------------------------


def activations(T: int, H: int, seed: int, device="cpu", outlier_p: float = 0.0,
                outlier_scale: float = 20.0, stream: int = 100) -> torch.Tensor:
    """x [T, H] bf16 ~N(0,1); with probability outlier_p an element is scaled by outlier_scale."""
    v = normal_f64(seed, stream, T * H, device)
    if outlier_p > 0:
        u = bits32(seed, stream + 1, _counters(T * H, device))
        thresh = int(outlier_p * 4294967296.0)
        v = torch.where(u < thresh, v * outlier_scale, v)
    return v.to(torch.float32).to(torch.bfloat16).reshape(T, H)


def routing_uniform(T: int, E: int, k: int, seed: int, device="cpu", stream: int = 200) -> torch.Tensor:
    """k distinct experts per token, uniform: the k largest of E hashed keys."""
    keys = bits32(seed, stream, _counters(T * E, device)).reshape(T, E)
    keys = keys * 1024 + torch.arange(E, device=device)  # unique keys break ties
    return torch.topk(keys, k, dim=1).indices.to(torch.int32)


def routing_zipf(T: int, E: int, k: int, seed: int, alpha: float = 1.1, device="cpu",
                 stream: int = 210) -> torch.Tensor:
    """k distinct experts per token, Zipf(alpha) popularity over a seeded permutation
    of experts, drawn by Gumbel-top-k on the log-probabilities."""
    perm_keys = bits32(seed, stream, _counters(E, device)) * 1024 + torch.arange(E, device=device)
    order = torch.argsort(perm_keys)  # rank r -> expert order[r]
    logp_rank = -alpha * torch.log(torch.arange(1, E + 1, dtype=torch.float64, device=device))
    logp = torch.empty(E, dtype=torch.float64, device=device)
    logp[order] = logp_rank
    u = (bits32(seed, stream + 1, _counters(T * E, device)).to(torch.float64) + 0.5) / 4294967296.0
    gumbel = -torch.log(-torch.log(u))
    keys = logp.unsqueeze(0) + gumbel.reshape(T, E)
    return torch.topk(keys, k, dim=1).indices.to(torch.int32)


def routing_hot_cold(T: int, E: int, k: int, seed: int, hot_frac: float = 0.10, n_empty: int = 16,
                     device="cpu", stream: int = 220) -> torch.Tensor:
    """Skewed routing: round(hot_frac*E) hot experts receive k/2 of every token's slots,
    n_empty experts receive none, the rest share the other k/2 slots uniformly."""
    n_hot = int(round(hot_frac * E))
    perm_keys = bits32(seed, stream, _counters(E, device)) * 1024 + torch.arange(E, device=device)
    order = torch.argsort(perm_keys)
    hot = order[:n_hot]
    cold = order[n_hot:E - n_empty]
    kh = k // 2
    kc = k - kh
    kh_keys = bits32(seed, stream + 1, _counters(T * n_hot, device)).reshape(T, n_hot) * 1024 + \
        torch.arange(n_hot, device=device)
    kc_keys = bits32(seed, stream + 2, _counters(T * cold.numel(), device)).reshape(T, -1) * 1024 + \
        torch.arange(cold.numel(), device=device)
    ids = torch.cat([hot[torch.topk(kh_keys, kh, dim=1).indices],
                     cold[torch.topk(kc_keys, kc, dim=1).indices]], dim=1)
    # interleave the slot order per token so hot slots are not always first
    slot_keys = bits32(seed, stream + 3, _counters(T * k, device)).reshape(T, k) * 16 + torch.arange(k, device=device)
    ids = torch.gather(ids, 1, torch.argsort(slot_keys, dim=1))
    return ids.to(torch.int32)


def router_weights(E: int, H: int, seed: int, device="cpu", stream: int = 400) -> torch.Tensor:
    """Router matrix [E, H] bf16 ~N(0, 1/H), so that logits of N(0,1) tokens are ~N(0, 1)."""
    v = normal_f64(seed, stream, E * H, device) / math.sqrt(H)
    return v.to(torch.float32).to(torch.bfloat16).reshape(E, H)


def routing_weights(T: int, k: int, seed: int, device="cpu", stream: int = 300) -> torch.Tensor:
    """float32 [T, k]: softmax over k N(0,1) logits."""
    logits = normal_f64(seed, stream, T * k, device).reshape(T, k)
    return torch.softmax(logits, dim=1).to(torch.float32)


# ---------------------------------------------------------------------------
# expert-weight blob
# ---------------------------------------------------------------------------

ALIGN = 256


def _align(x: int) -> int:
    return (x + ALIGN - 1) // ALIGN * ALIGN


@dataclass
class BlobLayout:
    wfmt: int
    E: int
    H: int
    I: int
    group: int
    expert_stride: int
    codes_off: list = field(default_factory=list)
    scales_off: list = field(default_factory=list)
    outer_off: list = field(default_factory=list)
    data_offset: int = 256

    @property
    def total_bytes(self) -> int:
        return self.data_offset + self.E * self.expert_stride

    def dims(self, m: int):
        return (self.H, self.I) if m == DOWN else (self.I, self.H)


def code_bytes(wfmt: int, N: int, K: int) -> int:
    return {FMT_BF16: N * K * 2, FMT_INT8_G128: N * K, FMT_INT4_G128: N * K // 2, FMT_NVFP4_G16: N * K // 2}[wfmt]


def scale_bytes(wfmt: int, N: int, K: int) -> int:
    return {FMT_BF16: 0, FMT_INT8_G128: N * (K // 128) * 2, FMT_INT4_G128: N * (K // 128) * 2,
            FMT_NVFP4_G16: N * (K // 16)}[wfmt]


def layout(wfmt: int, E: int, H: int, I: int) -> BlobLayout:
    group = {FMT_BF16: 0, FMT_INT8_G128: 128, FMT_INT4_G128: 128, FMT_NVFP4_G16: 16}[wfmt]
    L = BlobLayout(wfmt, E, H, I, group, 0)
    off = 0
    for m in (GATE, UP, DOWN):
        N, K = L.dims(m)
        L.codes_off.append(off)
        off = _align(off + code_bytes(wfmt, N, K))
        if scale_bytes(wfmt, N, K):
            L.scales_off.append(off)
            off = _align(off + scale_bytes(wfmt, N, K))
        else:
            L.scales_off.append(0)
        if wfmt == FMT_NVFP4_G16:
            L.outer_off.append(off)
            off = _align(off + 4)
        else:
            L.outer_off.append(0)
    L.expert_stride = off
    return L


def header_bytes(L: BlobLayout) -> bytes:
    h = bytearray(256)
    struct.pack_into("<4sIIIIIII", h, 0, b"MNWB", 1, L.wfmt, L.E, L.H, L.I, L.group, 256)
    struct.pack_into("<QQ", h, 32, L.data_offset, L.expert_stride)
    struct.pack_into("<3Q", h, 48, *L.codes_off)
    struct.pack_into("<3Q", h, 72, *L.scales_off)
    struct.pack_into("<3Q", h, 96, *L.outer_off)
    struct.pack_into("<Q", h, 120, L.total_bytes)
    struct.pack_into("<I", h, 252, zlib.crc32(bytes(h[:252])) & _M32)
    return bytes(h)


def _quantise_absmax(w: torch.Tensor, qmax: int, qmin: int):
    """Workload recipe for INT8/INT4 weights: per (row, 128 along K) group,
    s = fp16(absmax / qmax), q = clamp(round_half_even(w / s), qmin, qmax);
    an all-zero group gets s = 0, q = 0."""
    N, K = w.shape[-2], w.shape[-1]
    g = w.reshape(*w.shape[:-1], K // 128, 128)
    amax = g.abs().amax(dim=-1, keepdim=True)
    s16 = (amax / qmax).to(torch.float16)
    s = s16.to(torch.float64)
    q = torch.where(s > 0, torch.round(g / torch.where(s > 0, s, torch.ones_like(s))), torch.zeros_like(g))
    q = q.clamp(qmin, qmax).to(torch.int16).reshape(w.shape)
    return q, s16.reshape(*w.shape[:-1], K // 128)


def _pack_nibbles(q: torch.Tensor) -> torch.Tensor:
    """int [.., K] in [-8, 7] -> uint8 [.., K/2], even index in the low nibble."""
    u = (q.to(torch.int16) & 0xF).to(torch.uint8)
    return u[..., 0::2] | (u[..., 1::2] << 4)


def _nvfp4_matrix(seed: int, stream: int, E: int, N: int, K: int, device, sigma: float,
                  sf_range: str = "narrow"):
    """Direct draw of NVFP4 weights: E2M1 magnitude index from a fixed
    half-normal-like table, uniform sign.  sf_range "narrow" (the workloads):
    E4M3 block-scale bytes uniform in [0x30, 0x38] (0.5 .. 1.0), outer =
    sigma / 1.6 per matrix with a gentle per-expert jitter.  sf_range "full"
    (edge-case tests): block-scale bytes uniform over every non-negative
    finite E4M3 code 0x00 .. 0x7E (zero, the subnormals 2^-9 .. 7 * 2^-9, up
    to 448), and outer scales spread over 2^-3 .. 2^3 around a base chosen so
    that the weights' RMS stays near sigma."""
    n = E * N * K
    b = bits32(seed, stream, _counters(n, device))
    # magnitude index 0..7 -> thresholds on 16 bits (cumulative probabilities)
    cum = torch.tensor([11000, 25000, 38000, 48500, 56000, 62000, 64900, 65536], dtype=torch.int64, device=device)
    mag = torch.searchsorted(cum, (b & 0xFFFF), right=True).clamp_max(7)
    sign = (b >> 16) & 1
    codes = (mag | (sign << 3)).to(torch.uint8).reshape(E, N, K)
    packed = codes[..., 0::2] | (codes[..., 1::2] << 4)
    sb = bits32(seed, stream + 1, _counters(E * N * (K // 16), device))
    jit = bits32(seed, stream + 2, _counters(E, device)).to(torch.float64) / 4294967296.0
    if sf_range == "full":
        sf = (sb % 127).to(torch.uint8).reshape(E, N, K // 16)
        # RMS of a block scale drawn uniformly over the 127 codes is about 110,
        # of an E2M1 value from the table about 1.6
        outer = ((sigma / 176.0) * torch.pow(2.0, 6.0 * jit - 3.0)).to(torch.float32)
    else:
        sf = (0x30 + (sb % 9)).to(torch.uint8).reshape(E, N, K // 16)
        outer = ((sigma / 1.6) * (0.75 + 0.5 * jit)).to(torch.float32)
    return packed, sf, outer


def expert_blob(wfmt: int, E: int, H: int, I: int, seed: int, sigma: float = 0.02,
                device="cpu", stream: int = 1000, nvfp4_sf_range: str = "narrow"):
    """Build the packed expert blob.  Returns (blob uint8 tensor on `device`,
    header bytes, BlobLayout).  nvfp4_sf_range: see _nvfp4_matrix."""
    L = layout(wfmt, E, H, I)
    body = torch.zeros((E, L.expert_stride), dtype=torch.uint8, device=device)
    for m in (GATE, UP, DOWN):
        N, K = L.dims(m)
        st = stream + 10 * m
        c0 = L.codes_off[m]
        if wfmt == FMT_NVFP4_G16:
            packed, sf, outer = _nvfp4_matrix(seed, st, E, N, K, device, sigma, nvfp4_sf_range)
            body[:, c0:c0 + N * K // 2] = packed.reshape(E, -1)
            s0 = L.scales_off[m]
            body[:, s0:s0 + N * K // 16] = sf.reshape(E, -1)
            o0 = L.outer_off[m]
            body[:, o0:o0 + 4] = outer.reshape(E, 1).view(torch.uint8).reshape(E, 4)
            continue
        # blocks of experts at a time to bound the working set
        per = N * K
        step = max(1, min(E, (1 << 25) // per))
        for e0 in range(0, E, step):
            ne = min(step, E - e0)
            w = normal_f64(seed, st, ne * per, device, start=e0 * per).reshape(ne, N, K) * sigma
            rows = body[e0:e0 + ne]
            if wfmt == FMT_BF16:
                rows[:, c0:c0 + per * 2] = w.to(torch.float32).to(torch.bfloat16).view(torch.uint8).reshape(ne, -1)
                continue
            if wfmt == FMT_INT8_G128:
                q, s16 = _quantise_absmax(w, 127, -127)
                rows[:, c0:c0 + per] = q.to(torch.int8).view(torch.uint8).reshape(ne, -1)
            else:
                q, s16 = _quantise_absmax(w, 7, -8)
                rows[:, c0:c0 + per // 2] = _pack_nibbles(q).reshape(ne, -1)
            s0 = L.scales_off[m]
            rows[:, s0:s0 + N * (K // 128) * 2] = s16.contiguous().view(torch.uint8).reshape(ne, -1)
    hdr = header_bytes(L)
    blob = torch.empty((L.total_bytes,), dtype=torch.uint8, device=device)
    blob[:256] = torch.frombuffer(bytearray(hdr), dtype=torch.uint8).to(device)
    blob[256:] = body.reshape(-1)
    return blob, hdr, L


# ---------------------------------------------------------------------------
# the workloads
# ---------------------------------------------------------------------------


@dataclass
class Workload:
    name: str
    T: int
    H: int
    E: int
    I: int
    k: int
    wfmt: int
    act: int
    sigma: float
    routing: str          # "uniform" | "zipf" | "hot_cold"
    seed: int
    outlier_p: float = 0.0

    @property
    def P(self) -> int:
        return self.T * self.k


WORKLOADS = {
    "tiny_w8a16": Workload("tiny_w8a16", 32, 256, 8, 128, 2, FMT_INT8_G128, ACT_BF16, 0.02, "uniform", 0),
    "decode_w4a16": Workload("decode_w4a16", 256, 2048, 256, 512, 8, FMT_INT4_G128, ACT_BF16, 0.02, "uniform", 1),
    "w8a8_2048": Workload("w8a8_2048", 2048, 2048, 256, 512, 8, FMT_INT8_G128, ACT_INT8_G128, 0.02, "uniform", 2,
                          outlier_p=0.01),
    "prefill_nvfp4": Workload("prefill_nvfp4", 8192, 2048, 256, 512, 8, FMT_NVFP4_G16, ACT_NVFP4_G16, 0.02, "zipf", 3),
    "large_w4a16": Workload("large_w4a16", 4096, 4096, 256, 1536, 8, FMT_INT4_G128, ACT_BF16, 0.015, "hot_cold", 4),
    "large_bf16": Workload("large_bf16", 4096, 4096, 256, 1536, 8, FMT_BF16, ACT_BF16, 0.015, "hot_cold", 4),
}


def make_inputs(wl: Workload, device="cpu"):
    """(x bf16 [T,H], ids int32 [T,k], w float32 [T,k], blob uint8, header bytes, layout)."""
    x = activations(wl.T, wl.H, wl.seed, device, outlier_p=wl.outlier_p)
    if wl.routing == "uniform":
        ids = routing_uniform(wl.T, wl.E, wl.k, wl.seed, device)
    elif wl.routing == "zipf":
        ids = routing_zipf(wl.T, wl.E, wl.k, wl.seed, device=device)
    else:
        ids = routing_hot_cold(wl.T, wl.E, wl.k, wl.seed, device=device)
    w = routing_weights(wl.T, wl.k, wl.seed, device)
    blob, hdr, L = expert_blob(wl.wfmt, wl.E, wl.H, wl.I, wl.seed, wl.sigma, device)
    return x, ids, w, blob, hdr, L


def bf16_bits_np(t: torch.Tensor):
    """Host numpy uint16 view of a bf16 tensor."""
    return t.detach().to("cpu").contiguous().view(torch.int16).numpy().view("uint16")


def algorithmic_bytes(wl: Workload, ids: torch.Tensor) -> int:
    """Bytes the layer must move at minimum: each touched expert's three
    matrices (codes + scales) once, x read once, out written once."""
    L = layout(wl.wfmt, wl.E, wl.H, wl.I)
    touched = int(torch.unique(ids[(ids >= 0) & (ids < wl.E)]).numel())
    per_expert = 0
    for m in (GATE, UP, DOWN):
        N, K = L.dims(m)
        per_expert += code_bytes(wl.wfmt, N, K) + scale_bytes(wl.wfmt, N, K) + (4 if wl.wfmt == FMT_NVFP4_G16 else 0)
    return touched * per_expert + 2 * wl.T * wl.H * 2


def flops(wl: Workload, ids: torch.Tensor) -> int:
    """2 * 3 * H * I per valid assignment."""
    valid = int(((ids >= 0) & (ids < wl.E)).sum())
    return 2 * 3 * wl.H * wl.I * valid


# ---------------------------------------------------------------------------
# the block-attention prefill workload (the second workload)
# ---------------------------------------------------------------------------


@dataclass
class AttnWorkload:
    name: str
    B: int       # sequences
    T: int       # prompt tokens per sequence
    Hq: int      # query heads
    Hkv: int     # key/value heads (grouped queries: Hq / Hkv per kv head)
    d: int       # head dimension
    blk: int     # block size of the block-causal mask
    seed: int


ATTN_WORKLOADS = {
    "attn_small": AttnWorkload("attn_small", 2, 300, 4, 2, 128, 32, 11),
    "attn_prefill_8k": AttnWorkload("attn_prefill_8k", 1, 8192, 16, 4, 128, 32, 12),
}


def attention_inputs(B: int, T: int, Hq: int, Hkv: int, d: int, seed: int, device="cpu"):
    """q [B,T,Hq,d], k and v [B,T,Hkv,d] bf16, each element ~N(0,1)."""
    q = normal_f64(seed, 500, B * T * Hq * d, device).to(torch.float32).to(torch.bfloat16).reshape(B, T, Hq, d)
    k = normal_f64(seed, 501, B * T * Hkv * d, device).to(torch.float32).to(torch.bfloat16).reshape(B, T, Hkv, d)
    v = normal_f64(seed, 502, B * T * Hkv * d, device).to(torch.float32).to(torch.bfloat16).reshape(B, T, Hkv, d)
    return q, k, v
