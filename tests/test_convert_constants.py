"""Host check of the INT4 -> FP16 operand conversion of the warp-MMA kernel's
FP16-row form (int4_j4): the constants are read from the kernel source and
the same bit operations and FP16 arithmetic are replayed exactly in numpy.
Every nibble value in every position of a code word must come out as its
signed integer, in the K slot that the {j, j+4} pairing assigns it."""
import os
import re

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "quantized_moe_expert_routed_gb300", "csrc", "mnw_gemm_warp.cuh")


def _constants():
    body = open(SRC).read()
    body = body[body.index("void int4_j4("):]
    body = body[:body.index("}")]
    lo = re.search(r"lo = f16x2_sub\(and_xor\(v, (0x[0-9A-Fa-f]+)u, (0x[0-9A-Fa-f]+)u\), (0x[0-9A-Fa-f]+)u\)", body)
    hi = re.search(r"hi = f16x2_fma\(and_xor\(v, (0x[0-9A-Fa-f]+)u, (0x[0-9A-Fa-f]+)u\), (0x[0-9A-Fa-f]+)u, "
                   r"(0x[0-9A-Fa-f]+)u\)", body)
    shift = re.search(r"kOdd \? w >> (\d+) : w", body)
    assert lo and hi and shift, "int4_j4 changed shape; update this test"
    return ([int(g, 16) for g in lo.groups()], [int(g, 16) for g in hi.groups()], int(shift.group(1)))


def _halves(x):
    """uint32 -> the two FP16 values (low half, high half)."""
    x = np.asarray(x, np.uint32)
    return (x & 0xFFFF).astype(np.uint16).view(np.float16), (x >> 16).astype(np.uint16).view(np.float16)


def _j4(w, odd, consts):
    (m_lo, c_lo, s_lo), (m_hi, c_hi, mul, add), sh = consts
    v = (w >> sh) if odd else w
    a_lo = (v & m_lo) ^ c_lo
    a_hi = (v & m_hi) ^ c_hi
    lo = [x - y for x, y in zip(_halves(a_lo), _halves(s_lo))]              # one FP16 subtraction each
    hi = [np.float16(np.float32(x) * np.float32(m) + np.float32(b))       # fma: exact product, one rounding
          for x, m, b in zip(_halves(a_hi), _halves(mul), _halves(add))]
    return lo, hi


def test_every_nibble_in_every_position_decodes_exactly():
    consts = _constants()
    rng = np.random.default_rng(0)
    for pos in range(8):
        for n in range(16):
            w = rng.integers(0, 2 ** 32, 64, dtype=np.uint64).astype(np.uint32)
            w = (w & ~np.uint32(0xF << (4 * pos))) | np.uint32(n << (4 * pos))
            want = n - 16 if n >= 8 else n
            # slots: even k-step -> lo = K {0,4}, hi = K {1,5}; odd -> lo = K {2,6}, hi = K {3,7}
            j = pos % 4
            lo, hi = _j4(w, j >= 2, consts)
            out = (lo if j % 2 == 0 else hi)[1 if pos >= 4 else 0]
            assert np.all(out.astype(np.float64) == want), (pos, n)


CONVERT = os.path.join(ROOT, "quantized_moe_expert_routed_gb300", "csrc", "mnw_convert.cuh")
ROUTE = os.path.join(ROOT, "quantized_moe_expert_routed_gb300", "csrc", "mnw_route.cu")


def _prmt(a, b, sel):
    """PTX prmt.b32 (default mode): result byte i is byte (sel >> 4i) & 7 of {b:a}."""
    a = np.asarray(a, np.uint64)
    b = np.asarray(b, np.uint64)
    src = a | (b << np.uint64(32))
    out = np.zeros_like(a)
    for i in range(4):
        k = (sel >> (4 * i)) & 7
        out |= ((src >> np.uint64(8 * k)) & np.uint64(0xFF)) << np.uint64(8 * i)
    return out.astype(np.uint32)


def test_natural_pair_int4_and_int8_to_fp16():
    conv = open(CONVERT).read()
    for expr in ("prmt(w[i], hi, 0x0400u + 0x0101u * b)",
                 "f16x2_sub(and_xor(x, 0x000F000Fu, 0x64086408u), 0x64086408u)",
                 "f16x2_sub(prmt(u, 0x64646464u, 0x4140u), 0x64806480u)",
                 "f16x2_sub(prmt(u, 0x64646464u, 0x4342u), 0x64806480u)",
                 "const uint32_t u = w[i] ^ 0x80808080u;"):
        assert expr in conv, expr   # the replay below follows these lines
    rng = np.random.default_rng(1)
    w = rng.integers(0, 2 ** 32, 4096, dtype=np.uint64).astype(np.uint32)
    nib = np.stack([(w >> (4 * i)) & 0xF for i in range(8)]).astype(np.int64)
    q4 = np.where(nib >= 8, nib - 16, nib)                      # element e = nibble e, signed
    hi = w >> 4
    for b in range(4):                                           # INT4: byte b -> elements 2b, 2b+1
        x = _prmt(w, hi, 0x0400 + 0x0101 * b)
        a = (x & 0x000F000F) ^ 0x64086408
        lo, hh = _halves(a)
        c0, c1 = _halves(np.uint32(0x64086408))
        assert np.array_equal((lo - c0).astype(np.int64), q4[2 * b])
        assert np.array_equal((hh - c1).astype(np.int64), q4[2 * b + 1])
    u = w ^ np.uint32(0x80808080)                                # INT8: bytes 0..3 -> elements 0..3
    q8 = np.stack([((w >> (8 * i)) & 0xFF).astype(np.int64) for i in range(4)])
    q8 = np.where(q8 >= 128, q8 - 256, q8)
    for sel, e0 in ((0x4140, 0), (0x4342, 2)):
        lo, hh = _halves(_prmt(u, np.full_like(u, 0x64646464), sel))
        c0, c1 = _halves(np.uint32(0x64806480))
        assert np.array_equal((lo - c0).astype(np.int64), q8[e0])
        assert np.array_equal((hh - c1).astype(np.int64), q8[e0 + 1])


def test_fp16_row_exponent_rule_matches_the_oracle():
    """The gather kernel derives the row exponent from the largest BF16 bit
    pattern: e = clamp((bits >> 7) - 141, -110, 113).  Replayed on the host it
    must give the oracle's encoding bit for bit."""
    import torch
    import oracle as O
    assert "const int e = min(113, max(-110, static_cast<int>(m >> 7) - 141));" in open(ROUTE).read()
    rng = np.random.default_rng(2)
    x = rng.standard_normal((64, 256)) * np.exp2(rng.integers(-90, 90, (64, 1)).astype(np.float64))
    x[3] = 0.0
    xb = torch.tensor(x, dtype=torch.float32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    codes, factor = O.encode_f16_rows(xb)
    for r in range(64):
        m = int((xb[r] & 0x7FFF).max())
        e = min(113, max(-110, (m >> 7) - 141))
        vals = (xb[r].astype(np.uint32) << 16).view(np.float32)
        got = (vals * np.float32(2.0 ** -e)).astype(np.float16).view(np.uint16)  # exact scaling, one rounding
        assert factor[r] == np.float32(2.0 ** e)
        assert np.array_equal(got, codes[r]), r
