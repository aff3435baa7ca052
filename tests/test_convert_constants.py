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
