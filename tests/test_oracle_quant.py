"""Oracle pins for the dynamic activation quantisers (INT8 per 128, NVFP4)."""
import numpy as np
import torch

import oracle as O


def _bf16_bits(v):
    return torch.tensor(np.asarray(v, np.float64)).to(torch.float32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _bf16_vals(bits):
    return torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).to(torch.float64).numpy()


def test_int8_roundtrip_bound_and_extremes():
    rng = np.random.default_rng(0)
    x = rng.standard_normal((37, 512)) * np.exp(rng.uniform(-3, 3, (37, 1)))
    x[3, 128:256] = 0.0  # an all-zero group
    xb = _bf16_bits(x)
    q, s = O.quant_int8_g128(xb)
    xv = _bf16_vals(xb)
    for r in range(37):
        for g in range(4):
            grp = xv[r, g * 128:(g + 1) * 128]
            qq = q[r, g * 128:(g + 1) * 128].astype(np.int64)
            sc = float(s[r, g])
            if not np.any(grp):
                assert sc == 0.0 and not np.any(qq)
                continue
            assert np.max(np.abs(qq)) == 127           # the absmax element maps to +-127
            # half a step, plus the rounding of the binary32 quotient x / scale
            assert np.all(np.abs(grp - qq * sc) <= sc / 2 + np.abs(grp) * 2.0 ** -23)
            assert abs(sc * 127 - np.max(np.abs(grp))) <= np.max(np.abs(grp)) * 2 ** -23
            assert np.all(np.sign(qq) * np.sign(grp) >= 0)


def test_int8_exact_multiples_roundtrip():
    # scale 2^-4 exactly: amax = 127 * 2^-4; every value m * 2^-4 must give code m
    m = np.arange(-127, 128)
    m = np.concatenate([m, m[:1]])[:256].reshape(2, 128)
    m[:, 0] = 127
    xb = _bf16_bits(m * 2.0 ** -4)
    q, s = O.quant_int8_g128(xb)
    assert np.all(s == 2.0 ** -4)
    assert np.array_equal(q.astype(np.int64), m)


def _grid_row(rng, o_exp, K):
    """A row whose values lie on the NVFP4 grid for outer = 2^o_exp."""
    outer = 2.0 ** o_exp
    e2 = np.array([0.0, 0.5, 1, 1.5, 2, 3, 4, 6])
    sbs = [448.0, 1.0, 0.5, 2.0, 0.25]
    vals = np.zeros(K)
    for b in range(K // 16):
        sb = sbs[b % 5] if b else 448.0   # block 0 carries the row amax 2688 * outer
        mag = rng.choice(e2, 16)
        mag[rng.integers(16)] = 6.0      # block amax = 6 * sb * outer
        vals[b * 16:(b + 1) * 16] = mag * rng.choice([-1, 1], 16) * sb * outer
    return vals


def test_nvfp4_grid_values_roundtrip_exactly():
    rng = np.random.default_rng(2)
    K = 256
    x = np.stack([_grid_row(rng, e, K) for e in (-10, -4, 0)])
    xb = _bf16_bits(x)
    assert np.array_equal(_bf16_vals(xb), x)   # grid values are bf16-exact
    codes, sf, outer = O.quant_nvfp4_g16(xb)
    for r in range(3):
        for kk in range(K):
            c = (codes[r, kk // 2] >> (4 * (kk & 1))) & 0xF
            v = O.e2m1_to_double(int(c)) * O.e4m3_to_double(int(sf[r, kk // 16])) * float(outer[r])
            if x[r, kk] == 0:
                assert v == 0
            else:
                assert v == x[r, kk], (r, kk)


def test_nvfp4_error_bound_and_zero_row():
    rng = np.random.default_rng(3)
    x = rng.standard_normal((9, 512)) * 3
    x[4] = 0.0
    xb = _bf16_bits(x)
    xv = _bf16_vals(xb)
    codes, sf, outer = O.quant_nvfp4_g16(xb)
    assert outer[4] == 0 and not codes[4].any() and not sf[4].any()
    for r in (0, 1, 8):
        assert outer[r] == np.float32(np.float32(np.max(np.abs(xv[r]))) / np.float32(2688.0))
        for b in range(512 // 16):
            d = float(np.float32(O.e4m3_to_double(int(sf[r, b])) * np.float32(outer[r])))
            blk = xv[r, b * 16:(b + 1) * 16]
            for i in range(16):
                kk = b * 16 + i
                c = int((codes[r, kk // 2] >> (4 * (kk & 1))) & 0xF)
                v = O.e2m1_to_double(c) * d
                t = abs(blk[i]) / d
                # half the E2M1 grid spacing around t, unless saturated at 6
                half = 0.25 if t < 2 else 0.5 if t < 4 else 1.0
                if t <= 6:
                    assert abs(abs(v) - abs(blk[i])) <= half * d * (1 + 1e-6), (r, kk)
                else:
                    assert abs(v) == 6 * d
