"""Oracle pins for the FP16 row encoding (FP16 codes, power-of-two row
factor) and the grouped GEMM that reads it.

The encoding is the CUDA path's operand form for INT8/INT4-weight gate/up
GEMMs with BF16 activations on FP16 tensor cores: an exact re-encoding of a
BF16 row, so the GEMM over it must equal the BF16-activation GEMM."""
import numpy as np
import pytest
import torch

import oracle as O
import synth as S


def _bf16_bits(v):
    return torch.tensor(np.asarray(v, np.float64)).to(torch.float32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _bf16_vals(bits):
    return torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).to(torch.float64).numpy()


def _f16_vals(bits):
    return bits.view(np.float16).astype(np.float64)


def test_fp16_encoder_matches_numpy_rounding():
    # numpy's double -> half conversion rounds to nearest even: an independent
    # implementation of the same IEEE rounding, across normal, subnormal,
    # overflowing and exactly-halfway inputs.
    rng = np.random.default_rng(5)
    v = rng.standard_normal(4000) * np.exp2(rng.integers(-30, 18, 4000))
    ties = 1.0 + (np.arange(0, 1023) + 0.5) * 2.0 ** -10  # halfway between neighbouring FP16 values in [1, 2)
    v = np.concatenate([v, ties, -ties, [0.0, -0.0, 65504.0, 65519.9, 65520.0, 1e6, 2.0 ** -24, 2.0 ** -25,
                                         3 * 2.0 ** -26, 2.0 ** -14 * (1 - 2.0 ** -11)]])
    got = np.array([O.fp16_from_double(float(a)) for a in v], np.uint16)
    with np.errstate(over="ignore"):
        want = v.astype(np.float16).view(np.uint16)
    assert np.array_equal(got, want)


def test_hand_worked_row():
    # amax = 3 = 1.5 * 2^1 -> e = 1 - 14 = -13, factor 2^-13, codes x * 2^13:
    # 8192 = 2^13 -> 0x7000; -24576 = -1.5 * 2^14 -> 0xF600; 4096 = 2^12 -> 0x6C00; 0.
    codes, factor = O.encode_f16_rows(_bf16_bits([[1.0, -3.0, 0.5, 0.0]]))
    assert factor[0] == 2.0 ** -13
    assert codes[0].tolist() == [0x7000, 0xF600, 0x6C00, 0x0000]


def test_rows_scale_into_range_and_roundtrip_exactly():
    rng = np.random.default_rng(6)
    R, K = 40, 256
    x = rng.standard_normal((R, K)) * np.exp2(rng.integers(-60, 60, (R, 1)))
    x[5] *= 1e-30
    x[6] *= 1e30
    x[7, :] = 0.0
    x[8, :] = 0.0
    x[8, 17] = -2.0 ** -133  # the smallest BF16 subnormal
    xb = _bf16_bits(x)
    codes, factor = O.encode_f16_rows(xb)
    xv = _bf16_vals(xb)
    for r in range(R):
        amax = np.max(np.abs(xv[r]))
        e = np.log2(float(factor[r]))
        assert e == np.round(e)
        if r in (7, 8):
            assert factor[r] == 2.0 ** -110
        else:
            # the largest magnitude lands in [2^14, 2^15)
            assert 2.0 ** 14 <= amax / factor[r] < 2.0 ** 15
        keep = np.abs(xv[r]) >= amax * 2.0 ** -28
        dec = _f16_vals(codes[r]) * float(factor[r])
        assert np.array_equal(dec[keep], xv[r][keep])  # exact where FP16 stays normal
        # every code is the RNE FP16 value of x * 2^-e (numpy's rounding)
        want = (xv[r] / float(factor[r])).astype(np.float16).view(np.uint16)
        assert np.array_equal(codes[r], want)


def test_largest_bf16_does_not_overflow():
    big = float(_bf16_vals(np.array([0x7F7F], np.uint16))[0])  # largest finite BF16
    codes, factor = O.encode_f16_rows(_bf16_bits([[big, -big / 3, 1.0]]))
    assert factor[0] == 2.0 ** 113
    assert np.all(np.isfinite(_f16_vals(codes[0])))
    assert _f16_vals(codes[0])[0] * 2.0 ** 113 == big


def test_nonfinite_rows_are_rejected():
    with pytest.raises(Exception):
        O.encode_f16_rows(np.array([[0x3F80, 0x7F80]], np.uint16))  # 1.0, +Inf


@pytest.mark.parametrize("wfmt", [S.FMT_INT8_G128, S.FMT_INT4_G128])
def test_gemm_f16rows_equals_bf16_gemm_on_encoded_rows(wfmt):
    # The encoding is exact for these rows, the factor a power of two: the FP64
    # sums are the same numbers scaled, so both GEMMs give the same bits.
    wl = S.Workload("f16rows_pin", 6, 256, 4, 128, 2, wfmt, S.ACT_BF16, 0.02, "uniform", 3)
    x, ids, w, blob, hdr, L = S.make_inputs(wl)
    blob = blob.numpy()
    xb = S.bf16_bits_np(x)
    xb[1] = _bf16_bits(_bf16_vals(xb[1]) * 2.0 ** 40)
    xb[2] = _bf16_bits(_bf16_vals(xb[2]) * 2.0 ** -50)
    off, sorted_assign, pos, _ = O.permute(ids.numpy(), wl.E)
    a = xb[np.maximum(sorted_assign, 0) // wl.k]
    codes, factor = O.encode_f16_rows(a)
    for kind in (O.KIND_GATE_UP,):
        want = O.gemm_a16(blob, kind, a, off)
        got = O.gemm_f16rows(blob, kind, codes, factor, off)
        assert np.array_equal(got, want)
    # a dropped factor must show
    bad = O.gemm_f16rows(blob, O.KIND_GATE_UP, codes, np.ones_like(factor), off)
    assert not np.array_equal(bad, want)


def test_f16rows_is_not_a_layer_mode():
    wl = S.Workload("f16rows_mode", 4, 128, 4, 128, 2, S.FMT_INT8_G128, S.ACT_BF16, 0.02, "uniform", 4)
    x, ids, w, blob, hdr, L = S.make_inputs(wl)
    with pytest.raises(Exception):
        O.moe_forward(blob.numpy(), O.ACT_F16_ROWS, S.bf16_bits_np(x), ids.numpy(), w.numpy())
