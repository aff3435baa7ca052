"""Pins of the oracle's unfused-activation comparison path: the gate-only and
up-only grouped GEMMs against dense float64 expansions of the expert
matrices, and bf16(SiLU(g) * u) against its closed form."""
import math

import numpy as np
import pytest
import torch

import oracle as O
import synth as S
from test_oracle_layer import bf16_round, bf16_vals, close_bf16, dense_weights, silu


@pytest.mark.parametrize("wfmt", [S.FMT_BF16, S.FMT_INT8_G128, S.FMT_INT4_G128])
def test_single_matrix_gemms_match_dense_expansion(wfmt):
    E, H, I, T, k = 3, 256, 256, 6, 2
    blob, hdr, L = S.expert_blob(wfmt, E, H, I, seed=31 + wfmt)
    ids = S.routing_uniform(T, E, k, seed=32)
    x = S.activations(T, H, seed=33)
    off, sa, pos, _ = O.permute(ids.numpy(), E)
    xp = S.bf16_bits_np(x)[sa // k]
    b = blob.numpy()
    for kind, m in ((O.KIND_GATE, S.GATE), (O.KIND_UP, S.UP)):
        got = O.gemm_a16(b, kind, xp, off)
        assert got.shape == (T * k, I)
        for e in range(E):
            W = dense_weights(b, L, e, m)
            for p in range(off[e], off[e + 1]):
                assert close_bf16(got[p], W @ bf16_vals(xp[p]))
    # and the fused gate/up of the same rows is SiLU of the two, up to the extra roundings
    g = bf16_vals(O.gemm_a16(b, O.KIND_GATE, xp, off))
    u = bf16_vals(O.gemm_a16(b, O.KIND_UP, xp, off))
    fused = bf16_vals(O.gemm_a16(b, O.KIND_GATE_UP, xp, off))
    assert np.linalg.norm(fused - silu(g) * u) <= 1e-2 * np.linalg.norm(fused)


def test_single_matrix_gemm_a4_and_a8():
    E, H, I, T, k = 2, 256, 256, 5, 2
    blob, hdr, L = S.expert_blob(S.FMT_NVFP4_G16, E, H, I, seed=41)
    ids = S.routing_uniform(T, E, k, seed=42)
    x = S.bf16_bits_np(S.activations(T, H, seed=43))
    off, sa, pos, _ = O.permute(ids.numpy(), E)
    c, sf, o = O.quant_nvfp4_g16(x[sa // k])
    b = blob.numpy()
    g4 = O.gemm_a4(b, O.KIND_GATE, c, sf, o, off)
    # activations decoded from their codes, weights expanded densely
    from test_oracle_layer import E2M1, E4M3
    for p in range(T * k):
        e = int(np.searchsorted(off, p, side="right") - 1)
        a = np.empty(H)
        a[0::2] = E2M1[c[p] & 0xF]
        a[1::2] = E2M1[c[p] >> 4]
        a = a * np.repeat(E4M3[sf[p]], 16) * float(o[p])
        assert close_bf16(g4[p], dense_weights(b, L, e, S.GATE) @ a)
    blob8, _, L8 = S.expert_blob(S.FMT_INT8_G128, E, H, I, seed=44)
    q, s = O.quant_int8_g128(x[sa // k])
    u8, dots = O.gemm_a8(blob8.numpy(), O.KIND_UP, q, s, off, want_dots=True)
    assert dots.shape == (T * k, I, H // 128)
    for p in range(T * k):
        e = int(np.searchsorted(off, p, side="right") - 1)
        W = dense_weights(blob8.numpy(), L8, e, S.UP)
        a = q[p].astype(np.float64) * np.repeat(s[p].astype(np.float64), 128)
        assert close_bf16(u8[p], W @ a)


def test_silu_mul_closed_form():
    g = np.array([0.0, 1.0, -1.0, 20.0, -20.0, 3.5, -0.125, 1e-3], np.float64)
    u = np.array([1.0, 2.0, 3.0, 0.5, 4.0, -1.5, 8.0, 1000.0], np.float64)
    gb, ub = bf16_round(g), bf16_round(u)
    got = bf16_vals(O.silu_mul(gb, ub))
    gv, uv = bf16_vals(gb), bf16_vals(ub)
    want = [gi / (1.0 + math.exp(-gi)) * ui for gi, ui in zip(gv, uv)]
    assert np.array_equal(got, bf16_vals(bf16_round(want)))
    assert got[0] == 0.0 and got[4] == bf16_vals(bf16_round([-20.0 / (1 + math.exp(20.0)) * 4.0]))[0]
    rng = np.random.default_rng(0)
    g2 = bf16_round(rng.normal(0, 3, 4096))
    u2 = bf16_round(rng.normal(0, 1, 4096))
    ref = bf16_round(silu(bf16_vals(g2)) * bf16_vals(u2))
    assert np.array_equal(O.silu_mul(g2, u2), ref)
