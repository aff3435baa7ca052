"""Oracle pins for the expert GEMMs, the combine and the whole layer.

The cross-checks decode each weight format with library routines and lookup
tables built from the formats' stated value sets (numpy float16, torch
float8_e4m3fn / bfloat16, the E2M1 value list), expand whole expert matrices
and use dense float64 matmuls: a different route from the oracle's
element-by-element decode.
"""
import math
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle as O
import synth as S

E2M1 = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0, -0.0, -0.5, -1.0, -1.5, -2.0, -3.0, -4.0, -6.0])
INT4 = np.array([0, 1, 2, 3, 4, 5, 6, 7, -8, -7, -6, -5, -4, -3, -2, -1], np.float64)
E4M3 = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()


def bf16_vals(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16).copy()).view(torch.bfloat16).to(torch.float64).numpy()


def bf16_round(v):
    return torch.from_numpy(np.asarray(v, np.float64)).to(torch.float32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def dense_weights(blob, L, e, m):
    """Expand matrix m of expert e to float64 [N, K] with library decoders."""
    b = blob.numpy() if isinstance(blob, torch.Tensor) else blob
    N, K = L.dims(m)
    base = L.data_offset + e * L.expert_stride
    c0 = base + L.codes_off[m]
    if L.wfmt == S.FMT_BF16:
        return bf16_vals(b[c0:c0 + N * K * 2].view(np.uint16)).reshape(N, K)
    s0 = base + L.scales_off[m]
    if L.wfmt in (S.FMT_INT8_G128, S.FMT_INT4_G128):
        sc = b[s0:s0 + N * (K // 128) * 2].view(np.float16).astype(np.float64).reshape(N, K // 128)
        if L.wfmt == S.FMT_INT8_G128:
            q = b[c0:c0 + N * K].view(np.int8).astype(np.float64).reshape(N, K)
        else:
            by = b[c0:c0 + N * K // 2].reshape(N, K // 2)
            q = np.empty((N, K))
            q[:, 0::2] = INT4[by & 0xF]
            q[:, 1::2] = INT4[by >> 4]
        return q * np.repeat(sc, 128, axis=1)
    by = b[c0:c0 + N * K // 2].reshape(N, K // 2)
    v = np.empty((N, K))
    v[:, 0::2] = E2M1[by & 0xF]
    v[:, 1::2] = E2M1[by >> 4]
    sf = E4M3[b[s0:s0 + N * (K // 16)]].reshape(N, K // 16)
    outer = float(b[base + L.outer_off[m]: base + L.outer_off[m] + 4].view(np.float32)[0])
    return v * np.repeat(sf, 16, axis=1) * outer


def silu(g):
    return g / (1.0 + np.exp(-g))


def ffn_dense(blob, L, e, xrow):
    g = dense_weights(blob, L, e, S.GATE) @ xrow
    u = dense_weights(blob, L, e, S.UP) @ xrow
    h = bf16_vals(bf16_round(silu(g) * u))
    return bf16_vals(bf16_round(dense_weights(blob, L, e, S.DOWN) @ h))


def close_bf16(a_bits, b_vals, ulps=2):
    """a (bf16 bits) equals b (float64, before the final BF16 rounding) up to
    that rounding: within `ulps` BF16 ulps almost everywhere, relative L2
    error below 3e-3 (one BF16 rounding is at most 2^-9 relative)."""
    a = bf16_vals(a_bits)
    tol = np.abs(b_vals) * 2.0 ** -8 * ulps + 1e-30
    bad = np.abs(a - b_vals) > tol
    return bad.mean() <= 1e-2 and np.linalg.norm(a - b_vals) <= 3e-3 * (np.linalg.norm(b_vals) + 1e-30)


@pytest.mark.parametrize("wfmt", [S.FMT_BF16, S.FMT_INT8_G128, S.FMT_INT4_G128])
def test_a16_forward_matches_dense_expansion(wfmt):
    E, H, I, T, k = 4, 256, 128, 6, 2
    blob, hdr, L = S.expert_blob(wfmt, E, H, I, seed=11)
    x = S.activations(T, H, 12)
    ids = S.routing_uniform(T, E, k, 13)
    w = S.routing_weights(T, k, 14)
    xb = S.bf16_bits_np(x)
    out = O.moe_forward(blob.numpy(), S.ACT_BF16, xb, ids.numpy(), w.numpy())
    xv = bf16_vals(xb)
    for t in range(T):
        acc = np.zeros(H)
        for j in range(k):
            acc += float(w[t, j]) * ffn_dense(blob, L, int(ids[t, j]), xv[t])
        assert close_bf16(out[t], acc)


def test_gemm_a16_gate_up_and_down_rows():
    E, H, I = 3, 256, 256
    blob, hdr, L = S.expert_blob(S.FMT_INT4_G128, E, H, I, seed=21)
    offsets = np.array([0, 2, 2, 5], np.int32)
    a = S.bf16_bits_np(S.activations(5, H, 22))
    h = O.gemm_a16(blob.numpy(), O.KIND_GATE_UP, a, offsets)
    av = bf16_vals(a)
    for p, e in enumerate([0, 0, 2, 2, 2]):
        g = dense_weights(blob, L, e, S.GATE) @ av[p]
        u = dense_weights(blob, L, e, S.UP) @ av[p]
        assert close_bf16(h[p], silu(g) * u)
    y = O.gemm_a16(blob.numpy(), O.KIND_DOWN, h, offsets)
    hv = bf16_vals(h)
    for p, e in enumerate([0, 0, 2, 2, 2]):
        assert close_bf16(y[p], dense_weights(blob, L, e, S.DOWN) @ hv[p])


@pytest.mark.parametrize("wfmt", [S.FMT_INT8_G128, S.FMT_INT4_G128])
def test_a8_group_dots_brute_force(wfmt):
    E, H, I = 2, 256, 128
    blob, hdr, L = S.expert_blob(wfmt, E, H, I, seed=31)
    x = S.bf16_bits_np(S.activations(3, H, 32, outlier_p=0.05))
    q, s = O.quant_int8_g128(x)
    offsets = np.array([0, 1, 3], np.int32)
    h, dots = O.gemm_a8(blob.numpy(), O.KIND_GATE_UP, q, s, offsets, want_dots=True)
    b = blob.numpy()
    for p, e in enumerate([0, 1, 1]):
        for m in (S.GATE, S.UP):
            base = L.data_offset + e * L.expert_stride
            N, K = L.dims(m)
            c0 = base + L.codes_off[m]
            if wfmt == S.FMT_INT8_G128:
                qw = b[c0:c0 + N * K].view(np.int8).astype(np.int64).reshape(N, K)
            else:
                by = b[c0:c0 + N * K // 2].reshape(N, K // 2)
                qw = np.empty((N, K), np.int64)
                qw[:, 0::2] = INT4[by & 0xF]
                qw[:, 1::2] = INT4[by >> 4]
            for n in range(0, N, 17):
                for g in range(K // 128):
                    want = sum(int(q[p, kk]) * int(qw[n, kk]) for kk in range(g * 128, g * 128 + 128))
                    assert dots[p, m * N + n, g] == want
        # the scaled FP combination of the groups
        g_ = np.zeros(I)
        u_ = np.zeros(I)
        sw_g = dense_weights(blob, L, e, S.GATE)  # q * s, so q*s_w summed per group with s_a
        sw_u = dense_weights(blob, L, e, S.UP)
        qa = q[p].astype(np.float64) * np.repeat(s[p].astype(np.float64), 128)
        g_ = sw_g @ qa
        u_ = sw_u @ qa
        assert close_bf16(h[p], silu(g_) * u_)


def test_a4_forward_matches_dense_expansion():
    E, H, I, T, k = 3, 256, 256, 4, 2
    blob, hdr, L = S.expert_blob(S.FMT_NVFP4_G16, E, H, I, seed=41)
    x = S.bf16_bits_np(S.activations(T, H, 42))
    ids = S.routing_uniform(T, E, k, 43).numpy()
    w = S.routing_weights(T, k, 44).numpy()
    out = O.moe_forward(blob.numpy(), S.ACT_NVFP4_G16, x, ids, w)

    def deq(codes, sf, outer):
        K = codes.shape[-1] * 2
        v = np.empty(K)
        v[0::2] = E2M1[codes & 0xF]
        v[1::2] = E2M1[codes >> 4]
        return v * np.repeat(E4M3[sf], 16) * float(outer)

    for t in range(T):
        acc = np.zeros(H)
        c, sf, o = O.quant_nvfp4_g16(x[t:t + 1])
        xa = deq(c[0], sf[0], o[0])
        for j in range(k):
            e = int(ids[t, j])
            g = dense_weights(blob, L, e, S.GATE) @ xa
            u = dense_weights(blob, L, e, S.UP) @ xa
            hb = bf16_round(silu(g) * u)
            c2, sf2, o2 = O.quant_nvfp4_g16(hb[None, :])
            y = bf16_vals(bf16_round(dense_weights(blob, L, e, S.DOWN) @ deq(c2[0], sf2[0], o2[0])))
            acc += float(w[t, j]) * y
        assert close_bf16(out[t], acc)


def test_identity_experts_closed_form():
    """BF16 experts with gate = a*Id, up = Id, down = Id: the FFN reduces to
    h_i = bf16(SiLU(a x_i) x_i) and y = h."""
    H = I = 128
    L = S.layout(S.FMT_BF16, 1, H, I)
    body = np.zeros(L.expert_stride, np.uint8)
    a = 0.5
    for m, scale in ((S.GATE, a), (S.UP, 1.0), (S.DOWN, 1.0)):
        eye = bf16_round(np.eye(H) * scale)
        body[L.codes_off[m]:L.codes_off[m] + H * H * 2] = eye.view(np.uint8).reshape(-1)
    blob = np.concatenate([np.frombuffer(S.header_bytes(L), np.uint8), body])
    x = S.bf16_bits_np(S.activations(3, H, 51))
    out = O.moe_forward(blob, S.ACT_BF16, x, np.zeros((3, 1), np.int32), np.ones((3, 1), np.float32))
    xv = bf16_vals(x)
    for t in range(3):
        for i in range(H):
            want = a * xv[t, i] / (1 + math.exp(-a * xv[t, i])) * xv[t, i]
            got = bf16_vals(out[t, i:i + 1])[0]
            assert abs(got - want) <= abs(want) * 2.0 ** -8 + 1e-45


def test_layer_invariants():
    E, H, I, T, k = 4, 256, 128, 8, 3
    blob, hdr, L = S.expert_blob(S.FMT_INT4_G128, E, H, I, seed=61)
    x = S.bf16_bits_np(S.activations(T, H, 62))
    ids = S.routing_uniform(T, E, k, 63).numpy()
    w = S.routing_weights(T, k, 64).numpy()
    b = blob.numpy()
    out = O.moe_forward(b, S.ACT_BF16, x, ids, w)
    # token order: permuting tokens permutes outputs exactly
    perm = np.random.default_rng(0).permutation(T)
    assert np.array_equal(O.moe_forward(b, S.ACT_BF16, x[perm], ids[perm], w[perm]), out[perm])
    # a subset of rows equals the same rows of the full run
    rows = np.array([5, 1, 6], np.int32)
    assert np.array_equal(O.moe_forward(b, S.ACT_BF16, x, ids, w, rows=rows), out[rows])
    # zero input -> zero output
    z = O.moe_forward(b, S.ACT_BF16, np.zeros_like(x), ids, w)
    assert not np.any(bf16_vals(z))
    # slot order does not matter beyond rounding; doubling w doubles out exactly
    assert np.array_equal(bf16_vals(O.moe_forward(b, S.ACT_BF16, x, ids, 2 * w)), 2 * bf16_vals(out))
    # out-of-range ids are dropped: same as routing weight 0 for that slot
    ids2 = ids.copy(); ids2[:, 1] = E + 3
    w2 = w.copy(); w2[:, 1] = 0.0
    assert np.array_equal(O.moe_forward(b, S.ACT_BF16, x, ids2, w), O.moe_forward(b, S.ACT_BF16, x, ids, w2))


def test_identical_experts_scale_by_weight_sum():
    E, H, I, T, k = 3, 128, 128, 4, 3
    one, hdr, L1 = S.expert_blob(S.FMT_INT8_G128, 1, H, I, seed=71)
    L = S.layout(S.FMT_INT8_G128, E, H, I)
    body = np.tile(one.numpy()[256:], E)
    blob = np.concatenate([np.frombuffer(S.header_bytes(L), np.uint8), body])
    x = S.bf16_bits_np(S.activations(T, H, 72))
    ids = np.tile(np.arange(E, dtype=np.int32), (T, 1))
    w = S.routing_weights(T, k, 73).numpy()
    out = O.moe_forward(blob, S.ACT_BF16, x, ids, w)
    y = O.moe_forward(blob, S.ACT_BF16, x, ids[:, :1], np.ones((T, 1), np.float32))
    for t in range(T):
        s = sum(float(v) for v in w[t])
        assert np.array_equal(out[t], bf16_round(s * bf16_vals(y[t])))


def test_combine_exact_rational():
    rng = np.random.default_rng(5)
    T, k, H = 3, 4, 8
    y = bf16_round(rng.integers(-64, 64, (T * k, H)) / 16.0)
    w = np.array([[0.5, 0.25, 0.125, 0.125]] * T, np.float32)
    pos = np.arange(T * k, dtype=np.int32)
    pos[5] = -1
    out = O.combine(y, pos, w, T, k)
    yv = bf16_vals(y)
    for t in range(T):
        for c in range(H):
            s = sum(Fraction(float(w[t, j])) * Fraction(float(yv[t * k + j, c]))
                    for j in range(k) if pos[t * k + j] >= 0)
            assert Fraction(float(bf16_vals(out[t, c:c + 1])[0])) == s  # exact: few bits
