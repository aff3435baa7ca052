"""Pins of the oracle's block attention (the second workload) against facts
that hold whatever the implementation: the single-key and equal-score cases,
the two-key logistic closed form, invariance under permuting the allowed
keys, the mask's reach, grouped query heads as replicated kv heads, causal
masking as full attention on the prefix, the hard-attention limit and
convexity.  Model: minnow README, "Quantization" (Block FlashAttention for
long-prompt prefill)."""
import math

import numpy as np
import pytest
import torch

import oracle as O
import synth as S


def _bf16(a):
    return torch.tensor(np.asarray(a, np.float32)).to(torch.bfloat16).view(torch.uint16).numpy()


def _f(bits):
    return torch.tensor(bits.view(np.int16)).view(torch.bfloat16).float().numpy().astype(np.float64)


def _inputs(B, T, Hq, Hkv, d, seed):
    q, k, v = S.attention_inputs(B, T, Hq, Hkv, d, seed)
    u = lambda t: t.view(torch.uint16).numpy()
    return u(q), u(k), u(v)


def test_first_causal_token_returns_its_own_value():
    q, k, v = _inputs(1, 6, 4, 2, 16, 1)
    out = O.attention(q, k, v, blk=1, scale=0.25)
    for h in range(4):
        assert np.array_equal(out[0, 0, h], _f(v[0, 0, h // 2]))


def test_equal_scores_average_the_allowed_values():
    B, T, Hq, Hkv, d, blk = 1, 70, 2, 1, 8, 32
    _, k, v = _inputs(B, T, Hq, Hkv, d, 2)
    q = np.zeros((B, T, Hq, d), np.uint16)  # every score is 0
    out = O.attention(q, k, v, blk=blk, scale=1.0)
    vf = _f(v)
    for t in (0, 31, 32, 40, 63, 64, 69):
        kmax = min(T, (t // blk + 1) * blk)
        want = vf[0, :kmax, 0].mean(axis=0)
        np.testing.assert_allclose(out[0, t, 0], want, rtol=1e-12, atol=1e-14)
        np.testing.assert_allclose(out[0, t, 1], want, rtol=1e-12, atol=1e-14)


def test_two_keys_follow_the_logistic_function():
    # one query direction, two keys a*e0 and b*e0: weights 1 - sig, sig with sig = 1 / (1 + exp(-(s1 - s0)))
    d, scale = 4, 0.7
    qv = np.zeros((1, 2, 1, d)); qv[..., 0] = 1.5
    kv = np.zeros((1, 2, 1, d)); kv[0, 0, 0, 0] = -0.75; kv[0, 1, 0, 0] = 2.25
    vv = np.array([[[[1.0, -2.0, 0.5, 3.0]], [[-1.0, 4.0, 0.25, -3.0]]]])
    out = O.attention(_bf16(qv), _bf16(kv), _bf16(vv), blk=2, scale=scale)
    s0, s1 = scale * 1.5 * -0.75, scale * 1.5 * 2.25
    sig = 1.0 / (1.0 + math.exp(-(s1 - s0)))
    want = vv[0, 0, 0] * (1 - sig) + vv[0, 1, 0] * sig
    for t in range(2):
        np.testing.assert_allclose(out[0, t, 0], want, rtol=1e-13, atol=1e-13)


def test_bidirectional_output_does_not_depend_on_key_order():
    B, T, Hq, Hkv, d = 1, 40, 2, 2, 16
    q, k, v = _inputs(B, T, Hq, Hkv, d, 3)
    perm = np.random.default_rng(0).permutation(T)
    a = O.attention(q, k, v, blk=T, scale=0.3)
    b = O.attention(q, k[:, perm], v[:, perm], blk=T, scale=0.3)
    np.testing.assert_allclose(a, b, rtol=1e-12, atol=1e-13)
    # a key paired with another key's value changes the result
    v2 = v.copy(); v2[:, [0, 1]] = v2[:, [1, 0]]
    assert not np.allclose(O.attention(q, k, v2, blk=T, scale=0.3), a)


def test_the_mask_reaches_exactly_the_earlier_and_own_blocks():
    B, T, Hq, Hkv, d, blk = 1, 96, 1, 1, 8, 32
    q, k, v = _inputs(B, T, Hq, Hkv, d, 4)
    base = O.attention(q, k, v, blk=blk, scale=0.5)
    t = 40  # block 1: keys 0..63 allowed
    k2, v2 = k.copy(), v.copy()
    k2[0, 64:] = _bf16(np.full((32, 1, d), 3.0)); v2[0, 64:] = _bf16(np.full((32, 1, d), 100.0))
    out = O.attention(q, k2, v2, blk=blk, scale=0.5)
    assert np.array_equal(out[0, :64], base[0, :64])  # blocks 0 and 1 never see block 2
    assert not np.allclose(out[0, 64:], base[0, 64:])
    v3 = v.copy(); v3[0, 63] = _bf16(np.full((1, d), 100.0))  # the last key of t's own block
    assert not np.allclose(O.attention(q, k, v3, blk=blk, scale=0.5)[0, t], base[0, t])
    assert np.array_equal(O.attention(q, k, v3, blk=blk, scale=0.5)[0, :32], base[0, :32])


def test_grouped_query_heads_equal_replicated_kv_heads():
    B, T, Hq, Hkv, d = 2, 20, 4, 2, 8
    q, k, v = _inputs(B, T, Hq, Hkv, d, 5)
    a = O.attention(q, k, v, blk=4, scale=0.4)
    rep = [0, 0, 1, 1]
    b = O.attention(q, k[:, :, rep], v[:, :, rep], blk=4, scale=0.4)
    assert np.array_equal(a, b)


def test_causal_token_is_full_attention_on_its_prefix():
    B, T, Hq, Hkv, d = 1, 24, 2, 1, 8
    q, k, v = _inputs(B, T, Hq, Hkv, d, 6)
    causal = O.attention(q, k, v, blk=1, scale=0.6)
    for t in (3, 11, 23):
        pre = O.attention(q[:, :t + 1], k[:, :t + 1], v[:, :t + 1], blk=t + 1, scale=0.6)
        np.testing.assert_allclose(causal[0, t], pre[0, t], rtol=1e-13, atol=1e-14)


def test_large_scale_tends_to_the_argmax_value():
    B, T, Hq, Hkv, d = 1, 12, 1, 1, 8
    q, k, v = _inputs(B, T, Hq, Hkv, d, 7)
    qf, kf, vf = _f(q), _f(k), _f(v)
    s = np.einsum("c,jc->j", qf[0, T - 1, 0], kf[0, :, 0])
    order = np.argsort(s)
    gap = s[order[-1]] - s[order[-2]]
    assert gap > 0.05
    scale = 400.0 / gap
    out = O.attention(q, k, v, blk=T, scale=scale)
    bound = (T - 1) * math.exp(-scale * gap) * 2 * np.abs(vf).max()
    np.testing.assert_allclose(out[0, T - 1, 0], vf[0, order[-1], 0], atol=max(bound, 1e-15))


def test_outputs_are_convex_combinations_of_allowed_values():
    B, T, Hq, Hkv, d, blk = 1, 64, 2, 2, 16, 16
    q, k, v = _inputs(B, T, Hq, Hkv, d, 8)
    out = O.attention(q, k, v, blk=blk, scale=0.9)
    vf = _f(v)
    for t in range(T):
        kmax = (t // blk + 1) * blk
        for h in range(Hq):
            lo = vf[0, :kmax, h].min(axis=0)
            hi = vf[0, :kmax, h].max(axis=0)
            assert np.all(out[0, t, h] >= lo - 1e-12) and np.all(out[0, t, h] <= hi + 1e-12)


def test_selected_rows_match_the_full_output():
    B, T, Hq, Hkv, d = 2, 33, 2, 1, 8
    q, k, v = _inputs(B, T, Hq, Hkv, d, 9)
    full = O.attention(q, k, v, blk=8, scale=0.5)
    rows = np.array([0, 7, 32, 33, 65], np.int32)
    part = O.attention(q, k, v, blk=8, scale=0.5, rows=rows)
    for i, r in enumerate(rows):
        assert np.array_equal(part[i], full[r // T, r % T])


def test_bad_arguments_are_rejected():
    q, k, v = _inputs(1, 4, 3, 2, 8, 10)  # 3 query heads over 2 kv heads
    with pytest.raises(ValueError):
        O.attention(q, k, v, blk=1, scale=1.0)
