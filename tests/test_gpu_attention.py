"""Block attention for prompt prefill (the second workload) on the GPU,
compared with the FP64 oracle element by element.

Tolerance, from the kernel's arithmetic: the scores and the softmax are FP32
(relative error far below 2^-9), the probabilities enter the second product
rounded to BF16 and the row sum is taken over the same rounded values, so the
output is an exact convex combination of the v rows whose weights are each
within a relative 2^-8 of the true ones; the result is rounded to BF16 (2^-9).
Hence |out - ref| <= 2^-8 * max|v| + 2^-8 * |ref| + 1e-5 per element.
Model: minnow README, "Quantization" (Block FlashAttention)."""
import numpy as np
import pytest
import torch

import oracle as O
import synth as S

pytestmark = pytest.mark.gpu


def _u16(t):
    return t.detach().cpu().contiguous().view(torch.uint16).numpy()


def _run(B, T, Hq, Hkv, blk, seed, d=128):
    import quantized_moe_expert_routed_gb300 as M
    q, k, v = S.attention_inputs(B, T, Hq, Hkv, d, seed, device="cuda")
    scale = 1.0 / np.sqrt(d)
    out = M.mnw_attn_prefill(q, k, v, blk, scale)
    torch.cuda.synchronize()
    return q, k, v, out, scale


def _check(got, ref, v_bf16_host, Hq, Hkv):
    vmax = np.abs(torch.tensor(v_bf16_host.view(np.int16)).view(torch.bfloat16).float().numpy()).max()
    tol = 2.0 ** -8 * vmax + 2.0 ** -8 * np.abs(ref) + 1e-5
    err = np.abs(got - ref)
    assert np.all(np.isfinite(got))
    bad = np.argwhere(err > tol)
    assert bad.size == 0, f"{bad.shape[0]} elements off, first {bad[:3].tolist()}, max err {err.max():.3g}"
    rel = np.linalg.norm(got - ref) / np.linalg.norm(ref)
    assert rel < 5e-3, rel


@pytest.mark.parametrize("B,T,Hq,Hkv,blk", [
    (1, 128, 1, 1, 32),     # one query tile, one key tile
    (2, 300, 4, 2, 32),     # ragged tail, grouped heads, two sequences
    (1, 257, 2, 2, 1),      # causal, one row into a third tile
    (1, 200, 2, 1, 4096),   # bidirectional
    (1, 384, 2, 2, 64),
    (1, 130, 2, 2, 7),      # blocks that do not divide the tile
    (1, 640, 2, 1, 200),    # blocks wider than a tile
    (1, 1, 2, 1, 32),       # one token
    (3, 129, 8, 1, 32),     # three sequences, 8 query heads on one kv head, one row into a second tile
    (1, 256, 2, 2, 100),    # early rows of a tile see no key of its second tile
])
def test_attention_matches_oracle(B, T, Hq, Hkv, blk):
    q, k, v, out, scale = _run(B, T, Hq, Hkv, blk, seed=100 + T + blk)
    ref = O.attention(_u16(q), _u16(k), _u16(v), blk, scale)
    got = out.float().cpu().numpy().astype(np.float64)
    _check(got, ref, _u16(v), Hq, Hkv)


def test_attention_full_size_sampled_rows():
    wl = S.ATTN_WORKLOADS["attn_prefill_8k"]
    q, k, v, out, scale = _run(wl.B, wl.T, wl.Hq, wl.Hkv, wl.blk, wl.seed, wl.d)
    rng = np.random.default_rng(5)
    rows = np.unique(np.concatenate([[0, 31, 32, 127, 128, 4095, 4096, wl.T - 1],
                                     rng.integers(0, wl.B * wl.T, 16)])).astype(np.int32)
    ref = O.attention(_u16(q), _u16(k), _u16(v), wl.blk, scale, rows=rows)
    flat = out.reshape(wl.B * wl.T, wl.Hq, wl.d)
    got = flat[torch.as_tensor(rows, device=out.device).long()].float().cpu().numpy().astype(np.float64)
    _check(got, ref, _u16(v), wl.Hq, wl.Hkv)


def test_attention_is_deterministic_and_leaves_no_error():
    import quantized_moe_expert_routed_gb300 as M
    q, k, v = S.attention_inputs(1, 520, 4, 2, 128, 9, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    a = M.mnw_attn_prefill(q, k, v, 32, 0.09, err=err)
    b = M.mnw_attn_prefill(q, k, v, 32, 0.09, err=err)
    torch.cuda.synchronize()
    assert torch.equal(a, b)
    assert int(err.item()) == 0


def test_attention_large_scores_stay_finite():
    # scores far from zero: the running maximum moves by more than 2^8 several times
    import quantized_moe_expert_routed_gb300 as M
    q, k, v = S.attention_inputs(1, 512, 2, 1, 128, 10, device="cuda")
    ramp = torch.linspace(0.1, 6.0, 512, device="cuda").view(1, 512, 1, 1)
    k = (k.float() * ramp).to(torch.bfloat16)
    out = M.mnw_attn_prefill(q, k, v, 1, 0.5)
    torch.cuda.synchronize()
    ref = O.attention(_u16(q), _u16(k), _u16(v), 1, 0.5)
    _check(out.float().cpu().numpy().astype(np.float64), ref, _u16(v), 2, 1)
