"""Pins of the oracle's router (GPU routing path of the decode blocks): the
chosen experts and their weights against a brute-force restatement in plain
Python (float64 dot products, a full sort, math.exp), the tie rule, and the
special cases k = 1 and k = E."""
import math

import numpy as np
import pytest
import torch

import oracle as O
import synth as S


def _bf16(v):
    return S.to_bf16_bits(torch.as_tensor(v, dtype=torch.float64)).numpy().view(np.uint16)


def _vals(bits):
    return torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).double().numpy()


def _brute(x_bits, wr_bits, k):
    x, wr = _vals(x_bits), _vals(wr_bits)
    ids, ws = [], []
    for t in range(x.shape[0]):
        logits = [math.fsum(float(a) * float(b) for a, b in zip(x[t], wr[e])) for e in range(wr.shape[0])]
        order = sorted(range(len(logits)), key=lambda e: (-logits[e], e))[:k]
        top = logits[order[0]]
        den = math.fsum(math.exp(logits[e] - top) for e in order)
        ids.append(order)
        ws.append([math.exp(logits[e] - top) / den for e in order])
    return np.array(ids, np.int32), np.array(ws)


@pytest.mark.parametrize("T,H,E,k,seed", [(5, 8, 6, 3, 0), (7, 32, 16, 4, 1), (3, 64, 9, 9, 2), (4, 16, 5, 1, 3)])
def test_router_matches_brute_force(T, H, E, k, seed):
    x = S.activations(T, H, seed=seed)
    wr = S.activations(E, H, seed=seed + 10)
    xb, wrb = S.bf16_bits_np(x), S.bf16_bits_np(wr)
    ids, w, logits = O.route(xb, wrb, k)
    bids, bw = _brute(xb, wrb, k)
    assert np.array_equal(ids, bids)
    assert np.allclose(w, bw, rtol=2 ** -23, atol=0)
    assert np.allclose(w.sum(axis=1), 1.0, atol=1e-6)
    assert np.all(np.diff(w, axis=1) <= 0)  # largest logit first, weights descending


def test_router_ties_go_to_the_lower_expert_index():
    # experts 1, 3 and 4 have identical rows (equal logits); expert 0 is lower
    H = 8
    row = [0.5, -1, 2, 0.25, 0, 1, -0.5, 3]
    wr = np.stack([_bf16([-1.0] * H), _bf16(row), _bf16([0.0] * H), _bf16(row), _bf16(row)])
    x = np.stack([_bf16([1.0] * H)])
    ids, w, _ = O.route(x, wr, 3)
    assert ids.tolist() == [[1, 3, 4]]
    assert np.allclose(w, 1.0 / 3.0)
    ids, w, _ = O.route(x, wr, 4)
    assert ids.tolist() == [[1, 3, 4, 2]]   # logit 0 beats -8


def test_router_k1_and_k_equal_e():
    x = S.bf16_bits_np(S.activations(6, 16, seed=4))
    wr = S.bf16_bits_np(S.activations(5, 16, seed=5))
    ids1, w1, logits = O.route(x, wr, 1)
    assert np.array_equal(ids1[:, 0], np.argmax(logits, axis=1)) and np.all(w1 == 1.0)
    idsE, wE, _ = O.route(x, wr, 5)
    for t in range(6):
        assert sorted(idsE[t].tolist()) == list(range(5))
        assert np.all(np.diff(logits[t][idsE[t]]) <= 0)
    with pytest.raises(ValueError):
        O.route(x, wr, 6)
