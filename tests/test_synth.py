"""The seeded generator: determinism, blob header, and the storage rule pinned
by the pages' printed checkpoint sizes."""
import os

import numpy as np
import pytest
import torch

import oracle as O
import synth as S

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_generator_is_deterministic_and_seeded():
    a = S.activations(4, 256, 7)
    b = S.activations(4, 256, 7)
    c = S.activations(4, 256, 8)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    assert not torch.equal(a.view(torch.int16), c.view(torch.int16))
    v = S.activations(64, 1024, 3).float()
    assert abs(v.mean().item()) < 0.02 and abs(v.std().item() - 1) < 0.02


def test_routing_shapes_and_distinctness():
    for ids in (S.routing_uniform(50, 16, 4, 1), S.routing_zipf(50, 16, 4, 1), S.routing_hot_cold(50, 40, 8, 1)):
        assert ids.dtype == torch.int32
        for row in ids.tolist():
            assert len(set(row)) == len(row)
    hc = S.routing_hot_cold(400, 256, 8, 4)
    counts = torch.bincount(hc.reshape(-1).long(), minlength=256)
    assert int((counts == 0).sum()) == 16
    assert int(counts.sort(descending=True).values[:26].sum()) == 400 * 4
    w = S.routing_weights(10, 8, 1)
    assert torch.allclose(w.sum(1), torch.ones(10))


def _oracle_down(b, wfmt, off):
    """One down-GEMM row through the oracle entry that matches the blob's format
    (K = I = 256)."""
    if wfmt == S.FMT_NVFP4_G16:
        return O.gemm_a4(b, 1, np.zeros((1, 128), np.uint8), np.zeros((1, 16), np.uint8),
                         np.zeros((1,), np.float32), off)
    return O.gemm_a16(b, 1, np.zeros((1, 256), np.uint16), off)


@pytest.mark.parametrize("wfmt", [0, 1, 2, 3])
def test_blob_header_parses_in_oracle(wfmt):
    blob, hdr, L = S.expert_blob(wfmt, 2, 256, 256, seed=3)
    # the oracle's own parser accepts the header; a flipped byte breaks the CRC
    b = blob.numpy().copy()
    off = np.array([0, 1, 1], np.int32)
    _oracle_down(b, wfmt, off)
    b[20] ^= 1
    with pytest.raises(ValueError):
        _oracle_down(b, wfmt, off)


def _sizes():
    out = {}
    with open(os.path.join(GOLDEN, "checkpoint_sizes.txt")) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if line:
                model, fmt, size, dec = line.split()
                out[(model, fmt)] = (float(size), int(dec))
    return out


def _bytes_per_weight(wfmt):
    N, K = 4096, 4096  # big enough that 256-byte alignment and the outer scale vanish
    return (S.code_bytes(wfmt, N, K) + S.scale_bytes(wfmt, N, K)) / (N * K)


def test_storage_rule_predicts_the_printed_checkpoint_sizes():
    """Only routed experts change between checkpoints, so size = rest + R * bytes/weight.
    BF16 and INT8 fix R and rest; the INT4 and NVFP4 sizes the pages print must follow."""
    sizes = _sizes()
    bpw = {f: _bytes_per_weight(c) for f, c in (("bf16", 0), ("int8", 1), ("int4", 2), ("nvfp4", 3))}
    assert bpw == {"bf16": 2.0, "int8": 1.015625, "int4": 0.515625, "nvfp4": 0.5625}
    for model in ("flash", "mini"):
        b16, d = sizes[(model, "bf16")]
        i8, _ = sizes[(model, "int8")]
        half = 0.5 * 10.0 ** -d
        lo_hi = []
        for db in (-half, half):
            for di in (-half, half):
                R = ((b16 + db) - (i8 + di)) / (bpw["bf16"] - bpw["int8"])
                rest = (b16 + db) - R * bpw["bf16"]
                lo_hi.append({f: rest + R * bpw[f] for f in ("int4", "nvfp4")})
        for f in ("int4", "nvfp4"):
            printed, _ = sizes[(model, f)]
            lo = min(p[f] for p in lo_hi) - half
            hi = max(p[f] for p in lo_hi) + half
            assert lo <= printed <= hi, (model, f, lo, printed, hi)
    # the flash figures are printed to 0.01 GiB: the prediction lands within it
    R = (191.66 - 100.11) / (2 - 1.015625)
    rest = 191.66 - 2 * R
    assert abs(rest + R * 0.515625 - 53.61) < 0.01
    assert abs(rest + R * 0.5625 - 57.97) < 0.01
