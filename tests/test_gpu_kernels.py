"""GPU parity of each C-ABI call against the CPU oracle, on seeded inputs that
span several tiles, ragged token tiles and empty experts."""
import numpy as np
import pytest
import torch

import oracle as O
import synth as S
from gpu_util import REL_L2_NVFP4, assert_close, to_np_bits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def M():
    import quantized_moe_expert_routed_gb300 as M
    M.load()
    return M


DEV = "cuda"


@pytest.mark.parametrize("T,k,E,bad", [(1, 1, 1, False), (37, 2, 8, False), (256, 8, 256, False),
                                       (255, 8, 128, True), (257, 8, 64, False), (512, 8, 256, True),
                                       (1024, 8, 1024, True), (1025, 8, 256, False),
                                       (2048, 8, 256, True), (8192, 8, 256, False), (33, 3, 1024, True),
                                       (2048, 8, 1024, True), (1100, 8, 256, True), (1030, 9, 256, False)])
def test_permute_bitexact(M, T, k, E, bad):
    ids = S.routing_uniform(T, E, k, seed=T + E) if k <= E else None
    ids = ids.clone()
    if bad:
        ids[::7, 0] = E + 5
        ids[3, -1] = -2
    x = S.activations(T, 256, seed=5)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    off, sa, pos, xp = M.mnw_moe_permute(ids.to(DEV), E, x=x.to(DEV), err=err)
    o_off, o_sa, o_pos, dropped = O.permute(ids.numpy(), E)
    assert np.array_equal(off.cpu().numpy(), o_off)
    assert np.array_equal(sa.cpu().numpy(), o_sa)
    assert np.array_equal(pos.cpu().numpy(), o_pos)
    assert (M.mnw_moe_read_error(err) != 0) == (dropped > 0)
    # gathered rows are the tokens' rows, zero where no assignment
    xb = x.view(torch.int16)
    want = torch.zeros((T * k, 256), dtype=torch.int16)
    valid = torch.from_numpy(o_sa) >= 0
    want[valid] = xb[torch.from_numpy(o_sa)[valid].long() // k]
    assert torch.equal(xp.cpu().view(torch.int16), want)


def _ids_with_duplicates(T, k, E, seed):
    """Routing with repeated experts: some tokens name one expert twice or
    more, and the first 32 assignments (one warp's batch) all name expert
    min(3, E - 1); the rest are drawn with replacement, so most warp batches
    hold several lanes with the same id."""
    g = torch.Generator().manual_seed(seed)
    ids = torch.randint(0, E, (T, k), generator=g, dtype=torch.int32)
    ids[::5, 1 % k] = ids[::5, 0]             # a duplicate inside one token
    ids.view(-1)[:min(32, T * k)] = min(3, E - 1)  # a whole warp batch on one expert
    return ids


# (T, k, E): one shape per permute variant -- one CTA of 8 warps (<= 2048
# assignments), one CTA of 16 warps (<= 8192), count/scan/place over many CTAs,
# and the 32-warp CTA for batches the chunked variant does not take
@pytest.mark.parametrize("T,k,E", [(64, 8, 16), (37, 3, 4), (512, 8, 64), (2048, 8, 256), (1030, 9, 256)])
def test_permute_duplicate_ids_bitexact(M, T, k, E):
    """Duplicate ids within a token are separate assignments, ranked by their
    flat index (stable), exactly as the oracle's counting sort."""
    ids = _ids_with_duplicates(T, k, E, seed=T * 31 + E)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    off, sa, pos, _ = M.mnw_moe_permute(ids.to(DEV), E, err=err)
    o_off, o_sa, o_pos, dropped = O.permute(ids.numpy(), E)
    assert dropped == 0 and M.mnw_moe_read_error(err) == 0
    assert np.array_equal(off.cpu().numpy(), o_off)
    assert np.array_equal(sa.cpu().numpy(), o_sa)
    assert np.array_equal(pos.cpu().numpy(), o_pos)


@pytest.mark.parametrize("T,k,E", [(64, 8, 16), (37, 3, 4), (512, 8, 64), (2048, 8, 256), (1030, 9, 256)])
@pytest.mark.parametrize("shift", [1, 2, 3])
def test_permute_unaligned_ids_bitexact(M, T, k, E, shift):
    """ids that start off a 16-byte boundary (the kernels then read them with
    4-byte loads) give the same permutation as aligned ones and the oracle."""
    ids = _ids_with_duplicates(T, k, E, seed=T * 17 + E + shift)
    buf = torch.full((T * k + 8,), -7, dtype=torch.int32, device=DEV)
    view = buf[shift:shift + T * k].view(T, k)
    view.copy_(ids.to(DEV))
    assert view.data_ptr() % 16 != 0
    off, sa, pos, _ = M.mnw_moe_permute(view, E)
    o_off, o_sa, o_pos, dropped = O.permute(ids.numpy(), E)
    assert dropped == 0
    assert np.array_equal(off.cpu().numpy(), o_off)
    assert np.array_equal(sa.cpu().numpy(), o_sa)
    assert np.array_equal(pos.cpu().numpy(), o_pos)


# K: rows of up to 1024 values (a row per warp in registers, one to four
# 16-byte words per lane), odd group counts, and longer rows cut into chunks
# of 512 (2048, 4096) or 256 values (4352)
@pytest.mark.parametrize("R,K,gather", [(1, 128, False), (37, 512, False), (300, 2048, True), (5, 384, False),
                                        (9, 1024, False), (40, 1536, True), (3, 4096, False), (2, 4352, False)])
def test_quantize_int8_bitexact(M, R, K, gather):
    x = S.activations(R, K, seed=R, outlier_p=0.01)
    x[min(3, R - 1), :128] = 0  # an all-zero group
    idx = None
    src = x
    if gather:
        idx = torch.arange(R * 2, dtype=torch.int32).flip(0)[:R].contiguous()
        idx[5] = -1
        src = torch.zeros_like(x)
        for r in range(R):
            if idx[r] >= 0:
                src[r] = x[int(idx[r]) // 2]
        x_in = x
    else:
        x_in = x
    codes, scales = M.mnw_moe_quantize_act(M.ACT_INT8_G128, x_in.to(DEV),
                                          row_index=None if idx is None else idx.to(DEV), index_div=2, rows=R)
    oc, osc = O.quant_int8_g128(S.bf16_bits_np(src))
    assert np.array_equal(codes.cpu().numpy(), oc)
    assert np.array_equal(scales.cpu().numpy().view(np.uint32), osc.view(np.uint32))


# K: blocks that do not fill the last lane pass (272), rows of up to 1024
# values (a row per warp in registers) and longer rows (the two-pass kernel)
@pytest.mark.parametrize("R,K,gather", [(1, 256, False), (29, 512, False), (200, 2048, True), (4, 272, False),
                                        (16, 1024, True), (3, 4096, False), (2, 4608, False), (5, 1536, False),
                                        (11, 1040, False), (9, 2048, False)])
def test_quantize_nvfp4_bitexact(M, R, K, gather):
    x = S.activations(R, K, seed=R + 1)
    x[0, 5] = -1e-6        # tiny negative: rounds to E2M1 zero, sign kept
    x[min(2, R - 1)] = 0   # a zero row
    idx = None
    src = x
    if gather:
        idx = torch.arange(R, dtype=torch.int32).flip(0).contiguous()
        idx[7] = -1
        src = torch.zeros_like(x)
        for r in range(R):
            if idx[r] >= 0:
                src[r] = x[int(idx[r])]
    codes, sf, outer = M.mnw_moe_quantize_act(M.ACT_NVFP4_G16, x.to(DEV),
                                             row_index=None if idx is None else idx.to(DEV), index_div=1, rows=R)
    oc, osf, oo = O.quant_nvfp4_g16(S.bf16_bits_np(src))
    assert np.array_equal(outer.cpu().numpy().view(np.uint32), oo.view(np.uint32))
    assert np.array_equal(sf.cpu().numpy(), osf)
    assert np.array_equal(codes.cpu().numpy(), oc)


def test_combine_matches_oracle(M):
    T, k, H = 67, 8, 512
    P = T * k
    y = S.activations(P, H, seed=9)
    pos = torch.randperm(P, generator=torch.Generator().manual_seed(0)).to(torch.int32)
    pos[::11] = -1
    w = S.routing_weights(T, k, seed=3)
    out = M.mnw_moe_combine(y.to(DEV), pos.to(DEV), w.to(DEV))
    want = O.combine(S.bf16_bits_np(y), pos.numpy(), w.numpy(), T, k)
    assert_close(out, want, rel_l2=2e-3, max_abs=1e-2, what="combine")


# ---- grouped GEMMs --------------------------------------------------------------

SHAPES = [
    # (E, H, I, T, k): ragged decode-like tiles, and multi-tile prefill-like experts
    (8, 512, 256, 40, 2),
    (4, 512, 256, 300, 2),
]


def _setup(wfmt, E, H, I, T, k, seed, outlier_p=0.0):
    """Seeded blob, routing and activations.  Outliers (x20, as in the W8A8
    workload) only where the A8 path is tested: elsewhere they push |h| past
    4, where one BF16 ulp alone exceeds the 2e-2 absolute bound."""
    blob, hdr, L = S.expert_blob(wfmt, E, H, I, seed=seed)
    ids = S.routing_uniform(T, E, k, seed=seed + 1)
    x = S.activations(T, H, seed=seed + 2, outlier_p=outlier_p)
    return blob, hdr, ids, x


@pytest.mark.parametrize("wfmt,fn", [(S.FMT_BF16, "mnw_moe_grouped_gemm_bf16"),
                                     (S.FMT_INT8_G128, "mnw_moe_grouped_gemm_w8a16"),
                                     (S.FMT_INT4_G128, "mnw_moe_grouped_gemm_w4a16")])
@pytest.mark.parametrize("shape", SHAPES)
def test_gemm_a16(M, wfmt, fn, shape):
    E, H, I, T, k = shape
    blob, hdr, ids, x = _setup(wfmt, E, H, I, T, k, seed=7 * wfmt + T)
    layer = M.Layer(blob.to(DEV), hdr)
    off, sa, pos, xp = M.mnw_moe_permute(ids.to(DEV), E, x=x.to(DEV))
    h = getattr(M, fn)(layer, M.KIND_GATE_UP, xp, off)
    y = getattr(M, fn)(layer, M.KIND_DOWN, h, off)
    o_off = off.cpu().numpy()
    xp_bits = to_np_bits(xp)
    oh = O.gemm_a16(blob.numpy(), O.KIND_GATE_UP, xp_bits, o_off)
    assert_close(h, oh, what=f"{fn} gate_up")
    oy = O.gemm_a16(blob.numpy(), O.KIND_DOWN, to_np_bits(h), o_off)
    assert_close(y, oy, what=f"{fn} down")


@pytest.mark.parametrize("wfmt,fn", [(S.FMT_INT8_G128, "mnw_moe_grouped_gemm_w8a8"),
                                     (S.FMT_INT4_G128, "mnw_moe_grouped_gemm_w4a8")])
@pytest.mark.parametrize("shape", SHAPES)
def test_gemm_a8_group_dots_bitexact(M, wfmt, fn, shape):
    E, H, I, T, k = shape
    blob, hdr, ids, x = _setup(wfmt, E, H, I, T, k, seed=11 * wfmt + T, outlier_p=0.01)
    layer = M.Layer(blob.to(DEV), hdr)
    off, sa, pos, _ = M.mnw_moe_permute(ids.to(DEV), E)
    q, s = M.mnw_moe_quantize_act(M.ACT_INT8_G128, x.to(DEV), row_index=sa, index_div=k)
    h, dots = getattr(M, fn)(layer, M.KIND_GATE_UP, q, s, off, want_dots=True)
    o_off = off.cpu().numpy()
    oh, odots = O.gemm_a8(blob.numpy(), O.KIND_GATE_UP, q.cpu().numpy(), s.cpu().numpy(), o_off, want_dots=True)
    valid = int(o_off[-1])
    assert np.array_equal(dots.cpu().numpy()[:valid], odots[:valid])
    assert_close(h, oh, what=f"{fn} gate_up")
    hq, hs = M.mnw_moe_quantize_act(M.ACT_INT8_G128, h)
    y, ydots = getattr(M, fn)(layer, M.KIND_DOWN, hq, hs, off, want_dots=True)
    oy, oydots = O.gemm_a8(blob.numpy(), O.KIND_DOWN, hq.cpu().numpy(), hs.cpu().numpy(), o_off, want_dots=True)
    assert np.array_equal(ydots.cpu().numpy()[:valid], oydots[:valid])
    assert_close(y, oy, what=f"{fn} down")


@pytest.mark.parametrize("shape", [(8, 512, 256, 40, 2), (4, 512, 512, 300, 2)])
def test_gemm_nvfp4(M, shape):
    E, H, I, T, k = shape
    blob, hdr, ids, x = _setup(S.FMT_NVFP4_G16, E, H, I, T, k, seed=13 + T)
    layer = M.Layer(blob.to(DEV), hdr)
    off, sa, pos, _ = M.mnw_moe_permute(ids.to(DEV), E)
    c, sf, o = M.mnw_moe_quantize_act(M.ACT_NVFP4_G16, x.to(DEV), row_index=sa, index_div=k)
    h = M.mnw_moe_grouped_gemm_nvfp4(layer, M.KIND_GATE_UP, c, sf, o, off)
    o_off = off.cpu().numpy()
    oh = O.gemm_a4(blob.numpy(), O.KIND_GATE_UP, c.cpu().numpy(), sf.cpu().numpy(), o.cpu().numpy(), o_off)
    assert_close(h, oh, rel_l2=REL_L2_NVFP4, what="nvfp4 gate_up")
    hc, hsf, ho = M.mnw_moe_quantize_act(M.ACT_NVFP4_G16, h)
    y = M.mnw_moe_grouped_gemm_nvfp4(layer, M.KIND_DOWN, hc, hsf, ho, off)
    oy = O.gemm_a4(blob.numpy(), O.KIND_DOWN, hc.cpu().numpy(), hsf.cpu().numpy(), ho.cpu().numpy(), o_off)
    assert_close(y, oy, rel_l2=REL_L2_NVFP4, what="nvfp4 down")


@pytest.mark.parametrize("shape", [(8, 512, 256, 40, 2), (4, 512, 512, 300, 2)])
def test_gemm_nvfp4_full_scale_range(M, shape):
    """NVFP4 weights whose E4M3 block scales cover every non-negative finite
    code (zero, subnormals, up to 448) and whose per-matrix outer scales
    spread over a factor of 256: the block-scale decode is exercised over its
    whole range."""
    E, H, I, T, k = shape
    # sigma keeps |h| well below 1, where one BF16 ulp is inside the absolute bound
    blob, hdr, L = S.expert_blob(S.FMT_NVFP4_G16, E, H, I, seed=41 + T, sigma=0.006, nvfp4_sf_range="full")
    sf_bytes = blob.numpy()[L.data_offset + L.scales_off[0]:][:I * H // 16]
    assert sf_bytes.min() == 0 and sf_bytes.max() == 0x7E and ((sf_bytes > 0) & (sf_bytes < 8)).any()
    ids = S.routing_uniform(T, E, k, seed=42 + T)
    x = S.activations(T, H, seed=43 + T)
    layer = M.Layer(blob.to(DEV), hdr)
    off, sa, pos, _ = M.mnw_moe_permute(ids.to(DEV), E)
    c, sf, o = M.mnw_moe_quantize_act(M.ACT_NVFP4_G16, x.to(DEV), row_index=sa, index_div=k)
    h = M.mnw_moe_grouped_gemm_nvfp4(layer, M.KIND_GATE_UP, c, sf, o, off)
    o_off = off.cpu().numpy()
    oh = O.gemm_a4(blob.numpy(), O.KIND_GATE_UP, c.cpu().numpy(), sf.cpu().numpy(), o.cpu().numpy(), o_off)
    assert_close(h, oh, rel_l2=REL_L2_NVFP4, what="nvfp4 full-range gate_up")
    hc, hsf, ho = M.mnw_moe_quantize_act(M.ACT_NVFP4_G16, h)
    y = M.mnw_moe_grouped_gemm_nvfp4(layer, M.KIND_DOWN, hc, hsf, ho, off)
    oy = O.gemm_a4(blob.numpy(), O.KIND_DOWN, hc.cpu().numpy(), hsf.cpu().numpy(), ho.cpu().numpy(), o_off)
    assert_close(y, oy, rel_l2=REL_L2_NVFP4, what="nvfp4 full-range down")


def test_gemm_empty_experts_and_zero_rows(M):
    E, H, I = 6, 256, 256
    blob, hdr, L = S.expert_blob(S.FMT_INT4_G128, E, H, I, seed=3)
    layer = M.Layer(blob.to(DEV), hdr)
    ids = torch.tensor([[5], [5], [0], [5]], dtype=torch.int32)   # experts 1-4 empty
    x = S.activations(4, H, seed=4)
    off, sa, pos, xp = M.mnw_moe_permute(ids.to(DEV), E, x=x.to(DEV))
    h = M.mnw_moe_grouped_gemm_w4a16(layer, M.KIND_GATE_UP, xp, off)
    oh = O.gemm_a16(blob.numpy(), O.KIND_GATE_UP, to_np_bits(xp), off.cpu().numpy())
    assert_close(h, oh, what="empty experts")


@pytest.mark.parametrize("wfmt,act", [(S.FMT_INT4_G128, S.ACT_BF16), (S.FMT_INT8_G128, S.ACT_BF16),
                                      (S.FMT_INT4_G128, S.ACT_INT8_G128), (S.FMT_INT8_G128, S.ACT_INT8_G128)])
@pytest.mark.parametrize("T,k,E", [(40, 2, 8), (64, 8, 16), (130, 4, 8)])
def test_warp_and_tcgen05_paths_agree_bitwise(M, wfmt, act, T, k, E):
    """Both grouped-GEMM kernels sum each 128-wide group on the tensor cores in
    FP32 and combine the groups with the same FP32 operations.  With INT8
    activations every group dot is an exact integer, so the outputs are
    identical bits; with BF16 activations the in-group FP32 sums may round in
    a different order, so the outputs agree to that rounding."""
    H, I = 512, 256
    blob, hdr, ids, x = _setup(wfmt, E, H, I, T, k, seed=17 * T + wfmt)
    layer = M.Layer(blob.to(DEV), hdr)
    off, sa, pos, xp = M.mnw_moe_permute(ids.to(DEV), E, x=x.to(DEV))
    outs = []
    try:
        for path in (M.PATH_TCGEN05, M.PATH_WARP_MMA):
            M.mnw_moe_set_gemm_path(path)
            if act == S.ACT_BF16:
                fn = M.mnw_moe_grouped_gemm_w4a16 if wfmt == S.FMT_INT4_G128 else M.mnw_moe_grouped_gemm_w8a16
                h = fn(layer, M.KIND_GATE_UP, xp, off)
                y = fn(layer, M.KIND_DOWN, h, off)
                outs.append((h, y, None))
            else:
                fn = M.mnw_moe_grouped_gemm_w4a8 if wfmt == S.FMT_INT4_G128 else M.mnw_moe_grouped_gemm_w8a8
                q, s = M.mnw_moe_quantize_act(M.ACT_INT8_G128, x.to(DEV), row_index=sa, index_div=k)
                h, dots = fn(layer, M.KIND_GATE_UP, q, s, off, want_dots=True)
                hq, hs = M.mnw_moe_quantize_act(M.ACT_INT8_G128, h)
                y = fn(layer, M.KIND_DOWN, hq, hs, off)
                outs.append((h, y, dots))
    finally:
        M.mnw_moe_set_gemm_path(M.PATH_AUTO)
    (h0, y0, d0), (h1, y1, d1) = outs
    if act == S.ACT_INT8_G128:
        assert torch.equal(h0.view(torch.int16), h1.view(torch.int16))
        assert torch.equal(y0.view(torch.int16), y1.view(torch.int16))
    else:
        for p0, p1 in ((h0, h1), (y0, y1)):
            a, b = p0.double(), p1.double()
            assert (a - b).norm() <= 2e-3 * b.norm()
            assert ((a - b).abs() > b.abs() * 2.0 ** -7 + 1e-6).float().mean() <= 1e-3
    if d0 is not None:
        valid = int(off[-1])
        assert torch.equal(d0[:valid], d1[:valid])
    # and the warp path matches the oracle
    o_off = off.cpu().numpy()
    if act == S.ACT_BF16:
        oh = O.gemm_a16(blob.numpy(), O.KIND_GATE_UP, to_np_bits(xp), o_off)
    else:
        oh = O.gemm_a8(blob.numpy(), O.KIND_GATE_UP, q.cpu().numpy(), s.cpu().numpy(), o_off)
    assert_close(h1, oh, what="warp path gate_up")


# ---- FP16 row form: INT8/INT4 weights, BF16 activations on FP16 tensor cores -----

def _f16_row_inputs(R, K, seed):
    """Activations with rows far from unit scale: tiny, huge, zero, and one
    holding the largest finite BF16 magnitude."""
    x = S.activations(R, K, seed=seed).float()
    for r, f in ((2, 1e-20), (4, 1e25), (6, 0.0), (9, 3e-3)):
        if r < R:
            x[r] *= f
    x = x.to(torch.bfloat16)
    if R > 7:
        x.view(torch.int16)[7, 1] = 0x7F7F
    return x


@pytest.mark.parametrize("R,K,gather", [(1, 128, False), (37, 512, False), (300, 2048, True), (64, 7168, True)])
def test_quantize_f16_rows_bitexact(M, R, K, gather):
    x = _f16_row_inputs(R, K, seed=R + 3)
    idx = None
    src = x
    if gather:
        idx = torch.arange(R * 2, dtype=torch.int32).flip(0)[:R].contiguous()
        idx[5] = -1
        src = torch.zeros_like(x)
        for r in range(R):
            if idx[r] >= 0:
                src[r] = x[int(idx[r]) // 2]
    codes, outer = M.mnw_moe_quantize_act(M.ACT_F16_ROWS, x.to(DEV),
                                          row_index=None if idx is None else idx.to(DEV), index_div=2, rows=R)
    oc, of = O.encode_f16_rows(S.bf16_bits_np(src))
    if idx is not None:
        dropped = (idx < 0).numpy()
        oc[dropped] = 0
        of[dropped] = 1.0  # a negative row index: zero codes, factor 1
    assert np.array_equal(codes.cpu().view(torch.int16).numpy().view(np.uint16), oc)
    assert np.array_equal(outer.cpu().numpy().view(np.uint32), of.view(np.uint32))


@pytest.mark.parametrize("wfmt,fn", [(S.FMT_INT8_G128, "mnw_moe_grouped_gemm_w8a16_f16rows"),
                                     (S.FMT_INT4_G128, "mnw_moe_grouped_gemm_w4a16_f16rows")])
@pytest.mark.parametrize("shape", SHAPES + [(16, 1024, 512, 400, 4)])
def test_gemm_f16rows(M, wfmt, fn, shape):
    E, H, I, T, k = shape
    blob, hdr, ids, x = _setup(wfmt, E, H, I, T, k, seed=17 * wfmt + T)
    layer = M.Layer(blob.to(DEV), hdr)
    off, sa, pos, xp = M.mnw_moe_permute(ids.to(DEV), E, x=x.to(DEV))
    a, f = M.mnw_moe_quantize_act(M.ACT_F16_ROWS, x.to(DEV), row_index=sa, index_div=k)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    h = getattr(M, fn)(layer, M.KIND_GATE_UP, a, f, off, err=err)
    assert int(err.item()) == 0
    o_off = off.cpu().numpy()
    # the definition: the W8A16/W4A16 GEMM of the original BF16 rows
    oh_def = O.gemm_a16(blob.numpy(), O.KIND_GATE_UP, to_np_bits(xp), o_off)
    assert_close(h, oh_def, what=f"{fn} gate_up vs the BF16-row definition")
    # and the oracle's GEMM over the same encoded rows
    oh = O.gemm_f16rows(blob.numpy(), O.KIND_GATE_UP, a.cpu().view(torch.int16).numpy().view(np.uint16),
                        f.cpu().numpy(), o_off)
    assert_close(h, oh, what=f"{fn} gate_up")
    ha, hf = M.mnw_moe_quantize_act(M.ACT_F16_ROWS, h)
    y = getattr(M, fn)(layer, M.KIND_DOWN, ha, hf, off, err=err)
    assert int(err.item()) == 0
    oy_def = O.gemm_a16(blob.numpy(), O.KIND_DOWN, to_np_bits(h), o_off)
    assert_close(y, oy_def, what=f"{fn} down vs the BF16-row definition")
    oy = O.gemm_f16rows(blob.numpy(), O.KIND_DOWN, ha.cpu().view(torch.int16).numpy().view(np.uint16),
                        hf.cpu().numpy(), o_off)
    assert_close(y, oy, what=f"{fn} down")


def test_gemm_f16rows_rejects_bad_kind_format_and_out_of_range_scales(M):
    E, H, I, T, k = 4, 256, 256, 16, 2
    blob, hdr, ids, x = _setup(S.FMT_INT8_G128, E, H, I, T, k, seed=21)
    layer = M.Layer(blob.to(DEV), hdr)
    off, sa, pos, _ = M.mnw_moe_permute(ids.to(DEV), E)
    a, f = M.mnw_moe_quantize_act(M.ACT_F16_ROWS, x.to(DEV), row_index=sa, index_div=k)
    with pytest.raises(M.MnwError, match="invalid"):
        M.mnw_moe_grouped_gemm_w8a16_f16rows(layer, 7, a, f, off)
    with pytest.raises(M.MnwError, match="mode not allowed"):
        M.mnw_moe_grouped_gemm_w4a16_f16rows(layer, M.KIND_GATE_UP, a, f, off)  # INT8 layer
    # scales near 65504 / 127: some fp16(q * s) would overflow
    big, hdr_b, _ = S.expert_blob(S.FMT_INT8_G128, E, H, I, seed=22, sigma=5.0e4)
    with pytest.raises(M.MnwError, match="unsupported"):
        M.mnw_moe_grouped_gemm_w8a16_f16rows(M.Layer(big.to(DEV), hdr_b), M.KIND_GATE_UP, a, f, off)
    # scales below 2^-14: some fp16(q * s) would be subnormal
    tiny, hdr_t, _ = S.expert_blob(S.FMT_INT4_G128, E, H, I, seed=23, sigma=1.0e-6)
    with pytest.raises(M.MnwError, match="unsupported"):
        M.mnw_moe_grouped_gemm_w4a16_f16rows(M.Layer(tiny.to(DEV), hdr_t), M.KIND_GATE_UP, a, f, off)


def test_standalone_gemm_graph_replay_on_two_streams(M):
    """A standalone grouped-GEMM call keeps no state between calls (on the
    warp-MMA kernel its CTAs take work units in a static order): two captured
    launches replayed concurrently on two streams, several times, give the
    eager result bit for bit."""
    E, H, I, T, k = 64, 512, 256, 96, 4  # 6 tokens per expert: the warp-MMA kernel
    blob, hdr, ids, x = _setup(S.FMT_INT4_G128, E, H, I, T, k, seed=71)
    layer = M.Layer(blob.to(DEV), hdr)
    off, sa, pos, xp = M.mnw_moe_permute(ids.to(DEV), E, x=x.to(DEV))
    ref = M.mnw_moe_grouped_gemm_w4a16(layer, M.KIND_GATE_UP, xp, off)
    torch.cuda.synchronize()
    lib = M.load()
    import ctypes
    P = T * k
    outs = [torch.full_like(ref, float("nan")) for _ in range(2)]
    graphs = []
    for o in outs:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            rc = lib.mnw_moe_grouped_gemm_w4a16(layer.handle, M.KIND_GATE_UP, ctypes.c_void_p(xp.data_ptr()),
                                                ctypes.c_void_p(off.data_ptr()), P, ctypes.c_void_p(o.data_ptr()),
                                                None, ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
        assert rc == 0
        graphs.append(g)
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    for _ in range(3):
        for g, s in zip(graphs, streams):
            s.wait_stream(torch.cuda.current_stream())
            with torch.cuda.stream(s):
                g.replay()
    torch.cuda.synchronize()
    for o in outs:
        assert torch.equal(o.view(torch.int16), ref.view(torch.int16))


@pytest.mark.parametrize("wfmt", [S.FMT_INT4_G128, S.FMT_INT8_G128, S.FMT_BF16])
@pytest.mark.parametrize("T,k,E,H,I", [(300, 4, 8, 512, 256), (40, 2, 8, 512, 256), (700, 2, 16, 512, 256),
                                       (33, 8, 64, 512, 768)])
def test_row_tile_kernel_forced_matches_oracle(M, wfmt, T, k, E, H, I):
    """The row-tile tcgen05 kernel (tokens as M, 256 weight rows as N) forced on
    every shape: token tiles of 1..128 rows, experts with several tiles, empty
    experts, feature tiles of 128 (gate/up) and 256 (down) columns.  INT
    weights take FP16 rows, BF16 weights BF16 rows."""
    blob, hdr, ids, x = _setup(wfmt, E, H, I, T, k, seed=5 * T + wfmt)
    ids[: T // 3, 0] = 1  # a crowded expert (several token tiles)
    if E > 8:
        ids[ids == 5] = 6  # an empty expert
    layer = M.Layer(blob.to(DEV), hdr)
    off, sa, pos, xp = M.mnw_moe_permute(ids.to(DEV), E, x=x.to(DEV))
    o_off = off.cpu().numpy()
    M.mnw_moe_set_gemm_path(M.PATH_ROWS)
    try:
        if wfmt == S.FMT_BF16:
            h = M.mnw_moe_grouped_gemm_bf16(layer, M.KIND_GATE_UP, xp, off)
            y = M.mnw_moe_grouped_gemm_bf16(layer, M.KIND_DOWN, h, off)
        else:
            fn = M.mnw_moe_grouped_gemm_w4a16_f16rows if wfmt == S.FMT_INT4_G128 else \
                M.mnw_moe_grouped_gemm_w8a16_f16rows
            a, f = M.mnw_moe_quantize_act(M.ACT_F16_ROWS, x.to(DEV), row_index=sa, index_div=k)
            h = fn(layer, M.KIND_GATE_UP, a, f, off)
            ha, hf = M.mnw_moe_quantize_act(M.ACT_F16_ROWS, h)
            y = fn(layer, M.KIND_DOWN, ha, hf, off)
    finally:
        M.mnw_moe_set_gemm_path(M.PATH_AUTO)
    assert_close(h, O.gemm_a16(blob.numpy(), O.KIND_GATE_UP, to_np_bits(xp), o_off), what="row tiles gate_up")
    assert_close(y, O.gemm_a16(blob.numpy(), O.KIND_DOWN, to_np_bits(h), o_off), what="row tiles down")


@pytest.mark.parametrize("path", ["rows", "tcgen05"])
@pytest.mark.parametrize("T,k,E,H,I", [(300, 4, 8, 512, 512), (40, 2, 8, 1024, 512), (700, 2, 16, 2048, 512),
                                       (33, 8, 64, 512, 1024)])
def test_a8_kernels_forced_match_oracle(M, path, T, k, E, H, I):
    """W8A8 on the row-tile kernel (tokens as M, 128 weight rows as N, one
    accumulator per 128-K group, running sums in registers) and on the
    weight-tile kernel, each forced on every shape: ragged and crowded experts,
    an empty one, group dots bit for bit, the fused pair and the single gate
    and up matrices of the unfused path, and down."""
    blob, hdr, ids, x = _setup(S.FMT_INT8_G128, E, H, I, T, k, seed=7 * T + E, outlier_p=0.01)
    ids[: T // 3, 0] = 1  # a crowded expert
    if E > 8:
        ids[ids == 5] = 6  # an empty expert
    layer = M.Layer(blob.to(DEV), hdr)
    off, sa, pos, _ = M.mnw_moe_permute(ids.to(DEV), E)
    o_off = off.cpu().numpy()
    valid = int(o_off[-1])
    q, s = M.mnw_moe_quantize_act(M.ACT_INT8_G128, x.to(DEV), row_index=sa, index_div=k)
    qn, sn = q.cpu().numpy(), s.cpu().numpy()
    M.mnw_moe_set_gemm_path(M.PATH_ROWS if path == "rows" else M.PATH_TCGEN05)
    try:
        for kind, okind in ((M.KIND_GATE_UP, O.KIND_GATE_UP), (M.KIND_GATE, O.KIND_GATE), (M.KIND_UP, O.KIND_UP)):
            h, dots = M.mnw_moe_grouped_gemm_w8a8(layer, kind, q, s, off, want_dots=True)
            oh, odots = O.gemm_a8(blob.numpy(), okind, qn, sn, o_off, want_dots=True)
            assert np.array_equal(dots.cpu().numpy()[:valid], odots[:valid]), (path, kind)
            assert_close(h, oh, what=f"w8a8 {path} kind {kind}")
        h2, _ = M.mnw_moe_grouped_gemm_w8a8(layer, M.KIND_GATE_UP, q, s, off, want_dots=True)
        hq, hs = M.mnw_moe_quantize_act(M.ACT_INT8_G128, h2)
        y, ydots = M.mnw_moe_grouped_gemm_w8a8(layer, M.KIND_DOWN, hq, hs, off, want_dots=True)
        oy, oydots = O.gemm_a8(blob.numpy(), O.KIND_DOWN, hq.cpu().numpy(), hs.cpu().numpy(), o_off, want_dots=True)
        assert np.array_equal(ydots.cpu().numpy()[:valid], oydots[:valid]), path
        assert_close(y, oy, what=f"w8a8 {path} down")
    finally:
        M.mnw_moe_set_gemm_path(M.PATH_AUTO)
