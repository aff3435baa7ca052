"""The unfused-activation comparison path: gate-only and up-only grouped
GEMMs on every kernel and format against the oracle, the SiLU * mul step
against the oracle's, and the whole layer with the fused activation switched
off against the oracle's unfused composition."""
import numpy as np
import pytest
import torch

import oracle as O
import synth as S
from gpu_util import REL_L2, REL_L2_NVFP4, assert_close, to_np_bits

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def M():
    import quantized_moe_expert_routed_gb300 as M
    M.load()
    return M


def test_silu_mul_matches_oracle(M):
    g = (S.activations(64, 512, seed=1).float() * 3).to(torch.bfloat16)
    u = S.activations(64, 512, seed=2)
    h = M.mnw_moe_silu_mul(g.to(DEV), u.to(DEV))
    want = O.silu_mul(S.bf16_bits_np(g), S.bf16_bits_np(u))
    assert_close(h, want, rel_l2=2e-3, max_abs=2e-2, what="silu_mul")
    # at most one BF16 ulp apart anywhere
    a, b = h.cpu().view(torch.int16).numpy().astype(np.int32), want.view(np.int16).astype(np.int32)
    assert np.abs(a - b).max() <= 1


@pytest.mark.parametrize("path", ["warp", "rows", "tcgen05"])
@pytest.mark.parametrize("wfmt", [S.FMT_INT4_G128, S.FMT_INT8_G128])
def test_single_matrix_gemms_int(M, path, wfmt):
    E, H, I, T, k = 8, 512, 256, 60, 4
    blob, hdr, L = S.expert_blob(wfmt, E, H, I, seed=9 + wfmt)
    ids = S.routing_uniform(T, E, k, seed=10)
    x = S.activations(T, H, seed=11)
    layer = M.Layer(blob.to(DEV), hdr)
    off, sa, pos, xp = M.mnw_moe_permute(ids.to(DEV), E, x=x.to(DEV))
    a, f = M.mnw_moe_quantize_act(M.ACT_F16_ROWS, x.to(DEV), row_index=sa, index_div=k)
    fn16 = M.mnw_moe_grouped_gemm_w4a16_f16rows if wfmt == S.FMT_INT4_G128 else M.mnw_moe_grouped_gemm_w8a16_f16rows
    fnbf = M.mnw_moe_grouped_gemm_w4a16 if wfmt == S.FMT_INT4_G128 else M.mnw_moe_grouped_gemm_w8a16
    M.mnw_moe_set_gemm_path({"warp": M.PATH_WARP_MMA, "rows": M.PATH_ROWS, "tcgen05": M.PATH_TCGEN05}[path])
    try:
        outs = {kind: (fn16(layer, kind, a, f, off), fnbf(layer, kind, xp, off)) for kind in (M.KIND_GATE, M.KIND_UP)}
    finally:
        M.mnw_moe_set_gemm_path(M.PATH_AUTO)
    o_off = off.cpu().numpy()
    for kind, (o16, obf) in outs.items():
        want = O.gemm_a16(blob.numpy(), kind, to_np_bits(xp), o_off)
        assert_close(o16, want, what=f"{path} f16rows kind {kind}")
        assert_close(obf, want, what=f"{path} bf16 kind {kind}")


def test_single_matrix_gemms_a8_a4_bf16(M):
    E, H, I, T, k = 8, 512, 512, 100, 4
    ids = S.routing_uniform(T, E, k, seed=20)
    x = S.activations(T, H, seed=21)
    # A8: group dots bit-exact
    blob, hdr, L = S.expert_blob(S.FMT_INT8_G128, E, H, I, seed=22)
    layer = M.Layer(blob.to(DEV), hdr)
    off, sa, pos, _ = M.mnw_moe_permute(ids.to(DEV), E)
    q, s = M.mnw_moe_quantize_act(M.ACT_INT8_G128, x.to(DEV), row_index=sa, index_div=k)
    o_off = off.cpu().numpy()
    for kind in (M.KIND_GATE, M.KIND_UP):
        out, dots = M.mnw_moe_grouped_gemm_w8a8(layer, kind, q, s, off, want_dots=True)
        want, wdots = O.gemm_a8(blob.numpy(), kind, q.cpu().numpy(), s.cpu().numpy(), o_off, want_dots=True)
        valid = int(o_off[-1])
        assert np.array_equal(dots.cpu().numpy()[:valid], wdots[:valid])
        assert_close(out, want, what=f"w8a8 kind {kind}")
    # NVFP4
    blob, hdr, L = S.expert_blob(S.FMT_NVFP4_G16, E, H, I, seed=23)
    layer = M.Layer(blob.to(DEV), hdr)
    c, sf, o = M.mnw_moe_quantize_act(M.ACT_NVFP4_G16, x.to(DEV), row_index=sa, index_div=k)
    for kind in (M.KIND_GATE, M.KIND_UP):
        out = M.mnw_moe_grouped_gemm_nvfp4(layer, kind, c, sf, o, off)
        want = O.gemm_a4(blob.numpy(), kind, c.cpu().numpy(), sf.cpu().numpy(), o.cpu().numpy(), o_off)
        assert_close(out, want, rel_l2=REL_L2_NVFP4, what=f"nvfp4 kind {kind}")
    # BF16 weights
    blob, hdr, L = S.expert_blob(S.FMT_BF16, E, H, I, seed=24)
    layer = M.Layer(blob.to(DEV), hdr)
    off, sa, pos, xp = M.mnw_moe_permute(ids.to(DEV), E, x=x.to(DEV))
    for kind in (M.KIND_GATE, M.KIND_UP):
        out = M.mnw_moe_grouped_gemm_bf16(layer, kind, xp, off)
        assert_close(out, O.gemm_a16(blob.numpy(), kind, to_np_bits(xp), o_off), what=f"bf16 kind {kind}")


def _oracle_unfused_layer(blob, act, x_bits, ids, w, E, k):
    """The unfused layer composed from oracle steps: permute, (quantise x),
    gate-only and up-only GEMMs (BF16 g, u), SiLU * mul, (quantise h), down,
    combine."""
    T = ids.shape[0]
    off, sa, pos, _ = O.permute(ids, E)
    valid = int(off[-1])
    xr = x_bits[np.maximum(sa, 0) // k]
    xr[valid:] = 0
    if act == S.ACT_BF16:
        g = O.gemm_a16(blob, O.KIND_GATE, xr, off)
        u = O.gemm_a16(blob, O.KIND_UP, xr, off)
    elif act == S.ACT_INT8_G128:
        q, s = O.quant_int8_g128(xr)
        g = O.gemm_a8(blob, O.KIND_GATE, q, s, off)
        u = O.gemm_a8(blob, O.KIND_UP, q, s, off)
    else:
        c, sf, o = O.quant_nvfp4_g16(xr)
        g = O.gemm_a4(blob, O.KIND_GATE, c, sf, o, off)
        u = O.gemm_a4(blob, O.KIND_UP, c, sf, o, off)
    h = O.silu_mul(g, u)
    if act == S.ACT_BF16:
        y = O.gemm_a16(blob, O.KIND_DOWN, h, off)
    elif act == S.ACT_INT8_G128:
        q, s = O.quant_int8_g128(h)
        y = O.gemm_a8(blob, O.KIND_DOWN, q, s, off)
    else:
        c, sf, o = O.quant_nvfp4_g16(h)
        y = O.gemm_a4(blob, O.KIND_DOWN, c, sf, o, off)
    return O.combine(y, pos, w, T, k)


@pytest.mark.parametrize("name", ["decode_w4a16", "w8a8_2048", "prefill_nvfp4", "large_bf16", "large_w4a16"])
def test_forward_unfused_matches_oracle(M, name):
    wl = S.WORKLOADS[name]
    wl = S.Workload(**{**wl.__dict__, "T": 64, "E": 64, "H": 512,
                       "I": 512 if wl.wfmt == S.FMT_NVFP4_G16 else 256})
    x, ids, w, blob, hdr, L = S.make_inputs(wl, device=DEV)
    layer = M.Layer(blob, hdr)
    M.mnw_moe_set_fused_activation(False)
    try:
        out = M.mnw_moe_forward(layer, wl.act, x, ids, w)
    finally:
        M.mnw_moe_set_fused_activation(True)
    fused = M.mnw_moe_forward(layer, wl.act, x, ids, w)
    want = _oracle_unfused_layer(blob.cpu().numpy(), wl.act, S.bf16_bits_np(x), ids.cpu().numpy(), w.cpu().numpy(),
                                 wl.E, wl.k)
    tol = REL_L2_NVFP4 if wl.act == S.ACT_NVFP4_G16 else REL_L2
    assert_close(out, want, rel_l2=tol, what=f"{name} unfused")
    # the two paths differ only by the BF16 rounding of g and u -- amplified in
    # the A4 mode, where h is re-quantised to E2M1 before the down GEMM
    a, b = out.double(), fused.double()
    assert (a - b).norm() <= (5 if wl.act == S.ACT_NVFP4_G16 else 2) * tol * b.norm()
