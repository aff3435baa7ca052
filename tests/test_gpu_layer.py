"""Whole-layer parity: mnw_moe_forward against the oracle's token-by-token
layer, on every workload (small ones in full, large ones on sampled tokens,
each token's output depending only on its own row)."""
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


def _run(M, wl, rows=None, scale_down=None):
    if scale_down:
        wl = S.Workload(**{**wl.__dict__, **scale_down})
    x, ids, w, blob, hdr, L = S.make_inputs(wl, device=DEV)
    layer = M.Layer(blob, hdr)
    ws = M.workspace(layer, wl.act, wl.T, wl.k)
    out = M.mnw_moe_forward(layer, wl.act, x, ids, w, ws=ws)
    err = M.mnw_moe_read_error(M.workspace_error_word(ws))
    assert err == 0
    if rows is None:
        rows = np.arange(wl.T, dtype=np.int32)
    want = O.moe_forward(blob.cpu().numpy(), wl.act, S.bf16_bits_np(x), ids.cpu().numpy(), w.cpu().numpy(),
                         rows=rows)
    got = out[torch.from_numpy(rows).long().to(DEV)]
    tol = REL_L2_NVFP4 if wl.act == S.ACT_NVFP4_G16 else REL_L2
    return assert_close(got, want, rel_l2=tol, what=wl.name)


def test_tiny_w8a16_full(M):
    _run(M, S.WORKLOADS["tiny_w8a16"])


@pytest.mark.parametrize("name", ["decode_w4a16", "w8a8_2048", "prefill_nvfp4", "large_w4a16", "large_bf16"])
def test_small_versions_full(M, name):
    """Each workload's formats, modes and routing at a size the oracle runs in full."""
    wl = S.WORKLOADS[name]
    small = dict(T=48, E=64, H=512, I=256 if wl.wfmt != S.FMT_NVFP4_G16 else 512)
    _run(M, wl, scale_down=small)


@pytest.mark.parametrize("wfmt,act", [(S.FMT_BF16, S.ACT_BF16), (S.FMT_INT8_G128, S.ACT_BF16),
                                      (S.FMT_INT4_G128, S.ACT_BF16), (S.FMT_INT8_G128, S.ACT_INT8_G128),
                                      (S.FMT_INT4_G128, S.ACT_INT8_G128), (S.FMT_NVFP4_G16, S.ACT_NVFP4_G16)])
@pytest.mark.parametrize("T,E,k", [(1, 8, 8), (1, 1, 1), (3, 4, 1)])
def test_degenerate_shapes(M, wfmt, act, T, E, k):
    """One token routed to every expert, a single expert, and three tokens of
    top-1 over four experts (some experts empty): every format and mode."""
    wl = S.Workload("degenerate", T, 256, E, 256, k, wfmt, act, 0.02, "uniform", 70 + T + E + k)
    _run(M, wl)


@pytest.mark.parametrize("name,nrows", [("decode_w4a16", 16), ("w8a8_2048", 8), ("prefill_nvfp4", 8),
                                        ("large_w4a16", 3), ("large_bf16", 3)])
def test_full_size_sampled(M, name, nrows):
    wl = S.WORKLOADS[name]
    rows = np.linspace(0, wl.T - 1, nrows).astype(np.int32)
    _run(M, wl, rows=rows)


@pytest.mark.parametrize("T,E,sigma", [(48, 16, 0.004), (600, 8, 0.0015)])
def test_nvfp4_layer_full_scale_range(M, T, E, sigma):
    """The NVFP4 layer with weight block scales over every non-negative finite
    E4M3 code and outer scales spread over a factor of 64 (sigma keeps |h|
    below about 2, where one BF16 ulp is inside the absolute bound)."""
    H, I, k = 512, 512, 4
    x = S.activations(T, H, seed=51 + T).to(DEV)
    ids = S.routing_uniform(T, E, k, seed=52 + T).to(DEV)
    w = S.routing_weights(T, k, seed=53 + T).to(DEV)
    blob, hdr, L = S.expert_blob(S.FMT_NVFP4_G16, E, H, I, seed=54 + T, sigma=sigma, device=DEV,
                                 nvfp4_sf_range="full")
    layer = M.Layer(blob, hdr)
    ws = M.workspace(layer, S.ACT_NVFP4_G16, T, k)
    out = M.mnw_moe_forward(layer, S.ACT_NVFP4_G16, x, ids, w, ws=ws)
    assert M.mnw_moe_read_error(M.workspace_error_word(ws)) == 0
    want = O.moe_forward(blob.cpu().numpy(), S.ACT_NVFP4_G16, S.bf16_bits_np(x), ids.cpu().numpy(),
                         w.cpu().numpy(), rows=np.arange(T, dtype=np.int32))
    assert_close(out, want, rel_l2=REL_L2_NVFP4, what="nvfp4 layer, full scale range")


@pytest.mark.parametrize("name", ["tiny_w8a16", "decode_w4a16"])
@pytest.mark.parametrize("pinned", ["all", "none", "mixed"])
def test_forward_host_buffers(M, name, pinned):
    """Host buffers: mapped page-locked ones are used in place, pageable ones
    staged; either way the same bits as the device-buffer call."""
    wl = S.WORKLOADS[name]
    x, ids, w, blob, hdr, L = S.make_inputs(wl, device=DEV)
    layer = M.Layer(blob, hdr)
    ws = M.workspace(layer, wl.act, wl.T, wl.k, host=True)
    pin = {"all": (True, True, True, True), "none": (False, False, False, False),
           "mixed": (False, True, False, True)}[pinned]  # x, ids, w, out
    host = lambda t, p: t.cpu().pin_memory() if p else t.cpu().clone()
    out_h = torch.empty((wl.T, wl.H), dtype=torch.bfloat16)
    out_h = out_h.pin_memory() if pin[3] else out_h
    M.mnw_moe_forward_host(layer, wl.act, host(x, pin[0]), host(ids, pin[1]), host(w, pin[2]), ws, out_h)
    ref = M.mnw_moe_forward(layer, wl.act, x, ids, w)
    assert torch.equal(out_h.view(torch.int16), ref.cpu().view(torch.int16))


def test_deterministic_and_bad_ids(M):
    wl = S.Workload(**{**S.WORKLOADS["decode_w4a16"].__dict__, "E": 32, "H": 512, "I": 256})
    x, ids, w, blob, hdr, L = S.make_inputs(wl, device=DEV)
    layer = M.Layer(blob, hdr)
    a = M.mnw_moe_forward(layer, wl.act, x, ids, w)
    b = M.mnw_moe_forward(layer, wl.act, x, ids, w)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    ids2 = ids.clone()
    ids2[0, 0] = 1000
    ws = M.workspace(layer, wl.act, wl.T, wl.k)
    M.mnw_moe_forward(layer, wl.act, x, ids2, w, ws=ws)
    assert M.mnw_moe_read_error(M.workspace_error_word(ws)) & M.DEVERR_BAD_EXPERT_ID


def _run_custom(M, wl, x_scale_rows=None, relative_only=False):
    """Whole layer vs the oracle on every row.  Rows far from unit scale (the
    rescaled ones, or all of them with relative_only) are held to the relative
    L2 bound row by row; the others to both stated bounds."""
    x, ids, w, blob, hdr, L = S.make_inputs(wl, device=DEV)
    big = sorted(x_scale_rows or {})
    for r in big:
        x[r] = (x[r].float() * x_scale_rows[r]).to(torch.bfloat16)
    layer = M.Layer(blob, hdr)
    ws = M.workspace(layer, wl.act, wl.T, wl.k)
    out = M.mnw_moe_forward(layer, wl.act, x, ids, w, ws=ws)
    assert M.mnw_moe_read_error(M.workspace_error_word(ws)) == 0
    want = O.moe_forward(blob.cpu().numpy(), wl.act, S.bf16_bits_np(x), ids.cpu().numpy(), w.cpu().numpy(),
                         rows=np.arange(wl.T, dtype=np.int32))
    got = out.detach().float().cpu().double().numpy()
    ref = torch.from_numpy(np.ascontiguousarray(want).view(np.int16).copy()).view(torch.bfloat16).double().numpy()
    assert np.all(np.isfinite(got)), wl.name
    per_row = [r for r in range(wl.T) if relative_only or r in big]
    for r in per_row:
        rel = np.linalg.norm(got[r] - ref[r]) / max(np.linalg.norm(ref[r]), 1e-30)
        assert rel <= REL_L2, f"{wl.name}: row {r} rel_l2={rel:.3e}"
    normal = [r for r in range(wl.T) if r not in per_row]
    if normal:
        idx = torch.tensor(normal, device=DEV)
        assert_close(out[idx], np.ascontiguousarray(want[normal]), rel_l2=REL_L2, what=wl.name)


@pytest.mark.parametrize("wfmt", [S.FMT_INT8_G128, S.FMT_INT4_G128])
def test_fp16_operand_path(M, wfmt):
    """INT weights with 64 tokens per expert: the forward path runs gate/up on
    FP16 operands (rows scaled by powers of two, weights fp16(q * s)); rows far
    outside FP16's range exercise the row factors."""
    wl = S.Workload("fp16_path", 256, 512, 16, 256, 4, wfmt, S.ACT_BF16, 0.02, "uniform", 11)
    _run_custom(M, wl, x_scale_rows={3: 3.0e5, 77: 1.0e9, 200: 1.0e-6})


def test_fp16_operand_path_falls_back_for_large_scales(M):
    """Weights whose fp16(q * s) could overflow keep the exact grouped path."""
    wl = S.Workload("big_scales", 256, 512, 16, 256, 4, S.FMT_INT8_G128, S.ACT_BF16, 5.0e4, "uniform", 12)
    _run_custom(M, wl, relative_only=True)


@pytest.mark.parametrize("wfmt", [S.FMT_INT4_G128, S.FMT_INT8_G128])
@pytest.mark.parametrize("T,E,k", [(24, 64, 2), (40, 16, 2), (200, 16, 4), (64, 8, 8)])
def test_forward_warp_tile_dependency(M, wfmt, T, E, k):
    """On the warp-MMA kernel the down launch follows the gate/up launch tile by
    tile (tile counters in the workspace instead of a wait for the whole
    launch).  Scheduling only: the layer must give the same bits as the same
    kernels launched one after the other, on repeated calls with one
    workspace, and match the oracle.  Token tiles of 8, 16 and 32 rows."""
    wl = S.Workload("warp_dep", T, 512, E, 256, k, wfmt, S.ACT_BF16, 0.02, "uniform", 31 + T)
    x, ids, w, blob, hdr, L = S.make_inputs(wl, device=DEV)
    if T == 64:
        ids[:, 0] = 3  # one crowded expert, some empty ones
    M.mnw_moe_set_gemm_path(M.PATH_WARP_MMA)
    try:
        layer = M.Layer(blob, hdr)
        ws = M.workspace(layer, wl.act, T, k)
        out1 = M.mnw_moe_forward(layer, wl.act, x, ids, w, ws=ws).clone()
        assert M.mnw_moe_read_error(M.workspace_error_word(ws)) == 0
        out2 = M.mnw_moe_forward(layer, wl.act, x, ids, w, ws=ws)
        assert M.mnw_moe_read_error(M.workspace_error_word(ws)) == 0
        assert torch.equal(out1.view(torch.int16), out2.view(torch.int16))
        # the same kernels, launched one after the other through the ABI
        off, sa, pos, _ = M.mnw_moe_permute(ids, E)
        a, f = M.mnw_moe_quantize_act(M.ACT_F16_ROWS, x, row_index=sa, index_div=k)
        gu = {S.FMT_INT4_G128: M.mnw_moe_grouped_gemm_w4a16_f16rows,
              S.FMT_INT8_G128: M.mnw_moe_grouped_gemm_w8a16_f16rows}[wfmt]
        dn = {S.FMT_INT4_G128: M.mnw_moe_grouped_gemm_w4a16, S.FMT_INT8_G128: M.mnw_moe_grouped_gemm_w8a16}[wfmt]
        h = gu(layer, M.KIND_GATE_UP, a, f, off)
        y = dn(layer, M.KIND_DOWN, h, off)
        out3 = M.mnw_moe_combine(y, pos, w)
        assert torch.equal(out1.view(torch.int16), out3.view(torch.int16))
    finally:
        M.mnw_moe_set_gemm_path(M.PATH_AUTO)
    want = O.moe_forward(blob.cpu().numpy(), wl.act, S.bf16_bits_np(x), ids.cpu().numpy(), w.cpu().numpy(),
                         rows=np.arange(T, dtype=np.int32))
    assert_close(out1, want, rel_l2=REL_L2, what="warp tile dependency")


@pytest.mark.parametrize("name", ["decode_w4a16", "w8a8_2048", "prefill_nvfp4"])
def test_forward_replays_from_a_cuda_graph(M, name):
    """The layer's launches (memset, permute, quantisers, GEMMs chained with
    programmatic dependent launch, the linked decode GEMMs, combine) captured
    once in a CUDA graph and replayed: the same bits as the eager call, replay
    after replay, with new inputs copied into the captured buffers between
    replays."""
    wl = S.WORKLOADS[name]
    if name != "decode_w4a16":
        wl = S.Workload(**{**wl.__dict__, "T": 256, "E": 64, "H": 512, "I": 512})
    x, ids, w, blob, hdr, L = S.make_inputs(wl, device=DEV)
    layer = M.Layer(blob, hdr)
    ws = M.workspace(layer, wl.act, wl.T, wl.k)
    out = torch.empty((wl.T, wl.H), dtype=torch.bfloat16, device=DEV)
    ref = M.mnw_moe_forward(layer, wl.act, x, ids, w, ws=ws, out=out).clone()  # eager (also the one-time set-up)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        M.mnw_moe_forward(layer, wl.act, x, ids, w, ws=ws, out=out)
    for _ in range(3):
        out.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert M.mnw_moe_read_error(M.workspace_error_word(ws)) == 0
        assert torch.equal(out.view(torch.int16), ref.view(torch.int16))
    # new inputs in the captured buffers
    x2 = S.activations(wl.T, wl.H, seed=wl.seed + 77).to(DEV)
    x.copy_(x2)
    g.replay()
    torch.cuda.synchronize()
    eager = M.mnw_moe_forward(layer, wl.act, x, ids, w)
    assert torch.equal(out.view(torch.int16), eager.view(torch.int16))
