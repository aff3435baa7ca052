"""The allocation-free entry point (mnw_moe_forward_static), for callers that
cannot allocate device memory: it runs the same kernels as mnw_moe_forward
with the intermediates in an array compiled into the library, so its output
must be the same bits as mnw_moe_forward with a caller workspace, call after
call, and device memory must not change while it runs.  Collected last on
purpose."""
import ctypes

import pytest
import torch

import synth as S

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def M():
    import quantized_moe_expert_routed_gb300 as M
    M.load()
    return M


# the two workloads that fit, plus small A8 and A4 layers (their workspace
# layouts hold INT8 / NVFP4 codes and scales)
CASES = {
    "tiny_w8a16": S.WORKLOADS["tiny_w8a16"],
    "decode_w4a16": S.WORKLOADS["decode_w4a16"],
    "small_w8a8": S.Workload("small_w8a8", 64, 512, 16, 256, 4, S.FMT_INT8_G128, S.ACT_INT8_G128, 0.02, "uniform", 61,
                             outlier_p=0.01),
    "small_nvfp4": S.Workload("small_nvfp4", 64, 512, 16, 512, 4, S.FMT_NVFP4_G16, S.ACT_NVFP4_G16, 0.02, "zipf", 62),
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_static_forward_matches_workspace_forward_twice(M, name):
    wl = CASES[name]
    x, ids, w, blob, hdr, L = S.make_inputs(wl, device=DEV)
    layer = M.Layer(blob, hdr)
    assert M.mnw_moe_workspace_size(layer, wl.act, wl.T, wl.k) <= M.STATIC_WS_BYTES
    ref = M.mnw_moe_forward(layer, wl.act, x, ids, w)
    err = torch.full((1,), -1, dtype=torch.int32, device=DEV)
    outs = [torch.full_like(ref, float("nan")) for _ in range(3)]
    M.mnw_moe_forward_static(layer, wl.act, x, ids, w, out=outs[0], err=err)  # first call: one-time set-up
    torch.cuda.synchronize()
    free_before = torch.cuda.mem_get_info()[0]
    for call in (1, 2):
        M.mnw_moe_forward_static(layer, wl.act, x, ids, w, out=outs[call], err=err)
        torch.cuda.synchronize()
        assert int(err.item()) == 0, f"call {call}: device error word {int(err.item()):#x}"
    assert torch.cuda.mem_get_info()[0] == free_before, "device memory changed during the static calls"
    for call in range(3):
        assert torch.equal(outs[call].view(torch.int16), ref.view(torch.int16)), f"{name} static call {call}"


def test_static_forward_rejects_oversized_requests(M):
    wl = S.WORKLOADS["tiny_w8a16"]
    x, ids, w, blob, hdr, L = S.make_inputs(wl, device=DEV)
    layer = M.Layer(blob, hdr)
    T = 100000  # needs far more than the built-in array holds
    assert M.mnw_moe_workspace_size(layer, wl.act, T, wl.k) > M.STATIC_WS_BYTES
    lib = M.load()
    rc = lib.mnw_moe_forward_static(layer.handle, wl.act, ctypes.c_void_p(x.data_ptr()),
                                    ctypes.c_void_p(ids.data_ptr()), ctypes.c_void_p(w.data_ptr()), T, wl.k,
                                    ctypes.c_void_p(x.data_ptr()), None, None)
    assert rc == 4  # MNW_E_WORKSPACE_TOO_SMALL, nothing enqueued


def test_static_forward_zero_tokens_clears_error_word(M):
    wl = S.WORKLOADS["tiny_w8a16"]
    x, ids, w, blob, hdr, L = S.make_inputs(wl, device=DEV)
    layer = M.Layer(blob, hdr)
    err = torch.full((1,), -1, dtype=torch.int32, device=DEV)
    lib = M.load()
    rc = lib.mnw_moe_forward_static(layer.handle, wl.act, ctypes.c_void_p(x.data_ptr()),
                                    ctypes.c_void_p(ids.data_ptr()), ctypes.c_void_p(w.data_ptr()), 0, wl.k,
                                    ctypes.c_void_p(x.data_ptr()), ctypes.c_void_p(err.data_ptr()),
                                    ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    torch.cuda.synchronize()
    assert rc == 0 and int(err.item()) == 0
