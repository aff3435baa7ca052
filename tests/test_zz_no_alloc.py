"""The allocation-free entry point (mnw_moe_forward_static), for callers that
cannot allocate device memory: it must give the same layer output as
mnw_moe_forward with a caller workspace, call after call, while the library
allocates nothing.  Collected last on purpose."""
import ctypes

import pytest
import torch

import synth as S
from gpu_util import REL_L2, assert_close, to_np_bits

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def M():
    import quantized_moe_expert_routed_gb300 as M
    M.load()
    return M


@pytest.mark.parametrize("name", ["tiny_w8a16", "decode_w4a16"])
def test_static_forward_matches_workspace_forward_twice(M, name):
    wl = S.WORKLOADS[name]
    x, ids, w, blob, hdr, L = S.make_inputs(wl, device=DEV)
    layer = M.Layer(blob, hdr)
    assert M.mnw_moe_workspace_size(layer, wl.act, wl.T, wl.k) <= M.STATIC_WS_BYTES
    ref = M.mnw_moe_forward(layer, wl.act, x, ids, w)
    err = torch.full((1,), -1, dtype=torch.int32, device=DEV)
    for call in range(2):
        out = torch.full_like(ref, float("nan"))
        M.mnw_moe_forward_static(layer, wl.act, x, ids, w, out=out, err=err)
        torch.cuda.synchronize()
        assert int(err.item()) == 0, f"call {call}: device error word {int(err.item()):#x}"
        assert_close(out, to_np_bits(ref), rel_l2=REL_L2, what=f"{name} static call {call}")


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
