"""Failure detection on the GPU, without a fault: a bounded wait that nothing
completes must give up after its limit, report MNW_DEVERR_TIMEOUT through the
caller's device error word, make the CTA's other waiting role leave through
the abort flag, and leave the context usable for the next layer call."""
import time

import pytest
import torch

import synth as S
from gpu_util import assert_close, to_np_bits

pytestmark = pytest.mark.gpu
DEV = "cuda"
MNW_DEVERR_TIMEOUT = 0x2


@pytest.fixture(scope="module")
def M():
    import quantized_moe_expert_routed_gb300 as M
    M.load()
    return M


@pytest.mark.parametrize("limit_us", [2000, 20000])
def test_wait_that_nothing_completes_times_out(M, limit_us):
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    left_early = torch.zeros(1, dtype=torch.int32, device=DEV)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    M.mnw_moe_selftest_wait_timeout(limit_us, err, left_early)
    torch.cuda.synchronize()
    elapsed = time.perf_counter() - t0
    assert int(err.item()) == MNW_DEVERR_TIMEOUT
    # the second warp left through the abort flag, not its own 2 s limit
    assert int(left_early.item()) == 1
    assert limit_us * 1e-6 <= elapsed < 1.0


def test_context_usable_after_timeout(M):
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    left_early = torch.zeros(1, dtype=torch.int32, device=DEV)
    M.mnw_moe_selftest_wait_timeout(5000, err, left_early)
    torch.cuda.synchronize()
    assert int(err.item()) == MNW_DEVERR_TIMEOUT
    # a whole layer still runs, matches a second run bit for bit, and reports no error
    wl = S.WORKLOADS["tiny_w8a16"]
    x, ids, w, blob, hdr, L = S.make_inputs(wl, device=DEV)
    layer = M.Layer(blob, hdr)
    ws = M.workspace(layer, wl.act, wl.T, wl.k)
    out1 = M.mnw_moe_forward(layer, wl.act, x, ids, w, ws=ws).clone()
    assert M.mnw_moe_read_error(M.workspace_error_word(ws)) == 0
    out2 = M.mnw_moe_forward(layer, wl.act, x, ids, w, ws=ws)
    assert (to_np_bits(out1) == to_np_bits(out2)).all()


def test_selftest_rejects_bad_limits(M):
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    with pytest.raises(RuntimeError):
        M.mnw_moe_selftest_wait_timeout(0, err, err)
    with pytest.raises(RuntimeError):
        M.mnw_moe_selftest_wait_timeout(2_000_000, err, err)


def test_counter_wait_times_out_without_fault(M):
    """The wait a dependent launch does on a token-tile counter: a counter that
    nothing raises ends in MNW_DEVERR_TIMEOUT after the limit, a satisfied one
    returns at once, and the context stays usable."""
    counter = torch.zeros(1, dtype=torch.int32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    t0 = time.perf_counter()
    M.mnw_moe_selftest_counter_timeout(20000, counter, 1, err)
    torch.cuda.synchronize()
    waited = time.perf_counter() - t0
    assert int(err.item()) == MNW_DEVERR_TIMEOUT
    assert waited >= 0.02
    counter.fill_(3)
    err.zero_()
    M.mnw_moe_selftest_counter_timeout(1000000, counter, 3, err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    with pytest.raises(M.MnwError):
        M.mnw_moe_selftest_counter_timeout(0, counter, 1, err)
