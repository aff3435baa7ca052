"""GPU routing fused with the permutation (mnw_moe_route) and the layer with
GPU routing (mnw_moe_forward_routed), against the oracle's router and layer.

The expert choice is an integer decided by floating point: the kernel's FP32
logits and the oracle's FP64 ones may differ in their last bits, so ids are
compared with the oracle exactly wherever the oracle's logits leave a margin
wider than the FP32 accumulation bound between neighbours, and everywhere
they must be the top-k of the kernel's own logits under the stated rule
(largest first, lower index on ties).  The permutation of the chosen ids is
compared bit for bit."""
import math

import numpy as np
import pytest
import torch

import oracle as O
import synth as S
from gpu_util import REL_L2, REL_L2_NVFP4, assert_close

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def M():
    import quantized_moe_expert_routed_gb300 as M
    M.load()
    return M


def _f32_bound(x, wr):
    """Per-logit bound on FP32 accumulation error: H * 2^-24 * sum_h |x_h w_h|."""
    xa = x.double().abs().cpu()
    wa = wr.double().abs().cpu()
    return (xa @ wa.T).numpy() * x.shape[1] * 2.0 ** -24


def _topk_rule(logits_row, k):
    return sorted(range(len(logits_row)), key=lambda e: (-logits_row[e], e))[:k]


def _check_route(M, x, wr, k, scratch=None):
    T, H = x.shape
    E = wr.shape[0]
    ids, w, off, sa, pos, logits = M.mnw_moe_route(x, wr, k, scratch=scratch)
    ids_c, w_c, lg = ids.cpu().numpy(), w.cpu().numpy(), logits.cpu().numpy().astype(np.float64)
    o_ids, o_w, o_lg = O.route(S.bf16_bits_np(x), S.bf16_bits_np(wr), k)
    bound = _f32_bound(x, wr)
    diff = np.abs(lg - o_lg)
    assert np.all(diff <= bound + 1e-30), "logits outside the FP32 accumulation bound"
    margin = 2 * diff.max()  # no two logits closer than this can have swapped ranks
    exact = 0
    for t in range(T):
        # the kernel's choice is the rule applied to its own logits
        assert ids_c[t].tolist() == _topk_rule(lg[t].tolist(), k), f"token {t}"
        # and its weights are the softmax of its logits
        l = lg[t][ids_c[t]]
        p = np.exp(l - l[0])
        assert np.allclose(w_c[t], p / p.sum(), rtol=2e-6, atol=1e-7), f"token {t} weights"
        # where the oracle's ranking has margins wider than twice the bound, the same ids
        order = np.array(_topk_rule(o_lg[t].tolist(), min(k + 1, E)))
        gaps = -np.diff(o_lg[t][order])
        if np.all(gaps > margin):
            assert ids_c[t].tolist() == o_ids[t].tolist(), f"token {t}"
            assert np.allclose(w_c[t], o_w[t], rtol=1e-4, atol=1e-6)
            exact += 1
    # the permutation of the chosen ids, bit for bit
    o_off, o_sa, o_pos, dropped = O.permute(ids_c, E)
    assert dropped == 0
    assert np.array_equal(off.cpu().numpy(), o_off)
    assert np.array_equal(sa.cpu().numpy(), o_sa)
    assert np.array_equal(pos.cpu().numpy(), o_pos)
    return exact, ids, w


# (T, H, E, k): one 32-token decode block, the 256-token decode batch, a
# ragged batch, tiny, one above 4096 assignments (the permutation then runs
# in its own launches), 1024 experts, and batches of 1024 tokens or more
# (32-token tiles), with up to 256 and with more than 256 experts
@pytest.mark.parametrize("T,H,E,k", [(32, 2048, 256, 8), (256, 2048, 256, 8), (300, 512, 64, 4), (5, 256, 8, 2),
                                     (700, 512, 256, 8), (64, 1024, 1024, 8), (17, 128, 40, 1),
                                     (1100, 512, 256, 4), (1030, 256, 600, 2), (1024, 128, 16, 2)])
def test_route_matches_oracle(M, T, H, E, k):
    x = S.activations(T, H, seed=T + E).to(DEV)
    wr = S.router_weights(E, H, seed=H + k).to(DEV)
    exact, _, _ = _check_route(M, x, wr, k)
    assert exact >= 0.9 * T  # almost every token has a clear ranking


def test_route_ties_and_repeated_calls(M):
    """Experts with identical router rows have identical FP32 logits: the lower
    index comes first, as in the oracle.  The arrival counters return to zero,
    so a second call on the same scratch gives the same result."""
    T, H, E, k = 48, 512, 32, 6
    wr = S.router_weights(E, H, seed=3)
    for dup, src in ((5, 2), (9, 2), (20, 11), (21, 11), (31, 0)):
        wr[dup] = wr[src]
    x = S.activations(T, H, seed=4).to(DEV)
    wr = wr.to(DEV)
    scratch = torch.zeros(M.load().mnw_moe_route_scratch_size(T, E) + 256, dtype=torch.uint8, device=DEV)
    _, ids1, w1 = _check_route(M, x, wr, k, scratch=scratch)
    _, ids2, w2 = _check_route(M, x, wr, k, scratch=scratch)
    assert torch.equal(ids1, ids2) and torch.equal(w1, w2)
    o_ids, _, _ = O.route(S.bf16_bits_np(x), S.bf16_bits_np(wr), k)
    lg = M.mnw_moe_route(x, wr, k)[5].cpu().numpy()
    for t in range(T):
        for a, b in ((2, 5), (2, 9), (11, 20), (11, 21), (0, 31)):
            assert lg[t][a] == lg[t][b]
            ia, ib = ids1[t].tolist(), ids1[t].tolist()
            if a in ia and b in ib:
                assert ia.index(a) < ib.index(b)


@pytest.mark.parametrize("name", ["decode_w4a16", "w8a8_2048", "prefill_nvfp4", "large_bf16", "tiny_w8a16"])
def test_forward_routed_matches_forward_on_the_routers_choice(M, name):
    """The layer with GPU routing: ids_out / w_out are the router's choice, and
    the output is the same bits as mnw_moe_forward on that choice, within the
    layer tolerance of the oracle."""
    wl = S.WORKLOADS[name]
    wl = S.Workload(**{**wl.__dict__, "T": min(wl.T, 96), "E": min(wl.E, 64), "H": min(wl.H, 512),
                       "I": min(wl.I, 512 if wl.wfmt == S.FMT_NVFP4_G16 else 256)})
    x, _, _, blob, hdr, L = S.make_inputs(wl, device=DEV)
    wr = S.router_weights(wl.E, wl.H, seed=wl.seed + 7).to(DEV)
    layer = M.Layer(blob, hdr)
    out, ids, w = M.mnw_moe_forward_routed(layer, wl.act, x, wr, wl.k)
    r_ids, r_w = M.mnw_moe_route(x, wr, wl.k)[:2]
    assert torch.equal(ids, r_ids) and torch.equal(w, r_w)
    ref = M.mnw_moe_forward(layer, wl.act, x, ids, w)
    assert torch.equal(out.view(torch.int16), ref.view(torch.int16))
    want = O.moe_forward(blob.cpu().numpy(), wl.act, S.bf16_bits_np(x), ids.cpu().numpy(), w.cpu().numpy(),
                         rows=np.arange(wl.T, dtype=np.int32))
    tol = REL_L2_NVFP4 if wl.act == S.ACT_NVFP4_G16 else REL_L2
    assert_close(out, want, rel_l2=tol, what=f"{name} routed")


@pytest.mark.parametrize("name", ["decode_w4a16", "prefill_nvfp4"])
def test_host_routing_comparison_path(M, name):
    """Host routing: the same logits, the same rule and the same permutation
    computed on the host, so ids and the permutation agree with GPU routing
    exactly and the weights to the last FP32 bits of exp."""
    wl = S.WORKLOADS[name]
    wl = S.Workload(**{**wl.__dict__, "T": 300, "E": 64, "H": 512,
                       "I": 512 if wl.wfmt == S.FMT_NVFP4_G16 else 256})
    x, _, _, blob, hdr, L = S.make_inputs(wl, device=DEV)
    wr = S.router_weights(wl.E, wl.H, seed=wl.seed + 9).to(DEV)
    layer = M.Layer(blob, hdr)
    out_gpu, ids_gpu, w_gpu = M.mnw_moe_forward_routed(layer, wl.act, x, wr, wl.k)
    M.mnw_moe_set_host_routing(True)
    try:
        out_host, ids_host, w_host = M.mnw_moe_forward_routed(layer, wl.act, x, wr, wl.k)
    finally:
        M.mnw_moe_set_host_routing(False)
    assert torch.equal(ids_gpu, ids_host)
    assert torch.allclose(w_gpu, w_host, rtol=1e-6, atol=1e-7)
    tol = REL_L2_NVFP4 if wl.act == S.ACT_NVFP4_G16 else REL_L2
    want = O.moe_forward(blob.cpu().numpy(), wl.act, S.bf16_bits_np(x), ids_host.cpu().numpy(),
                         w_host.cpu().numpy(), rows=np.arange(wl.T, dtype=np.int32))
    assert_close(out_host, want, rel_l2=tol, what=f"{name} host routing")
    assert (out_host.double() - out_gpu.double()).norm() <= 1e-3 * out_gpu.double().norm()
