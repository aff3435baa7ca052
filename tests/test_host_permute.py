"""The library's host-side permutation (the host-routing comparison path):
no GPU, bit-exact against the oracle's permutation on the routing patterns
of the workloads, dropped and duplicate ids, and the edge sizes."""
import numpy as np
import pytest

import oracle as O
import synth as S


@pytest.fixture(scope="module")
def M():
    import quantized_moe_expert_routed_gb300 as M
    M.load()
    return M


def _check(M, ids, E):
    off, sa, pos, dropped = M.mnw_moe_permute_host(ids, E)
    o_off, o_sa, o_pos, o_dropped = O.permute(ids, E)
    assert np.array_equal(off, o_off)
    assert np.array_equal(sa, o_sa)
    assert np.array_equal(pos, o_pos)
    assert dropped == o_dropped


@pytest.mark.parametrize("T,k,E", [(1, 1, 1), (37, 2, 8), (256, 8, 256), (2048, 8, 256), (8192, 8, 256),
                                   (33, 3, 1024), (1030, 9, 256)])
def test_matches_oracle_uniform(M, T, k, E):
    _check(M, S.routing_uniform(T, E, k, seed=T + E).numpy(), E)


@pytest.mark.parametrize("routing", ["zipf", "hot_cold"])
def test_matches_oracle_skewed_and_bad_ids(M, routing):
    E = 256
    gen = S.routing_zipf if routing == "zipf" else S.routing_hot_cold
    ids = gen(512, E, 8, seed=3).numpy().copy()
    _check(M, ids, E)
    ids[::7, 0] = E + 5    # out of range: dropped
    ids[3, -1] = -2        # negative: dropped
    ids[10, :] = ids[10, 0]  # duplicates count as separate assignments
    _check(M, ids, E)


def test_all_dropped_and_single_expert(M):
    _check(M, np.full((16, 4), 9, np.int32), 4)   # every id out of range
    _check(M, np.zeros((16, 4), np.int32), 1)     # one expert takes everything


def test_argument_checks(M):
    with pytest.raises(M.MnwError):
        M.mnw_moe_permute_host(np.zeros((4, 40), np.int32), 64)   # k > 32
    with pytest.raises(M.MnwError):
        M.mnw_moe_permute_host(np.zeros((4, 2), np.int32), 2000)  # E > 1024
    off, sa, pos, dropped = M.mnw_moe_permute_host(np.zeros((0, 2), np.int32), 8)  # T = 0: no-op
    assert dropped == 0
