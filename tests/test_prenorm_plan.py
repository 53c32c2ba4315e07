"""Launch plan of the Pre-LN forward, from the host logic alone (CPU): how
many heads share a chunk of row statistics, whether cluster pairs share the
prologue, how many chunks each CTA's prologue covers."""
import numpy as np
import pytest

import masked_head_attention_gb300 as mha


def test_prenorm_workload_plan():
    # B32 H16 Lq2048 Lk2048 D64 on 152 SMs: four heads per chunk, 1024 chunks,
    # 6.7 per CTA, all in the prologue's table, shared by cluster pairs.
    pl = mha.plan_prenorm(32, 16, 2048, 2048, 64, 152)
    assert pl == dict(G=4, n_hg=4, cs=2, pre_chunks=7, grid=152, n_chunks=1024)
    # Statistics from the caller's array (the no-allocation entry point): the
    # finest chunks, no prologue, no clusters.
    pl = mha.plan_prenorm(32, 16, 2048, 2048, 64, 152, stats_given=True)
    assert pl == dict(G=1, n_hg=16, cs=1, pre_chunks=0, grid=152, n_chunks=4096)


def test_small_problem_clamps_the_grid_and_pairs():
    pl = mha.plan_prenorm(1, 2, 130, 150, 64, 152)
    assert pl == dict(G=1, n_hg=2, cs=2, pre_chunks=1, grid=2, n_chunks=2)


def test_no_prologue_at_d128_and_no_pairs_on_odd_grids():
    pl = mha.plan_prenorm(4, 8, 1024, 512, 128, 152)
    assert pl["pre_chunks"] == 0 and pl["cs"] == 1
    pl = mha.plan_prenorm(32, 16, 2048, 2048, 64, 151)
    assert pl["cs"] == 1 and pl["grid"] == 151
    # One CTA walking more chunks than the table holds: the first 32 in the
    # prologue, the rest at their chunk starts.
    pl = mha.plan_prenorm(1, 1, 40 * 256 - 70, 100, 64, 1)
    assert pl == dict(G=1, n_hg=1, cs=1, pre_chunks=32, grid=1, n_chunks=40)


@pytest.mark.parametrize("seed", range(8))
def test_plan_invariants(seed):
    r = np.random.default_rng(seed)
    for _ in range(200):
        B = int(r.integers(1, 65))
        H = int(r.choice([1, 2, 3, 4, 6, 8, 12, 16, 32]))
        D = int(r.choice([64, 128]))
        Lq = int(r.integers(1, 9000))
        Lk = int(r.integers(0, 9000))
        grid = int(r.choice([1, 2, 3, 76, 151, 152]))
        given = bool(r.random() < 0.3)
        pl = mha.plan_prenorm(B, H, Lq, Lk, D, grid, stats_given=given)
        n_items = B * H * ((Lq + 255) // 256)
        what = (B, H, Lq, Lk, D, grid, given, pl)
        assert H % pl["G"] == 0 and pl["n_hg"] * pl["G"] == H, what
        assert pl["n_chunks"] * pl["G"] == n_items, what
        assert 1 <= pl["grid"] <= min(grid, pl["n_chunks"]), what
        per_cta = -(-pl["n_chunks"] // pl["grid"])
        assert 0 <= pl["pre_chunks"] <= min(per_cta, 32), what
        if given or D == 128:
            assert pl["pre_chunks"] == 0 and pl["cs"] == 1, what
        if pl["cs"] == 2:
            # Every chunk of every CTA is in the table, and the pair shares
            # whole row blocks.
            assert pl["pre_chunks"] == per_cta and pl["n_hg"] % 2 == 0 and pl["grid"] % 2 == 0, what
        else:
            assert pl["cs"] == 1, what


def test_plan_rejects_bad_sizes():
    for args in ((0, 1, 1, 1, 64, 1), (1, 1, 1, 1, 96, 1), (1, 1, 1, 1, 64, 0), (1, 0, 5, 5, 64, 4)):
        with pytest.raises(mha.MhaError):
            mha.plan_prenorm(*args)
