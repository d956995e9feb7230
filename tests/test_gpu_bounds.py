"""GPU tests of the block-level key bounds and the bounded decode indexer
(include/dsa.h: dsa_index_bounds_update, dsa_index_score_bounded) against the
oracle.

The bounded indexer must leave the top-K unchanged: its index sets are
compared with the oracle's exactly; every score it computes equals the
oracle's; every tile it leaves out is -inf and holds no position whose exact
score reaches the row's K-th largest.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from workloads import device as wdev
from gpu_common import code, lib, need_gpu, to_dev

pytestmark = pytest.mark.gpu

LAT = dict(Hq=64, Dqk=576, Dv=512, latent=True, H_i=64, D_i=128, idx_dtype="fp8")
TINY = dict(Hq=16, Dqk=128, Dv=128, latent=False, H_i=4, D_i=64, idx_dtype="bf16")
TILE = 128


def _codes(t):
    """Device key pool / bounds -> numpy codes (uint16 for bf16, uint8 for E4M3)."""
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).cpu().numpy().view(np.uint16)
    return t.cpu().numpy()


def _bounds(dsa, case, d, lay, kb=None, seq=None, pos=None):
    if kb is None:
        kb = torch.zeros((case.num_blocks, 2, case.D_i), dtype=d.kidx_pool.dtype, device="cuda")
    ws = dsa.workspace(dsa.index_bounds_update_workspace_size())
    dsa.index_bounds_update(lay, d.kidx_pool, kb, ws, seq=seq, pos=pos)
    torch.cuda.synchronize()
    assert dsa.get_status(ws) == 0
    return kb


def _assert_bounds_equal(kb, case, kidx_pool, seq_lens):
    ref, cached = oracle.page_bounds(case.block_table, seq_lens, case.bs, case.num_blocks,
                                     kidx_pool, code(case))
    got = _codes(kb)
    np.testing.assert_array_equal(got[cached], ref[cached])


def _bounded(dsa, case, d, lay, kb):
    """Bounded scores, their top-K, and (tiles left out, tiles bounded)."""
    ld = int(case.seq_lens.max())
    ld = (ld + 3) // 4 * 4
    scores = torch.empty((case.B, ld), dtype=torch.float32, device="cuda")
    ws = dsa.workspace(dsa.index_score_bounded_workspace_size(case.B, case.H_i, case.D_i, ld,
                                                              case.K))
    dsa.index_score_bounded(lay, d.q_idx, d.w, d.kidx_pool, kb, case.K, scores, ws)
    idx = torch.empty((case.B, case.K), dtype=torch.int32, device="cuda")
    wt = dsa.workspace(dsa.topk_workspace_size(case.B, ld, case.K))
    dsa.topk(scores, d.n_elig, case.K, idx, wt)
    torch.cuda.synchronize()
    assert dsa.get_status(ws) == 0 and dsa.get_status(wt) == 0
    return scores.cpu().numpy(), idx.cpu().numpy(), dsa.index_bounded_stats(ws)


def _check(case, kidx_pool, s, idx):
    """Exact selection; computed scores exact; left-out tiles whole, -inf, and
    below the row's K-th largest exact score.  Returns tiles left out."""
    s_ref = oracle.index_score(case.block_table, case.seq_lens, case.bs, case.num_blocks,
                               case.q_seq, case.q_pos, case.q_idx, case.w, kidx_pool, code(case),
                               s.shape[1])
    np.testing.assert_array_equal(idx, oracle.topk(s_ref, case.n_elig, case.K))
    left = 0
    for b in range(case.B):
        n = int(case.n_elig[b])
        row, ref = s[b, :n], s_ref[b, :n]
        out = np.isneginf(row) & np.isfinite(ref)
        np.testing.assert_array_equal(row[~out], ref[~out], err_msg=f"row {b}")
        tiles = np.unique(np.nonzero(out)[0] // TILE)
        for t in tiles:
            assert out[t * TILE:min(n, (t + 1) * TILE)].all(), f"row {b}: tile {t} partly left out"
        if len(tiles):
            kth = np.sort(ref)[::-1][case.K - 1]
            assert ref[out].max() < kth, f"row {b}: a left-out score reaches the K-th largest"
        left += len(tiles)
    return left


def _cold_pages(case, hot_tiles, seed):
    """The key pool with every cached page set to zero keys except those of a
    few 128-position tiles per sequence: the cold pages' bounds are 0, below
    the hot tiles' scores.  (With at least K hot positions, in whole tiles, the
    first scored tiles set a positive threshold; with fewer, the row's K-th
    largest score is 0, every cold position ties at it, and nothing may be
    left out.)"""
    rng = np.random.default_rng(seed)
    kp = case.kidx_pool.copy()
    zero = W.encode_int(np.zeros(1, np.int64), "bf16" if case.idx_dtype == "bf16" else "fp8")[0]
    for b in range(case.B):
        P = (int(case.seq_lens[b]) + case.bs - 1) // case.bs
        T = (P + 1) // 2
        hot = set(rng.choice(T, size=min(hot_tiles, T), replace=False).tolist())
        for j in range(P):
            if j // 2 not in hot:
                kp[case.block_table[b, j]] = zero
    return kp


@pytest.mark.parametrize("shapes", [LAT, TINY], ids=["fp8-64x128", "bf16-4x64"])
def test_bounds_of_every_page_then_after_appends(shapes):
    """Bounds of every cached page, byte-exact; then one row appended to each
    sequence (into a partly filled page) and only the touched pages recomputed:
    every cached page matches the oracle on the new cache."""
    need_gpu()
    dsa = lib()
    c = W.make_case("bounds", seed=801, seq_lens=(1000, 3001, 77), K=64, **shapes)
    d = wdev.upload(c, "cuda")
    lay = wdev.layout_of(c, d)
    kb = _bounds(dsa, c, d, lay)
    _assert_bounds_equal(kb, c, c.kidx_pool, c.seq_lens)
    # append: position L_b of every sequence (all inside their last page)
    L = c.seq_lens.astype(np.int64)
    assert np.all(L % c.bs != 0)
    rng = np.random.default_rng(802)
    new = W.encode_int(rng.integers(-8, 9, size=(c.B, c.D_i)),
                       "bf16" if c.idx_dtype == "bf16" else "fp8")
    seq = np.arange(c.B, dtype=np.int32)
    pos = L.astype(np.int32)
    lens2 = (L + 1).astype(np.int32)
    lay2 = dsa.PagedLayout(d.block_table, to_dev(lens2), c.bs, c.num_blocks, int(lens2.max()))
    ws = dsa.workspace(dsa.cache_write_workspace_size())
    dsa.cache_write(lay2, to_dev(seq), to_dev(pos), ws, kidx_new=to_dev(new), kidx_pool=d.kidx_pool)
    _bounds(dsa, c, d, lay2, kb=kb, seq=to_dev(seq), pos=to_dev(pos))
    pool2, bad = oracle.cache_write(c.block_table, c.bs, c.num_blocks, seq, pos, new, c.kidx_pool)
    assert not bad
    np.testing.assert_array_equal(_codes(d.kidx_pool), pool2)
    _assert_bounds_equal(kb, c, pool2, lens2)


def test_bounded_indexer_on_random_keys_selects_exactly():
    """Keys drawn per position (the workloads' distribution): every page's bound
    covers the row's largest scores, so little or nothing is left out; the
    selection is exact either way."""
    need_gpu()
    dsa = lib()
    c = W.make_case("bounded-random", seed=811, seq_lens=(9000, 3000, 20000, 700), K=2048, **LAT)
    d = wdev.upload(c, "cuda")
    lay = wdev.layout_of(c, d)
    kb = _bounds(dsa, c, d, lay)
    s, idx, (skipped, total) = _bounded(dsa, c, d, lay, kb)
    left = _check(c, c.kidx_pool, s, idx)
    assert left == skipped
    assert total == sum((int(L) + TILE - 1) // TILE for L in c.seq_lens)


@pytest.mark.parametrize("shapes,lens,K,hot", [
    (LAT, (9000, 5000, 12000), 512, 6),
    (TINY, (4096, 1500), 256, 3),
], ids=["fp8-64x128", "bf16-4x64"])
def test_bounded_indexer_leaves_out_cold_tiles_and_selects_exactly(shapes, lens, K, hot):
    """A cache whose pages differ: all but a few tiles per sequence hold zero
    keys.  Their tiles are left out (keys not read, scores -inf) and the
    selection is still exact."""
    need_gpu()
    dsa = lib()
    c = W.make_case("bounded-cold", seed=821, seq_lens=lens, K=K, **shapes)
    c.kidx_pool = _cold_pages(c, hot, 822)
    d = wdev.upload(c, "cuda")
    lay = wdev.layout_of(c, d)
    kb = _bounds(dsa, c, d, lay)
    s, idx, (skipped, total) = _bounded(dsa, c, d, lay, kb)
    left = _check(c, c.kidx_pool, s, idx)
    assert left == skipped
    assert skipped >= total // 2, (skipped, total)


def test_bounded_indexer_short_sequences_leave_nothing_out():
    """Sequences with at most K positions: every position is selected, nothing
    may be left out."""
    need_gpu()
    dsa = lib()
    c = W.make_case("bounded-short", seed=831, seq_lens=(100, 2048, 1), K=2048, **LAT)
    c.kidx_pool = _cold_pages(c, 1, 832)
    d = wdev.upload(c, "cuda")
    lay = wdev.layout_of(c, d)
    kb = _bounds(dsa, c, d, lay)
    s, idx, (skipped, total) = _bounded(dsa, c, d, lay, kb)
    assert _check(c, c.kidx_pool, s, idx) == 0 and skipped == 0
