"""The seeded input generator against the recipe the tests and the bench rely
on: value sets and distributions, the paged layout (a permutation of the
page pool handed to the sequences in order), the NaN poisoning of every
cached slot past a sequence's end, query positions, and determinism.  Small
cases, CPU only."""
import numpy as np
import pytest
import torch

import workloads as W


def _bf16(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).float().numpy()


def _keys(codes, dtype):
    if dtype == "bf16":
        return _bf16(codes)
    return torch.from_numpy(np.ascontiguousarray(codes)).view(torch.float8_e4m3fn).float().numpy()


@pytest.mark.parametrize("shapes", [W.TINY, W.LATENT])
def test_values_layout_and_poison(shapes):
    kw = dict(shapes)
    kw["K"] = 64
    L = np.array([130, 64, 1, 257], np.int32)
    c = W.make_case("recipe", seed=5, seq_lens=L, **kw)
    bs, B = c.bs, c.B
    # layout: pages of all sequences are one permutation of the pool, -1 past the end
    used = [c.block_table[b, :(int(L[b]) + bs - 1) // bs] for b in range(B)]
    allp = np.concatenate(used)
    assert sorted(allp.tolist()) == list(range(c.num_blocks))
    for b in range(B):
        assert np.all(c.block_table[b, len(used[b]):] == -1)
    # decode queries: one per sequence at its last position, n_elig = L
    assert np.array_equal(c.q_seq, np.arange(B)) and np.array_equal(c.q_pos, L - 1)
    assert np.array_equal(c.n_elig, L)
    # indexer operands: integers in [-8, 8] (exact in bf16 and E4M3), weights in {0..4}
    qi = _keys(c.q_idx, c.idx_dtype)
    assert np.all(qi == np.round(qi)) and qi.min() >= -8 and qi.max() <= 8
    assert set(np.unique(c.w).tolist()) <= {0.0, 1.0, 2.0, 3.0, 4.0} and c.w.dtype == np.float32
    # cached slots of the sequences: finite; slots past each sequence's end: NaN
    k = _bf16(c.k_pool)
    ki = _keys(c.kidx_pool, c.idx_dtype)
    for b in range(B):
        n = int(L[b])
        pages = used[b]
        rows = k[pages].reshape(-1, k.shape[-1])
        krow = ki[pages].reshape(-1, ki.shape[-1])
        assert np.all(np.isfinite(rows[:n])) and np.all(np.isfinite(krow[:n]))
        assert np.all(np.isnan(rows[n:])) and np.all(np.isnan(krow[n:]))
        assert np.all(krow[:n] == np.round(krow[:n])) and np.abs(krow[:n]).max() <= 8
    if c.latent:
        assert c.v_pool is c.k_pool
    # q and the K rows: bf16 of N(0, 1)
    q = _bf16(c.q).ravel()
    assert abs(q.mean()) < 0.05 and abs(q.std() - 1.0) < 0.05
    live = np.concatenate([k[used[b]].reshape(-1, k.shape[-1])[:int(L[b])] for b in range(B)])
    assert abs(live.mean()) < 0.05 and abs(live.std() - 1.0) < 0.05
    assert c.sm_scale == pytest.approx(1.0 / np.sqrt(c.Dqk), rel=1e-6)


def test_prefill_queries_and_determinism():
    tiny = {k: v for k, v in W.TINY.items() if k != "K"}
    c = W.make_case("p", seed=9, kind="prefill", T=300, K=64, **tiny)
    assert np.array_equal(c.q_pos, np.arange(300)) and np.all(c.q_seq == 0)
    assert np.array_equal(c.n_elig, np.arange(1, 301))
    c2 = W.make_case("p", seed=9, kind="prefill", T=300, K=64, **tiny)
    for f in ("q", "k_pool", "v_pool", "q_idx", "kidx_pool", "w", "block_table"):
        assert getattr(c, f).tobytes() == getattr(c2, f).tobytes(), f   # same seed, same bytes
    c3 = W.make_case("p", seed=10, kind="prefill", T=300, K=64, **tiny)
    assert not np.array_equal(c.q, c3.q)


def test_dec_batch_lengths():
    L = W.dec_batch_lens()
    assert L.shape == (32,) and L.dtype == np.int32
    assert L.min() >= 8192 and L.max() <= 32768
    assert np.array_equal(L, W.dec_batch_lens())       # seeded
    assert len(np.unique(L)) > 16                        # drawn, not constant
