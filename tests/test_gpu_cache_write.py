"""GPU parity of dsa_cache_write (through the C ABI) against the oracle's
cache write, and the write-then-gather alignment of the paged layout.

Bar: every byte of every pool equal to the oracle's; the pipeline run over a
cache the kernel wrote meets the usual parity bar against the oracle run over
the original cache.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import workloads as W
from gpu_common import (DevicePipeline, assert_out_close, assert_scores_equal, fresh_layout, lib,
                        logical_rows, need_gpu, oracle_attn, oracle_scores, to_dev, to_host)
from workloads import device as wdev

pytestmark = pytest.mark.gpu

LAT_SHAPES = dict(Hq=64, Dqk=576, Dv=512, latent=True, H_i=64, D_i=128, idx_dtype="fp8")
TINY_SHAPES = dict(Hq=16, Dqk=128, Dv=128, latent=False, H_i=4, D_i=64, idx_dtype="bf16")


def _write(dsa, layout, seq, pos, kv_rows, kv_pool, ki_rows, ki_pool, ws):
    dsa.cache_write(layout, to_dev(seq), to_dev(pos), ws, kv_new=kv_rows, kv_pool=kv_pool,
                    kidx_new=ki_rows, kidx_pool=ki_pool)


@pytest.mark.parametrize("shapes,lens,stride_pad", [(LAT_SHAPES, (300,), 0),
                                                     (LAT_SHAPES, (1, 64, 65, 700), 64),
                                                     (TINY_SHAPES, (129, 1000, 33), 8)])
def test_cache_write_bulk_prefill_is_byte_exact(shapes, lens, stride_pad):
    """A whole prompt per sequence into pages of a fresh table, in a shuffled
    row order, K/V rows into a pool whose rows may be wider than the row."""
    need_gpu()
    dsa = lib()
    c = W.make_case("cw", seed=500 + len(lens), seq_lens=lens, K=64, **shapes)
    bt2, nb2 = fresh_layout(c, 17 + len(lens), 3)
    rng = np.random.default_rng(23)
    seq = np.concatenate([np.full(int(L), b, np.int32) for b, L in enumerate(c.seq_lens)])
    pos = np.concatenate([np.arange(int(L), dtype=np.int32) for L in c.seq_lens])
    order = rng.permutation(seq.shape[0])
    seq, pos = seq[order], pos[order]
    kv_rows = np.concatenate([logical_rows(c, c.k_pool, b, int(L)) for b, L in enumerate(c.seq_lens)])
    ki_rows = np.concatenate([logical_rows(c, c.kidx_pool, b, int(L))
                              for b, L in enumerate(c.seq_lens)])
    kv_rows, ki_rows = kv_rows[order], ki_rows[order]
    W_ = c.Dkv + stride_pad
    kv0 = rng.integers(0, 1 << 16, size=(nb2, c.bs, W_), dtype=np.uint16)
    ki0 = rng.integers(0, 1 << 16, size=(nb2, c.bs, c.D_i)).astype(c.kidx_pool.dtype)
    kv_want, bad1 = oracle.cache_write(bt2, c.bs, nb2, seq, pos, kv_rows, kv0)
    ki_want, bad2 = oracle.cache_write(bt2, c.bs, nb2, seq, pos, ki_rows, ki0)
    assert not bad1 and not bad2

    lay = dsa.PagedLayout(to_dev(bt2), to_dev(c.seq_lens), c.bs, nb2, c.max_len)
    kv_pool, ki_pool = to_dev(kv0), to_dev(ki0)
    ws = dsa.workspace(dsa.cache_write_workspace_size())
    n0 = dsa.launch_count()
    _write(dsa, lay, seq, pos, to_dev(kv_rows), kv_pool, to_dev(ki_rows), ki_pool, ws)
    assert dsa.launch_count() == n0 + 1
    torch.cuda.synchronize()
    np.testing.assert_array_equal(to_host(kv_pool, kv0), kv_want)
    np.testing.assert_array_equal(to_host(ki_pool, ki0), ki_want)
    assert dsa.get_status(ws) == 0


def test_cache_write_decode_append_then_pipeline_matches_oracle():
    """Decode append: each sequence's newest row is missing from the cache
    (pages hold garbage there); the kernel writes it, then the three stages
    run over the written cache and must match the oracle on the original."""
    need_gpu()
    dsa = lib()
    c = W.make_case("cw-append", seed=510, seq_lens=(100, 2048, 2049, 5000, 8191), K=2048,
                    **LAT_SHAPES)
    last = (c.seq_lens - 1).astype(np.int32)
    seq = np.arange(c.B, dtype=np.int32)
    pages = c.block_table[seq, last // c.bs]
    kv_rows = c.k_pool[pages, last % c.bs].copy()
    ki_rows = c.kidx_pool[pages, last % c.bs].copy()
    g = DevicePipeline(c)
    # overwrite the newest rows with garbage on the device, then append them
    garbage_kv = torch.full((c.B, c.Dkv), float("nan"), dtype=torch.bfloat16, device="cuda")
    garbage_ki = torch.full((c.B, c.D_i), 0x7F, dtype=torch.uint8, device="cuda")
    ws = dsa.workspace(dsa.cache_write_workspace_size())
    _write(dsa, g.layout, seq, last, garbage_kv, g.d.k_pool, garbage_ki, g.d.kidx_pool, ws)
    torch.cuda.synchronize()
    assert not np.array_equal(to_host(g.d.k_pool, c.k_pool), c.k_pool)
    _write(dsa, g.layout, seq, last, to_dev(kv_rows), g.d.k_pool, to_dev(ki_rows),
           g.d.kidx_pool, ws)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(to_host(g.d.k_pool, c.k_pool), c.k_pool)
    np.testing.assert_array_equal(to_host(g.d.kidx_pool, c.kidx_pool), c.kidx_pool)
    s = g.scores().cpu().numpy()
    s_ref = oracle_scores(c, ld=s.shape[1])
    assert_scores_equal(s, s_ref, c.n_elig)
    idx = g.topk().cpu().numpy()
    idx_ref = oracle.topk(s_ref, c.n_elig, c.K)
    np.testing.assert_array_equal(idx, idx_ref)
    out, lse = g.attn()
    out_ref, lse_ref = oracle_attn(c, idx_ref)
    assert_out_close(out, lse, out_ref, lse_ref, "append")
    assert g.status() == 0 and dsa.get_status(ws) == 0


def test_cache_write_prefill_written_cache_serves_decode():
    """Prefill path writes the prompt (K/V and indexer keys) into an empty
    paged cache; a decode step of the same sequence over that cache equals
    the oracle's decode step over the original cache."""
    need_gpu()
    dsa = lib()
    T = 3000
    c = W.make_case("cw-prefill", seed=520, seq_lens=(T,), K=2048, **LAT_SHAPES)
    bt2, nb2 = fresh_layout(c, 29, 2)
    seq = np.zeros(T, np.int32)
    pos = np.arange(T, dtype=np.int32)
    lay = dsa.PagedLayout(to_dev(bt2), to_dev(c.seq_lens), c.bs, nb2, c.max_len)
    kv_pool = torch.zeros((nb2, c.bs, c.Dkv), dtype=torch.bfloat16, device="cuda")
    ki_pool = torch.zeros((nb2, c.bs, c.D_i), dtype=torch.uint8, device="cuda")
    ws = dsa.workspace(dsa.cache_write_workspace_size())
    _write(dsa, lay, seq, pos, to_dev(logical_rows(c, c.k_pool, 0, T)), kv_pool,
           to_dev(logical_rows(c, c.kidx_pool, 0, T)), ki_pool, ws)
    d = wdev.upload(c)
    pipe = dsa.Pipeline(lay, kind="decode", Nq=c.Nq, Hq=c.Hq, Dqk=c.Dqk, Dv=c.Dv, H_i=c.H_i,
                        D_i=c.D_i, K=c.K)
    dsa.index_score(lay, d.q_idx, d.w, ki_pool, pipe.scores, pipe.ws_index)
    s = pipe.scores.cpu().numpy()
    s_ref = oracle_scores(c, ld=s.shape[1])
    assert_scores_equal(s, s_ref, c.n_elig)
    dsa.topk(pipe.scores, d.n_elig, c.K, pipe.idx, pipe.ws_topk)
    idx_ref = oracle.topk(s_ref, c.n_elig, c.K)
    np.testing.assert_array_equal(pipe.idx.cpu().numpy(), idx_ref)
    dsa.sparse_attn_decode(lay, d.q, kv_pool, kv_pool, pipe.idx, c.sm_scale, pipe.out, pipe.lse,
                           pipe.ws_attn)
    out_ref, lse_ref = oracle_attn(c, idx_ref)
    assert_out_close(pipe.out, pipe.lse, out_ref, lse_ref, "prefill-written")
    assert pipe.status() == 0 and dsa.get_status(ws) == 0


def test_cache_write_flags_rows_without_a_destination():
    need_gpu()
    dsa = lib()
    c = W.make_case("cw-bad", seed=530, seq_lens=(70, 33, 128), bs=16, K=8, extra_pages=2,
                    **TINY_SHAPES)
    past = c.block_table.shape[1] * c.bs
    unused = int(np.argmax(c.block_table[1] < 0)) * c.bs
    bt = c.block_table.copy()
    bt[2, 1] = c.num_blocks + 7                                   # page id out of range
    seq = np.array([-1, c.B, 0, 0, 1, 2, 2, 0], np.int32)
    pos = np.array([0, 0, -1, past, unused, 20, 3, 69], np.int32)
    rng = np.random.default_rng(31)
    kv_rows = rng.integers(0, 1 << 16, size=(8, c.Dkv), dtype=np.uint16)
    ki_rows = rng.integers(0, 1 << 16, size=(8, c.D_i), dtype=np.uint16)
    kv_want, bad = oracle.cache_write(bt, c.bs, c.num_blocks, seq, pos, kv_rows, c.k_pool)
    ki_want, _ = oracle.cache_write(bt, c.bs, c.num_blocks, seq, pos, ki_rows, c.kidx_pool)
    assert bad
    lay = dsa.PagedLayout(to_dev(bt), to_dev(c.seq_lens), c.bs, c.num_blocks, c.max_len)
    kv_pool, ki_pool = to_dev(c.k_pool), to_dev(c.kidx_pool)
    ws = dsa.workspace(dsa.cache_write_workspace_size())
    _write(dsa, lay, seq, pos, to_dev(kv_rows), kv_pool, to_dev(ki_rows), ki_pool, ws)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(to_host(kv_pool, c.k_pool), kv_want)
    np.testing.assert_array_equal(to_host(ki_pool, c.kidx_pool), ki_want)
    assert dsa.get_status(ws) == 1                                # DSA_STATUS_BAD_BLOCK
    assert dsa.get_status(ws) == 0                                # cleared by the read


def test_cache_write_duplicates_leave_pieces_of_the_rows():
    """64 rows written to one position in one call: the writes race, so each
    16-byte piece of the row holds that piece of one of them (the rows are
    constant, so a piece is 8 equal values in 1..64), and nothing else
    changes."""
    need_gpu()
    dsa = lib()
    c = W.make_case("cw-dup", seed=540, seq_lens=(64,), bs=64, K=8, **TINY_SHAPES)
    seq = np.zeros(64, np.int32)
    pos = np.full(64, 17, np.int32)
    rows = np.repeat(np.arange(64, dtype=np.uint16)[:, None] + 1, c.Dkv, axis=1)
    lay = dsa.PagedLayout(to_dev(c.block_table), to_dev(c.seq_lens), c.bs, c.num_blocks, c.max_len)
    kv_pool = to_dev(c.k_pool)
    ws = dsa.workspace(dsa.cache_write_workspace_size())
    dsa.cache_write(lay, to_dev(seq), to_dev(pos), ws, kv_new=to_dev(rows), kv_pool=kv_pool)
    got = to_host(kv_pool, c.k_pool)
    page = c.block_table[0, 0]
    row = got[page, 17]
    for g in range(c.Dkv // 8):
        piece = row[8 * g:8 * g + 8]
        assert np.all(piece == piece[0]) and 1 <= int(piece[0]) <= 64, (g, piece)
    mask = np.ones(got.shape[:2], bool)
    mask[page, 17] = False
    np.testing.assert_array_equal(got[mask], c.k_pool[mask])


def test_cache_write_host_errors_launch_nothing():
    need_gpu()
    dsa = lib()
    c = W.make_case("cw-err", seed=550, seq_lens=(64,), bs=64, K=8, **TINY_SHAPES)
    lay = dsa.PagedLayout(to_dev(c.block_table), to_dev(c.seq_lens), c.bs, c.num_blocks, c.max_len)
    kv_pool = to_dev(c.k_pool)
    ws = dsa.workspace(dsa.cache_write_workspace_size())
    seq = to_dev(np.zeros(4, np.int32))
    pos = to_dev(np.arange(4, dtype=np.int32))
    L = dsa.lib()
    n0 = dsa.launch_count()
    vp = ctypes.c_void_p
    rows = torch.zeros((4, 12), dtype=torch.bfloat16, device="cuda")   # 12: not a multiple of 8
    rc = L.dsa_cache_write(lay.c(), vp(seq.data_ptr()), vp(pos.data_ptr()), 4, vp(rows.data_ptr()),
                           12, vp(kv_pool.data_ptr()), c.Dkv, None, 0, 0, None,
                           vp(ws.data_ptr()), ws.numel(), None)
    assert rc == -1
    rc = L.dsa_cache_write(lay.c(), vp(seq.data_ptr()), vp(pos.data_ptr()), 4, None, 0, None, 0,
                           None, 0, 0, None, vp(ws.data_ptr()), ws.numel(), None)
    assert rc == -1                                                    # nothing to write
    rc = L.dsa_cache_write(lay.c(), vp(seq.data_ptr()), vp(pos.data_ptr()), 0, None, 0, None, 0,
                           None, 0, 0, None, vp(ws.data_ptr()), ws.numel(), None)
    assert rc == 0                                                     # N = 0: nothing to do
    assert dsa.launch_count() == n0
