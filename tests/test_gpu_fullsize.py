"""Parity at the full sizes of the five workloads, in the launch configuration
bench.py times (the binding's stage calls on one Pipeline).

Where the oracle cannot afford a whole workload, it checks sampled outputs it
can compute one by one (score prefixes, sampled prefill rows), and the rest is
checked through properties that hold at any size (the selection definition on
the GPU's own scores, the closed-form answer of the tie construction).
"""
import numpy as np
import pytest

import oracle
import workloads as W
from gpu_common import (GpuRun, assert_out_close, assert_scores_equal, check_topk_definition,
                        need_gpu, oracle_attn, oracle_scores)

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


def _scores_prefix(c, n_pos):
    """Oracle scores of the first n_pos positions of every decode sequence."""
    lens = np.minimum(c.seq_lens, n_pos).astype(np.int32)
    return oracle.index_score(c.block_table, lens, c.bs, c.num_blocks, c.q_seq,
                              (lens - 1).astype(np.int32), c.q_idx, c.w, c.kidx_pool,
                              oracle.BF16 if c.idx_dtype == "bf16" else oracle.FP8_E4M3, n_pos)


def test_dec_tiny_full():
    need_gpu()
    c = W.config("dec-tiny")
    g = GpuRun(c)
    out, lse = g.all()
    s_ref = oracle_scores(c)
    assert_scores_equal(g.pipe.scores.cpu().numpy(), s_ref, c.n_elig)
    idx_ref = oracle.topk(s_ref, c.n_elig, c.K)
    np.testing.assert_array_equal(g.pipe.idx.cpu().numpy(), idx_ref)
    out_ref, lse_ref = oracle_attn(c, idx_ref)
    assert_out_close(out, lse, out_ref, lse_ref, "dec-tiny")
    assert g.status() == 0


def test_dec_batch_full():
    need_gpu()
    c = W.config("dec-batch")
    g = GpuRun(c)
    out, lse = g.all()
    s_ref = oracle_scores(c)
    assert_scores_equal(g.pipe.scores.cpu().numpy(), s_ref, c.n_elig)
    idx_ref = oracle.topk(s_ref, c.n_elig, c.K)
    np.testing.assert_array_equal(g.pipe.idx.cpu().numpy(), idx_ref)
    out_ref, lse_ref = oracle_attn(c, idx_ref)
    assert_out_close(out, lse, out_ref, lse_ref, "dec-batch")
    assert g.status() == 0


def test_long_dec_full_tie_closed_form():
    need_gpu()
    c = W.config("long-dec")
    g = GpuRun(c)
    out, lse = g.all()
    s = g.pipe.scores.cpu().numpy()
    s_ref = _scores_prefix(c, 8192)
    for b in range(c.B):
        np.testing.assert_array_equal(s[b, :8192], s_ref[b])
        tied = c.tie_positions[b]
        L = int(c.seq_lens[b])
        mx = s[b, :L].max()
        assert np.all(s[b, tied] == mx) and (s[b, :L] == mx).sum() == len(tied)
    idx = g.pipe.idx.cpu().numpy()
    for b in range(c.B):
        assert idx[b].tolist() == c.tie_positions[b][:c.K].tolist()
    out_ref, lse_ref = oracle_attn(c, idx)
    assert_out_close(out, lse, out_ref, lse_ref, "long-dec")
    assert g.status() == 0


def test_million_full_sampled():
    need_gpu()
    c = W.config("million")
    g = GpuRun(c)
    out, lse = g.all()
    s = g.pipe.scores.cpu().numpy()
    s_ref = _scores_prefix(c, 4096)
    for b in range(c.B):
        np.testing.assert_array_equal(s[b, :4096], s_ref[b])
    idx = g.pipe.idx.cpu().numpy()
    for b in range(c.B):
        check_topk_definition(s[b], int(c.seq_lens[b]), c.K, idx[b])
        assert np.all(np.isfinite(s[b, :int(c.seq_lens[b])]))
    out_ref, lse_ref = oracle_attn(c, idx)
    assert_out_close(out, lse, out_ref, lse_ref, "million")
    assert g.status() == 0


def test_prefill_full_sampled_rows():
    need_gpu()
    c = W.config("prefill")
    g = GpuRun(c)
    out, lse = g.all()
    rng = np.random.default_rng(0)
    rows = np.unique(np.r_[[0, 1, 2, 127, 128, 2046, 2047, 2048, 2049, 8191, 16383],
                           rng.integers(0, c.Nq, 12)])
    s_ref = oracle_scores(c, rows=rows)
    assert_scores_equal(g.pipe.scores.cpu().numpy()[rows], s_ref, c.n_elig[rows])
    idx_ref = oracle.topk(s_ref, c.n_elig[rows], c.K)
    np.testing.assert_array_equal(g.pipe.idx.cpu().numpy()[rows], idx_ref)
    out_ref, lse_ref = oracle_attn(c, idx_ref, rows=rows)
    assert_out_close(out[rows], lse[rows], out_ref, lse_ref, "prefill rows")
    assert g.status() == 0
