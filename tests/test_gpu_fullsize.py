"""Parity at the full sizes of the five workloads, in the launch configuration
bench.py times (the binding's stage calls on one Pipeline).

Every score and every index set of every workload is compared with the CPU
oracle: the oracle stays single-threaded, and the workload's rows (or
sequences) are shared out over worker processes (``oracle_pool``), one oracle
call per shard.  Attention outputs are compared on every query of the decode
workloads and, for the 16384-token prefill, on 2048 seeded rows plus the edge
rows (the first positions, where a query sees fewer than K positions, the
rows around K, and the last).
"""
import numpy as np
import pytest

import oracle
import workloads as W
from gpu_common import DevicePipeline, assert_out_close, assert_scores_equal, need_gpu, oracle_attn
from oracle_pool import OraclePool

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


def _gpu(c):
    """The three stages on the GPU; results copied to the host."""
    g = DevicePipeline(c)
    out, lse = g.all()
    res = dict(scores=g.pipe.scores.cpu().numpy(), idx=g.pipe.idx.cpu().numpy(),
               out=out.float().cpu().numpy().astype(np.float64),
               lse=lse.cpu().numpy().astype(np.float64), status=g.status(), ld=g.pipe.ld)
    del g
    return res


def _full_parity(c, attn_rows=None):
    """Scores and index sets of every query against the oracle; attention on
    attn_rows (all queries when None)."""
    need_gpu()
    r = _gpu(c)
    assert r["status"] == 0
    rows = np.arange(c.Nq) if attn_rows is None else np.asarray(attn_rows)
    with OraclePool(c) as pool:
        s_ref, idx_ref = pool.scores_and_topk(c.max_len)
        assert_scores_equal(r["scores"], s_ref, c.n_elig)
        np.testing.assert_array_equal(r["idx"], idx_ref)
        if len(rows) > 64:
            out_ref, lse_ref = pool.attention(rows, idx_ref[rows])
        else:
            out_ref, lse_ref = oracle_attn(c, idx_ref[rows], rows=rows)
    assert_out_close(r["out"][rows], r["lse"][rows], out_ref, lse_ref, c.name)
    return r, idx_ref


def test_dec_tiny_full():
    _full_parity(W.config("dec-tiny"))


def test_dec_batch_full():
    _full_parity(W.config("dec-batch"))


def test_long_dec_full():
    """Every score row in full, the oracle's index sets, and the tie
    construction's closed form (the 2048 lowest tied positions)."""
    c = W.config("long-dec")
    r, idx_ref = _full_parity(c)
    for b in range(c.B):
        L = int(c.seq_lens[b])
        tied = c.tie_positions[b]
        mx = r["scores"][b, :L].max()
        assert np.all(r["scores"][b, tied] == mx) and (r["scores"][b, :L] == mx).sum() == len(tied)
        assert idx_ref[b].tolist() == tied[:c.K].tolist()


def test_million_full():
    _full_parity(W.config("million"))


def test_prefill_full():
    """All 16384 score rows and index sets; attention on 2048 seeded rows plus
    the edge rows."""
    c = W.config("prefill")
    rng = np.random.default_rng(2024)
    edge = [0, 1, 2, 3, 63, 64, 127, 128, 511, 512, 513, 2046, 2047, 2048, 2049, 4095, 8191,
            16382, 16383]
    rows = np.unique(np.r_[edge, rng.choice(c.Nq, 2048, replace=False)])
    _full_parity(c, attn_rows=rows)
