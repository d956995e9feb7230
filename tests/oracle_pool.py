"""The CPU oracle over whole workloads, sharded across worker processes.

The oracle itself stays what it is: plain, single-threaded C code called
through ``oracle``.  This module only splits a full-size workload into shards
of query rows (or whole sequences) and runs one oracle call per shard in a
pool of worker processes, so that the parity tests can compare every score,
every index set and thousands of attention rows at the workloads' full sizes
instead of samples.

Workers are started with the ``spawn`` method (never forked from a process
that has touched the GPU) and import only ``numpy`` and ``oracle``.  The
case's arrays reach them as ``.npy`` files in a private temporary directory,
opened memory-mapped, so a 1 GB key pool is shared through the page cache
rather than copied into every worker; results come back the same way, through
memory-mapped output files the parent creates.
"""
from __future__ import annotations

import multiprocessing as mp
import os
import shutil
import tempfile

import numpy as np

import oracle

_IDX_CODES = {"bf16": oracle.BF16, "fp8": oracle.FP8_E4M3}


def _open(path):
    return np.load(path, mmap_mode="r")


# ----------------------------------------------------------- worker side --
def _score_topk_shard(job):
    """Oracle scores of rows [r0, r1) of a case, then the oracle's top-K over
    them; both written into the parent's output files."""
    (files, r0, r1, ld, K, code, bs, nb, scores_path, idx_path) = job
    a = {k: _open(p) for k, p in files.items()}
    rows = np.arange(r0, r1)
    s = oracle.index_score(a["block_table"], a["seq_lens"], bs, nb, a["q_seq"][rows],
                           a["q_pos"][rows], a["q_idx"][rows], a["w"][rows], a["kidx_pool"],
                           code, ld)
    idx = oracle.topk(s, a["n_elig"][rows], K)
    out_s = np.load(scores_path, mmap_mode="r+")
    out_i = np.load(idx_path, mmap_mode="r+")
    out_s[r0:r1] = s
    out_i[r0:r1] = idx
    out_s.flush()
    out_i.flush()
    return r1 - r0


def _attn_shard(job):
    """Oracle attention of the given rows over the given index sets."""
    (files, rows, idx, sm_scale, Dv, bs, nb, out_path, lse_path, slot0) = job
    a = {k: _open(p) for k, p in files.items()}
    rows = np.asarray(rows)
    v_pool = a["v_pool"] if "v_pool" in a else a["k_pool"]
    out, lse = oracle.sparse_attn(a["block_table"], a["seq_lens"], bs, nb, a["q_seq"][rows],
                                  a["q"][rows], a["k_pool"], v_pool, idx, sm_scale, Dv=Dv)
    o = np.load(out_path, mmap_mode="r+")
    l = np.load(lse_path, mmap_mode="r+")
    o[slot0:slot0 + len(rows)] = out
    l[slot0:slot0 + len(rows)] = lse
    o.flush()
    l.flush()
    return len(rows)


# ----------------------------------------------------------- parent side --
def _balanced_shards(cost, n_shards):
    """Cut rows 0..len(cost)-1 into at most n_shards contiguous ranges of
    roughly equal total cost."""
    c = np.cumsum(np.asarray(cost, dtype=np.float64))
    total = float(c[-1]) if len(c) else 0.0
    bounds = [0]
    for k in range(1, n_shards):
        r = int(np.searchsorted(c, total * k / n_shards, side="left")) + 1
        if bounds[-1] < r < len(cost):
            bounds.append(r)
    bounds.append(len(cost))
    return [(bounds[i], bounds[i + 1]) for i in range(len(bounds) - 1)]


class OraclePool:
    """``with OraclePool(case) as pool:`` -- the case's arrays written once to a
    temporary directory, a spawn-started process pool over them."""

    def __init__(self, case, workers=None):
        self.case = case
        self.workers = max(1, int(workers or os.cpu_count() or 1))
        self.dir = tempfile.mkdtemp(prefix="dsa_oracle_pool_")
        self.files = {}
        self.pool = None

    def _inputs(self, names):
        """The files of the named case arrays, each written on first use."""
        for n in names:
            if n not in self.files:
                p = os.path.join(self.dir, n + ".npy")
                np.save(p, np.ascontiguousarray(getattr(self.case, n)))
                self.files[n] = p
        return {n: self.files[n] for n in names}

    def __enter__(self):
        self.pool = mp.get_context("spawn").Pool(self.workers)
        return self

    def __exit__(self, *exc):
        if self.pool is not None:
            self.pool.terminate()
            self.pool.join()
        shutil.rmtree(self.dir, ignore_errors=True)
        return False

    def _out(self, name, shape, dtype):
        p = os.path.join(self.dir, name + ".npy")
        np.lib.format.open_memmap(p, mode="w+", dtype=dtype, shape=shape).flush()
        return p

    def scores_and_topk(self, ld):
        """(scores [Nq, ld] fp32, idx [Nq, K] int32) of every query of the case,
        each row from one oracle call on the shard holding it."""
        c = self.case
        cost = np.minimum(c.n_elig.astype(np.int64), ld) + 64
        shards = _balanced_shards(cost, 4 * self.workers)
        sp = self._out("out_scores", (c.Nq, int(ld)), np.float32)
        ip = self._out("out_idx", (c.Nq, c.K), np.int32)
        code = _IDX_CODES[c.idx_dtype]
        files = self._inputs(["block_table", "seq_lens", "q_seq", "q_pos", "n_elig", "q_idx", "w",
                              "kidx_pool"])
        jobs = [(files, r0, r1, int(ld), int(c.K), code, int(c.bs), int(c.num_blocks), sp, ip)
                for r0, r1 in shards]
        done = sum(self.pool.imap_unordered(_score_topk_shard, jobs))
        assert done == c.Nq
        return np.array(np.load(sp, mmap_mode="r")), np.array(np.load(ip, mmap_mode="r"))

    def attention(self, rows, idx):
        """(out [len(rows), Hq, Dv] fp64, lse [len(rows), Hq] fp64) of the given
        query rows over the given index sets (one row of idx per row)."""
        c = self.case
        rows = np.asarray(rows, dtype=np.int64)
        idx = np.ascontiguousarray(idx, dtype=np.int32)
        op = self._out("out_attn", (len(rows), c.Hq, c.Dv), np.float64)
        lp = self._out("out_lse", (len(rows), c.Hq), np.float64)
        n_shards = min(len(rows), 4 * self.workers)
        bounds = np.linspace(0, len(rows), n_shards + 1).astype(np.int64)
        files = self._inputs(["block_table", "seq_lens", "q_seq", "q", "k_pool"] +
                             ([] if c.latent else ["v_pool"]))
        jobs = [(files, rows[b0:b1], idx[b0:b1], float(c.sm_scale), int(c.Dv), int(c.bs),
                 int(c.num_blocks), op, lp, int(b0))
                for b0, b1 in zip(bounds[:-1], bounds[1:]) if b1 > b0]
        done = sum(self.pool.imap_unordered(_attn_shard, jobs))
        assert done == len(rows)
        return np.array(np.load(op, mmap_mode="r")), np.array(np.load(lp, mmap_mode="r"))
