"""CPU oracle for the DSA sparse-attention hot path -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
reference arm of ``bench.py`` may import this package.  The library's product
path never touches it, and it never touches the product path: the two meet only
through the seeded inputs of ``workloads``.

The arithmetic lives in ``dsa_oracle.c`` (plain C, fp64, one thread); this
module builds it with gcc and marshals numpy arrays into it.  Each function
cites the passage it follows:

* ``index_score`` -- "Day-0 Adaptation of Trillion-Parameter MoE Models on
  Domestic GPUs", section 3 (1) Index Selection ("similarity scoring", read as
  the ReLU-weighted sum over indexer heads of q_idx . k_idx), restricted to
  causal positions.
* ``topk`` -- same page, section 3 (1) (the top-K selection), with the tie rule
  of "Day-0 Adaptation of Ultra-Large-Scale MoE Models on Heterogeneous AI
  Accelerators", section 4 ("Determinism of index selection"): equal scores go
  to the lower position.
* ``sparse_attn`` -- first page, section 3 (3) and the execution chain of the
  third page, section 4: exact softmax attention over the gathered rows only.
* the paged layout -- first page, section 3 (2): pages contiguous inside, an
  index table jumping between pages.
* ``cache_write`` -- "Day-0 Adaptation of Ultra-Large-Scale MoE Models on
  Heterogeneous AI Accelerators", section 4: new rows are written into the
  KV cache in the block layout, at the rows the decode gather reads (plain
  numpy, one row at a time).
* ``page_bounds`` / ``page_score_bound`` -- "Day-0 Adaptation of
  Trillion-Parameter MoE Models on Domestic GPUs", section 3 (3) (incremental
  decode-time selection that reuses an index structure): per page, per key
  dimension, the largest and smallest cached key, and the bound they give on
  every score of the page (plain numpy, fp64, page by page).

Every function is pinned by the ``-m "not gpu"`` tests in ``tests/`` against
closed forms, invariants, library special cases and brute force; none of the
pins calls back into this module's own arithmetic to check itself.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "dsa_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

BF16 = 0
FP8_E4M3 = 1


def build(force: bool = False) -> str:
    """Compile ``dsa_oracle.c`` into ``liboracle.so`` (gcc, -O2, no SIMD flags)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.run(
            ["gcc", "-O2", "-std=c11", "-Wall", "-shared", "-fPIC", "-o", tmp, _SRC, "-lm"],
            check=True,
        )
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            i32p = ctypes.POINTER(ctypes.c_int32)
            vp = ctypes.c_void_p
            lib.oracle_decode.restype = ctypes.c_double
            lib.oracle_decode.argtypes = [ctypes.c_int, ctypes.c_uint32]
            lib.oracle_index_score.restype = ctypes.c_int
            lib.oracle_index_score.argtypes = [
                ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, i32p, i32p,
                ctypes.c_int, i32p, i32p, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                vp, vp, vp, ctypes.c_int64, vp]
            lib.oracle_topk.restype = ctypes.c_int
            lib.oracle_topk.argtypes = [vp, ctypes.c_int64, i32p, ctypes.c_int, ctypes.c_int, i32p]
            lib.oracle_sparse_attn.restype = ctypes.c_int
            lib.oracle_sparse_attn.argtypes = [
                ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, i32p, i32p,
                ctypes.c_int, i32p, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                vp, vp, ctypes.c_int64, vp, ctypes.c_int64, i32p, ctypes.c_int,
                ctypes.c_double, vp, vp]
            _lib = lib
    return _lib


class OracleError(RuntimeError):
    pass


def _i32(a):
    a = np.ascontiguousarray(a, dtype=np.int32)
    return a, a.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))


def _raw(a, dtype_code):
    want = np.uint16 if dtype_code == BF16 else np.uint8
    a = np.ascontiguousarray(a)
    if a.dtype != want:
        raise TypeError(f"encoded array must be {want.__name__}, got {a.dtype}")
    return a


def decode(dtype_code: int, raw: int) -> float:
    """Exact value of one stored bf16 (raw uint16) or FP8 E4M3 (raw uint8) code."""
    return float(_load().oracle_decode(int(dtype_code), int(raw)))


def index_score(block_table, seq_lens, bs, num_blocks, q_seq, q_pos, q_idx, w, kidx_pool,
                dtype_code, ld):
    """Scores [Nq, ld] fp32: ReLU-weighted head sum over causal positions, -inf elsewhere.

    q_idx: encoded [Nq, H, D]; w: fp32 [Nq, H]; kidx_pool: encoded [NB, bs, D].
    """
    lib = _load()
    bt, btp = _i32(block_table)
    sl, slp = _i32(seq_lens)
    qs, qsp = _i32(q_seq)
    qp, qpp = _i32(q_pos)
    q_idx = _raw(q_idx, dtype_code)
    kidx_pool = _raw(kidx_pool, dtype_code)
    w = np.ascontiguousarray(w, dtype=np.float32)
    Nq, H, D = q_idx.shape
    assert kidx_pool.shape[-1] == D and kidx_pool.shape[-2] == bs
    out = np.empty((Nq, int(ld)), dtype=np.float32)
    rc = lib.oracle_index_score(
        int(sl.shape[0]), int(bs), int(num_blocks), int(bt.shape[1]), btp, slp,
        int(Nq), qsp, qpp, int(H), int(D), int(dtype_code),
        q_idx.ctypes.data, w.ctypes.data, kidx_pool.ctypes.data, int(ld), out.ctypes.data)
    if rc != 0:
        raise OracleError(f"oracle_index_score returned {rc}")
    return out


def topk(scores, n_elig, K):
    """idx [Nq, K] int32: top-K by (score desc, position asc), ascending, -1 padded."""
    lib = _load()
    scores = np.ascontiguousarray(scores, dtype=np.float32)
    ne, nep = _i32(n_elig)
    Nq, ld = scores.shape
    idx = np.empty((Nq, int(K)), dtype=np.int32)
    rc = lib.oracle_topk(scores.ctypes.data, int(ld), nep, int(Nq), int(K),
                         idx.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)))
    if rc != 0:
        raise OracleError(f"oracle_topk returned {rc}")
    return idx


def sparse_attn(block_table, seq_lens, bs, num_blocks, q_seq, q, k_pool, v_pool, idx, sm_scale,
                Dv=None):
    """(out [Nq, Hq, Dv] fp64, lse [Nq, Hq] fp64): exact softmax attention over idx rows.

    q: bf16 bits uint16 [Nq, Hq, Dqk]; k_pool/v_pool: bf16 bits uint16 [NB, bs, D*];
    v_pool may be the same array as k_pool (latent cache, V = first Dv dims).
    """
    lib = _load()
    bt, btp = _i32(block_table)
    sl, slp = _i32(seq_lens)
    qs, qsp = _i32(q_seq)
    ix, ixp = _i32(idx)
    q = _raw(q, BF16)
    k_pool = _raw(k_pool, BF16)
    v_pool = _raw(v_pool, BF16)
    Nq, Hq, Dqk = q.shape
    k_stride = int(k_pool.shape[-1])
    v_stride = int(v_pool.shape[-1])
    if Dv is None:
        Dv = v_stride
    assert Dqk <= k_stride and Dv <= v_stride
    K = int(ix.shape[1])
    out = np.empty((Nq, Hq, int(Dv)), dtype=np.float64)
    lse = np.empty((Nq, Hq), dtype=np.float64)
    rc = lib.oracle_sparse_attn(
        int(sl.shape[0]), int(bs), int(num_blocks), int(bt.shape[1]), btp, slp,
        int(Nq), qsp, int(Hq), int(Dqk), int(Dv),
        q.ctypes.data, k_pool.ctypes.data, k_stride, v_pool.ctypes.data, v_stride,
        ixp, K, float(sm_scale), out.ctypes.data, lse.ctypes.data)
    if rc != 0:
        raise OracleError(f"oracle_sparse_attn returned {rc}")
    return out, lse


def cache_write(block_table, bs, num_blocks, seq, pos, new_rows, pool):
    """(pool', bad): pool [NB, bs, W] with row i of new_rows [N, w <= W] stored
    at position pos[i] of sequence seq[i]; bad is True when some row had no
    valid destination (sequence outside the table, position past its row of
    the table, or a page id outside [0, NB)) and was skipped.

    "Day-0 Adaptation of Ultra-Large-Scale MoE Models on Heterogeneous AI
    Accelerators", section 4 (KV cache write in the block layout; the layout
    written must match the gather of decode), with the mapping of "Day-0
    Adaptation of Trillion-Parameter MoE Models on Domestic GPUs", section 3
    (2): position p lives in page block_table[b][p // bs], row p % bs.  Rows
    are written in order, so of two rows with one destination the later wins.
    """
    bt = np.asarray(block_table)
    out = np.array(pool, copy=True)
    assert out.shape[0] == num_blocks and out.shape[1] == bs
    new_rows = np.asarray(new_rows)
    w = new_rows.shape[1]
    bad = False
    for i in range(len(seq)):
        b, p = int(seq[i]), int(pos[i])
        if b < 0 or b >= bt.shape[0] or p < 0 or p // bs >= bt.shape[1]:
            bad = True
            continue
        page = int(bt[b, p // bs])
        if page < 0 or page >= num_blocks:
            bad = True
            continue
        out[page, p % bs, :w] = new_rows[i]
    return out, bad


_TABLES = {}


def _decode_table(dtype_code):
    """Value of every code of the format (bf16: 65536 codes, E4M3: 256)."""
    if dtype_code not in _TABLES:
        n = 65536 if dtype_code == BF16 else 256
        lib = _load()
        _TABLES[dtype_code] = np.array([lib.oracle_decode(int(dtype_code), c) for c in range(n)],
                                       dtype=np.float64)
    return _TABLES[dtype_code]


def page_bounds(block_table, seq_lens, bs, num_blocks, kidx_pool, dtype_code):
    """(bounds, cached): bounds [NB, 2, D] codes (the pool's dtype) holding, for
    every page some sequence caches a position in, per dimension the code of
    the largest key (row 0) and of the smallest key (row 1) over the page's
    cached positions -- the first such row on ties; cached [NB] bool marks
    those pages (the others are zero).

    "Day-0 Adaptation of Trillion-Parameter MoE Models on Domestic GPUs",
    section 3 (3): the index structure a decode step reuses, kept per page.
    """
    table = _decode_table(dtype_code)
    pool = _raw(kidx_pool, dtype_code)
    bt = np.asarray(block_table)
    D = pool.shape[-1]
    out = np.zeros((num_blocks, 2, D), dtype=pool.dtype)
    cached = np.zeros(num_blocks, dtype=bool)
    for b in range(bt.shape[0]):
        L = int(seq_lens[b])
        for j in range((L + bs - 1) // bs):
            page = int(bt[b, j])
            n = min(bs, L - j * bs)
            codes = pool[page, :n]                 # [n, D]
            vals = table[codes.astype(np.int64)]
            out[page, 0] = codes[np.argmax(vals, axis=0), np.arange(D)]
            out[page, 1] = codes[np.argmin(vals, axis=0), np.arange(D)]
            cached[page] = True
    return out, cached


def page_score_bound(q_idx, w, bounds, dtype_code):
    """UB [NB] fp64 for one query: sum_h (w_h >= 0 ? w_h relu(hi_h) : w_h relu(lo_h))
    with hi_h = sum_d max(q_hd kmax_d, q_hd kmin_d), lo_h the same with min, so
    that every score of a page's cached positions is at most its UB.

    q_idx: encoded [H, D]; w: [H]; bounds: [NB, 2, D] codes from page_bounds.
    """
    table = _decode_table(dtype_code)
    q = table[_raw(q_idx, dtype_code).astype(np.int64)]          # [H, D]
    kx = table[np.asarray(bounds)[:, 0].astype(np.int64)]          # [NB, D]
    kn = table[np.asarray(bounds)[:, 1].astype(np.int64)]
    w = np.asarray(w, dtype=np.float64)
    ub = np.zeros(kx.shape[0])
    for h in range(q.shape[0]):
        u = q[h][None, :] * kx
        v = q[h][None, :] * kn
        hi = np.maximum(u, v).sum(axis=1)
        lo = np.minimum(u, v).sum(axis=1)
        ub += w[h] * np.maximum(hi if w[h] >= 0 else lo, 0.0)
    return ub
