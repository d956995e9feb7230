"""Python binding of libdsa.so -- the DSA sparse-attention hot path for GB300.

Argument marshalling only: every stage runs in the library's CUDA kernels.
PyTorch supplies device memory and the current CUDA stream; tensors are passed
as raw device pointers to the C ABI declared in ``include/dsa.h``.

Stages (names as in the C ABI):

* :func:`index_score` -- indexer score of every cached position, ReLU-weighted
  over indexer heads ("Day-0 Adaptation of Trillion-Parameter MoE Models on
  Domestic GPUs", section 3 (1));
* :func:`topk` -- exact top-K per query, ties to the lower position ("Day-0
  Adaptation of Ultra-Large-Scale MoE Models on Heterogeneous AI
  Accelerators", section 4);
* :func:`sparse_attn_decode` / :func:`sparse_attn_prefill` -- exact softmax
  attention over the selected rows gathered through the block table (first
  page, section 3 (2)-(3)).

:func:`decode` and :func:`prefill` chain the three stages with workspaces
allocated through torch.  There is no CPU fallback: importing this package
raises if ``libdsa.so`` has not been built, and every call raises
:class:`DsaError` if the library reports an error.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass
from typing import Optional

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libdsa.so")

DSA_OK = 0
DSA_BF16 = 0
DSA_FP8_E4M3 = 1
STATUS_BAD_BLOCK = 0x1
STATUS_BAD_INDEX = 0x2
STATUS_BAD_LENGTH = 0x4
STATUS_TIMEOUT = 0x8

if not os.path.exists(LIB_PATH):
    raise ImportError(
        f"{LIB_PATH} is missing: build it first (python -c 'import __graft_entry__ as g; g.build()')")

_lib = ctypes.CDLL(LIB_PATH)


class DsaError(RuntimeError):
    def __init__(self, code: int, where: str):
        msg = _lib.dsa_last_error_string().decode(errors="replace")
        super().__init__(f"{where} failed with code {code}: {msg}")
        self.code = code


class PagedLayoutC(ctypes.Structure):
    _fields_ = [("block_size", ctypes.c_int32), ("num_blocks", ctypes.c_int32),
                ("max_blocks_per_seq", ctypes.c_int32), ("batch", ctypes.c_int32),
                ("max_seq_len", ctypes.c_int32), ("reserved_", ctypes.c_int32),
                ("block_table", ctypes.c_void_p), ("seq_lens", ctypes.c_void_p)]


_vp, _i, _i64, _sz, _f = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t, ctypes.c_float
_LP = ctypes.POINTER(PagedLayoutC)


def _sig(name, restype, argtypes):
    fn = getattr(_lib, name)
    fn.restype = restype
    fn.argtypes = argtypes
    return fn


_sig("dsa_version", _i, [])
_sig("dsa_launch_count", ctypes.c_uint64, [])
_sig("dsa_last_error_string", ctypes.c_char_p, [])
_sig("dsa_get_status", _i, [_vp, _vp, ctypes.POINTER(ctypes.c_int32), _i])
_sig("dsa_selftest_bounded_wait", _i, [_i, ctypes.c_uint64, _vp, _sz, _vp])
_sig("dsa_index_score_workspace_size", _sz, [_i, _i, _i, _i64])
_sig("dsa_index_score", _i, [_LP, _vp, _vp, _vp, _i, _i, _i, _vp, _vp, _i, _vp, _i64, _vp, _sz, _vp])
_sig("dsa_index_score_prefill_workspace_size", _sz, [_i, _i, _i, _i64])
_sig("dsa_index_score_prefill", _i, [_LP, _i, _vp, _vp, _vp, _i, _i, _i, _vp, _i, _vp, _i64, _vp, _sz,
                                     _vp])
_sig("dsa_topk_workspace_size", _sz, [_i, _i64, _i])
_sig("dsa_topk", _i, [_vp, _i64, _vp, _i, _i, _vp, _vp, _sz, _vp])
_sig("dsa_topk_noalloc", _i, [_vp, _i64, _vp, _i, _i, _vp, _vp])
_sig("dsa_topk_noalloc_scratch_bytes", _sz, [])
_sig("dsa_decode_step_workspace_size", _sz, [_i, _i, _i, _i64, _i, _i, _i, _i])
_sig("dsa_decode_step", _i, [_LP, _vp, _vp, _i64, _vp, _vp, _i64, _vp, _vp, _i, _vp, _vp, _i, _i,
                             _vp, _i, _i, _i, _i, _f, _vp, _i64, _vp, _vp, _vp, _vp, _sz, _vp])
_sig("dsa_prefill_step_workspace_size", _sz, [_i, _i, _i, _i64, _i, _i, _i, _i])
_sig("dsa_prefill_step", _i, [_LP, _i, _vp, _vp, _i, _vp, _vp, _i64, _vp, _vp, _i64, _vp, _vp, _i,
                              _vp, _vp, _i, _i, _vp, _i, _i, _i, _i, _f, _vp, _i64, _vp, _vp, _vp,
                              _vp, _sz, _vp])
_sig("dsa_prefill_step_chunked_workspace_size", _sz, [_i, _i, _i, _i64, _i, _i, _i, _i, _i])
_sig("dsa_prefill_step_chunked", _i, [_LP, _i, _vp, _vp, _i, _vp, _vp, _i64, _vp, _vp, _i64, _vp,
                                      _vp, _i, _vp, _vp, _i, _i, _vp, _i, _i, _i, _i, _f, _i64, _i,
                                      _vp, _vp, _vp, _vp, _sz, _vp])
_sig("dsa_index_bounds_update_workspace_size", _sz, [])
_sig("dsa_index_bounds_update", _i, [_LP, _vp, _vp, _i, _vp, _i, _i, _vp, _vp, _sz, _vp])
_sig("dsa_index_score_bounded_workspace_size", _sz, [_i, _i, _i, _i64, _i])
_sig("dsa_index_score_bounded", _i, [_LP, _vp, _vp, _vp, _i, _i, _i, _vp, _i, _vp, _i64, _vp, _sz,
                                     _vp])
_sig("dsa_index_bounded_stats", _i, [_vp, _vp, ctypes.POINTER(ctypes.c_uint64),
                                     ctypes.POINTER(ctypes.c_uint64)])
_sig("dsa_cache_write_workspace_size", _sz, [])
_sig("dsa_cache_write", _i, [_LP, _vp, _vp, _i, _vp, _i, _vp, _i64, _vp, _i, _i, _vp, _vp, _sz, _vp])
_sig("dsa_sparse_attn_decode_workspace_size", _sz, [_i, _i, _i, _i, _i])
_sig("dsa_sparse_attn_decode", _i, [_LP, _vp, _vp, _i64, _vp, _i64, _i, _i, _i, _vp, _i, _f, _vp,
                                    _vp, _vp, _sz, _vp])
_sig("dsa_sparse_attn_prefill_workspace_size", _sz, [_i, _i, _i, _i, _i])
_sig("dsa_sparse_attn_prefill", _i, [_LP, _vp, _vp, _i64, _vp, _i64, _i, _i, _i, _vp, _vp, _i, _vp,
                                     _i, _f, _vp, _vp, _vp, _sz, _vp])

SYMBOLS = ("dsa_version", "dsa_launch_count", "dsa_last_error_string", "dsa_get_status",
           "dsa_selftest_bounded_wait",
           "dsa_index_score_workspace_size", "dsa_index_score",
           "dsa_index_score_prefill_workspace_size", "dsa_index_score_prefill",
           "dsa_topk_workspace_size",
           "dsa_topk", "dsa_topk_noalloc", "dsa_topk_noalloc_scratch_bytes",
           "dsa_sparse_attn_decode_workspace_size", "dsa_sparse_attn_decode",
           "dsa_sparse_attn_prefill_workspace_size", "dsa_sparse_attn_prefill",
           "dsa_cache_write_workspace_size", "dsa_cache_write",
           "dsa_decode_step_workspace_size", "dsa_decode_step",
           "dsa_prefill_step_workspace_size", "dsa_prefill_step",
           "dsa_prefill_step_chunked_workspace_size", "dsa_prefill_step_chunked",
           "dsa_index_bounds_update_workspace_size", "dsa_index_bounds_update",
           "dsa_index_score_bounded_workspace_size", "dsa_index_score_bounded",
           "dsa_index_bounded_stats")


def lib() -> ctypes.CDLL:
    return _lib


def version() -> int:
    return int(_lib.dsa_version())


def launch_count() -> int:
    """Kernels launched by libdsa.so in this process so far."""
    return int(_lib.dsa_launch_count())


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not t.is_contiguous():
        raise ValueError("tensors must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


class _Args:
    """The operands of one call, checked so that no kernel can run outside
    them: as each is added, its element size and element count (at least
    what the call touches); then, in ptrs(), that every one of them and the
    layout live on the GPU.  Sizes are checked for all operands before
    residency for any, so that each check can be exercised with host
    tensors."""

    def __init__(self, layout: Optional["PagedLayout"] = None):
        self._t = []
        self._layout = layout

    def add(self, t: Optional[torch.Tensor], name: str, elt=None, numel: Optional[int] = None):
        if t is not None:
            if elt is not None and t.element_size() not in elt:
                raise TypeError(f"{name}: {t.dtype} has {t.element_size()}-byte elements; "
                                f"the call needs {' or '.join(str(e) for e in elt)}")
            if numel is not None and t.numel() < numel:
                raise ValueError(f"{name}: {t.numel()} elements; the call needs at least "
                                 f"{numel}")
        self._t.append((t, name))
        return self

    def ptrs(self):
        for t, name in self._t:
            if t is not None and not t.is_cuda:
                raise ValueError(f"{name}: a CUDA tensor is required")
        lay = self._layout
        if lay is not None and not (lay.block_table.is_cuda and lay.seq_lens.is_cuda):
            raise ValueError("layout: block_table and seq_lens must be CUDA tensors")
        return [_ptr(t) for t, _ in self._t]


def _rows(layout: "PagedLayout", width: int) -> int:
    """Elements of a paged pool of `width`-element rows."""
    return int(layout.num_blocks) * int(layout.block_size) * int(width)


_F32, _I32, _BF16, _KEY, _WS = (4,), (4,), (2,), (1, 2), (1,)  # element sizes (bytes)


_raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)


def _stream(stream=None):
    """The CUDA stream handle to launch on: `stream`, else the current stream
    of the current device (read as a raw handle when torch offers that, which
    costs a fraction of building a torch Stream object on every call)."""
    if stream is not None:
        return ctypes.c_void_p(stream.cuda_stream)
    if _raw_stream is not None:
        return ctypes.c_void_p(_raw_stream(torch.cuda.current_device()))
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _check(rc: int, where: str):
    if rc != DSA_OK:
        raise DsaError(rc, where)


def _elt_dtype(t: torch.Tensor) -> int:
    return DSA_FP8_E4M3 if t.element_size() == 1 else DSA_BF16


@dataclass
class PagedLayout:
    """Block table + sequence lengths on the device (tensors kept alive here)."""

    block_table: torch.Tensor  # int32 [B, max_blocks]
    seq_lens: torch.Tensor     # int32 [B]
    block_size: int
    num_blocks: int
    max_seq_len: int

    def __post_init__(self):
        if self.block_table.dtype != torch.int32 or self.seq_lens.dtype != torch.int32:
            raise TypeError("block_table and seq_lens must be int32")
        self._c = PagedLayoutC(int(self.block_size), int(self.num_blocks),
                               int(self.block_table.shape[1]), int(self.block_table.shape[0]),
                               int(self.max_seq_len), 0, self.block_table.data_ptr(),
                               self.seq_lens.data_ptr())

    @property
    def batch(self) -> int:
        return int(self.block_table.shape[0])

    def c(self):
        return ctypes.byref(self._c)


def workspace(nbytes: int, device=None) -> torch.Tensor:
    """Zero-filled device workspace (uint8), 256-byte aligned by the allocator."""
    return torch.zeros(max(int(nbytes), 256), dtype=torch.uint8, device=device or "cuda")


def index_score_workspace_size(Nq, H_i, D_i, ld) -> int:
    return int(_lib.dsa_index_score_workspace_size(Nq, H_i, D_i, ld))


def topk_workspace_size(Nq, ld, K) -> int:
    return int(_lib.dsa_topk_workspace_size(Nq, ld, K))


def sparse_attn_decode_workspace_size(B, Hq, Dqk, Dv, K) -> int:
    return int(_lib.dsa_sparse_attn_decode_workspace_size(B, Hq, Dqk, Dv, K))


def sparse_attn_prefill_workspace_size(Nq, Hq, Dqk, Dv, K) -> int:
    return int(_lib.dsa_sparse_attn_prefill_workspace_size(Nq, Hq, Dqk, Dv, K))


def index_score(layout: PagedLayout, q_idx, w, kidx_pool, scores, ws, q_seq=None, q_pos=None,
                stream=None):
    """scores[Nq, ld] <- indexer scores (see include/dsa.h, dsa_index_score)."""
    Nq, H_i, D_i = q_idx.shape
    ld = scores.shape[1]
    a = _Args(layout).add(q_idx, "q_idx", _KEY).add(w, "w", _F32, Nq * H_i)
    a.add(kidx_pool, "kidx_pool", (q_idx.element_size(),), _rows(layout, D_i))
    a.add(q_seq, "q_seq", _I32, Nq).add(q_pos, "q_pos", _I32, Nq)
    a.add(scores, "scores", _F32, Nq * ld).add(ws, "ws", _WS)
    pq, pw, pk, pseq, ppos, ps, pws = a.ptrs()
    rc = _lib.dsa_index_score(layout.c(), pq, pw, pk, _elt_dtype(kidx_pool), H_i, D_i, pseq, ppos,
                              Nq, ps, ld, pws, ws.numel(), _stream(stream))
    _check(rc, "dsa_index_score")


def index_score_prefill(layout: PagedLayout, seq, q_idx, w, kidx_pool, scores, ws, q_pos=None,
                        stream=None):
    """scores[Nq, ld] <- indexer scores of Nq queries of sequence `seq`."""
    Nq, H_i, D_i = q_idx.shape
    ld = scores.shape[1]
    a = _Args(layout).add(q_idx, "q_idx", _KEY).add(w, "w", _F32, Nq * H_i)
    a.add(kidx_pool, "kidx_pool", (q_idx.element_size(),), _rows(layout, D_i))
    a.add(q_pos, "q_pos", _I32, Nq).add(scores, "scores", _F32, Nq * ld).add(ws, "ws", _WS)
    pq, pw, pk, ppos, ps, pws = a.ptrs()
    rc = _lib.dsa_index_score_prefill(layout.c(), int(seq), pq, pw, pk, _elt_dtype(kidx_pool), H_i,
                                      D_i, ppos, Nq, ps, ld, pws, ws.numel(), _stream(stream))
    _check(rc, "dsa_index_score_prefill")


def topk(scores, n_eligible, K, idx, ws, stream=None):
    """idx[Nq, K] <- top-K positions, ascending, -1 padded."""
    Nq, ld = scores.shape
    K = int(K)
    a = _Args().add(scores, "scores", _F32).add(n_eligible, "n_eligible", _I32, Nq)
    a.add(idx, "idx", _I32, Nq * K).add(ws, "ws", _WS)
    ps, pn, pi, pws = a.ptrs()
    rc = _lib.dsa_topk(ps, ld, pn, Nq, K, pi, pws, ws.numel(), _stream(stream))
    _check(rc, "dsa_topk")


# Size of the fixed scratch array dsa_topk_noalloc uses, as the loaded library
# reports it (DSA_TOPK_NOALLOC_SCRATCH_BYTES in include/dsa.h).
TOPK_NOALLOC_SCRATCH_BYTES = int(_lib.dsa_topk_noalloc_scratch_bytes())


def topk_noalloc(scores, n_eligible, K, idx, stream=None):
    """dsa_topk without a workspace, for callers that may not allocate device
    memory: the scratch is a fixed array inside the library, shared by every
    call (calls that overlap on the GPU race)."""
    Nq, ld = scores.shape
    K = int(K)
    a = _Args().add(scores, "scores", _F32).add(n_eligible, "n_eligible", _I32, Nq)
    a.add(idx, "idx", _I32, Nq * K)
    ps, pn, pi = a.ptrs()
    rc = _lib.dsa_topk_noalloc(ps, ld, pn, Nq, K, pi, _stream(stream))
    _check(rc, "dsa_topk_noalloc")


def sparse_attn_decode(layout: PagedLayout, q, k_pool, v_pool, idx, sm_scale, out, lse, ws,
                       stream=None):
    B, Hq, Dqk = q.shape
    Dv, K = out.shape[2], idx.shape[1]
    ks, vs = k_pool.shape[-1], v_pool.shape[-1]
    a = _Args(layout).add(q, "q", _BF16).add(k_pool, "k_pool", _BF16, _rows(layout, ks))
    a.add(v_pool, "v_pool", _BF16, _rows(layout, vs)).add(idx, "idx", _I32, B * K)
    a.add(out, "out", _BF16, B * Hq * Dv).add(lse, "lse", _F32, B * Hq)
    a.add(ws, "ws", _WS)
    pq, pk, pv, pi, po, pl, pws = a.ptrs()
    rc = _lib.dsa_sparse_attn_decode(layout.c(), pq, pk, ks, pv, vs, Hq, Dqk, Dv, pi, K,
                                     float(sm_scale), po, pl, pws, ws.numel(), _stream(stream))
    _check(rc, "dsa_sparse_attn_decode")


def sparse_attn_prefill(layout: PagedLayout, q, k_pool, v_pool, idx, sm_scale, out, lse, ws,
                        q_seq=None, q_pos=None, stream=None):
    Nq, Hq, Dqk = q.shape
    Dv, K = out.shape[2], idx.shape[1]
    ks, vs = k_pool.shape[-1], v_pool.shape[-1]
    a = _Args(layout).add(q, "q", _BF16).add(k_pool, "k_pool", _BF16, _rows(layout, ks))
    a.add(v_pool, "v_pool", _BF16, _rows(layout, vs)).add(idx, "idx", _I32, Nq * K)
    a.add(out, "out", _BF16, Nq * Hq * Dv).add(lse, "lse", _F32, Nq * Hq)
    a.add(q_seq, "q_seq", _I32, Nq).add(q_pos, "q_pos", _I32, Nq).add(ws, "ws", _WS)
    pq, pk, pv, pi, po, pl, pseq, ppos, pws = a.ptrs()
    rc = _lib.dsa_sparse_attn_prefill(layout.c(), pq, pk, ks, pv, vs, Hq, Dqk, Dv, pseq, ppos, Nq,
                                      pi, K, float(sm_scale), po, pl, pws, ws.numel(),
                                      _stream(stream))
    _check(rc, "dsa_sparse_attn_prefill")


def cache_write_workspace_size() -> int:
    return int(_lib.dsa_cache_write_workspace_size())


def cache_write(layout: PagedLayout, seq, pos, ws, kv_new=None, kv_pool=None, kidx_new=None,
                kidx_pool=None, stream=None):
    """Store row i of kv_new / kidx_new at position pos[i] of sequence seq[i] of
    kv_pool / kidx_pool, through the block table (include/dsa.h, dsa_cache_write).

    kv_new [N, row_elems] bf16 into kv_pool [NB, bs, stride >= row_elems];
    kidx_new [N, D_i] into kidx_pool [NB, bs, D_i] (bf16 or FP8 E4M3).
    """
    N = int(seq.shape[0])
    row_elems = int(kv_new.shape[-1]) if kv_new is not None else 0
    stride = int(kv_pool.shape[-1]) if kv_pool is not None else 0
    D_i = int(kidx_new.shape[-1]) if kidx_new is not None else 0
    kdt = _elt_dtype(kidx_new) if kidx_new is not None else DSA_BF16
    ke = (kidx_new.element_size(),) if kidx_new is not None else _KEY
    a = _Args(layout).add(seq, "seq", _I32, N).add(pos, "pos", _I32, N)
    a.add(kv_new, "kv_new", _BF16, N * row_elems)
    a.add(kv_pool, "kv_pool", _BF16, _rows(layout, stride) if kv_new is not None else None)
    a.add(kidx_new, "kidx_new", _KEY, N * D_i)
    a.add(kidx_pool, "kidx_pool", ke, _rows(layout, D_i) if kidx_new is not None else None)
    a.add(ws, "ws", _WS)
    pseq, ppos, pkv, pkp, pin, pip, pws = a.ptrs()
    rc = _lib.dsa_cache_write(layout.c(), pseq, ppos, N, pkv, row_elems, pkp, stride, pin, D_i, kdt,
                              pip, pws, ws.numel(), _stream(stream))
    _check(rc, "dsa_cache_write")


def index_bounds_update_workspace_size() -> int:
    return int(_lib.dsa_index_bounds_update_workspace_size())


def index_bounds_update(layout: PagedLayout, kidx_pool, kbound_pool, ws, seq=None, pos=None,
                        stream=None):
    """Recompute the key bounds of the pages holding rows (seq[i], pos[i]), or of
    every cached page when seq and pos are None (include/dsa.h,
    dsa_index_bounds_update).  kbound_pool [NB, 2, D_i] in the keys' dtype."""
    D_i = int(kidx_pool.shape[-1])
    N = int(seq.shape[0]) if seq is not None else 0
    ke = (kidx_pool.element_size(),)
    a = _Args(layout).add(seq, "seq", _I32, N).add(pos, "pos", _I32, N)
    a.add(kidx_pool, "kidx_pool", ke, _rows(layout, D_i))
    a.add(kbound_pool, "kbound_pool", ke, layout.num_blocks * 2 * D_i).add(ws, "ws", _WS)
    pseq, ppos, pk, pb, pws = a.ptrs()
    rc = _lib.dsa_index_bounds_update(layout.c(), pseq, ppos, N, pk, D_i, _elt_dtype(kidx_pool),
                                      pb, pws, ws.numel(), _stream(stream))
    _check(rc, "dsa_index_bounds_update")


def index_score_bounded_workspace_size(B, H_i, D_i, ld, K) -> int:
    return int(_lib.dsa_index_score_bounded_workspace_size(B, H_i, D_i, ld, K))


def index_score_bounded(layout: PagedLayout, q_idx, w, kidx_pool, kbound_pool, K, scores, ws,
                        stream=None):
    """Decode indexer scores that leave out the tiles which cannot reach the
    top-K (include/dsa.h, dsa_index_score_bounded); dsa_topk over the row then
    selects exactly what it selects over dsa_index_score's row."""
    B, H_i, D_i = q_idx.shape
    ld = scores.shape[1]
    ke = (kidx_pool.element_size(),)
    a = _Args(layout).add(q_idx, "q_idx", _KEY).add(w, "w", _F32, B * H_i)
    a.add(kidx_pool, "kidx_pool", ke, _rows(layout, D_i))
    a.add(kbound_pool, "kbound_pool", ke, layout.num_blocks * 2 * D_i)
    a.add(scores, "scores", _F32, B * ld).add(ws, "ws", _WS)
    pq, pw, pk, pb, ps, pws = a.ptrs()
    rc = _lib.dsa_index_score_bounded(layout.c(), pq, pw, pk, _elt_dtype(kidx_pool), H_i, D_i, pb,
                                      int(K), ps, ld, pws, ws.numel(), _stream(stream))
    _check(rc, "dsa_index_score_bounded")


def index_bounded_stats(ws, stream=None):
    """(tiles left out, tiles bounded) by the last dsa_index_score_bounded call on ws."""
    sk, tot = ctypes.c_uint64(0), ctypes.c_uint64(0)
    rc = _lib.dsa_index_bounded_stats(ctypes.c_void_p(ws.data_ptr()), _stream(stream),
                                      ctypes.byref(sk), ctypes.byref(tot))
    _check(rc, "dsa_index_bounded_stats")
    return int(sk.value), int(tot.value)


def decode_step_workspace_size(B, H_i, D_i, ld, Hq, Dqk, Dv, K) -> int:
    return int(_lib.dsa_decode_step_workspace_size(B, H_i, D_i, ld, Hq, Dqk, Dv, K))


def prefill_step_workspace_size(Nq, H_i, D_i, ld, Hq, Dqk, Dv, K) -> int:
    return int(_lib.dsa_prefill_step_workspace_size(Nq, H_i, D_i, ld, Hq, Dqk, Dv, K))


def decode_step(layout: PagedLayout, k_new, k_pool, kidx_new, kidx_pool, q_idx, w, q, K, sm_scale,
                scores, idx, out, lse, ws, v_new=None, v_pool=None, stream=None):
    """One incremental decode step (include/dsa.h, dsa_decode_step): append each
    sequence's new K/V and indexer-key rows at position seq_lens[b] - 1, then
    score, select and attend.  v_pool None: V is the first Dv dims of the K row."""
    B, Hq, Dqk = q.shape
    a = _Args(layout)
    H_i, D_i = q_idx.shape[1], q_idx.shape[2]
    Dv, K, ld = out.shape[2], int(K), scores.shape[1]
    vp = k_pool if v_pool is None else v_pool
    ks, vs = k_pool.shape[-1], vp.shape[-1]
    ke = (q_idx.element_size(),)
    a.add(k_new, "k_new", _BF16, B * Dqk).add(k_pool, "k_pool", _BF16, _rows(layout, ks))
    a.add(v_new, "v_new", _BF16, B * Dv).add(vp, "v_pool", _BF16, _rows(layout, vs))
    a.add(kidx_new, "kidx_new", ke, B * D_i).add(kidx_pool, "kidx_pool", ke, _rows(layout, D_i))
    a.add(q_idx, "q_idx", _KEY).add(w, "w", _F32, B * H_i).add(q, "q", _BF16)
    a.add(scores, "scores", _F32, B * ld).add(idx, "idx", _I32, B * K)
    a.add(out, "out", _BF16, B * Hq * Dv).add(lse, "lse", _F32, B * Hq).add(ws, "ws", _WS)
    (pkn, pkp, pvn, pvp, pin, pip, pqi, pw, pq, ps, pi, po, pl, pws) = a.ptrs()
    rc = _lib.dsa_decode_step(layout.c(), pkn, pkp, ks, pvn, pvp, vs, pin, pip,
                              _elt_dtype(kidx_pool), pqi, pw, H_i, D_i, pq, Hq, Dqk, Dv, K,
                              float(sm_scale), ps, ld, pi, po, pl, pws, ws.numel(),
                              _stream(stream))
    _check(rc, "dsa_decode_step")


def prefill_step(layout: PagedLayout, seq, q_pos, n_eligible, k_new, k_pool, kidx_new, kidx_pool,
                 q_idx, w, q, K, sm_scale, scores, idx, out, lse, ws, v_new=None, v_pool=None,
                 stream=None):
    """A prompt (or a chunk after an existing prefix) of sequence `seq` in one
    call (include/dsa.h, dsa_prefill_step): its rows are written at q_pos, then
    scored, selected and attended."""
    Nq, Hq, Dqk = q.shape
    a = _Args(layout).add(q_pos, "q_pos", _I32, Nq).add(n_eligible, "n_eligible", _I32, Nq)
    H_i, D_i = q_idx.shape[1], q_idx.shape[2]
    Dv, K, ld = out.shape[2], int(K), scores.shape[1]
    vp = k_pool if v_pool is None else v_pool
    ks, vs = k_pool.shape[-1], vp.shape[-1]
    ke = (q_idx.element_size(),)
    a.add(k_new, "k_new", _BF16, Nq * Dqk).add(k_pool, "k_pool", _BF16, _rows(layout, ks))
    a.add(v_new, "v_new", _BF16, Nq * Dv).add(vp, "v_pool", _BF16, _rows(layout, vs))
    a.add(kidx_new, "kidx_new", ke, Nq * D_i).add(kidx_pool, "kidx_pool", ke, _rows(layout, D_i))
    a.add(q_idx, "q_idx", _KEY).add(w, "w", _F32, Nq * H_i).add(q, "q", _BF16)
    a.add(scores, "scores", _F32, Nq * ld).add(idx, "idx", _I32, Nq * K)
    a.add(out, "out", _BF16, Nq * Hq * Dv).add(lse, "lse", _F32, Nq * Hq).add(ws, "ws", _WS)
    (ppos, pn, pkn, pkp, pvn, pvp, pin, pip, pqi, pw, pq, ps, pi, po, pl, pws) = a.ptrs()
    rc = _lib.dsa_prefill_step(layout.c(), int(seq), ppos, pn, Nq, pkn, pkp, ks, pvn, pvp, vs,
                               pin, pip, _elt_dtype(kidx_pool), pqi, pw, H_i, D_i, pq, Hq, Dqk, Dv,
                               K, float(sm_scale), ps, ld, pi, po, pl, pws, ws.numel(),
                               _stream(stream))
    _check(rc, "dsa_prefill_step")


def prefill_step_chunked_workspace_size(Nq, H_i, D_i, ld, Hq, Dqk, Dv, K, chunk=0) -> int:
    return int(_lib.dsa_prefill_step_chunked_workspace_size(Nq, H_i, D_i, ld, Hq, Dqk, Dv, K,
                                                            int(chunk)))


def prefill_step_chunked(layout: PagedLayout, seq, q_pos, n_eligible, k_new, k_pool, kidx_new,
                         kidx_pool, q_idx, w, q, K, sm_scale, ld, idx, out, lse, ws, chunk=0,
                         v_new=None, v_pool=None, stream=None):
    """dsa_prefill_step without the score matrix (include/dsa.h,
    dsa_prefill_step_chunked): queries scored and selected `chunk` at a time
    (0: automatic) through a scratch in the workspace."""
    Nq, Hq, Dqk = q.shape
    a = _Args(layout).add(q_pos, "q_pos", _I32, Nq).add(n_eligible, "n_eligible", _I32, Nq)
    H_i, D_i = q_idx.shape[1], q_idx.shape[2]
    Dv, K, ld = out.shape[2], int(K), int(ld)
    vp = k_pool if v_pool is None else v_pool
    ks, vs = k_pool.shape[-1], vp.shape[-1]
    ke = (q_idx.element_size(),)
    a.add(k_new, "k_new", _BF16, Nq * Dqk).add(k_pool, "k_pool", _BF16, _rows(layout, ks))
    a.add(v_new, "v_new", _BF16, Nq * Dv).add(vp, "v_pool", _BF16, _rows(layout, vs))
    a.add(kidx_new, "kidx_new", ke, Nq * D_i).add(kidx_pool, "kidx_pool", ke, _rows(layout, D_i))
    a.add(q_idx, "q_idx", _KEY).add(w, "w", _F32, Nq * H_i).add(q, "q", _BF16)
    a.add(idx, "idx", _I32, Nq * K).add(out, "out", _BF16, Nq * Hq * Dv)
    a.add(lse, "lse", _F32, Nq * Hq).add(ws, "ws", _WS)
    (ppos, pn, pkn, pkp, pvn, pvp, pin, pip, pqi, pw, pq, pi, po, pl, pws) = a.ptrs()
    rc = _lib.dsa_prefill_step_chunked(layout.c(), int(seq), ppos, pn, Nq, pkn, pkp, ks, pvn, pvp,
                                       vs, pin, pip, _elt_dtype(kidx_pool), pqi, pw, H_i, D_i, pq,
                                       Hq, Dqk, Dv, K, float(sm_scale), ld, int(chunk), pi, po, pl,
                                       pws, ws.numel(), _stream(stream))
    _check(rc, "dsa_prefill_step_chunked")


def get_status(ws, clear: bool = True, stream=None) -> int:
    v = ctypes.c_int32(0)
    (pws,) = _Args().add(ws, "ws", _WS).ptrs()
    _check(_lib.dsa_get_status(pws, _stream(stream), ctypes.byref(v), int(clear)),
           "dsa_get_status")
    return int(v.value)


class Pipeline:
    """The three stages of one decode or prefill step with preallocated buffers.

    kind="decode": one query per sequence at position L_b - 1 (q [B, Hq, Dqk]).
    kind="prefill": Nq queries of sequence `prefill_seq` at positions q_pos (the
    indexer then shares key tiles across queries); prefill_seq=None scores
    queries of any sequences given by q_seq.
    Buffers (scores, idx, out, lse, workspaces) are allocated once through torch.
    """

    def __init__(self, layout: PagedLayout, *, kind: str, Nq: int, Hq: int, Dqk: int, Dv: int,
                 H_i: int, D_i: int, K: int, ld: Optional[int] = None, device="cuda",
                 prefill_seq: Optional[int] = 0):
        self.layout, self.kind, self.K = layout, kind, int(K)
        self.prefill_seq = prefill_seq
        self.Nq, self.Hq, self.Dqk, self.Dv = int(Nq), int(Hq), int(Dqk), int(Dv)
        # default row stride: the longest row rounded up to 4 scores, so that
        # every row starts on a 16-byte boundary (top-K then loads it with
        # 16-byte copies)
        self.ld = int(ld if ld is not None else (max(layout.max_seq_len, 1) + 3) // 4 * 4)
        self.scores = torch.empty((self.Nq, self.ld), dtype=torch.float32, device=device)
        self.idx = torch.empty((self.Nq, self.K), dtype=torch.int32, device=device)
        self.out = torch.empty((self.Nq, Hq, Dv), dtype=torch.bfloat16, device=device)
        self.lse = torch.empty((self.Nq, Hq), dtype=torch.float32, device=device)
        self.ws_index = workspace(index_score_workspace_size(self.Nq, H_i, D_i, self.ld), device)
        self.ws_topk = workspace(topk_workspace_size(self.Nq, self.ld, self.K), device)
        if kind == "decode":
            n = sparse_attn_decode_workspace_size(self.Nq, Hq, Dqk, Dv, self.K)
        else:
            n = sparse_attn_prefill_workspace_size(self.Nq, Hq, Dqk, Dv, self.K)
        self.ws_attn = workspace(n, device)

    def run(self, q, q_idx, w, kidx_pool, k_pool, v_pool, sm_scale, n_eligible=None, q_seq=None,
            q_pos=None, stream=None):
        if n_eligible is None:
            if self.kind != "decode":
                raise ValueError("prefill needs n_eligible (q_pos + 1)")
            n_eligible = self.layout.seq_lens
        if self.kind == "decode" or self.prefill_seq is None:
            index_score(self.layout, q_idx, w, kidx_pool, self.scores, self.ws_index, q_seq=q_seq,
                        q_pos=q_pos, stream=stream)
        else:
            index_score_prefill(self.layout, self.prefill_seq, q_idx, w, kidx_pool, self.scores,
                                self.ws_index, q_pos=q_pos, stream=stream)
        topk(self.scores, n_eligible, self.K, self.idx, self.ws_topk, stream=stream)
        if self.kind == "decode":
            sparse_attn_decode(self.layout, q, k_pool, v_pool, self.idx, sm_scale, self.out,
                               self.lse, self.ws_attn, stream=stream)
        else:
            sparse_attn_prefill(self.layout, q, k_pool, v_pool, self.idx, sm_scale, self.out,
                                self.lse, self.ws_attn, q_seq=q_seq, q_pos=q_pos, stream=stream)
        return self.out

    def status(self) -> int:
        return (get_status(self.ws_index) | get_status(self.ws_topk) | get_status(self.ws_attn))
