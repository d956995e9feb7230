"""Upload a :class:`workloads.Case` to a CUDA device as torch tensors.

Marshalling only (copies and dtype views), no arithmetic of the method.
"""
from __future__ import annotations

from types import SimpleNamespace

import numpy as np
import torch


def _t(a: np.ndarray, device, dtype=None) -> torch.Tensor:
    t = torch.from_numpy(np.ascontiguousarray(a))
    if dtype is not None:
        t = t.view(dtype)
    return t.to(device, non_blocking=False)


def upload(case, device="cuda", with_queries: bool = True) -> SimpleNamespace:
    """Device tensors of a case.  bf16 arrays become torch.bfloat16, E4M3 arrays
    torch.uint8 (raw codes); the latent cache uploads one pool used for K and V."""
    d = SimpleNamespace()
    d.block_table = _t(case.block_table, device)
    d.seq_lens = _t(case.seq_lens, device)
    d.q_seq = _t(case.q_seq, device)
    d.q_pos = _t(case.q_pos, device)
    d.n_elig = _t(case.n_elig, device)
    d.k_pool = _t(case.k_pool.view(np.int16), device, torch.bfloat16)
    d.v_pool = d.k_pool if case.latent else _t(case.v_pool.view(np.int16), device, torch.bfloat16)
    if case.idx_dtype == "bf16":
        d.kidx_pool = _t(case.kidx_pool.view(np.int16), device, torch.bfloat16)
    else:
        d.kidx_pool = _t(case.kidx_pool, device)
    if with_queries:
        upload_queries(case, d, device)
    return d


def upload_queries(case, d: SimpleNamespace, device="cuda") -> SimpleNamespace:
    d.q = _t(case.q.view(np.int16), device, torch.bfloat16)
    if case.idx_dtype == "bf16":
        d.q_idx = _t(case.q_idx.view(np.int16), device, torch.bfloat16)
    else:
        d.q_idx = _t(case.q_idx, device)
    d.w = _t(case.w, device)
    return d


def layout_of(case, d: SimpleNamespace):
    """The binding's PagedLayout for an uploaded case."""
    import sparse_attention_score_gb300 as dsa
    return dsa.PagedLayout(d.block_table, d.seq_lens, case.bs, case.num_blocks, case.max_len)
