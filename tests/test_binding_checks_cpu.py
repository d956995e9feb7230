"""The binding refuses, before anything reaches the C ABI, tensors that would
send a kernel outside them: elements of the wrong size, fewer elements than
the call touches, host memory.  Runs on CPU: each case fails one check
(element size and count are checked before residency, so host tensors reach
every check)."""
import pytest
import torch

from gpu_common import lib

dsa = lib()


def _layout(nb=4, bs=64, B=2):
    bt = torch.arange(nb, dtype=torch.int32).reshape(B, nb // B)
    return dsa.PagedLayout(bt, torch.full((B,), 100, dtype=torch.int32), bs, nb, 128)


def test_topk_checks_element_size_count_and_residency():
    s = torch.zeros((3, 40), dtype=torch.float32)
    n = torch.full((3,), 40, dtype=torch.int32)
    idx = torch.empty((3, 8), dtype=torch.int32)
    ws = torch.zeros(1024, dtype=torch.uint8)
    with pytest.raises(TypeError, match="scores"):
        dsa.topk(s.half(), n, 8, idx, ws)
    with pytest.raises(TypeError, match="n_eligible"):
        dsa.topk(s, n.long(), 8, idx, ws)
    with pytest.raises(ValueError, match="n_eligible"):
        dsa.topk(s, n[:2], 8, idx, ws)
    with pytest.raises(ValueError, match="idx"):
        dsa.topk(s, n, 9, idx, ws)                 # K = 9 needs 27 entries, idx has 24
    with pytest.raises(TypeError, match="ws"):
        dsa.topk(s, n, 8, idx, ws.float())         # sizes are passed in bytes
    with pytest.raises(ValueError, match="CUDA"):
        dsa.topk(s, n, 8, idx, ws)
    with pytest.raises(ValueError, match="CUDA"):
        dsa.topk_noalloc(s, n, 8, idx)


def test_attention_checks_operands_against_the_layout():
    lay = _layout()
    B, Hq, Dqk, Dv, K = 2, 4, 64, 64, 16
    q = torch.zeros((B, Hq, Dqk), dtype=torch.bfloat16)
    pool = torch.zeros((4, 64, Dqk), dtype=torch.bfloat16)
    idx = torch.zeros((B, K), dtype=torch.int32)
    out = torch.empty((B, Hq, Dv), dtype=torch.bfloat16)
    lse = torch.empty((B, Hq), dtype=torch.float32)
    ws = torch.zeros(4096, dtype=torch.uint8)
    with pytest.raises(TypeError, match="q"):
        dsa.sparse_attn_decode(lay, q.float(), pool, pool, idx, 0.1, out, lse, ws)
    with pytest.raises(ValueError, match="k_pool"):
        dsa.sparse_attn_decode(lay, q, pool[:3], pool, idx, 0.1, out, lse, ws)  # 3 of 4 pages
    with pytest.raises(ValueError, match="idx"):
        dsa.sparse_attn_decode(lay, q, pool, pool, idx[:1], 0.1, out, lse, ws)
    with pytest.raises(ValueError, match="out"):
        dsa.sparse_attn_decode(lay, q, pool, pool, idx, 0.1, out[:, :2], lse, ws)
    with pytest.raises(ValueError, match="q_pos"):
        dsa.sparse_attn_prefill(lay, q, pool, pool, idx, 0.1, out, lse, ws,
                                q_pos=torch.zeros(1, dtype=torch.int32))
    with pytest.raises(ValueError, match="CUDA"):
        dsa.sparse_attn_decode(lay, q, pool, pool, idx, 0.1, out, lse, ws)


def test_index_score_and_cache_write_checks():
    lay = _layout()
    Nq, H_i, D_i, ld = 2, 4, 64, 128
    q_idx = torch.zeros((Nq, H_i, D_i), dtype=torch.bfloat16)
    w = torch.zeros((Nq, H_i), dtype=torch.float32)
    kidx = torch.zeros((4, 64, D_i), dtype=torch.bfloat16)
    scores = torch.empty((Nq, ld), dtype=torch.float32)
    ws = torch.zeros(1024, dtype=torch.uint8)
    with pytest.raises(TypeError, match="kidx_pool"):      # keys of another element size
        dsa.index_score(lay, q_idx, w, kidx.view(torch.uint8), scores, ws)
    with pytest.raises(ValueError, match="w"):
        dsa.index_score(lay, q_idx, w[:1], kidx, scores, ws)
    with pytest.raises(ValueError, match="q_seq"):
        dsa.index_score(lay, q_idx, w, kidx, scores, ws, q_seq=torch.zeros(1, dtype=torch.int32))
    with pytest.raises(ValueError, match="CUDA"):
        dsa.index_score(lay, q_idx, w, kidx, scores, ws)
    seq = torch.zeros(3, dtype=torch.int32)
    pos = torch.arange(3, dtype=torch.int32)
    rows = torch.zeros((3, Dv := 64), dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="kv_pool"):
        dsa.cache_write(lay, seq, pos, ws, kv_new=rows, kv_pool=torch.zeros((2, 64, Dv),
                                                                            dtype=torch.bfloat16))
    with pytest.raises(ValueError, match="kv_new"):
        dsa.cache_write(lay, seq, pos, ws, kv_new=rows[:2],
                        kv_pool=torch.zeros((4, 64, Dv), dtype=torch.bfloat16))
