"""Whole-step entry points through the C ABI against the oracle: incremental
decode steps (each appends its token's K/V and indexer-key rows, then scores,
selects and attends) and a prompt prefilled in two chunks.

Bar: scores and index sets bit-exact, attention within max-abs 1e-2 and
mean-abs 2e-3 of the fp64 oracle, every written cache row byte-exact.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from gpu_common import (assert_out_close, assert_scores_equal, code, fresh_layout, lib,
                        logical_rows, need_gpu, to_dev, to_host)

pytestmark = pytest.mark.gpu

LAT_SHAPES = dict(Hq=64, Dqk=576, Dv=512, latent=True, H_i=64, D_i=128, idx_dtype="fp8")


def _queries(rng, n, case):
    q = W.encode_bf16(rng.standard_normal((n, case.Hq, case.Dqk)).astype(np.float32))
    q_idx = W.encode_int(rng.integers(-8, 9, size=(n, case.H_i, case.D_i), dtype=np.int8),
                         case.idx_dtype)
    w = rng.integers(0, 5, size=(n, case.H_i)).astype(np.float32)
    return q, q_idx, w


@pytest.mark.parametrize("shapes,bs", [("latent", 64), ("tiny", 64), ("latent", 32),
                                       ("tiny", 128)])
def test_incremental_decode_steps(shapes, bs):
    """Three decode steps on a cache whose newest rows are not written yet:
    each step appends one row per sequence and must match the oracle on the
    cache as it stands after that step (pages of 64 positions, and of 32 and
    128, where the append lands at other in-page offsets and the indexer
    takes its CUDA-core path)."""
    need_gpu()
    dsa = lib()
    S = 3
    if shapes == "latent":
        c = W.make_case("steps", seed=700 + bs, seq_lens=(700, 2100, 4100), K=512, bs=bs,
                        **LAT_SHAPES)
    else:
        c = W.make_case("steps", seed=701 + bs, seq_lens=(300, 1000, 70, 4097), K=256, bs=bs,
                        Hq=16, Dqk=128, Dv=128, latent=False, H_i=4, D_i=64, idx_dtype="bf16")
    final = c.seq_lens.copy()
    B = c.B
    # device caches with the last S rows of every sequence overwritten by garbage
    kp, ip = c.k_pool.copy(), c.kidx_pool.copy()
    vp = None if c.latent else c.v_pool.copy()
    for b in range(B):
        for p in range(int(final[b]) - S, int(final[b])):
            page, row = c.block_table[b, p // c.bs], p % c.bs
            kp[page, row] = W.BF16_NAN
            ip[page, row] = W.BF16_NAN if c.idx_dtype == "bf16" else W.E4M3_NAN
            if vp is not None:
                vp[page, row] = W.BF16_NAN
    k_pool, kidx_pool = to_dev(kp), to_dev(ip)
    v_pool = None if vp is None else to_dev(vp)
    bt = to_dev(c.block_table)
    seq_lens = to_dev((final - S).astype(np.int32))
    lay = dsa.PagedLayout(bt, seq_lens, c.bs, c.num_blocks, int(final.max()))
    ld = int(final.max())
    scores = torch.empty((B, ld), dtype=torch.float32, device="cuda")
    idx = torch.empty((B, c.K), dtype=torch.int32, device="cuda")
    out = torch.empty((B, c.Hq, c.Dv), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((B, c.Hq), dtype=torch.float32, device="cuda")
    ws = dsa.workspace(dsa.decode_step_workspace_size(B, c.H_i, c.D_i, ld, c.Hq, c.Dqk, c.Dv, c.K))
    rng = np.random.default_rng(77)
    for s in range(S):
        L = (final - S + s + 1).astype(np.int32)
        seq_lens.copy_(torch.from_numpy(L))
        pages = c.block_table[np.arange(B), (L - 1) // c.bs]
        k_new = c.k_pool[pages, (L - 1) % c.bs]
        i_new = c.kidx_pool[pages, (L - 1) % c.bs]
        v_new = None if c.latent else c.v_pool[pages, (L - 1) % c.bs]
        q, q_idx, w = _queries(rng, B, c)
        dsa.decode_step(lay, to_dev(k_new), k_pool, to_dev(i_new), kidx_pool, to_dev(q_idx),
                        to_dev(w), to_dev(q), c.K, c.sm_scale, scores, idx, out, lse, ws,
                        v_new=None if v_new is None else to_dev(v_new), v_pool=v_pool)
        torch.cuda.synchronize()
        q_seq = np.arange(B, dtype=np.int32)
        s_ref = oracle.index_score(c.block_table, L, c.bs, c.num_blocks, q_seq, L - 1, q_idx, w,
                                   c.kidx_pool, code(c), ld)
        assert_scores_equal(scores.cpu().numpy(), s_ref, L)
        idx_ref = oracle.topk(s_ref, L, c.K)
        np.testing.assert_array_equal(idx.cpu().numpy(), idx_ref)
        o_ref, l_ref = oracle.sparse_attn(c.block_table, L, c.bs, c.num_blocks, q_seq, q,
                                          c.k_pool, c.v_pool, idx_ref, c.sm_scale, Dv=c.Dv)
        assert_out_close(out, lse, o_ref, l_ref, f"step {s}")
    np.testing.assert_array_equal(to_host(k_pool, c.k_pool), c.k_pool)
    np.testing.assert_array_equal(to_host(kidx_pool, c.kidx_pool), c.kidx_pool)
    if v_pool is not None:
        np.testing.assert_array_equal(to_host(v_pool, c.v_pool), c.v_pool)
    assert dsa.get_status(ws) == 0


def test_prefill_step_in_two_chunks():
    """A 600-token prompt prefilled as positions 0..399 then 400..599 into an
    empty cache: each call writes its rows, then scores, selects and attends
    causally over everything written so far."""
    need_gpu()
    dsa = lib()
    T = 600
    c = W.make_case("prefill-steps", seed=710, kind="prefill", T=T, K=256, **LAT_SHAPES)
    bt2, nb2 = fresh_layout(c, 31, 2)
    lay = dsa.PagedLayout(to_dev(bt2), to_dev(c.seq_lens), c.bs, nb2, T)
    k_pool = torch.zeros((nb2, c.bs, c.Dkv), dtype=torch.bfloat16, device="cuda")
    kidx_pool = torch.zeros((nb2, c.bs, c.D_i), dtype=torch.uint8, device="cuda")
    rows_k = logical_rows(c, c.k_pool, 0, T)
    rows_i = logical_rows(c, c.kidx_pool, 0, T)
    for lo, hi in ((0, 400), (400, 600)):
        n = hi - lo
        r = np.arange(lo, hi)
        scores = torch.empty((n, T), dtype=torch.float32, device="cuda")
        idx = torch.empty((n, c.K), dtype=torch.int32, device="cuda")
        out = torch.empty((n, c.Hq, c.Dv), dtype=torch.bfloat16, device="cuda")
        lse = torch.empty((n, c.Hq), dtype=torch.float32, device="cuda")
        ws = dsa.workspace(dsa.prefill_step_workspace_size(n, c.H_i, c.D_i, T, c.Hq, c.Dqk, c.Dv,
                                                           c.K))
        dsa.prefill_step(lay, 0, to_dev(c.q_pos[r]), to_dev(c.n_elig[r]), to_dev(rows_k[r]),
                         k_pool, to_dev(rows_i[r]), kidx_pool, to_dev(c.q_idx[r]), to_dev(c.w[r]),
                         to_dev(c.q[r]), c.K, c.sm_scale, scores, idx, out, lse, ws)
        torch.cuda.synchronize()
        s_ref = oracle.index_score(c.block_table, c.seq_lens, c.bs, c.num_blocks, c.q_seq[r],
                                   c.q_pos[r], c.q_idx[r], c.w[r], c.kidx_pool, code(c), T)
        assert_scores_equal(scores.cpu().numpy(), s_ref, c.n_elig[r])
        idx_ref = oracle.topk(s_ref, c.n_elig[r], c.K)
        np.testing.assert_array_equal(idx.cpu().numpy(), idx_ref)
        o_ref, l_ref = oracle.sparse_attn(c.block_table, c.seq_lens, c.bs, c.num_blocks,
                                          c.q_seq[r], c.q[r], c.k_pool, c.v_pool, idx_ref,
                                          c.sm_scale, Dv=c.Dv)
        assert_out_close(out, lse, o_ref, l_ref, f"chunk {lo}")
        assert dsa.get_status(ws) == 0


@pytest.mark.parametrize("chunk", [0, 16, 112, 1000])
def test_prefill_step_chunked_matches_the_oracle(chunk):
    """dsa_prefill_step_chunked: the prefill step without the score matrix.
    A 1300-token prompt (latent shapes, FP8 indexer, K = 256) is written,
    scored and selected in chunks of `chunk` queries through one scratch
    region (0: the automatic size, here one chunk; 16 and 112: many chunks and
    a ragged last one), then attended; index sets and outputs are compared with
    the oracle on every query, and with the staged step's."""
    need_gpu()
    dsa = lib()
    T = 1300
    c = W.make_case("prefill-chunked", seed=730, kind="prefill", T=T, K=256, **LAT_SHAPES)
    bt2, nb2 = fresh_layout(c, 37, 2)
    lay = dsa.PagedLayout(to_dev(bt2), to_dev(c.seq_lens), c.bs, nb2, T)
    rows_k = logical_rows(c, c.k_pool, 0, T)
    rows_i = logical_rows(c, c.kidx_pool, 0, T)
    r = np.arange(T)
    res = {}
    for mode in ("chunked", "staged"):
        k_pool = torch.zeros((nb2, c.bs, c.Dkv), dtype=torch.bfloat16, device="cuda")
        kidx_pool = torch.zeros((nb2, c.bs, c.D_i), dtype=torch.uint8, device="cuda")
        idx = torch.full((T, c.K), 7, dtype=torch.int32, device="cuda")
        out = torch.empty((T, c.Hq, c.Dv), dtype=torch.bfloat16, device="cuda")
        lse = torch.empty((T, c.Hq), dtype=torch.float32, device="cuda")
        args = (lay, 0, to_dev(c.q_pos), to_dev(c.n_elig), to_dev(rows_k), k_pool,
                to_dev(rows_i), kidx_pool, to_dev(c.q_idx), to_dev(c.w), to_dev(c.q), c.K,
                c.sm_scale)
        if mode == "chunked":
            ws = dsa.workspace(dsa.prefill_step_chunked_workspace_size(
                T, c.H_i, c.D_i, T, c.Hq, c.Dqk, c.Dv, c.K, chunk))
            dsa.prefill_step_chunked(*args, T, idx, out, lse, ws, chunk=chunk)
        else:
            scores = torch.empty((T, T), dtype=torch.float32, device="cuda")
            ws = dsa.workspace(dsa.prefill_step_workspace_size(T, c.H_i, c.D_i, T, c.Hq, c.Dqk,
                                                               c.Dv, c.K))
            dsa.prefill_step(*args, scores, idx, out, lse, ws)
        torch.cuda.synchronize()
        assert dsa.get_status(ws) == 0
        res[mode] = (idx.cpu().numpy(), out, lse)
    s_ref = oracle.index_score(c.block_table, c.seq_lens, c.bs, c.num_blocks, c.q_seq, c.q_pos,
                               c.q_idx, c.w, c.kidx_pool, code(c), T)
    idx_ref = oracle.topk(s_ref, c.n_elig, c.K)
    np.testing.assert_array_equal(res["chunked"][0], idx_ref)
    np.testing.assert_array_equal(res["chunked"][0], res["staged"][0])
    o_ref, l_ref = oracle.sparse_attn(c.block_table, c.seq_lens, c.bs, c.num_blocks, c.q_seq,
                                      c.q, c.k_pool, c.v_pool, idx_ref, c.sm_scale, Dv=c.Dv)
    assert_out_close(res["chunked"][1], res["chunked"][2], o_ref, l_ref, f"chunk {chunk}")
    assert torch.equal(res["chunked"][1], res["staged"][1])

