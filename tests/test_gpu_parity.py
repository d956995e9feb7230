"""GPU parity of the CUDA path (through the C ABI) against the CPU oracle, on
small seeded cases that still span several tiles and ragged tails.

Bar: scores and index sets bit-exact; attention within max-abs 1e-2 and
mean-abs 2e-3 of the fp64 oracle.  Each stage is also fed the oracle's own
upstream result, so that a failure is pinned to one stage.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from gpu_common import (DevicePipeline, assert_out_close, assert_scores_equal, check_topk_definition,
                        need_gpu, oracle_attn, oracle_scores)

pytestmark = pytest.mark.gpu

TINY_SHAPES = dict(Hq=16, Dqk=128, Dv=128, latent=False, H_i=4, D_i=64, idx_dtype="bf16")
LAT_SHAPES = dict(Hq=64, Dqk=576, Dv=512, latent=True, H_i=64, D_i=128, idx_dtype="fp8")


def _full_check(case, ld=None):
    need_gpu()
    g = DevicePipeline(case, ld=ld)
    s = g.scores().cpu().numpy()
    s_ref = oracle_scores(case, ld=s.shape[1])
    assert_scores_equal(s, s_ref, case.n_elig)
    idx = g.topk().cpu().numpy()
    idx_ref = oracle.topk(s_ref, case.n_elig, case.K)
    np.testing.assert_array_equal(idx, idx_ref)
    out, lse = g.attn()
    out_ref, lse_ref = oracle_attn(case, idx_ref)
    assert_out_close(out, lse, out_ref, lse_ref, case.name)
    assert g.status() == 0
    return g


@pytest.mark.parametrize("lens", [(4096,), (1, 63, 64, 65, 1000, 3000)])
def test_tiny_shapes_pipeline(lens):
    c = W.make_case("tiny", seed=100 + len(lens), seq_lens=lens, K=256, **TINY_SHAPES)
    _full_check(c)


@pytest.mark.parametrize("lens,K", [((100, 2048, 2049, 5000, 8191), 2048),
                                    ((700, 129, 4097), 64)])
def test_latent_shapes_pipeline(lens, K):
    c = W.make_case("latent", seed=200 + K, seq_lens=lens, K=K, **dict(LAT_SHAPES))
    _full_check(c)


@pytest.mark.parametrize("bs,shapes,K", [
    (1, "tiny", 64), (16, "tiny", 256), (256, "latent", 512), (1024, "latent", 2048),
    (48, "latent", 300),
], ids=["bs1-tiny", "bs16-tiny", "bs256-latent", "bs1024-latent", "bs48-latent"])
def test_pipeline_page_sizes(bs, shapes, K):
    """Pages of other sizes than 64 positions (the tensor-core indexer's
    page), down to one position and up to the largest size the layout takes:
    the page table is read per position in every stage, and the indexer
    takes its CUDA-core path."""
    sh = TINY_SHAPES if shapes == "tiny" else LAT_SHAPES
    c = W.make_case(f"bs{bs}", seed=350 + bs, seq_lens=(bs * 3 + 5, 2 * K + 1, 70), bs=bs, K=K,
                    **dict(sh))
    _full_check(c)


def test_latent_bf16_indexer_and_extra_ld():
    shapes = dict(LAT_SHAPES, idx_dtype="bf16")
    c = W.make_case("latent-bf16", seed=301, seq_lens=(1500, 333), K=512, extra_pages=3, **shapes)
    _full_check(c, ld=c.max_len + 77)


def test_prefill_small_all_rows():
    c = W.make_case("prefill-small", seed=400, kind="prefill", T=300, K=64, **LAT_SHAPES)
    _full_check(c)


def test_prefill_sampled_rows_k2048():
    need_gpu()
    c = W.make_case("prefill-2600", seed=401, kind="prefill", T=2600, K=2048, **LAT_SHAPES)
    g = DevicePipeline(c)
    out, lse = g.all()
    rows = np.array([0, 1, 63, 64, 1000, 2046, 2047, 2048, 2049, 2500, 2599])
    s_ref = oracle_scores(c, rows=rows)
    assert_scores_equal(g.pipe.scores.cpu().numpy()[rows], s_ref, c.n_elig[rows])
    idx_ref = oracle.topk(s_ref, c.n_elig[rows], c.K)
    np.testing.assert_array_equal(g.pipe.idx.cpu().numpy()[rows], idx_ref)
    out_ref, lse_ref = oracle_attn(c, idx_ref, rows=rows)
    assert_out_close(out[rows], lse[rows], out_ref, lse_ref, "prefill rows")
    assert g.status() == 0


def test_topk_stage_alone_heavy_ties_and_edges():
    need_gpu()
    import sparse_attention_score_gb300 as dsa
    rng = np.random.default_rng(5)
    Nq, ld = 9, 5000
    s = rng.integers(0, 4, size=(Nq, ld)).astype(np.float32)
    s[1] = rng.standard_normal(ld).astype(np.float32)
    s[2] = 0.0
    s[2, ::2] = -0.0                       # -0 ties +0
    s[3, :] = -np.inf
    s[4] = np.float32(7.0)
    n = np.array([5000, 4999, 3000, 100, 17, 0, 1, 2048, 2049], np.int32)
    for K in (1, 5, 2048, 4096):
        st = torch.from_numpy(s).cuda()
        ne = torch.from_numpy(n).cuda()
        idx = torch.empty((Nq, K), dtype=torch.int32, device="cuda")
        ws = dsa.workspace(dsa.topk_workspace_size(Nq, ld, K))
        dsa.topk(st, ne, K, idx, ws)
        got = idx.cpu().numpy()
        want = oracle.topk(s, n, K)
        np.testing.assert_array_equal(got, want)
        for r in range(Nq):
            check_topk_definition(s[r], int(n[r]), K, got[r])
        assert dsa.get_status(ws) == 0


def test_attention_stage_alone_on_oracle_indices():
    need_gpu()
    c = W.make_case("attn-only", seed=500, seq_lens=(3000, 70, 2100), K=2048, **LAT_SHAPES)
    g = DevicePipeline(c)
    rng = np.random.default_rng(1)
    idx = np.full((c.B, c.K), -1, np.int32)
    for b in range(c.B):
        L = int(c.seq_lens[b])
        pick = np.sort(rng.choice(L, size=min(L, c.K - 37), replace=False))
        idx[b, :len(pick)] = pick
    out, lse = g.attn(torch.from_numpy(idx).cuda())
    out_ref, lse_ref = oracle_attn(c, idx)
    assert_out_close(out, lse, out_ref, lse_ref, "attn-only")


def test_edge_cases_k1_zero_weights_empty_row():
    need_gpu()
    c = W.make_case("edges", seed=600, seq_lens=(500, 1, 64), K=1, **TINY_SHAPES)
    _full_check(c)
    c2 = W.make_case("zero-w", seed=601, seq_lens=(900, 300), K=256, **TINY_SHAPES)
    c2.w[:] = 0.0
    g = _full_check(c2)
    idx = g.pipe.idx.cpu().numpy()
    assert idx[0].tolist() == list(range(256))       # all scores tie at 0
    # an empty row (no eligible position) gives -1 indices, zero output and -inf lse
    c3 = W.make_case("empty", seed=602, seq_lens=(200,), K=16, **TINY_SHAPES)
    g3 = DevicePipeline(c3)
    g3.scores()
    g3.topk(n_elig=torch.zeros(1, dtype=torch.int32, device="cuda"))
    assert np.all(g3.pipe.idx.cpu().numpy() == -1)
    out, lse = g3.attn()
    assert torch.all(out == 0) and torch.all(torch.isinf(lse)) and torch.all(lse < 0)


def test_block_table_permutation_gives_identical_results():
    need_gpu()
    c = W.make_case("perm", seed=700, seq_lens=(1200, 2500), K=512, **LAT_SHAPES)
    g1 = DevicePipeline(c)
    o1, l1 = g1.all()
    perm = np.random.default_rng(9).permutation(c.num_blocks)
    c2 = W.make_case("perm", seed=700, seq_lens=(1200, 2500), K=512, **LAT_SHAPES)
    kp = np.empty_like(c2.k_pool)
    kp[perm] = c2.k_pool
    ki = np.empty_like(c2.kidx_pool)
    ki[perm] = c2.kidx_pool
    c2.k_pool = c2.v_pool = kp
    c2.kidx_pool = ki
    c2.block_table = np.where(c2.block_table >= 0, perm[np.maximum(c2.block_table, 0)],
                              -1).astype(np.int32)
    g2 = DevicePipeline(c2)
    o2, l2 = g2.all()
    assert torch.equal(g1.pipe.idx, g2.pipe.idx)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_bad_block_id_is_flagged_not_faulted():
    need_gpu()
    import sparse_attention_score_gb300 as dsa
    c = W.make_case("bad-block", seed=800, seq_lens=(640, 300), K=64, **TINY_SHAPES)
    c.block_table[0, 3] = c.num_blocks + 1000      # positions 192..255 of sequence 0
    g = DevicePipeline(c)
    s = g.scores().cpu().numpy()
    assert np.all(s[0, 192:256] == -np.inf) and np.all(np.isfinite(s[0, :192]))
    assert dsa.get_status(g.pipe.ws_index) & dsa.STATUS_BAD_BLOCK
    # attention on an index past the sequence end: row skipped, flagged
    idx = np.full((c.B, c.K), -1, np.int32)
    idx[0, :3] = [5, 10, 639]
    idx[1, :3] = [0, 299, 300]                      # 300 >= L_1
    out, lse = g.attn(torch.from_numpy(idx).cuda())
    assert dsa.get_status(g.pipe.ws_attn) & dsa.STATUS_BAD_INDEX
    ok = idx.copy()
    ok[1, 2] = -1
    c.block_table[0, 3] = 0                          # oracle needs a valid table for row 0
    out_ref, lse_ref = oracle_attn(c, ok)
    assert_out_close(out[1:], lse[1:], out_ref[1:], lse_ref[1:], "skipped row")


def test_fp8_indexer_adversarial_exactness():
    """Integer dot products up to +-8192 per head (14 significant bits) with
    mixtures of large and small products: the FP8 tensor-core accumulation must
    keep every bit, so scores stay bit-exact."""
    need_gpu()
    c = W.make_case("fp8-adv", seed=900, seq_lens=(1100, 700, 257), K=128, **LAT_SHAPES)
    rng = np.random.default_rng(2)
    D = c.D_i
    pats = [np.full(D, 8), np.full(D, -8), np.r_[np.full(64, 8), np.full(64, 1)],
            np.r_[np.full(64, 8), np.full(64, -8)], np.r_[np.full(127, 8), [1]],
            np.tile([8, 1], D // 2), np.tile([8, -8, 1, 1], D // 4), np.full(D, 1)]
    q = np.empty((c.Nq, c.H_i, D), np.int64)
    for r in range(c.Nq):
        for h in range(c.H_i):
            q[r, h] = pats[(r + h) % len(pats)] * (1 if h % 3 else -1)
    k = np.empty(c.kidx_pool.shape, np.int64)
    flat = k.reshape(-1, D)
    for i in range(flat.shape[0]):
        flat[i] = pats[rng.integers(len(pats))] if i % 5 else rng.integers(-8, 9, D)
    c.q_idx = W.encode_int(q, "fp8")
    c.kidx_pool = W.encode_int(k, "fp8")
    c.w[:] = 4.0
    g = DevicePipeline(c)
    s = g.scores().cpu().numpy()
    s_ref = oracle_scores(c, ld=s.shape[1])
    assert s_ref[np.isfinite(s_ref)].max() >= 8192 * 4
    assert_scores_equal(s, s_ref, c.n_elig)


@pytest.mark.parametrize("Nq,K,cs", [(64, 512, 2), (32, 2048, 4), (16, 2048, 8), (4, 2048, 16),
                                     (8, 2048, 16)])
def test_attention_cluster_merge_splits(Nq, K, cs):
    """Every query split evenly over cs CTAs of one thread-block cluster (on a
    152-SM GB300: 128 CTAs of two or four 128-row tiles, or 64 and 128 CTAs
    of one tile for 16 per query), merged inside the attention kernel:
    outputs and lse against the oracle, with sequences shorter than one
    CTA's share (some CTAs of a cluster hold no usable row) and one of a
    single position.  The launch count shows whether the merge kernel ran:
    not for clusters of 2 and 4; splits over eight or 16 CTAs are merged by
    it (clusters of eight such CTAs are not all resident at once on a GB300,
    and clusters of 16 measured slower than the merge kernel)."""
    need_gpu()
    import sparse_attention_score_gb300 as dsa
    rng = np.random.default_rng(1200 + cs)
    lens = rng.integers(K // 2, 3 * K, size=Nq)
    lens[:4] = (1, 100, K // 4 + 3, K)
    c = W.make_case("cluster", seed=1300 + cs, seq_lens=tuple(int(x) for x in lens), K=K,
                    **LAT_SHAPES)
    idx = np.full((c.Nq, K), -1, np.int32)
    for b in range(c.Nq):
        L = int(c.seq_lens[b])
        n = min(K, L)
        idx[b, :n] = np.sort(rng.choice(L, size=n, replace=False))
    g = DevicePipeline(c)
    ix = torch.from_numpy(idx).cuda()
    g.attn(ix)  # first call: one-off per-process setup
    torch.cuda.synchronize()
    n0 = dsa.launch_count()
    out, lse = g.attn(ix)
    torch.cuda.synchronize()
    launches = dsa.launch_count() - n0
    out_ref, lse_ref = oracle_attn(c, idx)
    assert_out_close(out, lse, out_ref, lse_ref, f"cluster{cs}")
    assert g.status() == 0
    if torch.cuda.get_device_properties(0).multi_processor_count == 152:
        assert launches == (1 if cs <= 4 else 2), launches


@pytest.mark.parametrize("Nq,K,launches", [(1, 64, 1), (1, 256, 1), (3, 512, 2), (1, 2048, 2)],
                         ids=["S2-cluster", "S8-cluster", "S16-combine", "S64-combine"])
def test_cuda_core_attention_split_merges(Nq, K, launches):
    """The CUDA-core attention (16 heads x 128, separate K and V pools) splits
    each query's rows over S = min(304 / Nq, K / 32, 64) CTAs: with S <= 8
    they form a thread-block cluster and merge inside the kernel (one
    launch), otherwise the combine kernel merges them (two).  Outputs and lse
    against the oracle, with a sequence shorter than one split's share."""
    need_gpu()
    import sparse_attention_score_gb300 as dsa
    rng = np.random.default_rng(1400 + K + Nq)
    lens = [int(x) for x in rng.integers(K, 3 * K, size=Nq)]
    lens[0] = max(1, K // 9)
    c = W.make_case("split", seed=1500 + K, seq_lens=tuple(lens), K=K, **TINY_SHAPES)
    idx = np.full((c.Nq, K), -1, np.int32)
    for b in range(c.Nq):
        L = int(c.seq_lens[b])
        n = min(K, L)
        idx[b, :n] = np.sort(rng.choice(L, size=n, replace=False))
    g = DevicePipeline(c)
    ix = torch.from_numpy(idx).cuda()
    g.attn(ix)
    torch.cuda.synchronize()
    n0 = dsa.launch_count()
    out, lse = g.attn(ix)
    torch.cuda.synchronize()
    got = dsa.launch_count() - n0
    out_ref, lse_ref = oracle_attn(c, idx)
    assert_out_close(out, lse, out_ref, lse_ref, f"split K={K}")
    assert g.status() == 0
    if torch.cuda.get_device_properties(0).multi_processor_count == 152:
        assert got == launches, got


def test_attention_running_max_rescale_path():
    """Scores that jump by far more than 2^8 from one 128-row tile to the next
    (for even heads only) force the O rescale in the online softmax."""
    need_gpu()
    c = W.make_case("rescale", seed=950, seq_lens=(700, 1500), K=512, **LAT_SHAPES)
    kp = c.k_pool.astype(np.uint16).copy()
    lvl = [0.0, 0.25, 0.5, 1.0]
    for b in range(c.B):
        L = int(c.seq_lens[b])
        for p in range(L):
            page, slot = c.block_table[b, p // c.bs], p % c.bs
            val = lvl[min(p // 128, 3)]
            row = np.full(c.Dqk, val, np.float32)
            row[c.Dv:] = val
            # keep V informative: first dims carry the position
            row[0] = (p % 97) / 97.0
            kp[page, slot] = W.encode_bf16(row)
    c.k_pool = c.v_pool = kp
    qf = np.ones((c.Nq, c.Hq, c.Dqk), np.float32)
    qf[:, 1::2, :] = -1.0
    qf[:, :, 0] = 0.0
    c.q = W.encode_bf16(qf)
    g = DevicePipeline(c)
    idx = np.full((c.B, c.K), -1, np.int32)
    for b in range(c.B):
        n = min(c.K, int(c.seq_lens[b]))
        idx[b, :n] = np.arange(n)
    out, lse = g.attn(torch.from_numpy(idx).cuda())
    out_ref, lse_ref = oracle_attn(c, idx)
    assert_out_close(out, lse, out_ref, lse_ref, "rescale")
    assert g.status() == 0


@pytest.mark.parametrize("K", [1, 2047, 2048, 9000])
def test_topk_long_rows_ties_across_blocks(K):
    """Rows longer than one shared-memory block take the block + merge path;
    heavy ties straddle block boundaries, so the lower-position rule must hold
    across blocks."""
    need_gpu()
    import sparse_attention_score_gb300 as dsa
    rng = np.random.default_rng(11 + K)
    Nq, ld = 5, 150001
    s = rng.integers(0, 3, size=(Nq, ld)).astype(np.float32)
    s[1] = rng.standard_normal(ld).astype(np.float32)
    s[2, :] = 5.0                                  # one value everywhere
    s[3, 100000:] = 9.0                            # winners all in later blocks
    n = np.array([150001, 149000, 120000, 150001, 60000], np.int32)
    st, ne = torch.from_numpy(s).cuda(), torch.from_numpy(n).cuda()
    idx = torch.empty((Nq, K), dtype=torch.int32, device="cuda")
    ws = dsa.workspace(dsa.topk_workspace_size(Nq, ld, K))
    dsa.topk(st, ne, K, idx, ws)
    got = idx.cpu().numpy()
    np.testing.assert_array_equal(got, oracle.topk(s, n, K))
    assert dsa.get_status(ws) == 0


@pytest.mark.parametrize("ld,K", [(100000, 20000), (200000, 65536)])
def test_topk_row_at_a_time_path_large_k(ld, K):
    """K too large for the blocks' winners to fit one merge (K x blocks >
    49152, up to the largest K the call takes): the row-at-a-time radix
    kernel.  Ties, a constant row, NaN / +-inf / -0, rows shorter than K and
    an empty row, against the oracle."""
    need_gpu()
    import sparse_attention_score_gb300 as dsa
    assert dsa.topk_workspace_size(4, ld, K) == 256      # no block scratch: that path
    rng = np.random.default_rng(ld + K)
    Nq = 4
    s = rng.integers(0, 5, size=(Nq, ld)).astype(np.float32)
    s[1] = rng.standard_normal(ld).astype(np.float32)
    s[1, rng.choice(ld, 40, replace=False)] = np.array(
        [np.nan] * 10 + [np.inf] * 10 + [-np.inf] * 10 + [-0.0] * 10, np.float32)
    s[2, :] = 2.0
    n = np.array([ld, ld - 7, K // 2, 0], np.int32)
    st, ne = torch.from_numpy(s).cuda(), torch.from_numpy(n).cuda()
    idx = torch.full((Nq, K), 7, dtype=torch.int32, device="cuda")
    ws = dsa.workspace(dsa.topk_workspace_size(Nq, ld, K))
    dsa.topk(st, ne, K, idx, ws)
    # the oracle takes only numbers; NaN ranks below every value, and row 1
    # keeps K of its ~ld finite scores, so neither NaN nor -inf is reached
    ref = oracle.topk(np.where(np.isnan(s), np.float32(-1e30), s), n, K)
    np.testing.assert_array_equal(idx.cpu().numpy(), ref)
    assert dsa.get_status(ws) == 0


def test_topk_long_rows_short_rows_and_special_values():
    """The block + merge path on rows that leave blocks empty or short: no
    eligible position, fewer than K (then no block bounds the merge), exactly
    K across a block boundary, NaN (ranks below every value), -inf and -0
    against +0, and winners only in the last block.  ld is odd, so every row
    after the first starts off a 16-byte boundary."""
    need_gpu()
    import sparse_attention_score_gb300 as dsa
    rng = np.random.default_rng(4242)
    Nq, ld, K = 8, 100003, 2048
    s = rng.integers(0, 3, size=(Nq, ld)).astype(np.float32)
    s[2, ::7] = np.nan
    s[3, ::5] = -np.inf
    s[3, 1::5] = -0.0
    s[4, :] = np.nan
    s[4, 5000:5010] = 1.0
    s[5, :] = -0.0
    s[5, 1::2] = 0.0
    s[6, 90000:] = 7.0
    n = np.array([0, 100, 1500, ld, 40000, 60000, ld, K], np.int32)
    st, ne = torch.from_numpy(s).cuda(), torch.from_numpy(n).cuda()
    idx = torch.empty((Nq, K), dtype=torch.int32, device="cuda")
    ws = dsa.workspace(dsa.topk_workspace_size(Nq, ld, K))
    dsa.topk(st, ne, K, idx, ws)
    got = idx.cpu().numpy()
    # NaN ranks below every value: in rows without -inf a finite score below
    # all others orders the same, and the oracle takes only numbers
    ref = oracle.topk(np.where(np.isnan(s), np.float32(-1e30), s), n, K)
    np.testing.assert_array_equal(got, ref)
    assert dsa.get_status(ws) == 0
    # the same workspace again, after a call of another shape left data in it
    s2 = rng.standard_normal((3, 70001)).astype(np.float32)
    n2 = np.array([70001, 33, 50000], np.int32)
    idx2 = torch.empty((3, 512), dtype=torch.int32, device="cuda")
    ws2 = dsa.workspace(max(dsa.topk_workspace_size(3, 70001, 512), ws.numel()))
    dsa.topk(torch.from_numpy(s2).cuda(), torch.from_numpy(n2).cuda(), 512, idx2, ws2)
    dsa.topk(st, ne, K, idx, ws2)
    np.testing.assert_array_equal(idx2.cpu().numpy(), oracle.topk(s2, n2, 512))
    np.testing.assert_array_equal(idx.cpu().numpy(), ref)


def test_topk_more_rows_than_one_grid_dimension_holds():
    """70,000 rows (one CTA each) exceed the 65,535 blocks of a grid's y and z
    dimensions; the rows run on x."""
    need_gpu()
    import sparse_attention_score_gb300 as dsa
    rng = np.random.default_rng(70000)
    Nq, ld, K = 70000, 64, 8
    s = rng.integers(0, 6, size=(Nq, ld)).astype(np.float32)
    n = rng.integers(0, ld + 1, size=Nq).astype(np.int32)
    idx = torch.empty((Nq, K), dtype=torch.int32, device="cuda")
    ws = dsa.workspace(dsa.topk_workspace_size(Nq, ld, K))
    dsa.topk(torch.from_numpy(s).cuda(), torch.from_numpy(n).cuda(), K, idx, ws)
    np.testing.assert_array_equal(idx.cpu().numpy(), oracle.topk(s, n, K))
    assert dsa.get_status(ws) == 0


@pytest.mark.parametrize("ld,K", [(20000, 2048), (65536, 4096), (4097, 7)])
def test_topk_single_block_rows_ties_and_edges(ld, K):
    """Rows of 4K..64K positions (one shared-memory block each): heavy ties,
    empty, short and exact-K rows, one value everywhere, -0 against +0, and
    winners only at the end of the row."""
    need_gpu()
    import sparse_attention_score_gb300 as dsa
    rng = np.random.default_rng(ld + K)
    Nq = 9
    s = rng.integers(0, 4, size=(Nq, ld)).astype(np.float32)
    s[1] = rng.standard_normal(ld).astype(np.float32)
    s[2, :] = 5.0
    s[3, ld - ld // 9:] = 9.0
    s[4, ::3] = -0.0
    n = np.array([ld, ld - 1, ld // 2, ld, 4096, 0, 1, K, K + 1], np.int32)
    st, ne = torch.from_numpy(s).cuda(), torch.from_numpy(n).cuda()
    idx = torch.empty((Nq, K), dtype=torch.int32, device="cuda")
    ws = dsa.workspace(dsa.topk_workspace_size(Nq, ld, K))
    dsa.topk(st, ne, K, idx, ws)
    got = idx.cpu().numpy()
    np.testing.assert_array_equal(got, oracle.topk(s, n, K))
    assert dsa.get_status(ws) == 0


def test_prefill_indexer_both_entry_points():
    """The prefill form (queries of one sequence sharing key tiles) and the
    general form (explicit q_seq) give the oracle's scores bit for bit."""
    need_gpu()
    c = W.make_case("prefill-idx", seed=990, kind="prefill", T=1300, K=256, **LAT_SHAPES)
    g = DevicePipeline(c)
    s_ref = oracle_scores(c)
    assert_scores_equal(g.scores().cpu().numpy(), s_ref, c.n_elig)
    assert_scores_equal(g.scores_general().cpu().numpy(), s_ref, c.n_elig)
    assert g.status() == 0


def test_prefill_indexer_query_subset_ragged_block():
    """37 queries at scattered positions (a ragged last block of 16)."""
    need_gpu()
    rows = np.sort(np.random.default_rng(4).choice(3000, 37, replace=False))
    c = W.make_case("prefill-sub", seed=991, kind="prefill", T=3000, K=512, q_rows=rows,
                    **LAT_SHAPES)
    g = DevicePipeline(c)
    s_ref = oracle_scores(c)
    assert_scores_equal(g.scores().cpu().numpy(), s_ref, c.n_elig)
    idx = g.topk().cpu().numpy()
    np.testing.assert_array_equal(idx, oracle.topk(s_ref, c.n_elig, c.K))
    assert g.status() == 0


# ------------------------------------------------ mixed prefill/decode batch --
def _mixed(seed, lens, nq, K):
    return W.make_case("mixed", seed=seed, kind="mixed", seq_lens=lens, q_per_seq=nq, K=K,
                       **LAT_SHAPES)


def test_mixed_prefill_decode_batch_one_launch_per_stage():
    """One batch holding a prefill chunk over an existing prefix, two decode
    steps, a whole short prompt and a one-page prompt: each stage is one call
    of the general entry points (explicit q_seq / q_pos)."""
    need_gpu()
    c = _mixed(600, (3000, 700, 5000, 129, 64), (100, 1, 1, 129, 64), 128)
    g = DevicePipeline(c)
    dsa = g.dsa
    n0 = dsa.launch_count()
    d = g.d
    g.pipe.run(d.q, d.q_idx, d.w, d.kidx_pool, d.k_pool, d.v_pool, c.sm_scale,
               n_eligible=d.n_elig, q_seq=d.q_seq, q_pos=d.q_pos)
    launches = dsa.launch_count() - n0
    s = g.pipe.scores.cpu().numpy()
    s_ref = oracle_scores(c, ld=s.shape[1])
    assert_scores_equal(s, s_ref, c.n_elig)
    idx_ref = oracle.topk(s_ref, c.n_elig, c.K)
    np.testing.assert_array_equal(g.pipe.idx.cpu().numpy(), idx_ref)
    out_ref, lse_ref = oracle_attn(c, idx_ref)
    assert_out_close(g.pipe.out, g.pipe.lse, out_ref, lse_ref, "mixed")
    assert g.status() == 0
    assert launches <= 6, launches


def test_mixed_batch_rows_do_not_interfere():
    """Each sequence's rows of a mixed batch equal the rows of that sequence
    run alone: scores and indices bit for bit, attention within the bar."""
    need_gpu()
    lens, nq = (2100, 900, 300), (40, 1, 300)
    c = _mixed(610, lens, nq, 256)
    g = DevicePipeline(c)
    g.scores_general()
    s_all = g.pipe.scores.cpu().numpy()
    idx_all = g.topk().cpu().numpy()
    out_all, _ = g.attn()
    out_all = out_all.float().cpu().numpy()
    start = 0
    for b, (L, n) in enumerate(zip(lens, nq)):
        rows = np.arange(start, start + n)
        start += n
        solo = W.make_case("solo", seed=610, kind="mixed", seq_lens=lens, q_per_seq=nq, K=256,
                           **LAT_SHAPES)
        # the same cache, only sequence b's queries
        for f in ("q_seq", "q_pos", "n_elig", "q", "q_idx", "w"):
            setattr(solo, f, getattr(c, f)[rows])
        gs = DevicePipeline(solo)
        gs.scores_general()
        s = gs.pipe.scores.cpu().numpy()
        for r in range(n):
            m = int(c.n_elig[rows[r]])
            np.testing.assert_array_equal(s[r, :m], s_all[rows[r], :m])
        np.testing.assert_array_equal(gs.topk().cpu().numpy(), idx_all[rows])
        o, _ = gs.attn()
        err = np.abs(o.float().cpu().numpy() - out_all[rows])
        assert err.max() <= 1e-2 + 2.0 ** -9 * np.abs(out_all[rows]).max(), (b, err.max())


def test_variable_length_prefill_batch():
    """Several whole prompts of different lengths (ragged pages) in one batch."""
    need_gpu()
    lens = (300, 129, 64, 450, 1)
    c = _mixed(620, lens, lens, 64)
    _full_check(c)


def _random_selection(rng, Nq, K, hi):
    """idx [Nq, K]: for query r, distinct positions below hi[r] in random order,
    with -1 entries scattered among them (padding need not be at the end)."""
    idx = np.full((Nq, K), -1, np.int32)
    for r in range(Nq):
        n = min(int(hi[r]), K - K // 7)
        row = np.full(K, -1, np.int32)
        row[:n] = rng.choice(int(hi[r]), size=n, replace=False)
        idx[r] = rng.permutation(row)
    return idx


@pytest.mark.parametrize("name,kw,K", [
    # 5 heads (3 warps idle), Dqk 72 (2-way bank conflicts), Dv 8 (4 active lanes)
    ("odd-dv8", dict(seq_lens=(3000, 700, 1), Hq=5, Dqk=72, Dv=8), 1000),
    # Dv 200: the last pair block is partly outside Dv; many splits per query
    ("odd-dv200", dict(seq_lens=(5000, 2500), Hq=9, Dqk=64, Dv=200), 1500),
    # q of 64 heads x 1536 leaves room for 4-row tiles only
    ("tile4", dict(seq_lens=(900, 1300), Hq=64, Dqk=1536, Dv=512), 300),
])
def test_cuda_core_attention_tiles_and_odd_shapes(name, kw, K):
    """The CUDA-core attention kernel (shapes the tensor-core kernel does not
    take): odd head counts and value widths, tiles shorter than 32 rows,
    selections in random order with -1 entries anywhere."""
    need_gpu()
    c = W.make_case(name, seed=1700 + K, K=K, latent=False, H_i=4, D_i=64, idx_dtype="bf16", **kw)
    g = DevicePipeline(c)
    rng = np.random.default_rng(K)
    idx = _random_selection(rng, c.Nq, c.K, c.seq_lens[c.q_seq])
    out, lse = g.attn(torch.from_numpy(idx).cuda())
    out_ref, lse_ref = oracle_attn(c, idx)
    assert_out_close(out, lse, out_ref, lse_ref, name)
    assert g.status() == 0


def test_cuda_core_attention_long_ranges_per_cta():
    """Enough queries that each CTA takes all K selected rows of its query:
    600 rows = three passes of row lookups, 19 tiles (the last one ragged)."""
    need_gpu()
    rows = np.sort(np.random.default_rng(3).choice(1200, size=400, replace=False))
    c = W.make_case("long-range", seed=1750, kind="prefill", T=1200, q_rows=rows, K=600,
                    **TINY_SHAPES)
    g = DevicePipeline(c)
    rng = np.random.default_rng(4)
    idx = _random_selection(rng, c.Nq, c.K, c.q_pos + 1)
    out, lse = g.attn(torch.from_numpy(idx).cuda())
    out_ref, lse_ref = oracle_attn(c, idx)
    assert_out_close(out, lse, out_ref, lse_ref, "long-range")
    assert g.status() == 0
