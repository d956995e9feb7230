"""Pins of the CPU oracle against facts that do not come from the oracle itself.

Each test fixes one part of the oracle with a closed form, an invariant, a
special case that reduces to a library routine (torch SDPA, numpy matmul), a
hand-worked example under tests/golden/, or brute force on tiny inputs --
chosen so that a dropped term, a wrong sign or index, or a transposed operand
in the oracle fails at least one of them.
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle
import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ----------------------------------------------------------------- helpers --
def bf16_to_f64(u16):
    """Independent bf16 decode through torch (library routine)."""
    t = torch.from_numpy(np.ascontiguousarray(u16).view(np.int16))
    return t.view(torch.bfloat16).double().numpy()


def e4m3_to_f64(u8):
    t = torch.from_numpy(np.ascontiguousarray(u8))
    return t.view(torch.float8_e4m3fn).double().numpy()


def idx_to_f64(case, a):
    return bf16_to_f64(a) if case.idx_dtype == "bf16" else e4m3_to_f64(a)


def code(case):
    return oracle.BF16 if case.idx_dtype == "bf16" else oracle.FP8_E4M3


def scores_of(case, q_idx=None, w=None, kidx_pool=None, block_table=None, ld=None):
    return oracle.index_score(
        case.block_table if block_table is None else block_table, case.seq_lens, case.bs,
        case.num_blocks, case.q_seq, case.q_pos,
        case.q_idx if q_idx is None else q_idx, case.w if w is None else w,
        case.kidx_pool if kidx_pool is None else kidx_pool, code(case),
        case.max_len if ld is None else ld)


def logical_rows(case, pool, b):
    """Rows of sequence b in logical order, read through the block table."""
    L = int(case.seq_lens[b])
    pages = case.block_table[b, :(L + case.bs - 1) // case.bs]
    return pool[pages].reshape(-1, pool.shape[-1])[:L]


def read_golden(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if line:
                rows.append(line.split())
    return rows


# ------------------------------------------------------- storage formats --
def test_e4m3_decode_matches_spec_table():
    for c, v in read_golden("e4m3_codes.txt"):
        got = oracle.decode(oracle.FP8_E4M3, int(c, 16))
        if v == "nan":
            assert math.isnan(got)
        else:
            assert got == float(v) and math.copysign(1, got) == math.copysign(1, float(v)), c


def test_bf16_decode_matches_spec_table():
    for c, v in read_golden("bf16_codes.txt"):
        got = oracle.decode(oracle.BF16, int(c, 16))
        if v == "nan":
            assert math.isnan(got)
        else:
            assert got == float(v) and math.copysign(1, got) == math.copysign(1, float(v)), c


def test_all_e4m3_codes_match_torch():
    ref = e4m3_to_f64(np.arange(256, dtype=np.uint8))
    for c in range(256):
        got = oracle.decode(oracle.FP8_E4M3, c)
        assert (math.isnan(got) and math.isnan(ref[c])) or got == ref[c], hex(c)


# --------------------------------------------------------------- scoring --
def _golden_case():
    g = {r[0]: r[1:] for r in read_golden("index_tiny.txt")}
    bs = int(g["bs"][0])
    bt = np.array([[int(x) for x in g["block_table"]]], dtype=np.int32)
    L = int(g["seq_len"][0])
    qi = np.array([int(x) for x in g["q_idx"]]).reshape(1, 2, 3)
    w = np.array([[float(x) for x in g["w"]]], dtype=np.float32)
    k = np.array([int(x) for x in g["k"]]).reshape(L, 3)
    pool = np.full((2, bs, 3), W.BF16_NAN, dtype=np.uint16)
    for p in range(L):
        pool[bt[0, p // bs], p % bs] = W.encode_int(k[p], "bf16")
    return g, bs, bt, L, W.encode_int(qi, "bf16"), w, pool


def test_index_score_golden_tiny():
    g, bs, bt, L, qi, w, pool = _golden_case()
    s = oracle.index_score(bt, [L], bs, 2, [0], [L - 1], qi, w, pool, oracle.BF16, 4)
    want = np.array([float(x) for x in g["scores"]], dtype=np.float32)
    np.testing.assert_array_equal(s[0], want)
    for key in ("top1", "top2", "top3", "top5"):
        K = int(key[3:])
        idx = oracle.topk(s, [L], K)
        assert idx[0].tolist() == [int(x) for x in g[key]], key


def _small_case(dtype="bf16", seed=11, lens=(70, 33, 128), H=3, D=8):
    return W.make_case(seed=seed, seq_lens=lens, bs=16, Hq=2, Dqk=16, Dv=16, H_i=H, D_i=D,
                       idx_dtype=dtype, K=8, extra_pages=2)


@pytest.mark.parametrize("dtype", ["bf16", "fp8"])
def test_score_one_hot_query_is_relu_of_key_coordinate(dtype):
    c = _small_case(dtype, H=1)
    for d in (0, 5):
        qi = np.zeros((c.Nq, 1, c.D_i), dtype=np.int64)
        qi[:, 0, d] = 1
        s = scores_of(c, q_idx=W.encode_int(qi, dtype), w=np.ones((c.Nq, 1), np.float32))
        for b in range(c.B):
            k = idx_to_f64(c, logical_rows(c, c.kidx_pool, b))
            L = int(c.seq_lens[b])
            np.testing.assert_array_equal(s[b, :L], np.maximum(k[:, d], 0.0))


@pytest.mark.parametrize("dtype", ["bf16", "fp8"])
def test_score_relu_identities(dtype):
    """ReLU(x) - ReLU(-x) = x and ReLU(x) + ReLU(-x) = |x|: negating every key turns
    the score difference into the plain linear form w^T (Q k) (numpy matmul)."""
    c = _small_case(dtype)
    vals = idx_to_f64(c, c.kidx_pool)
    nanmask = np.isnan(vals)
    neg = W.encode_int(-np.where(nanmask, 0, vals).astype(np.int64), dtype)
    # poisoned rows stay poisoned
    neg[nanmask] = c.kidx_pool[nanmask]
    s_pos = scores_of(c).astype(np.float64)
    s_neg = scores_of(c, kidx_pool=neg).astype(np.float64)
    for b in range(c.B):
        L = int(c.seq_lens[b])
        k = idx_to_f64(c, logical_rows(c, c.kidx_pool, b))       # [L, D]
        Q = idx_to_f64(c, c.q_idx[b])                             # [H, D]
        dots = k @ Q.T                                            # [L, H]
        lin = dots @ c.w[b].astype(np.float64)
        ab = np.abs(dots) @ c.w[b].astype(np.float64)
        np.testing.assert_array_equal(s_pos[b, :L] - s_neg[b, :L], lin)
        np.testing.assert_array_equal(s_pos[b, :L] + s_neg[b, :L], ab)


def test_score_causal_mask_and_exact_integers():
    c = W.make_case(seed=3, kind="prefill", T=100, bs=16, Hq=2, Dqk=16, Dv=16, H_i=4, D_i=16,
                    idx_dtype="fp8", K=8)
    s = scores_of(c, ld=c.max_len)
    for r in range(c.Nq):
        t = int(c.q_pos[r])
        assert np.all(np.isfinite(s[r, :t + 1]))
        assert np.all(s[r, t + 1:] == -np.inf)
        assert np.all(s[r, :t + 1] >= 0) and np.all(np.rint(s[r, :t + 1]) == s[r, :t + 1])
    # fp32 exactness bound of the integer scores: H * 4 * (8*8*D)
    assert s[np.isfinite(s)].max() <= 4 * 4 * 64 * 16 < 2 ** 24


def test_score_zero_weights_is_zero():
    c = _small_case("fp8")
    s = scores_of(c, w=np.zeros_like(c.w))
    for b in range(c.B):
        L = int(c.seq_lens[b])
        assert np.all(s[b, :L] == 0.0)


def test_score_block_table_permutation_invariance():
    """Same logical cache under another page permutation: identical scores."""
    c = _small_case("fp8", seed=5)
    rng = np.random.default_rng(0)
    perm = rng.permutation(c.num_blocks)           # old page -> new page
    new_pool = np.empty_like(c.kidx_pool)
    new_pool[perm] = c.kidx_pool
    bt2 = np.where(c.block_table >= 0, perm[np.maximum(c.block_table, 0)], -1).astype(np.int32)
    np.testing.assert_array_equal(scores_of(c), scores_of(c, kidx_pool=new_pool, block_table=bt2))


def test_score_ignores_padding_rows():
    """The last page's tail is NaN-poisoned: no finite score may depend on it."""
    c = _small_case("bf16", seed=8, lens=(17, 31))
    s = scores_of(c)
    for b in range(c.B):
        assert np.all(np.isfinite(s[b, :int(c.seq_lens[b])]))


# ----------------------------------------------------------------- top-K --
def _check_topk_definition(s, n, K, idx):
    """Checker of the selection definition (not a re-implementation): exactly
    min(K, n) distinct eligible positions, ascending, -1 padded, and every kept
    position beats every dropped one under (score desc, position asc)."""
    m = min(K, n)
    kept = idx[:m]
    assert np.all(idx[m:] == -1)
    assert np.all(np.diff(kept) > 0) and (m == 0 or (kept[0] >= 0 and kept[-1] < n))
    keep = np.zeros(n, bool)
    keep[kept] = True
    if m and m < n:
        ks, dp = s[:n][keep], np.nonzero(~keep)[0]
        ds = s[:n][~keep]
        # worst kept vs best dropped
        wk = np.lexsort((-kept, ks))[0]   # lowest score, highest position among kept
        bd = np.lexsort((dp, -ds))[0]     # highest score, lowest position among dropped
        assert ks[wk] > ds[bd] or (ks[wk] == ds[bd] and kept[wk] < dp[bd])


def test_topk_brute_force_tiny_with_ties():
    rng = np.random.default_rng(1)
    for trial in range(300):
        n = int(rng.integers(0, 40))
        ld = n + int(rng.integers(0, 4))
        vals = rng.integers(0, 4, size=ld).astype(np.float32)   # heavy ties
        if trial % 3 == 0:
            vals = rng.standard_normal(ld).astype(np.float32)
        vals[n:] = -np.inf
        for K in (1, 3, max(n - 1, 1), max(n, 1), n + 5):
            idx = oracle.topk(vals[None, :], [n], K)[0]
            brute = sorted(range(n), key=lambda p: (-float(vals[p]), p))[:K]
            assert idx[:len(brute)].tolist() == sorted(brute)
            assert np.all(idx[len(brute):] == -1)
            _check_topk_definition(vals, n, K, idx)


def test_topk_zero_scores_closed_form():
    s = np.zeros((2, 50), np.float32)
    idx = oracle.topk(s, [50, 7], 10)
    assert idx[0].tolist() == list(range(10))
    assert idx[1].tolist() == list(range(7)) + [-1] * 3


def test_topk_negative_zero_ties_positive_zero():
    s = np.array([[-0.0, 0.0, -1.0], [0.0, -0.0, -1.0]], np.float32)
    assert oracle.topk(s, [3, 3], 1)[:, 0].tolist() == [0, 0]


def test_topk_rejects_nan():
    with pytest.raises(oracle.OracleError):
        oracle.topk(np.array([[1.0, np.nan]], np.float32), [2], 1)


def test_tie_construction_closed_form():
    """long-dec recipe at small size: the tied subset holds the unique maximum, so
    top-K is the K lowest tied positions -- fixed by construction, no oracle."""
    c = W.make_case(seed=3, seq_lens=(3000, 2500, 1200), bs=64, Hq=2, Dqk=16, Dv=16,
                    H_i=8, D_i=32, idx_dtype="fp8", K=48, tie_frac=0.05)
    s = scores_of(c)
    idx = oracle.topk(s, c.n_elig, c.K)
    for b in range(c.B):
        tied = c.tie_positions[b]
        assert len(tied) > c.K
        assert idx[b].tolist() == tied[:c.K].tolist()
        L = int(c.seq_lens[b])
        mx = s[b, :L].max()
        assert np.all(s[b, tied] == mx)
        assert (s[b, :L] == mx).sum() == len(tied)


# ------------------------------------------------------------- attention --
def _dense_sdpa(q, k, v, scale, causal_offsets=None):
    """torch SDPA in fp64: q [Nq, H, D], k/v [Nq, L, D] -> [Nq, H, Dv]."""
    out = []
    for r in range(q.shape[0]):
        qq = torch.from_numpy(q[r])[None, :, None, :]          # [1, H, 1, D]
        kk = torch.from_numpy(k[r])[None, None].expand(1, q.shape[1], -1, -1)
        vv = torch.from_numpy(v[r])[None, None].expand(1, q.shape[1], -1, -1)
        o = torch.nn.functional.scaled_dot_product_attention(qq, kk, vv, scale=scale)
        out.append(o[0, :, 0, :].numpy())
    return np.stack(out)


def _attn(c, idx, q=None, k_pool=None, v_pool=None):
    return oracle.sparse_attn(c.block_table, c.seq_lens, c.bs, c.num_blocks, c.q_seq,
                              c.q if q is None else q, c.k_pool if k_pool is None else k_pool,
                              c.v_pool if v_pool is None else v_pool, idx, c.sm_scale, Dv=c.Dv)


@pytest.mark.parametrize("latent", [False, True])
def test_attention_with_all_positions_is_dense_sdpa(latent):
    """K >= L selects every position: sparse attention = dense attention (SDPA)."""
    kw = dict(Hq=4, Dqk=24, Dv=16, latent=True) if latent else dict(Hq=3, Dqk=16, Dv=8)
    c = W.make_case(seed=21, seq_lens=(50, 17, 64), bs=16, H_i=2, D_i=8, K=80, **kw)
    s = scores_of(c)
    idx = oracle.topk(s, c.n_elig, c.K)
    for b in range(c.B):
        assert idx[b, :c.seq_lens[b]].tolist() == list(range(c.seq_lens[b]))
    out, lse = _attn(c, idx)
    for b in range(c.B):
        kr = bf16_to_f64(logical_rows(c, c.k_pool, b))[:, :c.Dqk]
        vr = bf16_to_f64(logical_rows(c, c.v_pool, b))[:, :c.Dv]
        want = _dense_sdpa(bf16_to_f64(c.q[b:b + 1]), kr[None], vr[None], c.sm_scale)[0]
        np.testing.assert_allclose(out[b], want, rtol=1e-12, atol=1e-12)
        z = c.sm_scale * bf16_to_f64(c.q[b]) @ kr.T
        np.testing.assert_allclose(lse[b], torch.logsumexp(torch.from_numpy(z), -1).numpy(),
                                   rtol=1e-12)


def test_attention_prefill_causal_is_dense_causal_sdpa():
    c = W.make_case(seed=4, kind="prefill", T=40, bs=16, Hq=2, Dqk=16, Dv=16, latent=True,
                    H_i=2, D_i=8, K=64)
    idx = oracle.topk(scores_of(c), c.n_elig, c.K)
    out, _ = _attn(c, idx)
    rows = bf16_to_f64(logical_rows(c, c.k_pool, 0))
    q = torch.from_numpy(bf16_to_f64(c.q)).permute(1, 0, 2)[None]       # [1, H, T, D]
    kk = torch.from_numpy(rows)[None, None].expand(1, c.Hq, -1, -1)
    want = torch.nn.functional.scaled_dot_product_attention(
        q, kk, kk[..., :c.Dv], is_causal=True, scale=c.sm_scale)[0].permute(1, 0, 2).numpy()
    np.testing.assert_allclose(out, want, rtol=1e-11, atol=1e-12)


def test_attention_single_row_returns_that_row():
    c = W.make_case(seed=6, seq_lens=(90,), bs=16, Hq=4, Dqk=16, Dv=16, H_i=2, D_i=8, K=1)
    for p in (0, 37, 89):
        out, lse = _attn(c, np.array([[p]], np.int32))
        v = bf16_to_f64(logical_rows(c, c.v_pool, 0))[p]
        k = bf16_to_f64(logical_rows(c, c.k_pool, 0))[p]
        np.testing.assert_array_equal(out[0], np.broadcast_to(v, out[0].shape))
        np.testing.assert_allclose(lse[0], c.sm_scale * (bf16_to_f64(c.q[0]) @ k), rtol=1e-13)


def test_attention_constant_values_and_zero_query():
    c = W.make_case(seed=7, seq_lens=(70,), bs=16, Hq=2, Dqk=16, Dv=16, H_i=2, D_i=8, K=20)
    idx = np.array([[1, 5, 9, 33, 60, 69] + [-1] * 14], np.int32)
    vconst = c.v_pool.copy()
    vconst[...] = W.encode_bf16(np.float32(0.75))
    out, _ = _attn(c, idx, v_pool=vconst)
    np.testing.assert_allclose(out, 0.75, rtol=0, atol=1e-15)
    qz = np.zeros_like(c.q)
    out, lse = _attn(c, idx, q=qz)
    vr = bf16_to_f64(logical_rows(c, c.v_pool, 0))[idx[0, :6]]
    np.testing.assert_allclose(out[0], np.broadcast_to(vr.mean(0), out[0].shape), rtol=1e-13)
    np.testing.assert_allclose(lse, math.log(6), rtol=1e-15)


def test_attention_two_rows_closed_form():
    """Two rows, one head: z = (0, 1) -> out = (V0 + e V1) / (1 + e)."""
    bs = 4
    bt = np.array([[0]], np.int32)
    q = W.encode_bf16(np.array([[[1.0, 0.0]]], np.float32))
    k = np.zeros((1, bs, 2), np.float32)
    k[0, 0] = [0.0, 5.0]
    k[0, 1] = [1.0, 7.0]
    v = np.zeros((1, bs, 2), np.float32)
    v[0, 0] = [1.0, 0.0]
    v[0, 1] = [0.0, 2.0]
    out, lse = oracle.sparse_attn(bt, [2], bs, 1, [0], q, W.encode_bf16(k), W.encode_bf16(v),
                                  np.array([[0, 1]], np.int32), 1.0)
    e = math.e
    np.testing.assert_allclose(out[0, 0], [1 / (1 + e), 2 * e / (1 + e)], rtol=1e-15)
    np.testing.assert_allclose(lse[0, 0], math.log(1 + e), rtol=1e-15)


def test_attention_is_a_set_function_and_skips_padding():
    c = W.make_case(seed=9, seq_lens=(120, 64), bs=16, Hq=2, Dqk=16, Dv=16, H_i=2, D_i=8, K=10)
    idx = np.array([[3, 7, 50, 119, 0, -1, -1, -1, -1, -1],
                    [63, 1, 2, -1, -1, 30, -1, -1, -1, -1]], np.int32)
    out1, lse1 = _attn(c, idx)
    shuf = np.array([[119, -1, 0, 50, -1, 3, -1, 7, -1, -1],
                     [-1, 30, -1, 2, -1, 1, -1, 63, -1, -1]], np.int32)
    out2, lse2 = _attn(c, shuf)
    np.testing.assert_allclose(out1, out2, rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(lse1, lse2, rtol=1e-14)


def test_attention_block_table_permutation_invariance():
    c = W.make_case(seed=10, seq_lens=(100, 40), bs=16, Hq=2, Dqk=16, Dv=16, H_i=2, D_i=8, K=30)
    idx = oracle.topk(scores_of(c), c.n_elig, c.K)
    out1, _ = _attn(c, idx)
    perm = np.random.default_rng(3).permutation(c.num_blocks)
    kp = np.empty_like(c.k_pool)
    kp[perm] = c.k_pool
    vp = np.empty_like(c.v_pool)
    vp[perm] = c.v_pool
    bt2 = np.where(c.block_table >= 0, perm[np.maximum(c.block_table, 0)], -1).astype(np.int32)
    out2, _ = oracle.sparse_attn(bt2, c.seq_lens, c.bs, c.num_blocks, c.q_seq, c.q, kp, vp, idx,
                                 c.sm_scale, Dv=c.Dv)
    np.testing.assert_array_equal(out1, out2)


def test_prefill_row_equals_decode_of_prefix():
    """Prefill query t over the cache equals decode with L = t + 1 on the same cache
    (prefill/decode layout alignment)."""
    c = W.make_case(seed=12, kind="prefill", T=150, bs=16, Hq=2, Dqk=16, Dv=16, latent=True,
                    H_i=3, D_i=8, idx_dtype="fp8", K=32)
    s = scores_of(c)
    idx = oracle.topk(s, c.n_elig, c.K)
    out, lse = _attn(c, idx)
    for t in (0, 31, 32, 100, 149):
        sl = np.array([t + 1], np.int32)
        sd = oracle.index_score(c.block_table, sl, c.bs, c.num_blocks, [0], [t], c.q_idx[t:t + 1],
                                c.w[t:t + 1], c.kidx_pool, oracle.FP8_E4M3, c.max_len)
        np.testing.assert_array_equal(sd[0], s[t])
        idd = oracle.topk(sd, sl, c.K)
        np.testing.assert_array_equal(idd[0], idx[t])
        od, ld = oracle.sparse_attn(c.block_table, sl, c.bs, c.num_blocks, [0], c.q[t:t + 1],
                                    c.k_pool, c.v_pool, idd, c.sm_scale, Dv=c.Dv)
        np.testing.assert_array_equal(od[0], out[t])


def test_oracle_reports_bad_block_table():
    c = _small_case("bf16")
    bt = c.block_table.copy()
    bt[0, 1] = c.num_blocks + 5
    with pytest.raises(oracle.OracleError):
        scores_of(c, block_table=bt)


# ------------------------------------------------------------- cache write --
def _logical_write_all(c, pool_src, bt, num_blocks, fill):
    """Write every cached position of every sequence of c (rows read from
    pool_src through c's own table) into a pool of `fill` laid out by bt."""
    seq = np.concatenate([np.full(int(L), b, np.int32) for b, L in enumerate(c.seq_lens)])
    pos = np.concatenate([np.arange(int(L), dtype=np.int32) for L in c.seq_lens])
    rows = np.concatenate([logical_rows(c, pool_src, b) for b in range(c.B)])
    dst = np.full((num_blocks, c.bs, pool_src.shape[-1]), fill, pool_src.dtype)
    return seq, pos, rows, dst


def test_cache_write_round_trip_through_the_page_view():
    """Rows written one by one land where the page view (pages of the table,
    reshaped to rows) reads them back; nothing else changes."""
    c = _small_case("bf16")
    seq, pos, rows, dst = _logical_write_all(c, c.k_pool, c.block_table, c.num_blocks, 0x7FC1)
    out, bad = oracle.cache_write(c.block_table, c.bs, c.num_blocks, seq, pos, rows, dst)
    assert not bad
    for b in range(c.B):
        np.testing.assert_array_equal(logical_rows(c, out, b), logical_rows(c, c.k_pool, b))
    untouched = np.all(out.reshape(-1, out.shape[-1]) == 0x7FC1, axis=1).sum()
    assert untouched == c.num_blocks * c.bs - int(c.seq_lens.sum())


def test_cache_write_order_of_distinct_rows_is_irrelevant_and_last_duplicate_wins():
    c = _small_case("fp8")
    seq, pos, rows, dst = _logical_write_all(c, c.kidx_pool, c.block_table, c.num_blocks, 0)
    a, _ = oracle.cache_write(c.block_table, c.bs, c.num_blocks, seq, pos, rows, dst)
    perm = np.random.default_rng(5).permutation(seq.shape[0])
    b, _ = oracle.cache_write(c.block_table, c.bs, c.num_blocks, seq[perm], pos[perm], rows[perm],
                              dst)
    np.testing.assert_array_equal(a, b)
    two = np.stack([np.full(c.D_i, 3, np.uint8), np.full(c.D_i, 9, np.uint8)])
    d2, _ = oracle.cache_write(c.block_table, c.bs, c.num_blocks, [1, 1], [5, 5], two, dst)
    page = c.block_table[1, 0]
    np.testing.assert_array_equal(d2[page, 5], two[1])


def test_cache_write_skips_rows_without_a_destination_and_keeps_wide_rows_tails():
    c = _small_case("bf16")
    dst = np.full((c.num_blocks, c.bs, c.Dkv), 0x1234, np.uint16)
    rows = np.arange(6 * 5, dtype=np.uint16).reshape(6, 5)       # 5 of Dkv columns
    past = c.block_table.shape[1] * c.bs
    unused = int(np.argmax(c.block_table[1] < 0)) * c.bs           # first page slot set to -1
    assert c.block_table[1, unused // c.bs] < 0
    seq = [-1, c.B, 0, 0, 1, 2]
    pos = [0, 0, -1, past, unused, 3]
    out, bad = oracle.cache_write(c.block_table, c.bs, c.num_blocks, seq, pos, rows, dst)
    assert bad
    page = c.block_table[2, 0]
    np.testing.assert_array_equal(out[page, 3, :5], rows[5])
    assert np.all(out[page, 3, 5:] == 0x1234)
    changed = np.argwhere(np.any(out != dst, axis=-1))
    assert changed.tolist() == [[page, 3]]


def test_cache_written_at_prefill_serves_the_decode_gather():
    """Prefill writes a prompt into pages of a fresh table; every stage read
    through that table gives what it gives on the original cache (the block
    layout written must match the gather that decode reads)."""
    c = W.make_case(seed=13, seq_lens=(150, 77), bs=16, Hq=2, Dqk=24, Dv=16, latent=True,
                    H_i=3, D_i=16, idx_dtype="fp8", K=40)
    nb2 = c.num_blocks + 4
    perm = np.random.default_rng(8).permutation(nb2).astype(np.int32)
    bt2 = np.full_like(c.block_table, -1)
    used = c.block_table >= 0
    bt2[used] = perm[:int(used.sum())]
    seq, pos, rows_k, dst_k = _logical_write_all(c, c.k_pool, bt2, nb2, 0)
    _, _, rows_i, dst_i = _logical_write_all(c, c.kidx_pool, bt2, nb2, 0)
    kp, bad_k = oracle.cache_write(bt2, c.bs, nb2, seq, pos, rows_k, dst_k)
    ip, bad_i = oracle.cache_write(bt2, c.bs, nb2, seq, pos, rows_i, dst_i)
    assert not bad_k and not bad_i
    s1 = scores_of(c)
    s2 = oracle.index_score(bt2, c.seq_lens, c.bs, nb2, c.q_seq, c.q_pos, c.q_idx, c.w, ip,
                            code(c), c.max_len)
    np.testing.assert_array_equal(s1, s2)
    idx = oracle.topk(s1, c.n_elig, c.K)
    o1, l1 = _attn(c, idx)
    o2, l2 = oracle.sparse_attn(bt2, c.seq_lens, c.bs, nb2, c.q_seq, c.q, kp, kp, idx, c.sm_scale,
                                Dv=c.Dv)
    np.testing.assert_array_equal(o1, o2)
    np.testing.assert_array_equal(l1, l2)


def test_mixed_batch_row_equals_decode_of_its_prefix():
    """A mixed batch (prefill chunk + decode + whole prompt) is row by row the
    decode of each query's prefix: a query at position t of sequence b sees
    exactly positions 0..t of b."""
    c = W.make_case(seed=14, kind="mixed", seq_lens=(90, 40, 33), q_per_seq=(20, 1, 33), bs=16,
                    Hq=2, Dqk=16, Dv=16, latent=True, H_i=2, D_i=8, idx_dtype="bf16", K=12)
    assert c.q_seq.tolist() == [0] * 20 + [1] + [2] * 33
    assert c.q_pos.tolist() == list(range(70, 90)) + [39] + list(range(33))
    s = scores_of(c)
    idx = oracle.topk(s, c.n_elig, c.K)
    out, _ = _attn(c, idx)
    for r in (0, 19, 20, 21, 53):
        b, t = int(c.q_seq[r]), int(c.q_pos[r])
        sl = c.seq_lens.copy()
        sl[b] = t + 1
        sd = oracle.index_score(c.block_table, sl, c.bs, c.num_blocks, [b], [t], c.q_idx[r:r + 1],
                                c.w[r:r + 1], c.kidx_pool, code(c), c.max_len)
        np.testing.assert_array_equal(sd[0], s[r])
        od, _ = oracle.sparse_attn(c.block_table, sl, c.bs, c.num_blocks, [b], c.q[r:r + 1],
                                   c.k_pool, c.v_pool, idx[r:r + 1], c.sm_scale, Dv=c.Dv)
        np.testing.assert_array_equal(od[0], out[r])


def _torch_decode(codes, dtype_code):
    """Values of stored codes through torch's own conversions (independent of
    the oracle's decoder)."""
    c = np.ascontiguousarray(codes)
    if dtype_code == oracle.BF16:
        return torch.from_numpy(c.astype(np.int16)).view(torch.bfloat16).double().numpy()
    return torch.from_numpy(c.astype(np.uint8)).view(torch.float8_e4m3fn).double().numpy()


@pytest.mark.parametrize("dtype", [oracle.BF16, oracle.FP8_E4M3])
def test_page_bounds_brute_force(dtype):
    """Per page and dimension, the largest and smallest key over the page's
    cached positions (first occurrence on ties), by plain loops over a tiny
    permuted layout with a ragged last page and one sequence of length 1."""
    rng = np.random.default_rng(91)
    bs, D, seq_lens = 4, 32, (5, 8, 1)
    pages_per = [(L + bs - 1) // bs for L in seq_lens]
    NB = sum(pages_per) + 2
    perm = rng.permutation(NB)
    bt = np.full((3, 2), -1, np.int32)
    k = 0
    for b, n in enumerate(pages_per):
        for j in range(n):
            bt[b, j] = perm[k]
            k += 1
    vals = rng.integers(-8, 9, size=(NB, bs, D))
    vals[0, :, 0] = 0                                # ties (and +0 / -0 for bf16 below)
    pool = W.encode_int(vals, "bf16" if dtype == oracle.BF16 else "fp8")
    if dtype == oracle.BF16:
        pool[0, 1, 0] = 0x8000                       # -0.0 ties +0.0
    got, cached = oracle.page_bounds(bt, np.array(seq_lens), bs, NB, pool, dtype)
    for b, L in enumerate(seq_lens):
        for j in range(pages_per[b]):
            page = bt[b, j]
            n = min(bs, L - j * bs)
            assert cached[page]
            for d in range(D):
                v = _torch_decode(pool[page, :n, d], dtype)
                imax = max(range(n), key=lambda r: (v[r], -r))
                imin = min(range(n), key=lambda r: (v[r], r))
                assert got[page, 0, d] == pool[page, imax, d]
                assert got[page, 1, d] == pool[page, imin, d]
    assert cached.sum() == sum(pages_per)


@pytest.mark.parametrize("dtype", [oracle.BF16, oracle.FP8_E4M3])
def test_page_score_bound_holds_and_is_tight_on_constant_pages(dtype):
    """Every score of a page's cached positions is at most the page's bound
    (checked against the oracle's own scores, weights of both signs); a page
    whose cached keys are all equal is bounded by exactly its score."""
    rng = np.random.default_rng(93)
    dname = "bf16" if dtype == oracle.BF16 else "fp8"
    c = W.make_case("bounds", seed=94, seq_lens=(300, 130), K=16, Hq=4, Dqk=64, Dv=64,
                    latent=False, H_i=8, D_i=32, idx_dtype=dname)
    w = rng.integers(-3, 4, size=c.w.shape).astype(np.float32)
    kp = c.kidx_pool.copy()
    # page 1 of sequence 0: every cached key the same row
    kp[c.block_table[0, 1]] = kp[c.block_table[0, 1], 0]
    scores = oracle.index_score(c.block_table, c.seq_lens, c.bs, c.num_blocks, c.q_seq, c.q_pos,
                                c.q_idx, w, kp, dtype, int(c.seq_lens.max()))
    bounds, cached = oracle.page_bounds(c.block_table, c.seq_lens, c.bs, c.num_blocks, kp, dtype)
    for b in range(c.B):
        ub = oracle.page_score_bound(c.q_idx[b], w[b], bounds, dtype)
        L = int(c.seq_lens[b])
        for j in range((L + c.bs - 1) // c.bs):
            page = c.block_table[b, j]
            s = scores[b, j * c.bs:min(L, (j + 1) * c.bs)]
            assert s.max() <= ub[page] + 1e-9 * max(1.0, abs(ub[page]))
            if b == 0 and j == 1:
                assert np.all(s == s[0])
                assert ub[page] == pytest.approx(float(s[0]), abs=1e-9)
