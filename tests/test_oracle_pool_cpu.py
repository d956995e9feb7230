"""CPU checks of the parity tests' own machinery: the sharded oracle runner
gives exactly what one oracle call over the whole case gives, and the bf16
rounding used by the attention tolerance is the correctly rounded one."""
import numpy as np
import torch

import oracle
import workloads as W
from gpu_common import bf16_nearest, out_errors
from oracle_pool import OraclePool, _balanced_shards


def test_balanced_shards_cover_every_row_once():
    for n, k in ((1, 8), (7, 64), (1000, 16), (16384, 64)):
        cost = np.arange(n) + 1
        sh = _balanced_shards(cost, k)
        assert sh[0][0] == 0 and sh[-1][1] == n
        assert all(a < b for a, b in sh) and all(sh[i][1] == sh[i + 1][0] for i in range(len(sh) - 1))
        assert len(sh) <= k


def test_pool_equals_one_oracle_call_prefill_and_decode():
    cases = [W.make_case("pool-pre", seed=5, kind="prefill", T=700, Hq=8, Dqk=64, Dv=32,
                         H_i=4, D_i=32, idx_dtype="fp8", K=96),
             W.make_case("pool-dec", seed=6, seq_lens=(300, 1000, 77, 513), Hq=4, Dqk=64, Dv=64,
                         latent=True, H_i=3, D_i=64, idx_dtype="bf16", K=128)]
    for c in cases:
        code = oracle.BF16 if c.idx_dtype == "bf16" else oracle.FP8_E4M3
        s1 = oracle.index_score(c.block_table, c.seq_lens, c.bs, c.num_blocks, c.q_seq, c.q_pos,
                                c.q_idx, c.w, c.kidx_pool, code, c.max_len)
        i1 = oracle.topk(s1, c.n_elig, c.K)
        rows = np.array([0, 2, c.Nq - 1])
        o1, l1 = oracle.sparse_attn(c.block_table, c.seq_lens, c.bs, c.num_blocks, c.q_seq[rows],
                                    c.q[rows], c.k_pool, c.v_pool, i1[rows], c.sm_scale, Dv=c.Dv)
        with OraclePool(c, workers=3) as pool:
            s2, i2 = pool.scores_and_topk(c.max_len)
            o2, l2 = pool.attention(rows, i1[rows])
        np.testing.assert_array_equal(s1, s2)
        np.testing.assert_array_equal(i1, i2)
        np.testing.assert_array_equal(o1, o2)
        np.testing.assert_array_equal(l1, l2)


def test_bf16_nearest_matches_torch_on_float32_values():
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.standard_normal(20000) * 4, rng.standard_normal(2000) * 1e-3,
                        [0.0, -0.0, 1.0, -3.0, 5.125, 1e-30]]).astype(np.float32)
    want = torch.from_numpy(x).to(torch.bfloat16).double().numpy()
    np.testing.assert_array_equal(bf16_nearest(x.astype(np.float64)), want)


def test_bf16_nearest_rounds_float64_once():
    # 1 + 2^-8 is the midpoint of 1 and 1 + 2^-7: ties go to the even 1.0;
    # a hair above it (not representable in float32) must round up, which a
    # rounding through float32 first would miss
    assert bf16_nearest(np.array([1.0 + 2.0 ** -8]))[0] == 1.0
    assert bf16_nearest(np.array([1.0 + 2.0 ** -8 + 2.0 ** -40]))[0] == 1.0 + 2.0 ** -7
    assert bf16_nearest(np.array([-(1.0 + 2.0 ** -8 + 2.0 ** -40)]))[0] == -(1.0 + 2.0 ** -7)
    assert bf16_nearest(np.array([3.0 * 2.0 ** -8 + 1.0]))[0] == 1.0 + 2.0 ** -6


def test_tolerance_exempts_only_the_store_rounding():
    ref = np.array([0.5, 2.0, 5.007, 5.007, 100.3])
    gpu = np.array([0.5095, 2.0099, bf16_nearest(np.array([5.007]))[0], 5.04, 100.5])
    _, ok = out_errors(gpu, ref)
    # 0.5 and 2.0: plain bar; 5.007: its bf16 neighbour passes, a further
    # value (one bf16 step away) does not; 100.3 -> bf16 is 100.5: passes
    assert ok.tolist() == [True, True, True, False, True]
    _, ok = out_errors(np.array([2.0105]), np.array([2.0]))
    assert not ok[0]
