"""Shared helpers of the GPU parity tests (CUDA path through the C ABI vs the oracle)."""
import numpy as np
import pytest
import torch

import oracle
from workloads import device as wdev

# Tolerances on attention outputs against the fp64 oracle (bf16 I/O, fp32
# accumulation): max-abs 1e-2 and mean-abs 2e-3 on out; lse to 1e-3 absolute.
# The output is stored as bf16.  Only that store's own rounding is exempt from
# the max-abs bar: an element passes when it is within 1e-2 of the exact
# value, or within 1e-2 of the exact value rounded to bf16 (the nearest
# representable output; the two differ only where the rounding alone moves a
# value by more than 1e-2, i.e. |out| >= 4).  The mean-abs bar is taken
# against the exact value.
OUT_MAX_ABS = 1e-2
OUT_MEAN_ABS = 2e-3
LSE_ABS = 1e-3


def bf16_nearest(x):
    """float64 values rounded to the nearest bfloat16 value (ties to an even
    significand), returned as float64.  Rounds once, from the float64 value:
    the candidates are the bf16 neighbours of its float32 rounding, and the
    nearest of them to x itself is taken."""
    x = np.asarray(x, dtype=np.float64)
    a = np.abs(x)
    top = a.astype(np.float32).view(np.uint32).astype(np.int64) & 0xFFFF0000
    cands = np.stack([np.maximum(top - 0x10000, 0), top, top + 0x10000])
    vals = cands.astype(np.uint32).view(np.float32).astype(np.float64)
    dist = np.abs(vals - a[None])
    best = dist.min(axis=0)
    # among the nearest candidates prefer the one with an even last bit
    even = ((cands >> 16) & 1) == 0
    score = np.where(dist == best[None], np.where(even, 0, 1), 2)
    pick = np.take_along_axis(vals, score.argmin(axis=0)[None], axis=0)[0]
    return np.copysign(pick, x)


def out_errors(o, ref):
    """Per-element error against the exact value, and whether each element
    meets the max-abs bar with only the bf16 store's rounding exempt."""
    err = np.abs(o - ref)
    ok = (err <= OUT_MAX_ABS) | (np.abs(o - bf16_nearest(ref)) <= OUT_MAX_ABS)
    return err, ok


def need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def lib():
    import __graft_entry__
    __graft_entry__.build_library()
    import sparse_attention_score_gb300 as dsa
    return dsa


def code(case):
    return oracle.BF16 if case.idx_dtype == "bf16" else oracle.FP8_E4M3


def oracle_scores(case, ld=None, rows=None):
    rows = np.arange(case.Nq) if rows is None else np.asarray(rows)
    return oracle.index_score(case.block_table, case.seq_lens, case.bs, case.num_blocks,
                              case.q_seq[rows], case.q_pos[rows], case.q_idx[rows], case.w[rows],
                              case.kidx_pool, code(case), case.max_len if ld is None else ld)


def oracle_attn(case, idx, rows=None):
    rows = np.arange(case.Nq) if rows is None else np.asarray(rows)
    return oracle.sparse_attn(case.block_table, case.seq_lens, case.bs, case.num_blocks,
                              case.q_seq[rows], case.q[rows], case.k_pool, case.v_pool, idx,
                              case.sm_scale, Dv=case.Dv)


class DevicePipeline:
    """Runs the three stages of a case on the GPU through the binding."""

    def __init__(self, case, dsa=None, ld=None, device="cuda"):
        self.dsa = dsa or lib()
        self.case = case
        self.d = wdev.upload(case, device)
        self.layout = wdev.layout_of(case, self.d)
        kind = "decode" if case.kind == "decode" else "prefill"
        self.pipe = self.dsa.Pipeline(self.layout, kind=kind, Nq=case.Nq, Hq=case.Hq, Dqk=case.Dqk,
                                      Dv=case.Dv, H_i=case.H_i, D_i=case.D_i, K=case.K, ld=ld,
                                      device=device,
                                      prefill_seq=None if case.kind == "mixed" else 0)

    def scores(self):
        d, p = self.d, self.pipe
        if self.case.kind == "mixed":
            return self.scores_general()
        if self.case.kind == "decode":
            self.dsa.index_score(self.layout, d.q_idx, d.w, d.kidx_pool, p.scores, p.ws_index)
        else:
            self.dsa.index_score_prefill(self.layout, 0, d.q_idx, d.w, d.kidx_pool, p.scores,
                                         p.ws_index, q_pos=d.q_pos)
        return p.scores

    def scores_general(self):
        """The general entry point (explicit q_seq) on the same inputs."""
        d, p = self.d, self.pipe
        self.dsa.index_score(self.layout, d.q_idx, d.w, d.kidx_pool, p.scores, p.ws_index,
                             q_seq=d.q_seq, q_pos=d.q_pos)
        return p.scores

    def topk(self, scores=None, n_elig=None):
        p = self.pipe
        s = p.scores if scores is None else scores
        ne = self.d.n_elig if n_elig is None else n_elig
        self.dsa.topk(s, ne, self.case.K, p.idx, p.ws_topk)
        return p.idx

    def attn(self, idx=None):
        d, p, c = self.d, self.pipe, self.case
        ix = p.idx if idx is None else idx
        if c.kind == "decode":
            self.dsa.sparse_attn_decode(self.layout, d.q, d.k_pool, d.v_pool, ix, c.sm_scale, p.out,
                                        p.lse, p.ws_attn)
        else:
            self.dsa.sparse_attn_prefill(self.layout, d.q, d.k_pool, d.v_pool, ix, c.sm_scale,
                                         p.out, p.lse, p.ws_attn, q_seq=d.q_seq,
                                         q_pos=d.q_pos)
        return p.out, p.lse

    def all(self):
        self.scores()
        self.topk()
        return self.attn()

    def status(self):
        return self.pipe.status()


def assert_scores_equal(s_gpu, s_ref, n_elig):
    """Bit-exact on every eligible entry of every row (entries past a row's
    eligible count are not part of the output contract)."""
    for r in range(s_ref.shape[0]):
        n = int(n_elig[r])
        np.testing.assert_array_equal(s_gpu[r, :n], s_ref[r, :n], err_msg=f"row {r}")


def assert_out_close(out_gpu, lse_gpu, out_ref, lse_ref, what=""):
    o = out_gpu.float().cpu().numpy().astype(np.float64) if hasattr(out_gpu, "cpu") else \
        np.asarray(out_gpu, dtype=np.float64)
    assert np.all(np.isfinite(o)), f"{what}: non-finite output"
    err, ok = out_errors(o, out_ref)
    if not ok.all():
        bad = np.argwhere(~ok)[0]
        raise AssertionError(f"{what}: {int((~ok).sum())} elements beyond max-abs {OUT_MAX_ABS} "
                             f"(first at {tuple(bad)}: gpu {o[tuple(bad)]!r}, "
                             f"exact {out_ref[tuple(bad)]!r})")
    assert err.mean() <= OUT_MEAN_ABS, f"{what}: mean-abs {err.mean():.3e}"
    if lse_gpu is not None:
        l = lse_gpu.cpu().numpy().astype(np.float64) if hasattr(lse_gpu, "cpu") else \
            np.asarray(lse_gpu, dtype=np.float64)
        fin = np.isfinite(lse_ref)
        assert np.array_equal(np.isfinite(l), fin), f"{what}: lse finiteness differs"
        if fin.any():
            assert np.abs(l[fin] - lse_ref[fin]).max() <= LSE_ABS, f"{what}: lse"
    return float(err.max()), float(err.mean())


def check_topk_definition(s, n, K, idx):
    """Validity of a selection against its scores (used where the oracle cannot
    afford a full row): kept set of size min(K,n), ascending, -1 padded, and the
    worst kept beats the best dropped under (score desc, position asc)."""
    s = np.where(s == 0, 0.0, s).astype(np.float32)  # -0 ties +0
    m = min(K, n)
    kept = idx[:m].astype(np.int64)
    assert np.all(idx[m:] == -1)
    assert np.all(np.diff(kept) > 0) and (m == 0 or (kept[0] >= 0 and kept[-1] < n))
    if m == 0 or m == n:
        return
    keep = np.zeros(n, bool)
    keep[kept] = True
    ks = s[:n][keep]
    dp = np.nonzero(~keep)[0]
    ds = s[:n][~keep]
    wk = np.lexsort((-kept, ks))[0]
    bd = np.lexsort((dp, -ds))[0]
    assert ks[wk] > ds[bd] or (ks[wk] == ds[bd] and kept[wk] < dp[bd])


# ------------------------------------------------ host <-> device marshalling --
def logical_rows(case, pool, b, L):
    """Rows 0..L-1 of sequence b read through the case's block table."""
    pages = case.block_table[b, :(L + case.bs - 1) // case.bs]
    return pool[pages].reshape(-1, pool.shape[-1])[:L]


def to_dev(a):
    """Host array -> device tensor of the same bytes (uint16 -> bf16 view)."""
    t = torch.from_numpy(np.ascontiguousarray(a))
    if a.dtype == np.uint16:
        t = t.view(torch.int16).view(torch.bfloat16)
    return t.cuda()


def to_host(t, like):
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).cpu().numpy().view(np.uint16)
    return t.cpu().numpy().astype(like.dtype, copy=False)


def fresh_layout(case, seed, extra):
    """Another page assignment for the same sequences, with spare pages."""
    nb2 = case.num_blocks + extra
    perm = np.random.default_rng(seed).permutation(nb2).astype(np.int32)
    bt2 = np.full_like(case.block_table, -1)
    used = case.block_table >= 0
    bt2[used] = perm[:int(used.sum())]
    return bt2, nb2
