"""Seeded synthetic inputs for the DSA sparse-attention hot path.

This module is the only code shared by the CUDA path's tests/benchmark and the
CPU oracle.  It draws random numbers, encodes them into the storage formats the
kernels read (bf16, FP8 E4M3) and assigns pages of the paged cache; it holds
none of the method's arithmetic (no scoring, no selection, no attention).

Workloads (sizes as the pages' scenarios are stated for this library):

=========  ==============================================================
dec-tiny   decode, B=1, L=4096, 16 query heads x 128, separate K and V
           pools (MQA), indexer 4 heads x 64 in bf16, top-K 256
dec-batch  decode, B=32, L ~ U[8192, 32768], 64 query heads sharing one
           latent KV row of 576 (V = first 512 dims), indexer 64 x 128 in
           FP8 E4M3, top-K 2048
prefill    causal prefill of one 16384-token sequence, dec-batch shapes
long-dec   decode, B=4, L = 262144/196608/131072/65536, dec-batch shapes,
           ~5% of positions tie at the maximum indexer score
million    decode, B=8, L = 1,048,576 each, dec-batch shapes (~10.7 GB)
=========  ==============================================================

Value distributions: q and K/V rows bf16(N(0,1)); q_idx and k_idx integers
uniform in [-8, 8] stored exactly as bf16 or E4M3; head weights integers
uniform in [0, 4] as fp32.  The block table is one seeded permutation of the
whole page pool, handed to the sequences in order; the tail of a sequence's
last page (and any extra page no table points to) can be poisoned with NaN so
that a kernel that reads outside the layout is caught.

Tie construction ("long-dec"): per sequence a sign vector s in {-1,+1}^D is
drawn; indexer queries are q_idx[h,d] = s_d * U{0..8} with q_idx[0,0] != 0 and
w[0] >= 1; a seeded subset of ~5% of positions gets k = 8 s, every other
position draws each k_d from [-8, 8] without the value 8 s_d.  Then
q_h . k <= 8 |q_h|_1 = q_h . (8 s) for every head, with strict inequality for
head 0, so the subset ties at the unique maximum score by construction and the
exact top-K is the subset's K lowest positions -- no score is computed here.
"""
from __future__ import annotations

import concurrent.futures
import dataclasses
import math
import os
from typing import Optional

import numpy as np
import torch

BF16_NAN = np.uint16(0x7FC0)
E4M3_NAN = np.uint8(0x7F)

# Storage codes for the 17 integers -8..8, produced by torch's own
# round-to-nearest conversions (both formats hold these integers exactly).
_INT_VALUES = torch.arange(-8, 9, dtype=torch.float32)
_BF16_OF_INT = _INT_VALUES.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16).copy()
_E4M3_OF_INT = _INT_VALUES.to(torch.float8_e4m3fn).view(torch.uint8).numpy().copy()


def encode_int(vals: np.ndarray, dtype: str) -> np.ndarray:
    """Encode integers in [-8, 8] as bf16 (uint16 bits) or E4M3 (uint8 bits)."""
    table = _BF16_OF_INT if dtype == "bf16" else _E4M3_OF_INT
    vals = np.asarray(vals)
    out = np.empty(vals.shape, dtype=table.dtype)
    flat_in, flat_out = vals.reshape(-1), out.reshape(-1)
    step = 1 << 26  # in slices, so that the index temporaries stay small
    for s in range(0, flat_in.size, step):
        flat_out[s:s + step] = table[flat_in[s:s + step].astype(np.int64) + 8]
    return out


def encode_bf16(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (nearest-even, via torch) and return the bits."""
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _normal_bf16(rng: np.random.Generator, shape, chunk: int = 1 << 22) -> np.ndarray:
    """bf16(N(0,1)) bits.  Chunk c draws from its own child of one seed taken from
    rng, so the values do not depend on how many threads fill the chunks."""
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.uint16)
    base = np.random.SeedSequence(int(rng.integers(0, 2**63 - 1)))
    nchunks = (n + chunk - 1) // chunk
    kids = base.spawn(nchunks)

    def fill(c):
        s, e = c * chunk, min(n, (c + 1) * chunk)
        g = np.random.Generator(np.random.PCG64(kids[c]))
        out[s:e] = encode_bf16(g.standard_normal(e - s, dtype=np.float32))

    if nchunks <= 1:
        for c in range(nchunks):
            fill(c)
    else:
        workers = min(nchunks, os.cpu_count() or 1, 32)
        with concurrent.futures.ThreadPoolExecutor(workers) as ex:
            list(ex.map(fill, range(nchunks)))
    return out.reshape(shape)


@dataclasses.dataclass
class Case:
    """One synthetic problem: paged cache + queries, as host numpy arrays."""

    name: str
    kind: str  # "decode", "prefill" or "mixed"
    seed: int
    # paged layout
    bs: int
    num_blocks: int
    seq_lens: np.ndarray      # int32 [B]
    block_table: np.ndarray   # int32 [B, max_blocks], -1 past a sequence's pages
    # queries
    q_seq: np.ndarray         # int32 [Nq] sequence of each query
    q_pos: np.ndarray         # int32 [Nq] absolute position of each query
    n_elig: np.ndarray        # int32 [Nq] positions a query may see (q_pos + 1)
    # attention operands
    Hq: int
    Dqk: int
    Dv: int
    latent: bool              # V rows are the first Dv dims of the K rows
    q: np.ndarray             # uint16 bf16 bits [Nq, Hq, Dqk]
    k_pool: np.ndarray        # uint16 bf16 bits [NB, bs, Dkv]
    v_pool: np.ndarray        # same object as k_pool when latent
    # indexer operands
    H_i: int
    D_i: int
    idx_dtype: str            # "bf16" or "fp8"
    q_idx: np.ndarray         # encoded [Nq, H_i, D_i]
    kidx_pool: np.ndarray     # encoded [NB, bs, D_i]
    w: np.ndarray             # float32 [Nq, H_i]
    K: int
    sm_scale: float
    tie_positions: Optional[list] = None  # per sequence, sorted positions tied at the max

    @property
    def B(self) -> int:
        return int(self.seq_lens.shape[0])

    @property
    def Nq(self) -> int:
        return int(self.q_seq.shape[0])

    @property
    def max_blocks(self) -> int:
        return int(self.block_table.shape[1])

    @property
    def max_len(self) -> int:
        return int(self.seq_lens.max()) if self.B else 0

    @property
    def Dkv(self) -> int:
        return int(self.k_pool.shape[-1])


def _layout(rng, seq_lens, bs, extra_pages=0):
    nblk = [(int(L) + bs - 1) // bs for L in seq_lens]
    nb_used = sum(nblk)
    num_blocks = nb_used + extra_pages
    perm = rng.permutation(num_blocks).astype(np.int32)
    max_blocks = max(nblk) if nblk else 1
    bt = np.full((len(seq_lens), max(max_blocks, 1)), -1, dtype=np.int32)
    off = 0
    for b, n in enumerate(nblk):
        bt[b, :n] = perm[off:off + n]
        off += n
    return num_blocks, bt, perm[nb_used:]


def make_case(name: str = "custom", *, seed: int = 0, kind: str = "decode",
              seq_lens=(4096,), T: int = 0, bs: int = 64,
              Hq: int = 16, Dqk: int = 128, Dv: int = 128, latent: bool = False,
              H_i: int = 4, D_i: int = 64, idx_dtype: str = "bf16", K: int = 256,
              tie_frac: float = 0.0, poison: bool = True, extra_pages: int = 0,
              q_rows=None, q_per_seq=None) -> Case:
    """Draw one case.  kind="prefill" uses a single sequence of T tokens with one
    query per token (q_pos = t); kind="decode" has one query per sequence at its
    last position; kind="mixed" gives sequence b the q_per_seq[b] queries at its
    last positions (1: a decode step, L_b: a whole prompt, in between: a prefill
    chunk over an existing prefix).  q_rows (prefill only) keeps a subset of the
    T queries."""
    rng = np.random.Generator(np.random.PCG64(seed))
    if kind == "prefill":
        seq_lens = np.array([T], dtype=np.int32)
    else:
        seq_lens = np.asarray(seq_lens, dtype=np.int32)
    B = int(seq_lens.shape[0])
    num_blocks, bt, spare = _layout(rng, seq_lens, bs, extra_pages)

    if kind == "prefill":
        q_pos = np.arange(T, dtype=np.int32) if q_rows is None else np.asarray(q_rows, np.int32)
        q_seq = np.zeros_like(q_pos)
    elif kind == "mixed":
        n_q = np.asarray(q_per_seq, dtype=np.int64)
        assert n_q.shape == (B,) and np.all(n_q >= 1) and np.all(n_q <= seq_lens)
        q_seq = np.repeat(np.arange(B, dtype=np.int32), n_q)
        q_pos = np.concatenate([np.arange(int(L) - int(n), int(L), dtype=np.int32)
                                for L, n in zip(seq_lens, n_q)])
    else:
        q_seq = np.arange(B, dtype=np.int32)
        q_pos = (seq_lens - 1).astype(np.int32)
    Nq = int(q_seq.shape[0])
    n_elig = (q_pos + 1).astype(np.int32)

    Dkv = Dqk
    k_pool = _normal_bf16(rng, (num_blocks, bs, Dkv))
    v_pool = k_pool if latent else _normal_bf16(rng, (num_blocks, bs, Dv))
    q = _normal_bf16(rng, (Nq, Hq, Dqk))

    tie_positions = None
    if tie_frac > 0.0:
        sign = rng.choice(np.array([-1, 1], dtype=np.int8), size=(B, D_i))
        qi = (sign[:, None, :] * rng.integers(0, 9, size=(B, H_i, D_i), dtype=np.int8)).astype(np.int8)
        qi[:, 0, 0] = sign[:, 0] * rng.integers(1, 9, size=B, dtype=np.int8)
        w_int = rng.integers(0, 5, size=(B, H_i))
        w_int[:, 0] = rng.integers(1, 5, size=B)
        kint = np.zeros((num_blocks, bs, D_i), dtype=np.int8)
        tie_positions = []
        for b in range(B):
            L = int(seq_lens[b])
            u = rng.integers(0, 16, size=(L, D_i), dtype=np.int8)
            # U{-8..8} without 8*s_d: s_d=+1 -> -8..7, s_d=-1 -> -7..8
            vals = u - np.where(sign[b] > 0, 8, 7).astype(np.int8)[None, :]
            n_tie = int(round(tie_frac * L))
            tied = np.sort(rng.choice(L, size=n_tie, replace=False)).astype(np.int64)
            vals[tied] = (8 * sign[b]).astype(np.int8)[None, :]
            tie_positions.append(tied.astype(np.int32))
            pages = bt[b, :(L + bs - 1) // bs]
            full = (L // bs) * bs
            kint[pages[:L // bs]] = vals[:full].reshape(-1, bs, D_i)
            if full < L:
                kint[pages[-1], :L - full] = vals[full:]
        if kind != "decode":
            raise ValueError("tie construction is defined for decode cases")
        q_idx = encode_int(qi, idx_dtype)
        kidx_pool = encode_int(kint, idx_dtype)
        w = w_int.astype(np.float32)
    else:
        q_idx = encode_int(rng.integers(-8, 9, size=(Nq, H_i, D_i), dtype=np.int8), idx_dtype)
        kidx_pool = encode_int(rng.integers(-8, 9, size=(num_blocks, bs, D_i), dtype=np.int8),
                               idx_dtype)
        w = rng.integers(0, 5, size=(Nq, H_i)).astype(np.float32)

    if poison:
        nan_idx = BF16_NAN if idx_dtype == "bf16" else E4M3_NAN
        for b in range(B):
            L = int(seq_lens[b])
            if L % bs:
                page = bt[b, L // bs]
                k_pool[page, L % bs:] = BF16_NAN
                if not latent:
                    v_pool[page, L % bs:] = BF16_NAN
                kidx_pool[page, L % bs:] = nan_idx
        for page in spare:
            k_pool[page] = BF16_NAN
            if not latent:
                v_pool[page] = BF16_NAN
            kidx_pool[page] = nan_idx

    return Case(name=name, kind=kind, seed=seed, bs=bs, num_blocks=num_blocks,
                seq_lens=seq_lens, block_table=bt, q_seq=q_seq, q_pos=q_pos, n_elig=n_elig,
                Hq=Hq, Dqk=Dqk, Dv=Dv, latent=latent, q=q, k_pool=k_pool, v_pool=v_pool,
                H_i=H_i, D_i=D_i, idx_dtype=idx_dtype, q_idx=q_idx, kidx_pool=kidx_pool, w=w,
                K=K, sm_scale=float(np.float32(1.0 / math.sqrt(Dqk))),
                tie_positions=tie_positions)


LATENT = dict(Hq=64, Dqk=576, Dv=512, latent=True, H_i=64, D_i=128, idx_dtype="fp8", K=2048)
TINY = dict(Hq=16, Dqk=128, Dv=128, latent=False, H_i=4, D_i=64, idx_dtype="bf16", K=256)


def dec_batch_lens(seed: int = 1, B: int = 32, lo: int = 8192, hi: int = 32768) -> np.ndarray:
    rng = np.random.Generator(np.random.PCG64(seed + 1000))
    return rng.integers(lo, hi + 1, size=B).astype(np.int32)


def config(name: str, **overrides) -> Case:
    """The five named workloads (seeds 0-4 in this order); overrides shrink them for tests."""
    if name == "dec-tiny":
        kw = dict(seed=0, kind="decode", seq_lens=(4096,), **TINY)
    elif name == "dec-batch":
        kw = dict(seed=1, kind="decode", seq_lens=dec_batch_lens(), **LATENT)
    elif name == "prefill":
        kw = dict(seed=2, kind="prefill", T=16384, **LATENT)
    elif name == "long-dec":
        kw = dict(seed=3, kind="decode", seq_lens=(262144, 196608, 131072, 65536),
                  tie_frac=0.05, **LATENT)
    elif name == "million":
        kw = dict(seed=4, kind="decode", seq_lens=(1 << 20,) * 8, **LATENT)
    else:
        raise KeyError(name)
    kw.update(overrides)
    return make_case(name, **kw)


NAMES = ("dec-tiny", "dec-batch", "prefill", "long-dec", "million")
