// index_prefill_tc.cu -- tensor-core indexer score for a prefill: many queries
// of one sequence scored against its causal prefix (FP8 E4M3 keys, 64
// indexer heads of dimension 128, pages of 64 positions).
//
// "Day-0 Adaptation of Trillion-Parameter MoE Models on Domestic GPUs",
// section 3 (3): the prefill stage processes the whole prompt at once and is
// compute-intensive.  Scoring is a dense causal contraction
//     D[p][(r, h)] = k_idx[p] . q_idx[r][h]
// followed by s[r][p] = sum_h w[r][h] * max(0, D[p][(r, h)]) for p <= q_pos[r].
//
// Queries are taken in blocks of 16 whose indexer heads (16 x 64 x 128 B =
// 128 KB) stay in shared memory while the block's key tiles stream past:
// per 128-position tile, four tcgen05.mma.kind::f8f6f4 groups of N = 256
// (4 queries x 64 heads) accumulate into two alternating 256-column TMEM
// buffers.  Sixteen epilogue warps (four per TMEM lane quadrant, one per
// query of the group's four) apply ReLU, the head weights and the head sum,
// and store the scores of the causal positions; the epilogue is bound by its
// instruction latency, so more warps per quadrant hide more of it.  Work items (block, key tile) are laid end
// to end and split evenly over one CTA per SM, which balances the triangle.
// Warp roles: 0-15 epilogue, 16 TMA producer, 17 TMEM owner + MMA issuer.
// Every wait is bounded (DSA_STATUS_TIMEOUT, then the CTA winds down).
#include "device_common.cuh"
#include "dsa_internal.cuh"
#include "sm100.cuh"

namespace dsa {

namespace {

using namespace sm100;

constexpr int kQB = 16;          // queries per block
constexpr int kGroupQ = 4;       // queries per MMA (N = 256)
constexpr int kGroups = kQB / kGroupQ;
constexpr int kHeads = 64;
constexpr int kRowBytes = 128;
constexpr int kTileRows = 128;
constexpr int kStages = 4;
constexpr int kTileBytes = kTileRows * kRowBytes;
constexpr int kPageBytes = 64 * kRowBytes;
constexpr int kGroupBytes = kGroupQ * kHeads * kRowBytes;  // 32 KB
constexpr int kMaxBlocks = 2048;                           // Nq <= 32768
constexpr int kEpiWarps = 16;                              // epilogue warps
constexpr int kEpiThreads = kEpiWarps * 32;
constexpr int kQPerWarp = kGroupQ / (kEpiWarps / 4);       // queries per epilogue warp
constexpr int kProducerWarp = kEpiWarps, kMmaWarp = kEpiWarps + 1;
constexpr int kThreads = kEpiThreads + 64;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kIdesc = instr_desc(128, kGroupQ * kHeads, 0, 0);

struct __align__(1024) Smem {
  uint8_t b[kGroups][kGroupBytes];   // 128 KB: q_idx of the current block
  uint8_t a[kStages][kTileBytes];    // 64 KB: key tiles
  float w[kQB][kHeads];              // head weights of the current block
  uint64_t full[kStages], empty[kStages], bfull, bempty, accfull[2], accempty[2], done, epsync;
  uint32_t tmem_base;
  int abort;
  int prefix[kMaxBlocks + 1];
};

__device__ __forceinline__ void fail(Smem& s, int* status) {
  s.abort = 1;
  flag_status(status, DSA_STATUS_TIMEOUT);
}

__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile int* abort) {
  return __all_sync(0xffffffffu, mbar_wait(bar, parity, abort));
}

struct SeqInfo {
  long long L;
};

// eligible positions of query r: p <= q_pos[r] and p < L
__device__ __forceinline__ long long elig(const IndexParams& a, long long L, int r) {
  if (r >= a.Nq) return 0;
  long long last = a.q_pos ? (long long)__ldg(&a.q_pos[r]) : (long long)r;
  if (last > L - 1) last = L - 1;
  return last + 1 > 0 ? last + 1 : 0;
}

__global__ void __launch_bounds__(kThreads, 1)
    k_index_prefill_tc(const __grid_constant__ CUtensorMap map_k,
                       const __grid_constant__ CUtensorMap map_q, IndexParams a) {
  extern __shared__ uint8_t smraw[];
  Smem& s = *reinterpret_cast<Smem*>((reinterpret_cast<uintptr_t>(smraw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nblocks = (a.Nq + kQB - 1) / kQB;
  launch_dependents();
  if (threadIdx.x == 0) {
    s.prefix[0] = 0;
    s.abort = 0;
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&s.full[i], 1);
      mbar_init(&s.empty[i], 1);
    }
    mbar_init(&s.bfull, 1);
    mbar_init(&s.bempty, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s.accfull[i], 1);
      mbar_init(&s.accempty[i], kEpiThreads);
    }
    mbar_init(&s.done, 1);
    mbar_init(&s.epsync, kEpiThreads);
    fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(&s.tmem_base, kTmemCols);
    tmem_relinquish();
  }
  if (warp == kProducerWarp && lane == 0) {
    tma_prefetch_desc(&map_k);
    tma_prefetch_desc(&map_q);
  }
  grid_dependency_wait();  // inputs below may come from the previous kernel
  const int b = a.seq_const;
  long long L = 0;
  if (b >= 0 && b < a.lay.batch) {
    L = __ldg(&a.lay.seq_lens[b]);
    const long long cap = (long long)a.lay.maxb * a.lay.bs;
    if (L > cap || L > a.ld) {
      if (blockIdx.x == 0 && threadIdx.x == 0) flag_status(a.status, DSA_STATUS_BAD_LENGTH);
      L = L < cap ? L : cap;
      L = L < a.ld ? L : a.ld;
    }
  } else if (blockIdx.x == 0 && threadIdx.x == 0) {
    flag_status(a.status, DSA_STATUS_BAD_INDEX);
  }

  // key tiles per query block (the block's largest eligible count)
  for (int bi = threadIdx.x; bi < nblocks; bi += kThreads) {
    long long n = 0;
    for (int j = 0; j < kQB; ++j) {
      const long long e = elig(a, L, bi * kQB + j);
      n = e > n ? e : n;
    }
    s.prefix[bi + 1] = (int)((n + kTileRows - 1) / kTileRows);
  }
  __syncthreads();
  if (warp == 0) {
    const int per = (nblocks + 31) / 32;
    const int i0 = 1 + lane * per, i1 = min(nblocks + 1, i0 + per);
    int sum = 0;
    for (int i = i0; i < i1; ++i) sum += s.prefix[i];
    int incl = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += t;
    }
    int run = incl - sum;
    for (int i = i0; i < i1; ++i) {
      run += s.prefix[i];
      s.prefix[i] = run;
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  const uint32_t tbase = s.tmem_base;
  const int total = s.prefix[nblocks];
  const int lo = (int)((long long)blockIdx.x * total / gridDim.x);
  const int hi = (int)((long long)(blockIdx.x + 1) * total / gridDim.x);
  auto block_of = [&](int item) {
    int l = 0, h = nblocks - 1;
    while (l < h) {
      const int m = (l + h + 1) >> 1;
      if (s.prefix[m] <= item) l = m; else h = m - 1;
    }
    return l;
  };

  if (warp == kProducerWarp) {
    // ------------------------------------------------------------ producer --
    if (lane == 0 && lo < hi) {
      int bi = block_of(lo), cur = -1, nbl = 0, stage = 0, issued = 0;
      uint32_t phase = 0, issued_parity[kStages];
      bool ok = true;
      for (int item = lo; item < hi; ++item) {
        while (s.prefix[bi + 1] <= item) ++bi;
        if (bi != cur) {
          if (nbl > 0 && !mbar_wait(&s.bempty, (nbl - 1) & 1, &s.abort)) { ok = false; break; }
          mbar_arrive_expect_tx(&s.bfull, kGroups * kGroupBytes);
          for (int g = 0; g < kGroups; ++g)
            tma_load_2d(s.b[g], &map_q, &s.bfull, 0, (bi * kQB + g * kGroupQ) * kHeads);
          ++nbl;
          cur = bi;
        }
        const long long p0 = (long long)(item - s.prefix[bi]) * kTileRows;
        const long long rows = min((long long)kTileRows, L - p0);
        const int pages = rows > 64 ? 2 : 1;
        if (!mbar_wait(&s.empty[stage], phase ^ 1, &s.abort)) { ok = false; break; }
        mbar_arrive_expect_tx(&s.full[stage], pages * kPageBytes);
        for (int pg = 0; pg < pages; ++pg) {
          int page = __ldg(&a.lay.bt[(long long)b * a.lay.maxb + p0 / 64 + pg]);
          if (page < 0 || page >= a.lay.nb) page = 0;  // the epilogue flags and masks it
          tma_load_2d(s.a[stage] + pg * kPageBytes, &map_k, &s.full[stage], 0, page * 64);
        }
        issued_parity[stage] = phase;
        ++issued;
        if (++stage == kStages) {
          stage = 0;
          phase ^= 1;
        }
      }
      if (!ok) fail(s, a.status);
      const int pend = issued < kStages ? issued : kStages;
      for (int i = 0; i < pend; ++i) {
        const int st = (stage - 1 - i + 2 * kStages) % kStages;
        mbar_wait(&s.full[st], issued_parity[st], &s.abort, 100000000ull);
      }
    }
  } else if (warp == kMmaWarp) {
    // -------------------------------------------------------- MMA issuer --
    if (lane == 0 && lo < hi) {
      int bi = block_of(lo), cur = -1, nbl = 0, stage = 0, it = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int item = lo; item < hi && ok; ++item) {
        while (s.prefix[bi + 1] <= item) ++bi;
        if (bi != cur) {
          if (nbl > 0) mma_commit(&s.bempty);
          if (!mbar_wait(&s.bfull, nbl & 1, &s.abort)) { ok = false; break; }
          ++nbl;
          cur = bi;
        }
        if (!mbar_wait(&s.full[stage], phase, &s.abort)) { ok = false; break; }
        tc_fence_after();
        const uint32_t a0 = smem_u32(s.a[stage]);
        for (int g = 0; g < kGroups; ++g, ++it) {
          const int acc = it & 1;
          if (!mbar_wait(&s.accempty[acc], ((it >> 1) & 1) ^ 1, &s.abort)) { ok = false; break; }
          tc_fence_after();
          const uint32_t b0 = smem_u32(s.b[g]);
#pragma unroll
          for (int k = 0; k < kRowBytes / 32; ++k)
            mma_f8f6f4(tbase + acc * 256, smem_desc(a0 + 32 * k, 16, 1024, kSwizzle128B),
                       smem_desc(b0 + 32 * k, 16, 1024, kSwizzle128B), kIdesc, k > 0);
          mma_commit(&s.accfull[acc]);
        }
        mma_commit(&s.empty[stage]);
        if (++stage == kStages) {
          stage = 0;
          phase ^= 1;
        }
      }
      if (!ok) fail(s, a.status);
      mma_commit(&s.done);
      mbar_wait(&s.done, 0, &s.abort, 100000000ull);
    }
  } else {
    // ----------------------------------------------------------- epilogue --
    const int quad = warp & 3, qsel = warp >> 2;  // lanes 32*quad.., queries kQPerWarp*qsel..
    const int et = threadIdx.x;                    // 0..kEpiThreads-1
    uint32_t ep = 0;
    if (lo < hi) {
      int bi = block_of(lo), cur = -1, it = 0;
      bool ok = true;
      long long n_q[kQPerWarp * kGroups];  // eligible counts of this thread's queries
      for (int item = lo; item < hi && ok; ++item) {
        while (s.prefix[bi + 1] <= item) ++bi;
        if (bi != cur) {
          // all epilogue threads are past the previous block's items here
          mbar_arrive(&s.epsync);
          if (!warp_wait(&s.epsync, ep, &s.abort)) { ok = false; break; }
          ep ^= 1;
          for (int i = et; i < kQB * kHeads; i += kEpiThreads) {
            const int r = bi * kQB + i / kHeads;
            s.w[i / kHeads][i % kHeads] = r < a.Nq ? __ldg(&a.w[(long long)r * kHeads + i % kHeads]) : 0.0f;
          }
          mbar_arrive(&s.epsync);
          if (!warp_wait(&s.epsync, ep, &s.abort)) { ok = false; break; }
          ep ^= 1;
#pragma unroll
          for (int g = 0; g < kGroups; ++g)
#pragma unroll
            for (int j = 0; j < kQPerWarp; ++j)
              n_q[kQPerWarp * g + j] = elig(a, L, bi * kQB + g * kGroupQ + kQPerWarp * qsel + j);
          cur = bi;
        }
        const long long p = (long long)(item - s.prefix[bi]) * kTileRows + quad * 32 + lane;
        bool page_ok = true;
        if (p < L) {
          const int page = __ldg(&a.lay.bt[(long long)b * a.lay.maxb + p / 64]);
          page_ok = page >= 0 && page < a.lay.nb;
        }
        for (int g = 0; g < kGroups; ++g, ++it) {
          const int acc = it & 1;
          if (!warp_wait(&s.accfull[acc], (it >> 1) & 1, &s.abort)) { ok = false; break; }
          tc_fence_after();
          float sc[kQPerWarp];
#pragma unroll
          for (int j = 0; j < kQPerWarp; ++j) {
            const int ql = g * kGroupQ + kQPerWarp * qsel + j;  // query within the block
            const uint32_t taddr = tbase + ((uint32_t)(quad * 32) << 16) + acc * 256 +
                                   (kQPerWarp * qsel + j) * kHeads;
            // the weights are read four at a time: with one shared-memory load
            // per FMA the shared-memory pipe paced the epilogue
            const float4* wq = reinterpret_cast<const float4*>(s.w[ql]);
            uint32_t v[32];
            float s0 = 0.0f, s1 = 0.0f;
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
              tmem_ld_32cols(taddr + 32 * hh, v);
              tmem_wait_ld();
#pragma unroll
              for (int h = 0; h < 32; h += 4) {
                const float4 wv = wq[(32 * hh + h) >> 2];
                s0 = fmaf(wv.x, fmaxf(__uint_as_float(v[h]), 0.0f), s0);
                s1 = fmaf(wv.y, fmaxf(__uint_as_float(v[h + 1]), 0.0f), s1);
                s0 = fmaf(wv.z, fmaxf(__uint_as_float(v[h + 2]), 0.0f), s0);
                s1 = fmaf(wv.w, fmaxf(__uint_as_float(v[h + 3]), 0.0f), s1);
              }
            }
            sc[j] = (s0 + s1) + 0.0f;
          }
          tc_fence_before();
          mbar_arrive(&s.accempty[acc]);
#pragma unroll
          for (int j = 0; j < kQPerWarp; ++j) {
            const int r = bi * kQB + g * kGroupQ + kQPerWarp * qsel + j;
            if (p < n_q[kQPerWarp * g + j]) {
              float out = sc[j];
              if (!page_ok) {
                flag_status(a.status, DSA_STATUS_BAD_BLOCK);
                out = -INFINITY;
              }
              a.scores[(long long)r * a.ld + p] = out;
            }
          }
        }
      }
      if (!ok) fail(s, a.status);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tbase, kTmemCols);
  }
}

}  // namespace

bool index_prefill_tc_eligible(const IndexParams& p) {
  return p.dtype == DSA_FP8_E4M3 && p.H == kHeads && p.D == kRowBytes && p.lay.bs == 64 &&
         p.Nq >= 1 && p.Nq <= kMaxBlocks * kQB && p.seq_const >= 0 &&
         (reinterpret_cast<uintptr_t>(p.w) & 15u) == 0;
}

int launch_index_prefill_tc(const IndexParams& p, cudaStream_t s) {
  CUtensorMap mk, mq;
  int rc = make_tmap_2d(&mk, p.kidx, true, kRowBytes, (uint64_t)p.lay.nb * 64, kRowBytes,
                        kRowBytes, 64);
  if (rc) return rc;
  rc = make_tmap_2d(&mq, p.q_idx, true, kRowBytes, (uint64_t)p.Nq * kHeads, kRowBytes, kRowBytes,
                    kGroupQ * kHeads);
  if (rc) return rc;
  const size_t smem = sizeof(Smem) + 1024;
  rc = ensure_dynamic_smem((const void*)k_index_prefill_tc, (int)smem,
                          "index_score prefill (tensor cores)");
  if (rc) return rc;
  const long long nblocks = (p.Nq + kQB - 1) / kQB;
  const long long max_items = nblocks * ((p.ld + kTileRows - 1) / kTileRows);
  long long grid = sm_count();
  if (grid > max_items) grid = max_items;
  if (grid < 1) grid = 1;
  const cudaError_t e =
      launch_pdl(k_index_prefill_tc, dim3((unsigned)grid), dim3(kThreads), smem, s, mk, mq, p);
  count_launch();
  if (e != cudaSuccess) return set_error(DSA_ERR_CUDA, cudaGetErrorString(e));
  return check_launch("index_score prefill (tensor cores)");
}

}  // namespace dsa
