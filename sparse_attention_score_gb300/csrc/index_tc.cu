// index_tc.cu -- tensor-core indexer score for FP8 E4M3 indexer keys with 64
// indexer heads of dimension 128 on a paged cache of 64-position pages.
//
// "Day-0 Adaptation of Trillion-Parameter MoE Models on Domestic GPUs",
// section 3 (1): score every cached position of the query's sequence with the
// lightweight indexer, s[p] = sum_h w[h] * max(0, q_idx[h] . k_idx[p]).
//
// Per 128-position tile this is one small GEMM: A = the tile's keys
// (128 positions x 128 bytes, K-major, exactly one 128-byte swizzle row per
// position), B = the query's 64 indexer heads (64 x 128 bytes), D = 128 x 64
// fp32 accumulators in TMEM, produced by four tcgen05.mma.kind::f8f6f4
// (K = 32 each).  The epilogue reads one TMEM lane (= one position) per
// thread, applies ReLU, the head weights and the head sum, and stores the
// fp32 score.  With the integer-valued inputs of the pages' workloads every
// product and partial sum is an integer below 2^14 per head, so the score is
// exact.
//
// Warp roles (192 threads, persistent, 2 CTAs per SM):
//   warps 0-3  epilogue: TMEM -> registers -> ReLU . w -> global scores
//   warp 4     TMA producer: block-table lookup, two 8 KB page loads per tile
//   warp 5     TMEM allocation and MMA issue (one lane)
// Tiles of all queries are laid end to end and split evenly over the CTAs.
// Every wait is bounded; on a timeout the CTA sets DSA_STATUS_TIMEOUT, drains
// its own copies and MMAs, frees TMEM and returns.
#include "device_common.cuh"
#include "dsa_internal.cuh"
#include "sm100.cuh"

namespace dsa {

namespace {

using namespace sm100;

constexpr int kStages = 4;
constexpr int kTileRows = 128;
constexpr int kRowBytes = 128;  // D_i = 128 FP8 codes
constexpr int kHeads = 64;      // MMA N
constexpr int kTileBytes = kTileRows * kRowBytes;
constexpr int kPageBytes = 64 * kRowBytes;
constexpr int kQBytes = kHeads * kRowBytes;
constexpr int kMaxQueries = 2048;
constexpr int kThreads = 192;
constexpr uint32_t kTmemCols = 128;  // two 64-column accumulators
constexpr uint32_t kIdesc = instr_desc(128, kHeads, 0, 0);

struct __align__(1024) Smem {
  uint8_t a[kStages][kTileBytes];
  uint8_t b[2][kQBytes];
  uint64_t full[kStages], empty[kStages], bfull[2], bempty[2], accfull[2], accempty[2], done;
  uint32_t tmem_base;
  int abort;
  int prefix[kMaxQueries + 1];  // tiles of queries [0, r)
};

struct Query {
  int b;       // sequence
  long long n; // eligible positions
};

__device__ __forceinline__ Query query_info(const IndexParams& a, int r) {
  Query q{-1, 0};
  const int b = a.seq_const >= 0 ? a.seq_const : (a.q_seq ? __ldg(&a.q_seq[r]) : r);
  if (b < 0 || b >= a.lay.batch) return q;
  long long L = __ldg(&a.lay.seq_lens[b]);
  const long long cap = (long long)a.lay.maxb * a.lay.bs;
  if (L > cap) L = cap;
  if (L > a.ld) L = a.ld;
  long long last = a.q_pos ? (long long)__ldg(&a.q_pos[r]) : L - 1;
  if (last > L - 1) last = L - 1;
  q.b = b;
  q.n = last + 1 > 0 ? last + 1 : 0;
  return q;
}

// Walks the flattened tile list in order, tracking the current query.
struct Cursor {
  int r;
  __device__ void seek(const Smem& s, int nq, int item) {
    int lo = 0, hi = nq;  // last r with prefix[r] <= item
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (s.prefix[mid] <= item) lo = mid; else hi = mid - 1;
    }
    r = lo;
  }
  __device__ void advance(const Smem& s, int item) {
    while (s.prefix[r + 1] <= item) ++r;
  }
};

// Tile t of query r left out by the caller's skip mask.
__device__ __forceinline__ bool tile_skipped(const IndexParams& a, int r, long long t) {
  return a.skip && __ldg(&a.skip[(long long)r * a.skip_stride + t]) != 0;
}

__device__ __forceinline__ void fail(Smem& s, int* status) {
  s.abort = 1;
  flag_status(status, DSA_STATUS_TIMEOUT);
}

__global__ void __launch_bounds__(kThreads, 2)
    k_index_tc(const __grid_constant__ CUtensorMap map_k, const __grid_constant__ CUtensorMap map_q,
               IndexParams a) {
  extern __shared__ uint8_t smraw[];
  Smem& s = *reinterpret_cast<Smem*>((reinterpret_cast<uintptr_t>(smraw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nq = a.Nq;
  launch_dependents();

  if (threadIdx.x == 0) {
    s.prefix[0] = 0;
    s.abort = 0;
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&s.full[i], 1);
      mbar_init(&s.empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s.bfull[i], 1);
      mbar_init(&s.bempty[i], 1);
      mbar_init(&s.accfull[i], 1);
      mbar_init(&s.accempty[i], 128);
    }
    mbar_init(&s.done, 1);
    fence_mbar_init();
  }
  if (warp == 5) {
    tmem_alloc(&s.tmem_base, kTmemCols);
    tmem_relinquish();
  }
  if (warp == 4 && lane == 0) {
    tma_prefetch_desc(&map_k);
    tma_prefetch_desc(&map_q);
  }
  grid_dependency_wait();  // inputs below may come from the previous kernel
  // tiles per query, then an exclusive prefix (one warp)
  for (int r = threadIdx.x; r < nq; r += kThreads) {
    const Query q = query_info(a, r);
    s.prefix[r + 1] = (int)((q.n + kTileRows - 1) / kTileRows);
    if (blockIdx.x == 0) {
      if (q.b < 0) {
        flag_status(a.status, DSA_STATUS_BAD_INDEX);
      } else {
        const long long L = __ldg(&a.lay.seq_lens[q.b]);
        if (L > (long long)a.lay.maxb * a.lay.bs || L > a.ld)
          flag_status(a.status, DSA_STATUS_BAD_LENGTH);
      }
    }
  }
  __syncthreads();
  if (warp == 0) {
    // inclusive scan of prefix[1..nq] by one warp, chunked per lane
    const int per = (nq + 31) / 32;
    const int i0 = 1 + lane * per, i1 = min(nq + 1, i0 + per);
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
  const int total = s.prefix[nq];
  const int lo = (int)((long long)blockIdx.x * total / gridDim.x);
  const int hi = (int)((long long)(blockIdx.x + 1) * total / gridDim.x);

  if (warp == 4) {
    // ------------------------------------------------------ TMA producer --
    if (lane == 0 && lo < hi) {
      // The block-table entries of tile i + 1 are loaded while tile i waits
      // for its stage, so their latency is off the issue path.
      struct TileLoad {
        int r, pages;
        long long p0;
        int page[2];
      };
      Cursor ca;
      ca.seek(s, nq, lo);
      int acur = -1;
      Query aq{};
      auto look = [&](int item) {
        TileLoad t;
        ca.advance(s, item);
        if (ca.r != acur) {
          acur = ca.r;
          aq = query_info(a, acur);
        }
        t.r = acur;
        t.p0 = (long long)(item - s.prefix[acur]) * kTileRows;
        const long long rows = min((long long)kTileRows, aq.n - t.p0);
        t.pages = (int)((rows + 63) / 64);
#pragma unroll
        for (int pg = 0; pg < 2; ++pg) {
          int page = 0;
          if (pg < t.pages) page = __ldg(&a.lay.bt[(long long)aq.b * a.lay.maxb + t.p0 / 64 + pg]);
          t.page[pg] = page;
        }
        return t;
      };
      TileLoad nxt = look(lo);
      int cur = -1, nb = 0, stage = 0;
      uint32_t phase = 0;
      uint32_t issued_parity[kStages];
      int issued = 0;
      for (int item = lo; item < hi; ++item) {
        const TileLoad t = nxt;
        if (item + 1 < hi) nxt = look(item + 1);
        // skipped tiles take no stage: the MMA issuer and the epilogue skip
        // the same items
        if (tile_skipped(a, t.r, t.p0 / kTileRows)) continue;
        if (t.r != cur) {
          cur = t.r;
          const int slot = nb & 1;
          if (nb >= 2 && !mbar_wait(&s.bempty[slot], ((nb >> 1) - 1) & 1, &s.abort)) {
            fail(s, a.status);
            break;
          }
          mbar_arrive_expect_tx(&s.bfull[slot], kQBytes);
          tma_load_2d(s.b[slot], &map_q, &s.bfull[slot], 0, cur * kHeads);
          ++nb;
        }
        if (!mbar_wait(&s.empty[stage], phase ^ 1, &s.abort)) {
          fail(s, a.status);
          break;
        }
        mbar_arrive_expect_tx(&s.full[stage], t.pages * kPageBytes);
        for (int pg = 0; pg < t.pages; ++pg) {
          int page = t.page[pg];
          if (page < 0 || page >= a.lay.nb) page = 0;  // epilogue flags and masks it
          tma_load_2d(s.a[stage] + pg * kPageBytes, &map_k, &s.full[stage], 0, page * 64);
        }
        issued_parity[stage] = phase;
        ++issued;
        if (++stage == kStages) {
          stage = 0;
          phase ^= 1;
        }
      }
      // drain: the last (up to kStages) loads must land before the CTA exits
      const int pend = issued < kStages ? issued : kStages;
      for (int i = 0; i < pend; ++i) {
        const int st = (stage - 1 - i + 2 * kStages) % kStages;
        mbar_wait(&s.full[st], issued_parity[st], &s.abort, 100000000ull);
      }
    }
  } else if (warp == 5) {
    // -------------------------------------------------------- MMA issuer --
    if (lane == 0 && lo < hi) {
      Cursor c;
      c.seek(s, nq, lo);
      int cur = -1, nb = 0, stage = 0, slot = 0, it = 0;
      uint32_t phase = 0;
      for (int item = lo; item < hi; ++item) {
        c.advance(s, item);
        if (tile_skipped(a, c.r, item - s.prefix[c.r])) continue;
        if (c.r != cur) {
          if (nb > 0) mma_commit(&s.bempty[(nb - 1) & 1]);
          cur = c.r;
          slot = nb & 1;
          if (!mbar_wait(&s.bfull[slot], (nb >> 1) & 1, &s.abort)) {
            fail(s, a.status);
            break;
          }
          ++nb;
        }
        const int acc = it & 1;
        if (!mbar_wait(&s.accempty[acc], ((it >> 1) & 1) ^ 1, &s.abort)) {
          fail(s, a.status);
          break;
        }
        tc_fence_after();
        if (!mbar_wait(&s.full[stage], phase, &s.abort)) {
          fail(s, a.status);
          break;
        }
        tc_fence_after();
        const uint32_t a0 = smem_u32(s.a[stage]), b0 = smem_u32(s.b[slot]);
#pragma unroll
        for (int k = 0; k < kRowBytes / 32; ++k) {
          mma_f8f6f4(tbase + acc * kHeads, smem_desc(a0 + 32 * k, 16, 1024, kSwizzle128B),
                     smem_desc(b0 + 32 * k, 16, 1024, kSwizzle128B), kIdesc, k > 0);
        }
        mma_commit(&s.empty[stage]);
        mma_commit(&s.accfull[acc]);
        if (++stage == kStages) {
          stage = 0;
          phase ^= 1;
        }
        ++it;
      }
      // every MMA issued by this thread must finish before TMEM is freed
      mma_commit(&s.done);
      mbar_wait(&s.done, 0, &s.abort, 100000000ull);
    }
  } else {
    // ----------------------------------------------------------- epilogue --
    if (lo < hi) {
      Cursor c;
      c.seek(s, nq, lo);
      int cur = -1, it = 0;
      Query q{};
      float w[kHeads];
      for (int item = lo; item < hi; ++item) {
        c.advance(s, item);
        if (c.r != cur) {
          cur = c.r;
          q = query_info(a, cur);
          const float4* wp = reinterpret_cast<const float4*>(a.w + (long long)cur * kHeads);
#pragma unroll
          for (int j = 0; j < kHeads / 4; ++j) {
            const float4 v = __ldg(wp + j);
            w[4 * j] = v.x;
            w[4 * j + 1] = v.y;
            w[4 * j + 2] = v.z;
            w[4 * j + 3] = v.w;
          }
        }
        if (tile_skipped(a, cur, item - s.prefix[cur])) {
          const long long p = (long long)(item - s.prefix[cur]) * kTileRows + warp * 32 + lane;
          if (p < q.n &&
              __ldg(&a.skip[(long long)cur * a.skip_stride + (item - s.prefix[cur])]) == kSkipInf)
            a.scores[(long long)cur * a.ld + p] = -INFINITY;
          continue;
        }
        const int acc = it & 1;
        // this lane's position and its page id, loaded before the wait for
        // the accumulator so that the load is not on the path to the store
        const long long p = (long long)(item - s.prefix[cur]) * kTileRows + warp * 32 + lane;
        const int page = p < q.n ? __ldg(&a.lay.bt[(long long)q.b * a.lay.maxb + p / 64]) : 0;
        // warp-uniform outcome: the TMEM loads below are .sync.aligned
        const bool ok = __all_sync(0xffffffffu, mbar_wait(&s.accfull[acc], (it >> 1) & 1, &s.abort));
        if (!ok) {
          fail(s, a.status);
          break;
        }
        tc_fence_after();
        const uint32_t taddr = tbase + ((uint32_t)(warp * 32) << 16) + acc * kHeads;
        uint32_t v[32];
        float sc0 = 0.0f, sc1 = 0.0f;
        tmem_ld_32cols(taddr, v);
        tmem_wait_ld();
#pragma unroll
        for (int h = 0; h < 32; h += 2) {
          sc0 = fmaf(w[h], fmaxf(__uint_as_float(v[h]), 0.0f), sc0);
          sc1 = fmaf(w[h + 1], fmaxf(__uint_as_float(v[h + 1]), 0.0f), sc1);
        }
        tmem_ld_32cols(taddr + 32, v);
        tmem_wait_ld();
#pragma unroll
        for (int h = 0; h < 32; h += 2) {
          sc0 = fmaf(w[32 + h], fmaxf(__uint_as_float(v[h]), 0.0f), sc0);
          sc1 = fmaf(w[33 + h], fmaxf(__uint_as_float(v[h + 1]), 0.0f), sc1);
        }
        tc_fence_before();
        mbar_arrive(&s.accempty[acc]);
        if (p < q.n) {
          float out = (sc0 + sc1) + 0.0f;
          if (page < 0 || page >= a.lay.nb) {
            flag_status(a.status, DSA_STATUS_BAD_BLOCK);
            out = -INFINITY;
          }
          a.scores[(long long)cur * a.ld + p] = out;
        }
        ++it;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 5) {
    tc_fence_after();
    tmem_dealloc(tbase, kTmemCols);
  }
}

}  // namespace

bool index_tc_eligible(const IndexParams& p) {
  return p.dtype == DSA_FP8_E4M3 && p.H == kHeads && p.D == kRowBytes && p.lay.bs == 64 &&
         p.Nq >= 1 && p.Nq <= kMaxQueries &&
         (reinterpret_cast<uintptr_t>(p.w) & 15u) == 0;
}

int launch_index_tc(const IndexParams& p, cudaStream_t s) {
  CUtensorMap mk, mq;
  int rc = make_tmap_2d(&mk, p.kidx, true, kRowBytes, (uint64_t)p.lay.nb * 64, kRowBytes,
                        kRowBytes, 64);
  if (rc) return rc;
  rc = make_tmap_2d(&mq, p.q_idx, true, kRowBytes, (uint64_t)p.Nq * kHeads, kRowBytes, kRowBytes,
                    kHeads);
  if (rc) return rc;
  const size_t smem = sizeof(Smem) + 1024;
  rc = ensure_dynamic_smem((const void*)k_index_tc, (int)smem, "index_score (tensor cores)");
  if (rc) return rc;
  const long long max_tiles = (long long)p.Nq * ((p.ld + kTileRows - 1) / kTileRows);
  long long grid = 2LL * sm_count();
  if (grid > max_tiles) grid = max_tiles;
  if (grid < 1) grid = 1;
  const cudaError_t e = launch_pdl(k_index_tc, dim3((unsigned)grid), dim3(kThreads), smem, s, mk, mq, p);
  count_launch();
  if (e != cudaSuccess) return set_error(DSA_ERR_CUDA, cudaGetErrorString(e));
  return check_launch("index_score (tensor cores)");
}

}  // namespace dsa
