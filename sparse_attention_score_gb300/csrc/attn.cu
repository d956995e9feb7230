// attn.cu -- stage 3 of the DSA path: exact softmax attention over the
// selected positions, their K/V rows gathered through the block table.
//
// "Day-0 Adaptation of Trillion-Parameter MoE Models on Domestic GPUs",
// section 3 (3) (prefill and decode paths) and "Day-0 Adaptation of
// Ultra-Large-Scale MoE Models on Heterogeneous AI Accelerators", section 4
// (cache gather + sparse attention).  For query r, head h and selected rows j:
//     z_j = sm_scale * q[r][h] . K_j,   out = sum_j softmax(z)_j V_j.
// Softmax runs online in fp32 (log2 domain).  The K selected rows of a query
// may be split into S ranges processed by different CTAs; each writes an
// unnormalised partial (o, m, l) and a combine kernel merges them:
//     M = max_s m_s,  l = sum_s l_s 2^(m_s - M),  o = sum_s o_s 2^(m_s - M) / l.
//
// This file holds the CUDA-core kernel, used for every shape the tensor-core
// kernel (attn_tc.cu) does not cover.
#include "device_common.cuh"
#include "dsa_internal.cuh"

namespace dsa {

namespace {

constexpr int kAttnThreads = 256;
constexpr int kAttnWarps = kAttnThreads / 32;

// grid (S, Nq); warp w owns heads w, w+8, ...; lane l owns dims l, l+32, ...
template <int HPW, int DVL>
__global__ void __launch_bounds__(kAttnThreads) k_attn_generic(AttnParams a) {
  extern __shared__ __align__(16) unsigned char smraw[];
  const int Hq = a.Hq, Dqk = a.Dqk, Dv = a.Dv;
  grid_dependency_wait();
  launch_dependents();
  __nv_bfloat16* qs = reinterpret_cast<__nv_bfloat16*>(smraw);          // [Hq][Dqk]
  float* krow = reinterpret_cast<float*>(smraw + (size_t)Hq * Dqk * 2);  // [Dqk]
  float* vrow = krow + Dqk;                                               // [Dv]
  __shared__ long long row_sh;

  const int r = blockIdx.y, split = blockIdx.x, S = gridDim.x;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int b = a.q_seq ? __ldg(&a.q_seq[r]) : (a.seq_const >= 0 ? a.seq_const : r);
  const bool b_ok = b >= 0 && b < a.lay.batch;

  for (int i = threadIdx.x; i < Hq * Dqk / 8; i += kAttnThreads)
    reinterpret_cast<uint4*>(qs)[i] =
        __ldg(reinterpret_cast<const uint4*>(a.q + (long long)r * Hq * Dqk) + i);

  float m[HPW], l[HPW], o[HPW][DVL];
#pragma unroll
  for (int i = 0; i < HPW; ++i) {
    m[i] = -INFINITY;
    l[i] = 0.0f;
#pragma unroll
    for (int k = 0; k < DVL; ++k) o[i][k] = 0.0f;
  }

  const int per = (a.K + S - 1) / S;
  const int j0 = split * per, j1 = min(a.K, j0 + per);
  long long L = b_ok ? (long long)__ldg(&a.lay.seq_lens[b]) : 0;
  if (a.q_pos) {
    const long long qp = (long long)__ldg(&a.q_pos[r]) + 1;  // positions <= q_pos
    if (qp < L) L = qp;
  }
  for (int j = j0; j < j1; ++j) {
    if (threadIdx.x == 0) {
      long long row = -1;
      const int p = __ldg(&a.idx[(long long)r * a.K + j]);
      if (!b_ok) {
        if (j == j0) flag_status(a.status, DSA_STATUS_BAD_INDEX);
      } else if (p >= 0) {
        if (p >= L) {
          flag_status(a.status, DSA_STATUS_BAD_INDEX);
        } else {
          row = phys_row(a.lay.bt, a.lay.maxb, a.lay.bs, a.lay.nb, b, p);
          if (row < 0) flag_status(a.status, DSA_STATUS_BAD_BLOCK);
        }
      }
      row_sh = row;
    }
    __syncthreads();
    const long long row = row_sh;
    if (row < 0) {
      __syncthreads();
      continue;
    }
    const __nv_bfloat16* kr = a.kp + row * a.ks;
    const __nv_bfloat16* vr = a.vp + row * a.vs;
    for (int d = threadIdx.x; d < Dqk; d += kAttnThreads) krow[d] = __bfloat162float(kr[d]);
    for (int d = threadIdx.x; d < Dv; d += kAttnThreads) vrow[d] = __bfloat162float(vr[d]);
    __syncthreads();
#pragma unroll
    for (int i = 0; i < HPW; ++i) {
      const int h = warp + kAttnWarps * i;
      if (h < Hq) {
        float dot = 0.0f;
        for (int d = lane; d < Dqk; d += 32)
          dot = fmaf(__bfloat162float(qs[h * Dqk + d]), krow[d], dot);
        dot = warp_sum(dot);
        const float z = dot * a.scale_log2;
        const float mn = fmaxf(m[i], z);
        const float c = exp2f(m[i] - mn);
        const float pz = exp2f(z - mn);
        l[i] = l[i] * c + pz;
#pragma unroll
        for (int k = 0; k < DVL; ++k) {
          const int d = lane + 32 * k;
          const float v = d < Dv ? vrow[d] : 0.0f;
          o[i][k] = fmaf(o[i][k], c, pz * v);
        }
        m[i] = mn;
      }
    }
    __syncthreads();
  }

#pragma unroll
  for (int i = 0; i < HPW; ++i) {
    const int h = warp + kAttnWarps * i;
    if (h >= Hq) continue;
    if (S == 1) {
      const float inv = l[i] > 0.0f ? 1.0f / l[i] : 0.0f;
      __nv_bfloat16* dst = a.out + ((long long)r * Hq + h) * Dv;
#pragma unroll
      for (int k = 0; k < DVL; ++k) {
        const int d = lane + 32 * k;
        if (d < Dv) dst[d] = __float2bfloat16(o[i][k] * inv);
      }
      if (a.lse && lane == 0)
        a.lse[(long long)r * Hq + h] =
            l[i] > 0.0f ? (m[i] + log2f(l[i])) * 0.6931471805599453f : -INFINITY;
    } else {
      float* po = a.part_o + (((long long)r * S + split) * Hq + h) * Dv;
#pragma unroll
      for (int k = 0; k < DVL; ++k) {
        const int d = lane + 32 * k;
        if (d < Dv) po[d] = o[i][k];
      }
      if (lane == 0) {
        float* pml = a.part_ml + (((long long)r * S + split) * Hq + h) * 2;
        pml[0] = m[i];
        pml[1] = l[i];
      }
    }
  }
}

// grid (Hq, Nq): merge the S partials of one (query, head).
__global__ void __launch_bounds__(128) k_attn_combine(AttnParams a) {
  grid_dependency_wait();
  launch_dependents();
  const int h = blockIdx.x, r = blockIdx.y, S = a.S, Hq = a.Hq, Dv = a.Dv;
  __shared__ float wsh[64];
  __shared__ float lsum_sh, mmax_sh;
  if (threadIdx.x == 0) {
    float M = -INFINITY;
    for (int s = 0; s < S; ++s) {
      const float* pml = a.part_ml + (((long long)r * S + s) * Hq + h) * 2;
      if (pml[1] > 0.0f) M = fmaxf(M, pml[0]);
    }
    float lsum = 0.0f;
    for (int s = 0; s < S; ++s) {
      const float* pml = a.part_ml + (((long long)r * S + s) * Hq + h) * 2;
      const float wgt = pml[1] > 0.0f ? exp2f(pml[0] - M) : 0.0f;
      wsh[s] = wgt;
      lsum += pml[1] * wgt;
    }
    lsum_sh = lsum;
    mmax_sh = M;
  }
  __syncthreads();
  const float lsum = lsum_sh;
  const float inv = lsum > 0.0f ? 1.0f / lsum : 0.0f;
  for (int d = threadIdx.x; d < Dv; d += blockDim.x) {
    float acc = 0.0f;
    for (int s = 0; s < S; ++s)
      acc = fmaf(wsh[s], a.part_o[(((long long)r * S + s) * Hq + h) * Dv + d], acc);
    a.out[((long long)r * Hq + h) * Dv + d] = __float2bfloat16(acc * inv);
  }
  if (a.lse && threadIdx.x == 0)
    a.lse[(long long)r * Hq + h] =
        lsum > 0.0f ? (mmax_sh + log2f(lsum)) * 0.6931471805599453f : -INFINITY;
}

constexpr int kMaxSplits = 64;

int choose_splits(int Nq, int K) {
  int s = (2 * 152 + Nq - 1) / (Nq > 0 ? Nq : 1);
  int maxs = K / 64;
  if (maxs < 1) maxs = 1;
  if (s > maxs) s = maxs;
  if (s > kMaxSplits) s = kMaxSplits;
  if (s < 1) s = 1;
  return s;
}

template <int HPW, int DVL>
int launch_generic(const AttnParams& p, cudaStream_t s) {
  auto kern = k_attn_generic<HPW, DVL>;
  const size_t smem = (size_t)p.Hq * p.Dqk * 2 + sizeof(float) * (p.Dqk + p.Dv);
  const int arc = ensure_dynamic_smem((const void*)kern, 200 * 1024, "sparse_attn");
  if (arc) return arc;
  kern<<<dim3(p.S, p.Nq), kAttnThreads, smem, s>>>(p);
  count_launch();
  return check_launch("sparse_attn");
}

template <int HPW>
int launch_dv(const AttnParams& p, cudaStream_t s) {
  const int dvl = (p.Dv + 31) / 32;
  if (dvl <= 4) return launch_generic<HPW, 4>(p, s);
  if (dvl <= 8) return launch_generic<HPW, 8>(p, s);
  return launch_generic<HPW, 16>(p, s);
}

}  // namespace

bool attn_supported(int Hq, int Dqk, int Dv) {
  return Hq >= 1 && Hq <= 64 && Dqk >= 8 && Dv >= 8 && Dqk % 8 == 0 && Dv % 8 == 0 &&
         Dv <= 512 && (size_t)Hq * Dqk * 2 + 4 * (Dqk + Dv) <= 200 * 1024;
}

size_t attn_ws(int Nq, int Hq, int Dqk, int Dv, int K, bool) {
  const int S = choose_splits(Nq, K);
  size_t generic = kWsHeader;
  if (S > 1) generic += sizeof(float) * (size_t)Nq * S * Hq * ((size_t)Dv + 2);
  size_t tc = 0;
  if (Hq == 64 && Dqk == 576 && Dv == 512) tc = attn_tc_ws(Nq);
  return generic > tc ? generic : tc;
}

int launch_attn(AttnParams p, bool /*decode*/, void* ws, size_t ws_bytes, cudaStream_t s) {
  if (p.Nq == 0) return DSA_OK;
  if (attn_tc_eligible(p) && ws_bytes >= attn_tc_ws(p.Nq)) return launch_attn_tc(p, ws, s);
  p.S = choose_splits(p.Nq, p.K);
  if (p.S > 1) {
    p.part_o = reinterpret_cast<float*>((char*)ws + kWsHeader);
    p.part_ml = p.part_o + (size_t)p.Nq * p.S * p.Hq * p.Dv;
  }
  const int hpw = (p.Hq + kAttnWarps - 1) / kAttnWarps;
  int rc;
  if (hpw <= 1) rc = launch_dv<1>(p, s);
  else if (hpw <= 2) rc = launch_dv<2>(p, s);
  else if (hpw <= 4) rc = launch_dv<4>(p, s);
  else rc = launch_dv<8>(p, s);
  if (rc != DSA_OK || p.S == 1) return rc;
  k_attn_combine<<<dim3(p.Hq, p.Nq), 128, 0, s>>>(p);
  count_launch();
  return check_launch("sparse_attn combine");
}

}  // namespace dsa
