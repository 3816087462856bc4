// fp32 attention forward on CUDA cores (the exactness path).
//
// Same computation as the bf16 kernel, the online-softmax update of
// "Building a FlashAttention-2 forward kernel in pure NumPy" ("Step 3: Online
// softmax core", "Step 4: The tiled forward kernel"), kept in fp32 from end to
// end: scores, probabilities and the accumulator never leave fp32, and the
// exponentials are the accurate expf.
//
// Queries and keys may differ in length; the causal mask then allows key j
// for query i when j <= i + (Nk - Nq), and a query with no allowed key gets
// O = 0 and LSE = -inf (the same reading as the 16-bit kernel).
//
// A CTA owns 32 query rows of one plane (four warps, eight rows each) and
// streams 32-key K/V tiles through shared memory.  Lane l scores key l of the
// tile; row max and row sum are warp-shuffle reductions; lane l accumulates
// output columns l, l+32, l+64, l+96.
#pragma once

#include "ptx.cuh"

namespace attn {

struct F32Params {
  float* o;
  float* lse;
  const int* cu_seqlens;    // query offsets; nullptr for the dense layout
  const int* cu_seqlens_k;  // key offsets (packed layout only)
  int nseq;
  int planes;
  int rows;    // query rows per plane (dense) or total query tokens (packed)
  int rows_k;  // key rows per plane (dense) or total key tokens (packed)
  int n_qblk;  // dense: ceil(Nq/32); packed: upper bound on 32-row blocks
  int D;
  int causal;
  float scale;
  unsigned int* err;
};

constexpr int kF32BM = 32;
constexpr int kF32BN = 32;

__device__ __forceinline__ bool f32_decode(const F32Params& p, int& plane, int& row_base,
                                           int& seq_len, int& kv_base, int& kv_len, int& qblk) {
  const int t = blockIdx.x;
  plane = t % p.planes;
  const int vb = t / p.planes;
  if (p.cu_seqlens == nullptr) {
    qblk = p.n_qblk - 1 - vb;
    row_base = 0;
    seq_len = p.rows;
    kv_base = 0;
    kv_len = p.rows_k;
    return qblk >= 0;
  }
  int cum = 0;
  for (int s = 0; s < p.nseq; ++s) {
    const int a = __ldg(p.cu_seqlens + s), e = __ldg(p.cu_seqlens + s + 1);
    if (a < 0 || e < a || e > p.rows) {
      if (threadIdx.x == 0) atomicOr(p.err, kDevErrBounds);
      return false;
    }
    const int nb = (e - a + kF32BM - 1) / kF32BM;
    if (vb < cum + nb) {
      const int ak = __ldg(p.cu_seqlens_k + s), ek = __ldg(p.cu_seqlens_k + s + 1);
      if (ak < 0 || ek < ak || ek > p.rows_k) {
        if (threadIdx.x == 0) atomicOr(p.err, kDevErrBounds);
        return false;
      }
      row_base = a;
      seq_len = e - a;
      kv_base = ak;
      kv_len = ek - ak;
      qblk = nb - 1 - (vb - cum);
      return true;
    }
    cum += nb;
  }
  return false;
}

__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
  return x;
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

// NC = number of 32-column groups of the head dim (D <= 32*NC).
template <int NC>
__global__ void __launch_bounds__(128)
    attn_fwd_f32_kernel(const float* __restrict__ q, const float* __restrict__ k,
                        const float* __restrict__ v, const F32Params p) {
  constexpr int BM = kF32BM, BN = kF32BN, RPW = BM / 4;
  extern __shared__ float sm[];
  const int D = p.D;
  const int KS = D + 1;  // padded K row stride: lanes read distinct banks
  float* sQ = sm;                 // [BM][D]
  float* sK = sQ + BM * D;        // [BN][D+1]
  float* sV = sK + BN * KS;       // [BN][D]

  int plane, row_base, seq_len, kv_base, kv_len, qblk;
  if (!f32_decode(p, plane, row_base, seq_len, kv_base, kv_len, qblk)) return;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int q_row0 = qblk * BM;
  const int off = kv_len - seq_len;  // causal alignment of queries to keys
  const size_t plane_off = static_cast<size_t>(plane) * p.rows + row_base;
  const size_t kv_off = static_cast<size_t>(plane) * p.rows_k + kv_base;
  const float* qp = q + plane_off * D;
  const float* kp = k + kv_off * D;
  const float* vp = v + kv_off * D;

  for (int idx = threadIdx.x; idx < BM * D; idx += blockDim.x) {
    const int r = idx / D, d = idx % D;
    sQ[idx] = (q_row0 + r < seq_len) ? qp[static_cast<size_t>(q_row0 + r) * D + d] : 0.f;
  }

  float m[RPW], l[RPW], acc[RPW][NC];
#pragma unroll
  for (int r = 0; r < RPW; ++r) {
    m[r] = -INFINITY;
    l[r] = 0.f;
#pragma unroll
    for (int c = 0; c < NC; ++c) acc[r][c] = 0.f;
  }

  const int kend = p.causal ? max(0, min(kv_len, q_row0 + BM + off)) : kv_len;
  for (int kv0 = 0; kv0 < kend; kv0 += BN) {
    __syncthreads();
    for (int idx = threadIdx.x; idx < BN * D; idx += blockDim.x) {
      const int r = idx / D, d = idx % D;
      const bool in = kv0 + r < kv_len;
      sK[r * KS + d] = in ? kp[static_cast<size_t>(kv0 + r) * D + d] : 0.f;
      sV[r * D + d] = in ? vp[static_cast<size_t>(kv0 + r) * D + d] : 0.f;
    }
    __syncthreads();
    const int key = kv0 + lane;
#pragma unroll
    for (int r = 0; r < RPW; ++r) {
      const int lr = warp * RPW + r;
      const int row = q_row0 + lr;
      float s = 0.f;
      for (int d = 0; d < D; ++d) s = fmaf(sQ[lr * D + d], sK[lane * KS + d], s);
      const bool allowed = key < kv_len && (!p.causal || key <= row + off);
      s = allowed ? s * p.scale : -INFINITY;
      const float m_new = fmaxf(m[r], warp_max(s));
      const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
      const float alpha = expf(m[r] - m_use);
      const float pj = expf(s - m_use);
      l[r] = l[r] * alpha + warp_sum(pj);
#pragma unroll
      for (int c = 0; c < NC; ++c) acc[r][c] *= alpha;
      for (int jj = 0; jj < BN; ++jj) {
        const float pb = __shfl_sync(0xffffffffu, pj, jj);
#pragma unroll
        for (int c = 0; c < NC; ++c) {
          const int d = lane + 32 * c;
          if (d < D) acc[r][c] = fmaf(pb, sV[jj * D + d], acc[r][c]);
        }
      }
      m[r] = m_new;
    }
  }

#pragma unroll
  for (int r = 0; r < RPW; ++r) {
    const int row = q_row0 + warp * RPW + r;
    if (row >= seq_len) continue;
    const size_t g = plane_off + row;
    // l == 0 only for a row that saw no allowed key: O = 0, LSE = -inf
    const float inv = (l[r] > 0.f) ? 1.f / l[r] : 0.f;
#pragma unroll
    for (int c = 0; c < NC; ++c) {
      const int d = lane + 32 * c;
      if (d < D) p.o[g * D + d] = acc[r][c] * inv;
    }
    if (lane == 0) p.lse[g] = (l[r] > 0.f) ? m[r] + logf(l[r]) : -INFINITY;
  }
}

}  // namespace attn
