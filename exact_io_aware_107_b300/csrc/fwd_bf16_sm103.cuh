// bf16 attention forward for sm_103a: TMA + mbarrier pipeline, tcgen05 MMAs
// with TMEM accumulators, online softmax in base 2.
//
// What it computes is the exact scaled-dot-product attention forward
// O = softmax(scale * Q K^T + causal mask) V together with the per-row
// log-sum-exp, by the online-softmax update of "Building a FlashAttention-2
// forward kernel in pure NumPy" (sections "Architecture Overview" and
// "Step 3: Online softmax core"): a running max m, a running sum l with
// l * 2^m = sum of 2^(scores seen), an output accumulator rescaled by
// 2^(m_old - m_new) and a final division by l.  Query tiles are outer and
// key/value tiles stream past them, the order of "Hands-on build guide: tiled
// self-attention kernel with online softmax in pure NumPy" ("Architecture
// Overview").  Key tiles above the causal diagonal are never visited ("Python
// Attention Mechanisms Explained", section "Causal Masking and Incremental
// Decoding").
//
// CTA layout (320 threads, one CTA per SM):
//   warps 0-3  softmax for query tile 0 (thread t owns row t = TMEM lane t)
//   warps 4-7  softmax for query tile 1
//   warp  8    tcgen05 MMA issuer (lane 0) and TMEM owner
//   warp  9    TMA producer (lane 0)
// A CTA covers 256 query rows (two 128-row tiles) of one (batch, head) plane
// or one packed sequence of one head.
//
// TMEM (512 columns x 128 lanes, fp32 cells):
//   [  0,128) S0 = Q0 K^T   (P0 as packed bf16 overwrites its first 64 columns)
//   [128,256) S1 = Q1 K^T   (P1 likewise)
//   [256,256+D) O0, [256+D, 256+2D) O1
//
// Shared memory (1024-byte aligned; every tile is 128 rows x D bf16 stored as
// D/64 chunks of 128 rows x 128 bytes, 128-byte swizzled, as TMA writes them):
//   Q0, Q1, then NSTAGE ring slots holding K_0, V_0, K_1, V_1, ... in order.
//
// Rescaling is lazy: a row keeps its reference max until a tile raises the
// max by more than 8 (base-2 units), so P stays <= 2^8 and most tiles need no
// O rescale at all.  This is exact: l and O are scaled by the same reference,
// and the final O / l and LSE = m_ref + log2(l) do not depend on when the
// reference moved.
#pragma once

#include "ptx.cuh"

namespace attn {

struct Bf16Params {
  __nv_bfloat16* o;
  float* lse;
  const int* cu_seqlens;  // nullptr for the dense layout
  int nseq;               // packed layout: number of sequences
  int planes;             // dense: B*H; packed: H
  int rows;               // dense: N; packed: total tokens
  int n_qblk;             // dense: ceil(N/256); packed: upper bound on 256-row blocks
  int causal;
  float scale_log2;       // scale * log2(e)
  unsigned long long timeout_ns;
  unsigned int* err;
};

template <int D>
struct Bf16Cfg {
  static constexpr int BM = 128;                  // query rows per tile
  static constexpr int BN = 128;                  // keys per K/V tile
  static constexpr int NSTAGE = (D == 128) ? 4 : 8;
  static constexpr int CHUNK_BYTES = BM * 128;    // 128 rows x 128 bytes
  static constexpr int NCHUNK = D / 64;
  static constexpr int TILE_BYTES = BM * D * 2;
  static constexpr int Q_OFF = 0;
  static constexpr int KV_OFF = 2 * TILE_BYTES;
  static constexpr int BAR_OFF = KV_OFF + NSTAGE * TILE_BYTES;
  // q_full, kv_full[NSTAGE], kv_empty[NSTAGE], s_full[2], p_full[2], o_full[2], mma_done
  static constexpr int NBAR = 1 + 2 * NSTAGE + 2 + 2 + 2 + 1;
  static constexpr int MISC_OFF = BAR_OFF + NBAR * 8;
  static constexpr int SMEM_BYTES = MISC_OFF + 16;
  static constexpr int SMEM_ALLOC = SMEM_BYTES + 1024;
  static constexpr int THREADS = 320;
  static constexpr uint32_t TMEM_COLS = 512;
  static constexpr uint32_t S_COL0 = 0, S_COL1 = 128;
  static constexpr uint32_t O_COL0 = 256, O_COL1 = 256 + D;
  static_assert(D == 64 || D == 128, "head dim");
  static_assert(SMEM_ALLOC <= 232448, "shared memory");
};

// Work decode, uniform across the CTA.  Returns false when the CTA has no work.
__device__ __forceinline__ bool bf16_decode(const Bf16Params& p, int& plane, int& row_base,
                                            int& seq_len, int& qblk) {
  const int t = blockIdx.x;
  plane = t % p.planes;
  const int vb = t / p.planes;
  if (p.cu_seqlens == nullptr) {
    // heaviest causal blocks (largest query index) are launched first
    qblk = p.n_qblk - 1 - vb;
    row_base = 0;
    seq_len = p.rows;
    return qblk >= 0;
  }
  int cum = 0;
  for (int s = 0; s < p.nseq; ++s) {
    const int a = __ldg(p.cu_seqlens + s), e = __ldg(p.cu_seqlens + s + 1);
    if (a < 0 || e < a || e > p.rows) {
      if (threadIdx.x == 0) atomicOr(p.err, kDevErrBounds);
      return false;
    }
    const int nb = (e - a + 255) / 256;
    if (vb < cum + nb) {
      row_base = a;
      seq_len = e - a;
      qblk = nb - 1 - (vb - cum);
      return true;
    }
    cum += nb;
  }
  return false;
}

template <int D>
__device__ __forceinline__ void bf16_issue_s(uint32_t d_tmem, uint32_t q_smem, uint32_t k_smem) {
  using C = Bf16Cfg<D>;
  constexpr uint32_t idesc = idesc_bf16_f32(128, C::BN, 0, 0);
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk) {
    const uint32_t off = (kk / 4) * C::CHUNK_BYTES + (kk % 4) * 32;
    const uint64_t a = sdesc_sw128(q_smem + off, 16, 1024);
    const uint64_t b = sdesc_sw128(k_smem + off, 16, 1024);
    umma_ss(d_tmem, a, b, idesc, kk > 0 ? 1u : 0u);
  }
}

template <int D>
__device__ __forceinline__ void bf16_issue_pv(uint32_t d_tmem, uint32_t p_tmem, uint32_t v_smem,
                                              uint32_t accumulate) {
  using C = Bf16Cfg<D>;
  constexpr uint32_t idesc = idesc_bf16_f32(128, D, 0, 1);
#pragma unroll
  for (int kk = 0; kk < C::BN / 16; ++kk) {
    // V is the MN-major B operand: 16 keys = two 8-row groups of 128-byte rows
    const uint64_t b = sdesc_sw128(v_smem + kk * 16 * 128, C::CHUNK_BYTES, 1024);
    umma_ts(d_tmem, p_tmem + kk * 8, b, idesc, (accumulate || kk > 0) ? 1u : 0u);
  }
}

template <int D>
__global__ void __launch_bounds__(320, 1)
    attn_fwd_bf16_kernel(const __grid_constant__ CUtensorMap tmQ,
                         const __grid_constant__ CUtensorMap tmK,
                         const __grid_constant__ CUtensorMap tmV, const Bf16Params p) {
  using C = Bf16Cfg<D>;
  constexpr int NS = C::NSTAGE;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::BAR_OFF);
  uint64_t* q_full = bars;
  uint64_t* kv_full = bars + 1;
  uint64_t* kv_empty = kv_full + NS;
  uint64_t* s_full = kv_empty + NS;
  uint64_t* p_full = s_full + 2;
  uint64_t* o_full = p_full + 2;
  uint64_t* mma_done = o_full + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::MISC_OFF);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::MISC_OFF + 4);

  int plane, row_base, seq_len, qblk;
  if (!bf16_decode(p, plane, row_base, seq_len, qblk)) return;

  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int s = 0; s < NS; ++s) {
      mbar_init(&kv_full[s], 1);
      mbar_init(&kv_empty[s], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s_full[i], 1);
      mbar_init(&p_full[i], 128);
      mbar_init(&o_full[i], 1);
    }
    mbar_init(mma_done, 1);
    *abort_flag = 0;
    mbar_fence_init();
  }
  if (warp == 8) {
    tmem_alloc(tmem_slot, C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const WaitCtl ctl{abort_flag, p.err, p.timeout_ns};

  const int q_row0 = qblk * 256;  // first query row of the CTA, relative to the sequence
  const bool has_q1 = q_row0 + 128 < seq_len;
  const int nkv = (seq_len + C::BN - 1) / C::BN;
  const int n0 = p.causal ? min(nkv, 2 * qblk + 1) : nkv;
  const int n1 = has_q1 ? (p.causal ? min(nkv, 2 * qblk + 2) : nkv) : 0;
  const int nmax = max(n0, n1);
  const uint32_t smem_base = smem_u32(smem);

  if (warp < 8) {
    // ------------------------------------------------------------ softmax
    const int ti = warp / 4;              // query tile
    const int t = threadIdx.x - 128 * ti;  // row within the tile
    const uint32_t lane_off = static_cast<uint32_t>(32 * (warp % 4)) << 16;
    const uint32_t tS = tmem + lane_off + (ti ? C::S_COL1 : C::S_COL0);
    const uint32_t tO = tmem + lane_off + (ti ? C::O_COL1 : C::O_COL0);
    const int n_i = ti ? n1 : n0;
    const int row = q_row0 + 128 * ti + t;
    const float cl2 = p.scale_log2;
    float m_ref = -INFINITY;
    float l = 0.f;
    bool ok = true;
    for (int j = 0; j < n_i; ++j) {
      if (!mbar_wait(&s_full[ti], j & 1, ctl)) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t sr[128];
      tmem_ld64_wait(tS, *reinterpret_cast<uint32_t(*)[64]>(&sr[0]));
      tmem_ld64_wait(tS + 64, *reinterpret_cast<uint32_t(*)[64]>(&sr[64]));
      float* s = reinterpret_cast<float*>(sr);
      const int kv0 = j * C::BN;
      const bool need_mask = (kv0 + C::BN > seq_len) || (p.causal && kv0 + C::BN - 1 > q_row0 + 128 * ti);
      if (need_mask) {
        const int lim = p.causal ? min(seq_len - 1, row) : (seq_len - 1);
#pragma unroll
        for (int c = 0; c < 128; ++c)
          if (kv0 + c > lim) s[c] = -INFINITY;
      }
      float mx[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) mx[e] = s[e];
#pragma unroll
      for (int c = 8; c < 128; c += 8)
#pragma unroll
        for (int e = 0; e < 8; ++e) mx[e] = fmaxf(mx[e], s[c + e]);
      const float mt =
          fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])),
                fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7]))) * cl2;
      float m_new = m_ref;
      float alpha = 1.f;
      bool resc = false;
      if (mt > m_ref + 8.f) {
        m_new = mt;
        alpha = ex2_approx(m_ref - m_new);
        resc = (j > 0);
      }
      const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
      float sum[4] = {0.f, 0.f, 0.f, 0.f};
      uint32_t pk[64];
#pragma unroll
      for (int c = 0; c < 64; ++c) {
        const float a = ex2_approx(fmaf(s[2 * c], cl2, -m_use));
        const float b = ex2_approx(fmaf(s[2 * c + 1], cl2, -m_use));
        sum[(2 * c) & 3] += a;
        sum[(2 * c + 1) & 3] += b;
        pk[c] = pack_bf16x2(a, b);
      }
      l = l * alpha + ((sum[0] + sum[1]) + (sum[2] + sum[3]));
      tmem_st32(tS, *reinterpret_cast<uint32_t(*)[32]>(&pk[0]));
      tmem_st32(tS + 32, *reinterpret_cast<uint32_t(*)[32]>(&pk[32]));
      if (__any_sync(0xffffffffu, resc)) {
        const float f = resc ? alpha : 1.f;
#pragma unroll
        for (int cc = 0; cc < D / 32; ++cc) {
          uint32_t o[32];
          tmem_ld32_wait(tO + 32 * cc, o);
#pragma unroll
          for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * f);
          tmem_st32(tO + 32 * cc, o);
        }
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&p_full[ti]);
      m_ref = m_new;
    }
    if (ok && n_i > 0 && mbar_wait(&o_full[ti], 0, ctl)) {
      tc_fence_after();
      const bool valid = row < seq_len;
      const size_t grow = static_cast<size_t>(plane) * p.rows + row_base + row;
      const float inv_l = 1.f / l;
      uint4* dst = reinterpret_cast<uint4*>(p.o + grow * D);
#pragma unroll
      for (int cc = 0; cc < D / 32; ++cc) {
        uint32_t o[32];
        tmem_ld32_wait(tO + 32 * cc, o);
        uint32_t h[16];
#pragma unroll
        for (int e = 0; e < 16; ++e)
          h[e] = pack_bf16x2(__uint_as_float(o[2 * e]) * inv_l, __uint_as_float(o[2 * e + 1]) * inv_l);
        if (valid) {
#pragma unroll
          for (int v = 0; v < 4; ++v)
            dst[cc * 4 + v] = make_uint4(h[4 * v], h[4 * v + 1], h[4 * v + 2], h[4 * v + 3]);
        }
      }
      if (valid) p.lse[grow] = (m_ref + log2f(l)) * 0.69314718055994530942f;
    }
  } else if (warp == 8) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t q0 = smem_base + C::Q_OFF;
      const uint32_t q1 = q0 + C::TILE_BYTES;
      const uint32_t kvb = smem_base + C::KV_OFF;
      bool ok = mbar_wait(q_full, 0, ctl);
      if (ok) ok = mbar_wait(&kv_full[0], 0, ctl);
      if (ok) {
        tc_fence_after();
        if (n0 > 0) {
          bf16_issue_s<D>(tmem + C::S_COL0, q0, kvb);
          umma_commit(&s_full[0]);
        }
        if (n1 > 0) {
          bf16_issue_s<D>(tmem + C::S_COL1, q1, kvb);
          umma_commit(&s_full[1]);
        }
        umma_commit(&kv_empty[0]);
      }
      for (int j = 0; ok && j < nmax; ++j) {
        const int tv = 2 * j + 1, tk = 2 * j + 2;
        const int sv = tv % NS, sk = tk % NS;
        const bool next = j + 1 < nmax;
        if (!mbar_wait(&kv_full[sv], (tv / NS) & 1, ctl)) break;
        if (next && !mbar_wait(&kv_full[sk], (tk / NS) & 1, ctl)) break;
        tc_fence_after();
        for (int ti = 0; ti < 2; ++ti) {
          const int n_i = ti ? n1 : n0;
          if (j >= n_i) continue;
          if (!mbar_wait(&p_full[ti], j & 1, ctl)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sc = ti ? C::S_COL1 : C::S_COL0;
          const uint32_t oc = ti ? C::O_COL1 : C::O_COL0;
          bf16_issue_pv<D>(tmem + oc, tmem + sc, kvb + sv * C::TILE_BYTES, j > 0 ? 1u : 0u);
          if (j + 1 < n_i) {
            bf16_issue_s<D>(tmem + sc, ti ? q1 : q0, kvb + sk * C::TILE_BYTES);
            umma_commit(&s_full[ti]);
          } else {
            umma_commit(&o_full[ti]);
          }
        }
        if (!ok) break;
        umma_commit(&kv_empty[sv]);
        if (next) umma_commit(&kv_empty[sk]);
      }
      // every MMA issued so far must finish before TMEM and shared memory are released
      umma_commit(mma_done);
      mbar_wait_drain(mma_done, 0, ctl);
    }
  } else {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      const int pc = plane;
      const int qr = row_base + q_row0;
      mbar_arrive_expect_tx(q_full, (has_q1 ? 2 : 1) * C::TILE_BYTES);
#pragma unroll
      for (int c = 0; c < C::NCHUNK; ++c)
        tma_load_3d(smem + C::Q_OFF + c * C::CHUNK_BYTES, &tmQ, q_full, c * 64, qr, pc);
      if (has_q1) {
#pragma unroll
        for (int c = 0; c < C::NCHUNK; ++c)
          tma_load_3d(smem + C::Q_OFF + C::TILE_BYTES + c * C::CHUNK_BYTES, &tmQ, q_full, c * 64,
                      qr + 128, pc);
      }
      int issued = 0;
      for (int t = 0; t < 2 * nmax; ++t) {
        const int s = t % NS, u = t / NS;
        if (u > 0 && !mbar_wait(&kv_empty[s], (u - 1) & 1, ctl)) break;
        const int j = t >> 1;
        const CUtensorMap* m = (t & 1) ? &tmV : &tmK;
        mbar_arrive_expect_tx(&kv_full[s], C::TILE_BYTES);
#pragma unroll
        for (int c = 0; c < C::NCHUNK; ++c)
          tma_load_3d(smem + C::KV_OFF + s * C::TILE_BYTES + c * C::CHUNK_BYTES, m, &kv_full[s],
                      c * 64, row_base + j * C::BN, pc);
        issued = t + 1;
      }
      // drain: every copy issued must land before the CTA may exit
      mbar_wait_drain(q_full, 0, ctl);
      for (int t = max(0, issued - NS); t < issued; ++t)
        mbar_wait_drain(&kv_full[t % NS], (t / NS) & 1, ctl);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 8) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

}  // namespace attn
