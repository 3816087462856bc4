// bf16 KV-cache decode for sm_103a: a few new query rows attend to every key
// of a long cache, without a mask (the incremental-decoding form of "Python
// Attention Mechanisms Explained: From Self-Attention to Flash Attention",
// section "Causal Masking and Incremental Decoding": the new token's query
// against the cached keys and values, is_causal=False).
//
// The work is bound by reading K and V once from HBM, so the keys of each
// (batch, head) plane are split across CTAs and every CTA streams its slice
// through shared memory with TMA, the online-softmax update of "Building a
// FlashAttention-2 forward kernel in pure NumPy" ("Step 3: Online softmax
// core") turning each slice into a partial (O_c, LSE_c).  The partials are
// then merged exactly: LSE = ln sum_c exp(LSE_c), O = sum_c exp(LSE_c - LSE) O_c
// (the same invariant, l * exp(m) = sum of exp(scores seen), applied to whole
// slices).  With one slice per plane the CTA writes the final O and LSE.
//
// CTA: 8 compute warps in two groups that take alternate 128-key tiles, plus
// one TMA producer warp.  Keys arrive in the forward kernel's swizzled tile
// layout; warp w of a group works on keys 32w..32w+31 of its tile, keeps its
// own running max / sums / output for the query rows, and the eight warps are
// merged at the end.  The 1..8 query rows are the M dimension of warp-level
// MMAs (decode_rows_mma), so each key is read once per warp with ldmatrix and
// scored against every row at once; on CUDA cores (lane = key) the work per
// key grew with the rows and already bounded a single row below the HBM
// rate.  P is rounded to bf16 for P.V, and O is divided by the sum of the
// rounded weights (LSE keeps the fp32 sum).
#pragma once

#include "ptx.cuh"

namespace attn {

struct DecodeParams {
  void* o;          // bf16 (planes, nq, D)
  float* lse;       // (planes, nq)
  float* ws_o;      // (planes, nsplit, nq, D) fp32 partial outputs (nsplit > 1)
  float* ws_lse;    // (planes, nsplit, nq) partial LSE (nsplit > 1)
  const void* q;    // bf16 (planes, nq, D)
  int planes;
  int nq;           // query rows per plane, 1..kDecodeMaxQ
  int nk;           // cached keys per plane
  int nsplit;       // key slices per plane
  int chunk;        // keys per slice (a multiple of 128)
  float scale_log2;
  int stall;        // abort-path test: CTA 0 waits on a phase nothing completes
  unsigned long long timeout_ns;
  unsigned int* err;
};

constexpr int kDecodeMaxQ = 8;

template <int D>
struct DecCfg {
  static constexpr int TK = 128;                 // keys per tile
  static constexpr int NSTAGE = (D == 128) ? 3 : 3;
  static constexpr int CHUNK_BYTES = TK * 128;
  static constexpr int NCHUNK = D / 64;
  static constexpr int TILE_BYTES = TK * D * 2;
  static constexpr int K_OFF = 0;
  static constexpr int V_OFF = NSTAGE * TILE_BYTES;
  static constexpr int BAR_OFF = 2 * NSTAGE * TILE_BYTES;
  static constexpr int NBAR = 2 * NSTAGE;
  static constexpr int MISC_OFF = BAR_OFF + NBAR * 8;
  static constexpr int SMEM_ALLOC = MISC_OFF + 16 + 1024;
  // after the key loop the merge arrays reuse the (drained) K/V stages:
  // m, l, l_o: float [8][MAXQ]; o: float [8][MAXQ][D]
  static constexpr int M_OFF = 0;
  static constexpr int O_OFF = 3 * 8 * kDecodeMaxQ * 4;
  static constexpr int WARPS = 8;                                 // compute warps
  static constexpr int THREADS = 32 * WARPS + 32;
  static_assert(O_OFF + WARPS * kDecodeMaxQ * D * 4 <= BAR_OFF, "merge area fits the stages");
  static_assert(SMEM_ALLOC <= 232448, "shared memory");
};

__device__ __forceinline__ float bf16lo(uint32_t x) { return __uint_as_float(x << 16); }
__device__ __forceinline__ float bf16hi(uint32_t x) { return __uint_as_float(x & 0xffff0000u); }

// ---- warp-level tensor-core helpers
// Four 8x8 16-bit matrices from shared memory; lane L gives the address of row
// L % 8 of matrix L / 8 and receives (row L / 4, columns 2(L % 4), 2(L % 4)+1)
// of each matrix (with .trans: rows 2(L % 4), 2(L % 4)+1 of column L / 4).
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
// C (16x8, fp32) += A (16x16, bf16, rows) * B (16x8, bf16, columns).  The
// kernel feeds at most 8 rows, so A's registers for rows 8-15 are zero and
// C's c[2], c[3] stay zero.
__device__ __forceinline__ void mma_bf16_16816(float (&c)[4], uint32_t a0, uint32_t a2,
                                               uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(0u), "r"(a2), "r"(0u), "r"(b0), "r"(b1));
}
// Shared-memory address of the 16-byte unit u (dims 8u..8u+7) of row `key` of
// a tile stored as TMA writes it (chunks of 64 dims, 128-byte swizzle).
template <int CHUNK_BYTES>
__device__ __forceinline__ uint32_t tile_unit(uint32_t base, int key, int u) {
  return base + static_cast<uint32_t>((u >> 3) * CHUNK_BYTES + key * 128 +
                                      (((u & 7) ^ (key & 7)) << 4));
}

// ---- 1..8 query rows: one warp-level MMA tile per 8 keys.  The rows are the
// M dimension of mma.m16n8k16 (rows nq..15 are zero), so Q sits in A
// fragments for the whole slice, K and V are read once per warp with
// ldmatrix, and P stays in registers between S = Q K^T and O += P V (the
// accumulator of two 8-key tiles is the A fragment of the next MMA).  Lane L
// works on query row L / 4 (g) and, in each 8-key tile, keys 2(L % 4) and
// 2(L % 4)+1 (c).
template <int D>
struct DecMmaRows {
  float m = -INFINITY;  // running max of row g (base 2)
  float l = 0.f;        // sum of the probabilities (fp32; for LSE)
  float lo = 0.f;       // sum of the probabilities as rounded for P.V (for O)
  float o[D / 8][4];    // O fragments: [dims 8n..8n+7][row g: c, c+1 | row g+8: 0, 0]
};

template <int D>
__device__ __forceinline__ void decode_rows_mma(DecMmaRows<D>& st, const DecodeParams& p,
                                                uint32_t sbase, uint64_t* full, uint64_t* empty,
                                                const WaitCtl& ctl, int plane, int k_begin,
                                                int k_end, int ntiles, int grp, int wq, int lane,
                                                bool& ok) {
  using C = DecCfg<D>;
  constexpr int NS = C::NSTAGE;
  const int g = lane >> 2, c = lane & 3;
  // Q rows 0..7 as A fragments: [k block of 16 dims][dims 2c, 2c+1 | 2c+8, 2c+9]
  uint32_t qa[D / 16][2];
  const uint32_t* qg = reinterpret_cast<const uint32_t*>(
      static_cast<const uint16_t*>(p.q) +
      (static_cast<size_t>(plane) * p.nq + (g < p.nq ? g : 0)) * D);
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk) {
    qa[kk][0] = (g < p.nq) ? qg[8 * kk + c] : 0u;
    qa[kk][1] = (g < p.nq) ? qg[8 * kk + 4 + c] : 0u;
  }
#pragma unroll
  for (int n = 0; n < D / 8; ++n)
#pragma unroll
    for (int e = 0; e < 4; ++e) st.o[n][e] = 0.f;
  for (int t = grp; t < ntiles; t += 2) {
    const int s = t % NS;
    // The two groups read the ring in interleaved order, so the previous use
    // of this stage (tile t - NS) belongs to the other group and may not have
    // landed yet; a parity wait on full[s] would then match the phase of
    // tile t - 2*NS.  Waiting first until tile t - NS has been read (its
    // empty phase) puts full[s] in tile t's phase, one phase apart at most.
    if (t >= NS && !__all_sync(0xffffffffu, mbar_wait(&empty[s], ((t / NS) - 1) & 1, ctl))) {
      ok = false;
      break;
    }
    if (!__all_sync(0xffffffffu, mbar_wait(&full[s], (t / NS) & 1, ctl))) {
      ok = false;
      break;
    }
    const uint32_t kt = sbase + C::K_OFF + s * C::TILE_BYTES;
    const uint32_t vt = sbase + C::V_OFF + s * C::TILE_BYTES;
    const int kw = 32 * wq;  // this warp's first key within the tile
    // S = Q K^T for the warp's 32 keys: four 8-key tiles
    float sa[4][4];
#pragma unroll
    for (int nt = 0; nt < 4; ++nt) {
#pragma unroll
      for (int e = 0; e < 4; ++e) sa[nt][e] = 0.f;
#pragma unroll
      for (int kp = 0; kp < D / 32; ++kp) {
        // dims 32kp + 8(L/8) .. +7 of key kw + 8nt + L%8: B fragments of two k blocks
        uint32_t b[4];
        ldsm_x4(tile_unit<C::CHUNK_BYTES>(kt, kw + 8 * nt + (lane & 7), 4 * kp + (lane >> 3)), b);
        mma_bf16_16816(sa[nt], qa[2 * kp][0], qa[2 * kp][1], b[0], b[1]);
        mma_bf16_16816(sa[nt], qa[2 * kp + 1][0], qa[2 * kp + 1][1], b[2], b[3]);
      }
    }
    // online softmax of row g over the 32 keys (4 lanes share a row)
    const int key0 = k_begin + t * C::TK + kw + 2 * c;
    float x[8];
#pragma unroll
    for (int nt = 0; nt < 4; ++nt)
#pragma unroll
      for (int h = 0; h < 2; ++h)
        x[2 * nt + h] = (key0 + 8 * nt + h < k_end) ? sa[nt][h] * p.scale_log2 : -INFINITY;
    float mx = fmaxf(fmaxf(fmaxf(x[0], x[1]), fmaxf(x[2], x[3])),
                     fmaxf(fmaxf(x[4], x[5]), fmaxf(x[6], x[7])));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
    const float m_new = fmaxf(st.m, mx);
    const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
    const float alpha = ex2_approx(st.m - m_use);
    uint32_t pa[4];
    float sum = 0.f, sum_r = 0.f;
#pragma unroll
    for (int nt = 0; nt < 4; ++nt) {
      const float p0 = ex2_approx(x[2 * nt] - m_use);
      const float p1 = ex2_approx(x[2 * nt + 1] - m_use);
      pa[nt] = pack_bf16x2(p0, p1);
      sum += p0 + p1;
      sum_r += bf16lo(pa[nt]) + bf16hi(pa[nt]);
    }
    sum += __shfl_xor_sync(0xffffffffu, sum, 1);
    sum += __shfl_xor_sync(0xffffffffu, sum, 2);
    sum_r += __shfl_xor_sync(0xffffffffu, sum_r, 1);
    sum_r += __shfl_xor_sync(0xffffffffu, sum_r, 2);
    st.l = st.l * alpha + sum;
    st.lo = st.lo * alpha + sum_r;
    st.m = m_new;
#pragma unroll
    for (int n = 0; n < D / 8; ++n) {
      st.o[n][0] *= alpha;
      st.o[n][1] *= alpha;
    }
    // O += P V: two k steps of 16 keys; V's rows are keys, so B comes transposed
#pragma unroll
    for (int ks = 0; ks < 2; ++ks) {
#pragma unroll
      for (int np = 0; np < D / 16; ++np) {
        // matrix L/8: keys +8((L/8)&1), dims 16np + 8((L/8)>>1)
        const int i = lane >> 3;
        uint32_t b[4];
        ldsm_x4_trans(tile_unit<C::CHUNK_BYTES>(vt, kw + 16 * ks + 8 * (i & 1) + (lane & 7),
                                                2 * np + (i >> 1)),
                      b);
        mma_bf16_16816(st.o[2 * np], pa[2 * ks], pa[2 * ks + 1], b[0], b[1]);
        mma_bf16_16816(st.o[2 * np + 1], pa[2 * ks], pa[2 * ks + 1], b[2], b[3]);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);
  }
}

// The warp's partial (m, l, l_o, O) of its rows into the merge arrays.
template <int D>
__device__ __forceinline__ void decode_rows_mma_store(const DecMmaRows<D>& st, float* ms,
                                                      float* ls, float* los, float* os, int warp,
                                                      int lane, int nq) {
  const int g = lane >> 2, c = lane & 3;
  if (g >= nq) return;
  const int row = warp * kDecodeMaxQ + g;
  if (c == 0) {
    ms[row] = st.m;
    ls[row] = st.l;
    los[row] = st.lo;
  }
#pragma unroll
  for (int n = 0; n < D / 8; ++n)
    *reinterpret_cast<float2*>(os + row * D + 8 * n + 2 * c) = make_float2(st.o[n][0], st.o[n][1]);
}

// The decode kernel: key slices of a plane per CTA, 1..8 query rows.
template <int D>
__global__ void __launch_bounds__(288)
    attn_decode_bf16_kernel(const __grid_constant__ CUtensorMap tmK,
                            const __grid_constant__ CUtensorMap tmV, const DecodeParams p) {
  using C = DecCfg<D>;
  constexpr int NS = C::NSTAGE;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::BAR_OFF);
  uint64_t* empty = full + NS;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::MISC_OFF);
  float* ms = reinterpret_cast<float*>(smem + C::M_OFF);
  float* ls = ms + C::WARPS * kDecodeMaxQ;   // sums of the probabilities (for LSE)
  float* los = ls + C::WARPS * kDecodeMaxQ;  // sums of the weights P.V used (for O)
  float* os = reinterpret_cast<float*>(smem + C::O_OFF);

  const int plane = blockIdx.x / p.nsplit;
  const int split = blockIdx.x - plane * p.nsplit;
  const int k_begin = split * p.chunk;
  const int k_end = min(p.nk, k_begin + p.chunk);
  const int ntiles = (k_end - k_begin + C::TK - 1) / C::TK;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int nq = p.nq;

  if (threadIdx.x == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 4);  // the four warps of the group that read the tile
    }
    *abort_flag = 0;
    mbar_fence_init();
  }
  __syncthreads();
  const WaitCtl ctl{abort_flag, p.err, p.timeout_ns};
  const uint32_t sbase = smem_u32(smem);

  if (warp == C::WARPS) {
    // ------------------------------------------------------------ TMA producer
    int t = 0;
    // abort-path test: empty[0] completes only once tile 0 (not loaded yet)
    // has been read, so this wait runs out of budget and the CTA aborts
    const bool stalled = p.stall && blockIdx.x == 0 &&
                         !__all_sync(0xffffffffu, mbar_wait(&empty[0], 0, ctl));
    for (; !stalled && t < ntiles; ++t) {
      const int s = t % NS, u = t / NS;
      if (u > 0 && !__all_sync(0xffffffffu, mbar_wait(&empty[s], (u - 1) & 1, ctl))) break;
      mbar_arrive_expect_tx_warp(&full[s], 2 * C::TILE_BYTES);
      const int row = k_begin + t * C::TK;
#pragma unroll
      for (int c = 0; c < C::NCHUNK; ++c) {
        tma_load_3d_warp(sbase + C::K_OFF + s * C::TILE_BYTES + c * C::CHUNK_BYTES, &tmK,
                         smem_u32(&full[s]), c * 64, row, plane);
        tma_load_3d_warp(sbase + C::V_OFF + s * C::TILE_BYTES + c * C::CHUNK_BYTES, &tmV,
                         smem_u32(&full[s]), c * 64, row, plane);
      }
    }
    for (int d = max(0, t - NS); d < t; ++d) mbar_wait_drain(&full[d % NS], (d / NS) & 1, ctl);
  } else {
    // ------------------------------------------------------------ compute warps
    const int grp = warp / 4;  // tiles t with t % 2 == grp
    const int wq = warp % 4;   // key quarter within a tile
    bool ok = true;
    DecMmaRows<D> st;
    decode_rows_mma<D>(st, p, sbase, full, empty, ctl, plane, k_begin, k_end, ntiles, grp, wq,
                       lane, ok);
    // merge the eight warps through shared memory (the drained K/V stages):
    // every compute warp must be past its last tile before the area is reused
    asm volatile("bar.sync 1, %0;" ::"n"(32 * C::WARPS) : "memory");
    // after an abort, copies may still be landing in the stages: skip the merge
    ok = !*abort_flag;
    if (ok) decode_rows_mma_store<D>(st, ms, ls, los, os, warp, lane, nq);
    asm volatile("bar.sync 1, %0;" ::"n"(32 * C::WARPS) : "memory");
    if (ok && !*abort_flag) {
      for (int i = threadIdx.x; i < nq * D; i += 32 * C::WARPS) {
        const int qi = i / D, d = i - qi * D;
        float mt = -INFINITY;
#pragma unroll
        for (int w = 0; w < C::WARPS; ++w) mt = fmaxf(mt, ms[w * kDecodeMaxQ + qi]);
        const float mu = (mt == -INFINITY) ? 0.f : mt;
        float lt = 0.f, lot = 0.f, ot = 0.f;
#pragma unroll
        for (int w = 0; w < C::WARPS; ++w) {
          const float f = ex2_approx(ms[w * kDecodeMaxQ + qi] - mu);
          lt += f * ls[w * kDecodeMaxQ + qi];
          lot += f * los[w * kDecodeMaxQ + qi];
          ot += f * os[(w * kDecodeMaxQ + qi) * D + d];
        }
        const float out = (lot > 0.f) ? ot / lot : 0.f;
        const float lse = (mu + log2f(lt)) * 0.69314718055994530942f;
        if (p.nsplit == 1) {
          const size_t g = static_cast<size_t>(plane) * nq + qi;
          static_cast<uint16_t*>(p.o)[g * D + d] =
              static_cast<uint16_t>(pack_bf16x2(out, 0.f) & 0xffffu);
          if (d == 0) p.lse[g] = lse;
        } else {
          const size_t g = (static_cast<size_t>(plane) * p.nsplit + split) * nq + qi;
          p.ws_o[g * D + d] = out;
          if (d == 0) p.ws_lse[g] = lse;
        }
      }
    }
  }
}

// Merges the per-slice partials of every (plane, query row): one CTA of D
// threads per row.
template <int D>
__global__ void __launch_bounds__(128) attn_decode_merge_kernel(const DecodeParams p) {
  const int row = blockIdx.x;  // plane * nq + qi
  const int plane = row / p.nq, qi = row - plane * p.nq;
  const int d = threadIdx.x;
  float mx = -INFINITY;
  for (int c = 0; c < p.nsplit; ++c)
    mx = fmaxf(mx, p.ws_lse[(static_cast<size_t>(plane) * p.nsplit + c) * p.nq + qi]);
  const float mu = (mx == -INFINITY) ? 0.f : mx;
  float den = 0.f, acc = 0.f;
  for (int c = 0; c < p.nsplit; ++c) {
    const size_t g = (static_cast<size_t>(plane) * p.nsplit + c) * p.nq + qi;
    const float f = expf(p.ws_lse[g] - mu);
    den += f;
    if (d < D) acc += f * p.ws_o[g * D + d];
  }
  if (d < D)
    static_cast<uint16_t*>(p.o)[static_cast<size_t>(row) * D + d] =
        static_cast<uint16_t>(pack_bf16x2(acc / den, 0.f) & 0xffffu);
  if (d == 0) p.lse[row] = mu + logf(den);
}

}  // namespace attn
