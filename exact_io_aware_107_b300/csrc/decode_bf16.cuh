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
// layout; warp w of a group scores keys 32w..32w+31 of its tile (lane = key,
// so the row reads of the 32 lanes hit distinct banks thanks to the swizzle),
// keeps its own running max / sum / output for the query rows, and the eight
// warps are merged at the end.  For P.V, lane l accumulates output columns
// [D/32 * l, D/32 * (l+1)).
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
  static constexpr int Q_OFF = 2 * NSTAGE * TILE_BYTES;          // float [MAXQ][D]
  static constexpr int BAR_OFF = Q_OFF + kDecodeMaxQ * D * 4;
  static constexpr int NBAR = 2 * NSTAGE;
  static constexpr int MISC_OFF = BAR_OFF + NBAR * 8;
  static constexpr int SMEM_ALLOC = MISC_OFF + 16 + 1024;
  // after the key loop the merge arrays reuse the (drained) K/V stages:
  // m, l: float [8][MAXQ]; o: float [8][MAXQ][D]
  static constexpr int M_OFF = 0;
  static constexpr int O_OFF = 2 * 8 * kDecodeMaxQ * 4;
  static constexpr int WARPS = 8;                                 // compute warps
  static constexpr int THREADS = 32 * WARPS + 32;
  static constexpr int CPL = D / 32;                             // output columns per lane
  static_assert(O_OFF + WARPS * kDecodeMaxQ * D * 4 <= Q_OFF, "merge area fits the stages");
  static_assert(SMEM_ALLOC <= 232448, "shared memory");
};

__device__ __forceinline__ float bf16lo(uint32_t x) { return __uint_as_float(x << 16); }
__device__ __forceinline__ float bf16hi(uint32_t x) { return __uint_as_float(x & 0xffff0000u); }

// NQ: query-row bucket (1, 2, 4 or 8); rows nq..NQ-1 of the bucket are idle.
template <int D, int NQ>
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
  float* qs = reinterpret_cast<float*>(smem + C::Q_OFF);
  float* ms = reinterpret_cast<float*>(smem + C::M_OFF);
  float* ls = ms + C::WARPS * kDecodeMaxQ;
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
  const uint16_t* qg = static_cast<const uint16_t*>(p.q) + static_cast<size_t>(plane) * nq * D;
  for (int i = threadIdx.x; i < nq * D; i += blockDim.x)
    qs[i] = __uint_as_float(static_cast<uint32_t>(qg[i]) << 16);
  __syncthreads();
  const WaitCtl ctl{abort_flag, p.err, p.timeout_ns};
  const uint32_t sbase = smem_u32(smem);

  if (warp == C::WARPS) {
    // ------------------------------------------------------------ TMA producer
    int t = 0;
    for (; t < ntiles; ++t) {
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
    float m[NQ], l[NQ], o[NQ][C::CPL];
#pragma unroll
    for (int qi = 0; qi < NQ; ++qi) {
      m[qi] = -INFINITY;
      l[qi] = 0.f;
#pragma unroll
      for (int e = 0; e < C::CPL; ++e) o[qi][e] = 0.f;
    }
    const int grp = warp / 4;               // tiles t with t % 2 == grp
    const int wq = warp % 4;                // key quarter within a tile
    const int r = 32 * wq + lane;           // this lane's key row within a tile
    bool ok = true;
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
      const uint8_t* kt = smem + C::K_OFF + s * C::TILE_BYTES;
      const uint8_t* vt = smem + C::V_OFF + s * C::TILE_BYTES;
      // scores of this lane's key against every query row
      float sc4[NQ][4];
#pragma unroll
      for (int qi = 0; qi < NQ; ++qi)
#pragma unroll
        for (int e = 0; e < 4; ++e) sc4[qi][e] = 0.f;
#pragma unroll
      for (int u = 0; u < D / 8; ++u) {
        const int phys = (u % 8) ^ (r & 7);
        const uint4 kv = *reinterpret_cast<const uint4*>(kt + (u / 8) * C::CHUNK_BYTES + r * 128 +
                                                         phys * 16);
        const float kf[8] = {bf16lo(kv.x), bf16hi(kv.x), bf16lo(kv.y), bf16hi(kv.y),
                             bf16lo(kv.z), bf16hi(kv.z), bf16lo(kv.w), bf16hi(kv.w)};
#pragma unroll
        for (int qi = 0; qi < NQ; ++qi) {
          if (qi < nq) {
            const float4 q0 = *reinterpret_cast<const float4*>(qs + qi * D + u * 8);
            const float4 q1 = *reinterpret_cast<const float4*>(qs + qi * D + u * 8 + 4);
            sc4[qi][0] = fmaf(q0.x, kf[0], sc4[qi][0]);
            sc4[qi][1] = fmaf(q0.y, kf[1], sc4[qi][1]);
            sc4[qi][2] = fmaf(q0.z, kf[2], sc4[qi][2]);
            sc4[qi][3] = fmaf(q0.w, kf[3], sc4[qi][3]);
            sc4[qi][0] = fmaf(q1.x, kf[4], sc4[qi][0]);
            sc4[qi][1] = fmaf(q1.y, kf[5], sc4[qi][1]);
            sc4[qi][2] = fmaf(q1.z, kf[6], sc4[qi][2]);
            sc4[qi][3] = fmaf(q1.w, kf[7], sc4[qi][3]);
          }
        }
      }
      float sc[NQ];
#pragma unroll
      for (int qi = 0; qi < NQ; ++qi)
        sc[qi] = (sc4[qi][0] + sc4[qi][1]) + (sc4[qi][2] + sc4[qi][3]);
      const bool valid = k_begin + t * C::TK + r < k_end;
      // online softmax per query row, over this warp's 32 keys, in base 2
      float pj[NQ];
#pragma unroll
      for (int qi = 0; qi < NQ; ++qi) {
        if (qi < nq) {
          const float x = valid ? sc[qi] * p.scale_log2 : -INFINITY;
          float mx = x;
#pragma unroll
          for (int off = 16; off > 0; off >>= 1)
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
          const float m_new = fmaxf(m[qi], mx);
          const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
          const float alpha = ex2_approx(m[qi] - m_use);
          const float pv = ex2_approx(x - m_use);
          float sum = pv;
#pragma unroll
          for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
          l[qi] = l[qi] * alpha + sum;
#pragma unroll
          for (int e = 0; e < C::CPL; ++e) o[qi][e] *= alpha;
          m[qi] = m_new;
          pj[qi] = pv;
        }
      }
      // P.V: lane l owns columns [CPL*l, CPL*(l+1))
#pragma unroll 4
      for (int j = 0; j < 32; ++j) {
        const int rv = 32 * wq + j;
        float vf[C::CPL];
        if constexpr (D == 128) {
          const int c = lane / 16;
          const int byte = 8 * (lane % 16);
          const int phys = (byte / 16) ^ (rv & 7);
          const uint2 vv = *reinterpret_cast<const uint2*>(vt + c * C::CHUNK_BYTES + rv * 128 +
                                                           phys * 16 + (byte % 16));
          vf[0] = bf16lo(vv.x);
          vf[1] = bf16hi(vv.x);
          vf[C::CPL > 2 ? 2 : 0] = bf16lo(vv.y);
          vf[C::CPL > 3 ? 3 : 0] = bf16hi(vv.y);
        } else {
          const int byte = 4 * lane;
          const int phys = (byte / 16) ^ (rv & 7);
          const uint32_t vv =
              *reinterpret_cast<const uint32_t*>(vt + rv * 128 + phys * 16 + (byte % 16));
          vf[0] = bf16lo(vv);
          vf[C::CPL > 1 ? 1 : 0] = bf16hi(vv);
        }
#pragma unroll
        for (int qi = 0; qi < NQ; ++qi) {
          if (qi < nq) {
            const float pb = __shfl_sync(0xffffffffu, pj[qi], j);
#pragma unroll
            for (int e = 0; e < C::CPL; ++e) o[qi][e] = fmaf(pb, vf[e], o[qi][e]);
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
    }
    // merge the eight warps through shared memory (the drained K/V stages):
    // every compute warp must be past its last tile before the area is reused
    asm volatile("bar.sync 1, %0;" ::"n"(32 * C::WARPS) : "memory");
    // after an abort, copies may still be landing in the stages: skip the merge
    ok = !*abort_flag;
    if (ok) {
#pragma unroll
      for (int qi = 0; qi < NQ; ++qi) {
        if (qi < nq) {
          if (lane == 0) {
            ms[warp * kDecodeMaxQ + qi] = m[qi];
            ls[warp * kDecodeMaxQ + qi] = l[qi];
          }
#pragma unroll
          for (int e = 0; e < C::CPL; ++e)
            os[(warp * kDecodeMaxQ + qi) * D + C::CPL * lane + e] = o[qi][e];
        }
      }
    }
    asm volatile("bar.sync 1, %0;" ::"n"(32 * C::WARPS) : "memory");
    if (ok && !*abort_flag) {
      for (int i = threadIdx.x; i < nq * D; i += 32 * C::WARPS) {
        const int qi = i / D, d = i - qi * D;
        float mt = -INFINITY;
#pragma unroll
        for (int w = 0; w < C::WARPS; ++w) mt = fmaxf(mt, ms[w * kDecodeMaxQ + qi]);
        const float mu = (mt == -INFINITY) ? 0.f : mt;
        float lt = 0.f, ot = 0.f;
#pragma unroll
        for (int w = 0; w < C::WARPS; ++w) {
          const float f = ex2_approx(ms[w * kDecodeMaxQ + qi] - mu);
          lt += f * ls[w * kDecodeMaxQ + qi];
          ot += f * os[(w * kDecodeMaxQ + qi) * D + d];
        }
        const float out = ot / lt;
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
