// 16-bit (bf16 or fp16) attention backward for sm_103a: TMA + mbarrier
// pipeline, tcgen05 MMAs with TMEM accumulators.
//
// What it computes is the gradient of the forward for an upstream gradient
// dO, the backward pass that "Building a FlashAttention-2 forward kernel in
// pure NumPy" names as the next extension ("Extending It: Your Roadmap to
// Senior-Level"): the forward's log-sum-exp is kept, the probabilities are
// rebuilt tile by tile from it (P_ij = exp(scale q_i.k_j - LSE_i)), and
//
//     dV = P^T dO,   dP = dO V^T,   dS = P * (dP - Delta),
//     dQ = scale dS K,   dK = scale dS^T Q,   Delta_i = dO_i . O_i.
//
// Masked entries (the causal mask, aligned like the forward's: key j is
// allowed for query i when j <= i + Nk - Nq) have P = 0 and so contribute
// nothing.
//
// Three kernels run in order on the caller's stream:
//   attn_bwd_prep_kernel   Delta_i = dO_i . O_i (fp32) and a zeroed fp32 dQ
//                          accumulator, both in the caller's workspace;
//   attn_bwd_bf16_kernel   persistent, one CTA per SM: it takes 128-key tiles
//                          of one plane (work items, heaviest first) from a
//                          counter of the launch; for each it keeps dK and dV
//                          for its keys in TMEM, streams the query tiles that
//                          see those keys, and adds each tile's dQ
//                          contribution to the fp32 accumulator;
//   attn_bwd_dq_kernel     dQ = scale * accumulator, rounded once.
//
// CTA layout of the main kernel (448 threads):
//   warps 0-7  "P/dS" warps: warp w owns key rows 32*(w%4).. (TMEM lanes) and
//              the query columns 64*(w/4) .. +63 of each tile, so two warps
//              share each SM sub-partition and hide each other's latency.
//              P^T = 2^(S^T * scale*log2e - LSE_q*log2e) goes back into TMEM
//              as 16-bit pairs for the dV MMA; dS^T = P^T (dP^T - Delta_q) is
//              written to shared memory for the dK and dQ MMAs.
//   warps 8-11 "dQ" warpgroup: thread t owns query row t of the dQ tile;
//              it loads its whole row from TMEM into registers (which frees
//              the columns for the next dP^T at once), then stages each
//              32 x 32 block in shared memory and adds it to the fp32
//              accumulator with a TMA reduction (whole 128-byte lines, far
//              fewer L2 operations than per-thread atomics).  At the end it
//              writes dK.
//   warp  12   tcgen05 MMA issuer and TMEM owner.
//   warp  13   TMA producer: takes the key tiles and hands them to the other
//              warps through a ring in shared memory; loads K and V per key
//              tile (as soon as the previous tile's MMAs are done with them),
//              Q and dO per query tile, and each query tile's -LSE*log2(e)
//              and -Delta into shared memory, read from global memory before
//              the stage is free so their latency hides behind the wait.
//
// Key tiles follow each other without a pause in the pipeline: every
// per-query-tile barrier counts the query tiles of all key tiles so far; the
// P/dS warps write the finished dV, the dQ warps the finished dK, while the
// next key tile's K and V load and its first S^T is computed (the next tile's
// first dK MMA waits until dK has been read out, acc_empty; its first dV MMA
// needs the P/dS warps' next P, which they compute after reading dV).
//
// TMEM columns (fp32 cells, 128 lanes): dV [0, D), dK [D, 2D),
// S^T [2D, 2D+128) (P^T for queries 0-63 overwrites its columns 0-31 and
// for queries 64-127 its columns 64-95, each half in columns it has read), dP^T
// [2D+128, 2D+256) (dS^T as 16-bit pairs overwrites the same columns of it,
// the A operand of dK += dS^T Q); each tile's dQ (lanes = queries) reuses the
// dP^T columns after that dK MMA.
//
// Shared memory: K, V (the current key tile), two Q stages, one dO stage, the dS
// tile, the per-stage LSE/Delta vectors and two 4 KB dQ staging buffers per
// dQ warp (about 226 KB: the kernel takes the dynamic shared memory base as
// it comes, 1024-byte aligned, and refuses to run otherwise).  Every 128 x D
// tile is stored as TMA writes it: D/64 chunks of 128 rows x 128 bytes,
// 128-byte swizzled.  The
// dS tile is written in the same format with keys as rows and queries along
// the row: the MN-major A operand of dQ = dS K (M = queries).  dK += dS^T Q
// (M = keys) takes dS^T from TMEM instead, which saves the tile's second read
// from shared memory, the resource that bounds this kernel.
//
// MMA order per query tile i:  dP_i (two halves of 64 queries, each as soon as
// the previous dQ has left its columns), [P_i ready] dV += P_i^T dO_i, S_{i+1},
// [dS_i ready] dK += dS_i^T Q_i, dQ_i = dS_i K.  S_{i+1} overwrites the
// columns P_i was read from, and dQ_i the columns dS_i^T was read from, which
// the tensor pipe orders after the MMAs that read them.
#pragma once

#include <cuda_fp16.h>

#include "ptx.cuh"

namespace attn {

// 32 lanes x 16 columns of TMEM from 16 registers per thread (asynchronous;
// pair with tmem_wait_st).  Only the backward stores 16-column slices.
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
      "r"(r[15])
      : "memory");
}

struct BwdParams {
  const void* o;            // forward output, layout of q (prep kernel)
  const void* dout;         // upstream gradient, layout of q
  const float* lse;         // forward log-sum-exp, natural log, layout (planes, rows)
  float* delta;             // workspace: Delta, layout of lse
  float* dq_acc;            // workspace: fp32 dQ accumulator, layout of q
  void* dq;
  void* dk;
  void* dv;
  const int* cu_seqlens;    // query offsets; nullptr for the dense layout
  const int* cu_seqlens_k;  // key offsets (packed layout only)
  int nseq;
  int planes;               // dense: B*H; packed: H
  int rows;                 // query rows per plane (dense Nq; packed total query tokens)
  int rows_k;               // key rows per plane (dense Nk; packed total key tokens)
  int n_kblk;               // dense: ceil(Nk/128)
  int n_tiles;              // packed: an upper bound on the key tiles
  int causal;
  float scale;
  float scale_log2;         // scale * log2(e)
  int stall;                // abort-path test: CTA 0 waits on a phase nothing completes
  unsigned long long timeout_ns;
  unsigned int* err;
  // Work counter of this launch (next key tile, CTAs finished), zero at launch
  // and reset to zero by the last CTA to finish.
  unsigned int* sched;
};

// Depth of the shared-memory ring through which the TMA producer hands the
// key tiles it takes to the other warps.
constexpr int kBwdRing = 4;
constexpr uint32_t kBwdSlotBytes = 48;

template <int D>
struct BwdCfg {
  static constexpr int BM = 128;                  // queries per tile
  static constexpr int BN = 128;                  // keys per CTA
  static constexpr int CHUNK_BYTES = 128 * 128;   // 128 rows x 128 bytes
  static constexpr int NCHUNK = D / 64;
  static constexpr int TILE_BYTES = 128 * D * 2;
  static constexpr int K_OFF = 0;
  static constexpr int V_OFF = TILE_BYTES;
  static constexpr int Q_OFF = 2 * TILE_BYTES;    // two stages
  static constexpr int DO_OFF = 4 * TILE_BYTES;   // one stage
  static constexpr int DS_OFF = 5 * TILE_BYTES;
  static constexpr int DS_BYTES = 2 * CHUNK_BYTES;  // 128 keys x 128 queries
  static constexpr int STAT_OFF = DS_OFF + DS_BYTES;
  static constexpr int STAT_BYTES = 2 * 256 * 4;  // per stage: -LSE*log2e[128], -Delta[128]
  static constexpr int STG_OFF = STAT_OFF + STAT_BYTES;   // dQ staging: 4 warps x 2 x 4 KB
  static constexpr int STG_BYTES = 4 * 2 * 4096;
  static constexpr int BAR_OFF = STG_OFF + STG_BYTES;
  // kv_full, q_full[2], q_empty[2], do_full, do_empty, s_full, dp_full[2], p_full,
  // ds_full, ds_empty, dq_full, dq_empty[2], mma_done, kv_empty, acc_full, acc_empty,
  // tile_full[kBwdRing], tile_empty[kBwdRing]
  static constexpr int TILE_BAR = 20;  // index of tile_full[0]
  static constexpr int NBAR = TILE_BAR + 2 * kBwdRing;
  static constexpr int MISC_OFF = BAR_OFF + NBAR * 8;
  static constexpr int RING_OFF = (MISC_OFF + 16 + 15) / 16 * 16;  // kBwdRing slots of 48 bytes
  static constexpr int SMEM_BYTES = RING_OFF + kBwdRing * kBwdSlotBytes;
  // at least 117 KB, so that one CTA (which takes all of TMEM) runs per SM
  static constexpr int SMEM_ALLOC = (SMEM_BYTES > 119808) ? SMEM_BYTES : 119808;
  static constexpr int THREADS = 448;
  static constexpr uint32_t TMEM_COLS = 512;
  static constexpr uint32_t DV_COL = 0, DK_COL = D, S_COL = 2 * D, DP_COL = 2 * D + 128;
  // D = 64 leaves 128 columns free: dQ gets its own, so that dP^T of the next
  // query tile does not wait for dQ to leave the dP^T columns, and dP^T is one
  // N = 128 MMA group instead of two halves (DQ_OWN).  At D = 128 dQ reuses the
  // dP^T columns.
  static constexpr bool DQ_OWN = (D == 64);
  static constexpr uint32_t DQ_COL = DQ_OWN ? DP_COL + 128 : DP_COL;
  static_assert(D == 64 || D == 128, "head dim");
  static_assert(DP_COL + 128 <= TMEM_COLS && DQ_COL + (DQ_OWN ? D : 0) <= TMEM_COLS,
                "tensor memory");
  static_assert(SMEM_ALLOC <= 232448, "shared memory");
};

// A key tile and the query tiles that see it.
struct BwdTile {
  int plane;
  int q_base, q_len;    // the sequence's first query row in the maps, and its query count
  int kv_base, kv_len;  // likewise for keys
  int kblk;             // 128-key block within the sequence
  int qt0, nqt;         // first query tile that sees a key of the block, and the tile count
};

// Work item t.  Dense layout: key block t / planes of plane t % planes, so
// the blocks that see the most query tiles under the causal mask (block 0)
// come first and the CTAs, taking the items in order as they free up, end
// within about one light item of each other.  Packed layout: key blocks
// sequence by sequence.  Returns false past the last item (or when
// cu_seqlens is malformed).
__device__ __forceinline__ bool bwd_tile(const BwdParams& p, int t, BwdTile& w) {
  w.plane = t % p.planes;
  const int vb = t / p.planes;
  if (p.cu_seqlens == nullptr) {
    if (vb >= p.n_kblk) return false;
    w.kblk = vb;
    w.q_base = 0;
    w.q_len = p.rows;
    w.kv_base = 0;
    w.kv_len = p.rows_k;
  } else {
    int cum = 0;
    bool found = false;
    for (int s = 0; s < p.nseq; ++s) {
      const int ak = __ldg(p.cu_seqlens_k + s), ek = __ldg(p.cu_seqlens_k + s + 1);
      if (ak < 0 || ek < ak || ek > p.rows_k) {
        if ((threadIdx.x % 32) == 0) atomicOr(p.err, kDevErrBounds);
        return false;
      }
      const int nb = (ek - ak + 127) / 128;
      if (vb < cum + nb) {
        const int a = __ldg(p.cu_seqlens + s), e = __ldg(p.cu_seqlens + s + 1);
        if (a < 0 || e < a || e > p.rows) {
          if ((threadIdx.x % 32) == 0) atomicOr(p.err, kDevErrBounds);
          return false;
        }
        w.q_base = a;
        w.q_len = e - a;
        w.kv_base = ak;
        w.kv_len = ek - ak;
        w.kblk = vb - cum;
        found = true;
        break;
      }
      cum += nb;
    }
    if (!found) return false;
  }
  const int nq_tiles = (w.q_len + 127) / 128;
  int first = 0;
  if (p.causal) {
    // the first query that sees key k0 is k0 - (Nk - Nq)
    const int r = w.kblk * 128 - (w.kv_len - w.q_len);
    first = r <= 0 ? 0 : r / 128;
  }
  w.qt0 = min(first, nq_tiles);
  w.nqt = nq_tiles - w.qt0;
  return true;
}

// The key tiles the producer takes reach the other warps through a ring of
// kBwdRing slots in shared memory (32-bit shared addresses: the first slot,
// the first tile_full barrier; the tile_empty barriers follow them): a slot
// holds the tile or the end of the walk, tile_full[slot] completes when it is
// written, tile_empty[slot] when all thirteen readers have copied it.
__device__ __forceinline__ bool bwd_publish(uint32_t ring, uint32_t full, int n, bool run,
                                            const BwdTile& w, const WaitCtl& ctl) {
  const uint32_t slot = static_cast<uint32_t>(n % kBwdRing);
  const uint32_t lap = static_cast<uint32_t>(n / kBwdRing);
  const uint32_t empty = full + 8 * kBwdRing;
  if (lap > 0 && !__all_sync(0xffffffffu, mbar_wait_at(empty + 8 * slot, (lap - 1) & 1, ctl)))
    return false;
  if ((threadIdx.x % 32) == 0) {
    const uint32_t a = ring + kBwdSlotBytes * slot;
    st_shared_v4(a, run ? 1u : 0u, w.plane, w.q_base, w.q_len);
    st_shared_v4(a + 16, w.kv_base, w.kv_len, w.kblk, w.qt0);
    st_shared_v4(a + 32, w.nqt, 0u, 0u, 0u);
    mbar_arrive_at(full + 8 * slot);  // release: the slot's contents are visible to its readers
  }
  __syncwarp();
  return true;
}

// Reader (warp-uniform): the n-th key tile; false at the end of the walk or
// when the CTA is aborting.  A reader that keeps the slot (kRelease false)
// reads words of it again later (bwd_slot_word) instead of holding them in
// registers through its loop, and releases it with bwd_release.  Words of a
// slot: 0 run, 1 plane, 2 q_base, 3 q_len, 4 kv_base, 5 kv_len, 6 kblk, 7 qt0,
// 8 nqt.
template <bool kRelease = true>
__device__ __forceinline__ bool bwd_read(uint32_t ring, uint32_t full, int n, BwdTile& w,
                                         const WaitCtl& ctl) {
  const uint32_t slot = static_cast<uint32_t>(n % kBwdRing);
  const uint32_t lap = static_cast<uint32_t>(n / kBwdRing);
  if (!__all_sync(0xffffffffu, mbar_wait_at(full + 8 * slot, lap & 1, ctl))) return false;
  const uint32_t a = ring + kBwdSlotBytes * slot;
  uint32_t r0[4], r1[4], r2[4];
  ld_shared_v4(a, r0);
  ld_shared_v4(a + 16, r1);
  ld_shared_v4(a + 32, r2);
  w.plane = static_cast<int>(r0[1]);
  w.q_base = static_cast<int>(r0[2]);
  w.q_len = static_cast<int>(r0[3]);
  w.kv_base = static_cast<int>(r1[0]);
  w.kv_len = static_cast<int>(r1[1]);
  w.kblk = static_cast<int>(r1[2]);
  w.qt0 = static_cast<int>(r1[3]);
  w.nqt = static_cast<int>(r2[0]);
  if (kRelease) {
    __syncwarp();
    if ((threadIdx.x % 32) == 0) mbar_arrive_at(full + 8 * kBwdRing + 8 * slot);
  }
  return r0[0] != 0;
}

__device__ __forceinline__ int bwd_slot_word(uint32_t ring, int n, int word) {
  uint32_t v;
  asm volatile("ld.shared.u32 %0, [%1];"
               : "=r"(v)
               : "r"(ring + kBwdSlotBytes * static_cast<uint32_t>(n % kBwdRing) + 4 * word)
               : "memory");
  return static_cast<int>(v);
}

__device__ __forceinline__ void bwd_release(uint32_t full, int n) {
  __syncwarp();
  if ((threadIdx.x % 32) == 0)
    mbar_arrive_at(full + 8 * kBwdRing + 8 * static_cast<uint32_t>(n % kBwdRing));
}

// First element of key row `row` of the key tile in slot n of the ring, in a
// (planes, rows_k, D) tensor.
template <int D>
__device__ __forceinline__ uint16_t* bwd_slot_key_row(void* base, int rows_k, uint32_t ring,
                                                      int n, int row) {
  const size_t r = static_cast<size_t>(bwd_slot_word(ring, n, 1)) * rows_k +
                   bwd_slot_word(ring, n, 4) + bwd_slot_word(ring, n, 6) * 128 + row;
  return static_cast<uint16_t*>(base) + r * D;
}

// acc (+)= A B over kdim/16 steps with both operands K-major in shared memory.
template <int KDIM>
__device__ __forceinline__ void bwd_mma_kk(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                           uint32_t accumulate) {
#pragma unroll
  for (int kk = 0; kk < KDIM / 16; ++kk) {
    const uint32_t off = ((kk / 4) * (128 * 128) + (kk % 4) * 32) >> 4;
    umma_ss_warp(d_tmem, a + off, b + off, idesc, (accumulate || kk > 0) ? 1u : 0u);
  }
}

// NCOL columns of one key row of dK or dV from TMEM (scaled by mul and
// rounded), or zeros, to global memory.
template <int NCOL, bool F16>
__device__ __forceinline__ void bwd_store_row(uint32_t t_src, uint16_t* dst, bool valid, float mul,
                                              bool zero) {
#pragma unroll
  for (int cc = 0; cc < NCOL / 32; ++cc) {
    uint32_t r[32];
    if (!zero) {
      tmem_ld32_wait(t_src + 32 * cc, r);
    } else {
#pragma unroll
      for (int e = 0; e < 32; ++e) r[e] = 0u;
    }
    uint32_t h[16];
#pragma unroll
    for (int e = 0; e < 16; ++e)
      h[e] = pack_16x2<F16>(__uint_as_float(r[2 * e]) * mul, __uint_as_float(r[2 * e + 1]) * mul);
    if (valid) {
      uint4* d4 = reinterpret_cast<uint4*>(dst + 32 * cc);
#pragma unroll
      for (int v = 0; v < 4; ++v)
        d4[v] = make_uint4(h[4 * v], h[4 * v + 1], h[4 * v + 2], h[4 * v + 3]);
    }
  }
}

template <int D, bool F16>
__global__ void __launch_bounds__(448, 1)
    attn_bwd_bf16_kernel(const __grid_constant__ CUtensorMap tmQ,
                         const __grid_constant__ CUtensorMap tmK,
                         const __grid_constant__ CUtensorMap tmV,
                         const __grid_constant__ CUtensorMap tmDO,
                         const __grid_constant__ CUtensorMap tmDQ, const BwdParams p) {
  using C = BwdCfg<D>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = smem_raw;
  if ((smem_u32(smem) & 1023u) != 0) {  // the swizzled layout needs a 1024-byte aligned base
    if (threadIdx.x == 0) {
      atomicOr(p.err, kDevErrLayout);
      sched_done(p.sched);
    }
    return;
  }
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::BAR_OFF);
  uint64_t* kv_full = bars;
  uint64_t* q_full = bars + 1;   // [2]
  uint64_t* q_empty = bars + 3;  // [2]
  uint64_t* do_full = bars + 5;
  uint64_t* do_empty = bars + 6;
  uint64_t* s_full = bars + 7;
  uint64_t* dp_full = bars + 8;    // [2]: query columns 0-63, 64-127
  uint64_t* p_full = bars + 10;
  uint64_t* ds_full = bars + 11;
  uint64_t* ds_empty = bars + 12;
  uint64_t* dq_full = bars + 13;
  uint64_t* dq_empty = bars + 14;  // [2]: TMEM columns 0-63, 64-127 read
  uint64_t* mma_done = bars + 16;  // every MMA of the CTA is complete
  uint64_t* kv_empty = bars + 17;  // the key tile's MMAs are done with K and V
  uint64_t* acc_full = bars + 18;  // the key tile's dK and dV are final in TMEM
  uint64_t* acc_empty = bars + 19; // dK has been read out of TMEM
  uint64_t* tile_bars = bars + C::TILE_BAR;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::MISC_OFF);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::MISC_OFF + 4);
  float* stat = reinterpret_cast<float*>(smem + C::STAT_OFF);

  {
    BwdTile w0;
    if (!bwd_tile(p, static_cast<int>(blockIdx.x), w0)) {  // uniform: no work for this CTA
      if (threadIdx.x == 0) sched_done(p.sched);
      return;
    }
  }

  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;

  if (threadIdx.x == 0) {
    mbar_init(kv_full, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&q_full[i], 1 + 32);  // 32 producer lanes (LSE/Delta) + the expect_tx arrival
      mbar_init(&q_empty[i], 1);
    }
    mbar_init(do_full, 1);
    mbar_init(do_empty, 1);
    mbar_init(s_full, 1);
    mbar_init(&dp_full[0], 1);
    mbar_init(&dp_full[1], 1);
    mbar_init(p_full, 256);
    mbar_init(ds_full, 256);
    mbar_init(ds_empty, 1);
    mbar_init(dq_full, 1);
    mbar_init(&dq_empty[0], 128);
    mbar_init(&dq_empty[1], 128);
    mbar_init(mma_done, 1);
    mbar_init(kv_empty, 1);
    mbar_init(acc_full, 1);
    mbar_init(acc_empty, 128);
    for (int i = 0; i < kBwdRing; ++i) {
      mbar_init(&tile_bars[i], 1);
      mbar_init(&tile_bars[kBwdRing + i], 13);  // P/dS warps, dQ warps, the MMA warp
    }
    *abort_flag = 0;
    mbar_fence_init();
  }
  if (warp == 12) {
    tmem_alloc(tmem_slot, C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const WaitCtl ctl{abort_flag, p.err, p.timeout_ns};
  const uint32_t smem_base = smem_u32(smem);
  const uint32_t ring = smem_base + C::RING_OFF;
  const uint32_t ring_bar = smem_base + C::BAR_OFF + 8 * C::TILE_BAR;
  auto wait = [&](uint64_t* bar, uint32_t parity) {
    return __all_sync(0xffffffffu, mbar_wait(bar, parity, ctl));
  };

  // Every role walks the same key tiles (the producer takes them and publishes
  // them in the ring); g counts the query tiles of all key tiles so far (the
  // phases of the per-query-tile barriers), kt the key tiles with queries (the
  // phases of kv_full, kv_empty, acc_full, acc_empty).
  if (warp < 8) {
    // ------------------------------------------------------------ P and dS
    const int hf = warp >> 2;              // query columns 64*hf .. 64*hf+63 of each tile
    const int t = threadIdx.x & 127;       // key row within the tile
    const uint32_t lane_off = static_cast<uint32_t>(32 * (warp & 3)) << 16;
    const uint32_t tS = tmem + lane_off + C::S_COL + 64 * hf;
    const uint32_t tDP = tmem + lane_off + C::DP_COL + 64 * hf;
    const uint64_t c2 = f32x2(p.scale_log2, p.scale_log2);
    const uint32_t ds_row = smem_base + C::DS_OFF + hf * C::CHUNK_BYTES + t * 128;
    bool ok = true;
    int g = 0;
    uint32_t kt = 0;
    for (int nt = 0; ok; ++nt) {
      // the slot of the previous key tile was kept for its epilogue
      if (nt > 0) bwd_release(ring_bar, nt - 1);
      BwdTile w;
      if (!bwd_read<false>(ring, ring_bar, nt, w, ctl)) break;
      const int n = w.nqt;
      const int key = w.kblk * C::BN + t;
      const bool key_ok = key < w.kv_len;
      if (n == 0) {
        // no query sees these keys: their gradients are zero
        if (warp < 4) {
          bwd_store_row<D, F16>(0, bwd_slot_key_row<D>(p.dv, p.rows_k, ring, nt, t), key_ok, 1.f,
                                true);
          bwd_store_row<D, F16>(0, bwd_slot_key_row<D>(p.dk, p.rows_k, ring, nt, t), key_ok, 1.f,
                                true);
        }
        continue;
      }
      // With q0 = qt0*BM + 64*hf + i*BM the first query of this half of query
      // tile i and off = kv_len - q_len the causal alignment: columns c < cmin =
      // key - off - q0 are future queries for this key, and the tile needs the
      // mask when the key tile's last key k0 + BN - 1 lies past q0 + off.
      const int qb = w.qt0 * C::BM + 64 * hf;
      const int cm0 = p.causal ? key - (w.kv_len - w.q_len) - qb : -1;
      const int mth = w.kblk * C::BN + C::BN - 1 - (w.kv_len - w.q_len) - qb;
      for (int i = 0; i < n; ++i, ++g) {
        const int st = g & 1;
        const float* nlse = stat + st * 256 + 64 * hf;  // -LSE * log2(e) per query column
        const float* dlt = nlse + 128;                  // -Delta per query column
        if (!wait(s_full, g & 1)) {
          ok = false;
          break;
        }
        tc_fence_after();
        uint32_t sr[64];
        tmem_ld64_wait(tS, sr);
        const int cmin = p.causal ? cm0 - i * C::BM : -1;
        const bool need_mask = !key_ok || (p.causal && mth > i * C::BM);
        uint32_t pk[32];
#pragma unroll
        for (int c4 = 0; c4 < 16; ++c4) {
          const uint4 nl = *reinterpret_cast<const uint4*>(nlse + 4 * c4);
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const int c = 2 * c4 + h;
            const uint64_t x2 = ffma2(u32x2(sr[2 * c], sr[2 * c + 1]), c2,
                                      h ? u32x2(nl.z, nl.w) : u32x2(nl.x, nl.y));
            float a = ex2_approx(lo_f32(x2));
            float b = ex2_approx(hi_f32(x2));
            if (need_mask) {
              if (!key_ok || 2 * c < cmin) a = 0.f;
              if (!key_ok || 2 * c + 1 < cmin) b = 0.f;
            }
            pk[c] = pack_16x2<F16>(a, b);
          }
        }
        // P^T as 16-bit pairs into the first 32 of the 64 columns just read
        tmem_st32(tS, pk);
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(p_full);

        if (!wait(&dp_full[hf], g & 1)) {
          ok = false;
          break;
        }
        tc_fence_after();
        // the previous dS must have been read by its dK and dQ MMAs
        if (g > 0 && !wait(ds_empty, (g - 1) & 1)) {
          ok = false;
          break;
        }
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
          uint32_t dr[32];
          tmem_ld32_wait(tDP + 32 * cc, dr);
          uint32_t h[16];
#pragma unroll
          for (int e4 = 0; e4 < 8; ++e4) {
            // -Delta for four query columns
            const uint4 nd = *reinterpret_cast<const uint4*>(dlt + 32 * cc + 4 * e4);
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
              const int e = 2 * e4 + hh;
              const uint32_t pp = pk[16 * cc + e];
              float plo, phi;
              if constexpr (F16) {
                const __half2 hv = *reinterpret_cast<const __half2*>(&pp);
                plo = __low2float(hv);
                phi = __high2float(hv);
              } else {
                plo = __uint_as_float(pp << 16);
                phi = __uint_as_float(pp & 0xffff0000u);
              }
              const uint64_t d2 = fadd2(u32x2(dr[2 * e], dr[2 * e + 1]),
                                        hh ? u32x2(nd.z, nd.w) : u32x2(nd.x, nd.y));
              const uint64_t s2 = fmul2(f32x2(plo, phi), d2);
              h[e] = pack_16x2<F16>(lo_f32(s2), hi_f32(s2));
            }
          }
          // dS^T as 16-bit pairs into this half's dP^T columns already read
          // (the A operand of dK += dS^T Q)
          tmem_st16(tDP + 16 * cc, h);
          // 32 queries = 64 bytes = four 16-byte units of this key's 128-byte row
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const uint32_t unit = static_cast<uint32_t>(cc * 4 + u) ^ static_cast<uint32_t>(t & 7);
            st_shared_v4(ds_row + unit * 16, h[4 * u], h[4 * u + 1], h[4 * u + 2], h[4 * u + 3]);
          }
        }
        fence_proxy_async_smem();
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(ds_full);
      }
      if (!ok) break;
      // dV epilogue: this warp's half of the columns.  The next key tile's
      // first dV MMA overwrites them only after this warp's next P arrival,
      // which comes after these loads.
      if (!wait(acc_full, kt & 1)) {
        ok = false;
        break;
      }
      tc_fence_after();
      bwd_store_row<D / 2, F16>(tmem + lane_off + C::DV_COL + (D / 2) * hf,
                                bwd_slot_key_row<D>(p.dv, p.rows_k, ring, nt, t) + (D / 2) * hf,
                                key_ok, 1.f, false);
      ++kt;
    }
  } else if (warp < 12) {
    // ------------------------------------------------------------ dQ drain
    const int t = threadIdx.x - 256;  // query row within the tile
    const uint32_t lane_off = static_cast<uint32_t>(32 * (warp - 8)) << 16;
    const uint32_t tQ = tmem + lane_off + C::DQ_COL;
    // Rows of the tile past the sequence's end carry dQ = 0 exactly (their P
    // and dS columns are zero), so a box that reaches into the next plane's or
    // sequence's rows adds zeros there; rows past the whole tensor are clipped.
    bool ok = true;
    const uint32_t stg = smem_base + C::STG_OFF + (warp - 8) * 8192 + lane * 128;
    int nstaged = 0;
    int g = 0;
    uint32_t kt = 0;
    for (int nt = 0; ok; ++nt) {
      // the slot of the previous key tile was kept for its epilogue
      if (nt > 0) bwd_release(ring_bar, nt - 1);
      BwdTile w;
      if (!bwd_read<false>(ring, ring_bar, nt, w, ctl)) break;
      const int n = w.nqt;
      if (n == 0) continue;
      // first dQ accumulator row of this warp's 32 rows of query tile 0
      const int rb = w.plane * p.rows + w.q_base + w.qt0 * C::BM + 32 * (warp - 8);
      for (int i = 0; i < n; ++i, ++g) {
        if (!wait(dq_full, g & 1)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const int row0 = rb + i * C::BM;
        // Two halves of 64 columns: each is released for the next dP^T half as
        // soon as it is in registers, then staged and reduced.
#pragma unroll
        for (int hq = 0; hq < 2; ++hq) {
          constexpr int NC = (D < 64) ? D : 64;  // columns per half (the second is empty at D = 64)
          uint32_t r[64];
          if (hq * 64 < D) {
            tmem_ld64_wait(tQ + 64 * hq, r);
          }
          tc_fence_before();
          mbar_arrive(&dq_empty[hq]);
          if (hq * 64 >= D) continue;
#pragma unroll
          for (int cc = 0; cc < NC / 32; ++cc) {
            const uint32_t buf = stg + (nstaged & 1) * 4096;
            // the reduction that last read this buffer must be done with it
            if (lane == 0 && nstaged >= 2) bulk_wait_group_read<1>();
            __syncwarp();
#pragma unroll
            for (int u = 0; u < 8; ++u)
              st_shared_v4(buf + ((u ^ (lane & 7)) * 16), r[32 * cc + 4 * u],
                           r[32 * cc + 4 * u + 1], r[32 * cc + 4 * u + 2], r[32 * cc + 4 * u + 3]);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              tma_reduce_add_2d(&tmDQ, buf - lane * 128, 64 * hq + 32 * cc, row0);
              bulk_commit_group();
            }
            ++nstaged;
          }
        }
      }
      if (!ok) break;
      // dK epilogue (dK = scale * dS^T Q); the next key tile's first dK MMA
      // waits for acc_empty
      if (!wait(acc_full, kt & 1)) {
        ok = false;
        break;
      }
      tc_fence_after();
      bwd_store_row<D, F16>(tmem + lane_off + C::DK_COL,
                            bwd_slot_key_row<D>(p.dk, p.rows_k, ring, nt, t),
                            bwd_slot_word(ring, nt, 6) * C::BN + t < bwd_slot_word(ring, nt, 5),
                            p.scale, false);
      tc_fence_before();
      mbar_arrive(acc_empty);
      ++kt;
    }
    if (lane == 0) bulk_wait_group<0>();
  } else if (warp == 12) {
    // ------------------------------------------------------------ MMA issuer
    constexpr uint32_t id_s = idesc_bf16_f32(128, 128, 0, 0, F16);   // S^T
    constexpr uint32_t id_s64 = idesc_bf16_f32(128, 64, 0, 0, F16);   // half of dP^T
    constexpr uint32_t id_kv = idesc_bf16_f32(128, D, 0, 1, F16);   // dV (TS), dK
    constexpr uint32_t id_dq = idesc_bf16_f32(128, D, 1, 1, F16);   // dQ: A MN-major
    const uint64_t kA = sdesc_sw128(smem_base + C::K_OFF, 16, 1024);
    const uint64_t vA = sdesc_sw128(smem_base + C::V_OFF, 16, 1024);
    const uint64_t kMN = sdesc_sw128(smem_base + C::K_OFF, C::CHUNK_BYTES, 1024);
    const uint64_t doK = sdesc_sw128(smem_base + C::DO_OFF, 16, 1024);
    const uint64_t doMN = sdesc_sw128(smem_base + C::DO_OFF, C::CHUNK_BYTES, 1024);
    const uint64_t dsMN = sdesc_sw128(smem_base + C::DS_OFF, C::CHUNK_BYTES, 1024);
    const uint64_t qK[2] = {sdesc_sw128(smem_base + C::Q_OFF, 16, 1024),
                            sdesc_sw128(smem_base + C::Q_OFF + C::TILE_BYTES, 16, 1024)};
    const uint64_t qMN[2] = {sdesc_sw128(smem_base + C::Q_OFF, C::CHUNK_BYTES, 1024),
                             sdesc_sw128(smem_base + C::Q_OFF + C::TILE_BYTES, C::CHUNK_BYTES,
                                         1024)};
    const uint32_t tS = tmem + C::S_COL, tDP = tmem + C::DP_COL;
    const uint32_t tDV = tmem + C::DV_COL, tDK = tmem + C::DK_COL;
    // abort-path test: mma_done completes only after this warp's own final
    // commit, so this wait runs out of budget and the whole CTA aborts
    bool ok = !p.stall || blockIdx.x != 0 || wait(mma_done, 0);
    int g = 0;
    uint32_t kt = 0;
    for (int nt = 0; ok; ++nt) {
      BwdTile w;
      if (!bwd_read(ring, ring_bar, nt, w, ctl)) break;
      const int n = w.nqt;
      if (n == 0) continue;
      if (!wait(kv_full, kt & 1) || !wait(&q_full[g & 1], (g >> 1) & 1)) {
        ok = false;
        break;
      }
      tc_fence_after();
      bwd_mma_kk<D>(tS, kA, qK[g & 1], id_s, 0);  // S_0^T = K Q_0^T
      umma_commit_warp(s_full);
      for (int i = 0; i < n; ++i, ++g) {
        const int st = g & 1;
        // dP_i^T = V dO_i^T in two halves of 64 queries, each into columns the
        // previous dQ tile has left
        if (!wait(do_full, g & 1)) {
          ok = false;
          break;
        }
        if constexpr (C::DQ_OWN) {
          tc_fence_after();
          bwd_mma_kk<D>(tDP, vA, doK, id_s, 0);
          umma_commit_warp(&dp_full[0]);
          umma_commit_warp(&dp_full[1]);
        } else {
          for (int hq = 0; hq < 2; ++hq) {
            if (g > 0 && !wait(&dq_empty[hq], (g - 1) & 1)) {
              ok = false;
              break;
            }
            tc_fence_after();
            bwd_mma_kk<D>(tDP + 64 * hq, vA, doK + ((hq * 64 * 128) >> 4), id_s64, 0);
            umma_commit_warp(&dp_full[hq]);
          }
          if (!ok) break;
        }
        // dV += P_i^T dO_i  (P^T from TMEM, 16 queries = 8 packed columns per step)
        if (!wait(p_full, g & 1)) {
          ok = false;
          break;
        }
        tc_fence_after();
        // queries 16kk..16kk+15: packed columns (kk/4)*64 + (kk%4)*8 of S^T
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          umma_ts_warp(tDV, tS + (kk / 4) * 64 + (kk % 4) * 8, doMN + ((kk * 2048) >> 4), id_kv,
                       (i > 0 || kk > 0) ? 1u : 0u);
        umma_commit_warp(do_empty);
        // S_{i+1}^T (its columns held P_i, read by the MMAs just issued)
        if (i + 1 < n) {
          if (!wait(&q_full[(g + 1) & 1], ((g + 1) >> 1) & 1)) {
            ok = false;
            break;
          }
          tc_fence_after();
          bwd_mma_kk<D>(tS, kA, qK[(g + 1) & 1], id_s, 0);
          umma_commit_warp(s_full);
        }
        // dK += dS_i^T Q_i and dQ_i = dS_i K
        if (!wait(ds_full, g & 1)) {
          ok = false;
          break;
        }
        // the first dK of a key tile overwrites the previous tile's dK, which
        // the dQ warps must have read out
        if (i == 0 && kt > 0 && !wait(acc_empty, (kt - 1) & 1)) {
          ok = false;
          break;
        }
        tc_fence_after();
        // dS^T from TMEM: queries 16kk..16kk+15 are packed columns
        // (kk/4)*64 + (kk%4)*8 of the dP^T region
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          umma_ts_warp(tDK, tDP + (kk / 4) * 64 + (kk % 4) * 8, qMN[st] + ((kk * 2048) >> 4),
                       id_kv, (i > 0 || kk > 0) ? 1u : 0u);
        umma_commit_warp(&q_empty[st]);
        if constexpr (C::DQ_OWN) {
          // the previous dQ must have left its own columns
          if (g > 0 && (!wait(&dq_empty[0], (g - 1) & 1) || !wait(&dq_empty[1], (g - 1) & 1))) {
            ok = false;
            break;
          }
          tc_fence_after();
        }
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          umma_ss_warp(C::DQ_OWN ? tmem + C::DQ_COL : tDP, dsMN + ((kk * 2048) >> 4),
                       kMN + ((kk * 2048) >> 4), id_dq, kk > 0 ? 1u : 0u);
        umma_commit_warp(dq_full);
        umma_commit_warp(ds_empty);
      }
      if (!ok) break;
      // the key tile's last MMAs: dK and dV are final, K and V free
      umma_commit_warp(acc_full);
      umma_commit_warp(kv_empty);
      ++kt;
    }
    // every MMA issued must finish before TMEM and shared memory are released
    umma_commit_warp(mma_done);
    mbar_wait_drain(mma_done, 0, ctl);
  } else {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      tma_prefetch_desc(&tmDO);
    }
    __syncwarp();
    int nq_issued = 0, ndo_issued = 0;
    int g = 0;
    uint32_t kt = 0;  // K/V loads issued
    bool ok = true;
    // K and V of key tile w into their buffers
    auto load_kv = [&](const BwdTile& w) {
      const int krow = w.kv_base + w.kblk * C::BN;
      mbar_arrive_expect_tx_warp(kv_full, 2 * C::TILE_BYTES);
#pragma unroll
      for (int c = 0; c < C::NCHUNK; ++c) {
        tma_load_3d_warp(smem_base + C::K_OFF + c * C::CHUNK_BYTES, &tmK, smem_u32(kv_full),
                         c * 64, krow, w.plane);
        tma_load_3d_warp(smem_base + C::V_OFF + c * C::CHUNK_BYTES, &tmV, smem_u32(kv_full),
                         c * 64, krow, w.plane);
      }
      ++kt;
    };
    for (int nt = 0; ok; ++nt) {
      BwdTile w;
      const bool run = bwd_tile(p, sched_take(p.sched, nt), w);
      if (!bwd_publish(ring, ring_bar, nt, run, w, ctl) || !run) break;
      const int n = w.nqt;
      if (n == 0) continue;
      // the CTA's first key tile: nothing holds the K/V buffers yet; a later
      // tile loads them as soon as the previous tile's MMAs are done with them.
      // That load takes ~3 us, queued on the TMA unit behind the previous
      // tile's dQ reductions; L2 prefetches of K and V when the tile is taken
      // (bulk tensor or per-lane) did not shorten it and slowed the kernel.
      bool kv_loaded = false;
      if (kt == 0) {
        load_kv(w);
        kv_loaded = true;
      }
      for (int i = 0; i < n; ++i, ++g) {
        const int st = g & 1;
        const int q0 = (w.qt0 + i) * C::BM;
        // this tile's LSE (as -LSE*log2e) and -Delta, fetched before the stage is
        // free so that their latency hides behind the wait; columns past the
        // sequence get -inf and 0, so their P and dS are zero
        float nl[4], dl[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int q = q0 + lane * 4 + e;
          nl[e] = -INFINITY;
          dl[e] = 0.f;
          if (q < w.q_len) {
            const size_t gq = static_cast<size_t>(w.plane) * p.rows + w.q_base + q;
            nl[e] = -__ldg(p.lse + gq) * 1.4426950408889634f;
            dl[e] = -__ldg(p.delta + gq);
          }
        }
        if (!kv_loaded) {
          // K and V of a later key tile, as soon as the previous key tile's
          // MMAs are done with them: the first S and dP of this tile wait
          // for them, its first Q and dO tiles may follow
          if (!wait(kv_empty, (kt - 1) & 1)) {
            ok = false;
            break;
          }
          load_kv(w);
          kv_loaded = true;
        }
        if (g >= 2 && !wait(&q_empty[st], ((g >> 1) - 1) & 1)) {
          ok = false;
          break;
        }
        mbar_arrive_expect_tx_warp(&q_full[st], C::TILE_BYTES);
#pragma unroll
        for (int c = 0; c < C::NCHUNK; ++c)
          tma_load_3d_warp(smem_base + C::Q_OFF + st * C::TILE_BYTES + c * C::CHUNK_BYTES, &tmQ,
                           smem_u32(&q_full[st]), c * 64, w.q_base + q0, w.plane);
        float* sdst = stat + st * 256;
        *reinterpret_cast<float4*>(sdst + lane * 4) = make_float4(nl[0], nl[1], nl[2], nl[3]);
        *reinterpret_cast<float4*>(sdst + 128 + lane * 4) = make_float4(dl[0], dl[1], dl[2], dl[3]);
        mbar_arrive(&q_full[st]);
        ++nq_issued;
        if (g >= 1 && !wait(do_empty, (g - 1) & 1)) {
          ok = false;
          break;
        }
        mbar_arrive_expect_tx_warp(do_full, C::TILE_BYTES);
#pragma unroll
        for (int c = 0; c < C::NCHUNK; ++c)
          tma_load_3d_warp(smem_base + C::DO_OFF + c * C::CHUNK_BYTES, &tmDO, smem_u32(do_full),
                           c * 64, w.q_base + q0, w.plane);
        ++ndo_issued;
      }
    }
    // drain: every copy issued must land before the CTA may exit
    if (kt > 0) mbar_wait_drain(kv_full, (kt - 1) & 1, ctl);
    for (int i = max(0, nq_issued - 2); i < nq_issued; ++i)
      mbar_wait_drain(&q_full[i & 1], (i >> 1) & 1, ctl);
    if (ndo_issued > 0) mbar_wait_drain(do_full, (ndo_issued - 1) & 1, ctl);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 12) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
  if (threadIdx.x == 0) sched_done(p.sched);
}

// Delta_i = dO_i . O_i in fp32, and a zeroed dQ accumulator row; 16 threads per row.
template <int D, bool F16>
__global__ void __launch_bounds__(256) attn_bwd_prep_kernel(const BwdParams p, long long nrows) {
  constexpr int EPT = D / 16;  // elements per thread (8 or 4)
  const long long gid = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  const long long row = gid / 16;
  const int sub = static_cast<int>(gid % 16);
  const bool valid = row < nrows;
  float acc = 0.f;
  if (valid) {
    const uint16_t* o = static_cast<const uint16_t*>(p.o) + row * D + sub * EPT;
    const uint16_t* g = static_cast<const uint16_t*>(p.dout) + row * D + sub * EPT;
    uint32_t ov[4], gv[4];
    if constexpr (EPT == 8) {
      const uint4 a = *reinterpret_cast<const uint4*>(o);
      const uint4 b = *reinterpret_cast<const uint4*>(g);
      ov[0] = a.x; ov[1] = a.y; ov[2] = a.z; ov[3] = a.w;
      gv[0] = b.x; gv[1] = b.y; gv[2] = b.z; gv[3] = b.w;
    } else {
      const uint2 a = *reinterpret_cast<const uint2*>(o);
      const uint2 b = *reinterpret_cast<const uint2*>(g);
      ov[0] = a.x; ov[1] = a.y; ov[2] = 0u; ov[3] = 0u;
      gv[0] = b.x; gv[1] = b.y; gv[2] = 0u; gv[3] = 0u;
    }
#pragma unroll
    for (int e = 0; e < EPT / 2; ++e) {
      float o0, o1, g0, g1;
      if constexpr (F16) {
        const __half2 ho = *reinterpret_cast<const __half2*>(&ov[e]);
        const __half2 hg = *reinterpret_cast<const __half2*>(&gv[e]);
        o0 = __low2float(ho); o1 = __high2float(ho);
        g0 = __low2float(hg); g1 = __high2float(hg);
      } else {
        o0 = __uint_as_float(ov[e] << 16); o1 = __uint_as_float(ov[e] & 0xffff0000u);
        g0 = __uint_as_float(gv[e] << 16); g1 = __uint_as_float(gv[e] & 0xffff0000u);
      }
      acc = fmaf(o0, g0, acc);
      acc = fmaf(o1, g1, acc);
    }
    float4* z = reinterpret_cast<float4*>(p.dq_acc + row * D + sub * EPT);
#pragma unroll
    for (int e = 0; e < EPT / 4; ++e) z[e] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
#pragma unroll
  for (int o = 8; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
  if (valid && sub == 0) p.delta[row] = acc;
}

// dQ = scale * accumulator, rounded once; 8 elements per thread.
template <bool F16>
__global__ void __launch_bounds__(256) attn_bwd_dq_kernel(const BwdParams p, long long n8) {
  const long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= n8) return;
  const float4 a = reinterpret_cast<const float4*>(p.dq_acc)[2 * i];
  const float4 b = reinterpret_cast<const float4*>(p.dq_acc)[2 * i + 1];
  const float s = p.scale;
  reinterpret_cast<uint4*>(p.dq)[i] =
      make_uint4(pack_16x2<F16>(a.x * s, a.y * s), pack_16x2<F16>(a.z * s, a.w * s),
                 pack_16x2<F16>(b.x * s, b.y * s), pack_16x2<F16>(b.z * s, b.w * s));
}

}  // namespace attn
