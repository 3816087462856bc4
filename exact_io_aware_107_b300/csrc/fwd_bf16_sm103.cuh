// 16-bit (bf16 or fp16) attention forward for sm_103a: persistent CTAs, TMA +
// mbarrier pipeline, tcgen05 MMAs with TMEM accumulators, online softmax in
// base 2.  The element type only changes the MMA instruction descriptor, the
// TMA element type (set by the host) and the rounding of P and O.
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
// Queries and keys may differ in length (cross-attention, named in the same
// page's section "The Core Idea").  The causal mask then aligns the last query
// with the last key: key j is allowed for query i when j <= i + (Nk - Nq),
// which is j <= i when Nq == Nk.  A query with no allowed key (i < Nq - Nk)
// gets O = 0 and LSE = -inf.
//
// CTA layout (320 threads, one persistent CTA per SM):
//   warps 0-3  softmax and epilogue for query tile 0 (thread t owns row t =
//              TMEM lane t)
//   warps 4-7  softmax and epilogue for query tile 1
//   warp  8    tcgen05 MMA issuer (lane 0) and TMEM owner
//   warp  9    TMA producer (lane 0)
// A work tile is 256 query rows (two 128-row query tiles) of one (batch,
// head) plane or of one packed sequence of one head.  The TMA producer
// decodes each tile this CTA runs (the causal and packed layouts take work
// items from a counter of the launch as they go, the dense non-causal layout
// walks a static list) and hands it to the MMA and softmax warps through a
// small ring in shared memory.
//
// TMEM (512 columns x 128 lanes, fp32 cells):
//   [  0,128) S0 = Q0 K^T   (D = 128: P0 as packed bf16 overwrites its first 64 columns)
//   [128,256) S1 = Q1 K^T   (P1 likewise)
//   [256,256+D) O0, [256+D, 256+2D) O1
//   D = 64 (bf16) only: [384,448) P0, [448,512) P1.  With P in its own columns the MMA
//   warp issues S_i of the next key tile before P_i V of this one, so the
//   softmax waits only for the S MMAs; it then waits for that P V (p_free)
//   before it overwrites P_i or rescales O_i.  At D = 128 S_i of the next key
//   tile must follow P_i V, whose P it overwrites, and the commit after it
//   also covers that P V, so O_i is quiescent whenever S_i is ready.
//
// Shared memory (1024-byte aligned; every tile is 128 rows x D bf16 stored as
// D/64 chunks of 128 rows x 128 bytes, 128-byte swizzled, as TMA writes them):
//   Q0, Q1 (each with its own full/empty barriers, so the next work tile's
//   Q0 loads as soon as the last S0 of the current one is done), then NSTAGE
//   ring slots holding K_0, V_0, K_1, V_1, ... of every work tile in turn.
//   The producer issues the next tile's K_0 and V_0 before it waits for the
//   Q buffers, so a tile change costs little more than one Q load.
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
  void* o;                  // bf16 or fp16 output, same layout as q
  float* lse;
  const int* cu_seqlens;    // query offsets; nullptr for the dense layout
  const int* cu_seqlens_k;  // key offsets (packed layout only)
  int nseq;                 // packed layout: number of sequences
  int planes;               // dense: B*H; packed: H
  int rows;                 // query rows per plane (dense: Nq; packed: total query tokens)
  int rows_k;               // key rows per plane (dense: Nk; packed: total key tokens)
  int n_qblk;               // dense: ceil(Nq/256)
  int n_tiles;            // packed: an upper bound on the work items (block pairs)
  int tail_planes;        // dense causal: planes handed out as single blocks at the end
  int causal;
  float scale_log2;       // scale * log2(e)
  int stall;              // abort-path test: CTA 0 waits on a phase nothing completes
  unsigned long long timeout_ns;
  unsigned int* err;
  // Work counter of this launch (next item, CTAs finished), zero at launch
  // and reset to zero by the last CTA to finish; used by the causal and
  // packed layouts, whose work items are handed out in order to whichever
  // CTA asks first.
  unsigned int* sched;
};

// Depth of the shared-memory ring through which the TMA producer hands the
// work tiles it takes to the MMA and softmax warps.
constexpr int kItemRing = 4;

// Packed layouts with at most this many sequences take them longest first.
constexpr int kSortMaxSeq = 256;

template <int D>
struct Bf16Cfg {
  static constexpr int BM = 128;                  // query rows per tile
  static constexpr int BN = 128;                  // keys per K/V tile
  static constexpr int NSTAGE = (D == 128) ? 5 : 10;
  static constexpr int CHUNK_BYTES = BM * 128;    // 128 rows x 128 bytes
  static constexpr int NCHUNK = D / 64;
  static constexpr int TILE_BYTES = BM * D * 2;
  static constexpr int Q_OFF = 0;
  static constexpr int KV_OFF = 2 * TILE_BYTES;
  static constexpr int BAR_OFF = KV_OFF + NSTAGE * TILE_BYTES;
  // q_full[2], q_empty[2], kv_full[NSTAGE], kv_empty[NSTAGE], s_full[2], p_full[2],
  // o_full[2], mma_done, p_free[2], item_full[kItemRing], item_empty[kItemRing]
  static constexpr int NBAR = 4 + 2 * NSTAGE + 6 + 1 + 2 + 2 * kItemRing;
  static constexpr int ITEM_FULL_BAR = 4 + 2 * NSTAGE + 6 + 1 + 2;  // index in the barriers
  static constexpr int ITEM_EMPTY_BAR = ITEM_FULL_BAR + kItemRing;
  static constexpr int MISC_OFF = BAR_OFF + NBAR * 8;
  // the work tiles in flight (kItemRing slots of 48 bytes, 16-byte aligned)
  static constexpr int ITEM_OFF = (MISC_OFF + 16 + 15) / 16 * 16;
  // packed layout: the sequences in decreasing length (up to kSortMaxSeq of them)
  static constexpr int ORDER_OFF = ITEM_OFF + 48 * kItemRing;
  static constexpr int SMEM_BYTES = ORDER_OFF + 2 * kSortMaxSeq;
  static constexpr int SMEM_ALLOC = SMEM_BYTES + 1024;
  static constexpr int THREADS = 320;
  static constexpr uint32_t TMEM_COLS = 512;
  static constexpr uint32_t S_COL0 = 0, S_COL1 = 128;
  static constexpr uint32_t O_COL0 = 256, O_COL1 = 256 + D;
  // D = 64 leaves 128 columns free: P gets its own, so that the next S can be
  // issued before P V (SPLIT_P); at D = 128 P overwrites the first half of S.
  static constexpr bool SPLIT_P = (D == 64);
  static constexpr uint32_t P_COL0 = SPLIT_P ? 384 : S_COL0;
  static constexpr uint32_t P_COL1 = SPLIT_P ? 448 : S_COL1;
  static_assert(D == 64 || D == 128, "head dim");
  static_assert(SMEM_ALLOC <= 232448, "shared memory");
};

// One work tile: up to 256 query rows (two 128-row query tiles) of one plane
// or sequence.
struct WorkTile {
  int plane;     // tensor-map plane coordinate (dense: b*H+h; packed: h)
  int row_base;  // first query row of the sequence in the query map (0 when dense)
  int seq_len;   // query rows of the sequence
  int kv_base;   // first key row of the sequence in the key/value maps
  int kv_len;    // keys of the sequence
  int q0;        // first row of query tile 0 within the sequence (tile 1 follows it)
  bool has_q1;   // a second 128-row query tile follows
  int n0, n1;    // key tiles visited by query tile 0 and 1 (0: none, or tile absent)
};

// Cursor over packed sequences (in the order the schedule takes them); every
// CTA's list positions increase, so the walk over cu_seqlens only moves forward.
struct SeqCursor {
  int s = 0;
  int cum = 0;  // work items of the sequences before position s
};

// The packed sequences in decreasing length (ties by index) into order[]:
// each thread ranks some of them against all.  The comparison is a strict
// total order, so the ranks are a permutation whatever cu_seqlens holds (a
// malformed array is caught later, when the walk reads the entry).
__device__ __forceinline__ void bf16_sort_sequences(const Bf16Params& p, uint16_t* order) {
  for (int s = threadIdx.x; s < p.nseq; s += blockDim.x) {
    const int len = __ldg(p.cu_seqlens + s + 1) - __ldg(p.cu_seqlens + s);
    int rank = 0;
    for (int t = 0; t < p.nseq; ++t) {
      const int lt = __ldg(p.cu_seqlens + t + 1) - __ldg(p.cu_seqlens + t);
      rank += (lt > len) || (lt == len && t < s);
    }
    order[rank] = static_cast<uint16_t>(s);
  }
}

enum TileStep { kTileEnd = 0, kTileRun = 1, kTileSkip = 2 };

// The query-tile geometry of w once its plane, rows and q0 are set: the key
// tiles each of its two query tiles visits (causal: up to the last key its
// last row may see).  A query tile whose rows see no key at all has n_i == 0:
// no loads and no MMAs, its softmax warps write O = 0 and LSE = -inf directly.
__device__ __forceinline__ int bf16_geometry(const Bf16Params& p, WorkTile& w, bool single) {
  const int nkv = (w.kv_len + 127) / 128;
  const int off = w.kv_len - w.seq_len;
  auto visited = [&](int q0) {
    if (!p.causal) return nkv;
    const int last = min(q0 + 127, w.seq_len - 1) + off;
    return last < 0 ? 0 : min(nkv, last / 128 + 1);
  };
  w.has_q1 = !single && w.q0 + 128 < w.seq_len;
  w.n0 = visited(w.q0);
  w.n1 = w.has_q1 ? visited(w.q0 + 128) : 0;
  return kTileRun;
}

// Dense non-causal layout, a static schedule: every 256-row block costs the
// same, so the list holds single blocks, plane-major, one round of gridDim.x
// per iteration.  When the last round is at most half full, its blocks are
// split into single 128-row query tiles, one per CTA, so that the last round
// takes about half as long.  Returns the it-th tile of this CTA, or kTileEnd.
__device__ __forceinline__ int bf16_tile_static(const Bf16Params& p, int it, WorkTile& w) {
  const int grid = static_cast<int>(gridDim.x);
  const int c = static_cast<int>(blockIdx.x);
  w.row_base = 0;
  w.seq_len = p.rows;
  w.kv_base = 0;
  w.kv_len = p.rows_k;
  const int nblk = p.planes * p.n_qblk;
  const int full = nblk / grid;  // rounds with a block for every CTA
  const int rem = nblk - full * grid;
  bool single = false;
  int u;
  if (it < full) {
    u = it * grid + c;
  } else {
    if (it > full || rem == 0) return kTileEnd;
    single = 2 * rem <= grid;
    if (c >= (single ? 2 * rem : rem)) return kTileEnd;
    u = full * grid + (single ? c / 2 : c);
  }
  w.plane = u / p.n_qblk;
  w.q0 = (u - w.plane * p.n_qblk) * 256 + (single ? 128 * (c & 1) : 0);
  if (w.q0 >= w.seq_len) return kTileEnd;  // the second tile of a short last block
  return bf16_geometry(p, w, single);
}

// Work item u of the causal dense and the packed layouts; half h = 0 is its
// first (heavier) 256-row block, h = 1 its second, if any.  The items are
// handed out in list order to whichever CTA asks first, and the list runs
// from heavy to light, so the CTAs end within about one light item of each
// other.
//
// Dense causal: pairs of 256-row blocks of one plane, block b with its mirror
// n-1-b, so that every pair costs the same under the causal mask; pairs are
// plane-major (the CTAs in flight share few planes and their K/V stay in
// L2).  The last tail_planes planes (about one round of pairs) come as single
// blocks instead, heaviest first (block n-1 of each of those planes, then
// block n-2, ...), which fills the last round evenly.
//
// Packed: pairs of mirror blocks within one sequence of one head, the pairs
// of a (sequence, head) consecutive (its K/V stays in L2), the heads of a
// sequence next, and the sequences longest first (order[], when the kernel
// could sort them; else as given), so that the pairs, whose cost grows with
// the sequence length, come in decreasing cost.  A CTA's items come in
// increasing u, so its walk over cu_seqlens (cur) only moves forward.
//
// Returns kTileEnd past the last item (or when cu_seqlens is malformed) and
// kTileSkip for a half that does not exist.
__device__ __forceinline__ int bf16_item(const Bf16Params& p, const uint16_t* order, int u, int h,
                                         SeqCursor& cur, WorkTile& w) {
  if (p.cu_seqlens == nullptr) {
    w.row_base = 0;
    w.seq_len = p.rows;
    w.kv_base = 0;
    w.kv_len = p.rows_k;
    const int npp = (p.n_qblk + 1) / 2;  // pairs per plane
    const int pair_planes = p.planes - p.tail_planes;
    const int n_pairs = pair_planes * npp;
    if (u < n_pairs) {
      w.plane = u / npp;
      const int pb = u - w.plane * npp;
      const int heavy = p.n_qblk - 1 - pb;
      if (h) {
        if (pb == heavy) return kTileSkip;
        w.q0 = pb * 256;
      } else {
        w.q0 = heavy * 256;
      }
    } else {
      const int v = u - n_pairs;
      if (v >= p.tail_planes * p.n_qblk) return kTileEnd;
      if (h) return kTileSkip;
      w.plane = pair_planes + v % p.tail_planes;
      w.q0 = (p.n_qblk - 1 - v / p.tail_planes) * 256;
    }
    return bf16_geometry(p, w, false);
  }
  if (u >= p.n_tiles) return kTileEnd;
  while (cur.s < p.nseq) {
    const int sq = order ? static_cast<int>(order[cur.s]) : cur.s;
    const int a = __ldg(p.cu_seqlens + sq), e = __ldg(p.cu_seqlens + sq + 1);
    if (a < 0 || e < a || e > p.rows) {
      if ((threadIdx.x % 32) == 0) atomicOr(p.err, kDevErrBounds);
      return kTileEnd;
    }
    const int nb = (e - a + 255) / 256;
    const int npp = (nb + 1) / 2;
    if (u < cur.cum + npp * p.planes) {
      const int ak = __ldg(p.cu_seqlens_k + sq), ek = __ldg(p.cu_seqlens_k + sq + 1);
      if (ak < 0 || ek < ak || ek > p.rows_k) {
        if ((threadIdx.x % 32) == 0) atomicOr(p.err, kDevErrBounds);
        return kTileEnd;
      }
      const int r = u - cur.cum;
      w.plane = r / npp;
      const int pb = r - w.plane * npp;
      const int heavy = nb - 1 - pb;
      if (h) {
        if (pb == heavy) return kTileSkip;
        w.q0 = pb * 256;
      } else {
        w.q0 = heavy * 256;
      }
      w.row_base = a;
      w.seq_len = e - a;
      w.kv_base = ak;
      w.kv_len = ek - ak;
      return bf16_geometry(p, w, false);
    }
    cur.cum += npp * p.planes;
    ++cur.s;
  }
  return kTileEnd;
}

// The producer's walk over the work tiles.
struct TileWalk {
  int k = 0;     // items (static schedule: iterations) taken so far
  int u = 0;     // current item
  int half = 2;  // next half of the current item (2: take a new item)
  SeqCursor cur;
};

// Next work tile of this CTA, decoded by the TMA producer warp (a
// warp-uniform call).  Static schedule: the next tile of the list.  Item
// schedule: the halves of the current item, then a new item: the CTA's first
// is blockIdx.x, every later one the next free position of the launch's
// counter (past the first gridDim.x).  kTileSkip marks a half that does not
// exist.
__device__ __forceinline__ int bf16_take(const Bf16Params& p, const uint16_t* order,
                                         TileWalk& src, WorkTile& w) {
  if (p.sched == nullptr) return bf16_tile_static(p, src.k++, w);
  if (src.half == 2) {
    src.u = sched_take(p.sched, src.k++);
    src.half = 0;
  }
  return bf16_item(p, order, src.u, src.half++, src.cur, w);
}

// The tiles the producer takes reach the MMA and softmax warps through a ring
// of kItemRing slots in shared memory: a slot holds the tile (or the end of
// the walk) as twelve 32-bit words, item_full[slot] completes when it is
// written, item_empty[slot] when all nine readers have copied it.  Addresses
// are 32-bit shared-memory addresses: the ring's first slot and the first
// item_full barrier (the item_empty barriers follow them).
constexpr uint32_t kItemSlotBytes = 48;

// Producer: publish the n-th tile (step is kTileRun or kTileEnd).
__device__ __forceinline__ bool bf16_publish(uint32_t ring, uint32_t full, int n, int step,
                                             const WorkTile& w, const WaitCtl& ctl) {
  const uint32_t slot = static_cast<uint32_t>(n % kItemRing);
  const uint32_t lap = static_cast<uint32_t>(n / kItemRing);
  const uint32_t empty = full + 8 * kItemRing;
  if (lap > 0 && !__all_sync(0xffffffffu, mbar_wait_at(empty + 8 * slot, (lap - 1) & 1, ctl)))
    return false;
  if ((threadIdx.x % 32) == 0) {
    const uint32_t a = ring + kItemSlotBytes * slot;
    st_shared_v4(a, step, w.plane, w.row_base, w.seq_len);
    st_shared_v4(a + 16, w.kv_base, w.kv_len, w.q0, w.has_q1 ? 1 : 0);
    st_shared_v4(a + 32, w.n0, w.n1, 0, 0);
    mbar_arrive_at(full + 8 * slot);  // release: the slot's contents are visible to its readers
  }
  __syncwarp();
  return true;
}

// Reader (MMA or softmax warp, warp-uniform): the n-th tile; kTileEnd at the
// end of the walk or when the CTA is aborting.
template <bool kRelease = true>
__device__ __forceinline__ int bf16_read(uint32_t ring, uint32_t full, int n, WorkTile& w,
                                         const WaitCtl& ctl) {
  const uint32_t slot = static_cast<uint32_t>(n % kItemRing);
  const uint32_t lap = static_cast<uint32_t>(n / kItemRing);
  if (!__all_sync(0xffffffffu, mbar_wait_at(full + 8 * slot, lap & 1, ctl))) return kTileEnd;
  const uint32_t a = ring + kItemSlotBytes * slot;
  uint32_t r0[4], r1[4], r2[4];
  ld_shared_v4(a, r0);
  ld_shared_v4(a + 16, r1);
  ld_shared_v4(a + 32, r2);
  w.plane = static_cast<int>(r0[1]);
  w.row_base = static_cast<int>(r0[2]);
  w.seq_len = static_cast<int>(r0[3]);
  w.kv_base = static_cast<int>(r1[0]);
  w.kv_len = static_cast<int>(r1[1]);
  w.q0 = static_cast<int>(r1[2]);
  w.has_q1 = r1[3] != 0;
  w.n0 = static_cast<int>(r2[0]);
  w.n1 = static_cast<int>(r2[1]);
  if (kRelease) {
    __syncwarp();
    if ((threadIdx.x % 32) == 0) mbar_arrive_at(full + 8 * kItemRing + 8 * slot);
  }
  return static_cast<int>(r0[0]);
}

// A reader that keeps its slot until the end of the tile (the softmax warps,
// whose registers are scarcest) reads the plane, first row and length of the
// tile again from it when it writes O, instead of holding them in registers
// through the key loop, and releases the slot when it takes the next tile.
// Words of a slot: 0 step, 1 plane, 2 row_base, 3 seq_len, 4 kv_base,
// 5 kv_len, 6 q0, 7 has_q1, 8 n0, 9 n1.
__device__ __forceinline__ uint32_t bf16_slot_word(uint32_t ring, int n, int word) {
  uint32_t v;
  asm volatile("ld.shared.u32 %0, [%1];"
               : "=r"(v)
               : "r"(ring + kItemSlotBytes * static_cast<uint32_t>(n % kItemRing) + 4 * word)
               : "memory");
  return v;
}
__device__ __forceinline__ void bf16_release(uint32_t full, int n) {
  __syncwarp();
  if ((threadIdx.x % 32) == 0)
    mbar_arrive_at(full + 8 * kItemRing + 8 * static_cast<uint32_t>(n % kItemRing));
}

// S = Q K^T for one 128x128 tile: D/16 MMAs of K=16.  q_desc/k_desc are the
// descriptors of the tiles' first bytes; the start-address field (bits 0-13,
// bytes / 16) is advanced in place, which cannot carry out of the field
// because shared addresses stay below 256 KB.
template <int D, bool F16>
__device__ __forceinline__ void bf16_issue_s(uint32_t d_tmem, uint64_t q_desc, uint64_t k_desc) {
  using C = Bf16Cfg<D>;
  constexpr uint32_t idesc = idesc_bf16_f32(128, C::BN, 0, 0, F16);
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk) {
    const uint32_t off = ((kk / 4) * C::CHUNK_BYTES + (kk % 4) * 32) >> 4;
    umma_ss_warp(d_tmem, q_desc + off, k_desc + off, idesc, kk > 0 ? 1u : 0u);
  }
}

// O (+)= P V: P (bf16 pairs) from TMEM columns p_tmem.., V tile from v_desc.
template <int D, bool F16>
__device__ __forceinline__ void bf16_issue_pv(uint32_t d_tmem, uint32_t p_tmem, uint64_t v_desc,
                                              uint32_t accumulate) {
  using C = Bf16Cfg<D>;
  constexpr uint32_t idesc = idesc_bf16_f32(128, D, 0, 1, F16);
#pragma unroll
  for (int kk = 0; kk < C::BN / 16; ++kk) {
    // V is the MN-major B operand: 16 keys = two 8-row groups of 128-byte rows
    umma_ts_warp(d_tmem, p_tmem + kk * 8, v_desc + ((kk * 16 * 128) >> 4), idesc,
                 (accumulate || kk > 0) ? 1u : 0u);
  }
}

template <int D, bool F16>
__global__ void __launch_bounds__(320, 1)
    attn_fwd_bf16_kernel(const __grid_constant__ CUtensorMap tmQ,
                         const __grid_constant__ CUtensorMap tmK,
                         const __grid_constant__ CUtensorMap tmV, const Bf16Params p) {
  using C = Bf16Cfg<D>;
  constexpr int NS = C::NSTAGE;
  // P in its own columns at D = 64 for bf16; the fp16 build of that layout
  // spills registers at the 168-register cap and runs 6 % slower, so fp16
  // keeps P in its S columns
  constexpr bool kSplitP = C::SPLIT_P && !F16;
  constexpr uint32_t kPCol0 = kSplitP ? C::P_COL0 : C::S_COL0;
  constexpr uint32_t kPCol1 = kSplitP ? C::P_COL1 : C::S_COL1;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::BAR_OFF);
  uint64_t* q_full = bars;          // [2]
  uint64_t* q_empty = bars + 2;     // [2]
  uint64_t* kv_full = bars + 4;     // [NS]
  uint64_t* kv_empty = kv_full + NS;
  uint64_t* s_full = kv_empty + NS;  // [2]
  uint64_t* p_full = s_full + 2;     // [2]
  uint64_t* o_full = p_full + 2;     // [2]
  uint64_t* mma_done = o_full + 2;
  uint64_t* p_free = mma_done + 1;   // [2] (kSplitP: the P V of the last P is complete)
  uint64_t* item_full = bars + C::ITEM_FULL_BAR;  // [kItemRing]
  uint64_t* item_empty = bars + C::ITEM_EMPTY_BAR;  // [kItemRing]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::MISC_OFF);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::MISC_OFF + 4);

  // packed layout: every role walks the sequences in the same order
  uint16_t* order = nullptr;
  if (p.cu_seqlens != nullptr && p.nseq <= kSortMaxSeq) {
    order = reinterpret_cast<uint16_t*>(smem + C::ORDER_OFF);
    bf16_sort_sequences(p, order);
    __syncthreads();
  }
  {
    SeqCursor c0;
    WorkTile w0;
    const int first = p.sched ? bf16_item(p, order, static_cast<int>(blockIdx.x), 0, c0, w0)
                              : bf16_tile_static(p, 0, w0);
    if (first != kTileRun) {  // uniform: no work for this CTA
      if (p.sched && threadIdx.x == 0) sched_done(p.sched);
      return;
    }
  }

  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;

  if (threadIdx.x == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(&q_full[i], 1);
      mbar_init(&q_empty[i], 1);
      mbar_init(&s_full[i], 1);
      mbar_init(&p_full[i], 128);
      mbar_init(&o_full[i], 1);
      mbar_init(&p_free[i], 1);
    }
    for (int s = 0; s < NS; ++s) {
      mbar_init(&kv_full[s], 1);
      mbar_init(&kv_empty[s], 1);
    }
    mbar_init(mma_done, 1);
    for (int i = 0; i < kItemRing; ++i) {
      mbar_init(&item_full[i], 1);
      mbar_init(&item_empty[i], 9);  // the eight softmax warps and the MMA warp
    }
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
  const uint32_t smem_base = smem_u32(smem);
  const uint32_t item_ring = smem_base + C::ITEM_OFF;
  const uint32_t item_bar = smem_base + C::BAR_OFF + 8 * C::ITEM_FULL_BAR;
  int n_tile = 0;  // work tiles read (MMA and softmax warps) or published (producer)

  if (warp < 8) {
    // ------------------------------------------------------------ softmax
    const int ti = warp / 4;               // query tile of this warpgroup
    const int t = threadIdx.x - 128 * ti;  // row within the tile
    const uint32_t lane_off = static_cast<uint32_t>(32 * (warp % 4)) << 16;
    const uint32_t tS = tmem + lane_off + (ti ? C::S_COL1 : C::S_COL0);
    const uint32_t tO = tmem + lane_off + (ti ? C::O_COL1 : C::O_COL0);
    const uint32_t tP = tmem + lane_off + (ti ? kPCol1 : kPCol0);
    uint32_t n_pst = 0;  // P tiles stored by this warpgroup so far (kSplitP)
    const float cl2 = p.scale_log2;
    const uint64_t c2 = f32x2(cl2, cl2);
    uint32_t n_s = 0, n_o = 0;  // s_full / o_full phases consumed so far
    WorkTile w;
    for (;; ++n_tile) {
      if (n_tile > 0) bf16_release(item_bar, n_tile - 1);
      const int step = bf16_read<false>(item_ring, item_bar, n_tile, w, ctl);
      if (step == kTileEnd) break;
      if (step == kTileSkip || (ti == 1 && !w.has_q1)) continue;
      const int n_i = ti ? w.n1 : w.n0;
      const int q_first = w.q0 + 128 * ti;  // first row of this query tile
      const int row = q_first + t;
      const int off = w.kv_len - w.seq_len;         // causal alignment of queries to keys
      if (n_i == 0) {
        // every row of this tile sees no key
        if (row < static_cast<int>(bf16_slot_word(item_ring, n_tile, 3))) {
          const size_t grow = static_cast<size_t>(bf16_slot_word(item_ring, n_tile, 1)) * p.rows +
                              bf16_slot_word(item_ring, n_tile, 2) + row;
          uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.o) + grow * D);
#pragma unroll
          for (int v = 0; v < D / 8; ++v) dst[v] = make_uint4(0u, 0u, 0u, 0u);
          p.lse[grow] = -INFINITY;
        }
        continue;
      }
      float m_ref = -INFINITY;
      float l = 0.f;    // row sum of the probabilities (for LSE)
      float l_o = 0.f;  // the same with each tile's largest term as rounded (for O)
      bool ok = true;
      for (int j = 0; j < n_i; ++j) {
        // warp-uniform outcome: the TMEM loads below are warp-collective
        if (!__all_sync(0xffffffffu, mbar_wait(&s_full[ti], n_s & 1, ctl))) {
          ok = false;
          break;
        }
        ++n_s;
        tc_fence_after();
        uint32_t sr[128];
        tmem_ld128_wait(tS, sr);
        const int kv0 = j * C::BN;
        const bool need_mask =
            (kv0 + C::BN > w.kv_len) || (p.causal && kv0 + C::BN - 1 > q_first + off);
        if (need_mask) {
          const int lim = p.causal ? min(w.kv_len - 1, row + off) : (w.kv_len - 1);
#pragma unroll
          for (int c = 0; c < 128; ++c)
            if (kv0 + c > lim) sr[c] = __float_as_uint(-INFINITY);
        }
        const float mraw = row_max<128>(sr);
        const float mt = mraw * cl2;
        if constexpr (kSplitP) {
          // The S just loaded was issued before the P V of the previous key
          // tile: that P V must be complete before its P columns are
          // overwritten and O is rescaled (it has had the load's latency to
          // finish, so this rarely waits).
          if (n_pst > 0 && !__all_sync(0xffffffffu, mbar_wait(&p_free[ti], (n_pst - 1) & 1, ctl))) {
            ok = false;
            break;
          }
          ++n_pst;
          tc_fence_after();
        }
        float m_new = m_ref;
        float alpha = 1.f;
        bool resc = false;
        if (mt > m_ref + 8.f) {
          m_new = mt;
          alpha = ex2_approx(m_ref - m_new);
          resc = (j > 0);
        }
        const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
        const uint64_t nm2 = f32x2(-m_use, -m_use);
        // The tile's largest probability, computed exactly as the loop below
        // computes it, and the error its rounding to 16 bits makes.  O is
        // divided by the row sum corrected by these errors, so that the term
        // that dominates a peaked row enters numerator and denominator alike
        // (its P can be up to 2^8 under the lazy rescale, and a relative 2^-8
        // on it would otherwise move O by up to 2^-8 |V|); LSE keeps the sum
        // of the unrounded probabilities.
        const float pmx = ex2_approx(fmaf(mraw, cl2, -m_use));
        const float pmx_err = lo_f32(unpack_16x2<F16>(pack_16x2<F16>(pmx, 0.f))) - pmx;
        uint64_t acc2[2] = {0ull, 0ull};
        uint32_t pk[64];
#pragma unroll
        for (int c = 0; c < 64; ++c) {
          const uint64_t x2 = ffma2(u32x2(sr[2 * c], sr[2 * c + 1]), c2, nm2);
          const float a = ex2_approx(lo_f32(x2));
          const float b = ex2_approx(hi_f32(x2));
          acc2[c & 1] = fadd2(acc2[c & 1], f32x2(a, b));
          pk[c] = pack_16x2<F16>(a, b);
        }
        const uint64_t sum2 = fadd2(acc2[0], acc2[1]);
        const float tile_sum = lo_f32(sum2) + hi_f32(sum2);
        l = l * alpha + tile_sum;
        l_o = l_o * alpha + (tile_sum + pmx_err);
        tmem_st32(tP, *reinterpret_cast<uint32_t(*)[32]>(&pk[0]));
        tmem_st32(tP + 32, *reinterpret_cast<uint32_t(*)[32]>(&pk[32]));
        if (__any_sync(0xffffffffu, resc)) {
          const float f = resc ? alpha : 1.f;
          const uint64_t f2 = f32x2(f, f);
#pragma unroll
          for (int cc = 0; cc < D / 32; ++cc) {
            uint32_t o[32];
            tmem_ld32_wait(tO + 32 * cc, o);
#pragma unroll
            for (int e = 0; e < 16; ++e) {
              const uint64_t v = fmul2(u32x2(o[2 * e], o[2 * e + 1]), f2);
              o[2 * e] = static_cast<uint32_t>(v);
              o[2 * e + 1] = static_cast<uint32_t>(v >> 32);
            }
            tmem_st32(tO + 32 * cc, o);
          }
        }
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(&p_full[ti]);
        m_ref = m_new;
      }
      if (!ok || !__all_sync(0xffffffffu, mbar_wait(&o_full[ti], n_o & 1, ctl))) break;
      ++n_o;
      tc_fence_after();
      const bool valid = row < static_cast<int>(bf16_slot_word(item_ring, n_tile, 3));
      const size_t grow = static_cast<size_t>(bf16_slot_word(item_ring, n_tile, 1)) * p.rows +
                          bf16_slot_word(item_ring, n_tile, 2) + row;
      // l == 0 only for a row that saw no allowed key: O = 0, LSE = -inf
      const float inv_l = (l > 0.f) ? 1.f / l_o : 0.f;
      uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.o) + grow * D);
#pragma unroll
      for (int cc = 0; cc < D / 32; ++cc) {
        uint32_t o[32];
        tmem_ld32_wait(tO + 32 * cc, o);
        uint32_t h[16];
#pragma unroll
        for (int e = 0; e < 16; ++e)
          h[e] = pack_16x2<F16>(__uint_as_float(o[2 * e]) * inv_l,
                                __uint_as_float(o[2 * e + 1]) * inv_l);
        if (valid) {
#pragma unroll
          for (int v = 0; v < 4; ++v)
            dst[cc * 4 + v] = make_uint4(h[4 * v], h[4 * v + 1], h[4 * v + 2], h[4 * v + 3]);
        }
      }
      if (valid) p.lse[grow] = (l > 0.f) ? (m_ref + log2f(l)) * 0.69314718055994530942f : -INFINITY;
    }
  } else if (warp == 8) {
    // ------------------------------------------------------------ MMA issuer
    // The whole warp runs this loop so every operand is warp-uniform; one
    // elected lane issues each tcgen05 instruction.
    const uint64_t qd[2] = {sdesc_sw128(smem_base + C::Q_OFF, 16, 1024),
                            sdesc_sw128(smem_base + C::Q_OFF + C::TILE_BYTES, 16, 1024)};
    const uint64_t kd0 = sdesc_sw128(smem_base + C::KV_OFF, 16, 1024);
    const uint64_t vd0 = sdesc_sw128(smem_base + C::KV_OFF, C::CHUNK_BYTES, 1024);
    constexpr uint32_t kSlotDesc = C::TILE_BYTES >> 4;  // descriptor step between ring slots
    uint32_t n_q[2] = {0, 0}, n_p[2] = {0, 0};
    int g = 0;  // ring position of the tile's K_0
    bool ok = true;
    WorkTile w;
    auto wait = [&](uint64_t* bar, uint32_t parity) {
      return __all_sync(0xffffffffu, mbar_wait(bar, parity, ctl));
    };
    // abort-path test: mma_done completes only after this warp's own final
    // commit, so this wait runs out of budget and the whole CTA aborts
    if (p.stall && blockIdx.x == 0) ok = wait(mma_done, 0);
    while (ok) {
      const int step = bf16_read(item_ring, item_bar, n_tile++, w, ctl);
      if (step == kTileEnd) break;
      if (step == kTileSkip) continue;
      const int nmax = max(w.n0, w.n1);
      if (nmax == 0) continue;  // no key for either query tile
      if (!wait(&kv_full[g % NS], (g / NS) & 1)) {
        ok = false;
        break;
      }
      const uint64_t k0 = kd0 + (g % NS) * kSlotDesc;
      for (int ti = 0; ti < 2; ++ti) {
        const int n_i = ti ? w.n1 : w.n0;
        if (n_i == 0) continue;
        if (!wait(&q_full[ti], n_q[ti] & 1)) {
          ok = false;
          break;
        }
        ++n_q[ti];
        tc_fence_after();
        bf16_issue_s<D, F16>(tmem + (ti ? C::S_COL1 : C::S_COL0), qd[ti], k0);
        umma_commit_warp(&s_full[ti]);
        if (n_i == 1) umma_commit_warp(&q_empty[ti]);
      }
      if (!ok) break;
      umma_commit_warp(&kv_empty[g % NS]);
      for (int j = 0; j < nmax; ++j) {
        const int gv = g + 2 * j + 1, gk = g + 2 * j + 2;
        const bool next = j + 1 < nmax;
        if (!wait(&kv_full[gv % NS], (gv / NS) & 1) ||
            (next && !wait(&kv_full[gk % NS], (gk / NS) & 1))) {
          ok = false;
          break;
        }
        tc_fence_after();
        for (int ti = 0; ti < 2; ++ti) {
          const int n_i = ti ? w.n1 : w.n0;
          if (j >= n_i) continue;
          if (!wait(&p_full[ti], n_p[ti] & 1)) {
            ok = false;
            break;
          }
          ++n_p[ti];
          tc_fence_after();
          const uint32_t sc = ti ? C::S_COL1 : C::S_COL0;
          const uint32_t oc = ti ? C::O_COL1 : C::O_COL0;
          const uint32_t pc = ti ? kPCol1 : kPCol0;
          if constexpr (kSplitP) {
            // S of the next key tile first: the softmax waits for it, while
            // this P V runs behind it
            if (j + 1 < n_i) {
              bf16_issue_s<D, F16>(tmem + sc, qd[ti], kd0 + (gk % NS) * kSlotDesc);
              umma_commit_warp(&s_full[ti]);
              if (j + 2 == n_i) umma_commit_warp(&q_empty[ti]);  // that was the last S of Q_ti
            }
            bf16_issue_pv<D, F16>(tmem + oc, tmem + pc, vd0 + (gv % NS) * kSlotDesc,
                                  j > 0 ? 1u : 0u);
            umma_commit_warp(&p_free[ti]);
            if (ti == ((j < w.n1) ? 1 : 0)) umma_commit_warp(&kv_empty[gv % NS]);
            if (j + 1 >= n_i) umma_commit_warp(&o_full[ti]);
          } else {
            bf16_issue_pv<D, F16>(tmem + oc, tmem + pc, vd0 + (gv % NS) * kSlotDesc,
                                  j > 0 ? 1u : 0u);
            // V_j is free for the producer as soon as its last reader is done
            if (ti == ((j < w.n1) ? 1 : 0)) umma_commit_warp(&kv_empty[gv % NS]);
            if (j + 1 < n_i) {
              bf16_issue_s<D, F16>(tmem + sc, qd[ti], kd0 + (gk % NS) * kSlotDesc);
              umma_commit_warp(&s_full[ti]);
              if (j + 2 == n_i) umma_commit_warp(&q_empty[ti]);  // that was the last S of Q_ti
            } else {
              umma_commit_warp(&o_full[ti]);
            }
          }
        }
        if (!ok) break;
        if (next) umma_commit_warp(&kv_empty[gk % NS]);
      }
      g += 2 * nmax;
    }
    // every MMA issued so far must finish before TMEM and shared memory are released
    umma_commit_warp(mma_done);
    mbar_wait_drain(mma_done, 0, ctl);
  } else {
    // ------------------------------------------------------------ TMA producer
    // Whole warp, one elected lane issues (operands stay warp-uniform).
    if (lane == 0) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
    }
    __syncwarp();
    uint32_t n_q[2] = {0, 0};
    int g = 0;  // ring positions issued
    bool ok = true;
    WorkTile w;
    auto wait = [&](uint64_t* bar, uint32_t parity) {
      return __all_sync(0xffffffffu, mbar_wait(bar, parity, ctl));
    };
    const uint32_t kv_smem = smem_base + C::KV_OFF;
    // one K or V tile into the next ring slot
    auto load_kv = [&](int t) -> bool {
      const int s = g % NS, u = g / NS;
      if (u > 0 && !wait(&kv_empty[s], (u - 1) & 1)) return false;
      mbar_arrive_expect_tx_warp(&kv_full[s], C::TILE_BYTES);
#pragma unroll
      for (int c = 0; c < C::NCHUNK; ++c)
        tma_load_3d_warp(kv_smem + s * C::TILE_BYTES + c * C::CHUNK_BYTES, (t & 1) ? &tmV : &tmK,
                         smem_u32(&kv_full[s]), c * 64, w.kv_base + (t >> 1) * C::BN, w.plane);
      ++g;
      return true;
    };
    TileWalk walk;
    while (ok) {
      const int step = bf16_take(p, order, walk, w);
      if (step == kTileSkip) continue;
      ok = bf16_publish(item_ring, item_bar, n_tile++, step, w, ctl);
      if (step == kTileEnd) break;
      const int nkv = 2 * max(w.n0, w.n1);
      // K_0 and V_0 first: their slots are freed by the previous tile alone
      const int head = min(2, nkv);
      for (int t = 0; ok && t < head; ++t) ok = load_kv(t);
      for (int ti = 0; ok && ti < 2; ++ti) {
        if ((ti ? w.n1 : w.n0) == 0) continue;
        if (n_q[ti] > 0 && !wait(&q_empty[ti], (n_q[ti] - 1) & 1)) {
          ok = false;
          break;
        }
        mbar_arrive_expect_tx_warp(&q_full[ti], C::TILE_BYTES);
#pragma unroll
        for (int c = 0; c < C::NCHUNK; ++c)
          tma_load_3d_warp(smem_base + C::Q_OFF + ti * C::TILE_BYTES + c * C::CHUNK_BYTES, &tmQ,
                           smem_u32(&q_full[ti]), c * 64, w.row_base + w.q0 + 128 * ti,
                           w.plane);
        ++n_q[ti];
      }
      for (int t = head; ok && t < nkv; ++t) ok = load_kv(t);
    }
    // drain: every copy issued must land before the CTA may exit
    for (int ti = 0; ti < 2; ++ti)
      if (n_q[ti] > 0) mbar_wait_drain(&q_full[ti], (n_q[ti] - 1) & 1, ctl);
    for (int t = max(0, g - NS); t < g; ++t)
      mbar_wait_drain(&kv_full[t % NS], (t / NS) & 1, ctl);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 8) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
  if (p.sched && threadIdx.x == 0) sched_done(p.sched);
}

}  // namespace attn
