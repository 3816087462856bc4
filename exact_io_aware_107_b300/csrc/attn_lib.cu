// C ABI of the attention forward: argument checks, TMA descriptors, launches.
//
// One translation unit holds the device error word and every kernel, so the
// library needs no relocatable device code.
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <algorithm>
#include <mutex>

#include "../../include/attn_b300.h"
#include "bwd_bf16_sm103.cuh"
#include "decode_bf16.cuh"
#include "fwd_bf16_sm103.cuh"
#include "fwd_f32.cuh"
#include "ptx.cuh"

namespace attn {

__device__ unsigned int g_dev_error;

// Work counters of the persistent kernels (the forward's causal and packed
// schedules, the backward): a launch takes the next of kSchedSlots slots (two
// words each, padded to 32 bytes), which every launch leaves at zero when its
// last CTA ends.  Launches in flight at the same time use different slots
// unless kSchedSlots of them are; replays of one captured launch reuse its
// slot and must not overlap.
constexpr int kSchedSlots = 256;
constexpr int kSchedStride = 8;  // words per slot
__device__ unsigned int g_sched[kSchedSlots * kSchedStride];

// Scratch of attn_decode_noalloc: the per-slice decode partials of one call
// (see include/attn_b300.h).  Fixed size, one copy per device, shared by every
// call of that entry point.
constexpr size_t kNoAllocScratchBytes = ATTN_NOALLOC_SCRATCH_BYTES;
static __device__ __align__(256) float g_decode_scratch[kNoAllocScratchBytes / sizeof(float)];

namespace {

constexpr int kMaxDevices = 64;
std::atomic<unsigned long long> g_timeout_ns{1000000000ull};
// Smallest wait budget attn_set_wait_timeout_ns accepts.
constexpr unsigned long long kMinTimeoutNs = 1000000ull;
// Set by attn_set_fault_injection: launches made while it is on stall CTA 0.
std::atomic<int> g_stall{0};

struct DeviceState {
  int checked = 0;  // 0 unknown, 1 ok, -1 wrong arch
  unsigned int* err = nullptr;
  unsigned int* sched = nullptr;             // g_sched on this device
  std::atomic<unsigned int> sched_next{0};   // slot of the next launch
  bool attrs_set = false;
  int sms = 0;
};
DeviceState g_dev[kMaxDevices];
std::mutex g_mu;

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;

template <int D>
bool set_decode_smem() {
  return cudaFuncSetAttribute(attn_decode_bf16_kernel<D>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize,
                              DecCfg<D>::SMEM_ALLOC) != cudaSuccess;
}

template <int D>
void launch_decode_kernel(unsigned grid, cudaStream_t s, const CUtensorMap& mk,
                          const CUtensorMap& mv, const DecodeParams& p) {
  attn_decode_bf16_kernel<D><<<grid, DecCfg<D>::THREADS, DecCfg<D>::SMEM_ALLOC, s>>>(mk, mv, p);
}

// Read-only stream of device memory (a measurement helper): one CTA per SM
// copies chunks of 32 KB with 1-D TMA bulk copies into a 4-stage shared-memory
// ring (128 KB in flight per SM; TMA bulk rings read HBM fastest in sweeps of
// load shapes on B300) and
// folds every 32-bit word with XOR; each warp XORs its fold into *out, so the
// data is really read.  Every wait is bounded; after an abort the CTA still
// waits for the copies it issued before it exits.
constexpr int kProbeStages = 4;
constexpr int kProbeChunk = 32768;
constexpr int kProbeSmem = kProbeStages * kProbeChunk + 64;

__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes,
                                          uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
      ::"r"(dst), "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
      : "memory");
}

__global__ void __launch_bounds__(256)
    hbm_read_probe_kernel(const uint8_t* __restrict__ p, unsigned long long bytes,
                          unsigned int* out, unsigned long long timeout, unsigned int* err) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* ring = smem_raw;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem_raw + kProbeStages * kProbeChunk);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(full + kProbeStages);
  const unsigned long long nchunks = (bytes + kProbeChunk - 1) / kProbeChunk;
  const unsigned long long mine =
      nchunks > blockIdx.x ? (nchunks - 1 - blockIdx.x) / gridDim.x + 1 : 0;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kProbeStages; ++s) mbar_init(&full[s], 1);
    *abort_flag = 0;
    mbar_fence_init();
  }
  __syncthreads();
  const WaitCtl ctl{abort_flag, err, timeout};
  const uint32_t ring_s = smem_u32(ring);
  auto chunk_bytes = [&](unsigned long long k) {
    const unsigned long long off = (blockIdx.x + k * gridDim.x) * kProbeChunk;
    return static_cast<uint32_t>(bytes - off < kProbeChunk ? bytes - off : kProbeChunk);
  };
  auto issue = [&](unsigned long long k) {
    const int s = static_cast<int>(k % kProbeStages);
    const uint32_t n = chunk_bytes(k);
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(
                     smem_u32(&full[s])),
                 "r"(n)
                 : "memory");
    bulk_load(ring_s + s * kProbeChunk, p + (blockIdx.x + k * gridDim.x) * kProbeChunk, n,
              smem_u32(&full[s]));
  };
  if (threadIdx.x == 0)
    for (unsigned long long k = 0; k < mine && k < kProbeStages; ++k) issue(k);
  uint32_t acc = 0;
  unsigned long long k = 0;
  bool ok = true;
  for (; k < mine; ++k) {
    const int s = static_cast<int>(k % kProbeStages);
    ok = __syncthreads_and(mbar_wait(&full[s], static_cast<uint32_t>((k / kProbeStages) & 1), ctl));
    if (!ok) break;
    const uint4* c = reinterpret_cast<const uint4*>(ring + s * kProbeChunk);
    const int n16 = static_cast<int>(chunk_bytes(k) / 16);
    for (int i = threadIdx.x; i < n16; i += blockDim.x) {
      const uint4 a = c[i];
      acc ^= a.x ^ a.y ^ a.z ^ a.w;
    }
    __syncthreads();
    if (threadIdx.x == 0 && k + kProbeStages < mine) {
      fence_proxy_async_smem();  // the generic reads of the slot come before the copy into it
      issue(k + kProbeStages);
    }
  }
  if (!ok) {
    if (threadIdx.x == 0)
      for (unsigned long long d = k; d < mine && d < k + kProbeStages; ++d)
        mbar_wait_drain(&full[d % kProbeStages],
                        static_cast<uint32_t>((d / kProbeStages) & 1), ctl);
    __syncthreads();
    return;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) acc ^= __shfl_xor_sync(0xffffffffu, acc, o);
  if ((threadIdx.x & 31) == 0) atomicXor(out, acc);
}

// The work counter of the next persistent launch on this device.
unsigned int* next_sched_slot(DeviceState* st) {
  return st->sched + (st->sched_next.fetch_add(1) % kSchedSlots) * kSchedStride;
}

// Checks the current device once and fetches what the launches need.
int prepare_device(DeviceState** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return ATTN_ERR_LAUNCH;
  }
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceState& st = g_dev[dev];
  if (st.checked == 0) {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) {
      cudaGetLastError();
      return ATTN_ERR_LAUNCH;
    }
    if (major != 10 || minor != 3) {
      st.checked = -1;
    } else {
      void* p = nullptr;
      if (cudaGetSymbolAddress(&p, g_dev_error) != cudaSuccess) {
        cudaGetLastError();
        return ATTN_ERR_LAUNCH;
      }
      st.err = static_cast<unsigned int*>(p);
      void* ps = nullptr;
      if (cudaGetSymbolAddress(&ps, g_sched) != cudaSuccess || ps == nullptr) {
        cudaGetLastError();
        return ATTN_ERR_LAUNCH;
      }
      st.sched = static_cast<unsigned int*>(ps);
      if (cudaDeviceGetAttribute(&st.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
          st.sms < 1) {
        cudaGetLastError();
        return ATTN_ERR_LAUNCH;
      }
      if (g_encode == nullptr) {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                             cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess || fn == nullptr) {
          cudaGetLastError();
          return ATTN_ERR_LAUNCH;
        }
        g_encode = reinterpret_cast<EncodeTiledFn>(fn);
      }
      st.checked = 1;
    }
  }
  if (st.checked < 0) return ATTN_ERR_ARCH;
  if (!st.attrs_set) {
    if (cudaFuncSetAttribute(attn_fwd_bf16_kernel<64, false>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             Bf16Cfg<64>::SMEM_ALLOC) != cudaSuccess ||
        cudaFuncSetAttribute(attn_fwd_bf16_kernel<128, false>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             Bf16Cfg<128>::SMEM_ALLOC) != cudaSuccess ||
        cudaFuncSetAttribute(attn_fwd_bf16_kernel<64, true>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             Bf16Cfg<64>::SMEM_ALLOC) != cudaSuccess ||
        cudaFuncSetAttribute(attn_fwd_bf16_kernel<128, true>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             Bf16Cfg<128>::SMEM_ALLOC) != cudaSuccess) {
      cudaGetLastError();
      return ATTN_ERR_LAUNCH;
    }
    if (set_decode_smem<64>() || set_decode_smem<128>()) {
      cudaGetLastError();
      return ATTN_ERR_LAUNCH;
    }
    if (cudaFuncSetAttribute(attn_bwd_bf16_kernel<64, false>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             BwdCfg<64>::SMEM_ALLOC) != cudaSuccess ||
        cudaFuncSetAttribute(attn_bwd_bf16_kernel<128, false>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             BwdCfg<128>::SMEM_ALLOC) != cudaSuccess ||
        cudaFuncSetAttribute(attn_bwd_bf16_kernel<64, true>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             BwdCfg<64>::SMEM_ALLOC) != cudaSuccess ||
        cudaFuncSetAttribute(attn_bwd_bf16_kernel<128, true>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             BwdCfg<128>::SMEM_ALLOC) != cudaSuccess) {
      cudaGetLastError();
      return ATTN_ERR_LAUNCH;
    }
    if (cudaFuncSetAttribute(hbm_read_probe_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kProbeSmem) != cudaSuccess) {
      cudaGetLastError();
      return ATTN_ERR_LAUNCH;
    }
    const int f32_smem = (2 * kF32BM * 128 + kF32BN * 129) * 4;
    if (cudaFuncSetAttribute(attn_fwd_f32_kernel<4>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             f32_smem) != cudaSuccess) {
      cudaGetLastError();
      return ATTN_ERR_LAUNCH;
    }
    st.attrs_set = true;
  }
  *out = &st;
  return ATTN_OK;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Argument checks shared by every forward entry point.  Nk == 0 is allowed
// (every query then sees no key), and k, v may be NULL in that case.
int check_common(const void* q, const void* k, const void* v, const void* o, const void* lse,
                 int B, int H, int Nq, int Nk, const int* cu_q, const int* cu_k, float scale) {
  if (B < 1 || H < 1 || Nq < 0 || Nk < 0) return ATTN_ERR_SHAPE;
  if ((cu_q == nullptr) != (cu_k == nullptr)) return ATTN_ERR_NULL;
  if (!(std::isfinite(scale) && scale > 0.f)) return ATTN_ERR_SCALE;
  if (Nq == 0) return ATTN_OK;
  if (!q || !o || !lse || (Nk > 0 && (!k || !v))) return ATTN_ERR_NULL;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) ||
      !aligned(lse, 4))
    return ATTN_ERR_ALIGN;
  if ((cu_q && !aligned(cu_q, 4)) || (cu_k && !aligned(cu_k, 4))) return ATTN_ERR_ALIGN;
  // element counts must fit the 64-bit offsets and the int row indices
  const long long planes = cu_q ? static_cast<long long>(H) : 1LL * B * H;
  if (planes > (1LL << 31) - 1) return ATTN_ERR_SHAPE;
  if (planes * Nq > (1LL << 40) || planes * Nk > (1LL << 40)) return ATTN_ERR_SHAPE;
  return ATTN_OK;
}

int encode_16bit_map(CUtensorMap* map, const void* base, int D, int rows, int planes, bool f16) {
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(rows),
                              static_cast<cuuint64_t>(planes)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(D) * 2,
                                 static_cast<cuuint64_t>(rows) * D * 2};
  const cuuint32_t box[3] = {64, 128, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r = g_encode(map,
                              f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                              3, const_cast<void*>(base),
                              dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? ATTN_OK : ATTN_ERR_LAUNCH;
}

__global__ void wait_selftest_kernel(unsigned long long budget, unsigned int* err) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    mbar_fence_init();
  }
  __syncthreads();
  const WaitCtl ctl{&abort_flag, err, budget};
  if (threadIdx.x == 0) mbar_wait(&bar, 0, ctl);  // nothing ever arrives
  __syncthreads();
}



// 16-bit (bf16 or fp16) forward on the tcgen05 kernel.
int fwd_16bit(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
              int Nq, int Nk, int D, const int* cu_q, const int* cu_k, int causal, float scale,
              cudaStream_t s, bool f16) {
  if (D != 64 && D != 128) return ATTN_ERR_HEADDIM;
  if (Nq == 0) return ATTN_OK;
  DeviceState* st = nullptr;
  int rc = prepare_device(&st);
  if (rc != ATTN_OK) return rc;

  const int planes = cu_q ? H : B * H;
  CUtensorMap mq, mk, mv;
  if (encode_16bit_map(&mq, q, D, Nq, planes, f16) != ATTN_OK) return ATTN_ERR_LAUNCH;
  if (Nk > 0) {
    if (encode_16bit_map(&mk, k, D, Nk, planes, f16) != ATTN_OK ||
        encode_16bit_map(&mv, v, D, Nk, planes, f16) != ATTN_OK)
      return ATTN_ERR_LAUNCH;
  } else {
    mk = mq;  // no key: the kernel issues no K/V load
    mv = mq;
  }

  Bf16Params p;
  p.o = o;
  p.lse = lse;
  p.cu_seqlens = cu_q;
  p.cu_seqlens_k = cu_k;
  p.nseq = cu_q ? B : 0;
  p.planes = planes;
  p.rows = Nq;
  p.rows_k = Nk;
  p.n_qblk = (Nq + 255) / 256;
  // work items: packed -> pairs of mirror blocks of one sequence and head (an
  // upper bound: the sequences' blocks number at most Nq/256 + B, so their
  // pairs at most half that plus B); dense causal -> pairs of mirror blocks of
  // one plane, then the single blocks of the last tail_planes planes (about
  // one round of pairs); dense non-causal -> single blocks, the last round
  // possibly split into single query tiles (up to twice as many CTAs as blocks)
  const long long blocks = 1LL * p.n_qblk * planes;
  const long long npp = (p.n_qblk + 1) / 2;
  const long long tail = std::min<long long>(planes, (st->sms + npp - 1) / npp);
  p.tail_planes = (!cu_q && causal) ? static_cast<int>(tail) : 0;
  const long long items =
      cu_q ? 1LL * ((Nq / 256 + B) / 2 + B) * H
           : (causal ? (planes - tail) * npp + tail * p.n_qblk : 2 * blocks);
  if (items > 0x7fffffffLL || blocks > 0x7fffffffLL) return ATTN_ERR_SHAPE;
  p.n_tiles = static_cast<int>(items);
  p.causal = causal ? 1 : 0;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.stall = g_stall.load();
  p.timeout_ns = g_timeout_ns.load();
  p.err = st->err;
  // the causal and packed schedules hand out their items from a counter
  p.sched = (cu_q || causal) ? next_sched_slot(st) : nullptr;

  const unsigned grid = static_cast<unsigned>(std::min<long long>(items, st->sms));
  if (D == 64) {
    if (f16)
      attn_fwd_bf16_kernel<64, true><<<grid, Bf16Cfg<64>::THREADS, Bf16Cfg<64>::SMEM_ALLOC, s>>>(
          mq, mk, mv, p);
    else
      attn_fwd_bf16_kernel<64, false><<<grid, Bf16Cfg<64>::THREADS, Bf16Cfg<64>::SMEM_ALLOC, s>>>(
          mq, mk, mv, p);
  } else {
    if (f16)
      attn_fwd_bf16_kernel<128, true><<<grid, Bf16Cfg<128>::THREADS, Bf16Cfg<128>::SMEM_ALLOC,
                                        s>>>(mq, mk, mv, p);
    else
      attn_fwd_bf16_kernel<128, false><<<grid, Bf16Cfg<128>::THREADS, Bf16Cfg<128>::SMEM_ALLOC,
                                         s>>>(mq, mk, mv, p);
  }
  return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_LAUNCH;
}

// fp32 forward on CUDA cores.
int fwd_f32(const float* q, const float* k, const float* v, float* o, float* lse, int B, int H,
            int Nq, int Nk, int D, const int* cu_q, const int* cu_k, int causal, float scale,
            cudaStream_t s) {
  if (D < 1 || D > 128) return ATTN_ERR_HEADDIM;
  if (Nq == 0) return ATTN_OK;
  DeviceState* st = nullptr;
  const int rc = prepare_device(&st);
  if (rc != ATTN_OK) return rc;

  F32Params p;
  p.o = o;
  p.lse = lse;
  p.cu_seqlens = cu_q;
  p.cu_seqlens_k = cu_k;
  p.nseq = cu_q ? B : 0;
  p.planes = cu_q ? H : B * H;
  p.rows = Nq;
  p.rows_k = Nk;
  p.n_qblk = cu_q ? (Nq / kF32BM + B) : (Nq + kF32BM - 1) / kF32BM;
  p.D = D;
  p.causal = causal ? 1 : 0;
  p.scale = scale;
  p.err = st->err;
  const long long grid = 1LL * p.n_qblk * p.planes;
  if (grid > 0x7fffffffLL) return ATTN_ERR_SHAPE;
  const int smem = (2 * kF32BM * D + kF32BN * (D + 1)) * 4;
  attn_fwd_f32_kernel<4><<<static_cast<unsigned>(grid), 128, smem, s>>>(q, k, v, p);
  return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_LAUNCH;
}

// Every forward entry point ends here.
int fwd_any(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
            int Nq, int Nk, int D, const int* cu_q, const int* cu_k, int causal, float scale,
            int dtype, void* stream) {
  const int rc = check_common(q, k, v, o, lse, B, H, Nq, Nk, cu_q, cu_k, scale);
  if (rc != ATTN_OK) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  switch (dtype) {
    case ATTN_BF16:
    case ATTN_F16:
      return fwd_16bit(q, k, v, o, lse, B, H, Nq, Nk, D, cu_q, cu_k, causal, scale, s,
                       dtype == ATTN_F16);
    case ATTN_F32:
      return fwd_f32(static_cast<const float*>(q), static_cast<const float*>(k),
                     static_cast<const float*>(v), static_cast<float*>(o), lse, B, H, Nq, Nk, D,
                     cu_q, cu_k, causal, scale, s);
    default:
      return ATTN_ERR_DTYPE;
  }
}

// Workspace of the backward: Delta (fp32 per query row, padded to 256 bytes)
// followed by the fp32 dQ accumulator.
size_t bwd_delta_bytes(long long qrows) {
  return ((static_cast<size_t>(qrows) * 4 + 255) / 256) * 256;
}
size_t bwd_workspace_bytes(long long planes, long long nq, int D) {
  return bwd_delta_bytes(planes * nq) + static_cast<size_t>(planes * nq) * D * 4;
}

template <int D, bool F16>
void launch_bwd_kernels(unsigned grid, cudaStream_t s, const CUtensorMap& mq,
                        const CUtensorMap& mk, const CUtensorMap& mv, const CUtensorMap& mdo,
                        const CUtensorMap& mdq, const BwdParams& p, long long qrows) {
  if (qrows > 0) {
    const long long threads = qrows * 16;
    attn_bwd_prep_kernel<D, F16><<<static_cast<unsigned>((threads + 255) / 256), 256, 0, s>>>(
        p, qrows);
  }
  if (grid > 0)
    attn_bwd_bf16_kernel<D, F16><<<grid, BwdCfg<D>::THREADS, BwdCfg<D>::SMEM_ALLOC, s>>>(
        mq, mk, mv, mdo, mdq, p);
  if (qrows > 0) {
    const long long n8 = qrows * D / 8;
    attn_bwd_dq_kernel<F16><<<static_cast<unsigned>((n8 + 255) / 256), 256, 0, s>>>(p, n8);
  }
}

int bwd_16bit(const void* q, const void* k, const void* v, const void* o, const float* lse,
              const void* dout, void* dq, void* dk, void* dv, int B, int H, int Nq, int Nk, int D,
              const int* cu_q, const int* cu_k, int causal, float scale, bool f16,
              void* workspace, unsigned long long workspace_bytes, cudaStream_t s) {
  if (D != 64 && D != 128) return ATTN_ERR_HEADDIM;
  const int planes = cu_q ? H : B * H;
  const long long qrows = 1LL * planes * Nq;
  if (qrows > 0) {
    if (!q || !dout || !dq || !o || !lse || !workspace) return ATTN_ERR_NULL;
    if (!aligned(q, 16) || !aligned(dout, 16) || !aligned(dq, 16) || !aligned(o, 16) ||
        !aligned(lse, 4) || !aligned(workspace, 16))
      return ATTN_ERR_ALIGN;
    if (workspace_bytes < bwd_workspace_bytes(planes, Nq, D)) return ATTN_ERR_SCRATCH;
  }
  if (Nk > 0) {
    if (!k || !v || !dk || !dv) return ATTN_ERR_NULL;
    if (!aligned(k, 16) || !aligned(v, 16) || !aligned(dk, 16) || !aligned(dv, 16))
      return ATTN_ERR_ALIGN;
  }
  if ((cu_q && !aligned(cu_q, 4)) || (cu_k && !aligned(cu_k, 4))) return ATTN_ERR_ALIGN;
  DeviceState* st = nullptr;
  int rc = prepare_device(&st);
  if (rc != ATTN_OK) return rc;

  // With no key the main kernel has no tile: the prep and dQ kernels alone
  // write dQ = 0.  With no query it writes dK = dV = 0 and reads no query.
  CUtensorMap mq, mk, mv, mdo;
  if (Nk > 0) {
    if (encode_16bit_map(&mk, k, D, Nk, planes, f16) != ATTN_OK ||
        encode_16bit_map(&mv, v, D, Nk, planes, f16) != ATTN_OK)
      return ATTN_ERR_LAUNCH;
  }
  if (Nq > 0) {
    if (encode_16bit_map(&mq, q, D, Nq, planes, f16) != ATTN_OK ||
        encode_16bit_map(&mdo, dout, D, Nq, planes, f16) != ATTN_OK)
      return ATTN_ERR_LAUNCH;
  }
  if (Nk == 0) {
    mk = mq;
    mv = mq;
  }
  if (Nq == 0) {
    mq = mk;
    mdo = mk;
  }
  CUtensorMap mdq = mq;

  BwdParams p;
  p.o = o;
  p.dout = dout;
  p.lse = lse;
  p.delta = static_cast<float*>(workspace);
  p.dq_acc = workspace ? reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) +
                                                  bwd_delta_bytes(qrows))
                       : nullptr;
  if (qrows > 0) {
    // the fp32 dQ accumulator as a 2-D tensor (D, planes * rows), 32 x 32 boxes
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(qrows)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(D) * 4};
    const cuuint32_t box[2] = {32, 32};
    const cuuint32_t estr[2] = {1, 1};
    if (g_encode(&mdq, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, p.dq_acc, dims, strides, box, estr,
                 CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                 CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) !=
        CUDA_SUCCESS)
      return ATTN_ERR_LAUNCH;
  }
  p.dq = dq;
  p.dk = dk;
  p.dv = dv;
  p.cu_seqlens = cu_q;
  p.cu_seqlens_k = cu_k;
  p.nseq = cu_q ? B : 0;
  p.planes = planes;
  p.rows = Nq;
  p.rows_k = Nk;
  p.n_kblk = (Nk + 127) / 128;
  const long long tiles = Nk == 0 ? 0 : (cu_q ? (1LL * (Nk / 128 + B)) : 1LL * p.n_kblk);
  // persistent: one CTA per SM at most, taking the key tiles (work items)
  // from the launch's counter, heaviest first
  const long long items = tiles * planes;
  if (items > 0x7fffffffLL) return ATTN_ERR_SHAPE;
  const long long grid = std::min<long long>(items, st->sms);
  p.n_tiles = static_cast<int>(tiles);
  p.causal = causal ? 1 : 0;
  p.scale = scale;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.stall = g_stall.load();
  p.timeout_ns = g_timeout_ns.load();
  p.err = st->err;
  p.sched = next_sched_slot(st);
  const unsigned g = static_cast<unsigned>(grid);
  if (D == 64) {
    if (f16)
      launch_bwd_kernels<64, true>(g, s, mq, mk, mv, mdo, mdq, p, qrows);
    else
      launch_bwd_kernels<64, false>(g, s, mq, mk, mv, mdo, mdq, p, qrows);
  } else {
    if (f16)
      launch_bwd_kernels<128, true>(g, s, mq, mk, mv, mdo, mdq, p, qrows);
    else
      launch_bwd_kernels<128, false>(g, s, mq, mk, mv, mdo, mdq, p, qrows);
  }
  return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_LAUNCH;
}

// Key slices per plane for the decode kernel: enough CTAs to cover every SM
// about twice (bandwidth needs many loads in flight), slices of whole tiles.
struct DecodePlan {
  int nsplit;
  int chunk;
  size_t ws_bytes;
};

DecodePlan plan_decode(int planes, int nq, int nk, int D, int sms) {
  const int tiles = (nk + 127) / 128;
  const int per_sm = (D == 64) ? 4 : 2;
  long long want = (1LL * per_sm * sms + planes - 1) / planes;
  want = std::max(1LL, std::min<long long>(want, tiles));
  const int chunk = static_cast<int>((tiles + want - 1) / want) * 128;
  const int nsplit = (nk + chunk - 1) / chunk;
  DecodePlan d;
  d.nsplit = nsplit;
  d.chunk = chunk;
  d.ws_bytes = nsplit > 1 ? static_cast<size_t>(planes) * nsplit * nq * (D + 1) * sizeof(float) : 0;
  return d;
}

int check_decode(const void* q, const void* k, const void* v, const void* o, const void* lse,
                 int B, int H, int Nq, int Nk, int D, float scale) {
  if (B < 1 || H < 1 || Nq < 1 || Nq > kDecodeMaxQ || Nk < 1) return ATTN_ERR_SHAPE;
  if (D != 64 && D != 128) return ATTN_ERR_HEADDIM;
  if (!(std::isfinite(scale) && scale > 0.f)) return ATTN_ERR_SCALE;
  if (!q || !k || !v || !o || !lse) return ATTN_ERR_NULL;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) ||
      !aligned(lse, 4))
    return ATTN_ERR_ALIGN;
  const long long planes = 1LL * B * H;
  if (planes > (1 << 24) || planes * Nk > (1LL << 40)) return ATTN_ERR_SHAPE;
  return ATTN_OK;
}

// Launches the decode kernels with the given split plan and workspace.
int launch_decode(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                  int Nq, int Nk, int D, float scale, const DecodePlan& plan, float* ws,
                  DeviceState* st, cudaStream_t s) {
  const int planes = B * H;
  CUtensorMap mk, mv;
  if (encode_16bit_map(&mk, k, D, Nk, planes, false) != ATTN_OK ||
      encode_16bit_map(&mv, v, D, Nk, planes, false) != ATTN_OK)
    return ATTN_ERR_LAUNCH;
  DecodeParams p;
  p.o = o;
  p.lse = lse;
  p.ws_o = ws;
  p.ws_lse = ws ? ws + static_cast<size_t>(planes) * plan.nsplit * Nq * D : nullptr;
  p.q = q;
  p.planes = planes;
  p.nq = Nq;
  p.nk = Nk;
  p.nsplit = plan.nsplit;
  p.chunk = plan.chunk;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.stall = g_stall.load();
  p.timeout_ns = g_timeout_ns.load();
  p.err = st->err;
  const unsigned grid = static_cast<unsigned>(planes * plan.nsplit);
  if (D == 64)
    launch_decode_kernel<64>(grid, s, mk, mv, p);
  else
    launch_decode_kernel<128>(grid, s, mk, mv, p);
  if (plan.nsplit > 1) {
    const unsigned rows = static_cast<unsigned>(planes * Nq);
    if (D == 64)
      attn_decode_merge_kernel<64><<<rows, 64, 0, s>>>(p);
    else
      attn_decode_merge_kernel<128><<<rows, 128, 0, s>>>(p);
  }
  return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_LAUNCH;
}

}  // namespace
}  // namespace attn

using namespace attn;

extern "C" int attn_decode_workspace_bytes(int B, int H, int Nq, int Nk, int D,
                                           unsigned long long* bytes) {
  if (!bytes) return ATTN_ERR_NULL;
  if (B < 1 || H < 1 || Nq < 1 || Nq > kDecodeMaxQ || Nk < 1) return ATTN_ERR_SHAPE;
  if (D != 64 && D != 128) return ATTN_ERR_HEADDIM;
  // the plane limit of the decode entry points (B * H is then an int)
  if (1LL * B * H > (1 << 24)) return ATTN_ERR_SHAPE;
  DeviceState* st = nullptr;
  const int rc = prepare_device(&st);
  if (rc != ATTN_OK) return rc;
  *bytes = plan_decode(B * H, Nq, Nk, D, st->sms).ws_bytes;
  return ATTN_OK;
}

namespace {
// Device address of g_decode_scratch, looked up once per device (with that
// device current) by the first attn_decode_noalloc call on it.  In host code
// the array's name only stands in for the symbol; it is not an address the
// kernels may be given.
float* g_scratch_addr[kMaxDevices] = {};
std::mutex g_scratch_mu;

int noalloc_scratch(float** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return ATTN_ERR_LAUNCH;
  }
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (g_scratch_addr[dev] == nullptr) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_decode_scratch) != cudaSuccess || ptr == nullptr) {
      cudaGetLastError();
      return ATTN_ERR_LAUNCH;
    }
    g_scratch_addr[dev] = static_cast<float*>(ptr);
  }
  *out = g_scratch_addr[dev];
  return ATTN_OK;
}
}  // namespace

extern "C" int attn_decode_noalloc(const void* q, const void* k, const void* v, void* o,
                                   float* lse, int B, int H, int Nq, int Nk, int D, float scale,
                                   void* stream) {
  int rc = check_decode(q, k, v, o, lse, B, H, Nq, Nk, D, scale);
  if (rc != ATTN_OK) return rc;
  DeviceState* st = nullptr;
  rc = prepare_device(&st);
  if (rc != ATTN_OK) return rc;
  const DecodePlan plan = plan_decode(B * H, Nq, Nk, D, st->sms);
  if (plan.ws_bytes > kNoAllocScratchBytes) return ATTN_ERR_SCRATCH;
  float* scratch = nullptr;
  if (plan.nsplit > 1) {
    rc = noalloc_scratch(&scratch);
    if (rc != ATTN_OK) return rc;
  }
  return launch_decode(q, k, v, o, lse, B, H, Nq, Nk, D, scale, plan, scratch, st,
                       static_cast<cudaStream_t>(stream));
}

extern "C" int attn_decode(const void* q, const void* k, const void* v, void* o, float* lse,
                           int B, int H, int Nq, int Nk, int D, float scale, void* workspace,
                           unsigned long long workspace_bytes, void* stream) {
  int rc = check_decode(q, k, v, o, lse, B, H, Nq, Nk, D, scale);
  if (rc != ATTN_OK) return rc;
  if (workspace && !aligned(workspace, 16)) return ATTN_ERR_ALIGN;
  DeviceState* st = nullptr;
  rc = prepare_device(&st);
  if (rc != ATTN_OK) return rc;
  DecodePlan plan = plan_decode(B * H, Nq, Nk, D, st->sms);
  if (plan.nsplit > 1 && (workspace == nullptr || workspace_bytes < plan.ws_bytes)) {
    // no (or too small a) workspace: one slice per plane, written directly
    plan.nsplit = 1;
    plan.chunk = ((Nk + 127) / 128) * 128;
    plan.ws_bytes = 0;
  }
  return launch_decode(q, k, v, o, lse, B, H, Nq, Nk, D, scale, plan,
                       plan.nsplit > 1 ? static_cast<float*>(workspace) : nullptr, st,
                       static_cast<cudaStream_t>(stream));
}

extern "C" int attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                        int H, int N, int D, const int* cu_seqlens, int causal, float scale,
                        void* stream) {
  return fwd_any(q, k, v, o, lse, B, H, N, N, D, cu_seqlens, cu_seqlens, causal, scale, ATTN_BF16,
                 stream);
}

extern "C" int attn_fwd_f16(const void* q, const void* k, const void* v, void* o, float* lse,
                            int B, int H, int N, int D, const int* cu_seqlens, int causal,
                            float scale, void* stream) {
  return fwd_any(q, k, v, o, lse, B, H, N, N, D, cu_seqlens, cu_seqlens, causal, scale, ATTN_F16,
                 stream);
}

extern "C" int attn_fwd_f32(const float* q, const float* k, const float* v, float* o, float* lse,
                            int B, int H, int N, int D, const int* cu_seqlens, int causal,
                            float scale, void* stream) {
  return fwd_any(q, k, v, o, lse, B, H, N, N, D, cu_seqlens, cu_seqlens, causal, scale, ATTN_F32,
                 stream);
}

extern "C" int attn_fwd_cross(const void* q, const void* k, const void* v, void* o, float* lse,
                              int B, int H, int Nq, int Nk, int D, const int* cu_seqlens_q,
                              const int* cu_seqlens_k, int causal, float scale, int dtype,
                              void* stream) {
  return fwd_any(q, k, v, o, lse, B, H, Nq, Nk, D, cu_seqlens_q, cu_seqlens_k, causal, scale,
                 dtype, stream);
}

namespace {
// Host-buffer forward: copies in, kernels and copies out of successive chunks
// of planes run on three streams of their own (created once per device), so
// that the two copy directions and the kernels overlap.
constexpr int kHostChunks = 8;

struct HostPipe {
  bool ready = false;
  cudaStream_t h2d = nullptr, comp = nullptr, d2h = nullptr;
  cudaEvent_t start = nullptr, done = nullptr;
  cudaEvent_t in_ready[2] = {}, out_ready[2] = {}, slot_free[2] = {};
  std::mutex mu;  // one call enqueues at a time on a device
};
HostPipe g_pipe[kMaxDevices];

int host_pipe(HostPipe** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return ATTN_ERR_LAUNCH;
  }
  HostPipe& hp = g_pipe[dev];
  std::lock_guard<std::mutex> lock(g_mu);
  if (!hp.ready) {
    bool ok = cudaStreamCreateWithFlags(&hp.h2d, cudaStreamNonBlocking) == cudaSuccess &&
              cudaStreamCreateWithFlags(&hp.comp, cudaStreamNonBlocking) == cudaSuccess &&
              cudaStreamCreateWithFlags(&hp.d2h, cudaStreamNonBlocking) == cudaSuccess &&
              cudaEventCreateWithFlags(&hp.start, cudaEventDisableTiming) == cudaSuccess &&
              cudaEventCreateWithFlags(&hp.done, cudaEventDisableTiming) == cudaSuccess;
    for (int i = 0; ok && i < 2; ++i)
      ok = cudaEventCreateWithFlags(&hp.in_ready[i], cudaEventDisableTiming) == cudaSuccess &&
           cudaEventCreateWithFlags(&hp.out_ready[i], cudaEventDisableTiming) == cudaSuccess &&
           cudaEventCreateWithFlags(&hp.slot_free[i], cudaEventDisableTiming) == cudaSuccess;
    if (!ok) {
      cudaGetLastError();
      return ATTN_ERR_LAUNCH;
    }
    hp.ready = true;
  }
  *out = &hp;
  return ATTN_OK;
}

size_t round256(size_t x) { return (x + 255) / 256 * 256; }

struct HostPlan {
  long long ppc;     // planes per chunk
  long long nchunk;
  size_t tile;       // bytes of one q/k/v/o chunk buffer
  size_t lse;        // bytes of one lse chunk buffer
  size_t slot;       // bytes of one slot (q, k, v, o, lse)
};

HostPlan host_plan(long long planes, int N, int D, size_t elt) {
  HostPlan h;
  const long long chunks = std::min<long long>(planes, kHostChunks);
  h.ppc = (planes + chunks - 1) / chunks;
  h.nchunk = (planes + h.ppc - 1) / h.ppc;
  h.tile = round256(static_cast<size_t>(h.ppc) * N * D * elt);
  h.lse = round256(static_cast<size_t>(h.ppc) * N * 4);
  h.slot = 4 * h.tile + h.lse;
  return h;
}

size_t dtype_size(int dtype) { return dtype == ATTN_F32 ? 4 : 2; }
}  // namespace

extern "C" int attn_fwd_host_workspace_bytes(int B, int H, int N, int D, int dtype,
                                             unsigned long long* bytes) {
  if (!bytes) return ATTN_ERR_NULL;
  if (B < 1 || H < 1 || N < 0) return ATTN_ERR_SHAPE;
  if (dtype != ATTN_BF16 && dtype != ATTN_F16 && dtype != ATTN_F32) return ATTN_ERR_DTYPE;
  *bytes = N == 0 ? 0 : 2 * host_plan(1LL * B * H, N, D, dtype_size(dtype)).slot;
  return ATTN_OK;
}

extern "C" int attn_fwd_host(const void* q, const void* k, const void* v, void* o, float* lse,
                             int B, int H, int N, int D, int causal, float scale, int dtype,
                             void* workspace, unsigned long long workspace_bytes, void* stream) {
  if (B < 1 || H < 1 || N < 0) return ATTN_ERR_SHAPE;
  if (!(std::isfinite(scale) && scale > 0.f)) return ATTN_ERR_SCALE;
  if (dtype != ATTN_BF16 && dtype != ATTN_F16 && dtype != ATTN_F32) return ATTN_ERR_DTYPE;
  if (dtype == ATTN_F32 ? (D < 1 || D > 128) : (D != 64 && D != 128)) return ATTN_ERR_HEADDIM;
  if (N == 0) return ATTN_OK;
  if (!q || !k || !v || !o || !lse || !workspace) return ATTN_ERR_NULL;
  if (!aligned(workspace, 256)) return ATTN_ERR_ALIGN;
  const long long planes = 1LL * B * H;
  if (planes * N > (1LL << 40)) return ATTN_ERR_SHAPE;
  const size_t elt = dtype_size(dtype);
  const HostPlan hp = host_plan(planes, N, D, elt);
  if (workspace_bytes < 2 * hp.slot) return ATTN_ERR_SCRATCH;
  DeviceState* st = nullptr;
  int rc = prepare_device(&st);
  if (rc != ATTN_OK) return rc;
  HostPipe* pp = nullptr;
  rc = host_pipe(&pp);
  if (rc != ATTN_OK) return rc;

  std::lock_guard<std::mutex> lock(pp->mu);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  bool ok = cudaEventRecord(pp->start, s) == cudaSuccess &&
            cudaStreamWaitEvent(pp->h2d, pp->start, 0) == cudaSuccess &&
            cudaStreamWaitEvent(pp->comp, pp->start, 0) == cudaSuccess &&
            cudaStreamWaitEvent(pp->d2h, pp->start, 0) == cudaSuccess;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  for (long long c = 0; ok && c < hp.nchunk; ++c) {
    const int slot = static_cast<int>(c & 1);
    const long long p0 = c * hp.ppc;
    const long long np = std::min(hp.ppc, planes - p0);
    const size_t in_bytes = static_cast<size_t>(np) * N * D * elt;
    const size_t in_off = static_cast<size_t>(p0) * N * D * elt;
    const size_t lse_bytes = static_cast<size_t>(np) * N * 4;
    const size_t lse_off = static_cast<size_t>(p0) * N;
    uint8_t* base = ws + slot * hp.slot;
    uint8_t *dq = base, *dk = base + hp.tile, *dv = base + 2 * hp.tile, *dout = base + 3 * hp.tile;
    float* dlse = reinterpret_cast<float*>(base + 4 * hp.tile);
    // inputs of chunk c go where chunk c-2 was: wait until its outputs are read back
    if (c >= 2) ok = cudaStreamWaitEvent(pp->h2d, pp->slot_free[slot], 0) == cudaSuccess;
    ok = ok &&
         cudaMemcpyAsync(dq, static_cast<const uint8_t*>(q) + in_off, in_bytes,
                         cudaMemcpyHostToDevice, pp->h2d) == cudaSuccess &&
         cudaMemcpyAsync(dk, static_cast<const uint8_t*>(k) + in_off, in_bytes,
                         cudaMemcpyHostToDevice, pp->h2d) == cudaSuccess &&
         cudaMemcpyAsync(dv, static_cast<const uint8_t*>(v) + in_off, in_bytes,
                         cudaMemcpyHostToDevice, pp->h2d) == cudaSuccess &&
         cudaEventRecord(pp->in_ready[slot], pp->h2d) == cudaSuccess &&
         cudaStreamWaitEvent(pp->comp, pp->in_ready[slot], 0) == cudaSuccess;
    if (!ok) break;
    rc = fwd_any(dq, dk, dv, dout, dlse, 1, static_cast<int>(np), N, N, D, nullptr, nullptr,
                 causal, scale, dtype, pp->comp);
    if (rc != ATTN_OK) break;
    ok = cudaEventRecord(pp->out_ready[slot], pp->comp) == cudaSuccess &&
         cudaStreamWaitEvent(pp->d2h, pp->out_ready[slot], 0) == cudaSuccess &&
         cudaMemcpyAsync(static_cast<uint8_t*>(o) + in_off, dout, in_bytes,
                         cudaMemcpyDeviceToHost, pp->d2h) == cudaSuccess &&
         cudaMemcpyAsync(lse + lse_off, dlse, lse_bytes, cudaMemcpyDeviceToHost, pp->d2h) ==
             cudaSuccess &&
         cudaEventRecord(pp->slot_free[slot], pp->d2h) == cudaSuccess;
  }
  // the caller's stream continues once the last copy back is done
  ok = ok && cudaEventRecord(pp->done, pp->d2h) == cudaSuccess &&
       cudaStreamWaitEvent(s, pp->done, 0) == cudaSuccess;
  if (rc != ATTN_OK) return rc;
  if (!ok) {
    cudaGetLastError();
    return ATTN_ERR_LAUNCH;
  }
  return ATTN_OK;
}

extern "C" int attn_bwd_workspace_bytes(int B, int H, int Nq, int D, int packed,
                                        unsigned long long* bytes) {
  if (!bytes) return ATTN_ERR_NULL;
  if (B < 1 || H < 1 || Nq < 0) return ATTN_ERR_SHAPE;
  if (D != 64 && D != 128) return ATTN_ERR_HEADDIM;
  const long long planes = packed ? H : 1LL * B * H;
  *bytes = Nq == 0 ? 0 : bwd_workspace_bytes(planes, Nq, D);
  return ATTN_OK;
}

extern "C" int attn_bwd(const void* q, const void* k, const void* v, const void* o,
                        const float* lse, const void* dout, void* dq, void* dk, void* dv, int B,
                        int H, int Nq, int Nk, int D, const int* cu_seqlens_q,
                        const int* cu_seqlens_k, int causal, float scale, int dtype,
                        void* workspace, unsigned long long workspace_bytes, void* stream) {
  // the forward's checks cover q, k, v, the shapes, the offsets and the scale
  // (o and lse stand in for the forward's outputs)
  int rc = check_common(q, k, v, o, lse, B, H, Nq, Nk, cu_seqlens_q, cu_seqlens_k, scale);
  if (rc != ATTN_OK) return rc;
  if (dtype != ATTN_BF16 && dtype != ATTN_F16) return ATTN_ERR_DTYPE;
  if (Nq == 0 && Nk == 0) return ATTN_OK;
  return bwd_16bit(q, k, v, o, lse, dout, dq, dk, dv, B, H, Nq, Nk, D, cu_seqlens_q,
                   cu_seqlens_k, causal, scale, dtype == ATTN_F16, workspace, workspace_bytes,
                   static_cast<cudaStream_t>(stream));
}

extern "C" const char* attn_strerror(int status) {
  switch (status) {
    case ATTN_OK: return "ok";
    case ATTN_ERR_NULL: return "a required pointer is NULL";
    case ATTN_ERR_SHAPE: return "invalid shape (B, H >= 1, N >= 0, sizes within index range)";
    case ATTN_ERR_HEADDIM: return "head dimension not supported by this entry point";
    case ATTN_ERR_ALIGN: return "tensor pointers must be 16-byte aligned (lse, cu_seqlens 4-byte)";
    case ATTN_ERR_ARCH: return "current device is not compute capability 10.3 (sm_103a)";
    case ATTN_ERR_LAUNCH: return "CUDA runtime error during set-up or launch";
    case ATTN_ERR_TIMEOUT: return "a bounded wait inside a kernel ran out of time";
    case ATTN_ERR_BOUNDS: return "cu_seqlens entries outside [0, N] or decreasing";
    case ATTN_ERR_SCALE: return "scale must be finite and > 0";
    case ATTN_ERR_SCRATCH:
      return "the workspace (or the built-in decode scratch) is too small for this problem";
    case ATTN_ERR_DTYPE: return "element type not one of ATTN_BF16, ATTN_F16, ATTN_F32";
    default: return "unknown status";
  }
}

extern "C" int attn_get_device_error(void* stream) {
  DeviceState* st = nullptr;
  int rc = prepare_device(&st);
  if (rc != ATTN_OK) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  unsigned int v = 0;
  if (cudaStreamSynchronize(s) != cudaSuccess ||
      cudaMemcpyFromSymbolAsync(&v, g_dev_error, sizeof(v), 0, cudaMemcpyDeviceToHost, s) !=
          cudaSuccess ||
      cudaMemsetAsync(st->err, 0, sizeof(unsigned int), s) != cudaSuccess ||
      cudaStreamSynchronize(s) != cudaSuccess) {
    cudaGetLastError();
    return ATTN_ERR_LAUNCH;
  }
  if (v & kDevErrTimeout) return ATTN_ERR_TIMEOUT;
  if (v & kDevErrBounds) return ATTN_ERR_BOUNDS;
  if (v & kDevErrLayout) return ATTN_ERR_LAUNCH;
  return ATTN_OK;
}

extern "C" int attn_set_wait_timeout_ns(unsigned long long ns) {
  if (ns < kMinTimeoutNs) return ATTN_ERR_SHAPE;
  g_timeout_ns.store(ns);
  return ATTN_OK;
}

extern "C" int attn_set_fault_injection(int on) {
  if (on != 0 && on != 1) return ATTN_ERR_SHAPE;
  g_stall.store(on);
  return ATTN_OK;
}

extern "C" int attn_wait_selftest(unsigned long long timeout_ns, void* stream) {
  if (timeout_ns == 0) return ATTN_ERR_SHAPE;
  DeviceState* st = nullptr;
  int rc = prepare_device(&st);
  if (rc != ATTN_OK) return rc;
  wait_selftest_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(timeout_ns, st->err);
  return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_LAUNCH;
}

extern "C" int attn_hbm_read_probe(const void* buf, unsigned long long bytes, unsigned int* out,
                                   void* stream) {
  if (!buf || !out) return ATTN_ERR_NULL;
  if (bytes == 0 || bytes % 16 != 0) return ATTN_ERR_SHAPE;
  if (!aligned(buf, 16) || !aligned(out, 4)) return ATTN_ERR_ALIGN;
  DeviceState* st = nullptr;
  const int rc = prepare_device(&st);
  if (rc != ATTN_OK) return rc;
  hbm_read_probe_kernel<<<st->sms, 256, kProbeSmem, static_cast<cudaStream_t>(stream)>>>(
      static_cast<const uint8_t*>(buf), bytes, out, g_timeout_ns.load(), st->err);
  return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_LAUNCH;
}

extern "C" int attn_version(void) { return 201; }
