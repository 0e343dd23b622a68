// Rank order of the selected positions: the optional sorted output of the
// radix_topk pseudocode's final step ("Technical Deep Dive | ... Triton-TLE
// ... TopK Selector", section "02. Traditional GPU Approach: Radix Selection").
//
// One block per row.  Each selected position p becomes the 64-bit composite
// (~key(p) << 32) | p, so ascending composites are descending values with
// ties by lower position (the selector's own order: +0.0 above -0.0, -inf
// lowest, subnormals in place, through the same order-preserving key); empty
// slots (-1) become all ones and sort last.  The composites are sorted in
// shared memory by a bitonic network and written back in place.
#include <algorithm>
#include <cstring>
#include <mutex>
#include <type_traits>

#include "tks.h"
#include "tks_device.cuh"
#include "tks_internal.h"

namespace tks {
namespace {
using namespace k256;  // key map and dependent-launch helpers

constexpr int kOrderThreads = 1024;

// The composite of selected position p (all ones for an empty slot).
template <int DT>
__device__ __forceinline__ unsigned long long composite(const unsigned char* row,
                                                        int64_t row_stride, int p) {
  if (p < 0 || p >= row_stride) return ~0ull;
  const uint32_t key = DT == 0 ? key_f32(*reinterpret_cast<const uint32_t*>(row + (int64_t)p * 4))
                               : key_bf16(*reinterpret_cast<const uint16_t*>(row + (int64_t)p * 2));
  const uint32_t inv = DT == 0 ? ~key : (~key & 0xFFFFu);
  return ((unsigned long long)inv << 32) | (uint32_t)p;
}

// Fills comp[0, n) with the composites of the first k slots of sel (empty
// beyond k), nt threads; each thread has all its loads of one step in flight
// (every composite is two dependent loads).
template <int DT>
__device__ __forceinline__ void gather_composites(unsigned long long* comp, int n, const int32_t* sel,
                                                  int k, const unsigned char* row,
                                                  int64_t row_stride, int nt) {
  constexpr int kG = 8;
  for (int i0 = (int)threadIdx.x; i0 < n; i0 += kG * nt) {
    int p[kG];
#pragma unroll
    for (int j = 0; j < kG; ++j) {
      const int i = i0 + j * nt;
      p[j] = i < k ? sel[i] : -1;
    }
    unsigned long long c[kG];
#pragma unroll
    for (int j = 0; j < kG; ++j) c[j] = composite<DT>(row, row_stride, p[j]);
#pragma unroll
    for (int j = 0; j < kG; ++j)
      if (i0 + j * nt < n) comp[i0 + j * nt] = c[j];
  }
}
static_assert(kOrderKMax == TKS_SORTED_K_MAX, "the C header states the limit");

template <int DT>
__global__ void __launch_bounds__(kOrderThreads) tks_order_kernel(const unsigned char* logits,
                                                                  int64_t row_stride, int32_t k,
                                                                  int32_t n, int32_t* out) {
  extern __shared__ __align__(16) unsigned long long comp[];
  grid_launch_dependents();
  grid_dependency_wait();  // out is written by the kernel ahead in the stream
  const int64_t r = blockIdx.x;
  int32_t* o = out + r * k;
  const unsigned char* row = logits + r * row_stride * (DT == 0 ? 4 : 2);
  gather_composites<DT>(comp, n, o, k, row, row_stride, (int)blockDim.x);
  __syncthreads();
  // Bitonic network, ascending (n a power of two, >= 64 or the whole row in
  // one warp).  Steps whose partner lies within the same 64-element segment
  // run in registers: each warp takes a segment, lane l holding elements
  // 2l and 2l+1 (stride 1 inside the lane, strides 2..32 by shuffles); the
  // other steps go through shared memory.
  const int nseg = n >= 64 ? n / 64 : 1;
  const int seg_len = n >= 64 ? 64 : n;
  const int warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
  const int lane = (int)(threadIdx.x & 31u);
  // one compare-exchange step with partner stride S (< 64) inside a segment
  auto seg_step = [&](unsigned long long& x0, unsigned long long& x1, int e0, int size, auto S) {
    constexpr int kS = decltype(S)::value;
    if constexpr (kS == 1) {
      const bool up = (e0 & size) == 0;  // e0 is the lower index of the pair
      const unsigned long long lo = x0 < x1 ? x0 : x1, hi = x0 < x1 ? x1 : x0;
      x0 = up ? lo : hi;
      x1 = up ? hi : lo;
    } else {
      constexpr int kLm = kS >> 1;  // partner lane
      const unsigned long long y0 = __shfl_xor_sync(0xffffffffu, x0, kLm);
      const unsigned long long y1 = __shfl_xor_sync(0xffffffffu, x1, kLm);
      const bool lower = (lane & kLm) == 0;
      // the lower index of an ascending pair keeps the smaller value
      const bool keep_min0 = lower == ((e0 & size) == 0);
      const bool keep_min1 = lower == (((e0 + 1) & size) == 0);
      x0 = (keep_min0 == (y0 < x0)) ? y0 : x0;
      x1 = (keep_min1 == (y1 < x1)) ? y1 : x1;
    }
  };
  // the steps of one size with strides 32 .. 1 (those of the size below 64 only)
  auto seg_level = [&](unsigned long long& x0, unsigned long long& x1, int e0, int size) {
    if (size >= 64) seg_step(x0, x1, e0, size, std::integral_constant<int, 32>{});
    if (size >= 32) seg_step(x0, x1, e0, size, std::integral_constant<int, 16>{});
    if (size >= 16) seg_step(x0, x1, e0, size, std::integral_constant<int, 8>{});
    if (size >= 8) seg_step(x0, x1, e0, size, std::integral_constant<int, 4>{});
    if (size >= 4) seg_step(x0, x1, e0, size, std::integral_constant<int, 2>{});
    seg_step(x0, x1, e0, size, std::integral_constant<int, 1>{});
  };
  // every step with stride < 64 of sizes in [size_lo, size_hi]
  auto in_segments = [&](int size_lo, int size_hi) {
    for (int sg = warp; sg < nseg; sg += nwarps) {
      const int e0 = sg * seg_len + 2 * lane;
      const bool live = 2 * lane < seg_len;
      unsigned long long x0 = live ? comp[e0] : ~0ull, x1 = live ? comp[e0 + 1] : ~0ull;
      for (int size = size_lo; size <= size_hi; size <<= 1) seg_level(x0, x1, e0, size);
      if (live) {
        comp[e0] = x0;
        comp[e0 + 1] = x1;
      }
    }
    __syncthreads();
  };
  in_segments(2, n < 64 ? n : 64);
  for (int size = 128; size <= n; size <<= 1) {
    for (int stride = size >> 1; stride >= 64; stride >>= 1) {
      for (int t = threadIdx.x; t < (n >> 1); t += blockDim.x) {
        const int i = 2 * t - (t & (stride - 1));
        const int j = i + stride;
        const unsigned long long a = comp[i], b = comp[j];
        const bool up = (i & size) == 0;
        if ((a > b) == up) {
          comp[i] = b;
          comp[j] = a;
        }
      }
      __syncthreads();
    }
    in_segments(size, size);
  }
  for (int i = threadIdx.x; i < k; i += blockDim.x) {
    const unsigned long long c = comp[i];
    o[i] = c == ~0ull ? -1 : (int32_t)(uint32_t)c;
  }
}

// Rank order of a few rows over many blocks.  Block (row, tile) holds the
// row's k composites in shared memory and places the TILE slots of its tile:
// a slot's place is the number of composites below its own (composites of
// selected positions are distinct; empty slots -- the last ones of a row
// shorter than k -- keep their place), counted by kRankThreads / TILE
// threads over interleaved parts of the row.  Reads the unordered selection
// sel and writes out, so blocks need not wait for one another.
constexpr int kRankThreads = 512;

template <int DT, int TILE>
__global__ void __launch_bounds__(kRankThreads) tks_rank_kernel(const unsigned char* logits,
                                                                int64_t row_stride, int32_t k,
                                                                const int32_t* sel, int32_t* out,
                                                                int32_t tiles) {
  constexpr int kLanes = kRankThreads / TILE;  // threads per slot, within one warp
  static_assert(kLanes <= 32 && 32 % kLanes == 0, "a slot's threads share a warp");
  extern __shared__ __align__(16) unsigned long long comp[];
  grid_launch_dependents();
  grid_dependency_wait();  // sel is written by the kernel ahead in the stream
  const int64_t r = blockIdx.x / tiles;
  const int tile = (int)(blockIdx.x % tiles);
  const int32_t* srow = sel + r * k;
  const unsigned char* row = logits + r * row_stride * (DT == 0 ? 4 : 2);
  gather_composites<DT>(comp, k, srow, k, row, row_stride, kRankThreads);
  __syncthreads();
  const int slot = tile * TILE + (int)threadIdx.x / kLanes;
  const int sub = (int)threadIdx.x % kLanes;
  const unsigned long long c = slot < k ? comp[slot] : ~0ull;
  unsigned below = 0u;
  if (c != ~0ull) {
#pragma unroll 4
    for (int f = sub; f < k; f += kLanes) below += comp[f] < c ? 1u : 0u;
  }
#pragma unroll
  for (int d = kLanes / 2; d > 0; d >>= 1) below += __shfl_xor_sync(0xffffffffu, below, d);
  if (slot < k && sub == 0)
    out[r * k + (c == ~0ull ? slot : (int)below)] = c == ~0ull ? -1 : (int32_t)(uint32_t)c;
}

std::mutex g_order_mu;
bool g_order_attr[2] = {false, false};  // shared-memory opt-in set (per process; all devices)
bool g_rank_attr[6] = {false, false, false, false, false, false};  // per dtype and tile
constexpr size_t kRankSmemMin = 120 * 1024;
static_assert((size_t)kRankKMax * sizeof(unsigned long long) <= kRankSmemMin, "opt-in covers every k");

}  // namespace

cudaError_t launch_rank_order(const void* logits, int32_t batch, int64_t row_stride, int32_t k,
                              int32_t dtype, int32_t* out, cudaStream_t stream) {
  int n = 2;
  while (n < k) n <<= 1;
  const size_t smem = (size_t)n * sizeof(unsigned long long);
  {
    std::lock_guard<std::mutex> lock(g_order_mu);
    if (!g_order_attr[dtype]) {
      const cudaError_t e = dtype == TKS_F32
          ? cudaFuncSetAttribute(tks_order_kernel<0>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)(kOrderKMax * sizeof(unsigned long long)))
          : cudaFuncSetAttribute(tks_order_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)(kOrderKMax * sizeof(unsigned long long)));
      if (e != cudaSuccess) return e;
      g_order_attr[dtype] = true;
    }
  }
  cudaLaunchConfig_t cfg;
  std::memset(&cfg, 0, sizeof cfg);
  cfg.gridDim = dim3((unsigned)batch, 1, 1);
  // whole warps (the in-segment steps shuffle across all 32 lanes)
  const int threads = n / 2 < 32 ? 32 : (n / 2 < kOrderThreads ? n / 2 : kOrderThreads);
  cfg.blockDim = dim3((unsigned)threads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  std::memset(attr, 0, sizeof attr);
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const unsigned char* lg = static_cast<const unsigned char*>(logits);
  return dtype == TKS_F32 ? cudaLaunchKernelEx(&cfg, tks_order_kernel<0>, lg, row_stride, k, n, out)
                          : cudaLaunchKernelEx(&cfg, tks_order_kernel<1>, lg, row_stride, k, n, out);
}

cudaError_t launch_rank_order_rows(const void* logits, int32_t batch, int64_t row_stride,
                                   int32_t k, int32_t dtype, const int32_t* sel, int32_t* out,
                                   cudaStream_t stream) {
  // the smallest tile that keeps the grid within one block per SM
  int sms = 0, dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return cudaErrorUnknown;
  const int tile = (int64_t)batch * ((k + 15) / 16) <= sms ? 16
                   : (int64_t)batch * ((k + 31) / 32) <= sms ? 32 : 64;
  const int tiles = (k + tile - 1) / tile;
  // at least kRankSmemMin of shared memory: one block per SM, so a row's
  // blocks spread over the device instead of sharing a few SMs
  const size_t smem = std::max((size_t)k * sizeof(unsigned long long), kRankSmemMin);
  using Kern = void (*)(const unsigned char*, int64_t, int32_t, const int32_t*, int32_t*, int32_t);
  Kern kern = dtype == TKS_F32 ? (tile == 16 ? tks_rank_kernel<0, 16>
                                  : tile == 32 ? tks_rank_kernel<0, 32> : tks_rank_kernel<0, 64>)
                               : (tile == 16 ? tks_rank_kernel<1, 16>
                                  : tile == 32 ? tks_rank_kernel<1, 32> : tks_rank_kernel<1, 64>);
  {
    std::lock_guard<std::mutex> lock(g_order_mu);
    const int idx = dtype * 3 + (tile == 16 ? 0 : tile == 32 ? 1 : 2);
    if (!g_rank_attr[idx]) {
      const cudaError_t e =
          cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kRankSmemMin);
      if (e != cudaSuccess) return e;
      g_rank_attr[idx] = true;
    }
  }
  cudaLaunchConfig_t cfg;
  std::memset(&cfg, 0, sizeof cfg);
  cfg.gridDim = dim3((unsigned)(batch * tiles), 1, 1);
  cfg.blockDim = dim3((unsigned)kRankThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  std::memset(attr, 0, sizeof attr);
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const unsigned char* lg = static_cast<const unsigned char*>(logits);
  return cudaLaunchKernelEx(&cfg, kern, lg, row_stride, k, sel, out, (int32_t)tiles);
}

}  // namespace tks
