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
  for (int i = threadIdx.x; i < n; i += blockDim.x) {
    unsigned long long c = ~0ull;
    const int p = i < k ? o[i] : -1;
    if (p >= 0 && p < row_stride) {
      const uint32_t key = DT == 0 ? key_f32(*reinterpret_cast<const uint32_t*>(row + (int64_t)p * 4))
                                   : key_bf16(*reinterpret_cast<const uint16_t*>(row + (int64_t)p * 2));
      const uint32_t inv = DT == 0 ? ~key : (~key & 0xFFFFu);
      c = ((unsigned long long)inv << 32) | (uint32_t)p;
    }
    comp[i] = c;
  }
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

std::mutex g_order_mu;
bool g_order_attr[2] = {false, false};  // shared-memory opt-in set (per process; all devices)

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

}  // namespace tks
