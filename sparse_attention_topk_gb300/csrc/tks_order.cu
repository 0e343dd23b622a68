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

#include "tks.h"
#include "tks_device.cuh"
#include "tks_internal.h"

namespace tks {
namespace {

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
  // bitonic network, ascending; n is a power of two
  for (int size = 2; size <= n; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
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
  cfg.blockDim = dim3((unsigned)(n / 2 < kOrderThreads ? n / 2 : kOrderThreads), 1, 1);
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
