// Top-k index selection by radix selection on GB300 (sm_103a).
//
// Method ("Technical Deep Dive | How to Use FlagOS's New Triton-TLE Language
// to Build a TopK Selector Faster Than FlashInfer", section "02. Traditional
// GPU Approach: Radix Selection"): map logits to order-preserving unsigned
// keys, take digits from the most significant bits down, histogram each digit,
// keep only the bin that holds the k-th element, and finally collect every
// element above the threshold.  Ties at the k-th value go to the lowest
// positions (the page's collection step scans the row in order); here that is
// obtained by extending each key with its inverted position, so the digit
// walk simply continues into the position bits when values tie.
//
// Layout of the work (one kernel launch per call; the kernel itself is in
// tks_kernel.cuh, built here with 256 threads per block and in
// tks_select512.cu with 512):
//  * A row is split into `group` contiguous slices, one thread block (one
//    per SM) each.  Each block copies its slice from HBM once, with a bulk
//    asynchronous copy (TMA, non-tensor form) into shared memory, and builds
//    a 4096-bin histogram of the top 12 key bits on chip.
//  * With group > 1 the blocks of a row add their histograms together, in
//    L2 behind a bounded barrier, or, when the row is one thread-block
//    cluster, in block 0's shared memory behind cluster barriers; every
//    block then finds the threshold bin itself (the page's "TLE distributed"
//    idea of summing block histograms and continuing with the new threshold,
//    section "5. Triton-TLE").  The adds return each block's offset inside
//    every bin, so each block can later write its selected positions to
//    fixed output slots with no further coordination.
//  * As soon as the bin holding the k-th element has few enough members
//    (the page's "early stop when the bucket is small", section "03."),
//    blocks write every position above the bin to the output and push the
//    bin's (key, position) pairs to a candidate buffer; block 0 of the row
//    refines those candidates on chip and writes the rest.
//  * With group == 1 (many rows) a block owns whole rows and needs no
//    cross-block step at all.
//  * A row whose keys are all equal (a constant row, all -inf) is answered
//    right after the first round with its lowest positions.
// No tensor cores: this is a streaming selection, not a contraction.

#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>
#include <cstring>
#include <map>
#include <mutex>
#include <utility>

#include "tks.h"
#include "tks_kernel.cuh"  // the 256-thread kernel, namespace tks::k256
#include "tks_internal.h"

namespace tks {
using namespace k256;  // shared-memory, workspace and status constants (equal for k512)

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
namespace {

struct DeviceInfo {
  int sms = 0;
  int blocks_per_sm = 0;
  int max_cluster = 1;  // largest thread-block cluster of the selection kernel
  bool ok = false;
};

struct Workspace {
  unsigned char* ptr = nullptr;
  size_t bytes = 0;
  int slots = 0;
};

std::mutex g_mu;
std::map<int, DeviceInfo> g_dev;
std::map<std::pair<int, void*>, Workspace> g_ws;

std::atomic<long long> g_force_group{0};
std::atomic<long long> g_spin_limit_ns{1000000000LL};
std::atomic<long long> g_min_per_block{4096};
constexpr long long kLoneRowMax = 4096;  // rows this short are never split
std::atomic<long long> g_test_skip_arrive{0};

int device_info(int dev, DeviceInfo* out) {
  auto it = g_dev.find(dev);
  if (it != g_dev.end()) {
    *out = it->second;
    return out->ok ? TKS_OK : TKS_E_UNSUPPORTED;
  }
  DeviceInfo d;
  int major = 0, minor = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
    cudaGetLastError();
    g_dev[dev] = d;
    *out = d;
    return TKS_E_UNSUPPORTED;
  }
  if (major == 10 && minor == 3) {
    int b256 = 0, b512 = 0, c256 = 1, c512 = 1;
    const bool good = k256::setup_select(&b256, &c256) && k512::setup_select(&b512, &c512);
    d.blocks_per_sm = b256 < b512 ? b256 : b512;  // a plan's grid fits either block size
    d.max_cluster = c256 < c512 ? c256 : c512;
    d.ok = good && d.blocks_per_sm >= 1;
    if (!good) cudaGetLastError();
  }
  g_dev[dev] = d;
  *out = d;
  return d.ok ? TKS_OK : TKS_E_UNSUPPORTED;
}

// Block size: rows split into large slices run with 512 threads (measured:
// 64 ragged 64K rows over 2 blocks of 128 KiB, 17.6 -> 17.2 us); smaller
// slices (four 1M-element bf16 rows over 37 blocks of 56 KiB: 14.1 us with
// 256, 14.7 with 512) and whole rows per block are faster with 256 (fewer
// warps for the control steps).
constexpr long long kBigSliceBytes = 96 * 1024;
std::atomic<long long> g_force_threads{0};

int plan_threads(int32_t batch, int64_t row_stride, int32_t dtype, int group) {
  const long long forced = g_force_threads.load();
  if (forced == 256 || forced == 512) return (int)forced;
  (void)batch;
  const long long es = dtype == TKS_F32 ? 4 : 2;
  return group > 1 && (row_stride + group - 1) / group * es >= kBigSliceBytes ? 512 : 256;
}

// Rows split over one thread-block cluster (its blocks merge through
// distributed shared memory and the cluster barrier) only when asked for:
// TKS_OPT_CLUSTER n >= 2 gives clusters of n blocks.  Automatically (0) and
// with 1, split rows merge through L2: measured back to back, fp32 rows of
// 32K to 512K elements took 9.1-10.0 us split through L2 at about 4096
// elements per block and 9.8-12.0 us in the clusters chosen before (up to 16
// blocks of about 32 KiB).
std::atomic<long long> g_cluster_opt{0};

int plan_cluster(const DeviceInfo& d, int32_t batch, int64_t row_stride, int32_t dtype) {
  const long long opt = g_cluster_opt.load();
  if (opt < 2 || g_force_group.load() > 0 || d.max_cluster < 2) return 0;
  const long long es = dtype == TKS_F32 ? 4 : 2;
  if (row_stride <= kLoneRowMax) return 0;
  const int n = (int)(opt < d.max_cluster ? opt : d.max_cluster);
  const int cap = d.sms * d.blocks_per_sm;
  if ((long long)batch * n > cap - 1) return 0;
  if ((row_stride + n - 1) / n * es > kSliceBytes) return 0;  // slices stay on chip
  return n;
}

void plan_launch(const DeviceInfo& d, int32_t batch, int64_t row_stride, int* group, int* grid,
                 int32_t dtype = TKS_F32, bool* cluster = nullptr) {
  const int cap = d.sms * d.blocks_per_sm;
  if (cluster != nullptr) *cluster = false;
  if (batch >= cap) {
    *group = 1;
    *grid = cap;
    return;
  }
  const int cl = cluster != nullptr ? plan_cluster(d, batch, row_stride, dtype) : 0;
  if (cl >= 2) {
    *group = cl;
    *grid = batch * cl;
    if (cluster != nullptr) *cluster = true;
    return;
  }
  // Rows split over blocks leave one block slot of the device free when they
  // can, so that the blocks of the next call are all resident by the time the
  // finishing block of this one is done.
  const int per = (cap > 1 ? cap - 1 : cap) / batch;
  long long g;
  const long long forced = g_force_group.load();
  if (forced > 0) {
    g = forced;
  } else {
    // short rows stay on one block (a split costs a round trip through L2
    // that a block of their size does not make up for); longer ones get a
    // block per g_min_per_block elements
    const long long mpb = g_min_per_block.load() > 0 ? g_min_per_block.load() : 1;
    g = row_stride <= kLoneRowMax ? 1 : (row_stride + mpb - 1) / mpb;
  }
  if (g > per) g = per;
  if (g < 1) g = 1;
  *group = (int)g;
  *grid = batch * (int)g;
}

int workspace_slots(const DeviceInfo& d) { return d.sms * d.blocks_per_sm; }

// The slice length the kernel gives each of `group` blocks of a row of
// row_stride elements: a ceiling share rounded up to whole 16-byte vectors.
int32_t slice_chunk(int64_t row_stride, int group, int32_t dtype) {
  const int64_t v = dtype == TKS_F32 ? 4 : 2;
  return (int32_t)(((row_stride + group - 1) / group + v - 1) / v * v);
}

// Whether every block's slice of a row of up to row_stride elements split
// over `group` blocks fits the on-chip copy (its 16-byte vectors, with one
// partial vector at each end), so the kernel without the streamed path may
// be used.
bool slices_fit_on_chip(int64_t row_stride, int group, int32_t dtype) {
  const int64_t es = dtype == TKS_F32 ? 4 : 2, v = 16 / es;
  const int64_t chunk = ((row_stride + group - 1) / group + v - 1) / v * v;
  return (chunk / v + 2) * 16 <= (int64_t)kSliceBytes;
}

// Layout: status header | slot headers and counters | candidate slots |
// unordered selections of the rank-ordered path for a few rows.
size_t workspace_rank_offset(int slots) {
  return kWsHeaderBytes + (size_t)slots * (kSlotBytes + kCandSlotBytes);
}
constexpr size_t kRankScratchBytes = (size_t)kRankMaxRows * kRankKMax * sizeof(int32_t);
size_t workspace_bytes(const DeviceInfo& d) {
  return workspace_rank_offset(workspace_slots(d)) + kRankScratchBytes;
}

// Counters start at zero, candidate slots at all ones ("not written").
cudaError_t workspace_clear(const Workspace& w, int slots, cudaStream_t stream) {
  const size_t zero_bytes = kWsHeaderBytes + (size_t)slots * kSlotBytes;
  cudaError_t e = cudaMemsetAsync(w.ptr, 0, zero_bytes, stream);
  if (e == cudaSuccess) e = cudaMemsetAsync(w.ptr + zero_bytes, 0xFF, w.bytes - zero_bytes, stream);
  return e;
}

int get_workspace(int dev, void* stream, const DeviceInfo& d, Workspace* out) {
  auto key = std::make_pair(dev, stream);
  auto it = g_ws.find(key);
  if (it != g_ws.end()) {
    *out = it->second;
    return TKS_OK;
  }
  Workspace w;
  w.bytes = workspace_bytes(d);
  w.slots = workspace_slots(d);
  if (cudaMalloc(&w.ptr, w.bytes) != cudaSuccess) {
    cudaGetLastError();
    return TKS_E_CUDA;
  }
  if (workspace_clear(w, w.slots, (cudaStream_t)stream) != cudaSuccess) {
    cudaGetLastError();
    cudaFree(w.ptr);
    return TKS_E_CUDA;
  }
  g_ws[key] = w;
  *out = w;
  return TKS_OK;
}

}  // namespace
}  // namespace tks

using namespace tks;

// Launch attributes: programmatic stream serialisation (the kernel may be
// scheduled while the previous kernel of the stream finishes; it waits for it
// before its first memory access), and a cooperative launch when the blocks of
// a row wait for one another, so that they are all resident.
static void set_launch_attrs(cudaLaunchConfig_t* cfg, cudaLaunchAttribute* attr, int group,
                             bool cluster = false) {
  std::memset(attr, 0, 2 * sizeof(cudaLaunchAttribute));
  int n = 0;
  attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[n].val.programmaticStreamSerializationAllowed = 1;
  ++n;
  if (cluster) {  // a row's blocks are one cluster, co-scheduled by construction
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = (unsigned)group;
    attr[n].val.clusterDim.y = 1;
    attr[n].val.clusterDim.z = 1;
    ++n;
  } else if (group > 1) {
    attr[n].id = cudaLaunchAttributeCooperative;
    attr[n].val.cooperative = 1;
    ++n;
  }
  cfg->attrs = attr;
  cfg->numAttrs = (unsigned)n;
}

// Argument checks shared by the entry points (nothing is touched on the device).
static int check_args(const void* logits, int32_t batch, int64_t row_stride, int32_t k,
                      int32_t dtype, const int32_t* out_idx) {
  if (batch < 0 || row_stride < 0 || row_stride > INT32_MAX || k < 1 || k > TKS_K_MAX)
    return TKS_E_INVAL;
  if (dtype != TKS_F32 && dtype != TKS_BF16) return TKS_E_INVAL;
  if (batch == 0) return TKS_OK;
  const int es = dtype == TKS_F32 ? 4 : 2;
  if (out_idx == nullptr || ((uintptr_t)out_idx & 3u) != 0) return TKS_E_INVAL;
  if (row_stride > 0 && (logits == nullptr || ((uintptr_t)logits % (uintptr_t)es) != 0))
    return TKS_E_INVAL;
  if ((int64_t)batch * row_stride > (INT64_MAX / 4)) return TKS_E_INVAL;
  return TKS_OK;
}

// The selection launch behind tks_topk_indices and tks_topk_indices_host;
// host_src: the pointers are device addresses of page-locked host memory.
static int select_launch(const void* logits, const int32_t* row_len, int32_t batch,
                         int64_t row_stride, int32_t k, int32_t dtype, int32_t* out_idx,
                         void* stream, bool host_src) {
  const int arg = check_args(logits, batch, row_stride, k, dtype, out_idx);
  if (arg != TKS_OK || batch == 0) return arg;

  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return TKS_E_UNSUPPORTED;
  }
  DeviceInfo d;
  Workspace w;
  {
    std::lock_guard<std::mutex> lock(g_mu);
    int rc = device_info(dev, &d);
    if (rc != TKS_OK) return rc;
    rc = get_workspace(dev, stream, d, &w);
    if (rc != TKS_OK) return rc;
  }
  int group = 1, grid = 1;
  bool cluster = false;
  plan_launch(d, batch, row_stride, &group, &grid, dtype, &cluster);

  Params p{};
  p.logits = static_cast<const unsigned char*>(logits);
  p.row_len = row_len;
  p.row_stride = row_stride;
  p.batch = batch;
  p.k = k;
  p.out = out_idx;
  p.group = group;
  p.test_skip_arrive = g_test_skip_arrive.load() ? 1 : 0;
  p.ws = w.ptr;
  p.slots = w.slots;
  p.spin_limit_ns = g_spin_limit_ns.load();
  p.cluster = cluster ? 1 : 0;
  p.host_src = host_src ? 1 : 0;
  p.chunk = slice_chunk(row_stride, group, dtype);
  // (the kernel without the streamed, host-memory, cluster and whole-row paths)
  const bool lean = group > 1 && !cluster && !host_src && slices_fit_on_chip(row_stride, group, dtype);

  cudaLaunchConfig_t cfg;
  std::memset(&cfg, 0, sizeof cfg);
  cfg.gridDim = dim3((unsigned)grid, 1, 1);
  cfg.stream = (cudaStream_t)stream;
  cudaLaunchAttribute attr[2];
  set_launch_attrs(&cfg, attr, group, cluster);
  cudaError_t e = plan_threads(batch, row_stride, dtype, group) == 512
                      ? k512::launch_select(cfg, p, dtype, lean)
                      : k256::launch_select(cfg, p, dtype, lean);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return TKS_E_CUDA;
  }
  return TKS_OK;
}

extern "C" int tks_topk_indices(const void* logits, const int32_t* row_len, int32_t batch,
                                int64_t row_stride, int32_t k, int32_t dtype, int32_t* out_idx,
                                void* stream) {
  return select_launch(logits, row_len, batch, row_stride, k, dtype, out_idx, stream, false);
}

// The device address of page-locked host memory (cudaHostAlloc, cudaMallocHost
// or cudaHostRegister), or nullptr when p is not such memory.
static void* host_to_device(const void* p) {
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  return a.type == cudaMemoryTypeHost ? a.devicePointer : nullptr;
}

extern "C" int tks_topk_indices_host(const void* logits, const int32_t* row_len, int32_t batch,
                                     int64_t row_stride, int32_t k, int32_t dtype,
                                     int32_t* out_idx, void* stream) {
  if (batch == 0)  // nothing is read or written: the arguments are only checked
    return select_launch(logits, row_len, batch, row_stride, k, dtype, out_idx, stream, true);
  if (batch < 0 || out_idx == nullptr) return TKS_E_INVAL;
  const void* dl = row_stride > 0 && logits != nullptr ? host_to_device(logits) : nullptr;
  void* dout = host_to_device(out_idx);
  const void* drl = row_len != nullptr ? host_to_device(row_len) : nullptr;
  if (dout == nullptr || (row_stride > 0 && dl == nullptr) || (row_len != nullptr && drl == nullptr))
    return TKS_E_INVAL;
  return select_launch(dl, static_cast<const int32_t*>(drl), batch, row_stride, k, dtype,
                       static_cast<int32_t*>(dout), stream, true);
}

extern "C" int tks_topk_indices_sorted(const void* logits, const int32_t* row_len, int32_t batch,
                                       int64_t row_stride, int32_t k, int32_t dtype, int32_t* out_idx,
                                       void* stream) {
  if (k > kOrderKMax) return TKS_E_INVAL;
  if (batch >= 1 && batch <= kRankMaxRows && k <= kRankKMax) {
    // A few rows: the selection goes to the stream's scratch, and the rank
    // kernel writes the ordered rows to out_idx from there over many blocks.
    const int arg = check_args(logits, batch, row_stride, k, dtype, out_idx);
    if (arg != TKS_OK) return arg;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
      cudaGetLastError();
      return TKS_E_UNSUPPORTED;
    }
    DeviceInfo d;
    Workspace w;
    {
      std::lock_guard<std::mutex> lock(g_mu);
      int rc = device_info(dev, &d);
      if (rc != TKS_OK) return rc;
      rc = get_workspace(dev, stream, d, &w);
      if (rc != TKS_OK) return rc;
    }
    int32_t* sel = reinterpret_cast<int32_t*>(w.ptr + workspace_rank_offset(w.slots));
    const int rc = select_launch(logits, row_len, batch, row_stride, k, dtype, sel, stream, false);
    if (rc != TKS_OK) return rc;
    if (launch_rank_order_rows(logits, batch, row_stride, k, dtype, sel, out_idx,
                               (cudaStream_t)stream) != cudaSuccess) {
      cudaGetLastError();
      return TKS_E_CUDA;
    }
    return TKS_OK;
  }
  const int rc = tks_topk_indices(logits, row_len, batch, row_stride, k, dtype, out_idx, stream);
  if (rc != TKS_OK || batch == 0) return rc;
  if (launch_rank_order(logits, batch, row_stride, k, dtype, out_idx, (cudaStream_t)stream) !=
      cudaSuccess) {
    cudaGetLastError();
    return TKS_E_CUDA;
  }
  return TKS_OK;
}

extern "C" int tks_device_status(void* stream) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return TKS_E_UNSUPPORTED;
  }
  if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) {
    cudaGetLastError();
    return TKS_E_CUDA;
  }
  Workspace w;
  {
    std::lock_guard<std::mutex> lock(g_mu);
    auto it = g_ws.find(std::make_pair(dev, stream));
    if (it == g_ws.end()) return TKS_OK;
    w = it->second;
  }
  unsigned st = 0;
  if (cudaMemcpyAsync(&st, w.ptr, sizeof st, cudaMemcpyDeviceToHost, (cudaStream_t)stream) !=
          cudaSuccess ||
      cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) {
    cudaGetLastError();
    return TKS_E_CUDA;
  }
  if (st == 0) return TKS_OK;
  if (workspace_clear(w, w.slots, (cudaStream_t)stream) != cudaSuccess ||
      cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) {
    cudaGetLastError();
    return TKS_E_CUDA;
  }
  if (st & kStatTimeout) return TKS_E_TIMEOUT;
  if (st & kStatInternal) return TKS_E_INTERNAL;
  return TKS_E_ROW_LEN;
}

extern "C" const char* tks_status_string(int status) {
  switch (status) {
    case TKS_OK: return "ok";
    case TKS_E_INVAL: return "invalid argument";
    case TKS_E_UNSUPPORTED: return "no supported CUDA device (needs compute capability 10.3)";
    case TKS_E_CUDA: return "CUDA runtime error";
    case TKS_E_TIMEOUT: return "a device-side wait between thread blocks timed out";
    case TKS_E_INTERNAL: return "device-side consistency check failed";
    case TKS_E_ROW_LEN: return "a row length was outside [0, row_stride] and was clamped";
    case TKS_E_TOO_LARGE: return "more rows than the allocation-free entry point's fixed scratch holds";
    default: return "unknown status";
  }
}

extern "C" int tks_version(void) { return 100; }

extern "C" int tks_release(void) {
  std::lock_guard<std::mutex> lock(g_mu);
  int rc = TKS_OK;
  int cur = 0;
  cudaGetDevice(&cur);
  for (auto& kv : g_ws) {
    cudaSetDevice(kv.first.first);
    if (cudaFree(kv.second.ptr) != cudaSuccess) rc = TKS_E_CUDA;
  }
  cudaSetDevice(cur);
  cudaGetLastError();
  g_ws.clear();
  return rc;
}

extern "C" int tks_set_option(int option, int64_t value) {
  if (value < 0) return TKS_E_INVAL;
  switch (option) {
    case TKS_OPT_FORCE_GROUP: g_force_group.store(value); return TKS_OK;
    case TKS_OPT_SPIN_LIMIT_NS: g_spin_limit_ns.store(value > 0 ? value : 1); return TKS_OK;
    case TKS_OPT_MIN_PER_BLOCK: g_min_per_block.store(value > 0 ? value : 4096); return TKS_OK;
    case TKS_OPT_TEST_SKIP_ARRIVE: g_test_skip_arrive.store(value ? 1 : 0); return TKS_OK;
    case TKS_OPT_CLUSTER: g_cluster_opt.store(value); return TKS_OK;
    case TKS_OPT_FORCE_THREADS:
      if (value != 0 && value != 256 && value != 512) return TKS_E_INVAL;
      g_force_threads.store(value);
      return TKS_OK;
    default: return TKS_E_INVAL;
  }
}

extern "C" int tks_plan(int32_t batch, int64_t row_stride, int32_t k, int32_t dtype, int32_t* group,
                        int32_t* grid) {
  if (batch < 1 || row_stride < 0 || k < 1 || (dtype != TKS_F32 && dtype != TKS_BF16))
    return TKS_E_INVAL;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return TKS_E_UNSUPPORTED;
  }
  DeviceInfo d;
  {
    std::lock_guard<std::mutex> lock(g_mu);
    const int rc = device_info(dev, &d);
    if (rc != TKS_OK) return rc;
  }
  int g = 1, gr = 1;
  bool cl = false;
  plan_launch(d, batch, row_stride, &g, &gr, dtype, &cl);
  if (group) *group = g;
  if (grid) *grid = gr;
  return TKS_OK;
}

// ---------------------------------------------------------------------------
// Allocation-free entry point.  Same selection, but its scratch (status word,
// per-row counters, candidate words) lives in a fixed array compiled into this
// library instead of a workspace the library allocates.
// ---------------------------------------------------------------------------
namespace tks {
namespace {
constexpr size_t kNoAllocBytes =
    kWsHeaderBytes + (size_t)TKS_NOALLOC_MAX_ROWS * (kSlotBytes + kCandSlotBytes);
std::map<int, unsigned char*> g_noalloc_addr;  // device -> device address of the array
}  // namespace
}  // namespace tks

// About 2.9 MB on every device that loads this library, held until exit.
static __device__ __align__(256) unsigned char g_noalloc_scratch[tks::kNoAllocBytes];

extern "C" int tks_topk_indices_noalloc(const void* logits, const int32_t* row_len, int32_t batch,
                                        int64_t row_stride, int32_t k, int32_t dtype,
                                        int32_t* out_idx, void* stream) {
  // the same argument checks as tks_topk_indices, then the array's row limit
  const int arg = check_args(logits, batch, row_stride, k, dtype, out_idx);
  if (arg != TKS_OK || batch == 0) return arg;
  if (batch > TKS_NOALLOC_MAX_ROWS) return TKS_E_TOO_LARGE;

  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return TKS_E_UNSUPPORTED;
  }
  DeviceInfo d;
  unsigned char* ws = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_mu);
    const int rc = device_info(dev, &d);
    if (rc != TKS_OK) return rc;
    auto it = g_noalloc_addr.find(dev);
    if (it == g_noalloc_addr.end()) {
      // Host code only sees a stand-in for the array; its device address is
      // looked up once per device, with that device current.
      void* ptr = nullptr;
      if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || ptr == nullptr) {
        cudaGetLastError();
        return TKS_E_CUDA;
      }
      it = g_noalloc_addr.emplace(dev, static_cast<unsigned char*>(ptr)).first;
    }
    ws = it->second;
  }
  int group = 1, grid = 1;
  plan_launch(d, batch, row_stride, &group, &grid);

  // The array keeps whatever the previous call left: clear the status word and
  // the counters of the rows used, and mark their candidate words unwritten.
  const cudaStream_t s = (cudaStream_t)stream;
  const size_t zero_bytes = kWsHeaderBytes + (group > 1 ? (size_t)batch * kSlotBytes : 0);
  if (cudaMemsetAsync(ws, 0, zero_bytes, s) != cudaSuccess ||
      (group > 1 && cudaMemsetAsync(ws + kWsHeaderBytes + (size_t)TKS_NOALLOC_MAX_ROWS * kSlotBytes, 0xFF,
                                    (size_t)batch * kCandSlotBytes, s) != cudaSuccess)) {
    cudaGetLastError();
    return TKS_E_CUDA;
  }

  Params p{};
  p.logits = static_cast<const unsigned char*>(logits);
  p.row_len = row_len;
  p.row_stride = row_stride;
  p.batch = batch;
  p.k = k;
  p.out = out_idx;
  p.group = group;
  p.test_skip_arrive = 0;
  p.ws = ws;
  p.slots = TKS_NOALLOC_MAX_ROWS;
  p.spin_limit_ns = g_spin_limit_ns.load();
  p.cluster = 0;
  p.host_src = 0;
  p.chunk = slice_chunk(row_stride, group, dtype);
  const bool lean = group > 1 && slices_fit_on_chip(row_stride, group, dtype);

  cudaLaunchConfig_t cfg;
  std::memset(&cfg, 0, sizeof cfg);
  cfg.gridDim = dim3((unsigned)grid, 1, 1);
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  set_launch_attrs(&cfg, attr, group);
  const cudaError_t e = plan_threads(batch, row_stride, dtype, group) == 512
                            ? k512::launch_select(cfg, p, dtype, lean)
                            : k256::launch_select(cfg, p, dtype, lean);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return TKS_E_CUDA;
  }
  return TKS_OK;
}
