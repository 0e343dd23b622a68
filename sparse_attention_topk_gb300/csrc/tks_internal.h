// Internal interface between the translation units of libtks (not part of
// the C ABI).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace tks {

// Arguments of the selection kernel (both block sizes).
struct Params {
  const unsigned char* logits;
  const int32_t* row_len;
  int64_t row_stride;
  int32_t batch;
  int32_t k;
  int32_t* out;
  int32_t group;
  int32_t test_skip_arrive;
  unsigned char* ws;
  int32_t slots;
  long long spin_limit_ns;
  int32_t cluster;  // 1: each row's `group` blocks form one thread-block cluster
  int32_t host_src; // 1: logits and row lengths are page-locked host memory (plain loads only)
  int32_t chunk;    // slice length of a row of row_stride elements split over `group` blocks
};

// The selection kernel's launcher and set-up for each block size (256 and 512
// threads): launch_select fills in the block size and shared memory of `base`;
// setup_select opts in to the shared memory and to clusters of up to 16 blocks and
// reports the blocks per SM and the largest cluster the device schedules.
namespace k256 {
cudaError_t launch_select(const cudaLaunchConfig_t& base, const Params& p, int32_t dtype,
                          bool lean);
bool setup_select(int* blocks_per_sm, int* max_cluster);
}  // namespace k256
namespace k512 {
cudaError_t launch_select(const cudaLaunchConfig_t& base, const Params& p, int32_t dtype,
                          bool lean);
bool setup_select(int* blocks_per_sm, int* max_cluster);
}  // namespace k512

// Largest k tks_topk_indices_sorted accepts: a row's k composite keys are
// sorted in one block's shared memory.
constexpr int kOrderKMax = 16384;

// Enqueues the rank ordering of out[batch][k] on `stream`: each row's
// selected positions (k slots, -1 for none) are reordered by value key
// descending, then position ascending, -1 slots last.  logits and dtype are
// those of the selection that wrote out.  Waits (programmatic dependency) for
// the kernel ahead of it in the stream before reading out.
cudaError_t launch_rank_order(const void* logits, int32_t batch, int64_t row_stride, int32_t k,
                              int32_t dtype, int32_t* out, cudaStream_t stream);

// The same order for at most kRankMaxRows rows of k <= kRankKMax, spread over
// many blocks: reads the unordered selection sel[batch][k] (device memory the
// call owns, written by the kernel ahead in the stream) and writes the ordered
// rows to out.
constexpr int kRankMaxRows = 8;
constexpr int kRankKMax = 4096;
cudaError_t launch_rank_order_rows(const void* logits, int32_t batch, int64_t row_stride,
                                   int32_t k, int32_t dtype, const int32_t* sel, int32_t* out,
                                   cudaStream_t stream);

}  // namespace tks
