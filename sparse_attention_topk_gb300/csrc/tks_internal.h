// Internal interface between the translation units of libtks (not part of
// the C ABI).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace tks {

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

}  // namespace tks
