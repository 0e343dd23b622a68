// The selection kernel built with 512 threads per block (namespace tks::k512),
// used for rows split into large slices; see tks_kernel.cuh.
#define TKS_THREADS 512
#define TKS_VARIANT k512
#include "tks_kernel.cuh"

namespace tks {
static_assert(k512::kSmemBytes == 230400 && k512::kSlotBytes > 0,
              "the 512-thread kernel shares the 256-thread kernel's layout");
}  // namespace tks
