// Device building blocks of the top-k selector: the order-preserving key map,
// the digit schedule, block-wide scans, histogram updates, TMA bulk copies and
// bounded waits.  Written for sm_103a (GB300).
#pragma once

#include <cstdint>

namespace tks {

// ---------------------------------------------------------------------------
// Shape constants
// ---------------------------------------------------------------------------
constexpr int kThreads = 1024;               // one block per SM, 32 warps
constexpr int kWarps = kThreads / 32;
constexpr int kMaxDigitBits = 12;            // widest digit: 4096 bins (16 KiB of counters)
constexpr int kMaxBins = 1 << kMaxDigitBits;
constexpr int kMaxRounds = 6;                // fp32: 3 key digits + up to 3 position digits
constexpr int kSliceBytes = 160 * 1024;      // on-chip copy of a block's slice of the row
constexpr int kLocalCandCap = 6144;          // (key, position) pairs kept by a lone block
constexpr int kGroupCandCap = kSliceBytes / 8;  // pairs the finishing block can hold
constexpr int kChunks = 4;                   // bulk copies (and mbarriers) per slice

// Dynamic shared memory layout.
constexpr int kHistOff = 0;
constexpr int kCtlOff = kHistOff + kMaxBins * 4;
constexpr int kCtlBytes = 1024;
constexpr int kSliceOff = kCtlOff + kCtlBytes;
constexpr int kLocalCandOff = kSliceOff + kSliceBytes;
constexpr int kSmemBytes = kLocalCandOff + kLocalCandCap * 8;  // 230400 B <= 227 KiB

// Device status bits (kept in the workspace, read by tks_device_status).
constexpr unsigned kStatTimeout = 1u << 0;
constexpr unsigned kStatRowLen = 1u << 1;
constexpr unsigned kStatInternal = 1u << 2;

// Per-row workspace for rows split over several blocks ("slot").
struct SlotHdr {
  unsigned arrive;           // barrier arrivals, monotonic within a call
  unsigned done;             // blocks finished with the row
  unsigned long long alloc;  // low 32 bits: output slots taken; high 32: candidates pushed
  unsigned pad[12];
};
static_assert(sizeof(SlotHdr) == 64, "slot header is one 64-byte line");
constexpr size_t kSlotHistOff = sizeof(SlotHdr);
constexpr size_t kSlotCandOff = kSlotHistOff + size_t(kMaxRounds) * kMaxBins * 4;
constexpr size_t kSlotBytes = (kSlotCandOff + size_t(kGroupCandCap) * 8 + 255) & ~size_t(255);
constexpr size_t kWsHeaderBytes = 256;  // status word + padding

// Shared-memory control block.
struct Ctl {
  unsigned long long mbar[kChunks];
  unsigned long long warp64[kWarps];
  unsigned warp32[kWarps];
  unsigned pick_bin, pick_above, pick_cnt;
  unsigned ok;
  unsigned long long base64;
  unsigned out_count;
  unsigned cand_count;
  unsigned is_last;
};
static_assert(sizeof(Ctl) <= kCtlBytes, "control block fits");

// ---------------------------------------------------------------------------
// Keys: the "Mapping" step.  Negative floats have every bit flipped, the rest
// get the sign bit set; unsigned order of the result equals the float order,
// with -0.0 just below +0.0, -inf lowest and subnormals in place.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t key_f32(uint32_t u) {
  return u ^ ((uint32_t)((int32_t)u >> 31) | 0x80000000u);
}
__device__ __forceinline__ uint32_t key_bf16(uint32_t u16) {
  return (u16 ^ ((uint32_t)((int32_t)(u16 << 16) >> 31) | 0x8000u)) & 0xFFFFu;
}

// ---------------------------------------------------------------------------
// Digit schedule.  The composite key of a position is (value key, inverted
// position): ranking by it descending is exactly the selector's order, and it
// is unique, so digit selection always ends with an exact threshold.
//   fp32 value keys: 12 + 10 + 10 bits; bf16: 12 + 4 bits;
//   then the inverted position, ceil(log2 len) bits, in digits of <= 12 bits.
// ---------------------------------------------------------------------------
struct Digit {
  int on_pos;  // 0: value key, 1: inverted position
  int shift;
  int bits;
};

template <int DT>
__device__ __forceinline__ int key_rounds() { return DT == 0 ? 3 : 2; }

template <int DT>
__device__ __forceinline__ Digit digit_of_round(int t, int pos_bits) {
  if (DT == 0) {
    if (t == 0) return {0, 20, 12};
    if (t == 1) return {0, 10, 10};
    if (t == 2) return {0, 0, 10};
    t -= 3;
  } else {
    if (t == 0) return {0, 4, 12};
    if (t == 1) return {0, 0, 4};
    t -= 2;
  }
  int rem = pos_bits - 12 * t;
  int b = rem < 12 ? rem : 12;
  return {1, rem - b, b};
}

template <int DT>
__device__ __forceinline__ int num_rounds(int pos_bits) {
  return key_rounds<DT>() + (pos_bits + 11) / 12;
}

// Resolved leading bits of the composite key and their chosen values.
struct Prefix {
  uint32_t kmask, kpref, pmask, ppref;
};

__device__ __forceinline__ void prefix_extend(Prefix& p, Digit d, uint32_t bin) {
  uint32_t m = ((1u << d.bits) - 1u) << d.shift;
  if (d.on_pos) {
    p.pmask |= m;
    p.ppref |= bin << d.shift;
  } else {
    p.kmask |= m;
    p.kpref |= bin << d.shift;
  }
}

// Compare the resolved leading bits of (key, inv) with the prefix: 1 above, 0 equal, -1 below.
__device__ __forceinline__ int prefix_cmp(const Prefix& p, uint32_t key, uint32_t inv) {
  uint32_t a = key & p.kmask;
  if (a != p.kpref) return a > p.kpref ? 1 : -1;
  uint32_t b = inv & p.pmask;
  if (b != p.ppref) return b > p.ppref ? 1 : -1;
  return 0;
}

__device__ __forceinline__ uint32_t digit_value(Digit d, uint32_t key, uint32_t inv) {
  return ((d.on_pos ? inv : key) >> d.shift) & ((1u << d.bits) - 1u);
}

// ---------------------------------------------------------------------------
// Small PTX helpers
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ unsigned long long globaltimer_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ unsigned ld_acquire_u32(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ unsigned ld_cg_u32(const unsigned* p) {
  unsigned v;
  asm volatile("ld.global.cg.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ unsigned long long ld_cg_u64(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.global.cg.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ uint2 ld_cg_u2(const uint2* p) {
  uint2 v;
  asm volatile("ld.global.cg.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void red_add_u32(unsigned* p, unsigned v) {
  asm volatile("red.relaxed.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ uint4 ld_nc_v4(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// mbarrier + bulk copy (TMA, non-tensor form).
__device__ __forceinline__ void mbar_init(unsigned long long* bar, unsigned count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(unsigned long long* bar, unsigned bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(unsigned long long* bar, unsigned parity) {
  unsigned ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ void bulk_copy_g2s(void* dst, const void* src, unsigned bytes,
                                              unsigned long long* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// ---------------------------------------------------------------------------
// Block-wide scans (kThreads threads, all must call)
// ---------------------------------------------------------------------------

// Sum of v over threads with a higher index (exclusive suffix sum).  *total gets the sum.
__device__ __forceinline__ unsigned block_suffix_excl(unsigned v, unsigned* total, Ctl* ctl) {
  const unsigned lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  unsigned x = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    unsigned y = __shfl_down_sync(0xffffffffu, x, off);
    if (lane + off < 32) x += y;
  }
  // x = sum over lanes >= lane
  if (lane == 0) ctl->warp32[warp] = x;
  __syncthreads();
  if (warp == 0) {
    unsigned w = ctl->warp32[lane];
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      unsigned y = __shfl_down_sync(0xffffffffu, w, off);
      if (lane + off < 32) w += y;
    }
    ctl->warp32[lane] = w;  // sum over warps >= lane
  }
  __syncthreads();
  unsigned higher_warps = warp + 1 < kWarps ? ctl->warp32[warp + 1] : 0u;
  *total = ctl->warp32[0];
  unsigned r = (x - v) + higher_warps;
  __syncthreads();  // warp32 reusable afterwards
  return r;
}

// Exclusive prefix sum of a 64-bit value over threads in index order; *total gets the sum.
__device__ __forceinline__ unsigned long long block_prefix_excl64(unsigned long long v,
                                                                  unsigned long long* total,
                                                                  Ctl* ctl) {
  const unsigned lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  unsigned long long x = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    unsigned long long y = __shfl_up_sync(0xffffffffu, x, off);
    if (lane >= (unsigned)off) x += y;
  }
  if (lane == 31) ctl->warp64[warp] = x;
  __syncthreads();
  if (warp == 0) {
    unsigned long long w = ctl->warp64[lane];
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      unsigned long long y = __shfl_up_sync(0xffffffffu, w, off);
      if (lane >= (unsigned)off) w += y;
    }
    ctl->warp64[lane] = w;  // inclusive over warps <= lane
  }
  __syncthreads();
  unsigned long long lower = warp > 0 ? ctl->warp64[warp - 1] : 0ull;
  *total = ctl->warp64[kWarps - 1];
  unsigned long long r = (x - v) + lower;
  __syncthreads();
  return r;
}

// ---------------------------------------------------------------------------
// Histogram update, called by all 32 lanes of a warp.  When every valid lane
// of the warp hits the same bin (constant or plateau rows) one lane adds the
// whole count; otherwise each valid lane adds one.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void hist_add(unsigned* h, uint32_t d, bool valid) {
  const unsigned full = 0xffffffffu;
  unsigned vm = __ballot_sync(full, valid);
  if (vm == 0) return;
  int first = __ffs(vm) - 1;
  uint32_t d0 = __shfl_sync(full, d, first);
  bool same = __all_sync(full, !valid || d == d0);
  if (same) {
    if ((int)(threadIdx.x & 31) == first) atomicAdd(&h[d0], (unsigned)__popc(vm));
  } else if (valid) {
    atomicAdd(&h[d], 1u);
  }
}

// ---------------------------------------------------------------------------
// Threshold scan: the bin holding the k_rem-th largest element (1-based) of
// the histogram, the count strictly above it and its own count.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void find_bin(const unsigned* h, int nb, unsigned k_rem, Ctl* ctl) {
  const int per = (nb + kThreads - 1) / kThreads;
  const int b0 = threadIdx.x * per;
  unsigned s = 0;
  for (int i = 0; i < per; ++i) {
    int b = b0 + i;
    if (b < nb) s += h[b];
  }
  unsigned total;
  unsigned above = block_suffix_excl(s, &total, ctl);
  if (s != 0 && above < k_rem && k_rem <= above + s) {
    unsigned acc = above;
    for (int i = per - 1; i >= 0; --i) {
      int b = b0 + i;
      if (b >= nb) continue;
      unsigned c = h[b];
      if (k_rem <= acc + c) {
        ctl->pick_bin = (unsigned)b;
        ctl->pick_above = acc;
        ctl->pick_cnt = c;
        break;
      }
      acc += c;
    }
  }
  __syncthreads();
}

}  // namespace tks
