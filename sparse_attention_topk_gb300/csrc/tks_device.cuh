// Device building blocks of the top-k selector: the order-preserving key map,
// the digit schedule, block-wide scans, histogram and slot counters, bulk
// asynchronous copies and bounded waits.  Written for sm_103a (GB300).
#pragma once

#include <cstdint>

#ifndef TKS_VARIANT
#define TKS_VARIANT k256
#endif

namespace tks {
namespace TKS_VARIANT {

// ---------------------------------------------------------------------------
// Shape constants
// ---------------------------------------------------------------------------
// 256 threads per block, one block per SM.  Control steps (scans, threshold
// search, bookkeeping) are issued once per warp, so fewer warps make them
// faster; the streaming steps are bound by data, not by the warp count.
#ifndef TKS_THREADS
#define TKS_THREADS 256
#endif
constexpr int kThreads = TKS_THREADS;
constexpr int kWarps = kThreads / 32;
constexpr int kMaxDigitBits = 12;            // widest digit: 4096 bins (16 KiB of counters)
constexpr int kMaxBins = 1 << kMaxDigitBits;
constexpr int kMaxRounds = 6;                // fp32: 3 key digits + up to 3 position digits
constexpr int kSliceBytes = 160 * 1024;      // on-chip copy of a block's slice of the row
constexpr int kLocalCandCap = 4096;          // (key, position) pairs kept by a lone block
constexpr int kGroupCandCap = kSliceBytes / 8;  // pairs the finishing block can hold
#ifndef TKS_CHUNKS
#define TKS_CHUNKS 1
#endif
constexpr int kChunks = TKS_CHUNKS;          // bulk copies (and mbarriers) per slice
constexpr int kPassVecs = 4;                 // vectors a thread loads per step of a pass

// Dynamic shared memory layout.
constexpr int kHistOff = 0;                          // counts, then exclusive suffix sums
constexpr int kOffsOff = kHistOff + kMaxBins * 4;    // this block's offset inside each bin
constexpr int kCtlOff = kOffsOff + kMaxBins * 4;
constexpr int kCtlBytes = 1024;
constexpr int kSliceOff = kCtlOff + kCtlBytes;
constexpr int kLocalCandOff = kSliceOff + kSliceBytes;
constexpr int kSmemBytes = kLocalCandOff + kLocalCandCap * 8;  // 230400 B <= 227 KiB

// Device status bits (kept in the workspace, read by tks_device_status).
constexpr unsigned kStatTimeout = 1u << 0;
constexpr unsigned kStatRowLen = 1u << 1;
constexpr unsigned kStatInternal = 1u << 2;

// Per-row workspace for rows split over several blocks ("slot").  Calls on
// a slot alternate between two sets of counters by the parity of `epoch`, so
// the set a call uses was cleared during the previous call and nothing has to
// be reset at the end of a call.
struct SlotHdr {
  unsigned epoch;       // calls that used this slot so far
  unsigned used[2];     // digit rounds the last call of each parity used
  // Candidate words [0, cand_dirty) the last call left written: the next call
  // puts them back to all ones before its first row barrier.
  unsigned cand_dirty;
  // Per parity, in one 16-byte word so that one load reads them together:
  // barrier arrivals (monotonic within a call), 1 + the highest nonempty
  // first-digit bin of the row (0 = none yet), and the highest of the blocks'
  // first-round floors (no block's floor lies above the row's threshold bin).
  struct alignas(16) {
    unsigned arrive;
    unsigned top;
    unsigned floor;
    unsigned pad;
  } sync[2];
  // Per parity: OR of the row's first-round keys and OR of their complements
  // (their AND, inverted, so that both start from zero): equal iff every key
  // of the row is the same.
  unsigned keyset[2][2];
};
static_assert(sizeof(SlotHdr) == 64, "slot header is one 64-byte line");
constexpr size_t kSlotHistOff = sizeof(SlotHdr);
constexpr size_t kSlotHistWords = size_t(kMaxRounds) * kMaxBins;  // per parity
constexpr size_t kSlotBytes = (kSlotHistOff + 2 * kSlotHistWords * 4 + 255) & ~size_t(255);
// Candidate slots: one 64-bit word (key | position << 32) each; all ones
// means "not written yet" (a position is always below 2^31).
constexpr size_t kCandSlotBytes = size_t(kGroupCandCap) * 8;
constexpr unsigned long long kCandEmpty = ~0ull;
constexpr size_t kWsHeaderBytes = 256;  // status word + padding

// Shared-memory control block.
struct Ctl {
  unsigned long long mbar[kChunks];
  unsigned warp32[kWarps + 1];
  unsigned pick_bin, pick_above, pick_cnt;
  unsigned ok;
  unsigned top;
  unsigned lo;                 // first-round floor bin of this block
  unsigned sink;               // keeps an atomic's returned value live
  unsigned kor, knand;         // OR of the keys and OR of their complements: block's, then row's
  unsigned red[4 * kWarps];
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

__device__ __forceinline__ unsigned lane_id() { return threadIdx.x & 31u; }

// Programmatic dependent launch: let the next grid of the stream be scheduled
// early / wait until the previous grid of the stream is complete and its
// memory operations are visible.
__device__ __forceinline__ void grid_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void grid_dependency_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

// Plain global loads (also valid on page-locked host memory mapped into the
// device's address space).
__device__ __forceinline__ uint4 ld_v4(const void* p) {
  uint4 v;
  asm volatile("ld.global.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}
__device__ __forceinline__ int ld_s32(const int32_t* p) {
  int v;
  asm volatile("ld.global.s32 %0, [%1];" : "=r"(v) : "l"(p));
  return v;
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
// The logits are read exactly once: ask L2 to evict them first, so they do
// not push the kernel's own counters and candidates out.
__device__ __forceinline__ void bulk_copy_g2s(void* dst, const void* src, unsigned bytes,
                                              unsigned long long* bar, unsigned long long policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, "
      "[%3], %4;" ::"r"(smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}
__device__ __forceinline__ unsigned long long policy_evict_first() {
  unsigned long long p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// ---------------------------------------------------------------------------
// Block-wide scan (kThreads threads, all must call): sum of v over threads
// with a higher index.  *total gets the sum over all threads.  scratch holds
// kWarps words (ctl->warp32 by default); without the trailing barrier the
// caller must pass a barrier before scratch is written again.
// ---------------------------------------------------------------------------
__device__ __forceinline__ unsigned block_suffix_excl(unsigned v, unsigned* total, Ctl* ctl,
                                                      unsigned* scratch = nullptr,
                                                      bool trailing_sync = true) {
  const unsigned lane = lane_id(), warp = threadIdx.x >> 5;
  if (scratch == nullptr) scratch = ctl->warp32;
  unsigned x = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    unsigned y = __shfl_down_sync(0xffffffffu, x, off);
    if (lane + off < 32) x += y;
  }
  // x = sum over lanes >= lane of this warp
  if (lane == 0) scratch[warp] = x;
  __syncthreads();
  unsigned higher = 0, all = 0;
#pragma unroll
  for (int w = 0; w < kWarps; ++w) {
    const unsigned s = scratch[w];
    all += s;
    if (w > (int)warp) higher += s;
  }
  *total = all;
  if (trailing_sync) __syncthreads();  // scratch reusable afterwards
  return (x - v) + higher;
}

// ---------------------------------------------------------------------------
// Threshold scan over h[0..nb): the bin holding the k_rem-th largest element
// (1-based), the count strictly above it and its own count.  Rewrites h in
// place into exclusive suffix sums (h[i] = number of elements in bins > i),
// which later give every emitted element its output slot.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void note_pick(Ctl* ctl, unsigned bin, unsigned above, unsigned c,
                                          unsigned k_rem) {
  if (above < k_rem && k_rem <= above + c) {
    ctl->pick_bin = bin;
    ctl->pick_above = above;
    ctl->pick_cnt = c;
  }
}

// The same over bins [lo, hi) only, up to 4 bins per thread (hi - lo <=
// 4 * kThreads); bins outside the range are neither read nor written.
__device__ __forceinline__ void pick_and_suffix_range(unsigned* h, int lo, int hi, unsigned k_rem,
                                                      Ctl* ctl) {
  const int n = hi - lo;
  const int per = (n + kThreads - 1) / kThreads;  // 0..4
  const int b0 = lo + (int)threadIdx.x * per;
  unsigned c[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) c[i] = (i < per && b0 + i < hi) ? h[b0 + i] : 0u;
  const unsigned s = c[0] + c[1] + c[2] + c[3];
  unsigned total;
  unsigned acc = block_suffix_excl(s, &total, ctl);
#pragma unroll
  for (int i = 3; i >= 0; --i) {
    if (i < per && b0 + i < hi) {
      note_pick(ctl, (unsigned)(b0 + i), acc, c[i], k_rem);
      h[b0 + i] = acc;
    }
    acc += c[i];
  }
  __syncthreads();
}

__device__ __forceinline__ void pick_and_suffix(unsigned* h, int nb, unsigned k_rem, Ctl* ctl) {
  const unsigned lane = lane_id(), warp = threadIdx.x >> 5;
  if (nb >= kWarps * 128) {
    // Warp w owns a contiguous run of 128*Q bins; lane l reads 16-byte vector
    // q*32 + l of it, so every access is conflict-free.  Bin order inside the
    // run is (q, lane, element).
    const int Q = nb / (kWarps * 128);  // 1, 2 or 4
    uint4* h4 = reinterpret_cast<uint4*>(h) + warp * 32 * Q;
    uint4 v[4];
    unsigned tot[4], sq[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      v[q] = q < Q ? h4[q * 32 + lane] : make_uint4(0u, 0u, 0u, 0u);
      const unsigned t = v[q].x + v[q].y + v[q].z + v[q].w;
      unsigned x = t;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const unsigned y = __shfl_down_sync(0xffffffffu, x, off);
        if (lane + off < 32) x += y;
      }
      sq[q] = x - t;                                 // lanes above, same q
      tot[q] = __shfl_sync(0xffffffffu, x, 0);       // all lanes, same q
    }
    unsigned above_q[4], acc = 0;
#pragma unroll
    for (int q = 3; q >= 0; --q) {
      above_q[q] = acc;
      acc += tot[q];
    }
    if (lane == 0) ctl->warp32[warp] = acc;
    __syncthreads();
    unsigned higher = 0;
#pragma unroll
    for (int w = 0; w < kWarps; ++w)
      if (w > (int)warp) higher += ctl->warp32[w];
    const unsigned base_bin = warp * 128 * Q + lane * 4;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      if (q >= Q) continue;
      unsigned a = higher + above_q[q] + sq[q];
      const unsigned bq = base_bin + q * 128;
      uint4 o;
      o.w = a; note_pick(ctl, bq + 3, a, v[q].w, k_rem); a += v[q].w;
      o.z = a; note_pick(ctl, bq + 2, a, v[q].z, k_rem); a += v[q].z;
      o.y = a; note_pick(ctl, bq + 1, a, v[q].y, k_rem); a += v[q].y;
      o.x = a; note_pick(ctl, bq + 0, a, v[q].x, k_rem);
      h4[q * 32 + lane] = o;
    }
    __syncthreads();
    return;
  }
  // Small digits: thread t owns `per` consecutive bins.
  pick_and_suffix_range(h, 0, nb, k_rem, ctl);
}

// Block-wide OR and AND of per-thread partial results for two words
// (all threads call; every thread gets the totals).
__device__ __forceinline__ void block_or_and(uint32_t& or_a, uint32_t& and_a, uint32_t& or_b,
                                             uint32_t& and_b, Ctl* ctl) {
  or_a = __reduce_or_sync(0xffffffffu, or_a);
  and_a = __reduce_and_sync(0xffffffffu, and_a);
  or_b = __reduce_or_sync(0xffffffffu, or_b);
  and_b = __reduce_and_sync(0xffffffffu, and_b);
  const unsigned warp = threadIdx.x >> 5;
  if (lane_id() == 0) {
    ctl->red[4 * warp + 0] = or_a;
    ctl->red[4 * warp + 1] = and_a;
    ctl->red[4 * warp + 2] = or_b;
    ctl->red[4 * warp + 3] = and_b;
  }
  __syncthreads();
  or_a = 0u; and_a = ~0u; or_b = 0u; and_b = ~0u;
#pragma unroll
  for (int w = 0; w < kWarps; ++w) {
    or_a |= ctl->red[4 * w + 0];
    and_a &= ctl->red[4 * w + 1];
    or_b |= ctl->red[4 * w + 2];
    and_b &= ctl->red[4 * w + 3];
  }
  __syncthreads();
}

__device__ __forceinline__ void red_release_add_u32(unsigned* p, unsigned v) {
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Thread-block clusters: shared memory of another block of the cluster
// (distributed shared memory) and the cluster barrier.
__device__ __forceinline__ uint32_t dsmem_map(const void* p, unsigned rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_u32(p)), "r"(rank));
  return r;
}
__device__ __forceinline__ unsigned dsmem_atom_add(uint32_t addr, unsigned v) {
  unsigned old;
  asm volatile("atom.shared::cluster.add.u32 %0, [%1], %2;" : "=r"(old) : "r"(addr), "r"(v) : "memory");
  return old;
}
__device__ __forceinline__ void dsmem_red_max(uint32_t addr, unsigned v) {
  asm volatile("red.shared::cluster.max.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}
__device__ __forceinline__ unsigned dsmem_ld(uint32_t addr) {
  unsigned v;
  asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
  return v;
}
__device__ __forceinline__ void cluster_arrive() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ uint4 ld_acquire_v4(const void* p) {
  uint4 v;
  asm volatile("ld.acquire.gpu.global.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p)
               : "memory");
  return v;
}

__device__ __forceinline__ unsigned long long ld_acquire_u64(const void* p) {
  unsigned long long v;
  asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

// Predicated forms (no branch around the access): a shared-memory add and a
// global store that happen only when p holds.
__device__ __forceinline__ void red_shared_add_if(bool p, unsigned* addr, unsigned v) {
  asm volatile(
      "{\n\t.reg .pred q;\n\tsetp.ne.u32 q, %0, 0;\n\t@q red.shared.add.u32 [%1], %2;\n\t}" ::"r"(
          (unsigned)p),
      "r"(smem_u32(addr)), "r"(v)
      : "memory");
}
__device__ __forceinline__ void st_global_s32_if(bool p, int32_t* addr, int32_t v) {
  asm volatile("{\n\t.reg .pred q;\n\tsetp.ne.u32 q, %0, 0;\n\t@q st.global.s32 [%1], %2;\n\t}" ::"r"(
                   (unsigned)p),
               "l"(addr), "r"(v)
               : "memory");
}

// Candidate words in global memory, written and polled without caching.
__device__ __forceinline__ void st_relaxed_u64(unsigned long long* p, unsigned long long v) {
  asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ unsigned long long ld_relaxed_u64(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ uint4 ld_relaxed_v4(const void* p) {
  uint4 v;
  asm volatile("ld.relaxed.gpu.global.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p)
               : "memory");
  return v;
}

}  // namespace TKS_VARIANT
}  // namespace tks
