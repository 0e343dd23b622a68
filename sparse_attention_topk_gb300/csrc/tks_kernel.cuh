// Device code of the top-k selector: element sources, the digit rounds, the
// cross-block merge, emission and the on-chip finish, and the kernel.  Included
// once per block size: TKS_THREADS threads per block, in namespace
// tks::TKS_VARIANT (k256: tks_select.cu, k512: tks_select512.cu).
#pragma once

#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>

#include "tks.h"
#include "tks_device.cuh"
#include "tks_internal.h"

// 1: the first-round histogram of resident slices uses warp-aggregated adds
// (a measurement build; the library proper uses plain shared-memory adds).
#ifndef TKS_HIST_AGGREGATE
#define TKS_HIST_AGGREGATE 0
#endif

namespace tks {
namespace TKS_VARIANT {


template <int DT>
struct Elt;
template <>
struct Elt<0> {  // fp32
  static constexpr int ES = 4;
  static constexpr int V = 4;
  static constexpr int kShift0 = 20;
  __device__ static __forceinline__ uint32_t key(uint32_t raw) { return key_f32(raw); }
  __device__ static __forceinline__ uint32_t lane(const uint4& x, int j) {
    return j == 0 ? x.x : j == 1 ? x.y : j == 2 ? x.z : x.w;
  }
  __device__ static __forceinline__ uint32_t load(const unsigned char* row, int i) {
    return *reinterpret_cast<const uint32_t*>(row + (int64_t)i * 4);
  }
  __device__ static __forceinline__ void store(unsigned char* dst, uint32_t raw) {
    *reinterpret_cast<uint32_t*>(dst) = raw;
  }
  // For a threshold key t0 of a value >= +0.0 (top key bit set): key(raw) >=
  // t0 exactly when the raw bits, read as a signed integer, are >= sthr(t0)
  // (negative values have the sign bit set and lie below every such value).
  __device__ static __forceinline__ int sraw(const uint4& x, int j) { return (int)lane(x, j); }
  __device__ static __forceinline__ int sthr(uint32_t t0) { return (int)(t0 ^ 0x80000000u); }
  static constexpr uint32_t kKeyTop = 0x80000000u;
};
template <>
struct Elt<1> {  // bf16
  static constexpr int ES = 2;
  static constexpr int V = 8;
  static constexpr int kShift0 = 4;
  __device__ static __forceinline__ uint32_t key(uint32_t raw) { return key_bf16(raw); }
  __device__ static __forceinline__ uint32_t lane(const uint4& x, int j) {
    uint32_t w = (j >> 1) == 0 ? x.x : (j >> 1) == 1 ? x.y : (j >> 1) == 2 ? x.z : x.w;
    return (j & 1) ? (w >> 16) : (w & 0xFFFFu);
  }
  __device__ static __forceinline__ uint32_t load(const unsigned char* row, int i) {
    return *reinterpret_cast<const uint16_t*>(row + (int64_t)i * 2);
  }
  __device__ static __forceinline__ void store(unsigned char* dst, uint32_t raw) {
    *reinterpret_cast<uint16_t*>(dst) = (uint16_t)raw;
  }
  // (as for fp32, on the 16-bit patterns)
  __device__ static __forceinline__ int sraw(const uint4& x, int j) {
    const uint32_t w = (j >> 1) == 0 ? x.x : (j >> 1) == 1 ? x.y : (j >> 1) == 2 ? x.z : x.w;
    return (j & 1) ? (int)w >> 16 : (int)(w << 16) >> 16;
  }
  __device__ static __forceinline__ int sthr(uint32_t t0) { return (int)(int16_t)(uint16_t)(t0 ^ 0x8000u); }
  static constexpr uint32_t kKeyTop = 0x8000u;
};

// One block's share of a row.
struct Slice {
  int lo, hi;  // positions [lo, hi)
  int bl, bh;  // 16-byte aligned body [bl, bh)
  int o;       // position held by byte 0 of the on-chip copy
  int nvec;    // 16-byte vectors of the on-chip copy
  int vb0;     // first whole vector of the body in the on-chip copy (0 or 1)
  int nbv;     // whole vectors in the body
  bool resident;
};

// ---------------------------------------------------------------------------
// Element sources.  visit(f) calls f(key[U], pos[U], vm) for groups of U
// elements, bit j of vm set when element j is real.  Each thread walks its
// own groups independently (f must not use warp-wide operations): shared
// memory atomics on GB300 absorb same-address conflicts inside a warp, so a
// plain strided loop with plain atomics is the fastest form of every pass.
// ---------------------------------------------------------------------------
template <int DT>
struct SliceSrc {
  static constexpr int U = Elt<DT>::V;
  const unsigned char* row;  // the row in global memory
  const unsigned char* sm;   // on-chip copy (resident slices)
  Slice s;
  bool plain;                // plain loads only (the row is in host memory)

  template <class F>
  __device__ __forceinline__ void vec(const uint4& x, int i0, unsigned vm, F& f) const {
    using E = Elt<DT>;
    uint32_t key[U];
    int pos[U];
#pragma unroll
    for (int j = 0; j < U; ++j) {
      key[j] = E::key(E::lane(x, j));
      pos[j] = i0 + j;
    }
    f(key, pos, vm);
  }

  // Whole vectors [va, vb) of the on-chip copy, four loads in flight per
  // thread (each iteration is otherwise one serial chain of latencies).
  template <class F>
  __device__ __forceinline__ void visit_range(int va, int vb, F&& f) const {
    constexpr int B = kPassVecs;
    const uint4* sv = reinterpret_cast<const uint4*>(sm);
    for (int v0 = va + (int)threadIdx.x; v0 < vb; v0 += B * kThreads) {
      uint4 x[B];
#pragma unroll
      for (int b = 0; b < B; ++b) {
        const int v = v0 + b * kThreads;
        x[b] = v < vb ? sv[v] : make_uint4(0u, 0u, 0u, 0u);
      }
#pragma unroll
      for (int b = 0; b < B; ++b) {
        const int v = v0 + b * kThreads;
        if (v < vb) vec(x[b], s.o + v * U, (1u << U) - 1u, f);
      }
    }
  }

  // The first-round histogram with warp-aggregated adds (the build with
  // TKS_HIST_AGGREGATE=1, kept to measure that choice against the plain adds
  // of visit_range): the lanes of a warp that hold the same bin (match_any)
  // add their count with one atomic.  Every lane runs the same number of
  // steps, as match_any needs all 32.
  __device__ __forceinline__ void hist_aggregated(int va, int vb, unsigned* h) const {
    using E = Elt<DT>;
    const uint4* sv = reinterpret_cast<const uint4*>(sm);
    for (int v0 = va; v0 < vb; v0 += kThreads) {
      const int v = v0 + (int)threadIdx.x;
      const uint4 x = v < vb ? sv[v] : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
      for (int j = 0; j < U; ++j) {
        const uint32_t bin = E::key(E::lane(x, j)) >> E::kShift0;
        const unsigned m = __match_any_sync(0xffffffffu, v < vb ? bin : 0xFFFFFFFFu);
        if (v < vb && __ffs((int)m) - 1 == (int)lane_id()) atomicAdd(&h[bin], (unsigned)__popc(m));
      }
    }
  }

  // The partial first and last vectors of the on-chip copy (threads 0 and 1).
  template <class F>
  __device__ __forceinline__ void visit_edges(F&& f) const {
    const int head = s.vb0 ? 0 : -1;
    const int tail = s.vb0 + s.nbv < s.nvec ? s.vb0 + s.nbv : -1;
    const int v = threadIdx.x == 0 ? head : threadIdx.x == 1 ? tail : -1;
    if (v < 0 || (threadIdx.x == 1 && tail == head)) return;
    const int i0 = s.o + v * U;
    unsigned vm = (1u << U) - 1u;
    if (i0 < s.lo) vm &= ~0u << (s.lo - i0);
    if (i0 + U > s.hi) vm &= (1u << max(0, s.hi - i0)) - 1u;
    vec(reinterpret_cast<const uint4*>(sm)[v], i0, vm, f);
  }

  // The body's whole vectors by plain loads from global memory into the
  // on-chip copy, each counted on the way (the first pass of a row held in
  // host memory, where bulk copies are not used).
  template <class F>
  __device__ __forceinline__ void load_visit_body(unsigned char* dst, F&& f) const {
    using E = Elt<DT>;
    const uint4* body = reinterpret_cast<const uint4*>(row + (int64_t)s.bl * E::ES);
    uint4* out = reinterpret_cast<uint4*>(dst) + s.vb0;
    const int nv = s.nbv;
    constexpr int kAhead = 8;
    for (int v0 = (int)threadIdx.x; v0 < nv; v0 += kAhead * kThreads) {
      uint4 x[kAhead];
#pragma unroll
      for (int a = 0; a < kAhead; ++a) {
        const int v = v0 + a * kThreads;
        x[a] = v < nv ? ld_v4(body + v) : make_uint4(0u, 0u, 0u, 0u);
      }
#pragma unroll
      for (int a = 0; a < kAhead; ++a) {
        const int v = v0 + a * kThreads;
        if (v < nv) {
          out[v] = x[a];
          vec(x[a], s.bl + v * U, (1u << U) - 1u, f);
        }
      }
    }
  }

  // Straight from global memory (slices too large to keep on chip).
  template <class F>
  __device__ __forceinline__ void visit_global(F&& f) const {
    using E = Elt<DT>;
    const int nh = s.bl - s.lo, nt = s.hi - s.bh;
    if ((int)threadIdx.x < nh + nt) {  // the unaligned head and tail, one element per thread
      const int i = (int)threadIdx.x < nh ? s.lo + (int)threadIdx.x : s.bh + ((int)threadIdx.x - nh);
      uint32_t key[U];
      int pos[U];
#pragma unroll
      for (int j = 0; j < U; ++j) {
        key[j] = E::key(j == 0 ? E::load(row, i) : 0u);
        pos[j] = i;
      }
      f(key, pos, 1u);
    }
    const uint4* body = reinterpret_cast<const uint4*>(row + (int64_t)s.bl * E::ES);
    const int nv = (s.bh - s.bl) / U;
    constexpr int kAhead = 4;
    for (int v0 = (int)threadIdx.x; v0 < nv; v0 += kAhead * kThreads) {
      uint4 x[kAhead];
#pragma unroll
      for (int a = 0; a < kAhead; ++a) {
        const int v = v0 + a * kThreads;
        x[a] = v >= nv ? make_uint4(0u, 0u, 0u, 0u) : plain ? ld_v4(body + v) : ld_nc_v4(body + v);
      }
#pragma unroll
      for (int a = 0; a < kAhead; ++a) {
        const int v = v0 + a * kThreads;
        if (v < nv) vec(x[a], s.bl + v * U, (1u << U) - 1u, f);
      }
    }
  }

  template <class F>
  __device__ __forceinline__ void visit(F&& f) const {
    if (s.resident) {
      visit_range(s.vb0, s.vb0 + s.nbv, f);
      visit_edges(f);
    } else {
      visit_global(f);
    }
  }
};

// (key, position) pairs in shared memory, four per call (strided by the
// block size, so the loads of a warp are contiguous).
struct CandSrc {
  static constexpr int U = 4;
  const uint2* c;
  unsigned n;
  template <class F>
  __device__ __forceinline__ void visit(F&& f) const {
    for (unsigned i0 = threadIdx.x; i0 < n; i0 += U * kThreads) {
      uint32_t key[U];
      int pos[U];
      unsigned vm = 0u;
#pragma unroll
      for (int j = 0; j < U; ++j) {
        const unsigned i = i0 + j * kThreads;
        const uint2 e = i < n ? c[i] : make_uint2(0u, 0u);
        key[j] = e.x;
        pos[j] = (int)e.y;
        vm |= (i < n ? 1u : 0u) << j;
      }
      f(key, pos, vm);
    }
  }
};

// ---------------------------------------------------------------------------
// Block-level steps
// ---------------------------------------------------------------------------

// Zeroes counters [0, n) (n rounded up to a multiple of 4; arrays hold kMaxBins).
__device__ __forceinline__ void zero_counters(unsigned* h, int n) {
  uint4* h4 = reinterpret_cast<uint4*>(h);
  for (int i = threadIdx.x; i < (n + 3) / 4; i += kThreads) h4[i] = make_uint4(0u, 0u, 0u, 0u);
}

// Largest valid key of a group of U elements (0 if none).
template <int U>
__device__ __forceinline__ uint32_t key_max(const uint32_t (&key)[U], unsigned vm) {
  uint32_t a = 0u;
#pragma unroll
  for (int j = 0; j < U; ++j) a = max(a, ((vm >> j) & 1u) ? key[j] : 0u);
  return a;
}

// Histogram of digit D over the elements that match the prefix.
template <class Src>
__device__ __forceinline__ void hist_round(const Src& src, unsigned* h, const Prefix& P, Digit D,
                                           uint32_t pmax) {
  constexpr int U = Src::U;
  src.visit([&](const uint32_t(&key)[U], const int(&pos)[U], unsigned vm) {
#pragma unroll
    for (int j = 0; j < U; ++j) {
      const uint32_t inv = pmax - (uint32_t)pos[j];
      if (((vm >> j) & 1u) && prefix_cmp(P, key[j], inv) == 0)
        atomicAdd(&h[digit_value(D, key[j], inv)], 1u);
    }
  });
}

// Spin (bounded) until a bulk copy's mbarrier phase completes.  On time-out
// records the error and clears ctl->ok; returns either way.
__device__ __forceinline__ void mbar_wait_bounded(unsigned long long* bar, unsigned parity,
                                                  long long limit, Ctl* ctl, unsigned* status) {
  if (mbar_try_wait(bar, parity)) return;
  const unsigned long long t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if ((long long)(globaltimer_ns() - t0) > limit) {
      ctl->ok = 0u;
      atomicOr(status, kStatTimeout);
      return;
    }
  }
}

// The row barrier after a merge, then the row's counts of bins [lo, top)
// replace the local ones in h[].  When use_top (the first round), top is the
// row's maximum and lo is raised to the row's highest floor (both from the
// word beside the arrival count), else top is nb; they are left in ctl->lo
// and ctl->top.  Bounded: on time-out records the error and returns false.
__device__ __forceinline__ bool merge_wait_load(unsigned* h, int lo, int nb, const unsigned* g,
                                                unsigned* sync_word, bool use_top, unsigned target,
                                                bool skip_arrive, long long limit, Ctl* ctl,
                                                unsigned* status) {
  constexpr int kPer = kMaxBins / kThreads;
  if (threadIdx.x == 0) {
    // release: this block's adds (all returned before the caller's barrier)
    // are visible to any block that sees the arrival
    if (!skip_arrive) red_release_add_u32(&sync_word[0], 1u);
    unsigned ok = 1u;
    uint4 w = ld_acquire_v4(sync_word);
    if (w.x < target) {
      const unsigned long long t0 = globaltimer_ns();
      while ((w = ld_acquire_v4(sync_word)).x < target) {
        if ((long long)(globaltimer_ns() - t0) > limit) {
          ok = 0u;
          atomicOr(status, kStatTimeout);
          break;
        }
      }
    }
    ctl->top = use_top ? min((unsigned)nb, w.y) : (unsigned)nb;
    ctl->lo = use_top ? max((unsigned)lo, w.z) : (unsigned)lo;
    ctl->ok = ok;
  }
  __syncthreads();
  if (!ctl->ok) return false;
  const int top = (int)ctl->top;
  lo = (int)ctl->lo;
  if (top - lo <= kThreads) {
    const int b = lo + (int)threadIdx.x;
    if (b < top) h[b] = __ldcg(g + b);
  } else {
    unsigned c[kPer];
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
      const int b = j * kThreads + threadIdx.x;
      c[j] = (b >= lo && b < top) ? __ldcg(g + b) : 0u;
    }
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
      const int b = j * kThreads + threadIdx.x;
      if (b >= lo && b < top) h[b] = c[j];
    }
  }
  __syncthreads();
  return true;
}

// Adds this block's counts of all nb bins into the row's L2 histogram g
// (rounds after the first).  The value each add returns is this block's
// offset inside that bin across the row, kept in offs[] to place the block's
// elements in the output later without any further coordination.  Then the
// row barrier and the row's counts in h[0, nb).
__device__ __forceinline__ bool group_merge(unsigned* h, unsigned* offs, int nb, unsigned* g,
                                            unsigned* sync_pair, unsigned target, long long limit,
                                            Ctl* ctl, unsigned* status) {
  constexpr int kPer = kMaxBins / kThreads;
  unsigned c[kPer];
#pragma unroll
  for (int j = 0; j < kPer; ++j) {
    const int b = j * kThreads + threadIdx.x;
    c[j] = b < nb ? h[b] : 0u;
  }
#pragma unroll
  for (int j = 0; j < kPer; ++j) c[j] = c[j] ? atomicAdd(&g[j * kThreads + threadIdx.x], c[j]) : 0u;
#pragma unroll
  for (int j = 0; j < kPer; ++j) {
    const int b = j * kThreads + threadIdx.x;
    if (b < nb) offs[b] = c[j];
  }
  __syncthreads();
  return merge_wait_load(h, 0, nb, g, sync_pair, false, target, false, limit, ctl, status);
}

// Round 0: this block's bounds and, for a row split over blocks, the merge.
// A bin can hold the row's threshold only if fewer than k of this block's
// elements lie above it (the row's k-th largest is at least this block's k-th
// largest): the lowest such bin is the block's floor, *lo.  *hi is 1 + the
// highest nonempty bin, of the row when split, else of the block.  Both come
// from one block-wide scan over per-thread sums of kPer consecutive bins.
// When split, the block's counts of bins [*lo, block top) go into the row's
// L2 histogram g (warp-wide adds over consecutive bins; the value each add
// returns is this block's offset inside the bin, kept in offs[]), the block
// top into the word beside the arrival count, and after the row barrier
// h[*lo, *hi) holds the row's counts.
__device__ __forceinline__ bool round0_bounds_merge(unsigned* h, unsigned* offs, unsigned k,
                                                    bool split, unsigned* g, unsigned* sync_pair,
                                                    unsigned target, bool skip_arrive,
                                                    long long limit, Ctl* ctl, unsigned* status,
                                                    int* lo, int* hi, unsigned* gh, bool* cl_pending) {
  constexpr int kPer = kMaxBins / kThreads;
  constexpr int Q = kPer / 4;  // 16-byte vectors of bins per thread
  static_assert(kPer % 4 == 0 && 8 % Q == 0, "bins per thread");
  const int b0 = (int)threadIdx.x * kPer;
  // The sum of my bins, reading my vectors in a rotated order so that the
  // lanes of a warp spread over all banks.
  unsigned S = 0u;
#pragma unroll
  for (int q = 0; q < Q; ++q) {
    const uint4 v = reinterpret_cast<const uint4*>(h + b0)[(q + (int)threadIdx.x / (8 / Q)) % Q];
    S += (v.x + v.y) + (v.z + v.w);
  }
  unsigned total;
  // (the scan's scratch is ctl->red, not needed again before the next barrier)
  const unsigned A = block_suffix_excl(S, &total, ctl, ctl->red, false);  // elements above my bins
  const bool floor_mine = A < k && (threadIdx.x == 0 || A + S >= k);
  const bool top_mine = A == 0u && S != 0u;  // my bins hold the highest nonempty one
  if (floor_mine || top_mine) {
    unsigned c[kPer];
#pragma unroll
    for (int q = 0; q < Q; ++q) {
      const uint4 v = reinterpret_cast<const uint4*>(h + b0)[q];
      c[4 * q] = v.x;
      c[4 * q + 1] = v.y;
      c[4 * q + 2] = v.z;
      c[4 * q + 3] = v.w;
    }
    // the floor: the lowest of my bins with fewer than k above it
    unsigned above = A;
    int f = 0, tj = 0;
#pragma unroll
    for (int j = kPer - 1; j >= 0; --j) {
      if (above < k) f = j;
      above += c[j];
    }
#pragma unroll
    for (int j = 0; j < kPer; ++j)
      if (c[j] != 0u) tj = j;
    if (floor_mine) ctl->lo = (unsigned)(b0 + f);
    if (top_mine) ctl->top = (unsigned)(b0 + tj + 1);
  }
  if (total == 0u && threadIdx.x == 0) ctl->top = 0u;
  __syncthreads();
  const int l = (int)ctl->lo, top = (int)ctl->top;
  *lo = l;
  if (!split) {
    *hi = top;
    return true;
  }
  if (gh != nullptr) {
    unsigned c[kPer];
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
      const int b = j * kThreads + threadIdx.x;
      c[j] = (b >= l && b < top) ? h[b] : 0u;
    }
    // The row is one thread-block cluster: the adds go to block 0's shared
    // histogram gh (distributed shared memory), each returning this block's
    // offset inside the bin; the cluster barrier replaces the L2 barrier.
    cluster_wait();  // every block has cleared its gh (each arrived when it did)
    const uint32_t g0 = dsmem_map(gh, 0u);
    unsigned r2[kPer];
#pragma unroll
    for (int j = 0; j < kPer; ++j)
      r2[j] = c[j] ? dsmem_atom_add(g0 + 4u * (j * kThreads + threadIdx.x), c[j]) : 0u;
    if (threadIdx.x == 0 && top > 0) dsmem_red_max(g0 + 4u * kMaxBins, (unsigned)top);
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
      const int b = j * kThreads + threadIdx.x;
      if (b >= l && b < top) offs[b] = r2[j];
    }
    cluster_arrive();  // every block's adds are done
    cluster_wait();
    const int rtop = (int)min((unsigned)kMaxBins, dsmem_ld(g0 + 4u * kMaxBins));
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
      const int b = j * kThreads + threadIdx.x;
      if (b >= l && b < rtop) h[b] = dsmem_ld(g0 + 4u * b);
    }
    // done with block 0's words; the matching wait comes before the block exits
    cluster_arrive();
    *cl_pending = true;
    __syncthreads();
    *hi = rtop;
    return ctl->ok != 0u;
  }
  // the bins of the window [l, top), one per thread: add, keep the offset
  for (int b = l + (int)threadIdx.x; b < top; b += kThreads) {
    const unsigned cb = h[b];
    offs[b] = cb ? atomicAdd(&g[b], cb) : 0u;
  }
  // atomics with return, so they have been performed by the arrival
  if (threadIdx.x == 0) {
    const unsigned a = top > 0 ? atomicMax(&sync_pair[1], (unsigned)top) : 0u;
    ctl->sink = a + atomicMax(&sync_pair[2], (unsigned)l);
  }
  __syncthreads();  // also: every thread has read ctl->top before it is rewritten
  if (!merge_wait_load(h, l, kMaxBins, g, sync_pair, true, target, skip_arrive, limit, ctl, status))
    return false;
  *lo = (int)ctl->lo;
  *hi = (int)ctl->top;
  return true;
}

// Finds the threshold bin among bins [lo, hi) of h[0..nb) (the caller knows
// it lies there) and turns those bins into exclusive suffix sums; false (and
// an error) if the counts are inconsistent, which cannot happen unless memory
// was corrupted.
__device__ __forceinline__ bool pick_bin_range(unsigned* h, int lo, int hi, int nb, unsigned k_rem,
                                               Ctl* ctl, unsigned* status, unsigned* bin,
                                               unsigned* above, unsigned* cnt) {
  if (threadIdx.x == 0) ctl->pick_bin = 0xFFFFFFFFu;
  if (hi - lo <= 4 * kThreads) {
    pick_and_suffix_range(h, lo, hi, k_rem, ctl);
  } else {
    for (int i = threadIdx.x; i < nb; i += kThreads)
      if (i < lo || i >= hi) h[i] = 0u;
    __syncthreads();
    pick_and_suffix(h, nb, k_rem, ctl);
  }
  *bin = ctl->pick_bin;
  *above = ctl->pick_above;
  *cnt = ctl->pick_cnt;
  if (*bin == 0xFFFFFFFFu) {
    if (threadIdx.x == 0) atomicOr(status, kStatInternal);
    return false;
  }
  return true;
}

// Finds the threshold bin of h[0..nb) and turns h into exclusive suffix sums;
// false (and an error) if the counts are inconsistent, which cannot happen
// unless memory was corrupted.
// The bin of h[0, nb) holding the k_rem-th largest count from the top, with
// the count above it and its own count (into ctl->pick_*), from one
// block-wide scan over per-thread sums of kPer consecutive bins.  Leaves no
// suffix sums behind.
__device__ __forceinline__ void pick_scan(const unsigned* h, int nb, unsigned k_rem, Ctl* ctl) {
  constexpr int kPer = kMaxBins / kThreads;
  static_assert(kPer % 4 == 0, "bins per thread");
  const int b0 = (int)threadIdx.x * kPer;
  unsigned c[kPer];
  if (b0 + kPer <= nb) {
#pragma unroll
    for (int q = 0; q < kPer / 4; ++q) {
      const uint4 v = reinterpret_cast<const uint4*>(h + b0)[q];
      c[4 * q] = v.x;
      c[4 * q + 1] = v.y;
      c[4 * q + 2] = v.z;
      c[4 * q + 3] = v.w;
    }
  } else {
#pragma unroll
    for (int j = 0; j < kPer; ++j) c[j] = b0 + j < nb ? h[b0 + j] : 0u;
  }
  unsigned S = 0u;
#pragma unroll
  for (int j = 0; j < kPer; ++j) S += c[j];
  unsigned total;
  const unsigned A = block_suffix_excl(S, &total, ctl);
  if (A < k_rem && A + S >= k_rem) {
    unsigned above = A;
#pragma unroll
    for (int j = kPer - 1; j >= 0; --j) {
      if (above < k_rem && above + c[j] >= k_rem) {
        ctl->pick_bin = (unsigned)(b0 + j);
        ctl->pick_above = above;
        ctl->pick_cnt = c[j];
      }
      above += c[j];
    }
  }
  __syncthreads();
}

__device__ __forceinline__ bool pick_bin(unsigned* h, int nb, unsigned k_rem, Ctl* ctl,
                                         unsigned* status, unsigned* bin, unsigned* above,
                                         unsigned* cnt) {
  if (threadIdx.x == 0) ctl->pick_bin = 0xFFFFFFFFu;
  pick_scan(h, nb, k_rem, ctl);
  *bin = ctl->pick_bin;
  *above = ctl->pick_above;
  *cnt = ctl->pick_cnt;
  if (*bin == 0xFFFFFFFFu) {
    if (threadIdx.x == 0) atomicOr(status, kStatInternal);
    return false;
  }
  return true;
}

// What happens to the elements of the threshold round's bins.
enum RoundEnd {
  kEndFinal = 0,    // the threshold bin is taken whole: emit bins >= bin
  kEndCollect = 1,  // emit bins > bin, bin's elements become candidates
  kEndAbove = 2     // emit bins > bin, another digit round follows
};

// Stores a candidate (key, position) as one 64-bit word.  Global slots are
// polled by the finishing block, so they are written with a single relaxed
// store that is never torn.
__device__ __forceinline__ void put_cand(uint2* cand, unsigned i, uint32_t key, int pos,
                                         bool global) {
  const unsigned long long w = (unsigned long long)key | ((unsigned long long)(uint32_t)pos << 32);
  if (global)
    st_relaxed_u64(reinterpret_cast<unsigned long long*>(cand) + i, w);
  else
    reinterpret_cast<unsigned long long*>(cand)[i] = w;
}

// One pass over the source: every element that matches the prefix before
// this round and lands in an emitted bin goes to output slot
//   base + (elements of the row in higher bins) + (its rank inside its bin),
// the rank coming from this block's running offset offs[bin]; candidates go
// to cand[offs[bin]++].
template <class Src>
__device__ __forceinline__ void emit_round(const Src& src, const Prefix& P, Digit D, unsigned bin, int end,
                           unsigned base, const unsigned* suf, unsigned* offs, uint32_t pmax,
                           int32_t* out_row, unsigned k, uint2* cand, bool cand_global,
                           unsigned cap, unsigned* status) {
  constexpr int U = Src::U;
  bool bad = false;
  // Every emitted element has (key & qmask) >= qval, and that part of the
  // key is monotone in the key: groups whose largest key fails it are skipped.
  uint32_t qmask = P.kmask, qval = P.kpref;
  if (!D.on_pos) {
    qmask |= ((1u << D.bits) - 1u) << D.shift;
    qval |= bin << D.shift;
  }
  src.visit([&](const uint32_t(&key)[U], const int(&pos)[U], unsigned vm) {
    if ((key_max<U>(key, vm) & qmask) < qval) return;  // nothing here reaches the threshold
#pragma unroll
    for (int j = 0; j < U; ++j) {
      const uint32_t inv = pmax - (uint32_t)pos[j];
      if (!((vm >> j) & 1u) || prefix_cmp(P, key[j], inv) != 0) continue;
      const uint32_t d = digit_value(D, key[j], inv);
      const bool to_cand = end == kEndCollect && d == bin;
      if (!(d > bin || (end == kEndFinal && d == bin) || to_cand)) continue;
      const unsigned o = atomicAdd(&offs[d], 1u);  // rank inside the bin, row-wide
      if (to_cand) {
        if (o < cap)
          put_cand(cand, o, key[j], pos[j], cand_global);
        else
          bad = true;
      } else {
        const unsigned slot = base + suf[d] + o;
        if (slot < k)
          out_row[slot] = pos[j];
        else
          bad = true;
      }
    }
  });
  if (bad) atomicOr(status, kStatInternal);
}

// First-round emission from a resident slice, as a plain pass: whole vectors
// (four loads in flight per thread), one compare per element (in the first
// round an element is written exactly when its key reaches t0), and the
// write path only for the elements that pass.  The partial edge vectors go
// through visit_edges.
// (suf[d - suf_lo]: the row's elements in the bins above bin d)
template <int DT>
__device__ __forceinline__ void emit_first_resident(const SliceSrc<DT>& src, uint32_t t0,
                                                    const Digit& D, unsigned bin, int end,
                                                    unsigned base, const unsigned* suf, int suf_lo,
                                                    unsigned* offs, int32_t* out_row, unsigned k,
                                                    uint2* cand, bool cand_global, unsigned cap,
                                                    unsigned* status) {
  using E = Elt<DT>;
  constexpr int U = E::V;
  constexpr int B = kPassVecs;
  bool bad = false;
  // an element of bin d with rank o inside the bin
  auto place = [&](uint32_t key, int pos, uint32_t d, unsigned o) {
    if (end == kEndCollect && d == bin) {
      if (o < cap)
        put_cand(cand, o, key, pos, cand_global);
      else
        bad = true;
    } else {
      const unsigned slot = base + suf[(int)d - suf_lo] + o;
      if (slot < k)
        out_row[slot] = pos;
      else
        bad = true;
    }
  };
  auto write = [&](uint32_t key, int pos) {
    const uint32_t d = key >> D.shift;
    place(key, pos, d, atomicAdd(&offs[d], 1u));  // rank inside the bin, row-wide
  };
  const Slice& s = src.s;
  const uint4* sv = reinterpret_cast<const uint4*>(src.sm);
  const int va = s.vb0, vb = s.vb0 + s.nbv;
  const int st0 = E::sthr(t0);
  for (int v0 = va + (int)threadIdx.x; v0 < vb; v0 += B * kThreads) {
    uint4 x[B];
#pragma unroll
    for (int b = 0; b < B; ++b) {
      const int v = v0 + b * kThreads;
      x[b] = v < vb ? sv[v] : make_uint4(0u, 0u, 0u, 0u);
    }
    // which of the B * U elements are written (a compact unrolled test) ...
    unsigned sel = 0u;
    if (t0 >= E::kKeyTop) {
#pragma unroll
      for (int b = 0; b < B; ++b) {
        const int v = v0 + b * kThreads;
#pragma unroll
        for (int j = 0; j < U; ++j) sel |= (v < vb && E::sraw(x[b], j) >= st0 ? 1u : 0u) << (b * U + j);
      }
    } else {
#pragma unroll
      for (int b = 0; b < B; ++b) {
        const int v = v0 + b * kThreads;
#pragma unroll
        for (int j = 0; j < U; ++j)
          sel |= (v < vb && E::key(E::lane(x[b], j)) >= t0 ? 1u : 0u) << (b * U + j);
      }
    }
    // ... then one copy of the write path for those (rare) elements, keys
    // re-read from shared memory, so the loop stays small; two at a time, so
    // that two chains of (load, atomic, store) latencies overlap
    while (sel) {
      const int q0 = __ffs((int)sel) - 1;
      sel &= sel - 1u;
      const int q1 = sel ? __ffs((int)sel) - 1 : -1;
      sel &= sel - 1u;
      const int pos0 = s.o + (v0 + (q0 / U) * kThreads) * U + q0 % U;
      const int pos1 = s.o + (v0 + (max(q1, 0) / U) * kThreads) * U + max(q1, 0) % U;
      const uint32_t key0 = E::key(E::load(src.sm, pos0 - s.o));  // resident: on chip
      const uint32_t key1 = E::key(E::load(src.sm, pos1 - s.o));
      const uint32_t d0 = key0 >> D.shift, d1 = key1 >> D.shift;
      const unsigned o0 = atomicAdd(&offs[d0], 1u);
      const unsigned o1 = q1 >= 0 ? atomicAdd(&offs[d1], 1u) : 0u;
      place(key0, pos0, d0, o0);
      if (q1 >= 0) place(key1, pos1, d1, o1);
    }
  }
  src.visit_edges([&](const uint32_t(&key)[U], const int(&pos)[U], unsigned vm) {
#pragma unroll
    for (int j = 0; j < U; ++j)
      if (((vm >> j) & 1u) && key[j] >= t0) write(key[j], pos[j]);
  });
  if (bad) atomicOr(status, kStatInternal);
}

// A later round over a resident slice as a plain pass (as emit_first_resident):
// elements that match the prefix P go into the digit-D histogram h (count)
// or, when emitting, are written if their digit is above bin (or equal, per
// end).  Vectors whose largest key cannot match P are skipped.
template <int DT, bool kEmit>
__device__ __forceinline__ void later_pass_resident(const SliceSrc<DT>& src, const Prefix& P,
                                                    const Digit& D, uint32_t pmax, unsigned* h,
                                                    unsigned bin, int end, unsigned base,
                                                    const unsigned* suf, unsigned* offs,
                                                    int32_t* out_row, unsigned k, uint2* cand,
                                                    bool cand_global, unsigned cap,
                                                    unsigned* status) {
  using E = Elt<DT>;
  constexpr int U = E::V;
  constexpr int B = kPassVecs;
  bool bad = false;
  auto element = [&](uint32_t key, int pos) {
    const uint32_t inv = pmax - (uint32_t)pos;
    if ((key & P.kmask) != P.kpref || (inv & P.pmask) != P.ppref) return;
    const uint32_t d = digit_value(D, key, inv);
    if (!kEmit) {
      atomicAdd(&h[d], 1u);
      return;
    }
    if (d < bin || (d == bin && end == kEndAbove)) return;
    const unsigned o = atomicAdd(&offs[d], 1u);  // rank inside the bin, row-wide
    if (end == kEndCollect && d == bin) {
      if (o < cap)
        put_cand(cand, o, key, pos, cand_global);
      else
        bad = true;
    } else {
      const unsigned slot = base + suf[d] + o;
      if (slot < k)
        out_row[slot] = pos;
      else
        bad = true;
    }
  };
  // keys at or above this can match the prefix (it is a leading-bits prefix)
  const uint32_t kmin = P.kpref;
  const Slice& s = src.s;
  const uint4* sv = reinterpret_cast<const uint4*>(src.sm);
  const int va = s.vb0, vb = s.vb0 + s.nbv;
  for (int v0 = va + (int)threadIdx.x; v0 < vb; v0 += B * kThreads) {
    uint4 x[B];
#pragma unroll
    for (int b = 0; b < B; ++b) {
      const int v = v0 + b * kThreads;
      x[b] = v < vb ? sv[v] : make_uint4(0u, 0u, 0u, 0u);
    }
    if (!kEmit) {
      // counting: a few operations per element, all inline
#pragma unroll
      for (int b = 0; b < B; ++b) {
        const int v = v0 + b * kThreads;
        if (v >= vb) continue;
#pragma unroll
        for (int j = 0; j < U; ++j) {
          const uint32_t key = E::key(E::lane(x[b], j));
          if (key < kmin) continue;
          const int pos = s.o + v * U + j;
          const uint32_t inv = pmax - (uint32_t)pos;
          if ((key & P.kmask) == P.kpref && (inv & P.pmask) == P.ppref)
            atomicAdd(&h[digit_value(D, key, inv)], 1u);
        }
      }
    } else {
      // emitting: which elements are written (a compact unrolled test), then
      // one copy of the write path for those, so the loop stays small
      unsigned sel = 0u;
#pragma unroll
      for (int b = 0; b < B; ++b) {
        const int v = v0 + b * kThreads;
#pragma unroll
        for (int j = 0; j < U; ++j) {
          const uint32_t key = E::key(E::lane(x[b], j));
          const uint32_t inv = pmax - (uint32_t)(s.o + v * U + j);
          const uint32_t d = digit_value(D, key, inv);
          const bool w = v < vb && (key & P.kmask) == P.kpref && (inv & P.pmask) == P.ppref &&
                         (d > bin || (d == bin && end != kEndAbove));
          sel |= (w ? 1u : 0u) << (b * U + j);
        }
      }
      while (sel) {
        const int q = __ffs((int)sel) - 1;
        sel &= sel - 1u;
        const int pos = s.o + (v0 + (q / U) * kThreads) * U + q % U;
        element(E::key(E::load(src.sm, pos - s.o)), pos);  // resident: on chip
      }
    }
  }
  src.visit_edges([&](const uint32_t(&key)[U], const int(&pos)[U], unsigned vm) {
#pragma unroll
    for (int j = 0; j < U; ++j)
      if ((vm >> j) & 1u) element(key[j], pos[j]);
  });
  if (bad) atomicOr(status, kStatInternal);
}

// The highest still-varying bits (at most `width`) of the composite key:
// value key first, then the inverted position.  False when nothing varies.
__device__ __forceinline__ bool next_digit(uint32_t& vk, uint32_t& vp, int width, Digit* D) {
  const bool on_pos = vk == 0u;
  uint32_t& v = on_pos ? vp : vk;
  if (!v) return false;
  const int hi = 31 - __clz((int)v);
  const int lowest = __ffs((int)v) - 1;  // no digit reaches below the lowest varying bit
  const int lo = max(lowest, hi >= width - 1 ? hi - (width - 1) : 0);
  *D = {on_pos ? 1 : 0, lo, hi - lo + 1};
  v &= ~(((1u << (hi - lo + 1)) - 1u) << lo);
  return true;
}

// Digit width for a round over n elements: about two bins per element, so the
// threshold bin usually ends up with one element (and the rounds end), while
// small candidate sets get small, cheap histograms.
__device__ __forceinline__ int digit_width(unsigned n) {
  const int lg = 32 - __clz((int)max(n, 1u));  // ceil-ish log2(n) + 1
  return min(kMaxDigitBits, max(4, lg + 1));
}

// Refines candidates held on chip until the k_rem wanted among them are
// known, then writes them after the k - k_rem already emitted.  Bits that are
// equal in every candidate join the prefix at once; digits are taken from the
// highest bits that still differ, so no round is spent on a constant digit.
// (or_*, and_*: OR and AND of the candidates' keys and inverted positions.)
__device__ __forceinline__ void finish_on_chip(const uint2* cand, unsigned n, unsigned k_rem, Prefix P,
                               uint32_t or_k, uint32_t and_k, uint32_t or_i, uint32_t and_i,
                               uint32_t pmax, unsigned* h, int32_t* out_row, unsigned k, Ctl* ctl,
                               unsigned* status) {
  const CandSrc src{cand, n};
  const unsigned out_base = k - k_rem;
  uint32_t vk = (or_k ^ and_k) & ~P.kmask;
  uint32_t vp = (or_i ^ and_i) & pmax & ~P.pmask;
  const uint32_t ck = ~(or_k ^ and_k) & ~P.kmask, cp = ~(or_i ^ and_i) & pmax & ~P.pmask;
  P.kmask |= ck;
  P.kpref |= and_k & ck;
  P.pmask |= cp;
  P.ppref |= and_i & cp;
  unsigned live = n;  // elements matching the prefix
  for (;;) {
    Digit D;
    if (!next_digit(vk, vp, digit_width(live), &D)) {
      if (threadIdx.x == 0) atomicOr(status, kStatInternal);
      return;
    }
    const int nb = 1 << D.bits;
    zero_counters(h, nb);
    __syncthreads();
    hist_round(src, h, P, D, pmax);
    __syncthreads();
    unsigned bin, above, cnt;
    if (!pick_bin(h, nb, k_rem, ctl, status, &bin, &above, &cnt)) return;
    prefix_extend(P, D, bin);
    k_rem -= above;
    if (cnt == k_rem) break;
    live = cnt;
  }
  // Write every candidate at or above the final prefix into consecutive
  // slots: count per warp, scan over warps, then each warp writes its
  // selected candidates in order (coalesced stores).
  const unsigned lane = lane_id(), warp = threadIdx.x >> 5;
  constexpr int B = 4;
  const unsigned iters = (n + B * kThreads - 1) / (B * kThreads);
  unsigned mine = 0u;
  for (unsigned it = 0; it < iters; ++it) {
    uint2 e[B];
#pragma unroll
    for (int b = 0; b < B; ++b) {
      const unsigned i = (it * B + b) * kThreads + threadIdx.x;
      e[b] = i < n ? cand[i] : make_uint2(0u, 0u);
    }
#pragma unroll
    for (int b = 0; b < B; ++b) {
      const unsigned i = (it * B + b) * kThreads + threadIdx.x;
      const bool sel = i < n && prefix_cmp(P, e[b].x, pmax - e[b].y) >= 0;
      mine += (unsigned)__popc(__ballot_sync(0xffffffffu, sel));
    }
  }
  if (lane == 0) ctl->warp32[warp] = mine;
  __syncthreads();
  unsigned wbase = out_base;
#pragma unroll
  for (int w = 0; w < kWarps; ++w)
    if (w < (int)warp) wbase += ctl->warp32[w];
  bool bad = false;
  const unsigned lt = (1u << lane) - 1u;
  for (unsigned it = 0; it < iters; ++it) {
    uint2 e[B];
#pragma unroll
    for (int b = 0; b < B; ++b) {
      const unsigned i = (it * B + b) * kThreads + threadIdx.x;
      e[b] = i < n ? cand[i] : make_uint2(0u, 0u);
    }
#pragma unroll
    for (int b = 0; b < B; ++b) {
      const unsigned i = (it * B + b) * kThreads + threadIdx.x;
      const bool sel = i < n && prefix_cmp(P, e[b].x, pmax - e[b].y) >= 0;
      const unsigned m = __ballot_sync(0xffffffffu, sel);
      if (sel) {
        const unsigned slot = wbase + (unsigned)__popc(m & lt);
        if (slot < k)
          out_row[slot] = (int)e[b].y;
        else
          bad = true;
      }
      wbase += (unsigned)__popc(m);
    }
  }
  if (bad) atomicOr(status, kStatInternal);
}

// Digits of the register finisher are at most kPickBits wide, so that one
// warp finds the threshold bin among kPickBins counters.
constexpr int kPickBits = 8;
constexpr int kPickBins = 1 << kPickBits;

// The threshold bin of a digit round: the bin holding the k_rem-th largest
// element, the count above it and its own count (bin all ones when the counts
// hold fewer than k_rem elements).
struct Pick {
  unsigned bin, above, cnt;
};

// Every lane of the calling warp gets the pick over the counts h[0,
// kPickBins).  Lane l owns bins [8l, 8l + 8), read in an order that spreads
// the lanes over all banks; a suffix scan over the lanes finds the lane that
// holds the threshold, which broadcasts its bin.
__device__ __forceinline__ Pick warp_pick(const unsigned* h, unsigned k_rem) {
  static_assert(kPickBins == 256, "eight bins per lane");
  const unsigned lane = lane_id();
  const uint4* h4 = reinterpret_cast<const uint4*>(h) + 2 * lane;
  const bool rot = ((lane >> 2) & 1u) != 0u;
  const uint4 a = h4[rot ? 1 : 0], b = h4[rot ? 0 : 1];
  const uint4 lo4 = rot ? b : a, hi4 = rot ? a : b;
  const unsigned c[8] = {lo4.x, lo4.y, lo4.z, lo4.w, hi4.x, hi4.y, hi4.z, hi4.w};
  const unsigned S = ((c[0] + c[1]) + (c[2] + c[3])) + ((c[4] + c[5]) + (c[6] + c[7]));
  unsigned x = S;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const unsigned y = __shfl_down_sync(0xffffffffu, x, off);
    if (lane + off < 32) x += y;
  }
  const unsigned A = x - S;  // counts in the lanes above
  const bool mine = A < k_rem && A + S >= k_rem;
  unsigned bin = 0u, above = 0u, cnt = 0u, acc = A;
#pragma unroll
  for (int j = 7; j >= 0; --j) {
    if (acc < k_rem && acc + c[j] >= k_rem) {
      bin = 8u * lane + (unsigned)j;
      above = acc;
      cnt = c[j];
    }
    acc += c[j];
  }
  const unsigned m = __ballot_sync(0xffffffffu, mine);
  if (m == 0u) return {0xFFFFFFFFu, 0u, 0u};
  const int src = __ffs((int)m) - 1;
  return {__shfl_sync(0xffffffffu, bin, src), __shfl_sync(0xffffffffu, above, src),
          __shfl_sync(0xffffffffu, cnt, src)};
}

// Every lane of the calling warp gets the pick over the counts h[lo, hi) (at
// most 32 bins, one per lane) for k_rem, and the warp writes the exclusive
// suffix sums of those bins (the elements in the bins above each) to
// sw[b - lo].  No branch around the warp-wide steps.
__device__ __forceinline__ Pick warp_window_pick(const unsigned* h, int lo, int hi, unsigned k_rem,
                                                 unsigned* sw) {
  const unsigned lane = lane_id();
  const int b = lo + (int)lane;
  const bool in = b < hi;
  const unsigned c = in ? h[b] : 0u;
  unsigned x = c;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const unsigned y = __shfl_down_sync(0xffffffffu, x, off);
    x += lane + off < 32 ? y : 0u;
  }
  const unsigned a = x - c;  // the elements in the bins above mine
  if (in) sw[lane] = a;
  const bool found = in && a < k_rem && a + c >= k_rem;
  const unsigned m = __ballot_sync(0xffffffffu, found);
  if (m == 0u) return {0xFFFFFFFFu, 0u, 0u};
  const int src = __ffs((int)m) - 1;
  return {(unsigned)(lo + src), __shfl_sync(0xffffffffu, a, src), __shfl_sync(0xffffffffu, c, src)};
}

// Candidates a thread keeps in registers in the register finisher.
constexpr int kRegCand = 8;
constexpr unsigned kRegCandCap = (unsigned)kRegCand * kThreads;

// A digit over the composite key (value key, inverted position) that may
// span both fields: kb value-key bits from bit klo, then pb position bits
// from bit plo (position bits only once no value-key bit below the digit
// still varies, so digit order stays the composite order).
struct Digit2 {
  int klo, kb, plo, pb;
};

__device__ __forceinline__ bool next_digit2(uint32_t& vk, uint32_t& vp, int width, Digit2* D) {
  D->kb = 0;
  D->pb = 0;
  D->klo = 0;
  D->plo = 0;
  int w = width;
  if (vk) {
    const int hi = 31 - __clz((int)vk);
    const int lo = max(__ffs((int)vk) - 1, hi - (w - 1));
    D->klo = lo;
    D->kb = hi - lo + 1;
    vk &= ~(((1u << D->kb) - 1u) << lo);
    w -= D->kb;
    if (vk) return true;  // lower value-key bits still vary: no position bits yet
  }
  if (w > 0 && vp) {
    const int hi = 31 - __clz((int)vp);
    const int lo = max(__ffs((int)vp) - 1, hi - (w - 1));
    D->plo = lo;
    D->pb = hi - lo + 1;
    vp &= ~(((1u << D->pb) - 1u) << lo);
  }
  return D->kb + D->pb > 0;
}

__device__ __forceinline__ uint32_t digit2_value(const Digit2& D, uint32_t key, uint32_t inv) {
  const uint32_t kpart = (key >> D.klo) & ((1u << D.kb) - 1u);
  const uint32_t ppart = (inv >> D.plo) & ((1u << D.pb) - 1u);
  return (kpart << D.pb) | ppart;
}

// The finish for up to kRegCandCap candidates, held in registers: thread t
// owns candidates t + j * kThreads (j < kRegCand) as (key, inverted
// position) with an `alive` bit (still inside the prefix) and a `sel` bit
// (known to be selected).  A digit round is then one predicated atomic per
// alive candidate and a bit update, with no rereading and no prefix tests.
// Digits cover only bits that differ among the candidates and may run from
// the value key into the position, so ties are usually broken in the same
// round.  Writes the k_rem selected positions after the k - k_rem already
// emitted.
__device__ __forceinline__ void finish_in_registers(const uint32_t (&ck)[kRegCand],
                                                    const uint32_t (&ci)[kRegCand], unsigned alive,
                                                    unsigned k_rem, const Prefix& P, uint32_t or_k,
                                                    uint32_t and_k, uint32_t or_i, uint32_t and_i,
                                                    unsigned n, uint32_t pmax, unsigned* h,
                                                    int32_t* out_row, unsigned k, Ctl* ctl,
                                                    unsigned* status, bool counters_clear = false) {
  const unsigned out_base = k - k_rem;
  uint32_t vk = (or_k ^ and_k) & ~P.kmask;
  uint32_t vp = (or_i ^ and_i) & pmax & ~P.pmask;
  // three sets of kPickBins counters, used by the rounds in turn: a round
  // clears the set the next one counts into, and every warp finds the
  // threshold bin itself, so that a round needs one barrier (the caller may
  // have cleared them already, off the critical path)
  if (!counters_clear) {
    for (int i = threadIdx.x; i < 3 * kPickBins; i += kThreads) h[i] = 0u;
    __syncthreads();
  }
  unsigned sel = 0u;
  unsigned live = n;
  for (int r = 0;; ++r) {
    Digit2 D;
    if (!next_digit2(vk, vp, min(kPickBits, digit_width(live)), &D)) {
      if (threadIdx.x == 0) atomicOr(status, kStatInternal);
      return;
    }
    unsigned* cur = h + (r % 3) * kPickBins;
    unsigned* nxt = h + ((r + 1) % 3) * kPickBins;
    uint32_t d[kRegCand];
#pragma unroll
    for (int j = 0; j < kRegCand; ++j) {
      d[j] = digit2_value(D, ck[j], ci[j]);
      red_shared_add_if((alive >> j) & 1u, &cur[d[j]], 1u);
    }
    for (int i = threadIdx.x; i < kPickBins; i += kThreads) nxt[i] = 0u;
    __syncthreads();
    const Pick pk = warp_pick(cur, k_rem);
    if (pk.bin == 0xFFFFFFFFu) {
      if (threadIdx.x == 0) atomicOr(status, kStatInternal);
      return;
    }
    // (branch-free: a live candidate above the bin is selected, one in it
    // stays live, the rest drop out)
    unsigned up = 0u, in = 0u;
#pragma unroll
    for (int j = 0; j < kRegCand; ++j) {
      up |= (d[j] > pk.bin ? 1u : 0u) << j;
      in |= (d[j] == pk.bin ? 1u : 0u) << j;
    }
    sel |= alive & up;
    alive &= in;
    k_rem -= pk.above;
    if (pk.cnt == k_rem) {
      sel |= alive;
      break;
    }
    live = pk.cnt;
  }
  // Distinct slots from out_base on: each warp takes a run of them after the
  // runs of the warps before it, its lanes place their candidates by ballot
  // ranks (predicated stores, no branch per candidate).
  const unsigned lane = lane_id(), lt = (1u << lane) - 1u, warp = threadIdx.x >> 5;
  unsigned m[kRegCand];
  unsigned wtotal = 0u;
#pragma unroll
  for (int j = 0; j < kRegCand; ++j) {
    m[j] = __ballot_sync(0xffffffffu, (sel >> j) & 1u);
    wtotal += (unsigned)__popc(m[j]);
  }
  if (lane == 0) ctl->warp32[warp] = wtotal;
  __syncthreads();
  unsigned slot = out_base;
#pragma unroll
  for (int w = 0; w < kWarps; ++w) slot += w < (int)warp ? ctl->warp32[w] : 0u;
  bool bad = false;
#pragma unroll
  for (int j = 0; j < kRegCand; ++j) {
    const bool s_j = ((sel >> j) & 1u) != 0u;
    const unsigned sj = slot + (unsigned)__popc(m[j] & lt);
    st_global_s32_if(s_j && sj < k, out_row + sj, (int32_t)(pmax - ci[j]));
    bad |= s_j && sj >= k;
    slot += (unsigned)__popc(m[j]);
  }
  if (bad) atomicOr(status, kStatInternal);
}

// Row r's valid length, clamped into [0, row_stride] (*bad: it was not).
__device__ __forceinline__ uint32_t row_length(const Params& p, int r, bool* bad) {
  int64_t Lr = !p.row_len ? p.row_stride
              : p.host_src ? (int64_t)ld_s32(p.row_len + r) : (int64_t)__ldg(p.row_len + r);
  *bad = Lr < 0 || Lr > p.row_stride;
  if (*bad) Lr = Lr < 0 ? 0 : p.row_stride;
  return (uint32_t)Lr;
}

// Block `part`'s slice of a row of L elements starting at `row`, with 16-byte
// aligned interior boundaries.
// chunk: the slice length for a row of L elements, when the caller knows it
// (0: computed here).
template <int DT>
__device__ __forceinline__ Slice slice_geometry(uint32_t L, int part, int group,
                                                const unsigned char* row, uint32_t chunk = 0u) {
  using E = Elt<DT>;
  const uint32_t V = E::V;
  const uint32_t mis = (uint32_t)(((uintptr_t)row & 15u) / E::ES);
  auto align_up = [&](uint32_t i) -> uint32_t { return i + ((V - ((mis + i) & (V - 1u))) & (V - 1u)); };
  auto align_down = [&](uint32_t i) -> uint32_t { return i - ((mis + i) & (V - 1u)); };
  if (chunk == 0u) chunk = ((L + (uint32_t)group - 1u) / (uint32_t)group + V - 1u) & ~(V - 1u);
  Slice s;
  s.lo = part == 0 ? 0 : (int)min(L, align_up((uint32_t)part * chunk));
  s.hi = part == group - 1 ? (int)L : (int)min(L, align_up((uint32_t)(part + 1) * chunk));
  s.bl = (int)min((uint32_t)s.hi, align_up((uint32_t)s.lo));
  s.bh = max(s.bl, (int)align_down((uint32_t)s.hi));
  s.o = s.lo < s.bl ? s.bl - (int)V : s.bl;
  s.nvec = (s.hi - s.o + (int)V - 1) / (int)V;
  s.vb0 = s.lo < s.bl ? 1 : 0;
  s.nbv = (s.bh - s.bl) / (int)V;
  s.resident = s.nvec * 16 <= kSliceBytes;
  return s;
}

// Thread 0: the bulk copies of a resident slice's whole vectors into the
// on-chip copy, each chunk on its own mbarrier.
// fence: the buffer may hold generic-proxy writes of this block (an earlier
// row, a finish) that must be ordered before the copy overwrites it; the
// first copy of a block's only row needs none.
template <int DT>
__device__ __forceinline__ void issue_slice_copy(const Slice& s, const unsigned char* row,
                                                 unsigned char* sl, Ctl* ctl, bool fence = true) {
  using E = Elt<DT>;
  if (fence) fence_proxy_async_smem();
  const unsigned long long pol = policy_evict_first();
  for (int c = 0; c < kChunks; ++c) {
    const int c0 = s.nbv * c / kChunks, c1 = s.nbv * (c + 1) / kChunks;
    if (c1 > c0) {
      const unsigned bytes = (unsigned)(c1 - c0) * 16u;
      mbar_arrive_expect_tx(&ctl->mbar[c], bytes);
      bulk_copy_g2s(sl + (size_t)(s.vb0 + c0) * 16, row + (int64_t)s.bl * E::ES + (int64_t)c0 * 16,
                    bytes, &ctl->mbar[c], pol);
    }
  }
}

// The OR and the complement OR of the keys of this block's slice into
// ctl->kor / ctl->knand (equal-as-complements iff every key is the same); for
// a row split over blocks (keyset != nullptr) those of the whole row, through
// the slot's key-set words and one more row barrier (bounded: on time-out
// records the error and returns false).
template <class Src>
__device__ __forceinline__ bool row_key_set(const Src& src, unsigned* keyset, unsigned* arrive,
                                            unsigned target, long long limit, Ctl* ctl,
                                            unsigned* status) {
  constexpr int U = Src::U;
  if (threadIdx.x == 0) {
    ctl->kor = 0u;
    ctl->knand = 0u;
  }
  uint32_t kor = 0u, kand = ~0u;
  src.visit([&](const uint32_t(&key)[U], const int(&)[U], unsigned vm) {
#pragma unroll
    for (int j = 0; j < U; ++j)
      if ((vm >> j) & 1u) {
        kor |= key[j];
        kand &= key[j];
      }
  });
  kor = __reduce_or_sync(0xffffffffu, kor);
  kand = __reduce_and_sync(0xffffffffu, kand);
  __syncthreads();  // (the words are clear)
  if ((threadIdx.x & 31u) == 0u) {
    if (kor != 0u) atomicOr(&ctl->kor, kor);
    if (~kand != 0u) atomicOr(&ctl->knand, ~kand);
  }
  __syncthreads();
  if (keyset != nullptr && threadIdx.x == 0) {
    if (ctl->kor != 0u) atomicOr(&keyset[0], ctl->kor);
    if (ctl->knand != 0u) atomicOr(&keyset[1], ctl->knand);
    red_release_add_u32(arrive, 1u);  // releases the two ORs
    unsigned ok = 1u;
    const unsigned long long t0 = globaltimer_ns();
    while ((unsigned)ld_acquire_u64(arrive) < target) {
      if ((long long)(globaltimer_ns() - t0) > limit) {
        ok = 0u;
        atomicOr(status, kStatTimeout);
        break;
      }
    }
    const unsigned long long ks = ld_relaxed_u64(reinterpret_cast<const unsigned long long*>(keyset));
    ctl->kor = (unsigned)ks;
    ctl->knand = (unsigned)(ks >> 32);
    ctl->ok = ok;
  }
  __syncthreads();
  return ctl->ok != 0u;
}

// Candidate words [0, dirty) that the previous call on this slot left
// written go back to all ones, each block of the row taking a share.  Called
// before the row's first barrier, which orders these stores before every
// candidate word of this call is written or polled.
__device__ __forceinline__ void reset_candidates(uint2* cand, unsigned dirty, int part, int group) {
  unsigned long long* gc = reinterpret_cast<unsigned long long*>(cand);
  dirty = min(dirty, (unsigned)kGroupCandCap);
  const unsigned per = (dirty + (unsigned)group - 1u) / (unsigned)group;
  const unsigned a = min(dirty, (unsigned)part * per), b = min(dirty, a + per);
  for (unsigned i = a + threadIdx.x; i < b; i += kThreads) st_relaxed_u64(gc + i, kCandEmpty);
}

// Clears the other parity's counters of a slot, used by the previous call on
// it, for the next one; blocks 1..group-1 of the row each take a share.
__device__ __forceinline__ void clear_other_parity(SlotHdr* slot, unsigned par, unsigned used_other,
                                                   int part, int group) {
  const unsigned helpers = (unsigned)group - 1u, me = (unsigned)part - 1u;
  unsigned* other = reinterpret_cast<unsigned*>(reinterpret_cast<unsigned char*>(slot) + kSlotHistOff) +
                    (size_t)(par ^ 1u) * kSlotHistWords;
  const unsigned words = min(used_other, (unsigned)kMaxRounds) * (unsigned)kMaxBins;
  const unsigned per = ((words / 4 + helpers - 1) / helpers) * 4;
  const unsigned w0 = min(words, me * per), w1 = min(words, w0 + per);
  for (unsigned i = w0 / 4 + threadIdx.x; i < w1 / 4; i += kThreads)
    reinterpret_cast<uint4*>(other)[i] = make_uint4(0u, 0u, 0u, 0u);
  if (me == 0 && threadIdx.x == 0) {
    slot->sync[par ^ 1u].arrive = 0u;
    slot->sync[par ^ 1u].top = 0u;
    slot->sync[par ^ 1u].floor = 0u;
    slot->keyset[par ^ 1u][0] = 0u;
    slot->keyset[par ^ 1u][1] = 0u;
  }
}

// A row length carried from one row to the next: the clamped length, bit 31
// set when it had to be clamped; kLenUnknown when not loaded yet.
constexpr uint32_t kLenUnknown = 0xFFFFFFFFu;

// Selects the top k of row r with this block as part `part` of `group`.
// Returns false after an unrecoverable device-side error.  copy_issued: the
// bulk copy of this row's slice is already in flight (issued by this block at
// the end of its previous row); on return, whether that holds for the next.
// len_carry: row r's length if already loaded; on return, the next row's.
// kLean: a row split over blocks whose slices all fit on chip, logits in
// device memory, no cluster -- the other paths are not compiled in.
template <int DT, bool kLean>
__device__ __forceinline__ bool select_row(const Params& p, int r, int part, unsigned char* smem,
                                           unsigned& phase_bits, bool& cl_pending,
                                           bool& copy_issued, uint32_t& len_carry) {
  using E = Elt<DT>;
  Ctl* ctl = reinterpret_cast<Ctl*>(smem + kCtlOff);
  unsigned* h = reinterpret_cast<unsigned*>(smem + kHistOff);
  unsigned* offs = reinterpret_cast<unsigned*>(smem + kOffsOff);
  unsigned char* sl = smem + kSliceOff;
  uint2* lcand = reinterpret_cast<uint2*>(smem + kLocalCandOff);
  unsigned* status = reinterpret_cast<unsigned*>(p.ws);
  const int group = p.group;
  const unsigned k = (unsigned)p.k;
  int32_t* out_row = p.out + (int64_t)r * p.k;

  __syncthreads();  // the previous row is done with shared memory
  if (threadIdx.x == 0) ctl->ok = 1u;

  // This row's slot (rows split over blocks): its header is read now and
  // used at the first merge.
  SlotHdr* slot = nullptr;
  uint4 hdr = make_uint4(0u, 0u, 0u, 0u);
  if (group > 1) {
    slot = reinterpret_cast<SlotHdr*>(p.ws + kWsHeaderBytes + (size_t)r * kSlotBytes);
    hdr = ld_relaxed_v4(slot);  // epoch, used[0], used[1], cand_dirty
  }

  // Valid length (clamped; a bad one is reported); for a block that owns
  // whole rows also the next row's, whose copy it issues early.
  bool bad_len;
  uint32_t L;
  if (len_carry != kLenUnknown) {
    L = len_carry & 0x7FFFFFFFu;
    bad_len = (len_carry >> 31) != 0u;
  } else {
    L = row_length(p, r, &bad_len);
  }
  // This block's slice, with 16-byte aligned interior boundaries (the lean
  // kernel has issued its copy on entry).
  const unsigned char* row = p.logits + (int64_t)r * p.row_stride * E::ES;
  const Slice s = slice_geometry<DT>(L, part, group, row, p.row_len ? 0u : (uint32_t)p.chunk);
  const int r_next = r + (int)gridDim.x;
  const bool has_next = group == 1 && r_next < p.batch;
  bool bad_next = false;  // (reported by the next row's own call)
  const uint32_t L_next = has_next ? row_length(p, r_next, &bad_next) : 0u;
  auto carry_next = [&] { len_carry = has_next ? (L_next | (bad_next ? 0x80000000u : 0u)) : kLenUnknown; };
  zero_counters(h, kMaxBins);
  // cluster rows merge into block 0's histogram in the (here unused) local
  // candidate area: bins, then the row's top
  unsigned* gh = !kLean && p.cluster ? reinterpret_cast<unsigned*>(lcand) : nullptr;
  if (gh != nullptr) {
    zero_counters(gh, kMaxBins + 4);
    // this block's gh is clear; the matching wait comes right before the adds,
    // so the barrier's latency hides behind the copy and the histogram
    __syncthreads();
    cluster_arrive();
    cl_pending = true;  // (consumed by the wait before the adds, or at exit)
  }
  if (bad_len && threadIdx.x == 0 && part == 0) atomicOr(status, kStatRowLen);

  // Rows with no more than k elements: every position, then -1.
  if (L <= k) {
    for (uint32_t i = (uint32_t)part * kThreads + threadIdx.x; i < k; i += (uint32_t)kThreads * group)
      out_row[i] = i < L ? (int32_t)i : -1;
    carry_next();
    return true;
  }

  const int pos_bits = 32 - __clz((int)(L - 1u));  // 1..31
  const uint32_t pmax = (1u << pos_bits) - 1u;
  const int nr = num_rounds<DT>(pos_bits);

  const SliceSrc<DT> src{row, sl, s, p.host_src != 0};

  // ---- round 0: one pass over HBM, histogram of the top 12 key bits ----
  constexpr int U = SliceSrc<DT>::U;
  auto f0 = [&](const uint32_t(&key)[U], const int(&)[U], unsigned vm) {
#pragma unroll
    for (int j = 0; j < U; ++j)
      if ((vm >> j) & 1u) atomicAdd(&h[key[j] >> E::kShift0], 1u);
  };
  if (!kLean && s.resident && p.host_src) {
    // a row in host memory: plain loads into the on-chip copy, counted as they arrive
    const int nh = s.bl - s.lo, nt = s.hi - s.bh;
    if ((int)threadIdx.x < nh + nt) {
      const int i = (int)threadIdx.x < nh ? s.lo + (int)threadIdx.x : s.bh + ((int)threadIdx.x - nh);
      E::store(sl + (size_t)(i - s.o) * E::ES, E::load(row, i));
    }
    src.load_visit_body(sl, f0);
    __syncthreads();
    src.visit_edges(f0);
  } else if (kLean || s.resident) {
    const int vb0 = s.vb0, nbv = s.nbv;
    // (a block that owns whole rows may have issued this copy already, at the
    // end of its previous row)
    if (!kLean && threadIdx.x == 0 && !copy_issued) issue_slice_copy<DT>(s, row, sl, ctl);
    copy_issued = false;
    // the unaligned head and tail by plain loads
    const int nh = s.bl - s.lo, nt = s.hi - s.bh;
    if ((int)threadIdx.x < nh + nt) {
      const int i = (int)threadIdx.x < nh ? s.lo + (int)threadIdx.x : s.bh + ((int)threadIdx.x - nh);
      E::store(sl + (size_t)(i - s.o) * E::ES, E::load(row, i));
    }
    __syncthreads();
    src.visit_edges(f0);
#pragma unroll
    for (int c = 0; c < kChunks; ++c) {
      const int c0 = nbv * c / kChunks, c1 = nbv * (c + 1) / kChunks;
      if (c1 > c0) {
        mbar_wait_bounded(&ctl->mbar[c], (phase_bits >> c) & 1u, p.spin_limit_ns, ctl, status);
        phase_bits ^= 1u << c;
#if TKS_HIST_AGGREGATE
        src.hist_aggregated(vb0 + c0, vb0 + c1, h);
#else
        src.visit_range(vb0 + c0, vb0 + c1, f0);
#endif
      }
    }
  } else {
    __syncthreads();
    src.visit_global(f0);
  }
  __syncthreads();
  // (a cluster row goes through its cluster barriers even when its copy
  // failed: the other blocks of the cluster wait for it there)
  if (!ctl->ok && gh == nullptr) return false;

  // Counters of this call's parity; the other parity's are cleared below.
  const unsigned epoch = hdr.x, par = epoch & 1u;
  const unsigned used_other = par ? hdr.y : hdr.z;
  unsigned* slot_hist = nullptr;
  uint2* slot_cand = nullptr;
  if (group > 1) {
    slot_hist = reinterpret_cast<unsigned*>(reinterpret_cast<unsigned char*>(slot) + kSlotHistOff) +
                (size_t)par * kSlotHistWords;
    slot_cand = reinterpret_cast<uint2*>(p.ws + kWsHeaderBytes + (size_t)p.slots * kSlotBytes +
                                         (size_t)r * kCandSlotBytes);
  }

  // ---- digit rounds: merge, threshold, emit; until the threshold bin is
  //      taken whole or is small enough to finish on one block ----
  Prefix P = {0u, 0u, 0u, 0u};  // resolved digits before round t
  unsigned k_rem = k;           // still to select among elements matching P
  unsigned base = 0;            // output slots already assigned to earlier rounds
  int t = 0;
  int end = kEndAbove;
  unsigned cnt = 0;
  const unsigned cap = group > 1 ? (unsigned)kGroupCandCap : (unsigned)kLocalCandCap;
  uint2* cand = group > 1 ? slot_cand : lcand;
  unsigned nbar = 0u;  // L2 row barriers passed (each adds `group` arrivals)
  for (;;) {
    const Digit D = digit_of_round<DT>(t, pos_bits);
    const int nb = 1 << D.bits;
    if (t > 0) {
      zero_counters(h, nb);
      __syncthreads();
      if (kLean || s.resident)
        later_pass_resident<DT, false>(src, P, D, pmax, h, 0u, 0, 0u, nullptr, nullptr, nullptr, 0u,
                                       nullptr, false, 0u, status);
      else
        hist_round(src, h, P, D, pmax);
      __syncthreads();
    }
    int lo = 0, hi = nb;
    if (t == 0) {
      if (group > 1) reset_candidates(slot_cand, hdr.w, part, group);
      const bool skip = p.test_skip_arrive && part == 0;
      if (!round0_bounds_merge(h, offs, k, group > 1, group > 1 ? slot_hist : nullptr,
                               group > 1 ? &slot->sync[par].arrive : nullptr, (unsigned)group, skip,
                               p.spin_limit_ns, ctl, status, &lo, &hi, gh, &cl_pending))
        return false;
      if (gh == nullptr && group > 1) ++nbar;  // the first round's L2 barrier
      // every block of the call has read the epoch: the next call may use the other set
      // (and until this call says how many candidate words it wrote, the next
      // one resets them all)
      if (group > 1 && part == 0 && threadIdx.x == 0) {
        slot->epoch = epoch + 1u;
        slot->cand_dirty = (unsigned)kGroupCandCap;
      }
      // One first-digit bin holds the whole row: if every key is the same,
      // the answer is the k lowest positions.  Each block ORs and ANDs its
      // keys; a split row exchanges them through the slot (one more row
      // barrier); then each block writes its share and stops.  (Cluster rows
      // go on with the digit rounds.)
      if (gh == nullptr && hi > 0 && h[hi - 1] == L) {
        if (!row_key_set(src, group > 1 ? slot->keyset[par] : nullptr,
                         group > 1 ? &slot->sync[par].arrive : nullptr,
                         (unsigned)group * (nbar + 1u), p.spin_limit_ns, ctl, status))
          return false;
        if (group > 1) ++nbar;
        if (ctl->kor == ~ctl->knand) {
          for (int i = s.lo + (int)threadIdx.x; i < min(s.hi, (int)k); i += kThreads) out_row[i] = i;
          end = kEndFinal;
          break;
        }
      }
    } else if (group > 1) {
      if (!group_merge(h, offs, nb, slot_hist + (size_t)t * kMaxBins, &slot->sync[par].arrive,
                       (unsigned)group * (nbar + 1u), p.spin_limit_ns, ctl, status))
        return false;
      ++nbar;
    }
    if (group == 1) zero_counters(offs, nb);
    unsigned bin, above;
    const unsigned* suf = h;  // the row's elements above each bin of this round
    int suf_lo = 0;
    // (the warps' own suffix sums: in the lean kernel's unused local
    // candidate area; for a whole row on chip, in the slice buffer's tail when
    // the slice leaves it free)
    unsigned* sw_base =
        kLean ? reinterpret_cast<unsigned*>(lcand)
        : (group == 1 && s.resident && s.nvec * 16 <= kSliceBytes - kWarps * 128)
            ? reinterpret_cast<unsigned*>(sl + kSliceBytes - kWarps * 128)
            : nullptr;
    if (sw_base != nullptr && t == 0 && hi - lo <= 32) {
      // every warp finds the threshold bin and keeps its own suffix sums: no
      // block-wide step
      unsigned* sw = sw_base + (threadIdx.x >> 5) * 32u;
      const Pick pk = warp_window_pick(h, lo, hi, k_rem, sw);
      __syncwarp();
      if (pk.bin == 0xFFFFFFFFu) {
        if (threadIdx.x == 0) atomicOr(status, kStatInternal);
        return false;
      }
      bin = pk.bin;
      above = pk.above;
      cnt = pk.cnt;
      suf = sw;
      suf_lo = lo;
    } else if (!pick_bin_range(h, lo, hi, nb, k_rem, ctl, status, &bin, &above, &cnt)) {
      return false;
    }
    const unsigned need = k_rem - above;
    end = cnt == need ? kEndFinal : cnt <= cap ? kEndCollect : kEndAbove;
    // (a round that only passes the threshold on, with nothing above its bin
    // anywhere in the row, has nothing to emit)
    if (end != kEndAbove || above != 0u) {
      const uint32_t t0 = (end == kEndAbove ? bin + 1u : bin) << D.shift;
      if (t == 0 && (kLean || s.resident) && !(end == kEndAbove && t0 == 0u))
        emit_first_resident(src, t0, D, bin, end, base, suf, suf_lo, offs, out_row, k, cand,
                            group > 1, cap, status);
      else if (suf != h) {
        // (the warp-kept suffix sums serve the first-round pass above only,
        // which a first round that has anything to emit always takes)
        if (threadIdx.x == 0) atomicOr(status, kStatInternal);
        return false;
      } else if (kLean || s.resident)
        later_pass_resident<DT, true>(src, P, D, pmax, nullptr, bin, end, base, h, offs, out_row, k,
                                      cand, group > 1, cap, status);
      else
        emit_round(src, P, D, bin, end, base, h, offs, pmax, out_row, k, cand, group > 1, cap,
                   status);
    }
    prefix_extend(P, D, bin);
    base += above;
    k_rem = need;
    if (end != kEndAbove) break;
    __syncthreads();
    if (++t >= nr) {
      if (threadIdx.x == 0) atomicOr(status, kStatInternal);
      return false;
    }
  }

  if (!kLean && group == 1) {
    // The slice copy is read for the last time: the next row's copy can start
    // now and land while this row finishes.
    const unsigned char* row_next = p.logits + (int64_t)r_next * p.row_stride * E::ES;
    const Slice s_next = slice_geometry<DT>(L_next, 0, 1, row_next);
    copy_issued = !p.host_src && L_next > k && s_next.resident;
    carry_next();
    if (copy_issued) {
      __syncthreads();
      if (threadIdx.x == 0) issue_slice_copy<DT>(s_next, row_next, sl, ctl);
    }
    if (end == kEndCollect && cnt <= kRegCandCap) {
      __syncthreads();
      uint32_t ck[kRegCand], ci[kRegCand];
      unsigned alive = 0u;
      uint32_t ok_ = 0u, ak = ~0u, oi = 0u, ai = ~0u;
#pragma unroll
      for (int j = 0; j < kRegCand; ++j) {
        const unsigned i = j * kThreads + threadIdx.x;
        const uint2 c = i < cnt ? lcand[i] : make_uint2(0u, 0u);
        ck[j] = c.x;
        ci[j] = pmax - c.y;
        if (i < cnt) {
          alive |= 1u << j;
          ok_ |= ck[j]; ak &= ck[j]; oi |= ci[j]; ai &= ci[j];
        }
      }
      block_or_and(ok_, ak, oi, ai, ctl);
      finish_in_registers(ck, ci, alive, k_rem, P, ok_, ak, oi, ai, cnt, pmax, h, out_row, k, ctl,
                          status);
    } else if (end == kEndCollect) {
      __syncthreads();
      uint32_t ok_ = 0u, ak = ~0u, oi = 0u, ai = ~0u;
      for (unsigned i = threadIdx.x; i < cnt; i += kThreads) {
        const uint2 e = lcand[i];
        const uint32_t inv = pmax - e.y;
        ok_ |= e.x; ak &= e.x; oi |= inv; ai &= inv;
      }
      block_or_and(ok_, ak, oi, ai, ctl);
      finish_on_chip(lcand, cnt, k_rem, P, ok_, ak, oi, ai, pmax, h, out_row, k, ctl, status);
    }
    return true;
  }

  // ---- rows split over blocks ----
  // For the next call on this slot: the digit rounds used (their counters are
  // cleared by the next call of the other parity) and the candidate words
  // written (reset by the next call).
  if (part == 0 && threadIdx.x == 0) {
    slot->used[par] = (unsigned)(t + 1);
    slot->cand_dirty = end == kEndCollect ? cnt : 0u;
  }
  if (part == 0) {
    if (end == kEndCollect && cnt <= kRegCandCap) {
      // Gather the row's candidates straight into registers as they land
      // (each word starts as all ones), then finish in registers.  The
      // finisher's counters are cleared first, while the candidates land
      // (after every warp is done with this block's emission).
      __syncthreads();
      for (int i = threadIdx.x; i < 3 * kPickBins; i += kThreads) h[i] = 0u;
      unsigned long long* gc = reinterpret_cast<unsigned long long*>(slot_cand);
      unsigned long long e[kRegCand];
#pragma unroll
      for (int j = 0; j < kRegCand; ++j) {
        const unsigned i = j * kThreads + threadIdx.x;
        e[j] = i < cnt ? ld_relaxed_u64(gc + i) : 0ull;
      }
      const unsigned long long t0 = globaltimer_ns();
      for (;;) {
        bool missing = false;
#pragma unroll
        for (int j = 0; j < kRegCand; ++j) {
          const unsigned i = j * kThreads + threadIdx.x;
          if (i < cnt && e[j] == kCandEmpty) {
            e[j] = ld_relaxed_u64(gc + i);
            missing = true;
          }
        }
        if (!missing) break;
        if ((long long)(globaltimer_ns() - t0) > p.spin_limit_ns) {
          ctl->ok = 0u;
          atomicOr(status, kStatTimeout);
          break;
        }
      }
      uint32_t ck[kRegCand], ci[kRegCand];
      unsigned alive = 0u;
      uint32_t ok_ = 0u, ak = ~0u, oi = 0u, ai = ~0u;
#pragma unroll
      for (int j = 0; j < kRegCand; ++j) {
        const bool in = j * kThreads + threadIdx.x < cnt;
        ck[j] = (uint32_t)e[j];
        ci[j] = pmax - (uint32_t)(e[j] >> 32);
        alive |= (in ? 1u : 0u) << j;
        ok_ |= in ? ck[j] : 0u;
        ak &= in ? ck[j] : ~0u;
        oi |= in ? ci[j] : 0u;
        ai &= in ? ci[j] : ~0u;
      }
      block_or_and(ok_, ak, oi, ai, ctl);
      if (!ctl->ok) return false;
      finish_in_registers(ck, ci, alive, k_rem, P, ok_, ak, oi, ai, cnt, pmax, h, out_row, k, ctl,
                          status, true);
    } else if (end == kEndCollect) {
      // Gather the row's candidates as they land (each slot starts as all
      // ones), then finish.
      // The candidates go where this block's slice copy was: every thread must
      // be done reading it (the emission pass) first.
      __syncthreads();
      uint2* fc = reinterpret_cast<uint2*>(sl);
      unsigned long long* gc = reinterpret_cast<unsigned long long*>(slot_cand);
      uint32_t ok_ = 0u, ak = ~0u, oi = 0u, ai = ~0u;
      const unsigned long long t0 = globaltimer_ns();
      for (unsigned i0 = 0; i0 < cnt; i0 += 8u * kThreads) {
        unsigned long long e[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const unsigned i = i0 + j * kThreads + threadIdx.x;
          e[j] = i < cnt ? ld_relaxed_u64(gc + i) : 0ull;
        }
        // re-poll every still-empty word together until all have landed
        for (;;) {
          bool missing = false;
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const unsigned i = i0 + j * kThreads + threadIdx.x;
            if (i < cnt && e[j] == kCandEmpty) {
              e[j] = ld_relaxed_u64(gc + i);
              missing = true;
            }
          }
          if (!missing) break;
          if ((long long)(globaltimer_ns() - t0) > p.spin_limit_ns) {
            ctl->ok = 0u;
            atomicOr(status, kStatTimeout);
            break;
          }
        }
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const unsigned i = i0 + j * kThreads + threadIdx.x;
          if (i >= cnt) continue;
          const uint2 c2 = make_uint2((uint32_t)e[j], (uint32_t)(e[j] >> 32));
          fc[i] = c2;
          const uint32_t inv = pmax - c2.y;
          ok_ |= c2.x; ak &= c2.x; oi |= inv; ai &= inv;
        }
      }
      block_or_and(ok_, ak, oi, ai, ctl);
      if (!ctl->ok) return false;
      finish_on_chip(fc, cnt, k_rem, P, ok_, ak, oi, ai, pmax, h, out_row, k, ctl, status);
    }
  } else {
    clear_other_parity(slot, par, used_other, part, group);
  }
  return true;
}


template <int DT, bool kLean>
__global__ void __launch_bounds__(kThreads, 1) tks_select_kernel(const Params p) {
  extern __shared__ __align__(128) unsigned char smem[];
  Ctl* ctl = reinterpret_cast<Ctl*>(smem + kCtlOff);
  // The next kernel of the stream may be scheduled as soon as SMs free up;
  // it waits below before touching memory, so this one runs ahead too.
  grid_launch_dependents();
  if (threadIdx.x == 0) {
    for (int c = 0; c < kChunks; ++c) mbar_init(&ctl->mbar[c], 1u);
    fence_mbar_init();
  }
  // Everything before this point is on-chip; the kernel ahead in the stream
  // (its writes to the inputs, the outputs and the workspace included) is
  // complete after it.
  grid_dependency_wait();
  // The slice copy of the block's first row goes out before anything else
  // (the lean kernel's one row; the first row of a block that owns whole rows
  // in device memory, when it fits on chip).
  bool first_issued = false;
  if (threadIdx.x == 0 && (kLean || (p.group == 1 && !p.host_src && !p.cluster))) {
    const int r = blockIdx.x / p.group, part = (int)blockIdx.x - r * p.group;
    bool bad;
    const uint32_t L = r < p.batch ? row_length(p, r, &bad) : 0u;
    if (L > (uint32_t)p.k) {
      const unsigned char* row = p.logits + (int64_t)r * p.row_stride * Elt<DT>::ES;
      const Slice s = slice_geometry<DT>(L, part, p.group, row, p.row_len ? 0u : (uint32_t)p.chunk);
      if (kLean || s.resident) {
        issue_slice_copy<DT>(s, row, smem + kSliceOff, ctl, false);
        first_issued = true;
      }
    }
  }
  __syncthreads();
  unsigned phase_bits = 0u;
  bool cl_pending = false;  // arrived at the cluster barrier that ends block 0's reads
  if (kLean || p.group > 1) {
    const int r = blockIdx.x / p.group;
    bool copy_issued = false;
    uint32_t len_carry = kLenUnknown;
    if (r < p.batch)
      select_row<DT, kLean>(p, r, (int)blockIdx.x - r * p.group, smem, phase_bits, cl_pending, copy_issued,
                            len_carry);
  } else {
    bool copy_issued = first_issued;   // this (then the next) row's slice copy is in flight
    uint32_t len_carry = kLenUnknown;  // the next row's length, once loaded
    for (int r = blockIdx.x; r < p.batch; r += gridDim.x)
      if (!select_row<DT, kLean>(p, r, 0, smem, phase_bits, cl_pending, copy_issued, len_carry))
        break;
  }
  // block 0 of a cluster keeps its shared memory until the others have read it
  if (cl_pending) cluster_wait();
}

// This block size's launcher and set-up (declared in tks_internal.h).
cudaError_t launch_select(const cudaLaunchConfig_t& base, const Params& p, int32_t dtype,
                          bool lean) {
  cudaLaunchConfig_t cfg = base;
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = kSmemBytes;
  if (lean)
    return dtype == TKS_F32 ? cudaLaunchKernelEx(&cfg, tks_select_kernel<0, true>, p)
                            : cudaLaunchKernelEx(&cfg, tks_select_kernel<1, true>, p);
  return dtype == TKS_F32 ? cudaLaunchKernelEx(&cfg, tks_select_kernel<0, false>, p)
                          : cudaLaunchKernelEx(&cfg, tks_select_kernel<1, false>, p);
}

bool setup_select(int* blocks_per_sm, int* max_cluster) {
  bool good = cudaFuncSetAttribute(tks_select_kernel<0, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   kSmemBytes) == cudaSuccess;
  good &= cudaFuncSetAttribute(tks_select_kernel<1, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               kSmemBytes) == cudaSuccess;
  good &= cudaFuncSetAttribute(tks_select_kernel<0, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               kSmemBytes) == cudaSuccess;
  good &= cudaFuncSetAttribute(tks_select_kernel<1, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               kSmemBytes) == cudaSuccess;
  // clusters of up to 16 blocks (one block per SM)
  good &= cudaFuncSetAttribute(tks_select_kernel<0, false>, cudaFuncAttributeNonPortableClusterSizeAllowed,
                               1) == cudaSuccess;
  good &= cudaFuncSetAttribute(tks_select_kernel<1, false>, cudaFuncAttributeNonPortableClusterSizeAllowed,
                               1) == cudaSuccess;
  int c0 = 0, c1 = 0;
  cudaLaunchConfig_t q;
  std::memset(&q, 0, sizeof q);
  q.gridDim = dim3(16, 1, 1);
  q.blockDim = dim3(kThreads, 1, 1);
  q.dynamicSmemBytes = kSmemBytes;
  cudaLaunchAttribute qa[1];
  qa[0].id = cudaLaunchAttributeClusterDimension;
  qa[0].val.clusterDim.x = 1;
  qa[0].val.clusterDim.y = 1;
  qa[0].val.clusterDim.z = 1;
  q.attrs = qa;
  q.numAttrs = 1;
  if (cudaOccupancyMaxPotentialClusterSize(&c0, tks_select_kernel<0, false>, &q) != cudaSuccess ||
      cudaOccupancyMaxPotentialClusterSize(&c1, tks_select_kernel<1, false>, &q) != cudaSuccess) {
    cudaGetLastError();
    c0 = c1 = 1;  // no clusters: rows merge through L2
  }
  *max_cluster = c0 < c1 ? c0 : c1;
  int b0 = 0, b1 = 0;
  good &= cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b0, tks_select_kernel<0, false>, kThreads,
                                                        kSmemBytes) == cudaSuccess;
  good &= cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b1, tks_select_kernel<1, false>, kThreads,
                                                        kSmemBytes) == cudaSuccess;
  *blocks_per_sm = b0 < b1 ? b0 : b1;
  return good;
}

}  // namespace TKS_VARIANT
}  // namespace tks
