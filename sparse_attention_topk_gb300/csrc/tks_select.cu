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
// Layout of the work (one kernel launch per call):
//  * A row is split into `group` contiguous slices, one thread block (256
//    threads, one per SM) each.  Each block copies its slice from HBM once,
//    with bulk asynchronous copies (TMA, non-tensor form) into shared memory,
//    and builds a 4096-bin histogram of the top 12 key bits on chip.
//  * With group > 1 the blocks of a row add their histograms into one in L2
//    and meet at a bounded barrier; every block then finds the threshold bin
//    itself (the page's "TLE distributed" idea of summing block histograms
//    and continuing with the new threshold, section "5. Triton-TLE").  The
//    adds return each block's offset inside every bin, so each block can
//    later write its selected positions to fixed output slots with no
//    further coordination.
//  * As soon as the bin holding the k-th element has few enough members
//    (the page's "early stop when the bucket is small", section "03."),
//    blocks write every position above the bin to the output and push the
//    bin's (key, position) pairs to a candidate buffer; the last block to
//    finish refines those candidates on chip and writes the rest.
//  * With group == 1 (many rows) a block owns whole rows and needs no
//    cross-block step at all.
// No tensor cores: this is a streaming selection, not a contraction.

#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>
#include <cstring>
#include <map>
#include <mutex>
#include <utility>

#include "tks.h"
#include "tks_device.cuh"
#include "tks_internal.h"

namespace tks {

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
};

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

  // The key of position pos of this slice (on chip when resident).
  __device__ __forceinline__ uint32_t key_at(int pos) const {
    using E = Elt<DT>;
    return E::key(s.resident ? E::load(sm, pos - s.o) : E::load(row, pos));
  }

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
        x[a] = v < nv ? ld_nc_v4(body + v) : make_uint4(0u, 0u, 0u, 0u);
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
// replace the local ones in h[].  top is the row's maximum (from the word
// beside the arrival count) when use_top, else nb; it is left in ctl->top.
// Bounded: on time-out records the error and returns false.
__device__ __forceinline__ bool merge_wait_load(unsigned* h, int lo, int nb, const unsigned* g,
                                                unsigned* sync_pair, bool use_top, unsigned target,
                                                bool skip_arrive, long long limit, Ctl* ctl,
                                                unsigned* status) {
  constexpr int kPer = kMaxBins / kThreads;
  if (threadIdx.x == 0) {
    // release: this block's adds (all returned before the caller's barrier)
    // are visible to any block that sees the arrival
    if (!skip_arrive) red_release_add_u32(&sync_pair[0], 1u);
    unsigned ok = 1u;
    unsigned long long w = ld_acquire_u64(sync_pair);
    if ((unsigned)w < target) {
      const unsigned long long t0 = globaltimer_ns();
      while ((unsigned)(w = ld_acquire_u64(sync_pair)) < target) {
        if ((long long)(globaltimer_ns() - t0) > limit) {
          ok = 0u;
          atomicOr(status, kStatTimeout);
          break;
        }
      }
    }
    ctl->top = use_top ? min((unsigned)nb, (unsigned)(w >> 32)) : (unsigned)nb;
    ctl->ok = ok;
  }
  __syncthreads();
  if (!ctl->ok) return false;
  const int top = (int)ctl->top;
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
                                                    int* lo, int* hi) {
  constexpr int kPer = kMaxBins / kThreads;
  static_assert(kPer % 4 == 0, "bins per thread");
  const int b0 = (int)threadIdx.x * kPer;
  unsigned c[kPer];
#pragma unroll
  for (int q = 0; q < kPer / 4; ++q) {
    const uint4 v = reinterpret_cast<const uint4*>(h + b0)[q];
    c[4 * q] = v.x;
    c[4 * q + 1] = v.y;
    c[4 * q + 2] = v.z;
    c[4 * q + 3] = v.w;
  }
  unsigned S = 0u;
#pragma unroll
  for (int j = 0; j < kPer; ++j) S += c[j];
  unsigned total;
  const unsigned A = block_suffix_excl(S, &total, ctl);  // this block's elements above my bins
  if (A < k && (threadIdx.x == 0 || A + S >= k)) {
    // the floor is mine: the lowest of my bins with fewer than k above it
    unsigned above = A;
    int f = 0;
#pragma unroll
    for (int j = kPer - 1; j >= 0; --j) {
      if (above < k) f = j;
      above += c[j];
    }
    ctl->lo = (unsigned)(b0 + f);
  }
  if (A == 0u && S != 0u) {  // my bins hold the highest nonempty one
    int tj = 0;
#pragma unroll
    for (int j = 0; j < kPer; ++j)
      if (c[j] != 0u) tj = j;
    ctl->top = (unsigned)(b0 + tj + 1);
  }
  if (total == 0u && threadIdx.x == 0) ctl->top = 0u;
  __syncthreads();
  const int l = (int)ctl->lo, top = (int)ctl->top;
  *lo = l;
  if (!split) {
    *hi = top;
    return true;
  }
#pragma unroll
  for (int j = 0; j < kPer; ++j) {
    const int b = j * kThreads + threadIdx.x;
    c[j] = (b >= l && b < top) ? h[b] : 0u;
  }
#pragma unroll
  for (int j = 0; j < kPer; ++j) c[j] = c[j] ? atomicAdd(&g[j * kThreads + threadIdx.x], c[j]) : 0u;
  // an atomic with return, so it has been performed by the arrival
  if (threadIdx.x == 0 && top > 0) ctl->sink = atomicMax(&sync_pair[1], (unsigned)top);
#pragma unroll
  for (int j = 0; j < kPer; ++j) {
    const int b = j * kThreads + threadIdx.x;
    if (b >= l && b < top) offs[b] = c[j];
  }
  __syncthreads();  // also: every thread has read ctl->top before it is rewritten
  if (!merge_wait_load(h, l, kMaxBins, g, sync_pair, true, target, skip_arrive, limit, ctl, status))
    return false;
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
template <int DT>
__device__ __forceinline__ void emit_first_resident(const SliceSrc<DT>& src, uint32_t t0,
                                                    const Digit& D, unsigned bin, int end,
                                                    unsigned base, const unsigned* suf,
                                                    unsigned* offs, int32_t* out_row, unsigned k,
                                                    uint2* cand, bool cand_global, unsigned cap,
                                                    unsigned* status) {
  using E = Elt<DT>;
  constexpr int U = E::V;
  constexpr int B = kPassVecs;
  bool bad = false;
  auto write = [&](uint32_t key, int pos) {
    const uint32_t d = key >> D.shift;
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
    // which of the B * U elements are written (a compact unrolled test) ...
    unsigned sel = 0u;
#pragma unroll
    for (int b = 0; b < B; ++b) {
      const int v = v0 + b * kThreads;
#pragma unroll
      for (int j = 0; j < U; ++j)
        sel |= (v < vb && E::key(E::lane(x[b], j)) >= t0 ? 1u : 0u) << (b * U + j);
    }
    // ... then one copy of the write path for those (rare) elements, keys
    // re-read from shared memory, so the loop stays small
    while (sel) {
      const int q = __ffs((int)sel) - 1;
      sel &= sel - 1u;
      const int pos = s.o + (v0 + (q / U) * kThreads) * U + q % U;
      write(E::key(E::load(src.sm, pos - s.o)), pos);  // resident: on chip
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
                                                    unsigned* status) {
  const unsigned out_base = k - k_rem;
  uint32_t vk = (or_k ^ and_k) & ~P.kmask;
  uint32_t vp = (or_i ^ and_i) & pmax & ~P.pmask;
  if (threadIdx.x == 0) ctl->emit_n = 0u;  // read after the rounds' barriers
  unsigned sel = 0u;
  unsigned live = n;
  for (;;) {
    Digit2 D;
    if (!next_digit2(vk, vp, digit_width(live), &D)) {
      if (threadIdx.x == 0) atomicOr(status, kStatInternal);
      return;
    }
    const int nb = 1 << (D.kb + D.pb);
    zero_counters(h, nb);
    __syncthreads();
    uint32_t d[kRegCand];
#pragma unroll
    for (int j = 0; j < kRegCand; ++j) {
      d[j] = digit2_value(D, ck[j], ci[j]);
      if ((alive >> j) & 1u) atomicAdd(&h[d[j]], 1u);
    }
    __syncthreads();
    unsigned bin, above, cnt;
    if (!pick_bin(h, nb, k_rem, ctl, status, &bin, &above, &cnt)) return;
#pragma unroll
    for (int j = 0; j < kRegCand; ++j) {
      if (!((alive >> j) & 1u)) continue;
      if (d[j] > bin) sel |= 1u << j;
      if (d[j] != bin) alive &= ~(1u << j);
    }
    k_rem -= above;
    if (cnt == k_rem) {
      sel |= alive;
      break;
    }
    live = cnt;
  }
  // Distinct slots from out_base on: each warp takes a run of them with one
  // shared add, its lanes place their candidates by ballot ranks.
  const unsigned lane = lane_id(), lt = (1u << lane) - 1u;
  unsigned m[kRegCand];
  unsigned wtotal = 0u;
#pragma unroll
  for (int j = 0; j < kRegCand; ++j) {
    m[j] = __ballot_sync(0xffffffffu, (sel >> j) & 1u);
    wtotal += (unsigned)__popc(m[j]);
  }
  unsigned wbase = 0u;
  if (lane == 0 && wtotal) wbase = atomicAdd(&ctl->emit_n, wtotal);
  unsigned slot = out_base + __shfl_sync(0xffffffffu, wbase, 0);
  bool bad = false;
#pragma unroll
  for (int j = 0; j < kRegCand; ++j) {
    if ((sel >> j) & 1u) {
      const unsigned sj = slot + (unsigned)__popc(m[j] & lt);
      if (sj < k)
        out_row[sj] = (int)(pmax - ci[j]);
      else
        bad = true;
    }
    slot += (unsigned)__popc(m[j]);
  }
  if (bad) atomicOr(status, kStatInternal);
}

// Selects the top k of row r with this block as part `part` of `group`.
// Returns false after an unrecoverable device-side error.
template <int DT>
__device__ __forceinline__ bool select_row(const Params& p, int r, int part, unsigned char* smem,
                           unsigned& phase_bits) {
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
    slot = reinterpret_cast<SlotHdr*>(p.ws + kWsHeaderBytes + (size_t)(blockIdx.x / group) * kSlotBytes);
    hdr = ld_relaxed_v4(slot);  // epoch, used[0], used[1]
  }

  // Valid length (clamped; a bad one is reported).
  int64_t Lr = p.row_len ? (int64_t)__ldg(p.row_len + r) : p.row_stride;
  zero_counters(h, kMaxBins);
  if (Lr < 0 || Lr > p.row_stride) {
    if (threadIdx.x == 0 && part == 0) atomicOr(status, kStatRowLen);
    Lr = Lr < 0 ? 0 : p.row_stride;
  }
  const uint32_t L = (uint32_t)Lr;

  // Rows with no more than k elements: every position, then -1.
  if (L <= k) {
    for (uint32_t i = (uint32_t)part * kThreads + threadIdx.x; i < k; i += (uint32_t)kThreads * group)
      out_row[i] = i < L ? (int32_t)i : -1;
    return true;
  }

  const int pos_bits = 32 - __clz((int)(L - 1u));  // 1..31
  const uint32_t pmax = (1u << pos_bits) - 1u;
  const int nr = num_rounds<DT>(pos_bits);

  // This block's slice, with 16-byte aligned interior boundaries.
  const unsigned char* row = p.logits + (int64_t)r * p.row_stride * E::ES;
  const uint32_t V = E::V;
  const uint32_t mis = (uint32_t)(((uintptr_t)row & 15u) / E::ES);
  auto align_up = [&](uint32_t i) -> uint32_t { return i + ((V - ((mis + i) & (V - 1u))) & (V - 1u)); };
  auto align_down = [&](uint32_t i) -> uint32_t { return i - ((mis + i) & (V - 1u)); };
  const uint32_t chunk = ((L + (uint32_t)group - 1u) / (uint32_t)group + V - 1u) & ~(V - 1u);
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
  const SliceSrc<DT> src{row, sl, s};

  // ---- round 0: one pass over HBM, histogram of the top 12 key bits ----
  constexpr int U = SliceSrc<DT>::U;
  auto f0 = [&](const uint32_t(&key)[U], const int(&)[U], unsigned vm) {
#pragma unroll
    for (int j = 0; j < U; ++j)
      if ((vm >> j) & 1u) atomicAdd(&h[key[j] >> E::kShift0], 1u);
  };
  if (s.resident) {
    const int vb0 = s.vb0, nbv = s.nbv;
    if (threadIdx.x == 0) {
      fence_proxy_async_smem();
      const unsigned long long pol = policy_evict_first();
      for (int c = 0; c < kChunks; ++c) {
        const int c0 = nbv * c / kChunks, c1 = nbv * (c + 1) / kChunks;
        if (c1 > c0) {
          const unsigned bytes = (unsigned)(c1 - c0) * 16u;
          mbar_arrive_expect_tx(&ctl->mbar[c], bytes);
          bulk_copy_g2s(sl + (size_t)(vb0 + c0) * 16, row + (int64_t)s.bl * E::ES + (int64_t)c0 * 16,
                        bytes, &ctl->mbar[c], pol);
        }
      }
    }
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
        src.visit_range(vb0 + c0, vb0 + c1, f0);
      }
    }
  } else {
    __syncthreads();
    src.visit_global(f0);
  }
  __syncthreads();
  if (!ctl->ok) return false;

  // Counters of this call's parity; the other parity's are cleared below.
  const unsigned epoch = hdr.x, par = epoch & 1u;
  const unsigned used_other = par ? hdr.y : hdr.z;
  unsigned* slot_hist = nullptr;
  uint2* slot_cand = nullptr;
  if (group > 1) {
    slot_hist = reinterpret_cast<unsigned*>(reinterpret_cast<unsigned char*>(slot) + kSlotHistOff) +
                (size_t)par * kSlotHistWords;
    slot_cand = reinterpret_cast<uint2*>(p.ws + kWsHeaderBytes + (size_t)p.slots * kSlotBytes +
                                         (size_t)(blockIdx.x / group) * kCandSlotBytes);
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
  for (;;) {
    const Digit D = digit_of_round<DT>(t, pos_bits);
    const int nb = 1 << D.bits;
    if (t > 0) {
      zero_counters(h, nb);
      __syncthreads();
      if (s.resident)
        later_pass_resident<DT, false>(src, P, D, pmax, h, 0u, 0, 0u, nullptr, nullptr, nullptr, 0u,
                                       nullptr, false, 0u, status);
      else
        hist_round(src, h, P, D, pmax);
      __syncthreads();
    }
    int lo = 0, hi = nb;
    if (t == 0) {
      const bool skip = p.test_skip_arrive && part == 0;
      if (!round0_bounds_merge(h, offs, k, group > 1, group > 1 ? slot_hist : nullptr,
                               group > 1 ? &slot->sync[par].arrive : nullptr, (unsigned)group, skip,
                               p.spin_limit_ns, ctl, status, &lo, &hi))
        return false;
      // every block of the call has read the epoch: the next call may use the other set
      if (group > 1 && part == 0 && threadIdx.x == 0) slot->epoch = epoch + 1u;
    } else if (group > 1) {
      if (!group_merge(h, offs, nb, slot_hist + (size_t)t * kMaxBins, &slot->sync[par].arrive,
                       (unsigned)group * (t + 1), p.spin_limit_ns, ctl, status))
        return false;
    }
    if (group == 1) zero_counters(offs, nb);
    unsigned bin, above;
    if (!pick_bin_range(h, lo, hi, nb, k_rem, ctl, status, &bin, &above, &cnt)) return false;
    const unsigned need = k_rem - above;
    end = cnt == need ? kEndFinal : cnt <= cap ? kEndCollect : kEndAbove;
    // (a round that only passes the threshold on, with nothing above its bin
    // anywhere in the row, has nothing to emit)
    if (end != kEndAbove || above != 0u) {
      const uint32_t t0 = (end == kEndAbove ? bin + 1u : bin) << D.shift;
      if (t == 0 && s.resident && !(end == kEndAbove && t0 == 0u))
        emit_first_resident(src, t0, D, bin, end, base, h, offs, out_row, k, cand, group > 1, cap,
                            status);
      else if (s.resident)
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

  if (group == 1) {
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
  if (part == 0) {
    if (end == kEndCollect && cnt <= kRegCandCap) {
      // Gather the row's candidates straight into registers as they land
      // (each word starts as all ones), put the words back to all ones for
      // the next call, then finish in registers.
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
        const unsigned i = j * kThreads + threadIdx.x;
        ck[j] = (uint32_t)e[j];
        ci[j] = pmax - (uint32_t)(e[j] >> 32);
        if (i < cnt) {
          gc[i] = kCandEmpty;
          alive |= 1u << j;
          ok_ |= ck[j]; ak &= ck[j]; oi |= ci[j]; ai &= ci[j];
        }
      }
      block_or_and(ok_, ak, oi, ai, ctl);
      if (!ctl->ok) return false;
      finish_in_registers(ck, ci, alive, k_rem, P, ok_, ak, oi, ai, cnt, pmax, h, out_row, k, ctl,
                          status);
    } else if (end == kEndCollect) {
      // Gather the row's candidates as they land (each slot starts as all
      // ones), put the slots back to all ones for the next call, then finish.
      uint2* fc = reinterpret_cast<uint2*>(sl);  // this block's slice copy is no longer needed
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
          gc[i] = kCandEmpty;
          const uint32_t inv = pmax - c2.y;
          ok_ |= c2.x; ak &= c2.x; oi |= inv; ai &= inv;
        }
      }
      block_or_and(ok_, ak, oi, ai, ctl);
      if (!ctl->ok) return false;
      finish_on_chip(fc, cnt, k_rem, P, ok_, ak, oi, ai, pmax, h, out_row, k, ctl, status);
    }
    if (threadIdx.x == 0) slot->used[par] = (unsigned)(t + 1);
  } else {
    // Clear the other parity's counters, used by the previous call on this
    // slot, for the next one; the blocks other than the finisher share it.
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
    }
  }
  return true;
}

template <int DT>
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
  __syncthreads();
  unsigned phase_bits = 0u;
  if (p.group > 1) {
    const int r = blockIdx.x / p.group;
    if (r < p.batch) select_row<DT>(p, r, blockIdx.x % p.group, smem, phase_bits);
  } else {
    for (int r = blockIdx.x; r < p.batch; r += gridDim.x)
      if (!select_row<DT>(p, r, 0, smem, phase_bits)) break;
  }
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
namespace {

struct DeviceInfo {
  int sms = 0;
  int blocks_per_sm = 0;
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
std::atomic<long long> g_min_per_block{2048};
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
    bool good = true;
    good &= cudaFuncSetAttribute(tks_select_kernel<0>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 kSmemBytes) == cudaSuccess;
    good &= cudaFuncSetAttribute(tks_select_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 kSmemBytes) == cudaSuccess;
    int b0 = 0, b1 = 0;
    good &= cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b0, tks_select_kernel<0>, kThreads,
                                                          kSmemBytes) == cudaSuccess;
    good &= cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b1, tks_select_kernel<1>, kThreads,
                                                          kSmemBytes) == cudaSuccess;
    d.blocks_per_sm = b0 < b1 ? b0 : b1;
    d.ok = good && d.blocks_per_sm >= 1;
    if (!good) cudaGetLastError();
  }
  g_dev[dev] = d;
  *out = d;
  return d.ok ? TKS_OK : TKS_E_UNSUPPORTED;
}

void plan_launch(const DeviceInfo& d, int32_t batch, int64_t row_stride, int* group, int* grid) {
  const int cap = d.sms * d.blocks_per_sm;
  if (batch >= cap) {
    *group = 1;
    *grid = cap;
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

// Layout: status header | slot headers and counters | candidate slots.
size_t workspace_bytes(const DeviceInfo& d) {
  return kWsHeaderBytes + (size_t)workspace_slots(d) * (kSlotBytes + kCandSlotBytes);
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
static void set_launch_attrs(cudaLaunchConfig_t* cfg, cudaLaunchAttribute* attr, int group) {
  std::memset(attr, 0, 2 * sizeof(cudaLaunchAttribute));
  int n = 0;
  attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[n].val.programmaticStreamSerializationAllowed = 1;
  ++n;
  if (group > 1) {
    attr[n].id = cudaLaunchAttributeCooperative;
    attr[n].val.cooperative = 1;
    ++n;
  }
  cfg->attrs = attr;
  cfg->numAttrs = (unsigned)n;
}

extern "C" int tks_topk_indices(const void* logits, const int32_t* row_len, int32_t batch,
                                int64_t row_stride, int32_t k, int32_t dtype, int32_t* out_idx,
                                void* stream) {
  if (batch < 0 || row_stride < 0 || row_stride > INT32_MAX || k < 1 || k > TKS_K_MAX)
    return TKS_E_INVAL;
  if (dtype != TKS_F32 && dtype != TKS_BF16) return TKS_E_INVAL;
  if (batch == 0) return TKS_OK;
  const int es = dtype == TKS_F32 ? 4 : 2;
  if (out_idx == nullptr || ((uintptr_t)out_idx & 3u) != 0) return TKS_E_INVAL;
  if (row_stride > 0 && (logits == nullptr || ((uintptr_t)logits % (uintptr_t)es) != 0))
    return TKS_E_INVAL;
  if ((int64_t)batch * row_stride > (INT64_MAX / 4)) return TKS_E_INVAL;

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
  plan_launch(d, batch, row_stride, &group, &grid);

  Params p;
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

  cudaLaunchConfig_t cfg;
  std::memset(&cfg, 0, sizeof cfg);
  cfg.gridDim = dim3((unsigned)grid, 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = (cudaStream_t)stream;
  cudaLaunchAttribute attr[2];
  set_launch_attrs(&cfg, attr, group);
  cudaError_t e = dtype == TKS_F32 ? cudaLaunchKernelEx(&cfg, tks_select_kernel<0>, p)
                                   : cudaLaunchKernelEx(&cfg, tks_select_kernel<1>, p);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return TKS_E_CUDA;
  }
  return TKS_OK;
}

extern "C" int tks_topk_indices_sorted(const void* logits, const int32_t* row_len, int32_t batch,
                                       int64_t row_stride, int32_t k, int32_t dtype, int32_t* out_idx,
                                       void* stream) {
  if (k > kOrderKMax) return TKS_E_INVAL;
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
    case TKS_OPT_MIN_PER_BLOCK: g_min_per_block.store(value > 0 ? value : 2048); return TKS_OK;
    case TKS_OPT_TEST_SKIP_ARRIVE: g_test_skip_arrive.store(value ? 1 : 0); return TKS_OK;
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
  plan_launch(d, batch, row_stride, &g, &gr);
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
  if (batch < 0 || row_stride < 0 || row_stride > INT32_MAX || k < 1 || k > TKS_K_MAX)
    return TKS_E_INVAL;
  if (dtype != TKS_F32 && dtype != TKS_BF16) return TKS_E_INVAL;
  if (batch == 0) return TKS_OK;
  if (batch > TKS_NOALLOC_MAX_ROWS) return TKS_E_TOO_LARGE;
  const int es = dtype == TKS_F32 ? 4 : 2;
  if (out_idx == nullptr || ((uintptr_t)out_idx & 3u) != 0) return TKS_E_INVAL;
  if (row_stride > 0 && (logits == nullptr || ((uintptr_t)logits % (uintptr_t)es) != 0))
    return TKS_E_INVAL;

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

  Params p;
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

  cudaLaunchConfig_t cfg;
  std::memset(&cfg, 0, sizeof cfg);
  cfg.gridDim = dim3((unsigned)grid, 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  set_launch_attrs(&cfg, attr, group);
  const cudaError_t e = dtype == TKS_F32 ? cudaLaunchKernelEx(&cfg, tks_select_kernel<0>, p)
                                         : cudaLaunchKernelEx(&cfg, tks_select_kernel<1>, p);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return TKS_E_CUDA;
  }
  return TKS_OK;
}
