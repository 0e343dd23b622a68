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
//  * A row is split into `group` contiguous slices, one thread block (1024
//    threads, one per SM) each.  Each block copies its slice from HBM once,
//    with bulk asynchronous copies (TMA, non-tensor form) into shared memory,
//    and builds a 4096-bin histogram of the top 12 key bits on chip.
//  * With group > 1 the blocks of a row add their histograms into one in L2
//    and meet at a bounded barrier; every block then finds the threshold bin
//    itself (the page's "TLE distributed" idea of summing block histograms
//    and continuing with the new threshold, section "5. Triton-TLE").
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
  bool resident;
};

// ---------------------------------------------------------------------------
// Element sources.  visit(f) calls f(key, position, valid) with all 32 lanes
// of each warp together (f may use warp intrinsics); the order in which a
// thread meets its elements is the same on every visit.
// ---------------------------------------------------------------------------
template <int DT>
struct SliceSrc {
  const unsigned char* row;  // the row in global memory
  const unsigned char* sm;   // on-chip copy (resident slices)
  Slice s;

  template <class F>
  __device__ __forceinline__ void visit_vecs(int va, int vb, F&& f) const {
    using E = Elt<DT>;
    for (int v0 = va; v0 < vb; v0 += kThreads) {
      const int v = v0 + (int)threadIdx.x;
      const bool in = v < vb;
      uint4 x = make_uint4(0u, 0u, 0u, 0u);
      if (in) x = reinterpret_cast<const uint4*>(sm)[v];
      const int i0 = s.o + v * E::V;
#pragma unroll
      for (int j = 0; j < E::V; ++j) {
        const int i = i0 + j;
        f(E::key(E::lane(x, j)), i, in && i >= s.lo && i < s.hi);
      }
    }
  }

  template <class F>
  __device__ __forceinline__ void visit_global(F&& f) const {
    using E = Elt<DT>;
    const int nh = s.bl - s.lo, nt = s.hi - s.bh;
    if ((threadIdx.x >> 5) == 0) {
      const int l = threadIdx.x & 31;
      const bool v = l < nh + nt;
      const int i = l < nh ? s.lo + l : s.bh + (l - nh);
      const uint32_t raw = v ? E::load(row, i) : 0u;
      f(E::key(raw), i, v);
    }
    const uint4* body = reinterpret_cast<const uint4*>(row + (int64_t)s.bl * E::ES);
    const int nv = (s.bh - s.bl) / E::V;
    constexpr int U = 4;
    for (int v0 = 0; v0 < nv; v0 += U * kThreads) {
      uint4 x[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int v = v0 + u * kThreads + (int)threadIdx.x;
        x[u] = v < nv ? ld_nc_v4(body + v) : make_uint4(0u, 0u, 0u, 0u);
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int v = v0 + u * kThreads + (int)threadIdx.x;
#pragma unroll
        for (int j = 0; j < E::V; ++j) f(E::key(E::lane(x[u], j)), s.bl + v * E::V + j, v < nv);
      }
    }
  }

  template <class F>
  __device__ __forceinline__ void visit(F&& f) const {
    if (s.resident)
      visit_vecs(0, s.nvec, f);
    else
      visit_global(f);
  }
};

// (key, position) pairs in shared memory.
struct CandSrc {
  const uint2* c;
  unsigned n;
  template <class F>
  __device__ __forceinline__ void visit(F&& f) const {
    for (unsigned i0 = 0; i0 < n; i0 += kThreads) {
      const unsigned i = i0 + threadIdx.x;
      const bool v = i < n;
      const uint2 e = v ? c[i] : make_uint2(0u, 0u);
      f(e.x, (int)e.y, v);
    }
  }
};

// ---------------------------------------------------------------------------
// Block-level steps
// ---------------------------------------------------------------------------

__device__ __forceinline__ void zero_hist(unsigned* h, int nb) {
  for (int i = threadIdx.x; i < nb; i += kThreads) h[i] = 0u;
}

// Histogram of digit D over the elements that match the prefix.
template <class Src>
__device__ __forceinline__ void hist_round(const Src& src, unsigned* h, const Prefix& P, Digit D,
                                           uint32_t pmax) {
  src.visit([&](uint32_t key, int pos, bool valid) {
    const uint32_t inv = pmax - (uint32_t)pos;
    const bool m = valid && prefix_cmp(P, key, inv) == 0;
    hist_add(h, digit_value(D, key, inv), m);
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

// Adds this block's histogram into the row's L2 histogram, waits (bounded)
// until every block of the row has done the same, then loads the sum.
__device__ bool group_merge(unsigned* h, int nb, unsigned* g, SlotHdr* slot, unsigned target,
                            bool skip_arrive, long long limit, Ctl* ctl, unsigned* status) {
  for (int i = threadIdx.x; i < nb; i += kThreads) {
    const unsigned c = h[i];
    if (c) red_add_u32(&g[i], c);
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    if (!skip_arrive) atomicAdd(&slot->arrive, 1u);
    unsigned ok = 1u;
    if (ld_acquire_u32(&slot->arrive) < target) {
      const unsigned long long t0 = globaltimer_ns();
      while (ld_acquire_u32(&slot->arrive) < target) {
        if ((long long)(globaltimer_ns() - t0) > limit) {
          ok = 0u;
          atomicOr(status, kStatTimeout);
          break;
        }
      }
    }
    __threadfence();
    ctl->ok = ok;
  }
  __syncthreads();
  if (!ctl->ok) return false;
  for (int i = threadIdx.x; i < nb; i += kThreads) h[i] = ld_cg_u32(&g[i]);
  __syncthreads();
  return true;
}

// Output slots and candidate slots come from one 64-bit counter: low half
// output positions, high half candidates.
struct Reserve {
  unsigned long long* global;  // slot->alloc (rows split over blocks), else null
};

// Writes every element whose resolved prefix is above P (and, unless
// `collect`, equal to P) to the output row; with `collect` the elements equal
// to P go to `cand` as (key, position) pairs.  Two passes over the source:
// count, one reservation per block, then write.
template <class Src>
__device__ void emit(const Src& src, const Prefix& P, uint32_t pmax, bool collect, Reserve res,
                     int32_t* out_row, unsigned k, uint2* cand, unsigned cap, Ctl* ctl,
                     unsigned* status) {
  unsigned ne = 0, nc = 0;
  src.visit([&](uint32_t key, int pos, bool valid) {
    if (!valid) return;
    const int c = prefix_cmp(P, key, pmax - (uint32_t)pos);
    if (c > 0 || (c == 0 && !collect))
      ++ne;
    else if (c == 0)
      ++nc;
  });
  unsigned long long total;
  const unsigned long long mine =
      block_prefix_excl64(((unsigned long long)nc << 32) | ne, &total, ctl);
  if (threadIdx.x == 0) {
    unsigned long long base;
    if (res.global) {
      base = total ? atomicAdd(res.global, total) : 0ull;
    } else {
      base = ((unsigned long long)ctl->cand_count << 32) | ctl->out_count;
      ctl->out_count += (unsigned)total;
      ctl->cand_count += (unsigned)(total >> 32);
    }
    ctl->base64 = base;
  }
  __syncthreads();
  const unsigned long long base = ctl->base64;
  unsigned eo = (unsigned)base + (unsigned)mine;
  unsigned co = (unsigned)(base >> 32) + (unsigned)(mine >> 32);
  bool bad = false;
  src.visit([&](uint32_t key, int pos, bool valid) {
    if (!valid) return;
    const int c = prefix_cmp(P, key, pmax - (uint32_t)pos);
    if (c > 0 || (c == 0 && !collect)) {
      if (eo < k)
        out_row[eo] = pos;
      else
        bad = true;
      ++eo;
    } else if (c == 0) {
      if (co < cap)
        cand[co] = make_uint2(key, (uint32_t)pos);
      else
        bad = true;
      ++co;
    }
  });
  if (bad) atomicOr(status, kStatInternal);
  __syncthreads();
}

// Finds the threshold bin for round D; false (and an error) if the counts
// are inconsistent, which cannot happen unless memory was corrupted.
__device__ __forceinline__ bool pick_bin(const unsigned* h, int nb, unsigned k_rem, Ctl* ctl,
                                         unsigned* status, unsigned* bin, unsigned* above,
                                         unsigned* cnt) {
  if (threadIdx.x == 0) ctl->pick_bin = 0xFFFFFFFFu;
  find_bin(h, nb, k_rem, ctl);
  *bin = ctl->pick_bin;
  *above = ctl->pick_above;
  *cnt = ctl->pick_cnt;
  if (*bin == 0xFFFFFFFFu) {
    if (threadIdx.x == 0) atomicOr(status, kStatInternal);
    return false;
  }
  return true;
}

// Refines candidates held on chip until the k_rem wanted among them are
// known, then writes them.  Rounds continue at digit t.
template <int DT>
__device__ void finish_on_chip(const uint2* cand, unsigned n, unsigned k_rem, Prefix P, int t,
                               int pos_bits, uint32_t pmax, unsigned* h, int32_t* out_row,
                               unsigned k, Ctl* ctl, unsigned* status) {
  const CandSrc src{cand, n};
  const int nr = num_rounds<DT>(pos_bits);
  for (;;) {
    if (t >= nr) {
      if (threadIdx.x == 0) atomicOr(status, kStatInternal);
      return;
    }
    const Digit D = digit_of_round<DT>(t, pos_bits);
    const int nb = 1 << D.bits;
    zero_hist(h, nb);
    __syncthreads();
    hist_round(src, h, P, D, pmax);
    __syncthreads();
    unsigned bin, above, cnt;
    if (!pick_bin(h, nb, k_rem, ctl, status, &bin, &above, &cnt)) return;
    prefix_extend(P, D, bin);
    k_rem -= above;
    if (cnt == k_rem) break;
    ++t;
  }
  emit(src, P, pmax, false, Reserve{nullptr}, out_row, k, nullptr, 0u, ctl, status);
}

// Selects the top k of row r with this block as part `part` of `group`.
// Returns false after an unrecoverable device-side error.
template <int DT>
__device__ bool select_row(const Params& p, int r, int part, unsigned char* smem,
                           unsigned& phase_bits) {
  using E = Elt<DT>;
  Ctl* ctl = reinterpret_cast<Ctl*>(smem + kCtlOff);
  unsigned* h = reinterpret_cast<unsigned*>(smem + kHistOff);
  unsigned char* sl = smem + kSliceOff;
  uint2* lcand = reinterpret_cast<uint2*>(smem + kLocalCandOff);
  unsigned* status = reinterpret_cast<unsigned*>(p.ws);
  const int group = p.group;
  const unsigned k = (unsigned)p.k;
  int32_t* out_row = p.out + (int64_t)r * p.k;

  __syncthreads();  // the previous row is done with ctl
  if (threadIdx.x == 0) {
    ctl->ok = 1u;
    ctl->out_count = 0u;
    ctl->cand_count = 0u;
  }

  // Valid length (clamped; a bad one is reported).
  int64_t Lr = p.row_len ? (int64_t)__ldg(p.row_len + r) : p.row_stride;
  if (Lr < 0 || Lr > p.row_stride) {
    if (threadIdx.x == 0 && part == 0) atomicOr(status, kStatRowLen);
    Lr = Lr < 0 ? 0 : p.row_stride;
  }
  const int L = (int)Lr;

  // Rows with no more than k elements: every position, then -1.
  if ((unsigned)L <= k) {
    for (int64_t i = (int64_t)part * kThreads + threadIdx.x; i < (int64_t)k;
         i += (int64_t)kThreads * group)
      out_row[i] = i < L ? (int32_t)i : -1;
    return true;
  }

  const int pos_bits = 32 - __clz(L - 1);  // 1..31
  const uint32_t pmax = (pos_bits == 32) ? 0xFFFFFFFFu : ((1u << pos_bits) - 1u);
  const int nr = num_rounds<DT>(pos_bits);

  // This block's slice, with 16-byte aligned interior boundaries.
  const unsigned char* row = p.logits + (int64_t)r * p.row_stride * E::ES;
  const int mis = (int)(((uintptr_t)row & 15u) / E::ES);
  auto align_up = [&](int64_t i) -> int64_t { return i + (E::V - (mis + i) % E::V) % E::V; };
  auto align_down = [&](int64_t i) -> int64_t { return i - (mis + i) % E::V; };
  const int64_t chunk = (((int64_t)L + group - 1) / group + E::V - 1) / E::V * E::V;
  Slice s;
  s.lo = part == 0 ? 0 : (int)min((int64_t)L, align_up((int64_t)part * chunk));
  s.hi = part == group - 1 ? L : (int)min((int64_t)L, align_up((int64_t)(part + 1) * chunk));
  s.bl = (int)min((int64_t)s.hi, align_up(s.lo));
  s.bh = (int)max((int64_t)s.bl, align_down(s.hi));
  s.o = s.lo < s.bl ? s.bl - E::V : s.bl;
  s.nvec = (s.hi - s.o + E::V - 1) / E::V;
  s.resident = (int64_t)s.nvec * 16 <= kSliceBytes;
  const SliceSrc<DT> src{row, sl, s};

  SlotHdr* slot = nullptr;
  unsigned* slot_hist = nullptr;
  uint2* slot_cand = nullptr;
  if (group > 1) {
    unsigned char* base = p.ws + kWsHeaderBytes + (size_t)(blockIdx.x / group) * kSlotBytes;
    slot = reinterpret_cast<SlotHdr*>(base);
    slot_hist = reinterpret_cast<unsigned*>(base + kSlotHistOff);
    slot_cand = reinterpret_cast<uint2*>(base + kSlotCandOff);
  }

  // ---- round 0: one pass over HBM, histogram of the top 12 key bits ----
  zero_hist(h, kMaxBins);
  if (s.resident) {
    const int vb0 = s.lo < s.bl ? 1 : 0;
    const int nbv = (s.bh - s.bl) / E::V;
    if (threadIdx.x == 0) {
      fence_proxy_async_smem();
      for (int c = 0; c < kChunks; ++c) {
        const int c0 = (int)((int64_t)nbv * c / kChunks), c1 = (int)((int64_t)nbv * (c + 1) / kChunks);
        if (c1 > c0) {
          const unsigned bytes = (unsigned)(c1 - c0) * 16u;
          mbar_arrive_expect_tx(&ctl->mbar[c], bytes);
          bulk_copy_g2s(sl + (size_t)(vb0 + c0) * 16, row + (int64_t)s.bl * E::ES + (int64_t)c0 * 16,
                        bytes, &ctl->mbar[c]);
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
    auto f0 = [&](uint32_t key, int, bool valid) { hist_add(h, key >> E::kShift0, valid); };
    src.visit_vecs(0, vb0, f0);
    src.visit_vecs(vb0 + nbv, s.nvec, f0);
    for (int c = 0; c < kChunks; ++c) {
      const int c0 = (int)((int64_t)nbv * c / kChunks), c1 = (int)((int64_t)nbv * (c + 1) / kChunks);
      if (c1 > c0) {
        mbar_wait_bounded(&ctl->mbar[c], (phase_bits >> c) & 1u, p.spin_limit_ns, ctl, status);
        phase_bits ^= 1u << c;
        src.visit_vecs(vb0 + c0, vb0 + c1, f0);
      }
    }
  } else {
    __syncthreads();
    src.visit_global([&](uint32_t key, int, bool valid) { hist_add(h, key >> E::kShift0, valid); });
  }
  __syncthreads();
  if (!ctl->ok) return false;

  // ---- digit rounds until the threshold bin is small or exact ----
  Prefix P = {0u, 0u, 0u, 0u};
  unsigned k_rem = k;
  int t = 0;
  bool collect = false;
  const unsigned cap = group > 1 ? (unsigned)kGroupCandCap : (unsigned)kLocalCandCap;
  for (;;) {
    const Digit D = digit_of_round<DT>(t, pos_bits);
    const int nb = 1 << D.bits;
    if (t > 0) {
      zero_hist(h, nb);
      __syncthreads();
      hist_round(src, h, P, D, pmax);
      __syncthreads();
    }
    if (group > 1) {
      const bool skip = p.test_skip_arrive && part == 0 && t == 0;
      if (!group_merge(h, nb, slot_hist + (size_t)t * kMaxBins, slot, (unsigned)group * (t + 1), skip,
                       p.spin_limit_ns, ctl, status))
        return false;
    }
    unsigned bin, above, cnt;
    if (!pick_bin(h, nb, k_rem, ctl, status, &bin, &above, &cnt)) return false;
    prefix_extend(P, D, bin);
    k_rem -= above;
    if (cnt == k_rem) break;  // the whole bin is selected
    if (cnt <= cap) {         // few enough to finish on one block
      collect = true;
      break;
    }
    if (++t >= nr) {
      if (threadIdx.x == 0) atomicOr(status, kStatInternal);
      return false;
    }
  }

  // ---- collection ----
  if (group == 1) {
    emit(src, P, pmax, collect, Reserve{nullptr}, out_row, k, lcand, cap, ctl, status);
    if (collect) {
      const unsigned n = min(ctl->cand_count, cap);
      finish_on_chip<DT>(lcand, n, k_rem, P, t + 1, pos_bits, pmax, h, out_row, k, ctl, status);
    }
    return true;
  }

  emit(src, P, pmax, collect, Reserve{&slot->alloc}, out_row, k, slot_cand, cap, ctl, status);
  if (threadIdx.x == 0) {
    __threadfence();
    const unsigned old = atomicAdd(&slot->done, 1u);
    ctl->is_last = (old == (unsigned)group - 1u) ? 1u : 0u;
    if (ctl->is_last) __threadfence();
  }
  __syncthreads();
  if (!ctl->is_last) return true;

  // The last block of the row: finish the candidates, then reset the slot.
  if (collect) {
    const unsigned long long a = ld_cg_u64(&slot->alloc);
    const unsigned n = min((unsigned)(a >> 32), cap);
    uint2* fc = reinterpret_cast<uint2*>(sl);  // this block's slice copy is no longer needed
    for (unsigned i = threadIdx.x; i < n; i += kThreads) fc[i] = ld_cg_u2(slot_cand + i);
    if (threadIdx.x == 0) {
      ctl->out_count = (unsigned)a;
      ctl->cand_count = 0u;
    }
    __syncthreads();
    finish_on_chip<DT>(fc, n, k_rem, P, t + 1, pos_bits, pmax, h, out_row, k, ctl, status);
  }
  for (int i = threadIdx.x; i < (t + 1) * kMaxBins; i += kThreads) slot_hist[i] = 0u;
  if (threadIdx.x == 0) {
    slot->arrive = 0u;
    slot->done = 0u;
    slot->alloc = 0ull;
  }
  return true;
}

template <int DT>
__global__ void __launch_bounds__(kThreads, 1) tks_select_kernel(const Params p) {
  extern __shared__ __align__(128) unsigned char smem[];
  Ctl* ctl = reinterpret_cast<Ctl*>(smem + kCtlOff);
  if (threadIdx.x == 0) {
    for (int c = 0; c < kChunks; ++c) mbar_init(&ctl->mbar[c], 1u);
    fence_mbar_init();
  }
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
};

std::mutex g_mu;
std::map<int, DeviceInfo> g_dev;
std::map<std::pair<int, void*>, Workspace> g_ws;

std::atomic<long long> g_force_group{0};
std::atomic<long long> g_spin_limit_ns{1000000000LL};
std::atomic<long long> g_min_per_block{4096};
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
  const int per = cap / batch;
  long long g;
  const long long forced = g_force_group.load();
  if (forced > 0) {
    g = forced;
  } else {
    const long long mpb = g_min_per_block.load() > 0 ? g_min_per_block.load() : 1;
    g = (row_stride + mpb - 1) / mpb;
  }
  if (g > per) g = per;
  if (g < 1) g = 1;
  *group = (int)g;
  *grid = batch * (int)g;
}

size_t workspace_bytes(const DeviceInfo& d) {
  return kWsHeaderBytes + (size_t)d.sms * d.blocks_per_sm * kSlotBytes;
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
  if (cudaMalloc(&w.ptr, w.bytes) != cudaSuccess) {
    cudaGetLastError();
    return TKS_E_CUDA;
  }
  if (cudaMemsetAsync(w.ptr, 0, w.bytes, (cudaStream_t)stream) != cudaSuccess) {
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
  p.spin_limit_ns = g_spin_limit_ns.load();

  cudaLaunchConfig_t cfg;
  std::memset(&cfg, 0, sizeof cfg);
  cfg.gridDim = dim3((unsigned)grid, 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = (cudaStream_t)stream;
  cudaLaunchAttribute attr[1];
  std::memset(attr, 0, sizeof attr);
  if (group > 1) {
    // blocks of a row wait for one another: they must all be resident
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
  }
  cudaError_t e = dtype == TKS_F32 ? cudaLaunchKernelEx(&cfg, tks_select_kernel<0>, p)
                                   : cudaLaunchKernelEx(&cfg, tks_select_kernel<1>, p);
  if (e != cudaSuccess) {
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
  if (cudaMemsetAsync(w.ptr, 0, w.bytes, (cudaStream_t)stream) != cudaSuccess ||
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
