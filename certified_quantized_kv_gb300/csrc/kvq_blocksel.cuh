// kvq_blocksel.cuh -- block-wide (BS_THREADS-thread) reductions and the "top blocks covering a
// target" selection used by the top-K* pass and by rungs 1-2 of the ladder.
//
// Selection rule ("Runtime-Certified Bounded-Error Quantized Attention", gist.science
// technical summary, Method §3): take blocks in descending value, ties to the lower
// block index, until the taken weight reaches the target.  Values v_i in [0, 1] are
// passed as keys (fp32 bits, order-preserving for v >= 0; 0 = not a candidate) and
// weighted in fixed point, w_i = floor(v_i 2^62), so every sum is an exact integer and
// the choice does not depend on summation order.
//
// Method: one block reduction gives the total weight, the number of candidates and the
// smallest and largest candidate key (the first level's histograms are cleared
// meanwhile).  The threshold key is then narrowed by histogram levels over the current
// key range [lo, hi], cut linearly into 1024 buckets (keys are order-preserving fp32
// bits, so this is a logarithmic cut of the values): each group of warps accumulates
// its keys' weights into a private histogram, the warps' running totals of the summed
// histograms locate the warp that holds the bucket where the weight from the top
// reaches the target, that warp finds the bucket, and the bucket's key range becomes the
// next [lo, hi]; its keys are gathered in the same pass that counts them.  Once it holds
// at most SEL_CAND keys they are ranked exactly (one key value left: ties go to the lower
// indices).  Near-uniform values usually need a single level.
#pragma once

#include "kvq_common.cuh"

namespace kvq {

constexpr int BS_THREADS = 512;                   // per (sequence, head): latency-bound work
constexpr int BS_WARPS = BS_THREADS / 32;
constexpr int BS_NHIST = 4;                        // private histograms, BS_WARPS / BS_NHIST warps each
constexpr int BS_BPT = 1024 / BS_THREADS;          // histogram buckets per thread in the scan
static_assert(SEL_CAND <= BS_THREADS, "one thread per exactly ranked candidate");
static_assert(BS_WARPS % BS_NHIST == 0 && 1024 % BS_THREADS == 0, "block shape");

struct BlockRed {
  unsigned long long u[BS_WARPS];   // per-warp totals of block_excl_scan_u64
};

// Exclusive prefix sum over the block in thread order; *total = the block total.
__device__ __forceinline__ unsigned long long block_excl_scan_u64(unsigned long long v, BlockRed& r,
                                                                  unsigned long long* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  unsigned long long incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned long long t = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += t;
  }
  __syncthreads();
  if (lane == 31) r.u[warp] = incl;
  __syncthreads();
  unsigned long long before = 0, tot = 0;
#pragma unroll
  for (int w = 0; w < BS_WARPS; ++w) {
    if (w < warp) before += r.u[w];
    tot += r.u[w];
  }
  *total = tot;
  return before + incl - v;
}

// Exact 64-bit add to a shared-memory bucket with two native 32-bit atomics (a 64-bit
// shared atomic add is a compare-and-swap loop, slow when many lanes hit one bucket):
// the low word's wrap-around, seen in the value the atomic returns, carries into the
// high word, so the bucket read as a 64-bit integer is the exact sum.
__device__ __forceinline__ void hist_add(unsigned long long* bucket, unsigned long long w) {
  uint32_t* h = reinterpret_cast<uint32_t*>(bucket);   // little endian: h[0] low, h[1] high
  const uint32_t lo = (uint32_t)w, hi = (uint32_t)(w >> 32);
  const uint32_t old = atomicAdd(&h[0], lo);
  const uint32_t carry = (old + lo < old) ? 1u : 0u;
  if (hi + carry) atomicAdd(&h[1], hi + carry);
}

// Blocks owned by a thread in the per-block passes of the selection and combine kernels and
// of block_select_top: the contiguous range [tid kpt, tid kpt + kpt), kpt = sel_kpt(n) a
// multiple of 4 (one 16-byte load of fp32 values per four blocks).  A thread reads back
// only the keys it wrote itself, so no barrier separates writing the keys and selecting.
__device__ __forceinline__ int sel_kpt(int n) {
  return ((n + 4 * BS_THREADS - 1) / (4 * BS_THREADS)) * 4;
}

// floor(d 1024 / span) for 0 <= d < span <= 2^32: the fp32 estimate d 1024 inv_span is
// within 2^-12 of the quotient (three roundings of at most 2^-24 relative each, quotient
// below 1024), so its floor is off by at most one, and one exact 64-bit comparison each
// way corrects it.  The bucket edges must be exact: the next level's key range is the
// crossing bucket's, ceil(b span / 1024) .. ceil((b + 1) span / 1024) - 1 above lo.
__device__ __forceinline__ uint32_t sel_bucket(uint32_t d, unsigned long long span, float inv_span) {
  const unsigned long long x = (unsigned long long)d << 10;
  uint32_t q = (uint32_t)fminf((float)x * inv_span, 1023.f);
  if ((unsigned long long)q * span > x) --q;
  else if ((unsigned long long)(q + 1u) * span <= x) ++q;
  return q;
}

// Shared-memory workspace of block_select_top, at the start of the kernel's dynamic shared
// memory; the keys (one per block, padded to 16) follow it.
struct BlockSelSmem {
  unsigned long long hist[BS_NHIST][1024];   // private histograms of groups of warps
  alignas(16) int cidx[SEL_CAND];
  alignas(16) uint32_t ckey[SEL_CAND];
  int order[SEL_CAND];
  unsigned long long wtot[BS_WARPS];         // per-warp weight totals (statistics, scan)
  int wnz[BS_WARPS];
  uint32_t kmin[BS_WARPS], kmax[BS_WARPS];
  unsigned long long above;
  unsigned long long take_w;
  uint32_t prefix;
  int ncand;
  int cnt;
  int last;
  BlockRed red;
};

__device__ __forceinline__ BlockSelSmem& sel_smem() {
  extern __shared__ __align__(16) unsigned char kvq_sel_dsm[];
  return *reinterpret_cast<BlockSelSmem*>(kvq_sel_dsm);
}
__device__ __forceinline__ uint32_t* sel_keys() {
  extern __shared__ __align__(16) unsigned char kvq_sel_dsm[];
  return reinterpret_cast<uint32_t*>(kvq_sel_dsm + sizeof(BlockSelSmem));
}

// Sums and extrema over the 16 warps' slots: lane l takes slot l mod 16 and the lanes of
// each half warp combine theirs, so every lane ends with the block's value.
__device__ __forceinline__ float xw_sum(float v) {
#pragma unroll
  for (int o = 8; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ float xw_max(float v) {
#pragma unroll
  for (int o = 8; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ unsigned long long xw_sum_u64(unsigned long long v) {
#pragma unroll
  for (int o = 8; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
static_assert(BS_WARPS == 16, "cross-warp reductions take one slot per lane of a half warp");

struct SelResult {
  int count;                    // blocks taken
  unsigned long long taken;     // their weight
};

// Marks (marks[i] = 1) the blocks with the largest keys, ties to the lower index, until
// the taken weight reaches target; keys are the n keys after the workspace, each thread's
// own range written by that thread.  Every thread of the block must call it; the result is
// the same in every thread.  Barriers: one after the statistics, four per histogram level
// (accumulate, scan, crossing, gather), one at the end.
static __device__ __noinline__ SelResult block_select_top(int n, unsigned long long target, uint8_t* marks) {
  BlockSelSmem& ws = sel_smem();
  const uint32_t* keys = sel_keys();
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int kpt = sel_kpt(n);
  const int i0 = min(n, tid * kpt), i1 = min(n, i0 + kpt);
  // the first level's histograms are cleared while the statistics are taken
  {
    uint4* hz = reinterpret_cast<uint4*>(&ws.hist[0][0]);
#pragma unroll
    for (int d = 0; d < BS_NHIST * 1024 / 2 / BS_THREADS; ++d) hz[tid + BS_THREADS * d] = make_uint4(0, 0, 0, 0);
  }
  if (tid == 0) ws.ncand = 0;   // the previous call read it before its last barrier
  // total weight, candidates (nonzero keys) and their key range
  unsigned long long tot = 0;
  int nz = 0;
  uint32_t lo = 0xffffffffu, hi = 0u;
  for (int i = i0; i < i1; ++i) {
    const uint32_t k = keys[i];
    if (k != 0u) {
      tot += key_weight(k);
      ++nz;
      lo = min(lo, k);
      hi = max(hi, k);
    }
  }
  tot = warp_sum_u64(tot);
  nz = (int)__reduce_add_sync(0xffffffffu, (unsigned)nz);
  lo = __reduce_min_sync(0xffffffffu, lo);
  hi = __reduce_max_sync(0xffffffffu, hi);
  if (lane == 0) {
    ws.wtot[warp] = tot;
    ws.wnz[warp] = nz;
    ws.kmin[warp] = lo;
    ws.kmax[warp] = hi;
  }
  __syncthreads();
  if (tid == 0) ws.cnt = 0;     // every thread has read the previous call's count
  tot = xw_sum_u64(ws.wtot[lane & 15]);
  nz = (int)(__reduce_add_sync(0xffffffffu, (unsigned)ws.wnz[lane & 15]) >> 1);   // each slot twice
  lo = __reduce_min_sync(0xffffffffu, ws.kmin[lane & 15]);
  hi = __reduce_max_sync(0xffffffffu, ws.kmax[lane & 15]);
  SelResult res;
  res.count = 0;
  res.taken = 0ull;
  if (target == 0ull || tot < target) {
    if (target != 0ull) {   // out of reach: take every candidate
      for (int i = i0; i < i1; ++i)
        if (keys[i] != 0u) marks[i] = 1;
      res.count = nz;
      res.taken = tot;
    }
    __syncthreads();   // every warp has read the per-warp slots before the next call writes them
    return res;
  }
  // candidates in [glo, ghi] to ws.cidx / ws.ckey (ws.ncand counts them all; those past
  // SEL_CAND are not stored), one shared atomic per warp and step
  auto gather = [&](uint32_t glo, uint32_t ghi) {
    const unsigned lt_mask = (1u << lane) - 1u;
    for (int j = 0; j < kpt; ++j) {
      const int i = i0 + j;
      const uint32_t k = i < i1 ? keys[i] : 0u;
      const bool c = k != 0u && k >= glo && k <= ghi;
      const unsigned m = __ballot_sync(0xffffffffu, c);
      if (m == 0u) continue;
      int base = 0;
      if (lane == __ffs(m) - 1) base = atomicAdd(&ws.ncand, __popc(m));
      base = __shfl_sync(0xffffffffu, base, __ffs(m) - 1);
      if (c) {
        const int slot = base + __popc(m & lt_mask);
        if (slot < SEL_CAND) {
          ws.cidx[slot] = i;
          ws.ckey[slot] = k;
        }
      }
    }
  };
  // candidates are the keys in [lo, hi]; `above` = weight of the keys above hi
  unsigned long long above = 0;
  int ncand = nz;
  if (ncand <= SEL_CAND) {
    gather(lo, hi);
    __syncthreads();
  }
  for (int level = 0; ncand > SEL_CAND && hi > lo && level < 4; ++level) {
    if (level > 0) {
      uint4* hz = reinterpret_cast<uint4*>(&ws.hist[0][0]);
#pragma unroll
      for (int d = 0; d < BS_NHIST * 1024 / 2 / BS_THREADS; ++d) hz[tid + BS_THREADS * d] = make_uint4(0, 0, 0, 0);
      __syncthreads();
      if (tid == 0) ws.ncand = 0;   // read by every thread before the barrier above
    }
    const unsigned long long span = (unsigned long long)(hi - lo) + 1ull;
    const float inv_span = 1.0f / (float)span;
    const int hg = warp / (BS_WARPS / BS_NHIST);
    for (int i = i0; i < i1; ++i) {
      const uint32_t k = keys[i];
      if (k != 0u && k >= lo && k <= hi)
        hist_add(&ws.hist[hg][sel_bucket(k - lo, span, inv_span)], key_weight(k));
    }
    __syncthreads();
    // thread t owns buckets 1023 - BS_BPT t - j, j < BS_BPT (descending): warp 0 the top ones
    unsigned long long bw[BS_BPT], run = 0;
#pragma unroll
    for (int j = 0; j < BS_BPT; ++j) {
      const int bk = 1023 - BS_BPT * tid - j;
      unsigned long long sum = 0;
#pragma unroll
      for (int w = 0; w < BS_NHIST; ++w) sum += ws.hist[w][bk];
      bw[j] = sum;
      run += sum;
    }
    unsigned long long incl = run;   // inclusive scan within the warp
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const unsigned long long t = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += t;
    }
    if (lane == 31) ws.wtot[warp] = incl;
    __syncthreads();
    // the warp holding the crossing: the first whose running total (from the top) reaches
    // the target; only its threads look for the bucket
    unsigned long long winc = ws.wtot[lane & 15];
#pragma unroll
    for (int o = 1; o < 16; o <<= 1) {
      const unsigned long long t = __shfl_up_sync(0xffffffffu, winc, o, 16);
      if ((lane & 15) >= o) winc += t;
    }
    const unsigned cross = __ballot_sync(0xffffffffu, lane < 16 && above + winc >= target);
    const int wstar = __ffs(cross) - 1;
    const unsigned long long before = __shfl_sync(0xffffffffu, winc, wstar > 0 ? wstar - 1 : 0);
    if (warp == wstar) {
      unsigned long long c = above + (wstar > 0 ? before : 0ull) + (incl - run);
#pragma unroll
      for (int j = 0; j < BS_BPT; ++j) {
        if (c < target && c + bw[j] >= target) {
          ws.prefix = (uint32_t)(1023 - BS_BPT * tid - j);
          ws.above = c;
        }
        c += bw[j];
      }
    }
    __syncthreads();
    // the crossing bucket b holds the keys lo + ceil(b span / 1024) .. lo + ceil((b + 1) span / 1024) - 1
    const unsigned long long b = ws.prefix;
    above = ws.above;
    const uint32_t nlo = lo + (uint32_t)((b * span + 1023ull) / 1024ull);
    const uint32_t nhi = lo + (uint32_t)(((b + 1ull) * span + 1023ull) / 1024ull) - 1u;
    lo = nlo;
    hi = nhi;
    gather(lo, hi);
    __syncthreads();
    ncand = ws.ncand;
  }
  const unsigned long long rem = target - above;
  int cnt = 0;
  unsigned long long take_w = 0;
  bool small = false;   // the candidates were ranked by warp 0 alone
  if (ncand > SEL_CAND) {
    // one key value left (lo == hi) with more keys than the exact ranking takes: ties,
    // lowest indices first
    const unsigned long long wt = key_weight(lo);
    const unsigned long long need = wt ? (rem + wt - 1) / wt : 0ull;
    int mine = 0;
    for (int i = i0; i < i1; ++i) mine += (keys[i] != 0u && keys[i] == lo);
    unsigned long long ties;
    unsigned long long rank = block_excl_scan_u64((unsigned long long)mine, ws.red, &ties);
    for (int i = i0; i < i1; ++i) {
      const uint32_t k = keys[i];
      if (k == 0u) continue;
      if (k > lo) { marks[i] = 1; ++cnt; }
      else if (k == lo) {
        if (rank < need) { marks[i] = 1; ++cnt; }
        ++rank;
      }
    }
    take_w = (need < ties ? need : ties) * wt;
  } else {
    const int nc = ncand;   // gathered in ws.cidx / ws.ckey
    for (int i = i0; i < i1; ++i)
      if (keys[i] > hi) { marks[i] = 1; ++cnt; }
    if (nc <= 32) {
      // few candidates: warp 0 ranks them with shuffles (no block barrier)
      if (warp == 0) {
        const bool live = lane < nc;
        const uint32_t ka = live ? ws.ckey[lane] : 0u;
        const int ia = live ? ws.cidx[lane] : 0x7fffffff;
        const unsigned long long wa = live ? key_weight(ka) : 0ull;
        // weight of the candidates ranked before this one (key descending, index
        // ascending); weights are non-negative, so a candidate is taken exactly when that
        // weight is below the remainder, and the one whose running weight reaches it is
        // the last taken
        unsigned long long excl = 0ull, tot_c = 0ull;
        for (int j = 0; j < nc; ++j) {
          const uint32_t kb = __shfl_sync(0xffffffffu, ka, j);
          const int ib = __shfl_sync(0xffffffffu, ia, j);
          const unsigned long long wb = __shfl_sync(0xffffffffu, wa, j);
          if ((kb > ka) || (kb == ka && ib < ia)) excl += wb;
          tot_c += wb;
        }
        const unsigned crossing = __ballot_sync(0xffffffffu, live && excl < rem && excl + wa >= rem);
        const unsigned long long tw = crossing ? __shfl_sync(0xffffffffu, excl + wa, __ffs(crossing) - 1) : tot_c;
        if (live && excl < rem) { marks[ia] = 1; ++cnt; }
        if (lane == 0) ws.take_w = tw;   // read after the closing barrier
      }
      small = true;
    } else {
      const int nc4 = (nc + 3) & ~3;
      if (tid >= nc && tid < nc4) ws.ckey[tid] = 0u;   // padding ranks below every candidate
      __syncthreads();
      // rank of candidate a = number of candidates before it (key descending, index
      // ascending); nc <= SEL_CAND <= BS_THREADS, four candidates per 16-byte load
      if (tid < nc) {
        const uint32_t ka = ws.ckey[tid];
        const int ia = ws.cidx[tid];
        int rank = 0;
#pragma unroll 4
        for (int b4 = 0; b4 < nc4; b4 += 4) {
          const uint4 kb = *reinterpret_cast<const uint4*>(&ws.ckey[b4]);
          const int4 ib = *reinterpret_cast<const int4*>(&ws.cidx[b4]);
          rank += (kb.x > ka) || (kb.x == ka && ib.x < ia);
          rank += (kb.y > ka) || (kb.y == ka && ib.y < ia);
          rank += (kb.z > ka) || (kb.z == ka && ib.z < ia);
          rank += (kb.w > ka) || (kb.w == ka && ib.w < ia);
        }
        ws.order[rank] = tid;
      }
      if (tid == 0) { ws.last = nc - 1; ws.take_w = 0ull; }
      __syncthreads();
      // running weight in rank order; thread r handles rank r (nc <= SEL_CAND <= BS_THREADS)
      const unsigned long long w = (tid < nc) ? key_weight(ws.ckey[ws.order[tid]]) : 0ull;
      unsigned long long tot_c;
      const unsigned long long excl = block_excl_scan_u64(w, ws.red, &tot_c);
      if (tid < nc && excl < rem && excl + w >= rem) { ws.last = tid; ws.take_w = excl + w; }
      __syncthreads();
      const int last = ws.last;
      take_w = (ws.take_w != 0ull || last < 0) ? ws.take_w : tot_c;
      if (tid <= last && tid < nc) { marks[ws.cidx[ws.order[tid]]] = 1; ++cnt; }
    }
  }
  cnt = (int)__reduce_add_sync(0xffffffffu, (unsigned)cnt);
  if (lane == 0 && cnt) atomicAdd(&ws.cnt, cnt);
  __syncthreads();
  res.count = ws.cnt;
  res.taken = above + (small ? ws.take_w : take_w);
  return res;
}

}  // namespace kvq
