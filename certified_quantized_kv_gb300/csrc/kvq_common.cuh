// kvq_common.cuh -- layouts, launch views and device helpers shared by the kernels.
//
// Method: "Runtime-Certified Bounded-Error Quantized Attention" (gist.science technical
// summary), Method §1-§3.  This header fixes the tier-1 byte layouts, which are chosen
// so that every hot-loop load is a coalesced 16-byte load that lands directly in the
// register fragment of an mma.sync.m16n8k16 tile (no shared-memory staging, no bank
// conflicts):
//
//  K codes (INT8), per 64-token block, 8192 bytes:
//    offset((w*4 + j)*32 + lane)*16 + byte, w = token>>4 (MMA row tile), lane = gid*4+tig
//    row  = 16w + gid + 8*(j>>1),   channel = 32*tig + 16*(j&1) + byte.
//    In k-step kk (0..7) the MMA column 2tig(+1) is channel 32tig+4kk(+1) and column
//    2tig+8(+9) is channel 32tig+4kk+2(+3): a thread's 32 channels are contiguous.
//  V codes (INT4), per block, 4096 bytes: 16-byte chunk ((g*2 + mt)*32 + lane), word kk,
//    g = channel>>5 (value group, = warp), mt = (channel>>4)&1, gid = channel&7,
//    chhalf = (channel>>3)&1, tig = token>>4, kk = (token>>2)&3, tpos = token&3;
//    nibble bit position 4*((tpos>>1)*2 + chhalf) + 16*(tpos&1).
//    For PV the MMA runs channels as rows and tokens as the k dimension; MMA column
//    2tig(+1) of k-step kk is token 16tig+4kk(+1), column 2tig+8(+9) token 16tig+4kk+2(+3).
//  V scale/offset, per block, 1024 bytes: half2 (scale, offset) at [group][token].
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace kvq {

constexpr int D = 128;           // head_dim
constexpr int BLK = 64;          // tokens per block
constexpr int VG = 32;           // channels per value group
constexpr int NG = D / VG;       // value groups per token
constexpr int MAXREP = 4;        // query heads per KV head held in one MMA tile
constexpr int KC_BYTES = BLK * D;          // 8192
constexpr int VC_BYTES = BLK * D / 2;      // 4096
constexpr int VSV_WORDS = BLK * NG;        // 256 half2
constexpr int F16_BLOCK_BYTES = BLK * D * 2;  // 16384 bytes of FP16 per block (K or V)
constexpr int CHUNK = 16;        // blocks per work item of the streaming kernels
constexpr float KAPPA = 0.5f + 1.0f / 256.0f;
constexpr float INV_SQRT_D = 0.088388347648318440550f;  // 1/sqrt(128), rounded to fp32

// Per (sequence, query head) state of one decode call.
struct HeadState {
  float M;          // reference >= every score of the head (exp(s - M) <= 1)
  float lse_int8;   // log-sum-exp over all tokens with INT8 scores for full blocks
  float tail_lse;   // log-sum-exp of the partial block's exact scores (-inf if none)
  int k_star;       // |S_h|
  int rank_ok;
  int planned;      // rung asked for after the first pass: 0, 1, 2, or 3 (rank failure)
  int level1;       // rung after the second pass (0..3)
  int level;        // final rung (0..4)
  float e_key, e_val;
  int n_vprom;
  int pad;
};

// Per (sequence, KV head) state.
struct GroupState {
  int need_round1;
  int need_dense;
  int n_kprom0, n_kprom1, n_vprom1;
  int pad;
  long long bytes;
};

// Everything a kernel needs to address one layer of the cache plus the call's scratch.
struct LayerView {
  // shape
  int B, Hq, Hkv, n_rep, BG;
  int nb;          // full blocks of the layer
  int n_tail;      // tokens in the partial block (0..63)
  int nbmax;       // block capacity per (sequence, KV head)
  long long cap;   // token capacity of tier 2 per (sequence, KV head)
  // tier 1 of this layer
  const int8_t* kc;      // [BG][nbmax][8192]
  const __half* ks;      // [BG][nbmax][128]
  const uint8_t* vc;     // [BG][nbmax][4096]
  const __half2* vsv;    // [BG][nbmax][256]
  const float* eta;      // [BG][nbmax]
  const uint32_t* vmin;  // [BG][128] order-preserving encoding
  const uint32_t* vmax;
  const uint32_t* kscale_max;  // [BG] fp16 bits of the largest key scale
  const uint32_t* vscale_max;  // [BG] fp16 bits of the largest value scale
  const __half* tail_k;  // [BG][64][128]
  const __half* tail_v;
  // tier 2 of this layer (device addresses of mapped pinned host memory)
  const __half* t2k;     // [BG][cap][128]
  const __half* t2v;
  // call inputs / outputs (device)
  const __half* q;       // [B][Hq][128]
  __half* out;           // [B][Hq][128]
  float tau, eps;
  float l4_frac;
  int rank_positions;
  int debug;
  // scratch
  float* shat;           // [B][Hq][nbmax*64]
  float* lse8;           // [B][Hq][nbmax]
  float* delta;
  float* lse16;
  uint8_t* sel;          // [B][Hq][nbmax]
  uint8_t* kprom0;       // [BG][nbmax]
  uint8_t* kprom1;
  uint8_t* vprom1;
  HeadState* hst;        // [B*Hq]
  GroupState* gst;       // [BG]
  float* part;           // [BG][nbmax/CHUNK+1][MAXREP][D+4] partials of the mixed pass
  float* dpart;          // [BG][nbmax/CHUNK+1][MAXREP][D+4] partials of the dense pass
  unsigned int* counters;  // work queues and completion counters (self-resetting)
};

// counters layout
constexpr int CNT_SCORE_Q = 0;      // work queue of the scoring pass
constexpr int CNT_SCORE_EXIT = 1;
constexpr int CNT_MIX_Q = 2;
constexpr int CNT_MIX_EXIT = 3;
constexpr int CNT_DENSE_Q = 4;
constexpr int CNT_DENSE_EXIT = 5;
constexpr int CNT_GROUP_BASE = 16;  // + stage*BG + hs: per-group completion counters
constexpr int N_STAGE_COUNTERS = 3;

// ---------------------------------------------------------------------------------
// small helpers
// ---------------------------------------------------------------------------------

__device__ __forceinline__ uint32_t f2ord(float f) {
  uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float ord2f(uint32_t u) {
  return __uint_as_float((u & 0x80000000u) ? (u & 0x7fffffffu) : ~u);
}

// D = A(16x16, f16, row) * B(16x8, f16, col) + C, fp32 accumulate.
__device__ __forceinline__ void mma16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t h2_as_u32(__half2 h) { return *reinterpret_cast<uint32_t*>(&h); }
__device__ __forceinline__ __half2 u32_as_h2(uint32_t u) { return *reinterpret_cast<__half2*>(&u); }

// Four signed INT8 codes (one 32-bit word) -> two f16x2 registers, exactly.
// Bias each byte to unsigned (b + 128), place it under the exponent pattern 0x64 so the
// half reads 1024 + (b + 128), then subtract 1152.  Every step is exact in binary16.
__device__ __forceinline__ void i8x4_to_f16(uint32_t w, uint32_t& lo, uint32_t& hi) {
  const uint32_t x = w ^ 0x80808080u;
  const uint32_t l = __byte_perm(x, 0x64646464u, 0x4140);
  const uint32_t h = __byte_perm(x, 0x64646464u, 0x4342);
  const __half2 bias = u32_as_h2(0x64806480u);  // (1152, 1152)
  lo = h2_as_u32(__hsub2(u32_as_h2(l), bias));
  hi = h2_as_u32(__hsub2(u32_as_h2(h), bias));
}

// Nibble pair i of a V-code word (bits 4i..4i+3 and 16+4i..16+4i+3) -> f16x2, exactly:
// 0x6400 | n reads 1024 + n; subtracting 1024 leaves n.
__device__ __forceinline__ uint32_t nib_to_f16(uint32_t w, int i) {
  const uint32_t t = ((w >> (4 * i)) & 0x000F000Fu) | 0x64006400u;
  return h2_as_u32(__hsub2(u32_as_h2(t), u32_as_h2(0x64006400u)));
}

// x = hi + lo with hi = rn16(x), lo = rn16(x - hi); exact unless lo is subnormal.
__device__ __forceinline__ void split_hl(float x, __half& hi, __half& lo) {
  hi = __float2half_rn(x);
  lo = __float2half_rn(x - __half2float(hi));
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ double warp_sum_d(double v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Power-of-two prescale so that |x| * 2^e <= 2^14 for |x| <= xmax (keeps split halves
// normal and far from overflow).  Returns 2^e as a float.
__device__ __forceinline__ float prescale_for(float xmax) {
  if (!(xmax > 0.f)) return 1.f;
  int e;
  frexpf(xmax, &e);             // xmax = m * 2^e, m in [0.5, 1)
  int s = 14 - e;
  s = max(-100, min(100, s));
  return ldexpf(1.f, s);
}

// ---------------------------------------------------------------------------------
// Warp-cooperative "top blocks covering a target" selection (radix select).
//
// Among n values v_i >= 0 with fixed-point weights F_i (uint64, F_i = v_i/scale * 2^62),
// take blocks in descending v (ties: lower index first) until their F sum reaches
// target.  Keys are the fp32 bit patterns of v (order-preserving for v >= 0).  Zero
// values are never taken.  mark(i) is called for every taken block; the call returns
// their count and stores the sum of their weights in *taken (same value in every lane).
// Fixed-point integer sums make the choice independent of
// summation order.  hist: 256 uint64 of shared memory owned by this warp.
// ---------------------------------------------------------------------------------
template <typename KeyFn, typename WeightFn, typename MarkFn>
__device__ int warp_select_top(int n, unsigned long long target, KeyFn key_of, WeightFn w_of,
                               MarkFn mark, unsigned long long* hist,
                               unsigned long long* taken) {
  const int lane = threadIdx.x & 31;
  *taken = 0ull;
  if (target == 0ull) return 0;
  // total weight of strictly positive keys
  unsigned long long tot = 0;
  for (int i = lane; i < n; i += 32) {
    if (key_of(i) != 0u) tot += w_of(i);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) tot += __shfl_xor_sync(0xffffffffu, tot, o);
  if (tot < target) {  // the target is out of reach: take every positive block
    *taken = tot;
    int cnt = 0;
    for (int base = 0; base < n; base += 32) {   // uniform trip count for the ballot
      const int i = base + lane;
      const bool t = (i < n) && key_of(i) != 0u;
      if (t) mark(i);
      cnt += __popc(__ballot_sync(0xffffffffu, t));
    }
    return cnt;
  }
  uint32_t prefix = 0;             // decided high bits of the threshold key
  unsigned long long above = 0;    // weight of keys strictly above the current prefix range
  for (int pass = 0; pass < 4; ++pass) {
    const int shift = 24 - 8 * pass;
    for (int d = lane; d < 256; d += 32) hist[d] = 0ull;
    __syncwarp();
    for (int i = lane; i < n; i += 32) {
      const uint32_t k = key_of(i);
      if (k == 0u) continue;
      const bool match = (pass == 0) || ((k >> (shift + 8)) == prefix);
      if (match) atomicAdd(&hist[(k >> shift) & 255u], w_of(i));
    }
    __syncwarp();
    // lane L owns digits 255-8L .. 248-8L (descending); suffix scan from the top
    unsigned long long loc[8];
    unsigned long long run = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      loc[j] = hist[255 - 8 * lane - j];
      run += loc[j];
    }
    unsigned long long incl = run;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const unsigned long long t = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += t;
    }
    const unsigned long long excl = incl - run;
    // find first digit (from the top) where above + cumulative >= target
    int found = -1;
    unsigned long long before = 0;
    {
      unsigned long long c = above + excl;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        if (found < 0 && c + loc[j] >= target) {
          found = 255 - 8 * lane - j;
          before = c;
        }
        c += loc[j];
      }
    }
    const unsigned int has = __ballot_sync(0xffffffffu, found >= 0);
    const int src = __ffs(has) - 1;  // lowest lane = highest digits
    const int dsel = __shfl_sync(0xffffffffu, found, src);
    above = __shfl_sync(0xffffffffu, before, src);
    prefix = (prefix << 8) | (uint32_t)dsel;
    __syncwarp();
  }
  // prefix is now the full threshold key; `above` = weight of keys > prefix.
  // ties: take the lowest-index blocks with key == prefix until the target is met.
  unsigned long long wt = 0;
  for (int i = lane; i < n; i += 32)
    if (key_of(i) == prefix) { wt = w_of(i); }
  // all ties share one key, hence one weight (weights are a function of the key)
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const unsigned long long t = __shfl_xor_sync(0xffffffffu, wt, o);
    wt = wt > t ? wt : t;
  }
  const unsigned long long rem = target - above;
  const unsigned long long need = wt ? (rem + wt - 1) / wt : 0ull;
  int cnt = 0;
  unsigned long long ties_seen = 0;
  for (int base = 0; base < n; base += 32) {
    const int i = base + lane;
    const uint32_t k = (i < n) ? key_of(i) : 0u;
    const bool gt = (i < n) && k != 0u && k > prefix;
    const bool eq = (i < n) && k != 0u && k == prefix;
    const unsigned int eqm = __ballot_sync(0xffffffffu, eq);
    const unsigned long long rank = ties_seen + __popc(eqm & ((1u << lane) - 1u));
    const bool take = gt || (eq && rank < need);
    if (take) mark(i);
    cnt += __popc(__ballot_sync(0xffffffffu, take));
    ties_seen += __popc(eqm);
  }
  const unsigned long long nt = need < ties_seen ? need : ties_seen;
  *taken = above + nt * wt;
  return cnt;
}

}  // namespace kvq
