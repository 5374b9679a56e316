// kvq_common.cuh -- layouts, launch views and device helpers shared by the kernels.
//
// Method: "Runtime-Certified Bounded-Error Quantized Attention" (gist.science technical
// summary), Method §1-§3.  This header fixes the tier-1 byte layouts, which are chosen
// so that every hot-loop load is a coalesced 16-byte load that lands directly in the
// register fragment of an mma.sync.m16n8k16 tile (no shared-memory staging, no bank
// conflicts):
//
//  K codes (INT8, stored offset binary: byte = code + 128), per 64-token block, 8192 bytes:
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
constexpr int CHUNK = 16;        // most blocks per work item of the mixed and dense passes
constexpr int ITEMS_PER_CTA = 3; // work items per resident CTA the split aims for
constexpr float KAPPA = 0.5f + 1.0f / 256.0f;
constexpr float INV_SQRT_D = 0.088388347648318440550f;  // 1/sqrt(128), rounded to fp32

// Per (sequence, query head) state of one decode call.
struct HeadState {
  float M;          // softmax reference of the head: after the selection the largest INT8
                    // block log-mass or partial-block score (>= every INT8 score); after a
                    // combine the largest reference of that pass's work items (>= every
                    // score the pass used)
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
  int nbmax;       // block capacity per (sequence, KV head), a multiple of 16
  int chunk;       // blocks per work item of the mixed and dense passes (1..CHUNK)
  int nslot;       // partial slots per KV group (>= the work items of a group)
  int nparts;      // partial slots the combine kernel adds (0: one per work item)
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
  const __half* t2v;     // nullptr with FP16 values in tier 1
  const __half* v16;     // [BG][nbmax][64][128] FP16 values in tier 1, or nullptr (INT4)
  // call inputs / outputs (device)
  const __half* q;       // [B][Hq][128]
  __half* out;           // [B][Hq][128]
  float tau, eps;
  float l4_frac;
  float v_tol;           // budget on E_val alone (+inf: none)
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
  float* part;           // [BG][nslot][MAXREP][D+4] partials of the mixed pass: D
                         // channel sums, then the weight sum l and the item's reference M
                         // (weights are exp(s - M))
  float* part1;          // same shape: deltas of the second mixed pass
  float* red0;           // [B*Hq][D+4] the first pass's partials summed (channels, then l)
  float* dpart;          // [BG][nslot][MAXREP][D+4] partials of the dense pass
  unsigned int* counters;  // work queues and completion counters (self-resetting)
  // cross-step residency of FP16 tier-2 blocks in HBM (nres == 0: off)
  int nres;              // slots of this layer
  unsigned int call_id;  // certified decode calls of this layer so far (stamps slot use)
  int* rslot_k;          // [BG][nbmax] slot holding the block's keys, or -1
  int* rslot_v;          // [BG][nbmax] slot holding the block's values, or -1
  __half* rpool;         // [nres][64][128]
  int* rowner;           // [nres] (kv << 30) | (hs * nbmax + blk), or -1
  unsigned int* rstamp;  // [nres] call_id of the last call that used the slot
  int* rfree;            // [nres] free slots (the first rstate[RS_NFREE] entries)
  unsigned int* rstate;  // RS_* below
  unsigned long long* rbytes;  // [2] bytes served from slots, bytes read over the host link
};

// residency state words
constexpr int RS_NFREE = 0;   // free slots at the start of the call (rfree[0, NFREE))
constexpr int RS_TAKEN = 1;   // claims during the call (from the top of the free stack)
constexpr int RS_USED = 2;    // slots holding a block after the last eviction pass
constexpr int RS_PUSHED = 3;  // slots freed by the running eviction pass
constexpr int RS_DONE = 4;    // CTAs of the running eviction pass that have finished
constexpr int RS_WORDS = 8;

// counters layout
constexpr int CNT_MIX_Q = 2;
constexpr int CNT_MIX_EXIT = 3;
constexpr int CNT_DENSE_Q = 4;
constexpr int CNT_DENSE_EXIT = 5;
constexpr int CNT_ANY_DENSE = 6;    // set when a head reaches rung 3 (reset by the finaliser)
constexpr int CNT_NEED_R1 = 7;      // set when a head plans rung 1 or 2 (reset by the finaliser)
constexpr int CNT_BOUNDS = 8;       // KVQ_DEBUG_BOUNDS: site of the first violation (0: none)
constexpr int CNT_BOUNDS_AT = 9;    // ... and the index that was out of range (low 32 bits)
constexpr int CNT_GROUP_BASE = 16;  // + stage*BG + hs: per-group completion counters
constexpr int N_STAGE_COUNTERS = 3;
// + b after the four per-group stages: heads of sequence b at rung 3 after the ladder
// plan (kept by the combine kernels, read by the dense pass, cleared by the finaliser)
__host__ __device__ constexpr int cnt_rung3(int BG, int b) { return CNT_GROUP_BASE + 4 * BG + b; }

// ---------------------------------------------------------------------------------
// bounds checks (KVQ_DEBUG_BOUNDS)
// ---------------------------------------------------------------------------------

constexpr int DBG_BOUNDS = 0x10;   // the KVQ_DEBUG_BOUNDS bit of kvq_set_debug
// Kernels that check their indices; the host turns a recorded site into the kernel name.
enum BoundsSite : unsigned {
  SITE_SCORE = 1, SITE_SELECT, SITE_MIX0, SITE_MIX, SITE_COMBINE, SITE_TAIL, SITE_DENSE,
  SITE_FINAL, SITE_APPEND, SITE_COUNT
};

// With DBG_BOUNDS set, an index about to address an array of n elements is checked: the
// first index outside [0, n) of the call is recorded (site, index) in two counter words
// and false is returned, so the caller skips the access.  Nothing traps; the host reads
// the words after the call.  Without the flag this is one test of a uniform value.
__device__ __forceinline__ bool bounds_ok(unsigned int* counters, int debug, long long i, long long n,
                                          unsigned site) {
  if (!(debug & DBG_BOUNDS) || (i >= 0 && i < n)) return true;
  if (atomicCAS(&counters[CNT_BOUNDS], 0u, site) == 0u) counters[CNT_BOUNDS_AT] = (unsigned int)i;
  return false;
}

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

// q . k over the D channels of one FP16 row in fp32, fused multiply-adds in channel order
// (16-byte loads; both rows 16-byte aligned).
__device__ __forceinline__ float dot_f16_row(const __half* q, const __half* k) {
  const uint4* q4 = reinterpret_cast<const uint4*>(q);
  const uint4* k4 = reinterpret_cast<const uint4*>(k);
  float s = 0.f;
#pragma unroll 4
  for (int i = 0; i < D / 8; ++i) {
    const uint4 qv = q4[i], kv = k4[i];
    const uint32_t qw[4] = {qv.x, qv.y, qv.z, qv.w}, kw[4] = {kv.x, kv.y, kv.z, kv.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float2 qq = __half22float2(u32_as_h2(qw[j])), kk = __half22float2(u32_as_h2(kw[j]));
      s = fmaf(qq.x, kk.x, s);
      s = fmaf(qq.y, kk.y, s);
    }
  }
  return s;
}

// Four INT8 codes stored offset binary (byte = code + 128; one 32-bit word) -> two
// f16x2 registers, exactly: placed under the exponent pattern 0x64 a byte reads as the
// half 1024 + byte, and subtracting 1152 leaves the code.  Every step is exact in binary16.
__device__ __forceinline__ void i8x4_to_f16(uint32_t w, uint32_t& lo, uint32_t& hi) {
  const uint32_t l = __byte_perm(w, 0x64646464u, 0x4140);
  const uint32_t h = __byte_perm(w, 0x64646464u, 0x4342);
  const __half2 bias = u32_as_h2(0x64806480u);  // (1152, 1152)
  lo = h2_as_u32(__hsub2(u32_as_h2(l), bias));
  hi = h2_as_u32(__hsub2(u32_as_h2(h), bias));
}

// The four nibble pairs of a V-code word (pair i: bits 4i..4i+3 and 16+4i..16+4i+3) ->
// f16x2 MMA operands a0..a3 in five instructions, read as binary16 subnormals: with a zero
// exponent field the bits m of a half encode m * 2^-24 exactly.  Pairs 0 and 2 (of w, and
// of w with bytes 1 and 3 moved down by a byte permute) sit at bits 0-3 and 16-19 and read
// n * 2^-24; pairs 1 and 3 sit at bits 4-7 and 20-23 and read 16 n * 2^-24 = n * 2^-20.
// The tensor cores take subnormal f16 operands as they are (checked on GB300 against an
// fp64 sum: the accumulated error stays within 2.7e-6 of the sum of |products|, against
// 7.6e-7 for the same products with normal operands), so an MMA over these operands
// gives the code-weighted sum times 2^-24 in the rows of pairs 0/2 (A-fragment rows gid)
// and times 2^-20 in the rows of pairs 1/3 (rows gid + 8); NIB_ROW_SCALE_* undo that.
constexpr float NIB_ROW_SCALE_LO = 16777216.f;   // 2^24: accumulator rows gid
constexpr float NIB_ROW_SCALE_HI = 1048576.f;    // 2^20: accumulator rows gid + 8
__device__ __forceinline__ void nib8_to_sub_f16x4(uint32_t w, uint32_t& a0, uint32_t& a1, uint32_t& a2,
                                                  uint32_t& a3) {
  const uint32_t x = __byte_perm(w, 0u, 0x4341);   // bytes 1 and 3 of w into bytes 0 and 2
  a0 = w & 0x000F000Fu;
  a1 = w & 0x00F000F0u;
  a2 = x & 0x000F000Fu;
  a3 = x & 0x00F000F0u;
}

// 2^x by the hardware's base-2 exponential (ex2.approx: relative error about 2^-22;
// results below 2^-126 flush to zero).  e^x is 2^(x log2 e).
constexpr float LOG2E_F = 1.4426950408889634f;
__device__ __forceinline__ float exp2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
// Base-2 exponent e of the prescale 2^e chosen by prescale_for (0 when xmax <= 0).
__device__ __forceinline__ int prescale_exp(float xmax) {
  if (!(xmax > 0.f)) return 0;
  int e;
  frexpf(xmax, &e);
  return max(-100, min(100, 14 - e));
}

// Packed fp32 pairs (two lanes of one 64-bit register pair per instruction).
__device__ __forceinline__ unsigned long long f2_bits(float2 v) {
  return ((unsigned long long)__float_as_uint(v.y) << 32) | __float_as_uint(v.x);
}
__device__ __forceinline__ float2 bits_f2(unsigned long long u) {
  return make_float2(__uint_as_float((uint32_t)u), __uint_as_float((uint32_t)(u >> 32)));
}
__device__ __forceinline__ float2 mul2(float2 a, float2 b) {
  unsigned long long r;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(f2_bits(a)), "l"(f2_bits(b)));
  return bits_f2(r);
}
__device__ __forceinline__ float2 sub2(float2 a, float2 b) {
  unsigned long long r;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(f2_bits(a)), "l"(f2_bits(b)));
  return bits_f2(r);
}
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) {
  unsigned long long r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(f2_bits(a)), "l"(f2_bits(b)), "l"(f2_bits(c)));
  return bits_f2(r);
}
__device__ __forceinline__ float2 add2(float2 a, float2 b) {
  unsigned long long r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(f2_bits(a)), "l"(f2_bits(b)));
  return bits_f2(r);
}

// Programmatic dependent launch: a kernel launched with programmatic stream
// serialisation may start while the previous kernel of the stream drains; pdl_wait()
// returns once that kernel has completed and its writes are visible (at once when the
// launch had no such dependency).  pdl_trigger() lets the next kernel start launching.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Asynchronous 16-byte global -> shared copies (cp.async, L2 only) with an L2 eviction
// hint: tier-1 streams are read once per call, so they are marked evict-first and do not
// push the smaller reused arrays out of L2.
__device__ __forceinline__ unsigned long long evict_first_policy() {
  unsigned long long pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}
__device__ __forceinline__ void cp_async16_hint(void* dst_smem, const void* src, unsigned long long pol) {
  const unsigned d = (unsigned)__cvta_generic_to_shared(dst_smem);
  asm volatile("cp.async.cg.shared.global.L2::cache_hint [%0], [%1], 16, %2;"
               :: "r"(d), "l"(src), "l"(pol) : "memory");
}
__device__ __forceinline__ void cp_async16(void* dst_smem, const void* src) {
  const unsigned d = (unsigned)__cvta_generic_to_shared(dst_smem);
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" :: "r"(d), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" :: "n"(N) : "memory"); }

__device__ __forceinline__ uint32_t word_of(const uint4& v, int i) {
  return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w;
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
// Power-of-two prescale so that |x| * 2^e <= 2^14 for |x| <= xmax (keeps split halves
// normal and far from overflow).  Returns 2^e as a float.
__device__ __forceinline__ float prescale_for(float xmax) {
  return ldexpf(1.f, prescale_exp(xmax));   // xmax = m 2^e, m in [0.5, 1): 2^(14 - e)
}

// ---------------------------------------------------------------------------------
// Fixed-point weights of selection keys (see kvq_blocksel.cuh)
// ---------------------------------------------------------------------------------
__device__ __forceinline__ unsigned long long key_weight(uint32_t key) {
  // floor(v * 2^62) for v = bits `key` in [0, 1], with integer shifts only (no FP64):
  // v = m * 2^(e - 150) with the 24-bit significand m, so v * 2^62 = m * 2^(e - 88).
  const int e = (int)(key >> 23);
  if (e == 0) return 0ull;                     // zero or below 2^-126: weight 0
  const unsigned long long m = (unsigned long long)((key & 0x7fffffu) | 0x800000u);
  const int sh = e - 88;
  if (sh >= 0) return m << sh;                 // e <= 127 keeps this below 2^63
  if (sh <= -24) return 0ull;
  return m >> (-sh);
}

__device__ __forceinline__ unsigned long long warp_sum_u64(unsigned long long v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

constexpr int SEL_CAND = 256;   // candidates ranked exactly by block_select_top

}  // namespace kvq
