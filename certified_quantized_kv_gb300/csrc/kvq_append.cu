// kvq_append.cu -- quantise-and-append into tier 1, and the tier-1 export for tests.
//
// "Runtime-Certified Bounded-Error Quantized Attention" (gist.science technical summary),
// Method §1 (tier 1: per-channel INT8 keys, per-group INT4 values with scale/offset, a
// per-block error annotation) and Method §2 (value ranges tracked for E_key).
// Readings: key scale per (64-token block, channel) = fp16 rounded up of max|K|/127,
// symmetric codes rint(K/s) clamped to +-127; value group = 32 channels of one token,
// offset = group min, scale = fp16 rounded up of (max-min)/15, codes rint((v-o)/s) in
// [0, 15]; eta_b = max |v - v_hat| over the block.  IEEE fp32 divides (__fdiv_rn) and
// explicit round-to-nearest intrinsics make the codes bit-identical to any IEEE host.
#include "kvq_common.cuh"
#include "kvq_launch.h"

namespace kvq {

struct AppendArgs {
  const __half* k;   // [BG][n][128]
  const __half* v;
  int n, pos;        // new tokens, tokens already cached
  int first_blk;     // pos / 64
  int8_t* kc; __half* ks; uint8_t* vc; __half2* vsv; float* eta;
  uint32_t* vmin; uint32_t* vmax; uint32_t* kscale_max; uint32_t* vscale_max;
  const __half* tail_k_in;  // [BG][64][128] partial block before this append
  const __half* tail_v_in;
  __half* tail_k_out;       // [BG][64][128] partial block after it
  __half* tail_v_out;
  int nbmax;
  __half* v16;              // FP16 values of full blocks (value_bits 16), or nullptr
  unsigned int* counters;   // bounds-check words (KVQ_DEBUG_BOUNDS)
  int debug;
  int BG;
};

__device__ __forceinline__ int kc_offset(int t, int c) {
  const int w = t >> 4, r = t & 15, gid = r & 7, rowhalf = r >> 3;
  const int tig = c >> 5, cc = c & 31, chunkhalf = cc >> 4, byte = cc & 15;
  const int j = rowhalf * 2 + chunkhalf;
  return ((w * 4 + j) * 32 + gid * 4 + tig) * 16 + byte;
}

// byte offset of the 32-bit word and bit position of the nibble for (token, channel)
__device__ __forceinline__ void vc_offset(int t, int c, int& word_byte, int& bit) {
  const int g = c >> 5, cg = c & 31, mt = cg >> 4, r = cg & 15, gid = r & 7, chhalf = r >> 3;
  const int tig = t >> 4, tt = t & 15, kk = tt >> 2, tpos = tt & 3;
  const int reg = (tpos >> 1) * 2 + chhalf;
  bit = 4 * reg + 16 * (tpos & 1);
  word_byte = ((g * 2 + mt) * 32 + gid * 4 + tig) * 16 + kk * 4;
}

constexpr int SROW = D + 8;   // padded shared row (272 bytes): fewer bank conflicts
constexpr int APP_R = 2;      // blocks per CTA (value-range and scale-maximum atomics once per CTA)

// Codes are rint(x / s) for an IEEE fp32 divide followed by rounding to the nearest
// integer, ties to even.  They are computed through the reciprocal r = rn(1 / s):
// q = rn(x r) is within 3 * 2^-24 |x / s| of rn(x / s), so rint(q) is the code unless q
// lies within a margin of a half-integer -- 2^-15 for keys (|x / s| <= 127.5, error below
// 2.3e-5), 2^-17 for values (|x / s| <= 15.5, error below 2.8e-6).  Every 32-bit code
// word whose quotients all clear the margin keeps the fast codes; the others are formed
// again by dividing exactly.  rint(q) itself is q + 1.5 * 2^23 - 1.5 * 2^23 (the sum's
// unit in the last place is 1, so the addition rounds q to an integer, ties to even), and
// the sum's bit pattern is 0x4B400000 + rint(q), which the packing uses directly.
constexpr float RND_C = 12582912.f;            // 1.5 * 2^23
constexpr uint32_t RND_BITS = 0x4B400000u;     // bit pattern of RND_C
constexpr float KEY_TIE_MARGIN = 0.000030517578125f;   // 2^-15
constexpr float VAL_TIE_MARGIN = 0.00000762939453125f; // 2^-17
// packed = sum_e (bits_e << 8e) + KC_INIT = sum_e (code_e + 128) << 8e (mod 2^32)
constexpr uint32_t KC_INIT = (uint32_t)(128u - RND_BITS) + ((uint32_t)(128u - RND_BITS) << 8) +
                             ((uint32_t)(128u - RND_BITS) << 16) + ((uint32_t)(128u - RND_BITS) << 24);
__host__ __device__ constexpr uint32_t vc_shift(int tpos, int chhalf) { return 4 * ((tpos >> 1) * 2 + chhalf) + 16 * (tpos & 1); }
__host__ __device__ constexpr uint32_t vc_init() {
  uint32_t w = 0u;
  for (int tpos = 0; tpos < 4; ++tpos)
    for (int chhalf = 0; chhalf < 2; ++chhalf) w -= RND_BITS << vc_shift(tpos, chhalf);
  return w;
}
constexpr uint32_t VC_INIT = vc_init();   // word = sum (bits << shift) + VC_INIT = sum code << shift

// rint(x / s) by the IEEE divide (the exact path)
__device__ __forceinline__ int rint_div_exact(float x, float s) {
  return s > 0.f ? (int)rintf(__fdiv_rn(x, s)) : 0;
}

// Staged values: 16-byte chunk k of row t sits at chunk k ^ ((t >> 4) & 3), so that the
// value-code pass, whose lanes read four rows 16 apart in one instruction, hits distinct
// banks.  Index of element (t, c) in a row.
__device__ __forceinline__ int svi(int t, int c) { return ((((c >> 3) ^ (t >> 4)) & 3) | ((c >> 3) & ~3)) * 8 + (c & 7); }

// One CTA per run of up to APP_R touched blocks of one (sequence x KV head), 128 threads.
// Each block's FP16 tokens (old partial-block tokens, then new ones) are staged in shared
// memory with 16-byte loads (VEC; element loads when the caller's buffers are not 16-byte
// aligned).  Per-channel maxima and value ranges are taken in exact packed-half
// arithmetic, two channels and half of the rows per thread.  A completed block is
// quantised with each thread producing whole 16-byte chunks of the fragment-ordered key
// and value layouts, written straight to tier 1; the lanes of a warp are assigned so
// that each quarter warp's shared-memory reads fall in distinct banks or broadcast.
// Codes come from the reciprocal, with an exact division where a quotient is near a
// half-integer: bit-identical to dividing every element.
template <bool VEC>
__global__ void __launch_bounds__(128, 5) append_kernel(AppendArgs a) {
  __shared__ __align__(16) __half sk[BLK][SROW];
  __shared__ __align__(16) __half sv[BLK][SROW];   // chunks swizzled (svi)
  __shared__ __align__(16) float kscale[D];
  __shared__ __align__(16) float krcp[D];
  __shared__ __align__(16) float4 vsm[NG][BLK];    // (scale, scale, offset, offset) per (group, token)
  __shared__ __align__(16) float2 vrr[NG][BLK + 4];   // (rn(1 / scale), same) at t + t / 16
  __shared__ __half2 xred[3][D / 2];   // the second row half's partial maxima / minima
  __shared__ float red[4];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int hs = blockIdx.y;
  const int cp = tid & 63, rh = tid >> 6;   // statistics role: channels 2cp, 2cp+1; rows 32rh..+31
  const int cgid = lane & 7, ctig = lane >> 3;   // code role: fragment (gid, tig) of this lane
  const int end = a.pos + a.n;              // tokens after the append
  const int last_blk = (end - 1) / BLK;
  if (!bounds_ok(a.counters, a.debug, hs, a.BG, SITE_APPEND)) return;
  const __half2 hinf = __floats2half2_rn(INFINITY, INFINITY);
  __half2 vlo = hinf, vhi = __hneg2(hinf);   // value range of the new tokens (this role)
  uint32_t smax_k = 0u, smax_v = 0u;         // largest key / value scale bits (thread's own)

  for (int rb = 0; rb < APP_R; ++rb) {
    const int blk = a.first_blk + blockIdx.x * APP_R + rb;
    if (blk > last_blk) break;
    if (!bounds_ok(a.counters, a.debug, blk, a.nbmax, SITE_APPEND)) break;
    const int t0 = blk * BLK;                         // first token of the block
    const int rows = min(t0 + BLK, end) - t0;
    const bool complete = rows == BLK;
    if (rb > 0) __syncthreads();   // the previous block is done with the staging buffers

    // ---- gather the block's FP16 tokens ----
    if (VEC && t0 >= a.pos && rows == BLK) {
      // a whole block of the caller's tokens: one base address per block
      const __half* kp = a.k + ((size_t)hs * a.n + (size_t)(t0 - a.pos)) * D;
      const __half* vp = a.v + ((size_t)hs * a.n + (size_t)(t0 - a.pos)) * D;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int i = tid + 128 * j, row = i >> 4, col = (i & 15) * 8;
        cp_async16(&sk[row][col], kp + (size_t)i * 8);
        cp_async16(&sv[row][svi(row, col)], vp + (size_t)i * 8);
      }
      cp_async_commit();
      cp_async_wait<0>();
    } else if (VEC) {
      // straight into shared memory (cp.async): no registers held while the loads fly
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int i = tid + 128 * j, row = i >> 4, col = (i & 15) * 8;
        const int t = t0 + row;
        if (row < rows) {
          const size_t o = (t < a.pos) ? ((size_t)hs * BLK + row) * D + col
                                       : ((size_t)hs * a.n + (t - a.pos)) * D + col;
          const __half* kp = (t < a.pos) ? a.tail_k_in : a.k;
          const __half* vp = (t < a.pos) ? a.tail_v_in : a.v;
          cp_async16(&sk[row][col], kp + o);
          cp_async16(&sv[row][svi(row, col)], vp + o);
        } else {
          *reinterpret_cast<uint4*>(&sk[row][col]) = make_uint4(0, 0, 0, 0);
          *reinterpret_cast<uint4*>(&sv[row][svi(row, col)]) = make_uint4(0, 0, 0, 0);
        }
      }
      cp_async_commit();
      cp_async_wait<0>();
    } else {
      for (int row = 0; row < rows; ++row) {
        const int t = t0 + row;
        const size_t o = (t < a.pos) ? ((size_t)hs * BLK + row) * D + tid
                                     : ((size_t)hs * a.n + (t - a.pos)) * D + tid;
        sk[row][tid] = (t < a.pos) ? a.tail_k_in[o] : a.k[o];
        sv[row][svi(row, tid)] = (t < a.pos) ? a.tail_v_in[o] : a.v[o];
      }
    }
    __syncthreads();

    // ---- value ranges over the new tokens (exact in binary16) ----
    {
      const int r0 = max(a.pos, t0) - t0;
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {   // rows 32rh + 16hh + [0, 16): one swizzled column
        const int rbase = 32 * rh + 16 * hh;
        const __half* col = &sv[rbase][svi(rbase, 2 * cp)];
        if (r0 <= rbase && rbase + 16 <= rows) {
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const __half2 v2 = *reinterpret_cast<const __half2*>(col + i * SROW);
            vlo = __hmin2(vlo, v2);
            vhi = __hmax2(vhi, v2);
          }
        } else {
          for (int i = max(0, r0 - rbase); i < min(16, rows - rbase); ++i) {
            const __half2 v2 = *reinterpret_cast<const __half2*>(col + i * SROW);
            vlo = __hmin2(vlo, v2);
            vhi = __hmax2(vhi, v2);
          }
        }
      }
    }

    if (!complete) {
      // the block stays FP16 (it is the last one): copy its old and new tokens to the
      // outgoing partial buffer
      for (int i = tid; i < rows * (D / 8); i += 128) {
        const int row = i >> 4, col = (i & 15) * 8;
        const size_t o = ((size_t)hs * BLK + row) * D + col;
        *reinterpret_cast<uint4*>(a.tail_k_out + o) = *reinterpret_cast<const uint4*>(&sk[row][col]);
        *reinterpret_cast<uint4*>(a.tail_v_out + o) = *reinterpret_cast<const uint4*>(&sv[row][svi(row, col)]);
      }
      break;
    }
    const size_t blk_index = (size_t)hs * a.nbmax + blk;

    // ---- key scales: one fp16 per channel, rounded up; their reciprocals ----
    {
      __half2 m2 = __float2half2_rn(0.f);
#pragma unroll 8
      for (int row = 32 * rh; row < 32 * rh + 32; ++row)
        m2 = __hmax2(m2, __habs2(*reinterpret_cast<const __half2*>(&sk[row][2 * cp])));
      xred[rh][cp] = m2;
      __syncthreads();
      // thread = channel: the larger of the two row halves' maxima
      const __half2 p0 = xred[0][tid >> 1], p1 = xred[1][tid >> 1];
      const float amax = (tid & 1) ? fmaxf(__high2float(p0), __high2float(p1)) : fmaxf(__low2float(p0), __low2float(p1));
      const __half s_h = __float2half_ru(__fdiv_rn(amax, 127.f));
      a.ks[blk_index * D + tid] = s_h;
      const float f = __half2float(s_h);
      kscale[tid] = f;
      krcp[tid] = f > 0.f ? __frcp_rn(f) : 0.f;
      smax_k = max(smax_k, (uint32_t)__half_as_ushort(s_h));
    }
    if (a.v16) {
      // FP16-values configuration: the block's values are stored as they are; eta = 0
      __half* dst = a.v16 + blk_index * (BLK * D);
      for (int i = tid; i < BLK * (D / 8); i += 128) {
        const int row = i >> 4, col = (i & 15) * 8;
        *reinterpret_cast<uint4*>(dst + row * D + col) = *reinterpret_cast<const uint4*>(&sv[row][svi(row, col)]);
      }
    } else {
      // ---- value scale/offset per (token, 32-channel group): offset = min, scale rounded up ----
#pragma unroll
      for (int pp = 0; pp < 2; ++pp) {
        const int p = tid + 128 * pp, t = p & 63, g = p >> 6;
        __half2 mn2 = hinf, mx2 = __hneg2(hinf);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const uint4 w = *reinterpret_cast<const uint4*>(&sv[t][svi(t, g * VG + 8 * q)]);
          const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            mn2 = __hmin2(mn2, u32_as_h2(ww[e]));
            mx2 = __hmax2(mx2, u32_as_h2(ww[e]));
          }
        }
        const float mn = fminf(__low2float(mn2), __high2float(mn2));
        const float mx = fmaxf(__low2float(mx2), __high2float(mx2));
        const __half vs_h = __float2half_ru(__fdiv_rn(__fsub_rn(mx, mn), 15.f));
        const __half vo_h = __float2half_rn(mn);  // exact: mn is an fp16 value
        a.vsv[blk_index * VSV_WORDS + g * BLK + t] = __halves2half2(vs_h, vo_h);
        const float vs = __half2float(vs_h);
        vsm[g][t] = make_float4(vs, vs, mn, mn);
        const float vr = vs > 0.f ? __frcp_rn(vs) : 0.f;
        vrr[g][t + (t >> 4)] = make_float2(vr, vr);
        smax_v = max(smax_v, (uint32_t)__half_as_ushort(vs_h));
      }
    }
    __syncthreads();

    // ---- key codes: 512 chunks of 16 codes (one token, 16 channels) in fragment order ----
    // chunk ((w * 4 + jj) * 32 + gid * 4 + tig): w = j, jj = warp; a quarter warp shares tig
    {
      const float2 C2 = make_float2(RND_C, RND_C);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int q = (j * 4 + warp) * 32 + cgid * 4 + ctig;
        const int t = j * 16 + (warp >> 1) * 8 + cgid;
        const int c0 = ctig * 32 + (warp & 1) * 16;
        uint32_t word[4];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const uint4 kh = *reinterpret_cast<const uint4*>(&sk[t][c0 + 8 * h]);
          const uint32_t kw[4] = {kh.x, kh.y, kh.z, kh.w};
#pragma unroll
          for (int uu = 0; uu < 2; ++uu) {
            const int u = 2 * h + uu, cc = c0 + 4 * u;
            const float4 rc = *reinterpret_cast<const float4*>(&krcp[cc]);
            // |code| <= 127 without clamping: s >= rn(amax / 127) makes |K / s| < 127.5
            uint32_t packed = KC_INIT;
            float dmax = 0.f;
#pragma unroll
            for (int pr = 0; pr < 2; ++pr) {
              const float2 x = __half22float2(u32_as_h2(kw[2 * uu + pr]));
              const float2 qq = mul2(x, pr ? make_float2(rc.z, rc.w) : make_float2(rc.x, rc.y));
              const float2 tt = add2(qq, C2);
              const float2 d = sub2(qq, sub2(tt, C2));
              dmax = fmaxf(dmax, fmaxf(fabsf(d.x), fabsf(d.y)));
              packed += __float_as_uint(tt.x) << (16 * pr);
              packed += __float_as_uint(tt.y) << (16 * pr + 8);
            }
            if (dmax > 0.5f - KEY_TIE_MARGIN) {   // a quotient near a half-integer: divide
              packed = 0u;
#pragma unroll 1
              for (int e = 0; e < 4; ++e) {
                const uint32_t kwe = (e >> 1) ? kw[2 * uu + 1] : kw[2 * uu];
                const float xe = __half2float(__ushort_as_half((unsigned short)(kwe >> (16 * (e & 1)))));
                packed |= (uint32_t)(rint_div_exact(xe, kscale[cc + e]) + 128) << (8 * e);
              }
            }
            word[u] = packed;
          }
        }
        reinterpret_cast<uint4*>(a.kc + blk_index * KC_BYTES)[q] = make_uint4(word[0], word[1], word[2], word[3]);
      }
    }

    // ---- value codes: 256 chunks of 4 words of 8 nibbles (4 tokens x 2 channels) ----
    // chunk ((g * 2 + mt) * 32 + gid * 4 + tig), word kk: g = warp; a quarter warp shares tig
    float errmax = 0.f;
    if (!a.v16) {
      const int g = warp;
      const float2 C2 = make_float2(RND_C, RND_C);
#pragma unroll 1
      for (int mt = 0; mt < 2; ++mt) {
        const int cb = g * VG + mt * 16 + cgid;
        // this lane's tokens are 16 ctig + [0, 16): one swizzle for all of them
        const __half* colA = &sv[ctig * 16][svi(ctig * 16, cb)];
        const __half* colB = &sv[ctig * 16][svi(ctig * 16, cb + 8)];
        const float4* inf = &vsm[g][ctig * 16];
        const float2* rcp = &vrr[g][ctig * 17];   // padded: the two 16-token groups of a half warp use distinct banks
        uint32_t word[4];
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          uint32_t wv = VC_INIT;
          float dmax = 0.f, werr = 0.f;   // the word's largest |q - rint(q)| and |v - v_hat|
#pragma unroll
          for (int tpos = 0; tpos < 4; ++tpos) {
            const int i = kk * 4 + tpos;
            const float4 so = inf[i];     // (scale, scale, offset, offset)
            const float2 r2 = rcp[i];
            const float2 f = make_float2(__half2float(colA[i * SROW]), __half2float(colB[i * SROW]));
            // 0 <= (v - o) / s < 15.5 (s rounded up from (max - min) / 15): no clamping
            const float2 qq = mul2(sub2(f, make_float2(so.z, so.w)), r2);
            const float2 tt = add2(qq, C2);
            const float2 k = sub2(tt, C2);
            const float2 d = sub2(qq, k);
            dmax = fmaxf(dmax, fmaxf(fabsf(d.x), fabsf(d.y)));
            const float2 vhat = add2(mul2(make_float2(so.x, so.y), k), make_float2(so.z, so.w));
            const float2 err = sub2(f, vhat);
            werr = fmaxf(werr, fmaxf(fabsf(err.x), fabsf(err.y)));
            wv += __float_as_uint(tt.x) << vc_shift(tpos, 0);
            wv += __float_as_uint(tt.y) << vc_shift(tpos, 1);
          }
          if (dmax > 0.5f - VAL_TIE_MARGIN) {   // a quotient near a half-integer: divide
            wv = 0u;
            werr = 0.f;
#pragma unroll 1
            for (int e = 0; e < 8; ++e) {
              const int i = kk * 4 + (e >> 1);
              const float4 so = inf[i];
              const float fv = __half2float((e & 1) ? colB[i * SROW] : colA[i * SROW]);
              const int code = rint_div_exact(__fsub_rn(fv, so.z), so.x);
              const float vhat = __fadd_rn(__fmul_rn(so.x, (float)code), so.z);
              werr = fmaxf(werr, fabsf(__fsub_rn(fv, vhat)));
              wv |= (uint32_t)code << vc_shift(e >> 1, e & 1);
            }
          }
          errmax = fmaxf(errmax, werr);
          word[kk] = wv;
        }
        reinterpret_cast<uint4*>(a.vc + blk_index * VC_BYTES)[(g * 2 + mt) * 32 + cgid * 4 + ctig] =
            make_uint4(word[0], word[1], word[2], word[3]);
      }
    }
    errmax = warp_max(errmax);
    if (lane == 0) red[warp] = errmax;
    __syncthreads();
    if (tid == 0) a.eta[blk_index] = fmaxf(fmaxf(red[0], red[1]), fmaxf(red[2], red[3]));
  }

  // ---- value ranges and scale maxima of the CTA's blocks: one atomic per channel ----
  __syncthreads();
  if (rh == 1) {
    xred[1][cp] = vlo;
    xred[2][cp] = vhi;
  }
  __syncthreads();
  if (rh == 0) {
    vlo = __hmin2(vlo, xred[1][cp]);
    vhi = __hmax2(vhi, xred[2][cp]);
    const float2 l2 = __half22float2(vlo), h2 = __half22float2(vhi);
    if (l2.x <= h2.x) {   // the channel pair saw new tokens
      atomicMin(&a.vmin[hs * D + 2 * cp], f2ord(l2.x));
      atomicMin(&a.vmin[hs * D + 2 * cp + 1], f2ord(l2.y));
      atomicMax(&a.vmax[hs * D + 2 * cp], f2ord(h2.x));
      atomicMax(&a.vmax[hs * D + 2 * cp + 1], f2ord(h2.y));
    }
  }
  smax_k = __reduce_max_sync(0xffffffffu, smax_k);
  smax_v = __reduce_max_sync(0xffffffffu, smax_v);
  if (lane == 0) {
    if (smax_k) atomicMax(&a.kscale_max[hs], smax_k);
    if (smax_v) atomicMax(&a.vscale_max[hs], smax_v);
  }
}

// Canonical-layout copy of one block of tier 1 (tests and diagnostics).
struct ExportArgs {
  const int8_t* kc; const __half* ks; const uint8_t* vc; const __half2* vsv; const float* eta;
  const uint32_t* vmin; const uint32_t* vmax;
  int8_t* okc; __half* oks; uint8_t* ovc; __half* ovs; __half* ovo; float* oeta;
  float* ovmin; float* ovmax;
  int nb, nbmax;
};

__global__ void __launch_bounds__(128) export_tier1_kernel(ExportArgs a) {
  const int c = threadIdx.x;
  const int hs = blockIdx.y;
  const int blk = blockIdx.x;
  if (blk >= a.nb) {  // one extra column of CTAs copies the value ranges
    if (blk == a.nb) {
      if (a.ovmin) a.ovmin[hs * D + c] = ord2f(a.vmin[hs * D + c]);
      if (a.ovmax) a.ovmax[hs * D + c] = ord2f(a.vmax[hs * D + c]);
    }
    return;
  }
  const size_t src = (size_t)hs * a.nbmax + blk;
  const size_t dst = (size_t)hs * a.nb + blk;
  for (int t = 0; t < BLK; ++t) {
    if (a.okc)   // stored offset binary (code + 128)
      a.okc[(dst * BLK + t) * D + c] = (int8_t)((int)(uint8_t)a.kc[src * KC_BYTES + kc_offset(t, c)] - 128);
    if (a.ovc) {
      int wb, bit;
      vc_offset(t, c, wb, bit);
      const uint32_t w = *reinterpret_cast<const uint32_t*>(a.vc + src * VC_BYTES + wb);
      a.ovc[(dst * BLK + t) * D + c] = (uint8_t)((w >> bit) & 0xfu);
    }
  }
  if (a.oks) a.oks[dst * D + c] = a.ks[src * D + c];
  for (int p = c; p < BLK * NG && (a.ovs || a.ovo); p += 128) {
    const int t = p >> 2, g = p & 3;
    const __half2 so = a.vsv[src * VSV_WORDS + g * BLK + t];
    if (a.ovs) a.ovs[(dst * BLK + t) * NG + g] = __low2half(so);
    if (a.ovo) a.ovo[(dst * BLK + t) * NG + g] = __high2half(so);
  }
  if (c == 0 && a.oeta) a.oeta[dst] = a.eta[src];
}

cudaError_t launch_append(const LayerAppend& L, const void* k, const void* v, int n, int pos,
                          cudaStream_t st) {
  if (n <= 0) return cudaSuccess;
  AppendArgs a;
  a.k = static_cast<const __half*>(k);
  a.v = static_cast<const __half*>(v);
  a.n = n;
  a.pos = pos;
  a.first_blk = pos / BLK;
  a.kc = L.kc; a.ks = L.ks; a.vc = L.vc; a.vsv = L.vsv; a.eta = L.eta;
  a.vmin = L.vmin; a.vmax = L.vmax; a.kscale_max = L.kscale_max; a.vscale_max = L.vscale_max;
  a.tail_k_in = L.tail_k_in; a.tail_v_in = L.tail_v_in;
  a.tail_k_out = L.tail_k_out; a.tail_v_out = L.tail_v_out; a.nbmax = L.nbmax;
  a.v16 = L.v16;
  a.counters = L.counters; a.debug = L.debug; a.BG = L.BG;
  const int last_blk = (pos + n - 1) / BLK;
  dim3 grid((last_blk - a.first_blk + APP_R) / APP_R, L.BG);
  const bool aligned = ((reinterpret_cast<uintptr_t>(k) | reinterpret_cast<uintptr_t>(v)) & 15u) == 0;
  if (aligned) append_kernel<true><<<grid, 128, 0, st>>>(a);
  else append_kernel<false><<<grid, 128, 0, st>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_export_tier1(const LayerAppend& L, int nb, void* kc, void* ks, void* vc,
                                void* vs, void* vo, float* eta, float* vmin, float* vmax,
                                cudaStream_t st) {
  ExportArgs a;
  a.kc = L.kc; a.ks = L.ks; a.vc = L.vc; a.vsv = L.vsv; a.eta = L.eta;
  a.vmin = L.vmin; a.vmax = L.vmax;
  a.okc = static_cast<int8_t*>(kc); a.oks = static_cast<__half*>(ks);
  a.ovc = static_cast<uint8_t*>(vc); a.ovs = static_cast<__half*>(vs);
  a.ovo = static_cast<__half*>(vo); a.oeta = eta; a.ovmin = vmin; a.ovmax = vmax;
  if (L.v16) { a.ovc = nullptr; a.ovs = nullptr; a.ovo = nullptr; }   // no INT4 values exist
  a.nb = nb; a.nbmax = L.nbmax;
  dim3 grid(nb + 1, L.BG);
  export_tier1_kernel<<<grid, 128, 0, st>>>(a);
  return cudaGetLastError();
}

}  // namespace kvq
