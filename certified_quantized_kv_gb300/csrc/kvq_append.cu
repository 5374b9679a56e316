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

// One CTA per (touched block, sequence x KV head), 128 threads.  The block's FP16 tokens
// (old partial-block tokens, then new ones) are staged in shared memory with 16-byte
// loads (VEC; element loads when the caller's buffers are not 16-byte aligned).  A
// completed block is quantised with each thread producing whole 16-byte key chunks and
// whole 32-bit value words of the fragment-ordered layouts, written straight to tier 1.
template <bool VEC>
__global__ void __launch_bounds__(128) append_kernel(AppendArgs a) {
  __shared__ __align__(16) __half sk[BLK][SROW];
  __shared__ __align__(16) __half sv[BLK][SROW];
  __shared__ __align__(16) float kscale[D];
  __shared__ float vsc[BLK][NG], voff[BLK][NG];
  __shared__ float red[4];
  __shared__ uint32_t smax_k, smax_v;

  const int tid = threadIdx.x;
  const int hs = blockIdx.y;
  const int blk = a.first_blk + blockIdx.x;
  if (!bounds_ok(a.counters, a.debug, blk, a.nbmax, SITE_APPEND) ||
      !bounds_ok(a.counters, a.debug, hs, a.BG, SITE_APPEND))
    return;
  const int t0 = blk * BLK;                         // first token of the block
  const int end = a.pos + a.n;                      // tokens after the append
  const int t_hi = min(t0 + BLK, end);
  const int rows = t_hi - t0;
  const bool complete = rows == BLK;

  // ---- gather the block's FP16 tokens ----
  if (VEC) {
    uint4 kr[8], vr[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int i = tid + 128 * j, row = i >> 4, col = (i & 15) * 8;
      const int t = t0 + row;
      kr[j] = make_uint4(0, 0, 0, 0);
      vr[j] = kr[j];
      if (row < rows) {
        const size_t o = (t < a.pos) ? ((size_t)hs * BLK + row) * D + col
                                     : ((size_t)hs * a.n + (t - a.pos)) * D + col;
        const __half* kp = (t < a.pos) ? a.tail_k_in : a.k;
        const __half* vp = (t < a.pos) ? a.tail_v_in : a.v;
        kr[j] = *reinterpret_cast<const uint4*>(kp + o);
        vr[j] = *reinterpret_cast<const uint4*>(vp + o);
      }
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int i = tid + 128 * j, row = i >> 4, col = (i & 15) * 8;
      *reinterpret_cast<uint4*>(&sk[row][col]) = kr[j];
      *reinterpret_cast<uint4*>(&sv[row][col]) = vr[j];
    }
  } else {
    for (int row = 0; row < rows; ++row) {
      const int t = t0 + row;
      const size_t o = (t < a.pos) ? ((size_t)hs * BLK + row) * D + tid
                                   : ((size_t)hs * a.n + (t - a.pos)) * D + tid;
      sk[row][tid] = (t < a.pos) ? a.tail_k_in[o] : a.k[o];
      sv[row][tid] = (t < a.pos) ? a.tail_v_in[o] : a.v[o];
    }
  }
  __syncthreads();

  // ---- value ranges over the new tokens (thread = channel) ----
  {
    const int r0 = max(a.pos, t0) - t0;
    if (r0 < rows) {
      float lo = INFINITY, hi = -INFINITY;
      for (int row = r0; row < rows; ++row) {
        const float f = __half2float(sv[row][tid]);
        lo = fminf(lo, f);
        hi = fmaxf(hi, f);
      }
      atomicMin(&a.vmin[hs * D + tid], f2ord(lo));
      atomicMax(&a.vmax[hs * D + tid], f2ord(hi));
    }
  }

  if (!complete) {
    // the block stays FP16: copy it (old and new tokens) to the outgoing partial buffer
    for (int i = tid; i < rows * (D / 8); i += 128) {
      const int row = i >> 4, col = (i & 15) * 8;
      const size_t o = ((size_t)hs * BLK + row) * D + col;
      *reinterpret_cast<uint4*>(a.tail_k_out + o) = *reinterpret_cast<const uint4*>(&sk[row][col]);
      *reinterpret_cast<uint4*>(a.tail_v_out + o) = *reinterpret_cast<const uint4*>(&sv[row][col]);
    }
    return;
  }
  if (tid == 0) { smax_k = 0u; smax_v = 0u; }
  const size_t blk_index = (size_t)hs * a.nbmax + blk;

  // ---- key scales: one fp16 per channel, rounded up (thread = channel) ----
  {
    float amax = 0.f;
    for (int t = 0; t < BLK; ++t) amax = fmaxf(amax, fabsf(__half2float(sk[t][tid])));
    const __half s_h = __float2half_ru(__fdiv_rn(amax, 127.f));
    a.ks[blk_index * D + tid] = s_h;
    kscale[tid] = __half2float(s_h);
    __syncthreads();   // smax_k initialised, kscale complete
    atomicMax(&smax_k, (uint32_t)__half_as_ushort(s_h));
  }
  if (a.v16) {
    // FP16-values configuration: the block's values are stored as they are; eta = 0
    __half* dst = a.v16 + blk_index * (BLK * D);
    for (int i = tid; i < BLK * (D / 8); i += 128) {
      const int row = i >> 4, col = (i & 15) * 8;
      *reinterpret_cast<uint4*>(dst + row * D + col) = *reinterpret_cast<const uint4*>(&sv[row][col]);
    }
  }
  // ---- value scale/offset per (token, 32-channel group): offset = min, scale rounded up ----
  for (int p = tid; p < BLK * NG && !a.v16; p += 128) {
    const int t = p >> 2, g = p & 3;
    float mn = INFINITY, mx = -INFINITY;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const uint4 w = *reinterpret_cast<const uint4*>(&sv[t][g * VG + 8 * q]);
      const __half2* h2 = reinterpret_cast<const __half2*>(&w);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 f = __half22float2(h2[e]);
        mn = fminf(mn, fminf(f.x, f.y));
        mx = fmaxf(mx, fmaxf(f.x, f.y));
      }
    }
    const __half vs_h = __float2half_ru(__fdiv_rn(__fsub_rn(mx, mn), 15.f));
    const __half vo_h = __float2half_rn(mn);  // exact: mn is an fp16 value
    a.vsv[blk_index * VSV_WORDS + g * BLK + t] = __halves2half2(vs_h, vo_h);
    vsc[t][g] = __half2float(vs_h);
    voff[t][g] = mn;
    atomicMax(&smax_v, (uint32_t)__half_as_ushort(vs_h));
  }
  __syncthreads();

  // ---- key codes: 512 chunks of 16 codes (one token, 16 channels) in fragment order ----
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int q = tid + 128 * j;            // chunk index = ((w * 4 + jj) * 32 + gid * 4 + tig)
    const int tig = q & 3, gid = (q >> 2) & 7, jj = (q >> 5) & 3, w = q >> 7;
    const int t = w * 16 + (jj >> 1) * 8 + gid;
    const int c0 = tig * 32 + (jj & 1) * 16;
    uint32_t word[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const uint2 kh = *reinterpret_cast<const uint2*>(&sk[t][c0 + 4 * u]);
      const float4 sc = *reinterpret_cast<const float4*>(&kscale[c0 + 4 * u]);
      const __half2* h2 = reinterpret_cast<const __half2*>(&kh);
      const float2 f01 = __half22float2(h2[0]), f23 = __half22float2(h2[1]);
      const float fv[4] = {f01.x, f01.y, f23.x, f23.y}, sv4[4] = {sc.x, sc.y, sc.z, sc.w};
      uint32_t packed = 0u;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        int code = 0;
        if (sv4[e] > 0.f) {
          const float r = rintf(__fdiv_rn(fv[e], sv4[e]));
          code = (int)fminf(fmaxf(r, -127.f), 127.f);
        }
        packed |= ((uint32_t)(code + 128)) << (8 * e);   // offset binary: code + 128
      }
      word[u] = packed;
    }
    reinterpret_cast<uint4*>(a.kc + blk_index * KC_BYTES)[q] = make_uint4(word[0], word[1], word[2], word[3]);
  }

  // ---- value codes: 1024 words of 8 nibbles (4 tokens x 2 channels) in fragment order ----
  float errmax = 0.f;
#pragma unroll 2
  for (int j = 0; j < 8 && !a.v16; ++j) {
    const int wi = tid + 128 * j;           // word = ((g * 2 + mt) * 32 + gid * 4 + tig) * 4 + kk
    const int kk = wi & 3, tig = (wi >> 2) & 3, gid = (wi >> 4) & 7, mt = (wi >> 7) & 1, g = wi >> 8;
    const int cb = g * VG + mt * 16 + gid;
    uint32_t word = 0u;
#pragma unroll
    for (int tpos = 0; tpos < 4; ++tpos) {
      const int t = tig * 16 + kk * 4 + tpos;
      const float vs = vsc[t][g], mn = voff[t][g];
#pragma unroll
      for (int chhalf = 0; chhalf < 2; ++chhalf) {
        const float f = __half2float(sv[t][cb + 8 * chhalf]);
        int code = 0;
        if (vs > 0.f) {
          const float r = rintf(__fdiv_rn(__fsub_rn(f, mn), vs));
          code = (int)fminf(fmaxf(r, 0.f), 15.f);
        }
        const float vhat = __fadd_rn(__fmul_rn(vs, (float)code), mn);
        errmax = fmaxf(errmax, fabsf(__fsub_rn(f, vhat)));
        word |= ((uint32_t)code) << (4 * ((tpos >> 1) * 2 + chhalf) + 16 * (tpos & 1));
      }
    }
    reinterpret_cast<uint32_t*>(a.vc + blk_index * VC_BYTES)[wi] = word;
  }
  errmax = warp_max(errmax);
  if ((tid & 31) == 0) red[tid >> 5] = errmax;
  __syncthreads();
  if (tid == 0) {
    a.eta[blk_index] = fmaxf(fmaxf(red[0], red[1]), fmaxf(red[2], red[3]));
    atomicMax(&a.kscale_max[hs], smax_k);
    atomicMax(&a.vscale_max[hs], smax_v);
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
  dim3 grid(last_blk - a.first_blk + 1, L.BG);
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
