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

// One CTA per (touched block, sequence x KV head); 128 threads, thread = channel.
__global__ void __launch_bounds__(128) append_kernel(AppendArgs a) {
  __shared__ __half sk[BLK][D];
  __shared__ __half sv[BLK][D];
  __shared__ uint32_t kcode[KC_BYTES / 4];
  __shared__ uint32_t vcode[VC_BYTES / 4];
  __shared__ float red[4];
  __shared__ uint32_t smax_k, smax_v;

  const int c = threadIdx.x;
  const int hs = blockIdx.y;
  const int blk = a.first_blk + blockIdx.x;
  const int t0 = blk * BLK;                         // first token of the block
  const int end = a.pos + a.n;                      // tokens after the append
  const int t_hi = min(t0 + BLK, end);
  const bool complete = (t0 + BLK) <= end;

  // gather the block's FP16 tokens: old partial-block tokens, then new ones
  float lo = INFINITY, hi = -INFINITY;
  for (int t = t0; t < t_hi; ++t) {
    __half kv, vv;
    if (t < a.pos) {
      const size_t o = ((size_t)hs * BLK + (t - t0)) * D + c;
      kv = a.tail_k_in[o];
      vv = a.tail_v_in[o];
    } else {
      const size_t o = ((size_t)hs * a.n + (t - a.pos)) * D + c;
      kv = a.k[o];
      vv = a.v[o];
      const float f = __half2float(vv);
      lo = fminf(lo, f);
      hi = fmaxf(hi, f);
    }
    sk[t - t0][c] = kv;
    sv[t - t0][c] = vv;
  }
  if (t_hi > a.pos) {
    atomicMin(&a.vmin[hs * D + c], f2ord(lo));
    atomicMax(&a.vmax[hs * D + c], f2ord(hi));
  }

  if (!complete) {
    // the block stays FP16: write it (old and new tokens) to the outgoing partial buffer
    for (int t = t0; t < t_hi; ++t) {
      const size_t o = ((size_t)hs * BLK + (t - t0)) * D + c;
      a.tail_k_out[o] = sk[t - t0][c];
      a.tail_v_out[o] = sv[t - t0][c];
    }
    return;
  }

  for (int i = c; i < KC_BYTES / 4; i += 128) kcode[i] = 0u;
  for (int i = c; i < VC_BYTES / 4; i += 128) vcode[i] = 0u;
  if (c == 0) { smax_k = 0u; smax_v = 0u; }
  __syncthreads();

  // ---- keys: one fp16 scale per channel, rounded up; symmetric INT8 codes ----
  float amax = 0.f;
  for (int t = 0; t < BLK; ++t) amax = fmaxf(amax, fabsf(__half2float(sk[t][c])));
  const __half s_h = __float2half_ru(__fdiv_rn(amax, 127.f));
  const float s = __half2float(s_h);
  const size_t blk_index = (size_t)hs * a.nbmax + blk;
  a.ks[blk_index * D + c] = s_h;
  atomicMax(&smax_k, (uint32_t)__half_as_ushort(s_h));
  for (int t = 0; t < BLK; ++t) {
    int code = 0;
    if (s > 0.f) {
      const float r = rintf(__fdiv_rn(__half2float(sk[t][c]), s));
      code = (int)fminf(fmaxf(r, -127.f), 127.f);
    }
    const int off = kc_offset(t, c);
    atomicOr(&kcode[off >> 2], ((uint32_t)(code & 0xff)) << (8 * (off & 3)));
  }

  // ---- values: per (token, 32-channel group) offset = min, scale rounded up; INT4 ----
  float errmax = 0.f;
  for (int p = c; p < BLK * NG; p += 128) {
    const int t = p >> 2, g = p & 3;
    float mn = INFINITY, mx = -INFINITY;
    for (int j = 0; j < VG; ++j) {
      const float f = __half2float(sv[t][g * VG + j]);
      mn = fminf(mn, f);
      mx = fmaxf(mx, f);
    }
    const __half vs_h = __float2half_ru(__fdiv_rn(__fsub_rn(mx, mn), 15.f));
    const float vs = __half2float(vs_h);
    const __half vo_h = __float2half_rn(mn);  // exact: mn is an fp16 value
    atomicMax(&smax_v, (uint32_t)__half_as_ushort(vs_h));
    a.vsv[blk_index * VSV_WORDS + g * BLK + t] = __halves2half2(vs_h, vo_h);
    for (int j = 0; j < VG; ++j) {
      const int ch = g * VG + j;
      const float f = __half2float(sv[t][ch]);
      int code = 0;
      if (vs > 0.f) {
        const float r = rintf(__fdiv_rn(__fsub_rn(f, mn), vs));
        code = (int)fminf(fmaxf(r, 0.f), 15.f);
      }
      const float vhat = __fadd_rn(__fmul_rn(vs, (float)code), mn);
      errmax = fmaxf(errmax, fabsf(__fsub_rn(f, vhat)));
      int wb, bit;
      vc_offset(t, ch, wb, bit);
      atomicOr(&vcode[wb >> 2], ((uint32_t)code) << bit);
    }
  }
  errmax = warp_max(errmax);
  if ((c & 31) == 0) red[c >> 5] = errmax;
  __syncthreads();

  // ---- write the block: coalesced 16-byte stores of the fragment-ordered codes ----
  {
    const uint4* src = reinterpret_cast<const uint4*>(kcode);
    uint4* dst = reinterpret_cast<uint4*>(a.kc + blk_index * KC_BYTES);
    for (int i = c; i < KC_BYTES / 16; i += 128) dst[i] = src[i];
    const uint4* srcv = reinterpret_cast<const uint4*>(vcode);
    uint4* dstv = reinterpret_cast<uint4*>(a.vc + blk_index * VC_BYTES);
    for (int i = c; i < VC_BYTES / 16; i += 128) dstv[i] = srcv[i];
  }
  if (c == 0) {
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
    if (a.okc) a.okc[(dst * BLK + t) * D + c] = a.kc[src * KC_BYTES + kc_offset(t, c)];
    if (a.ovc) {
      int wb, bit;
      vc_offset(t, c, wb, bit);
      const uint32_t w = *reinterpret_cast<const uint32_t*>(a.vc + src * VC_BYTES + wb);
      a.ovc[(dst * BLK + t) * D + c] = (uint8_t)((w >> bit) & 0xfu);
    }
  }
  if (a.oks) a.oks[dst * D + c] = a.ks[src * D + c];
  for (int p = c; p < BLK * NG; p += 128) {
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
  const int last_blk = (pos + n - 1) / BLK;
  dim3 grid(last_blk - a.first_blk + 1, L.BG);
  append_kernel<<<grid, 128, 0, st>>>(a);
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
  a.nb = nb; a.nbmax = L.nbmax;
  dim3 grid(nb + 1, L.BG);
  export_tier1_kernel<<<grid, 128, 0, st>>>(a);
  return cudaGetLastError();
}

}  // namespace kvq
