// kvq_tail.cu -- the INT4 value pass over blocks that keep their INT8 scores: softmax
// weights from the stored INT8 scores times the INT4 value reconstructions.
//
// "Runtime-Certified Bounded-Error Quantized Attention" (gist.science technical summary),
// Method §1 (INT4 values per 32-channel group with scale and offset) and Method §3 (the
// tail of the context keeps its INT8 scores).  For a block b and query head h:
//   p_t = exp(s_hat_t - M_h),  sum_t p_t v_hat_t = sum_t (p_t s_{t,g}) code_{t,c} + sum_t p_t o_{t,g}
// with g the value group of channel c.  The first sum runs on the tensor cores as in the
// mixed pass (channels as MMA rows, tokens as k, the eight columns = four heads x the hi
// and lo halves of p s 2^e, exact in f16), the second on the CUDA cores.
//
// This pass runs in the uncertified call, where no block is paged in: every full block
// of the layer keeps its INT8 scores and INT4 values.
//
// Work split: one warp per run of consecutive blocks of one KV group (runs per group =
// warps / groups), no CTA barrier; each block's codes, scales/offsets and scores reach
// shared memory by cp.async through a two-stage ring per warp, so the next block is in
// flight while the current one is multiplied.  Each run writes one partial (sum p v_hat,
// sum p and the reference M per head) into its own slot, which the combine kernel adds
// in a fixed order.  The weights carry a prescale 2^e from the start
// (p 2^e = 2^((s - M) log2 e + e)) and are split once per token into binary16 halves
// p_hi + p_lo; each product p s (s a binary16 scale) is then formed as two binary16
// halves in three packed-half instructions per token pair: hi = rn(p_hi s), the exact
// remainder p_hi s - hi by a fused multiply-add, plus p_lo s in a second one (together
// within about 2^-21 of p s).  The INT4 codes enter the MMA as binary16 subnormals (see
// nib8_to_sub_f16x4); both scalings are undone once per run.
#include "kvq_common.cuh"
#include "kvq_launch.h"

namespace kvq {

namespace {

constexpr int TAIL_CTAS_PER_SM = 4;
constexpr int TAIL_STAGES = 2;
// B words of one value group: [head][hi, lo][token pair], rows of 32 pairs padded to 36
// words so that the eight lanes of a quarter warp read disjoint banks.
constexpr int TW_ROW = 36;
constexpr int TW_WORDS = MAXREP * 2 * TW_ROW;   // per warp

// One block's tail data in shared memory: INT4 codes (this lane's chunks at lane + 32 j),
// (scale, offset) per value group and token, and the INT8 scores of the group's heads.
struct __align__(16) TailStage {
  uint4 codes[VC_BYTES / 16];          // 256 chunks
  uint4 so[VSV_WORDS / 4];             // 64 x 4 half2: [group][token]
  float4 s[MAXREP * BLK / 4];          // [head][token]
};

}  // namespace

__global__ void __launch_bounds__(128, TAIL_CTAS_PER_SM) tail_kernel(LayerView V, int runs) {
  extern __shared__ __align__(16) unsigned char tail_dsm[];
  const int warp = threadIdx.x >> 5;
  TailStage* ring = reinterpret_cast<TailStage*>(tail_dsm) + warp * TAIL_STAGES;
  uint32_t* tw = reinterpret_cast<uint32_t*>(tail_dsm + sizeof(TailStage) * TAIL_STAGES * 4) + warp * TW_WORDS;
  pdl_trigger();
  pdl_wait();   // scores of the scoring pass, reference maxima of the selection
  const int lane = threadIdx.x & 31;
  const int gid = lane >> 2, tig = lane & 3;
  const int hp = lane >> 3, sub = lane & 7;   // product role: head hp, tokens 8 sub + [0, 8)
  const int nwarps = gridDim.x * (blockDim.x >> 5);
  const int wid = blockIdx.x * (blockDim.x >> 5) + warp;
  const int NCH = V.nslot;
  const unsigned long long pol = evict_first_policy();

  for (int unit = wid; unit < V.BG * runs; unit += nwarps) {
    const int hs = unit / runs, run = unit % runs;
    const int b0 = (int)((long long)run * V.nb / runs);
    const int b1 = (int)((long long)(run + 1) * V.nb / runs);
    const int hrow = hs * V.n_rep;
    const bool act = hp < V.n_rep;
    if (!bounds_ok(V.counters, V.debug, hs, V.BG, SITE_TAIL) ||
        !bounds_ok(V.counters, V.debug, run, V.nslot, SITE_TAIL) ||
        !bounds_ok(V.counters, V.debug, b1, (long long)V.nbmax + 1, SITE_TAIL))
      continue;
    const float M = act ? V.hst[hrow + hp].M : 0.f;
    // weights p 2^e <= 2^e must be finite binary16 values: e <= 15
    const int pre_e = min(15, prescale_exp(__half2float(__ushort_as_half((unsigned short)V.vscale_max[hs]))));
    const float pre_ef = (float)pre_e;
    int pb = b0;   // producer: next block to copy
    auto issue = [&](int st) {
      if (pb < b1) {
        const size_t bi = (size_t)hs * V.nbmax + pb;
        TailStage& T = ring[st];
        const uint4* vc = reinterpret_cast<const uint4*>(V.vc + bi * VC_BYTES);
#pragma unroll
        for (int j = 0; j < 8; ++j) cp_async16_hint(&T.codes[lane + 32 * j], vc + lane + 32 * j, pol);
        const uint4* so = reinterpret_cast<const uint4*>(V.vsv + bi * VSV_WORDS);
        cp_async16_hint(&T.so[lane], so + lane, pol);
        cp_async16_hint(&T.so[lane + 32], so + lane + 32, pol);
#pragma unroll
        for (int j = 0; j < 2; ++j) {   // 64 float4 of scores: head j * 2 + lane / 16
          const int idx = lane + 32 * j, h = idx >> 4;
          if (h < V.n_rep)
            cp_async16_hint(&T.s[idx], V.shat + (size_t)(hrow + h) * ((size_t)V.nbmax * BLK) + (size_t)pb * BLK + 4 * (idx & 15), pol);
        }
        ++pb;
      }
      cp_async_commit();
    };

    float acc[NG][2][4];
#pragma unroll
    for (int g = 0; g < NG; ++g)
#pragma unroll
      for (int mt = 0; mt < 2; ++mt)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[g][mt][j] = 0.f;
    float2 off[NG];   // sum p o per value group, head hp, tokens of this lane (pairs)
#pragma unroll
    for (int g = 0; g < NG; ++g) off[g] = make_float2(0.f, 0.f);
    float lsum = 0.f;  // sum p, head hp, tokens of this lane

    issue(0);
    int it = 0;
    for (int blk = b0; blk < b1; ++blk, ++it) {
      issue((it + 1) % TAIL_STAGES);
      cp_async_wait<1>();
      __syncwarp();
      const TailStage& T = ring[it % TAIL_STAGES];
      // weights of head hp at tokens 8 sub + [0, 8), times 2^e: fp32 pairs and their
      // binary16 halves (token pair i = tokens 8 sub + 2i, +1)
      float2 pf[4];
      __half2 ph[4], pl[4];
      {
        const float4 sa = T.s[hp * (BLK / 4) + 2 * sub], sb = T.s[hp * (BLK / 4) + 2 * sub + 1];
        const float sv[8] = {sa.x, sa.y, sa.z, sa.w, sb.x, sb.y, sb.z, sb.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float p0 = act ? exp2_approx(fmaf(sv[2 * i] - M, LOG2E_F, pre_ef)) : 0.f;
          const float p1 = act ? exp2_approx(fmaf(sv[2 * i + 1] - M, LOG2E_F, pre_ef)) : 0.f;
          lsum += p0 + p1;
          pf[i] = make_float2(p0, p1);
          ph[i] = __floats2half2_rn(p0, p1);
          const float2 r = sub2(pf[i], __half22float2(ph[i]));   // exact
          pl[i] = __floats2half2_rn(r.x, r.y);
        }
      }
#pragma unroll
      for (int g = 0; g < NG; ++g) {
        // products p_t s_{t,g} 2^e of head hp, tokens 8 sub + [0, 8), as hi + lo halves
        const uint4 S0 = T.so[g * (BLK / 4) + 2 * sub], S1 = T.so[g * (BLK / 4) + 2 * sub + 1];
        uint32_t hw[4], lw[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {   // token pair 4 sub + i: tokens 8 sub + 2i, +1
          const uint4& S = (i < 2) ? S0 : S1;
          const __half2 a = u32_as_h2(word_of(S, 2 * (i & 1)));       // (scale, offset) of token 2i
          const __half2 c = u32_as_h2(word_of(S, 2 * (i & 1) + 1));   // ... of token 2i + 1
          const __half2 s2 = __lows2half2(a, c), o2 = __highs2half2(a, c);
          const __half2 hi = __hmul2_rn(ph[i], s2);
          __half2 lo = __hfma2(ph[i], s2, __hneg2(hi));   // p_hi s - hi, exact
          lo = __hfma2(pl[i], s2, lo);
          hw[i] = h2_as_u32(hi);
          lw[i] = h2_as_u32(lo);
          off[g] = fma2(pf[i], __half22float2(o2), off[g]);
        }
        uint32_t* wr = tw + hp * (2 * TW_ROW) + 4 * sub;
        *reinterpret_cast<uint4*>(wr) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
        *reinterpret_cast<uint4*>(wr + TW_ROW) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
        __syncwarp();
        // B fragments of column gid = (head gid>>1, hi or lo): k-step kk takes token pairs
        // 8 tig + 2kk (tokens 16 tig + 4kk + {0,1}) and 8 tig + 2kk + 1 ({2,3})
        const uint32_t* rd = tw + (gid >> 1) * (2 * TW_ROW) + (gid & 1) * TW_ROW + 8 * tig;
        const uint4 B0 = *reinterpret_cast<const uint4*>(rd), B1 = *reinterpret_cast<const uint4*>(rd + 4);
        const uint32_t bb[8] = {B0.x, B0.y, B0.z, B0.w, B1.x, B1.y, B1.z, B1.w};
#pragma unroll
        for (int mt = 0; mt < 2; ++mt) {
          const uint4 Cw = T.codes[lane + 32 * (2 * g + mt)];
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            uint32_t a0, a1, a2, a3;
            nib8_to_sub_f16x4(word_of(Cw, kk), a0, a1, a2, a3);
            mma16816(acc[g][mt], a0, a1, a2, a3, bb[2 * kk], bb[2 * kk + 1]);
          }
        }
        __syncwarp();   // every lane has read the B words before the next group's
      }
    }
    cp_async_wait<0>();
    __syncwarp();

    // head hp's sums are spread over its eight product lanes
    float offs[NG];
#pragma unroll
    for (int g = 0; g < NG; ++g) {
      offs[g] = off[g].x + off[g].y;
      offs[g] += __shfl_xor_sync(0xffffffffu, offs[g], 1);
      offs[g] += __shfl_xor_sync(0xffffffffu, offs[g], 2);
      offs[g] += __shfl_xor_sync(0xffffffffu, offs[g], 4);
    }
    lsum += __shfl_xor_sync(0xffffffffu, lsum, 1);
    lsum += __shfl_xor_sync(0xffffffffu, lsum, 2);
    lsum += __shfl_xor_sync(0xffffffffu, lsum, 4);
    // this lane writes head tig: its offsets sit in lane 8 tig
    float offh[NG];
#pragma unroll
    for (int g = 0; g < NG; ++g) offh[g] = __shfl_sync(0xffffffffu, offs[g], 8 * tig);
    // undo 2^e (weights) and 2^-24 / 2^-20 (subnormal code rows); powers of two, exact
    const float inv = ldexpf(1.f, -pre_e);
    const float inv_lo = inv * NIB_ROW_SCALE_LO, inv_hi = inv * NIB_ROW_SCALE_HI;
    float* pp = V.part + (((size_t)hs * NCH + run) * MAXREP) * (D + 4);
    if (tig < V.n_rep) {
      float* pr = pp + tig * (D + 4);
#pragma unroll
      for (int g = 0; g < NG; ++g)
#pragma unroll
        for (int mt = 0; mt < 2; ++mt) {
          const int c0 = 32 * g + 16 * mt + gid;
          pr[c0] = (acc[g][mt][0] + acc[g][mt][1]) * inv_lo + offh[g] * inv;
          pr[c0 + 8] = (acc[g][mt][2] + acc[g][mt][3]) * inv_hi + offh[g] * inv;
        }
    }
    if (sub == 0 && act) {
      pp[hp * (D + 4) + D] = lsum * inv;
      pp[hp * (D + 4) + D + 1] = M;
    }
  }
}

int tail_runs(int num_sms, int groups) {
  const int warps = num_sms * TAIL_CTAS_PER_SM * 4;
  return groups >= warps ? 1 : warps / groups;
}

cudaError_t launch_tail(const LayerView& V, int runs, int num_sms, cudaStream_t st) {
  int grid = num_sms * TAIL_CTAS_PER_SM;
  const int units = V.BG * runs;
  if (grid * 4 > units) grid = (units + 3) / 4;
  const size_t dyn = (sizeof(TailStage) * TAIL_STAGES + TW_WORDS * 4) * 4;   // 4 warps
  cudaError_t e = cudaFuncSetAttribute(tail_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)dyn);
  if (e != cudaSuccess) return e;
  return launch_dependent(tail_kernel, dim3(grid), dim3(128), dyn, st, V, runs);
}

}  // namespace kvq
