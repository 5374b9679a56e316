// kvq_score.cu -- light INT8 scoring pass fused with the adaptive top-K* selection.
//
// "Runtime-Certified Bounded-Error Quantized Attention" (gist.science technical summary),
// Method §3 ("a lightweight scoring pass with INT8 keys estimates per-block attention
// mass; the top-K* blocks covering tau_cov of the estimated mass are promoted to FP16
// keys") and Method §2 (the per-token score perturbation Delta, computed from the
// quantisation scales and the query).
//
// Per 64-token block and KV head the pass computes, for every query head of the group,
//   s_hat_t  = (1/sqrt(D)) sum_c q_c s_{b,c} code_{t,c}            (all 64 tokens)
//   lse8_b   = log sum_t exp(s_hat_t)
//   Delta_b  = kappa (1/sqrt(D)) sum_c |q_c| s_{b,c},   kappa = 1/2 + 2^-8
// on the tensor cores: tokens are the MMA rows, channels the k dimension and the eight
// MMA columns hold the four query heads twice, as the high and low fp16 halves of the
// exact fp32 product q_c s_{b,c} (scaled by a power of two), so the f16 MMA reproduces
// the fp32 product exactly.  The INT8 codes convert to f16 exactly in registers.
//
// A second kernel (one CTA per sequence and query head) selects, per query head,
// the fewest blocks covering tau_cov of exp(lse8_b - LSE) (descending mass, ties to the
// lower block index; the partial FP16 block counts as covered), with fixed-point sums so
// the choice does not depend on summation order; the union over the group is the set of
// blocks whose FP16 keys are paged in.
#include "kvq_common.cuh"
#include "kvq_blocksel.cuh"
#include "kvq_launch.h"

namespace kvq {

namespace {

struct ScoreSmem {
  uint4 bfrag[2][32][4];             // B fragments per lane, double-buffered by block parity
  float dsum[2][4][MAXREP];          // partial sum |q| s  [parity][warp][head]
  float red_m[2][4][MAXREP];         // per-warp block max  [parity][warp][head]
  float red_l[2][4][MAXREP];
  float qmax[MAXREP];
  int item;
};


__device__ __forceinline__ size_t head_row(const LayerView& V, int b, int g, int r) {
  return (size_t)b * V.Hq + (size_t)g * V.n_rep + r;
}

}  // namespace

__global__ void __launch_bounds__(128, 6) score_kernel(LayerView V) {
  __shared__ ScoreSmem sm;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int gid = lane >> 2, tig = lane & 3;
  const int nch = max(1, (V.nb + SCORE_CHUNK - 1) / SCORE_CHUNK);
  const int total = V.BG * nch;

  int cur_hs = -1;
  uint4 qv = make_uint4(0, 0, 0, 0);  // q of head gid>>1, channels 32tig + 8warp + [0, 8)
  float pre = 1.f;                     // prescale of head gid>>1
  float sc_out = 0.f;                  // output scale of head tig
  int par = 0;

  for (;;) {
    if (tid == 0) sm.item = (int)atomicAdd(&V.counters[CNT_SCORE_Q], 1u);
    __syncthreads();
    const int item = sm.item;
    if (item >= total) break;
    const int hs = item / nch, ch = item % nch;
    const int b = hs / V.Hkv, g = hs % V.Hkv;

    if (hs != cur_hs) {
      cur_hs = hs;
      // per-head max |q| (warp = head slot)
      if (warp < V.n_rep) {
        const __half* q = V.q + head_row(V, b, g, warp) * D;
        float m = 0.f;
        for (int c = lane; c < D; c += 32) m = fmaxf(m, fabsf(__half2float(q[c])));
        m = warp_max(m);
        if (lane == 0) sm.qmax[warp] = m;
      } else if (lane == 0) {
        sm.qmax[warp] = 0.f;
      }
      __syncthreads();
      const float smax = __half2float(__ushort_as_half((unsigned short)V.kscale_max[hs]));
      const int r = gid >> 1;
      if (r < V.n_rep) {
        qv = *reinterpret_cast<const uint4*>(V.q + head_row(V, b, g, r) * D + 32 * tig + 8 * warp);
        pre = prescale_for(sm.qmax[r] * smax);
      } else {
        qv = make_uint4(0, 0, 0, 0);
        pre = 1.f;
      }
      sc_out = (tig < V.n_rep) ? INV_SQRT_D / prescale_for(sm.qmax[tig] * smax) : 0.f;
    }

    const int blk_begin = ch * SCORE_CHUNK;
    const int blk_end = min(V.nb, blk_begin + SCORE_CHUNK);
    // software pipeline: the next block's codes and scales are in flight while the
    // current block is multiplied
    uint4 N0, N1, N2, N3, NS;
    if (blk_begin < blk_end) {
      const size_t bi = (size_t)hs * V.nbmax + blk_begin;
      const uint4* kp = reinterpret_cast<const uint4*>(V.kc + bi * KC_BYTES) + (warp * 4) * 32 + lane;
      N0 = __ldcs(kp); N1 = __ldcs(kp + 32); N2 = __ldcs(kp + 64); N3 = __ldcs(kp + 96);
      NS = *reinterpret_cast<const uint4*>(V.ks + bi * D + 32 * tig + 8 * warp);
    }
    for (int blk = blk_begin; blk < blk_end; ++blk, par ^= 1) {
      // A operand: this warp's 16 rows, 4 x 16 bytes per lane, coalesced
      const uint4 R0 = N0, R1 = N1, R2 = N2, R3 = N3, sv = NS;
      if (blk + 1 < blk_end) {
        const size_t bn = (size_t)hs * V.nbmax + blk + 1;
        const uint4* kp = reinterpret_cast<const uint4*>(V.kc + bn * KC_BYTES) + (warp * 4) * 32 + lane;
        N0 = __ldcs(kp); N1 = __ldcs(kp + 32); N2 = __ldcs(kp + 64); N3 = __ldcs(kp + 96);
        NS = *reinterpret_cast<const uint4*>(V.ks + bn * D + 32 * tig + 8 * warp);
      }
      // B operand: hi/lo halves of q_c s_c 2^e for the thread's 8 channels
      {
        const __half* qh = reinterpret_cast<const __half*>(&qv);
        const __half* sh = reinterpret_cast<const __half*>(&sv);
        uint32_t bw[4];
        float dp = 0.f;
#pragma unroll
        for (int i = 0; i < 8; i += 2) {
          const float w0 = __half2float(qh[i]) * __half2float(sh[i]);        // exact
          const float w1 = __half2float(qh[i + 1]) * __half2float(sh[i + 1]);
          dp += fabsf(w0) + fabsf(w1);
          __half h0, l0, h1, l1;
          split_hl(w0 * pre, h0, l0);
          split_hl(w1 * pre, h1, l1);
          const __half2 pk = (gid & 1) ? __halves2half2(l0, l1) : __halves2half2(h0, h1);
          bw[i >> 1] = h2_as_u32(pk);
        }
        sm.bfrag[par][lane][warp ^ ((lane >> 1) & 3)] = make_uint4(bw[0], bw[1], bw[2], bw[3]);
        dp += __shfl_xor_sync(0xffffffffu, dp, 1);
        dp += __shfl_xor_sync(0xffffffffu, dp, 2);
        if (tig == 0 && (gid & 1) == 0) sm.dsum[par][warp][gid >> 1] = dp;
      }
      __syncthreads();
      float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int kq = 0; kq < 4; ++kq) {
        const uint4 bv = sm.bfrag[par][lane][kq ^ ((lane >> 1) & 3)];
        // k-steps 2kq and 2kq+1
#pragma unroll
        for (int s = 0; s < 2; ++s) {
          const int kk = 2 * kq + s;
          const uint4& ra = (kk < 4) ? R0 : R1;
          const uint4& rb = (kk < 4) ? R2 : R3;
          const int wi = kk & 3;
          const uint32_t wa = (wi == 0) ? ra.x : (wi == 1) ? ra.y : (wi == 2) ? ra.z : ra.w;
          const uint32_t wb = (wi == 0) ? rb.x : (wi == 1) ? rb.y : (wi == 2) ? rb.z : rb.w;
          uint32_t a0, a2, a1, a3;
          i8x4_to_f16(wa, a0, a2);
          i8x4_to_f16(wb, a1, a3);
          const uint32_t b0 = s ? bv.z : bv.x;
          const uint32_t b1 = s ? bv.w : bv.y;
          mma16816(acc, a0, a1, a2, a3, b0, b1);
        }
      }
      // epilogue: thread holds head tig, tokens 16warp+gid and 16warp+gid+8
      const float x0 = (acc[0] + acc[1]) * sc_out;
      const float x1 = (acc[2] + acc[3]) * sc_out;
      if (tig < V.n_rep) {
        float* sh = V.shat + head_row(V, b, g, tig) * ((size_t)V.nbmax * BLK) + (size_t)blk * BLK + 16 * warp + gid;
        sh[0] = x0;
        sh[8] = x1;
      }
      float m = fmaxf(x0, x1);
      m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 4));
      m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 8));
      m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 16));
      float l = expf(x0 - m) + expf(x1 - m);
      l += __shfl_xor_sync(0xffffffffu, l, 4);
      l += __shfl_xor_sync(0xffffffffu, l, 8);
      l += __shfl_xor_sync(0xffffffffu, l, 16);
      if (gid == 0) {
        sm.red_m[par][warp][tig] = m;
        sm.red_l[par][warp][tig] = l;
      }
      __syncthreads();
      if (tid < V.n_rep) {
        const int r = tid;
        float M = sm.red_m[par][0][r];
        for (int w = 1; w < 4; ++w) M = fmaxf(M, sm.red_m[par][w][r]);
        float L = 0.f, ds = 0.f;
        for (int w = 0; w < 4; ++w) {
          L += sm.red_l[par][w][r] * expf(sm.red_m[par][w][r] - M);
          ds += sm.dsum[par][w][r];
        }
        const size_t hb = head_row(V, b, g, r);
        V.lse8[hb * V.nbmax + blk] = M + logf(L);
        V.delta[hb * V.nbmax + blk] = KAPPA * INV_SQRT_D * ds;
      }
    }

    __syncthreads();
  }
  if (tid == 0) {
    const unsigned int old = atomicAdd(&V.counters[CNT_SCORE_EXIT], 1u);
    if (old == gridDim.x - 1) {
      V.counters[CNT_SCORE_Q] = 0u;
      V.counters[CNT_SCORE_EXIT] = 0u;
    }
  }
}

// One CTA of 256 threads per (sequence, query head): the top-K* selection.  The last
// head of each KV group to finish forms the group's union of selected blocks.
__global__ void __launch_bounds__(BS_THREADS) select_kernel(LayerView V) {
  extern __shared__ __align__(16) unsigned char sel_dsm[];
  BlockSelSmem& ws = *reinterpret_cast<BlockSelSmem*>(sel_dsm);
  uint32_t* keys = reinterpret_cast<uint32_t*>(sel_dsm + sizeof(BlockSelSmem));   // [nb padded]
  float* xs = reinterpret_cast<float*>(keys);                                         // same storage
  __shared__ float tail_s[BLK];
  __shared__ int is_last;
  const int tid = threadIdx.x;
  const int bh = blockIdx.x;
  const int b = bh / V.Hq, h = bh % V.Hq, g = h / V.n_rep;
  const int hs = b * V.Hkv + g;
  const int nb = V.nb, nbp = (nb + 15) & ~15;
  const size_t hb = (size_t)bh;
  // exact scores of the partial FP16 block (counts as covered)
  float tmax = -INFINITY;
  if (tid < V.n_tail) {
    const __half* q = V.q + hb * D;
    const __half* k = V.tail_k + ((size_t)hs * BLK + tid) * D;
    float sc = 0.f;
    for (int c = 0; c < D; c += 2) {
      const float2 kk = __half22float2(*reinterpret_cast<const __half2*>(k + c));
      const float2 qq = __half22float2(*reinterpret_cast<const __half2*>(q + c));
      sc = fmaf(qq.x, kk.x, sc);
      sc = fmaf(qq.y, kk.y, sc);
    }
    sc *= INV_SQRT_D;
    tail_s[tid] = sc;
    tmax = sc;
  }
  tmax = block_max(tmax, ws.red);
  const float tl = block_sum(tid < V.n_tail ? expf(tail_s[tid] - tmax) : 0.f, ws.red);
  const float tail_lse = V.n_tail > 0 ? tmax + logf(tl) : -INFINITY;
  // block log-masses: staged in shared memory (16-byte loads; rows padded to 16 blocks)
  const float* lse8 = V.lse8 + hb * V.nbmax;
  const float* dl = V.delta + hb * V.nbmax;
  float m = -INFINITY, mref = -INFINITY;
  for (int i4 = tid; i4 < nbp / 4; i4 += BS_THREADS) {
    const float4 x = reinterpret_cast<const float4*>(lse8)[i4];
    const float4 d = reinterpret_cast<const float4*>(dl)[i4];
    const float xv[4] = {x.x, x.y, x.z, x.w}, dv[4] = {d.x, d.y, d.z, d.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      if (4 * i4 + j < nb) {
        m = fmaxf(m, xv[j]);
        mref = fmaxf(mref, xv[j] + dv[j]);
      }
    }
    reinterpret_cast<float4*>(xs)[i4] = x;
  }
  m = block_max(fmaxf(m, tail_lse), ws.red);
  mref = block_max(fmaxf(mref, tmax), ws.red);
  float sp = 0.f;
  for (int i = tid; i < nb; i += BS_THREADS) sp += expf(xs[i] - m);
  float s = block_sum(sp, ws.red);
  if (V.n_tail > 0) s += expf(tail_lse - m);
  const float LSE = m + logf(s);
  const double tail_mass = (V.n_tail > 0) ? (double)expf(tail_lse - LSE) : 0.0;
  const double need = (double)V.tau - tail_mass;
  unsigned long long target = 0ull;
  if (need > 0.0) target = (unsigned long long)ceil(need * 4611686018427387904.0);
  uint8_t* sel = V.sel + hb * V.nbmax;
  for (int i16 = tid; i16 < nbp / 16; i16 += BS_THREADS) reinterpret_cast<uint4*>(sel)[i16] = make_uint4(0, 0, 0, 0);
  for (int i = tid; i < nb; i += BS_THREADS) keys[i] = __float_as_uint(expf(xs[i] - LSE));   // mass
  __syncthreads();
  unsigned long long taken = 0;
  const int kstar = block_select_top(nb, keys, target, [&](int i) { sel[i] = 1; }, ws, &taken);
  if (tid == 0) {
    HeadState hsd;
    hsd.M = mref;
    hsd.lse_int8 = LSE;
    hsd.tail_lse = tail_lse;
    hsd.k_star = kstar;
    hsd.rank_ok = 1;
    hsd.planned = 0;
    hsd.level1 = 0;
    hsd.level = -1;
    hsd.e_key = 0.f;
    hsd.e_val = 0.f;
    hsd.n_vprom = 0;
    hsd.pad = 0;
    V.hst[hb] = hsd;
  }
  // the last head of the group to finish forms the union (blocks whose FP16 keys are
  // paged in); the padding bytes of every sel row are zero
  __syncthreads();
  if (tid == 0) {
    __threadfence();
    const unsigned int old = atomicAdd(&V.counters[CNT_GROUP_BASE + hs], 1u);
    is_last = (old == (unsigned int)(V.n_rep - 1));
  }
  __syncthreads();
  if (!is_last) return;
  __threadfence();
  int cnt = 0;
  for (int i16 = tid; i16 < nbp / 16; i16 += BS_THREADS) {
    uint4 u = make_uint4(0, 0, 0, 0);
    for (int r = 0; r < V.n_rep; ++r) {
      const uint4 x = __ldcg(reinterpret_cast<const uint4*>(V.sel + ((size_t)b * V.Hq + g * V.n_rep + r) * V.nbmax) + i16);
      u.x |= x.x; u.y |= x.y; u.z |= x.z; u.w |= x.w;
    }
    reinterpret_cast<uint4*>(V.kprom0 + (size_t)hs * V.nbmax)[i16] = u;
    reinterpret_cast<uint4*>(V.kprom1 + (size_t)hs * V.nbmax)[i16] = u;
    reinterpret_cast<uint4*>(V.vprom1 + (size_t)hs * V.nbmax)[i16] = make_uint4(0, 0, 0, 0);
    cnt += __popc(u.x) + __popc(u.y) + __popc(u.z) + __popc(u.w);
  }
  cnt = block_sum_int(cnt, ws.red);
  if (tid == 0) {
    GroupState gs;
    gs.need_round1 = 0;
    gs.need_dense = 0;
    gs.n_kprom0 = cnt;
    gs.n_kprom1 = cnt;
    gs.n_vprom1 = 0;
    gs.pad = 0;
    gs.bytes = (long long)cnt * F16_BLOCK_BYTES;
    V.gst[hs] = gs;
    V.counters[CNT_GROUP_BASE + hs] = 0u;
  }
}

size_t select_smem_bytes(int nb) {
  return sizeof(BlockSelSmem) + (size_t)((nb + 15) & ~15) * 4;
}

int score_grid(int num_sms) { return num_sms * 6; }

cudaError_t launch_score(const LayerView& V, int grid, cudaStream_t st) {
  score_kernel<<<grid, 128, 0, st>>>(V);
  return cudaGetLastError();
}

cudaError_t launch_select(const LayerView& V, cudaStream_t st) {
  const size_t dyn = select_smem_bytes(V.nb);
  cudaError_t e = cudaFuncSetAttribute(select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)dyn);
  if (e != cudaSuccess) return e;
  select_kernel<<<V.B * V.Hq, BS_THREADS, dyn, st>>>(V);
  return cudaGetLastError();
}

}  // namespace kvq
