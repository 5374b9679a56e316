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
// on the tensor cores, one warp per block:
// tokens are the MMA rows, channels the k dimension and the eight
// MMA columns hold the four query heads twice, as the high and low fp16 halves of the
// exact fp32 product q_c s_{b,c} (scaled by a power of two), so the f16 MMA reproduces
// the fp32 product exactly.  The 512 products of a block are formed once per warp (16 per
// lane) and exchanged through shared memory in B-fragment order.  The INT8 codes convert
// to f16 exactly in registers.
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

__device__ __forceinline__ size_t head_row(const LayerView& V, int b, int g, int r) {
  return (size_t)b * V.Hq + (size_t)g * V.n_rep + r;
}

}  // namespace

// Warp-per-block scoring: every warp owns a contiguous range of the (KV group, block)
// sequence and processes each block alone -- B fragments, 4 MMA row tiles, the block
// log-mass by shuffles -- with no CTA barrier.  Codes and scales reach shared memory by
// cp.async in half blocks (two row tiles) through a two-stage ring per warp: every lane
// copies exactly the 16-byte chunks of its own MMA fragments, so the next half block is
// in flight while the current one is multiplied and no registers hold it.  The stream
// is read once, so the copies carry an L2 evict-first hint.
constexpr int SCORE_CTAS_PER_SM = 4;
constexpr int SCORE_STAGES = 2;
// B words of one block: [head][hi, lo][channel pair], a pair index j stored at
// j + 4 (j / 16) and the lo row 80 words after the hi row, so that the eight lanes of a
// quarter warp read disjoint banks.
constexpr int BW_ROW = 80;
constexpr int BW_HEAD = 2 * BW_ROW;
constexpr int BW_WORDS = MAXREP * BW_HEAD;   // per warp

struct __align__(16) ScoreHalf {   // row tiles 2h, 2h+1 of a block; the scales with h = 0
  uint4 codes[256];
  uint4 scales[16];
};

__global__ void __launch_bounds__(128, SCORE_CTAS_PER_SM) score_kernel(LayerView V) {
  extern __shared__ __align__(16) unsigned char score_dsm[];
  const int warp = threadIdx.x >> 5;
  ScoreHalf* ring = reinterpret_cast<ScoreHalf*>(score_dsm) + warp * SCORE_STAGES;
  uint32_t* bw = reinterpret_cast<uint32_t*>(score_dsm + sizeof(ScoreHalf) * SCORE_STAGES * 4) + warp * BW_WORDS;
  pdl_trigger();
  const int lane = threadIdx.x & 31;
  const int gid = lane >> 2, tig = lane & 3;
  const int hp = lane >> 3, sub = lane & 7;   // product role: head hp, channels 16 sub + [0, 16)
  const unsigned long long pol = evict_first_policy();
  const long long total = (long long)V.BG * V.nb;
  const long long nwarps = (long long)gridDim.x * (blockDim.x >> 5);
  const long long wid = (long long)blockIdx.x * (blockDim.x >> 5) + warp;
  const long long per = (total + nwarps - 1) / nwarps;
  const long long g0 = wid * per;
  const int count = (int)max(0ll, min(total, g0 + per) - g0);
  const int units = 2 * count;   // half blocks

  // producer: copies half block u into ring slot u % SCORE_STAGES (one commit group each)
  int phs = (int)(g0 / V.nb), pblk = (int)(g0 % V.nb);
  auto issue = [&](int u) {
    if (u < units) {
      const int h = u & 1;
      if (h == 0 && pblk == V.nb) { pblk = 0; ++phs; }
      const size_t pbi = (size_t)phs * V.nbmax + pblk;
      ScoreHalf& st = ring[u % SCORE_STAGES];
      if (bounds_ok(V.counters, V.debug, (long long)pbi, (long long)V.BG * V.nbmax, SITE_SCORE)) {
        const uint4* kp = reinterpret_cast<const uint4*>(V.kc + pbi * KC_BYTES) + 256 * h;
#pragma unroll
        for (int j = 0; j < 8; ++j) cp_async16_hint(&st.codes[lane + 32 * j], kp + lane + 32 * j, pol);
        if (h == 0 && lane < 16)
          cp_async16_hint(&st.scales[lane], reinterpret_cast<const uint4*>(V.ks + pbi * D) + lane, pol);
      }
      if (h == 1) ++pblk;
    }
    cp_async_commit();
  };
#pragma unroll
  for (int u = 0; u < SCORE_STAGES - 1; ++u) issue(u);

  int cur_hs = -1;
  float2 qp2[8];                    // q 2^e of head hp at channels 16 sub + [0, 16) (exact)
  float inv_pre = 1.f;              // 2^-e of head hp
  float sc_out = 0.f;               // output scale of head tig
  // the group's queries: max |q| per head, this lane's slice, the power-of-two prescale
  auto setup_q = [&](int hs_q) {
    cur_hs = hs_q;
    const int hrow = hs_q * V.n_rep;
    const float smax = __half2float(__ushort_as_half((unsigned short)V.kscale_max[hs_q]));
    float qm[MAXREP];
#pragma unroll
    for (int r = 0; r < MAXREP; ++r) {
      float m = 0.f;
      if (r < V.n_rep) {
        const __half2 v = *reinterpret_cast<const __half2*>(V.q + (size_t)(hrow + r) * D + 4 * lane);
        const __half2 w = *reinterpret_cast<const __half2*>(V.q + (size_t)(hrow + r) * D + 4 * lane + 2);
        m = fmaxf(fmaxf(fabsf(__low2float(v)), fabsf(__high2float(v))),
                  fmaxf(fabsf(__low2float(w)), fabsf(__high2float(w))));
      }
      qm[r] = warp_max(m);
    }
    float qmr = 0.f, qmt = 0.f;
#pragma unroll
    for (int k = 0; k < MAXREP; ++k) {
      qmr = (k == hp) ? qm[k] : qmr;
      qmt = (k == tig) ? qm[k] : qmt;
    }
    if (hp < V.n_rep) {
      const float pre = prescale_for(qmr * smax);
      const uint4* qp = reinterpret_cast<const uint4*>(V.q + (size_t)(hrow + hp) * D + 16 * sub);
      const uint4 u0 = qp[0], u1 = qp[1];
#pragma unroll
      for (int i = 0; i < 8; ++i)
        qp2[i] = mul2(__half22float2(u32_as_h2(word_of(i < 4 ? u0 : u1, i & 3))), make_float2(pre, pre));
      inv_pre = 1.f / pre;
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i) qp2[i] = make_float2(0.f, 0.f);
      inv_pre = 1.f;
    }
    sc_out = (tig < V.n_rep) ? INV_SQRT_D / prescale_for(qmt * smax) : 0.f;
  };
  if (units > 0) setup_q((int)(g0 / V.nb));   // overlaps the first copy

  int hs = (int)(g0 / V.nb), blk = (int)(g0 % V.nb) - 1;
  bool wok = true;   // the block's result rows are inside the score scratch
  uint32_t bf[16];
  float x[8];
  for (int u = 0; u < units; ++u) {
    issue(u + SCORE_STAGES - 1);
    cp_async_wait<SCORE_STAGES - 1>();   // half block u has landed (this lane's copies)
    __syncwarp();                        // ... and every lane's (the scales are shared)
    const ScoreHalf& cur = ring[u % SCORE_STAGES];
    const int h = u & 1;
    if (h == 0) {
      if (++blk == V.nb) { blk = 0; ++hs; }
      wok = bounds_ok(V.counters, V.debug, (long long)hs * V.nbmax + blk, (long long)V.BG * V.nbmax, SITE_SCORE);
      if (hs != cur_hs) setup_q(hs);
      // products q_c s_c 2^e of head hp at channels 16 sub + [0, 16), split hi + lo
      const uint4 S0 = cur.scales[2 * sub], S1 = cur.scales[2 * sub + 1];
      uint32_t hw[8], lw[8];
      float dp = 0.f;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float2 s2 = __half22float2(u32_as_h2(word_of(i < 4 ? S0 : S1, i & 3)));
        const float2 w = mul2(qp2[i], s2);                            // exact products
        dp += fabsf(w.x) + fabsf(w.y);
        const __half2 hi = __floats2half2_rn(w.x, w.y);
        const float2 rem = sub2(w, __half22float2(hi));               // exact remainders
        hw[i] = h2_as_u32(hi);
        lw[i] = h2_as_u32(__floats2half2_rn(rem.x, rem.y));
      }
      {   // pairs 8 sub + [0, 8) at 8 sub + 4 (sub / 2) + [0, 8)
        uint32_t* ph = bw + hp * BW_HEAD + 8 * sub + 4 * (sub >> 1);
        *reinterpret_cast<uint4*>(ph) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
        *reinterpret_cast<uint4*>(ph + 4) = make_uint4(hw[4], hw[5], hw[6], hw[7]);
        *reinterpret_cast<uint4*>(ph + BW_ROW) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
        *reinterpret_cast<uint4*>(ph + BW_ROW + 4) = make_uint4(lw[4], lw[5], lw[6], lw[7]);
      }
      dp += __shfl_xor_sync(0xffffffffu, dp, 1);   // sum_c |q_c| s_c 2^e of head hp
      dp += __shfl_xor_sync(0xffffffffu, dp, 2);
      dp += __shfl_xor_sync(0xffffffffu, dp, 4);
      if (wok && sub == 0 && hp < V.n_rep)
        V.delta[(size_t)(hs * V.n_rep + hp) * V.nbmax + blk] = KAPPA * INV_SQRT_D * (dp * inv_pre);
      __syncwarp();
      // B fragments of column gid = (head gid>>1, hi or lo): k-step kk takes pairs
      // 16 tig + 2kk (channels 32tig + 4kk + {0,1}) and 16 tig + 2kk + 1 ({2,3})
      const uint4* pb = reinterpret_cast<const uint4*>(bw + (gid >> 1) * BW_HEAD + (gid & 1) * BW_ROW + 20 * tig);
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        const uint4 v = pb[m];
        bf[4 * m] = v.x; bf[4 * m + 1] = v.y; bf[4 * m + 2] = v.z; bf[4 * m + 3] = v.w;
      }
    }
#pragma unroll
    for (int ww = 0; ww < 2; ++ww) {     // MMA row tile 2h + ww: tokens 16(2h + ww) + [0, 16)
      const uint4 R0 = cur.codes[lane + 128 * ww], R1 = cur.codes[lane + 128 * ww + 32];
      const uint4 R2 = cur.codes[lane + 128 * ww + 64], R3 = cur.codes[lane + 128 * ww + 96];
      float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};   // two chains: k-steps 0-3, 4-7
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        const uint4& ra = (kk < 4) ? R0 : R1;
        const uint4& rb = (kk < 4) ? R2 : R3;
        const uint32_t wa = word_of(ra, kk & 3), wb = word_of(rb, kk & 3);
        uint32_t a0, a2, a1, a3;
        i8x4_to_f16(wa, a0, a2);
        i8x4_to_f16(wb, a1, a3);
        mma16816(acc[kk >> 2], a0, a1, a2, a3, bf[2 * kk], bf[2 * kk + 1]);
      }
      // head tig, tokens 16w + gid and 16w + gid + 8 (w = 2h + ww)
      const float2 c0 = add2(make_float2(acc[0][0], acc[0][2]), make_float2(acc[0][1], acc[0][3]));
      const float2 c1 = add2(make_float2(acc[1][0], acc[1][2]), make_float2(acc[1][1], acc[1][3]));
      const float2 xs = mul2(add2(c0, c1), make_float2(sc_out, sc_out));
      if (h == 0) { x[2 * ww] = xs.x; x[2 * ww + 1] = xs.y; }
      else { x[4 + 2 * ww] = xs.x; x[5 + 2 * ww] = xs.y; }
    }
    __syncwarp();   // every lane is done with this slot before it is refilled
    if (h == 1) {
      const int hrow = hs * V.n_rep;   // query-head row of slot 0 (b Hq + g n_rep)
      if (wok && tig < V.n_rep) {
        float* sh = V.shat + (size_t)(hrow + tig) * ((size_t)V.nbmax * BLK) + (size_t)blk * BLK + gid;
#pragma unroll
        for (int w = 0; w < 4; ++w) {
          sh[16 * w] = x[2 * w];
          sh[16 * w + 8] = x[2 * w + 1];
        }
      }
      // block log-mass of head tig over its 64 tokens (8 per lane, 8 lanes per head)
      float m = x[0];
#pragma unroll
      for (int i = 1; i < 8; ++i) m = fmaxf(m, x[i]);
      m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 4));
      m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 8));
      m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 16));
      float l = 0.f;
#pragma unroll
      for (int i = 0; i < 8; ++i) l += __expf(x[i] - m);   // relative error ~2^-22: inside the selection band
      l += __shfl_xor_sync(0xffffffffu, l, 4);
      l += __shfl_xor_sync(0xffffffffu, l, 8);
      l += __shfl_xor_sync(0xffffffffu, l, 16);
      // lane tig (gid 0) holds lse of head tig
      if (wok && gid == 0 && tig < V.n_rep)
        V.lse8[(size_t)(hrow + tig) * V.nbmax + blk] = m + logf(l);
    }
  }
  cp_async_wait<0>();
}

// One CTA of BS_THREADS threads per (sequence, query head): the top-K* selection.  The last
// head of each KV group to finish forms the group's union of selected blocks.
__global__ void __launch_bounds__(BS_THREADS) select_kernel(LayerView V) {
  pdl_trigger();
  pdl_wait();   // scores of the scoring pass
  uint32_t* keys = sel_keys();                           // [nb padded], after the selection's workspace
  float* xs = reinterpret_cast<float*>(keys);            // same storage: the log-masses first
  __shared__ float wm[BS_WARPS], wsum[BS_WARPS], wtm[BS_WARPS], wtl[BS_WARPS];
  __shared__ int is_last, ucnt;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int bh = blockIdx.x;
  const int b = bh / V.Hq, h = bh % V.Hq, g = h / V.n_rep;
  const int hs = b * V.Hkv + g;
  const int nb = V.nb, nbp = (nb + 15) & ~15;
  const size_t hb = (size_t)bh;
  if (!bounds_ok(V.counters, V.debug, nb, (long long)V.nbmax + 1, SITE_SELECT) ||
      !bounds_ok(V.counters, V.debug, hs, V.BG, SITE_SELECT))
    return;
  // this thread's blocks: [i0, i1), log-masses staged in shared memory (16-byte loads;
  // rows are padded to 16 blocks)
  const int kpt = sel_kpt(nb);
  const int i0 = min(nb, tid * kpt), i1 = min(nb, i0 + kpt);
  const float* lse8 = V.lse8 + hb * V.nbmax;
  float m = -INFINITY;
  for (int i = i0; i < i1; i += 4) {
    const float4 x = reinterpret_cast<const float4*>(lse8)[i >> 2];
    reinterpret_cast<float4*>(xs)[i >> 2] = x;
    const float xv[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
    for (int j = 0; j < 4; ++j)
      if (i + j < i1) m = fmaxf(m, xv[j]);
  }
  // exact scores of the partial FP16 block (covered by definition): one score per thread
  float sc = -INFINITY;
  if (tid < V.n_tail)
    sc = dot_f16_row(V.q + hb * D, V.tail_k + ((size_t)hs * BLK + tid) * D) * INV_SQRT_D;
  float tm = -INFINITY;
  // maxima and sums of exp(x - maximum), of the blocks and of the partial block: each warp
  // sums against its own maximum (order-preserving bits, one reduction), and the warps'
  // sums are moved to the block's maximum in one cross-warp round
  m = ord2f(__reduce_max_sync(0xffffffffu, f2ord(m)));
  float sp = 0.f;
  for (int i = i0; i < i1; ++i) sp += expf(xs[i] - m);
  sp = warp_sum(sp);
  float tl = 0.f;
  if (warp < 2) {   // BLK <= 64 partial-block tokens
    tm = ord2f(__reduce_max_sync(0xffffffffu, f2ord(sc)));
    tl = warp_sum(tid < V.n_tail ? expf(sc - tm) : 0.f);
  }
  if (lane == 0) { wm[warp] = m; wsum[warp] = sp; wtm[warp] = tm; wtl[warp] = tl; }
  __syncthreads();
  {
    const float mv = wm[lane & 15], tv = wtm[lane & 15];
    m = ord2f(__reduce_max_sync(0xffffffffu, f2ord(mv)));
    tm = ord2f(__reduce_max_sync(0xffffffffu, f2ord(tv)));
    sp = xw_sum(mv == m ? wsum[lane & 15] : wsum[lane & 15] * expf(mv - m));
    tl = xw_sum(tv == tm ? wtl[lane & 15] : wtl[lane & 15] * expf(tv - tm));
  }
  const float tail_lse = V.n_tail > 0 ? tm + logf(tl) : -INFINITY;
  // softmax reference of the passes that follow: >= every INT8 score (a block's log-mass
  // bounds its scores) and every partial-block score; a pass that meets a larger FP16
  // score raises its own reference
  const float mref = fmaxf(m, tm);
  // log-sum-exp over the blocks (sum sp relative to m) and the partial block
  const float mm = fmaxf(m, tail_lse);
  float s = (nb > 0 ? sp * expf(m - mm) : 0.f) + (V.n_tail > 0 ? expf(tail_lse - mm) : 0.f);
  const float LSE = mm + logf(s);
  // target weight ceil((tau - tail mass) 2^62), in fp32 (FP64 is a narrow unit here)
  const float tail_mass = (V.n_tail > 0) ? expf(tail_lse - LSE) : 0.f;
  const float need = V.tau - tail_mass;
  unsigned long long target = 0ull;
  if (need > 0.f) target = need >= 1.f ? (1ull << 62) : __float2ull_ru(need * 0x1p62f);
  uint8_t* sel = V.sel + hb * V.nbmax;
  // cleared before the selection's first barrier, marked after it
  for (int i16 = tid; i16 < nbp / 16; i16 += BS_THREADS) reinterpret_cast<uint4*>(sel)[i16] = make_uint4(0, 0, 0, 0);
  for (int i = i0; i < i1; ++i) keys[i] = __float_as_uint(expf(xs[i] - LSE));   // mass
  const SelResult sr = block_select_top(nb, target, sel);
  // the last head of the group to finish forms the union (blocks whose FP16 keys are
  // paged in); every mark of this head precedes the selection's closing barrier, and the
  // padding bytes of every sel row are zero
  if (tid == 0) {
    HeadState hsd;
    hsd.M = mref;
    hsd.lse_int8 = LSE;
    hsd.tail_lse = tail_lse;
    hsd.k_star = sr.count;
    hsd.rank_ok = 1;
    hsd.planned = 0;
    hsd.level1 = 0;
    hsd.level = -1;
    hsd.e_key = 0.f;
    hsd.e_val = 0.f;
    hsd.n_vprom = 0;
    hsd.pad = 0;
    V.hst[hb] = hsd;
    ucnt = 0;
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
  cnt = (int)__reduce_add_sync(0xffffffffu, (unsigned)cnt);
  if (lane == 0 && cnt) atomicAdd(&ucnt, cnt);
  __syncthreads();
  if (tid == 0) {
    GroupState gs;
    gs.need_round1 = 0;
    gs.need_dense = 0;
    gs.n_kprom0 = ucnt;
    gs.n_kprom1 = ucnt;
    gs.n_vprom1 = 0;
    gs.pad = 0;
    gs.bytes = (long long)ucnt * F16_BLOCK_BYTES;
    V.gst[hs] = gs;
    V.counters[CNT_GROUP_BASE + hs] = 0u;
  }
}

size_t select_smem_bytes(int nb) {
  return sizeof(BlockSelSmem) + (size_t)((nb + 15) & ~15) * 4;
}

int score_grid(int num_sms) { return num_sms * SCORE_CTAS_PER_SM; }

cudaError_t launch_score(const LayerView& V, int grid, cudaStream_t st) {
  const long long total = (long long)V.BG * V.nb;
  if (total == 0) return cudaSuccess;   // nothing to score (only a partial block)
  if ((long long)grid * 4 > total) grid = (int)((total + 3) / 4);
  const size_t dyn = (sizeof(ScoreHalf) * SCORE_STAGES + BW_WORDS * 4) * 4;   // 4 warps
  cudaError_t e = cudaFuncSetAttribute(score_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)dyn);
  if (e != cudaSuccess) return e;
  score_kernel<<<grid, 128, dyn, st>>>(V);
  return cudaGetLastError();
}

cudaError_t launch_select(const LayerView& V, cudaStream_t st) {
  const size_t dyn = select_smem_bytes(V.nb);
  cudaError_t e = cudaFuncSetAttribute(select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)dyn);
  if (e != cudaSuccess) return e;
  return launch_dependent(select_kernel, dim3(V.B * V.Hq), dim3(BS_THREADS), dyn, st, V);
}

}  // namespace kvq
