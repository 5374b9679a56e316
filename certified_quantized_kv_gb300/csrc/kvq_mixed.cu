// kvq_mixed.cu -- fused mixed-precision split-K softmax x V with the runtime certificate.
//
// "Runtime-Certified Bounded-Error Quantized Attention" (gist.science technical summary):
//   Method §1  FP16 originals of promoted blocks come from tier 2 (pinned host memory,
//              read here directly over the host link);
//   Method §2  E_key from the total variation between exact and approximate softmax,
//              bounded through the per-token perturbation Delta; E_val = sum of
//              attention mass times eta_b over blocks with INT4 values;
//   Method §3  promoted blocks use FP16 keys, the tail keeps INT8 scores; the ranking
//              check compares INT8 and FP16 orderings of the selected blocks; rungs 1
//              (more FP16 keys) and 2 (FP16 values) of the fallback ladder.
// Readings (certificate of one query head, p_hat = softmax of the mixed scores):
//   S = sum over INT8 blocks of mass_b (e^Delta_b - 1),  A = sum over INT8 blocks of
//   mass_b e^-Delta_b + mass of FP16-key blocks + mass of the partial block,
//   E_key = S / A * max_c (vmax_c - vmin_c),  E_val = sum over INT4-value blocks of
//   mass_b * eta_b.  Ranking check: the top-R blocks of S_h by INT8 and by FP16 block
//   log-mass agree (ties to the lower index).  Rung 1 adds INT8 blocks in descending
//   mass_b (e^Delta_b - 1) until the projected E_key <= eps/2; rung 2 pages in FP16
//   values in descending mass_b eta_b until the projected E_key + E_val <= eps.
//
// Work split: a persistent grid takes (KV group, run of up to 16 blocks) items from a
// queue; short layers use shorter runs so that every CTA gets several items.  Each warp
// owns one 32-channel value group and multiplies the weights p_t = exp(s'_t - M) of the
// group's query heads into V: INT4 codes on the tensor cores (channels as MMA rows, tokens
// as k, the eight MMA columns = four heads x hi/lo halves of p * scale), FP16 values on the
// CUDA cores.  M >= every score, so no online rescaling is needed.
//   mixed_kernel_r0 (first pass, INT4 values): a block that keeps its INT8 scores is
//     handled by each warp alone, from its own cp.async ring; a block with FP16 keys is
//     read from tier 2 and scored by the whole CTA.
//   mixed_kernel (second pass; first pass with FP16 values in VRAM): the CTA forms each
//     block's weights in shared memory, with a barrier per block.
// combine_kernel (one CTA per sequence and query head) adds the item partials in a fixed
// order and writes the output, the certificate and the ladder plan.
#include "kvq_common.cuh"
#include "kvq_blocksel.cuh"
#include "kvq_launch.h"
#include "kvq_resident.cuh"

namespace kvq {

namespace {

constexpr int KROW = D + 8;   // padded FP16 row (272 bytes): conflict-free 16-byte reads
// B words of one value group: [head][hi, lo][token pair], rows of 32 pairs padded to 36
// words so that the eight lanes of a quarter warp read disjoint banks.
constexpr int MW_ROW = 36;
constexpr int MW_WORDS = MAXREP * 2 * MW_ROW;   // per warp

struct __align__(16) MixSmem {
  float p[2][MAXREP][BLK];    // INT4-path weights
  float pn[2][MAXREP][BLK];   // FP16-value weights / FP16 scores
  float qf[MAXREP][D];
  float fac[MAXREP];          // per head: factor that moved the item's sums to a raised reference
  uint32_t bw[4][MW_WORDS];   // per warp: the INT4-path B words of its value group
  struct {
    __half kbuf[BLK][KROW];
    __half vbuf[BLK][D];
  } st;
  int item;
  int skip;
  int res[4];                 // residency picks: keys [0..1], values [2..3]
};


__device__ __forceinline__ size_t head_row(const LayerView& V, int b, int g, int r) {
  return (size_t)b * V.Hq + (size_t)g * V.n_rep + r;
}

__device__ __forceinline__ unsigned long long fixed62(float x) {
  // x in [0, 1] -> x * 2^62 (rounded toward zero); the shares are formed in fp32, since
  // FP64 is a narrow unit on this part and the inputs are fp32 sums
  if (!(x > 0.f)) return 0ull;
  if (x >= 1.f) return 1ull << 62;
  return __float2ull_rz(x * 0x1p62f);
}

// Copy one FP16 block (64 x 128, 16 KiB) from tier 2 (or its resident copy) into shared
// memory rows of `stride` halves (128 threads), and into `copy` (a free resident slot)
// when given.  A thread issues all eight of its 16-byte loads before the first store, so
// the block costs one host-link round trip instead of eight.
template <int STRIDE>
__device__ __forceinline__ void load_f16_block(__half* dst, const __half* src, __half* copy) {
  const uint4* s = reinterpret_cast<const uint4*>(src);
  uint4 r[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) r[j] = s[threadIdx.x + 128 * j];
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const int i = threadIdx.x + 128 * j, row = i >> 4, col = (i & 15) * 8;
    *reinterpret_cast<uint4*>(dst + row * STRIDE + col) = r[j];
  }
  if (copy) {
#pragma unroll
    for (int j = 0; j < 8; ++j) reinterpret_cast<uint4*>(copy)[threadIdx.x + 128 * j] = r[j];
  }
}

// FP16 scores of one block for the group's heads, s = (q . k) / sqrt(D) in fp32 in channel
// order: thread t (of 128) takes token t % 64 and heads 2 (t / 64) and 2 (t / 64) + 1.
__device__ __forceinline__ void score_f16_block(const __half (*kbuf)[KROW], const float (*qf)[D],
                                                float (*out)[BLK]) {
  const int t = threadIdx.x & 63, rp = (threadIdx.x >> 6) * 2;
  float s0 = 0.f, s1 = 0.f;
#pragma unroll 4
  for (int c = 0; c < D; c += 8) {
    const uint4 kv = *reinterpret_cast<const uint4*>(&kbuf[t][c]);
    const __half2* k2 = reinterpret_cast<const __half2*>(&kv);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float2 kf = __half22float2(k2[j]);
      s0 = fmaf(qf[rp][c + 2 * j], kf.x, s0);
      s0 = fmaf(qf[rp][c + 2 * j + 1], kf.y, s0);
      s1 = fmaf(qf[rp + 1][c + 2 * j], kf.x, s1);
      s1 = fmaf(qf[rp + 1][c + 2 * j + 1], kf.y, s1);
    }
  }
  out[rp][t] = s0 * INV_SQRT_D;
  out[rp + 1][t] = s1 * INV_SQRT_D;
}

}  // namespace

__global__ void __launch_bounds__(128, 4) mixed_kernel(LayerView V, int round) {
  pdl_trigger();
  pdl_wait();   // selection (round 0) or ladder plan (round 1)
  __shared__ MixSmem sm;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int gid = lane >> 2, tig = lane & 3;
  const int nch = max(1, (V.nb + V.chunk - 1) / V.chunk);
  const int NCH = V.nslot;
  const int total = V.BG * nch;
  int par = 0;
  int cur_hs = -1;
  float pre_v = 1.f;
  const bool v16 = V.v16 != nullptr;   // FP16 values in tier 1 (no INT4 codes)
  if (round == 1 && V.counters[CNT_NEED_R1] == 0u) return;   // no head planned rung 1 or 2

  for (;;) {
    if (tid == 0) {
      int it = (int)atomicAdd(&V.counters[CNT_MIX_Q], 1u);
      int skip = 0;
      if (it < total && round == 1) skip = !V.gst[it / nch].need_round1;
      sm.item = it;
      sm.skip = skip;
    }
    __syncthreads();
    const int item = sm.item;
    if (item >= total) break;
    if (sm.skip) { __syncthreads(); continue; }
    const int hs = item / nch, ch = item % nch;
    const int b = hs / V.Hkv, g = hs % V.Hkv;
    {   // the item's group, partial slot, blocks (tier 1, scratch) and tier-2 rows
      const long long be = min(V.nb, (ch + 1) * V.chunk);
      if (!bounds_ok(V.counters, V.debug, hs, V.BG, SITE_MIX) ||
          !bounds_ok(V.counters, V.debug, ch, V.nslot, SITE_MIX) ||
          !bounds_ok(V.counters, V.debug, be, (long long)V.nbmax + 1, SITE_MIX) ||
          !bounds_ok(V.counters, V.debug, be * BLK, V.cap + 1, SITE_MIX)) {
        __syncthreads();
        continue;
      }
    }

    if (hs != cur_hs) {
      cur_hs = hs;
      for (int i = tid; i < MAXREP * D; i += blockDim.x) {
        const int r = i / D, c = i % D;
        sm.qf[r][c] = (r < V.n_rep) ? __half2float(V.q[head_row(V, b, g, r) * D + c]) : 0.f;
      }
      pre_v = prescale_for(__half2float(__ushort_as_half((unsigned short)V.vscale_max[hs])));
      __syncthreads();
    }
    // the item's softmax reference for head `warp`: the head's reference after the
    // selection (round 0) or the first combine (round 1), raised only where an FP16-key
    // block of this item scores above it (its sums so far are then rescaled)
    float Mr = (warp < V.n_rep) ? V.hst[head_row(V, b, g, warp)].M : 0.f;

    float acc[2][4];
#pragma unroll
    for (int i = 0; i < 2; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;
    float acc16[4] = {0.f, 0.f, 0.f, 0.f};
    float off = 0.f;     // sum p * offset for head lane/8 (this lane's tokens), group = warp
    float lsum = 0.f;    // sum p for head = warp

    const int blk_end = min(V.nb, (ch + 1) * V.chunk);
    for (int blk = ch * V.chunk; blk < blk_end; ++blk) {
      const size_t bi = (size_t)hs * V.nbmax + blk;
      const bool kp0 = V.kprom0[bi] != 0;
      bool newk = false, vp = false;
      if (round == 1) {
        newk = !kp0 && V.kprom1[bi] != 0;
        vp = V.vprom1[bi] != 0;
        if (!newk && !vp) continue;   // precision unchanged: contribution unchanged
      }
      // FP16 values: paged in for this block (rung 2), or resident in tier 1
      const bool use16 = vp || v16;
      par ^= 1;
      const int r = warp;
      const bool act = r < V.n_rep;
      float* shat_r = V.shat + head_row(V, b, g, act ? r : 0) * ((size_t)V.nbmax * BLK) + (size_t)blk * BLK;
      const bool need_k16 = (round == 0) ? kp0 : newk;
      // ---- stage 1: probabilities of the block's 64 tokens for the group's heads ----
      // Round 0: p = exp(s' - M), s' = FP16 score on promoted blocks (computed from tier 2
      // and kept in the score scratch for the second pass), INT8 score elsewhere.
      // Round 1: INT4 weights = p_new - p_old (or -p_old where the values are promoted);
      // FP16-value weights = p_new.
      float so0 = 0.f, so1 = 0.f;
      if (act && (round == 1 || !kp0)) {
        so0 = __ldcs(shat_r + lane);
        so1 = __ldcs(shat_r + lane + 32);
      }
      float sn0 = so0, sn1 = so1;
      if (need_k16) {
        const ResPick pk = res_pick(V, 0, bi, sm.res);
        load_f16_block<KROW>(&sm.st.kbuf[0][0],
                             res_src(V, pk, V.t2k + ((size_t)hs * V.cap + (size_t)blk * BLK) * D),
                             res_dst(V, pk));
        res_commit(V, 0, bi, pk);
        __syncthreads();
        score_f16_block(sm.st.kbuf, sm.qf, sm.pn[par]);
        __syncthreads();
        sn0 = sm.pn[par][r][lane];
        sn1 = sm.pn[par][r][lane + 32];
        float fac = 1.f;
        if (act) {
          const float m = warp_max(fmaxf(sn0, sn1));
          const float l = warp_sum(expf(sn0 - m) + expf(sn1 - m));
          if (lane == 0) V.lse16[head_row(V, b, g, r) * V.nbmax + blk] = m + logf(l);
          shat_r[lane] = sn0;
          shat_r[lane + 32] = sn1;
          if (m > Mr) {
            fac = expf(Mr - m);
            Mr = m;
            lsum *= fac;   // head `warp`'s weight sum, before this block's weights join it
          }
        }
        if (lane == 0) sm.fac[r] = fac;
      }
      float pn0 = 0.f, pn1 = 0.f, pi0 = 0.f, pi1 = 0.f;
      if (act) {
        const float M = Mr;
        if (round == 0) {
          pn0 = kp0 ? expf(sn0 - M) : __expf(sn0 - M);
          pn1 = kp0 ? expf(sn1 - M) : __expf(sn1 - M);
          pi0 = pn0;
          pi1 = pn1;
          lsum += pn0 + pn1;
        } else {
          const float po0 = kp0 ? expf(so0 - M) : __expf(so0 - M);   // as the first pass
          const float po1 = kp0 ? expf(so1 - M) : __expf(so1 - M);
          pn0 = newk ? expf(sn0 - M) : po0;
          pn1 = newk ? expf(sn1 - M) : po1;
          pi0 = vp ? -po0 : pn0 - po0;
          pi1 = vp ? -po1 : pn1 - po1;
          lsum += (pn0 - po0) + (pn1 - po1);
          if (v16) {   // resident FP16 values: only the change of weight is added
            pn0 -= po0;
            pn1 -= po1;
          }
        }
      }
      sm.p[par][r][lane] = pi0;
      sm.p[par][r][lane + 32] = pi1;
      sm.pn[par][r][lane] = pn0;
      sm.pn[par][r][lane + 32] = pn1;
      __syncthreads();
      if (need_k16) {   // sums so far to the raised references (factor 1 where unchanged)
        const float ft = sm.fac[tig], fh = sm.fac[lane >> 3];
#pragma unroll
        for (int i = 0; i < 2; ++i)
#pragma unroll
          for (int j = 0; j < 4; ++j) acc[i][j] *= ft;   // accumulator columns: head tig
#pragma unroll
        for (int j = 0; j < 4; ++j) acc16[j] *= ft;     // FP16 values: head tig
        off *= fh;                                       // offsets: head lane / 8
      }
      // ---- stage 2: weights x V for the warp's value group ----
      if (!v16) {
        const uint4* vcp = reinterpret_cast<const uint4*>(V.vc + bi * VC_BYTES) + (warp * 2) * 32 + lane;
        const uint4 C0 = __ldcs(vcp), C1 = __ldcs(vcp + 32);
        // products p_t s_{t,g} 2^e of head hp = lane / 8 at tokens 8 (lane % 8) + [0, 8), as
        // hi + lo halves, formed once per warp and exchanged as B fragments
        {
          const int hp = lane >> 3, sub = lane & 7;
          const uint4* svp = reinterpret_cast<const uint4*>(V.vsv + bi * VSV_WORDS + warp * BLK + 8 * sub);
          const uint4 S0 = __ldcs(svp), S1 = __ldcs(svp + 1);        // (scale, offset), 8 tokens
          const float4 pa = *reinterpret_cast<const float4*>(&sm.p[par][hp][8 * sub]);
          const float4 pb = *reinterpret_cast<const float4*>(&sm.p[par][hp][8 * sub + 4]);
          const float pv[8] = {pa.x, pa.y, pa.z, pa.w, pb.x, pb.y, pb.z, pb.w};
          const uint32_t sw[8] = {S0.x, S0.y, S0.z, S0.w, S1.x, S1.y, S1.z, S1.w};
          uint32_t hw[4], lw[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) {   // token pair 4 sub + i
            const float2 a = __half22float2(u32_as_h2(sw[2 * i])), c = __half22float2(u32_as_h2(sw[2 * i + 1]));
            const float2 p2 = make_float2(pv[2 * i], pv[2 * i + 1]);
            off = fmaf(p2.x, a.y, off);
            off = fmaf(p2.y, c.y, off);
            const float2 w = mul2(mul2(p2, make_float2(a.x, c.x)), make_float2(pre_v, pre_v));
            const __half2 hi = __floats2half2_rn(w.x, w.y);
            const float2 rem = sub2(w, __half22float2(hi));   // exact remainders
            hw[i] = h2_as_u32(hi);
            lw[i] = h2_as_u32(__floats2half2_rn(rem.x, rem.y));
          }
          uint32_t* wr = sm.bw[warp] + hp * (2 * MW_ROW) + 4 * sub;
          *reinterpret_cast<uint4*>(wr) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
          *reinterpret_cast<uint4*>(wr + MW_ROW) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
        }
        __syncwarp();
        // column gid = (head gid>>1, hi or lo): k-step kk takes token pairs 8 tig + 2kk and
        // 8 tig + 2kk + 1 (tokens 16 tig + 4kk + {0,1} and {2,3})
        uint32_t bb0[4], bb1[4];
        {
          const uint32_t* rd = sm.bw[warp] + (gid >> 1) * (2 * MW_ROW) + (gid & 1) * MW_ROW + 8 * tig;
          const uint4 B0 = *reinterpret_cast<const uint4*>(rd), B1 = *reinterpret_cast<const uint4*>(rd + 4);
          bb0[0] = B0.x; bb1[0] = B0.y; bb0[1] = B0.z; bb1[1] = B0.w;
          bb0[2] = B1.x; bb1[2] = B1.y; bb0[3] = B1.z; bb1[3] = B1.w;
        }
#pragma unroll
        for (int mt = 0; mt < 2; ++mt) {
          const uint4 C = mt ? C1 : C0;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint32_t w = (kk == 0) ? C.x : (kk == 1) ? C.y : (kk == 2) ? C.z : C.w;
            uint32_t a0, a1, a2, a3;
            nib8_to_sub_f16x4(w, a0, a1, a2, a3);
            mma16816(acc[mt], a0, a1, a2, a3, bb0[kk], bb1[kk]);
          }
        }
      }
      if (use16) {
        const ResPick pv = v16 ? ResPick{-1, -1} : res_pick(V, 1, bi, sm.res + 2);
        load_f16_block<D>(&sm.st.vbuf[0][0],
                          v16 ? V.v16 + bi * (BLK * D)
                              : res_src(V, pv, V.t2v + ((size_t)hs * V.cap + (size_t)blk * BLK) * D),
                          res_dst(V, pv));
        res_commit(V, 1, bi, pv);
        __syncthreads();
        const int c0 = 32 * warp + gid;
        const float* pr = sm.pn[par][tig];
        for (int t = 0; t < BLK; ++t) {
          const float pt = pr[t];
          acc16[0] = fmaf(pt, __half2float(sm.st.vbuf[t][c0]), acc16[0]);
          acc16[1] = fmaf(pt, __half2float(sm.st.vbuf[t][c0 + 8]), acc16[1]);
          acc16[2] = fmaf(pt, __half2float(sm.st.vbuf[t][c0 + 16]), acc16[2]);
          acc16[3] = fmaf(pt, __half2float(sm.st.vbuf[t][c0 + 24]), acc16[3]);
        }
      }
    }

    // ---- write this chunk's partial: l and acc[D] per head ----
    off += __shfl_xor_sync(0xffffffffu, off, 1);   // head lane/8: its eight product lanes
    off += __shfl_xor_sync(0xffffffffu, off, 2);
    off += __shfl_xor_sync(0xffffffffu, off, 4);
    const float offh = __shfl_sync(0xffffffffu, off, 8 * tig);  // head tig
    // undo 2^e (the products) and 2^-24 / 2^-20 (subnormal code rows); powers of two
    const float inv = 1.f / pre_v;
    const float inv_lo = inv * NIB_ROW_SCALE_LO, inv_hi = inv * NIB_ROW_SCALE_HI;
    float* pp = (round == 0 ? V.part : V.part1) + (((size_t)hs * NCH + ch) * MAXREP) * (D + 4);
    if (tig < V.n_rep) {
      float* pr = pp + tig * (D + 4);
      const int c0 = 32 * warp + gid;
      pr[c0] = (acc[0][0] + acc[0][1]) * inv_lo + acc16[0] + offh;
      pr[c0 + 8] = (acc[0][2] + acc[0][3]) * inv_hi + acc16[1] + offh;
      pr[c0 + 16] = (acc[1][0] + acc[1][1]) * inv_lo + acc16[2] + offh;
      pr[c0 + 24] = (acc[1][2] + acc[1][3]) * inv_hi + acc16[3] + offh;
    }
    lsum = warp_sum(lsum);
    if (lane == 0 && warp < V.n_rep) {
      pp[warp * (D + 4) + D] = lsum;
      pp[warp * (D + 4) + D + 1] = Mr;
    }

    __syncthreads();
  }
  if (tid == 0) {
    const unsigned int old = atomicAdd(&V.counters[CNT_MIX_EXIT], 1u);
    if (old == gridDim.x - 1) {
      V.counters[CNT_MIX_Q] = 0u;
      V.counters[CNT_MIX_EXIT] = 0u;
    }
  }
}

// Per-block values of four consecutive blocks read by the certificate pass.
struct BlockQuad {
  uchar4 kf, vf, sl;        // FP16-key flag, FP16-value flag, selected (ranking check)
  float4 l8, l16, dl, eta;  // log-masses (INT8, FP16 scores), Delta_b, eta_b
};

// One CTA of BS_THREADS threads per (sequence, query head): combine the work-item partials
// of a pass for the head, add the partial block, write the output and the certificate
// and, after the first pass, run the ranking check and plan rungs 1-2.
// One instantiation per pass (`round`): each carries only its own code, which matters for a
// kernel that runs once per head on an otherwise idle SM (cold instruction fetch).
template <int round>
__global__ void __launch_bounds__(BS_THREADS) combine_kernel(LayerView V) {
  pdl_trigger();
  pdl_wait();   // partials of the mixed pass
  uint32_t* keys = sel_keys();   // [nb padded], after the selection's workspace
  __shared__ __align__(16) float acc_s[BS_WARPS][D];
  __shared__ float l_s[BS_WARPS], m_s[BS_WARPS], tl_s[2];
  __shared__ float tail_p[BLK];
  __shared__ int wk[BS_WARPS], wv[BS_WARPS];
  __shared__ float cR[BS_WARPS], cS[BS_WARPS], cA[BS_WARPS], cE[BS_WARPS];
  __shared__ uint32_t c8[BS_WARPS], c16[BS_WARPS];
  __shared__ int ci8[BS_WARPS], ci16[BS_WARPS];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int bh = blockIdx.x;
  const int b = bh / V.Hq, h = bh % V.Hq, g = h / V.n_rep, r = h % V.n_rep;
  const int hs = b * V.Hkv + g;
  const size_t hb = (size_t)bh;
  const int nb = V.nb;
  const int nch = V.nparts > 0 ? V.nparts : max(1, (nb + V.chunk - 1) / V.chunk);
  const int NCH = V.nslot;
  if (!bounds_ok(V.counters, V.debug, hs, V.BG, SITE_COMBINE) ||
      !bounds_ok(V.counters, V.debug, nch, (long long)NCH + 1, SITE_COMBINE) ||
      !bounds_ok(V.counters, V.debug, nb, (long long)V.nbmax + 1, SITE_COMBINE))
    return;
  const uint8_t* kfl = (round == 0 ? V.kprom0 : V.kprom1) + (size_t)hs * V.nbmax;
  // first pass: no FP16 values yet (every head's rung 2 plans against this empty set,
  // while its marks accumulate in vprom1 for the second pass)
  const uint8_t* vfl = round == 0 ? nullptr : V.vprom1 + (size_t)hs * V.nbmax;
  HeadState hsd = V.hst[hb];
  if (round == 1) {
    if (!V.gst[hs].need_round1) return;
    const bool planned12 = hsd.planned == 1 || hsd.planned == 2;
    if (r != 0 && !planned12) return;
    // the group's promoted key and value blocks of the second pass (head r = 0 records them)
    int nk = 0, nv = 0;
    for (int i16 = tid; i16 < (nb + 15) / 16; i16 += BS_THREADS) {
      const uint4 a = reinterpret_cast<const uint4*>(V.kprom1 + (size_t)hs * V.nbmax)[i16];
      const uint4 c = reinterpret_cast<const uint4*>(V.vprom1 + (size_t)hs * V.nbmax)[i16];
      nk += __popc(a.x) + __popc(a.y) + __popc(a.z) + __popc(a.w);
      nv += __popc(c.x) + __popc(c.y) + __popc(c.z) + __popc(c.w);
    }
    nk = (int)__reduce_add_sync(0xffffffffu, (unsigned)nk);
    nv = (int)__reduce_add_sync(0xffffffffu, (unsigned)nv);
    if (lane == 0) { wk[warp] = nk; wv[warp] = nv; }
    if (!planned12) {   // head 0 of the group, not re-run itself: the counts only
      __syncthreads();
      if (tid == 0) {
        nk = 0; nv = 0;
        for (int w = 0; w < BS_WARPS; ++w) { nk += wk[w]; nv += wv[w]; }
        GroupState gs = V.gst[hs];
        gs.n_kprom1 = nk;
        gs.n_vprom1 = nv;
        gs.bytes += (long long)(nk - gs.n_kprom0 + nv) * F16_BLOCK_BYTES;
        V.gst[hs] = gs;
      }
      return;
    }
    // otherwise thread 0 reads the counts after the merge barrier below
  }
  const float M_prev = hsd.M;   // reference of the selection (round 0) or the first pass's sums (round 1)
  // (1) work-item partials of this pass, in a fixed order: warp w takes items w, w + 16, ...
  //     (lane = four channels) in batches of eight, its sums kept relative to the largest
  //     item reference seen so far (rescaled when it rises; a factor of exactly 1 for
  //     every item that kept the head's reference)
  {
    const float* P = (round == 0) ? V.part : V.part1;
    float Mw = -INFINITY, l = 0.f;
    float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int base = warp; base < nch; base += BS_WARPS * 8) {
      float Mi[8], Li[8];
      float4 x[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int ch = base + BS_WARPS * j;
        if (ch < nch) {
          const size_t o = (((size_t)hs * NCH + ch) * MAXREP + r) * (D + 4);
          Mi[j] = P[o + D + 1];
          Li[j] = P[o + D];
          x[j] = *reinterpret_cast<const float4*>(P + o + 4 * lane);
        } else {
          Mi[j] = -INFINITY;
          Li[j] = 0.f;
          x[j] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
      }
      float Mb = Mw;
#pragma unroll
      for (int j = 0; j < 8; ++j) Mb = fmaxf(Mb, Mi[j]);
      if (Mb > Mw) {
        const float f = expf(Mw - Mb);
        a.x *= f; a.y *= f; a.z *= f; a.w *= f;
        l *= f;
        Mw = Mb;
      }
#pragma unroll
      for (int j = 0; j < 8; ++j) {   // a partial at reference -inf still adds its (zero or NaN) sums
        const float w = (Mi[j] == Mw) ? 1.f : expf(Mi[j] - Mw);
        a.x = fmaf(x[j].x, w, a.x); a.y = fmaf(x[j].y, w, a.y);
        a.z = fmaf(x[j].z, w, a.z); a.w = fmaf(x[j].w, w, a.w);
        l = fmaf(Li[j], w, l);
      }
    }
    *reinterpret_cast<float4*>(&acc_s[warp][4 * lane]) = a;
    if (lane == 0) { l_s[warp] = l; m_s[warp] = Mw; }
  }
  // (2) the partial FP16 block with exact scores, weighted against M_prev (which bounds
  //     every partial-block score)
  {
    float lt = 0.f;
    if (tid < V.n_tail) {
      const float sc = dot_f16_row(V.q + hb * D, V.tail_k + ((size_t)hs * BLK + tid) * D);
      lt = expf(sc * INV_SQRT_D - M_prev);
      tail_p[tid] = lt;
    }
    if (warp < 2) {   // BLK <= 64 tail tokens
      lt = warp_sum(lt);
      if (lane == 0) tl_s[warp] = lt;
    }
  }
  // this thread's blocks for the certificate pass, the first four read before the barrier
  const int kpt = sel_kpt(nb);
  const int i0 = min(nb, tid * kpt), i1 = min(nb, i0 + kpt);
  const bool rank0 = round == 0 && hsd.k_star > 1;   // first ranking position in the pass
  const uint8_t* sel = V.sel + hb * V.nbmax;
  const float* lse8 = V.lse8 + hb * V.nbmax;
  const float* lse16 = V.lse16 + hb * V.nbmax;
  const float* dl = V.delta + hb * V.nbmax;
  const float* eta = V.eta + (size_t)hs * V.nbmax;
  auto load_quad = [&](int i) {
    BlockQuad q;
    const int i4 = i >> 2;   // rows are padded to 16 blocks, 16-byte aligned
    q.kf = reinterpret_cast<const uchar4*>(kfl)[i4];
    q.vf = vfl ? reinterpret_cast<const uchar4*>(vfl)[i4] : make_uchar4(0, 0, 0, 0);
    q.sl = rank0 ? reinterpret_cast<const uchar4*>(sel)[i4] : make_uchar4(0, 0, 0, 0);
    q.l8 = reinterpret_cast<const float4*>(lse8)[i4];
    q.l16 = reinterpret_cast<const float4*>(lse16)[i4];
    q.dl = reinterpret_cast<const float4*>(dl)[i4];
    q.eta = reinterpret_cast<const float4*>(eta)[i4];
    return q;
  };
  BlockQuad q0;
  if (i0 < i1) q0 = load_quad(i0);
  // value range R = max_c (vmax_c - vmin_c)
  float R = tid < D ? ord2f(V.vmax[hs * D + tid]) - ord2f(V.vmin[hs * D + tid]) : -INFINITY;
  __syncthreads();
  if (round == 1 && tid == 0) {
    int nk = 0, nv = 0;
    for (int w = 0; w < BS_WARPS; ++w) { nk += wk[w]; nv += wv[w]; }
    if (r == 0) {
      GroupState gs = V.gst[hs];
      gs.n_kprom1 = nk;
      gs.n_vprom1 = nv;
      // the second pass pages in only the newly promoted key blocks and the value blocks
      gs.bytes += (long long)(nk - gs.n_kprom0 + nv) * F16_BLOCK_BYTES;
      V.gst[hs] = gs;
    }
    hsd.n_vprom = nv;
  }
  // the pass's reference Mc: the largest of the warps' (and M_prev); lane l holds warp
  // l mod 16's factor to it
  const float mw = m_s[lane & 15];
  const float Mc = fmaxf(M_prev, xw_max(mw));
  const float fw = (mw == Mc) ? 1.f : expf(mw - Mc);
  const float w_prev = (M_prev == Mc) ? 1.f : expf(M_prev - Mc);   // first-pass sums and tail
  const float lt = (tl_s[0] + tl_s[1]) * w_prev;
  float* red = V.red0 + hb * (D + 4);
  float L0 = xw_sum(l_s[lane & 15] * fw);
  if (round == 1) L0 += red[D] * w_prev;
  const float L = L0 + lt;
  if (round == 0 && tid == 0) red[D] = L0;
  if (tid < D) {
    float a = (round == 1) ? red[tid] * w_prev : 0.f;
#pragma unroll
    for (int w = 0; w < BS_WARPS; ++w) a = fmaf(acc_s[w][tid], __shfl_sync(0xffffffffu, fw, w), a);
    if (round == 0) red[tid] = a;
    float at = 0.f;
    for (int t = 0; t < V.n_tail; ++t)
      at = fmaf(tail_p[t], __half2float(V.tail_v[((size_t)hs * BLK + t) * D + tid]), at);
    a = fmaf(at, w_prev, a);
    V.out[hb * D + tid] = __float2half_rn(a / L);
  }
  hsd.M = Mc;
  // (3) certificate; in the first pass also the first ranking position (the best selected
  //     block by INT8 and by FP16 log-mass, ties to the lower index) and each block's
  //     rung-2 weight mass_b eta_b (kept in `keys`, normalised if rung 2 is planned)
  const float LSEp = Mc + logf(L);
  const float tail_mass = lt / L;
  float S = 0.f, A = 0.f, Ev = 0.f;
  float b8 = -INFINITY, b16 = -INFINITY;
  int i8 = 0x7fffffff, i16 = 0x7fffffff;
  for (int i = i0; i < i1; i += 4) {
    const BlockQuad q = (i == i0) ? q0 : load_quad(i);
    const unsigned char kf[4] = {q.kf.x, q.kf.y, q.kf.z, q.kf.w}, vf[4] = {q.vf.x, q.vf.y, q.vf.z, q.vf.w};
    const unsigned char sv[4] = {q.sl.x, q.sl.y, q.sl.z, q.sl.w};
    const float a8[4] = {q.l8.x, q.l8.y, q.l8.z, q.l8.w}, a16[4] = {q.l16.x, q.l16.y, q.l16.z, q.l16.w};
    const float dd[4] = {q.dl.x, q.dl.y, q.dl.z, q.dl.w}, ee[4] = {q.eta.x, q.eta.y, q.eta.z, q.eta.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      if (i + j >= i1) break;
      const bool kp = kf[j] != 0;
      const float pm = expf((kp ? a16[j] : a8[j]) - LSEp);
      if (kp) {
        A += pm;
      } else {
        S += pm * expm1f(dd[j]);
        A += pm * expf(-dd[j]);
      }
      const float pe = pm * ee[j];
      if (!vf[j]) Ev += pe;
      if (round == 0) keys[i + j] = __float_as_uint(pe);
      if (sv[j]) {   // this thread's blocks are visited in ascending index order
        if (a8[j] > b8 || (a8[j] == b8 && i + j < i8)) { b8 = a8[j]; i8 = i + j; }
        if (a16[j] > b16 || (a16[j] == b16 && i + j < i16)) { b16 = a16[j]; i16 = i + j; }
      }
    }
  }
  // one cross-warp round: R (max), S, A, Ev (sums) and the two arg-maxima (largest value,
  // then lowest index; value order by the order-preserving bits)
  {
    R = warp_max(R);
    S = warp_sum(S);
    A = warp_sum(A);
    Ev = warp_sum(Ev);
    uint32_t o8 = f2ord(b8), o16 = f2ord(b16);
    o8 = __reduce_max_sync(0xffffffffu, o8);
    o16 = __reduce_max_sync(0xffffffffu, o16);
    i8 = (int)__reduce_min_sync(0xffffffffu, f2ord(b8) == o8 ? (unsigned)i8 : 0x7fffffffu);
    i16 = (int)__reduce_min_sync(0xffffffffu, f2ord(b16) == o16 ? (unsigned)i16 : 0x7fffffffu);
    if (lane == 0) {
      cR[warp] = R; cS[warp] = S; cA[warp] = A; cE[warp] = Ev;
      c8[warp] = o8; c16[warp] = o16; ci8[warp] = i8; ci16[warp] = i16;
    }
    __syncthreads();
    const int l16 = lane & 15;
    R = xw_max(cR[l16]);
    S = xw_sum(cS[l16]);
    A = xw_sum(cA[l16]);
    Ev = xw_sum(cE[l16]);
    o8 = __reduce_max_sync(0xffffffffu, c8[l16]);
    o16 = __reduce_max_sync(0xffffffffu, c16[l16]);
    i8 = (int)__reduce_min_sync(0xffffffffu, c8[l16] == o8 ? (unsigned)ci8[l16] : 0x7fffffffu);
    i16 = (int)__reduce_min_sync(0xffffffffu, c16[l16] == o16 ? (unsigned)ci16[l16] : 0x7fffffffu);
    b8 = ord2f(o8);
    b16 = ord2f(o16);
  }
  A += tail_mass;
  const float e_key = S / A * R;
  const float e_val = Ev;
  hsd.e_key = e_key;
  hsd.e_val = e_val;
  if (round == 1) {
    hsd.level1 = (e_key + e_val <= V.eps && e_val <= V.v_tol) ? hsd.planned : 3;
    if (tid == 0) {
      V.hst[hb] = hsd;
      if (hsd.level1 == 3) {
        V.counters[CNT_ANY_DENSE] = 1u;
        atomicAdd(&V.counters[cnt_rung3(V.BG, b)], 1u);
      }
    }
    return;
  }
  // (4) ranking-consistency check over S_h: the top-R positions by INT8 and FP16 log-mass
  //     (position 1 came with the certificate pass)
  bool ok = true;
  if (hsd.k_star > 1) {
    ok = (i8 == i16);
    float last8 = b8, last16 = b16;
    int idx8 = i8, idx16 = i16;
    const int R_rank = min(V.rank_positions, hsd.k_star);
#pragma unroll 1
    for (int pos = 1; pos < R_rank && ok; ++pos) {
      float c8v = -INFINITY, c16v = -INFINITY;
      int j8 = 0x7fffffff, j16 = 0x7fffffff;
      for (int i4 = tid; i4 < (nb + 3) / 4; i4 += BS_THREADS) {
        const uchar4 s4 = reinterpret_cast<const uchar4*>(sel)[i4];
        if ((s4.x | s4.y | s4.z | s4.w) == 0) continue;
        const float4 l8 = reinterpret_cast<const float4*>(lse8)[i4];
        const float4 l16 = reinterpret_cast<const float4*>(lse16)[i4];
        const unsigned char sv[4] = {s4.x, s4.y, s4.z, s4.w};
        const float a8[4] = {l8.x, l8.y, l8.z, l8.w}, a16[4] = {l16.x, l16.y, l16.z, l16.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int i = 4 * i4 + j;
          if (i >= nb || !sv[j]) continue;
          const float x8 = a8[j], x16 = a16[j];
          const bool after8 = (x8 < last8) || (x8 == last8 && i > idx8);
          const bool after16 = (x16 < last16) || (x16 == last16 && i > idx16);
          if (after8 && (x8 > c8v || (x8 == c8v && i < j8))) { c8v = x8; j8 = i; }
          if (after16 && (x16 > c16v || (x16 == c16v && i < j16))) { c16v = x16; j16 = i; }
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float ob8 = __shfl_xor_sync(0xffffffffu, c8v, o);
        const int oi8 = __shfl_xor_sync(0xffffffffu, j8, o);
        if (ob8 > c8v || (ob8 == c8v && oi8 < j8)) { c8v = ob8; j8 = oi8; }
        const float ob16 = __shfl_xor_sync(0xffffffffu, c16v, o);
        const int oi16 = __shfl_xor_sync(0xffffffffu, j16, o);
        if (ob16 > c16v || (ob16 == c16v && oi16 < j16)) { c16v = ob16; j16 = oi16; }
      }
      __syncthreads();   // the previous position's slots have been read
      if (lane == 0) {
        cR[warp] = c8v; ci8[warp] = j8;
        cS[warp] = c16v; ci16[warp] = j16;
      }
      __syncthreads();
      for (int w = 0; w < BS_WARPS; ++w) {
        const float ob8 = cR[w], ob16 = cS[w];
        const int oi8 = ci8[w], oi16 = ci16[w];
        if (ob8 > c8v || (ob8 == c8v && oi8 < j8)) { c8v = ob8; j8 = oi8; }
        if (ob16 > c16v || (ob16 == c16v && oi16 < j16)) { c16v = ob16; j16 = oi16; }
      }
      ok = (j8 == j16);
      last8 = c8v; idx8 = j8; last16 = c16v; idx16 = j16;
    }
  }
  if (V.debug & 0x1) ok = false;
  hsd.rank_ok = ok ? 1 : 0;
  int planned = 0;
  if (!ok) {
    planned = 3;
  } else if (!(e_key + e_val <= V.eps && e_val <= V.v_tol)) {
    const float eps = V.eps;
    float S_proj = S;
    bool keys_rung2 = true;   // keys still hold the certificate pass's mass_b eta_b
    uint8_t* k1 = V.kprom1 + (size_t)hs * V.nbmax;
    uint8_t* v1 = V.vprom1 + (size_t)hs * V.nbmax;
    if (e_key > eps * 0.5f) {
      planned = 1;
      keys_rung2 = false;
      // rung 1: INT8 blocks by descending mass_b (e^Delta_b - 1) until the removed share
      // of S reaches 1 - eps A / (2 R S)
      const float need = 1.f - eps * A / (2.f * R * S);
#pragma unroll 1
      for (int i = i0; i < i1; i += 4) {
        const uchar4 kf4 = reinterpret_cast<const uchar4*>(kfl)[i >> 2];
        const float4 l8 = reinterpret_cast<const float4*>(lse8)[i >> 2];
        const float4 d4 = reinterpret_cast<const float4*>(dl)[i >> 2];
        const unsigned char kf[4] = {kf4.x, kf4.y, kf4.z, kf4.w};
        const float a8[4] = {l8.x, l8.y, l8.z, l8.w}, dd[4] = {d4.x, d4.y, d4.z, d4.w};
#pragma unroll
        for (int j = 0; j < 4; ++j)
          if (i + j < i1)
            keys[i + j] = kf[j] ? 0u : __float_as_uint(expf(a8[j] - LSEp) * expm1f(dd[j]) / S);
      }
      const SelResult sr = block_select_top(nb, fixed62(need), k1);
      S_proj = S * (1.f - __ull2float_rn(sr.taken) * 0x1p-62f);
      if (S_proj < 0.f) S_proj = 0.f;
    }
    const float ekey_proj = S_proj / A * R;
    if (!(ekey_proj + e_val <= eps && e_val <= V.v_tol)) {
      planned = 2;
      if (e_val > 0.f) {
        // rung 2: FP16 values by descending mass_b eta_b until the projected
        // E_key + E_val <= eps and E_val <= v_tol (every block is a candidate: no values
        // are FP16 yet)
        const float target = fminf(eps - ekey_proj, V.v_tol);
        const float need = 1.f - target / e_val;
        for (int i = i0; i < i1; i += 4) {
          if (keys_rung2) {
#pragma unroll
            for (int j = 0; j < 4; ++j)
              if (i + j < i1) keys[i + j] = __float_as_uint(__uint_as_float(keys[i + j]) / e_val);
          } else {
            const uchar4 kf4 = reinterpret_cast<const uchar4*>(kfl)[i >> 2];
            const float4 l8 = reinterpret_cast<const float4*>(lse8)[i >> 2];
            const float4 l16 = reinterpret_cast<const float4*>(lse16)[i >> 2];
            const float4 e4 = reinterpret_cast<const float4*>(eta)[i >> 2];
            const unsigned char kf[4] = {kf4.x, kf4.y, kf4.z, kf4.w};
            const float a8[4] = {l8.x, l8.y, l8.z, l8.w}, a16[4] = {l16.x, l16.y, l16.z, l16.w};
            const float ee[4] = {e4.x, e4.y, e4.z, e4.w};
#pragma unroll
            for (int j = 0; j < 4; ++j)
              if (i + j < i1)
                keys[i + j] = __float_as_uint(expf((kf[j] ? a16[j] : a8[j]) - LSEp) * ee[j] / e_val);
          }
        }
        block_select_top(nb, fixed62(need), v1);
      }
    }
    if (tid == 0 && planned > 0) {
      V.gst[hs].need_round1 = 1;
      V.counters[CNT_NEED_R1] = 1u;
    }
  }
  hsd.planned = planned;
  hsd.level1 = planned;   // rungs 1/2 are confirmed, or raised to 3, by the second pass
  if (tid == 0) {
    V.hst[hb] = hsd;
    if (planned == 3) {
      V.counters[CNT_ANY_DENSE] = 1u;
      atomicAdd(&V.counters[cnt_rung3(V.BG, b)], 1u);
    }
  }
}

namespace {

// Round 0 with INT4 values in VRAM.  Every block needs the INT4 codes and scale/offset of
// its values; a block that keeps its INT8 scores needs nothing else, a block with FP16
// keys needs its keys from tier 2 (or a resident copy) scored by the whole CTA.
//  - Blocks that keep INT8 scores are dealt to the warps by position in the work item
//    (block j to warp j mod 4), and a warp multiplies each of its blocks whole, all four
//    value groups, as the INT4 tail pass does: the weights of head hp at tokens
//    8 sub + [0, 8) split once into binary16 halves, each group's products p s 2^e as
//    exact halves by packed-half TwoProduct FMAs, INT4 codes as binary16 subnormals into
//    the MMA.  Its copies come from a two-stage cp.async ring that holds its own
//    positions only (the first one copied before the item's FP16-key flags are known; a
//    position whose keys turn out FP16 leaves an empty group in the ring).
//  - A block with FP16 keys is scored by the whole CTA between barriers, as before; each
//    warp then multiplies the weights into its own value group, whose codes and
//    scale/offset it loads directly while the keys are read.
//  - The item's reference M per head starts at the selection's and rises only where an
//    FP16-key block scores above it; every sum is then rescaled, so each item's partial
//    depends on its own blocks alone.  At the end of the item the four warps' sums meet
//    in shared memory and one partial per item is written, as before.
constexpr int R0_STAGES = 2;
constexpr int R0_CTAS_PER_SM = 3;
static_assert(CHUNK <= 32, "one FP16-key flag per lane of a warp");

// One block that keeps its INT8 scores, whole: INT4 codes (a lane's chunks at lane + 32 j),
// (scale, offset) per value group and token, and the INT8 scores of the group's heads.
struct __align__(16) R0Stage {
  uint4 codes[VC_BYTES / 16];     // 256 chunks
  uint4 so[VSV_WORDS / 4];        // 64 x 4 half2: [group][token]
  float4 s[MAXREP * BLK / 4];     // [head][token]
};

struct __align__(16) R0Smem {     // dynamic shared memory
  R0Stage ring[4][R0_STAGES];     // per warp
  uint32_t tw[4][MW_WORDS];       // per warp: the B words of one value group
  float p[MAXREP][BLK];           // weights of an FP16-key block
  float s16[MAXREP][BLK];         // its FP16 scores
  float qf[MAXREP][D];
  float M[MAXREP];                // the item's reference per head after an FP16-key block
  float fac[MAXREP];              // factor that moved the item's sums to that reference
  union {
    __half kbuf[BLK][KROW];                   // keys of an FP16-key block
    float red[4][NG][MAXREP][VG];             // item end: each warp's sums per group, head, channel
  } u;
  float lred[4][MAXREP];          // item end: each warp's weight sums per head
  int item;
  int res[2];
};

}  // namespace

__global__ void __launch_bounds__(128, R0_CTAS_PER_SM) mixed_kernel_r0(LayerView V) {
  pdl_trigger();
  pdl_wait();   // selection: FP16-key flags, reference maxima; scores of the scoring pass
  extern __shared__ __align__(16) unsigned char r0_dsm[];
  R0Smem& sm = *reinterpret_cast<R0Smem*>(r0_dsm);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int gid = lane >> 2, tig = lane & 3;
  const int hp = lane >> 3, sub = lane & 7;   // weight role: head hp, tokens 8 sub + [0, 8)
  const int nch = max(1, (V.nb + V.chunk - 1) / V.chunk);
  const int NCH = V.nslot;
  const int total = V.BG * nch;
  const bool act = hp < V.n_rep;              // head hp exists
  const bool wact = warp < V.n_rep;           // head `warp` exists (FP16-key role)
  const unsigned long long pol = evict_first_policy();
  R0Stage* ring = sm.ring[warp];
  uint32_t* tw = sm.tw[warp];
  int cur_hs = -1;
  int pre_e = 0;
  float pre_v = 1.f, pre_ef = 0.f;

  for (;;) {
    if (tid == 0) sm.item = (int)atomicAdd(&V.counters[CNT_MIX_Q], 1u);
    __syncthreads();
    const int item = sm.item;
    if (item >= total) break;
    const int hs = item / nch, ch = item % nch;
    const int b = hs / V.Hkv, g = hs % V.Hkv;
    const size_t hrow = head_row(V, b, g, 0);
    {   // the item's group, partial slot, blocks (tier 1, scratch) and tier-2 rows
      const long long be = min(V.nb, (ch + 1) * V.chunk);
      if (!bounds_ok(V.counters, V.debug, hs, V.BG, SITE_MIX0) ||
          !bounds_ok(V.counters, V.debug, ch, V.nslot, SITE_MIX0) ||
          !bounds_ok(V.counters, V.debug, be, (long long)V.nbmax + 1, SITE_MIX0) ||
          !bounds_ok(V.counters, V.debug, be * BLK, V.cap + 1, SITE_MIX0)) {
        __syncthreads();
        continue;
      }
    }
    if (hs != cur_hs) {
      cur_hs = hs;
      for (int i = tid; i < MAXREP * D; i += blockDim.x) {
        const int r = i / D, c = i % D;
        sm.qf[r][c] = (r < V.n_rep) ? __half2float(V.q[(hrow + r) * D + c]) : 0.f;
      }
      // weights p 2^e <= 2^e must be finite binary16 values on the INT8 path: e <= 15
      pre_e = min(15, prescale_exp(__half2float(__ushort_as_half((unsigned short)V.vscale_max[hs]))));
      pre_v = ldexpf(1.f, pre_e);
      pre_ef = (float)pre_e;
      __syncthreads();
    }
    float Mh = act ? V.hst[hrow + hp].M : 0.f;      // head hp: weights, offsets, sums
    float Mw = wact ? V.hst[hrow + warp].M : 0.f;   // head `warp`: FP16 scoring role

    const int blk0 = ch * V.chunk, blk_end = min(V.nb, blk0 + V.chunk);
    const int nblk = blk_end - blk0;
    const size_t bi0 = (size_t)hs * V.nbmax + blk0;
    unsigned kmask = 0;   // bit j: block blk0 + j has FP16 keys
    // copy of this warp's k-th position (block blk0 + warp + 4k) into slot k % R0_STAGES:
    // the whole block if it keeps its INT8 scores (or when `always`), else nothing; one
    // commit group either way
    auto issue = [&](int k, bool always) {
      const int j = warp + 4 * k;
      if (j < nblk && (always || !((kmask >> j) & 1u))) {
        const size_t bi = bi0 + j;
        R0Stage& T = ring[k % R0_STAGES];
        const uint4* vc = reinterpret_cast<const uint4*>(V.vc + bi * VC_BYTES);
#pragma unroll
        for (int jj = 0; jj < 8; ++jj) cp_async16_hint(&T.codes[lane + 32 * jj], vc + lane + 32 * jj, pol);
        const uint4* so = reinterpret_cast<const uint4*>(V.vsv + bi * VSV_WORDS);
        cp_async16_hint(&T.so[lane], so + lane, pol);
        cp_async16_hint(&T.so[lane + 32], so + lane + 32, pol);
#pragma unroll
        for (int jj = 0; jj < 2; ++jj) {   // 64 float4 of scores: head (lane + 32 jj) / 16
          const int idx = lane + 32 * jj, h = idx >> 4;
          if (h < V.n_rep)
            cp_async16_hint(&T.s[idx], V.shat + (hrow + h) * ((size_t)V.nbmax * BLK) + (size_t)(blk0 + j) * BLK + 4 * (idx & 15), pol);
        }
      }
      cp_async_commit();
    };
    // the first position is copied before the item's FP16-key flags arrive
    issue(0, true);
    {
      const unsigned char f = (lane < nblk) ? V.kprom0[bi0 + lane] : 0;
      kmask = __ballot_sync(0xffffffffu, f != 0);
    }
    issue(1, false);

    float accT[NG][2][4];   // INT8-score blocks of this warp: all four groups
#pragma unroll
    for (int gg = 0; gg < NG; ++gg)
#pragma unroll
      for (int mt = 0; mt < 2; ++mt)
#pragma unroll
        for (int j = 0; j < 4; ++j) accT[gg][mt][j] = 0.f;
    float2 offT[NG];        // sum p o per group, head hp, this lane's tokens (pairs)
#pragma unroll
    for (int gg = 0; gg < NG; ++gg) offT[gg] = make_float2(0.f, 0.f);
    float accF[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};   // FP16-key blocks: group `warp`
    float offF = 0.f;       // sum p o, group `warp`, head hp, this lane's tokens
    float lsumT = 0.f, lsumF = 0.f;   // sum p, head hp, this lane's tokens

    for (int j = 0; j < nblk; ++j) {
      const int blk = blk0 + j;
      if ((kmask >> j) & 1u) {
        // ---- FP16 keys from tier 2 (or their resident copy), scored by the whole CTA;
        //      the FP16 scores replace the INT8 ones in the score scratch for round 1 ----
        const size_t bi = (size_t)hs * V.nbmax + blk;
        // this warp's value group of the block: codes (two chunks) and the (scale,
        // offset) of this lane's eight tokens, loaded while the keys are read
        const uint4* vcp = reinterpret_cast<const uint4*>(V.vc + bi * VC_BYTES);
        const uint4 vcode0 = vcp[lane + 32 * (2 * warp)], vcode1 = vcp[lane + 32 * (2 * warp + 1)];
        const uint4* sop = reinterpret_cast<const uint4*>(V.vsv + bi * VSV_WORDS + warp * BLK);
        const uint4 S0 = sop[2 * sub], S1 = sop[2 * sub + 1];
        const ResPick pk = res_pick(V, 0, bi, sm.res);
        load_f16_block<KROW>(&sm.u.kbuf[0][0],
                             res_src(V, pk, V.t2k + ((size_t)hs * V.cap + (size_t)blk * BLK) * D),
                             res_dst(V, pk));
        res_commit(V, 0, bi, pk);
        __syncthreads();
        score_f16_block(sm.u.kbuf, sm.qf, sm.s16);
        __syncthreads();
        float p0 = 0.f, p1 = 0.f, fac = 1.f;
        if (wact) {
          const float sn0 = sm.s16[warp][lane], sn1 = sm.s16[warp][lane + 32];
          const float m = warp_max(fmaxf(sn0, sn1));
          const float l = warp_sum(expf(sn0 - m) + expf(sn1 - m));
          if (lane == 0) V.lse16[(hrow + warp) * V.nbmax + blk] = m + logf(l);
          float* shat_r = V.shat + (hrow + warp) * ((size_t)V.nbmax * BLK) + (size_t)blk * BLK;
          shat_r[lane] = sn0;
          shat_r[lane + 32] = sn1;
          if (m > Mw) {   // an FP16 score above the reference: raise it, rescale the sums
            fac = expf(Mw - m);
            Mw = m;
          }
          p0 = expf(sn0 - Mw) * pre_v;
          p1 = expf(sn1 - Mw) * pre_v;
        }
        if (lane == 0) {
          sm.fac[warp] = fac;
          sm.M[warp] = Mw;
        }
        sm.p[warp][lane] = p0;
        sm.p[warp][lane + 32] = p1;
        __syncthreads();
        {
          const float ft = sm.fac[tig], fh = sm.fac[hp];   // accumulator columns: head tig
          if (__any_sync(0xffffffffu, ft != 1.f || fh != 1.f)) {
#pragma unroll
            for (int gg = 0; gg < NG; ++gg) {
#pragma unroll
              for (int mt = 0; mt < 2; ++mt)
#pragma unroll
                for (int q = 0; q < 4; ++q) accT[gg][mt][q] *= ft;
              offT[gg].x *= fh;
              offT[gg].y *= fh;
            }
#pragma unroll
            for (int mt = 0; mt < 2; ++mt)
#pragma unroll
              for (int q = 0; q < 4; ++q) accF[mt][q] *= ft;
            offF *= fh;
            lsumT *= fh;
            lsumF *= fh;
          }
          if (act) Mh = sm.M[hp];
        }
        float pv[8];
        {
          const float4 pa = *reinterpret_cast<const float4*>(&sm.p[hp][8 * sub]);
          const float4 pc = *reinterpret_cast<const float4*>(&sm.p[hp][8 * sub + 4]);
          pv[0] = pa.x; pv[1] = pa.y; pv[2] = pa.z; pv[3] = pa.w;
          pv[4] = pc.x; pv[5] = pc.y; pv[6] = pc.z; pv[7] = pc.w;
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) lsumF += pv[i];
        // products p_t s_{t,g} 2^e of head hp at tokens 8 sub + [0, 8) as hi + lo halves,
        // exchanged through shared memory as B fragments
        {
          const uint32_t sw[8] = {S0.x, S0.y, S0.z, S0.w, S1.x, S1.y, S1.z, S1.w};
          uint32_t hw[4], lw[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) {   // token pair 4 sub + i
            const float2 a = __half22float2(u32_as_h2(sw[2 * i])), c = __half22float2(u32_as_h2(sw[2 * i + 1]));
            const float2 p2 = make_float2(pv[2 * i], pv[2 * i + 1]);
            offF = fmaf(p2.x, a.y, offF);
            offF = fmaf(p2.y, c.y, offF);
            const float2 w = mul2(p2, make_float2(a.x, c.x));
            const __half2 hi = __floats2half2_rn(w.x, w.y);
            const float2 rem = sub2(w, __half22float2(hi));   // exact remainders
            hw[i] = h2_as_u32(hi);
            lw[i] = h2_as_u32(__floats2half2_rn(rem.x, rem.y));
          }
          uint32_t* wr = tw + hp * (2 * MW_ROW) + 4 * sub;
          *reinterpret_cast<uint4*>(wr) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
          *reinterpret_cast<uint4*>(wr + MW_ROW) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
        }
        __syncwarp();
        {
          // column gid = (head gid>>1, hi or lo): k-step kk takes token pairs 8 tig + 2kk and
          // 8 tig + 2kk + 1 (tokens 16 tig + 4kk + {0,1} and {2,3})
          const uint32_t* rd = tw + (gid >> 1) * (2 * MW_ROW) + (gid & 1) * MW_ROW + 8 * tig;
          const uint4 B0 = *reinterpret_cast<const uint4*>(rd), B1 = *reinterpret_cast<const uint4*>(rd + 4);
          const uint32_t bb[8] = {B0.x, B0.y, B0.z, B0.w, B1.x, B1.y, B1.z, B1.w};
#pragma unroll
          for (int mt = 0; mt < 2; ++mt) {
            const uint4 Cw = mt ? vcode1 : vcode0;
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              uint32_t a0, a1, a2, a3;
              nib8_to_sub_f16x4(word_of(Cw, kk), a0, a1, a2, a3);
              mma16816(accF[mt], a0, a1, a2, a3, bb[2 * kk], bb[2 * kk + 1]);
            }
          }
        }
        __syncwarp();   // every lane has read the B words
      }
      if ((j & 3) != warp) continue;
      // ---- this warp's position: its ring slot (empty if the keys are FP16) ----
      const int k = j >> 2;
      cp_async_wait<R0_STAGES - 1>();
      __syncwarp();
      if (!((kmask >> j) & 1u)) {
        const R0Stage& T = ring[k % R0_STAGES];
        // weights of head hp at tokens 8 sub + [0, 8), times 2^e, with their binary16
        // halves (token pair i = tokens 8 sub + 2i, +1)
        float2 pf[4];
        __half2 ph[4], pl[4];
        {
          const float4 sa = T.s[hp * (BLK / 4) + 2 * sub], sb = T.s[hp * (BLK / 4) + 2 * sub + 1];
          const float sv[8] = {sa.x, sa.y, sa.z, sa.w, sb.x, sb.y, sb.z, sb.w};
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float p0 = act ? exp2_approx(fmaf(sv[2 * i] - Mh, LOG2E_F, pre_ef)) : 0.f;
            const float p1 = act ? exp2_approx(fmaf(sv[2 * i + 1] - Mh, LOG2E_F, pre_ef)) : 0.f;
            lsumT += p0 + p1;
            pf[i] = make_float2(p0, p1);
            ph[i] = __floats2half2_rn(p0, p1);
            const float2 r = sub2(pf[i], __half22float2(ph[i]));   // exact
            pl[i] = __floats2half2_rn(r.x, r.y);
          }
        }
#pragma unroll
        for (int gg = 0; gg < NG; ++gg) {
          const uint4 S0 = T.so[gg * (BLK / 4) + 2 * sub], S1 = T.so[gg * (BLK / 4) + 2 * sub + 1];
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
            offT[gg] = fma2(pf[i], __half22float2(o2), offT[gg]);
          }
          uint32_t* wr = tw + hp * (2 * MW_ROW) + 4 * sub;
          *reinterpret_cast<uint4*>(wr) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
          *reinterpret_cast<uint4*>(wr + MW_ROW) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
          __syncwarp();
          const uint32_t* rd = tw + (gid >> 1) * (2 * MW_ROW) + (gid & 1) * MW_ROW + 8 * tig;
          const uint4 B0 = *reinterpret_cast<const uint4*>(rd), B1 = *reinterpret_cast<const uint4*>(rd + 4);
          const uint32_t bb[8] = {B0.x, B0.y, B0.z, B0.w, B1.x, B1.y, B1.z, B1.w};
#pragma unroll
          for (int mt = 0; mt < 2; ++mt) {
            const uint4 Cw = T.codes[lane + 32 * (2 * gg + mt)];
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              uint32_t a0, a1, a2, a3;
              nib8_to_sub_f16x4(word_of(Cw, kk), a0, a1, a2, a3);
              mma16816(accT[gg][mt], a0, a1, a2, a3, bb[2 * kk], bb[2 * kk + 1]);
            }
          }
          __syncwarp();   // every lane has read the B words before the next group's
        }
      }
      __syncwarp();       // the slot is free: refill it with position k + 2
      issue(k + R0_STAGES, false);
    }
    cp_async_wait<0>();
    __syncwarp();

    // ---- this item's partial: the four warps' sums meet in shared memory ----
    float offs[NG];
#pragma unroll
    for (int gg = 0; gg < NG; ++gg) {
      offs[gg] = offT[gg].x + offT[gg].y + (gg == warp ? offF : 0.f);
      offs[gg] += __shfl_xor_sync(0xffffffffu, offs[gg], 1);   // head hp: its eight product lanes
      offs[gg] += __shfl_xor_sync(0xffffffffu, offs[gg], 2);
      offs[gg] += __shfl_xor_sync(0xffffffffu, offs[gg], 4);
    }
    float lsum = lsumT + (warp == 0 ? lsumF : 0.f);   // the FP16-key weights are the same in every warp
    lsum += __shfl_xor_sync(0xffffffffu, lsum, 1);
    lsum += __shfl_xor_sync(0xffffffffu, lsum, 2);
    lsum += __shfl_xor_sync(0xffffffffu, lsum, 4);
    // undo 2^e (weights) and 2^-24 / 2^-20 (subnormal code rows); powers of two, exact
    const float inv = ldexpf(1.f, -pre_e);
    const float inv_lo = inv * NIB_ROW_SCALE_LO, inv_hi = inv * NIB_ROW_SCALE_HI;
#pragma unroll
    for (int gg = 0; gg < NG; ++gg) {
      const float offh = __shfl_sync(0xffffffffu, offs[gg], 8 * tig);   // head tig
      float* rr = sm.u.red[warp][gg][tig];
#pragma unroll
      for (int mt = 0; mt < 2; ++mt) {
        float lo = accT[gg][mt][0] + accT[gg][mt][1], hi = accT[gg][mt][2] + accT[gg][mt][3];
        if (gg == warp) {
          lo += accF[mt][0] + accF[mt][1];
          hi += accF[mt][2] + accF[mt][3];
        }
        rr[16 * mt + gid] = lo * inv_lo + offh * inv;
        rr[16 * mt + gid + 8] = hi * inv_hi + offh * inv;
      }
    }
    if (sub == 0) sm.lred[warp][hp] = lsum;
    __syncthreads();
    float* pp = V.part + (((size_t)hs * NCH + ch) * MAXREP) * (D + 4);
    for (int h = 0; h < V.n_rep; ++h) {   // warp = value group, lane = channel
      const float s = ((sm.u.red[0][warp][h][lane] + sm.u.red[1][warp][h][lane]) + sm.u.red[2][warp][h][lane]) +
                      sm.u.red[3][warp][h][lane];
      pp[h * (D + 4) + VG * warp + lane] = s;
    }
    if (warp == 0 && sub == 0 && act) {
      const float l = ((sm.lred[0][hp] + sm.lred[1][hp]) + sm.lred[2][hp]) + sm.lred[3][hp];
      pp[hp * (D + 4) + D] = l * inv;
      pp[hp * (D + 4) + D + 1] = Mh;
    }
    __syncthreads();
  }
  if (tid == 0) {
    const unsigned int old = atomicAdd(&V.counters[CNT_MIX_EXIT], 1u);
    if (old == gridDim.x - 1) {
      V.counters[CNT_MIX_Q] = 0u;
      V.counters[CNT_MIX_EXIT] = 0u;
    }
  }
}

int mixed_grid(int num_sms) { return num_sms * 4; }

cudaError_t launch_mixed(const LayerView& V, int round, int grid, cudaStream_t st) {
  if (round == 0 && V.v16 == nullptr) {
    const int g0 = grid / 4 * R0_CTAS_PER_SM;   // grid = 4 CTAs per SM; round 0 holds fewer
    cudaError_t e = cudaFuncSetAttribute(mixed_kernel_r0, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)sizeof(R0Smem));
    if (e != cudaSuccess) return e;
    return launch_dependent(mixed_kernel_r0, dim3(g0), dim3(128), sizeof(R0Smem), st, V);
  }
  return launch_dependent(mixed_kernel, dim3(grid), dim3(128), 0, st, V, round);
}

cudaError_t launch_combine(const LayerView& V, int round, cudaStream_t st) {
  const size_t dyn = sizeof(BlockSelSmem) + (size_t)((V.nb + 15) & ~15) * 4;
  auto* k = round == 0 ? combine_kernel<0> : combine_kernel<1>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)dyn);
  if (e != cudaSuccess) return e;
  return launch_dependent(k, dim3(V.B * V.Hq), dim3(BS_THREADS), dyn, st, V);
}

}  // namespace kvq
