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
// Work split: a persistent grid takes (KV group, 16-block chunk) items from a queue.
// For each block the CTA first produces p_t = exp(s'_t - M) for the four query heads in
// shared memory -- from the stored INT8 scores, or from FP16 keys read from tier 2 -- and
// then each warp (one 32-channel value group) multiplies them into V: INT4 codes on the
// tensor cores (channels as MMA rows, tokens as k, the eight MMA columns = four heads x
// hi/lo halves of p * scale), FP16 values of promoted blocks on the CUDA cores.  M >= every
// score, so no online rescaling is needed.  The CTA that completes a group combines the
// chunk partials in a fixed order and writes the output, certificate and ladder plan.
#include "kvq_common.cuh"
#include "kvq_launch.h"

namespace kvq {

namespace {

constexpr int KROW = D + 8;   // padded FP16 row (272 bytes): conflict-free 16-byte reads

struct __align__(16) MixSmem {
  float p[2][MAXREP][BLK];
  float qf[MAXREP][D];
  float M[MAXREP];
  union __align__(16) {
    struct {
      __half kbuf[BLK][KROW];
      __half vbuf[BLK][D];
    } st;
    struct {
      unsigned long long hist[4][256];
      float tail_s[MAXREP][BLK];
      float l[MAXREP];
      float lse[MAXREP];
      float red[4];
      int cnt[4];
    } cb;
  } u;
  int item;
  int is_last;
  int skip;
};

__device__ __forceinline__ size_t head_row(const LayerView& V, int b, int g, int r) {
  return (size_t)b * V.Hq + (size_t)g * V.n_rep + r;
}

__device__ __forceinline__ unsigned long long fixed62(double x) {
  // x in [0, 1] -> x * 2^62 (rounded toward zero)
  if (!(x > 0.0)) return 0ull;
  if (x >= 1.0) return 4611686018427387904ull;
  return (unsigned long long)(x * 4611686018427387904.0);
}

// Copy one FP16 block (64 x 128) from tier 2 into shared memory with row stride KROW.
__device__ __forceinline__ void load_f16_block(__half (*dst)[KROW], const __half* src) {
  const uint4* s = reinterpret_cast<const uint4*>(src);
  for (int i = threadIdx.x; i < BLK * D / 8; i += blockDim.x) {
    const int row = i >> 4, col = (i & 15) * 8;
    *reinterpret_cast<uint4*>(&dst[row][col]) = s[i];
  }
}
__device__ __forceinline__ void load_f16_block_dense(__half (*dst)[D], const __half* src) {
  const uint4* s = reinterpret_cast<const uint4*>(src);
  for (int i = threadIdx.x; i < BLK * D / 8; i += blockDim.x) {
    const int row = i >> 4, col = (i & 15) * 8;
    *reinterpret_cast<uint4*>(&dst[row][col]) = s[i];
  }
}

// Combine the chunk partials of one group, add the partial block, write outputs and the
// certificate; in the first pass also run the ranking check and plan rungs 1 and 2.
__device__ void combine_group(const LayerView& V, int hs, int round, MixSmem& sm) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int b = hs / V.Hkv, g = hs % V.Hkv;
  const int nb = V.nb;
  const int nch = max(1, (nb + CHUNK - 1) / CHUNK);
  const int NCH = V.nbmax / CHUNK + 1;
  const uint8_t* kfl = (round == 0 ? V.kprom0 : V.kprom1) + (size_t)hs * V.nbmax;
  const uint8_t* vfl = V.vprom1 + (size_t)hs * V.nbmax;

  // which heads take this pass's result
  bool take[MAXREP];
  for (int r = 0; r < MAXREP; ++r) {
    take[r] = false;
    if (r < V.n_rep) {
      const HeadState& h = V.hst[head_row(V, b, g, r)];
      take[r] = (round == 0) || (h.planned == 1 || h.planned == 2);
    }
  }

  // (1) chunk partials in fixed order: thread = channel
  float acc[MAXREP];
  for (int r = 0; r < MAXREP; ++r) acc[r] = 0.f;
  for (int c = 0; c < nch; ++c) {
    const float* pp = V.part + (((size_t)hs * NCH + c) * MAXREP) * (D + 4);
    for (int r = 0; r < V.n_rep; ++r) acc[r] += pp[r * (D + 4) + tid];
  }
  if (warp < V.n_rep) {
    float l = 0.f;
    for (int c = lane; c < nch; c += 32)
      l += V.part[(((size_t)hs * NCH + c) * MAXREP + warp) * (D + 4) + D];
    l = warp_sum(l);
    // (2) partial FP16 block: exact scores
    const size_t hb = head_row(V, b, g, warp);
    const float M = V.hst[hb].M;
    const __half* q = V.q + hb * D;
    float lt = 0.f;
    for (int t = lane; t < V.n_tail; t += 32) {
      const __half* k = V.tail_k + ((size_t)hs * BLK + t) * D;
      float s = 0.f;
      for (int c = 0; c < D; c += 2) {
        const float2 kk = __half22float2(*reinterpret_cast<const __half2*>(k + c));
        const float2 qq = __half22float2(*reinterpret_cast<const __half2*>(q + c));
        s = fmaf(qq.x, kk.x, s);
        s = fmaf(qq.y, kk.y, s);
      }
      const float p = expf(s * INV_SQRT_D - M);
      sm.u.cb.tail_s[warp][t] = p;
      lt += p;
    }
    lt = warp_sum(lt);
    if (lane == 0) {
      sm.u.cb.l[warp] = l + lt;
      sm.u.cb.lse[warp] = lt;  // tail mass numerator, normalised below
    }
  }
  __syncthreads();
  for (int r = 0; r < V.n_rep; ++r) {
    float a = acc[r];
    for (int t = 0; t < V.n_tail; ++t)
      a += sm.u.cb.tail_s[r][t] * __half2float(V.tail_v[((size_t)hs * BLK + t) * D + tid]);
    if (take[r]) {
      const size_t hb = head_row(V, b, g, r);
      V.out[hb * D + tid] = __float2half_rn(a / sm.u.cb.l[r]);
    }
  }
  // value range R = max_c (vmax_c - vmin_c)
  float rng = ord2f(V.vmax[hs * D + tid]) - ord2f(V.vmin[hs * D + tid]);
  rng = warp_max(rng);
  if (lane == 0) sm.u.cb.red[warp] = rng;
  __syncthreads();
  const float R = fmaxf(fmaxf(sm.u.cb.red[0], sm.u.cb.red[1]), fmaxf(sm.u.cb.red[2], sm.u.cb.red[3]));

  // (3) certificate per head: warp = head slot
  if (warp < V.n_rep && take[warp]) {
    const int r = warp;
    const size_t hb = head_row(V, b, g, r);
    HeadState hsd = V.hst[hb];
    const float L = sm.u.cb.l[r];
    const float LSEp = hsd.M + logf(L);
    const float tail_mass = sm.u.cb.lse[r] / L;
    const float* lse8 = V.lse8 + hb * V.nbmax;
    const float* lse16 = V.lse16 + hb * V.nbmax;
    const float* dl = V.delta + hb * V.nbmax;
    const float* eta = V.eta + (size_t)hs * V.nbmax;
    float S = 0.f, A = 0.f, Ev = 0.f;
    for (int i = lane; i < nb; i += 32) {
      const bool kp = kfl[i] != 0;
      const float pm = expf((kp ? lse16[i] : lse8[i]) - LSEp);
      if (kp) {
        A += pm;
      } else {
        S += pm * expm1f(dl[i]);
        A += pm * expf(-dl[i]);
      }
      if (!vfl[i]) Ev += pm * eta[i];
    }
    S = warp_sum(S);
    A = warp_sum(A) + tail_mass;
    Ev = warp_sum(Ev);
    const float e_key = S / A * R;
    const float e_val = Ev;
    hsd.e_key = e_key;
    hsd.e_val = e_val;

    if (round == 0) {
      // ranking-consistency check over S_h: top-R positions by INT8 and by FP16 log-mass
      const uint8_t* sel = V.sel + hb * V.nbmax;
      bool ok = true;
      if (hsd.k_star > 1) {
        float last8 = INFINITY, last16 = INFINITY;
        int idx8 = -1, idx16 = -1;
        const int R_rank = min(V.rank_positions, hsd.k_star);
        for (int pos = 0; pos < R_rank && ok; ++pos) {
          // next entry after (last, idx) in descending order, ties to lower index
          float b8 = -INFINITY, b16 = -INFINITY;
          int i8 = 0x7fffffff, i16 = 0x7fffffff;
          for (int i = lane; i < nb; i += 32) {
            if (!sel[i]) continue;
            const float x8 = lse8[i], x16 = lse16[i];
            const bool after8 = (x8 < last8) || (x8 == last8 && i > idx8);
            const bool after16 = (x16 < last16) || (x16 == last16 && i > idx16);
            if (after8 && (x8 > b8 || (x8 == b8 && i < i8))) { b8 = x8; i8 = i; }
            if (after16 && (x16 > b16 || (x16 == b16 && i < i16))) { b16 = x16; i16 = i; }
          }
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) {
            const float ob8 = __shfl_xor_sync(0xffffffffu, b8, o);
            const int oi8 = __shfl_xor_sync(0xffffffffu, i8, o);
            if (ob8 > b8 || (ob8 == b8 && oi8 < i8)) { b8 = ob8; i8 = oi8; }
            const float ob16 = __shfl_xor_sync(0xffffffffu, b16, o);
            const int oi16 = __shfl_xor_sync(0xffffffffu, i16, o);
            if (ob16 > b16 || (ob16 == b16 && oi16 < i16)) { b16 = ob16; i16 = oi16; }
          }
          ok = (i8 == i16);
          last8 = b8; idx8 = i8; last16 = b16; idx16 = i16;
        }
      }
      if (V.debug & 0x1) ok = false;
      hsd.rank_ok = ok ? 1 : 0;
      int planned = 0;
      if (!ok) {
        planned = 3;
      } else if (!(e_key + e_val <= V.eps)) {
        const float eps = V.eps;
        float S_proj = S;
        uint8_t* k1 = V.kprom1 + (size_t)hs * V.nbmax;
        uint8_t* v1 = V.vprom1 + (size_t)hs * V.nbmax;
        if (e_key > eps * 0.5f) {
          planned = 1;
          // rung 1: take INT8 blocks by descending mass_b (e^Delta_b - 1) until the
          // removed share reaches S - eps A / (2R)
          const double need = 1.0 - (double)eps * (double)A / (2.0 * (double)R * (double)S);
          auto key_of = [&](int i) -> uint32_t {
            if (kfl[i]) return 0u;
            const float pm = expf(lse8[i] - LSEp);
            return __float_as_uint(pm * expm1f(dl[i]));
          };
          auto w_of = [&](int i) -> unsigned long long {
            return fixed62((double)__uint_as_float(key_of(i)) / (double)S);
          };
          auto mark = [&](int i) { k1[i] = 1; };
          unsigned long long taken = 0;
          warp_select_top(nb, fixed62(need), key_of, w_of, mark, sm.u.cb.hist[warp], &taken);
          S_proj = (float)((double)S * (1.0 - (double)taken / 4611686018427387904.0));
          if (S_proj < 0.f) S_proj = 0.f;
        }
        const float ekey_proj = S_proj / A * R;
        if (!(ekey_proj + e_val <= eps)) {
          planned = 2;
          if (e_val > 0.f) {
            const double need = 1.0 - ((double)eps - (double)ekey_proj) / (double)e_val;
            auto key_of = [&](int i) -> uint32_t {
              if (vfl[i]) return 0u;
              const float pm = expf((kfl[i] ? lse16[i] : lse8[i]) - LSEp);
              return __float_as_uint(pm * eta[i]);
            };
            auto w_of = [&](int i) -> unsigned long long {
              return fixed62((double)__uint_as_float(key_of(i)) / (double)e_val);
            };
            auto mark = [&](int i) { v1[i] = 1; };
            unsigned long long taken = 0;
            warp_select_top(nb, fixed62(need), key_of, w_of, mark, sm.u.cb.hist[warp], &taken);
          }
        }
      }
      hsd.planned = planned;
      hsd.level1 = planned;  // rungs 1/2 are confirmed (or raised to 3) by the second pass
    } else {
      hsd.level1 = (e_key + e_val <= V.eps) ? hsd.planned : 3;
    }
    if (lane == 0) V.hst[hb] = hsd;
  }
  __syncthreads();
  // group bookkeeping
  if (round == 0) {
    if (tid == 0) {
      int need = 0;
      for (int r = 0; r < V.n_rep; ++r) {
        const int p = V.hst[head_row(V, b, g, r)].planned;
        need |= (p == 1 || p == 2);
      }
      V.gst[hs].need_round1 = need;
    }
  } else {
    int nk = 0, nv = 0;
    for (int i = tid; i < nb; i += blockDim.x) {
      nk += V.kprom1[(size_t)hs * V.nbmax + i];
      nv += V.vprom1[(size_t)hs * V.nbmax + i];
    }
    nk = (int)warp_sum((float)nk);
    nv = (int)warp_sum((float)nv);
    if (lane == 0) sm.u.cb.cnt[warp] = nk | (nv << 16);
    __syncthreads();
    if (tid == 0) {
      int tk = 0, tv = 0;
      for (int w = 0; w < 4; ++w) { tk += sm.u.cb.cnt[w] & 0xffff; tv += sm.u.cb.cnt[w] >> 16; }
      GroupState gs = V.gst[hs];
      gs.n_kprom1 = tk;
      gs.n_vprom1 = tv;
      gs.bytes += (long long)(tk + tv) * F16_BLOCK_BYTES;
      V.gst[hs] = gs;
      for (int r = 0; r < V.n_rep; ++r) {
        HeadState& h = V.hst[head_row(V, b, g, r)];
        if (h.planned == 1 || h.planned == 2) h.n_vprom = tv;
      }
    }
  }
}

}  // namespace

__global__ void __launch_bounds__(128) mixed_kernel(LayerView V, int round) {
  __shared__ MixSmem sm;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int gid = lane >> 2, tig = lane & 3;
  const int nch = max(1, (V.nb + CHUNK - 1) / CHUNK);
  const int NCH = V.nbmax / CHUNK + 1;
  const int total = V.BG * nch;
  unsigned int* cnt_group = V.counters + CNT_GROUP_BASE + (1 + round) * V.BG;
  const uint8_t* kflags = round == 0 ? V.kprom0 : V.kprom1;
  int par = 0;
  int cur_hs = -1;
  float pre_v = 1.f;

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

    if (hs != cur_hs) {
      cur_hs = hs;
      for (int i = tid; i < MAXREP * D; i += blockDim.x) {
        const int r = i / D, c = i % D;
        sm.qf[r][c] = (r < V.n_rep) ? __half2float(V.q[head_row(V, b, g, r) * D + c]) : 0.f;
      }
      if (tid < MAXREP) sm.M[tid] = (tid < V.n_rep) ? V.hst[head_row(V, b, g, tid)].M : 0.f;
      pre_v = prescale_for(__half2float(__ushort_as_half((unsigned short)V.vscale_max[hs])));
      __syncthreads();
    }

    float acc[2][4];
#pragma unroll
    for (int i = 0; i < 2; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;
    float acc16[4] = {0.f, 0.f, 0.f, 0.f};
    float off = 0.f;     // sum p * offset for head gid>>1, group = warp
    float lsum = 0.f;    // sum p for head = warp

    const int blk_end = min(V.nb, (ch + 1) * CHUNK);
    for (int blk = ch * CHUNK; blk < blk_end; ++blk, par ^= 1) {
      const size_t bi = (size_t)hs * V.nbmax + blk;
      const bool kp = kflags[bi] != 0;
      const bool vp = (round == 1) && V.vprom1[bi] != 0;
      // ---- stage 1: p_t = exp(s'_t - M) for the group's query heads ----
      if (!kp) {
        const int r = warp;
        float p0 = 0.f, p1 = 0.f;
        if (r < V.n_rep) {
          const float2 s2 = __ldcs(reinterpret_cast<const float2*>(
              V.shat + head_row(V, b, g, r) * ((size_t)V.nbmax * BLK) + (size_t)blk * BLK + 2 * lane));
          p0 = __expf(s2.x - sm.M[r]);
          p1 = __expf(s2.y - sm.M[r]);
        }
        sm.p[par][r][2 * lane] = p0;
        sm.p[par][r][2 * lane + 1] = p1;
        lsum += p0 + p1;
      } else {
        load_f16_block(sm.u.st.kbuf, V.t2k + ((size_t)hs * V.cap + (size_t)blk * BLK) * D);
        __syncthreads();
        {
          const int t = tid & 63, rp = (tid >> 6) * 2;  // heads rp, rp+1
          float s0 = 0.f, s1 = 0.f;
#pragma unroll 4
          for (int c = 0; c < D; c += 8) {
            const uint4 kv = *reinterpret_cast<const uint4*>(&sm.u.st.kbuf[t][c]);
            const __half2* k2 = reinterpret_cast<const __half2*>(&kv);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const float2 kf = __half22float2(k2[j]);
              s0 = fmaf(sm.qf[rp][c + 2 * j], kf.x, s0);
              s0 = fmaf(sm.qf[rp][c + 2 * j + 1], kf.y, s0);
              s1 = fmaf(sm.qf[rp + 1][c + 2 * j], kf.x, s1);
              s1 = fmaf(sm.qf[rp + 1][c + 2 * j + 1], kf.y, s1);
            }
          }
          sm.p[par][rp][t] = s0 * INV_SQRT_D;
          sm.p[par][rp + 1][t] = s1 * INV_SQRT_D;
        }
        __syncthreads();
        {
          const int r = warp;
          const float x0 = sm.p[par][r][lane], x1 = sm.p[par][r][lane + 32];
          float p0 = 0.f, p1 = 0.f;
          if (r < V.n_rep) {
            const float m = warp_max(fmaxf(x0, x1));
            const float l = warp_sum(expf(x0 - m) + expf(x1 - m));
            if (lane == 0) V.lse16[head_row(V, b, g, r) * V.nbmax + blk] = m + logf(l);
            p0 = expf(x0 - sm.M[r]);
            p1 = expf(x1 - sm.M[r]);
          }
          sm.p[par][r][lane] = p0;
          sm.p[par][r][lane + 32] = p1;
          lsum += p0 + p1;
        }
      }
      __syncthreads();
      // ---- stage 2: p x V for the warp's value group ----
      if (!vp) {
        const uint4* vcp = reinterpret_cast<const uint4*>(V.vc + bi * VC_BYTES) + (warp * 2) * 32 + lane;
        const uint4 C0 = __ldcs(vcp), C1 = __ldcs(vcp + 32);
        const uint4* svp = reinterpret_cast<const uint4*>(V.vsv + bi * VSV_WORDS + warp * BLK + 16 * tig);
        const int r = gid >> 1;
        const float* pr = &sm.p[par][r][16 * tig];
        uint32_t bb0[4], bb1[4];
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          const uint4 so = __ldcs(svp + kk);                       // tokens 4kk .. 4kk+3
          const float4 pp = *reinterpret_cast<const float4*>(pr + 4 * kk);
          const __half2* so2 = reinterpret_cast<const __half2*>(&so);
          const float pv[4] = {pp.x, pp.y, pp.z, pp.w};
          __half sel[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float2 sof = __half22float2(so2[i]);
            off = fmaf(pv[i], sof.y, off);
            __half hi, lo;
            split_hl(pv[i] * sof.x * pre_v, hi, lo);
            sel[i] = (gid & 1) ? lo : hi;
          }
          bb0[kk] = h2_as_u32(__halves2half2(sel[0], sel[1]));
          bb1[kk] = h2_as_u32(__halves2half2(sel[2], sel[3]));
        }
#pragma unroll
        for (int mt = 0; mt < 2; ++mt) {
          const uint4 C = mt ? C1 : C0;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint32_t w = (kk == 0) ? C.x : (kk == 1) ? C.y : (kk == 2) ? C.z : C.w;
            mma16816(acc[mt], nib_to_f16(w, 0), nib_to_f16(w, 1), nib_to_f16(w, 2),
                     nib_to_f16(w, 3), bb0[kk], bb1[kk]);
          }
        }
      } else {
        load_f16_block_dense(sm.u.st.vbuf, V.t2v + ((size_t)hs * V.cap + (size_t)blk * BLK) * D);
        __syncthreads();
        const int c0 = 32 * warp + gid;
        const float* pr = sm.p[par][tig];
        for (int t = 0; t < BLK; ++t) {
          const float pt = pr[t];
          acc16[0] = fmaf(pt, __half2float(sm.u.st.vbuf[t][c0]), acc16[0]);
          acc16[1] = fmaf(pt, __half2float(sm.u.st.vbuf[t][c0 + 8]), acc16[1]);
          acc16[2] = fmaf(pt, __half2float(sm.u.st.vbuf[t][c0 + 16]), acc16[2]);
          acc16[3] = fmaf(pt, __half2float(sm.u.st.vbuf[t][c0 + 24]), acc16[3]);
        }
      }
    }

    // ---- write this chunk's partial: l and acc[D] per head ----
    off += __shfl_xor_sync(0xffffffffu, off, 1);
    off += __shfl_xor_sync(0xffffffffu, off, 2);
    const float offh = __shfl_sync(0xffffffffu, off, 8 * tig);  // head tig, hi lane
    const float inv = 1.f / pre_v;
    float* pp = V.part + (((size_t)hs * NCH + ch) * MAXREP) * (D + 4);
    if (tig < V.n_rep) {
      float* pr = pp + tig * (D + 4);
      const int c0 = 32 * warp + gid;
      pr[c0] = (acc[0][0] + acc[0][1]) * inv + acc16[0] + offh;
      pr[c0 + 8] = (acc[0][2] + acc[0][3]) * inv + acc16[1] + offh;
      pr[c0 + 16] = (acc[1][0] + acc[1][1]) * inv + acc16[2] + offh;
      pr[c0 + 24] = (acc[1][2] + acc[1][3]) * inv + acc16[3] + offh;
    }
    lsum = warp_sum(lsum);
    if (lane == 0 && warp < V.n_rep) pp[warp * (D + 4) + D] = lsum;

    __syncthreads();
    if (tid == 0) {
      __threadfence();
      const unsigned int old = atomicAdd(&cnt_group[hs], 1u);
      sm.is_last = (old == (unsigned int)(nch - 1));
    }
    __syncthreads();
    if (sm.is_last) {
      __threadfence();
      combine_group(V, hs, round, sm);
      if (tid == 0) cnt_group[hs] = 0u;
      cur_hs = -1;  // the union was reused by the combine
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
  mixed_kernel<<<grid, 128, 0, st>>>(V, round);
  return cudaGetLastError();
}

}  // namespace kvq
