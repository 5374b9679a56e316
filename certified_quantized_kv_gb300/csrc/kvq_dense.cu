// kvq_dense.cu -- rungs 3 and 4 of the fallback ladder: exact dense FP16 attention over
// tier 2, and the final certificate write-out.
//
// "Runtime-Certified Bounded-Error Quantized Attention" (gist.science technical summary),
// Method §1 (fallback pages FP16 data in from tier 2 and runs exact dense attention for
// the affected head or layer), Method §3 (rung 3: per-head dense when the ranking check
// fails; rung 4: the whole layer dense) and Contributions ("deterministic recovery":
// O_dense is returned when the certified bound cannot be met).
// Readings: a head that failed its ranking check, or whose bound still exceeds eps after
// rungs 1-2, is recomputed densely (rung 3); when at least l4_head_fraction of a
// sequence's query heads are at rung 3, or tau_cov = 1, every head of that sequence is
// (rung 4).  Dense heads report E_key = E_val = 0.
//
// The kernel reads FP16 keys and values straight from pinned host memory over the host
// link (split-K over runs of up to 16 blocks, online softmax per run), which is the bound of
// this path; the CUDA cores keep up with the link, so no tensor-core tiling is used.  For
// the key blocks this call already paged in, the exact scores kept by the mixed pass are
// reused and only the values cross the link.
#include "kvq_common.cuh"
#include "kvq_launch.h"
#include "kvq_resident.cuh"
#include "kvq.h"

namespace kvq {

namespace {

struct __align__(16) DenseSmem {
  __half kbuf[BLK][D + 8];
  __half vbuf[BLK][D];
  float qf[MAXREP][D];
  float s[MAXREP][BLK];
  float red[MAXREP][4];
  float cacc[4][D];         // final merge: each warp's sums for one head (channels)
  float cml[4][2];          // ... and its reference and weight sum
  int item;
  int mask;
  int is_last;
  int res[4];   // residency picks: keys [0..1], values [2..3]
};

__device__ __forceinline__ size_t head_row(const LayerView& V, int b, int g, int r) {
  return (size_t)b * V.Hq + (size_t)g * V.n_rep + r;
}

// Heads of group hs that need dense attention (bit r = head slot r).
__device__ int dense_mask(const LayerView& V, int hs, int all_dense) {
  const int b = hs / V.Hkv, g = hs % V.Hkv;
  const int full = (1 << V.n_rep) - 1;
  if (all_dense) return full;
  const unsigned int n3 = V.counters[cnt_rung3(V.BG, b)];   // heads of sequence b at rung 3
  if (n3 == 0u) return 0;
  if ((float)n3 >= V.l4_frac * (float)V.Hq) return full;
  int m = 0;
  for (int r = 0; r < V.n_rep; ++r)
    if (V.hst[head_row(V, b, g, r)].level1 == 3) m |= 1 << r;
  return m;
}

__device__ void combine_dense(const LayerView& V, int hs, int mask, int all_dense, DenseSmem& sm) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int b = hs / V.Hkv, g = hs % V.Hkv;
  const int nch = max(1, (V.nb + V.chunk - 1) / V.chunk);
  const int NCH = V.nslot;
  // partial block exact scores (warp = head slot)
  if (warp < V.n_rep) {
    const __half* q = V.q + head_row(V, b, g, warp) * D;
    for (int t = lane; t < BLK; t += 32) {
      float s = -INFINITY;
      if (t < V.n_tail) s = dot_f16_row(q, V.tail_k + ((size_t)hs * BLK + t) * D) * INV_SQRT_D;
      sm.s[warp][t] = s;
    }
  }
  __syncthreads();
  const int nchv = V.nb > 0 ? nch : 0;
  if (__popc(mask) == 1) {
    // one dense head (rung 3): the four warps split its chunk partials (warp w takes
    // chunks w, w + 4, ... in batches of eight; lane = four channels), each summing
    // against its own running reference so that its loads go out together; thread =
    // channel then adds the four warps' sums in warp order and the partial block's tokens
    const int r = __ffs(mask) - 1;
    const float* P = V.dpart + ((size_t)hs * NCH * MAXREP + r) * (D + 4);   // chunk c at + c MAXREP (D + 4)
    float Mw = -INFINITY, L = 0.f;
    float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int base = warp; base < nchv; base += 4 * 8) {
      float Mi[8], Li[8];
      float4 x[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int c = base + 4 * j;
        if (c < nchv) {
          const float* pp = P + (size_t)c * MAXREP * (D + 4);
          Mi[j] = pp[D];
          Li[j] = pp[D + 1];
          x[j] = *reinterpret_cast<const float4*>(pp + 4 * lane);
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
        L *= f;
        Mw = Mb;
      }
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        // a chunk at reference -inf still adds its sums (zero, or NaN from NaN inputs)
        const float w = (Mi[j] == Mw) ? 1.f : expf(Mi[j] - Mw);
        a.x = fmaf(x[j].x, w, a.x); a.y = fmaf(x[j].y, w, a.y);
        a.z = fmaf(x[j].z, w, a.z); a.w = fmaf(x[j].w, w, a.w);
        L = fmaf(Li[j], w, L);
      }
    }
    *reinterpret_cast<float4*>(&sm.cacc[warp][4 * lane]) = a;
    if (lane == 0) { sm.cml[warp][0] = Mw; sm.cml[warp][1] = L; }
    __syncthreads();
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < 4; ++w) M = fmaxf(M, sm.cml[w][0]);
    for (int t = 0; t < V.n_tail; ++t) M = fmaxf(M, sm.s[r][t]);
    float acc = 0.f, Lt = 0.f;
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      const float mw = sm.cml[w][0];
      const float f = (mw == -INFINITY) ? 0.f : expf(mw - M);
      acc = fmaf(sm.cacc[w][tid], f, acc);
      Lt = fmaf(sm.cml[w][1], f, Lt);
    }
    for (int t = 0; t < V.n_tail; ++t) {
      const float p = expf(sm.s[r][t] - M);
      Lt += p;
      acc = fmaf(p, __half2float(V.tail_v[((size_t)hs * BLK + t) * D + tid]), acc);
    }
    V.out[head_row(V, b, g, r) * D + tid] = __float2half_rn(acc / Lt);
  } else {
    // several dense heads (rung 4): warp r combines head slot r's chunk partials (lane =
    // four channels): the global max over the chunk maxima and the partial block, then
    // the rescaled sums in chunk order
    const int r = warp;
    if (r < V.n_rep && (mask >> r & 1)) {
      const float* P = V.dpart + ((size_t)hs * NCH * MAXREP + r) * (D + 4);   // chunk c at + c MAXREP (D + 4)
      float M = -INFINITY;
      for (int c = lane; c < nchv; c += 32) M = fmaxf(M, P[(size_t)c * MAXREP * (D + 4) + D]);
      for (int t = lane; t < V.n_tail; t += 32) M = fmaxf(M, sm.s[r][t]);
      M = warp_max(M);
      float L = 0.f;
      float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 16
      for (int c = 0; c < nchv; ++c) {   // sixteen partials' loads in flight per lane
        const float* pp = P + (size_t)c * MAXREP * (D + 4);
        const float w = expf(pp[D] - M);
        const float4 x = *reinterpret_cast<const float4*>(pp + 4 * lane);
        L += pp[D + 1] * w;
        a.x += x.x * w; a.y += x.y * w; a.z += x.z * w; a.w += x.w * w;
      }
      for (int t = 0; t < V.n_tail; ++t) {
        const float p = expf(sm.s[r][t] - M);
        const uint2 vv = *reinterpret_cast<const uint2*>(V.tail_v + ((size_t)hs * BLK + t) * D + 4 * lane);
        const float2 v01 = __half22float2(u32_as_h2(vv.x)), v23 = __half22float2(u32_as_h2(vv.y));
        L += p;
        a.x += p * v01.x; a.y += p * v01.y; a.z += p * v23.x; a.w += p * v23.y;
      }
      __half2* o = reinterpret_cast<__half2*>(V.out + head_row(V, b, g, r) * D + 4 * lane);
      o[0] = __floats2half2_rn(a.x / L, a.y / L);
      o[1] = __floats2half2_rn(a.z / L, a.w / L);
    }
  }
  __syncthreads();
  if (tid == 0) {
    const unsigned int n3 = all_dense ? 0u : V.counters[cnt_rung3(V.BG, b)];
    const bool l4 = all_dense || ((float)n3 >= V.l4_frac * (float)V.Hq);
    for (int r = 0; r < V.n_rep; ++r) {
      HeadState& h = V.hst[head_row(V, b, g, r)];
      if (all_dense) {
        h.M = 0.f; h.lse_int8 = 0.f; h.tail_lse = 0.f;
        h.k_star = V.nb; h.rank_ok = 1; h.planned = 0; h.level1 = 0; h.n_vprom = 0;
      }
      if (mask >> r & 1) {
        h.level = l4 ? 4 : 3;
        h.e_key = 0.f;
        h.e_val = 0.f;
      }
    }
    GroupState& gs = V.gst[hs];
    if (all_dense) {
      gs.need_round1 = 0; gs.n_kprom0 = 0; gs.n_kprom1 = 0; gs.n_vprom1 = 0; gs.bytes = 0;
    }
    gs.need_dense = 1;
    // tier-2 values of every block (none when FP16 values are resident) and the keys of the
    // blocks whose FP16 scores this call does not already hold
    gs.bytes += ((long long)(V.nb - gs.n_kprom1) + (V.v16 ? 0LL : (long long)V.nb)) * F16_BLOCK_BYTES;
  }
}

}  // namespace

__global__ void __launch_bounds__(128) dense_kernel(LayerView V, int all_dense) {
  pdl_trigger();
  pdl_wait();   // ladder levels of the combine kernels
  __shared__ DenseSmem sm;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int nch = max(1, (V.nb + V.chunk - 1) / V.chunk);
  const int NCH = V.nslot;
  const int total = V.BG * nch;
  unsigned int* cnt_group = V.counters + CNT_GROUP_BASE + 3 * V.BG;
  int cur_hs = -1;
  if (!all_dense && V.counters[CNT_ANY_DENSE] == 0u) return;   // no head reached rung 3

  for (;;) {
    if (tid == 0) {
      const int it = (int)atomicAdd(&V.counters[CNT_DENSE_Q], 1u);
      sm.item = it;
      sm.mask = (it < total) ? dense_mask(V, it / nch, all_dense) : 0;
    }
    __syncthreads();
    const int item = sm.item;
    const int mask = sm.mask;
    if (item >= total) break;
    if (mask == 0) { __syncthreads(); continue; }
    const int hs = item / nch, ch = item % nch;
    const int b = hs / V.Hkv, g = hs % V.Hkv;
    {   // the item's group, partial slot, blocks (tier 1, scratch) and tier-2 rows
      const long long be = min(V.nb, (ch + 1) * V.chunk);
      if (!bounds_ok(V.counters, V.debug, hs, V.BG, SITE_DENSE) ||
          !bounds_ok(V.counters, V.debug, ch, V.nslot, SITE_DENSE) ||
          !bounds_ok(V.counters, V.debug, be, (long long)V.nbmax + 1, SITE_DENSE) ||
          !bounds_ok(V.counters, V.debug, be * BLK, V.cap + 1, SITE_DENSE)) {
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
      __syncthreads();
    }
    // online softmax over the chunk; thread = channel, all four head slots
    float m[MAXREP], l[MAXREP], a[MAXREP];
#pragma unroll
    for (int r = 0; r < MAXREP; ++r) { m[r] = -INFINITY; l[r] = 0.f; a[r] = 0.f; }
    const int blk_end = min(V.nb, (ch + 1) * V.chunk);
    for (int blk = ch * V.chunk; blk < blk_end; ++blk) {
      const size_t src = ((size_t)hs * V.cap + (size_t)blk * BLK) * D;
      // FP16 keys this call already paged in: their exact scores are in the score scratch
      const bool have_s = !all_dense && V.kprom1[(size_t)hs * V.nbmax + blk];
      {
        // tier 2 or the blocks' resident copies; all sixteen 16-byte loads of a thread in
        // flight before the first store
        const size_t bi = (size_t)hs * V.nbmax + blk;
        const ResPick pk = have_s ? ResPick{-1, -1} : res_pick(V, 0, bi, sm.res);
        const ResPick pv = V.v16 ? ResPick{-1, -1} : res_pick(V, 1, bi, sm.res + 2);
        const uint4* ks = reinterpret_cast<const uint4*>(res_src(V, pk, V.t2k + src));
        const uint4* vs = reinterpret_cast<const uint4*>(
            V.v16 ? V.v16 + bi * (BLK * D) : res_src(V, pv, V.t2v + src));   // FP16 values
        uint4* kcopy = reinterpret_cast<uint4*>(res_dst(V, pk));
        uint4* vcopy = reinterpret_cast<uint4*>(res_dst(V, pv));
        uint4 rk[8], rv[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          rv[j] = vs[tid + 128 * j];
          if (!have_s) rk[j] = ks[tid + 128 * j];
        }
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const int i = tid + 128 * j, row = i >> 4, col = (i & 15) * 8;
          if (!have_s) *reinterpret_cast<uint4*>(&sm.kbuf[row][col]) = rk[j];
          *reinterpret_cast<uint4*>(&sm.vbuf[row][col]) = rv[j];
        }
        if (kcopy) {
#pragma unroll
          for (int j = 0; j < 8; ++j) kcopy[tid + 128 * j] = rk[j];
        }
        if (vcopy) {
#pragma unroll
          for (int j = 0; j < 8; ++j) vcopy[tid + 128 * j] = rv[j];
        }
        res_commit(V, 0, bi, pk);
        res_commit(V, 1, bi, pv);
      }
      __syncthreads();
      if (have_s) {
        const int t = tid & 63, rp = (tid >> 6) * 2;
        const size_t o = (size_t)blk * BLK + t;
        const size_t row = (size_t)V.nbmax * BLK;
        sm.s[rp][t] = (rp < V.n_rep) ? V.shat[head_row(V, b, g, rp) * row + o] : 0.f;
        sm.s[rp + 1][t] = (rp + 1 < V.n_rep) ? V.shat[head_row(V, b, g, rp + 1) * row + o] : 0.f;
      } else {
        const int t = tid & 63, rp = (tid >> 6) * 2;
        float s0 = 0.f, s1 = 0.f;
        for (int c = 0; c < D; c += 8) {
          const uint4 kv = *reinterpret_cast<const uint4*>(&sm.kbuf[t][c]);
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
        sm.s[rp][t] = s0 * INV_SQRT_D;
        sm.s[rp + 1][t] = s1 * INV_SQRT_D;
      }
      __syncthreads();
      {  // block max per head, then p_t = exp(s_t - m_new) in place (warp = head slot)
        const int r = warp;
        const float x0 = sm.s[r][lane], x1 = sm.s[r][lane + 32];
        const float mn = fmaxf(m[r], warp_max(fmaxf(x0, x1)));
        const float p0 = expf(x0 - mn), p1 = expf(x1 - mn);
        sm.s[r][lane] = p0;
        sm.s[r][lane + 32] = p1;
        const float ls = warp_sum(p0 + p1);
        if (lane == 0) { sm.red[r][0] = mn; sm.red[r][1] = ls; }
      }
      __syncthreads();
#pragma unroll
      for (int r = 0; r < MAXREP; ++r) {   // head slots r < n_rep (unrolled: m, l, a stay in registers)
        if (r < V.n_rep) {
          const float mn = sm.red[r][0];
          const float sc = (m[r] == -INFINITY) ? 0.f : expf(m[r] - mn);
          float as = 0.f;
          for (int t = 0; t < BLK; ++t) as = fmaf(sm.s[r][t], __half2float(sm.vbuf[t][tid]), as);
          l[r] = l[r] * sc + sm.red[r][1];
          a[r] = a[r] * sc + as;
          m[r] = mn;
        }
      }
      __syncthreads();
    }
    float* pp = V.dpart + (((size_t)hs * NCH + ch) * MAXREP) * (D + 4);
#pragma unroll
    for (int r = 0; r < MAXREP; ++r) {
      if (r < V.n_rep) {
        pp[r * (D + 4) + tid] = a[r];
        if (tid == 0) {
          pp[r * (D + 4) + D] = m[r];
          pp[r * (D + 4) + D + 1] = l[r];
        }
      }
    }
    __syncthreads();
    if (tid == 0) {
      __threadfence();
      const unsigned int old = atomicAdd(&cnt_group[hs], 1u);
      sm.is_last = (old == (unsigned int)(nch - 1));
    }
    __syncthreads();
    if (sm.is_last) {
      __threadfence();
      combine_dense(V, hs, mask, all_dense, sm);
      if (tid == 0) cnt_group[hs] = 0u;
    }
    __syncthreads();
  }
  if (tid == 0) {
    const unsigned int old = atomicAdd(&V.counters[CNT_DENSE_EXIT], 1u);
    if (old == gridDim.x - 1) {
      V.counters[CNT_DENSE_Q] = 0u;
      V.counters[CNT_DENSE_EXIT] = 0u;
    }
  }
}

// Final certificates and per-sequence ladder level; one CTA per sequence.
__global__ void finalize_kernel(LayerView V, kvq_certificate* cert, int32_t* level) {
  pdl_wait();   // every head's state
  const int b = blockIdx.x;
  __shared__ int mx;
  if (threadIdx.x == 0) mx = 0;
  __syncthreads();
  for (int h = threadIdx.x; h < V.Hq; h += blockDim.x) {
    HeadState& s = V.hst[(size_t)b * V.Hq + h];
    if (s.level < 0) s.level = s.level1;
    const int g = h / V.n_rep;
    kvq_certificate c;
    c.e_key = s.e_key;
    c.e_val = s.e_val;
    c.rank_ok = s.rank_ok;
    c.level = s.level;
    c.k_star = s.k_star;
    c.n_val_promoted = s.n_vprom;
    c.promoted_bytes = V.gst[(size_t)b * V.Hkv + g].bytes;
    if (cert) cert[(size_t)b * V.Hq + h] = c;
    atomicMax(&mx, s.level);
  }
  __syncthreads();
  if (threadIdx.x == 0 && level) level[b] = mx;
  if (threadIdx.x == 0) V.counters[cnt_rung3(V.BG, b)] = 0u;   // consumed by the dense pass
  if (b == 0 && threadIdx.x == 0) {   // the flags of this call have been consumed
    V.counters[CNT_ANY_DENSE] = 0u;
    V.counters[CNT_NEED_R1] = 0u;
  }
}

int dense_grid(int num_sms) { return num_sms * 3; }

cudaError_t launch_dense(const LayerView& V, int all_dense, int grid, cudaStream_t st) {
  return launch_dependent(dense_kernel, dim3(grid), dim3(128), 0, st, V, all_dense);
}

cudaError_t launch_finalize(const LayerView& V, kvq_certificate* cert, int32_t* level,
                            cudaStream_t st) {
  return launch_dependent(finalize_kernel, dim3(V.B), dim3(128), 0, st, V, cert, level);
}

}  // namespace kvq
