// kvq_dense_hbm.cu -- exact dense FP16 decode attention over keys and values held in
// device memory: the dense baseline that the certified path is set against.
//
// "Runtime-Certified Bounded-Error Quantized Attention" (gist.science technical summary):
// Method §1 names dense FP16 attention as the ground truth the ladder falls back to, and
// Results (performance overhead) quotes the certified step's latency against dense FP16
// attention with the whole FP16 cache in VRAM.  This file computes that reference,
// softmax(q K^T / sqrt(D)) V per query head (head h uses KV head h / n_rep), on one GPU.
//
// Design (HBM bound: 512 bytes of K and V per token and KV head, read once):
//  - Persistent CTAs of four consumer warps and one producer warp.  The (sequence x KV
//    head, 64-token block) pairs are numbered group-major and cut into one contiguous
//    range per CTA, so every CTA streams the same number of blocks.
//  - The producer's elected lane streams each block's keys and values (two 64 x 64
//    channel halves of each, 32 KiB) into a three-stage shared-memory ring with tensor
//    memory accelerator copies (128-byte swizzle, so the matrix loads below hit 32
//    distinct banks), completion signalled on a "full" mbarrier per stage; consumer
//    warps release a stage on its "empty" mbarrier.  Every wait is bounded in time.
//  - Consumer warp w owns tokens 16w..16w+15 of each block.  Scores run on the tensor
//    cores transposed, S^T = Q K^T with the query rows as the A operand: rows 0-3 and
//    4-7 both hold the group's four query heads, so the accumulator of lane (gid, tig)
//    holds head gid & 3 at tokens 2tig, 2tig+1, 8+2tig, 9+2tig -- exactly the tokens of
//    the B fragment of the PV product for MMA column gid.  Columns 0-3 take the f16
//    high halves of the softmax weights, columns 4-7 the low halves (weight minus its
//    f16 rounding), so P V = V^T (P_hi + P_lo) is exact to about 2^-22 with no data
//    exchange between lanes.  V^T fragments come from transposing matrix loads.
//  - Each warp keeps an online softmax (running maximum in the base-2 domain, weight
//    sum, 128 x 8 accumulator) per group; when its range leaves a group the four warps
//    merge through shared memory and write one partial (channels, maximum, sum) per head
//    into the caller's workspace.  A second kernel adds a head's partials in a fixed
//    order and writes the FP16 output.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <initializer_list>
#include <mutex>
#include <string>

#include "kvq.h"
#include "kvq_common.cuh"
#include "kvq_launch.h"

namespace kvq {
void set_last_error(const std::string& msg);
}

namespace {

using namespace kvq;

constexpr int DH_STAGES = 3;
constexpr int DH_CONSUMERS = 4;                       // consumer warps (16 tokens each)
constexpr int DH_THREADS = 32 * (DH_CONSUMERS + 1);   // + one producer warp
constexpr int DH_HALF = BLK * 64 * 2;                 // 8 KiB: 64 tokens x 64 channels
constexpr int DH_STAGE_BYTES = 4 * DH_HALF;           // K lo, K hi, V lo, V hi
constexpr int DH_PART = D + 4;                        // floats per (slot, head) partial
constexpr int DH_CTAS_PER_SM = 2;
constexpr unsigned long long DH_WAIT_NS = 2000000000ull;   // bounded waits: 2 s
constexpr size_t DH_SMEM = 1024 /* alignment slack */ + DH_STAGES * DH_STAGE_BYTES + 64 /* barriers */ +
                           16 /* flags */ + DH_CONSUMERS * MAXREP * DH_PART * sizeof(float);

struct DhArgs {
  const __half* q;   // [B][Hq][128]
  __half* out;       // [B][Hq][128]
  float* part;       // [BG][S][MAXREP][DH_PART]
  long long T;       // blocks over all groups: BG * nbt
  int nbt;           // blocks per group, ceil(N / 64)
  int N, B, Hq, Hkv, n_rep, BG, S, grid;
};

// CTA whose block range holds block x (ranges [floor(i T / grid), floor((i + 1) T / grid))).
__host__ __device__ __forceinline__ int cta_of(long long x, long long T, int grid) {
  return (int)(((x + 1) * (long long)grid - 1) / T);
}

__device__ __forceinline__ unsigned long long global_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ bool mbar_try(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok) : "r"(bar), "r"(parity) : "memory");
  return ok != 0;
}

// Wait for phase `parity` of an mbarrier for at most DH_WAIT_NS; false (and the CTA's
// failure flag set) when the time runs out or another thread of the CTA already failed.
__device__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity, volatile int* failed) {
  if (mbar_try(bar, parity)) return true;
  const unsigned long long t0 = global_ns();
  for (;;) {
    if (mbar_try(bar, parity)) return true;
    if (*failed) return false;
    if (global_ns() - t0 > DH_WAIT_NS) {
      *failed = 1;
      return false;
    }
  }
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& d0, uint32_t& d1, uint32_t& d2, uint32_t& d3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(d0), "=r"(d1), "=r"(d2), "=r"(d3) : "r"(addr) : "memory");
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& d0, uint32_t& d1, uint32_t& d2, uint32_t& d3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(d0), "=r"(d1), "=r"(d2), "=r"(d3) : "r"(addr) : "memory");
}

// One 64 x 64 tile of a [BG][N][128] FP16 tensor (coordinates: channel, token, group)
// into shared memory, completing `bytes` on the mbarrier.
__device__ __forceinline__ void tma_tile(uint32_t dst, const CUtensorMap* map, int x, int y, int z,
                                         uint32_t bar, unsigned long long pol) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3, %4}], [%5], %6;"
      :: "r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(bar), "l"(pol)
      : "memory");
}

__global__ void __launch_bounds__(DH_THREADS, DH_CTAS_PER_SM)
    dense_hbm_kernel(const __grid_constant__ CUtensorMap tk, const __grid_constant__ CUtensorMap tv,
                     DhArgs a) {
  extern __shared__ unsigned char dh_raw[];
  const uint32_t raw = (uint32_t)__cvta_generic_to_shared(dh_raw);
  const uint32_t pad = ((raw + 1023u) & ~1023u) - raw;   // swizzled tiles want 1024-byte alignment
  unsigned char* base = dh_raw + pad;
  const uint32_t sbase = raw + pad;
  const uint32_t bar_full = sbase + DH_STAGES * DH_STAGE_BYTES;   // [DH_STAGES] x 8 bytes
  const uint32_t bar_empty = bar_full + 8 * DH_STAGES;
  volatile int* failed = reinterpret_cast<volatile int*>(base + DH_STAGES * DH_STAGE_BYTES + 64);
  float* merge = reinterpret_cast<float*>(base + DH_STAGES * DH_STAGE_BYTES + 64 + 16);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long x0 = (long long)blockIdx.x * a.T / a.grid;
  const long long x1 = (long long)(blockIdx.x + 1) * a.T / a.grid;

  if (threadIdx.x == 0) {
    for (int s = 0; s < DH_STAGES; ++s) {
      asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" :: "r"(bar_full + 8 * s) : "memory");
      asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" :: "r"(bar_empty + 8 * s), "r"(DH_CONSUMERS) : "memory");
    }
    *failed = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  __syncthreads();
  pdl_trigger();

  if (warp == DH_CONSUMERS) {
    // ---- producer: one elected lane streams the CTA's blocks through the ring ----
    if (lane == 0) {
      asm volatile("prefetch.tensormap [%0];" :: "l"(reinterpret_cast<uint64_t>(&tk)) : "memory");
      asm volatile("prefetch.tensormap [%0];" :: "l"(reinterpret_cast<uint64_t>(&tv)) : "memory");
      const unsigned long long pol = evict_first_policy();
      int it = 0;
      for (long long x = x0; x < x1; ++x, ++it) {
        const int s = it % DH_STAGES;
        if (it >= DH_STAGES && !mbar_wait_bounded(bar_empty + 8 * s, (uint32_t)((it / DH_STAGES) - 1) & 1u, failed))
          break;
        const int bg = (int)(x / a.nbt), blk = (int)(x - (long long)bg * a.nbt);
        const uint32_t st = sbase + s * DH_STAGE_BYTES, fb = bar_full + 8 * s;
        asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" :: "r"(fb), "r"(DH_STAGE_BYTES) : "memory");
        tma_tile(st, &tk, 0, blk * BLK, bg, fb, pol);
        tma_tile(st + DH_HALF, &tk, 64, blk * BLK, bg, fb, pol);
        tma_tile(st + 2 * DH_HALF, &tv, 0, blk * BLK, bg, fb, pol);
        tma_tile(st + 3 * DH_HALF, &tv, 64, blk * BLK, bg, fb, pol);
      }
    }
    return;
  }

  // ---- consumers ----
  const int w = warp;
  const int gid = lane >> 2, tig = lane & 3;
  const int hq = gid & 3;               // head of this lane's score rows
  const bool lo_col = gid >= 4;         // this lane's PV B column takes the low halves
  const int mi = lane >> 3, r8 = lane & 7;   // matrix-load role: matrix mi, row r8
  const int tok = 16 * w + 8 * (mi >> 1) + r8;   // token row this lane addresses
  const uint32_t row_off = (uint32_t)tok * 128u;
  const float sc = LOG2E_F * INV_SQRT_D;

  uint32_t qa0[8], qa2[8];
  float acc[8][4];
  float m = -INFINITY, l = 0.f;
  int cur = -1;
  bool bad = false;

  auto flush = [&](int bg) {
    // weight sums over the four lanes of a row group; high + low columns of each head
    float lt = l + __shfl_xor_sync(0xffffffffu, l, 1);
    lt += __shfl_xor_sync(0xffffffffu, lt, 2);
#pragma unroll
    for (int mt = 0; mt < 8; ++mt)
#pragma unroll
      for (int j = 0; j < 4; ++j) acc[mt][j] += __shfl_xor_sync(0xffffffffu, acc[mt][j], 2);
    float* mb = merge + w * (MAXREP * DH_PART);
    if (tig < 2) {
#pragma unroll
      for (int mt = 0; mt < 8; ++mt) {
        const int c0 = 16 * mt + gid;
        mb[(2 * tig) * DH_PART + c0] = acc[mt][0];
        mb[(2 * tig + 1) * DH_PART + c0] = acc[mt][1];
        mb[(2 * tig) * DH_PART + c0 + 8] = acc[mt][2];
        mb[(2 * tig + 1) * DH_PART + c0 + 8] = acc[mt][3];
      }
    }
    if (tig == 0 && gid < 4) {
      mb[gid * DH_PART + D] = bad ? __int_as_float(0x7fc00000) : m;
      mb[gid * DH_PART + D + 1] = lt;
    }
    asm volatile("bar.sync 1, %0;" :: "r"(32 * DH_CONSUMERS) : "memory");
    const int c = threadIdx.x;   // 0..127: one channel per consumer thread
    const int slot = (int)blockIdx.x - cta_of((long long)bg * a.nbt, a.T, a.grid);
    for (int h = 0; h < a.n_rep; ++h) {
      float M = -INFINITY;
#pragma unroll
      for (int ww = 0; ww < DH_CONSUMERS; ++ww) M = fmaxf(M, merge[(ww * MAXREP + h) * DH_PART + D]);
      float L = 0.f, O = 0.f;
#pragma unroll
      for (int ww = 0; ww < DH_CONSUMERS; ++ww) {
        const float* p = merge + (ww * MAXREP + h) * DH_PART;
        const float mw = p[D];
        const float f = (mw == -INFINITY) ? 0.f : exp2_approx(mw - M);
        L = fmaf(p[D + 1], f, L);
        O = fmaf(p[c], f, O);
      }
      float* dst = a.part + (((size_t)bg * a.S + slot) * MAXREP + h) * DH_PART;
      dst[c] = O;
      if (c == 0) {
        dst[D] = M;
        dst[D + 1] = L;
      }
    }
    asm volatile("bar.sync 1, %0;" :: "r"(32 * DH_CONSUMERS) : "memory");
  };

  int it = 0;
  for (long long x = x0; x < x1; ++x, ++it) {
    const int bg = (int)(x / a.nbt), blk = (int)(x - (long long)bg * a.nbt);
    if (bg != cur) {
      if (cur >= 0) flush(cur);
      cur = bg;
      const int b = bg / a.Hkv, g = bg - b * a.Hkv;
      const bool live = hq < a.n_rep;
      const __half* qrow = a.q + ((size_t)b * a.Hq + g * a.n_rep + (live ? hq : 0)) * D;
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        qa0[kk] = live ? *reinterpret_cast<const uint32_t*>(qrow + 16 * kk + 2 * tig) : 0u;
        qa2[kk] = live ? *reinterpret_cast<const uint32_t*>(qrow + 16 * kk + 8 + 2 * tig) : 0u;
      }
#pragma unroll
      for (int mt = 0; mt < 8; ++mt)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[mt][j] = 0.f;
      m = -INFINITY;
      l = 0.f;
    }
    const int s = it % DH_STAGES;
    const bool got = mbar_wait_bounded(bar_full + 8 * s, (uint32_t)(it / DH_STAGES) & 1u, failed);
    const bool ok = __all_sync(0xffffffffu, got);
    bad = bad || !ok;
    const int tbase = blk * BLK + 16 * w;   // first token of this warp's slice
    if (ok && tbase < a.N) {
      const uint32_t st = sbase + s * DH_STAGE_BYTES;
      // scores S^T: rows = heads (twice), columns = 8 tokens per n-tile
      float sacc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        const int chunk = 2 * (kk & 3) + (mi & 1);
        uint32_t d0, d1, d2, d3;
        ldsm_x4(st + (kk >> 2) * DH_HALF + row_off + ((uint32_t)(chunk ^ r8) << 4), d0, d1, d2, d3);
        mma16816(sacc[0], qa0[kk], 0u, qa2[kk], 0u, d0, d1);
        mma16816(sacc[1], qa0[kk], 0u, qa2[kk], 0u, d2, d3);
      }
      float s2[4] = {sacc[0][0] * sc, sacc[0][1] * sc, sacc[1][0] * sc, sacc[1][1] * sc};
      if (tbase + 16 > a.N) {
        const int tt[4] = {2 * tig, 2 * tig + 1, 8 + 2 * tig, 9 + 2 * tig};
#pragma unroll
        for (int j = 0; j < 4; ++j)
          if (tbase + tt[j] >= a.N) s2[j] = -INFINITY;
      }
      float bm = fmaxf(fmaxf(s2[0], s2[1]), fmaxf(s2[2], s2[3]));
      bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, 1));
      bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, 2));
      const float mn = fmaxf(m, bm);            // finite: token tbase is valid
      const float alpha = exp2_approx(m - mn);  // 0 on the group's first slice
      float p[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) p[j] = exp2_approx(s2[j] - mn);
      l = fmaf(l, alpha, (p[0] + p[1]) + (p[2] + p[3]));
      m = mn;
      if (__any_sync(0xffffffffu, alpha != 1.f)) {
        // accumulator columns 2tig, 2tig+1 are heads 2(tig & 1) and 2(tig & 1) + 1
        const float a0 = __shfl_sync(0xffffffffu, alpha, 8 * (tig & 1));
        const float a1 = __shfl_sync(0xffffffffu, alpha, 8 * (tig & 1) + 4);
#pragma unroll
        for (int mt = 0; mt < 8; ++mt) {
          acc[mt][0] *= a0;
          acc[mt][1] *= a1;
          acc[mt][2] *= a0;
          acc[mt][3] *= a1;
        }
      }
      // B fragments of PV: k = tokens (2tig, 2tig+1 | 8+2tig, 9+2tig), column gid
      const __half2 h01 = __floats2half2_rn(p[0], p[1]), h23 = __floats2half2_rn(p[2], p[3]);
      uint32_t b0 = h2_as_u32(h01), b1 = h2_as_u32(h23);
      if (lo_col) {
        const float2 r01 = sub2(make_float2(p[0], p[1]), __half22float2(h01));
        const float2 r23 = sub2(make_float2(p[2], p[3]), __half22float2(h23));
        b0 = h2_as_u32(__floats2half2_rn(r01.x, r01.y));
        b1 = h2_as_u32(__floats2half2_rn(r23.x, r23.y));
      }
      // O^T += V^T P: rows = 16 channels per m-tile, k = the slice's 16 tokens
#pragma unroll
      for (int mt = 0; mt < 8; ++mt) {
        const int chunk = 2 * (mt & 3) + (mi & 1);
        uint32_t v0, v1, v2, v3;
        ldsm_x4_t(st + 2 * DH_HALF + (mt >> 2) * DH_HALF + row_off + ((uint32_t)(chunk ^ r8) << 4), v0, v1, v2, v3);
        mma16816(acc[mt], v0, v1, v2, v3, b0, b1);
      }
    }
    __syncwarp();
    if (lane == 0 && ok) asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" :: "r"(bar_empty + 8 * s) : "memory");
  }
  if (cur >= 0) flush(cur);
}

// One CTA per query head: adds the head's partials in slot order.
__global__ void __launch_bounds__(128) dense_hbm_combine_kernel(DhArgs a) {
  pdl_wait();
  const int bh = blockIdx.x, b = bh / a.Hq, h = bh - b * a.Hq;
  const int g = h / a.n_rep, r = h - g * a.n_rep, bg = b * a.Hkv + g;
  const long long first = (long long)bg * a.nbt;
  const int s0 = cta_of(first, a.T, a.grid), s1 = cta_of(first + a.nbt - 1, a.T, a.grid);
  const int ns = s1 - s0 + 1;
  const float* p = a.part + ((size_t)bg * a.S * MAXREP + r) * DH_PART;
  const int c = threadIdx.x;
  float M = -INFINITY;
  for (int s = 0; s < ns; ++s) M = fmaxf(M, p[(size_t)s * MAXREP * DH_PART + D]);
  float L = 0.f, O = 0.f;
  for (int s = 0; s < ns; ++s) {
    const float* ps = p + (size_t)s * MAXREP * DH_PART;
    const float f = exp2_approx(ps[D] - M);
    L = fmaf(ps[D + 1], f, L);
    O = fmaf(ps[c], f, O);
  }
  a.out[((size_t)b * a.Hq + h) * D + c] = __float2half_rn(O / L);
}

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;
cudaError_t g_encode_err = cudaSuccess;

cudaError_t encode_fn(PFN_cuTensorMapEncodeTiled_v12000* fn) {
  std::call_once(g_encode_once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    g_encode_err = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q);
    if (g_encode_err == cudaSuccess && q != cudaDriverEntryPointSuccess) g_encode_err = cudaErrorNotSupported;
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  *fn = g_encode;
  return g_encode_err;
}

// [BG][N][128] FP16 as a 3-D tensor (channel, token, group), 64 x 64 x 1 boxes, 128-byte swizzle.
bool make_map(CUtensorMap* map, const void* base, int N, int BG, PFN_cuTensorMapEncodeTiled_v12000 enc) {
  const cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)N, (cuuint64_t)BG};
  const cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)N * D * 2};
  const cuuint32_t box[3] = {64, (cuuint32_t)BLK, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

struct DhShape {
  long long T;
  int nbt, BG, grid, S;
};

// Grid and partial slots of a call on the current device.
cudaError_t dh_shape(int batch, int n_kv_heads, int n_tokens, DhShape* sh) {
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  sh->BG = batch * n_kv_heads;
  sh->nbt = (n_tokens + BLK - 1) / BLK;
  sh->T = (long long)sh->BG * sh->nbt;
  long long grid = (long long)std::max(1, sms) * DH_CTAS_PER_SM;
  if (grid > sh->T) grid = sh->T;
  sh->grid = (int)grid;
  int S = 1;
  for (int bg = 0; bg < sh->BG; ++bg) {
    const long long f = (long long)bg * sh->nbt;
    S = std::max(S, cta_of(f + sh->nbt - 1, sh->T, sh->grid) - cta_of(f, sh->T, sh->grid) + 1);
  }
  sh->S = S;
  return cudaSuccess;
}

const char* dh_shape_error(int batch, int n_q_heads, int n_kv_heads, int n_tokens) {
  if (batch < 1 || n_q_heads < 1 || n_kv_heads < 1 || n_tokens < 1)
    return "batch, n_q_heads, n_kv_heads and n_tokens must be >= 1";
  if (n_q_heads % n_kv_heads != 0 || n_q_heads / n_kv_heads > MAXREP)
    return "n_q_heads / n_kv_heads must be an integer in 1..4";
  if ((long long)batch * n_kv_heads > (1ll << 30) || (long long)batch * n_q_heads > (1ll << 30))
    return "batch x heads too large";
  return nullptr;
}

bool on_device(const void* p, int dev) {
  cudaPointerAttributes at;
  if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  if (at.type == cudaMemoryTypeDevice) return at.device == dev;
  return at.type == cudaMemoryTypeManaged;
}

size_t dh_workspace_bytes(const DhShape& sh) {
  return (size_t)sh.BG * sh.S * MAXREP * DH_PART * sizeof(float);
}

}  // namespace

extern "C" kvq_status kvq_dense_attention_workspace(int batch, int n_q_heads, int n_kv_heads, int n_tokens,
                                                    size_t* bytes) {
  if (!bytes) {
    kvq::set_last_error("kvq_dense_attention_workspace: NULL output");
    return KVQ_ERR_INVALID;
  }
  if (const char* msg = dh_shape_error(batch, n_q_heads, n_kv_heads, n_tokens)) {
    kvq::set_last_error(std::string("kvq_dense_attention_workspace: ") + msg);
    return KVQ_ERR_INVALID;
  }
  DhShape sh;
  const cudaError_t e = dh_shape(batch, n_kv_heads, n_tokens, &sh);
  if (e != cudaSuccess) {
    cudaGetLastError();
    kvq::set_last_error(std::string("kvq_dense_attention_workspace: ") + cudaGetErrorString(e));
    return KVQ_ERR_CUDA;
  }
  *bytes = dh_workspace_bytes(sh);
  return KVQ_OK;
}

extern "C" kvq_status kvq_dense_attention(const void* q, const void* k, const void* v, int batch, int n_q_heads,
                                          int n_kv_heads, int n_tokens, void* out, void* workspace,
                                          size_t workspace_bytes, void* stream) {
  if (!q || !k || !v || !out || !workspace) {
    kvq::set_last_error("kvq_dense_attention: NULL buffer");
    return KVQ_ERR_INVALID;
  }
  if (const char* msg = dh_shape_error(batch, n_q_heads, n_kv_heads, n_tokens)) {
    kvq::set_last_error(std::string("kvq_dense_attention: ") + msg);
    return KVQ_ERR_INVALID;
  }
  int cur = 0;
  if (cudaGetDevice(&cur) != cudaSuccess) {
    cudaGetLastError();
    kvq::set_last_error("kvq_dense_attention: no current CUDA device");
    return KVQ_ERR_CUDA;
  }
  for (const void* p : {q, k, v, static_cast<const void*>(out), static_cast<const void*>(workspace)}) {
    if (!on_device(p, cur)) {
      kvq::set_last_error("kvq_dense_attention: q, k, v, out and workspace must be device memory of the "
                          "current device");
      return KVQ_ERR_INVALID;
    }
    if (reinterpret_cast<uintptr_t>(p) % 16 != 0) {
      kvq::set_last_error("kvq_dense_attention: q, k, v, out and workspace must be 16-byte aligned");
      return KVQ_ERR_INVALID;
    }
  }
  DhShape sh;
  cudaError_t e = dh_shape(batch, n_kv_heads, n_tokens, &sh);
  if (e != cudaSuccess) {
    cudaGetLastError();
    kvq::set_last_error(std::string("kvq_dense_attention: ") + cudaGetErrorString(e));
    return KVQ_ERR_CUDA;
  }
  if (workspace_bytes < dh_workspace_bytes(sh)) {
    kvq::set_last_error("kvq_dense_attention: workspace smaller than kvq_dense_attention_workspace reports");
    return KVQ_ERR_INVALID;
  }
  PFN_cuTensorMapEncodeTiled_v12000 enc = nullptr;
  e = encode_fn(&enc);
  if (e != cudaSuccess || !enc) {
    kvq::set_last_error("kvq_dense_attention: the driver's tensor-map encoder is unavailable");
    return KVQ_ERR_CUDA;
  }
  CUtensorMap mk, mv;
  if (!make_map(&mk, k, n_tokens, sh.BG, enc) || !make_map(&mv, v, n_tokens, sh.BG, enc)) {
    kvq::set_last_error("kvq_dense_attention: tensor-map encoding of k or v failed");
    return KVQ_ERR_INVALID;
  }
  DhArgs a;
  a.q = static_cast<const __half*>(q);
  a.out = static_cast<__half*>(out);
  a.part = static_cast<float*>(workspace);
  a.T = sh.T;
  a.nbt = sh.nbt;
  a.N = n_tokens;
  a.B = batch;
  a.Hq = n_q_heads;
  a.Hkv = n_kv_heads;
  a.n_rep = n_q_heads / n_kv_heads;
  a.BG = sh.BG;
  a.S = sh.S;
  a.grid = sh.grid;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  e = cudaFuncSetAttribute(dense_hbm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)DH_SMEM);
  if (e == cudaSuccess) {
    dense_hbm_kernel<<<sh.grid, DH_THREADS, DH_SMEM, st>>>(mk, mv, a);
    e = cudaGetLastError();
  }
  if (e == cudaSuccess) e = launch_dependent(dense_hbm_combine_kernel, dim3(batch * n_q_heads), dim3(D), 0, st, a);
  if (e != cudaSuccess) {
    kvq::set_last_error(std::string("kvq_dense_attention: launch: ") + cudaGetErrorString(e));
    return KVQ_ERR_CUDA;
  }
  return KVQ_OK;
}
