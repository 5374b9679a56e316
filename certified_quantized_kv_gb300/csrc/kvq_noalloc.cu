// kvq_noalloc.cu -- exact dense FP16 decode attention that allocates no memory.
//
// The paper has no counterpart to this entry point.  It serves callers that cannot
// allocate device memory at the point of the call: a process whose device memory is
// fully reserved by another framework's pool, an allocator-free embedding that only
// owns fixed buffers, or code that must not fail on allocation mid-step.  It computes
// the same dense attention as the ladder's dense rungs (split-K over 16-block chunks,
// online softmax per chunk, fixed-order combine), but over caller-owned FP16 keys and
// values, and keeps its split-K partials and work counters in one file-scope device
// array of NOALLOC_SCRATCH_BYTES instead of memory from cudaMalloc.
//
// The array is shared by every call on a device and keeps the previous call's
// contents; each call clears the counters it needs before its kernel runs.  Calls
// whose kernels overlap on the GPU (two streams, or two host threads) race on the
// array and must be serialised by the caller.
#include <cstdint>
#include <initializer_list>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <string>

#include "kvq.h"
#include "kvq_common.cuh"

namespace kvq {
void set_last_error(const std::string& msg);
}

namespace {

using namespace kvq;

constexpr size_t NOALLOC_SCRATCH_BYTES = 8u << 20;   // 8 MiB per device
constexpr int NA_CHUNK = 16;                           // blocks per work item
constexpr int NA_PART = MAXREP * (D + 4);              // floats per (group, chunk) partial

static __device__ __align__(256) unsigned char g_noalloc_scratch[NOALLOC_SCRATCH_BYTES];


struct NaArgs {
  const __half* q;    // [B][Hq][128]
  const __half* k;    // [B][Hkv][N][128]
  const __half* v;
  __half* out;        // [B][Hq][128]
  int B, Hq, Hkv, n_rep, BG, N, nch;
  unsigned int* cnt;  // [2 + BG]: work queue, exit count, per-group completion
  float* part;        // [BG][nch][MAXREP][D + 4]
};

struct __align__(16) NaSmem {
  __half kbuf[BLK][D + 8];
  __half vbuf[BLK][D];
  float qf[MAXREP][D];
  float s[MAXREP][BLK];
  float red[MAXREP][2];
  int item;
  int is_last;
};

__global__ void __launch_bounds__(128) noalloc_dense_kernel(NaArgs a) {
  __shared__ NaSmem sm;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int total = a.BG * a.nch;
  int cur_hs = -1;
  for (;;) {
    if (tid == 0) sm.item = (int)atomicAdd(&a.cnt[0], 1u);
    __syncthreads();
    const int item = sm.item;
    if (item >= total) break;
    const int hs = item / a.nch, ch = item % a.nch;
    const int b = hs / a.Hkv, g = hs % a.Hkv;
    if (hs != cur_hs) {
      cur_hs = hs;
      for (int i = tid; i < MAXREP * D; i += blockDim.x) {
        const int r = i / D, c = i % D;
        sm.qf[r][c] = (r < a.n_rep) ? __half2float(a.q[((size_t)b * a.Hq + g * a.n_rep + r) * D + c]) : 0.f;
      }
      __syncthreads();
    }
    float m[MAXREP], l[MAXREP], acc[MAXREP];
    for (int r = 0; r < MAXREP; ++r) { m[r] = -INFINITY; l[r] = 0.f; acc[r] = 0.f; }
    const int t_begin = ch * NA_CHUNK * BLK;
    const int t_end = min(a.N, t_begin + NA_CHUNK * BLK);
    for (int t0 = t_begin; t0 < t_end; t0 += BLK) {
      const int nvalid = min(BLK, t_end - t0);
      for (int i = tid; i < BLK * D / 8; i += blockDim.x) {
        const int row = i >> 4, col = (i & 15) * 8;
        uint4 kv = make_uint4(0, 0, 0, 0), vv = make_uint4(0, 0, 0, 0);
        if (row < nvalid) {
          const size_t o = ((size_t)hs * a.N + t0 + row) * D + col;
          kv = *reinterpret_cast<const uint4*>(a.k + o);
          vv = *reinterpret_cast<const uint4*>(a.v + o);
        }
        *reinterpret_cast<uint4*>(&sm.kbuf[row][col]) = kv;
        *reinterpret_cast<uint4*>(&sm.vbuf[row][col]) = vv;
      }
      __syncthreads();
      {
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
        sm.s[rp][t] = (t < nvalid) ? s0 * INV_SQRT_D : -INFINITY;
        sm.s[rp + 1][t] = (t < nvalid) ? s1 * INV_SQRT_D : -INFINITY;
      }
      __syncthreads();
      {
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
      for (int r = 0; r < a.n_rep; ++r) {
        const float mn = sm.red[r][0];
        const float sc = (m[r] == -INFINITY) ? 0.f : expf(m[r] - mn);
        float as = 0.f;
        for (int t = 0; t < BLK; ++t) as = fmaf(sm.s[r][t], __half2float(sm.vbuf[t][tid]), as);
        l[r] = l[r] * sc + sm.red[r][1];
        acc[r] = acc[r] * sc + as;
        m[r] = mn;
      }
      __syncthreads();
    }
    float* pp = a.part + ((size_t)hs * a.nch + ch) * NA_PART;
    for (int r = 0; r < a.n_rep; ++r) {
      pp[r * (D + 4) + tid] = acc[r];
      if (tid == 0) {
        pp[r * (D + 4) + D] = m[r];
        pp[r * (D + 4) + D + 1] = l[r];
      }
    }
    __syncthreads();
    if (tid == 0) {
      __threadfence();
      const unsigned int old = atomicAdd(&a.cnt[2 + hs], 1u);
      sm.is_last = (old == (unsigned int)(a.nch - 1));
    }
    __syncthreads();
    if (sm.is_last) {
      __threadfence();
      for (int r = 0; r < a.n_rep; ++r) {
        float M = -INFINITY;
        for (int c = 0; c < a.nch; ++c) M = fmaxf(M, a.part[((size_t)hs * a.nch + c) * NA_PART + r * (D + 4) + D]);
        float L = 0.f, o = 0.f;
        for (int c = 0; c < a.nch; ++c) {
          const float* q = a.part + ((size_t)hs * a.nch + c) * NA_PART + r * (D + 4);
          const float w = expf(q[D] - M);
          L += q[D + 1] * w;
          o += q[tid] * w;
        }
        a.out[((size_t)b * a.Hq + g * a.n_rep + r) * D + tid] = __float2half_rn(o / L);
      }
    }
    __syncthreads();
  }
}

// Device address of this device's scratch array, looked up on every call (the lookup is
// cheap and allocates nothing; the first one on a device also makes the driver load this
// library's device code there, which is when the array's memory is reserved).  Looking
// it up each time keeps the address right if the device code was loaded again.
cudaError_t scratch_for_current_device(void** out) {
  void* p = nullptr;
  const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
  if (e != cudaSuccess) return e;
  *out = p;
  return cudaSuccess;
}

// Device (or managed) memory of device `dev`: the kernel runs on the current device, so a
// buffer of another device would be read through a foreign address.
bool on_device(const void* p, int dev) {
  cudaPointerAttributes at;
  if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  if (at.type == cudaMemoryTypeDevice) return at.device == dev;
  return at.type == cudaMemoryTypeManaged;
}

}  // namespace

extern "C" kvq_status kvq_dense_decode_noalloc(const void* q, const void* k, const void* v,
                                               int batch, int n_q_heads, int n_kv_heads,
                                               int n_tokens, void* out, void* stream) {
  if (!q || !k || !v || !out) {
    kvq::set_last_error("kvq_dense_decode_noalloc: NULL buffer");
    return KVQ_ERR_INVALID;
  }
  if (batch < 1 || n_kv_heads < 1 || n_q_heads < 1 || n_tokens < 1 || n_q_heads % n_kv_heads != 0 ||
      n_q_heads / n_kv_heads > MAXREP) {
    kvq::set_last_error("kvq_dense_decode_noalloc: need batch, heads, n_tokens >= 1 and "
                        "n_q_heads / n_kv_heads an integer in 1..4");
    return KVQ_ERR_INVALID;
  }
  int cur = 0;
  if (cudaGetDevice(&cur) != cudaSuccess) {
    cudaGetLastError();
    kvq::set_last_error("kvq_dense_decode_noalloc: no current CUDA device");
    return KVQ_ERR_CUDA;
  }
  if (!on_device(q, cur) || !on_device(k, cur) || !on_device(v, cur) || !on_device(out, cur)) {
    kvq::set_last_error("kvq_dense_decode_noalloc: q, k, v and out must be device memory of the "
                        "current device");
    return KVQ_ERR_INVALID;
  }
  for (const void* p : {q, k, v, static_cast<const void*>(out)}) {
    if (reinterpret_cast<uintptr_t>(p) % 16 != 0) {   // 16-byte vector accesses
      kvq::set_last_error("kvq_dense_decode_noalloc: q, k, v and out must be 16-byte aligned");
      return KVQ_ERR_INVALID;
    }
  }
  const int BG = batch * n_kv_heads;
  const int nch = (n_tokens + NA_CHUNK * BLK - 1) / (NA_CHUNK * BLK);
  const size_t cnt_bytes = ((size_t)(2 + BG) * sizeof(unsigned int) + 255) / 256 * 256;
  const size_t need = cnt_bytes + (size_t)BG * nch * NA_PART * sizeof(float);
  if (need > NOALLOC_SCRATCH_BYTES) {
    kvq::set_last_error("kvq_dense_decode_noalloc: batch * n_kv_heads * ceil(n_tokens / 1024) "
                        "partials exceed the fixed 8 MiB device scratch");
    return KVQ_ERR_CAPACITY;
  }
  void* base = nullptr;
  cudaError_t e = scratch_for_current_device(&base);
  if (e != cudaSuccess) {
    kvq::set_last_error(std::string("kvq_dense_decode_noalloc: scratch lookup: ") + cudaGetErrorString(e));
    return KVQ_ERR_CUDA;
  }
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  e = cudaMemsetAsync(base, 0, cnt_bytes, st);
  if (e != cudaSuccess) {
    kvq::set_last_error(std::string("kvq_dense_decode_noalloc: clear: ") + cudaGetErrorString(e));
    return KVQ_ERR_CUDA;
  }
  NaArgs a;
  a.q = static_cast<const __half*>(q);
  a.k = static_cast<const __half*>(k);
  a.v = static_cast<const __half*>(v);
  a.out = static_cast<__half*>(out);
  a.B = batch; a.Hq = n_q_heads; a.Hkv = n_kv_heads; a.n_rep = n_q_heads / n_kv_heads;
  a.BG = BG; a.N = n_tokens; a.nch = nch;
  a.cnt = static_cast<unsigned int*>(base);
  a.part = reinterpret_cast<float*>(static_cast<char*>(base) + cnt_bytes);
  int sms = 0;
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, cur);
  const int grid = std::min(BG * nch, std::max(1, sms) * 3);
  noalloc_dense_kernel<<<grid, 128, 0, st>>>(a);
  e = cudaGetLastError();
  if (e != cudaSuccess) {
    kvq::set_last_error(std::string("kvq_dense_decode_noalloc: launch: ") + cudaGetErrorString(e));
    return KVQ_ERR_CUDA;
  }
  return KVQ_OK;
}
