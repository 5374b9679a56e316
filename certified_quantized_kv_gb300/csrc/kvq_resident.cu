// kvq_resident.cu -- eviction pass of the cross-step residency of FP16 tier-2 blocks
// (an option of this library, not of the paper; see kvq_resident.cuh).
//
// After a certified decode call of a layer: every slot whose block that call did not
// use is freed (its table entry cleared), and the free list is rebuilt in ascending slot
// order, so the next call claims slots deterministically.  One CTA of 1024 threads.
#include <algorithm>

#include "kvq_common.cuh"
#include "kvq_launch.h"

namespace kvq {

__global__ void __launch_bounds__(1024) residency_kernel(LayerView V) {
  pdl_wait();   // every use of this call has been stamped
  __shared__ int wcount[32];
  __shared__ int chunk_total;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  int base = 0;
  for (int s0 = 0; s0 < V.nres; s0 += 1024) {
    const int s = s0 + tid;
    bool fr = false;
    if (s < V.nres) {
      const int own = V.rowner[s];
      const bool keep = own >= 0 && V.rstamp[s] == V.call_id;
      if (own >= 0 && !keep) {
        ((own >> 30) ? V.rslot_v : V.rslot_k)[own & 0x3fffffff] = -1;
        V.rowner[s] = -1;
      }
      fr = !keep;
    }
    const unsigned int m = __ballot_sync(0xffffffffu, fr);
    if (lane == 0) wcount[warp] = __popc(m);
    __syncthreads();
    if (warp == 0) {   // exclusive scan of the 32 warp counts
      const int v = wcount[lane];
      int x = v;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
      }
      wcount[lane] = x - v;
      if (lane == 31) chunk_total = x;
    }
    __syncthreads();
    if (fr) V.rfree[base + wcount[warp] + __popc(m & ((1u << lane) - 1u))] = s;
    base += chunk_total;
    __syncthreads();
  }
  if (tid == 0) {
    V.rstate[RS_NFREE] = (unsigned int)base;
    V.rstate[RS_TAKEN] = 0u;
    V.rstate[RS_USED] = (unsigned int)(V.nres - base);
  }
}

// Initial state: every slot free, in order.
__global__ void residency_init_kernel(int* rfree, int* rowner, unsigned int* rstamp, int n) {
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) {
    rfree[i] = i;
    rowner[i] = -1;
    rstamp[i] = 0u;
  }
}

cudaError_t launch_residency(const LayerView& V, cudaStream_t st) {
  if (V.nres == 0) return cudaSuccess;
  return launch_dependent(residency_kernel, dim3(1), dim3(1024), 0, st, V);
}

cudaError_t launch_residency_init(int* rfree, int* rowner, unsigned int* rstamp, int n, cudaStream_t st) {
  if (n == 0) return cudaSuccess;
  residency_init_kernel<<<std::min(64, (n + 255) / 256), 256, 0, st>>>(rfree, rowner, rstamp, n);
  return cudaGetLastError();
}

}  // namespace kvq
