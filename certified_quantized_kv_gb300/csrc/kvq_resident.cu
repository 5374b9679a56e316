// kvq_resident.cu -- eviction pass of the cross-step residency of FP16 tier-2 blocks
// (an option of this library, not of the paper; see kvq_resident.cuh).
//
// After a certified decode call of a layer, one thread per slot: a slot whose block
// that call did not use is freed (its table entry cleared) and pushed onto the free
// stack above the entries no claim of the call reached; the last CTA to finish
// publishes the new stack height and clears the claim counter.
#include <algorithm>

#include "kvq_common.cuh"
#include "kvq_launch.h"

namespace kvq {

constexpr int RES_THREADS = 256;

__global__ void __launch_bounds__(RES_THREADS) residency_kernel(LayerView V) {
  pdl_wait();   // every use of this call has been stamped
  __shared__ bool last;
  const unsigned int nfree = V.rstate[RS_NFREE], taken = V.rstate[RS_TAKEN];
  const unsigned int base = nfree - min(taken, nfree);   // unclaimed entries stay at the bottom
  const int s = blockIdx.x * RES_THREADS + threadIdx.x;
  if (s < V.nres) {
    const int own = V.rowner[s];
    if (own >= 0 && V.rstamp[s] != V.call_id) {
      ((own >> 30) ? V.rslot_v : V.rslot_k)[own & 0x3fffffff] = -1;
      V.rowner[s] = -1;
      V.rfree[base + atomicAdd(&V.rstate[RS_PUSHED], 1u)] = s;
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    last = atomicAdd(&V.rstate[RS_DONE], 1u) == gridDim.x - 1;
  }
  __syncthreads();
  if (last && threadIdx.x == 0) {
    __threadfence();
    const unsigned int n = base + atomicAdd(&V.rstate[RS_PUSHED], 0u);
    V.rstate[RS_NFREE] = n;
    V.rstate[RS_TAKEN] = 0u;
    V.rstate[RS_USED] = (unsigned int)V.nres - n;
    V.rstate[RS_PUSHED] = 0u;
    V.rstate[RS_DONE] = 0u;
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
  return launch_dependent(residency_kernel, dim3((V.nres + RES_THREADS - 1) / RES_THREADS),
                          dim3(RES_THREADS), 0, st, V);
}

cudaError_t launch_residency_init(int* rfree, int* rowner, unsigned int* rstamp, int n, cudaStream_t st) {
  if (n == 0) return cudaSuccess;
  residency_init_kernel<<<std::min(64, (n + 255) / 256), 256, 0, st>>>(rfree, rowner, rstamp, n);
  return cudaGetLastError();
}

}  // namespace kvq
