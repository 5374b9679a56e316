// kvq_launch.h -- host-side launchers of the kernels (internal to the library).
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "kvq.h"
#include "kvq_common.cuh"

namespace kvq {

// Pointers of one layer's tier 1 and partial-block buffers, for the append path.
struct LayerAppend {
  int BG, nbmax;
  int8_t* kc; __half* ks; uint8_t* vc; __half2* vsv; float* eta;
  uint32_t* vmin; uint32_t* vmax; uint32_t* kscale_max; uint32_t* vscale_max;
  __half* v16;   // FP16 values of full blocks (value_bits 16), or nullptr
  const __half* tail_k_in; const __half* tail_v_in;
  __half* tail_k_out; __half* tail_v_out;
  unsigned int* counters;   // bounds-check words (KVQ_DEBUG_BOUNDS)
  int debug;
};

cudaError_t launch_append(const LayerAppend& L, const void* k, const void* v, int n, int pos,
                          cudaStream_t st);
cudaError_t launch_export_tier1(const LayerAppend& L, int nb, void* kc, void* ks, void* vc,
                                void* vs, void* vo, float* eta, float* vmin, float* vmax,
                                cudaStream_t st);

// Launch `k` as a programmatic dependent of the previous kernel in `st`: its CTAs may be
// scheduled while that kernel drains and wait in pdl_wait() for its results.
template <typename... P, typename... A>
cudaError_t launch_dependent(void (*k)(P...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                             A&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, k, static_cast<A&&>(args)...);
}

// Decode pipeline (kvq_score.cu, kvq_mixed.cu, kvq_dense.cu).
int score_grid(int num_sms);
int mixed_grid(int num_sms);
int dense_grid(int num_sms);
cudaError_t launch_score(const LayerView& V, int grid, cudaStream_t st);
cudaError_t launch_select(const LayerView& V, cudaStream_t st);
cudaError_t launch_mixed(const LayerView& V, int round, int grid, cudaStream_t st);
cudaError_t launch_combine(const LayerView& V, int round, cudaStream_t st);
int tail_runs(int num_sms, int groups);
cudaError_t launch_tail(const LayerView& V, int runs, int num_sms, cudaStream_t st);
cudaError_t launch_dense(const LayerView& V, int all_dense, int grid, cudaStream_t st);
cudaError_t launch_finalize(const LayerView& V, kvq_certificate* cert, int32_t* level,
                            cudaStream_t st);

// Cross-step residency of FP16 tier-2 blocks (kvq_resident.cu).
cudaError_t launch_residency(const LayerView& V, cudaStream_t st);
cudaError_t launch_residency_init(int* rfree, int* rowner, unsigned int* rstamp, int n, cudaStream_t st);

}  // namespace kvq
