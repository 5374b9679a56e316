// kvq_resident.cuh -- cross-step residency of FP16 tier-2 blocks in HBM (device side).
//
// An option of this library, not a step of the paper's method: each layer may keep up
// to `nres` FP16 blocks (keys or values, 16 KiB each) that earlier decode calls paged in
// from tier 2, so that a later call reads them from HBM instead of over the host link.
// The copies are bit-identical to tier 2, so outputs and certificates do not change.
//
// Per FP16 block a CTA (128 threads) is about to read, thread 0 looks the block up in
// the layer's slot table; on a hit the CTA reads the slot, on a miss it reads tier 2 and,
// while a free slot is left, copies the block into it as it goes (claims pop the free
// stack from the top).  Slot use is stamped with the layer's call number; after each
// certified call an eviction pass frees the slots that call did not use and pushes them
// back onto the stack.  Which slot a block lands in depends on timing; which blocks are
// resident, and every output, does not.
#pragma once

#include "kvq_common.cuh"

namespace kvq {

struct ResPick {
  int slot;    // slot holding the block (read it from HBM), or -1
  int admit;   // on a miss: free slot to fill with the block, or -1
};

// Where this CTA reads FP16 block (kv: 0 keys, 1 values) of table entry `bi` =
// hs * nbmax + blk from.  Thread 0 decides and broadcasts through `sh` (two ints of
// shared memory that no other pick of the same CTA uses before a later barrier); one
// __syncthreads.  With residency off: {-1, -1} and no barrier.
__device__ __forceinline__ ResPick res_pick(const LayerView& V, int kv, size_t bi, int* sh) {
  if (V.nres == 0) return {-1, -1};
  if (threadIdx.x == 0) {
    const int s = (kv ? V.rslot_v : V.rslot_k)[bi];
    int adm = -1;
    if (s >= 0) {
      V.rstamp[s] = V.call_id;
      atomicAdd(&V.rbytes[0], (unsigned long long)F16_BLOCK_BYTES);
    } else {
      const unsigned int t = atomicAdd(&V.rstate[RS_TAKEN], 1u);
      const unsigned int nfree = V.rstate[RS_NFREE];   // constant during the call
      if (t < nfree) adm = V.rfree[nfree - 1u - t];
      atomicAdd(&V.rbytes[1], (unsigned long long)F16_BLOCK_BYTES);
    }
    sh[0] = s;
    sh[1] = adm;
  }
  __syncthreads();
  return {sh[0], sh[1]};
}

// Source address of the block: its slot, or `tier2`.
__device__ __forceinline__ const __half* res_src(const LayerView& V, const ResPick& p, const __half* tier2) {
  return p.slot >= 0 ? V.rpool + (size_t)p.slot * (BLK * D) : tier2;
}

// Destination of the copy a missed block makes on its way in (nullptr: none).
__device__ __forceinline__ __half* res_dst(const LayerView& V, const ResPick& p) {
  return p.admit >= 0 ? V.rpool + (size_t)p.admit * (BLK * D) : nullptr;
}

// Record the filled slot.  The copy is visible to the later kernels of this call and to
// later calls (kernel boundaries order it); no kernel reads a block it admits itself.
__device__ __forceinline__ void res_commit(const LayerView& V, int kv, size_t bi, const ResPick& p) {
  if (threadIdx.x == 0 && p.admit >= 0) {
    V.rowner[p.admit] = (kv << 30) | (int)bi;
    V.rstamp[p.admit] = V.call_id;
    (kv ? V.rslot_v : V.rslot_k)[bi] = p.admit;
  }
}

}  // namespace kvq
