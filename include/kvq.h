/*
 * kvq.h -- C ABI of the certified quantized-KV decode-attention library (GB300, sm_103a).
 *
 * The method is "Runtime-Certified Bounded-Error Quantized Attention" (gist.science
 * technical summary).  Section names used below:
 *   Method §1  tiered storage: tier 1 in VRAM holds per-channel INT8 keys, per-group INT4
 *              values, their scale/offset metadata and a per-block error annotation;
 *              tier 2 keeps the unquantised FP16 keys and values in pinned system RAM as
 *              the ground truth for fallback.
 *   Method §2  two-term error decomposition: E_key bounds the total-variation distortion
 *              of the softmax caused by key quantisation through the per-token score
 *              perturbation Delta; E_val bounds the INT4 value reconstruction error as the
 *              attention-mass-weighted sum of the per-block errors eta_b.  Both come from
 *              quantities already tracked (scales, query norms, value ranges).
 *   Method §3  a light INT8 scoring pass estimates per-block attention mass; the top-K*
 *              blocks covering tau_cov of it get FP16 keys from tier 2; a ranking check
 *              compares INT8 and FP16 block orderings; a four-rung fallback ladder (more
 *              coverage, FP16 values, per-head dense, per-layer dense) follows.
 *   Contributions, "deterministic recovery": when the certified bound cannot be met the
 *              returned output is the dense FP16 attention O_dense.
 *
 * Conventions for every call
 *   - Shapes: B = batch, Hq = query heads, Hkv = KV heads, D = head_dim = 128, blocks of
 *     64 tokens, value groups of 32 channels.  Query head h uses KV head h / (Hq / Hkv).
 *   - FP16 data is IEEE binary16, passed as void*.
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream).  Work is enqueued on
 *     it in stream order; a call returns once its work is enqueued, unless it says
 *     otherwise.  One cache must not be used from two streams at once: every call
 *     reuses the cache's scratch memory.
 *   - Errors: every call returns a kvq_status; kvq_last_error() gives the text of the
 *     calling thread's last failure.  A failed call leaves the cache as it was, except
 *     after KVQ_ERR_CUDA, which reports an error of the CUDA runtime (the context may be
 *     unusable).
 *   - Inputs must be finite.
 */
#ifndef KVQ_H_
#define KVQ_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum kvq_status {
  KVQ_OK = 0,
  KVQ_ERR_INVALID = 1,   /* bad argument, NULL pointer, unsupported shape, empty cache */
  KVQ_ERR_OOM = 2,       /* device memory allocation failed */
  KVQ_ERR_HOST_OOM = 3,  /* pinned host (tier-2) allocation failed */
  KVQ_ERR_CAPACITY = 4,  /* append beyond max_ctx tokens */
  KVQ_ERR_CUDA = 5,      /* a CUDA runtime call failed */
  KVQ_ERR_TIMEOUT = 6    /* reserved for bounded device waits */
} kvq_status;

/* Cache shape and the method's open parameters.  head_dim must be 128, block_tokens 64
 * and value_group 32; n_q_heads / n_kv_heads must be 1, 2, 3 or 4. */
typedef struct kvq_config {
  int n_layers;
  int batch;
  int n_q_heads;
  int n_kv_heads;
  int head_dim;
  int block_tokens;
  int value_group;
  int max_ctx;             /* tokens per sequence and layer, at most 2097152 */
  int rank_positions;      /* ranking check compares the top-R blocks (R >= 1; default 1) */
  float l4_head_fraction;  /* rung 4 when >= this fraction of a sequence's heads are at
                              rung 3 (in (0, 1]; default 0.5) */
  int value_bits;          /* 4 (or 0): INT4 values in VRAM, FP16 values in tier 2 (the
                              paper's configuration).  16: the paper's FP16-values ablation
                              (Results, structured reasoning): values stay FP16 in VRAM,
                              tier 2 holds keys only, E_val = 0 and rung 2 pages nothing
                              in; VRAM per token and KV head 388 B instead of 212 B (dense
                              FP16: 512 B) */
  float v_tol;             /* value tolerance: a head is certified only if also E_val <=
                              v_tol, and rung 2 pages in values until it holds (the paper's
                              v_tol, Results: structured reasoning).  0 (or +inf): no budget
                              beyond eps.  Must not be negative or NaN. */
  int resident_blocks;     /* cross-step residency (not part of the paper: an option of
                              this library).  Each layer may keep up to this many FP16
                              tier-2 blocks (keys or values, 16 KiB each) in device memory
                              across decode calls, so that a block paged in again by a
                              later call is read from HBM instead of over the host link.
                              A block read from tier 2 takes a free slot if one is left;
                              after each certified call the slots its layer did not use in
                              that call are freed.  Outputs and certificates are unchanged
                              (the copies are bit-identical).  Costs resident_blocks x
                              16 KiB of device memory per layer.  0 (the default): none. */
} kvq_config;

/* Per-head certificate of one decode call (Method §2, §3). */
typedef struct kvq_certificate {
  float e_key;             /* bound on the key-quantisation error of the output (max-abs) */
  float e_val;             /* bound on the value-reconstruction error (max-abs) */
  int32_t rank_ok;         /* 1 if the INT8 and FP16 rankings of the selected blocks agree */
  int32_t level;           /* ladder rung reached: 0 certified as is, 1 coverage expanded,
                              2 values promoted, 3 per-head dense, 4 per-layer dense */
  int32_t k_star;          /* blocks selected for this head by the top-K* pass */
  int32_t n_val_promoted;  /* value blocks paged in for the head's certified result */
  int64_t promoted_bytes;  /* FP16 tier-2 bytes paged in for this head's KV group during
                              the call (same for all heads of the group).  With
                              resident_blocks > 0 part of them may come from the resident
                              copies in HBM (kvq_residency_stats) */
} kvq_certificate;

typedef struct kvq_cache kvq_cache;

/* Debug flags for kvq_set_debug. */
#define KVQ_DEBUG_FORCE_RANK_FAIL 0x1  /* every ranking check reports inconsistency */
#define KVQ_DEBUG_FORCE_DENSE     0x2  /* every head takes rung 4 */
#define KVQ_DEBUG_SYNC            0x4  /* synchronise and check after every kernel */
#define KVQ_DEBUG_PROFILE         0x8  /* time every kernel with CUDA events */
#define KVQ_DEBUG_BOUNDS          0x10 /* kernels check the indices they address tier 1, tier 2
                                          and scratch with; the first one out of range is
                                          recorded (the access skipped, nothing traps) and
                                          the call synchronises and returns KVQ_ERR_INVALID
                                          naming the kernel */
#define KVQ_DEBUG_FAIL_MIRROR     0x20 /* test aid: kvq_append's tier-2 mirror copy reports a
                                          CUDA error without being issued; the call returns
                                          KVQ_ERR_CUDA and the cache keeps its length */

/* kvq_cache_create -- allocate tier 1 (device), tier 2 (pinned, mapped host memory) and
 * scratch for `n_layers` layers of `batch` sequences of up to `max_ctx` tokens (Method §1).
 * The library owns all of it until kvq_cache_destroy.  Uses the current CUDA device.
 * Errors: KVQ_ERR_INVALID (cfg NULL or unsupported), KVQ_ERR_OOM, KVQ_ERR_HOST_OOM,
 * KVQ_ERR_CUDA (no usable CUDA device, or initialising tier 1 failed). */
kvq_status kvq_cache_create(const kvq_config* cfg, kvq_cache** out);

/* kvq_cache_destroy -- synchronise the device and free everything.  NULL is a no-op. */
kvq_status kvq_cache_destroy(kvq_cache* cache);

/* kvq_append -- quantise-and-append `n_tokens` new tokens to every sequence of `layer`
 * (Method §1).  k and v are caller-owned device buffers [B, Hkv, n_tokens, D] of FP16,
 * 16-byte aligned.
 * Full 64-token blocks are quantised into tier 1 (INT8 keys with one fp16 scale per
 * block and channel; INT4 values with fp16 scale and offset per token and 32-channel
 * group; eta_b = max |v - v_hat| over the block); the partial last block stays FP16 in
 * VRAM until it fills.  Every token is also mirrored to tier 2 by a copy on an internal
 * side stream that `stream` waits for before any later work, so k and v may be reused
 * by later work on `stream`.  n_tokens = 0 is a no-op.
 * Errors: KVQ_ERR_INVALID (layer out of range, NULL, host or unaligned buffers,
 * n_tokens < 0), KVQ_ERR_CAPACITY (length would exceed max_ctx), KVQ_ERR_CUDA. */
kvq_status kvq_append(kvq_cache* cache, int layer, const void* k, const void* v,
                      int n_tokens, void* stream);

/* kvq_decode_attention -- certified decode attention of one query token per sequence
 * against the cached `layer` (Method §2, §3; deterministic recovery).
 *   q            [B, Hq, D] FP16, device or host memory
 *   tau_cov      coverage target in (0, 1]; tau_cov == 1 takes rung 4 for every head
 *   eps          certificate budget on E_key + E_val (max-abs over the head's output),
 *                eps >= 0; +inf accepts every head whose ranking check passes
 *   out          [B, Hq, D] FP16, device or host memory
 *   cert         [B * Hq] certificates (may be NULL), device or host memory
 *   ladder_level [B] highest rung reached per sequence (may be NULL), device or host
 * Host memory for any of q, out, cert or ladder_level is staged through the cache's own
 * device buffers.  Page-locked host buffers (cudaHostAlloc, cudaHostRegister) are copied
 * in stream order, like cudaMemcpyAsync: q is read when the stream reaches the call, and
 * out, cert and ladder_level hold the results once the stream has completed it.  If any
 * host buffer is pageable, the call synchronises `stream` before returning, so every
 * result is in place on return.  Device buffers are used in
 * place and must be aligned: q and out to 16 bytes, cert to 8, ladder_level to 4.  Tier-2 blocks are read
 * directly by the kernels through the host link (NVLink-C2C); no host round trip
 * happens inside the call.
 * Errors: KVQ_ERR_INVALID (layer out of range, empty layer, tau_cov outside (0, 1],
 * eps < 0 or NaN, NULL q/out, unaligned device buffers), KVQ_ERR_CUDA. */
kvq_status kvq_decode_attention(kvq_cache* cache, int layer, const void* q, float tau_cov,
                                float eps, void* out, kvq_certificate* cert,
                                int32_t* ladder_level, void* stream);

/* kvq_decode_attention_uncertified -- plain quantized decode attention: INT8 key scores
 * and INT4 values on every full block, exact FP16 on the partial block.  No block is
 * paged in from tier 2, no ranking check runs and no rung of the fallback ladder is
 * taken.  This is the uncertified INT8/INT4 baseline that the paper sets against the
 * certified path (Experiments, retrieval), and the speed ceiling of the tier-1 data.
 *   q, out, stream  as kvq_decode_attention
 *   cert            [B * Hq] (may be NULL): e_key and e_val are the bounds of this output,
 *                   computed as in kvq_decode_attention but not enforced; rank_ok 1,
 *                   level 0, k_star 0, n_val_promoted 0, promoted_bytes 0.
 * Debug flags that force rungs are ignored.  The selection state it leaves (nothing
 * selected) is what kvq_export_decode_state reports afterwards.
 * Errors: KVQ_ERR_INVALID (layer out of range, empty layer, NULL q/out, unaligned
 * device buffers), KVQ_ERR_CUDA. */
kvq_status kvq_decode_attention_uncertified(kvq_cache* cache, int layer, const void* q,
                                            void* out, kvq_certificate* cert, void* stream);

/* kvq_last_error -- text of the calling thread's last error ("" if none).  The pointer
 * stays valid until the thread's next failing call. */
const char* kvq_last_error(void);

/* kvq_set_debug -- set KVQ_DEBUG_* flags on the cache (0 clears them). */
kvq_status kvq_set_debug(kvq_cache* cache, int flags);

/* kvq_cache_length -- tokens currently cached for `layer`. */
kvq_status kvq_cache_length(const kvq_cache* cache, int layer, int* n_tokens);

/* kvq_export_tier1 -- copy the tier-1 contents of `layer` into caller device buffers in
 * canonical layout (nb = full blocks of the layer); any pointer may be NULL to skip it:
 *   kc int8 [B, Hkv, nb, 64, D]        ks fp16 [B, Hkv, nb, D]
 *   vc uint8 [B, Hkv, nb, 64, D] (one code 0..15 per byte)
 *   vs fp16 [B, Hkv, nb, 64, D/32]     vo fp16 [B, Hkv, nb, 64, D/32]
 *   eta float [B, Hkv, nb]             vmin, vmax float [B, Hkv, D]
 * Stream-ordered.  Errors: KVQ_ERR_INVALID, KVQ_ERR_CUDA. */
kvq_status kvq_export_tier1(kvq_cache* cache, int layer, void* kc, void* ks, void* vc,
                            void* vs, void* vo, float* eta, float* vmin, float* vmax,
                            void* stream);

/* kvq_export_decode_state -- copy the selection state of the last decode call into caller
 * device buffers (any may be NULL).  nb = full blocks of that call's layer.
 *   sel    uint8 [B, Hq, nb]   1 if the block is in the head's top-K* set S_h
 *   kprom0 uint8 [B, Hkv, nb]  FP16-key blocks of the first pass (union of S_h)
 *   kprom1 uint8 [B, Hkv, nb]  FP16-key blocks after rung 1 (== kprom0 if not run)
 *   vprom1 uint8 [B, Hkv, nb]  FP16-value blocks after rung 2
 *   lse8   float [B, Hq, nb]   INT8 block log-mass;  delta float [B, Hq, nb]  Delta_b
 * Stream-ordered.  Errors: KVQ_ERR_INVALID (no decode yet), KVQ_ERR_CUDA. */
kvq_status kvq_export_decode_state(kvq_cache* cache, uint8_t* sel, uint8_t* kprom0,
                                   uint8_t* kprom1, uint8_t* vprom1, float* lse8,
                                   float* delta, void* stream);

/* Per-kernel timing collected while KVQ_DEBUG_PROFILE is set. */
typedef struct kvq_kernel_stat {
  char name[32];
  int64_t launches;
  double total_ms;
} kvq_kernel_stat;

/* kvq_profile_read -- synchronise the cache's streams and return up to `max` kernel
 * statistics accumulated since the last reset (n = entries written).  reset != 0 clears
 * them afterwards.  Errors: KVQ_ERR_INVALID, KVQ_ERR_CUDA. */
kvq_status kvq_profile_read(kvq_cache* cache, kvq_kernel_stat* stats, int max, int* n,
                            int reset);

/* kvq_residency_stats -- FP16 block traffic of `layer`'s certified decode calls since the
 * last reset (cross-step residency, see kvq_config.resident_blocks): bytes of tier-2
 * blocks served from resident copies in device memory, bytes read over the host link,
 * and the slots currently holding a block.  Any output pointer may be NULL; reset != 0
 * clears the two byte counters.  Synchronises the device.
 * Errors: KVQ_ERR_INVALID (NULL cache, layer out of range), KVQ_ERR_CUDA. */
kvq_status kvq_residency_stats(kvq_cache* cache, int layer, int64_t* resident_bytes,
                               int64_t* host_bytes, int32_t* slots_in_use, int reset);

/* kvq_debug_fill_tier2 -- a test aid, not part of the paper: waits for the device, then
 * overwrites every FP16 element of `layer`'s tier 2 (the keys, and the values when they
 * live there) with the binary16 bit pattern `bits`.  Calls that page blocks in from
 * tier 2 afterwards see the pattern, so a test can show which passes never read it.
 * Errors: KVQ_ERR_INVALID (NULL cache, layer out of range), KVQ_ERR_CUDA. */
kvq_status kvq_debug_fill_tier2(kvq_cache* cache, int layer, uint16_t bits);

/* kvq_dense_attention_workspace -- device workspace bytes that kvq_dense_attention needs
 * for this shape on the current device (it depends on the device's SM count).
 * Errors: KVQ_ERR_INVALID (NULL bytes, bad shape), KVQ_ERR_CUDA. */
kvq_status kvq_dense_attention_workspace(int batch, int n_q_heads, int n_kv_heads, int n_tokens,
                                         size_t* bytes);

/* kvq_dense_attention -- exact dense FP16 decode attention, softmax(q K^T / sqrt(D)) V,
 * over keys and values held in device memory.  This is the dense FP16 attention that
 * Method §1 names as the ground truth and that Results (performance overhead) sets the
 * certified step against; the library uses it as that baseline on the same GPU.
 *   q         [B, Hq, D] FP16, device;  k, v [B, Hkv, n_tokens, D] FP16, device
 *   out       [B, Hq, D] FP16, device (caller-owned)
 *   workspace device buffer of at least kvq_dense_attention_workspace(...) bytes,
 *             caller-owned; its contents need no initialisation and are overwritten
 *   Hq / Hkv in 1..4, n_tokens >= 1; q, k, v, out and workspace 16-byte aligned and on
 *   the current device.
 * Two kernels on `stream`: a split pass that streams every key and value once from HBM
 * and a fixed-order combine.  Every device-side wait of the split pass is bounded (2 s);
 * a wait that runs out, which does not happen in correct operation, makes the affected
 * heads' outputs NaN.  Calls that share a workspace must not overlap on the GPU.
 * Stream-ordered.  Errors: KVQ_ERR_INVALID (NULL, host, unaligned or other-device
 * pointers, bad shape, workspace too small), KVQ_ERR_CUDA. */
kvq_status kvq_dense_attention(const void* q, const void* k, const void* v, int batch, int n_q_heads,
                               int n_kv_heads, int n_tokens, void* out, void* workspace,
                               size_t workspace_bytes, void* stream);

/* kvq_dense_decode_noalloc -- exact dense FP16 decode attention that allocates no memory.
 * The paper has no counterpart to this call.  It is for callers that cannot allocate
 * device memory when they call: a process whose device memory is fully held by another
 * framework's pool, an embedding that owns only fixed buffers, or a step that must not
 * fail on allocation.  It computes softmax(q K^T / sqrt(D)) V -- the same dense attention
 * as the ladder's rungs 3-4 -- over caller-owned FP16 keys and values, keeping its
 * split-K partials and counters in one static 8 MiB device array instead of calling
 * cudaMalloc, cudaFree or any allocating routine.
 *   q   [B, Hq, D] FP16, device;  k, v [B, Hkv, n_tokens, D] FP16, device
 *   out [B, Hq, D] FP16, device (caller-owned);  Hq / Hkv in 1..4, n_tokens >= 1
 *   q, k, v and out 16-byte aligned
 * Size limit: B * Hkv * ceil(n_tokens / 1024) * 2112 bytes of partials (plus a few
 * counters) must fit in the 8 MiB array, e.g. B * Hkv = 8 with up to 507904 tokens.
 * The array exists once per device that loads the library and is held until the
 * process exits.  Every call, with the device current, looks up the array's device
 * address (no allocation); make the first call on a device before any stream capture.
 * With the CUDA driver's lazy loading that first call is also when the library's device
 * code, and with it the 8 MiB array, is loaded onto the device: make it while 8 MiB of
 * device memory are still free (before another pool takes the rest), or it fails with
 * KVQ_ERR_CUDA.  After a cudaDeviceReset the next call loads the array again.
 * Every call shares the array and clears the counters it needs itself; calls whose work
 * overlaps on the GPU (other streams, other host threads) race on it and must be
 * serialised.  The kernel runs on the current device, on `stream`.
 * Stream-ordered.  Errors: KVQ_ERR_INVALID (NULL, host, unaligned or other-device
 * pointers, bad shape), KVQ_ERR_CAPACITY (beyond the size limit), KVQ_ERR_CUDA. */
kvq_status kvq_dense_decode_noalloc(const void* q, const void* k, const void* v, int batch,
                                    int n_q_heads, int n_kv_heads, int n_tokens, void* out,
                                    void* stream);

#ifdef __cplusplus
}
#endif

#endif /* KVQ_H_ */
