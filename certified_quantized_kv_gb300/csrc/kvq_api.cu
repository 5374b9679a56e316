// kvq_api.cu -- the C ABI (include/kvq.h): cache lifetime, append, certified decode,
// exports for tests, per-kernel timing.
//
// Orchestration of one decode call ("Runtime-Certified Bounded-Error Quantized
// Attention", gist.science technical summary, Method §1-§3): the INT8 scoring pass, the
// top-K* selection, the mixed-precision pass and its combine (certificate and ladder
// plan), a second mixed pass and combine for groups that asked for rungs 1-2, the dense
// rungs 3-4 and the certificate write-out -- eight stream-ordered launches (a ninth, the
// eviction pass, with cross-step residency) with no host round trip; every
// data-dependent decision is taken on the device.
#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>

#include <algorithm>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <cstdint>
#include <string>
#include <vector>

#include "kvq.h"
#include "kvq_common.cuh"
#include "kvq_launch.h"

using namespace kvq;

namespace {

thread_local std::string g_err;

kvq_status fail(kvq_status s, const std::string& msg) {
  g_err = msg;
  return s;
}
kvq_status cuda_fail(cudaError_t e, const char* where) {
  g_err = std::string(where) + ": " + cudaGetErrorString(e);
  return KVQ_ERR_CUDA;
}

#define KVQ_CUDA(call, where)                      \
  do {                                             \
    cudaError_t e_ = (call);                       \
    if (e_ != cudaSuccess) return cuda_fail(e_, where); \
  } while (0)

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Names of the kernels that record bounds violations (BoundsSite order).
const char* kBoundsSites[SITE_COUNT] = {"", "score", "select", "mixed_round0",
                                        "mixed (second pass or FP16 values)", "combine",
                                        "int4_tail", "dense_fallback", "finalize",
                                        "quantize_append"};

bool aligned(const void* p, size_t a) { return reinterpret_cast<uintptr_t>(p) % a == 0; }

__global__ void fill_u32(uint32_t* p, uint32_t v, size_t n) {
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x) p[i] = v;
}

enum KernelId { K_SCORE = 0, K_SELECT, K_MIX0, K_COMB0, K_MIX1, K_COMB1, K_DENSE, K_FINAL,
                K_APPEND, K_TAIL, K_RESIDENT, K_COUNT };
const char* kKernelNames[K_COUNT] = {"score", "select", "mixed_round0", "combine_round0",
                                     "mixed_round1", "combine_round1", "dense_fallback",
                                     "finalize", "quantize_append", "int4_tail", "residency"};

}  // namespace

namespace kvq {
// Lets other translation units of the library report through kvq_last_error().
void set_last_error(const std::string& msg) { g_err = msg; }
}  // namespace kvq

struct kvq_cache {
  kvq_config cfg;
  int device = 0, num_sms = 0;
  int nslot = 0;      // partial slots per KV group of the split-K passes
  int B = 0, Hq = 0, Hkv = 0, n_rep = 0, BG = 0, nbmax = 0, nbmax_used = 0, L = 0;
  long long cap = 0;  // tier-2 tokens per (sequence, KV head)
  std::vector<int> n_tokens;
  std::vector<int> tail_parity;
  // tier 1, all layers in one allocation
  char* t1 = nullptr;
  size_t off_kc = 0, off_ks = 0, off_vc = 0, off_vsv = 0, off_eta = 0, off_vmin = 0, off_vmax = 0,
         off_ksm = 0, off_vsm = 0, off_tail = 0, off_v16 = 0, t1_layer = 0;
  bool v16 = false;   // FP16 values in tier 1 (value_bits 16); tier 2 then holds keys only
  // tier 2: pinned, mapped host memory, per layer
  std::vector<__half*> t2k_host, t2v_host;
  std::vector<__half*> t2k_dev, t2v_dev;
  // scratch
  char* scr = nullptr;
  float *shat = nullptr, *lse8 = nullptr, *delta = nullptr, *lse16 = nullptr;
  uint8_t *sel = nullptr, *kprom0 = nullptr, *kprom1 = nullptr, *vprom1 = nullptr;
  HeadState* hst = nullptr;
  GroupState* gst = nullptr;
  float *part = nullptr, *part1 = nullptr, *dpart = nullptr, *red0 = nullptr;
  unsigned int* counters = nullptr;
  __half *q_stage = nullptr, *out_stage = nullptr;
  kvq_certificate* cert_stage = nullptr;
  int32_t* level_stage = nullptr;
  // cross-step residency of FP16 tier-2 blocks, all layers in one allocation
  int nres = 0;
  char* res = nullptr;
  size_t res_layer = 0, off_rk = 0, off_rv = 0, off_rown = 0, off_rstamp = 0, off_rfree = 0,
         off_rstate = 0, off_rbytes = 0, off_rpool = 0;
  std::vector<unsigned int> call_id;   // certified decode calls per layer
  cudaStream_t side = nullptr;
  cudaEvent_t ev_in = nullptr, ev_mirror = nullptr;
  int debug = 0;
  int last_layer = -1, last_nb = 0;
  // profiling
  struct Rec { int id; cudaEvent_t a, b; };
  std::vector<Rec> recs;
  std::vector<cudaEvent_t> ev_pool;
  double prof_ms[K_COUNT] = {0};
  long long prof_n[K_COUNT] = {0};
};

namespace {

int8_t* layer_kc(kvq_cache* c, int l) { return reinterpret_cast<int8_t*>(c->t1 + c->t1_layer * l + c->off_kc); }
__half* layer_ks(kvq_cache* c, int l) { return reinterpret_cast<__half*>(c->t1 + c->t1_layer * l + c->off_ks); }
uint8_t* layer_vc(kvq_cache* c, int l) { return reinterpret_cast<uint8_t*>(c->t1 + c->t1_layer * l + c->off_vc); }
__half2* layer_vsv(kvq_cache* c, int l) { return reinterpret_cast<__half2*>(c->t1 + c->t1_layer * l + c->off_vsv); }
float* layer_eta(kvq_cache* c, int l) { return reinterpret_cast<float*>(c->t1 + c->t1_layer * l + c->off_eta); }
uint32_t* layer_vmin(kvq_cache* c, int l) { return reinterpret_cast<uint32_t*>(c->t1 + c->t1_layer * l + c->off_vmin); }
uint32_t* layer_vmax(kvq_cache* c, int l) { return reinterpret_cast<uint32_t*>(c->t1 + c->t1_layer * l + c->off_vmax); }
uint32_t* layer_ksm(kvq_cache* c, int l) { return reinterpret_cast<uint32_t*>(c->t1 + c->t1_layer * l + c->off_ksm); }
uint32_t* layer_vsm(kvq_cache* c, int l) { return reinterpret_cast<uint32_t*>(c->t1 + c->t1_layer * l + c->off_vsm); }
__half* layer_v16(kvq_cache* c, int l) {
  return c->v16 ? reinterpret_cast<__half*>(c->t1 + c->t1_layer * l + c->off_v16) : nullptr;
}
// partial-block buffers: [parity][K|V][BG][64][128]
__half* layer_tail(kvq_cache* c, int l, int parity, int kv) {
  __half* base = reinterpret_cast<__half*>(c->t1 + c->t1_layer * l + c->off_tail);
  return base + ((size_t)(parity * 2 + kv) * c->BG) * BLK * D;
}

LayerAppend append_view(kvq_cache* c, int l) {
  LayerAppend a;
  a.BG = c->BG;
  a.nbmax = c->nbmax;
  a.kc = layer_kc(c, l); a.ks = layer_ks(c, l); a.vc = layer_vc(c, l); a.vsv = layer_vsv(c, l);
  a.eta = layer_eta(c, l); a.vmin = layer_vmin(c, l); a.vmax = layer_vmax(c, l);
  a.kscale_max = layer_ksm(c, l); a.vscale_max = layer_vsm(c, l);
  a.v16 = layer_v16(c, l);
  const int p = c->tail_parity[l];
  a.tail_k_in = layer_tail(c, l, p, 0); a.tail_v_in = layer_tail(c, l, p, 1);
  a.tail_k_out = layer_tail(c, l, 1 - p, 0); a.tail_v_out = layer_tail(c, l, 1 - p, 1);
  a.counters = c->counters;
  a.debug = c->debug;
  return a;
}

// KVQ_DEBUG_BOUNDS: the two bounds words are cleared before a call's kernels and read
// (after a synchronise) once they have run; a recorded site fails the call.
kvq_status bounds_clear(kvq_cache* c, cudaStream_t st) {
  if (!(c->debug & KVQ_DEBUG_BOUNDS)) return KVQ_OK;
  KVQ_CUDA(cudaMemsetAsync(c->counters + CNT_BOUNDS, 0, 2 * sizeof(unsigned int), st), "bounds: clear");
  return KVQ_OK;
}
kvq_status bounds_report(kvq_cache* c, cudaStream_t st, const std::string& f) {
  if (!(c->debug & KVQ_DEBUG_BOUNDS)) return KVQ_OK;
  unsigned int w[2] = {0u, 0u};
  KVQ_CUDA(cudaMemcpyAsync(w, c->counters + CNT_BOUNDS, sizeof(w), cudaMemcpyDeviceToHost, st), "bounds: read");
  KVQ_CUDA(cudaStreamSynchronize(st), "bounds: sync");
  if (w[0] == 0u) return KVQ_OK;
  const char* site = w[0] < SITE_COUNT ? kBoundsSites[w[0]] : "unknown kernel";
  return fail(KVQ_ERR_INVALID, f + ": bounds check failed in " + site + " (index " + std::to_string(w[1]) +
                                   " out of range); the access was skipped");
}

bool is_device_ptr(const void* p) {
  cudaPointerAttributes at;
  if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return at.type == cudaMemoryTypeDevice || at.type == cudaMemoryTypeManaged;
}

// Page-locked host memory (cudaHostAlloc, cudaHostRegister): copies to and from it are
// ordered on the stream without the host waiting.
bool is_pinned_host_ptr(const void* p) {
  cudaPointerAttributes at;
  if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return at.type == cudaMemoryTypeHost;
}

cudaEvent_t pooled_event(kvq_cache* c) {
  if (!c->ev_pool.empty()) {
    cudaEvent_t e = c->ev_pool.back();
    c->ev_pool.pop_back();
    return e;
  }
  cudaEvent_t e;
  cudaEventCreate(&e);
  return e;
}

// Makes the cache's device current for the duration of a call and restores the
// caller's device afterwards (a process may drive caches on several GPUs).
struct DeviceGuard {
  int prev = -1;
  explicit DeviceGuard(int dev) {
    if (cudaGetDevice(&prev) == cudaSuccess && prev != dev) cudaSetDevice(dev);
    else prev = -1;
  }
  ~DeviceGuard() { if (prev >= 0) cudaSetDevice(prev); }
};

// One launch of the pipeline: an NVTX range named after the kernel (visible to any
// attached profiler; a no-op otherwise), CUDA events around it in profiling mode, and a
// synchronising error check in debug-sync mode.
struct KernelScope {
  kvq_cache* c;
  int id;
  cudaStream_t st;
  cudaEvent_t a = nullptr;
  bool open = true;
  KernelScope(kvq_cache* c_, int id_, cudaStream_t st_) : c(c_), id(id_), st(st_) {
    nvtxRangePushA(kKernelNames[id]);
    if (c->debug & KVQ_DEBUG_PROFILE) {
      a = pooled_event(c);
      cudaEventRecord(a, st);
    }
  }
  ~KernelScope() { if (open) nvtxRangePop(); }
  cudaError_t done(cudaError_t e) {
    nvtxRangePop();
    open = false;
    if (e != cudaSuccess) return e;
    if (c->debug & KVQ_DEBUG_PROFILE) {
      cudaEvent_t b = pooled_event(c);
      cudaEventRecord(b, st);
      c->recs.push_back({id, a, b});
    }
    if (c->debug & KVQ_DEBUG_SYNC) {
      e = cudaStreamSynchronize(st);
      if (e == cudaSuccess) e = cudaGetLastError();
    }
    return e;
  }
};

void free_all(kvq_cache* c) {
  if (!c) return;
  cudaDeviceSynchronize();
  for (auto& r : c->recs) { c->ev_pool.push_back(r.a); c->ev_pool.push_back(r.b); }
  for (auto e : c->ev_pool) cudaEventDestroy(e);
  if (c->t1) cudaFree(c->t1);
  if (c->scr) cudaFree(c->scr);
  if (c->res) cudaFree(c->res);
  for (auto p : c->t2k_host) if (p) cudaFreeHost(p);
  for (auto p : c->t2v_host) if (p) cudaFreeHost(p);
  if (c->side) cudaStreamDestroy(c->side);
  if (c->ev_in) cudaEventDestroy(c->ev_in);
  if (c->ev_mirror) cudaEventDestroy(c->ev_mirror);
  delete c;
}

}  // namespace

// Blocks per work item of the split-K passes: at least ITEMS_PER_CTA items per resident
// CTA when the layer is small (short contexts are latency-bound: every item reads its
// blocks one after another), at most CHUNK blocks per item otherwise.
static int decode_split(const kvq_cache* c, int nb) {
  const long long target = (long long)ITEMS_PER_CTA * kvq::mixed_grid(c->num_sms);
  const long long per = ((long long)c->BG * nb + target - 1) / target;
  return (int)std::min<long long>(kvq::CHUNK, std::max<long long>(1, per));
}

static kvq_status decode_impl(kvq_cache* c, int layer, const void* q, float tau, float eps,
                              void* out, kvq_certificate* cert, int32_t* ladder_level,
                              void* stream, bool certified, const char* fn);

extern "C" {

const char* kvq_last_error(void) { return g_err.c_str(); }

kvq_status kvq_cache_create(const kvq_config* cfg, kvq_cache** out) {
  if (!cfg || !out) return fail(KVQ_ERR_INVALID, "kvq_cache_create: NULL argument");
  *out = nullptr;
  const kvq_config& k = *cfg;
  if (k.head_dim != D) return fail(KVQ_ERR_INVALID, "head_dim must be 128");
  if (k.block_tokens != BLK) return fail(KVQ_ERR_INVALID, "block_tokens must be 64");
  if (k.value_group != VG) return fail(KVQ_ERR_INVALID, "value_group must be 32");
  if (k.n_layers < 1 || k.batch < 1 || k.n_kv_heads < 1 || k.n_q_heads < 1 || k.max_ctx < 1)
    return fail(KVQ_ERR_INVALID, "n_layers, batch, heads and max_ctx must be >= 1");
  if (k.n_q_heads % k.n_kv_heads != 0 || k.n_q_heads / k.n_kv_heads > MAXREP)
    return fail(KVQ_ERR_INVALID, "n_q_heads / n_kv_heads must be an integer in 1..4");
  if (k.rank_positions < 1) return fail(KVQ_ERR_INVALID, "rank_positions must be >= 1");
  if (k.max_ctx > (1 << 21))   // selection keeps one key per block in shared memory
    return fail(KVQ_ERR_INVALID, "max_ctx must be <= 2097152 tokens");
  if (!(k.l4_head_fraction > 0.f && k.l4_head_fraction <= 1.f))
    return fail(KVQ_ERR_INVALID, "l4_head_fraction must be in (0, 1]");
  if (k.value_bits != 0 && k.value_bits != 4 && k.value_bits != 16)
    return fail(KVQ_ERR_INVALID, "value_bits must be 4 (or 0) or 16");
  if (!(k.v_tol >= 0.f)) return fail(KVQ_ERR_INVALID, "v_tol must be >= 0 (0: no value budget)");
  if (k.resident_blocks < 0) return fail(KVQ_ERR_INVALID, "resident_blocks must be >= 0");

  int dev = 0, sms = 0;
  cudaError_t de = cudaGetDevice(&dev);
  if (de == cudaSuccess) de = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (de != cudaSuccess || sms < 1) {
    cudaGetLastError();
    return fail(KVQ_ERR_CUDA, std::string("kvq_cache_create: no usable CUDA device: ") +
                                  (de != cudaSuccess ? cudaGetErrorString(de) : "no multiprocessors"));
  }
  kvq_cache* c = new kvq_cache();
  c->cfg = k;
  c->device = dev;
  c->num_sms = sms;
  c->B = k.batch; c->Hq = k.n_q_heads; c->Hkv = k.n_kv_heads; c->n_rep = k.n_q_heads / k.n_kv_heads;
  c->BG = c->B * c->Hkv; c->L = k.n_layers;
  c->nbmax_used = k.max_ctx / BLK;
  c->nbmax = (std::max(1, c->nbmax_used) + 15) / 16 * 16;   // row stride of per-block arrays
  c->cap = (long long)((k.max_ctx + BLK - 1) / BLK) * BLK;
  c->n_tokens.assign(c->L, 0);
  c->tail_parity.assign(c->L, 0);
  c->v16 = k.value_bits == 16;

  // ---- tier 1 (INT4 value codes and scale/offset, or FP16 values) ----
  const size_t BG = c->BG, nbm = c->nbmax;
  const size_t n4 = c->v16 ? 0 : BG * nbm, n16 = c->v16 ? BG * nbm : 0;
  size_t o = 0;
  c->off_kc = o;   o = align_up(o + BG * nbm * KC_BYTES, 256);
  c->off_ks = o;   o = align_up(o + BG * nbm * D * 2, 256);
  c->off_vc = o;   o = align_up(o + n4 * VC_BYTES, 256);
  c->off_vsv = o;  o = align_up(o + n4 * VSV_WORDS * 4, 256);
  c->off_v16 = o;  o = align_up(o + n16 * BLK * D * 2, 256);
  c->off_eta = o;  o = align_up(o + BG * nbm * 4, 256);
  c->off_vmin = o; o = align_up(o + BG * D * 4, 256);
  c->off_vmax = o; o = align_up(o + BG * D * 4, 256);
  c->off_ksm = o;  o = align_up(o + BG * 4, 256);
  c->off_vsm = o;  o = align_up(o + BG * 4, 256);
  c->off_tail = o; o = align_up(o + 4 * BG * BLK * D * 2, 256);
  c->t1_layer = o;
  if (cudaMalloc(&c->t1, c->t1_layer * c->L) != cudaSuccess) {
    cudaGetLastError();
    free_all(c);
    return fail(KVQ_ERR_OOM, "tier-1 device allocation failed");
  }
  cudaError_t ie = cudaMemset(c->t1, 0, c->t1_layer * c->L);
  for (int l = 0; l < c->L && ie == cudaSuccess; ++l) {
    fill_u32<<<64, 256>>>(layer_vmin(c, l), 0xFF800000u, BG * D);  // encoding of +inf
    fill_u32<<<64, 256>>>(layer_vmax(c, l), 0x007FFFFFu, BG * D);  // encoding of -inf
    ie = cudaGetLastError();
  }
  if (ie != cudaSuccess) {
    free_all(c);
    return fail(KVQ_ERR_CUDA, std::string("kvq_cache_create: tier-1 initialisation: ") + cudaGetErrorString(ie));
  }

  // ---- tier 2: pinned, mapped host memory ----
  const size_t t2bytes = (size_t)BG * c->cap * D * sizeof(__half);
  c->t2k_host.assign(c->L, nullptr); c->t2v_host.assign(c->L, nullptr);
  c->t2k_dev.assign(c->L, nullptr); c->t2v_dev.assign(c->L, nullptr);
  for (int l = 0; l < c->L; ++l) {
    for (int kv = 0; kv < (c->v16 ? 1 : 2); ++kv) {   // FP16 values need no tier-2 copy
      void* h = nullptr;
      if (cudaHostAlloc(&h, t2bytes, cudaHostAllocMapped | cudaHostAllocPortable) != cudaSuccess) {
        cudaGetLastError();
        free_all(c);
        return fail(KVQ_ERR_HOST_OOM, "tier-2 pinned host allocation failed");
      }
      void* d = nullptr;
      if (cudaHostGetDevicePointer(&d, h, 0) != cudaSuccess) {
        cudaGetLastError();
        (kv ? c->t2v_host : c->t2k_host)[l] = static_cast<__half*>(h);
        free_all(c);
        return fail(KVQ_ERR_HOST_OOM, "tier-2 memory is not mapped into the device");
      }
      (kv ? c->t2v_host : c->t2k_host)[l] = static_cast<__half*>(h);
      (kv ? c->t2v_dev : c->t2k_dev)[l] = static_cast<__half*>(d);
    }
  }

  // ---- scratch ----
  const size_t HQ = (size_t)c->B * c->Hq;
  // partial slots per group: enough for every split decode_split() can choose and for
  // the INT4 value pass's runs (tail_runs), whichever asks for more
  const size_t target = (size_t)ITEMS_PER_CTA * mixed_grid(c->num_sms);
  const size_t NCH = std::max({nbm / CHUNK + 1, (target + BG - 1) / BG + 1,
                               (size_t)tail_runs(c->num_sms, (int)BG) + 1});
  c->nslot = (int)NCH;
  o = 0;
  const size_t s_shat = o;  o = align_up(o + HQ * nbm * BLK * 4, 256);
  const size_t s_lse8 = o;  o = align_up(o + HQ * nbm * 4, 256);
  const size_t s_delta = o; o = align_up(o + HQ * nbm * 4, 256);
  const size_t s_lse16 = o; o = align_up(o + HQ * nbm * 4, 256);
  const size_t s_sel = o;   o = align_up(o + HQ * nbm, 256);
  const size_t s_kp0 = o;   o = align_up(o + BG * nbm, 256);
  const size_t s_kp1 = o;   o = align_up(o + BG * nbm, 256);
  const size_t s_vp1 = o;   o = align_up(o + BG * nbm, 256);
  const size_t s_hst = o;   o = align_up(o + HQ * sizeof(HeadState), 256);
  const size_t s_gst = o;   o = align_up(o + BG * sizeof(GroupState), 256);
  const size_t s_part = o;  o = align_up(o + BG * NCH * MAXREP * (D + 4) * 4, 256);
  const size_t s_part1 = o; o = align_up(o + BG * NCH * MAXREP * (D + 4) * 4, 256);
  const size_t s_red0 = o;  o = align_up(o + HQ * (D + 4) * 4, 256);
  const size_t s_dpart = o; o = align_up(o + BG * NCH * MAXREP * (D + 4) * 4, 256);
  const size_t s_cnt = o;   o = align_up(o + (CNT_GROUP_BASE + 4 * BG + c->B) * 4, 256);
  const size_t s_q = o;     o = align_up(o + HQ * D * 2, 256);
  const size_t s_out = o;   o = align_up(o + HQ * D * 2, 256);
  const size_t s_cert = o;  o = align_up(o + HQ * sizeof(kvq_certificate), 256);
  const size_t s_lvl = o;   o = align_up(o + c->B * 4, 256);
  if (cudaMalloc(&c->scr, o) != cudaSuccess) {
    cudaGetLastError();
    free_all(c);
    return fail(KVQ_ERR_OOM, "scratch device allocation failed");
  }
  cudaMemset(c->scr, 0, o);
  c->shat = reinterpret_cast<float*>(c->scr + s_shat);
  c->lse8 = reinterpret_cast<float*>(c->scr + s_lse8);
  c->delta = reinterpret_cast<float*>(c->scr + s_delta);
  c->lse16 = reinterpret_cast<float*>(c->scr + s_lse16);
  c->sel = reinterpret_cast<uint8_t*>(c->scr + s_sel);
  c->kprom0 = reinterpret_cast<uint8_t*>(c->scr + s_kp0);
  c->kprom1 = reinterpret_cast<uint8_t*>(c->scr + s_kp1);
  c->vprom1 = reinterpret_cast<uint8_t*>(c->scr + s_vp1);
  c->hst = reinterpret_cast<HeadState*>(c->scr + s_hst);
  c->gst = reinterpret_cast<GroupState*>(c->scr + s_gst);
  c->part = reinterpret_cast<float*>(c->scr + s_part);
  c->part1 = reinterpret_cast<float*>(c->scr + s_part1);
  c->red0 = reinterpret_cast<float*>(c->scr + s_red0);
  c->dpart = reinterpret_cast<float*>(c->scr + s_dpart);
  c->counters = reinterpret_cast<unsigned int*>(c->scr + s_cnt);
  c->q_stage = reinterpret_cast<__half*>(c->scr + s_q);
  c->out_stage = reinterpret_cast<__half*>(c->scr + s_out);
  c->cert_stage = reinterpret_cast<kvq_certificate*>(c->scr + s_cert);
  c->level_stage = reinterpret_cast<int32_t*>(c->scr + s_lvl);

  // ---- cross-step residency (resident_blocks slots of 16 KiB per layer) ----
  c->call_id.assign(c->L, 0u);
  c->nres = k.resident_blocks;
  if (c->nres > 0) {
    if ((size_t)BG * nbm >= (1u << 30))
      { free_all(c); return fail(KVQ_ERR_INVALID, "resident_blocks: cache too large for the slot table"); }
    const size_t S = (size_t)c->nres;
    o = 0;
    c->off_rk = o;     o = align_up(o + BG * nbm * 4, 256);
    c->off_rv = o;     o = align_up(o + BG * nbm * 4, 256);
    c->off_rown = o;   o = align_up(o + S * 4, 256);
    c->off_rstamp = o; o = align_up(o + S * 4, 256);
    c->off_rfree = o;  o = align_up(o + S * 4, 256);
    c->off_rstate = o; o = align_up(o + RS_WORDS * 4, 256);
    c->off_rbytes = o; o = align_up(o + 2 * 8, 256);
    c->off_rpool = o;  o = align_up(o + S * F16_BLOCK_BYTES, 256);
    c->res_layer = o;
    if (cudaMalloc(&c->res, c->res_layer * c->L) != cudaSuccess) {
      cudaGetLastError();
      free_all(c);
      return fail(KVQ_ERR_OOM, "residency device allocation failed");
    }
    for (int l = 0; l < c->L; ++l) {
      char* r = c->res + c->res_layer * l;
      cudaMemset(r + c->off_rk, 0xff, BG * nbm * 4);   // -1: not resident
      cudaMemset(r + c->off_rv, 0xff, BG * nbm * 4);
      const unsigned int st0[RS_WORDS] = {(unsigned int)S, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
      cudaMemcpy(r + c->off_rstate, st0, sizeof st0, cudaMemcpyHostToDevice);
      cudaMemset(r + c->off_rbytes, 0, 16);
      launch_residency_init(reinterpret_cast<int*>(r + c->off_rfree), reinterpret_cast<int*>(r + c->off_rown),
                            reinterpret_cast<unsigned int*>(r + c->off_rstamp), c->nres, 0);
    }
  }

  if (cudaStreamCreateWithFlags(&c->side, cudaStreamNonBlocking) != cudaSuccess ||
      cudaEventCreateWithFlags(&c->ev_in, cudaEventDisableTiming) != cudaSuccess ||
      cudaEventCreateWithFlags(&c->ev_mirror, cudaEventDisableTiming) != cudaSuccess) {
    cudaError_t e = cudaGetLastError();
    free_all(c);
    return cuda_fail(e, "kvq_cache_create: stream/event");
  }
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) {
    free_all(c);
    return cuda_fail(e, "kvq_cache_create");
  }
  *out = c;
  return KVQ_OK;
}

kvq_status kvq_cache_destroy(kvq_cache* cache) {
  if (!cache) return KVQ_OK;
  DeviceGuard dg(cache->device);
  free_all(cache);
  return KVQ_OK;
}

kvq_status kvq_set_debug(kvq_cache* c, int flags) {
  if (!c) return fail(KVQ_ERR_INVALID, "kvq_set_debug: NULL cache");
  c->debug = flags;
  return KVQ_OK;
}

kvq_status kvq_cache_length(const kvq_cache* c, int layer, int* n) {
  if (!c || !n) return fail(KVQ_ERR_INVALID, "kvq_cache_length: NULL argument");
  if (layer < 0 || layer >= c->L) return fail(KVQ_ERR_INVALID, "layer out of range");
  *n = c->n_tokens[layer];
  return KVQ_OK;
}

kvq_status kvq_append(kvq_cache* c, int layer, const void* k, const void* v, int n, void* stream) {
  if (!c) return fail(KVQ_ERR_INVALID, "kvq_append: NULL cache");
  if (layer < 0 || layer >= c->L) return fail(KVQ_ERR_INVALID, "kvq_append: layer out of range");
  DeviceGuard dg(c->device);
  if (n < 0) return fail(KVQ_ERR_INVALID, "kvq_append: n_tokens < 0");
  if (n == 0) return KVQ_OK;
  if (!k || !v) return fail(KVQ_ERR_INVALID, "kvq_append: NULL k or v");
  if (!is_device_ptr(k) || !is_device_ptr(v))
    return fail(KVQ_ERR_INVALID, "kvq_append: k and v must be device memory");
  if (!aligned(k, 16) || !aligned(v, 16))   // read with 16-byte loads
    return fail(KVQ_ERR_INVALID, "kvq_append: k and v must be 16-byte aligned");
  const int pos = c->n_tokens[layer];
  if ((long long)pos + n > c->cfg.max_ctx)
    return fail(KVQ_ERR_CAPACITY, "kvq_append: cache capacity (max_ctx) exceeded");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const size_t dpitch = (size_t)c->cap * D * sizeof(__half);
  const size_t width = (size_t)n * D * sizeof(__half);
  if (pos % BLK + n < BLK) {
    // Every new token stays in the FP16 partial block, which no decode reads from tier 2.
    // The mirror then copies the tokens from the partial-block buffer the kernel writes
    // (not from the caller's buffers) and is not joined: the call costs one launch.
    // Earlier mirrors may still read the buffer this kernel overwrites (the ping-pong
    // partner of the last append): they are waited for first.
    KVQ_CUDA(cudaStreamWaitEvent(st, c->ev_mirror, 0), "kvq_append: wait mirror");
    if (kvq_status bs = bounds_clear(c, st)) return bs;
    {
      KernelScope ks(c, K_APPEND, st);
      KVQ_CUDA(ks.done(launch_append(append_view(c, layer), k, v, n, pos, st)), "quantize_append");
    }
    if (kvq_status bs = bounds_report(c, st, "kvq_append")) return bs;
    KVQ_CUDA(cudaEventRecord(c->ev_in, st), "kvq_append: event");
    KVQ_CUDA(cudaStreamWaitEvent(c->side, c->ev_in, 0), "kvq_append: wait");
    const int p_out = 1 - c->tail_parity[layer];
    const size_t spitch = (size_t)BLK * D * sizeof(__half);
    const size_t row0 = (size_t)(pos % BLK) * D;
    if (c->debug & KVQ_DEBUG_FAIL_MIRROR)
      return cuda_fail(cudaErrorInvalidValue, "kvq_append: mirror K (injected failure)");
    KVQ_CUDA(cudaMemcpy2DAsync(c->t2k_host[layer] + (size_t)pos * D, dpitch,
                               layer_tail(c, layer, p_out, 0) + row0, spitch, width, c->BG,
                               cudaMemcpyDeviceToHost, c->side), "kvq_append: mirror K");
    if (!c->v16)
      KVQ_CUDA(cudaMemcpy2DAsync(c->t2v_host[layer] + (size_t)pos * D, dpitch,
                                 layer_tail(c, layer, p_out, 1) + row0, spitch, width, c->BG,
                                 cudaMemcpyDeviceToHost, c->side), "kvq_append: mirror V");
    KVQ_CUDA(cudaEventRecord(c->ev_mirror, c->side), "kvq_append: event");
    c->n_tokens[layer] = pos + n;
    c->tail_parity[layer] ^= 1;
    return KVQ_OK;
  }
  // tier-2 mirror of the caller's tokens on the side stream, overlapped with
  // quantisation and joined before the call returns (a completed block may be paged in
  // by the next decode, and the caller may reuse k and v)
  KVQ_CUDA(cudaEventRecord(c->ev_in, st), "kvq_append: event");
  KVQ_CUDA(cudaStreamWaitEvent(c->side, c->ev_in, 0), "kvq_append: wait");
  if (c->debug & KVQ_DEBUG_FAIL_MIRROR)
    return cuda_fail(cudaErrorInvalidValue, "kvq_append: mirror K (injected failure)");
  KVQ_CUDA(cudaMemcpy2DAsync(c->t2k_host[layer] + (size_t)pos * D, dpitch, k, width, width, c->BG,
                             cudaMemcpyDeviceToHost, c->side), "kvq_append: mirror K");
  if (!c->v16)
    KVQ_CUDA(cudaMemcpy2DAsync(c->t2v_host[layer] + (size_t)pos * D, dpitch, v, width, width, c->BG,
                               cudaMemcpyDeviceToHost, c->side), "kvq_append: mirror V");
  KVQ_CUDA(cudaEventRecord(c->ev_mirror, c->side), "kvq_append: event");
  if (kvq_status bs = bounds_clear(c, st)) return bs;
  {
    KernelScope ks(c, K_APPEND, st);
    KVQ_CUDA(ks.done(launch_append(append_view(c, layer), k, v, n, pos, st)), "quantize_append");
  }
  KVQ_CUDA(cudaStreamWaitEvent(st, c->ev_mirror, 0), "kvq_append: join");
  if (kvq_status bs = bounds_report(c, st, "kvq_append")) return bs;
  c->n_tokens[layer] = pos + n;
  c->tail_parity[layer] ^= 1;
  return KVQ_OK;
}

kvq_status kvq_decode_attention(kvq_cache* c, int layer, const void* q, float tau, float eps,
                                void* out, kvq_certificate* cert, int32_t* ladder_level,
                                void* stream) {
  if (!(tau > 0.f && tau <= 1.f)) return fail(KVQ_ERR_INVALID, "kvq_decode_attention: tau_cov must be in (0, 1]");
  if (!(eps >= 0.f)) return fail(KVQ_ERR_INVALID, "kvq_decode_attention: eps must be >= 0");
  return decode_impl(c, layer, q, tau, eps, out, cert, ladder_level, stream, true, "kvq_decode_attention");
}

kvq_status kvq_decode_attention_uncertified(kvq_cache* c, int layer, const void* q, void* out,
                                            kvq_certificate* cert, void* stream) {
  // an empty selection (tau_cov = 0) and no bound to meet (eps = +inf): INT8 scores and
  // INT4 values on every full block
  return decode_impl(c, layer, q, 0.f, INFINITY, out, cert, nullptr, stream, false,
                     "kvq_decode_attention_uncertified");
}

}  // extern "C"

static kvq_status decode_impl(kvq_cache* c, int layer, const void* q, float tau, float eps,
                              void* out, kvq_certificate* cert, int32_t* ladder_level,
                              void* stream, bool certified, const char* fn) {
  const std::string f(fn);
  if (!c) return fail(KVQ_ERR_INVALID, f + ": NULL cache");
  DeviceGuard dg(c->device);
  if (layer < 0 || layer >= c->L) return fail(KVQ_ERR_INVALID, f + ": layer out of range");
  if (!q || !out) return fail(KVQ_ERR_INVALID, f + ": NULL q or out");
  const int N = c->n_tokens[layer];
  if (N == 0) return fail(KVQ_ERR_INVALID, f + ": layer holds no tokens");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const size_t HQ = (size_t)c->B * c->Hq;
  const bool q_dev = is_device_ptr(q), out_dev = is_device_ptr(out);
  const bool cert_dev = cert && is_device_ptr(cert);
  const bool lvl_dev = ladder_level && is_device_ptr(ladder_level);
  // pageable host buffers make the call wait for its copies; page-locked ones are copied
  // in stream order (valid once the stream has reached them)
  const bool pageable_any = (!q_dev && !is_pinned_host_ptr(q)) || (!out_dev && !is_pinned_host_ptr(out)) ||
                            (cert && !cert_dev && !is_pinned_host_ptr(cert)) ||
                            (ladder_level && !lvl_dev && !is_pinned_host_ptr(ladder_level));
  // device buffers are read and written in place with vector accesses (host buffers are
  // staged through the cache's own)
  if ((q_dev && !aligned(q, 16)) || (out_dev && !aligned(out, 16)))
    return fail(KVQ_ERR_INVALID, f + ": device q and out must be 16-byte aligned");
  if ((cert_dev && !aligned(cert, alignof(kvq_certificate))) || (lvl_dev && !aligned(ladder_level, 4)))
    return fail(KVQ_ERR_INVALID, f + ": device cert must be 8-byte and ladder_level 4-byte aligned");
  const __half* qd = static_cast<const __half*>(q);
  if (!q_dev) {
    KVQ_CUDA(cudaMemcpyAsync(c->q_stage, q, HQ * D * 2, cudaMemcpyHostToDevice, st), "stage q");
    qd = c->q_stage;
  }
  __half* od = out_dev ? static_cast<__half*>(out) : c->out_stage;
  kvq_certificate* cd = cert_dev ? cert : c->cert_stage;
  int32_t* ld = lvl_dev ? ladder_level : c->level_stage;

  LayerView V;
  V.B = c->B; V.Hq = c->Hq; V.Hkv = c->Hkv; V.n_rep = c->n_rep; V.BG = c->BG;
  V.nb = N / BLK; V.n_tail = N % BLK; V.nbmax = c->nbmax; V.cap = c->cap;
  V.chunk = decode_split(c, V.nb); V.nslot = c->nslot; V.nparts = 0;
  if (std::max(1, (V.nb + V.chunk - 1) / V.chunk) > V.nslot)
    return fail(KVQ_ERR_INVALID, f + ": more work items per KV group than partial slots");
  V.kc = layer_kc(c, layer); V.ks = layer_ks(c, layer); V.vc = layer_vc(c, layer);
  V.vsv = layer_vsv(c, layer); V.eta = layer_eta(c, layer);
  V.vmin = layer_vmin(c, layer); V.vmax = layer_vmax(c, layer);
  V.kscale_max = layer_ksm(c, layer); V.vscale_max = layer_vsm(c, layer);
  const int p = c->tail_parity[layer];
  V.tail_k = layer_tail(c, layer, p, 0); V.tail_v = layer_tail(c, layer, p, 1);
  V.t2k = c->t2k_dev[layer]; V.t2v = c->t2v_dev[layer]; V.v16 = layer_v16(c, layer);
  V.q = qd; V.out = od; V.tau = tau; V.eps = eps;
  V.l4_frac = c->cfg.l4_head_fraction; V.rank_positions = c->cfg.rank_positions;
  V.v_tol = (certified && c->cfg.v_tol > 0.f) ? c->cfg.v_tol : INFINITY;
  V.debug = certified ? c->debug : (c->debug & ~(KVQ_DEBUG_FORCE_RANK_FAIL | KVQ_DEBUG_FORCE_DENSE));
  V.shat = c->shat; V.lse8 = c->lse8; V.delta = c->delta; V.lse16 = c->lse16; V.sel = c->sel;
  V.kprom0 = c->kprom0; V.kprom1 = c->kprom1; V.vprom1 = c->vprom1;
  V.hst = c->hst; V.gst = c->gst; V.part = c->part; V.dpart = c->dpart; V.counters = c->counters;
  V.part1 = c->part1; V.red0 = c->red0;
  V.nres = 0; V.call_id = 0u;
  V.rslot_k = V.rslot_v = nullptr; V.rpool = nullptr; V.rowner = nullptr; V.rstamp = nullptr;
  V.rfree = nullptr; V.rstate = nullptr; V.rbytes = nullptr;
  if (certified && c->nres > 0) {   // only certified calls page FP16 blocks in
    char* r = c->res + c->res_layer * layer;
    V.nres = c->nres;
    V.call_id = ++c->call_id[layer];
    V.rslot_k = reinterpret_cast<int*>(r + c->off_rk);
    V.rslot_v = reinterpret_cast<int*>(r + c->off_rv);
    V.rowner = reinterpret_cast<int*>(r + c->off_rown);
    V.rstamp = reinterpret_cast<unsigned int*>(r + c->off_rstamp);
    V.rfree = reinterpret_cast<int*>(r + c->off_rfree);
    V.rstate = reinterpret_cast<unsigned int*>(r + c->off_rstate);
    V.rbytes = reinterpret_cast<unsigned long long*>(r + c->off_rbytes);
    V.rpool = reinterpret_cast<__half*>(r + c->off_rpool);
  }

  const bool all_dense = certified && ((tau >= 1.f) || (c->debug & KVQ_DEBUG_FORCE_DENSE));
  if (kvq_status bs = bounds_clear(c, st)) return bs;
  if (!all_dense) {
    { KernelScope s(c, K_SCORE, st); KVQ_CUDA(s.done(launch_score(V, score_grid(c->num_sms), st)), "score"); }
    { KernelScope s(c, K_SELECT, st); KVQ_CUDA(s.done(launch_select(V, st)), "select"); }
    if (certified || c->v16) {
      KernelScope s(c, K_MIX0, st);
      KVQ_CUDA(s.done(launch_mixed(V, 0, mixed_grid(c->num_sms), st)), "mixed_round0");
    } else {
      // nothing is paged in: the INT4 value pass over every block, one partial per run
      const int runs = tail_runs(c->num_sms, V.BG);
      if (runs > V.nslot) return fail(KVQ_ERR_INVALID, f + ": more INT4-pass runs than partial slots");
      KernelScope s(c, K_TAIL, st);
      KVQ_CUDA(s.done(launch_tail(V, runs, c->num_sms, st)), "int4_tail");
      V.nparts = runs;
    }
    { KernelScope s(c, K_COMB0, st); KVQ_CUDA(s.done(launch_combine(V, 0, st)), "combine_round0"); }
    if (certified) {
      { KernelScope s(c, K_MIX1, st); KVQ_CUDA(s.done(launch_mixed(V, 1, mixed_grid(c->num_sms), st)), "mixed_round1"); }
      { KernelScope s(c, K_COMB1, st); KVQ_CUDA(s.done(launch_combine(V, 1, st)), "combine_round1"); }
    }
  }
  if (certified) {
    KernelScope s(c, K_DENSE, st);
    KVQ_CUDA(s.done(launch_dense(V, all_dense ? 1 : 0, dense_grid(c->num_sms), st)), "dense_fallback");
  }
  { KernelScope s(c, K_FINAL, st); KVQ_CUDA(s.done(launch_finalize(V, cd, ld, st)), "finalize"); }
  if (V.nres > 0) { KernelScope s(c, K_RESIDENT, st); KVQ_CUDA(s.done(launch_residency(V, st)), "residency"); }
  if (kvq_status bs = bounds_report(c, st, f)) return bs;

  if (!out_dev) KVQ_CUDA(cudaMemcpyAsync(out, od, HQ * D * 2, cudaMemcpyDeviceToHost, st), "copy out");
  if (cert && !cert_dev) KVQ_CUDA(cudaMemcpyAsync(cert, cd, HQ * sizeof(kvq_certificate), cudaMemcpyDeviceToHost, st), "copy cert");
  if (ladder_level && !lvl_dev) KVQ_CUDA(cudaMemcpyAsync(ladder_level, ld, c->B * 4, cudaMemcpyDeviceToHost, st), "copy level");
  if (pageable_any) KVQ_CUDA(cudaStreamSynchronize(st), (f + ": sync").c_str());
  c->last_layer = layer;
  c->last_nb = all_dense ? -1 : V.nb;
  return KVQ_OK;
}

extern "C" {

kvq_status kvq_export_tier1(kvq_cache* c, int layer, void* kc, void* ks, void* vc, void* vs,
                            void* vo, float* eta, float* vmin, float* vmax, void* stream) {
  if (!c) return fail(KVQ_ERR_INVALID, "kvq_export_tier1: NULL cache");
  DeviceGuard dg(c->device);
  if (layer < 0 || layer >= c->L) return fail(KVQ_ERR_INVALID, "kvq_export_tier1: layer out of range");
  const int nb = c->n_tokens[layer] / BLK;
  KVQ_CUDA(launch_export_tier1(append_view(c, layer), nb, kc, ks, vc, vs, vo, eta, vmin, vmax,
                               static_cast<cudaStream_t>(stream)), "export_tier1");
  return KVQ_OK;
}

kvq_status kvq_export_decode_state(kvq_cache* c, uint8_t* sel, uint8_t* kprom0, uint8_t* kprom1,
                                   uint8_t* vprom1, float* lse8, float* delta, void* stream) {
  if (!c) return fail(KVQ_ERR_INVALID, "kvq_export_decode_state: NULL cache");
  DeviceGuard dg(c->device);
  if (c->last_layer < 0 || c->last_nb < 0)
    return fail(KVQ_ERR_INVALID, "kvq_export_decode_state: no certified decode call yet");
  const int nb = c->last_nb;
  if (nb == 0) return KVQ_OK;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const size_t HQ = (size_t)c->B * c->Hq, nbm = c->nbmax;
  auto cp = [&](void* dst, const void* src, size_t elem, size_t rows) -> cudaError_t {
    if (!dst) return cudaSuccess;
    return cudaMemcpy2DAsync(dst, nb * elem, src, nbm * elem, nb * elem, rows, cudaMemcpyDeviceToDevice, st);
  };
  KVQ_CUDA(cp(sel, c->sel, 1, HQ), "export sel");
  KVQ_CUDA(cp(kprom0, c->kprom0, 1, c->BG), "export kprom0");
  KVQ_CUDA(cp(kprom1, c->kprom1, 1, c->BG), "export kprom1");
  KVQ_CUDA(cp(vprom1, c->vprom1, 1, c->BG), "export vprom1");
  KVQ_CUDA(cp(lse8, c->lse8, 4, HQ), "export lse8");
  KVQ_CUDA(cp(delta, c->delta, 4, HQ), "export delta");
  return KVQ_OK;
}

kvq_status kvq_profile_read(kvq_cache* c, kvq_kernel_stat* stats, int max, int* n, int reset) {
  if (!c || !n || (max > 0 && !stats)) return fail(KVQ_ERR_INVALID, "kvq_profile_read: NULL argument");
  DeviceGuard dg(c->device);
  for (auto& r : c->recs) {
    KVQ_CUDA(cudaEventSynchronize(r.b), "kvq_profile_read: sync");
    float ms = 0.f;
    KVQ_CUDA(cudaEventElapsedTime(&ms, r.a, r.b), "kvq_profile_read: elapsed");
    c->prof_ms[r.id] += ms;
    c->prof_n[r.id] += 1;
    c->ev_pool.push_back(r.a);
    c->ev_pool.push_back(r.b);
  }
  c->recs.clear();
  int w = 0;
  for (int i = 0; i < K_COUNT && w < max; ++i) {
    if (c->prof_n[i] == 0) continue;
    std::memset(&stats[w], 0, sizeof(kvq_kernel_stat));
    std::strncpy(stats[w].name, kKernelNames[i], sizeof(stats[w].name) - 1);
    stats[w].launches = c->prof_n[i];
    stats[w].total_ms = c->prof_ms[i];
    ++w;
  }
  *n = w;
  if (reset) {
    for (int i = 0; i < K_COUNT; ++i) { c->prof_ms[i] = 0; c->prof_n[i] = 0; }
  }
  return KVQ_OK;
}

kvq_status kvq_residency_stats(kvq_cache* c, int layer, int64_t* resident_bytes,
                               int64_t* host_bytes, int32_t* slots_in_use, int reset) {
  if (!c) return fail(KVQ_ERR_INVALID, "kvq_residency_stats: NULL cache");
  if (layer < 0 || layer >= c->L) return fail(KVQ_ERR_INVALID, "kvq_residency_stats: layer out of range");
  DeviceGuard dg(c->device);
  unsigned long long b[2] = {0ull, 0ull};
  unsigned int stt[RS_WORDS] = {};
  if (c->nres > 0) {
    char* r = c->res + c->res_layer * layer;
    KVQ_CUDA(cudaDeviceSynchronize(), "kvq_residency_stats: sync");
    KVQ_CUDA(cudaMemcpy(b, r + c->off_rbytes, sizeof b, cudaMemcpyDeviceToHost), "kvq_residency_stats: read");
    KVQ_CUDA(cudaMemcpy(stt, r + c->off_rstate, sizeof stt, cudaMemcpyDeviceToHost), "kvq_residency_stats: read");
    if (reset) KVQ_CUDA(cudaMemset(r + c->off_rbytes, 0, sizeof b), "kvq_residency_stats: reset");
  }
  if (resident_bytes) *resident_bytes = (int64_t)b[0];
  if (host_bytes) *host_bytes = (int64_t)b[1];
  if (slots_in_use) *slots_in_use = (int32_t)stt[RS_USED];
  return KVQ_OK;
}

kvq_status kvq_debug_fill_tier2(kvq_cache* c, int layer, uint16_t bits) {
  if (!c) return fail(KVQ_ERR_INVALID, "kvq_debug_fill_tier2: NULL cache");
  if (layer < 0 || layer >= c->L) return fail(KVQ_ERR_INVALID, "kvq_debug_fill_tier2: layer out of range");
  DeviceGuard dg(c->device);
  KVQ_CUDA(cudaDeviceSynchronize(), "kvq_debug_fill_tier2: sync");   // no copy or kernel in flight
  const size_t n = (size_t)c->BG * c->cap * D;
  uint16_t* k = reinterpret_cast<uint16_t*>(c->t2k_host[layer]);
  std::fill(k, k + n, bits);
  if (!c->v16) {
    uint16_t* v = reinterpret_cast<uint16_t*>(c->t2v_host[layer]);
    std::fill(v, v + n, bits);
  }
  return KVQ_OK;
}

}  // extern "C"
