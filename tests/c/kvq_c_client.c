/*
 * Plain C client of the kvq C ABI (no Python, no torch): builds a small cache from
 * seeded pseudo-random FP16 keys and values, decodes with tau_cov = 1 (rung 4: exact
 * dense attention over tier 2, "Runtime-Certified Bounded-Error Quantized Attention",
 * Contributions: deterministic recovery) and with tau_cov = 0.99, passing host buffers,
 * and checks the dense result against a double-precision softmax attention computed
 * here.  Exit status 0 on success.
 */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime_api.h>

#include "kvq.h"

enum { B = 1, HQ = 8, HKV = 2, D = 128, N = 64 * 5 + 17 };

static uint64_t rng_state = 0x9E3779B97F4A7C15ull;
static double uniform01(void) {   /* splitmix64 */
  uint64_t z = (rng_state += 0x9E3779B97F4A7C15ull);
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  z ^= z >> 31;
  return (double)(z >> 11) * (1.0 / 9007199254740992.0);
}

/* float -> binary16 (round to nearest even), for |x| well inside the normal range */
static uint16_t to_half(float f) {
  uint32_t x;
  memcpy(&x, &f, 4);
  const uint32_t sign = (x >> 16) & 0x8000u;
  int32_t e = (int32_t)((x >> 23) & 0xff) - 127 + 15;
  uint32_t m = x & 0x7fffffu;
  if (e <= 0) return (uint16_t)sign;               /* tiny values flush to zero here */
  uint32_t h = sign | ((uint32_t)e << 10) | (m >> 13);
  const uint32_t rest = m & 0x1fffu;
  if (rest > 0x1000u || (rest == 0x1000u && (h & 1u))) h += 1;
  return (uint16_t)h;
}
static double from_half(uint16_t h) {
  const int e = (h >> 10) & 0x1f, m = h & 0x3ff;
  const double v = e == 0 ? ldexp(m, -24) : ldexp(1024 + m, e - 25);
  return (h & 0x8000u) ? -v : v;
}

static double gauss(void) {
  const double u = uniform01() + 1e-12, v = uniform01();
  return sqrt(-2.0 * log(u)) * cos(6.283185307179586 * v);
}

#define CHECK(call)                                                              \
  do {                                                                           \
    kvq_status s_ = (call);                                                      \
    if (s_ != KVQ_OK) {                                                          \
      fprintf(stderr, "%s failed: %d (%s)\n", #call, (int)s_, kvq_last_error());  \
      return 1;                                                                  \
    }                                                                            \
  } while (0)

int main(void) {
  const size_t kv_elems = (size_t)B * HKV * N * D, q_elems = (size_t)B * HQ * D;
  uint16_t* k = malloc(kv_elems * 2);
  uint16_t* v = malloc(kv_elems * 2);
  uint16_t* q = malloc(q_elems * 2);
  uint16_t* out = malloc(q_elems * 2);
  kvq_certificate cert[B * HQ];
  int32_t level[B];
  for (size_t i = 0; i < kv_elems; ++i) k[i] = to_half((float)(2.0 * gauss()));
  for (size_t i = 0; i < kv_elems; ++i) v[i] = to_half((float)gauss());
  for (size_t i = 0; i < q_elems; ++i) q[i] = to_half((float)gauss());

  void *dk = NULL, *dv = NULL;
  if (cudaMalloc(&dk, kv_elems * 2) != cudaSuccess || cudaMalloc(&dv, kv_elems * 2) != cudaSuccess) {
    fprintf(stderr, "cudaMalloc failed\n");
    return 1;
  }
  cudaMemcpy(dk, k, kv_elems * 2, cudaMemcpyHostToDevice);
  cudaMemcpy(dv, v, kv_elems * 2, cudaMemcpyHostToDevice);

  kvq_config cfg;
  memset(&cfg, 0, sizeof cfg);
  cfg.n_layers = 1; cfg.batch = B; cfg.n_q_heads = HQ; cfg.n_kv_heads = HKV;
  cfg.head_dim = D; cfg.block_tokens = 64; cfg.value_group = 32; cfg.max_ctx = N;
  cfg.rank_positions = 1; cfg.l4_head_fraction = 0.5f;
  kvq_cache* cache = NULL;
  CHECK(kvq_cache_create(&cfg, &cache));
  CHECK(kvq_append(cache, 0, dk, dv, N, NULL));

  /* tau_cov = 1: every head at rung 4, out = fp16(O_dense) */
  CHECK(kvq_decode_attention(cache, 0, q, 1.0f, 0.25f, out, cert, level, NULL));
  double worst = 0.0;
  for (int h = 0; h < HQ; ++h) {
    const int g = h / (HQ / HKV);
    double s[N], mx = -INFINITY, l = 0.0;
    for (int t = 0; t < N; ++t) {
      double acc = 0.0;
      for (int c = 0; c < D; ++c)
        acc += from_half(q[h * D + c]) * from_half(k[((size_t)g * N + t) * D + c]);
      s[t] = acc / sqrt((double)D);
      if (s[t] > mx) mx = s[t];
    }
    for (int t = 0; t < N; ++t) { s[t] = exp(s[t] - mx); l += s[t]; }
    for (int c = 0; c < D; ++c) {
      double o = 0.0;
      for (int t = 0; t < N; ++t) o += s[t] * from_half(v[((size_t)g * N + t) * D + c]);
      o /= l;
      const double err = fabs(from_half(out[h * D + c]) - o);
      if (err > 2e-3 + 1e-2 * fabs(o)) {
        fprintf(stderr, "head %d channel %d: %g vs %g\n", h, c, from_half(out[h * D + c]), o);
        return 1;
      }
      if (err > worst) worst = err;
    }
    if (cert[h].level != 4 || cert[h].e_key != 0.f || cert[h].e_val != 0.f) {
      fprintf(stderr, "head %d: level %d, bounds %g %g\n", h, cert[h].level, cert[h].e_key, cert[h].e_val);
      return 1;
    }
  }
  if (level[0] != 4) { fprintf(stderr, "ladder level %d\n", level[0]); return 1; }

  /* certified call: every head reports a level in 0..4 and non-negative bounds */
  CHECK(kvq_decode_attention(cache, 0, q, 0.99f, 0.25f, out, cert, level, NULL));
  for (int h = 0; h < HQ; ++h)
    if (cert[h].level < 0 || cert[h].level > 4 || !(cert[h].e_key >= 0.f) || !(cert[h].e_val >= 0.f)) {
      fprintf(stderr, "head %d: bad certificate\n", h);
      return 1;
    }
  /* argument errors come back as status codes */
  if (kvq_decode_attention(cache, 0, q, 0.0f, 0.25f, out, NULL, NULL, NULL) != KVQ_ERR_INVALID) return 1;
  if (kvq_append(cache, 0, dk, dv, 1, NULL) != KVQ_ERR_CAPACITY) return 1;

  CHECK(kvq_cache_destroy(cache));
  cudaFree(dk);
  cudaFree(dv);
  printf("c client ok: max-abs error %.3g, ladder level %d\n", worst, level[0]);
  free(k); free(v); free(q); free(out);
  return 0;
}
