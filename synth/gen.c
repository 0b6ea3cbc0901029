/*
 * Seeded synthetic inputs for the sparse KV-cache offloading decode path.
 *
 * This module is shared by the CPU oracle side and the CUDA side as the ONE
 * source of input tensors. It holds none of the method's arithmetic: only
 * random streams, a Box-Muller normal transform and an fp32->bf16 rounding.
 *
 * Streams are counter based: value(seed, tid, idx) = mix(mix(seed ^ mix(tid))
 * + (idx + 1) * GAMMA), where mix is the splitmix64 finaliser (Steele, Lea,
 * Flood, "Fast splittable pseudorandom number generators", OOPSLA 2014) and
 * GAMMA its golden-ratio increment. A tensor id (tid) packs a kind tag with
 * (layer, request); the index is a flat element index. Every value is thus
 * independent of how many threads fill a buffer or in which order.
 *
 * Normals: Box-Muller (1958) on two 53-bit uniforms, in fp64, then rounded to
 * fp32 and from fp32 to bf16 with round-to-nearest-even.
 *
 * Workload shape (PulseInfer Guide, "The Long-Context Decoding Memory Wall";
 * "SoloHead Sparse Selection"): Llama-3-shaped K/V ~ N(0,1), a fraction of
 * heavy-hitter blocks whose keys are shifted along a per-KV-head unit direction,
 * queries following an AR(1) process across decode steps.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define GAMMA 0x9E3779B97F4A7C15ULL

enum {
  SY_KIND_K = 1, SY_KIND_V = 2, SY_KIND_Q = 3, SY_KIND_HEAVY = 4, SY_KIND_DIR = 5,
  SY_KIND_RESIDENT = 6, SY_KIND_BUDGET = 7, SY_KIND_FRAC = 8, SY_KIND_MISC = 9
};

static inline uint64_t sy_mix(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
  return z ^ (z >> 31);
}

uint64_t sy_tid(int kind, int a, int b) {
  return ((uint64_t)(uint32_t)kind << 56) ^ ((uint64_t)(uint32_t)a << 28) ^ (uint64_t)(uint32_t)b;
}

static inline uint64_t sy_base(uint64_t seed, uint64_t tid) { return sy_mix(seed ^ sy_mix(tid + GAMMA)); }

static inline uint64_t sy_at(uint64_t base, uint64_t idx) { return sy_mix(base + (idx + 1ULL) * GAMMA); }

uint64_t sy_u64(uint64_t seed, uint64_t tid, uint64_t idx) { return sy_at(sy_base(seed, tid), idx); }

/* uniform in [0, 1) with 53 random bits */
static inline double sy_unit(uint64_t x) { return (double)(x >> 11) * (1.0 / 9007199254740992.0); }

/* Box-Muller pair from stream elements 2p and 2p+1 */
static inline void sy_normal_pair(uint64_t base, uint64_t p, double* z0, double* z1) {
  double u1 = 1.0 - sy_unit(sy_at(base, 2 * p));     /* (0, 1] */
  double u2 = sy_unit(sy_at(base, 2 * p + 1));       /* [0, 1) */
  double r = sqrt(-2.0 * log(u1));
  double a = 6.283185307179586476925286766559 * u2;
  *z0 = r * cos(a);
  *z1 = r * sin(a);
}

double sy_normal(uint64_t seed, uint64_t tid, uint64_t idx) {
  double z0, z1;
  sy_normal_pair(sy_base(seed, tid), idx >> 1, &z0, &z1);
  return (idx & 1) ? z1 : z0;
}

/* fp32 -> bf16 bits, round to nearest even (finite inputs) */
static inline uint16_t sy_f32_to_bf16(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  if ((u & 0x7F800000u) == 0x7F800000u) return (uint16_t)((u >> 16) | ((u & 0xFFFF) ? 0x40 : 0));
  uint32_t lsb = (u >> 16) & 1u;
  u += 0x7FFFu + lsb;
  return (uint16_t)(u >> 16);
}

uint16_t sy_bf16_of_double(double x) { return sy_f32_to_bf16((float)x); }

/* n normals of one stream, rounded to bf16 */
void sy_normal_bf16(uint64_t seed, uint64_t tid, uint64_t start, int64_t n, uint16_t* out) {
  uint64_t base = sy_base(seed, tid);
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; i++) {
    uint64_t idx = start + (uint64_t)i;
    double z0, z1;
    sy_normal_pair(base, idx >> 1, &z0, &z1);
    out[i] = sy_f32_to_bf16((float)((idx & 1) ? z1 : z0));
  }
}

/* Heavy-hitter block mask of one (host layer, request): round(frac * nb)
 * distinct blocks drawn by a partial Fisher-Yates shuffle of 0..nb-1. */
int sy_heavy_mask(uint64_t seed, int hl, int r, int nb, double frac, uint8_t* mask) {
  int nh = (int)floor(frac * (double)nb + 0.5);
  if (nh > nb) nh = nb;
  memset(mask, 0, (size_t)nb);
  if (nh <= 0) return 0;
  int* perm = (int*)malloc(sizeof(int) * (size_t)nb);
  if (!perm) return -1;
  for (int i = 0; i < nb; i++) perm[i] = i;
  uint64_t base = sy_base(seed, sy_tid(SY_KIND_HEAVY, hl, r));
  for (int i = 0; i < nh; i++) {
    int j = i + (int)(sy_at(base, (uint64_t)i) % (uint64_t)(nb - i));
    int t = perm[i]; perm[i] = perm[j]; perm[j] = t;
  }
  for (int i = 0; i < nh; i++) mask[perm[i]] = 1;
  free(perm);
  return nh;
}

/* Unit direction (fp64) of one (host layer, request, kv head) for the shift */
void sy_direction(uint64_t seed, int hl, int r, int g, int D, double* u) {
  uint64_t tid = sy_tid(SY_KIND_DIR, hl, r);
  double s = 0.0;
  for (int d = 0; d < D; d++) { u[d] = sy_normal(seed, tid, (uint64_t)g * (uint64_t)D + (uint64_t)d); s += u[d] * u[d]; }
  double inv = 1.0 / sqrt(s);
  for (int d = 0; d < D; d++) u[d] *= inv;
}

/*
 * Fill the host KV region of one (host layer hl, request r):
 *   dst[b][g][kv][t][d] bf16, b < max_blocks, kv 0 = K, 1 = V.
 * Token tt = b*B + t (tt < ntok) takes K = N(0,1) (+ shift * u_g if its block is
 * heavy) and V = N(0,1), keyed by (tt*Hkv + g)*D + d so values do not depend on
 * the block size. Slots past ntok are zero.
 */
int sy_fill_kv(uint64_t seed, int hl, int r, int ntok, int max_blocks, int Hkv, int B, int D,
               double heavy_frac, double heavy_shift, uint16_t* dst) {
  if (D % 2) return -1;
  int nb0 = (ntok + B - 1) / B;
  if (nb0 > max_blocks) return -2;
  uint8_t* mask = (uint8_t*)calloc((size_t)(max_blocks > 0 ? max_blocks : 1), 1);
  double* dir = (double*)calloc((size_t)Hkv * (size_t)D, sizeof(double));
  if (!mask || !dir) { free(mask); free(dir); return -3; }
  if (heavy_frac > 0.0) {
    if (sy_heavy_mask(seed, hl, r, nb0, heavy_frac, mask) < 0) { free(mask); free(dir); return -3; }
    for (int g = 0; g < Hkv; g++) sy_direction(seed, hl, r, g, D, dir + (size_t)g * D);
  }
  uint64_t bk = sy_base(seed, sy_tid(SY_KIND_K, hl, r));
  uint64_t bv = sy_base(seed, sy_tid(SY_KIND_V, hl, r));
  const size_t blk = (size_t)Hkv * 2 * B * D;
#pragma omp parallel for schedule(dynamic, 4)
  for (int b = 0; b < max_blocks; b++) {
    uint16_t* out = dst + (size_t)b * blk;
    for (int g = 0; g < Hkv; g++) {
      uint16_t* ko = out + ((size_t)g * 2 + 0) * B * D;
      uint16_t* vo = out + ((size_t)g * 2 + 1) * B * D;
      const double* u = dir + (size_t)g * D;
      for (int t = 0; t < B; t++) {
        int tt = b * B + t;
        if (tt >= ntok) {
          memset(ko + (size_t)t * D, 0, (size_t)D * 2);
          memset(vo + (size_t)t * D, 0, (size_t)D * 2);
          continue;
        }
        uint64_t e0 = ((uint64_t)tt * (uint64_t)Hkv + (uint64_t)g) * (uint64_t)D;
        for (int d = 0; d < D; d += 2) {
          double k0, k1, v0, v1;
          sy_normal_pair(bk, (e0 + (uint64_t)d) >> 1, &k0, &k1);
          sy_normal_pair(bv, (e0 + (uint64_t)d) >> 1, &v0, &v1);
          if (mask[b]) { k0 += heavy_shift * u[d]; k1 += heavy_shift * u[d + 1]; }
          ko[(size_t)t * D + d] = sy_f32_to_bf16((float)k0);
          ko[(size_t)t * D + d + 1] = sy_f32_to_bf16((float)k1);
          vo[(size_t)t * D + d] = sy_f32_to_bf16((float)v0);
          vo[(size_t)t * D + d + 1] = sy_f32_to_bf16((float)v1);
        }
      }
    }
  }
  free(mask);
  free(dir);
  return 0;
}

/* K and V of one appended token tt of (hl, r): k_out[g][d], v_out[g][d] (no shift) */
void sy_token_kv(uint64_t seed, int hl, int r, int tt, int Hkv, int D, uint16_t* k_out, uint16_t* v_out) {
  uint64_t bk = sy_base(seed, sy_tid(SY_KIND_K, hl, r));
  uint64_t bv = sy_base(seed, sy_tid(SY_KIND_V, hl, r));
  for (int g = 0; g < Hkv; g++) {
    uint64_t e0 = ((uint64_t)tt * (uint64_t)Hkv + (uint64_t)g) * (uint64_t)D;
    for (int d = 0; d < D; d += 2) {
      double k0, k1, v0, v1;
      sy_normal_pair(bk, (e0 + (uint64_t)d) >> 1, &k0, &k1);
      sy_normal_pair(bv, (e0 + (uint64_t)d) >> 1, &v0, &v1);
      k_out[g * D + d] = sy_f32_to_bf16((float)k0);
      k_out[g * D + d + 1] = sy_f32_to_bf16((float)k1);
      v_out[g * D + d] = sy_f32_to_bf16((float)v0);
      v_out[g * D + d + 1] = sy_f32_to_bf16((float)v1);
    }
  }
}

/*
 * Queries of `steps` decode steps for (layer l, request r): AR(1) per element,
 * x_0 = z_0, x_s = rho*x_{s-1} + sqrt(1-rho^2)*z_s, state kept in fp32 and
 * rounded to bf16 each step. out[s][h][d], with row stride `step_stride`
 * elements between consecutive steps.
 */
void sy_q_ar1(uint64_t seed, int l, int r, int Hq, int D, int steps, double rho, uint16_t* out,
              int64_t step_stride) {
  uint64_t base = sy_base(seed, sy_tid(SY_KIND_Q, l, r));
  double c = sqrt(1.0 - rho * rho);
  int E = Hq * D;
  for (int e = 0; e < E; e++) {
    float x = 0.0f;
    for (int s = 0; s < steps; s++) {
      uint64_t idx = (uint64_t)s * (uint64_t)E + (uint64_t)e;
      double z0, z1;
      sy_normal_pair(base, idx >> 1, &z0, &z1);
      double z = (idx & 1) ? z1 : z0;
      x = (s == 0) ? (float)z : (float)(rho * (double)x + c * z);
      out[(int64_t)s * step_stride + e] = sy_f32_to_bf16(x);
    }
  }
}

/* integer uniform in [lo, hi] (inclusive) of stream (kind, a, b) at idx */
int64_t sy_uniform_int(uint64_t seed, int kind, int a, int b, uint64_t idx, int64_t lo, int64_t hi) {
  uint64_t span = (uint64_t)(hi - lo + 1);
  return lo + (int64_t)(sy_u64(seed, sy_tid(kind, a, b), idx) % span);
}

/* real uniform in [lo, hi) of stream (kind, a, b) at idx */
double sy_uniform_real(uint64_t seed, int kind, int a, int b, uint64_t idx, double lo, double hi) {
  return lo + (hi - lo) * sy_unit(sy_u64(seed, sy_tid(kind, a, b), idx));
}

/* n distinct values of 0..nb-1 (partial Fisher-Yates of stream (kind, a, b)),
 * written sorted ascending; used for initial pool residency samples */
int sy_sample_sorted(uint64_t seed, int kind, int a, int b, int nb, int n, int* out, int* scratch) {
  if (n > nb) n = nb;
  for (int i = 0; i < nb; i++) scratch[i] = i;
  uint64_t base = sy_base(seed, sy_tid(kind, a, b));
  for (int i = 0; i < n; i++) {
    int j = i + (int)(sy_at(base, (uint64_t)i) % (uint64_t)(nb - i));
    int t = scratch[i]; scratch[i] = scratch[j]; scratch[j] = t;
  }
  /* insertion into a 0/1 map keeps it sorted without a library sort */
  for (int i = 0; i < nb; i++) out[i] = 0;
  for (int i = 0; i < n; i++) out[scratch[i]] = 1;
  int m = 0;
  for (int i = 0; i < nb; i++) if (out[i]) scratch[m++] = i;
  for (int i = 0; i < n; i++) out[i] = scratch[i];
  return n;
}
