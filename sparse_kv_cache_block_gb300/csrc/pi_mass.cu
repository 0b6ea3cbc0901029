// Attention-mass diagnostic: the share of each query head's full softmax
// attention that a block selection keeps.
//
// PulseInfer Guide, "SoloHead Sparse Selection", "2. High Attention Mass
// Preservation": the shared block set is judged by how much of every head's
// attention mass its blocks still hold, next to independent per-head sets.
//
// Off the decode path: every key of the layer is read from the mapped host
// store (the pool holds only the recalled blocks), so one call moves
// Hkv*ntok*D*2 bytes per request over the host link and is bound by it.
//
// Kernel 1, one CTA per (chunk of tokens, request, KV head): the selected
// blocks sit in a shared-memory bitmap; a warp reads whole key rows (D/8 lanes
// of 16 bytes per token), each lane dots its 8 elements with the group's G
// queries (fp32, in registers) and a xor tree over the row's lanes completes the
// logits; every row keeps an online (max, sum over all tokens, sum over
// selected tokens) per head, merged across the warp and the CTA by fixed trees.
// Kernel 2 merges the chunks in chunk order.
#include <math.h>

#include "pi_internal.cuh"

namespace {

constexpr int kMassThreads = 256;
constexpr int kMassChunksMax = 32;

struct MassParams {
  const uint8_t* host;      // device address of the host store
  size_t region_bytes;      // bytes of one (host layer, request) region
  int hl, layer, L, R, Hkv, G, B, max_blocks, cap, per_head, chunks;
  float scale;              // 1/sqrt(D)
  const int* ntok;          // [R][L]
  const uint16_t* q;        // [R][Hq][D] bf16
  const int* sel;           // [R][cap] or [R][Hkv][cap]
  const int* nsel;          // [R] or [R][Hkv]
  float4* part;             // [R][Hkv][chunks][G]: (m, sum all, sum selected, -)
  float* mass;              // [R][Hq]
  unsigned* status;
};

struct MassAcc {
  float m, la, ls;
};

// Fold (m2, la2, ls2) into a; a side with no tokens (m = -inf) scales by 0.
__device__ __forceinline__ void mass_fold(MassAcc& a, float m2, float la2, float ls2) {
  const float M = fmaxf(a.m, m2);
  if (M == -INFINITY) return;
  const float ca = a.m == -INFINITY ? 0.f : expf(a.m - M);
  const float c2 = m2 == -INFINITY ? 0.f : expf(m2 - M);
  a.la = a.la * ca + la2 * c2;
  a.ls = a.ls * ca + ls2 * c2;
  a.m = M;
}

template <int D>
__global__ void __launch_bounds__(kMassThreads) mass_part_kernel(MassParams a) {
  extern __shared__ float4 mass_smem[];
  const int G = a.G;
  float* qf = reinterpret_cast<float*>(mass_smem);                  // [G][D]
  unsigned* bits = reinterpret_cast<unsigned*>(qf + G * D);         // [ceil(max_blocks/32)]
  float* red = reinterpret_cast<float*>(bits + ((a.max_blocks + 31) >> 5));  // [warps][G][3]

  const int unit = blockIdx.y;
  const int r = unit / a.Hkv, g = unit - r * a.Hkv;
  const int c = blockIdx.x;
  const int tid = threadIdx.x;
  const int n_tok = a.ntok[r * a.L + a.layer];
  const int nb = (n_tok + a.B - 1) / a.B;
  const int words = (a.max_blocks + 31) >> 5;

  const uint16_t* qg = a.q + ((size_t)r * a.Hkv * G + (size_t)g * G) * D;
  for (int i = tid; i < G * D; i += kMassThreads) qf[i] = __uint_as_float((uint32_t)qg[i] << 16);
  for (int i = tid; i < words; i += kMassThreads) bits[i] = 0;
  __syncthreads();
  const int su = a.per_head ? unit : r;
  int ns = a.nsel[su];
  if (ns < 0 || ns > a.cap) {
    if (tid == 0 && c == 0) pi_flag(a.status, PI_DEV_BAD_INDEX);
    ns = ns < 0 ? 0 : a.cap;
  }
  const int* sl = a.sel + (size_t)su * a.cap;
  for (int i = tid; i < ns; i += kMassThreads) {
    const int b = sl[i];
    if (b >= 0 && b < nb)
      atomicOr(&bits[b >> 5], 1u << (b & 31));
    else if (c == 0)
      pi_flag(a.status, PI_DEV_BAD_INDEX);
  }
  __syncthreads();

  // a token's key row is D/8 lanes x 16 bytes: a warp reads 32/(D/8) whole rows
  // per load instruction (full 128-byte lines over the host link); each lane
  // keeps its 8 elements of the group's queries in registers
  constexpr int LPT = D / 8;      // lanes per token
  constexpr int TPW = 32 / LPT;   // tokens per warp pass
  constexpr int kPass = 4;        // passes whose loads are in flight together
  const int lane = tid & 31, warp = tid >> 5;
  const int sub = lane / LPT, part = lane % LPT;
  float qr[8][8];
#pragma unroll
  for (int j = 0; j < 8; j++)
#pragma unroll
    for (int e = 0; e < 8; e++) qr[j][e] = (j < G) ? qf[j * D + part * 8 + e] : 0.f;

  MassAcc acc[8];
#pragma unroll
  for (int j = 0; j < 8; j++) acc[j] = {-INFINITY, 0.f, 0.f};

  const int per = (n_tok + a.chunks - 1) / a.chunks;
  const int t0 = c * per, t1 = min(n_tok, t0 + per);
  const uint8_t* region = a.host + ((size_t)a.hl * a.R + r) * a.region_bytes;
  const size_t half = (size_t)a.B * D * 2;  // one head's K (or V) of a block, bytes
  constexpr int kWarps = kMassThreads / 32;
  for (int tb = t0 + warp * kPass * TPW; tb < t1; tb += kWarps * kPass * TPW) {
    uint4 kv[kPass];
#pragma unroll
    for (int u = 0; u < kPass; u++) {
      const int t = tb + u * TPW + sub;
      kv[u] = make_uint4(0u, 0u, 0u, 0u);
      if (t < t1) {
        const int b = t / a.B, i = t - b * a.B;
        kv[u] = *reinterpret_cast<const uint4*>(region + (size_t)(b * a.Hkv + g) * 2 * half + (size_t)i * D * 2 +
                                                (size_t)part * 16);
      }
    }
#pragma unroll
    for (int u = 0; u < kPass; u++) {
      const int t = tb + u * TPW + sub;
      const uint32_t w[4] = {kv[u].x, kv[u].y, kv[u].z, kv[u].w};
      float k[8];
#pragma unroll
      for (int e = 0; e < 4; e++) {
        k[2 * e] = pi_bf16_lo(w[e]);
        k[2 * e + 1] = pi_bf16_hi(w[e]);
      }
      float z[8];
#pragma unroll
      for (int j = 0; j < 8; j++) {
        z[j] = 0.f;
        if (j < G) {
#pragma unroll
          for (int e = 0; e < 8; e++) z[j] = fmaf(qr[j][e], k[e], z[j]);
          // the row's LPT lanes: xor tree, every lane ends with the full dot
#pragma unroll
          for (int off = LPT / 2; off > 0; off >>= 1) z[j] += __shfl_xor_sync(0xffffffffu, z[j], off);
        }
      }
      if (t < t1) {
        const int b = t / a.B;
        const float in = (bits[b >> 5] >> (b & 31)) & 1u ? 1.f : 0.f;
#pragma unroll
        for (int j = 0; j < 8; j++) {
          if (j < G) {
            const float zj = z[j] * a.scale;
            if (zj > acc[j].m) {
              const float cm = acc[j].m == -INFINITY ? 0.f : expf(acc[j].m - zj);
              acc[j].la = acc[j].la * cm + 1.f;
              acc[j].ls = acc[j].ls * cm + in;
              acc[j].m = zj;
            } else {
              const float e = expf(zj - acc[j].m);
              acc[j].la += e;
              acc[j].ls += in * e;
            }
          }
        }
      }
    }
  }

  // merge across the CTA: the lanes of one row hold the same sums, so the warp
  // merges its rows (xor offsets >= LPT), then the warps in order
#pragma unroll
  for (int j = 0; j < 8; j++) {
    if (j < G) {
#pragma unroll
      for (int off = 16; off >= LPT; off >>= 1) {
        const float m2 = __shfl_xor_sync(0xffffffffu, acc[j].m, off);
        const float la2 = __shfl_xor_sync(0xffffffffu, acc[j].la, off);
        const float ls2 = __shfl_xor_sync(0xffffffffu, acc[j].ls, off);
        mass_fold(acc[j], m2, la2, ls2);
      }
      if (lane == 0) {
        float* o = red + (warp * G + j) * 3;
        o[0] = acc[j].m;
        o[1] = acc[j].la;
        o[2] = acc[j].ls;
      }
    }
  }
  __syncthreads();
  if (tid < G) {
    MassAcc s = {-INFINITY, 0.f, 0.f};
    for (int w = 0; w < kMassThreads / 32; w++) {
      const float* o = red + (w * G + tid) * 3;
      mass_fold(s, o[0], o[1], o[2]);
    }
    a.part[((size_t)unit * a.chunks + c) * G + tid] = make_float4(s.m, s.la, s.ls, 0.f);
  }
}

__global__ void mass_merge_kernel(MassParams a) {
  const int Hq = a.Hkv * a.G;
  const int idx = blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= a.R * Hq) return;
  const int r = idx / Hq, h = idx - r * Hq;
  const int g = h / a.G, j = h - g * a.G;
  MassAcc s = {-INFINITY, 0.f, 0.f};
  const float4* pp = a.part + (size_t)(r * a.Hkv + g) * a.chunks * a.G + j;
  for (int c = 0; c < a.chunks; c++) {
    const float4 v = pp[(size_t)c * a.G];
    mass_fold(s, v.x, v.y, v.z);
  }
  a.mass[idx] = s.la > 0.f ? s.ls / s.la : 0.f;
}

}  // namespace

extern "C" pi_status pi_attention_mass(pi_pool* p, int layer, const void* q, const int* sel, const int* nsel,
                                       int per_head, float* mass, pi_stream s) {
  if (!p || layer < 0 || layer >= p->L || !q || !sel || !nsel || !mass) return PI_ERR_INVALID;
  if (per_head != 0 && per_head != 1) return PI_ERR_INVALID;
  if (reinterpret_cast<uintptr_t>(q) & 1) return PI_ERR_INVALID;
  const size_t part_per_layer = (size_t)p->R * p->Hq * kMassChunksMax;
  if (!p->mass_part) {
    if (cudaMalloc(reinterpret_cast<void**>(&p->mass_part), part_per_layer * p->L * sizeof(float4)) != cudaSuccess) {
      cudaGetLastError();
      p->mass_part = nullptr;
      return PI_ERR_OOM;
    }
  }
  MassParams a{};
  a.host = p->host_dev;
  a.region_bytes = p->region_bytes;
  a.hl = layer % p->host_layers;
  a.layer = layer;
  a.L = p->L;
  a.R = p->R;
  a.Hkv = p->Hkv;
  a.G = p->G;
  a.B = p->B;
  a.max_blocks = p->max_blocks;
  a.cap = p->cap;
  a.per_head = per_head;
  const int units = p->R * p->Hkv;
  a.chunks = std::max(1, std::min(kMassChunksMax, (2 * p->num_sms + units - 1) / units));
  a.scale = 1.0f / sqrtf((float)p->D);
  a.ntok = p->ntok;
  a.q = static_cast<const uint16_t*>(q);
  a.sel = sel;
  a.nsel = nsel;
  a.part = p->mass_part + part_per_layer * layer;
  a.mass = mass;
  a.status = p->dev_status;
  const size_t smem = (size_t)p->G * p->D * sizeof(float) + (size_t)((p->max_blocks + 31) >> 5) * sizeof(unsigned) +
                      (size_t)(kMassThreads / 32) * p->G * 3 * sizeof(float);
  cudaStream_t st = reinterpret_cast<cudaStream_t>(s);
  dim3 grid(a.chunks, units);
  if (p->D == 128)
    mass_part_kernel<128><<<grid, kMassThreads, smem, st>>>(a);
  else
    mass_part_kernel<64><<<grid, kMassThreads, smem, st>>>(a);
  PI_CUDA_TRY(cudaGetLastError());
  const int n = p->R * p->Hq;
  mass_merge_kernel<<<(n + 255) / 256, 256, 0, st>>>(a);
  PI_CUDA_TRY(cudaGetLastError());
  return PI_OK;
}
