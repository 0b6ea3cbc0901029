// Block summaries, token append and SoloHead-style shared top-k selection.
//
// "PulseInfer Guide: I/O-Centric Sparse KV Cache Offloading", section "SoloHead
// Sparse Selection": one block set is chosen for all heads of a layer so a
// recall moves whole blocks instead of per-head fragments. The guide leaves the
// per-block importance undefined; this library scores a block by
// sum_h q_h . kmean[b, h/G] in fp32, where kmean is the per-KV-head mean key of
// the block (the summary kept for every block), and keeps the W most recent
// blocks unconditionally.
//
// Bit-exact contract with the CPU oracle: summaries are a sequential fp32 sum in
// token order divided by the token count (IEEE division); the score uses one
// fixed fp32 order (per-lane fused multiply-add over elements 128c+4*lane+j,
// then a xor butterfly); ties go to the lower block index.
//
// A selection is a set of work items (a chunk of one unit's candidates); the
// stand-alone kernel runs one item per CTA, the fused select + gather kernel
// lets a few CTAs claim the items one after another and then copy the recalls.
#include <map>
#include <mutex>
#include <tuple>

#include "pi_gather.cuh"
#include "pi_internal.cuh"
#include "pi_plan.cuh"

namespace {

constexpr int kSelThreads = 256;

// ------------------------------------------------------------------ a-1
// grid (blocks in range, R); one thread per 8 consecutive elements of one head.
// The keys come from the host store through the GPU's mapping (or from device
// memory): each thread keeps eight 16-byte token rows in flight, then adds them
// in token order, so the sum is the sequential fp32 sum.
constexpr int kSumDepth = 8;
__global__ void summaries_kernel(const uint8_t* __restrict__ src, long long src_req_stride,
                                 const int* __restrict__ ntok_new, int* __restrict__ ntok, float* __restrict__ kmean,
                                 float* __restrict__ tail_sum, int layer, int L, int Hkv, int B, int D, int max_blocks,
                                 int b0) {
  const int r = blockIdx.y;
  const int nt = ntok_new[r];
  if (blockIdx.x == 0 && threadIdx.x == 0) ntok[(size_t)r * L + layer] = nt;
  const int nb = (nt + B - 1) / B;
  const int b = b0 + blockIdx.x;
  if (b >= nb) return;
  const int nv = min(B, nt - b * B);
  const int e = threadIdx.x * 8;
  if (e >= Hkv * D) return;
  const int g = e / D, d = e % D;
  const size_t block_bytes = (size_t)Hkv * 2 * B * D * 2;
  const uint8_t* row = src + (size_t)r * src_req_stride + (size_t)b * block_bytes + ((size_t)g * 2 * B * D + d) * 2;
  float s[8];
#pragma unroll
  for (int j = 0; j < 8; j++) s[j] = 0.0f;
  for (int t0 = 0; t0 < nv; t0 += kSumDepth) {
    uint4 v[kSumDepth];
#pragma unroll
    for (int k = 0; k < kSumDepth; k++)
      if (t0 + k < nv) v[k] = pi_ld_stream(reinterpret_cast<const uint4*>(row + (size_t)(t0 + k) * D * 2));
#pragma unroll
    for (int k = 0; k < kSumDepth; k++) {
      if (t0 + k >= nv) break;
      const uint32_t w[4] = {v[k].x, v[k].y, v[k].z, v[k].w};
#pragma unroll
      for (int j = 0; j < 4; j++) {
        s[2 * j] = __fadd_rn(s[2 * j], pi_bf16_lo(w[j]));
        s[2 * j + 1] = __fadd_rn(s[2 * j + 1], pi_bf16_hi(w[j]));
      }
    }
  }
  const size_t rl = (size_t)r * L + layer;
  float* km = kmean + ((rl * max_blocks + b) * Hkv + g) * D + d;
  const float fn = (float)nv;
  float m[8];
#pragma unroll
  for (int j = 0; j < 8; j++) m[j] = __fdiv_rn(s[j], fn);
  reinterpret_cast<float4*>(km)[0] = make_float4(m[0], m[1], m[2], m[3]);
  reinterpret_cast<float4*>(km)[1] = make_float4(m[4], m[5], m[6], m[7]);
  if (b == nb - 1) {
    float* ts = tail_sum + (rl * Hkv + g) * D + d;
    reinterpret_cast<float4*>(ts)[0] = make_float4(s[0], s[1], s[2], s[3]);
    reinterpret_cast<float4*>(ts)[1] = make_float4(s[4], s[5], s[6], s[7]);
  }
}

// ------------------------------------------------------------------ a-7
struct AppendParams {
  const uint8_t* k_new;
  const uint8_t* v_new;
  uint8_t* host_dev;      // device address of the host store
  uint8_t* pool;
  const long long* slot_base;
  const int* P;
  const int* slot_of;
  int* ntok;
  float* kmean;
  float* tail_sum;
  unsigned* status;
  int layer, L, R, Hkv, B, D, U, max_blocks, host_layer;
  int r0;                 // first request of this launch (one CTA per request)
  int write_host;         // 0: the decode-step gather writes the host copy instead
};

// grid R; one thread per 8 consecutive elements of one head
__global__ void append_kernel(AppendParams a) {
  const int r = a.r0 + blockIdx.x;
  const size_t rl = (size_t)r * a.L + a.layer;
  const int t = a.ntok[rl];
  const int b = t / a.B, tp = t % a.B;
  const int e = threadIdx.x * 8;
  const bool active = e < a.Hkv * a.D;
  if (b >= a.max_blocks) {
    if (threadIdx.x == 0) pi_flag(a.status, PI_DEV_BAD_INDEX);
    return;
  }
  if (active) {
    const int g = e / a.D, d = e % a.D;
    const size_t block_bytes = (size_t)a.Hkv * 2 * a.B * a.D * 2;
    const uint4 kv = *reinterpret_cast<const uint4*>(a.k_new + (((size_t)r * a.Hkv + g) * a.D + d) * 2);
    const uint4 vv = *reinterpret_cast<const uint4*>(a.v_new + (((size_t)r * a.Hkv + g) * a.D + d) * 2);
    const size_t in_block_k = (((size_t)g * 2 + 0) * a.B + tp) * a.D * 2 + (size_t)d * 2;
    const size_t in_block_v = (((size_t)g * 2 + 1) * a.B + tp) * a.D * 2 + (size_t)d * 2;
    uint8_t* host_blk =
        a.host_dev + (((size_t)a.host_layer * a.R + r) * a.max_blocks + b) * block_bytes;
    if (a.write_host) {
      *reinterpret_cast<uint4*>(host_blk + in_block_k) = kv;
      *reinterpret_cast<uint4*>(host_blk + in_block_v) = vv;
    }
    const int u = (a.U == 1) ? 0 : g;
    const int slot = a.slot_of[(rl * a.U + u) * a.max_blocks + b];
    if (slot >= 0) {
      if (slot >= a.P[rl]) {
        pi_flag(a.status, PI_DEV_BAD_INDEX);
      } else {
        const long long gs = a.slot_base[rl] + slot;
        uint8_t* pool_blk = a.pool + (size_t)gs * block_bytes;
        *reinterpret_cast<uint4*>(pool_blk + in_block_k) = kv;
        *reinterpret_cast<uint4*>(pool_blk + in_block_v) = vv;
      }
    }
    // running fp32 sum of the block's keys in token order == a fresh sequential sum
    float* ts = a.tail_sum + (rl * a.Hkv + g) * a.D + d;
    float* km = a.kmean + ((rl * a.max_blocks + b) * a.Hkv + g) * a.D + d;
    const uint32_t w[4] = {kv.x, kv.y, kv.z, kv.w};
    const float fn = (float)(tp + 1);
#pragma unroll
    for (int j = 0; j < 4; j++) {
      float s0 = (tp == 0) ? 0.0f : ts[2 * j];
      float s1 = (tp == 0) ? 0.0f : ts[2 * j + 1];
      s0 = __fadd_rn(s0, pi_bf16_lo(w[j]));
      s1 = __fadd_rn(s1, pi_bf16_hi(w[j]));
      ts[2 * j] = s0;
      ts[2 * j + 1] = s1;
      km[2 * j] = __fdiv_rn(s0, fn);
      km[2 * j + 1] = __fdiv_rn(s1, fn);
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) a.ntok[rl] = t + 1;
}

// ------------------------------------------------------------------ a-2
struct SelParams {
  const uint16_t* q;
  const int* k_per_req;
  int* sel;
  int* nsel;
  const float* kmean;
  const int* ntok;
  float* scores;       // [R*U][max_blocks] for this layer
  unsigned* counter;   // [R*U] for this layer
  unsigned* status;
  int layer, L, Hq, Hkv, G, D, B, max_blocks, W, k_max, cap, U, bpc;
  // fused recall plan (decode-step pipeline); table == nullptr disables it
  int* table;
  const int* slot_of;
  const int* block_of;
  const int* P;
  int* plan_n;
  int4* plan;
  long long* counts;
  int p_max;
  int* slot_stamp;     // least-recently-selected policy, else nullptr
  int* epoch;
  int lru_p2;
  int map_cache_blocks;  // fused plan: blocks of slot_of_block cached in shared memory (0: read global)
  int map_cache_slots;   // and slots of block_of_slot
  int u0;                // first unit of this launch (grid.y covers u0 ..)
  int consensus;         // rank blocks by the consensus score (shared selection only)
  float lambda;          // its weight on the group mean
  int ring_stages;       // consensus: bulk-copy stages of 8 blocks' summaries
  int dyn_plan_off;      // bytes of dynamic shared memory before the plan scratch (consensus: ring + c_g)
  int empty_first;       // the layer is held whole in HBM
  int q_vec;             // q is 16-byte aligned: the query sums load 16 bytes at a time
  int binned_off;        // last-CTA top-k by value bins: its scratch (keys, bins, list, state) at this
                         // byte offset of dynamic shared memory, sized for binned_cap candidates (0: radix)
  int binned_cap;
};

__device__ __forceinline__ uint32_t order_key(float f) {
  uint32_t u = __float_as_uint(f);
  if ((u << 1) == 0) u = 0;  // -0.0 ranks as +0.0
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

constexpr int kKeysPerThread = 16;  // candidates a thread keeps in registers (4096 per CTA)

// Consensus ranking ("PulseInfer Guide", "SoloHead Sparse Selection", "1.
// Consensus Scoring Mechanism"): per GQA group g, c_g = max_h S(h, b) + lambda x
// (sum_h S(h, b) / G) with S(h, b) = q_h . kmean[b, g]; the block's score is
// the sum of c_g over g ascending. The CTA streams its candidates' summaries
// through a ring of bulk-copy stages (8 blocks each); warp w owns one 128-float
// chunk of [Hkv][D] (one group for D = 128, two for D = 64) and keeps its lanes'
// query values of that chunk's heads in registers. Per (block, chunk): lane i of
// a group holds the partial dot of each head over d = 4i .. 4i+3 (fused
// multiply-add); the group's P = pow2(G) head sums are formed by a reduce-
// scatter (each round a lane keeps half its values and adds its partner's at
// the same positions) and butterfly rounds, so head j ends in lane j*(n/P); the
// max is a butterfly max, the sum a pairwise tree over the padded heads. Every
// step is rounded exactly as the oracle's fixed order prescribes.
// Shape of the reduction for one lane, fixed for a warp (n = D/4 lanes per
// group, P = pow2(G); every offset a power of two).
struct ConsShape {
  int off[3];      // reduce-scatter offset of the rounds with 8, 4, 2 values (0: round skipped)
  int bfly;        // first butterfly offset after the scatter, n / (2P) (0: none)
  int tree;        // lane distance between neighbouring heads, n / P
  int n;           // lanes per group
  int jh;          // the head this lane holds after the scatter
  int G;
  float inv_g;     // 1 / G when G is a power of two (exact), else 0: divide
};

__device__ __forceinline__ ConsShape cons_shape(int lane, int D, int G) {
  ConsShape c;
  c.n = D / 4;
  int P = 1, lgP = 0;
  while (P < G) {
    P <<= 1;
    lgP++;
  }
  int lgn = (D == 128) ? 5 : 4;
#pragma unroll
  for (int lv = 0; lv < 3; lv++) {
    const int lgm = 3 - lv;  // rounds with m = 2^lgm values
    c.off[lv] = (lgm <= lgP) ? (1 << (lgn + lgm - 1 - lgP)) : 0;
  }
  c.bfly = (lgn - 1 - lgP >= 0) ? (1 << (lgn - 1 - lgP)) : 0;
  c.tree = 1 << (lgn - lgP);
  c.jh = (lane & (c.n - 1)) >> (lgn - lgP);
  c.G = G;
  c.inv_g = (P == G) ? 1.0f / (float)G : 0.0f;
  return c;
}

__device__ __forceinline__ float consensus_chunk(const float4 k4, const float4 (&qv)[8], bool valid, int lane,
                                                 const ConsShape& cs, float lambda) {
  float a[8];
#pragma unroll
  for (int j = 0; j < 8; j++) {
    a[j] = 0.0f;
    if (j < cs.G && valid) {
      a[j] = __fmaf_rn(qv[j].x, k4.x, a[j]);
      a[j] = __fmaf_rn(qv[j].y, k4.y, a[j]);
      a[j] = __fmaf_rn(qv[j].z, k4.z, a[j]);
      a[j] = __fmaf_rn(qv[j].w, k4.w, a[j]);
    }
  }
#pragma unroll
  for (int lv = 0; lv < 3; lv++) {
    const int h = 4 >> lv;  // values kept this round
    const int off = cs.off[lv];
    if (off == 0) continue;
    const bool up = (lane & off) != 0;
#pragma unroll
    for (int x = 0; x < h; x++) {
      const float send = up ? a[x] : a[x + h];
      const float keep = up ? a[x + h] : a[x];
      a[x] = __fadd_rn(keep, __shfl_xor_sync(0xffffffffu, send, off));
    }
  }
#pragma unroll
  for (int k = 0; k < 5; k++) {
    const int off = cs.bfly >> k;
    if (off == 0) break;
    a[0] = __fadd_rn(a[0], __shfl_xor_sync(0xffffffffu, a[0], off));
  }
  float mv = (cs.jh < cs.G) ? a[0] : -INFINITY;
  float sv = (cs.jh < cs.G) ? a[0] : 0.0f;
#pragma unroll
  for (int k = 0; k < 3; k++) {
    const int o = cs.tree << k;
    if (o >= cs.n) break;
    mv = fmaxf(mv, __shfl_xor_sync(0xffffffffu, mv, o));
    sv = __fadd_rn(sv, __shfl_xor_sync(0xffffffffu, sv, o));
  }
  const float mean = (cs.inv_g != 0.0f) ? __fmul_rn(sv, cs.inv_g) : __fdiv_rn(sv, (float)cs.G);
  return __fadd_rn(mv, __fmul_rn(lambda, mean));
}

// dst[0..n) = src[0..n): PER loads per thread in flight before the first store
template <int PER>
__device__ __forceinline__ void stage_ints(int* dst, const int* src, int n) {
  for (int base = 0; base < n; base += PER * kSelThreads) {
    int v[PER];
#pragma unroll
    for (int i = 0; i < PER; i++) {
      const int j = base + threadIdx.x + i * kSelThreads;
      v[i] = (j < n) ? __ldcg(src + j) : 0;
    }
#pragma unroll
    for (int i = 0; i < PER; i++) {
      const int j = base + threadIdx.x + i * kSelThreads;
      if (j < n) dst[j] = v[i];
    }
  }
}

// One work item of a selection: the scores of chunk `chunk` (of nchunks) of unit
// u's candidates; the CTA that finishes the unit's last chunk then runs its
// top-k (and, with a table, its recall plan) and returns true. Every branch is
// uniform across the CTA; a CTA may run several items one after another.
// Scores of unit u's candidates [b_begin, b_end): sink(b, score) once per block,
// from one thread. Every branch is uniform across the CTA (it synchronises).
template <class Sink>
__device__ __forceinline__ void select_score(const SelParams& p, const int u, const int b_begin, const int b_end,
                                             Sink&& sink) {
  __shared__ __align__(16) float qs[1024];
  extern __shared__ __align__(16) uint32_t dyn[];  // consensus ring + group scores first
  const int r = u / p.U;
  const int g = (p.U == 1) ? 0 : u % p.U;
  const int E = (p.U == 1) ? p.Hkv * p.D : p.D;
  const int goff = (p.U == 1) ? 0 : g * p.D;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const size_t rl = (size_t)r * p.L + p.layer;
  constexpr int NW = kSelThreads / 32;

  // mean-key scores of one block set per request may stream the candidates'
  // summaries through a ring of bulk-copy stages (NW blocks per stage, one per
  // warp): the first stages are in flight while the query sums are formed
  const bool mk_ring = !p.consensus && p.ring_stages > 0;
  const int mk_nblk = max(0, b_end - b_begin);
  const int mk_nst = (mk_nblk + NW - 1) / NW;
  const int mk_stage = NW * E * 4;
  uint8_t* mk_ring_base = reinterpret_cast<uint8_t*>(dyn);
  uint64_t* mk_full = reinterpret_cast<uint64_t*>(mk_ring_base + (size_t)p.ring_stages * mk_stage);
  const float* mk_src = p.kmean + (rl * p.max_blocks + (size_t)b_begin) * E;
  auto mk_issue = [&](int it) {
    const int st = it % p.ring_stages;
    const unsigned bytes = (unsigned)(min(NW, mk_nblk - it * NW) * E * 4);
    pi_mbar_arrive_expect_tx(&mk_full[st], bytes);
    pi_bulk_load(mk_ring_base + (size_t)st * mk_stage, mk_src + (size_t)it * NW * E, bytes, &mk_full[st]);
  };
  if (mk_ring && b_begin + mk_nblk > p.max_blocks) {
    // a range past the unit's summaries is never copied (recorded, nothing scored)
    if (threadIdx.x == 0) pi_flag(p.status, PI_DEV_LAUNCH_SIZE);
    return;
  }
  // the ring's first stages are issued at once by the first thread that has no
  // query elements to load (with 16-byte query loads, thread E/8), so neither
  // waits for the other; without such a thread, thread 0 issues them right
  // after its query loads
  const int ring_thread = (!p.consensus && p.q_vec && E / 8 < kSelThreads) ? E / 8 : 0;
  auto mk_start = [&]() {
    if (mk_ring && threadIdx.x == ring_thread) {
      for (int st = 0; st < p.ring_stages; st++) pi_mbar_init(&mk_full[st], 1);
      pi_fence_barrier_init();
      for (int it = 0; it < min(p.ring_stages, mk_nst); it++) mk_issue(it);
    }
  };

  // qsum[e] = sum over the group's query heads (ascending) of q[h][d], fp32
  // (the mean-key score; the consensus ranking reads the heads one by one). A
  // thread takes 8 consecutive elements and loads each head's 16 bytes of them
  // at once (every load in flight before the first sum); queries that are not
  // 16-byte aligned take the element-wise loop.
  if (!p.consensus && p.q_vec) {
    const int e0 = threadIdx.x * 8;
    if (e0 < E) {
      const int gg = (p.U == 1) ? e0 / p.D : g;
      const uint16_t* qh = p.q + ((size_t)r * p.Hq + (size_t)gg * p.G) * p.D + e0 % p.D;
      uint4 v[8];
#pragma unroll
      for (int j = 0; j < 8; j++)
        if (j < p.G) v[j] = *reinterpret_cast<const uint4*>(qh + (size_t)j * p.D);
      mk_start();
      float acc[8];
#pragma unroll
      for (int i = 0; i < 8; i++) acc[i] = 0.0f;
#pragma unroll
      for (int j = 0; j < 8; j++) {
        if (j >= p.G) break;
        const uint32_t w[4] = {v[j].x, v[j].y, v[j].z, v[j].w};
#pragma unroll
        for (int i = 0; i < 4; i++) {
          acc[2 * i] = __fadd_rn(acc[2 * i], pi_bf16_lo(w[i]));
          acc[2 * i + 1] = __fadd_rn(acc[2 * i + 1], pi_bf16_hi(w[i]));
        }
      }
      reinterpret_cast<float4*>(qs + e0)[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
      reinterpret_cast<float4*>(qs + e0)[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
    } else {
      mk_start();
    }
  } else {
    mk_start();
    for (int e = threadIdx.x; e < E && !p.consensus; e += kSelThreads) {
      const int gg = (p.U == 1) ? e / p.D : g;
      const int d = e % p.D;
      const uint16_t* qh = p.q + ((size_t)r * p.Hq + (size_t)gg * p.G) * p.D + d;
      float s = 0.0f;
      for (int j = 0; j < p.G; j++) s = __fadd_rn(s, __uint_as_float((uint32_t)qh[(size_t)j * p.D] << 16));
      qs[e] = s;
    }
  }
  __syncthreads();

  // scores of this CTA's candidates: one warp per block, canonical lane order,
  // two blocks per pass so sixteen 16-byte loads per lane are in flight (or from
  // the ring)
  const int chunks = (E + 127) / 128;
  if (mk_ring) {
    float4 qv[8];  // this lane's query sums of chunk c: elements 128c + 4 lane .. +3
#pragma unroll
    for (int c = 0; c < 8; c++) {
      const int e = 128 * c + 4 * lane;
      qv[c] = (c < chunks && e < E) ? *reinterpret_cast<const float4*>(qs + e) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    bool ok = true;
    for (int it = 0; it < mk_nst; it++) {
      const int st = it % p.ring_stages;
      if (!pi_mbar_wait_bounded(&mk_full[st], (it / p.ring_stages) & 1, p.status)) ok = false;
      const int nb_it = min(NW, mk_nblk - it * NW);
      if (ok && warp < nb_it) {
        const float* kb = reinterpret_cast<const float*>(mk_ring_base + (size_t)st * mk_stage) + (size_t)warp * E;
        float acc = 0.0f;
#pragma unroll
        for (int c = 0; c < 8; c++) {
          const int e = 128 * c + 4 * lane;
          if (c < chunks && e < E) {
            const float4 k4 = *reinterpret_cast<const float4*>(kb + e);
            acc = __fmaf_rn(qv[c].x, k4.x, acc);
            acc = __fmaf_rn(qv[c].y, k4.y, acc);
            acc = __fmaf_rn(qv[c].z, k4.z, acc);
            acc = __fmaf_rn(qv[c].w, k4.w, acc);
          }
        }
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) acc = __fadd_rn(acc, __shfl_xor_sync(0xffffffffu, acc, off));
        if (lane == 0) sink(b_begin + it * NW + warp, acc);
      }
      // every warp is done with stage st: refill it (a failed wait stops the ring)
      ok = __syncthreads_and(ok) != 0;
      if (!ok) break;
      if (threadIdx.x == 0 && it + p.ring_stages < mk_nst) mk_issue(it + p.ring_stages);
    }
    if (!ok && threadIdx.x == 0)
      for (int it = 0; it < mk_nst; it++) pi_mbar_wait_bounded(&mk_full[it % p.ring_stages], (it / p.ring_stages) & 1, p.status);
    __syncthreads();
    if (threadIdx.x == 0)
      for (int st = 0; st < p.ring_stages; st++) pi_mbar_inval(&mk_full[st]);
    return;
  }
  if (p.consensus) {
    // ring of bulk-copy stages of NW blocks' summaries; then the groups' c_g
    // per block in shared memory, summed over the groups at the end
    const int NS = p.ring_stages;
    const int stage_bytes = NW * E * 4;
    uint8_t* ring = reinterpret_cast<uint8_t*>(dyn);
    uint64_t* full = reinterpret_cast<uint64_t*>(ring + (size_t)NS * stage_bytes);
    float* cg_s = reinterpret_cast<float*>(full + NS);  // [bpc][Hkv]
    const int nblk = max(0, b_end - b_begin);
    const int nst = (nblk + NW - 1) / NW;
    const float* src0 = p.kmean + (rl * p.max_blocks + (size_t)b_begin) * E;
    auto issue = [&](int it) {
      const int s = it % NS;
      const unsigned bytes = (unsigned)(min(NW, nblk - it * NW) * E * 4);
      pi_mbar_arrive_expect_tx(&full[s], bytes);
      pi_bulk_load(ring + (size_t)s * stage_bytes, src0 + (size_t)it * NW * E, bytes, &full[s]);
    };
    if (threadIdx.x == 0) {
      for (int s = 0; s < NS; s++) pi_mbar_init(&full[s], 1);
      pi_fence_barrier_init();
      for (int it = 0; it < min(NS, nst); it++) issue(it);
    }
    // warp w: chunk c = w % chunks, block slot w / chunks of every wpc blocks
    const int wpc = NW / chunks;
    const bool active = warp < chunks * wpc;
    const int c = warp % chunks, slot = warp / chunks;
    const int e0 = 128 * c + 4 * lane;
    const bool valid = active && e0 < E;
    const int gl = valid ? e0 / p.D : 0;
    const int d0 = e0 % p.D;
    const int n = p.D / 4;
    const ConsShape cs = cons_shape(lane, p.D, p.G);
    float4 qv[8];
#pragma unroll
    for (int j = 0; j < 8; j++) {
      qv[j] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
      if (valid && j < p.G) {
        const uint16_t* qh = p.q + ((size_t)r * p.Hq + (size_t)gl * p.G + j) * p.D + d0;
        const uint32_t lo = *reinterpret_cast<const uint32_t*>(qh);
        const uint32_t hi = *reinterpret_cast<const uint32_t*>(qh + 2);
        qv[j] = make_float4(__uint_as_float(lo << 16), __uint_as_float(lo & 0xffff0000u), __uint_as_float(hi << 16),
                            __uint_as_float(hi & 0xffff0000u));
      }
    }
    __syncthreads();  // the ring's barriers are initialised
    bool ok = true;
    for (int it = 0; it < nst; it++) {
      const int s = it % NS;
      if (!pi_mbar_wait_bounded(&full[s], (it / NS) & 1, p.status)) ok = false;
      if (ok && active) {
        const int nb_it = min(NW, nblk - it * NW);
        for (int x = slot; x < nb_it; x += wpc) {
          const float* kb = reinterpret_cast<const float*>(ring + (size_t)s * stage_bytes) + (size_t)x * E;
          const float4 k4 = valid ? *reinterpret_cast<const float4*>(kb + e0) : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
          const float cg = consensus_chunk(k4, qv, valid, lane, cs, p.lambda);
          if (valid && (lane & (n - 1)) == 0) cg_s[(size_t)(it * NW + x) * p.Hkv + gl] = cg;
        }
      }
      // every warp is done with stage s: refill it (a failed wait stops the ring)
      ok = __syncthreads_and(ok) != 0;
      if (!ok) break;
      if (threadIdx.x == 0 && it + NS < nst) issue(it + NS);
    }
    if (!ok && threadIdx.x == 0)
      for (int it = 0; it < nst; it++) pi_mbar_wait_bounded(&full[it % NS], (it / NS) & 1, p.status);
    __syncthreads();
    // the ring's barriers are done with (a later item of the same CTA sets them up again)
    if (threadIdx.x == 0)
      for (int s = 0; s < NS; s++) pi_mbar_inval(&full[s]);
    for (int bl = threadIdx.x; bl < nblk; bl += kSelThreads) {
      float total = 0.0f;
      for (int g2 = 0; g2 < p.Hkv; g2++) total = __fadd_rn(total, cg_s[(size_t)bl * p.Hkv + g2]);
      sink(b_begin + bl, total);
    }
  }
  for (int b = b_begin + warp; b < b_end && !p.consensus; b += 2 * NW) {
    const int b2 = b + NW;
    const bool two = b2 < b_end;
    const float* km = p.kmean + ((rl * p.max_blocks + b) * p.Hkv) * p.D + goff;
    const float* km2 = p.kmean + ((rl * p.max_blocks + (two ? b2 : b)) * p.Hkv) * p.D + goff;
    float4 kv[8], kv2[8];
#pragma unroll
    for (int c = 0; c < 8; c++) {
      const int e = 128 * c + 4 * lane;
      if (c < chunks && e < E) {
        kv[c] = __ldg(reinterpret_cast<const float4*>(km + e));
        if (two) kv2[c] = __ldg(reinterpret_cast<const float4*>(km2 + e));
      }
    }
    float acc = 0.0f, acc2 = 0.0f;
#pragma unroll
    for (int c = 0; c < 8; c++) {
      const int e = 128 * c + 4 * lane;
      if (c < chunks && e < E) {
        const float4 qv = *reinterpret_cast<const float4*>(qs + e);
        acc = __fmaf_rn(qv.x, kv[c].x, acc);
        acc = __fmaf_rn(qv.y, kv[c].y, acc);
        acc = __fmaf_rn(qv.z, kv[c].z, acc);
        acc = __fmaf_rn(qv.w, kv[c].w, acc);
        if (two) {
          acc2 = __fmaf_rn(qv.x, kv2[c].x, acc2);
          acc2 = __fmaf_rn(qv.y, kv2[c].y, acc2);
          acc2 = __fmaf_rn(qv.z, kv2[c].z, acc2);
          acc2 = __fmaf_rn(qv.w, kv2[c].w, acc2);
        }
      }
    }
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) {
      acc = __fadd_rn(acc, __shfl_xor_sync(0xffffffffu, acc, off));
      acc2 = __fadd_rn(acc2, __shfl_xor_sync(0xffffffffu, acc2, off));
    }
    if (lane == 0) {
      sink(b, acc);
      if (two) sink(b2, acc2);
    }
  }
}

// Top-k by value bins (used by the last CTA of a unit and by the cluster form):
// the candidates' scores are spread over kBins equal-width bins between their
// minimum and maximum; a bin index never decreases as the score grows, so only
// the bin holding the k-th largest score needs resolving further.
constexpr int kBins = kSelThreads;  // one bin per thread
constexpr int kExactMax = 64;       // boundary candidates ranked directly
constexpr int kBinLevels = 6;       // bin refinements before direct ranking regardless

struct FoldArgs {
  // the decode step's append of one token per request, done by the leader CTA
  // (nullptr k_new: no append); its host write-through rides in the gather
  const uint8_t* k_new;
  const uint8_t* v_new;
  uint8_t* pool;
  const long long* slot_base;
  float* tail_sum;
  int* ntok_w;
};

struct ClusterArgs {
  int keys_off, hist_off, list_off, state_off;  // leader's scratch in dynamic shared memory (bytes)
  int cap_keys;                                 // candidates that scratch holds
  FoldArgs f;
};

__device__ __forceinline__ int score_bin(float v, float lo, float inv) {
  const float x = fminf(__fmul_rn(__fsub_rn(v, lo), inv), (float)(kBins - 1));
  return x > 0.0f ? __float2int_rz(x) : 0;
}

// min and max score over the candidates still open (state 2)
__device__ __forceinline__ void open_range(const float* s, const uint8_t* st, int n, float* red, float& lo,
                                           float& hi) {
  constexpr int NW = kSelThreads / 32;
  float a = INFINITY, b = -INFINITY;
  for (int j = threadIdx.x; j < n; j += kSelThreads)
    if (st[j] == 2) {
      a = fminf(a, s[j]);
      b = fmaxf(b, s[j]);
    }
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) {
    a = fminf(a, __shfl_xor_sync(0xffffffffu, a, o));
    b = fmaxf(b, __shfl_xor_sync(0xffffffffu, b, o));
  }
  if ((threadIdx.x & 31) == 0) {
    red[threadIdx.x >> 5] = a;
    red[NW + (threadIdx.x >> 5)] = b;
  }
  __syncthreads();
  a = INFINITY;
  b = -INFINITY;
#pragma unroll
  for (int w = 0; w < NW; w++) {
    a = fminf(a, red[w]);
    b = fmaxf(b, red[NW + w]);
  }
  __syncthreads();
  lo = a;
  hi = b;
}

// The kk largest of s[0..n) (ties: lower index), written ascending to out.
// st: n bytes of state (0 out, 1 taken, 2 open); hist: kBins ints per warp;
// list: 2n ints (8-byte aligned). Every thread of the CTA calls it. Returns the
// count written.
__device__ int topk_binned(const float* s, int n, int kk, uint8_t* st, int* hist, int* list, int* warp_sums,
                           int* bc, float* red, int* out) {
  constexpr int NW = kSelThreads / 32;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint8_t init = (kk >= n) ? 1 : (kk <= 0 ? 0 : 2);
  int need = (init == 2) ? kk : 0;
  bool equal_open = false;  // every open candidate has the same score
  // the state of every candidate and the range of the open ones in one pass
  float lo, hi;
  {
    float a = INFINITY, b = -INFINITY;
    for (int j = tid; j < n; j += kSelThreads) {
      st[j] = init;
      a = fminf(a, s[j]);
      b = fmaxf(b, s[j]);
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) {
      a = fminf(a, __shfl_xor_sync(0xffffffffu, a, o));
      b = fmaxf(b, __shfl_xor_sync(0xffffffffu, b, o));
    }
    if (lane == 0) {
      red[warp] = a;
      red[NW + warp] = b;
    }
    __syncthreads();
    a = INFINITY;
    b = -INFINITY;
#pragma unroll
    for (int w = 0; w < NW; w++) {
      a = fminf(a, red[w]);
      b = fmaxf(b, red[NW + w]);
    }
    lo = a;
    hi = b;
    __syncthreads();  // red is reused below
  }
  for (int level = 0; need > 0; level++) {
    if (level > 0) open_range(s, st, n, red, lo, hi);
    if (!(lo < hi)) {
      equal_open = true;
      break;
    }
    if (level >= kBinLevels) break;
    const float inv = __fdiv_rn((float)kBins, __fsub_rn(hi, lo));
    // one histogram per warp (its atomics never queue behind another warp's),
    // then thread b adds bin b over the warps
#pragma unroll
    for (int w = 0; w < NW; w++) hist[w * kBins + tid] = 0;
    __syncthreads();
    for (int j = tid; j < n; j += kSelThreads)
      if (st[j] == 2) atomicAdd(&hist[warp * kBins + score_bin(s[j], lo, inv)], 1);
    __syncthreads();
    {
      int c = 0;
#pragma unroll
      for (int w = 0; w < NW; w++) c += hist[w * kBins + tid];
      hist[tid] = c;  // bin tid of warp 0's histogram, read only by this thread above
    }
    __syncthreads();
    if (warp == 0) {
      // boundary bin: count(bins above) < need <= count(bins above) + its own;
      // lane i holds bins 255-8i .. 248-8i (descending)
      int cnt[8], own = 0;
#pragma unroll
      for (int t = 0; t < 8; t++) {
        cnt[t] = hist[kBins - 1 - 8 * lane - t];
        own += cnt[t];
      }
      int incl = own;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      const unsigned hit = __ballot_sync(0xffffffffu, incl >= need);
      if (lane == __ffs(hit) - 1) {
        int acc = incl - own;
#pragma unroll
        for (int t = 0; t < 8; t++) {
          if (acc + cnt[t] >= need) {
            bc[0] = kBins - 1 - 8 * lane - t;
            bc[1] = acc;
            bc[2] = cnt[t];
            break;
          }
          acc += cnt[t];
        }
      }
    }
    __syncthreads();
    const int tb = bc[0], above = bc[1], m = bc[2];
    for (int j = tid; j < n; j += kSelThreads)
      if (st[j] == 2) {
        const int bn = score_bin(s[j], lo, inv);
        st[j] = (bn > tb) ? 1 : (bn == tb ? 2 : 0);
      }
    need -= above;
    __syncthreads();  // bc and st are read by every thread before they change again
    if (need == m) {
      for (int j = tid; j < n; j += kSelThreads)
        if (st[j] == 2) st[j] = 1;
      need = 0;
      __syncthreads();
    }
    if (m <= kExactMax) break;
  }
  const int per = (n + kSelThreads - 1) / kSelThreads;
  const int j0 = min(n, tid * per), j1 = min(n, j0 + per);
  if (need > 0 && equal_open) {
    // equal scores: the lowest indices go first
    int c = 0;
    for (int j = j0; j < j1; j++) c += (st[j] == 2) ? 1 : 0;
    int tot;
    int before = pi_plan::cta_excl_scan<kSelThreads>(c, warp_sums, tot);
    for (int j = j0; j < j1; j++)
      if (st[j] == 2) st[j] = (before++ < need) ? 1 : 0;
    __syncthreads();
  } else if (need > 0) {
    // few open candidates: rank each against the others directly, from a list
    // of (score, index) pairs (one shared load per comparison, eight in flight)
    if (tid == 0) bc[3] = 0;
    __syncthreads();
    float2* pairs = reinterpret_cast<float2*>(list);  // list holds 2n ints
    for (int j = tid; j < n; j += kSelThreads)
      if (st[j] == 2) pairs[atomicAdd(&bc[3], 1)] = make_float2(s[j], __int_as_float(j));
    __syncthreads();
    const int m = bc[3];
    for (int i = tid; i < m; i += kSelThreads) {
      const float2 me = pairs[i];
      const int j = __float_as_int(me.y);
      int rank = 0;
      int x = 0;
      for (; x + 8 <= m; x += 8) {
        float2 o[8];
#pragma unroll
        for (int t = 0; t < 8; t++) o[t] = pairs[x + t];
#pragma unroll
        for (int t = 0; t < 8; t++)
          rank += (o[t].x > me.x || (o[t].x == me.x && __float_as_int(o[t].y) < j)) ? 1 : 0;
      }
      for (; x < m; x++) {
        const float2 o = pairs[x];
        rank += (o.x > me.x || (o.x == me.x && __float_as_int(o.y) < j)) ? 1 : 0;
      }
      st[j] = (rank < need) ? 1 : 0;
    }
    __syncthreads();
  }
  // ascending output of the taken candidates
  int c = 0;
  for (int j = j0; j < j1; j++) c += (st[j] == 1) ? 1 : 0;
  int tot;
  int pos = pi_plan::cta_excl_scan<kSelThreads>(c, warp_sums, tot);
  for (int j = j0; j < j1; j++)
    if (st[j] == 1 && pos < kk) out[pos++] = j;
  return tot;
}

// Candidates a thread keeps in registers in the register form of the top-k
// (up to kRegKeys * kSelThreads = 4096 candidates).
constexpr int kRegKeys = 16;

// The same top-k with every candidate's score in registers: thread t owns
// candidates [t*per, t*per + per) of [0, n) in v[0..per), so every pass over
// the candidates is register work and the output is one scan. flag: n bytes;
// pairs: n (score, index) pairs; hist: kBins ints per warp. Returns the count
// written to out.
__device__ int topk_regs(int n, int kk, const float (&v)[kRegKeys], int per, int* hist, float2* pairs,
                         uint8_t* flag, int* warp_sums, int* bc, float* red, int* out) {
  constexpr int NW = kSelThreads / 32;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int j0 = tid * per;
  unsigned valid = 0;
#pragma unroll
  for (int i = 0; i < kRegKeys; i++)
    if (i < per && j0 + i < n) valid |= 1u << i;
  unsigned open = 0, taken = 0;
  int need = 0;
  if (kk >= n) {
    taken = valid;
  } else if (kk > 0) {
    open = valid;
    need = kk;
  }
  bool equal_open = false;
  for (int level = 0; need > 0; level++) {
    float a = INFINITY, b = -INFINITY;
#pragma unroll
    for (int i = 0; i < kRegKeys; i++)
      if (open & (1u << i)) {
        a = fminf(a, v[i]);
        b = fmaxf(b, v[i]);
      }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) {
      a = fminf(a, __shfl_xor_sync(0xffffffffu, a, o));
      b = fmaxf(b, __shfl_xor_sync(0xffffffffu, b, o));
    }
    if (lane == 0) {
      red[warp] = a;
      red[NW + warp] = b;
    }
#pragma unroll
    for (int w = 0; w < NW; w++) hist[w * kBins + tid] = 0;
    __syncthreads();
    float lo = INFINITY, hi = -INFINITY;
#pragma unroll
    for (int w = 0; w < NW; w++) {
      lo = fminf(lo, red[w]);
      hi = fmaxf(hi, red[NW + w]);
    }
    if (!(lo < hi)) {
      equal_open = true;
      break;
    }
    if (level >= kBinLevels) break;
    const float inv = __fdiv_rn((float)kBins, __fsub_rn(hi, lo));
    int bins[kRegKeys];
#pragma unroll
    for (int i = 0; i < kRegKeys; i++) {
      bins[i] = score_bin(v[i], lo, inv);
      if (open & (1u << i)) atomicAdd(&hist[warp * kBins + bins[i]], 1);
    }
    __syncthreads();
    {
      int c = 0;
#pragma unroll
      for (int w = 0; w < NW; w++) c += hist[w * kBins + tid];
      hist[tid] = c;
    }
    __syncthreads();
    if (warp == 0) {
      int cnt[8], own = 0;
#pragma unroll
      for (int t = 0; t < 8; t++) {
        cnt[t] = hist[kBins - 1 - 8 * lane - t];
        own += cnt[t];
      }
      int incl = own;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      const unsigned hit = __ballot_sync(0xffffffffu, incl >= need);
      if (lane == __ffs(hit) - 1) {
        int acc = incl - own;
#pragma unroll
        for (int t = 0; t < 8; t++) {
          if (acc + cnt[t] >= need) {
            bc[0] = kBins - 1 - 8 * lane - t;
            bc[1] = acc;
            bc[2] = cnt[t];
            break;
          }
          acc += cnt[t];
        }
      }
    }
    __syncthreads();
    const int tb = bc[0], above = bc[1], m = bc[2];
#pragma unroll
    for (int i = 0; i < kRegKeys; i++)
      if (open & (1u << i)) {
        if (bins[i] > tb) taken |= 1u << i;
        if (bins[i] != tb) open &= ~(1u << i);
      }
    need -= above;
    __syncthreads();  // red, hist and bc are rewritten by the next level
    if (need == m) {
      taken |= open;
      open = 0;
      need = 0;
    }
    if (m <= kExactMax) break;
  }
  if (need > 0 && equal_open) {
    // equal scores: the lowest indices go first
    int tot;
    int before = pi_plan::cta_excl_scan<kSelThreads>(__popc(open), warp_sums, tot);
#pragma unroll
    for (int i = 0; i < kRegKeys; i++)
      if (open & (1u << i)) {
        if (before < need) taken |= 1u << i;
        before++;
      }
    open = 0;
  } else if (need > 0) {
    // few open candidates: rank each against the others directly
    if (tid == 0) bc[3] = 0;
    __syncthreads();
#pragma unroll
    for (int i = 0; i < kRegKeys; i++)
      if (open & (1u << i)) pairs[atomicAdd(&bc[3], 1)] = make_float2(v[i], __int_as_float(j0 + i));
    __syncthreads();
    const int m = bc[3];
    for (int x0 = tid; x0 < m; x0 += kSelThreads) {
      const float2 me = pairs[x0];
      const int j = __float_as_int(me.y);
      int rank = 0;
      int x = 0;
      for (; x + 8 <= m; x += 8) {
        float2 o[8];
#pragma unroll
        for (int t = 0; t < 8; t++) o[t] = pairs[x + t];
#pragma unroll
        for (int t = 0; t < 8; t++)
          rank += (o[t].x > me.x || (o[t].x == me.x && __float_as_int(o[t].y) < j)) ? 1 : 0;
      }
      for (; x < m; x++) {
        const float2 o = pairs[x];
        rank += (o.x > me.x || (o.x == me.x && __float_as_int(o.y) < j)) ? 1 : 0;
      }
      flag[j] = (rank < need) ? 1 : 0;
    }
    __syncthreads();
#pragma unroll
    for (int i = 0; i < kRegKeys; i++)
      if ((open & (1u << i)) && flag[j0 + i]) taken |= 1u << i;
  }
  // ascending output of the taken candidates
  int tot;
  int pos = pi_plan::cta_excl_scan<kSelThreads>(__popc(taken), warp_sums, tot);
#pragma unroll
  for (int i = 0; i < kRegKeys; i++)
    if ((taken & (1u << i)) && pos < kk) out[pos++] = j0 + i;
  return tot;
}

__device__ __forceinline__ bool select_item(const SelParams& p, const int u, const int chunk, const int nchunks) {
  __shared__ int hist[512];
  __shared__ int warp_sums[kSelThreads / 32];
  __shared__ int bcast[4];
  extern __shared__ __align__(16) uint32_t dyn[];  // plan scratch, then the slot-map cache
  const int r = u / p.U;
  const int g = (p.U == 1) ? 0 : u % p.U;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const size_t rl = (size_t)r * p.L + p.layer;
  const int nt = p.ntok[rl];
  int nb = (nt + p.B - 1) / p.B;
  int ncand = max(0, nb - p.W);
  if (ncand > nchunks * p.bpc || nb > p.max_blocks) {
    // more candidates than the launch was sized for (a token count the host did
    // not know of): flagged, and only the candidates the launch covers compete
    if (threadIdx.x == 0) pi_flag(p.status, PI_DEV_LAUNCH_SIZE);
    nb = min(nb, p.max_blocks);
    ncand = min(max(0, nb - p.W), nchunks * p.bpc);
  }
  const int kreq_early = p.k_per_req[r];  // read now: the tail needs it right away

  const int b_begin = chunk * p.bpc;
  const int b_end = min(ncand, b_begin + p.bpc);
  float* sc = p.scores + (size_t)u * p.max_blocks;
  select_score(p, u, b_begin, b_end, [&](int b, float v) { sc[b] = v; });

  // the last CTA of this unit to finish runs the top-k
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) {
    const unsigned done = atomicAdd(p.counter + u, 1u);
    bcast[0] = (done == (unsigned)nchunks - 1) ? 1 : 0;
  }
  __syncthreads();
  if (!bcast[0]) return false;
  if (threadIdx.x == 0) p.counter[u] = 0;  // ready for the next call
  __threadfence();

  const int kk = min(max(0, min(kreq_early, p.k_max)), ncand);
  int* out = p.sel + (size_t)u * p.cap;
  // fused plan: read this unit's slot maps now (one round of loads, held in
  // registers, then stored), so the plan runs from shared memory
  const size_t rlu_m = rl * p.U + g;
  const int P_r = p.P[rl];
  int* sob_c = nullptr;
  int* bos_c = nullptr;
  if (p.table && p.map_cache_blocks >= nb && p.map_cache_slots >= P_r) {
    unsigned char* after = reinterpret_cast<unsigned char*>(dyn) + p.dyn_plan_off +
                           pi_plan::plan_smem_bytes(p.max_blocks, p.cap, p.slot_stamp ? p.lru_p2 : 0);
    sob_c = reinterpret_cast<int*>(after);
    bos_c = sob_c + p.map_cache_blocks;
    stage_ints<kKeysPerThread>(sob_c, p.slot_of + rlu_m * p.max_blocks, nb);
    stage_ints<kKeysPerThread>(bos_c, p.block_of + rlu_m * p.p_max, P_r);
  }
  int out_n = 0;
  if (p.binned_off > 0 && ncand <= p.binned_cap && ncand <= kRegKeys * kSelThreads) {
    // every score straight into registers (each thread a contiguous run), then
    // the binned top-k on them
    uint8_t* bsm = reinterpret_cast<uint8_t*>(dyn) + p.binned_off;
    const int capk = (p.binned_cap + 3) & ~3;
    constexpr size_t hist_bytes = (size_t)kBins * 4 * (kSelThreads / 32);
    const int per = (((ncand + kSelThreads - 1) / kSelThreads) + 3) & ~3;
    const int j0 = threadIdx.x * per;
    float v[kRegKeys];
#pragma unroll
    for (int i = 0; i < kRegKeys; i++) v[i] = (i < per && j0 + i < ncand) ? __ldcg(sc + j0 + i) : 0.0f;
    out_n = topk_regs(ncand, kk, v, per, reinterpret_cast<int*>(bsm + (size_t)capk * 4),
                      reinterpret_cast<float2*>(bsm + (size_t)capk * 4 + hist_bytes),
                      bsm + (size_t)capk * 4 + hist_bytes + (size_t)capk * 8, warp_sums, bcast,
                      reinterpret_cast<float*>(hist), out);
  } else if (p.binned_off > 0 && ncand <= p.binned_cap) {
    // every score into shared memory in one round of loads, then the binned top-k
    uint8_t* bsm = reinterpret_cast<uint8_t*>(dyn) + p.binned_off;
    float* keys = reinterpret_cast<float*>(bsm);
    const int capk = (p.binned_cap + 3) & ~3;
    for (int base = 0; base < ncand; base += kSelThreads * 8) {
      float v[8];
#pragma unroll
      for (int i = 0; i < 8; i++) {
        const int b = base + threadIdx.x + i * kSelThreads;
        v[i] = (b < ncand) ? __ldcg(sc + b) : 0.0f;
      }
#pragma unroll
      for (int i = 0; i < 8; i++) {
        const int b = base + threadIdx.x + i * kSelThreads;
        if (b < ncand) keys[b] = v[i];
      }
    }
    __syncthreads();
    constexpr size_t hist_bytes = (size_t)kBins * 4 * (kSelThreads / 32);
    out_n = topk_binned(keys, ncand, kk, bsm + (size_t)capk * 4 + hist_bytes + (size_t)capk * 8,
                        reinterpret_cast<int*>(bsm + (size_t)capk * 4),
                        reinterpret_cast<int*>(bsm + (size_t)capk * 4 + hist_bytes), warp_sums, bcast,
                        reinterpret_cast<float*>(hist), out);
  } else {
  // candidate keys: up to kKeysPerThread per thread in registers, each thread
  // owning a contiguous run of block ids; more candidates than that are read
  // from the score buffer where they are used
  const bool in_regs = ncand <= kKeysPerThread * kSelThreads;
  const int per = in_regs ? (ncand + kSelThreads - 1) / kSelThreads : 0;
  const int b_lo = threadIdx.x * per;
  uint32_t kr[kKeysPerThread];
#pragma unroll
  for (int i = 0; i < kKeysPerThread; i++)
    kr[i] = (i < per && b_lo + i < ncand) ? order_key(__ldcg(sc + b_lo + i)) : 0u;
  hist[threadIdx.x] = 0;  // kSelThreads == 256 bins, two buffers
  __syncthreads();

  uint32_t T = 0;      // key of the kk-th largest candidate
  int need_eq = 0;     // how many candidates equal to T to take (lowest indices)
  const bool take_all = (kk == ncand);
  if (kk > 0 && !take_all) {
    uint32_t prefix = 0, mask = 0;
    int remaining = kk;
    int pass = 0;
    for (int shift = 24; shift >= 0; shift -= 8, pass++) {
      int* h_cur = hist + 256 * (pass & 1);
      int* h_nxt = hist + 256 * ((pass + 1) & 1);
      if (in_regs && per <= 4) {
        // few keys per thread: lanes of a warp with the same digit add once (the
        // leading digits of nearby scores coincide, so plain atomics would queue
        // on a few bins); with more keys per thread the matching costs more
        // than the queueing it saves (measured)
#pragma unroll
        for (int i = 0; i < 4; i++) {
          if (i >= per) break;
          const bool take = b_lo + i < ncand && (kr[i] & mask) == prefix;
          const unsigned act = __ballot_sync(0xffffffffu, take);
          if (take) {
            const unsigned digit = (kr[i] >> shift) & 255;
            const unsigned peers = __match_any_sync(act, digit);
            if (lane == __ffs(peers) - 1) atomicAdd(&h_cur[digit], __popc(peers));
          }
        }
      } else if (in_regs) {
#pragma unroll
        for (int i = 0; i < kKeysPerThread; i++)
          if (i < per && b_lo + i < ncand && (kr[i] & mask) == prefix) atomicAdd(&h_cur[(kr[i] >> shift) & 255], 1);
      } else {
        for (int b = threadIdx.x; b < ncand; b += kSelThreads) {
          const uint32_t key = order_key(__ldcg(sc + b));
          if ((key & mask) == prefix) atomicAdd(&h_cur[(key >> shift) & 255], 1);
        }
      }
      __syncthreads();
      if (warp == 0) {
        // lane owns digits 255-8*lane .. 248-8*lane (descending)
        int cnt[8], own = 0;
#pragma unroll
        for (int j = 0; j < 8; j++) {
          cnt[j] = h_cur[255 - 8 * lane - j];
          own += cnt[j];
        }
        int incl = own;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          int y = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += y;
        }
        const unsigned hit = __ballot_sync(0xffffffffu, incl >= remaining);
        const int first = __ffs(hit) - 1;
        if (lane == first) {
          int before = incl - own;
          int digit = 255 - 8 * lane - 7;
#pragma unroll
          for (int j = 0; j < 8; j++) {
            if (before + cnt[j] >= remaining) {
              digit = 255 - 8 * lane - j;
              break;
            }
            before += cnt[j];
          }
          bcast[1] = digit;
          bcast[2] = remaining - before;
        }
      } else {
        // the other warps clear the next pass's histogram meanwhile
        for (int i = threadIdx.x - 32; i < 256; i += kSelThreads - 32) h_nxt[i] = 0;
      }
      __syncthreads();
      // (bcast is rewritten only after the next pass's first barrier, which every
      // thread reaches after reading it here)
      prefix |= (uint32_t)bcast[1] << shift;
      mask |= 0xFFu << shift;
      remaining = bcast[2];
    }
    T = prefix;
    need_eq = remaining;
  }

  // stable compaction in block order: all keys > T, then the first need_eq == T
  if (kk > 0 && in_regs) {
    // one scan of (greater, equal) counts per thread, then each thread places
    // its own run in order
    int gt_c = 0, eq_c = 0;
#pragma unroll
    for (int i = 0; i < kKeysPerThread; i++)
      if (i < per && b_lo + i < ncand) {
        gt_c += (take_all || kr[i] > T) ? 1 : 0;
        eq_c += (!take_all && kr[i] == T) ? 1 : 0;
      }
    int tot;
    const int ex = pi_plan::cta_excl_scan<kSelThreads>((gt_c << 16) | eq_c, warp_sums, tot);
    int gt_before = ex >> 16, eq_before = ex & 0xffff;
#pragma unroll
    for (int i = 0; i < kKeysPerThread; i++)
      if (i < per && b_lo + i < ncand) {
        const bool gt = take_all || kr[i] > T;
        const bool eq = !take_all && kr[i] == T;
        if (gt) {
          const int pos = gt_before + min(eq_before, need_eq);
          if (pos < kk) out[pos] = b_lo + i;
          gt_before++;
        } else if (eq) {
          if (eq_before < need_eq && gt_before + eq_before < kk) out[gt_before + eq_before] = b_lo + i;
          eq_before++;
        }
      }
    out_n = (tot >> 16) + min(tot & 0xffff, need_eq);
  } else if (kk > 0) {
    int eq_seen = 0;
    for (int base = 0; base < ncand; base += kSelThreads) {
      const int b = base + threadIdx.x;
      int gt = 0, eq = 0;
      if (b < ncand) {
        if (take_all) {
          gt = 1;
        } else {
          const uint32_t key = order_key(__ldcg(sc + b));
          gt = key > T;
          eq = key == T;
        }
      }
      int eq_total;
      const int eq_before = pi_plan::cta_excl_scan<kSelThreads>(eq, warp_sums, eq_total);
      const int take = gt || (eq && (eq_seen + eq_before) < need_eq);
      int take_total;
      const int pos = pi_plan::cta_excl_scan<kSelThreads>(take, warp_sums, take_total);
      if (take && out_n + pos < kk) out[out_n + pos] = b;
      out_n += take_total;
      eq_seen += eq_total;
    }
  }
  }  // radix path
  // the W most recent blocks follow (they are the highest block ids)
  const int nrecent = nb - ncand;
  for (int j = threadIdx.x; j < nrecent; j += kSelThreads) out[kk + j] = ncand + j;
  if (threadIdx.x == 0) {
    if (out_n != kk) pi_flag(p.status, PI_DEV_BAD_INDEX);
    p.nsel[u] = kk + nrecent;
  }
  if (p.table == nullptr) return true;

  // fused recall plan of this unit (the selection is in global memory, written
  // by this CTA; the barrier makes it visible to every thread of the CTA)
  __syncthreads();
  const int words = (p.max_blocks + 31) / 32;
  unsigned char* plb = reinterpret_cast<unsigned char*>(dyn) + p.dyn_plan_off;
  unsigned long long* lkeys = reinterpret_cast<unsigned long long*>(plb);
  uint32_t* pl = reinterpret_cast<uint32_t*>(plb + sizeof(unsigned long long) * (p.slot_stamp ? p.lru_p2 : 0));
  pi_plan::UnitArgs a;
  a.sel = out;
  a.n = kk + nrecent;
  const size_t rlu = rl * p.U + g;
  a.sob = sob_c ? sob_c : p.slot_of + rlu * p.max_blocks;
  a.bos = bos_c ? bos_c : p.block_of + rlu * p.p_max;
  a.P = p.P[rl];
  a.max_blocks = p.max_blocks;
  a.table = p.table + (size_t)u * p.cap;
  a.plan = p.plan + (size_t)u * p.cap;
  a.plan_n = p.plan_n + u;
  a.counts = p.counts;
  a.status = p.status;
  a.stamp = p.slot_stamp ? p.slot_stamp + rlu * p.p_max : nullptr;
  a.epoch = p.slot_stamp ? p.epoch + rlu : nullptr;
  a.empty_first = p.empty_first;
  pi_plan::plan_unit<kSelThreads>(a, pl, reinterpret_cast<int*>(pl) + words, reinterpret_cast<int*>(pl) + words + p.cap,
                                  warp_sums, lkeys, p.lru_p2);
  return true;
}

__global__ void __launch_bounds__(kSelThreads) select_kernel(SelParams p) {
  select_item(p, p.u0 + blockIdx.y, blockIdx.x, gridDim.x);
}

struct FusedArgs {
  unsigned long long* claim;      // this layer's item counter (only grows)
  unsigned long long claim_base;  // its value when this launch starts
  unsigned* ready;                // [R*U] of this layer: epoch once a unit's plan is written
  unsigned epoch;
  int units, chunks, items;       // units p.u0 .. p.u0+units-1; items = units x chunks
};

// Selection, recall plan and UVA gather of one layer in one launch on a few SMs
// (the decode step's fused form). Phase 1: each CTA claims selection items
// (unit-major, so the first units' plans come out first) from a counter until
// none are left; the CTA that completes a unit's last item runs its top-k and
// plan and publishes them with a release store of the launch's epoch. Phase 2:
// every CTA walks the units in order, waits (bounded) for each unit's flag, and
// copies its share of the unit's missing blocks in 32 KiB items. A CTA only
// waits once every item has been claimed by a running CTA, and items never
// wait, so the launch finishes whatever the CTAs' residency.
__global__ void __launch_bounds__(kSelThreads) select_gather_kernel(SelParams p, GatherParams g, FusedArgs f) {
  __shared__ int claim_s;
  if (g.k_new && blockIdx.x == 0) pi_gather_write_through<kSelThreads>(g);
  for (;;) {
    __syncthreads();  // the previous item is done with shared memory and claim_s
    if (threadIdx.x == 0) claim_s = (int)min(atomicAdd(f.claim, 1ULL) - f.claim_base, (unsigned long long)f.items);
    __syncthreads();
    const int it = claim_s;
    if (it >= f.items) break;
    const int v = it / f.chunks;
    if (select_item(p, p.u0 + v, it - v * f.chunks, f.chunks)) {
      __threadfence();
      __syncthreads();
      if (threadIdx.x == 0) pi_st_release(f.ready + p.u0 + v, f.epoch);
    }
  }
  constexpr int kDepth = 8;
  constexpr int kChunk = kSelThreads * 16 * kDepth;
  const int chunk = min(g.copy_bytes, kChunk);
  const int cpe = (g.copy_bytes + chunk - 1) / chunk;
  const int F = gridDim.x;
  long long rot = 0;  // items of the earlier units: the next unit's first item goes to CTA rot % F
  for (int v = 0; v < f.units; v++) {
    __syncthreads();
    if (threadIdx.x == 0) claim_s = pi_wait_flag_bounded(f.ready + p.u0 + v, f.epoch, p.status) ? 1 : 0;
    __syncthreads();
    if (!claim_s) continue;  // timed out: recorded in the status word, the unit is skipped
    const long long items = (long long)__ldcg(g.plan_n + v) * cpe;
    const long long first = ((long long)blockIdx.x - rot % F + F) % F;
    for (long long i = first; i < items; i += F)
      pi_gather_item<kDepth, kSelThreads>(g, v, (int)(i / cpe), (int)(i % cpe), chunk, 0);
    rot += items;
  }
}

// ------------------------------------------------------------------ a-2 in clusters
// The selection of one unit as one thread-block cluster of cs CTAs: CTA c scores
// candidates [c*bpc, (c+1)*bpc) and stores each score straight into the shared
// memory of the cluster's first CTA (the leader); after one cluster barrier the
// leader holds every score of the unit and runs the top-k (and, in the decode
// step, the recall plan) from shared memory. Nothing goes through global memory
// and no CTA has to find out it finished last.
//
// Top-k by value bins: the candidates' scores are spread over kBins equal-width
// bins between their minimum and maximum; a bin index is a non-decreasing
// function of the score (subtraction, multiplication and truncation rounded in
// one direction), so every candidate in a bin above the one holding the k-th
// largest score is taken, every one below is not, and only the boundary bin is
// resolved further: again by bins, or, once few candidates are left, by ranking
// them exactly by (score descending, block index ascending).
// The decode step's append for request r (leader CTA): the token at position t
// goes into its block's pool slot when that block is resident (a block recalled
// in this step gets it from the gather instead), and the block's running key sum
// and summary take it (the same fp32 arithmetic as the stand-alone append).
__device__ __forceinline__ void fold_append(const SelParams& p, const FoldArgs& f, int r, size_t rl, int t) {
  const int b = t / p.B, tp = t % p.B;
  if (b >= p.max_blocks) {
    if (threadIdx.x == 0) pi_flag(p.status, PI_DEV_BAD_INDEX);
    return;
  }
  const size_t block_bytes = (size_t)p.Hkv * 2 * p.B * p.D * 2;
  const int slot = p.slot_of[rl * p.max_blocks + b];
  const int P_r = p.P[rl];
  for (int e = threadIdx.x * 8; e < p.Hkv * p.D; e += kSelThreads * 8) {
    const int g = e / p.D, d = e % p.D;
    const uint4 kv = *reinterpret_cast<const uint4*>(f.k_new + (((size_t)r * p.Hkv + g) * p.D + d) * 2);
    if (slot >= 0) {
      if (slot >= P_r) {
        pi_flag(p.status, PI_DEV_BAD_INDEX);
      } else {
        const uint4 vv = *reinterpret_cast<const uint4*>(f.v_new + (((size_t)r * p.Hkv + g) * p.D + d) * 2);
        uint8_t* blk = f.pool + (size_t)(f.slot_base[rl] + slot) * block_bytes;
        *reinterpret_cast<uint4*>(blk + ((((size_t)g * 2 + 0) * p.B + tp) * p.D + d) * 2) = kv;
        *reinterpret_cast<uint4*>(blk + ((((size_t)g * 2 + 1) * p.B + tp) * p.D + d) * 2) = vv;
      }
    }
    float* ts = f.tail_sum + (rl * p.Hkv + g) * p.D + d;
    float* km = const_cast<float*>(p.kmean) + ((rl * p.max_blocks + b) * p.Hkv + g) * p.D + d;
    const uint32_t w[4] = {kv.x, kv.y, kv.z, kv.w};
    const float fn = (float)(tp + 1);
#pragma unroll
    for (int j = 0; j < 4; j++) {
      float s0 = (tp == 0) ? 0.0f : ts[2 * j];
      float s1 = (tp == 0) ? 0.0f : ts[2 * j + 1];
      s0 = __fadd_rn(s0, pi_bf16_lo(w[j]));
      s1 = __fadd_rn(s1, pi_bf16_hi(w[j]));
      ts[2 * j] = s0;
      ts[2 * j + 1] = s1;
      km[2 * j] = __fdiv_rn(s0, fn);
      km[2 * j + 1] = __fdiv_rn(s1, fn);
    }
  }
}

// grid (cs, units), cluster (cs, 1, 1): CTA blockIdx.x of unit p.u0 + blockIdx.y
__global__ void __launch_bounds__(kSelThreads) select_cluster_kernel(SelParams p, ClusterArgs c) {
  __shared__ int warp_sums[kSelThreads / 32];
  __shared__ int bc[4];
  __shared__ float red[2 * (kSelThreads / 32)];
  extern __shared__ __align__(16) uint32_t dyn[];
  pi_grid_dep_wait();  // what earlier kernels wrote (token counts, summaries, maps) is visible from here on
  const int u = p.u0 + blockIdx.y;
  const int rank = blockIdx.x;
  const bool leader = rank == 0;
  const int r = u / p.U;
  const int g = (p.U == 1) ? 0 : u % p.U;
  const size_t rl = (size_t)r * p.L + p.layer;
  const bool fold = c.f.k_new != nullptr;
  const int nt_old = p.ntok[rl];
  const int nt = nt_old + (fold ? 1 : 0);
  const int nb = (nt + p.B - 1) / p.B;
  int ncand = max(0, nb - p.W);
  if (ncand > c.cap_keys || ncand > (int)gridDim.x * p.bpc) {
    // more candidates than the launch was sized for (a token count the host did
    // not know of): flagged, and only the first ones compete
    if (threadIdx.x == 0) pi_flag(p.status, PI_DEV_LAUNCH_SIZE);
    ncand = min(c.cap_keys, (int)gridDim.x * p.bpc);
  }
  uint8_t* sm = reinterpret_cast<uint8_t*>(dyn);
  float* keys = reinterpret_cast<float*>(sm + c.keys_off);
  const int kreq_early = leader ? p.k_per_req[r] : 0;  // read now: the tail needs it right away

  // leader: this unit's slot maps into shared memory, in flight during the scoring
  const size_t rlu = rl * p.U + g;
  const int P_r = p.P[rl];
  int* sob_c = nullptr;
  int* bos_c = nullptr;
  if (leader && p.table && p.map_cache_blocks >= nb && p.map_cache_slots >= P_r) {
    uint8_t* after = sm + p.dyn_plan_off + pi_plan::plan_smem_bytes(p.max_blocks, p.cap, p.slot_stamp ? p.lru_p2 : 0);
    sob_c = reinterpret_cast<int*>(after);
    bos_c = sob_c + p.map_cache_blocks;
    for (int i = threadIdx.x; i < nb; i += kSelThreads) pi_cp_async4(sob_c + i, p.slot_of + rlu * p.max_blocks + i);
    for (int i = threadIdx.x; i < P_r; i += kSelThreads) pi_cp_async4(bos_c + i, p.block_of + rlu * p.p_max + i);
    pi_cp_async_commit();
  }
  if (leader && fold) fold_append(p, c.f, r, rl, nt_old);

  // this CTA's candidates, scored into the leader's key array
  const int b_begin = rank * p.bpc;
  const int b_end = min(ncand, b_begin + p.bpc);
  const uint32_t keys_leader = pi_cluster_map(pi_smem_addr(keys), 0);
  select_score(p, u, b_begin, b_end, [&](int b, float v) { pi_st_cluster_f32(keys_leader + 4u * (uint32_t)b, v); });
  pi_grid_dep_trigger();
  pi_cluster_sync();  // every score of the unit is in the leader's shared memory
  if (!leader) return;
  if (fold && threadIdx.x == 0) c.f.ntok_w[rl] = nt;  // every CTA of the unit has read the old count

  const int kk = min(max(0, min(kreq_early, p.k_max)), ncand);
  int* out = p.sel + (size_t)u * p.cap;
  int out_n;
  if (ncand <= kRegKeys * kSelThreads) {
    // the keys into registers (a contiguous run per thread, 16-byte loads)
    const int per = (((ncand + kSelThreads - 1) / kSelThreads) + 3) & ~3;
    const int j0 = threadIdx.x * per;
    float v[kRegKeys];
#pragma unroll
    for (int q4 = 0; q4 < kRegKeys / 4; q4++) {
      float4 f = make_float4(0.f, 0.f, 0.f, 0.f);
      if (4 * q4 < per && j0 + 4 * q4 < ncand) f = *reinterpret_cast<const float4*>(keys + j0 + 4 * q4);
      v[4 * q4] = f.x;
      v[4 * q4 + 1] = f.y;
      v[4 * q4 + 2] = f.z;
      v[4 * q4 + 3] = f.w;
    }
    out_n = topk_regs(ncand, kk, v, per, reinterpret_cast<int*>(sm + c.hist_off),
                      reinterpret_cast<float2*>(sm + c.list_off), reinterpret_cast<uint8_t*>(sm + c.state_off),
                      warp_sums, bc, red, out);
  } else {
    out_n = topk_binned(keys, ncand, kk, reinterpret_cast<uint8_t*>(sm + c.state_off),
                        reinterpret_cast<int*>(sm + c.hist_off), reinterpret_cast<int*>(sm + c.list_off), warp_sums,
                        bc, red, out);
  }
  const int nrecent = min(nb, p.W);  // the W most recent blocks follow (the highest ids)
  for (int j = threadIdx.x; j < nrecent; j += kSelThreads) out[kk + j] = nb - nrecent + j;
  if (threadIdx.x == 0) {
    if (out_n != kk) pi_flag(p.status, PI_DEV_BAD_INDEX);
    p.nsel[u] = kk + nrecent;
  }
  if (p.table == nullptr) return;

  // recall plan of this unit from shared memory
  pi_cp_async_wait_all();
  __syncthreads();  // the selection and the cached maps are visible to every thread
  const int words = (p.max_blocks + 31) / 32;
  unsigned char* plb = sm + p.dyn_plan_off;
  unsigned long long* lkeys = reinterpret_cast<unsigned long long*>(plb);
  uint32_t* pl = reinterpret_cast<uint32_t*>(plb + sizeof(unsigned long long) * (p.slot_stamp ? p.lru_p2 : 0));
  pi_plan::UnitArgs a;
  a.sel = out;
  a.n = kk + nrecent;
  a.sob = sob_c ? sob_c : p.slot_of + rlu * p.max_blocks;
  a.bos = bos_c ? bos_c : p.block_of + rlu * p.p_max;
  a.P = P_r;
  a.max_blocks = p.max_blocks;
  a.table = p.table + (size_t)u * p.cap;
  a.plan = p.plan + (size_t)u * p.cap;
  a.plan_n = p.plan_n + u;
  a.counts = p.counts;
  a.status = p.status;
  a.stamp = p.slot_stamp ? p.slot_stamp + rlu * p.p_max : nullptr;
  a.epoch = p.slot_stamp ? p.epoch + rlu : nullptr;
  a.empty_first = p.empty_first;
  pi_plan::plan_unit<kSelThreads>(a, pl, reinterpret_cast<int*>(pl) + words, reinterpret_cast<int*>(pl) + words + p.cap,
                                  warp_sums, lkeys, p.lru_p2);
}

}  // namespace

// ---------------------------------------------------------------------- launchers
cudaError_t pi_launch_summaries(pi_pool* p, int layer, const uint8_t* src, bool src_is_host, int b0, int b1,
                                cudaStream_t s, const int* ntok_new) {
  (void)src_is_host;
  if (b1 <= b0) return cudaSuccess;
  dim3 grid(b1 - b0, p->R);
  int threads = (p->Hkv * p->D) / 8;
  long long stride = (long long)p->region_bytes;
  summaries_kernel<<<grid, threads, 0, s>>>(src, stride, ntok_new, p->ntok, p->kmean, p->tail_sum, layer, p->L,
                                            p->Hkv, p->B, p->D, p->max_blocks, b0);
  return cudaGetLastError();
}

cudaError_t pi_launch_append(pi_pool* p, int layer, const void* k_new, const void* v_new, cudaStream_t s,
                             bool write_host, int r0, int nr) {
  AppendParams a;
  a.write_host = write_host ? 1 : 0;
  a.k_new = (const uint8_t*)k_new;
  a.v_new = (const uint8_t*)v_new;
  a.host_dev = p->host_dev;
  a.pool = p->pool;
  a.slot_base = p->slot_base;
  a.P = p->P;
  a.slot_of = p->slot_of;
  a.ntok = p->ntok;
  a.kmean = p->kmean;
  a.tail_sum = p->tail_sum;
  a.status = p->dev_status;
  a.layer = layer;
  a.L = p->L;
  a.R = p->R;
  a.Hkv = p->Hkv;
  a.B = p->B;
  a.D = p->D;
  a.U = p->U;
  a.max_blocks = p->max_blocks;
  a.host_layer = layer % p->host_layers;
  int threads = (p->Hkv * p->D) / 8;
  if (nr < 0) nr = p->R;
  a.r0 = r0;
  if (nr == 0) return cudaSuccess;
  append_kernel<<<nr, threads, 0, s>>>(a);
  return cudaGetLastError();
}

// Largest candidate count the binned top-k takes (every score, a state byte and
// a list entry per candidate in shared memory).
constexpr int kClusterMaxCand = 16384;
// Up to this many candidates per unit the cluster form is used by default
// (measured faster there); more candidates keep the last-CTA form, whose launch
// spreads evenly over every SM (a unit's cluster holds at most 16 CTAs, so few
// units with many candidates leave SMs idle or need a second wave of clusters).
constexpr int kClusterFormMaxCand = 1024;

// Parameters, chunk count and dynamic shared memory of a selection launch over
// requests r0 .. r0+nr-1 whose grid should hold about `target` CTAs.
static void prepare_select(pi_pool* p, int layer, const void* q, const int* k_per_req, int* sel, int* nsel,
                           int* fused_table, int mode, int r0, int nr, long long target, SelParams& sp, int& chunks,
                           size_t& smem, int* ncand_out = nullptr) {
  sp.q = (const uint16_t*)q;
  sp.q_vec = (reinterpret_cast<uintptr_t>(q) & 15) == 0 ? 1 : 0;
  sp.k_per_req = k_per_req;
  sp.sel = sel;
  sp.nsel = nsel;
  sp.kmean = p->kmean;
  sp.ntok = p->ntok;
  const size_t RU = (size_t)p->R * p->U;
  sp.scores = p->sel_scores + (size_t)layer * RU * p->max_blocks;
  sp.counter = p->sel_counter + (size_t)layer * RU;
  sp.status = p->dev_status;
  sp.layer = layer;
  sp.L = p->L;
  sp.Hq = p->Hq;
  sp.Hkv = p->Hkv;
  sp.G = p->G;
  sp.D = p->D;
  sp.B = p->B;
  sp.max_blocks = p->max_blocks;
  sp.W = p->W;
  sp.k_max = p->k_max;
  sp.cap = p->cap;
  sp.U = p->U;
  // candidates bounded by the largest token count of this layer (host mirror)
  int nb_max = 0;
  for (int r = 0; r < p->R; r++) {
    int nt = p->ntok_h[(size_t)r * p->L + layer];
    nb_max = max(nb_max, (nt + p->B - 1) / p->B);
  }
  const int ncand_max = max(0, nb_max - p->W);
  if (ncand_out) *ncand_out = ncand_max;
  // about `target` CTAs, at least 8 blocks (one per warp) each (rounded down:
  // one more chunk per unit would spill into a second wave)
  const long long units_launch = (long long)nr * p->U;
  chunks = (int)max(1LL, target / units_launch);
  int bpc = (ncand_max + chunks - 1) / chunks;
  bpc = ((max(bpc, 8) + 7) / 8) * 8;
  chunks = max(1, (ncand_max + bpc - 1) / bpc);
  sp.bpc = bpc;
  sp.table = fused_table;
  sp.slot_of = p->slot_of;
  sp.block_of = p->block_of;
  sp.P = p->P;
  sp.plan_n = p->plan_n + (size_t)layer * RU;
  sp.plan = p->plan + (size_t)layer * RU * p->cap;
  sp.counts = p->recall_counts + (size_t)layer * 4;
  sp.p_max = p->p_max;
  const bool lru = p->cfg.evict_policy == PI_EVICT_LRU;
  sp.slot_stamp = lru ? p->slot_stamp : nullptr;
  sp.epoch = lru ? p->epoch : nullptr;
  sp.lru_p2 = lru ? p->lru_p2 : 0;
  sp.consensus = (mode == PI_CONSENSUS) ? 1 : 0;
  sp.empty_first = p->pinned_h.empty() ? 0 : p->pinned_h[layer];
  sp.lambda = p->consensus_lambda;
  sp.ring_stages = 0;
  sp.dyn_plan_off = 0;
  if (sp.consensus) {
    // about 64 KiB of summaries in flight per CTA (two CTAs per SM), then the
    // groups' c_g of the chunk
    const int stage_bytes = 8 * p->Hkv * p->D * 4;
    sp.ring_stages = max(2, min(8, 65536 / stage_bytes));
    sp.dyn_plan_off = sp.ring_stages * stage_bytes + sp.ring_stages * 8 + ((bpc * p->Hkv * 4 + 15) & ~15);
  } else if (p->U == 1) {
    // mean-key scores: a ring of bulk-copy stages (about 96 KiB in flight per CTA,
    // two CTAs per SM), so the loads of a CTA never wait for its arithmetic and
    // an SM keeps enough bytes in flight to cover the latency of a loaded HBM
    const int stage_bytes = 8 * p->Hkv * p->D * 4;
    sp.ring_stages = max(2, min(8, 98304 / stage_bytes));
    sp.dyn_plan_off = (sp.ring_stages * stage_bytes + sp.ring_stages * 8 + 15) & ~15;
  }
  smem = sp.dyn_plan_off;
  if (fused_table) smem += pi_plan::plan_smem_bytes(p->max_blocks, p->cap, sp.lru_p2);
  // slot maps cached for the fused plan when they are small (cached only up to
  // the largest block count of this layer; nothing beyond it is ever looked up)
  sp.map_cache_blocks = 0;
  sp.map_cache_slots = 0;
  if (fused_table && nb_max <= 4096 && p->p_max <= 4096) {
    sp.map_cache_blocks = (nb_max + 3) & ~3;
    sp.map_cache_slots = (p->p_max + 3) & ~3;
    smem += sizeof(int) * (size_t)(sp.map_cache_blocks + sp.map_cache_slots);
  }
  // the last CTA's top-k by value bins: keys, bins, list and state bytes, in the
  // score ring when it is large enough (the ring is idle once the scores are
  // written), else after everything else
  sp.binned_off = 0;
  sp.binned_cap = 0;
  if (ncand_max <= kClusterMaxCand) {
    const size_t capk = (size_t)((ncand_max + 3) & ~3);
    const size_t need = capk * 4 + (size_t)kBins * 4 * (kSelThreads / 32) + capk * 8 + ((capk + 15) & ~(size_t)15);
    sp.binned_cap = (int)capk;
    if (sp.ring_stages > 0 && 16 + need <= (size_t)sp.dyn_plan_off - (size_t)sp.ring_stages * 8 -
                                               (sp.consensus ? (size_t)((bpc * p->Hkv * 4 + 15) & ~15) : 0)) {
      sp.binned_off = 16;  // offset 0 means "radix"
    } else {
      smem = (smem + 15) & ~(size_t)15;
      if (smem == 0) smem = 16;
      sp.binned_off = (int)smem;
      smem += need;
    }
  }
  sp.u0 = r0 * p->U;
}


// How many clusters of cs CTAs with smem bytes each can be resident at once
// (0: none), cached per device, cluster size and shared-memory size.
static int select_cluster_capacity(int cs, size_t smem) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  static std::mutex mu;
  static std::map<std::tuple<int, int, size_t>, int> known;
  std::lock_guard<std::mutex> lock(mu);
  auto key = std::make_tuple(dev, cs, smem);
  auto it = known.find(key);
  if (it != known.end()) return it->second;
  int n = 0;
  bool ok = pi_smem_optin(reinterpret_cast<const void*>(select_cluster_kernel), (int)smem) == cudaSuccess;
  if (ok) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(cs, 1);
    cfg.blockDim = dim3(kSelThreads);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = cs;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaOccupancyMaxActiveClusters(&n, select_cluster_kernel, &cfg) != cudaSuccess) n = 0;
  }
  cudaGetLastError();  // a refused size is not an error of the next call
  known[key] = n;
  return n;
}

cudaError_t pi_launch_select(pi_pool* p, int layer, const void* q, const int* k_per_req, int* sel, int* nsel,
                             cudaStream_t s, int* fused_table, int mode, int r0, int nr, const void* k_new,
                             const void* v_new, bool pdl) {
  if (mode < 0) mode = p->mode;
  if (nr < 0) nr = p->R;
  if (nr == 0) return cudaSuccess;
  SelParams sp;
  int chunks = 1, ncand_max = 0;
  size_t smem = 0;
  // enough CTAs to cover every SM twice
  prepare_select(p, layer, q, k_per_req, sel, nsel, fused_table, mode, r0, nr, 2LL * p->num_sms, sp, chunks, smem,
                 &ncand_max);
  const long long units = (long long)nr * p->U;
  // the append folds into the cluster launch for one block set per request with a
  // recent window (the new token's block is then never a candidate); otherwise
  // the append kernel runs first
  const bool fold = k_new && p->U == 1 && p->W >= 1;
  if (k_new && !fold) {
    cudaError_t e = pi_launch_append(p, layer, k_new, v_new, s, false, r0, nr);
    if (e != cudaSuccess) return e;
  }
  if (p->select_cluster_on &&
      ncand_max <= (p->select_cluster_ctas > 0 ? kClusterMaxCand : kClusterFormMaxCand)) {
    const int cap_c = (ncand_max + 3) & ~3;
    SelParams sc = sp;
    ClusterArgs ca;
    ca.cap_keys = cap_c;
    ca.f.k_new = fold ? (const uint8_t*)k_new : nullptr;
    ca.f.v_new = fold ? (const uint8_t*)v_new : nullptr;
    ca.f.pool = p->pool;
    ca.f.slot_base = p->slot_base;
    ca.f.tail_sum = p->tail_sum;
    ca.f.ntok_w = p->ntok;
    // mean-key scores of one block set per request stream through a ring of
    // bulk-copy stages of 8 blocks (about 160 KiB in flight: one CTA per SM, or
    // 64 KiB and two CTAs per SM when the large ring's clusters would not all be
    // resident at once); the consensus score (G x the arithmetic) and head-wise
    // units (strided summary rows) keep two CTAs per SM
    const bool ring = !sc.consensus && p->U == 1;
    const int stage_bytes = 8 * p->Hkv * p->D * 4;
    const int ring_big = max(2, min(8, 163840 / stage_bytes));   // one CTA per SM
    const int ring_small = max(2, min(8, 65536 / stage_bytes));  // two CTAs per SM
    if (ring) sc.ring_stages = ring_big;
    const long long per_sm = ring ? 1 : 2;
    // dynamic shared memory for bpc candidates per CTA: the score ring (and the
    // consensus group scores, sized by bpc), the plan scratch and slot-map cache
    // (leader), then the leader's keys, bins, list and state
    auto layout = [&](int bpc_) -> size_t {
      sc.bpc = bpc_;
      size_t off = 0;
      if (sc.consensus) {
        sc.dyn_plan_off = sc.ring_stages * stage_bytes + sc.ring_stages * 8 + ((bpc_ * p->Hkv * 4 + 15) & ~15);
        off = sc.dyn_plan_off;
      } else if (ring) {
        sc.dyn_plan_off = (sc.ring_stages * stage_bytes + sc.ring_stages * 8 + 15) & ~15;
        off = sc.dyn_plan_off;
      }
      if (fused_table) off += pi_plan::plan_smem_bytes(p->max_blocks, p->cap, sc.lru_p2);
      off += sizeof(int) * (size_t)(sc.map_cache_blocks + sc.map_cache_slots);
      off = (off + 15) & ~(size_t)15;
      ca.keys_off = (int)off;
      off += (size_t)cap_c * 4;
      ca.hist_off = (int)off;
      off += (size_t)kBins * 4 * (kSelThreads / 32);
      ca.list_off = (int)off;
      off += (size_t)cap_c * 8;
      ca.state_off = (int)off;
      off += ((size_t)cap_c + 15) & ~(size_t)15;
      return off;
    };
    // one cluster of cs CTAs per unit: cs up to 16 with the launch's CTAs about
    // per_sm per SM and at least 8 candidates per CTA, then as large as still
    // lets every cluster of the launch be resident at once (the clusters need
    // no second wave)
    int cs = 1;
    while (cs < 16 && units * (cs * 2) <= per_sm * p->num_sms && (cs * 2) * 8 <= ncand_max) cs *= 2;
    if (p->select_cluster_ctas > 0) cs = max(1, min(p->select_cluster_ctas, (ncand_max + 7) / 8));
    for (; cs >= 1; cs = (cs > 1 ? cs / 2 : 0)) {
      const int bpc = ((((max(ncand_max, 1) + cs - 1) / cs) + 7) / 8) * 8;
      const int cs_used = max(1, (ncand_max + bpc - 1) / bpc);
      // the large ring first; when its clusters would not all be resident at
      // once, the small ring (two CTAs per SM) before a smaller cluster
      bool fits = false;
      size_t dsm = 0;
      for (int attempt = 0; attempt < (ring ? 2 : 1) && !fits; attempt++) {
        if (ring) sc.ring_stages = attempt == 0 ? ring_big : ring_small;
        dsm = layout(bpc);
        if (dsm > 220 * 1024) continue;
        const int cap_clusters = select_cluster_capacity(cs_used, dsm);
        if (cap_clusters <= 0) continue;
        // a launch larger than one wave of clusters is still correct (clusters
        // wait for room); prefer a smaller cluster that fits in one wave
        if (cs_used > 1 && units > cap_clusters && p->select_cluster_ctas == 0) continue;
        fits = true;
      }
      if (!fits) continue;
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3(cs_used, (unsigned)units);
      cfg.blockDim = dim3(kSelThreads);
      cfg.dynamicSmemBytes = dsm;
      cfg.stream = s;
      cudaLaunchAttribute attr[2];
      attr[0].id = cudaLaunchAttributeClusterDimension;
      attr[0].val.clusterDim.x = cs_used;
      attr[0].val.clusterDim.y = 1;
      attr[0].val.clusterDim.z = 1;
      attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
      attr[1].val.programmaticStreamSerializationAllowed = 1;
      cfg.attrs = attr;
      cfg.numAttrs = pdl ? 2 : 1;
      return cudaLaunchKernelEx(&cfg, select_cluster_kernel, sc, ca);
    }
  }
  if (fold) {
    cudaError_t e = pi_launch_append(p, layer, k_new, v_new, s, false, r0, nr);
    if (e != cudaSuccess) return e;
  }
  cudaError_t e0 = pi_smem_optin(reinterpret_cast<const void*>(select_kernel), (int)smem);
  if (e0 != cudaSuccess) return e0;
  dim3 grid(chunks, (unsigned)units);
  select_kernel<<<grid, kSelThreads, smem, s>>>(sp);
  return cudaGetLastError();
}

cudaError_t pi_launch_select_gather(pi_pool* p, int layer, const void* q, const int* k_per_req, int* sel, int* nsel,
                                    int* table, const void* k_new, const void* v_new, cudaStream_t s, int r0,
                                    int nr) {
  if (nr < 0) nr = p->R;
  if (nr == 0) return cudaSuccess;
  const int ctas = p->fused_ctas > 0 ? p->fused_ctas : max(1, p->num_sms / 4);
  FusedArgs f;
  SelParams sp;
  size_t smem = 0;
  // two selection items per CTA: a CTA that finishes early takes another
  prepare_select(p, layer, q, k_per_req, sel, nsel, table, p->mode, r0, nr, 2LL * ctas, sp, f.chunks, smem);
  GatherParams g = pi_gather_params(p, layer);
  g.plan_n += (size_t)r0 * p->U;
  g.plan += (size_t)r0 * p->U * p->cap;
  g.r0 = r0;
  g.nr = nr;
  g.units = nr * p->U;
  g.k_new = (const uint8_t*)k_new;
  g.v_new = (const uint8_t*)v_new;
  f.units = nr * p->U;
  f.items = f.units * f.chunks;
  const size_t ci = (size_t)layer * p->R * p->U + (size_t)r0 * p->U;  // counter of (layer, first unit)
  f.claim = p->fused_claim + ci;
  f.claim_base = p->fused_base[ci];
  f.ready = p->fused_ready + (size_t)layer * p->R * p->U;
  f.epoch = ++p->fused_epoch[layer];
  cudaError_t e0 = pi_smem_optin(reinterpret_cast<const void*>(select_gather_kernel), (int)smem);
  if (e0 != cudaSuccess) return e0;
  select_gather_kernel<<<ctas, kSelThreads, smem, s>>>(sp, g, f);
  cudaError_t e = cudaGetLastError();
  // every CTA claims until a claim fails: the counter grows by the items plus one per CTA
  if (e == cudaSuccess) p->fused_base[ci] += (unsigned long long)f.items + (unsigned long long)ctas;
  return e;
}

// ---------------------------------------------------------------------- API
extern "C" pi_status pi_update_summaries(pi_pool* p, int layer, const void* k_dev, int block_begin, int block_end,
                                         const int* ntok_host, pi_stream s) {
  if (!p || layer < 0 || layer >= p->L || !ntok_host || block_begin < 0 || block_end < block_begin)
    return PI_ERR_INVALID;
  for (int r = 0; r < p->R; r++)
    if (ntok_host[r] < 0 || (long long)ntok_host[r] > (long long)p->max_blocks * p->B) return PI_ERR_INVALID;
  if (block_end > p->max_blocks) block_end = p->max_blocks;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(s);
  int* stage = p->ntok_stage + (size_t)layer * p->R;
  PI_CUDA_TRY(cudaMemcpyAsync(stage, ntok_host, sizeof(int) * p->R, cudaMemcpyHostToDevice, st));
  const uint8_t* src = k_dev ? (const uint8_t*)k_dev
                             : p->host_dev + (size_t)(layer % p->host_layers) * p->R * p->region_bytes;
  int b1 = block_end;
  if (b1 <= block_begin) b1 = block_begin + 1;  // still record the counts
  PI_CUDA_TRY(pi_launch_summaries(p, layer, src, k_dev == nullptr, block_begin, b1, st, stage));
  for (int r = 0; r < p->R; r++) p->ntok_h[(size_t)r * p->L + layer] = ntok_host[r];
  return PI_OK;
}

extern "C" pi_status pi_append_kv(pi_pool* p, int layer, const void* k_new, const void* v_new, pi_stream s) {
  if (!p || layer < 0 || layer >= p->L || !k_new || !v_new) return PI_ERR_INVALID;
  if ((reinterpret_cast<uintptr_t>(k_new) | reinterpret_cast<uintptr_t>(v_new)) & 15) return PI_ERR_INVALID;
  for (int r = 0; r < p->R; r++)
    if ((long long)p->ntok_h[(size_t)r * p->L + layer] + 1 > (long long)p->max_blocks * p->B) return PI_ERR_INVALID;
  PI_CUDA_TRY(pi_launch_append(p, layer, k_new, v_new, reinterpret_cast<cudaStream_t>(s)));
  for (int r = 0; r < p->R; r++) p->ntok_h[(size_t)r * p->L + layer] += 1;
  return PI_OK;
}

extern "C" pi_status pi_select_topk(pi_pool* p, int layer, const void* q, const int* k_per_req, int mode, int* sel,
                                    int* nsel, pi_stream s) {
  if (!p || layer < 0 || layer >= p->L || !q || !k_per_req || !sel || !nsel) return PI_ERR_INVALID;
  // pools of one block set per request rank by either score; head-wise pools only per head
  if (p->U == 1 ? (mode != PI_SHARED && mode != PI_CONSENSUS) : mode != PI_HEADWISE) return PI_ERR_STATE;
  if (reinterpret_cast<uintptr_t>(q) & 3) return PI_ERR_INVALID;
  PI_CUDA_TRY(pi_launch_select(p, layer, q, k_per_req, sel, nsel, reinterpret_cast<cudaStream_t>(s), nullptr, mode));
  return PI_OK;
}

// Load the selection kernels on the current device and give each the largest
// dynamic shared memory the device allows, once, when a pool is created: a
// later launch then never loads a kernel or changes an attribute while other
// work of the pool is in flight (the cluster form's size changes as the
// context grows; the last-CTA form may first run many steps into a decode).
cudaError_t pi_prepare_select_kernels() {
  int dev = 0, optin = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  if (e != cudaSuccess) return e;
  const void* fns[] = {reinterpret_cast<const void*>(summaries_kernel), reinterpret_cast<const void*>(append_kernel),
                       reinterpret_cast<const void*>(select_kernel), reinterpret_cast<const void*>(select_gather_kernel),
                       reinterpret_cast<const void*>(select_cluster_kernel)};
  for (const void* fn : fns) {
    cudaFuncAttributes a;
    e = cudaFuncGetAttributes(&a, fn);
    if (e != cudaSuccess) return e;
    e = pi_smem_optin(fn, optin - (int)a.sharedSizeBytes);
    if (e != cudaSuccess) return e;
  }
  return cudaFuncSetAttribute(select_cluster_kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
}
