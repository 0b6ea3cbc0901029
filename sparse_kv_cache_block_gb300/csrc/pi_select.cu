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
#include "pi_gather.cuh"
#include "pi_internal.cuh"
#include "pi_plan.cuh"

namespace {

constexpr int kSelThreads = 256;

__device__ __forceinline__ float bf16_at(const uint16_t* p) { return __uint_as_float((uint32_t)(*p) << 16); }

// ------------------------------------------------------------------ a-1
// grid (blocks in range, R); one thread per 8 consecutive elements of one head.
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
  for (int t = 0; t < nv; t++) {
    uint4 v = *reinterpret_cast<const uint4*>(row + (size_t)t * D * 2);
    uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int j = 0; j < 4; j++) {
      s[2 * j] = __fadd_rn(s[2 * j], pi_bf16_lo(w[j]));
      s[2 * j + 1] = __fadd_rn(s[2 * j + 1], pi_bf16_hi(w[j]));
    }
  }
  const size_t rl = (size_t)r * L + layer;
  float* km = kmean + ((rl * max_blocks + b) * Hkv + g) * D + d;
  const float fn = (float)nv;
#pragma unroll
  for (int j = 0; j < 8; j++) km[j] = __fdiv_rn(s[j], fn);
  if (b == nb - 1) {
    float* ts = tail_sum + (rl * Hkv + g) * D + d;
#pragma unroll
    for (int j = 0; j < 8; j++) ts[j] = s[j];
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
__device__ __forceinline__ bool select_item(const SelParams& p, const int u, const int chunk, const int nchunks) {
  __shared__ __align__(16) float qs[1024];
  __shared__ int hist[512];
  __shared__ int warp_sums[kSelThreads / 32];
  __shared__ int bcast[4];
  extern __shared__ __align__(16) uint32_t dyn[];  // plan scratch, then the slot-map cache
  const int r = u / p.U;
  const int g = (p.U == 1) ? 0 : u % p.U;
  const int E = (p.U == 1) ? p.Hkv * p.D : p.D;
  const int goff = (p.U == 1) ? 0 : g * p.D;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const size_t rl = (size_t)r * p.L + p.layer;
  const int nt = p.ntok[rl];
  const int nb = (nt + p.B - 1) / p.B;
  const int ncand = max(0, nb - p.W);

  // qsum[e] = sum over the group's query heads (ascending) of q[h][d], fp32
  // (the mean-key score; the consensus ranking reads the heads one by one)
  for (int e = threadIdx.x; e < E && !p.consensus; e += kSelThreads) {
    const int gg = (p.U == 1) ? e / p.D : g;
    const int d = e % p.D;
    const uint16_t* qh = p.q + ((size_t)r * p.Hq + (size_t)gg * p.G) * p.D + d;
    float s = 0.0f;
    for (int j = 0; j < p.G; j++) s = __fadd_rn(s, bf16_at(qh + (size_t)j * p.D));
    qs[e] = s;
  }
  __syncthreads();

  // scores of this CTA's candidates: one warp per block, canonical lane order,
  // two blocks per pass so sixteen 16-byte loads per lane are in flight
  const int b_begin = chunk * p.bpc;
  const int b_end = min(ncand, b_begin + p.bpc);
  float* sc = p.scores + (size_t)u * p.max_blocks;
  const int chunks = (E + 127) / 128;
  constexpr int NW = kSelThreads / 32;
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
      sc[b_begin + bl] = total;
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
      sc[b] = acc;
      if (two) sc[b2] = acc2;
    }
  }

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

  int kreq = p.k_per_req[r];
  kreq = max(0, min(kreq, p.k_max));
  const int kk = min(kreq, ncand);
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
  int out_n = 0;
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

// Parameters, chunk count and dynamic shared memory of a selection launch over
// requests r0 .. r0+nr-1 whose grid should hold about `target` CTAs.
static void prepare_select(pi_pool* p, int layer, const void* q, const int* k_per_req, int* sel, int* nsel,
                           int* fused_table, int mode, int r0, int nr, long long target, SelParams& sp, int& chunks,
                           size_t& smem) {
  sp.q = (const uint16_t*)q;
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
  sp.u0 = r0 * p->U;
}

cudaError_t pi_launch_select(pi_pool* p, int layer, const void* q, const int* k_per_req, int* sel, int* nsel,
                             cudaStream_t s, int* fused_table, int mode, int r0, int nr) {
  if (mode < 0) mode = p->mode;
  if (nr < 0) nr = p->R;
  if (nr == 0) return cudaSuccess;
  SelParams sp;
  int chunks = 1;
  size_t smem = 0;
  // enough CTAs to cover every SM twice
  prepare_select(p, layer, q, k_per_req, sel, nsel, fused_table, mode, r0, nr, 2LL * p->num_sms, sp, chunks, smem);
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  dim3 grid(chunks, (unsigned)(nr * p->U));
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
  if (smem > 48 * 1024) {
    cudaError_t e =
        cudaFuncSetAttribute(select_gather_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
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
