// GQA sparse decode attention over the pool, read through the block table.
//
// "PulseInfer Guide: I/O-Centric Sparse KV Cache Offloading", section
// "PulseInfer Architectural Foundations": recalled blocks land in a paged KV
// pool in HBM and attention runs over them; "SoloHead Sparse Selection": the
// selected block set is shared by the query heads of a GQA group.
//
// Design (GB300): one CTA per (request, KV head, split of the selected blocks).
// A producer warp streams each selected block's K and V of that head (one slot =
// [Hkv][K|V][B][D], so a head's K+V is 4*B*D contiguous bytes) into a ring of
// shared-memory stages with 2D TMA loads (128-byte swizzle) signalled on
// mbarriers. Four consumer warps each take 16-token tiles and run bf16
// mma.sync with the tokens on the M side and the G query heads of the group on
// the N side (N = 8, padded when G < 8):
//   S^T[tok][h]  = K[tok][:] . q[h][:]          (fp32 accumulate)
//   O^T[d][h]   += V^T[d][tok] . P^T[tok][h]     (P in bf16, fp32 accumulate)
// P^T's operand fragment is the register transpose (movmatrix) of S^T's
// accumulator fragment, so P never touches shared memory. Online softmax in the
// log2 domain, fp32. Warps merge in shared memory. The 2..8 splits of a unit run
// as one thread-block cluster: each stores its partial (m, l, O) into the first
// CTA's shared memory, which merges them (or, where that extra shared memory
// would cost occupancy, every CTA merges a slice from its peers' partials);
// other split counts merge through a small global partial buffer, finalised by
// the last CTA of the unit.
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstdio>
#include <mutex>

#include "pi_internal.cuh"

namespace {

constexpr int kConsumerWarps = 4;
constexpr int kThreads = (kConsumerWarps + 1) * 32;

struct AttnParams {
  const uint16_t* q;
  const int* sel;
  const int* table;
  const int* nsel;
  const int* ntok;
  const long long* slot_base;
  const int* P;
  float* part_o;      // this layer: [R*Hkv][splits_max][G][D]
  float2* part_ml;    // this layer: [R*Hkv][splits_max][G]
  unsigned* counter;  // this layer: [R*Hkv]
  uint16_t* out;
  float* lse;
  float* logits;
  unsigned* status;
  int layer, L, Hq, Hkv, G, U, cap, splits, splits_max, bps;
  int cluster;        // 1: the splits of a unit form one thread-block cluster and merge through DSMEM
  int push;           // with cluster: every split stores its partial into the first CTA's shared memory
                      // (after the regular layout), which merges them alone
  int u0, nunits;     // the launch covers units u0 .. u0+nunits-1 (grid.y)
  float scale, scale_log2;
};

template <int D, int B>
struct AttnShape {
  static constexpr int kStage = 4 * B * D;  // K + V of one head of one block, bytes
  static constexpr int kNS = (98304 / kStage) < 2 ? 2 : ((98304 / kStage) > 8 ? 8 : (98304 / kStage));
  static constexpr int kSub = B * 128;      // one 64-column swizzled sub-tile
  static constexpr int kSelCap = 512;        // selected blocks one CTA may take
  static constexpr int kSmem = kNS * kStage + 1024 + 2 * kNS * 8 + 64 + 2 * kSelCap * 4;
  static constexpr int kMergeCap = (kNS * kStage) / 8;  // split (m, l) pairs the merge stages in shared memory
  // a CTA's merged partial for the cluster merge ([8][D] fp32 + [8] (m, l)), after
  // the warps' [4][G][D] + [4][G][2] in the (idle) stage memory
  static constexpr int kClusterPart = kConsumerWarps * 8 * D * 4 + kConsumerWarps * 8 * 2 * 4;
  static_assert(kClusterPart + 8 * D * 4 + 8 * 8 <= kNS * kStage, "cluster partial must fit the stage memory");
};

__device__ __forceinline__ void consumer_sync() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

// one output element: O = acc / l in bf16; d == 0 also writes lse = (M + log2 l) ln 2
__device__ __forceinline__ void store_out(const AttnParams& p, int r, int hq, int d, int D, float acc, float lsum,
                                          float M) {
  const float v = (lsum > 0.0f) ? acc / lsum : 0.0f;
  const __nv_bfloat16 bv = __float2bfloat16_rn(v);
  p.out[((size_t)r * p.Hq + hq) * D + d] = *reinterpret_cast<const uint16_t*>(&bv);
  if (p.lse && d == 0)
    p.lse[(size_t)r * p.Hq + hq] = (lsum > 0.0f) ? (M + log2f(lsum)) * 0.69314718055994530942f : -INFINITY;
}

template <int D, int B>
__global__ void __launch_bounds__(kThreads) attn_kernel(const __grid_constant__ CUtensorMap tmap, AttnParams p) {
  using S = AttnShape<D, B>;
  constexpr int NS = S::kNS;
  constexpr int TPB = B / 16;
  constexpr int KS = D / 16;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = pi_smem_addr(smem_raw);
  uint8_t* smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + NS * S::kStage);
  uint64_t* empty = full + NS;
  int* flags = reinterpret_cast<int*>(empty + NS);
  int* s_blk = flags + 16;            // this CTA's selected block ids
  int* s_slot = s_blk + S::kSelCap;   // and their pool slots

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == kConsumerWarps * 32) pi_tmap_prefetch(&tmap);
  pi_grid_dep_wait();  // selections, tables and token counts of earlier kernels are visible from here on
  pi_grid_dep_trigger();
  const int u = p.u0 + blockIdx.y;
  const int r = u / p.Hkv, g = u % p.Hkv;
  const int su = (p.U == 1) ? r : u;
  const int* selu = p.sel + (size_t)su * p.cap;
  const int* tabu = p.table + (size_t)su * p.cap;
  int n = p.nsel[su];
  const int split = blockIdx.x;
  const int i0 = split * p.bps;
  // the split's table entries are read up to the split's end (a row holds cap
  // entries) without waiting for the selection count, so that every load of
  // the prologue is in flight at once
  const int span = min(S::kSelCap, max(0, min(p.bps, p.cap - i0)));
  for (int i = threadIdx.x; i < span; i += kThreads) {
    s_blk[i] = selu[i0 + i];
    s_slot[i] = tabu[i0 + i];
  }
  const int nt = p.ntok[(size_t)r * p.L + p.layer];
  const int Pr = p.P[(size_t)r * p.L + p.layer];
  const long long gbase = p.slot_base[(size_t)r * p.L + p.layer];
  const int gid = lane >> 2, tig = lane & 3;
  uint32_t qb[KS][2];  // this group's query rows as the mma's B fragments (consumer warps)
  if (warp < kConsumerWarps) {
    const uint16_t* qrow = p.q + ((size_t)r * p.Hq + (size_t)g * p.G + gid) * D;
#pragma unroll
    for (int ks = 0; ks < KS; ks++) {
      qb[ks][0] = (gid < p.G) ? *reinterpret_cast<const uint32_t*>(qrow + ks * 16 + 2 * tig) : 0u;
      qb[ks][1] = (gid < p.G) ? *reinterpret_cast<const uint32_t*>(qrow + ks * 16 + 8 + 2 * tig) : 0u;
    }
  }
  if (n < 0 || n > p.cap) {
    if (threadIdx.x == 0) pi_flag(p.status, PI_DEV_BAD_INDEX);
    n = 0;
  }
  const int nblk = min(span, max(0, n - i0));

  if (threadIdx.x == 0) {
    for (int s = 0; s < NS; s++) {
      pi_mbar_init(&full[s], 1);
      pi_mbar_init(&empty[s], kConsumerWarps);
    }
    flags[0] = 0;
    pi_fence_barrier_init();
  }
  __syncthreads();

  if (warp == kConsumerWarps) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int issued = 0;
      for (int it = 0; it < nblk; it++) {
        const int s = it % NS;
        if (it >= NS && !pi_mbar_wait_bounded(&empty[s], ((it / NS) - 1) & 1, p.status)) break;
        int slot = s_slot[it];
        if (slot < 0 || slot >= Pr) {
          pi_flag(p.status, PI_DEV_BAD_INDEX);
          slot = 0;  // keep the barrier accounting whole; the unit's output is flagged
        }
        const int row_k = (int)(((gbase + slot) * p.Hkv + g) * 2 * B);
        uint8_t* ks = smem + s * S::kStage;
        uint8_t* vs = ks + B * D * 2;
        pi_mbar_arrive_expect_tx(&full[s], S::kStage);
#pragma unroll
        for (int h = 0; h < D / 64; h++) {
          pi_tma_load_2d(ks + h * S::kSub, &tmap, h * 64, row_k, &full[s]);
          pi_tma_load_2d(vs + h * S::kSub, &tmap, h * 64, row_k + B, &full[s]);
        }
        issued = it + 1;
      }
      // drain: every issued load has landed before the CTA may exit
      for (int it = max(0, issued - NS); it < issued; it++) pi_mbar_wait_bounded(&full[it % NS], (it / NS) & 1, p.status);
    }
  } else {
    // ------------------------------------------------------------ consumers
    float o[KS][4];
#pragma unroll
    for (int mt = 0; mt < KS; mt++) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.0f;
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.0f, l1 = 0.0f;
    const int h0 = 2 * tig, h1 = 2 * tig + 1;
    const int mat = lane >> 3, r8 = lane & 7;

    for (int it = 0; it < nblk; it++) {
      const int s = it % NS;
      if (!pi_mbar_wait_bounded(&full[s], (it / NS) & 1, p.status)) break;
      const int b = s_blk[it];
      int nv = nt - b * B;
      nv = nv > B ? B : nv;
      // a block whose slot is out of range was flagged by the producer, which
      // loaded slot 0 in its place to keep the barriers whole: skip its tokens
      const int sl = s_slot[it];
      if (b < 0 || sl < 0 || sl >= Pr) nv = 0;
      const uint32_t ks_base = pi_smem_addr(smem + s * S::kStage);
      const uint32_t vs_base = ks_base + B * D * 2;
#pragma unroll
      for (int j = 0; j < TPB; j++) {
        if (((it * TPB + j) & (kConsumerWarps - 1)) != warp) continue;
        const int t0 = j * 16;
        float c[4] = {0.0f, 0.0f, 0.0f, 0.0f};
        {
          const int tok = t0 + r8 + ((mat & 1) << 3);
#pragma unroll
          for (int ks = 0; ks < KS; ks++) {
            const int chunk = ((ks * 16) & 63) / 8 + (mat >> 1);
            const uint32_t addr = ks_base + ((ks * 16) / 64) * S::kSub + tok * 128 + ((chunk ^ (tok & 7)) << 4);
            uint32_t a[4];
            pi_ldmatrix_x4(a, addr);
            pi_mma_bf16(c, a, qb[ks][0], qb[ks][1]);
          }
        }
        const int ta = t0 + gid, tb = t0 + gid + 8;
        if (p.logits) {
          float* lg = p.logits + ((size_t)r * p.Hq + (size_t)g * p.G) * p.cap * B + (size_t)(i0 + it) * B;
          const size_t hs = (size_t)p.cap * B;
          if (h0 < p.G && ta < nv) lg[h0 * hs + ta] = c[0] * p.scale;
          if (h1 < p.G && ta < nv) lg[h1 * hs + ta] = c[1] * p.scale;
          if (h0 < p.G && tb < nv) lg[h0 * hs + tb] = c[2] * p.scale;
          if (h1 < p.G && tb < nv) lg[h1 * hs + tb] = c[3] * p.scale;
        }
        const float z0 = (ta < nv) ? c[0] * p.scale_log2 : -INFINITY;
        const float z1 = (ta < nv) ? c[1] * p.scale_log2 : -INFINITY;
        const float z2 = (tb < nv) ? c[2] * p.scale_log2 : -INFINITY;
        const float z3 = (tb < nv) ? c[3] * p.scale_log2 : -INFINITY;
        float mx0 = fmaxf(z0, z2), mx1 = fmaxf(z1, z3);
#pragma unroll
        for (int off = 4; off <= 16; off <<= 1) {
          mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
          mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
        }
        const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
        const float al0 = (mn0 == -INFINITY) ? 1.0f : pi_exp2(m0 - mn0);
        const float al1 = (mn1 == -INFINITY) ? 1.0f : pi_exp2(m1 - mn1);
        const float p0 = (mn0 == -INFINITY) ? 0.0f : pi_exp2(z0 - mn0);
        const float p1 = (mn1 == -INFINITY) ? 0.0f : pi_exp2(z1 - mn1);
        const float p2 = (mn0 == -INFINITY) ? 0.0f : pi_exp2(z2 - mn0);
        const float p3 = (mn1 == -INFINITY) ? 0.0f : pi_exp2(z3 - mn1);
        m0 = mn0;
        m1 = mn1;
        const uint32_t x0 = pi_pack_bf16(p0, p1);  // tokens t0+gid:   heads 2tig, 2tig+1
        const uint32_t x1 = pi_pack_bf16(p2, p3);  // tokens t0+gid+8
        // the row sums take the fp32 weights (the log-sum-exp keeps fp32 accuracy);
        // only the PV product sees them rounded to bf16
        l0 = l0 * al0 + (p0 + p2);
        l1 = l1 * al1 + (p1 + p3);
        const uint32_t b0 = pi_movmatrix_trans(x0);
        const uint32_t b1 = pi_movmatrix_trans(x1);
        {
          const int tok = t0 + r8 + ((mat >> 1) << 3);
#pragma unroll
          for (int mt = 0; mt < KS; mt++) {
            o[mt][0] *= al0;
            o[mt][1] *= al1;
            o[mt][2] *= al0;
            o[mt][3] *= al1;
            const int chunk = ((mt * 16) & 63) / 8 + (mat & 1);
            const uint32_t addr = vs_base + ((mt * 16) / 64) * S::kSub + tok * 128 + ((chunk ^ (tok & 7)) << 4);
            uint32_t a[4];
            pi_ldmatrix_x4_trans(a, addr);
            pi_mma_bf16(o[mt], a, b0, b1);
          }
        }
      }
      __syncwarp();
      if (lane == 0) pi_mbar_arrive(&empty[s]);
    }
    // row sums over the 8 lanes holding the other tokens of the same heads
#pragma unroll
    for (int off = 4; off <= 16; off <<= 1) {
      l0 += __shfl_xor_sync(0xffffffffu, l0, off);
      l1 += __shfl_xor_sync(0xffffffffu, l1, off);
    }
    consumer_sync();  // every consumer is done reading the stages
    float* ow = reinterpret_cast<float*>(smem);                 // [4][G][D]
    float* mlw = ow + kConsumerWarps * p.G * D;                 // [4][G][2]
#pragma unroll
    for (int mt = 0; mt < KS; mt++) {
      const int d = mt * 16 + gid;
      if (h0 < p.G) {
        ow[(warp * p.G + h0) * D + d] = o[mt][0];
        ow[(warp * p.G + h0) * D + d + 8] = o[mt][2];
      }
      if (h1 < p.G) {
        ow[(warp * p.G + h1) * D + d] = o[mt][1];
        ow[(warp * p.G + h1) * D + d + 8] = o[mt][3];
      }
    }
    if (gid == 0) {
      if (h0 < p.G) { mlw[(warp * p.G + h0) * 2] = m0; mlw[(warp * p.G + h0) * 2 + 1] = l0; }
      if (h1 < p.G) { mlw[(warp * p.G + h1) * 2] = m1; mlw[(warp * p.G + h1) * 2 + 1] = l1; }
    }
    consumer_sync();
    if (p.splits == 1) {
      // one CTA holds the whole unit: normalise and write the output here
      for (int e = threadIdx.x; e < p.G * D; e += 128) {
        const int h = e / D, d = e % D;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kConsumerWarps; w++) M = fmaxf(M, mlw[(w * p.G + h) * 2]);
        float acc = 0.0f, lsum = 0.0f;
        if (M != -INFINITY) {
#pragma unroll
          for (int w = 0; w < kConsumerWarps; w++) {
            const float f = pi_exp2(mlw[(w * p.G + h) * 2] - M);
            acc += f * ow[(w * p.G + h) * D + d];
            lsum += f * mlw[(w * p.G + h) * 2 + 1];
          }
        }
        store_out(p, r, g * p.G + h, d, D, acc, lsum, M);
      }
    } else if (p.cluster && p.push) {
      // this CTA's partial goes straight into the first CTA's push region, slot =
      // split: [splits][G][D] fp32, then [splits][G] (m, l); the cluster barrier
      // below orders these stores before the first CTA reads them
      const uint32_t region = pi_cluster_map(pi_smem_addr(smem_raw + S::kSmem), 0);
      const uint32_t po_r = region + (uint32_t)(split * p.G * D) * 4u;
      const uint32_t ml_r = region + (uint32_t)(p.splits * p.G * D) * 4u + (uint32_t)(split * p.G) * 8u;
      for (int e = threadIdx.x; e < p.G * D; e += 128) {
        const int h = e / D, d = e % D;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kConsumerWarps; w++) M = fmaxf(M, mlw[(w * p.G + h) * 2]);
        float acc = 0.0f, lsum = 0.0f;
        if (M != -INFINITY) {
#pragma unroll
          for (int w = 0; w < kConsumerWarps; w++) {
            const float f = pi_exp2(mlw[(w * p.G + h) * 2] - M);
            acc += f * ow[(w * p.G + h) * D + d];
            lsum += f * mlw[(w * p.G + h) * 2 + 1];
          }
        }
        pi_st_cluster_f32(po_r + (uint32_t)e * 4u, acc);
        if (d == 0) pi_st_cluster_f2(ml_r + (uint32_t)h * 8u, make_float2(M, lsum));
      }
    } else if (p.cluster) {
      // this CTA's partial stays in its own shared memory; the cluster merges below
      float* cpo = reinterpret_cast<float*>(smem + S::kClusterPart);  // [G][D]
      float2* cpml = reinterpret_cast<float2*>(cpo + p.G * D);        // [G]
      for (int e = threadIdx.x; e < p.G * D; e += 128) {
        const int h = e / D, d = e % D;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kConsumerWarps; w++) M = fmaxf(M, mlw[(w * p.G + h) * 2]);
        float acc = 0.0f, lsum = 0.0f;
        if (M != -INFINITY) {
#pragma unroll
          for (int w = 0; w < kConsumerWarps; w++) {
            const float f = pi_exp2(mlw[(w * p.G + h) * 2] - M);
            acc += f * ow[(w * p.G + h) * D + d];
            lsum += f * mlw[(w * p.G + h) * 2 + 1];
          }
        }
        cpo[h * D + d] = acc;
        if (d == 0) cpml[h] = make_float2(M, lsum);
      }
    } else {
      const int au = r * p.Hkv + g;
      float* po = p.part_o + ((size_t)au * p.splits_max + split) * p.G * D;
      float2* pml = p.part_ml + ((size_t)au * p.splits_max + split) * p.G;
      for (int e = threadIdx.x; e < p.G * D; e += 128) {
        const int h = e / D, d = e % D;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kConsumerWarps; w++) M = fmaxf(M, mlw[(w * p.G + h) * 2]);
        float acc = 0.0f, lsum = 0.0f;
        if (M != -INFINITY) {
#pragma unroll
          for (int w = 0; w < kConsumerWarps; w++) {
            const float f = pi_exp2(mlw[(w * p.G + h) * 2] - M);
            acc += f * ow[(w * p.G + h) * D + d];
            lsum += f * mlw[(w * p.G + h) * 2 + 1];
          }
        }
        po[h * D + d] = acc;
        if (d == 0) pml[h] = make_float2(M, lsum);
      }
      __threadfence();
      consumer_sync();
      if (threadIdx.x == 0) {
        const unsigned done = atomicAdd(p.counter + au, 1u);
        flags[0] = (done == (unsigned)p.splits - 1) ? 1 : 0;
      }
      consumer_sync();
      if (flags[0]) {
        if (threadIdx.x == 0) p.counter[au] = 0;
        __threadfence();
        const int G = p.G, ns = p.splits;
        const float* pob = p.part_o + (size_t)au * p.splits_max * G * D;
        const float2* pmb = p.part_ml + (size_t)au * p.splits_max * G;
        // every split's (m, l) in one round of loads into the (now idle) stage
        // memory; more than fits is read from L2 where it is used
        float2* sml = reinterpret_cast<float2*>(smem);
        const bool staged = ns * G <= S::kMergeCap;
        if (staged)
          for (int t = threadIdx.x; t < ns * G; t += 128) sml[t] = __ldcg(&pmb[t]);
        consumer_sync();
        auto ml_at = [&](int i) -> float2 { return staged ? sml[i] : __ldcg(&pmb[i]); };
        float2* shead = reinterpret_cast<float2*>(s_blk);  // [G] merged (M, l)
        if (threadIdx.x < G) {
          const int h = threadIdx.x;
          float M = -INFINITY;
          for (int s = 0; s < ns; s++) M = fmaxf(M, ml_at(s * G + h).x);
          float lsum = 0.0f;
          if (M != -INFINITY)
            for (int s = 0; s < ns; s++) {
              const float2 ml = ml_at(s * G + h);
              lsum += pi_exp2(ml.x - M) * ml.y;
            }
          shead[h] = make_float2(M, lsum);
        }
        consumer_sync();
        const float4* pob4 = reinterpret_cast<const float4*>(pob);
        for (int e4 = threadIdx.x; e4 < G * D / 4; e4 += 128) {
          const int h = (4 * e4) / D, d = (4 * e4) % D;
          const float2 head = shead[h];
          float4 acc = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
          if (head.x != -INFINITY) {
#pragma unroll 4
            for (int s = 0; s < ns; s++) {
              const float f = pi_exp2(ml_at(s * G + h).x - head.x);
              const float4 v = __ldcg(pob4 + (size_t)s * (G * D / 4) + e4);
              acc.x += f * v.x;
              acc.y += f * v.y;
              acc.z += f * v.z;
              acc.w += f * v.w;
            }
          }
          const int hq = g * G + h;
          store_out(p, r, hq, d, D, acc.x, head.y, head.x);
          store_out(p, r, hq, d + 1, D, acc.y, head.y, head.x);
          store_out(p, r, hq, d + 2, D, acc.z, head.y, head.x);
          store_out(p, r, hq, d + 3, D, acc.w, head.y, head.x);
        }
      }
    }  // more than one split
  }
  __syncthreads();
  if (p.cluster && p.push) {
    // the first CTA merges every split's partial from its own shared memory, in
    // split order (the same arithmetic as the pulled merge below)
    pi_cluster_sync();
    if (split != 0) return;
    const int G = p.G, ns = p.splits;
    const float* po_s = reinterpret_cast<const float*>(smem_raw + S::kSmem);  // [ns][G][D]
    const float2* ml_s = reinterpret_cast<const float2*>(po_s + ns * G * D);   // [ns][G]
    for (int e4 = threadIdx.x; e4 < G * D / 4; e4 += kThreads) {
      const int h = (4 * e4) / D, d = (4 * e4) % D;
      float M = -INFINITY;
      for (int c = 0; c < ns; c++) M = fmaxf(M, ml_s[c * G + h].x);
      float4 acc = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
      float lsum = 0.0f;
      if (M != -INFINITY) {
        for (int c = 0; c < ns; c++) {
          const float2 ml = ml_s[c * G + h];
          const float f = pi_exp2(ml.x - M);
          const float4 v = reinterpret_cast<const float4*>(po_s + (size_t)c * G * D)[e4];
          acc.x += f * v.x;
          acc.y += f * v.y;
          acc.z += f * v.z;
          acc.w += f * v.w;
          lsum += f * ml.y;
        }
      }
      const int hq = g * G + h;
      store_out(p, r, hq, d, D, acc.x, lsum, M);
      store_out(p, r, hq, d + 1, D, acc.y, lsum, M);
      store_out(p, r, hq, d + 2, D, acc.z, lsum, M);
      store_out(p, r, hq, d + 3, D, acc.w, lsum, M);
    }
  } else if (p.cluster) {
    // every CTA of the cluster (the unit's splits, rank = split) merges a slice of
    // the output from all the partials, read from the peers' shared memory
    pi_cluster_sync();
    const int G = p.G, ns = p.splits;
    const int n4 = G * D / 4;
    const int per = (n4 + ns - 1) / ns;
    const uint32_t cpo_local = pi_smem_addr(smem + S::kClusterPart);
    const uint32_t cpml_local = cpo_local + G * D * 4;
    const int e_end = min(n4, (split + 1) * per);
    for (int e4 = split * per + threadIdx.x; e4 < e_end; e4 += kThreads) {
      const int h = (4 * e4) / D, d = (4 * e4) % D;
      float M = -INFINITY;
      for (int c = 0; c < ns; c++) M = fmaxf(M, pi_ld_cluster_f2(pi_cluster_map(cpml_local + h * 8, c)).x);
      float4 acc = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
      float lsum = 0.0f;
      if (M != -INFINITY) {
        for (int c = 0; c < ns; c++) {
          const float2 ml = pi_ld_cluster_f2(pi_cluster_map(cpml_local + h * 8, c));
          const float f = pi_exp2(ml.x - M);
          const float4 v = pi_ld_cluster_f4(pi_cluster_map(cpo_local + e4 * 16, c));
          acc.x += f * v.x;
          acc.y += f * v.y;
          acc.z += f * v.z;
          acc.w += f * v.w;
          lsum += f * ml.y;
        }
      }
      const int hq = g * G + h;
      store_out(p, r, hq, d, D, acc.x, lsum, M);
      store_out(p, r, hq, d + 1, D, acc.y, lsum, M);
      store_out(p, r, hq, d + 2, D, acc.z, lsum, M);
      store_out(p, r, hq, d + 3, D, acc.w, lsum, M);
    }
    pi_cluster_sync();  // a CTA's partial must outlive every peer's reads of it
  }
}

// Bytes of the first CTA's push region: every split's partial [G][D] fp32 and (m, l).
int push_bytes(int splits, int G, int D) { return splits * (G * D * 4 + G * 8); }

template <int D, int B>
cudaError_t launch_attn(pi_pool* p, AttnParams ap, cudaStream_t s, bool pdl) {
  using S = AttnShape<D, B>;
  // the push merge takes shared memory beyond the regular layout; it is used
  // only where that keeps the kernel's CTAs per SM
  const int smem0 = S::kSmem;
  const int smem1 = S::kSmem + push_bytes(ap.splits, ap.G, D);
  ap.push = (ap.cluster && (228 * 1024) / (smem1 + 1024) >= (228 * 1024) / (smem0 + 1024)) ? 1 : 0;
  const int smem = ap.push ? smem1 : smem0;
  cudaError_t e = pi_smem_optin(reinterpret_cast<const void*>(attn_kernel<D, B>), smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(ap.splits, ap.nunits);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  // programmatic dependent launch: the CTAs launch and prefetch while the
  // previous kernel on the stream drains, and wait for it before any read
  cudaLaunchAttribute attr[2];
  int na = 0;
  if (pdl) {
    attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[na].val.programmaticStreamSerializationAllowed = 1;
    na++;
  }
  if (ap.cluster) {
    attr[na].id = cudaLaunchAttributeClusterDimension;
    attr[na].val.clusterDim.x = ap.splits;
    attr[na].val.clusterDim.y = 1;
    attr[na].val.clusterDim.z = 1;
    na++;
  }
  cfg.attrs = attr;
  cfg.numAttrs = na;
  return cudaLaunchKernelEx(&cfg, attn_kernel<D, B>, p->tmap, ap);
}

int attn_smem_bytes(int D, int B) {
  if (D == 128) {
    switch (B) {
      case 16: return AttnShape<128, 16>::kSmem;
      case 32: return AttnShape<128, 32>::kSmem;
      case 64: return AttnShape<128, 64>::kSmem;
      case 128: return AttnShape<128, 128>::kSmem;
    }
  } else {
    switch (B) {
      case 16: return AttnShape<64, 16>::kSmem;
      case 32: return AttnShape<64, 32>::kSmem;
      case 64: return AttnShape<64, 64>::kSmem;
      case 128: return AttnShape<64, 128>::kSmem;
    }
  }
  return 227 * 1024;
}

}  // namespace

int pi_attention_smem(int D, int B) { return attn_smem_bytes(D, B); }

// Load every attention kernel on the current device and opt it in to the
// device's largest dynamic shared memory once, when a pool is created (the
// regular layout and any push region of the cluster merge fit under it, so no
// kernel loads or attribute changes happen while a decode step is in flight).
cudaError_t pi_prepare_attention_kernels() {
  int dev = 0, optin = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  auto one = [&](const void* fn, int bytes) {
    if (e != cudaSuccess) return;
    cudaFuncAttributes a;
    e = cudaFuncGetAttributes(&a, fn);
    if (e == cudaSuccess) e = pi_smem_optin(fn, std::max(bytes, optin - (int)a.sharedSizeBytes));
  };
  one(reinterpret_cast<const void*>(attn_kernel<128, 16>), AttnShape<128, 16>::kSmem);
  one(reinterpret_cast<const void*>(attn_kernel<128, 32>), AttnShape<128, 32>::kSmem);
  one(reinterpret_cast<const void*>(attn_kernel<128, 64>), AttnShape<128, 64>::kSmem);
  one(reinterpret_cast<const void*>(attn_kernel<128, 128>), AttnShape<128, 128>::kSmem);
  one(reinterpret_cast<const void*>(attn_kernel<64, 16>), AttnShape<64, 16>::kSmem);
  one(reinterpret_cast<const void*>(attn_kernel<64, 32>), AttnShape<64, 32>::kSmem);
  one(reinterpret_cast<const void*>(attn_kernel<64, 64>), AttnShape<64, 64>::kSmem);
  one(reinterpret_cast<const void*>(attn_kernel<64, 128>), AttnShape<64, 128>::kSmem);
  return e;
}

cudaError_t pi_launch_attention(pi_pool* p, int layer, const void* q, const int* sel, const int* table,
                                const int* nsel, void* out, float* lse, float* logits, cudaStream_t s, int r0,
                                int nr, bool pdl) {
  if (nr < 0) nr = p->R;
  if (nr == 0) return cudaSuccess;
  AttnParams ap;
  ap.u0 = r0 * p->Hkv;
  ap.nunits = nr * p->Hkv;
  ap.q = (const uint16_t*)q;
  ap.sel = sel;
  ap.table = table;
  ap.nsel = nsel;
  ap.ntok = p->ntok;
  ap.slot_base = p->slot_base;
  ap.P = p->P;
  const size_t units = (size_t)p->R * p->Hkv;
  ap.part_o = p->attn_o + (size_t)layer * units * p->attn_max_splits * p->G * p->D;
  ap.part_ml = p->attn_ml + (size_t)layer * units * p->attn_max_splits * p->G;
  ap.counter = p->attn_counter + (size_t)layer * units;
  ap.out = (uint16_t*)out;
  ap.lse = lse;
  ap.logits = logits;
  ap.status = p->dev_status;
  ap.layer = layer;
  ap.L = p->L;
  ap.Hq = p->Hq;
  ap.Hkv = p->Hkv;
  ap.G = p->G;
  ap.U = p->U;
  ap.cap = p->cap;
  ap.splits_max = p->attn_max_splits;
  // split the selection so the grid fills the GPU in one wave at the kernel's
  // occupancy, with at most 512 selected blocks per CTA
  const int smem = attn_smem_bytes(p->D, p->B);
  const int per_sm = max(1, (228 * 1024) / (smem + 1024));
  int splits = (int)(((long long)per_sm * p->num_sms) / (long long)ap.nunits);
  if (p->attn_splits > 0) splits = p->attn_splits;
  splits = max(splits, (p->cap + 511) / 512);
  splits = max(1, min(splits, p->attn_max_splits));
  int bps = (p->cap + splits - 1) / splits;
  splits = (p->cap + bps - 1) / bps;
  ap.splits = splits;
  ap.bps = bps;
  ap.cluster = (p->attn_cluster && splits >= 2 && splits <= 8) ? 1 : 0;
  ap.scale = 1.0f / sqrtf((float)p->D);
  ap.scale_log2 = ap.scale * 1.4426950408889634f;
  if (p->D == 128) {
    switch (p->B) {
      case 16: return launch_attn<128, 16>(p, ap, s, pdl);
      case 32: return launch_attn<128, 32>(p, ap, s, pdl);
      case 64: return launch_attn<128, 64>(p, ap, s, pdl);
      case 128: return launch_attn<128, 128>(p, ap, s, pdl);
    }
  } else if (p->D == 64) {
    switch (p->B) {
      case 16: return launch_attn<64, 16>(p, ap, s, pdl);
      case 32: return launch_attn<64, 32>(p, ap, s, pdl);
      case 64: return launch_attn<64, 64>(p, ap, s, pdl);
      case 128: return launch_attn<64, 128>(p, ap, s, pdl);
    }
  }
  return cudaErrorInvalidValue;
}

extern "C" pi_status pi_sparse_decode(pi_pool* p, int layer, const void* q, const int* sel, const int* table,
                                      const int* nsel, void* out, float* lse, float* logits, pi_stream s) {
  if (!p || layer < 0 || layer >= p->L || !q || !sel || !table || !nsel || !out) return PI_ERR_INVALID;
  if (reinterpret_cast<uintptr_t>(q) & 3) return PI_ERR_INVALID;
  if (!p->tmap_ok) return PI_ERR_STATE;
  PI_CUDA_TRY(pi_launch_attention(p, layer, q, sel, table, nsel, out, lse, logits, reinterpret_cast<cudaStream_t>(s)));
  return PI_OK;
}

// ----------------------------------------------------------------------------
// Attention with no allocation (no pool, no cudaMalloc).
//
// For callers that cannot allocate device memory: engines that reserve all HBM
// up front in their own arena and forbid further cudaMalloc calls, or code that
// runs where a runtime allocation would stall or fail. They own the paged KV
// buffer, tables and outputs; the split-K partials, merge counters and per-request
// slot bases this kernel needs live in the fixed array below, which every GPU that
// loads the library holds until the process exits.
namespace {

constexpr int kNoAllocMaxUnits = 1024;   // batch * KV heads
constexpr int kNoAllocMaxParts = 2048;   // units * splits
constexpr int kNoAllocMaxCap = 512;      // selected blocks per request
constexpr int kNoAllocMaxGD = 8 * 128;   // query heads per group * head_dim

struct NoAllocLayout {
  static constexpr size_t o_bytes = (size_t)kNoAllocMaxParts * kNoAllocMaxGD * sizeof(float);
  static constexpr size_t ml_bytes = (size_t)kNoAllocMaxParts * 8 * sizeof(float2);
  static constexpr size_t ctr_bytes = (size_t)kNoAllocMaxUnits * sizeof(unsigned);
  static constexpr size_t base_bytes = (size_t)kNoAllocMaxUnits * sizeof(long long);
  static constexpr size_t p_bytes = (size_t)kNoAllocMaxUnits * sizeof(int);
  static constexpr size_t o_off = 0;
  static constexpr size_t ml_off = o_off + o_bytes;
  static constexpr size_t ctr_off = ml_off + ml_bytes;
  static constexpr size_t base_off = ctr_off + ctr_bytes;
  static constexpr size_t p_off = base_off + base_bytes;
  static constexpr size_t status_off = p_off + p_bytes;
  static constexpr size_t total = status_off + 256;
};

static __device__ __align__(256) unsigned char g_noalloc_scratch[NoAllocLayout::total];

constexpr int kNoAllocMaxDevices = 64;
std::mutex g_noalloc_mu;
unsigned char* g_noalloc_ptr[kNoAllocMaxDevices] = {};

// Counters and the status word start at zero; every request's slots start at
// global slot 0 of the caller's buffer and are bounded by its slot count.
__global__ void noalloc_prepare_kernel(unsigned char* scratch, int batch, int units, int n_slots) {
  unsigned* ctr = reinterpret_cast<unsigned*>(scratch + NoAllocLayout::ctr_off);
  long long* base = reinterpret_cast<long long*>(scratch + NoAllocLayout::base_off);
  int* P = reinterpret_cast<int*>(scratch + NoAllocLayout::p_off);
  for (int i = threadIdx.x; i < units; i += blockDim.x) ctr[i] = 0u;
  for (int r = threadIdx.x; r < batch; r += blockDim.x) {
    base[r] = 0;
    P[r] = n_slots;
  }
  if (threadIdx.x == 0) *reinterpret_cast<unsigned*>(scratch + NoAllocLayout::status_off) = 0u;
}

template <int D, int B>
cudaError_t launch_attn_noalloc(const CUtensorMap& tmap, const AttnParams& ap, int units, cudaStream_t s) {
  using S = AttnShape<D, B>;
  cudaError_t e = pi_smem_optin(reinterpret_cast<const void*>(attn_kernel<D, B>), S::kSmem);
  if (e != cudaSuccess) return e;
  dim3 grid(ap.splits, units);
  attn_kernel<D, B><<<grid, kThreads, S::kSmem, s>>>(tmap, ap);
  return cudaGetLastError();
}

}  // namespace

extern "C" pi_status pi_sparse_decode_noalloc_status(pi_stream stream) {
  int dev = 0;
  PI_CUDA_TRY(cudaGetDevice(&dev));
  if (dev < 0 || dev >= kNoAllocMaxDevices) return PI_ERR_INVALID;
  unsigned char* scratch = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    scratch = g_noalloc_ptr[dev];
  }
  if (!scratch) return PI_ERR_STATE;  // no call on this device yet
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  unsigned w = 0;
  PI_CUDA_TRY(cudaMemcpyAsync(&w, scratch + NoAllocLayout::status_off, sizeof(unsigned), cudaMemcpyDeviceToHost, s));
  PI_CUDA_TRY(cudaStreamSynchronize(s));
  if (w & PI_DEV_BAD_INDEX) return PI_ERR_DEVICE;
  if (w & PI_DEV_TIMEOUT) return PI_ERR_TIMEOUT;
  return PI_OK;
}

extern "C" pi_status pi_sparse_decode_noalloc(const void* kv_slots, long long n_slots, int batch, int hq, int hkv,
                                              int head_dim, int block_tokens, int cap, const void* q, const int* sel,
                                              const int* slot_table, const int* nsel, const int* ntok, void* out,
                                              float* lse, pi_stream stream) {
  if (!kv_slots || !q || !sel || !slot_table || !nsel || !ntok || !out) return PI_ERR_INVALID;
  if (batch <= 0 || hq <= 0 || hkv <= 0 || hq % hkv != 0 || hq / hkv > 8 || n_slots <= 0 || cap <= 0)
    return PI_ERR_INVALID;
  if (head_dim != 64 && head_dim != 128) return PI_ERR_INVALID;
  if (block_tokens != 16 && block_tokens != 32 && block_tokens != 64 && block_tokens != 128) return PI_ERR_INVALID;
  // the fixed scratch bounds every size this entry point accepts
  const long long units = (long long)batch * hkv;
  if (units > kNoAllocMaxUnits || cap > kNoAllocMaxCap) return PI_ERR_INVALID;
  if ((long long)(hq / hkv) * head_dim > kNoAllocMaxGD) return PI_ERR_INVALID;
  const unsigned long long rows = (unsigned long long)n_slots * hkv * 2 * block_tokens;
  if (rows >= (1ULL << 31)) return PI_ERR_INVALID;
  if ((reinterpret_cast<uintptr_t>(kv_slots) & 15) || (reinterpret_cast<uintptr_t>(q) & 3)) return PI_ERR_INVALID;

  int dev = 0;
  PI_CUDA_TRY(cudaGetDevice(&dev));
  if (dev < 0 || dev >= kNoAllocMaxDevices) return PI_ERR_INVALID;
  unsigned char* scratch = nullptr;
  {
    // first call on this device: resolve the array's device address (this device is current)
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    if (!g_noalloc_ptr[dev]) {
      void* ptr = nullptr;
      cudaError_t e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
      if (e != cudaSuccess || !ptr) {
        pi_note_cuda_error(e, "cudaGetSymbolAddress(g_noalloc_scratch)", __FILE__, __LINE__);
        return PI_ERR_CUDA;
      }
      g_noalloc_ptr[dev] = static_cast<unsigned char*>(ptr);
    }
    scratch = g_noalloc_ptr[dev];
  }

  void* fn = nullptr;
  cudaDriverEntryPointQueryResult qres;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &qres) != cudaSuccess ||
      qres != cudaDriverEntryPointSuccess || !fn) {
    cudaGetLastError();
    return PI_ERR_CUDA;
  }
  CUtensorMap tmap;
  cuuint64_t dims[2] = {(cuuint64_t)head_dim, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)head_dim * 2};
  cuuint32_t box[2] = {64, (cuuint32_t)block_tokens};
  cuuint32_t estr[2] = {1, 1};
  if (reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn)(
          &tmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(kv_slots), dims, strides, box, estr,
          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return PI_ERR_INVALID;

  int num_sms = 0;
  PI_CUDA_TRY(cudaDeviceGetAttribute(&num_sms, cudaDevAttrMultiProcessorCount, dev));
  const int G = hq / hkv;
  const int smem = attn_smem_bytes(head_dim, block_tokens);
  const int per_sm = max(1, (228 * 1024) / (smem + 1024));
  int splits = (int)(((long long)per_sm * max(num_sms, 1)) / units);
  splits = max(1, min(splits, min(cap, (int)(kNoAllocMaxParts / units))));
  int bps = (cap + splits - 1) / splits;
  splits = (cap + bps - 1) / bps;

  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  noalloc_prepare_kernel<<<1, 256, 0, s>>>(scratch, batch, (int)units, (int)min(n_slots, (long long)INT_MAX));
  PI_CUDA_TRY(cudaGetLastError());

  AttnParams ap;
  ap.q = (const uint16_t*)q;
  ap.sel = sel;
  ap.table = slot_table;
  ap.nsel = nsel;
  ap.ntok = ntok;
  ap.slot_base = reinterpret_cast<const long long*>(scratch + NoAllocLayout::base_off);
  ap.P = reinterpret_cast<const int*>(scratch + NoAllocLayout::p_off);
  ap.part_o = reinterpret_cast<float*>(scratch + NoAllocLayout::o_off);
  ap.part_ml = reinterpret_cast<float2*>(scratch + NoAllocLayout::ml_off);
  ap.counter = reinterpret_cast<unsigned*>(scratch + NoAllocLayout::ctr_off);
  ap.out = (uint16_t*)out;
  ap.lse = lse;
  ap.logits = nullptr;
  ap.status = reinterpret_cast<unsigned*>(scratch + NoAllocLayout::status_off);
  ap.layer = 0;
  ap.L = 1;
  ap.Hq = hq;
  ap.Hkv = hkv;
  ap.G = G;
  ap.U = 1;
  ap.cap = cap;
  ap.splits = splits;
  ap.splits_max = splits;
  ap.bps = bps;
  ap.u0 = 0;
  ap.nunits = (int)units;
  ap.cluster = 0;
  ap.push = 0;
  ap.scale = 1.0f / sqrtf((float)head_dim);
  ap.scale_log2 = ap.scale * 1.4426950408889634f;
  cudaError_t e = cudaErrorInvalidValue;
  if (head_dim == 128) {
    switch (block_tokens) {
      case 16: e = launch_attn_noalloc<128, 16>(tmap, ap, (int)units, s); break;
      case 32: e = launch_attn_noalloc<128, 32>(tmap, ap, (int)units, s); break;
      case 64: e = launch_attn_noalloc<128, 64>(tmap, ap, (int)units, s); break;
      case 128: e = launch_attn_noalloc<128, 128>(tmap, ap, (int)units, s); break;
    }
  } else {
    switch (block_tokens) {
      case 16: e = launch_attn_noalloc<64, 16>(tmap, ap, (int)units, s); break;
      case 32: e = launch_attn_noalloc<64, 32>(tmap, ap, (int)units, s); break;
      case 64: e = launch_attn_noalloc<64, 64>(tmap, ap, (int)units, s); break;
      case 128: e = launch_attn_noalloc<64, 128>(tmap, ap, (int)units, s); break;
    }
  }
  PI_CUDA_TRY(e);
  return PI_OK;
}
