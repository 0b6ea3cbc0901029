// Copy side of a recall: the parameters of a gather and the per-item device
// code, shared by the stand-alone gather kernel and the fused select + gather
// kernel.
//
// "PulseInfer Guide: I/O-Centric Sparse KV Cache Offloading", "The
// Gather-Scatter I/O Engine": each missing block is copied from the host store
// into the pool slot its plan entry names, and the slot maps are committed.
#pragma once

#include "pi_internal.cuh"

struct GatherParams {
  const int* plan_n;
  const int4* plan;
  int* slot_of;
  int* block_of;
  int* slot_stamp;           // stamped at commit under the least-recently-selected policy
  const uint8_t* host_src;   // device address of this layer's host store (request 0)
  uint8_t* host_dst;         // same memory, writable (write-through of new tokens)
  const uint8_t* stage_src;  // staged arm: device staging buffer (entries e_begin..)
  uint8_t* pool;
  const long long* slot_base;
  const int* P;
  const int* ntok;           // [R][L] (after this step's append)
  const uint8_t* k_new;      // optional [R][Hkv][D]: this step's token of this layer
  const uint8_t* v_new;
  unsigned* status;
  long long region_bytes;
  long long e_begin, e_end;  // entry range to process (global plan order)
  int layer, L, R, U, Hkv, B, D, max_blocks, p_max, cap, units, copy_bytes, block_bytes, do_copy, do_commit;
  int r0, nr;                // requests of this launch: r0 .. r0+nr-1 (units r0*U ..; plan pointers offset)
};

// Parameters of a gather over every request of `layer` (plan pointers at unit 0).
GatherParams pi_gather_params(pi_pool* p, int layer);

#ifdef __CUDACC__
__device__ __forceinline__ uint4 pi_ld_stream(const uint4* ptr) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(ptr));
  return v;
}

// Write this step's token of every request of the launch through to the host
// store (one CTA).
template <int THREADS>
__device__ __forceinline__ void pi_gather_write_through(const GatherParams& g) {
  const int row_bytes = g.D * 2;
  const int row_words = row_bytes / 16;
  const int per_req = g.Hkv * 2 * row_words;  // 16-byte words of K and V rows
  for (int w = threadIdx.x; w < g.nr * per_req; w += THREADS) {
    const int r = g.r0 + w / per_req, rem = w % per_req;
    const int g_ = rem / (2 * row_words), kv = (rem / row_words) & 1, x = rem % row_words;
    const int t = g.ntok[(size_t)r * g.L + g.layer] - 1;
    if (t < 0 || t / g.B >= g.max_blocks) continue;
    const int b = t / g.B, tp = t % g.B;
    const uint8_t* src = (kv ? g.v_new : g.k_new) + (((size_t)r * g.Hkv + g_) * g.D) * 2 + (size_t)x * 16;
    uint8_t* dst = g.host_dst + (size_t)r * g.region_bytes + (size_t)b * g.block_bytes +
                   (((size_t)g_ * 2 + kv) * g.B + tp) * row_bytes + (size_t)x * 16;
    *reinterpret_cast<uint4*>(dst) = *reinterpret_cast<const uint4*>(src);
  }
}

// One item of a gather: chunk c (of `chunk` bytes) of plan entry j of the
// launch's unit u (plan pointers offset to the launch). The CTA copies the
// chunk with DEPTH 16-byte loads in flight per thread, rewrites the rows of
// this step's token when the chunk holds them, and the item of chunk 0 commits
// the entry's slot maps. stage_idx: the entry's position in the staging buffer
// (staged arm). The plan is read through L2 (it may have been written by
// another CTA of the same launch). Every branch is uniform across the CTA.
template <int DEPTH, int THREADS>
__device__ __forceinline__ void pi_gather_item(const GatherParams& g, int u, int j, int c, int chunk,
                                               long long stage_idx) {
  const int row_bytes = g.D * 2;
  const int row_words = row_bytes / 16;
  const int4 pe = __ldcg(g.plan + (size_t)u * g.cap + j);
  const int r = g.r0 + u / g.U, gu = u % g.U;
  const int Pr = g.P[(size_t)r * g.L + g.layer];
  const bool ok = pe.x >= 0 && pe.x < g.max_blocks && pe.y >= 0 && pe.y < Pr && pe.z < g.max_blocks;
  if (!ok) {
    if (threadIdx.x == 0) pi_flag(g.status, PI_DEV_BAD_INDEX);
    return;
  }
  const size_t head_off = (g.U > 1) ? (size_t)gu * g.copy_bytes : 0;
  if (g.do_copy) {
    const size_t off = (size_t)c * chunk;
    const int len = min(chunk, g.copy_bytes - c * chunk);
    const uint8_t* src = g.stage_src ? g.stage_src + (size_t)stage_idx * g.copy_bytes + off
                                     : g.host_src + (size_t)r * g.region_bytes + (size_t)pe.x * g.block_bytes +
                                           head_off + off;
    uint8_t* blk = g.pool + (size_t)(g.slot_base[(size_t)r * g.L + g.layer] + pe.y) * g.block_bytes;
    uint8_t* dst = blk + head_off + off;
    const uint4* s4 = reinterpret_cast<const uint4*>(src);
    uint4* d4 = reinterpret_cast<uint4*>(dst);
    const int words = len >> 4;
    for (int w = threadIdx.x; w < words; w += THREADS * DEPTH) {
      uint4 v[DEPTH];
#pragma unroll
      for (int k = 0; k < DEPTH; k++)
        if (w + k * THREADS < words) v[k] = pi_ld_stream(s4 + w + k * THREADS);
#pragma unroll
      for (int k = 0; k < DEPTH; k++)
        if (w + k * THREADS < words) d4[w + k * THREADS] = v[k];
    }
    if (g.k_new) {
      const int t = g.ntok[(size_t)r * g.L + g.layer] - 1;
      if (t >= 0 && t / g.B == pe.x) {
        // this block holds the new token: rewrite its rows that fall in this chunk
        __syncthreads();
        const int tp = t % g.B;
        const int heads = (g.U > 1) ? 1 : g.Hkv;
        for (int w = threadIdx.x; w < heads * 2 * row_words; w += THREADS) {
          const int hh = w / (2 * row_words), kv = (w / row_words) & 1, x = w % row_words;
          const int g_ = (g.U > 1) ? gu : hh;
          const size_t rel = (((size_t)g_ * 2 + kv) * g.B + tp) * row_bytes + (size_t)x * 16;  // in the block
          const size_t lo_b = head_off + off, hi_b = head_off + off + len;
          if (rel >= lo_b && rel < hi_b) {
            const uint8_t* tsrc = (kv ? g.v_new : g.k_new) + (((size_t)r * g.Hkv + g_) * g.D) * 2 + (size_t)x * 16;
            *reinterpret_cast<uint4*>(blk + rel) = *reinterpret_cast<const uint4*>(tsrc);
          }
        }
      }
    }
  }
  if (g.do_commit && c == 0 && threadIdx.x == 0) {
    const size_t rlu = ((size_t)r * g.L + g.layer) * g.U + gu;
    int* sob = g.slot_of + rlu * g.max_blocks;
    int* bos = g.block_of + rlu * g.p_max;
    if (pe.z >= 0) sob[pe.z] = -1;
    sob[pe.x] = pe.y;
    bos[pe.y] = pe.x;
    if (g.slot_stamp) g.slot_stamp[rlu * g.p_max + pe.y] = pe.w;
  }
}
#endif
