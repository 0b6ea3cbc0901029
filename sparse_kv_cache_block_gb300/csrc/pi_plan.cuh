// Recall plan of one unit (a request, or a request x KV head in head-wise
// pools), run by one CTA: which selected units are missing from the pool, which
// slots are free, and which missing unit goes to which free slot.
//
// "PulseInfer Guide: I/O-Centric Sparse KV Cache Offloading", section "The
// Gather-Scatter I/O Engine": recalled blocks are written into their pool page
// slots. The rule here (the library's reading): missing = selected units
// without a slot, in selection (ascending block) order; free = slots that are
// empty or hold an unselected unit, ascending; the i-th missing unit takes the
// i-th free slot, evicting what it held. Maps are not touched here; the copy
// kernel commits them.
#pragma once

#include "pi_internal.cuh"

namespace pi_plan {

// Exclusive scan over a CTA of NT threads; every thread must call it.
template <int NT>
__device__ __forceinline__ int cta_excl_scan(int v, int* warp_sums, int& total) {
  constexpr int NW = NT / 32;
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) warp_sums[w] = x;
  __syncthreads();
  if (w == 0) {
    int s = (lane < NW) ? warp_sums[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int y = __shfl_up_sync(0xffffffffu, s, o);
      if (lane >= o) s += y;
    }
    if (lane < NW) warp_sums[lane] = s;
  }
  __syncthreads();
  const int before = (w == 0) ? 0 : warp_sums[w - 1];
  total = warp_sums[NW - 1];
  __syncthreads();
  return before + x - v;
}

// free-slot counts up to this are ordered by counting ranks, larger ones by a
// bitonic sort
constexpr int kRankSortMax = 1024;

struct UnitArgs {
  const int* sel;        // this unit's selection [n], ascending
  int n;
  int* stamp;            // least-recently-selected policy: this unit's slot stamps [P], else nullptr
  int* epoch;            // and its epoch counter
  const int* sob;        // this unit's slot_of_block [max_blocks]
  const int* bos;        // this unit's block_of_slot [P]
  int P, max_blocks;
  int* table;            // out [n]
  int4* plan;            // out [cap]: (unit block, slot, evicted block, 0)
  int* plan_n;           // out: number of plan entries
  long long* counts;     // [0] misses, [1] hits (accumulated)
  unsigned* status;
  int empty_first;       // layer held whole in HBM: empty slots before stale ones (lowest-slot rule)
};

// Shared memory: bits [ceil(max_blocks/32)] + miss_pos [cap] + free_list [cap];
// with the least-recently-selected policy also keys [lru_p2] (8-byte aligned).
template <int NT>
__device__ void plan_unit(const UnitArgs& a, unsigned* bits, int* miss_pos, int* free_list, int* warp_sums,
                          unsigned long long* keys = nullptr, int lru_p2 = 0) {
  const int words = (a.max_blocks + 31) / 32;
  const int n = a.n;
  for (int w = threadIdx.x; w < words; w += NT) bits[w] = 0u;
  __syncthreads();
  for (int i = threadIdx.x; i < n; i += NT) {
    const int b = a.sel[i];
    if (b >= 0 && b < a.max_blocks) atomicOr(&bits[b >> 5], 1u << (b & 31));
  }
  __syncthreads();

  int nm = 0;
  for (int base = 0; base < n; base += NT) {
    const int i = base + threadIdx.x;
    int miss = 0;
    if (i < n) {
      const int b = a.sel[i];
      if (b < 0 || b >= a.max_blocks) {
        pi_flag(a.status, PI_DEV_BAD_INDEX);
        a.table[i] = -1;
      } else {
        const int s = a.sob[b];
        if (s < 0) {
          miss = 1;
        } else if (s >= a.P) {
          pi_flag(a.status, PI_DEV_BAD_INDEX);
          a.table[i] = -1;
        } else {
          a.table[i] = s;
        }
      }
    }
    int tot;
    const int pos = cta_excl_scan<NT>(miss, warp_sums, tot);
    if (miss) miss_pos[nm + pos] = i;
    nm += tot;
  }

  int nf = 0;
  if (a.stamp) {
    // least recently selected first: every free slot keyed by (stamp + 1, slot),
    // sorted ascending; empty slots carry stamp -1 and come first
    const int e_new = *a.epoch + 1;
    for (int base = 0; base < a.P; base += NT) {
      const int s = base + threadIdx.x;
      int fr = 0;
      if (s < a.P) {
        const int bb = a.bos[s];
        if (bb < 0) fr = 1;
        else if (bb >= a.max_blocks) pi_flag(a.status, PI_DEV_BAD_INDEX);
        else fr = ((bits[bb >> 5] >> (bb & 31)) & 1u) ? 0 : 1;
      }
      int tot;
      const int pos = cta_excl_scan<NT>(fr, warp_sums, tot);
      if (fr) {
        const int st = (a.bos[s] < 0) ? -1 : a.stamp[s];
        keys[nf + pos] = ((unsigned long long)(unsigned)(st + 1) << 32) | (unsigned)s;
      }
      nf += tot;
    }
    __syncthreads();
    if (nf <= kRankSortMax) {
      // few free slots: each key's rank is the number of smaller keys (keys are
      // unique: the slot index is in the low word); the nm lowest ranks are taken
      for (int i = threadIdx.x; i < nf; i += NT) {
        const unsigned long long x = keys[i];
        int rank = 0;
        for (int j = 0; j < nf; j++) rank += (keys[j] < x) ? 1 : 0;
        if (rank < nm) free_list[rank] = (int)(x & 0xffffffffu);
      }
    } else {
      int n2 = 1;
      while (n2 < nf) n2 <<= 1;
      if (n2 > lru_p2) {
        if (threadIdx.x == 0) pi_flag(a.status, PI_DEV_BAD_INDEX);
        n2 = 0;
        nf = 0;
      }
      for (int i = nf + threadIdx.x; i < n2; i += NT) keys[i] = ~0ull;
      __syncthreads();
      for (int k = 2; k <= n2; k <<= 1)
        for (int j = k >> 1; j > 0; j >>= 1) {
          for (int i = threadIdx.x; i < n2; i += NT) {
            const int ix = i ^ j;
            if (ix > i) {
              const unsigned long long x = keys[i], y = keys[ix];
              const bool up = (i & k) == 0;
              if ((x > y) == up) {
                keys[i] = y;
                keys[ix] = x;
              }
            }
          }
          __syncthreads();
        }
      for (int j = threadIdx.x; j < nm && j < nf; j += NT) free_list[j] = (int)(keys[j] & 0xffffffffu);
    }
    // stamp the slots of the hits now; new entries are stamped at commit
    for (int i = threadIdx.x; i < n; i += NT) {
      const int b = a.sel[i];
      if (b >= 0 && b < a.max_blocks) {
        const int s = a.sob[b];
        if (s >= 0 && s < a.P) a.stamp[s] = e_new;
      }
    }
    __syncthreads();
  }
  // lowest free slot first; a layer held whole in HBM takes its empty slots
  // before the slots of unselected blocks (two passes), so it evicts nothing
  // while room is left
  const int passes = a.empty_first ? 2 : 1;
  for (int pass = 0; pass < passes && nf < nm && !a.stamp; pass++)
    for (int base = 0; base < a.P && nf < nm; base += NT) {
      const int s = base + threadIdx.x;
      int fr = 0;
      if (s < a.P) {
        const int bb = a.bos[s];
        if (bb < 0) {
          fr = (passes == 1 || pass == 0) ? 1 : 0;
        } else if (bb >= a.max_blocks) {
          if (pass == passes - 1) pi_flag(a.status, PI_DEV_BAD_INDEX);
        } else if (passes == 1 || pass == 1) {
          fr = ((bits[bb >> 5] >> (bb & 31)) & 1u) ? 0 : 1;
        }
      }
      int tot;
      const int pos = cta_excl_scan<NT>(fr, warp_sums, tot);
      if (fr && nf + pos < nm) free_list[nf + pos] = s;
      nf += tot;
    }
  if (nf < nm) {
    if (threadIdx.x == 0) {
      pi_flag(a.status, PI_DEV_POOL_FULL);
      *a.plan_n = 0;
    }
    for (int j = threadIdx.x; j < nm; j += NT) a.table[miss_pos[j]] = -1;
    return;
  }
  const int stamp_new = a.stamp ? *a.epoch + 1 : 0;
  for (int j = threadIdx.x; j < nm; j += NT) {
    const int i = miss_pos[j];
    const int s = free_list[j];
    a.plan[j] = make_int4(a.sel[i], s, a.bos[s], stamp_new);
    a.table[i] = s;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    if (a.stamp) *a.epoch = stamp_new;
    *a.plan_n = nm;
    atomicAdd(reinterpret_cast<unsigned long long*>(a.counts + 0), (unsigned long long)nm);
    atomicAdd(reinterpret_cast<unsigned long long*>(a.counts + 1), (unsigned long long)(n - nm));
  }
}

// smallest power of two >= n (n >= 1)
__host__ __device__ inline int pow2_at_least(int n) {
  int p = 1;
  while (p < n) p <<= 1;
  return p;
}

// bytes of dynamic shared memory plan_unit needs; layout: [keys u64 x lru_p2]
// [bits][miss_pos][free_list]
__host__ __device__ inline size_t plan_smem_bytes(int max_blocks, int cap, int lru_p2 = 0) {
  return sizeof(unsigned long long) * (size_t)lru_p2 +
         sizeof(int) * ((size_t)(max_blocks + 31) / 32 + 2 * (size_t)cap);
}

}  // namespace pi_plan
