// Recall engine: pool plan, UVA gather kernel, and the measured copy arms.
//
// "PulseInfer Guide: I/O-Centric Sparse KV Cache Offloading":
//  - "The Small-Packet PCIe DMA Tax": one host->device copy per small paged
//    block loses most of the link bandwidth to per-transfer overhead.
//  - "The Gather-Scatter I/O Engine": gather the scattered blocks, move them in
//    one bulk transfer, scatter them into their pool page slots.
// On GB300 the GPU reads the pinned host store directly through its mapping
// (NVLink-C2C or PCIe), so the default arm is one gather kernel that copies every
// missing block straight into its slot: no staging, no host round trip. The
// per-run cudaMemcpyAsync arm and the guide's three-phase staged arm are kept as
// measured comparisons.
#include <omp.h>

#include <chrono>
#include <cstring>

#include "pi_internal.cuh"

namespace {

constexpr int kPlanThreads = 256;
constexpr int kGatherThreads = 256;
constexpr int kChunkBytes = kGatherThreads * 16 * 4;  // 16 KiB per CTA iteration

__device__ __forceinline__ int cta_excl_scan(int v, int* warp_sums, int& total) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  constexpr int NW = kPlanThreads / 32;
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

struct PlanParams {
  const int* sel;
  const int* nsel;
  int* table;
  const int* slot_of;
  const int* block_of;
  int* plan_n;
  int4* plan;
  const int* P;
  long long* counts;  // [0] misses, [1] hits
  unsigned* status;
  int layer, L, U, max_blocks, p_max, cap;
};

// One CTA per unit (request, or request x KV head). Writes the table and the
// plan; the maps are committed later by the copy kernel.
__global__ void __launch_bounds__(kPlanThreads) plan_kernel(PlanParams p) {
  extern __shared__ int sm[];
  const int words = (p.max_blocks + 31) / 32;
  unsigned* bits = reinterpret_cast<unsigned*>(sm);
  int* miss_pos = sm + words;
  int* free_list = miss_pos + p.cap;
  __shared__ int warp_sums[kPlanThreads / 32];

  const int u = blockIdx.x;
  const int r = u / p.U, gu = u % p.U;
  const size_t rlu = ((size_t)r * p.L + p.layer) * p.U + gu;
  const int* sob = p.slot_of + rlu * p.max_blocks;
  const int* bos = p.block_of + rlu * p.p_max;
  const int Pr = p.P[r];
  const int* su = p.sel + (size_t)u * p.cap;
  int* tab = p.table + (size_t)u * p.cap;
  int n = p.nsel[u];
  if (n < 0 || n > p.cap) {
    if (threadIdx.x == 0) pi_flag(p.status, PI_DEV_BAD_INDEX);
    n = 0;
  }
  for (int w = threadIdx.x; w < words; w += kPlanThreads) bits[w] = 0u;
  __syncthreads();
  for (int i = threadIdx.x; i < n; i += kPlanThreads) {
    const int b = su[i];
    if (b >= 0 && b < p.max_blocks) atomicOr(&bits[b >> 5], 1u << (b & 31));
  }
  __syncthreads();

  // missing = selected without a slot, in selection (ascending) order
  int nm = 0;
  for (int base = 0; base < n; base += kPlanThreads) {
    const int i = base + threadIdx.x;
    int miss = 0;
    if (i < n) {
      const int b = su[i];
      if (b < 0 || b >= p.max_blocks) {
        pi_flag(p.status, PI_DEV_BAD_INDEX);
        tab[i] = -1;
      } else {
        const int s = sob[b];
        if (s < 0) {
          miss = 1;
        } else if (s >= Pr) {
          pi_flag(p.status, PI_DEV_BAD_INDEX);
          tab[i] = -1;
        } else {
          tab[i] = s;
        }
      }
    }
    int tot;
    const int pos = cta_excl_scan(miss, warp_sums, tot);
    if (miss) miss_pos[nm + pos] = i;
    nm += tot;
  }

  // free = slots empty or holding an unselected block, ascending; first nm only
  int nf = 0;
  for (int base = 0; base < Pr && nf < nm; base += kPlanThreads) {
    const int s = base + threadIdx.x;
    int fr = 0;
    if (s < Pr) {
      const int bb = bos[s];
      if (bb < 0) {
        fr = 1;
      } else if (bb >= p.max_blocks) {
        pi_flag(p.status, PI_DEV_BAD_INDEX);
      } else {
        fr = ((bits[bb >> 5] >> (bb & 31)) & 1u) ? 0 : 1;
      }
    }
    int tot;
    const int pos = cta_excl_scan(fr, warp_sums, tot);
    if (fr && nf + pos < nm) free_list[nf + pos] = s;
    nf += tot;
  }
  if (nf < nm) {
    if (threadIdx.x == 0) {
      pi_flag(p.status, PI_DEV_POOL_FULL);
      p.plan_n[u] = 0;
    }
    for (int j = threadIdx.x; j < nm; j += kPlanThreads) tab[miss_pos[j]] = -1;
    return;
  }
  int4* pl = p.plan + (size_t)u * p.cap;
  for (int j = threadIdx.x; j < nm; j += kPlanThreads) {
    const int i = miss_pos[j];
    const int s = free_list[j];
    pl[j] = make_int4(su[i], s, bos[s], 0);
    tab[i] = s;
  }
  if (threadIdx.x == 0) {
    p.plan_n[u] = nm;
    atomicAdd(reinterpret_cast<unsigned long long*>(p.counts + 0), (unsigned long long)nm);
    atomicAdd(reinterpret_cast<unsigned long long*>(p.counts + 1), (unsigned long long)(n - nm));
  }
}

struct GatherParams {
  const int* plan_n;
  const int4* plan;
  int* slot_of;
  int* block_of;
  const uint8_t* host_src;   // device address of this layer's host store (request 0)
  const uint8_t* stage_src;  // staged arm: device staging buffer (entries e_begin..)
  uint8_t* pool;
  const long long* slot_base;
  const int* P;
  unsigned* status;
  long long region_bytes;
  long long e_begin, e_end;  // entry range to process (global plan order)
  int layer, L, U, max_blocks, p_max, cap, units, copy_bytes, block_bytes, do_copy, do_commit;
};

__device__ __forceinline__ uint4 ld_stream(const uint4* ptr) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(ptr));
  return v;
}

// Grid-stride over (plan entry, 16 KiB chunk). Each thread keeps four 16-byte
// loads in flight, so a CTA has 16 KiB outstanding on the host link.
__global__ void __launch_bounds__(kGatherThreads) gather_kernel(GatherParams g) {
  extern __shared__ long long prefix[];  // [units + 1]
  __shared__ int warp_sums[kGatherThreads / 32];
  // prefix sums of the per-unit plan counts (every CTA computes its own copy)
  long long run = 0;
  for (int base = 0; base < g.units; base += kGatherThreads) {
    const int u = base + threadIdx.x;
    const int v = (u < g.units) ? g.plan_n[u] : 0;
    // reuse the plan kernel's scan shape
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    if (lane == 31) warp_sums[w] = x;
    __syncthreads();
    int before = 0, tot = 0;
    for (int k = 0; k < kGatherThreads / 32; k++) {
      if (k < w) before += warp_sums[k];
      tot += warp_sums[k];
    }
    if (u < g.units) prefix[u] = run + before + x - v;
    run += tot;
    __syncthreads();
  }
  if (threadIdx.x == 0) prefix[g.units] = run;
  __syncthreads();
  const long long total_entries = run;
  const long long e0 = g.e_begin, e1 = min(g.e_end, total_entries);
  if (e1 <= e0) return;
  const int chunk = min(g.copy_bytes, kChunkBytes);
  const int cpe = g.do_copy ? (g.copy_bytes + chunk - 1) / chunk : 1;
  const long long items = (e1 - e0) * cpe;
  for (long long it = blockIdx.x; it < items; it += gridDim.x) {
    const long long e = e0 + it / cpe;
    const int c = (int)(it % cpe);
    // unit owning entry e: last u with prefix[u] <= e
    int lo = 0, hi = g.units - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (prefix[mid] <= e) lo = mid; else hi = mid - 1;
    }
    const int u = lo;
    const int j = (int)(e - prefix[u]);
    const int4 pe = g.plan[(size_t)u * g.cap + j];
    const int r = u / g.U, gu = u % g.U;
    const int Pr = g.P[r];
    const bool ok = pe.x >= 0 && pe.x < g.max_blocks && pe.y >= 0 && pe.y < Pr && pe.z < g.max_blocks;
    if (!ok) {
      if (threadIdx.x == 0) pi_flag(g.status, PI_DEV_BAD_INDEX);
      continue;
    }
    const size_t head_off = (g.U > 1) ? (size_t)gu * g.copy_bytes : 0;
    if (g.do_copy) {
      const size_t off = (size_t)c * chunk;
      const int len = min(chunk, g.copy_bytes - c * chunk);
      const uint8_t* src = g.stage_src ? g.stage_src + (size_t)(e - e0) * g.copy_bytes + off
                                       : g.host_src + (size_t)r * g.region_bytes +
                                             (size_t)pe.x * g.block_bytes + head_off + off;
      uint8_t* dst = g.pool + (size_t)(g.slot_base[r] + (long long)g.layer * Pr + pe.y) * g.block_bytes + head_off + off;
      const uint4* s4 = reinterpret_cast<const uint4*>(src);
      uint4* d4 = reinterpret_cast<uint4*>(dst);
      const int words = len >> 4;
      for (int w = threadIdx.x; w < words; w += kGatherThreads * 4) {
        uint4 v[4];
#pragma unroll
        for (int k = 0; k < 4; k++)
          if (w + k * kGatherThreads < words) v[k] = ld_stream(s4 + w + k * kGatherThreads);
#pragma unroll
        for (int k = 0; k < 4; k++)
          if (w + k * kGatherThreads < words) d4[w + k * kGatherThreads] = v[k];
      }
    }
    if (g.do_commit && c == 0 && threadIdx.x == 0) {
      const size_t rlu = ((size_t)r * g.L + g.layer) * g.U + gu;
      int* sob = g.slot_of + rlu * g.max_blocks;
      int* bos = g.block_of + rlu * g.p_max;
      if (pe.z >= 0) sob[pe.z] = -1;
      sob[pe.x] = pe.y;
      bos[pe.y] = pe.x;
    }
  }
}

}  // namespace

cudaError_t pi_launch_plan(pi_pool* p, int layer, const int* sel, const int* nsel, int* table, cudaStream_t s) {
  PlanParams pp;
  pp.sel = sel;
  pp.nsel = nsel;
  pp.table = table;
  pp.slot_of = p->slot_of;
  pp.block_of = p->block_of;
  const size_t RU = (size_t)p->R * p->U;
  pp.plan_n = p->plan_n + (size_t)layer * RU;
  pp.plan = p->plan + (size_t)layer * RU * p->cap;
  pp.P = p->P;
  pp.counts = p->recall_counts + (size_t)layer * 4;
  pp.status = p->dev_status;
  pp.layer = layer;
  pp.L = p->L;
  pp.U = p->U;
  pp.max_blocks = p->max_blocks;
  pp.p_max = p->p_max;
  pp.cap = p->cap;
  const size_t smem = sizeof(int) * ((p->max_blocks + 31) / 32 + 2 * (size_t)p->cap);
  if (smem > 48 * 1024) cudaFuncSetAttribute(plan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  plan_kernel<<<(unsigned)RU, kPlanThreads, smem, s>>>(pp);
  return cudaGetLastError();
}

static GatherParams gather_params(pi_pool* p, int layer) {
  GatherParams g;
  const size_t RU = (size_t)p->R * p->U;
  g.plan_n = p->plan_n + (size_t)layer * RU;
  g.plan = p->plan + (size_t)layer * RU * p->cap;
  g.slot_of = p->slot_of;
  g.block_of = p->block_of;
  g.host_src = p->host_dev + (size_t)(layer % p->host_layers) * p->R * p->region_bytes;
  g.stage_src = nullptr;
  g.pool = p->pool;
  g.slot_base = p->slot_base;
  g.P = p->P;
  g.status = p->dev_status;
  g.region_bytes = (long long)p->region_bytes;
  g.e_begin = 0;
  g.e_end = 1LL << 62;
  g.layer = layer;
  g.L = p->L;
  g.U = p->U;
  g.max_blocks = p->max_blocks;
  g.p_max = p->p_max;
  g.cap = p->cap;
  g.units = (int)RU;
  g.copy_bytes = (int)p->copy_bytes;
  g.block_bytes = (int)p->block_bytes;
  g.do_copy = 1;
  g.do_commit = 1;
  return g;
}

static cudaError_t launch_gather(pi_pool* p, const GatherParams& g, cudaStream_t s) {
  const size_t smem = sizeof(long long) * ((size_t)g.units + 1);
  if (smem > 48 * 1024) cudaFuncSetAttribute(gather_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  int ctas = p->cfg.gather_ctas > 0 ? p->cfg.gather_ctas : 2 * p->num_sms;
  gather_kernel<<<ctas, kGatherThreads, smem, s>>>(g);
  return cudaGetLastError();
}

cudaError_t pi_launch_gather(pi_pool* p, int layer, const uint8_t* stage_src, bool copy, bool commit,
                             cudaStream_t s) {
  GatherParams g = gather_params(p, layer);
  g.stage_src = stage_src;
  g.do_copy = copy ? 1 : 0;
  g.do_commit = commit ? 1 : 0;
  return launch_gather(p, g, s);
}

// Read the plan of `layer` back to the host (one D2H copy, one sync).
static pi_status fetch_plan(pi_pool* p, int layer, cudaStream_t st, double* wait_ms) {
  const size_t RU = (size_t)p->R * p->U;
  p->plan_n_h.resize(RU);
  p->plan_h.resize(RU * p->cap);
  PI_CUDA_TRY(cudaMemcpyAsync(p->plan_n_h.data(), p->plan_n + (size_t)layer * RU, sizeof(int) * RU,
                              cudaMemcpyDeviceToHost, st));
  PI_CUDA_TRY(cudaMemcpyAsync(p->plan_h.data(), p->plan + (size_t)layer * RU * p->cap, sizeof(int4) * RU * p->cap,
                              cudaMemcpyDeviceToHost, st));
  auto t0 = std::chrono::steady_clock::now();
  PI_CUDA_TRY(cudaStreamSynchronize(st));
  auto t1 = std::chrono::steady_clock::now();
  if (wait_ms) *wait_ms += std::chrono::duration<double, std::milli>(t1 - t0).count();
  return PI_OK;
}

struct CopyRun {
  size_t src_off, dst_off, bytes;
};

// Host-side copy list in plan order, adjacent units merged into runs.
static void build_runs(pi_pool* p, int layer, std::vector<CopyRun>& runs, long long& frags) {
  runs.clear();
  frags = 0;
  const size_t RU = (size_t)p->R * p->U;
  const size_t hl_base = (size_t)(layer % p->host_layers) * p->R * p->region_bytes;
  for (size_t u = 0; u < RU; u++) {
    const int r = (int)(u / p->U), gu = (int)(u % p->U);
    const size_t head_off = (p->U > 1) ? (size_t)gu * p->copy_bytes : 0;
    const int n = p->plan_n_h[u];
    for (int j = 0; j < n; j++) {
      const int4 pe = p->plan_h[u * p->cap + j];
      CopyRun c;
      c.src_off = hl_base + (size_t)r * p->region_bytes + (size_t)pe.x * p->block_bytes + head_off;
      c.dst_off = (size_t)pi_global_slot(p, r, layer, pe.y) * p->block_bytes + head_off;
      c.bytes = p->copy_bytes;
      frags++;
      if (!runs.empty() && runs.back().src_off + runs.back().bytes == c.src_off &&
          runs.back().dst_off + runs.back().bytes == c.dst_off && p->U == 1) {
        runs.back().bytes += c.bytes;
      } else {
        runs.push_back(c);
      }
    }
  }
}

static pi_status fill_counts(pi_pool* p, int layer, cudaStream_t st, pi_recall_stats* stats) {
  long long c[2] = {0, 0};
  PI_CUDA_TRY(cudaMemcpyAsync(c, p->recall_counts + (size_t)layer * 4, sizeof(c), cudaMemcpyDeviceToHost, st));
  PI_CUDA_TRY(cudaStreamSynchronize(st));
  stats->hits += c[1];
  return PI_OK;
}

pi_status pi_recall_impl(pi_pool* p, int layer, const int* sel, const int* nsel, int method, int* table,
                         pi_recall_stats* stats, cudaStream_t st) {
  if (!p || layer < 0 || layer >= p->L || !sel || !nsel || !table) return PI_ERR_INVALID;
  if (method != PI_RECALL_UVA && method != PI_RECALL_MEMCPY && method != PI_RECALL_STAGED) return PI_ERR_INVALID;
  p->recall_calls++;
  if (p->fault_recall_at > 0 && p->recall_calls == p->fault_recall_at) return PI_ERR_FAULT_INJECTED;
  pi_recall_stats local{};
  if (stats) PI_CUDA_TRY(cudaMemsetAsync(p->recall_counts + (size_t)layer * 4, 0, sizeof(long long) * 4, st));
  PI_CUDA_TRY(pi_launch_plan(p, layer, sel, nsel, table, st));
  if (method == PI_RECALL_UVA) {
    PI_CUDA_TRY(pi_launch_gather(p, layer, nullptr, true, true, st));
    if (stats) {
      pi_status s = fetch_plan(p, layer, st, nullptr);
      if (s != PI_OK) return s;
      std::vector<CopyRun> runs;
      long long frags;
      build_runs(p, layer, runs, frags);
      local.fragments = frags;
      local.runs = (long long)runs.size();
      local.bytes = frags * (long long)p->copy_bytes;
      local.api_calls = 0;
    }
  } else {
    pi_status s = fetch_plan(p, layer, st, &local.host_wait_ms);
    if (s != PI_OK) return s;
    std::vector<CopyRun> runs;
    long long frags;
    build_runs(p, layer, runs, frags);
    local.fragments = frags;
    local.runs = (long long)runs.size();
    local.bytes = frags * (long long)p->copy_bytes;
    if (method == PI_RECALL_MEMCPY) {
      for (const CopyRun& c : runs) {
        PI_CUDA_TRY(cudaMemcpyAsync(p->pool + c.dst_off, p->host + c.src_off, c.bytes, cudaMemcpyHostToDevice, st));
        local.api_calls++;
      }
    } else {
      // staged: CPU gather into pinned staging -> one bulk copy -> GPU scatter
      if (!p->stage_host) {
        long long units = p->cfg.staging_blocks > 0 ? p->cfg.staging_blocks
                                                    : (long long)((256ull << 20) / p->copy_bytes);
        if (units < 1) units = 1;
        if (cudaHostAlloc(reinterpret_cast<void**>(&p->stage_host), (size_t)units * p->copy_bytes,
                          cudaHostAllocDefault) != cudaSuccess) {
          cudaGetLastError();
          p->stage_host = nullptr;
          return PI_ERR_HOST_ALLOC;
        }
        if (cudaMalloc(reinterpret_cast<void**>(&p->stage_dev), (size_t)units * p->copy_bytes) != cudaSuccess) {
          cudaGetLastError();
          cudaFreeHost(p->stage_host);
          p->stage_host = nullptr;
          return PI_ERR_OOM;
        }
        p->stage_units = units;
      }
      // entry list in plan order
      const size_t RU = (size_t)p->R * p->U;
      const size_t hl_base = (size_t)(layer % p->host_layers) * p->R * p->region_bytes;
      std::vector<size_t> src;
      src.reserve((size_t)frags);
      for (size_t u = 0; u < RU; u++) {
        const int r = (int)(u / p->U), gu = (int)(u % p->U);
        const size_t head_off = (p->U > 1) ? (size_t)gu * p->copy_bytes : 0;
        for (int j = 0; j < p->plan_n_h[u]; j++) {
          const int4 pe = p->plan_h[u * p->cap + j];
          src.push_back(hl_base + (size_t)r * p->region_bytes + (size_t)pe.x * p->block_bytes + head_off);
        }
      }
      const long long N = (long long)src.size();
      for (long long e0 = 0; e0 < N; e0 += p->stage_units) {
        const long long e1 = std::min(N, e0 + p->stage_units);
        auto t0 = std::chrono::steady_clock::now();
        const size_t cb = p->copy_bytes;
        uint8_t* stage = p->stage_host;
        const uint8_t* host = p->host;
#pragma omp parallel for schedule(static)
        for (long long e = e0; e < e1; e++) memcpy(stage + (size_t)(e - e0) * cb, host + src[(size_t)e], cb);
        auto t1 = std::chrono::steady_clock::now();
        local.cpu_gather_ms += std::chrono::duration<double, std::milli>(t1 - t0).count();
        PI_CUDA_TRY(cudaMemcpyAsync(p->stage_dev, p->stage_host, (size_t)(e1 - e0) * cb, cudaMemcpyHostToDevice, st));
        local.api_calls++;
        GatherParams g = gather_params(p, layer);
        g.stage_src = p->stage_dev;
        g.e_begin = e0;
        g.e_end = e1;
        g.do_copy = 1;
        g.do_commit = 0;
        PI_CUDA_TRY(launch_gather(p, g, st));
        if (e1 < N) PI_CUDA_TRY(cudaStreamSynchronize(st));  // staging reused by the next batch
      }
    }
    // every copy is enqueued: commit the maps
    PI_CUDA_TRY(pi_launch_gather(p, layer, nullptr, false, true, st));
  }
  if (stats) {
    pi_status s = fill_counts(p, layer, st, &local);
    if (s != PI_OK) return s;
    stats->bytes += local.bytes;
    stats->fragments += local.fragments;
    stats->runs += local.runs;
    stats->api_calls += local.api_calls;
    stats->hits += local.hits;
    stats->host_wait_ms += local.host_wait_ms;
    stats->cpu_gather_ms += local.cpu_gather_ms;
  }
  return PI_OK;
}

extern "C" pi_status pi_recall(pi_pool* p, int layer, const int* sel, const int* nsel, int method, int* table,
                               pi_recall_stats* stats, pi_stream s) {
  if (stats) memset(stats, 0, sizeof(*stats));
  return pi_recall_impl(p, layer, sel, nsel, method, table, stats, reinterpret_cast<cudaStream_t>(s));
}
