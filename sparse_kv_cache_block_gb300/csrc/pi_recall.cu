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

#include "pi_gather.cuh"
#include "pi_internal.cuh"
#include "pi_plan.cuh"

namespace {

constexpr int kPlanThreads = 256;


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
  int* slot_stamp;    // nullptr unless the least-recently-selected policy is on
  int* epoch;
  int layer, L, U, max_blocks, p_max, cap, lru_p2;
  int empty_first;    // the layer is held whole in HBM
};

// One CTA per unit (request, or request x KV head). Writes the table and the
// plan; the maps are committed later by the copy kernel.
__global__ void __launch_bounds__(kPlanThreads) plan_kernel(PlanParams p) {
  extern __shared__ __align__(16) unsigned char smraw[];
  __shared__ int warp_sums[kPlanThreads / 32];
  const int words = (p.max_blocks + 31) / 32;
  unsigned long long* keys = reinterpret_cast<unsigned long long*>(smraw);
  int* sm = reinterpret_cast<int*>(smraw + sizeof(unsigned long long) * (p.slot_stamp ? p.lru_p2 : 0));
  const int u = blockIdx.x;
  const int r = u / p.U, gu = u % p.U;
  const size_t rlu = ((size_t)r * p.L + p.layer) * p.U + gu;
  int n = p.nsel[u];
  if (n < 0 || n > p.cap) {
    if (threadIdx.x == 0) pi_flag(p.status, PI_DEV_BAD_INDEX);
    n = 0;
  }
  pi_plan::UnitArgs a;
  a.sel = p.sel + (size_t)u * p.cap;
  a.n = n;
  a.sob = p.slot_of + rlu * p.max_blocks;
  a.bos = p.block_of + rlu * p.p_max;
  a.P = p.P[(size_t)r * p.L + p.layer];
  a.max_blocks = p.max_blocks;
  a.table = p.table + (size_t)u * p.cap;
  a.plan = p.plan + (size_t)u * p.cap;
  a.plan_n = p.plan_n + u;
  a.counts = p.counts;
  a.status = p.status;
  a.stamp = p.slot_stamp ? p.slot_stamp + rlu * p.p_max : nullptr;
  a.epoch = p.slot_stamp ? p.epoch + rlu : nullptr;
  a.empty_first = p.empty_first;
  pi_plan::plan_unit<kPlanThreads>(a, reinterpret_cast<unsigned*>(sm), sm + words, sm + words + p.cap, warp_sums,
                                   keys, p.lru_p2);
}

// Grid-stride over (plan entry, chunk of 256 x 16 x DEPTH bytes). Each thread
// keeps DEPTH 16-byte loads in flight (DEPTH = 8: 32 KiB outstanding per CTA).
// With k_new set (decode-step pipeline), CTA 0 also writes this step's token of
// every request through to the host store, and a CTA that copies a chunk of the
// block holding that token overwrites the token's rows from k_new/v_new, so the
// pool never depends on when the host write lands.
template <int kGatherDepth, int kGatherThreads>
__global__ void __launch_bounds__(kGatherThreads) gather_kernel(GatherParams g) {
  constexpr int kChunkBytes = kGatherThreads * 16 * kGatherDepth;
  extern __shared__ long long prefix[];  // [units + 1]
  __shared__ int warp_sums[kGatherThreads / 32];
  if (g.k_new && blockIdx.x == 0) pi_gather_write_through<kGatherThreads>(g);
  // prefix sums of the per-unit plan counts (every CTA computes its own copy)
  long long run = 0;
  for (int base = 0; base < g.units; base += kGatherThreads) {
    const int u = base + threadIdx.x;
    const int v = (u < g.units) ? g.plan_n[u] : 0;
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
    int lo = 0, hi = g.units - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (prefix[mid] <= e) lo = mid; else hi = mid - 1;
    }
    pi_gather_item<kGatherDepth, kGatherThreads>(g, lo, (int)(e - prefix[lo]), c, chunk, e - e0);
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
  const bool lru = p->cfg.evict_policy == PI_EVICT_LRU;
  pp.slot_stamp = lru ? p->slot_stamp : nullptr;
  pp.epoch = lru ? p->epoch : nullptr;
  pp.lru_p2 = lru ? p->lru_p2 : 0;
  pp.empty_first = p->pinned_h.empty() ? 0 : p->pinned_h[layer];
  const size_t smem = pi_plan::plan_smem_bytes(p->max_blocks, p->cap, pp.lru_p2);
  cudaError_t e0 = pi_smem_optin(reinterpret_cast<const void*>(plan_kernel), (int)smem);
  if (e0 != cudaSuccess) return e0;
  plan_kernel<<<(unsigned)RU, kPlanThreads, smem, s>>>(pp);
  return cudaGetLastError();
}

GatherParams pi_gather_params(pi_pool* p, int layer) {
  GatherParams g;
  const size_t RU = (size_t)p->R * p->U;
  g.plan_n = p->plan_n + (size_t)layer * RU;
  g.plan = p->plan + (size_t)layer * RU * p->cap;
  g.slot_of = p->slot_of;
  g.block_of = p->block_of;
  g.slot_stamp = (p->cfg.evict_policy == PI_EVICT_LRU) ? p->slot_stamp : nullptr;
  g.host_src = p->host_dev + (size_t)(layer % p->host_layers) * p->R * p->region_bytes;
  g.host_dst = p->host_dev + (size_t)(layer % p->host_layers) * p->R * p->region_bytes;
  g.stage_src = nullptr;
  g.ntok = p->ntok;
  g.k_new = nullptr;
  g.v_new = nullptr;
  g.pool = p->pool;
  g.slot_base = p->slot_base;
  g.P = p->P;
  g.status = p->dev_status;
  g.region_bytes = (long long)p->region_bytes;
  g.e_begin = 0;
  g.e_end = 1LL << 62;
  g.layer = layer;
  g.L = p->L;
  g.R = p->R;
  g.U = p->U;
  g.Hkv = p->Hkv;
  g.B = p->B;
  g.D = p->D;
  g.max_blocks = p->max_blocks;
  g.p_max = p->p_max;
  g.cap = p->cap;
  g.units = (int)RU;
  g.r0 = 0;
  g.nr = p->R;
  g.copy_bytes = (int)p->copy_bytes;
  g.block_bytes = (int)p->block_bytes;
  g.do_copy = 1;
  g.do_commit = 1;
  return g;
}

template <int DEPTH, int THREADS>
static cudaError_t launch_gather_t(int ctas, size_t smem, const GatherParams& g, cudaStream_t s) {
  cudaError_t e = pi_smem_optin(reinterpret_cast<const void*>(gather_kernel<DEPTH, THREADS>), (int)smem);
  if (e != cudaSuccess) return e;
  gather_kernel<DEPTH, THREADS><<<ctas, THREADS, smem, s>>>(g);
  return cudaGetLastError();
}

template <int THREADS>
static cudaError_t launch_gather_d(int depth, int ctas, size_t smem, const GatherParams& g, cudaStream_t s) {
  switch (depth) {
    case 2: return launch_gather_t<2, THREADS>(ctas, smem, g, s);
    case 4: return launch_gather_t<4, THREADS>(ctas, smem, g, s);
    case 16:
      // 1024-thread CTAs have 64 registers per thread: sixteen loads in flight would spill
      if constexpr (THREADS <= 256) return launch_gather_t<16, THREADS>(ctas, smem, g, s);
      return launch_gather_t<8, THREADS>(ctas, smem, g, s);
    default: return launch_gather_t<8, THREADS>(ctas, smem, g, s);
  }
}

// Exclusive (default): 1024-thread CTAs on a quarter of the SMs that reserve
// enough shared memory that no attention CTA fits beside them, so the
// long-latency host-link reads stay on a few SMs and the other SMs' memory
// requests never queue behind them (measured: attention in the decode step drops
// from ~110 us to ~40-55 us per layer; the step runs 12 % faster).
// Shared: 256-thread CTAs, one per SM, beside whatever else runs. Copy units
// under 32 KiB (one KV head's fragment of small blocks in the head-wise arm)
// always take the shared shape: a 1024-thread CTA would leave most threads idle
// on each unit (measured: 8 KiB fragments move 120 GB/s exclusive, 184 shared).
// paired: another gather may run at the same time on a second copy stream; the
// default grid is then half as wide, so both together hold a quarter of the SMs
// (measured: 3 % more tokens/s than a quarter each).
static cudaError_t launch_gather(pi_pool* p, const GatherParams& g, cudaStream_t s, bool paired) {
  size_t smem = sizeof(long long) * ((size_t)g.units + 1);
  if (p->gather_exclusive && g.copy_bytes >= 32768) {
    const int ctas = p->cfg.gather_ctas > 0 ? p->cfg.gather_ctas : max(1, p->num_sms / (paired ? 8 : 4));
    const size_t attn = (size_t)pi_attention_smem(p->D, p->B);
    const size_t sm_bytes = 228 * 1024, reserve = 1024;
    size_t pad = (sm_bytes > attn + 2 * reserve) ? sm_bytes - attn - 2 * reserve + 1024 : 0;
    if (pad > 220 * 1024) pad = 220 * 1024;
    if (smem < pad) smem = pad;
    return launch_gather_d<1024>(p->cfg.gather_depth, ctas, smem, g, s);
  }
  const int ctas = p->cfg.gather_ctas > 0 ? p->cfg.gather_ctas : p->num_sms;
  return launch_gather_d<256>(p->cfg.gather_depth, ctas, smem, g, s);
}

cudaError_t pi_launch_gather(pi_pool* p, int layer, const uint8_t* stage_src, bool copy, bool commit,
                             cudaStream_t s, const void* k_new, const void* v_new, int r0, int nr, bool paired) {
  GatherParams g = pi_gather_params(p, layer);
  if (nr >= 0) {
    // requests r0 .. r0+nr-1 only: their units' plans (the staged arm always takes every request)
    g.plan_n += (size_t)r0 * p->U;
    g.plan += (size_t)r0 * p->U * p->cap;
    g.r0 = r0;
    g.nr = nr;
    g.units = nr * p->U;
  }
  g.stage_src = stage_src;
  g.k_new = (const uint8_t*)k_new;
  g.v_new = (const uint8_t*)v_new;
  g.do_copy = copy ? 1 : 0;
  g.do_commit = commit ? 1 : 0;
  return launch_gather(p, g, s, paired);
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
        GatherParams g = pi_gather_params(p, layer);
        g.stage_src = p->stage_dev;
        g.e_begin = e0;
        g.e_end = e1;
        g.do_copy = 1;
        g.do_commit = 0;
        PI_CUDA_TRY(launch_gather(p, g, st, false));
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
