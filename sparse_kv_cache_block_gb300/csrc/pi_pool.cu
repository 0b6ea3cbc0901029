#include <algorithm>
// Pool lifetime, views, residency control, device status and fault injection.
//
// The pool follows the architecture of "PulseInfer Guide: I/O-Centric Sparse
// KV Cache Offloading", section "PulseInfer Architectural Foundations": a
// global offloaded KV store in host DRAM (here pinned and mapped into the GPU's
// address space so kernels can read it directly), and a paged KV block pool in
// HBM that recalled blocks are written into.
#include <cudaTypedefs.h>
#include <sys/mman.h>

#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <map>
#include <mutex>
#include <utility>
#include <vector>

#include "pi_internal.cuh"

static thread_local char g_last_cuda_error[256];

void pi_note_cuda_error(cudaError_t e, const char* what, const char* file, int line) {
  snprintf(g_last_cuda_error, sizeof(g_last_cuda_error), "%s: %s (%s:%d)", cudaGetErrorString(e), what, file, line);
  if (getenv("PI_VERBOSE")) fprintf(stderr, "[pi] %s\n", g_last_cuda_error);
}

cudaError_t pi_smem_optin(const void* fn, int bytes) {
  if (bytes <= 48 * 1024) return cudaSuccess;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  static std::mutex mu;
  static std::map<std::pair<const void*, int>, int> done;  // (kernel, device) -> bytes set
  std::lock_guard<std::mutex> lock(mu);
  int& have = done[std::make_pair(fn, dev)];
  if (have >= bytes) return cudaSuccess;
  e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess) have = bytes;
  return e;
}

extern "C" int pi_abi_version(void) { return PI_ABI_VERSION; }

extern "C" const char* pi_status_str(pi_status s) {
  switch (s) {
    case PI_OK: return "ok";
    case PI_ERR_INVALID: return "invalid argument";
    case PI_ERR_CUDA: return "CUDA error";
    case PI_ERR_OOM: return "device out of memory";
    case PI_ERR_HOST_ALLOC: return "pinned host allocation failed";
    case PI_ERR_POOL_FULL: return "pool has fewer free slots than missing blocks";
    case PI_ERR_TIMEOUT: return "bounded device wait timed out";
    case PI_ERR_DEVICE: return "device-side index check failed";
    case PI_ERR_STATE: return "call not valid in this pool state or mode";
    case PI_ERR_FAULT_INJECTED: return "injected fault";
  }
  return "unknown status";
}

static void pool_free(pi_pool* p) {
  if (!p) return;
  for (auto e : p->ev_sel) cudaEventDestroy(e);
  for (auto e : p->ev_rec) cudaEventDestroy(e);
  if (p->ev_start) cudaEventDestroy(p->ev_start);
  for (auto e : p->ev_att) cudaEventDestroy(e);
  if (p->attn_stream) cudaStreamDestroy(p->attn_stream);
  if (p->copy2) cudaStreamDestroy(p->copy2);
  for (auto st : p->grp_stream)
    if (st) cudaStreamDestroy(st);
  for (auto e : p->grp_ev)
    if (e) cudaEventDestroy(e);
  for (auto e : p->grp_done)
    if (e) cudaEventDestroy(e);
  for (auto e : p->tev) cudaEventDestroy(e);
  void* dev_ptrs[] = {p->pool,       p->slot_base,  p->P,          p->kmean,       p->tail_sum,    p->ntok,
                      p->slot_of,    p->block_of,   p->dev_status, p->sel_scores,  p->sel_counter, p->plan_n,
                      p->plan,       p->recall_counts, p->attn_o,  p->attn_ml,     p->attn_counter, p->step_sel,
                      p->step_nsel,  p->step_table, p->step_in,    p->step_out,    p->stage_dev,
                      p->ntok_stage, p->slot_stamp, p->epoch,      p->mass_part,
                      p->fused_claim, p->fused_ready};
  for (void* d : dev_ptrs)
    if (d) cudaFree(d);
  if (p->host) {
    if (p->host_mmapped) {
      cudaHostUnregister(p->host);
      munmap(p->host_map, p->host_map_bytes);
    } else {
      cudaFreeHost(p->host);
    }
  }
  if (p->stage_host) cudaFreeHost(p->stage_host);
  delete p;
}

static pi_status parse_fault(pi_pool* p, const char* spec) {
  p->fault_recall_at = 0;
  if (!spec || !*spec) return PI_OK;
  long long n = 0;
  if (sscanf(spec, "recall_fail@%lld", &n) == 1 && n > 0) {
    p->fault_recall_at = n;
    p->recall_calls = 0;
    return PI_OK;
  }
  if (strcmp(spec, "pinned_alloc_fail") == 0) return PI_OK;  // only meaningful at creation
  return PI_ERR_INVALID;
}

static bool valid_config(const pi_config& c) {
  if (c.layers <= 0 || c.batch <= 0 || c.hq <= 0 || c.hkv <= 0) return false;
  if (c.hq % c.hkv != 0 || c.hq / c.hkv > 8) return false;
  if (c.head_dim != 64 && c.head_dim != 128) return false;
  if (c.block_tokens != 16 && c.block_tokens != 32 && c.block_tokens != 64 && c.block_tokens != 128) return false;
  if (c.max_blocks <= 0 || c.max_blocks > 65536) return false;
  if (c.k_max < 0 || c.window < 0 || c.k_max + c.window <= 0) return false;
  if ((long long)c.max_blocks * c.block_tokens > (1LL << 30)) return false;
  if (c.select_mode != PI_SHARED && c.select_mode != PI_HEADWISE && c.select_mode != PI_CONSENSUS) return false;
  if (c.host_layers < 0 || c.host_layers > c.layers) return false;
  if (c.hkv * c.head_dim > 1024) return false;  // selection keeps one block's summary per warp pass
  if (c.gather_depth != 0 && c.gather_depth != 2 && c.gather_depth != 4 && c.gather_depth != 8 &&
      c.gather_depth != 16)
    return false;
  if (c.host_alloc != 0 && c.host_alloc != 1) return false;
  if (c.evict_policy != PI_EVICT_ASCENDING && c.evict_policy != PI_EVICT_LRU) return false;
  if (c.gather_ctas < 0) return false;
  if (c.pin_layers < 0 || c.pin_layers > c.layers) return false;
  int cap = c.k_max + c.window;
  if (c.pool_slots_per_req) {
    for (int r = 0; r < c.batch; r++)
      if (c.pool_slots_per_req[r] < cap) return false;
  } else if (c.pool_slots < cap) {
    return false;
  }
  return true;
}

template <typename T>
static pi_status dalloc(T** ptr, size_t count, bool zero = true, int fill_byte = 0) {
  size_t bytes = count * sizeof(T);
  if (bytes == 0) bytes = sizeof(T);
  if (cudaMalloc(reinterpret_cast<void**>(ptr), bytes) != cudaSuccess) {
    cudaGetLastError();
    *ptr = nullptr;
    return PI_ERR_OOM;
  }
  if (zero && cudaMemset(*ptr, fill_byte, bytes) != cudaSuccess) return PI_ERR_CUDA;
  return PI_OK;
}

extern "C" pi_status pi_pool_create(const pi_config* cfg, pi_pool** out) {
  if (!cfg || !out) return PI_ERR_INVALID;
  *out = nullptr;
  if (!valid_config(*cfg)) return PI_ERR_INVALID;
  pi_pool* p = new pi_pool();
  p->cfg = *cfg;
  p->cfg.pool_slots_per_req = nullptr;  // do not keep the caller's pointer
  p->L = cfg->layers;
  p->R = cfg->batch;
  p->Hq = cfg->hq;
  p->Hkv = cfg->hkv;
  p->D = cfg->head_dim;
  p->B = cfg->block_tokens;
  p->G = p->Hq / p->Hkv;
  p->max_blocks = cfg->max_blocks;
  p->k_max = cfg->k_max;
  p->W = cfg->window;
  p->cap = p->k_max + p->W;
  p->mode = cfg->select_mode;
  p->U = (p->mode == PI_HEADWISE) ? p->Hkv : 1;
  p->host_layers = cfg->host_layers > 0 ? cfg->host_layers : p->L;
  p->frag_bytes = (size_t)2 * p->B * p->D * 2;
  p->block_bytes = p->frag_bytes * p->Hkv;
  p->copy_bytes = (p->mode == PI_HEADWISE) ? p->frag_bytes : p->block_bytes;
  p->region_bytes = p->block_bytes * (size_t)p->max_blocks;
  p->ntok_h.assign((size_t)p->R * p->L, 0);

  if (cudaGetDevice(&p->device) != cudaSuccess) { pool_free(p); return PI_ERR_CUDA; }
  cudaDeviceGetAttribute(&p->num_sms, cudaDevAttrMultiProcessorCount, p->device);
  if (p->num_sms <= 0) p->num_sms = 148;

  const char* fault = getenv("PI_FAULT");
  if (parse_fault(p, fault) != PI_OK) { pool_free(p); return PI_ERR_INVALID; }

  // slots per (request, layer): P_r, and room for every block in the pinnable
  // layers (the first ceil(n/2) and the last floor(n/2)); global slot offsets
  p->P_h.resize(p->R);
  p->slot_base_h.resize((size_t)p->R * p->L);
  p->P_rl_h.resize((size_t)p->R * p->L);
  p->cap_rl_h.resize((size_t)p->R * p->L);
  p->pinned_h.assign(p->L, 0);
  p->pinnable_h.assign(p->L, 0);
  const int pin_lo = (cfg->pin_layers + 1) / 2, pin_hi = cfg->pin_layers / 2;
  long long acc = 0;
  for (int r = 0; r < p->R; r++) {
    p->P_h[r] = cfg->pool_slots_per_req ? cfg->pool_slots_per_req[r] : cfg->pool_slots;
    for (int l = 0; l < p->L; l++) {
      const size_t rl = (size_t)r * p->L + l;
      const bool pinnable = l < pin_lo || l >= p->L - pin_hi;
      p->pinnable_h[l] = pinnable ? 1 : 0;
      p->cap_rl_h[rl] = pinnable ? std::max(p->P_h[r], p->max_blocks) : p->P_h[r];
      p->P_rl_h[rl] = p->P_h[r];
      p->slot_base_h[rl] = acc;
      acc += p->cap_rl_h[rl];
      p->p_max = std::max(p->p_max, p->cap_rl_h[rl]);
    }
  }
  p->total_slots = acc;
  p->lru_p2 = 1;
  while (p->lru_p2 < p->p_max) p->lru_p2 <<= 1;
  if (p->lru_p2 > 8192) {  // the least-recently-selected sort keeps all free slots in shared memory
    if (cfg->evict_policy == PI_EVICT_LRU) { pool_free(p); return PI_ERR_INVALID; }
  }

  // host store: pinned and mapped
  p->host_bytes = p->region_bytes * (size_t)p->host_layers * (size_t)p->R;
  if (fault && strcmp(fault, "pinned_alloc_fail") == 0) { pool_free(p); return PI_ERR_HOST_ALLOC; }
  if (cfg->host_alloc == 1) {
    // reserve extra so the store can start on a huge-page boundary (512 MiB covers
    // the largest transparent huge page of 4 KiB / 16 KiB / 64 KiB base-page kernels)
    const size_t align = (size_t)512 << 20;
    p->host_map_bytes = p->host_bytes + align;
    void* raw = mmap(nullptr, p->host_map_bytes, PROT_READ | PROT_WRITE, MAP_PRIVATE | MAP_ANONYMOUS, -1, 0);
    if (raw == MAP_FAILED) {
      pool_free(p);
      return PI_ERR_HOST_ALLOC;
    }
    p->host_map = raw;
    void* m = reinterpret_cast<void*>((reinterpret_cast<uintptr_t>(raw) + align - 1) & ~(uintptr_t)(align - 1));
    madvise(m, p->host_bytes, MADV_HUGEPAGE);  // advice only: the kernel may decline
    memset(m, 0, p->host_bytes);               // fault the pages in before pinning
    if (cudaHostRegister(m, p->host_bytes, cudaHostRegisterMapped | cudaHostRegisterPortable) != cudaSuccess) {
      cudaGetLastError();
      munmap(raw, p->host_map_bytes);
      p->host_map = nullptr;
      pool_free(p);
      return PI_ERR_HOST_ALLOC;
    }
    p->host = static_cast<uint8_t*>(m);
    p->host_mmapped = true;
  } else {
    if (cudaHostAlloc(reinterpret_cast<void**>(&p->host), p->host_bytes,
                      cudaHostAllocMapped | cudaHostAllocPortable) != cudaSuccess) {
      cudaGetLastError();
      p->host = nullptr;
      pool_free(p);
      return PI_ERR_HOST_ALLOC;
    }
    memset(p->host, 0, p->host_bytes);
  }
  if (cudaHostGetDevicePointer(reinterpret_cast<void**>(&p->host_dev), p->host, 0) != cudaSuccess) {
    pool_free(p);
    return PI_ERR_CUDA;
  }

  pi_status st = PI_OK;
  const size_t RL = (size_t)p->R * p->L, RU = (size_t)p->R * p->U;
#define TRY_ALLOC(expr)      \
  do {                       \
    st = (expr);             \
    if (st != PI_OK) {       \
      pool_free(p);          \
      return st;             \
    }                        \
  } while (0)
  TRY_ALLOC(dalloc(&p->pool, (size_t)p->total_slots * p->block_bytes));
  TRY_ALLOC(dalloc(&p->slot_base, (size_t)p->R * p->L, false));
  TRY_ALLOC(dalloc(&p->P, (size_t)p->R * p->L, false));
  TRY_ALLOC(dalloc(&p->kmean, RL * p->max_blocks * p->Hkv * p->D));
  TRY_ALLOC(dalloc(&p->tail_sum, RL * p->Hkv * p->D));
  TRY_ALLOC(dalloc(&p->ntok, RL));
  TRY_ALLOC(dalloc(&p->ntok_stage, RL));
  TRY_ALLOC(dalloc(&p->slot_of, RL * p->U * p->max_blocks, true, 0xFF));
  TRY_ALLOC(dalloc(&p->block_of, RL * p->U * p->p_max, true, 0xFF));
  TRY_ALLOC(dalloc(&p->slot_stamp, RL * p->U * p->p_max, true, 0xFF));
  TRY_ALLOC(dalloc(&p->epoch, RL * p->U));
  TRY_ALLOC(dalloc(&p->dev_status, 1));
  TRY_ALLOC(dalloc(&p->sel_scores, (size_t)p->L * RU * p->max_blocks));
  TRY_ALLOC(dalloc(&p->sel_counter, (size_t)p->L * RU));
  TRY_ALLOC(dalloc(&p->fused_claim, (size_t)p->L * RU));
  TRY_ALLOC(dalloc(&p->fused_ready, (size_t)p->L * RU));
  p->fused_base.assign((size_t)p->L * RU, 0ULL);
  p->fused_epoch.assign(p->L, 0u);
  TRY_ALLOC(dalloc(&p->plan_n, (size_t)p->L * RU));
  TRY_ALLOC(dalloc(&p->plan, (size_t)p->L * RU * p->cap));
  TRY_ALLOC(dalloc(&p->recall_counts, (size_t)p->L * 4));
  // attention split-K partials: enough splits to give every SM work at any batch
  {
    int units = p->R * p->Hkv;
    int s = (8 * p->num_sms + units - 1) / units;
    if (s < 1) s = 1;
    if (s > p->cap) s = p->cap;
    if (s < (p->cap + 511) / 512) s = (p->cap + 511) / 512;
    p->attn_max_splits = s;
  }
  TRY_ALLOC(dalloc(&p->attn_o, (size_t)p->L * p->R * p->Hkv * p->attn_max_splits * p->G * p->D, false));
  TRY_ALLOC(dalloc(&p->attn_ml, (size_t)p->L * p->R * p->Hkv * p->attn_max_splits * p->G, false));
  TRY_ALLOC(dalloc(&p->attn_counter, (size_t)p->L * p->R * p->Hkv));
  TRY_ALLOC(dalloc(&p->step_sel, (size_t)p->L * RU * p->cap));
  TRY_ALLOC(dalloc(&p->step_nsel, (size_t)p->L * RU));
  TRY_ALLOC(dalloc(&p->step_table, (size_t)p->L * RU * p->cap));
  p->step_in_bytes = (size_t)p->L * p->R * ((size_t)p->Hq * p->D * 2 + (size_t)2 * p->Hkv * p->D * 2 + 4);
  p->step_out_bytes = (size_t)p->L * p->R * ((size_t)p->Hq * p->D * 2 + (size_t)p->Hq * 4);
  TRY_ALLOC(dalloc(&p->step_in, p->step_in_bytes, false));
  TRY_ALLOC(dalloc(&p->step_out, p->step_out_bytes, false));
#undef TRY_ALLOC

  if (cudaMemcpy(p->slot_base, p->slot_base_h.data(), sizeof(long long) * p->R * p->L, cudaMemcpyHostToDevice) !=
          cudaSuccess ||
      cudaMemcpy(p->P, p->P_rl_h.data(), sizeof(int) * p->R * p->L, cudaMemcpyHostToDevice) != cudaSuccess) {
    pool_free(p);
    return PI_ERR_CUDA;
  }

  if (cudaEventCreateWithFlags(&p->ev_start, cudaEventDisableTiming) != cudaSuccess) {
    pool_free(p);
    return PI_ERR_CUDA;
  }
  p->ev_att.resize(p->L, nullptr);
  for (int l = 0; l < p->L; l++)
    if (cudaEventCreateWithFlags(&p->ev_att[l], cudaEventDisableTiming) != cudaSuccess) {
      pool_free(p);
      return PI_ERR_CUDA;
    }
  if (cudaStreamCreateWithFlags(&p->attn_stream, cudaStreamNonBlocking) != cudaSuccess ||
      cudaStreamCreateWithFlags(&p->copy2, cudaStreamNonBlocking) != cudaSuccess) {
    pool_free(p);
    return PI_ERR_CUDA;
  }
  p->ev_sel.resize(p->L);
  p->ev_rec.resize(p->L);
  for (int l = 0; l < p->L; l++) {
    if (cudaEventCreateWithFlags(&p->ev_sel[l], cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&p->ev_rec[l], cudaEventDisableTiming) != cudaSuccess) {
      pool_free(p);
      return PI_ERR_CUDA;
    }
  }
  if (!pi_make_tmap(p)) {
    pool_free(p);
    return PI_ERR_CUDA;
  }
  // every kernel of the decode path loaded and opted in to its shared memory now,
  // not in the middle of a decode
  if (pi_prepare_select_kernels() != cudaSuccess || pi_prepare_attention_kernels() != cudaSuccess) {
    cudaGetLastError();
    pool_free(p);
    return PI_ERR_CUDA;
  }
  if (cudaDeviceSynchronize() != cudaSuccess) {
    pool_free(p);
    return PI_ERR_CUDA;
  }
  *out = p;
  return PI_OK;
}

extern "C" pi_status pi_pool_destroy(pi_pool* p) {
  if (!p) return PI_ERR_INVALID;
  cudaDeviceSynchronize();
  pool_free(p);
  return PI_OK;
}

extern "C" pi_status pi_pool_get_config(const pi_pool* p, pi_config* out) {
  if (!p || !out) return PI_ERR_INVALID;
  *out = p->cfg;
  return PI_OK;
}

extern "C" pi_status pi_pool_get_views(pi_pool* p, pi_pool_views* v) {
  if (!p || !v) return PI_ERR_INVALID;
  v->pool = p->pool;
  v->slot_base = p->slot_base_h.data();
  v->slots_per_req = p->P_h.data();
  v->slots_rl = p->P_rl_h.data();
  v->capacity_rl = p->cap_rl_h.data();
  v->total_slots = p->total_slots;
  v->dev_status = p->dev_status;
  v->kmean = p->kmean;
  v->ntok = p->ntok;
  v->slot_of_block = p->slot_of;
  v->block_of_slot = p->block_of;
  v->p_max = p->p_max;
  v->step_sel = p->step_sel;
  v->step_nsel = p->step_nsel;
  v->step_table = p->step_table;
  v->block_bytes = p->block_bytes;
  v->frag_bytes = p->frag_bytes;
  v->host_region_bytes = p->region_bytes;
  v->slot_stamp = p->slot_stamp;
  return PI_OK;
}

extern "C" void* pi_host_kv(pi_pool* p, int layer, int req) {
  if (!p || layer < 0 || layer >= p->L || req < 0 || req >= p->R) return nullptr;
  int hl = layer % p->host_layers;
  return p->host + ((size_t)hl * p->R + req) * p->region_bytes;
}

extern "C" pi_status pi_set_fault(pi_pool* p, const char* spec) {
  if (!p) return PI_ERR_INVALID;
  return parse_fault(p, spec);
}

extern "C" pi_status pi_get_device_status(pi_pool* p) {
  if (!p) return PI_ERR_INVALID;
  PI_CUDA_TRY(cudaDeviceSynchronize());
  unsigned w = 0;
  PI_CUDA_TRY(cudaMemcpy(&w, p->dev_status, sizeof(unsigned), cudaMemcpyDeviceToHost));
  if (w & (PI_DEV_BAD_INDEX | PI_DEV_LAUNCH_SIZE)) return PI_ERR_DEVICE;
  if (w & PI_DEV_TIMEOUT) return PI_ERR_TIMEOUT;
  if (w & PI_DEV_POOL_FULL) return PI_ERR_POOL_FULL;
  return PI_OK;
}

extern "C" pi_status pi_clear_device_status(pi_pool* p) {
  if (!p) return PI_ERR_INVALID;
  PI_CUDA_TRY(cudaDeviceSynchronize());
  PI_CUDA_TRY(cudaMemset(p->dev_status, 0, sizeof(unsigned)));
  // a kernel that gave up on a wait may have left its completion counters behind
  PI_CUDA_TRY(cudaMemset(p->sel_counter, 0, sizeof(unsigned) * p->L * p->R * p->U));
  PI_CUDA_TRY(cudaMemset(p->attn_counter, 0, sizeof(unsigned) * p->L * p->R * p->Hkv));
  PI_CUDA_TRY(cudaMemset(p->fused_claim, 0, sizeof(unsigned long long) * p->L * p->R * p->U));
  p->fused_base.assign((size_t)p->L * p->R * p->U, 0ULL);
  return PI_OK;
}

extern "C" pi_status pi_pool_flush(pi_pool* p, int layer, pi_stream s) {
  if (!p || layer < -1 || layer >= p->L) return PI_ERR_INVALID;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(s);
  for (int r = 0; r < p->R; r++)
    for (int l = 0; l < p->L; l++) {
      if (layer >= 0 && l != layer) continue;
      size_t rl = (size_t)r * p->L + l;
      PI_CUDA_TRY(cudaMemsetAsync(p->slot_of + rl * p->U * p->max_blocks, 0xFF,
                                  sizeof(int) * p->U * p->max_blocks, st));
      PI_CUDA_TRY(cudaMemsetAsync(p->block_of + rl * p->U * p->p_max, 0xFF, sizeof(int) * p->U * p->p_max, st));
      PI_CUDA_TRY(cudaMemsetAsync(p->slot_stamp + rl * p->U * p->p_max, 0xFF, sizeof(int) * p->U * p->p_max, st));
      PI_CUDA_TRY(cudaMemsetAsync(p->epoch + rl * p->U, 0, sizeof(int) * p->U, st));
    }
  return PI_OK;
}

extern "C" pi_status pi_pool_preload(pi_pool* p, int layer, int req, const int* blocks, int n, pi_stream s) {
  if (!p || layer < 0 || layer >= p->L || req < 0 || req >= p->R || n < 0 || (n > 0 && !blocks))
    return PI_ERR_INVALID;
  if (p->U != 1) return PI_ERR_STATE;
  if (n > p->P_rl_h[(size_t)req * p->L + layer]) return PI_ERR_INVALID;
  for (int i = 0; i < n; i++) {
    if (blocks[i] < 0 || blocks[i] >= p->max_blocks) return PI_ERR_INVALID;
    if (i > 0 && blocks[i] <= blocks[i - 1]) return PI_ERR_INVALID;
  }
  cudaStream_t st = reinterpret_cast<cudaStream_t>(s);
  PI_CUDA_TRY(cudaStreamSynchronize(st));
  size_t rl = (size_t)req * p->L + layer;
  std::vector<int> sob(p->max_blocks, -1), bos(p->p_max, -1);
  for (int i = 0; i < n; i++) {
    sob[blocks[i]] = i;
    bos[i] = blocks[i];
  }
  PI_CUDA_TRY(cudaMemcpy(p->slot_of + rl * p->max_blocks, sob.data(), sizeof(int) * p->max_blocks,
                         cudaMemcpyHostToDevice));
  PI_CUDA_TRY(cudaMemcpy(p->block_of + rl * p->p_max, bos.data(), sizeof(int) * p->p_max, cudaMemcpyHostToDevice));
  std::vector<int> stamps(p->p_max, -1);
  for (int i = 0; i < n; i++) stamps[i] = 0;  // preloaded blocks count as selected at epoch 0
  PI_CUDA_TRY(cudaMemcpy(p->slot_stamp + rl * p->p_max, stamps.data(), sizeof(int) * p->p_max, cudaMemcpyHostToDevice));
  PI_CUDA_TRY(cudaMemset(p->epoch + rl, 0, sizeof(int)));
  const uint8_t* src = (const uint8_t*)pi_host_kv(p, layer, req);
  for (int i = 0; i < n; i++) {
    uint8_t* dst = p->pool + (size_t)pi_global_slot(p, req, layer, i) * p->block_bytes;
    PI_CUDA_TRY(cudaMemcpyAsync(dst, src + (size_t)blocks[i] * p->block_bytes, p->block_bytes,
                                cudaMemcpyHostToDevice, st));
  }
  PI_CUDA_TRY(cudaStreamSynchronize(st));
  return PI_OK;
}

// Tensor map over the device pool seen as rows of D bf16 (one row = one token of
// one head's K or V). Row of (global slot gs, head g, kv, token t) =
// ((gs * Hkv + g) * 2 + kv) * B + t. Boxes are 64 elements (128 bytes) wide and
// B rows high, 128-byte swizzled, so a block's K or V of one head is D/64 boxes.
bool pi_make_tmap(pi_pool* p) {
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess || !fn) {
    cudaGetLastError();
    return false;
  }
  auto encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  unsigned long long rows = (unsigned long long)p->total_slots * p->Hkv * 2 * p->B;
  if (rows >= (1ULL << 31)) return false;
  cuuint64_t dims[2] = {(cuuint64_t)p->D, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)p->D * 2};
  cuuint32_t box[2] = {64, (cuuint32_t)p->B};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = encode(&p->tmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, p->pool, dims, strides, box, estr,
                      CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                      CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  p->tmap_ok = (r == CUDA_SUCCESS);
  return p->tmap_ok;
}

// One thread waits on a phase of an mbarrier that never completes (its expected
// arrival count is 2 and nothing arrives); the bounded wait gives up and flags.
static __global__ void bounded_wait_selftest_kernel(unsigned* status, long long limit) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    pi_mbar_init(&bar, 2);
    pi_fence_barrier_init();
    pi_mbar_wait_bounded(&bar, 0, status, limit);
  }
}

extern "C" pi_status pi_selftest_bounded_wait(pi_pool* p, long long limit_cycles) {
  if (!p || limit_cycles < 1 || limit_cycles > 2000000000LL) return PI_ERR_INVALID;
  bounded_wait_selftest_kernel<<<1, 32>>>(p->dev_status, limit_cycles);
  PI_CUDA_TRY(cudaGetLastError());
  return pi_get_device_status(p);
}

extern "C" pi_status pi_pool_set_gather(pi_pool* p, int ctas, int depth, int exclusive) {
  if (!p || ctas < 0 || (depth != 2 && depth != 4 && depth != 8 && depth != 16)) return PI_ERR_INVALID;
  p->cfg.gather_ctas = ctas;
  p->cfg.gather_depth = depth;
  p->gather_exclusive = exclusive != 0;
  return PI_OK;
}

extern "C" pi_status pi_pool_set_consensus_lambda(pi_pool* p, float lambda) {
  if (!p || !(lambda >= 0.0f) || !(lambda <= 1e30f)) return PI_ERR_INVALID;
  p->consensus_lambda = lambda;
  return PI_OK;
}

// ------------------------------------------------------------------ IO-adaptive admission
// "PulseInfer Guide", section "Interruptible Layer-Wise Scheduling & Adaptive
// Admission", "2. IO-Adaptive Offloading Admission": under a saturated link the
// most active layers (the first and the last) stay whole in HBM; under a quiet
// link they are offloaded again. A pinned layer uses the room the pool reserved
// for every block of each request, so once its blocks have been recalled it
// recalls nothing; releasing it drops the blocks held beyond P_r from the maps.
static pi_status set_layer_slots(pi_pool* p, int layer, bool pinned) {
  PI_CUDA_TRY(cudaDeviceSynchronize());
  std::vector<int> sob(p->max_blocks), bos(p->p_max), stamp(p->p_max);
  for (int r = 0; r < p->R; r++) {
    const size_t rl = (size_t)r * p->L + layer;
    const int keep = p->P_h[r];
    if (!pinned && p->P_rl_h[rl] > keep) {
      for (int u = 0; u < p->U; u++) {
        const size_t rlu = rl * p->U + u;
        int* sob_d = p->slot_of + rlu * p->max_blocks;
        int* bos_d = p->block_of + rlu * p->p_max;
        int* st_d = p->slot_stamp + rlu * p->p_max;
        PI_CUDA_TRY(cudaMemcpy(sob.data(), sob_d, sizeof(int) * p->max_blocks, cudaMemcpyDeviceToHost));
        PI_CUDA_TRY(cudaMemcpy(bos.data(), bos_d, sizeof(int) * p->p_max, cudaMemcpyDeviceToHost));
        PI_CUDA_TRY(cudaMemcpy(stamp.data(), st_d, sizeof(int) * p->p_max, cudaMemcpyDeviceToHost));
        for (int s = keep; s < p->P_rl_h[rl]; s++) {
          const int b = bos[s];
          if (b >= 0 && b < p->max_blocks) sob[b] = -1;
          bos[s] = -1;
          stamp[s] = -1;
        }
        PI_CUDA_TRY(cudaMemcpy(sob_d, sob.data(), sizeof(int) * p->max_blocks, cudaMemcpyHostToDevice));
        PI_CUDA_TRY(cudaMemcpy(bos_d, bos.data(), sizeof(int) * p->p_max, cudaMemcpyHostToDevice));
        PI_CUDA_TRY(cudaMemcpy(st_d, stamp.data(), sizeof(int) * p->p_max, cudaMemcpyHostToDevice));
      }
    }
    p->P_rl_h[rl] = pinned ? p->cap_rl_h[rl] : keep;
    PI_CUDA_TRY(cudaMemcpy(p->P + rl, &p->P_rl_h[rl], sizeof(int), cudaMemcpyHostToDevice));
  }
  p->pinned_h[layer] = pinned ? 1 : 0;
  if (pinned) {
    p->pin_order.push_back(layer);
  } else {
    for (size_t i = 0; i < p->pin_order.size(); i++)
      if (p->pin_order[i] == layer) {
        p->pin_order.erase(p->pin_order.begin() + (long)i);
        break;
      }
  }
  return PI_OK;
}

extern "C" pi_status pi_pool_pin_layer(pi_pool* p, int layer, int pinned) {
  if (!p || layer < 0 || layer >= p->L || (pinned != 0 && pinned != 1)) return PI_ERR_INVALID;
  if (!p->pinnable_h[layer]) return PI_ERR_INVALID;
  if (p->pinned_h[layer] == pinned) return PI_OK;
  return set_layer_slots(p, layer, pinned != 0);
}

extern "C" pi_status pi_admission_decide(int layers, const int* pinnable, const int* pinned, int last_pinned,
                                         double link_util, int* layer, int* pin) {
  if (layers <= 0 || !pinnable || !pinned || !layer || !pin || !(link_util >= 0.0)) return PI_ERR_INVALID;
  // the layer named as pinned last must be a pinnable layer that is still pinned
  if (last_pinned >= layers || (last_pinned >= 0 && (!pinnable[last_pinned] || !pinned[last_pinned])))
    return PI_ERR_INVALID;
  *layer = -1;
  *pin = 0;
  if (link_util > 0.85) {
    // the most active layers first: 0, L-1, 1, L-2, ...
    for (int i = 0; i < layers; i++) {
      const int l = (i % 2 == 0) ? i / 2 : layers - 1 - i / 2;
      if (pinnable[l] && !pinned[l]) {
        *layer = l;
        *pin = 1;
        break;
      }
    }
  } else if (link_util < 0.5 && last_pinned >= 0) {
    *layer = last_pinned;
    *pin = 0;
  }
  return PI_OK;
}

extern "C" pi_status pi_pool_recall_totals(pi_pool* p, long long* recalled, long long* hits, int reset) {
  if (!p || !recalled || !hits || (reset != 0 && reset != 1)) return PI_ERR_INVALID;
  PI_CUDA_TRY(cudaDeviceSynchronize());
  std::vector<long long> c((size_t)4 * p->L);
  PI_CUDA_TRY(cudaMemcpy(c.data(), p->recall_counts, sizeof(long long) * c.size(), cudaMemcpyDeviceToHost));
  long long m = 0, h = 0;
  for (int l = 0; l < p->L; l++) {
    m += c[(size_t)l * 4 + 0];
    h += c[(size_t)l * 4 + 1];
  }
  if (reset) PI_CUDA_TRY(cudaMemset(p->recall_counts, 0, sizeof(long long) * c.size()));
  *recalled = m;
  *hits = h;
  return PI_OK;
}

extern "C" pi_status pi_pool_admission(pi_pool* p, double link_util, int* layer, int* pinned) {
  if (!p || !layer || !pinned || !(link_util >= 0.0)) return PI_ERR_INVALID;
  int l = -1, pin = 0;
  pi_status st = pi_admission_decide(p->L, p->pinnable_h.data(), p->pinned_h.data(),
                                     p->pin_order.empty() ? -1 : p->pin_order.back(), link_util, &l, &pin);
  if (st != PI_OK) return st;
  if (l >= 0) {
    st = set_layer_slots(p, l, pin == 1);
    if (st != PI_OK) return st;
  }
  *layer = l;
  *pinned = pin;
  return PI_OK;
}

extern "C" pi_status pi_pool_set_evict(pi_pool* p, int policy) {
  if (!p || (policy != PI_EVICT_ASCENDING && policy != PI_EVICT_LRU)) return PI_ERR_INVALID;
  if (policy == PI_EVICT_LRU && p->lru_p2 > 8192) return PI_ERR_INVALID;
  p->cfg.evict_policy = policy;
  return PI_OK;
}
