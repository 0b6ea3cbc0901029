// Internal declarations of the GB300 sparse KV-cache offloading library.
// Host-side pool state, device-side helpers (status word, bounded waits, TMA,
// mma) and the kernel launchers shared by the translation units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include <algorithm>
#include <string>
#include <vector>

#include "../../include/pi.h"

// --------------------------------------------------------------- device status
// Sticky error bits, OR-ed by kernels; never a trap.
enum : unsigned {
  PI_DEV_BAD_INDEX = 1u,   // an index read from memory was out of range (access skipped)
  PI_DEV_TIMEOUT = 2u,     // a bounded wait ran out
  PI_DEV_POOL_FULL = 4u,   // plan found fewer free slots than missing units
  PI_DEV_LAUNCH_SIZE = 8u, // a kernel met more work than its launch was sized for (the excess skipped)
};

#define PI_CUDA_TRY(expr)                                   \
  do {                                                      \
    cudaError_t _e = (expr);                                \
    if (_e != cudaSuccess) {                                \
      pi_note_cuda_error(_e, #expr, __FILE__, __LINE__);    \
      return PI_ERR_CUDA;                                   \
    }                                                       \
  } while (0)

void pi_note_cuda_error(cudaError_t e, const char* what, const char* file, int line);

// Opt kernel `fn` in to `bytes` of dynamic shared memory (above the default 48
// KiB) on the current device. The attribute belongs to the device's context, so
// it is set once per (kernel, device) and again only for a larger size; safe to
// call from several host threads.
cudaError_t pi_smem_optin(const void* fn, int bytes);

// --------------------------------------------------------------- pool
struct pi_pool {
  pi_config cfg{};
  int L = 0, R = 0, Hq = 0, Hkv = 0, D = 0, B = 0, G = 0;
  int max_blocks = 0, cap = 0, W = 0, k_max = 0, mode = PI_SHARED, U = 1, host_layers = 0;
  float consensus_lambda = 0.5f;  // PI_CONSENSUS: weight of the group mean
  int p_max = 0;
  size_t block_bytes = 0, frag_bytes = 0, copy_bytes = 0, region_bytes = 0;
  int device = 0, num_sms = 0;

  // host store (pinned, mapped)
  uint8_t* host = nullptr;       // host address
  uint8_t* host_dev = nullptr;   // device address of the same memory
  size_t host_bytes = 0;
  bool host_mmapped = false;     // mmap + cudaHostRegister instead of cudaHostAlloc
  void* host_map = nullptr;      // the whole mapping (the store starts at an aligned offset in it)
  size_t host_map_bytes = 0;

  // device state
  uint8_t* pool = nullptr;       // all slots
  long long total_slots = 0;
  std::vector<long long> slot_base_h;  // [R][L] first global slot of (r, l)
  std::vector<int> P_h;           // [R] configured slots per (request, layer)
  std::vector<int> P_rl_h;        // [R][L] slots in use (P_r, or the room of a pinned layer)
  std::vector<int> cap_rl_h;      // [R][L] slots reserved
  std::vector<int> pinned_h;      // [L] 1 = held whole in HBM
  std::vector<int> pinnable_h;    // [L] 1 = room reserved for every block
  std::vector<int> pin_order;     // admission: layers pinned, most recent last
  long long* slot_base = nullptr; // device [R][L]
  int* P = nullptr;               // device [R][L] slots in use
  float* kmean = nullptr;         // [R][L][max_blocks][Hkv][D]
  float* tail_sum = nullptr;      // [R][L][Hkv][D]
  int* ntok = nullptr;            // [R][L]
  std::vector<int> ntok_h;        // host mirror [R][L]
  int* slot_of = nullptr;         // [R][L][U][max_blocks]
  int* block_of = nullptr;        // [R][L][U][p_max]
  int* slot_stamp = nullptr;      // [R][L][U][p_max] last selection epoch (least-recently-selected policy)
  int* epoch = nullptr;           // [R][L][U]
  int lru_p2 = 0;                 // power of two >= p_max (sort width of the policy)
  unsigned* dev_status = nullptr;

  // per-layer scratch
  float* sel_scores = nullptr;    // [L][R*U][max_blocks]
  unsigned* sel_counter = nullptr;// [L][R*U]
  int* plan_n = nullptr;          // [L][R*U]
  int4* plan = nullptr;           // [L][R*U][cap]  (unit block, slot, evicted block, 0)
  long long* recall_counts = nullptr; // [L][4]: misses, hits (device-accumulated per call)
  int attn_max_splits = 0;
  float* attn_o = nullptr;        // [L][R*Hkv][max_splits][G][D]
  float2* attn_ml = nullptr;      // [L][R*Hkv][max_splits][G]  (m log2-domain, l)
  unsigned* attn_counter = nullptr; // [L][R*Hkv]

  // decode-step buffers
  int* step_sel = nullptr;        // [L][R][U][cap]
  int* step_nsel = nullptr;       // [L][R][U]
  int* step_table = nullptr;      // [L][R][U][cap]
  uint8_t* step_in = nullptr;     // host-variant staging of q/k/v/budget on device
  uint8_t* step_out = nullptr;    // host-variant device out/lse
  size_t step_in_bytes = 0, step_out_bytes = 0;
  std::vector<cudaEvent_t> ev_sel, ev_rec;
  cudaEvent_t ev_start = nullptr;
  int* ntok_stage = nullptr;      // [L][R] token counts staged by pi_update_summaries

  // staged arm
  uint8_t* stage_host = nullptr;  // pinned
  uint8_t* stage_dev = nullptr;
  long long stage_units = 0;
  std::vector<int4> plan_h;       // host copy of a plan
  std::vector<int> plan_n_h;

  // attention tensor map over the whole device pool (rows of D bf16)
  CUtensorMap tmap{};
  bool tmap_ok = false;

  // per-kernel timing inside pi_decode_step: events [step][layer][kind][2]
  std::vector<cudaEvent_t> tev;
  int timing_steps = 0, timing_used = 0;
  int timing_groups = 1;  // event slots per layer (request groups of the dependent schedule)

  // decode-step pipeline: layers selected ahead of attention (0 = all)
  int select_ahead = 1;
  // attention on a library-owned third stream (selection then runs freely ahead
  // and consecutive steps overlap); ev_att[l] = attention of layer l done
  bool attn_stream_on = true;
  cudaStream_t attn_stream = nullptr;
  std::vector<cudaEvent_t> ev_att;
  // interruptible layer-wise scheduling: with dependent queries a request
  // group's selection of layer l+1 follows its attention of layer l; groups
  // interleave on the copy stream (group 0 on the caller's compute stream)
  bool copy2_on = true;           // UVA gathers of odd layers on a second, pool-owned copy stream
  cudaStream_t copy2 = nullptr;
  int sched_dependent = 0;
  int sched_groups = 1;
  cudaStream_t grp_stream[8] = {};
  std::vector<cudaEvent_t> grp_ev;  // [L][8][2]: selected, recalled
  cudaEvent_t grp_done[8] = {};
  // gather on a few SMs of its own (1024-thread CTAs holding enough shared memory
  // to keep attention CTAs away)
  bool gather_exclusive = true;
  bool attn_cluster = true;       // splits 2..8 of a unit merge through DSMEM in a cluster
  bool select_cluster_on = true;  // selection as one thread-block cluster per unit (else the last-CTA form)
  int select_cluster_ctas = 0;    // CTAs per unit of the cluster form (0 = about two CTAs per SM)
  int attn_splits = 0;            // attention split count override (0 = one wave at full occupancy)

  // fused selection + gather (UVA arm of the decode step): one launch per layer (or
  // request group) on a few SMs; its CTAs claim selection items from a counter that
  // only grows, one per (layer, first unit of the launch) so that request groups'
  // launches of one layer may overlap (fused_base = its value when the next launch
  // starts), and a unit's plan is published to the launch's other CTAs by
  // fused_ready = epoch
  bool fused_on = false;
  int fused_ctas = 0;                    // 0 = a quarter of the SMs
  unsigned long long* fused_claim = nullptr;  // [L][R*U]
  unsigned* fused_ready = nullptr;       // [L][R*U]
  std::vector<unsigned long long> fused_base;  // [L][R*U]
  std::vector<unsigned> fused_epoch;     // [L]

  // attention-mass diagnostic: per-chunk partials [L][R][Hq][kMassChunksMax], allocated on first use
  float4* mass_part = nullptr;

  // fault injection
  long long fault_recall_at = 0;
  long long recall_calls = 0;
};

// --------------------------------------------------------------- helpers
static inline long long pi_global_slot(const pi_pool* p, int r, int l, int s) {
  return p->slot_base_h[(size_t)r * p->L + l] + s;
}

// kernel launchers (return cudaGetLastError of the launch)
cudaError_t pi_launch_summaries(pi_pool* p, int layer, const uint8_t* src, bool src_is_host, int b0, int b1,
                                cudaStream_t s, const int* ntok_new);
// r0, nr: the launch covers requests r0 .. r0+nr-1 (nr < 0: every request)
cudaError_t pi_launch_append(pi_pool* p, int layer, const void* k_new, const void* v_new, cudaStream_t s,
                             bool write_host = true, int r0 = 0, int nr = -1);
// fused_table != nullptr: the last CTA of each unit also writes the recall plan and the table
// mode: PI_SHARED / PI_CONSENSUS ranking on pools of one block set per request
// (U = 1), PI_HEADWISE on head-wise pools; -1 = the pool's own mode
// k_new / v_new (optional, decode step with the UVA recall): this layer's new
// tokens, appended by the selection launch itself where it can (else by the
// append kernel first, with the host write-through left to the gather)
// pdl: launch with programmatic dependent launch (the stand-alone calls; the
// decode step, whose launches are separated by stream events, does not)
cudaError_t pi_launch_select(pi_pool* p, int layer, const void* q, const int* k_per_req, int* sel, int* nsel,
                             cudaStream_t s, int* fused_table = nullptr, int mode = -1, int r0 = 0, int nr = -1,
                             const void* k_new = nullptr, const void* v_new = nullptr, bool pdl = true);
cudaError_t pi_launch_plan(pi_pool* p, int layer, const int* sel, const int* nsel, int* table, cudaStream_t s);
// selection + plan + UVA gather of requests r0 .. r0+nr-1 in one launch (decode step)
cudaError_t pi_launch_select_gather(pi_pool* p, int layer, const void* q, const int* k_per_req, int* sel, int* nsel,
                                    int* table, const void* k_new, const void* v_new, cudaStream_t s, int r0 = 0,
                                    int nr = -1);
cudaError_t pi_launch_gather(pi_pool* p, int layer, const uint8_t* stage_src, bool copy, bool commit,
                             cudaStream_t s, const void* k_new = nullptr, const void* v_new = nullptr, int r0 = 0,
                             int nr = -1, bool paired = false);
cudaError_t pi_launch_attention(pi_pool* p, int layer, const void* q, const int* sel, const int* table,
                                const int* nsel, void* out, float* lse, float* logits, cudaStream_t s, int r0 = 0,
                                int nr = -1, bool pdl = true);
bool pi_make_tmap(pi_pool* p);
// load the selection / attention kernels and set their shared-memory opt-in once
cudaError_t pi_prepare_select_kernels();
cudaError_t pi_prepare_attention_kernels();
int pi_attention_smem(int D, int B);  // dynamic shared memory of one attention CTA

// --------------------------------------------------------------- device helpers
#ifdef __CUDACC__
__device__ __forceinline__ void pi_flag(unsigned* status, unsigned bit) { atomicOr(status, bit); }

__device__ __forceinline__ float pi_bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float pi_bf16_hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }

__device__ __forceinline__ uint32_t pi_smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void pi_mbar_init(uint64_t* bar, unsigned count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(pi_smem_addr(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void pi_mbar_arrive(uint64_t* bar) {
  asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(pi_smem_addr(bar))
               : "memory");
}

__device__ __forceinline__ void pi_mbar_arrive_expect_tx(uint64_t* bar, unsigned bytes) {
  asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(
                   pi_smem_addr(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool pi_mbar_try_wait(uint64_t* bar, unsigned parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(pi_smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait for the phase of `parity` to complete; gives up after ~`limit` cycles
// (about a second), flags PI_DEV_TIMEOUT and returns false.
__device__ __forceinline__ bool pi_mbar_wait_bounded(uint64_t* bar, unsigned parity, unsigned* status,
                                                     long long limit = 2000000000LL) {
  if (pi_mbar_try_wait(bar, parity)) return true;
  long long t0 = clock64();
  while (!pi_mbar_try_wait(bar, parity)) {
    if (clock64() - t0 > limit) {
      pi_flag(status, PI_DEV_TIMEOUT);
      return false;
    }
  }
  return true;
}

__device__ __forceinline__ void pi_fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void pi_mbar_inval(uint64_t* bar) {
  asm volatile("mbarrier.inval.shared::cta.b64 [%0];" ::"r"(pi_smem_addr(bar)) : "memory");
}

// Flags one CTA publishes to the other CTAs of the same launch.
__device__ __forceinline__ void pi_st_release(unsigned* addr, unsigned v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(addr), "r"(v) : "memory");
}

__device__ __forceinline__ unsigned pi_ld_acquire(const unsigned* addr) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(addr) : "memory");
  return v;
}

// Wait until *flag == want; gives up after `limit` cycles (about a second at the
// default), records PI_DEV_TIMEOUT and returns false.
__device__ __forceinline__ bool pi_wait_flag_bounded(const unsigned* flag, unsigned want, unsigned* status,
                                                     long long limit = 2000000000LL) {
  if (pi_ld_acquire(flag) == want) return true;
  const long long t0 = clock64();
  while (pi_ld_acquire(flag) != want) {
    if (clock64() - t0 > limit) {
      pi_flag(status, PI_DEV_TIMEOUT);
      return false;
    }
    __nanosleep(200);
  }
  return true;
}

// 2D tiled TMA load global -> shared, completion on an mbarrier.
__device__ __forceinline__ void pi_tma_load_2d(void* smem_dst, const CUtensorMap* map, int x, int y, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::
          "r"(pi_smem_addr(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(pi_smem_addr(bar))
      : "memory");
}

// Fetch a tensor map (kernel parameter) into the descriptor cache ahead of its first use.
__device__ __forceinline__ void pi_tmap_prefetch(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// 1D bulk copy global -> this CTA's shared memory (both addresses 16-byte
// aligned, size a multiple of 16), completing on an mbarrier's transaction count.
__device__ __forceinline__ void pi_bulk_load(void* smem_dst, const void* src, unsigned bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          pi_smem_addr(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(pi_smem_addr(bar))
      : "memory");
}

// Thread-block clusters: the same shared-memory offset in CTA `rank` of this
// cluster, loads through that window, and a full cluster barrier (every thread
// of every CTA arrives; release/acquire order shared-memory writes before peers'
// reads).
__device__ __forceinline__ uint32_t pi_cluster_map(uint32_t smem_addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_addr), "r"(rank));
  return r;
}
__device__ __forceinline__ float2 pi_ld_cluster_f2(uint32_t addr) {
  float2 v;
  asm volatile("ld.shared::cluster.v2.f32 {%0, %1}, [%2];" : "=f"(v.x), "=f"(v.y) : "r"(addr) : "memory");
  return v;
}
__device__ __forceinline__ float4 pi_ld_cluster_f4(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(addr)
               : "memory");
  return v;
}
__device__ __forceinline__ void pi_st_cluster_f32(uint32_t addr, float v) {
  asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}
__device__ __forceinline__ void pi_st_cluster_f2(uint32_t addr, float2 v) {
  asm volatile("st.shared::cluster.v2.f32 [%0], {%1, %2};" ::"r"(addr), "f"(v.x), "f"(v.y) : "memory");
}
// Programmatic dependent launch: wait until the grids this one depends on have
// completed and their writes are visible (a no-op for a launch without the
// attribute), and let the next grid on the stream start its own launch.
__device__ __forceinline__ void pi_grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pi_grid_dep_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
// 4-byte asynchronous global -> shared copies (both 4-byte aligned), waited for as a group
__device__ __forceinline__ void pi_cp_async4(void* smem_dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(pi_smem_addr(smem_dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void pi_cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void pi_cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }
__device__ __forceinline__ void pi_cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ void pi_ldmatrix_x4(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

__device__ __forceinline__ void pi_ldmatrix_x4_trans(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

__device__ __forceinline__ uint32_t pi_movmatrix_trans(uint32_t x) {
  uint32_t y;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}

// D(16x8 fp32) += A(16x16 bf16, row) * B(16x8 bf16, col)
__device__ __forceinline__ void pi_mma_bf16(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t pi_pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ float pi_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
#endif
