/*
 * pi.h -- C ABI of the GB300 sparse KV-cache offloading decode path.
 *
 * One GPU, one process. The library owns a pool: a pinned, GPU-mapped host KV
 * store (most blocks live here), a device block pool of recalled blocks, the
 * per-block key summaries, the slot maps and all scratch. Callers own the
 * per-call device buffers (queries, selections, tables, outputs), typically
 * PyTorch tensors, and pass raw device pointers and CUDA streams.
 *
 * Method (page title, section):
 *  - "PulseInfer: I/O-Centric Sparse KV Cache Offloading for Efficient
 *    Long-Context LLM Decoding", Abstract: KV blocks stay in CPU DRAM, selected
 *    blocks are recalled on demand; one block set shared by the heads (SoloHead)
 *    and a gathering recall path replace many small per-head copies by one;
 *    recall is overlapped with decode layer by layer.
 *  - "PulseInfer Guide: I/O-Centric Sparse KV Cache Offloading":
 *    "SoloHead Sparse Selection" (one block set shared by all heads of a layer),
 *    "The Gather-Scatter I/O Engine" (blocks land in pool page slots),
 *    "The Small-Packet PCIe DMA Tax" (paged blocks of B tokens),
 *    "Interruptible Layer-Wise Scheduling" (recall of one layer hides behind
 *    compute of another).
 * The pages name SoloHead but never define its block score. This library fixes
 * one definition (see pi_select_topk).
 *
 * Notation: L layers, R requests (batch), Hq query heads, Hkv KV heads,
 * G = Hq/Hkv, D head_dim, B tokens per block, P pool slots per (request, layer),
 * cap = k_max + window, bf16 = IEEE bfloat16 bit patterns (uint16).
 *
 * Layouts (row-major, innermost last):
 *  host store, per (layer, request):  [max_blocks][Hkv][2 (K,V)][B][D] bf16
 *    -> a block is BB = 2*Hkv*B*D*2 contiguous bytes, one head's K+V of a block
 *       (a "fragment") FB = 2*B*D*2 contiguous bytes.
 *  device pool: one slot = one block in the same [Hkv][2][B][D] layout.
 *  q: [R][Hq][D] bf16; out: [R][Hq][D] bf16; lse: [R][Hq] fp32 (natural log).
 *  sel / table: [R][cap] int32 (shared mode) or [R][Hkv][cap] (head-wise mode);
 *  nsel: [R] or [R][Hkv] int32.
 *
 * Errors: every call checks its arguments on the host and returns a status; no
 * call aborts. Kernels never trap: a bad index or a wait that runs out sets a
 * sticky device status word, read by pi_get_device_status. Calls are
 * asynchronous on the given stream unless stated. Calls of the same kind on the
 * same layer must be stream-ordered; different layers may run concurrently.
 */
#ifndef PI_H
#define PI_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define PI_ABI_VERSION 1

/* cudaStream_t without pulling in CUDA headers; NULL = legacy default stream. */
typedef struct CUstream_st* pi_stream;

typedef enum {
  PI_OK = 0,
  PI_ERR_INVALID = 1,        /* bad argument or size; nothing was enqueued */
  PI_ERR_CUDA = 2,           /* a CUDA runtime call failed */
  PI_ERR_OOM = 3,            /* device allocation failed */
  PI_ERR_HOST_ALLOC = 4,     /* pinned host allocation failed */
  PI_ERR_POOL_FULL = 5,      /* more missing blocks than free slots */
  PI_ERR_TIMEOUT = 6,        /* a bounded device wait ran out */
  PI_ERR_DEVICE = 7,         /* a kernel flagged an out-of-range index */
  PI_ERR_STATE = 8,          /* call not valid in the pool's state/mode */
  PI_ERR_FAULT_INJECTED = 9  /* host-side fault injection fired */
} pi_status;

enum { PI_SHARED = 0, PI_HEADWISE = 1, PI_CONSENSUS = 2 };
enum { PI_RECALL_UVA = 0, PI_RECALL_MEMCPY = 1, PI_RECALL_STAGED = 2 };
enum { PI_EVICT_ASCENDING = 0, PI_EVICT_LRU = 1 };

typedef struct pi_config {
  int layers, batch, hq, hkv, head_dim, block_tokens;
  int max_blocks;            /* host/summary capacity per (layer, request), blocks */
  int pool_slots;            /* P per (request, layer); must be >= k_max + window */
  int k_max;                 /* largest top-k a call may ask for */
  int window;                /* W most recent blocks always selected */
  int select_mode;           /* PI_SHARED (one block set per request and layer),
                                PI_CONSENSUS (the same, ranked by the consensus
                                score) or PI_HEADWISE (one per KV head: the
                                comparison arm) */
  int host_layers;           /* 0 = layers. Else the host store holds host_layers
                                layers and layer l reads host layer l % host_layers
                                (capacity fallback; appends must then carry the same
                                tokens for aliased layers). */
  int staging_blocks;        /* staged recall arm: staging capacity in copy units
                                (0 = as many as fit in 256 MiB) */
  int gather_ctas;           /* UVA gather kernel grid (0 = default; see pi_pool_set_gather) */
  int gather_depth;          /* 16-byte loads in flight per gather thread: 2, 4, 8 or 16
                                (0 = 8) */
  int evict_policy;          /* which free slots a recall takes first: PI_EVICT_ASCENDING
                                (lowest slot index) or PI_EVICT_LRU (empty slots, then
                                the block selected longest ago); placed before host_alloc */
  int host_alloc;            /* host store allocation: 0 = cudaHostAlloc (pinned,
                                mapped); 1 = anonymous mmap advised for transparent huge
                                pages, then cudaHostRegister (pinned, mapped); measured
                                on GB300: the UVA gather's scattered block reads run
                                about 4x slower through mapping 1, sequential reads
                                alike, so 0 is the one to use */
  int pin_layers;            /* layers that can be held whole in HBM (IO-adaptive
                                admission): the first ceil(n/2) and the last
                                floor(n/2) layers get room for max_blocks blocks per
                                request (0 = none) */
  const int* pool_slots_per_req; /* optional host [batch]: per-request P (each
                                >= k_max + window); NULL = pool_slots for all */
} pi_config;

typedef struct pi_pool pi_pool;

typedef struct pi_recall_stats {
  long long bytes;           /* bytes copied host -> pool */
  long long fragments;       /* copy units moved (blocks; block-heads head-wise) */
  long long runs;            /* contiguous runs after merging adjacent units */
  long long api_calls;       /* cudaMemcpyAsync calls issued (0 for the UVA kernel) */
  long long hits;            /* selected units already resident */
  double host_wait_ms;       /* host time blocked on the plan (memcpy, staged arms) */
  double cpu_gather_ms;      /* staged arm: CPU gather time */
} pi_recall_stats;

typedef struct pi_step_stats {
  pi_recall_stats recall;    /* summed over layers */
  long long selected;        /* selected units summed over layers and requests */
} pi_step_stats;

/* Pointers into library-owned device state, for inspection and tests. */
typedef struct pi_pool_views {
  void* pool;                /* device pool base (slots of BB bytes) */
  const long long* slot_base;/* host [batch][layers]: first global slot of (r, l);
                                global slot of (r, l, s) = slot_base[r*layers + l] + s */
  const int* slots_per_req;  /* host [batch]: the configured P_r */
  float* kmean;              /* device [R][L][max_blocks][Hkv][D] fp32 summaries */
  int* ntok;                 /* device [R][L] tokens held */
  int* slot_of_block;        /* device [R][L][U][max_blocks], U = 1 or Hkv; -1 = absent */
  int* block_of_slot;        /* device [R][L][U][P_max]; -1 = empty */
  int p_max;
  int* step_sel;             /* device [L][R][U][cap]: selections of pi_decode_step */
  int* step_nsel;            /* device [L][R][U] */
  int* step_table;           /* device [L][R][U][cap] */
  size_t block_bytes, frag_bytes, host_region_bytes;
  int* slot_stamp;           /* device [R][L][U][P_max]: epoch a slot's block was last
                                selected (-1 never); maintained under PI_EVICT_LRU */
  const int* slots_rl;       /* host [batch][layers]: slots in use for (r, l) (P_r, or
                                the room of a pinned layer) */
  const int* capacity_rl;    /* host [batch][layers]: slots reserved for (r, l) */
  long long total_slots;     /* slots of the whole pool */
  const unsigned* dev_status;/* device: the sticky status word's raw bits (1 an index out of
                                range, 2 a bounded wait ran out, 4 a pool too small, 8 more work
                                than a launch was sized for); pi_get_device_status maps them */
} pi_pool_views;

/* ------------------------------------------------------------------ lifetime */
int pi_abi_version(void);
const char* pi_status_str(pi_status s);

/* Create a pool on the current CUDA device. Allocates the pinned mapped host
 * store (host_layers*batch*max_blocks*BB bytes, zero-filled), the device pool
 * (zeroed; all slots empty), summaries, maps and scratch. Honors the host-side
 * fault hook PI_FAULT=pinned_alloc_fail (environment) for tests.
 * Errors: PI_ERR_INVALID (sizes: head_dim in {64,128}, block_tokens in
 * {16,32,64,128}, Hq % Hkv == 0, Hq/Hkv <= 8, max_blocks <= 65536, P >= cap),
 * PI_ERR_HOST_ALLOC, PI_ERR_OOM. On error *out is NULL and nothing leaks. */
pi_status pi_pool_create(const pi_config* cfg, pi_pool** out);
pi_status pi_pool_destroy(pi_pool* p);   /* synchronizes the device first */
pi_status pi_pool_get_config(const pi_pool* p, pi_config* out);
pi_status pi_pool_get_views(pi_pool* p, pi_pool_views* out);

/* Host pointer (pinned, writable by the caller) to the KV region of (layer,
 * request): [max_blocks][Hkv][2][B][D] bf16. Aliased layers share a region.
 * Fill it before pi_update_summaries; later changes go through pi_append_kv.
 * NULL on a bad index. */
void* pi_host_kv(pi_pool* p, int layer, int req);

/* ------------------------------------------------------------------ a-1 summaries */
/* Set the token count of every request of `layer` (host array ntok[R]) and
 * compute the block summaries kmean[b][g][:] = (sum over the block's valid
 * tokens, in token order, of K in fp32) / valid, for blocks
 * [block_begin, block_end) clipped to each request's block count. Keys are read
 * from k_dev (device, same layout as the host region of that layer, per request
 * consecutive) or, if k_dev is NULL, from the host store through the GPU's
 * mapping of it. Also seeds the running sum of each request's last block.
 * Score definition: PulseInfer Guide, "SoloHead Sparse Selection" names a
 * per-block importance; the per-KV-head mean key is this library's reading.
 * Errors: PI_ERR_INVALID (layer, range, ntok > max_blocks*B). */
pi_status pi_update_summaries(pi_pool* p, int layer, const void* k_dev, int block_begin, int block_end,
                              const int* ntok_host, pi_stream s);

/* ------------------------------------------------------------------ a-7 append */
/* Append one decoded token per request to `layer`: k_new/v_new device
 * [R][Hkv][D] bf16. Writes through to the host store and, if the token's block
 * is resident, to its pool slot; updates that block's summary from the running
 * fp32 sum (bit-identical to recomputing it in token order) and the token
 * count. Errors: PI_ERR_INVALID when a request would exceed max_blocks*B. */
pi_status pi_append_kv(pi_pool* p, int layer, const void* k_new, const void* v_new, pi_stream s);

/* ------------------------------------------------------------------ a-2 select */
/* SoloHead-style shared block selection of `layer` for every request.
 * score(b) = sum over query heads h of q_h . kmean[b, h / G], evaluated in fp32
 * as sum_g qsum_g . kmean[b, g] with qsum_g = sum_{h in g} q_h (head order) and
 * a fixed 32-lane order: lane i accumulates elements 128c+4i+j with fused
 * multiply-add (c, then j ascending), then a xor-butterfly 16,8,4,2,1.
 * Candidates: blocks 0 .. nb-W-1 (nb = ceil(ntok/B)); pick min(k_r, candidates)
 * by (score descending, block index ascending; -0.0 equals +0.0), add the W most
 * recent blocks, write ascending to sel[r][0..nsel[r]). k_per_req: device [R],
 * each clamped to [0, k_max]. Head-wise pools (PI_HEADWISE) select per KV head g
 * with score_g(b) = qsum_g . kmean[b, g] into sel[r][g][..]. mode = PI_CONSENSUS
 * ranks by the consensus score instead (PulseInfer Guide, "SoloHead Sparse
 * Selection", "1. Consensus Scoring Mechanism"): per GQA group g the per-head
 * scores S(h, b) = q_h . kmean[b, g] (D/4 lanes, lane i accumulates d = 4i + j by
 * fused multiply-add, then a xor-butterfly D/8 .. 1), c_g = max_h S + lambda x
 * (sum_h S / G) with each operation rounded to fp32, score(b) = sum of c_g over
 * g ascending; same candidates, ties and output. Pools of one block set per
 * request (select_mode PI_SHARED or PI_CONSENSUS) accept PI_SHARED and
 * PI_CONSENSUS; head-wise pools accept PI_HEADWISE; otherwise PI_ERR_STATE.
 * Scores must be finite (NaN inputs are a caller error).
 * Source: PulseInfer Guide, "SoloHead Sparse Selection"; the abstract of the
 * PulseInfer paper (SoloHead coalesces head-wise fragmented recalls). */
pi_status pi_select_topk(pi_pool* p, int layer, const void* q, const int* k_per_req, int mode, int* sel,
                         int* nsel, pi_stream s);

/* ------------------------------------------------------------------ a-3/a-4 recall */
/* Make every selected unit of `layer` resident and write its slot to table.
 * Plan (per request, or per request and KV head in head-wise pools): missing =
 * selected units without a slot, ascending; free = slots empty or holding an
 * unselected unit, ascending; the i-th missing unit takes the i-th free slot.
 * Copy: each missing unit's bytes (a BB block, or an FB fragment head-wise) go
 * from the host store to its slot, by
 *   PI_RECALL_UVA    one gather kernel reading the mapped host store (no host
 *                    sync; the plan stays on the device),
 *   PI_RECALL_MEMCPY one cudaMemcpyAsync per run of adjacent units (the plan is
 *                    read back: one device->host copy and one host sync),
 *   PI_RECALL_STAGED CPU threads gather into a pinned staging buffer, one bulk
 *                    cudaMemcpyAsync, a GPU scatter kernel (the guide's three
 *                    phases; host sync as above).
 * Maps are committed only after the copy is enqueued: an error (including an
 * injected fault) leaves them unchanged. stats (optional) is filled after the
 * call's work completes (this adds a host sync to the UVA arm).
 * Source: PulseInfer Guide, "The Gather-Scatter I/O Engine" and "The Small-Packet
 * PCIe DMA Tax"; the PulseInfer abstract (gather-scatter I/O engine).
 * Errors: PI_ERR_INVALID, PI_ERR_CUDA, PI_ERR_FAULT_INJECTED (PI_FAULT=recall_fail@N
 * fails the N-th recall call, counted from 1, before any map change). */
pi_status pi_recall(pi_pool* p, int layer, const int* sel, const int* nsel, int method, int* table,
                    pi_recall_stats* stats, pi_stream s);

/* Place blocks[0..n) (ascending, host array) of (layer, req) in slots 0..n-1
 * and copy their bytes from the host store (initial residency). Synchronous.
 * Errors: PI_ERR_INVALID (n > P_r, unsorted, out of range, head-wise pool). */
pi_status pi_pool_preload(pi_pool* p, int layer, int req, const int* blocks, int n, pi_stream s);

/* Switch the eviction policy for recalls issued afterwards (PI_EVICT_ASCENDING
 * or PI_EVICT_LRU; head-wise pools included). Least-recently-selected is this
 * library's variant: the pages leave eviction open. */
pi_status pi_pool_set_evict(pi_pool* p, int policy);

/* IO-adaptive offloading admission (PulseInfer Guide, "Interruptible Layer-Wise
 * Scheduling & Adaptive Admission", "2. IO-Adaptive Offloading Admission").
 * pinned = 1 holds `layer` whole in HBM: each request of it uses the room the
 * pool reserved for all its blocks (config pin_layers: the first ceil(n/2) and
 * last floor(n/2) layers), so once a block has been recalled it stays and the
 * layer recalls nothing new beyond first use; pinned = 0 returns the layer to
 * P_r slots and drops the blocks held in slots >= P_r from the maps (their next
 * selection recalls them). Selection, the recall rule and every result are
 * unchanged; only residency differs. Synchronizes the device. PI_ERR_INVALID
 * for a layer without reserved room. */
pi_status pi_pool_pin_layer(pi_pool* p, int layer, int pinned);

/* One admission decision from the host link's measured utilisation (recalled
 * bytes per second over the link's peak, 0..1): above 0.85 the next pinnable
 * layer in the order 0, L-1, 1, L-2, ... is pinned; below 0.5 the layer pinned
 * last is released; otherwise nothing changes (the guide's thresholds). *layer =
 * the layer changed (-1: none), *pinned = its new state. Synchronizes the device
 * when it changes a layer. */
pi_status pi_pool_admission(pi_pool* p, double link_util, int* layer, int* pinned);

/* The admission rule of pi_pool_admission alone, on host arrays (no pool, no
 * device): pinnable[l], pinned[l] (0/1, host [layers]) and last_pinned (the layer
 * pinned most recently and still pinned, -1: none). Writes the decision to
 * *layer (-1: none) and *pin (1 pin, 0 release) without changing anything.
 * Source: PulseInfer Guide, "Interruptible Layer-Wise Scheduling & Adaptive
 * Admission", "2. IO-Adaptive Offloading Admission" (the two utilisation
 * thresholds).
 * Errors: PI_ERR_INVALID (layers <= 0, a null array or output, link_util
 * negative or NaN, last_pinned >= layers, or last_pinned >= 0 naming a layer
 * that is not pinnable or not pinned); outputs are untouched then. */
pi_status pi_admission_decide(int layers, const int* pinnable, const int* pinned, int last_pinned, double link_util,
                              int* layer, int* pin);

/* Recall counters the device accumulates over every recall plan (the decode
 * step's selections with plan, pi_recall) since the pool was created or last
 * reset, summed over layers: *recalled = blocks copied into the pool (misses),
 * *hits = selected blocks found resident. A decode step with statistics
 * (pi_decode_step with stats) zeroes them at its start. Synchronizes the
 * device; reset = 1 zeroes them after reading. Errors: PI_ERR_INVALID (null
 * pool or output, reset not 0 or 1). */
pi_status pi_pool_recall_totals(pi_pool* p, long long* recalled, long long* hits, int reset);

/* Weight lambda of the group mean in the consensus score (default 0.5, the
 * guide's "typical" value; its worked example uses 1). Applies to later
 * PI_CONSENSUS selections. PI_ERR_INVALID unless 0 <= lambda <= 1e30. */
pi_status pi_pool_set_consensus_lambda(pi_pool* p, float lambda);

/* Retune the UVA gather: grid size (CTAs; 0 = default), 16-byte loads in flight
 * per thread (2, 4, 8 or 16) and placement: exclusive = 1 (the default) runs
 * 1024-thread CTAs (default: a quarter of the SMs, an eighth per gather when
 * the decode step pairs gathers on two copy streams) that reserve enough shared
 * memory to keep attention CTAs off their SMs, so host-link reads stay on a few
 * SMs; exclusive = 0 runs 256-thread CTAs, one per SM, beside other kernels.
 * Copy units under 32 KiB always take the 256-thread shape. Applies to calls
 * issued afterwards. */
pi_status pi_pool_set_gather(pi_pool* p, int ctas, int depth, int exclusive);

/* Forget residency of `layer` (-1 = all layers): every slot empty. Bytes stay. */
pi_status pi_pool_flush(pi_pool* p, int layer, pi_stream s);

/* ------------------------------------------------------------------ a-5 attention */
/* GQA sparse decode attention of `layer` over the resident selected blocks:
 * for query head h (KV head g = h / G) the tokens of sel[..][0..nsel) (ascending
 * block, then token; a block b holds min(B, ntok - b*B) valid tokens) read from
 * the pool through table; z = q_h . K / sqrt(D) in fp32 from bf16 products;
 * softmax and the weighted sum of V accumulate in fp32 (weights enter the PV
 * product as bf16); out rounded to bf16. lse (optional) = log-sum-exp of z.
 * logits (optional, debugging) fp32 [R][Hq][cap][B] receives z of valid tokens.
 * An empty selection gives out = 0, lse = -inf.
 * Source: PulseInfer Guide, "PulseInfer Architectural Foundations" (attention
 * over the recalled pool blocks) and "SoloHead Sparse Selection" (GQA).
 * Errors: PI_ERR_INVALID. */
pi_status pi_sparse_decode(pi_pool* p, int layer, const void* q, const int* sel, const int* table,
                           const int* nsel, void* out, float* lse, float* logits, pi_stream s);

/* Sparse decode attention that allocates nothing. The pages have no counterpart:
 * this entry point exists for callers that cannot call cudaMalloc, such as
 * serving engines that reserve all device memory in their own arena up front
 * and forbid later allocations. It computes what pi_sparse_decode computes
 * (shared selection only) over a caller-owned paged KV buffer, without a pool:
 *   kv_slots   device, n_slots slots of [hkv][2 (K,V)][block_tokens][head_dim]
 *              bf16 (16-byte aligned); slot_table [batch][cap] gives, for each
 *              selected block, its slot index in kv_slots;
 *   q [batch][hq][head_dim] bf16, sel [batch][cap] ascending block ids, nsel
 *   [batch], ntok [batch] tokens held per request (all device);
 *   out [batch][hq][head_dim] bf16, lse [batch][hq] fp32 (optional).
 * Its scratch (split-K partials, merge counters, per-request slot bases; about
 * 8.3 MiB) is one fixed array in device memory that every GPU loading the
 * library holds until the process exits. Limits: batch*hkv <= 1024,
 * cap <= 512, (hq/hkv)*head_dim <= 1024, hq/hkv <= 8; larger sizes return
 * PI_ERR_INVALID. The first call on a device resolves the array's address on
 * that device (make it before any stream capture). Every call shares the array:
 * each call clears what must start at zero, and calls that overlap on the GPU
 * (other streams, other threads) race. Problems found on the device are not
 * returned by this call (it returns once the work is enqueued); they are
 * recorded in a status word inside the array, which the call clears when it
 * starts and pi_sparse_decode_noalloc_status reads: a table entry outside
 * [0, n_slots) (that block is not read: its keys and values are skipped), nsel
 * outside [0, cap] (the request's output is zeros) or a bounded wait that ran
 * out (the output is partial). */
pi_status pi_sparse_decode_noalloc(const void* kv_slots, long long n_slots, int batch, int hq, int hkv,
                                   int head_dim, int block_tokens, int cap, const void* q, const int* sel,
                                   const int* slot_table, const int* nsel, const int* ntok, void* out, float* lse,
                                   pi_stream s);

/* The device-side outcome of the last pi_sparse_decode_noalloc call on the
 * current device, read once the work enqueued on s has finished (synchronizes
 * s; allocates nothing): PI_OK, PI_ERR_DEVICE (an out-of-range table entry or
 * selection count), PI_ERR_TIMEOUT (a bounded wait ran out), PI_ERR_STATE (no
 * call on this device yet). Like the entry point it has no counterpart in the
 * pages. */
pi_status pi_sparse_decode_noalloc_status(pi_stream s);

/* Attention mass a block selection keeps: a diagnostic, off the decode path.
 * For request r and query head h (group g = h / G), with z_t = q_h . K_t /
 * sqrt(D) over all ntok tokens t of (r, layer):
 *   mass[r][h] = sum over t in a selected block of exp(z_t) / sum over all t of exp(z_t),
 * the share of h's full softmax attention that the selection keeps. per_head = 0:
 * sel [R][cap], nsel [R] (one set per request: PI_SHARED / PI_CONSENSUS);
 * per_head = 1: sel [R][Hkv][cap], nsel [R][Hkv] (head h uses its group's set).
 * Independent of the pool's select_mode, so selections from pools of either kind
 * over the same tokens can be compared. A block listed twice counts once.
 * K is read from the host store through the mapping, so the whole context of
 * the layer crosses the host link (Hkv*ntok*D*2 bytes per request). Logits and
 * sums in fp32, combined per chunk of tokens by a log-sum-exp merge in a fixed
 * order (deterministic). mass = 0 where ntok = 0. q, sel, nsel, mass: device.
 * A selected index outside [0, nb) is skipped and flags PI_ERR_DEVICE. The first
 * call allocates the pool's scratch for it (a synchronizing cudaMalloc).
 * Source: PulseInfer Guide, "SoloHead Sparse Selection", "2. High Attention Mass
 * Preservation" (the shared set keeps nearly the attention mass that independent
 * per-head sets keep while moving fewer bytes).
 * Errors: PI_ERR_INVALID, PI_ERR_OOM, PI_ERR_CUDA. */
pi_status pi_attention_mass(pi_pool* p, int layer, const void* q, const int* sel, const int* nsel, int per_head,
                            float* mass, pi_stream s);

/* ------------------------------------------------------------------ a-6 pipeline */
/* One decode step over all layers with the recall of layer l+1 overlapped with
 * attention of layer l: compute stream runs append, select and attention; the
 * copy stream runs recall; events order them (no host sync with PI_RECALL_UVA).
 * q_all [L][R][Hq][D] bf16, k_new_all/v_new_all [L][R][Hkv][D] bf16 (both NULL:
 * no append), k_budget [L][R] int32, out_all [L][R][Hq][D] bf16, lse_all
 * [L][R][Hq] fp32 (optional); all device. Selections and tables land in the
 * pool's per-layer step buffers (pi_pool_views). stats: optional (adds a sync).
 * Source: PulseInfer abstract and Guide, "Interruptible Layer-Wise Scheduling". */
pi_status pi_decode_step(pi_pool* p, const void* q_all, const void* k_new_all, const void* v_new_all,
                         const int* k_budget, int method, void* out_all, float* lse_all, pi_stream compute,
                         pi_stream copy, pi_step_stats* stats);

/* Shape of pi_decode_step's pipeline (default: attention_stream = 1).
 * attention_stream = 0: two streams, the
 * caller's compute stream runs append, selection and attention, selection running
 * select_ahead layers in front of attention (1 = the next layer only, 0 = every
 * layer first). attention_stream = 1: attention runs on a stream the pool owns,
 * selection runs ahead as far as the data allow, and consecutive steps overlap
 * (select_ahead is ignored); the caller's compute stream still completes after
 * the whole step. Results are identical in every shape. Synchronizes the device. */
pi_status pi_pool_set_pipeline(pi_pool* p, int select_ahead, int attention_stream);

/* Interruptible layer-wise scheduling (PulseInfer Guide, "Interruptible
 * Layer-Wise Scheduling"). dependent = 1 models a model whose query of layer
 * l+1 comes out of its layer l: in pi_decode_step a request's selection of
 * layer l+1 waits for its attention of layer l (the query is still read from
 * q_all). The batch splits into `groups` contiguous request groups (request r
 * in group g when g*R/groups <= r < (g+1)*R/groups); each group's chain (append,
 * selection + plan, recall, attention, layer after layer) runs on its own
 * stream (group 0 on the caller's compute stream, the others on streams the
 * pool owns) and the copy stream takes the groups' recalls in turn, so one
 * group's recall of layer l streams over the host link while the others
 * compute. groups = 1 is the rigid order (nothing overlaps the recall).
 * dependent = 0 (the default): every layer's query is known up front and
 * selections run ahead (pi_pool_set_pipeline). The dependent schedule takes
 * UVA recall only (pi_decode_step returns PI_ERR_INVALID for other methods).
 * Selections, tables, slot maps and recalled bytes are identical under every
 * schedule; attention outputs may differ in floating-point summation order
 * (a launch over fewer requests splits the selected blocks over more CTAs).
 * Synchronizes the device.
 * PI_ERR_INVALID unless dependent is 0 or 1 and 1 <= groups <= min(8, batch). */
pi_status pi_pool_set_schedule(pi_pool* p, int dependent, int groups);

/* Copy streams of the UVA recall in pi_decode_step (default schedules): n = 2
 * (the default) runs odd layers' gathers on a second stream the pool owns, so a
 * gather's start overlaps the previous gather's tail (each still follows its
 * layer's selection and precedes its attention; measured 6-8 % more tokens/s);
 * n = 1 runs every gather on the caller's copy stream. Results are identical.
 * Synchronizes the device. PI_ERR_INVALID unless n is 1 or 2. */
pi_status pi_pool_set_copy_streams(pi_pool* p, int n);

/* Fused selection + recall (on = 1): in pi_decode_step with PI_RECALL_UVA, the
 * selection, recall plan and gather of a layer (of a request group, under the
 * dependent schedule) run as one launch of `ctas` CTAs on the copy stream (0 =
 * a quarter of the SMs) instead of a selection on the compute stream and a
 * gather on the copy stream. Its CTAs first claim selection items (a chunk of a
 * unit's candidates) from a counter; the CTA that completes a unit's last chunk
 * runs the unit's top-k and plan and publishes them through a flag; then every
 * CTA copies its share of each unit's missing blocks once the unit's flag is
 * set (bounded wait: PI_ERR_TIMEOUT in the status word, the unit skipped). A CTA
 * waits only after every item has been taken by a running CTA, so the launch
 * completes whatever the CTAs' residency. Results are identical to the unfused
 * step. Under the dependent schedule each request group's launch runs on the
 * group's stream (groups share the link instead of taking turns on the copy
 * stream); launches over the same requests of one layer stay stream-ordered.
 * Source: the guide's "The Gather-Scatter I/O Engine" (selected blocks gathered
 * straight into pool slots); running the three steps as one launch is this
 * library's design.
 * Synchronizes the device. Errors: PI_ERR_INVALID. */
pi_status pi_pool_set_fused(pi_pool* p, int on, int ctas);

/* Split count of the attention kernel (CTAs per request and KV head; 0 = the
 * default: one wave at the kernel's occupancy). Clamped to what the pool's
 * scratch holds. Results change only by floating-point summation order. */
pi_status pi_pool_set_attention(pi_pool* p, int splits);

/* Shape of the selection launch (pi_select_topk and the decode step's selection).
 * cluster = 1 (the default): each unit (a request, or a request and KV head) is
 * one thread-block cluster whose CTAs score a share of the candidates each and
 * store the scores in the shared memory of the cluster's first CTA, which then
 * runs the top-k and, in the decode step, the recall plan and the token append;
 * ctas_per_unit = CTAs per cluster (1..16; 0 = about two CTAs per SM over the
 * launch). cluster = 0: the earlier form, where the scores go through global
 * memory and the unit's last CTA to finish runs the top-k. Results are
 * identical. Library tuning; the pages have no counterpart. PI_ERR_INVALID
 * unless cluster is 0 or 1 and 0 <= ctas_per_unit <= 16. */
pi_status pi_pool_set_selection(pi_pool* p, int cluster, int ctas_per_unit);

/* How the splits of one (request, KV head) combine. on = 1 (the default): when a
 * unit has 2..8 splits they are launched as one thread-block cluster and merge
 * their partial (m, l, O) through distributed shared memory; otherwise (on = 0,
 * one split, or more than 8) they merge through a global partial buffer
 * finalised by the unit's last CTA. Results change only by floating-point
 * summation order (the same order in both merges). PI_ERR_INVALID unless on is
 * 0 or 1. Library tuning; the pages have no counterpart. */
pi_status pi_pool_set_attention_cluster(pi_pool* p, int on);

/* pi_decode_step with HOST inputs and outputs (pinned or pageable): copies
 * q_all, k_new_all, v_new_all, k_budget host->device into pool-owned buffers,
 * runs the step and copies out_all (and lse_all if non-NULL) back. Returns after
 * the outputs are on the host. */
pi_status pi_decode_step_host(pi_pool* p, const void* q_all, const void* k_new_all, const void* v_new_all,
                              const int* k_budget, int method, void* out_all, float* lse_all,
                              pi_stream compute, pi_stream copy);

/* ------------------------------------------------------------------ timing */
enum { PI_K_APPEND = 0, PI_K_SELECT = 1, PI_K_PLAN = 2, PI_K_GATHER = 3, PI_K_ATTENTION = 4, PI_K_KINDS = 5 };

typedef struct pi_kernel_timing {
  long long launches;        /* kernels of this kind timed */
  double total_ms;           /* sum of their CUDA-event durations */
  double busy_ms;            /* length of the union of their [start, end] intervals
                                (less than total_ms when launches overlap) */
} pi_kernel_timing;

/* Enable per-kernel CUDA-event timing inside pi_decode_step for the next
 * max_steps steps (0 disables and frees the events). Each kernel launch of the
 * step is bracketed by two events on the stream it runs on. */
pi_status pi_pool_set_timing(pi_pool* p, int max_steps);
/* Synchronizes, sums the recorded durations per kind into out[PI_K_KINDS] and
 * resets the recording. */
pi_status pi_pool_get_timing(pi_pool* p, pi_kernel_timing* out);

/* ------------------------------------------------------------------ status */
/* Synchronizes the device, returns PI_OK or the first device-side error
 * (PI_ERR_DEVICE, PI_ERR_TIMEOUT, PI_ERR_POOL_FULL) recorded since the last clear.
 * PI_ERR_DEVICE covers an index read from memory out of range and a kernel that
 * met more work than its launch was sized for (in both cases the excess is
 * skipped, never accessed). */
pi_status pi_get_device_status(pi_pool* p);
pi_status pi_clear_device_status(pi_pool* p);

/* Self-test of the bounded device wait every kernel uses: one thread waits on an
 * mbarrier phase that nothing completes, gives up after limit_cycles (clock64;
 * 1..2e9), records PI_ERR_TIMEOUT in the status word and exits. The context
 * stays usable. Synchronous; returns the status word it read. */
pi_status pi_selftest_bounded_wait(pi_pool* p, long long limit_cycles);

/* Host-side fault injection for tests: "recall_fail@N" or "" (off). The
 * environment variable PI_FAULT is read once at pool creation. */
pi_status pi_set_fault(pi_pool* p, const char* spec);

#ifdef __cplusplus
}
#endif
#endif /* PI_H */
