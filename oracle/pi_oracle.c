/*
 * CPU ORACLE of the sparse KV-cache offloading decode path. TEST
 * INFRASTRUCTURE ONLY: tests, the smoke check and the benchmark's CPU-baseline
 * leg call it; the product path never does. It shares no code with the CUDA
 * library. Plain loops, no SIMD intrinsics, compiled with -ffp-contract=off.
 *
 * Sources (page title, section):
 *  [A] "PulseInfer: I/O-Centric Sparse KV Cache Offloading for Efficient
 *      Long-Context LLM Decoding", Abstract: most KV blocks live in CPU DRAM and
 *      only selected blocks are recalled; one shared block set (SoloHead) and
 *      a gathering recall path turn the recall into few large copies.
 *  [G] "PulseInfer Guide: I/O-Centric Sparse KV Cache Offloading":
 *      "SoloHead Sparse Selection" (one block set shared by all heads),
 *      "The Gather-Scatter I/O Engine" (recalled blocks land in pool page slots),
 *      "The Small-Packet PCIe DMA Tax" (paged blocks of B tokens),
 *      "PulseInfer Architectural Foundations" (attention over the pool).
 *
 * The pages name SoloHead but leave the block score S(h,b) undefined. This
 * library fixes it: every KV block keeps the per-KV-head mean of its keys, and
 * score(b) = sum over all query heads h of q_h . kmean[b, group(h)] in fp32,
 * group(h) = h / (Hq/Hkv). Top-k over the non-recent blocks (score descending,
 * lower block index first on ties) plus the W most recent blocks. The guide's
 * consensus rule (largest per-head score + lambda x mean, per GQA group) is a
 * second ranking over the same summaries (or_consensus_score).
 *
 * Precision: the score decides integer outputs (selected block ids), so the
 * oracle evaluates it in fp32 in one fixed order (below) that the GPU follows
 * too; everything else (attention) is fp64 and the GPU is compared within a
 * tolerance.
 *
 * Host KV layout of one (layer, request): [block][kv head g][K=0|V=1][token t][d] bf16.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------ bf16 */
static float or_bf16(uint16_t h) {
  uint32_t u = (uint32_t)h << 16;
  float f;
  memcpy(&f, &u, 4);
  return f;
}

/* fp64 -> bf16 bits, round to nearest even, done directly on the fp64 value:
 * scale so the bf16 quantum becomes 1, round with nearbyint (RNE in the default
 * rounding mode; exact because the scale is a power of two), scale back. */
uint16_t or_bf16_rne(double x) {
  if (isnan(x)) return 0x7FC0;
  if (x == 0.0) return signbit(x) ? 0x8000 : 0x0000;
  int e;
  (void)frexp(x, &e);                   /* |x| = m * 2^e, m in [0.5, 1) */
  int qexp = e - 8;                     /* 8 significant bits */
  if (qexp < -133) qexp = -133;         /* bf16 subnormal quantum */
  double y = ldexp(nearbyint(ldexp(x, -qexp)), qexp);
  if (fabs(y) >= 0x1p128) return signbit(x) ? 0xFF80 : 0x7F80;
  float f = (float)y;                   /* exact: y has <= 8 significant bits */
  uint32_t u;
  memcpy(&u, &f, 4);
  return (uint16_t)(u >> 16);
}

/* ------------------------------------------------------------------ a-1 summary */
/* kmean[g][d] = (sum over the first n_valid tokens, in token order, fp32) / n_valid.
 * blk: one block [Hkv][2][B][D]. */
void or_block_summary(const uint16_t* blk, int Hkv, int B, int D, int n_valid, float* kmean) {
  for (int g = 0; g < Hkv; g++) {
    const uint16_t* K = blk + (size_t)g * 2 * B * D;
    for (int d = 0; d < D; d++) {
      float s = 0.0f;
      for (int t = 0; t < n_valid; t++) s = s + or_bf16(K[(size_t)t * D + d]);
      kmean[(size_t)g * D + d] = (n_valid > 0) ? s / (float)n_valid : 0.0f;
    }
  }
}

/* summaries of blocks 0..nb-1 of a host region holding ntok tokens */
void or_region_summaries(const uint16_t* region, int ntok, int Hkv, int B, int D, float* kmean_all) {
  int nb = (ntok + B - 1) / B;
  size_t bs = (size_t)Hkv * 2 * B * D;
  for (int b = 0; b < nb; b++) {
    int nv = ntok - b * B;
    if (nv > B) nv = B;
    or_block_summary(region + (size_t)b * bs, Hkv, B, D, nv, kmean_all + (size_t)b * Hkv * D);
  }
}

/* ------------------------------------------------------------------ a-2 score */
/* qsum[g][d] = sum over the query heads of group g (ascending h) of q[h][d], fp32.
 * sum_h q_h . kmean[group(h)] = sum_g qsum[g] . kmean[g]: the per-head sum is
 * regrouped by KV head (exact in real arithmetic), which is the fixed order. */
void or_qsum(const uint16_t* q, int Hq, int Hkv, int D, float* qsum) {
  int G = Hq / Hkv;
  for (int g = 0; g < Hkv; g++)
    for (int d = 0; d < D; d++) {
      float s = 0.0f;
      for (int j = 0; j < G; j++) s = s + or_bf16(q[(size_t)(g * G + j) * D + d]);
      qsum[(size_t)g * D + d] = s;
    }
}

/* Canonical fp32 dot product of length E (E % 4 == 0): 32 partial sums, partial i
 * takes elements e = 128c + 4i + j (c ascending, then j = 0..3) with fused
 * multiply-add; then five butterfly rounds acc[i] <- acc[i] + acc[i ^ off] for
 * off = 16, 8, 4, 2, 1, all partials updated from the previous round's values.
 * The result is acc[0] (all partials are equal after the last round). */
float or_score(const float* qs, const float* km, int E) {
  float acc[32], nxt[32];
  for (int i = 0; i < 32; i++) acc[i] = 0.0f;
  int chunks = (E + 127) / 128;
  for (int i = 0; i < 32; i++)
    for (int c = 0; c < chunks; c++)
      for (int j = 0; j < 4; j++) {
        int e = 128 * c + 4 * i + j;
        if (e < E) acc[i] = fmaf(qs[e], km[e], acc[i]);
      }
  for (int off = 16; off >= 1; off >>= 1) {
    for (int i = 0; i < 32; i++) nxt[i] = acc[i] + acc[i ^ off];
    for (int i = 0; i < 32; i++) acc[i] = nxt[i];
  }
  return acc[0];
}

/* ------------------------------------------------------------------ a-2 top-k */
typedef struct { float s; int b; } or_cand;

static int or_cand_cmp(const void* pa, const void* pb) {
  const or_cand* a = (const or_cand*)pa;
  const or_cand* b = (const or_cand*)pb;
  if (a->s > b->s) return -1;   /* higher score first; -0.0 == +0.0 */
  if (a->s < b->s) return 1;
  return (a->b < b->b) ? -1 : (a->b > b->b);  /* then lower block index */
}

static int or_int_cmp(const void* pa, const void* pb) {
  int a = *(const int*)pa, b = *(const int*)pb;
  return (a > b) - (a < b);
}

/* Candidates are blocks 0..nb-W-1 (the W most recent are always kept). Take the
 * first min(k, ncand) candidates under (score desc, index asc), add the recent
 * blocks, output ascending. Returns nsel. Scores must be finite. */
int or_select_topk(const float* score, int nb, int k, int W, int* sel) {
  int ncand = nb - W;
  if (ncand < 0) ncand = 0;
  int kk = k < ncand ? k : ncand;
  if (kk < 0) kk = 0;
  or_cand* c = (or_cand*)malloc(sizeof(or_cand) * (size_t)(ncand > 0 ? ncand : 1));
  for (int b = 0; b < ncand; b++) { c[b].s = score[b]; c[b].b = b; }
  qsort(c, (size_t)ncand, sizeof(or_cand), or_cand_cmp);
  int n = 0;
  for (int i = 0; i < kk; i++) sel[n++] = c[i].b;
  for (int b = ncand; b < nb; b++) sel[n++] = b;
  free(c);
  qsort(sel, (size_t)n, sizeof(int), or_int_cmp);
  return n;
}

/* Shared selection of one (request, layer). q [Hq][D] bf16, kmean_all [nb][Hkv][D].
 * scores_out (optional) receives score[b] for candidates. */
int or_select_shared(const uint16_t* q, const float* kmean_all, int nb, int Hq, int Hkv, int D, int k,
                     int W, int* sel, float* scores_out) {
  int E = Hkv * D;
  float* qs = (float*)malloc(sizeof(float) * (size_t)E);
  float* sc = (float*)malloc(sizeof(float) * (size_t)(nb > 0 ? nb : 1));
  or_qsum(q, Hq, Hkv, D, qs);
  int ncand = nb - W > 0 ? nb - W : 0;
  for (int b = 0; b < ncand; b++) sc[b] = or_score(qs, kmean_all + (size_t)b * E, E);
  if (scores_out) memcpy(scores_out, sc, sizeof(float) * (size_t)ncand);
  int n = or_select_topk(sc, nb, k, W, sel);
  free(qs);
  free(sc);
  return n;
}

/* Head-wise selection (comparison arm): for KV head g, score_g[b] =
 * qsum[g] . kmean[b, g] over D elements, its own top-k. sel [Hkv][cap]. */
void or_select_headwise(const uint16_t* q, const float* kmean_all, int nb, int Hq, int Hkv, int D, int k,
                        int W, int cap, int* sel, int* nsel) {
  int E = Hkv * D;
  float* qs = (float*)malloc(sizeof(float) * (size_t)E);
  float* sc = (float*)malloc(sizeof(float) * (size_t)(nb > 0 ? nb : 1));
  or_qsum(q, Hq, Hkv, D, qs);
  int ncand = nb - W > 0 ? nb - W : 0;
  for (int g = 0; g < Hkv; g++) {
    for (int b = 0; b < ncand; b++) sc[b] = or_score(qs + (size_t)g * D, kmean_all + (size_t)b * E + (size_t)g * D, D);
    nsel[g] = or_select_topk(sc, nb, k, W, sel + (size_t)g * cap);
  }
  free(qs);
  free(sc);
}

/* ------------------------------------------------------------------ consensus score */
/* [G] "SoloHead Sparse Selection", "1. Consensus Scoring Mechanism": within one
 * GQA group, a block's consensus score is the largest of the group's per-head
 * scores plus lambda times their mean (the guide's figure uses lambda = 1, its
 * formula "typically" 0.5). The per-head score S(h, b) is left undefined there;
 * this library reads it the same way as the shared score: S(h, b) = q_h .
 * kmean[b, group(h)], in one fixed fp32 order (below). The pages speak of one
 * group; a request with several KV heads sums the groups' consensus scores
 * (g ascending) so that one block set serves the whole request, as in the
 * shared selection. */

/* One head's score alone: D/4 partial sums, partial i takes d = 4i + j (j =
 * 0..3) by fused multiply-add, then butterfly rounds acc[i] <- acc[i] +
 * acc[i ^ off] for off = D/8 .. 1. (The group order below with one head.) */
float or_head_score(const uint16_t* qh, const float* kmg, int D) {
  float acc[32], nxt[32];
  int n = D / 4;
  for (int i = 0; i < n; i++) {
    acc[i] = 0.0f;
    for (int j = 0; j < 4; j++) acc[i] = fmaf(or_bf16(qh[4 * i + j]), kmg[4 * i + j], acc[i]);
  }
  for (int off = n / 2; off >= 1; off >>= 1) {
    for (int i = 0; i < n; i++) nxt[i] = acc[i] + acc[i ^ off];
    for (int i = 0; i < n; i++) acc[i] = nxt[i];
  }
  return acc[0];
}

/* The G scores of one group's heads together, in the fixed order: P = the
 * smallest power of two >= G (heads G..P-1 are zero rows); n = D/4 partials per
 * head, partial i of head j = fused multiply-add over d = 4i + t (t = 0..3).
 * Then for m = P, P/2, .., 2 with off = n*m/(2P): partial i keeps the half of
 * its m values selected by bit `off` of i (the upper half when set) and adds,
 * position by position, what partial i^off holds at the same positions; then
 * butterfly rounds on the one value left for off = n/(2P) .. 1. Head j's score
 * is then held by partial j*(n/P). out[0..G). */
void or_group_head_scores(const uint16_t* qg, const float* kmg, int G, int D, float* out) {
  int n = D / 4, P = 1;
  while (P < G) P <<= 1;
  float v[32][8], nv[32][8];
  for (int i = 0; i < n; i++)
    for (int j = 0; j < P; j++) {
      v[i][j] = 0.0f;
      if (j < G)
        for (int t = 0; t < 4; t++) v[i][j] = fmaf(or_bf16(qg[(size_t)j * D + 4 * i + t]), kmg[4 * i + t], v[i][j]);
    }
  for (int m = P; m >= 2; m >>= 1) {
    int off = n * m / (2 * P), h = m / 2;
    for (int i = 0; i < n; i++) {
      int up = (i & off) != 0;
      for (int x = 0; x < h; x++) nv[i][x] = v[i][up ? x + h : x] + v[i ^ off][up ? x + h : x];
    }
    for (int i = 0; i < n; i++)
      for (int x = 0; x < h; x++) v[i][x] = nv[i][x];
  }
  for (int off = n / (2 * P); off >= 1; off >>= 1) {
    for (int i = 0; i < n; i++) nv[i][0] = v[i][0] + v[i ^ off][0];
    for (int i = 0; i < n; i++) v[i][0] = nv[i][0];
  }
  for (int j = 0; j < G; j++) out[j] = v[j * (n / P)][0];
}

/* km_b: one block's summaries [Hkv][D]. Per group: the head scores as above;
 * m = the largest; s = their sum as a pairwise tree over the P padded heads
 * (pairs j, j^1; then j, j^2; ...; zero for padded heads); c = m + lambda *
 * (s / G), each step rounded to fp32; the result is the sum of c over the
 * groups (g ascending). */
float or_consensus_score(const uint16_t* q, const float* km_b, int Hq, int Hkv, int D, float lambda) {
  int G = Hq / Hkv, P = 1;
  while (P < G) P <<= 1;
  float total = 0.0f;
  for (int g = 0; g < Hkv; g++) {
    float hs[8], w[8], nw[8];
    or_group_head_scores(q + (size_t)g * G * D, km_b + (size_t)g * D, G, D, hs);
    float m = hs[0];
    for (int j = 1; j < G; j++)
      if (hs[j] > m) m = hs[j];
    for (int j = 0; j < P; j++) w[j] = (j < G) ? hs[j] : 0.0f;
    for (int o = 1; o < P; o <<= 1) {
      for (int j = 0; j < P; j++) nw[j] = w[j] + w[j ^ o];
      for (int j = 0; j < P; j++) w[j] = nw[j];
    }
    float mean = w[0] / (float)G;
    float t = lambda * mean;
    float c = m + t;
    total = total + c;
  }
  return total;
}

/* Consensus selection of one (request, layer): the same top-k rule as the
 * shared selection over consensus scores. */
int or_select_consensus(const uint16_t* q, const float* kmean_all, int nb, int Hq, int Hkv, int D, int k, int W,
                        float lambda, int* sel, float* scores_out) {
  int E = Hkv * D;
  float* sc = (float*)malloc(sizeof(float) * (size_t)(nb > 0 ? nb : 1));
  int ncand = nb - W > 0 ? nb - W : 0;
  for (int b = 0; b < ncand; b++) sc[b] = or_consensus_score(q, kmean_all + (size_t)b * E, Hq, Hkv, D, lambda);
  if (scores_out) memcpy(scores_out, sc, sizeof(float) * (size_t)ncand);
  int n = or_select_topk(sc, nb, k, W, sel);
  free(sc);
  return n;
}

/* ------------------------------------------------------------------ a-3 pool plan */
/* One pool of P slots. missing = selected blocks without a slot (ascending);
 * free = slots that are empty or hold a block not selected (ascending); the i-th
 * missing block takes the i-th free slot, evicting what that slot held.
 * table[i] = slot of sel[i] afterwards. Maps are updated in place.
 * Returns the number of missing blocks, or -1 if they outnumber the free slots
 * (maps untouched then). miss_block/miss_slot/evicted (optional) list the moves. */
int or_recall_plan(const int* sel, int nsel, int* slot_of_block, int* block_of_slot, int P, int* table,
                   int* miss_block, int* miss_slot, int* evicted) {
  int nmiss = 0, nfree = 0;
  int* missing = (int*)malloc(sizeof(int) * (size_t)(nsel > 0 ? nsel : 1));
  int* freel = (int*)malloc(sizeof(int) * (size_t)(P > 0 ? P : 1));
  for (int i = 0; i < nsel; i++)
    if (slot_of_block[sel[i]] < 0) missing[nmiss++] = sel[i];
  for (int s = 0; s < P; s++) {
    int b = block_of_slot[s];
    int keep = 0;
    if (b >= 0)
      for (int i = 0; i < nsel; i++)
        if (sel[i] == b) { keep = 1; break; }
    if (!keep) freel[nfree++] = s;
  }
  if (nmiss > nfree) { free(missing); free(freel); return -1; }
  for (int i = 0; i < nmiss; i++) {
    int s = freel[i];
    int old = block_of_slot[s];
    if (old >= 0) slot_of_block[old] = -1;
    slot_of_block[missing[i]] = s;
    block_of_slot[s] = missing[i];
    if (miss_block) miss_block[i] = missing[i];
    if (miss_slot) miss_slot[i] = s;
    if (evicted) evicted[i] = old;
  }
  for (int i = 0; i < nsel; i++) table[i] = slot_of_block[sel[i]];
  free(missing);
  free(freel);
  return nmiss;
}

/* Plan of a layer held whole in HBM ([G] "2. IO-Adaptive Offloading Admission":
 * the most active layers are retained in GPU HBM). Such a layer has room for
 * every block, so a recall takes the empty slots first (ascending) and only then
 * slots holding an unselected block (ascending): nothing is evicted while room
 * is left. Otherwise as or_recall_plan. */
int or_recall_plan_pinned(const int* sel, int nsel, int* slot_of_block, int* block_of_slot, int P, int* table,
                          int* miss_block, int* miss_slot, int* evicted) {
  int nmiss = 0, nfree = 0;
  int* missing = (int*)malloc(sizeof(int) * (size_t)(nsel > 0 ? nsel : 1));
  int* freel = (int*)malloc(sizeof(int) * (size_t)(P > 0 ? P : 1));
  for (int i = 0; i < nsel; i++)
    if (slot_of_block[sel[i]] < 0) missing[nmiss++] = sel[i];
  for (int pass = 0; pass < 2; pass++)
    for (int s = 0; s < P; s++) {
      int b = block_of_slot[s];
      if (pass == 0) {
        if (b < 0) freel[nfree++] = s;
        continue;
      }
      if (b < 0) continue;
      int keep = 0;
      for (int i = 0; i < nsel; i++)
        if (sel[i] == b) { keep = 1; break; }
      if (!keep) freel[nfree++] = s;
    }
  if (nmiss > nfree) { free(missing); free(freel); return -1; }
  for (int i = 0; i < nmiss; i++) {
    int s = freel[i];
    int old = block_of_slot[s];
    if (old >= 0) slot_of_block[old] = -1;
    slot_of_block[missing[i]] = s;
    block_of_slot[s] = missing[i];
    if (miss_block) miss_block[i] = missing[i];
    if (miss_slot) miss_slot[i] = s;
    if (evicted) evicted[i] = old;
  }
  for (int i = 0; i < nsel; i++) table[i] = slot_of_block[sel[i]];
  free(missing);
  free(freel);
  return nmiss;
}

/* Least-recently-selected variant of the plan (a pool policy option; the pages
 * leave eviction open). stamp[s] is the epoch at which slot s's block was last
 * selected (-1: never, or the slot is empty). This call is epoch `epoch`: the
 * free slots (empty or holding an unselected block) are taken in order of
 * (stamp ascending, slot ascending), so empty slots go first and among occupied
 * ones the block selected longest ago is evicted first. Every selected block's
 * slot is stamped with `epoch` afterwards. Otherwise as or_recall_plan. */
typedef struct { int stamp, slot; } or_free_cand;

static int or_free_cmp(const void* pa, const void* pb) {
  const or_free_cand* a = (const or_free_cand*)pa;
  const or_free_cand* b = (const or_free_cand*)pb;
  if (a->stamp != b->stamp) return (a->stamp < b->stamp) ? -1 : 1;
  return (a->slot > b->slot) - (a->slot < b->slot);
}

int or_recall_plan_lru(const int* sel, int nsel, int* slot_of_block, int* block_of_slot, int* stamp, int P,
                       int epoch, int* table, int* miss_block, int* miss_slot, int* evicted) {
  int nmiss = 0, nfree = 0;
  int* missing = (int*)malloc(sizeof(int) * (size_t)(nsel > 0 ? nsel : 1));
  or_free_cand* freel = (or_free_cand*)malloc(sizeof(or_free_cand) * (size_t)(P > 0 ? P : 1));
  for (int i = 0; i < nsel; i++)
    if (slot_of_block[sel[i]] < 0) missing[nmiss++] = sel[i];
  for (int s = 0; s < P; s++) {
    int b = block_of_slot[s];
    int keep = 0;
    if (b >= 0)
      for (int i = 0; i < nsel; i++)
        if (sel[i] == b) { keep = 1; break; }
    if (!keep) {
      freel[nfree].stamp = (b >= 0) ? stamp[s] : -1;
      freel[nfree].slot = s;
      nfree++;
    }
  }
  if (nmiss > nfree) { free(missing); free(freel); return -1; }
  qsort(freel, (size_t)nfree, sizeof(or_free_cand), or_free_cmp);
  for (int i = 0; i < nmiss; i++) {
    int s = freel[i].slot;
    int old = block_of_slot[s];
    if (old >= 0) slot_of_block[old] = -1;
    slot_of_block[missing[i]] = s;
    block_of_slot[s] = missing[i];
    if (miss_block) miss_block[i] = missing[i];
    if (miss_slot) miss_slot[i] = s;
    if (evicted) evicted[i] = old;
  }
  for (int i = 0; i < nsel; i++) {
    table[i] = slot_of_block[sel[i]];
    stamp[table[i]] = epoch;
  }
  free(missing);
  free(freel);
  return nmiss;
}

/* ------------------------------------------------------------------ a-5 attention */
/* Sparse GQA decode attention of one (request, layer) in fp64. For query head h
 * (KV head g = h / G) the tokens are those of the selected blocks, ascending block
 * then token, valid tokens only (block b holds min(B, ntok - b*B) tokens).
 * z_j = q_h . K_j / sqrt(D); m = max z; p_j = exp(z_j - m); lse = m + log(sum p);
 * out = sum p_j V_j / sum p, rounded to bf16 (RNE). An empty selection gives
 * out = 0 and lse = -inf. logits (optional) [Hq][nsel][B] receives z (others
 * left untouched). sel may differ per KV head: sel_g = sel + g*sel_stride,
 * nsel_g = nsel[g * nsel_stride_g] (shared: strides 0). */
void or_attention(const uint16_t* q, const uint16_t* region, const int* sel, int sel_stride,
                  const int* nsel, int nsel_stride, int ntok, int Hq, int Hkv, int B, int D,
                  uint16_t* out, double* lse, double* logits, int logits_cap) {
  int G = Hq / Hkv;
  size_t bs = (size_t)Hkv * 2 * B * D;
  double scale = 1.0 / sqrt((double)D);
  int maxtok = 0;
  for (int g = 0; g < Hkv; g++) {
    int n = nsel[(size_t)g * nsel_stride];
    if (n * B > maxtok) maxtok = n * B;
  }
  double* z = (double*)malloc(sizeof(double) * (size_t)(maxtok > 0 ? maxtok : 1));
  int* zt = (int*)malloc(sizeof(int) * (size_t)(maxtok > 0 ? maxtok : 1));
  double* acc = (double*)malloc(sizeof(double) * (size_t)D);
  for (int h = 0; h < Hq; h++) {
    int g = h / G;
    const int* sg = sel + (size_t)g * sel_stride;
    int ns = nsel[(size_t)g * nsel_stride];
    int n = 0;
    double m = -INFINITY;
    for (int i = 0; i < ns; i++) {
      int b = sg[i];
      int nv = ntok - b * B;
      if (nv > B) nv = B;
      const uint16_t* K = region + (size_t)b * bs + (size_t)g * 2 * B * D;
      for (int t = 0; t < nv; t++) {
        double s = 0.0;
        for (int d = 0; d < D; d++) s += (double)or_bf16(q[(size_t)h * D + d]) * (double)or_bf16(K[(size_t)t * D + d]);
        s *= scale;
        z[n] = s;
        zt[n] = (i * B + t);
        if (logits) logits[((size_t)h * logits_cap + i) * B + t] = s;
        if (s > m) m = s;
        n++;
      }
    }
    if (n == 0) {
      for (int d = 0; d < D; d++) out[(size_t)h * D + d] = 0;
      if (lse) lse[h] = -INFINITY;
      continue;
    }
    double l = 0.0;
    for (int d = 0; d < D; d++) acc[d] = 0.0;
    for (int j = 0; j < n; j++) {
      double p = exp(z[j] - m);
      l += p;
      int i = zt[j] / B, t = zt[j] % B;
      const uint16_t* V = region + (size_t)sg[i] * bs + ((size_t)g * 2 + 1) * B * D;
      for (int d = 0; d < D; d++) acc[d] += p * (double)or_bf16(V[(size_t)t * D + d]);
    }
    for (int d = 0; d < D; d++) out[(size_t)h * D + d] = or_bf16_rne(acc[d] / l);
    if (lse) lse[h] = m + log(l);
  }
  free(z);
  free(zt);
  free(acc);
}
