// Layer-wise decode step.
//
// "PulseInfer Guide: I/O-Centric Sparse KV Cache Offloading", section
// "Interruptible Layer-Wise Scheduling", and the PulseInfer abstract: recall of
// one layer's blocks runs while the GPU computes another layer, so variable
// recall latency hides behind compute. Three shapes, all ordered by events only:
//  - default: the compute stream runs append and selection (+ plan) of every
//    layer in turn, the copy stream the gathers, a pool-owned stream the
//    attention; recall(l) waits for select(l), attention(l) for recall(l);
//  - two streams: attention on the compute stream, selection select_ahead
//    layers in front of it;
//  - dependent queries: per request group, append, selection, recall and
//    attention of layer after layer on the group's stream, the groups' recalls
//    taking turns on the copy stream.
// With the fused form (pi_pool_set_fused) the selection, plan and gather of a
// layer (or a request group's share of it) are one launch on the copy stream.
// With the UVA gather arm no step needs the host.
#include <algorithm>
#include <cstring>
#include <utility>
#include <vector>

#include "pi_internal.cuh"

pi_status pi_recall_impl(pi_pool* p, int layer, const int* sel, const int* nsel, int method, int* table,
                         pi_recall_stats* stats, cudaStream_t st);

// event pair of (layer, request group, kind) for the step being recorded, or nullptr
static cudaEvent_t* tev_of(pi_pool* p, int l, int kind, int grp = 0) {
  if (p->timing_used >= p->timing_steps || grp >= p->timing_groups) return nullptr;
  return &p->tev[((((size_t)p->timing_used * p->L + l) * p->timing_groups + grp) * PI_K_KINDS + kind) * 2];
}

#define PI_TIMED(l, kind, stream, launch_expr) PI_TIMED_G(l, 0, kind, stream, launch_expr)
#define PI_TIMED_G(l, grp, kind, stream, launch_expr)              \
  do {                                                             \
    cudaEvent_t* _ev = tev_of(p, (l), (kind), (grp));              \
    if (_ev) PI_CUDA_TRY(cudaEventRecord(_ev[0], (stream)));       \
    PI_CUDA_TRY(launch_expr);                                      \
    if (_ev) PI_CUDA_TRY(cudaEventRecord(_ev[1], (stream)));       \
  } while (0)

cudaError_t pi_launch_plan(pi_pool* p, int layer, const int* sel, const int* nsel, int* table, cudaStream_t s);

static pi_status step_impl(pi_pool* p, const uint8_t* q_all, const uint8_t* k_new_all, const uint8_t* v_new_all,
                           const int* k_budget, int method, uint8_t* out_all, float* lse_all, cudaStream_t cs,
                           cudaStream_t ys, pi_step_stats* stats) {
  const size_t q_bytes = (size_t)p->R * p->Hq * p->D * 2;
  const size_t kv_bytes = (size_t)p->R * p->Hkv * p->D * 2;
  const size_t RU = (size_t)p->R * p->U;
  const bool append = (k_new_all != nullptr);
  if (append)
    for (int l = 0; l < p->L; l++)
      for (int r = 0; r < p->R; r++)
        if ((long long)p->ntok_h[(size_t)r * p->L + l] + 1 > (long long)p->max_blocks * p->B) return PI_ERR_INVALID;
  if (stats) {
    memset(stats, 0, sizeof(*stats));
    PI_CUDA_TRY(cudaMemsetAsync(p->recall_counts, 0, sizeof(long long) * 4 * p->L, ys));
  }
  // the copy stream must not run ahead of work the caller queued on the compute stream
  PI_CUDA_TRY(cudaEventRecord(p->ev_start, cs));
  PI_CUDA_TRY(cudaStreamWaitEvent(ys, p->ev_start, 0));

  auto sel_of = [&](int l) { return p->step_sel + (size_t)l * RU * p->cap; };
  auto nsel_of = [&](int l) { return p->step_nsel + (size_t)l * RU; };
  auto tab_of = [&](int l) { return p->step_table + (size_t)l * RU * p->cap; };
  // UVA arm: the plan runs in the selection kernel's last CTA and the gather
  // writes the new tokens through to the host store, so the copy stream carries
  // only the gather and the compute stream never waits on host-memory writes.
  const bool uva = (method == PI_RECALL_UVA);
  // fused: selection, plan and gather of a layer run as one launch on the copy
  // stream (the compute stream keeps only the append)
  const bool fused = uva && p->fused_on;
  // UVA arm, separate selection: the selection launch appends the new tokens
  // itself (its leader CTAs), so the compute stream's chain starts with it
  const bool fold = append && uva && !fused;
  auto select = [&](int l) -> pi_status {
    if (append && !fold)
      PI_TIMED(l, PI_K_APPEND, cs,
               pi_launch_append(p, l, k_new_all + (size_t)l * kv_bytes, v_new_all + (size_t)l * kv_bytes, cs, !uva));
    if (append)
      for (int r = 0; r < p->R; r++) p->ntok_h[(size_t)r * p->L + l] += 1;
    if (!fused)
      PI_TIMED(l, PI_K_SELECT, cs,
               pi_launch_select(p, l, q_all + (size_t)l * q_bytes, k_budget + (size_t)l * p->R, sel_of(l), nsel_of(l),
                                cs, uva ? tab_of(l) : nullptr, -1, 0, -1,
                                fold ? k_new_all + (size_t)l * kv_bytes : nullptr,
                                fold ? v_new_all + (size_t)l * kv_bytes : nullptr, false));
    PI_CUDA_TRY(cudaEventRecord(p->ev_sel[l], cs));
    return PI_OK;
  };

  // with two copy streams the UVA gathers of odd layers run on the pool's second
  // one, so a gather's start overlaps the previous gather's tail
  const bool two_copies = uva && p->copy2_on;
  if (two_copies) PI_CUDA_TRY(cudaStreamWaitEvent(p->copy2, p->ev_start, 0));
  auto recall_layer = [&](int l) -> pi_status {
    cudaStream_t rs = (two_copies && (l & 1)) ? p->copy2 : ys;
    PI_CUDA_TRY(cudaStreamWaitEvent(rs, p->ev_sel[l], 0));
    if (uva) {
      p->recall_calls++;
      if (p->fault_recall_at > 0 && p->recall_calls == p->fault_recall_at) return PI_ERR_FAULT_INJECTED;
      const uint8_t* kn = append ? k_new_all + (size_t)l * kv_bytes : nullptr;
      const uint8_t* vn = append ? v_new_all + (size_t)l * kv_bytes : nullptr;
      if (fused)
        PI_TIMED(l, PI_K_GATHER, rs,
                 pi_launch_select_gather(p, l, q_all + (size_t)l * q_bytes, k_budget + (size_t)l * p->R, sel_of(l),
                                         nsel_of(l), tab_of(l), kn, vn, rs));
      else
        PI_TIMED(l, PI_K_GATHER, rs, pi_launch_gather(p, l, nullptr, true, true, rs, kn, vn, 0, -1, two_copies));
    } else {
      pi_status s2 = pi_recall_impl(p, l, sel_of(l), nsel_of(l), method, tab_of(l), nullptr, rs);
      if (s2 != PI_OK) return s2;
    }
    PI_CUDA_TRY(cudaEventRecord(p->ev_rec[l], rs));
    return PI_OK;
  };
  auto attend_layer = [&](int l, cudaStream_t as) -> pi_status {
    PI_CUDA_TRY(cudaStreamWaitEvent(as, p->ev_rec[l], 0));
    PI_TIMED(l, PI_K_ATTENTION, as,
             pi_launch_attention(p, l, q_all + (size_t)l * q_bytes, sel_of(l), tab_of(l), nsel_of(l),
                                 out_all + (size_t)l * q_bytes, lse_all ? lse_all + (size_t)l * p->R * p->Hq : nullptr,
                                 nullptr, as, 0, -1, false));
    return PI_OK;
  };
  pi_status st = PI_OK;
  if (p->sched_dependent) {
    // Interruptible layer-wise scheduling ("PulseInfer Guide", section
    // "Interruptible Layer-Wise Scheduling"): a request's query of layer l+1
    // comes out of its layer l, so each request group's chain runs append,
    // selection (+ plan), recall, attention layer after layer on its own
    // stream; the copy stream takes the groups' recalls in turn, so one group's
    // recall of layer l streams while the others compute.
    if (!uva) return PI_ERR_INVALID;
    const int M = p->sched_groups;
    cudaStream_t gs[8];
    int r0[8], nr[8];
    for (int g = 0; g < M; g++) {
      r0[g] = (int)((long long)g * p->R / M);
      nr[g] = (int)((long long)(g + 1) * p->R / M) - r0[g];
      gs[g] = (g == 0) ? cs : p->grp_stream[g];
      if (g > 0) PI_CUDA_TRY(cudaStreamWaitEvent(gs[g], p->ev_start, 0));
    }
    for (int l = 0; l < p->L; l++)
      for (int g = 0; g < M; g++) {
        cudaStream_t s = gs[g];
        cudaEvent_t* ev = &p->grp_ev[((size_t)l * 8 + g) * 2];
        if (append) {
          PI_TIMED_G(l, g, PI_K_APPEND, s,
                     pi_launch_append(p, l, k_new_all + (size_t)l * kv_bytes, v_new_all + (size_t)l * kv_bytes, s,
                                      false, r0[g], nr[g]));
          for (int r = r0[g]; r < r0[g] + nr[g]; r++) p->ntok_h[(size_t)r * p->L + l] += 1;
        }
        p->recall_calls++;
        if (p->fault_recall_at > 0 && p->recall_calls == p->fault_recall_at) return PI_ERR_FAULT_INJECTED;
        const uint8_t* kn = append ? k_new_all + (size_t)l * kv_bytes : nullptr;
        const uint8_t* vn = append ? v_new_all + (size_t)l * kv_bytes : nullptr;
        if (fused) {
          // the fused launch stays on the group's stream: the groups' launches
          // share the link instead of taking turns on the copy stream
          PI_TIMED_G(l, g, PI_K_GATHER, s,
                     pi_launch_select_gather(p, l, q_all + (size_t)l * q_bytes, k_budget + (size_t)l * p->R,
                                             sel_of(l), nsel_of(l), tab_of(l), kn, vn, s, r0[g], nr[g]));
        } else {
          PI_TIMED_G(l, g, PI_K_SELECT, s,
                     pi_launch_select(p, l, q_all + (size_t)l * q_bytes, k_budget + (size_t)l * p->R, sel_of(l),
                                      nsel_of(l), s, tab_of(l), -1, r0[g], nr[g], nullptr, nullptr, false));
          PI_CUDA_TRY(cudaEventRecord(ev[0], s));
          PI_CUDA_TRY(cudaStreamWaitEvent(ys, ev[0], 0));
          PI_TIMED_G(l, g, PI_K_GATHER, ys, pi_launch_gather(p, l, nullptr, true, true, ys, kn, vn, r0[g], nr[g]));
          PI_CUDA_TRY(cudaEventRecord(ev[1], ys));
          PI_CUDA_TRY(cudaStreamWaitEvent(s, ev[1], 0));
        }
        PI_TIMED_G(l, g, PI_K_ATTENTION, s,
                   pi_launch_attention(p, l, q_all + (size_t)l * q_bytes, sel_of(l), tab_of(l), nsel_of(l),
                                       out_all + (size_t)l * q_bytes,
                                       lse_all ? lse_all + (size_t)l * p->R * p->Hq : nullptr, nullptr, s, r0[g],
                                       nr[g], false));
      }
    // the caller's compute stream completes after every group's last attention
    for (int g = 1; g < M; g++) {
      PI_CUDA_TRY(cudaEventRecord(p->grp_done[g], gs[g]));
      PI_CUDA_TRY(cudaStreamWaitEvent(cs, p->grp_done[g], 0));
    }
  } else if (p->attn_stream_on) {
    // three streams: compute runs append + select, copy runs the gather, the
    // pool's own stream runs attention. append(l) of this step waits for
    // attention(l) of the previous step (which reads the token count, selection
    // and table this step overwrites); nothing else orders the layers, so
    // selection runs ahead and consecutive steps overlap.
    cudaStream_t as = p->attn_stream;
    PI_CUDA_TRY(cudaStreamWaitEvent(as, p->ev_start, 0));
    for (int l = 0; l < p->L; l++) {
      PI_CUDA_TRY(cudaStreamWaitEvent(cs, p->ev_att[l], 0));
      st = select(l);
      if (st != PI_OK) return st;
      st = recall_layer(l);
      if (st != PI_OK) return st;
      st = attend_layer(l, as);
      if (st != PI_OK) return st;
      PI_CUDA_TRY(cudaEventRecord(p->ev_att[l], as));
    }
    // the caller's compute stream completes after every layer's attention
    PI_CUDA_TRY(cudaStreamWaitEvent(cs, p->ev_att[p->L - 1], 0));
  } else {
    // selections run `ahead` layers in front of attention (0: every layer first).
    // Any depth gives the same results: a layer's plan reads only maps committed by
    // the previous step's gather of that layer, which the compute stream has
    // already waited for; deeper lookahead only keeps the copy stream fed.
    const int ahead = (p->select_ahead <= 0 || p->select_ahead > p->L) ? p->L : p->select_ahead;
    int next_sel = 0;
    auto select_upto = [&](int upto) -> pi_status {
      for (; next_sel <= upto && next_sel < p->L; next_sel++) {
        pi_status s2 = select(next_sel);
        if (s2 != PI_OK) return s2;
      }
      return PI_OK;
    };
    st = select_upto(ahead - 1);
    if (st != PI_OK) return st;
    for (int l = 0; l < p->L; l++) {
      st = recall_layer(l);
      if (st != PI_OK) return st;
      st = select_upto(l + ahead);
      if (st != PI_OK) return st;
      st = attend_layer(l, cs);
      if (st != PI_OK) return st;
    }
  }
  if (p->timing_used < p->timing_steps) p->timing_used++;
  if (stats) {
    std::vector<long long> c((size_t)4 * p->L);
    PI_CUDA_TRY(cudaStreamSynchronize(cs));
    PI_CUDA_TRY(cudaStreamSynchronize(ys));
    PI_CUDA_TRY(cudaStreamSynchronize(p->attn_stream));
    for (int g = 1; g < 8; g++)
      if (p->grp_stream[g]) PI_CUDA_TRY(cudaStreamSynchronize(p->grp_stream[g]));
    if (p->copy2) PI_CUDA_TRY(cudaStreamSynchronize(p->copy2));
    PI_CUDA_TRY(cudaMemcpy(c.data(), p->recall_counts, sizeof(long long) * 4 * p->L, cudaMemcpyDeviceToHost));
    std::vector<int> ns((size_t)p->L * RU);
    PI_CUDA_TRY(cudaMemcpy(ns.data(), p->step_nsel, sizeof(int) * ns.size(), cudaMemcpyDeviceToHost));
    for (int l = 0; l < p->L; l++) {
      stats->recall.fragments += c[(size_t)l * 4 + 0];
      stats->recall.hits += c[(size_t)l * 4 + 1];
    }
    for (int v : ns) stats->selected += v;
    stats->recall.bytes = stats->recall.fragments * (long long)p->copy_bytes;
    stats->recall.runs = stats->recall.fragments;
  }
  return PI_OK;
}

extern "C" pi_status pi_decode_step(pi_pool* p, const void* q_all, const void* k_new_all, const void* v_new_all,
                                    const int* k_budget, int method, void* out_all, float* lse_all, pi_stream compute,
                                    pi_stream copy, pi_step_stats* stats) {
  if (!p || !q_all || !k_budget || !out_all) return PI_ERR_INVALID;
  if ((k_new_all == nullptr) != (v_new_all == nullptr)) return PI_ERR_INVALID;
  if (method != PI_RECALL_UVA && method != PI_RECALL_MEMCPY && method != PI_RECALL_STAGED) return PI_ERR_INVALID;
  if (reinterpret_cast<uintptr_t>(q_all) & 3) return PI_ERR_INVALID;
  if (k_new_all && ((reinterpret_cast<uintptr_t>(k_new_all) | reinterpret_cast<uintptr_t>(v_new_all)) & 15))
    return PI_ERR_INVALID;
  return step_impl(p, (const uint8_t*)q_all, (const uint8_t*)k_new_all, (const uint8_t*)v_new_all, k_budget, method,
                   (uint8_t*)out_all, lse_all, reinterpret_cast<cudaStream_t>(compute),
                   reinterpret_cast<cudaStream_t>(copy), stats);
}

extern "C" pi_status pi_decode_step_host(pi_pool* p, const void* q_all, const void* k_new_all, const void* v_new_all,
                                         const int* k_budget, int method, void* out_all, float* lse_all,
                                         pi_stream compute, pi_stream copy) {
  if (!p || !q_all || !k_budget || !out_all) return PI_ERR_INVALID;
  if ((k_new_all == nullptr) != (v_new_all == nullptr)) return PI_ERR_INVALID;
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(compute);
  const size_t q_total = (size_t)p->L * p->R * p->Hq * p->D * 2;
  const size_t kv_total = (size_t)p->L * p->R * p->Hkv * p->D * 2;
  const size_t b_total = (size_t)p->L * p->R * sizeof(int);
  uint8_t* dq = p->step_in;
  uint8_t* dk = dq + q_total;
  uint8_t* dv = dk + kv_total;
  int* db = reinterpret_cast<int*>(dv + kv_total);
  uint8_t* dout = p->step_out;
  float* dlse = reinterpret_cast<float*>(dout + q_total);
  PI_CUDA_TRY(cudaMemcpyAsync(dq, q_all, q_total, cudaMemcpyHostToDevice, cs));
  if (k_new_all) {
    PI_CUDA_TRY(cudaMemcpyAsync(dk, k_new_all, kv_total, cudaMemcpyHostToDevice, cs));
    PI_CUDA_TRY(cudaMemcpyAsync(dv, v_new_all, kv_total, cudaMemcpyHostToDevice, cs));
  }
  PI_CUDA_TRY(cudaMemcpyAsync(db, k_budget, b_total, cudaMemcpyHostToDevice, cs));
  pi_status st = step_impl(p, dq, k_new_all ? dk : nullptr, k_new_all ? dv : nullptr, db, method, dout,
                           lse_all ? dlse : nullptr, cs, reinterpret_cast<cudaStream_t>(copy), nullptr);
  if (st != PI_OK) return st;
  PI_CUDA_TRY(cudaMemcpyAsync(out_all, dout, q_total, cudaMemcpyDeviceToHost, cs));
  if (lse_all)
    PI_CUDA_TRY(cudaMemcpyAsync(lse_all, dlse, (size_t)p->L * p->R * p->Hq * sizeof(float), cudaMemcpyDeviceToHost, cs));
  PI_CUDA_TRY(cudaStreamSynchronize(cs));
  return PI_OK;
}

extern "C" pi_status pi_pool_set_timing(pi_pool* p, int max_steps) {
  if (!p || max_steps < 0) return PI_ERR_INVALID;
  PI_CUDA_TRY(cudaDeviceSynchronize());
  for (auto e : p->tev) cudaEventDestroy(e);
  p->tev.clear();
  p->timing_steps = 0;
  p->timing_used = 0;
  if (max_steps == 0) return PI_OK;
  p->timing_groups = p->sched_dependent ? p->sched_groups : 1;
  const size_t n = (size_t)max_steps * p->L * p->timing_groups * PI_K_KINDS * 2;
  p->tev.resize(n, nullptr);
  for (size_t i = 0; i < n; i++) PI_CUDA_TRY(cudaEventCreate(&p->tev[i]));
  p->timing_steps = max_steps;
  return PI_OK;
}

extern "C" pi_status pi_pool_get_timing(pi_pool* p, pi_kernel_timing* out) {
  if (!p || !out) return PI_ERR_INVALID;
  PI_CUDA_TRY(cudaDeviceSynchronize());
  for (int k = 0; k < PI_K_KINDS; k++) out[k] = pi_kernel_timing{0, 0.0, 0.0};
  std::vector<std::pair<double, double>> iv[PI_K_KINDS];
  cudaEvent_t ref = nullptr;  // the first recorded start: the origin of every interval
  for (int s = 0; s < p->timing_used; s++)
    for (int lg = 0; lg < p->L * p->timing_groups; lg++)
      for (int k = 0; k < PI_K_KINDS; k++) {
        cudaEvent_t* ev = &p->tev[(((size_t)s * p->L * p->timing_groups + lg) * PI_K_KINDS + k) * 2];
        float ms = 0.0f, t0 = 0.0f;
        // a kind that did not run in this step leaves its pair unrecorded
        if (cudaEventQuery(ev[1]) != cudaSuccess) { cudaGetLastError(); continue; }
        if (cudaEventElapsedTime(&ms, ev[0], ev[1]) != cudaSuccess) { cudaGetLastError(); continue; }
        if (!ref) ref = ev[0];
        if (cudaEventElapsedTime(&t0, ref, ev[0]) != cudaSuccess) { cudaGetLastError(); continue; }
        out[k].launches++;
        out[k].total_ms += ms;
        iv[k].push_back({(double)t0, (double)t0 + ms});
      }
  for (int k = 0; k < PI_K_KINDS; k++) {
    std::sort(iv[k].begin(), iv[k].end());
    double end = -1e300;
    for (const auto& x : iv[k]) {
      const double a = std::max(x.first, end);
      if (x.second > a) out[k].busy_ms += x.second - a;
      end = std::max(end, x.second);
    }
  }
  p->timing_used = 0;
  return PI_OK;
}

extern "C" pi_status pi_pool_set_pipeline(pi_pool* p, int select_ahead, int attention_stream) {
  if (!p || select_ahead < 0) return PI_ERR_INVALID;
  PI_CUDA_TRY(cudaDeviceSynchronize());  // no step of the old mode may still run
  p->select_ahead = select_ahead;
  p->attn_stream_on = attention_stream != 0;
  return PI_OK;
}

extern "C" pi_status pi_pool_set_fused(pi_pool* p, int on, int ctas) {
  if (!p || (on != 0 && on != 1) || ctas < 0) return PI_ERR_INVALID;
  PI_CUDA_TRY(cudaDeviceSynchronize());
  p->fused_on = (on == 1);
  p->fused_ctas = ctas;
  // fresh timing events: a kind the new form no longer launches keeps no old times
  if (p->timing_steps > 0) return pi_pool_set_timing(p, p->timing_steps);
  return PI_OK;
}

extern "C" pi_status pi_pool_set_copy_streams(pi_pool* p, int n) {
  if (!p || (n != 1 && n != 2)) return PI_ERR_INVALID;
  PI_CUDA_TRY(cudaDeviceSynchronize());
  if (n == 2 && !p->copy2) PI_CUDA_TRY(cudaStreamCreateWithFlags(&p->copy2, cudaStreamNonBlocking));
  p->copy2_on = (n == 2);
  return PI_OK;
}

extern "C" pi_status pi_pool_set_schedule(pi_pool* p, int dependent, int groups) {
  if (!p || (dependent != 0 && dependent != 1) || groups < 1 || groups > 8 || groups > p->R) return PI_ERR_INVALID;
  PI_CUDA_TRY(cudaDeviceSynchronize());  // no step of the old schedule may still run
  if (dependent) {
    if (p->grp_ev.empty()) {
      p->grp_ev.resize((size_t)p->L * 8 * 2, nullptr);
      for (auto& e : p->grp_ev) PI_CUDA_TRY(cudaEventCreateWithFlags(&e, cudaEventDisableTiming));
    }
    for (int g = 1; g < groups; g++) {
      if (!p->grp_stream[g]) PI_CUDA_TRY(cudaStreamCreateWithFlags(&p->grp_stream[g], cudaStreamNonBlocking));
      if (!p->grp_done[g]) PI_CUDA_TRY(cudaEventCreateWithFlags(&p->grp_done[g], cudaEventDisableTiming));
    }
  }
  p->sched_dependent = dependent;
  p->sched_groups = dependent ? groups : 1;
  return PI_OK;
}

extern "C" pi_status pi_pool_set_attention_cluster(pi_pool* p, int on) {
  if (!p || (on != 0 && on != 1)) return PI_ERR_INVALID;
  p->attn_cluster = on != 0;
  return PI_OK;
}

extern "C" pi_status pi_pool_set_selection(pi_pool* p, int cluster, int ctas_per_unit) {
  if (!p || (cluster != 0 && cluster != 1) || ctas_per_unit < 0 || ctas_per_unit > 16) return PI_ERR_INVALID;
  p->select_cluster_on = cluster != 0;
  p->select_cluster_ctas = ctas_per_unit;
  return PI_OK;
}

extern "C" pi_status pi_pool_set_attention(pi_pool* p, int splits) {
  if (!p || splits < 0) return PI_ERR_INVALID;
  p->attn_splits = splits;
  return PI_OK;
}
