// The LongFlow fused decode step (attention + zero-cost score + in-place
// eviction) and the prefill kernel, for sm_103a.
//
// One launch handles one layer for every (sequence, KV head) unit.  A
// thread-block cluster of C CTAs owns one unit; CTA `rank` streams the slots
// [rank*chunk, (rank+1)*chunk) of that unit:
//
//   phase A  K tiles (+ ||v||_1 and positions) arrive through a ring of
//            1-D bulk TMA copies into shared memory; each warp computes the
//            G query heads' logits of its slots and keeps them in shared
//            memory (they are needed again for the exact score);
//   softmax  the CTA's local max m_h and p_{h,i} = 2^(s_{h,i} - m_h), l_h;
//   phase B  V tiles arrive through the same ring; o_h += p_{h,i} v_i;
//   combine  the cluster exchanges (m_h, l_h) and the partial outputs through
//            distributed shared memory, adds the new token as one more key,
//            writes out_h, and scores every unprotected slot exactly:
//            score_i = ||v_i||_1 * sum_h p_{h,i} 2^(m_h - M_h) / L_h;
//   evict    the leader CTA takes the lowest (score, slot) over the cluster
//            and overwrites that slot with the new token in place.
//
// Logits are kept pre-multiplied by log2(e) so every exponential is an exp2.
// No global scratch is used, no CTA waits on another CTA except through the
// hardware cluster barrier, and every mbarrier wait is bounded.
#pragma once

#include <cooperative_groups.h>
#include <limits.h>
#include <math.h>

#include "lf_device.cuh"
#include "longflow.h"

namespace lf {
namespace cg = cooperative_groups;

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kTile = 32;        // slots per staged tile
constexpr int kMaxCluster = 16;
constexpr int kMaxStages = 16;
constexpr int kMaxGroup = 8;

struct DecodeArgs {
  const void* q;       // [batch][q_heads][D]
  const void* k_new;   // [batch][kv_heads][D]
  const void* v_new;   // [batch][kv_heads][D]
  void* out;           // [batch][q_heads][D]
  int32_t* evicted;    // [batch][kv_heads]
  void* K;             // this layer's [batch][kv_heads][slot_stride][D]
  void* V;
  float* vnorm;        // this layer's [batch][kv_heads][slot_stride]
  int32_t* pos;
  int32_t* count;      // this layer's [batch][kv_heads]
  int32_t* next_pos;
  const int32_t* budget;  // [batch]
  int32_t* err;
  float* acc;          // H2O: this layer's attention mass per slot (as vnorm), else null
  int32_t* pending;    // deferred: this layer's chosen slot per unit (as count), else null
  float* lw_score;     // layer scope: one layer's per-slot scores (as vnorm), else null
  int32_t* lw_req;     // layer scope: [batch][kv_heads] 1 = scores written this step
  float* lw_anew;      // layer scope: [batch][kv_heads] the new token's attention mass
  int batch, kv_heads, q_heads, slot_stride, capacity, window, chunk, stages, evict;
  int score, norm, sinks, deferred, scope;  // the policy (lf_config)
  int strict;          // a step on a full slab is an error (R-KV: compress first)
  float scale_log2;    // log2(e) / sqrt(D)
};

// ---- eviction rules shared by every decode kernel ------------------------------
//
// Per unit, from its occupancy n, next position p, budget and (deferred) the
// slot chosen at the previous step:
//   same step   attend over the n cached slots + the new token; once n >= budget
//               choose among slots with sinks <= pos < p - W and write the new
//               token there, else append at slot n;
//   deferred    the new token takes slot n while n < budget, else the slot chosen
//               before (`excl`: its old token is neither attended nor a
//               candidate); once the buffer is full after the write, choose among
//               slots with sinks <= pos < p + 1 - W the slot the next token takes.
struct UnitRule {
  bool full;      // n >= budget with eviction on: this step replaces a token
  bool choosing;  // a victim is chosen this step
  int plim;       // a slot is a candidate iff sinks <= pos < plim (and not excl)
  int excl;       // slot whose old token is dropped before attention (deferred), or -1
};

__device__ __forceinline__ UnitRule unit_rule(const DecodeArgs& a, int n, int p, int pend,
                                              int bud, bool state_ok) {
  UnitRule r;
  r.full = state_ok && a.evict && n >= bud;
  if (a.deferred && a.evict) {
    r.choosing = state_ok && n + 1 >= bud;
    r.plim = p + 1 - a.window;
    r.excl = r.full ? pend : -1;
  } else {
    r.choosing = r.full;
    r.plim = p - a.window;
    r.excl = -1;
  }
  return r;
}

// Candidate weights carry the candidate flag in the sign bit, so that a slot
// that is not a candidate still carries its value (the H2O accumulator must be
// written back for every slot, and it may be +0).
__device__ __forceinline__ float flag_protected(float x) {
  return __int_as_float(__float_as_int(x) | (int)0x80000000);
}
__device__ __forceinline__ bool is_candidate(float w) { return __float_as_int(w) >= 0; }

// ||v|| of one stored value row, by one warp (fp32, lane-strided then a tree).
template <typename T, int D>
__device__ __forceinline__ float warp_value_norm(const T* v, int norm, int lane) {
  float s = 0.f;
  if (norm == 2) {
    for (int e = lane; e < D; e += 32) {
      const float x = to_f32(v[e]);
      s = fmaf(x, x, s);
    }
    return sqrtf(warp_sum(s));
  }
  for (int e = lane; e < D; e += 32) s += fabsf(to_f32(v[e]));
  return warp_sum(s);
}

// The unit leader's decision once the cluster's lowest (score, slot) is known
// (`fi`, INT_MAX if none): the slot the new token takes (-1: none) and the slot
// reported as evicted, with the unit's bookkeeping written to global memory
// (count, next position, the deferred choice, the layer-scope request).
struct LeaderOut {
  int slot;
  int evicted;
};

__device__ __forceinline__ LeaderOut leader_decide(const DecodeArgs& a, int unit, int n, int p,
                                                   int pend, int bud, bool state_ok,
                                                   bool any_fail, const UnitRule& r, int fi,
                                                   float anew) {
  const bool layer = a.evict && a.scope == LF_SCOPE_LAYER;
  const bool deferred = a.evict && a.deferred;
  int chosen = -1;
  if (r.choosing && !layer) {
    if (fi != INT_MAX) chosen = fi;
    else if (!any_fail) atomicOr(a.err, LF_DEVERR_STATE);  // no candidate
  }
  int slot = -1, evicted = -1;
  if (deferred) {
    slot = r.full ? pend : n;
    evicted = r.full ? pend : -1;
    if (r.full && pend < 0) {  // a full buffer without a chosen slot
      if (!any_fail) atomicOr(a.err, LF_DEVERR_STATE);
      slot = evicted = -1;
    }
  } else if (r.full) {
    slot = evicted = layer ? -1 : chosen;  // layer scope: the selection kernel writes
  } else {
    slot = (n < (a.evict ? bud : a.capacity)) ? n : -1;
    if (slot < 0 && a.strict && state_ok && !any_fail) atomicOr(a.err, LF_DEVERR_STATE);
  }
  if (!state_ok) atomicOr(a.err, LF_DEVERR_STATE);
  if (any_fail || !state_ok) slot = evicted = -1;
  a.evicted[unit] = evicted;
  if (state_ok && !any_fail) {
    if (!r.full && slot >= 0) a.count[unit] = n + 1;
    a.next_pos[unit] = p + 1;
    if (deferred && !layer && r.choosing) a.pending[unit] = chosen;
    if (layer) {
      a.lw_req[unit] = r.choosing ? n + 1 : 0;  // slots scored, + 1
      a.lw_anew[unit] = anew;
    }
  }
  return {slot, evicted};
}

// In-place overwrite of one slot (guide, "Static Memory Pre-Allocation and
// In-Place Eviction", step 3): K, V, ||v|| (fp32, from the stored value), the
// position and, with the H2O score, the new token's own attention mass.  Called
// by `nthreads` threads numbered `tid`; threads 0..31 form one warp.
template <typename T, int D>
__device__ __forceinline__ void write_slot(const DecodeArgs& a, size_t ubase, int slot,
                                           const T* kn, const T* vn, int p, float anew, int tid,
                                           int nthreads) {
  T* Kd = reinterpret_cast<T*>(a.K) + (ubase + slot) * D;
  T* Vd = reinterpret_cast<T*>(a.V) + (ubase + slot) * D;
  for (int e = tid; e < D; e += nthreads) {
    Kd[e] = kn[e];
    Vd[e] = vn[e];
  }
  if (tid < 32) {
    const float nv = warp_value_norm<T, D>(vn, a.norm, tid);
    if (tid == 0) {
      a.vnorm[ubase + slot] = nv;
      a.pos[ubase + slot] = p;
      if (a.acc) a.acc[ubase + slot] = anew;
    }
  }
}

// Shared-memory plan, shared by the host (launch size) and the kernel.
template <typename T, int D, int G>
struct DecodePlan {
  static constexpr int kStageData = kTile * D * (int)sizeof(T);
  static constexpr int kStageBytes = kStageData + 2 * kTile * 4;  // + ||v||_1, pos
  static constexpr int kPvTpr = D / 4;               // threads per V row (4 elements each)
  static constexpr int kPvGroups = kThreads / kPvTpr;
  static constexpr int kPvBufBytes = kPvGroups * G * D * 4;
  // fixed header
  static constexpr int kOffBars = 0;                  // kMaxStages mbarriers
  static constexpr int kOffStats = 128;               // 6 x kMaxGroup floats
  static constexpr int kOffBest = kOffStats + 6 * kMaxGroup * 4;  // kMaxCluster (score, slot, flag)
  static constexpr int kOffRed = kOffBest + 3 * kMaxCluster * 4;  // kWarps x kMaxGroup floats + ints
  static constexpr int kOffDecision = kOffRed + 2 * kWarps * kMaxGroup * 4;
  static constexpr int kHeader = 2048;
  static_assert(kOffDecision + 16 <= kHeader, "header overflow");
  static constexpr int kOffOpart = kHeader;           // G x D floats
  static constexpr int kOffRing = (kOffOpart + G * D * 4 + 127) / 128 * 128;

  __host__ __device__ static constexpr int ring_bytes(int stages) {
    return ((stages * kStageBytes > kPvBufBytes ? stages * kStageBytes : kPvBufBytes) + 127) / 128 *
           128;
  }
  __host__ __device__ static constexpr int off_logits(int stages) {
    return kOffRing + ring_bytes(stages);
  }
  __host__ __device__ static constexpr int off_weights(int stages, int chunk) {
    return off_logits(stages) + chunk * G * 4;
  }
  __host__ __device__ static constexpr int smem_bytes(int stages, int chunk) {
    return off_weights(stages, chunk) + chunk * 4;
  }
};

// Shared-memory pieces the cluster combine reads and writes.
struct CombineSmem {
  float* m_loc;   // [kMaxGroup] this CTA's max logit per head (log2 domain)
  float* l_loc;   // [kMaxGroup] sum of 2^(s - m_loc) over this CTA's slots
  float* s_new;   // [kMaxGroup] the new token's logit per head
  float* cmul;    // [kMaxGroup] 2^(m_loc - M) / L per head
  float* m_glb;   // [kMaxGroup] M: max over the cluster and the new token
  float* l_glb;   // [kMaxGroup] L: softmax denominator over the unit
  float* best_s;  // [kMaxCluster] per-rank lowest score (leader's copy is filled)
  int* best_i;    // [kMaxCluster] per-rank victim slot
  int* fail_in;   // [kMaxCluster] per-rank abort flags
  float* red;     // [kWarps * kMaxGroup] reduction scratch
  int* red_i;     // [kWarps * kMaxGroup]
  int* decision;  // [2] slot written, victim
  float* o_part;  // [G][D] this CTA's unnormalised output, relative to m_loc
  const float* p; // [rows][G] 2^(s - m_loc) of this CTA's slots
  const float* w; // [rows] ||v|| (H2O: the accumulator) of each slot, sign bit set
                  // when the slot is not a candidate
};

// Cluster-wide combine of one unit: merge (m, l) and the partial outputs over
// DSMEM, add the new token as one more key, write out, score every candidate
// exactly, and let the leader CTA overwrite the lowest-scored slot.  Called by
// all NT threads of every CTA of the cluster.
template <typename T, int D, int G, int NT>
__device__ __forceinline__ void combine_and_evict(
    const DecodeArgs& a, cg::cluster_group& cluster, const CombineSmem& sm, int C, int rank, int b,
    int g, int unit, size_t ubase, int n, int p, int pend, int bud, bool state_ok,
    const UnitRule& rl, int s0, int rows, bool aborted, const T* qg, const T* kn, const T* vn) {
  constexpr int NW = NT / 32;
  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int warp = tid >> 5;
  // The new token's logits, computed redundantly by every CTA of the cluster.
  for (int h = warp; h < G; h += NW) {
    float s = 0.f;
    for (int e = lane; e < D; e += 32) s = fmaf(to_f32(qg[(size_t)h * D + e]), to_f32(kn[e]), s);
    s = warp_sum(s);
    if (lane == 0) sm.s_new[h] = s * a.scale_log2;
  }
  // #1: every CTA has started (DSMEM may be touched from here on) and its
  // m_loc, l_loc and o_part are visible to the cluster.
  cluster.sync();
  if (tid == 0 && aborted) *cluster.map_shared_rank(&sm.fail_in[rank], 0) = 1;

  if (tid < G) {
    const int h = tid;
    float M = sm.s_new[h];
    for (int r = 0; r < C; ++r) M = fmaxf(M, *cluster.map_shared_rank(&sm.m_loc[h], r));
    float L = exp2f(sm.s_new[h] - M);
    for (int r = 0; r < C; ++r) {
      const float mr = *cluster.map_shared_rank(&sm.m_loc[h], r);
      if (mr != -INFINITY) L += *cluster.map_shared_rank(&sm.l_loc[h], r) * exp2f(mr - M);
    }
    sm.m_glb[h] = M;
    sm.l_glb[h] = L;
    sm.cmul[h] = (sm.m_loc[h] != -INFINITY) ? exp2f(sm.m_loc[h] - M) / L : 0.f;
    if (!(isfinite(M) && isfinite(L) && L > 0.f)) atomicOr(a.err, LF_DEVERR_NONFINITE);
  }
  __syncthreads();

  // Output: the cluster's threads share the G x D elements.
  {
    T* og = reinterpret_cast<T*>(a.out) + ((size_t)b * a.q_heads + (size_t)g * G) * D;
    for (int idx = rank * NT + tid; idx < G * D; idx += C * NT) {
      const int h = idx / D;
      const int e = idx - h * D;
      float acc = exp2f(sm.s_new[h] - sm.m_glb[h]) * to_f32(vn[e]);
      for (int r = 0; r < C; ++r) {
        const float mr = *cluster.map_shared_rank(&sm.m_loc[h], r);
        if (mr != -INFINITY)
          acc += *cluster.map_shared_rank(&sm.o_part[idx], r) * exp2f(mr - sm.m_glb[h]);
      }
      from_f32(acc / sm.l_glb[h], &og[(size_t)h * D + e]);
    }
  }

  // Exact scores of this CTA's slots and the lowest (score, slot) of its
  // candidates.  LongFlow: ||v_i|| sum_h alpha_{h,i}.  H2O: the slot's
  // accumulator plus this step's sum_h alpha_{h,i}, written back for every slot
  // but the dropped one before cluster barrier #2 (the leader overwrites the
  // written slot after it).  Layer scope: every score goes to the scratch for
  // the selection kernel.
  const bool h2o = a.evict && a.score == LF_SCORE_H2O;
  const bool layer = a.evict && a.scope == LF_SCOPE_LAYER;
  float bs = INFINITY;
  int bi = INT_MAX;
  if ((rl.choosing || h2o) && !aborted) {
    float cm[G];
#pragma unroll
    for (int h = 0; h < G; ++h) cm[h] = sm.cmul[h];
    for (int i = tid; i < rows; i += NT) {
      const int slot = s0 + i;
      if (slot == rl.excl) {
        if (layer && rl.choosing) a.lw_score[ubase + slot] = INFINITY;
        continue;
      }
      const float w = sm.w[i];
      const float val = fabsf(w);
      float as = 0.f;
#pragma unroll
      for (int h = 0; h < G; ++h) as = fmaf(sm.p[(size_t)i * G + h], cm[h], as);
      const float sc = h2o ? val + as : val * as;
      if (h2o) a.acc[ubase + slot] = sc;
      if (rl.choosing) {
        if (layer) {
          a.lw_score[ubase + slot] = is_candidate(w) ? sc : INFINITY;
        } else if (is_candidate(w) && better(sc, slot, bs, bi)) {
          bs = sc;
          bi = slot;
        }
      }
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float os = __shfl_xor_sync(0xffffffffu, bs, o);
    const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
    if (better(os, oi, bs, bi)) {
      bs = os;
      bi = oi;
    }
  }
  if (lane == 0) {
    sm.red[warp] = bs;
    sm.red_i[warp] = bi;
  }
  __syncthreads();
  if (tid == 0) {
    for (int w = 1; w < NW; ++w)
      if (better(sm.red[w], sm.red_i[w], bs, bi)) {
        bs = sm.red[w];
        bi = sm.red_i[w];
      }
    *cluster.map_shared_rank(&sm.best_s[rank], 0) = bs;
    *cluster.map_shared_rank(&sm.best_i[rank], 0) = bi;
  }
  cluster.sync();  // #2: all slot reads of the step are done; minima are at the leader
  if (rank != 0) return;

  float anew = 0.f;  // the new token's attention mass (tid 0)
  if (tid == 0) {
    bool any_fail = false;
    for (int r = 0; r < C; ++r) any_fail = any_fail || sm.fail_in[r] != 0;
    float fs = INFINITY;
    int fi = INT_MAX;
    for (int r = 0; r < C; ++r)
      if (better(sm.best_s[r], sm.best_i[r], fs, fi)) {
        fs = sm.best_s[r];
        fi = sm.best_i[r];
      }
#pragma unroll
    for (int h = 0; h < G; ++h) anew += exp2f(sm.s_new[h] - sm.m_glb[h]) / sm.l_glb[h];
    const LeaderOut d = leader_decide(a, unit, n, p, pend, bud, state_ok, any_fail, rl, fi, anew);
    sm.decision[0] = d.slot;
  }
  __syncthreads();
  const int slot = sm.decision[0];
  if (slot >= 0) write_slot<T, D>(a, ubase, slot, kn, vn, p, anew, tid, NT);
}

template <typename T, int D, int G>
__global__ void __launch_bounds__(kThreads, 2) decode_step_simt_kernel(const DecodeArgs a) {
  using P = DecodePlan<T, D, G>;
  constexpr int V = ElemTraits<T>::kPer16B;  // elements per 16-byte chunk
  constexpr int NC = D / V;                  // chunks per row
  constexpr int LPS = NC < 8 ? NC : 8;       // lanes sharing one slot's dot product
  constexpr int CPL = NC / LPS;              // chunks per lane
  constexpr int SPW = 32 / LPS;              // slots per warp pass
  constexpr int SPP = kWarps * SPW;          // slots per CTA pass
  static_assert(NC % LPS == 0 && 32 % LPS == 0, "bad row split");
  static_assert(G <= kWarps && G <= kMaxGroup, "group too large");

  cg::cluster_group cluster = cg::this_cluster();
  const int C = (int)cluster.num_blocks();
  const int rank = (int)cluster.block_rank();
  const int g = blockIdx.y;
  const int b = blockIdx.z;
  const int unit = b * a.kv_heads + g;
  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int warp = tid >> 5;
  const int S = a.stages;

  extern __shared__ __align__(1024) unsigned char smem[];
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + P::kOffBars);
  float* m_loc = reinterpret_cast<float*>(smem + P::kOffStats);
  float* l_loc = m_loc + kMaxGroup;
  float* s_new = l_loc + kMaxGroup;
  float* cmul = s_new + kMaxGroup;
  float* m_glb = cmul + kMaxGroup;
  float* l_glb = m_glb + kMaxGroup;
  float* best_s = reinterpret_cast<float*>(smem + P::kOffBest);
  int* best_i = reinterpret_cast<int*>(best_s + kMaxCluster);
  int* fail_in = best_i + kMaxCluster;
  float* red = reinterpret_cast<float*>(smem + P::kOffRed);
  int* red_i = reinterpret_cast<int*>(red + kWarps * kMaxGroup);
  int* decision = reinterpret_cast<int*>(smem + P::kOffDecision);
  float* o_part = reinterpret_cast<float*>(smem + P::kOffOpart);
  unsigned char* ring = smem + P::kOffRing;
  float* lg = reinterpret_cast<float*>(smem + P::off_logits(S));
  float* wv = reinterpret_cast<float*>(smem + P::off_weights(S, a.chunk));

  const int n = a.count[unit];
  const int p = a.next_pos[unit];
  const int bud = a.budget[b];
  // Read before the leader may update it (after cluster barrier #2).
  const int pend = (a.evict && a.deferred) ? a.pending[unit] : -1;
  const bool state_ok = (n >= 0 && n <= a.capacity && p >= n);
  const UnitRule rl = unit_rule(a, n, p, pend, bud, state_ok);
  const int s0 = rank * a.chunk;
  const int s1 = state_ok ? min(s0 + a.chunk, n) : s0;
  const int rows = max(0, s1 - s0);
  const int ntile = (rows + kTile - 1) / kTile;
  const int total = 2 * ntile;  // K tiles then V tiles through one ring

  const size_t ubase = (size_t)unit * a.slot_stride;
  const T* Ku = reinterpret_cast<const T*>(a.K) + ubase * D;
  const T* Vu = reinterpret_cast<const T*>(a.V) + ubase * D;
  // ||v|| per slot, or the H2O accumulator: the value a candidate is scored from
  const float* vnu = (a.evict && a.score == LF_SCORE_H2O) ? a.acc + ubase : a.vnorm + ubase;
  const int32_t* posu = a.pos + ubase;
  const T* qg = reinterpret_cast<const T*>(a.q) + ((size_t)b * a.q_heads + (size_t)g * G) * D;
  const T* kn = reinterpret_cast<const T*>(a.k_new) + (size_t)unit * D;
  const T* vn = reinterpret_cast<const T*>(a.v_new) + (size_t)unit * D;

  if (tid == 0) {
    for (int s = 0; s < S; ++s) mbar_init(&bars[s], 1);
    fence_mbar_init();
  }
  if (tid < kMaxCluster) {
    best_s[tid] = INFINITY;
    best_i[tid] = INT_MAX;
    fail_in[tid] = 0;
  }
  __syncthreads();

  const uint64_t policy = l2_evict_first_policy();
  auto issue = [&](int t) {
    const int st = t % S;
    const bool isK = t < ntile;
    const int j = isK ? t : t - ntile;
    const int r0 = s0 + j * kTile;
    const int r = min(kTile, s1 - r0);
    unsigned char* dst = ring + (size_t)st * P::kStageBytes;
    const uint32_t data_bytes = (uint32_t)(r * D * (int)sizeof(T));
    // ||v||_1 and pos are 4-byte fields: copy whole 16-byte groups (the slab's
    // slot stride is a multiple of 32, so this stays inside the unit).
    const uint32_t small_bytes = isK ? (uint32_t)(((r + 3) & ~3) * 4) : 0u;
    mbar_arrive_expect_tx(&bars[st], data_bytes + 2u * small_bytes);
    bulk_g2s(dst, (isK ? Ku : Vu) + (size_t)r0 * D, data_bytes, &bars[st], policy);
    if (isK) {
      bulk_g2s(dst + P::kStageData, vnu + r0, small_bytes, &bars[st], policy);
      bulk_g2s(dst + P::kStageData + kTile * 4, posu + r0, small_bytes, &bars[st], policy);
    }
  };
  int issued = 0;
  if (tid == 0) {
    issued = min(S, total);
    for (int t = 0; t < issued; ++t) issue(t);
  }

  // This lane's slice of the group's queries, pre-scaled by log2(e)/sqrt(D).
  const int sub = lane % LPS;
  const int rsl = lane / LPS;
  float qr[G][CPL * V];
#pragma unroll
  for (int h = 0; h < G; ++h)
#pragma unroll
    for (int c = 0; c < CPL; ++c) {
      load16_f32(qg + (size_t)h * D + (sub + LPS * c) * V, &qr[h][c * V]);
#pragma unroll
      for (int v = 0; v < V; ++v) qr[h][c * V + v] *= a.scale_log2;
    }

  const int plim = rl.plim;  // a slot is a candidate iff sinks <= pos < plim (and not excl)
  const int pv_e0 = (tid % P::kPvTpr) * 4;
  const int pv_grp = tid / P::kPvTpr;
  float pv[G][4];
#pragma unroll
  for (int h = 0; h < G; ++h)
#pragma unroll
    for (int v = 0; v < 4; ++v) pv[h][v] = 0.f;

  bool failed = false;
  int t_stop = total;
  for (int t = 0; t < total; ++t) {
    const int st = t % S;
    bool ok = mbar_wait_bounded(&bars[st], (uint32_t)((t / S) & 1));
    ok = __all_sync(0xffffffffu, ok);
    const unsigned char* stage = ring + (size_t)st * P::kStageBytes;
    const bool isK = t < ntile;
    const int j = isK ? t : t - ntile;
    const int off = j * kTile;
    const int r = min(kTile, rows - off);
    if (ok && isK) {
      const T* Kt = reinterpret_cast<const T*>(stage);
#pragma unroll
      for (int ps = 0; ps < kTile; ps += SPP) {
        const int rr = ps + warp * SPW + rsl;
        float acc[G];
#pragma unroll
        for (int h = 0; h < G; ++h) acc[h] = 0.f;
        if (rr < r) {
#pragma unroll
          for (int c = 0; c < CPL; ++c) {
            float x[V];
            load16_f32(Kt + (size_t)rr * D + (sub + LPS * c) * V, x);
#pragma unroll
            for (int h = 0; h < G; ++h)
#pragma unroll
              for (int v = 0; v < V; ++v) acc[h] = fmaf(qr[h][c * V + v], x[v], acc[h]);
          }
        }
#pragma unroll
        for (int o = 1; o < LPS; o <<= 1)
#pragma unroll
          for (int h = 0; h < G; ++h) acc[h] += __shfl_xor_sync(0xffffffffu, acc[h], o);
        if (rr < r) {
#pragma unroll
          for (int h = 0; h < G; ++h)
            if (sub == h % LPS)
              lg[(size_t)(off + rr) * G + h] = (s0 + off + rr == rl.excl) ? -INFINITY : acc[h];
        }
      }
      const float* vn_t = reinterpret_cast<const float*>(stage + P::kStageData);
      const int32_t* pos_t = reinterpret_cast<const int32_t*>(stage + P::kStageData + kTile * 4);
      if (tid < r) {
        const int ps = pos_t[tid];
        const bool cand = (s0 + off + tid != rl.excl) && ps < plim && ps >= a.sinks;
        wv[off + tid] = cand ? vn_t[tid] : flag_protected(vn_t[tid]);
      }
    } else if (ok) {
      const T* Vt = reinterpret_cast<const T*>(stage);
      for (int rr = pv_grp; rr < r; rr += P::kPvGroups) {
        float x[4];
        load4_f32(Vt + (size_t)rr * D + pv_e0, x);
        const float* pp = lg + (size_t)(off + rr) * G;
#pragma unroll
        for (int h = 0; h < G; ++h) {
          const float ph = pp[h];
#pragma unroll
          for (int v = 0; v < 4; ++v) pv[h][v] = fmaf(ph, x[v], pv[h][v]);
        }
      }
    }
    failed = failed || !ok;
    if (__syncthreads_or(failed)) {  // uniform: every thread leaves together
      t_stop = t;
      break;
    }
    if (tid == 0 && t + S < total) {
      issue(t + S);
      issued = t + S + 1;
    }
    if (t == ntile - 1) {
      // Local softmax statistics over this CTA's slots: m_h, p = 2^(s - m_h), l_h.
      float mx[G];
#pragma unroll
      for (int h = 0; h < G; ++h) mx[h] = -INFINITY;
      for (int i = tid; i < rows; i += kThreads)
#pragma unroll
        for (int h = 0; h < G; ++h) mx[h] = fmaxf(mx[h], lg[(size_t)i * G + h]);
#pragma unroll
      for (int h = 0; h < G; ++h) mx[h] = warp_max(mx[h]);
      if (lane == 0)
#pragma unroll
        for (int h = 0; h < G; ++h) red[warp * kMaxGroup + h] = mx[h];
      __syncthreads();
      if (tid < G) {
        float m = -INFINITY;
        for (int w = 0; w < kWarps; ++w) m = fmaxf(m, red[w * kMaxGroup + tid]);
        m_loc[tid] = m;
      }
      __syncthreads();
      float sm[G];
#pragma unroll
      for (int h = 0; h < G; ++h) sm[h] = 0.f;
      for (int i = tid; i < rows; i += kThreads)
#pragma unroll
        for (int h = 0; h < G; ++h) {
          const float x = lg[(size_t)i * G + h];
          const float e = (x == -INFINITY) ? 0.f : exp2f(x - m_loc[h]);  // dropped slot
          lg[(size_t)i * G + h] = e;
          sm[h] += e;
        }
#pragma unroll
      for (int h = 0; h < G; ++h) sm[h] = warp_sum(sm[h]);
      if (lane == 0)
#pragma unroll
        for (int h = 0; h < G; ++h) red[warp * kMaxGroup + h] = sm[h];
      __syncthreads();
      if (tid < G) {
        float s = 0.f;
        for (int w = 0; w < kWarps; ++w) s += red[w * kMaxGroup + tid];
        l_loc[tid] = s;
      }
      __syncthreads();
    }
  }
  const bool aborted = (t_stop < total);
  if (aborted && tid == 0) {
    // Retire every copy still in flight into our shared memory, then report.
    for (int t = t_stop; t < issued; ++t)
      (void)mbar_wait_bounded(&bars[t % S], (uint32_t)((t / S) & 1));
    atomicOr(a.err, LF_DEVERR_TIMEOUT);
  }
  if (rows == 0 || aborted) {
    if (tid < G) {
      m_loc[tid] = -INFINITY;
      l_loc[tid] = 0.f;
    }
#pragma unroll
    for (int h = 0; h < G; ++h)
#pragma unroll
      for (int v = 0; v < 4; ++v) pv[h][v] = 0.f;
  }

  // Reduce the partial outputs of the P.V thread groups (the ring is idle now).
  float* pvbuf = reinterpret_cast<float*>(ring);
  __syncthreads();
#pragma unroll
  for (int h = 0; h < G; ++h)
#pragma unroll
    for (int v = 0; v < 4; ++v) pvbuf[((size_t)pv_grp * G + h) * D + pv_e0 + v] = pv[h][v];
  __syncthreads();
  for (int idx = tid; idx < G * D; idx += kThreads) {
    float s = 0.f;
    for (int grp = 0; grp < P::kPvGroups; ++grp) s += pvbuf[(size_t)grp * G * D + idx];
    o_part[idx] = s;
  }
  CombineSmem cs{m_loc, l_loc, s_new, cmul, m_glb, l_glb, best_s, best_i, fail_in, red, red_i,
                 decision, o_part, lg, wv};
  combine_and_evict<T, D, G, kThreads>(a, cluster, cs, C, rank, b, g, unit, ubase, n, p, pend,
                                       bud, state_ok, rl, s0, rows, aborted, qg, kn, vn);
}

// ---- layer scope: the shared victim ------------------------------------------

// After the attention kernel of a step, one CTA per sequence adds its KV heads'
// per-slot scores (+inf for slots that are not candidates), takes the lowest
// (ties to the lowest slot), and either records it as the slot the next token
// takes (deferred) or writes every KV head's new token into it.
constexpr int kSelThreads = 1024;
constexpr int kSelWarps = kSelThreads / 32;

template <typename T, int D>
__global__ void __launch_bounds__(kSelThreads) select_layer_kernel(const DecodeArgs a) {
  __shared__ float rs[kSelWarps];
  __shared__ int ri[kSelWarps];
  __shared__ int pick;
  const int b = blockIdx.x;
  const int u0 = b * a.kv_heads;
  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int warp = tid >> 5;
  // Launched as a programmatic dependent of the decode grid: wait until that
  // grid has completed and its writes are visible.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  // The next decode grid may be scheduled now; it still waits for this grid.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  // Every KV head's attention kernel leaves the same request: the slots it
  // scored, + 1 (0: nothing to choose this step).
  const int req = a.lw_req[u0];
  bool same = true;
  for (int g = 1; g < a.kv_heads; ++g) same = same && a.lw_req[u0 + g] == req;
  if (req == 0 && same) return;
  __syncthreads();  // every thread has read the requests
  if (!same || req < 2) {
    if (tid == 0) atomicOr(a.err, LF_DEVERR_STATE);
    for (int g = tid; g < a.kv_heads; g += kSelThreads) a.lw_req[u0 + g] = 0;
    return;
  }
  const int scored = req - 1;
  float bs = INFINITY;
  int bi = INT_MAX;
  // Four consecutive slots per thread and step, one 16-byte load per KV head
  // (every scratch row starts on a 16-byte boundary: slot_stride is a multiple
  // of 32); the heads are summed in order, slots past `scored` are skipped.
  for (int i0 = 4 * tid; i0 < scored; i0 += 4 * kSelThreads) {
    float sc[4] = {0.f, 0.f, 0.f, 0.f};
    for (int g = 0; g < a.kv_heads; ++g) {
      const float4 x =
          *reinterpret_cast<const float4*>(a.lw_score + (size_t)(u0 + g) * a.slot_stride + i0);
      sc[0] += x.x;
      sc[1] += x.y;
      sc[2] += x.z;
      sc[3] += x.w;
    }
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int i = i0 + q;
      if (i < scored && sc[q] < INFINITY && better(sc[q], i, bs, bi)) {
        bs = sc[q];
        bi = i;
      }
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float os = __shfl_xor_sync(0xffffffffu, bs, o);
    const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
    if (better(os, oi, bs, bi)) {
      bs = os;
      bi = oi;
    }
  }
  if (lane == 0) {
    rs[warp] = bs;
    ri[warp] = bi;
  }
  __syncthreads();
  if (tid == 0) {
    for (int w = 1; w < kSelWarps; ++w)
      if (better(rs[w], ri[w], bs, bi)) {
        bs = rs[w];
        bi = ri[w];
      }
    pick = (bi == INT_MAX) ? -1 : bi;
    if (pick < 0) atomicOr(a.err, LF_DEVERR_STATE);  // no candidate
  }
  __syncthreads();
  const int e = pick;
  if (a.deferred) {
    for (int g = tid; g < a.kv_heads; g += kSelThreads) a.pending[u0 + g] = e;
  } else {
    for (int g = warp; g < a.kv_heads; g += kSelWarps) {
      const int u = u0 + g;
      if (e >= 0) {
        const size_t ubase = (size_t)u * a.slot_stride;
        const T* kn = reinterpret_cast<const T*>(a.k_new) + (size_t)u * D;
        const T* vn = reinterpret_cast<const T*>(a.v_new) + (size_t)u * D;
        write_slot<T, D>(a, ubase, e, kn, vn, a.next_pos[u] - 1, a.lw_anew[u], lane, 32);
      }
      if (lane == 0) a.evicted[u] = e;
    }
  }
  for (int g = tid; g < a.kv_heads; g += kSelThreads) a.lw_req[u0 + g] = 0;
}

// ---- prefill ----------------------------------------------------------------

struct PrefillArgs {
  const void* k;          // [batch][kv_heads][max_prompt][D]
  const void* v;
  const int32_t* plen;    // [batch]
  void* K;                // this layer's slab
  void* V;
  float* vnorm;
  int32_t* pos;
  int32_t* count;
  int32_t* next_pos;
  float* acc;             // H2O accumulators (zeroed), or null
  int32_t* pending;       // deferred choice (set to -1), or null
  int kv_heads, max_prompt, slot_stride, norm;
};

// grid (kv_heads, batch); one CTA copies one unit's prompt rows.
template <typename T, int D>
__global__ void __launch_bounds__(kThreads) prefill_kernel(const PrefillArgs a) {
  const int g = blockIdx.x;
  const int b = blockIdx.y;
  const int unit = b * a.kv_heads + g;
  const int P = a.plen[b];
  const size_t src0 = (size_t)unit * a.max_prompt * D;
  const size_t dst0 = (size_t)unit * a.slot_stride * D;
  // Rows 0..P-1 are contiguous on both sides: copy them as 16-byte words.
  const size_t words = (size_t)P * D * sizeof(T) / 16;
  const uint4* ks = reinterpret_cast<const uint4*>(reinterpret_cast<const T*>(a.k) + src0);
  const uint4* vs = reinterpret_cast<const uint4*>(reinterpret_cast<const T*>(a.v) + src0);
  uint4* kd = reinterpret_cast<uint4*>(reinterpret_cast<T*>(a.K) + dst0);
  uint4* vd = reinterpret_cast<uint4*>(reinterpret_cast<T*>(a.V) + dst0);
  for (size_t w = threadIdx.x; w < words; w += kThreads) {
    kd[w] = ks[w];
    vd[w] = vs[w];
  }
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const T* vrow0 = reinterpret_cast<const T*>(a.v) + src0;
  const size_t ubase = (size_t)unit * a.slot_stride;
  for (int i = warp; i < a.slot_stride; i += kWarps) {
    const float nv = (i < P) ? warp_value_norm<T, D>(vrow0 + (size_t)i * D, a.norm, lane) : 0.f;
    if (lane == 0) {
      a.vnorm[ubase + i] = nv;
      a.pos[ubase + i] = (i < P) ? i : -1;
      if (a.acc) a.acc[ubase + i] = 0.f;
    }
  }
  if (threadIdx.x == 0) {
    a.count[unit] = P;
    a.next_pos[unit] = P;
    if (a.pending) a.pending[unit] = -1;
  }
}

}  // namespace lf
