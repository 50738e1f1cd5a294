// The LongFlow fused decode step on the 5th-generation tensor cores (tcgen05):
// a persistent, warp-specialised kernel for bf16 storage, head_dim 128 and
// group size G <= 8.
//
// Work decomposition.  A thread-block cluster of C CTAs walks a list of
// (sequence, KV head) units: cluster j takes units j, j + NC, j + 2 NC, ...
// (NC clusters are resident, one CTA per SM).  CTA `rank` owns the slots
// [rank*chunk, (rank+1)*chunk) of every unit it visits.
//
// Per unit, both contractions run as tcgen05.mma with fp32 accumulators in
// tensor memory:
//   phase A  S^T[slot][h] = K[slot][:] . q_h     M = 128 slots, N = 16 (G heads,
//            A = K tile (K-major), B = q         zero-padded), K = d: 8 MMAs / tile
//   phase B  O^T[e][c]   = sum_slot V[slot][e] P^T[c][slot]
//            A = V tile (MN-major), B = P^T      M = 128 = d, N = 16, K = 128 slots
//            rows c < G hold bf16(p_h), rows G+h hold bf16(p_h - bf16(p_h)), so
//            O = O_hi + O_lo carries p to ~16 significant bits.
// The softmax runs in two passes over the CTA's slots: all logits first (kept
// in shared memory, needed again for the exact score), then p = 2^(s - m)
// with the CTA's exact max m, so nothing is rescaled.
//
// Warp roles (256 threads):
//   warp 4  producer: a ring of 2-D tensor-TMA copies (K then V tiles of
//           128 slots x 256 bytes, 128-byte swizzle) that runs ahead across
//           units, waiting only for stages the tensor cores have read;
//   warp 5  MMA: writes the q operand and issues every tcgen05.mma;
//   warps 0-3  epilogue (thread i <-> TMEM lane i): logits, softmax
//           statistics, P^T and the output accumulator of one unit, then a
//           hand-off of double-buffered state to
//   warps 6-7  tail: the exchange, exact scores, and the leader's output and
//           eviction of that unit, while warps 0-3 go on with the next unit.
// Exchange (no cluster barrier inside the loop, so no other warp stops for
// it): every CTA sends its (m_h, l_h) to all CTAs of the
// cluster with st.async into an mbarrier-counted slot; each CTA then knows
// the unit's max M_h and denominator L_h, scores its own candidates exactly,
//   score_i = ||v_i||_1 * sum_h p_{h,i} 2^(m_h - M_h) / L_h,
// and sends its partial output and its lowest (score, slot) to the unit's
// leader CTA (rank = item mod C), which adds the new token as one more key,
// writes the output, and overwrites the victim slot in place.
// Every wait is bounded; on expiry the step is skipped and LF_DEVERR_TIMEOUT
// is raised.
#pragma once

#include <cuda.h>

#include "lf_decode.cuh"

namespace lf {

constexpr int kTcCompute = 128;   // epilogue threads: warps 0-3, TMEM lanes 0..127
constexpr int kTcProducerWarp = 4;
constexpr int kTcMmaWarp = 5;
constexpr int kTcTailWarp0 = 6;   // tail warps 6 and 7
constexpr int kTcTail = 64;
constexpr int kTcThreads = 256;
constexpr int kTcTile = 128;      // slots per tile (the MMA M of phase A)
constexpr int kTcSBufs = 16;      // logit accumulators in flight between MMA and epilogue
constexpr int kTcLookahead = 2;   // K tiles of the next unit issued before V of this one
constexpr int kTcPBufs = 4;       // P^T tiles in flight between the compute warps and MMA
constexpr int kScoreRows = 4;     // rows a tail thread scores per pass (loads issued together)
#ifndef LF_PREFETCH_TILES
#define LF_PREFETCH_TILES 8
#endif
// K tiles of a CTA's first unit brought into L2 before the grid dependency wait.
constexpr int kPrefetchTiles = LF_PREFETCH_TILES;
// kTcSBufs x 16 columns of S + 16 columns of O, rounded to a power of two.  All
// 512 columns of the SM: the host sizes shared memory so that exactly one CTA
// is resident per SM, so the allocation never waits.
constexpr int kTcTmemCols = 512;
constexpr int kTcMaxItems = 512;  // units one cluster may visit in one launch
constexpr int kTcItemInts = 8;    // ints per entry of the shared-memory item table
constexpr int kTcMaxPlan = 152;   // clusters a launch plan can describe (one per SM at most)

// Planned launches: at most this many CTAs share a unit.
constexpr int kMaxSplitParts = 16;

struct TcArgs {
  CUtensorMap k64, k16, v64, v16;  // 2-D views [rows][128] of K and V, boxes {64,64} / {64,16}
  DecodeArgs a;
  int row_base;                    // tensor row of this layer's first slot
  int max_items;                   // units one cluster may visit (sizes the item table)
  // Planned launches (kernel instantiated with kSplit).  Cluster j takes the
  // whole units j, j + plan_nc, ... below plan_rounds * plan_nc, and before them
  // one contiguous range of the units past the whole rounds (units in order,
  // slots in order within a unit): from slot cut_slot[j] of unit cut_unit[j] to
  // where cluster j + 1 starts (cut plan_nc is (units, 0)).  A unit cut inside
  // (cut_slot > 0) is shared by the clusters whose ranges meet it; they exchange
  // through global memory (all clusters are co-resident: the grid is
  // persistent).  A cluster's parts (at most two: of the unit its range starts
  // inside, then of the unit it ends inside) are its first items, then the
  // units wholly inside its range, then its whole rounds.  The last part of a
  // unit runs to the unit's occupied count at launch time.
  int plan_nc;                     // clusters of the plan (gridDim.y); 0: whole units
  int plan_rounds;                 // whole units per cluster
  float* split_stat;               // [plan_nc][kMaxSplitParts][2 kMaxGroup]: (m_h, l_h) per part
  float* split_fin;                // [plan_nc][kMaxSplitParts][G D + 4]: partial output,
                                   //   score, slot, flag per part
  int* split_cnt;                  // [plan_nc][2]: arrivals at the two exchanges
  int cut_unit[kTcMaxPlan + 1];
  int cut_slot[kTcMaxPlan + 1];    // multiples of 4
  // The host's guess at cluster j's first unit and its occupied slots, for the
  // L2 prefetch before the grid dependency wait (a hint: the copies proper read
  // the counts from memory); hint_n[j] <= 0 or another first unit: no prefetch.
  int hint_unit[kTcMaxPlan];
  int hint_n[kTcMaxPlan];
};

// One cluster's part of a shared unit in a planned launch.
struct TcPiece {
  int unit, lo, hi;  // slots [lo, hi) of the unit (hi = INT_MAX: to its occupied count)
  int info;          // exchange row (its first inner cut) << 16 | index among the
                     //   unit's clusters (0 leads) << 8 | clusters sharing the unit
};

// The parts of cluster j's range: of the unit it starts inside, then of the
// unit it ends inside (one part when it lies inside a single unit); and the
// units wholly inside it, [*w0, *w1).  Returns the number of parts (0-2).
__device__ __forceinline__ int plan_pieces(const TcArgs& ta, int j, TcPiece* pc, int* w0,
                                           int* w1) {
  const int nc = ta.plan_nc;
  const int u0 = ta.cut_unit[j], s0 = ta.cut_slot[j];
  const int u1 = ta.cut_unit[j + 1], s1 = ta.cut_slot[j + 1];
  auto inner = [&](int c, int u) {
    return c >= 1 && c < nc && ta.cut_unit[c] == u && ta.cut_slot[c] > 0;
  };
  int np = 0;
  if (s0 > 0) {  // the range starts inside unit u0
    int jmin = j, jmax = j;
    while (inner(jmin - 1, u0)) --jmin;
    while (inner(jmax + 1, u0)) ++jmax;
    pc[np++] = {u0, s0, (u1 == u0) ? s1 : INT_MAX,
                (jmin << 16) | ((j - jmin + 1) << 8) | (jmax - jmin + 2)};
  }
  if (s1 > 0 && !(s0 > 0 && u1 == u0)) {  // it ends inside unit u1 and holds slot 0
    int jmax = j + 1;
    while (inner(jmax + 1, u1)) ++jmax;
    pc[np++] = {u1, 0, s1, ((j + 1) << 16) | (jmax - j + 1)};
  }
  *w0 = (s0 > 0) ? u0 + 1 : u0;  // units wholly inside the range
  *w1 = max(*w0, u1);
  return np;
}

// Split launches: spin, with a bound, until another CTA of this persistent grid
// (all of them are resident) has counted itself in.
__device__ __forceinline__ int ld_acquire_gpu(const int* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ bool wait_count_bounded(const int* cnt, int target) {
  if (ld_acquire_gpu(cnt) >= target) return true;
  const unsigned long long t0 = global_ns();
  for (;;) {
#pragma unroll 1
    for (int i = 0; i < 32; ++i) {
      if (ld_acquire_gpu(cnt) >= target) return true;
      __nanosleep(32);
    }
    if (global_ns() - t0 > kWaitLimitNs) return false;
  }
}

// sum_h row[h] cm[h], the FMAs in head order (vector loads of the logit row).
template <int G>
__device__ __forceinline__ float group_dot(const float* row, const float* cm) {
  float as = 0.f;
  if constexpr (G % 4 == 0) {
#pragma unroll
    for (int h = 0; h < G; h += 4) {
      const float4 x = *reinterpret_cast<const float4*>(row + h);
      as = fmaf(x.x, cm[h], as);
      as = fmaf(x.y, cm[h + 1], as);
      as = fmaf(x.z, cm[h + 2], as);
      as = fmaf(x.w, cm[h + 3], as);
    }
  } else if constexpr (G == 2) {
    const float2 x = *reinterpret_cast<const float2*>(row);
    as = fmaf(x.x, cm[0], as);
    as = fmaf(x.y, cm[1], as);
  } else {
#pragma unroll
    for (int h = 0; h < G; ++h) as = fmaf(row[h], cm[h], as);
  }
  return as;
}

template <int G>
struct TcPlan {
  static constexpr int D = 128;
  static constexpr int kBlock = kTcTile * 128;  // [128 rows][64 bf16], swizzled: 16 KB
  static constexpr int kStage = 2 * kBlock;     // one K or V tile: 32 KB
  static constexpr int kQBytes = 2 * 16 * 128;  // q^T operand [16][128], 2 blocks
  static constexpr int kPTile = 2 * 16 * 128;   // P^T operand of one tile [16][128 slots]
  static constexpr int kFinBytes = G * D * 4 + 16;  // one CTA's partial output + (score, slot)
  // header: barriers, statistics, reductions, exchange slots, unit metadata
  static constexpr int kOffBars = 0;     // 112 mbarriers
  static constexpr int kOffStats = 896;  // m_loc[2], l_loc[2], s_new[2], cmul, m_glb, l_glb
  static constexpr int kOffRed = kOffStats + 9 * kMaxGroup * 4;
  static constexpr int kOffMisc = kOffRed + 4 * kMaxGroup * 4 + 16;
  // the leader's output scales: 2^(m_r - M) / L per part r and head, and the new token's
  static constexpr int kOffOutScale = 1408;  // [kMaxSplitParts + 1][kMaxGroup] floats
  // planned launches: the tail's copy of a shared unit's parts' (m, l)
  static constexpr int kOffPieceStats = 2048;                // [kMaxSplitParts][2G] floats
  static constexpr int kOffStatIn = 3072;                    // [2][kMaxCluster][2G] floats
  static constexpr int kOffOpart = kOffStatIn + 2 * kMaxCluster * 2 * kMaxGroup * 4;  // [2][G][D]
  static_assert(kOffMisc + 80 <= kOffOutScale, "header overflow");
  static_assert(kOffOutScale + (kMaxSplitParts + 1) * kMaxGroup * 4 <= kOffPieceStats,
                "header overflow");
  static_assert(kMaxCluster <= kMaxSplitParts, "output scales sized for the larger count");
  static_assert(kOffPieceStats + kMaxSplitParts * 2 * kMaxGroup * 4 <= kOffStatIn,
                "header overflow");
  static_assert(16 + 16 + 2 * kTcSBufs + 2 * kTcPBufs + 16 <= kOffStats / 8, "too many barriers");
  static constexpr int kOffNew = kOffOpart + 2 * G * D * 4;  // [2][k | v][D] the new token
  static constexpr int kOffQ = (kOffNew + 2 * 2 * D * 2 + 1023) / 1024 * 1024;  // [2] buffers
  static constexpr int kOffRing = kOffQ + 2 * kQBytes;

  __host__ __device__ static constexpr int off_p(int stages) { return kOffRing + stages * kStage; }
  __host__ __device__ static constexpr int off_fin(int stages) {
    return off_p(stages) + kTcPBufs * kPTile;
  }
  __host__ __device__ static constexpr int off_lg(int stages, int cluster) {
    return off_fin(stages) + cluster * kFinBytes;
  }
  __host__ __device__ static constexpr int vn_bytes(int chunk) { return (chunk + 3) / 4 * 16; }
  // Eviction needs two logit buffers (the tail warps score unit k while the
  // epilogue fills unit k+1) and the ||v||_1 / position / weight buffers; the
  // read-only full-KV mode needs one logit buffer and none of the others.
  __host__ __device__ static constexpr int off_vn(int stages, int chunk, int cluster, int evict) {
    return (off_lg(stages, cluster) + (evict ? 2 : 1) * chunk * G * 4 + 15) / 16 * 16;
  }
  // vn[2], pos[2] (raw, from the slab) then w[2] (candidate weights), each vn_bytes(chunk);
  // then the item table: (count, next position, deferred choice, budget, unit, first
  // slot, end slot, part) per item visited.
  __host__ __device__ static constexpr int off_items(int stages, int chunk, int cluster,
                                                     int evict) {
    return off_vn(stages, chunk, cluster, evict) + (evict ? 6 * vn_bytes(chunk) : 0);
  }
  __host__ __device__ static constexpr int smem_bytes(int stages, int chunk, int cluster,
                                                      int evict, int items) {
    return off_items(stages, chunk, cluster, evict) + items * kTcItemInts * 4 +
           1024;  // + alignment slack
  }
};

// The L2 prefetch of a CTA's first unit before the grid dependency wait (see
// the kernel): rows [lo, hi) of unit u clipped to its n occupied slots, this
// CTA's share of them, as the copies proper will read them (64-row boxes, then
// 16-row granules, up to kPrefetchTiles tiles), its norms and positions, and
// the group's queries.  Out of line: a launch without hints pays nothing for it.
template <int G>
__device__ __noinline__ void prefetch_first_unit(const TcArgs& ta, int u, int lo, int hi, int n,
                                                 int C, int rank) {
  constexpr int D = 128;
  using T = __nv_bfloat16;
  const DecodeArgs& a = ta.a;
  const int lo2 = min(lo, n);
  const int hi2 = min(hi, n);
  const int per = ((hi2 - lo2 + C - 1) / C + 3) & ~3;
  const int base = lo2 + rank * per;
  const int rows = max(0, min(per, hi2 - base));
  const int row0 = ta.row_base + u * a.slot_stride + base;
  const int lim = min((rows + 15) & ~15, kPrefetchTiles * kTcTile);
  int r = 0;
  for (; r + 64 <= lim; r += 64) {
    tma_prefetch_l2_2d(&ta.k64, 0, row0 + r);
    tma_prefetch_l2_2d(&ta.k64, 64, row0 + r);
  }
  for (; r < lim; r += 16) {
    tma_prefetch_l2_2d(&ta.k16, 0, row0 + r);
    tma_prefetch_l2_2d(&ta.k16, 64, row0 + r);
  }
  if (rows > 0 && a.evict) {
    const size_t ub = (size_t)u * a.slot_stride + base;
    const uint32_t small = (uint32_t)(((rows + 3) & ~3) * 4);
    bulk_prefetch_l2((a.score == LF_SCORE_H2O ? a.acc : a.vnorm) + ub, small);
    bulk_prefetch_l2(a.pos + ub, small);
  }
  const int bb = u / a.kv_heads;
  bulk_prefetch_l2(reinterpret_cast<const T*>(a.q) +
                       ((size_t)bb * a.q_heads + (size_t)(u - bb * a.kv_heads) * G) * D,
                   (uint32_t)(G * D * sizeof(T)));
}

template <int G, bool kSplit = false>
__global__ void __launch_bounds__(kTcThreads, 1)
    decode_step_tc_kernel(const __grid_constant__ TcArgs ta) {
  constexpr int D = 128;
  using P = TcPlan<G>;
  using T = __nv_bfloat16;
  static_assert(2 * G <= 16, "group too large for N = 16");
  static_assert(D == kTcCompute, "one compute thread per output element / TMEM lane");
  const DecodeArgs& a = ta.a;

  cg::cluster_group cluster = cg::this_cluster();
  const int C = (int)cluster.num_blocks();
  const int rank = (int)cluster.block_rank();
  const int NC = (int)gridDim.y;
  const int j = (int)blockIdx.y;
  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int warp = tid >> 5;
  const int S = a.stages;
  const int chunk = a.chunk;
  const int units = a.batch * a.kv_heads;
  // Whole-unit launches: cluster j takes units j, j + NC, ...  Planned
  // launches: its parts of shared units first (every cluster's range takes
  // about as long, so the parts of a unit finish about together and the
  // exchanges through L2 overlap the stream of the whole units after them),
  // then the units wholly inside its range, then plan_rounds whole units.
  const bool planned = kSplit && ta.plan_nc == NC;
  TcPiece pcs[2];
  int w0 = 0, w1 = 0;
  const int npc = planned ? plan_pieces(ta, j, pcs, &w0, &w1) : 0;  // parts, exchanged via L2
  const int nitems = planned ? npc + (w1 - w0) + ta.plan_rounds
                             : ((j < units) ? (units - j + NC - 1) / NC : 0);
  if (nitems > ta.max_items || (kSplit && !planned) ||
      (npc > 0 && (pcs[0].info & 0xff) * C > kMaxSplitParts) ||
      (npc > 1 && (pcs[1].info & 0xff) * C > kMaxSplitParts)) {
    // the host sized the item table for fewer units, or the plan does not fit
    if (threadIdx.x == 0 && cg::this_cluster().block_rank() == 0) atomicOr(ta.a.err, LF_DEVERR_STATE);
    return;
  }

  extern __shared__ __align__(1024) unsigned char smem_raw[];
  // The 128-byte swizzle phase of TMA writes and MMA reads follows address
  // bits 7-9: start the carve-up on a 1024-byte boundary (1 KB is reserved).
  unsigned char* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + P::kOffBars);
  uint64_t* full = bars;                   // [16] stage landed
  uint64_t* empty = bars + 16;             // [16] stage read by the tensor cores
  uint64_t* sfull = bars + 32;             // [kTcSBufs] logits ready in TMEM
  uint64_t* sfree = sfull + kTcSBufs;      // [kTcSBufs] logits read by the compute warps
  uint64_t* pready = sfree + kTcSBufs;     // [kTcPBufs] P^T tile written
  uint64_t* pfree = pready + kTcPBufs;     // [kTcPBufs] P^T tile read by the tensor cores
  uint64_t* ofull = pfree + kTcPBufs;      // output accumulator complete
  uint64_t* aux = ofull + 1;               // [2] ||v||_1 and positions landed
  uint64_t* auxfree = aux + 2;             // [2] ... read by the epilogue warps
  uint64_t* statb = auxfree + 2;           // [2] all CTAs' (m, l) arrived
  uint64_t* finb = statb + 2;              // all CTAs' partial outputs arrived (leader)
  uint64_t* qfree = finb + 1;              // [2] q operand buffer read by the tensor cores
  uint64_t* handoff = qfree + 2;           // [2] epilogue -> tail: a unit's state is ready
  uint64_t* taildone = handoff + 2;        // [2] tail -> epilogue: that state is consumed
  uint64_t* drain = taildone + 2;          // every MMA complete
  uint64_t* statrdy = drain + 1;           // [2] epilogue -> tail: (m, l), logits, weights
  uint64_t* gstat = statrdy + 2;           // tail -> epilogue: the last unit's scales (once)
  uint64_t* escore = gstat + 1;            // epilogue -> tail: its share of the last unit's scores
  float* m_loc = reinterpret_cast<float*>(smem + P::kOffStats);  // [2][kMaxGroup]
  float* l_loc = m_loc + 2 * kMaxGroup;                          // [2][kMaxGroup]
  float* s_new = l_loc + 2 * kMaxGroup;                          // [2][kMaxGroup]
  float* cmul = s_new + 2 * kMaxGroup;
  float* m_glb = cmul + kMaxGroup;
  float* l_glb = m_glb + kMaxGroup;
  float* osc = reinterpret_cast<float*>(smem + P::kOffOutScale);  // [parts + 1][kMaxGroup]
  float* red = reinterpret_cast<float*>(smem + P::kOffRed);  // epilogue: [4][kMaxGroup]
  float* red_t = red + 4 * kMaxGroup;                        // tail: [2] scores
  int* red_ti = reinterpret_cast<int*>(red_t + 2);           // tail: [2] slots
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + P::kOffMisc);
  int* decision = reinterpret_cast<int*>(smem + P::kOffMisc + 8);
  volatile int* fail_any = reinterpret_cast<volatile int*>(smem + P::kOffMisc + 16);
  volatile int* uflag = reinterpret_cast<volatile int*>(smem + P::kOffMisc + 24);  // [2]
  volatile int* split_flag = reinterpret_cast<volatile int*>(smem + P::kOffMisc + 40);
  volatile int* gscore_ok = reinterpret_cast<volatile int*>(smem + P::kOffMisc + 44);
  float* esc_s = reinterpret_cast<float*>(smem + P::kOffMisc + 48);  // [4] epilogue warps' lowest
  int* esc_i = reinterpret_cast<int*>(smem + P::kOffMisc + 64);      // [4]
  float* stat_in = reinterpret_cast<float*>(smem + P::kOffStatIn);  // [2][C][2G]
  int* items = reinterpret_cast<int*>(smem + P::off_items(S, chunk, C, a.evict));  // [nitems][8]
  float* opbase = reinterpret_cast<float*>(smem + P::kOffOpart);     // [2][G][D]
  unsigned char* qbuf = smem + P::kOffQ;
  unsigned char* ring = smem + P::kOffRing;
  unsigned char* ptile = smem + P::off_p(S);      // [kTcPBufs] P^T tiles
  unsigned char* fin_in = smem + P::off_fin(S);   // [C][kFinBytes]
  float* lgbase = reinterpret_cast<float*>(smem + P::off_lg(S, C));  // [2][chunk][G]
  unsigned char* vnbase = smem + P::off_vn(S, chunk, C, a.evict);
  const int lgpar = a.evict ? 1 : 0;  // logit buffers alternate only when scores are needed

  // ---- set-up ---------------------------------------------------------------
  // Everything up to griddepcontrol.wait touches only this CTA's own shared and
  // tensor memory, so with programmatic dependent launch it overlaps the tail
  // of the previous launch on the stream.
  if (tid == kTcProducerWarp * 32) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int i = 0; i < kTcSBufs; ++i) {
      mbar_init(&sfull[i], 1);
      mbar_init(&sfree[i], 4);
    }
    mbar_init(ofull, 1);
    mbar_init(finb, 1);
    for (int i = 0; i < kTcPBufs; ++i) {
      mbar_init(&pready[i], 4);
      mbar_init(&pfree[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&aux[i], 1);
      mbar_init(&auxfree[i], 4);   // the four epilogue warps
      mbar_init(&statb[i], 1);
      mbar_init(&qfree[i], 1);
      mbar_init(&handoff[i], 4);   // the four epilogue warps
      mbar_init(&taildone[i], 2);  // the two tail warps
      mbar_init(&statrdy[i], 1);
    }
    mbar_init(drain, 1);
    mbar_init(gstat, 1);
    mbar_init(escore, 4);  // the four epilogue warps
    fence_mbar_init();
    // The tensor maps are kernel parameters: fetch them before the wait below.
    tma_prefetch_desc(&ta.k64);
    tma_prefetch_desc(&ta.k16);
    tma_prefetch_desc(&ta.v64);
    tma_prefetch_desc(&ta.v16);
    // While the previous grid on the stream finishes (its last units leave HBM
    // mostly idle), bring the first K tiles of this CTA's first unit, its norms
    // and positions and its queries into L2.  A hint only: the copies proper
    // come after the wait below and read memory again; the occupancy is the
    // host's (a kernel parameter: no global load holds up the set-up), so a
    // wrong value costs bandwidth and nothing else.
    int u = j, lo = 0, hi = INT_MAX;
    if (npc > 0) {
      u = pcs[0].unit;
      lo = pcs[0].lo;
      hi = pcs[0].hi;
    } else if (w1 > w0) {
      u = w0;
    }
    if (nitems > 0 && kPrefetchTiles > 0 && j < kTcMaxPlan && ta.hint_unit[j] == u &&
        ta.hint_n[j] > 0)
      prefetch_first_unit<G>(ta, u, lo, hi, min(ta.hint_n[j], a.capacity), C, rank);
  }
  if (tid == 0) *fail_any = 0;
  // Operand buffers start at zero (padding rows of q^T and P^T stay zero).
  {
    uint4* z = reinterpret_cast<uint4*>(qbuf);
    for (int i = tid; i < 2 * P::kQBytes / 16; i += kTcThreads) z[i] = make_uint4(0, 0, 0, 0);
    z = reinterpret_cast<uint4*>(ptile);
    for (int i = tid; i < kTcPBufs * P::kPTile / 16; i += kTcThreads) z[i] = make_uint4(0, 0, 0, 0);
  }
  if (warp == 0) {
    tmem_alloc(tmem_slot, kTcTmemCols);
    tmem_relinquish();
  }
  // Global memory from here on: wait until the previous grid on the stream has
  // completed and its writes are visible (this kernel never lets a dependent
  // grid pass its own wait early, so back-to-back steps of one layer stay ordered).
  asm volatile("griddepcontrol.wait;" ::: "memory");
  // Let the next grid on the stream be scheduled now: its CTAs take SMs as this
  // grid's CTAs exit and run their set-up there, but none of them passes its own
  // griddepcontrol.wait before this whole grid has completed.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  // Occupancy and position of every unit this cluster visits, read once: the
  // leaders update them during the launch, every role must see the old values.
  // (A unit shared with other clusters is updated by its leader only after
  // every part has sent its partial output, so all of them have read it.)
  for (int k = tid; k < nitems; k += kTcThreads) {
    int u, lo = 0, hi = INT_MAX, part = 0;
    if (k < npc) {
      u = pcs[k].unit;
      lo = pcs[k].lo;
      hi = pcs[k].hi;
      part = pcs[k].info;  // the low byte (clusters sharing the unit) is >= 2: never 0
    } else if (k < npc + (w1 - w0)) {
      u = w0 + (k - npc);  // a unit wholly inside the range
    } else {
      u = j + (k - npc - (w1 - w0)) * NC;
    }
    int* it = items + kTcItemInts * k;
    it[0] = a.count[u];
    it[1] = a.next_pos[u];
    it[2] = (a.evict && a.deferred) ? a.pending[u] : -1;
    it[3] = a.budget[u / a.kv_heads];
    it[4] = u;
    it[5] = lo;
    it[6] = hi;
    it[7] = part;
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // Every CTA of the cluster has started: shared memory may be addressed remotely.
  cluster.sync();
  const uint32_t tmem = *tmem_slot;
  const uint32_t tO = tmem + 16 * kTcSBufs;

  auto unit_of = [&](int k) { return items[kTcItemInts * k + 4]; };
  // The launch's last item, a whole unit with the plain LongFlow score: the
  // epilogue warps, idle after it, score the rows from `split` on while the tail
  // warps score the rows before it, so that the launch ends sooner.
  auto last_shared_scoring = [&](int k, const UnitRule& rl) {
    return k == nitems - 1 && items[kTcItemInts * k + 7] == 0 && rl.choosing &&
           a.score != LF_SCORE_H2O && a.scope != LF_SCOPE_LAYER;
  };
  auto score_split = [](int rows) { return (rows / 3) & ~3; };
  auto is_piece = [&](int k) { return kSplit && items[kTcItemInts * k + 7] != 0; };
  // This CTA's share of item k: the occupied slots of the unit (of a shared
  // unit: of this cluster's range of it, clipped to the occupied count) are
  // split evenly over the cluster, in multiples of 4 from a multiple of 4, so
  // a partly filled unit keeps every CTA busy.  Returns the slot count and
  // sets `base`, the first slot.
  auto unit_rows = [&](int k, int& n, int& p, bool& ok, int& base) {
    const int* it = items + kTcItemInts * k;
    n = it[0];
    p = it[1];
    ok = (n >= 0 && n <= a.capacity && p >= n);
    const int lo = min(it[5], max(n, 0));
    const int hi = min(it[6], max(n, 0));
    const int per = ((hi - lo + C - 1) / C + 3) & ~3;  // <= chunk since n <= capacity
    base = lo + rank * per;
    return ok ? max(0, min(per, hi - base)) : 0;
  };

  // Tile order through the ring, shared by the producer and the MMA warp.  For
  // the non-empty units u0, u1, ... of this CTA:
  //   K(u0), then for each x: K(u_{x+1})[0, L), V(u_x), K(u_{x+1})[L, end)
  // with L = min(tiles, kTcLookahead): the next unit's first logits are computed
  // while the epilogue warps finish the softmax of u_x, so the tensor cores and
  // the TMA stream do not wait for it.  L stays below the accumulator count,
  // which the epilogue frees before it needs V(u_x).  A pending
  // V(u_x) is issued on its own as soon as the walk reaches unit u_x + 2
  // (empty units in between): the producer then waits for the tail warps to be
  // done with u_x, which needs V(u_x) -- so every wait looks strictly back.
  if (warp == kTcProducerWarp) {
    // ---- producer: the ring of K / V tiles and the per-unit ||v||_1, pos ----------
    if (lane == 0) {
      const uint64_t pol = l2_evict_first_policy();
      bool fail = false;
      int tt = 0;  // tiles produced
      // Each step of the walk is up to five segments in ring order, issued by one
      // loop (one copy of the issue code): 0, a pending V(prev) that the walk has
      // passed; 1, unit k's norms and positions; 2, its first K tiles (all of them
      // when nothing is pending); 3, V(prev); 4, the rest of its K tiles.  Step
      // nitems only flushes.
      int prev = -1, prev_rows = 0, prev_base = 0;
      for (int k = 0; k <= nitems && !fail; ++k) {
        const bool flush = prev >= 0 && (k == nitems || prev <= k - 2);
        const int fk = prev, frows = prev_rows, fbase = prev_base;
        if (flush) prev = -1;
        int rows = 0, base = 0, ntile = 0, L = 0;
        if (k < nitems) {
          int n, p;
          bool ok;
          rows = unit_rows(k, n, p, ok, base);
          ntile = (rows + kTcTile - 1) / kTcTile;
          L = (prev < 0) ? ntile : min(ntile, kTcLookahead);
        }
        const bool pend = prev >= 0 && rows > 0;  // V(prev) between this unit's K tiles
#pragma unroll 1
        for (int si = 0; si < 5 && !fail; ++si) {
          // this segment: unit item gk (rows, first slot), kind, tiles [t0, t1)
          int gk = k, grows = rows, gbase = base, t0 = 0, t1 = 0;
          bool isK = true;
          if (si == 0 || si == 3) {
            if (si == 0 ? !flush : !pend) continue;
            gk = (si == 0) ? fk : prev;
            grows = (si == 0) ? frows : prev_rows;
            gbase = (si == 0) ? fbase : prev_base;
            isK = false;
            t1 = (grows + kTcTile - 1) / kTcTile;
          } else if (si == 1) {
            if (k == nitems) continue;
            // unit k's ||v||_1 (H2O: accumulators) and positions, once the
            // epilogue has read this parity's buffers (unit k - 2)
            const int b2 = k & 1;
            if (k >= 2 && !mbar_wait_bounded(&auxfree[b2], (uint32_t)(((k >> 1) - 1) & 1))) {
              fail = true;
              break;
            }
            if (rows > 0 && a.evict) {
              const size_t ub = (size_t)unit_of(k) * a.slot_stride + base;
              const uint32_t small = (uint32_t)(((rows + 3) & ~3) * 4);
              unsigned char* vdst = vnbase + b2 * P::vn_bytes(chunk);
              unsigned char* pdst = vnbase + (2 + b2) * P::vn_bytes(chunk);
              mbar_arrive_expect_tx(&aux[b2], 2u * small);
              bulk_g2s(vdst, (a.score == LF_SCORE_H2O ? a.acc : a.vnorm) + ub, small, &aux[b2],
                       pol);
              bulk_g2s(pdst, a.pos + ub, small, &aux[b2], pol);
            } else {
              mbar_arrive(&aux[b2]);  // nothing to load: complete the phase
            }
            continue;
          } else {
            t0 = (si == 2) ? 0 : L;
            t1 = (si == 2) ? L : ntile;
          }
          // Tiles [t0, t1) of the unit (K or V) into the ring.
          const int unit_row = ta.row_base + unit_of(gk) * a.slot_stride + gbase;
          const void* m64 = isK ? (const void*)&ta.k64 : (const void*)&ta.v64;
          const void* m16 = isK ? (const void*)&ta.k16 : (const void*)&ta.v16;
#pragma unroll 1
          for (int t = t0; t < t1; ++t, ++tt) {
            const int st = tt % S;
            if (tt >= S && !mbar_wait_bounded(&empty[st], (uint32_t)(((tt / S) - 1) & 1))) {
              fail = true;
              break;
            }
            const int r0 = t * kTcTile;
            const int rr = (min(kTcTile, grows - r0) + 15) & ~15;  // 16-row granules
            unsigned char* dst = ring + (size_t)st * P::kStage;
            mbar_arrive_expect_tx(&full[st], (uint32_t)(rr * D * 2));
            for (int blk = 0; blk < 2; ++blk) {
              int ro = 0;
              for (; ro + 64 <= rr; ro += 64)
                tma_load_2d(dst + blk * P::kBlock + ro * 128, m64, blk * 64, unit_row + r0 + ro,
                            &full[st], pol);
              for (; ro < rr; ro += 16)
                tma_load_2d(dst + blk * P::kBlock + ro * 128, m16, blk * 64, unit_row + r0 + ro,
                            &full[st], pol);
            }
          }
        }
        if (k < nitems && rows > 0) {
          prev = k;
          prev_rows = rows;
          prev_base = base;
        }
      }
      // Every copy issued lands before the CTA may exit.
      for (int t = max(0, tt - S); t < tt; ++t)
        (void)mbar_wait_bounded(&full[t % S], (uint32_t)((t / S) & 1));
      if (fail) {
        *fail_any = 1;
        atomicOr(a.err, LF_DEVERR_TIMEOUT);
      }
    }
    __syncwarp();
  } else if (warp == kTcMmaWarp) {
    // ---- MMA warp: the q operand (all lanes) and every tcgen05.mma (lane 0) --------
    constexpr uint32_t kIdA = idesc_bf16_f32(128, 16, false, false);
    constexpr uint32_t kIdB = idesc_bf16_f32(128, 16, true, false);
    bool fail = false;
    int tt = 0, kt = 0, pt = 0, nn = 0;  // tiles, K tiles, P^T tiles, non-empty units
    int nq[2] = {0, 0};
    // K tiles [t0, t1) of a unit: S^T = K . q^T into the next free logit accumulator.
    auto mma_k = [&](int t0, int t1, uint32_t qaddr) {
#pragma unroll 1
      for (int t = t0; t < t1 && !fail; ++t, ++tt, ++kt) {
        const int st = tt % S;
        const int buf = kt % kTcSBufs;
        if (!mbar_wait_bounded(&full[st], (uint32_t)((tt / S) & 1)) ||
            (kt >= kTcSBufs &&
             !mbar_wait_bounded(&sfree[buf], (uint32_t)(((kt / kTcSBufs) - 1) & 1)))) {
          fail = true;
          break;
        }
        tc_fence_after();
        const uint32_t sbase = smem_u32(ring + (size_t)st * P::kStage);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t ko = (uint32_t)((kk >> 2) * P::kBlock + (kk & 3) * 32);
          const uint32_t qo = (uint32_t)((kk >> 2) * 2048 + (kk & 3) * 32);
          tc_mma_bf16(tmem + 16 * buf, sw128_desc(sbase + ko, 16, 1024),
                      sw128_desc(qaddr + qo, 16, 1024), kIdA, kk > 0 ? 1u : 0u);
        }
        tc_commit(&sfull[buf]);
        tc_commit(&empty[st]);
      }
    };
    // All V tiles of a unit: O^T += V^T . P^T, then signal the output.
    auto mma_v = [&](int rows) {
      const int ntile = (rows + kTcTile - 1) / kTcTile;
#pragma unroll 1
      for (int vt = 0; vt < ntile && !fail; ++vt, ++tt, ++pt) {
        const int st = tt % S;
        const int pb = pt % kTcPBufs;
        if (!mbar_wait_bounded(&pready[pb], (uint32_t)((pt / kTcPBufs) & 1)) ||
            !mbar_wait_bounded(&full[st], (uint32_t)((tt / S) & 1))) {
          fail = true;
          break;
        }
        tc_fence_after();
        const uint32_t sbase = smem_u32(ring + (size_t)st * P::kStage);
        const int ksteps = (min(kTcTile, rows - vt * kTcTile) + 15) >> 4;
        const uint32_t pbase = smem_u32(ptile + (size_t)pb * P::kPTile);
        for (int jj = 0; jj < ksteps; ++jj) {
          const uint32_t po = (uint32_t)((jj >> 2) * 2048 + (jj & 3) * 32);
          tc_mma_bf16(tO, sw128_desc(sbase + jj * 2048, P::kBlock, 1024),
                      sw128_desc(pbase + po, 16, 1024), kIdB, (vt > 0 || jj > 0) ? 1u : 0u);
        }
        tc_commit(&empty[st]);
        tc_commit(&pfree[pb]);
      }
      tc_commit(ofull);
    };
    // The group's queries of unit item kk, 16-byte chunk c = lane + 32 i, loaded
    // into registers one unit ahead: the load's latency then passes while this
    // warp issues the previous unit's MMAs instead of holding up the ring.
    constexpr int kQChunks = (G * 16 + 31) / 32;
    uint4 qreg[kQChunks];
    int qreg_item = -1;
    auto load_q = [&](int kk) {
      const int uu = unit_of(kk);
      const int bb = uu / a.kv_heads;
      const int gg = uu - bb * a.kv_heads;
      const T* qsrc =
          reinterpret_cast<const T*>(a.q) + ((size_t)bb * a.q_heads + (size_t)gg * G) * D;
#pragma unroll
      for (int i = 0; i < kQChunks; ++i) {
        const int c = lane + 32 * i;
        if (c < G * 16)
          qreg[i] = *reinterpret_cast<const uint4*>(qsrc + (size_t)(c >> 4) * D + (c & 15) * 8);
      }
      qreg_item = kk;
    };
    if (nitems > 0) load_q(0);
    // The producer's walk, step by step: its tile segments in ring order (0, a
    // pending V(prev); 2, unit k's first K tiles; 3, V(prev); 4, the rest of its
    // K tiles), issued by lane 0 through one copy of each MMA loop.
    int prev = -1, prev_rows = 0;
    for (int k = 0; k <= nitems && !fail; ++k) {
      const bool flush = prev >= 0 && (k == nitems || prev <= k - 2);
      const int frows = prev_rows;
      if (flush) prev = -1;
      int rows = 0, qb = 0, ntile = 0, L = 0;
      uint32_t qaddr = 0;
      if (k < nitems) {
        int n, p, base;
        bool ok;
        rows = unit_rows(k, n, p, ok, base);
      }
      if (rows > 0) {
        ntile = (rows + kTcTile - 1) / kTcTile;
        L = (prev < 0) ? ntile : min(ntile, kTcLookahead);
        qb = nn & 1;
        unsigned char* qdst = qbuf + qb * P::kQBytes;
        // The buffer's previous contents (two units ago) must have been read.
        bool okq = true;
        if (lane == 0 && nq[qb] > 0)
          okq = mbar_wait_bounded(&qfree[qb], (uint32_t)((nq[qb] - 1) & 1));
        if (__shfl_sync(0xffffffffu, okq ? 1 : 0, 0) == 0) {
          fail = true;
          break;
        }
        // q^T rows h < G: the group's queries (16-byte chunks, 128-byte swizzle).
        if (qreg_item != k) load_q(k);   // not fetched ahead (an empty unit came between)
#pragma unroll
        for (int i = 0; i < kQChunks; ++i) {
          const int c = lane + 32 * i;
          if (c < G * 16) {
            const int h = c >> 4;
            const int ch = c & 15;
            *reinterpret_cast<uint4*>(qdst + (ch >> 3) * 2048 + h * 128 + (((ch & 7) ^ (h & 7)) << 4)) =
                qreg[i];
          }
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (k + 1 < nitems) load_q(k + 1);   // the next unit's queries, in the background
        qaddr = smem_u32(qdst);
      }
      const bool pend = prev >= 0 && rows > 0;
      if (lane == 0) {
#pragma unroll 1
        for (int si = 0; si < 5 && !fail; ++si) {
          if (si == 0 || si == 3) {
            if (si == 0 ? !flush : !pend) continue;
            mma_v(si == 0 ? frows : prev_rows);
          } else if (si != 1 && rows > 0) {
            mma_k(si == 2 ? 0 : L, si == 2 ? L : ntile, qaddr);
          }
        }
        if (rows > 0) tc_commit(&qfree[qb]);
      }
      if (rows > 0) {
        nq[qb] += 1;
        nn += 1;
        prev = k;
        prev_rows = rows;
      }
      fail = __shfl_sync(0xffffffffu, fail ? 1 : 0, 0) != 0;
    }
    if (lane == 0) {
      // Every MMA issued completes before tensor memory is released.
      tc_commit(drain);
      (void)mbar_wait_bounded(drain, 0);
      if (fail) {
        *fail_any = 1;
        atomicOr(a.err, LF_DEVERR_TIMEOUT);
      }
    }
    __syncwarp();
  } else if (warp < kTcTailWarp0) {
    // ---- epilogue warps 0-3 (thread i <-> TMEM lane i) ---------------------------
    // A shared unit (planned launch): this CTA's (m_h, l_h) go to the unit's other
    // parts through global memory as soon as they are final, from here rather
    // than from the tail warps, so that no cluster's exchange waits for another
    // cluster's tail to reach that unit.  Thread 0, after m_loc / l_loc are written.
    auto publish_stats = [&](int k, int b2) {
      const int part = items[kTcItemInts * k + 7];
      const int xi = part >> 16;
      const int me = ((part >> 8) & 0xff) * C + rank;
      float* gst = ta.split_stat + ((size_t)xi * kMaxSplitParts + me) * 2 * kMaxGroup;
#pragma unroll
      for (int h = 0; h < kMaxGroup; ++h) {
        gst[h] = h < G ? m_loc[b2 * kMaxGroup + h] : -INFINITY;
        gst[kMaxGroup + h] = h < G ? l_loc[b2 * kMaxGroup + h] : 0.f;
      }
      __threadfence();
      atomicAdd(ta.split_cnt + 2 * xi, 1);
    };
    // The epilogue warps' share of the last unit's scores (rows from score_split
    // on), once the tail warps have the unit's scales; the lowest (score, slot)
    // of each warp goes to the tail warps.  Every path arrives on `escore`.
    auto epilogue_scores = [&](int rows, int base, const UnitRule& rl, const float* lg,
                               const float* w_s, bool have) {
      const bool ok = __all_sync(0xffffffffu, mbar_wait_bounded(gstat, 0));
      float bs = INFINITY;
      int bi = INT_MAX;
      if (ok && have && gscore_ok[0]) {
        float cm[G];
#pragma unroll
        for (int h = 0; h < G; ++h) cm[h] = cmul[h];
#pragma unroll 1
        for (int i0 = score_split(rows) + tid; i0 < rows; i0 += kScoreRows * kTcCompute) {
          float wv[kScoreRows], asv[kScoreRows];
#pragma unroll
          for (int jr = 0; jr < kScoreRows; ++jr) {
            const int i = i0 + jr * kTcCompute;
            wv[jr] = 0.f;
            asv[jr] = 0.f;
            if (i < rows) {
              wv[jr] = w_s[i];
              asv[jr] = group_dot<G>(lg + (size_t)i * G, cm);
            }
          }
#pragma unroll
          for (int jr = 0; jr < kScoreRows; ++jr) {
            const int i = i0 + jr * kTcCompute;
            const int slot = base + i;
            if (i >= rows) break;
            if (slot == rl.excl) continue;
            const float sc = fabsf(wv[jr]) * asv[jr];
            if (is_candidate(wv[jr]) && better(sc, slot, bs, bi)) {
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
        esc_s[warp] = bs;
        esc_i[warp] = bi;
        mbar_arrive(escore);
      }
      if (!ok && tid == 0) {
        *fail_any = 1;
        atomicOr(a.err, LF_DEVERR_TIMEOUT);
      }
    };
    int kt = 0, ne = 0, pt = 0;
    for (int k = 0; k < nitems; ++k) {
      int n, p, base;
      bool state_ok;
      const int rows = unit_rows(k, n, p, state_ok, base);
      const int ntile = (rows + kTcTile - 1) / kTcTile;
      const int b2 = k & 1;
      float* lg = lgbase + (size_t)(b2 & lgpar) * chunk * G;
      float* o_part = opbase + (size_t)b2 * G * D;
      const float* vn_s = reinterpret_cast<const float*>(vnbase + b2 * P::vn_bytes(chunk));
      const int32_t* pos_s =
          reinterpret_cast<const int32_t*>(vnbase + (2 + b2) * P::vn_bytes(chunk));
      float* w_s = reinterpret_cast<float*>(vnbase + (4 + b2) * P::vn_bytes(chunk));
      const int bud = items[kTcItemInts * k + 3];
      const UnitRule rl = unit_rule(a, n, p, items[kTcItemInts * k + 2], bud, state_ok);
      const int plim = rl.plim;  // a slot is a candidate iff sinks <= pos < plim (and not excl)
      const int excl = rl.excl - base;  // this CTA's row of the dropped slot (deferred)

      // The tail warps must be done with this parity's buffers (unit k - 2).
      bool bad = false;
      if (k >= 2)
        bad = !__all_sync(0xffffffffu, mbar_wait_bounded(&taildone[b2],
                                                         (uint32_t)(((k >> 1) - 1) & 1)));
      bad = bad || !__all_sync(0xffffffffu,
                               mbar_wait_bounded(&aux[b2], (uint32_t)((k >> 1) & 1)));

      // Phase A epilogue: logits of this CTA's slots, their max, candidate weights.
      float mx[G];
#pragma unroll
      for (int h = 0; h < G; ++h) mx[h] = -INFINITY;
#pragma unroll 1
      for (int t = 0; t < ntile && !bad; ++t, ++kt) {
        const int buf = kt % kTcSBufs;
        if (!__all_sync(0xffffffffu,
                        mbar_wait_bounded(&sfull[buf], (uint32_t)((kt / kTcSBufs) & 1)))) {
          bad = true;
          break;
        }
        tc_fence_after();
        float acc[8];
        tmem_ld8(tmem + 16 * buf + ((uint32_t)(warp * 32) << 16), acc);
        tmem_wait_ld();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sfree[buf]);
        const int i = t * kTcTile + tid;
        if (i < rows) {
          const bool dropped = (i == excl);
#pragma unroll
          for (int h = 0; h < G; ++h) {
            const float s = dropped ? -INFINITY : acc[h] * a.scale_log2;
            lg[(size_t)i * G + h] = s;
            mx[h] = fmaxf(mx[h], s);
          }
          if (lgpar) {
            const int ps = pos_s[i];
            const bool cand = !dropped && ps < plim && ps >= a.sinks;
            w_s[i] = cand ? vn_s[i] : flag_protected(vn_s[i]);
          }
        }
      }
      const bool any_bad = named_bar_or(1, kTcCompute, bad);
      // The raw ||v||_1 / positions buffer may be refilled for unit k + 2.
      if (lane == 0) mbar_arrive(&auxfree[b2]);
      bool bad2 = false;
      if (rows > 0 && !any_bad) {
#pragma unroll
        for (int h = 0; h < G; ++h) mx[h] = warp_max(mx[h]);
        if (lane == 0)
#pragma unroll
          for (int h = 0; h < G; ++h) red[warp * kMaxGroup + h] = mx[h];
        named_bar_sync(1, kTcCompute);
        float ml[G], sm[G];
#pragma unroll
        for (int h = 0; h < G; ++h) {
          float m = -INFINITY;
          for (int w = 0; w < 4; ++w) m = fmaxf(m, red[w * kMaxGroup + h]);
          ml[h] = m;
          sm[h] = 0.f;
        }
        // p = 2^(s - m) (kept in fp32 for the score) and the bf16 hi/lo P^T operand,
        // ahead of the MMAs in a ring of kTcPBufs tiles; slots past `rows` are zero.
#pragma unroll 1
        for (int vt = 0; vt < ntile; ++vt, ++pt) {
          const int pb = pt % kTcPBufs;
          if (pt >= kTcPBufs &&
              !__all_sync(0xffffffffu, mbar_wait_bounded(&pfree[pb],
                                                         (uint32_t)(((pt / kTcPBufs) - 1) & 1)))) {
            bad2 = true;  // the MMA warp stopped; it reports the error
            break;
          }
          const int i = vt * kTcTile + tid;
          unsigned char* ptb = ptile + (size_t)pb * P::kPTile + ((tid >> 6) & 1) * 2048;
          const int c = tid & 63;
#pragma unroll
          for (int h = 0; h < G; ++h) {
            float pv = 0.f;
            if (i < rows) {
              const float x = lg[(size_t)i * G + h];
              pv = (x == -INFINITY) ? 0.f : exp2f(x - ml[h]);  // the dropped slot: 0
              lg[(size_t)i * G + h] = pv;
              sm[h] += pv;
            }
            const T hi = __float2bfloat16_rn(pv);
            const T lo = __float2bfloat16_rn(pv - __bfloat162float(hi));
            *reinterpret_cast<T*>(ptb + sw128_offset(h, c)) = hi;
            *reinterpret_cast<T*>(ptb + sw128_offset(G + h, c)) = lo;
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(&pready[pb]);
        }
#pragma unroll
        for (int h = 0; h < G; ++h) sm[h] = warp_sum(sm[h]);
        named_bar_sync(1, kTcCompute);  // every warp has read red[] (the maxima)
        if (lane == 0)
#pragma unroll
          for (int h = 0; h < G; ++h) red[warp * kMaxGroup + h] = sm[h];
        named_bar_sync(1, kTcCompute);
        if (tid < G) {
          float sl = 0.f;
          for (int w = 0; w < 4; ++w) sl += red[w * kMaxGroup + tid];
          m_loc[b2 * kMaxGroup + tid] = ml[tid];
          l_loc[b2 * kMaxGroup + tid] = sl;
        }
        // This CTA's (m, l), logits and candidate weights are final: the tail
        // warps exchange and score them while the unit's V tiles still stream.
        __syncwarp();
        if (tid == 0) {
          if (is_piece(k)) publish_stats(k, b2);
          mbar_arrive(&statrdy[b2]);
        }
        if (last_shared_scoring(k, rl)) epilogue_scores(rows, base, rl, lg, w_s, !bad2);
        // The output accumulator: thread e <-> TMEM lane e <-> output element e.
        if (!bad2 && __all_sync(0xffffffffu, mbar_wait_bounded(ofull, (uint32_t)(ne & 1)))) {
          tc_fence_after();
          float o[16];
          tmem_ld16(tO + ((uint32_t)(warp * 32) << 16), o);
          tmem_wait_ld();
          tc_fence_before();
#pragma unroll
          for (int h = 0; h < G; ++h) o_part[h * D + tid] = o[h] + o[G + h];
        } else {
          bad2 = true;
        }
      } else {
        // Nothing of this unit here (or a wait ran out): no statistics.
        if (tid < G) {
          m_loc[b2 * kMaxGroup + tid] = -INFINITY;
          l_loc[b2 * kMaxGroup + tid] = 0.f;
        }
        __syncwarp();
        if (tid == 0) {
          if (is_piece(k)) publish_stats(k, b2);
          mbar_arrive(&statrdy[b2]);
        }
        if (last_shared_scoring(k, rl)) epilogue_scores(rows, base, rl, lg, w_s, false);
      }
      if (rows > 0) ne += 1;
      const bool failed = any_bad || named_bar_or(1, kTcCompute, bad2);
      if (rows == 0 || failed) {
#pragma unroll
        for (int h = 0; h < G; ++h) o_part[h * D + tid] = 0.f;
      }
      if (tid == 0) uflag[b2] = failed ? 1 : 0;
      if (failed && tid == 0) {
        *fail_any = 1;
        atomicOr(a.err, LF_DEVERR_TIMEOUT);
      }
      // Hand the unit over to the tail warps (release of the writes above).
      named_bar_sync(1, kTcCompute);
      if (lane == 0) mbar_arrive(&handoff[b2]);
    }
  } else {
    // ---- tail warps 6-7: exchange, exact scores, leader's output and eviction -----
    const int tt_id = tid - kTcTailWarp0 * 32;  // 0..63
    const int twarp = tt_id >> 5;
    // The new token's k and v and the group's queries of an item, in 16-byte
    // chunks, loaded into registers one item ahead: under a saturated HBM their
    // latency is microseconds, and it passes while the tail works on the
    // previous unit.  Tail thread t holds query chunks c = t + 64 i (head c / 16,
    // elements 8 (c mod 16) ...), key chunk t mod 16 and, for t < 16, value chunk t.
    constexpr int kNq = (G * 16 + kTcTail - 1) / kTcTail;
    uint4 nq[kNq], nk = make_uint4(0, 0, 0, 0), nv = make_uint4(0, 0, 0, 0);
    auto load_new = [&](int kk) {
      const int uu = unit_of(kk);
      const int bb = uu / a.kv_heads;
      const uint4* qs = reinterpret_cast<const uint4*>(
          reinterpret_cast<const T*>(a.q) + ((size_t)bb * a.q_heads + (size_t)(uu - bb * a.kv_heads) * G) * D);
#pragma unroll
      for (int i = 0; i < kNq; ++i) {
        const int c = tt_id + kTcTail * i;
        nq[i] = (c < G * 16) ? qs[c] : make_uint4(0, 0, 0, 0);
      }
      nk = reinterpret_cast<const uint4*>(reinterpret_cast<const T*>(a.k_new) + (size_t)uu * D)[tt_id & 15];
      if (tt_id < 16)
        nv = reinterpret_cast<const uint4*>(reinterpret_cast<const T*>(a.v_new) + (size_t)uu * D)[tt_id];
    };
    if (nitems > 0) load_new(0);
    for (int k = 0; k < nitems; ++k) {
      int n, p, base;
      bool state_ok;
      const int rows = unit_rows(k, n, p, state_ok, base);
      const int u = unit_of(k);
      const int b = u / a.kv_heads;
      const int g = u - b * a.kv_heads;
      const int bud = items[kTcItemInts * k + 3];
      const int pend = items[kTcItemInts * k + 2];
      const UnitRule rl = unit_rule(a, n, p, pend, bud, state_ok);
      const bool h2o = a.evict && a.score == LF_SCORE_H2O;
      const bool layer = a.evict && a.scope == LF_SCOPE_LAYER;
      const int b2 = k & 1;
      const float* lg = lgbase + (size_t)(b2 & lgpar) * chunk * G;
      const float* o_part = opbase + (size_t)b2 * G * D;
      const float* w_s = reinterpret_cast<const float*>(vnbase + (4 + b2) * P::vn_bytes(chunk));
      const size_t ubase = (size_t)u * a.slot_stride;
      float* snw = s_new + b2 * kMaxGroup;
      const float* mlc = m_loc + b2 * kMaxGroup;
      const float* llc = l_loc + b2 * kMaxGroup;
      // The new token's k and v in shared memory for the leader's output and slot
      // write (the barrier after the statistics wait below orders the copy for
      // both tail warps), and its logits (every CTA computes them): the dot
      // products of this thread's query chunks with the key chunk, summed over
      // the 16 threads of a head.
      T* nkv = reinterpret_cast<T*>(smem + P::kOffNew) + (size_t)b2 * 2 * D;  // [k | v]
      if (tt_id < 16) {
        reinterpret_cast<uint4*>(nkv)[tt_id] = nk;
        reinterpret_cast<uint4*>(nkv + D)[tt_id] = nv;
      }
#pragma unroll
      for (int i = 0; i < kNq; ++i) {
        const int c = tt_id + kTcTail * i;
        const uint32_t qw[4] = {nq[i].x, nq[i].y, nq[i].z, nq[i].w};
        const uint32_t kw[4] = {nk.x, nk.y, nk.z, nk.w};
        float s = 0.f;
#pragma unroll
        for (int x = 0; x < 4; ++x) {
          const float2 qf = bf2_to_f2(qw[x]);
          const float2 kf = bf2_to_f2(kw[x]);
          s = fmaf(qf.x, kf.x, s);
          s = fmaf(qf.y, kf.y, s);
        }
#pragma unroll
        for (int o = 8; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
        if ((tt_id & 15) == 0 && c < G * 16) snw[c >> 4] = s * a.scale_log2;
      }
      // The next item's, in the background.
      if (k + 1 < nitems) load_new(k + 1);
      // This CTA's (m, l), logits and weights: exchanged and scored while the
      // unit's V tiles still stream.
      const bool got_loc = __all_sync(
          0xffffffffu, mbar_wait_bounded(&statrdy[b2], (uint32_t)((k >> 1) & 1)));
      named_bar_sync(2, kTcTail);
      // The partial output and the unit's failure flag, once the output
      // accumulator is read (the epilogue's hand-off).  Every tail thread calls it.
      auto unit_handoff = [&]() -> bool {
        const bool got = __all_sync(
            0xffffffffu, mbar_wait_bounded(&handoff[b2], (uint32_t)((k >> 1) & 1)));
        named_bar_sync(2, kTcTail);
        return !got || !got_loc || uflag[b2] != 0;
      };

      if constexpr (kSplit) {
        if (is_piece(k)) {
          // ---- a unit shared with other clusters (a planned launch): both
          // exchanges go through global memory, counted by atomics.  The parts
          // are the CTAs of the clusters whose ranges meet the unit, in
          // cluster then rank order; part 0 leads. ----
          const int part = items[kTcItemInts * k + 7];
          const int xi = part >> 16;                      // exchange slot
          const int np = (part & 0xff) * C;               // parts (<= kMaxSplitParts)
          const int me = ((part >> 8) & 0xff) * C + rank; // this CTA's part
          constexpr int kFinF = G * D + 4;  // floats per part: output, score, slot, flag
          int* cnt = ta.split_cnt + 2 * xi;
          const float* gst = ta.split_stat + (size_t)xi * kMaxSplitParts * 2 * kMaxGroup;
          float* gfn = ta.split_fin + (size_t)xi * kMaxSplitParts * kFinF;
          // local copy (not stat_in: a cluster peer may already be sending the
          // next whole unit's statistics there)
          float* sst = reinterpret_cast<float*>(smem + P::kOffPieceStats);
          // Exchange 1: every part's (m_h, l_h), published by the epilogue warps.
          if (tt_id == 0) {
            split_flag[0] = wait_count_bounded(cnt, np) ? 1 : 0;
            __threadfence();
          }
          named_bar_sync(2, kTcTail);
          const bool got_stats = split_flag[0] != 0;
          for (int i = tt_id; i < np * 2 * kMaxGroup; i += kTcTail) sst[i] = __ldcg(gst + i);
          named_bar_sync(2, kTcTail);
          if (tt_id < G) {
            const int h = tt_id;
            float M = snw[h];
#pragma unroll 1
            for (int r = 0; r < np; ++r) M = fmaxf(M, sst[r * 2 * kMaxGroup + h]);
            float L = exp2f(snw[h] - M);
#pragma unroll 1
            for (int r = 0; r < np; ++r) {
              const float mr = sst[r * 2 * kMaxGroup + h];
              if (mr != -INFINITY) L += sst[r * 2 * kMaxGroup + kMaxGroup + h] * exp2f(mr - M);
            }
            m_glb[h] = M;
            l_glb[h] = L;
            cmul[h] = (mlc[h] != -INFINITY) ? exp2f(mlc[h] - M) / L : 0.f;
            // the leader's output scales: each part's, then the new token's
#pragma unroll 1
            for (int r = 0; r < np; ++r) {
              const float mr = sst[r * 2 * kMaxGroup + h];
              osc[r * kMaxGroup + h] = (mr != -INFINITY) ? exp2f(mr - M) / L : 0.f;
            }
            osc[np * kMaxGroup + h] = exp2f(snw[h] - M) / L;
            if (!(isfinite(M) && isfinite(L) && L > 0.f)) atomicOr(a.err, LF_DEVERR_NONFINITE);
          }
          const bool stats_ok = !named_bar_or(2, kTcTail, !got_stats);
          if (!stats_ok && tt_id == 0) {
            *fail_any = 1;
            atomicOr(a.err, LF_DEVERR_TIMEOUT);
          }
          // Exact scores of this CTA's slots, its lowest candidate (LongFlow:
          // ||v_i|| sum_h alpha_{h,i}; H2O: the slot's accumulator plus this
          // step's sum_h alpha_{h,i}, scored on every step to update it).  Layer
          // scope: every score goes to the scratch for the selection kernel,
          // after the hand-off, so that a failed unit leaves it alone.
          const bool early = !layer;
          bool unit_failed = early ? false : unit_handoff();
          float bs = INFINITY;
          int bi = INT_MAX;
          const bool pscoring = (rl.choosing || h2o) && !unit_failed && got_loc && stats_ok;
          if (pscoring && (rl.choosing || layer)) {
            float cm[G];
#pragma unroll
            for (int h = 0; h < G; ++h) cm[h] = cmul[h];
            if (!layer) {
#pragma unroll 1
              for (int i0 = tt_id; i0 < rows; i0 += kScoreRows * kTcTail) {
                float wv[kScoreRows], asv[kScoreRows];
#pragma unroll
                for (int jr = 0; jr < kScoreRows; ++jr) {
                  const int i = i0 + jr * kTcTail;
                  wv[jr] = 0.f;
                  asv[jr] = 0.f;
                  if (i < rows) {
                    wv[jr] = w_s[i];
                    asv[jr] = group_dot<G>(lg + (size_t)i * G, cm);
                  }
                }
#pragma unroll
                for (int jr = 0; jr < kScoreRows; ++jr) {
                  const int i = i0 + jr * kTcTail;
                  const int slot = base + i;
                  if (i >= rows) break;
                  const float w = wv[jr];
                  const float sc = h2o ? fabsf(w) + asv[jr] : fabsf(w) * asv[jr];
                  if (slot != rl.excl && rl.choosing && is_candidate(w) && better(sc, slot, bs, bi)) {
                    bs = sc;
                    bi = slot;
                  }
                }
              }
            } else {
#pragma unroll 1
              for (int i = tt_id; i < rows; i += kTcTail) {
                const int slot = base + i;
                if (slot == rl.excl) {
                  if (rl.choosing) a.lw_score[ubase + slot] = INFINITY;
                  continue;
                }
                const float w = w_s[i];
                const float as = group_dot<G>(lg + (size_t)i * G, cm);
                const float sc = h2o ? fabsf(w) + as : fabsf(w) * as;
                if (h2o) a.acc[ubase + slot] = sc;
                if (rl.choosing) a.lw_score[ubase + slot] = is_candidate(w) ? sc : INFINITY;
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
            red_t[twarp] = bs;
            red_ti[twarp] = bi;
          }
          named_bar_sync(2, kTcTail);
          if (early) unit_failed = unit_handoff();
          // H2O, per-KV-head scope: write back the accumulators of this part's
          // slots except the dropped slot and the part's lowest candidate, which
          // the leader writes (it may be the victim, which takes the new token's).
          if (pscoring && h2o && !layer && !unit_failed) {
            int ci = red_ti[0];
            if (better(red_t[1], red_ti[1], red_t[0], red_ti[0])) ci = red_ti[1];
            float cm[G];
#pragma unroll
            for (int h = 0; h < G; ++h) cm[h] = cmul[h];
#pragma unroll 1
            for (int i = tt_id; i < rows; i += kTcTail) {
              const int slot = base + i;
              if (slot == rl.excl || slot == ci) continue;
              a.acc[ubase + slot] = fabsf(w_s[i]) + group_dot<G>(lg + (size_t)i * G, cm);
            }
          }
          // Exchange 2: partial output, lowest (score, slot) and failure flag to part 0.
          for (int c = tt_id; c < G * D; c += kTcTail) gfn[(size_t)me * kFinF + c] = o_part[c];
          if (tt_id == 0) {
            float cs = red_t[0];
            int ci = red_ti[0];
            if (better(red_t[1], red_ti[1], cs, ci)) {
              cs = red_t[1];
              ci = red_ti[1];
            }
            const bool fl = unit_failed || !stats_ok || *fail_any;
            gfn[(size_t)me * kFinF + G * D] = cs;
            gfn[(size_t)me * kFinF + G * D + 1] = __int_as_float(ci);
            gfn[(size_t)me * kFinF + G * D + 2] = fl ? 1.f : 0.f;
          }
          __threadfence();
          named_bar_sync(2, kTcTail);
          if (tt_id == 0) atomicAdd(cnt + 1, 1);
          if (me == 0) {
            if (tt_id == 0) {
              split_flag[0] = wait_count_bounded(cnt + 1, np) ? 1 : 0;
              __threadfence();
            }
            named_bar_sync(2, kTcTail);
            const bool all_got = split_flag[0] != 0;
            // Every part's lowest (score, slot) and failure flag: one part per
            // lane of warp 0, loaded together, then reduced.
            float fs = INFINITY;
            int fi = INT_MAX;
            bool any_fail = !all_got || !stats_ok;
            float rs = INFINITY;   // warp 0, lane r < np: part r's lowest (score, slot)
            int ri = INT_MAX;
            if (twarp == 0) {
              float rf = 0.f;
              if (lane < np) {
                const float* tl = gfn + (size_t)lane * kFinF + G * D;
                rs = __ldcg(tl);
                ri = __float_as_int(__ldcg(tl + 1));
                rf = __ldcg(tl + 2);
              }
              any_fail = any_fail || __any_sync(0xffffffffu, rf != 0.f);
              fs = rs;
              fi = ri;
#pragma unroll
              for (int o = 16; o > 0; o >>= 1) {
                const float os = __shfl_xor_sync(0xffffffffu, fs, o);
                const int oi = __shfl_xor_sync(0xffffffffu, fi, o);
                if (better(os, oi, fs, fi)) {
                  fs = os;
                  fi = oi;
                }
              }
            }
            if (twarp == 1) {
              // Output (warp 1): the new token + every part's partial output, in part
              // order; each part's elements of this lane loaded together.
              if (all_got && stats_ok) {
                constexpr int kEl = G * D / 32;
                T* og = reinterpret_cast<T*>(a.out) + ((size_t)b * a.q_heads + (size_t)g * G) * D;
                float acc[kEl];
#pragma unroll
                for (int i = 0; i < kEl; ++i) {
                  const int h = (lane + 32 * i) / D;
                  const int e = (lane + 32 * i) - h * D;
                  acc[i] = to_f32(nkv[D + e]) * osc[np * kMaxGroup + h];
                }
#pragma unroll 1
                for (int r = 0; r < np; ++r) {
                  float part[kEl];
#pragma unroll
                  for (int i = 0; i < kEl; ++i)
                    part[i] = __ldcg(gfn + (size_t)r * kFinF + lane + 32 * i);
#pragma unroll
                  for (int i = 0; i < kEl; ++i)
                    acc[i] = fmaf(part[i], osc[r * kMaxGroup + (lane + 32 * i) / D], acc[i]);
                }
#pragma unroll
                for (int i = 0; i < kEl; ++i) {
                  const int idx = lane + 32 * i;
                  const int h = idx / D;
                  from_f32(acc[i], &og[(size_t)h * D + (idx - h * D)]);
                }
              }
            } else {
              // The decision and the slot write (warp 0), beside the output.
              float anew = 0.f;
              if (lane == 0) {
#pragma unroll
                for (int h = 0; h < G; ++h) anew += osc[np * kMaxGroup + h];
                const LeaderOut d =
                    leader_decide(a, u, n, p, pend, bud, state_ok, any_fail, rl, fi, anew);
                decision[0] = d.slot;
                // every part is through both exchanges: ready for the next launch
                cnt[0] = 0;
                cnt[1] = 0;
              }
              __syncwarp();
              const int slot = decision[0];
              // H2O, per-KV-head scope: the accumulators of the parts' lowest
              // candidates (their scores), except the slot the new token takes.
              if (h2o && !layer && state_ok && !__any_sync(0xffffffffu, any_fail) && lane < np &&
                  ri != INT_MAX && ri != slot)
                a.acc[ubase + ri] = rs;
              if (slot >= 0) write_slot<T, D>(a, ubase, slot, nkv, nkv + D, p, anew, lane, 32);
            }
          }
          named_bar_sync(2, kTcTail);
          if (lane == 0) mbar_arrive(&taildone[b2]);
          continue;
        }
      }

      // Exchange 1: every CTA's (m_h, l_h) to every CTA of the cluster.
      float* sin = stat_in + (size_t)b2 * kMaxCluster * 2 * kMaxGroup;
      if (tt_id == 0) {
        mbar_arrive_expect_tx(&statb[b2], (uint32_t)(C * 2 * kMaxGroup * 4));
        const uint32_t src = smem_u32(sin + (size_t)rank * 2 * kMaxGroup);
        const uint32_t bar = smem_u32(&statb[b2]);
        uint32_t v[2 * kMaxGroup];
#pragma unroll
        for (int h = 0; h < kMaxGroup; ++h) {
          v[h] = __float_as_uint(h < G ? mlc[h] : -INFINITY);
          v[kMaxGroup + h] = __float_as_uint(h < G ? llc[h] : 0.f);
        }
#pragma unroll 1
        for (int r = 0; r < C; ++r) {
          const uint32_t ra = mapa_u32(src, (uint32_t)r);
          const uint32_t rb = mapa_u32(bar, (uint32_t)r);
#pragma unroll
          for (int q4 = 0; q4 < 2 * kMaxGroup; q4 += 4)
            st_async_v4(ra + q4 * 4, v[q4], v[q4 + 1], v[q4 + 2], v[q4 + 3], rb);
        }
      }
      // statb[b2] completes once per whole unit of parity b2 (the shared units
      // first in a planned launch do not use it).
      const int npc_items = planned ? npc : 0;
      const int k0 = npc_items + ((k - npc_items) & 1);  // first whole item of this parity
      const uint32_t stat_phase = (uint32_t)(((k - k0) >> 1) & 1);
      const bool got_stats = __all_sync(
          0xffffffffu, mbar_wait_cluster_bounded(&statb[b2], stat_phase));
      if (tt_id < G) {
        const int h = tt_id;
        float M = snw[h];
#pragma unroll 1
        for (int r = 0; r < C; ++r) M = fmaxf(M, sin[r * 2 * kMaxGroup + h]);
        float L = exp2f(snw[h] - M);
#pragma unroll 1
        for (int r = 0; r < C; ++r) {
          const float mr = sin[r * 2 * kMaxGroup + h];
          if (mr != -INFINITY) L += sin[r * 2 * kMaxGroup + kMaxGroup + h] * exp2f(mr - M);
        }
        m_glb[h] = M;
        l_glb[h] = L;
        cmul[h] = (mlc[h] != -INFINITY) ? exp2f(mlc[h] - M) / L : 0.f;
        // the leader's output scales: each CTA's, then the new token's
#pragma unroll 1
        for (int r = 0; r < C; ++r) {
          const float mr = sin[r * 2 * kMaxGroup + h];
          osc[r * kMaxGroup + h] = (mr != -INFINITY) ? exp2f(mr - M) / L : 0.f;
        }
        osc[C * kMaxGroup + h] = exp2f(snw[h] - M) / L;
        if (!(isfinite(M) && isfinite(L) && L > 0.f)) atomicOr(a.err, LF_DEVERR_NONFINITE);
      }
      const bool stats_ok = !named_bar_or(2, kTcTail, !got_stats);
      if (!stats_ok && tt_id == 0) {
        *fail_any = 1;
        atomicOr(a.err, LF_DEVERR_TIMEOUT);
      }

      // Exact scores of this CTA's slots and the lowest (score, slot) of its
      // candidates.  LongFlow: ||v_i|| sum_h alpha_{h,i}.  H2O: the slot's
      // accumulator plus this step's sum_h alpha_{h,i}.  Layer scope: every score
      // goes to the scratch for the selection kernel, and the H2O accumulators
      // are written back here.  The per-KV-head scores are taken before the
      // hand-off; every write to global memory (the scratch, the accumulators)
      // waits for it, so that a failed unit leaves them alone.
      const bool early = !layer;
      bool unit_failed = early ? false : unit_handoff();
      float bs = INFINITY;
      int bi = INT_MAX;
      const bool scoring = (rl.choosing || h2o) && !unit_failed && got_loc && stats_ok;
      // The launch's last unit: the epilogue warps score the rows from `srows` on.
      const bool shared_last = last_shared_scoring(k, rl);
      const int srows = shared_last ? score_split(rows) : rows;
      if (shared_last && tt_id == 0) {
        gscore_ok[0] = scoring ? 1 : 0;
        mbar_arrive(gstat);  // the scales (cmul) are final: the named barrier above
      }
      if (scoring) {
        float cm[G];
#pragma unroll
        for (int h = 0; h < G; ++h) cm[h] = cmul[h];
        if (!layer) {
          // The lowest (score, slot) of this CTA's candidates, kScoreRows rows per
          // pass with their loads issued together (the result does not depend on
          // the order rows are visited in).
#pragma unroll 1
          for (int i0 = tt_id; i0 < srows; i0 += kScoreRows * kTcTail) {
            float wv[kScoreRows], asv[kScoreRows];
#pragma unroll
            for (int jr = 0; jr < kScoreRows; ++jr) {
              const int i = i0 + jr * kTcTail;
              wv[jr] = 0.f;
              asv[jr] = 0.f;
              if (i < srows) {
                wv[jr] = w_s[i];
                asv[jr] = group_dot<G>(lg + (size_t)i * G, cm);
              }
            }
#pragma unroll
            for (int jr = 0; jr < kScoreRows; ++jr) {
              const int i = i0 + jr * kTcTail;
              const int slot = base + i;
              if (i >= srows) break;
              const float w = wv[jr];
              const float sc = h2o ? fabsf(w) + asv[jr] : fabsf(w) * asv[jr];
              if (slot != rl.excl && rl.choosing && is_candidate(w) && better(sc, slot, bs, bi)) {
                bs = sc;
                bi = slot;
              }
            }
          }
        } else {
          // Layer scope: every score to the scratch (+inf for a non-candidate),
          // and the H2O accumulators written back.
#pragma unroll 1
          for (int i = tt_id; i < srows; i += kTcTail) {
            const int slot = base + i;
            if (slot == rl.excl) {
              if (rl.choosing) a.lw_score[ubase + slot] = INFINITY;
              continue;
            }
            const float w = w_s[i];
            const float as = group_dot<G>(lg + (size_t)i * G, cm);
            const float sc = h2o ? fabsf(w) + as : fabsf(w) * as;
            if (h2o) a.acc[ubase + slot] = sc;
            if (rl.choosing) a.lw_score[ubase + slot] = is_candidate(w) ? sc : INFINITY;
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
        red_t[twarp] = bs;
        red_ti[twarp] = bi;
      }
      named_bar_sync(2, kTcTail);
      if (early) unit_failed = unit_handoff();
      // H2O, per-KV-head scope: write back the accumulators of this CTA's slots
      // except the dropped slot and the CTA's lowest candidate.  The leader
      // writes that one (it may be the victim, which takes the new token's), so
      // no slot has two writers.
      if (scoring && h2o && !layer && !unit_failed) {
        int ci = red_ti[0];
        float cs = red_t[0];
        if (better(red_t[1], red_ti[1], cs, ci)) ci = red_ti[1];
        float cm[G];
#pragma unroll
        for (int h = 0; h < G; ++h) cm[h] = cmul[h];
#pragma unroll 1
        for (int i = tt_id; i < rows; i += kTcTail) {
          const int slot = base + i;
          if (slot == rl.excl || slot == ci) continue;
          const float as = group_dot<G>(lg + (size_t)i * G, cm);
          a.acc[ubase + slot] = fabsf(w_s[i]) + as;
        }
      }

      // Exchange 2: partial output and lowest (score, slot) to the unit's leader.
      // One receive buffer suffices: a peer can send the leader's next unit only
      // after the leader has sent its own statistics for it, i.e. finished this one.
      const int leader = (k - npc_items) % C;
      unsigned char* fin = fin_in;
      if (rank == leader && tt_id == 0) mbar_arrive_expect_tx(finb, (uint32_t)(C * P::kFinBytes));
      {
        const uint32_t dst = mapa_u32(smem_u32(fin + (size_t)rank * P::kFinBytes), (uint32_t)leader);
        const uint32_t rb = mapa_u32(smem_u32(finb), (uint32_t)leader);
        for (int c = tt_id; c < G * D / 4; c += kTcTail) {
          const uint4 v = *reinterpret_cast<const uint4*>(o_part + c * 4);
          st_async_v4(dst + c * 16, v.x, v.y, v.z, v.w, rb);
        }
        if (tt_id == 0) {
          if (better(red_t[1], red_ti[1], bs, bi)) {
            bs = red_t[1];
            bi = red_ti[1];
          }
          if (shared_last) {  // the epilogue warps' share
            if (!mbar_wait_bounded(escore, 0)) {
              *fail_any = 1;
              atomicOr(a.err, LF_DEVERR_TIMEOUT);
            }
            for (int w = 0; w < 4; ++w)
              if (better(esc_s[w], esc_i[w], bs, bi)) {
                bs = esc_s[w];
                bi = esc_i[w];
              }
          }
          const uint32_t flag = (unit_failed || !stats_ok || *fail_any) ? 1u : 0u;
          st_async_v4(dst + G * D * 4, __float_as_uint(bs), (uint32_t)bi, flag, 0u, rb);
        }
      }
      if (rank == leader) {
        // finb completes once per whole unit this CTA leads (not for a shared unit).
        const uint32_t fin_phase = (uint32_t)(((k - npc_items) / C) & 1);
        const bool got = __all_sync(0xffffffffu, mbar_wait_cluster_bounded(finb, fin_phase));
        const bool all_got = !named_bar_or(2, kTcTail, !got);
        if (twarp == 1) {
          // Output (warp 1): the new token + every CTA's partial output, in rank
          // order.  Lane l takes elements [4l, 4l + 4) of every head row, each
          // CTA's rows loaded together as 16-byte vectors.
          if (all_got && stats_ok) {
            static_assert(D == 32 * 4, "four elements of a head row per lane");
            T* og = reinterpret_cast<T*>(a.out) + ((size_t)b * a.q_heads + (size_t)g * G) * D;
            const int e0 = lane * 4;
            float acc[G][4];
#pragma unroll
            for (int h = 0; h < G; ++h) {
              const float sn = osc[C * kMaxGroup + h];
#pragma unroll
              for (int x = 0; x < 4; ++x) acc[h][x] = to_f32(nkv[D + e0 + x]) * sn;
            }
#pragma unroll 1
            for (int r = 0; r < C; ++r) {
              const float* fr = reinterpret_cast<const float*>(fin + (size_t)r * P::kFinBytes);
              float4 pr[G];
#pragma unroll
              for (int h = 0; h < G; ++h) pr[h] = *reinterpret_cast<const float4*>(fr + h * D + e0);
#pragma unroll
              for (int h = 0; h < G; ++h) {
                const float sc = osc[r * kMaxGroup + h];
                acc[h][0] = fmaf(pr[h].x, sc, acc[h][0]);
                acc[h][1] = fmaf(pr[h].y, sc, acc[h][1]);
                acc[h][2] = fmaf(pr[h].z, sc, acc[h][2]);
                acc[h][3] = fmaf(pr[h].w, sc, acc[h][3]);
              }
            }
#pragma unroll
            for (int h = 0; h < G; ++h)
#pragma unroll
              for (int x = 0; x < 4; ++x) from_f32(acc[h][x], &og[(size_t)h * D + e0 + x]);
          }
        } else {
          // The decision and the slot write (warp 0), beside the output.
          float anew = 0.f;  // the new token's attention mass (lane 0)
          if (lane == 0) {
            bool any_fail = !all_got || !stats_ok;
            float fs = INFINITY;
            int fi = INT_MAX;
#pragma unroll 1
            for (int r = 0; r < C; ++r) {
              const uint32_t* tail =
                  reinterpret_cast<const uint32_t*>(fin + (size_t)r * P::kFinBytes + G * D * 4);
              any_fail = any_fail || tail[2] != 0;
              const float rs = __uint_as_float(tail[0]);
              const int ri = (int)tail[1];
              if (better(rs, ri, fs, fi)) {
                fs = rs;
                fi = ri;
              }
            }
#pragma unroll
            for (int h = 0; h < G; ++h) anew += osc[C * kMaxGroup + h];
            const LeaderOut d =
                leader_decide(a, u, n, p, pend, bud, state_ok, any_fail, rl, fi, anew);
            decision[0] = d.slot;
            // H2O: the accumulators of the CTAs' lowest candidates (their scores),
            // except the slot the new token takes.
            if (h2o && !layer && state_ok && !any_fail)
#pragma unroll 1
              for (int r = 0; r < C; ++r) {
                const uint32_t* tail =
                    reinterpret_cast<const uint32_t*>(fin + (size_t)r * P::kFinBytes + G * D * 4);
                const int ri = (int)tail[1];
                if (ri != INT_MAX && ri != d.slot) a.acc[ubase + ri] = __uint_as_float(tail[0]);
              }
          }
          __syncwarp();
          const int slot = decision[0];
          if (slot >= 0) write_slot<T, D>(a, ubase, slot, nkv, nkv + D, p, anew, lane, 32);
        }
      }
      // Release this parity's buffers (logits, partial output, statistics).
      named_bar_sync(2, kTcTail);
      if (lane == 0) mbar_arrive(&taildone[b2]);
    }
  }

  // ---- teardown ---------------------------------------------------------------
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, kTcTmemCols);
  }
  // No CTA leaves while a peer may still address its shared memory.
  cluster.sync();
}

}  // namespace lf
