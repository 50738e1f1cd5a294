// C ABI of the LongFlow fused decode step: cache creation, prefill, decode,
// error checks and the slab layout.  Declarations and semantics are in
// include/longflow.h.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <climits>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <new>
#include <string>
#include <vector>

#include "lf_decode_tc.cuh"
#include "lf_kernels.h"
#include "lf_rkv.h"
#include "longflow.h"

// A launch plan: every cluster takes `rounds` whole units round-robin (the
// units below rounds * nc), and before them one contiguous range of the units
// past the whole rounds, cut so that the clusters' loads come out level (parts
// first, so every cluster's parts start together and take about as long).
// When those units are few, only as many clusters take ranges as keep every
// shared unit within lf::kMaxSplitParts CTAs.
struct Plan {
  int rounds;
  int cut_unit[lf::kTcMaxPlan + 1], cut_slot[lf::kTcMaxPlan + 1];
};

struct lf_cache {
  int layers, batch, kv_heads, q_heads, head_dim, capacity, slot_stride, window;
  int dtype, evict, cluster, stages, chunk, smem, device;
  int score, norm, sinks, deferred, scope;  // the policy (zero unless LongFlow eviction, but norm)
  int kevict;     // what the decode kernels do: 1 LongFlow eviction, 0 append (off and R-KV)
  int rkv_buffer, rkv_alpha, rkv_beta;      // R-KV parameters (evict = LF_EVICT_RKV)
  float rkv_lambda, rkv_tau;
  int items;      // tensor-core path: units one cluster may visit per launch
  size_t elem_bytes;
  void* K;
  void* V;
  float* vnorm;
  int32_t* pos;
  int32_t* count;
  int32_t* next_pos;
  int32_t* budget;
  int32_t* err;
  int32_t* plen;  // [layers][batch] prompt lengths uploaded by lf_prefill_fill
  float* acc;     // H2O: attention mass per slot, else null
  int32_t* pending;   // deferred: chosen slot per unit, else null
  float* lw_score;    // layer scope: one layer's per-slot scores, else null
  int32_t* lw_req;    // layer scope: [batch][kv_heads] requests, else null
  float* lw_anew;     // layer scope: [batch][kv_heads] new tokens' attention mass
  void* small;    // one allocation holding vnorm..lw_anew
  lf::KernelEntry kern;
  int threads;    // CTA size of the decode kernel
  int grid_y;     // tensor-core path: resident clusters (persistent grid)
  int plan_ok;    // tensor-core path: planned launches allowed (policy and kernel)
  // Per layer and sequence, the host's count of occupied slots (the prompt plus
  // the decode steps since, capped at the sequence's limit; cut back by an R-KV
  // compression).  It only steers the launch plan: host state, ordered like the
  // calls; a wrong count costs balance, never correctness.
  std::vector<int32_t> occ;  // [layers][batch]
  std::vector<int32_t> occ_limit;  // [batch]: budget (LongFlow) or capacity (append modes)
  std::vector<int32_t> plan_n;     // scratch: one layer's counts per unit
  // Per layer, the occupancies of its last planning and the outcome: the same
  // counts give the same plan, so a layer in steady state plans once.
  std::vector<int32_t> memo_occ;       // [layers][batch]; -1: not planned yet
  std::vector<signed char> memo_used;  // [layers]: the plan was taken
  std::vector<Plan> memo_plan;         // [layers]
  float* split_stat;  // planned launches' exchanges through global memory (see TcArgs)
  float* split_fin;
  int32_t* split_cnt;
  CUtensorMap tmaps[4];  // tensor-core path: K and V as 2-D [rows][head_dim], two box heights
};

namespace {

thread_local std::string g_last_error;
thread_local int g_last_status = LF_OK;

// A call starts with no recorded failure.
void clear_last() {
  g_last_error.clear();
  g_last_status = LF_OK;
}

// Planned launches only once every sequence of the layer holds this many tokens
// (below it the exchanges through L2 cost more than the balance gains: measured
// at batch 32 on 2-CTA clusters, two-part shared units were 4-9% slower from
// 1408 slots down to 640, even at 1664, 7-9% faster from 2048 up).
#ifndef LF_PLAN_MIN_SLOTS
#define LF_PLAN_MIN_SLOTS 2048
#endif
constexpr int kPlanMinSlots = LF_PLAN_MIN_SLOTS;

// Slot rows per CTA below which a decode launch gets no prefetch hints.
constexpr long long kPrefetchMinRows = 2048;

// Host cost model of one launch, in CTA slot rows (one row of K and V streamed
// by one CTA, ~12.5 ns in a steady launch): every item a CTA visits adds a unit
// boundary, and every part of a shared unit adds its two exchanges through L2.
// Measured at batch 64 on 2-CTA clusters (512 units of 3276 slots on 76
// clusters): a plan of 6.74 units and two parts per cluster took 146.6 us per
// launch against 149.5 us for 7 whole units, about 1.3 us (~100 rows) per part.
#ifndef LF_PLAN_ITEM_COST
#define LF_PLAN_ITEM_COST 32
#endif
#ifndef LF_PLAN_PART_COST
#define LF_PLAN_PART_COST 64
#endif
constexpr long long kItemCost = LF_PLAN_ITEM_COST;
constexpr long long kPartCost = LF_PLAN_PART_COST;

// Costs every cluster of `pl` as the kernel will run it: false when a shared
// unit needs more than lf::kMaxSplitParts CTAs or a cluster more items than
// the table holds.  `worst` is the costliest cluster's cost and fixed[j] the
// part of cluster j's cost that its range adds beyond its slots (items, parts).
bool cost_plan(const Plan& pl, const std::vector<int32_t>& n, int c, int nc, int max_items,
               const std::vector<long long>& load, long long* worst,
               std::vector<long long>* fixed) {
  // Clusters sharing the unit of inner cut q: 1 + the unit's inner cuts, which
  // are consecutive (cuts never go back).
  int pos[lf::kTcMaxPlan + 1], tot[lf::kTcMaxPlan + 1];
  auto same = [&](int q, int r) {  // cuts q and r: inner cuts of one unit
    return pl.cut_slot[q] > 0 && pl.cut_slot[r] > 0 && pl.cut_unit[q] == pl.cut_unit[r];
  };
  for (int q = 1; q < nc; ++q) pos[q] = (q > 1 && same(q - 1, q)) ? pos[q - 1] + 1 : 1;
  for (int q = nc - 1; q >= 1; --q) tot[q] = (q + 1 < nc && same(q, q + 1)) ? tot[q + 1] : pos[q];
  auto parts_of = [&](int q) { return 1 + tot[q]; };
  *worst = 0;
  for (int j = 0; j < nc; ++j) {
    const int u0 = pl.cut_unit[j], s0 = pl.cut_slot[j];
    const int u1 = pl.cut_unit[j + 1], s1 = pl.cut_slot[j + 1];
    long long cost = load[j], fx = 0;
    int items = pl.rounds;
    if (s0 > 0) {
      const long long hi = (u1 == u0) ? s1 : n[u0];
      cost += (std::max(0LL, hi - s0) + c - 1) / c;
      fx += kItemCost + kPartCost;
      ++items;
      if (parts_of(j) * c > lf::kMaxSplitParts) return false;
    }
    if (s1 > 0 && !(s0 > 0 && u1 == u0)) {
      cost += ((long long)std::min(s1, n[u1]) + c - 1) / c;
      fx += kItemCost + kPartCost;
      ++items;
      if (parts_of(j + 1) * c > lf::kMaxSplitParts) return false;
    }
    for (int w = (s0 > 0) ? u0 + 1 : u0; w < u1; ++w) {  // units wholly inside the range
      cost += (n[w] + c - 1) / c;
      fx += kItemCost;
      ++items;
    }
    if (items > max_items) return false;
    (*fixed)[j] = fx;
    *worst = std::max(*worst, cost + fx);
  }
  return true;
}

// Cuts for level `level`: clusters 0, 1, ... take, in turn, the units past the
// whole rounds from where the last range ended, each as far as its cost stays
// within the level, every part and unit of the range paying its fixed cost
// where it falls.  False when the ranges end before the last unit does.
bool walk_plan(const std::vector<int32_t>& n, int c, int ncp, int nc, int first,
               const std::vector<long long>& load, double level, long long gran, long long least,
               Plan* pl) {
  const int units = (int)n.size();
  int u = first;
  long long s = 0;  // the walk's position: slot s of unit u
  pl->cut_unit[0] = first;
  pl->cut_slot[0] = 0;
  for (int j = 0; j < nc; ++j) {
    if (j < ncp && u < units) {
      double cap = (level - (double)load[j]) * c;  // slots left to this cluster
      while (u < units) {
        const long long rest = n[u] - s;
        const double fixed = (double)(kItemCost + (s > 0 ? kPartCost : 0)) * c;
        if ((double)rest + fixed <= cap) {  // the rest of unit u fits
          cap -= (double)rest + fixed;
          ++u;
          s = 0;
          continue;
        }
        // A part of unit u: from s, as many slots as the level leaves, on the grid.
        const double room = cap - (double)(kItemCost + kPartCost) * c;
        const long long x = room > 0 ? (long long)(room / (double)gran) * gran : 0;
        if (x >= least && rest - x >= least) {
          s += x;
        } else if (x >= least) {
          // The unit's tail would be short: leave the next range a part of
          // `least` slots, or take the whole unit when that leaves too little.
          const long long x2 = (rest - least) / gran * gran;
          if (x2 >= least) {
            s += x2;
          } else {
            ++u;
            s = 0;
          }
        }
        break;
      }
    }
    pl->cut_unit[j + 1] = (u < units) ? u : units;
    pl->cut_slot[j + 1] = (u < units) ? (int)s : 0;
  }
  return u >= units;
}

// Fills `pl` for units of n[u] occupied slots on nc clusters of c CTAs; returns
// the costliest cluster's cost (CTA slot rows), or -1 when no plan applies.
// Two ways to cut the ranges, the cheaper kept: lengths levelled on the
// clusters' loads alone (the fixed costs of parts and units fall where the
// cuts do), and the walk above at the lowest level that covers every unit.
long long make_plan(const std::vector<int32_t>& n, int c, int nc, int max_items, Plan* pl) {
  const int units = (int)n.size();
  const int rounds = units / nc, first = rounds * nc;
  if (first == units || nc > lf::kTcMaxPlan) return -1;
  const long long gran = 32LL * c;                      // cut points: 32 slots per CTA
  const long long least = (long long)lf::kTcTile * c;   // parts: one tile per CTA at least
  std::vector<long long> load((size_t)nc, 0);           // whole-unit cost per cluster
  for (int j = 0; j < nc; ++j)
    for (int k = 0; k < rounds; ++k) load[j] += (n[j + k * nc] + c - 1) / c + kItemCost;
  long long total = 0, longest = 1;                     // slots past the whole rounds
  for (int u = first; u < units; ++u) {
    total += n[u];
    longest = std::max(longest, (long long)n[u]);
  }
  // Ranges of at least `span` slots keep a unit within kMaxSplitParts / c clusters.
  const int most = lf::kMaxSplitParts / c;
  if (most < 2) return -1;
  const long long span = (longest + most - 2) / (most - 1) + 2 * gran;
  const int ncp = (int)std::max(1LL, std::min<long long>(nc, total / span));
  std::vector<long long> fixed((size_t)nc, 0);
  long long best = -1, worst = 0;
  Plan trial;
  // Level: range lengths f_j = c (level - load_j), at least 0, summing to
  // `total` over the first ncp clusters; cut points at the running sums,
  // rounded to the grid and moved off short parts.
  double lo_l = 0, hi_l = (double)total / c + 1;
  for (int j = 0; j < ncp; ++j) hi_l = std::max(hi_l, (double)load[j] + (double)total / c + 1);
  for (int it = 0; it < 48; ++it) {
    const double mid = 0.5 * (lo_l + hi_l);
    double sum = 0;
    for (int j = 0; j < ncp; ++j) sum += std::max(0.0, (mid - load[j]) * c);
    (sum < total ? lo_l : hi_l) = mid;
  }
  trial.rounds = rounds;
  trial.cut_unit[0] = first;
  trial.cut_slot[0] = 0;
  double at = 0;
  int u = first;
  long long before = 0;  // slots of the units [first, u)
  for (int j = 1; j <= nc; ++j) {
    if (j >= ncp) {
      trial.cut_unit[j] = units;
      trial.cut_slot[j] = 0;
      continue;
    }
    at += std::max(0.0, (hi_l - load[j - 1]) * c);
    const long long t = std::min((long long)at, total);
    while (u < units && before + n[u] <= t) before += n[u++];
    int cu = u, cs = 0;
    if (u < units) {
      const long long off = (t - before) / gran * gran;
      if (off >= least && n[u] - off >= least) cs = (int)off;
      else if (off >= least) cu = u + 1;  // the unit's tail is short: it stays on the left
    }
    if (cu < trial.cut_unit[j - 1] ||
        (cu == trial.cut_unit[j - 1] && cs < trial.cut_slot[j - 1])) {  // never go back
      cu = trial.cut_unit[j - 1];
      cs = trial.cut_slot[j - 1];
    }
    trial.cut_unit[j] = cu;
    trial.cut_slot[j] = cs;
  }
  if (cost_plan(trial, n, c, nc, max_items, load, &worst, &fixed)) {
    *pl = trial;
    best = worst;
  }
  // The walk: the lowest level (bisection) at which the ranges cover every unit.
  double lo_w = 0, hi_w = 0;
  for (int j = 0; j < ncp; ++j) hi_w = std::max(hi_w, (double)load[j]);
  hi_w += (double)total / c + (double)(units - first + 2) * (kItemCost + kPartCost) + 1;
  trial.rounds = rounds;
  if (walk_plan(n, c, ncp, nc, first, load, hi_w, gran, least, &trial)) {
    for (int it = 0; it < 40; ++it) {
      const double mid = 0.5 * (lo_w + hi_w);
      (walk_plan(n, c, ncp, nc, first, load, mid, gran, least, &trial) ? hi_w : lo_w) = mid;
    }
    if (walk_plan(n, c, ncp, nc, first, load, hi_w, gran, least, &trial) &&
        cost_plan(trial, n, c, nc, max_items, load, &worst, &fixed) &&
        (best < 0 || worst < best)) {
      *pl = trial;
      best = worst;
    }
  }
  return best;
}

// Cost of the whole-unit launch: cluster j visits units j, j + nc, ...
long long round_robin_cost(const std::vector<int32_t>& n, int c, int nc) {
  long long worst = 0;
  for (int j = 0; j < nc; ++j) {
    long long cost = 0;
    for (int u = j; u < (int)n.size(); u += nc) cost += (n[u] + c - 1) / c + kItemCost;
    worst = std::max(worst, cost);
  }
  return worst;
}

int fail(int code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  g_last_status = code;
  return code;
}

int cuda_fail(cudaError_t e, const char* what) {
  const int code = (e == cudaErrorMemoryAllocation) ? LF_ERR_OOM : LF_ERR_CUDA;
  (void)cudaGetLastError();  // clear a non-sticky error
  return fail(code, "%s: %s", what, cudaGetErrorString(e));
}

inline size_t round_up(size_t x, size_t m) { return (x + m - 1) / m * m; }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// How many clusters of this shape can be resident at once (0: none).
int active_clusters(const void* fn, int cluster, int grid_y, int grid_z, int smem, int threads) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(cluster, grid_y, grid_z);
  cfg.blockDim = dim3(threads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = cluster;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, fn, &cfg) != cudaSuccess) {
    (void)cudaGetLastError();
    return 0;
  }
  return n;
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// K and V slabs as 2-D tensors [rows = every slot of every unit][head_dim]
// (bf16), read in boxes of 64 columns x {64, 16} rows with the 128-byte
// swizzle the tensor-core descriptors expect.
int encode_tensor_maps(lf_cache* c, size_t n_rows) {
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                                   cudaEnableDefault, &q);
  if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !fn)
    return fail(LF_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  if (n_rows >= (1ull << 31)) return fail(LF_ERR_UNSUPPORTED, "slab has too many rows for TMA");
  EncodeTiledFn encode = reinterpret_cast<EncodeTiledFn>(fn);
  const cuuint64_t dims[2] = {(cuuint64_t)c->head_dim, (cuuint64_t)n_rows};
  const cuuint64_t strides[1] = {(cuuint64_t)c->head_dim * 2};
  const cuuint32_t estr[2] = {1, 1};
  void* bases[4] = {c->K, c->K, c->V, c->V};
  const cuuint32_t heights[4] = {64, 16, 64, 16};
  for (int i = 0; i < 4; ++i) {
    const cuuint32_t box[2] = {64, heights[i]};
    CUresult r = encode(&c->tmaps[i], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, bases[i], dims, strides,
                        box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(LF_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
  }
  return LF_OK;
}

// The plan of the next decode step of `layer`: true, with `pl` filled, when it
// costs less than whole units (cost model above) and every sequence is long
// enough for the exchanges to pay.
bool plan_layer(lf_cache* c, int layer, Plan* pl) {
  if (!c->plan_ok) return false;
  const int32_t* occ = c->occ.data() + (size_t)layer * c->batch;
  int32_t* memo = c->memo_occ.data() + (size_t)layer * c->batch;
  if (std::equal(occ, occ + c->batch, memo)) {
    if (c->memo_used[layer]) *pl = c->memo_plan[layer];
    return c->memo_used[layer] != 0;
  }
  int shortest = INT_MAX;
  for (int b = 0; b < c->batch; ++b) {
    shortest = std::min(shortest, occ[b]);
    for (int g = 0; g < c->kv_heads; ++g) c->plan_n[(size_t)b * c->kv_heads + g] = occ[b];
  }
  bool used = false;
  if (shortest >= kPlanMinSlots) {
    const long long rr = round_robin_cost(c->plan_n, c->cluster, c->grid_y);
    const long long pc = make_plan(c->plan_n, c->cluster, c->grid_y, c->items, pl);
    used = pc >= 0 && pc < rr;
  }
  std::copy(occ, occ + c->batch, memo);
  c->memo_used[layer] = used ? 1 : 0;
  if (used) c->memo_plan[layer] = *pl;
  return used;
}

void destroy_memory(lf_cache* c) {
  if (c->K) cudaFree(c->K);
  if (c->V) cudaFree(c->V);
  if (c->small) cudaFree(c->small);
  c->K = c->V = c->small = nullptr;
}

}  // namespace

void lf::set_last_error(int code, const std::string& msg) {
  g_last_error = msg;
  g_last_status = code;
}

void lf::clear_last_error() { clear_last(); }

extern "C" {

const char* lf_last_error(void) { return g_last_error.c_str(); }

int lf_last_status(void) { return g_last_status; }

int lf_abi_version(void) { return LF_ABI_VERSION; }

lf_cache* lf_cache_create(int layers, int batch, int kv_heads, int q_heads, int head_dim,
                          int budget, int window) {
  return lf_cache_create_ex(layers, batch, kv_heads, q_heads, head_dim, budget, window, nullptr);
}

lf_cache* lf_cache_create_ex(int layers, int batch, int kv_heads, int q_heads, int head_dim,
                             int capacity, int window, const lf_config* cfg) {
  clear_last();
  lf_config def = {LF_BF16, 1, nullptr, 0, 0, LF_KERNEL_AUTO, LF_SCORE_LONGFLOW, 1, 0, 0,
                   LF_SCOPE_KV_HEAD, 0, 0, 0, 0.f, 0.f};
  lf_config c = cfg ? *cfg : def;
  if (layers < 1 || batch < 1 || kv_heads < 1 || q_heads < 1 || capacity < 1 || window < 0) {
    fail(LF_ERR_ARG, "layers, batch, heads and capacity must be >= 1 and window >= 0");
    return nullptr;
  }
  if (batch > 65535 || kv_heads > 65535) {
    fail(LF_ERR_ARG, "batch and kv_heads must be <= 65535");
    return nullptr;
  }
  if (q_heads % kv_heads != 0) {
    fail(LF_ERR_ARG, "q_heads (%d) must be a multiple of kv_heads (%d)", q_heads, kv_heads);
    return nullptr;
  }
  if (c.dtype != LF_BF16 && c.dtype != LF_F32) {
    fail(LF_ERR_ARG, "dtype must be LF_BF16 or LF_F32");
    return nullptr;
  }
  if (c.evict < LF_EVICT_OFF || c.evict > LF_EVICT_RKV) {
    fail(LF_ERR_ARG, "evict must be LF_EVICT_OFF, LF_EVICT_LONGFLOW or LF_EVICT_RKV");
    return nullptr;
  }
  const bool rkv = c.evict == LF_EVICT_RKV;
  if (c.cluster != 0 && (c.cluster < 1 || c.cluster > lf::kMaxCluster ||
                         (c.cluster & (c.cluster - 1)) != 0)) {
    fail(LF_ERR_ARG, "cluster must be 0 (auto) or a power of two <= %d", lf::kMaxCluster);
    return nullptr;
  }
  if (c.stages != 0 && (c.stages < 2 || c.stages > lf::kMaxStages)) {
    fail(LF_ERR_ARG, "stages must be 0 (auto) or in [2, %d]", lf::kMaxStages);
    return nullptr;
  }
  if (c.kernel < LF_KERNEL_AUTO || c.kernel > LF_KERNEL_TENSOR_CORE) {
    fail(LF_ERR_ARG, "kernel must be LF_KERNEL_AUTO, LF_KERNEL_SIMT or LF_KERNEL_TENSOR_CORE");
    return nullptr;
  }
  if (c.norm == 0) c.norm = 1;
  if ((c.score != LF_SCORE_LONGFLOW && c.score != LF_SCORE_H2O) || (c.norm != 1 && c.norm != 2) ||
      c.sinks < 0 || (c.deferred != 0 && c.deferred != 1) ||
      (c.scope != LF_SCOPE_KV_HEAD && c.scope != LF_SCOPE_LAYER)) {
    fail(LF_ERR_ARG, "policy: score must be LF_SCORE_LONGFLOW or LF_SCORE_H2O, norm 1 or 2, "
         "sinks >= 0, deferred 0 or 1, scope LF_SCOPE_KV_HEAD or LF_SCOPE_LAYER");
    return nullptr;
  }
  if (c.evict != LF_EVICT_LONGFLOW) {  // no LongFlow eviction: the policy has nothing to decide
    c.score = LF_SCORE_LONGFLOW;
    c.sinks = c.deferred = 0;
    c.scope = LF_SCOPE_KV_HEAD;
  }
  const int kevict = (c.evict == LF_EVICT_LONGFLOW) ? 1 : 0;
  if (rkv) {  // the README's defaults, then the limits of the compression kernel
    if (c.rkv_buffer == 0) c.rkv_buffer = 128;
    if (c.rkv_alpha == 0) c.rkv_alpha = 8;
    if (c.rkv_beta == 0) c.rkv_beta = 1;
    if (c.rkv_lambda == 0.f) c.rkv_lambda = 0.1f;
    if (c.rkv_tau == 0.f) c.rkv_tau = 0.9f;
    const int grp = q_heads / kv_heads;
    if (c.dtype != LF_BF16 || head_dim != 128 || (grp != 1 && grp != 2 && grp != 4 && grp != 8)) {
      fail(LF_ERR_UNSUPPORTED, "R-KV compression is built for bf16, head_dim 128, group 1/2/4/8");
      return nullptr;
    }
    if (c.budgets) {
      fail(LF_ERR_ARG, "R-KV takes no per-sequence budgets");
      return nullptr;
    }
    if (capacity > lf::kRkvMaxSlots || c.rkv_buffer < 1 || c.rkv_alpha < 1 || c.rkv_beta < 1 ||
        capacity - c.rkv_buffer <= c.rkv_alpha || c.rkv_alpha * grp > 64 ||
        !(c.rkv_lambda > 0.f && c.rkv_lambda <= 1.f) || !(c.rkv_tau > 0.f && c.rkv_tau <= 1.f)) {
      fail(LF_ERR_ARG, "R-KV: need capacity <= %d, buffer >= 1, alpha < capacity - buffer, "
           "alpha * group <= 64, beta >= 1, lambda and tau in (0, 1]", lf::kRkvMaxSlots);
      return nullptr;
    }
  }
  const int group = q_heads / kv_heads;
  lf::KernelEntry kern;
  bool found = false;
  if (c.dtype == LF_BF16 && c.kernel != LF_KERNEL_SIMT)
    found = lf::find_kernels_tc(head_dim, group, &kern);
  if (!found && c.kernel == LF_KERNEL_TENSOR_CORE) {
    fail(LF_ERR_UNSUPPORTED, "the tensor-core kernel needs bf16 storage, head_dim 128 and group "
         "size 1/2/4/8");
    return nullptr;
  }
  if (!found)
    found = (c.dtype == LF_BF16) ? lf::find_kernels_bf16(head_dim, group, &kern)
                                 : lf::find_kernels_f32(head_dim, group, &kern);
  if (!found) {
    fail(LF_ERR_UNSUPPORTED, "no kernel for head_dim %d and group size %d (built: head_dim "
         "16/32/64/128, group 1/2/4/8)", head_dim, group);
    return nullptr;
  }
  // Per-sequence budgets.
  int min_budget = capacity;
  if (c.budgets) {
    for (int b = 0; b < batch; ++b) {
      if (c.budgets[b] < 1 || c.budgets[b] > capacity) {
        fail(LF_ERR_ARG, "budget[%d] = %d outside [1, capacity %d]", b, c.budgets[b], capacity);
        return nullptr;
      }
      min_budget = std::min(min_budget, (int)c.budgets[b]);
    }
  }
  if (kevict && window + c.sinks >= min_budget) {
    fail(LF_ERR_ARG, "window + sinks (%d + %d) must be smaller than every budget (min %d)", window,
         c.sinks, min_budget);
    return nullptr;
  }
  if (kevict && c.deferred && window < 1) {
    fail(LF_ERR_ARG, "deferred eviction needs window >= 1 (the new token is protected)");
    return nullptr;
  }
  if (capacity > INT_MAX / 2) {
    fail(LF_ERR_ARG, "capacity too large");
    return nullptr;
  }

  int device = 0;
  cudaError_t e = cudaGetDevice(&device);
  if (e != cudaSuccess) {
    cuda_fail(e, "cudaGetDevice");
    return nullptr;
  }
  int num_sms = 0, max_optin = 0, max_sm_smem = 0;
  if ((e = cudaDeviceGetAttribute(&max_sm_smem, cudaDevAttrMaxSharedMemoryPerMultiprocessor,
                                  device)) != cudaSuccess ||
      (e = cudaDeviceGetAttribute(&num_sms, cudaDevAttrMultiProcessorCount, device)) != cudaSuccess ||
      (e = cudaDeviceGetAttribute(&max_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, device)) !=
          cudaSuccess) {
    cuda_fail(e, "cudaDeviceGetAttribute");
    return nullptr;
  }
  auto set_attributes = [&](const lf::KernelEntry& k) -> bool {
    if ((e = cudaFuncSetAttribute(k.decode, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  max_optin)) != cudaSuccess ||
        (e = cudaFuncSetAttribute(k.decode, cudaFuncAttributeNonPortableClusterSizeAllowed, 1)) !=
            cudaSuccess ||
        (k.decode_split &&
         ((e = cudaFuncSetAttribute(k.decode_split, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    max_optin)) != cudaSuccess ||
          (e = cudaFuncSetAttribute(k.decode_split,
                                    cudaFuncAttributeNonPortableClusterSizeAllowed, 1)) !=
              cudaSuccess))) {
      cuda_fail(e, "cudaFuncSetAttribute");
      return false;
    }
    return true;
  };
  if (!set_attributes(kern)) return nullptr;

  // Launch shape.  CUDA-core kernel: one cluster of C CTAs per unit; prefer
  // the smallest C giving at least 8 CTAs per SM with >= 128 slots per CTA.
  // Tensor-core kernel: persistent, one CTA per SM; prefer the smallest C
  // whose per-CTA chunk fits next to a ring of `stages` 32 KB tiles.  The
  // caller may force C and the ring depth.
  bool tc = (kern.kind == lf::kTensorCore);
  int threads = tc ? lf::kTcThreads : lf::kThreads;
  const int units = batch * kv_heads;
  int stages = c.stages ? c.stages : (tc ? 3 : 4);
  // The shared memory, resident clusters and item-table size of one cluster size;
  // false if it does not fit.
  int chunk = 0, smem = 0, grid_y = 0, items = 0, resident = 0;
  auto try_shape = [&](int cl) -> bool {
    chunk = (int)round_up((size_t)((capacity + cl - 1) / cl), 4);
    int fits = 0;
    if (tc) {
      // The persistent grid visits ceil(units / resident clusters) units per
      // cluster; its item table is sized for that.  Start from the most
      // clusters the SMs could hold and grow the table if fewer are resident.
      // (+ 2: a planned launch adds the parts of up to two shared units)
      const int most = std::max(1, num_sms / cl);
      items = (units + most - 1) / most + 2;
      for (int pass = 0; pass < 4; ++pass) {
        smem = kern.smem_bytes(stages, chunk, cl, kevict, items);
        // The tensor-core kernel takes all of an SM's tensor memory: ask for more
        // than half of its shared memory so that never two CTAs share an SM.
        smem = std::max(smem, max_sm_smem / 2 + 1024);
        fits = (smem <= max_optin) ? active_clusters(kern.decode, cl, 1, 1, smem, threads) : 0;
        if (fits <= 0) break;
        resident = fits;
        grid_y = std::min(fits, units);
        const int need = (units + grid_y - 1) / grid_y + 2;
        if (need <= items) break;
        items = need;
        fits = 0;
      }
      if (fits > 0 && items > lf::kTcMaxItems) fits = 0;
    } else {
      smem = kern.smem_bytes(stages, chunk, cl, kevict, 0);
      if (smem <= max_optin)
        fits = active_clusters(kern.decode, cl, kv_heads, batch, smem, threads);
    }
    return fits > 0;
  };
  auto first_cluster = [&]() {
    int cl = c.cluster;
    if (cl == 0) {
      cl = 1;
      if (!tc)
        while (cl < lf::kMaxCluster && (long long)units * cl < 8LL * num_sms &&
               (capacity + 2 * cl - 1) / (2 * cl) >= 128)
          cl *= 2;
    }
    return cl;
  };
  int cluster = first_cluster();
  for (;;) {
    if (try_shape(cluster)) break;
    if (c.cluster != 0 || cluster >= lf::kMaxCluster) {
      // The tensor-core kernel chosen by default may not take a very large
      // layer (its per-cluster item table holds kTcMaxItems units, and long
      // units need large clusters): the CUDA-core kernel, one cluster per unit,
      // takes any number of units.
      lf::KernelEntry simt;
      if (tc && c.kernel == LF_KERNEL_AUTO && c.cluster == 0 &&
          lf::find_kernels_bf16(head_dim, group, &simt)) {
        if (!set_attributes(simt)) return nullptr;
        kern = simt;
        tc = false;
        threads = lf::kThreads;
        stages = c.stages ? c.stages : 4;
        cluster = first_cluster();
        continue;
      }
      fail(LF_ERR_UNSUPPORTED, "launch does not fit: cluster %d, %d stages, %d slots per CTA need "
           "%d bytes of shared memory (max %d)", cluster, stages, chunk, smem, max_optin);
      return nullptr;
    }
    cluster *= 2;
  }
  if (tc && c.cluster == 0) {
    // Tensor-core kernel: of the smallest cluster that fits and the next two,
    // take the one with the least estimated time per launch: rounds of units per
    // cluster x (K and V tiles per CTA x ~0.7 us + ~3 us per unit boundary).
    // More CTAs per unit pay when the units do not fill the SMs (64 units of
    // 512 slots: 2-CTA clusters 14.5 us, 1-CTA 16.8 us) and cost when they do.
    auto cost = [&](int cl) {
      const long long rounds = (units + grid_y - 1) / grid_y;
      const long long tiles = 2LL * ((((capacity + cl - 1) / cl) + lf::kTcTile - 1) / lf::kTcTile);
      return rounds * (7 * tiles + 30);
    };
    int best = cluster;
    long long best_cost = cost(cluster);
    for (int cl = cluster * 2; cl <= std::min(cluster * 4, lf::kMaxCluster); cl *= 2) {
      if (!try_shape(cl)) continue;
      const long long cc = cost(cl);
      if (cc < best_cost) {
        best = cl;
        best_cost = cc;
      }
    }
    cluster = best;
    if (!try_shape(cluster)) {  // restore the chosen shape (it fitted above)
      fail(LF_ERR_UNSUPPORTED, "launch shape changed while choosing it");
      return nullptr;
    }
  }

  lf_cache* cache = new (std::nothrow) lf_cache();
  if (!cache) {
    fail(LF_ERR_OOM, "host allocation failed");
    return nullptr;
  }
  cache->layers = layers;
  cache->batch = batch;
  cache->kv_heads = kv_heads;
  cache->q_heads = q_heads;
  cache->head_dim = head_dim;
  cache->capacity = capacity;
  cache->slot_stride = (int)round_up((size_t)capacity, 32);
  cache->window = window;
  cache->dtype = c.dtype;
  cache->evict = c.evict;
  cache->kevict = kevict;
  cache->rkv_buffer = c.rkv_buffer;
  cache->rkv_alpha = c.rkv_alpha;
  cache->rkv_beta = c.rkv_beta;
  cache->rkv_lambda = c.rkv_lambda;
  cache->rkv_tau = c.rkv_tau;
  cache->cluster = cluster;
  cache->stages = stages;
  cache->chunk = chunk;
  cache->smem = smem;
  cache->device = device;
  cache->elem_bytes = (size_t)kern.elem_bytes;
  cache->kern = kern;
  cache->threads = threads;
  cache->grid_y = grid_y;
  cache->items = items;
  cache->occ.assign((size_t)layers * batch, 0);
  cache->occ_limit.resize((size_t)batch);
  for (int b = 0; b < batch; ++b)  // append modes fill the slab to its capacity
    cache->occ_limit[b] = (kevict && c.budgets) ? c.budgets[b] : capacity;
  cache->plan_n.assign((size_t)units, 0);
  cache->memo_occ.assign((size_t)layers * batch, -1);
  cache->memo_used.assign((size_t)layers, 0);
  // Planned launches: the layer's slots cut into equal contiguous ranges, one
  // per cluster, when that balances better than whole units (decided per step
  // on the host), for every policy.
  if (tc) {
    if (kern.decode_split && resident <= lf::kTcMaxPlan &&
        2 * cluster <= lf::kMaxSplitParts) {
      cache->plan_ok = 1;
      cache->memo_plan.resize((size_t)layers);
      // every resident cluster, also when there are fewer units: a plan cuts
      // units into parts for the clusters a whole-unit launch would leave idle
      cache->grid_y = resident;
    }
  }
  cache->score = c.score;
  cache->norm = c.norm;
  cache->sinks = c.sinks;
  cache->deferred = c.deferred;
  cache->scope = c.scope;

  const size_t n_units = (size_t)layers * batch * kv_heads;
  const size_t n_slots = n_units * cache->slot_stride;
  const size_t kv_bytes = n_slots * head_dim * cache->elem_bytes;
  // small block: vnorm, pos [n_slots]; count, next_pos [n_units]; budget [batch];
  // err [1]; plen [layers*batch] -- each piece 256-byte aligned.
  size_t off_vnorm = 0;
  size_t off_pos = round_up(off_vnorm + n_slots * 4, 256);
  size_t off_count = round_up(off_pos + n_slots * 4, 256);
  size_t off_next = round_up(off_count + n_units * 4, 256);
  size_t off_budget = round_up(off_next + n_units * 4, 256);
  size_t off_err = round_up(off_budget + (size_t)batch * 4, 256);
  size_t off_plen = round_up(off_err + 4, 256);
  // policy state: acc [n_slots] (H2O); pending [n_units] (deferred); one layer's
  // lw_score [slots], lw_req and lw_anew [units] (layer scope)
  const size_t lunits = (size_t)batch * kv_heads;
  const bool h2o = c.score == LF_SCORE_H2O, layer = c.scope == LF_SCOPE_LAYER;
  size_t off_acc = round_up(off_plen + (size_t)layers * batch * 4, 256);
  size_t off_pend = round_up(off_acc + (h2o ? n_slots * 4 : 0), 256);
  size_t off_lws = round_up(off_pend + (c.deferred ? n_units * 4 : 0), 256);
  size_t off_lwr = round_up(off_lws + (layer ? lunits * cache->slot_stride * 4 : 0), 256);
  size_t off_lwa = round_up(off_lwr + (layer ? lunits * 4 : 0), 256);
  // planned launches, per exchange slot (one per cluster): [kMaxSplitParts][2
  // kMaxGroup] statistics, [kMaxSplitParts][G d + 4] partial outputs, [2] counters
  // (one row per cut point: cache->grid_y, every resident cluster)
  const size_t nxs = cache->plan_ok ? (size_t)cache->grid_y : 0;
  const size_t nsp = nxs * lf::kMaxSplitParts;
  size_t off_sst = round_up(off_lwa + (layer ? lunits * 4 : 0), 256);
  size_t off_sfn = round_up(off_sst + nsp * 2 * lf::kMaxGroup * 4, 256);
  size_t off_scn = round_up(off_sfn + nsp * ((size_t)group * head_dim + 4) * 4, 256);
  size_t small_bytes = round_up(off_scn + nxs * 2 * 4, 256);

  if ((e = cudaMalloc(&cache->K, kv_bytes)) != cudaSuccess ||
      (e = cudaMalloc(&cache->V, kv_bytes)) != cudaSuccess ||
      (e = cudaMalloc(&cache->small, small_bytes)) != cudaSuccess) {
    cuda_fail(e, "cudaMalloc of the slab");
    destroy_memory(cache);
    delete cache;
    return nullptr;
  }
  char* s = static_cast<char*>(cache->small);
  cache->vnorm = reinterpret_cast<float*>(s + off_vnorm);
  cache->pos = reinterpret_cast<int32_t*>(s + off_pos);
  cache->count = reinterpret_cast<int32_t*>(s + off_count);
  cache->next_pos = reinterpret_cast<int32_t*>(s + off_next);
  cache->budget = reinterpret_cast<int32_t*>(s + off_budget);
  cache->err = reinterpret_cast<int32_t*>(s + off_err);
  cache->plen = reinterpret_cast<int32_t*>(s + off_plen);
  cache->acc = h2o ? reinterpret_cast<float*>(s + off_acc) : nullptr;
  cache->pending = c.deferred ? reinterpret_cast<int32_t*>(s + off_pend) : nullptr;
  cache->lw_score = layer ? reinterpret_cast<float*>(s + off_lws) : nullptr;
  cache->lw_req = layer ? reinterpret_cast<int32_t*>(s + off_lwr) : nullptr;
  cache->lw_anew = layer ? reinterpret_cast<float*>(s + off_lwa) : nullptr;
  cache->split_stat = cache->plan_ok ? reinterpret_cast<float*>(s + off_sst) : nullptr;
  cache->split_fin = cache->plan_ok ? reinterpret_cast<float*>(s + off_sfn) : nullptr;
  cache->split_cnt = cache->plan_ok ? reinterpret_cast<int32_t*>(s + off_scn) : nullptr;

  // Empty state: no occupied slot, positions -1, ||v||_1 0, K/V zero.
  int32_t* hb = new (std::nothrow) int32_t[batch];
  if (!hb) {
    fail(LF_ERR_OOM, "host allocation failed");
    destroy_memory(cache);
    delete cache;
    return nullptr;
  }
  for (int b = 0; b < batch; ++b)
    hb[b] = c.budgets ? c.budgets[b] : (rkv ? capacity - c.rkv_buffer : capacity);
  if ((e = cudaMemset(cache->small, 0, small_bytes)) != cudaSuccess ||
      (e = cudaMemset(cache->pos, 0xff, n_slots * 4)) != cudaSuccess ||
      (cache->pending && (e = cudaMemset(cache->pending, 0xff, n_units * 4)) != cudaSuccess) ||
      (e = cudaMemset(cache->K, 0, kv_bytes)) != cudaSuccess ||
      (e = cudaMemset(cache->V, 0, kv_bytes)) != cudaSuccess ||
      (e = cudaMemcpy(cache->budget, hb, (size_t)batch * 4, cudaMemcpyHostToDevice)) !=
          cudaSuccess ||
      (e = cudaDeviceSynchronize()) != cudaSuccess) {
    delete[] hb;
    cuda_fail(e, "initialising the slab");
    destroy_memory(cache);
    delete cache;
    return nullptr;
  }
  delete[] hb;
  if (rkv) {
    e = cudaFuncSetAttribute(lf::find_rkv_kernel(group), cudaFuncAttributeMaxDynamicSharedMemorySize,
                             lf::rkv_smem_bytes());
    if (e != cudaSuccess) {
      cuda_fail(e, "cudaFuncSetAttribute (R-KV compression)");
      destroy_memory(cache);
      delete cache;
      return nullptr;
    }
  }
  if (tc || rkv) {
    const int code = encode_tensor_maps(cache, n_slots);
    if (code != LF_OK) {
      destroy_memory(cache);
      delete cache;
      return nullptr;
    }
  }
  return cache;
}

int lf_cache_destroy(lf_cache* cache) {
  clear_last();
  if (!cache) return LF_OK;
  destroy_memory(cache);
  delete cache;
  return LF_OK;
}

int lf_prefill_fill(lf_cache* cache, int layer, const void* k, const void* v,
                    const int32_t* prompt_len, int max_prompt, lf_stream_t stream) {
  clear_last();
  if (!cache) return fail(LF_ERR_ARG, "null cache");
  if (layer < 0 || layer >= cache->layers)
    return fail(LF_ERR_ARG, "layer %d outside [0, %d)", layer, cache->layers);
  if (!prompt_len) return fail(LF_ERR_ARG, "null prompt_len");
  if (max_prompt < 0) return fail(LF_ERR_ARG, "max_prompt < 0");
  int longest = 0;
  for (int b = 0; b < cache->batch; ++b) {
    const int P = prompt_len[b];
    if (P < 0 || P > max_prompt)
      return fail(LF_ERR_ARG, "prompt_len[%d] = %d outside [0, max_prompt %d]", b, P, max_prompt);
    longest = std::max(longest, P);
  }
  // Limits need the budgets, which live on the device; the host mirror below
  // is read back only here, outside any step.
  int32_t* hb = new (std::nothrow) int32_t[cache->batch];
  if (!hb) return fail(LF_ERR_OOM, "host allocation failed");
  cudaError_t e = cudaMemcpy(hb, cache->budget, (size_t)cache->batch * 4, cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) {
    delete[] hb;
    return cuda_fail(e, "reading budgets");
  }
  for (int b = 0; b < cache->batch; ++b) {
    // deferred: the step that fills the buffer chooses the first victim
    const int limit = cache->kevict ? hb[b] - (cache->deferred ? 1 : 0) : cache->capacity;
    if (prompt_len[b] > limit) {
      delete[] hb;
      return fail(LF_ERR_ARG, "prompt_len[%d] = %d exceeds the buffer (%d%s); feed the rest "
                  "through lf_decode_step", b, prompt_len[b], limit,
                  cache->deferred ? ": budget - 1 in deferred mode" : "");
    }
  }
  delete[] hb;
  if (longest > 0 && (!k || !v)) return fail(LF_ERR_ARG, "null k or v");
  if (longest > 0 && (!aligned16(k) || !aligned16(v)))
    return fail(LF_ERR_ARG, "k and v must be 16-byte aligned");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int32_t* dplen = cache->plen + (size_t)layer * cache->batch;
  if ((e = cudaMemcpyAsync(dplen, prompt_len, (size_t)cache->batch * 4, cudaMemcpyHostToDevice,
                           st)) != cudaSuccess)
    return cuda_fail(e, "uploading prompt lengths");
  const size_t layer_units = (size_t)cache->batch * cache->kv_heads;
  const size_t layer_slots = layer_units * cache->slot_stride;
  lf::PrefillArgs a;
  a.k = k;
  a.v = v;
  a.plen = dplen;
  a.K = static_cast<char*>(cache->K) + layer * layer_slots * cache->head_dim * cache->elem_bytes;
  a.V = static_cast<char*>(cache->V) + layer * layer_slots * cache->head_dim * cache->elem_bytes;
  a.vnorm = cache->vnorm + layer * layer_slots;
  a.pos = cache->pos + layer * layer_slots;
  a.count = cache->count + layer * layer_units;
  a.next_pos = cache->next_pos + layer * layer_units;
  a.acc = cache->acc ? cache->acc + layer * layer_slots : nullptr;
  a.pending = cache->pending ? cache->pending + layer * layer_units : nullptr;
  a.kv_heads = cache->kv_heads;
  a.max_prompt = max_prompt;
  a.slot_stride = cache->slot_stride;
  a.norm = cache->norm;
  void* args[] = {&a};
  e = cudaLaunchKernel(cache->kern.prefill, dim3(cache->kv_heads, cache->batch, 1),
                       dim3(lf::kThreads, 1, 1), args, 0, st);
  if (e != cudaSuccess) return cuda_fail(e, "prefill launch");
  for (int b = 0; b < cache->batch; ++b)
    cache->occ[(size_t)layer * cache->batch + b] = std::min(prompt_len[b], cache->occ_limit[b]);
  return LF_OK;
}

int lf_decode_step(lf_cache* cache, int layer, const void* q, const void* k_new,
                   const void* v_new, void* out, int32_t* evicted_slot, lf_stream_t stream) {
  if (!cache) return fail(LF_ERR_ARG, "null cache");
  if (layer < 0 || layer >= cache->layers)
    return fail(LF_ERR_ARG, "layer %d outside [0, %d)", layer, cache->layers);
  if (!q || !k_new || !v_new || !out || !evicted_slot)
    return fail(LF_ERR_ARG, "null q, k_new, v_new, out or evicted_slot");
  if (!aligned16(q) || !aligned16(k_new) || !aligned16(v_new))
    return fail(LF_ERR_ARG, "q, k_new and v_new must be 16-byte aligned");
  const size_t layer_units = (size_t)cache->batch * cache->kv_heads;
  const size_t layer_slots = layer_units * cache->slot_stride;
  lf::DecodeArgs a;
  a.q = q;
  a.k_new = k_new;
  a.v_new = v_new;
  a.out = out;
  a.evicted = evicted_slot;
  a.K = static_cast<char*>(cache->K) + layer * layer_slots * cache->head_dim * cache->elem_bytes;
  a.V = static_cast<char*>(cache->V) + layer * layer_slots * cache->head_dim * cache->elem_bytes;
  a.vnorm = cache->vnorm + layer * layer_slots;
  a.pos = cache->pos + layer * layer_slots;
  a.count = cache->count + layer * layer_units;
  a.next_pos = cache->next_pos + layer * layer_units;
  a.budget = cache->budget;
  a.err = cache->err;
  a.acc = cache->acc ? cache->acc + layer * layer_slots : nullptr;
  a.pending = cache->pending ? cache->pending + layer * layer_units : nullptr;
  a.lw_score = cache->lw_score;  // one layer's scratch, reused by every layer
  a.lw_req = cache->lw_req;
  a.lw_anew = cache->lw_anew;
  a.score = cache->score;
  a.norm = cache->norm;
  a.sinks = cache->sinks;
  a.deferred = cache->deferred;
  a.scope = cache->scope;
  a.batch = cache->batch;
  a.kv_heads = cache->kv_heads;
  a.q_heads = cache->q_heads;
  a.slot_stride = cache->slot_stride;
  a.capacity = cache->capacity;
  a.window = cache->window;
  a.chunk = cache->chunk;
  a.stages = cache->stages;
  a.evict = cache->kevict;
  a.strict = (cache->evict == LF_EVICT_RKV) ? 1 : 0;
  a.scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)cache->head_dim));

  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = (cache->kern.kind == lf::kTensorCore)
                    ? dim3(cache->cluster, cache->grid_y, 1)
                    : dim3(cache->cluster, cache->kv_heads, cache->batch);
  cfg.blockDim = dim3(cache->threads, 1, 1);
  cfg.dynamicSmemBytes = cache->smem;
  cfg.stream = static_cast<cudaStream_t>(stream);
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = cache->cluster;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  // Tensor-core kernel: programmatic dependent launch (its prologue overlaps the
  // previous grid; it waits for that grid before touching global memory).
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = (cache->kern.kind == lf::kTensorCore) ? 2 : 1;
  cudaError_t e;
  if (cache->kern.kind == lf::kTensorCore) {
    lf::TcArgs ta;
    ta.k64 = cache->tmaps[0];
    ta.k16 = cache->tmaps[1];
    ta.v64 = cache->tmaps[2];
    ta.v16 = cache->tmaps[3];
    ta.a = a;
    ta.row_base = (int)(layer * layer_slots);
    ta.max_items = cache->items;
    ta.plan_nc = 0;
    ta.split_stat = cache->split_stat;
    ta.split_fin = cache->split_fin;
    ta.split_cnt = cache->split_cnt;
    Plan pl;
    const bool planned = plan_layer(cache, layer, &pl);
    if (planned) {
      ta.plan_nc = cache->grid_y;
      ta.plan_rounds = pl.rounds;
      for (int j = 0; j <= cache->grid_y; ++j) {
        ta.cut_unit[j] = pl.cut_unit[j];
        ta.cut_slot[j] = pl.cut_slot[j];
      }
    }
    // Each cluster's first unit (the kernel's item order: the part its range
    // starts inside, else the part it ends inside, else a whole unit of the
    // range, else its first round) and the host's count of its slots, for the
    // kernel's L2 prefetch before its grid dependency wait.  Only for launches
    // of at least kPrefetchMinRows slot rows per CTA: a short launch's CTAs
    // start as the previous grid ends, and the prefetch then delays them
    // (measured on qwen3-0.6b, 215 rows per CTA: 11.2 -> 12.1 us per launch).
    const int units = cache->batch * cache->kv_heads;
    const int32_t* occ = cache->occ.data() + (size_t)layer * cache->batch;
    long long slots = 0;
    for (int b = 0; b < cache->batch; ++b) slots += (long long)occ[b] * cache->kv_heads;
    const bool hint = slots >= (long long)kPrefetchMinRows * cache->grid_y * cache->cluster;
    for (int j = 0; j < lf::kTcMaxPlan; ++j) {
      int u = -1;
      if (hint && j < cache->grid_y) {
        if (!planned) {
          u = j < units ? j : -1;
        } else {
          const int u0 = pl.cut_unit[j], s0 = pl.cut_slot[j];
          const int u1 = pl.cut_unit[j + 1], s1 = pl.cut_slot[j + 1];
          u = s0 > 0 ? u0 : s1 > 0 ? u1 : u1 > u0 ? u0 : (pl.rounds > 0 ? j : -1);
        }
      }
      ta.hint_unit[j] = u;
      ta.hint_n[j] = (u >= 0 && u < units) ? occ[u / cache->kv_heads] : 0;
    }
    void* args[] = {&ta};
    e = cudaLaunchKernelExC(&cfg, planned ? cache->kern.decode_split : cache->kern.decode, args);
  } else {
    void* args[] = {&a};
    e = cudaLaunchKernelExC(&cfg, cache->kern.decode, args);
  }
  if (e != cudaSuccess) return cuda_fail(e, "decode launch");
  for (int b = 0; b < cache->batch; ++b) {
    int32_t& o = cache->occ[(size_t)layer * cache->batch + b];
    o = std::min(o + 1, cache->occ_limit[b]);
  }
  if (cache->scope == LF_SCOPE_LAYER) {
    // The shared victim of every sequence, once all its KV heads have scored.
    // Programmatic dependent launch: its CTAs are placed while the decode grid
    // drains and wait for it in griddepcontrol.wait.
    void* args[] = {&a};
    cudaLaunchConfig_t sc = {};
    sc.gridDim = dim3(cache->batch, 1, 1);
    sc.blockDim = dim3(lf::kSelThreads, 1, 1);
    sc.dynamicSmemBytes = 0;
    sc.stream = static_cast<cudaStream_t>(stream);
    cudaLaunchAttribute sa[1];
    sa[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    sa[0].val.programmaticStreamSerializationAllowed = 1;
    sc.attrs = sa;
    sc.numAttrs = 1;
    e = cudaLaunchKernelExC(&sc, cache->kern.select, args);
    if (e != cudaSuccess) return cuda_fail(e, "layer-scope selection launch");
  }
  return LF_OK;
}

int lf_rkv_compress(lf_cache* cache, int layer, const void* q_obs, lf_stream_t stream) {
  if (!cache) return fail(LF_ERR_ARG, "null cache");
  if (cache->evict != LF_EVICT_RKV) return fail(LF_ERR_ARG, "not an R-KV cache (evict != LF_EVICT_RKV)");
  if (layer < 0 || layer >= cache->layers)
    return fail(LF_ERR_ARG, "layer %d outside [0, %d)", layer, cache->layers);
  if (!q_obs || !aligned16(q_obs)) return fail(LF_ERR_ARG, "q_obs must be non-null and 16-byte aligned");
  const int group = cache->q_heads / cache->kv_heads;
  const size_t layer_units = (size_t)cache->batch * cache->kv_heads;
  const size_t layer_slots = layer_units * cache->slot_stride;
  lf::RkvArgs ra;
  ra.kmap = cache->tmaps[0];
  ra.q_obs = static_cast<const __nv_bfloat16*>(q_obs);
  ra.K = static_cast<__nv_bfloat16*>(cache->K) + layer * layer_slots * cache->head_dim;
  ra.V = static_cast<__nv_bfloat16*>(cache->V) + layer * layer_slots * cache->head_dim;
  ra.vnorm = cache->vnorm + layer * layer_slots;
  ra.pos = cache->pos + layer * layer_slots;
  ra.count = cache->count + layer * layer_units;
  ra.next_pos = cache->next_pos + layer * layer_units;
  ra.err = cache->err;
  ra.kv_heads = cache->kv_heads;
  ra.q_heads = cache->q_heads;
  ra.slot_stride = cache->slot_stride;
  ra.budget = cache->capacity - cache->rkv_buffer;
  ra.alpha = cache->rkv_alpha;
  ra.beta = cache->rkv_beta;
  ra.row_base = (int)(layer * layer_slots);
  ra.lam = cache->rkv_lambda;
  ra.tau = cache->rkv_tau;
  ra.scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)cache->head_dim));
  void* args[] = {&ra};
  cudaError_t e = cudaLaunchKernel(lf::find_rkv_kernel(group), dim3((unsigned)layer_units, 1, 1),
                                   dim3((unsigned)lf::rkv_threads(), 1, 1), args, lf::rkv_smem_bytes(),
                                   static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "R-KV compression launch");
  // every sequence is back at the budget (or at most that: it was below it)
  for (int b = 0; b < cache->batch; ++b) {
    int32_t& o = cache->occ[(size_t)layer * cache->batch + b];
    o = std::min(o, ra.budget);
  }
  return LF_OK;
}

int lf_cache_check(lf_cache* cache, lf_stream_t stream, int32_t* bits) {
  clear_last();
  if (bits) *bits = 0;
  if (!cache) return fail(LF_ERR_ARG, "null cache");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int32_t word = 0;
  cudaError_t e;
  if ((e = cudaStreamSynchronize(st)) != cudaSuccess) return cuda_fail(e, "stream synchronize");
  if ((e = cudaMemcpy(&word, cache->err, 4, cudaMemcpyDeviceToHost)) != cudaSuccess)
    return cuda_fail(e, "reading the error word");
  if ((e = cudaMemset(cache->err, 0, 4)) != cudaSuccess ||
      // an expired wait can leave a split launch's exchange counters mid-count
      ((word & LF_DEVERR_TIMEOUT) && cache->split_cnt &&
       (e = cudaMemset(cache->split_cnt, 0, (size_t)cache->grid_y * 2 * 4)) != cudaSuccess) ||
      (e = cudaDeviceSynchronize()) != cudaSuccess)
    return cuda_fail(e, "clearing the error word");
  if (bits) *bits = word;
  if (word != 0) return fail(LF_ERR_DEVICE, "device error word 0x%x", (unsigned)word);
  return LF_OK;
}

int lf_launch_plan(lf_cache* cache, int layer, int32_t* rounds, int32_t* cut_unit,
                   int32_t* cut_slot, int max_cuts) {
  clear_last();
  if (!cache) return fail(LF_ERR_ARG, "null cache");
  if (layer < 0 || layer >= cache->layers)
    return fail(LF_ERR_ARG, "layer %d outside [0, %d)", layer, cache->layers);
  Plan pl;
  if (!plan_layer(cache, layer, &pl)) return 0;
  const int nc = cache->grid_y;
  if (cut_unit || cut_slot) {
    if (!cut_unit || !cut_slot || max_cuts < nc + 1)
      return fail(LF_ERR_ARG, "need cut_unit and cut_slot of >= %d entries", nc + 1);
    for (int j = 0; j <= nc; ++j) {
      cut_unit[j] = pl.cut_unit[j];
      cut_slot[j] = pl.cut_slot[j];
    }
  }
  if (rounds) *rounds = pl.rounds;
  return nc;
}

int lf_launch_plan_for(const int32_t* occupancy, int units, int cluster, int clusters,
                       int max_items, int32_t* rounds, int32_t* cut_unit, int32_t* cut_slot) {
  clear_last();
  if (!occupancy || units < 1 || cluster < 1 || clusters < 1 || clusters > lf::kTcMaxPlan ||
      max_items < 1 || !rounds || !cut_unit || !cut_slot)
    return fail(LF_ERR_ARG, "bad plan arguments (clusters <= %d)", lf::kTcMaxPlan);
  std::vector<int32_t> n(occupancy, occupancy + units);
  for (int u = 0; u < units; ++u)
    if (n[u] < 0) return fail(LF_ERR_ARG, "occupancy[%d] < 0", u);
  Plan pl;
  const long long pc = make_plan(n, cluster, clusters, max_items, &pl);
  if (pc < 0 || pc >= round_robin_cost(n, cluster, clusters)) return 0;
  *rounds = pl.rounds;
  for (int j = 0; j <= clusters; ++j) {
    cut_unit[j] = pl.cut_unit[j];
    cut_slot[j] = pl.cut_slot[j];
  }
  return clusters;
}

int lf_cache_layout(const lf_cache* cache, lf_layout* out) {
  clear_last();
  if (!cache || !out) return fail(LF_ERR_ARG, "null cache or layout");
  out->layers = cache->layers;
  out->batch = cache->batch;
  out->kv_heads = cache->kv_heads;
  out->q_heads = cache->q_heads;
  out->head_dim = cache->head_dim;
  out->capacity = cache->capacity;
  out->slot_stride = cache->slot_stride;
  out->window = cache->window;
  out->dtype = cache->dtype;
  out->evict = cache->evict;
  out->cluster = cache->cluster;
  out->stages = cache->stages;
  out->kernel = cache->kern.kind == lf::kTensorCore ? LF_KERNEL_TENSOR_CORE : LF_KERNEL_SIMT;
  out->k = cache->K;
  out->v = cache->V;
  out->vnorm = cache->vnorm;
  out->pos = cache->pos;
  out->count = cache->count;
  out->next_pos = cache->next_pos;
  out->budget = cache->budget;
  out->err = cache->err;
  out->score = cache->score;
  out->norm = cache->norm;
  out->sinks = cache->sinks;
  out->deferred = cache->deferred;
  out->scope = cache->scope;
  out->acc = cache->acc;
  out->pending = cache->pending;
  out->rkv_buffer = cache->rkv_buffer;
  out->rkv_alpha = cache->rkv_alpha;
  out->rkv_beta = cache->rkv_beta;
  out->rkv_lambda = cache->rkv_lambda;
  out->rkv_tau = cache->rkv_tau;
  out->split_units = cache->plan_ok ? cache->grid_y : 0;
  out->split_cnt = cache->split_cnt;
  return LF_OK;
}

}  // extern "C"
