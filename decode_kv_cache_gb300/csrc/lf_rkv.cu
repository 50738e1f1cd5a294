// R-KV's buffered compression step on the tensor cores (bf16 storage, head
// dim 128): the baseline the LongFlow pages compare against.  Its README
// ("GitHub - Zefan-Cai/R-KV", section "Method", stages 2-4) scores every
// cached token of a KV head by
//   importance  I_i = mean over the observation queries of their softmax
//               weight on i (over every cached token);
//   redundancy  R_i = 1 when at least beta later tokens have a key cosine
//               >= tau with token i, else 0;
//   joint       Z_i = lambda I_i - (1 - lambda) R_i,
// keeps the alpha latest tokens and the best-scoring others up to the budget,
// and (static slab) moves the kept buffer tokens into the freed slots.
//
// One CTA per (sequence, KV head) unit, n <= 4096 cached tokens:
//   pass 1  per 128-token tile, S = K_tile . Q_obs^T on the tensor cores
//           (M = 128, N = alpha * G padded to 16); online max / sum of every
//           observation query's softmax over all tokens;
//   pass 2  per 128-token row block I: importance of its tokens, then the key
//           dot products K_I . K_J^T (M = N = 128) for every J >= I, streamed
//           through a 3-stage TMA ring into three TMEM accumulators (the MMAs
//           run two blocks ahead; each warp hands an accumulator back as soon
//           as it has loaded it); each pair (i, j) is looked at once and a
//           near-duplicate pair counts for the older token.  The B x B cosine
//           matrix never leaves the chip;
//   select  a bitonic sort of (Z, position) keys, observation tokens first;
//   move    kept buffer tokens into the freed retained slots.
// Every wait is bounded; on expiry the unit is left as it was and
// LF_DEVERR_TIMEOUT is raised.
#include <cuda.h>
#include <cuda_runtime.h>

#include <climits>

#include "lf_device.cuh"
#include "lf_rkv.h"
#include "longflow.h"

namespace lf {

namespace {

constexpr int kRkThreads = 256;
constexpr int kRkTile = 128;
constexpr int kRkStages = 3;
constexpr int kRkStage = kRkTile * 256;     // one K tile [128 rows][128 d] bf16: 32 KB
constexpr int kRkBlock = kRkTile * 128;     // one 64-column half of it: 16 KB
constexpr int kRkQRows = 64;                // observation query rows (alpha * G <= 64)
constexpr int kRkQBlock = kRkQRows * 128;   // one 64-column half of the query operand: 8 KB

// Shared-memory plan (offsets from a 1024-byte aligned base).
constexpr int kOffBars = 0;        // full[3], afull, impfull, accfull[3], accfree[3]
constexpr int kRkAcc = 3;          // key dot-product accumulators, 128 TMEM columns each
constexpr int kOffTmem = 128;
constexpr int kOffMisc = 144;      // [0] fail flag, [1] move count, [2] list length check
constexpr int kOffStats = 256;     // m[64], l[64]
constexpr int kOffRed = 1024;      // [4 quarters][64 columns][2]
constexpr int kOffNmin = 3072;     // per 32-slot chunk: smallest ||k|| (128 chunks)
constexpr int kOffA = 4096;
constexpr int kOffRing = kOffA + kRkStage;
constexpr int kOffQ = kOffRing + kRkStages * kRkStage;
constexpr int kOffPos = kOffQ + 2 * kRkQBlock;
constexpr int kOffInv = kOffPos + kRkvMaxSlots * 4;
constexpr int kOffCnt = kOffInv + kRkvMaxSlots * 4;
constexpr int kOffZ = kOffCnt + kRkvMaxSlots * 4;
constexpr int kSmem = kOffZ + kRkvMaxSlots * 4 + 1024;  // + alignment slack
static_assert(kOffA % 1024 == 0 && kOffRing % 1024 == 0 && kOffQ % 1024 == 0, "alignment");
// the sort reuses the ring: 64-bit keys then 16-bit slot indices
static_assert(kRkvMaxSlots * 10 <= kRkStages * kRkStage, "sort space");

__device__ __forceinline__ uint32_t orderable(float z) {
  const uint32_t u = __float_as_uint(z);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

template <int G>
__global__ void __launch_bounds__(kRkThreads, 1) rkv_compress_kernel(const __grid_constant__ RkvArgs ra) {
  using T = __nv_bfloat16;
  constexpr int D = 128;
  const int unit = blockIdx.x;
  const int b = unit / ra.kv_heads;
  const int g = unit - b * ra.kv_heads;
  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int warp = tid >> 5;
  const int quarter = warp & 3;     // TMEM lanes 32*quarter .. +31
  const int half = warp >> 2;       // which half of the accumulator's columns
  const int QN = ra.alpha * G;      // observation query rows
  const int QN16 = (QN + 15) & ~15;
  const size_t ubase = (size_t)unit * ra.slot_stride;

  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kOffBars);
  uint64_t* afull = full + 3;
  uint64_t* impfull = full + 4;
  uint64_t* accfull = full + 5;   // [3] MMAs of a block complete
  uint64_t* accfree = full + 8;   // [3] every warp has loaded the block
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffTmem);
  volatile int* misc = reinterpret_cast<volatile int*>(smem + kOffMisc);
  float* m_col = reinterpret_cast<float*>(smem + kOffStats);
  float* l_col = m_col + kRkQRows;
  float* red = reinterpret_cast<float*>(smem + kOffRed);
  float* nmin = reinterpret_cast<float*>(smem + kOffNmin);
  unsigned char* abuf = smem + kOffA;
  unsigned char* ring = smem + kOffRing;
  unsigned char* qop = smem + kOffQ;
  int32_t* pos_s = reinterpret_cast<int32_t*>(smem + kOffPos);
  float* inv_s = reinterpret_cast<float*>(smem + kOffInv);
  int* cnt_s = reinterpret_cast<int*>(smem + kOffCnt);
  float* z_s = reinterpret_cast<float*>(smem + kOffZ);

  const int n = ra.count[unit];
  if (n <= ra.budget) return;   // nothing above the budget: uniform for the CTA
  if (n > kRkvMaxSlots || n > ra.slot_stride) {
    if (tid == 0) atomicOr(ra.err, LF_DEVERR_STATE);
    return;
  }
  const int nb = (n + kRkTile - 1) / kRkTile;
  const int pnext = ra.next_pos[unit];

  // ---- set-up: barriers, tensor memory, positions, 1/||k||, the query operand --
  if (tid == 0) {
    for (int i = 0; i < 8; ++i) mbar_init(&full[i], 1);
    for (int i = 0; i < kRkAcc; ++i) mbar_init(&accfree[i], kRkThreads / 32);
    fence_mbar_init();
    misc[0] = 0;
  }
  if (warp == 0) {
    __syncwarp();  // warp-collective allocation (thread 0 initialised the barriers alone)
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  for (int i = tid; i < kRkvMaxSlots; i += kRkThreads) {
    pos_s[i] = (i < n) ? ra.pos[ubase + i] : INT_MIN;
    cnt_s[i] = 0;
    z_s[i] = 0.f;
    inv_s[i] = 0.f;   // ||k_i||^2 accumulates here in pass 1, then becomes 1/||k_i||
  }
  // the observation queries as the B operand: row j*G + h = query head g*G + h
  // of observation j; rows >= QN stay zero
  for (int i = tid; i < 2 * kRkQBlock / 16; i += kRkThreads)
    reinterpret_cast<uint4*>(qop)[i] = make_uint4(0, 0, 0, 0);
  __syncthreads();
  for (int c = tid; c < QN * 16; c += kRkThreads) {
    const int r = c >> 4;          // query row
    const int ch = c & 15;         // 16-byte chunk of the 256-byte row
    const int j = r / G, h = r - (r / G) * G;
    const T* src = ra.q_obs + (((size_t)b * ra.alpha + j) * ra.q_heads + (size_t)g * G + h) * D;
    const uint4 v = *reinterpret_cast<const uint4*>(src + ch * 8);
    *reinterpret_cast<uint4*>(qop + (ch >> 3) * kRkQBlock + r * 128 + (((ch & 7) ^ (r & 7)) << 4)) = v;
  }
  __syncthreads();
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tm = *tmem_slot;
  const uint32_t t_imp = tm + kRkAcc * 128;   // importance logits, QN16 <= 64 columns
  // K tiles are read again for every row block: ask L2 to keep them
  const uint64_t pol = l2_evict_last_policy();
  const int row0 = ra.row_base + (int)ubase;
  const uint32_t id_imp = idesc_bf16_f32(128, QN16, false, false);
  const uint32_t id_s = idesc_bf16_f32(128, 128, false, false);
  const uint32_t lanes = (uint32_t)(quarter * 32) << 16;
  bool ok = true;
  int n_a = 0, n_imp = 0;   // uses of the A-tile and importance barriers
  int issued = 0;           // ring tiles requested (thread 0)

  // Load K tile t (rows 128 t ..) into dst, counted on bar (thread 0).
  auto load_tile = [&](unsigned char* dst, int t, uint64_t* bar) {
    mbar_arrive_expect_tx(bar, (uint32_t)kRkStage);
    for (int blk = 0; blk < 2; ++blk)
      for (int ro = 0; ro < kRkTile; ro += 64)
        tma_load_2d(dst + blk * kRkBlock + ro * 128, &ra.kmap, blk * 64, row0 + t * kRkTile + ro,
                    bar, pol);
  };
  // Importance logits of the A tile into t_imp (thread 0).
  auto mma_imp = [&]() {
    const uint32_t a0 = smem_u32(abuf), q0 = smem_u32(qop);
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk)
      tc_mma_bf16(t_imp, sw128_desc(a0 + (kk >> 2) * kRkBlock + (kk & 3) * 32, 16, 1024),
                  sw128_desc(q0 + (kk >> 2) * kRkQBlock + (kk & 3) * 32, 16, 1024), id_imp,
                  kk > 0 ? 1u : 0u);
    tc_commit(impfull);
  };
  // Row block I of A: load it and compute its importance logits (all threads);
  // returns this thread's 32 logits (columns 32*half ..) scaled to log2 units.
  auto a_tile_logits = [&](int I, float* s) -> bool {
    if (tid == 0) load_tile(abuf, I, afull);
    bool got = mbar_wait_bounded(afull, (uint32_t)(n_a & 1));
    ++n_a;
    if (tid == 0 && got) {
      tc_fence_after();
      mma_imp();
    }
    got = got && mbar_wait_bounded(impfull, (uint32_t)(n_imp & 1));
    ++n_imp;
    got = __syncthreads_and(got);
    if (!got) return false;
    tc_fence_after();
    __syncwarp();  // tcgen05.ld is warp-collective
    tmem_ld32(t_imp + lanes + (uint32_t)(half * 32), s);
    tmem_wait_ld();
    const int row = I * kRkTile + quarter * 32 + lane;
#pragma unroll
    for (int c = 0; c < 32; ++c)
      s[c] = (row < n && half * 32 + c < QN) ? s[c] * ra.scale_log2 : -INFINITY;
    return true;
  };

  // ---- pass 1: every observation query's max and softmax denominator ------------
  if (tid < kRkQRows) {
    m_col[tid] = -INFINITY;
    l_col[tid] = 0.f;
  }
  for (int I = 0; I < nb && ok; ++I) {
    float s[32];
    ok = a_tile_logits(I, s);
    if (!ok) break;
    {
      // ||k||^2 of this thread's token, d-half `half`, from the tile in shared memory
      // (row r of the 64-column block at r * 128 bytes, 16-byte chunks swizzled by r mod 8)
      const int r = quarter * 32 + lane;
      const int row = I * kRkTile + r;
      const unsigned char* rp = abuf + half * kRkBlock + r * 128;
      float ss = 0.f;
#pragma unroll
      for (int ch = 0; ch < 8; ++ch) {
        const uint4 w = *reinterpret_cast<const uint4*>(rp + ((ch ^ (r & 7)) << 4));
        const __nv_bfloat162* h2 = reinterpret_cast<const __nv_bfloat162*>(&w);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 f = __bfloat1622float2(h2[e]);
          ss = fmaf(f.x, f.x, fmaf(f.y, f.y, ss));
        }
      }
      if (row < n) atomicAdd(&inv_s[row], ss);
    }
#pragma unroll
    for (int c = 0; c < 32; ++c) {
      const float wm = warp_max(s[c]);
      const float e = (s[c] == -INFINITY) ? 0.f : exp2f(s[c] - wm);
      const float ws = warp_sum(e);
      if (lane == 0) {
        red[(quarter * kRkQRows + half * 32 + c) * 2] = wm;
        red[(quarter * kRkQRows + half * 32 + c) * 2 + 1] = ws;
      }
    }
    tc_fence_before();
    __syncthreads();
    if (tid < QN) {
      float m = m_col[tid], l = l_col[tid];
      for (int q = 0; q < 4; ++q) {
        const float bm = red[(q * kRkQRows + tid) * 2], bl = red[(q * kRkQRows + tid) * 2 + 1];
        if (bm == -INFINITY) continue;
        const float mn = fmaxf(m, bm);
        l = (m == -INFINITY ? 0.f : l * exp2f(m - mn)) + bl * exp2f(bm - mn);
        m = mn;
      }
      m_col[tid] = m;
      l_col[tid] = l;
    }
    __syncthreads();
  }

  // 1/||k_i|| (0 for a zero key: never similar), and the smallest ||k|| of every
  // 32-slot chunk for the quick rejection below
  __syncthreads();
  for (int i = tid; i < n; i += kRkThreads) {
    const float ss = inv_s[i];
    inv_s[i] = (ss > 0.f) ? rsqrtf(ss) : 0.f;
  }
  __syncthreads();
  if (tid < kRkvMaxSlots / 32) {
    float mn = INFINITY;
    for (int c = 0; c < 32; ++c) {
      const float iv = inv_s[tid * 32 + c];
      if (iv > 0.f) mn = fminf(mn, 1.f / iv);
    }
    nmin[tid] = mn;
  }
  __syncthreads();

  // ---- pass 2: importance, then near-duplicate counts over blocks J >= I ---------
  int tglob = 0;   // K tiles through the ring so far
  for (int I = 0; I < nb && ok; ++I) {
    const int row = I * kRkTile + quarter * 32 + lane;   // this thread's token
    {
      float s[32];
      ok = a_tile_logits(I, s);
      if (!ok) break;
      float part = 0.f;
#pragma unroll
      for (int c = 0; c < 32; ++c) {
        const int col = half * 32 + c;
        if (col < QN && s[c] != -INFINITY) part += exp2f(s[c] - m_col[col]) / l_col[col];
      }
      if (row < n) atomicAdd(&z_s[row], part / (float)QN);
    }
    const float inv_i = (row < n) ? inv_s[row] : 0.f;
    const float thr_i = (inv_i > 0.f) ? ra.tau / inv_i : INFINITY;   // tau * ||k_i||
    const int pos_i = pos_s[min(row, kRkvMaxSlots - 1)];
    int cnt = 0;
    // prologue: the first tiles of this row block's column walk, and its first MMA
    const int njb = nb - I;
    if (tid == 0) {
      for (int q = 0; q < kRkStages && q < njb; ++q)
        load_tile(ring + ((tglob + q) % kRkStages) * kRkStage, I + q, &full[(tglob + q) % kRkStages]);
      issued = tglob + min(kRkStages, njb);
    }
    auto mma_s = [&](int t) -> bool {   // K_I . K_J^T of ring tile t into accumulator t % 3
      const int st = t % kRkStages;
      const int acc = t % kRkAcc;
      if (!mbar_wait_bounded(&full[st], (uint32_t)((t / kRkStages) & 1))) return false;
      // the accumulator's previous block (tile t - 3) has been loaded by every warp
      if (t >= kRkAcc && !mbar_wait_bounded(&accfree[acc], (uint32_t)(((t / kRkAcc) - 1) & 1)))
        return false;
      tc_fence_after();
      const uint32_t a0 = smem_u32(abuf), b0 = smem_u32(ring + st * kRkStage);
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk)
        tc_mma_bf16(tm + (uint32_t)(acc * 128),
                    sw128_desc(a0 + (kk >> 2) * kRkBlock + (kk & 3) * 32, 16, 1024),
                    sw128_desc(b0 + (kk >> 2) * kRkBlock + (kk & 3) * 32, 16, 1024), id_s,
                    kk > 0 ? 1u : 0u);
      tc_commit(&accfull[acc]);
      return true;
    };
    // the first two blocks' MMAs (the MMAs then run two blocks ahead of the epilogue)
    if (tid == 0) {
      if (!mma_s(tglob)) misc[0] = 1;
      if (njb > 1 && !misc[0] && !mma_s(tglob + 1)) misc[0] = 1;
    }
    for (int J = I; J < nb; ++J) {
      const int t = tglob + (J - I);
      const int acc = t % kRkAcc;
      if (tid == 0 && J + 2 < nb && !misc[0] && !mma_s(t + 2)) misc[0] = 1;
      const bool got = (misc[0] == 0) &&
                       mbar_wait_bounded(&accfull[acc], (uint32_t)((t / kRkAcc) & 1));
      if (!__all_sync(0xffffffffu, got)) {
        misc[0] = 1;
        ok = false;
        break;
      }
      tc_fence_after();
      // the stage of tile t is free again (its MMAs completed): refill it
      if (tid == 0 && J + kRkStages < nb) {
        load_tile(ring + (t % kRkStages) * kRkStage, J + kRkStages, &full[t % kRkStages]);
        issued = t + kRkStages + 1;
      }
      // columns 64*half .. +63 of block J: both warp-collective loads first, then
      // hand the accumulator back, then each thread's own (divergent) tests
      float v[2][32];
      __syncwarp();
      tmem_ld32(tm + (uint32_t)(acc * 128) + lanes + (uint32_t)(half * 64), v[0]);
      tmem_ld32(tm + (uint32_t)(acc * 128) + lanes + (uint32_t)(half * 64 + 32), v[1]);
      tmem_wait_ld();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&accfree[acc]);
#pragma unroll
      for (int cc = 0; cc < 2; ++cc) {
        const int j0 = J * kRkTile + half * 64 + cc * 32;   // first column token
        float mx = -INFINITY;
#pragma unroll
        for (int c = 0; c < 32; ++c) mx = fmaxf(mx, v[cc][c]);
        // quick rejection: cos >= tau needs S_ij >= tau ||k_i|| ||k_j|| >= thr_i * min ||k_j||
        if (mx < thr_i * nmin[j0 >> 5]) continue;
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          const int j = j0 + c;
          const bool valid = row < n && j < n && (J != I || j > row);
          if (valid && v[cc][c] * inv_s[j] >= thr_i) {
            if (pos_s[j] > pos_i) ++cnt;                 // a later near-duplicate of i
            else atomicAdd(&cnt_s[j], 1);                 // i is the later one: j is older
          }
        }
      }
    }
    // every warp is through this row block (and every accumulator it used is free)
    ok = __syncthreads_and(ok && misc[0] == 0);
    tglob += njb;
    if (!ok) break;
    if (row < n && cnt) atomicAdd(&cnt_s[row], cnt);
    __syncthreads();
    // block I is final: Z_i = lambda I_i - (1 - lambda) R_i
    if (half == 0 && row < n) {
      const float red_i = (cnt_s[row] >= ra.beta) ? 1.f : 0.f;
      z_s[row] = ra.lam * z_s[row] - (1.f - ra.lam) * red_i;
    }
  }
  ok = __syncthreads_and(ok && misc[0] == 0);

  // ---- selection: observation tokens first, then Z descending, ties to later ----
  if (ok) {
    int np2 = 256;
    while (np2 < n) np2 <<= 1;
    unsigned long long* key = reinterpret_cast<unsigned long long*>(ring);
    uint16_t* idx = reinterpret_cast<uint16_t*>(ring + kRkvMaxSlots * 8);
    for (int i = tid; i < np2; i += kRkThreads) {
      if (i < n) {
        const bool obs = pos_s[i] >= pnext - ra.alpha;
        const uint32_t hi = obs ? 0xFFFFFFFFu : orderable(z_s[i]);
        key[i] = ((unsigned long long)hi << 32) | (uint32_t)pos_s[i];
      } else {
        key[i] = 0ull;
      }
      idx[i] = (uint16_t)i;
    }
    __syncthreads();
    // bitonic sort, descending
    for (int kk = 2; kk <= np2; kk <<= 1) {
      for (int jj = kk >> 1; jj > 0; jj >>= 1) {
        for (int i = tid; i < np2; i += kRkThreads) {
          const int ixj = i ^ jj;
          if (ixj > i) {
            const bool desc = (i & kk) == 0;
            const unsigned long long a = key[i], c = key[ixj];
            if (desc ? (a < c) : (a > c)) {
              key[i] = c;
              key[ixj] = a;
              const uint16_t t = idx[i];
              idx[i] = idx[ixj];
              idx[ixj] = t;
            }
          }
        }
        __syncthreads();
      }
    }
    // kept flags (reuse the counts)
    for (int i = tid; i < kRkvMaxSlots; i += kRkThreads) cnt_s[i] = 0;
    __syncthreads();
    for (int r = tid; r < ra.budget; r += kRkThreads) cnt_s[idx[r]] = 1;
    __syncthreads();
    // ---- move: kept buffer tokens into the freed retained slots, in slot order ----
    int* freed = reinterpret_cast<int*>(ring);                  // reuse the ring
    int* movers = freed + kRkvMaxSlots;
    if (warp == 0) {   // ballot scans: freed retained slots and kept buffer slots, in order
      int nf = 0, nm = 0;
      for (int s0 = 0; s0 < n; s0 += 32) {
        const int sl = s0 + lane;
        const bool is_freed = sl < ra.budget && !cnt_s[sl];
        const bool is_mover = sl >= ra.budget && sl < n && cnt_s[sl];
        const unsigned fb = __ballot_sync(0xffffffffu, is_freed);
        const unsigned mb = __ballot_sync(0xffffffffu, is_mover);
        const unsigned below = (1u << lane) - 1u;
        if (is_freed) freed[nf + __popc(fb & below)] = sl;
        if (is_mover) movers[nm + __popc(mb & below)] = sl;
        nf += __popc(fb);
        nm += __popc(mb);
      }
      if (lane == 0) misc[1] = (nf == nm) ? nm : -1;
    }
    __syncthreads();
    const int nmove = misc[1];
    if (nmove < 0) {
      if (tid == 0) atomicOr(ra.err, LF_DEVERR_STATE);
    } else {
      T* Kw = ra.K + ubase * D;
      T* Vw = ra.V + ubase * D;
      for (int m = warp; m < nmove; m += kRkThreads / 32) {
        const int src = movers[m], dst = freed[m];
        const uint4* from = reinterpret_cast<const uint4*>(lane < 16 ? Kw + (size_t)src * D
                                                                       : Vw + (size_t)src * D);
        uint4* to = reinterpret_cast<uint4*>(lane < 16 ? Kw + (size_t)dst * D : Vw + (size_t)dst * D);
        to[lane & 15] = from[lane & 15];
        if (lane == 0) {
          ra.pos[ubase + dst] = pos_s[src];
          ra.vnorm[ubase + dst] = ra.vnorm[ubase + src];
        }
      }
      __syncthreads();
      for (int s = ra.budget + tid; s < n; s += kRkThreads) ra.pos[ubase + s] = -1;
      if (tid == 0) ra.count[unit] = ra.budget;
    }
  } else if (tid == 0) {
    // A wait ran out: leave the unit as it was, and let every copy this CTA
    // requested land before its shared memory is released.
    atomicOr(ra.err, LF_DEVERR_TIMEOUT);
    for (int t = max(0, issued - kRkStages); t < issued; ++t)
      (void)mbar_wait_bounded(&full[t % kRkStages], (uint32_t)((t / kRkStages) & 1));
    if (n_a > 0) (void)mbar_wait_bounded(afull, (uint32_t)((n_a - 1) & 1));
  }

  // ---- teardown ----------------------------------------------------------------
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tm, 512);
  }
}

}  // namespace

int rkv_smem_bytes() { return kSmem; }

const void* find_rkv_kernel(int group) {
  switch (group) {
    case 1: return reinterpret_cast<const void*>(&rkv_compress_kernel<1>);
    case 2: return reinterpret_cast<const void*>(&rkv_compress_kernel<2>);
    case 4: return reinterpret_cast<const void*>(&rkv_compress_kernel<4>);
    case 8: return reinterpret_cast<const void*>(&rkv_compress_kernel<8>);
    default: return nullptr;
  }
}

}  // namespace lf
