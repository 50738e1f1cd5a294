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
// One CTA per (sequence, KV head) unit, n <= 4096 cached tokens, with the
// warps split by role: a producer warp streams K tiles through a 3-stage TMA
// ring, an MMA warp issues every tcgen05.mma, and eight epilogue warps read
// the accumulators (thread <-> token row, each warp half of the columns).
//   pass 1  per 128-token tile, S = K_tile . Q_obs^T (M = 128, N = alpha * G
//           padded to 16) into one of two TMEM accumulators; every epilogue
//           thread keeps an online max / sum per observation query over its own
//           rows, and ||k||^2 of its row from the tile in shared memory; the
//           rows are merged once at the end;
//   pass 2  per 128-token row block I (held in its own buffer): importance of
//           its tokens, then the key dot products K_I . K_J^T (M = N = 128) for
//           every J >= I, the column tiles streamed through the ring into three
//           TMEM accumulators; a stage is refilled as soon as its MMAs
//           complete, so the stream runs ahead of the epilogue; each pair
//           (i, j) is looked at once and a near-duplicate pair counts for the
//           older token.  The column tiles of row block I come in the order
//           I+2, ..., then I+1, and the stage that holds tile I+1 becomes the
//           next row block's buffer (the old one takes its place in the ring),
//           so no row block is loaded twice and none waits for its load.  The
//           B x B cosine matrix never leaves the chip;
//   select  a radix select of the (Z, position) keys for the budget-th largest,
//           observation tokens first;
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

constexpr int kRkEpiWarps = 8;               // epilogue warps 0-7
constexpr int kRkEpi = kRkEpiWarps * 32;
constexpr int kRkProducerWarp = 8;
constexpr int kRkMmaWarp = 9;                // MMA warps 9 and 10: even and odd blocks
constexpr int kRkThreads = 352;
constexpr int kRkTile = 128;
constexpr int kRkStages = 3;
constexpr int kRkStage = kRkTile * 256;     // one K tile [128 rows][128 d] bf16: 32 KB
constexpr int kRkBlock = kRkTile * 128;     // one 64-column half of it: 16 KB
constexpr int kRkQRows = 64;                // observation query rows (alpha * G <= 64)
constexpr int kRkQBlock = kRkQRows * 128;   // one 64-column half of the query operand: 8 KB
constexpr int kRkAcc = 3;                   // key dot-product accumulators, 128 TMEM columns each
constexpr int kRkImpCol = kRkAcc * 128;     // two importance accumulators, 64 columns each
constexpr int kRkPrefetch = 6;              // ring tiles requested into L2 ahead of their load

// Pass 2 takes the row blocks in pairs p: I0 = 2p and I1 = 2p + 1 (when below
// nb), and streams each column tile J > I1 once for both: first I1+3 .. nb-1,
// then I1+2, then I1+1.  The last two become the next pair's row blocks.
__device__ __forceinline__ int pair_tiles(int I1, int nb) { return I1 < nb ? nb - I1 - 1 : 0; }
__device__ __forceinline__ int pair_kept(int m) { return m < 2 ? m : 2; }
__device__ __forceinline__ int pair_tile(int I1, int k, int m) {
  if (k < m - pair_kept(m)) return I1 + 3 + k;
  return k == m - 1 ? I1 + 1 : I1 + 2;
}

// A position in the producer's tile walk: pass 1 tile k, then column tile j of
// pair p; `keep` marks a tile that becomes the next pair's row block 1 (I1+2)
// or 0 (I1+1), else -1.
struct Walk {
  int k, p, j, keep;
};

// Shared-memory buffers behind the ring stages and the pair's two row blocks.
struct Bufs {
  unsigned char* stage[kRkStages];
  unsigned char* a[2];
  __device__ void swap(int st, int which) {
    unsigned char* t = stage[st];
    stage[st] = a[which];
    a[which] = t;
  }
};

// Shared-memory plan (offsets from a 1024-byte aligned base).
constexpr int kRkBars = 2 * kRkStages + 13;   // mbarriers (see the kernel)
constexpr int kOffBars = 0;
constexpr int kOffTmem = 256;
constexpr int kOffMisc = 272;      // [0] fail flag, [1] move count, [2] row blocks landed
constexpr int kOffStats = 512;     // m[64], l[64]
constexpr int kOffRed = 1024;      // [4 quarters][64 columns][2]
constexpr int kOffNmin = 3072;     // per 32-slot chunk: smallest ||k|| (128 chunks)
constexpr int kOffA = 4096;        // the two row blocks of pass 2
constexpr int kOffRing = kOffA + 2 * kRkStage;
constexpr int kOffQ = kOffRing + kRkStages * kRkStage;
constexpr int kOffInv = kOffQ + 2 * kRkQBlock;
constexpr int kOffCnt = kOffInv + kRkvMaxSlots * 4;       // 16-bit counts, two per word
constexpr int kOffZ = kOffCnt + kRkvMaxSlots * 2;
constexpr int kSmem = kOffZ + kRkvMaxSlots * 4 + 1024;  // + alignment slack
static_assert(kOffA % 1024 == 0 && kOffRing % 1024 == 0 && kOffQ % 1024 == 0, "alignment");
static_assert(kOffMisc + 16 <= kOffStats && kOffStats + 2 * kRkQRows * 4 <= kOffRed, "header");
// the sort reuses the ring: 64-bit keys then 16-bit slot indices
static_assert(kRkvMaxSlots * 10 <= kRkStages * kRkStage, "sort space");
static_assert(kOffBars + kRkBars * 8 <= kOffTmem, "barriers");

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
  const int quarter = warp & 3;     // epilogue: TMEM lanes 32*quarter .. +31
  const int half = (warp >> 2) & 1;  // epilogue: which half of the accumulator's columns
  const int QN = ra.alpha * G;      // observation query rows
  const int QN16 = (QN + 15) & ~15;
  const size_t ubase = (size_t)unit * ra.slot_stride;

  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffBars);
  // barriers: full / empty per ring stage, then the fixed ones
  uint64_t* full = bars;                      // [kRkStages] ring stage landed
  uint64_t* empty = bars + kRkStages;         // [kRkStages] ring stage read (by the epilogue)
  uint64_t* fixed = bars + 2 * kRkStages;
  uint64_t* afull = fixed;                    // row block 0 landed
  uint64_t* drain2 = fixed + 1;               // every MMA of the second MMA warp complete
  uint64_t* impfull = fixed + 2;              // [2] importance logits ready
  uint64_t* impfree = fixed + 4;              // [2] ... loaded by every epilogue warp
  uint64_t* accfull = fixed + 6;              // [3] key dot products of a block ready
  uint64_t* accfree = fixed + 9;              // [3] ... loaded by every epilogue warp
  uint64_t* drain = fixed + 12;               // every MMA of the first MMA warp complete
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffTmem);
  volatile int* misc = reinterpret_cast<volatile int*>(smem + kOffMisc);
  float* m_col = reinterpret_cast<float*>(smem + kOffStats);
  float* l_col = m_col + kRkQRows;
  float* red = reinterpret_cast<float*>(smem + kOffRed);
  float* nmin = reinterpret_cast<float*>(smem + kOffNmin);
  unsigned char* abuf = smem + kOffA;
  unsigned char* ring = smem + kOffRing;
  unsigned char* qop = smem + kOffQ;
  const int32_t* posg = ra.pos + ubase;   // positions, read from global memory (L2)
  float* inv_s = reinterpret_cast<float*>(smem + kOffInv);
  // Near-duplicate counts, 16 bits per token (at most n - 1 < 65536: no carry
  // into the neighbour), added with 32-bit atomics on the word holding them.
  uint32_t* cnt_w = reinterpret_cast<uint32_t*>(smem + kOffCnt);
  auto cnt_add = [&](int i, int v) { atomicAdd(&cnt_w[i >> 1], (uint32_t)v << ((i & 1) * 16)); };
  auto cnt_get = [&](int i) { return (int)((cnt_w[i >> 1] >> ((i & 1) * 16)) & 0xFFFFu); };
  float* z_s = reinterpret_cast<float*>(smem + kOffZ);

  const int n = ra.count[unit];
  if (n <= ra.budget) return;   // nothing above the budget: uniform for the CTA
  if (n > kRkvMaxSlots || n > ra.slot_stride) {
    if (tid == 0) atomicOr(ra.err, LF_DEVERR_STATE);
    return;
  }
  const int nb = (n + kRkTile - 1) / kRkTile;
  const int pnext = ra.next_pos[unit];

  // ---- set-up: barriers, tensor memory, positions, the query operand -------------
  if (tid == 0) {
    for (int i = 0; i < kRkBars; ++i) {  // impfree, accfree: one arrival per epilogue warp
      const bool per_warp = (&bars[i] >= impfree && &bars[i] < impfree + 2) ||
                            (&bars[i] >= accfree && &bars[i] < accfree + kRkAcc);
      mbar_init(&bars[i], per_warp ? kRkEpiWarps : 1);
    }
    fence_mbar_init();
    misc[0] = 0;
    misc[2] = 0;
  }
  if (warp == 0) {
    __syncwarp();  // warp-collective allocation (thread 0 initialised the barriers alone)
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  for (int i = tid; i < kRkvMaxSlots; i += kRkThreads) {
    if (i < kRkvMaxSlots / 2) cnt_w[i] = 0u;
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
  const int row0 = ra.row_base + (int)ubase;

  // K tiles are read again for every row block: ask L2 to keep them
  const uint64_t pol = l2_evict_last_policy();
  auto load_tile_tx = [&](unsigned char* dst, int t, uint64_t* bar) {  // bytes announced by the caller
    for (int blk = 0; blk < 2; ++blk)
      for (int ro = 0; ro < kRkTile; ro += 64)
        tma_load_2d(dst + blk * kRkBlock + ro * 128, &ra.kmap, blk * 64, row0 + t * kRkTile + ro,
                    bar, pol);
  };
  auto load_tile = [&](unsigned char* dst, int t, uint64_t* bar) {
    mbar_arrive_expect_tx(bar, (uint32_t)kRkStage);
    load_tile_tx(dst, t, bar);
  };

  // The producer's tile walk (loads, L2 requests), in the order the MMA warps
  // and the epilogue take the tiles: pass 1 tiles 0..nb-1, then per pair its
  // column tiles in pair_tile order; -1 at the end.
  auto next = [&](Walk& w) -> int {
    w.keep = -1;
    if (w.k < nb) return w.k++;
    for (;;) {
      const int I1 = 2 * w.p + 1;
      if (I1 >= nb) return -1;   // no pair from here on has column tiles
      const int m = pair_tiles(I1, nb);
      if (w.j < m) {
        const int k = w.j++;
        if (k == m - 1) w.keep = 0;
        else if (pair_kept(m) == 2 && k == m - 2) w.keep = 1;
        return pair_tile(I1, k, m);
      }
      ++w.p;
      w.j = 0;
    }
  };
  // The buffers behind the ring's stages and the row blocks (the producer and
  // the MMA warps make the same swaps: the producer when it loads a kept tile,
  // the MMA warps when the pair is done with the old row blocks).
  auto initial_bufs = [&]() {
    Bufs b;
    for (int i = 0; i < kRkStages; ++i) b.stage[i] = ring + i * kRkStage;
    b.a[0] = abuf;
    b.a[1] = abuf + kRkStage;
    return b;
  };

  if (warp == kRkProducerWarp) {
    // ---- producer: the ring's tile sequence, pass 1 tiles 0..nb-1, then for
    // each pair of row blocks its column tiles.  The ring is
    // latency-bound (the tiles mostly come from L2), so every tile is also
    // requested into L2 kRkPrefetch places ahead of its load. ----------------------
    if (lane == 0) {
      Walk ahead{0, 0, 0, -1};
      for (int q = 0; q < kRkPrefetch; ++q) {
        const int t = next(ahead);
        if (t < 0) break;
        for (int ro = 0; ro < kRkTile; ro += 64)
          for (int blk = 0; blk < 2; ++blk)
            tma_prefetch_l2_2d(&ra.kmap, blk * 64, row0 + t * kRkTile + ro);
      }
      Walk cur{0, 0, 0, -1};
      Bufs bf = initial_bufs();
      int tt = 0;       // ring tiles issued
      for (int t = next(cur); t >= 0; t = next(cur), ++tt) {
        const int st = tt % kRkStages;
        if (tt >= kRkStages &&
            (misc[0] || !mbar_wait_bounded(&empty[st], (uint32_t)(((tt / kRkStages) - 1) & 1)))) {
          misc[0] = 1;
          break;
        }
        load_tile(bf.stage[st], t, &full[st]);
        if (cur.keep >= 0) bf.swap(st, cur.keep);  // the next pair's row block
        const int tp = next(ahead);
        if (tp >= 0)
          for (int ro = 0; ro < kRkTile; ro += 64)
            for (int blk = 0; blk < 2; ++blk)
              tma_prefetch_l2_2d(&ra.kmap, blk * 64, row0 + tp * kRkTile + ro);
      }
      // every copy issued lands before the CTA may exit
      for (int t = max(0, tt - kRkStages); t < tt; ++t)
        (void)mbar_wait_bounded(&full[t % kRkStages], (uint32_t)((t / kRkStages) & 1));
    }
    __syncwarp();
  } else if (warp == kRkMmaWarp || warp == kRkMmaWarp + 1) {
    // ---- MMA warps (lane 0 of each): the same tile order as the producer.  The
    // two warps take turns, item by item (a tile's importance in pass 1, and in
    // pass 2 a row block's importance and its key dot-product blocks), so that
    // one issues while the other waits on its barriers: a single issuing thread
    // left the tensor cores idle between blocks.  Both walk every item to keep
    // the same counters; each waits only for what its own MMAs read. ----------
    if (lane == 0) {
      const int par = warp - kRkMmaWarp;
      const uint32_t id_imp = idesc_bf16_f32(128, QN16, false, false);
      const uint32_t id_s = idesc_bf16_f32(128, 128, false, false);
      const uint32_t q0 = smem_u32(qop);
      bool fail = false;
      int rt = 0;   // ring tiles consumed
      int it = 0;   // importance items (accumulator it % 2 = the warp that takes it)
      int at = 0;   // key dot-product blocks (accumulator at % kRkAcc)
      auto wait = [&](uint64_t* bar, uint32_t parity) {
        if (!fail && (misc[0] || !mbar_wait_bounded(bar, parity))) fail = true;
        return !fail;
      };
      // S = tile . Q^T into importance accumulator it % 2, by warp it % 2
      auto mma_imp = [&](uint32_t a0) {
        const int ib = it & 1;
        if (ib == par && !fail) {
          if (it >= 2 && !wait(&impfree[ib], (uint32_t)(((it >> 1) - 1) & 1))) return;
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk)
            tc_mma_bf16(tm + (uint32_t)(kRkImpCol + ib * 64),
                        sw128_desc(a0 + (kk >> 2) * kRkBlock + (kk & 3) * 32, 16, 1024),
                        sw128_desc(q0 + (kk >> 2) * kRkQBlock + (kk & 3) * 32, 16, 1024),
                        id_imp, kk > 0 ? 1u : 0u);
          tc_commit(&impfull[ib]);
        }
        ++it;
      };
      // row blocks 0 and 1 (the others come through the ring): request them now
      if (par == 0) {
        mbar_arrive_expect_tx(afull, (uint32_t)((nb > 1 ? 2 : 1) * kRkStage));
        load_tile_tx(abuf, 0, afull);
        if (nb > 1) load_tile_tx(abuf + kRkStage, 1, afull);
      }
      // pass 1: the stage is released by the epilogue (it also reads ||k|| there)
      for (int t = 0; t < nb && !fail; ++t) {
        const int st = rt % kRkStages;
        if ((it & 1) == par) {
          if (!wait(&full[st], (uint32_t)((rt / kRkStages) & 1))) break;
          tc_fence_after();
        }
        mma_imp(smem_u32(ring + st * kRkStage));
        ++rt;
      }
      // pass 2, in pairs of row blocks
      Bufs bf = initial_bufs();
      volatile int* landed = misc + 2;   // kept tiles known to have landed
      int kept_before = 0;               // kept tiles of the pairs so far
      // One key dot-product block into accumulator at % kRkAcc, by warp at % 2:
      // A = aop's 128 keys, B = bop's; st >= 0: bop is ring stage st.  `mark`:
      // the tile becomes a row block of the next pair, count it as landed.
      auto block = [&](uint32_t aop, uint32_t bop, int st, bool mark) {
        const int acc = at % kRkAcc;
        if ((at & 1) == par && !fail) {
          if (at >= kRkAcc && !wait(&accfree[acc], (uint32_t)(((at / kRkAcc) - 1) & 1))) return;
          if (st >= 0 && !wait(&full[st], (uint32_t)((rt / kRkStages) & 1))) return;
          if (mark) {
            __threadfence_block();
            atomicAdd(const_cast<int*>(landed), 1);
          }
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk)
            tc_mma_bf16(tm + (uint32_t)(acc * 128),
                        sw128_desc(aop + (kk >> 2) * kRkBlock + (kk & 3) * 32, 16, 1024),
                        sw128_desc(bop + (kk >> 2) * kRkBlock + (kk & 3) * 32, 16, 1024), id_s,
                        kk > 0 ? 1u : 0u);
          tc_commit(&accfull[acc]);
        }
        ++at;
      };
      for (int p = 0; 2 * p < nb && !fail; ++p) {
        const int I1 = 2 * p + 1;
        const bool has1 = I1 < nb;
        const int m = pair_tiles(I1, nb);
        // The pair's row blocks have landed: rows 0 and 1 by their own copy, the
        // others as the previous pair's kept tiles, which one of the two warps
        // waited for and counted (a stage's barrier may have moved on to its
        // next tile by the time the other warp gets here).
        if (p == 0) {
          if (!wait(afull, 0)) break;
        } else if (*landed < kept_before) {
          const unsigned long long t0 = global_ns();
          while (*landed < kept_before && !misc[0]) {
            __nanosleep(32);
            if (global_ns() - t0 > kWaitLimitNs) break;
          }
          if (*landed < kept_before) {
            fail = true;
            break;
          }
        }
        __threadfence_block();
        tc_fence_after();
        const uint32_t a0 = smem_u32(bf.a[0]), a1 = smem_u32(bf.a[1]);
        mma_imp(a0);
        if (has1) mma_imp(a1);
        block(a0, a0, -1, false);        // K_I0 . K_I0^T
        if (has1) {
          block(a0, a1, -1, false);      // K_I0 . K_I1^T
          block(a1, a1, -1, false);      // K_I1 . K_I1^T
        }
        int keep_st[2] = {-1, -1};
        for (int k = 0; k < m && !fail; ++k) {
          const int st = rt % kRkStages;
          const int keep = (k == m - 1) ? 0 : (pair_kept(m) == 2 && k == m - 2) ? 1 : -1;
          const uint32_t b0 = smem_u32(bf.stage[st]);
          block(a0, b0, st, keep >= 0);
          block(a1, b0, st, false);
          if (keep >= 0) keep_st[keep] = st;
          ++rt;
        }
        // The epilogue hands the kept tiles' stages back after the pair's last
        // block, so after every MMA on the old row blocks, whose buffers take
        // their places in the ring.
        if (keep_st[1] >= 0) bf.swap(keep_st[1], 1);
        if (keep_st[0] >= 0) bf.swap(keep_st[0], 0);
        kept_before += pair_kept(m);
      }
      if (fail) misc[0] = 1;
      // every MMA issued completes before tensor memory is released, and row
      // block 0 lands before the CTA may exit
      uint64_t* dr = par == 0 ? drain : drain2;
      tc_commit(dr);
      (void)mbar_wait_bounded(dr, 0);
      if (par == 0) (void)mbar_wait_bounded(afull, 0);
    }
    __syncwarp();
  } else {
    // ---- epilogue warps 0-7 ------------------------------------------------------
    const int r = quarter * 32 + lane;              // this thread's row of a tile
    const uint32_t lanes = (uint32_t)(quarter * 32) << 16;
    bool bad = false;                               // this warp gave up waiting
    auto wait = [&](uint64_t* bar, uint32_t parity) {
      if (!bad && (misc[0] || !__all_sync(0xffffffffu, mbar_wait_bounded(bar, parity)))) {
        bad = true;
        if (lane == 0) misc[0] = 1;
      }
      return !bad;
    };
    // importance logits of accumulator it % 2 (32 columns from 32 * half),
    // scaled to log2 units; -inf outside the tokens and the query rows
    int it = 0;
    auto imp_logits = [&](int row, float* s) -> bool {
      const int ib = it & 1;
      const bool got = wait(&impfull[ib], (uint32_t)((it >> 1) & 1));
      ++it;
      if (!got) return false;
      tc_fence_after();
      __syncwarp();  // tcgen05.ld is warp-collective
      tmem_ld32(tm + (uint32_t)(kRkImpCol + ib * 64) + lanes + (uint32_t)(half * 32), s);
      tmem_wait_ld();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&impfree[ib]);
#pragma unroll
      for (int c = 0; c < 32; ++c)
        s[c] = (row < n && half * 32 + c < QN) ? s[c] * ra.scale_log2 : -INFINITY;
      return true;
    };

    // ---- pass 1: every observation query's max and softmax denominator, kept
    // per thread over its own rows (online), and ||k||^2 --------------------------
    float m[32], l[32];
#pragma unroll
    for (int c = 0; c < 32; ++c) {
      m[c] = -INFINITY;
      l[c] = 0.f;
    }
    for (int t = 0; t < nb; ++t) {
      const int row = t * kRkTile + r;
      const int st = t % kRkStages;
      float s[32];
      const bool got = imp_logits(row, s) && wait(&full[st], (uint32_t)((t / kRkStages) & 1));
      if (got) {
        // ||k||^2 of this thread's token, d-half `half`, from the tile in shared memory
        // (row r of the 64-column block at r * 128 bytes, 16-byte chunks swizzled by r mod 8)
        const unsigned char* rp = ring + st * kRkStage + half * kRkBlock + r * 128;
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
      // every epilogue warp has read the stage (the MMAs on it completed before
      // the logits were ready): hand it back to the producer
      named_bar_sync(1, kRkEpi);
      if (tid == 0 && !misc[0]) mbar_arrive(&empty[st]);
      if (got) {
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          const float x = s[c];
          const float mn = fmaxf(m[c], x);   // branch-free: every lane the same path
          if (mn != -INFINITY) {
            l[c] = l[c] * exp2f(m[c] - mn) + exp2f(x - mn);
            m[c] = mn;
          }
        }
      }
    }
    // merge the rows: the 32 lanes of the warp, then the four quarters
#pragma unroll
    for (int c = 0; c < 32; ++c) {
      float mc = m[c], lc = l[c];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float mo = __shfl_xor_sync(0xffffffffu, mc, o);
        const float lo = __shfl_xor_sync(0xffffffffu, lc, o);
        const float mn = fmaxf(mc, mo);
        if (mn != -INFINITY) {
          lc = lc * exp2f(mc - mn) + lo * exp2f(mo - mn);
          mc = mn;
        }
      }
      if (lane == 0) {
        red[(quarter * kRkQRows + half * 32 + c) * 2] = mc;
        red[(quarter * kRkQRows + half * 32 + c) * 2 + 1] = lc;
      }
    }
    named_bar_sync(1, kRkEpi);
    if (tid < QN) {
      float mc = -INFINITY, lc = 0.f;
      for (int q = 0; q < 4; ++q) {
        const float bm = red[(q * kRkQRows + tid) * 2], bl = red[(q * kRkQRows + tid) * 2 + 1];
        if (bm == -INFINITY) continue;
        const float mn = fmaxf(mc, bm);
        lc = (mc == -INFINITY ? 0.f : lc * exp2f(mc - mn)) + bl * exp2f(bm - mn);
        mc = mn;
      }
      m_col[tid] = mc;
      l_col[tid] = lc;
    }
    // 1/||k_i|| (0 for a zero key: never similar), and the smallest ||k|| of every
    // 32-slot chunk for the quick rejection below
    for (int i = tid; i < n; i += kRkEpi) {
      const float ss = inv_s[i];
      inv_s[i] = (ss > 0.f) ? rsqrtf(ss) : 0.f;
    }
    named_bar_sync(1, kRkEpi);
    if (tid < kRkvMaxSlots / 32) {
      float mn = INFINITY;
      for (int c = 0; c < 32; ++c) {
        const float iv = inv_s[tid * 32 + c];
        if (iv > 0.f) mn = fminf(mn, 1.f / iv);
      }
      nmin[tid] = mn;
    }
    named_bar_sync(1, kRkEpi);

    // ---- pass 2: importance, then near-duplicate counts over blocks J >= I, ----
    // in the MMA warps' order: per pair, both row blocks' importance, the blocks
    // (I0, I0), (I0, I1), (I1, I1), then (I0, J), (I1, J) per column tile.
    int at = 0;
    int rt = nb;   // ring tiles consumed (pass 1 took nb)
    // This thread's token of a row block: its importance, then its state.
    struct RowState {
      int row, pos;
      float thr;
      int cnt;
    };
    auto row_start = [&](int I) -> RowState {
      RowState rs;
      rs.row = I * kRkTile + r;
      float s[32];
      if (imp_logits(rs.row, s)) {
        float part = 0.f;
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          const int col = half * 32 + c;
          if (col < QN && s[c] != -INFINITY) part += exp2f(s[c] - m_col[col]) / l_col[col];
        }
        if (rs.row < n) atomicAdd(&z_s[rs.row], part / (float)QN);
      }
      const float inv_i = (rs.row < n) ? inv_s[rs.row] : 0.f;
      rs.thr = (inv_i > 0.f) ? ra.tau / inv_i : INFINITY;   // tau * ||k_i||
      rs.pos = (rs.row < n) ? posg[rs.row] : INT_MIN;
      rs.cnt = 0;
      return rs;
    };
    // Block `at` (row block of rs, column block J; diag: J is rs's own row
    // block, only j > row counts); release: ring stage to hand back once its
    // products are read (-1: none), release2 a second one.
    auto take_block = [&](RowState& rs, int J, bool diag, int release, int release2) {
      const int acc = at % kRkAcc;
      const bool got = wait(&accfull[acc], (uint32_t)((at / kRkAcc) & 1));
      ++at;
      if (!got) return;
      // every block so far is complete: those stages may be refilled
      if (tid == 0) {
        if (release >= 0) mbar_arrive(&empty[release]);
        if (release2 >= 0) mbar_arrive(&empty[release2]);
      }
      tc_fence_after();
      // columns 64*half .. +63 of block J: both warp-collective loads first, then
      // hand the accumulator back, then each thread's own tests
      float v[2][32];
      __syncwarp();
      tmem_ld32(tm + (uint32_t)(acc * 128) + lanes + (uint32_t)(half * 64), v[0]);
      tmem_ld32(tm + (uint32_t)(acc * 128) + lanes + (uint32_t)(half * 64 + 32), v[1]);
      tmem_wait_ld();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&accfree[acc]);
      const int row = rs.row;
      const float thr_i = rs.thr;
#pragma unroll
      for (int cc = 0; cc < 2; ++cc) {
        const int j0 = J * kRkTile + half * 64 + cc * 32;   // first column token
        float mx = -INFINITY;
#pragma unroll
        for (int c = 0; c < 32; ++c) mx = fmaxf(mx, v[cc][c]);
        // quick rejection: cos >= tau needs S_ij >= tau ||k_i|| ||k_j|| >= thr_i * min ||k_j||
        const bool rejected = mx < thr_i * nmin[j0 >> 5];
        if (__all_sync(0xffffffffu, rejected)) continue;
        // The exact test on every column, the same instructions for every lane
        // (the chunk's 1/||k_j|| are broadcast loads), as a mask of hits.
        uint32_t hits = 0;
        const float4* iv4 = reinterpret_cast<const float4*>(inv_s + j0);
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const float4 w = iv4[q];
          hits |= (v[cc][4 * q] * w.x >= thr_i ? 1u : 0u) << (4 * q);
          hits |= (v[cc][4 * q + 1] * w.y >= thr_i ? 1u : 0u) << (4 * q + 1);
          hits |= (v[cc][4 * q + 2] * w.z >= thr_i ? 1u : 0u) << (4 * q + 2);
          hits |= (v[cc][4 * q + 3] * w.w >= thr_i ? 1u : 0u) << (4 * q + 3);
        }
        // only tokens (j < n), and on a diagonal block only j > row
        const int lim = n - j0;
        if (rejected || row >= n || lim <= 0) hits = 0;
        else if (lim < 32) hits &= (1u << lim) - 1u;
        if (diag) {
          const int d = row - j0 + 1;   // columns c >= d have j > row
          if (d >= 32) hits = 0;
          else if (d > 0) hits &= ~((1u << d) - 1u);
        }
        while (hits) {
          const int j = j0 + __ffs(hits) - 1;
          hits &= hits - 1u;
          if (posg[j] > rs.pos) ++rs.cnt;               // a later near-duplicate of i
          else cnt_add(j, 1);                           // i is the later one: j is older
        }
      }
    };
    for (int p = 0; 2 * p < nb; ++p) {
      const int I0 = 2 * p, I1 = I0 + 1;
      const bool has1 = I1 < nb;
      const int m = pair_tiles(I1, nb);
      RowState r0 = row_start(I0);
      RowState r1 = has1 ? row_start(I1) : r0;
      take_block(r0, I0, true, -1, -1);
      if (has1) {
        take_block(r0, I1, false, -1, -1);
        take_block(r1, I1, true, -1, -1);
      }
      // A tile's stage goes back after its second block, but the tile kept as
      // the next pair's row block 1 only with the last block of the pair: the
      // old row block 1, whose buffer refills that stage, is read until then.
      int held = -1;
      for (int k = 0; k < m; ++k) {
        const int J = pair_tile(I1, k, m);
        const int st = (rt++) % kRkStages;
        const bool keep1 = pair_kept(m) == 2 && k == m - 2;
        take_block(r0, J, false, -1, -1);
        take_block(r1, J, false, keep1 ? -1 : st, k == m - 1 ? held : -1);
        if (keep1) held = st;
      }
      if (r0.row < n && r0.cnt) cnt_add(r0.row, r0.cnt);
      if (has1 && r1.row < n && r1.cnt) cnt_add(r1.row, r1.cnt);
    }
  }
  const bool ok = __syncthreads_and(misc[0] == 0);

  // ---- selection: observation tokens first, then Z descending, ties to later ----
  // Every token gets a unique 64-bit key (observation flag or orderable Z, then
  // its position); the `budget` largest keys stay.  A radix select finds the
  // m-th smallest key, m = n - budget, 8 bits per pass from the top: count the
  // keys that share the prefix found so far by their next byte, then take the
  // byte in which the remaining rank falls.  Tokens above that key are kept.
  if (ok) {
    // every count is in: Z_i = lambda I_i - (1 - lambda) R_i
    for (int i = tid; i < n; i += kRkThreads)
      z_s[i] = ra.lam * z_s[i] - (1.f - ra.lam) * ((cnt_get(i) >= ra.beta) ? 1.f : 0.f);
    __syncthreads();
    unsigned long long* key = reinterpret_cast<unsigned long long*>(ring);   // [n]
    int* hist = reinterpret_cast<int*>(ring + kRkvMaxSlots * 8);            // [256]
    unsigned long long* sel_prefix = reinterpret_cast<unsigned long long*>(smem + kOffMisc + 16);
    int* sel_rank = reinterpret_cast<int*>(smem + kOffMisc + 24);
    for (int i = tid; i < n; i += kRkThreads) {
      const int pi = posg[i];
      const bool obs = pi >= pnext - ra.alpha;
      const uint32_t hi = obs ? 0xFFFFFFFFu : orderable(z_s[i]);
      key[i] = ((unsigned long long)hi << 32) | (uint32_t)pi;
    }
    if (tid == 0) {
      *sel_prefix = 0ull;
      *sel_rank = n - ra.budget;   // 1-based rank of the largest dropped key
    }
    const int nwalk = (n + kRkThreads - 1) / kRkThreads * kRkThreads;
    for (int shift = 56; shift >= 0; shift -= 8) {
      if (tid < 256) hist[tid] = 0;
      __syncthreads();
      const unsigned long long prefix = *sel_prefix;
      const unsigned long long hmask = (shift == 56) ? 0ull : (~0ull << (shift + 8));
      // warp-aggregated counts: lanes with the same byte add once
      for (int i = tid; i < nwalk; i += kRkThreads) {
        int digit = 256;
        if (i < n) {
          const unsigned long long k = key[i];
          if ((k & hmask) == prefix) digit = (int)((k >> shift) & 255u);
        }
        const unsigned peers = __match_any_sync(0xffffffffu, digit);
        if (digit < 256 && lane == __ffs(peers) - 1) atomicAdd(&hist[digit], __popc(peers));
      }
      __syncthreads();
      if (warp == 0) {
        // lane L holds bytes 8L .. 8L+7; find the byte where the rank falls
        int c[8], sum = 0;
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          c[q] = hist[lane * 8 + q];
          sum += c[q];
        }
        int incl = sum;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int y = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += y;
        }
        const int rank = *sel_rank;
        const int excl = incl - sum;
        if (rank > excl && rank <= incl) {
          // the first of this lane's bytes at which the running count reaches the rank
          int below = excl, qs = 7;
          bool found = false;
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            if (!found && below + c[q] >= rank) {
              qs = q;
              found = true;
            } else if (!found) {
              below += c[q];
            }
          }
          *sel_prefix = prefix | ((unsigned long long)(lane * 8 + qs) << shift);
          *sel_rank = rank - below;
        }
      }
      __syncthreads();
    }
    // kept flags: every key above the largest dropped one
    const unsigned long long kcut = *sel_prefix;
    int* kept = reinterpret_cast<int*>(z_s);   // Z is in the keys now: reuse its space
    for (int i = tid; i < kRkvMaxSlots; i += kRkThreads) kept[i] = (i < n && key[i] > kcut) ? 1 : 0;
    __syncthreads();
    // ---- move: kept buffer tokens into the freed retained slots, in slot order ----
    int* freed = reinterpret_cast<int*>(ring);                  // reuse the ring
    int* movers = freed + kRkvMaxSlots;
    if (warp == 0) {   // ballot scans: freed retained slots and kept buffer slots, in order
      int nf = 0, nm = 0;
      for (int s0 = 0; s0 < n; s0 += 32) {
        const int sl = s0 + lane;
        const bool is_freed = sl < ra.budget && !kept[sl];
        const bool is_mover = sl >= ra.budget && sl < n && kept[sl];
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
          ra.pos[ubase + dst] = posg[src];   // src >= budget > dst: never a moved slot
          ra.vnorm[ubase + dst] = ra.vnorm[ubase + src];
        }
      }
      __syncthreads();
      for (int s = ra.budget + tid; s < n; s += kRkThreads) ra.pos[ubase + s] = -1;
      if (tid == 0) ra.count[unit] = ra.budget;
    }
  } else if (tid == 0) {
    // A wait ran out: leave the unit as it was (the producer has waited for every
    // copy it requested, the MMA warp for every MMA).
    atomicOr(ra.err, LF_DEVERR_TIMEOUT);
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

int rkv_threads() { return kRkThreads; }

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
