// Causal (or full) prefill attention forward on sm_103a: TMA + tcgen05 + TMEM.
//
// What it computes: "Why your local LLM feels dumber than it is" (Part 3.14),
// section "What attention is trying to calculate" -- O = softmax(scale*QK^T) V
// per query row over the keys it may see (causal: keys j <= i), plus the
// natural-log LSE of each row.
//
// How (the tiled flow of "Streaming process -- How the SM works inside a
// transformer", Steps 3-8 and its code snippet, redesigned for tcgen05):
//   * the kernel is persistent: one CTA per SM walks a list of work tiles
//     (one 128-row Q tile of one (sequence, query head) each), longest causal
//     tiles first, and keeps its pipelines running across tile boundaries.
//     Sequences are a batch of equal length, packed (cu_seqlens), or new
//     tokens whose keys come from a paged KV cache (block table);
//   * two producer warps stream Q (once per tile, Step 3) and the K and V
//     tiles (128 keys; 64 at d = 256) through shared-memory rings with
//     mbarrier full/empty pairs (Step 6).  Q is double-buffered (single at
//     d = 256), so the next tile's Q arrives while this tile still runs; two K
//     stages, two V stages (three at d = 64).  With a paged cache each lane
//     issues one 16-token page copy;
//   * one warp issues S_j = Q K_j^T into TMEM (Step 4).  S is triple-buffered
//     in TMEM, so the tensor core computes S two steps ahead of softmax.  A
//     second warp issues O += P_j V_j with P (bf16, over the first half of
//     S_j's columns) read straight from TMEM once softmax has written it
//     (Step 7).  Each issuing warp runs its loop converged and one elected
//     lane issues: with warp-uniform operands a tcgen05.mma issues in about
//     the 64 cycles a 128x128x16 product takes, and two issuers let one wait
//     on a barrier while the other keeps the tensor core fed;
//   * eight softmax warps, each with 16 whole rows of the tile (four threads
//     per row through the 16x256b TMEM access shape).  Each thread reads its
//     scores from TMEM, masks, takes the row max (two shuffles within the
//     row's four threads), exponentiates with ex2 and keeps its share of the
//     running sum (Step 5).  No warp waits for another, so the two softmax
//     warps that share a scheduler interleave their phases.  O is rescaled
//     only when the row max has grown by more than 2^8 since it was last
//     applied -- exact either way, because O and l always refer to the same
//     max;
//   * at the end of a tile the softmax warps hand l and the row max to a
//     fourth warpgroup and go straight on to the next tile.  That epilogue
//     warpgroup (one thread per row) writes LSE = m*scale + ln(l), waits for
//     the last P_j V_j, reads O out of TMEM, releases it for the next tile's
//     first product, divides by l, rounds to bf16 and stores the tile with
//     TMA through a 128B-swizzled staging panel (Step 8).  Tile boundaries
//     therefore cost the softmax warps almost nothing;
//   * the first tile's Q, K and V loads are issued by the thread that sets up
//     the barriers, before the CTA-wide barrier and the TMEM allocation.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cfloat>
#include <cstdint>

#include "prefill.h"
#include "prefill_tile.cuh"
#include "prefill_walk.cuh"
#include "sm103.cuh"

namespace attn {

__device__ uint32_t g_prefill_status;

namespace {

using pf::BM;                    // query rows per work tile (TMEM lanes)
constexpr int NSB = 3;           // S buffers in TMEM
constexpr int NUM_THREADS = 512; // 8 softmax warps, 2 TMA warps, 2 MMA warps, 4 epilogue warps
constexpr int PRODUCER_WARP = 8; // loads Q and streams K
constexpr int V_WARP = 11;       // streams V
constexpr int MMA_WARP = 9;      // issues S = Q K^T, owns the TMEM allocation
constexpr int PV_WARP = 10;      // issues O += P V
constexpr int EPI_WARP0 = 12;    // warps 12..15: epilogue, one thread per row
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t REG_SOFTMAX = 168, REG_OTHER = 64, REG_EPI = 112;  // registers per thread, see below
static_assert(8 * 32 * REG_SOFTMAX + 4 * 32 * REG_OTHER + 4 * 32 * REG_EPI == 128 * NUM_THREADS, "register split");
using pf::PANEL_ROW;             // bytes of one 128B-swizzle panel row: 64 bf16

// Tiling and shared-memory layout per head dim.  d <= 128: 128-key K/V tiles, two Q buffers (the
// next tile's Q loads while this one runs), two K stages and two V stages (three at d = 64).
// d = 256: 64-key tiles, one Q buffer and two stages of each, so that Q and the rings fit in
// shared memory and O (256 columns) plus three S buffers fit in the 512 TMEM columns.
template <int D>
struct Layout {
  static constexpr int BN = D <= 128 ? 128 : 64;        // keys per K/V tile
  static constexpr int Q_STAGES = D <= 128 ? 2 : 1;     // Q buffers
  static constexpr int K_STAGES = 2;                    // K_j is free as soon as S_j is done
  static constexpr int V_STAGES = D <= 64 ? 3 : 2;      // V_j is held until P_j V_j is done
  static constexpr int CHUNKS = D / 64;                 // 64-column panels per row
  static constexpr int Q_PANEL = BM * PANEL_ROW;        // one panel of a Q (or output) tile
  static constexpr int KV_PANEL = BN * PANEL_ROW;       // one panel of a K or V tile
  static constexpr int Q_BYTES = CHUNKS * Q_PANEL;
  static constexpr int KV_BYTES = CHUNKS * KV_PANEL;
  static constexpr uint32_t O_COL = NSB * BN;           // O accumulator columns start here
  static constexpr int OGRP = D < 128 ? D : 128;        // O columns the epilogue holds at once
  static constexpr int Q_OFF = 0;
  static constexpr int K_OFF = Q_OFF + Q_STAGES * Q_BYTES;
  static constexpr int V_OFF = K_OFF + K_STAGES * KV_BYTES;
  static constexpr int OST_OFF = V_OFF + V_STAGES * KV_BYTES;   // output staging: one 64-column panel
  // a tile's row sums and row maxima, handed to the epilogue: [2 tiles][2][128]
  static constexpr int XL_OFF = OST_OFF + Q_PANEL;
  static constexpr int BAR_OFF = XL_OFF + 2 * 2 * 128 * 4;
  // q_full[Q], q_empty[Q], k_full[K], k_empty[K], v_full[V], v_empty[V], s_full[3], p_full[3],
  // pv_done[3], o_full, o_free, mma_done[2], l_full[2], l_empty[2]
  static constexpr int NUM_BARS = 2 * Q_STAGES + 2 * K_STAGES + 2 * V_STAGES + 3 * NSB + 4 + 4;
  static constexpr int SLOT_OFF = BAR_OFF + NUM_BARS * 8;
  static constexpr int USED = SLOT_OFF + 16;
  // The dynamic shared memory window starts 1 KB-aligned (checked at run time); never below
  // ~114 KB, so that one CTA (and its 512 TMEM columns) holds an SM.
  static constexpr int ALLOC = USED > 116 * 1024 ? USED : 116 * 1024;
  static_assert(ALLOC <= 232448, "shared memory budget");
  static_assert(O_COL + D <= TMEM_COLS, "TMEM budget");
  static_assert(BN == 64 || BN == 128, "the softmax takes 8 or 16 groups of 8 columns");
  static_assert((BN / 16) * CHUNKS <= 32, "one paged K/V copy per producer lane");
};

using pf::WorkTile;

// The walk over this kernel's work tiles (one query head each), in the order of Base (pf::TileWalk
// or pf::BlockedTileWalk); errors go to this kernel's status.
template <class Base>
struct WalkOf : Base {
  __device__ __forceinline__ bool next(const PrefillParams& p, WorkTile& t) {
    return Base::next(p, t, &g_prefill_status);
  }
};

template <int D, class TileWalk>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    prefill_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                       const __grid_constant__ CUtensorMap tm_vrow, const PrefillParams p) {
  using L = Layout<D>;
  extern __shared__ __align__(1024) uint8_t smem[];
  if ((smem_u32(smem) & 1023u) != 0) {  // 128B-swizzled tiles need 1 KB alignment
    if (threadIdx.x == 0) set_error(&g_prefill_status, kDevMisaligned);
    return;
  }
  uint8_t* sQ = smem + L::Q_OFF;
  uint8_t* sK = smem + L::K_OFF;
  uint8_t* sV = smem + L::V_OFF;
  uint8_t* sO = smem + L::OST_OFF;
  float* xl = reinterpret_cast<float*>(smem + L::XL_OFF);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::BAR_OFF);
  constexpr int BN = L::BN, Q_STAGES = L::Q_STAGES, K_STAGES = L::K_STAGES, V_STAGES = L::V_STAGES;
  constexpr uint32_t O_COL = L::O_COL;
  uint64_t* q_full = bars;                 // [Q_STAGES]
  uint64_t* q_empty = q_full + Q_STAGES;   // [Q_STAGES]: every S product of the buffer's tile is done
  uint64_t* k_full = q_empty + Q_STAGES;
  uint64_t* k_empty = k_full + K_STAGES;
  uint64_t* v_full = k_empty + K_STAGES;
  uint64_t* v_empty = v_full + V_STAGES;
  uint64_t* s_full = v_empty + V_STAGES;
  uint64_t* p_full = s_full + NSB;
  uint64_t* pv_done = p_full + NSB;   // [3]: P_j V_j done, per S buffer
  uint64_t* o_full = pv_done + NSB;
  uint64_t* o_free = o_full + 1;      // the epilogue has read O out of TMEM
  uint64_t* mma_done = o_free + 1;    // [2]: each issuer's last MMA done
  uint64_t* l_full = mma_done + 2;    // [2]: a tile's row sums and maxima are in xl
  uint64_t* l_empty = l_full + 2;     // [2]: the epilogue has read them
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::SLOT_OFF);

  // The warp index and the TMEM base are made visibly warp-uniform (a broadcast from lane 0): the
  // compiler then keeps them, and everything the MMA operands are built from, in uniform
  // registers, and tcgen05.mma issues at the tensor core's rate instead of half of it.
  const int warp = __shfl_sync(0xffffffffu, static_cast<int>(threadIdx.x >> 5), 0);
  const int lane = threadIdx.x & 31;
  const int G = p.Hq / p.Hkv;
  // a wait taken by a whole warp, which passes only if every lane's does
  auto wait = [&](uint64_t* bar, uint32_t parity) { return __all_sync(0xffffffffu, mbar_wait(bar, parity)); };
  auto tile_nkv = [&](const WorkTile& t) { return pf::tile_nkv<BN>(p, t); };
  // Paged K/V: the physical page of each of the BN / 16 pages of key tile j (-1 past the sequence).
  // The producers read them before waiting for a free stage, so the reads overlap the wait.
  auto fetch_pages = [&](const WorkTile& t, int j, int (&pids)[BN / 16]) {
    const int32_t* bt = p.block_table + static_cast<size_t>(t.b) * p.max_blocks;
#pragma unroll
    for (int pp = 0; pp < BN / 16; ++pp) {
      const int page = j * (BN / 16) + pp;
      pids[pp] = page * 16 < t.kv_len ? bt[page] : -1;
    }
  };
  // K or V tile j of work tile t into one ring stage (one expect_tx for all of its boxes)
  auto load_kv = [&](uint8_t* dst, const CUtensorMap* map, bool is_v, uint64_t* bar, int g, const WorkTile& t,
                     int j, const int (&pids)[BN / 16]) {
    mbar_arrive_expect_tx(bar, L::KV_BYTES);
    if (p.kv_lens == nullptr) {
      for (int c = 0; c < L::CHUNKS; ++c)
        tma_load_3d(dst + c * L::KV_PANEL, map, bar, g * D + c * 64, t.base + j * BN, t.z);
      return;
    }
    // paged: BN / 16 pages of 16 rows.  Pages past the sequence are read from rows past the cache,
    // which the copy fills with zeros.
    const int oob = p.num_blocks * 16;
#pragma unroll
    for (int pp = 0; pp < BN / 16; ++pp) {
      const int valid = t.kv_len - (j * (BN / 16) + pp) * 16;  // rows of this page that hold keys
      int row0 = oob;
      if (valid > 0) {
        int pid = pids[pp];
        if (pid < 0 || pid >= p.num_blocks) {
          set_error(&g_prefill_status, kDevBadPage);
          pid = 0;
        }
        row0 = pid * 16;
      }
      uint8_t* pd = dst + pp * 16 * PANEL_ROW;
      if (is_v && valid > 0 && valid < 16) {
        // the rows past the last key must be finite (P is 0 there, but 0 * NaN is not): row by row,
        // the tail from past the cache
#pragma unroll 1
        for (int r = 0; r < 16; ++r)
#pragma unroll 1
          for (int c = 0; c < L::CHUNKS; ++c)
            tma_load_3d(pd + c * L::KV_PANEL + r * PANEL_ROW, &tm_vrow, bar, c * 64, g, r < valid ? row0 + r : oob);
      } else {
        for (int c = 0; c < L::CHUNKS; ++c) tma_load_3d(pd + c * L::KV_PANEL, map, bar, c * 64, g, row0);
      }
    }
  };
  // loads of the first tile that are issued before the CTA barrier: Q, and as many K and V
  // tiles as the rings hold
  auto first_loads = [&](int nst) {
    TileWalk w;
    WorkTile t;
    if (!w.next(p, t)) return 0;
    const int n = tile_nkv(t);
    return n < nst ? n : nst;
  };

  if (warp == PRODUCER_WARP && lane == 0) {
    for (int s = 0; s < Q_STAGES; ++s) {
      mbar_init(&q_full[s], 1);
      mbar_init(&q_empty[s], 1);
    }
    for (int s = 0; s < K_STAGES; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&k_empty[s], 1);
    }
    for (int s = 0; s < V_STAGES; ++s) {
      mbar_init(&v_full[s], 1);
      mbar_init(&v_empty[s], 1);
    }
    for (int s = 0; s < NSB; ++s) {
      mbar_init(&s_full[s], 1);
      mbar_init(&p_full[s], 8);   // one arrival per softmax warp
      mbar_init(&pv_done[s], 1);
    }
    mbar_init(o_full, 1);
    mbar_init(o_free, 4);          // one arrival per epilogue warp
    mbar_init(&mma_done[0], 1);
    mbar_init(&mma_done[1], 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(&l_full[s], 8);    // one arrival per softmax warp
      mbar_init(&l_empty[s], 4);   // one arrival per epilogue warp
    }
    fence_mbar_init();
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
    tma_prefetch_desc(&tm_o);
    TileWalk w;
    WorkTile t;
    if (w.next(p, t)) {
      const int g = t.hq / G;
      mbar_arrive_expect_tx(q_full, L::Q_BYTES);
      for (int c = 0; c < L::CHUNKS; ++c)
        tma_load_3d(sQ + c * L::Q_PANEL, &tm_q, q_full, t.hq * D + c * 64, t.base + t.qt * BM, t.z);
      const int nk = first_loads(K_STAGES), nv = first_loads(V_STAGES);
      int pids[BN / 16] = {};
      for (int j = 0; j < nk; ++j) {
        if (p.kv_lens != nullptr) fetch_pages(t, j, pids);
        load_kv(sK + j * L::KV_BYTES, &tm_k, false, &k_full[j], g, t, j, pids);
      }
      for (int j = 0; j < nv; ++j) {
        if (p.kv_lens != nullptr) fetch_pages(t, j, pids);
        load_kv(sV + j * L::KV_BYTES, &tm_v, true, &v_full[j], g, t, j, pids);
      }
    }
  }
  if (warp == MMA_WARP) {
    tmem_alloc(tmem_slot, TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = __shfl_sync(0xffffffffu, *tmem_slot, 0);

  // Each warpgroup sets its register budget at the top of its branch, so that the compiler
  // allocates the role's code within it: the softmax warps take 168 registers per thread, the
  // loading and MMA warps 64, the epilogue 112 (launched with 128 x 512 = 65536).
  if (warp >= PRODUCER_WARP && warp < EPI_WARP0) {
    regs_dec<REG_OTHER>();
    if (warp == PRODUCER_WARP || warp == V_WARP) {
      // ------------------------------------------------------------ TMA producers
      // Warp 8 loads Q and the K tiles, warp 11 the V tiles; each waits only on its own ring.
      // Counters run across work tiles, so the rings never drain between tiles.  The whole warp runs
      // the loop: with paged K/V, lane l reads the physical page of page l of the tile and the lanes
      // issue one 16-row copy each, so the many small copies of a tile leave in one instruction.
      {
        const bool is_k = warp == PRODUCER_WARP;
        const int nst = is_k ? K_STAGES : V_STAGES;
        uint64_t* full = is_k ? k_full : v_full;
        uint64_t* empty = is_k ? k_empty : v_empty;
        uint8_t* ring = is_k ? sK : sV;
        const CUtensorMap* map = is_k ? &tm_k : &tm_v;
        const int npre = first_loads(nst);
        constexpr int PAGES = BN / 16;
        bool ok = true;
        int issued = npre, nq = 0;
        TileWalk walk;
        WorkTile t;
        for (int k = 0; ok && walk.next(p, t); ++k) {
          const int g = t.hq / G;
          if (is_k) {
            // Q of tile k goes to buffer k % Q_STAGES once every S = Q K^T product of tile
            // k - Q_STAGES is done: with two buffers it loads while the previous tile still runs
            if (k > 0) {
              const int qs = k % Q_STAGES;
              if (k >= Q_STAGES) {
                ok = __all_sync(0xffffffffu, mbar_wait(&q_empty[qs], ((k / Q_STAGES) - 1) & 1));
                if (!ok) break;
              }
              if (lane == 0) {
                mbar_arrive_expect_tx(&q_full[qs], L::Q_BYTES);
                for (int c = 0; c < L::CHUNKS; ++c)
                  tma_load_3d(sQ + qs * L::Q_BYTES + c * L::Q_PANEL, &tm_q, &q_full[qs], t.hq * D + c * 64,
                              t.base + t.qt * BM, t.z);
              }
            }
            nq = k + 1;
          }
          const int nkv = tile_nkv(t);
          for (int j = (k == 0 ? npre : 0); j < nkv; ++j) {
            const int st = issued % nst;
            uint8_t* dst = ring + st * L::KV_BYTES;
            // paged: lane l < PAGES reads the physical page of page l of this tile before the wait
            int my_pid = -1;
            if (p.kv_lens != nullptr && lane < PAGES) {
              const int page = j * PAGES + lane;
              if (page * 16 < t.kv_len) my_pid = p.block_table[static_cast<size_t>(t.b) * p.max_blocks + page];
            }
            ok = __all_sync(0xffffffffu, mbar_wait(&empty[st], ((issued / nst) & 1) ^ 1));
            if (!ok) break;
            if (lane == 0) mbar_arrive_expect_tx(&full[st], L::KV_BYTES);
            __syncwarp();
            if (p.kv_lens == nullptr) {
              if (lane < L::CHUNKS)
                tma_load_3d(dst + lane * L::KV_PANEL, map, &full[st], g * D + lane * 64, t.base + j * BN, t.z);
            } else {
              // lane l: page l / CHUNKS, 64-column chunk l % CHUNKS.  Pages past the sequence are read
              // from rows past the cache, which the copy fills with zeros.
              const int pp = lane / L::CHUNKS, c = lane % L::CHUNKS;
              int pid = __shfl_sync(0xffffffffu, my_pid, pp < PAGES ? pp : 0);
              if (pp < PAGES) {
                const int oob = p.num_blocks * 16;
                const int valid = t.kv_len - (j * PAGES + pp) * 16;  // rows of this page that hold keys
                int row0 = oob;
                if (valid > 0) {
                  if (pid < 0 || pid >= p.num_blocks) {
                    set_error(&g_prefill_status, kDevBadPage);
                    pid = 0;
                  }
                  row0 = pid * 16;
                }
                uint8_t* pd = dst + c * L::KV_PANEL + pp * 16 * PANEL_ROW;
                if (!is_k && valid > 0 && valid < 16) {
                  // the V rows past the last key must be finite (P is 0 there, but 0 * NaN is not):
                  // row by row, the tail from past the cache
                  for (int r = 0; r < 16; ++r)
                    tma_load_3d(pd + r * PANEL_ROW, &tm_vrow, &full[st], c * 64, g, r < valid ? row0 + r : oob);
                } else {
                  tma_load_3d(pd, map, &full[st], c * 64, g, row0);
                }
              }
            }
            ++issued;
          }
        }
        if (lane == 0) {
          if (!ok) set_error(&g_prefill_status, kDevWaitTimeout);
          // Drain: every copy started here must have landed before the CTA exits.  The newest
          // copy of each stage is the one whose phase is current.
          for (int i = (issued > nst ? issued - nst : 0); i < issued; ++i) mbar_wait(&full[i % nst], (i / nst) & 1);
          for (int i = (nq > Q_STAGES ? nq - Q_STAGES : 0); i < nq; ++i)
            mbar_wait(&q_full[i % Q_STAGES], (i / Q_STAGES) & 1);
        }
      }
    } else if (warp == MMA_WARP) {
      // ------------------------------------------------------------ S = Q K^T issue
      // S of global step gs goes to TMEM buffer gs % 3, which held P of step gs - 3: wait until
      // that P.V is done.  The whole warp runs the loop; one elected lane issues.
      {
        constexpr uint32_t IDESC_S = idesc_bf16_f32(BM, BN, 0);   // Q (K-major) x K (K-major)
        bool ok = true;
        int gs = 0;
        TileWalk walk;
        WorkTile t;
        for (int k = 0; ok && walk.next(p, t); ++k) {
          const int qs = k % Q_STAGES;
          if (!wait(&q_full[qs], (k / Q_STAGES) & 1)) { ok = false; break; }
          const uint32_t qbase = smem_u32(sQ + qs * L::Q_BYTES);
          const int nkv = tile_nkv(t);
          for (int j = 0; j < nkv; ++j, ++gs) {
            const int sb = gs % NSB;
            const int st = gs % K_STAGES;
            if ((gs >= NSB && !wait(&pv_done[sb], ((gs - NSB) / NSB) & 1)) ||
                !wait(&k_full[st], (gs / K_STAGES) & 1)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t kbase = smem_u32(sK + st * L::KV_BYTES);
            const uint32_t s_tmem = tmem + sb * BN;
  #pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
              // 16 columns of d: panel kk / 4, 32 bytes into its 128-byte rows
              const uint32_t qoff = (kk >> 2) * L::Q_PANEL + (kk & 3) * 32;
              const uint32_t koff = (kk >> 2) * L::KV_PANEL + (kk & 3) * 32;
              umma_ss_warp(s_tmem, smem_desc_sw128(qbase + qoff, 16, 1024), smem_desc_sw128(kbase + koff, 16, 1024),
                           IDESC_S, kk > 0 ? 1u : 0u);
            }
            umma_commit_warp(&s_full[sb]);
            umma_commit_warp(&k_empty[st]);
          }
          umma_commit_warp(&q_empty[qs]);  // the buffer may take another Q once these products are done
        }
        if (!ok) set_error(&g_prefill_status, kDevWaitTimeout);
        umma_commit_warp(&mma_done[0]);
        if (!wait(&mma_done[0], 0)) set_error(&g_prefill_status, kDevWaitTimeout);
      }
    } else if (warp == PV_WARP) {
      // ------------------------------------------------------------ O += P V issue
      // The whole warp runs the loop; one elected lane issues.
      {
        constexpr uint32_t IDESC_O = idesc_bf16_f32(BM, D, 1);    // P (TMEM) x V (MN-major)
        const uint32_t o_tmem = tmem + O_COL;
        bool ok = true;
        int gs = 0;
        TileWalk walk;
        WorkTile t;
        for (int k = 0; ok && walk.next(p, t); ++k) {
          // the first product of a tile overwrites O: the previous tile's epilogue must have read it
          if (k > 0 && !wait(o_free, (k - 1) & 1)) { ok = false; break; }
          const int nkv = tile_nkv(t);
          for (int j = 0; j < nkv; ++j, ++gs) {
            const int sb = gs % NSB;
            const int st = gs % V_STAGES;
            if (!wait(&p_full[sb], (gs / NSB) & 1) || !wait(&v_full[st], (gs / V_STAGES) & 1)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t vbase = smem_u32(sV + st * L::KV_BYTES);
            const uint32_t p_tmem = tmem + sb * BN;
  #pragma unroll
            for (int kk = 0; kk < BN / 16; ++kk) {
              // 16 keys = two 8-row swizzle atoms; d panels are BN*128 bytes apart
              umma_ts_warp(o_tmem, p_tmem + kk * 8, smem_desc_sw128(vbase + kk * 16 * 128, BN * 128, 1024), IDESC_O,
                           (j > 0 || kk > 0) ? 1u : 0u);
            }
            umma_commit_warp(&pv_done[sb]);
            umma_commit_warp(&v_empty[st]);
            if (j == nkv - 1) umma_commit_warp(o_full);
          }
        }
        if (!ok) set_error(&g_prefill_status, kDevWaitTimeout);
        umma_commit_warp(&mma_done[1]);
        if (!wait(&mma_done[1], 0)) set_error(&g_prefill_status, kDevWaitTimeout);
      }
    }
  } else if (warp < PRODUCER_WARP) {
    regs_inc<REG_SOFTMAX>();
    // ------------------------------------------------------------ softmax (prefill_tile.cuh)
    // Warp w takes the 16 rows r0 .. r0 + 15 of each tile, four threads per row.
    const int r0 = (warp & 3) * 32 + (warp >> 2) * 16;
    const int ra = r0 + (lane >> 2);  // row a; row b is ra + 8
    const int cq = 2 * (lane & 3);    // this thread's first column in each group of 8
    const uint32_t lane_base = static_cast<uint32_t>(r0) << 16;
    const float c2 = p.scale_log2;
    const uint64_t c2x2 = f2_pack(c2, c2);
    bool ok = true;
    int gs = 0;
    TileWalk walk;
    WorkTile t;
    pf::SoftmaxRows rows;
    for (int k = 0; walk.next(p, t); ++k) {
      const int qa = t.q_off + t.qt * BM + ra;  // positions of rows a and b among the keys
      const int nkv = tile_nkv(t);
      rows.reset();
      for (int j = 0; j < nkv; ++j, ++gs) {
        const int sb = gs % NSB;
        if (ok) ok = __all_sync(0xffffffffu, mbar_wait(&s_full[sb], (gs / NSB) & 1));
        tc_fence_after();
        pf::softmax_step<BN, D, NSB>(p, t, j, gs, tmem + lane_base + sb * BN, tmem + lane_base + O_COL, qa, qa + 8,
                                     cq, c2, c2x2, pv_done, rows, ok);
        if (lane == 0) mbar_arrive(&p_full[sb]);  // one arrival per warp: 256 would queue on the barrier
      }
      pf::softmax_tile_end(k, ra, lane, rows, l_empty, l_full, xl, ok);
    }
    if (!ok) set_error(&g_prefill_status, kDevWaitTimeout);
  } else {
    regs_dec<REG_EPI>();
    // ------------------------------------------------------------ epilogue (prefill_tile.cuh)
    const int row = (warp & 3) * 32 + lane;
    const int et = threadIdx.x - EPI_WARP0 * 32;
    const uint32_t o_row = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16) + O_COL;
    auto release_o = [&]() {
      if (lane == 0) mbar_arrive(o_free);
    };
    bool ok = true;
    TileWalk walk;
    WorkTile t;
    for (int k = 0; walk.next(p, t); ++k)
      pf::epilogue_tile<D, L::OGRP>(p, t, k, row, et, lane, o_row, xl, l_full, l_empty, o_full, sO, &tm_o, release_o,
                                   ok);
    if (!ok) set_error(&g_prefill_status, kDevWaitTimeout);
    if (et == 0) tma_store_wait0();
  }

  __syncwarp();  // single-lane roles rejoin their warps before the CTA barrier
  tc_fence_before();
  __syncthreads();
  if (warp == MMA_WARP) {
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

// one persistent CTA per SM of the current device (sms), or one per work tile if fewer
template <int D, class Walk>
cudaError_t launch(const PrefillMaps& m, const PrefillParams& p, int sms, cudaStream_t stream) {
  auto kern = prefill_fwd_kernel<D, Walk>;
  const int smem = Layout<D>::ALLOC;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const long long tiles = static_cast<long long>(p.num_qblocks) * p.B * p.Hq;
  const int grid = static_cast<int>(tiles < sms ? tiles : sms);
  kern<<<grid, NUM_THREADS, smem, stream>>>(m.q, m.k, m.v, m.o, m.v_row, p);
  return cudaGetLastError();
}

}  // namespace

int prefill_rows_per_cta() { return BM; }
int prefill_tile_rows() { return BM; }
int prefill_kv_tile_rows(int d) { return d <= 128 ? Layout<128>::BN : Layout<256>::BN; }

cudaError_t prefill_launch(int d, const PrefillMaps& maps, const PrefillParams& p, bool blocked, int sms,
                           cudaStream_t stream) {
  using Plain = WalkOf<pf::TileWalk>;
  using Blocked = WalkOf<pf::BlockedTileWalk>;
  if (d == 64) return blocked ? launch<64, Blocked>(maps, p, sms, stream) : launch<64, Plain>(maps, p, sms, stream);
  if (d == 128) return blocked ? launch<128, Blocked>(maps, p, sms, stream) : launch<128, Plain>(maps, p, sms, stream);
  if (d == 256) return blocked ? launch<256, Blocked>(maps, p, sms, stream) : launch<256, Plain>(maps, p, sms, stream);
  return cudaErrorInvalidValue;
}

cudaError_t prefill_status(uint32_t* out, bool clear) {
  uint32_t pair = 0;
  cudaError_t e = cudaMemcpyFromSymbol(out, g_prefill_status, sizeof(uint32_t));
  if (e == cudaSuccess && clear) {
    const uint32_t zero = 0;
    e = cudaMemcpyToSymbol(g_prefill_status, &zero, sizeof(uint32_t));
  }
  if (e == cudaSuccess) e = prefill_cta2_status(&pair, clear);
  if (e == cudaSuccess && *out == 0) *out = pair;
  return e;
}

}  // namespace attn
