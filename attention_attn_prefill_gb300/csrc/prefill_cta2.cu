// Causal (or full) prefill attention forward on sm_103a, head dim 128, as CTA pairs: the two CTAs of a
// cluster take two query heads of one KV head (the same query tile of each), and every tcgen05.mma
// is a 256-row product over both SMs (cta_group::2).
//
// What it computes: "Why your local LLM feels dumber than it is" (Part 3.14), section "What attention
// is trying to calculate" -- O = softmax(scale*QK^T) V per query row over the keys it may see (causal:
// keys j <= i), plus the natural-log LSE of each row -- with the tiled online softmax of "Streaming
// process -- How the SM works inside a transformer", Steps 3-8.
//
// How it differs from the single-head kernel (prefill.cu), whose softmax, rescaling and epilogue it
// shares:
//   * CTA r of a pair holds the 128 query rows of head 2p + r (Q, double-buffered), the K tile's keys
//     64r .. 64r + 63 and the V tile's head-dim columns 64r .. 64r + 63.  The even CTA issues
//     S = Q K^T as one M = 256, N = 128 product (A split by rows, B by keys) and O += P V as one
//     M = 256, N = 128 product (P from each CTA's TMEM, V split by columns); each CTA gets its own
//     128 rows of S and O in its TMEM.  So each CTA streams half of every K and V tile: its rings
//     hold four 16 KB stages each, twice the lookahead of the single-head kernel at the same shared
//     memory, and one issue stream feeds two SMs;
//   * both CTAs' copies complete on the even CTA's full barriers.  The even CTA arms each of them for
//     both halves before the first copy and again right after its MMA issuer has consumed a phase,
//     before the commit that frees the stage, so no copy can land on a phase that is not armed yet.
//     The even CTA's commits reach both CTAs' barriers (multicast); the odd CTA's softmax and
//     epilogue warps arrive on the even CTA's p_full and o_free (relaxed arrivals, after their TMEM
//     stores or loads have completed and a tcgen05 fence);
//   * packed sequences (cu_seqlens) and paged K/V (block table) take the instances with PACKED set:
//     each CTA copies its half of a K tile as 4 pages x 2 panels and its V panel as 8 pages.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <type_traits>

#include "prefill.h"
#include "prefill_tile.cuh"
#include "prefill_walk.cuh"
#include "sm103.cuh"

namespace attn {

__device__ uint32_t g_prefill_cta2_status;

namespace {

using pf::BM;
using pf::PANEL_ROW;
using pf::WorkTile;

constexpr int D = 128;           // head dim
constexpr int BN = 128;          // keys per step
constexpr int CHUNKS = D / 64;   // 64-column panels per row
constexpr int NSB = 3;           // S buffers in TMEM
constexpr int NUM_THREADS = 512; // 8 softmax warps, 2 TMA warps, 2 MMA warps, 4 epilogue warps
constexpr int PRODUCER_WARP = 8; // loads Q and streams K
constexpr int MMA_WARP = 9;      // issues S = Q K^T (even CTA), owns the TMEM allocation
constexpr int PV_WARP = 10;      // issues O += P V (even CTA)
constexpr int V_WARP = 11;       // streams V
constexpr int EPI_WARP0 = 12;    // warps 12..15: epilogue, one thread per row
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t REG_SOFTMAX = 168, REG_OTHER = 72, REG_EPI = 104;
static_assert(8 * 32 * REG_SOFTMAX + 4 * 32 * REG_OTHER + 4 * 32 * REG_EPI == 128 * NUM_THREADS, "register split");

constexpr int Q_STAGES = 2, K_STAGES = 4, V_STAGES = 4;
constexpr int Q_PANEL = BM * PANEL_ROW;        // one panel of a Q (or output) tile: 16 KB
constexpr int Q_BYTES = CHUNKS * Q_PANEL;      // this CTA's 128 query rows
constexpr int KH_ROWS = BN / 2;                // keys of a K tile held by one CTA
constexpr int KH_PANEL = KH_ROWS * PANEL_ROW;  // 8 KB
constexpr int K_BYTES = CHUNKS * KH_PANEL;     // this CTA's half of a K tile: 16 KB
constexpr int V_BYTES = BN * PANEL_ROW;        // all BN keys, this CTA's 64 head-dim columns: 16 KB
constexpr int OGRP = D;                        // O columns the epilogue holds at once
constexpr uint32_t O_COL = NSB * BN;           // O accumulator columns start here
constexpr int Q_OFF = 0;
constexpr int K_OFF = Q_OFF + Q_STAGES * Q_BYTES;
constexpr int V_OFF = K_OFF + K_STAGES * K_BYTES;
constexpr int OST_OFF = V_OFF + V_STAGES * V_BYTES;  // output staging: one 64-column panel
constexpr int XL_OFF = OST_OFF + Q_PANEL;            // row sums and maxima for the epilogue [2 tiles][2][128]
constexpr int BAR_OFF = XL_OFF + 2 * 2 * 128 * 4;
// q_full[Q], q_empty[Q], k_full[K], k_empty[K], v_full[V], v_empty[V], s_full[3], p_full[3], pv_done[3],
// o_full, o_free, mma_done[2], l_full[2], l_empty[2]
constexpr int NUM_BARS = 2 * Q_STAGES + 2 * K_STAGES + 2 * V_STAGES + 3 * NSB + 4 + 4;
constexpr int SLOT_OFF = BAR_OFF + NUM_BARS * 8;
constexpr int SMEM_BYTES = SLOT_OFF + 16;
static_assert(SMEM_BYTES <= 232448, "shared memory budget");
static_assert(O_COL + D <= TMEM_COLS, "TMEM budget");
constexpr uint16_t BOTH = 3, EVEN = 1;  // CTA masks for multicast commits

// Work units: (query tile, sequence, head pair), longest first, dealt out in a zigzag over the
// clusters; CTA r of the pair takes head 2 * pair + r.  The host sets the divisors to B * Hq / 2
// (units per query-tile level) and Hq / 2.
struct PairWalk {
  int v = 0;
  __device__ __forceinline__ bool next(const PrefillParams& p, WorkTile& t, int rank) {
    const int G = static_cast<int>(num_clusters_x()), c = static_cast<int>(cluster_id_x());
    const int pairs = p.Hq >> 1;
    const int per_qt = p.B * pairs;
    const int total = per_qt * p.num_qblocks;
    const int idx = v * G + ((v & 1) ? (G - 1 - c) : c);
    ++v;
    if (idx >= total) return false;
    const int level = static_cast<int>(p.div_level.div(static_cast<uint32_t>(idx)));
    t.qt = p.num_qblocks - 1 - level;
    const int rem = idx - level * per_qt;
    t.b = static_cast<int>(p.div_heads.div(static_cast<uint32_t>(rem)));
    t.hq = 2 * (rem - t.b * pairs) + rank;
    t.base = 0;
    t.z = t.b;
    t.len = t.kv_len = p.S;
    t.q_off = 0;
    return true;
  }
};

// PairWalk's list in blocks of p.seq_block consecutive (sequence, head pair) units, whole KV heads,
// band by band of query-tile levels (equal-length batches whose keys and values exceed three
// quarters of L2; see PrefillParams::seq_block).
struct LaneBlockedPairWalk {
  int v = 0;
  __device__ __forceinline__ bool next(const PrefillParams& p, WorkTile& t, int rank) {
    const int G = static_cast<int>(num_clusters_x()), c = static_cast<int>(cluster_id_x());
    const int pairs = p.Hq >> 1;
    const int units = p.B * pairs;
    while (true) {
      const int idx = v * G + ((v & 1) ? (G - 1 - c) : c);
      ++v;
      int level, u;
      const int k = pf::lane_band_unit(p, idx, units, level, u);
      if (k == 0) return false;
      if (k == 1) continue;
      t.qt = p.num_qblocks - 1 - level;
      t.b = static_cast<int>(p.div_heads.div(static_cast<uint32_t>(u)));
      t.hq = 2 * (u - t.b * pairs) + rank;
      t.base = 0;
      t.z = t.b;
      t.len = t.kv_len = p.S;
      t.q_off = 0;
      return true;
    }
  }
};

// The same list for packed sequences (cu_seqlens, and with paged K/V kv_lens): units past a sequence's
// end are skipped, alike in both CTAs of a pair, and a sequence with bad bounds is recorded and skipped.
// BLOCKED, chunked prefill over a paged cache larger than half of L2: the list is cut into blocks of
// p.seq_block sequences, each block walked longest unit first before the next, so that a block's
// cached keys and values stay in L2 while all its query tiles stream them.  Every block counts
// p.seq_block sequences; the last one's units past the batch are skipped.  BLOCKED, packed prompts
// (no kv_lens) larger than three quarters of L2: the banded lane-blocked order of
// LaneBlockedPairWalk.  It is a separate instance: where the batch fits L2 the extra index
// arithmetic measured 2-3% slower.
template <bool BLOCKED>
struct PackedPairWalk {
  int v = 0;
  __device__ __forceinline__ bool next(const PrefillParams& p, WorkTile& t, int rank) {
    const int G = static_cast<int>(num_clusters_x()), c = static_cast<int>(cluster_id_x());
    const int pairs = p.Hq >> 1;
    if constexpr (BLOCKED) {
      if (p.kv_lens == nullptr) {  // packed prompts: lanes and bands
        const int units = p.B * pairs;
        while (true) {
          const int idx = v * G + ((v & 1) ? (G - 1 - c) : c);
          ++v;
          int level, u;
          const int k = pf::lane_band_unit(p, idx, units, level, u);
          if (k == 0) return false;
          if (k == 1) continue;
          t.qt = p.num_qblocks - 1 - level;
          t.b = static_cast<int>(p.div_heads.div(static_cast<uint32_t>(u)));
          t.hq = 2 * (u - t.b * pairs) + rank;
          const int s0 = p.cu_seqlens[t.b], s1 = p.cu_seqlens[t.b + 1];
          if (s0 < 0 || s1 < s0 || s1 > p.S || s1 - s0 > p.num_qblocks * BM) {
            if (rank == 0) set_error(&g_prefill_cta2_status, kDevBadSeqlens);
            continue;  // the sequence is skipped
          }
          t.base = s0;
          t.z = 0;
          t.len = t.kv_len = s1 - s0;
          t.q_off = 0;
          if (t.qt * BM < t.len) return true;
        }
      }
    }
    const int seqs = BLOCKED ? (p.B + p.seq_block - 1) / p.seq_block * p.seq_block : p.B;
    const int total = seqs * pairs * p.num_qblocks;
    while (true) {
      const int idx = v * G + ((v & 1) ? (G - 1 - c) : c);
      ++v;
      if (idx >= total) return false;
      int r = idx, b0 = 0, per_qt = p.B * pairs;
      if constexpr (BLOCKED) {
        const int blk = static_cast<int>(p.div_block.div(static_cast<uint32_t>(idx)));
        r = idx - blk * p.seq_block * pairs * p.num_qblocks;
        b0 = blk * p.seq_block;
        per_qt = p.seq_block * pairs;
      }
      const int level = static_cast<int>((BLOCKED ? p.div_block_level : p.div_level).div(static_cast<uint32_t>(r)));
      t.qt = p.num_qblocks - 1 - level;
      const int rem = r - level * per_qt;
      const int bi = static_cast<int>(p.div_heads.div(static_cast<uint32_t>(rem)));
      t.b = b0 + bi;
      t.hq = 2 * (rem - bi * pairs) + rank;
      if (BLOCKED && t.b >= p.B) continue;  // past the batch, in the last block
      const int s0 = p.cu_seqlens[t.b], s1 = p.cu_seqlens[t.b + 1];
      const int kvl = p.kv_lens != nullptr ? p.kv_lens[t.b] : s1 - s0;
      if (s0 < 0 || s1 < s0 || s1 > p.S || s1 - s0 > p.num_qblocks * BM || kvl < s1 - s0 ||
          (p.kv_lens != nullptr && kvl > p.max_blocks * 16)) {
        if (rank == 0) set_error(&g_prefill_cta2_status, kDevBadSeqlens);
        continue;  // the sequence is skipped
      }
      t.base = s0;
      t.z = 0;
      t.len = s1 - s0;
      t.kv_len = kvl;
      t.q_off = kvl - t.len;
      if (t.qt * BM < t.len) return true;
    }
  }
};

// PACKED: packed sequences (PackedPairWalk), with contiguous or paged K/V; tm_vrow (one-row V boxes,
// paged K/V only) fetches the last, partial page of a sequence row by row.  BLOCKED: the packed walk in
// blocks of sequences; without PACKED, the equal-length walk in blocks of units (LaneBlockedPairWalk).
template <bool PACKED, bool BLOCKED>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(NUM_THREADS, 1)
    prefill_cta2_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                        const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                        const __grid_constant__ CUtensorMap tm_vrow, const PrefillParams p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  if ((smem_u32(smem) & 1023u) != 0) {  // both CTAs see the same launch: both return
    if (threadIdx.x == 0) set_error(&g_prefill_cta2_status, kDevMisaligned);
    return;
  }
  uint8_t* sQ = smem + Q_OFF;
  uint8_t* sK = smem + K_OFF;
  uint8_t* sV = smem + V_OFF;
  uint8_t* sO = smem + OST_OFF;
  float* xl = reinterpret_cast<float*>(smem + XL_OFF);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + BAR_OFF);
  uint64_t* q_full = bars;                 // [Q_STAGES] (even CTA): both CTAs' Q rows are in
  uint64_t* q_empty = q_full + Q_STAGES;   // [Q_STAGES]: every S product of the buffer's tile is done
  uint64_t* k_full = q_empty + Q_STAGES;   // (even CTA) both halves of the K tile are in
  uint64_t* k_empty = k_full + K_STAGES;
  uint64_t* v_full = k_empty + K_STAGES;   // (even CTA) both halves of the V tile are in
  uint64_t* v_empty = v_full + V_STAGES;
  uint64_t* s_full = v_empty + V_STAGES;
  uint64_t* p_full = s_full + NSB;         // (even CTA) both CTAs' P are in TMEM
  uint64_t* pv_done = p_full + NSB;        // [3]: P_j V_j done, per S buffer
  uint64_t* o_full = pv_done + NSB;
  uint64_t* o_free = o_full + 1;           // (even CTA) both epilogues have read O out of TMEM
  uint64_t* mma_done = o_free + 1;         // [2]: each issuer's last MMA done (even CTA)
  uint64_t* l_full = mma_done + 2;         // [2]: a tile's row sums and maxima are in xl
  uint64_t* l_empty = l_full + 2;          // [2]: the epilogue has read them
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + SLOT_OFF);

  // warp index and TMEM base made visibly warp-uniform, so the MMA operands stay in uniform registers
  const int warp = __shfl_sync(0xffffffffu, static_cast<int>(threadIdx.x >> 5), 0);
  const int lane = threadIdx.x & 31;
  const int rank = static_cast<int>(cluster_ctarank());
  const int G = p.Hq / p.Hkv;
  auto wait = [&](uint64_t* bar, uint32_t parity) { return __all_sync(0xffffffffu, mbar_wait(bar, parity)); };
  auto tile_nkv = [&](const WorkTile& t) { return pf::tile_nkv<BN>(p, t); };
  struct Walk
      : std::conditional_t<PACKED, PackedPairWalk<BLOCKED>, std::conditional_t<BLOCKED, LaneBlockedPairWalk, PairWalk>> {
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
      mbar_init(&p_full[s], 16);  // one arrival per softmax warp of both CTAs
      mbar_init(&pv_done[s], 1);
    }
    mbar_init(o_full, 1);
    mbar_init(o_free, 8);          // one arrival per epilogue warp of both CTAs
    mbar_init(&mma_done[0], 1);
    mbar_init(&mma_done[1], 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(&l_full[s], 8);    // one arrival per softmax warp
      mbar_init(&l_empty[s], 4);   // one arrival per epilogue warp
    }
    if (rank == 0) {
      // arm the first phase of every full barrier for both CTAs' halves
      for (int s = 0; s < Q_STAGES; ++s) mbar_arrive_expect_tx(&q_full[s], 2 * Q_BYTES);
      for (int s = 0; s < K_STAGES; ++s) mbar_arrive_expect_tx(&k_full[s], 2 * K_BYTES);
      for (int s = 0; s < V_STAGES; ++s) mbar_arrive_expect_tx(&v_full[s], 2 * V_BYTES);
    }
    fence_mbar_init();
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
    tma_prefetch_desc(&tm_o);
  }
  if (warp == MMA_WARP) {
    tmem_alloc_pair(tmem_slot, TMEM_COLS);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // both CTAs' barriers exist before any copy, commit or arrival crosses the pair
  tc_fence_after();
  const uint32_t tmem = __shfl_sync(0xffffffffu, *tmem_slot, 0);

  // Each warpgroup sets its register budget at the top of its branch: 168 registers per thread for
  // the softmax warps, 72 for the loading and MMA warps, 104 for the epilogue.
  if (warp >= PRODUCER_WARP && warp < EPI_WARP0) {
    regs_dec<REG_OTHER>();
    if (warp == PRODUCER_WARP || warp == V_WARP) {
      // ------------------------------------------------------------ TMA producers (both CTAs)
      // Warp 8 loads Q and this CTA's half of each K tile, warp 11 its half of each V tile; each
      // waits on its own ring's empty barriers, which the even CTA's commits reach.  The copies
      // complete on the even CTA's full barriers, already armed for both halves.
      const bool is_k = warp == PRODUCER_WARP;
      const int nst = is_k ? K_STAGES : V_STAGES;
      uint64_t* full = is_k ? k_full : v_full;
      uint64_t* empty = is_k ? k_empty : v_empty;
      bool ok = true;
      int issued = 0, nq = 0;
      Walk walk;
      WorkTile t;
      for (int k = 0; ok && walk.next(p, t, rank); ++k) {
        const int g = t.hq / G;
        if (is_k) {
          const int qs = k % Q_STAGES;
          if (k >= Q_STAGES) {
            ok = wait(&q_empty[qs], ((k / Q_STAGES) - 1) & 1);
            if (!ok) break;
          }
          if (lane == 0) {
            const uint32_t bar = cluster_addr(&q_full[qs], 0);
            for (int c = 0; c < CHUNKS; ++c) {
              if constexpr (PACKED)
                tma_load_3d_pair(sQ + qs * Q_BYTES + c * Q_PANEL, &tm_q, bar, t.hq * D + c * 64, t.base + t.qt * BM,
                                 t.z);
              else
                tma_load_3d_pair(sQ + qs * Q_BYTES + c * Q_PANEL, &tm_q, bar, t.hq * D + c * 64, t.qt * BM, t.z);
            }
          }
          nq = k + 1;
        }
        const int nkv = tile_nkv(t);
        for (int j = 0; j < nkv; ++j) {
          const int st = issued % nst;
          // paged K/V: lane l reads, before the wait, the physical page of this CTA's l-th page of the
          // key tile -- for K its half (keys 64 * rank .. + 63: 4 pages), for V all 8 pages
          constexpr int PAGES = BN / 16;
          const int npg = is_k ? PAGES / 2 : PAGES;
          const int page_first = is_k ? j * PAGES + rank * (PAGES / 2) : j * PAGES;
          int my_pid = -1;
          if constexpr (PACKED) {
            if (p.kv_lens != nullptr && lane < npg && (page_first + lane) * 16 < t.kv_len)
              my_pid = p.block_table[static_cast<size_t>(t.b) * p.max_blocks + page_first + lane];
          }
          ok = wait(&empty[st], ((issued / nst) & 1) ^ 1);
          if (!ok) break;
          const uint32_t bar = cluster_addr(&full[st], 0);
          if constexpr (!PACKED) {
            if (is_k) {
              // keys j * BN + 64 * rank .. + 63, both 64-column panels of d
              if (lane < CHUNKS)
                tma_load_3d_pair(sK + st * K_BYTES + lane * KH_PANEL, &tm_k, bar, g * D + lane * 64,
                                 j * BN + rank * KH_ROWS, t.z);
            } else if (lane == 0) {
              // all BN keys, head-dim columns 64 * rank .. + 63
              tma_load_3d_pair(sV + st * V_BYTES, &tm_v, bar, g * D + rank * 64, j * BN, t.z);
            }
          } else if (p.kv_lens == nullptr) {
            // packed sequences, contiguous K/V: the same boxes from the sequence's first token
            if (is_k) {
              if (lane < CHUNKS)
                tma_load_3d_pair(sK + st * K_BYTES + lane * KH_PANEL, &tm_k, bar, g * D + lane * 64,
                                 t.base + j * BN + rank * KH_ROWS, t.z);
            } else if (lane == 0) {
              tma_load_3d_pair(sV + st * V_BYTES, &tm_v, bar, g * D + rank * 64, t.base + j * BN, t.z);
            }
          } else {
            // paged K/V, one 16-row box per page: K lane l takes page l / 2 of this CTA's half and
            // panel l % 2 of d; V lane l takes page l and this CTA's panel (rank).  Pages past the
            // sequence are read from rows past the cache, which the copy fills with zeros.
            const int src = is_k ? lane / CHUNKS : lane;
            int pid = __shfl_sync(0xffffffffu, my_pid, src < npg ? src : 0);
            const int pp = src, c = is_k ? lane % CHUNKS : rank;
            if (is_k ? lane < npg * CHUNKS : lane < npg) {
              const int oob = p.num_blocks * 16;
              const int valid = t.kv_len - (page_first + pp) * 16;  // rows of this page that hold keys
              int row0 = oob;
              if (valid > 0) {
                if (pid < 0 || pid >= p.num_blocks) {
                  set_error(&g_prefill_cta2_status, kDevBadPage);
                  pid = 0;
                }
                row0 = pid * 16;
              }
              uint8_t* dst = is_k ? sK + st * K_BYTES + c * KH_PANEL + pp * 16 * PANEL_ROW
                                  : sV + st * V_BYTES + pp * 16 * PANEL_ROW;
              if (!is_k && valid > 0 && valid < 16) {
                // the V rows past the last key must be finite (P is 0 there, but 0 * NaN is not):
                // row by row, the tail from past the cache
#pragma unroll 1
                for (int r = 0; r < 16; ++r)
                  tma_load_3d_pair(dst + r * PANEL_ROW, &tm_vrow, bar, c * 64, g, r < valid ? row0 + r : oob);
              } else {
                tma_load_3d_pair(dst, is_k ? &tm_k : &tm_v, bar, c * 64, g, row0);
              }
            }
          }
          ++issued;
        }
      }
      if (lane == 0) {
        if (!ok) set_error(&g_prefill_cta2_status, kDevWaitTimeout);
        // Drain (even CTA, which holds the full barriers): every copy of the pair must have landed
        // before the CTAs exit.  The newest copy of each stage is the one whose phase is current.
        if (rank == 0) {
          for (int i = (issued > nst ? issued - nst : 0); i < issued; ++i)
            mbar_wait(&full[i % nst], (i / nst) & 1);
          for (int i = (nq > Q_STAGES ? nq - Q_STAGES : 0); i < nq; ++i)
            mbar_wait(&q_full[i % Q_STAGES], (i / Q_STAGES) & 1);
        }
      }
    } else if (warp == MMA_WARP && rank == 0) {
      // ------------------------------------------------------------ S = Q K^T issue (even CTA)
      // S of global step gs goes to TMEM buffer gs % 3 (in both SMs), which held P of step gs - 3:
      // wait until that P.V is done.  The whole warp runs the loop; one elected lane issues.
      constexpr uint32_t IDESC_S = idesc_bf16_f32(2 * BM, BN, 0);  // Q (K-major) x K (K-major), M = 256
      bool ok = true;
      int gs = 0;
      Walk walk;
      WorkTile t;
      for (int k = 0; ok && walk.next(p, t, rank); ++k) {
        const int qs = k % Q_STAGES;
        if (!wait(&q_full[qs], (k / Q_STAGES) & 1)) {
          ok = false;
          break;
        }
        if (lane == 0) mbar_arrive_expect_tx(&q_full[qs], 2 * Q_BYTES);  // arm its next phase
        const uint32_t qbase = smem_u32(sQ + qs * Q_BYTES);
        const int nkv = tile_nkv(t);
        for (int j = 0; j < nkv; ++j, ++gs) {
          const int sb = gs % NSB;
          const int st = gs % K_STAGES;
          if ((gs >= NSB && !wait(&pv_done[sb], ((gs - NSB) / NSB) & 1)) || !wait(&k_full[st], (gs / K_STAGES) & 1)) {
            ok = false;
            break;
          }
          if (lane == 0) mbar_arrive_expect_tx(&k_full[st], 2 * K_BYTES);  // arm its next phase
          tc_fence_after();
          const uint32_t kbase = smem_u32(sK + st * K_BYTES);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            // 16 columns of d: panel kk / 4, 32 bytes into its 128-byte rows
            const uint32_t qoff = (kk >> 2) * Q_PANEL + (kk & 3) * 32;
            const uint32_t koff = (kk >> 2) * KH_PANEL + (kk & 3) * 32;
            umma_ss_pair_warp(tmem + sb * BN, smem_desc_sw128(qbase + qoff, 16, 1024),
                              smem_desc_sw128(kbase + koff, 16, 1024), IDESC_S, kk > 0 ? 1u : 0u);
          }
          umma_commit_pair_warp(&s_full[sb], BOTH);
          umma_commit_pair_warp(&k_empty[st], BOTH);
        }
        umma_commit_pair_warp(&q_empty[qs], BOTH);  // the buffers may take another Q once these are done
      }
      if (!ok) set_error(&g_prefill_cta2_status, kDevWaitTimeout);
      umma_commit_pair_warp(&mma_done[0], EVEN);
      if (!wait(&mma_done[0], 0)) set_error(&g_prefill_cta2_status, kDevWaitTimeout);
    } else if (warp == PV_WARP && rank == 0) {
      // ------------------------------------------------------------ O += P V issue (even CTA)
      constexpr uint32_t IDESC_O = idesc_bf16_f32(2 * BM, D, 1);  // P (TMEM) x V (MN-major), M = 256
      const uint32_t o_tmem = tmem + O_COL;
      bool ok = true;
      int gs = 0;
      Walk walk;
      WorkTile t;
      for (int k = 0; ok && walk.next(p, t, rank); ++k) {
        // the first product of a tile overwrites O: both epilogues must have read the previous one
        if (k > 0 && !wait(o_free, (k - 1) & 1)) {
          ok = false;
          break;
        }
        const int nkv = tile_nkv(t);
        for (int j = 0; j < nkv; ++j, ++gs) {
          const int sb = gs % NSB;
          const int st = gs % V_STAGES;
          if (!wait(&p_full[sb], (gs / NSB) & 1) || !wait(&v_full[st], (gs / V_STAGES) & 1)) {
            ok = false;
            break;
          }
          if (lane == 0) mbar_arrive_expect_tx(&v_full[st], 2 * V_BYTES);  // arm its next phase
          tc_fence_after();
          const uint32_t vbase = smem_u32(sV + st * V_BYTES);
          const uint32_t p_tmem = tmem + sb * BN;
#pragma unroll
          for (int kk = 0; kk < BN / 16; ++kk)  // 16 keys = two 8-row swizzle atoms of this CTA's panel
            umma_ts_pair_warp(o_tmem, p_tmem + kk * 8, smem_desc_sw128(vbase + kk * 16 * 128, BN * 128, 1024),
                              IDESC_O, (j > 0 || kk > 0) ? 1u : 0u);
          umma_commit_pair_warp(&pv_done[sb], BOTH);
          umma_commit_pair_warp(&v_empty[st], BOTH);
          if (j == nkv - 1) umma_commit_pair_warp(o_full, BOTH);
        }
      }
      if (!ok) set_error(&g_prefill_cta2_status, kDevWaitTimeout);
      umma_commit_pair_warp(&mma_done[1], EVEN);
      if (!wait(&mma_done[1], 0)) set_error(&g_prefill_cta2_status, kDevWaitTimeout);
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
    Walk walk;
    WorkTile t;
    pf::SoftmaxRows rows;
    for (int k = 0; walk.next(p, t, rank); ++k) {
      const int qa = t.q_off + t.qt * BM + ra;  // positions of rows a and b among the keys
      const int nkv = tile_nkv(t);
      rows.reset();
      for (int j = 0; j < nkv; ++j, ++gs) {
        const int sb = gs % NSB;
        if (ok) ok = __all_sync(0xffffffffu, mbar_wait(&s_full[sb], (gs / NSB) & 1));
        tc_fence_after();
        pf::softmax_step<BN, D, NSB>(p, t, j, gs, tmem + lane_base + sb * BN, tmem + lane_base + O_COL, qa, qa + 8,
                                     cq, c2, c2x2, pv_done, rows, ok);
        if (lane == 0) mbar_arrive_remote(cluster_addr(&p_full[sb], 0));  // one per warp, on the even CTA's barrier
      }
      pf::softmax_tile_end(k, ra, lane, rows, l_empty, l_full, xl, ok);
    }
    if (!ok) set_error(&g_prefill_cta2_status, kDevWaitTimeout);
  } else {
    regs_dec<REG_EPI>();
    // ------------------------------------------------------------ epilogue (prefill_tile.cuh)
    const int row = (warp & 3) * 32 + lane;
    const int et = threadIdx.x - EPI_WARP0 * 32;
    const uint32_t o_row = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16) + O_COL;
    auto release_o = [&]() {
      if (lane == 0) mbar_arrive_remote(cluster_addr(o_free, 0));
    };
    bool ok = true;
    Walk walk;
    WorkTile t;
    for (int k = 0; walk.next(p, t, rank); ++k)
      pf::epilogue_tile<D, OGRP>(p, t, k, row, et, lane, o_row, xl, l_full, l_empty, o_full, sO, &tm_o, release_o,
                                   ok);
    if (!ok) set_error(&g_prefill_cta2_status, kDevWaitTimeout);
    if (et == 0) tma_store_wait0();
  }


  __syncwarp();  // single-lane roles rejoin their warps before the CTA barrier
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // the even CTA's products have finished with the odd CTA's memory
  if (warp == MMA_WARP) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, TMEM_COLS);
  }
}

}  // namespace

bool prefill_cta2_supported(int d, int Hq, int Hkv, bool packed) {
  (void)packed;  // packed and paged batches take the kernel's packed instance
  return d == D && Hkv > 0 && Hq % Hkv == 0 && (Hq / Hkv) % 2 == 0;
}

cudaError_t prefill_cta2_launch(const PrefillMaps& m, const PrefillParams& p_in, bool blocked, int sms,
                                cudaStream_t stream) {
  const bool packed = p_in.cu_seqlens != nullptr;
  auto kern = !packed ? (blocked ? prefill_cta2_kernel<false, true> : prefill_cta2_kernel<false, false>)
                      : (blocked ? prefill_cta2_kernel<true, true> : prefill_cta2_kernel<true, false>);
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
  if (e != cudaSuccess) return e;
  PrefillParams p = p_in;
  p.div_heads = FastDiv::make(static_cast<uint32_t>(p.Hq / 2));
  p.div_level = FastDiv::make(static_cast<uint32_t>(p.B * (p.Hq / 2)));
  if (packed && p.kv_lens != nullptr) {  // the paged blocked walk's divisors, in head pairs (the host counted heads)
    p.div_block_level = FastDiv::make(static_cast<uint32_t>(p.seq_block * (p.Hq / 2)));
    p.div_block = FastDiv::make(static_cast<uint32_t>(p.seq_block * (p.Hq / 2) * p.num_qblocks));
  }
  const long long units = static_cast<long long>(p.num_qblocks) * p.B * (p.Hq / 2);
  const int clusters = static_cast<int>(units < sms / 2 ? units : sms / 2);  // one pair per two SMs
  kern<<<2 * clusters, NUM_THREADS, SMEM_BYTES, stream>>>(m.q, m.k, m.v, m.o, m.v_row, p);
  return cudaGetLastError();
}

int prefill_cta2_k_rows() { return KH_ROWS; }

cudaError_t prefill_cta2_status(uint32_t* out, bool clear) {
  cudaError_t e = cudaMemcpyFromSymbol(out, g_prefill_cta2_status, sizeof(uint32_t));
  if (e == cudaSuccess && clear) {
    const uint32_t zero = 0;
    e = cudaMemcpyToSymbol(g_prefill_cta2_status, &zero, sizeof(uint32_t));
  }
  return e;
}

}  // namespace attn
