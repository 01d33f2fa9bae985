// Work tiles of the prefill kernels and the order in which a persistent CTA walks them.
//
// A work tile is one 128-row query tile of one (sequence, query head).  Tiles are ordered
// longest first -- the causal cost of a tile grows with its query tile -- and dealt out in a zigzag
// over the CTAs, so that every CTA gets about the same number of key steps.  Every role of a CTA
// walks the list with its own walker and sees the same tiles, so no tile list passes between roles.
#pragma once

#include <cstdint>

#include "prefill.h"
#include "sm103.cuh"

namespace attn {
namespace pf {

constexpr int BM = 128;         // query rows per work tile (TMEM lanes)
constexpr int PANEL_ROW = 128;  // bytes of one 128B-swizzle panel row: 64 bf16

struct WorkTile {
  int b, hq, qt;  // sequence, query head (or head group), query tile within the sequence
  int base, z;    // row and batch coordinates of the sequence's first query token in the maps
  int len;        // query tokens of the sequence
  int kv_len;     // keys of the sequence (len, or its cached tokens with paged K/V)
  int q_off;      // position of its first query among the keys (kv_len - len with paged K/V, else 0)
};

// Key tiles of BN keys that a work tile's queries see: all of the sequence's keys, or (causal) those
// up to the position of the tile's last query.
template <int BN>
__device__ __forceinline__ int kv_tiles(const WorkTile& t) {
  return (t.kv_len + BN - 1) / BN;
}

template <int BN>
__device__ __forceinline__ int tile_nkv(const PrefillParams& p, const WorkTile& t) {
  const int all = kv_tiles<BN>(t);
  const int diag = (t.q_off + t.qt * BM + BM - 1) / BN + 1;
  return p.causal && diag < all ? diag : all;
}

// A packed sequence shorter than the longest one has no tiles at the top query-tile levels: every
// role skips those alike.  The divisions go through the multipliers in the parameters, which costs
// the roles a few cycles per tile instead of hundreds.
struct TileWalk {
  int v = 0;
  // 32-bit index arithmetic: the host keeps tiles x 2 below 2^31
  __device__ __forceinline__ bool next(const PrefillParams& p, WorkTile& t, uint32_t* status) {
    const int G = gridDim.x, c = blockIdx.x;
    const int per_qt = p.B * p.Hq;
    const int total = per_qt * p.num_qblocks;
    while (true) {
      const int idx = v * G + ((v & 1) ? (G - 1 - c) : c);
      ++v;
      if (idx >= total) return false;
      const int level = static_cast<int>(p.div_level.div(static_cast<uint32_t>(idx)));
      t.qt = p.num_qblocks - 1 - level;
      const int rem = idx - level * per_qt;
      t.b = static_cast<int>(p.div_heads.div(static_cast<uint32_t>(rem)));
      t.hq = rem - t.b * p.Hq;
      if (p.cu_seqlens == nullptr) {
        t.base = 0;
        t.z = t.b;
        t.len = t.kv_len = p.S;
        t.q_off = 0;
        return true;
      }
      const int s0 = p.cu_seqlens[t.b], s1 = p.cu_seqlens[t.b + 1];
      const int kvl = p.kv_lens != nullptr ? p.kv_lens[t.b] : s1 - s0;
      if (s0 < 0 || s1 < s0 || s1 > p.S || s1 - s0 > p.num_qblocks * BM || kvl < s1 - s0 ||
          (p.kv_lens != nullptr && kvl > p.max_blocks * 16)) {
        set_error(status, kDevBadSeqlens);
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

// Work index idx of the banded, lane-blocked order over `units` (sequence, head) units (see
// PrefillParams::seq_block): its query-tile level and unit.  Returns 0 past the list, 1 for a slot
// to skip (a level past the last band's or a unit past the last block's), 2 otherwise.
__device__ __forceinline__ int lane_band_unit(const PrefillParams& p, int idx, int units, int& level, int& u) {
  const int band = (p.num_qblocks + kBlockedBands - 1) / kBlockedBands;  // levels a band
  const int per_bb = p.seq_block * band;
  const int per_band = static_cast<int>(p.div_block_level.div(static_cast<uint32_t>(units + p.seq_block - 1))) * per_bb;
  if (idx >= kBlockedBands * per_band) return 0;
  const int bnd = static_cast<int>(p.div_block.div(static_cast<uint32_t>(idx)));
  const int r1 = idx - bnd * per_band;
  const int blk = static_cast<int>(p.div_block_level_last.div(static_cast<uint32_t>(r1)));
  const int r2 = r1 - blk * per_bb;
  const int lb = static_cast<int>(p.div_block_level.div(static_cast<uint32_t>(r2)));
  level = bnd * band + lb;
  u = blk * p.seq_block + (r2 - lb * p.seq_block);
  return (level >= p.num_qblocks || u >= units) ? 1 : 2;
}

// The same list in blocks whose keys and values fit in part of L2, each block walked longest tile
// first; used when all of a batch's keys and values do not fit in L2, so that the query tiles of one
// level do not evict what the next level reads again.  Chunked prefill over a paged cache goes in
// blocks of p.seq_block sequences; equal-length batches and packed prompts in blocks of p.seq_block
// (sequence, query head) units, whole KV heads, band by band of query-tile levels (see
// PrefillParams::seq_block).
struct BlockedTileWalk {
  int v = 0;
  __device__ __forceinline__ bool next(const PrefillParams& p, WorkTile& t, uint32_t* status) {
    const int G = gridDim.x, c = blockIdx.x;
    if (p.kv_lens == nullptr) {  // equal-length batches and packed prompts: lanes and bands
      const int units = p.B * p.Hq;
      while (true) {
        const int idx = v * G + ((v & 1) ? (G - 1 - c) : c);
        ++v;
        int level, u;
        const int k = lane_band_unit(p, idx, units, level, u);
        if (k == 0) return false;
        if (k == 1) continue;
        t.qt = p.num_qblocks - 1 - level;
        t.b = static_cast<int>(p.div_heads.div(static_cast<uint32_t>(u)));
        t.hq = u - t.b * p.Hq;
        if (p.cu_seqlens == nullptr) {
          t.base = 0;
          t.z = t.b;
          t.len = t.kv_len = p.S;
          t.q_off = 0;
          return true;
        }
        const int s0 = p.cu_seqlens[t.b], s1 = p.cu_seqlens[t.b + 1];
        if (s0 < 0 || s1 < s0 || s1 > p.S || s1 - s0 > p.num_qblocks * BM) {
          set_error(status, kDevBadSeqlens);
          continue;  // the sequence is skipped
        }
        t.base = s0;
        t.z = 0;
        t.len = t.kv_len = s1 - s0;
        t.q_off = 0;
        if (t.qt * BM < t.len) return true;
      }
    }
    const int total = p.B * p.Hq * p.num_qblocks;
    const int per_block = p.seq_block * p.Hq * p.num_qblocks;
    while (true) {
      const int idx = v * G + ((v & 1) ? (G - 1 - c) : c);
      ++v;
      if (idx >= total) return false;
      const int blk = static_cast<int>(p.div_block.div(static_cast<uint32_t>(idx)));
      const int r = idx - blk * per_block;
      const int b0 = blk * p.seq_block;
      const bool last = b0 + p.seq_block > p.B;
      const int per_qt = (last ? p.B - b0 : p.seq_block) * p.Hq;
      const int level = static_cast<int>((last ? p.div_block_level_last : p.div_block_level).div(static_cast<uint32_t>(r)));
      t.qt = p.num_qblocks - 1 - level;
      const int rem = r - level * per_qt;
      const int bi = static_cast<int>(p.div_heads.div(static_cast<uint32_t>(rem)));
      t.b = b0 + bi;
      t.hq = rem - bi * p.Hq;
      if (p.cu_seqlens == nullptr) {
        t.base = 0;
        t.z = t.b;
        t.len = t.kv_len = p.S;
        t.q_off = 0;
        return true;
      }
      const int s0 = p.cu_seqlens[t.b], s1 = p.cu_seqlens[t.b + 1];
      const int kvl = p.kv_lens != nullptr ? p.kv_lens[t.b] : s1 - s0;
      if (s0 < 0 || s1 < s0 || s1 > p.S || s1 - s0 > p.num_qblocks * BM || kvl < s1 - s0 ||
          (p.kv_lens != nullptr && kvl > p.max_blocks * 16)) {
        set_error(status, kDevBadSeqlens);
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

}  // namespace pf
}  // namespace attn
