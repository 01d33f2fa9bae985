// Internal interface between the C-ABI layer and the decode kernels.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

namespace attn {

// TMA descriptors of the paged caches: 3-D maps {d, Hkv, num_blocks*page},
// 64-element x 1-head x 16-token boxes, 128-byte swizzle.
struct DecodeMaps {
  CUtensorMap k, v;
};

struct DecodeParams {
  const __nv_bfloat16* q;      // [N][Hq][d]
  const int32_t* block_table;  // [N][max_blocks]
  const int32_t* seq_lens;     // [N]
  __nv_bfloat16* o;            // [N][Hq][d]    (write_final)
  float* lse;                  // [N][Hq] or null (write_final)
  float* part_o;               // [N][Hq][splits][d]
  float* part_m;               // [N][Hq][splits]
  float* part_l;               // [N][Hq][splits]
  int N, Hq, Hkv, G;
  int max_blocks, num_blocks;
  int splits;       // grid extent along splits (partial slots per row)
  int split_pages;  // > 0: pages per split; 0: ceil(pages / num_splits) per sequence
  int num_splits;
  float scale;
  float scale_log2;
  int write_final;  // 1: write o / lse directly (one split)
  // Backend-numerics emulation (read only by the emulating kernel variant):
  int emu;            // EmuNumerics value
  int rr_tile_pages;  // > 0: groups take tiles of this many pages round-robin (num_splits groups)
  int granule_pages;  // pages per block of the num_splits rule (>= 1)
  int warp_groups;    // 1: each warp owns a whole group (fixed-size groups of split_pages pages)
};

// Decode numerics of other backends that the emulating split kernel and merge reproduce:
// where the groups come from, what a group stores, and how the groups are merged.
enum EmuNumerics : int {
  kEmuNone = 0,
  kEmuTriton = 1,  // contiguous groups of 16-token tiles; f32 weighted-value sum; merged at the largest max
  kEmuFa2 = 2,     // contiguous groups of 64-token blocks; f32 normalised output; merged by log-sums
  kEmuXqa = 3,     // 256-token tiles round-robin; bf16 weights in the sum; bf16 normalised output
  kEmuTrt = 4,     // one group per 128-token tile; bf16 weighted-value sum; ordered running merge
};

// Balanced ("stream-K") decode: every warp of a persistent grid takes an equal
// contiguous share of the flattened (sequence, KV head, page) list and writes
// one partial record per (sequence, KV head) it touches; a combine merges them.
struct BalancedParams {
  const __nv_bfloat16* q;      // [N][Hq][d]
  const int32_t* block_table;  // [N][max_blocks]
  const int32_t* seq_lens;     // [N]
  __nv_bfloat16* o;            // [N][Hq][d]
  float* lse;                  // [N][Hq] or null
  float* rec;                  // records: o [R][G][d], then m [R][G], then l [R][G]; R = warps + N*Hkv
  int N, Hq, Hkv, G;
  int max_blocks, num_blocks;
  int warps_total;             // number of worker warps in the split grid
  float scale;
  float scale_log2;
};

size_t decode_balanced_records(int warps_total, int N, int Hkv);
int decode_balanced_warps(int d);  // worker warps of the split grid on the current device (0 on error)
cudaError_t decode_balanced_launch(int d, const DecodeMaps& maps, const BalancedParams& p, cudaStream_t stream);

cudaError_t decode_split_launch(int d, const DecodeMaps& maps, const DecodeParams& p, cudaStream_t stream);
// The split kernel's emulating variant (p.emu != kEmuNone): always writes partials.
cudaError_t decode_split_emulated_launch(int d, const DecodeMaps& maps, const DecodeParams& p, cudaStream_t stream);
// Merge of emulated partials in the chosen backend's float32 operation order; o32 and o may be null.
cudaError_t merge_emulated_launch(int numerics, const float* part_o, const float* part_m, const float* part_l,
                                  int rows, int splits, int d, float* o32, void* o, float* lse, cudaStream_t stream);
int decode_split_ctas_per_sm(int d);  // resident split-kernel CTAs per SM on the current device (0 on error)
// Which slots of a row the combine visits.  seq_lens == null: all of them (a slot counts if its l > 0).
// Otherwise row r belongs to sequence r / Hq, whose groups follow the split kernel's geometry
// (split_pages > 0 pages per group, else ceil(pages / num_splits)); only those slots are read.
struct CombineGeometry {
  const int32_t* seq_lens;
  int Hq, max_blocks, split_pages, num_splits;
};
cudaError_t combine_launch(int d, const float* part_o, const float* part_m, const float* part_l, int rows,
                           int splits, const CombineGeometry& geo, void* o, float* lse, cudaStream_t stream);
cudaError_t decode_status(uint32_t* out, bool clear);

}  // namespace attn
