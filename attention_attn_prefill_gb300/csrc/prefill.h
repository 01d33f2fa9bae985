// Internal interface between the C-ABI layer and the prefill kernel.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

namespace attn {

// TMA descriptors of one prefill call.  Q/O: [B][S][Hq*d], K/V: [B][S][Hkv*d] (B = 1 for packed
// sequences); 3-D maps, 64-element x 128-row boxes, 128-byte swizzle.
struct PrefillMaps {
  CUtensorMap q, k, v, o;
  CUtensorMap v_row;  // paged K/V only: V with one-row boxes, for the last page of a sequence
};

// Two layouts share one kernel:
//   * fixed length (cu_seqlens == null): B sequences of S tokens, maps [B][S][H*d], LSE [B][Hq][S];
//   * packed (cu_seqlens != null): B sequences of cu_seqlens[n+1] - cu_seqlens[n] tokens stored
//     back to back, S = total tokens, maps [1][S][H*d], LSE [Hq][S].
//   * paged K/V (kv_lens != null, packed queries): sequence n's keys are its kv_lens[n] cached tokens,
//     read through block_table (16-token pages; maps {d, Hkv, num_blocks*16}); its packed queries are
//     the last cu_seqlens[n+1] - cu_seqlens[n] of them.
// x / d for 0 <= x < 2^31 by a multiply-high, an add and a shift: the round-up method of
// Granlund and Montgomery, "Division by Invariant Integers using Multiplication" (1994), section 4,
// with s = ceil(log2 d) and m = floor(2^32 (2^s - d) / d) + 1 < 2^32.
struct FastDiv {
  uint32_t m = 1, s = 0;
  static FastDiv make(uint32_t d) {  // d >= 1
    FastDiv f;
    if (d == 0) d = 1;
    while ((1ull << f.s) < d) ++f.s;
    f.m = static_cast<uint32_t>(((1ull << 32) * ((1ull << f.s) - d)) / d + 1);
    return f;
  }
#ifdef __CUDACC__
  __device__ __forceinline__ uint32_t div(uint32_t x) const {
    return static_cast<uint32_t>((static_cast<uint64_t>(__umulhi(x, m)) + x) >> s);
  }
#endif
};

struct PrefillParams {
  float* lse;                  // LSE (see above) or null
  void* o;                     // output base (bf16), for the rows of a partial packed tile
  const int32_t* cu_seqlens;   // [B + 1] or null
  const int32_t* kv_lens;      // [B] cached tokens per sequence (paged K/V), or null
  const int32_t* block_table;  // [B][max_blocks] (paged K/V)
  int max_blocks, num_blocks;  // (paged K/V)
  int B, Hq, Hkv, S;
  float scale;       // natural-units score scale
  float scale_log2;  // scale * log2(e)
  int causal;
  int num_qblocks;   // query tiles of the longest sequence: ceil(S or max_seqlen / 128)
  FastDiv div_heads;  // by Hq
  FastDiv div_level;  // by B * Hq: work tiles per query-tile level
  // Blocked walks (BlockedTileWalk and the CTA-pair kernel's blocked instances), taken when a batch's
  // keys and values do not fit in L2; the host picks the instance.
  //  * Packed sequences: blocks of seq_block sequences (the last block may hold fewer), each block
  //    longest tile first; the divisors are by seq_block * heads (work tiles per query-tile level of
  //    a full block), (B - (blocks - 1) * seq_block) * heads (the same for the last block) and
  //    seq_block * heads * num_qblocks (work tiles of a full block).
  //  * Equal-length batches: the work units (sequence, query head) -- (sequence, head pair) in the
  //    CTA-pair kernel -- numbered b * heads + h, in blocks of seq_block consecutive units (whole KV
  //    heads), and the query-tile levels in kBlockedBands bands of band = ceil(num_qblocks /
  //    kBlockedBands) levels, longest first.  Band by band, block by block, each block's levels of
  //    the band longest first: a block's keys and values stay in L2 over a band, and the walk ends
  //    on the shortest tiles.  The divisors are by seq_block, seq_block * band and blocks *
  //    seq_block * band (the tiles of one band); levels and units past the batch are skipped.
  // (The two share fields: a larger parameter block measured about 1% slower on every cell.)
  int seq_block;
  FastDiv div_block_level;
  FastDiv div_block_level_last;
  FastDiv div_block;
};

constexpr int kBlockedBands = 4;

int prefill_rows_per_cta();
int prefill_tile_rows();            // rows of a Q / O box
int prefill_kv_tile_rows(int d);    // rows of a K / V box for head dim d
// blocked: take the blocked walk's instance (PrefillParams::seq_block); sms: the current device's SMs
cudaError_t prefill_launch(int d, const PrefillMaps& maps, const PrefillParams& p, bool blocked, int sms,
                           cudaStream_t stream);
cudaError_t prefill_status(uint32_t* out, bool clear);  // both prefill kernels' status words

// CTA-pair kernel (prefill_cta2.cu): head dim 128, an even number of query heads per KV head, a batch
// of equal-length sequences.  Its K map has boxes of prefill_cta2_k_rows() rows (a CTA's half of a
// K tile); Q, V and O maps are as for the single-head kernel.
bool prefill_cta2_supported(int d, int Hq, int Hkv, bool packed);
int prefill_cta2_k_rows();
cudaError_t prefill_cta2_launch(const PrefillMaps& maps, const PrefillParams& p, bool blocked, int sms,
                                cudaStream_t stream);
cudaError_t prefill_cta2_status(uint32_t* out, bool clear);

}  // namespace attn
