// Internal interface between the C-ABI layer and the prefill kernel.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

namespace attn {

// TMA descriptors of one prefill call.  Q/O: [B][S][Hq*d], K/V: [B][S][Hkv*d]
// (3-D maps, 64-element x 128-row boxes, 128-byte swizzle).
struct PrefillMaps {
  CUtensorMap q, k, v, o;
};

struct PrefillParams {
  float* lse;        // [B][Hq][S] or null
  int B, Hq, Hkv, S;
  float scale;       // natural-units score scale
  float scale_log2;  // scale * log2(e)
  int causal;
  int num_qblocks;   // ceil(S / rows per CTA)
  int n_kv_total;    // ceil(S / 128)
};

int prefill_rows_per_cta();
int prefill_tile_rows();
cudaError_t prefill_launch(int d, const PrefillMaps& maps, const PrefillParams& p, cudaStream_t stream);
cudaError_t prefill_status(uint32_t* out, bool clear);

}  // namespace attn
