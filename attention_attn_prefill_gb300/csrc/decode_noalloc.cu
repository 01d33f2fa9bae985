// attn_decode_paged_noalloc: the paged decode for callers that cannot allocate.
//
// attn_decode_paged needs a caller-supplied workspace for its per-split
// partials whenever a sequence is split.  Some callers cannot provide one: a
// plugin inside a host framework that owns all device memory and hands out no
// scratch buffers, or a serving loop whose policy forbids any device
// allocation once it has started.  This entry point takes the same inputs
// and outputs but keeps the partials in a fixed array that lives in the
// library's own device memory (file scope, below), so it never allocates.
//
// The array is ATTN_DECODE_NOALLOC_SCRATCH_BYTES (32 MiB) on every device that
// loads the library, held until the process exits.  Calls share it: two calls
// whose work overlaps on the GPU (different streams, or different host
// threads) race on it.  In every split mode, balanced mode included, the
// split kernel writes each partial a call's combine reads, earlier in the
// same call, so stale contents from an earlier call are never read and
// nothing needs clearing.
//
// The entry point hands the array to attn_decode_paged as its workspace, with
// the array's size as workspace_bytes.  So every check runs in that call's own
// order: argument errors first, and ATTN_ERR_WORKSPACE (the partials would not
// fit) last, before anything is enqueued.
//
// The array's address is looked up once per device ordinal and kept.  It
// belongs to the runtime's primary context of that device, so the cache
// assumes that context is the one current at every call and is never reset
// (cudaDeviceReset) while the library is in use.
#include <cuda_runtime.h>

#include <cstddef>
#include <mutex>

#include "attn.h"

namespace {

constexpr size_t kScratchBytes = ATTN_DECODE_NOALLOC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_decode_scratch[kScratchBytes];

// Device address of g_decode_scratch per device ordinal.  In host code the
// array's name is only a host-side stand-in, so the address must come from
// cudaGetSymbolAddress, asked once per device with that device current.
void* g_scratch_addr[kMaxDevices];
std::mutex g_scratch_mutex;

attn_status_t scratch_of_current_device(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return ATTN_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  if (g_scratch_addr[dev] == nullptr) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_decode_scratch) != cudaSuccess || ptr == nullptr) return ATTN_ERR_CUDA;
    g_scratch_addr[dev] = ptr;
  }
  *out = g_scratch_addr[dev];
  return ATTN_OK;
}

}  // namespace

extern "C" attn_status_t attn_decode_paged_noalloc(const void* q, const void* k_cache, const void* v_cache,
                                                   const int32_t* block_table, const int32_t* seq_lens, void* o,
                                                   float* lse, int num_seqs, int Hq, int Hkv, int d, int page_size,
                                                   int max_blocks_per_seq, int num_blocks, int num_splits,
                                                   int split_tokens, float scale, void* stream) {
  void* scratch = nullptr;
  const attn_status_t st = scratch_of_current_device(&scratch);
  if (st != ATTN_OK) return st;
  return attn_decode_paged(q, k_cache, v_cache, block_table, seq_lens, o, lse, num_seqs, Hq, Hkv, d, page_size,
                           max_blocks_per_seq, num_blocks, num_splits, split_tokens, scale, scratch, kScratchBytes,
                           stream);
}
