// C-ABI entry point for a prefill whose inputs and outputs live in host memory (include/attn.h,
// attn_prefill_host): the transfers are part of the call and overlap the compute.
//
// The queries of the sequence are cut into chunks of rows.  Chunk c attends to keys 0 .. the end of
// chunk c, which is exactly its rows of the causal prefill ("Why your local LLM feels dumber than it
// is" (Part 3.14), section "What attention is trying to calculate": a row sees the keys up to its own
// position), so it runs as one chunked prefill (attn_prefill_paged) against the sequence's own keys
// and values, read as a paged cache whose block table is the identity.  Three streams carry the
// work: the caller's stream runs the chunks' prefills, and two streams the library owns carry the
// host-to-device and device-to-host copies.  Chunk c + 1 is copied in while chunk c is computed and
// chunk c - 1 copied out, and the two copy directions run at once on the host link.
//
// The streams and events are created once per device and kept for the life of the process; a mutex
// serialises the enqueueing of concurrent calls.  A call's copies wait for the work already on the
// caller's stream, so calls on one stream run one after the other; calls on different streams can
// overlap on the GPU (the copy streams are shared, in the order the calls were made).
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <mutex>

#include "attn.h"

namespace attn {
namespace {

constexpr int kPage = 16;
constexpr int kMaxChunks = 64;
constexpr int kMaxDevices = 64;
constexpr size_t kAlign = 256;

size_t round_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

// Byte offsets of the workspace regions: the sequence's q, k, v (K and V padded to whole pages), o
// and LSE (chunk-major: chunk c's [Hq, rows_c] block at float offset Hq * row0), the identity block
// table and four int32 per chunk {0, rows_c, end_c, 0}: the chunk's cu_seqlens_q and seq_lens.
struct Layout {
  size_t q, k, v, o, lse, table, meta, total;
  int rows, chunks, pages;
};

bool make_layout(int S, int Hq, int Hkv, int d, int chunks, Layout* L) {
  if (S < 1 || Hq < 1 || Hkv < 1 || d < 1 || chunks < 1 || chunks > kMaxChunks) return false;
  if (S > (1 << 30) || static_cast<int64_t>(Hq) * d > (1 << 30)) return false;
  L->rows = (S + chunks - 1) / chunks;
  L->chunks = (S + L->rows - 1) / L->rows;  // chunks that hold rows
  L->pages = (S + kPage - 1) / kPage;
  const size_t q_bytes = static_cast<size_t>(S) * Hq * d * 2;
  const size_t kv_bytes = static_cast<size_t>(L->pages) * kPage * Hkv * d * 2;
  size_t at = 0;
  L->q = at;
  at += round_up(q_bytes);
  L->k = at;
  at += round_up(kv_bytes);
  L->v = at;
  at += round_up(kv_bytes);
  L->o = at;
  at += round_up(q_bytes);
  L->lse = at;
  at += round_up(static_cast<size_t>(S) * Hq * 4);
  L->table = at;
  at += round_up(static_cast<size_t>(L->pages) * 4);
  L->meta = at;
  at += round_up(static_cast<size_t>(kMaxChunks) * 4 * 4);
  L->total = at;
  return true;
}

// The identity block table and the chunks' {0, rows_c, keys_c, 0}: keys_c is the end of chunk c
// (causal) or S (every row sees every key).
__global__ void host_prefill_tables_kernel(int32_t* table, int pages, int32_t* meta, int S, int rows, int chunks,
                                           int causal) {
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < pages; i += gridDim.x * blockDim.x) table[i] = i;
  if (blockIdx.x == 0) {
    for (int c = threadIdx.x; c < chunks; c += blockDim.x) {
      const int r0 = c * rows;
      const int r1 = r0 + rows < S ? r0 + rows : S;
      meta[4 * c] = 0;
      meta[4 * c + 1] = r1 - r0;
      meta[4 * c + 2] = causal ? r1 : S;
      meta[4 * c + 3] = 0;
    }
  }
}

struct CopyStreams {
  bool ready = false;
  cudaStream_t in = nullptr, out = nullptr;
  cudaEvent_t start = nullptr, arrived = nullptr, done = nullptr, finished = nullptr;
};

std::mutex g_mutex;
CopyStreams g_streams[kMaxDevices];

// The current device's copy streams and events (created on first use).  Called under g_mutex.
cudaError_t copy_streams(CopyStreams** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  CopyStreams& s = g_streams[dev];
  if (!s.ready) {
    if ((e = cudaStreamCreateWithFlags(&s.in, cudaStreamNonBlocking)) != cudaSuccess) return e;
    if ((e = cudaStreamCreateWithFlags(&s.out, cudaStreamNonBlocking)) != cudaSuccess) return e;
    for (cudaEvent_t* ev : {&s.start, &s.arrived, &s.done, &s.finished})
      if ((e = cudaEventCreateWithFlags(ev, cudaEventDisableTiming)) != cudaSuccess) return e;
    s.ready = true;
  }
  *out = &s;
  return cudaSuccess;
}

}  // namespace
}  // namespace attn

using namespace attn;  // the helpers above

extern "C" {

size_t attn_prefill_host_workspace_bytes(int S, int Hq, int Hkv, int d, int chunks) {
  Layout L;
  if (Hkv < 1 || Hq % Hkv != 0 || (d != 64 && d != 128 && d != 256) || !make_layout(S, Hq, Hkv, d, chunks, &L))
    return 0;
  return L.total;
}

attn_status_t attn_prefill_host(const void* q_host, const void* k_host, const void* v_host, void* o_host,
                                float* lse_host, int S, int Hq, int Hkv, int d, float scale, int causal, int chunks,
                                void* workspace, size_t workspace_bytes, void* stream) {
  if (q_host == nullptr || k_host == nullptr || v_host == nullptr || o_host == nullptr || workspace == nullptr)
    return ATTN_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(workspace) % kAlign != 0) return ATTN_ERR_INVALID_ARG;
  if (Hkv < 1 || Hq < 1 || Hq % Hkv != 0) return ATTN_ERR_INVALID_ARG;
  if (d != 64 && d != 128 && d != 256) return ATTN_ERR_UNSUPPORTED;
  Layout L;
  if (!make_layout(S, Hq, Hkv, d, chunks, &L)) return ATTN_ERR_INVALID_ARG;
  if (workspace_bytes < L.total) return ATTN_ERR_WORKSPACE;
  // the first chunk's call checks scale and the rest of the arguments; checking scale here keeps an
  // invalid call from enqueueing anything
  if (!std::isfinite(scale) || !(scale > 0.f)) return ATTN_ERR_INVALID_ARG;

  uint8_t* ws = static_cast<uint8_t*>(workspace);
  uint8_t* q = ws + L.q;
  uint8_t* k = ws + L.k;
  uint8_t* v = ws + L.v;
  uint8_t* o = ws + L.o;
  float* lse = reinterpret_cast<float*>(ws + L.lse);
  int32_t* table = reinterpret_cast<int32_t*>(ws + L.table);
  int32_t* meta = reinterpret_cast<int32_t*>(ws + L.meta);
  const size_t q_row = static_cast<size_t>(Hq) * d * 2, kv_row = static_cast<size_t>(Hkv) * d * 2;
  const uint8_t* qh = static_cast<const uint8_t*>(q_host);
  const uint8_t* kh = static_cast<const uint8_t*>(k_host);
  const uint8_t* vh = static_cast<const uint8_t*>(v_host);
  uint8_t* oh = static_cast<uint8_t*>(o_host);
  cudaStream_t st = static_cast<cudaStream_t>(stream);

  std::lock_guard<std::mutex> lock(g_mutex);
  CopyStreams* cs = nullptr;
  if (copy_streams(&cs) != cudaSuccess) return ATTN_ERR_CUDA;
  cudaError_t e = cudaSuccess;
  auto ok = [&](cudaError_t r) {
    if (e == cudaSuccess) e = r;
    return e == cudaSuccess;
  };
  // the copies wait for the work the caller enqueued before this call
  if (!ok(cudaEventRecord(cs->start, st)) || !ok(cudaStreamWaitEvent(cs->in, cs->start, 0)) ||
      !ok(cudaStreamWaitEvent(cs->out, cs->start, 0)))
    return ATTN_ERR_CUDA;
  host_prefill_tables_kernel<<<(L.pages + 255) / 256, 256, 0, cs->in>>>(table, L.pages, meta, S, L.rows, L.chunks,
                                                                        causal ? 1 : 0);
  if (!ok(cudaGetLastError())) return ATTN_ERR_CUDA;
  for (int c = 0; c < L.chunks; ++c) {
    const int r0 = c * L.rows;
    const int r1 = r0 + L.rows < S ? r0 + L.rows : S;
    const int n = r1 - r0;
    // chunk c's rows of q in, with its rows of k and v (causal), or with all of k and v before the
    // first chunk (every row sees every key)
    const int k0 = causal ? r0 : 0, k1 = causal ? r1 : (c == 0 ? S : 0);
    if (!ok(cudaMemcpyAsync(q + r0 * q_row, qh + r0 * q_row, n * q_row, cudaMemcpyHostToDevice, cs->in)))
      return ATTN_ERR_CUDA;
    if (k1 > k0 &&
        (!ok(cudaMemcpyAsync(k + k0 * kv_row, kh + k0 * kv_row, (k1 - k0) * kv_row, cudaMemcpyHostToDevice, cs->in)) ||
         !ok(cudaMemcpyAsync(v + k0 * kv_row, vh + k0 * kv_row, (k1 - k0) * kv_row, cudaMemcpyHostToDevice, cs->in))))
      return ATTN_ERR_CUDA;
    if (!ok(cudaEventRecord(cs->arrived, cs->in)) || !ok(cudaStreamWaitEvent(st, cs->arrived, 0))) return ATTN_ERR_CUDA;
    // its prefill: rows r0 .. r1 - 1 against keys 0 .. keys_c - 1 through the identity block table
    float* lse_c = lse_host != nullptr ? lse + static_cast<size_t>(Hq) * r0 : nullptr;
    const attn_status_t s = attn_prefill_paged(q + r0 * q_row, k, v, table, meta + 4 * c, meta + 4 * c + 2,
                                               o + r0 * q_row, lse_c, 1, L.rows, n, Hq, Hkv, d, kPage, L.pages,
                                               L.pages, scale, causal, st);
    if (s != ATTN_OK) return s;
    // its rows of o (and of each head's LSE) out
    if (!ok(cudaEventRecord(cs->done, st)) || !ok(cudaStreamWaitEvent(cs->out, cs->done, 0)) ||
        !ok(cudaMemcpyAsync(oh + r0 * q_row, o + r0 * q_row, n * q_row, cudaMemcpyDeviceToHost, cs->out)))
      return ATTN_ERR_CUDA;
    if (lse_host != nullptr &&
        !ok(cudaMemcpy2DAsync(lse_host + r0, static_cast<size_t>(S) * 4, lse_c, static_cast<size_t>(n) * 4,
                              static_cast<size_t>(n) * 4, Hq, cudaMemcpyDeviceToHost, cs->out)))
      return ATTN_ERR_CUDA;
  }
  // later work on the caller's stream waits for the last copy out
  if (!ok(cudaEventRecord(cs->finished, cs->out)) || !ok(cudaStreamWaitEvent(st, cs->finished, 0)))
    return ATTN_ERR_CUDA;
  return ATTN_OK;
}

}  // extern "C"
