// C-ABI layer of libattn.so: argument checks, TMA descriptor encoding and
// kernel dispatch.  See include/attn.h for the contract of each entry point.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cmath>
#include <vector>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "attn.h"
#include "decode.h"
#include "prefill.h"

namespace {

constexpr int kVersion = 100;  // 0.1.0
constexpr int kPage = 16;
constexpr int kAutoMaxSplits = 128;  // largest split count the automatic choice considers

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  });
  return fn;
}

// 3-D bf16 tensor map; dims innermost first, strides in bytes for dims 1 and 2.
bool encode_3d(CUtensorMap* map, const void* base, uint64_t d0, uint64_t d1, uint64_t d2, uint64_t stride1,
               uint64_t stride2, uint32_t b0, uint32_t b1, uint32_t b2) {
  auto fn = encode_fn();
  if (fn == nullptr) return false;
  const cuuint64_t dims[3] = {d0, d1, d2};
  const cuuint64_t strides[2] = {stride1, stride2};
  const cuuint32_t box[3] = {b0, b1, b2};
  const cuuint32_t estride[3] = {1, 1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estride,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

attn_status_t from_cuda(cudaError_t e) { return e == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA; }

}  // namespace

extern "C" {

const char* attn_status_string(attn_status_t s) {
  switch (s) {
    case ATTN_OK: return "ATTN_OK";
    case ATTN_ERR_INVALID_ARG: return "ATTN_ERR_INVALID_ARG";
    case ATTN_ERR_UNSUPPORTED: return "ATTN_ERR_UNSUPPORTED";
    case ATTN_ERR_WORKSPACE: return "ATTN_ERR_WORKSPACE";
    case ATTN_ERR_CUDA: return "ATTN_ERR_CUDA";
    case ATTN_ERR_DEVICE: return "ATTN_ERR_DEVICE";
  }
  return "ATTN_ERR_UNKNOWN";
}

int attn_version(void) { return kVersion; }

namespace {

// Paged K/V for the chunked prefill entry point (absent for the others).
struct PagedKV {
  const void* k_cache;
  const void* v_cache;
  const int32_t* block_table;
  const int32_t* kv_lens;
  int max_blocks, num_blocks;
};

// Shared by the prefill entry points: `batch` sequences of `rows` tokens each in the maps (one
// packed batch of `rows` tokens for packed sequences).
attn_status_t prefill_common(const void* q, const void* k, const void* v, void* o, float* lse, int batch, int Hq,
                             int Hkv, int rows, int d, float scale, int causal, const int32_t* cu_seqlens,
                             int num_seqs, int max_seqlen, const PagedKV* paged, void* stream) {
  if (q == nullptr || o == nullptr) return ATTN_ERR_INVALID_ARG;
  if (paged == nullptr && (k == nullptr || v == nullptr || !aligned16(k) || !aligned16(v))) return ATTN_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(o)) return ATTN_ERR_INVALID_ARG;
  if (lse != nullptr && (reinterpret_cast<uintptr_t>(lse) & 3u)) return ATTN_ERR_INVALID_ARG;
  if (batch < 1 || rows < 1 || Hq < 1 || Hkv < 1 || Hq % Hkv != 0) return ATTN_ERR_INVALID_ARG;
  if (!std::isfinite(scale) || !(scale > 0.f)) return ATTN_ERR_INVALID_ARG;  // masked keys stay -inf only under a positive scale
  if (d != 64 && d != 128 && d != 256) return ATTN_ERR_UNSUPPORTED;
  // TMA coordinates are int32 and each map dimension must stay below 2^32
  if (static_cast<int64_t>(Hq) * d > (1 << 30) || rows > (1 << 30) || batch > 65535 || Hq > 65535 ||
      num_seqs > (1 << 24))
    return ATTN_ERR_INVALID_ARG;

  attn::PrefillMaps maps;
  std::memset(&maps, 0, sizeof(maps));
  const uint64_t q_row = static_cast<uint64_t>(Hq) * d * 2, kv_row = static_cast<uint64_t>(Hkv) * d * 2;
  const uint32_t box = static_cast<uint32_t>(attn::prefill_tile_rows());
  const uint32_t kv_box = static_cast<uint32_t>(attn::prefill_kv_tile_rows(d));
  // equal-length batches at d = 128 with an even number of query heads per KV head run as CTA pairs,
  // whose K boxes hold one CTA's half of a key tile
  const bool cta2 = attn::prefill_cta2_supported(d, Hq, Hkv, cu_seqlens != nullptr || paged != nullptr);
  const uint32_t k_box = cta2 ? static_cast<uint32_t>(attn::prefill_cta2_k_rows()) : kv_box;
  if (!encode_3d(&maps.q, q, static_cast<uint64_t>(Hq) * d, rows, batch, q_row, q_row * rows, 64, box, 1) ||
      !encode_3d(&maps.o, o, static_cast<uint64_t>(Hq) * d, rows, batch, q_row, q_row * rows, 64, box, 1))
    return ATTN_ERR_CUDA;
  if (paged == nullptr) {
    if (!encode_3d(&maps.k, k, static_cast<uint64_t>(Hkv) * d, rows, batch, kv_row, kv_row * rows, 64, k_box, 1) ||
        !encode_3d(&maps.v, v, static_cast<uint64_t>(Hkv) * d, rows, batch, kv_row, kv_row * rows, 64, kv_box, 1))
      return ATTN_ERR_CUDA;
  } else {
    // {d, Hkv, num_blocks * 16}: 64-column x 1-head x 16-row boxes (one page), V also 1-row boxes
    const uint64_t tokens = static_cast<uint64_t>(paged->num_blocks) * kPage;
    if (!encode_3d(&maps.k, paged->k_cache, d, Hkv, tokens, static_cast<uint64_t>(d) * 2, kv_row, 64, 1, kPage) ||
        !encode_3d(&maps.v, paged->v_cache, d, Hkv, tokens, static_cast<uint64_t>(d) * 2, kv_row, 64, 1, kPage) ||
        !encode_3d(&maps.v_row, paged->v_cache, d, Hkv, tokens, static_cast<uint64_t>(d) * 2, kv_row, 64, 1, 1))
      return ATTN_ERR_CUDA;
  }

  attn::PrefillParams p;
  p.lse = lse;
  p.o = o;
  p.cu_seqlens = cu_seqlens;
  p.kv_lens = paged != nullptr ? paged->kv_lens : nullptr;
  p.block_table = paged != nullptr ? paged->block_table : nullptr;
  p.max_blocks = paged != nullptr ? paged->max_blocks : 0;
  p.num_blocks = paged != nullptr ? paged->num_blocks : 0;
  p.B = cu_seqlens != nullptr ? num_seqs : batch;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.S = rows;
  p.scale = scale;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.causal = causal ? 1 : 0;
  const int per_cta = attn::prefill_rows_per_cta();
  const int longest = cu_seqlens != nullptr ? max_seqlen : rows;
  p.num_qblocks = (longest + per_cta - 1) / per_cta;
  if (p.num_qblocks > 65535) return ATTN_ERR_INVALID_ARG;
  // the kernel's tile walk indexes (query tile, sequence, head) in 32 bits
  if (static_cast<int64_t>(p.num_qblocks) * p.B * p.Hq > (int64_t(1) << 30)) return ATTN_ERR_INVALID_ARG;
  p.div_heads = attn::FastDiv::make(static_cast<uint32_t>(p.Hq));
  p.div_level = attn::FastDiv::make(static_cast<uint32_t>(p.B * p.Hq));
  // Chunked prefill over a paged cache whose keys and values (at most max_blocks pages a sequence)
  // exceed half of L2 is walked in blocks of sequences whose keys and values take at most an eighth
  // of L2: every query tile streams its sequence's whole cached context, and level by level over all
  // sequences that context would come from HBM once per level.  The L2 is two partitions, one per
  // die, and the walk overlaps the end of one block with the start of the next, so the blocks are
  // kept well under half of it: an eighth measured 1.5-2.3% faster than half, a quarter in between.
  // (For prompts prefilled from scratch the plain longest-first walk measured faster: there the
  // blocks' tails are unbalanced.)
  p.seq_block = p.B;
  int l2_bytes = 0, sms = 0, dev = 0;  // of the current device, at every call
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&l2_bytes, cudaDevAttrL2CacheSize, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms < 2)
    return ATTN_ERR_CUDA;
  if (paged != nullptr) {
    const int64_t kv_max = std::max<int64_t>(max_seqlen, static_cast<int64_t>(paged->max_blocks) * kPage);
    const int64_t kv_seq_bytes = std::max<int64_t>(1, kv_max * Hkv * d * 2 * 2);
    if (kv_seq_bytes * p.B > l2_bytes / 2)
      p.seq_block = static_cast<int>(std::min<int64_t>(p.B, std::max<int64_t>(1, (l2_bytes / 8) / kv_seq_bytes)));
  }
  const int blocks = (p.B + p.seq_block - 1) / p.seq_block;
  p.div_block_level = attn::FastDiv::make(static_cast<uint32_t>(p.seq_block * p.Hq));
  p.div_block_level_last = attn::FastDiv::make(static_cast<uint32_t>((p.B - (blocks - 1) * p.seq_block) * p.Hq));
  p.div_block = attn::FastDiv::make(static_cast<uint32_t>(p.seq_block * p.Hq * p.num_qblocks));
  // Equal-length batches and packed prompts whose keys and values exceed three quarters of L2 at
  // d = 128, or one and a half times L2 at d = 64 and 256, go the same way in blocks of whole KV
  // heads: (sequence, KV head) "lanes" (sized for the longest sequence) whose keys and values take at
  // most an eighth of L2, with the query-tile levels in bands, so that a lane's keys and values are
  // read from HBM once a band rather than once a level.  Measured at d = 128: MHA 4 x 32 heads at
  // S = 4096 -29%; 32 query / 8 KV heads at 4 x 8192 or 8 x 4096 (134 MB) -3 to -6%; at half of L2
  // (sweep S = 4096) no gain.  At d = 64: MHA 4 x 32 heads at S = 8192 (268 MB) -10%, but 32 query /
  // 8 KV heads at 8 x 8192 (134 MB) +1%.  At d = 256: MHA 2 x 16 heads at S = 8192 (268 MB) -5%, but
  // 1 x 16 heads (134 MB) +4%.
  bool blocked = p.seq_block < p.B;
  if (paged == nullptr) {
    const int64_t lane_bytes = static_cast<int64_t>(cu_seqlens != nullptr ? max_seqlen : rows) * d * 2 * 2;
    const int64_t kv_bytes = static_cast<int64_t>(rows) * batch * Hkv * d * 2 * 2;  // rows: all tokens if packed
    if ((d == 128 ? 4 : 2) * kv_bytes > 3 * static_cast<int64_t>(l2_bytes)) {
      const int per_lane = cta2 ? Hq / Hkv / 2 : Hq / Hkv;  // work units of one KV head (head pairs or heads)
      const int64_t units = static_cast<int64_t>(p.B) * Hkv * per_lane;
      const int64_t lanes = std::max<int64_t>(1, (l2_bytes / 8) / lane_bytes);
      if (lanes * per_lane < units) {
        // blocks of whole KV heads, bands of levels (PrefillParams::seq_block)
        const int64_t ub = lanes * per_lane, nblk = (units + ub - 1) / ub;
        const int64_t band = (p.num_qblocks + attn::kBlockedBands - 1) / attn::kBlockedBands;
        if (attn::kBlockedBands * nblk * ub * band > (int64_t(1) << 30)) return ATTN_ERR_INVALID_ARG;
        p.seq_block = static_cast<int>(ub);
        p.div_block_level = attn::FastDiv::make(static_cast<uint32_t>(ub));
        p.div_block_level_last = attn::FastDiv::make(static_cast<uint32_t>(ub * band));
        p.div_block = attn::FastDiv::make(static_cast<uint32_t>(nblk * ub * band));
        blocked = true;
      }
    }
  }
  if (cta2) return from_cuda(attn::prefill_cta2_launch(maps, p, blocked, sms, static_cast<cudaStream_t>(stream)));
  return from_cuda(attn::prefill_launch(d, maps, p, blocked, sms, static_cast<cudaStream_t>(stream)));
}

}  // namespace

attn_status_t attn_prefill(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq, int Hkv,
                           int S, int d, float scale, int causal, void* stream) {
  return prefill_common(q, k, v, o, lse, B, Hq, Hkv, S, d, scale, causal, nullptr, 0, 0, nullptr, stream);
}

attn_status_t attn_prefill_varlen(const void* q, const void* k, const void* v, void* o, float* lse,
                                  const int32_t* cu_seqlens, int num_seqs, int max_seqlen, int total_tokens, int Hq,
                                  int Hkv, int d, float scale, int causal, void* stream) {
  if (cu_seqlens == nullptr || (reinterpret_cast<uintptr_t>(cu_seqlens) & 3u)) return ATTN_ERR_INVALID_ARG;
  if (num_seqs < 1 || max_seqlen < 1 || total_tokens < 1) return ATTN_ERR_INVALID_ARG;
  return prefill_common(q, k, v, o, lse, 1, Hq, Hkv, total_tokens, d, scale, causal, cu_seqlens, num_seqs,
                        max_seqlen, nullptr, stream);
}

attn_status_t attn_prefill_paged(const void* q, const void* k_cache, const void* v_cache, const int32_t* block_table,
                                 const int32_t* cu_seqlens_q, const int32_t* seq_lens, void* o, float* lse,
                                 int num_seqs, int max_seqlen_q, int total_q, int Hq, int Hkv, int d, int page_size,
                                 int max_blocks_per_seq, int num_blocks, float scale, int causal, void* stream) {
  auto aligned4 = [](const void* ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 3u) == 0; };
  if (k_cache == nullptr || v_cache == nullptr || !aligned16(k_cache) || !aligned16(v_cache)) return ATTN_ERR_INVALID_ARG;
  if (block_table == nullptr || cu_seqlens_q == nullptr || seq_lens == nullptr || !aligned4(block_table) ||
      !aligned4(cu_seqlens_q) || !aligned4(seq_lens))
    return ATTN_ERR_INVALID_ARG;
  if (num_seqs < 1 || max_seqlen_q < 1 || total_q < 1 || max_blocks_per_seq < 1 || num_blocks < 1)
    return ATTN_ERR_INVALID_ARG;
  if (page_size != kPage) return ATTN_ERR_UNSUPPORTED;
  if (static_cast<int64_t>(num_blocks) * kPage > (int64_t(1) << 30) ||
      static_cast<int64_t>(max_blocks_per_seq) * kPage > (int64_t(1) << 30))
    return ATTN_ERR_INVALID_ARG;
  const PagedKV paged{k_cache, v_cache, block_table, seq_lens, max_blocks_per_seq, num_blocks};
  return prefill_common(q, nullptr, nullptr, o, lse, 1, Hq, Hkv, total_q, d, scale, causal, cu_seqlens_q, num_seqs,
                        max_seqlen_q, &paged, stream);
}

int attn_decode_num_slots(int max_blocks_per_seq, int page_size, int num_splits, int split_tokens) {
  if (max_blocks_per_seq < 1 || page_size != kPage) return 0;
  if (split_tokens > 0) {
    if (split_tokens % page_size) return 0;
    const int64_t max_tokens = static_cast<int64_t>(max_blocks_per_seq) * page_size;
    return static_cast<int>((max_tokens + split_tokens - 1) / split_tokens);
  }
  if (split_tokens < 0 || num_splits < 1) return 0;
  return num_splits < max_blocks_per_seq ? num_splits : max_blocks_per_seq;
}

int attn_split_heuristic(int units, int capacity, int blocks, int max_splits) {
  if (units < 1 || capacity < 1 || blocks < 1 || max_splits < 1) return 0;
  int limit = max_splits < capacity ? max_splits : capacity;
  if (blocks < limit) limit = blocks;
  auto per_group = [&](int c) { return (blocks + c - 1) / c; };
  auto efficiency = [&](int c) {
    const double w = static_cast<double>(units) * c / capacity;
    return w / std::ceil(w);
  };
  // a count is a candidate only if it changes the number of blocks per group
  auto candidate = [&](int c) { return c == 1 || per_group(c) != per_group(c - 1); };
  double best = 0.0;
  for (int c = 1; c <= limit; ++c)
    if (candidate(c) && efficiency(c) > best) best = efficiency(c);
  for (int c = 1; c <= limit; ++c)
    if (candidate(c) && efficiency(c) >= 0.85 * best) return c;
  return 1;
}

int attn_decode_auto_splits(int num_seqs, int Hkv, int d, int max_blocks_per_seq) {
  if (num_seqs < 1 || Hkv < 1 || max_blocks_per_seq < 1 || (d != 128 && d != 256)) return 0;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  const int per_sm = attn::decode_split_ctas_per_sm(d);
  if (per_sm < 1) return 0;
  return attn_split_heuristic(num_seqs * Hkv, sms * per_sm, max_blocks_per_seq, kAutoMaxSplits);
}

int attn_split_tokens_rule(const int32_t* seq_lens, int num_seqs, int Hkv, int capacity, int max_blocks_per_seq) {
  if (seq_lens == nullptr || num_seqs < 1 || Hkv < 1 || capacity < 1 || max_blocks_per_seq < 1) return 0;
  const int64_t max_tokens = static_cast<int64_t>(max_blocks_per_seq) * kPage;
  if (max_tokens > (int64_t(1) << 30)) return 0;
  std::vector<int> pages(num_seqs);
  int max_pages = 0;
  int64_t total = 0;
  for (int n = 0; n < num_seqs; ++n) {
    const int64_t L = std::min<int64_t>(std::max<int64_t>(seq_lens[n], 0), max_tokens);
    pages[n] = static_cast<int>((L + kPage - 1) / kPage);
    max_pages = std::max(max_pages, pages[n]);
    total += pages[n];
  }
  if (max_pages == 0) return kPage;  // nothing to read: any group size serves
  auto items = [&](int span) {
    int64_t groups = 0;
    for (int p : pages) groups += (p + span - 1) / span;
    return groups * Hkv;
  };
  constexpr int kMinPages = 32;  // 512 tokens
  const int64_t work = total * Hkv;  // pages of all (sequence, KV head) pairs
  int span = 0;
  if (items(max_pages) <= capacity) {
    // one wave: the smallest span whose groups all fit (items falls as span grows)
    int lo = 1, hi = max_pages;
    while (lo < hi) {
      const int mid = lo + (hi - lo) / 2;
      if (items(mid) <= capacity) hi = mid; else lo = mid + 1;
    }
    lo = std::max(lo, std::min(kMinPages, max_pages));
    // kept only if its groups are near-equal: at most 5/4 of the average work per CTA
    if (4 * static_cast<int64_t>(lo) * capacity <= 5 * work || lo == std::min(kMinPages, max_pages)) span = lo;
  }
  if (span == 0) {
    // several waves: about three waves of equal power-of-two groups
    const int64_t target = std::max<int64_t>(kMinPages, work / (3 * static_cast<int64_t>(capacity)));
    span = kMinPages;
    while (static_cast<int64_t>(span) * 2 <= target) span *= 2;
    span = std::min(span, max_pages);
  }
  return span * kPage;
}

int attn_decode_auto_split_tokens(const int32_t* seq_lens, int num_seqs, int Hkv, int d, int max_blocks_per_seq) {
  if (seq_lens == nullptr || num_seqs < 1 || Hkv < 1 || max_blocks_per_seq < 1 || (d != 128 && d != 256)) return 0;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  const int per_sm = attn::decode_split_ctas_per_sm(d);
  if (per_sm < 1) return 0;
  return attn_split_tokens_rule(seq_lens, num_seqs, Hkv, sms * per_sm, max_blocks_per_seq);
}

size_t attn_decode_workspace_bytes(int num_seqs, int Hq, int d, int slots) {
  if (num_seqs < 1 || Hq < 1 || d < 1 || slots < 1) return 0;
  if (slots == 1) return 0;
  return static_cast<size_t>(num_seqs) * Hq * slots * (static_cast<size_t>(d) + 2) * sizeof(float);
}

size_t attn_decode_balanced_workspace_bytes(int num_seqs, int Hq, int Hkv, int d) {
  if (num_seqs < 1 || Hq < 1 || Hkv < 1 || Hq % Hkv != 0 || (d != 128 && d != 256)) return 0;
  const int warps = attn::decode_balanced_warps(d);
  if (warps <= 0) return 0;
  return attn::decode_balanced_records(warps, num_seqs, Hkv) * (Hq / Hkv) * (static_cast<size_t>(d) + 2) *
         sizeof(float);
}

}  // extern "C"

namespace {

// Argument checks shared by the paged decode entry points.
attn_status_t check_decode_args(const void* q, const void* k_cache, const void* v_cache, const int32_t* block_table,
                                const int32_t* seq_lens, const void* o, const float* lse, int num_seqs, int Hq,
                                int Hkv, int d, int page_size, int max_blocks_per_seq, int num_blocks, float scale) {
  if (q == nullptr || k_cache == nullptr || v_cache == nullptr || block_table == nullptr || seq_lens == nullptr ||
      o == nullptr)
    return ATTN_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(o) ||
      (reinterpret_cast<uintptr_t>(block_table) & 3u) || (reinterpret_cast<uintptr_t>(seq_lens) & 3u))
    return ATTN_ERR_INVALID_ARG;
  if (lse != nullptr && (reinterpret_cast<uintptr_t>(lse) & 3u)) return ATTN_ERR_INVALID_ARG;
  if (num_seqs < 1 || Hq < 1 || Hkv < 1 || Hq % Hkv != 0 || max_blocks_per_seq < 1 || num_blocks < 1)
    return ATTN_ERR_INVALID_ARG;
  // masked keys stay -inf only under a positive scale
  if (!std::isfinite(scale) || !(scale > 0.f)) return ATTN_ERR_INVALID_ARG;
  if (page_size != kPage) return ATTN_ERR_UNSUPPORTED;
  if (d != 128 && d != 256) return ATTN_ERR_UNSUPPORTED;
  if (Hq / Hkv > 16) return ATTN_ERR_UNSUPPORTED;  // query heads per KV head fill at most 16 MMA rows
  if (num_seqs > 65535 || Hkv > 65535) return ATTN_ERR_INVALID_ARG;
  if (static_cast<int64_t>(num_seqs) * Hq > (int64_t(1) << 30)) return ATTN_ERR_INVALID_ARG;  // rows of the combine
  if (static_cast<int64_t>(num_blocks) * page_size > (int64_t(1) << 31) - 1) return ATTN_ERR_INVALID_ARG;
  return ATTN_OK;
}

// TMA maps of the paged caches: {d, Hkv, num_blocks * page} with 64 x 1 x page boxes.
bool encode_cache_maps(attn::DecodeMaps* maps, const void* k_cache, const void* v_cache, int Hkv, int d,
                       int num_blocks, int page_size) {
  const uint64_t row = static_cast<uint64_t>(Hkv) * d * 2;
  const uint64_t tokens = static_cast<uint64_t>(num_blocks) * page_size;
  return encode_3d(&maps->k, k_cache, d, Hkv, tokens, static_cast<uint64_t>(d) * 2, row, 64, 1, page_size) &&
         encode_3d(&maps->v, v_cache, d, Hkv, tokens, static_cast<uint64_t>(d) * 2, row, 64, 1, page_size);
}

// Fields of the split kernel's parameters common to every mode.
attn::DecodeParams decode_params(const void* q, const int32_t* block_table, const int32_t* seq_lens, void* o,
                                 float* lse, int num_seqs, int Hq, int Hkv, int max_blocks_per_seq, int num_blocks,
                                 float scale) {
  attn::DecodeParams p = {};
  p.q = static_cast<const __nv_bfloat16*>(q);
  p.block_table = block_table;
  p.seq_lens = seq_lens;
  p.o = static_cast<__nv_bfloat16*>(o);
  p.lse = lse;
  p.N = num_seqs;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.G = Hq / Hkv;
  p.max_blocks = max_blocks_per_seq;
  p.num_blocks = num_blocks;
  p.scale = scale;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.emu = attn::kEmuNone;
  p.granule_pages = 1;
  return p;
}

static_assert(int{ATTN_NUMERICS_TRITON} == int{attn::kEmuTriton} && int{ATTN_NUMERICS_FA2} == int{attn::kEmuFa2} &&
                  int{ATTN_NUMERICS_XQA} == int{attn::kEmuXqa} && int{ATTN_NUMERICS_TRT} == int{attn::kEmuTrt},
              "public and internal numerics codes must agree");

bool numerics_valid(int numerics) { return numerics >= ATTN_NUMERICS_TRITON && numerics <= ATTN_NUMERICS_TRT; }

constexpr int kTrtTileTokens = 128;     // one TensorRT-LLM partial per 128-token tile
constexpr int kXqaTileTokens = 256;     // XQA deals 256-token tiles round-robin
constexpr int kFa2BlockTokens = 64;     // FlashAttention 2 splits whole 64-token blocks
constexpr int kTritonSegments = 16;     // Triton always uses 16 groups

}  // namespace

extern "C" {

attn_status_t attn_decode_paged(const void* q, const void* k_cache, const void* v_cache, const int32_t* block_table,
                                const int32_t* seq_lens, void* o, float* lse, int num_seqs, int Hq, int Hkv, int d,
                                int page_size, int max_blocks_per_seq, int num_blocks, int num_splits,
                                int split_tokens, float scale, void* workspace, size_t workspace_bytes,
                                void* stream) {
  const attn_status_t chk = check_decode_args(q, k_cache, v_cache, block_table, seq_lens, o, lse, num_seqs, Hq, Hkv,
                                              d, page_size, max_blocks_per_seq, num_blocks, scale);
  if (chk != ATTN_OK) return chk;
  if (num_splits == 0 && split_tokens == 0) {
    // balanced mode: equal shares of all pages per worker warp, then a combine
    attn::BalancedParams bp;
    bp.warps_total = attn::decode_balanced_warps(d);
    if (bp.warps_total <= 0) return ATTN_ERR_CUDA;
    const size_t need = attn_decode_balanced_workspace_bytes(num_seqs, Hq, Hkv, d);
    if (workspace == nullptr || workspace_bytes < need || !aligned16(workspace)) return ATTN_ERR_WORKSPACE;
    attn::DecodeMaps bmaps;
    if (!encode_cache_maps(&bmaps, k_cache, v_cache, Hkv, d, num_blocks, page_size)) return ATTN_ERR_CUDA;
    bp.q = static_cast<const __nv_bfloat16*>(q);
    bp.block_table = block_table;
    bp.seq_lens = seq_lens;
    bp.o = static_cast<__nv_bfloat16*>(o);
    bp.lse = lse;
    bp.rec = static_cast<float*>(workspace);
    bp.N = num_seqs;
    bp.Hq = Hq;
    bp.Hkv = Hkv;
    bp.G = Hq / Hkv;
    bp.max_blocks = max_blocks_per_seq;
    bp.num_blocks = num_blocks;
    bp.scale = scale;
    bp.scale_log2 = scale * 1.4426950408889634f;
    return from_cuda(attn::decode_balanced_launch(d, bmaps, bp, static_cast<cudaStream_t>(stream)));
  }
  const int slots = attn_decode_num_slots(max_blocks_per_seq, page_size, num_splits, split_tokens);
  if (slots < 1 || slots > 65535) return ATTN_ERR_INVALID_ARG;
  const size_t need = attn_decode_workspace_bytes(num_seqs, Hq, d, slots);
  if (need > 0 && (workspace == nullptr || workspace_bytes < need || !aligned16(workspace)))
    return ATTN_ERR_WORKSPACE;

  attn::DecodeMaps maps;
  if (!encode_cache_maps(&maps, k_cache, v_cache, Hkv, d, num_blocks, page_size)) return ATTN_ERR_CUDA;

  attn::DecodeParams p = decode_params(q, block_table, seq_lens, o, lse, num_seqs, Hq, Hkv, max_blocks_per_seq,
                                       num_blocks, scale);
  p.splits = slots;
  p.split_pages = split_tokens > 0 ? split_tokens / page_size : 0;
  p.num_splits = split_tokens > 0 ? 0 : slots;
  p.write_final = slots == 1 ? 1 : 0;
  float* ws = static_cast<float*>(workspace);
  const size_t nrow = static_cast<size_t>(num_seqs) * Hq;
  p.part_o = slots > 1 ? ws : nullptr;
  p.part_m = slots > 1 ? ws + nrow * slots * d : nullptr;
  p.part_l = slots > 1 ? ws + nrow * slots * (d + 1) : nullptr;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = attn::decode_split_launch(d, maps, p, st);
  if (e != cudaSuccess) return ATTN_ERR_CUDA;
  if (slots > 1) {
    const attn::CombineGeometry geo{seq_lens, Hq, max_blocks_per_seq, p.split_pages, p.num_splits};
    e = attn::combine_launch(d, p.part_o, p.part_m, p.part_l, static_cast<int>(nrow), slots, geo, o, lse, st);
  }
  return from_cuda(e);
}

attn_status_t attn_combine(const float* part_o, const float* part_m, const float* part_l, int rows,
                           int num_splits, int d, void* o, float* lse, void* stream) {
  if (part_o == nullptr || part_m == nullptr || part_l == nullptr || o == nullptr) return ATTN_ERR_INVALID_ARG;
  if (!aligned16(part_o) || !aligned16(o) || (reinterpret_cast<uintptr_t>(part_m) & 3u) ||
      (reinterpret_cast<uintptr_t>(part_l) & 3u))
    return ATTN_ERR_INVALID_ARG;
  if (lse != nullptr && (reinterpret_cast<uintptr_t>(lse) & 3u)) return ATTN_ERR_INVALID_ARG;
  if (rows < 1 || num_splits < 1) return ATTN_ERR_INVALID_ARG;
  if (d != 64 && d != 128 && d != 256) return ATTN_ERR_UNSUPPORTED;
  const attn::CombineGeometry all_slots{nullptr, 1, 1, 0, 1};
  return from_cuda(attn::combine_launch(d, part_o, part_m, part_l, rows, num_splits, all_slots, o, lse,
                                        static_cast<cudaStream_t>(stream)));
}

int attn_emulated_partitions(int numerics, int num_seqs, int Hkv, int max_tokens, int sm_count) {
  if (!numerics_valid(numerics) || num_seqs < 1 || Hkv < 1 || max_tokens < 1 || sm_count < 1) return 0;
  const int64_t units = static_cast<int64_t>(num_seqs) * Hkv;
  switch (numerics) {
    case ATTN_NUMERICS_TRITON:
      return kTritonSegments;
    case ATTN_NUMERICS_FA2:
      if (units > (int64_t(1) << 30) || sm_count > (1 << 29)) return 0;
      return attn_split_heuristic(static_cast<int>(units), 2 * sm_count,
                                  (max_tokens + kFa2BlockTokens - 1) / kFa2BlockTokens, kAutoMaxSplits);
    case ATTN_NUMERICS_XQA: {
      const int64_t share = sm_count / units;
      const int tiles = (max_tokens + kXqaTileTokens - 1) / kXqaTileTokens;
      return share < 1 ? 1 : (share < tiles ? static_cast<int>(share) : tiles);
    }
    default:
      return (max_tokens + kTrtTileTokens - 1) / kTrtTileTokens;
  }
}

int attn_emulated_num_slots(int numerics, int max_blocks_per_seq, int page_size, int partitions) {
  if (!numerics_valid(numerics) || max_blocks_per_seq < 1 || page_size != kPage) return 0;
  if (numerics == ATTN_NUMERICS_TRT) {
    const int64_t slots = (static_cast<int64_t>(max_blocks_per_seq) * page_size + kTrtTileTokens - 1) / kTrtTileTokens;
    return slots > 65535 ? 0 : static_cast<int>(slots);
  }
  return partitions >= 1 && partitions <= 65535 ? partitions : 0;
}

size_t attn_emulated_workspace_bytes(int num_seqs, int Hq, int d, int slots) {
  if (num_seqs < 1 || Hq < 1 || d < 1 || slots < 1) return 0;
  return static_cast<size_t>(num_seqs) * Hq * slots * (static_cast<size_t>(d) + 2) * sizeof(float);
}

attn_status_t attn_decode_paged_emulated(const void* q, const void* k_cache, const void* v_cache,
                                         const int32_t* block_table, const int32_t* seq_lens, void* o, float* lse,
                                         int num_seqs, int Hq, int Hkv, int d, int page_size, int max_blocks_per_seq,
                                         int num_blocks, int numerics, int partitions, float scale, void* workspace,
                                         size_t workspace_bytes, void* stream) {
  const attn_status_t chk = check_decode_args(q, k_cache, v_cache, block_table, seq_lens, o, lse, num_seqs, Hq, Hkv,
                                              d, page_size, max_blocks_per_seq, num_blocks, scale);
  if (chk != ATTN_OK) return chk;
  if (!numerics_valid(numerics)) return ATTN_ERR_INVALID_ARG;
  const int slots = attn_emulated_num_slots(numerics, max_blocks_per_seq, page_size, partitions);
  if (slots < 1) return ATTN_ERR_INVALID_ARG;
  const size_t need = attn_emulated_workspace_bytes(num_seqs, Hq, d, slots);
  if (workspace == nullptr || workspace_bytes < need || !aligned16(workspace)) return ATTN_ERR_WORKSPACE;

  attn::DecodeMaps maps;
  if (!encode_cache_maps(&maps, k_cache, v_cache, Hkv, d, num_blocks, page_size)) return ATTN_ERR_CUDA;
  attn::DecodeParams p = decode_params(q, block_table, seq_lens, o, lse, num_seqs, Hq, Hkv, max_blocks_per_seq,
                                       num_blocks, scale);
  p.emu = numerics;
  p.splits = slots;
  p.write_final = 0;
  p.num_splits = slots;
  switch (numerics) {
    case ATTN_NUMERICS_FA2:
      p.granule_pages = kFa2BlockTokens / kPage;
      break;
    case ATTN_NUMERICS_XQA:
      p.rr_tile_pages = kXqaTileTokens / kPage;
      break;
    case ATTN_NUMERICS_TRT:
      p.split_pages = kTrtTileTokens / kPage;
      p.num_splits = 0;
      p.warp_groups = 1;  // 8-page groups: one per warp
      break;
    default:
      break;
  }
  float* ws = static_cast<float*>(workspace);
  const size_t nrow = static_cast<size_t>(num_seqs) * Hq;
  p.part_o = ws;
  p.part_m = ws + nrow * slots * d;
  p.part_l = ws + nrow * slots * (d + 1);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = attn::decode_split_emulated_launch(d, maps, p, st);
  if (e != cudaSuccess) return ATTN_ERR_CUDA;
  return from_cuda(attn::merge_emulated_launch(numerics, p.part_o, p.part_m, p.part_l, static_cast<int>(nrow), slots,
                                               d, nullptr, o, lse, st));
}

attn_status_t attn_merge_emulated(int numerics, const float* part_o, const float* part_m, const float* part_l,
                                  int rows, int num_splits, int d, float* o_f32, void* o, float* lse, void* stream) {
  if (!numerics_valid(numerics)) return ATTN_ERR_INVALID_ARG;
  if (part_o == nullptr || part_m == nullptr || part_l == nullptr || (o_f32 == nullptr && o == nullptr))
    return ATTN_ERR_INVALID_ARG;
  auto misaligned = [](const void* ptr, uintptr_t a) { return (reinterpret_cast<uintptr_t>(ptr) & (a - 1)) != 0; };
  if (misaligned(part_o, 4) || misaligned(part_m, 4) || misaligned(part_l, 4) || misaligned(o_f32, 4) ||
      misaligned(o, 2) || misaligned(lse, 4))
    return ATTN_ERR_INVALID_ARG;
  if (rows < 1 || num_splits < 1 || d < 1 || d > 1024) return ATTN_ERR_INVALID_ARG;
  return from_cuda(attn::merge_emulated_launch(numerics, part_o, part_m, part_l, rows, num_splits, d, o_f32, o, lse,
                                               static_cast<cudaStream_t>(stream)));
}

attn_status_t attn_device_status(uint32_t* code, int clear) {
  if (code == nullptr) return ATTN_ERR_INVALID_ARG;
  if (cudaDeviceSynchronize() != cudaSuccess) return ATTN_ERR_CUDA;
  uint32_t a = 0, b = 0;
  if (attn::prefill_status(&a, clear != 0) != cudaSuccess) return ATTN_ERR_CUDA;
  if (attn::decode_status(&b, clear != 0) != cudaSuccess) return ATTN_ERR_CUDA;
  *code = a != 0 ? a : b;
  return ATTN_OK;
}

}  // extern "C"
