// Paged split-KV decode and the log-sum-exp combine on sm_103a.
//
// What it computes: one query token per sequence attends to all seq_len
// cached tokens ("Why your local LLM feels dumber than it is" (Part 3.14),
// section "What attention is trying to calculate"), read through a block
// table of 16-token pages ("GPU Datapath: Where Every Byte Moves in One LLM
// Inference Step", section D "Paged decode attention -- the zero-reuse
// stream").  The history is cut into contiguous page-aligned groups; each
// group yields a partial (normalised output, local max, local sum) and the
// partials are merged with weights l_i * exp(m_i - M) (section "Why the
// calculation is split into groups").
//
// Split kernel: one CTA per (split, KV head, sequence).  Each of its warps
// owns every NW-th page of the split and runs its own TMA pipeline: the page's
// K and V rows for this KV head arrive as 16-row x 128-byte panels (128-byte
// swizzle) on an mbarrier.  The G query heads that share the KV head form the
// rows of a 16 x d matrix (padded with zeros), so S = Q K^T and O += P V are
// m16n8k16 tensor-core products: at d = 256 and G = 8 the stream needs about
// 8 flops per byte, more than the FP32 pipes sustain next to HBM.  Online
// softmax runs in registers with quad shuffles; O is rescaled lazily.  The
// warps' states are merged in shared memory; the CTA writes either the final
// bf16 output + LSE (one split) or its partial.
//
// Combine kernel: one warp per (sequence, query head) merges the partials.  It is
// launched as a programmatic dependent of the split kernel, which signals at the
// end of each CTA: the combine's CTAs are scheduled once every split CTA has
// written its share (earlier, they would take the registers the split kernel's
// later waves need) and wait (griddepcontrol.wait) until all of it is visible,
// which hides the second launch.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cfloat>
#include <cstdint>

#include "decode.h"
#include "sm103.cuh"

namespace attn {

__device__ uint32_t g_decode_status;

#ifdef ATTN_TEST_DROP_COPY
// Test-only builds (never the product library): when set, warp 0 of split CTA (0, 0, 0) never
// requests its first page, so the wait for it runs out (after ATTN_WAIT_LIMIT_NS) and the kernel
// takes its unwinding path and records kDevWaitTimeout.
__device__ int g_test_drop_copy;
#endif

namespace {

constexpr int PAGE = 16;
constexpr int PANEL_BYTES = PAGE * 128;  // 16 token rows x 64 bf16
constexpr float RESCALE_LOG2_THRESHOLD = 8.0f;
constexpr float LN2 = 0.693147180559945309f;

template <int D, int NW, int NS>
struct DLayout {
  static constexpr int PANELS = D / 64;
  static constexpr int KV_BYTES = PANELS * PANEL_BYTES;  // one page of K (or V) for one KV head
  static constexpr int STAGE_BYTES = 2 * KV_BYTES;
  static constexpr int Q_OFF = 0;
  static constexpr int Q_BYTES = 16 * D * 2;
  static constexpr int STAGE_OFF = (Q_OFF + Q_BYTES + 1023) & ~1023;
  static constexpr int WARP_BYTES = NS * STAGE_BYTES;
  static constexpr int BAR_OFF = STAGE_OFF + NW * WARP_BYTES;
  static constexpr int USED = BAR_OFF + NW * NS * 8;
  static constexpr int ALLOC = USED + 1024;
  // per-warp merge record (after its pipeline drains): m[16], l[16], o[16][D]
  static constexpr int MERGE_BYTES = 32 * 4 + 16 * D * 4;
  static_assert(MERGE_BYTES <= WARP_BYTES, "merge record must fit in a warp's stages");
};

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ void mma_bf16(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Byte offset of element (row, x) in a stack of 128B-swizzled 16-row panels.
__device__ __forceinline__ uint32_t panel_off(int row, int x) {
  const int u = (x & 63) >> 3;
  return (x >> 6) * PANEL_BYTES + row * 128 + ((u ^ (row & 7)) << 4) + (x & 7) * 2;
}

// Pages [first, end) of sequence n that split s owns.
__device__ __forceinline__ void split_pages(const DecodeParams& p, int L, int s, int& first, int& end) {
  const int pages = (L + PAGE - 1) / PAGE;
  int span = p.split_pages;
  if (span <= 0) span = (pages + p.num_splits - 1) / p.num_splits;
  first = s * span;
  end = first + span < pages ? first + span : pages;
  if (span <= 0 || first > pages) first = end = pages;
}

// Pages of group s in the emulating variant.  Round-robin groups (tp > 0) own the tiles
// s, s + num_splits, ... of tp pages each: page i of the group is first + (i / tp) * stride + i % tp,
// and end - first is their count.  Otherwise the group is contiguous, [first, end), with the
// num_splits rule counted in blocks of granule_pages pages.
__device__ __forceinline__ void emu_group_pages(const DecodeParams& p, int L, int s, int& first, int& end, int& tp,
                                                int& stride) {
  const int pages = (L + PAGE - 1) / PAGE;
  tp = p.rr_tile_pages;
  stride = 0;
  if (tp > 0) {
    const int P = p.num_splits;
    const int tiles = (pages + tp - 1) / tp;
    const int c = tiles > s ? (tiles - 1 - s) / P + 1 : 0;  // tiles of this group
    first = s * tp;
    stride = P * tp;
    int count = 0;
    if (c > 0) {
      const int last = (s + (c - 1) * P) * tp;  // first page of the group's last tile
      count = (c - 1) * tp + (pages - last < tp ? pages - last : tp);
    }
    end = first + count;
    return;
  }
  int span = p.split_pages;
  if (span <= 0) {
    const int gr = p.granule_pages;
    span = gr * (((pages + gr - 1) / gr + p.num_splits - 1) / p.num_splits);
  }
  first = s * span;
  end = first + span < pages ? first + span : pages;
  if (span <= 0 || first > pages) first = end = pages;
}

__device__ __forceinline__ float bf16_lo(uint32_t x) { return __uint_as_float(x << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t x) { return __uint_as_float(x & 0xffff0000u); }

// This lane's rows of the 16-row tiles (query heads): a = lane/4, b = lane/4 + 8.
template <int D>
struct WarpRows {
  float m_a, m_b;       // raw-score maxima that o and l refer to
  float l_a, l_b;       // this lane's shares of the row sums
  float o[D / 8][4];    // unnormalised output, m16n8 accumulator layout
  __device__ __forceinline__ void reset() {
    m_a = m_b = -INFINITY;
    l_a = l_b = 0.f;
#pragma unroll
    for (int i = 0; i < D / 8; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
  }
};

// ldmatrix row addresses of this lane: Q (A operand), K panels (B, as stored), V panels (B, transposed).
struct FragRows {
  int a_row, a_colh, kb_tok, kb_colh, vb_tok, vb_colh;
  __device__ __forceinline__ explicit FragRows(int lane)
      : a_row(((lane >> 3) & 1) * 8 + (lane & 7)),
        a_colh((lane >> 4) * 8),
        kb_tok((lane >> 4) * 8 + (lane & 7)),
        kb_colh(((lane >> 3) & 1) * 8),
        vb_tok(((lane >> 3) & 1) * 8 + (lane & 7)),
        vb_colh((lane >> 4) * 8) {}
};

// One 16-token page, already in shared memory (K, then V, as 16 x 128 B swizzled panels), for the
// 16 query rows of a warp: S = Q K^T, masking of the tokens past the sequence (`valid` of them are
// real), the online softmax and O += P V.  Q comes from registers (qa, d <= 128) or from the swizzled
// rows at q_base.  `first`: the page starts the rows' state.  exact_max: every increase of a row's
// max rescales (else only past 2^8); bf16_sum: the row sums add the bf16-rounded weights that P V
// uses (else the unrounded ones).
template <int D, bool Q_IN_REGS>
__device__ __forceinline__ void decode_page(uint8_t* st, int valid, bool first, bool exact_max, bool bf16_sum,
                                            const uint32_t (&qa)[Q_IN_REGS ? D / 16 : 1][4], uint32_t q_base,
                                            const FragRows& fr, float c2, int lane, WarpRows<D>& w) {
  constexpr int KV_BYTES = (D / 64) * PANEL_BYTES;
  const uint32_t k_base = smem_u32(st);
  const uint32_t v_base = k_base + KV_BYTES;
  if (valid < PAGE) {
    // zero the V rows past the end of the sequence: P is 0 there, but 0 * NaN would not be
    for (int i = lane; i < (PAGE - valid) * (D / 8); i += 32) {
      const int r = valid + i / (D / 8);
      const int x = (i % (D / 8)) * 8;
      *reinterpret_cast<uint4*>(st + KV_BYTES + panel_off(r, x)) = make_uint4(0, 0, 0, 0);
    }
    __syncwarp();
  }
  // ---- S = Q K^T (16 heads x 16 tokens)
  float sacc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk) {
    uint32_t a[4];
    if constexpr (Q_IN_REGS) {
      a[0] = qa[kk][0]; a[1] = qa[kk][1]; a[2] = qa[kk][2]; a[3] = qa[kk][3];
    } else {
      const int x = kk * 16 + fr.a_colh;
      ldsm_x4(q_base + fr.a_row * (D * 2) + (((x >> 3) ^ (fr.a_row & 7)) << 4), a[0], a[1], a[2], a[3]);
    }
    uint32_t b0, b1, b2, b3;
    ldsm_x4(k_base + panel_off(fr.kb_tok, kk * 16 + fr.kb_colh), b0, b1, b2, b3);
    mma_bf16(sacc[0], a, b0, b1);
    mma_bf16(sacc[1], a, b2, b3);
  }
  // ---- mask tokens past seq_len (also hides NaN keys there)
  const int colq = 2 * (lane & 3);
#pragma unroll
  for (int nb = 0; nb < 2; ++nb)
#pragma unroll
    for (int e = 0; e < 4; ++e)
      if (nb * 8 + colq + (e & 1) >= valid) sacc[nb][e] = -INFINITY;
  // ---- online softmax, rows a = lane/4 and b = lane/4 + 8
  float mx_a = fmaxf(fmaxf(sacc[0][0], sacc[0][1]), fmaxf(sacc[1][0], sacc[1][1]));
  float mx_b = fmaxf(fmaxf(sacc[0][2], sacc[0][3]), fmaxf(sacc[1][2], sacc[1][3]));
  mx_a = fmaxf(mx_a, __shfl_xor_sync(0xffffffffu, mx_a, 1));
  mx_a = fmaxf(mx_a, __shfl_xor_sync(0xffffffffu, mx_a, 2));
  mx_b = fmaxf(mx_b, __shfl_xor_sync(0xffffffffu, mx_b, 1));
  mx_b = fmaxf(mx_b, __shfl_xor_sync(0xffffffffu, mx_b, 2));
  float al_a = 1.f, al_b = 1.f;
  bool rs = false;
  if (first) {
    w.m_a = mx_a;
    w.m_b = mx_b;
  } else {
    if (exact_max ? mx_a > w.m_a : (mx_a - w.m_a) * c2 > RESCALE_LOG2_THRESHOLD) {
      al_a = ex2_approx((w.m_a - mx_a) * c2);
      w.l_a *= al_a;
      w.m_a = mx_a;
      rs = true;
    }
    if (exact_max ? mx_b > w.m_b : (mx_b - w.m_b) * c2 > RESCALE_LOG2_THRESHOLD) {
      al_b = ex2_approx((w.m_b - mx_b) * c2);
      w.l_b *= al_b;
      w.m_b = mx_b;
      rs = true;
    }
  }
  if (__any_sync(0xffffffffu, rs)) {
#pragma unroll
    for (int i = 0; i < D / 8; ++i) {
      w.o[i][0] *= al_a; w.o[i][1] *= al_a;
      w.o[i][2] *= al_b; w.o[i][3] *= al_b;
    }
  }
  const float mb_a = w.m_a * c2, mb_b = w.m_b * c2;
  float pr[2][4];
#pragma unroll
  for (int nb = 0; nb < 2; ++nb) {
    pr[nb][0] = ex2_approx(fmaf(sacc[nb][0], c2, -mb_a));
    pr[nb][1] = ex2_approx(fmaf(sacc[nb][1], c2, -mb_a));
    pr[nb][2] = ex2_approx(fmaf(sacc[nb][2], c2, -mb_b));
    pr[nb][3] = ex2_approx(fmaf(sacc[nb][3], c2, -mb_b));
    if (!bf16_sum) {
      w.l_a += pr[nb][0] + pr[nb][1];
      w.l_b += pr[nb][2] + pr[nb][3];
    }
  }
  uint32_t pa[4];
  pa[0] = pack_bf16x2(pr[0][0], pr[0][1]);
  pa[1] = pack_bf16x2(pr[0][2], pr[0][3]);
  pa[2] = pack_bf16x2(pr[1][0], pr[1][1]);
  pa[3] = pack_bf16x2(pr[1][2], pr[1][3]);
  if (bf16_sum) {
    w.l_a += (bf16_lo(pa[0]) + bf16_hi(pa[0])) + (bf16_lo(pa[2]) + bf16_hi(pa[2]));
    w.l_b += (bf16_lo(pa[1]) + bf16_hi(pa[1])) + (bf16_lo(pa[3]) + bf16_hi(pa[3]));
  }
  // ---- O += P V
#pragma unroll
  for (int nb = 0; nb < D / 8; nb += 2) {
    uint32_t b0, b1, b2, b3;
    ldsm_x4_t(v_base + panel_off(fr.vb_tok, nb * 8 + fr.vb_colh), b0, b1, b2, b3);
    mma_bf16(w.o[nb], pa, b0, b1);
    mma_bf16(w.o[nb + 1], pa, b2, b3);
  }
  __syncwarp();
}

// EMU: the variant that reproduces another backend's decode numerics (p.emu): its group
// geometry, an exact running max (every increase rescales), XQA's bf16 weights in the sum,
// and the backend's stored value (normalised or not, f32 or bf16-rounded).  Always writes partials.
// With p.warp_groups (small fixed-size groups) each warp owns a whole group, CTA x serving
// groups x * NW .. x * NW + NW - 1, and writes that group's partial from its own record.
template <int D, int NW, int NS, bool EMU>
__global__ void __launch_bounds__(NW * 32)
    decode_split_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                        const DecodeParams p) {
  using L = DLayout<D, NW, NS>;
  constexpr bool Q_IN_REGS = (D <= 128);
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  uint8_t* sQ = smem + L::Q_OFF;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::BAR_OFF);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int s = blockIdx.x;
  const int g = blockIdx.y;
  const int n = blockIdx.z;
  const int G = p.G;
  int seq_len = p.seq_lens[n];
  if (seq_len < 0 || seq_len > p.max_blocks * PAGE) {
    // a length the block table cannot cover: record it and stay inside the table
    if (threadIdx.x == 0) set_error(&g_decode_status, kDevBadSplit);
    seq_len = seq_len < 0 ? 0 : p.max_blocks * PAGE;
  }
  // group of this warp and its share of the group's pages: page i of the share is wstart + k * wstep
  const bool wg = EMU && p.warp_groups;
  const int wstart = wg ? 0 : warp, wstep = wg ? 1 : NW;
  int pfirst, pend, rr_tp = 0, rr_stride = 0;
  if constexpr (EMU)
    emu_group_pages(p, seq_len, wg ? s * NW + warp : s, pfirst, pend, rr_tp, rr_stride);
  else
    split_pages(p, seq_len, s, pfirst, pend);
  const int npages = pend - pfirst;
  // page of the sequence that the group's i-th page is
  auto page_at = [&](int i) -> int {
    if constexpr (EMU) {
      if (rr_tp > 0) return pfirst + (i / rr_tp) * rr_stride + i % rr_tp;
    }
    return pfirst + i;
  };
  const bool xqa_sum = EMU && p.emu == kEmuXqa;  // the sum adds the bf16-rounded weights
  if constexpr (!EMU) {
    // An empty group writes nothing: the combine visits only the groups a sequence has.
    if (npages <= 0 && !p.write_final) {
      asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
      return;
    }
  }

  uint8_t* my_stages = smem + L::STAGE_OFF + warp * L::WARP_BYTES;
  uint64_t* my_bars = bars + warp * NS;
  const int n_my = npages > wstart ? (npages - wstart + wstep - 1) / wstep : 0;

  auto issue = [&](int k) {
#ifdef ATTN_TEST_DROP_COPY
    if (g_test_drop_copy && k == 0 && warp == 0 && blockIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0) return;
#endif
    const int pi = page_at(wstart + k * wstep);
    int pid = p.block_table[static_cast<size_t>(n) * p.max_blocks + pi];
    if (pid < 0 || pid >= p.num_blocks) {
      set_error(&g_decode_status, kDevBadPage);
      pid = 0;
    }
    uint8_t* st = my_stages + (k % NS) * L::STAGE_BYTES;
    uint64_t* bar = &my_bars[k % NS];
    mbar_arrive_expect_tx(bar, L::STAGE_BYTES);
#pragma unroll
    for (int c = 0; c < L::PANELS; ++c) {
      tma_load_3d(st + c * PANEL_BYTES, &tm_k, bar, c * 64, g, pid * PAGE);
      tma_load_3d(st + L::KV_BYTES + c * PANEL_BYTES, &tm_v, bar, c * 64, g, pid * PAGE);
    }
  };

  // Each warp's lane 0 sets up its own barriers and requests its first pages at once; the Q rows
  // arrive meanwhile, and the CTA barrier below makes both visible to every thread.
  if (lane == 0) {
    for (int i = 0; i < NS; ++i) mbar_init(&my_bars[i], 1);
    fence_mbar_init();
    for (int k = 0; k < n_my && k < NS; ++k) issue(k);
  }
  // Q rows of the G heads sharing KV head g (rows >= G are zero), swizzled by 16-byte unit.
  for (int i = threadIdx.x; i < 16 * (D / 8); i += NW * 32) {
    const int r = i / (D / 8);
    const int u = i % (D / 8);
    uint4 v = make_uint4(0, 0, 0, 0);
    if (r < G)
      v = *reinterpret_cast<const uint4*>(p.q + ((static_cast<size_t>(n) * p.Hq + g * G + r) * D + u * 8));
    *reinterpret_cast<uint4*>(sQ + r * (D * 2) + ((u ^ (r & 7)) << 4)) = v;
  }
  __syncthreads();

  const uint32_t q_base = smem_u32(sQ);
  const FragRows fr(lane);
  uint32_t qa[Q_IN_REGS ? D / 16 : 1][4];
  if constexpr (Q_IN_REGS) {
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
      const int x = kk * 16 + fr.a_colh;
      ldsm_x4(q_base + fr.a_row * (D * 2) + (((x >> 3) ^ (fr.a_row & 7)) << 4), qa[kk][0], qa[kk][1], qa[kk][2],
              qa[kk][3]);
    }
  }

  const float c2 = p.scale_log2;
  WarpRows<D> w;
  w.reset();

  bool ok = true;
  int consumed = 0;
  for (int k = 0; k < n_my; ++k) {
    ok = __all_sync(0xffffffffu, mbar_wait(&my_bars[k % NS], (k / NS) & 1));
    if (!ok) break;
    consumed = k + 1;
    uint8_t* st = my_stages + (k % NS) * L::STAGE_BYTES;
    const int tok0 = page_at(wstart + k * wstep) * PAGE;
    const int valid = seq_len - tok0 < PAGE ? seq_len - tok0 : PAGE;
    decode_page<D, Q_IN_REGS>(st, valid, k == 0, EMU, xqa_sum, qa, q_base, fr, c2, lane, w);
    if (lane == 0 && k + NS < n_my) {
      fence_proxy_async_smem();
      issue(k + NS);
    }
    __syncwarp();
  }
  if (!ok) {
    set_error(&g_decode_status, kDevWaitTimeout);
    // drain copies still in flight before the stage memory is reused
    if (lane == 0)
      for (int k = consumed; k < n_my && k < consumed + NS; ++k) mbar_wait(&my_bars[k % NS], (k / NS) & 1);
  }
  __syncwarp();

  // ---- per-warp record: m (log2-scaled), l, unnormalised o, rows < 16
  w.l_a += __shfl_xor_sync(0xffffffffu, w.l_a, 1);
  w.l_a += __shfl_xor_sync(0xffffffffu, w.l_a, 2);
  w.l_b += __shfl_xor_sync(0xffffffffu, w.l_b, 1);
  w.l_b += __shfl_xor_sync(0xffffffffu, w.l_b, 2);
  float* rec_m = reinterpret_cast<float*>(my_stages);
  float* rec_l = rec_m + 16;
  float* rec_o = rec_m + 32;
  const int ra = lane >> 2, rb = ra + 8;
  if ((lane & 3) == 0) {
    const bool any = n_my > 0;
    rec_m[ra] = any ? w.m_a * c2 : -INFINITY;
    rec_m[rb] = any ? w.m_b * c2 : -INFINITY;
    rec_l[ra] = any ? w.l_a : 0.f;
    rec_l[rb] = any ? w.l_b : 0.f;
  }
#pragma unroll
  for (int nb = 0; nb < D / 8; ++nb) {
    const int x = nb * 8 + 2 * (lane & 3);
    *reinterpret_cast<float2*>(rec_o + ra * D + x) = make_float2(w.o[nb][0], w.o[nb][1]);
    *reinterpret_cast<float2*>(rec_o + rb * D + x) = make_float2(w.o[nb][2], w.o[nb][3]);
  }
  __syncthreads();

  const uint8_t* rec0 = smem + L::STAGE_OFF;
  // a group's partial, from its max M (log2-scaled), sum Lsum and unnormalised output O
  auto write_partial = [&](size_t slot, int x, float M, float Lsum, float O) {
    float val = (Lsum > 0.f) ? O / Lsum : 0.f;
    if constexpr (EMU) {
      if (p.emu == kEmuTriton || p.emu == kEmuTrt) val = O;  // the weighted-value sum itself
      if (p.emu == kEmuXqa || p.emu == kEmuTrt) val = __bfloat162float(__float2bfloat16_rn(val));
    }
    p.part_o[slot * D + x] = val;
    if (x == 0) {
      p.part_m[slot] = (Lsum > 0.f) ? M * LN2 : -INFINITY;
      p.part_l[slot] = Lsum;
    }
  };
  if (wg) {
    // ---- one group per warp: its record is the group's partial (D is a power of two: shifts only)
#pragma unroll 1
    for (int w = 0; w < NW; ++w) {
      const int grp = s * NW + w;
      if (grp >= p.splits) break;
      const float* rm = reinterpret_cast<const float*>(rec0 + w * L::WARP_BYTES);
      for (int i = threadIdx.x; i < G * D; i += NW * 32) {
        const int r = i / D, x = i % D;
        const size_t row = static_cast<size_t>(n) * p.Hq + g * G + r;
        write_partial(row * p.splits + grp, x, rm[r], rm[16 + r], rm[32 + r * D + x]);
      }
    }
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    return;
  }
  // ---- merge the warps and write the final output or this split's partial
  for (int i = threadIdx.x; i < G * D; i += NW * 32) {
    const int r = i / D, x = i % D;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < NW; ++w) M = fmaxf(M, reinterpret_cast<const float*>(rec0 + w * L::WARP_BYTES)[r]);
    float Lsum = 0.f, O = 0.f;
    if (M != -INFINITY) {
#pragma unroll
      for (int w = 0; w < NW; ++w) {
        const float* rm = reinterpret_cast<const float*>(rec0 + w * L::WARP_BYTES);
        const float wm = rm[r];
        if (wm == -INFINITY) continue;
        const float f = ex2_approx(wm - M);
        Lsum += rm[16 + r] * f;
        O += rm[32 + r * D + x] * f;
      }
    }
    const int hq = g * G + r;
    const size_t row = static_cast<size_t>(n) * p.Hq + hq;
    if (p.write_final) {
      const float out = (Lsum > 0.f) ? O / Lsum : 0.f;
      p.o[row * D + x] = __float2bfloat16_rn(out);
      if (x == 0 && p.lse != nullptr) p.lse[row] = (Lsum > 0.f) ? (M + log2f(Lsum)) * LN2 : -INFINITY;
    } else {
      write_partial(row * p.splits + s, x, M, Lsum, O);
    }
  }
  // the dependent combine may be scheduled once every CTA has written its share
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Merge of the partials of each row (sequence, query head): O = sum_i w_i o_i / sum_i w_i with
// w_i = l_i exp(m_i - M), M = max of the non-empty slots' m_i, LSE = M + ln sum_i w_i.
//
// WPR warps share a row and take its slots round-robin, each loading U slots at a time so that
// their loads are in flight together; the warps' sums (all at the same M) are then added through
// shared memory.  With a row's group count known (geo.seq_lens != null) only its groups
// are visited, so slots past them need not have been written; otherwise every slot is visited and
// a slot counts only if its l_i > 0.
template <int D, int WPR>
__global__ void __launch_bounds__(256) combine_kernel(const float* __restrict__ part_o,
                                                      const float* __restrict__ part_m,
                                                      const float* __restrict__ part_l, int rows, int splits,
                                                      CombineGeometry geo, __nv_bfloat16* __restrict__ o,
                                                      float* __restrict__ lse) {
  // the partials come from the preceding kernel in the stream: wait until they are all visible
  asm volatile("griddepcontrol.wait;" ::: "memory");
  constexpr int RPC = 8 / WPR;           // rows per CTA of 8 warps
  constexpr int PER = D / 32;            // output columns per lane
  constexpr int U = 8;                   // slots in flight per warp
  __shared__ __align__(16) float s_acc[WPR > 1 ? 8 : 1][WPR > 1 ? D : 1];
  __shared__ float s_w[8];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int wr = warp % WPR;
  const int row = blockIdx.x * RPC + warp / WPR;
  const bool live = row < rows;
  int nvalid = splits;
  if (live && geo.seq_lens != nullptr) {
    int L = geo.seq_lens[row / geo.Hq];
    L = L < 0 ? 0 : (L > geo.max_blocks * PAGE ? geo.max_blocks * PAGE : L);
    const int pages = (L + PAGE - 1) / PAGE;
    const int span = geo.split_pages > 0 ? geo.split_pages : (pages + geo.num_splits - 1) / geo.num_splits;
    const int groups = span > 0 ? (pages + span - 1) / span : 0;
    nvalid = groups < splits ? groups : splits;
  }
  const size_t rbase = static_cast<size_t>(live ? row : 0) * splits;
  const float* pm = part_m + rbase;
  const float* pl = part_l + rbase;
  float M = -INFINITY;
  if (live) {
    // all of a lane's loads of a pass are issued before any is used
    for (int i0 = lane; i0 < nvalid; i0 += 32 * 4) {
      float lv[4], mv[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int i = i0 + 32 * u;
        lv[u] = i < nvalid ? pl[i] : 0.f;
        mv[u] = i < nvalid ? pm[i] : -INFINITY;
      }
#pragma unroll
      for (int u = 0; u < 4; ++u)
        if (lv[u] > 0.f) M = fmaxf(M, mv[u]);
    }
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
  float acc[PER];
#pragma unroll
  for (int e = 0; e < PER; ++e) acc[e] = 0.f;
  float W = 0.f;
  if (live && M != -INFINITY) {
    const float* po = part_o + rbase * D + lane * PER;
    for (int i0 = wr; i0 < nvalid; i0 += WPR * U) {
      float li[U], mi[U], v[U][PER];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int i = i0 + u * WPR;
        li[u] = 0.f;
        mi[u] = -INFINITY;
        if (i < nvalid) {
          li[u] = pl[i];
          mi[u] = pm[i];
          const float* src = po + static_cast<size_t>(i) * D;
#pragma unroll
          for (int e = 0; e < PER; e += (PER >= 4 ? 4 : 2)) {
            if constexpr (PER >= 4) {
              const float4 t = *reinterpret_cast<const float4*>(src + e);
              v[u][e] = t.x; v[u][e + 1] = t.y; v[u][e + 2] = t.z; v[u][e + 3] = t.w;
            } else {
              const float2 t = *reinterpret_cast<const float2*>(src + e);
              v[u][e] = t.x; v[u][e + 1] = t.y;
            }
          }
        }
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        if (!(li[u] > 0.f)) continue;  // an empty group carries no weight (its stored values are not read)
        const float w = li[u] * expf(mi[u] - M);
        W += w;
#pragma unroll
        for (int e = 0; e < PER; ++e) acc[e] = fmaf(w, v[u][e], acc[e]);
      }
    }
  }
  if constexpr (WPR > 1) {
#pragma unroll
    for (int e = 0; e < PER; ++e) s_acc[warp][lane * PER + e] = acc[e];
    if (lane == 0) s_w[warp] = W;
    __syncthreads();
    if (wr != 0) return;
#pragma unroll
    for (int j = 1; j < WPR; ++j) {
#pragma unroll
      for (int e = 0; e < PER; ++e) acc[e] += s_acc[warp + j][lane * PER + e];
      W += s_w[warp + j];
    }
  }
  if (!live) return;
  const float inv = W > 0.f ? 1.f / W : 0.f;
  __nv_bfloat16* dst = o + static_cast<size_t>(row) * D + lane * PER;
#pragma unroll
  for (int e = 0; e < PER; e += 2) {
    *reinterpret_cast<__nv_bfloat162*>(dst + e) = __floats2bfloat162_rn(acc[e] * inv, acc[e + 1] * inv);
  }
  if (lse != nullptr && lane == 0) lse[row] = W > 0.f ? M + logf(W) : -INFINITY;
}

// ----------------------------------------------------------------------------
// Balanced decode.  The pages of all sequences, for every KV head, form one
// list ordered by (sequence, KV head, page); worker warp u of the persistent
// grid takes the contiguous share [u W / Wp, (u+1) W / Wp) of its W pages, so
// every warp streams the same number of bytes whatever the length mix.  With
// the KV head inside the sequence, warps running side by side read the other
// heads' slices of the same physical pages.  A warp writes one partial record
// per (sequence n, KV head g) its share touches, at index u + n Hkv + g
// (distinct for all warps, because shares are contiguous and ordered).  The
// combine finds the warps covering (n, g) arithmetically.
// ----------------------------------------------------------------------------

__device__ __forceinline__ int pages_of(const int32_t* lens, int n, int max_blocks) {
  int L = lens[n];
  L = L < 0 ? 0 : (L > max_blocks * PAGE ? max_blocks * PAGE : L);
  return (L + PAGE - 1) / PAGE;
}

__device__ __forceinline__ int clamped_len(const int32_t* lens, int n, int max_blocks) {
  const int L = lens[n];
  return L < 0 ? 0 : (L > max_blocks * PAGE ? max_blocks * PAGE : L);
}

// Warp-wide: total pages per KV head, and (if want >= 0) the first sequence n whose
// inclusive page prefix exceeds `want`, with the prefix before it.  All lanes get the results.
__device__ __forceinline__ void page_scan(const int32_t* lens, int N, int max_blocks, int lane, long long want,
                                          long long& total, int& n_at, long long& before, int mult = 1) {
  total = 0;
  n_at = N;
  before = 0;
  for (int base = 0; base < N; base += 32) {
    const int n = base + lane;
    const int pg = n < N ? mult * pages_of(lens, n, max_blocks) : 0;
    int incl = pg;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int t = __shfl_up_sync(0xffffffffu, incl, off);
      if (lane >= off) incl += t;
    }
    const long long excl_g = total + incl - pg;  // pages before sequence n
    if (n_at == N && want >= 0) {
      const unsigned hit = __ballot_sync(0xffffffffu, n < N && pg > 0 && excl_g <= want && want < excl_g + pg);
      if (hit) {
        const int src = __ffs(hit) - 1;
        n_at = base + src;
        before = __shfl_sync(0xffffffffu, excl_g, src);
      }
    }
    total += __shfl_sync(0xffffffffu, incl, 31);
  }
}

// Walks the (sequence, KV head, page) list, skipping empty sequences.
struct PageCursor {
  int n, g, p, np;  // sequence, KV head, page within it, pages of that sequence
  __device__ __forceinline__ void advance(const int32_t* lens, int N, int Hkv, int max_blocks) {
    if (++p < np) return;
    p = 0;
    if (++g < Hkv) return;
    g = 0;
    do {
      if (++n == N) n = 0;  // only reached past the end of the list, where nothing is read
      np = pages_of(lens, n, max_blocks);
    } while (np == 0);
  }
};

template <int D, int NW, int NS>
struct BLayout {
  static constexpr int PANELS = D / 64;
  static constexpr int KV_BYTES = PANELS * PANEL_BYTES;
  static constexpr int STAGE_BYTES = 2 * KV_BYTES;
  static constexpr int WARP_BYTES = NS * STAGE_BYTES;
  static constexpr int Q_BYTES = 16 * D * 2;  // one warp's Q rows
  static constexpr int Q_OFF = NW * WARP_BYTES;
  static constexpr int BAR_OFF = Q_OFF + NW * Q_BYTES;
  static constexpr int ALLOC = BAR_OFF + NW * NS * 8;  // the dynamic window is 1 KB-aligned (checked)
};

template <int D, int NW, int NS>
__global__ void __launch_bounds__(NW * 32)
    decode_balanced_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                           const BalancedParams p) {
  using L = BLayout<D, NW, NS>;
  constexpr bool Q_IN_REGS = (D <= 128);
  extern __shared__ __align__(1024) uint8_t smem[];
  if ((smem_u32(smem) & 1023u) != 0) {
    if (threadIdx.x == 0) set_error(&g_decode_status, kDevMisaligned);
    return;
  }
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::BAR_OFF);
  if (threadIdx.x == 0) {
    for (int i = 0; i < NW * NS; ++i) mbar_init(&bars[i], 1);
    fence_mbar_init();
  }
  if (blockIdx.x == 0)
    for (int i = threadIdx.x; i < p.N; i += NW * 32)
      if (p.seq_lens[i] < 0 || p.seq_lens[i] > p.max_blocks * PAGE) set_error(&g_decode_status, kDevBadSplit);
  __syncthreads();

  const int N = p.N, G = p.G;
  const int u = blockIdx.x * NW + warp;
  long long W, dummy_before;
  int dummy_n;
  page_scan(p.seq_lens, N, p.max_blocks, lane, -1, W, dummy_n, dummy_before, p.Hkv);
  const long long lo = static_cast<long long>(u) * W / p.warps_total;
  const long long hi = static_cast<long long>(u + 1) * W / p.warps_total;
  const int npg = static_cast<int>(hi - lo);
  if (npg <= 0) return;  // nothing to stream (warps never sync with each other after the setup)

  // cursor at the first page of this warp's share
  PageCursor cur;
  {
    long long tot, before;
    int n_at;
    page_scan(p.seq_lens, N, p.max_blocks, lane, lo, tot, n_at, before, p.Hkv);
    cur.n = n_at;
    cur.np = pages_of(p.seq_lens, n_at, p.max_blocks);
    const int r = static_cast<int>(lo - before);
    cur.g = r / cur.np;
    cur.p = r % cur.np;
  }
  PageCursor icur = cur;  // the issuing lane's cursor runs NS pages ahead

  uint8_t* my_stages = smem + warp * L::WARP_BYTES;
  uint64_t* my_bars = bars + warp * NS;
  uint8_t* sQ = smem + L::Q_OFF + warp * L::Q_BYTES;
  const uint32_t q_base = smem_u32(sQ);

  int nissued = 0;  // pages this warp's lane 0 has requested
  auto issue = [&](int k) {
    nissued = k + 1;
    int pid = p.block_table[static_cast<size_t>(icur.n) * p.max_blocks + icur.p];
    if (pid < 0 || pid >= p.num_blocks) {
      set_error(&g_decode_status, kDevBadPage);
      pid = 0;
    }
    uint8_t* st = my_stages + (k % NS) * L::STAGE_BYTES;
    uint64_t* bar = &my_bars[k % NS];
    mbar_arrive_expect_tx(bar, L::STAGE_BYTES);
#pragma unroll
    for (int c = 0; c < L::PANELS; ++c) {
      tma_load_3d(st + c * PANEL_BYTES, &tm_k, bar, c * 64, icur.g, pid * PAGE);
      tma_load_3d(st + L::KV_BYTES + c * PANEL_BYTES, &tm_v, bar, c * 64, icur.g, pid * PAGE);
    }
    icur.advance(p.seq_lens, N, p.Hkv, p.max_blocks);
  };
  if (lane == 0)
    for (int k = 0; k < npg && k < NS; ++k) issue(k);
  __syncwarp();

  const FragRows fr(lane);
  const float c2 = p.scale_log2;
  const size_t R = static_cast<size_t>(p.warps_total) + static_cast<size_t>(p.Hkv) * N;

  uint32_t qa[Q_IN_REGS ? D / 16 : 1][4];
  WarpRows<D> w;
  w.reset();
  int seg_g = -1, seg_n = -1, seg_len = 0;
  bool first = true;

  // finish the current (g, n) segment: partial record = normalised o, max (natural units), sum
  auto flush = [&]() {
    float la = w.l_a, lb = w.l_b;
    la += __shfl_xor_sync(0xffffffffu, la, 1);
    la += __shfl_xor_sync(0xffffffffu, la, 2);
    lb += __shfl_xor_sync(0xffffffffu, lb, 1);
    lb += __shfl_xor_sync(0xffffffffu, lb, 2);
    const size_t idx = static_cast<size_t>(u) + static_cast<size_t>(seg_n) * p.Hkv + seg_g;
    const int ra = lane >> 2, rb = ra + 8;
    float* ro = p.rec + idx * G * D;
    const float ia = la > 0.f ? 1.f / la : 0.f, ib = lb > 0.f ? 1.f / lb : 0.f;
#pragma unroll
    for (int nb = 0; nb < D / 8; ++nb) {
      const int x = nb * 8 + 2 * (lane & 3);
      if (ra < G) *reinterpret_cast<float2*>(ro + ra * D + x) = make_float2(w.o[nb][0] * ia, w.o[nb][1] * ia);
      if (rb < G) *reinterpret_cast<float2*>(ro + rb * D + x) = make_float2(w.o[nb][2] * ib, w.o[nb][3] * ib);
    }
    if ((lane & 3) == 0) {
      float* rm = p.rec + R * G * D + idx * G;
      float* rl = rm + R * G;
      if (ra < G) { rm[ra] = la > 0.f ? w.m_a * p.scale : -INFINITY; rl[ra] = la; }
      if (rb < G) { rm[rb] = lb > 0.f ? w.m_b * p.scale : -INFINITY; rl[rb] = lb; }
    }
  };

  bool ok = true;
  int consumed = 0;
  for (int k = 0; k < npg; ++k) {
    ok = __all_sync(0xffffffffu, mbar_wait(&my_bars[k % NS], (k / NS) & 1));
    if (!ok) break;
    consumed = k + 1;
    if (cur.g != seg_g || cur.n != seg_n) {
      if (seg_g >= 0) flush();
      seg_g = cur.g;
      seg_n = cur.n;
      seg_len = clamped_len(p.seq_lens, seg_n, p.max_blocks);
      // Q rows of the G heads of KV head g for sequence n (rows >= G zero), 16-byte units swizzled
      for (int i = lane; i < 16 * (D / 8); i += 32) {
        const int r = i / (D / 8);
        const int c = i % (D / 8);
        uint4 v = make_uint4(0, 0, 0, 0);
        if (r < G)
          v = *reinterpret_cast<const uint4*>(p.q + ((static_cast<size_t>(seg_n) * p.Hq + seg_g * G + r) * D + c * 8));
        *reinterpret_cast<uint4*>(sQ + r * (D * 2) + ((c ^ (r & 7)) << 4)) = v;
      }
      __syncwarp();
      if constexpr (Q_IN_REGS) {
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const int x = kk * 16 + fr.a_colh;
          ldsm_x4(q_base + fr.a_row * (D * 2) + (((x >> 3) ^ (fr.a_row & 7)) << 4), qa[kk][0], qa[kk][1], qa[kk][2],
                  qa[kk][3]);
        }
      }
      w.reset();
      first = true;
    }
    uint8_t* st = my_stages + (k % NS) * L::STAGE_BYTES;
    const int tok0 = cur.p * PAGE;
    const int valid = seg_len - tok0 < PAGE ? seg_len - tok0 : PAGE;
    decode_page<D, Q_IN_REGS>(st, valid, first, false, false, qa, q_base, fr, c2, lane, w);
    first = false;
    if (lane == 0 && k + NS < npg) {
      fence_proxy_async_smem();
      issue(k + NS);
    }
    __syncwarp();
    cur.advance(p.seq_lens, N, p.Hkv, p.max_blocks);
  }
  if (!ok) {
    set_error(&g_decode_status, kDevWaitTimeout);
    // copies still in flight must land before this warp's stages can be released
    if (lane == 0)
      for (int k = consumed; k < nissued; ++k) mbar_wait(&my_bars[k % NS], (k / NS) & 1);
    return;
  }
  flush();
}

// WPR warps per (sequence n, query head hq), 8 / WPR rows per CTA of 8 warps: merge the records of
// the worker warps that covered (g, n).  Every warp of a row finds the covering range and its largest
// max; the row's warps then take its records round-robin, U at a time so that their loads are in
// flight together, and their sums (all at the same max) are added through shared memory.
template <int D, int WPR>
__global__ void __launch_bounds__(256) combine_balanced_kernel(const BalancedParams p) {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  constexpr int RPC = 8 / WPR;         // rows per CTA
  constexpr int PER = D / 32;          // output columns per lane
  constexpr int U = D <= 128 ? 8 : 4;  // records in flight per warp
  __shared__ __align__(16) float s_acc[WPR > 1 ? 8 : 1][WPR > 1 ? D : 1];
  __shared__ float s_w[8];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int wr = warp % WPR;
  const int row_raw = blockIdx.x * RPC + warp / WPR;
  const bool live = row_raw < p.N * p.Hq;
  const int row = live ? row_raw : 0;
  const int n = row / p.Hq, hq = row % p.Hq;
  const int G = p.G, g = hq / G, r = hq % G;
  long long Wt, before;
  int n_at;
  page_scan(p.seq_lens, p.N, p.max_blocks, lane, -1, Wt, n_at, before, p.Hkv);
  float acc[PER];
#pragma unroll
  for (int e = 0; e < PER; ++e) acc[e] = 0.f;
  float M = -INFINITY, W = 0.f;
  const int np = live ? pages_of(p.seq_lens, n, p.max_blocks) : 0;
  if (np > 0) {
    // pages of the sequences before n (each appears once per KV head in the list)
    long long pre = 0;
    for (int base = 0; base < n; base += 32) {
      const int m2 = base + lane;
      int pg = m2 < n ? pages_of(p.seq_lens, m2, p.max_blocks) : 0;
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) pg += __shfl_xor_sync(0xffffffffu, pg, off);
      pre += pg;
    }
    const long long Wp = p.warps_total;
    const long long start = static_cast<long long>(p.Hkv) * pre + static_cast<long long>(g) * np, last = start + np - 1;
    const int u0 = static_cast<int>(((start + 1) * Wp - 1) / Wt);
    const int u1 = static_cast<int>(((last + 1) * Wp - 1) / Wt);
    const size_t R = static_cast<size_t>(p.warps_total) + static_cast<size_t>(p.Hkv) * p.N;
    const size_t j = static_cast<size_t>(n) * p.Hkv + g;
    const float* rm = p.rec + R * G * D;
    const float* rl = rm + R * G;
    // a warp whose share is empty (fewer pages than warps) wrote no record
    auto has_pages = [&](int uu) { return (uu + 1) * Wt / Wp > uu * Wt / Wp; };
    for (int uu = u0 + lane; uu <= u1; uu += 32) {
      const size_t idx = uu + j;
      if (has_pages(uu) && rl[idx * G + r] > 0.f) M = fmaxf(M, rm[idx * G + r]);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
    if (M != -INFINITY) {
      for (int u_0 = u0 + wr; u_0 <= u1; u_0 += WPR * U) {
        float li[U], mi[U], v[U][PER];
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const int uu = u_0 + u * WPR;
          li[u] = 0.f;
          mi[u] = -INFINITY;
          if (uu <= u1 && has_pages(uu)) {
            const size_t idx = uu + j;
            li[u] = rl[idx * G + r];
            mi[u] = rm[idx * G + r];
            const float* src = p.rec + (idx * G + r) * D + lane * PER;
#pragma unroll
            for (int e = 0; e < PER; e += 4) {
              const float4 t = *reinterpret_cast<const float4*>(src + e);
              v[u][e] = t.x; v[u][e + 1] = t.y; v[u][e + 2] = t.z; v[u][e + 3] = t.w;
            }
          }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
          if (!(li[u] > 0.f)) continue;
          const float w = li[u] * expf(mi[u] - M);
          W += w;
#pragma unroll
          for (int e = 0; e < PER; ++e) acc[e] = fmaf(w, v[u][e], acc[e]);
        }
      }
    }
  }
  if constexpr (WPR > 1) {
#pragma unroll
    for (int e = 0; e < PER; ++e) s_acc[warp][lane * PER + e] = acc[e];
    if (lane == 0) s_w[warp] = W;
    __syncthreads();
    if (wr != 0) return;
#pragma unroll
    for (int w = 1; w < WPR; ++w) {
#pragma unroll
      for (int e = 0; e < PER; ++e) acc[e] += s_acc[warp + w][lane * PER + e];
      W += s_w[warp + w];
    }
  }
  if (!live) return;
  const float inv = W > 0.f ? 1.f / W : 0.f;
  __nv_bfloat16* dst = p.o + static_cast<size_t>(row) * D + lane * PER;
#pragma unroll
  for (int e = 0; e < PER; e += 2)
    *reinterpret_cast<__nv_bfloat162*>(dst + e) = __floats2bfloat162_rn(acc[e] * inv, acc[e + 1] * inv);
  if (p.lse != nullptr && lane == 0) p.lse[row] = W > 0.f ? M + logf(W) : -INFINITY;
}

template <int D, int NW, int NS, int CTAS_PER_SM>
cudaError_t launch_balanced(const DecodeMaps& m, const BalancedParams& p, cudaStream_t stream) {
  auto kern = decode_balanced_kernel<D, NW, NS>;
  const int smem = BLayout<D, NW, NS>::ALLOC;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  kern<<<p.warps_total / NW, NW * 32, smem, stream>>>(m.k, m.v, p);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  // a row's records are spread over the warps that covered it; with few rows, several warps share a row
  int dev = 0, sms = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
  const long long rows = static_cast<long long>(p.N) * p.Hq;
  const int wpr = rows * 8 <= 16LL * sms ? 8 : rows * 2 <= 16LL * sms ? 2 : 1;
  cfg.gridDim = dim3(static_cast<unsigned>((rows + 8 / wpr - 1) / (8 / wpr)));
  cfg.blockDim = dim3(256);
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (wpr == 8) return cudaLaunchKernelEx(&cfg, combine_balanced_kernel<D, 8>, p);
  if (wpr == 2) return cudaLaunchKernelEx(&cfg, combine_balanced_kernel<D, 2>, p);
  return cudaLaunchKernelEx(&cfg, combine_balanced_kernel<D, 1>, p);
}

template <int D, int NW, int NS, bool EMU = false>
cudaError_t launch_split(const DecodeMaps& m, const DecodeParams& p, cudaStream_t stream) {
  auto kern = decode_split_kernel<D, NW, NS, EMU>;
  const int smem = DLayout<D, NW, NS>::ALLOC;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  dim3 grid(EMU && p.warp_groups ? (p.splits + NW - 1) / NW : p.splits, p.Hkv, p.N);
  kern<<<grid, NW * 32, smem, stream>>>(m.k, m.v, p);
  return cudaGetLastError();
}

template <int D, int NW, int NS>
int split_ctas_per_sm() {
  auto kern = decode_split_kernel<D, NW, NS, false>;
  const int smem = DLayout<D, NW, NS>::ALLOC;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess) return 0;
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, NW * 32, smem) != cudaSuccess) return 0;
  return n;
}

}  // namespace

int decode_split_ctas_per_sm(int d) {
  if (d == 128) return split_ctas_per_sm<128, 4, 2>();
  if (d == 256) return split_ctas_per_sm<256, 3, 2>();
  return 0;
}

namespace {

// 4 warps x 2 pages in flight (3 CTAs per SM) at d = 128; 3 warps x 2 pages (2 CTAs per SM) at
// d = 256: more resident warps per SM than deeper per-warp pipelines, measured on GB300.  A grid
// of no more CTAs than SMs (one short batch) takes CTAs of twice the warps instead (8 at d = 128,
// 6 at d = 256, one CTA per SM), so that each SM keeps twice as many pages in flight.
template <bool EMU>
cudaError_t launch_split_for(int d, const DecodeMaps& maps, const DecodeParams& p, cudaStream_t stream) {
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  const int nw = d == 128 ? 4 : 3;  // warps per CTA of the default shape
  const long long xs = EMU && p.warp_groups ? (p.splits + nw - 1) / nw : p.splits;
  const bool few = xs * p.Hkv * p.N <= sms && !(EMU && p.warp_groups);
  if (d == 128) return few ? launch_split<128, 8, 2, EMU>(maps, p, stream) : launch_split<128, 4, 2, EMU>(maps, p, stream);
  if (d == 256) return few ? launch_split<256, 6, 2, EMU>(maps, p, stream) : launch_split<256, 3, 2, EMU>(maps, p, stream);
  return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t decode_split_launch(int d, const DecodeMaps& maps, const DecodeParams& p, cudaStream_t stream) {
  return launch_split_for<false>(d, maps, p, stream);
}

cudaError_t decode_split_emulated_launch(int d, const DecodeMaps& maps, const DecodeParams& p, cudaStream_t stream) {
  if (p.emu == kEmuNone || p.write_final) return cudaErrorInvalidValue;
  return launch_split_for<true>(d, maps, p, stream);
}

namespace {

template <int D>
cudaError_t launch_combine(const float* part_o, const float* part_m, const float* part_l, int rows, int splits,
                           const CombineGeometry& geo, __nv_bfloat16* o, float* lse, cudaStream_t stream) {
  // warps per row: enough that each warp has about U slots, at most the CTA's 8, and fewer when
  // the rows alone give every SM work
  constexpr int U = 8;  // slots a warp has in flight (as in the kernel)
  int wpr = splits <= U ? 1 : splits <= 2 * U ? 2 : splits <= 4 * U ? 4 : 8;
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  while (wpr > 1 && static_cast<long long>(rows) * wpr > 16LL * sms) wpr /= 2;
  void (*kern)(const float*, const float*, const float*, int, int, CombineGeometry, __nv_bfloat16*, float*) =
      wpr == 1 ? combine_kernel<D, 1> : wpr == 2 ? combine_kernel<D, 2> : wpr == 4 ? combine_kernel<D, 4>
                                                                                 : combine_kernel<D, 8>;
  // programmatic dependent launch: may begin before the previous kernel in the stream has finished
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  const int rpc = 8 / wpr;
  cfg.gridDim = dim3((rows + rpc - 1) / rpc);
  cfg.blockDim = dim3(256);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, part_o, part_m, part_l, rows, splits, geo, o, lse);
}

}  // namespace

cudaError_t combine_launch(int d, const float* part_o, const float* part_m, const float* part_l, int rows,
                           int splits, const CombineGeometry& geo, void* o, float* lse, cudaStream_t stream) {
  auto* out = static_cast<__nv_bfloat16*>(o);
  if (d == 128) return launch_combine<128>(part_o, part_m, part_l, rows, splits, geo, out, lse, stream);
  if (d == 256) return launch_combine<256>(part_o, part_m, part_l, rows, splits, geo, out, lse, stream);
  if (d == 64) return launch_combine<64>(part_o, part_m, part_l, rows, splits, geo, out, lse, stream);
  return cudaErrorInvalidValue;
}

// Worker warps per CTA, pages in flight per warp and CTAs per SM of the balanced kernel.
template <int D> struct BalCfg;
template <> struct BalCfg<128> { static constexpr int NW = 3, NS = 2, CTAS = 3; };  // 60 KB per CTA
template <> struct BalCfg<256> { static constexpr int NW = 2, NS = 2, CTAS = 2; };  // 80 KB per CTA

size_t decode_balanced_records(int warps_total, int N, int Hkv) {
  return static_cast<size_t>(warps_total) + static_cast<size_t>(Hkv) * N;
}

int decode_balanced_warps(int d) {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  if (d == 128) return sms * BalCfg<128>::CTAS * BalCfg<128>::NW;
  if (d == 256) return sms * BalCfg<256>::CTAS * BalCfg<256>::NW;
  return 0;
}

cudaError_t decode_balanced_launch(int d, const DecodeMaps& maps, const BalancedParams& p, cudaStream_t stream) {
  if (d == 128) {
    using C = BalCfg<128>;
    if (p.warps_total % C::NW) return cudaErrorInvalidValue;
    return launch_balanced<128, C::NW, C::NS, C::CTAS>(maps, p, stream);
  }
  if (d == 256) {
    using C = BalCfg<256>;
    if (p.warps_total % C::NW) return cudaErrorInvalidValue;
    return launch_balanced<256, C::NW, C::NS, C::CTAS>(maps, p, stream);
  }
  return cudaErrorInvalidValue;
}

#ifdef ATTN_TEST_DROP_COPY
extern "C" int attn_test_drop_copy(int on) {
  return static_cast<int>(cudaMemcpyToSymbol(g_test_drop_copy, &on, sizeof(int)));
}
#endif

cudaError_t decode_status(uint32_t* out, bool clear) {
  cudaError_t e = cudaMemcpyFromSymbol(out, g_decode_status, sizeof(uint32_t));
  if (e == cudaSuccess && clear) {
    const uint32_t zero = 0;
    e = cudaMemcpyToSymbol(g_decode_status, &zero, sizeof(uint32_t));
  }
  return e;
}

}  // namespace attn
