// Causal (or full) prefill attention forward on sm_103a: TMA + tcgen05 + TMEM.
//
// What it computes: "Why your local LLM feels dumber than it is" (Part 3.14),
// section "What attention is trying to calculate" -- O = softmax(scale*QK^T) V
// per query row over the keys it may see (causal: keys j <= i), plus the
// natural-log LSE of each row.
//
// How (the tiled flow of "Streaming process -- How the SM works inside a
// transformer", Steps 3-8 and its code snippet, redesigned for tcgen05):
//   * one CTA owns two 128-row Q tiles of one (batch, query head); TMA loads
//     each Q tile once (Step 3);
//   * a producer warp streams 128-key K and V tiles through a two-stage
//     shared-memory ring with mbarrier full/empty pairs (Step 6);
//   * one thread of the MMA warp issues S = Q K^T into TMEM (Step 4) and, once
//     softmax has written P, O += P V with P read straight from TMEM (Step 7);
//   * eight softmax warps (one thread per query row, one warpgroup per Q tile)
//     read S from TMEM, mask, take the running max, exponentiate with ex2 and
//     keep the running sum (Step 5); O is rescaled only when the max has grown
//     by more than 2^8 since it was last applied (exact either way, because
//     O and l always share the same reference max);
//   * the epilogue divides by l, rounds to bf16, stages the tile in shared
//     memory and stores it with TMA; LSE = m*scale + ln(l) (Step 8).
// The two Q tiles ping-pong: while one warpgroup runs softmax on its S, the
// tensor core works on the other tile's S or P.V.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cfloat>
#include <cstdint>

#include "prefill.h"
#include "sm103.cuh"

namespace attn {

__device__ uint32_t g_prefill_status;

namespace {

constexpr int BM = 128;          // query rows per Q tile (TMEM lanes)
constexpr int BN = 128;          // keys per K/V tile
constexpr int NQT = 2;           // Q tiles per CTA
constexpr int KV_STAGES = 2;
constexpr int NUM_THREADS = 320; // 8 softmax warps, 1 TMA warp, 1 MMA warp
constexpr int PRODUCER_WARP = 8;
constexpr int MMA_WARP = 9;
constexpr uint32_t TMEM_COLS = 512;
constexpr float RESCALE_LOG2_THRESHOLD = 8.0f;
constexpr int CHUNK_BYTES = 128 * 128;   // 128 rows x 128 B (64 bf16): one 128B-swizzle panel

template <int D>
struct Layout {
  static constexpr int CHUNKS = D / 64;
  static constexpr int TILE_BYTES = 128 * D * 2;
  static constexpr int Q_OFF = 0;
  static constexpr int K_OFF = Q_OFF + NQT * TILE_BYTES;
  static constexpr int V_OFF = K_OFF + KV_STAGES * TILE_BYTES;
  static constexpr int BAR_OFF = V_OFF + KV_STAGES * TILE_BYTES;
  static constexpr int NUM_BARS = 17;
  static constexpr int SLOT_OFF = BAR_OFF + NUM_BARS * 8;
  static constexpr int USED = SLOT_OFF + 16;
  // + 1 KB for aligning the base; never below ~114 KB so that one CTA holds an SM
  static constexpr int ALLOC = (USED + 1024) > 116 * 1024 ? (USED + 1024) : 116 * 1024;
};

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

template <int D>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    prefill_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                       const PrefillParams p) {
  using L = Layout<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  uint8_t* sQ = smem + L::Q_OFF;
  uint8_t* sK = smem + L::K_OFF;
  uint8_t* sV = smem + L::V_OFF;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::BAR_OFF);
  uint64_t* q_full = bars + 0;
  uint64_t* k_full = bars + 2;
  uint64_t* k_empty = bars + 4;
  uint64_t* v_full = bars + 6;
  uint64_t* v_empty = bars + 8;
  uint64_t* s_full = bars + 10;
  uint64_t* p_full = bars + 12;
  uint64_t* o_full = bars + 14;
  uint64_t* mma_done = bars + 16;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::SLOT_OFF);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int hq = blockIdx.x;
  const int qb = p.num_qblocks - 1 - static_cast<int>(blockIdx.y);  // longest causal rows first
  const int b = blockIdx.z;
  const int g = hq / (p.Hq / p.Hkv);
  const int q0 = qb * (NQT * BM);
  const int ntiles = (q0 + BM < p.S) ? 2 : 1;
  int nkv[NQT];
#pragma unroll
  for (int t = 0; t < NQT; ++t) nkv[t] = p.causal ? ((q0 + t * BM) / BN + 1) : p.n_kv_total;
  const int nkv_max = nkv[ntiles - 1];

  if (threadIdx.x == 0) {
    for (int t = 0; t < NQT; ++t) {
      mbar_init(&q_full[t], 1);
      mbar_init(&s_full[t], 1);
      mbar_init(&p_full[t], BM);
      mbar_init(&o_full[t], 1);
    }
    for (int s = 0; s < KV_STAGES; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&k_empty[s], 1);
      mbar_init(&v_full[s], 1);
      mbar_init(&v_empty[s], 1);
    }
    mbar_init(mma_done, 1);
    fence_mbar_init();
  }
  if (warp == MMA_WARP) {
    tmem_alloc(tmem_slot, TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == PRODUCER_WARP) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      tma_prefetch_desc(&tm_o);
      for (int t = 0; t < ntiles; ++t) {
        mbar_arrive_expect_tx(&q_full[t], L::TILE_BYTES);
        for (int c = 0; c < L::CHUNKS; ++c)
          tma_load_3d(sQ + t * L::TILE_BYTES + c * CHUNK_BYTES, &tm_q, &q_full[t], hq * D + c * 64, q0 + t * BM, b);
      }
      int nk = 0, nv = 0;  // K and V tiles issued
      for (int j = 0; j < nkv_max; ++j) {
        const int st = j & 1;
        const uint32_t ph = (j >> 1) & 1;
        if (!mbar_wait(&k_empty[st], ph ^ 1)) { set_error(&g_prefill_status, kDevWaitTimeout); break; }
        mbar_arrive_expect_tx(&k_full[st], L::TILE_BYTES);
        for (int c = 0; c < L::CHUNKS; ++c)
          tma_load_3d(sK + st * L::TILE_BYTES + c * CHUNK_BYTES, &tm_k, &k_full[st], g * D + c * 64, j * BN, b);
        nk = j + 1;
        if (!mbar_wait(&v_empty[st], ph ^ 1)) { set_error(&g_prefill_status, kDevWaitTimeout); break; }
        mbar_arrive_expect_tx(&v_full[st], L::TILE_BYTES);
        for (int c = 0; c < L::CHUNKS; ++c)
          tma_load_3d(sV + st * L::TILE_BYTES + c * CHUNK_BYTES, &tm_v, &v_full[st], g * D + c * 64, j * BN, b);
        nv = j + 1;
      }
      // Drain: every copy this warp started must have landed before the CTA exits.
      // The last KV_STAGES copies are the newest in their stages, so their phases are current.
      for (int j = (nk > KV_STAGES ? nk - KV_STAGES : 0); j < nk; ++j) mbar_wait(&k_full[j & 1], (j >> 1) & 1);
      for (int j = (nv > KV_STAGES ? nv - KV_STAGES : 0); j < nv; ++j) mbar_wait(&v_full[j & 1], (j >> 1) & 1);
      for (int t = 0; t < ntiles; ++t) mbar_wait(&q_full[t], 0);
    }
  } else if (warp == MMA_WARP) {
    // ------------------------------------------------------------ MMA issue
    if (lane == 0) {
      constexpr uint32_t IDESC_S = idesc_bf16_f32(BM, BN, 0);   // Q (K-major) x K (K-major)
      constexpr uint32_t IDESC_O = idesc_bf16_f32(BM, D, 1);    // P (TMEM)   x V (MN-major)
      bool ok = true;
      for (int t = 0; t < ntiles && ok; ++t) ok = mbar_wait(&q_full[t], 0);
      tc_fence_after();
      for (int j = 0; ok && j <= nkv_max; ++j) {
        for (int t = 0; t < ntiles; ++t) {
          const uint32_t s_tmem = tmem + t * 256;
          const uint32_t o_tmem = tmem + t * 256 + 128;
          if (j >= 1 && j - 1 < nkv[t]) {
            // O_t += P_t(j-1) V(j-1)
            const int jj = j - 1;
            const int st = jj & 1;
            if (!mbar_wait(&p_full[t], jj & 1) || !mbar_wait(&v_full[st], (jj >> 1) & 1)) { ok = false; break; }
            tc_fence_after();
            const uint32_t vbase = smem_u32(sV + st * L::TILE_BYTES);
#pragma unroll
            for (int kk = 0; kk < BN / 16; ++kk) {
              // 16 keys = two 8-row swizzle atoms; d panels are BN*128 bytes apart
              const uint64_t bdesc = smem_desc_sw128(vbase + kk * 16 * 128, BN * 128, 1024);
              umma_ts(o_tmem, s_tmem + kk * 8, bdesc, IDESC_O, (jj > 0 || kk > 0) ? 1u : 0u);
            }
            if (jj == nkv[t] - 1) umma_commit(&o_full[t]);
            if (t == ntiles - 1) umma_commit(&v_empty[st]);
          }
          if (j < nkv[t]) {
            // S_t(j) = Q_t K(j)^T
            const int st = j & 1;
            if (!mbar_wait(&k_full[st], (j >> 1) & 1)) { ok = false; break; }
            tc_fence_after();
            const uint32_t qbase = smem_u32(sQ + t * L::TILE_BYTES);
            const uint32_t kbase = smem_u32(sK + st * L::TILE_BYTES);
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
              const uint32_t koff = (kk >> 2) * CHUNK_BYTES + (kk & 3) * 32;
              const uint64_t adesc = smem_desc_sw128(qbase + koff, 16, 1024);
              const uint64_t bdesc = smem_desc_sw128(kbase + koff, 16, 1024);
              umma_ss(s_tmem, adesc, bdesc, IDESC_S, kk > 0 ? 1u : 0u);
            }
            umma_commit(&s_full[t]);
            if (t == ntiles - 1) umma_commit(&k_empty[st]);
          }
        }
      }
      if (!ok) set_error(&g_prefill_status, kDevWaitTimeout);
      umma_commit(mma_done);
      if (!mbar_wait(mma_done, 0)) set_error(&g_prefill_status, kDevWaitTimeout);
    }
  } else {
    // ------------------------------------------------------------ softmax + epilogue
    const int t = warp >> 2;
    if (t < ntiles) {
      const int row = (warp & 3) * 32 + lane;
      const int q = q0 + t * BM + row;
      const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
      const uint32_t s_tmem = tmem + lane_base + t * 256;
      const uint32_t o_tmem = s_tmem + 128;
      const float c2 = p.scale_log2;
      float m_used = -FLT_MAX;  // raw-score max the current O and l refer to
      float l = 0.f;
      bool ok = true;
      for (int j = 0; j < nkv[t]; ++j) {
        ok = __all_sync(0xffffffffu, mbar_wait(&s_full[t], j & 1));
        if (!ok) break;
        tc_fence_after();
        uint32_t sr[4][32];
#pragma unroll
        for (int c4 = 0; c4 < 4; ++c4) tmem_ld32(s_tmem + c4 * 32, sr[c4]);
        tmem_ld_wait();
        const bool need_mask = (p.causal && j == nkv[t] - 1) || (j == p.n_kv_total - 1 && (p.S % BN) != 0);
        if (need_mask) {
          const int key0 = j * BN;
#pragma unroll
          for (int c = 0; c < 128; ++c) {
            const int key = key0 + c;
            if ((p.causal && key > q) || key >= p.S) sr[c >> 5][c & 31] = __float_as_uint(-INFINITY);
          }
        }
        float mx0 = -INFINITY, mx1 = -INFINITY, mx2 = -INFINITY, mx3 = -INFINITY;
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          mx0 = fmaxf(mx0, __uint_as_float(sr[0][c]));
          mx1 = fmaxf(mx1, __uint_as_float(sr[1][c]));
          mx2 = fmaxf(mx2, __uint_as_float(sr[2][c]));
          mx3 = fmaxf(mx3, __uint_as_float(sr[3][c]));
        }
        const float mx = fmaxf(fmaxf(mx0, mx1), fmaxf(mx2, mx3));
        float alpha = 1.f;
        bool rescale_o = false;
        if (j == 0) {
          m_used = mx;
        } else if ((mx - m_used) * c2 > RESCALE_LOG2_THRESHOLD) {
          alpha = ex2_approx((m_used - mx) * c2);
          l *= alpha;
          rescale_o = true;
          m_used = mx;
        }
        const float mb = (m_used == -INFINITY) ? 0.f : m_used * c2;
        float rs0 = 0.f, rs1 = 0.f;
        uint32_t pk[2][32];
#pragma unroll
        for (int c = 0; c < 64; ++c) {
          const float x0 = __uint_as_float(sr[(2 * c) >> 5][(2 * c) & 31]);
          const float x1 = __uint_as_float(sr[(2 * c + 1) >> 5][(2 * c + 1) & 31]);
          const float p0 = ex2_approx(fmaf(x0, c2, -mb));
          const float p1 = ex2_approx(fmaf(x1, c2, -mb));
          rs0 += p0;
          rs1 += p1;
          pk[c >> 5][c & 31] = pack_bf16x2(p0, p1);
        }
        l += rs0 + rs1;
        // P (bf16, two per column) overwrites the first 64 columns of S
        tmem_st32(s_tmem, pk[0]);
        tmem_st32(s_tmem + 32, pk[1]);
        if (__any_sync(0xffffffffu, rescale_o)) {
          // P.V of the previous tile has completed: S of this tile was issued after it.
#pragma unroll 1
          for (int c4 = 0; c4 < D / 32; ++c4) {
            uint32_t r[32];
            tmem_ld32(o_tmem + c4 * 32, r);
            tmem_ld_wait();
#pragma unroll
            for (int c = 0; c < 32; ++c) r[c] = __float_as_uint(__uint_as_float(r[c]) * alpha);
            tmem_st32(o_tmem + c4 * 32, r);
          }
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(&p_full[t]);
      }
      // ---- epilogue: O / l -> bf16 -> smem (128B-swizzled, the Q tile's panels) -> TMA store
      if (ok) ok = mbar_wait(&o_full[t], 0);
      ok = __all_sync(0xffffffffu, ok);
      uint8_t* stage = sQ + t * L::TILE_BYTES;
      if (ok) {
        tc_fence_after();
        const float inv_l = 1.f / l;
#pragma unroll 1
        for (int c4 = 0; c4 < D / 32; ++c4) {
          uint32_t r[32];
          tmem_ld32(o_tmem + c4 * 32, r);
          tmem_ld_wait();
          uint8_t* panel = stage + (c4 >> 1) * CHUNK_BYTES + row * 128;
          const int u0 = (c4 & 1) * 4;
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            uint4 w;
            w.x = pack_bf16x2(__uint_as_float(r[8 * u + 0]) * inv_l, __uint_as_float(r[8 * u + 1]) * inv_l);
            w.y = pack_bf16x2(__uint_as_float(r[8 * u + 2]) * inv_l, __uint_as_float(r[8 * u + 3]) * inv_l);
            w.z = pack_bf16x2(__uint_as_float(r[8 * u + 4]) * inv_l, __uint_as_float(r[8 * u + 5]) * inv_l);
            w.w = pack_bf16x2(__uint_as_float(r[8 * u + 6]) * inv_l, __uint_as_float(r[8 * u + 7]) * inv_l);
            *reinterpret_cast<uint4*>(panel + (((u0 + u) ^ (row & 7)) << 4)) = w;
          }
        }
        if (p.lse != nullptr && q < p.S)
          p.lse[(static_cast<size_t>(b) * p.Hq + hq) * p.S + q] = m_used * p.scale + logf(l);
        fence_proxy_async_smem();
      } else {
        set_error(&g_prefill_status, kDevWaitTimeout);
      }
      named_barrier_sync(1 + t, BM);
      if (ok && row == 0) {
        for (int c = 0; c < L::CHUNKS; ++c) tma_store_3d(&tm_o, stage + c * CHUNK_BYTES, hq * D + c * 64, q0 + t * BM, b);
        tma_store_commit();
        tma_store_wait0();
      }
    }
  }

  __syncwarp();  // single-lane roles rejoin their warps before the CTA barrier
  tc_fence_before();
  __syncthreads();
  if (warp == MMA_WARP) {
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

template <int D>
cudaError_t launch(const PrefillMaps& m, const PrefillParams& p, cudaStream_t stream) {
  auto kern = prefill_fwd_kernel<D>;
  const int smem = Layout<D>::ALLOC;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  dim3 grid(p.Hq, p.num_qblocks, p.B);
  kern<<<grid, NUM_THREADS, smem, stream>>>(m.q, m.k, m.v, m.o, p);
  return cudaGetLastError();
}

}  // namespace

int prefill_rows_per_cta() { return NQT * BM; }
int prefill_tile_rows() { return BM; }

cudaError_t prefill_launch(int d, const PrefillMaps& maps, const PrefillParams& p, cudaStream_t stream) {
  if (d == 64) return launch<64>(maps, p, stream);
  if (d == 128) return launch<128>(maps, p, stream);
  return cudaErrorInvalidValue;
}

cudaError_t prefill_status(uint32_t* out, bool clear) {
  cudaError_t e = cudaMemcpyFromSymbol(out, g_prefill_status, sizeof(uint32_t));
  if (e == cudaSuccess && clear) {
    const uint32_t zero = 0;
    e = cudaMemcpyToSymbol(g_prefill_status, &zero, sizeof(uint32_t));
  }
  return e;
}

}  // namespace attn
