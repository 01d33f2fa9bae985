// Per-tile work of the softmax warps (one key step; the end of a tile) and of the epilogue warps,
// shared by both prefill kernels (one CTA per tile in prefill.cu, CTA pairs in prefill_cta2.cu).
//
// Warp w takes 16 whole rows of the 128-row tile: TMEM lanes r0 .. r0 + 15 with r0 = 32 (w % 4) +
// 16 (w / 4).  Through the 16x256b TMEM shape four threads share a row: thread t holds rows r0 + t/4
// ("a") and r0 + t/4 + 8 ("b"), columns 8i + 2(t % 4) and 8i + 2(t % 4) + 1 of each group i of 8
// columns.  A row max is then two shuffles, and no warp waits for another.
//
// Online softmax ("Streaming process -- How the SM works inside a transformer", Step 5, with the lazy
// rescale of this library): the exponentials are taken
// against a reference max per row.  That is exact for any reference, because O and l always refer to
// the same one, and nothing overflows while every p stays below 2^32.  The first step of a tile
// takes the score of key 0 (visible to every row of a first key tile) as the reference, one shuffle
// instead of a row max.  Every step keeps the reference unless one of this thread's partial row sums
// leaves that range.  Only then does it take the row max, move the reference (rescaling O and l when
// the max has grown by more than 2^8, except on the first step, which has no O or l yet) and compute
// its P again.
#pragma once

#include <cstdint>

#include "prefill.h"
#include "prefill_walk.cuh"
#include "sm103.cuh"

namespace attn {
namespace pf {

constexpr float RESCALE_LOG2_THRESHOLD = 8.0f;
constexpr float P_PARTIAL_LIMIT = 4294967296.0f;  // 2^32: bound on a thread's share of a step's row sum

// One thread's softmax state for its rows a and b of the current tile.
struct SoftmaxRows {
  float m_a, m_b;  // raw-score maxima that O and l currently refer to
  float l_a, l_b;  // this thread's shares of the row sums
  __device__ __forceinline__ void reset() {
    m_a = m_b = -INFINITY;
    l_a = l_b = 0.f;
  }
};

// Key step j (global step gs) of tile t: S in TMEM (s_tmem, this warp's lanes) becomes P (bf16
// pairs in the first BN / 2 columns of the same buffer); O (o_tmem, this warp's lanes, D columns)
// is rescaled when the reference max moves.  qa / qb: positions of rows a and b among the keys;
// cq: this thread's first column in each group of 8.  The caller has waited for S and, after this
// returns, signals that P is ready.  A wait that runs out of time clears `ok`.
template <int BN, int D, int NSB>
__device__ __forceinline__ void softmax_step(const PrefillParams& p, const WorkTile& t, int j, int gs,
                                             uint32_t s_tmem, uint32_t o_tmem, int qa, int qb, int cq, float c2,
                                             uint64_t c2x2, uint64_t* pv_done, SoftmaxRows& st, bool& ok) {
  constexpr int NG = BN / 8;  // 8-column groups per S tile
  const int lane_row0 = (threadIdx.x & 31) & ~3;
  uint32_t sr[4 * NG];
  tmem_ld16_256b<NG>(s_tmem, sr);
  tmem_ld_wait();
  // last visible column of each row in this tile: below BN - 1 only where the tile crosses
  // the causal diagonal or the end of the sequence
  const int key0 = j * BN;
  int lim_a = t.kv_len - 1 - key0, lim_b = lim_a;
  if (p.causal) {
    lim_a = min(lim_a, qa - key0);
    lim_b = min(lim_b, qb - key0);
  }
  // 64-key steps (d = 256) skip the groups of 8 columns past the last visible column of every row
  // of this warp: their weights are 0 without masking or exponentials.  (With 128-key steps the
  // extra test measured slower, so those steps mask every column.)
  constexpr bool SKIP = (BN == 64);
  const int lim_w = SKIP ? __reduce_max_sync(0xffffffffu, max(lim_a, lim_b)) : BN - 1;
  if (min(lim_a, lim_b) < BN - 1) {
#pragma unroll
    for (int i = 0; i < NG; ++i) {
      if (SKIP && 8 * i > lim_w) continue;
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int c = 8 * i + cq + e;
        if (c > lim_a) sr[4 * i + e] = __float_as_uint(-INFINITY);
        if (c > lim_b) sr[4 * i + 2 + e] = __float_as_uint(-INFINITY);
      }
    }
  }
  float alpha_a = 1.f, alpha_b = 1.f;
  bool rescale_o = false;
  uint32_t pk[2 * NG];
  float ps_a = 0.f, ps_b = 0.f;  // this step's shares of the two row sums
  if (j == 0) {
    // first key tile: key 0 is visible to every row, so its score is a finite reference (the thread
    // holding column 0 of the row shares it); a later overflow check falls back to the row max
    st.m_a = __shfl_sync(0xffffffffu, __uint_as_float(sr[0]), lane_row0);
    st.m_b = __shfl_sync(0xffffffffu, __uint_as_float(sr[2]), lane_row0);
  }
  const bool need_max = __any_sync(0xffffffffu, !(st.m_a > -INFINITY) || !(st.m_b > -INFINITY));
  for (int pass = need_max ? 1 : 0; pass < 2; ++pass) {
    if (pass == 1) {
      float mxa = -INFINITY, mxb = -INFINITY;
#pragma unroll
      for (int i = 0; i < NG; ++i) {
        if (SKIP && 8 * i > lim_w) continue;
        mxa = fmax3(mxa, __uint_as_float(sr[4 * i]), __uint_as_float(sr[4 * i + 1]));
        mxb = fmax3(mxb, __uint_as_float(sr[4 * i + 2]), __uint_as_float(sr[4 * i + 3]));
      }
      mxa = fmaxf(mxa, __shfl_xor_sync(0xffffffffu, mxa, 1));
      mxb = fmaxf(mxb, __shfl_xor_sync(0xffffffffu, mxb, 1));
      mxa = fmaxf(mxa, __shfl_xor_sync(0xffffffffu, mxa, 2));
      mxb = fmaxf(mxb, __shfl_xor_sync(0xffffffffu, mxb, 2));
      if (j == 0 || !(st.m_a > -INFINITY)) {  // step 0 has no O or l of this tile yet: nothing to rescale
        st.m_a = mxa;
      } else if ((mxa - st.m_a) * c2 > RESCALE_LOG2_THRESHOLD) {
        alpha_a = ex2_approx((st.m_a - mxa) * c2);
        st.l_a *= alpha_a;
        st.m_a = mxa;
        rescale_o = true;
      }
      if (j == 0 || !(st.m_b > -INFINITY)) {
        st.m_b = mxb;
      } else if ((mxb - st.m_b) * c2 > RESCALE_LOG2_THRESHOLD) {
        alpha_b = ex2_approx((st.m_b - mxb) * c2);
        st.l_b *= alpha_b;
        st.m_b = mxb;
        rescale_o = true;
      }
    }
    const float mba = (st.m_a == -INFINITY) ? 0.f : st.m_a * c2;
    const float mbb = (st.m_b == -INFINITY) ? 0.f : st.m_b * c2;
    const uint64_t nma = f2_pack(-mba, -mba), nmb = f2_pack(-mbb, -mbb);
    // p = 2^(s*scale*log2e - m*scale*log2e) in f32x2 pairs.  P (bf16, two per column) goes to
    // the first BN / 2 columns of this S buffer: the pair of columns 8i + cq, + 1 to column
    // 4i + cq/2, which is where the 16x128b shape puts this thread's registers 2i (row a) and
    // 2i + 1 (row b).
    uint64_t acc_a = 0ull, acc_b = 0ull;
#pragma unroll
    for (int i = 0; i < NG; ++i) {
      if (SKIP && 8 * i > lim_w) {
        pk[2 * i] = pk[2 * i + 1] = 0u;
        continue;
      }
      float x0, x1;
      f2_unpack(f2_fma(f2_pack(__uint_as_float(sr[4 * i]), __uint_as_float(sr[4 * i + 1])), c2x2, nma), x0, x1);
      const float pa0 = ex2_approx(x0), pa1 = ex2_approx(x1);
      f2_unpack(f2_fma(f2_pack(__uint_as_float(sr[4 * i + 2]), __uint_as_float(sr[4 * i + 3])), c2x2, nmb), x0,
                x1);
      const float pb0 = ex2_approx(x0), pb1 = ex2_approx(x1);
      acc_a = f2_add(acc_a, f2_pack(pa0, pa1));
      acc_b = f2_add(acc_b, f2_pack(pb0, pb1));
      pk[2 * i] = pack_bf16x2(pa0, pa1);
      pk[2 * i + 1] = pack_bf16x2(pb0, pb1);
    }
    float a0, a1, b0, b1;
    f2_unpack(acc_a, a0, a1);
    f2_unpack(acc_b, b0, b1);
    ps_a = a0 + a1;
    ps_b = b0 + b1;
    if (pass == 1 || !__any_sync(0xffffffffu, !(ps_a <= P_PARTIAL_LIMIT) || !(ps_b <= P_PARTIAL_LIMIT))) break;
  }
  st.l_a += ps_a;
  st.l_b += ps_b;
  tmem_st16_128b<NG>(s_tmem, pk);
  if (__any_sync(0xffffffffu, rescale_o)) {
    // O must hold P V of the previous step before it is rescaled
    if (ok) ok = __all_sync(0xffffffffu, mbar_wait(&pv_done[(gs - 1) % NSB], ((gs - 1) / NSB) & 1));
    tc_fence_after();
#pragma unroll 1
    for (int c64 = 0; c64 < D; c64 += 64) {
      uint32_t r[32];
      tmem_ld16_256b_x8(o_tmem + c64, r);
      tmem_ld_wait();
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        r[4 * i] = __float_as_uint(__uint_as_float(r[4 * i]) * alpha_a);
        r[4 * i + 1] = __float_as_uint(__uint_as_float(r[4 * i + 1]) * alpha_a);
        r[4 * i + 2] = __float_as_uint(__uint_as_float(r[4 * i + 2]) * alpha_b);
        r[4 * i + 3] = __float_as_uint(__uint_as_float(r[4 * i + 3]) * alpha_b);
      }
      tmem_st16_256b_x8(o_tmem + c64, r);
    }
  }
  tmem_st_wait();
  tc_fence_before();
  __syncwarp();
}

// End of tile k: add the four threads' shares of each row sum and hand l and the row max of rows
// ra and ra + 8 to the epilogue warps (two buffers in xl, [2][l, m][128]), which write LSE and
// divide O by l; the softmax warps go straight on.
__device__ __forceinline__ void softmax_tile_end(int k, int ra, int lane, SoftmaxRows& st, uint64_t* l_empty,
                                                 uint64_t* l_full, float* xl, bool& ok) {
  st.l_a += __shfl_xor_sync(0xffffffffu, st.l_a, 1);
  st.l_b += __shfl_xor_sync(0xffffffffu, st.l_b, 1);
  st.l_a += __shfl_xor_sync(0xffffffffu, st.l_a, 2);
  st.l_b += __shfl_xor_sync(0xffffffffu, st.l_b, 2);
  const int tb = k & 1;
  if (ok) ok = __all_sync(0xffffffffu, mbar_wait(&l_empty[tb], ((k >> 1) & 1) ^ 1));
  float* xt = xl + tb * 2 * 128;
  if ((lane & 3) == 0) {
    xt[ra] = st.l_a;
    xt[ra + 8] = st.l_b;
    xt[128 + ra] = st.m_a;
    xt[128 + ra + 8] = st.m_b;
  }
  __syncwarp();
  if (lane == 0) mbar_arrive(&l_full[tb]);
}

// Epilogue of tile t, the k-th tile of this CTA, by the 128 epilogue threads, one per row
// ("Streaming process -- How the SM works inside a transformer", Step 8): wait for the tile's row
// sums and maxima and write LSE = m * scale + ln l; wait for the tile's last P.V, read O out of TMEM
// (o_row: this thread's lane, D columns) in groups of OGRP columns as bf16 pairs after the division
// by l, and call release_o() once all of O has been read; then store 64-column panels through the
// staging buffer sO with TMA.  The last tile of a packed sequence that ends inside it is written
// row by row instead, so that the rows of the next sequence are left alone.
template <int D, int OGRP, class ReleaseO>
__device__ __forceinline__ void epilogue_tile(const PrefillParams& p, const WorkTile& t, int k, int row, int et,
                                              int lane, uint32_t o_row, const float* xl, uint64_t* l_full,
                                              uint64_t* l_empty, uint64_t* o_full, uint8_t* sO,
                                              const CUtensorMap* tm_o, ReleaseO release_o, bool& ok) {
  const int tb = k & 1;
  if (ok) ok = __all_sync(0xffffffffu, mbar_wait(&l_full[tb], (k >> 1) & 1));
  const float* xt = xl + tb * 2 * 128;
  const float l = xt[row];
  const float m_row = xt[128 + row];
  __syncwarp();
  if (lane == 0) mbar_arrive(&l_empty[tb]);
  const float inv_l = 1.f / l;
  const uint64_t il2 = f2_pack(inv_l, inv_l);
  if (p.lse != nullptr && t.qt * BM + row < t.len)
    p.lse[(static_cast<size_t>(t.z) * p.Hq + t.hq) * p.S + t.base + t.qt * BM + row] = m_row * p.scale + logf(l);
  if (ok) ok = __all_sync(0xffffffffu, mbar_wait(o_full, k & 1));
  tc_fence_after();
  const bool rowwise = p.cu_seqlens != nullptr && t.qt * BM + BM > t.len;
#pragma unroll 1
  for (int g0 = 0; g0 < D; g0 += OGRP) {
    uint32_t ob[OGRP / 2];
#pragma unroll
    for (int c4 = 0; c4 < OGRP / 32; ++c4) {
      uint32_t r[32];
      tmem_ld32(o_row + g0 + c4 * 32, r);
      tmem_ld_wait();
#pragma unroll
      for (int c = 0; c < 16; ++c) {
        float o0, o1;
        f2_unpack(f2_mul(f2_pack(__uint_as_float(r[2 * c]), __uint_as_float(r[2 * c + 1])), il2), o0, o1);
        ob[c4 * 16 + c] = pack_bf16x2(o0, o1);
      }
    }
    if (g0 + OGRP == D) {
      tc_fence_before();
      __syncwarp();
      release_o();  // the next tile's first P.V may overwrite O
    }
    if (rowwise) {
      if (t.qt * BM + row < t.len) {
        uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.o) +
                                              (static_cast<size_t>(t.base + t.qt * BM + row) * p.Hq + t.hq) * D + g0);
#pragma unroll
        for (int u = 0; u < OGRP / 8; ++u) dst[u] = make_uint4(ob[4 * u], ob[4 * u + 1], ob[4 * u + 2], ob[4 * u + 3]);
      }
      continue;
    }
    uint8_t* line = sO + row * PANEL_ROW;
#pragma unroll
    for (int c = 0; c < OGRP / 64; ++c) {
      if (et == 0) tma_store_wait_read0();  // the previous panel's store has read the staging buffer
      named_barrier_sync(2, 128);
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const uint4 w =
            make_uint4(ob[32 * c + 4 * u], ob[32 * c + 4 * u + 1], ob[32 * c + 4 * u + 2], ob[32 * c + 4 * u + 3]);
        *reinterpret_cast<uint4*>(line + ((u ^ (row & 7)) << 4)) = w;
      }
      fence_proxy_async_smem();
      named_barrier_sync(2, 128);
      if (et == 0) {
        tma_store_3d(tm_o, sO, t.hq * D + g0 + c * 64, t.base + t.qt * BM, t.z);
        tma_store_commit();
      }
    }
  }
}

}  // namespace pf
}  // namespace attn
