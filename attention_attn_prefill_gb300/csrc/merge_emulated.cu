// Merges of split-KV decode partials in the float32 operation order of other backends.
//
// "Why your local LLM feels dumber than it is" (Part 3.14), section "Backend
// names expand into four decode algorithms", describes how four decode
// backends combine their groups.  This kernel reproduces each combination
// step by step in float32, with every add, multiply and divide rounded on its
// own (no fused multiply-add) and every exp / log evaluated in double precision
// and rounded once to float32:
//   Triton   top = max m_i;  c_i = exp(m_i - top);  L += l_i c_i;  N += n_i c_i;  out = N / L
//   FA2      lse_i = m_i + log l_i;  top = max lse_i;  w_i = exp(lse_i - top);
//            W += w_i;  N += o_i w_i;  out = N / W
//   XQA      top = max m_i;  w_i = l_i exp(m_i - top);  W += w_i;  N += o_i w_i;  out = N / W
//   TRT      one group after another: M' = max(M, m_i);  a = exp(M - M') (0 before the first
//            group);  b = exp(m_i - M');  L = L a + l_i b;  N = N a + bf16(n_i) b;  out = N / L
// Groups are visited in slot order; slots with l_i <= 0 are empty and skipped.  The
// log-sum-exp the library also returns is the largest max (or log-sum) plus log of the
// merged sum, rounded the same way.
//
// One CTA per row: the per-slot factors of a chunk of slots are computed in parallel (the
// running maxima of the ordered merge by a warp-wide max scan) and kept in shared memory; then
// every thread runs the sequential accumulation for its own NC consecutive output components.
// The stored values reach the additions ahead of them, so that the loads overlap while the
// additions stay in slot order: either the next U slots are loaded into registers while the
// current U are added, or (d of 128 or 256) a ring of NST shared-memory stages of SB slots each is
// filled with 16-byte cp.async copies, NST - 1 stages ahead.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "decode.h"

namespace attn {
namespace {

constexpr int MT = 128;     // threads per row
constexpr int CHUNK = 256;  // slots whose factors are staged at once
constexpr int MAX_D = 1024;

__device__ __forceinline__ float exp_rn(float x) { return static_cast<float>(exp(static_cast<double>(x))); }
__device__ __forceinline__ float log_rn(float x) { return static_cast<float>(log(static_cast<double>(x))); }
__device__ __forceinline__ float bf16_rn(float x) { return __bfloat162float(__float2bfloat16_rn(x)); }

// FA2's group statistic: m + log l, each step rounded.
__device__ __forceinline__ float log_sum(float m, float l) { return __fadd_rn(m, log_rn(l)); }

__device__ __forceinline__ void cp_async16(void* smem_dst, const void* gmem_src) {
  const uint32_t dst = static_cast<uint32_t>(__cvta_generic_to_shared(smem_dst));
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(gmem_src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// NC: output components per thread (d <= MT * NC).  NST == 0: the next U slots' values are loaded
// into registers; NST > 0: a ring of NST stages of SB slots in dynamic shared memory (d == MT * NC,
// part_o 16-byte aligned).
template <int NC, int U, int NST, int SB>
__global__ void __launch_bounds__(MT) merge_emulated_kernel(const float* __restrict__ part_o,
                                                            const float* __restrict__ part_m,
                                                            const float* __restrict__ part_l, int splits, int d,
                                                            int mode, float* __restrict__ o32,
                                                            __nv_bfloat16* __restrict__ o, float* __restrict__ lse) {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  __shared__ float f_a[CHUNK], f_b[CHUNK], f_l[CHUNK], f_m[CHUNK];
  __shared__ float red[MT / 32];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const size_t row = blockIdx.x;
  const float* pm = part_m + row * splits;
  const float* pl = part_l + row * splits;
  const float* po = part_o + row * splits * static_cast<size_t>(d);

  // largest max (log-sum for FA2) over the non-empty groups; the ordered merge keeps a running one
  float top = -INFINITY;
  if (mode != kEmuTrt) {
    for (int i = tid; i < splits; i += MT) {
      const float l = pl[i];
      if (l > 0.f) top = fmaxf(top, mode == kEmuFa2 ? log_sum(pm[i], l) : pm[i]);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) top = fmaxf(top, __shfl_xor_sync(0xffffffffu, top, off));
    if (lane == 0) red[warp] = top;
    __syncthreads();
    top = fmaxf(fmaxf(red[0], red[1]), fmaxf(red[2], red[3]));
  }

  const int x0 = tid * NC;  // this thread's first output component
  float acc[NC];
#pragma unroll
  for (int c = 0; c < NC; ++c) acc[c] = 0.f;
  float wsum = 0.f;
  float run = -INFINITY;  // ordered merge: running max before the current chunk
  bool any = false;

  for (int base = 0; base < splits; base += CHUNK) {
    const int n = splits - base < CHUNK ? splits - base : CHUNK;
    // the chunk's group sums and maxima, loaded by all threads at once
    for (int j = tid; j < n; j += MT) {
      f_l[j] = pl[base + j];
      f_m[j] = pm[base + j];
    }
    __syncthreads();
    if (mode == kEmuTrt) {
      // warp 0: running max before (f_a) and after (f_b) each slot, by a max scan over the live slots
      if (warp == 0) {
        for (int j0 = 0; j0 < n; j0 += 32) {
          const int j = j0 + lane;
          const float l = j < n ? f_l[j] : 0.f;
          const float v = l > 0.f ? f_m[j] : -INFINITY;
          float incl = v;
#pragma unroll
          for (int off = 1; off < 32; off <<= 1) {
            const float t = __shfl_up_sync(0xffffffffu, incl, off);
            if (lane >= off) incl = fmaxf(incl, t);
          }
          incl = fmaxf(incl, run);
          float excl = __shfl_up_sync(0xffffffffu, incl, 1);
          if (lane == 0) excl = run;
          if (j < n) {
            f_a[j] = excl;
            f_b[j] = incl;
          }
          run = __shfl_sync(0xffffffffu, incl, 31);
        }
      }
      __syncthreads();
      for (int j = tid; j < n; j += MT) {
        const float l = f_l[j];
        if (!(l > 0.f)) continue;
        const float before = f_a[j], after = f_b[j];
        f_a[j] = before == -INFINITY ? 0.f : exp_rn(__fsub_rn(before, after));  // keeps the running state
        f_b[j] = exp_rn(__fsub_rn(f_m[j], after));                                // takes the new group
      }
    } else {
      for (int j = tid; j < n; j += MT) {
        const float l = f_l[j];
        if (!(l > 0.f)) continue;
        const float m = f_m[j];
        if (mode == kEmuFa2)
          f_a[j] = exp_rn(__fsub_rn(log_sum(m, l), top));
        else if (mode == kEmuXqa)
          f_a[j] = __fmul_rn(l, exp_rn(__fsub_rn(m, top)));
        else
          f_a[j] = exp_rn(__fsub_rn(m, top));
      }
    }
    __syncthreads();
    // the groups in slot order, each thread on its own components
    auto add = [&](int j, const float (&v)[NC]) {
      const float l = f_l[j];
      if (!(l > 0.f)) return;
      any = true;
      if (mode == kEmuTrt) {
        const float a = f_a[j], b = f_b[j];
        wsum = __fadd_rn(__fmul_rn(wsum, a), __fmul_rn(l, b));
#pragma unroll
        for (int c = 0; c < NC; ++c) acc[c] = __fadd_rn(__fmul_rn(acc[c], a), __fmul_rn(bf16_rn(v[c]), b));
      } else {
        const float w = f_a[j];
        wsum = __fadd_rn(wsum, mode == kEmuTriton ? __fmul_rn(l, w) : w);
#pragma unroll
        for (int c = 0; c < NC; ++c) acc[c] = __fadd_rn(acc[c], __fmul_rn(v[c], w));
      }
    };
    if constexpr (NST == 0) {
      // the values of the next U slots are loaded while the current U are added
      auto load_batch = [&](float (&v)[U][NC], int j0) {
#pragma unroll
        for (int u = 0; u < U; ++u) {
          // indices clamped into the row, so that every load is in bounds; the value is dropped there
          const int j = j0 + u < n ? j0 + u : n - 1;
          const float* src = po + static_cast<size_t>(base + j) * d;
#pragma unroll
          for (int c = 0; c < NC; ++c) {
            const int x = x0 + c < d ? x0 + c : d - 1;
            v[u][c] = (j0 + u < n && x0 + c < d) ? src[x] : 0.f;
          }
        }
      };
      float cur[U][NC], nxt[U][NC];
      load_batch(cur, 0);
      for (int j0 = 0; j0 < n; j0 += U) {
        if (j0 + U < n) load_batch(nxt, j0 + U);
#pragma unroll
        for (int u = 0; u < U; ++u)
          if (j0 + u < n) add(j0 + u, cur[u]);
#pragma unroll
        for (int u = 0; u < U; ++u)
#pragma unroll
          for (int c = 0; c < NC; ++c) cur[u][c] = nxt[u][c];
      }
    } else {
      // stage t holds slots t * SB .. of this chunk in buffer t % NST; NST - 1 stages are in flight
      extern __shared__ float4 ring4[];
      float* ring = reinterpret_cast<float*>(ring4);
      constexpr int D = MT * NC;
      const int nst = (n + SB - 1) / SB;
      auto issue = [&](int t) {
        const int j0 = t * SB;
        const int cnt = n - j0 < SB ? n - j0 : SB;
        const float* src = po + static_cast<size_t>(base + j0) * D;
        float* dst = ring + (t % NST) * (SB * D);
        for (int q = tid; q < cnt * (D / 4); q += MT) cp_async16(dst + 4 * q, src + 4 * q);
      };
#pragma unroll
      for (int t = 0; t < NST - 1; ++t) {
        if (t < nst) issue(t);
        cp_async_commit();
      }
      for (int t = 0; t < nst; ++t) {
        cp_async_wait<NST - 2>();  // this thread's copies of stage t have landed ...
        __syncthreads();           // ... and everyone's
        const float* buf = ring + (t % NST) * (SB * D) + x0;
        const int j0 = t * SB;
        const int cnt = n - j0 < SB ? n - j0 : SB;
        for (int u = 0; u < cnt; ++u) {  // (measured: unrolling this loop makes it slower)
          float v[NC];
#pragma unroll
          for (int c = 0; c < NC; ++c) v[c] = buf[u * D + c];
          add(j0 + u, v);
        }
        __syncthreads();  // buffer t % NST is free again
        if (t + NST - 1 < nst) issue(t + NST - 1);
        cp_async_commit();  // an empty group past the end keeps the count uniform
      }
      cp_async_wait<0>();
    }
    __syncthreads();
  }
  if (mode == kEmuTrt) top = run;

#pragma unroll
  for (int c = 0; c < NC; ++c) {
    const int x = x0 + c;
    if (x >= d) continue;
    const float out = any ? __fdiv_rn(acc[c], wsum) : 0.f;
    if (o32 != nullptr) o32[row * d + x] = out;
    if (o != nullptr) o[row * d + x] = __float2bfloat16_rn(out);
  }
  if (lse != nullptr && tid == 0) lse[row] = any ? __fadd_rn(top, log_rn(wsum)) : -INFINITY;
}

}  // namespace

cudaError_t merge_emulated_launch(int numerics, const float* part_o, const float* part_m, const float* part_l,
                                  int rows, int splits, int d, float* o32, void* o, float* lse, cudaStream_t stream) {
  if (numerics < kEmuTriton || numerics > kEmuTrt || rows < 1 || splits < 1 || d < 1 || d > MAX_D)
    return cudaErrorInvalidValue;
  using Kern = void (*)(const float*, const float*, const float*, int, int, int, float*, __nv_bfloat16*, float*);
  Kern kern = merge_emulated_kernel<8, 8, 0, 0>;
  if (d <= MT)
    kern = merge_emulated_kernel<1, 16, 0, 0>;
  else if (d <= 2 * MT)
    kern = merge_emulated_kernel<2, 32, 0, 0>;
  else if (d <= 4 * MT)
    kern = merge_emulated_kernel<4, 16, 0, 0>;
  // staged loads for rows of many groups at the head dims of the decode kernels, when the stored values
  // are 16-byte aligned (with fewer groups, a row has too little to pipeline and the ring's shared
  // memory only leaves fewer rows in flight)
  int smem = 0;
  if ((d == 128 || d == 256) && splits >= 96 && (reinterpret_cast<uintptr_t>(part_o) & 15u) == 0) {
    constexpr int NST = 6, SB = 16;
    smem = NST * SB * d * static_cast<int>(sizeof(float));
    kern = d == 128 ? merge_emulated_kernel<1, 1, NST, SB> : merge_emulated_kernel<2, 1, NST, SB>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
  }
  // programmatic dependent launch: the partials may come from the kernel just before it
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(rows);
  cfg.blockDim = dim3(MT);
  cfg.dynamicSmemBytes = static_cast<size_t>(smem);
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, part_o, part_m, part_l, splits, d, numerics, o32,
                            static_cast<__nv_bfloat16*>(o), lse);
}

}  // namespace attn
