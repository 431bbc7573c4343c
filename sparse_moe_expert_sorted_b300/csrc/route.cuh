// a1: router logits in the fixed fp32 order R, top-k by (logit desc, id asc),
// softmax weights.
//
// Pages: a small router selects a few experts per token, e.g. 6 of 256
// (banandre.com, "The 284B Model on a 32GB GPU Trick", section "Sparsity Is a
// Lie (But a Useful One)").
//
// Order R, which makes the logits (and so the ids) reproducible bit for bit:
//   - Lane j of a warp owns the 8-element chunks c = j, j + 32, j + 64, ...
//   - The lane adds its products in ascending element order.  Each product is
//     formed in fp32 (exact for bf16 * bf16) and each add rounds (mul and add
//     are kept separate, never contracted).
//   - The lanes then combine by a shuffle-xor butterfly over 16, 8, 4, 2, 1.
//   - The bias is added last.
#pragma once
#include "common.cuh"
#include "permute.cuh"

namespace ftmoe {

constexpr int kRouteWarps = 8;            // warps per CTA
constexpr int kSelectSmallT = 64;         // T up to this: the last CTA selects (no 2nd kernel)

struct RouteArgs {
  const uint16_t* x;
  const uint16_t* wr;
  const float* bias;
  int T, E, d, k, renorm;
  float* logits;        // [T][E] (caller's buffer or workspace)
  int32_t* ids;
  float* w;
  unsigned* counter;    // zero between calls
  // optional (layer call, small batches): the last CTA also sorts the pairs (ftmoe_permute's outputs)
  int32_t* perm_off;
  int32_t* perm_sp;
  int32_t* perm_pp;
};

// Packed pairs of fp32 values (low half = first) and the packed IEEE operations on them.
__device__ __forceinline__ uint64_t f32x2_pack(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void f32x2_unpack(uint64_t v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t f32x2_mul(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ uint64_t f32x2_add(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}

// Warp-level top-k of one token's E logits.  Lane r ends up holding rank r
// (value and id); the first k lanes write ids and weights.
__device__ __forceinline__ void select_token(const RouteArgs& a, int t, int lane) {
  constexpr int MAXJ = 32;  // E <= 1024: lane holds experts lane, lane + 32, ...
  constexpr int NONE = 0x7FFFFFFF;
  const int E = a.E;
  float v[MAXJ];
  const float* row = a.logits + size_t(t) * E;
#pragma unroll
  for (int j = 0; j < MAXJ; ++j) {
    const int e = j * 32 + lane;
    v[j] = (e < E) ? __ldcg(row + e) : -INFINITY;
  }
  uint32_t taken = 0;
  float my_v = -INFINITY;
  int my_i = NONE;
  for (int r = 0; r < a.k; ++r) {
    float bv = -INFINITY;
    int bi = NONE;
#pragma unroll
    for (int j = 0; j < MAXJ; ++j) {
      const int e = j * 32 + lane;
      const bool ok = (e < E) && !((taken >> j) & 1u);
      if (ok && (bi == NONE || v[j] > bv)) {  // ascending e: an equal value keeps the lower id
        bv = v[j];
        bi = e;
      }
    }
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) {
      const float ov = __shfl_xor_sync(0xFFFFFFFFu, bv, off);
      const int oi = __shfl_xor_sync(0xFFFFFFFFu, bi, off);
      if (oi != NONE && (bi == NONE || ov > bv || (ov == bv && oi < bi))) {
        bv = ov;
        bi = oi;
      }
    }
    if ((bi & 31) == lane) taken |= 1u << (bi >> 5);
    if (lane == r) {
      my_v = bv;
      my_i = bi;
    }
  }
  const float m = __shfl_sync(0xFFFFFFFFu, my_v, 0);  // rank 0 holds the largest logit
  float part = 0.f;
  if (a.renorm) {
    part = (lane < a.k) ? expf(my_v - m) : 0.f;
  } else {
#pragma unroll
    for (int j = 0; j < MAXJ; ++j)
      if (j * 32 + lane < E) part += expf(v[j] - m);
  }
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) part += __shfl_xor_sync(0xFFFFFFFFu, part, off);
  if (lane < a.k) {
    a.ids[size_t(t) * a.k + lane] = my_i;
    a.w[size_t(t) * a.k + lane] = expf(my_v - m) / part;
  }
}

// Each warp: EW experts x TW tokens of logits.  Grid-stride over items.
// The lane's chunks are loaded RB at a time before any is used, so RB loads per
// operand are in flight; they are still added in ascending chunk order.
template <int EW, int TW, int RB>
__global__ void __launch_bounds__(kRouteWarps * 32)
route_logits_kernel(RouteArgs a, int fused_select) {
  pdl_wait();
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int n_eg = (a.E + EW - 1) / EW;
  const int n_tt = (a.T + TW - 1) / TW;
  const int n_items = n_eg * n_tt;
  const int S = a.d >> 8;  // chunks per lane
  for (int item = blockIdx.x * kRouteWarps + warp; item < n_items; item += gridDim.x * kRouteWarps) {
    const int eg = item % n_eg;
    const int tt = item / n_eg;
    const int e0 = eg * EW, t0 = tt * TW;
    float acc[EW][TW];
#pragma unroll
    for (int i = 0; i < EW; ++i)
#pragma unroll
      for (int j = 0; j < TW; ++j) acc[i][j] = 0.f;
    // Even TW: two tokens' accumulators share one packed f32x2 register, so one packed multiply
    // and one packed add (each two independent IEEE fp32 operations, round to nearest) do the
    // work of two; every accumulator still sees its products in the same order.
    constexpr int TP = (TW % 2 == 0) ? TW / 2 : 1;
    uint64_t acc2[EW][TP];
#pragma unroll
    for (int i = 0; i < EW; ++i)
#pragma unroll
      for (int q = 0; q < TP; ++q) acc2[i][q] = 0ull;
    for (int s0 = 0; s0 < S; s0 += RB) {
      uint4 wv[RB][EW], xv[RB][TW];
#pragma unroll
      for (int b = 0; b < RB; ++b) {
        const int c = min(s0 + b, S - 1) * 32 + lane;
#pragma unroll
        for (int i = 0; i < EW; ++i) {
          int e = min(e0 + i, a.E - 1);
          wv[b][i] = __ldg(reinterpret_cast<const uint4*>(a.wr + size_t(e) * a.d) + c);
        }
#pragma unroll
        for (int j = 0; j < TW; ++j) {
          int t = min(t0 + j, a.T - 1);
          xv[b][j] = __ldg(reinterpret_cast<const uint4*>(a.x + size_t(t) * a.d) + c);
        }
      }
#pragma unroll
      for (int b = 0; b < RB; ++b) {
        if (s0 + b < S) {
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            if constexpr (TW % 2 == 0) {
              uint64_t xp[TP];
#pragma unroll
              for (int q = 0; q < TP; ++q) {
                const uint32_t x0 = (&xv[b][2 * q].x)[u >> 1], x1 = (&xv[b][2 * q + 1].x)[u >> 1];
                xp[q] = f32x2_pack((u & 1) ? bf16_hi(x0) : bf16_lo(x0), (u & 1) ? bf16_hi(x1) : bf16_lo(x1));
              }
#pragma unroll
              for (int i = 0; i < EW; ++i) {
                const uint32_t ww = (&wv[b][i].x)[u >> 1];
                const float wf = (u & 1) ? bf16_hi(ww) : bf16_lo(ww);
                const uint64_t w2 = f32x2_pack(wf, wf);
#pragma unroll
                for (int q = 0; q < TP; ++q) acc2[i][q] = f32x2_add(acc2[i][q], f32x2_mul(xp[q], w2));
              }
            } else {
#pragma unroll
              for (int i = 0; i < EW; ++i) {
                const uint32_t ww = (&wv[b][i].x)[u >> 1];
                const float wf = (u & 1) ? bf16_hi(ww) : bf16_lo(ww);
#pragma unroll
                for (int j = 0; j < TW; ++j) {
                  const uint32_t xx = (&xv[b][j].x)[u >> 1];
                  const float xf = (u & 1) ? bf16_hi(xx) : bf16_lo(xx);
                  acc[i][j] = __fadd_rn(acc[i][j], __fmul_rn(xf, wf));
                }
              }
            }
          }
        }
      }
    }
    if constexpr (TW % 2 == 0) {
#pragma unroll
      for (int i = 0; i < EW; ++i)
#pragma unroll
        for (int q = 0; q < TP; ++q) f32x2_unpack(acc2[i][q], acc[i][2 * q], acc[i][2 * q + 1]);
    }
#pragma unroll
    for (int i = 0; i < EW; ++i)
#pragma unroll
      for (int j = 0; j < TW; ++j) {
        float v = acc[i][j];
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) v = __fadd_rn(v, __shfl_xor_sync(0xFFFFFFFFu, v, off));
        acc[i][j] = v;
      }
    if (lane == 0) {
#pragma unroll
      for (int i = 0; i < EW; ++i)
#pragma unroll
        for (int j = 0; j < TW; ++j) {
          const int e = e0 + i, t = t0 + j;
          if (e < a.E && t < a.T) {
            float v = acc[i][j];
            if (a.bias) v = __fadd_rn(v, a.bias[e]);
            a.logits[size_t(t) * a.E + e] = v;
          }
        }
    }
  }
  if (!fused_select) return;
  // Last CTA to finish selects for every token (small T only).
  __shared__ unsigned s_last;
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) {
    unsigned prev = atomicAdd(a.counter, 1u);
    s_last = (prev == gridDim.x - 1);
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  for (int t = warp; t < a.T; t += kRouteWarps) select_token(a, t, lane);
  if (threadIdx.x == 0) *a.counter = 0u;  // leave the counter zero for the next call
  if (a.perm_off) {
    extern __shared__ int s_perm[];
    __syncthreads();
    permute_block(a.ids, a.T * a.k, a.E, a.perm_off, a.perm_sp, a.perm_pp, s_perm);
  }
}

__global__ void __launch_bounds__(kRouteWarps * 32) route_select_kernel(RouteArgs a) {
  pdl_wait();
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  for (int t = blockIdx.x * kRouteWarps + warp; t < a.T; t += gridDim.x * kRouteWarps) select_token(a, t, lane);
}

}  // namespace ftmoe
