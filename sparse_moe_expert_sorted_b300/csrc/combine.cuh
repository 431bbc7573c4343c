// a5: weighted combine and exact merge.
//
// Pages: the partial sums over a split of the selected experts add up to the
// full output, with no approximation, once the layer completes (banandre.com, "The 284B Model on a 32GB GPU
// Trick", section "The q* Policy: Math Instead of Guesses").
//
//   out[t][n] = partial_b[t][n] + sum over resident ranks r (ascending) of w[t][r] * y[pair_pos[t*k+r]][n]
//
// One thread handles four consecutive columns, so loads and stores are 128-bit.
#pragma once
#include "common.cuh"

namespace ftmoe {

struct CombineArgs {
  int T, k, d, E;
  int C;                     // slots of the arena: an entry >= C was skipped by the FFN (not resident)
  const float* y;
  const int32_t* pair_pos;
  const float* topk_w;
  const int32_t* topk_ids;
  const int32_t* slot_of;
  const float* partial_b;
  float* out_f32;
  uint16_t* out_bf16;
};

__global__ void __launch_bounds__(256) combine_kernel(CombineArgs a) {
  pdl_wait();
  const int q = a.d / 4;
  // the bf16 cast of an out that already holds the sum (no y, partial_b == out_f32): out_f32
  // is only read
  float* out_f32 = (a.y == nullptr && a.out_f32 == a.partial_b) ? nullptr : a.out_f32;
  const long long total = (long long)a.T * q;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < total;
       i += (long long)gridDim.x * blockDim.x) {
    const int t = int(i / q), c4 = int(i % q);
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    if (a.partial_b) acc = reinterpret_cast<const float4*>(a.partial_b + size_t(t) * a.d)[c4];
    if (a.y) {
      for (int r = 0; r < a.k; ++r) {
        const int p = t * a.k + r;
        if (a.slot_of) {
          int e = a.topk_ids[p];
          if (e < 0 || e >= a.E) {
            set_dev_err(DEV_ERR_BAD_ID);
            continue;
          }
          const int slot = a.slot_of[e];
          if (slot < 0 || slot >= a.C) continue;
        }
        const float w = a.topk_w[p];
        const float4 v = reinterpret_cast<const float4*>(a.y + size_t(a.pair_pos[p]) * a.d)[c4];
        acc.x = fmaf(w, v.x, acc.x);
        acc.y = fmaf(w, v.y, acc.y);
        acc.z = fmaf(w, v.z, acc.z);
        acc.w = fmaf(w, v.w, acc.w);
      }
    }
    if (out_f32) reinterpret_cast<float4*>(out_f32 + size_t(t) * a.d)[c4] = acc;
    if (a.out_bf16) {
      __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x, acc.y);
      __nv_bfloat162 hi = __floats2bfloat162_rn(acc.z, acc.w);
      uint2 pk;
      pk.x = *reinterpret_cast<uint32_t*>(&lo);
      pk.y = *reinterpret_cast<uint32_t*>(&hi);
      reinterpret_cast<uint2*>(a.out_bf16 + size_t(t) * a.d)[c4] = pk;
    }
  }
}

}  // namespace ftmoe
