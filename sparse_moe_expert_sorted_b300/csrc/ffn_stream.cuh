// a4 (+a5): grouped SwiGLU expert FFN on CUDA cores, streaming the packed weights.
//
// Pages: each routed expert is a small feed-forward network (banandre.com,
// "The 284B Model on a 32GB GPU Trick", section "Sparsity Is a Lie").  Resident
// experts are read from GPU expert slots (zubnet.ai, "FreeToken, Unsloth GGUF
// ... consumer hardware").
//
// With few tokens per expert, a layer is a stream of the selected experts'
// packed weights through the SMs.  The weights are used directly, with no
// activation quantisation; it is bound by HBM bandwidth.
//
// Work items are (expert, token tile of kTokTile rows, output row).  Each
// warp takes a contiguous range of items, so consecutive items read
// consecutive weight rows.  Inside an item, lane l reads every 32nd unit of
// the row (64 elements for gate/up, 32 for down) with 128-bit streaming
// loads.  It decodes the codes to fp32 with their block scale and
// accumulates fp32 dot products for the tile's tokens.  A warp butterfly
// finishes the dot products.
//
//   kernel 1 (gate/up): h[j][:] = silu(g) * u for every sorted row j.  h is fp32 [P][f] in the workspace.
//   kernel 2 (down):    y[j][n] = sum_i h[j][i] W_d[n][i].  It writes y (sorted rows), or
//                       adds w_p * y into out[t][n] (the fused combine).
#pragma once
#include "common.cuh"
#include "permute.cuh"

namespace ftmoe {

constexpr int kFfnWarps = 8;
constexpr int kTokTile = 8;

struct FfnArgs {
  int E, k, d, f, C;
  const uint8_t* gate;
  const uint8_t* up;
  const uint8_t* down;
  const uint8_t* gate_s;
  const uint8_t* up_s;
  const uint8_t* down_s;
  const float* tscale;     // NVFP4 [C][3], else nullptr
  const int32_t* slot_of;  // [E] or nullptr (slot e)
  const uint16_t* x;       // [T][d]
  int T;
  const int32_t* offsets;
  const int32_t* sorted_pair;
  const float* topk_w;     // nullptr: write y; else add w*y into out
  float* y_or_out;
  float* h;                // [P][f]
  // layer call only (decode kernel): zero y_or_out (the fused-combine accumulator) before any
  // add, and afterwards write its bf16 copy here (nullptr = neither)
  uint16_t* out_bf16;
  const uint8_t* prep_dec;  // prepared decode layout of the arena (NVFP4 / MXFP4), or nullptr
};

template <int FMT>
struct FmtTraits {
  static constexpr int kBits = FMT == FTMOE_BF16 ? 16 : (FMT == FTMOE_FP8_B128 ? 8 : 4);
  static __host__ __device__ size_t row_bytes(int K) { return size_t(K) * kBits / 8; }
  // scale bytes of one [N][K] matrix (FP8: floats)
  static __host__ __device__ size_t scale_bytes(int N, int K) {
    if (FMT == FTMOE_NVFP4) return size_t(N) * (K / 16);
    if (FMT == FTMOE_MXFP4) return size_t(N) * (K / 32);
    if (FMT == FTMOE_FP8_B128) return size_t(N / 128) * (K / 128) * sizeof(float);
    return 0;
  }
};

// U consecutive elements (a "unit") of one weight row, raw then decoded by 16s.
template <int FMT, int U>
struct Unit {
  static constexpr int kBits = FmtTraits<FMT>::kBits;
  static constexpr int kWords = U * kBits / 32;
  uint32_t w[kWords];
  uint32_t sc;  // FP4 block-scale bytes of this unit
  float sf;     // FP8 block scale

  // row: codes of the row; srow: FP4 scale row; fp8_srow: FP8 scale row (block row n/128)
  __device__ __forceinline__ void load(const uint8_t* row, const uint8_t* srow, const float* fp8_srow, int u) {
    const uint8_t* p = row + size_t(u) * (U * kBits / 8);
#pragma unroll
    for (int i = 0; i < kWords / 4; ++i) {
      uint4 v = ld_stream16(p + 16 * i);
      w[4 * i + 0] = v.x;
      w[4 * i + 1] = v.y;
      w[4 * i + 2] = v.z;
      w[4 * i + 3] = v.w;
    }
    if (FMT == FTMOE_NVFP4) {
      sc = (U == 64) ? __ldg(reinterpret_cast<const uint32_t*>(srow) + u)
                     : __ldg(reinterpret_cast<const uint16_t*>(srow) + u);
    } else if (FMT == FTMOE_MXFP4) {
      sc = (U == 64) ? __ldg(reinterpret_cast<const uint16_t*>(srow) + u) : __ldg(srow + u);
    } else if (FMT == FTMOE_FP8_B128) {
      sf = __ldg(fp8_srow + (U * u) / 128);
    }
  }

  // elements [16q, 16q + 16) of the unit, scale applied
  __device__ __forceinline__ void decode16(int q, float out[16]) const {
    if (FMT == FTMOE_NVFP4 || FMT == FTMOE_MXFP4) {
      const float s = (FMT == FTMOE_NVFP4) ? e4m3_to_float((sc >> (8 * q)) & 0xFFu)
                                           : e8m0_to_float((sc >> (8 * (q >> 1))) & 0xFFu);
#pragma unroll
      for (int hw = 0; hw < 2; ++hw) {
        uint32_t hh[4];
        e2m1x8_to_f16x8(w[2 * q + hw], hh);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          float2 f2 = f16x2_to_float2(hh[i]);
          out[8 * hw + 2 * i] = f2.x * s;
          out[8 * hw + 2 * i + 1] = f2.y * s;
        }
      }
    } else if (FMT == FTMOE_FP8_B128) {
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint32_t v = w[4 * q + i];
        float2 a = e4m3x2_to_float2(uint16_t(v & 0xFFFFu));
        float2 b = e4m3x2_to_float2(uint16_t(v >> 16));
        out[4 * i + 0] = a.x * sf;
        out[4 * i + 1] = a.y * sf;
        out[4 * i + 2] = b.x * sf;
        out[4 * i + 3] = b.y * sf;
      }
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        out[2 * i] = bf16_lo(w[8 * q + i]);
        out[2 * i + 1] = bf16_hi(w[8 * q + i]);
      }
    }
  }
};

// s_start[e] = first item of expert e (exclusive scan); s_start[E] = total items.
__device__ __forceinline__ int build_item_starts(const FfnArgs& a, int rows, int* s_start, int* s_warp_tot) {
  for (int e = threadIdx.x; e < a.E; e += blockDim.x) {
    const int n = a.offsets[e + 1] - a.offsets[e];
    int slot = a.slot_of ? a.slot_of[e] : e;
    if (slot >= a.C) {
      if (n > 0) set_dev_err(DEV_ERR_BAD_SLOT);
      slot = -1;
    }
    s_start[e] = (n > 0 && slot >= 0) ? ((n + kTokTile - 1) / kTokTile) * rows : 0;
  }
  __syncthreads();
  const int total = block_exclusive_scan(s_start, a.E, s_warp_tot);
  if (threadIdx.x == 0) s_start[a.E] = total;
  __syncthreads();
  return total;
}

__device__ __forceinline__ int find_expert(const int* s_start, int E, int item) {
  int lo = 0, hi = E - 1;  // largest e with s_start[e] <= item
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (s_start[mid] <= item) lo = mid; else hi = mid - 1;
  }
  return lo;
}

template <int FMT>
__global__ void __launch_bounds__(kFfnWarps * 32) ffn_gate_up_kernel(FfnArgs a) {
  __shared__ int s_start[1025];
  __shared__ int s_warp_tot[33];
  pdl_wait();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int total = build_item_starts(a, a.f, s_start, s_warp_tot);
  const long long G = (long long)gridDim.x * kFfnWarps;
  const long long g = (long long)blockIdx.x * kFfnWarps + warp;
  const int i0 = int(g * total / G), i1 = int((g + 1) * total / G);
  using Tr = FmtTraits<FMT>;
  const size_t rb = Tr::row_bytes(a.d);
  const size_t mat_bytes = rb * a.f;
  const size_t smat = Tr::scale_bytes(a.f, a.d);
  const int units = a.d / 64;
  int e = i0 < i1 ? find_expert(s_start, a.E, i0) : 0;
  for (int item = i0; item < i1; ++item) {
    while (item >= s_start[e + 1]) ++e;
    const int local = item - s_start[e];
    const int tile = local / a.f, row = local % a.f;
    const int slot = a.slot_of ? a.slot_of[e] : e;
    const int n0 = a.offsets[e] + tile * kTokTile;
    const int nt = min(kTokTile, a.offsets[e + 1] - n0);
    int tok[kTokTile];
#pragma unroll
    for (int j = 0; j < kTokTile; ++j) tok[j] = (j < nt) ? a.sorted_pair[n0 + j] / a.k : 0;
    const uint8_t* grow = a.gate + slot * mat_bytes + row * rb;
    const uint8_t* urow = a.up + slot * mat_bytes + row * rb;
    const uint8_t* gsrow = nullptr;
    const uint8_t* usrow = nullptr;
    const float* gfrow = nullptr;
    const float* ufrow = nullptr;
    if (FMT == FTMOE_NVFP4 || FMT == FTMOE_MXFP4) {
      const size_t sr = (FMT == FTMOE_NVFP4) ? a.d / 16 : a.d / 32;
      gsrow = a.gate_s + slot * smat + row * sr;
      usrow = a.up_s + slot * smat + row * sr;
    } else if (FMT == FTMOE_FP8_B128) {
      const size_t nkb = a.d / 128;
      gfrow = reinterpret_cast<const float*>(a.gate_s + slot * smat) + (row / 128) * nkb;
      ufrow = reinterpret_cast<const float*>(a.up_s + slot * smat) + (row / 128) * nkb;
    }
    float ag[kTokTile], au[kTokTile];
#pragma unroll
    for (int j = 0; j < kTokTile; ++j) ag[j] = au[j] = 0.f;
    for (int u = lane; u < units; u += 32) {
      Unit<FMT, 64> gu, uu;
      gu.load(grow, gsrow, gfrow, u);
      uu.load(urow, usrow, ufrow, u);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        float wg[16], wu[16];
        gu.decode16(q, wg);
        uu.decode16(q, wu);
#pragma unroll
        for (int j = 0; j < kTokTile; ++j) {
          if (j < nt) {
            const uint4* xp = reinterpret_cast<const uint4*>(a.x + size_t(tok[j]) * a.d + 64 * u + 16 * q);
            const uint4 x0 = __ldg(xp), x1 = __ldg(xp + 1);
            const uint32_t xw[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
            float sg = 0.f, su = 0.f;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const float xa = bf16_lo(xw[i]), xb = bf16_hi(xw[i]);
              sg = fmaf(wg[2 * i], xa, sg);
              sg = fmaf(wg[2 * i + 1], xb, sg);
              su = fmaf(wu[2 * i], xa, su);
              su = fmaf(wu[2 * i + 1], xb, su);
            }
            ag[j] += sg;
            au[j] += su;
          }
        }
      }
    }
    const float tsg = a.tscale ? a.tscale[slot * 3 + 0] : 1.f;
    const float tsu = a.tscale ? a.tscale[slot * 3 + 1] : 1.f;
#pragma unroll
    for (int j = 0; j < kTokTile; ++j) {
      if (j < nt) {
        float vg = ag[j], vu = au[j];
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) {
          vg += __shfl_xor_sync(0xFFFFFFFFu, vg, off);
          vu += __shfl_xor_sync(0xFFFFFFFFu, vu, off);
        }
        if (lane == j) {
          const float gg = vg * tsg, uu = vu * tsu;
          a.h[size_t(n0 + j) * a.f + row] = gg / (1.f + expf(-gg)) * uu;
        }
      }
    }
  }
}

template <int FMT>
__global__ void __launch_bounds__(kFfnWarps * 32) ffn_down_kernel(FfnArgs a) {
  __shared__ int s_start[1025];
  __shared__ int s_warp_tot[33];
  pdl_wait();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int total = build_item_starts(a, a.d, s_start, s_warp_tot);
  const long long G = (long long)gridDim.x * kFfnWarps;
  const long long g = (long long)blockIdx.x * kFfnWarps + warp;
  const int i0 = int(g * total / G), i1 = int((g + 1) * total / G);
  using Tr = FmtTraits<FMT>;
  const size_t rb = Tr::row_bytes(a.f);
  const size_t mat_bytes = rb * a.d;
  const size_t smat = Tr::scale_bytes(a.d, a.f);
  const int units = a.f / 32;
  int e = i0 < i1 ? find_expert(s_start, a.E, i0) : 0;
  for (int item = i0; item < i1; ++item) {
    while (item >= s_start[e + 1]) ++e;
    const int local = item - s_start[e];
    const int tile = local / a.d, row = local % a.d;
    const int slot = a.slot_of ? a.slot_of[e] : e;
    const int n0 = a.offsets[e] + tile * kTokTile;
    const int nt = min(kTokTile, a.offsets[e + 1] - n0);
    const uint8_t* drow = a.down + slot * mat_bytes + row * rb;
    const uint8_t* dsrow = nullptr;
    const float* dfrow = nullptr;
    if (FMT == FTMOE_NVFP4 || FMT == FTMOE_MXFP4) {
      const size_t sr = (FMT == FTMOE_NVFP4) ? a.f / 16 : a.f / 32;
      dsrow = a.down_s + slot * smat + row * sr;
    } else if (FMT == FTMOE_FP8_B128) {
      dfrow = reinterpret_cast<const float*>(a.down_s + slot * smat) + (row / 128) * (a.f / 128);
    }
    float acc[kTokTile];
#pragma unroll
    for (int j = 0; j < kTokTile; ++j) acc[j] = 0.f;
    for (int u = lane; u < units; u += 32) {
      Unit<FMT, 32> du;
      du.load(drow, dsrow, dfrow, u);
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        float wd[16];
        du.decode16(q, wd);
#pragma unroll
        for (int j = 0; j < kTokTile; ++j) {
          if (j < nt) {
            const float4* hp = reinterpret_cast<const float4*>(a.h + size_t(n0 + j) * a.f + 32 * u + 16 * q);
            float s = 0.f;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const float4 hv = hp[i];
              s = fmaf(wd[4 * i + 0], hv.x, s);
              s = fmaf(wd[4 * i + 1], hv.y, s);
              s = fmaf(wd[4 * i + 2], hv.z, s);
              s = fmaf(wd[4 * i + 3], hv.w, s);
            }
            acc[j] += s;
          }
        }
      }
    }
    const float tsd = a.tscale ? a.tscale[slot * 3 + 2] : 1.f;
#pragma unroll
    for (int j = 0; j < kTokTile; ++j) {
      if (j < nt) {
        float v = acc[j];
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, off);
        if (lane == j) {
          v *= tsd;
          if (a.topk_w) {
            const int p = a.sorted_pair[n0 + j];
            atomicAdd(a.y_or_out + size_t(p / a.k) * a.d + row, a.topk_w[p] * v);
          } else {
            a.y_or_out[size_t(n0 + j) * a.d + row] = v;
          }
        }
      }
    }
  }
}

}  // namespace ftmoe
