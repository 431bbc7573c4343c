// a4 (+a5) decode path for the block-scaled 4-bit formats (NVFP4, MXFP4):
// the grouped SwiGLU expert FFN with few tokens per expert, as a stream of the
// selected experts' packed weights through warp-level tensor-core MMAs.
//
// Pages: resident experts are computed on GPU tensor cores from expert slots
// (zubnet.ai, "FreeToken, Unsloth GGUF ... consumer hardware"); in decode a
// token touches a few experts (banandre.com, "The 284B Model on a 32GB
// GPU Trick", section "Sparsity Is a Lie").  A decode layer reads each
// selected expert's weights once, so it is bound by HBM bandwidth.
//
// Work unit = (expert, 16 weight rows).  One CTA of 4 warps takes a unit and
// splits K four ways; each warp issues the loads of up to 8 super-blocks of
// its K range before it computes, so a unit's bytes are in flight together.
// The unit's tokens (a group of up to 8) are staged once in shared memory as
// f16, so the MMA loop reads its B fragments there.  The partial sums of the
// four warps meet in shared memory.
//
// MMA: mma.sync m16n8k16, f16 operands, fp32 accumulation.  Weights are the A
// operand (16 rows), tokens the B operand (8 per MMA; a unit's tokens run in
// passes of 8).  The dot product does not depend on the order of K,
// so K is permuted to match the loads: in each 64-element super-block, lane
// (g = lane / 4, t = lane % 4) loads the 8 code bytes of elements
// [16 t, 16 t + 16) of rows g and g + 8 (one NVFP4 scale block), and MMA step
// j takes elements 16 t + 4 j + {0, 1} as logical columns {2t, 2t + 1} and
// 16 t + 4 j + {2, 3} as {2t + 8, 2t + 9}.  The tokens' x (or h) elements
// follow the same map.
//
// Dequantisation: E2M1 -> f16 is exact.  NVFP4: code * E4M3 scale has at most
// 6 significant bits and lies in [2^-10, 2688], so the f16 product is exact;
// the per-tensor fp32 scale is applied to the result.  MXFP4: the E8M0 scales
// of a chunk (up to 8 super-blocks) are rebased on their maximum E0 (f16 factor
// 2^(e - E0) <= 1) and the chunk's partial sum is multiplied by 2^(E0 - 127)
// in fp32.
//
// Activations: x (bf16) and h (fp32) are rounded to f16 (bf16 -> f16 is exact
// in f16's normal range).  A non-finite result flags FTMOE_ERR_DEVICE_CHECK:
// inputs beyond the f16 range (|v| > 65504) are outside this path.
//
// One persistent kernel (dec_ffn_kernel) runs both halves, with a grid barrier between:
//   phase A  h[j][n] = silu(g) * u for the expert's sorted rows j (fp32 [P][f])
//   phase B  y = h W_down^T: written in sorted order, or w * y added into out (fused combine)
// Called by the layer forward, it also zeroes out first and, after a second barrier, writes
// the bf16 copy of out.
#pragma once
#include "common.cuh"
#include "ffn_stream.cuh"

namespace ftmoe {

constexpr int kDecWarps = 4;
constexpr int kDecChunk = 8;    // super-blocks per loaded chunk

__device__ __forceinline__ void mma_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                          uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// one byte (two E2M1 codes, element 2i in the low nibble) -> f16x2 (low half = element 2i)
__device__ __forceinline__ uint32_t e2m1_byte_f16x2(uint32_t word, int byte) {
  uint32_t r;
  const uint32_t b = (word >> (8 * byte)) & 0xFFu;
  asm("{\n\t.reg .b8 q;\n\tcvt.u8.u32 q, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, q;\n\t}" : "=r"(r) : "r"(b));
  return r;
}
__device__ __forceinline__ uint32_t hmul2(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}
// an E4M3 code -> f16x2 holding its value twice (exact)
__device__ __forceinline__ uint32_t e4m3_f16x2(uint32_t code) {
  uint32_t r;
  const uint16_t v = uint16_t(code | (code << 8));
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(v));
  return r;
}
// 2^d for d <= 0 as f16x2 (0 below the f16 subnormal range)
__device__ __forceinline__ uint32_t pow2_f16x2(int d) {
  uint32_t h = 0;
  if (d >= -14) h = uint32_t(15 + d) << 10;
  else if (d >= -24) h = 1u << (d + 24);
  return h | (h << 16);
}
// two floats -> f16x2 (lo, hi)
__device__ __forceinline__ uint32_t f16x2_of(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// Token staging in shared memory: up to 8 rows of K f16 values, row stride K + 8
// (the 16-byte pad spreads the 8 rows of a fragment load over distinct banks).
__device__ __forceinline__ int stage_stride(int K) { return K + 8; }

// x rows (bf16) of tokens [i0, i0 + n) of the unit -> f16 rows in s_x (all threads)
__device__ __forceinline__ void stage_x_bf16(uint16_t* s_x, const FfnArgs& a, int lo, int i0, int n, int K) {
  const int per = K / 8;                       // 16-byte chunks per row
  const int st = stage_stride(K);
  for (int c = threadIdx.x; c < n * per; c += blockDim.x) {
    const int q = c / per, cc = c % per;
    const uint16_t* row = a.x + size_t(a.sorted_pair[lo + i0 + q] / a.k) * a.d;
    const uint4 v = __ldg(reinterpret_cast<const uint4*>(row) + cc);
    uint4 h;
    h.x = f16x2_of(bf16_lo(v.x), bf16_hi(v.x));
    h.y = f16x2_of(bf16_lo(v.y), bf16_hi(v.y));
    h.z = f16x2_of(bf16_lo(v.z), bf16_hi(v.z));
    h.w = f16x2_of(bf16_lo(v.w), bf16_hi(v.w));
    *reinterpret_cast<uint4*>(s_x + q * st + 8 * cc) = h;
  }
}
// h rows (fp32 [*][K], sorted order) of tokens [i0, i0 + n) -> f16 rows in s_x.  Read
// through L2 (ld.cg): in the fused kernel h was written by other CTAs of the same grid.
__device__ __forceinline__ void stage_h_f32(uint16_t* s_x, const float* h, int K, int lo, int i0, int n) {
  const int per = K / 8;
  const int st = stage_stride(K);
  for (int c = threadIdx.x; c < n * per; c += blockDim.x) {
    const int q = c / per, cc = c % per;
    const float4* row = reinterpret_cast<const float4*>(h + size_t(lo + i0 + q) * K) + 2 * cc;
    const float4 v0 = __ldcg(row), v1 = __ldcg(row + 1);
    uint4 h;
    h.x = f16x2_of(v0.x, v0.y);
    h.y = f16x2_of(v0.z, v0.w);
    h.z = f16x2_of(v1.x, v1.y);
    h.w = f16x2_of(v1.z, v1.w);
    *reinterpret_cast<uint4*>(s_x + q * st + 8 * cc) = h;
  }
}

// The core, in two halves so that a chunk's weight loads can be issued before the
// tokens are staged.  NM weight matrices (1: down, 2: gate + up) x 16 rows; a chunk is up
// to kDecChunk super-blocks of this warp's K range.
//   rows[m][0|1]: code rows g and g + 8;  srows[m][0|1]: their scale rows
template <int FMT, int NM>
struct DecChunk {
  uint2 code[NM][2][kDecChunk];
  uint32_t sc[NM][2][kDecChunk];
  int sb0, nc;

  // every weight load of the chunk (clamped to the range, so no branch)
  __device__ __forceinline__ void load(const uint8_t* const (&rows)[NM][2], const uint8_t* const (&srows)[NM][2],
                                       int sb_start, int sb_hi, int t) {
    sb0 = sb_start;
    nc = min(kDecChunk, sb_hi - sb0);
#pragma unroll
    for (int m = 0; m < NM; ++m)
#pragma unroll
      for (int r = 0; r < 2; ++r)
#pragma unroll
        for (int c = 0; c < kDecChunk; ++c) {
          const int sb = sb0 + min(c, nc - 1);
          code[m][r][c] = __ldcs(reinterpret_cast<const uint2*>(rows[m][r] + 32 * sb + 8 * t));
          if (FMT == FTMOE_NVFP4)
            sc[m][r][c] = __ldg(reinterpret_cast<const uint32_t*>(srows[m][r]) + sb);
          else
            sc[m][r][c] = __ldg(reinterpret_cast<const uint16_t*>(srows[m][r]) + sb);
        }
  }

  // MMAs of the chunk against the staged tokens (xrow = this lane's token row + 16 t); adds into acc
  __device__ __forceinline__ void compute(const uint16_t* xrow, int t, float (&acc)[NM][4]) const {
    int e0[NM][2];
#pragma unroll
    for (int m = 0; m < NM; ++m)
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        e0[m][r] = 0;
        if (FMT == FTMOE_MXFP4) {
#pragma unroll
          for (int c = 0; c < kDecChunk; ++c)
            if (c < nc) e0[m][r] = max(e0[m][r], int(max(sc[m][r][c] & 0xFFu, sc[m][r][c] >> 8)));
        }
      }
    float part[NM][4];
#pragma unroll
    for (int m = 0; m < NM; ++m)
#pragma unroll
      for (int i = 0; i < 4; ++i) part[m][i] = 0.f;
#pragma unroll
    for (int c = 0; c < kDecChunk; ++c) {
      if (c < nc) {
        const uint16_t* xp = xrow + 64 * (sb0 + c);
        const uint4 x0 = *reinterpret_cast<const uint4*>(xp);
        const uint4 x1 = *reinterpret_cast<const uint4*>(xp + 8);
        const uint32_t B[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
#pragma unroll
        for (int m = 0; m < NM; ++m) {
          uint32_t pre0, pre1;
          if (FMT == FTMOE_NVFP4) {
            pre0 = e4m3_f16x2((sc[m][0][c] >> (8 * t)) & 0xFFu);
            pre1 = e4m3_f16x2((sc[m][1][c] >> (8 * t)) & 0xFFu);
          } else {
            pre0 = pow2_f16x2(int((sc[m][0][c] >> (8 * (t >> 1))) & 0xFFu) - e0[m][0]);
            pre1 = pow2_f16x2(int((sc[m][1][c] >> (8 * (t >> 1))) & 0xFFu) - e0[m][1]);
          }
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const uint32_t wg = j < 2 ? code[m][0][c].x : code[m][0][c].y;
            const uint32_t wh = j < 2 ? code[m][1][c].x : code[m][1][c].y;
            const int b = 2 * (j & 1);
            const uint32_t a0 = hmul2(e2m1_byte_f16x2(wg, b), pre0);
            const uint32_t a1 = hmul2(e2m1_byte_f16x2(wh, b), pre1);
            const uint32_t a2 = hmul2(e2m1_byte_f16x2(wg, b + 1), pre0);
            const uint32_t a3 = hmul2(e2m1_byte_f16x2(wh, b + 1), pre1);
            if (FMT == FTMOE_MXFP4) mma_16816(part[m], a0, a1, a2, a3, B[2 * j], B[2 * j + 1]);
            else mma_16816(acc[m], a0, a1, a2, a3, B[2 * j], B[2 * j + 1]);
          }
        }
      }
    }
    if (FMT == FTMOE_MXFP4) {
#pragma unroll
      for (int m = 0; m < NM; ++m) {
        const float f0 = e8m0_to_float(uint32_t(e0[m][0])), f1 = e8m0_to_float(uint32_t(e0[m][1]));
        acc[m][0] = fmaf(f0, part[m][0], acc[m][0]);
        acc[m][1] = fmaf(f0, part[m][1], acc[m][1]);
        acc[m][2] = fmaf(f1, part[m][2], acc[m][2]);
        acc[m][3] = fmaf(f1, part[m][3], acc[m][3]);
      }
    }
  }
};

// One pass over the warp's K range for the tokens staged by `stage` (a callable run by
// the whole CTA, followed by a barrier): the first chunk's loads go out before the staging.
// ch: the chunk registers; preloaded: ch already holds the first chunk of this pass.
template <int FMT, int NM, typename Stage>
__device__ __forceinline__ void dec_pass(const uint8_t* const (&rows)[NM][2], const uint8_t* const (&srows)[NM][2],
                                         const uint16_t* s_x, int K, int sb_lo, int sb_hi, int g, int t,
                                         Stage stage, float (&acc)[NM][4], DecChunk<FMT, NM>& ch, bool preloaded) {
#pragma unroll
  for (int m = 0; m < NM; ++m)
#pragma unroll
    for (int i = 0; i < 4; ++i) acc[m][i] = 0.f;
  if (!preloaded && sb_lo < sb_hi) ch.load(rows, srows, sb_lo, sb_hi, t);
  stage();
  __syncthreads();
  const uint16_t* xrow = s_x + g * stage_stride(K) + 16 * t;
  for (int sb0 = sb_lo; sb0 < sb_hi; sb0 += kDecChunk) {
    if (sb0 > sb_lo) ch.load(rows, srows, sb0, sb_hi, t);
    ch.compute(xrow, t, acc);
  }
}

// Shared reduction buffer: [warp][matrix][row 16][token 8]
template <int NM>
struct DecRed {
  float v[kDecWarps][NM][16][8];
};

template <int NM>
__device__ __forceinline__ void dec_store_partials(DecRed<NM>& s, int warp, int g, int t, const float (&acc)[NM][4]) {
#pragma unroll
  for (int m = 0; m < NM; ++m) {
    s.v[warp][m][g][2 * t] = acc[m][0];
    s.v[warp][m][g][2 * t + 1] = acc[m][1];
    s.v[warp][m][g + 8][2 * t] = acc[m][2];
    s.v[warp][m][g + 8][2 * t + 1] = acc[m][3];
  }
}



// Grid-wide barrier of a grid whose CTAs are all resident (the launch sizes the grid by
// occupancy).  count returns to 0 after each barrier; gen is only incremented.  The wait is
// bounded: false = gave up (FTMOE_ERR_TIMEOUT recorded).
__device__ __forceinline__ bool grid_barrier(unsigned* count, unsigned* gen, int* s_flag) {
  __syncthreads();
  if (threadIdx.x == 0) {
    int ok = 1;
    const unsigned g = *reinterpret_cast<volatile unsigned*>(gen);
    __threadfence();
    if (atomicAdd(count, 1u) == gridDim.x - 1) {
      *reinterpret_cast<volatile unsigned*>(count) = 0u;
      __threadfence();
      atomicAdd(gen, 1u);
    } else {
      unsigned long long t0 = 0;
      asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t0));
      for (uint32_t it = 0; *reinterpret_cast<volatile unsigned*>(gen) == g; ++it) {
        if ((it & 63u) == 63u) {
          unsigned long long t1;
          asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t1));
          if (t1 - t0 > 2000000000ull) {
            ok = 0;
            set_dev_err(DEV_ERR_GRID_TIMEOUT);
            break;
          }
        }
        __nanosleep(64);
      }
    }
    __threadfence();
    *s_flag = ok;
  }
  __syncthreads();
  return *s_flag != 0;
}

// Dynamic shared memory of the decode kernel: expert ranks [1025] ints, the reduction
// buffer, the staged tokens.  Every region starts on a 16-byte boundary (the staged rows
// are read and written with 16-byte vector accesses).
constexpr size_t kDecOffRed = (1025 * 4 + 15) / 16 * 16;
constexpr size_t kDecOffX = kDecOffRed + (sizeof(DecRed<2>) + 15) / 16 * 16;
__host__ __device__ constexpr size_t dec_smem_bytes(int Kmax) { return kDecOffX + size_t(8) * (Kmax + 8) * 2; }
static_assert(kDecOffRed % 16 == 0 && kDecOffX % 16 == 0, "decode shared-memory regions must be 16-byte aligned");

// s_rank[e] = resident experts with rows below e; returns their number.  (All threads.)
__device__ __forceinline__ int dec_expert_ranks(const FfnArgs& a, int* s_rank) {
  for (int e = threadIdx.x; e < a.E; e += blockDim.x) {
    const int cnt = a.offsets[e + 1] - a.offsets[e];
    int slot = a.slot_of ? a.slot_of[e] : e;
    if (slot >= a.C) {
      if (cnt > 0 && blockIdx.x == 0) set_dev_err(DEV_ERR_BAD_SLOT);
      slot = -1;
    }
    s_rank[e] = (cnt > 0 && slot >= 0) ? 1 : 0;
  }
  __syncthreads();
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    int run = 0;
    for (int base = 0; base < a.E; base += 32) {
      const int e = base + lane;
      const int n = e < a.E ? s_rank[e] : 0;
      int incl = n;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int o = __shfl_up_sync(0xFFFFFFFFu, incl, off);
        if (lane >= off) incl += o;
      }
      if (e < a.E) s_rank[e] = run + incl - n;
      run += __shfl_sync(0xFFFFFFFFu, incl, 31);
    }
    if (lane == 0) s_rank[a.E] = run;
  }
  __syncthreads();
  return s_rank[a.E];
}

// Rows of one unit: weight row pointers, scale rows, tokens.
struct DecUnit {
  int e, n0, slot, lo, cnt;
};
__device__ __forceinline__ DecUnit dec_unit(const FfnArgs& a, const int* s_rank, int unit, int per_expert) {
  DecUnit u;
  const int r = unit / per_expert;
  u.e = find_expert(s_rank, a.E, r);   // largest e with s_rank[e] <= r: the expert of rank r
  u.n0 = (unit - r * per_expert) * 16;
  u.slot = a.slot_of ? a.slot_of[u.e] : u.e;
  u.lo = a.offsets[u.e];
  u.cnt = a.offsets[u.e + 1] - u.lo;
  return u;
}

template <int FMT>
struct DecDown {
  const uint8_t* rows[1][2];
  const uint8_t* srows[1][2];
  __device__ __forceinline__ DecDown(const FfnArgs& a, const DecUnit& u, int g) {
    const size_t rowb = size_t(a.f) / 2, mat = rowb * a.d;
    const size_t srow = (FMT == FTMOE_NVFP4) ? a.f / 16 : a.f / 32, smat = srow * a.d;
    rows[0][0] = a.down + u.slot * mat + (u.n0 + g) * rowb;
    rows[0][1] = a.down + u.slot * mat + (u.n0 + g + 8) * rowb;
    srows[0][0] = a.down_s + u.slot * smat + (u.n0 + g) * srow;
    srows[0][1] = a.down_s + u.slot * smat + (u.n0 + g + 8) * srow;
  }
};

// One kernel for both halves of the FFN:
//   phase A  units of 16 gate/up rows: h[j][n] = silu(g) * u for the expert's sorted rows j
//   barrier  (every h written); the first phase-B unit's weights are already loading
//   phase B  units of 16 down rows: y = h W_down^T, written in sorted order or added as w * y
//            into out (fused combine)
template <int FMT>
__global__ void __launch_bounds__(kDecWarps * 32) dec_ffn_kernel(FfnArgs a, unsigned* bar_count, unsigned* bar_gen) {
  extern __shared__ __align__(16) uint8_t dsm[];
  int* s_rank = reinterpret_cast<int*>(dsm);
  DecRed<2>& s_red2 = *reinterpret_cast<DecRed<2>*>(dsm + kDecOffRed);
  DecRed<1>& s_red1 = *reinterpret_cast<DecRed<1>*>(dsm + kDecOffRed);
  uint16_t* s_x = reinterpret_cast<uint16_t*>(dsm + kDecOffX);
  __shared__ int s_flag;
  pdl_wait();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int g = lane >> 2, t = lane & 3;
  const int nres = dec_expert_ranks(a, s_rank);
  const int row = threadIdx.x & 15, tok = threadIdx.x >> 4;   // epilogue: thread -> (row, token)

  // layer call: the fused-combine accumulator starts at zero (ordered before every add by the barrier)
  if (a.out_bf16) {
    float4* o = reinterpret_cast<float4*>(a.y_or_out);
    const long long n4 = (long long)a.T * a.d / 4;
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n4; i += (long long)gridDim.x * blockDim.x)
      o[i] = make_float4(0.f, 0.f, 0.f, 0.f);
  }

  // ---------------- phase A: gate / up ----------------
  {
    const int per = a.f / 16;
    const int nsb = a.d / 64;
    const int sb_lo = warp * nsb / kDecWarps, sb_hi = (warp + 1) * nsb / kDecWarps;
    const size_t rowb = size_t(a.d) / 2, mat = rowb * a.f;
    const size_t srow = (FMT == FTMOE_NVFP4) ? a.d / 16 : a.d / 32, smat = srow * a.f;
    for (int unit = blockIdx.x; unit < nres * per; unit += gridDim.x) {
      const DecUnit u = dec_unit(a, s_rank, unit, per);
      const uint8_t* const rows[2][2] = {
          {a.gate + u.slot * mat + (u.n0 + g) * rowb, a.gate + u.slot * mat + (u.n0 + g + 8) * rowb},
          {a.up + u.slot * mat + (u.n0 + g) * rowb, a.up + u.slot * mat + (u.n0 + g + 8) * rowb}};
      const uint8_t* const srows[2][2] = {
          {a.gate_s + u.slot * smat + (u.n0 + g) * srow, a.gate_s + u.slot * smat + (u.n0 + g + 8) * srow},
          {a.up_s + u.slot * smat + (u.n0 + g) * srow, a.up_s + u.slot * smat + (u.n0 + g + 8) * srow}};
      const float tsg = a.tscale ? a.tscale[u.slot * 3 + 0] : 1.f;
      const float tsu = a.tscale ? a.tscale[u.slot * 3 + 1] : 1.f;
      for (int p0 = 0; p0 < u.cnt; p0 += 8) {
        const int n = min(8, u.cnt - p0);
        float acc[2][4];
        DecChunk<FMT, 2> ch;
        dec_pass<FMT, 2>(rows, srows, s_x, a.d, sb_lo, sb_hi, g, t,
                         [&] { stage_x_bf16(s_x, a, u.lo, p0, n, a.d); }, acc, ch, false);
        dec_store_partials<2>(s_red2, warp, g, t, acc);
        __syncthreads();
        if (tok < n) {
          float gs = 0.f, us = 0.f;
#pragma unroll
          for (int w = 0; w < kDecWarps; ++w) {
            gs += s_red2.v[w][0][row][tok];
            us += s_red2.v[w][1][row][tok];
          }
          const float gg = gs * tsg, uu = us * tsu;
          const float h = gg / (1.f + expf(-gg)) * uu;
          if (!isfinite(h)) set_dev_err(DEV_ERR_NONFINITE);
          a.h[size_t(u.lo + p0 + tok) * a.f + u.n0 + row] = h;
        }
        __syncthreads();
      }
    }
  }

  // ---------------- phase B: down ----------------
  const int per = a.d / 16;
  const int nsb = a.f / 64;
  const int sb_lo = warp * nsb / kDecWarps, sb_hi = (warp + 1) * nsb / kDecWarps;
  const int total = nres * per;
  DecChunk<FMT, 1> pre;     // phase-B chunk registers; the first unit's first chunk loads before the barrier
  const bool have_pre = blockIdx.x < total && sb_lo < sb_hi;
  if (have_pre) {
    const DecUnit u = dec_unit(a, s_rank, blockIdx.x, per);
    const DecDown<FMT> w(a, u, g);
    pre.load(w.rows, w.srows, sb_lo, sb_hi, t);
  }
  if (!grid_barrier(bar_count, bar_gen, &s_flag)) return;
  const float* hbase = a.h;
  for (int unit = blockIdx.x; unit < total; unit += gridDim.x) {
    const DecUnit u = dec_unit(a, s_rank, unit, per);
    const DecDown<FMT> w(a, u, g);
    const float tsd = a.tscale ? a.tscale[u.slot * 3 + 2] : 1.f;
    for (int p0 = 0; p0 < u.cnt; p0 += 8) {
      const int n = min(8, u.cnt - p0);
      float acc[1][4];
      const bool use_pre = have_pre && unit == int(blockIdx.x) && p0 == 0;
      dec_pass<FMT, 1>(w.rows, w.srows, s_x, a.f, sb_lo, sb_hi, g, t,
                       [&] { stage_h_f32(s_x, hbase, a.f, u.lo, p0, n); }, acc, pre, use_pre);
      dec_store_partials<1>(s_red1, warp, g, t, acc);
      __syncthreads();
      if (tok < n) {
        float y = 0.f;
#pragma unroll
        for (int ww = 0; ww < kDecWarps; ++ww) y += s_red1.v[ww][0][row][tok];
        y *= tsd;
        if (!isfinite(y)) set_dev_err(DEV_ERR_NONFINITE);
        const int i = p0 + tok;
        if (a.topk_w) {
          const int p = a.sorted_pair[u.lo + i];
          atomicAdd(a.y_or_out + size_t(p / a.k) * a.d + u.n0 + row, a.topk_w[p] * y);
        } else {
          a.y_or_out[size_t(u.lo + i) * a.d + u.n0 + row] = y;
        }
      }
      __syncthreads();
    }
  }
  // layer call: every add has landed; cast the output to bf16 (round to nearest even)
  if (a.out_bf16) {
    if (!grid_barrier(bar_count, bar_gen, &s_flag)) return;
    const float4* o = reinterpret_cast<const float4*>(a.y_or_out);
    uint2* ob = reinterpret_cast<uint2*>(a.out_bf16);
    const long long n4 = (long long)a.T * a.d / 4;
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n4; i += (long long)gridDim.x * blockDim.x) {
      const float4 v = __ldcg(o + i);
      __nv_bfloat162 lo = __floats2bfloat162_rn(v.x, v.y), hi = __floats2bfloat162_rn(v.z, v.w);
      ob[i] = make_uint2(*reinterpret_cast<uint32_t*>(&lo), *reinterpret_cast<uint32_t*>(&hi));
    }
  }
}

}  // namespace ftmoe
