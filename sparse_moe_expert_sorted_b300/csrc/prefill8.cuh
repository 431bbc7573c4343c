// a3 + a4 (+a5) prefill path for FP8_B128 weights: the grouped SwiGLU expert FFN
// on tcgen05 tensor cores (kind::f8f6f4, E4M3 x E4M3 -> fp32) with FP8 activations.
//
// Pages: resident experts run on GPU tensor cores from expert slots, with FP8
// among the weight formats (zubnet.ai, "FreeToken, Unsloth GGUF ... consumer
// hardware"); a prefill chunk touches nearly every expert (banandre.com, "The 284B
// Model on a 32GB GPU Trick", section "The Three Failure Modes").
//
// Scales.  Weights carry one fp32 scale per 128 x 128 block; activations carry one
// fp32 scale per (row, 128 columns) by the library's rule (s = amax / 448, q =
// E4M3(v / s)).  No tcgen05 scale kind takes fp32 scales, so each 128-wide K step
// (one scale block of both operands) is its own MMA group: 4 MMAs (K = 32 each)
// write a fresh partial P_kb into one of two TMEM buffers, and the epilogue warps
// add P_kb * s_x[row, kb] * s_w[block, kb] into fp32 registers while the tensor
// cores fill the other buffer.
//
// Kernels (one stream, in order):
//   quantize8_kernel   x -> per-token E4M3 codes + fp32 scales (once per token)
//   gather8_kernel     padded expert-sorted rows <- the tokens' codes; scales
//                      transposed to [K/128][rows] (a K step's scales are contiguous)
//   gemm8_kernel<0>    [gate | up] tile (128 + 128 columns); epilogue h = silu(g) * u,
//                      quantised to E4M3 per (row, 128 columns)
//   gemm8_kernel<1>    down tile (256 columns); epilogue adds w * y into out[token]
//                      (fused combine) or writes y in sorted order
// GEMM CTA (persistent, one per SM): warp 0 TMA producer (3-stage ring), warp 1 TMEM
// owner and MMA issuer, warps 2-9 epilogue (warp w reads TMEM lanes 32 (w % 4) ..,
// columns [64 h, 64 h + 64) of both 128-column blocks, h = (w - 2) / 4).
#pragma once
#include "prefill.cuh"

namespace ftmoe {

constexpr int kG8Stages = 3;
constexpr int kG8MaxKB = 64;   // K / 128 steps supported (K <= 8192)

// FP8 quantisation of 128 values held 4 per lane by one warp: s = amax / 448, q = E4M3(v / s)
// (IEEE fp32 divisions, a zero of v's sign when s == 0).  Returns s; codes in c (4 bytes, element 0 low).
__device__ __forceinline__ float quant_fp8_warp(const float (&v)[4], uint32_t& c) {
  float amax = fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3])));
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, off));
  const float s = amax / 448.0f;
  uint32_t b[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) b[i] = s > 0.f ? e4m3_code(v[i] / s) : e4m3_code(copysignf(0.f, v[i]));
  c = b[0] | (b[1] << 8) | (b[2] << 16) | (b[3] << 24);
  return s;
}

// x [T][d] bf16 -> codes [T][d], scales [T][d/128] (one warp per 128-element block)
__global__ void __launch_bounds__(256) quantize8_kernel(const uint16_t* x, int T, int d, uint8_t* codes,
                                                        float* scales) {
  pdl_wait();
  const int lane = threadIdx.x & 31;
  const int nb = d / 128;
  const long long blocks = (long long)T * nb;
  for (long long bi = (long long)blockIdx.x * 8 + (threadIdx.x >> 5); bi < blocks; bi += (long long)gridDim.x * 8) {
    const long long t = bi / nb;
    const int b = int(bi % nb);
    const uint2 raw = __ldg(reinterpret_cast<const uint2*>(x + t * d + 128 * b) + lane);
    const float v[4] = {bf16_lo(raw.x), bf16_hi(raw.x), bf16_lo(raw.y), bf16_hi(raw.y)};
    uint32_t c;
    const float s = quant_fp8_warp(v, c);
    reinterpret_cast<uint32_t*>(codes + t * d + 128 * b)[lane] = c;
    if (lane == 0) scales[bi] = s;
  }
}

struct Gather8Args {
  const uint8_t* xq_tok;   // [T][d]
  const float* sx_tok;     // [T][d/128]
  int d, k, E, C, P;
  const int32_t* offsets;
  const int32_t* sorted_pair;
  const int32_t* slot_of;
  uint8_t* xq;             // [rows_cap][d]
  float* sx;               // [d/128][rows_cap]
  int rows_cap;
  float4* zero_out;
  long long zero_n4;
  const float* topk_w;     // or nullptr
  int4* rowmeta;           // [rows_cap] row_meta of each padded row
};

__global__ void __launch_bounds__(kActqWarps * 32) gather8_kernel(Gather8Args a) {
  __shared__ int s_mt[1025];
  __shared__ int s_tmp[33];
  pdl_wait();
  if (a.zero_out) {
    const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < a.zero_n4;
         i += (long long)gridDim.x * blockDim.x)
      a.zero_out[i] = z;
  }
  const int MT = build_mtile_starts(a.offsets, a.slot_of, a.E, a.C, a.rows_cap / kTileM, s_mt, s_tmp);
  const int lane = threadIdx.x & 31;
  const int nb = a.d / 128;
  const int rows = MT * kTileM;
  for (int j = blockIdx.x * kActqWarps + (threadIdx.x >> 5); j < rows; j += gridDim.x * kActqWarps) {
    const int e = expert_of_mtile(s_mt, a.E, j / kTileM);
    const int i = j - s_mt[e] * kTileM;
    const int lo = a.offsets[e];
    int tok = -1;
    if (i < a.offsets[e + 1] - lo) {
      const int p = a.sorted_pair[lo + i];
      if (p >= 0 && p < a.P) tok = p / a.k;
      else set_dev_err(DEV_ERR_BAD_PAIR);
      if (lane == 0) a.rowmeta[j] = row_meta(lo + i, tok >= 0 ? p : -1, a.k, a.topk_w);
    } else if (lane == 0) {
      a.rowmeta[j] = make_int4(-1, -1, 0, 0);
    }
    const uint4* src = reinterpret_cast<const uint4*>(a.xq_tok + size_t(tok < 0 ? 0 : tok) * a.d);
    uint4* dst = reinterpret_cast<uint4*>(a.xq + size_t(j) * a.d);
    for (int c = lane; c < a.d / 16; c += 32) dst[c] = tok >= 0 ? __ldg(src + c) : make_uint4(0u, 0u, 0u, 0u);
    for (int b = lane; b < nb; b += 32) a.sx[size_t(b) * a.rows_cap + j] = tok >= 0 ? __ldg(a.sx_tok + size_t(tok) * nb + b) : 0.f;
  }
}

struct Gemm8Args {
  int E, k, d, f, C, P;
  int rows_cap;
  const int32_t* offsets;
  const int32_t* sorted_pair;
  const int32_t* slot_of;
  const float* sx;          // activation scales [K/128][rows_cap]
  const float* sw0;         // weight block scales: MODE 0 gate, MODE 1 down   [C][N/128][K/128]
  const float* sw1;         // MODE 0 up
  uint8_t* hq;              // MODE 0: h codes [rows_cap][f]
  float* sh;                // MODE 0: h scales [f/128][rows_cap]
  const float* topk_w;      // MODE 1: fused combine weights, or nullptr (write y)
  float* out;               // MODE 1: out [T][d] (fused) or y [P][d] (sorted)
  const int4* rowmeta;      // MODE 1: row_meta of each padded row
};

template <int MODE>
struct G8Cfg {
  static constexpr int N = 256;
  static constexpr int A_BYTES = kTileM * 128;
  static constexpr int B_BYTES = N * 128;
  static constexpr int STAGE_TX = A_BYTES + B_BYTES;
  static constexpr int OFF_A = 0;
  static constexpr int OFF_B = OFF_A + kG8Stages * A_BYTES;
  static constexpr int OFF_BAR = OFF_B + kG8Stages * B_BYTES;   // full[S], empty[S], tfull[2], tempty[2], done
  static constexpr int OFF_MISC = OFF_BAR + (2 * kG8Stages + 5) * 8;
  static constexpr int OFF_MT = OFF_MISC + 16;                   // s_mt[1025], s_tmp[33]
  static constexpr int OFF_SW = (OFF_MT + (1025 + 33) * 4 + 15) / 16 * 16;   // [2][kG8MaxKB] weight scales of the tile
  static constexpr int OFF_AMAX = OFF_SW + 2 * kG8MaxKB * 4;     // MODE 0: [2][128] per-half row amax
  static constexpr int STG_W = 32 + 4;                           // MODE 1: staging row stride (floats)
  static constexpr int OFF_STG = OFF_AMAX + 2 * 128 * 4;
  static constexpr int STG_BYTES = MODE == 1 ? kEpiWarps * 32 * STG_W * 4 : 0;
  static constexpr int SMEM = OFF_STG + STG_BYTES + 1024;
  static constexpr uint32_t IDESC = idesc_f8(kTileM, N);
  static_assert(SMEM <= 232448, "one CTA's opt-in shared memory");
  static_assert(STAGE_TX < (1 << 20), "an mbarrier's transaction count");
  static_assert(OFF_BAR % 8 == 0 && A_BYTES % 1024 == 0 && B_BYTES % 1024 == 0, "aligned barriers and stages");
};

// Epilogue-only barrier: named barrier 2 over the 8 epilogue warps.
__device__ __forceinline__ void g8_epi_sync() { asm volatile("bar.sync 2, %0;" ::"r"(kEpiWarps * 32) : "memory"); }

template <int MODE>
__global__ void __launch_bounds__(kGemmThreads, 1)
gemm8_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB0,
             const __grid_constant__ CUtensorMap tmB1, Gemm8Args a) {
  using Cfg = G8Cfg<MODE>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sb = smem_u32(smem);
  const uint32_t bar_full = sb + Cfg::OFF_BAR, bar_empty = bar_full + 8 * kG8Stages;
  const uint32_t bar_tfull = bar_empty + 8 * kG8Stages, bar_tempty = bar_tfull + 16, bar_done = bar_tempty + 16;
  uint32_t* s_tslot = reinterpret_cast<uint32_t*>(smem + Cfg::OFF_MISC);
  volatile int* s_abort = reinterpret_cast<volatile int*>(smem + Cfg::OFF_MISC + 4);
  int* s_mt = reinterpret_cast<int*>(smem + Cfg::OFF_MT);
  int* s_tmp = s_mt + 1025;
  float* s_sw = reinterpret_cast<float*>(smem + Cfg::OFF_SW);
  float* s_amax = reinterpret_cast<float*>(smem + Cfg::OFF_AMAX);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kG8Stages; ++s) {
      mbar_init(bar_full + 8 * s, 1);
      mbar_init(bar_empty + 8 * s, 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar_tfull + 8 * b, 1);
      mbar_init(bar_tempty + 8 * b, kEpiWarps);
    }
    mbar_init(bar_done, 1);
    *s_abort = 0;
    mbar_fence_init();
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmB0);
    if (MODE == 0) prefetch_tmap(&tmB1);
  }
  if (warp == 1) tmem_alloc(smem_u32(s_tslot), 512);
  pdl_wait();
  const int MT = build_mtile_starts(a.offsets, a.slot_of, a.E, a.C, a.rows_cap / kTileM, s_mt, s_tmp);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *s_tslot;

  const int K = MODE == 0 ? a.d : a.f;
  const int KS = K / 128;                      // K steps = scale blocks = stages per tile
  const int NT = MODE == 0 ? a.f / 128 : a.d / 256;
  const int tiles = MT * NT;

  if (warp == 0) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      uint32_t stage = 0, ph = 0;
      int issued = 0;
      bool ok = true;
      for (int tile = blockIdx.x; tile < tiles && ok; tile += gridDim.x) {
        const int mt = tile / NT, nt = tile % NT;
        const int e = expert_of_mtile(s_mt, a.E, mt);
        const int slot = a.slot_of ? a.slot_of[e] : e;
        const int brow = MODE == 0 ? slot * a.f + nt * 128 : slot * a.d + nt * 256;
        for (int ks = 0; ks < KS; ++ks) {
          if (!mbar_wait(bar_empty + 8 * stage, ph ^ 1, s_abort)) { ok = false; break; }
          const uint32_t fb = bar_full + 8 * stage;
          mbar_arrive_expect_tx(fb, Cfg::STAGE_TX);
          const uint32_t sA = sb + Cfg::OFF_A + stage * Cfg::A_BYTES;
          const uint32_t sB = sb + Cfg::OFF_B + stage * Cfg::B_BYTES;
          tma_load_2d(sA, &tmA, ks * 128, mt * kTileM, fb);
          if (MODE == 0) {
            tma_load_2d(sB, &tmB0, ks * 128, brow, fb);
            tma_load_2d(sB + 128 * 128, &tmB1, ks * 128, brow, fb);
          } else {
            tma_load_2d(sB, &tmB0, ks * 128, brow, fb);
          }
          ++issued;
          if (++stage == kG8Stages) { stage = 0; ph ^= 1; }
        }
      }
      if (!ok) {
        set_dev_err(DEV_ERR_TIMEOUT);
        *s_abort = 1;
        for (int i = 0; i < kG8Stages && i < issued; ++i) {
          if (stage == 0) { stage = kG8Stages; ph ^= 1; }
          --stage;
          mbar_wait(bar_full + 8 * stage, ph, nullptr);
        }
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer: one partial per K step, alternating TMEM buffers ----------------
    if (lane == 0) {
      uint32_t stage = 0, ph = 0, buf = 0, bph = 0;
      bool ok = true;
      for (int tile = blockIdx.x; tile < tiles && ok; tile += gridDim.x) {
        for (int ks = 0; ks < KS; ++ks) {
          if (!mbar_wait(bar_full + 8 * stage, ph, s_abort)) { ok = false; break; }
          if (!mbar_wait(bar_tempty + 8 * buf, bph ^ 1, s_abort)) { ok = false; break; }
          tc_fence_after();
          const uint32_t sA = sb + Cfg::OFF_A + stage * Cfg::A_BYTES;
          const uint32_t sB = sb + Cfg::OFF_B + stage * Cfg::B_BYTES;
          const uint32_t d_tmem = tmem + buf * 256;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            mma_f8(d_tmem, desc_sw128(sA + 32 * kk), desc_sw128(sB + 32 * kk), Cfg::IDESC, kk != 0);
          tc_commit(bar_empty + 8 * stage);
          tc_commit(bar_tfull + 8 * buf);
          if (++stage == kG8Stages) { stage = 0; ph ^= 1; }
          buf ^= 1;
          if (buf == 0) bph ^= 1;
        }
      }
      if (!ok) {
        set_dev_err(DEV_ERR_TIMEOUT);
        *s_abort = 1;
      }
      tc_commit(bar_done);
      mbar_wait(bar_done, 0, nullptr);
    }
  } else {
    // ---------------- epilogue: promotion of every K step, then the tile's epilogue ----------------
    const int q = warp & 3;
    const int half = (warp - 2) >> 2;
    const int r = q * 32 + lane;
    const int et = threadIdx.x - 64;          // epilogue thread 0..255
    // On a failed wait `ok` turns false; the loops keep their shape (every epilogue warp
    // reaches every named barrier) and skip the work.
    uint32_t buf = 0, bph = 0;
    bool ok = true;
    for (int tile = blockIdx.x; tile < tiles; tile += gridDim.x) {
      const int mt = tile / NT, nt = tile % NT;
      const int e = expert_of_mtile(s_mt, a.E, mt);
      const int slot = a.slot_of ? a.slot_of[e] : e;
      const int j = mt * kTileM + r;
      const int4 meta = MODE == 1 ? __ldg(a.rowmeta + j) : make_int4(-1, -1, 0, 0);   // used after the K loop
      // the tile's weight block scales (two 128-column blocks x KS steps)
      g8_epi_sync();
      for (int i = et; i < 2 * KS; i += kEpiWarps * 32) {
        const int blk = i / KS, kb = i % KS;
        float v;
        if (MODE == 0) v = (blk ? a.sw1 : a.sw0)[(size_t(slot) * (a.f / 128) + nt) * KS + kb];
        else v = a.sw0[(size_t(slot) * (a.d / 128) + 2 * nt + blk) * KS + kb];
        s_sw[blk * kG8MaxKB + kb] = v;
      }
      g8_epi_sync();
      float acc[2][64];
#pragma unroll
      for (int b = 0; b < 2; ++b)
#pragma unroll
        for (int i = 0; i < 64; ++i) acc[b][i] = 0.f;
      float sx_next = __ldcg(a.sx + j);
      for (int ks = 0; ks < KS; ++ks) {
        const float sx = sx_next;
        if (ks + 1 < KS) sx_next = __ldcg(a.sx + size_t(ks + 1) * a.rows_cap + j);
        if (ok && !mbar_wait(bar_tfull + 8 * buf, bph, s_abort)) {
          if (lane == 0) {
            set_dev_err(DEV_ERR_TIMEOUT);
            *s_abort = 1;
          }
          ok = false;
        }
        if (!ok) continue;
        tc_fence_after();
        const uint32_t tb = tmem + (uint32_t(q * 32) << 16) + buf * 256 + half * 64;
#pragma unroll
        for (int b = 0; b < 2; ++b) {
          const float sc = sx * s_sw[b * kG8MaxKB + ks];
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            uint32_t p0[16], p1[16];
            tc_ld16(tb + b * 128 + 32 * c, p0);
            tc_ld16(tb + b * 128 + 32 * c + 16, p1);
            tc_wait_ld();
            tc_reg_fence(p0);
            tc_reg_fence(p1);
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              acc[b][32 * c + i] = fmaf(__uint_as_float(p0[i]), sc, acc[b][32 * c + i]);
              acc[b][32 * c + 16 + i] = fmaf(__uint_as_float(p1[i]), sc, acc[b][32 * c + 16 + i]);
            }
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_tempty + 8 * buf);
        buf ^= 1;
        if (buf == 0) bph ^= 1;
      }
      if (MODE == 0) {
        // h = silu(g) * u over this thread's 64 columns, then E4M3 per (row, 128 columns)
        float amax = 0.f;
#pragma unroll
        for (int i = 0; i < 64; ++i) {
          const float g = acc[0][i];
          const float h = __fdividef(g, 1.f + __expf(-g)) * acc[1][i];
          acc[0][i] = h;
          amax = fmaxf(amax, fabsf(h));
        }
        s_amax[half * 128 + r] = amax;
        g8_epi_sync();
        amax = fmaxf(s_amax[r], s_amax[128 + r]);
        if (!ok) continue;
        const float s = amax / 448.0f;
        const float inv = s > 0.f ? 1.0f / s : 0.f;
        uint4* dst = reinterpret_cast<uint4*>(a.hq + size_t(j) * a.f + nt * 128 + half * 64);
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t w[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int o = 16 * c + 4 * i;
            w[i] = e4m3_code(acc[0][o] * inv) | (e4m3_code(acc[0][o + 1] * inv) << 8) |
                   (e4m3_code(acc[0][o + 2] * inv) << 16) | (e4m3_code(acc[0][o + 3] * inv) << 24);
          }
          dst[c] = make_uint4(w[0], w[1], w[2], w[3]);
        }
        if (half == 0) a.sh[size_t(nt) * a.rows_cap + j] = s;
      } else if (ok) {
        if (a.topk_w) {
          // fused combine: stage w * y (32 rows x 32 columns at a time), add row by row
          float* stg = reinterpret_cast<float*>(smem + Cfg::OFF_STG) + (warp - 2) * 32 * Cfg::STG_W;
          const int tok = meta.y;
          const float w = __int_as_float(meta.z);
#pragma unroll
          for (int b = 0; b < 2; ++b)
#pragma unroll
            for (int c = 0; c < 2; ++c) {
              float* my = stg + lane * Cfg::STG_W;
#pragma unroll
              for (int i4 = 0; i4 < 8; ++i4)
                reinterpret_cast<float4*>(my)[i4] =
                    make_float4(w * acc[b][32 * c + 4 * i4], w * acc[b][32 * c + 4 * i4 + 1],
                                w * acc[b][32 * c + 4 * i4 + 2], w * acc[b][32 * c + 4 * i4 + 3]);
              __syncwarp();
              const int col0 = nt * 256 + b * 128 + half * 64 + 32 * c;
              const int sub = lane >> 3, cl = lane & 7;   // 4 rows per instruction, 8 lanes x float4 per row
#pragma unroll 2
              for (int r0 = 0; r0 < 32; r0 += 4) {
                const int rr = r0 + sub;
                const int t_r = __shfl_sync(0xFFFFFFFFu, tok, rr);
                const float4 val = reinterpret_cast<const float4*>(stg + rr * Cfg::STG_W)[cl];
                if (t_r >= 0) atomicAdd(reinterpret_cast<float4*>(a.out + size_t(t_r) * a.d + col0) + cl, val);
              }
              __syncwarp();
            }
        } else if (meta.x >= 0) {
          float* dst = a.out + size_t(meta.x) * a.d + nt * 256 + half * 64;
#pragma unroll
          for (int b = 0; b < 2; ++b)
#pragma unroll
            for (int i4 = 0; i4 < 16; ++i4)
              reinterpret_cast<float4*>(dst + b * 128)[i4] =
                  make_float4(acc[b][4 * i4], acc[b][4 * i4 + 1], acc[b][4 * i4 + 2], acc[b][4 * i4 + 3]);
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, 512);
}

}  // namespace ftmoe
