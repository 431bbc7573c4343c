// a3 + a4 (+a5) prefill path: the grouped SwiGLU expert FFN on tcgen05
// block-scaled tensor cores with NVFP4 activations.
//
// Pages: resident experts run on GPU tensor cores from expert slots, with
// NVFP4 among the weight formats (zubnet.ai, "FreeToken, Unsloth GGUF ...
// consumer hardware"); a prefill chunk of 8,192 tokens touches nearly every
// expert (asapai.co.kr, "Running 753B GLM-5.2 on a single workstation GPU",
// section "Abandoning fixed offloading in favor of measured bandwidth";
// banandre.com, "The 284B Model on a 32GB GPU Trick", section "The Three
// Failure Modes").  With hundreds of rows per expert the expert FFN is a
// dense contraction, so it runs as a grouped GEMM.
//
// FP4 tensor cores need both operands in a block-scaled 4-bit format, and the
// pages say nothing about activations.  The library's rule (one E4M3 scale
// per 16 elements, s = E4M3(amax / 6), q = E2M1(v / s), tensor scale 1) is
// applied to the gathered rows of x and to h.
//
// Rows.  The P = T*k pairs are in expert-sorted order (ftmoe_permute).  Each
// resident expert's rows are padded to a multiple of 128 ("M-tiles"), so an
// M-tile never mixes experts.  The padded row index of the i-th row of
// expert e is 128 * mt[e] + i, with mt[e] = sum over earlier resident
// experts of ceil(rows / 128).
//
// Scale factors.  An MMA with K = 64 reads four scales per row from tensor
// memory: row r of a 128-row block at lane r % 32 (every 32-lane quarter
// holds the same copy), column r / 32, byte = 16-element block within the
// 64.  In global memory one 128-row block of one K = 64 step is 512 bytes:
// byte (r % 32) * 16 + (r / 32) * 4 + kb.  tcgen05.cp moves such a block from
// shared memory into 4 TMEM columns.  Weight scales are repacked into this
// layout once (ftmoe_prepare_weights); activation scales are written in it.
//
// Kernels (one stream, in order):
//   quantize_act_kernel x -> per-token E2M1 codes + E4M3 scales (once per token)
//   actq_gather_kernel  padded rows <- the tokens' codes; scales into scale blocks
//   gemm_kernel<0, NH>  [gate | up] tile of N = 2 NH columns; epilogue
//                       h = silu(g) * u, quantised to codes + scale blocks
//   gemm_kernel<1, 128> down tile of 128 columns; epilogue adds w * y into
//                       out[token] (fused combine) or writes y in sorted order
//
// GEMM CTA (persistent, one per SM, static round robin over tiles):
//   warp 0      TMA producer: A, B tiles (128-byte swizzle) and scale blocks
//               into a kStages-deep shared-memory ring
//   warp 1      TMEM owner and MMA issuer (one thread)
//   warps 2-17  epilogue; warp w reads TMEM lanes 32 * (w % 4) .. + 31, a
//               quarter of each matrix's columns
//   warps 18-21 scale writers: each stage's scale blocks, shared memory ->
//               registers -> TMEM (tcgen05.st, one lane quarter per warp)
// TMEM: the down GEMM (N = 128) double-buffers its accumulator (columns 0 and
// 256) with the scale blocks of the stage in flight right after each (two
// buffers alternate); the gate/up GEMM (N = 256) has one accumulator at column
// 0, handed back as soon as the 16 epilogue warps hold it, and its two scale
// buffers from column 256.  Measured on B300: writing the scales with tcgen05.st from the
// scale warps costs the MMA issuer nothing, while tcgen05.cp copies issued
// between its MMAs serialise with them (the 8192-token gate/up GEMM spent
// ~80 us of ~210 us on them).
#pragma once
#include "tc.cuh"
#include "permute.cuh"

namespace ftmoe {

constexpr int kTileM = 128;
constexpr int kStages = 4;
constexpr int kEpiWarps = 8;
constexpr int kGemmThreads = (2 + kEpiWarps) * 32;
constexpr int kSfWarps = 4;                                  // FP4 GEMM: scale writers
constexpr int kNvEpiWarps = 16;                              // FP4 GEMM: epilogue warps (4 per lane quarter)
constexpr int kGemmNvThreads = (2 + kNvEpiWarps + kSfWarps) * 32;
constexpr int kStageK = 256;            // FP4 elements per stage (128 bytes per row)
constexpr int kSfBlock = 512;           // bytes of one 128-row x K=64 scale block

// s_mt[e] = first M-tile of expert e (resident experts with rows only); s_mt[E] = total.
// The total is clamped to max_mt (the workspace's row capacity / 128).
__device__ __forceinline__ int build_mtile_starts(const int32_t* offsets, const int32_t* slot_of, int E, int C,
                                                  int max_mt, int* s_mt, int* s_tmp) {
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    const int n = offsets[e + 1] - offsets[e];
    int slot = slot_of ? slot_of[e] : e;
    if (slot >= C) {
      if (n > 0) set_dev_err(DEV_ERR_BAD_SLOT);
      slot = -1;
    }
    s_mt[e] = (n > 0 && slot >= 0) ? (n + kTileM - 1) / kTileM : 0;
  }
  __syncthreads();
  int total = block_exclusive_scan(s_mt, E, s_tmp);
  if (total > max_mt) {
    if (threadIdx.x == 0) set_dev_err(DEV_ERR_ROWS);
    total = max_mt;
  }
  if (threadIdx.x == 0) s_mt[E] = total;
  __syncthreads();
  return total;
}

// largest e with s_mt[e] <= mt (experts with no tiles have s_mt[e] == s_mt[e+1])
__device__ __forceinline__ int expert_of_mtile(const int* s_mt, int E, int mt) {
  int lo = 0, hi = E - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (s_mt[mid] <= mt) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// byte offset of (row r of its 128-row block, 16-element block kb16 of the row) inside the
// scale blocks of a matrix with K/64 steps: [row / 128][kb16 / 4][512]
__device__ __forceinline__ size_t sf_offset(int row, int kb16, int ksteps) {
  const int r = row & 127;
  return (size_t(row >> 7) * ksteps + (kb16 >> 2)) * kSfBlock + (r & 31) * 16 + (r >> 5) * 4 + (kb16 & 3);
}

// NVFP4 quantisation of 16 values: returns the E4M3 scale code, codes in c (element 2i in the
// low nibble of byte i).  s = E4M3_rn_satfinite(amax / 6); q = E2M1_rn_satfinite(v / s), or a
// zero of v's sign when s == 0.  Divisions are IEEE fp32.
__device__ __forceinline__ uint32_t quant_nvfp4_16(const float (&v)[16], uint2& c) {
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(v[i]));
  const uint32_t sc = e4m3_code(amax / 6.0f);
  const float s = e4m3_to_float(uint8_t(sc));
  uint32_t b[8];
  if (s > 0.f) {
#pragma unroll
    for (int i = 0; i < 8; ++i) b[i] = e2m1x2(v[2 * i] / s, v[2 * i + 1] / s);
  } else {
#pragma unroll
    for (int i = 0; i < 8; ++i) b[i] = e2m1x2(copysignf(0.f, v[2 * i]), copysignf(0.f, v[2 * i + 1]));
  }
  c.x = b[0] | (b[1] << 8) | (b[2] << 16) | (b[3] << 24);
  c.y = b[4] | (b[5] << 8) | (b[6] << 16) | (b[7] << 24);
  return sc;
}

// The same block quantisation for h inside the GEMM epilogue: one division per
// block (1 / s), then products.  h codes are not compared bit for bit (h is
// computed in a different order than the oracle's anyway), so a product that
// differs from the quotient by an ulp only matters at exact rounding ties.
__device__ __forceinline__ uint32_t quant_nvfp4_16_fast(const float (&v)[16], uint2& c) {
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(v[i]));
  const uint32_t sc = e4m3_code(amax / 6.0f);
  const float s = e4m3_to_float(uint8_t(sc));
  const float inv = s > 0.f ? 1.0f / s : 0.f;
  uint32_t b[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) b[i] = e2m1x2(v[2 * i] * inv, v[2 * i + 1] * inv);
  c.x = b[0] | (b[1] << 8) | (b[2] << 16) | (b[3] << 24);
  c.y = b[4] | (b[5] << 8) | (b[6] << 16) | (b[7] << 24);
  return sc;
}

// ---------------------------------------------------------------------------
// a3: gather + quantise the padded rows of x
// ---------------------------------------------------------------------------
struct ActqArgs {
  const uint8_t* xq_tok;   // per-token codes [T][d/2] (quantize_act_kernel)
  const uint8_t* sf_tok;   // per-token scales [T][d/16]
  int T, d, k, E, C, P;
  const int32_t* offsets;
  const int32_t* sorted_pair;
  const int32_t* slot_of;
  uint8_t* xq;        // [rows_cap][d/2]
  uint8_t* sfa;       // [rows_cap/128][d/64][512]
  int rows_cap;
  float4* zero_out;   // optional: zeroed first (T*d/4 float4)
  long long zero_n4;
  const float* topk_w;   // or nullptr
  int4* rowmeta;         // [rows_cap] per padded row (row_meta)
};

// Per padded row, for the down GEMM's epilogue: {sorted index of the pair or -1, token or -1,
// the pair's combine weight (fp32 bits; 0 without topk_w), 0}.  Written by the gather kernel,
// which reads the sorted pairs anyway, so the epilogue needs one load per row instead of a
// chain of three (offsets -> sorted pair -> weight).
__device__ __forceinline__ int4 row_meta(int yrow, int p, int k, const float* topk_w) {
  return make_int4(yrow, p >= 0 ? p / k : -1, (p >= 0 && topk_w) ? __float_as_int(topk_w[p]) : 0, 0);
}

constexpr int kActqWarps = 8;

// One warp per 32 consecutive padded rows: lane i first resolves row j0 + i (expert, sorted
// pair, token) so the warp pays the chain of dependent loads once per 32 rows, writes the row's
// metadata and its scale words, then the warp copies the 32 rows' codes 16 bytes per lane.
__global__ void __launch_bounds__(kActqWarps * 32) actq_gather_kernel(ActqArgs a) {
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
  const int nb = a.d / 16;           // scale bytes per row
  const int ksteps = a.d / 64;       // scale words per row
  const int row_bytes = a.d / 2;
  const int n16 = row_bytes / 16;    // 16-byte pieces of a row's codes
  const int rows = MT * kTileM;      // a multiple of 32
  for (int j0 = (blockIdx.x * kActqWarps + (threadIdx.x >> 5)) * 32; j0 < rows; j0 += gridDim.x * kActqWarps * 32) {
    const int j = j0 + lane;
    const int e = expert_of_mtile(s_mt, a.E, j / kTileM);
    const int i = j - s_mt[e] * kTileM;
    const int lo = a.offsets[e];
    int tok = -1;
    int4 meta = make_int4(-1, -1, 0, 0);
    if (i < a.offsets[e + 1] - lo) {
      int p = a.sorted_pair[lo + i];
      if (p >= 0 && p < a.P) {
        tok = p / a.k;
      } else {
        set_dev_err(DEV_ERR_BAD_PAIR);
        p = -1;
      }
      meta = row_meta(lo + i, p, a.k, a.topk_w);
    }
    a.rowmeta[j] = meta;
    // scale words of row j: the four E4M3 scales of K = 64 step ks (little-endian) go to byte
    // (r % 32) * 16 + (r / 32) * 4 of the step's 512-byte block
    {
      const uint32_t* ss = reinterpret_cast<const uint32_t*>(a.sf_tok + size_t(tok < 0 ? 0 : tok) * nb);
      const int r = j & (kTileM - 1);
      uint8_t* blk = a.sfa + size_t(j / kTileM) * ksteps * kSfBlock + (r & 31) * 16 + (r >> 5) * 4;
#pragma unroll 8
      for (int ks = 0; ks < ksteps; ++ks)
        *reinterpret_cast<uint32_t*>(blk + size_t(ks) * kSfBlock) = tok >= 0 ? __ldg(ss + ks) : 0u;
    }
    // codes of the 32 rows, four rows' loads in flight at a time
    for (int r0 = 0; r0 < 32; r0 += 4) {
      int tr[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) tr[q] = __shfl_sync(0xFFFFFFFFu, tok, r0 + q);
      for (int c0 = 0; c0 < n16; c0 += 64) {
        uint4 v[4][2];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const uint4* src = reinterpret_cast<const uint4*>(a.xq_tok + size_t(tr[q] < 0 ? 0 : tr[q]) * row_bytes);
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const int c = c0 + 32 * h + lane;
            v[q][h] = (tr[q] >= 0 && c < n16) ? __ldg(src + c) : make_uint4(0u, 0u, 0u, 0u);
          }
        }
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          uint4* dst = reinterpret_cast<uint4*>(a.xq + size_t(j0 + r0 + q) * row_bytes);
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const int c = c0 + 32 * h + lane;
            if (c < n16) dst[c] = v[q][h];
          }
        }
      }
    }
  }
}

// The same rule in token order with plain layouts (ftmoe_quantize_act):
// codes [T][d/2], scales [T][d/16].  One warp per row.
__global__ void __launch_bounds__(kActqWarps * 32)
quantize_act_kernel(const uint16_t* x, int T, int d, uint8_t* codes, uint8_t* scales) {
  pdl_wait();
  const int lane = threadIdx.x & 31;
  const int nb = d / 16;
  for (int t = blockIdx.x * kActqWarps + (threadIdx.x >> 5); t < T; t += gridDim.x * kActqWarps) {
    for (int b = lane; b < nb; b += 32) {
      const uint4* src = reinterpret_cast<const uint4*>(x + size_t(t) * d + 16 * b);
      const uint4 v0 = __ldg(src), v1 = __ldg(src + 1);
      const uint32_t w[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
      float f[16];
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        f[2 * q] = bf16_lo(w[q]);
        f[2 * q + 1] = bf16_hi(w[q]);
      }
      uint2 c;
      const uint32_t sc = quant_nvfp4_16(f, c);
      reinterpret_cast<uint2*>(codes + size_t(t) * (d / 2))[b] = c;
      scales[size_t(t) * nb + b] = uint8_t(sc);
    }
  }
}

// ---------------------------------------------------------------------------
// Weight scale repack (ftmoe_prepare_weights): canonical E4M3 [N][K/16] -> scale blocks
// ---------------------------------------------------------------------------
// gate/up: per slot, per N-tile of NH gate rows + NH up rows, in ceil(2 NH / 128)
// 128-row blocks (rows past 2 NH zero): [C][f/NH][d/64][atoms][512]
// down: [C][d/128][f/64][512]
__global__ void prep_sf_gate_up_kernel(const uint8_t* gs, const uint8_t* us, int C, int d, int f, int nh,
                                       uint8_t* out) {
  const int ks = d / 64, nt = f / nh, atoms = (2 * nh + 127) / 128;
  const long long total = (long long)C * nt * ks * atoms * kSfBlock;
  for (long long o = (long long)blockIdx.x * blockDim.x + threadIdx.x; o < total; o += (long long)gridDim.x * blockDim.x) {
    long long t = o;
    const int pos = int(t % kSfBlock); t /= kSfBlock;
    const int atom = int(t % atoms); t /= atoms;
    const int kst = int(t % ks); t /= ks;
    const int n = int(t % nt); t /= nt;
    const int slot = int(t);
    const int r = atom * 128 + ((pos & 15) >> 2) * 32 + (pos >> 4);
    const int kb = kst * 4 + (pos & 3);
    uint8_t v = 0;
    if (r < nh) v = gs[(size_t(slot) * f + n * nh + r) * (d / 16) + kb];
    else if (r < 2 * nh) v = us[(size_t(slot) * f + n * nh + (r - nh)) * (d / 16) + kb];
    out[o] = v;
  }
}

__global__ void prep_sf_down_kernel(const uint8_t* ds, int C, int d, int f, uint8_t* out) {
  const int ks = f / 64, nt = d / 128;
  const long long total = (long long)C * nt * ks * kSfBlock;
  for (long long o = (long long)blockIdx.x * blockDim.x + threadIdx.x; o < total; o += (long long)gridDim.x * blockDim.x) {
    long long t = o;
    const int pos = int(t % kSfBlock); t /= kSfBlock;
    const int kst = int(t % ks); t /= ks;
    const int n = int(t % nt); t /= nt;
    const int slot = int(t);
    const int r = ((pos & 15) >> 2) * 32 + (pos >> 4);
    out[o] = ds[(size_t(slot) * d + n * 128 + r) * (f / 16) + kst * 4 + (pos & 3)];
  }
}

// ---------------------------------------------------------------------------
// grouped block-scaled GEMM
// ---------------------------------------------------------------------------
struct GemmArgs {
  int E, k, d, f, C, P;
  int rows_cap;
  const int32_t* offsets;
  const int32_t* sorted_pair;
  const int32_t* slot_of;
  const uint8_t* sfa;       // activation scale blocks [rows_cap/128][K/64][512]
  const uint8_t* sfb;       // prepared weight scale blocks
  const float* tscale;      // [C][3]
  uint8_t* hq;              // MODE 0: h codes [rows_cap][f/2]
  uint8_t* sfh;             // MODE 0: h scale blocks [rows_cap/128][f/64][512]
  const float* topk_w;      // MODE 1: fused combine weights, or nullptr (write y)
  float* out;               // MODE 1: out [T][d] (fused) or y [P][d] (sorted)
  const int4* rowmeta;      // MODE 1: row_meta of each padded row
};

template <int MODE, int NH>
struct GemmCfg {
  static constexpr int N = MODE == 0 ? 2 * NH : NH;      // MMA N
  static constexpr int A_BYTES = kTileM * 128;
  static constexpr int B_BYTES = N * 128;
  static constexpr int SFA_BYTES = 4 * kSfBlock;
  static constexpr int SFB_ATOMS = (N + 127) / 128;
  static constexpr int SFB_BYTES = 4 * SFB_ATOMS * kSfBlock;
  static constexpr int STAGE_TX = A_BYTES + B_BYTES;        // on full[s]
  static constexpr int SF_TX = SFA_BYTES + SFB_BYTES;         // on sfld[s]
  static constexpr int OFF_A = 0;
  static constexpr int OFF_B = OFF_A + kStages * A_BYTES;
  static constexpr int OFF_SFA = OFF_B + kStages * B_BYTES;
  static constexpr int OFF_SFB = OFF_SFA + kStages * SFA_BYTES;
  // full[S], empty[S], tfull[2], tempty[2], done, sf_full[2], sf_free[2], sfld[S]
  static constexpr int OFF_BAR = OFF_SFB + kStages * SFB_BYTES;
  static constexpr int OFF_MISC = OFF_BAR + (3 * kStages + 9) * 8;
  // TMEM columns of one stage's scales: SFA 4 per K = 64 step, then SFB 4 per step and 128-row
  // atom.  Two accumulators (columns 0 and 256) when an accumulator and a scale buffer fit in
  // 256 columns, the scale buffers right after each; else one accumulator at column 0 and the
  // two scale buffers from column 256.
  static constexpr int SF_COLS = 16 + 16 * SFB_ATOMS;
  static constexpr int ACC_BUFS = N + SF_COLS <= 256 ? 2 : 1;
  // epilogue warps at work: all 16 for gate/up; 8 for the down GEMM, whose combine then issues
  // half as many (and twice as long) bulk reductions (measured faster)
  static constexpr int EPI_ACTIVE = MODE == 0 ? kNvEpiWarps : 8;
  static constexpr int EPI_COLS = NH / (EPI_ACTIVE / 4);        // columns of each matrix per epilogue warp
  __host__ __device__ static constexpr uint32_t sf_col(uint32_t buf) {
    return ACC_BUFS == 2 ? buf * 256 + N : 256 + buf * SF_COLS;
  }
  static constexpr int OFF_MT = OFF_MISC + 16;                     // int s_mt[1025], s_tmp[33]
  // MODE 1: per epilogue warp, its 32 rows x EPI_COLS columns of the tile (row stride padded by 4 floats)
  static constexpr int STG_STRIDE = EPI_COLS + 4;
  static constexpr int OFF_STG = (OFF_MT + (1025 + 33) * 4 + 15) / 16 * 16;
  static constexpr int STG_BYTES = MODE == 1 ? EPI_ACTIVE * 32 * STG_STRIDE * 4 : 0;
  static constexpr int SMEM = OFF_STG + STG_BYTES + 1024;        // + alignment slack
  static constexpr uint32_t IDESC = idesc_mxf4(kTileM, N, 0);
  static_assert(N % 16 == 0 && N <= 256, "MMA N");
  static_assert(ACC_BUFS == 2 || N + 2 * SF_COLS <= 512 - 256 + N, "accumulators + scale columns within 512 TMEM columns");
  static_assert(ACC_BUFS == 2 || 256 + 2 * SF_COLS <= 512, "scale buffers after the single accumulator");
  static_assert(EPI_COLS % 16 == 0, "whole 16-column TMEM loads per epilogue warp");
  static_assert(B_BYTES % 1024 == 0 && A_BYTES % 1024 == 0, "1024-byte aligned stage buffers");
  static_assert(SMEM <= 232448, "one CTA's opt-in shared memory");
  static_assert(STAGE_TX < (1 << 20), "an mbarrier's transaction count");
  static_assert(OFF_BAR % 8 == 0, "8-byte aligned mbarriers");
};

template <int MODE, int NH>
__global__ void __launch_bounds__(kGemmNvThreads, 1)
gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB0,
            const __grid_constant__ CUtensorMap tmB1, GemmArgs a) {
  using Cfg = GemmCfg<MODE, NH>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sb = smem_u32(smem);
  const uint32_t bar_full = sb + Cfg::OFF_BAR, bar_empty = bar_full + 8 * kStages;
  const uint32_t bar_tfull = bar_empty + 8 * kStages, bar_tempty = bar_tfull + 16, bar_done = bar_tempty + 16;
  const uint32_t bar_sffull = bar_done + 8, bar_sffree = bar_sffull + 16, bar_sfld = bar_sffree + 16;
  uint32_t* s_tslot = reinterpret_cast<uint32_t*>(smem + Cfg::OFF_MISC);
  volatile int* s_abort = reinterpret_cast<volatile int*>(smem + Cfg::OFF_MISC + 4);
  int* s_mt = reinterpret_cast<int*>(smem + Cfg::OFF_MT);
  int* s_tmp = s_mt + 1025;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(bar_full + 8 * s, 1);
      mbar_init(bar_empty + 8 * s, 1);
      mbar_init(bar_sfld + 8 * s, 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar_tfull + 8 * b, 1);
      mbar_init(bar_tempty + 8 * b, Cfg::EPI_ACTIVE);
      mbar_init(bar_sffull + 8 * b, kSfWarps);
      mbar_init(bar_sffree + 8 * b, 1);
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
  const int KS = K / kStageK;                 // stages per tile
  const int ksteps = K / 64;                  // K = 64 steps per row
  const int NT = MODE == 0 ? a.f / NH : a.d / NH;
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
        const int brow = slot * (MODE == 0 ? a.f : a.d) + nt * NH;
        const uint8_t* sfa_src = a.sfa + size_t(mt) * ksteps * kSfBlock;
        const uint8_t* sfb_src = a.sfb + (size_t(slot) * NT + nt) * ksteps * Cfg::SFB_ATOMS * kSfBlock;
        for (int ks = 0; ks < KS; ++ks) {
          if (!mbar_wait(bar_empty + 8 * stage, ph ^ 1, s_abort)) { ok = false; break; }
          // the scales first, on their own barrier: the scale warps can move them into TMEM
          // before the (larger) A and B tiles have landed
          const uint32_t fs = bar_sfld + 8 * stage;
          mbar_arrive_expect_tx(fs, Cfg::SF_TX);
          bulk_load(sb + Cfg::OFF_SFA + stage * Cfg::SFA_BYTES, sfa_src + size_t(ks) * Cfg::SFA_BYTES,
                    Cfg::SFA_BYTES, fs);
          bulk_load(sb + Cfg::OFF_SFB + stage * Cfg::SFB_BYTES, sfb_src + size_t(ks) * Cfg::SFB_BYTES,
                    Cfg::SFB_BYTES, fs);
          const uint32_t fb = bar_full + 8 * stage;
          mbar_arrive_expect_tx(fb, Cfg::STAGE_TX);
          const uint32_t sA = sb + Cfg::OFF_A + stage * Cfg::A_BYTES;
          const uint32_t sB = sb + Cfg::OFF_B + stage * Cfg::B_BYTES;
          tma_load_2d(sA, &tmA, ks * 128, mt * kTileM, fb);
          tma_load_2d(sB, &tmB0, ks * 128, brow, fb);
          if (MODE == 0) tma_load_2d(sB + NH * 128, &tmB1, ks * 128, brow, fb);
          ++issued;
          if (++stage == kStages) { stage = 0; ph ^= 1; }
        }
      }
      if (!ok) {
        set_dev_err(DEV_ERR_TIMEOUT);
        *s_abort = 1;
        // let the copies already issued land before the CTA can exit
        for (int i = 0; i < kStages && i < issued; ++i) {
          if (stage == 0) { stage = kStages; ph ^= 1; }
          --stage;
          mbar_wait(bar_full + 8 * stage, ph, nullptr);
          mbar_wait(bar_sfld + 8 * stage, ph, nullptr);
        }
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      uint32_t stage = 0, ph = 0, acc = 0, aph = 0, sfbuf = 0, sfph = 0;
      bool ok = true;
      for (int tile = blockIdx.x; tile < tiles && ok; tile += gridDim.x) {
        if (!mbar_wait(bar_tempty + 8 * acc, aph ^ 1, s_abort)) { ok = false; break; }
        tc_fence_after();
        const uint32_t d_tmem = tmem + acc * 256;      // acc stays 0 with one accumulator
        for (int ks = 0; ks < KS; ++ks) {
          if (!mbar_wait(bar_full + 8 * stage, ph, s_abort) || !mbar_wait(bar_sffull + 8 * sfbuf, sfph, s_abort)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sA = sb + Cfg::OFF_A + stage * Cfg::A_BYTES;
          const uint32_t sB = sb + Cfg::OFF_B + stage * Cfg::B_BYTES;
          const uint32_t sf_col = tmem + Cfg::sf_col(sfbuf);   // written by the scale warps
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            mma_nvf4(d_tmem, desc_sw128(sA + 32 * kk), desc_sw128(sB + 32 * kk), Cfg::IDESC, sf_col + 4 * kk,
                     sf_col + 16 + 4 * Cfg::SFB_ATOMS * kk, (ks | kk) != 0);
          tc_commit(bar_empty + 8 * stage);
          tc_commit(bar_sffree + 8 * sfbuf);
          sfbuf ^= 1;
          if (sfbuf == 0) sfph ^= 1;
          if (++stage == kStages) { stage = 0; ph ^= 1; }
        }
        if (!ok) break;
        tc_commit(bar_tfull + 8 * acc);
        if (Cfg::ACC_BUFS == 2) {
          acc ^= 1;
          if (acc == 0) aph ^= 1;
        } else {
          aph ^= 1;
        }
      }
      if (!ok) {
        set_dev_err(DEV_ERR_TIMEOUT);
        *s_abort = 1;
      }
      // every MMA of this CTA has completed before TMEM is released
      tc_commit(bar_done);
      mbar_wait(bar_done, 0, nullptr);
    }
  } else if (warp >= 2 + kNvEpiWarps) {
    // ---------------- scale writers ----------------
    // Lane l of the warp of quarter q writes TMEM lane 32 q + l: in every quarter, column
    // c of a K = 64 step holds bytes 16 l + 4 c .. + 3 of the step's 512-byte scale block
    // (the scales of row 32 c + l), the layout the block-scaled MMA reads.
    const int q = warp & 3;
    const uint32_t lane_base = tmem + (uint32_t(q * 32) << 16);
    uint32_t stage = 0, ph = 0, sfbuf = 0, sfph = 0;
    bool ok = true;
    for (int tile = blockIdx.x; tile < tiles && ok; tile += gridDim.x) {
      for (int ks = 0; ks < KS; ++ks) {
        if (!mbar_wait_warp(bar_sfld + 8 * stage, ph, s_abort) ||
            !mbar_wait_warp(bar_sffree + 8 * sfbuf, sfph ^ 1, s_abort)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint4* sfa = reinterpret_cast<const uint4*>(smem + Cfg::OFF_SFA + stage * Cfg::SFA_BYTES) + lane;
        const uint4* sfb = reinterpret_cast<const uint4*>(smem + Cfg::OFF_SFB + stage * Cfg::SFB_BYTES) + lane;
        uint32_t v[16];
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          const uint4 w = sfa[kk * (kSfBlock / 16)];
          v[4 * kk] = w.x; v[4 * kk + 1] = w.y; v[4 * kk + 2] = w.z; v[4 * kk + 3] = w.w;
        }
        const uint32_t col = lane_base + Cfg::sf_col(sfbuf);
        tc_st16(col, v);
#pragma unroll
        for (int h = 0; h < Cfg::SFB_ATOMS; ++h) {
#pragma unroll
          for (int i = 0; i < 4; ++i) {      // blocks 4h .. 4h + 3 in (kk, atom) order
            const uint4 w = sfb[(4 * h + i) * (kSfBlock / 16)];
            v[4 * i] = w.x; v[4 * i + 1] = w.y; v[4 * i + 2] = w.z; v[4 * i + 3] = w.w;
          }
          tc_st16(col + 16 + 16 * h, v);
        }
        tc_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_sffull + 8 * sfbuf);
        sfbuf ^= 1;
        if (sfbuf == 0) sfph ^= 1;
        if (++stage == kStages) { stage = 0; ph ^= 1; }
      }
    }
    if (!ok && lane == 0) {
      set_dev_err(DEV_ERR_TIMEOUT);
      *s_abort = 1;
    }
  } else {
    // ---------------- epilogue ----------------
    const int q = warp & 3;             // TMEM lane quarter of this warp
    const int part = (warp - 2) >> 2;   // which part of each matrix's columns (EPI_COLS each)
    const int r = q * 32 + lane;        // row within the M-tile
    uint32_t acc = 0, aph = 0;
    // warps beyond the active ones have no columns (the down GEMM)
    for (int tile = part < Cfg::EPI_ACTIVE / 4 ? int(blockIdx.x) : tiles; tile < tiles; tile += gridDim.x) {
      const int mt = tile / NT, nt = tile % NT;
      const int e = expert_of_mtile(s_mt, a.E, mt);
      const int slot = a.slot_of ? a.slot_of[e] : e;
      // tensor scales: gate and up (MODE 0), down (MODE 1); loaded before the wait
      const float ts0 = a.tscale ? a.tscale[slot * 3 + (MODE == 0 ? 0 : 2)] : 1.f;
      const float ts1 = (MODE == 0 && a.tscale) ? a.tscale[slot * 3 + 1] : 1.f;
      const int j = mt * kTileM + r;   // padded row
      const int4 meta = MODE == 1 ? __ldg(a.rowmeta + j) : make_int4(-1, -1, 0, 0);
      if (!mbar_wait(bar_tfull + 8 * acc, aph, s_abort)) {
        if (lane == 0) {
          set_dev_err(DEV_ERR_TIMEOUT);
          *s_abort = 1;
        }
        break;
      }
      tc_fence_after();
      const uint32_t tb = tmem + (uint32_t(q * 32) << 16) + acc * 256;
      // the accumulator goes back to the MMA issuer as soon as its values are in registers
      auto release = [&]() {
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_tempty + 8 * acc);
      };
      if (MODE == 0) {
        constexpr int NB = Cfg::EPI_COLS / 16;    // 16-column blocks per warp
        uint32_t g[NB][16], u[NB][16];
#pragma unroll
        for (int b = 0; b < NB; ++b) {
          tc_ld16(tb + part * Cfg::EPI_COLS + 16 * b, g[b]);
          tc_ld16(tb + NH + part * Cfg::EPI_COLS + 16 * b, u[b]);
        }
        tc_wait_ld();
#pragma unroll
        for (int b = 0; b < NB; ++b) {
          tc_reg_fence(g[b]);
          tc_reg_fence(u[b]);
        }
        release();
        const float tsg = ts0, tsu = ts1;
        const int fsteps = a.f / 64;
#pragma unroll
        for (int b = 0; b < NB; ++b) {
          float hv[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float gg = __uint_as_float(g[b][i]) * tsg;
            const float uu = __uint_as_float(u[b][i]) * tsu;
            hv[i] = __fdividef(gg, 1.f + __expf(-gg)) * uu;
          }
          uint2 c;
          const uint32_t sc = quant_nvfp4_16_fast(hv, c);
          const int col = nt * NH + part * Cfg::EPI_COLS + 16 * b;
          *reinterpret_cast<uint2*>(a.hq + size_t(j) * (a.f / 2) + col / 2) = c;
          a.sfh[sf_offset(j, col / 16, fsteps)] = uint8_t(sc);
        }
      } else if (!a.topk_w) {
        // y in sorted order
        constexpr int NB = Cfg::EPI_COLS / 16;
        uint32_t v[NB][16];
#pragma unroll
        for (int b = 0; b < NB; ++b) tc_ld16(tb + part * Cfg::EPI_COLS + 16 * b, v[b]);
        tc_wait_ld();
#pragma unroll
        for (int b = 0; b < NB; ++b) tc_reg_fence(v[b]);
        release();
        if (meta.x >= 0) {
          const float tsd = ts0;
          float* dst = a.out + size_t(meta.x) * a.d + nt * NH + part * Cfg::EPI_COLS;
#pragma unroll
          for (int b = 0; b < NB; ++b)
#pragma unroll
            for (int i4 = 0; i4 < 4; ++i4)
              reinterpret_cast<float4*>(dst + 16 * b)[i4] =
                  make_float4(tsd * __uint_as_float(v[b][4 * i4]), tsd * __uint_as_float(v[b][4 * i4 + 1]),
                              tsd * __uint_as_float(v[b][4 * i4 + 2]), tsd * __uint_as_float(v[b][4 * i4 + 3]));
        }
      }
      if (MODE == 1 && a.topk_w) {
        // Fused combine.  Each lane stages w * y of its row in shared memory and hands it to
        // one asynchronous bulk reduce-add into out[token] (the reductions run beside the next
        // tile's epilogue; a lane's staging row is rewritten only after its reduction read it).
        constexpr int NB = Cfg::EPI_COLS / 16;
        constexpr int HC = Cfg::EPI_COLS;           // columns of this warp
        float* stg = reinterpret_cast<float*>(smem + Cfg::OFF_STG) + (warp - 2) * 32 * Cfg::STG_STRIDE;
        const int tok = meta.y;
        const float w = __int_as_float(meta.z) * ts0;
        uint32_t v[NB][16];
#pragma unroll
        for (int b = 0; b < NB; ++b) tc_ld16(tb + part * HC + 16 * b, v[b]);
        tc_wait_ld();
#pragma unroll
        for (int b = 0; b < NB; ++b) tc_reg_fence(v[b]);
        release();
        // the staging of the previous tile has been read by its bulk reductions
        bulk_wait_read0();
        __syncwarp();
        float* my = stg + lane * Cfg::STG_STRIDE;
#pragma unroll
        for (int b = 0; b < NB; ++b)
#pragma unroll
          for (int i4 = 0; i4 < 4; ++i4)
            reinterpret_cast<float4*>(my + 16 * b)[i4] =
                make_float4(w * __uint_as_float(v[b][4 * i4]), w * __uint_as_float(v[b][4 * i4 + 1]),
                            w * __uint_as_float(v[b][4 * i4 + 2]), w * __uint_as_float(v[b][4 * i4 + 3]));
        // each lane's row, HC floats, is added into out[token] by one bulk reduction
        fence_proxy_async_smem();
        if (tok >= 0) {
          bulk_reduce_add_f32(a.out + size_t(tok) * a.d + nt * NH + part * HC, smem_u32(my), uint32_t(HC * 4));
        }
        bulk_commit();
      }
      if (Cfg::ACC_BUFS == 2) {
        acc ^= 1;
        if (acc == 0) aph ^= 1;
      } else {
        aph ^= 1;
      }
    }
    if (MODE == 1) bulk_wait0();   // the fused combine's reductions have completed
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, 512);
}

}  // namespace ftmoe
