// a1 for long batches: router logits on tcgen05 tensor cores, then a per-token bound that
// narrows the experts whose order-R logits are needed to a few candidates; the ids and weights
// stay exactly those of the CUDA-core router (route.cuh), bit for bit.
//
// Pages: a small router selects a few experts per token, e.g. 6 of 256 (banandre.com, "The
// 284B Model on a 32GB GPU Trick", section "Sparsity Is a Lie (But a Useful One)").  At a
// prefill chunk of thousands of tokens the router is a dense [T x d] x [d x E] product.
//
// Kernels (one stream, in order; renormalised weights, 16 <= E <= 256, E % 16 == 0):
//   rtc_prep_kernel    per expert ||W_r[e]||_2 (an upper bound, rounded up); zeroes the counts
//   rtc_logits_kernel  tensor-core logits L~ = x W_r^T in fp32 (bf16 x bf16 products, fp32
//                      accumulation), M = 128 tokens per tile, N = E, K = 64 per stage; when
//                      the tiles fill less than half the SMs, two CTAs per tile each take half
//                      of K and the selection adds the two parts (one more fp32 rounding,
//                      inside the bound below)
//   rtc_select_kernel  one warp per token: the candidates, their order-R logits, the top-k
//   rtc_fallback_kernel  tokens with too many candidates: every logit in order R, then the
//                      exact selection
//
// The bound.  Order R and the tensor cores both approximate the exact dot product s_e =
// sum_i x_i w_ei (bf16 products are exact in fp32), each within a multiple of the fp32 unit
// roundoff times sum_i |x_i w_ei| <= ||x|| ||w_e||.  Order R adds each product through at most
// d/32 - 1 sequential adds and 5 butterfly adds, each rounding to nearest (2^-24).  For the
// tensor cores the reading is that each K = 16 step loses at most two ulps (2^-22) of the
// running magnitude, d/16 steps in all.  rtc_gamma doubles the sum of the two, and tau =
// gamma ||x|| max_e ||w_e|| bounds |L~_e - L_R_e| for every expert of the token.
#pragma once
#include "route.cuh"
#include "tc.cuh"

namespace ftmoe {

constexpr int kRtcStages = 4;
constexpr int kRtcEpiWarps = 4;
constexpr int kRtcThreads = (2 + kRtcEpiWarps) * 32;

// Twice the relative error bound of the two logits together (see the bound above).
__host__ __device__ inline float rtc_gamma(int d) {
  return 2.f * (float(d / 16) * 2.384185791015625e-07f + float(d / 32 + 5) * 5.9604644775390625e-08f);
}

// tcgen05 kind::f16: BF16 x BF16 -> F32, K-major A and B
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (uint32_t(N >> 3) << 17) | (uint32_t(M >> 4) << 24);
}
__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                         uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
      : "memory");
}

struct RtcArgs {
  const uint16_t* x;      // [T][d]
  const uint16_t* wr;     // [E][d]
  const float* bias;      // [E] or nullptr
  int T, E, d, k;
  float* logits;          // [T][E] workspace: the tensor-core logits (over K / ksplit, part 0)
  float* logits2;         // [T][E] workspace: part 1 of a split K (ksplit == 2)
  int ksplit;             // 1, or 2: two CTAs per 128-token tile, each over half of K
  float* wnorm;           // [E] workspace: ||W_r[e]||_2, rounded up
  int32_t* fb_list;       // [T] workspace: tokens left to the fallback
  unsigned* fb_count;     // workspace header word: their number (zeroed by rtc_prep_kernel)
  unsigned* extra_count;  // workspace header word: tokens with more than k candidates (zeroed there too)
  int32_t* ids;           // [T][k]
  float* w;               // [T][k]
};

// An upper bound on sqrt(ss) from an fp32 sum of squares ss of at most 4096 / 32 + 5 sequential
// roundings (relative error < 1e-5), and at least 2^-30 (squares that underflow lose less than
// d * 2^-149 in all).
__device__ __forceinline__ float rtc_norm_bound(float ss) {
  return fmaxf(sqrtf(ss * 1.0001f) * 1.0001f, 9.313225746154785e-10f);
}

// One warp per expert: ||W_r[e]||_2 bounded from above.
__global__ void __launch_bounds__(256) rtc_prep_kernel(RtcArgs a) {
  pdl_wait();
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    *a.fb_count = 0u;
    *a.extra_count = 0u;
  }
  const int lane = threadIdx.x & 31;
  for (int e = blockIdx.x * 8 + (threadIdx.x >> 5); e < a.E; e += gridDim.x * 8) {
    const uint4* row = reinterpret_cast<const uint4*>(a.wr + size_t(e) * a.d);
    float ss = 0.f;
    for (int i = lane; i < a.d / 8; i += 32) {
      const uint4 v = __ldg(row + i);
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const uint32_t q = (&v.x)[u];
        ss = fmaf(bf16_lo(q), bf16_lo(q), ss);
        ss = fmaf(bf16_hi(q), bf16_hi(q), ss);
      }
    }
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) ss += __shfl_xor_sync(0xFFFFFFFFu, ss, off);
    if (lane == 0) a.wnorm[e] = rtc_norm_bound(ss);
  }
}

// Shared memory of the logits kernel: kRtcStages x (A 16 KB + B N x 128 B), barriers.
__host__ __device__ inline int rtc_smem(int N) { return kRtcStages * (kTileM * 128 + N * 128) + 128 + 1024; }

__global__ void __launch_bounds__(kRtcThreads, 1)
rtc_logits_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW, RtcArgs a,
                  int N) {
  extern __shared__ uint8_t rtc_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(rtc_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sb = smem_u32(smem);
  const int A_BYTES = kTileM * 128, B_BYTES = N * 128;
  const int OFF_B = kRtcStages * A_BYTES, OFF_BAR = OFF_B + kRtcStages * B_BYTES;
  const uint32_t bar_full = sb + OFF_BAR, bar_empty = bar_full + 8 * kRtcStages;
  const uint32_t bar_tfull = bar_empty + 8 * kRtcStages, bar_tempty = bar_tfull + 8, bar_done = bar_tempty + 8;
  uint32_t* s_tslot = reinterpret_cast<uint32_t*>(smem + OFF_BAR + 8 * (2 * kRtcStages + 3));
  volatile int* s_abort = reinterpret_cast<volatile int*>(smem + OFF_BAR + 8 * (2 * kRtcStages + 3) + 4);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kRtcStages; ++s) {
      mbar_init(bar_full + 8 * s, 1);
      mbar_init(bar_empty + 8 * s, 1);
    }
    mbar_init(bar_tfull, 1);
    mbar_init(bar_tempty, kRtcEpiWarps);
    mbar_init(bar_done, 1);
    *s_abort = 0;
    mbar_fence_init();
    prefetch_tmap(&tmX);
    prefetch_tmap(&tmW);
  }
  const uint32_t ncols = N <= 32 ? 32u : N <= 64 ? 64u : N <= 128 ? 128u : 256u;   // fp32 columns, a power of 2
  if (warp == 1) tmem_alloc(smem_u32(s_tslot), ncols);
  pdl_wait();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *s_tslot;
  // work items: (tile, part of K); item i = tile * ksplit + part
  const int tiles = (a.T + kTileM - 1) / kTileM * a.ksplit;
  const int KS = a.d / 64 / a.ksplit;
  if (warp == 0) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      uint32_t stage = 0, ph = 0;
      int issued = 0;
      bool ok = true;
      for (int item = blockIdx.x; item < tiles && ok; item += gridDim.x) {
        const int tile = item / a.ksplit, k0 = (item % a.ksplit) * KS;
        for (int ks = 0; ks < KS; ++ks) {
          if (!mbar_wait(bar_empty + 8 * stage, ph ^ 1, s_abort)) {
            ok = false;
            break;
          }
          const uint32_t fb = bar_full + 8 * stage;
          mbar_arrive_expect_tx(fb, uint32_t(A_BYTES + B_BYTES));
          tma_load_2d(sb + stage * A_BYTES, &tmX, (k0 + ks) * 128, tile * kTileM, fb);
          tma_load_2d(sb + OFF_B + stage * B_BYTES, &tmW, (k0 + ks) * 128, 0, fb);
          ++issued;
          if (++stage == kRtcStages) {
            stage = 0;
            ph ^= 1;
          }
        }
      }
      if (!ok) {
        set_dev_err(DEV_ERR_TIMEOUT);
        *s_abort = 1;
        for (int i = 0; i < kRtcStages && i < issued; ++i) {   // the copies in flight land first
          if (stage == 0) {
            stage = kRtcStages;
            ph ^= 1;
          }
          --stage;
          mbar_wait(bar_full + 8 * stage, ph, nullptr);
        }
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      uint32_t stage = 0, ph = 0, tph = 0;
      bool ok = true;
      const uint32_t idesc = idesc_bf16(kTileM, N);
      for (int tile = blockIdx.x; tile < tiles && ok; tile += gridDim.x) {
        if (!mbar_wait(bar_tempty, tph ^ 1, s_abort)) {
          ok = false;
          break;
        }
        tc_fence_after();
        for (int ks = 0; ks < KS; ++ks) {
          if (!mbar_wait(bar_full + 8 * stage, ph, s_abort)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sA = sb + stage * A_BYTES, sB = sb + OFF_B + stage * B_BYTES;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)   // K = 16 bf16 (32 bytes) per instruction
            mma_bf16(tmem, desc_sw128(sA + 32 * kk), desc_sw128(sB + 32 * kk), idesc, (ks | kk) != 0);
          tc_commit(bar_empty + 8 * stage);
          if (++stage == kRtcStages) {
            stage = 0;
            ph ^= 1;
          }
        }
        if (!ok) break;
        tc_commit(bar_tfull);
        tph ^= 1;
      }
      if (!ok) {
        set_dev_err(DEV_ERR_TIMEOUT);
        *s_abort = 1;
      }
      tc_commit(bar_done);
      mbar_wait(bar_done, 0, nullptr);
    }
  } else {
    // ---------------- epilogue: TMEM -> logits ----------------
    const int q = warp & 3;              // TMEM lane quarter of this warp
    const int r = q * 32 + lane;
    uint32_t tph = 0;
    for (int item = blockIdx.x; item < tiles; item += gridDim.x) {
      if (!mbar_wait(bar_tfull, tph, s_abort)) {
        if (lane == 0) {
          set_dev_err(DEV_ERR_TIMEOUT);
          *s_abort = 1;
        }
        break;
      }
      tc_fence_after();
      const int t = (item / a.ksplit) * kTileM + r;
      float* out = (item % a.ksplit) ? a.logits2 : a.logits;
      const uint32_t tb = tmem + (uint32_t(q * 32) << 16);
      for (int c0 = 0; c0 < N; c0 += 16) {
        uint32_t v[16];
        tc_ld16(tb + c0, v);
        tc_wait_ld();
        tc_reg_fence(v);
        if (t < a.T) {
          float* dst = out + size_t(t) * a.E + c0;
#pragma unroll
          for (int i = 0; i < 16; ++i)
            if (c0 + i < a.E) dst[i] = __uint_as_float(v[i]);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_tempty);
      tph ^= 1;
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, ncols);
}

// The order-R logit of expert e for the token whose x chunks this lane holds (xv[s] = chunk
// s * 32 + lane), without the bias: the CUDA-core router's arithmetic.
__device__ __forceinline__ float rtc_order_r(const uint4 (&xv)[16], const uint16_t* wrow, int S, int lane) {
  float acc = 0.f;
#pragma unroll
  for (int s = 0; s < 16; ++s) {
    if (s < S) {
      const uint4 wv = __ldg(reinterpret_cast<const uint4*>(wrow) + s * 32 + lane);
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const uint32_t xx = (&xv[s].x)[u >> 1], ww = (&wv.x)[u >> 1];
        const float xf = (u & 1) ? bf16_hi(xx) : bf16_lo(xx), wf = (u & 1) ? bf16_hi(ww) : bf16_lo(ww);
        acc = __fadd_rn(acc, __fmul_rn(xf, wf));
      }
    }
  }
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) acc = __fadd_rn(acc, __shfl_xor_sync(0xFFFFFFFFu, acc, off));
  return acc;
}

// Lane r < k holds (value, id) of rank r: writes ids and the renormalised weights with the
// arithmetic of the CUDA-core router's select step.
__device__ __forceinline__ void rtc_write(const RtcArgs& a, int t, int lane, float my_v, int my_i) {
  const float m = __shfl_sync(0xFFFFFFFFu, my_v, 0);
  float part = (lane < a.k) ? expf(my_v - m) : 0.f;
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) part += __shfl_xor_sync(0xFFFFFFFFu, part, off);
  if (lane < a.k) {
    a.ids[size_t(t) * a.k + lane] = my_i;
    a.w[size_t(t) * a.k + lane] = expf(my_v - m) / part;
  }
}

// One warp per token; SMAX = d / 256 at most (8 or 16), EJ = E / 32 at most (4 or 8).
//   1. V~ = L~ + bias for the token's E experts, and the k-th largest of them, kth.
//   2. Candidates C = {e : V~_e >= kth - delta}, delta = 2 tau + the bias adds' roundings.
//      Every expert outside C has an order-R value below each of the k largest V~ experts'
//      (all in C), so the order-R top-k lies in C.
//   3. The order-R logits of C, four experts at a time (four independent order-R chains; each
//      keeps its own order), then the exact top-k of C by (value desc, id asc): the ids, order
//      and weights of the CUDA-core router.
// A token with more than 32 candidates, or a non-finite V~ or bound, goes to the fallback list.
template <int SMAX, int EJ>
__global__ void __launch_bounds__(256, SMAX == 8 ? 3 : 2) rtc_select_kernel(RtcArgs a) {
  pdl_wait();
  const int lane = threadIdx.x & 31, wib = threadIdx.x >> 5;
  const int S = a.d >> 8;
  constexpr int NONE = 0x7FFFFFFF;
  __shared__ float s_wmax;
  __shared__ int s_cand[8][36];
  // the warp's token x, chunk s of lane l at [s * 32 + l] (dynamic: 8 warps x SMAX x 512 bytes)
  extern __shared__ uint4 rtc_sx[];
  uint4* sx = rtc_sx + wib * SMAX * 32;
  if (threadIdx.x < 32) {
    float m = 0.f;
    for (int e = lane; e < a.E; e += 32) m = fmaxf(m, a.wnorm[e]);
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, off));
    if (lane == 0) s_wmax = m;
  }
  __syncthreads();
  const float wmax = s_wmax;
  const float gamma = rtc_gamma(a.d);
  unsigned n_extra = 0;
  for (int t = blockIdx.x * 8 + wib; t < a.T; t += gridDim.x * 8) {
    // x of the token (for its norm here, and from shared memory for the candidates' logits)
    uint4 xv[SMAX];
    const uint4* xr = reinterpret_cast<const uint4*>(a.x + size_t(t) * a.d);
#pragma unroll
    for (int s = 0; s < SMAX; ++s) xv[s] = s < S ? __ldg(xr + s * 32 + lane) : make_uint4(0, 0, 0, 0);
    __syncwarp();                       // the previous token's reads of sx are done
#pragma unroll
    for (int s = 0; s < SMAX; ++s)
      if (s < S) sx[s * 32 + lane] = xv[s];
    float v[EJ];
    const float* row = a.logits + size_t(t) * a.E;
    const float* row2 = a.logits2 + size_t(t) * a.E;
    bool fin = true;
#pragma unroll
    for (int j = 0; j < EJ; ++j) {
      const int e = j * 32 + lane;
      v[j] = -INFINITY;
      if (e < a.E) {
        const float l = a.ksplit == 2 ? __fadd_rn(__ldcg(row + e), __ldcg(row2 + e)) : __ldcg(row + e);
        v[j] = a.bias ? __fadd_rn(l, __ldg(a.bias + e)) : l;
        fin = fin && isfinite(v[j]);
      }
    }
    float ss = 0.f;
#pragma unroll
    for (int s = 0; s < SMAX; ++s) {
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const uint32_t q = (&xv[s].x)[u];
        ss = fmaf(bf16_lo(q), bf16_lo(q), ss);
        ss = fmaf(bf16_hi(q), bf16_hi(q), ss);
      }
    }
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) ss += __shfl_xor_sync(0xFFFFFFFFu, ss, off);
    // 1. the k-th largest V~ (k rounds of a warp argmax)
    uint32_t taken = 0;
    float kth = -INFINITY;
    for (int rr = 0; rr < a.k; ++rr) {
      float bv = -INFINITY;
      int bi = NONE;
#pragma unroll
      for (int j = 0; j < EJ; ++j) {
        const int e = j * 32 + lane;
        if (e < a.E && !((taken >> j) & 1u) && (bi == NONE || v[j] > bv)) {
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
      kth = bv;
    }
    // 2. the candidates, in ascending id, into s_cand[wib][0..n)
    const float tau = gamma * rtc_norm_bound(ss) * wmax;
    const float delta = 2.f * tau + 8.f * 1.1920929e-07f * (fabsf(kth) + 2.f * tau);
    const float thr = kth - delta;
    const bool ok = __all_sync(0xFFFFFFFFu, fin) && isfinite(thr);
    int n = 0;
#pragma unroll
    for (int j = 0; j < EJ; ++j) {
      const bool c = ok && (j * 32 + lane < a.E) && v[j] >= thr;
      const uint32_t m = __ballot_sync(0xFFFFFFFFu, c);
      const int pos = n + __popc(m & ((1u << lane) - 1u));
      if (c && pos < 32) s_cand[wib][pos] = j * 32 + lane;
      n += __popc(m);
    }
    if (!ok || n > 32) {
      if (lane == 0) a.fb_list[atomicAdd(a.fb_count, 1u)] = t;
      continue;
    }
    n_extra += (n > a.k);
    __syncwarp();
    // 3. the candidates' order-R values, four at a time (two packed pairs of chains); the
    //    router rows' next chunks load while the current ones are used
    const int my_i = lane < n ? s_cand[wib][lane] : NONE;
    float myR = -INFINITY;
    for (int p0 = 0; p0 < n; p0 += 4) {
      const uint4* wrow[4];
#pragma unroll
      for (int q = 0; q < 4; ++q)
        wrow[q] = reinterpret_cast<const uint4*>(a.wr + size_t(s_cand[wib][min(p0 + q, n - 1)]) * a.d) + lane;
      uint64_t acc[2] = {0ull, 0ull};
      uint4 wb[2][4];
#pragma unroll
      for (int q = 0; q < 4; ++q) wb[0][q] = __ldg(wrow[q]);
#pragma unroll
      for (int s = 0; s < SMAX; ++s) {
        if (s < S) {
          if (s + 1 < S) {
#pragma unroll
            for (int q = 0; q < 4; ++q) wb[(s + 1) & 1][q] = __ldg(wrow[q] + (s + 1) * 32);
          }
          const uint4(&wv)[4] = wb[s & 1];
          const uint4 xs = sx[s * 32 + lane];
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            const uint32_t xx = (&xs.x)[u >> 1];
            const float xf = (u & 1) ? bf16_hi(xx) : bf16_lo(xx);
            const uint64_t x2 = f32x2_pack(xf, xf);
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const uint32_t w0 = (&wv[2 * h].x)[u >> 1], w1 = (&wv[2 * h + 1].x)[u >> 1];
              const uint64_t w2 = f32x2_pack((u & 1) ? bf16_hi(w0) : bf16_lo(w0), (u & 1) ? bf16_hi(w1) : bf16_lo(w1));
              acc[h] = f32x2_add(acc[h], f32x2_mul(x2, w2));
            }
          }
        }
      }
      float l[4];
      f32x2_unpack(acc[0], l[0], l[1]);
      f32x2_unpack(acc[1], l[2], l[3]);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) l[q] = __fadd_rn(l[q], __shfl_xor_sync(0xFFFFFFFFu, l[q], off));
        if (p0 + q < n && lane == p0 + q) myR = l[q];
      }
    }
    __syncwarp();                       // s_cand is rewritten by the next token
    if (a.bias && lane < n) myR = __fadd_rn(myR, __ldg(a.bias + my_i));
    int rank = 0;
    for (int o = 0; o < n; ++o) {
      const float ov = __shfl_sync(0xFFFFFFFFu, myR, o);
      const int oi = __shfl_sync(0xFFFFFFFFu, my_i, o);
      rank += (ov > myR) || (ov == myR && oi < my_i);
    }
    // lane r < k <- (value, id) of rank r
    float out_v = 0.f;
    int out_i = 0;
    for (int o = 0; o < n; ++o) {
      const int ro = __shfl_sync(0xFFFFFFFFu, rank, o);
      const float ov = __shfl_sync(0xFFFFFFFFu, myR, o);
      const int oi = __shfl_sync(0xFFFFFFFFu, my_i, o);
      if (lane == ro) {
        out_v = ov;
        out_i = oi;
      }
    }
    rtc_write(a, t, lane, out_v, out_i);
  }
  if (lane == 0 && n_extra) atomicAdd(a.extra_count, n_extra);
}

// The listed tokens: all E logits in order R (one warp per expert group), then the exact
// selection from them.  A CTA takes tokens i, i + grid, ...
__global__ void __launch_bounds__(256) rtc_fallback_kernel(RtcArgs a) {
  pdl_wait();
  __shared__ float s_l[256];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int S = a.d >> 8;
  const unsigned n = *reinterpret_cast<volatile unsigned*>(a.fb_count);
  for (unsigned i = blockIdx.x; i < n; i += gridDim.x) {
    const int t = a.fb_list[i];
    uint4 xv[16];
    const uint4* xr = reinterpret_cast<const uint4*>(a.x + size_t(t) * a.d);
#pragma unroll
    for (int s = 0; s < 16; ++s) xv[s] = s < S ? __ldg(xr + s * 32 + lane) : make_uint4(0, 0, 0, 0);
    for (int e = warp; e < a.E; e += 8) {
      float l = rtc_order_r(xv, a.wr + size_t(e) * a.d, S, lane);
      if (a.bias) l = __fadd_rn(l, a.bias[e]);
      if (lane == 0) s_l[e] = l;
    }
    __syncthreads();
    if (warp == 0) {
      // exact top-k of the order-R logits (the CUDA-core select step)
      constexpr int NONE = 0x7FFFFFFF;
      float v[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) v[j] = (j * 32 + lane < a.E) ? s_l[j * 32 + lane] : -INFINITY;
      uint32_t taken = 0;
      float my_v = -INFINITY;
      int my_i = NONE;
      for (int rr = 0; rr < a.k; ++rr) {
        float bv = -INFINITY;
        int bi = NONE;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const int e = j * 32 + lane;
          const bool ok = (e < a.E) && !((taken >> j) & 1u);
          if (ok && (bi == NONE || v[j] > bv)) {
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
        if (lane == rr) {
          my_v = bv;
          my_i = bi;
        }
      }
      rtc_write(a, t, lane, my_v, my_i);
    }
    __syncthreads();
  }
}

}  // namespace ftmoe
