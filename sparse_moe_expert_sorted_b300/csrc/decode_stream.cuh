// a4 (+a5) decode path for NVFP4 / MXFP4, streaming form: the selected experts'
// weights flow through a shared-memory ring filled by bulk copies, and
// consumer warps run the warp-level MMAs of decode.cuh on them.
//
// Pages: resident experts are computed on GPU tensor cores from expert slots
// (zubnet.ai, "FreeToken, Unsloth GGUF ... consumer hardware"); in decode a
// token touches a handful of experts (banandre.com, "The 284B Model on a 32GB
// GPU Trick", section "Sparsity Is a Lie"), so a decode layer is a stream of
// those experts' weights and is bound by HBM bandwidth.
//
// Persistent kernel, one CTA per SM (all resident):
//   warp 0       producer: for each work item of this CTA, waits for a free
//                stage and fills it with ONE bulk copy: the item's tile in the
//                prepared decode layout (below) is contiguous.  Few large copies
//                keep the copy engine's per-copy cost small.
//   warps 1-16   consumers: MMAs on the staged rows against the tokens staged
//                in shared memory as f16; partials of the 8 warps meet in
//                shared memory; epilogue.
// Work items, in order: phase A (gate/up) then phase B (down).  An item is
// (expert, group of up to 8 tokens, block of rows); a stage is one item's rows.  Each CTA takes a contiguous
// range of items, so consecutive items share the staged tokens.
//   phase A item: 16 gate + 16 up rows; the consumer warps split K.
//   phase B item: 32 down rows; consumer warp w takes row tile w & 1 and K part w >> 1.
// Prepared decode layout (ftmoe_prepare_weights), per slot: phase-A tiles (16 gate
// rows + 16 up rows, ffn/16 of them) then phase-B tiles (32 down rows, d/32 of them).
// A tile of R rows of one matrix stores its codes chunk-major, [K/32 chunks][R rows][16
// bytes], then the scales block-major, [K/16 (NVFP4) or K/32 (MXFP4) blocks][R rows].  A
// phase-A tile is [gate codes][up codes][gate scales][up scales].  In this order the
// 8 rows of an MMA fragment load sit side by side, so every shared-memory fragment read
// covers contiguous 128-byte lines (no bank conflicts).
// Between the phases the consumers meet at a grid barrier (every h written);
// the producer does not wait there, so the first down weights are already in
// flight.  The layer call also zeroes out first and casts it to bf16 last.
#pragma once
#include "decode.cuh"
#include "tc.cuh"

namespace ftmoe {

constexpr int kSdCons = 16;                    // consumer warps
constexpr int kSdThreads = (1 + kSdCons) * 32;
constexpr int kSdRowsA = 16;                   // gate (and up) rows per phase-A item
constexpr int kSdRowsB = 32;                   // down rows per phase-B item
// per-expert info: item starts (A, B), first row, rows, slot, tensor scales (3); then the token group
__host__ __device__ inline int sd_info_ints(int E) { return 8 * (E + 8) + 32; }

// Bytes of one prepared tile: phase A (16 gate + 16 up rows, K = d), phase B (32 down rows, K = f).
__host__ __device__ inline int sd_block_bytes_a(int d, int fmt) {
  return 2 * kSdRowsA * (d / 2 + d / (fmt == FTMOE_NVFP4 ? 16 : 32));
}
__host__ __device__ inline int sd_block_bytes_b(int f, int fmt) {
  return kSdRowsB * (f / 2 + f / (fmt == FTMOE_NVFP4 ? 16 : 32));
}
// Prepared decode bytes of one slot.
__host__ __device__ inline size_t sd_slot_bytes(int d, int f, int fmt) {
  return size_t(f / kSdRowsA) * sd_block_bytes_a(d, fmt) + size_t(d / kSdRowsB) * sd_block_bytes_b(f, fmt);
}

// Repack canonical codes + scales into the prepared decode layout (one thread per output byte).
__global__ void prep_decode_kernel(const uint8_t* gate, const uint8_t* up, const uint8_t* down, const uint8_t* gs,
                                   const uint8_t* us, const uint8_t* ds, int C, int d, int f, int fmt, uint8_t* out) {
  const int sdiv = fmt == FTMOE_NVFP4 ? 16 : 32;
  const long long ba = sd_block_bytes_a(d, fmt), bb = sd_block_bytes_b(f, fmt);
  const long long na = f / kSdRowsA, nb = d / kSdRowsB;
  const long long per_slot = na * ba + nb * bb;
  const long long total = per_slot * C;
  for (long long o = (long long)blockIdx.x * blockDim.x + threadIdx.x; o < total; o += (long long)gridDim.x * blockDim.x) {
    const long long slot = o / per_slot;
    long long r = o % per_slot;
    uint8_t v;
    if (r < na * ba) {
      const long long tile = r / ba;
      long long q = r % ba;
      const long long cbytes = kSdRowsA * (d / 2);          // one matrix's codes in the tile
      if (q < 2 * cbytes) {
        const int m = int(q / cbytes);
        q %= cbytes;
        const long long chunk = q / (kSdRowsA * 16), row = (q / 16) % kSdRowsA, byte = q % 16;
        const uint8_t* src = m ? up : gate;
        v = src[(slot * f + tile * kSdRowsA + row) * (d / 2) + chunk * 16 + byte];
      } else {
        q -= 2 * cbytes;
        const long long sbytes = kSdRowsA * (d / sdiv);
        const int m = int(q / sbytes);
        q %= sbytes;
        const long long blk = q / kSdRowsA, row = q % kSdRowsA;
        const uint8_t* src = m ? us : gs;
        v = src[(slot * f + tile * kSdRowsA + row) * (d / sdiv) + blk];
      }
    } else {
      r -= na * ba;
      const long long tile = r / bb;
      long long q = r % bb;
      const long long cbytes = kSdRowsB * (f / 2);
      if (q < cbytes) {
        const long long chunk = q / (kSdRowsB * 16), row = (q / 16) % kSdRowsB, byte = q % 16;
        v = down[(slot * d + tile * kSdRowsB + row) * (f / 2) + chunk * 16 + byte];
      } else {
        q -= cbytes;
        const long long blk = q / kSdRowsB, row = q % kSdRowsB;
        v = ds[(slot * d + tile * kSdRowsB + row) * (f / sdiv) + blk];
      }
    }
    out[o] = v;
  }
}

// Layout of one stage and of the kernel's shared memory, for one (d, f, format).  A stage
// holds whole rows (K = d in phase A, f in phase B), so each matrix tile is one contiguous
// run of the canonical layout and lands with one bulk copy: codes [rows][K/2], then
// scales [rows][K/16 or K/32].
struct SdLayout {
  int kcA, nkA, kcB, nkB;     // K per stage and stages per item, phase A (K = d) and B (K = f)
  int csA, ssA, csB, ssB;     // code / scale row strides in the stage (bytes)
  int stage_bytes, stages;
  int xrows, estride;         // staged token rows; per-expert info stride (ints)
  int off_x, off_red, off_rank, off_bar, smem;
};

// xrows: tokens staged at once (min(8, T))
__host__ __device__ inline SdLayout sd_layout(int E, int d, int f, int fmt, int xrows, int max_smem) {
  SdLayout L;
  L.xrows = xrows;
  L.estride = E + 8;
  const int sdiv = fmt == FTMOE_NVFP4 ? 16 : 32;
  L.kcA = d;
  L.nkA = 1;
  L.kcB = f;
  L.nkB = 1;
  L.csA = d / 2;
  L.ssA = d / sdiv;
  L.csB = f / 2;
  L.ssB = f / sdiv;
  const int sa = sd_block_bytes_a(d, fmt), sb = sd_block_bytes_b(f, fmt);
  L.stage_bytes = ((sa > sb ? sa : sb) + 127) / 128 * 128;
  const int kx = d > f ? d : f;
  const int xbytes = (xrows * (kx + 8) * 2 + 127) / 128 * 128;
  const int red = kSdCons * 2 * 16 * 8 * 4;
  const int fixed = xbytes + red + sd_info_ints(E) * 4 + 256;
  L.stages = (max_smem - 1024 - fixed) / L.stage_bytes;
  if (L.stages > 4) L.stages = 4;
  L.off_x = L.stages * L.stage_bytes;
  L.off_red = L.off_x + xbytes;
  L.off_rank = L.off_red + red;
  L.off_bar = L.off_rank + (sd_info_ints(E) * 4 + 15) / 16 * 16;
  L.smem = L.off_bar + 256 + 128;
  return L;
}

// Whether the streaming kernel takes this shape: E <= 512 and at least 2 stages of
// shared memory.  (Every tile copy is a multiple of 16 bytes at a 16-byte boundary:
// d and f are multiples of 128.)
__host__ inline bool sd_supported(int E, int d, int f, int fmt, int xrows, int max_smem) {
  if (fmt != FTMOE_NVFP4 && fmt != FTMOE_MXFP4) return false;
  if (E > 1024) return false;
  return sd_layout(E, d, f, fmt, xrows, max_smem).stages >= 2;
}

// items per resident expert: rows-blocks x token groups
__device__ __forceinline__ int sd_groups(int cnt, int xrows) { return (cnt + xrows - 1) / xrows; }

// s_a[e], s_b[e]: first phase-A / phase-B item of expert e; totals in s_a[E], s_b[E].
// s_lo, s_cnt, s_slot: the expert's first sorted row, rows and slot.  All threads of the CTA.
__device__ __forceinline__ void sd_items(const FfnArgs& a, int xrows, int* s_a, int* s_b, int* s_lo, int* s_cnt,
                                         int* s_slot, float* s_ts) {
  const int ua = a.f / kSdRowsA, ub = a.d / kSdRowsB;
  for (int e = threadIdx.x; e < a.E; e += blockDim.x) {
    const int lo = a.offsets[e];
    const int cnt = a.offsets[e + 1] - lo;
    int slot = a.slot_of ? a.slot_of[e] : e;
    if (slot >= a.C) {
      if (cnt > 0 && blockIdx.x == 0) set_dev_err(DEV_ERR_BAD_SLOT);
      slot = -1;
    }
    s_lo[e] = lo;
    s_cnt[e] = cnt;
    s_slot[e] = slot;
#pragma unroll
    for (int m = 0; m < 3; ++m) s_ts[3 * e + m] = (a.tscale && slot >= 0) ? a.tscale[slot * 3 + m] : 1.f;
    const int gr = (cnt > 0 && slot >= 0) ? sd_groups(cnt, xrows) : 0;
    s_a[e] = gr * ua;
    s_b[e] = gr * ub;
  }
  __syncthreads();
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    int ra = 0, rb = 0;
    for (int base = 0; base < a.E; base += 32) {
      const int e = base + lane;
      const int na = e < a.E ? s_a[e] : 0, nb = e < a.E ? s_b[e] : 0;
      int ia = na, ib = nb;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int oa = __shfl_up_sync(0xFFFFFFFFu, ia, off), ob = __shfl_up_sync(0xFFFFFFFFu, ib, off);
        if (lane >= off) {
          ia += oa;
          ib += ob;
        }
      }
      if (e < a.E) {
        s_a[e] = ra + ia - na;
        s_b[e] = rb + ib - nb;
      }
      ra += __shfl_sync(0xFFFFFFFFu, ia, 31);
      rb += __shfl_sync(0xFFFFFFFFu, ib, 31);
    }
    if (lane == 0) {
      s_a[a.E] = ra;
      s_b[a.E] = rb;
    }
  }
  __syncthreads();
}

struct SdItem {
  int e, slot, lo, cnt, grp, n0;   // expert, slot, first sorted row, tokens, token group, row block
};
// Items of one CTA are visited in increasing order; *e tracks the expert (start it at -1).
__device__ __forceinline__ SdItem sd_item(const int* s_start, const int* s_lo, const int* s_cnt, const int* s_slot,
                                          int E, int item, int blocks, int* e) {
  if (*e < 0) *e = find_expert(s_start, E, item);
  while (item >= s_start[*e + 1]) ++*e;
  SdItem it;
  it.e = *e;
  const int local = item - s_start[it.e];
  it.grp = local / blocks;
  it.n0 = local % blocks;
  it.slot = s_slot[it.e];
  it.lo = s_lo[it.e];
  it.cnt = s_cnt[it.e];
  return it;
}

// Consumer-only barrier (named barrier 1, the 8 consumer warps).
__device__ __forceinline__ void sd_cons_sync() { asm volatile("bar.sync 1, %0;" ::"r"(kSdCons * 32) : "memory"); }

// MMAs of NT 16-row tiles (NT = 2: gate and up, sharing the token fragments) over
// super-blocks [sb_lo, sb_hi) of a staged tile.  Tile m: codes at cbase[m], scales at
// sbase[m], in a prepared block of R rows; this lane's fragment rows are r and r + 8.
template <int FMT, int NT>
__device__ __forceinline__ void sd_tiles_mma(const uint8_t* const (&cbase)[NT], const uint8_t* const (&sbase)[NT],
                                             int R, int r, const uint16_t* xrow, int sb_lo, int sb_hi, int t,
                                             float (&acc)[NT][4]) {
  const int half = (t & 1) * 8;
  for (int sb0 = sb_lo; sb0 < sb_hi; sb0 += 8) {
    const int nc = min(8, sb_hi - sb0);
    // MXFP4: rebase the chunk's scales on their maximum exponent
    int e0[NT][2];
#pragma unroll
    for (int m = 0; m < NT; ++m) {
      e0[m][0] = e0[m][1] = 0;
      if (FMT == FTMOE_MXFP4) {
        for (int b = 2 * sb0; b < 2 * (sb0 + nc); ++b) {
          e0[m][0] = max(e0[m][0], int(sbase[m][b * R + r]));
          e0[m][1] = max(e0[m][1], int(sbase[m][b * R + r + 8]));
        }
      }
    }
    float part[NT][4];
#pragma unroll
    for (int m = 0; m < NT; ++m)
#pragma unroll
      for (int i = 0; i < 4; ++i) part[m][i] = 0.f;
#pragma unroll 1
    for (int c = 0; c < nc; ++c) {
      const int sb = sb0 + c;
      const uint16_t* xp = xrow + 64 * sb;
      const uint4 x0 = *reinterpret_cast<const uint4*>(xp);
      const uint4 x1 = *reinterpret_cast<const uint4*>(xp + 8);
      const uint32_t B[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
      const int chunk = 2 * sb + (t >> 1);
#pragma unroll
      for (int m = 0; m < NT; ++m) {
        const uint2 ca = *reinterpret_cast<const uint2*>(cbase[m] + (chunk * R + r) * 16 + half);
        const uint2 cb = *reinterpret_cast<const uint2*>(cbase[m] + (chunk * R + r + 8) * 16 + half);
        uint32_t pre0, pre1;
        if (FMT == FTMOE_NVFP4) {
          pre0 = e4m3_f16x2(sbase[m][(4 * sb + t) * R + r]);
          pre1 = e4m3_f16x2(sbase[m][(4 * sb + t) * R + r + 8]);
        } else {
          pre0 = pow2_f16x2(int(sbase[m][(2 * sb + (t >> 1)) * R + r]) - e0[m][0]);
          pre1 = pow2_f16x2(int(sbase[m][(2 * sb + (t >> 1)) * R + r + 8]) - e0[m][1]);
        }
        // byte i of the lane's 8 code bytes -> fa[i] (row r), fb[i] (row r + 8)
        uint32_t fa[8], fb[8];
        e2m1x8_to_f16x8(ca.x, *reinterpret_cast<uint32_t(*)[4]>(fa));
        e2m1x8_to_f16x8(ca.y, *reinterpret_cast<uint32_t(*)[4]>(fa + 4));
        e2m1x8_to_f16x8(cb.x, *reinterpret_cast<uint32_t(*)[4]>(fb));
        e2m1x8_to_f16x8(cb.y, *reinterpret_cast<uint32_t(*)[4]>(fb + 4));
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          fa[i] = hmul2(fa[i], pre0);
          fb[i] = hmul2(fb[i], pre1);
        }
        // MMA step j: bytes 2j (columns 2t, 2t+1) and 2j + 1 (columns 2t+8, 2t+9)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          if (FMT == FTMOE_MXFP4)
            mma_16816(part[m], fa[2 * j], fb[2 * j], fa[2 * j + 1], fb[2 * j + 1], B[2 * j], B[2 * j + 1]);
          else
            mma_16816(acc[m], fa[2 * j], fb[2 * j], fa[2 * j + 1], fb[2 * j + 1], B[2 * j], B[2 * j + 1]);
        }
      }
    }
    if (FMT == FTMOE_MXFP4) {
#pragma unroll
      for (int m = 0; m < NT; ++m) {
        const float f0 = e8m0_to_float(uint32_t(e0[m][0])), f1 = e8m0_to_float(uint32_t(e0[m][1]));
        acc[m][0] = fmaf(f0, part[m][0], acc[m][0]);
        acc[m][1] = fmaf(f0, part[m][1], acc[m][1]);
        acc[m][2] = fmaf(f1, part[m][2], acc[m][2]);
        acc[m][3] = fmaf(f1, part[m][3], acc[m][3]);
      }
    }
  }
}

template <int FMT>
__global__ void __launch_bounds__(kSdThreads, 1)
sd_ffn_kernel(FfnArgs a, SdLayout Ls, unsigned* bar_count, unsigned* bar_gen) {
  extern __shared__ uint8_t sd_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(sd_raw) + 127) & ~uintptr_t(127));
  uint16_t* s_x = reinterpret_cast<uint16_t*>(sm + Ls.off_x);
  float* s_red = reinterpret_cast<float*>(sm + Ls.off_red);   // [warp][m][16][8]
  const int es = Ls.estride;
  int* s_a = reinterpret_cast<int*>(sm + Ls.off_rank);
  int* s_b = s_a + es;
  int* s_lo = s_a + 2 * es;
  int* s_cnt = s_a + 3 * es;
  int* s_slot = s_a + 4 * es;
  float* s_ts = reinterpret_cast<float*>(s_a + 5 * es);   // [E][3]
  int* s_tok = s_a + 8 * es;                               // token group: x row of each token
  float* s_w = reinterpret_cast<float*>(s_a + 8 * es + 8); // and its combine weight
  const uint32_t bars = smem_u32(sm + Ls.off_bar);              // full[4], empty[4]
  int* s_flag = reinterpret_cast<int*>(sm + Ls.off_bar + 128);
  volatile int* s_abort = reinterpret_cast<volatile int*>(sm + Ls.off_bar + 132);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int S = Ls.stages;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(bars + 8 * s, 1);
      mbar_init(bars + 64 + 8 * s, kSdCons);
    }
    *s_abort = 0;
    mbar_fence_init();
  }
  pdl_wait();
  sd_items(a, Ls.xrows, s_a, s_b, s_lo, s_cnt, s_slot, s_ts);   // all threads, ends with __syncthreads
  const int NA = s_a[a.E], NB = s_b[a.E];
  const int G = gridDim.x, b = blockIdx.x;
  const int a_lo = int((long long)NA * b / G), a_hi = int((long long)NA * (b + 1) / G);
  const int b_lo = int((long long)NB * b / G), b_hi = int((long long)NB * (b + 1) / G);
  const int ua = a.f / kSdRowsA, ub = a.d / kSdRowsB;
  const size_t blk_a = sd_block_bytes_a(a.d, FMT), blk_b = sd_block_bytes_b(a.f, FMT);
  const size_t slot_bytes = sd_slot_bytes(a.d, a.f, FMT);

  if (warp == 0) {
    // ---------------- producer ----------------
    uint32_t stage = 0, ph = 0;
    bool ok = true;
    for (int phase = 0; phase < 2 && ok; ++phase) {
      const int i0 = phase ? b_lo : a_lo, i1 = phase ? b_hi : a_hi;
      const int kc = phase ? Ls.kcB : Ls.kcA, nk = phase ? Ls.nkB : Ls.nkA;
      const int cs = phase ? Ls.csB : Ls.csA, ss = phase ? Ls.ssB : Ls.ssA;
      const int K = phase ? a.f : a.d, N = phase ? a.d : a.f;
      const int nrows = phase ? kSdRowsB : 2 * kSdRowsA;
      const uint32_t bytes = uint32_t(phase ? blk_b : blk_a);
      int ecur = -1;
      for (int item = i0; item < i1 && ok; ++item) {
        const SdItem it = sd_item(phase ? s_b : s_a, s_lo, s_cnt, s_slot, a.E, item, phase ? ub : ua, &ecur);
        for (int kk = 0; kk < nk; ++kk) {
          if (!mbar_wait(bars + 64 + 8 * stage, ph ^ 1, s_abort)) {
            ok = false;
            break;
          }
          if (lane == 0) {
            mbar_arrive_expect_tx(bars + 8 * stage, bytes);
            const uint8_t* src = a.prep_dec + size_t(it.slot) * slot_bytes +
                                 (phase ? size_t(a.f / kSdRowsA) * blk_a + size_t(it.n0) * blk_b
                                        : size_t(it.n0) * blk_a);
            bulk_load(smem_u32(sm + stage * Ls.stage_bytes), src, bytes, bars + 8 * stage);
          }
          __syncwarp();
          if (++stage == uint32_t(S)) {
            stage = 0;
            ph ^= 1;
          }
        }
      }
    }
    if (!ok) {
      if (lane == 0) {
        set_dev_err(DEV_ERR_TIMEOUT);
        *s_abort = 1;
      }
    }
    // let every copy issued land before the CTA can exit: wait for the last uses of each stage
    if (lane == 0) {
      for (int i = 0; i < S; ++i) {
        if (stage == 0) {
          stage = S;
          ph ^= 1;
        }
        --stage;
        mbar_wait(bars + 8 * stage, ph, nullptr);
      }
    }
    return;
  }

  // ---------------- consumers ----------------
  const int cw = warp - 1;                 // consumer warp 0..7
  const int ct = threadIdx.x - 32;         // consumer thread 0..255
  const int g = lane >> 2, t = lane & 3;
  uint32_t stage = 0, ph = 0;
  bool ok = true;

  if (a.out_bf16) {
    float4* o = reinterpret_cast<float4*>(a.y_or_out);
    const long long n4 = (long long)a.T * a.d / 4;
    for (long long i = (long long)b * (kSdCons * 32) + ct; i < n4; i += (long long)G * kSdCons * 32)
      o[i] = make_float4(0.f, 0.f, 0.f, 0.f);
  }

  for (int phase = 0; phase < 2; ++phase) {
    const int i0 = phase ? b_lo : a_lo, i1 = phase ? b_hi : a_hi;
    const int kc = phase ? Ls.kcB : Ls.kcA, nk = phase ? Ls.nkB : Ls.nkA;
    const int cs = phase ? Ls.csB : Ls.csA, ss = phase ? Ls.ssB : Ls.ssA;
    const int K = phase ? a.f : a.d;
    const int nrows = phase ? kSdRowsB : 2 * kSdRowsA;
    const int st_x = K + 8;                // staged token row stride (f16)
    if (phase == 1) {
      // every h of every CTA is written before any is read
      sd_cons_sync();
      if (ct == 0) {
        int okb = 1;
        const unsigned gg = *reinterpret_cast<volatile unsigned*>(bar_gen);
        __threadfence();
        if (atomicAdd(bar_count, 1u) == unsigned(G) - 1) {
          *reinterpret_cast<volatile unsigned*>(bar_count) = 0u;
          __threadfence();
          atomicAdd(bar_gen, 1u);
        } else {
          const unsigned long long t0 = globaltimer_ns();
          for (uint32_t it = 0; *reinterpret_cast<volatile unsigned*>(bar_gen) == gg; ++it) {
            if ((it & 63u) == 63u && globaltimer_ns() - t0 > kWaitLimitNs) {
              okb = 0;
              set_dev_err(DEV_ERR_GRID_TIMEOUT);
              break;
            }
            __nanosleep(64);
          }
        }
        __threadfence();
        *s_flag = okb;
      }
      sd_cons_sync();
      if (!*s_flag) {
        ok = false;
        *s_abort = 1;
      }
    }
    // On a failed wait `ok` turns false and the loops keep their shape (every consumer
    // warp still reaches every barrier), skipping work, so no warp is left waiting.
    int staged_e = -1, staged_g = -1, ecur = -1;
    for (int item = i0; item < i1; ++item) {
      const SdItem it = sd_item(phase ? s_b : s_a, s_lo, s_cnt, s_slot, a.E, item, phase ? ub : ua, &ecur);
      const int p0 = it.grp * Ls.xrows, n = min(Ls.xrows, it.cnt - p0);
      if (it.e != staged_e || it.grp != staged_g) {
        sd_cons_sync();   // every warp is done with the previous tokens
        if (ct < n) {
          const int p = a.sorted_pair[it.lo + p0 + ct];
          s_tok[ct] = p / a.k;
          s_w[ct] = a.topk_w ? a.topk_w[p] : 0.f;
        }
        if (phase == 0) {
          const int per = K / 8;
          for (int c = ct; c < n * per; c += kSdCons * 32) {
            const int q = c / per, cc = c % per;
            const uint16_t* row = a.x + size_t(a.sorted_pair[it.lo + p0 + q] / a.k) * a.d;
            const uint4 v = __ldg(reinterpret_cast<const uint4*>(row) + cc);
            uint4 hh;
            hh.x = f16x2_of(bf16_lo(v.x), bf16_hi(v.x));
            hh.y = f16x2_of(bf16_lo(v.y), bf16_hi(v.y));
            hh.z = f16x2_of(bf16_lo(v.z), bf16_hi(v.z));
            hh.w = f16x2_of(bf16_lo(v.w), bf16_hi(v.w));
            *reinterpret_cast<uint4*>(s_x + q * st_x + 8 * cc) = hh;
          }
        } else {
          const int per = K / 8;
          for (int c = ct; c < n * per; c += kSdCons * 32) {
            const int q = c / per, cc = c % per;
            const float4* row = reinterpret_cast<const float4*>(a.h + size_t(it.lo + p0 + q) * a.f) + 2 * cc;
            const float4 v0 = __ldcg(row), v1 = __ldcg(row + 1);
            uint4 hh;
            hh.x = f16x2_of(v0.x, v0.y);
            hh.y = f16x2_of(v0.z, v0.w);
            hh.z = f16x2_of(v1.x, v1.y);
            hh.w = f16x2_of(v1.z, v1.w);
            *reinterpret_cast<uint4*>(s_x + q * st_x + 8 * cc) = hh;
          }
        }
        staged_e = it.e;
        staged_g = it.grp;
        sd_cons_sync();
      }
      // warp's share: phase A: both matrices, K eighth cw; phase B: row tile cw & 1, K quarter cw >> 1
      float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
      const int nsb = kc / 64;
      const int parts = phase ? kSdCons / 2 : kSdCons;
      const int kp = phase ? (cw >> 1) : cw;
      const int sb_lo = kp * nsb / parts, sb_hi = (kp + 1) * nsb / parts;
      for (int kk = 0; kk < nk; ++kk) {
        if (ok && !mbar_wait(bars + 8 * stage, ph, s_abort)) {
          ok = false;
          *s_abort = 1;
        }
        const uint8_t* base = sm + stage * Ls.stage_bytes;
        // MMA token column g: rows past the staged ones read the last staged row (results unused)
        const uint16_t* xrow = s_x + min(g, Ls.xrows - 1) * st_x + kk * kc + 16 * t;
        if (!ok) {
          // skip the work; the stage is still released below
        } else if (phase == 0) {
          // [gate codes][up codes][gate scales][up scales], 16 rows each
          const int cb = kSdRowsA * (a.d / 2), sbb = kSdRowsA * ss;
          const uint8_t* const cbase[2] = {base, base + cb};
          const uint8_t* const sbase[2] = {base + 2 * cb, base + 2 * cb + sbb};
          sd_tiles_mma<FMT, 2>(cbase, sbase, kSdRowsA, g, xrow, sb_lo, sb_hi, t, acc);
        } else {
          // [down codes][down scales], 32 rows; this warp's 16-row half
          const int tile = cw & 1;
          const uint8_t* const cbase[1] = {base};
          const uint8_t* const sbase[1] = {base + kSdRowsB * (a.f / 2)};
          float (&acc1)[1][4] = *reinterpret_cast<float(*)[1][4]>(&acc[0]);
          sd_tiles_mma<FMT, 1>(cbase, sbase, kSdRowsB, tile * 16 + g, xrow, sb_lo, sb_hi, t, acc1);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(bars + 64 + 8 * stage);
        if (++stage == uint32_t(S)) {
          stage = 0;
          ph ^= 1;
        }
      }
      // partials -> shared memory: [warp][m][row 16][token 8]
      float* my = s_red + cw * 2 * 128;
#pragma unroll
      for (int m = 0; m < 2; ++m) {
        my[m * 128 + g * 8 + 2 * t] = acc[m][0];
        my[m * 128 + g * 8 + 2 * t + 1] = acc[m][1];
        my[m * 128 + (g + 8) * 8 + 2 * t] = acc[m][2];
        my[m * 128 + (g + 8) * 8 + 2 * t + 1] = acc[m][3];
      }
      sd_cons_sync();
      if (!ok) {
        // nothing to write
      } else if (phase == 0) {
        if (ct < 128) {
          const int row = ct & 15, tok = ct >> 4;
          if (tok < n) {
            float gs = 0.f, us = 0.f;
#pragma unroll
            for (int w = 0; w < kSdCons; ++w) {
              gs += s_red[w * 256 + row * 8 + tok];
              us += s_red[w * 256 + 128 + row * 8 + tok];
            }
            const float tsg = s_ts[3 * it.e + 0], tsu = s_ts[3 * it.e + 1];
            const float gg = gs * tsg, uu = us * tsu;
            const float h = gg / (1.f + expf(-gg)) * uu;
            if (!isfinite(h)) set_dev_err(DEV_ERR_NONFINITE);
            a.h[size_t(it.lo + p0 + tok) * a.f + it.n0 * kSdRowsA + row] = h;
          }
        }
      } else {
        const int tile = (ct >> 7) & 1, row = ct & 15, tok = (ct >> 4) & 7;
        if (ct < 256 && tok < n) {
          float y = 0.f;
#pragma unroll
          for (int q = 0; q < kSdCons / 2; ++q) y += s_red[(2 * q + tile) * 256 + row * 8 + tok];
          y *= s_ts[3 * it.e + 2];
          if (!isfinite(y)) set_dev_err(DEV_ERR_NONFINITE);
          const int i = p0 + tok;
          const int col = it.n0 * kSdRowsB + tile * 16 + row;
          if (a.topk_w) {
            atomicAdd(a.y_or_out + size_t(s_tok[tok]) * a.d + col, s_w[tok] * y);
          } else {
            a.y_or_out[size_t(it.lo + i) * a.d + col] = y;
          }
        }
      }
      sd_cons_sync();   // s_red is free again
    }
  }
  if (!ok) set_dev_err(DEV_ERR_TIMEOUT);
  if (a.out_bf16) {
    // every add of every CTA has landed: cast out to bf16
    sd_cons_sync();
    if (ct == 0) {
      int okb = 1;
      const unsigned gg = *reinterpret_cast<volatile unsigned*>(bar_gen);
      __threadfence();
      if (atomicAdd(bar_count, 1u) == unsigned(G) - 1) {
        *reinterpret_cast<volatile unsigned*>(bar_count) = 0u;
        __threadfence();
        atomicAdd(bar_gen, 1u);
      } else {
        const unsigned long long t0 = globaltimer_ns();
        for (uint32_t it = 0; *reinterpret_cast<volatile unsigned*>(bar_gen) == gg; ++it) {
          if ((it & 63u) == 63u && globaltimer_ns() - t0 > kWaitLimitNs) {
            okb = 0;
            set_dev_err(DEV_ERR_GRID_TIMEOUT);
            break;
          }
          __nanosleep(64);
        }
      }
      __threadfence();
      *s_flag = okb;
    }
    sd_cons_sync();
    if (!*s_flag || !ok) return;
    const float4* o = reinterpret_cast<const float4*>(a.y_or_out);
    uint2* ob = reinterpret_cast<uint2*>(a.out_bf16);
    const long long n4 = (long long)a.T * a.d / 4;
    for (long long i = (long long)b * (kSdCons * 32) + ct; i < n4; i += (long long)G * kSdCons * 32) {
      const float4 v = __ldcg(o + i);
      __nv_bfloat162 lo = __floats2bfloat162_rn(v.x, v.y), hi = __floats2bfloat162_rn(v.z, v.w);
      ob[i] = make_uint2(*reinterpret_cast<uint32_t*>(&lo), *reinterpret_cast<uint32_t*>(&hi));
    }
  }
}

}  // namespace ftmoe
