// a4 (+a5, and a1 + a2 in the layer call) decode path for NVFP4 / MXFP4, streaming
// form: the selected experts' weights flow through a shared-memory ring filled by bulk
// copies, and consumer warps run the warp-level MMAs of decode.cuh on them.
//
// Pages: resident experts are computed on GPU tensor cores from expert slots
// (zubnet.ai, "FreeToken, Unsloth GGUF ... consumer hardware"); in decode a
// token touches a few experts (banandre.com, "The 284B Model on a 32GB
// GPU Trick", section "Sparsity Is a Lie"), so a decode layer is a stream of
// those experts' weights and is bound by HBM bandwidth.
//
// Persistent kernel, one CTA per SM (all resident):
//   warp 0       producer: for each work item of this CTA, waits for a free
//                stage and fills it with ONE bulk copy: the item's tile in the
//                prepared decode layout (below) is contiguous.  Few large copies
//                keep the copy engine's per-copy cost small.
//   warps 1-16   consumers: MMAs on the staged rows against the tokens staged
//                in shared memory as f16.
//   warp 17      epilogue: reduces the consumers' partial sums and writes h or y.
// Work items, in order: phase A (gate/up) then phase B (down).  An item is
// (expert, group of up to 8 tokens, block of rows); a stage is one item's rows.  Each CTA
// takes a contiguous range of items, so consecutive items share the staged tokens (the
// one-token layer call takes its gate/up items strided instead; see ROUTE below).
//   phase A item: 16 gate + 16 up rows; the consumer warps split K.
//   phase B item: 32 down rows; consumer warp w takes row tile w & 1 and K part w >> 1.
// Prepared decode layout (ftmoe_prepare_weights), per slot: phase-A tiles (16 gate
// rows + 16 up rows, ffn/16 of them) then phase-B tiles (32 down rows, d/32 of them).
// A tile of R rows of one matrix stores its codes chunk-major, [K/32 chunks][R rows][16
// bytes], then the scales block-major, [K/16 (NVFP4) or K/32 (MXFP4) blocks][R rows].  A
// phase-A tile is [gate codes][up codes][gate scales][up scales].  In this order the
// 8 rows of an MMA fragment load sit side by side, so every shared-memory fragment read
// covers contiguous 128-byte lines (no bank conflicts).
//
// Cross-warp reduction without a CTA barrier: each consumer warp writes its partial
// sums of an item into one of two reduction buffers (item parity) and counts itself in,
// then goes on to the next item.  The epilogue warp waits for the 16 counts, sums the
// partials in warp order (results do not depend on timing), writes h or y and frees the
// buffer.  h is kept as f16 (the precision the down MMA reads it in).
//
// Between the phases: ftmoe_expert_ffn meets at a grid sync (every h written).  The layer
// call (ROUTE) instead counts the finished gate/up items of each expert, and a down item
// waits only for its own expert.  The producer never waits there, so the first down
// weights are already in flight.
//
// ROUTE (ftmoe_layer_forward with few tokens): the router, top-k and expert sort run in
// the same kernel.  Before its programmatic-launch wait each CTA copies the router rows
// of its experts (e = CTA, CTA + grid, ...) to shared memory (weights only); it then
// computes their logits in the router's fixed order R, and after one grid sync every CTA
// selects the top-k of all tokens itself (a rank count in shared memory) and sorts the
// pairs by expert.  With one token, gate/up items go to CTAs strided by the grid (every
// expert shares the staged x) so the first experts finish early, and down ranges run in
// reverse CTA order.  The combine is a merge: the down epilogue writes y per pair; the last
// of a token's resident pairs to finish a 32-column block sums w * y over the token's
// ranks in ascending order (as ftmoe_combine does) and writes out in fp32 and bf16.
#pragma once
#include "decode.cuh"
#include "tc.cuh"

namespace ftmoe {

constexpr int kSdCons = 16;                    // consumer warps
constexpr int kSdEpiWarp = 1 + kSdCons;        // the epilogue warp (after producer and consumers)
constexpr int kSdThreads = (2 + kSdCons) * 32;
constexpr int kSdRowsA = 16;                   // gate (and up) rows per phase-A item
constexpr int kSdRowsB = 32;                   // down rows per phase-B item
// per-expert info: item starts (A, B), first row, rows, slot, tensor scales (3); then the token
// group (token, weight and pair of each row, 8 each) and the scan's chunk totals (2 x 32)
__host__ __device__ inline int sd_info_ints(int E) { return 8 * (E + 8) + 96; }

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

constexpr int kSdMaxStages = 6;
constexpr int kSdRedBufs = 2;       // reduction buffers at most (items alternate between them)
constexpr int kSdCopyPieces = 8;    // bulk copies per streamed weight block
constexpr int kSdRouteMaxT = 8;     // tokens the fused router takes (one token group per expert)

// Layout of one stage and of the kernel's shared memory, for one (d, f, format).  A stage
// holds one item's tile (whole rows: K = d in phase A, f in phase B), which lands with one
// bulk copy.
struct SdLayout {
  int stage_bytes, stages;
  int xrows, estride;         // staged token rows; per-expert info stride (ints)
  int nred;                   // floats per reduction buffer: [warp][m 2][row 16][xrows]
  int nbufs;                  // reduction buffers: 2, or 1 where two would leave fewer than 2 stages
  int route_ints;             // fused router scratch (0 without it)
  int off_x, off_red, off_rank, off_route, off_bar, smem;
};

// fused router scratch: logits [T][E], ids/values/weights/resident flags/sorted pairs [T*k], expected merges [T], offsets [E+1]
__host__ __device__ inline int sd_route_ints(int E, int T, int k) { return T * E + 5 * T * k + T + E + 1; }

// T: tokens of the call (xrows = min(8, T)); route: with the fused router
__host__ __device__ inline SdLayout sd_layout(int E, int d, int f, int fmt, int T, int k, bool route, int max_smem) {
  SdLayout L;
  L.xrows = T < 8 ? T : 8;
  L.estride = E + 8;
  const int sa = sd_block_bytes_a(d, fmt), sb = sd_block_bytes_b(f, fmt);
  L.stage_bytes = ((sa > sb ? sa : sb) + 127) / 128 * 128;
  const int kx = d > f ? d : f;
  const int xbytes = (L.xrows * (kx + 8) * 2 + 127) / 128 * 128;
  L.nred = kSdCons * 2 * 16 * L.xrows;
  const int info = (sd_info_ints(E) * 4 + 15) / 16 * 16;
  L.route_ints = route ? sd_route_ints(E, T, k) : 0;
  const int rbytes = (L.route_ints * 4 + 15) / 16 * 16;
  int red = 0;
  for (L.nbufs = kSdRedBufs; L.nbufs >= 1; --L.nbufs) {
    red = L.nbufs * L.nred * 4;
    L.stages = (max_smem - 1024 - (xbytes + red + info + rbytes + 256)) / L.stage_bytes;
    if (L.stages >= 2 || L.nbufs == 1) break;
  }
  if (L.stages > kSdMaxStages) L.stages = kSdMaxStages;
  L.off_x = L.stages * L.stage_bytes;
  L.off_red = L.off_x + xbytes;
  L.off_rank = L.off_red + red;
  L.off_route = L.off_rank + info;
  L.off_bar = L.off_route + rbytes;
  L.smem = L.off_bar + 256 + 128;
  return L;
}

// Whether the streaming kernel takes this shape: E <= 1024 and at least 2 stages of
// shared memory.  (Every tile copy is a multiple of 16 bytes at a 16-byte boundary:
// d and f are multiples of 128.)
__host__ inline bool sd_supported(int E, int d, int f, int fmt, int T, int k, int max_smem) {
  if (fmt != FTMOE_NVFP4 && fmt != FTMOE_MXFP4) return false;
  if (E > 1024) return false;
  return sd_layout(E, d, f, fmt, T, k, false, max_smem).stages >= 2;
}
// Whether the layer call can fuse the router: T <= 8, the rank count small
// (T * E * E <= 2^22 compares), and this CTA's router rows fit in the ring.
__host__ inline bool sd_route_supported(int E, int d, int f, int fmt, int T, int k, int grid, int max_smem) {
  if (fmt != FTMOE_NVFP4 && fmt != FTMOE_MXFP4) return false;
  if (E > 1024 || T < 1 || T > kSdRouteMaxT || (long long)T * E * E > (1ll << 22)) return false;
  const SdLayout L = sd_layout(E, d, f, fmt, T, k, true, max_smem);
  if (L.stages < 2) return false;
  const long long rows = (E + grid - 1) / grid;
  return rows * d * 2 <= (long long)L.stages * L.stage_bytes;
}

// items per resident expert: rows-blocks x token groups
__device__ __forceinline__ int sd_groups(int cnt, int xrows) { return (cnt + xrows - 1) / xrows; }

// s_a[e], s_b[e]: first phase-A / phase-B item of expert e; totals in s_a[E], s_b[E].
// s_lo, s_cnt, s_slot: the expert's first sorted row, rows and slot (slot_src: the slot table,
// global or a shared copy, or nullptr = slot e).  s_scan: 64 ints of scratch.  All threads.
// The tensor scales are left to sd_tensor_scales (they are needed only by the epilogues).
__device__ __forceinline__ void sd_items(const FfnArgs& a, const int32_t* offsets, const int32_t* slot_src, int xrows,
                                         int* s_a, int* s_b, int* s_lo, int* s_cnt, int* s_slot, int* s_scan) {
  const int ua = a.f / kSdRowsA, ub = a.d / kSdRowsB;
  for (int e = threadIdx.x; e < a.E; e += blockDim.x) {
    const int lo = offsets[e];
    const int cnt = offsets[e + 1] - lo;
    int slot = slot_src ? slot_src[e] : e;
    if (slot >= a.C) {
      if (cnt > 0 && blockIdx.x == 0) set_dev_err(DEV_ERR_BAD_SLOT);
      slot = -1;
    }
    s_lo[e] = lo;
    s_cnt[e] = cnt;
    s_slot[e] = slot;
    const int gr = (cnt > 0 && slot >= 0) ? sd_groups(cnt, xrows) : 0;
    s_a[e] = gr * ua;
    s_b[e] = gr * ub;
  }
  __syncthreads();
  // exclusive scan of s_a and s_b: each warp scans 32-expert chunks, then the chunk totals
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
  const int nch = (a.E + 31) / 32;
  for (int c = warp; c < nch; c += nw) {
    const int e = c * 32 + lane;
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
      s_a[e] = ia - na;
      s_b[e] = ib - nb;
    }
    if (lane == 31) {
      s_scan[c] = ia;
      s_scan[32 + c] = ib;
    }
  }
  __syncthreads();
  if (warp == 0) {
    const int ta = lane < nch ? s_scan[lane] : 0, tb = lane < nch ? s_scan[32 + lane] : 0;
    int ia = ta, ib = tb;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int oa = __shfl_up_sync(0xFFFFFFFFu, ia, off), ob = __shfl_up_sync(0xFFFFFFFFu, ib, off);
      if (lane >= off) {
        ia += oa;
        ib += ob;
      }
    }
    __syncwarp();
    if (lane < nch) {
      s_scan[lane] = ia - ta;
      s_scan[32 + lane] = ib - tb;
    }
    if (lane == 31) {
      s_a[a.E] = ia;
      s_b[a.E] = ib;
    }
  }
  __syncthreads();
  for (int e = threadIdx.x; e < a.E; e += blockDim.x) {
    s_a[e] += s_scan[e >> 5];
    s_b[e] += s_scan[32 + (e >> 5)];
  }
  __syncthreads();
}

// Tensor scales of the experts that have items (threads i0, i0 + step, ...).
__device__ __forceinline__ void sd_tensor_scales(const FfnArgs& a, const int* s_a, const int* s_slot, float* s_ts,
                                                 int i0, int step) {
  for (int e = i0; e < a.E; e += step) {
    if (s_a[e + 1] > s_a[e]) {
      const int slot = s_slot[e];
#pragma unroll
      for (int m = 0; m < 3; ++m) s_ts[3 * e + m] = a.tscale ? a.tscale[slot * 3 + m] : 1.f;
    }
  }
}

struct SdItem {
  int e, slot, lo, cnt, grp, n0;   // expert, slot, first sorted row, tokens, token group, row block
};
// Walks a CTA's items in increasing order without divisions: `it` holds the current item
// (expert e, token group grp, row block n0 < blocks); sd_item_first places it on the first
// item, sd_item_next moves it to the following one.
__device__ __forceinline__ void sd_item_load(SdItem& it, const int* s_lo, const int* s_cnt, const int* s_slot) {
  it.slot = s_slot[it.e];
  it.lo = s_lo[it.e];
  it.cnt = s_cnt[it.e];
}
__device__ __forceinline__ void sd_item_first(SdItem& it, const int* s_start, const int* s_lo, const int* s_cnt,
                                              const int* s_slot, int E, int item, int blocks) {
  it.e = find_expert(s_start, E, item);
  while (item >= s_start[it.e + 1]) ++it.e;
  const int local = item - s_start[it.e];
  it.grp = local / blocks;
  it.n0 = local - it.grp * blocks;
  sd_item_load(it, s_lo, s_cnt, s_slot);
}
__device__ __forceinline__ void sd_item_next(SdItem& it, const int* s_start, const int* s_lo, const int* s_cnt,
                                             const int* s_slot, int item, int blocks) {
  if (item < s_start[it.e + 1]) {
    if (++it.n0 == blocks) {
      it.n0 = 0;
      ++it.grp;
    }
    return;
  }
  do {
    ++it.e;
  } while (item >= s_start[it.e + 1]);
  it.grp = 0;
  it.n0 = 0;
  sd_item_load(it, s_lo, s_cnt, s_slot);
}

// Barrier of the consumer warps and the epilogue warp (named barrier 1; the producer is not in it).
__device__ __forceinline__ void sd_work_sync() { asm volatile("bar.sync 1, %0;" ::"r"((kSdCons + 1) * 32) : "memory"); }

// MMAs of NT 16-row tiles (NT = 2: gate and up, sharing the token fragments) over
// super-blocks [sb_lo, sb_hi) of a staged tile.  Tile m: codes at cbase[m], scales at
// sbase[m], in a prepared block of R rows; this lane's fragment rows are r and r + 8.
// Addresses advance by constant strides per super-block (R is a compile-time constant).
template <int FMT, int NT, int R>
__device__ __forceinline__ void sd_tiles_mma(const uint8_t* const (&cbase)[NT], const uint8_t* const (&sbase)[NT],
                                             int r, const uint16_t* xrow, int sb_lo, int sb_hi, int t,
                                             float (&acc)[NT][4]) {
  constexpr int kCodeStep = 32 * R;                               // bytes of codes per super-block
  constexpr int kScaleStep = (FMT == FTMOE_NVFP4 ? 4 : 2) * R;    // bytes of scales per super-block
  const uint8_t* pc[NT];
  const uint8_t* ps[NT];
#pragma unroll
  for (int m = 0; m < NT; ++m) {
    pc[m] = cbase[m] + ((t >> 1) * R + r) * 16 + (t & 1) * 8 + sb_lo * kCodeStep;
    ps[m] = sbase[m] + (FMT == FTMOE_NVFP4 ? t : (t >> 1)) * R + r + sb_lo * kScaleStep;
  }
  const uint16_t* px = xrow + 64 * sb_lo;
  for (int sb0 = sb_lo; sb0 < sb_hi; sb0 += 8) {
    const int nc = min(8, sb_hi - sb0);
    // MXFP4: rebase the chunk's scales on their maximum exponent.  The maximum runs over both
    // 32-blocks of every super-block, so the four lanes of a row (whose products one MMA
    // sums) share it.
    int e0[NT][2];
#pragma unroll
    for (int m = 0; m < NT; ++m) {
      e0[m][0] = e0[m][1] = 0;
      if (FMT == FTMOE_MXFP4) {
        const uint8_t* q = sbase[m] + r + sb0 * kScaleStep;
        for (int bk = 0; bk < 2 * nc; ++bk) {
          e0[m][0] = max(e0[m][0], int(q[bk * R]));
          e0[m][1] = max(e0[m][1], int(q[bk * R + 8]));
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
      const uint4 x0 = *reinterpret_cast<const uint4*>(px);
      const uint4 x1 = *reinterpret_cast<const uint4*>(px + 8);
      px += 64;
      const uint32_t B[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
#pragma unroll
      for (int m = 0; m < NT; ++m) {
        const uint2 ca = *reinterpret_cast<const uint2*>(pc[m]);
        const uint2 cb = *reinterpret_cast<const uint2*>(pc[m] + 128);
        uint32_t pre0, pre1;
        if (FMT == FTMOE_NVFP4) {
          pre0 = e4m3_f16x2(ps[m][0]);
          pre1 = e4m3_f16x2(ps[m][8]);
        } else {
          pre0 = pow2_f16x2(int(ps[m][0]) - e0[m][0]);
          pre1 = pow2_f16x2(int(ps[m][8]) - e0[m][1]);
        }
        pc[m] += kCodeStep;
        ps[m] += kScaleStep;
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

// Fused router and merge of the layer call (ROUTE): router, outputs and workspace.
struct SdRoute {
  const uint16_t* wr;    // [E][d] bf16 router weights
  const float* bias;     // [E] or nullptr
  int renorm;
  float* logits;         // [T][E] workspace
  int32_t* ids;          // [T][k] out
  float* tw;             // [T][k] out
  unsigned* ready;       // [E] workspace: finished gate/up items per expert (zeroed by the kernel)
  unsigned* merge;       // [T][d/32] workspace: finished down blocks per (token, 32 columns) (zeroed likewise)
  float* ybuf;           // [T*k][d] workspace: y of each (token, rank) pair
  float* out_f32;        // [T][d]
  uint16_t* out_bf16;    // [T][d] or nullptr
  float* part;           // [grid][d] workspace of the slice form: each CTA's partial output
};

__device__ __forceinline__ unsigned long long atom_add_release_u64(unsigned long long* p, unsigned long long v) {
  unsigned long long old;
  asm volatile("atom.add.release.gpu.global.u64 %0, [%1], %2;" : "=l"(old) : "l"(p), "l"(v) : "memory");
  return old;
}
__device__ __forceinline__ unsigned long long ld_acquire_u64(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}
// Release add without a result: the earlier writes of this thread, and those ordered before
// it by a __syncwarp, are visible before the add.
__device__ __forceinline__ void red_add_release(unsigned* p, unsigned v) {
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ unsigned atom_add_acq_rel(unsigned* p, unsigned v) {
  unsigned old;
  asm volatile("atom.add.acq_rel.gpu.global.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}
__device__ __forceinline__ unsigned ld_acquire_u32(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Grid sync of a kernel whose grid is one CTA per SM (one thread per CTA calls it).  The
// arrival counter only grows and is a multiple of the grid size between syncs, so this
// sync ends when it reaches the next multiple.  false = gave up (time limit or abort).
__device__ __forceinline__ bool grid_sync_mono(unsigned long long* w, volatile int* abort) {
  const unsigned long long G = gridDim.x;
  const unsigned long long old = atom_add_release_u64(w, 1ull);
  const unsigned long long target = (old / G + 1) * G;
  const unsigned long long t0 = globaltimer_ns(), lim = wait_limit_ns();
  for (uint32_t it = 0; ld_acquire_u64(w) < target; ++it) {
    if ((it & 63u) == 63u) {
      if (abort && *abort) return false;
      if (globaltimer_ns() - t0 > lim) return false;
    }
  }
  return true;
}

// Waits until *v >= target (bounded); false = gave up.
__device__ __forceinline__ bool wait_count(const unsigned* v, unsigned target, volatile int* abort) {
  const unsigned long long t0 = globaltimer_ns(), lim = wait_limit_ns();
  for (uint32_t it = 0; ld_acquire_u32(v) < target; ++it) {
    if ((it & 63u) == 63u) {
      if (abort && *abort) return false;
      if (globaltimer_ns() - t0 > lim) return false;
    }
  }
  return true;
}

// Router logits of this CTA's experts e = b, b + G, ... for all T tokens, in order R (the
// router's fixed fp32 order: lane j adds the products of its 8-element chunks j, j + 32, ...
// in ascending element order, unfused; lanes combine by a xor butterfly 16 .. 1; bias last).
// Router rows are in shared memory (srow), x is read from global memory.  Consumer warps.
// cl_logit: 0 = write r.logits (global); else the shared-memory address of s_logit [T][E], and
// the logit goes to that address in each of the cl_n CTAs of the cluster (lane q to rank q).
__device__ __forceinline__ void sd_route_logits(const FfnArgs& a, const SdRoute& r, const uint8_t* srow, int ne,
                                                int cw, int lane, int e_first, int e_step, uint32_t cl_logit = 0,
                                                int cl_n = 0) {
  const int S = a.d >> 8;    // chunks per lane
  for (int item = cw; item < ne * a.T; item += kSdCons) {
    const int i = item / a.T, t = item - i * a.T;
    const int e = e_first + i * e_step;
    const uint4* wrow = reinterpret_cast<const uint4*>(srow + size_t(i) * a.d * 2);
    const uint4* xr = reinterpret_cast<const uint4*>(a.x + size_t(t) * a.d);
    const float bias = r.bias ? __ldg(r.bias + e) : 0.f;   // issued beside the x loads
    float acc = 0.f;
    for (int s0 = 0; s0 < S; s0 += 8) {
      uint4 xv[8];
#pragma unroll
      for (int q = 0; q < 8; ++q) xv[q] = __ldg(xr + min(s0 + q, S - 1) * 32 + lane);
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        if (s0 + q < S) {
          const uint4 wv = wrow[(s0 + q) * 32 + lane];
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            const uint32_t ww = (&wv.x)[u >> 1], xx = (&xv[q].x)[u >> 1];
            const float wf = (u & 1) ? bf16_hi(ww) : bf16_lo(ww);
            const float xf = (u & 1) ? bf16_hi(xx) : bf16_lo(xx);
            acc = __fadd_rn(acc, __fmul_rn(xf, wf));
          }
        }
      }
    }
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) acc = __fadd_rn(acc, __shfl_xor_sync(0xFFFFFFFFu, acc, off));
    if (r.bias) acc = __fadd_rn(acc, bias);
    if (cl_logit) {
      if (lane < cl_n) st_cluster_f32(mapa_shared(cl_logit + 4u * uint32_t(t * a.E + e), uint32_t(lane)), acc);
    } else if (lane == 0) {
      r.logits[size_t(t) * a.E + e] = acc;
    }
  }
}

// Router logits of the cluster form: this CTA's experts e_first + i (i < ne) for T tokens, in
// order R (as sd_route_logits), each written into s_logit of every CTA of the cluster.  Warp cw
// takes experts cw and cw + 16 together: x of the token is loaded once into registers with the
// two biases, and the two experts' chains run side by side (their arithmetic is unchanged).
// d <= 2048 (at most 8 chunks per lane).  Consumer warps.  The router rows arrive by one bulk
// copy on rows_bar: a warp waits for it after issuing its first x and bias loads, so that their
// latency overlaps the copy.  Returns false if that wait gave up (abort or wait limit).
__device__ __forceinline__ bool sl_route_logits_cl(const FfnArgs& a, const SdRoute& r, const uint8_t* srow, int ne,
                                                   int cw, int lane, int e_first, uint32_t cl_logit, int cl_n,
                                                   uint32_t rows_bar, volatile int* abort) {
  const int S = a.d >> 8;    // chunks per lane (<= 8)
  bool rows_ready = false;
  for (int i0 = cw; i0 < ne; i0 += 2 * kSdCons) {
    const int i1 = i0 + kSdCons;
    const bool two = i1 < ne;
    const int e0 = e_first + i0, e1 = e_first + (two ? i1 : i0);
    const uint4* w0 = reinterpret_cast<const uint4*>(srow + size_t(i0) * a.d * 2);
    const uint4* w1 = reinterpret_cast<const uint4*>(srow + size_t(two ? i1 : i0) * a.d * 2);
    for (int t = 0; t < a.T; ++t) {
      const uint4* xr = reinterpret_cast<const uint4*>(a.x + size_t(t) * a.d);
      uint4 xv[8];
#pragma unroll
      for (int q = 0; q < 8; ++q) xv[q] = q < S ? __ldg(xr + q * 32 + lane) : make_uint4(0, 0, 0, 0);
      const float b0 = r.bias ? __ldg(r.bias + e0) : 0.f, b1 = r.bias ? __ldg(r.bias + e1) : 0.f;
      if (!rows_ready) {
        if (!mbar_wait_warp(rows_bar, 0, abort)) return false;
        rows_ready = true;
      }
      float acc0 = 0.f, acc1 = 0.f;
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        if (q < S) {
          const uint4 wv0 = w0[q * 32 + lane], wv1 = w1[q * 32 + lane];
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            const uint32_t xx = (&xv[q].x)[u >> 1], ww0 = (&wv0.x)[u >> 1], ww1 = (&wv1.x)[u >> 1];
            const float xf = (u & 1) ? bf16_hi(xx) : bf16_lo(xx);
            acc0 = __fadd_rn(acc0, __fmul_rn(xf, (u & 1) ? bf16_hi(ww0) : bf16_lo(ww0)));
            acc1 = __fadd_rn(acc1, __fmul_rn(xf, (u & 1) ? bf16_hi(ww1) : bf16_lo(ww1)));
          }
        }
      }
#pragma unroll
      for (int off = 16; off >= 1; off >>= 1) {
        acc0 = __fadd_rn(acc0, __shfl_xor_sync(0xFFFFFFFFu, acc0, off));
        acc1 = __fadd_rn(acc1, __shfl_xor_sync(0xFFFFFFFFu, acc1, off));
      }
      if (r.bias) {
        acc0 = __fadd_rn(acc0, b0);
        acc1 = __fadd_rn(acc1, b1);
      }
      if (lane < cl_n) {
        st_cluster_f32(mapa_shared(cl_logit + 4u * uint32_t(t * a.E + e0), uint32_t(lane)), acc0);
        if (two) st_cluster_f32(mapa_shared(cl_logit + 4u * uint32_t(t * a.E + e1), uint32_t(lane)), acc1);
      }
    }
  }
  return true;
}

// Top-k of every token by (logit desc, id asc; NaN last), softmax weights, and the stable
// sort of the pairs by expert, all in shared memory (every CTA computes the same).  All
// threads; ends with __syncthreads.  CTA 0 writes ids and weights.
// logits_in_smem: s_logit already holds the logits (the cluster form); else they are read from r.logits.
__device__ __forceinline__ void sd_route_select(const FfnArgs& a, const SdRoute& r, float* s_logit, int* s_ids,
                                                float* s_val, float* s_wt, int* s_sp, int* s_off,
                                                bool logits_in_smem = false) {
  const int T = a.T, E = a.E, k = a.k, P = T * k;
  const int tid = threadIdx.x, nt = blockDim.x, warp = tid >> 5, lane = tid & 31;
  if (!logits_in_smem) {
    for (int i = tid; i < T * E; i += nt) s_logit[i] = __ldcg(r.logits + i);
    __syncthreads();
  }
  // rank of (t, e) = experts that come before it; the first k ranks are the selection.
  // Four neighbouring threads share a (t, e) and split the comparisons four ways.
  const int n4 = 4 * T * E, n4w = (n4 + 31) & ~31;   // whole warps take part in the shuffles
  for (int i4 = tid; i4 < n4w; i4 += nt) {
    const bool act = i4 < n4;
    const int i = act ? i4 >> 2 : 0, part = i4 & 3;
    const int t = i / E, e = i - t * E;
    const float v = s_logit[i];
    const float* row = s_logit + t * E;
    // part p compares against j = p, p + 4, ...: the four parts of a warp read four
    // neighbouring words (no bank conflict), and the counts add up to the same rank
    const int j1 = act ? E : 0;
    int rank = 0;
    if (!isnan(v)) {
#pragma unroll 8
      for (int j = part; j < j1; j += 4) {
        const float u = row[j];
        rank += (u > v) || (u == v && j < e);
      }
    } else {
#pragma unroll 8
      for (int j = part; j < j1; j += 4) rank += !isnan(row[j]) || j < e;
    }
    rank += __shfl_xor_sync(0xFFFFFFFFu, rank, 1);
    rank += __shfl_xor_sync(0xFFFFFFFFu, rank, 2);
    if (act && part == 0 && rank < k) {
      s_ids[t * k + rank] = e;
      s_val[t * k + rank] = v;
    }
  }
  __syncthreads();
  // weights: warp t, the same arithmetic as the router's select step
  for (int t = warp; t < T; t += nt >> 5) {
    const float m = s_val[t * k];
    float part = 0.f;
    if (r.renorm) {
      part = lane < k ? expf(s_val[t * k + lane] - m) : 0.f;
    } else {
      for (int e = lane; e < E; e += 32) part += expf(s_logit[t * E + e] - m);
    }
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) part += __shfl_xor_sync(0xFFFFFFFFu, part, off);
    if (lane < k) {
      const float w = expf(s_val[t * k + lane] - m) / part;
      s_wt[t * k + lane] = w;
      if (blockIdx.x == 0) {
        r.ids[t * k + lane] = s_ids[t * k + lane];
        r.tw[t * k + lane] = w;
      }
    }
  }
  // expert offsets (pairs with a smaller id), then positions (stable within an expert)
  for (int e = tid; e <= E; e += nt) {
    int c = 0;
#pragma unroll 8
    for (int p = 0; p < P; ++p) c += s_ids[p] < e;
    s_off[e] = c;
  }
  __syncthreads();
  for (int p = tid; p < P; p += nt) {
    const int e = s_ids[p];
    int pos = s_off[e];
#pragma unroll 8
    for (int q = 0; q < p; ++q) pos += s_ids[q] == e;
    s_sp[pos] = p;
  }
  __syncthreads();
}

template <int FMT, bool ROUTE>
__global__ void __launch_bounds__(kSdThreads, 1)
sd_ffn_kernel(FfnArgs a, SdLayout Ls, SdRoute ra, unsigned long long* gsync) {
  extern __shared__ uint8_t sd_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(sd_raw) + 127) & ~uintptr_t(127));
  uint16_t* s_x = reinterpret_cast<uint16_t*>(sm + Ls.off_x);
  float* s_red = reinterpret_cast<float*>(sm + Ls.off_red);   // [buffer][warp][m][16][xrows]
  const int es = Ls.estride;
  int* s_a = reinterpret_cast<int*>(sm + Ls.off_rank);
  int* s_b = s_a + es;
  int* s_lo = s_a + 2 * es;
  int* s_cnt = s_a + 3 * es;
  int* s_slot = s_a + 4 * es;
  float* s_ts = reinterpret_cast<float*>(s_a + 5 * es);   // [E][3]
  int* s_tok = s_a + 8 * es;                               // token group: token of each row
  float* s_w = reinterpret_cast<float*>(s_a + 8 * es + 8); // its combine weight
  int* s_pair = s_a + 8 * es + 16;                         // its pair index
  int* s_scan = s_a + 8 * es + 32;                         // [64] scan scratch
  // fused router scratch
  float* s_logit = reinterpret_cast<float*>(sm + Ls.off_route);
  const int P = a.T * a.k;
  int* s_ids = reinterpret_cast<int*>(s_logit + (ROUTE ? a.T * a.E : 0));
  float* s_val = reinterpret_cast<float*>(s_ids + P);
  float* s_wt = s_val + P;
  int* s_res = reinterpret_cast<int*>(s_wt + P);
  int* s_sp = s_res + P;
  int* s_expect = s_sp + P;
  int* s_off = s_expect + a.T;
  const uint32_t bars = smem_u32(sm + Ls.off_bar);   // full[8] at 0, empty[8] at 64, router rows at 128
  // reduction buffers: red_full[i] (16 consumer arrivals: partials in) at 136 + 8i,
  // red_empty[i] (the epilogue warp's arrival: partials read) at 152 + 8i
  const uint32_t red_full = bars + 136, red_empty = bars + 152;
  volatile int* s_flag = reinterpret_cast<volatile int*>(sm + Ls.off_bar + 176);
  volatile int* s_abort = reinterpret_cast<volatile int*>(sm + Ls.off_bar + 180);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int S = Ls.stages;
  const int G = gridDim.x, b = blockIdx.x;

  if (tid == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(bars + 8 * s, 1);
      mbar_init(bars + 64 + 8 * s, kSdCons);
    }
    mbar_init(bars + 128, 1);
    for (int i = 0; i < kSdRedBufs; ++i) {
      mbar_init(red_full + 8 * i, kSdCons);
      mbar_init(red_empty + 8 * i, 1);
    }
    *s_flag = 1;
    *s_abort = 0;
    mbar_fence_init();
  }
  __syncthreads();
  bool ok = true;
  const int ne = ROUTE ? (a.E > b ? (a.E - b + G - 1) / G : 0) : 0;   // router rows of this CTA
  if (ROUTE) {
    // router rows are weights: their copy may start before the previous kernel has finished
    if (tid == 0 && ne > 0) {
      mbar_arrive_expect_tx(bars + 128, uint32_t(ne * a.d * 2));
      for (int i = 0; i < ne; ++i)
        bulk_load(smem_u32(sm + size_t(i) * a.d * 2), ra.wr + size_t(b + i * G) * a.d, uint32_t(a.d * 2), bars + 128);
    }
  }
  pdl_wait();
  if (ROUTE) {
    // the slot table is read now, while the router step runs
    if (a.slot_of)
      for (int e = tid; e < a.E; e += kSdThreads) s_slot[e] = a.slot_of[e];
    // this call's counters start at zero (the grid sync below orders this before any count)
    const int nz = a.E + a.T * (a.d / 32);
    for (int i = b * kSdThreads + tid; i < nz; i += G * kSdThreads) {
      if (i < a.E) ra.ready[i] = 0u;
      else ra.merge[i - a.E] = 0u;
    }
    if (warp >= 1 && warp <= kSdCons && ne > 0) {
      if (mbar_wait_warp(bars + 128, 0, s_abort)) {
        sd_route_logits(a, ra, sm, ne, warp - 1, lane, b, G);
      } else {
        *s_abort = 1;
      }
    }
    __syncthreads();
    // (the sync's release add orders the CTA's logits, made visible to thread 0 by the barrier)
    if (tid == 0 && !grid_sync_mono(gsync, nullptr)) *s_abort = 1;
    __syncthreads();
    if (*s_abort) {
      ok = false;
      if (tid == 0) set_dev_err(DEV_ERR_GRID_TIMEOUT);
    }
    sd_route_select(a, ra, s_logit, s_ids, s_val, s_wt, s_sp, s_off);
  }
  // the pairs sorted by expert: this kernel's own (ROUTE) or the caller's
  const int32_t* offsets = ROUTE ? s_off : a.offsets;
  const int32_t* spair = ROUTE ? s_sp : a.sorted_pair;
  // slot table: the copy taken during the router step (ROUTE) or the caller's
  const int32_t* slot_src = ROUTE ? (a.slot_of ? s_slot : nullptr) : a.slot_of;
  sd_items(a, offsets, slot_src, Ls.xrows, s_a, s_b, s_lo, s_cnt, s_slot, s_scan);   // all threads
  const int NA = s_a[a.E], NB = s_b[a.E];
  // item ranges of this CTA (32-bit: items * grid stays far below 2^32)
  const int a_lo = int(unsigned(NA) * unsigned(b) / unsigned(G)), a_hi = int(unsigned(NA) * unsigned(b + 1) / unsigned(G));
  // one-token layer call: down ranges in reverse CTA order, so the CTAs that finish their (strided)
  // gate/up items first take the experts whose gate/up items finished first
  const int bb = (ROUTE && a.T == 1) ? G - 1 - b : b;
  const int b_lo = int(unsigned(NB) * unsigned(bb) / unsigned(G)), b_hi = int(unsigned(NB) * unsigned(bb + 1) / unsigned(G));
  const int ua = a.f / kSdRowsA, ub = a.d / kSdRowsB;
  // Item sequence of a phase: contiguous [lo, hi), except the gate/up items of a one-token layer
  // call, which a CTA takes strided by the grid (b, b + G, ...).  With one token every expert
  // shares the staged x, and the strided order finishes the first experts' gate/up items
  // early, so their down items need not wait for the slowest CTA.
  const bool strided_a = ROUTE && a.T == 1;
  auto seq_first = [&](int phase) { return (phase == 0 && strided_a) ? b : (phase ? b_lo : a_lo); };
  auto seq_step = [&](int phase) { return (phase == 0 && strided_a) ? G : 1; };
  auto seq_count = [&](int phase) {
    if (phase == 0 && strided_a) return NA > b ? (NA - b + G - 1) / G : 0;
    return phase ? b_hi - b_lo : a_hi - a_lo;
  };
  const size_t blk_a = sd_block_bytes_a(a.d, FMT), blk_b = sd_block_bytes_b(a.f, FMT);
  const size_t slot_bytes = sd_slot_bytes(a.d, a.f, FMT);

  if (warp == 0) {
    // ---------------- producer ----------------
    uint32_t stage = 0, ph = 0;
    bool pok = ok;
    for (int phase = 0; phase < 2 && pok; ++phase) {
      const int first = seq_first(phase), step = seq_step(phase), count = seq_count(phase);
      const uint32_t bytes = uint32_t(phase ? blk_b : blk_a);
      SdItem it;
      for (int q = 0; q < count && pok; ++q) {
        const int item = first + q * step;
        if (q == 0 || step != 1) sd_item_first(it, phase ? s_b : s_a, s_lo, s_cnt, s_slot, a.E, item, phase ? ub : ua);
        else sd_item_next(it, phase ? s_b : s_a, s_lo, s_cnt, s_slot, item, phase ? ub : ua);
        if (!mbar_wait_warp(bars + 64 + 8 * stage, ph ^ 1, s_abort)) {
          pok = false;
          break;
        }
        if (lane == 0) {
          mbar_arrive_expect_tx(bars + 8 * stage, bytes);
          const uint8_t* src = a.prep_dec + size_t(it.slot) * slot_bytes +
                               (phase ? size_t(a.f / kSdRowsA) * blk_a + size_t(it.n0) * blk_b
                                      : size_t(it.n0) * blk_a);
          bulk_load_split(smem_u32(sm + stage * Ls.stage_bytes), src, bytes, bars + 8 * stage, kSdCopyPieces);
        }
        __syncwarp();
        if (++stage == uint32_t(S)) {
          stage = 0;
          ph ^= 1;
        }
      }
    }
    if (!pok && ok && lane == 0) {
      set_dev_err(DEV_ERR_TIMEOUT);
      *s_abort = 1;
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
      if (ROUTE && ne > 0 && !ok) mbar_wait(bars + 128, 0, nullptr);   // the router rows' copy
    }
    return;
  }

  const int xr = Ls.xrows;
  uint16_t* h16 = reinterpret_cast<uint16_t*>(a.h);
  if (warp == kSdEpiWarp) {
    // ---------------- epilogue warp ----------------
    // Per item, in the consumers' order: wait until the 16 partials are in, reduce them
    // (in warp order), write h / y, free the buffer.  It meets the consumers at their
    // named barriers, so the token group it reads is the current one.
    sd_tensor_scales(a, s_a, s_slot, s_ts, lane, 32);
    if (ROUTE) {
      // which pairs are resident, how many merges each token expects; a token without a
      // resident expert gets zeros (no merge reaches it).  Only this warp reads these.
      for (int p = lane; p < P; p += 32) s_res[p] = s_slot[s_ids[p]] >= 0;
      __syncwarp();
      for (int tk = lane; tk < a.T; tk += 32) {
        int c = 0;
        for (int q = 0; q < a.k; ++q) c += s_res[tk * a.k + q];
        s_expect[tk] = c;
      }
      __syncwarp();
      for (int tk = b; tk < a.T; tk += G) {
        if (s_expect[tk] == 0) {
          for (int c = lane; c < a.d; c += 32) {
            ra.out_f32[size_t(tk) * a.d + c] = 0.f;
            if (ra.out_bf16) ra.out_bf16[size_t(tk) * a.d + c] = 0;
          }
        }
      }
    }
    __syncwarp();
    bool eok = ok;
    int jred = 0;
    unsigned pend_n = 0;   // finished gate/up items of the current expert not yet published
    for (int phase = 0; phase < 2; ++phase) {
      const int first = seq_first(phase), step = seq_step(phase), count = seq_count(phase);
      if (!ROUTE && phase == 1) {
        sd_work_sync();   // the consumers' grid sync happens between these
        sd_work_sync();
        if (!*s_flag) eok = false;
      }
      int staged_e = -1, staged_g = -1;
      SdItem it;
      for (int q = 0; q < count; ++q) {
        const int item = first + q * step;
        if (q == 0 || step != 1) sd_item_first(it, phase ? s_b : s_a, s_lo, s_cnt, s_slot, a.E, item, phase ? ub : ua);
        else sd_item_next(it, phase ? s_b : s_a, s_lo, s_cnt, s_slot, item, phase ? ub : ua);
        const int p0 = it.grp * xr, n = min(xr, it.cnt - p0);
        if (step != 1 ? q == 0 : (it.e != staged_e || it.grp != staged_g)) {
          sd_work_sync();   // (consumers restage the tokens between the two)
          sd_work_sync();
          if (!*s_flag) eok = false;
          staged_e = it.e;
          staged_g = it.grp;
        }
        const int buf = jred & (Ls.nbufs - 1), use = jred >> (Ls.nbufs - 1);
        ++jred;
        if (eok && !mbar_wait_warp(red_full + 8 * buf, use & 1, s_abort)) {
          eok = false;
          *s_abort = 1;
        }
        if (!eok) continue;
        const float* rb = s_red + buf * Ls.nred;
        if (phase == 0) {
          // h = silu(gate) * up for the item's 16 rows and n tokens, stored as f16.  Lane: row
          // lane & 15, tokens (lane >> 4) + 2j.
          float gs[4], us[4];
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const int row = lane & 15, tok = (lane >> 4) + 2 * j;
            gs[j] = us[j] = 0.f;
            if (tok < n) {
#pragma unroll 4
              for (int w = 0; w < kSdCons; ++w) {
                gs[j] += rb[((w * 2 + 0) * 16 + row) * xr + tok];
                us[j] += rb[((w * 2 + 1) * 16 + row) * xr + tok];
              }
            }
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(red_empty + 8 * buf);   // the buffer is free again
          const float tsg = s_ts[3 * it.e + 0], tsu = s_ts[3 * it.e + 1];
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const int row = lane & 15, tok = (lane >> 4) + 2 * j;
            if (tok < n) {
              const float gg = gs[j] * tsg, uu = us[j] * tsu;
              const float h = __fdividef(gg, 1.f + __expf(-gg)) * uu;
              if (!isfinite(h)) set_dev_err(DEV_ERR_NONFINITE);
              h16[size_t(it.lo + p0 + tok) * a.f + it.n0 * kSdRowsA + row] = __half_as_ushort(__float2half_rn(h));
            }
          }
          if (ROUTE) {
            // publish the expert's finished items once, after its last item in this CTA
            ++pend_n;
            if (q + 1 == count || item + step >= s_a[it.e + 1]) {
              __syncwarp();
              if (lane == 0) red_add_release(ra.ready + it.e, pend_n);   // orders the warp's h stores
              pend_n = 0;
            }
          }
        } else {
          // y for the item's 32 columns (lane) and n tokens
          float yv[8];
          const int tile = lane >> 4, row = lane & 15;
#pragma unroll
          for (int tok = 0; tok < 8; ++tok) {
            yv[tok] = 0.f;
            if (tok < n) {
#pragma unroll 4
              for (int q = 0; q < kSdCons / 2; ++q) yv[tok] += rb[(((2 * q + tile) * 2) * 16 + row) * xr + tok];
            }
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(red_empty + 8 * buf);   // the buffer is free again
          const float tsd = s_ts[3 * it.e + 2];
          const int gcol = it.n0 * kSdRowsB + lane;
#pragma unroll
          for (int tok = 0; tok < 8; ++tok) {
            if (tok < n) {
              const float y = yv[tok] * tsd;
              if (!isfinite(y)) set_dev_err(DEV_ERR_NONFINITE);
              if (ROUTE) {
                ra.ybuf[size_t(s_pair[tok]) * a.d + gcol] = y;
              } else if (a.topk_w) {
                atomicAdd(a.y_or_out + size_t(s_tok[tok]) * a.d + gcol, s_w[tok] * y);
              } else {
                a.y_or_out[size_t(it.lo + p0 + tok) * a.d + gcol] = y;
              }
            }
          }
          if (ROUTE) {
            // count this pair in on each of its tokens' 32-column blocks; the last one merges
            __syncwarp();
            int fin = 0;
            if (lane < n) {
              const int tk = s_tok[lane];
              const unsigned old = atom_add_acq_rel(ra.merge + size_t(tk) * (a.d / 32) + it.n0, 1u);
              fin = int(old) + 1 == s_expect[tk];
            }
            unsigned fm = __ballot_sync(0xFFFFFFFFu, fin);   // (the acq_rel add acquired the others' y)
            while (fm) {
              const int tok = __ffs(fm) - 1;
              fm &= fm - 1;
              const int tk = s_tok[tok];
              float o = 0.f;
              for (int q0 = 0; q0 < a.k; q0 += 8) {
                float yq[8];
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                  const int pr = tk * a.k + q0 + q;
                  yq[q] = (q0 + q < a.k && s_res[pr]) ? __ldcg(ra.ybuf + size_t(pr) * a.d + gcol) : 0.f;
                }
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                  const int pr = tk * a.k + q0 + q;
                  if (q0 + q < a.k && s_res[pr]) o = fmaf(s_wt[pr], yq[q], o);
                }
              }
              ra.out_f32[size_t(tk) * a.d + gcol] = o;
              if (ra.out_bf16) ra.out_bf16[size_t(tk) * a.d + gcol] = __bfloat16_as_ushort(__float2bfloat16_rn(o));
            }
          }
        }
      }
    }
    if (!eok && ok) set_dev_err(DEV_ERR_TIMEOUT);
    if (!ROUTE && a.out_bf16) {
      sd_work_sync();
      sd_work_sync();
    }
    return;
  }

  // ---------------- consumers ----------------
  const int cw = warp - 1;                 // consumer warp 0..15
  const int ct = tid - 32;                 // consumer thread 0..511
  const int g = lane >> 2, t = lane & 3;
  uint32_t stage = 0, ph = 0;
  int jred = 0;                            // items done: picks the reduction buffer

  if (!ROUTE && a.out_bf16) {
    float4* o = reinterpret_cast<float4*>(a.y_or_out);
    const long long n4 = (long long)a.T * a.d / 4;
    for (long long i = (long long)b * (kSdCons * 32) + ct; i < n4; i += (long long)G * kSdCons * 32)
      o[i] = make_float4(0.f, 0.f, 0.f, 0.f);
  }

  for (int phase = 0; phase < 2; ++phase) {
    const int first = seq_first(phase), step = seq_step(phase), count = seq_count(phase);
    const int K = phase ? a.f : a.d;
    const int st_x = K + 8;                // staged token row stride (f16)
    if (!ROUTE && phase == 1) {
      // every h of every CTA is written before any is read (the epilogue warp is done with phase A)
      sd_work_sync();
      if (ct == 0) {
        __threadfence();
        if (!grid_sync_mono(gsync, s_abort)) {
          *s_flag = 0;
          set_dev_err(DEV_ERR_GRID_TIMEOUT);
        }
      }
      sd_work_sync();
      if (!*s_flag) {
        ok = false;
        *s_abort = 1;
      }
    }
    // On a failed wait `ok` turns false and the loops keep their shape (every warp still
    // reaches every named barrier), skipping work, so no warp is left waiting.
    int staged_e = -1, staged_g = -1;
    // warp's share: phase A: both matrices, K sixteenth cw; phase B: row tile cw & 1, K eighth cw >> 1
    const int nsb = K / 64;
    const int parts = phase ? kSdCons / 2 : kSdCons;
    const int kp = phase ? (cw >> 1) : cw;
    const int sb_lo = kp * nsb / parts, sb_hi = (kp + 1) * nsb / parts;
    SdItem it;
    for (int q = 0; q < count; ++q) {
      const int item = first + q * step;
      if (q == 0 || step != 1) sd_item_first(it, phase ? s_b : s_a, s_lo, s_cnt, s_slot, a.E, item, phase ? ub : ua);
      else sd_item_next(it, phase ? s_b : s_a, s_lo, s_cnt, s_slot, item, phase ? ub : ua);
      const int p0 = it.grp * xr, n = min(xr, it.cnt - p0);
      if (step != 1 ? q == 0 : (it.e != staged_e || it.grp != staged_g)) {
        if (ROUTE && phase == 1 && ct == 0 && ok) {
          // the expert's h is complete once all of its gate/up items have counted in
          if (!wait_count(ra.ready + it.e, unsigned(s_a[it.e + 1] - s_a[it.e]), s_abort)) {
            *s_flag = 0;
            set_dev_err(DEV_ERR_GRID_TIMEOUT);
          }
        }
        sd_work_sync();   // every warp is done with the previous tokens (and their epilogues)
        if (!*s_flag) {
          ok = false;
          *s_abort = 1;
        }
        if (ct < n) {
          const int p = spair[it.lo + p0 + ct];
          s_pair[ct] = p;
          s_tok[ct] = p / a.k;
          s_w[ct] = a.topk_w ? a.topk_w[p] : 0.f;
        }
        if (ok) {
          const int per = K / 8;
          if (phase == 0) {
            for (int c = ct; c < n * per; c += kSdCons * 32) {
              const int q = c / per, cc = c % per;
              const uint16_t* row = a.x + size_t(spair[it.lo + p0 + q] / a.k) * a.d;
              const uint4 v = __ldg(reinterpret_cast<const uint4*>(row) + cc);
              uint4 hh;
              hh.x = f16x2_of(bf16_lo(v.x), bf16_hi(v.x));
              hh.y = f16x2_of(bf16_lo(v.y), bf16_hi(v.y));
              hh.z = f16x2_of(bf16_lo(v.z), bf16_hi(v.z));
              hh.w = f16x2_of(bf16_lo(v.w), bf16_hi(v.w));
              *reinterpret_cast<uint4*>(s_x + q * st_x + 8 * cc) = hh;
            }
          } else {
            for (int c = ct; c < n * per; c += kSdCons * 32) {
              const int q = c / per, cc = c % per;
              const uint4 v = __ldcg(reinterpret_cast<const uint4*>(h16 + size_t(it.lo + p0 + q) * a.f) + cc);
              *reinterpret_cast<uint4*>(s_x + q * st_x + 8 * cc) = v;
            }
          }
        }
        staged_e = it.e;
        staged_g = it.grp;
        sd_work_sync();
      }
      float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
      if (ok && !mbar_wait_warp(bars + 8 * stage, ph, s_abort)) {
        ok = false;
        *s_abort = 1;
      }
      if (ok) {
        const uint8_t* base = sm + stage * Ls.stage_bytes;
        // MMA token column g: rows past the staged ones read the last staged row (results unused)
        const uint16_t* xrow = s_x + min(g, xr - 1) * st_x + 16 * t;
        if (phase == 0) {
          // [gate codes][up codes][gate scales][up scales], 16 rows each
          const int cb = kSdRowsA * (a.d / 2), sbb = kSdRowsA * (a.d / (FMT == FTMOE_NVFP4 ? 16 : 32));
          const uint8_t* const cbase[2] = {base, base + cb};
          const uint8_t* const sbase[2] = {base + 2 * cb, base + 2 * cb + sbb};
          sd_tiles_mma<FMT, 2, kSdRowsA>(cbase, sbase, g, xrow, sb_lo, sb_hi, t, acc);
        } else {
          // [down codes][down scales], 32 rows; this warp's 16-row half
          const int tile = cw & 1;
          const uint8_t* const cbase[1] = {base};
          const uint8_t* const sbase[1] = {base + kSdRowsB * (a.f / 2)};
          float (&acc1)[1][4] = *reinterpret_cast<float(*)[1][4]>(&acc[0]);
          sd_tiles_mma<FMT, 1, kSdRowsB>(cbase, sbase, tile * 16 + g, xrow, sb_lo, sb_hi, t, acc1);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(bars + 64 + 8 * stage);
      if (++stage == uint32_t(S)) {
        stage = 0;
        ph ^= 1;
      }
      // ---- partials -> reduction buffer; the epilogue warp takes it from there ----
      const int buf = jred & (Ls.nbufs - 1), use = jred >> (Ls.nbufs - 1);
      ++jred;
      float* rb = s_red + buf * Ls.nred;
      if (ok && !mbar_wait_warp(red_empty + 8 * buf, (use & 1) ^ 1, s_abort)) {
        ok = false;
        *s_abort = 1;
      }
      if (!ok) continue;
      const int nm = phase ? 1 : 2;
      for (int m = 0; m < nm; ++m) {
        float* my = rb + ((cw * 2 + m) * 16) * xr;
        if (2 * t < xr) {
          my[g * xr + 2 * t] = acc[m][0];
          my[(g + 8) * xr + 2 * t] = acc[m][2];
        }
        if (2 * t + 1 < xr) {
          my[g * xr + 2 * t + 1] = acc[m][1];
          my[(g + 8) * xr + 2 * t + 1] = acc[m][3];
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(red_full + 8 * buf);
    }
  }
  if (!ok) set_dev_err(DEV_ERR_TIMEOUT);
  if (!ROUTE && a.out_bf16) {
    // every add of every CTA has landed: cast out to bf16
    sd_work_sync();
    if (ct == 0) {
      __threadfence();
      if (!grid_sync_mono(gsync, s_abort)) {
        *s_flag = 0;
        set_dev_err(DEV_ERR_GRID_TIMEOUT);
      }
    }
    sd_work_sync();
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


// ---------------------------------------------------------------------------
// Layer call, slice form (sl_layer_kernel): one token, or up to 8 with NVFP4 weights, d <= 2048.
// Each gate/up item (16 rows of h) also
// carries the down weights that read those 16 values: W_down[:, 16 n0 .. 16 n0 + 16) for all
// d rows, one NVFP4 block (half an MXFP4 block) of K per row.  Right after the epilogue warp
// has made the item's 16 h values, the consumer warps multiply them into the down slice
// (warp w takes rows [w d/16, (w + 1) d/16)) and keep the CTA's partial output for their
// rows in registers, across all of the CTA's items.  With several tokens the h values go by
// batch-token column (zeros for tokens the expert does not serve), so one register per (row,
// token) accumulates across experts.  There is no down phase and no wait on other CTAs' h;
// one grid sync at the end, then every CTA sums the partials of a block of outputs over the
// CTAs in CTA order (deterministic) and writes out in fp32 and bf16.
// The combine weight and the block scale multiply the fp32 MMA result of each slice, so
// out = sum over experts and slices of w * s * (W_slice h_slice): the combine's sum, regrouped.
//
// Prepared slice layout (after the decode layout, shapes with d <= 2048): per slot, per
// slice n0: codes [d/16 row tiles][32 lanes][4 B] (lane (g, t) of a tile: bytes 2t and 2t + 1
// of rows g and g + 8, i.e. K elements 4t .. 4t + 3, the MMA fragment of a K permutation
// that the h operand follows too), then the rows' scales [d] (byte per row).
__host__ __device__ inline bool sl_wanted(int d, int fmt) {
  return (fmt == FTMOE_NVFP4 || fmt == FTMOE_MXFP4) && d % 256 == 0 && d / 256 <= 8;
}
__host__ __device__ inline int sl_slice_bytes(int d) { return 9 * d; }
__host__ __device__ inline size_t sl_slot_bytes(int d, int f) { return size_t(f / kSdRowsA) * sl_slice_bytes(d); }

// Canonical down codes + scales -> slice layout (one thread per output byte).
__global__ void prep_slices_kernel(const uint8_t* down, const uint8_t* ds, int C, int d, int f, int fmt, uint8_t* out) {
  const long long sb = sl_slice_bytes(d);
  const long long per_slot = (long long)(f / kSdRowsA) * sb;
  const long long total = per_slot * C;
  for (long long o = (long long)blockIdx.x * blockDim.x + threadIdx.x; o < total; o += (long long)gridDim.x * blockDim.x) {
    const long long slot = o / per_slot;
    const long long r = o % per_slot;
    const long long n0 = r / sb, q = r % sb;
    uint8_t v;
    if (q < 8ll * d) {
      const long long rt = q / 128;
      const int L = int((q / 4) % 32), j = int(q % 4);
      const int g = L >> 2, t = L & 3;
      const long long row = rt * 16 + g + (j >= 2 ? 8 : 0);
      const int byte = 2 * t + (j & 1);
      v = down[(slot * d + row) * (f / 2) + 8 * n0 + byte];
    } else {
      const long long row = q - 8ll * d;
      v = fmt == FTMOE_NVFP4 ? ds[(slot * d + row) * (f / 16) + n0] : ds[(slot * d + row) * (f / 32) + n0 / 2];
    }
    out[o] = v;
  }
}

struct SlLayout {
  int blk_a, off_d, stage_bytes, stages, estride, nred, xr;
  int off_x, off_red, off_rank, off_route, off_h, off_bar, smem;
};
// T <= 8 tokens: one token group per expert (xr = T staged x rows)
__host__ __device__ inline SlLayout sl_layout(int E, int d, int fmt, int T, int k, int max_smem) {
  SlLayout L;
  L.xr = T;
  L.estride = E + 8;
  L.blk_a = sd_block_bytes_a(d, fmt);
  L.off_d = (L.blk_a + 127) / 128 * 128;
  L.stage_bytes = L.off_d + (sl_slice_bytes(d) + 127) / 128 * 128;
  L.nred = kSdCons * 2 * 16 * T;
  const int xbytes = (T * (d + 8) * 2 + 127) / 128 * 128;
  const int red = kSdRedBufs * L.nred * 4;
  const int info = (sd_info_ints(E) * 4 + 15) / 16 * 16;
  const int rbytes = (sd_route_ints(E, T, k) * 4 + 15) / 16 * 16;
  const int fixed = xbytes + red + info + rbytes + 512 + 256;
  L.stages = (max_smem - 1024 - fixed) / L.stage_bytes;
  if (L.stages > 4) L.stages = 4;
  L.off_x = L.stages * L.stage_bytes;
  L.off_red = L.off_x + xbytes;
  L.off_rank = L.off_red + red;
  L.off_route = L.off_rank + info;
  L.off_h = L.off_route + rbytes;
  L.off_bar = L.off_h + 512;                                   // h: [2 buffers][8 token columns][16] f16
  L.smem = L.off_bar + 256 + 128;
  return L;
}
// Whether a layer call of T tokens takes the slice form (the prepared slices exist for d).
__host__ inline bool sl_supported(int E, int d, int f, int fmt, int T, int k, int grid, int max_smem) {
  if (!sl_wanted(d, fmt) || T < 1 || T > kSdRouteMaxT || E > 1024 || (long long)T * E * E > (1ll << 22)) return false;
  const SlLayout L = sl_layout(E, d, fmt, T, k, max_smem);
  if (L.stages < 2) return false;
  const long long rows = (E + grid - 1) / grid;
  return rows * d * 2 <= (long long)L.stages * L.stage_bytes && f % kSdRowsA == 0;
}

// One token (the slice form with NCOL = 1): the top-k of the E logits in s_logit by (logit
// desc, id asc; NaN last), the weights with the router's arithmetic, then the resident
// selected experts in ascending id: s_rexp[j] the expert, s_rslot[j] its slot and s_sp[j] its
// pair (its rank) for j < *s_nres (their tensor scales are the epilogue warp's to load).  This replaces the
// general selection, pair sort and item scan, whose dependent shared-memory steps dominate a
// one-token call.  All threads; ends with __syncthreads.
// logits_in_smem: s_logit already holds the logits (the cluster form); else they are read from r.logits.
__device__ __forceinline__ void sl_select_t1(const FfnArgs& a, const SdRoute& r, float* s_logit, int* s_ids,
                                             float* s_val, float* s_wt, const int32_t* s_slot_in, int* s_rexp,
                                             int* s_rslot, int* s_sp, float* s_ts, uint32_t* s_bits, int* s_nres,
                                             bool logits_in_smem) {
  const int E = a.E, k = a.k;
  const int tid = threadIdx.x, nt = blockDim.x, warp = tid >> 5, lane = tid & 31;
  for (int i = tid; i < (E + 31) / 32; i += nt) s_bits[i] = 0u;
  if (!logits_in_smem) {
    for (int i = tid; i < E; i += nt) s_logit[i] = __ldcg(r.logits + i);
    __syncthreads();
  }
  // rank of e = experts before it, four threads per expert.  When E % 16 == 0 and 4 E threads
  // fit the block, thread (e, q) reads four-wide words 4i + q of the row: the four q of a warp
  // hit four different bank groups and the eight experts of a warp share each load (a
  // broadcast).  Otherwise part p compares against j = p, p + 4, ...
  const bool wide = (E & 15) == 0 && 4 * E <= nt;
  if (wide && tid < 4 * E) {
    const int e = tid >> 2, q = tid & 3;
    const float v = s_logit[e];
    const float4* row4 = reinterpret_cast<const float4*>(s_logit);
    int c0 = 0, c1 = 0, c2 = 0, c3 = 0;
    if (!isnan(v)) {
#pragma unroll 8
      for (int i = 0; i < (E >> 4); ++i) {
        const int j4 = 4 * i + q, j = 4 * j4;
        const float4 u = row4[j4];
        c0 += (u.x > v) || (u.x == v && j < e);
        c1 += (u.y > v) || (u.y == v && j + 1 < e);
        c2 += (u.z > v) || (u.z == v && j + 2 < e);
        c3 += (u.w > v) || (u.w == v && j + 3 < e);
      }
    } else {
      for (int j = q; j < E; j += 4) c0 += !isnan(s_logit[j]) || j < e;
    }
    int rank = (c0 + c1) + (c2 + c3);
    rank += __shfl_xor_sync(0xFFFFFFFFu, rank, 1);
    rank += __shfl_xor_sync(0xFFFFFFFFu, rank, 2);
    if (q == 0 && rank < k) {
      s_ids[rank] = e;
      s_val[rank] = v;
    }
  }
  const int n4 = wide ? 0 : 4 * E, n4w = (n4 + 31) & ~31;
  for (int i4 = tid; i4 < n4w; i4 += nt) {
    const bool act = i4 < n4;
    const int e = act ? i4 >> 2 : 0, part = i4 & 3;
    const float v = s_logit[e];
    const int j1 = act ? E : 0;
    int rank = 0;
    if (!isnan(v)) {
#pragma unroll 8
      for (int j = part; j < j1; j += 4) {
        const float u = s_logit[j];
        rank += (u > v) || (u == v && j < e);
      }
    } else {
#pragma unroll 8
      for (int j = part; j < j1; j += 4) rank += !isnan(s_logit[j]) || j < e;
    }
    rank += __shfl_xor_sync(0xFFFFFFFFu, rank, 1);
    rank += __shfl_xor_sync(0xFFFFFFFFu, rank, 2);
    if (act && part == 0 && rank < k) {
      s_ids[rank] = e;
      s_val[rank] = v;
    }
  }
  __syncthreads();
  if (warp == 0) {
    // weights: the router's select-step arithmetic (k <= 32: lane r holds rank r)
    const float m = s_val[0];
    float part = 0.f;
    if (r.renorm) {
      part = lane < k ? expf(s_val[lane] - m) : 0.f;
    } else {
      for (int e = lane; e < E; e += 32) part += expf(s_logit[e] - m);
    }
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) part += __shfl_xor_sync(0xFFFFFFFFu, part, off);
    int e = 0, slot = -1;
    if (lane < k) {
      e = s_ids[lane];
      const float w = expf(s_val[lane] - m) / part;
      s_wt[lane] = w;
      if (blockIdx.x == 0) {
        r.ids[lane] = e;
        r.tw[lane] = w;
      }
      slot = s_slot_in ? s_slot_in[e] : e;
      if (slot >= a.C) {
        if (blockIdx.x == 0) set_dev_err(DEV_ERR_BAD_SLOT);
        slot = -1;
      }
      if (slot >= 0) atomicOr(&s_bits[e >> 5], 1u << (e & 31));
    }
    __syncwarp();
    if (slot >= 0) {
      // position among the resident selected experts in ascending id
      int pos = __popc(s_bits[e >> 5] & ((1u << (e & 31)) - 1u));
      for (int w2 = 0; w2 < (e >> 5); ++w2) pos += __popc(s_bits[w2]);
      s_rexp[pos] = e;
      s_rslot[pos] = slot;
      s_sp[pos] = lane;
    }
    const int nres = __popc(__ballot_sync(0xFFFFFFFFu, slot >= 0));
    if (lane == 0) *s_nres = nres;
  }
  __syncthreads();
}

// NCOL: token columns a lane keeps partial outputs for (1 when T = 1: column 0 only; 2 otherwise).
// CL: the cluster form (launched in clusters of 2 to 8 CTAs, grid a multiple of the cluster):
//   - the CTAs of a cluster split the router rows (cluster rank r: experts [r E/n, (r+1) E/n)),
//     write each logit into the shared memory of every CTA of the cluster, and meet at a cluster
//     barrier: no grid-wide sync before the selection;
//   - at the end each CTA leaves its partial output in its shared memory; rank r of a cluster
//     sums slice r of the outputs over the cluster's CTAs in rank order (distributed shared
//     memory) and writes the cluster's partial of that slice; the last cluster to count in on a
//     slice (a counter in the workspace header, set back to 0 after use) sums the clusters'
//     partials in cluster order and writes out.  No CTA waits for another cluster, so the
//     kernel needs no co-residency beyond its own clusters.
// Either way the output is the combine's sum regrouped in a fixed order (deterministic).
template <int FMT, int NCOL, bool CL>
__global__ void __launch_bounds__(kSdThreads, 1)
sl_layer_kernel(FfnArgs a, SlLayout Ls, SdRoute ra, unsigned long long* gsync, const uint8_t* slices,
                unsigned* ccnt) {
  extern __shared__ uint8_t sl_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(sl_raw) + 127) & ~uintptr_t(127));
  uint16_t* s_x = reinterpret_cast<uint16_t*>(sm + Ls.off_x);
  float* s_red = reinterpret_cast<float*>(sm + Ls.off_red);   // [buffer][warp][m][16]
  uint16_t* s_h = reinterpret_cast<uint16_t*>(sm + Ls.off_h);   // [buffer][token column 8][16] f16
  const int es = Ls.estride;
  int* s_a = reinterpret_cast<int*>(sm + Ls.off_rank);
  int* s_b = s_a + es;
  int* s_lo = s_a + 2 * es;
  int* s_cnt = s_a + 3 * es;
  int* s_slot = s_a + 4 * es;
  float* s_ts = reinterpret_cast<float*>(s_a + 5 * es);   // [E][3]
  int* s_tok = s_a + 8 * es;                               // token group: token of each row
  int* s_scan = s_a + 8 * es + 32;
  float* s_logit = reinterpret_cast<float*>(sm + Ls.off_route);
  const int P = a.T * a.k;
  int* s_ids = reinterpret_cast<int*>(s_logit + a.T * a.E);
  float* s_val = reinterpret_cast<float*>(s_ids + P);
  float* s_wt = s_val + P;
  int* s_sp = reinterpret_cast<int*>(s_wt + 2 * P);
  int* s_off = s_sp + P + a.T;
  const int xr = Ls.xr;
  // barriers: full[4] 0, empty[4] 64 (16), router rows 128, red_full[2] 136 (16), red_empty[2]
  // 152 (1), h_full[2] 168 (1), h_empty[2] 184 (16); flags at 208
  const uint32_t bars = smem_u32(sm + Ls.off_bar);
  const uint32_t red_full = bars + 136, red_empty = bars + 152, h_full = bars + 168, h_empty = bars + 184;
  volatile int* s_flag = reinterpret_cast<volatile int*>(sm + Ls.off_bar + 208);
  volatile int* s_abort = reinterpret_cast<volatile int*>(sm + Ls.off_bar + 212);
  volatile int* s_last = reinterpret_cast<volatile int*>(sm + Ls.off_bar + 216);   // cluster form
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int S = Ls.stages;
  const int G = gridDim.x, b = blockIdx.x;

  if (tid == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(bars + 8 * s, 1);
      mbar_init(bars + 64 + 8 * s, kSdCons);
    }
    mbar_init(bars + 128, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(red_full + 8 * i, kSdCons);
      mbar_init(red_empty + 8 * i, 1);
      mbar_init(h_full + 8 * i, 1);
      mbar_init(h_empty + 8 * i, kSdCons);
    }
    *s_flag = 1;
    *s_abort = 0;
    mbar_fence_init();
  }
  __syncthreads();
  bool ok = true;
  // router rows of this CTA: experts e_first + i * e_step, i < ne
  const int csz = CL ? int(cluster_nctarank()) : 1, crank = CL ? int(cluster_ctarank()) : 0;
  const int epc = (a.E + csz - 1) / csz;
  const int e_first = CL ? crank * epc : b, e_step = CL ? 1 : G;
  const int ne = CL ? max(0, min(epc, a.E - crank * epc)) : (a.E > b ? (a.E - b + G - 1) / G : 0);
  if (tid == 0 && ne > 0) {
    // router rows are weights: their copy may start before the previous kernel has finished
    mbar_arrive_expect_tx(bars + 128, uint32_t(ne * a.d * 2));
    for (int i = 0; i < ne; ++i)
      bulk_load(smem_u32(sm + size_t(i) * a.d * 2), ra.wr + size_t(e_first + i * e_step) * a.d, uint32_t(a.d * 2),
                bars + 128);
  }
  // every CTA of the cluster has started before any writes into another's shared memory
  if (CL) asm volatile("barrier.cluster.arrive.relaxed.aligned;\n\tbarrier.cluster.wait.aligned;" ::: "memory");
  pdl_wait();
  // slot_of (which the previous kernel may have written) is loaded here and stored into shared
  // memory after the logits, so that its latency overlaps theirs (E <= 1024 <= 2 x 576 threads)
  static_assert(2 * kSdThreads >= 1024, "two slot_of entries per thread");
  int slot_v[2] = {0, 0};
  if (a.slot_of)
#pragma unroll
    for (int j = 0; j < 2; ++j)
      if (tid + j * kSdThreads < a.E) slot_v[j] = a.slot_of[tid + j * kSdThreads];
  if (warp >= 1 && warp <= kSdCons && ne > 0) {
    bool rok;
    if (CL) {
      rok = sl_route_logits_cl(a, ra, sm, ne, warp - 1, lane, e_first, smem_u32(s_logit), csz, bars + 128, s_abort);
    } else {
      rok = mbar_wait_warp(bars + 128, 0, s_abort);
      if (rok) sd_route_logits(a, ra, sm, ne, warp - 1, lane, e_first, e_step);
    }
    if (!rok) *s_abort = 1;
  }
  if (a.slot_of)
#pragma unroll
    for (int j = 0; j < 2; ++j)
      if (tid + j * kSdThreads < a.E) s_slot[tid + j * kSdThreads] = slot_v[j];
  __syncthreads();
  if (CL) {
    cluster_sync_all();   // every logit of the layer is now in this CTA's s_logit
  } else {
    if (tid == 0 && !grid_sync_mono(gsync, nullptr)) *s_abort = 1;
    __syncthreads();
  }
  // every CTA of this grid is resident (it passed the barrier above): the next kernel on the
  // stream may start its prologue on the SMs that this grid frees
  pdl_launch_dependents();
  if (*s_abort) {
    ok = false;
    if (tid == 0) set_dev_err(CL ? DEV_ERR_TIMEOUT : DEV_ERR_GRID_TIMEOUT);
  }
  const int ua = a.f / kSdRowsA;
  int* s_nres = s_scan + 40;
  if (NCOL == 1) {
    // one token: the resident selected experts in s_a (expert) and s_b (slot), their pairs in s_sp
    sl_select_t1(a, ra, s_logit, s_ids, s_val, s_wt, a.slot_of ? s_slot : nullptr, s_a, s_b, s_sp, s_ts,
                 reinterpret_cast<uint32_t*>(s_scan), s_nres, CL);
  } else {
    sd_route_select(a, ra, s_logit, s_ids, s_val, s_wt, s_sp, s_off, CL);
    sd_items(a, s_off, a.slot_of ? s_slot : nullptr, xr, s_a, s_b, s_lo, s_cnt, s_slot, s_scan);   // all threads
  }
  const int NA = NCOL == 1 ? *s_nres * ua : s_a[a.E];
  // item -> (expert, slot, first sorted row, rows, row block): one token by division, else a search
  auto item_at = [&](SdItem& it, int item) {
    if (NCOL == 1) {
      const int j = item / ua;
      it.e = s_a[j];
      it.slot = s_b[j];
      it.lo = j;
      it.cnt = 1;
      it.grp = 0;
      it.n0 = item - j * ua;
    } else {
      sd_item_first(it, s_a, s_lo, s_cnt, s_slot, a.E, item, ua);
    }
  };
  // items: one token takes b, b + G, ... (every expert shares the staged x); more tokens take a
  // contiguous range (x is restaged per expert)
  const bool strided = a.T == 1;
  const int a_lo = int(unsigned(NA) * unsigned(b) / unsigned(G)), a_hi = int(unsigned(NA) * unsigned(b + 1) / unsigned(G));
  const int first = strided ? b : a_lo, step = strided ? G : 1;
  const int count = strided ? (NA > b ? (NA - b + G - 1) / G : 0) : a_hi - a_lo;
  const size_t blk_a = size_t(Ls.blk_a);
  const size_t slot_bytes = sd_slot_bytes(a.d, a.f, FMT);
  const size_t slice_slot = sl_slot_bytes(a.d, a.f);
  const int RP = a.d / 256;                                // row tiles per consumer warp

  if (warp == 0) {
    // ---------------- producer ----------------
    uint32_t stage = 0, ph = 0;
    bool pok = ok;
    SdItem it;
    for (int q = 0; q < count && pok; ++q) {
      item_at(it, first + q * step);
      if (!mbar_wait_warp(bars + 64 + 8 * stage, ph ^ 1, s_abort)) {
        pok = false;
        break;
      }
      if (lane == 0) {
        const uint32_t full = bars + 8 * stage;
        mbar_arrive_expect_tx(full, uint32_t(blk_a + size_t(sl_slice_bytes(a.d))));
        uint8_t* dst = sm + stage * Ls.stage_bytes;
        bulk_load_split(smem_u32(dst), a.prep_dec + size_t(it.slot) * slot_bytes + size_t(it.n0) * blk_a,
                        uint32_t(blk_a), full, kSdCopyPieces);
        bulk_load_split(smem_u32(dst + Ls.off_d),
                        slices + size_t(it.slot) * slice_slot + size_t(it.n0) * sl_slice_bytes(a.d),
                        uint32_t(sl_slice_bytes(a.d)), full, kSdCopyPieces);
      }
      __syncwarp();
      if (++stage == uint32_t(S)) {
        stage = 0;
        ph ^= 1;
      }
    }
    if (!pok && ok && lane == 0) {
      set_dev_err(DEV_ERR_TIMEOUT);
      *s_abort = 1;
    }
    if (lane == 0) {
      for (int i = 0; i < S; ++i) {
        if (stage == 0) {
          stage = S;
          ph ^= 1;
        }
        --stage;
        mbar_wait(bars + 8 * stage, ph, nullptr);
      }
      if (ne > 0 && !ok) mbar_wait(bars + 128, 0, nullptr);
    }
    goto tail;
  }

  if (warp == kSdEpiWarp) {
    // ---------------- epilogue warp: h of each item into s_h ----------------
    if (NCOL != 1) {
      sd_tensor_scales(a, s_a, s_slot, s_ts, lane, 32);
    } else if (lane < *s_nres) {   // one token: the resident selected experts s_a[j], slots s_b[j]
#pragma unroll
      for (int m3 = 0; m3 < 3; ++m3) s_ts[3 * s_a[lane] + m3] = a.tscale ? a.tscale[s_b[lane] * 3 + m3] : 1.f;
    }
    __syncwarp();
    bool eok = ok;
    SdItem it;
    int staged_e = -1;
    for (int q = 0; q < count; ++q) {
      item_at(it, first + q * step);
      if (strided ? q == 0 : it.e != staged_e) {
        sd_work_sync();   // (the consumers stage x and the token group between these)
        sd_work_sync();
        if (!*s_flag) eok = false;
        staged_e = it.e;
      }
      const int n = min(xr, it.cnt);
      const int buf = q & 1, use = q >> 1;
      if (eok && !mbar_wait_warp(red_full + 8 * buf, use & 1, s_abort)) {
        eok = false;
        *s_abort = 1;
      }
      // lane: row lane & 15, group rows (lane >> 4) + 2j
      float gs[4], us[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        gs[j] = us[j] = 0.f;
        const int tok = (lane >> 4) + 2 * j;
        if (eok && tok < n) {
          const float* rb = s_red + buf * Ls.nred;
#pragma unroll 8
          for (int w = 0; w < kSdCons; ++w) {
            gs[j] += rb[((w * 2 + 0) * 16 + (lane & 15)) * xr + tok];
            us[j] += rb[((w * 2 + 1) * 16 + (lane & 15)) * xr + tok];
          }
        }
      }
      __syncwarp();
      if (eok && lane == 0) mbar_arrive(red_empty + 8 * buf);
      if (eok && !mbar_wait_warp(h_empty + 8 * buf, (use & 1) ^ 1, s_abort)) {
        eok = false;
        *s_abort = 1;
      }
      if (!eok) continue;
      // h by batch-token column (zeros for tokens this expert does not serve; one token: column 0
      // only, the other columns are never read into a kept result)
      uint16_t* hb = s_h + buf * 128;
      if (NCOL == 2) {
        for (int i = lane; i < 128; i += 32) hb[i] = 0;
        __syncwarp();
      }
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int tok = (lane >> 4) + 2 * j;
        if (tok < n) {
          const float gg = gs[j] * s_ts[3 * it.e + 0], uu = us[j] * s_ts[3 * it.e + 1];
          const float h = __fdividef(gg, 1.f + __expf(-gg)) * uu;
          if (!isfinite(h)) set_dev_err(DEV_ERR_NONFINITE);
          hb[s_tok[tok] * 16 + (lane & 15)] = __half_as_ushort(__float2half_rn(h));
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(h_full + 8 * buf);
    }
    if (!eok && ok) set_dev_err(DEV_ERR_TIMEOUT);
    sd_work_sync();   // (between these the consumers write their partials: cluster form; or meet the grid)
    sd_work_sync();
    goto tail;
  }

  // ---------------- consumers ----------------
  {
  const int cw = warp - 1;
  const int ct = tid - 32;
  const int g = lane >> 2, t = lane & 3;
  const int nsb = a.d / 64;
  const int sb_lo = cw * nsb / kSdCons, sb_hi = (cw + 1) * nsb / kSdCons;
  uint32_t stage = 0, ph = 0;
  float yacc[8][2][NCOL];   // [row tile][row g, g + 8][token 2t + j]
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int h2 = 0; h2 < 2; ++h2)
#pragma unroll
      for (int j = 0; j < NCOL; ++j) yacc[i][h2][j] = 0.f;
  // down slice of item j (stage dstage, expert de; this lane's two token columns 2t, 2t + 1
  // carry combine weights w0, w1): fragments of h, 16 x 16 MMAs, scaled partials
  auto down_part = [&](int j, uint32_t dstage, int de, float w0, float w1) {
    const int buf = j & 1, use = j >> 1;
    if (ok && !mbar_wait_warp(h_full + 8 * buf, use & 1, s_abort)) {
      ok = false;
      *s_abort = 1;
    }
    if (ok) {
      const uint32_t b0 = *reinterpret_cast<const uint32_t*>(s_h + buf * 128 + g * 16 + 4 * t);
      const uint32_t b1 = *reinterpret_cast<const uint32_t*>(s_h + buf * 128 + g * 16 + 4 * t + 2);
      __syncwarp();
      if (lane == 0) mbar_arrive(h_empty + 8 * buf);
      const uint8_t* dbase = sm + dstage * Ls.stage_bytes + Ls.off_d;
      const uint8_t* sbase = dbase + 8 * a.d;
      const float tsd = s_ts[3 * de + 2];   // (tensor scales: loaded by the epilogue warp before the first barrier)
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        if (i < RP) {
          const int rt = cw * RP + i;
          const uint32_t c4 = *reinterpret_cast<const uint32_t*>(dbase + (rt * 32 + lane) * 4);
          uint32_t fr[4];
          e2m1x8_to_f16x8(c4, fr);
          float dd[4] = {0.f, 0.f, 0.f, 0.f};
          mma_16816(dd, fr[0], fr[2], fr[1], fr[3], b0, b1);
          const uint8_t s0 = sbase[rt * 16 + g], s1 = sbase[rt * 16 + g + 8];
          const float f0 = (FMT == FTMOE_NVFP4 ? e4m3_to_float(s0) : e8m0_to_float(s0)) * tsd;
          const float f1 = (FMT == FTMOE_NVFP4 ? e4m3_to_float(s1) : e8m0_to_float(s1)) * tsd;
          yacc[i][0][0] = fmaf(f0 * w0, dd[0], yacc[i][0][0]);     // row g, token 2t
          yacc[i][1][0] = fmaf(f1 * w0, dd[2], yacc[i][1][0]);     // row g + 8, token 2t
          if (NCOL == 2) {
            yacc[i][0][NCOL - 1] = fmaf(f0 * w1, dd[1], yacc[i][0][NCOL - 1]);   // row g, token 2t + 1
            yacc[i][1][NCOL - 1] = fmaf(f1 * w1, dd[3], yacc[i][1][NCOL - 1]);   // row g + 8, token 2t + 1
          }
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(bars + 64 + 8 * dstage);   // the stage is free
  };
  int pend_e = -1, staged_e = -1;
  uint32_t pend_stage = 0;
  float pend_w0 = 0.f, pend_w1 = 0.f;
  const int st_x = a.d + 8;
  SdItem it;
  for (int q = 0; q < count; ++q) {
    item_at(it, first + q * step);
    const int n = min(xr, it.cnt);
    if (strided ? q == 0 : it.e != staged_e) {
      // the expert's token group: x rows (f16) and tokens (one token: staged once)
      sd_work_sync();
      if (!*s_flag) {
        ok = false;
        *s_abort = 1;
      }
      if (ct < n) s_tok[ct] = s_sp[it.lo + ct] / a.k;
      if (ok) {
        const int per = a.d / 8;
        for (int c = ct; c < n * per; c += kSdCons * 32) {
          const int qq = c / per, cc = c - qq * per;
          const uint16_t* row = a.x + size_t(s_sp[it.lo + qq] / a.k) * a.d;
          const uint4 v = __ldg(reinterpret_cast<const uint4*>(row) + cc);
          uint4 hh;
          hh.x = f16x2_of(bf16_lo(v.x), bf16_hi(v.x));
          hh.y = f16x2_of(bf16_lo(v.y), bf16_hi(v.y));
          hh.z = f16x2_of(bf16_lo(v.z), bf16_hi(v.z));
          hh.w = f16x2_of(bf16_lo(v.w), bf16_hi(v.w));
          *reinterpret_cast<uint4*>(s_x + qq * st_x + 8 * cc) = hh;
        }
      }
      staged_e = it.e;
      sd_work_sync();
    }
    // this lane's token columns 2t, 2t + 1: the expert's combine weight for each (0 if it does not serve it)
    float w0 = 0.f, w1 = 0.f;
    if (NCOL == 1) {
      if (t == 0) w0 = s_wt[s_sp[it.lo]];   // the one token's pair with this expert
    } else {
      for (int j = 0; j < n; ++j) {
        const int pj = s_sp[it.lo + j], tk = pj / a.k;
        if (tk == 2 * t) w0 = s_wt[pj];
        if (tk == 2 * t + 1) w1 = s_wt[pj];
      }
    }
    // gate/up partials of item q
    float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
    if (ok && !mbar_wait_warp(bars + 8 * stage, ph, s_abort)) {
      ok = false;
      *s_abort = 1;
    }
    if (ok) {
      const uint8_t* base = sm + stage * Ls.stage_bytes;
      const int cb = kSdRowsA * (a.d / 2), sbb = kSdRowsA * (a.d / (FMT == FTMOE_NVFP4 ? 16 : 32));
      const uint8_t* const cbase[2] = {base, base + cb};
      const uint8_t* const sbase[2] = {base + 2 * cb, base + 2 * cb + sbb};
      // MMA token column g: rows past the staged ones read the last staged row (results unused)
      sd_tiles_mma<FMT, 2, kSdRowsA>(cbase, sbase, g, s_x + min(g, xr - 1) * st_x + 16 * t, sb_lo, sb_hi, t, acc);
    }
    const int buf = q & 1, use = q >> 1;
    if (ok && !mbar_wait_warp(red_empty + 8 * buf, (use & 1) ^ 1, s_abort)) {
      ok = false;
      *s_abort = 1;
    }
    if (ok) {
      float* rb = s_red + buf * Ls.nred;
#pragma unroll
      for (int m = 0; m < 2; ++m) {
        float* my = rb + ((cw * 2 + m) * 16) * xr;
        if (2 * t < xr) {
          my[g * xr + 2 * t] = acc[m][0];
          my[(g + 8) * xr + 2 * t] = acc[m][2];
        }
        if (2 * t + 1 < xr) {
          my[g * xr + 2 * t + 1] = acc[m][1];
          my[(g + 8) * xr + 2 * t + 1] = acc[m][3];
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(red_full + 8 * buf);
    }
    // down slice of the previous item (its h is ready by now, or soon)
    if (q > 0) down_part(q - 1, pend_stage, pend_e, pend_w0, pend_w1);
    pend_e = it.e;
    pend_stage = stage;
    pend_w0 = w0;
    pend_w1 = w1;
    if (++stage == uint32_t(S)) {
      stage = 0;
      ph ^= 1;
    }
  }
  if (count > 0) down_part(count - 1, pend_stage, pend_e, pend_w0, pend_w1);
  // this CTA's partial output [token][row]: this lane holds tokens 2t, 2t + 1 of rows g, g + 8.
  // Grid form: to the workspace; cluster form: to this CTA's shared memory, over the ring's
  // bytes.  Every staged tile has landed by now, but another consumer warp may still be reading
  // the down slices of the last two items (a partial of more than off_d bytes reaches stage 0's
  // slice), so in the cluster form the consumers (and the epilogue warp) meet first.
  if (CL) sd_work_sync();
  float* pb = CL ? reinterpret_cast<float*>(sm) : ra.part + size_t(b) * a.T * a.d;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    if (i < RP) {
      const int r0 = (cw * RP + i) * 16 + g;
      if (2 * t < a.T) {
        pb[size_t(2 * t) * a.d + r0] = yacc[i][0][0];
        pb[size_t(2 * t) * a.d + r0 + 8] = yacc[i][1][0];
      }
      if (NCOL == 2 && 2 * t + 1 < a.T) {
        pb[size_t(2 * t + 1) * a.d + r0] = yacc[i][0][NCOL - 1];
        pb[size_t(2 * t + 1) * a.d + r0 + 8] = yacc[i][1][NCOL - 1];
      }
    }
  }
  if (!ok) set_dev_err(DEV_ERR_TIMEOUT);
  if (CL) {
    sd_work_sync();   // (the epilogue warp's second meeting; its first is before the writes above)
  } else {
    sd_work_sync();
    if (ct == 0) {
      __threadfence();
      if (!grid_sync_mono(gsync, s_abort)) {
        *s_flag = 0;
        set_dev_err(DEV_ERR_GRID_TIMEOUT);
      }
    }
    sd_work_sync();
    if (!*s_flag) return;
    // outputs [T d b / G, T d (b + 1) / G) of out [T][d]: sum the CTAs' partials in CTA order
    // (lane-strided, then a fixed butterfly), write out
    const unsigned nout = unsigned(a.T) * unsigned(a.d);
    const int o_lo = int(nout * unsigned(b) / unsigned(G)), o_hi = int(nout * unsigned(b + 1) / unsigned(G));
    for (int o = o_lo + cw; o < o_hi; o += kSdCons) {
      // this lane's partials c = lane, lane + 32, ... loaded together, then added in that order
      float v = 0.f;
      for (int c0 = lane; c0 < G; c0 += 32 * 8) {
        float pv[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) pv[u] = c0 + 32 * u < G ? __ldcg(ra.part + size_t(c0 + 32 * u) * nout + o) : 0.f;
#pragma unroll
        for (int u = 0; u < 8; ++u)
          if (c0 + 32 * u < G) v += pv[u];
      }
#pragma unroll
      for (int off = 16; off >= 1; off >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, off);
      if (lane == 0) {
        ra.out_f32[o] = v;
        if (ra.out_bf16) ra.out_bf16[o] = __bfloat16_as_ushort(__float2bfloat16_rn(v));
      }
    }
  }
  }   // consumers
tail:
  if (CL) {
    cluster_sync_all();   // every CTA of the cluster has its partial in shared memory
    const int n = a.T * a.d, ncl = G / csz, cid = b / csz;
    const int lo = int((long long)n * crank / csz), hi = int((long long)n * (crank + 1) / csz);
    const uint32_t part0 = smem_u32(sm);
    float* cpart = ra.part + size_t(cid) * n;
    for (int o = lo + tid; o < hi; o += kSdThreads) {
      float pv[kMaxClusterSize];   // the cluster's partials of output o, loaded together, added in rank order
#pragma unroll
      for (int q = 0; q < kMaxClusterSize; ++q)
        pv[q] = q < csz ? ld_cluster_f32(mapa_shared(part0 + 4u * uint32_t(o), uint32_t(q))) : 0.f;
      float v = 0.f;
#pragma unroll
      for (int q = 0; q < kMaxClusterSize; ++q)
        if (q < csz) v += pv[q];
      cpart[o] = v;
    }
    __syncthreads();
    // This CTA has read the cluster's shared memory for the last time: it counts in on the cluster
    // barrier now and waits on it just before it exits (no CTA leaves while another still reads
    // its shared memory), so neither the count-in below nor the final sum waits for the cluster.
    cluster_arrive_release();
    if (tid == 0)   // (release: the barrier above orders the CTA's cluster-partial writes before it)
      *s_last = atom_add_acq_rel(ccnt + crank, 1u) == unsigned(ncl - 1);
    __syncthreads();
    if (*s_last) {
      // slice [lo, hi) of out: the clusters' partials in cluster order
      for (int o = lo + tid; o < hi; o += kSdThreads) {
        float v = 0.f;   // in cluster order, sixteen loads in flight at a time
        for (int c0 = 0; c0 < ncl; c0 += 16) {
          float pv[16];
#pragma unroll
          for (int u = 0; u < 16; ++u) pv[u] = c0 + u < ncl ? __ldcg(ra.part + size_t(c0 + u) * n + o) : 0.f;
#pragma unroll
          for (int u = 0; u < 16; ++u)
            if (c0 + u < ncl) v += pv[u];
        }
        ra.out_f32[o] = v;
        if (ra.out_bf16) ra.out_bf16[o] = __bfloat16_as_ushort(__float2bfloat16_rn(v));
      }
      if (tid == 0) ccnt[crank] = 0u;   // zero again for the next call on this workspace
    }
    cluster_wait_acquire();
  }
}

}  // namespace ftmoe
