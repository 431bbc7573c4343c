// The decode-time expert cache around the global LRU: slot copies (fills from the host
// pool, moves within an arena, migration to a resized arena), the elastic resize of the
// LRU's slot map, and the q* split of a call's experts between two executors.
//
// Pages:
//   - a missed expert is either copied over the host link into the GPU cache or computed
//     where its weights are; for a step with m misses the engine fills q* ~= m B_P / B_H of
//     them (B_P: measured link bandwidth, B_H: measured host-memory bandwidth) and the two
//     partial sums merge exactly (banandre.com, "The 284B Model on a 32GB GPU Trick",
//     section "The q* Policy: Math Instead of Guesses");
//   - the cache is one global LRU that admits every missed expert (asapai.co.kr, "Running
//     753B GLM-5.2 on a single workstation GPU", section "Abandoning fixed offloading in
//     favor of measured bandwidth");
//   - at scheduler safe points the cache is rebuilt under a new VRAM budget without
//     reloading the host pool, and the pool is kept in its final layout in pinned host
//     memory (banandre.com, section "Elastic Memory: The VRAM Budget Is a Suggestion").
#pragma once
#include "lru.cuh"

namespace ftmoe {

// One byte range per slot of an arena array: slot s of src starts at src + s * src_stride,
// slot t of dst at dst + t * dst_stride; `bytes` per slot.  vec16: 16-byte copies (bases,
// strides and bytes are multiples of 16), else 4-byte copies.
struct SlotRegion {
  const uint8_t* src;
  uint8_t* dst;
  unsigned long long src_stride, dst_stride, bytes;
  int vec16;
};
constexpr int kMaxSlotRegions = 12;
struct SlotCopyArgs {
  SlotRegion r[kMaxSlotRegions];
  int nr;
  const int32_t* pairs;     // [n][2]: (source slot, destination slot)
  const int32_t* n_dev;     // device count of pairs, or nullptr
  int n_max;                // pairs available (the count is clamped to it)
  int src_C, dst_C;         // slots of the two arenas (a pair outside them is skipped, device error)
  int same;                 // 1: source and destination are the same arena (identity pairs skipped)
};

// Grid: x over 16-byte chunks of a slot (all regions back to back), y over pairs (strided).
// Source reads are plain loads, so the source may be device memory or pinned host memory
// that the device can address (zero-copy over the host link).
__global__ void __launch_bounds__(256) copy_slots_kernel(SlotCopyArgs a) {
  pdl_wait();
  int n = a.n_dev ? *a.n_dev : a.n_max;
  n = n < 0 ? 0 : (n > a.n_max ? a.n_max : n);
  for (int p = blockIdx.y; p < n; p += gridDim.y) {
    const int s = a.pairs[2 * p], t = a.pairs[2 * p + 1];
    if (s < 0 || s >= a.src_C || t < 0 || t >= a.dst_C) {
      if (threadIdx.x == 0 && blockIdx.x == 0) set_dev_err(DEV_ERR_BAD_SLOT);
      continue;
    }
    if (a.same && s == t) continue;
    for (int ri = 0; ri < a.nr; ++ri) {
      const SlotRegion& R = a.r[ri];
      const uint8_t* src = R.src + (unsigned long long)s * R.src_stride;
      uint8_t* dst = R.dst + (unsigned long long)t * R.dst_stride;
      if (R.vec16) {
        const unsigned long long n16 = R.bytes >> 4;
        const uint4* s4 = reinterpret_cast<const uint4*>(src);
        uint4* d4 = reinterpret_cast<uint4*>(dst);
        const unsigned long long step = (unsigned long long)gridDim.x * blockDim.x;
        unsigned long long i = (unsigned long long)blockIdx.x * blockDim.x + threadIdx.x;
        // four loads in flight per thread before their stores (the host link has a long latency)
        for (; i + 3 * step < n16; i += 4 * step) {
          const uint4 v0 = s4[i], v1 = s4[i + step], v2 = s4[i + 2 * step], v3 = s4[i + 3 * step];
          d4[i] = v0;
          d4[i + step] = v1;
          d4[i + 2 * step] = v2;
          d4[i + 3 * step] = v3;
        }
        for (; i < n16; i += step) d4[i] = s4[i];
      } else {
        const unsigned long long n4 = R.bytes >> 2;
        const uint32_t* s1 = reinterpret_cast<const uint32_t*>(src);
        uint32_t* d1 = reinterpret_cast<uint32_t*>(dst);
        for (unsigned long long i = (unsigned long long)blockIdx.x * blockDim.x + threadIdx.x; i < n4;
             i += (unsigned long long)gridDim.x * blockDim.x)
          d1[i] = s1[i];
      }
    }
  }
}

// Elastic resize of the LRU state (one thread: resizes happen at safe points, between
// calls).  Reads the old state, writes the new one (separate buffers):
//   - the first C_new keys of the recency list (most recent first) stay, the rest are
//     evicted (slot_of = -1);
//   - kept keys in slots < C_new keep their slot; kept keys in slots >= C_new, in
//     ascending slot order, take the freed slots < C_new in ascending order;
//   - moves[i] = (old slot, new slot) of every kept key in ascending old slot; *n_moves
//     = kept keys.  The recency order, the totals and "lowest free slot next" carry over.
// scratch: int32 [C_old] (new slot of each old slot, -1 = evicted).
__global__ void lru_resize_kernel(LruState o, LruState nw, int32_t* scratch, int32_t* moves, int32_t* n_moves) {
  pdl_wait();
  if (blockIdx.x != 0 || threadIdx.x != 0) return;
  const int LE = o.L * o.E;
  for (int i = 0; i < LE; ++i) nw.slot_of[i] = o.slot_of[i];
  for (int s = 0; s < o.C; ++s) scratch[s] = -1;
  // walk the recency list: the first C_new keys stay (bounded by C_old steps)
  int kept = 0, s = o.meta[0];
  for (int guard = 0; s >= 0 && guard < o.C; ++guard) {
    const int nx = o.nxt[s];
    if (s >= o.C) {
      set_dev_err(DEV_ERR_LRU_STATE);
      break;
    }
    if (kept < nw.C) {
      scratch[s] = s;   // provisional: keeps its slot
      ++kept;
    } else {
      const int key = o.key_of[s];
      if (key >= 0 && key < LE) nw.slot_of[key] = -1;
    }
    s = nx;
  }
  // kept keys above the new capacity move to the freed slots below it, both ascending
  int lo = 0;
  for (int hs = nw.C; hs < o.C; ++hs) {
    if (scratch[hs] < 0) continue;
    while (lo < nw.C && lo < o.C && scratch[lo] != -1) ++lo;   // skip kept slots and taken ones
    if (lo >= nw.C || lo >= o.C) {   // cannot happen: kept <= C_new
      set_dev_err(DEV_ERR_LRU_STATE);
      scratch[hs] = -1;
      continue;
    }
    scratch[hs] = lo;
    scratch[lo] = -2;   // taken (an old slot that was evicted, now a destination)
  }
  for (int t = 0; t < nw.C; ++t) {
    nw.key_of[t] = -1;
    nw.prv[t] = -1;
    nw.nxt[t] = -1;
  }
  int nm = 0;
  for (int os = 0; os < o.C; ++os) {
    const int t = scratch[os];
    if (t < 0) continue;
    const int key = o.key_of[os];
    nw.key_of[t] = key;
    if (key >= 0 && key < LE) nw.slot_of[key] = t;
    if (moves) {
      moves[2 * nm] = os;
      moves[2 * nm + 1] = t;
    }
    ++nm;
  }
  // recency list over the new slots, in the old order
  int head = -1, tail = -1, prev = -1;
  s = o.meta[0];
  for (int guard = 0; s >= 0 && s < o.C && guard < o.C; ++guard) {
    const int t = scratch[s];
    if (t >= 0) {
      nw.prv[t] = prev;
      if (prev >= 0) nw.nxt[prev] = t; else head = t;
      prev = t;
      tail = t;
    }
    s = o.nxt[s];
  }
  nw.meta[0] = head;
  nw.meta[1] = tail;
  nw.meta[2] = nm;   // occupied slots are 0 .. nm-1
  nw.meta[3] = 0;
  nw.totals[0] = o.totals[0];
  nw.totals[1] = o.totals[1];
  if (n_moves) *n_moves = nm;
}

// The q* split of one LRU call (the call's accesses: unique ids ascending, hit flags in
// that order).  Reads the LRU's slot table as the call left it.  One CTA.
//   counts[0] = m (misses of the call), [1] = fills now, [2] = fills later, [3] = experts of B.
struct SplitArgs {
  const int32_t* slot_of;    // the LRU table [L][E]
  const int32_t* ids;        // [B*k]
  int Bk, E, layer;
  const uint8_t* hit;        // [accesses]
  double link, host;         // q* bandwidths (GB/s), used when fill_override < 0
  int fill_override;         // >= 0: fill this many (clamped) instead of q*
  int32_t* slot_of_a;        // [E]
  int32_t* slot_of_b;        // [E]
  int32_t* fill_now;         // [<= E][2]
  int32_t* fill_later;       // [<= E][2]
  int32_t* counts;           // [4]
};

__global__ void __launch_bounds__(256) miss_split_kernel(SplitArgs a) {
  __shared__ uint32_t s_bits[32];   // E <= 1024
  pdl_wait();
  const int nwords = (a.E + 31) >> 5;
  for (int i = threadIdx.x; i < nwords; i += blockDim.x) s_bits[i] = 0u;
  for (int e = threadIdx.x; e < a.E; e += blockDim.x) {
    a.slot_of_a[e] = -1;
    a.slot_of_b[e] = -1;
  }
  __syncthreads();
  for (int i = threadIdx.x; i < a.Bk; i += blockDim.x) {
    const int e = a.ids[i];
    if (e < 0 || e >= a.E) {
      set_dev_err(DEV_ERR_BAD_ID);
      continue;
    }
    atomicOr(&s_bits[e >> 5], 1u << (e & 31));
  }
  __syncthreads();
  if (threadIdx.x != 0) return;
  // m: misses of the call
  int n_acc = 0, m = 0;
  for (int wd = 0; wd < nwords; ++wd) n_acc += __popc(s_bits[wd]);
  for (int i = 0; i < n_acc; ++i) m += a.hit[i] == 0;
  int n_fill;
  if (a.fill_override >= 0) {
    n_fill = a.fill_override;
  } else {
    const double q = double(m) * a.link / a.host;   // q* (IEEE fp64, as on the host)
    n_fill = int(floor(q + 0.5));
  }
  n_fill = n_fill < 0 ? 0 : (n_fill > m ? m : n_fill);
  int acc = 0, nn = 0, nl = 0, nb = 0;
  const int32_t* row = a.slot_of + size_t(a.layer) * a.E;
  for (int wd = 0; wd < nwords; ++wd) {
    uint32_t bits = s_bits[wd];
    while (bits) {
      const int e = (wd << 5) + __ffs(bits) - 1;
      bits &= bits - 1;
      const int s = row[e];
      const int pool = a.layer * a.E + e;
      if (s < 0) {
        a.slot_of_b[e] = pool;
        ++nb;
      } else if (a.hit[acc]) {
        a.slot_of_a[e] = s;
      } else if (nn < n_fill) {
        a.slot_of_a[e] = s;
        a.fill_now[2 * nn] = pool;
        a.fill_now[2 * nn + 1] = s;
        ++nn;
      } else {
        a.slot_of_b[e] = pool;
        a.fill_later[2 * nl] = pool;
        a.fill_later[2 * nl + 1] = s;
        ++nl;
        ++nb;
      }
      ++acc;
    }
  }
  a.counts[0] = m;
  a.counts[1] = nn;
  a.counts[2] = nl;
  a.counts[3] = nb;
}

}  // namespace ftmoe
