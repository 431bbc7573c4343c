// a2: stable expert-sorted permutation of the P = T*k (token, rank) pairs.
//
// The pages do not describe this step.  It is what computing each selected
// expert once over a batch requires (banandre.com, "The 284B Model on a 32GB
// GPU Trick", section "Sparsity Is a Lie (But a Useful One)").
//
// Definition (stable counting sort by expert id):
//   offsets[e]    = number of pairs with an id below e
//   sorted_pair   = the pairs ordered by (expert id, pair index)
//   pair_pos[p]   = position of pair p in sorted_pair
//
// Scheme:
//   - Pairs are cut into chunks of kPermChunk, one CTA per chunk.
//   - The position of a pair is
//       offsets[e] + (pairs of e in earlier chunks) + (pairs of e in earlier
//       warps of this chunk) + (pairs of e in lower lanes of its warp).
//     Every term is a count, so no atomic decides any order.
//   - One chunk needs a single kernel.  Several chunks first write per-chunk
//     histograms (permute_hist_kernel), then rank and scatter.
#pragma once
#include "common.cuh"

namespace ftmoe {

constexpr int kPermChunk = 1024;   // pairs per CTA (one per thread)

__device__ __forceinline__ int load_id(const int32_t* ids, int p, int E) {
  int e = ids[p];
  if (e < 0 || e >= E) {
    set_dev_err(DEV_ERR_BAD_ID);
    e = E - 1;
  }
  return e;
}

// hist[c][e] = number of pairs of chunk c with expert e.
__global__ void __launch_bounds__(kPermChunk) permute_hist_kernel(const int32_t* ids, int P, int E, int32_t* hist) {
  extern __shared__ int s_cnt[];  // [E]
  pdl_wait();
  for (int e = threadIdx.x; e < E; e += blockDim.x) s_cnt[e] = 0;
  __syncthreads();
  const int p = blockIdx.x * kPermChunk + threadIdx.x;
  if (p < P) atomicAdd(&s_cnt[load_id(ids, p, E)], 1);
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) hist[size_t(blockIdx.x) * E + e] = s_cnt[e];
}

// Block-wide exclusive scan of s[0..n) in place (n <= 4 * blockDim); returns the total.
__device__ int block_exclusive_scan(int* s, int n, int* s_warp_tot) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  // each thread owns up to 4 consecutive entries
  const int per = (n + blockDim.x - 1) / blockDim.x;
  const int base = threadIdx.x * per;
  int local = 0;
  for (int i = 0; i < per; ++i)
    if (base + i < n) local += s[base + i];
  int incl = local;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    int o = __shfl_up_sync(0xFFFFFFFFu, incl, off);
    if (lane >= off) incl += o;
  }
  if (lane == 31) s_warp_tot[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int v = (lane < nw) ? s_warp_tot[lane] : 0;
    int inc = v;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      int o = __shfl_up_sync(0xFFFFFFFFu, inc, off);
      if (lane >= off) inc += o;
    }
    if (lane < nw) s_warp_tot[lane] = inc - v;  // exclusive warp offsets
    if (lane == 31) s_warp_tot[32] = inc;       // total
  }
  __syncthreads();
  int run = s_warp_tot[warp] + incl - local;
  for (int i = 0; i < per; ++i)
    if (base + i < n) {
      int v = s[base + i];
      s[base + i] = run;
      run += v;
    }
  __syncthreads();
  return s_warp_tot[32];
}

// Rank and scatter one chunk.  hist == nullptr means a single chunk (counts made here).
__global__ void __launch_bounds__(kPermChunk)
permute_rank_kernel(const int32_t* ids, int P, int E, const int32_t* hist, int n_chunks,
                    int32_t* offsets, int32_t* sorted_pair, int32_t* pair_pos) {
  extern __shared__ int smem[];
  int* s_base = smem;              // [E]: first position of expert e for this chunk
  int* s_tot = smem + E;           // [E]: totals, then exclusive offsets
  int* s_wcnt = smem + 2 * E;      // [32][E]: per-warp counts, then per-warp bases
  __shared__ int s_warp_tot[33];
  pdl_wait();
  const int warp = threadIdx.x >> 5;
  const int c = blockIdx.x;
  const int p = c * kPermChunk + threadIdx.x;

  for (int i = threadIdx.x; i < 32 * E; i += blockDim.x) s_wcnt[i] = 0;
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    if (hist) {
      int before = 0, tot = 0;
      for (int cc = 0; cc < n_chunks; ++cc) {
        int h = hist[size_t(cc) * E + e];
        if (cc < c) before += h;
        tot += h;
      }
      s_base[e] = before;
      s_tot[e] = tot;
    } else {
      s_base[e] = 0;
      s_tot[e] = 0;
    }
  }
  __syncthreads();

  const bool active = p < P;
  const int e = active ? load_id(ids, p, E) : -1;
  const uint32_t act = __ballot_sync(0xFFFFFFFFu, active);
  int rank = 0;
  if (active) {
    const uint32_t same = __match_any_sync(act, e);
    rank = __popc(same & lanemask_lt());
    if (rank == 0) s_wcnt[warp * E + e] = __popc(same);
  }
  __syncthreads();
  // per expert: exclusive scan over warps; chunk count into the totals when single-chunk
  for (int x = threadIdx.x; x < E; x += blockDim.x) {
    int run = 0;
    for (int w = 0; w < 32; ++w) {
      int v = s_wcnt[w * E + x];
      s_wcnt[w * E + x] = run;
      run += v;
    }
    if (!hist) s_tot[x] = run;
  }
  __syncthreads();
  const int total = block_exclusive_scan(s_tot, E, s_warp_tot);
  if (c == 0) {
    for (int x = threadIdx.x; x < E; x += blockDim.x) offsets[x] = s_tot[x];
    if (threadIdx.x == 0) offsets[E] = total;
  }
  if (active) {
    const int pos = s_tot[e] + s_base[e] + s_wcnt[warp * E + e] + rank;
    sorted_pair[pos] = p;
    pair_pos[p] = pos;
  }
}

static inline size_t permute_rank_smem(int E) { return size_t(34) * E * sizeof(int); }

// The same stable counting sort done by one CTA over all P pairs, chunk by chunk in pair
// order (used by the router's last CTA for small batches).  Shared memory: permute_block_ints(E, nw)
// ints, nw = warps of the CTA; E <= 4 * blockDim.
__host__ __device__ inline int permute_block_ints(int E, int nw) { return (nw + 2) * E + 33; }

__device__ void permute_block(const int32_t* ids, int P, int E, int32_t* offsets, int32_t* sorted_pair,
                              int32_t* pair_pos, int* sm) {
  const int nw = blockDim.x >> 5, warp = threadIdx.x >> 5;
  int* s_base = sm;                  // [E]: first position of expert e for the current chunk
  int* s_wcnt = sm + E;              // [nw][E]: per-warp counts, then per-warp bases
  int* s_ctot = sm + (nw + 1) * E;   // [E]: the chunk's count per expert
  int* s_wtot = sm + (nw + 2) * E;   // [33]
  for (int e = threadIdx.x; e < E; e += blockDim.x) s_base[e] = 0;
  __syncthreads();
  for (int p = threadIdx.x; p < P; p += blockDim.x) atomicAdd(&s_base[load_id(ids, p, E)], 1);
  __syncthreads();
  const int total = block_exclusive_scan(s_base, E, s_wtot);
  for (int e = threadIdx.x; e < E; e += blockDim.x) offsets[e] = s_base[e];
  if (threadIdx.x == 0) offsets[E] = total;
  for (int base = 0; base < P; base += blockDim.x) {
    for (int i = threadIdx.x; i < nw * E; i += blockDim.x) s_wcnt[i] = 0;
    __syncthreads();
    const int p = base + threadIdx.x;
    const bool active = p < P;
    const int e = active ? load_id(ids, p, E) : -1;
    const uint32_t act = __ballot_sync(0xFFFFFFFFu, active);
    int rank = 0;
    if (active) {
      const uint32_t same = __match_any_sync(act, e);
      rank = __popc(same & lanemask_lt());
      if (rank == 0) s_wcnt[warp * E + e] = __popc(same);
    }
    __syncthreads();
    for (int x = threadIdx.x; x < E; x += blockDim.x) {
      int run = 0;
      for (int w = 0; w < nw; ++w) {
        const int v = s_wcnt[w * E + x];
        s_wcnt[w * E + x] = run;
        run += v;
      }
      s_ctot[x] = run;
    }
    __syncthreads();
    if (active) {
      const int pos = s_base[e] + s_wcnt[warp * E + e] + rank;
      sorted_pair[pos] = p;
      pair_pos[p] = pos;
    }
    __syncthreads();
    for (int x = threadIdx.x; x < E; x += blockDim.x) s_base[x] += s_ctot[x];
  }
}

}  // namespace ftmoe
