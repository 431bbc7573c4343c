// a6: global LRU slot map over (layer, expert) keys.
//
// Pages:
//   - at decode time one global LRU of experts admits every missed expert
//     (asapai.co.kr, "Running 753B GLM-5.2 on a single workstation GPU",
//     section "Abandoning fixed offloading in favor of measured bandwidth");
//   - it spans all MoE layers (banandre.com, "The 284B Model on a 32GB GPU
//     Trick", section "Semantic-Aware Caching: Because Agents Lie");
//   - it starts cold (same page, section "Elastic Memory").
//
// Reading:
//   - Each call makes one access per unique expert, in ascending id order.
//   - A hit moves the key to most-recent.
//   - A miss takes the lowest free slot.  Slots are never freed except by a
//     reset, so that is the count of used slots.  Otherwise the miss evicts
//     the least-recent key and reuses its slot.
//
// Device form: one CTA.  The state lives in shared memory for the whole
// launch:
//   - slot_of[L*E];
//   - key, prev and next per slot: a doubly linked recency list, head = most
//     recent, tail = least recent.
// The CTA's threads mark the experts of a call in a bitmap.  Thread 0 then
// walks the set bits in ascending order and applies each access in O(1).
// The sequence of accesses is inherently serial.
#pragma once
#include "common.cuh"

namespace ftmoe {

struct LruState {      // device memory owned by the handle
  int32_t* slot_of;    // [L*E]
  int32_t* key_of;     // [C]
  int32_t* prv;        // [C]
  int32_t* nxt;        // [C]
  int32_t* meta;       // [4]: head, tail, used, (pad)
  long long* totals;   // [2]: accesses, misses
  int L, E, C;
};

constexpr int kLruThreads = 256;

__device__ __forceinline__ void lru_unlink(int s, int* prv, int* nxt, int& head, int& tail) {
  const int p = prv[s], n = nxt[s];
  if (p >= 0) nxt[p] = n; else head = n;
  if (n >= 0) prv[n] = p; else tail = p;
}

__device__ __forceinline__ void lru_push_front(int s, int* prv, int* nxt, int& head, int& tail) {
  prv[s] = -1;
  nxt[s] = head;
  if (head >= 0) prv[head] = s;
  head = s;
  if (tail < 0) tail = s;
}

// Process a sequence of calls: call c = (layer c % Lc, ids of call c).
//   ids: [n_calls][B*k]; layer of call c = layer0 if n_layers_cycle == 0 else c % L.
__global__ void __launch_bounds__(kLruThreads)
lru_kernel(LruState st, const int32_t* ids, int n_calls, int Bk, int layer0, int cycle_layers,
           uint8_t* hit, int32_t* slot, int32_t* evicted, long long capacity, long long* counters_out) {
  extern __shared__ int sm[];
  int* s_slot_of = sm;                      // [L*E]
  int* s_key = s_slot_of + st.L * st.E;     // [C]
  int* s_prv = s_key + st.C;                // [C]
  int* s_nxt = s_prv + st.C;                // [C]
  uint32_t* s_bits = reinterpret_cast<uint32_t*>(s_nxt + st.C);  // [ceil(E/32)]
  __shared__ int s_meta[4];
  __shared__ long long s_tot[2];
  pdl_wait();
  const int LE = st.L * st.E;
  for (int i = threadIdx.x; i < LE; i += blockDim.x) s_slot_of[i] = st.slot_of[i];
  for (int i = threadIdx.x; i < st.C; i += blockDim.x) {
    s_key[i] = st.key_of[i];
    s_prv[i] = st.prv[i];
    s_nxt[i] = st.nxt[i];
  }
  if (threadIdx.x < 4) s_meta[threadIdx.x] = st.meta[threadIdx.x];
  if (threadIdx.x < 2) s_tot[threadIdx.x] = st.totals[threadIdx.x];
  const int nwords = (st.E + 31) >> 5;
  long long out_n = 0;  // thread 0 only
  for (int c = 0; c < n_calls; ++c) {
    const int layer = cycle_layers ? (c % st.L) : layer0;
    for (int i = threadIdx.x; i < nwords; i += blockDim.x) s_bits[i] = 0u;
    __syncthreads();
    for (int i = threadIdx.x; i < Bk; i += blockDim.x) {
      int e = ids[size_t(c) * Bk + i];
      if (e < 0 || e >= st.E) {
        set_dev_err(DEV_ERR_BAD_ID);
        continue;
      }
      atomicOr(&s_bits[e >> 5], 1u << (e & 31));
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      int head = s_meta[0], tail = s_meta[1], used = s_meta[2];
      long long acc = s_tot[0], miss = s_tot[1];
      for (int wd = 0; wd < nwords; ++wd) {
        uint32_t bits = s_bits[wd];
        while (bits) {
          const int e = (wd << 5) + __ffs(bits) - 1;
          bits &= bits - 1;
          const int key = layer * st.E + e;
          int s = s_slot_of[key];
          int h = 1, ev = -1;
          if (s >= st.C) {
            set_dev_err(DEV_ERR_LRU_STATE);
            bits = 0;
            wd = nwords;
            break;
          }
          if (s >= 0) {
            lru_unlink(s, s_prv, s_nxt, head, tail);
          } else {
            h = 0;
            ++miss;
            if (used < st.C) {
              s = used++;
            } else {
              s = tail;
              if (s < 0 || s >= st.C) {  // a broken list: report, stop this call
                set_dev_err(DEV_ERR_LRU_STATE);
                bits = 0;
                wd = nwords;
                break;
              }
              ev = s_key[s];
              if (ev >= 0 && ev < LE) s_slot_of[ev] = -1;
              lru_unlink(s, s_prv, s_nxt, head, tail);
            }
            s_key[s] = key;
            s_slot_of[key] = s;
          }
          lru_push_front(s, s_prv, s_nxt, head, tail);
          ++acc;
          if (out_n < capacity) {
            hit[out_n] = uint8_t(h);
            slot[out_n] = s;
            evicted[out_n] = ev;
          } else {
            set_dev_err(DEV_ERR_LRU_CAPACITY);
          }
          ++out_n;
        }
      }
      s_meta[0] = head;
      s_meta[1] = tail;
      s_meta[2] = used;
      s_tot[0] = acc;
      s_tot[1] = miss;
    }
    __syncthreads();
  }
  for (int i = threadIdx.x; i < LE; i += blockDim.x) st.slot_of[i] = s_slot_of[i];
  for (int i = threadIdx.x; i < st.C; i += blockDim.x) {
    st.key_of[i] = s_key[i];
    st.prv[i] = s_prv[i];
    st.nxt[i] = s_nxt[i];
  }
  if (threadIdx.x < 4) st.meta[threadIdx.x] = s_meta[threadIdx.x];
  if (threadIdx.x < 2) {
    st.totals[threadIdx.x] = s_tot[threadIdx.x];
    if (counters_out) counters_out[threadIdx.x] = s_tot[threadIdx.x];
  }
}

__global__ void lru_reset_kernel(LruState st) {
  pdl_wait();
  const int LE = st.L * st.E;
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < LE; i += gridDim.x * blockDim.x) st.slot_of[i] = -1;
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < st.C; i += gridDim.x * blockDim.x) {
    st.key_of[i] = -1;
    st.prv[i] = -1;
    st.nxt[i] = -1;
  }
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    st.meta[0] = -1;
    st.meta[1] = -1;
    st.meta[2] = 0;
    st.meta[3] = 0;
    st.totals[0] = 0;
    st.totals[1] = 0;
  }
}

static inline size_t lru_smem_bytes(int L, int E, int C) {
  return (size_t(L) * E + 3 * size_t(C) + (E + 31) / 32) * sizeof(int);
}

}  // namespace ftmoe
