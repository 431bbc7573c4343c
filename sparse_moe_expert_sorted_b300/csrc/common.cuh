// Shared device helpers: launch plumbing, the device error word, and the
// decoders of the weight storage formats (E2M1, E4M3, E8M0, bf16).
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <stdint.h>

#include "../../include/ftmoe.h"

namespace ftmoe {

// Device error word: first failing check wins; read and cleared by ftmoe_get_device_error.
__device__ int g_dev_err;

enum DevErr : int {
  DEV_ERR_BAD_ID = 1,        // a top-k id outside [0, E)
  DEV_ERR_BAD_SLOT = 2,      // slot_of[e] >= C
  DEV_ERR_LRU_CAPACITY = 3,  // replay output buffer too small
  DEV_ERR_BAD_LAYER = 4,
  DEV_ERR_LRU_STATE = 5,     // the recency list is inconsistent (never expected)
  DEV_ERR_TIMEOUT = 6,       // a bounded wait on an mbarrier gave up
  DEV_ERR_BAD_PAIR = 7,      // a sorted pair index outside [0, P)
  DEV_ERR_ROWS = 8,          // padded rows beyond the workspace's capacity
  DEV_ERR_NONFINITE = 9,     // a non-finite FFN value (inputs beyond the f16 range on the decode path)
  DEV_ERR_GRID_TIMEOUT = 10, // a bounded grid barrier gave up
};

__device__ __forceinline__ void set_dev_err(int code) { atomicCAS(&g_dev_err, 0, code); }

// Programmatic dependent launch.  Every kernel waits before it touches memory
// that an earlier kernel on the stream may still read or write; only reads
// of immutable data (weights) may come before the wait.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Workspace: the first FTMOE_WS_ZERO_BYTES bytes hold completion counters that
// are zero between calls; buffers follow at 256-byte aligned offsets.
constexpr size_t kWsCounterRoute = 0;     // uint32
constexpr size_t kWsCounterPermute = 4;   // uint32
constexpr size_t kWsBarrierCount = 16;    // uint32: grid barrier arrivals (back to 0 after each barrier)
constexpr size_t kWsBarrierGen = 20;      // uint32: grid barrier generation (only ever incremented)
// uint64: arrivals of the grid syncs of kernels whose grid is exactly one CTA per SM.  Only
// ever incremented, so it stays a multiple of that grid size between syncs.
constexpr size_t kWsGridSync = 24;
// uint32 [16]: per output slice, the clusters that have added their partial (the cluster form
// of the one-kernel decode layer, clusters of up to 16 CTAs; the last one sums and sets it
// back to 0).
constexpr size_t kWsClusterCnt = 64;
constexpr int kMaxClusterSize = 16;
// uint32: tokens the tensor-core router left to its full order-R fallback, and tokens for which
// it recomputed more than k logits in order R (both set by each such call).
constexpr size_t kWsRouteFallback = 128;
constexpr size_t kWsRouteExtra = 132;
constexpr size_t kWsHeader = FTMOE_WS_ZERO_BYTES;
static inline size_t align256(size_t v) { return (v + 255) & ~size_t(255); }

// ---------------------------------------------------------------------------
// number formats
// ---------------------------------------------------------------------------
__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }

// Four bytes of packed E2M1 pairs -> four f16x2 words (exact: every E2M1 value is an f16).
// Byte i holds elements 2i (low nibble) and 2i+1 (high nibble); word i holds them as (lo, hi).
__device__ __forceinline__ void e2m1x8_to_f16x8(uint32_t src, uint32_t out[4]) {
  asm("{\n\t"
      ".reg .b8 q0, q1, q2, q3;\n\t"
      "mov.b32 {q0, q1, q2, q3}, %4;\n\t"
      "cvt.rn.f16x2.e2m1x2 %0, q0;\n\t"
      "cvt.rn.f16x2.e2m1x2 %1, q1;\n\t"
      "cvt.rn.f16x2.e2m1x2 %2, q2;\n\t"
      "cvt.rn.f16x2.e2m1x2 %3, q3;\n\t"
      "}"
      : "=r"(out[0]), "=r"(out[1]), "=r"(out[2]), "=r"(out[3])
      : "r"(src));
}

__device__ __forceinline__ float2 f16x2_to_float2(uint32_t h) {
  __half2 v = *reinterpret_cast<__half2*>(&h);
  return __half22float2(v);
}

// Two E4M3 codes (low byte first) -> float2 (exact).
__device__ __forceinline__ float2 e4m3x2_to_float2(uint16_t v) {
  __half2_raw r = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(v), __NV_E4M3);
  __half2 h = *reinterpret_cast<__half2*>(&r);
  return __half22float2(h);
}

__device__ __forceinline__ float e4m3_to_float(uint8_t v) {
  __half_raw r = __nv_cvt_fp8_to_halfraw(static_cast<__nv_fp8_storage_t>(v), __NV_E4M3);
  return __half2float(*reinterpret_cast<__half*>(&r));
}

// E8M0: 2^(c - 127); c = 0 is the fp32 subnormal 2^-127; c = 255 is NaN.
__device__ __forceinline__ float e8m0_to_float(uint32_t c) {
  if (c == 0) return __uint_as_float(0x00400000u);
  if (c == 255) return __uint_as_float(0x7FC00000u);
  return __uint_as_float(c << 23);
}

// Streaming 128-bit load that does not allocate in L1 (weights are read once).
__device__ __forceinline__ uint4 ld_stream16(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ uint32_t lanemask_lt() {
  uint32_t m;
  asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
  return m;
}

}  // namespace ftmoe
