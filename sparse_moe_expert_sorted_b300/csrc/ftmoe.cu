// ftmoe C ABI: argument checks, workspace layout and kernel launches.
// All kernels live in this one translation unit (they share the device error word).
#include <array>
#include <cstdio>
#include <cstring>
#include <map>
#include <mutex>
#include <new>

#include "common.cuh"
#include "cache.cuh"
#include "combine.cuh"
#include "decode.cuh"
#include "decode_stream.cuh"
#include "ffn_stream.cuh"
#include "lru.cuh"
#include "permute.cuh"
#include "prefill.cuh"
#include "prefill8.cuh"
#include "route.cuh"
#include "route_tc.cuh"

using namespace ftmoe;

struct ftmoe_lru {
  LruState st;
  void* mem;
  int device;
};

namespace {

constexpr int kMaxDevices = 64;
int g_sms[kMaxDevices];

int num_sms() {
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= kMaxDevices) return 148;
  if (!g_sms[dev]) {
    int v = 0;
    cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev);
    g_sms[dev] = v > 0 ? v : 148;
  }
  return g_sms[dev];
}

inline cudaStream_t as_stream(void* s) { return reinterpret_cast<cudaStream_t>(s); }

// Launch with programmatic stream serialisation: the kernel may start while the
// previous kernel on the stream drains; it calls griddepcontrol.wait before
// touching dependent memory.
template <typename... KArgs, typename... Args>
ftmoe_status launch(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                    Args... args) {
  if (smem > 48 * 1024) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem)) != cudaSuccess)
      return FTMOE_ERR_CUDA;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t err = cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
  return err == cudaSuccess ? FTMOE_OK : FTMOE_ERR_CUDA;
}

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool desc_ok(const ftmoe_layer_desc* d) {
  if (!d) return false;
  if (d->E < 1 || d->E > 1024) return false;
  if (d->k < 1 || d->k > 32 || d->k > d->E) return false;
  if (d->d < 256 || d->d % 256) return false;
  if (d->ffn < 128 || d->ffn % 128) return false;
  if (d->fmt < FTMOE_BF16 || d->fmt > FTMOE_FP8_B128) return false;
  if (d->renorm != 0 && d->renorm != 1) return false;
  if (d->fmt == FTMOE_FP8_B128 && (d->d % 128 || d->ffn % 128)) return false;
  return true;
}

constexpr int kMaxT = 1 << 20;

inline int cdiv(long long a, long long b) { return int((a + b - 1) / b); }

// --- workspace layouts -------------------------------------------------------
// The tensor-core router (route_tc.cuh) takes long batches of renormalised routers of 16..256
// experts (a multiple of 16) and d <= 4096; it needs the logits in the workspace.
bool route_tc_ok(const ftmoe_layer_desc* d, int T) {
  return T >= FTMOE_PREFILL_MIN_T && d->renorm == 1 && d->E >= 16 && d->E <= 256 && d->E % 16 == 0 && d->d <= 4096;
}
// header | logits [T][E] | (tensor-core router) expert norms [E] | fallback tokens [T] |
// logits of the second half of K [T][E]
size_t route_ws(const ftmoe_layer_desc* d, int T, bool own_logits) {
  size_t n = kWsHeader;
  if (own_logits) {
    n += align256(size_t(T) * d->E * sizeof(float));
    if (route_tc_ok(d, T))
      n += align256(size_t(d->E) * 4) + align256(size_t(T) * 4) + align256(size_t(T) * d->E * sizeof(float));
  }
  return n;
}
size_t permute_ws(const ftmoe_layer_desc* d, int T) {
  const int P = T * d->k;
  const int nch = cdiv(P, kPermChunk);
  return kWsHeader + (nch > 1 ? align256(size_t(nch) * d->E * sizeof(int)) : 0);
}
// --- tensor-core prefill path (NVFP4) ---------------------------------------
int ffn_path(const ftmoe_layer_desc* d, int T) {
  if (T < FTMOE_PREFILL_MIN_T) return 0;
  if (d->fmt == FTMOE_NVFP4 && d->d % kStageK == 0 && d->ffn % kStageK == 0) return 1;
  if (d->fmt == FTMOE_FP8_B128 && d->d % 256 == 0 && d->ffn % 128 == 0 && d->d / 128 <= kG8MaxKB &&
      d->ffn / 128 <= kG8MaxKB)
    return 2;
  return 0;
}
// The streaming kernels of path 0 index their work items (8-token groups x rows) in 32-bit
// arithmetic, scaled by the grid in places.  A call stays far inside that range when the worst
// case, (pairs / 8 + E) groups times the wider matrix dimension, is at most 2^28 (a 16384-token
// chunk at d 4096 and top-6 needs 5.1e7); larger calls are refused, to be split by tokens.
bool path0_size_ok(const ftmoe_layer_desc* d, int T) {
  const long long groups = ((long long)T * d->k + 7) / 8 + d->E;
  return groups * std::max(d->d, d->ffn) <= (1ll << 28);
}
// N tile of the gate/up GEMM: NH gate rows + NH up rows
int gate_up_nh(const ftmoe_layer_desc* d) { return d->ffn % 128 == 0 ? 128 : 64; }

inline size_t align1k(size_t v) { return (v + 1023) & ~size_t(1023); }

// Padded row capacity: every resident expert's rows rounded up to 128.
size_t tc_rows_cap(const ftmoe_layer_desc* d, int T) {
  const size_t P = size_t(T) * d->k;
  const size_t r = P + size_t(kTileM - 1) * std::min<size_t>(d->E, P);
  return (r + kTileM - 1) / kTileM * kTileM;
}

// header | xq_tok [T][d/2] | sf_tok [T][d/16] | xq [R][d/2] | sfa [R][d/16] | hq [R][f/2] | sfh [R][f/16]
//        | rowmeta [R] int4
struct TcWs {
  size_t rows, xq_tok, sf_tok, xq, sfa, hq, sfh, rowmeta, total;
};
TcWs tc_ws(const ftmoe_layer_desc* d, int T) {
  TcWs w;
  w.rows = tc_rows_cap(d, T);
  size_t o = align1k(kWsHeader);
  w.xq_tok = o; o += align1k(size_t(T) * d->d / 2);
  w.sf_tok = o; o += align1k(size_t(T) * d->d / 16);
  w.xq = o; o += align1k(w.rows * d->d / 2);
  w.sfa = o; o += align1k(w.rows * d->d / 16);
  w.hq = o; o += align1k(w.rows * d->ffn / 2);
  w.sfh = o; o += align1k(w.rows * d->ffn / 16);
  w.rowmeta = o; o += align1k(w.rows * 16);
  w.total = o;
  return w;
}

// FP8 path: header | xq_tok [T][d] | sx_tok [T][d/128] | xq [R][d] | sx [d/128][R] | hq [R][f] | sh [f/128][R]
//           | rowmeta [R] int4
struct Tc8Ws {
  size_t rows, xq_tok, sx_tok, xq, sx, hq, sh, rowmeta, total;
};
Tc8Ws tc8_ws(const ftmoe_layer_desc* d, int T) {
  Tc8Ws w;
  w.rows = tc_rows_cap(d, T);
  size_t o = align1k(kWsHeader);
  w.xq_tok = o; o += align1k(size_t(T) * d->d);
  w.sx_tok = o; o += align1k(size_t(T) * (d->d / 128) * 4);
  w.xq = o; o += align1k(w.rows * d->d);
  w.sx = o; o += align1k(w.rows * (d->d / 128) * 4);
  w.hq = o; o += align1k(w.rows * d->ffn);
  w.sh = o; o += align1k(w.rows * (d->ffn / 128) * 4);
  w.rowmeta = o; o += align1k(w.rows * 16);
  w.total = o;
  return w;
}

size_t ffn_ws(const ftmoe_layer_desc* d, int T) {
  if (ffn_path(d, T) == 1) return tc_ws(d, T).total;
  if (ffn_path(d, T) == 2) return tc8_ws(d, T).total;
  const size_t P = size_t(T) * d->k;
  return kWsHeader + align256(P * d->ffn * sizeof(float));
}

// prepared scale blocks: gate/up [C][f/NH][d/64][atoms][512] | down [C][d/128][f/64][512]
size_t prep_gate_up_bytes(const ftmoe_layer_desc* d, int C) {
  const int nh = gate_up_nh(d);
  return size_t(C) * (d->ffn / nh) * (d->d / 64) * ((2 * nh + 127) / 128) * kSfBlock;
}
size_t prep_down_bytes(const ftmoe_layer_desc* d, int C) {
  return size_t(C) * (d->d / 128) * (d->ffn / 64) * kSfBlock;
}
// prepared buffer: [prefill scale blocks (NVFP4, d and ffn multiples of 256)][decode layout (NVFP4, MXFP4)]
size_t prep_prefill_bytes(const ftmoe_layer_desc* d, int C) {
  if (d->fmt != FTMOE_NVFP4 || d->d % kStageK || d->ffn % kStageK) return 0;
  return align1k(prep_gate_up_bytes(d, C)) + prep_down_bytes(d, C);
}
size_t prep_decode_offset(const ftmoe_layer_desc* d, int C) { return align1k(prep_prefill_bytes(d, C)); }
// decode layout [C][slot] then, where the one-token slice form applies (d <= 2048), the
// down slices [C][slot]
size_t prep_slices_bytes(const ftmoe_layer_desc* d, int C) {
  return sl_wanted(d->d, d->fmt) ? size_t(C) * sl_slot_bytes(d->d, d->ffn) : 0;
}
size_t prep_decode_bytes(const ftmoe_layer_desc* d, int C) {
  if (d->fmt != FTMOE_NVFP4 && d->fmt != FTMOE_MXFP4) return 0;
  return size_t(C) * sd_slot_bytes(d->d, d->ffn, d->fmt) + prep_slices_bytes(d, C);
}
size_t prep_slices_offset(const ftmoe_layer_desc* d, int C) {
  return prep_decode_offset(d, C) + size_t(C) * sd_slot_bytes(d->d, d->ffn, d->fmt);
}
size_t prep_bytes(const ftmoe_layer_desc* d, int C) {
  const size_t dec = prep_decode_bytes(d, C);
  return dec ? prep_decode_offset(d, C) + dec : prep_prefill_bytes(d, C);
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_tiled() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// 2D byte matrix [rows][row_bytes], boxes of 128 bytes x box_rows, 128-byte swizzle
bool make_map(CUtensorMap* m, const void* base, size_t row_bytes, size_t rows, int box_rows) {
  EncodeTiledFn enc = encode_tiled();
  if (!enc) return false;
  cuuint64_t dims[2] = {cuuint64_t(row_bytes), cuuint64_t(rows)};
  cuuint64_t strides[1] = {cuuint64_t(row_bytes)};
  cuuint32_t box[2] = {128u, cuuint32_t(box_rows)};
  cuuint32_t es[2] = {1u, 1u};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// perm_*: optional fused permutation (only when the router's last CTA selects, and P fits one CTA);
// *fused_perm tells whether it was done.
bool route_can_permute(const ftmoe_layer_desc* d, int T) {
  return T <= kSelectSmallT && T * d->k <= kPermChunk;
}
// tc: the logits are scratch (the caller does not read them), so the tensor-core router may
// take the call; its norms and fallback list follow the logits in the workspace.
ftmoe_status route_impl(const ftmoe_layer_desc* d, const uint16_t* x, const uint16_t* wr, const float* bias, int T,
                        int32_t* ids, float* w, float* logits, void* ws, cudaStream_t st, int32_t* perm_off = nullptr,
                        int32_t* perm_sp = nullptr, int32_t* perm_pp = nullptr, bool tc = false) {
  RouteArgs a;
  const bool fp = perm_off && route_can_permute(d, T);
  a.perm_off = fp ? perm_off : nullptr;
  a.perm_sp = fp ? perm_sp : nullptr;
  a.perm_pp = fp ? perm_pp : nullptr;
  const size_t psm = fp ? size_t(permute_block_ints(d->E, kRouteWarps)) * sizeof(int) : 0;
  a.x = x;
  a.wr = wr;
  a.bias = bias;
  a.T = T;
  a.E = d->E;
  a.d = d->d;
  a.k = d->k;
  a.renorm = d->renorm;
  a.logits = logits ? logits : reinterpret_cast<float*>(static_cast<char*>(ws) + kWsHeader);
  a.ids = ids;
  a.w = w;
  a.counter = reinterpret_cast<unsigned*>(static_cast<char*>(ws) + kWsCounterRoute);
  const int fused = T <= kSelectSmallT;
  const int sms = num_sms();
  ftmoe_status s;
  dim3 blk(kRouteWarps * 32);
  if (tc && route_tc_ok(d, T) && encode_tiled()) {
    RtcArgs r;
    r.x = x;
    r.wr = wr;
    r.bias = bias;
    r.T = T;
    r.E = d->E;
    r.d = d->d;
    r.k = d->k;
    r.logits = a.logits;
    char* extra = reinterpret_cast<char*>(a.logits) + align256(size_t(T) * d->E * sizeof(float));
    r.wnorm = reinterpret_cast<float*>(extra);
    r.fb_list = reinterpret_cast<int32_t*>(extra + align256(size_t(d->E) * 4));
    r.logits2 = reinterpret_cast<float*>(extra + align256(size_t(d->E) * 4) + align256(size_t(T) * 4));
    r.fb_count = reinterpret_cast<unsigned*>(static_cast<char*>(ws) + kWsRouteFallback);
    r.extra_count = reinterpret_cast<unsigned*>(static_cast<char*>(ws) + kWsRouteExtra);
    r.ids = ids;
    r.w = w;
    CUtensorMap tmX, tmW;
    if (!make_map(&tmX, x, size_t(d->d) * 2, size_t(T), kTileM) || !make_map(&tmW, wr, size_t(d->d) * 2, size_t(d->E), d->E))
      return FTMOE_ERR_CUDA;
    s = launch(rtc_prep_kernel, dim3(std::max(1, std::min(cdiv(d->E, 8), sms))), dim3(256), 0, st, r);
    if (s != FTMOE_OK) return s;
    const int tiles = cdiv(T, kTileM);
    // fewer tiles than half the SMs: two CTAs per tile, each over half of K
    r.ksplit = (2 * tiles <= sms && (d->d / 64) % 2 == 0) ? 2 : 1;
    s = launch(rtc_logits_kernel, dim3(std::min(tiles * r.ksplit, sms)), dim3(kRtcThreads), size_t(rtc_smem(d->E)), st,
               tmX, tmW, r, d->E);
    if (s != FTMOE_OK) return s;
    const dim3 sg(std::min(cdiv(T, 8), sms * 4));
    const size_t xs8 = 8 * 8 * 512, xs16 = 8 * 16 * 512;   // per-warp x rows in shared memory
    if (d->d <= 2048)
      s = d->E <= 128 ? launch(rtc_select_kernel<8, 4>, sg, dim3(256), xs8, st, r)
                      : launch(rtc_select_kernel<8, 8>, sg, dim3(256), xs8, st, r);
    else
      s = d->E <= 128 ? launch(rtc_select_kernel<16, 4>, sg, dim3(256), xs16, st, r)
                      : launch(rtc_select_kernel<16, 8>, sg, dim3(256), xs16, st, r);
    if (s != FTMOE_OK) return s;
    return launch(rtc_fallback_kernel, dim3(sms), dim3(256), 0, st, r);
  }
  if (T == 1) {
    const int items = d->E;
    s = launch(route_logits_kernel<1, 1, 8>, dim3(std::min(cdiv(items, kRouteWarps), sms * 8)), blk, psm, st, a,
               fused);
  } else if (T <= 64) {
    const int items = d->E * cdiv(T, 8);
    s = launch(route_logits_kernel<1, 8, 2>, dim3(std::min(cdiv(items, kRouteWarps), sms * 8)), blk, psm, st, a,
               fused);
  } else {
    const long long items = (long long)cdiv(d->E, 4) * cdiv(T, 8);
    s = launch(route_logits_kernel<4, 8, 1>, dim3((unsigned)std::min<long long>(cdiv(items, kRouteWarps), sms * 8)),
               blk, 0, st, a, fused);
  }
  if (s != FTMOE_OK || fused) return s;
  return launch(route_select_kernel, dim3(std::min(cdiv(T, kRouteWarps), sms * 8)), blk, 0, st, a);
}

ftmoe_status permute_impl(const ftmoe_layer_desc* d, const int32_t* ids, int T, int32_t* off, int32_t* sp,
                          int32_t* pp, void* ws, cudaStream_t st) {
  const int P = T * d->k;
  const int nch = cdiv(P, kPermChunk);
  const int E = d->E;
  if (nch == 1)
    return launch(permute_rank_kernel, dim3(1), dim3(kPermChunk), permute_rank_smem(E), st, ids, P, E,
                  (const int32_t*)nullptr, 1, off, sp, pp);
  int32_t* hist = reinterpret_cast<int32_t*>(static_cast<char*>(ws) + kWsHeader);
  ftmoe_status s = launch(permute_hist_kernel, dim3(nch), dim3(kPermChunk), size_t(E) * sizeof(int), st, ids, P, E, hist);
  if (s != FTMOE_OK) return s;
  return launch(permute_rank_kernel, dim3(nch), dim3(kPermChunk), permute_rank_smem(E), st, ids, P, E,
                (const int32_t*)hist, nch, off, sp, pp);
}

template <int FMT>
ftmoe_status ffn_stream_launch(const FfnArgs& a, int P, cudaStream_t st) {
  const int sms = num_sms();
  const long long tiles = cdiv(P, kTokTile) + std::min(a.E, P);
  const long long items_gu = tiles * a.f, items_d = tiles * a.d;
  const int cap = sms * 16;
  dim3 blk(kFfnWarps * 32);
  ftmoe_status s = launch(ffn_gate_up_kernel<FMT>, dim3((unsigned)std::min<long long>(cdiv(items_gu, kFfnWarps), cap)),
                          blk, 0, st, a);
  if (s != FTMOE_OK) return s;
  return launch(ffn_down_kernel<FMT>, dim3((unsigned)std::min<long long>(cdiv(items_d, kFfnWarps), cap)), blk, 0, st, a);
}

// CTAs of `kern` that fit on one SM with `smem` dynamic bytes (0 on error).
template <typename K>
int resident_ctas(K kern, int threads, size_t smem) {
  if (smem > 48 * 1024 &&
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem)) != cudaSuccess)
    return 0;
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, threads, smem) != cudaSuccess) return 0;
  return n;
}

// Decode path of the 4-bit block-scaled formats: one persistent kernel whose CTAs are all
// resident (its two phases meet at a grid barrier), over 16-row units.
// hdr: the workspace's zero header (grid barrier words).
int max_smem_optin() {
  int dev = 0, v = 0;
  cudaGetDevice(&dev);
  if (cudaDeviceGetAttribute(&v, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess || v <= 0) v = 232448;
  return v;
}

template <int FMT>
ftmoe_status ffn_dec_launch(const FfnArgs& a, int P, void* hdr, cudaStream_t st) {
  unsigned* cnt = reinterpret_cast<unsigned*>(static_cast<char*>(hdr) + kWsBarrierCount);
  unsigned* gen = reinterpret_cast<unsigned*>(static_cast<char*>(hdr) + kWsBarrierGen);
  const int ms = max_smem_optin();
  if (a.prep_dec && sd_supported(a.E, a.d, a.f, FMT, a.T, a.k, ms)) {
    // streaming form: one CTA per SM, bulk copies into a shared-memory ring
    const SdLayout Ls = sd_layout(a.E, a.d, a.f, FMT, a.T, a.k, false, ms);
    const int per_sm = resident_ctas(sd_ffn_kernel<FMT, false>, kSdThreads, size_t(Ls.smem));
    if (per_sm < 1) return FTMOE_ERR_CUDA;
    unsigned long long* gs = reinterpret_cast<unsigned long long*>(static_cast<char*>(hdr) + kWsGridSync);
    return launch(sd_ffn_kernel<FMT, false>, dim3(num_sms()), dim3(kSdThreads), size_t(Ls.smem), st, a, Ls, SdRoute{},
                  gs);
  }
  const size_t smem = dec_smem_bytes(std::max(a.d, a.f));
  const int per_sm = resident_ctas(dec_ffn_kernel<FMT>, kDecWarps * 32, smem);
  if (per_sm < 1) return FTMOE_ERR_CUDA;
  const long long experts = std::min(a.E, P);
  const long long units = experts * (std::max(a.d, a.f) / 16);
  const int grid = (int)std::min<long long>(units, (long long)per_sm * num_sms());
  return launch(dec_ffn_kernel<FMT>, dim3(grid), dim3(kDecWarps * 32), smem, st, a, cnt, gen);
}

bool weights_ok(const ftmoe_layer_desc* d, const ftmoe_weights* w) {
  if (!w) return false;
  if (w->fmt != d->fmt || w->d != d->d || w->ffn != d->ffn || w->C < 1) return false;
  if (!w->gate || !w->up || !w->down) return false;
  if (!aligned16(w->gate) || !aligned16(w->up) || !aligned16(w->down)) return false;
  if (d->fmt != FTMOE_BF16) {
    if (!w->gate_scale || !w->up_scale || !w->down_scale) return false;
    if (!aligned16(w->gate_scale) || !aligned16(w->up_scale) || !aligned16(w->down_scale)) return false;
  }
  if (d->fmt == FTMOE_NVFP4 && !w->tensor_scale) return false;
  return true;
}

template <int MODE, int NH>
ftmoe_status launch_gemm(const CUtensorMap& ta, const CUtensorMap& tb0, const CUtensorMap& tb1, const GemmArgs& g,
                         int max_tiles, cudaStream_t st) {
  const int grid = std::max(1, std::min(num_sms(), max_tiles));
  return launch(gemm_kernel<MODE, NH>, dim3(grid), dim3(kGemmNvThreads), size_t(GemmCfg<MODE, NH>::SMEM), st, ta, tb0,
                tb1, g);
}

// Path 1: gather + quantise x, gate/up GEMM (SwiGLU + quantise h), down GEMM (fused combine or y).
// zero_out: optional fp32 [T][d] zeroed by the first kernel (the layer call's accumulator).
ftmoe_status ffn_tc_impl(const ftmoe_layer_desc* d, const ftmoe_weights* w, const int32_t* slot_of,
                         const uint16_t* x, int T, const int32_t* off, const int32_t* sp, const float* topk_w,
                         float* y_or_out, void* ws, float* zero_out, cudaStream_t st) {
  if (!w->prepared || !aligned16(w->prepared)) return FTMOE_ERR_INVALID_ARG;
  const TcWs L = tc_ws(d, T);
  char* base = static_cast<char*>(ws);
  uint8_t* xq = reinterpret_cast<uint8_t*>(base + L.xq);
  uint8_t* sfa = reinterpret_cast<uint8_t*>(base + L.sfa);
  uint8_t* hq = reinterpret_cast<uint8_t*>(base + L.hq);
  uint8_t* sfh = reinterpret_cast<uint8_t*>(base + L.sfh);
  const int P = T * d->k;
  const int nh = gate_up_nh(d);
  const int sms = num_sms();

  uint8_t* xq_tok = reinterpret_cast<uint8_t*>(base + L.xq_tok);
  uint8_t* sf_tok = reinterpret_cast<uint8_t*>(base + L.sf_tok);
  ftmoe_status s = launch(quantize_act_kernel, dim3(std::min(cdiv(T, kActqWarps), sms * 8)), dim3(kActqWarps * 32), 0,
                          st, x, T, d->d, xq_tok, sf_tok);
  if (s != FTMOE_OK) return s;
  ActqArgs q;
  q.xq_tok = xq_tok;
  q.sf_tok = sf_tok;
  q.T = T;
  q.d = d->d;
  q.k = d->k;
  q.E = d->E;
  q.C = w->C;
  q.P = P;
  q.offsets = off;
  q.sorted_pair = sp;
  q.slot_of = slot_of;
  q.xq = xq;
  q.sfa = sfa;
  q.rows_cap = int(L.rows);
  q.zero_out = reinterpret_cast<float4*>(zero_out);
  q.zero_n4 = zero_out ? (long long)T * d->d / 4 : 0;
  q.topk_w = topk_w;
  q.rowmeta = reinterpret_cast<int4*>(base + L.rowmeta);
  s = launch(actq_gather_kernel, dim3(std::min(cdiv(L.rows, 32 * kActqWarps), sms * 8)),
                          dim3(kActqWarps * 32), 0, st, q);
  if (s != FTMOE_OK) return s;

  CUtensorMap tA1, tG, tU, tA2, tD;
  const size_t C = size_t(w->C);
  if (!make_map(&tA1, xq, d->d / 2, L.rows, kTileM) || !make_map(&tG, w->gate, d->d / 2, C * d->ffn, nh) ||
      !make_map(&tU, w->up, d->d / 2, C * d->ffn, nh) || !make_map(&tA2, hq, d->ffn / 2, L.rows, kTileM) ||
      !make_map(&tD, w->down, d->ffn / 2, C * d->d, 128))
    return FTMOE_ERR_CUDA;

  const uint8_t* prep = static_cast<const uint8_t*>(w->prepared);
  GemmArgs g;
  g.E = d->E;
  g.k = d->k;
  g.d = d->d;
  g.f = d->ffn;
  g.C = w->C;
  g.P = P;
  g.rows_cap = int(L.rows);
  g.offsets = off;
  g.sorted_pair = sp;
  g.slot_of = slot_of;
  g.tscale = w->tensor_scale;
  g.sfa = sfa;
  g.sfb = prep;
  g.hq = hq;
  g.sfh = sfh;
  g.topk_w = nullptr;
  g.out = nullptr;
  const int mts = int(L.rows / kTileM);
  s = nh == 128 ? launch_gemm<0, 128>(tA1, tG, tU, g, mts * (d->ffn / 128), st)
                : launch_gemm<0, 64>(tA1, tG, tU, g, mts * (d->ffn / 64), st);
  if (s != FTMOE_OK) return s;
  g.sfa = sfh;
  g.sfb = prep + align1k(prep_gate_up_bytes(d, w->C));
  g.hq = nullptr;
  g.sfh = nullptr;
  g.topk_w = topk_w;
  g.out = y_or_out;
  g.rowmeta = reinterpret_cast<const int4*>(base + L.rowmeta);
  return launch_gemm<1, 128>(tA2, tD, tD, g, mts * (d->d / 128), st);
}

// ws: buffers at ws + kWsHeader; hdr: the zero header that holds the call's counters.
// out_bf16 (decode kernel only, with topk_w): zero y_or_out first and write its bf16 copy last.
bool ffn_dec_kernel(const ftmoe_layer_desc* d, int T) {
  return ffn_path(d, T) == 0 && (d->fmt == FTMOE_NVFP4 || d->fmt == FTMOE_MXFP4);
}
template <int MODE>
ftmoe_status launch_gemm8(const CUtensorMap& ta, const CUtensorMap& tb0, const CUtensorMap& tb1, const Gemm8Args& g,
                          int max_tiles, cudaStream_t st) {
  const int grid = std::max(1, std::min(num_sms(), max_tiles));
  return launch(gemm8_kernel<MODE>, dim3(grid), dim3(kGemmThreads), size_t(G8Cfg<MODE>::SMEM), st, ta, tb0, tb1, g);
}

// 2D byte matrix [rows][row_bytes], boxes of 128 bytes x box_rows, 128-byte swizzle (box_rows <= 256)
// (make_map above); FP8 path: quantise, gather, gate/up GEMM (SwiGLU + E4M3 h), down GEMM.
ftmoe_status ffn_tc8_impl(const ftmoe_layer_desc* d, const ftmoe_weights* w, const int32_t* slot_of,
                          const uint16_t* x, int T, const int32_t* off, const int32_t* sp, const float* topk_w,
                          float* y_or_out, void* ws, float* zero_out, cudaStream_t st) {
  const Tc8Ws L = tc8_ws(d, T);
  char* base = static_cast<char*>(ws);
  uint8_t* xq_tok = reinterpret_cast<uint8_t*>(base + L.xq_tok);
  float* sx_tok = reinterpret_cast<float*>(base + L.sx_tok);
  uint8_t* xq = reinterpret_cast<uint8_t*>(base + L.xq);
  float* sx = reinterpret_cast<float*>(base + L.sx);
  uint8_t* hq = reinterpret_cast<uint8_t*>(base + L.hq);
  float* sh = reinterpret_cast<float*>(base + L.sh);
  const int P = T * d->k;
  const int sms = num_sms();
  const long long qblocks = (long long)T * (d->d / 128);
  ftmoe_status s = launch(quantize8_kernel, dim3((unsigned)std::min<long long>((qblocks + 7) / 8, sms * 16)), dim3(256),
                          0, st, x, T, d->d, xq_tok, sx_tok);
  if (s != FTMOE_OK) return s;
  Gather8Args q;
  q.xq_tok = xq_tok;
  q.sx_tok = sx_tok;
  q.d = d->d;
  q.k = d->k;
  q.E = d->E;
  q.C = w->C;
  q.P = P;
  q.offsets = off;
  q.sorted_pair = sp;
  q.slot_of = slot_of;
  q.xq = xq;
  q.sx = sx;
  q.rows_cap = int(L.rows);
  q.zero_out = reinterpret_cast<float4*>(zero_out);
  q.zero_n4 = zero_out ? (long long)T * d->d / 4 : 0;
  q.topk_w = topk_w;
  q.rowmeta = reinterpret_cast<int4*>(base + L.rowmeta);
  s = launch(gather8_kernel, dim3(std::min(cdiv(L.rows, kActqWarps), sms * 8)), dim3(kActqWarps * 32), 0, st, q);
  if (s != FTMOE_OK) return s;
  CUtensorMap tA1, tG, tU, tA2, tD;
  const size_t C = size_t(w->C);
  if (!make_map(&tA1, xq, d->d, L.rows, kTileM) || !make_map(&tG, w->gate, d->d, C * d->ffn, 128) ||
      !make_map(&tU, w->up, d->d, C * d->ffn, 128) || !make_map(&tA2, hq, d->ffn, L.rows, kTileM) ||
      !make_map(&tD, w->down, d->ffn, C * d->d, 256))
    return FTMOE_ERR_CUDA;
  Gemm8Args g;
  g.E = d->E;
  g.k = d->k;
  g.d = d->d;
  g.f = d->ffn;
  g.C = w->C;
  g.P = P;
  g.rows_cap = int(L.rows);
  g.offsets = off;
  g.sorted_pair = sp;
  g.slot_of = slot_of;
  g.sx = sx;
  g.sw0 = static_cast<const float*>(w->gate_scale);
  g.sw1 = static_cast<const float*>(w->up_scale);
  g.hq = hq;
  g.sh = sh;
  g.topk_w = nullptr;
  g.out = nullptr;
  const int mts = int(L.rows / kTileM);
  s = launch_gemm8<0>(tA1, tG, tU, g, mts * (d->ffn / 128), st);
  if (s != FTMOE_OK) return s;
  g.sx = sh;
  g.sw0 = static_cast<const float*>(w->down_scale);
  g.sw1 = nullptr;
  g.hq = nullptr;
  g.sh = nullptr;
  g.topk_w = topk_w;
  g.out = y_or_out;
  g.rowmeta = reinterpret_cast<const int4*>(base + L.rowmeta);
  return launch_gemm8<1>(tA2, tD, tD, g, mts * (d->d / 256), st);
}

FfnArgs make_ffn_args(const ftmoe_layer_desc* d, const ftmoe_weights* w, const int32_t* slot_of, const uint16_t* x,
                      int T, const int32_t* off, const int32_t* sp, const float* topk_w, float* y_or_out, void* ws,
                      uint16_t* out_bf16) {
  FfnArgs a;
  a.E = d->E;
  a.k = d->k;
  a.d = d->d;
  a.f = d->ffn;
  a.C = w->C;
  a.gate = static_cast<const uint8_t*>(w->gate);
  a.up = static_cast<const uint8_t*>(w->up);
  a.down = static_cast<const uint8_t*>(w->down);
  a.gate_s = static_cast<const uint8_t*>(w->gate_scale);
  a.up_s = static_cast<const uint8_t*>(w->up_scale);
  a.down_s = static_cast<const uint8_t*>(w->down_scale);
  a.tscale = d->fmt == FTMOE_NVFP4 ? w->tensor_scale : nullptr;
  a.slot_of = slot_of;
  a.x = x;
  a.T = T;
  a.offsets = off;
  a.sorted_pair = sp;
  a.topk_w = topk_w;
  a.y_or_out = y_or_out;
  a.h = reinterpret_cast<float*>(static_cast<char*>(ws) + kWsHeader);
  a.out_bf16 = out_bf16;
  a.prep_dec = (w->prepared && prep_decode_bytes(d, w->C))
                   ? static_cast<const uint8_t*>(w->prepared) + prep_decode_offset(d, w->C)
                   : nullptr;
  return a;
}

ftmoe_status ffn_impl(const ftmoe_layer_desc* d, const ftmoe_weights* w, const int32_t* slot_of, const uint16_t* x,
                      int T, const int32_t* off, const int32_t* sp, const float* topk_w, float* y_or_out, void* ws,
                      void* hdr, cudaStream_t st, uint16_t* out_bf16 = nullptr) {
  const FfnArgs a = make_ffn_args(d, w, slot_of, x, T, off, sp, topk_w, y_or_out, ws, out_bf16);
  const int P = T * d->k;
  if (ffn_path(d, T) == 1) return ffn_tc_impl(d, w, slot_of, x, T, off, sp, topk_w, y_or_out, ws, nullptr, st);
  if (ffn_path(d, T) == 2) return ffn_tc8_impl(d, w, slot_of, x, T, off, sp, topk_w, y_or_out, ws, nullptr, st);
  switch (d->fmt) {
    case FTMOE_BF16: return ffn_stream_launch<FTMOE_BF16>(a, P, st);
    case FTMOE_NVFP4: return ffn_dec_launch<FTMOE_NVFP4>(a, P, hdr, st);
    case FTMOE_MXFP4: return ffn_dec_launch<FTMOE_MXFP4>(a, P, hdr, st);
    case FTMOE_FP8_B128: return ffn_stream_launch<FTMOE_FP8_B128>(a, P, st);
  }
  return FTMOE_ERR_UNSUPPORTED;
}

// C: the arena's slot count when the caller knows it (the layer call), so that a slot_of
// entry the FFN skipped as out of range adds nothing here either; INT32_MAX otherwise.
ftmoe_status combine_impl(const ftmoe_layer_desc* d, int T, const float* y, const int32_t* pp, const float* w,
                          const int32_t* ids, const int32_t* slot_of, const float* pb, float* of, uint16_t* ob,
                          cudaStream_t st, int C = INT32_MAX) {
  CombineArgs a;
  a.T = T;
  a.k = d->k;
  a.d = d->d;
  a.E = d->E;
  a.C = C;
  a.y = y;
  a.pair_pos = pp;
  a.topk_w = w;
  a.topk_ids = ids;
  a.slot_of = slot_of;
  a.partial_b = pb;
  a.out_f32 = of;
  a.out_bf16 = ob;
  const long long n = (long long)T * (d->d / 4);
  return launch(combine_kernel, dim3((unsigned)std::min<long long>(cdiv(n, 256), num_sms() * 8)), dim3(256), 0, st, a);
}

// Device state of an LRU handle for (L, E, C) in one allocation: slot_of [L*E], key, prev and
// next per slot, meta [4], then the totals (int64 [2]).
bool lru_alloc(int L, int E, int C, LruState* st, void** mem) {
  const size_t n_int = size_t(L) * E + 3 * size_t(C) + 4;
  const size_t bytes = align256(n_int * sizeof(int32_t)) + 2 * sizeof(long long);
  void* m = nullptr;
  if (cudaMalloc(&m, bytes) != cudaSuccess) return false;
  int32_t* p = static_cast<int32_t*>(m);
  st->slot_of = p;
  st->key_of = p + size_t(L) * E;
  st->prv = st->key_of + C;
  st->nxt = st->prv + C;
  st->meta = st->nxt + C;
  st->totals = reinterpret_cast<long long*>(static_cast<char*>(m) + align256(n_int * sizeof(int32_t)));
  st->L = L;
  st->E = E;
  st->C = C;
  *mem = m;
  return true;
}

// Per-slot byte ranges of every array of an arena pair (same layer shape, both arenas in
// `fmt`), for slot copies.  The prepared layouts are copied part by part (their part
// offsets depend on each arena's slot count).  Returns the count, or -1 if the prepared
// buffers are not both present or both absent.
// parts: bit 0 = the prefill part of the prepared layout, bit 1 = the decode parts.
int slot_regions(const ftmoe_layer_desc* d, const ftmoe_weights* src, const ftmoe_weights* dst, SlotRegion* r,
                 int parts = 3) {
  int n = 0;
  auto add = [&](const void* s, void* t, size_t ss, size_t ts, size_t bytes) {
    if (!bytes) return;
    SlotRegion& R = r[n++];
    R.src = static_cast<const uint8_t*>(s);
    R.dst = static_cast<uint8_t*>(t);
    R.src_stride = ss;
    R.dst_stride = ts;
    R.bytes = bytes;
    R.vec16 = aligned16(s) && aligned16(t) && ss % 16 == 0 && ts % 16 == 0 && bytes % 16 == 0;
  };
  const size_t nd = size_t(d->ffn) * d->d;   // elements of one matrix
  size_t code = 0, scale = 0;
  switch (d->fmt) {
    case FTMOE_BF16: code = 2 * nd; break;
    case FTMOE_NVFP4: code = nd / 2; scale = nd / 16; break;
    case FTMOE_MXFP4: code = nd / 2; scale = nd / 32; break;
    case FTMOE_FP8_B128: code = nd; scale = (nd / (128 * 128)) * 4; break;
  }
  add(src->gate, const_cast<void*>(dst->gate), code, code, code);
  add(src->up, const_cast<void*>(dst->up), code, code, code);
  add(src->down, const_cast<void*>(dst->down), code, code, code);
  if (scale) {
    add(src->gate_scale, const_cast<void*>(dst->gate_scale), scale, scale, scale);
    add(src->up_scale, const_cast<void*>(dst->up_scale), scale, scale, scale);
    add(src->down_scale, const_cast<void*>(dst->down_scale), scale, scale, scale);
  }
  if (d->fmt == FTMOE_NVFP4) add(src->tensor_scale, const_cast<float*>(dst->tensor_scale), 12, 12, 12);
  const size_t pb = prep_bytes(d, 1);
  if (!pb) return n;
  if ((src->prepared == nullptr) != (dst->prepared == nullptr)) return -1;
  if (!src->prepared) return n;
  const uint8_t* sp = static_cast<const uint8_t*>(src->prepared);
  uint8_t* tp = static_cast<uint8_t*>(const_cast<void*>(dst->prepared));
  const int sC = src->C, tC = dst->C;
  if ((parts & 1) && prep_prefill_bytes(d, 1)) {
    const size_t gu = prep_gate_up_bytes(d, 1), dn = prep_down_bytes(d, 1);
    add(sp, tp, gu, gu, gu);
    add(sp + align1k(prep_gate_up_bytes(d, sC)), tp + align1k(prep_gate_up_bytes(d, tC)), dn, dn, dn);
  }
  if ((parts & 2) && prep_decode_bytes(d, 1)) {
    const size_t db = sd_slot_bytes(d->d, d->ffn, d->fmt);
    add(sp + prep_decode_offset(d, sC), tp + prep_decode_offset(d, tC), db, db, db);
    if (prep_slices_bytes(d, 1)) {
      const size_t sb = sl_slot_bytes(d->d, d->ffn);
      add(sp + prep_slices_offset(d, sC), tp + prep_slices_offset(d, tC), sb, sb, sb);
    }
  }
  return n;
}

}  // namespace

// =============================================================================
extern "C" {

int ftmoe_version(void) { return 100; }

const char* ftmoe_status_string(ftmoe_status s) {
  switch (s) {
    case FTMOE_OK: return "ok";
    case FTMOE_ERR_INVALID_ARG: return "invalid argument";
    case FTMOE_ERR_UNSUPPORTED: return "unsupported";
    case FTMOE_ERR_CUDA: return "CUDA error";
    case FTMOE_ERR_WORKSPACE: return "workspace too small";
    case FTMOE_ERR_TIMEOUT: return "device wait timed out";
    case FTMOE_ERR_DEVICE_CHECK: return "device-side check failed";
  }
  return "unknown status";
}

ftmoe_status ftmoe_set_wait_limit(unsigned long long ns) {
  const unsigned long long v = ns ? ns : kWaitLimitNs;
  return cudaMemcpyToSymbol(g_wait_limit_ns, &v, sizeof(v)) == cudaSuccess ? FTMOE_OK : FTMOE_ERR_CUDA;
}

ftmoe_status ftmoe_get_device_error(int* code, void* stream) {
  if (!code) return FTMOE_ERR_INVALID_ARG;
  cudaStream_t st = as_stream(stream);
  int v = 0;
  if (cudaMemcpyFromSymbolAsync(&v, g_dev_err, sizeof(int), 0, cudaMemcpyDeviceToHost, st) != cudaSuccess)
    return FTMOE_ERR_CUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return FTMOE_ERR_CUDA;
  const int zero = 0;
  if (cudaMemcpyToSymbolAsync(g_dev_err, &zero, sizeof(int), 0, cudaMemcpyHostToDevice, st) != cudaSuccess)
    return FTMOE_ERR_CUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return FTMOE_ERR_CUDA;
  *code = v;
  return FTMOE_OK;
}

size_t ftmoe_route_workspace_size(const ftmoe_layer_desc* d, int T) {
  if (!desc_ok(d) || T < 1) return 0;
  return route_ws(d, T, true);
}

ftmoe_status ftmoe_route(const ftmoe_layer_desc* d, const uint16_t* x, const uint16_t* wr, const float* bias, int T,
                         int32_t* ids, float* w, float* logits, void* ws, size_t ws_bytes, void* stream) {
  if (!desc_ok(d) || T < 1 || T > kMaxT || !x || !wr || !ids || !w || !ws) return FTMOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(wr)) return FTMOE_ERR_INVALID_ARG;
  if (ws_bytes < route_ws(d, T, logits == nullptr)) return FTMOE_ERR_WORKSPACE;
  return route_impl(d, x, wr, bias, T, ids, w, logits, ws, as_stream(stream), nullptr, nullptr, nullptr,
                    logits == nullptr);
}

size_t ftmoe_permute_workspace_size(const ftmoe_layer_desc* d, int T) {
  if (!desc_ok(d) || T < 1) return 0;
  return permute_ws(d, T);
}

ftmoe_status ftmoe_permute(const ftmoe_layer_desc* d, const int32_t* ids, int T, int32_t* off, int32_t* sp,
                           int32_t* pp, void* ws, size_t ws_bytes, void* stream) {
  if (!desc_ok(d) || T < 1 || T > kMaxT || !ids || !off || !sp || !pp || !ws) return FTMOE_ERR_INVALID_ARG;
  if (ws_bytes < permute_ws(d, T)) return FTMOE_ERR_WORKSPACE;
  return permute_impl(d, ids, T, off, sp, pp, ws, as_stream(stream));
}

size_t ftmoe_expert_ffn_workspace_size(const ftmoe_layer_desc* d, int T) {
  if (!desc_ok(d) || T < 1) return 0;
  return ffn_ws(d, T);
}

int ftmoe_expert_ffn_path(const ftmoe_layer_desc* d, int T) {
  if (!desc_ok(d) || T < 1) return -1;
  return ffn_path(d, T);
}

size_t ftmoe_prepare_weights_size(const ftmoe_layer_desc* d, int C) {
  if (!desc_ok(d) || C < 1) return 0;
  return prep_bytes(d, C);
}

ftmoe_status ftmoe_prepare_weights(const ftmoe_layer_desc* d, const ftmoe_weights* w, void* prep, size_t bytes,
                                   void* stream) {
  if (!desc_ok(d) || !weights_ok(d, w)) return FTMOE_ERR_INVALID_ARG;
  const size_t need = prep_bytes(d, w->C);
  if (need == 0) return FTMOE_OK;
  if (!prep || !aligned16(prep)) return FTMOE_ERR_INVALID_ARG;
  if (bytes < need) return FTMOE_ERR_WORKSPACE;
  cudaStream_t st = as_stream(stream);
  uint8_t* out = static_cast<uint8_t*>(prep);
  const int grid = num_sms() * 4;
  ftmoe_status s = FTMOE_OK;
  if (prep_prefill_bytes(d, w->C)) {
    s = launch(prep_sf_gate_up_kernel, dim3(grid), dim3(256), 0, st, static_cast<const uint8_t*>(w->gate_scale),
               static_cast<const uint8_t*>(w->up_scale), w->C, d->d, d->ffn, gate_up_nh(d), out);
    if (s != FTMOE_OK) return s;
    s = launch(prep_sf_down_kernel, dim3(grid), dim3(256), 0, st, static_cast<const uint8_t*>(w->down_scale), w->C,
               d->d, d->ffn, out + align1k(prep_gate_up_bytes(d, w->C)));
    if (s != FTMOE_OK) return s;
  }
  if (prep_decode_bytes(d, w->C)) {
    const uint8_t* g8 = static_cast<const uint8_t*>(w->gate);
    s = launch(prep_decode_kernel, dim3(grid), dim3(256), 0, st, g8, static_cast<const uint8_t*>(w->up),
               static_cast<const uint8_t*>(w->down), static_cast<const uint8_t*>(w->gate_scale),
               static_cast<const uint8_t*>(w->up_scale), static_cast<const uint8_t*>(w->down_scale), w->C, d->d,
               d->ffn, d->fmt, out + prep_decode_offset(d, w->C));
    if (s != FTMOE_OK) return s;
    if (prep_slices_bytes(d, w->C))
      s = launch(prep_slices_kernel, dim3(grid), dim3(256), 0, st, static_cast<const uint8_t*>(w->down),
                 static_cast<const uint8_t*>(w->down_scale), w->C, d->d, d->ffn, d->fmt,
                 out + prep_slices_offset(d, w->C));
  }
  return s;
}

ftmoe_status ftmoe_quantize_act(const ftmoe_layer_desc* d, const uint16_t* x, int T, uint8_t* codes, uint8_t* scales,
                                void* stream) {
  if (!desc_ok(d) || T < 1 || T > kMaxT || !x || !codes || !scales) return FTMOE_ERR_INVALID_ARG;
  if (!aligned16(x) || (reinterpret_cast<uintptr_t>(codes) & 7u)) return FTMOE_ERR_INVALID_ARG;
  if (d->fmt == FTMOE_FP8_B128) {
    if (reinterpret_cast<uintptr_t>(scales) & 3u) return FTMOE_ERR_INVALID_ARG;
    const long long qblocks = (long long)T * (d->d / 128);
    return launch(quantize8_kernel, dim3((unsigned)std::min<long long>((qblocks + 7) / 8, num_sms() * 16)), dim3(256),
                  0, as_stream(stream), x, T, d->d, codes, reinterpret_cast<float*>(scales));
  }
  return launch(quantize_act_kernel, dim3(std::min(cdiv(T, kActqWarps), num_sms() * 8)), dim3(kActqWarps * 32), 0,
                as_stream(stream), x, T, d->d, codes, scales);
}

ftmoe_status ftmoe_expert_ffn(const ftmoe_layer_desc* d, const ftmoe_weights* w, const int32_t* slot_of,
                              const uint16_t* x, int T, const int32_t* off, const int32_t* sp, const float* topk_w,
                              float* y_or_out, void* ws, size_t ws_bytes, void* stream) {
  if (!desc_ok(d) || T < 1 || T > kMaxT || !x || !off || !sp || !y_or_out || !ws) return FTMOE_ERR_INVALID_ARG;
  if (!weights_ok(d, w) || !aligned16(x) || !aligned16(y_or_out)) return FTMOE_ERR_INVALID_ARG;
  if (ffn_path(d, T) == 0 && !path0_size_ok(d, T)) return FTMOE_ERR_UNSUPPORTED;
  if (ws_bytes < ffn_ws(d, T)) return FTMOE_ERR_WORKSPACE;
  return ffn_impl(d, w, slot_of, x, T, off, sp, topk_w, y_or_out, ws, ws, as_stream(stream));
}

ftmoe_status ftmoe_combine(const ftmoe_layer_desc* d, int T, const float* y, const int32_t* pp, const float* w,
                           const int32_t* ids, const int32_t* slot_of, const float* pb, float* of, uint16_t* ob,
                           void* stream) {
  if (!desc_ok(d) || T < 1 || T > kMaxT || (!of && !ob)) return FTMOE_ERR_INVALID_ARG;
  if (y && (!pp || !w)) return FTMOE_ERR_INVALID_ARG;
  if (y && slot_of && !ids) return FTMOE_ERR_INVALID_ARG;
  if ((y && !aligned16(y)) || (pb && !aligned16(pb)) || (of && !aligned16(of))) return FTMOE_ERR_INVALID_ARG;
  if (ob && (reinterpret_cast<uintptr_t>(ob) & 7u)) return FTMOE_ERR_INVALID_ARG;
  return combine_impl(d, T, y, pp, w, ids, slot_of, pb, of, ob, as_stream(stream));
}

// --- LRU ---------------------------------------------------------------------
ftmoe_status ftmoe_lru_create(int L, int E, int C, ftmoe_lru** out) {
  if (!out || L < 1 || E < 1 || C < 1) return FTMOE_ERR_INVALID_ARG;
  if ((long long)L * E > INT32_MAX / 2) return FTMOE_ERR_INVALID_ARG;
  if (lru_smem_bytes(L, E, C) > 200 * 1024) return FTMOE_ERR_UNSUPPORTED;
  ftmoe_lru* h = new (std::nothrow) ftmoe_lru();
  if (!h) return FTMOE_ERR_CUDA;
  if (!lru_alloc(L, E, C, &h->st, &h->mem)) {
    delete h;
    return FTMOE_ERR_CUDA;
  }
  cudaGetDevice(&h->device);
  ftmoe_status s = ftmoe_lru_reset(h, nullptr);
  if (s == FTMOE_OK && cudaStreamSynchronize(nullptr) != cudaSuccess) s = FTMOE_ERR_CUDA;
  if (s != FTMOE_OK) {
    cudaFree(h->mem);
    delete h;
    return s;
  }
  *out = h;
  return FTMOE_OK;
}

ftmoe_status ftmoe_lru_reset(ftmoe_lru* h, void* stream) {
  if (!h) return FTMOE_ERR_INVALID_ARG;
  const int n = std::max(h->st.L * h->st.E, h->st.C);
  return launch(lru_reset_kernel, dim3(std::min(cdiv(n, 256), 64)), dim3(256), 0, as_stream(stream), h->st);
}

ftmoe_status ftmoe_lru_destroy(ftmoe_lru* h) {
  if (!h) return FTMOE_ERR_INVALID_ARG;
  cudaDeviceSynchronize();
  cudaError_t e = cudaFree(h->mem);
  delete h;
  return e == cudaSuccess ? FTMOE_OK : FTMOE_ERR_CUDA;
}

const int32_t* ftmoe_lru_slot_of(const ftmoe_lru* h) { return h ? h->st.slot_of : nullptr; }

ftmoe_status ftmoe_lru_copy_slot_of(const ftmoe_lru* h, int32_t* dst, void* stream) {
  if (!h || !dst) return FTMOE_ERR_INVALID_ARG;
  const size_t n = size_t(h->st.L) * h->st.E * sizeof(int32_t);
  return cudaMemcpyAsync(dst, h->st.slot_of, n, cudaMemcpyDeviceToDevice, as_stream(stream)) == cudaSuccess
             ? FTMOE_OK
             : FTMOE_ERR_CUDA;
}

ftmoe_status ftmoe_slot_lru(ftmoe_lru* h, int layer, const int32_t* ids, int B, int k, uint8_t* hit, int32_t* slot,
                            int32_t* ev, int64_t* counters, void* stream) {
  if (!h || !ids || !hit || !slot || !ev || B < 1 || k < 1) return FTMOE_ERR_INVALID_ARG;
  if ((long long)B * k > INT32_MAX) return FTMOE_ERR_INVALID_ARG;
  if (layer < 0 || layer >= h->st.L) return FTMOE_ERR_INVALID_ARG;
  const long long cap = std::min<long long>((long long)B * k, h->st.E);
  return launch(lru_kernel, dim3(1), dim3(kLruThreads), lru_smem_bytes(h->st.L, h->st.E, h->st.C),
                as_stream(stream), h->st, ids, 1, B * k, layer, 0, hit, slot, ev, cap,
                reinterpret_cast<long long*>(counters));
}

ftmoe_status ftmoe_slot_lru_replay(ftmoe_lru* h, const int32_t* trace, int steps, int B, int k, uint8_t* hit,
                                   int32_t* slot, int32_t* ev, int64_t capacity, int64_t* counters, void* stream) {
  if (!h || !trace || !hit || !slot || !ev || steps < 1 || B < 1 || k < 1 || capacity < 0) return FTMOE_ERR_INVALID_ARG;
  if ((long long)B * k > INT32_MAX || (long long)steps * h->st.L > INT32_MAX) return FTMOE_ERR_INVALID_ARG;
  return launch(lru_kernel, dim3(1), dim3(kLruThreads), lru_smem_bytes(h->st.L, h->st.E, h->st.C),
                as_stream(stream), h->st, trace, steps * h->st.L, B * k, 0, 1, hit, slot, ev, (long long)capacity,
                reinterpret_cast<long long*>(counters));
}

// --- expert cache: elastic resize, slot copies, the q* split ---------------------
int ftmoe_lru_capacity(const ftmoe_lru* h) { return h ? h->st.C : -1; }

ftmoe_status ftmoe_lru_resize(ftmoe_lru* h, int C_new, int32_t* moves, int32_t* n_moves, void* stream) {
  if (!h || C_new < 1) return FTMOE_ERR_INVALID_ARG;
  if (lru_smem_bytes(h->st.L, h->st.E, C_new) > 200 * 1024) return FTMOE_ERR_UNSUPPORTED;
  LruState nw;
  void* mem = nullptr;
  if (!lru_alloc(h->st.L, h->st.E, C_new, &nw, &mem)) return FTMOE_ERR_CUDA;
  int32_t* scratch = nullptr;
  if (cudaMalloc(&scratch, size_t(h->st.C) * sizeof(int32_t)) != cudaSuccess) {
    cudaFree(mem);
    return FTMOE_ERR_CUDA;
  }
  cudaStream_t st = as_stream(stream);
  ftmoe_status s = launch(lru_resize_kernel, dim3(1), dim3(32), 0, st, h->st, nw, scratch, moves, n_moves);
  if (s == FTMOE_OK && cudaStreamSynchronize(st) != cudaSuccess) s = FTMOE_ERR_CUDA;
  cudaFree(scratch);
  if (s != FTMOE_OK) {   // the old state stays in use
    cudaFree(mem);
    return s;
  }
  cudaFree(h->mem);
  h->mem = mem;
  h->st = nw;
  return FTMOE_OK;
}

ftmoe_status ftmoe_copy_slots(const ftmoe_layer_desc* d, const ftmoe_weights* src, const ftmoe_weights* dst,
                              const int32_t* pairs, const int32_t* n_pairs, int max_pairs, void* stream) {
  if (!desc_ok(d) || !weights_ok(d, src) || !weights_ok(d, dst) || max_pairs < 0) return FTMOE_ERR_INVALID_ARG;
  if (max_pairs > 0 && !pairs) return FTMOE_ERR_INVALID_ARG;
  if (max_pairs == 0) return FTMOE_OK;
  SlotCopyArgs a;
  memset(&a, 0, sizeof(a));
  a.nr = slot_regions(d, src, dst, a.r);
  if (a.nr < 0) return FTMOE_ERR_INVALID_ARG;
  a.pairs = pairs;
  a.n_dev = n_pairs;
  a.n_max = max_pairs;
  a.src_C = src->C;
  a.dst_C = dst->C;
  a.same = src->gate == dst->gate;
  unsigned long long big = 16;
  for (int i = 0; i < a.nr; ++i) big = std::max(big, a.r[i].bytes);
  const int gx = std::max(1, std::min(128, cdiv((long long)(big / 16), 1024)));
  const int gy = std::max(1, std::min(max_pairs, std::max(1, num_sms() * 16 / gx)));
  return launch(copy_slots_kernel, dim3(gx, std::min(gy, 65535)), dim3(256), 0, as_stream(stream), a);
}

double ftmoe_qstar(int m, double link_gbs, double host_gbs) {
  if (m < 0 || !(link_gbs > 0.0) || !(host_gbs > 0.0) || link_gbs > 1e300 || host_gbs > 1e300) return -1.0;
  return double(m) * link_gbs / host_gbs;
}

int ftmoe_qstar_fill_count(int m, double link_gbs, double host_gbs) {
  const double q = ftmoe_qstar(m, link_gbs, host_gbs);
  if (q < 0.0) return -1;
  const double n = floor(q + 0.5);
  return n < 0.0 ? 0 : (n > double(m) ? m : int(n));
}

ftmoe_status ftmoe_miss_split(const ftmoe_lru* h, int layer, const int32_t* ids, int B, int k, const uint8_t* hit,
                              double link_gbs, double host_gbs, int fill_override, int32_t* slot_of_a,
                              int32_t* slot_of_b, int32_t* fill_now, int32_t* fill_later, int32_t* counts,
                              void* stream) {
  if (!h || !ids || !hit || !slot_of_a || !slot_of_b || !fill_now || !fill_later || !counts) return FTMOE_ERR_INVALID_ARG;
  if (B < 1 || k < 1 || (long long)B * k > INT32_MAX || layer < 0 || layer >= h->st.L) return FTMOE_ERR_INVALID_ARG;
  if (fill_override < 0 && ftmoe_qstar(0, link_gbs, host_gbs) < 0.0) return FTMOE_ERR_INVALID_ARG;
  if (h->st.E > 1024) return FTMOE_ERR_UNSUPPORTED;
  SplitArgs a;
  a.slot_of = h->st.slot_of;
  a.ids = ids;
  a.Bk = B * k;
  a.E = h->st.E;
  a.layer = layer;
  a.hit = hit;
  a.link = link_gbs;
  a.host = host_gbs;
  a.fill_override = fill_override;
  a.slot_of_a = slot_of_a;
  a.slot_of_b = slot_of_b;
  a.fill_now = fill_now;
  a.fill_later = fill_later;
  a.counts = counts;
  return launch(miss_split_kernel, dim3(1), dim3(256), 0, as_stream(stream), a);
}

// --- whole layer -------------------------------------------------------------
// Workspace: header | ids | w | offsets | sorted_pair | pair_pos | y | (route/permute/ffn scratch, shared)
}  // extern "C"

namespace {
// Fused decode layer (router, expert FFN and merge in one kernel): few tokens, a 4-bit
// format with the prepared decode layout.  Its scratch: h (f16) | logits | ready | merge.
struct FusedWs {
  size_t h, logits, ready, merge, part, total;
};
FusedWs fused_ws(const ftmoe_layer_desc* d, int T) {
  FusedWs F;
  const size_t P = size_t(T) * d->k;
  size_t o = 0;
  F.h = o; o += align256(P * d->ffn * 2);
  F.logits = o; o += align256(size_t(T) * d->E * 4);
  F.ready = o; o += align256(size_t(d->E) * 4);
  F.merge = o; o += align256(size_t(T) * (d->d / 32) * 4);
  F.part = o;                                                     // slice form: each CTA's partial output
  if (sl_wanted(d->d, d->fmt)) o += align256(size_t(num_sms()) * T * d->d * 4);
  F.total = o;
  return F;
}
bool layer_fused_ok(const ftmoe_layer_desc* d, const ftmoe_weights* w, int T) {
  if (ffn_path(d, T) != 0 || !w->prepared || !prep_decode_bytes(d, w->C)) return false;
  return sd_route_supported(d->E, d->d, d->ffn, d->fmt, T, d->k, num_sms(), max_smem_optin());
}
// the one-token slice form (down projection per gate/up item, no down phase)
bool layer_slice_ok(const ftmoe_layer_desc* d, const ftmoe_weights* w, int T) {
  if (T < 1 || T > kSdRouteMaxT || ffn_path(d, T) != 0 || !w->prepared || !prep_slices_bytes(d, w->C)) return false;
  // more than one token: NVFP4 only (the MXFP4 instance with two token columns runs out of registers)
  if (T > 1 && d->fmt != FTMOE_NVFP4) return false;
  return sl_supported(d->E, d->d, d->ffn, d->fmt, T, d->k, num_sms(), max_smem_optin());
}
// Cluster form of the slice kernel: among cluster sizes 8, 4 and 2 whose CTAs each hold their
// share of the router rows in the ring, the one that places the most CTAs on the GPU (as many
// clusters as fit, one CTA per SM; on a tie the larger cluster).  More CTAs means fewer items
// per CTA, and an item beyond the ring's stages would wait for a stage to free.  {0, 0}: the
// grid form.  Cached per shape.
struct SlClusterPlan {
  int cs, grid;
};
template <int FMT, int NCOL>
SlClusterPlan sl_cluster_plan(const FfnArgs& a, const SlLayout& Ls) {
  static std::mutex mu;
  static std::map<std::array<int, 5>, SlClusterPlan> cache;
  int dev = 0;
  cudaGetDevice(&dev);
  const std::array<int, 5> key{dev, a.E, a.d, a.T, Ls.smem};
  std::lock_guard<std::mutex> lock(mu);
  auto it = cache.find(key);
  if (it != cache.end()) return it->second;
  SlClusterPlan plan{0, 0};
  auto kern = sl_layer_kernel<FMT, NCOL, true>;
  // Each CTA streams the router rows of E / cs experts before the selection (measured on
  // B300: ~2.9 us for 128 KB per SM), and the FFN items spread over the grid (~1.5 us per
  // item of a d 2048, ffn 768 NVFP4 expert).  The plan takes the cluster size with the least
  // estimated time of the two; 16 needs the non-portable cluster attribute.
  const double us_per_row_byte = 2.9 / (128.0 * 1024.0), us_per_item = 1.5;
  const long long items = (long long)std::min(a.E, a.T * a.k) * (a.f / kSdRowsA);
  double best = 1e30;
  if (resident_ctas(kern, kSdThreads, size_t(Ls.smem)) >= 1 &&
      cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) == cudaSuccess) {
    for (int cs : {16, 8, 4, 2}) {
      const long long epc = (a.E + cs - 1) / cs;
      // the ring holds this CTA's router rows, and at the end its partial output [T][d] (fp32)
      if (epc * a.d * 2 > (long long)Ls.stages * Ls.stage_bytes || num_sms() < cs) continue;
      if ((long long)a.T * a.d * 4 > (long long)Ls.stages * Ls.stage_bytes) continue;
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3(num_sms() / cs * cs);
      cfg.blockDim = dim3(kSdThreads);
      cfg.dynamicSmemBytes = size_t(Ls.smem);
      cudaLaunchAttribute at[1];
      at[0].id = cudaLaunchAttributeClusterDimension;
      at[0].val.clusterDim.x = unsigned(cs);
      at[0].val.clusterDim.y = 1;
      at[0].val.clusterDim.z = 1;
      cfg.attrs = at;
      cfg.numAttrs = 1;
      int n = 0;
      if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) {
        (void)cudaGetLastError();
        continue;
      }
      const int grid = std::min(n, num_sms() / cs) * cs;
      if (n < 1) continue;
      const double est = double(epc) * a.d * 2 * us_per_row_byte + double((items + grid - 1) / grid) * us_per_item;
      if (est < best) {
        best = est;
        plan = SlClusterPlan{cs, grid};
      }
    }
  }
  (void)cudaGetLastError();
  cache[key] = plan;
  return plan;
}

template <int FMT, int NCOL>
ftmoe_status layer_slice_launch(const FfnArgs& a, const SdRoute& r, void* hdr, const uint8_t* slices,
                                cudaStream_t st) {
  const SlLayout Ls = sl_layout(a.E, a.d, FMT, a.T, a.k, max_smem_optin());
  unsigned long long* gs = reinterpret_cast<unsigned long long*>(static_cast<char*>(hdr) + kWsGridSync);
  unsigned* ccnt = reinterpret_cast<unsigned*>(static_cast<char*>(hdr) + kWsClusterCnt);
  const SlClusterPlan plan = sl_cluster_plan<FMT, NCOL>(a, Ls);
  if (plan.cs > 0) {
    // the function's dynamic shared-memory bound is per function, and launches of other
    // shapes may have lowered it since the plan was made
    if (cudaFuncSetAttribute(sl_layer_kernel<FMT, NCOL, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             Ls.smem) != cudaSuccess)
      return FTMOE_ERR_CUDA;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(plan.grid);
    cfg.blockDim = dim3(kSdThreads);
    cfg.dynamicSmemBytes = size_t(Ls.smem);
    cfg.stream = st;
    cudaLaunchAttribute at[2];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = unsigned(plan.cs);
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    at[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, sl_layer_kernel<FMT, NCOL, true>, a, Ls, r, gs, slices, ccnt) == cudaSuccess
               ? FTMOE_OK
               : FTMOE_ERR_CUDA;
  }
  if (resident_ctas(sl_layer_kernel<FMT, NCOL, false>, kSdThreads, size_t(Ls.smem)) < 1) return FTMOE_ERR_CUDA;
  return launch(sl_layer_kernel<FMT, NCOL, false>, dim3(num_sms()), dim3(kSdThreads), size_t(Ls.smem), st, a, Ls, r,
                gs, slices, ccnt);
}
template <int FMT>
ftmoe_status layer_fused_launch(const FfnArgs& a, const SdRoute& r, void* hdr, cudaStream_t st) {
  const SdLayout Ls = sd_layout(a.E, a.d, a.f, FMT, a.T, a.k, true, max_smem_optin());
  if (resident_ctas(sd_ffn_kernel<FMT, true>, kSdThreads, size_t(Ls.smem)) < 1) return FTMOE_ERR_CUDA;
  unsigned long long* gs = reinterpret_cast<unsigned long long*>(static_cast<char*>(hdr) + kWsGridSync);
  return launch(sd_ffn_kernel<FMT, true>, dim3(num_sms()), dim3(kSdThreads), size_t(Ls.smem), st, a, Ls, r, gs);
}

struct LayerWs {
  size_t ids, w, off, sp, pp, y, scratch, total;
};
LayerWs layer_ws(const ftmoe_layer_desc* d, int T) {
  LayerWs L;
  const size_t P = size_t(T) * d->k;
  size_t o = kWsHeader;
  L.ids = o; o += align256(P * 4);
  L.w = o; o += align256(P * 4);
  L.off = o; o += align256(size_t(d->E + 1) * 4);
  L.sp = o; o += align256(P * 4);
  L.pp = o; o += align256(P * 4);
  L.y = o;
  if (ffn_path(d, T) == 0) o += align256(P * d->d * sizeof(float));
  L.scratch = o;
  // scratch regions reuse the same bytes after the header, so offset them by the header size
  const size_t sr = route_ws(d, T, true) - kWsHeader;
  const size_t sq = permute_ws(d, T) - kWsHeader;
  const size_t sf = ffn_ws(d, T) - kWsHeader;
  // the one-kernel forms' scratch only where one of them can run (few tokens, 4-bit weights)
  const bool fusable = T <= kSdRouteMaxT && ffn_path(d, T) == 0 && (d->fmt == FTMOE_NVFP4 || d->fmt == FTMOE_MXFP4);
  o += std::max(std::max(sr, sq), std::max(sf, fusable ? fused_ws(d, T).total : size_t(0)));
  L.total = o;
  return L;
}
}  // namespace

extern "C" {

size_t ftmoe_layer_workspace_size(const ftmoe_layer_desc* d, int T) {
  if (!desc_ok(d) || T < 1) return 0;
  return layer_ws(d, T).total;
}

int ftmoe_layer_path(const ftmoe_layer_desc* d, const ftmoe_weights* w, int T) {
  if (!desc_ok(d) || T < 1 || T > kMaxT || !weights_ok(d, w)) return -1;
  if (!layer_fused_ok(d, w, T)) return 0;
  return layer_slice_ok(d, w, T) ? 2 : 1;
}

ftmoe_status ftmoe_layer_forward(const ftmoe_layer_desc* d, const ftmoe_weights* w, const int32_t* slot_of,
                                 const uint16_t* x, const uint16_t* wr, const float* bias, int T, int32_t* ids,
                                 float* tw, float* out_f32, uint16_t* out_bf16, void* ws, size_t ws_bytes,
                                 void* stream) {
  if (!desc_ok(d) || T < 1 || T > kMaxT || !x || !wr || !out_f32 || !ws) return FTMOE_ERR_INVALID_ARG;
  if ((ids == nullptr) != (tw == nullptr)) return FTMOE_ERR_INVALID_ARG;
  if (!weights_ok(d, w) || !aligned16(x) || !aligned16(wr) || !aligned16(out_f32)) return FTMOE_ERR_INVALID_ARG;
  if (out_bf16 && (reinterpret_cast<uintptr_t>(out_bf16) & 7u)) return FTMOE_ERR_INVALID_ARG;
  if (ffn_path(d, T) == 0 && !path0_size_ok(d, T)) return FTMOE_ERR_UNSUPPORTED;
  const LayerWs L = layer_ws(d, T);
  if (ws_bytes < L.total) return FTMOE_ERR_WORKSPACE;
  char* base = static_cast<char*>(ws);
  cudaStream_t st = as_stream(stream);
  int32_t* ids_ = ids ? ids : reinterpret_cast<int32_t*>(base + L.ids);
  float* w_ = tw ? tw : reinterpret_cast<float*>(base + L.w);
  int32_t* off = reinterpret_cast<int32_t*>(base + L.off);
  int32_t* sp = reinterpret_cast<int32_t*>(base + L.sp);
  int32_t* pp = reinterpret_cast<int32_t*>(base + L.pp);
  float* y = reinterpret_cast<float*>(base + L.y);
  // The steps run in order on one stream, so they share one scratch region:
  // router logits, then the permutation histogram, then h.  Counters stay in
  // the caller's zero header at `base`.  The FFN addresses its buffer at
  // ws + kWsHeader, so it gets a view that ends its header where scratch starts.
  char* view = base + L.scratch - kWsHeader;
  ftmoe_status s;
  if (layer_fused_ok(d, w, T)) {
    // one kernel: router + sort + expert FFN + merge
    const FusedWs F = fused_ws(d, T);
    char* sc = base + L.scratch;
    FfnArgs a = make_ffn_args(d, w, slot_of, x, T, nullptr, nullptr, nullptr, out_f32, view, nullptr);
    a.h = reinterpret_cast<float*>(sc + F.h);
    SdRoute r;
    r.wr = wr;
    r.bias = bias;
    r.renorm = d->renorm;
    r.logits = reinterpret_cast<float*>(sc + F.logits);
    r.ids = ids_;
    r.tw = w_;
    r.ready = reinterpret_cast<unsigned*>(sc + F.ready);
    r.merge = reinterpret_cast<unsigned*>(sc + F.merge);
    r.ybuf = y;
    r.out_f32 = out_f32;
    r.out_bf16 = out_bf16;
    r.part = reinterpret_cast<float*>(sc + F.part);
    if (layer_slice_ok(d, w, T)) {
      const uint8_t* slices = static_cast<const uint8_t*>(w->prepared) + prep_slices_offset(d, w->C);
      if (T > 1) return layer_slice_launch<FTMOE_NVFP4, 2>(a, r, base, slices, st);   // NVFP4 only (layer_slice_ok)
      return d->fmt == FTMOE_NVFP4 ? layer_slice_launch<FTMOE_NVFP4, 1>(a, r, base, slices, st)
                                   : layer_slice_launch<FTMOE_MXFP4, 1>(a, r, base, slices, st);
    }
    return d->fmt == FTMOE_NVFP4 ? layer_fused_launch<FTMOE_NVFP4>(a, r, base, st)
                                 : layer_fused_launch<FTMOE_MXFP4>(a, r, base, st);
  }
  // route: logits go to the scratch region (the view's buffer area)
  s = route_impl(d, x, wr, bias, T, ids_, w_, reinterpret_cast<float*>(base + L.scratch), base, st, off, sp, pp, true);
  if (s != FTMOE_OK) return s;
  // permute: fused into the router for small batches; else its histogram lives in the scratch region too
  if (!route_can_permute(d, T)) {
    const int P = T * d->k;
    const int nch = cdiv(P, kPermChunk);
    if (nch == 1) {
      s = launch(permute_rank_kernel, dim3(1), dim3(kPermChunk), permute_rank_smem(d->E), st, (const int32_t*)ids_, P,
                 d->E, (const int32_t*)nullptr, 1, off, sp, pp);
    } else {
      int32_t* hist = reinterpret_cast<int32_t*>(base + L.scratch);
      s = launch(permute_hist_kernel, dim3(nch), dim3(kPermChunk), size_t(d->E) * sizeof(int), st,
                 (const int32_t*)ids_, P, d->E, hist);
      if (s == FTMOE_OK)
        s = launch(permute_rank_kernel, dim3(nch), dim3(kPermChunk), permute_rank_smem(d->E), st,
                   (const int32_t*)ids_, P, d->E, (const int32_t*)hist, nch, off, sp, pp);
    }
  }
  if (s != FTMOE_OK) return s;
  if (ffn_path(d, T) != 0) {
    // tensor-core path: out_f32 is zeroed by the gather kernel and the down GEMM adds w * y into it
    s = ffn_path(d, T) == 1 ? ffn_tc_impl(d, w, slot_of, x, T, off, sp, w_, out_f32, view, out_f32, st)
                            : ffn_tc8_impl(d, w, slot_of, x, T, off, sp, w_, out_f32, view, out_f32, st);
    if (s != FTMOE_OK || !out_bf16) return s;
    return combine_impl(d, T, nullptr, pp, w_, ids_, slot_of, out_f32, out_f32, out_bf16, st, w->C);
  }
  if (ffn_dec_kernel(d, T) && out_bf16) {
    // decode kernel: fused combine into out_f32, which it zeroes first and casts to bf16 last
    return ffn_impl(d, w, slot_of, x, T, off, sp, w_, out_f32, view, base, st, out_bf16);
  }
  s = ffn_impl(d, w, slot_of, x, T, off, sp, nullptr, y, view, base, st);
  if (s != FTMOE_OK) return s;
  return combine_impl(d, T, y, pp, w_, ids_, slot_of, nullptr, out_f32, out_bf16, st, w->C);
}

}  // extern "C"

// =============================================================================
// ftmoe_layer_forward_host: staging of x and of the bf16 output in the workspace, after the
// layer call's own bytes.
// =============================================================================
extern "C" size_t ftmoe_layer_host_workspace_size(const ftmoe_layer_desc* d, int T) {
  if (!desc_ok(d) || T < 1 || T > kMaxT) return 0;
  return align256(layer_ws(d, T).total) + 2 * align256(size_t(T) * d->d * 2);
}

extern "C" ftmoe_status ftmoe_layer_forward_host(const ftmoe_layer_desc* d, const ftmoe_weights* w,
                                                 const int32_t* slot_of, const uint16_t* x_host, const uint16_t* wr,
                                                 const float* bias, int T, int32_t* ids, float* tw, float* out_f32,
                                                 uint16_t* out_host, void* ws, size_t ws_bytes, void* stream) {
  if (!desc_ok(d) || T < 1 || T > kMaxT || !x_host || !out_host || !ws) return FTMOE_ERR_INVALID_ARG;
  const size_t need = ftmoe_layer_host_workspace_size(d, T);
  if (ws_bytes < need) return FTMOE_ERR_WORKSPACE;
  const size_t base = align256(layer_ws(d, T).total), xb = size_t(T) * d->d * 2;
  char* p = static_cast<char*>(ws);
  uint16_t* x_dev = reinterpret_cast<uint16_t*>(p + base);
  uint16_t* o_dev = reinterpret_cast<uint16_t*>(p + base + align256(xb));
  cudaStream_t st = as_stream(stream);
  if (cudaMemcpyAsync(x_dev, x_host, xb, cudaMemcpyHostToDevice, st) != cudaSuccess) return FTMOE_ERR_CUDA;
  const ftmoe_status s =
      ftmoe_layer_forward(d, w, slot_of, x_dev, wr, bias, T, ids, tw, out_f32, o_dev, ws, base, stream);
  if (s != FTMOE_OK) return s;
  return cudaMemcpyAsync(out_host, o_dev, xb, cudaMemcpyDeviceToHost, st) == cudaSuccess ? FTMOE_OK : FTMOE_ERR_CUDA;
}

// =============================================================================
// ftmoe_layer_graph: one host-buffer layer call captured from `stream` and instantiated.
// =============================================================================
struct ftmoe_layer_graph {
  cudaGraphExec_t exec;
};

extern "C" ftmoe_status ftmoe_layer_graph_create(const ftmoe_layer_desc* d, const ftmoe_weights* w,
                                                 const int32_t* slot_of, const uint16_t* x_host, const uint16_t* wr,
                                                 const float* bias, int T, int32_t* ids, float* tw, float* out_f32,
                                                 uint16_t* out_host, void* ws, size_t ws_bytes, void* stream,
                                                 ftmoe_layer_graph** out) {
  if (!out) return FTMOE_ERR_INVALID_ARG;
  *out = nullptr;
  if (!stream) return FTMOE_ERR_INVALID_ARG;
  // the host checks of the call itself, before any CUDA call
  if (!desc_ok(d) || T < 1 || T > kMaxT || !x_host || !out_host || !ws || !wr || !out_f32) return FTMOE_ERR_INVALID_ARG;
  if ((ids == nullptr) != (tw == nullptr) || !weights_ok(d, w)) return FTMOE_ERR_INVALID_ARG;
  if (ws_bytes < ftmoe_layer_host_workspace_size(d, T)) return FTMOE_ERR_WORKSPACE;
  cudaStream_t st = as_stream(stream);
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(st, &cap) != cudaSuccess) return FTMOE_ERR_CUDA;
  if (cap != cudaStreamCaptureStatusNone) return FTMOE_ERR_INVALID_ARG;
  if (cudaStreamBeginCapture(st, cudaStreamCaptureModeThreadLocal) != cudaSuccess) return FTMOE_ERR_CUDA;
  const ftmoe_status s =
      ftmoe_layer_forward_host(d, w, slot_of, x_host, wr, bias, T, ids, tw, out_f32, out_host, ws, ws_bytes, stream);
  cudaGraph_t g = nullptr;
  const cudaError_t e = cudaStreamEndCapture(st, &g);   // always: the stream leaves capture mode
  if (s != FTMOE_OK || e != cudaSuccess || !g) {
    if (g) cudaGraphDestroy(g);
    (void)cudaGetLastError();
    return s != FTMOE_OK ? s : FTMOE_ERR_CUDA;
  }
  cudaGraphExec_t x = nullptr;
  const cudaError_t ie = cudaGraphInstantiate(&x, g, 0);
  cudaGraphDestroy(g);
  if (ie != cudaSuccess || !x) {
    (void)cudaGetLastError();
    return FTMOE_ERR_CUDA;
  }
  ftmoe_layer_graph* h = new (std::nothrow) ftmoe_layer_graph{x};
  if (!h) {
    cudaGraphExecDestroy(x);
    return FTMOE_ERR_CUDA;
  }
  *out = h;
  return FTMOE_OK;
}

extern "C" ftmoe_status ftmoe_layer_graph_launch(ftmoe_layer_graph* h, void* stream) {
  if (!h) return FTMOE_ERR_INVALID_ARG;
  return cudaGraphLaunch(h->exec, as_stream(stream)) == cudaSuccess ? FTMOE_OK : FTMOE_ERR_CUDA;
}

extern "C" ftmoe_status ftmoe_layer_graph_destroy(ftmoe_layer_graph* h) {
  if (!h) return FTMOE_OK;
  const cudaError_t e = cudaGraphExecDestroy(h->exec);
  delete h;
  return e == cudaSuccess ? FTMOE_OK : FTMOE_ERR_CUDA;
}

// =============================================================================
// ftmoe_layers_streamed: L layers whose experts stream from a host pool through one or two
// device arenas; with two, layer l+1's experts are copied while layer l computes.
// =============================================================================
extern "C" ftmoe_status ftmoe_layers_streamed(const ftmoe_layer_desc* d, int L, const ftmoe_weights* pool,
                                              const ftmoe_weights* arenas, int n_arenas, const uint16_t* const* x,
                                              const uint16_t* const* wr, const float* const* bias, int T,
                                              float* const* out_f32, uint16_t* const* out_bf16, void* ws,
                                              size_t ws_bytes, void* compute_stream, void* copy_stream) {
  if (!desc_ok(d) || L < 1 || T < 1 || T > kMaxT || !pool || !arenas || n_arenas < 1 || n_arenas > 2)
    return FTMOE_ERR_INVALID_ARG;
  if (!x || !wr || !out_f32 || !ws || !x[0]) return FTMOE_ERR_INVALID_ARG;
  if (!weights_ok(d, pool) || (long long)pool->C < (long long)L * d->E) return FTMOE_ERR_INVALID_ARG;
  for (int b = 0; b < n_arenas; ++b)
    if (!weights_ok(d, &arenas[b]) || arenas[b].C < d->E) return FTMOE_ERR_INVALID_ARG;
  for (int l = 0; l < L; ++l) {
    if (!wr[l] || !out_f32[l]) return FTMOE_ERR_INVALID_ARG;
    if (!x[l] && (l == 0 || !out_bf16 || !out_bf16[l - 1])) return FTMOE_ERR_INVALID_ARG;
  }
  if (ws_bytes < layer_ws(d, T).total) return FTMOE_ERR_WORKSPACE;
  // what the call's path reads: the canonical arrays, plus the prefill part (tensor-core NVFP4
  // path) or the decode parts (decode path) of the prepared layout
  const int parts = ffn_path(d, T) == 1 ? 1 : (ffn_path(d, T) == 0 ? 2 : 0);
  SlotRegion reg[kMaxSlotRegions];
  const int nr = slot_regions(d, pool, &arenas[0], reg, parts);
  if (nr < 0) return FTMOE_ERR_INVALID_ARG;
  for (int b = 1; b < n_arenas; ++b) {
    SlotRegion other[kMaxSlotRegions];
    if (slot_regions(d, pool, &arenas[b], other, parts) != nr) return FTMOE_ERR_INVALID_ARG;
  }
  cudaStream_t cs = as_stream(compute_stream), ps = as_stream(copy_stream);
  cudaEvent_t filled[2] = {nullptr, nullptr}, done[2] = {nullptr, nullptr};
  ftmoe_status s = FTMOE_OK;
  for (int b = 0; b < n_arenas && s == FTMOE_OK; ++b)
    if (cudaEventCreateWithFlags(&filled[b], cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&done[b], cudaEventDisableTiming) != cudaSuccess)
      s = FTMOE_ERR_CUDA;
  // the copy stream starts after whatever the compute stream has queued (the arenas may be in use)
  if (s == FTMOE_OK && (cudaEventRecord(done[0], cs) != cudaSuccess || cudaStreamWaitEvent(ps, done[0], 0) != cudaSuccess))
    s = FTMOE_ERR_CUDA;
  const size_t E = size_t(d->E);
  for (int l = 0; l < L && s == FTMOE_OK; ++l) {
    const int b = l % n_arenas;
    const ftmoe_weights* A = &arenas[b];
    SlotRegion rb[kMaxSlotRegions];
    slot_regions(d, pool, A, rb, parts);
    if (l >= n_arenas && cudaStreamWaitEvent(ps, done[b], 0) != cudaSuccess) {
      s = FTMOE_ERR_CUDA;
      break;
    }
    // layer l's experts are slots l*E .. l*E + E - 1 of the pool: one contiguous range per array
    for (int i = 0; i < nr && s == FTMOE_OK; ++i)
      if (cudaMemcpyAsync(rb[i].dst, rb[i].src + size_t(l) * E * rb[i].src_stride, E * rb[i].bytes,
                          cudaMemcpyDefault, ps) != cudaSuccess)
        s = FTMOE_ERR_CUDA;
    if (s != FTMOE_OK || cudaEventRecord(filled[b], ps) != cudaSuccess || cudaStreamWaitEvent(cs, filled[b], 0) != cudaSuccess) {
      s = FTMOE_ERR_CUDA;
      break;
    }
    const uint16_t* xl = x[l] ? x[l] : out_bf16[l - 1];
    s = ftmoe_layer_forward(d, A, nullptr, xl, wr[l], bias ? bias[l] : nullptr, T, nullptr, nullptr, out_f32[l],
                            out_bf16 ? out_bf16[l] : nullptr, ws, ws_bytes, compute_stream);
    if (s == FTMOE_OK && cudaEventRecord(done[b], cs) != cudaSuccess) s = FTMOE_ERR_CUDA;
  }
  for (int b = 0; b < 2; ++b) {   // destroyed once their pending work completes
    if (filled[b]) cudaEventDestroy(filled[b]);
    if (done[b]) cudaEventDestroy(done[b]);
  }
  return s;
}

// =============================================================================
// ftmoe_route_noalloc: the router for callers that cannot allocate device memory.
//
// Its scratch (the completion counter and the [T][E] fp32 logits) lives in one
// fixed array that every GPU loading this library holds until the process
// exits.  Host code must not hand the array's name to a kernel: on the host it
// is only a stand-in symbol.  The device address comes from
// cudaGetSymbolAddress, taken once per device (with that device current) on
// the first call there.  Every call shares the array, so calls that overlap on
// the GPU race; each call zeroes the counter before its kernels run.
// =============================================================================
static __device__ __align__(256) unsigned char g_route_noalloc_scratch[FTMOE_WS_ZERO_BYTES +
                                                                       FTMOE_NOALLOC_MAX_LOGITS * sizeof(float)];

namespace {
std::mutex g_noalloc_mu;
void* g_noalloc_ptr[kMaxDevices];
unsigned long long g_noalloc_ctx[kMaxDevices];   // the context the address was taken in

typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long*);

// Unique id of the current context (0 if the driver cannot tell).  A device reset ends the
// context and reloads this library's module in the next one, at a possibly different address.
unsigned long long current_ctx_id() {
  static CtxGetCurrentFn get_cur = nullptr;
  static CtxGetIdFn get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_cur = reinterpret_cast<CtxGetCurrentFn>(p);
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<CtxGetIdFn>(p);
  });
  CUcontext c = nullptr;
  unsigned long long id = 0;
  if (!get_cur || !get_id || get_cur(&c) != CUDA_SUCCESS || !c || get_id(c, &id) != CUDA_SUCCESS) return 0;
  return id;
}

// Device address of the fixed scratch array on the current device: looked up on the first call
// in each context of a device (after a device reset, again), then reused.  While no context is
// current yet (id 0) it is looked up on every call; the lookup makes the context current.
ftmoe_status noalloc_scratch(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return FTMOE_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return FTMOE_ERR_UNSUPPORTED;
  const unsigned long long ctx = current_ctx_id();
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (!g_noalloc_ptr[dev] || ctx == 0 || g_noalloc_ctx[dev] != ctx) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_route_noalloc_scratch) != cudaSuccess || !p) return FTMOE_ERR_CUDA;
    g_noalloc_ptr[dev] = p;
    g_noalloc_ctx[dev] = ctx;
  }
  *out = g_noalloc_ptr[dev];
  return FTMOE_OK;
}
}  // namespace

extern "C" ftmoe_status ftmoe_route_noalloc(const ftmoe_layer_desc* d, const uint16_t* x, const uint16_t* wr,
                                            const float* bias, int T, int32_t* ids, float* w, void* stream) {
  if (!desc_ok(d) || T < 1 || T > kMaxT || !x || !wr || !ids || !w) return FTMOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(wr)) return FTMOE_ERR_INVALID_ARG;
  if (size_t(T) * size_t(d->E) > size_t(FTMOE_NOALLOC_MAX_LOGITS)) return FTMOE_ERR_WORKSPACE;
  void* ws = nullptr;
  const ftmoe_status s = noalloc_scratch(&ws);
  if (s != FTMOE_OK) return s;
  cudaStream_t st = as_stream(stream);
  if (cudaMemsetAsync(ws, 0, FTMOE_WS_ZERO_BYTES, st) != cudaSuccess) return FTMOE_ERR_CUDA;
  return route_impl(d, x, wr, bias, T, ids, w, nullptr, ws, st);
}
