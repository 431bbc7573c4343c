// Host-side check of the decode kernels' shared-memory layouts (sd_layout, sl_layout) over a
// sweep of layer shapes: for every shape a kernel accepts, the regions are ordered, aligned,
// large enough for what the kernels put there, and fit in the opt-in shared memory of one
// CTA (the slice form's ring also holds the cluster form's partial output).  Prints one line
// per failure and "checked N layouts"; exits 1 on any failure.
#include <cstdio>
#include "../../sparse_moe_expert_sorted_b300/csrc/decode_stream.cuh"

using namespace ftmoe;

static int fails = 0;
#define CHECK(c, ...)                                   \
  do {                                                  \
    if (!(c)) {                                         \
      if (fails < 50) {                                 \
        std::printf("FAIL %s: ", #c);                   \
        std::printf(__VA_ARGS__);                       \
        std::printf("\n");                              \
      }                                                 \
      ++fails;                                          \
    }                                                   \
  } while (0)

int main() {
  const int max_smem = 232448, grid = 148;
  const int Es[] = {1, 2, 8, 16, 64, 128, 148, 256, 300, 512, 1024};
  const int ds[] = {256, 512, 768, 1024, 2048, 3072, 4096, 6144, 8192};
  const int fs[] = {128, 256, 384, 512, 768, 1024, 2048, 4096, 8192};
  const int ks[] = {1, 2, 4, 6, 8, 32};
  const int Ts[] = {1, 2, 3, 4, 5, 6, 7, 8, 9, 16, 64, 255};
  long long n = 0;
  for (int fmt : {FTMOE_NVFP4, FTMOE_MXFP4})
    for (int E : Es)
      for (int d : ds)
        for (int f : fs)
          for (int k : ks) {
            if (k > E) continue;
            for (int T : Ts) {
              const int sa = sd_block_bytes_a(d, fmt), sb = sd_block_bytes_b(f, fmt);
              for (int route = 0; route < 2; ++route) {
                const bool ok = route ? sd_route_supported(E, d, f, fmt, T, k, grid, max_smem)
                                      : sd_supported(E, d, f, fmt, T, k, max_smem);
                if (!ok) continue;
                ++n;
                const SdLayout L = sd_layout(E, d, f, fmt, T, k, route != 0, max_smem);
                const int kx = d > f ? d : f;
                CHECK(L.stages >= 2 && L.stages <= kSdMaxStages, "E %d d %d f %d T %d", E, d, f, T);
                CHECK(L.stage_bytes % 128 == 0 && L.stage_bytes >= sa && L.stage_bytes >= sb, "d %d f %d", d, f);
                CHECK(sa % 16 == 0 && sb % 16 == 0, "bulk copy sizes d %d f %d", d, f);
                CHECK(L.off_x == L.stages * L.stage_bytes, "off_x");
                CHECK(L.off_red - L.off_x >= L.xrows * (kx + 8) * 2, "x rows E %d d %d f %d T %d", E, d, f, T);
                CHECK(L.off_rank - L.off_red >= L.nbufs * L.nred * 4, "reduction buffers");
                CHECK(L.nred == kSdCons * 2 * 16 * L.xrows && L.xrows == (T < 8 ? T : 8), "nred");
                CHECK(L.off_route - L.off_rank >= sd_info_ints(E) * 4, "info");
                CHECK(L.off_bar - L.off_route >= (route ? sd_route_ints(E, T, k) : 0) * 4, "router scratch");
                CHECK(L.off_x % 16 == 0 && L.off_red % 16 == 0 && L.off_rank % 16 == 0 && L.off_route % 16 == 0 &&
                          L.off_bar % 16 == 0, "16-byte regions");
                CHECK(L.smem - L.off_bar >= 256 + 128 && L.smem <= max_smem, "smem %d E %d d %d f %d T %d", L.smem,
                      E, d, f, T);
                CHECK(L.nbufs == 1 || L.nbufs == 2, "nbufs");
                if (route) {
                  const long long rows = (E + grid - 1) / grid;
                  CHECK(rows * d * 2 <= (long long)L.stages * L.stage_bytes, "router rows in the ring");
                }
              }
              if (T <= kSdRouteMaxT && sl_supported(E, d, f, fmt, T, k, grid, max_smem)) {
                ++n;
                const SlLayout S = sl_layout(E, d, fmt, T, k, max_smem);
                CHECK(sl_wanted(d, fmt) && d <= 2048, "slice form beyond d 2048");
                CHECK(S.stages >= 2 && S.stages <= 4, "slice stages");
                CHECK(S.off_d % 128 == 0 && S.off_d >= S.blk_a && S.blk_a == sa, "slice tile offset");
                CHECK(S.stage_bytes % 128 == 0 && S.stage_bytes >= S.off_d + sl_slice_bytes(d), "slice stage");
                CHECK(sl_slice_bytes(d) % 16 == 0 && S.blk_a % 16 == 0, "slice bulk copy sizes");
                CHECK(S.off_x == S.stages * S.stage_bytes, "slice off_x");
                CHECK(S.off_red - S.off_x >= T * (d + 8) * 2, "slice x rows");
                CHECK(S.off_rank - S.off_red >= kSdRedBufs * S.nred * 4 && S.nred == kSdCons * 2 * 16 * T, "slice red");
                CHECK(S.off_route - S.off_rank >= sd_info_ints(E) * 4, "slice info");
                CHECK(S.off_h - S.off_route >= sd_route_ints(E, T, k) * 4, "slice router scratch");
                CHECK(S.off_bar - S.off_h >= 2 * 8 * 16 * 2, "slice h buffers");
                CHECK(S.smem - S.off_bar >= 256 + 128 && S.smem <= max_smem, "slice smem %d", S.smem);
                CHECK(f % kSdRowsA == 0, "slice f");
                const long long rows = (E + grid - 1) / grid;
                CHECK(rows * d * 2 <= (long long)S.stages * S.stage_bytes, "slice router rows");
                // the cluster form leaves each CTA's partial output [T][d] (fp32) over the ring
                CHECK((long long)T * d * 4 <= (long long)S.stages * S.stage_bytes, "slice partial E %d d %d T %d", E,
                      d, T);
              }
            }
          }
  std::printf("checked %lld layouts, %d failures\n", n, fails);
  return fails ? 1 : 0;
}
