// FP8 latent-KV cache ("[DeepSeek v3.2] 上下文并行详解", section 1 核心改动总结:
// round-robin-split lifts the restriction that NSA prefill CP could not use an
// FP8 KV cache; the page names no format).  Row layout taken: the Dv value
// ("nope") columns as OCP FP8 E4M3 codes with one fp32 scale per tile of 128
// columns (scale = tile max|x| / 448, 1 for an all-zero tile), then the D - Dv
// rope columns as bf16, zero bytes up to a multiple of 16 (656 bytes for the
// DeepSeek-V3.2 latent row of 576).
//
// Codes round to nearest even and saturate at +-448 (the hardware conversion
// cvt.rn.satfinite.e4m3x2.f32), decided in fp32 on x / scale (IEEE division).
// Dequantised values are bf16(fp32(decode(code)) * scale): E4M3 -> f16 is
// exact, the product is one fp32 rounding, then round to nearest bf16.  The
// sparse attention consumes the dequantised rows.
//
// One warp per row; a lane holds 4 consecutive columns of a tile.  HBM-bound.
#include "dsa_common.cuh"
#include "internal.h"

namespace dsa {
namespace {

constexpr int kTile = 128;
constexpr int kRowsPerBlock = 8;

__device__ __forceinline__ uint32_t e4m3x2_sat(float lo, float hi) {
  uint32_t r;
  asm("{\n\t.reg .b16 t;\n\tcvt.rn.satfinite.e4m3x2.f32 t, %1, %2;\n\tcvt.u32.u16 %0, t;\n\t}"
      : "=r"(r)
      : "f"(hi), "f"(lo));
  return r;
}

struct Fp8Geom {
  int D, Dv, tiles, rope_units, row_bytes;  // rope_units: 4-byte units of the bf16 rope columns
};

__global__ void __launch_bounds__(kRowsPerBlock * 32) kv_fp8_quantize_kernel(const __nv_bfloat16 *__restrict__ kv,
                                                                            uint8_t *__restrict__ cache,
                                                                            int64_t num_rows, Fp8Geom g) {
  const int lane = threadIdx.x & 31;
  const int64_t row = static_cast<int64_t>(blockIdx.x) * kRowsPerBlock + (threadIdx.x >> 5);
  if (row >= num_rows) return;
  const __nv_bfloat16 *src = kv + row * g.D;
  uint8_t *dst = cache + row * g.row_bytes;
  // tiles in groups of kGroup: every load of a group is in flight before the
  // first reduction waits on one
  constexpr int kGroup = 4;
  for (int t0 = 0; t0 < g.tiles; t0 += kGroup) {
    float x[kGroup][4];
#pragma unroll
    for (int u = 0; u < kGroup; ++u) {
      const int t = t0 + u;
      const int c0 = t * kTile + 4 * lane;
      x[u][0] = x[u][1] = x[u][2] = x[u][3] = 0.f;
      if (t < g.tiles && 4 * lane < min(kTile, g.Dv - t * kTile)) {
        const uint2 v = *reinterpret_cast<const uint2 *>(src + c0);
        x[u][0] = __uint_as_float(v.x << 16);
        x[u][1] = __uint_as_float(v.x & 0xffff0000u);
        x[u][2] = __uint_as_float(v.y << 16);
        x[u][3] = __uint_as_float(v.y & 0xffff0000u);
      }
    }
#pragma unroll
    for (int u = 0; u < kGroup; ++u) {
      const int t = t0 + u;
      if (t >= g.tiles) break;
      const int c0 = t * kTile + 4 * lane;
      const bool mine = 4 * lane < min(kTile, g.Dv - t * kTile);
      float amax = fmaxf(fmaxf(fabsf(x[u][0]), fabsf(x[u][1])), fmaxf(fabsf(x[u][2]), fabsf(x[u][3])));
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
      const float scale = amax > 0.f ? __fdiv_rn(amax, 448.f) : 1.f;
      if (mine) {
        const uint32_t lo = e4m3x2_sat(__fdiv_rn(x[u][0], scale), __fdiv_rn(x[u][1], scale));
        const uint32_t hi = e4m3x2_sat(__fdiv_rn(x[u][2], scale), __fdiv_rn(x[u][3], scale));
        *reinterpret_cast<uint32_t *>(dst + c0) = lo | (hi << 16);
      }
      if (lane == 0) *reinterpret_cast<float *>(dst + g.Dv + 4 * t) = scale;
    }
  }
  // rope columns: the bf16 bytes as they are; then zero padding
  const uint32_t *rope_src = reinterpret_cast<const uint32_t *>(src + g.Dv);
  uint32_t *rope_dst = reinterpret_cast<uint32_t *>(dst + g.Dv + 4 * g.tiles);
  for (int u = lane; u < g.rope_units; u += 32) rope_dst[u] = rope_src[u];
  const int used = g.Dv + 4 * g.tiles + 4 * g.rope_units;
  for (int b = used + 4 * lane; b < g.row_bytes; b += 128) *reinterpret_cast<uint32_t *>(dst + b) = 0u;
}

__global__ void __launch_bounds__(kRowsPerBlock * 32) kv_fp8_dequantize_kernel(const uint8_t *__restrict__ cache,
                                                                              __nv_bfloat16 *__restrict__ kv,
                                                                              int64_t num_rows, Fp8Geom g) {
  const int lane = threadIdx.x & 31;
  const int64_t row = static_cast<int64_t>(blockIdx.x) * kRowsPerBlock + (threadIdx.x >> 5);
  if (row >= num_rows) return;
  const uint8_t *src = cache + row * g.row_bytes;
  __nv_bfloat16 *dst = kv + row * g.D;
#pragma unroll 4
  for (int t = 0; t < g.tiles; ++t) {
    const int width = min(kTile, g.Dv - t * kTile);
    const int c0 = t * kTile + 4 * lane;
    if (4 * lane >= width) continue;
    const float scale = *reinterpret_cast<const float *>(src + g.Dv + 4 * t);
    const uint32_t codes = *reinterpret_cast<const uint32_t *>(src + c0);
    float a, b, c, d;
    unpack_f16x2(e4m3x2_to_f16x2(codes & 0xffffu), a, b);
    unpack_f16x2(e4m3x2_to_f16x2(codes >> 16), c, d);
    uint2 o;
    o.x = pack_bf16x2(__fmul_rn(a, scale), __fmul_rn(b, scale));
    o.y = pack_bf16x2(__fmul_rn(c, scale), __fmul_rn(d, scale));
    *reinterpret_cast<uint2 *>(dst + c0) = o;
  }
  const uint32_t *rope_src = reinterpret_cast<const uint32_t *>(src + g.Dv + 4 * g.tiles);
  uint32_t *rope_dst = reinterpret_cast<uint32_t *>(dst + g.Dv);
  for (int u = lane; u < g.rope_units; u += 32) rope_dst[u] = rope_src[u];
}

dsa_status fp8_geom(int32_t D, int32_t Dv, Fp8Geom *g) {
  if (D < 1 || Dv < 1 || Dv > D || D > 65536) return DSA_ERR_SHAPE;
  if (Dv % 8 != 0 || (D - Dv) % 8 != 0) return DSA_ERR_SHAPE;
  g->D = D;
  g->Dv = Dv;
  g->tiles = (Dv + kTile - 1) / kTile;
  g->rope_units = (D - Dv) / 2;
  const int raw = Dv + 4 * g->tiles + 2 * (D - Dv);
  g->row_bytes = (raw + 15) / 16 * 16;
  return DSA_OK;
}

}  // namespace
}  // namespace dsa

using namespace dsa;

extern "C" dsa_status dsa_kv_fp8_row_bytes(int32_t D, int32_t Dv, size_t *bytes) {
  if (!bytes) return DSA_ERR_INVALID_ARG;
  Fp8Geom g;
  dsa_status st = fp8_geom(D, Dv, &g);
  if (st != DSA_OK) return st;
  *bytes = static_cast<size_t>(g.row_bytes);
  return DSA_OK;
}

extern "C" dsa_status dsa_kv_fp8_quantize(const void *kv, int32_t num_rows, int32_t D, int32_t Dv, void *cache,
                                          dsa_stream_t stream) {
  if (!kv || !cache) return DSA_ERR_INVALID_ARG;
  if (!aligned16(kv) || !aligned16(cache)) return DSA_ERR_INVALID_ARG;
  if (num_rows < 0) return DSA_ERR_SHAPE;
  Fp8Geom g;
  dsa_status st = fp8_geom(D, Dv, &g);
  if (st != DSA_OK) return st;
  if (num_rows == 0) return DSA_OK;
  const int64_t blocks = (static_cast<int64_t>(num_rows) + kRowsPerBlock - 1) / kRowsPerBlock;
  kv_fp8_quantize_kernel<<<static_cast<unsigned>(blocks), kRowsPerBlock * 32, 0,
                           reinterpret_cast<cudaStream_t>(stream)>>>(static_cast<const __nv_bfloat16 *>(kv),
                                                                      static_cast<uint8_t *>(cache), num_rows, g);
  return check_launch();
}

extern "C" dsa_status dsa_kv_fp8_dequantize(const void *cache, int32_t num_rows, int32_t D, int32_t Dv, void *kv,
                                            dsa_stream_t stream) {
  if (!kv || !cache) return DSA_ERR_INVALID_ARG;
  if (!aligned16(kv) || !aligned16(cache)) return DSA_ERR_INVALID_ARG;
  if (num_rows < 0) return DSA_ERR_SHAPE;
  Fp8Geom g;
  dsa_status st = fp8_geom(D, Dv, &g);
  if (st != DSA_OK) return st;
  if (num_rows == 0) return DSA_OK;
  const int64_t blocks = (static_cast<int64_t>(num_rows) + kRowsPerBlock - 1) / kRowsPerBlock;
  kv_fp8_dequantize_kernel<<<static_cast<unsigned>(blocks), kRowsPerBlock * 32, 0,
                             reinterpret_cast<cudaStream_t>(stream)>>>(static_cast<const uint8_t *>(cache),
                                                                        static_cast<__nv_bfloat16 *>(kv), num_rows, g);
  return check_launch();
}
