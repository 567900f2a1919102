// Split and rerange of the CP token layout ("[DeepSeek v3.2] 上下文并行详解",
// sections 2.B and 第三部分; "NSA Prefill CP 中两次 All-Gather 的作用说明",
// 第一次 All-Gather) and the head/token all-to-all of the attention outputs
// ("feat: DeepSeek-V4 DSA context-parallel on NPU", 单层前向数据流 (6)).  All
// are row gathers: dst row d <- the source row that map(d) points at, or zeros
// when map(d) is a pad slot.  HBM-bound byte copies, bit-exact.
//
// Large rows (>= 2 KB, e.g. 147,456-byte attention-query rows): one CTA
// copies a 16 KB piece of one row with 16-byte vectors, 8 loads in flight per
// thread.  Small rows (e.g. 256-byte indexer-weight rows): one warp per row.
#include "dsa_common.cuh"
#include "internal.h"

namespace dsa {
namespace {

// Each map gives, for destination row d, the element offset of its source row
// (in units of the copy's vector type; rows are `e` units long), or -1 for a
// pad row that is written as zeros.
struct SplitMap {  // dst [n_ranks][tpr] <- src [T]
  int64_t tpr, T;
  int32_t cp, rank, mode;  // rank < 0: all ranks
  __device__ __forceinline__ int64_t operator()(int64_t d, int64_t e) const {
    const int64_t r = rank < 0 ? d / tpr : rank;
    const int64_t i = rank < 0 ? d - r * tpr : d;
    const int64_t g = cp_row_of_slot(r, i, tpr, cp, mode);
    return g < T ? g * e : -1;
  }
};

struct RerangeMap {  // dst [T] <- src [cp][tpr]
  int64_t tpr;
  int32_t cp, mode;
  __device__ __forceinline__ int64_t operator()(int64_t g, int64_t e) const {
    int64_t r, i;
    cp_slot_of_row(g, tpr, cp, mode, r, i);
    return (r * tpr + i) * e;
  }
};

// dst [cp][T][H / cp] head slices <- src [cp][tpr][H]: destination row
// d = rd * T + g is heads rd * H / cp .. of token g, taken from the view that
// computed g (its slot there as in RerangeMap); a row is H / cp heads long.
struct HeadA2AMap {
  int64_t tpr, T;
  int32_t cp, mode;
  __device__ __forceinline__ int64_t operator()(int64_t d, int64_t e) const {
    const int64_t rd = d / T, g = d - rd * T;
    int64_t r, i;
    cp_slot_of_row(g, tpr, cp, mode, r, i);
    return ((r * tpr + i) * cp + rd) * e;  // a token row is cp slices of e units
  }
};

constexpr int kBigThreads = 128;
constexpr int kBigUnroll = 8;
constexpr int64_t kBigChunk = kBigThreads * kBigUnroll;  // elements per CTA

template <class T, class Map>
__global__ void __launch_bounds__(kBigThreads) copy_rows_big(const T *__restrict__ src, T *__restrict__ dst,
                                                             int64_t elems_per_row, Map map) {
  const int64_t row = blockIdx.x;
  const int64_t s = map(row, elems_per_row);
  const int64_t e0 = static_cast<int64_t>(blockIdx.y) * kBigChunk + threadIdx.x;
  const T *sp = src + s;
  T *dp = dst + row * elems_per_row;
  T v[kBigUnroll];
#pragma unroll
  for (int k = 0; k < kBigUnroll; ++k) {
    const int64_t e = e0 + k * kBigThreads;
    if (s >= 0 && e < elems_per_row) v[k] = __ldcs(sp + e);
    else v[k] = T{};
  }
#pragma unroll
  for (int k = 0; k < kBigUnroll; ++k) {
    const int64_t e = e0 + k * kBigThreads;
    if (e < elems_per_row) __stcs(dp + e, v[k]);
  }
}

template <class T, class Map>
__global__ void __launch_bounds__(256) copy_rows_small(const T *__restrict__ src, T *__restrict__ dst,
                                                       int64_t elems_per_row, int64_t n_rows, Map map) {
  const int64_t row = static_cast<int64_t>(blockIdx.x) * 8 + (threadIdx.x >> 5);
  if (row >= n_rows) return;
  const int64_t s = map(row, elems_per_row);
  for (int64_t e = threadIdx.x & 31; e < elems_per_row; e += 32)
    dst[row * elems_per_row + e] = s >= 0 ? src[s + e] : T{};
}

template <class Map>
dsa_status launch_copy(const void *src, void *dst, int64_t row_bytes, int64_t n_rows, Map map,
                       cudaStream_t stream) {
  if (n_rows == 0) return DSA_OK;
  const bool a16 = aligned16(src) && aligned16(dst) && (row_bytes % 16 == 0);
  const bool a4 = ((reinterpret_cast<uintptr_t>(src) | reinterpret_cast<uintptr_t>(dst)) % 4 == 0) &&
                  (row_bytes % 4 == 0);
  auto go = [&](auto tag) -> dsa_status {
    using T = decltype(tag);
    const int64_t elems = row_bytes / static_cast<int64_t>(sizeof(T));
    if (row_bytes >= 2048) {
      const int64_t chunks = (elems + kBigChunk - 1) / kBigChunk;
      if (chunks > 65535 || n_rows > INT32_MAX) return DSA_ERR_SHAPE;
      dim3 grid(static_cast<unsigned>(n_rows), static_cast<unsigned>(chunks));
      copy_rows_big<T, Map><<<grid, kBigThreads, 0, stream>>>(static_cast<const T *>(src), static_cast<T *>(dst),
                                                             elems, map);
    } else {
      const int64_t blocks = (n_rows + 7) / 8;
      if (blocks > INT32_MAX) return DSA_ERR_SHAPE;
      copy_rows_small<T, Map><<<static_cast<unsigned>(blocks), 256, 0, stream>>>(
          static_cast<const T *>(src), static_cast<T *>(dst), elems, n_rows, map);
    }
    return check_launch();
  };
  if (a16) return go(uint4{});
  if (a4) return go(uint32_t{});
  return go(uint8_t{});
}

}  // namespace
}  // namespace dsa

using namespace dsa;

extern "C" dsa_status dsa_cp_split(const void *src, int64_t row_bytes, int32_t num_tokens, int32_t cp_size,
                                   dsa_cp_mode mode, int32_t cp_rank, void *dst, dsa_stream_t stream) {
  if (!src || !dst) return DSA_ERR_INVALID_ARG;
  if (mode != DSA_CP_IN_SEQ_SPLIT && mode != DSA_CP_ROUND_ROBIN && mode != DSA_CP_HEAD_TAIL)
    return DSA_ERR_INVALID_ARG;
  if (cp_size < 1 || cp_rank < -1 || cp_rank >= cp_size) return DSA_ERR_INVALID_ARG;
  if (row_bytes <= 0 || num_tokens < 0) return DSA_ERR_SHAPE;
  int32_t pad = 0, tpr = 0;
  dsa_status st = dsa_cp_geometry(num_tokens, cp_size, &pad, &tpr);
  if (st != DSA_OK) return st;
  const int64_t n_rows = cp_rank < 0 ? static_cast<int64_t>(pad) : tpr;
  SplitMap map{tpr, num_tokens, cp_size, cp_rank, static_cast<int32_t>(mode)};
  return launch_copy(src, dst, row_bytes, n_rows, map, reinterpret_cast<cudaStream_t>(stream));
}

extern "C" dsa_status dsa_cp_rerange(const void *src, int64_t row_bytes, int32_t num_tokens, int32_t cp_size,
                                     dsa_cp_mode mode, void *dst, dsa_stream_t stream) {
  if (!src || !dst) return DSA_ERR_INVALID_ARG;
  if (mode != DSA_CP_IN_SEQ_SPLIT && mode != DSA_CP_ROUND_ROBIN && mode != DSA_CP_HEAD_TAIL)
    return DSA_ERR_INVALID_ARG;
  if (cp_size < 1) return DSA_ERR_INVALID_ARG;
  if (row_bytes <= 0 || num_tokens < 0) return DSA_ERR_SHAPE;
  int32_t pad = 0, tpr = 0;
  dsa_status st = dsa_cp_geometry(num_tokens, cp_size, &pad, &tpr);
  if (st != DSA_OK) return st;
  RerangeMap map{tpr, cp_size, static_cast<int32_t>(mode)};
  return launch_copy(src, dst, row_bytes, num_tokens, map, reinterpret_cast<cudaStream_t>(stream));
}

extern "C" dsa_status dsa_cp_all_to_all_heads(const void *src, int32_t num_heads, int64_t head_bytes,
                                              int32_t num_tokens, int32_t cp_size, dsa_cp_mode mode, void *dst,
                                              dsa_stream_t stream) {
  if (!src || !dst) return DSA_ERR_INVALID_ARG;
  if (mode != DSA_CP_IN_SEQ_SPLIT && mode != DSA_CP_ROUND_ROBIN && mode != DSA_CP_HEAD_TAIL)
    return DSA_ERR_INVALID_ARG;
  if (cp_size < 1) return DSA_ERR_INVALID_ARG;
  if (num_heads < 1 || num_heads % cp_size != 0 || head_bytes <= 0 || num_tokens < 0) return DSA_ERR_SHAPE;
  int32_t pad = 0, tpr = 0;
  dsa_status st = dsa_cp_geometry(num_tokens, cp_size, &pad, &tpr);
  if (st != DSA_OK) return st;
  const int64_t slice_bytes = head_bytes * (num_heads / cp_size);
  if (slice_bytes > (int64_t{1} << 40) / cp_size) return DSA_ERR_SHAPE;
  HeadA2AMap map{tpr, num_tokens, cp_size, static_cast<int32_t>(mode)};
  return launch_copy(src, dst, slice_bytes, static_cast<int64_t>(cp_size) * num_tokens, map,
                     reinterpret_cast<cudaStream_t>(stream));
}

// ------------------------------------------------------------------ one rank's rows to / from host memory
// A rank's slots are at most two runs of consecutive slots whose flat rows are
// evenly spaced (in-seq: one contiguous run; round-robin: one run of stride
// cp; head-tail: the head run and the tail run).  Each run is one 2D copy of
// the copy engines: rows of row_bytes, the flat side pitched by stride rows.
namespace dsa {
namespace {

struct RowRun {
  int64_t slot0, row0, n, stride;  // slots [slot0, slot0 + n) <-> flat rows row0 + k * stride
};

int rank_runs(int64_t T, int64_t tpr, int64_t cp, int64_t r, int mode, RowRun runs[2]) {
  auto clamp_n = [](int64_t v, int64_t hi) { return v < 0 ? int64_t{0} : (v > hi ? hi : v); };
  if (mode == DSA_CP_IN_SEQ_SPLIT) {
    runs[0] = {0, r * tpr, clamp_n(T - r * tpr, tpr), 1};
    return 1;
  }
  if (mode == DSA_CP_ROUND_ROBIN) {
    runs[0] = {0, r, r < T ? clamp_n((T - r + cp - 1) / cp, tpr) : 0, cp};
    return 1;
  }
  const int64_t h = (tpr + 1) / 2, t = tpr / 2;
  runs[0] = {0, r * h, clamp_n(T - r * h, h), 1};
  const int64_t tail0 = cp * h + (cp - 1 - r) * t;
  runs[1] = {h, tail0, clamp_n(T - tail0, t), 1};
  return 2;
}

dsa_status host_rows_copy(const void *src, void *dst, int64_t row_bytes, int32_t num_tokens, int32_t cp_size,
                          dsa_cp_mode mode, int32_t cp_rank, bool to_device, cudaStream_t stream) {
  if (!src || !dst) return DSA_ERR_INVALID_ARG;
  if (mode != DSA_CP_IN_SEQ_SPLIT && mode != DSA_CP_ROUND_ROBIN && mode != DSA_CP_HEAD_TAIL)
    return DSA_ERR_INVALID_ARG;
  if (cp_size < 1 || cp_rank < 0 || cp_rank >= cp_size) return DSA_ERR_INVALID_ARG;
  if (row_bytes <= 0 || num_tokens < 0) return DSA_ERR_SHAPE;
  int32_t pad = 0, tpr = 0;
  dsa_status st = dsa_cp_geometry(num_tokens, cp_size, &pad, &tpr);
  if (st != DSA_OK) return st;
  if (row_bytes > (int64_t{1} << 40) / (static_cast<int64_t>(cp_size) * (static_cast<int64_t>(pad) + 1)))
    return DSA_ERR_SHAPE;
  RowRun runs[2];
  const int nr = rank_runs(num_tokens, tpr, cp_size, cp_rank, static_cast<int>(mode), runs);
  for (int k = 0; k < nr; ++k) {
    const RowRun &u = runs[k];
    if (u.n == 0) continue;
    const size_t w = static_cast<size_t>(row_bytes), flat_pitch = static_cast<size_t>(u.stride * row_bytes);
    const char *s = static_cast<const char *>(src);
    char *d = static_cast<char *>(dst);
    cudaError_t e;
    if (to_device)
      e = cudaMemcpy2DAsync(d + u.slot0 * row_bytes, w, s + u.row0 * row_bytes, flat_pitch, w,
                            static_cast<size_t>(u.n), cudaMemcpyHostToDevice, stream);
    else
      e = cudaMemcpy2DAsync(d + u.row0 * row_bytes, flat_pitch, s + u.slot0 * row_bytes, w, w,
                            static_cast<size_t>(u.n), cudaMemcpyDeviceToHost, stream);
    if (e != cudaSuccess) return cuda_fail(e);
  }
  return DSA_OK;
}

}  // namespace
}  // namespace dsa

extern "C" dsa_status dsa_cp_split_from_host(const void *host_src, int64_t row_bytes, int32_t num_tokens,
                                             int32_t cp_size, dsa_cp_mode mode, int32_t cp_rank, void *dst,
                                             dsa_stream_t stream) {
  return host_rows_copy(host_src, dst, row_bytes, num_tokens, cp_size, mode, cp_rank, true,
                        reinterpret_cast<cudaStream_t>(stream));
}

extern "C" dsa_status dsa_cp_rerange_to_host(const void *src, int64_t row_bytes, int32_t num_tokens,
                                             int32_t cp_size, dsa_cp_mode mode, int32_t cp_rank, void *host_dst,
                                             dsa_stream_t stream) {
  return host_rows_copy(src, host_dst, row_bytes, num_tokens, cp_size, mode, cp_rank, false,
                        reinterpret_cast<cudaStream_t>(stream));
}
