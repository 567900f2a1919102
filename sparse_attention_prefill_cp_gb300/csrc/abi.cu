// Host-only parts of the C ABI: status strings, the device error word,
// CP geometry / metadata sizing, tensor-map encoding.
#include <cudaTypedefs.h>

#include <cstdio>
#include <mutex>

#include "internal.h"

namespace dsa {

// One error record per device: {first dsa_status a kernel recorded, site,
// detail, block}; read and cleared by dsa_poll_device_error.
static __device__ int g_device_error[4] = {0, 0, 0, 0};

static thread_local char t_last_cuda_error[256] = "";

dsa_status cuda_fail_msg(const char *msg) {
  snprintf(t_last_cuda_error, sizeof(t_last_cuda_error), "%s", msg);
  return DSA_ERR_CUDA;
}

dsa_status cuda_fail(cudaError_t e) {
  snprintf(t_last_cuda_error, sizeof(t_last_cuda_error), "%s: %s", cudaGetErrorName(e), cudaGetErrorString(e));
  return DSA_ERR_CUDA;
}

static constexpr int kMaxDevices = 64;
static int *s_error_word[kMaxDevices];
static std::mutex s_error_mutex;

int *device_error_word() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(s_error_mutex);
  if (!s_error_word[dev]) {
    void *p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_device_error);
    if (e != cudaSuccess) {
      cuda_fail(e);
      return nullptr;
    }
    s_error_word[dev] = static_cast<int *>(p);
  }
  return s_error_word[dev];
}

int num_sms() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 1;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) return 1;
  return n;
}

static PFN_cuTensorMapEncodeTiled_v12000 s_encode = nullptr;
static std::once_flag s_encode_once;

dsa_status encode_tensor_map(CUtensorMap *map, CUtensorMapDataType dtype, uint32_t rank, const void *base,
                             const uint64_t *dims, const uint64_t *strides_bytes, const uint32_t *box,
                             CUtensorMapSwizzle swizzle) {
  std::call_once(s_encode_once, [] {
    void *fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      s_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  if (!s_encode) return cuda_fail_msg("cuTensorMapEncodeTiled entry point not found");
  cuuint32_t elem_strides[3] = {1, 1, 1};
  CUresult r = s_encode(map, dtype, rank, const_cast<void *>(base), reinterpret_cast<const cuuint64_t *>(dims),
                        reinterpret_cast<const cuuint64_t *>(strides_bytes),
                        reinterpret_cast<const cuuint32_t *>(box), elem_strides, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    char buf[96];
    snprintf(buf, sizeof(buf), "cuTensorMapEncodeTiled failed (CUresult %d)", static_cast<int>(r));
    return cuda_fail_msg(buf);
  }
  return DSA_OK;
}

}  // namespace dsa

using namespace dsa;

extern "C" {

int32_t dsa_abi_version(void) { return DSA_CP_ABI_VERSION; }

const char *dsa_last_cuda_error(void) { return t_last_cuda_error; }

const char *dsa_status_string(dsa_status s) {
  switch (s) {
    case DSA_OK: return "DSA_OK";
    case DSA_ERR_INVALID_ARG: return "DSA_ERR_INVALID_ARG: invalid argument (null pointer, rank or mode out of range)";
    case DSA_ERR_SHAPE: return "DSA_ERR_SHAPE: inconsistent or out-of-range sizes";
    case DSA_ERR_UNSUPPORTED: return "DSA_ERR_UNSUPPORTED: dimension set not compiled into this library";
    case DSA_ERR_WORKSPACE: return "DSA_ERR_WORKSPACE: workspace too small";
    case DSA_ERR_CUDA: return "DSA_ERR_CUDA: a CUDA call failed (see dsa_last_cuda_error)";
    case DSA_ERR_DEVICE_TIMEOUT: return "DSA_ERR_DEVICE_TIMEOUT: a device-side wait ran past its limit";
    case DSA_ERR_DEVICE_BOUNDS: return "DSA_ERR_DEVICE_BOUNDS: a device-side index was out of range";
    case DSA_ERR_DEVICE_SEQ_LENS:
      return "DSA_ERR_DEVICE_SEQ_LENS: a seq_lens entry is below its query length (or the KV rows overflow int32)";
  }
  return "unknown dsa_status";
}

dsa_status dsa_cp_geometry(int32_t num_tokens, int32_t cp_size, int32_t *num_tokens_pad, int32_t *tokens_per_rank) {
  if (!num_tokens_pad || !tokens_per_rank || cp_size < 1) return DSA_ERR_INVALID_ARG;
  if (num_tokens < 0) return DSA_ERR_SHAPE;
  const int64_t tpr = (static_cast<int64_t>(num_tokens) + cp_size - 1) / cp_size;
  const int64_t pad = tpr * cp_size;
  if (pad > INT32_MAX) return DSA_ERR_SHAPE;
  *num_tokens_pad = static_cast<int32_t>(pad);
  *tokens_per_rank = static_cast<int32_t>(tpr);
  return DSA_OK;
}

dsa_status dsa_cp_metadata_sizes(int32_t batch, int32_t num_tokens, int32_t cp_size, size_t *ints_needed) {
  if (!ints_needed) return DSA_ERR_INVALID_ARG;
  if (batch < 0) return DSA_ERR_SHAPE;
  int32_t pad = 0, tpr = 0;
  dsa_status st = dsa_cp_geometry(num_tokens, cp_size, &pad, &tpr);
  if (st != DSA_OK) return st;
  *ints_needed = static_cast<size_t>(DSA_MD_NUM_SCALARS) + 2 * (static_cast<size_t>(batch) + 1) +
                 4 * static_cast<size_t>(batch) + static_cast<size_t>(tpr);
  return DSA_OK;
}

dsa_status dsa_cp_metadata_bind(int32_t *buffer, int32_t batch, int32_t num_tokens, int32_t cp_size,
                                dsa_cp_local_metadata *out) {
  if (!buffer || !out) return DSA_ERR_INVALID_ARG;
  size_t n = 0;
  dsa_status st = dsa_cp_metadata_sizes(batch, num_tokens, cp_size, &n);
  if (st != DSA_OK) return st;
  int32_t *p = buffer;
  const size_t B = static_cast<size_t>(batch);
  out->scalars = p;                p += DSA_MD_NUM_SCALARS;
  out->local_query_start_loc = p;  p += B + 1;
  out->local_seq_lens = p;         p += B;
  out->local_kv_start_loc = p;     p += B + 1;
  out->local_req_id = p;           p += B;
  out->local_req_kv_base = p;      p += B;
  out->local_req_pos_base = p;     p += B;
  out->local_token_pos = p;
  return DSA_OK;
}

dsa_status dsa_poll_device_error_detail(dsa_stream_t stream, int32_t *detail) {
  cudaError_t e = cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e);
  int *word = device_error_word();
  if (!word) return DSA_ERR_CUDA;
  int value[4] = {0, 0, 0, 0};
  e = cudaMemcpy(value, word, sizeof(value), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e);
  if (value[0] != 0) {
    const int zero[4] = {0, 0, 0, 0};
    e = cudaMemcpy(word, zero, sizeof(zero), cudaMemcpyHostToDevice);
    if (e != cudaSuccess) return cuda_fail(e);
  }
  if (detail)
    for (int i = 0; i < 3; ++i) detail[i] = value[i + 1];
  return static_cast<dsa_status>(value[0]);
}

dsa_status dsa_poll_device_error(dsa_stream_t stream) { return dsa_poll_device_error_detail(stream, nullptr); }

}  // extern "C"
