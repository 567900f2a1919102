// MLA sparse attention prefill for one CP view ("feat: DeepSeek-V4 DSA
// context-parallel on NPU", section 单层前向数据流 (4): local queries, the
// full shared latent KV, output [T_local, num_heads_FULL, Dv]).
//
// Per local query token: S = scale * Q K^T over its selected latent rows
// (Q: [128 heads, D], K = the gathered rows [n, D]), softmax over the rows
// with an optional per-head sink in the denominator, O = P V with V the
// first Dv columns of the same rows.
//
// GB300 layout (DeepSeek-V3.2 shapes, D = 576, Dv = 512): one fp32 O
// accumulator of 128 heads x 512 values fills an SM's whole tensor memory,
// so each token runs on a 2-CTA cluster.  CTA c owns value columns
// [256c, 256c + 256) and computes the partial QK over latent dims
// [256c, 256c + 256) + [512 + 32c, 512 + 32c + 32): the gathered rows split
// evenly (576 bytes per CTA per row, no row read twice) and the value
// columns are exactly the CTA's main QK chunks, so one smem tile serves as
// QK's K-major B and PV's MN-major B.  The partial S tiles are exchanged
// through distributed shared memory and summed (a + b == b + a bitwise, so
// both CTAs hold the same S and take the same softmax decisions).
//
// Per CTA, 10 warps: 0-3 softmax (one head row = one TMEM lane per thread),
// 4 MMA issue + TMEM owner, 5 Q TMA, 6-9 row gather (cp.async, 128B/64B
// swizzle written directly).  Key blocks of 64 rows, 3 smem stages; two S
// buffers in TMEM, P (bf16) written over its S buffer and fed to the PV MMA
// from TMEM.  The running max is rescaled lazily: O and l are rescaled only
// when a block's max exceeds the max in use by more than 2^8.
//
// The tiny shapes (H = 8, D = 64, Dv = 48) run the same kernel on one CTA
// with Q rows 8..127 zero-filled by the TMA.
#include "dsa_common.cuh"
#include "internal.h"

namespace dsa {
namespace {

template <int NMAIN_, bool TAIL_, int DVC_, bool SPLIT_>
struct AttnCfg {
  static constexpr int NMAIN = NMAIN_;  // 64-wide latent chunks per CTA (128B swizzle)
  static constexpr bool TAIL = TAIL_;   // plus one 32-wide chunk (64B swizzle)
  static constexpr int DVC = DVC_;      // value columns per CTA
  static constexpr bool SPLIT = SPLIT_; // 2-CTA cluster per token
  static constexpr int kBN = 64;        // selected rows per block
  static constexpr int kStages = 3;
  static constexpr int kThreads = 320;
  static constexpr int kQMain = NMAIN * 128 * 128;
  static constexpr int kQTail = TAIL ? 128 * 64 : 0;
  static constexpr int kStageMain = NMAIN * kBN * 128;
  static constexpr int kStageBytes = kStageMain + (TAIL ? kBN * 64 : 0);
  static constexpr int kUnitsPerRow = NMAIN * 8 + (TAIL ? 4 : 0);  // 16-byte pieces
  static constexpr int kQKSteps = NMAIN * 4 + (TAIL ? 2 : 0);
  static constexpr int kPVSteps = kBN / 16;
  static constexpr int kOCols = (DVC + 63) / 64 * 64;
  static constexpr int kSCol = kOCols;  // S / P buffers after O
  static constexpr int kTmemCols = (kOCols + 2 * kBN) <= 256 ? 256 : 512;
  static constexpr int kRecvStride = 68;  // floats per head row (padded against bank conflicts)
  static constexpr int kOffQ = 0;
  static constexpr int kOffStage = kOffQ + kQMain + kQTail;
  static constexpr int kOffRecv = kOffStage + kStages * kStageBytes;
  static constexpr int kOffBar = kOffRecv + (SPLIT ? 128 * kRecvStride * 4 : 0);
  static constexpr int kNumBars = 1 + 2 * kStages + 2 + 2 + 2 + 2;
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;
  static constexpr int kSmemUsed = kOffMisc + 32 + 1024;
  // the tiny variant asks for enough smem that at most two CTAs share an SM's TMEM
  static constexpr int kSmemBytes = kSmemUsed < 100 * 1024 && !SPLIT ? 100 * 1024 : kSmemUsed;
  static constexpr uint32_t kIdescQK = idesc_bf16(128, kBN, false, false);
  static constexpr uint32_t kIdescPV = idesc_bf16(128, DVC, false, true);
  static_assert(kOCols + 2 * kBN <= kTmemCols, "TMEM budget");
  static_assert(DVC % 16 == 0 && DVC <= NMAIN * 64, "value columns inside the main chunks");
  static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
};

using BigAttn = AttnCfg<4, true, 256, true>;
using TinyAttn = AttnCfg<1, false, 48, false>;

struct AttnParams {
  dsa_cp_local_metadata md;
  const __nv_bfloat16 *kv;   // [T][D]
  const int32_t *topk_idx;   // [tpr][topk]
  const float *sink;         // [H] or nullptr
  __nv_bfloat16 *out;        // [tpr][H][Dv]
  float scale_log2;          // softmax_scale * log2(e)
  int32_t topk, H, D, Dv, num_tokens;
  int *err;
};

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

template <class C>
__global__ void __launch_bounds__(C::kThreads, 1)
    sparse_attn_kernel(const __grid_constant__ CUtensorMap qmain_map, const __grid_constant__ CUtensorMap qtail_map,
                       const AttnParams P) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::kOffBar);
  uint64_t *q_full = bars;
  uint64_t *kv_full = q_full + 1;
  uint64_t *kv_empty = kv_full + C::kStages;
  uint64_t *s_full = kv_empty + C::kStages;
  uint64_t *p_full = s_full + 2;
  uint64_t *pv_done = p_full + 2;
  uint64_t *recv_full = pv_done + 2;
  uint64_t *recv_empty = recv_full + 1;
  int32_t *misc = reinterpret_cast<int32_t *>(smem + C::kOffMisc);  // [0] tmem, [1] base, [2] p
  float *recv = reinterpret_cast<float *>(smem + C::kOffRecv);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t crank = C::SPLIT ? cluster_ctarank() : 0u;
  const uint32_t peer = crank ^ 1u;
  const int slot = C::SPLIT ? static_cast<int>(blockIdx.x >> 1) : static_cast<int>(blockIdx.x);
  const int main_dim0 = C::SPLIT ? static_cast<int>(crank) * C::NMAIN * 64 : 0;
  const int tail_dim0 = C::NMAIN * 64 * (C::SPLIT ? 2 : 1) + 32 * static_cast<int>(crank);

  if (tid == 0) {
    int base = 0, p = -1;
    const int g = P.md.local_token_pos[slot];
    const int nb = P.md.scalars[DSA_MD_LOCAL_BATCH];
    if (g >= 0 && nb > 0) {
      const int j = find_local_request(P.md.local_query_start_loc, nb, slot);
      base = P.md.local_req_kv_base[j];
      p = g - base;
      if (p < 0 || g >= P.num_tokens) {
        record_error(P.err, DSA_ERR_DEVICE_BOUNDS, 44, slot);
        p = -1;
      }
    }
    misc[1] = base;
    misc[2] = p;
    mbar_init(q_full, 1);
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(&kv_full[s], 64);
      mbar_init(&kv_empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&s_full[b], 1);
      mbar_init(&p_full[b], 128);
      mbar_init(&pv_done[b], 1);
    }
    mbar_init(recv_full, 128);
    mbar_init(recv_empty, 128);
    fence_mbar_init();
  }
  if (warp == 4) {
    tmem_alloc(reinterpret_cast<uint32_t *>(&misc[0]), C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  if (C::SPLIT) cluster_sync();
  else __syncthreads();
  tc_fence_after();

  const uint32_t tmem = static_cast<uint32_t>(misc[0]);
  const int p = misc[2];
  const int n_valid = p >= 0 ? min(p + 1, P.topk) : 0;
  const int nb = (n_valid + C::kBN - 1) / C::kBN;
  __nv_bfloat16 *out_row = P.out + (static_cast<int64_t>(slot) * P.H) * P.Dv + main_dim0;

  if (nb == 0) {
    // pad slot: zero output rows
    if (warp < 4 && tid < P.H) {
      __nv_bfloat16 *o = out_row + static_cast<int64_t>(tid) * P.Dv;
      for (int c = 0; c < C::DVC; ++c) o[c] = __float2bfloat16(0.f);
    }
  } else if (warp == 5) {
    // ---------------- Q tile by TMA (rows beyond H arrive as zeros)
    if (lane == 0) {
      tma_prefetch_desc(&qmain_map);
      mbar_arrive_expect_tx(q_full, C::kQMain + C::kQTail);
      for (int i = 0; i < C::NMAIN; ++i)
        tma_load_3d(smem + C::kOffQ + i * 128 * 128, &qmain_map, main_dim0 + 64 * i, 0, slot, q_full);
      if (C::TAIL) tma_load_3d(smem + C::kOffQ + C::kQMain, &qtail_map, tail_dim0, 0, slot, q_full);
      mbar_wait(q_full, 0, P.err, 21);
    }
  } else if (warp >= 6) {
    // ---------------- gather of the selected rows: two groups of 64 threads take
    // alternate blocks, one selected row per thread
    const int ptid = tid - 192;
    const int group = ptid >> 6, r = ptid & 63;
    const int32_t *idx_row = P.topk_idx + static_cast<int64_t>(slot) * P.topk;
    for (int j = group; j < nb; j += 2) {
      const int s = j % C::kStages;
      if (!mbar_wait(&kv_empty[s], ((j / C::kStages) & 1) ^ 1, P.err, 22, j)) break;
      const int k = j * C::kBN + r;
      int row = k < n_valid ? __ldg(idx_row + k) : -1;
      if (k < n_valid && (row < 0 || row >= P.num_tokens)) {
        record_error(P.err, DSA_ERR_DEVICE_BOUNDS, 45, k);
        row = -1;
      }
      const __nv_bfloat16 *src = P.kv + static_cast<int64_t>(row < 0 ? 0 : row) * P.D;
      const uint32_t nbytes = row < 0 ? 0u : 16u;
      const uint32_t sb = smem_u32(smem + C::kOffStage + s * C::kStageBytes);
#pragma unroll
      for (int u = 0; u < C::kUnitsPerRow; ++u) {
        if (u < C::NMAIN * 8) {
          const int i = u >> 3, v = u & 7;
          cp_async_16(sb + i * (C::kBN * 128) + r * 128 + ((v ^ (r & 7)) << 4), src + main_dim0 + i * 64 + v * 8,
                      nbytes);
        } else {
          const int v = u - C::NMAIN * 8;
          cp_async_16(sb + C::kStageMain + r * 64 + ((v ^ ((r >> 1) & 3)) << 4), src + tail_dim0 + v * 8, nbytes);
        }
      }
      cp_async_commit();
      cp_async_wait<0>();
      fence_proxy_async_smem();
      mbar_arrive(&kv_full[s]);
    }
    cp_async_wait<0>();
  } else if (warp == 4) {
    // ---------------- MMA issuer
    if (lane == 0) {
      const uint32_t q_addr = smem_u32(smem + C::kOffQ);
      const uint32_t st_addr = smem_u32(smem + C::kOffStage);
      bool ok = mbar_wait(q_full, 0, P.err, 23);
      for (int j = 0; ok && j <= nb; ++j) {
        if (j < nb) {
          const int s = j % C::kStages, b = j & 1;
          if (!(ok = mbar_wait(&kv_full[s], (j / C::kStages) & 1, P.err, 24, j))) break;
          if (j >= 2 && !(ok = mbar_wait(&pv_done[b], ((j - 2) >> 1) & 1, P.err, 25, j))) break;
          tc_fence_after();
          const uint32_t kb = st_addr + s * C::kStageBytes;
#pragma unroll
          for (int k = 0; k < C::kQKSteps; ++k) {
            uint64_t a, bd;
            if (k < C::NMAIN * 4) {
              const int i = k >> 2, sub = k & 3;
              a = smem_desc(q_addr + i * 16384 + sub * 32, 16, 1024, kLayoutSW128);
              bd = smem_desc(kb + i * (C::kBN * 128) + sub * 32, 16, 1024, kLayoutSW128);
            } else {
              const int t = k - C::NMAIN * 4;
              a = smem_desc(q_addr + C::kQMain + t * 32, 16, 512, kLayoutSW64);
              bd = smem_desc(kb + C::kStageMain + t * 32, 16, 512, kLayoutSW64);
            }
            mma_ss(tmem + C::kSCol + b * C::kBN, a, bd, C::kIdescQK, k > 0 ? 1u : 0u);
          }
          mma_commit(&s_full[b]);
        }
        if (j >= 1) {
          const int i = j - 1, si = i % C::kStages, bi = i & 1;
          if (!(ok = mbar_wait(&p_full[bi], (i >> 1) & 1, P.err, 26, i))) break;
          tc_fence_after();
          const uint32_t vb = st_addr + si * C::kStageBytes;
#pragma unroll
          for (int k = 0; k < C::kPVSteps; ++k) {
            const uint64_t bd = smem_desc(vb + k * 2048, C::kBN * 128, 1024, kLayoutSW128);
            mma_ts(tmem, tmem + C::kSCol + bi * C::kBN + k * 8, bd, C::kIdescPV, (i > 0 || k > 0) ? 1u : 0u);
          }
          mma_commit(&pv_done[bi]);
          mma_commit(&kv_empty[si]);
        }
      }
    }
  } else {
    // ---------------- softmax: thread = head row h = TMEM lane
    const int h = tid;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(warp * 32) << 16);
    float m_used = -__builtin_huge_valf(), l = 0.f;
    float *my_recv = recv + h * C::kRecvStride;
    const uint32_t peer_recv = C::SPLIT ? map_to_cta(smem_u32(my_recv), peer) : 0u;
    bool ok = true;
    for (int i = 0; i < nb; ++i) {
      const int b = i & 1;
      // tcgen05.ld/st are warp-collective (.sync.aligned): every decision that
      // guards one is made warp-uniform, including the error path
      ok = __all_sync(0xffffffffu, mbar_wait(&s_full[b], (i >> 1) & 1, P.err, 27, i));
      if (!ok) break;
      tc_fence_after();
      float x[C::kBN];
      {
        uint32_t r0[32], r1[32];
        tmem_ld32(lane_base + C::kSCol + b * C::kBN, r0);
        tmem_ld32(lane_base + C::kSCol + b * C::kBN + 32, r1);
        tmem_ld_wait();
#pragma unroll
        for (int k = 0; k < 32; ++k) {
          x[k] = __uint_as_float(r0[k]);
          x[k + 32] = __uint_as_float(r1[k]);
        }
      }
      if (C::SPLIT) {
        ok = __all_sync(0xffffffffu, i == 0 || mbar_wait<true>(recv_empty, (i - 1) & 1, P.err, 28, i));
        if (!ok) break;
#pragma unroll
        for (int k = 0; k < C::kBN; k += 4) st_cluster_v4(peer_recv + k * 4, x[k], x[k + 1], x[k + 2], x[k + 3]);
        mbar_arrive_remote(recv_full, peer);
        ok = __all_sync(0xffffffffu, mbar_wait<true>(recv_full, i & 1, P.err, 29, i));
        if (!ok) break;
#pragma unroll
        for (int k = 0; k < C::kBN; k += 4) {
          const float4 v = *reinterpret_cast<const float4 *>(my_recv + k);
          x[k] += v.x;
          x[k + 1] += v.y;
          x[k + 2] += v.z;
          x[k + 3] += v.w;
        }
        mbar_arrive_remote(recv_empty, peer);
      }
      float mblk = -__builtin_huge_valf();
#pragma unroll
      for (int k = 0; k < C::kBN; ++k) {
        x[k] = (i * C::kBN + k < n_valid) ? x[k] * P.scale_log2 : -__builtin_huge_valf();
        mblk = fmaxf(mblk, x[k]);
      }
      // lazy rescale: only when some row of the warp saw its max grow by more
      // than 2^8; rows whose max did not grow get alpha = 1 (exact)
      if (__any_sync(0xffffffffu, mblk > m_used + 8.f)) {
        const float m_new = fmaxf(m_used, mblk);
        const float alpha = ex2(m_used - m_new);
        if (i >= 1) {
          // O holds PV(i-1): rescale it before PV(i) accumulates
          ok = __all_sync(0xffffffffu, mbar_wait(&pv_done[(i - 1) & 1], ((i - 1) >> 1) & 1, P.err, 30, i));
          if (!ok) break;
          tc_fence_after();
#pragma unroll 1
          for (int c = 0; c < C::kOCols; c += 32) {
            uint32_t r[32];
            tmem_ld32(lane_base + c, r);
            tmem_ld_wait();
#pragma unroll
            for (int k = 0; k < 32; ++k) r[k] = __float_as_uint(__uint_as_float(r[k]) * alpha);
            tmem_st32(lane_base + c, r);
          }
          tmem_st_wait();
        }
        l *= alpha;
        m_used = m_new;
      }
      uint32_t packed[32];
      float lsum = 0.f;
#pragma unroll
      for (int k = 0; k < C::kBN; k += 2) {
        const float a = ex2(x[k] - m_used), c = ex2(x[k + 1] - m_used);
        lsum += a + c;
        packed[k >> 1] = pack_bf16x2(a, c);
      }
      l += lsum;
      tmem_st32(lane_base + C::kSCol + b * C::kBN, packed);
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&p_full[b]);
    }
    ok = __all_sync(0xffffffffu, ok && mbar_wait(&pv_done[(nb - 1) & 1], ((nb - 1) >> 1) & 1, P.err, 31, nb));
    if (ok) {
      tc_fence_after();
      if (P.sink && h < P.H) l += ex2(P.sink[h] * 1.4426950408889634f - m_used);
      const float inv = 1.f / l;
      __nv_bfloat16 *o = out_row + static_cast<int64_t>(h) * P.Dv;
#pragma unroll 1
      for (int c = 0; c < C::kOCols; c += 32) {
        uint32_t r[32];
        tmem_ld32(lane_base + c, r);
        tmem_ld_wait();
        if (h < P.H) {
#pragma unroll
          for (int k = 0; k < 32; k += 8) {
            if (c + k < C::DVC) {
              uint4 v;
              v.x = pack_bf16x2(__uint_as_float(r[k + 0]) * inv, __uint_as_float(r[k + 1]) * inv);
              v.y = pack_bf16x2(__uint_as_float(r[k + 2]) * inv, __uint_as_float(r[k + 3]) * inv);
              v.z = pack_bf16x2(__uint_as_float(r[k + 4]) * inv, __uint_as_float(r[k + 5]) * inv);
              v.w = pack_bf16x2(__uint_as_float(r[k + 6]) * inv, __uint_as_float(r[k + 7]) * inv);
              *reinterpret_cast<uint4 *>(o + c + k) = v;
            }
          }
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 4) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
  if (C::SPLIT) cluster_sync();  // no CTA leaves while its peer may still touch its smem
}

template <class C>
dsa_status launch_attn(const void *q, int32_t tpr, const AttnParams &P, cudaStream_t stream) {
  CUtensorMap qmain, qtail;
  uint64_t dims[3] = {static_cast<uint64_t>(P.D), static_cast<uint64_t>(P.H), static_cast<uint64_t>(tpr)};
  uint64_t strides[2] = {static_cast<uint64_t>(P.D) * 2, static_cast<uint64_t>(P.H) * P.D * 2};
  uint32_t box_main[3] = {64, 128, 1};
  dsa_status st = encode_tensor_map(&qmain, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, q, dims, strides, box_main,
                                    CU_TENSOR_MAP_SWIZZLE_128B);
  if (st != DSA_OK) return st;
  if (C::TAIL) {
    uint32_t box_tail[3] = {32, 128, 1};
    st = encode_tensor_map(&qtail, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, q, dims, strides, box_tail,
                           CU_TENSOR_MAP_SWIZZLE_64B);
    if (st != DSA_OK) return st;
  } else {
    qtail = qmain;
  }
  cudaError_t e = cudaFuncSetAttribute(sparse_attn_kernel<C>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       C::kSmemBytes);
  if (e != cudaSuccess) return cuda_fail(e);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(tpr) * (C::SPLIT ? 2u : 1u));
  cfg.blockDim = dim3(C::kThreads);
  cfg.dynamicSmemBytes = C::kSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = C::SPLIT ? 2 : 1;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, sparse_attn_kernel<C>, qmain, qtail, P);
  if (e != cudaSuccess) return cuda_fail(e);
  return check_launch();
}

}  // namespace
}  // namespace dsa

using namespace dsa;

extern "C" dsa_status dsa_sparse_attn_prefill(const dsa_cp_local_metadata *md, int32_t batch, int32_t tpr,
                                              const void *q, const void *kv, int32_t num_tokens,
                                              const int32_t *topk_idx, int32_t topk, const float *attn_sink,
                                              float softmax_scale, int32_t H, int32_t D, int32_t Dv, void *out,
                                              dsa_stream_t stream) {
  if (!md || !q || !kv || !topk_idx || !out) return DSA_ERR_INVALID_ARG;
  if (!md->scalars || !md->local_query_start_loc || !md->local_req_kv_base || !md->local_token_pos)
    return DSA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(kv) || !aligned16(out)) return DSA_ERR_INVALID_ARG;
  if (batch < 0 || tpr < 0 || num_tokens < 1 || topk < 1) return DSA_ERR_SHAPE;
  if (!(softmax_scale > 0.f) || softmax_scale != softmax_scale) return DSA_ERR_INVALID_ARG;
  if (tpr == 0) return DSA_OK;
  if (static_cast<int64_t>(tpr) * 2 > INT32_MAX) return DSA_ERR_SHAPE;
  const bool big = H == 128 && D == 576 && Dv == 512 && topk == 2048;
  const bool tiny = H == 8 && D == 64 && Dv == 48 && topk == 64;
  if (!big && !tiny) return DSA_ERR_UNSUPPORTED;
  int *err = device_error_word();
  if (!err) return DSA_ERR_CUDA;
  AttnParams P{*md,
               static_cast<const __nv_bfloat16 *>(kv),
               topk_idx,
               attn_sink,
               static_cast<__nv_bfloat16 *>(out),
               static_cast<float>(static_cast<double>(softmax_scale) * 1.4426950408889634),
               topk,
               H,
               D,
               Dv,
               num_tokens,
               err};
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  return big ? launch_attn<BigAttn>(q, tpr, P, s) : launch_attn<TinyAttn>(q, tpr, P, s);
}
