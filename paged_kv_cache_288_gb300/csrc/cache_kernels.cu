// Cache writes: the slot scatter of new tokens and the whole-block copy of
// copy-on-write. Both are pure data movement with 16-byte vector accesses.
#include "common.cuh"
#include "internal.h"

namespace pa {
namespace {

// One CTA per token; each thread moves 8 elements (16 source bytes) of one
// KV head's row. For 16-bit caches the bits are copied; for an E4M3 cache
// each value is divided by its (block, head) scale in IEEE float32 and
// converted with round-to-nearest-even and saturation to +-448.
template <typename ST, typename CT>
__global__ void reshape_and_cache_kernel(const ST* __restrict__ key, const ST* __restrict__ value,
                                         CT* __restrict__ k_cache, CT* __restrict__ v_cache,
                                         const int64_t* __restrict__ slot_mapping,
                                         int num_kv_heads, int head_dim, int block_size,
                                         int num_blocks, const float* __restrict__ k_scale,
                                         const float* __restrict__ v_scale, int32_t* debug_err) {
  const int t = blockIdx.x;
  const int64_t slot = slot_mapping[t];
  if (slot < 0) return;
  if (slot >= static_cast<int64_t>(num_blocks) * block_size) {
    if (threadIdx.x == 0) flag_error(debug_err, PA_DEVERR_SLOT_RANGE);
    return;
  }
  const int64_t blk = slot / block_size;
  const int off = static_cast<int>(slot % block_size);
  const int chunks_per_head = head_dim / 8;
  const int chunks = num_kv_heads * chunks_per_head;
  for (int c = threadIdx.x; c < chunks; c += blockDim.x) {
    const int h = c / chunks_per_head;
    const int e = (c % chunks_per_head) * 8;
    const int64_t src = (static_cast<int64_t>(t) * num_kv_heads + h) * head_dim + e;
    const int64_t dst = ((blk * num_kv_heads + h) * block_size + off) * head_dim + e;
    if constexpr (!is_fp8<CT>::value) {
      static_assert(sizeof(ST) == sizeof(CT), "16-bit caches copy bits");
      *reinterpret_cast<uint4*>(k_cache + dst) = *reinterpret_cast<const uint4*>(key + src);
      *reinterpret_cast<uint4*>(v_cache + dst) = *reinterpret_cast<const uint4*>(value + src);
    } else {
      const float ks = k_scale[blk * num_kv_heads + h];
      const float vs = v_scale[blk * num_kv_heads + h];
      float kf[8], vf[8];
      load_float<ST, 8>(key + src, kf);
      load_float<ST, 8>(value + src, vf);
      uint2 ko, vo;
      uint8_t* kb = reinterpret_cast<uint8_t*>(&ko);
      uint8_t* vb = reinterpret_cast<uint8_t*>(&vo);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        kb[i] = __nv_cvt_float_to_fp8(__fdiv_rn(kf[i], ks), __NV_SATFINITE, __NV_E4M3);
        vb[i] = __nv_cvt_float_to_fp8(__fdiv_rn(vf[i], vs), __NV_SATFINITE, __NV_E4M3);
      }
      *reinterpret_cast<uint2*>(k_cache + dst) = ko;
      *reinterpret_cast<uint2*>(v_cache + dst) = vo;
    }
  }
}

// grid = (num_pairs, num_layers, 2: K then V). Each CTA copies one block of
// one cache with 16-byte loads and stores.
__global__ void copy_blocks_kernel(void* const* __restrict__ k_caches, void* const* __restrict__ v_caches,
                                   const int64_t* __restrict__ block_mapping, int num_blocks,
                                   int64_t block_vecs, int32_t* debug_err) {
  const int pair = blockIdx.x;
  const int layer = blockIdx.y;
  const int64_t src = block_mapping[2 * pair];
  const int64_t dst = block_mapping[2 * pair + 1];
  if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks) {
    if (threadIdx.x == 0 && layer == 0 && blockIdx.z == 0) flag_error(debug_err, PA_DEVERR_BLOCK_RANGE);
    return;
  }
  uint4* base = reinterpret_cast<uint4*>(blockIdx.z == 0 ? k_caches[layer] : v_caches[layer]);
  const uint4* s = base + src * block_vecs;
  uint4* d = base + dst * block_vecs;
  for (int64_t i = threadIdx.x; i < block_vecs; i += blockDim.x) d[i] = s[i];
}

// grid = (num_pairs, num_layers, 2: K then V). Each CTA moves one block of
// one cache of one layer between two pools (device memory or mapped pinned
// host memory), kSwapUnroll 16-byte vectors per thread in flight.
constexpr int kSwapThreads = 256;
constexpr int kSwapUnroll = 4;

__global__ void __launch_bounds__(kSwapThreads) swap_blocks_kernel(const __grid_constant__ SwapPools pools,
                                                                   const int64_t* __restrict__ block_mapping,
                                                                   int src_num_blocks, int dst_num_blocks,
                                                                   int64_t block_vecs, int32_t* debug_err) {
  const int pair = blockIdx.x;
  const int layer = blockIdx.y;
  const int kv = blockIdx.z;
  const int64_t src = block_mapping[2 * pair];
  const int64_t dst = block_mapping[2 * pair + 1];
  if (src < 0 || src >= src_num_blocks || dst < 0 || dst >= dst_num_blocks) {
    if (threadIdx.x == 0 && layer == 0 && kv == 0) flag_error(debug_err, PA_DEVERR_BLOCK_RANGE);
    return;
  }
  const uint4* s = static_cast<const uint4*>(pools.src[kv][layer]) + src * block_vecs;
  uint4* d = static_cast<uint4*>(pools.dst[kv][layer]) + dst * block_vecs;
  constexpr int kStep = kSwapThreads * kSwapUnroll;
  int64_t i = threadIdx.x;
  for (; i + (kSwapUnroll - 1) * kSwapThreads < block_vecs; i += kStep) {
    uint4 v[kSwapUnroll];
#pragma unroll
    for (int u = 0; u < kSwapUnroll; ++u) v[u] = __ldcs(s + i + u * kSwapThreads);
#pragma unroll
    for (int u = 0; u < kSwapUnroll; ++u) __stcs(d + i + u * kSwapThreads, v[u]);
  }
  for (; i < block_vecs; i += kSwapThreads) __stcs(d + i, __ldcs(s + i));
}

}  // namespace

cudaError_t launch_reshape_and_cache(const void* key, const void* value, void* k_cache,
                                     void* v_cache, const int64_t* slot_mapping, int num_tokens,
                                     int num_kv_heads, int head_dim, int block_size, int num_blocks,
                                     pa_dtype src_dtype, pa_dtype kv_dtype, const float* k_scale,
                                     const float* v_scale, int32_t* debug_err, cudaStream_t stream) {
  if (num_tokens == 0) return cudaSuccess;
  const int chunks = num_kv_heads * head_dim / 8;
  const int threads = chunks >= 256 ? 256 : ((chunks + 31) / 32) * 32;
  dim3 grid(num_tokens);
#define PA_RC(ST, CT)                                                                        \
  reshape_and_cache_kernel<ST, CT><<<grid, threads, 0, stream>>>(                            \
      static_cast<const ST*>(key), static_cast<const ST*>(value), static_cast<CT*>(k_cache), \
      static_cast<CT*>(v_cache), slot_mapping, num_kv_heads, head_dim, block_size,           \
      num_blocks, k_scale, v_scale, debug_err)
  if (kv_dtype == PA_F16) {
    PA_RC(f16, f16);
  } else if (kv_dtype == PA_BF16) {
    PA_RC(bf16, bf16);
  } else if (src_dtype == PA_F16) {
    PA_RC(f16, fp8);
  } else {
    PA_RC(bf16, fp8);
  }
#undef PA_RC
  cudaError_t err = cudaGetLastError();
  if (err == cudaSuccess) note_launches(1);
  return err;
}

cudaError_t launch_copy_blocks(void* const* k_caches, void* const* v_caches, int num_layers,
                               const int64_t* block_mapping, int num_pairs, int num_blocks,
                               size_t block_bytes, int32_t* debug_err, cudaStream_t stream) {
  if (num_pairs == 0 || num_layers == 0) return cudaSuccess;
  dim3 grid(num_pairs, num_layers, 2);
  copy_blocks_kernel<<<grid, 256, 0, stream>>>(k_caches, v_caches, block_mapping, num_blocks,
                                               static_cast<int64_t>(block_bytes / 16), debug_err);
  cudaError_t err = cudaGetLastError();
  if (err == cudaSuccess) note_launches(1);
  return err;
}

cudaError_t launch_swap_blocks(const SwapPools& pools, int num_layers, const int64_t* block_mapping,
                               int num_pairs, int src_num_blocks, int dst_num_blocks,
                               size_t block_bytes, int32_t* debug_err, cudaStream_t stream) {
  if (num_pairs == 0 || num_layers == 0) return cudaSuccess;
  dim3 grid(num_pairs, num_layers, 2);
  swap_blocks_kernel<<<grid, kSwapThreads, 0, stream>>>(pools, block_mapping, src_num_blocks,
                                                        dst_num_blocks,
                                                        static_cast<int64_t>(block_bytes / 16), debug_err);
  cudaError_t err = cudaGetLastError();
  if (err == cudaSuccess) note_launches(1);
  return err;
}

}  // namespace pa
