// Launchers shared between the translation units of the library. These are
// C++ (namespace pa); the C-ABI lives in pa_api.cu.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

#include "pa.h"

namespace pa {

struct DecodeParams;
struct PrefixGroups;

// Adds n to the process-wide count of kernels launched by this library.
void note_launches(int n);

// Raises the dynamic shared memory limit of kernel `fn` to `bytes` on the
// current device, once per device (a function attribute is per device);
// `done` holds one bit per device already set.
inline cudaError_t set_smem_limit_once(const void* fn, int bytes, std::atomic<unsigned long long>& done) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned long long bit = (dev >= 0 && dev < 64) ? (1ull << dev) : 0ull;
  if (bit != 0 && (done.load(std::memory_order_relaxed) & bit) != 0) return cudaSuccess;
  e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && bit != 0) done.fetch_or(bit, std::memory_order_relaxed);
  return e;
}

// 3-D TMA view of a cache [blocks, KV heads, block_size, head_dim] as (d, token
// in block, block x KV head), boxes of 128 bytes x min(block_size,
// tile_tokens) rows x heads_per_box adjacent KV heads, 128-byte swizzle
// (decode_tc.cu).
bool make_cache_map(CUtensorMap* map, const void* base, int head_dim, int elem, int block_size,
                    int tile_tokens, int64_t blocks_x_heads, int heads_per_box = 1);

// Sets the message pa_last_error_message() returns on this thread.
void set_last_error(const char* fmt, ...);

// Host-side checks of pa_decode's arguments other than the workspace:
// PA_OK, or the status pa_decode returns for them (message set).
pa_status validate_decode_args(const void* out, const void* q, const void* k_cache,
                               const void* v_cache, const int32_t* block_tables,
                               int32_t max_blocks_per_seq, const int32_t* context_lens,
                               int32_t num_seqs, int32_t num_heads, int32_t num_kv_heads,
                               int32_t head_dim, int32_t block_size, int32_t num_blocks,
                               float scale, pa_dtype q_dtype, pa_dtype kv_dtype,
                               const float* k_scale, const float* v_scale,
                               int32_t max_context_len, int32_t partition_size);

cudaError_t launch_reshape_and_cache(const void* key, const void* value, void* k_cache,
                                     void* v_cache, const int64_t* slot_mapping, int num_tokens,
                                     int num_kv_heads, int head_dim, int block_size, int num_blocks,
                                     pa_dtype src_dtype, pa_dtype kv_dtype, const float* k_scale,
                                     const float* v_scale, int32_t* debug_err, cudaStream_t stream);

cudaError_t launch_copy_blocks(void* const* k_caches, void* const* v_caches, int num_layers,
                               const int64_t* block_mapping, int num_pairs, int num_blocks,
                               size_t block_bytes, int32_t* debug_err, cudaStream_t stream);

// Paged prefill on tcgen05 (prefill_tc.cu).
bool prefill_supported(int group, int head_dim, pa_dtype dtype, int block_size);
cudaError_t launch_prefill_tc(void* out, const void* q, const void* k_cache, const void* v_cache,
                              const int32_t* block_tables, int max_blocks_per_seq,
                              const int32_t* context_lens, const int32_t* query_start, int num_seqs,
                              int num_tokens, int max_query_len, int num_heads, int num_kv_heads,
                              int block_size, int num_blocks, float scale, pa_dtype dtype,
                              int32_t* debug_err, cudaStream_t stream);

// Per-layer pool pointers of one swap, all device-accessible.
struct SwapPools {
  const void* src[2][PA_SWAP_MAX_LAYERS];  // [K, V][layer]
  void* dst[2][PA_SWAP_MAX_LAYERS];
};
cudaError_t launch_swap_blocks(const SwapPools& pools, int num_layers, const int64_t* block_mapping,
                               int num_pairs, int src_num_blocks, int dst_num_blocks,
                               size_t block_bytes, int32_t* debug_err, cudaStream_t stream);

// CUDA-core decode: grid (num_partitions, num_kv_heads, num_seqs), plus the
// partition reduce when num_partitions > 1.
cudaError_t launch_decode_simt(const DecodeParams& p, int head_dim, pa_dtype q_dtype,
                               pa_dtype kv_dtype, cudaStream_t stream);

// Merge of the split path's per-partition partials into the output rows;
// with pdl the launch may overlap the tail of the kernel before it.
cudaError_t launch_reduce_partitions(const DecodeParams& p, int head_dim, pa_dtype q_dtype,
                                     bool pdl, cudaStream_t stream);

// Tensor-core decode (GQA groups of 2/4/8). partition_size = 0: balanced schedule
// over all warps of the GPU with partial states merged by a second kernel
// (workspace of tc_auto_workspace_bytes); partition_size > 0: split path
// with partitions of that many tokens into p.ws_acc / p.ws_ml.
constexpr int kTcMaxSeqs = 2048;
bool tc_supported(int group, int head_dim, pa_dtype kv_dtype, int num_seqs, int partition_size);
size_t tc_auto_workspace_bytes(int num_seqs, int head_dim, int group, int num_sms);
cudaError_t launch_decode_tc(const DecodeParams& p, int head_dim, pa_dtype q_dtype,
                             pa_dtype kv_dtype, int partition_size, void* workspace, int num_sms,
                             cudaStream_t stream, const PrefixGroups* groups = nullptr);

// Shared-prefix attention (decode_prefix.cu): one CTA per (64 rows of a
// group's members x query heads, KV unit, group x chunk of the prefix),
// launched before the decode grid of the call; partial states go to
// groups.ws_prefix.
int prefix_row_tiles(int max_group_size, int group);
int prefix_max_chunk_len(int block_size);
int prefix_chunk_step(int block_size);
cudaError_t launch_prefix_attn(const DecodeParams& p, const PrefixGroups& groups, int head_dim,
                               pa_dtype dtype, cudaStream_t stream);

}  // namespace pa
