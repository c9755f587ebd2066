// pa_decode_split_noalloc: the split-context decode for callers that cannot
// allocate device memory.
//
// pa_decode's split path keeps its per-partition partial results in a
// workspace the caller allocates. Some callers have no allocator to ask: a
// plugin inside a host framework that owns every device allocation and hands
// its plugins none, or a runtime whose device memory is fixed at start-up
// (real-time and certified deployments forbid allocating afterwards). This
// entry point serves them with a scratch array
// that lives in the library itself: a file-scope __device__ array of fixed
// size, created when the library's module is loaded on a GPU and held by
// every GPU that loads the library until the process exits. No call here
// allocates or frees anything.
//
// The host cannot use the array's name as a device address (in host code it
// names a host-side stand-in). The first call on each device therefore looks
// up the device address with cudaGetSymbolAddress, with that device current,
// and remembers it; later calls on that device reuse it.
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace {

// 16 MiB, 256-byte aligned: enough for the split partials of, e.g., 64
// sequences x 32 heads x 8 partitions x head dim 128 (8.5 MB).
constexpr size_t kScratchBytes = size_t(16) << 20;
__device__ __align__(256) unsigned char g_decode_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mutex;
void* g_scratch_ptr[kMaxDevices] = {};

pa_status scratch_for_current_device(void** ptr, const char** why) {
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) {
    *why = cudaGetErrorString(err);
    return PA_ERR_CUDA;
  }
  if (dev < 0 || dev >= kMaxDevices) {
    *why = "device ordinal beyond the library's table";
    return PA_ERR_UNSUPPORTED;
  }
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    err = cudaGetSymbolAddress(&p, g_decode_scratch);
    if (err != cudaSuccess) {
      *why = cudaGetErrorString(err);
      return PA_ERR_CUDA;
    }
    g_scratch_ptr[dev] = p;
  }
  *ptr = g_scratch_ptr[dev];
  return PA_OK;
}

}  // namespace

extern "C" {

pa_status pa_decode_split_noalloc(void* out, const void* q, const void* k_cache,
                                  const void* v_cache, const int32_t* block_tables,
                                  int32_t max_blocks_per_seq, const int32_t* context_lens,
                                  int32_t num_seqs, int32_t num_heads, int32_t num_kv_heads,
                                  int32_t head_dim, int32_t block_size, int32_t num_blocks,
                                  float scale, pa_dtype q_dtype, pa_dtype kv_dtype,
                                  const float* k_scale, const float* v_scale,
                                  int32_t max_context_len, int32_t partition_size,
                                  int32_t* debug_err, cudaStream_t stream) {
  if (partition_size < 0) {
    pa::set_last_error("partition_size < 0");
    return PA_ERR_INVALID;
  }
  if (partition_size == 0) partition_size = 512;
  // the arguments first, so a bad one is reported as such and not as a size
  const pa_status v = pa::validate_decode_args(
      out, q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens, num_seqs,
      num_heads, num_kv_heads, head_dim, block_size, num_blocks, scale, q_dtype, kv_dtype,
      k_scale, v_scale, max_context_len, partition_size);
  if (v != PA_OK || num_seqs == 0) return v;
  const size_t need = pa_decode_workspace_size(num_seqs, num_heads, num_kv_heads, head_dim,
                                               max_context_len, partition_size);
  if (need > kScratchBytes) {
    pa::set_last_error("pa_decode_split_noalloc needs %zu scratch bytes for these sizes; its "
                       "built-in scratch holds %zu",
                       need, kScratchBytes);
    return PA_ERR_WORKSPACE;
  }
  void* scratch = nullptr;
  if (num_seqs > 0) {
    const char* why = "";
    pa_status s = scratch_for_current_device(&scratch, &why);
    if (s != PA_OK) {
      pa::set_last_error("pa_decode_split_noalloc scratch set-up: %s", why);
      return s;
    }
  }
  // Every partial slot the reduce reads is written by the partition kernel of
  // the same call, so nothing in the scratch needs clearing between calls.
  return pa_decode(out, q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens,
                   num_seqs, num_heads, num_kv_heads, head_dim, block_size, num_blocks, scale,
                   q_dtype, kv_dtype, k_scale, v_scale, max_context_len, partition_size, scratch,
                   kScratchBytes, debug_err, stream);
}

}  // extern "C"
