// The C ABI of the library: argument checks, schedule choice, launches.
#include <atomic>
#include <cmath>
#include <cstdio>
#include <cstdarg>
#include <string>

#include "common.cuh"
#include "internal.h"

namespace {

thread_local std::string g_last_error;
std::atomic<uint64_t> g_launches{0};

pa_status fail(pa_status s, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return s;
}

pa_status from_cuda(cudaError_t err, const char* what) {
  if (err == cudaSuccess) return PA_OK;
  return fail(PA_ERR_CUDA, "%s: %s", what, cudaGetErrorString(err));
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool is_16bit(pa_dtype t) { return t == PA_F16 || t == PA_BF16; }
bool valid_dtype(pa_dtype t) { return t == PA_F16 || t == PA_BF16 || t == PA_FP8_E4M3; }
bool supported_block_size(int bs) { return bs == 8 || bs == 16 || bs == 32 || bs == 64; }
// Query heads per KV head: 1, 2, 4, 8, or a multiple of 8 (up to MQA, where
// every query head shares one KV head). Groups above 8 are run as KV units of
// 8 query heads that read the same KV head.
bool supported_group(int g) { return g == 1 || g == 2 || g == 4 || (g >= 8 && g % 8 == 0); }
constexpr int kUnitHeads = 8;
int unit_group(int g) { return g > kUnitHeads ? kUnitHeads : g; }
bool supported_head_dim(int d) { return d == 64 || d == 128 || d == 256; }

constexpr int kAutoPartition = 512;

int num_partitions_for(int max_context_len, int partition_size) {
  return max_context_len <= 0 ? 1 : (max_context_len + partition_size - 1) / partition_size;
}

size_t split_workspace_bytes(int num_seqs, int num_heads, int head_dim, int nparts) {
  const size_t slots = static_cast<size_t>(num_seqs) * num_heads * nparts;
  const size_t acc = ((slots * head_dim * sizeof(float)) + 255) / 256 * 256;
  const size_t ml = ((slots * 2 * sizeof(float)) + 255) / 256 * 256;
  return acc + ml;
}

// The split schedule the library picks by itself, or 0 for a single pass.
int auto_partition(int max_context_len) {
  return max_context_len > kAutoPartition ? kAutoPartition : 0;
}

int current_sm_count() {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return sms;
}

// How the shared prefixes are cut: chunks of chunk_len keys (whole key tiles
// and whole blocks), as many as fit the prefix grid into one wave of two
// CTAs per SM (more chunks mean more partial states to write and merge, and
// a second wave); num_chunks covers the longest prefix.
struct PrefixPlan {
  int chunk_len = 0;
  int num_chunks = 0;
};

PrefixPlan prefix_plan(int num_groups, int max_group_size, int max_prefix_len, int units, int group,
                       int block_size, int sms) {
  PrefixPlan pl;
  if (num_groups <= 0 || max_group_size <= 0 || max_prefix_len <= 0) return pl;
  const int64_t per_set = static_cast<int64_t>(pa::prefix_row_tiles(max_group_size, group)) * units * num_groups;
  const int64_t target = 2 * static_cast<int64_t>(sms > 0 ? sms : 1);  // CTAs resident at once
  int64_t c = target / per_set;  // one wave when the rows allow it
  const int64_t cmax = (max_prefix_len + pa::prefix_chunk_step(block_size) - 1) / pa::prefix_chunk_step(block_size);
  if (c > cmax) c = cmax;
  if (c < 1) c = 1;
  const int step = pa::prefix_chunk_step(block_size);
  int64_t len = (max_prefix_len + c - 1) / c;
  len = (len + step - 1) / step * step;
  const int64_t cap = pa::prefix_max_chunk_len(block_size) / step * step;
  if (len > cap) len = cap;
  pl.chunk_len = static_cast<int>(len);
  pl.num_chunks = static_cast<int>((max_prefix_len + len - 1) / len);
  return pl;
}

}  // namespace

namespace pa {
void note_launches(int n) { g_launches.fetch_add(static_cast<uint64_t>(n), std::memory_order_relaxed); }

void set_last_error(const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
}
}  // namespace pa

extern "C" {

uint64_t pa_kernel_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

int pa_version(void) { return 100; }

const char* pa_status_string(pa_status status) {
  switch (status) {
    case PA_OK: return "PA_OK";
    case PA_ERR_INVALID: return "PA_ERR_INVALID";
    case PA_ERR_UNSUPPORTED: return "PA_ERR_UNSUPPORTED";
    case PA_ERR_CUDA: return "PA_ERR_CUDA";
    case PA_ERR_WORKSPACE: return "PA_ERR_WORKSPACE";
  }
  return "PA_ERR_UNKNOWN";
}

const char* pa_last_error_message(void) { return g_last_error.c_str(); }

pa_status pa_reshape_and_cache(const void* key, const void* value, void* k_cache, void* v_cache,
                               const int64_t* slot_mapping, int32_t num_tokens,
                               int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                               int32_t num_blocks, pa_dtype src_dtype, pa_dtype kv_dtype,
                               const float* k_scale, const float* v_scale, int32_t* debug_err,
                               cudaStream_t stream) {
  if (num_tokens < 0) return fail(PA_ERR_INVALID, "num_tokens < 0");
  if (num_kv_heads <= 0 || head_dim <= 0 || block_size <= 0 || num_blocks <= 0)
    return fail(PA_ERR_INVALID, "sizes must be positive");
  if (head_dim % 8 != 0) return fail(PA_ERR_INVALID, "head_dim must be a multiple of 8");
  if (!valid_dtype(src_dtype) || !valid_dtype(kv_dtype)) return fail(PA_ERR_INVALID, "bad dtype");
  if (!is_16bit(src_dtype)) return fail(PA_ERR_INVALID, "sources must be f16 or bf16");
  if (is_16bit(kv_dtype) && src_dtype != kv_dtype)
    return fail(PA_ERR_INVALID, "a 16-bit cache takes sources of its own type");
  if (kv_dtype == PA_FP8_E4M3 && (k_scale == nullptr || v_scale == nullptr))
    return fail(PA_ERR_INVALID, "an 8-bit cache needs k_scale and v_scale");
  if (num_tokens == 0) return PA_OK;
  if (!key || !value || !k_cache || !v_cache || !slot_mapping)
    return fail(PA_ERR_INVALID, "null tensor pointer");
  if (!aligned16(key) || !aligned16(value) || !aligned16(k_cache) || !aligned16(v_cache))
    return fail(PA_ERR_INVALID, "tensor pointers must be 16-byte aligned");
  return from_cuda(pa::launch_reshape_and_cache(key, value, k_cache, v_cache, slot_mapping,
                                                num_tokens, num_kv_heads, head_dim, block_size,
                                                num_blocks, src_dtype, kv_dtype, k_scale, v_scale,
                                                debug_err, stream),
                   "reshape_and_cache launch");
}

size_t pa_decode_workspace_size(int32_t num_seqs, int32_t num_heads, int32_t num_kv_heads,
                                int32_t head_dim, int32_t max_context_len,
                                int32_t partition_size) {
  (void)num_kv_heads;
  if (num_seqs <= 0 || num_heads <= 0 || head_dim <= 0 || max_context_len <= 0) return 0;
  if (partition_size > 0)
    return split_workspace_bytes(num_seqs, num_heads, head_dim,
                                 num_partitions_for(max_context_len, partition_size));
  // the library's own schedule: the tensor-core schedule's partial states, or
  // the CUDA-core split path, whichever needs more
  size_t need = 0;
  const int sms = current_sm_count();
  if (sms > 0 && num_kv_heads > 0 && num_heads % num_kv_heads == 0)
    need = pa::tc_auto_workspace_bytes(num_seqs, head_dim, unit_group(num_heads / num_kv_heads), sms);
  const int part = auto_partition(max_context_len);
  if (part > 0) {
    const size_t simt = split_workspace_bytes(num_seqs, num_heads, head_dim,
                                              num_partitions_for(max_context_len, part));
    if (simt > need) need = simt;
  }
  return need;
}

}  // extern "C"

namespace pa {

// The host-side checks of pa_decode's arguments (everything but the
// workspace), shared with pa_decode_split_noalloc.
pa_status validate_decode_args(const void* out, const void* q, const void* k_cache,
                               const void* v_cache, const int32_t* block_tables,
                               int32_t max_blocks_per_seq, const int32_t* context_lens,
                               int32_t num_seqs, int32_t num_heads, int32_t num_kv_heads,
                               int32_t head_dim, int32_t block_size, int32_t num_blocks,
                               float scale, pa_dtype q_dtype, pa_dtype kv_dtype,
                               const float* k_scale, const float* v_scale,
                               int32_t max_context_len, int32_t partition_size) {
  if (num_seqs < 0) return fail(PA_ERR_INVALID, "num_seqs < 0");
  if (num_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0 || block_size <= 0 ||
      num_blocks <= 0 || max_blocks_per_seq <= 0)
    return fail(PA_ERR_INVALID, "sizes must be positive");
  if (num_heads % num_kv_heads != 0)
    return fail(PA_ERR_INVALID, "num_heads must be a multiple of num_kv_heads");
  if (head_dim % 8 != 0) return fail(PA_ERR_INVALID, "head_dim must be a multiple of 8");
  if (!valid_dtype(q_dtype) || !valid_dtype(kv_dtype)) return fail(PA_ERR_INVALID, "bad dtype");
  if (!is_16bit(q_dtype)) return fail(PA_ERR_INVALID, "q must be f16 or bf16");
  if (is_16bit(kv_dtype) && q_dtype != kv_dtype)
    return fail(PA_ERR_INVALID, "q and a 16-bit cache must have the same type");
  if (kv_dtype == PA_FP8_E4M3 && (k_scale == nullptr || v_scale == nullptr))
    return fail(PA_ERR_INVALID, "an 8-bit cache needs k_scale and v_scale");
  if (!std::isfinite(scale)) return fail(PA_ERR_INVALID, "scale must be finite");
  if (max_context_len < 0) return fail(PA_ERR_INVALID, "max_context_len < 0");
  if (static_cast<int64_t>(max_context_len) > static_cast<int64_t>(max_blocks_per_seq) * block_size)
    return fail(PA_ERR_INVALID, "max_context_len exceeds max_blocks_per_seq * block_size");
  if (partition_size < 0) return fail(PA_ERR_INVALID, "partition_size < 0");
  if (partition_size > 0 && (partition_size % 16 != 0 || partition_size % block_size != 0))
    return fail(PA_ERR_INVALID, "partition_size must be a multiple of 16 and of block_size");
  if (!supported_block_size(block_size))
    return fail(PA_ERR_UNSUPPORTED, "block_size %d not in {8,16,32,64}", block_size);
  if (!supported_group(num_heads / num_kv_heads))
    return fail(PA_ERR_UNSUPPORTED, "num_heads/num_kv_heads %d not 1, 2, 4 or a multiple of 8",
                num_heads / num_kv_heads);
  if (!supported_head_dim(head_dim))
    return fail(PA_ERR_UNSUPPORTED, "head_dim %d not in {64,128,256}", head_dim);
  if (num_seqs > 65535) return fail(PA_ERR_UNSUPPORTED, "more than 65535 sequences");
  if (num_seqs == 0) return PA_OK;
  if (!out || !q || !k_cache || !v_cache || !block_tables || !context_lens)
    return fail(PA_ERR_INVALID, "null tensor pointer");
  if (!aligned16(out) || !aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache))
    return fail(PA_ERR_INVALID, "tensor pointers must be 16-byte aligned");
  return PA_OK;
}

}  // namespace pa

extern "C" {

pa_status pa_decode(void* out, const void* q, const void* k_cache, const void* v_cache,
                    const int32_t* block_tables, int32_t max_blocks_per_seq,
                    const int32_t* context_lens, int32_t num_seqs, int32_t num_heads,
                    int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                    int32_t num_blocks, float scale, pa_dtype q_dtype, pa_dtype kv_dtype,
                    const float* k_scale, const float* v_scale, int32_t max_context_len,
                    int32_t partition_size, void* workspace, size_t workspace_bytes,
                    int32_t* debug_err, cudaStream_t stream) {
  const pa_status v = pa::validate_decode_args(
      out, q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens, num_seqs,
      num_heads, num_kv_heads, head_dim, block_size, num_blocks, scale, q_dtype, kv_dtype,
      k_scale, v_scale, max_context_len, partition_size);
  if (v != PA_OK || num_seqs == 0) return v;
  if (workspace != nullptr && (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
    return fail(PA_ERR_INVALID, "workspace must be 256-byte aligned");

  pa::DecodeParams p{};
  p.out = out;
  p.q = q;
  p.k_cache = k_cache;
  p.v_cache = v_cache;
  p.block_tables = block_tables;
  p.context_lens = context_lens;
  p.k_scale = k_scale;
  p.v_scale = v_scale;
  p.debug_err = debug_err;
  p.max_blocks_per_seq = max_blocks_per_seq;
  p.num_seqs = num_seqs;
  p.num_heads = num_heads;
  // groups above 8 query heads: KV units of 8 query heads each, several per KV head
  const int group = unit_group(num_heads / num_kv_heads);
  p.kv_div = (num_heads / num_kv_heads) / group;
  p.kv_heads_phys = num_kv_heads;
  p.num_kv_heads = num_kv_heads * p.kv_div;
  p.block_size = block_size;
  p.num_blocks = num_blocks;
  p.max_context_len = max_context_len;
  p.scale_log2 = scale * pa::kLog2e;

  const bool tc = pa::tc_supported(group, head_dim, kv_dtype, num_seqs, partition_size > 0 ? partition_size : 0);
  if (partition_size > 0) {
    const int nparts = num_partitions_for(max_context_len, partition_size);
    const size_t need = split_workspace_bytes(num_seqs, num_heads, head_dim, nparts);
    if (workspace == nullptr || workspace_bytes < need)
      return fail(PA_ERR_WORKSPACE, "split decode needs %zu workspace bytes, got %zu", need,
                  workspace_bytes);
  }
  // every argument is checked: from here on the device is queried and used
  const int sms = current_sm_count();
  if (sms <= 0) return fail(PA_ERR_CUDA, "no current CUDA device");

  if (partition_size > 0) {
    const int nparts = num_partitions_for(max_context_len, partition_size);
    p.partition_size = partition_size;
    p.num_partitions = nparts;
    const size_t slots = static_cast<size_t>(num_seqs) * num_heads * nparts;
    p.ws_acc = static_cast<float*>(workspace);
    p.ws_ml = reinterpret_cast<float*>(static_cast<char*>(workspace) +
                                       ((slots * head_dim * sizeof(float)) + 255) / 256 * 256);
    if (tc)
      return from_cuda(pa::launch_decode_tc(p, head_dim, q_dtype, kv_dtype, partition_size,
                                            nullptr, sms, stream),
                       "decode launch");
    return from_cuda(pa::launch_decode_simt(p, head_dim, q_dtype, kv_dtype, stream),
                     "decode launch");
  }

  if (tc && workspace != nullptr &&
      workspace_bytes >= pa::tc_auto_workspace_bytes(num_seqs, head_dim, group, sms)) {
    p.partition_size = 0;
    p.num_partitions = 1;
    return from_cuda(pa::launch_decode_tc(p, head_dim, q_dtype, kv_dtype, 0, workspace, sms, stream),
                     "decode launch");
  }
  int part = auto_partition(max_context_len);
  if (part > 0) {
    const size_t need = split_workspace_bytes(num_seqs, num_heads, head_dim,
                                              num_partitions_for(max_context_len, part));
    if (workspace == nullptr || workspace_bytes < need) part = 0;
  }
  if (part > 0) {
    p.partition_size = part;
    p.num_partitions = num_partitions_for(max_context_len, part);
    const size_t slots = static_cast<size_t>(num_seqs) * num_heads * p.num_partitions;
    p.ws_acc = static_cast<float*>(workspace);
    p.ws_ml = reinterpret_cast<float*>(static_cast<char*>(workspace) +
                                       ((slots * head_dim * sizeof(float)) + 255) / 256 * 256);
  } else {
    // one pass over the whole sequence
    p.partition_size = max_context_len > 0 ? ((max_context_len + block_size - 1) / block_size) * block_size
                                           : block_size;
    p.num_partitions = 1;
  }
  return from_cuda(pa::launch_decode_simt(p, head_dim, q_dtype, kv_dtype, stream),
                   "decode launch");
}

size_t pa_decode_shared_prefix_workspace_size(int32_t num_seqs, int32_t num_heads,
                                              int32_t num_kv_heads, int32_t head_dim,
                                              int32_t block_size, int32_t num_groups,
                                              int32_t max_group_size, int32_t max_prefix_len) {
  if (num_seqs <= 0 || num_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0 || block_size <= 0 ||
      num_heads % num_kv_heads != 0)
    return 0;
  const int sms = current_sm_count();
  if (sms <= 0) return 0;
  const int group = unit_group(num_heads / num_kv_heads);
  const int units = num_heads / group;
  const size_t dec = pa::tc_auto_workspace_bytes(num_seqs, head_dim, group, sms);
  const PrefixPlan pl = prefix_plan(num_groups, max_group_size, max_prefix_len, units, group, block_size, sms);
  // a state per (sequence, unit, chunk) of the shared prefixes, and one per
  // (sequence, unit) for suffixes that one warp holds whole
  const size_t pre = static_cast<size_t>(num_seqs) * units * (pl.num_chunks + 1) *
                     pa::state_floats(group, head_dim) * sizeof(float);
  return dec + pre;
}

pa_status pa_decode_shared_prefix(void* out, const void* q, const void* k_cache, const void* v_cache,
                                  const int32_t* block_tables, int32_t max_blocks_per_seq,
                                  const int32_t* context_lens, int32_t num_seqs, int32_t num_heads,
                                  int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                                  int32_t num_blocks, float scale, pa_dtype dtype,
                                  int32_t max_context_len, const int32_t* group_start,
                                  const int32_t* group_prefix, int32_t num_groups,
                                  int32_t max_group_size, int32_t max_prefix_len, void* workspace,
                                  size_t workspace_bytes, int32_t* debug_err, cudaStream_t stream) {
  const pa_status v = pa::validate_decode_args(
      out, q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens, num_seqs, num_heads,
      num_kv_heads, head_dim, block_size, num_blocks, scale, dtype, dtype, nullptr, nullptr,
      max_context_len, 0);
  if (v != PA_OK) return v;
  if (!is_16bit(dtype)) return fail(PA_ERR_UNSUPPORTED, "shared-prefix decode takes f16 or bf16 caches");
  if (num_groups < 0 || max_group_size < 0 || max_prefix_len < 0)
    return fail(PA_ERR_INVALID, "negative group count or bound");
  if (num_groups > 0 && (group_start == nullptr || group_prefix == nullptr))
    return fail(PA_ERR_INVALID, "null group arrays");
  const int group = unit_group(num_heads / num_kv_heads);
  if (head_dim == 256 || num_seqs > pa::kTcMaxSeqs)
    return fail(PA_ERR_UNSUPPORTED, "shared-prefix decode takes head_dim 64 or 128 and at most %d sequences",
                pa::kTcMaxSeqs);
  if (num_seqs == 0) return PA_OK;
  if (workspace == nullptr || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
    return fail(PA_ERR_INVALID, "workspace must be a 256-byte aligned device buffer");
  const size_t need = pa_decode_shared_prefix_workspace_size(
      num_seqs, num_heads, num_kv_heads, head_dim, block_size, num_groups, max_group_size, max_prefix_len);
  if (need == 0) return fail(PA_ERR_CUDA, "no current CUDA device");
  if (workspace_bytes < need)
    return fail(PA_ERR_WORKSPACE, "shared-prefix decode needs %zu workspace bytes, got %zu", need,
                workspace_bytes);
  const int sms = current_sm_count();
  pa::DecodeParams p{};
  p.out = out;
  p.q = q;
  p.k_cache = k_cache;
  p.v_cache = v_cache;
  p.block_tables = block_tables;
  p.context_lens = context_lens;
  p.debug_err = debug_err;
  p.max_blocks_per_seq = max_blocks_per_seq;
  p.num_seqs = num_seqs;
  p.num_heads = num_heads;
  p.kv_div = (num_heads / num_kv_heads) / group;
  p.kv_heads_phys = num_kv_heads;
  p.num_kv_heads = num_kv_heads * p.kv_div;
  p.block_size = block_size;
  p.num_blocks = num_blocks;
  p.max_context_len = max_context_len;
  p.scale_log2 = scale * pa::kLog2e;
  p.partition_size = 0;
  p.num_partitions = 1;
  const PrefixPlan pl = prefix_plan(num_groups, max_group_size, max_prefix_len, p.num_kv_heads, group,
                                    block_size, sms);
  if (pl.num_chunks == 0)  // nothing shared: the library's own schedule
    return from_cuda(pa::launch_decode_tc(p, head_dim, dtype, dtype, 0, workspace, sms, stream),
                     "decode launch");
  if (static_cast<int64_t>(num_groups) * pl.num_chunks > 65535 ||
      pa::prefix_row_tiles(max_group_size, group) > 65535)
    return fail(PA_ERR_UNSUPPORTED, "too many groups or members for one prefix grid");
  pa::PrefixGroups pg{};
  pg.group_start = group_start;
  pg.group_prefix = group_prefix;
  pg.num_groups = num_groups;
  pg.max_group_size = max_group_size;
  pg.max_prefix_len = max_prefix_len;
  pg.chunk_len = pl.chunk_len;
  pg.num_chunks = pl.num_chunks;
  return from_cuda(pa::launch_decode_tc(p, head_dim, dtype, dtype, 0, workspace, sms, stream, &pg),
                   "shared-prefix decode launch");
}

pa_status pa_copy_blocks(void* const* k_caches, void* const* v_caches, int32_t num_layers,
                         const int64_t* block_mapping, int32_t num_pairs, int32_t num_blocks,
                         size_t block_bytes, int32_t* debug_err, cudaStream_t stream) {
  if (num_layers < 0 || num_pairs < 0) return fail(PA_ERR_INVALID, "negative count");
  if (num_blocks <= 0) return fail(PA_ERR_INVALID, "num_blocks must be positive");
  if (block_bytes == 0 || block_bytes % 16 != 0)
    return fail(PA_ERR_INVALID, "block_bytes must be a positive multiple of 16");
  if (num_layers == 0 || num_pairs == 0) return PA_OK;
  if (num_layers > 65535) return fail(PA_ERR_UNSUPPORTED, "more than 65535 layers");
  if (!k_caches || !v_caches || !block_mapping) return fail(PA_ERR_INVALID, "null pointer");
  return from_cuda(pa::launch_copy_blocks(k_caches, v_caches, num_layers, block_mapping,
                                          num_pairs, num_blocks, block_bytes, debug_err, stream),
                   "copy_blocks launch");
}

pa_status pa_prefill(void* out, const void* q, const void* k_cache, const void* v_cache,
                     const int32_t* block_tables, int32_t max_blocks_per_seq,
                     const int32_t* context_lens, const int32_t* query_start, int32_t num_seqs,
                     int32_t num_tokens, int32_t max_query_len, int32_t num_heads,
                     int32_t num_kv_heads, int32_t head_dim, int32_t block_size, int32_t num_blocks,
                     float scale, pa_dtype dtype, int32_t* debug_err, cudaStream_t stream) {
  if (num_seqs < 0 || num_tokens < 0 || max_query_len < 0) return fail(PA_ERR_INVALID, "negative count");
  if (num_heads <= 0 || num_kv_heads <= 0 || num_heads % num_kv_heads != 0)
    return fail(PA_ERR_INVALID, "num_heads must be a positive multiple of num_kv_heads");
  if (block_size != 8 && block_size != 16 && block_size != 32 && block_size != 64)
    return fail(PA_ERR_UNSUPPORTED, "block_size %d not in {8, 16, 32, 64}", block_size);
  if (num_blocks <= 0 || max_blocks_per_seq <= 0) return fail(PA_ERR_INVALID, "empty pool or table");
  if (dtype != PA_F16 && dtype != PA_BF16) return fail(PA_ERR_UNSUPPORTED, "prefill takes f16 or bf16");
  if (!pa::prefill_supported(num_heads / num_kv_heads, head_dim, dtype, block_size))
    return fail(PA_ERR_UNSUPPORTED, "prefill supports head_dim 128 and groups 1, 2, 4, 8");
  if (num_seqs == 0 || num_tokens == 0 || max_query_len == 0) return PA_OK;
  if (!out || !q || !k_cache || !v_cache || !block_tables || !context_lens || !query_start)
    return fail(PA_ERR_INVALID, "null pointer");
  if (reinterpret_cast<uintptr_t>(q) % 16 || reinterpret_cast<uintptr_t>(out) % 16 ||
      reinterpret_cast<uintptr_t>(k_cache) % 16 || reinterpret_cast<uintptr_t>(v_cache) % 16)
    return fail(PA_ERR_INVALID, "q, out and the caches must be 16-byte aligned");
  if (num_seqs > 65535) return fail(PA_ERR_UNSUPPORTED, "more than 65535 sequences");
  return from_cuda(pa::launch_prefill_tc(out, q, k_cache, v_cache, block_tables, max_blocks_per_seq,
                                         context_lens, query_start, num_seqs, num_tokens, max_query_len,
                                         num_heads, num_kv_heads, block_size, num_blocks, scale, dtype,
                                         debug_err, stream),
                   "prefill launch");
}

// The device-side address of `p` when the device can read and write it (device
// or managed memory, or pinned host memory mapped into the device's address
// space), else nullptr.
static const void* device_accessible(const void* p) {
  cudaPointerAttributes at{};
  if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
    cudaGetLastError();  // clear the sticky-free error of an unknown pointer
    return nullptr;
  }
  switch (at.type) {
    case cudaMemoryTypeDevice:
    case cudaMemoryTypeManaged:
      return p;
    case cudaMemoryTypeHost:
      return at.devicePointer;
    default:
      return nullptr;
  }
}

pa_status pa_swap_blocks(void* const* dst_k, void* const* dst_v, const void* const* src_k,
                         const void* const* src_v, int32_t num_layers,
                         const int64_t* block_mapping, int32_t num_pairs, int32_t src_num_blocks,
                         int32_t dst_num_blocks, size_t block_bytes, int32_t* debug_err,
                         cudaStream_t stream) {
  if (num_layers < 0 || num_pairs < 0) return fail(PA_ERR_INVALID, "negative count");
  if (num_layers > PA_SWAP_MAX_LAYERS)
    return fail(PA_ERR_UNSUPPORTED, "more than %d layers in one swap", PA_SWAP_MAX_LAYERS);
  if (src_num_blocks <= 0 || dst_num_blocks <= 0)
    return fail(PA_ERR_INVALID, "pool sizes must be positive");
  if (block_bytes == 0 || block_bytes % 16 != 0)
    return fail(PA_ERR_INVALID, "block_bytes must be a positive multiple of 16");
  if (num_layers == 0 || num_pairs == 0) return PA_OK;
  if (num_pairs > 2147483647 / 2) return fail(PA_ERR_UNSUPPORTED, "too many pairs");
  if (!dst_k || !dst_v || !src_k || !src_v || !block_mapping) return fail(PA_ERR_INVALID, "null pointer");
  pa::SwapPools pools{};
  for (int l = 0; l < num_layers; ++l) {
    const void* in[4] = {src_k[l], src_v[l], dst_k[l], dst_v[l]};
    const void* dev[4];
    for (int i = 0; i < 4; ++i) {
      if (in[i] == nullptr) return fail(PA_ERR_INVALID, "null pool pointer for layer %d", l);
      if (reinterpret_cast<uintptr_t>(in[i]) % 16 != 0)
        return fail(PA_ERR_INVALID, "pool pointer of layer %d is not 16-byte aligned", l);
      dev[i] = device_accessible(in[i]);
      if (dev[i] == nullptr)
        return fail(PA_ERR_INVALID,
                    "pool pointer of layer %d is neither device memory nor mapped pinned host memory", l);
    }
    pools.src[0][l] = dev[0];
    pools.src[1][l] = dev[1];
    pools.dst[0][l] = const_cast<void*>(dev[2]);
    pools.dst[1][l] = const_cast<void*>(dev[3]);
  }
  const void* map = device_accessible(block_mapping);
  if (map == nullptr)
    return fail(PA_ERR_INVALID, "block_mapping is neither device memory nor mapped pinned host memory");
  return from_cuda(pa::launch_swap_blocks(pools, num_layers, static_cast<const int64_t*>(map), num_pairs,
                                          src_num_blocks, dst_num_blocks, block_bytes, debug_err, stream),
                   "swap_blocks launch");
}

}  // extern "C"
