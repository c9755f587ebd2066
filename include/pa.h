/*
 * pa.h - paged KV-cache attention decode for NVIDIA GB300 (sm_103a).
 *
 * The KV cache is a pool of fixed-size physical blocks. A sequence owns a
 * block table that maps its logical block index to a physical block id, so
 * its blocks need not be contiguous (serving-paged-attention, section
 * "블록으로 쪼개고 표로 잇는다"; LLM의 Paged Attention, "Paged Attention의
 * 핵심 원리" items 1-2). Decode attention reads each sequence's scattered
 * blocks through its table.
 *
 * Conventions shared by every call:
 *  - Tensor arguments are DEVICE pointers owned by the caller. The library
 *    never allocates, frees or synchronises; it launches on `stream`
 *    asynchronously and returns.
 *  - Layouts are dense, row-major, with no padding:
 *      k_cache, v_cache   [num_blocks, num_kv_heads, block_size, head_dim]
 *      q, out             [num_seqs, num_heads, head_dim]
 *      key, value (new)   [num_tokens, num_kv_heads, head_dim]
 *      block_tables       int32 [num_seqs, max_blocks_per_seq]
 *      context_lens       int32 [num_seqs]
 *      slot_mapping       int64 [num_tokens]; slot = block*block_size+offset
 *      k_scale, v_scale   float32 [num_blocks, num_kv_heads] (8-bit KV only)
 *  - Query head h reads KV head h / (num_heads / num_kv_heads) (grouped-query
 *    attention with contiguous groups).
 *  - Every call returns a pa_status. Bad shapes, types, sizes, null or
 *    misaligned pointers are rejected before anything is launched. Values
 *    held in device memory (slots, table entries, context lengths) are
 *    checked by the kernels themselves: an out-of-range value is skipped
 *    (never dereferenced) and, when `debug_err` is non-NULL, the matching
 *    PA_DEVERR_* bit is OR-ed into *debug_err. `debug_err` is a caller-owned
 *    device int32, never cleared by the library.
 *  - PA_ERR_CUDA reports a launch error from the CUDA runtime; the message
 *    of the last failure on the calling thread is pa_last_error_message().
 */
#ifndef PA_H_
#define PA_H_

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  PA_OK = 0,
  PA_ERR_INVALID = 1,     /* a host-checked argument is wrong */
  PA_ERR_UNSUPPORTED = 2, /* valid, but not a shape/type the library runs */
  PA_ERR_CUDA = 3,        /* the CUDA runtime reported an error */
  PA_ERR_WORKSPACE = 4    /* the workspace given is too small */
} pa_status;

typedef enum {
  PA_F16 = 0,
  PA_BF16 = 1,
  PA_FP8_E4M3 = 2 /* OCP OFP8 E4M3: bias 7, max 448, no infinities */
} pa_dtype;

/* Bits OR-ed into *debug_err by the kernels. */
#define PA_DEVERR_SLOT_RANGE 0x1    /* slot >= num_blocks * block_size */
#define PA_DEVERR_BLOCK_RANGE 0x2   /* table entry or copy pair outside [0, num_blocks) */
#define PA_DEVERR_CONTEXT_RANGE 0x4 /* context length above max_context_len or the table width */
#define PA_DEVERR_TIMEOUT 0x8       /* a kernel gave up waiting for its own data copies (1 s) */
#define PA_DEVERR_LAYOUT 0x10       /* a kernel found its shared memory misaligned; nothing computed */
#define PA_DEVERR_QUERY_START 0x20  /* pa_prefill: query_start outside [0, num_tokens] or decreasing; clamped */
#define PA_DEVERR_Q_RANGE 0x40      /* pa_decode, 8-bit KV: a q value beyond the f16 range (|q| > 65504) */
#define PA_DEVERR_PREFIX 0x80       /* pa_decode_shared_prefix: a group description was clamped, or a
                                       member's table differs from its group's in the shared blocks */

/* Library version, major*10000 + minor*100 + patch. */
int pa_version(void);

/* Human-readable name of a status code (static storage). */
const char* pa_status_string(pa_status status);

/* Detail of the last failed call on this thread ("" if none). */
const char* pa_last_error_message(void);

/* Number of kernels this library has launched in this process (all threads). */
uint64_t pa_kernel_launch_count(void);

/*
 * pa_reshape_and_cache - write new tokens' K and V into their cache slots.
 *
 * For token t with s = slot_mapping[t] >= 0: block = s / block_size, offset
 * = s % block_size, and for every KV head h the row key[t, h, :] goes to
 * k_cache[block, h, offset, :] (value[t, h, :] to v_cache likewise). A slot
 * of -1 is a padding token and is skipped. This is the token-to-slot table
 * of vLLM의 핵심 이해: PagedAttention, section 6, applied to the block pool
 * of serving-paged-attention, "블록으로 쪼개고 표로 잇는다".
 *
 * src_dtype must equal kv_dtype for 16-bit caches, which receive the source
 * bits unchanged. For kv_dtype == PA_FP8_E4M3 (serving-paged-attention,
 * "실무에서 만지는 지점": an 8-bit KV cache) the sources are f16 or bf16 and
 * each stored code is e4m3(float(x) / scale[block, h]) with an IEEE float32
 * division and round-to-nearest-even conversion that saturates at +-448.
 * k_scale / v_scale are read only (NULL for 16-bit caches). head_dim must be
 * a multiple of 8; every tensor pointer must be 16-byte aligned.
 * Out-of-range slots set PA_DEVERR_SLOT_RANGE and are skipped.
 */
pa_status pa_reshape_and_cache(const void* key, const void* value, void* k_cache,
                               void* v_cache, const int64_t* slot_mapping,
                               int32_t num_tokens, int32_t num_kv_heads,
                               int32_t head_dim, int32_t block_size,
                               int32_t num_blocks, pa_dtype src_dtype,
                               pa_dtype kv_dtype, const float* k_scale,
                               const float* v_scale, int32_t* debug_err,
                               cudaStream_t stream);

/*
 * pa_decode - single-query attention of every sequence over its paged KV.
 *
 * For sequence i with L = context_lens[i] and query head h, with g = h / G:
 *   K, V = rows 0..L-1 of the sequence, gathered through block_tables[i]
 *          (logical block j lives in physical block block_tables[i, j];
 *          serving-paged-attention, "블록으로 쪼개고 표로 잇는다")
 *   out[i, h, :] = softmax(scale * K q[i, h]) V
 * computed with the online softmax (running max, running sum, rescaled
 * accumulator) of LLM 추론 확장, 품질·비용 절충 필수, in float32. Entries of a
 * table past ceil(L / block_size) and the unused tail of the last block are
 * never read as data. L == 0 gives an all-zero output row.
 *
 * Types: q_dtype == kv_dtype for 16-bit caches; with kv_dtype ==
 * PA_FP8_E4M3, q is f16 or bf16 and k_scale / v_scale give the per-(block,
 * KV head) dequantisation factors. out has q's type.
 *
 * max_context_len is a host-known upper bound on every context_lens[i]
 * (larger lengths are clamped to it and flag PA_DEVERR_CONTEXT_RANGE).
 * partition_size = 0 lets the library schedule the work; > 0 forces the
 * split-context path: partitions of that many tokens are attended
 * separately into float32 partials in `workspace`, then merged by a reduce
 * kernel (it must be a multiple of 16 and of block_size). The workspace is
 * caller-owned device memory of at least pa_decode_workspace_size() bytes,
 * 256-byte aligned; with partition_size = 0 and a smaller or NULL workspace
 * the library uses a schedule that needs none.
 *
 * With an 8-bit cache the tensor-core path multiplies q, converted to f16,
 * with the codes widened to f16: a q value beyond the f16 range (|q| > 65504)
 * becomes infinite, which the kernel reports with PA_DEVERR_Q_RANGE.
 *
 * Calls that overlap on the GPU: a call on the tensor-core path (groups of
 * up to 8 query heads per KV unit, head_dim 64 or 128, with a workspace)
 * takes one of 256 work counters inside the library, in turn, and its last
 * kernel sets it back to zero. Calls on one stream never overlap.
 * Two calls that run at the same time on the GPU (on different streams or
 * from several threads) share a counter when they were issued a multiple of
 * 256 calls apart, and every replay of a captured graph uses the counter its
 * capture took; calls sharing a counter must not overlap (the caller
 * serialises them), or work is skipped or done twice with no error flagged.
 *
 * Supported: num_heads / num_kv_heads (the group G) 1, 2, 4, or any multiple
 * of 8, which covers MHA (G = 1), GQA and MQA (num_kv_heads = 1, G =
 * num_heads; LLM 추론 확장, 품질·비용 절충 필수, the MHA/MQA/GQA passage);
 * head_dim in {64, 128, 256}; block_size in {8, 16, 32, 64}.
 */
pa_status pa_decode(void* out, const void* q, const void* k_cache,
                    const void* v_cache, const int32_t* block_tables,
                    int32_t max_blocks_per_seq, const int32_t* context_lens,
                    int32_t num_seqs, int32_t num_heads, int32_t num_kv_heads,
                    int32_t head_dim, int32_t block_size, int32_t num_blocks,
                    float scale, pa_dtype q_dtype, pa_dtype kv_dtype,
                    const float* k_scale, const float* v_scale,
                    int32_t max_context_len, int32_t partition_size,
                    void* workspace, size_t workspace_bytes,
                    int32_t* debug_err, cudaStream_t stream);

/*
 * Bytes of workspace pa_decode needs for these sizes on the current device
 * (partition_size as passed to pa_decode; 0 = the library's own schedule).
 */
size_t pa_decode_workspace_size(int32_t num_seqs, int32_t num_heads,
                                int32_t num_kv_heads, int32_t head_dim,
                                int32_t max_context_len, int32_t partition_size);

/*
 * pa_decode_shared_prefix - pa_decode for a batch whose sequences come in
 * groups that share the leading blocks of their tables, reading each shared
 * block once per group instead of once per sequence.
 *
 * When many requests open with one prompt, their tables point at the same
 * physical blocks for it (serving-paged-attention, "공유는 표를 베끼는 일이
 * 된다": a system prompt shared by 100 requests is stored once). The result
 * is pa_decode's, out[i, h] = softmax(scale * K q[i, h]) V over each
 * sequence's whole context; only the order of the work changes. The shared
 * tokens of a group are attended for all its members at once (their query
 * rows form a dense tile for the tensor cores) into partial softmax states,
 * which are merged with the states of each member's own suffix.
 *
 * Groups: group g is sequences group_start[g] .. group_start[g+1]-1 (DEVICE
 * int32 [num_groups + 1], non-decreasing, group_start[0] = 0,
 * group_start[num_groups] = num_seqs; a sequence in no group may sit in a
 * group of its own with prefix 0). Its members share their first
 * group_prefix[g] tokens (DEVICE int32 [num_groups], a multiple of
 * block_size, at most every member's context length): the first
 * group_prefix[g] / block_size entries of their tables are equal. The shared
 * blocks are read through the table of the group's first sequence.
 * max_group_size and max_prefix_len are host-known bounds on every group's
 * size and prefix (they size the grid). Descriptions that break these rules
 * are clamped so that nothing outside the arrays is read or written, and set
 * PA_DEVERR_PREFIX in *debug_err (the results are then undefined); so does a
 * member whose table differs from its group's first in the shared blocks.
 *
 * Other arguments as for pa_decode with partition_size = 0: dtype is the
 * type of q, out and both caches (PA_F16 or PA_BF16); head_dim 64 or 128;
 * the group sizes of pa_decode; at most 2048 sequences. The workspace
 * (caller-owned device memory, 256-byte aligned) must hold
 * pa_decode_shared_prefix_workspace_size() bytes for the same sizes on the
 * current device, else PA_ERR_WORKSPACE. The calls-that-overlap rule of
 * pa_decode applies.
 */
pa_status pa_decode_shared_prefix(void* out, const void* q, const void* k_cache,
                                  const void* v_cache, const int32_t* block_tables,
                                  int32_t max_blocks_per_seq, const int32_t* context_lens,
                                  int32_t num_seqs, int32_t num_heads, int32_t num_kv_heads,
                                  int32_t head_dim, int32_t block_size, int32_t num_blocks,
                                  float scale, pa_dtype dtype, int32_t max_context_len,
                                  const int32_t* group_start, const int32_t* group_prefix,
                                  int32_t num_groups, int32_t max_group_size,
                                  int32_t max_prefix_len, void* workspace,
                                  size_t workspace_bytes, int32_t* debug_err,
                                  cudaStream_t stream);

/* Bytes of workspace pa_decode_shared_prefix needs for these sizes on the
 * current device (0 for invalid sizes or without a device). */
size_t pa_decode_shared_prefix_workspace_size(int32_t num_seqs, int32_t num_heads,
                                              int32_t num_kv_heads, int32_t head_dim,
                                              int32_t block_size, int32_t num_groups,
                                              int32_t max_group_size,
                                              int32_t max_prefix_len);

/*
 * pa_copy_blocks - copy whole physical blocks, K and V, in every layer.
 *
 * For each pair p, src = block_mapping[2p], dst = block_mapping[2p+1], and
 * each layer l: block dst of k_caches[l] and v_caches[l] becomes a byte copy
 * of block src. This is the copy of copy-on-write: a request about to write
 * into a block that other tables share gets its own copy first
 * (serving-paged-attention, "공유는 표를 베끼는 일이 된다"; LLM의 Paged
 * Attention, "Paged Attention의 핵심 원리" item 3); redirecting the table
 * entry is the caller's job.
 *
 * k_caches / v_caches are DEVICE arrays of num_layers device pointers;
 * block_mapping is a DEVICE int64 array [num_pairs, 2]. block_bytes is the
 * size of one block of one cache (num_kv_heads * block_size * head_dim *
 * element size), a multiple of 16; cache pointers must be 16-byte aligned.
 * No dst may equal a src or another dst (one src may feed many dsts).
 * Pairs outside [0, num_blocks) set PA_DEVERR_BLOCK_RANGE and are skipped.
 */
pa_status pa_copy_blocks(void* const* k_caches, void* const* v_caches,
                         int32_t num_layers, const int64_t* block_mapping,
                         int32_t num_pairs, int32_t num_blocks,
                         size_t block_bytes, int32_t* debug_err,
                         cudaStream_t stream);

/*
 * pa_prefill - causal attention of each sequence's chunk of new query tokens
 * over its paged KV cache (the prompt, or a chunk of it after earlier chunks
 * were cached: chunked prefill).
 *
 * Prefill is the many-query step before decode (LLM 추론 확장, 품질·비용 절충
 * 필수, the prefill / decode split) and reads the same block tables
 * (serving-paged-attention, "블록으로 쪼개고 표로 잇는다"). Sequence i holds
 * context_lens[i] tokens whose K/V are in the caches (write the chunk's own
 * K/V with pa_reshape_and_cache first); its queries are the last
 * n_i = query_start[i+1] - query_start[i] of them, rows query_start[i] ..
 * query_start[i+1]-1 of q. Query j sits at position context_lens[i] - n_i + j
 * and attends to positions 0..that:
 *   out[query_start[i] + j, h] = softmax(scale * q . K[0..p]) V[0..p],
 * K, V of KV head h / (num_heads / num_kv_heads).
 *
 * q, out: DEVICE [num_tokens, num_heads, head_dim] of `dtype`, 16-byte
 * aligned; caches as for pa_decode, same dtype; block_tables, context_lens,
 * query_start (int32 [num_seqs + 1], non-decreasing, query_start[0] = 0,
 * query_start[num_seqs] = num_tokens): DEVICE. Entries outside [0,
 * num_tokens], or smaller than the entry before, are clamped into that range
 * (so no row outside q and out is read or written) and set
 * PA_DEVERR_QUERY_START. max_query_len bounds n_i (it
 * sizes the grid; chunks beyond it are not computed). Sequences whose
 * context is shorter than their chunk, or longer than the table holds, set
 * PA_DEVERR_CONTEXT_RANGE; table entries outside [0, num_blocks) set
 * PA_DEVERR_BLOCK_RANGE and their keys are skipped.
 *
 * Supported: dtype PA_F16 or PA_BF16, head_dim 128, num_heads / num_kv_heads
 * in {1, 2, 4, 8}, block_size in {8, 16, 32, 64}; others return
 * PA_ERR_UNSUPPORTED.
 */
pa_status pa_prefill(void* out, const void* q, const void* k_cache, const void* v_cache,
                     const int32_t* block_tables, int32_t max_blocks_per_seq,
                     const int32_t* context_lens, const int32_t* query_start,
                     int32_t num_seqs, int32_t num_tokens, int32_t max_query_len,
                     int32_t num_heads, int32_t num_kv_heads, int32_t head_dim,
                     int32_t block_size, int32_t num_blocks, float scale, pa_dtype dtype,
                     int32_t* debug_err, cudaStream_t stream);

/* Layers one pa_swap_blocks call moves at most. */
#define PA_SWAP_MAX_LAYERS 64

/*
 * pa_swap_blocks - move whole blocks, K and V, in every layer, between two
 * pools, typically the device pool and a pool in pinned host memory.
 *
 * This is the swap way of preempting a request when the pool runs out of
 * free blocks: its blocks are moved to CPU memory and brought back later,
 * which keeps the computed cache at the price of the transfer over the host
 * link (serving-paged-attention, "그래도 넘칠 때 — 선점", item "스왑").
 * For each pair p, src = block_mapping[2p], dst = block_mapping[2p+1], and
 * each layer l: block dst of dst_k[l] (dst_v[l]) becomes a byte copy of
 * block src of src_k[l] (src_v[l]). Swap-out passes the device caches as
 * src and the host pools as dst; swap-in the reverse. The caller updates
 * the block tables and frees or allocates the blocks.
 *
 * dst_k, dst_v, src_k, src_v are HOST arrays of num_layers pointers (1 <=
 * num_layers <= PA_SWAP_MAX_LAYERS). Each pointer, and block_mapping (int64
 * [num_pairs, 2]), must be device memory or pinned host memory mapped into
 * the device's address space (cudaHostAlloc / cudaHostRegister, torch
 * pin_memory); other pointers are refused with PA_ERR_INVALID before any
 * launch. Pointers are 16-byte aligned; block_bytes (one block of one cache
 * of one layer) is a positive multiple of 16; the src pools hold
 * src_num_blocks blocks, the dst pools dst_num_blocks. Pairs outside those
 * ranges set PA_DEVERR_BLOCK_RANGE in *debug_err (if not NULL) and are
 * skipped. dst blocks must be distinct and must not overlap the src blocks
 * of the same call. The call is asynchronous on `stream`; the caller keeps
 * every buffer alive and unmodified until the stream has passed it.
 */
pa_status pa_swap_blocks(void* const* dst_k, void* const* dst_v,
                         const void* const* src_k, const void* const* src_v,
                         int32_t num_layers, const int64_t* block_mapping,
                         int32_t num_pairs, int32_t src_num_blocks,
                         int32_t dst_num_blocks, size_t block_bytes,
                         int32_t* debug_err, cudaStream_t stream);

/*
 * pa_decode_split_noalloc - pa_decode's split-context path without a
 * caller-provided workspace. (The source pages have no counterpart; this is
 * an interface for callers, not a step of the method.)
 *
 * For callers that cannot allocate device memory: a plugin inside a host
 * framework that owns every device allocation and gives its plugins none, or
 * a runtime whose device memory is fixed at start-up (real-time and
 * certified deployments forbid allocating afterwards). The partial
 * results of the partitions go to a scratch array built into the library
 * (16 MiB, a file-scope __device__ array that every GPU loading the library
 * holds until the process exits). Nothing is allocated or freed by this call.
 *
 * Arguments and results are those of pa_decode with the split path forced
 * (partition_size 0 means 512 tokens). Sizes whose partials would not fit
 * the 16 MiB (pa_decode_workspace_size() above 16 MiB) are rejected with
 * PA_ERR_WORKSPACE and a message giving both sizes.
 *
 * The first call on a device looks up the scratch array's device address
 * (cudaGetSymbolAddress, with that device current) and keeps it; make that
 * first call before any stream capture. All calls share the one array, which
 * keeps the last call's contents: each call writes every partial it reads, so
 * nothing needs clearing, but calls whose kernels overlap on the GPU (on
 * different streams, or from different threads) race on the array and must
 * be serialised by the caller.
 */
pa_status pa_decode_split_noalloc(void* out, const void* q, const void* k_cache,
                                  const void* v_cache, const int32_t* block_tables,
                                  int32_t max_blocks_per_seq, const int32_t* context_lens,
                                  int32_t num_seqs, int32_t num_heads, int32_t num_kv_heads,
                                  int32_t head_dim, int32_t block_size, int32_t num_blocks,
                                  float scale, pa_dtype q_dtype, pa_dtype kv_dtype,
                                  const float* k_scale, const float* v_scale,
                                  int32_t max_context_len, int32_t partition_size,
                                  int32_t* debug_err, cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* PA_H_ */
