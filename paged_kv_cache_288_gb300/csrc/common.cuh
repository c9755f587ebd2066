// Device-side helpers shared by the kernels of this library: element types,
// vector loads that widen to float32, and the parameter blocks the C-ABI
// layer fills in.
#pragma once

#include <cuda_runtime.h>
#include <cuda_fp16.h>
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <stdint.h>

#include "pa.h"

namespace pa {

using f16 = __half;
using bf16 = __nv_bfloat16;
using fp8 = __nv_fp8_e4m3;

constexpr float kLog2e = 1.4426950408889634f;

template <typename T> struct is_fp8 { static constexpr bool value = false; };
template <> struct is_fp8<fp8> { static constexpr bool value = true; };

// Vector type holding N elements of T (N * sizeof(T) bytes, power of two).
template <int Bytes> struct VecOf;
template <> struct VecOf<2> { using type = uint16_t; };
template <> struct VecOf<4> { using type = uint32_t; };
template <> struct VecOf<8> { using type = uint2; };
template <> struct VecOf<16> { using type = uint4; };

__device__ __forceinline__ float2 pair_to_float2(uint32_t w, f16*) {
  __half2 h = *reinterpret_cast<__half2*>(&w);
  return __half22float2(h);
}
__device__ __forceinline__ float2 pair_to_float2(uint32_t w, bf16*) {
  __nv_bfloat162 h = *reinterpret_cast<__nv_bfloat162*>(&w);
  return __bfloat1622float2(h);
}
__device__ __forceinline__ float2 fp8pair_to_float2(uint16_t w) {
  __half2_raw r = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(w), __NV_E4M3);
  __half2 h = *reinterpret_cast<__half2*>(&r);
  return __half22float2(h);
}

// Load N consecutive elements of T at p (aligned to N*sizeof(T)) as floats.
template <typename T, int N>
__device__ __forceinline__ void load_float(const T* __restrict__ p, float (&f)[N]) {
  static_assert(N % 2 == 0, "pairs only");
  using V = typename VecOf<N * sizeof(T)>::type;
  V v = *reinterpret_cast<const V*>(p);
  if constexpr (is_fp8<T>::value) {
    const uint16_t* w = reinterpret_cast<const uint16_t*>(&v);
#pragma unroll
    for (int i = 0; i < N / 2; ++i) {
      float2 x = fp8pair_to_float2(w[i]);
      f[2 * i] = x.x;
      f[2 * i + 1] = x.y;
    }
  } else {
    const uint32_t* w = reinterpret_cast<const uint32_t*>(&v);
#pragma unroll
    for (int i = 0; i < N / 2; ++i) {
      float2 x = pair_to_float2(w[i], static_cast<T*>(nullptr));
      f[2 * i] = x.x;
      f[2 * i + 1] = x.y;
    }
  }
}

__device__ __forceinline__ f16 from_float(float x, f16*) { return __float2half_rn(x); }
__device__ __forceinline__ bf16 from_float(float x, bf16*) { return __float2bfloat16_rn(x); }

__device__ __forceinline__ void flag_error(int32_t* err, int32_t bit) {
  if (err != nullptr) atomicOr(err, bit);
}

// Everything a decode kernel reads; filled by the C-ABI layer.
struct DecodeParams {
  void* out;
  const void* q;
  const void* k_cache;
  const void* v_cache;
  const int32_t* block_tables;
  const int32_t* context_lens;
  const float* k_scale;
  const float* v_scale;
  float* ws_acc;   // [num_seqs, num_heads, num_partitions, head_dim] normalised partial outputs
  float* ws_ml;    // [num_seqs, num_heads, num_partitions, 2] (max in log2 units, sum)
  int32_t* debug_err;
  int32_t* claim;           // work counter the partition reduce rearms (tensor-core split path), or null
  int32_t max_blocks_per_seq;
  int32_t num_seqs;
  int32_t num_heads;
  int32_t num_kv_heads;     // KV units per sequence: KV heads, or slices of 8 query heads of one
  int32_t kv_heads_phys;    // KV heads in the cache layout
  int32_t kv_div;           // units per KV head (1, or G / 8 for groups above 8)
  int32_t block_size;
  int32_t num_blocks;
  int32_t max_context_len;
  int32_t partition_size;   // tokens per partition (multiple of block_size)
  int32_t num_partitions;   // partitions per sequence in the grid
  float scale_log2;         // softmax scale * log2(e)
};

// Groups of sequences that share the leading blocks of their tables (a common
// prompt prefix). Group g is sequences group_start[g] .. group_start[g+1]-1;
// every member's first group_prefix[g] tokens are the same physical blocks.
// The shared tokens are attended once per group (prefix_attn_kernel) into
// partial softmax states, which the merge combines with each member's own
// suffix.
struct PrefixGroups {
  const int32_t* group_start;   // device [num_groups + 1]
  const int32_t* group_prefix;  // device [num_groups], tokens (multiples of block_size)
  float* ws_prefix;             // [num_seqs * units * num_chunks] states of group * (D + 2) floats
  int32_t num_groups;
  int32_t max_group_size;       // members per group the prefix grid covers
  int32_t max_prefix_len;       // bound on every group's prefix; sizes the prefix grid
  int32_t chunk_len;            // keys per prefix chunk, a multiple of 16 and of block_size
  int32_t num_chunks;           // chunks of the longest prefix
};

// The member range [a, b) and the shared token count of group g, clamped so
// that no index leaves its array: ranges into [0, num_seqs], at most
// max_group_size members, the prefix into [0, min(max_prefix_len, table
// width)] and down to whole blocks. Returns true when anything was clamped.
__device__ __forceinline__ bool prefix_group(const PrefixGroups& pg, int g, int num_seqs,
                                             int max_blocks_per_seq, int block_size, int& a,
                                             int& b, int& len) {
  const int a0 = pg.group_start[g], b0 = pg.group_start[g + 1], p0 = pg.group_prefix[g];
  a = min(max(a0, 0), num_seqs);
  b = min(max(b0, a), num_seqs);
  bool clamped = a != a0 || b != b0;
  if (b - a > pg.max_group_size) {
    b = a + pg.max_group_size;
    clamped = true;
  }
  const int cap = min(pg.max_prefix_len, max_blocks_per_seq * block_size);
  len = min(max(p0, 0), cap);
  len -= len % block_size;
  return clamped || len != p0;
}

// Floats of one partial softmax state of a KV unit with `group` query heads:
// the unnormalised accumulators [group][head_dim], then the group's maxima and
// sums, padded to a multiple of 4 so that every state starts 16-byte aligned
// (the merge reads the accumulators as float4).
__host__ __device__ constexpr int state_floats(int group, int head_dim) {
  return group * head_dim + ((2 * group + 3) & ~3);
}

// KV head of the caches that KV unit u reads.
__device__ __forceinline__ int kv_head_of(const DecodeParams& p, int u) {
  return p.kv_div == 1 ? u : u / p.kv_div;
}

// Clamp a sequence's context length to what the table and the grid cover.
__device__ __forceinline__ int clamp_context(const DecodeParams& p, int seq) {
  int ctx = p.context_lens[seq];
  int cap = min(p.max_context_len, p.max_blocks_per_seq * p.block_size);
  if (ctx > cap) {
    flag_error(p.debug_err, PA_DEVERR_CONTEXT_RANGE);
    ctx = cap;
  }
  return ctx < 0 ? 0 : ctx;
}

}  // namespace pa
