// Paged prefill: causal attention of a chunk of new query tokens per sequence
// over its paged KV cache, on the 5th-generation tensor cores.
//
// Each sequence holds context_lens[i] tokens, the last n_i of which are its
// queries (their K/V already written by pa_reshape_and_cache); query j sits
// at position ctx_i - n_i + j and attends to the keys at positions 0..that.
// Prefill and decode read the same block tables (serving-paged-attention,
// "블록으로 쪼개고 표로 잇는다"); prefill is the many-query step before decode
// (LLM 추론 확장, 품질·비용 절충 필수, the prefill / decode split), which makes
// QK^T and PV dense tiles.
//
// One CTA of 4 warps per (query tile, KV head, sequence). A tile is 128 MMA
// rows: 128/G query tokens x the G query heads of the KV head, row r = token
// r/G, head r%G. Thread r owns row r (TMEM lane r). Per 128-key tile:
//   S = Q K^T   tcgen05.mma, M=128, N=128, K=128 (8 steps), Q and K tiles
//               K-major with 128-byte swizzle, loaded by TMA (K block by block
//               through the block table), S in TMEM columns 0..127;
//   softmax     each thread reads its row of S from TMEM, masks keys past its
//               position, keeps a running max in log2 units (the accumulator
//               is rescaled only when the max grows by more than 2^8), and
//               writes P (16-bit) to shared memory in the K-major swizzled
//               layout;
//   O += P V    tcgen05.mma with V as an MN-major operand straight from its
//               TMA tile, O in TMEM columns 128..255.
// K/V tiles are double-buffered; the next tile's TMA loads go out as soon as
// the MMA that read the buffer has completed. Every wait is bounded: on a
// timeout the CTA sets PA_DEVERR_TIMEOUT, waits briefly for its own tensor
// core work, frees its TMEM and returns.
#include "common.cuh"
#include "internal.h"
#include "ptx.cuh"

#include <cudaTypedefs.h>

namespace pa {
namespace {

constexpr int kPfThreads = 128;
constexpr int kPfRows = 128;                   // MMA M
constexpr int kPfKeys = 128;                   // keys per KV tile
constexpr int kPfD = 128;                      // head dim
constexpr int kHalf = kPfRows * 128;           // a 64-column half of a 128-row 16-bit tile
constexpr int kTile = 2 * kHalf;               // 32 KiB
constexpr int kSmemBytes = 1024 + 6 * kTile;   // Q, P, K[2], V[2] + alignment slack
constexpr uint32_t kTmemCols = 256;            // S: 0..127, O: 128..255
constexpr float kLazyRescale = 8.f;            // log2 units

struct PfParams {
  void* out;
  const int32_t* block_tables;
  const int32_t* context_lens;
  const int32_t* query_start;
  int32_t* debug_err;
  int max_blocks_per_seq;
  int num_heads;
  int num_kv_heads;
  int block_size;
  int num_blocks;
  int group;
  int tokens_per_tile;
  float scale_log2;
};

template <typename T>
__device__ __forceinline__ uint32_t pack2(float lo, float hi);
template <>
__device__ __forceinline__ uint32_t pack2<bf16>(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}
template <>
__device__ __forceinline__ uint32_t pack2<f16>(float lo, float hi) {
  __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

// Byte offset of the 16-byte chunk holding columns 8c..8c+7 of row r in a
// 128-row K-major tile stored as two 64-column halves with the 128-byte
// swizzle (the layout TMA writes and the MMA descriptors describe).
__device__ __forceinline__ uint32_t sw128_chunk(int r, int c) {
  return (c >> 3) * kHalf + r * 128 + (((c & 7) ^ (r & 7)) << 4);
}

template <typename T>
__global__ void __launch_bounds__(kPfThreads, 1)
    prefill_tc_kernel(const __grid_constant__ CUtensorMap tmap_q, const __grid_constant__ CUtensorMap tmap_k,
                      const __grid_constant__ CUtensorMap tmap_v, const PfParams p) {
  const int tile = blockIdx.x, kvh = blockIdx.y, seq = blockIdx.z;
  const int q0 = p.query_start[seq];
  const int n = p.query_start[seq + 1] - q0;
  const int G = p.group, TQ = p.tokens_per_tile;
  const int t0 = tile * TQ;
  if (t0 >= n) return;  // CTA-uniform, before any TMEM is held
  const int bs = p.block_size;
  int ctx = p.context_lens[seq];
  const int cap = p.max_blocks_per_seq * bs;
  if (ctx > cap || ctx < n) {
    // a context past the table, or shorter than the chunk of queries
    if (threadIdx.x == 0) flag_error(p.debug_err, PA_DEVERR_CONTEXT_RANGE);
    ctx = min(ctx, cap);
    if (ctx < n) return;
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r = threadIdx.x;  // this thread's row

  extern __shared__ unsigned char smem_raw[];
  unsigned char* sm = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                       ~static_cast<uintptr_t>(1023));
  const uint32_t sQ = smem_u32(sm);
  const uint32_t sP = sQ + kTile;
  const uint32_t sK0 = sQ + 2 * kTile;  // K[stage] = sK0 + stage * kTile
  const uint32_t sV0 = sQ + 4 * kTile;
  unsigned char* const pP = sm + kTile;
  unsigned char* const pV0 = sm + 4 * kTile;
  __shared__ uint64_t bars[5];  // Q, KV[0], KV[1], S done, PV done
  __shared__ uint32_t tmem_slot;
  const uint32_t bar_q = smem_u32(&bars[0]);
  const uint32_t bar_kv0 = smem_u32(&bars[1]);
  const uint32_t bar_s = smem_u32(&bars[3]);
  const uint32_t bar_o = smem_u32(&bars[4]);

  if (threadIdx.x == 0) {
    for (int i = 0; i < 5; ++i) mbar_init(smem_u32(&bars[i]), 1);
    mbar_init_fence();
  }
  if (warp == 0) tmem_alloc(smem_u32(&tmem_slot), kTmemCols);
  tc05_fence_before();
  __syncthreads();
  tc05_fence_after();
  const uint32_t tmem = tmem_slot;
  const uint32_t tmem_s = tmem, tmem_o = tmem + 128;
  const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;

  // the keys this tile needs: 0 .. position of its last query
  const int t_last = min(t0 + TQ, n) - 1;
  const int pos_last = ctx - n + t_last;
  const int nkt = pos_last / kPfKeys + 1;
  // this row's query position (rows past the chunk repeat the last position;
  // they are not stored)
  const int my_t = min(t0 + r / G, n - 1);
  const int my_pos = ctx - n + my_t;

  constexpr uint32_t kAB = std::is_same<T, bf16>::value ? 1u : 0u;
  constexpr uint32_t idesc_s = mma_idesc_f16(kAB, 0, kPfRows, kPfKeys);
  constexpr uint32_t idesc_o = mma_idesc_f16(kAB, 1, kPfRows, kPfD);
  const int blocks_per_tile = kPfKeys / bs;

  // TMA loads of key tile kt into stage st (thread 0): every block of the
  // tile that holds tokens of the context, both 64-column halves, K and V.
  auto issue_kv = [&](int kt, int st) {
    const uint32_t bar = bar_kv0 + st * 8;
    const int lb0 = kt * blocks_per_tile;
    int phys[kPfKeys / 8];
    int nload = 0;
    for (int j = 0; j < blocks_per_tile; ++j) {
      phys[j] = -1;
      const int lb = lb0 + j;
      if (lb * bs >= ctx) continue;
      const int b = p.block_tables[static_cast<int64_t>(seq) * p.max_blocks_per_seq + lb];
      if (b < 0 || b >= p.num_blocks) {
        flag_error(p.debug_err, PA_DEVERR_BLOCK_RANGE);
        continue;
      }
      phys[j] = b;
      ++nload;
    }
    mbar_arrive_expect_tx(bar, static_cast<uint32_t>(nload) * 4u * bs * 128u);
    for (int j = 0; j < blocks_per_tile; ++j) {
      if (phys[j] < 0) continue;
      const int z = phys[j] * p.num_kv_heads + kvh;
      for (int h = 0; h < 2; ++h) {
        const uint32_t off = st * kTile + h * kHalf + j * bs * 128;
        tma_load_3d(sK0 + off, &tmap_k, h * 64, 0, z, bar);
        tma_load_3d(sV0 + off, &tmap_v, h * 64, 0, z, bar);
      }
    }
  };

  if (threadIdx.x == 0) {
    mbar_arrive_expect_tx(bar_q, 2u * kHalf);
    for (int h = 0; h < 2; ++h) tma_load_3d(sQ + h * kHalf, &tmap_q, h * 64, kvh * G, q0 + t0, bar_q);
    issue_kv(0, 0);
    if (nkt > 1) issue_kv(1, 1);
  }

  float m_run = -INFINITY, l_run = 0.f;
  bool ok = true, aborted = false;
  for (int kt = 0; kt < nkt; ++kt) {
    const int st = kt & 1;
    const uint32_t kv_parity = (kt >> 1) & 1;
    // ---- S = Q K^T ----
    if (threadIdx.x == 0) {
      ok = (kt > 0 || mbar_wait_bounded(bar_q, 0)) && mbar_wait_bounded(bar_kv0 + st * 8, kv_parity);
      if (ok) {
        tc05_fence_after();
#pragma unroll
        for (int k = 0; k < kPfD / 16; ++k) {
          const uint32_t koff = (k >> 2) * kHalf + (k & 3) * 32;
          tc05_mma_ss(tmem_s, smem_desc_sw128(sQ + koff, 16, 1024),
                      smem_desc_sw128(sK0 + st * kTile + koff, 16, 1024), idesc_s, k > 0);
        }
        tc05_commit(bar_s);
      }
    }
    ok = mbar_wait_bounded(bar_s, kt & 1) && mbar_wait_bounded(bar_kv0 + st * 8, kv_parity);
    if (__syncthreads_or(!ok)) {
      aborted = true;
      break;
    }
    tc05_fence_after();

    // ---- softmax of this thread's row ----
    float s[kPfKeys];
#pragma unroll
    for (int c = 0; c < kPfKeys; c += 32) {
      uint32_t v[32];
      tmem_ld32(tmem_s + lane_base + c, v);
      tmem_wait_ld();
#pragma unroll
      for (int j = 0; j < 32; ++j) s[c + j] = __uint_as_float(v[j]);
    }
    const int key0 = kt * kPfKeys;
    float mx = -INFINITY;
#pragma unroll
    for (int c = 0; c < kPfKeys; ++c) {
      s[c] = key0 + c <= my_pos ? s[c] * p.scale_log2 : -INFINITY;
      mx = fmaxf(mx, s[c]);
    }
    float m_use = m_run, alpha = 1.f;
    if (mx > m_run + kLazyRescale || m_run == -INFINITY) {
      m_use = fmaxf(m_run, mx);
      alpha = m_run == -INFINITY ? 0.f : exp2f(m_run - m_use);
    }
    const float base = m_use == -INFINITY ? 0.f : m_use;
    float sum = 0.f;
#pragma unroll
    for (int c = 0; c < kPfKeys; ++c) {
      s[c] = exp2f(s[c] - base);
      sum += s[c];
    }
    l_run = l_run * alpha + sum;
    m_run = m_use;

    // the previous PV product is complete: P, O and the other K/V buffer are free
    if (kt > 0) {
      ok = mbar_wait_bounded(bar_o, (kt - 1) & 1);
      if (__syncthreads_or(!ok)) {
        aborted = true;
        break;
      }
      tc05_fence_after();
      if (threadIdx.x == 0 && kt + 1 < nkt) issue_kv(kt + 1, (kt + 1) & 1);
      // rescale O where this row's max moved (warps with no such row skip)
      if (__any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll
        for (int c = 0; c < kPfD; c += 32) {
          uint32_t v[32];
          tmem_ld32(tmem_o + lane_base + c, v);
          tmem_wait_ld();
#pragma unroll
          for (int j = 0; j < 32; ++j) v[j] = __float_as_uint(__uint_as_float(v[j]) * alpha);
          tmem_st32(tmem_o + lane_base + c, v);
        }
        tmem_wait_st();
      }
    }
    // keys past the context in the last tile: zero their V rows (stale or
    // unwritten shared memory must not meet a zero weight as NaN)
    const int valid = ctx - key0;
    if (valid < kPfKeys) {
      unsigned char* vt = pV0 + st * kTile;
      for (int i = threadIdx.x; i < (kPfKeys - valid) * 16; i += kPfThreads) {
        const int row = valid + i / 16, chunk = i % 16;
        *reinterpret_cast<uint4*>(vt + (chunk >> 3) * kHalf + row * 128 + (((chunk & 7) ^ (row & 7)) << 4)) =
            make_uint4(0u, 0u, 0u, 0u);
      }
    }
    // P in the K-major swizzled layout of the PV product's A operand
#pragma unroll
    for (int c = 0; c < kPfKeys; c += 8) {
      uint4 w;
      w.x = pack2<T>(s[c], s[c + 1]);
      w.y = pack2<T>(s[c + 2], s[c + 3]);
      w.z = pack2<T>(s[c + 4], s[c + 5]);
      w.w = pack2<T>(s[c + 6], s[c + 7]);
      *reinterpret_cast<uint4*>(pP + sw128_chunk(r, c >> 3)) = w;
    }
    fence_proxy_async_smem();
    tc05_fence_before();
    __syncthreads();

    // ---- O += P V ----
    if (threadIdx.x == 0) {
      tc05_fence_after();
#pragma unroll
      for (int k = 0; k < kPfKeys / 16; ++k) {
        tc05_mma_ss(tmem_o, smem_desc_sw128(sP + (k >> 2) * kHalf + (k & 3) * 32, 16, 1024),
                    smem_desc_sw128(sV0 + st * kTile + k * 16 * 128, kHalf, 1024), idesc_o,
                    (kt > 0 || k > 0) ? 1u : 0u);
      }
      tc05_commit(bar_o);
    }
  }

  if (!aborted) aborted = __syncthreads_or(!mbar_wait_bounded(bar_o, (nkt - 1) & 1));
  if (!aborted) {
    tc05_fence_after();
    // ---- out = O / l for the rows of the chunk ----
    const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
    const int tok = t0 + r / G;
    T* orow = static_cast<T*>(p.out) +
              (static_cast<int64_t>(q0 + min(tok, n - 1)) * p.num_heads + kvh * G + r % G) * kPfD;
#pragma unroll
    for (int c = 0; c < kPfD; c += 32) {
      uint32_t v[32];
      tmem_ld32(tmem_o + lane_base + c, v);
      tmem_wait_ld();
      if (tok < n) {
#pragma unroll
        for (int j = 0; j < 32; j += 8) {
          uint4 w;
          w.x = pack2<T>(__uint_as_float(v[j]) * inv, __uint_as_float(v[j + 1]) * inv);
          w.y = pack2<T>(__uint_as_float(v[j + 2]) * inv, __uint_as_float(v[j + 3]) * inv);
          w.z = pack2<T>(__uint_as_float(v[j + 4]) * inv, __uint_as_float(v[j + 5]) * inv);
          w.w = pack2<T>(__uint_as_float(v[j + 6]) * inv, __uint_as_float(v[j + 7]) * inv);
          *reinterpret_cast<uint4*>(orow + c + j) = w;
        }
      }
    }
  } else {
    if (threadIdx.x == 0) {
      flag_error(p.debug_err, PA_DEVERR_TIMEOUT);
      // let tensor-core work already issued finish before its TMEM goes away
      mbar_wait_bounded(bar_s, 0, 10000000ull);
      mbar_wait_bounded(bar_o, 0, 10000000ull);
    }
  }
  tc05_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, kTmemCols);
}

PFN_cuTensorMapEncodeTiled_v12000 pf_encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static bool tried = false;
  if (!tried) {
    tried = true;
    cudaDriverEntryPointQueryResult q;
    void* ptr = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  }
  return fn;
}

bool encode3d(CUtensorMap* map, const void* base, const cuuint64_t (&dims)[3], const cuuint64_t (&strides)[2],
              const cuuint32_t (&box)[3]) {
  auto fn = pf_encode_fn();
  if (fn == nullptr) return false;
  cuuint32_t es[3] = {1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT16, 3, const_cast<void*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool prefill_supported(int group, int head_dim, pa_dtype dtype, int block_size) {
  return head_dim == kPfD && (dtype == PA_F16 || dtype == PA_BF16) &&
         (group == 1 || group == 2 || group == 4 || group == 8) && block_size >= 8 && block_size <= 64;
}

cudaError_t launch_prefill_tc(void* out, const void* q, const void* k_cache, const void* v_cache,
                              const int32_t* block_tables, int max_blocks_per_seq,
                              const int32_t* context_lens, const int32_t* query_start, int num_seqs,
                              int num_tokens, int max_query_len, int num_heads, int num_kv_heads,
                              int block_size, int num_blocks, float scale, pa_dtype dtype,
                              int32_t* debug_err, cudaStream_t stream) {
  if (num_seqs == 0 || num_tokens == 0 || max_query_len == 0) return cudaSuccess;
  const int G = num_heads / num_kv_heads;
  PfParams pp{};
  pp.out = out;
  pp.block_tables = block_tables;
  pp.context_lens = context_lens;
  pp.query_start = query_start;
  pp.debug_err = debug_err;
  pp.max_blocks_per_seq = max_blocks_per_seq;
  pp.num_heads = num_heads;
  pp.num_kv_heads = num_kv_heads;
  pp.block_size = block_size;
  pp.num_blocks = num_blocks;
  pp.group = G;
  pp.tokens_per_tile = kPfRows / G;
  pp.scale_log2 = scale * 1.4426950408889634f;
  CUtensorMap mq, mk, mv;
  const cuuint64_t row = static_cast<cuuint64_t>(kPfD) * 2;
  if (!encode3d(&mq, q, {static_cast<cuuint64_t>(kPfD), static_cast<cuuint64_t>(num_heads),
                         static_cast<cuuint64_t>(num_tokens)},
                {row, row * num_heads}, {64, static_cast<cuuint32_t>(G), static_cast<cuuint32_t>(kPfRows / G)}))
    return cudaErrorInvalidValue;
  const cuuint64_t bxh = static_cast<cuuint64_t>(num_blocks) * num_kv_heads;
  const cuuint64_t kdims[3] = {static_cast<cuuint64_t>(kPfD), static_cast<cuuint64_t>(block_size), bxh};
  const cuuint64_t kstr[2] = {row, row * block_size};
  const cuuint32_t kbox[3] = {64, static_cast<cuuint32_t>(block_size), 1};
  if (!encode3d(&mk, k_cache, kdims, kstr, kbox) || !encode3d(&mv, v_cache, kdims, kstr, kbox))
    return cudaErrorInvalidValue;
  const int tiles = (max_query_len + pp.tokens_per_tile - 1) / pp.tokens_per_tile;
  dim3 grid(tiles, num_kv_heads, num_seqs);
  cudaError_t err;
  if (dtype == PA_BF16) {
    static bool set = false;
    if (!set) {
      err = cudaFuncSetAttribute(prefill_tc_kernel<bf16>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
      if (err != cudaSuccess) return err;
      set = true;
    }
    prefill_tc_kernel<bf16><<<grid, kPfThreads, kSmemBytes, stream>>>(mq, mk, mv, pp);
  } else {
    static bool set = false;
    if (!set) {
      err = cudaFuncSetAttribute(prefill_tc_kernel<f16>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
      if (err != cudaSuccess) return err;
      set = true;
    }
    prefill_tc_kernel<f16><<<grid, kPfThreads, kSmemBytes, stream>>>(mq, mk, mv, pp);
  }
  err = cudaGetLastError();
  if (err == cudaSuccess) note_launches(1);
  return err;
}

}  // namespace pa
