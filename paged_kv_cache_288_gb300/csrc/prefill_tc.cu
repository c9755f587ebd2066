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
// One CTA of 24 warps per (pair of query tiles, KV head, sequence). A query
// tile is 128 MMA rows: 128/G query tokens x the G query heads of the KV
// head, row r = token r/G, head r%G; the two tiles of a CTA share every K/V
// tile, which halves the TMA boxes per FLOP. Per 64-key tile:
//   S = Q K^T   tcgen05.mma, M=128, N=64, K=128 (8 steps) per query tile; Q
//               and K K-major with the 128-byte swizzle, loaded by TMA (K one
//               box per 16-token block and 64-column half, through the block
//               table); S double-buffered in TMEM (two 64-column buffers per
//               query tile), so the next S is computed during the softmax;
//   softmax     16 warps, two threads per row (32 keys each): read the row of
//               S from TMEM, mask keys past the row's position, keep a running
//               max in log2 units (O is rescaled only when the max grows by
//               more than 2^8), and store P (16-bit) in TMEM over the S it
//               came from;
//   O += P V    tcgen05.mma with A = P from TMEM and V an MN-major operand
//               straight from its TMA tile, O in TMEM (128 columns per query
//               tile).
// Warp roles: three K loaders (the first also loads Q) and three V loaders
// (a tile's boxes spread over them), one thread each issues S and PV.
// K and V tiles go through rings of 4 buffers, each refilled once the
// products that read it have completed. CTAs take the heaviest work first
// (see the work order below). Every wait is bounded: on a timeout the CTA
// sets PA_DEVERR_TIMEOUT, waits briefly for its own tensor core work, frees
// its TMEM and returns.
#include "common.cuh"
#include "internal.h"
#include "ptx.cuh"

#include <cudaTypedefs.h>

namespace pa {
namespace {

constexpr int kGroups = 2;                      // query tiles per CTA (they share the K/V tiles)
constexpr int kRowsPerGroup = 128;              // rows of a query tile
constexpr int kGroupThreads = 2 * kRowsPerGroup;        // two softmax threads per row
constexpr int kSoftThreads = kGroups * kGroupThreads;   // 16 softmax warps
// TMA issue: one thread issues only a few 2 KiB boxes per microsecond and
// lanes of one warp add little, so each of K and V has kLoadWarps loader
// warps with kLoadLanes issuing lanes each; box i (= 2 * block + half) of a
// tile goes to loader q = i % (kLoadWarps * kLoadLanes), which is lane
// q / kLoadWarps of loader warp q % kLoadWarps
constexpr int kLoadWarps = 3;
constexpr int kLoadLanes = 1;
constexpr int kLoaders = kLoadWarps * kLoadLanes;
// + role warps: K loaders (the first also loads Q), V loaders, S issue, PV issue
constexpr int kPfThreads = kSoftThreads + 32 * (2 * kLoadWarps + 2);
static_assert(kPfThreads % 128 == 0, "whole warpgroups");
// Registers: 24 warps are 6 per scheduler, which caps a thread at 80 at
// launch. The softmax warpgroups raise theirs to 96 and the role warpgroups
// lower theirs to 48 (setmaxnreg); the split must not exceed what the launch
// allocated, or the raise waits forever.
constexpr int kLaunchRegs = 80, kSoftRegs = 96, kRoleRegs = 48;
static_assert(kSoftThreads * kSoftRegs + (kPfThreads - kSoftThreads) * kRoleRegs <= kPfThreads * kLaunchRegs,
              "register split within the launch allocation");
constexpr int kPfRows = 128;                   // MMA M: rows of a query tile
constexpr int kPfKeys = 64;                    // keys per K/V tile (MMA N of S, K of PV)
constexpr int kPfD = 128;                      // head dim
constexpr int kStages = 4;                     // K and V tiles in flight
constexpr int kHalf = kPfRows * 128;           // a 64-column half of a 128-row 16-bit tile
constexpr int kTile = 2 * kHalf;               // a Q tile: 32 KiB
constexpr int kKVHalf = kPfKeys * 128;         // a 64-column half of a K/V tile: 8 KiB
constexpr int kKVTile = 2 * kKVHalf;           // a K/V tile: 16 KiB
// Q[2], K and V rings; barriers (512 B); row exchange (2 KiB)
constexpr int kSmemBytes = 2 * kTile + 2 * kStages * kKVTile + 1024 + 2048;
static_assert(kSmemBytes <= 227 * 1024, "shared memory per CTA");
// per group: S[2] (64 columns each; P, 16-bit, replaces its S in the first
// 32 columns), O (128 columns)
constexpr uint32_t kTmemCols = 512;
constexpr float kLazyRescale = 8.f;            // log2 units
constexpr int kRankMaxSeqs = 256;              // batches up to this size are ordered by work

struct PfParams {
  void* out;
  const int32_t* block_tables;
  const int32_t* context_lens;
  const int32_t* query_start;
  int32_t* debug_err;
  int max_blocks_per_seq;
  int num_tokens;
  int num_heads;
  int num_kv_heads;
  int block_size;
  int num_blocks;
  int group;
  int tokens_per_tile;
  float scale_log2;
};

// Rows [q0, q0 + n) of q and out that hold sequence i's queries, from
// query_start clamped into [0, num_tokens] (an entry below the one before it
// counts as that one), so no row outside q and out is ever addressed.
// Returns true when query_start had to be clamped.
__device__ __forceinline__ bool query_rows(const PfParams& p, int i, int& q0, int& n) {
  const int a = p.query_start[i], b = p.query_start[i + 1];
  const int lo = min(max(a, 0), p.num_tokens);
  const int hi = min(max(b, lo), p.num_tokens);
  q0 = lo;
  n = hi - lo;
  return a != lo || b != hi;
}

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

// A wait on an mbarrier that gives up after kWaitLimitNs, or as soon as
// another thread of the CTA has given up (*abort set).
__device__ __forceinline__ bool pf_wait(uint32_t bar, uint32_t parity, volatile int* abort) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (*abort) return false;
    if (globaltimer_ns() - t0 > kWaitLimitNs) {
      *abort = 1;
      return false;
    }
  }
  return true;
}

__device__ __forceinline__ void named_sync(int id, int threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

__device__ __forceinline__ void named_arrive(int id, int threads) {
  asm volatile("bar.arrive %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// 2^x of the special function unit, subnormal results flushed to zero (a
// softmax weight below 2^-126 is rounded to zero in 16 bits anyway)
__device__ __forceinline__ float ex2_ftz(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float max3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// (x0, x1) = (x0 * b + c, x1 * b + c) in one packed two-lane FMA
__device__ __forceinline__ void exp_arg2(float& x0, float& x1, float b, float c) {
  asm("{\n\t.reg .b64 ra, rb, rc;\n\t"
      "mov.b64 ra, {%0, %1};\n\tmov.b64 rb, {%2, %2};\n\tmov.b64 rc, {%3, %3};\n\t"
      "fma.rn.f32x2 ra, ra, rb, rc;\n\tmov.b64 {%0, %1}, ra;\n\t}"
      : "+f"(x0), "+f"(x1)
      : "f"(b), "f"(c));
}

// (s0, s1) += (x0, x1) in one packed two-lane add
__device__ __forceinline__ void add2(float& s0, float& s1, float x0, float x1) {
  asm("{\n\t.reg .b64 ra, rb;\n\t"
      "mov.b64 ra, {%0, %1};\n\tmov.b64 rb, {%2, %3};\n\t"
      "add.rn.f32x2 ra, ra, rb;\n\tmov.b64 {%0, %1}, ra;\n\t}"
      : "+f"(s0), "+f"(s1)
      : "f"(x0), "f"(x1));
}

template <typename T>
__global__ void __launch_bounds__(kPfThreads, 1)
    prefill_tc_kernel(const __grid_constant__ CUtensorMap tmap_q, const __grid_constant__ CUtensorMap tmap_k,
                      const __grid_constant__ CUtensorMap tmap_v, const PfParams p) {
  // All shared memory is dynamic (no static __shared__ variables), so its
  // base is the start of the CTA's shared window, which is 1024-aligned as
  // the 128-byte swizzle needs; the kernel checks rather than assumes it.
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  if (smem_u32(smem_raw) & 1023u) {
    if (threadIdx.x == 0) flag_error(p.debug_err, PA_DEVERR_LAYOUT);
    return;
  }
  unsigned char* const sm = smem_raw;

  // Work order. CTAs start in launch order (x fastest), so the launch index
  // L is mapped to the heaviest work first: sequences by decreasing work
  // n (2 ctx - n), within a sequence the query-tile pairs from the last (the
  // most keys) down, the KV heads fastest. This is list scheduling in
  // decreasing order, which keeps long CTAs out of the last wave.
  const int L = blockIdx.x + gridDim.x * (blockIdx.y + gridDim.y * blockIdx.z);
  const int kvh = L % gridDim.y;
  const int pair = gridDim.x - 1 - (L / gridDim.y) % gridDim.x;
  int seq = L / (gridDim.x * gridDim.y);
  if (gridDim.z > 1 && gridDim.z <= kRankMaxSeqs) {
    // the K ring is not in use yet: it holds each sequence's work
    unsigned long long* w = reinterpret_cast<unsigned long long*>(sm + kGroups * kTile);
    int& s_seq = *reinterpret_cast<int*>(sm + kGroups * kTile + kRankMaxSeqs * 8);
    const int nseq = gridDim.z;
    for (int i = threadIdx.x; i < nseq; i += blockDim.x) {
      int qi, ni;
      query_rows(p, i, qi, ni);
      const int ci = p.context_lens[i];
      w[i] = (ni > 0 && ci >= ni) ? static_cast<unsigned long long>(ni) * (2ull * ci - ni) : 0ull;
    }
    __syncthreads();
    for (int i = threadIdx.x; i < nseq; i += blockDim.x) {
      const unsigned long long wi = w[i];
      int rank = 0;
      for (int j = 0; j < nseq; ++j) {
        const unsigned long long wj = w[j];
        rank += (wj > wi || (wj == wi && j < i)) ? 1 : 0;
      }
      if (rank == seq) s_seq = i;  // ranks are a permutation: one writer
    }
    fence_proxy_async_smem();  // the ring is written by TMA later
    __syncthreads();
    seq = s_seq;
  }
  int q0, n;
  if (query_rows(p, seq, q0, n) && threadIdx.x == 0)
    flag_error(p.debug_err, PA_DEVERR_QUERY_START);
  const int G = p.group, TQ = p.tokens_per_tile;
  const int t0 = pair * kGroups * TQ;  // first query of the CTA's two tiles
  if (t0 >= n) return;                 // CTA-uniform, before any TMEM is held
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
  // Q[2] (32 KiB each) | K[kStages] | V[kStages] (16 KiB each) | barriers |
  // row exchange
  const uint32_t sQ0 = smem_u32(sm);
  const uint32_t sK0 = sQ0 + kGroups * kTile;
  const uint32_t sV0 = sK0 + kStages * kKVTile;
  unsigned char* const pV0 = sm + kGroups * kTile + kStages * kKVTile;
  constexpr int kTiles = kGroups * kTile + 2 * kStages * kKVTile;
  // barrier counts: kLoaders for a K or V tile (one arrival per issuing
  // thread), 1 for Q and the tensor-core completions, kGroupThreads for one
  // softmax group's threads (P written)
  enum {
    kQ,
    kKFull,
    kKFree = kKFull + kStages,
    kVFull = kKFree + kStages,
    kVFree = kVFull + kStages,
    kSFull = kVFree + kStages,      // [group][S buffer]: S computed
    kOFull = kSFull + 2 * kGroups,  // [group]: the group's PV products so far done
    kSFree = kOFull + kGroups,      // [group][S buffer]: the PV that read its P done
    kPFull = kSFree + 2 * kGroups,  // [group][S buffer]: P written
    kNumBars = kPFull + 2 * kGroups
  };
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + kTiles);
  uint32_t& tmem_slot = *reinterpret_cast<uint32_t*>(sm + kTiles + 512);
  int& s_abort = *reinterpret_cast<int*>(sm + kTiles + 516);
  // per row: each half's max, then its sum
  float(*s_half)[2][kRowsPerGroup] = reinterpret_cast<float(*)[2][kRowsPerGroup]>(sm + kTiles + 1024);
  static_assert(kNumBars * 8 <= 512, "barriers fit their slot");
  static_assert(kTiles + 1024 + kGroups * 2 * kRowsPerGroup * 4 <= kSmemBytes, "shared memory layout");
  auto bar = [&](int i) { return smem_u32(&bars[i]); };
  volatile int* abort = &s_abort;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kNumBars; ++i) {
      const bool tile_full = (i >= kKFull && i < kKFree) || (i >= kVFull && i < kVFree);
      mbar_init(bar(i), i >= kPFull ? static_cast<uint32_t>(kGroupThreads) : tile_full ? static_cast<uint32_t>(kLoaders) : 1u);
    }
    mbar_init_fence();
    s_abort = 0;
  }
  if (warp == 0) tmem_alloc(smem_u32(&tmem_slot), kTmemCols);
  tc05_fence_before();
  __syncthreads();
  tc05_fence_after();
  // group g: S[0], S[1] at columns 256g, 256g + 64 (64 each), O at 256g + 128;
  // P of S buffer b in its first 32 columns
  const uint32_t tmem = tmem_slot;

  // the keys the CTA needs: 0 .. position of its last query
  const int t_last = min(t0 + kGroups * TQ, n) - 1;
  const int pos_last = ctx - n + t_last;
  const int nkt = pos_last / kPfKeys + 1;
  const int blocks_per_tile = kPfKeys / bs;
  const int32_t* trow0 = p.block_tables + static_cast<int64_t>(seq) * p.max_blocks_per_seq;

  // Block-table entries reach the loaders 32 at a time (lane l of a loader
  // warp holds entry 32c + l of chunk c, one chunk read ahead), so the table
  // read's latency is not paid once per tile. A tile's entries are lanes
  // (kt % tiles_per_chunk) * blocks_per_tile + j.
  const int tiles_per_chunk = 32 / blocks_per_tile;  // block_size in {8, 16, 32, 64}
  const int nblk = (ctx + bs - 1) / bs;
  auto fetch_chunk = [&](int c) -> int {
    const int i = c * 32 + lane;
    return i < nblk ? __ldg(trow0 + i) : 0;
  };

  // TMA of loader q's share of one K or V tile: one 64-column box per block
  // and half, box i = 2j + h issued by loader i % kLoaders; every loader
  // arrives on the full barrier once (its count), with the bytes of its own
  // boxes
  auto load_tile = [&](const CUtensorMap* map, int q, uint32_t dst, uint32_t full, uint32_t freed,
                       uint32_t free_par, bool wait_free, int kt, const int (&ent)[kPfKeys / 8]) -> bool {
    const int lb0 = kt * blocks_per_tile;
    bool use[kPfKeys / 8];
    uint32_t nbox = 0;
#pragma unroll
    for (int j = 0; j < kPfKeys / 8; ++j) {
      use[j] = j < blocks_per_tile && lb0 + j < nblk;
      if (use[j] && (ent[j] < 0 || ent[j] >= p.num_blocks)) {
        flag_error(p.debug_err, PA_DEVERR_BLOCK_RANGE);
        use[j] = false;
      }
#pragma unroll
      for (int h = 0; h < 2; ++h) nbox += (use[j] && (2 * j + h) % kLoaders == q) ? 1u : 0u;
    }
    if (wait_free && !pf_wait(freed, free_par, abort)) return false;
    mbar_arrive_expect_tx(full, nbox * bs * 128u);
#pragma unroll
    for (int j = 0; j < kPfKeys / 8; ++j) {
      if (!use[j]) continue;
      const int z = ent[j] * p.num_kv_heads + kvh;
#pragma unroll
      for (int h = 0; h < 2; ++h)
        if ((2 * j + h) % kLoaders == q) tma_load_3d(dst + h * kKVHalf + j * bs * 128, map, h * 64, 0, z, full);
    }
    return true;
  };

  constexpr uint32_t kAB = std::is_same<T, bf16>::value ? 1u : 0u;
  if (warp >= kSoftThreads / 32) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRoleRegs));
    // ====== roles: K loaders (+Q), V loaders, S issue, PV issue ======
    const int role = warp - kSoftThreads / 32;
    if (role < 2 * kLoadWarps) {
      // K (the first kLoadWarps role warps; the first also loads Q) or V
      // tiles into a ring of kStages buffers, each refilled once both
      // products of the tile kStages back have read it
      const bool is_k = role < kLoadWarps;
      const int lw = is_k ? role : role - kLoadWarps;
      if (is_k && lw == 0 && lane == 0) {
        mbar_arrive_expect_tx(bar(kQ), 4u * kHalf);
        for (int g = 0; g < kGroups; ++g)
          for (int h = 0; h < 2; ++h)
            tma_load_3d(sQ0 + g * kTile + h * kHalf, &tmap_q, h * 64, kvh * G, q0 + t0 + g * TQ, bar(kQ));
      }
      const CUtensorMap* map = is_k ? &tmap_k : &tmap_v;
      const uint32_t dst0 = is_k ? sK0 : sV0;
      const int full = is_k ? kKFull : kVFull, freed = is_k ? kKFree : kVFree;
      int cur = fetch_chunk(0), nxt = fetch_chunk(1);
      for (int kt = 0; kt < nkt; ++kt) {
        const int st = kt % kStages, slot = kt % tiles_per_chunk;
        if (slot == 0 && kt > 0) {
          cur = nxt;
          nxt = fetch_chunk(kt / tiles_per_chunk + 1);
        }
        int ent[kPfKeys / 8];
#pragma unroll
        for (int j = 0; j < kPfKeys / 8; ++j) ent[j] = __shfl_sync(0xffffffffu, cur, (slot * blocks_per_tile + j) & 31);
        bool go = true;
        if (lane < kLoadLanes)
          go = load_tile(map, lw + kLoadWarps * lane, dst0 + st * kKVTile, bar(full + st), bar(freed + st), ((kt / kStages) - 1) & 1,
                         kt >= kStages, kt, ent);
        if (!__all_sync(0xffffffffu, go)) break;
      }
    } else if (lane == 0 && role == 2 * kLoadWarps) {
      // S[g][kt % 2] = Q[g] K^T for both groups once K arrived and the PV
      // product that read the P in that S buffer two tiles back is done
      constexpr uint32_t idesc_s = mma_idesc_f16(kAB, 0, kPfRows, kPfKeys);
      bool go = pf_wait(bar(kQ), 0, abort);
      for (int kt = 0; go && kt < nkt; ++kt) {
        const int st = kt % kStages, b = kt & 1;
        go = pf_wait(bar(kKFull + st), (kt / kStages) & 1, abort);
        for (int g = 0; go && g < kGroups; ++g) {
          if (kt >= 2 && !(go = pf_wait(bar(kSFree + 2 * g + b), ((kt - 2) >> 1) & 1, abort))) break;
          tc05_fence_after();
#pragma unroll
          for (int k = 0; k < kPfD / 16; ++k) {
            tc05_mma_ss(tmem + g * 256 + b * kPfKeys,
                        smem_desc_sw128(sQ0 + g * kTile + (k >> 2) * kHalf + (k & 3) * 32, 16, 1024),
                        smem_desc_sw128(sK0 + st * kKVTile + (k >> 2) * kKVHalf + (k & 3) * 32, 16, 1024),
                        idesc_s, k > 0);
          }
          tc05_commit(bar(kSFull + 2 * g + b));
        }
        if (go) tc05_commit(bar(kKFree + st));
      }
    } else if (lane == 0 && role == 2 * kLoadWarps + 1) {
      // O[g] += P[g] V for both groups once V arrived and the group wrote P
      // (A = P from tensor memory, 16 keys = 8 columns per step)
      constexpr uint32_t idesc_o = mma_idesc_f16(kAB, 1, kPfRows, kPfD);
      bool go = true;
      for (int kt = 0; go && kt < nkt; ++kt) {
        const int st = kt % kStages, b = kt & 1;
        go = pf_wait(bar(kVFull + st), (kt / kStages) & 1, abort);
        for (int g = 0; go && g < kGroups; ++g) {
          if (!(go = pf_wait(bar(kPFull + 2 * g + b), (kt >> 1) & 1, abort))) break;
          tc05_fence_after();
#pragma unroll
          for (int k = 0; k < kPfKeys / 16; ++k) {
            tc05_mma_ts(tmem + g * 256 + 128, tmem + g * 256 + b * kPfKeys + k * 8,
                        smem_desc_sw128(sV0 + st * kKVTile + k * 16 * 128, kKVHalf, 1024), idesc_o,
                        (kt > 0 || k > 0) ? 1u : 0u);
          }
          tc05_commit(bar(kOFull + g));
          tc05_commit(bar(kSFree + 2 * g + b));
        }
        if (go) tc05_commit(bar(kVFree + st));
      }
    }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kSoftRegs));
    // ====== softmax: group g = query tile g, two threads per row ======
    const int g = warp / 8;
    const int wg = warp % 8;
    const int r = (wg & 3) * 32 + lane;  // this thread's row of the group's tile
    const int hc = wg >> 2;              // its half of the columns
    const uint32_t lane_base = static_cast<uint32_t>((wg & 3) * 32) << 16;
    const uint32_t tmem_o = tmem + g * 256 + 128 + hc * (kPfD / 2);
    const int c0 = hc * (kPfKeys / 2);  // this thread's 32 keys of a tile
    // named barriers 3 + 2g + h: half h's exchange slot has been read by
    // the other half (half h waits on it before rewriting the slot)
    const int bar_mine = 3 + 2 * g + hc, bar_other = 3 + 2 * g + (1 - hc);
    const int tg0 = t0 + g * TQ;        // the group's first query
    // this row's query position (rows past the chunk repeat the last
    // position; they are not stored)
    const int my_t = min(tg0 + r / G, n - 1);
    const int my_pos = ctx - n + my_t;
    const int pos_first = ctx - n + min(tg0, n - 1);  // the group's earliest query position
    float m_run = -INFINITY, l_run = 0.f;
    // All threads of a group run every iteration and every named barrier,
    // also after a timeout (then they skip the work); `ok` is kept
    // warp-uniform for the warp-collective TMEM accesses.
    bool ok = true;
    for (int kt = 0; kt < nkt; ++kt) {
      const int b = kt & 1, st = kt % kStages;
      ok = __all_sync(0xffffffffu, ok && pf_wait(bar(kSFull + 2 * g + b), (kt >> 1) & 1, abort));
      const int key0 = kt * kPfKeys;
      float x[32];
      if (ok) {
        tc05_fence_after();
        uint32_t v[32];
        tmem_ld32(tmem + g * 256 + b * kPfKeys + c0 + lane_base, v);
        tmem_wait_ld();
#pragma unroll
        for (int j = 0; j < 32; ++j) x[j] = __uint_as_float(v[j]);
      } else {
#pragma unroll
        for (int j = 0; j < 32; ++j) x[j] = 0.f;
      }
      // only tiles that reach past the group's earliest query need the mask
      if (key0 + kPfKeys - 1 > pos_first) {
#pragma unroll
        for (int j = 0; j < 32; ++j)
          if (key0 + c0 + j > my_pos) x[j] = -INFINITY;
      }
      float mraw = max3(x[0], x[1], x[2]);
#pragma unroll
      for (int j = 3; j < 31; j += 2) mraw = max3(mraw, x[j], x[j + 1]);
      mraw = fmaxf(mraw, x[31]);
      // the row's two halves exchange their maxima through one slot each: a
      // slot is rewritten only after the other half has read it (bar_read)
      if (kt > 0) named_sync(bar_mine, kGroupThreads);
      s_half[g][hc][r] = mraw;
      // this barrier also orders both halves' S loads before either half's
      // P store into the same columns
      tc05_fence_before();
      named_sync(1 + g, kGroupThreads);
      tc05_fence_after();
      const float mx = fmaxf(s_half[g][0][r], s_half[g][1][r]) * p.scale_log2;  // scale > 0
      named_arrive(bar_other, kGroupThreads);
      float m_use = m_run, alpha = 1.f;
      if (mx > m_run + kLazyRescale || m_run == -INFINITY) {
        m_use = fmaxf(m_run, mx);
        alpha = m_run == -INFINITY ? 0.f : ex2_ftz(m_run - m_use);
      }
      const float nbase = m_use == -INFINITY ? 0.f : -m_use;
      float s0 = 0.f, s1 = 0.f;
#pragma unroll
      for (int j = 0; j < 32; j += 2) {
        exp_arg2(x[j], x[j + 1], p.scale_log2, nbase);
        x[j] = ex2_ftz(x[j]);
        x[j + 1] = ex2_ftz(x[j + 1]);
        add2(s0, s1, x[j], x[j + 1]);
      }
      l_run = l_run * alpha + (s0 + s1);  // this half's share of the row sum
      m_run = m_use;
      // P, 16-bit, two keys per column: this half's 32 keys go to columns
      // 16 hc .. 16 hc + 15 of the S buffer they came from
      uint32_t pw[16];
#pragma unroll
      for (int j = 0; j < 16; ++j) pw[j] = pack2<T>(x[2 * j], x[2 * j + 1]);
      // keys past the context in the last tile: zero their V rows (stale or
      // unwritten shared memory must not meet a zero weight as NaN); group 0
      // does it, before its P is signalled, and the PV issuer serves group 0
      // first
      const int valid = ctx - key0;
      if (g == 0 && valid < kPfKeys) {
        ok = ok && pf_wait(bar(kVFull + st), (kt / kStages) & 1, abort);
        unsigned char* vt = pV0 + st * kKVTile;
        for (int i = hc * kRowsPerGroup + r; ok && i < (kPfKeys - valid) * 16; i += kGroupThreads) {
          const int row = valid + i / 16, chunk = i % 16;
          *reinterpret_cast<uint4*>(vt + (chunk >> 3) * kKVHalf + row * 128 + (((chunk & 7) ^ (row & 7)) << 4)) =
              make_uint4(0u, 0u, 0u, 0u);
        }
        fence_proxy_async_smem();  // the PV product reads these rows
        ok = __all_sync(0xffffffffu, ok);
      }
      if (ok) tmem_st16(tmem + g * 256 + b * kPfKeys + hc * 16 + lane_base, pw);
      // O *= alpha, once the group's previous PV product is complete. Only a
      // warp whose running max moved waits for it; otherwise the softmax runs
      // ahead of the PV products.
      const bool resc = kt > 0 && __any_sync(0xffffffffu, alpha != 1.f);
      if (resc) ok = __all_sync(0xffffffffu, ok && pf_wait(bar(kOFull + g), (kt - 1) & 1, abort));
      if (ok && resc) {
        tc05_fence_after();
#pragma unroll
        for (int c = 0; c < kPfD / 2; c += 32) {
          uint32_t v[32];
          tmem_ld32(tmem_o + lane_base + c, v);
          tmem_wait_ld();
#pragma unroll
          for (int j = 0; j < 32; ++j) v[j] = __float_as_uint(__uint_as_float(v[j]) * alpha);
          tmem_st32(tmem_o + lane_base + c, v);
        }
      }
      if (ok) {
        tmem_wait_st();
        tc05_fence_before();
        mbar_arrive(bar(kPFull + 2 * g + b));
      }
    }
    ok = __all_sync(0xffffffffu, ok && pf_wait(bar(kOFull + g), (nkt - 1) & 1, abort));
    // ---- out = O / l for the rows of the chunk ----
    named_sync(bar_mine, kGroupThreads);
    s_half[g][hc][r] = l_run;
    named_sync(1 + g, kGroupThreads);
    if (ok) {
      tc05_fence_after();
      const float l = s_half[g][0][r] + s_half[g][1][r];
      const float inv = l > 0.f ? 1.f / l : 0.f;
      const int tok = tg0 + r / G;
      T* orow = static_cast<T*>(p.out) +
                (static_cast<int64_t>(q0 + min(tok, n - 1)) * p.num_heads + kvh * G + r % G) * kPfD + hc * (kPfD / 2);
#pragma unroll
      for (int c = 0; c < kPfD / 2; c += 32) {
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
    }
  }

  tc05_fence_before();
  __syncthreads();
  if (s_abort) {
    if (threadIdx.x == 0) {
      flag_error(p.debug_err, PA_DEVERR_TIMEOUT);
      // let tensor-core work already issued finish before its TMEM goes away
      for (int i = 0; i < kGroups; ++i) mbar_wait_bounded(bar(kOFull + i), 0, 10000000ull);
      for (int i = 0; i < 2 * kGroups; ++i) mbar_wait_bounded(bar(kSFull + i), 0, 10000000ull);
    }
    __syncthreads();
  }
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

template <int R>
bool encode(CUtensorMap* map, const void* base, const cuuint64_t (&dims)[R], const cuuint64_t (&strides)[R - 1],
            const cuuint32_t (&box)[R]) {
  auto fn = pf_encode_fn();
  if (fn == nullptr) return false;
  cuuint32_t es[R];
  for (int i = 0; i < R; ++i) es[i] = 1;
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT16, R, const_cast<void*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool prefill_supported(int group, int head_dim, pa_dtype dtype, int block_size) {
  return head_dim == kPfD && (dtype == PA_F16 || dtype == PA_BF16) &&
         (group == 1 || group == 2 || group == 4 || group == 8) &&
         (block_size == 8 || block_size == 16 || block_size == 32 || block_size == 64);
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
  pp.num_tokens = num_tokens;
  pp.num_heads = num_heads;
  pp.num_kv_heads = num_kv_heads;
  pp.block_size = block_size;
  pp.num_blocks = num_blocks;
  pp.group = G;
  pp.tokens_per_tile = kPfRows / G;
  pp.scale_log2 = scale * 1.4426950408889634f;
  CUtensorMap mq, mk, mv;
  const cuuint64_t row = static_cast<cuuint64_t>(kPfD) * 2;
  if (!encode<3>(&mq, q,
                 {static_cast<cuuint64_t>(kPfD), static_cast<cuuint64_t>(num_heads),
                  static_cast<cuuint64_t>(num_tokens)},
                 {row, row * num_heads}, {64, static_cast<cuuint32_t>(G), static_cast<cuuint32_t>(kPfRows / G)}))
    return cudaErrorInvalidValue;
  const cuuint64_t bxh = static_cast<cuuint64_t>(num_blocks) * num_kv_heads;
  const cuuint64_t bsz = static_cast<cuuint64_t>(block_size);
  const cuuint32_t bsb = static_cast<cuuint32_t>(block_size);
  // K and V: (column, row, block x head), one 64-column half of a block per box
  const cuuint64_t kdims[3] = {static_cast<cuuint64_t>(kPfD), bsz, bxh};
  const cuuint64_t kstr[2] = {row, row * bsz};
  const cuuint32_t kbox[3] = {64, bsb, 1};
  if (!encode<3>(&mk, k_cache, kdims, kstr, kbox) || !encode<3>(&mv, v_cache, kdims, kstr, kbox))
    return cudaErrorInvalidValue;
  const int tiles = (max_query_len + pp.tokens_per_tile - 1) / pp.tokens_per_tile;
  dim3 grid((tiles + kGroups - 1) / kGroups, num_kv_heads, num_seqs);
  cudaError_t err;
  if (dtype == PA_BF16) {
    static std::atomic<unsigned long long> set{0};
    err = set_smem_limit_once(reinterpret_cast<const void*>(prefill_tc_kernel<bf16>), kSmemBytes, set);
    if (err != cudaSuccess) return err;
    prefill_tc_kernel<bf16><<<grid, kPfThreads, kSmemBytes, stream>>>(mq, mk, mv, pp);
  } else {
    static std::atomic<unsigned long long> set{0};
    err = set_smem_limit_once(reinterpret_cast<const void*>(prefill_tc_kernel<f16>), kSmemBytes, set);
    if (err != cudaSuccess) return err;
    prefill_tc_kernel<f16><<<grid, kPfThreads, kSmemBytes, stream>>>(mq, mk, mv, pp);
  }
  err = cudaGetLastError();
  if (err == cudaSuccess) note_launches(1);
  return err;
}

}  // namespace pa
