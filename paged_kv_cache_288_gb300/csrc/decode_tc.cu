// Paged decode on the tensor cores, for GQA groups of 2, 4 or 8 query heads.
//
// Work. The context of every (sequence, KV head) is cut into 16-token tiles;
// all tiles of the batch form one flat list ordered (sequence, KV head,
// tile). Each warp of a persistent grid (8 warps per CTA, one CTA per SM)
// takes an equal contiguous share of that list, so every warp streams the
// same number of KV bytes whatever the mix of context lengths. A warp's share
// is a run of "pieces", one per (sequence, KV head) it touches; only the
// first and last piece can be partial. A warp that holds a whole (sequence,
// KV head) writes its output rows; partial pieces leave their online-softmax
// state (running max, running sum, unnormalised accumulator) in the
// workspace and tc_merge_kernel combines them. With a forced partition size
// the list is cut at partition boundaries instead, every piece is one whole
// partition, and the partition reduce of the split path combines them.
//
// Data movement. Each warp owns a ring of shared-memory slots, one 16-token
// K tile plus V tile per slot. It fetches its own tiles with 3-D TMA loads
// (box = 128 bytes of a row x up to 16 rows of one block of one KV head, 128B
// swizzle), completing on one mbarrier per slot, and runs as many tiles ahead
// as it has slots. Physical block ids come from the block table through a
// 32-entry window held one entry per lane.
//
// Math. With G query heads per KV head, S^T = K Q^T is a 16x16 by 16x8
// product per 16 d-columns (tokens in M, heads in N, G of the 8 columns
// used), issued as mma.sync m16n8k16 with float accumulators; P^T is moved
// from the accumulator layout into the B-operand layout with movmatrix; then
// O^T = V^T P^T, again m16n8k16, with V^T fragments read by ldmatrix.trans.
// The online softmax runs in log2 units on the accumulator fragments. E4M3
// tiles are widened to f16 in registers (K through a consistent permutation
// of the contraction index, V through one of the d rows) and their block
// scales are applied to S and to P.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <atomic>
#include <mutex>
#include <type_traits>

#include "common.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace pa {
namespace {

constexpr int kWarps16 = 8;     // warps of a CTA, 16-bit caches
constexpr int kWarpsFp8 = 12;   // warps of a CTA, E4M3 caches
constexpr int kMaxWarps = 12;   // the most of either (sizes the workspace)
constexpr int kRowTile = 16;   // MMA M: tokens per row tile
constexpr int kMaxG = 8;       // MMA N
constexpr uint32_t kFull = 0xffffffffu;
// inputs larger than this are not warmed into the L2 at the start of a call
constexpr int64_t kWarmBytes = 16ll << 20;

// A tile is TT tokens (16 or 32, one or two MMA row tiles) of one
// (sequence, KV unit): TT rows of K and TT rows of V of each of the unit's HP
// KV heads in one ring slot (head h's rows after head h-1's).
template <typename KT, int D, int TT, int HP = 1>
struct Geom {
  static constexpr int kElem = int(sizeof(KT));
  static constexpr int kRowBytes = D * kElem;
  static constexpr int kBoxW = 128 / kElem;        // elements in one 128-byte box row
  static constexpr int kBoxes = kRowBytes / 128;   // boxes across a row
  static constexpr int kBoxBytes = TT * HP * 128;  // one 128-byte column of the tile
  static constexpr int kRowTiles = TT / kRowTile * HP;  // 16-row tiles of K (or V) in a slot
  static constexpr uint32_t kFullMask = TT == 32 ? 0xffffffffu : 0xffffu;
  static constexpr int kTileBytes = TT * HP * kRowBytes;
  static constexpr int kSlotBytes = 2 * kTileBytes;
  // E4M3 tiles carry more conversion work per byte, so an SM runs more of
  // their warps (each with a shorter ring) to hide its latencies
  static constexpr int kWarps = kElem == 1 ? kWarpsFp8 : kWarps16;
  static constexpr int kSlots = kElem == 1 ? (kWarpsFp8 > 8 ? 2 : 3) : (kSlotBytes >= 8192 ? 3 : 6);
  static constexpr int kSteps = D / 16;            // 16-column steps of QK^T and PV
};

struct SlotMeta {
  float ks[4];    // E4M3 K scale of tokens 8i .. 8i+7
  float vs[4];    // E4M3 V scale
  uint32_t mask;  // bit t: token t of the tile holds data
  uint32_t pad[3];
};

struct TcParams {
  DecodeParams p;
  PrefixGroups pg;     // shared-prefix groups (group_start == nullptr: none)
  float* ws_slots;     // [6 * num_warps][group * (D + 2)] partial states (auto schedule)
  int32_t* claim;      // chunk counter of the auto schedule: 0 on entry, reset by the merge
  int32_t num_warps;   // warps that share the work
  int32_t part_tiles;  // tiles per partition (split path); 0 = auto schedule
  int32_t group;       // query heads per KV head
  int32_t short_share;  // static share /256 of short lists; 0 for MQA's split units
};

// The auto schedule: the first S of the U tiles are split evenly over the W
// warps (warp w: [w*S/W, (w+1)*S/W)); the rest are chunks of C >= kMinChunk
// tiles that warps claim from a counter when their share is done, so SMs
// that stream faster take more of them. At most 2W chunks.
// S is kStatic256/256 of U. When every unit is one KV head (or an E4M3 head
// pair) it is a shorter share for lists of fewer than kShortShare tiles per
// warp (kStatic256Short16/256 for 16-bit caches, kStatic256ShortFp8/256 for
// E4M3) and kStatic256Long/256 for longer ones. Measured:
// - 16-bit, short lists: the Llama-8B-shaped batch 92.8 us with 160 against
//   94.5 with 192; later 87.9 with 144, 89.5 with 160, 90.7 with 128; the
//   shared-prefix batch's suffixes 55.2 with 144 against 56.0 with 160.
// - E4M3 head pairs (about 18 tiles per warp): 70.9 with 160, 72.0 with 192,
//   77.0 with 144, 79.3 with 128.
// - long context bs 16 (108 tiles per warp): 167.1 with 224, 168.9 with 192.
// MQA's units of 8 query heads keep 192: the four units of a KV head gain
// from running side by side.
constexpr int kStatic256 = 192;
constexpr int kStatic256Short16 = 144;
constexpr int kStatic256ShortFp8 = 160;
constexpr int kStatic256Long = 224;
constexpr int64_t kShortShare = 64;
constexpr int64_t kMinChunk = 8;

struct Sched {
  int64_t S, C, K;
};

// short_share: the static share /256 of short lists, 0 for MQA's split units
__device__ __forceinline__ Sched make_sched(int64_t U, int64_t W, int short_share) {
  Sched sc;
  sc.S = U * (short_share == 0 ? kStatic256 : U < kShortShare * W ? short_share : kStatic256Long) / 256;
  const int64_t rest = U - sc.S;
  int64_t c = (rest + 2 * W - 1) / (2 * W);
  sc.C = c < kMinChunk ? kMinChunk : c;
  sc.K = (rest + sc.C - 1) / sc.C;
  return sc;
}

// Byte address of 16-byte chunk `chunk` of row `row` in a tile whose
// 128-byte columns are box_bytes apart (boxes of 8, 16 or 32 rows of one
// block stack in row order), chunks XOR-swizzled by row % 8 as the TMA 128B
// swizzle stores them.
template <int box_bytes>
__device__ __forceinline__ uint32_t tile_addr(uint32_t base, int row, int chunk) {
  return base + (chunk >> 3) * box_bytes + row * 128 + (((chunk & 7) ^ (row & 7)) << 4);
}

// Tiles of a sequence whose first `start` tokens are left to the shared-prefix
// kernel: tokens [start - start % TT, ctx) in tiles of TT (the tokens below
// `start` of the first tile are masked).
template <int TT>
__device__ __forceinline__ int seq_tiles(int ctx, int start) {
  if (ctx <= start) return 0;
  const int lo = start - start % TT;
  return (ctx - lo + TT - 1) / TT;
}

// Shared-prefix tokens of sequence i: the prefix of the group whose range
// holds it (binary search over group_start, which a valid description keeps
// non-decreasing), 0 outside every group.
__device__ __forceinline__ int seq_prefix_len(const PrefixGroups& pg, const DecodeParams& p, int i,
                                              int& group_len) {
  group_len = 0;
  if (pg.group_start == nullptr || pg.num_groups <= 0) return 0;
  int lo = 0, hi = pg.num_groups - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (pg.group_start[mid] <= i) lo = mid; else hi = mid - 1;
  }
  int a, b, len;
  prefix_group(pg, lo, p.num_seqs, p.max_blocks_per_seq, p.block_size, a, b, len);
  if (i < a || i >= b) return 0;
  group_len = len;
  return len;
}

// Bits [first, first + n) set, n <= 32.
__device__ __forceinline__ uint32_t bit_range(int first, int n) {
  return (n >= 32 ? 0xffffffffu : ((1u << n) - 1u)) << first;
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}
__device__ __forceinline__ uint32_t pack_f16(float lo, float hi) {
  __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

// Keep the 16-bit halves of a (token t, token t+1) register whose token holds data.
__device__ __forceinline__ uint32_t keep_tokens(uint32_t v, uint32_t mask, int t) {
  const uint32_t lo = (mask >> t) & 1u ? 0x0000ffffu : 0u;
  const uint32_t hi = (mask >> (t + 1)) & 1u ? 0xffff0000u : 0u;
  return v & (lo | hi);
}

// Position in the flat tile list, walked tile by tile.
struct Cursor {
  int64_t f;  // flat index
  int seq, kvh, t, tiles;
};

__device__ __forceinline__ int find_seq(const int* pref, int B, int Hkv, int64_t f) {
  int lo = 0, hi = B - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (static_cast<int64_t>(pref[mid]) * Hkv <= f) lo = mid; else hi = mid - 1;
  }
  return lo;
}

__device__ __forceinline__ void cursor_at(Cursor& c, int64_t f, const int* prefT, int B, int Hkv) {
  c.f = f;
  c.seq = find_seq(prefT, B, Hkv, f);
  c.tiles = prefT[c.seq + 1] - prefT[c.seq];
  const int64_t r = f - static_cast<int64_t>(prefT[c.seq]) * Hkv;
  c.kvh = static_cast<int>(r / c.tiles);
  c.t = static_cast<int>(r % c.tiles);
}

__device__ __forceinline__ void cursor_next(Cursor& c, const int* prefT, int B, int Hkv) {
  ++c.f;
  if (++c.t < c.tiles) return;
  c.t = 0;
  if (++c.kvh < Hkv) return;
  c.kvh = 0;
  do {
    ++c.seq;
  } while (c.seq < B && prefT[c.seq + 1] == prefT[c.seq]);
  if (c.seq < B) c.tiles = prefT[c.seq + 1] - prefT[c.seq];
}

template <typename QT, typename KT, int D, int TT, int HP>
__global__ void __launch_bounds__(Geom<KT, D, TT, HP>::kWarps * 32, 1)
decode_tc_kernel(const __grid_constant__ CUtensorMap tmap_k,
                 const __grid_constant__ CUtensorMap tmap_v, const TcParams tp) {
  using Gm = Geom<KT, D, TT, HP>;
  constexpr int kWarps = Gm::kWarps;
  constexpr int kThreads = kWarps * 32;
  constexpr int RT = Gm::kRowTiles;   // 16-row tiles of K (or V) in a slot
  constexpr int RS = TT / kRowTile;   // 16-token tiles of S
  constexpr bool kFp8 = is_fp8<KT>::value;
  constexpr int NS = Gm::kSlots;
  const DecodeParams& p = tp.p;
  const int B = p.num_seqs;
  const int Hkv = p.num_kv_heads;
  const int G = tp.group;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int g = lane >> 2;   // MMA group id: accumulator row, B-operand column
  const int tig = lane & 3;  // thread in group
  // HP = 2: a unit is two KV heads of G / 2 query heads each; MMA column c
  // belongs to the unit's KV head c / (G / 2). This lane's B-operand column
  // is g, its accumulator columns 2 tig and 2 tig + 1 (one KV head: G / 2 is
  // 2 or 4).
  const int hd_b = HP == 2 ? g / (G >> 1) : 0;
  const int hd_c = HP == 2 ? min((2 * tig) / (G >> 1), 1) : 0;

  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  unsigned char* slots = smem;
  SlotMeta* meta = reinterpret_cast<SlotMeta*>(slots + kWarps * NS * Gm::kSlotBytes);
  uint64_t* bars = reinterpret_cast<uint64_t*>(meta + kWarps * NS);
  int* s_ctx = reinterpret_cast<int*>(bars + kWarps * NS);
  int* s_prefT = s_ctx + B;
  int* s_prefP = s_prefT + B + 1;
  // tokens of each sequence left to the shared-prefix kernel; only with groups,
  // which never come with a forced partition size, so it reuses s_prefP
  const bool prefix_mode = tp.pg.group_start != nullptr;
  int* s_start = s_prefP;
  auto start_of = [&](int i) -> int { return prefix_mode ? s_start[i] : 0; };
  __shared__ int s_warp_sum[kWarps][2];
  __shared__ int64_t s_queue[kWarps][NS + 1][3];  // claimed ranges waiting: start, end, first slot

  if (threadIdx.x < kWarps * NS) mbar_init(smem_u32(&bars[threadIdx.x]), 1);
  if (threadIdx.x == 0) {
    prefetch_tensormap(&tmap_k);
    prefetch_tensormap(&tmap_v);
  }
  mbar_init_fence();
  griddep_wait();
  // Warm the L2 with the call's small inputs: q, the block tables and the
  // E4M3 scales, a 128-byte line per thread of the grid at a time. Every
  // warp's first tiles and q rows need them at once, and from HBM those
  // loads would queue behind the first tiles' own traffic.
  {
    const int64_t nthr = static_cast<int64_t>(gridDim.x) * kThreads;
    const int64_t me = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x;
    auto warm = [&](const void* base, int64_t bytes) {
      if (base == nullptr || bytes > kWarmBytes) return;
      const char* b = static_cast<const char*>(base);
      for (int64_t l = me; l * 128 < bytes; l += nthr) prefetch_l2(b + l * 128);
    };
    warm(p.q, static_cast<int64_t>(B) * p.num_heads * D * static_cast<int64_t>(sizeof(QT)));
    warm(p.block_tables, static_cast<int64_t>(B) * p.max_blocks_per_seq * 4);
    if constexpr (kFp8) {
      warm(p.k_scale, static_cast<int64_t>(p.num_blocks) * p.kv_heads_phys * 4);
      warm(p.v_scale, static_cast<int64_t>(p.num_blocks) * p.kv_heads_phys * 4);
    }
  }

  // ---- per-sequence tile and partition counts, and their exclusive prefix --
  const int per = (B + kThreads - 1) / kThreads;
  const int i0 = min(B, static_cast<int>(threadIdx.x) * per);
  const int i1 = min(B, i0 + per);
  int sum_t = 0, sum_p = 0;
  for (int i = i0; i < i1; ++i) {
    s_ctx[i] = clamp_context(p, i);
    if (prefix_mode) s_start[i] = 0;
  }
  if (prefix_mode) {
    // each group's members skip its shared tokens
    __syncthreads();
    for (int g = warp; g < tp.pg.num_groups; g += kWarps) {  // a warp per group, a lane per member
      int a, b, len;
      if (prefix_group(tp.pg, g, B, p.max_blocks_per_seq, p.block_size, a, b, len) && lane == 0)
        flag_error(p.debug_err, PA_DEVERR_PREFIX);
      for (int i = a + lane; i < b; i += 32) s_start[i] = len;
    }
    __syncthreads();
  }
  for (int i = i0; i < i1; ++i) {
    const int ctx = s_ctx[i];
    if (prefix_mode && s_start[i] > ctx) {
      flag_error(p.debug_err, PA_DEVERR_PREFIX);  // a member shorter than its group's prefix
      s_start[i] = ctx;
    }
    const int tl = seq_tiles<TT>(ctx, start_of(i));
    sum_t += tl;
    if (tp.part_tiles) sum_p += (tl + tp.part_tiles - 1) / tp.part_tiles;
  }
  int inc_t = sum_t, inc_p = sum_p;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int a = __shfl_up_sync(kFull, inc_t, off);
    const int b = __shfl_up_sync(kFull, inc_p, off);
    if (lane >= off) {
      inc_t += a;
      inc_p += b;
    }
  }
  if (lane == 31) {
    s_warp_sum[warp][0] = inc_t;
    s_warp_sum[warp][1] = inc_p;
  }
  __syncthreads();
  int run_t = inc_t - sum_t, run_p = inc_p - sum_p;
  for (int w = 0; w < warp; ++w) {
    run_t += s_warp_sum[w][0];
    run_p += s_warp_sum[w][1];
  }
  for (int i = i0; i < i1; ++i) {
    const int tl = seq_tiles<TT>(s_ctx[i], start_of(i));
    s_prefT[i] = run_t;
    if (tp.part_tiles) s_prefP[i] = run_p;
    run_t += tl;
    if (tp.part_tiles) run_p += (tl + tp.part_tiles - 1) / tp.part_tiles;
  }
  if (threadIdx.x == kThreads - 1) {
    s_prefT[B] = run_t;
    if (tp.part_tiles) s_prefP[B] = run_p;
  }
  __syncthreads();
  griddep_launch_dependents();

  // ---- this warp's share of the tile list --------------------------------
  const int64_t W = tp.num_warps;
  const int64_t wid = static_cast<int64_t>(blockIdx.x) * kWarps + warp;
  if (wid >= W) return;
  const int64_t U = static_cast<int64_t>(s_prefT[B]) * Hkv;
  int64_t f0, f1;
  int64_t S = U, C = 1, K = 0;  // static tiles, chunk size, chunks
  // split path: whole partitions; partition index -> its first tile
  const int64_t US = tp.part_tiles ? static_cast<int64_t>(s_prefP[B]) * Hkv : 0;
  auto part_to_tile = [&](int64_t s) -> int64_t {
    if (s >= US) return U;
    const int seq = find_seq(s_prefP, B, Hkv, s);
    const int np = s_prefP[seq + 1] - s_prefP[seq];
    const int64_t r = s - static_cast<int64_t>(s_prefP[seq]) * Hkv;
    const int kvh = static_cast<int>(r / np);
    const int pi = static_cast<int>(r % np);
    const int tiles = s_prefT[seq + 1] - s_prefT[seq];
    return static_cast<int64_t>(s_prefT[seq]) * Hkv + static_cast<int64_t>(kvh) * tiles +
           static_cast<int64_t>(pi) * tp.part_tiles;
  };
  int64_t SP = 0;  // split path: partitions shared out statically
  if (tp.part_tiles == 0) {
    const Sched sc = make_sched(U, W, tp.short_share);
    S = sc.S;
    C = sc.C;
    K = sc.K;
    f0 = wid * S / W;
    f1 = (wid + 1) * S / W;
  } else {
    // the first kStatic256/256 of the partitions in equal shares, the rest
    // claimed one partition at a time by warps whose share is done (SMs
    // stream at different rates)
    SP = tp.claim != nullptr ? US * kStatic256 / 256 : US;
    K = US - SP;
    f0 = part_to_tile(wid * SP / W);
    f1 = part_to_tile((wid + 1) * SP / W);
  }
  // claim the next chunk of the shared tail: its tile range and first slot
  auto claim = [&](int64_t& r0, int64_t& r1, int64_t& slot0) -> bool {
    if (K == 0) return false;
    int k = 0;
    if (lane == 0) k = atomicAdd(tp.claim, 1);
    k = __shfl_sync(kFull, k, 0);
    if (k >= K) return false;
    if (tp.part_tiles) {
      r0 = part_to_tile(SP + k);
      r1 = part_to_tile(SP + k + 1);
      slot0 = 0;  // partitions write their own partials
      return true;
    }
    r0 = S + static_cast<int64_t>(k) * C;
    r1 = r0 + C < U ? r0 + C : U;
    slot0 = 2 * W + 2 * static_cast<int64_t>(k);
    return true;
  };
  int64_t cr0 = f0, cr1 = f1, cslot = 2 * wid;  // the consumer's current range
  if (cr0 >= cr1 && !claim(cr0, cr1, cslot)) return;

  const int bs = p.block_size;
  const int lbs = 31 - __clz(bs);  // block sizes are powers of two
  const int width = p.max_blocks_per_seq;
  const int Hq = p.num_heads;
  const uint32_t slot_base0 = smem_u32(slots) + warp * NS * Gm::kSlotBytes;
  SlotMeta* my_meta = meta + warp * NS;
  const uint32_t bar_base = smem_u32(bars + warp * NS);

  // block-table window: lane l holds entry win_base + l of sequence win_seq
  // and, for E4M3 caches, that block's K and V scales for KV head win_kvh
  int win_seq = -1, win_base = 0, win_val = -1, win_kvh = -1;
  float win_ks = 1.f, win_vs = 1.f, win_ks1 = 1.f, win_vs1 = 1.f;  // (HP = 2: ks1, vs1 of the second head)
  auto table_entry = [&](int seq, int kvh, int j, float& ksc, float& vsc, float& ksc1, float& vsc1) -> int {
    if (seq != win_seq || j < win_base || j >= win_base + 32) {
      win_seq = seq;
      win_base = j;
      win_kvh = -1;
      const int jj = j + lane;
      win_val = jj < width ? p.block_tables[static_cast<int64_t>(seq) * width + jj] : -1;
    }
    if constexpr (kFp8) {
      if (kvh != win_kvh) {
        win_kvh = kvh;
        const bool ok = win_val >= 0 && win_val < p.num_blocks;
        const int64_t si = static_cast<int64_t>(ok ? win_val : 0) * p.kv_heads_phys +
                           (HP == 2 ? 2 * kvh : kv_head_of(p, kvh));
        win_ks = ok ? p.k_scale[si] : 1.f;
        win_vs = ok ? p.v_scale[si] : 1.f;
        if constexpr (HP == 2) {
          win_ks1 = ok ? p.k_scale[si + 1] : 1.f;
          win_vs1 = ok ? p.v_scale[si + 1] : 1.f;
        }
      }
      ksc = __shfl_sync(kFull, win_ks, j - win_base);
      vsc = __shfl_sync(kFull, win_vs, j - win_base);
      if constexpr (HP == 2) {
        ksc1 = __shfl_sync(kFull, win_ks1, j - win_base);
        vsc1 = __shfl_sync(kFull, win_vs1, j - win_base);
      }
    }
    return __shfl_sync(kFull, win_val, j - win_base);
  };

  // Issue the TMA loads of the tile under `c` into slot `s` (whole warp):
  // one box per 128-byte column per block the tile touches (a tile lies in
  // one block when the block holds at least TT tokens, else it spans
  // TT / block_size blocks).
  constexpr int kMaxSub = TT / 8;
  // K and V are read once: their lines leave the L2 first, so the partial
  // states the merge reads, q and the tables stay there
  const uint64_t kv_policy = l2_evict_first_policy();
  const uint64_t state_policy = l2_evict_last_policy();
  auto issue = [&](const Cursor& c, int s) {
    const int ctx = s_ctx[c.seq];
    const int st = start_of(c.seq);
    const int tok0 = st - st % TT + c.t * TT;
    const int valid = min(TT, ctx - tok0);
    const int skip = st > tok0 ? st - tok0 : 0;  // leading tokens of the shared prefix
    const uint32_t kdst = slot_base0 + s * Gm::kSlotBytes;
    const uint32_t vdst = kdst + Gm::kTileBytes;
    const uint32_t bar = bar_base + s * 8;
    const int bh = bs < TT ? bs : TT;  // rows per box
    const int nsub = TT / bh;
    uint32_t mask = 0, tx = 0;
    int phys[kMaxSub];
    float ks[kMaxSub], vs[kMaxSub];
    float ks1 = 1.f, vs1 = 1.f;  // HP = 2: the second head's scales (the tile lies in one block)
    const int off = tok0 & (bs - 1);  // 0 when the tile spans blocks
#pragma unroll
    for (int h = 0; h < kMaxSub; ++h) {
      phys[h] = -1;
      ks[h] = vs[h] = 1.f;
      float k1 = 1.f, v1 = 1.f;
      const int first = h * bh;
      if (h >= nsub || first >= valid || first < skip) continue;  // skip is a multiple of bh
      phys[h] = table_entry(c.seq, c.kvh, (tok0 >> lbs) + h, ks[h], vs[h], k1, v1);
      if (HP == 2 && h == 0) {
        ks1 = k1;
        vs1 = v1;
      }
      if (phys[h] < 0 || phys[h] >= p.num_blocks) {
        if (lane == 0) flag_error(p.debug_err, PA_DEVERR_BLOCK_RANGE);
        phys[h] = -1;
        continue;
      }
      mask |= bit_range(first, min(bh, valid - first));
      tx += 2u * HP * bh * Gm::kRowBytes;
    }
    // lane 0: the slot's token mask and, for E4M3 caches, the scales of its
    // 8-token groups (vector stores), then the expected bytes
    if (lane == 0) {
      SlotMeta& m = my_meta[s];
      if constexpr (kFp8 && HP == 2) {
        // the tile's block: each head's scales
        *reinterpret_cast<float4*>(m.ks) = make_float4(ks[0], ks1, 1.f, 1.f);
        *reinterpret_cast<float4*>(m.vs) = make_float4(vs[0], vs1, 1.f, 1.f);
      } else if constexpr (kFp8) {
        float k4[4], v4[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int h = (8 * i) / bh;  // the block holding tokens 8i .. 8i+7
          k4[i] = ks[0];
          v4[i] = vs[0];
#pragma unroll
          for (int q = 1; q < kMaxSub; ++q)
            if (h == q) {
              k4[i] = ks[q];
              v4[i] = vs[q];
            }
        }
        *reinterpret_cast<float4*>(m.ks) = make_float4(k4[0], k4[1], k4[2], k4[3]);
        *reinterpret_cast<float4*>(m.vs) = make_float4(v4[0], v4[1], v4[2], v4[3]);
      }
      m.mask = mask;
      mbar_arrive_expect_tx(bar, tx);
    }
    __syncwarp();
    // the boxes, one per lane: box i is column (i / 2) % kBoxes of block
    // i / (2 kBoxes), of K (i even) or V (i odd); a single thread issues
    // only a few boxes per microsecond
    constexpr int kPerSub = 2 * Gm::kBoxes;
    if (lane < kMaxSub * kPerSub) {
      const int h = lane / kPerSub, r = lane % kPerSub, b = r >> 1;
      int ph = phys[0];
#pragma unroll
      for (int q = 1; q < kMaxSub; ++q)
        if (h == q) ph = phys[q];
      if (ph >= 0) {
        // HP = 2: one box holds both heads' rows (heads 2u, 2u + 1 are adjacent)
        const int z = ph * p.kv_heads_phys + (HP == 2 ? 2 * c.kvh : kv_head_of(p, c.kvh));
        const uint32_t at = b * Gm::kBoxBytes + h * bh * 128;  // boxes of later blocks sit after earlier ones
        if (r & 1)
          tma_load_3d_hint(vdst + at, &tmap_v, b * Gm::kBoxW, off, z, bar, kv_policy);
        else
          tma_load_3d_hint(kdst + at, &tmap_k, b * Gm::kBoxW, off, z, bar, kv_policy);
      }
    }
  };

  // q of one (sequence, KV head) as MMA B fragments: column g = query head
  // kvh*G + g (zero for g >= G); 16-bit caches contract d in order, E4M3
  // caches in the permuted order their K fragments arrive in.
  // fetch_q issues the loads (E4M3: the four q elements of a step raw, as
  // two 16-bit pairs) and convert_q turns them into f16 fragments, so the
  // first q rows can be in flight while the first tiles are issued.
  uint32_t qb[Gm::kSteps][2];
  auto fetch_q = [&](int seq, int kvh) {
    const QT* qrow = static_cast<const QT*>(p.q) + (static_cast<int64_t>(seq) * Hq + kvh * G + g) * D;
#pragma unroll
    for (int k = 0; k < Gm::kSteps; ++k) {
      if (g >= G) {
        qb[k][0] = qb[k][1] = 0u;
      } else if constexpr (!kFp8) {
        qb[k][0] = *reinterpret_cast<const uint32_t*>(qrow + 16 * k + 2 * tig);
        qb[k][1] = *reinterpret_cast<const uint32_t*>(qrow + 16 * k + 8 + 2 * tig);
      } else {
        const uint2 r = *reinterpret_cast<const uint2*>(qrow + 16 * k + 4 * tig);
        qb[k][0] = r.x;
        qb[k][1] = r.y;
      }
    }
  };
  auto convert_q = [&]() {
    if constexpr (kFp8) {
#pragma unroll
      for (int k = 0; k < Gm::kSteps; ++k) {
        const float2 a = pair_to_float2(qb[k][0], static_cast<QT*>(nullptr));
        const float2 b = pair_to_float2(qb[k][1], static_cast<QT*>(nullptr));
        qb[k][0] = pack_f16(a.x, a.y);
        qb[k][1] = pack_f16(b.x, b.y);
        // beyond the f16 range q turns infinite: report it
        if (fmaxf(fmaxf(fabsf(a.x), fabsf(a.y)), fmaxf(fabsf(b.x), fabsf(b.y))) > 65504.f)
          flag_error(p.debug_err, PA_DEVERR_Q_RANGE);
      }
    }
  };
  auto load_q = [&](int seq, int kvh) {
    fetch_q(seq, kvh);
    convert_q();
  };

  // online-softmax state of the current piece: this lane's two heads
  // (columns 2*tig, 2*tig+1) and its 16 d rows per 16-row step
  float m0, m1, l0, l1;
  float o[Gm::kSteps][4];
  auto reset = [&]() {
    m0 = m1 = -INFINITY;
    l0 = l1 = 0.f;
#pragma unroll
    for (int k = 0; k < Gm::kSteps; ++k) o[k][0] = o[k][1] = o[k][2] = o[k][3] = 0.f;
  };

  // d index held in accumulator row r (0..15) of 16-row step k
  auto d_of = [&](int k, int upper) -> int {
    if constexpr (kFp8) return 16 * k + 2 * g + upper;
    else return 16 * k + g + 8 * upper;
  };

  // Write the finished piece: output rows, a partition partial, or a
  // per-warp partial state for the merge.
  auto flush = [&](int seq, int kvh, int part, bool whole, int64_t slot_index) {
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
      l0 += __shfl_xor_sync(kFull, l0, off);
      l1 += __shfl_xor_sync(kFull, l1, off);
    }
    const int h0 = 2 * tig, h1 = 2 * tig + 1;
    const bool prefixed = start_of(seq) > 0;
    if (whole && prefixed) {
      // a whole segment of a sequence with a shared prefix: its own state
      // slot, after the decode and shared-prefix states
      slot_index = 6 * static_cast<int64_t>(tp.num_warps) +
                   static_cast<int64_t>(B) * Hkv * tp.pg.num_chunks + static_cast<int64_t>(seq) * Hkv + kvh;
    }
    if (whole && tp.part_tiles == 0 && !prefixed) {
      QT* out = static_cast<QT*>(p.out);
      const float i0 = l0 > 0.f ? 1.f / l0 : 0.f;
      const float i1 = l1 > 0.f ? 1.f / l1 : 0.f;
      QT* r0 = out + (static_cast<int64_t>(seq) * Hq + kvh * G + h0) * D;
      QT* r1 = r0 + D;
#pragma unroll
      for (int k = 0; k < Gm::kSteps; ++k) {
        if constexpr (kFp8) {
          // rows d and d+1 are adjacent: one 32-bit store per head
          const int d = d_of(k, 0);
          if (h0 < G) {
            if constexpr (std::is_same<QT, bf16>::value)
              *reinterpret_cast<uint32_t*>(r0 + d) = pack_bf16(o[k][0] * i0, o[k][2] * i0);
            else
              *reinterpret_cast<uint32_t*>(r0 + d) = pack_f16(o[k][0] * i0, o[k][2] * i0);
          }
          if (h1 < G) {
            if constexpr (std::is_same<QT, bf16>::value)
              *reinterpret_cast<uint32_t*>(r1 + d) = pack_bf16(o[k][1] * i1, o[k][3] * i1);
            else
              *reinterpret_cast<uint32_t*>(r1 + d) = pack_f16(o[k][1] * i1, o[k][3] * i1);
          }
        } else {
          const int da = d_of(k, 0), db = d_of(k, 1);
          if (h0 < G) {
            r0[da] = from_float(o[k][0] * i0, static_cast<QT*>(nullptr));
            r0[db] = from_float(o[k][2] * i0, static_cast<QT*>(nullptr));
          }
          if (h1 < G) {
            r1[da] = from_float(o[k][1] * i1, static_cast<QT*>(nullptr));
            r1[db] = from_float(o[k][3] * i1, static_cast<QT*>(nullptr));
          }
        }
      }
    } else if (tp.part_tiles != 0) {
      // one whole partition: normalised partial plus (max, sum) for the reduce
      const int NP = p.num_partitions;
      const float i0 = l0 > 0.f ? 1.f / l0 : 0.f;
      const float i1 = l1 > 0.f ? 1.f / l1 : 0.f;
      const int64_t s0 = (static_cast<int64_t>(seq) * Hq + kvh * G + h0) * NP + part;
      const int64_t s1 = s0 + NP;
#pragma unroll
      for (int k = 0; k < Gm::kSteps; ++k) {
        const int da = d_of(k, 0), db = d_of(k, 1);
        if (h0 < G) {
          p.ws_acc[s0 * D + da] = o[k][0] * i0;
          p.ws_acc[s0 * D + db] = o[k][2] * i0;
        }
        if (h1 < G) {
          p.ws_acc[s1 * D + da] = o[k][1] * i1;
          p.ws_acc[s1 * D + db] = o[k][3] * i1;
        }
      }
      if (g == 0) {
        if (h0 < G) {
          p.ws_ml[s0 * 2] = m0;
          p.ws_ml[s0 * 2 + 1] = l0;
        }
        if (h1 < G) {
          p.ws_ml[s1 * 2] = m1;
          p.ws_ml[s1 * 2 + 1] = l1;
        }
      }
    } else {
      // part of a (sequence, KV head) shared with other warps
      // (16-bit caches: stored under an L2 evict-last policy for the merge;
      // measured on the Llama-8B-shaped batch 88.5 against 89.5 us, while
      // the E4M3 layer was 0.8 us slower with it)
      float* base = tp.ws_slots + slot_index * state_floats(G, D);
      auto put = [&](float* a, float v) {
        if constexpr (kFp8) *a = v;
        else st_global_hint(a, v, state_policy);
      };
#pragma unroll
      for (int k = 0; k < Gm::kSteps; ++k) {
        const int da = d_of(k, 0), db = d_of(k, 1);
        if (h0 < G) {
          put(base + h0 * D + da, o[k][0]);
          put(base + h0 * D + db, o[k][2]);
        }
        if (h1 < G) {
          put(base + h1 * D + da, o[k][1]);
          put(base + h1 * D + db, o[k][3]);
        }
      }
      if (g == 0) {
        if (h0 < G) {
          put(base + G * D + h0, m0);
          put(base + G * D + G + h0, l0);
        }
        if (h1 < G) {
          put(base + G * D + h1, m1);
          put(base + G * D + G + h1, l1);
        }
      }
    }
  };

  // ---- the warp's pipeline ----------------------------------------------
  // The producer side runs up to NS tiles ahead of the consumer side; when it
  // reaches the end of its range it claims the next one, which the consumer
  // takes over when it reaches the same point. Claimed ranges wait in a small
  // queue in shared memory (lane 0 writes, the warp reads): every waiting
  // range but the newest has a tile in the ring, so NS + 1 entries suffice
  // even when ranges are a single tile (a split-path partition of one tile).
  Cursor pc, cc;
  cursor_at(pc, cr0, s_prefT, B, Hkv);
  cc = pc;
  int64_t pr1 = cr1;
  int q_head = 0, q_count = 0;  // warp-uniform
  bool prod_done = false;
  auto advance_producer = [&]() {
    cursor_next(pc, s_prefT, B, Hkv);
    if (pc.f == pr1) {
      int64_t a, b, sl;
      if (claim(a, b, sl)) {
        int i = q_head + q_count;
        if (i > NS) i -= NS + 1;
        if (lane == 0) {
          s_queue[warp][i][0] = a;
          s_queue[warp][i][1] = b;
          s_queue[warp][i][2] = sl;
        }
        __syncwarp();
        ++q_count;
        pr1 = b;
        cursor_at(pc, a, s_prefT, B, Hkv);
      } else {
        prod_done = true;
      }
    }
  };
  fetch_q(cc.seq, cc.kvh);  // in flight while the first tiles are issued
  int pending = 0;
  for (int s = 0; s < NS && !prod_done; ++s) {
    issue(pc, s);
    advance_producer();
    ++pending;
  }
  convert_q();
  reset();
  int piece_t0 = cc.t;
  bool first_piece = true;
  uint32_t parity = 0;
  int s = 0;
  while (true) {
    const bool ok = mbar_wait_bounded(bar_base + s * 8, (parity >> s) & 1u);
    if (!__all_sync(kFull, ok)) {
      if (lane == 0) flag_error(p.debug_err, PA_DEVERR_TIMEOUT);
      // give copies still in flight a short while to land, then leave
      for (int q = 0; q < NS; ++q) mbar_wait_bounded(bar_base + q * 8, (parity >> q) & 1u, 10000000ull);
      return;
    }
    parity ^= 1u << s;
    --pending;
    const SlotMeta mt = my_meta[s];
    const uint32_t kbase = slot_base0 + s * Gm::kSlotBytes;
    const uint32_t vbase = kbase + Gm::kTileBytes;

    // S^T = K Q^T per 16-token row tile: rows = tokens, columns = query heads.
    // HP = 2: the two heads' K rows meet q with the other head's columns
    // zeroed (a block-diagonal q), both into the same accumulators.
    float sv[RS][4];
#pragma unroll
    for (int rs = 0; rs < RS; ++rs) {
      float sa[4] = {0.f, 0.f, 0.f, 0.f}, sb[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int hh = 0; hh < HP; ++hh) {
        const int rt = hh * RS + rs;
        const int row = rt * kRowTile + (lane & 15);
        [[maybe_unused]] const bool qon = HP == 1 || hd_b == hh;
        if constexpr (!kFp8) {
#pragma unroll
          for (int k = 0; k < Gm::kSteps; ++k) {
            uint32_t a[4];
            ldsm_x4(tile_addr<Gm::kBoxBytes>(kbase, row, 2 * k + (lane >> 4)), a[0], a[1], a[2], a[3]);
            if constexpr (std::is_same<KT, bf16>::value) mma_bf16((k & 1) ? sb : sa, a, qb[k][0], qb[k][1]);
            else mma_f16((k & 1) ? sb : sa, a, qb[k][0], qb[k][1]);
          }
        } else {
#pragma unroll
          for (int k = 0; k < Gm::kSteps; k += 2) {
            uint32_t r[4];
            ldsm_x4(tile_addr<Gm::kBoxBytes>(kbase, row, k + (lane >> 4)), r[0], r[1], r[2], r[3]);
            // a lane's four bytes of a row are d = 16c + 4tig .. +3: the low pair
            // feeds contraction slots 2tig, 2tig+1, the high pair 2tig+8, 2tig+9
            uint32_t a0[4], a1[4];
            e4m3x4_to_f16x2x2(r[0], a0[0], a0[2]);
            e4m3x4_to_f16x2x2(r[1], a0[1], a0[3]);
            e4m3x4_to_f16x2x2(r[2], a1[0], a1[2]);
            e4m3x4_to_f16x2x2(r[3], a1[1], a1[3]);
            mma_f16(sa, a0, qon ? qb[k][0] : 0u, qon ? qb[k][1] : 0u);
            mma_f16(sb, a1, qon ? qb[k + 1][0] : 0u, qon ? qb[k + 1][1] : 0u);
          }
        }
      }
      // the block's K scale for E4M3 caches (the slot's scales are only
      // written for them): per 8-token group, or (HP = 2) per head
      float sc0 = p.scale_log2, sc1 = p.scale_log2;
      if constexpr (kFp8 && HP == 2) {
        sc0 = sc1 = p.scale_log2 * (hd_c ? mt.ks[1] : mt.ks[0]);
      } else if constexpr (kFp8) {
        sc0 = p.scale_log2 * mt.ks[2 * rs];
        sc1 = p.scale_log2 * mt.ks[2 * rs + 1];
      }
      sv[rs][0] = (sa[0] + sb[0]) * sc0;
      sv[rs][1] = (sa[1] + sb[1]) * sc0;
      sv[rs][2] = (sa[2] + sb[2]) * sc1;
      sv[rs][3] = (sa[3] + sb[3]) * sc1;
    }
    const uint32_t mask = mt.mask;
    float x0 = -INFINITY, x1 = -INFINITY;
#pragma unroll
    for (int rs = 0; rs < RS; ++rs) {
      if (!((mask >> (rs * kRowTile + g)) & 1u)) sv[rs][0] = sv[rs][1] = -INFINITY;
      if (!((mask >> (rs * kRowTile + g + 8)) & 1u)) sv[rs][2] = sv[rs][3] = -INFINITY;
      x0 = fmaxf(x0, fmaxf(sv[rs][0], sv[rs][2]));
      x1 = fmaxf(x1, fmaxf(sv[rs][1], sv[rs][3]));
    }

    // online softmax (log2 units), per head column
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
      x0 = fmaxf(x0, __shfl_xor_sync(kFull, x0, off));
      x1 = fmaxf(x1, __shfl_xor_sync(kFull, x1, off));
    }
    const float n0 = fmaxf(m0, x0), n1 = fmaxf(m1, x1);
    if (__any_sync(kFull, n0 > m0 || n1 > m1)) {
      const float a0 = exp2f(m0 - n0), a1 = exp2f(m1 - n1);  // 0 while m is -inf
      m0 = n0;
      m1 = n1;
      l0 *= a0;
      l1 *= a1;
#pragma unroll
      for (int k = 0; k < Gm::kSteps; ++k) {
        o[k][0] *= a0;
        o[k][1] *= a1;
        o[k][2] *= a0;
        o[k][3] *= a1;
      }
    }
    const float b0 = m0 == -INFINITY ? 0.f : m0, b1 = m1 == -INFINITY ? 0.f : m1;
    // P^T of each row tile as B operands: transpose the accumulator-layout rows
    uint32_t pb[RS][2];
#pragma unroll
    for (int rs = 0; rs < RS; ++rs) {
      const float p0 = exp2f(sv[rs][0] - b0), p1 = exp2f(sv[rs][1] - b1);
      const float p2 = exp2f(sv[rs][2] - b0), p3 = exp2f(sv[rs][3] - b1);
      l0 += p0 + p2;
      l1 += p1 + p3;
      if constexpr (std::is_same<KT, bf16>::value) {
        pb[rs][0] = movmatrix_trans(pack_bf16(p0, p1));
        pb[rs][1] = movmatrix_trans(pack_bf16(p2, p3));
      } else if constexpr (!kFp8) {
        pb[rs][0] = movmatrix_trans(pack_f16(p0, p1));
        pb[rs][1] = movmatrix_trans(pack_f16(p2, p3));
      } else {
        const float v0 = HP == 2 ? (hd_c ? mt.vs[1] : mt.vs[0]) : mt.vs[2 * rs];
        const float v1 = HP == 2 ? v0 : mt.vs[2 * rs + 1];
        pb[rs][0] = movmatrix_trans(pack_f16(p0 * v0, p1 * v0));
        pb[rs][1] = movmatrix_trans(pack_f16(p2 * v1, p3 * v1));
      }
    }

    // O^T += V^T P^T: each row tile is one 16-token contraction step,
    // one 16-row step of d at a time
    // HP = 2: head h's V rows meet P^T with the other head's columns zeroed
    const bool partial = mask != Gm::kFullMask;
#pragma unroll
    for (int rt = 0; rt < RT; ++rt) {
      const int rs = rt % RS, hh = rt / RS;
      const int t0 = rs * kRowTile;     // the row tile's first token
      const int r0 = rt * kRowTile;     // its first row in the slot
      const bool pon = HP == 1 || hd_b == hh;
      const uint32_t pb0 = pon ? pb[rs][0] : 0u, pb1 = pon ? pb[rs][1] : 0u;
      if constexpr (!kFp8) {
#pragma unroll
        for (int k = 0; k < Gm::kSteps; ++k) {
          uint32_t a[4];
          ldsm_x4_trans(tile_addr<Gm::kBoxBytes>(vbase, r0 + (lane & 7) + ((lane >> 4) << 3),
                                                 2 * k + ((lane >> 3) & 1)),
                        a[0], a[1], a[2], a[3]);
          if (partial) {
            a[0] = keep_tokens(a[0], mask, t0 + 2 * tig);
            a[1] = keep_tokens(a[1], mask, t0 + 2 * tig);
            a[2] = keep_tokens(a[2], mask, t0 + 2 * tig + 8);
            a[3] = keep_tokens(a[3], mask, t0 + 2 * tig + 8);
          }
          if constexpr (std::is_same<KT, bf16>::value) mma_bf16(o[k], a, pb0, pb1);
          else mma_f16(o[k], a, pb0, pb1);
        }
      } else {
#pragma unroll
        for (int k = 0; k < Gm::kSteps; k += 2) {
          uint32_t r[4];
          ldsm_x4_trans(tile_addr<Gm::kBoxBytes>(vbase, r0 + (lane & 15), k + (lane >> 4)),
                        r[0], r[1], r[2], r[3]);
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            // tokens 0-7 / 8-15 of chunk k+h; bytes (t, d0), (t, d1), (t+1, d0),
            // (t+1, d1) regrouped as (d0: t, t+1) and (d1: t, t+1)
            uint32_t a[4];
            e4m3x4_to_f16x2x2(__byte_perm(r[2 * h], 0, 0x3120), a[0], a[1]);
            e4m3x4_to_f16x2x2(__byte_perm(r[2 * h + 1], 0, 0x3120), a[2], a[3]);
            if (partial) {
              a[0] = keep_tokens(a[0], mask, t0 + 2 * tig);
              a[1] = keep_tokens(a[1], mask, t0 + 2 * tig);
              a[2] = keep_tokens(a[2], mask, t0 + 2 * tig + 8);
              a[3] = keep_tokens(a[3], mask, t0 + 2 * tig + 8);
            }
            mma_f16(o[k + h], a, pb0, pb1);
          }
        }
      }
    }

    // the slot is free again: refill it with the tile NS ahead
    __syncwarp();
    fence_proxy_async_smem();
    if (!prod_done) {
      issue(pc, s);
      advance_producer();
      ++pending;
    }
    s = (s + 1 == NS) ? 0 : s + 1;

    // end of a piece?
    const int seq = cc.seq, kvh = cc.kvh, t = cc.t, tiles = cc.tiles;
    cursor_next(cc, s_prefT, B, Hkv);
    const bool range_end = cc.f == cr1;
    const bool new_segment = cc.t == 0 || (tp.part_tiles != 0 && cc.t % tp.part_tiles == 0);
    if (range_end || new_segment) {
      const int seg_t0 = tp.part_tiles ? (t / tp.part_tiles) * tp.part_tiles : 0;
      const int seg_t1 = tp.part_tiles ? min(tiles, seg_t0 + tp.part_tiles) : tiles;
      const bool whole = piece_t0 == seg_t0 && t + 1 == seg_t1;
      flush(seq, kvh, tp.part_tiles ? t / tp.part_tiles : 0, whole, first_piece ? cslot : cslot + 1);
      first_piece = false;
      if (range_end) {
        if (q_count == 0) break;
        cr0 = s_queue[warp][q_head][0];
        cr1 = s_queue[warp][q_head][1];
        cslot = s_queue[warp][q_head][2];
        q_head = q_head == NS ? 0 : q_head + 1;
        --q_count;
        first_piece = true;
        cursor_at(cc, cr0, s_prefT, B, Hkv);
      }
      reset();
      piece_t0 = cc.t;
      if (range_end || cc.seq != seq || cc.kvh != kvh) load_q(cc.seq, cc.kvh);
    }
  }
  (void)pending;
}

// Combine the partial states of every (sequence, KV head) that several
// ranges shared (launched as a programmatic dependent of the decode grid):
// with M = max_c m_c, out = sum_c 2^(m_c-M) acc_c / sum_c 2^(m_c-M) l_c.
// Sequences with no context get zero rows here. The rows are float4 elements
// of the G x D block, EPT per thread; when the block has fewer elements than
// the CTA has threads, the threads split the contributors into groups, so a
// step issues the loads of many contributors at once. Contributor slots are
// listed in shared memory 128 (or 256) at a time.
// - Up to 256 threads: the (max, sum) of every contributor in the list are
//   loaded by a thread each, a warp per head derives the weights, and a
//   running maximum carries the softmax across lists.
// - 1024 threads (long contributor lists): each thread keeps its own online
//   softmax (running maximum, denominator, weighted rows) over its group's
//   contributors, loading a contributor's rows with its maximum and sum, and
//   group 0 combines the groups at the end; no barrier stands between the
//   decode grid's completion and the loads (long context bs 16: 169.7 ->
//   168.2 us; slower on the E4M3 layer's short lists, 72.4 against 74.2).
// Threads of a merge CTA: 256, or 1024 when there are few pairs (their
// contributor lists are then long, and more threads keep more rows in flight),
// or 128 when most pairs have at most two contributors (fewer warps than twice
// the pairs) and the G x D block has at most 128 float4s: a 128-thread CTA
// fits on an SM beside the persistent decode CTA, so the first of them are
// resident, past their prologue, when the decode grid completes. (Measured:
// 128 threads were faster on batches of short pairs, 256 on the Llama-8B-
// shaped batch, about 2.4 contributors per pair.) Blocks of more than 128
// float4s with more pairs than one wave of 256-thread CTAs holds take 128
// threads of two elements each, so that one wave holds them all (the E4M3
// layer's head-pair blocks: 73.1 -> 72.4 us).
constexpr int kMergeThreads = 256;
constexpr int kMergeThreadsFew = 1024;
constexpr int kMergeThreadsSmall = 128;

template <typename QT, int D, int TT, int NT, int EPT = 1>
__global__ void __launch_bounds__(NT, 1024 / NT) tc_merge_kernel(const TcParams tp) {
  constexpr int kMergeThreads = NT;
  constexpr int kMergeChunk = NT >= 512 ? 256 : 128;  // contributors taken at a time
  constexpr bool kOnline = NT >= 512;  // long contributor lists: an online softmax per thread
  const DecodeParams& p = tp.p;
  if (blockIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0) {
    // the decode grid is complete: rearm its chunk counter for the next call
    griddep_wait();
    if (threadIdx.x == 0) *tp.claim = 0;
  }
  const int kvh = blockIdx.x;
  const int seq = blockIdx.y;
  const int G = tp.group;
  const int Hkv = p.num_kv_heads;
  const int B = p.num_seqs;
  QT* out = static_cast<QT*>(p.out) + (static_cast<int64_t>(seq) * p.num_heads + kvh * G) * D;

  // Until the wait below, only inputs are read (the decode grid writes none
  // of them): this sequence's tile offset in the list and the total, from
  // the clamped context lengths exactly as the decode grid computes them.
  __shared__ int s_sum[kMergeThreads / 32][2];
  int before = 0, total = 0;
  for (int i = threadIdx.x; i < B; i += kMergeThreads) {
    int glen;
    const int ctx = clamp_context(p, i);
    const int tl = seq_tiles<TT>(ctx, min(seq_prefix_len(tp.pg, p, i, glen), ctx));
    total += tl;
    if (i < seq) before += tl;
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    before += __shfl_xor_sync(0xffffffffu, before, off);
    total += __shfl_xor_sync(0xffffffffu, total, off);
  }
  if ((threadIdx.x & 31) == 0) {
    s_sum[threadIdx.x >> 5][0] = before;
    s_sum[threadIdx.x >> 5][1] = total;
  }
  __syncthreads();
  before = total = 0;
#pragma unroll
  for (int w = 0; w < kMergeThreads / 32; ++w) {
    before += s_sum[w][0];
    total += s_sum[w][1];
  }
  // the shared-prefix states of this sequence: one per chunk of its group's prefix
  int plen = 0;
  const int ctx_self = clamp_context(p, seq);
  const int start = min(seq_prefix_len(tp.pg, p, seq, plen), ctx_self);
  const int npre = plen > 0 ? (plen + tp.pg.chunk_len - 1) / tp.pg.chunk_len : 0;
  const int tiles = seq_tiles<TT>(ctx_self, start);
  if (tiles == 0 && npre == 0) {
    for (int i = threadIdx.x; i < G * D; i += kMergeThreads) out[i] = from_float(0.f, static_cast<QT*>(nullptr));
    return;
  }
  const int64_t U = static_cast<int64_t>(total) * Hkv;
  const int64_t W = tp.num_warps;
  const int64_t seg0 = static_cast<int64_t>(before) * Hkv + static_cast<int64_t>(kvh) * tiles;
  const int64_t seg1 = seg0 + tiles;
  // The schedule's quantities for this segment, derived by one thread and
  // shared (64-bit divisions are long instruction sequences).
  __shared__ int64_t s_sched[6];
  if (threadIdx.x == 0) {
    const Sched sc = make_sched(U, W, tp.short_share);
    const int64_t S = sc.S, C = sc.C;
    // static shares meeting [seg0, min(seg1, S)): warp w holds [w*S/W,
    // (w+1)*S/W), so the owner of tile x < S is ceil((x+1)W/S) - 1
    int64_t ws0 = 0, nstat = 0;
    if (tiles > 0 && seg0 < S) {
      const int64_t e = seg1 < S ? seg1 : S;
      ws0 = ((seg0 + 1) * W - 1) / S;
      nstat = (e * W - 1) / S - ws0 + 1;
    }
    // chunks meeting [max(seg0, S), seg1)
    int64_t k0 = 0, ndyn = 0;
    if (tiles > 0 && seg1 > S) {
      const int64_t a = seg0 > S ? seg0 : S;
      k0 = (a - S) / C;
      ndyn = (seg1 - 1 - S) / C - k0 + 1;
    }
    s_sched[0] = S;
    s_sched[1] = C;
    s_sched[2] = ws0;
    s_sched[3] = nstat;
    s_sched[4] = k0;
    s_sched[5] = ndyn;
  }
  __syncthreads();
  const int64_t S = s_sched[0], C = s_sched[1], ws0 = s_sched[2], nstat = s_sched[3], k0 = s_sched[4];
  const int ndec = static_cast<int>(nstat + s_sched[5]);
  if (ndec == 1 && npre == 0) return;  // one range held the whole segment and wrote the rows
  const int nc = ndec + npre;
  // a whole segment of a sequence with a shared prefix left its state in the
  // sequence's own slot, after the decode and shared-prefix states
  const bool own_slot = ndec == 1 && start > 0;

  // slot of contributor c: static shares first, then chunks; a range that
  // starts before the segment left it in its second slot; -1 for a warp
  // whose static share is empty (it wrote nothing)
  auto slot_of = [&](int c) -> int {
    if (c >= ndec)  // a shared-prefix state, stored after the 6W decode states
      return static_cast<int>(6 * W + (static_cast<int64_t>(seq) * Hkv + kvh) * tp.pg.num_chunks + (c - ndec));
    if (own_slot)
      return static_cast<int>(6 * W + static_cast<int64_t>(B) * Hkv * tp.pg.num_chunks +
                              static_cast<int64_t>(seq) * Hkv + kvh);
    if (c < nstat) {
      const int64_t w = ws0 + c;
      const int64_t st = w * S / W, en = (w + 1) * S / W;
      return st == en ? -1 : static_cast<int>((c == 0 && st < seg0) ? 2 * w + 1 : 2 * w);
    }
    const int64_t k = k0 + (c - nstat);
    const int64_t st = S + k * C;
    return static_cast<int>(2 * W + 2 * k + ((c == nstat && st < seg0) ? 1 : 0));
  };

  __shared__ int s_slot[kMergeChunk];
  const float* slots = tp.ws_slots;
  const int stride = state_floats(G, D);
  // the block's float4 elements (32..256); with gridDim.z > 1 this CTA takes
  // the z-th of gridDim.z equal slices of them (few pairs with many
  // contributors: more CTAs share each pair). A thread holds EPT elements of
  // the slice, nth apart.
  const int nes = G * D / 4 / static_cast<int>(gridDim.z);
  const int nth = nes / EPT;                 // threads that cover the slice once
  const int ngrp = kMergeThreads / nth;      // contributor groups
  const int el = threadIdx.x % nth;          // this thread's first element within the slice
  const int grp = threadIdx.x / nth;
  int e4[EPT], he[EPT];                      // this thread's elements and their heads
#pragma unroll
  for (int e = 0; e < EPT; ++e) {
    e4[e] = static_cast<int>(blockIdx.z) * nes + el + e * nth;
    he[e] = (4 * e4[e]) / D;
  }
  if constexpr (kOnline) {
    // each thread carries its own online softmax over the contributors of its
    // group: running maximum, denominator and weighted rows, per element
    float run[EPT], den[EPT];
    float4 acc[EPT];
#pragma unroll
    for (int e = 0; e < EPT; ++e) {
      run[e] = -INFINITY;
      den[e] = 0.f;
      acc[e] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    if (threadIdx.x < min(kMergeChunk, nc)) s_slot[threadIdx.x] = slot_of(threadIdx.x);
    __syncthreads();
    griddep_wait();  // the decode grid's partial states are complete from here on
    constexpr int kBatch = 4 / EPT;  // contributors a thread loads at a time (4 rows in flight)
    for (int cb = 0; cb < nc; cb += kMergeChunk) {
      const int nin = min(kMergeChunk, nc - cb);
      if (cb > 0) {
        __syncthreads();  // every thread is done with the previous chunk's slots
        if (threadIdx.x < nin) s_slot[threadIdx.x] = slot_of(cb + threadIdx.x);
        __syncthreads();
      }
      for (int j0 = grp; j0 < nin; j0 += kBatch * ngrp) {
        // one round of loads: each contributor's row elements, maximum and sum
        float4 v[kBatch][EPT];
        float m[kBatch][EPT], l[kBatch][EPT];
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
          const int j = j0 + u * ngrp;
          const int sl = j < nin ? s_slot[j] : -1;
          const float* st = slots + int64_t(sl) * stride;
#pragma unroll
          for (int e = 0; e < EPT; ++e) {
            v[u][e] = sl >= 0 ? __ldcg(reinterpret_cast<const float4*>(st) + e4[e]) : make_float4(0.f, 0.f, 0.f, 0.f);
            m[u][e] = sl >= 0 ? __ldcg(st + G * D + he[e]) : -INFINITY;
            l[u][e] = sl >= 0 ? __ldcg(st + G * D + G + he[e]) : 0.f;
          }
        }
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
#pragma unroll
          for (int e = 0; e < EPT; ++e) {
            const float mj = m[u][e];
            if (mj > run[e]) {
              const float a = exp2f(run[e] - mj);  // 0 while the running maximum is -inf
              den[e] *= a;
              acc[e].x *= a;
              acc[e].y *= a;
              acc[e].z *= a;
              acc[e].w *= a;
              run[e] = mj;
            }
            const float w = mj == -INFINITY ? 0.f : exp2f(mj - run[e]);
            den[e] += w * l[u][e];
            acc[e].x += w * v[u][e].x;
            acc[e].y += w * v[u][e].y;
            acc[e].z += w * v[u][e].z;
            acc[e].w += w * v[u][e].w;
          }
        }
      }
    }
    // the groups' states, combined by group 0
    __shared__ float4 s_acc[kMergeThreads * EPT];
    __shared__ float2 s_md[kMergeThreads * EPT];
    if (ngrp > 1) {
#pragma unroll
      for (int e = 0; e < EPT; ++e) {
        s_acc[threadIdx.x * EPT + e] = acc[e];
        s_md[threadIdx.x * EPT + e] = make_float2(run[e], den[e]);
      }
      __syncthreads();
    }
    if (grp == 0) {
#pragma unroll
      for (int e = 0; e < EPT; ++e) {
        float mx = run[e];
        for (int gi = 1; gi < ngrp; ++gi) mx = fmaxf(mx, s_md[(gi * nth + el) * EPT + e].x);
        const float a0 = run[e] == -INFINITY ? 0.f : exp2f(run[e] - mx);
        float4 t = make_float4(a0 * acc[e].x, a0 * acc[e].y, a0 * acc[e].z, a0 * acc[e].w);
        float d = a0 * den[e];
        for (int gi = 1; gi < ngrp; ++gi) {
          const int k = (gi * nth + el) * EPT + e;
          const float2 md = s_md[k];
          const float a = md.x == -INFINITY ? 0.f : exp2f(md.x - mx);
          const float4 u = s_acc[k];
          t.x += a * u.x;
          t.y += a * u.y;
          t.z += a * u.z;
          t.w += a * u.w;
          d += a * md.y;
        }
        const float inv = d > 0.f ? 1.f / d : 0.f;
        uint2 pk;
        if constexpr (std::is_same<QT, bf16>::value) {
          pk.x = pack_bf16(t.x * inv, t.y * inv);
          pk.y = pack_bf16(t.z * inv, t.w * inv);
        } else {
          pk.x = pack_f16(t.x * inv, t.y * inv);
          pk.y = pack_f16(t.z * inv, t.w * inv);
        }
        *reinterpret_cast<uint2*>(out + 4 * e4[e]) = pk;
      }
    }
  } else {
    __shared__ float s_w[kMergeChunk][kMaxG];  // max of each contributor, then its weight
    __shared__ float s_l[kMergeChunk][kMaxG];
    __shared__ float s_run[kMaxG], s_den[kMaxG], s_scale[kMaxG];
    __shared__ float4 s_part[kMergeThreads * EPT];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x < kMaxG) {
      s_run[threadIdx.x] = -INFINITY;
      s_den[threadIdx.x] = 0.f;
    }
    float4 acc[EPT];
#pragma unroll
    for (int e = 0; e < EPT; ++e) acc[e] = make_float4(0.f, 0.f, 0.f, 0.f);
    if (threadIdx.x < min(kMergeChunk, nc)) s_slot[threadIdx.x] = slot_of(threadIdx.x);
    __syncthreads();
    griddep_wait();  // the decode grid's partial states are complete from here on
    constexpr int kBatch = 4 / EPT;  // rows a thread loads at a time (4 float4s in flight)
    for (int cb = 0; cb < nc; cb += kMergeChunk) {
      const int nin = min(kMergeChunk, nc - cb);
      if (cb > 0) {
        if (threadIdx.x < nin) s_slot[threadIdx.x] = slot_of(cb + threadIdx.x);
        __syncthreads();
      }
      // one round of loads: each contributor's (max, sum) per head, and this
      // thread's first kBatch rows
      if (threadIdx.x < nin) {
        const int sl = s_slot[threadIdx.x];
#pragma unroll
        for (int h = 0; h < kMaxG; ++h) {
          const bool ok = sl >= 0 && h < G;
          s_w[threadIdx.x][h] = ok ? __ldcg(slots + int64_t(sl) * stride + G * D + h) : -INFINITY;
          s_l[threadIdx.x][h] = ok ? __ldcg(slots + int64_t(sl) * stride + G * D + G + h) : 0.f;
        }
      }
      float4 v[kBatch][EPT];
#pragma unroll
      for (int u = 0; u < kBatch; ++u) {
        const int j = grp + u * ngrp;
        const int sl = j < nin ? s_slot[j] : -1;
#pragma unroll
        for (int e = 0; e < EPT; ++e)
          v[u][e] = sl >= 0 ? __ldcg(reinterpret_cast<const float4*>(slots + int64_t(sl) * stride) + e4[e])
                            : make_float4(0.f, 0.f, 0.f, 0.f);
      }
      __syncthreads();
      // per head (warps take heads h, h + warps, ...): new running max,
      // rescale factor, weights, sum
      for (int h = warp; h < G; h += kMergeThreads / 32) {
        float cm = -INFINITY;
        for (int j = lane; j < nin; j += 32) cm = fmaxf(cm, s_w[j][h]);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) cm = fmaxf(cm, __shfl_xor_sync(0xffffffffu, cm, off));
        const float old = s_run[h];
        const float nm = fmaxf(old, cm);
        float d = 0.f;
        for (int j = lane; j < nin; j += 32) {
          const float m = s_w[j][h];
          const float w = m == -INFINITY ? 0.f : exp2f(m - nm);
          s_w[j][h] = w;
          d += w * s_l[j][h];
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) d += __shfl_xor_sync(0xffffffffu, d, off);
        __syncwarp();
        if (lane == 0) {
          const float scale = old == -INFINITY ? 0.f : exp2f(old - nm);
          s_scale[h] = scale;
          s_den[h] = s_den[h] * scale + d;
          s_run[h] = nm;
        }
      }
      __syncthreads();
      auto accumulate = [&](int j0) {
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
          const int j = j0 + u * ngrp;
#pragma unroll
          for (int e = 0; e < EPT; ++e) {
            const float wt = j < nin ? s_w[j][he[e]] : 0.f;
            acc[e].x += wt * v[u][e].x;
            acc[e].y += wt * v[u][e].y;
            acc[e].z += wt * v[u][e].z;
            acc[e].w += wt * v[u][e].w;
          }
        }
      };
#pragma unroll
      for (int e = 0; e < EPT; ++e) {
        const float sc_e = s_scale[he[e]];
        acc[e].x *= sc_e;
        acc[e].y *= sc_e;
        acc[e].z *= sc_e;
        acc[e].w *= sc_e;
      }
      accumulate(grp);
      // contributors beyond the first batch of this thread
      for (int j0 = grp + kBatch * ngrp; j0 < nin; j0 += kBatch * ngrp) {
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
          const int j = j0 + u * ngrp;
          const int sl = j < nin ? s_slot[j] : -1;
#pragma unroll
          for (int e = 0; e < EPT; ++e)
            v[u][e] = sl >= 0 ? __ldcg(reinterpret_cast<const float4*>(slots + int64_t(sl) * stride) + e4[e])
                              : make_float4(0.f, 0.f, 0.f, 0.f);
        }
        accumulate(j0);
      }
      __syncthreads();
    }
#pragma unroll
    for (int e = 0; e < EPT; ++e) s_part[threadIdx.x * EPT + e] = acc[e];
    __syncthreads();
    if (grp == 0) {
#pragma unroll
      for (int e = 0; e < EPT; ++e) {
        float4 t = acc[e];
        for (int gi = 1; gi < ngrp; ++gi) {
          const float4 u = s_part[(gi * nth + el) * EPT + e];
          t.x += u.x;
          t.y += u.y;
          t.z += u.z;
          t.w += u.w;
        }
        const float d = s_den[he[e]];
        const float inv = d > 0.f ? 1.f / d : 0.f;
        uint2 pk;
        if constexpr (std::is_same<QT, bf16>::value) {
          pk.x = pack_bf16(t.x * inv, t.y * inv);
          pk.y = pack_bf16(t.z * inv, t.w * inv);
        } else {
          pk.x = pack_f16(t.x * inv, t.y * inv);
          pk.y = pack_f16(t.z * inv, t.w * inv);
        }
        *reinterpret_cast<uint2*>(out + 4 * e4[e]) = pk;
      }
    }
  }
}

// ---- host side ----------------------------------------------------------

// Chunk counters of the auto schedule, one per call in flight (calls take
// them round robin). Module memory is zero when the library loads on a
// device and every call's merge kernel sets its counter back to zero, so the
// schedule needs nothing from the caller's memory.
constexpr int kClaimSlots = 256;
constexpr int kClaimDevices = 64;
__device__ int32_t g_claim_counters[kClaimSlots];
std::mutex g_claim_mutex;
int32_t* g_claim_base[kClaimDevices] = {};
std::atomic<unsigned> g_claim_next{0};

int32_t* next_claim_counter() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kClaimDevices) return nullptr;
  {
    std::lock_guard<std::mutex> lock(g_claim_mutex);
    if (g_claim_base[dev] == nullptr) {
      void* ptr = nullptr;
      if (cudaGetSymbolAddress(&ptr, g_claim_counters) != cudaSuccess) return nullptr;
      g_claim_base[dev] = static_cast<int32_t*>(ptr);
    }
  }
  return g_claim_base[dev] + (g_claim_next.fetch_add(1, std::memory_order_relaxed) % kClaimSlots);
}

}  // namespace

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static bool tried = false;
  if (!tried) {
    tried = true;
    cudaDriverEntryPointQueryResult q;
    void* ptr = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  }
  return fn;
}

// 3-D view of a cache: (d, token in block, block x KV head), boxes of 128
// bytes x min(block_size, 16) rows x 1, 128-byte swizzle.
bool make_cache_map(CUtensorMap* map, const void* base, int head_dim, int elem, int block_size,
                    int tile_tokens, int64_t blocks_x_heads, int heads_per_box) {
  auto fn = encode_fn();
  if (fn == nullptr) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(head_dim), static_cast<cuuint64_t>(block_size),
                        static_cast<cuuint64_t>(blocks_x_heads)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(head_dim) * elem,
                           static_cast<cuuint64_t>(head_dim) * elem * block_size};
  cuuint32_t box[3] = {static_cast<cuuint32_t>(128 / elem),
                       static_cast<cuuint32_t>(block_size < tile_tokens ? block_size : tile_tokens),
                       static_cast<cuuint32_t>(heads_per_box)};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(map, elem == 1 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_UINT16, 3,
                  const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

namespace {

template <typename QT, typename KT, int D, int TT, int HP>
size_t smem_bytes(int num_seqs) {
  using Gm = Geom<KT, D, TT, HP>;
  return 1024 + static_cast<size_t>(Gm::kWarps) * Gm::kSlots * (Gm::kSlotBytes + sizeof(SlotMeta) + 8) +
         (3 * static_cast<size_t>(num_seqs) + 2) * sizeof(int);
}

template <typename QT, typename KT, int D, int TT, int HP = 1>
cudaError_t launch_typed(const TcParams& tp, const void* k_cache, const void* v_cache, int num_sms,
                         cudaStream_t stream) {
  const DecodeParams& p = tp.p;
  CUtensorMap mk, mv;
  const int64_t bxh = static_cast<int64_t>(p.num_blocks) * p.kv_heads_phys;
  if (!make_cache_map(&mk, k_cache, D, int(sizeof(KT)), p.block_size, TT, bxh, HP) ||
      !make_cache_map(&mv, v_cache, D, int(sizeof(KT)), p.block_size, TT, bxh, HP))
    return cudaErrorInvalidValue;
  auto kernel = decode_tc_kernel<QT, KT, D, TT, HP>;
  static std::atomic<unsigned long long> attr_set{0};
  cudaError_t e = set_smem_limit_once(reinterpret_cast<const void*>(kernel),
                                      static_cast<int>(smem_bytes<QT, KT, D, TT, HP>(kTcMaxSeqs)), attr_set);
  if (e != cudaSuccess) return e;
  constexpr int kWarps = Geom<KT, D, TT, HP>::kWarps;
  const int grid = (tp.num_warps + kWarps - 1) / kWarps;
  if (tp.pg.group_start != nullptr) {
    // the shared prefixes first, on the whole GPU; the decode grid that
    // follows starts its work (griddepcontrol.wait) once they are complete
    e = launch_prefix_attn(p, tp.pg, D, std::is_same<QT, bf16>::value ? PA_BF16 : PA_F16, stream);
    if (e != cudaSuccess) return e;
  }
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kWarps * 32);
  cfg.dynamicSmemBytes = smem_bytes<QT, KT, D, TT, HP>(p.num_seqs);
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t err = cudaLaunchKernelEx(&cfg, kernel, mk, mv, tp);
  if (err != cudaSuccess) return err;
  note_launches(1);
  if (tp.part_tiles != 0) {
    err = launch_reduce_partitions(p, D, std::is_same<QT, bf16>::value ? PA_BF16 : PA_F16,
                                   /*pdl=*/true, stream);
    if (err != cudaSuccess) cudaMemsetAsync(tp.claim, 0, sizeof(int32_t), stream);  // rearm it ourselves
    return err;
  }
  cudaLaunchConfig_t mcfg = cfg;
  mcfg.gridDim = dim3(p.num_kv_heads, p.num_seqs);
  // few pairs: each is split over up to 4 CTAs by element slices (slices of
  // at least 32 float4s) so that more SMs share the merge
  const int64_t npairs = static_cast<int64_t>(p.num_seqs) * p.num_kv_heads;
  int zs = 1;
  while (zs < 4 && npairs * zs * 2 <= num_sms && (tp.group * D / 4) % (zs * 2) == 0 && tp.group * D / 4 / (zs * 2) >= 32)
    zs *= 2;
  mcfg.dynamicSmemBytes = 0;
  // more pairs than one wave of kMergeThreads-thread CTAs holds, each of more
  // than kMergeThreadsSmall float4s: kMergeThreadsSmall-thread CTAs of two
  // elements per thread, so that all of them are resident at once
  bool wide = false;
  if constexpr (D == 128)
    wide = tp.group * D / 4 > kMergeThreadsSmall && npairs > static_cast<int64_t>(num_sms) * (1024 / kMergeThreads);
  if (static_cast<int64_t>(p.num_seqs) * p.num_kv_heads <= num_sms) {
    mcfg.blockDim = dim3(kMergeThreadsFew);
    mcfg.gridDim.z = zs;
    err = cudaLaunchKernelEx(&mcfg, tc_merge_kernel<QT, D, TT, kMergeThreadsFew>, tp);
  } else if (wide) {
    if constexpr (D == 128) {
      mcfg.blockDim = dim3(kMergeThreadsSmall);
      err = cudaLaunchKernelEx(&mcfg, tc_merge_kernel<QT, D, TT, kMergeThreadsSmall, 2>, tp);
    }
  } else if (tp.group <= 4 && tp.group * D <= 4 * kMergeThreadsSmall &&
             tp.num_warps < 2 * static_cast<int64_t>(p.num_seqs) * p.num_kv_heads) {
    mcfg.blockDim = dim3(kMergeThreadsSmall);
    err = cudaLaunchKernelEx(&mcfg, tc_merge_kernel<QT, D, TT, kMergeThreadsSmall>, tp);
  } else {
    mcfg.blockDim = dim3(kMergeThreads);
    err = cudaLaunchKernelEx(&mcfg, tc_merge_kernel<QT, D, TT, kMergeThreads>, tp);
  }
  if (err == cudaSuccess) {
    note_launches(1);
  } else {
    cudaMemsetAsync(tp.claim, 0, sizeof(int32_t), stream);  // rearm the counter ourselves
  }
  return err;
}

}  // namespace

// E4M3 tiles carry half the bytes of 16-bit ones, so they take 32 tokens per
// pipeline step to keep the same work per step.
int tc_tile_tokens(pa_dtype kv_dtype) { return kv_dtype == PA_FP8_E4M3 ? 32 : 16; }

bool tc_supported(int group, int head_dim, pa_dtype kv_dtype, int num_seqs, int partition_size) {
  if (group < 1 || group > kMaxG) return false;
  if (num_seqs > kTcMaxSeqs) return false;
  if (partition_size % tc_tile_tokens(kv_dtype) != 0) return false;
  if (kv_dtype == PA_FP8_E4M3) return head_dim == 128;
  return head_dim == 64 || head_dim == 128;
}

int tc_num_warps(int num_sms, int64_t max_units, pa_dtype kv_dtype) {
  int64_t w = static_cast<int64_t>(num_sms) * (kv_dtype == PA_FP8_E4M3 ? kWarpsFp8 : kWarps16);
  if (max_units < w) w = max_units;
  return static_cast<int>(w < 1 ? 1 : w);
}

size_t tc_auto_workspace_bytes(int num_seqs, int head_dim, int group, int num_sms) {
  (void)num_seqs;
  // two partial states per static share and per chunk (at most 2W chunks);
  // E4M3 calls with 2 or 4 query heads per KV head run units of two KV heads,
  // whose states hold twice the query heads
  const size_t W = static_cast<size_t>(num_sms) * kMaxWarps;
  const int sg = (group == 2 || group == 4) ? 2 * group : group;
  const size_t slots = 6 * W * static_cast<size_t>(state_floats(sg, head_dim)) * sizeof(float);
  return slots;
}

cudaError_t launch_decode_tc(const DecodeParams& p, int head_dim, pa_dtype q_dtype,
                             pa_dtype kv_dtype, int partition_size, void* workspace, int num_sms,
                             cudaStream_t stream, const PrefixGroups* groups) {
  // E4M3 caches with 2 or 4 query heads per KV head: a unit is two adjacent
  // KV heads (their query heads fill the MMA's 8 columns), its tiles 16
  // tokens of both heads, one box per block for K and one for V
  const int gkv = p.num_heads / p.num_kv_heads;
  const bool pairs = kv_dtype == PA_FP8_E4M3 && head_dim == 128 && groups == nullptr && p.kv_div == 1 &&
                     (gkv == 2 || gkv == 4) && p.num_kv_heads % 2 == 0 && p.block_size >= 16;
  const int tt = pairs ? 16 : tc_tile_tokens(kv_dtype);
  const int part_tiles = partition_size / tt;
  TcParams tp{};
  tp.p = p;
  tp.short_share = p.kv_div != 1 ? 0 : kv_dtype == PA_FP8_E4M3 ? kStatic256ShortFp8 : kStatic256Short16;
  if (pairs) tp.p.num_kv_heads = p.num_kv_heads / 2;  // units
  tp.group = p.num_heads / tp.p.num_kv_heads;
  tp.part_tiles = part_tiles;
  const int64_t tiles_max = (static_cast<int64_t>(p.max_context_len) + tt - 1) / tt;
  if (part_tiles == 0) {
    tp.claim = next_claim_counter();
    if (tp.claim == nullptr) return cudaErrorInvalidDevice;
    tp.num_warps = tc_num_warps(num_sms, static_cast<int64_t>(p.num_seqs) * tp.p.num_kv_heads * tiles_max, kv_dtype);
    tp.ws_slots = static_cast<float*>(workspace);
    if (groups != nullptr) {
      // the shared-prefix states follow the 6W decode states
      tp.pg = *groups;
      tp.pg.ws_prefix = tp.ws_slots + 6 * static_cast<int64_t>(tp.num_warps) * state_floats(tp.group, head_dim);
    }
  } else {
    const int64_t parts_max = (tiles_max + part_tiles - 1) / part_tiles;
    tp.num_warps = tc_num_warps(num_sms, static_cast<int64_t>(p.num_seqs) * tp.p.num_kv_heads * parts_max, kv_dtype);
    // the tail of the partitions is claimed from a counter the reduce rearms
    tp.claim = next_claim_counter();
    if (tp.claim == nullptr) return cudaErrorInvalidDevice;
    tp.p.claim = tp.claim;
  }
  const void* kc = p.k_cache;
  const void* vc = p.v_cache;
  if (kv_dtype == PA_BF16) {
    if (head_dim == 128) return launch_typed<bf16, bf16, 128, 16>(tp, kc, vc, num_sms, stream);
    return launch_typed<bf16, bf16, 64, 16>(tp, kc, vc, num_sms, stream);
  }
  if (kv_dtype == PA_F16) {
    if (head_dim == 128) return launch_typed<f16, f16, 128, 16>(tp, kc, vc, num_sms, stream);
    return launch_typed<f16, f16, 64, 16>(tp, kc, vc, num_sms, stream);
  }
  if (pairs) {
    if (q_dtype == PA_BF16) return launch_typed<bf16, fp8, 128, 16, 2>(tp, kc, vc, num_sms, stream);
    return launch_typed<f16, fp8, 128, 16, 2>(tp, kc, vc, num_sms, stream);
  }
  if (q_dtype == PA_BF16) return launch_typed<bf16, fp8, 128, 32>(tp, kc, vc, num_sms, stream);
  return launch_typed<f16, fp8, 128, 32>(tp, kc, vc, num_sms, stream);
}

}  // namespace pa
