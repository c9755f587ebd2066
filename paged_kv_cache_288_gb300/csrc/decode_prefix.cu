// Decode attention over a prefix that many sequences share, read once per
// group of sequences.
//
// When many requests open with the same prompt, their block tables point at
// the same physical blocks for it (serving-paged-attention, "공유는 표를
// 베끼는 일이 된다": the system prompt of 100 requests is stored once). A
// per-sequence decode still streams those blocks once per sequence. Here the
// shared keys are attended once per group instead: the rows of the product
// are (member sequence, query head) pairs of one KV unit, so with 100 members
// and 4 heads per KV head a key tile meets 400 query rows, a real dense tile
// for the tensor cores.
//
// Work. A CTA of four warps takes 64 rows (16 per warp: member r / G, query
// head r % G of one KV unit) and one chunk of the group's shared keys; the
// grid is (row tiles, KV units, group x chunk). Its K and V tiles (64 keys,
// one 3-D TMA box per 128-byte column per block, issued by the first lanes
// of all four warps) go through a three-stage ring in shared memory that all
// warps read. Per tile and warp: S = Q K^T as
// mma.sync m16n8k16 with Q held as A fragments in registers and K^T as B
// fragments (ldmatrix), eight independent 8-key accumulators; the online
// softmax on the accumulators (running maximum in log2 units, running sum, O
// rescaled only when a maximum grows); P packed straight from the S
// accumulators into A fragments; O += P V with V through ldmatrix.trans. A
// 64-key tile gives each softmax step 128 tensor-core products, so the
// softmax chain is not what bounds a warp. Each row ends as a partial state
// (unnormalised O, maximum, sum) in the same layout as the decode kernel's
// partial states, one per (sequence, KV unit, chunk); the merge kernel
// combines them with the states of the member's own suffix.
//
// The grid runs before the decode grid of the same call, on the whole GPU;
// the decode grid (which streams only the members' own suffixes) starts its
// work once this grid is complete.
#include "common.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace pa {
namespace {

constexpr int kPxWarps = 4;
constexpr int kPxThreads = 32 * kPxWarps;
constexpr int kPxRows = 16 * kPxWarps;  // rows of a CTA
constexpr int kPxTile = 64;             // keys per ring stage
constexpr int kPxStages = 3;
constexpr int kPxMaxEntries = 256;      // block-table entries of one chunk held in shared memory
constexpr uint32_t kFullMask = 0xffffffffu;

template <int D>
struct PxGeom {
  static constexpr int kBoxes = D * 2 / 128;          // 128-byte columns of a row
  static constexpr int kBoxBytes = kPxTile * 128;     // one column of a 16-key tile
  static constexpr int kTileBytes = kPxTile * D * 2;  // K (or V) of one stage
  static constexpr int kStageBytes = 2 * kTileBytes;
  static constexpr int kSmemBytes = 1024 + kPxStages * kStageBytes + 2 * kPxStages * 8 + 16 +
                                    kPxMaxEntries * 4;
};

struct PxParams {
  DecodeParams p;
  PrefixGroups pg;
  int group;  // query heads per KV unit
};

// Address of 16-byte chunk `chunk` of key row `row` in a stage tile whose
// 128-byte columns are kBoxBytes apart, chunks swizzled by row % 8 as the TMA
// 128-byte swizzle stores them.
template <int box_bytes>
__device__ __forceinline__ uint32_t px_addr(uint32_t base, int row, int chunk) {
  return base + (chunk >> 3) * box_bytes + row * 128 + (((chunk & 7) ^ (row & 7)) << 4);
}

__device__ __forceinline__ uint32_t px_pack(float lo, float hi, bf16*) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}
__device__ __forceinline__ uint32_t px_pack(float lo, float hi, f16*) {
  __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

template <typename T>
__device__ __forceinline__ void px_mma(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  if constexpr (std::is_same<T, bf16>::value) mma_bf16(d, a, b0, b1);
  else mma_f16(d, a, b0, b1);
}

template <typename T, int D>
__global__ void __launch_bounds__(kPxThreads, 2)
prefix_attn_kernel(const __grid_constant__ CUtensorMap tmap_k, const __grid_constant__ CUtensorMap tmap_v,
                   const PxParams xp) {
  using Gm = PxGeom<D>;
  constexpr int KS = D / 16;        // 16-column steps of d
  constexpr int NT = kPxTile / 8;   // 8-key tiles of S
  const DecodeParams& p = xp.p;
  const PrefixGroups& pg = xp.pg;
  const int G = xp.group;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gid = lane >> 2, tig = lane & 3;

  const int unit = blockIdx.y;
  const int grp = blockIdx.z / pg.num_chunks;
  const int chunk = blockIdx.z % pg.num_chunks;
  const int bs = p.block_size;
  const int lbs = 31 - __clz(bs);  // block sizes are powers of two
  int a, b, plen;
  const bool clamped = prefix_group(pg, grp, p.num_seqs, p.max_blocks_per_seq, bs, a, b, plen);
  if (clamped && threadIdx.x == 0 && blockIdx.x == 0 && unit == 0 && chunk == 0)
    flag_error(p.debug_err, PA_DEVERR_PREFIX);
  const int rows = (b - a) * G;
  const int row0 = blockIdx.x * kPxRows;
  const int k0 = chunk * pg.chunk_len;
  const int k1 = min(plen, k0 + pg.chunk_len);
  if (row0 >= rows || k0 >= k1) return;  // uniform over the CTA, before any barrier
  const int ntiles = (k1 - k0 + kPxTile - 1) / kPxTile;

  extern __shared__ unsigned char px_smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(px_smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t stage0 = smem_u32(smem);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kPxStages * Gm::kStageBytes);
  int* s_abort = reinterpret_cast<int*>(bars + 2 * kPxStages);
  int* s_ent = s_abort + 4;
  auto full_bar = [&](int s) { return smem_u32(&bars[s]); };
  auto empty_bar = [&](int s) { return smem_u32(&bars[kPxStages + s]); };

  // the chunk's blocks, from the group's first member's table
  const int j0 = k0 >> lbs;
  const int nent = ((k1 - 1) >> lbs) - j0 + 1;  // <= chunk_len / bs <= kPxMaxEntries
  const int32_t* lead = p.block_tables + static_cast<int64_t>(a) * p.max_blocks_per_seq;
  bool bad = false;
  for (int i = threadIdx.x; i < nent; i += kPxThreads) {
    int e = lead[j0 + i];
    if (e < 0 || e >= p.num_blocks) {
      flag_error(p.debug_err, PA_DEVERR_BLOCK_RANGE);
      e = -1;
      bad = true;
    }
    s_ent[i] = e;
  }
  if (threadIdx.x < kPxStages) {
    mbar_init(full_bar(threadIdx.x), kPxWarps);  // each warp's first lane issues a share of a tile
    mbar_init(empty_bar(threadIdx.x), kPxWarps);
  }
  if (threadIdx.x == 0) *s_abort = 0;
  mbar_init_fence();
  // every block of the chunk in range: tiles inside the chunk need no masks
  const bool all_valid = __syncthreads_and(!bad);

  const int kvh = kv_head_of(p, unit);
  const int hkv = p.kv_heads_phys;
  // TMA of key tile i into stage s: one box per 128-byte column per block
  // the tile touches, K and V; blocks flagged out of range are skipped
  // (their keys are masked below). A single issuing thread manages only a
  // few boxes per microsecond, so the first lane of every warp issues its
  // share (box b goes to warp b % kPxWarps) and arrives on the stage's
  // barrier with the bytes of its own boxes.
  auto issue = [&](int i, int s) {
    const int t0 = k0 + i * kPxTile;
    const int bh = bs < kPxTile ? bs : kPxTile;  // rows per box
    const int nsub = kPxTile / bh;
    const uint32_t kdst = stage0 + s * Gm::kStageBytes;
    const uint32_t vdst = kdst + Gm::kTileBytes;
    constexpr int kBoxesPerSub = 2 * Gm::kBoxes;  // K and V columns of one block
    uint32_t tx = 0;
    for (int bx = warp; bx < nsub * kBoxesPerSub; bx += kPxWarps) {
      const int h = bx / kBoxesPerSub;
      const int tok = t0 + h * bh;
      if (tok < k1 && s_ent[(tok >> lbs) - j0] >= 0) tx += bh * 128;
    }
    mbar_arrive_expect_tx(full_bar(s), tx);
    for (int bx = warp; bx < nsub * kBoxesPerSub; bx += kPxWarps) {
      const int h = bx / kBoxesPerSub, r = bx % kBoxesPerSub;
      const int tok = t0 + h * bh;
      if (tok >= k1) continue;
      const int e = s_ent[(tok >> lbs) - j0];
      if (e < 0) continue;
      const int z = e * hkv + kvh;
      const int off = tok & (bs - 1);
      const int c = r >> 1;
      if ((r & 1) == 0)
        tma_load_3d(kdst + c * Gm::kBoxBytes + h * bh * 128, &tmap_k, c * 64, off, z, full_bar(s));
      else
        tma_load_3d(vdst + c * Gm::kBoxBytes + h * bh * 128, &tmap_v, c * 64, off, z, full_bar(s));
    }
  };
  if (lane == 0)
    for (int i = 0; i < kPxStages && i < ntiles; ++i) issue(i, i);

  // every member of this CTA's rows must hold the same blocks in the chunk
  // (checked by the first KV unit's CTAs only, while the first tiles load)
  if (unit == 0) {
    const int m0 = row0 / G, m1 = min(b - a, (row0 + kPxRows + G - 1) / G);
    for (int i = threadIdx.x; i < (m1 - m0) * nent; i += kPxThreads) {
      const int m = m0 + i / nent, j = i % nent;
      if (m == 0) continue;
      const int e = p.block_tables[static_cast<int64_t>(a + m) * p.max_blocks_per_seq + j0 + j];
      if (e != lead[j0 + j]) flag_error(p.debug_err, PA_DEVERR_PREFIX);
    }
  }

  // this warp's rows: gid and gid + 8 of its 16
  const int r_a = row0 + warp * 16 + gid, r_b = r_a + 8;
  const bool ok_a = r_a < rows, ok_b = r_b < rows;
  const int seq_a = a + (ok_a ? r_a / G : 0), seq_b = a + (ok_b ? r_b / G : 0);
  const int h_a = ok_a ? r_a % G : 0, h_b = ok_b ? r_b % G : 0;
  const T* qa = static_cast<const T*>(p.q) + (static_cast<int64_t>(seq_a) * p.num_heads + unit * G + h_a) * D;
  const T* qb = static_cast<const T*>(p.q) + (static_cast<int64_t>(seq_b) * p.num_heads + unit * G + h_b) * D;
  uint32_t qf[KS][4];
#pragma unroll
  for (int k = 0; k < KS; ++k) {
    qf[k][0] = ok_a ? *reinterpret_cast<const uint32_t*>(qa + 16 * k + 2 * tig) : 0u;
    qf[k][1] = ok_b ? *reinterpret_cast<const uint32_t*>(qb + 16 * k + 2 * tig) : 0u;
    qf[k][2] = ok_a ? *reinterpret_cast<const uint32_t*>(qa + 16 * k + 8 + 2 * tig) : 0u;
    qf[k][3] = ok_b ? *reinterpret_cast<const uint32_t*>(qb + 16 * k + 8 + 2 * tig) : 0u;
  }

  float o[2 * KS][4];
#pragma unroll
  for (int n = 0; n < 2 * KS; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
  float m_a = -INFINITY, m_b = -INFINITY, l_a = 0.f, l_b = 0.f;

  for (int i = 0; i < ntiles; ++i) {
    const int s = i % kPxStages;
    const uint32_t par = (i / kPxStages) & 1u;
    const bool got = mbar_wait_bounded(full_bar(s), par);
    if (!__all_sync(kFullMask, got)) {
      if (lane == 0) {
        flag_error(p.debug_err, PA_DEVERR_TIMEOUT);
        atomicExch(s_abort, 1);
      }
      break;
    }
    const uint32_t kbase = stage0 + s * Gm::kStageBytes;
    const uint32_t vbase = kbase + Gm::kTileBytes;
    const int t0 = k0 + i * kPxTile;

    // S = Q K^T: 16 rows x 64 keys, as eight independent 8-key tiles
    float sc[NT][4];
#pragma unroll
    for (int n = 0; n < NT; ++n) sc[n][0] = sc[n][1] = sc[n][2] = sc[n][3] = 0.f;
#pragma unroll
    for (int k = 0; k < KS; ++k) {
#pragma unroll
      for (int n = 0; n < NT; n += 2) {
        uint32_t r0, r1, r2, r3;
        ldsm_x4(px_addr<Gm::kBoxBytes>(kbase, 8 * n + (lane >> 4) * 8 + (lane & 7), 2 * k + ((lane >> 3) & 1)),
                r0, r1, r2, r3);
        px_mma<T>(sc[n], qf[k], r0, r1);
        px_mma<T>(sc[n + 1], qf[k], r2, r3);
      }
    }
#pragma unroll
    for (int n = 0; n < NT; ++n)
#pragma unroll
      for (int e = 0; e < 4; ++e) sc[n][e] *= p.scale_log2;
    // keys past the chunk, or in a block flagged out of range, do not count
    // (their rows of the stage hold stale data: scores are replaced, values
    // zeroed below, so no NaN or infinity reaches O)
    uint64_t vmask = ~0ull;  // bit k: key t0 + k is valid
    const bool full = all_valid && t0 + kPxTile <= k1;
    if (!full) {
      vmask = 0;
#pragma unroll
      for (int k = 0; k < kPxTile; k += 8) {
        const int tok = t0 + k;
        if (tok < k1 && s_ent[(tok >> lbs) - j0] >= 0)
          vmask |= static_cast<uint64_t>(tok + 8 <= k1 ? 0xffu : ((1u << (k1 - tok)) - 1u)) << k;
      }
#pragma unroll
      for (int n = 0; n < NT; ++n)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const bool valid = (vmask >> (8 * n + 2 * tig + e)) & 1ull;
          sc[n][e] = valid ? sc[n][e] : -INFINITY;
          sc[n][2 + e] = valid ? sc[n][2 + e] : -INFINITY;
        }
    }
    float x_a = -INFINITY, x_b = -INFINITY;
#pragma unroll
    for (int n = 0; n < NT; ++n) {
      x_a = fmaxf(x_a, fmaxf(sc[n][0], sc[n][1]));
      x_b = fmaxf(x_b, fmaxf(sc[n][2], sc[n][3]));
    }
#pragma unroll
    for (int off = 1; off < 4; off <<= 1) {
      x_a = fmaxf(x_a, __shfl_xor_sync(kFullMask, x_a, off));
      x_b = fmaxf(x_b, __shfl_xor_sync(kFullMask, x_b, off));
    }
    // rescale O only when some row's maximum grew (rarely, once the maxima settle)
    if (__any_sync(kFullMask, x_a > m_a || x_b > m_b)) {
      const float n_a = fmaxf(m_a, x_a), n_b = fmaxf(m_b, x_b);
      const float al_a = n_a == -INFINITY ? 1.f : exp2f(m_a - n_a);  // 0 while m is -inf
      const float al_b = n_b == -INFINITY ? 1.f : exp2f(m_b - n_b);
      m_a = n_a;
      m_b = n_b;
      l_a *= al_a;
      l_b *= al_b;
#pragma unroll
      for (int n = 0; n < 2 * KS; ++n) {
        o[n][0] *= al_a;
        o[n][1] *= al_a;
        o[n][2] *= al_b;
        o[n][3] *= al_b;
      }
    }
    const float b_a = m_a == -INFINITY ? 0.f : m_a, b_b = m_b == -INFINITY ? 0.f : m_b;
    // O += P V, one 16-key step at a time: P of keys 16j.. as the A operand
    // (rows gid / gid + 8), V rows 16j.. through transposed loads
#pragma unroll
    for (int j = 0; j < NT / 2; ++j) {
      float pr[2][4];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        pr[h][0] = exp2f(sc[2 * j + h][0] - b_a);
        pr[h][1] = exp2f(sc[2 * j + h][1] - b_a);
        pr[h][2] = exp2f(sc[2 * j + h][2] - b_b);
        pr[h][3] = exp2f(sc[2 * j + h][3] - b_b);
        l_a += pr[h][0] + pr[h][1];
        l_b += pr[h][2] + pr[h][3];
      }
      uint32_t pa4[4];
      pa4[0] = px_pack(pr[0][0], pr[0][1], static_cast<T*>(nullptr));
      pa4[1] = px_pack(pr[0][2], pr[0][3], static_cast<T*>(nullptr));
      pa4[2] = px_pack(pr[1][0], pr[1][1], static_cast<T*>(nullptr));
      pa4[3] = px_pack(pr[1][2], pr[1][3], static_cast<T*>(nullptr));
      const uint32_t km = static_cast<uint32_t>(vmask >> (16 * j)) & 0xffffu;
      const uint32_t lo = ((km >> (2 * tig)) & 1u ? 0x0000ffffu : 0u) | ((km >> (2 * tig + 1)) & 1u ? 0xffff0000u : 0u);
      const uint32_t hi = ((km >> (8 + 2 * tig)) & 1u ? 0x0000ffffu : 0u) |
                          ((km >> (9 + 2 * tig)) & 1u ? 0xffff0000u : 0u);
#pragma unroll
      for (int c = 0; c < KS; ++c) {
        uint32_t r0, r1, r2, r3;
        ldsm_x4_trans(px_addr<Gm::kBoxBytes>(vbase, 16 * j + ((lane >> 3) & 1) * 8 + (lane & 7), 2 * c + (lane >> 4)),
                      r0, r1, r2, r3);
        if (!full) {
          // r0, r2 hold keys 2tig, 2tig + 1 of the step; r1, r3 keys 8 + 2tig, 9 + 2tig
          r0 &= lo;
          r2 &= lo;
          r1 &= hi;
          r3 &= hi;
        }
        px_mma<T>(o[2 * c], pa4, r0, r1);
        px_mma<T>(o[2 * c + 1], pa4, r2, r3);
      }
    }

    // stage s is free again: once every warp is done with it, each warp's
    // first lane issues its share of the tile kPxStages ahead
    __syncwarp();
    if (lane == 0) mbar_arrive(empty_bar(s));
    if (lane == 0 && i + kPxStages < ntiles) {
      if (!mbar_wait_bounded(empty_bar(s), par)) {
        flag_error(p.debug_err, PA_DEVERR_TIMEOUT);
        atomicExch(s_abort, 1);
      } else {
        fence_proxy_async_smem();
        issue(i + kPxStages, s);
      }
    }
    __syncwarp();
    if (*reinterpret_cast<volatile int*>(s_abort)) break;
  }

  if (*reinterpret_cast<volatile int*>(s_abort) == 0) {
#pragma unroll
    for (int off = 1; off < 4; off <<= 1) {
      l_a += __shfl_xor_sync(kFullMask, l_a, off);
      l_b += __shfl_xor_sync(kFullMask, l_b, off);
    }
    const int stride = state_floats(G, D);
    const int64_t units = p.num_kv_heads;
    auto store_row = [&](bool ok, int seq, int h, float m, float l, int upper) {
      if (!ok) return;
      float* st = pg.ws_prefix + ((static_cast<int64_t>(seq) * units + unit) * pg.num_chunks + chunk) * stride;
#pragma unroll
      for (int n = 0; n < 2 * KS; ++n)
        *reinterpret_cast<float2*>(st + h * D + 8 * n + 2 * tig) =
            make_float2(o[n][2 * upper], o[n][2 * upper + 1]);
      if (tig == 0) {
        st[G * D + h] = m;
        st[G * D + G + h] = l;
      }
    };
    store_row(ok_a, seq_a, h_a, m_a, l_a, 0);
    store_row(ok_b, seq_b, h_b, m_b, l_b, 1);
  } else if (threadIdx.x == 0) {
    // give copies still in flight a short while to land before the CTA leaves
    for (int s = 0; s < kPxStages; ++s) mbar_wait_bounded(full_bar(s), 0, 10000000ull);
  }
}

template <typename T, int D>
cudaError_t launch_px(const PxParams& xp, dim3 grid, cudaStream_t stream) {
  const DecodeParams& p = xp.p;
  CUtensorMap mk, mv;
  const int64_t bxh = static_cast<int64_t>(p.num_blocks) * p.kv_heads_phys;
  if (!make_cache_map(&mk, p.k_cache, D, 2, p.block_size, kPxTile, bxh) ||
      !make_cache_map(&mv, p.v_cache, D, 2, p.block_size, kPxTile, bxh))
    return cudaErrorInvalidValue;
  auto kernel = prefix_attn_kernel<T, D>;
  static std::atomic<unsigned long long> attr_set{0};
  cudaError_t e = set_smem_limit_once(reinterpret_cast<const void*>(kernel), PxGeom<D>::kSmemBytes, attr_set);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(kPxThreads);
  cfg.dynamicSmemBytes = PxGeom<D>::kSmemBytes;
  cfg.stream = stream;
  e = cudaLaunchKernelEx(&cfg, kernel, mk, mv, xp);
  if (e == cudaSuccess) note_launches(1);
  return e;
}

}  // namespace

int prefix_row_tiles(int max_group_size, int group) {
  return static_cast<int>((static_cast<int64_t>(max_group_size) * group + kPxRows - 1) / kPxRows);
}

int prefix_chunk_step(int block_size) {
  // chunks are whole key tiles (and whole blocks)
  return block_size > kPxTile ? block_size : kPxTile;
}

int prefix_max_chunk_len(int block_size) {
  // the chunk's table entries fit the CTA's shared array
  return (kPxMaxEntries - 1) * block_size;
}

cudaError_t launch_prefix_attn(const DecodeParams& p, const PrefixGroups& pg, int head_dim,
                               pa_dtype dtype, cudaStream_t stream) {
  PxParams xp{};
  xp.p = p;
  xp.pg = pg;
  xp.group = p.num_heads / p.num_kv_heads;
  dim3 grid(prefix_row_tiles(pg.max_group_size, xp.group), p.num_kv_heads, pg.num_groups * pg.num_chunks);
  if (dtype == PA_BF16) {
    if (head_dim == 128) return launch_px<bf16, 128>(xp, grid, stream);
    return launch_px<bf16, 64>(xp, grid, stream);
  }
  if (head_dim == 128) return launch_px<f16, 128>(xp, grid, stream);
  return launch_px<f16, 64>(xp, grid, stream);
}

}  // namespace pa
