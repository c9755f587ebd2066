// General paged decode on the CUDA cores.
//
// One CTA of 4 warps handles one (partition, KV head, sequence). The warps
// take the partition's blocks round-robin. Lane l owns head_dim/32
// consecutive elements of every row, so a K or V row is one coalesced
// warp-wide load; q.k is a per-lane partial dot product finished with
// xor-shuffles. Each warp keeps the online-softmax state (running max m,
// running sum l, accumulator acc rescaled by exp(m_old - m_new)) for the G
// query heads of its KV head, four tokens at a time; the four warp states
// are merged through shared memory at the end. With a single partition the
// CTA writes the output row; otherwise it writes a normalised float32
// partial plus (m, l) and reduce_partitions_kernel merges them.
#include "common.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace pa {
namespace {

constexpr int kWarps = 4;
constexpr int kChunk = 4;  // tokens per online-softmax update

template <typename QT, typename KT, int D, int G>
__global__ void __launch_bounds__(kWarps * 32)
decode_simt_kernel(const DecodeParams p) {
  constexpr int EPL = D / 32;  // elements per lane
  constexpr bool kFp8 = is_fp8<KT>::value;
  const int part = blockIdx.x;
  const int kvh = blockIdx.y;
  const int seq = blockIdx.z;
  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;

  const int ctx = clamp_context(p, seq);
  const int tok_begin = part * p.partition_size;
  const int tok_end = min(ctx, tok_begin + p.partition_size);
  const bool single = p.num_partitions == 1;
  if (tok_begin >= tok_end && !(single && part == 0)) return;  // partition past the end

  // query rows of this KV head's group, widened to float
  float qf[G][EPL];
  const QT* q = static_cast<const QT*>(p.q);
#pragma unroll
  for (int j = 0; j < G; ++j)
    load_float<QT, EPL>(q + (static_cast<int64_t>(seq) * p.num_heads + kvh * G + j) * D + lane * EPL,
                        qf[j]);

  float m[G], l[G], acc[G][EPL];
#pragma unroll
  for (int j = 0; j < G; ++j) {
    m[j] = -INFINITY;
    l[j] = 0.f;
#pragma unroll
    for (int e = 0; e < EPL; ++e) acc[j][e] = 0.f;
  }

  const KT* kc = static_cast<const KT*>(p.k_cache);
  const KT* vc = static_cast<const KT*>(p.v_cache);
  const int bs = p.block_size;
  const int32_t* table = p.block_tables + static_cast<int64_t>(seq) * p.max_blocks_per_seq;
  const int blk_begin = tok_begin / bs;
  const int blk_end = (tok_end + bs - 1) / bs;

  for (int b = blk_begin + warp; b < blk_end; b += kWarps) {
    const int phys = table[b];
    if (phys < 0 || phys >= p.num_blocks) {
      if (lane == 0) flag_error(p.debug_err, PA_DEVERR_BLOCK_RANGE);
      continue;
    }
    const int valid = min(bs, tok_end - b * bs);
    const int64_t hi = static_cast<int64_t>(phys) * p.kv_heads_phys + kv_head_of(p, kvh);
    const int64_t row0 = hi * bs;
    float kscale = 1.f, vscale = 1.f;
    if constexpr (kFp8) {
      kscale = p.k_scale[hi];
      vscale = p.v_scale[hi];
    }
    for (int t0 = 0; t0 < valid; t0 += kChunk) {
      float kf[kChunk][EPL];
#pragma unroll
      for (int u = 0; u < kChunk; ++u) {
        if (t0 + u < valid) {
          load_float<KT, EPL>(kc + (row0 + t0 + u) * D + lane * EPL, kf[u]);
        } else {
#pragma unroll
          for (int e = 0; e < EPL; ++e) kf[u][e] = 0.f;
        }
      }
      float s[kChunk][G];
#pragma unroll
      for (int u = 0; u < kChunk; ++u)
#pragma unroll
        for (int j = 0; j < G; ++j) {
          float d = 0.f;
#pragma unroll
          for (int e = 0; e < EPL; ++e) d = fmaf(qf[j][e], kf[u][e], d);
          s[u][j] = d;
        }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1)
#pragma unroll
        for (int u = 0; u < kChunk; ++u)
#pragma unroll
          for (int j = 0; j < G; ++j) s[u][j] += __shfl_xor_sync(0xffffffffu, s[u][j], off);

      float vf[kChunk][EPL];
#pragma unroll
      for (int u = 0; u < kChunk; ++u) {
        if (t0 + u < valid) {
          load_float<KT, EPL>(vc + (row0 + t0 + u) * D + lane * EPL, vf[u]);
        } else {
#pragma unroll
          for (int e = 0; e < EPL; ++e) vf[u][e] = 0.f;
        }
      }
#pragma unroll
      for (int j = 0; j < G; ++j) {
        float cmax = -INFINITY;
#pragma unroll
        for (int u = 0; u < kChunk; ++u) {
          s[u][j] = (t0 + u < valid) ? s[u][j] * (p.scale_log2 * kscale) : -INFINITY;
          cmax = fmaxf(cmax, s[u][j]);
        }
        const float m_new = fmaxf(m[j], cmax);
        const float alpha = exp2f(m[j] - m_new);  // 0 when m[j] is -inf
        m[j] = m_new;
        float psum = 0.f;
        float pu[kChunk];
#pragma unroll
        for (int u = 0; u < kChunk; ++u) {
          pu[u] = exp2f(s[u][j] - m_new);
          psum += pu[u];
        }
        l[j] = l[j] * alpha + psum;
#pragma unroll
        for (int e = 0; e < EPL; ++e) {
          float a = acc[j][e] * alpha;
#pragma unroll
          for (int u = 0; u < kChunk; ++u) a = fmaf(pu[u] * vscale, vf[u][e], a);
          acc[j][e] = a;
        }
      }
    }
  }

  // merge the warps' states
  __shared__ float sm_m[kWarps][G];
  __shared__ float sm_l[kWarps][G];
  __shared__ float sm_acc[kWarps][G][D];
  if (lane == 0) {
#pragma unroll
    for (int j = 0; j < G; ++j) {
      sm_m[warp][j] = m[j];
      sm_l[warp][j] = l[j];
    }
  }
#pragma unroll
  for (int j = 0; j < G; ++j)
#pragma unroll
    for (int e = 0; e < EPL; ++e) sm_acc[warp][j][lane * EPL + e] = acc[j][e];
  __syncthreads();

  for (int idx = threadIdx.x; idx < G * D; idx += kWarps * 32) {
    const int j = idx / D;
    const int e = idx % D;
    float mt = -INFINITY;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) mt = fmaxf(mt, sm_m[w][j]);
    float lt = 0.f, at = 0.f;
    if (mt != -INFINITY) {
#pragma unroll
      for (int w = 0; w < kWarps; ++w) {
        const float f = exp2f(sm_m[w][j] - mt);
        lt += sm_l[w][j] * f;
        at += sm_acc[w][j][e] * f;
      }
    }
    const float o = lt > 0.f ? at / lt : 0.f;
    const int h = kvh * G + j;
    if (single) {
      QT* out = static_cast<QT*>(p.out);
      out[(static_cast<int64_t>(seq) * p.num_heads + h) * D + e] = from_float(o, static_cast<QT*>(nullptr));
    } else {
      const int64_t slot = (static_cast<int64_t>(seq) * p.num_heads + h) * p.num_partitions + part;
      p.ws_acc[slot * D + e] = o;
      if (e == 0) {
        p.ws_ml[slot * 2] = mt;
        p.ws_ml[slot * 2 + 1] = lt;
      }
    }
  }
}

// Merge the partitions of one (sequence, query head): with M = max_p m_p and
// w_p = 2^(m_p - M) * l_p, out = sum_p w_p * o_p / sum_p w_p (the partials
// o_p are normalised). Partitions are taken kReduceThreads at a time: one
// thread per partition loads its (m_p, l_p), and the rows are float4
// elements of o_p with the threads split into groups of partitions, so one
// round issues the loads of many partitions at once (kBatch per thread, all
// independent). A running maximum carries the merge across chunks, so any
// number of partitions fits the kernel's fixed shared memory.
constexpr int kReduceThreads = 256;

template <typename QT, int D>
__global__ void __launch_bounds__(kReduceThreads) reduce_partitions_kernel(const DecodeParams p) {
  constexpr int NT = kReduceThreads;
  constexpr int NE4 = D / 4;      // float4 elements per row: 16, 32 or 64
  constexpr int NGRP = NT / NE4;  // groups of partitions: 16, 8 or 4
  constexpr int kBatch = 4;       // row loads a thread keeps in flight
  constexpr int kWarpsR = NT / 32;
  griddep_wait();
  // the partition kernel is complete: rearm its work counter for the next call
  if (p.claim != nullptr && blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0) *p.claim = 0;
  const int h = blockIdx.x;
  const int seq = blockIdx.y;
  const int ctx = clamp_context(p, seq);
  const int nparts = min((ctx + p.partition_size - 1) / p.partition_size, p.num_partitions);
  const int64_t base = (static_cast<int64_t>(seq) * p.num_heads + h) * p.num_partitions;
  const int e4 = threadIdx.x % NE4, grp = threadIdx.x / NE4;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __shared__ float s_w[NT];
  __shared__ float s_red[kWarpsR];
  __shared__ float4 s_part[NT];
  const float4* rows = reinterpret_cast<const float4*>(p.ws_acc + base * D) + e4;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  float run = -INFINITY, den = 0.f;  // running maximum and denominator (uniform over the CTA)
  for (int c0 = 0; c0 < nparts; c0 += NT) {
    const int nin = min(NT, nparts - c0);
    float m = -INFINITY, l = 0.f;
    if (static_cast<int>(threadIdx.x) < nin) {
      const float2 ml = __ldcg(reinterpret_cast<const float2*>(p.ws_ml) + base + c0 + threadIdx.x);
      m = ml.x;
      l = ml.y;
    }
    float4 v[kBatch];
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      const int j = grp + u * NGRP;
      v[u] = j < nin ? __ldcg(rows + static_cast<int64_t>(c0 + j) * NE4) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    // the chunk's maximum
    float cm = m;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) cm = fmaxf(cm, __shfl_xor_sync(0xffffffffu, cm, off));
    if (lane == 0) s_red[warp] = cm;
    __syncthreads();
    cm = s_red[0];
#pragma unroll
    for (int w = 1; w < kWarpsR; ++w) cm = fmaxf(cm, s_red[w]);
    const float nm = fmaxf(run, cm);
    const float scale = run == -INFINITY ? 0.f : exp2f(run - nm);
    const float w = m == -INFINITY ? 0.f : exp2f(m - nm) * l;
    s_w[threadIdx.x] = w;
    float sw = w;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) sw += __shfl_xor_sync(0xffffffffu, sw, off);
    __syncthreads();  // every thread has read s_red (maxima) and written s_w
    if (lane == 0) s_red[warp] = sw;
    __syncthreads();
    float d = 0.f;
#pragma unroll
    for (int i = 0; i < kWarpsR; ++i) d += s_red[i];
    den = den * scale + d;
    run = nm;
    acc.x *= scale;
    acc.y *= scale;
    acc.z *= scale;
    acc.w *= scale;
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      const int j = grp + u * NGRP;
      const float wt = j < nin ? s_w[j] : 0.f;
      acc.x = fmaf(wt, v[u].x, acc.x);
      acc.y = fmaf(wt, v[u].y, acc.y);
      acc.z = fmaf(wt, v[u].z, acc.z);
      acc.w = fmaf(wt, v[u].w, acc.w);
    }
    // partitions beyond the first batch of this thread
    for (int j0 = grp + kBatch * NGRP; j0 < nin; j0 += kBatch * NGRP) {
#pragma unroll
      for (int u = 0; u < kBatch; ++u) {
        const int j = j0 + u * NGRP;
        v[u] = j < nin ? __ldcg(rows + static_cast<int64_t>(c0 + j) * NE4) : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int u = 0; u < kBatch; ++u) {
        const int j = j0 + u * NGRP;
        const float wt = j < nin ? s_w[j] : 0.f;
        acc.x = fmaf(wt, v[u].x, acc.x);
        acc.y = fmaf(wt, v[u].y, acc.y);
        acc.z = fmaf(wt, v[u].z, acc.z);
        acc.w = fmaf(wt, v[u].w, acc.w);
      }
    }
    __syncthreads();  // s_w and s_red are rewritten by the next chunk
  }
  s_part[threadIdx.x] = acc;
  __syncthreads();
  if (grp == 0) {
    float4 t = acc;
#pragma unroll
    for (int gi = 1; gi < NGRP; ++gi) {
      const float4 u = s_part[gi * NE4 + e4];
      t.x += u.x;
      t.y += u.y;
      t.z += u.z;
      t.w += u.w;
    }
    const float inv = den > 0.f ? 1.f / den : 0.f;
    QT* out = static_cast<QT*>(p.out) + (static_cast<int64_t>(seq) * p.num_heads + h) * D + 4 * e4;
    out[0] = from_float(t.x * inv, static_cast<QT*>(nullptr));
    out[1] = from_float(t.y * inv, static_cast<QT*>(nullptr));
    out[2] = from_float(t.z * inv, static_cast<QT*>(nullptr));
    out[3] = from_float(t.w * inv, static_cast<QT*>(nullptr));
  }
}

template <typename QT, typename KT, int D>
cudaError_t launch_d(const DecodeParams& p, int group, cudaStream_t stream) {
  dim3 grid(p.num_partitions, p.num_kv_heads, p.num_seqs);
  switch (group) {
    case 1: decode_simt_kernel<QT, KT, D, 1><<<grid, kWarps * 32, 0, stream>>>(p); break;
    case 2: decode_simt_kernel<QT, KT, D, 2><<<grid, kWarps * 32, 0, stream>>>(p); break;
    case 4: decode_simt_kernel<QT, KT, D, 4><<<grid, kWarps * 32, 0, stream>>>(p); break;
    case 8: decode_simt_kernel<QT, KT, D, 8><<<grid, kWarps * 32, 0, stream>>>(p); break;
    default: return cudaErrorInvalidValue;
  }
  cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  note_launches(1);
  if (p.num_partitions == 1) return err;
  dim3 rgrid(p.num_heads, p.num_seqs);
  reduce_partitions_kernel<QT, D><<<rgrid, kReduceThreads, 0, stream>>>(p);
  err = cudaGetLastError();
  if (err == cudaSuccess) note_launches(1);
  return err;
}

template <typename QT, int D>
cudaError_t launch_reduce_pdl(const DecodeParams& p, bool pdl, cudaStream_t stream) {
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.num_heads, p.num_seqs);
  cfg.blockDim = dim3(kReduceThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  cudaError_t err = cudaLaunchKernelEx(&cfg, reduce_partitions_kernel<QT, D>, p);
  if (err == cudaSuccess) note_launches(1);
  return err;
}

template <typename QT, typename KT>
cudaError_t launch_t(const DecodeParams& p, int head_dim, int group, cudaStream_t stream) {
  switch (head_dim) {
    case 64: return launch_d<QT, KT, 64>(p, group, stream);
    case 128: return launch_d<QT, KT, 128>(p, group, stream);
    case 256: return launch_d<QT, KT, 256>(p, group, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

cudaError_t launch_reduce_partitions(const DecodeParams& p, int head_dim, pa_dtype q_dtype,
                                     bool pdl, cudaStream_t stream) {
  const bool b = q_dtype == PA_BF16;
  switch (head_dim) {
    case 64: return b ? launch_reduce_pdl<bf16, 64>(p, pdl, stream) : launch_reduce_pdl<f16, 64>(p, pdl, stream);
    case 128: return b ? launch_reduce_pdl<bf16, 128>(p, pdl, stream) : launch_reduce_pdl<f16, 128>(p, pdl, stream);
    case 256: return b ? launch_reduce_pdl<bf16, 256>(p, pdl, stream) : launch_reduce_pdl<f16, 256>(p, pdl, stream);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_decode_simt(const DecodeParams& p, int head_dim, pa_dtype q_dtype,
                               pa_dtype kv_dtype, cudaStream_t stream) {
  if (p.num_seqs == 0) return cudaSuccess;
  const int group = p.num_heads / p.num_kv_heads;
  if (kv_dtype == PA_F16) return launch_t<f16, f16>(p, head_dim, group, stream);
  if (kv_dtype == PA_BF16) return launch_t<bf16, bf16>(p, head_dim, group, stream);
  if (q_dtype == PA_F16) return launch_t<f16, fp8>(p, head_dim, group, stream);
  return launch_t<bf16, fp8>(p, head_dim, group, stream);
}

}  // namespace pa
