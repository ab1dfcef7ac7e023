// Exact log-sum-exp merge of partial attention results ("ByteScale:
// Communication-Efficient Scaling of LLM Training with a 2048K Context Length
// on 16384 GPUs", research digest, section 3.2: the partial block of each ring
// step is combined with the others).  For one (row, head):
//   M = max_k lse_k,  lse = M + ln sum_k exp(lse_k - M),
//   o = sum_k exp(lse_k - lse) o_k.
// HBM-bound: one warp per (row, head), each lane streams float4 columns of
// every partial (coalesced 512-byte rows at d = 128), and each partial's lse
// is read once; bf16 output.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>

#include "internal.h"

namespace hdp {
namespace {

constexpr int kMergeThreads = 256;  // 8 warps, one (row, head) each

struct BlockSource {  // SPLIT workspace: partials addressed through the plan
  const float* o_part;    // [N_b][C][hq][d]
  const float* lse_part;  // [N_b][hq][C]
  const int32_t* cu;
  const int64_t* bo;
  int32_t n, C, hq;
  long long T;
};

struct RowSource {  // plain arrays: o_parts [m][rows][d], lse_parts [m][rows]
  const float* o_parts;
  const float* lse_parts;
  int32_t m;
  long long rows;
};

// One warp merges the m partials of one row.  lse_at(k) gives lse_k; o_at(k)
// points at o_k's d floats.  Each lse_k is read once: lane j holds the
// partials j, j + 32, ...; the running (max, sum of exp) pair is combined
// across lanes by shuffles, and in the weighted sum lane j's weight
// exp(lse_j - lse) is broadcast to the warp.  Eight partial rows are loaded
// per step (4 KB in flight per warp at d = 128).  Writes d bf16 to `out` and
// returns lse.
constexpr int kMergeUnroll = 8;

__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, off));
  return x;
}
__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) x += __shfl_xor_sync(0xffffffffu, x, off);
  return x;
}

template <int VEC, typename LseAt, typename OAt>
__device__ __forceinline__ float merge_row(int m, int d, int lane, LseAt lse_at, OAt o_at, __nv_bfloat16* out) {
  // pass 1: M = max_k lse_k and S = sum_k exp(lse_k - M), 32 partials at a time
  float M = -INFINITY, S = 0.f;
  float x0 = -INFINITY;  // lane's lse of the first 32 partials, kept for pass 2
  for (int c0 = 0; c0 < m; c0 += 32) {
    const float x = c0 + lane < m ? lse_at(c0 + lane) : -INFINITY;
    if (c0 == 0) x0 = x;
    const float Mn = fmaxf(M, warp_max(x));
    if (Mn != -INFINITY) {
      const float e = x == -INFINITY ? 0.f : expf(x - Mn);
      S = (M == -INFINITY ? 0.f : S * expf(M - Mn)) + warp_sum(e);
      M = Mn;
    }
  }
  float4 acc[VEC];
#pragma unroll
  for (int v = 0; v < VEC; ++v) acc[v] = make_float4(0.f, 0.f, 0.f, 0.f);
  float L = -INFINITY;
  if (M != -INFINITY) {
    L = M + logf(S);
    // pass 2: o = sum_k exp(lse_k - L) o_k
    for (int c0 = 0; c0 < m; c0 += 32) {
      const float x = c0 == 0 ? x0 : (c0 + lane < m ? lse_at(c0 + lane) : -INFINITY);
      const float wl = x == -INFINITY ? 0.f : expf(x - L);
      const int cn = m - c0 < 32 ? m - c0 : 32;
      for (int j0 = 0; j0 < cn; j0 += kMergeUnroll) {
        float w[kMergeUnroll];
        float4 xv[kMergeUnroll][VEC];
#pragma unroll
        for (int u = 0; u < kMergeUnroll; ++u) {
          const int j = j0 + u;
          w[u] = __shfl_sync(0xffffffffu, wl, j & 31);
          if (j >= cn) w[u] = 0.f;
          const float* ok = o_at(c0 + (j < cn ? j : j0));
#pragma unroll
          for (int v = 0; v < VEC; ++v) {
            const int c = (v * 32 + lane) * 4;
            xv[u][v] = (c < d && w[u] != 0.f) ? __ldcs(reinterpret_cast<const float4*>(ok + c))
                                               : make_float4(0.f, 0.f, 0.f, 0.f);
          }
        }
#pragma unroll
        for (int u = 0; u < kMergeUnroll; ++u)
#pragma unroll
          for (int v = 0; v < VEC; ++v) {
            acc[v].x = fmaf(w[u], xv[u][v].x, acc[v].x);
            acc[v].y = fmaf(w[u], xv[u][v].y, acc[v].y);
            acc[v].z = fmaf(w[u], xv[u][v].z, acc[v].z);
            acc[v].w = fmaf(w[u], xv[u][v].w, acc[v].w);
          }
      }
    }
  }
#pragma unroll
  for (int v = 0; v < VEC; ++v) {
    const int c = (v * 32 + lane) * 4;
    if (c < d) {
      __nv_bfloat162 lo = __floats2bfloat162_rn(acc[v].x, acc[v].y);
      __nv_bfloat162 hi = __floats2bfloat162_rn(acc[v].z, acc[v].w);
      uint2 pk;
      pk.x = *reinterpret_cast<uint32_t*>(&lo);
      pk.y = *reinterpret_cast<uint32_t*>(&hi);
      *reinterpret_cast<uint2*>(out + c) = pk;
    }
  }
  return L;
}

__device__ __forceinline__ int32_t doc_of(const int32_t* __restrict__ cu, int32_t n, long long t) {
  int32_t lo = 0, hi = n - 1;
  while (lo < hi) {
    const int32_t mid = (lo + hi + 1) >> 1;
    if (cu[mid] <= t)
      lo = mid;
    else
      hi = mid - 1;
  }
  return lo;
}

// SPLIT partials of the plan's causal blocks.  A work item is 32 rows of one
// 128-row query tile of the plan's FUSED work list (a query tile never
// straddles a chunk edge, since C % 128 == 0, so all its rows have the same
// chunk qc, the same m = qc + 1 partials and the same first block b0) for one
// head h; items run head-fastest, so the 32 warps of consecutive heads stream
// the same rows' partials (hq * d floats each) and output rows contiguously.
// Lane i owns row i for the lse pass: for each partial k the warp reads 32
// consecutive lse values (one 128-byte line), and each lane keeps its row's
// running (max, sum of exp).  The weighted sum then runs eight rows at a time,
// one partial of each per step (eight 512-byte rows in flight at d = 128);
// lane i recomputes row i's weight exp(lse_k - lse) from the lse line (now
// cached) and the eight weights are broadcast to the warp.
template <int VEC>
__global__ void __launch_bounds__(kMergeThreads) k_merge_blocks(BlockSource src, const int32_t* __restrict__ tiles,
                                                                long long ntiles, int d,
                                                                __nv_bfloat16* __restrict__ o,
                                                                float* __restrict__ lse) {
  const int lane = threadIdx.x & 31;
  const long long nwork = ntiles * 4 * src.hq;
  for (long long w = (static_cast<long long>(blockIdx.x) * kMergeThreads + threadIdx.x) >> 5; w < nwork;
       w += (static_cast<long long>(gridDim.x) * kMergeThreads) >> 5) {
    const long long ts = w / src.hq;  // (tile, 32-row sub-block)
    const int32_t h = static_cast<int32_t>(w - ts * src.hq);
    const long long ti = ts >> 2;
    const int sb = static_cast<int>(ts & 3);
    const int4 row0 = __ldg(reinterpret_cast<const int4*>(tiles + ti * 8));
    const int4 row1 = __ldg(reinterpret_cast<const int4*>(tiles + ti * 8 + 4));
    // row0 = {q_row0, q_rows, doc start, key range}; row1 = {-, row offset in the document, -, -}
    const int nrows = min(32, row0.y - sb * 32);
    if (nrows <= 0) continue;
    const long long t0 = static_cast<long long>(row0.x) + sb * 32;  // first token of the item
    const long long p0 = static_cast<long long>(row1.y) + sb * 32;  // its position in the document
    const long long qc = p0 / src.C;
    const long long r0 = p0 - qc * src.C;  // its row in the chunk
    const int32_t doc = doc_of(src.cu, src.n, t0);
    const long long b0 = src.bo[doc] + qc * (qc + 1) / 2;  // block (qc, 0)
    const int m = static_cast<int>(qc + 1);
    const float* lse_h = src.lse_part + (b0 * src.hq + h) * static_cast<long long>(src.C) + r0;
    const long long lse_step = static_cast<long long>(src.hq) * src.C;  // next block, same head and row
    const bool mine = lane < nrows;
    // lse pass: lane = row
    float M = -INFINITY, S = 0.f;
    for (int k = 0; k < m; ++k) {
      const float x = mine ? __ldg(lse_h + k * lse_step + lane) : -INFINITY;
      const float Mn = fmaxf(M, x);
      if (Mn != -INFINITY) {
        S = (M == -INFINITY ? 0.f : S * expf(M - Mn)) + (x == -INFINITY ? 0.f : expf(x - Mn));
        M = Mn;
      }
    }
    const float L = M == -INFINITY ? -INFINITY : M + logf(S);
    if (mine) lse[static_cast<long long>(h) * src.T + t0 + lane] = L;
    // weighted sum, eight rows at a time
    const long long o_step = static_cast<long long>(src.C) * src.hq * d;  // next block, same row and head
    const float* o_base = src.o_part + ((b0 * src.C + r0) * src.hq + h) * static_cast<long long>(d);
    for (int g0 = 0; g0 < nrows; g0 += 8) {
      float4 acc[8][VEC];
#pragma unroll
      for (int u = 0; u < 8; ++u)
#pragma unroll
        for (int v = 0; v < VEC; ++v) acc[u][v] = make_float4(0.f, 0.f, 0.f, 0.f);
      for (int k = 0; k < m; ++k) {
        float4 xv[8][VEC];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const float* orow = o_base + k * o_step + static_cast<long long>(g0 + u) * src.hq * d;
#pragma unroll
          for (int v = 0; v < VEC; ++v) {
            const int c = (v * 32 + lane) * 4;
            xv[u][v] = (c < d && g0 + u < nrows) ? __ldcs(reinterpret_cast<const float4*>(orow + c))
                                                  : make_float4(0.f, 0.f, 0.f, 0.f);
          }
        }
        const float x = mine ? __ldg(lse_h + k * lse_step + lane) : -INFINITY;
        const float wl = x == -INFINITY ? 0.f : expf(x - L);
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const float wu = __shfl_sync(0xffffffffu, wl, (g0 + u) & 31);
#pragma unroll
          for (int v = 0; v < VEC; ++v) {
            acc[u][v].x = fmaf(wu, xv[u][v].x, acc[u][v].x);
            acc[u][v].y = fmaf(wu, xv[u][v].y, acc[u][v].y);
            acc[u][v].z = fmaf(wu, xv[u][v].z, acc[u][v].z);
            acc[u][v].w = fmaf(wu, xv[u][v].w, acc[u][v].w);
          }
        }
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        if (g0 + u >= nrows) break;
        __nv_bfloat16* out = o + ((t0 + g0 + u) * src.hq + h) * static_cast<long long>(d);
#pragma unroll
        for (int v = 0; v < VEC; ++v) {
          const int c = (v * 32 + lane) * 4;
          if (c < d) {
            __nv_bfloat162 lo = __floats2bfloat162_rn(acc[u][v].x, acc[u][v].y);
            __nv_bfloat162 hi = __floats2bfloat162_rn(acc[u][v].z, acc[u][v].w);
            uint2 pk;
            pk.x = *reinterpret_cast<uint32_t*>(&lo);
            pk.y = *reinterpret_cast<uint32_t*>(&hi);
            *reinterpret_cast<uint2*>(out + c) = pk;
          }
        }
      }
    }
  }
}

template <int VEC>
__global__ void __launch_bounds__(kMergeThreads) k_merge_rows(RowSource src, int d, __nv_bfloat16* __restrict__ o,
                                                              float* __restrict__ lse) {
  const int lane = threadIdx.x & 31;
  for (long long r = (static_cast<long long>(blockIdx.x) * kMergeThreads + threadIdx.x) >> 5; r < src.rows;
       r += (static_cast<long long>(gridDim.x) * kMergeThreads) >> 5) {
    auto lse_at = [&](int k) { return __ldg(src.lse_parts + k * src.rows + r); };
    auto o_at = [&](int k) { return src.o_parts + (k * src.rows + r) * static_cast<long long>(d); };
    const float L = merge_row<VEC>(src.m, d, lane, lse_at, o_at, o + r * static_cast<long long>(d));
    if (lane == 0) lse[r] = L;
  }
}

int merge_grid(long long warps) {
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  long long g = (warps * 32 + kMergeThreads - 1) / kMergeThreads;
  const long long cap = static_cast<long long>(sms) * 16;
  if (g > cap) g = cap;
  if (g < 1) g = 1;
  return static_cast<int>(g);
}

}  // namespace

// Shared with attn_fwd.cu (SPLIT mode).
hdp_status_t launch_merge_blocks(const hdp_plan_s* plan, const float* o_part, const float* lse_part, int32_t hq,
                                 int32_t d, void* o, float* lse, cudaStream_t st) {
  BlockSource src{o_part, lse_part, plan->v.cu_seqlens, plan->v.block_offsets, plan->v.num_docs,
                  plan->v.capacity, hq, plan->v.total_tokens};
  const long long ntiles = plan->v.num_tiles_fused;
  const int g = merge_grid(ntiles * 4 * hq);
  if (d <= 128)
    k_merge_blocks<1><<<g, kMergeThreads, 0, st>>>(src, plan->v.tiles_fused, ntiles, d,
                                                   static_cast<__nv_bfloat16*>(o), lse);
  else
    k_merge_blocks<2><<<g, kMergeThreads, 0, st>>>(src, plan->v.tiles_fused, ntiles, d,
                                                   static_cast<__nv_bfloat16*>(o), lse);
  note_launch();
  HDP_CUDA_TRY(cudaGetLastError());
  return HDP_OK;
}

}  // namespace hdp

using namespace hdp;

extern "C" hdp_status_t hdp_lse_merge(hdp_plan_t plan, const float* o_part, const float* lse_part, int32_t hq,
                                      int32_t d, void* o, float* lse, void* stream) {
  if (!plan || !o_part || !lse_part || !o || !lse) return fail(HDP_ERR_INVALID_ARGUMENT, "hdp_lse_merge: NULL argument");
  if (hq < 1) return fail(HDP_ERR_INVALID_ARGUMENT, "hdp_lse_merge: hq must be >= 1");
  if (d != 64 && d != 128) return fail(HDP_ERR_UNSUPPORTED, "hdp_lse_merge: d must be 64 or 128");
  if (plan->v.capacity % kTile != 0)
    return fail(HDP_ERR_INVALID_ARGUMENT, "hdp_lse_merge: the plan's capacity must be a multiple of 128");
  if ((reinterpret_cast<uintptr_t>(o_part) & 15) || (reinterpret_cast<uintptr_t>(o) & 7))
    return fail(HDP_ERR_INVALID_ARGUMENT, "hdp_lse_merge: o_part must be 16-byte and o 8-byte aligned");
  return launch_merge_blocks(plan, o_part, lse_part, hq, d, o, lse, static_cast<cudaStream_t>(stream));
}

extern "C" hdp_status_t hdp_lse_merge_rows(int32_t m, int64_t rows, int32_t d, const float* o_parts,
                                           const float* lse_parts, void* o, float* lse, void* stream) {
  if (m < 1 || rows < 0 || d < 4 || d > 256 || d % 4 != 0)
    return fail(HDP_ERR_INVALID_ARGUMENT, "hdp_lse_merge_rows: need m >= 1, rows >= 0, d % 4 == 0, 4 <= d <= 256");
  if (rows == 0) return HDP_OK;
  if (!o_parts || !lse_parts || !o || !lse) return fail(HDP_ERR_INVALID_ARGUMENT, "hdp_lse_merge_rows: NULL argument");
  if ((reinterpret_cast<uintptr_t>(o_parts) & 15) || (reinterpret_cast<uintptr_t>(o) & 7))
    return fail(HDP_ERR_INVALID_ARGUMENT, "hdp_lse_merge_rows: o_parts must be 16-byte and o 8-byte aligned");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  RowSource src{o_parts, lse_parts, m, rows};
  const int g = merge_grid(rows);
  if (d <= 128)
    k_merge_rows<1><<<g, kMergeThreads, 0, st>>>(src, d, static_cast<__nv_bfloat16*>(o), lse);
  else
    k_merge_rows<2><<<g, kMergeThreads, 0, st>>>(src, d, static_cast<__nv_bfloat16*>(o), lse);
  note_launch();
  HDP_CUDA_TRY(cudaGetLastError());
  return HDP_OK;
}
