// Exact log-sum-exp merge of partial attention results ("ByteScale:
// Communication-Efficient Scaling of LLM Training with a 2048K Context Length
// on 16384 GPUs", research digest, section 3.2: the partial block of each ring
// step is combined with the others).  For one (row, head):
//   M = max_k lse_k,  lse = M + ln sum_k exp(lse_k - M),
//   o = sum_k exp(lse_k - lse) o_k.
// HBM-bound: one warp per (row, head), each lane streams float4 columns of
// every partial (coalesced 512-byte rows at d = 128); bf16 output.
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

// Merge m partials of one row.  lse_at(k) gives lse_k; o_at(k) gives a pointer
// to o_k's d floats.  Writes d bf16 to `out` and returns lse.
template <int VEC, typename LseAt, typename OAt>
__device__ __forceinline__ float merge_row(int m, int d, int lane, LseAt lse_at, OAt o_at, __nv_bfloat16* out) {
  float M = -INFINITY;
  for (int k = lane; k < m; k += 32) M = fmaxf(M, lse_at(k));
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
  float4 acc[VEC];
#pragma unroll
  for (int v = 0; v < VEC; ++v) acc[v] = make_float4(0.f, 0.f, 0.f, 0.f);
  float L = -INFINITY;
  if (M != -INFINITY) {
    float sum = 0.f;
    for (int k = lane; k < m; k += 32) sum += expf(lse_at(k) - M);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
    L = M + logf(sum);
    // four partials per step: their loads are independent, so up to four
    // 512-byte rows per warp are in flight
    for (int k0 = 0; k0 < m; k0 += 4) {
      float w[4];
      float4 x[4][VEC];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int k = k0 + u;
        w[u] = k < m ? expf(lse_at(k) - L) : 0.f;
        const float* ok = o_at(k < m ? k : k0);
#pragma unroll
        for (int v = 0; v < VEC; ++v) {
          const int c = (v * 32 + lane) * 4;
          x[u][v] = (c < d && w[u] != 0.f) ? __ldg(reinterpret_cast<const float4*>(ok + c))
                                            : make_float4(0.f, 0.f, 0.f, 0.f);
        }
      }
#pragma unroll
      for (int u = 0; u < 4; ++u)
#pragma unroll
        for (int v = 0; v < VEC; ++v) {
          acc[v].x = fmaf(w[u], x[u][v].x, acc[v].x);
          acc[v].y = fmaf(w[u], x[u][v].y, acc[v].y);
          acc[v].z = fmaf(w[u], x[u][v].z, acc[v].z);
          acc[v].w = fmaf(w[u], x[u][v].w, acc[v].w);
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

// Work item w = h * T + t (consecutive warps: consecutive tokens of one head).
template <int VEC>
__global__ void __launch_bounds__(kMergeThreads) k_merge_blocks(BlockSource src, int d, __nv_bfloat16* __restrict__ o,
                                                                float* __restrict__ lse) {
  const int lane = threadIdx.x & 31;
  const long long nwork = src.T * src.hq;
  for (long long w = (static_cast<long long>(blockIdx.x) * kMergeThreads + threadIdx.x) >> 5; w < nwork;
       w += (static_cast<long long>(gridDim.x) * kMergeThreads) >> 5) {
    const int32_t h = static_cast<int32_t>(w / src.T);
    const long long t = w - static_cast<long long>(h) * src.T;
    const int32_t doc = doc_of(src.cu, src.n, t);
    const long long p = t - src.cu[doc];
    const long long qc = p / src.C;
    const long long row = p - qc * src.C;
    const long long b0 = src.bo[doc] + qc * (qc + 1) / 2;  // block (qc, 0)
    const int m = static_cast<int>(qc + 1);
    auto lse_at = [&](int k) {
      return __ldg(src.lse_part + ((b0 + k) * src.hq + h) * static_cast<long long>(src.C) + row);
    };
    auto o_at = [&](int k) { return src.o_part + (((b0 + k) * src.C + row) * src.hq + h) * static_cast<long long>(d); };
    const float L = merge_row<VEC>(m, d, lane, lse_at, o_at, o + (t * src.hq + h) * static_cast<long long>(d));
    if (lane == 0) lse[static_cast<long long>(h) * src.T + t] = L;
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
  const int g = merge_grid(plan->v.total_tokens * hq);
  if (d <= 128)
    k_merge_blocks<1><<<g, kMergeThreads, 0, st>>>(src, d, static_cast<__nv_bfloat16*>(o), lse);
  else
    k_merge_blocks<2><<<g, kMergeThreads, 0, st>>>(src, d, static_cast<__nv_bfloat16*>(o), lse);
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
