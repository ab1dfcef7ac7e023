// Sharding plan, best-fit shard packing, query-tile work lists and per-shard
// FLOPs ("ByteScale: Communication-Efficient Scaling of LLM Training with a
// 2048K Context Length on 16384 GPUs", research digest, sections 1, 2, 3.1
// and Figure 2).
//
// Kernels:
//   k_plan_reduce / k_plan_scan_partials / k_plan_scan_write
//       three-phase (reduce, scan of CTA sums, re-scan) warp-shuffle prefix
//       sums of the per-document quantities: tokens, chunks ceil(s/C), causal
//       blocks n(n+1)/2, fused query tiles, split query tiles, sub-capacity
//       pieces.  Integer only, bit-exact.
//   k_fill_chunks / k_fill_blocks / k_fill_tiles_*
//       one thread per table row; the row's document is found by binary
//       search over the scanned offsets, the rest is closed-form.
//   k_radix_*     stable LSD radix sort of 32-bit keys with their indices,
//                 8 bits a pass over the bits the largest key needs (work
//                 lists heaviest first, pieces in best-fit-decreasing order).
//   k_shard_bfd   one CTA: sequential best fit over the sorted pieces with a
//                 block-wide argmin over the open shards.
//   k_flops_*     exact int64 per-shard FLOPs.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdio>
#include <string>

#include "internal.h"

namespace hdp {
namespace {

constexpr int kScanThreads = 256;
constexpr int kScanItems = 8;
constexpr int kScanTile = kScanThreads * kScanItems;  // documents per CTA
constexpr int kQ = 6;  // tokens, chunks, blocks, fused tiles, split tiles, pieces
constexpr int kPartial = 8;  // kQ sums + max length + invalid-length flag

// Per-document quantities (s >= 1).  32-bit unsigned division: every
// intermediate is below 2^31 for s, C < 2^31.
__device__ __forceinline__ void doc_quantities(int32_t s, int32_t C, bool split_ok, long long (&q)[kQ]) {
  const uint32_t su = static_cast<uint32_t>(s), cu = static_cast<uint32_t>(C);
  const uint32_t n = (su - 1u) / cu + 1u;   // ceil(s / C)
  const uint32_t last = su - (n - 1u) * cu;  // length of the last chunk, in [1, C]
  q[0] = s;
  q[1] = n;
  q[2] = static_cast<long long>(n) * (n + 1) / 2;
  q[3] = (su + kTile - 1) / kTile;
  if (split_ok) {
    const long long tpc = cu / kTile;
    const long long tl = (last + kTile - 1) / kTile;
    q[4] = tpc * (static_cast<long long>(n - 1) * n / 2) + tl * n;
  } else {
    q[4] = 0;
  }
  q[5] = last != cu ? 1 : 0;
}

// Exclusive scan of N int64 values over a 256-thread block; also returns the
// block totals.  Warp level: shuffle-up inclusive scan; block level: scan of
// the 8 warp sums by warp 0.
template <int N>
__device__ void block_exclusive_scan(long long (&x)[N], long long (&total)[N]) {
  __shared__ long long wsum[kScanThreads / 32][N];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  long long inc[N];
#pragma unroll
  for (int i = 0; i < N; ++i) inc[i] = x[i];
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
#pragma unroll
    for (int i = 0; i < N; ++i) {
      const long long y = __shfl_up_sync(0xffffffffu, inc[i], off);
      if (lane >= off) inc[i] += y;
    }
  }
  if (lane == 31) {
#pragma unroll
    for (int i = 0; i < N; ++i) wsum[warp][i] = inc[i];
  }
  __syncthreads();
  if (warp == 0) {
    constexpr int W = kScanThreads / 32;
    long long w[N];
#pragma unroll
    for (int i = 0; i < N; ++i) w[i] = lane < W ? wsum[lane][i] : 0;
#pragma unroll
    for (int off = 1; off < W; off <<= 1) {
#pragma unroll
      for (int i = 0; i < N; ++i) {
        const long long y = __shfl_up_sync(0xffffffffu, w[i], off);
        if (lane >= off) w[i] += y;
      }
    }
    if (lane < W) {
#pragma unroll
      for (int i = 0; i < N; ++i) wsum[lane][i] = w[i];
    }
  }
  __syncthreads();
#pragma unroll
  for (int i = 0; i < N; ++i) {
    const long long before = warp > 0 ? wsum[warp - 1][i] : 0;
    total[i] = wsum[kScanThreads / 32 - 1][i];
    x[i] = before + inc[i] - x[i];
  }
  __syncthreads();
}

__global__ void __launch_bounds__(kScanThreads) k_plan_reduce(const int32_t* __restrict__ lengths, int32_t n,
                                                              int32_t C, int split_ok,
                                                              long long* __restrict__ partials) {
  long long acc[kQ] = {0, 0, 0, 0, 0, 0};
  long long mx = 0, bad = 0;
  const long long base = static_cast<long long>(blockIdx.x) * kScanTile;
#pragma unroll
  for (int j = 0; j < kScanItems; ++j) {
    const long long i = base + j * kScanThreads + threadIdx.x;  // coalesced
    if (i < n) {
      const int32_t s = lengths[i];
      if (s < 1) {
        bad = 1;
      } else {
        long long q[kQ];
        doc_quantities(s, C, split_ok != 0, q);
#pragma unroll
        for (int k = 0; k < kQ; ++k) acc[k] += q[k];
        mx = s > mx ? s : mx;
      }
    }
  }
  // block reduction (sum, max, or) via the scan's totals
  long long tot[kQ];
  block_exclusive_scan<kQ>(acc, tot);
  __shared__ long long smx, sbad;
  if (threadIdx.x == 0) smx = 0, sbad = 0;
  __syncthreads();
  if (mx) atomicMax(reinterpret_cast<unsigned long long*>(&smx), static_cast<unsigned long long>(mx));
  if (bad) sbad = 1;
  __syncthreads();
  if (threadIdx.x == 0) {
    long long* p = partials + static_cast<long long>(blockIdx.x) * kPartial;
#pragma unroll
    for (int k = 0; k < kQ; ++k) p[k] = tot[k];
    p[6] = smx;
    p[7] = sbad;
  }
}

// One CTA: exclusive scan of the per-CTA sums (in place: partials[b][0..5]
// become CTA offsets) and the totals: {T, N_c, N_b, fused tiles, split tiles,
// pieces, max length, invalid flag}.  Also writes entry [n] of the offset
// arrays.
__global__ void __launch_bounds__(kScanThreads) k_plan_scan_partials(long long* __restrict__ partials, int nblk,
                                                                     int32_t n, long long* __restrict__ totals,
                                                                     int32_t* cu, int32_t* co, int64_t* bo,
                                                                     int64_t* tof, int64_t* tos, int32_t* po) {
  long long carry[kQ] = {0, 0, 0, 0, 0, 0};
  __shared__ long long smx, sbad;
  if (threadIdx.x == 0) smx = 0, sbad = 0;
  __syncthreads();
  for (int b0 = 0; b0 < nblk; b0 += kScanThreads) {
    const int b = b0 + threadIdx.x;
    long long x[kQ], tot[kQ];
    long long* p = partials + static_cast<long long>(b) * kPartial;
#pragma unroll
    for (int k = 0; k < kQ; ++k) x[k] = b < nblk ? p[k] : 0;
    if (b < nblk) {
      if (p[6]) atomicMax(reinterpret_cast<unsigned long long*>(&smx), static_cast<unsigned long long>(p[6]));
      if (p[7]) sbad = 1;
    }
    block_exclusive_scan<kQ>(x, tot);
    if (b < nblk) {
#pragma unroll
      for (int k = 0; k < kQ; ++k) p[k] = carry[k] + x[k];
    }
#pragma unroll
    for (int k = 0; k < kQ; ++k) carry[k] += tot[k];
  }
  __syncthreads();
  if (threadIdx.x == 0) {
#pragma unroll
    for (int k = 0; k < kQ; ++k) totals[k] = carry[k];
    totals[6] = smx;
    totals[7] = sbad;
    cu[n] = static_cast<int32_t>(carry[0]);
    co[n] = static_cast<int32_t>(carry[1]);
    bo[n] = carry[2];
    tof[n] = carry[3];
    tos[n] = carry[4];
    po[n] = static_cast<int32_t>(carry[5]);
  }
}

__global__ void __launch_bounds__(kScanThreads) k_plan_scan_write(const int32_t* __restrict__ lengths, int32_t n,
                                                                  int32_t C, int split_ok,
                                                                  const long long* __restrict__ partials,
                                                                  int32_t* __restrict__ cu, int32_t* __restrict__ co,
                                                                  int64_t* __restrict__ bo, int64_t* __restrict__ tof,
                                                                  int64_t* __restrict__ tos, int32_t* __restrict__ po) {
  __shared__ int32_t s_len[kScanTile];
  const long long base = static_cast<long long>(blockIdx.x) * kScanTile;
#pragma unroll
  for (int j = 0; j < kScanItems; ++j) {
    const long long i = base + j * kScanThreads + threadIdx.x;
    s_len[j * kScanThreads + threadIdx.x] = i < n ? lengths[i] : 0;
  }
  __syncthreads();
  // thread t owns documents base + t*8 .. base + t*8 + 7
  long long sum[kQ] = {0, 0, 0, 0, 0, 0}, tot[kQ];
#pragma unroll
  for (int j = 0; j < kScanItems; ++j) {
    const int32_t s = s_len[threadIdx.x * kScanItems + j];
    if (s >= 1) {
      long long q[kQ];
      doc_quantities(s, C, split_ok != 0, q);
#pragma unroll
      for (int k = 0; k < kQ; ++k) sum[k] += q[k];
    }
  }
  block_exclusive_scan<kQ>(sum, tot);
  const long long* p = partials + static_cast<long long>(blockIdx.x) * kPartial;
#pragma unroll
  for (int k = 0; k < kQ; ++k) sum[k] += p[k];
  // this thread's 8 consecutive documents: exclusive prefixes in registers,
  // then 16-byte stores
  const long long first = base + threadIdx.x * kScanItems;
  int32_t vcu[kScanItems], vco[kScanItems], vpo[kScanItems];
  long long vbo[kScanItems], vtf[kScanItems], vts[kScanItems];
#pragma unroll
  for (int j = 0; j < kScanItems; ++j) {
    vcu[j] = static_cast<int32_t>(sum[0]);
    vco[j] = static_cast<int32_t>(sum[1]);
    vbo[j] = sum[2];
    vtf[j] = sum[3];
    vts[j] = sum[4];
    vpo[j] = static_cast<int32_t>(sum[5]);
    const int32_t s = s_len[threadIdx.x * kScanItems + j];
    if (first + j < n && s >= 1) {
      long long q[kQ];
      doc_quantities(s, C, split_ok != 0, q);
#pragma unroll
      for (int k = 0; k < kQ; ++k) sum[k] += q[k];
    }
  }
  if (first + kScanItems <= n) {
    int4* c4 = reinterpret_cast<int4*>(cu + first);
    int4* o4 = reinterpret_cast<int4*>(co + first);
    int4* p4 = reinterpret_cast<int4*>(po + first);
    c4[0] = make_int4(vcu[0], vcu[1], vcu[2], vcu[3]);
    c4[1] = make_int4(vcu[4], vcu[5], vcu[6], vcu[7]);
    o4[0] = make_int4(vco[0], vco[1], vco[2], vco[3]);
    o4[1] = make_int4(vco[4], vco[5], vco[6], vco[7]);
    p4[0] = make_int4(vpo[0], vpo[1], vpo[2], vpo[3]);
    p4[1] = make_int4(vpo[4], vpo[5], vpo[6], vpo[7]);
    longlong2* b2 = reinterpret_cast<longlong2*>(bo + first);
    longlong2* f2 = reinterpret_cast<longlong2*>(tof + first);
    longlong2* s2 = reinterpret_cast<longlong2*>(tos + first);
#pragma unroll
    for (int j = 0; j < kScanItems / 2; ++j) {
      b2[j] = make_longlong2(vbo[2 * j], vbo[2 * j + 1]);
      f2[j] = make_longlong2(vtf[2 * j], vtf[2 * j + 1]);
      s2[j] = make_longlong2(vts[2 * j], vts[2 * j + 1]);
    }
  } else {
#pragma unroll
    for (int j = 0; j < kScanItems; ++j) {
      if (first + j < n) {
        cu[first + j] = vcu[j];
        co[first + j] = vco[j];
        po[first + j] = vpo[j];
        bo[first + j] = vbo[j];
        tof[first + j] = vtf[j];
        tos[first + j] = vts[j];
      }
    }
  }
}

// Largest i in [0, n) with off[i] <= x (off ascending, off[0] = 0 <= x).
template <typename T>
__device__ __forceinline__ int32_t upper_doc(const T* __restrict__ off, int32_t n, long long x) {
  int32_t lo = 0, hi = n - 1;
  while (lo < hi) {
    const int32_t mid = (lo + hi + 1) >> 1;
    if (static_cast<long long>(off[mid]) <= x)
      lo = mid;
    else
      hi = mid - 1;
  }
  return lo;
}

// Chunk table, causal pairs per chunk, and the shard of every chunk: full
// chunks take shard ids in chunk order (chunk c of document i is preceded by
// po[i] sub-capacity pieces); a piece takes the shard best fit gave it.
__global__ void k_fill_chunks(int32_t n, int32_t C, long long nc, const int32_t* __restrict__ cu,
                              const int32_t* __restrict__ co, const int32_t* __restrict__ po,
                              const int32_t* __restrict__ piece_shard, int32_t* __restrict__ chunk_table,
                              int64_t* __restrict__ chunk_pairs, int32_t* __restrict__ shard_of_chunk) {
  for (long long c = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; c < nc;
       c += static_cast<long long>(gridDim.x) * blockDim.x) {
    const int32_t doc = upper_doc(co, n, c);
    const long long idx = c - co[doc];
    const long long s = cu[doc + 1] - cu[doc];
    const long long a = idx * C;
    const long long len = s - a < C ? s - a : C;
    const long long b = a + len;
    int4 row;
    row.x = doc;
    row.y = static_cast<int32_t>(idx);
    row.z = static_cast<int32_t>(cu[doc] + a);
    row.w = static_cast<int32_t>(len);
    reinterpret_cast<int4*>(chunk_table)[c] = row;
    chunk_pairs[c] = (b * (b + 1) - a * (a + 1)) / 2;
    if (shard_of_chunk) shard_of_chunk[c] = len == C ? static_cast<int32_t>(c - po[doc]) : piece_shard[doc];
  }
}

// qc = largest q with q(q+1)/2 <= local.
__device__ __forceinline__ long long tri_root(long long local) {
  long long q = static_cast<long long>((sqrt(8.0 * static_cast<double>(local) + 1.0) - 1.0) * 0.5);
  while (q > 0 && q * (q + 1) / 2 > local) --q;
  while ((q + 1) * (q + 2) / 2 <= local) ++q;
  return q;
}

__global__ void k_fill_blocks(int32_t n, long long nb, const int32_t* __restrict__ co,
                              const int64_t* __restrict__ bo, int32_t* __restrict__ block_table) {
  for (long long b = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; b < nb;
       b += static_cast<long long>(gridDim.x) * blockDim.x) {
    const int32_t doc = upper_doc(bo, n, b);
    const long long local = b - bo[doc];
    const long long qc = tri_root(local);
    const long long kc = local - qc * (qc + 1) / 2;
    int2 row;
    row.x = static_cast<int32_t>(co[doc] + qc);
    row.y = static_cast<int32_t>(co[doc] + kc);
    reinterpret_cast<int2*>(block_table)[b] = row;
  }
}

__device__ __forceinline__ void store_tile(int32_t* out, long long t, int32_t q0, int32_t qrows, int32_t kv0,
                                           int32_t kvlen, int32_t blk, int32_t row_off, int32_t w, int32_t doc_len) {
  int4* o = reinterpret_cast<int4*>(out + t * 8);
  o[0] = make_int4(q0, qrows, kv0, kvlen);
  o[1] = make_int4(blk, row_off, w, doc_len);
}

// One row per document query tile: keys are the document's causal prefix.
// Sort key: w_max - weight (w_max >= every weight), so heaviest sorts first.
__global__ void k_fill_tiles_fused(int32_t n, long long ntiles, const int32_t* __restrict__ cu,
                                   const int64_t* __restrict__ tof, int32_t w_max, int32_t* __restrict__ rows,
                                   uint32_t* __restrict__ keys) {
  for (long long t = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; t < ntiles;
       t += static_cast<long long>(gridDim.x) * blockDim.x) {
    const int32_t doc = upper_doc(tof, n, t);
    const long long qt = t - tof[doc];
    const long long s = cu[doc + 1] - cu[doc];
    const long long qrows = s - qt * kTile < kTile ? s - qt * kTile : kTile;
    const long long kvlen = qt * kTile + qrows;
    const long long w = qt + 1;
    store_tile(rows, t, static_cast<int32_t>(cu[doc] + qt * kTile), static_cast<int32_t>(qrows), cu[doc],
               static_cast<int32_t>(kvlen), -1, static_cast<int32_t>(qt * kTile), static_cast<int32_t>(w),
               static_cast<int32_t>(s));
    keys[t] = static_cast<uint32_t>(w_max - w);
  }
}

// One row per query tile of every causal block (qc, kc); rows of a document
// are ordered by block (qc, kc ascending), then query tile.  Needs C % 128 == 0.
// Sort key: C / 128 - weight.
__global__ void k_fill_tiles_split(int32_t n, int32_t C, long long ntiles, const int32_t* __restrict__ cu,
                                   const int64_t* __restrict__ bo, const int64_t* __restrict__ tos,
                                   int32_t* __restrict__ rows, uint32_t* __restrict__ keys) {
  const long long tpc = C / kTile;
  for (long long t = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; t < ntiles;
       t += static_cast<long long>(gridDim.x) * blockDim.x) {
    const int32_t doc = upper_doc(tos, n, t);
    const long long local = t - tos[doc];
    const long long s = cu[doc + 1] - cu[doc];
    const long long nch = (s + C - 1) / C;
    const long long last = s - (nch - 1) * C;
    const long long tl = (last + kTile - 1) / kTile;
    const long long full_rows = tpc * ((nch - 1) * nch / 2);
    long long qc, kc, qt, blk_local;
    if (local < full_rows) {
      blk_local = local / tpc;
      qt = local % tpc;
      qc = tri_root(blk_local);
      kc = blk_local - qc * (qc + 1) / 2;
    } else {
      const long long r = local - full_rows;
      kc = r / tl;
      qt = r % tl;
      qc = nch - 1;
      blk_local = (nch - 1) * nch / 2 + kc;
    }
    const long long qlen = qc == nch - 1 ? last : C;
    const long long qrows = qlen - qt * kTile < kTile ? qlen - qt * kTile : kTile;
    const long long kvlen = kc == qc ? qt * kTile + qrows : C;
    const long long w = (kvlen + kTile - 1) / kTile;
    store_tile(rows, t, static_cast<int32_t>(cu[doc] + qc * C + qt * kTile), static_cast<int32_t>(qrows),
               static_cast<int32_t>(cu[doc] + kc * C), static_cast<int32_t>(kvlen),
               static_cast<int32_t>(bo[doc] + blk_local), static_cast<int32_t>(qt * kTile),
               static_cast<int32_t>(w), 0);
    keys[t] = static_cast<uint32_t>(tpc - w);
  }
}

// ---------------------------------------------------------------- radix sort
// Stable LSD radix sort of (32-bit key, index) pairs by key ascending, 8 bits a
// pass over only the bits the largest key needs.  A pass is three launches:
// block histograms, a scan per digit over the blocks, and a scatter that
// places each block's items in index order (so equal keys keep their order).
// The work lists sort by (largest weight - weight), the best-fit pieces by
// (C - piece length): heaviest / longest first, then index ascending.
constexpr int kRadixThreads = 256;  // also the number of digit values
constexpr int kRadixItems = 8;      // items per thread per block
constexpr int kRadixTile = kRadixThreads * kRadixItems;
constexpr int kRadixWarps = kRadixThreads / 32;

// counts[d * nb + b] = items of block b whose digit is d.
__global__ void __launch_bounds__(kRadixThreads) k_radix_hist(const uint32_t* __restrict__ keys, long long n,
                                                              int shift, uint32_t* __restrict__ counts, int nb) {
  __shared__ uint32_t h[kRadixThreads];
  h[threadIdx.x] = 0;
  __syncthreads();
  const long long base = static_cast<long long>(blockIdx.x) * kRadixTile;
#pragma unroll
  for (int j = 0; j < kRadixItems; ++j) {
    const long long i = base + j * kRadixThreads + threadIdx.x;
    if (i < n) atomicAdd(&h[(keys[i] >> shift) & 255u], 1u);
  }
  __syncthreads();
  counts[static_cast<long long>(threadIdx.x) * nb + blockIdx.x] = h[threadIdx.x];
}

// One CTA per digit: exclusive scan of its row of counts over the blocks, in
// place; totals[d] = the digit's count.
constexpr int kDigitScanThreads = 1024;
__global__ void __launch_bounds__(kDigitScanThreads) k_radix_digit_scan(uint32_t* __restrict__ counts, int nb,
                                                                        uint32_t* __restrict__ totals) {
  __shared__ uint32_t wsum[kDigitScanThreads / 32];
  __shared__ uint32_t carry;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t* row = counts + static_cast<long long>(blockIdx.x) * nb;
  if (threadIdx.x == 0) carry = 0;
  __syncthreads();
  for (int b0 = 0; b0 < nb; b0 += kDigitScanThreads) {
    const int i = b0 + threadIdx.x;
    const uint32_t x = i < nb ? row[i] : 0u;
    uint32_t v = x;  // inclusive scan inside the warp
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(0xffffffffu, v, o);
      if (lane >= o) v += y;
    }
    if (lane == 31) wsum[warp] = v;
    __syncthreads();
    if (warp == 0) {
      uint32_t w = wsum[lane];
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(0xffffffffu, w, o);
        if (lane >= o) w += y;
      }
      wsum[lane] = w;
    }
    __syncthreads();
    const uint32_t before = carry + (warp > 0 ? wsum[warp - 1] : 0u);
    if (i < nb) row[i] = before + v - x;
    __syncthreads();  // every thread has read carry
    if (threadIdx.x == kDigitScanThreads - 1) carry = before + v;
    __syncthreads();
  }
  if (threadIdx.x == 0) totals[blockIdx.x] = carry;
}

// Places every item of block b at digit_base[d] + counts[d][b] + (its rank
// among the block's items with digit d, in index order).  vals_in == nullptr:
// the value is the item's index (first pass).
__global__ void __launch_bounds__(kRadixThreads) k_radix_scatter(const uint32_t* __restrict__ keys_in,
                                                                 const uint32_t* __restrict__ vals_in,
                                                                 uint32_t* __restrict__ keys_out,
                                                                 uint32_t* __restrict__ vals_out, long long n,
                                                                 int shift, const uint32_t* __restrict__ counts,
                                                                 int nb, const uint32_t* __restrict__ totals) {
  __shared__ uint32_t wcnt[kRadixWarps][kRadixThreads];  // per round: digit counts per warp, then offsets
  __shared__ uint32_t base_d[kRadixThreads];             // where this block's items of digit d start
  __shared__ uint32_t wsum[kRadixWarps];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int d = threadIdx.x;  // one digit per thread for the per-digit steps
  {
    // exclusive scan of the digit totals -> start of each digit's output range
    const uint32_t x = totals[d];
    uint32_t v = x;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(0xffffffffu, v, o);
      if (lane >= o) v += y;
    }
    if (lane == 31) wsum[warp] = v;
    __syncthreads();
    uint32_t before = 0;
    for (int w = 0; w < warp; ++w) before += wsum[w];
    base_d[d] = before + v - x + counts[static_cast<long long>(d) * nb + blockIdx.x];
  }
  const long long base = static_cast<long long>(blockIdx.x) * kRadixTile;
  for (int j = 0; j < kRadixItems; ++j) {
#pragma unroll
    for (int e = lane; e < kRadixThreads; e += 32) wcnt[warp][e] = 0;
    __syncthreads();  // (first j: also orders base_d)
    const long long i = base + j * kRadixThreads + threadIdx.x;
    const bool valid = i < n;
    const uint32_t key = valid ? keys_in[i] : 0u;
    const uint32_t dig = valid ? (key >> shift) & 255u : 256u;  // 256: not an item
    const uint32_t peers = __match_any_sync(0xffffffffu, dig);
    const uint32_t rank = __popc(peers & ((1u << lane) - 1u));
    if (valid && rank == 0) wcnt[warp][dig] = __popc(peers);
    __syncthreads();
    {
      // per digit: items of earlier warps of this round, after earlier rounds
      uint32_t off = base_d[d];
#pragma unroll
      for (int w = 0; w < kRadixWarps; ++w) {
        const uint32_t c = wcnt[w][d];
        wcnt[w][d] = off;
        off += c;
      }
      base_d[d] = off;
    }
    __syncthreads();
    if (valid) {
      const uint32_t pos = wcnt[warp][dig] + rank;
      keys_out[pos] = key;
      vals_out[pos] = vals_in ? vals_in[i] : static_cast<uint32_t>(i);
    }
    __syncthreads();  // before the next round clears wcnt
  }
}

// Small inputs (n <= kSmallSort) in one launch: one CTA sorts (key, index)
// pairs packed as key << 32 | index with a bitonic network in shared memory
// (the index makes the order that of a stable sort by key).
constexpr int kSmallSort = 4096;
constexpr int kSmallSortThreads = 1024;
__global__ void __launch_bounds__(kSmallSortThreads) k_sort_small(const uint32_t* __restrict__ keys, int n,
                                                                  uint32_t* __restrict__ keys_out,
                                                                  uint32_t* __restrict__ perm_out) {
  __shared__ unsigned long long s[kSmallSort];
  int n2 = 1;
  while (n2 < n) n2 <<= 1;
  for (int i = threadIdx.x; i < n2; i += kSmallSortThreads)
    s[i] = i < n ? (static_cast<unsigned long long>(keys[i]) << 32) | static_cast<unsigned>(i) : ~0ull;
  __syncthreads();
  for (int k = 2; k <= n2; k <<= 1) {
    for (int j = k >> 1; j > 0; j >>= 1) {
      for (int i = threadIdx.x; i < n2 / 2; i += kSmallSortThreads) {
        const int lo = (i / j) * 2 * j + (i % j);
        const int hi = lo + j;
        const bool asc = (lo & k) == 0;
        const unsigned long long a = s[lo], b = s[hi];
        if ((a > b) == asc) {
          s[lo] = b;
          s[hi] = a;
        }
      }
      __syncthreads();
    }
  }
  for (int i = threadIdx.x; i < n; i += kSmallSortThreads) {
    keys_out[i] = static_cast<uint32_t>(s[i] >> 32);
    perm_out[i] = static_cast<uint32_t>(s[i] & 0xffffffffu);
  }
}

// out row i = rows[perm[i]] (perm == nullptr: the identity).
__global__ void k_gather_rows(const uint32_t* __restrict__ perm, long long count, const int32_t* __restrict__ rows,
                              int32_t* __restrict__ out) {
  for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < count;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const long long src = perm ? static_cast<long long>(perm[i]) : i;
    const int4* a = reinterpret_cast<const int4*>(rows + src * 8);
    int4* b = reinterpret_cast<int4*>(out + i * 8);
    b[0] = a[0];
    b[1] = a[1];
  }
}

// ---------------------------------------------------------------- best fit
// Sort key of document i: C - (length of its sub-capacity piece: a short
// document or a tail chunk), so ascending order is length descending (then
// document ascending, the sort being stable); documents without a piece (s a
// multiple of C, or an invalid length) get C and sort after every piece.
__global__ void k_piece_keys(int32_t n, int32_t C, const int32_t* __restrict__ lengths,
                             uint32_t* __restrict__ keys) {
  for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const int32_t s = lengths[i];
    const int32_t last = s >= 1 ? s % C : 0;
    keys[i] = static_cast<uint32_t>(last != 0 ? C - last : C);
  }
}

constexpr int kBfdThreads = 1024;

// Best fit over the pieces in sorted order: each goes to the open piece shard
// with the least remaining capacity that still fits (lowest id on ties), else
// opens a new shard.  Piece shards are numbered after the full-chunk shards.
// The piece and chunk counts come from the scan's totals on the device, so
// the plan's one host read-back carries the shard count too: totals[kPartial]
// becomes the number of shards, or -1 when there are more than kMaxPieces
// pieces (nothing else is written then).  piece_shard[doc] receives the shard
// of the document's piece.
__global__ void __launch_bounds__(kBfdThreads) k_shard_bfd(const uint32_t* __restrict__ keys,
                                                           const uint32_t* __restrict__ docs, int32_t C,
                                                           long long* __restrict__ totals,
                                                           int32_t* __restrict__ remaining,
                                                           int32_t* __restrict__ piece_shard) {
  const long long npc_total = totals[5];
  const int32_t nfull = static_cast<int32_t>(totals[1] - npc_total);
  if (npc_total > kMaxPieces || totals[7]) {
    if (threadIdx.x == 0) totals[kPartial] = -1;
    return;
  }
  const int32_t npieces = static_cast<int32_t>(npc_total);
  __shared__ unsigned long long wbest[kBfdThreads / 32];
  __shared__ int32_t s_open;
  if (threadIdx.x == 0) s_open = 0;
  __syncthreads();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int32_t p = 0; p < npieces; ++p) {
    const int32_t len = C - static_cast<int32_t>(keys[p]);
    const int32_t doc = docs ? static_cast<int32_t>(docs[p]) : p;
    const int32_t open = s_open;
    unsigned long long best = ~0ull;
    for (int32_t s = threadIdx.x; s < open; s += kBfdThreads) {
      const int32_t r = remaining[s];
      if (r >= len) {
        const unsigned long long cand = (static_cast<unsigned long long>(r) << 32) | static_cast<unsigned>(s);
        best = cand < best ? cand : best;
      }
    }
    if (open > 32) {
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) {
        const unsigned long long y = __shfl_xor_sync(0xffffffffu, best, off);
        best = y < best ? y : best;
      }
      if (lane == 0) wbest[warp] = best;
      __syncthreads();
      if (warp == 0) {
        best = wbest[lane];
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
          const unsigned long long y = __shfl_xor_sync(0xffffffffu, best, off);
          best = y < best ? y : best;
        }
      }
    } else if (warp == 0) {
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) {
        const unsigned long long y = __shfl_xor_sync(0xffffffffu, best, off);
        best = y < best ? y : best;
      }
    }
    if (threadIdx.x == 0) {
      int32_t sid;
      if (best == ~0ull) {
        sid = s_open;
        remaining[sid] = C - len;
        s_open = sid + 1;
      } else {
        sid = static_cast<int32_t>(best & 0xffffffffu);
        remaining[sid] -= len;
      }
      piece_shard[doc] = nfull + sid;
    }
    __syncthreads();
  }
  if (threadIdx.x == 0) totals[kPartial] = nfull + s_open;
}

// ---------------------------------------------------------------- FLOPs
__global__ void k_flops_zero(int64_t* out, int32_t ns) {
  for (int32_t i = blockIdx.x * blockDim.x + threadIdx.x; i < ns; i += gridDim.x * blockDim.x) out[i] = 0;
}
__global__ void k_flops_accum(const int64_t* __restrict__ pairs, const int32_t* __restrict__ shard, long long nc,
                              long long per_pair, int64_t* out) {
  for (long long c = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; c < nc;
       c += static_cast<long long>(gridDim.x) * blockDim.x) {
    atomicAdd(reinterpret_cast<unsigned long long*>(out + shard[c]),
              static_cast<unsigned long long>(pairs[c] * per_pair));
  }
}

// ---------------------------------------------------------------- host helpers
int grid_for(long long items, int threads, int cap = 1 << 16) {
  long long g = (items + threads - 1) / threads;
  if (g < 1) g = 1;
  if (g > cap) g = cap;
  return static_cast<int>(g);
}

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

int bit_length(uint32_t x) {
  int b = 0;
  while (x) {
    ++b;
    x >>= 1;
  }
  return b;
}

// Scratch of radix_sort for n items: two key and two value buffers of n
// entries, the per-(digit, block) counts and the 256 digit totals.
struct RadixScratch {
  uint32_t *k0, *v0, *k1, *v1, *counts, *totals;
};
size_t radix_scratch_bytes(long long n) {
  const long long nb = (n + kRadixTile - 1) / kRadixTile;
  return 4 * align256(sizeof(uint32_t) * (n > 0 ? n : 1)) + align256(sizeof(uint32_t) * 256 * (nb > 0 ? nb : 1)) +
         align256(sizeof(uint32_t) * 256);
}
RadixScratch radix_scratch(char* mem, long long n) {
  const long long nb = (n + kRadixTile - 1) / kRadixTile;
  const size_t a = align256(sizeof(uint32_t) * (n > 0 ? n : 1));
  RadixScratch r;
  r.k0 = reinterpret_cast<uint32_t*>(mem);
  r.v0 = reinterpret_cast<uint32_t*>(mem + a);
  r.k1 = reinterpret_cast<uint32_t*>(mem + 2 * a);
  r.v1 = reinterpret_cast<uint32_t*>(mem + 3 * a);
  r.counts = reinterpret_cast<uint32_t*>(mem + 4 * a);
  r.totals = reinterpret_cast<uint32_t*>(mem + 4 * a + align256(sizeof(uint32_t) * 256 * (nb > 0 ? nb : 1)));
  return r;
}

// Stable sort of the n keys in sc.k0 (every key <= max_key) with their
// indices: one launch when n <= kSmallSort, else the radix passes.  *keys / *perm receive the sorted keys and the source index of
// each position (perm == nullptr when no pass was needed: the identity,
// keys == sc.k0).
cudaError_t radix_sort(RadixScratch sc, long long n, uint32_t max_key, cudaStream_t st, const uint32_t** keys,
                       const uint32_t** perm) {
  const int passes = (bit_length(max_key) + 7) / 8;
  if (passes > 0 && n > 1 && n <= kSmallSort) {
    k_sort_small<<<1, kSmallSortThreads, 0, st>>>(sc.k0, static_cast<int>(n), sc.k1, sc.v1);
    note_launch();
    *keys = sc.k1;
    *perm = sc.v1;
    return cudaGetLastError();
  }
  const int nb = static_cast<int>((n + kRadixTile - 1) / kRadixTile);
  uint32_t *kin = sc.k0, *vin = nullptr, *kout = sc.k1, *vout = sc.v1;
  for (int p = 0; p < passes && n > 0; ++p) {
    const int shift = 8 * p;
    k_radix_hist<<<nb, kRadixThreads, 0, st>>>(kin, n, shift, sc.counts, nb);
    note_launch();
    k_radix_digit_scan<<<256, kDigitScanThreads, 0, st>>>(sc.counts, nb, sc.totals);
    note_launch();
    k_radix_scatter<<<nb, kRadixThreads, 0, st>>>(kin, vin, kout, vout, n, shift, sc.counts, nb, sc.totals);
    note_launch();
    // this pass's output is the next pass's input; its input buffers are free
    uint32_t* const free_k = kin;
    uint32_t* const free_v = vin ? vin : sc.v0;
    kin = kout;
    vin = vout;
    kout = free_k;
    vout = free_v;
  }
  *keys = kin;
  *perm = vin;
  return cudaGetLastError();
}


}  // namespace
}  // namespace hdp

using namespace hdp;

extern "C" hdp_status_t hdp_plan_create_ex(const int32_t* d_lengths, int32_t num_docs, int32_t capacity,
                                           uint32_t flags, void* stream, hdp_plan_t* out) {
  if (!out) return fail(HDP_ERR_INVALID_ARGUMENT, "hdp_plan_create: out is NULL");
  *out = nullptr;
  if (!d_lengths) return fail(HDP_ERR_INVALID_ARGUMENT, "hdp_plan_create: d_lengths is NULL");
  if (num_docs < 1) return fail(HDP_ERR_INVALID_ARGUMENT, "hdp_plan_create: num_docs must be >= 1");
  if (capacity < 1) return fail(HDP_ERR_INVALID_ARGUMENT, "hdp_plan_create: capacity must be >= 1");
  if (flags & ~(HDP_PLAN_NO_SHARDS | HDP_PLAN_NO_SPLIT))
    return fail(HDP_ERR_INVALID_ARGUMENT, "hdp_plan_create: unknown flags");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const bool split_ok = capacity % kTile == 0;
  const bool split_list = split_ok && !(flags & HDP_PLAN_NO_SPLIT);  // build the SPLIT work list
  const int32_t n = num_docs;
  const int nblk = static_cast<int>((static_cast<long long>(n) + kScanTile - 1) / kScanTile);

  // ---- phase 1: per-document offsets and best-fit shards (sizes known from n)
  // Every sub-capacity piece belongs to one document, so the pieces' sort keys,
  // the best-fit state and the per-document piece shards are sized by n and
  // run before the one host read-back, which then carries the shard count.
  const bool shards = !(flags & HDP_PLAN_NO_SHARDS);
  size_t off = 0;
  const size_t o_cu = off; off = align256(off + sizeof(int32_t) * (n + 1));
  const size_t o_co = off; off = align256(off + sizeof(int32_t) * (n + 1));
  const size_t o_bo = off; off = align256(off + sizeof(int64_t) * (n + 1));
  const size_t o_tof = off; off = align256(off + sizeof(int64_t) * (n + 1));
  const size_t o_tos = off; off = align256(off + sizeof(int64_t) * (n + 1));
  const size_t bytes1 = off;
  const size_t o_po = 0;  // scratch: piece offsets, CTA partials, totals, best-fit state
  size_t soff = align256(sizeof(int32_t) * (n + 1));
  const size_t o_part = soff; soff = align256(soff + sizeof(long long) * kPartial * nblk);
  const size_t o_tot = soff; soff = align256(soff + sizeof(long long) * (kPartial + 1));
  const size_t o_pkey = soff; soff = align256(soff + (shards ? radix_scratch_bytes(n) : 0));
  const size_t o_rem = soff; soff = align256(soff + (shards ? sizeof(int32_t) * std::min<long long>(n, kMaxPieces) : 0));
  const size_t o_psh = soff; soff = align256(soff + (shards ? sizeof(int32_t) * n : 0));
  const size_t sbytes = soff;

  int device = 0;
  HDP_CUDA_TRY(cudaGetDevice(&device));
  auto* plan = new (std::nothrow) hdp_plan_s;
  if (!plan) return fail(HDP_ERR_OUT_OF_MEMORY, "hdp_plan_create: host allocation failed");
  plan->device = device;
  plan->stream = st;
  plan->flags = flags;
  char* scratch = nullptr;
  char* mem1 = nullptr;
  auto cleanup = [&](hdp_status_t s) {
    if (scratch) cudaFreeAsync(scratch, st);
    if (mem1) cudaFreeAsync(mem1, st);
    if (plan->mem) cudaFreeAsync(plan->mem, st);
    delete plan;
    return s;
  };
  cudaError_t e = cudaMallocAsync(reinterpret_cast<void**>(&mem1), bytes1, st);
  if (e != cudaSuccess) return cleanup(fail_cuda(e, "cudaMallocAsync(plan offsets)"));
  e = cudaMallocAsync(reinterpret_cast<void**>(&scratch), sbytes, st);
  if (e != cudaSuccess) return cleanup(fail_cuda(e, "cudaMallocAsync(plan scratch)"));
  int32_t* cu = reinterpret_cast<int32_t*>(mem1 + o_cu);
  int32_t* co = reinterpret_cast<int32_t*>(mem1 + o_co);
  int64_t* bo = reinterpret_cast<int64_t*>(mem1 + o_bo);
  int64_t* tof = reinterpret_cast<int64_t*>(mem1 + o_tof);
  int64_t* tos = reinterpret_cast<int64_t*>(mem1 + o_tos);
  int32_t* po = reinterpret_cast<int32_t*>(scratch + o_po);
  long long* partials = reinterpret_cast<long long*>(scratch + o_part);
  long long* totals = reinterpret_cast<long long*>(scratch + o_tot);
  auto* rem = reinterpret_cast<int32_t*>(scratch + o_rem);
  auto* piece_shard = reinterpret_cast<int32_t*>(scratch + o_psh);

  k_plan_reduce<<<nblk, kScanThreads, 0, st>>>(d_lengths, n, capacity, split_ok, partials);
  note_launch();
  k_plan_scan_partials<<<1, kScanThreads, 0, st>>>(partials, nblk, n, totals, cu, co, bo, tof, tos, po);
  note_launch();
  k_plan_scan_write<<<nblk, kScanThreads, 0, st>>>(d_lengths, n, capacity, split_ok, partials, cu, co, bo, tof,
                                                   tos, po);
  note_launch();
  if (shards) {
    const RadixScratch ps = radix_scratch(scratch + o_pkey, n);
    k_piece_keys<<<grid_for(n, 256), 256, 0, st>>>(n, capacity, d_lengths, ps.k0);
    note_launch();
    const uint32_t *sorted_keys = nullptr, *sorted_docs = nullptr;
    e = radix_sort(ps, n, static_cast<uint32_t>(capacity), st, &sorted_keys, &sorted_docs);
    if (e != cudaSuccess) return cleanup(fail_cuda(e, "piece sort"));
    k_shard_bfd<<<1, kBfdThreads, 0, st>>>(sorted_keys, sorted_docs, capacity, totals, rem, piece_shard);
    note_launch();
  }
  e = cudaGetLastError();
  if (e != cudaSuccess) return cleanup(fail_cuda(e, "plan scan launch"));
  long long h_tot[kPartial + 1];
  e = cudaMemcpyAsync(h_tot, totals, sizeof h_tot, cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) {
    note_host_sync();
    e = cudaStreamSynchronize(st);
  }
  if (e != cudaSuccess) return cleanup(fail_cuda(e, "plan totals readback"));

  const long long T = h_tot[0], nc = h_tot[1], nb = h_tot[2], ntf = h_tot[3], nts = h_tot[4];
  if (h_tot[7]) return cleanup(fail(HDP_ERR_INVALID_ARGUMENT, "hdp_plan_create: every length must be >= 1"));
  if (T >= (1ll << 31))
    return cleanup(fail(HDP_ERR_INVALID_ARGUMENT, "hdp_plan_create: total tokens must be < 2^31"));
  if (nb >= (1ll << 31) || nts >= (1ll << 31))
    return cleanup(fail(HDP_ERR_UNSUPPORTED, "hdp_plan_create: more than 2^31 causal blocks or split tiles"));
  if (shards && h_tot[kPartial] < 0)
    return cleanup(fail(HDP_ERR_UNSUPPORTED,
                        "hdp_plan_create: more than 65536 sub-capacity pieces for best-fit packing "
                        "(use HDP_PLAN_NO_SHARDS)"));
  const int32_t h_ns = shards ? static_cast<int32_t>(h_tot[kPartial]) : 0;

  // ---- phase 2: tables sized by the totals
  off = 0;
  const size_t o_ct = off; off = align256(off + sizeof(int32_t) * 4 * nc);
  const size_t o_bt = off; off = align256(off + sizeof(int32_t) * 2 * nb);
  const size_t o_cp = off; off = align256(off + sizeof(int64_t) * nc);
  const size_t o_sc = off; off = align256(off + (shards ? sizeof(int32_t) * nc : 0));
  const size_t o_tf = off; off = align256(off + sizeof(int32_t) * 8 * ntf);
  const size_t o_ts = off; off = align256(off + (split_list ? sizeof(int32_t) * 8 * nts : 0));
  const size_t bytes2 = off;
  e = cudaMallocAsync(&plan->mem, bytes2, st);
  if (e != cudaSuccess) return cleanup(fail_cuda(e, "cudaMallocAsync(plan tables)"));
  char* m2 = static_cast<char*>(plan->mem);
  int32_t* chunk_table = reinterpret_cast<int32_t*>(m2 + o_ct);
  int32_t* block_table = reinterpret_cast<int32_t*>(m2 + o_bt);
  int64_t* chunk_pairs = reinterpret_cast<int64_t*>(m2 + o_cp);
  int32_t* shard_of_chunk = shards ? reinterpret_cast<int32_t*>(m2 + o_sc) : nullptr;
  int32_t* tiles_f = reinterpret_cast<int32_t*>(m2 + o_tf);
  int32_t* tiles_s = split_list ? reinterpret_cast<int32_t*>(m2 + o_ts) : nullptr;

  // sort scratch: radix-sort buffers + unsorted rows
  const long long nrows = std::max({ntf, split_list ? nts : 0ll, 1ll});
  char* sort_mem = nullptr;
  size_t so = radix_scratch_bytes(nrows);
  const size_t o_rows = so; so = align256(so + sizeof(int32_t) * 8 * nrows);
  e = cudaMallocAsync(reinterpret_cast<void**>(&sort_mem), so, st);
  if (e != cudaSuccess) return cleanup(fail_cuda(e, "cudaMallocAsync(plan sort scratch)"));
  const RadixScratch rs = radix_scratch(sort_mem, nrows);
  auto* rows = reinterpret_cast<int32_t*>(sort_mem + o_rows);
  const uint32_t *sorted_keys = nullptr, *perm = nullptr;
  auto cleanup2 = [&](hdp_status_t s) {
    cudaFreeAsync(sort_mem, st);
    return cleanup(s);
  };

  if (nc > 0) {
    k_fill_chunks<<<grid_for(nc, 256), 256, 0, st>>>(n, capacity, nc, cu, co, po, piece_shard, chunk_table,
                                                     chunk_pairs, shard_of_chunk);
    note_launch();
  }
  if (nb > 0) {
    k_fill_blocks<<<grid_for(nb, 256), 256, 0, st>>>(n, nb, co, bo, block_table);
    note_launch();
  }
  // fused work list
  // heaviest first: weights are 1 .. ceil(longest document / 128)
  const int32_t w_max = static_cast<int32_t>((h_tot[6] + kTile - 1) / kTile);
  k_fill_tiles_fused<<<grid_for(ntf, 256), 256, 0, st>>>(n, ntf, cu, tof, w_max, rows, rs.k0);
  note_launch();
  e = radix_sort(rs, ntf, static_cast<uint32_t>(w_max - 1), st, &sorted_keys, &perm);
  if (e != cudaSuccess) return cleanup2(fail_cuda(e, "work list sort"));
  k_gather_rows<<<grid_for(ntf, 256), 256, 0, st>>>(perm, ntf, rows, tiles_f);
  note_launch();
  // split work list
  if (split_list && nts > 0) {
    // weights are 1 .. C / 128
    k_fill_tiles_split<<<grid_for(nts, 256), 256, 0, st>>>(n, capacity, nts, cu, bo, tos, rows, rs.k0);
    note_launch();
    e = radix_sort(rs, nts, static_cast<uint32_t>(capacity / kTile - 1), st, &sorted_keys, &perm);
    if (e != cudaSuccess) return cleanup2(fail_cuda(e, "split work list sort"));
    k_gather_rows<<<grid_for(nts, 256), 256, 0, st>>>(perm, nts, rows, tiles_s);
    note_launch();
  }
  e = cudaGetLastError();
  if (e != cudaSuccess) return cleanup2(fail_cuda(e, "plan table launch"));
  cudaFreeAsync(sort_mem, st);
  cudaFreeAsync(scratch, st);

  // keep the phase-1 offsets: move them into the plan by keeping mem1 alive
  plan->v.num_docs = n;
  plan->v.capacity = capacity;
  plan->v.num_chunks = static_cast<int32_t>(nc);
  plan->v.num_shards = h_ns;
  plan->v.num_blocks = nb;
  plan->v.total_tokens = T;
  plan->v.max_doc_len = static_cast<int32_t>(h_tot[6]);
  plan->v.tile = kTile;
  plan->v.cu_seqlens = cu;
  plan->v.chunk_offsets = co;
  plan->v.block_offsets = bo;
  plan->v.chunk_table = chunk_table;
  plan->v.block_table = block_table;
  plan->v.chunk_pairs = chunk_pairs;
  plan->v.shard_of_chunk = shard_of_chunk;
  plan->v.tiles_fused = tiles_f;
  plan->v.num_tiles_fused = ntf;
  plan->v.tiles_split = tiles_s;
  plan->v.num_tiles_split = split_list ? nts : 0;
  plan->tile_offsets_fused = tof;
  plan->tile_offsets_split = tos;
  plan->mem1 = mem1;
  *out = plan;
  return HDP_OK;
}

extern "C" hdp_status_t hdp_plan_create(const int32_t* d_lengths, int32_t num_docs, int32_t capacity, void* stream,
                                        hdp_plan_t* out) {
  return hdp_plan_create_ex(d_lengths, num_docs, capacity, HDP_PLAN_DEFAULT, stream, out);
}

extern "C" hdp_status_t hdp_plan_view(hdp_plan_t plan, hdp_plan_view_t* view) {
  if (!plan || !view) return fail(HDP_ERR_INVALID_ARGUMENT, "hdp_plan_view: NULL argument");
  *view = plan->v;
  return HDP_OK;
}

extern "C" hdp_status_t hdp_plan_destroy(hdp_plan_t plan) {
  if (!plan) return HDP_OK;
  int cur = 0;
  cudaGetDevice(&cur);
  if (cur != plan->device) cudaSetDevice(plan->device);
  cudaError_t e1 = plan->mem ? cudaFreeAsync(plan->mem, plan->stream) : cudaSuccess;
  cudaError_t e2 = plan->mem1 ? cudaFreeAsync(plan->mem1, plan->stream) : cudaSuccess;
  if (cur != plan->device) cudaSetDevice(cur);
  delete plan;
  if (e1 != cudaSuccess) return fail_cuda(e1, "hdp_plan_destroy");
  if (e2 != cudaSuccess) return fail_cuda(e2, "hdp_plan_destroy");
  return HDP_OK;
}

extern "C" hdp_status_t hdp_flops_per_shard(hdp_plan_t plan, int32_t d, int32_t hq, int64_t* d_out, void* stream) {
  if (!plan || !d_out) return fail(HDP_ERR_INVALID_ARGUMENT, "hdp_flops_per_shard: NULL argument");
  if (d < 1 || hq < 1) return fail(HDP_ERR_INVALID_ARGUMENT, "hdp_flops_per_shard: d and hq must be >= 1");
  if (!plan->v.shard_of_chunk)
    return fail(HDP_ERR_INVALID_ARGUMENT, "hdp_flops_per_shard: plan was created without shards");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int32_t ns = plan->v.num_shards;
  k_flops_zero<<<grid_for(ns, 256), 256, 0, st>>>(d_out, ns);
  note_launch();
  k_flops_accum<<<grid_for(plan->v.num_chunks, 256), 256, 0, st>>>(
      plan->v.chunk_pairs, plan->v.shard_of_chunk, plan->v.num_chunks, 4ll * d * hq, d_out);
  note_launch();
  HDP_CUDA_TRY(cudaGetLastError());
  return HDP_OK;
}
