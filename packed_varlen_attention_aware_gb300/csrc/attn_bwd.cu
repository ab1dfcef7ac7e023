// Backward pass of document-masked causal attention on tcgen05 tensor cores.
// The training step timed in "ByteScale: Communication-Efficient Scaling of
// LLM Training with a 2048K Context Length on 16384 GPUs" (research digest,
// section 5: forward and backward bars) runs this after the forward of the
// same packed micro-batch; a query attends only to its own sequence
// (section 3.2), so the gradient of every document is independent.
//
// With P = exp(scale Q K^T - LSE) (causal, same document), D = rowsum(dO * O):
//   dV = P^T dO,  dS = P * (dO V^T - D),  dK = scale dS^T Q,  dQ = scale dS K.
//
// Two persistent kernels (one CTA per SM, 12 warps), so that no partial sum
// ever goes through global memory:
//  - dK/dV pass: a work unit is one key tile (128 keys of one document) for
//    one key/value head; it walks every query tile of the document from the
//    key tile's diagonal on, and for each every query head of that head's GQA
//    group (fully masked tiles are never touched); dK and dV accumulate in TMEM.
//  - dQ pass (further below): a unit is one query tile of one query head; it
//    walks the causal key tiles; dQ accumulates in TMEM.
// S and dP are computed by both passes (seven tile products instead of
// five), in exchange for no dQ reductions, which on this GPU are bounded by
// the L2's reduction throughput.
//   warps 0-7  compute warps (two per scheduler: TMEM lane quarter w % 4,
//              column half w / 4): thread = key row.  S^T and dP^T (keys on
//              the TMEM lanes) -> P^T and dS^T in bf16, written back into
//              TMEM for the dV / dK MMAs; at the end of a unit the dK and dV
//              rows -> bf16 outputs
//   warp 8     TMA producer        warp 9     MMA issuer + TMEM owner
// dK/dV pass, per query tile i of the unit (key tile j):
//   S^T  = K_j Q_i^T      dP^T = V_j dO_i^T           (SS, M = keys)
//   dV  += P^T dO_i       dK  += dS^T Q_i             (TS, A from TMEM)
// TMEM (512 columns): dV [0,D) dK [D,2D) S^T [2D,2D+128) dP^T [2D+128,2D+256);
// P^T aliases S^T's columns [0,32) and [64,96) (one block per column half),
// dS^T the same columns of dP^T.  The compute warps hand P^T and dS^T back
// separately, and the products are issued as
//   S(i) dP(i) | dV(i) S(i+1) | dK(i) dP(i+1) | dV(i+1) S(i+2) | ...
// so the tensor pipe runs two products while the warps compute each phase.
// Every wait is bounded; a timeout sets the device error word and all roles
// stop at the same point, drain and free TMEM.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <string>

#include "internal.h"
#include "sm103_ptx.cuh"

namespace hdp {

hdp_status_t make_bf16_tile_map(CUtensorMap* m, const void* base, long long T, int heads, int d);

namespace {

// Read-only global load that the compiler keeps where it is written (an
// ordinary __ldg may be sunk to its first use, past barriers, and then its
// whole latency is paid there).
__device__ __forceinline__ float ldg_f32_here(const float* p) {
  float v;
  asm volatile("ld.global.nc.f32 %0, [%1];" : "=f"(v) : "l"(p));
  return v;
}

constexpr int kBwdThreads = 384;
constexpr int kBwdProducer = 8;
constexpr int kBwdMma = 9;
constexpr uint32_t kDsBarrier = 2;  // named barrier of the eight compute warps
// Launched at 168 registers a thread (384 x 168 = 64,512); setmaxnreg then
// gives the compute warpgroups more: 2 x 128 x 200 + 128 x 104 = 64,512
// (dQ pass, and the dK/dV pass at d = 64), 2 x 128 x 208 + 128 x 88 =
// 64,512 (dK/dV pass at d = 128, whose compute warps hold P and dP rows).
constexpr int kBwdComputeRegs = 200;
constexpr int kBwdControlRegs = 104;
template <int D>
struct KvRegs {
  static constexpr int kCompute = D == 128 ? 208 : kBwdComputeRegs;
  static constexpr int kControl = D == 128 ? 88 : kBwdControlRegs;
  static_assert(2 * 128 * kCompute + 128 * kControl == 384 * 168, "register split must use the launch's pool");
};

constexpr int kErrBKv = 0x201, kErrBQ = 0x202, kErrBS = 0x203, kErrBP = 0x204, kErrBDkv = 0x207, kErrBDkvE = 0x208,
              kErrBKvE = 0x209, kErrBQE = 0x20a;

template <int D>
struct BwdSmem {
  static constexpr int kTileBytes = kTile * D * 2;  // 128 x D bf16
  static constexpr int kHalfBytes = kTile * 64 * 2;
  static constexpr int kQStages = 3;                // Q(i) is read last by dK(i): keep two tiles in flight
  static constexpr int kK = 0;
  static constexpr int kV = kK + kTileBytes;
  static constexpr int kQ = kV + kTileBytes;                    // 3 stages
  static constexpr int kDO = kQ + kQStages * kTileBytes;        // 2 stages
  static constexpr int kLse = kDO + 2 * kTileBytes;  // 128 fp32: -LSE log2(e) of the tile's queries
  static constexpr int kDl = kLse + kTile * 4;       // 128 fp32: -D scale of the tile's queries
  static constexpr int kBar = kDl + kTile * 4;
  static constexpr int kBytes = kBar + 256;
};

struct BwdBars {
  uint64_t kv_full, kv_empty;
  uint64_t q_full[3], q_empty[3], do_full[2], do_empty[2];
  uint64_t s_full, dp_full, p_full, ds_full, dkv_full, dkv_empty, drain;
  uint32_t tmem_base;
  int abort_word;
};

struct BwdParams {
  const int32_t* tiles;  // fused work list [ntiles][8]; walked backwards
  long long ntiles;
  long long block_kv;    // dK/dV pass: key tiles per block of units (see bwd_unit)
  long long block_q;     // dQ pass: query tiles per block of units (see dq_unit)
  int hq, hkv, group;
  long long T;
  float scale, scale_log2;
  const float* lse;      // [hq][T] natural log
  const float* dl;       // [hq][T] rowsum(dO * O)
  __nv_bfloat16* dq;     // [T][hq][D]
  __nv_bfloat16* dk;     // [T][hkv][D]
  __nv_bfloat16* dv;
  unsigned int* err;
  long long wait_budget;  // clocks before a role's wait gives up (drain waits keep their own budget)
};

struct BwdUnit {
  int k_row0, k_rows, doc_start, doc_len, j, n, kvh, iters;
};

// Units are taken in blocks of `block_kv` key tiles (a grid round covers
// heads_per_round heads of a block), KV head major inside a block: with one
// head per round (long documents) the CTAs of a round all walk the same
// head's Q / dO tiles, from the document's last query tile down, at about the
// same time, so each of those tiles is read from HBM about once per round.
__device__ __forceinline__ BwdUnit bwd_unit(const BwdParams& p, long long u) {
  const long long blk_units = p.block_kv * p.hkv;
  const long long blk = u / blk_units;
  const long long r0 = u - blk * blk_units;
  const long long t0 = blk * p.block_kv;
  const long long gb = p.ntiles - t0 < p.block_kv ? p.ntiles - t0 : p.block_kv;  // key tiles in this block
  const int kvh = static_cast<int>(r0 / gb);
  const long long ti = t0 + (r0 - kvh * gb);
  const int4* row = reinterpret_cast<const int4*>(p.tiles + (p.ntiles - 1 - ti) * 8);
  const int4 a = __ldg(row), b = __ldg(row + 1);
  BwdUnit x;
  x.k_row0 = a.x;
  x.k_rows = a.y;
  x.doc_start = a.z;
  x.doc_len = b.w;
  x.j = b.y / kTile;
  x.n = (x.doc_len + kTile - 1) / kTile;
  x.kvh = kvh;
  x.iters = p.group * (x.n - x.j);
  return x;
}

// The iterations of a unit: the query tiles from the document's last one down
// to the key tile's diagonal, and for each tile every query head of the GQA
// group.  Every unit of a document starts at the same tile and the units of
// one round share a KV head, so the CTAs of a round read the same Q / dO tiles
// at about the same time and those stay in L2.
__device__ __forceinline__ long long bwd_unit_index(long long k, int cta, int nctas) {
  return k * nctas + ((k & 1) ? (nctas - 1 - cta) : cta);
}

__device__ __forceinline__ void bwd_drain_wait(uint64_t* bar, uint32_t parity) {
  const uint32_t a = smem_u32(bar);
  const long long t0 = clock64();
  while (!mbar_try_wait(a, parity)) {
    if (clock64() - t0 > kWaitBudgetClocks / 4) break;
  }
}

template <int D>
__global__ void __launch_bounds__(kBwdThreads, 1)
    k_attn_bwd(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
               const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmDO,
               const BwdParams p) {
  using L = BwdSmem<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  BwdBars& bars = *reinterpret_cast<BwdBars*>(smem + L::kBar);
  volatile int* abort_word = &bars.abort_word;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long total_units = p.ntiles * p.hkv;
  const int cta = blockIdx.x, nctas = gridDim.x;

  if (threadIdx.x == 0) {
    mbar_init(&bars.kv_full, 1);
    mbar_init(&bars.kv_empty, 1);
    for (int s = 0; s < L::kQStages; ++s) {
      mbar_init(&bars.q_full[s], 1);
      mbar_init(&bars.q_empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bars.do_full[s], 1);
      mbar_init(&bars.do_empty[s], 1);
    }
    mbar_init(&bars.s_full, 1);
    mbar_init(&bars.dp_full, 1);
    mbar_init(&bars.p_full, 8);
    mbar_init(&bars.ds_full, 8);
    mbar_init(&bars.dkv_full, 1);
    mbar_init(&bars.dkv_empty, 8);
    mbar_init(&bars.drain, 1);
    bars.abort_word = 0;
    fence_mbarrier_init();
  }
  if (warp == kBwdMma) {
    tmem_alloc(&bars.tmem_base, 512);
    tmem_relinquish();
  }
  if (warp == kBwdProducer && lane == 0) {
    prefetch_tmap(&tmQ);
    prefetch_tmap(&tmK);
    prefetch_tmap(&tmV);
    prefetch_tmap(&tmDO);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars.tmem_base;
  const uint32_t tDV = tmem, tDK = tmem + D, tS = tmem + 2 * D, tDP = tmem + 2 * D + 128;

  if (warp >= 8) {
  // control warpgroup: producer, MMA issuer, two idle warps; registers go to the compute warps
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(KvRegs<D>::kControl));
  if (warp == kBwdProducer) {
    // ------------------------------------------------------------ TMA producer
    // Q of tile g goes to stage g % 3, dO to stage g % 2 (g counts the
    // query tiles of all units of this CTA); K and V once per unit.
    if (lane == 0) {
      int qs = 0;
      long long g = 0, q_armed = 0;    // tiles whose dO / Q loads were issued
      uint32_t units = 0, qround = 0;  // qround: completed passes over the Q stages
      bool ok = true;
      for (long long k = 0; ok; ++k) {
        const long long u = bwd_unit_index(k, cta, nctas);
        if (u >= total_units) break;
        const BwdUnit x = bwd_unit(p, u);
        if (units > 0 && !mbar_wait(&bars.kv_empty, (units - 1) & 1, abort_word, p.err, kErrBKvE, p.wait_budget)) {
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(&bars.kv_full, 2 * L::kTileBytes);
#pragma unroll
        for (int hb = 0; hb < D / 64; ++hb) {
          tma_load_3d(smem + L::kK + hb * L::kHalfBytes, &tmK, &bars.kv_full, hb * 64, x.kvh, x.k_row0);
          tma_load_3d(smem + L::kV + hb * L::kHalfBytes, &tmV, &bars.kv_full, hb * 64, x.kvh, x.k_row0);
        }
        ++units;
        int h = x.kvh * p.group, i = x.n - 1;  // query head and tile of iteration it
        for (int it = 0; it < x.iters; ++it) {
          const int q_row0 = x.doc_start + i * kTile;
          if (qround > 0 && !mbar_wait(&bars.q_empty[qs], (qround - 1) & 1, abort_word, p.err, kErrBQE, p.wait_budget)) {
            q_armed = g;
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&bars.q_full[qs], L::kTileBytes);
#pragma unroll
          for (int hb = 0; hb < D / 64; ++hb)
            tma_load_3d(smem + L::kQ + qs * L::kTileBytes + hb * L::kHalfBytes, &tmQ, &bars.q_full[qs], hb * 64, h,
                        q_row0);
          const int ds = static_cast<int>(g & 1);
          if (g >= 2 && !mbar_wait(&bars.do_empty[ds], ((g >> 1) - 1) & 1, abort_word, p.err, kErrBQE, p.wait_budget)) {
            q_armed = g + 1;
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&bars.do_full[ds], L::kTileBytes);
#pragma unroll
          for (int hb = 0; hb < D / 64; ++hb)
            tma_load_3d(smem + L::kDO + ds * L::kTileBytes + hb * L::kHalfBytes, &tmDO, &bars.do_full[ds], hb * 64,
                        h, q_row0);
          if (++qs == L::kQStages) {
            qs = 0;
            ++qround;
          }
          q_armed = ++g;
          if (h == (x.kvh + 1) * p.group - 1) {
            h = x.kvh * p.group;
            --i;
          } else {
            ++h;
          }
        }
      }
      if (!ok) {
        // every armed barrier completes once its bytes land: stage s of Q
        // was armed by the tiles t < q_armed with t % 3 == s, of dO by the
        // tiles t < g with t % 2 == s
        if (units > 0) bwd_drain_wait(&bars.kv_full, (units - 1) & 1);
        for (int s = 0; s < L::kQStages; ++s) {
          const long long uses = (q_armed + L::kQStages - 1 - s) / L::kQStages;
          if (uses > 0) bwd_drain_wait(&bars.q_full[s], static_cast<uint32_t>(uses - 1) & 1);
        }
        for (int s = 0; s < 2; ++s) {
          const long long uses = (g + 1 - s) / 2;
          if (uses > 0) bwd_drain_wait(&bars.do_full[s], static_cast<uint32_t>(uses - 1) & 1);
        }
      }
    }
    __syncwarp();
    tc_fence_before();
    named_barrier_sync(1, kBwdThreads);
  } else if (warp == kBwdMma) {
    // ------------------------------------------------------------ MMA issuer
    // Issue order, tile g then g + 1:
    //   ... S(g) dP(g) | P(g) | dV(g) S(g+1) | dS(g) | dK(g) dP(g+1) | P(g+1) | ...
    // so the tensor pipe computes dV(g) and S(g+1) while the compute warps
    // turn dP(g) into dS(g), and dK(g), dP(g+1) while they turn S(g+1) into
    // P(g+1).  S(g+1) overwrites the columns that hold P(g), and dP(g+1)
    // those of dS(g): the pipe executes in issue order, so the MMA that
    // reads them has already run.
    if (lane == 0) {
      constexpr uint32_t idesc_s = idesc_bf16_f32(128, 128, 0);   // K-major A and B
      constexpr uint32_t idesc_kv = idesc_bf16_f32(128, D, 1);    // A from TMEM, B MN-major
      constexpr uint64_t kTileUnits = L::kTileBytes >> 4;
      const uint64_t dK_k = sdesc_sw128(smem_u32(smem + L::kK), 16, 1024);
      const uint64_t dV_k = sdesc_sw128(smem_u32(smem + L::kV), 16, 1024);
      const uint64_t dQ_k = sdesc_sw128(smem_u32(smem + L::kQ), 16, 1024);
      const uint64_t dDO_k = sdesc_sw128(smem_u32(smem + L::kDO), 16, 1024);
      const uint64_t dQ_mn = sdesc_sw128(smem_u32(smem + L::kQ), L::kHalfBytes, 1024);
      const uint64_t dDO_mn = sdesc_sw128(smem_u32(smem + L::kDO), L::kHalfBytes, 1024);
      // S^T = K_j Q_g^T into tS
      auto issue_s = [&](int qs) {
        const uint64_t qk = dQ_k + static_cast<uint64_t>(qs) * kTileUnits;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint64_t off = static_cast<uint64_t>((kk >> 2) * L::kHalfBytes + (kk & 3) * 32) >> 4;
          umma_ss(tS, dK_k + off, qk + off, idesc_s, kk > 0);
        }
        umma_commit(&bars.s_full);
      };
      // dP^T = V_j dO_g^T into tDP
      auto issue_dp = [&](int ds) {
        const uint64_t dok = dDO_k + static_cast<uint64_t>(ds) * kTileUnits;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint64_t off = static_cast<uint64_t>((kk >> 2) * L::kHalfBytes + (kk & 3) * 32) >> 4;
          umma_ss(tDP, dV_k + off, dok + off, idesc_s, kk > 0);
        }
        umma_commit(&bars.dp_full);
      };
      long long g = 0;                 // current tile: S(g), dP(g) issued
      int qs = 0, qs_next = 1;         // Q stages of tiles g and g + 1
      uint32_t units = 0;              // index of the current unit
      long long k = 0;
      long long u = bwd_unit_index(0, cta, nctas);
      bool ok = u < total_units;
      BwdUnit x{};
      int it = 0;
      if (ok) {
        x = bwd_unit(p, u);
        ok = mbar_wait(&bars.kv_full, 0, abort_word, p.err, kErrBKv, p.wait_budget) &&
             mbar_wait(&bars.q_full[0], 0, abort_word, p.err, kErrBQ, p.wait_budget);
        if (ok) issue_s(0);
        if (ok) ok = mbar_wait(&bars.do_full[0], 0, abort_word, p.err, kErrBQ, p.wait_budget);
        if (ok) {
          issue_dp(0);
          if (x.iters == 1) umma_commit(&bars.kv_empty);
        }
      }
      while (ok) {
        const bool first = it == 0, last = it == x.iters - 1;
        const int ds = static_cast<int>(g & 1);
        // dV += P^T dO_g, once the compute warps have written P(g)
        ok = mbar_wait(&bars.p_full, g & 1, abort_word, p.err, kErrBP, p.wait_budget);
        if (ok && first && units > 0)
          ok = mbar_wait(&bars.dkv_empty, (units - 1) & 1, abort_word, p.err, kErrBDkvE, p.wait_budget);
        if (!ok) break;
        tc_fence_after();
        {
          const uint64_t domn = dDO_mn + static_cast<uint64_t>(ds) * kTileUnits;
#pragma unroll
          for (int kk = 0; kk < kTile / 16; ++kk)
            umma_ts(tDV, tS + kk * 8 + (kk >= 4 ? 32 : 0), domn + (static_cast<uint64_t>(kk * 2048) >> 4), idesc_kv,
                    (kk > 0 || !first) ? 1u : 0u);
        }
        umma_commit(&bars.do_empty[ds]);
        // the next tile: same unit, or the first tile of the next unit
        bool has_next = true, next_new_unit = false;
        BwdUnit xn = x;
        if (last) {
          const long long un = bwd_unit_index(k + 1, cta, nctas);
          has_next = un < total_units;
          next_new_unit = true;
          if (has_next) xn = bwd_unit(p, un);
        }
        if (has_next) {
          if (next_new_unit) ok = mbar_wait(&bars.kv_full, (units + 1) & 1, abort_word, p.err, kErrBKv, p.wait_budget);
          if (ok) ok = mbar_wait(&bars.q_full[qs_next], ((g + 1) / L::kQStages) & 1, abort_word, p.err, kErrBQ, p.wait_budget);
          if (!ok) break;
          issue_s(qs_next);
        }
        // dK += dS^T Q_g, once the compute warps have written dS(g)
        ok = mbar_wait(&bars.ds_full, g & 1, abort_word, p.err, kErrBP, p.wait_budget);
        if (!ok) break;
        tc_fence_after();
        {
          const uint64_t qmn = dQ_mn + static_cast<uint64_t>(qs) * kTileUnits;
#pragma unroll
          for (int kk = 0; kk < kTile / 16; ++kk)
            umma_ts(tDK, tDP + kk * 8 + (kk >= 4 ? 32 : 0), qmn + (static_cast<uint64_t>(kk * 2048) >> 4), idesc_kv,
                    (kk > 0 || !first) ? 1u : 0u);
        }
        umma_commit(&bars.q_empty[qs]);
        if (last) umma_commit(&bars.dkv_full);
        if (!has_next) break;
        ok = mbar_wait(&bars.do_full[ds ^ 1], ((g + 1) >> 1) & 1, abort_word, p.err, kErrBQ, p.wait_budget);
        if (!ok) break;
        issue_dp(ds ^ 1);
        // K and V of a unit are read last by the S and dP of its last tile
        if (next_new_unit) {
          x = xn;
          ++k;
          ++units;
          it = 0;
        } else {
          ++it;
        }
        if (it == x.iters - 1) umma_commit(&bars.kv_empty);
        ++g;
        qs = qs_next;
        qs_next = qs_next == L::kQStages - 1 ? 0 : qs_next + 1;
      }
      umma_commit(&bars.drain);
      bwd_drain_wait(&bars.drain, 0);
    }
    __syncwarp();
    tc_fence_before();
    named_barrier_sync(1, kBwdThreads);
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  } else {
    named_barrier_sync(1, kBwdThreads);  // idle warps
  }
  } else {
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(KvRegs<D>::kCompute));
    // ------------------------------------------------------------ compute warps 0-7
    // Warp w serves TMEM lane quarter qt = w % 4 (32 key rows) and column
    // half hf = w / 4 (64 query columns of S^T / dP^T), so two warps share
    // each scheduler.  Per query tile, two phases, each answered by the pipe:
    //   P:  P^T = exp2(S^T scale log2e - LSE log2e)  -> bf16 into S^T's columns
    //   dS: dS^T = P^T (dP^T scale - D scale)        -> bf16 into dP^T's columns
    // P stays in registers (fp32) from the first phase to the second.  At
    // the end of a unit the dK and dV rows go out in bf16.
    const int qt = warp & 3, hf = warp >> 2;
    const int r = qt * 32 + lane;
    const int t = threadIdx.x & 127;  // query of the tile whose LSE (warps 0-3) or D (4-7) this thread stages
    const uint32_t lane_off = static_cast<uint32_t>(qt * 32) << 16;
    float* lse2_s = reinterpret_cast<float*>(smem + L::kLse);
    float* dl_s = reinterpret_cast<float*>(smem + L::kDl);
    // LSE (warps 0-3) or D (warps 4-7) of query t of tile (h, i), 0 past the
    // document's end.  Nothing here uses the loaded value, so the load stays
    // in flight until the value is staged one tile later.
    const float* src = threadIdx.x < 128 ? p.lse : p.dl;
    const float mult = threadIdx.x < 128 ? -1.4426950408889634f : -p.scale;
    auto staged = [&](const BwdUnit& x, int h, int i) -> float {
      const int q_local = i * kTile + t;
      float v = 0.f;
      if (q_local < x.doc_len) v = ldg_f32_here(src + static_cast<long long>(h) * p.T + x.doc_start + q_local);
      return v;
    };
    long long g = 0;
    uint32_t units = 0;
    bool ok = true;
    for (long long k = 0; ok; ++k) {
      const long long u = bwd_unit_index(k, cta, nctas);
      if (u >= total_units) break;
      const BwdUnit x = bwd_unit(p, u);
      const int key_local = x.j * kTile + r;
      const bool key_ok = key_local < x.doc_len;
      // query tile i from n - 1 down to j; for each, every head of the group
      int i = x.n - 1, hi = 0;                       // this iteration's query tile and head in the group
      int nh = x.kvh * p.group, ni = x.n - 1;        // the tile `pre` is loaded for
      // Staging: -LSE log2(e) and -D scale (the addends of the FMAs below)
      // of a tile's queries are written once every warp is done with the
      // previous tile, behind the dS phase, where the warps wait for the next
      // S anyway.  The unit's first tile: every warp passed the previous
      // unit's last barrier.
      float pre = staged(x, nh, ni);
      if (threadIdx.x < 128)
        lse2_s[t] = pre * mult;
      else
        dl_s[t] = pre * mult;
      if (named_barrier_or(kDsBarrier, 256, !ok)) {
        ok = false;
        break;
      }
      for (int it = 0; it < x.iters; ++it) {
        if (ok) ok = __all_sync(0xffffffffu, mbar_wait(&bars.s_full, g & 1, abort_word, p.err, kErrBS, p.wait_budget));
        const int q_base = i * kTile;
        const int c_lo = key_local - q_base;  // query column c allowed iff c_lo <= c < c_hi
        const int c_hi = x.doc_len - q_base;
        // ---- P phase: both 32-column chunks of this half (after a failed
        // wait it runs on stale columns; every role is stopping by then)
        uint32_t pv[2][32];
        tc_fence_after();
        tmem_ld32(tS + lane_off + hf * 64, pv[0]);
        tmem_ld32(tS + lane_off + hf * 64 + 32, pv[1]);
        tmem_wait_ld();
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
          const int c0 = hf * 64 + cc * 32;
          uint32_t pk[16];
          if (key_ok && c0 >= c_lo && c0 + 32 <= c_hi) {
            const uint64_t c2 = pack_f32x2(p.scale_log2, p.scale_log2);
            const ulonglong2* l4 = reinterpret_cast<const ulonglong2*>(lse2_s + c0);
#pragma unroll
            for (int e2 = 0; e2 < 16; ++e2) {
              const ulonglong2 lv = l4[e2 >> 1];
              const uint64_t sp = (static_cast<uint64_t>(pv[cc][2 * e2 + 1]) << 32) | pv[cc][2 * e2];
              const uint64_t a = ffma_f32x2(sp, c2, (e2 & 1) ? lv.y : lv.x);
              const float p0 = ex2_approx(lo_f32(a)), p1 = ex2_approx(hi_f32(a));
              pv[cc][2 * e2] = __float_as_uint(p0);
              pv[cc][2 * e2 + 1] = __float_as_uint(p1);
              pk[e2] = pack_bf16x2(p0, p1);
            }
          } else {
#pragma unroll
            for (int e = 0; e < 32; ++e) {
              const int col = c0 + e;
              const bool allowed = key_ok && col >= c_lo && col < c_hi;
              pv[cc][e] = __float_as_uint(
                  allowed ? ex2_approx(fmaf(__uint_as_float(pv[cc][e]), p.scale_log2, lse2_s[col])) : 0.f);
            }
#pragma unroll
            for (int e2 = 0; e2 < 16; ++e2)
              pk[e2] = pack_bf16x2(__uint_as_float(pv[cc][2 * e2]), __uint_as_float(pv[cc][2 * e2 + 1]));
          }
          // chunk cc's pairs go to [64 hf + 16 cc, 64 hf + 16 cc + 16): this
          // half's own columns, already read
          tmem_st16(tS + lane_off + hf * 64 + cc * 16, pk);
        }
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars.p_full);
        // the next tile's LSE / D: it has a whole tile to land
        if (nh == (x.kvh + 1) * p.group - 1) {
          nh = x.kvh * p.group;
          --ni;
        } else {
          ++nh;
        }
        if (it + 1 < x.iters) pre = staged(x, nh, ni);
        // ---- dS phase
        if (ok) ok = __all_sync(0xffffffffu, mbar_wait(&bars.dp_full, g & 1, abort_word, p.err, kErrBS, p.wait_budget));
        if (ok) {
          tc_fence_after();
          uint32_t dpv[2][32];
          tmem_ld32(tDP + lane_off + hf * 64, dpv[0]);
          tmem_ld32(tDP + lane_off + hf * 64 + 32, dpv[1]);
          tmem_wait_ld();
          const uint64_t s2 = pack_f32x2(p.scale, p.scale);
#pragma unroll
          for (int cc = 0; cc < 2; ++cc) {
            // masked entries have P = 0 and a finite dP, so dS = 0 there
            const ulonglong2* d4 = reinterpret_cast<const ulonglong2*>(dl_s + hf * 64 + cc * 32);
            uint32_t pk[16];
#pragma unroll
            for (int e2 = 0; e2 < 16; ++e2) {
              const ulonglong2 dv = d4[e2 >> 1];
              const uint64_t pp = (static_cast<uint64_t>(pv[cc][2 * e2 + 1]) << 32) | pv[cc][2 * e2];
              const uint64_t dp = (static_cast<uint64_t>(dpv[cc][2 * e2 + 1]) << 32) | dpv[cc][2 * e2];
              const uint64_t dsv = fmul_f32x2(pp, ffma_f32x2(dp, s2, (e2 & 1) ? dv.y : dv.x));
              pk[e2] = pack_bf16x2(lo_f32(dsv), hi_f32(dsv));
            }
            tmem_st16(tDP + lane_off + hf * 64 + cc * 16, pk);
          }
          tmem_wait_st();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&bars.ds_full);
        }
        if (it + 1 < x.iters) {
          // every warp is done with this tile's LSE / D: stage the next
          // tile's, and make them visible before its P phase
          if (named_barrier_or(kDsBarrier, 256, !ok)) {
            ok = false;
            break;
          }
          if (threadIdx.x < 128)
            lse2_s[t] = pre * mult;
          else
            dl_s[t] = pre * mult;
          named_barrier_or(kDsBarrier, 256, false);
        }
        if (++hi == p.group) {
          hi = 0;
          --i;
        }
        ++g;
      }
      // a failed dP wait in the unit's last tile is seen by every warp here
      if (named_barrier_or(kDsBarrier, 256, !ok)) {
        ok = false;
        break;
      }
      // ---- the unit's dK and dV rows (thread = key row)
      ok = __all_sync(0xffffffffu, mbar_wait(&bars.dkv_full, units & 1, abort_word, p.err, kErrBDkv, p.wait_budget));
      if (named_barrier_or(kDsBarrier, 256, !ok)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const bool kv_ok = r < x.k_rows;
      const long long krow = (static_cast<long long>(x.k_row0) + r) * p.hkv + x.kvh;
#pragma unroll 1
      for (int which = 0; which < 2; ++which) {
        __nv_bfloat16* out = (which == 0 ? p.dv : p.dk) + krow * D + hf * (D / 2);
        const uint32_t col0 = (which == 0 ? tDV : tDK) + hf * (D / 2);
#pragma unroll 1
        for (int c = 0; c < D / 64; ++c) {
          uint32_t v[32];
          tmem_ld32(col0 + lane_off + c * 32, v);
          tmem_wait_ld();
          if (kv_ok) {
            uint4 w[4];
            uint32_t* wp = reinterpret_cast<uint32_t*>(w);
#pragma unroll
            for (int e = 0; e < 16; ++e) wp[e] = pack_bf16x2(__uint_as_float(v[2 * e]), __uint_as_float(v[2 * e + 1]));
            uint4* d4 = reinterpret_cast<uint4*>(out + c * 32);
#pragma unroll
            for (int e = 0; e < 4; ++e) d4[e] = w[e];
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars.dkv_empty);
      ++units;
    }
    named_barrier_sync(1, kBwdThreads);
  }
}

// ---------------------------------------------------------------- dQ pass
// Query-stationary: a unit is one query tile of one query head (the forward's
// heaviest-first work list, the heads of a tile next to each other so the CTAs
// of one GQA group read the same K / V tiles).  Per key tile j of the causal
// range: S = Q K_j^T, dP = dO V_j^T (SS), then dS = P * (dP - D) * scale from the
// compute warps into S's TMEM columns, and dQ += dS K_j (TS, A from TMEM).  dQ
// accumulates in TMEM over the whole range and is written once, in bf16.
// TMEM: S two buffers [0,128) [128,256), dP [256,384), dQ [384,384+D).  While
// the compute warps work on tile j the MMA thread already computes S(j+1) and,
// once they have read dP(j), dP(j+1).
template <int D>
struct DqSmem {
  static constexpr int kTileBytes = kTile * D * 2;
  static constexpr int kHalfBytes = kTile * 64 * 2;
  static constexpr int kKStages = 3;               // K(j) is read last by dQ(j), one tile later than V(j)
  static constexpr int kQ = 0;
  static constexpr int kDO = kQ + kTileBytes;
  static constexpr int kK = kDO + kTileBytes;               // 3 stages
  static constexpr int kV = kK + kKStages * kTileBytes;     // 2 stages
  static constexpr int kBar = kV + 2 * kTileBytes;
  static constexpr int kBytes = kBar + 256;
};

struct DqBars {
  uint64_t q_full, q_empty;
  uint64_t k_full[3], k_empty[3], v_full[2], v_empty[2];
  uint64_t s_full, dp_free, p_full[2], dq_full, dq_empty, drain;
  uint32_t tmem_base;
  int abort_word;
};

constexpr int kErrDQ = 0x301, kErrDKv = 0x302, kErrDS = 0x303, kErrDDp = 0x304, kErrDP = 0x305, kErrDDq = 0x306,
              kErrDDqE = 0x307, kErrDQE = 0x308, kErrDKvE = 0x309;

struct DqUnit {
  int q_row0, q_rows, doc_start, doc_len, i, ntk, h, kvh;
};

// Units in blocks of `block_q` query tiles (a grid round covers
// heads_per_round heads of a block), KV head major inside a block (then tile,
// then query head of the group): with one head per round the CTAs of a round
// stream the same head's K / V tiles together, for L2 reuse.
__device__ __forceinline__ DqUnit dq_unit(const BwdParams& p, long long u) {
  const long long blk_units = p.block_q * p.hq;
  const long long blk = u / blk_units;
  const long long r0 = u - blk * blk_units;
  const long long t0 = blk * p.block_q;
  const long long gb = p.ntiles - t0 < p.block_q ? p.ntiles - t0 : p.block_q;  // query tiles in this block
  const long long per_head = gb * p.group;
  const int kvh = static_cast<int>(r0 / per_head);
  const long long rem = r0 - kvh * per_head;
  const long long ti = t0 + rem / p.group;
  const int4* row = reinterpret_cast<const int4*>(p.tiles + ti * 8);
  const int4 a = __ldg(row), b = __ldg(row + 1);
  DqUnit x;
  x.q_row0 = a.x;
  x.q_rows = a.y;
  x.doc_start = a.z;
  x.ntk = (a.w + kTile - 1) / kTile;  // key tiles of the causal range
  x.i = b.y / kTile;
  x.doc_len = b.w;
  x.h = kvh * p.group + static_cast<int>(rem - (rem / p.group) * p.group);
  x.kvh = kvh;
  return x;
}

template <int D>
__global__ void __launch_bounds__(kBwdThreads, 1)
    k_attn_bwd_dq(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                  const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmDO,
                  const BwdParams p) {
  using L = DqSmem<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  DqBars& bars = *reinterpret_cast<DqBars*>(smem + L::kBar);
  volatile int* abort_word = &bars.abort_word;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long total_units = p.ntiles * p.hq;
  const int cta = blockIdx.x, nctas = gridDim.x;

  if (threadIdx.x == 0) {
    mbar_init(&bars.q_full, 1);
    mbar_init(&bars.q_empty, 1);
    for (int s = 0; s < L::kKStages; ++s) {
      mbar_init(&bars.k_full[s], 1);
      mbar_init(&bars.k_empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bars.v_full[s], 1);
      mbar_init(&bars.v_empty[s], 1);
    }
    mbar_init(&bars.s_full, 1);
    mbar_init(&bars.dp_free, 8);
    // two barriers for P: the compute warps could otherwise finish the tile
    // after next before the MMA thread has seen this one
    mbar_init(&bars.p_full[0], 8);
    mbar_init(&bars.p_full[1], 8);
    mbar_init(&bars.dq_full, 1);
    mbar_init(&bars.dq_empty, 8);
    mbar_init(&bars.drain, 1);
    bars.abort_word = 0;
    fence_mbarrier_init();
  }
  if (warp == kBwdMma) {
    tmem_alloc(&bars.tmem_base, 512);
    tmem_relinquish();
  }
  if (warp == kBwdProducer && lane == 0) {
    prefetch_tmap(&tmQ);
    prefetch_tmap(&tmK);
    prefetch_tmap(&tmV);
    prefetch_tmap(&tmDO);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars.tmem_base;
  const uint32_t tS0 = tmem, tDP = tmem + 256, tDQ = tmem + 384;

  if (warp >= 8) {
  // control warpgroup: producer, MMA issuer, two idle warps; registers go to the compute warps
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kBwdControlRegs));
  if (warp == kBwdProducer) {
    // ------------------------------------------------------------ TMA producer
    // K of key tile t (t counts the key tiles of all units of this CTA)
    // goes to stage t % 3, V to stage t % 2.
    if (lane == 0) {
      uint32_t units = 0, kround = 0;  // kround: completed passes over the K stages
      int ks = 0;
      long long kvc = 0, k_armed = 0;  // key tiles whose V / K loads were issued
      bool ok = true;
      for (long long k = 0; ok; ++k) {
        const long long u = bwd_unit_index(k, cta, nctas);
        if (u >= total_units) break;
        const DqUnit x = dq_unit(p, u);
        if (units > 0 && !mbar_wait(&bars.q_empty, (units - 1) & 1, abort_word, p.err, kErrDQE, p.wait_budget)) {
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(&bars.q_full, 2 * L::kTileBytes);
#pragma unroll
        for (int hb = 0; hb < D / 64; ++hb) {
          tma_load_3d(smem + L::kQ + hb * L::kHalfBytes, &tmQ, &bars.q_full, hb * 64, x.h, x.q_row0);
          tma_load_3d(smem + L::kDO + hb * L::kHalfBytes, &tmDO, &bars.q_full, hb * 64, x.h, x.q_row0);
        }
        ++units;
        for (int j = 0; j < x.ntk; ++j) {
          const int row0 = x.doc_start + j * kTile;
          if (kround > 0 && !mbar_wait(&bars.k_empty[ks], (kround - 1) & 1, abort_word, p.err, kErrDKvE, p.wait_budget)) {
            k_armed = kvc;
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&bars.k_full[ks], L::kTileBytes);
#pragma unroll
          for (int hb = 0; hb < D / 64; ++hb)
            tma_load_3d(smem + L::kK + ks * L::kTileBytes + hb * L::kHalfBytes, &tmK, &bars.k_full[ks], hb * 64,
                        x.kvh, row0);
          const int vs = static_cast<int>(kvc & 1);
          if (kvc >= 2 && !mbar_wait(&bars.v_empty[vs], ((kvc >> 1) - 1) & 1, abort_word, p.err, kErrDKvE, p.wait_budget)) {
            k_armed = kvc + 1;
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&bars.v_full[vs], L::kTileBytes);
#pragma unroll
          for (int hb = 0; hb < D / 64; ++hb)
            tma_load_3d(smem + L::kV + vs * L::kTileBytes + hb * L::kHalfBytes, &tmV, &bars.v_full[vs], hb * 64,
                        x.kvh, row0);
          if (++ks == L::kKStages) {
            ks = 0;
            ++kround;
          }
          k_armed = ++kvc;
        }
      }
      if (!ok) {
        // every armed barrier completes once its bytes land
        if (units > 0) bwd_drain_wait(&bars.q_full, (units - 1) & 1);
        for (int s = 0; s < L::kKStages; ++s) {
          const long long uses = (k_armed + L::kKStages - 1 - s) / L::kKStages;
          if (uses > 0) bwd_drain_wait(&bars.k_full[s], static_cast<uint32_t>(uses - 1) & 1);
        }
        for (int s = 0; s < 2; ++s) {
          const long long uses = (kvc + 1 - s) / 2;
          if (uses > 0) bwd_drain_wait(&bars.v_full[s], static_cast<uint32_t>(uses - 1) & 1);
        }
      }
    }
    __syncwarp();
    tc_fence_before();
    named_barrier_sync(1, kBwdThreads);
  } else if (warp == kBwdMma) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_s = idesc_bf16_f32(128, 128, 0);
      constexpr uint32_t idesc_q = idesc_bf16_f32(128, D, 1);
      constexpr uint64_t kTileUnits = L::kTileBytes >> 4;
      const uint64_t dQ_k = sdesc_sw128(smem_u32(smem + L::kQ), 16, 1024);
      const uint64_t dDO_k = sdesc_sw128(smem_u32(smem + L::kDO), 16, 1024);
      const uint64_t dK_k = sdesc_sw128(smem_u32(smem + L::kK), 16, 1024);
      const uint64_t dV_k = sdesc_sw128(smem_u32(smem + L::kV), 16, 1024);
      const uint64_t dK_mn = sdesc_sw128(smem_u32(smem + L::kK), L::kHalfBytes, 1024);
      uint32_t units = 0, kround = 0;
      int ks = 0, ks_prev = 0;  // K stages of this key tile and of the previous one
      long long kvc = 0;  // key tiles issued so far (all units): stages, S buffer and barrier phases
      bool ok = true;
      // dQ += dS(t) K(t) for global tile t (its dS sits in S buffer t & 1, its K in stage kst)
      auto issue_dq = [&](long long t, int kst, bool first_of_unit) -> bool {
        if (!mbar_wait(&bars.p_full[t & 1], (t >> 1) & 1, abort_word, p.err, kErrDP, p.wait_budget)) return false;
        if (first_of_unit && units > 0 &&
            !mbar_wait(&bars.dq_empty, (units - 1) & 1, abort_word, p.err, kErrDDqE, p.wait_budget))
          return false;
        tc_fence_after();
        const uint32_t a = tS0 + static_cast<uint32_t>(t & 1) * 128u;
        const uint64_t b = dK_mn + static_cast<uint64_t>(kst) * kTileUnits;
#pragma unroll
        for (int kk = 0; kk < kTile / 16; ++kk)
          umma_ts(tDQ, a + kk * 8 + (kk >= 4 ? 32 : 0), b + (static_cast<uint64_t>(kk * 2048) >> 4), idesc_q,
                  (first_of_unit && kk == 0) ? 0u : 1u);
        umma_commit(&bars.k_empty[kst]);
        return true;
      };
      for (long long k = 0; ok; ++k) {
        const long long u = bwd_unit_index(k, cta, nctas);
        if (u >= total_units) break;
        const DqUnit x = dq_unit(p, u);
        ok = mbar_wait(&bars.q_full, units & 1, abort_word, p.err, kErrDQ, p.wait_budget);
        if (!ok) break;
        for (int j = 0; j < x.ntk && ok; ++j) {
          const int st = static_cast<int>(kvc & 1);
          ok = mbar_wait(&bars.k_full[ks], kround & 1, abort_word, p.err, kErrDKv, p.wait_budget);
          if (!ok) break;
          // S(j) into buffer st: its previous dS was read by a dQ MMA issued earlier
          const uint64_t kd = dK_k + static_cast<uint64_t>(ks) * kTileUnits;
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint64_t off = static_cast<uint64_t>((kk >> 2) * L::kHalfBytes + (kk & 3) * 32) >> 4;
            umma_ss(tS0 + st * 128u, dQ_k + off, kd + off, idesc_s, kk > 0);
          }
          // dP(j) once the compute warps have read dP(j-1)
          if (kvc > 0) {
            ok = mbar_wait(&bars.dp_free, (kvc - 1) & 1, abort_word, p.err, kErrDDp, p.wait_budget);
            if (!ok) break;
            tc_fence_after();
          }
          ok = mbar_wait(&bars.v_full[st], (kvc >> 1) & 1, abort_word, p.err, kErrDKv, p.wait_budget);
          if (!ok) break;
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint64_t off = static_cast<uint64_t>((kk >> 2) * L::kHalfBytes + (kk & 3) * 32) >> 4;
            umma_ss(tDP, dDO_k + off, dV_k + st * kTileUnits + off, idesc_s, kk > 0);
          }
          umma_commit(&bars.v_empty[st]);  // V(j) is read by dP(j) alone
          umma_commit(&bars.s_full);
          if (j == x.ntk - 1) umma_commit(&bars.q_empty);  // Q and dO are read by then
          // dQ of the previous tile of this unit
          if (j > 0) ok = issue_dq(kvc - 1, ks_prev, j == 1);
          ks_prev = ks;
          if (++ks == L::kKStages) {
            ks = 0;
            ++kround;
          }
          ++kvc;
        }
        if (ok) ok = issue_dq(kvc - 1, ks_prev, x.ntk == 1);
        if (ok) umma_commit(&bars.dq_full);
        ++units;
      }
      umma_commit(&bars.drain);
      bwd_drain_wait(&bars.drain, 0);
    }
    __syncwarp();
    tc_fence_before();
    named_barrier_sync(1, kBwdThreads);
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  } else {
    named_barrier_sync(1, kBwdThreads);
  }
  } else {
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kBwdComputeRegs));
    // ------------------------------------------------------------ compute warps (thread = query row)
    const int qt = warp & 3, hf = warp >> 2;
    const int r = qt * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(qt * 32) << 16;
    long long tg = 0;
    uint32_t units = 0;
    bool ok = true;
    for (long long k = 0; ok; ++k) {
      const long long u = bwd_unit_index(k, cta, nctas);
      if (u >= total_units) break;
      const DqUnit x = dq_unit(p, u);
      const int q_local = x.i * kTile + r;
      const bool row_ok = r < x.q_rows;
      const long long tok = static_cast<long long>(x.q_row0) + r;
      const float lse2 = row_ok ? __ldg(p.lse + static_cast<long long>(x.h) * p.T + tok) * 1.4426950408889634f : 0.f;
      const float dlr = row_ok ? __ldg(p.dl + static_cast<long long>(x.h) * p.T + tok) : 0.f;
      const uint64_t c2 = pack_f32x2(p.scale_log2, p.scale_log2), s2 = pack_f32x2(p.scale, p.scale);
      const uint64_t nl2 = pack_f32x2(-lse2, -lse2), nd2 = pack_f32x2(-dlr * p.scale, -dlr * p.scale);
      for (int j = 0; j < x.ntk; ++j) {
        ok = __all_sync(0xffffffffu, mbar_wait(&bars.s_full, tg & 1, abort_word, p.err, kErrDS, p.wait_budget));
        if (!ok) break;
        tc_fence_after();
        const uint32_t tS = tS0 + static_cast<uint32_t>(tg & 1) * 128u;
        uint32_t sv[64], dpv[64];
        tmem_ld32(tS + lane_off + hf * 64, *reinterpret_cast<uint32_t(*)[32]>(sv));
        tmem_ld32(tS + lane_off + hf * 64 + 32, *reinterpret_cast<uint32_t(*)[32]>(sv + 32));
        tmem_ld32(tDP + lane_off + hf * 64, *reinterpret_cast<uint32_t(*)[32]>(dpv));
        tmem_ld32(tDP + lane_off + hf * 64 + 32, *reinterpret_cast<uint32_t(*)[32]>(dpv + 32));
        tmem_wait_ld();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars.dp_free);
        // key column c (doc-local key j*128 + 64 hf + c) is allowed iff it is <= q_local
        const int c_hi = row_ok ? q_local - (j * kTile + hf * 64) + 1 : 0;  // allowed: c < c_hi
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
          uint32_t pk[16];
          if (c_hi >= cc * 32 + 32) {
            // every key of the chunk is visible to this query: packed pairs
#pragma unroll
            for (int e2 = 0; e2 < 16; ++e2) {
              const int c = cc * 32 + 2 * e2;
              const uint64_t sp = (static_cast<uint64_t>(sv[c + 1]) << 32) | sv[c];
              const uint64_t dp = (static_cast<uint64_t>(dpv[c + 1]) << 32) | dpv[c];
              const uint64_t a = ffma_f32x2(sp, c2, nl2);
              const float p0 = ex2_approx(lo_f32(a)), p1 = ex2_approx(hi_f32(a));
              const uint64_t ds = fmul_f32x2(pack_f32x2(p0, p1), ffma_f32x2(dp, s2, nd2));
              pk[e2] = pack_bf16x2(lo_f32(ds), hi_f32(ds));
            }
          } else {
#pragma unroll
            for (int e = 0; e < 32; e += 2) {
              float dd[2];
#pragma unroll
              for (int t = 0; t < 2; ++t) {
                const int c = cc * 32 + e + t;
                const float pe = c < c_hi ? ex2_approx(fmaf(__uint_as_float(sv[c]), p.scale_log2, -lse2)) : 0.f;
                dd[t] = pe * (__uint_as_float(dpv[c]) - dlr) * p.scale;
              }
              pk[e / 2] = pack_bf16x2(dd[0], dd[1]);
            }
          }
          tmem_st16(tS + lane_off + hf * 64 + cc * 16, pk);
        }
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars.p_full[tg & 1]);
        ++tg;
      }
      if (!ok) break;
      // ---- dQ of the unit -> bf16 rows
      ok = __all_sync(0xffffffffu, mbar_wait(&bars.dq_full, units & 1, abort_word, p.err, kErrDDq, p.wait_budget));
      if (!ok) break;
      tc_fence_after();
      __nv_bfloat16* out = p.dq + (tok * p.hq + x.h) * static_cast<long long>(D) + hf * (D / 2);
#pragma unroll 1
      for (int c = 0; c < D / 64; ++c) {
        uint32_t v[32];
        tmem_ld32(tDQ + lane_off + hf * (D / 2) + c * 32, v);
        tmem_wait_ld();
        if (row_ok) {
          uint4 w[4];
          uint32_t* wp = reinterpret_cast<uint32_t*>(w);
#pragma unroll
          for (int e = 0; e < 16; ++e) wp[e] = pack_bf16x2(__uint_as_float(v[2 * e]), __uint_as_float(v[2 * e + 1]));
          uint4* d4 = reinterpret_cast<uint4*>(out + c * 32);
#pragma unroll
          for (int e = 0; e < 4; ++e) d4[e] = w[e];
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars.dq_empty);
      ++units;
    }
    named_barrier_sync(1, kBwdThreads);
  }
}

// D[h][t] = sum_c dO[t][h][c] * O[t][h][c]; 16 threads per (t, h) row, 8
// elements (16 bytes) per thread per step.
template <int D>
__global__ void k_bwd_delta(const __nv_bfloat16* __restrict__ o, const __nv_bfloat16* __restrict__ dout,
                            float* __restrict__ dl, long long rows, int hq, long long T) {
  const long long row = (blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x) / 16;
  const int sub = threadIdx.x & 15;
  float acc = 0.f;
  if (row < rows) {
#pragma unroll
    for (int c = sub * 8; c < D; c += 128) {
      const uint4 a = __ldg(reinterpret_cast<const uint4*>(o + row * D + c));
      const uint4 b = __ldg(reinterpret_cast<const uint4*>(dout + row * D + c));
      const __nv_bfloat162* a2 = reinterpret_cast<const __nv_bfloat162*>(&a);
      const __nv_bfloat162* b2 = reinterpret_cast<const __nv_bfloat162*>(&b);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 fa = __bfloat1622float2(a2[e]), fb = __bfloat1622float2(b2[e]);
        acc = fmaf(fa.x, fb.x, acc);
        acc = fmaf(fa.y, fb.y, acc);
      }
    }
  }
#pragma unroll
  for (int off = 8; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
  if (row < rows && sub == 0) {
    const long long t = row / hq;
    const int h = static_cast<int>(row - t * hq);
    dl[static_cast<long long>(h) * T + t] = acc;
  }
}

// dynamic shared memory of a launch = layout + 1 KB for the 1024-byte
// alignment of the swizzled tiles; the per-block opt-in limit is 227 KB
static_assert(BwdSmem<128>::kBytes + 1024 <= 227 * 1024, "dK/dV pass shared memory");
static_assert(DqSmem<128>::kBytes + 1024 <= 227 * 1024, "dQ pass shared memory");
static_assert(sizeof(BwdBars) <= 256 && sizeof(DqBars) <= 256, "barrier block");

size_t bwd_align256(size_t x) { return (x + 255) & ~size_t(255); }

void bwd_workspace(const hdp_plan_s* plan, int hq, size_t* total) {
  const size_t T = static_cast<size_t>(plan->v.total_tokens);
  *total = bwd_align256(T * hq * sizeof(float));  // D = rowsum(dout * o)
}

template <int D>
hdp_status_t launch_bwd(const hdp_plan_s* plan, const void* q, const void* k, const void* v, const void* o,
                        const float* lse, const void* dout, int hq, int hkv, float scale, float* dl, void* dq,
                        void* dk, void* dv, cudaStream_t st) {
  const long long T = plan->v.total_tokens;
  if (T == 0) return HDP_OK;
  CUtensorMap mq, mk, mv, mdo;
  hdp_status_t r;
  if ((r = make_bf16_tile_map(&mq, q, T, hq, D)) != HDP_OK) return r;
  if ((r = make_bf16_tile_map(&mk, k, T, hkv, D)) != HDP_OK) return r;
  if ((r = make_bf16_tile_map(&mv, v, T, hkv, D)) != HDP_OK) return r;
  if ((r = make_bf16_tile_map(&mdo, dout, T, hq, D)) != HDP_OK) return r;
  int dev = 0, sms = 0;
  HDP_CUDA_TRY(cudaGetDevice(&dev));
  HDP_CUDA_TRY(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
  // D = rowsum(dO * O)
  const long long rows = T * hq;
  k_bwd_delta<D><<<static_cast<unsigned>((rows * 16 + 255) / 256), 256, 0, st>>>(
      static_cast<const __nv_bfloat16*>(o), static_cast<const __nv_bfloat16*>(dout), dl, rows, hq, T);
  note_launch();
  HDP_CUDA_TRY(cudaGetLastError());
  BwdParams prm{};
  prm.tiles = plan->v.tiles_fused;
  prm.ntiles = plan->v.num_tiles_fused;
  prm.hq = hq;
  prm.hkv = hkv;
  prm.group = hq / hkv;
  prm.T = T;
  prm.scale = scale;
  prm.scale_log2 = scale * 1.4426950408889634f;
  prm.lse = lse;
  prm.dl = dl;
  prm.dq = static_cast<__nv_bfloat16*>(dq);
  prm.dk = static_cast<__nv_bfloat16*>(dk);
  prm.dv = static_cast<__nv_bfloat16*>(dv);
  prm.err = device_error_word();
  if (!prm.err) return fail(HDP_ERR_CUDA, "cannot resolve the device error word");
  prm.wait_budget = wait_budget_clocks();
  // dK, dV: one unit per (key tile, kv head)
  {
    const long long units = prm.ntiles * hkv;
    const int grid = static_cast<int>(units < sms ? units : sms);
    const long long bk = grid / heads_per_round(plan->v.max_doc_len, hkv);
    prm.block_kv = bk > 0 ? bk : 1;
    const int smem = BwdSmem<D>::kBytes + 1024;
    HDP_CUDA_TRY(cudaFuncSetAttribute(k_attn_bwd<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem));
    k_attn_bwd<D><<<grid, kBwdThreads, smem, st>>>(mq, mk, mv, mdo, prm);
    note_launch();
    HDP_CUDA_TRY(cudaGetLastError());
  }
  // dQ: one unit per (query tile, query head)
  {
    const long long units = prm.ntiles * hq;
    const int grid = static_cast<int>(units < sms ? units : sms);
    const long long bq = grid / (prm.group * heads_per_round(plan->v.max_doc_len, hkv));
    prm.block_q = bq > 0 ? bq : 1;
    const int smem = DqSmem<D>::kBytes + 1024;
    HDP_CUDA_TRY(cudaFuncSetAttribute(k_attn_bwd_dq<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem));
    k_attn_bwd_dq<D><<<grid, kBwdThreads, smem, st>>>(mq, mk, mv, mdo, prm);
    note_launch();
    HDP_CUDA_TRY(cudaGetLastError());
  }
  return HDP_OK;
}

}  // namespace
}  // namespace hdp

using namespace hdp;

extern "C" hdp_status_t hdp_attention_bwd_workspace_bytes(hdp_plan_t plan, int32_t hq, int32_t d, size_t* bytes) {
  if (!plan || !bytes) return fail(HDP_ERR_INVALID_ARGUMENT, "hdp_attention_bwd_workspace_bytes: NULL argument");
  if (hq < 1 || d < 1)
    return fail(HDP_ERR_INVALID_ARGUMENT, "hdp_attention_bwd_workspace_bytes: hq, d must be >= 1");
  bwd_workspace(plan, hq, bytes);
  return HDP_OK;
}

extern "C" hdp_status_t hdp_attention_bwd(hdp_plan_t plan, const void* q, const void* k, const void* v,
                                          const void* o, const float* lse, const void* dout, int32_t hq,
                                          int32_t hkv, int32_t d, float scale, void* workspace,
                                          size_t workspace_bytes, void* dq, void* dk, void* dv, void* stream) {
  if (!plan || !q || !k || !v || !o || !lse || !dout || !dq || !dk || !dv)
    return fail(HDP_ERR_INVALID_ARGUMENT, "hdp_attention_bwd: NULL argument");
  if (hq < 1 || hkv < 1 || hq % hkv != 0)
    return fail(HDP_ERR_INVALID_ARGUMENT, "hdp_attention_bwd: need hq >= 1, hkv >= 1, hq % hkv == 0");
  if (!(scale > 0.f)) return fail(HDP_ERR_INVALID_ARGUMENT, "hdp_attention_bwd: scale must be > 0");
  if (d != 64 && d != 128) return fail(HDP_ERR_UNSUPPORTED, "hdp_attention_bwd: d must be 64 or 128");
  const uintptr_t mis = reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k) |
                        reinterpret_cast<uintptr_t>(v) | reinterpret_cast<uintptr_t>(o) |
                        reinterpret_cast<uintptr_t>(dout) | reinterpret_cast<uintptr_t>(dq) |
                        reinterpret_cast<uintptr_t>(dk) | reinterpret_cast<uintptr_t>(dv);
  if (mis & 15)
    return fail(HDP_ERR_INVALID_ARGUMENT, "hdp_attention_bwd: q, k, v, o, dout, dq, dk, dv must be 16-byte aligned");
  size_t need = 0;
  bwd_workspace(plan, hq, &need);
  if (!workspace || workspace_bytes < need)
    return fail(HDP_ERR_INVALID_ARGUMENT,
                "hdp_attention_bwd: workspace too small (need " + std::to_string(need) + " bytes)");
  if (reinterpret_cast<uintptr_t>(workspace) & 255)
    return fail(HDP_ERR_INVALID_ARGUMENT, "hdp_attention_bwd: workspace must be 256-byte aligned");
  float* dl = static_cast<float*>(workspace);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  return d == 128 ? launch_bwd<128>(plan, q, k, v, o, lse, dout, hq, hkv, scale, dl, dq, dk, dv, st)
                  : launch_bwd<64>(plan, q, k, v, o, lse, dout, hq, hkv, scale, dl, dq, dk, dv, st);
}
