// Document-masked causal attention forward on tcgen05 tensor cores
// ("ByteScale: Communication-Efficient Scaling of LLM Training with a 2048K
// Context Length on 16384 GPUs", research digest, section 3.2: a query attends
// only to its own sequence; each C x C block of a long sequence is a partial
// result, and partials are combined by log-sum-exp).
//
// Design (one persistent CTA per SM, 12 warps):
//   warps 0-3  softmax for query slot 0     warps 4-7  softmax for query slot 1
//   warp 8     TMA producer                 warp 9     MMA issuer + TMEM owner
//   warps 10, 11 idle (they complete the control warpgroup)
// A work unit is one query tile (128 rows of one document, from the plan's
// heaviest-first work list) for one key/value head and a pair of query heads of
// that head's GQA group: both slots share every K/V tile.  Only the key tiles
// of the tile's causal range inside its own document are visited, so fully
// masked tiles are never loaded or computed; the mask is applied only on the
// tiles that straddle the diagonal or the end of the key range.
//
// Per key tile j and slot s:
//   S_s = Q_s K_j^T        tcgen05.mma, A and B from 128B-swizzled smem, D in TMEM
//   softmax_s              tcgen05.ld S, online max / exp2 / row sum in fp32,
//                          P (bf16) written back into S's TMEM columns
//   O_s += P_s V_j         tcgen05.mma with A = P from TMEM, B = V (MN-major smem)
// The online softmax keeps a stale running max unless it grows by more than
// 2^8, so O is rescaled only rarely; the final O/l and LSE use the same max, so
// the result is exact.  In SPLIT mode each block (q chunk, kv chunk) ends in a
// partial (O fp32, LSE) instead: the units are FUSED's (a query tile over its
// whole causal key range), and at each chunk boundary of that range the block
// just finished is written and the running max, l and O restart.  Each
// partial covers exactly its own C keys, and no block restarts a unit (a new
// Q tile, a refilled pipeline).
//
// Pacing (documents whose K and V rows of one head exceed L2): the CTAs of a
// round stream the same K/V tiles, and they share them through L2 only while
// they stay close together on the key range.  The SMs run at slightly
// different speeds (about 2 % apart, steadily), so unpaced CTAs drift apart by
// thousands of key tiles and each reads the tiles from HBM again.  So each
// producer publishes its position on its K/V stream, a pacer warp reads the
// positions of the other CTAs on the same stream, and the producer holds its
// next load while it is more than a window ahead of the slowest.  The
// kernel's duration was set by the slowest CTA anyway; what changes is that
// the K/V tiles come from L2 (fewer HBM reads, so more of the power budget
// for the SMs' clock).  Pacing is advisory: every hold is bounded, and it
// never changes what is computed.
//
// Every mbarrier wait is bounded; a timeout sets the device error word, all
// roles stop, in-flight copies and MMAs are drained, TMEM is freed.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstdio>
#include <mutex>

#include "internal.h"
#include "sm103_ptx.cuh"

namespace hdp {

hdp_status_t launch_merge_blocks(const hdp_plan_s* plan, const float* o_part, const float* lse_part, int32_t hq,
                                 int32_t d, void* o, float* lse, cudaStream_t st);

// Positions of the CTAs of a paced launch on their K/V streams (one slot per CTA).
__device__ unsigned long long g_pace[1024];

namespace {

// 12 warps = 3 warpgroups: two softmax warpgroups and one for the producer
// (warp 8), the MMA issuer (warp 9) and two idle warps.
// Launched at 168 registers a thread (384 x 168 = 64,512); setmaxnreg then moves registers to
// the softmax warpgroups: 2 x 128 x 176 + 128 x 152 = 64,512 (the MMA
// issuer's straight-line code needs the control share).
constexpr int kThreads = 384;
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;
constexpr int kPacerWarp = 10;
constexpr int kPaceEvery = 8;    // key tiles between published positions
constexpr int kPaceWindow = 24;  // key tiles a CTA may run ahead of the slowest on its stream
constexpr unsigned int kPaceDone = 0xFFFFFFu;
constexpr int kSoftmaxRegs = 176;
constexpr int kControlRegs = 152;
constexpr int kStages = 2;  // K and V ring depth
constexpr float kRescaleThreshold = 8.0f;  // log2 units: rescale O only when the max grows by > 2^8

// error codes recorded in the device error word
constexpr int kErrQFull = 0x101, kErrKFull = 0x102, kErrVFull = 0x103, kErrSFull = 0x104, kErrPFull = 0x105,
              kErrOFull = 0x106, kErrOEmpty = 0x107, kErrKEmpty = 0x108, kErrVEmpty = 0x109, kErrQEmpty = 0x10a,
              kErrKvEmpty = 0x10b;

template <int D>
struct SmemLayout {
  static constexpr int kTileBytes = kTile * D * 2;  // one 128 x D bf16 tile
  static constexpr int kHalfBytes = kTile * 64 * 2;  // one 64-column (128-byte) half
  static constexpr int kQ = 0;
  static constexpr int kK = kQ + 2 * kTileBytes;
  static constexpr int kV = kK + kStages * kTileBytes;
  static constexpr int kBar = kV + kStages * kTileBytes;
  static constexpr int kBytes = kBar + 512;
};

struct Bars {
  uint64_t q_full[2], q_empty[2];
  uint64_t kv_full[2];                 // one TMA group: K(j+1) and/or V(j)
  uint64_t kv_empty[2];                // the MMA thread has consumed that group's phase
  uint64_t k_empty[kStages], v_empty[kStages];
  uint64_t s_full[2], p_full[2], o_full[2], o_empty[2];
  uint64_t drain;  // private to the MMA thread: completion of all its MMAs at exit
  uint64_t pace_entry;  // this CTA's last published position (producer -> pacer)
  uint64_t pace_limit;  // stream << 32 | furthest key tile the producer may load (pacer -> producer)
  uint32_t tmem_base;
  int abort_word;
  int pace_done;        // the producer has finished
};

struct Params {
  const int32_t* tiles;  // [ntiles][8]
  long long ntiles;
  long long block_tiles;  // work-list tiles per block of units (see load_unit)
  int hq, hkv, group, npairs;
  float scale_log2;      // scale * log2(e)
  long long T;
  __nv_bfloat16* o;      // FUSED output [T][hq][D]
  float* lse;            // FUSED output [hq][T]
  float* o_part;         // SPLIT partials [N_b][C][hq][D]
  float* lse_part;       // SPLIT partials [N_b][hq][C]
  int C;
  int tpc;               // SPLIT: key tiles per chunk, C / 128
  int ndocs;
  const int32_t* cu;     // SPLIT: cu_seqlens [ndocs + 1]
  const int64_t* bo;     // SPLIT: first causal block of each document [ndocs + 1]
  unsigned int* err;
  unsigned long long* pace;  // per-CTA positions on the K/V streams, or nullptr: no pacing
  unsigned int pace_epoch;   // 8 bits, distinct for consecutive launches
  long long wait_budget;  // clocks before a role's wait gives up (drain waits keep their own budget)
};

struct Unit {
  int q_row0, q_rows, kv_row0, kv_len, blk, row_off;
  int kvh, h0;       // kv head, first query head of the pair
  bool valid1;       // slot 1 in use
  int ntiles_kv;
};

// Units are taken in blocks of `block_tiles` consecutive work-list tiles
// (grid / (pairs per head x heads per round), so a round of the persistent
// grid covers `heads_per_round` heads of one block); inside a block the order
// is KV head, then tile, then query-head pair.  With one head per round (long
// documents) the CTAs of a round all stream the same head's K/V (the same key
// prefix, for the tiles of one long document) at about the same time, and
// each K/V tile is read from HBM about once per round instead of once per
// CTA.  Blocks follow the heaviest-first order of the work list.
__device__ __forceinline__ Unit load_unit(const Params& p, long long u) {
  const long long per_tile = static_cast<long long>(p.hkv) * p.npairs;
  const long long blk_units = p.block_tiles * per_tile;
  const long long blk = u / blk_units;
  const long long r0 = u - blk * blk_units;
  const long long t0 = blk * p.block_tiles;
  const long long gb = p.ntiles - t0 < p.block_tiles ? p.ntiles - t0 : p.block_tiles;  // tiles in this block
  const long long per_head = gb * p.npairs;
  const int kvh = static_cast<int>(r0 / per_head);
  const long long rem = r0 - kvh * per_head;
  const long long ti = t0 + rem / p.npairs;
  const int r = kvh * p.npairs + static_cast<int>(rem - (rem / p.npairs) * p.npairs);
  const int4* row = reinterpret_cast<const int4*>(p.tiles + ti * 8);
  const int4 a = __ldg(row), b = __ldg(row + 1);
  Unit x;
  x.q_row0 = a.x;
  x.q_rows = a.y;
  x.kv_row0 = a.z;
  x.kv_len = a.w;
  x.blk = b.x;
  x.row_off = b.y;
  x.kvh = r / p.npairs;
  const int pair = r - x.kvh * p.npairs;
  x.h0 = x.kvh * p.group + 2 * pair;
  x.valid1 = 2 * pair + 1 < p.group;
  x.ntiles_kv = (x.kv_len + kTile - 1) / kTile;
  return x;
}

// Static snake schedule over the heaviest-first unit list.
__device__ __forceinline__ long long unit_index(long long k, int cta, int nctas) {
  const long long round = k / 1;  // one unit per CTA per round
  return round * nctas + ((round & 1) ? (nctas - 1 - cta) : cta);
}

// Bounded wait used only while tearing down after an abort (ignores the abort flag).
__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity) {
  const uint32_t a = smem_u32(bar);
  const long long t0 = clock64();
  while (!mbar_try_wait(a, parity)) {
    if (clock64() - t0 > kWaitBudgetClocks / 4) break;
  }
}

// Document holding token `start`: the d < n with cu[d] <= start < cu[d + 1].
// A 32-way search by the whole warp: each step the lanes probe 32 evenly
// spaced offsets of [lo, hi) and keep the span after the last one that is
// <= start, so n documents take ceil(log32 n) steps.
__device__ __forceinline__ int doc_at(const int32_t* __restrict__ cu, int n, int start, int lane) {
  int lo = 0, hi = n;  // cu[lo] <= start < cu[hi]
  while (hi - lo > 1) {
    const int step = (hi - lo + 31) >> 5;
    const int idx = lo + lane * step;
    const unsigned le = __ballot_sync(0xffffffffu, idx < hi && __ldg(cu + idx) <= start);
    lo += (31 - __clz(le)) * step;  // lane 0 probes lo itself, so le != 0
    hi = min(hi, lo + step);
  }
  return lo;
}

// SPLIT is a template argument, not a run-time flag, so the FUSED code carries
// no SPLIT state or branches (its softmax warps stay free of register spills).
template <int D, bool SPLIT>
__global__ void __launch_bounds__(kThreads, 1)
    k_attn_fwd(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
               const __grid_constant__ CUtensorMap tmV, const Params p) {
  using L = SmemLayout<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  Bars& bars = *reinterpret_cast<Bars*>(smem + L::kBar);
  volatile int* abort_word = &bars.abort_word;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  const long long total_units = p.ntiles * p.hkv * p.npairs;
  const int cta = blockIdx.x, nctas = gridDim.x;

  if (threadIdx.x == 0) {
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bars.q_full[s], 1);
      mbar_init(&bars.q_empty[s], 1);
      mbar_init(&bars.kv_full[s], 1);
      mbar_init(&bars.kv_empty[s], 1);
      mbar_init(&bars.s_full[s], 1);
      mbar_init(&bars.p_full[s], 4);  // one arrive per softmax warp
      mbar_init(&bars.o_full[s], 1);  // completes once per unit (its last P.V)
      mbar_init(&bars.o_empty[s], 4);
    }
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&bars.k_empty[s], 1);
      mbar_init(&bars.v_empty[s], 1);
    }
    mbar_init(&bars.drain, 1);
    bars.abort_word = 0;
    bars.pace_entry = 0;
    bars.pace_limit = 0;
    bars.pace_done = 0;
    fence_mbarrier_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(&bars.tmem_base, 512);
    tmem_relinquish();
  }
  if (warp == kProducerWarp && lane == 0) {
    prefetch_tmap(&tmQ);
    prefetch_tmap(&tmK);
    prefetch_tmap(&tmV);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars.tmem_base;
  // TMEM columns: S0 [0,128) S1 [128,256) O0 [256,256+D) O1 [256+D,256+2D); P_s aliases S_s[0,64)
  auto tS = [tmem](int slot) { return tmem + static_cast<uint32_t>(slot) * 128u; };
  auto tO = [tmem](int slot) { return tmem + 256u + static_cast<uint32_t>(slot) * D; };

  if (warp >= 8) {
  // control warpgroup: give registers back first, then split into roles
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kControlRegs));
  if (warp == kProducerWarp) {
    // ------------------------------------------------------------ TMA producer
    // Per unit: Q of both slots, then TMA groups {K(0)}, {V(0), K(1)}, ...,
    // {V(n-1)}; group j+1 is what the MMA thread needs for its tile-j step
    // (P.V(j) then S = Q K(j+1)^T), so one wait covers both operands.
    if (lane == 0) {
      uint32_t q_uses[2] = {0, 0};
      uint32_t gcount[2] = {0, 0};  // groups armed per kv_full barrier
      long long kload = 0, vload = 0, g = 0;
      bool ok = true;
      auto arm_group = [&](const Unit& x, int kj, int vj) -> bool {
        // kj / vj < 0: no K / V tile in this group
        if (kj >= 0) {
          const long long round = kload / kStages;
          if (round > 0 &&
              !mbar_wait(&bars.k_empty[kload % kStages], (round - 1) & 1, abort_word, p.err, kErrKEmpty,
                         p.wait_budget))
            return false;
        }
        if (vj >= 0) {
          const long long round = vload / kStages;
          if (round > 0 &&
              !mbar_wait(&bars.v_empty[vload % kStages], (round - 1) & 1, abort_word, p.err, kErrVEmpty,
                         p.wait_budget))
            return false;
        }
        // A group barrier is re-armed only after the MMA thread has consumed
        // its previous phase (group g-2).  Free K/V stages do not imply that,
        // and re-arming earlier could complete two phases before the MMA thread
        // looks, which it would then miss.
        uint64_t* bar = &bars.kv_full[g & 1];
        if (g >= 2 && !mbar_wait(&bars.kv_empty[g & 1], ((g >> 1) - 1) & 1, abort_word, p.err, kErrKvEmpty,
                                 p.wait_budget))
          return false;
        mbar_arrive_expect_tx(bar, (kj >= 0 ? L::kTileBytes : 0) + (vj >= 0 ? L::kTileBytes : 0));
        if (kj >= 0) {
          uint8_t* dst = smem + L::kK + (kload % kStages) * L::kTileBytes;
#pragma unroll
          for (int hb = 0; hb < D / 64; ++hb)
            tma_load_3d(dst + hb * L::kHalfBytes, &tmK, bar, hb * 64, x.kvh, x.kv_row0 + kj * kTile);
          ++kload;
        }
        if (vj >= 0) {
          uint8_t* dst = smem + L::kV + (vload % kStages) * L::kTileBytes;
#pragma unroll
          for (int hb = 0; hb < D / 64; ++hb)
            tma_load_3d(dst + hb * L::kHalfBytes, &tmV, bar, hb * 64, x.kvh, x.kv_row0 + vj * kTile);
          ++vload;
        }
        ++gcount[g & 1];
        ++g;
        return true;
      };
      for (long long k = 0; ok; ++k) {
        const long long u = unit_index(k, cta, nctas);
        if (u >= total_units) break;
        const Unit x = load_unit(p, u);
        for (int s = 0; s < 2 && ok; ++s) {
          if (s == 1 && !x.valid1) continue;
          if (q_uses[s] > 0)
            ok = mbar_wait(&bars.q_empty[s], (q_uses[s] - 1) & 1, abort_word, p.err, kErrQEmpty, p.wait_budget);
          if (!ok) break;
          ++q_uses[s];
          uint8_t* dst = smem + L::kQ + s * L::kTileBytes;
          mbar_arrive_expect_tx(&bars.q_full[s], L::kTileBytes);
#pragma unroll
          for (int hb = 0; hb < D / 64; ++hb)
            tma_load_3d(dst + hb * L::kHalfBytes, &tmQ, &bars.q_full[s], hb * 64, x.h0 + s, x.q_row0);
        }
        // K/V stream of this unit: CTAs on the same stream read the same K/V
        // tiles.  A published position is stream hash (bits 63-32) | launch
        // epoch (31-24) | key tile (23-0, kPaceDone once the unit is done).
        const uint32_t stream = (static_cast<uint32_t>(x.kv_row0) * 2654435761u) ^ (static_cast<uint32_t>(x.kvh) + 1u);
        const unsigned long long tag = (static_cast<unsigned long long>(stream) << 32) | ((p.pace_epoch & 0xFFu) << 24);
        if (ok) ok = arm_group(x, 0, -1);
        for (int j = 0; j < x.ntiles_kv && ok; ++j) {
          if (p.pace && (j % kPaceEvery) == 0) {
            const unsigned long long e = tag | static_cast<unsigned int>(j);
            *reinterpret_cast<volatile unsigned long long*>(p.pace + cta) = e;
            *reinterpret_cast<volatile unsigned long long*>(&bars.pace_entry) = e;
            // hold K(j+1) until the slowest CTA on this stream is within the window
            const long long t0 = clock64();
            for (;;) {
              const unsigned long long lim = *reinterpret_cast<volatile unsigned long long*>(&bars.pace_limit);
              if (static_cast<uint32_t>(lim >> 32) != stream || static_cast<unsigned int>(j) <= static_cast<unsigned int>(lim & 0xFFFFFFu))
                break;
              if (clock64() - t0 > p.wait_budget / 256 || *abort_word) break;  // advisory: give up and go on
              __nanosleep(128);
            }
          }
          ok = arm_group(x, j + 1 < x.ntiles_kv ? j + 1 : -1, j);
        }
        if (p.pace) {
          const unsigned long long e = tag | kPaceDone;
          *reinterpret_cast<volatile unsigned long long*>(p.pace + cta) = e;
          *reinterpret_cast<volatile unsigned long long*>(&bars.pace_entry) = e;
        }
      }
      *reinterpret_cast<volatile int*>(&bars.pace_done) = 1;
      // Drain: every armed barrier's last phase completes once its bytes
      // land, so no copy into this CTA's shared memory is still in flight when
      // it exits, also when another role gave up after this loop ended.  In a
      // normal run these phases completed long ago and each wait returns at
      // its first poll.
      for (int b = 0; b < 2; ++b)
        if (gcount[b] > 0) drain_wait(&bars.kv_full[b], (gcount[b] - 1) & 1);
      for (int s = 0; s < 2; ++s)
        if (q_uses[s] > 0) drain_wait(&bars.q_full[s], (q_uses[s] - 1) & 1);
    }
    __syncwarp();
    tc_fence_before();
    named_barrier_sync(1, kThreads);
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    // Per key tile j: for each slot P.V(j) followed at once by S = Q K(j+1)^T.
    // S(j+1) of a slot overwrites the TMEM columns that P(j) of the same slot
    // occupies; one thread issues the two back to back and they execute in
    // issue order.
    //
    // The tensor core's queue holds only about two MMAs, so every cycle the
    // issuing thread spends between two slots' MMA groups can leave it idle.
    // The thread therefore does the few waits its MMAs depend on itself, at
    // the group boundaries where it has nothing else to issue: the TMA group
    // holding V(j) and K(j+1), the slot's P(j), and (first tile of a unit)
    // the previous epilogue's read of O.  Each is one try-wait when already
    // complete; a cross-warp hand-off here cost about 250 cycles a slot.
    if (lane == 0) {
      constexpr uint32_t idesc_qk = idesc_bf16_f32(128, 128, 0);
      constexpr uint32_t idesc_pv = idesc_bf16_f32(128, D, 1);
      // Descriptors: base per buffer; K steps add compile-time offsets to the
      // start-address field (addresses stay below 256 KB, so no carry).
      const uint64_t dQ = sdesc_sw128(smem_u32(smem + L::kQ), 16, 1024);
      const uint64_t dK = sdesc_sw128(smem_u32(smem + L::kK), 16, 1024);
      const uint64_t dV = sdesc_sw128(smem_u32(smem + L::kV), L::kHalfBytes, 1024);
      constexpr uint64_t kTileUnits = L::kTileBytes >> 4;
      const uint64_t dK1 = dK + kTileUnits, dV1 = dV + kTileUnits;
      auto issue_qk = [&](int s, int kst) {
        const uint64_t qd = dQ + s * kTileUnits, kd = kst ? dK1 : dK;
        umma_ss_c<false>(tS(s), qd, kd, idesc_qk);
  #pragma unroll
        for (int kk = 1; kk < D / 16; ++kk) {
          const uint64_t off = static_cast<uint64_t>((kk >> 2) * L::kHalfBytes + (kk & 3) * 32) >> 4;
          umma_ss_c<true>(tS(s), qd + off, kd + off, idesc_qk);
        }
        umma_commit(&bars.s_full[s]);
      };
      auto issue_pv = [&](int s, int vst, bool accumulate) {
        const uint64_t vd = vst ? dV1 : dV;
        if (accumulate)
          umma_ts_c<true>(tO(s), tS(s), vd, idesc_pv);
        else
          umma_ts_c<false>(tO(s), tS(s), vd, idesc_pv);
  #pragma unroll
        for (int kk = 1; kk < kTile / 16; ++kk)
          umma_ts_c<true>(tO(s), tS(s) + kk * 8, vd + static_cast<uint64_t>(kk * 2048 >> 4), idesc_pv);
      };
      uint32_t q_uses[2] = {0, 0}, p_uses[2] = {0, 0}, units_done[2] = {0, 0};  // units_done: epilogues
      long long g = 0;
      bool ok = true;  // every wait so far succeeded
      auto wait_on = [&](uint64_t* bar, uint32_t parity, int code) {
        if (ok) ok = mbar_wait(bar, parity, abort_word, p.err, code, p.wait_budget);
      };
      auto wait_group = [&](int code) {  // one TMA group; the producer may re-arm its barrier afterwards
        wait_on(&bars.kv_full[g & 1], (g >> 1) & 1, code);
        if (ok) mbar_arrive(&bars.kv_empty[g & 1]);
        ++g;
      };
      // K and V stages advance together (n of each per unit), so one parity c
      // per unit fixes them: P.V(j) reads V stage c ^ (j & 1), S(j+1) K stage
      // c ^ 1 ^ (j & 1).  The steady key tiles are unrolled by two with those
      // stages as constants, and the last two tiles are peeled, so the issuing
      // thread runs straight-line code: per-MMA index arithmetic or commit
      // branches cost it tens of cycles a MMA.
      // key tile j of the unit; kind 0: steady (j < n - 2), 1: j = n - 2 (Q is
      // free after its S), 2: j = n - 1 (the unit's last P.V)
      // first / last: key tile j opens / closes an epilogue's span (the unit,
      // or one C-key chunk in SPLIT); call sites pass constants
      // where they can, so steady tiles carry no span bookkeeping
      auto tile = [&](const Unit& x, int nslots, int j, int vs, int ks, int kind, bool first, bool last) -> bool {
        for (int s = 0; s < nslots; ++s) {
          if (s == 0) wait_group(kErrVFull);
          if (first && units_done[s] > 0) wait_on(&bars.o_empty[s], (units_done[s] - 1) & 1, kErrOEmpty);
          wait_on(&bars.p_full[s], p_uses[s] & 1, kErrPFull);  // P_s(j) written, O_s rescaled
          ++p_uses[s];
          if (!ok) return false;
          tc_fence_after();
          issue_pv(s, vs, !first);
          if (last) {
            umma_commit(&bars.o_full[s]);
            ++units_done[s];
          }
          if (kind != 2) {
            issue_qk(s, ks);
            if (kind == 1) umma_commit(&bars.q_empty[s]);
          }
        }
        if (kind != 2) umma_commit(&bars.k_empty[ks]);
        umma_commit(&bars.v_empty[vs]);
        return true;
      };
      bool alive = true;
      int c = 0;  // stage parity at the start of a unit
      for (long long k = 0; alive; ++k) {
        const long long u = unit_index(k, cta, nctas);
        if (u >= total_units) break;
        const Unit x = load_unit(p, u);
        const int nslots = x.valid1 ? 2 : 1;
        const int n = x.ntiles_kv;
        // Q of every slot and the group holding K(0)
        for (int s = 0; s < nslots; ++s) wait_on(&bars.q_full[s], q_uses[s] & 1, kErrQFull);
        for (int s = 0; s < nslots; ++s) ++q_uses[s];
        wait_group(kErrKFull);
        if (!ok) break;
        tc_fence_after();
        for (int s = 0; s < nslots; ++s) {
          issue_qk(s, c);
          if (n == 1) umma_commit(&bars.q_empty[s]);
        }
        umma_commit(&bars.k_empty[c]);
        int j = 0;
        if constexpr (SPLIT) {
          // span by span: the span's first tile, its steady middle (as in
          // FUSED: constant stages, no bookkeeping), then its last tile and
          // the unit's last two (kinds 1 and 2) with flags taken at run time
          auto kind_of = [n](int jj) { return jj == n - 1 ? 2 : (jj == n - 2 ? 1 : 0); };
          while (alive && j < n) {
            const int je = min(j + p.tpc, n);
            alive = tile(x, nslots, j, c ^ (j & 1), c ^ 1 ^ (j & 1), kind_of(j), true, j == je - 1);
            ++j;
            const int steady_end = min(je - 1, n - 2);
            if ((c ^ (j & 1)) == 0) {
              for (; j + 1 < steady_end && alive; j += 2)
                alive = tile(x, nslots, j, 0, 1, 0, false, false) && tile(x, nslots, j + 1, 1, 0, 0, false, false);
            } else {
              for (; j + 1 < steady_end && alive; j += 2)
                alive = tile(x, nslots, j, 1, 0, 0, false, false) && tile(x, nslots, j + 1, 0, 1, 0, false, false);
            }
            for (; j < steady_end && alive; ++j)
              alive = tile(x, nslots, j, c ^ (j & 1), c ^ 1 ^ (j & 1), 0, false, false);
            for (; j < je && alive; ++j)
              alive = tile(x, nslots, j, c ^ (j & 1), c ^ 1 ^ (j & 1), kind_of(j), false, j == je - 1);
          }
        } else {
          if (c == 0) {
            for (; j + 1 < n - 2 && alive; j += 2)
              alive = tile(x, nslots, j, 0, 1, 0, j == 0, false) && tile(x, nslots, j + 1, 1, 0, 0, false, false);
          } else {
            for (; j + 1 < n - 2 && alive; j += 2)
              alive = tile(x, nslots, j, 1, 0, 0, j == 0, false) && tile(x, nslots, j + 1, 0, 1, 0, false, false);
          }
          for (; j < n - 2 && alive; ++j) alive = tile(x, nslots, j, c ^ (j & 1), c ^ 1 ^ (j & 1), 0, j == 0, false);
          if (alive && n >= 2) {
            alive = tile(x, nslots, j, c ^ (j & 1), c ^ 1 ^ (j & 1), 1, j == 0, false);
            ++j;
          }
          if (alive) alive = tile(x, nslots, j, c ^ (j & 1), 0, 2, j == 0, true);
        }
        if (!alive) break;
        c ^= n & 1;
      }
      // drain every MMA this thread issued before TMEM is released
      umma_commit(&bars.drain);
      drain_wait(&bars.drain, 0);
    }
    __syncwarp();
    tc_fence_before();
    named_barrier_sync(1, kThreads);  // every role is done with TMEM
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  } else {
    if (warp == kPacerWarp && p.pace) {
      // ---------------------------------------------------------- pacer
      // Publishes, for this CTA's producer, the furthest key tile it may load:
      // the least position among the CTAs of this launch on the same K/V
      // stream, plus the window.  Ends with the producer, on an abort, or when
      // this CTA's position has not moved for a whole wait budget.
      // Lane 0 takes every decision and the warp follows it, so the whole warp
      // reaches each shuffle and reduction together.
      unsigned long long last = 0;
      long long last_change = clock64();
      for (;;) {
        int stop = 0;
        unsigned long long me = 0;
        if (lane == 0) {
          me = *reinterpret_cast<volatile unsigned long long*>(&bars.pace_entry);
          stop = *reinterpret_cast<volatile int*>(&bars.pace_done) || *abort_word;
          if (me != last) {
            last = me;
            last_change = clock64();
          } else if (clock64() - last_change > p.wait_budget) {
            stop = 1;
          }
        }
        stop = __shfl_sync(0xffffffffu, stop, 0);
        me = __shfl_sync(0xffffffffu, me, 0);
        if (stop) break;
        if (me != 0) {
          const unsigned long long tag = me & ~0xFFFFFFull;
          unsigned int mn = kPaceDone;
          for (int i = lane; i < nctas; i += 32) {
            const unsigned long long e = *reinterpret_cast<volatile unsigned long long*>(p.pace + i);
            if ((e & ~0xFFFFFFull) == tag) mn = min(mn, static_cast<unsigned int>(e & 0xFFFFFFu));
          }
          mn = __reduce_min_sync(0xffffffffu, mn);
          if (lane == 0) {
            const unsigned int lim = mn >= kPaceDone - kPaceWindow ? kPaceDone : mn + kPaceWindow;
            *reinterpret_cast<volatile unsigned long long*>(&bars.pace_limit) = (tag & ~0xFFFFFFFFull) | lim;
          }
        }
        __syncwarp();
        __nanosleep(256);
      }
    }
    named_barrier_sync(1, kThreads);  // the two idle warps of the control warpgroup
  }
  } else {
    // ------------------------------------------------------------ softmax + epilogue
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kSoftmaxRegs));
    const int s = warp >> 2;                 // slot
    const int row = (warp & 3) * 32 + lane;  // TMEM lane = tile row
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint64_t scale2 = pack_f32x2(p.scale_log2, p.scale_log2);
    uint32_t s_count = 0, units_done = 0;
    bool ok = true;
    for (long long k = 0; ok; ++k) {
      const long long u = unit_index(k, cta, nctas);
      if (u >= total_units) break;
      const Unit x = load_unit(p, u);
      if (s == 1 && !x.valid1) continue;
      const int h = x.h0 + s;
      // doc-local query position relative to the first key of the range
      const int q_rel = x.q_row0 - x.kv_row0 + row;
      const int key_limit = min(q_rel + 1, x.kv_len);  // keys [0, key_limit) are allowed
      // SPLIT: the tile's chunk qc, its block (qc, 0), its first row
      // in the chunk
      int blk0 = 0, row0c = 0;
      if constexpr (SPLIT) {
        const int doc = doc_at(p.cu, p.ndocs, x.kv_row0, lane);
        const int qc = x.row_off / p.C;
        blk0 = static_cast<int>(__ldg(p.bo + doc) + static_cast<long long>(qc) * (qc + 1) / 2);
        row0c = x.row_off - qc * p.C;
      }
      // key tiles in spans: the unit's whole range, or one C-key chunk in
      // SPLIT; each span ends in its own epilogue
      const int nspan = SPLIT ? (x.ntiles_kv + p.tpc - 1) / p.tpc : 1;
      for (int b = 0; b < nspan && ok; ++b) {
        const int j0 = SPLIT ? b * p.tpc : 0;
        const int j1 = SPLIT ? min(j0 + p.tpc, x.ntiles_kv) : x.ntiles_kv;
        float m = -INFINITY, l = 0.f;
        for (int j = j0; j < j1 && ok; ++j) {
          const bool first = j == j0;
          ok = __all_sync(0xffffffffu,
                          mbar_wait(&bars.s_full[s], s_count & 1, abort_word, p.err, kErrSFull, p.wait_budget));
          if (!ok) break;
          ++s_count;
          tc_fence_after();
          const int lim = key_limit - j * kTile;  // allowed keys of this tile: [0, lim)
          uint32_t r[4][32];
          float mc[4];
          bool rescale_o = false;
          float alpha = 1.f;
          // p = 2^(s*scale*log2e - m) for one 32-column chunk: four packed
          // partial row sums, P packed to bf16 pairs and stored into the first
          // 64 columns of S (chunk c's keys land in columns [16c, 16c + 16)).
          auto exp_chunk = [&](int c, uint64_t negm2, uint64_t (&acc)[4]) {
            uint32_t pk[16];
#pragma unroll
            for (int i = 0; i < 32; i += 2) {
              const uint64_t t = ffma_f32x2(pack_f32x2(__uint_as_float(r[c][i]), __uint_as_float(r[c][i + 1])),
                                            scale2, negm2);
              const float p0 = ex2_approx(lo_f32(t));
              const float p1 = ex2_approx(hi_f32(t));
              acc[(i >> 1) & 3] = fadd_f32x2(acc[(i >> 1) & 3], pack_f32x2(p0, p1));
              pk[i / 2] = pack_bf16x2(p0, p1);
            }
            tmem_st16(tS(s) + lane_off + c * 16, pk);
          };
          auto row_sum = [](uint64_t (&acc)[4]) {
            const uint64_t a = fadd_f32x2(fadd_f32x2(acc[0], acc[1]), fadd_f32x2(acc[2], acc[3]));
            return lo_f32(a) + hi_f32(a);
          };
          if (__all_sync(0xffffffffu, !first && lim >= kTile)) {
            // Steady tile (no mask, running max known): each chunk's exponentials
            // are computed with the running max while the next chunk's load is
            // in flight; a chunk's P only overwrites S columns already loaded.
            // The row maxima come from the loads themselves.  If one of them
            // exceeds the running max by more than the threshold, the tile is
            // recomputed from the registers with the new max (rare).
            const uint64_t negm2 = pack_f32x2(-m, -m);
            uint64_t acc[4] = {0, 0, 0, 0};
            mc[0] = tmem_ld32_max(tS(s) + lane_off, r[0]);
            tmem_wait_ld();
#pragma unroll
            for (int c = 0; c < 4; ++c) {
              if (c < 3) mc[c + 1] = tmem_ld32_max(tS(s) + lane_off + (c + 1) * 32, r[c + 1]);
              exp_chunk(c, negm2, acc);
              if (c < 3) tmem_wait_ld();
            }
            const float mt_scaled = fmax3(fmaxf(mc[0], mc[1]), mc[2], mc[3]) * p.scale_log2;
            const bool grow = mt_scaled > m + kRescaleThreshold;
            if (__any_sync(0xffffffffu, grow)) {
              if (grow) {
                alpha = ex2_approx(m - mt_scaled);
                l *= alpha;
                m = mt_scaled;
                rescale_o = true;
              }
              tmem_wait_st();  // the first pass's stores land before they are overwritten
              const uint64_t negm2n = pack_f32x2(-m, -m);
              uint64_t acc2[4] = {0, 0, 0, 0};
#pragma unroll
              for (int c = 0; c < 4; ++c) exp_chunk(c, negm2n, acc2);
              l += row_sum(acc2);
            } else {
              l += row_sum(acc);
            }
          } else {
            // first tile, or a tile crossing the diagonal or the end of the key
            // range: load the whole row, mask, take the maximum over the allowed
            // keys, then the exponentials
#pragma unroll
            for (int c = 0; c < 4; ++c) mc[c] = tmem_ld32_max(tS(s) + lane_off + c * 32, r[c]);
            tmem_wait_ld();
            if (lim < kTile) {
#pragma unroll
              for (int c = 0; c < 4; ++c)
#pragma unroll
                for (int i = 0; i < 32; ++i)
                  if (c * 32 + i >= lim) r[c][i] = __float_as_uint(-INFINITY);
#pragma unroll
              for (int c = 0; c < 4; ++c) {
                mc[c] = __uint_as_float(r[c][0]);
#pragma unroll
                for (int i = 1; i < 31; i += 2)
                  mc[c] = fmax3(mc[c], __uint_as_float(r[c][i]), __uint_as_float(r[c][i + 1]));
                mc[c] = fmaxf(mc[c], __uint_as_float(r[c][31]));
              }
            }
            const float mt_scaled = fmax3(fmaxf(mc[0], mc[1]), mc[2], mc[3]) * p.scale_log2;
            if (mt_scaled > m + kRescaleThreshold || first) {
              const float m_new = fmaxf(m, mt_scaled);
              alpha = first ? 0.f : ex2_approx(m - m_new);
              l *= alpha;
              m = m_new;
              rescale_o = !first;
            }
            const uint64_t negm2 = pack_f32x2(-m, -m);
            uint64_t acc[4] = {0, 0, 0, 0};
#pragma unroll
            for (int c = 0; c < 4; ++c) exp_chunk(c, negm2, acc);
            l += row_sum(acc);
          }
          if (__any_sync(0xffffffffu, rescale_o)) {
            // P.V of tile j-1 is complete: S_s(j) was committed after it
#pragma unroll 1
            for (int c = 0; c < D / 32; ++c) {
              uint32_t o[32];
              tmem_ld32(tO(s) + lane_off + c * 32, o);
              tmem_wait_ld();
#pragma unroll
              for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
              tmem_st32(tO(s) + lane_off + c * 32, o);
            }
          }
          tmem_wait_st();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&bars.p_full[s]);
        }
        if (!ok) break;
        // ---- epilogue: wait for the span's last P.V, normalize, store
          if (!__all_sync(0xffffffffu, mbar_wait(&bars.o_full[s], units_done & 1, abort_word, p.err, kErrOFull,
                                                 p.wait_budget))) {
            ok = false;
            break;
          }
          tc_fence_after();
          const bool row_valid = row < x.q_rows;
          const float inv_l = 1.f / l;
          const float lse_val = (m + __log2f(l)) * 0.69314718055994530942f;
          const long long tok = static_cast<long long>(x.q_row0) + row;
          if constexpr (!SPLIT) {
            __nv_bfloat16* dst = p.o + (tok * p.hq + h) * static_cast<long long>(D);
#pragma unroll 1
            for (int c = 0; c < D / 32; ++c) {
              uint32_t o[32];
              tmem_ld32(tO(s) + lane_off + c * 32, o);
              tmem_wait_ld();
              if (row_valid) {
                uint4 w[4];
                uint32_t* wp = reinterpret_cast<uint32_t*>(w);
#pragma unroll
                for (int i = 0; i < 16; ++i)
                  wp[i] = pack_bf16x2(__uint_as_float(o[2 * i]) * inv_l, __uint_as_float(o[2 * i + 1]) * inv_l);
                uint4* d4 = reinterpret_cast<uint4*>(dst + c * 32);
#pragma unroll
                for (int i = 0; i < 4; ++i) d4[i] = w[i];
              }
            }
            if (row_valid) p.lse[static_cast<long long>(h) * p.T + tok] = lse_val;
          } else {
            const int blk = blk0 + b;
            const long long prow = static_cast<long long>(blk) * p.C + row0c + row;
            float* dst = p.o_part + (prow * p.hq + h) * static_cast<long long>(D);
#pragma unroll 1
            for (int c = 0; c < D / 32; ++c) {
              uint32_t o[32];
              tmem_ld32(tO(s) + lane_off + c * 32, o);
              tmem_wait_ld();
              if (row_valid) {
                float4* d4 = reinterpret_cast<float4*>(dst + c * 32);
#pragma unroll
                for (int i = 0; i < 8; ++i)
                  d4[i] = make_float4(__uint_as_float(o[4 * i]) * inv_l, __uint_as_float(o[4 * i + 1]) * inv_l,
                                      __uint_as_float(o[4 * i + 2]) * inv_l, __uint_as_float(o[4 * i + 3]) * inv_l);
              }
            }
            if (row_valid) p.lse_part[(static_cast<long long>(blk) * p.hq + h) * p.C + row0c + row] = lse_val;
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&bars.o_empty[s]);
          ++units_done;
      }
      if (!ok) break;
    }
    tc_fence_before();
    named_barrier_sync(1, kThreads);
  }
}

// ---------------------------------------------------------------- host side
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(f);
  });
  return fn;
}

// [T][heads][d] bf16 viewed as a 3-D tensor (d, heads, T); box = 64 columns x
// 1 head x 128 rows, 128-byte swizzle (the canonical K-major SW128 layout).
hdp_status_t make_map(CUtensorMap* m, const void* base, long long T, int heads, int d) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return fail(HDP_ERR_CUDA, "cuTensorMapEncodeTiled is unavailable");
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(heads), static_cast<cuuint64_t>(T)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 2, static_cast<cuuint64_t>(heads) * d * 2};
  cuuint32_t box[3] = {64, 1, static_cast<cuuint32_t>(kTile)};
  cuuint32_t es[3] = {1, 1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, es,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(HDP_ERR_CUDA, "cuTensorMapEncodeTiled failed (" + std::to_string(r) + ")");
  return HDP_OK;
}

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

}  // namespace

// Shared with the backward pass: the same tile map for any [T][heads][d] bf16 tensor.
hdp_status_t make_bf16_tile_map(CUtensorMap* m, const void* base, long long T, int heads, int d) {
  return make_map(m, base, T, heads, d);
}


namespace {

// Pacing table of a device and the launch epochs, shared by every launch of
// the library (both head sizes, all threads).  The table's address is
// resolved once per device, on the first paced launch with that device
// current; devices past the cache run unpaced.
std::mutex g_pace_mu;
unsigned long long* g_pace_ptr[64] = {nullptr};
std::atomic<unsigned int> g_pace_epoch{0};

hdp_status_t pace_table(int dev, unsigned long long** out) {
  *out = nullptr;
  if (dev < 0 || dev >= 64) return HDP_OK;
  std::lock_guard<std::mutex> lk(g_pace_mu);
  if (!g_pace_ptr[dev]) {
    void* a = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&a, g_pace);
    if (e != cudaSuccess) return fail_cuda(e, "cudaGetSymbolAddress(g_pace)");
    g_pace_ptr[dev] = static_cast<unsigned long long*>(a);
  }
  *out = g_pace_ptr[dev];
  return HDP_OK;
}

template <int D>
hdp_status_t launch(const hdp_plan_s* plan, const void* q, const void* k, const void* v, int hq, int hkv,
                    float scale, bool split, float* o_part, float* lse_part, void* o, float* lse, cudaStream_t st) {
  const long long T = plan->v.total_tokens;
  CUtensorMap mq, mk, mv;
  hdp_status_t r;
  if ((r = make_map(&mq, q, T, hq, D)) != HDP_OK) return r;
  if ((r = make_map(&mk, k, T, hkv, D)) != HDP_OK) return r;
  if ((r = make_map(&mv, v, T, hkv, D)) != HDP_OK) return r;
  // SPLIT walks the same fused units as FUSED.  Pacing when one head's K and
  // V rows of the longest document exceed L2 (they no longer stay in L2 for
  // a whole round on their own).
  int dev = 0, sms = 0, l2 = 0;
  HDP_CUDA_TRY(cudaGetDevice(&dev));
  HDP_CUDA_TRY(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
  HDP_CUDA_TRY(cudaDeviceGetAttribute(&l2, cudaDevAttrL2CacheSize, dev));
  const long long kv_head_bytes = 2LL * plan->v.max_doc_len * D * 2;
  const bool pace = kv_head_bytes > l2;
  Params prm{};
  prm.tiles = plan->v.tiles_fused;
  prm.ntiles = plan->v.num_tiles_fused;
  prm.hq = hq;
  prm.hkv = hkv;
  prm.group = hq / hkv;
  prm.npairs = (prm.group + 1) / 2;
  prm.scale_log2 = scale * 1.4426950408889634f;
  prm.T = T;
  prm.o = static_cast<__nv_bfloat16*>(o);
  prm.lse = lse;
  prm.o_part = o_part;
  prm.lse_part = lse_part;
  prm.C = plan->v.capacity;
  prm.tpc = plan->v.capacity / kTile;
  prm.ndocs = plan->v.num_docs;
  prm.cu = plan->v.cu_seqlens;
  prm.bo = plan->v.block_offsets;
  prm.err = device_error_word();
  if (!prm.err) return fail(HDP_ERR_CUDA, "cannot resolve the device error word");
  prm.wait_budget = wait_budget_clocks();
  prm.pace = nullptr;
  if (pace) {
    hdp_status_t pr = pace_table(dev, &prm.pace);
    if (pr != HDP_OK) return pr;
    prm.pace_epoch = g_pace_epoch.fetch_add(1) % 255u + 1u;  // never 0: zeroed slots match no launch
  }
  const long long units = prm.ntiles * hkv * prm.npairs;
  if (units == 0) return HDP_OK;
  const int grid = static_cast<int>(units < sms ? units : sms);
  if (grid > 1024) prm.pace = nullptr;
  const long long bt = grid / (prm.npairs * heads_per_round(plan->v.max_doc_len, hkv));
  prm.block_tiles = bt > 0 ? bt : 1;
  const int smem = SmemLayout<D>::kBytes + 1024;
  auto kernel = split ? k_attn_fwd<D, true> : k_attn_fwd<D, false>;
  HDP_CUDA_TRY(cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem));
  kernel<<<grid, kThreads, smem, st>>>(mq, mk, mv, prm);
  note_launch();
  HDP_CUDA_TRY(cudaGetLastError());
  return HDP_OK;
}

hdp_status_t split_workspace(const hdp_plan_s* plan, int hq, int d, size_t* o_bytes, size_t* total) {
  const size_t rows = static_cast<size_t>(plan->v.num_blocks) * plan->v.capacity;
  *o_bytes = align256(rows * hq * d * sizeof(float));
  *total = *o_bytes + align256(rows * hq * sizeof(float));
  return HDP_OK;
}

}  // namespace
}  // namespace hdp

using namespace hdp;

extern "C" hdp_status_t hdp_attention_workspace_bytes(hdp_plan_t plan, int32_t hq, int32_t d, int32_t mode,
                                                      size_t* bytes) {
  if (!plan || !bytes) return fail(HDP_ERR_INVALID_ARGUMENT, "hdp_attention_workspace_bytes: NULL argument");
  if (hq < 1 || d < 1) return fail(HDP_ERR_INVALID_ARGUMENT, "hdp_attention_workspace_bytes: hq, d must be >= 1");
  if (mode == HDP_MODE_FUSED) {
    *bytes = 0;
    return HDP_OK;
  }
  if (mode != HDP_MODE_SPLIT) return fail(HDP_ERR_INVALID_ARGUMENT, "hdp_attention_workspace_bytes: unknown mode");
  size_t ob = 0;
  return split_workspace(plan, hq, d, &ob, bytes);
}

extern "C" hdp_status_t hdp_attention_fwd(hdp_plan_t plan, const void* q, const void* k, const void* v, int32_t hq,
                                          int32_t hkv, int32_t d, float scale, int32_t mode, void* workspace,
                                          size_t workspace_bytes, void* o, float* lse, void* stream) {
  if (!plan || !q || !k || !v || !o || !lse) return fail(HDP_ERR_INVALID_ARGUMENT, "hdp_attention_fwd: NULL argument");
  if (hq < 1 || hkv < 1 || hq % hkv != 0)
    return fail(HDP_ERR_INVALID_ARGUMENT, "hdp_attention_fwd: need hq >= 1, hkv >= 1, hq % hkv == 0");
  if (!(scale > 0.f)) return fail(HDP_ERR_INVALID_ARGUMENT, "hdp_attention_fwd: scale must be > 0");
  if (mode != HDP_MODE_FUSED && mode != HDP_MODE_SPLIT)
    return fail(HDP_ERR_INVALID_ARGUMENT, "hdp_attention_fwd: unknown mode");
  if (d != 64 && d != 128) return fail(HDP_ERR_UNSUPPORTED, "hdp_attention_fwd: d must be 64 or 128");
  const uintptr_t mis = reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k) |
                        reinterpret_cast<uintptr_t>(v) | reinterpret_cast<uintptr_t>(o);
  if (mis & 15) return fail(HDP_ERR_INVALID_ARGUMENT, "hdp_attention_fwd: q, k, v, o must be 16-byte aligned");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const bool split = mode == HDP_MODE_SPLIT;
  float* o_part = nullptr;
  float* lse_part = nullptr;
  if (split) {
    if (plan->v.capacity % kTile != 0)
      return fail(HDP_ERR_INVALID_ARGUMENT, "hdp_attention_fwd: SPLIT needs capacity % 128 == 0");
    size_t ob = 0, need = 0;
    split_workspace(plan, hq, d, &ob, &need);
    if (!workspace || workspace_bytes < need)
      return fail(HDP_ERR_INVALID_ARGUMENT, "hdp_attention_fwd: SPLIT workspace too small (need " +
                                                std::to_string(need) + " bytes)");
    if (reinterpret_cast<uintptr_t>(workspace) & 255)
      return fail(HDP_ERR_INVALID_ARGUMENT, "hdp_attention_fwd: workspace must be 256-byte aligned");
    o_part = static_cast<float*>(workspace);
    lse_part = reinterpret_cast<float*>(static_cast<char*>(workspace) + ob);
  }
  hdp_status_t r = d == 128 ? launch<128>(plan, q, k, v, hq, hkv, scale, split, o_part, lse_part, o, lse, st)
                            : launch<64>(plan, q, k, v, hq, hkv, scale, split, o_part, lse_part, o, lse, st);
  if (r != HDP_OK || !split) return r;
  return launch_merge_blocks(plan, o_part, lse_part, hq, d, o, lse, st);
}

// ---------------------------------------------------------------- SPLIT without allocation
// Some callers cannot allocate device memory when they run attention:
// serving processes that reserve all device memory at start-up and forbid
// allocation on the request path, host programs whose own allocator owns the
// device memory, and callers that must not take the device-wide
// synchronisation cudaMalloc/cudaFree may imply.  For them SPLIT mode can use
// a fixed scratch array that is part of the library image instead of a
// caller-provided workspace.
namespace hdp {
namespace {

// Largest SPLIT workspace (partial O and LSE of every causal block) the
// static area holds; each GPU that loads the library reserves it until exit.
constexpr size_t kStaticSplitScratchBytes = size_t(64) << 20;
static __device__ __align__(256) unsigned char g_split_scratch[kStaticSplitScratchBytes];

std::mutex g_scratch_mu;
void* g_scratch_ptr[64] = {nullptr};

// Device address of g_split_scratch on the current device.  Resolved once per
// device, on the first call made with that device current.
hdp_status_t static_scratch(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail_cuda(e, "cudaGetDevice");
  if (dev < 0 || dev >= 64) return fail(HDP_ERR_UNSUPPORTED, "device index out of range for the static scratch");
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_split_scratch);
    if (e != cudaSuccess) return fail_cuda(e, "cudaGetSymbolAddress(g_split_scratch)");
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return HDP_OK;
}

}  // namespace
}  // namespace hdp

extern "C" hdp_status_t hdp_attention_fwd_split_noalloc(hdp_plan_t plan, const void* q, const void* k,
                                                        const void* v, int32_t hq, int32_t hkv, int32_t d,
                                                        float scale, void* o, float* lse, void* stream) {
  if (!plan) return fail(HDP_ERR_INVALID_ARGUMENT, "hdp_attention_fwd_split_noalloc: plan is NULL");
  if (hq < 1 || d < 1) return fail(HDP_ERR_INVALID_ARGUMENT, "hdp_attention_fwd_split_noalloc: hq, d must be >= 1");
  size_t ob = 0, need = 0;
  split_workspace(plan, hq, d, &ob, &need);
  if (need > kStaticSplitScratchBytes)
    return fail(HDP_ERR_INVALID_ARGUMENT,
                "hdp_attention_fwd_split_noalloc: this plan needs " + std::to_string(need) +
                    " bytes of SPLIT scratch, more than the static maximum of " +
                    std::to_string(kStaticSplitScratchBytes) + " bytes; use hdp_attention_fwd with a workspace");
  void* scratch = nullptr;
  hdp_status_t r = static_scratch(&scratch);
  if (r != HDP_OK) return r;
  return hdp_attention_fwd(plan, q, k, v, hq, hkv, d, scale, HDP_MODE_SPLIT, scratch, kStaticSplitScratchBytes, o,
                           lse, stream);
}
