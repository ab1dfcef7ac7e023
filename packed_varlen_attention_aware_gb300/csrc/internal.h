// Internal declarations shared by the library's translation units.
#pragma once
#include <cuda_runtime.h>

#include <cstdint>
#include <string>

#include "../../include/hdpattn.h"

namespace hdp {

constexpr int kTile = 128;             // query/key rows per attention tile
constexpr int64_t kMaxPieces = 65536;  // best-fit packing limit (sub-capacity pieces)

// Record a thread-local error message and return `st`.
hdp_status_t fail(hdp_status_t st, const std::string& msg);
hdp_status_t fail_cuda(cudaError_t e, const char* what);
#define HDP_CUDA_TRY(expr)                          \
  do {                                              \
    cudaError_t e_ = (expr);                        \
    if (e_ != cudaSuccess) return ::hdp::fail_cuda(e_, #expr); \
  } while (0)

// KV heads whose units share one round of a persistent attention grid.  One
// head per round makes the CTAs of a round stream the same head's tiles at
// about the same time (L2 reuse), which pays on long documents, whose causal
// prefixes outgrow the L2; with many short documents it would put units of
// very different sizes into one round, so every head takes part in each round
// there.  `max_doc_len` is the plan's longest document.
inline int heads_per_round(long long max_doc_len, int hkv) { return max_doc_len >= 65536 ? 1 : hkv; }

// Device error word shared by all kernels (bounded-wait timeouts, internal
// consistency checks).  Defined in api.cu; read by hdp_device_status.
unsigned int* device_error_word();

// Count one kernel enqueued by this library (reported by hdp_kernel_launch_count).
void note_launch();
// Count one host wait on a stream (reported by hdp_host_sync_count).
void note_host_sync();

// Budget, in SM clocks, of the attention forward's role waits (set by
// hdp_set_wait_budget; the default is about one second).
long long wait_budget_clocks();

}  // namespace hdp

struct hdp_plan_s {
  int device = 0;
  cudaStream_t stream = nullptr;
  uint32_t flags = 0;
  hdp_plan_view_t v{};
  void* mem = nullptr;   // stream-ordered allocation holding the N_c/N_b/tile-sized tables
  void* mem1 = nullptr;  // stream-ordered allocation holding the [n+1] offset arrays
  // internal tables (inside `mem`)
  const int64_t* tile_offsets_fused = nullptr;  // [n+1]
  const int64_t* tile_offsets_split = nullptr;  // [n+1]
};
