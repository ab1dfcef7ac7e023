// Status strings, thread-local error messages and the device error word.
#include <cuda_runtime.h>

#include <atomic>
#include <cstdio>
#include <mutex>
#include <string>

#include "internal.h"
#include "sm103_ptx.cuh"

namespace {
thread_local std::string g_last_error;
__device__ unsigned int g_device_error;  // 0 = ok, else a code from the kernels

std::mutex g_mu;
std::atomic<unsigned long long> g_launches{0};
std::atomic<unsigned long long> g_host_syncs{0};
std::atomic<long long> g_wait_budget{hdp::kWaitBudgetClocks};
unsigned int* g_err_ptr[64] = {nullptr};
}  // namespace

namespace hdp {

void note_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }
void note_host_sync() { g_host_syncs.fetch_add(1, std::memory_order_relaxed); }
long long wait_budget_clocks() { return g_wait_budget.load(std::memory_order_relaxed); }

hdp_status_t fail(hdp_status_t st, const std::string& msg) {
  g_last_error = msg;
  return st;
}

hdp_status_t fail_cuda(cudaError_t e, const char* what) {
  g_last_error = std::string(what) + ": " + cudaGetErrorName(e) + " (" + cudaGetErrorString(e) + ")";
  if (e == cudaErrorMemoryAllocation) return HDP_ERR_OUT_OF_MEMORY;
  return HDP_ERR_CUDA;
}

unsigned int* device_error_word() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_err_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_device_error) != cudaSuccess) return nullptr;
    g_err_ptr[dev] = static_cast<unsigned int*>(p);
  }
  return g_err_ptr[dev];
}

}  // namespace hdp

extern "C" {

const char* hdp_status_string(hdp_status_t s) {
  switch (s) {
    case HDP_OK: return "HDP_OK";
    case HDP_ERR_INVALID_ARGUMENT: return "HDP_ERR_INVALID_ARGUMENT";
    case HDP_ERR_UNSUPPORTED: return "HDP_ERR_UNSUPPORTED";
    case HDP_ERR_OUT_OF_MEMORY: return "HDP_ERR_OUT_OF_MEMORY";
    case HDP_ERR_CUDA: return "HDP_ERR_CUDA";
    case HDP_ERR_DEVICE_TIMEOUT: return "HDP_ERR_DEVICE_TIMEOUT";
  }
  return "HDP_ERR_UNKNOWN";
}

const char* hdp_last_error_message(void) { return g_last_error.c_str(); }

uint64_t hdp_kernel_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

uint64_t hdp_host_sync_count(void) { return g_host_syncs.load(std::memory_order_relaxed); }

hdp_status_t hdp_set_wait_budget(int64_t clocks) {
  g_wait_budget.store(clocks > 0 ? static_cast<long long>(clocks) : hdp::kWaitBudgetClocks,
                      std::memory_order_relaxed);
  return HDP_OK;
}

hdp_status_t hdp_device_status(void* stream) {
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  hdp::note_host_sync();
  HDP_CUDA_TRY(cudaStreamSynchronize(s));
  unsigned int* w = hdp::device_error_word();
  if (!w) return hdp::fail(HDP_ERR_CUDA, "cannot resolve the device error word");
  unsigned int code = 0, zero = 0;
  HDP_CUDA_TRY(cudaMemcpyFromSymbol(&code, g_device_error, sizeof code));
  if (code != 0) {
    HDP_CUDA_TRY(cudaMemcpyToSymbol(g_device_error, &zero, sizeof zero));
    char buf[128];
    std::snprintf(buf, sizeof buf, "a kernel's bounded wait expired (code %u)", code);
    return hdp::fail(HDP_ERR_DEVICE_TIMEOUT, buf);
  }
  return HDP_OK;
}

}  // extern "C"
