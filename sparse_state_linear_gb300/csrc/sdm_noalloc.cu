// sdm_noalloc.cu -- sdm_scan_noalloc: the scan for callers that cannot
// allocate device memory or hand the library a workspace.
//
// The scan needs scratch for its plan codes (one 16-bit code per token and
// touched row).  sdm_scan takes that scratch from the caller.  Here it is a
// fixed array in this file, in device memory that every GPU loading the
// library keeps until the process exits; no call allocates anything.
#include <cuda_runtime.h>

#include <mutex>

#include "common.cuh"
#include "internal.h"
#include "sdm.h"

namespace sdm {
namespace {

constexpr size_t kNoAllocScratchBytes = size_t(8) << 20;  // 8 MiB per device

// The scratch.  In host code this name is only a host-side stand-in for the
// device symbol: its device address comes from cudaGetSymbolAddress.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mu;
void* g_noalloc_ptr[kMaxDevices] = {};

// Device address of the scratch on the current device, looked up once per
// device (with that device current) and cached.
sdm_status noalloc_scratch(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return SDM_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_noalloc_mu);
  if (!g_noalloc_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return SDM_ERR_CUDA;
    g_noalloc_ptr[dev] = p;
  }
  *out = g_noalloc_ptr[dev];
  return SDM_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace
}  // namespace sdm

using namespace sdm;

extern "C" sdm_status sdm_scan_noalloc(const sdm_shape* shape, const int32_t* idx_w,
                                       const float* wt_w, const int32_t* idx_r,
                                       const float* wt_r, const void* alpha, const void* beta,
                                       const void* v, float* M, float* y, void* stream) {
  Dims d;
  sdm_status st = api_check_shape(shape, &d);
  if (st != SDM_OK) return st;
  if ((long long)d.B * d.H * d.T == 0) return SDM_OK;   // no work: pointers are not looked at
  const void* ptrs[] = {idx_w, wt_w, idx_r, wt_r, alpha, beta, v, M, y};
  for (const void* p : ptrs)
    if (!p || !aligned16(p)) return SDM_ERR_INVALID_ARG;
  // Problems whose plan codes do not fit the fixed scratch are refused.
  if (scan_workspace_bytes(d) > kNoAllocScratchBytes) return SDM_ERR_UNSUPPORTED;
  void* scratch = nullptr;
  if ((st = noalloc_scratch(&scratch)) != SDM_OK) return st;
  unsigned* status = nullptr;
  if ((st = api_status_ptr(&status)) != SDM_OK) return st;
  int depth = 0, col_slice = 0;
  api_scan_tuning(&depth, &col_slice);
  if (col_slice && d.dv % col_slice != 0) return SDM_ERR_INVALID_ARG;
  // Every code the scan reads is written by the plan kernel of this same
  // call, so nothing in the scratch has to start at zero.
  const cudaError_t e = launch_scan(d, idx_w, wt_w, idx_r, wt_r, alpha, beta, v, M, y, nullptr,
                                    scratch, depth, col_slice, status,
                                    static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? SDM_OK : SDM_ERR_CUDA;
}
