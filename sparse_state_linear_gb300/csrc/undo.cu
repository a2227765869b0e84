// undo.cu -- putting back a logged segment of the scan.
//
// [SDM notes] "Sparse Delta Memory：中文精读笔记", 2.9 and appendix A.3: the
// backward pass restores earlier states by undoing the in-place sparse
// writes.  The logged scan stores, for every step, each write row's value
// from just before that step's write; undoing a segment puts back, for every
// row it wrote, the copy logged at that row's earliest write (exact).
#include "common.cuh"
#include "internal.h"

namespace sdm {
namespace {

// A logged segment is undone by putting back, for every row it wrote, the
// copy logged at that row's earliest write in the segment.  Three passes
// over the segment's write sets, as stream-ordered launches (no ordering
// between steps is needed inside a pass):
//   clear  mark[chain][row] = 0 for every row the segment wrote;
//   mark   atomicMax(mark[chain][row], T - t), so the earliest step wins;
//   copy   the (t, j) whose mark equals T - t copies its logged row back.
struct UndoArgs {
  const int32_t* idx_w;
  const float* undo;
  float* M;
  uint32_t* mark;
  long long n;          // B * H * T * W write entries
  int T, W, dv;
  uint32_t N;
  unsigned* status;
};

constexpr int kUndoThreads = 256;

__global__ void __launch_bounds__(kUndoThreads) undo_mark_kernel(const UndoArgs U, int pass) {
  const long long stride = (long long)gridDim.x * kUndoThreads;
  for (long long e = (long long)blockIdx.x * kUndoThreads + threadIdx.x; e < U.n; e += stride) {
    const long long tw = (long long)U.T * U.W;
    const long long chain = e / tw;
    const int t = (int)((e - chain * tw) / U.W);
    const int row = __ldg(U.idx_w + e);
    if (row < 0 || (uint32_t)row >= U.N) {
      if (pass == 1) record_status(U.status, SDM_ERR_DEVICE_BOUNDS);
      continue;
    }
    uint32_t* mk = U.mark + chain * U.N + row;
    if (pass == 0)
      *mk = 0u;
    else
      atomicMax(mk, (uint32_t)(U.T - t));
  }
}

// One warp per write entry: 16-byte copies of the logged row.
__global__ void __launch_bounds__(kUndoThreads) undo_copy_kernel(const UndoArgs U) {
  const int lane = threadIdx.x & 31;
  const long long nwarps = (long long)gridDim.x * (kUndoThreads / 32);
  const long long tw = (long long)U.T * U.W;
  for (long long e = ((long long)blockIdx.x * kUndoThreads + threadIdx.x) >> 5; e < U.n;
       e += nwarps) {
    const long long chain = e / tw;
    const int t = (int)((e - chain * tw) / U.W);
    const int row = __ldg(U.idx_w + e);
    if (row < 0 || (uint32_t)row >= U.N) continue;
    if (U.mark[chain * U.N + row] != (uint32_t)(U.T - t)) continue;
    const float4* src = reinterpret_cast<const float4*>(U.undo + e * U.dv);
    float4* dst = reinterpret_cast<float4*>(U.M + (chain * U.N + row) * U.dv);
    for (int c = lane; c < U.dv / 4; c += 32) dst[c] = __ldg(src + c);
  }
}

}  // namespace

size_t undo_workspace_bytes(const Dims& d) {
  return (size_t)d.B * d.H * (size_t)d.N() * sizeof(uint32_t);
}

cudaError_t launch_undo(const Dims& d, const int32_t* idx_w, const float* undo, float* M,
                        void* workspace, unsigned* status, cudaStream_t stream) {
  const long long n = (long long)d.B * d.H * d.T * d.W;
  if (n == 0) return cudaSuccess;
  UndoArgs U{idx_w, undo, M, static_cast<uint32_t*>(workspace), n, d.T, d.W, d.dv,
             (uint32_t)d.N(), status};
  const long long sms = device_limits().sms;
  const long long want = (n + kUndoThreads - 1) / kUndoThreads;
  const unsigned blocks = (unsigned)(want < 8 * sms ? want : 8 * sms);
  undo_mark_kernel<<<blocks, kUndoThreads, 0, stream>>>(U, 0);
  undo_mark_kernel<<<blocks, kUndoThreads, 0, stream>>>(U, 1);
  const long long wantc = (n + kUndoThreads / 32 - 1) / (kUndoThreads / 32);
  const unsigned cblocks = (unsigned)(wantc < 16 * sms ? wantc : 16 * sms);
  undo_copy_kernel<<<cblocks, kUndoThreads, 0, stream>>>(U);
  return cudaGetLastError();
}

}  // namespace sdm
