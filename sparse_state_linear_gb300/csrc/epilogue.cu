// epilogue.cu -- per-head RMS-Norm and element-wise output gate on y.
//
// [SDM notes] "Sparse Delta Memory：中文精读笔记", 2.4 (after Eq. (5)): every
// head's read result y_t goes through an RMS-Norm and an element-wise output
// gate before the heads are mixed:
//   out = y / sqrt(mean_c y_c^2 + eps) * gamma[h] * g.
// One warp per (b, h, t) row: 16-byte loads, a warp sum of squares, then the
// scaled, gated row in bf16 or fp32.  Purely bandwidth-bound.
#include "common.cuh"
#include "internal.h"

namespace sdm {
namespace {

constexpr int kEpiThreads = 256;

struct EpiArgs {
  const float* y;
  const void* g;
  const float* gamma;
  void* out;
  long long rows;
  int H, T, dv;
  float eps;
  int g_dtype, out_dtype;
};

__device__ __forceinline__ float4 load4(const void* base, size_t i, int dt) {
  if (dt == SDM_F32) return __ldg(reinterpret_cast<const float4*>(base) + i);
  const uint2 w = __ldg(reinterpret_cast<const uint2*>(base) + i);
  return make_float4(bf16_bits_to_float(w.x & 0xffffu), bf16_bits_to_float(w.x >> 16),
                     bf16_bits_to_float(w.y & 0xffffu), bf16_bits_to_float(w.y >> 16));
}

__device__ __forceinline__ void store4(void* base, size_t i, int dt, float4 v) {
  if (dt == SDM_F32) {
    reinterpret_cast<float4*>(base)[i] = v;
    return;
  }
  const __nv_bfloat162 a = __floats2bfloat162_rn(v.x, v.y);
  const __nv_bfloat162 b = __floats2bfloat162_rn(v.z, v.w);
  uint2 w;
  w.x = *reinterpret_cast<const uint32_t*>(&a);
  w.y = *reinterpret_cast<const uint32_t*>(&b);
  reinterpret_cast<uint2*>(base)[i] = w;
}

__global__ void __launch_bounds__(kEpiThreads) rmsnorm_gate_kernel(const EpiArgs E) {
  const int lane = threadIdx.x & 31;
  const long long nwarps = (long long)gridDim.x * (kEpiThreads / 32);
  const int n4 = E.dv / 4;
  for (long long row = ((long long)blockIdx.x * kEpiThreads + threadIdx.x) >> 5; row < E.rows;
       row += nwarps) {
    const float4* yr = reinterpret_cast<const float4*>(E.y) + row * n4;
    float ss = 0.f;
    for (int c = lane; c < n4; c += 32) {
      const float4 v = __ldg(yr + c);
      ss = fmaf(v.x, v.x, ss);
      ss = fmaf(v.y, v.y, ss);
      ss = fmaf(v.z, v.z, ss);
      ss = fmaf(v.w, v.w, ss);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
    const float inv = 1.f / sqrtf(ss / (float)E.dv + E.eps);
    const int h = (int)((row / E.T) % E.H);
    const float4* gm = E.gamma ? reinterpret_cast<const float4*>(E.gamma) + (size_t)h * n4
                               : nullptr;
    for (int c = lane; c < n4; c += 32) {
      const float4 v = __ldg(yr + c);
      const float4 gt = load4(E.g, (size_t)row * n4 + c, E.g_dtype);
      const float4 sc = gm ? __ldg(gm + c) : make_float4(1.f, 1.f, 1.f, 1.f);
      store4(E.out, (size_t)row * n4 + c, E.out_dtype,
             make_float4(v.x * inv * sc.x * gt.x, v.y * inv * sc.y * gt.y,
                         v.z * inv * sc.z * gt.z, v.w * inv * sc.w * gt.w));
    }
  }
}

constexpr int kEpiSMs = 152;

}  // namespace

cudaError_t launch_rmsnorm_gate(const Dims& d, const float* y, const void* g, const float* gamma,
                                float eps, void* out, int out_dtype, cudaStream_t stream) {
  const long long rows = (long long)d.B * d.H * d.T;
  if (rows == 0) return cudaSuccess;
  EpiArgs E{y, g, gamma, out, rows, d.H, d.T, d.dv, eps, d.in_dtype, out_dtype};
  const long long want = (rows + kEpiThreads / 32 - 1) / (kEpiThreads / 32);
  const unsigned blocks = (unsigned)(want < 16 * kEpiSMs ? want : 16 * kEpiSMs);
  rmsnorm_gate_kernel<<<blocks, kEpiThreads, 0, stream>>>(E);
  return cudaGetLastError();
}

}  // namespace sdm
