// rowtraffic.cu -- a measured ceiling for the scan's memory traffic.
//
// The scan of [SDM notes] 2.4 (Eq. (3)-(5)) moves, per step of every
// (chain, column slice) unit, W + R random row pieces of the chain's table
// from HBM and W pieces back.  This kernel moves the same pieces in the same
// unit layout (one CTA per unit, rows drawn uniformly from the chain's own
// N rows, CW floats per piece, a few steps in flight) with no arithmetic and
// no dependency between steps, so its rate is what HBM gives this access
// pattern: the ceiling the scan is compared against besides the sequential
// copy peak.
//
// Each thread pipelines its own 16-byte copies with cp.async groups
// (commit / wait_group): a thread stores only what its own copies brought in,
// so no barrier and no spin-wait is involved.  Rows come from the lowbias32
// integer hash (Wellons' 2018 search; any well-mixed 32-bit hash would do).
#include "common.cuh"
#include "internal.h"

namespace sdm {
namespace {

constexpr int kRtThreads = 256;
constexpr int kRtDepth = 4;         // steps whose loads are in flight per unit

__device__ __forceinline__ uint32_t lowbias32(uint32_t x) {
  x ^= x >> 16;
  x *= 0x7feb352du;
  x ^= x >> 15;
  x *= 0x846ca68bu;
  x ^= x >> 16;
  return x;
}

template <int CW>
__global__ void __launch_bounds__(kRtThreads) row_traffic_kernel(const float* __restrict__ src,
                                                                 float* __restrict__ dst,
                                                                 long long rows, int dv, int T,
                                                                 int loads, int stores,
                                                                 uint32_t seed) {
  constexpr int CH = CW / 4;                 // 16-byte chunks per piece
  constexpr int PP = kRtThreads / CH;        // pieces per pass of the block
  extern __shared__ __align__(16) unsigned char smem[];
  const int slices = dv / CW;
  const uint32_t unit = blockIdx.x;
  const long long chain = unit / slices;
  const int slice = (int)(unit % slices);
  const size_t cbase = (size_t)chain * (size_t)rows * dv + (size_t)slice * CW;
  const int tid = threadIdx.x, c = tid % CH, r0 = tid / CH;
  const size_t stage = (size_t)loads * CW * 4;
  const uint32_t ukey = lowbias32(seed ^ (unit * 0x9e3779b9u));
  auto pick = [&](int t, int r, uint32_t salt) -> size_t {
    const uint32_t h = lowbias32(ukey ^ lowbias32((uint32_t)t * 0x85ebca6bu + (uint32_t)r + salt));
    return (size_t)(((uint64_t)h * (uint64_t)rows) >> 32);
  };
  for (int t = 0; t < T + kRtDepth - 1; ++t) {
    if (t < T) {
      unsigned char* st = smem + (size_t)(t % kRtDepth) * stage;
      for (int r = r0; r < loads; r += PP)
        cp_async16(st + (size_t)r * CW * 4 + 16 * c, src + cbase + pick(t, r, 0u) * dv + 4 * c);
    }
    cp_async_commit();
    cp_async_wait<kRtDepth - 1>();           // this thread's copies of step t - D + 1 landed
    const int tt = t - (kRtDepth - 1);
    if (tt < 0) continue;
    const unsigned char* st = smem + (size_t)(tt % kRtDepth) * stage;
    for (int r = r0; r < stores; r += PP) {
      const float4 v = *reinterpret_cast<const float4*>(st + (size_t)r * CW * 4 + 16 * c);
      *reinterpret_cast<float4*>(dst + cbase + pick(tt, r, 0x5bd1e995u) * dv + 4 * c) = v;
    }
  }
  cp_async_wait_all();
}

template <int CW>
cudaError_t launch_rt(const float* src, float* dst, long long chains, long long rows, int dv,
                      int T, int loads, int stores, uint32_t seed, cudaStream_t stream) {
  const size_t smem = (size_t)kRtDepth * loads * CW * 4;
  cudaError_t e = cudaFuncSetAttribute(row_traffic_kernel<CW>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const long long units = chains * (dv / CW);
  row_traffic_kernel<CW><<<(unsigned)units, kRtThreads, smem, stream>>>(src, dst, rows, dv, T,
                                                                       loads, stores, seed);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_row_traffic(const float* src, float* dst, long long chains, long long rows,
                               int dv, int col_slice, int T, int loads, int stores,
                               uint32_t seed, cudaStream_t stream) {
  if (col_slice == 16)
    return launch_rt<16>(src, dst, chains, rows, dv, T, loads, stores, seed, stream);
  if (col_slice == 32)
    return launch_rt<32>(src, dst, chains, rows, dv, T, loads, stores, seed, stream);
  return launch_rt<64>(src, dst, chains, rows, dv, T, loads, stores, seed, stream);
}

}  // namespace sdm
