// plan.cu -- the hazard plan of the scan: where each row's current value is.
//
// [SDM notes] "Sparse Delta Memory：中文精读笔记", 2.4, Eq. (3)-(5): step t
// writes its W slots and then reads its R slots, so a row a step touches may
// have been written by one of the few steps before it.  The scan fetches the
// rows of step t while steps t-depth+1 .. t-1 may still be writing them; for
// every row a step touches this kernel records where its current value will
// be: -1 = the fetched copy, (d << 6) | p = the on-chip copy that step t-d
// left at write position p (latest such d; reads also see d = 0, the step's
// own write), -2 = invalid (index out of range, or a slot repeated within one
// write set; both also recorded in the status word).
//
// Fully parallel over chains and blocks of 64 steps: one CTA hashes the write
// sets of its block plus the depth-1 steps before it into shared memory; two
// filters ("written once", "written again") answer nearly every lookup at
// once, and the rest are resolved on the table.
#include "common.cuh"
#include "internal.h"

namespace sdm {
namespace {

constexpr int kPlanTB = 64;          // steps per plan CTA
constexpr int kPlanThreads = 512;
constexpr int kPlanBuckets = 4096;   // hash buckets of 4 entries (uint32) each
constexpr int kPlanBloom = 2048;     // words of each filter (65536 bits)
constexpr int kPlanQCap = 160;       // per-warp queue of filter hits (< 32 + 4 * 32)
// Shared memory: entries, bucket counts, two filters, queues.
constexpr size_t kPlanSmem =
    sizeof(uint32_t) * (5 * kPlanBuckets + 2 * kPlanBloom + (kPlanThreads / 32) * kPlanQCap);

struct PlanArgs {
  const int32_t* idx_w;
  const int32_t* idx_r;
  int16_t* codes;
  int T, W, R, depth;
  int Ts;              // rows between chains in the index / code layouts
  uint32_t N;
  unsigned* status;
};

__device__ __forceinline__ uint32_t plan_bucket(uint32_t row) {
  return (row * 0x9E3779B1u) >> 20;
}
// Filter bit of a row: the row itself when the table has at most 65536 rows
// (an exact membership bitmap), else 16 bits of a multiplicative hash.
__device__ __forceinline__ uint32_t plan_bit(uint32_t row, uint32_t N) {
  return N <= 65536u ? row : (row * 0x9E3779B1u) >> 16;
}

// Entry = (row << 13) | (step - s0) << 6 | position; rows < 2^18, step offsets
// < 128 (kPlanTB + depth - 1), positions < 64.  An insert claims the next
// entry of the row's bucket by counting; a full bucket passes the entry on to
// the next one, whose count then exceeds 4 -- which tells lookups to go on.
__device__ __forceinline__ void plan_insert(uint32_t* tab, uint32_t* cnt, int row, uint32_t N,
                                            int ds, int j) {
  if (row < 0 || (uint32_t)row >= N) return;
  const uint32_t key = ((uint32_t)row << 13) | ((uint32_t)ds << 6) | (uint32_t)j;
  uint32_t b = plan_bucket((uint32_t)row);
  for (int i = 0; i < kPlanBuckets; ++i) {
    const uint32_t c = atomicAdd(&cnt[b], 1u);
    if (c < 4u) {
      tab[4 * b + c] = key;
      return;
    }
    b = (b + 1) & (kPlanBuckets - 1);
  }
}

// Code of row `row` at position k of step t (write rows k < W, then reads).
__device__ __forceinline__ int plan_code(const uint32_t* tab, const uint32_t* cnt,
                                         const PlanArgs& P, int s0, int row, int t, int k) {
  if (row < 0 || (uint32_t)row >= P.N) {
    record_status(P.status, SDM_ERR_DEVICE_BOUNDS);
    return -2;
  }
  // Latest writer s of this row with t-depth+1 <= s < t (<= t for reads).
  const bool is_w = k < P.W;
  const int lo = t - (P.depth - 1), hi = is_w ? t - 1 : t;
  int best = -1, bp = 0;
  bool dup = false;
  uint32_t b = plan_bucket((uint32_t)row);
  for (int i = 0; i < kPlanBuckets; ++i) {
    const uint32_t c = cnt[b];
    const uint4 e4 = reinterpret_cast<const uint4*>(tab)[b];
    const uint32_t ents[4] = {e4.x, e4.y, e4.z, e4.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const uint32_t ent = ents[e];
      if ((uint32_t)e < c && (ent >> 13) == (uint32_t)row) {
        const int s = s0 + (int)((ent >> 6) & 127u), p = (int)(ent & 63u);
        if (is_w && s == t && p != k) dup = true;
        if (s >= lo && s <= hi && s > best) {
          best = s;
          bp = p;
        }
      }
    }
    if (c <= 4u) break;
    b = (b + 1) & (kPlanBuckets - 1);
  }
  if (dup) {
    record_status(P.status, SDM_ERR_DUPLICATE_SLOT);
    return -2;
  }
  return best >= 0 ? ((t - best) << 6) | bp : -1;
}

// VEC (W and R multiples of 4): warp w owns steps w, w + 16, ... of the
// block and lane l positions 4l .. 4l+3 of a step, so no index needs a
// division; every thread first issues all of its index loads as 16-byte
// vectors.  Rows of the block's write sets also mark two 65536-bit filters,
// "written once" and "written again", so a read lookup that misses the first
// or a write lookup that misses the second (its own insert set the first)
// cannot have an earlier writer in the window and gets code -1 at once --
// nearly every lookup.  Filter hits queue per warp and are resolved 32 at a
// time on the hash table, so the probe loops run with full warps.
template <bool VEC>
__global__ void __launch_bounds__(kPlanThreads, 2) plan_kernel(const PlanArgs P) {
  extern __shared__ __align__(16) uint32_t tab[];
  uint32_t* cnt = tab + 4 * kPlanBuckets;
  uint32_t* once = cnt + kPlanBuckets;
  uint32_t* again = once + kPlanBloom;
  const int chain = blockIdx.y;
  const int t0 = blockIdx.x * kPlanTB;
  const int t1 = min(P.T, t0 + kPlanTB);
  const int s0 = max(0, t0 - (P.depth - 1));
  const int W = P.W, R = P.R, WR = W + R, CP = code_pitch(W, R);
  const size_t base = (size_t)chain * P.Ts;
  if constexpr (VEC) {
    constexpr int kWarps = kPlanThreads / 32;
    constexpr int kLook = kPlanTB / kWarps;                        // steps per warp
    constexpr int kIns = (kPlanTB + 15 + kWarps - 1) / kWarps;     // insert steps per warp
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int k = 4 * lane;
    const bool lk = k < WR, lw = k < W;
    const int32_t* iw = P.idx_w + base * W;
    const int32_t* ir = P.idx_r + base * R;
    int16_t* cb = P.codes + base * CP;
    uint32_t* q = again + kPlanBloom + warp * kPlanQCap;
    int4 look[kLook], irow[kIns];
#pragma unroll
    for (int i = 0; i < kLook; ++i) {
      const int t = t0 + warp + kWarps * i;
      if (t < t1 && lk)
        look[i] = __ldg(reinterpret_cast<const int4*>(lw ? iw + (size_t)t * W + k
                                                         : ir + (size_t)t * R + (k - W)));
    }
#pragma unroll
    for (int i = 0; i < kIns; ++i) {
      const int s = s0 + warp + kWarps * i;
      if (s < t1 && lw) irow[i] = __ldg(reinterpret_cast<const int4*>(iw + (size_t)s * W + k));
    }
    // Counts and filters are adjacent: one clear (entries need none).
    for (int i = threadIdx.x; i < (kPlanBuckets + 2 * kPlanBloom) / 4; i += kPlanThreads)
      reinterpret_cast<uint4*>(cnt)[i] = make_uint4(0u, 0u, 0u, 0u);
    __syncthreads();
#pragma unroll
    for (int i = 0; i < kIns; ++i) {
      const int ds = warp + kWarps * i;
      if (s0 + ds < t1 && lw) {
        const int r4[4] = {irow[i].x, irow[i].y, irow[i].z, irow[i].w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          if (r4[e] < 0 || (uint32_t)r4[e] >= P.N) continue;
          const uint32_t hb = plan_bit((uint32_t)r4[e], P.N), m = 1u << (hb & 31u);
          if (atomicOr(&once[hb >> 5], m) & m) atomicOr(&again[hb >> 5], m);
          plan_insert(tab, cnt, r4[e], P.N, ds, k + e);
        }
      }
    }
    __syncthreads();
    // Queued hit: (row << 13) | (dt << 7) | position.
    auto resolve = [&](uint32_t ent) {
      const int t = t0 + (int)((ent >> 7) & 63u), kk = (int)(ent & 127u);
      cb[(size_t)t * CP + kk] = (int16_t)plan_code(tab, cnt, P, s0, (int)(ent >> 13), t, kk);
    };
    int qn = 0;   // warp-uniform queue length
#pragma unroll
    for (int i = 0; i < kLook; ++i) {
      const int dt = warp + kWarps * i, t = t0 + dt;
      uint32_t hit = 0;
      const int r4[4] = {look[i].x, look[i].y, look[i].z, look[i].w};
      if (t < t1 && lk) {
        uint32_t c16[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          c16[e] = 0xffffu;                    // -1: the fetched copy
          if (r4[e] < 0 || (uint32_t)r4[e] >= P.N) {
            record_status(P.status, SDM_ERR_DEVICE_BOUNDS);
            c16[e] = 0xfffeu;                  // -2: invalid
          } else {
            const uint32_t hb = plan_bit((uint32_t)r4[e], P.N);
            hit |= (((lw ? again : once)[hb >> 5] >> (hb & 31u)) & 1u) << e;
          }
        }
        // Hits are overwritten after the warp barrier below.  CP is a
        // multiple of 8 and k of 4: one aligned 8-byte store.
        *reinterpret_cast<uint2*>(cb + (size_t)t * CP + k) =
            make_uint2(c16[0] | (c16[1] << 16), c16[2] | (c16[3] << 16));
      }
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const bool h = (hit >> e) & 1u;
        const unsigned bal = __ballot_sync(0xffffffffu, h);
        if (h)
          q[qn + __popc(bal & ((1u << lane) - 1u))] =
              ((uint32_t)r4[e] << 13) | ((uint32_t)dt << 7) | (uint32_t)(k + e);
        qn += __popc(bal);
      }
      __syncwarp();
      while (qn >= 32) {
        qn -= 32;
        resolve(q[qn + lane]);
      }
      __syncwarp();
    }
    if (lane < qn) resolve(q[lane]);
  } else {
    const int nins = (t1 - s0) * W;        // write slots of steps s0 .. t1-1, contiguous
    const int nlook = (t1 - t0) * WR;
    const int32_t* ins = P.idx_w + (base + s0) * W;
    for (int i = threadIdx.x; i < kPlanBuckets / 4; i += kPlanThreads)
      reinterpret_cast<uint4*>(cnt)[i] = make_uint4(0u, 0u, 0u, 0u);
    __syncthreads();
    for (int e = threadIdx.x; e < nins; e += kPlanThreads) {
      const int ds = e / W;
      plan_insert(tab, cnt, __ldg(ins + e), P.N, ds, e - ds * W);
    }
    __syncthreads();
    for (int e = threadIdx.x; e < nlook; e += kPlanThreads) {
      const int dt = e / WR, k = e - dt * WR, t = t0 + dt;
      const int row = k < W ? __ldg(P.idx_w + (base + t) * W + k)
                            : __ldg(P.idx_r + (base + t) * R + (k - W));
      P.codes[(base + t) * CP + k] = (int16_t)plan_code(tab, cnt, P, s0, row, t, k);
    }
  }
}

}  // namespace

cudaError_t launch_plan(const Dims& d, const int32_t* idx_w, const int32_t* idx_r,
                        int16_t* codes, int depth, unsigned* status, cudaStream_t stream) {
  const long long chains = (long long)d.B * d.H;
  if (chains == 0 || d.T == 0) return cudaSuccess;
  const bool vec = d.W % 4 == 0 && d.R % 4 == 0;
  auto* kern = vec ? plan_kernel<true> : plan_kernel<false>;
  cudaError_t e =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kPlanSmem);
  if (e != cudaSuccess) return e;
  PlanArgs P{idx_w, idx_r, codes, d.T, d.W, d.R, depth, d.Ts, (uint32_t)d.N(), status};
  dim3 grid((unsigned)((d.T + kPlanTB - 1) / kPlanTB), (unsigned)chains);
  kern<<<grid, kPlanThreads, kPlanSmem, stream>>>(P);
  return cudaGetLastError();
}

}  // namespace sdm
