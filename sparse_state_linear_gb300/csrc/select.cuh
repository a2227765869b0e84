// select.cuh -- exact warp-level product-key selection.
//
// [SDM notes] "Sparse Delta Memory：中文精读笔记", 2.3: every half keeps its
// top-k sub-scores, the k*k sums S_1[a] + S_2[b] are ranked and the best W
// (R) kept; 2.2: the weights are a softmax over the selected scores.
//
// Order used everywhere: x before y iff x.v > y.v, or x.v == y.v and
// x.id < y.id (ids: sub-index within a half, slot a*s + b after the merge).
// Floats compare as values (-0 == +0).  NaN scores are not supported.
//
// Selection = exact radix select of the k-th element on an order-preserving
// 32-bit key (8-bit digits, warp-shared histogram; stops as soon as the
// boundary digit holds exactly the elements still needed), ids break the
// remaining value ties, ballot compaction, then a register bitonic sort of
// the k <= 64 winners.  No step depends on scheduling, so results are
// bit-reproducible.
//
// Merge: only pairs with (a+1)(b+1) <= W can be among the best W (each other
// pair has at least W pairs at least as large above-left of it in the sorted
// k x k grid).  Ties at the W-th value could still let an excluded pair win
// on its lower slot, so the largest excluded sum is checked; if it reaches the
// W-th selected sum the full k*k grid is ranked instead.
#pragma once

#include "common.cuh"

namespace sdm {

constexpr int kMaxSel = 64;
constexpr unsigned kFull = 0xffffffffu;

__device__ __forceinline__ bool better(float va, uint32_t ia, float vb, uint32_t ib) {
  return va > vb || (va == vb && ia < ib);
}

// Order-preserving key: key(x) < key(y) iff x < y; -0 and +0 share a key.
__device__ __forceinline__ uint32_t order_key(float x) {
  uint32_t u = __float_as_uint(x);
  if ((u << 1) == 0u) u = 0u;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

constexpr int kTmpCap = 128;   // bucket-ordered candidates of the fast path

struct WarpScratch {
  uint32_t hist[256];          // digit / bucket counts; fast path: then scatter cursors
  uint32_t base[260];          // fast path: exclusive prefix of bucket counts
  union {
    struct {                   // radix path: unsorted winners
      float cand_v[kMaxSel];
      uint32_t cand_id[kMaxSel];
    };
    struct {                   // fast path: candidates in bucket order
      float tmp_v[kTmpCap];
      uint32_t tmp_id[kTmpCap];
    };
  };
  float out_v[kMaxSel];
  uint32_t out_id[kMaxSel];
};

// Locate the digit where the running count (from the top digit if
// `descending`, else from digit 0) reaches `need`.  Returns the digit, the
// count strictly before it and its own count.  Requires sum(hist) >= need.
__device__ __forceinline__ void find_digit(const uint32_t* hist, uint32_t need,
                                           bool descending, int lane, uint32_t& digit,
                                           uint32_t& before, uint32_t& cnt) {
  uint32_t c[8];
  uint32_t tot = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int d = descending ? (255 - 8 * lane - i) : (8 * lane + i);
    c[i] = hist[d];
    tot += c[i];
  }
  uint32_t inc = tot;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const uint32_t t = __shfl_up_sync(kFull, inc, off);
    if (lane >= off) inc += t;
  }
  const uint32_t exc = inc - tot;
  const unsigned m = __ballot_sync(kFull, exc < need && need <= inc);
  const int L = __ffs(m) - 1;
  uint32_t d_o = 0, b_o = 0, c_o = 0;
  if (lane == L) {
    uint32_t run = exc;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      if (run < need && need <= run + c[i]) {
        d_o = descending ? (255 - 8 * lane - i) : (8 * lane + i);
        b_o = run;
        c_o = c[i];
      }
      run += c[i];
    }
  }
  digit = __shfl_sync(kFull, d_o, L);
  before = __shfl_sync(kFull, b_o, L);
  cnt = __shfl_sync(kFull, c_o, L);
}

// Bitonic sort of 32*PL (value, id) pairs held PL per lane (element
// e = lane*PL + i), best first.
template <int PL>
__device__ __forceinline__ void bitonic_sort_best_first(float (&v)[PL], uint32_t (&id)[PL],
                                                        int lane) {
  constexpr int NTOT = 32 * PL;
#pragma unroll
  for (int k = 2; k <= NTOT; k <<= 1) {
#pragma unroll
    for (int j = k >> 1; j > 0; j >>= 1) {
      float pv[PL];
      uint32_t pid[PL];
#pragma unroll
      for (int i = 0; i < PL; ++i) {
        if (j < PL) {
          pv[i] = v[i ^ j];
          pid[i] = id[i ^ j];
        } else {
          pv[i] = __shfl_xor_sync(kFull, v[i], j / PL);
          pid[i] = __shfl_xor_sync(kFull, id[i], j / PL);
        }
      }
#pragma unroll
      for (int i = 0; i < PL; ++i) {
        const int e = lane * PL + i;
        const bool up = (e & k) == 0;
        const bool lower = (e & j) == 0;
        const bool take = (lower == up) ? better(pv[i], pid[i], v[i], id[i])
                                        : better(v[i], id[i], pv[i], pid[i]);
        if (take) {
          v[i] = pv[i];
          id[i] = pid[i];
        }
      }
    }
  }
}

// The best k (1 <= k <= 64 <= n) of the n elements given by src.get(e, v, id),
// written best first to ws.out_v / ws.out_id.  Whole warp, converged.
template <class Src>
__device__ void warp_topk_sorted(const Src& src, int n, int k, WarpScratch& ws, int lane) {
  uint32_t prefix = 0, need = (uint32_t)k;
  int shift = 32;
  bool exact = false;
  for (int pass = 0; pass < 4; ++pass) {
    shift -= 8;
    for (int i = lane; i < 256; i += 32) ws.hist[i] = 0u;
    __syncwarp();
    for (int e = lane; e < n; e += 32) {
      float v;
      uint32_t id;
      src.get(e, v, id);
      const uint32_t key = order_key(v);
      if (pass == 0 || (key >> (shift + 8)) == prefix)
        atomicAdd(&ws.hist[(key >> shift) & 255u], 1u);
    }
    __syncwarp();
    uint32_t d, before, cnt;
    find_digit(ws.hist, need, true, lane, d, before, cnt);
    need -= before;
    prefix = (prefix << 8) | d;
    __syncwarp();
    if (cnt == need) {
      exact = true;
      break;
    }
  }
  // Value ties at the full key: keep the `need` smallest ids among them.
  uint32_t idprefix = 0;
  int idshift = 24;
  if (!exact) {
    for (int pass = 0; pass < 3; ++pass) {
      idshift -= 8;
      for (int i = lane; i < 256; i += 32) ws.hist[i] = 0u;
      __syncwarp();
      for (int e = lane; e < n; e += 32) {
        float v;
        uint32_t id;
        src.get(e, v, id);
        if (order_key(v) == prefix && (pass == 0 || (id >> (idshift + 8)) == idprefix))
          atomicAdd(&ws.hist[(id >> idshift) & 255u], 1u);
      }
      __syncwarp();
      uint32_t d, before, cnt;
      find_digit(ws.hist, need, false, lane, d, before, cnt);
      need -= before;
      idprefix = (idprefix << 8) | d;
      __syncwarp();
      if (cnt == need) break;
    }
  }
  // Compaction of the k winners (any order) into ws.cand_*.
  int base = 0;
  for (int e0 = 0; e0 < n; e0 += 32) {
    const int e = e0 + lane;
    bool sel = false;
    float v = 0.f;
    uint32_t id = 0;
    if (e < n) {
      src.get(e, v, id);
      const uint32_t kp = order_key(v) >> shift;
      if (kp > prefix)
        sel = true;
      else if (kp == prefix)
        sel = exact ? true : ((id >> idshift) <= idprefix);
    }
    const unsigned m = __ballot_sync(kFull, sel);
    if (sel) {
      const int pos = min(base + __popc(m & ((1u << lane) - 1u)), kMaxSel - 1);
      ws.cand_v[pos] = v;
      ws.cand_id[pos] = id;
    }
    base += __popc(m);
  }
  __syncwarp();
  // Sort the winners, best first.
  if (k <= 32) {
    float v[1];
    uint32_t id[1];
    v[0] = lane < k ? ws.cand_v[lane] : -INFINITY;
    id[0] = lane < k ? ws.cand_id[lane] : 0xffffffffu;
    bitonic_sort_best_first<1>(v, id, lane);
    if (lane < k) {
      ws.out_v[lane] = v[0];
      ws.out_id[lane] = id[0];
    }
  } else {
    float v[2];
    uint32_t id[2];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const int e = 2 * lane + i;
      v[i] = e < k ? ws.cand_v[e] : -INFINITY;
      id[i] = e < k ? ws.cand_id[e] : 0xffffffffu;
    }
    bitonic_sort_best_first<2>(v, id, lane);
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const int e = 2 * lane + i;
      if (e < k) {
        ws.out_v[e] = v[i];
        ws.out_id[e] = id[i];
      }
    }
  }
  __syncwarp();
}

// Fast exact top-k for n <= 32*PL elements (values cached in registers).
// One pass buckets every value by its distance below the row maximum:
// bucket(v) = min(255, trunc((vmax - v) * 256 / (vmax - vmin))).  The map is
// monotone and equal values share a bucket, so an element in a lower bucket
// is strictly larger than any element in a higher one.  Buckets up to the one
// holding the k-th element are scattered in bucket order (counting sort) and
// every candidate's rank is its bucket's base plus the number of members of
// its own bucket that come first in (value desc, id asc).  Returns false
// (nothing written) when the data defeat the bucketing (all values equal, an
// infinite range, or more than kTmpCap candidates up to the boundary bucket);
// the caller then uses warp_topk_sorted.
template <int PL, class Src>
__device__ bool warp_topk_bucketed(const Src& src, int n, int k, WarpScratch& ws, int lane) {
  float v[PL];
  float vmax = -INFINITY, vmin = INFINITY;
#pragma unroll
  for (int i = 0; i < PL; ++i) {
    const int e = lane + 32 * i;
    v[i] = 0.f;
    if (e < n) {
      uint32_t id;
      src.get(e, v[i], id);
      vmax = fmaxf(vmax, v[i]);
      vmin = fminf(vmin, v[i]);
    }
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    vmax = fmaxf(vmax, __shfl_xor_sync(kFull, vmax, off));
    vmin = fminf(vmin, __shfl_xor_sync(kFull, vmin, off));
  }
  const float range = vmax - vmin;
  if (!(range > 0.f) || !(range < INFINITY)) return false;
  // Any positive scale keeps the map monotone (ranks are exact comparisons).
  const float scale = __fdividef(256.f, range);
  auto bucket = [&](float x) -> uint32_t {
    const float dd = (vmax - x) * scale;
    return min(255u, __float2uint_rz(dd));
  };
  {
    uint4* h4 = reinterpret_cast<uint4*>(ws.hist);
    h4[2 * lane] = make_uint4(0u, 0u, 0u, 0u);
    h4[2 * lane + 1] = make_uint4(0u, 0u, 0u, 0u);
  }
  __syncwarp();
  // Each element's arrival order within its bucket (the count before its
  // own increment) places it in bucket order later without a second pass of
  // atomics; the orders are kept as bytes, four to a register.
  constexpr int PW = (PL + 3) / 4;
  uint32_t ord[PW];
#pragma unroll
  for (int i = 0; i < PW; ++i) ord[i] = 0u;
#pragma unroll
  for (int i = 0; i < PL; ++i)
    if (lane + 32 * i < n) {
      const uint32_t o = atomicAdd(&ws.hist[bucket(v[i])], 1u);
      ord[i >> 2] |= (o & 255u) << (8 * (i & 3));
    }
  __syncwarp();
  // Exclusive prefix over buckets (lane owns 8 consecutive buckets).
  uint32_t c[8], tot = 0;
  {
    const uint4 a = reinterpret_cast<const uint4*>(ws.hist)[2 * lane];
    const uint4 b = reinterpret_cast<const uint4*>(ws.hist)[2 * lane + 1];
    c[0] = a.x; c[1] = a.y; c[2] = a.z; c[3] = a.w;
    c[4] = b.x; c[5] = b.y; c[6] = b.z; c[7] = b.w;
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) tot += c[i];
  uint32_t inc = tot;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const uint32_t t = __shfl_up_sync(kFull, inc, off);
    if (lane >= off) inc += t;
  }
  uint32_t run = inc - tot;
  uint32_t bstar = 256;          // boundary bucket (found by exactly one lane)
  uint32_t pre[8];
  __syncwarp();
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    pre[i] = run;
    if (run < (uint32_t)k && (uint32_t)k <= run + c[i]) bstar = 8 * lane + i;
    run += c[i];
  }
  {
    // Bucket bases.
    const uint4 a = make_uint4(pre[0], pre[1], pre[2], pre[3]);
    const uint4 b = make_uint4(pre[4], pre[5], pre[6], pre[7]);
    reinterpret_cast<uint4*>(ws.base)[2 * lane] = a;
    reinterpret_cast<uint4*>(ws.base)[2 * lane + 1] = b;
  }
  if (lane == 31) ws.base[256] = run;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) bstar = min(bstar, __shfl_xor_sync(kFull, bstar, off));
  __syncwarp();
  const uint32_t ncand = ws.base[bstar + 1];
  if (ncand > (uint32_t)kTmpCap) return false;
  // Scatter the candidates in bucket order: bucket base + arrival order
  // (counts never exceed n < 256 per bucket, so a byte holds the order).
#pragma unroll
  for (int i = 0; i < PL; ++i) {
    const int e = lane + 32 * i;
    if (e < n) {
      const uint32_t b = bucket(v[i]);
      if (b <= bstar) {
        const uint32_t pos = ws.base[b] + ((ord[i >> 2] >> (8 * (i & 3))) & 255u);
        ws.tmp_v[pos] = v[i];
        ws.tmp_id[pos] = src.id(e);
      }
    }
  }
  __syncwarp();
  // Exact rank of every candidate; the best k land in ws.out_* in order.
  for (uint32_t p = lane; p < ncand; p += 32) {
    const float pv = ws.tmp_v[p];
    const uint32_t pid = ws.tmp_id[p];
    const uint32_t b = bucket(pv);
    const uint32_t lo = ws.base[b], hi = ws.base[b + 1];
    uint32_t r = lo;
    for (uint32_t q = lo; q < hi; ++q) r += better(ws.tmp_v[q], ws.tmp_id[q], pv, pid) ? 1u : 0u;
    if (r < (uint32_t)k) {
      ws.out_v[r] = pv;
      ws.out_id[r] = pid;
    }
  }
  __syncwarp();
  return true;
}

// Best k of n (k <= 64): the bucketed path when it applies, else the radix one.
template <int PL, class Src>
__device__ __forceinline__ void warp_topk(const Src& src, int n, int k, WarpScratch& ws, int lane) {
  if (n <= 32 * PL && warp_topk_bucketed<PL>(src, n, k, ws, lane)) return;
  warp_topk_sorted(src, n, k, ws, lane);
}

// Element sources ------------------------------------------------------------

// One half's sub-scores: element j has value row[j] and id j.
struct RowSrc {
  const float* row;
  __device__ __forceinline__ void get(int e, float& v, uint32_t& id) const {
    v = row[e];
    id = (uint32_t)e;
  }
  __device__ __forceinline__ uint32_t id(int e) const { return (uint32_t)e; }
};

// Candidate pairs (a, b) listed in `pairs` as (a << 8) | b.
struct PairSrc {
  const float* v1;
  const uint32_t* id1;
  const float* v2;
  const uint32_t* id2;
  const uint16_t* pairs;
  uint32_t s;
  __device__ __forceinline__ void get(int e, float& v, uint32_t& id) const {
    const uint32_t ab = pairs[e];
    const uint32_t a = ab >> 8, b = ab & 255u;
    v = __fadd_rn(v1[a], v2[b]);
    id = id1[a] * s + id2[b];
  }
  __device__ __forceinline__ uint32_t id(int e) const {
    const uint32_t ab = pairs[e];
    return id1[ab >> 8] * s + id2[ab & 255u];
  }
};

// The full k x k grid, element e = a*k + b.
struct GridSrc {
  const float* v1;
  const uint32_t* id1;
  const float* v2;
  const uint32_t* id2;
  int k;
  uint32_t s;
  __device__ __forceinline__ void get(int e, float& v, uint32_t& id) const {
    const int a = e / k, b = e - a * k;
    v = __fadd_rn(v1[a], v2[b]);
    id = id1[a] * s + id2[b];
  }
  __device__ __forceinline__ uint32_t id(int e) const {
    const int a = e / k, b = e - a * k;
    return id1[a] * s + id2[b];
  }
};

// Pairs (a, b), a, b < k, with (a+1)(b+1) <= nsel, written a-major.  Whole
// warp; returns their number (at least nsel when nsel <= k*k).
__device__ __forceinline__ int build_stair(int nsel, int k, uint16_t* pairs, int lane) {
  const int a0 = lane, a1 = lane + 32;
  const int c0 = a0 < k ? min(k, nsel / (a0 + 1)) : 0;
  const int c1 = a1 < k ? min(k, nsel / (a1 + 1)) : 0;
  int i0 = c0, i1 = c1;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int t0 = __shfl_up_sync(kFull, i0, off);
    const int t1 = __shfl_up_sync(kFull, i1, off);
    if (lane >= off) {
      i0 += t0;
      i1 += t1;
    }
  }
  const int tot0 = __shfl_sync(kFull, i0, 31);
  const int tot1 = __shfl_sync(kFull, i1, 31);
  const int o0 = i0 - c0, o1 = tot0 + i1 - c1;
  for (int b = 0; b < c0; ++b) pairs[o0 + b] = (uint16_t)((a0 << 8) | b);
  for (int b = 0; b < c1; ++b) pairs[o1 + b] = (uint16_t)((a1 << 8) | b);
  __syncwarp();
  return tot0 + tot1;
}

// Best nsel slots of the two sorted half lists, best first, into ws.out_*.
// `bcut` (optional) holds nsel / (a + 1) for a < k.
__device__ __forceinline__ void warp_merge(const float* v1, const uint32_t* id1,
                                           const float* v2, const uint32_t* id2, int k,
                                           int nsel, uint32_t s, const uint16_t* stair,
                                           int nstair, WarpScratch& ws, int lane,
                                           const int* bcut = nullptr) {
  PairSrc ps{v1, id1, v2, id2, stair, s};
  warp_topk<10>(ps, nstair, nsel, ws, lane);
  const float cw = ws.out_v[nsel - 1];
  bool tie = false;
  for (int a = lane; a < k; a += 32) {
    const int b = bcut ? bcut[a] : nsel / (a + 1);
    if (b < k && __fadd_rn(v1[a], v2[b]) >= cw) tie = true;
  }
  if (__any_sync(kFull, tie)) {
    GridSrc gs{v1, id1, v2, id2, k, s};
    warp_topk_sorted(gs, k * k, nsel, ws, lane);
  }
}

// Softmax of ov[0..nsel) and store of slots oi and weights (best first).
__device__ __forceinline__ void softmax_store(const float* ov, const uint32_t* oi, int nsel,
                                              int32_t* idx_out, float* wt_out, int lane) {
  const float m = ov[0];
  const float e0 = lane < nsel ? expf(ov[lane] - m) : 0.f;
  const float e1 = lane + 32 < nsel ? expf(ov[lane + 32] - m) : 0.f;
  float sum = e0 + e1;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(kFull, sum, off);
  if (lane < nsel) {
    idx_out[lane] = (int32_t)oi[lane];
    wt_out[lane] = e0 / sum;
  }
  if (lane + 32 < nsel) {
    idx_out[lane + 32] = (int32_t)oi[lane + 32];
    wt_out[lane + 32] = e1 / sum;
  }
}
__device__ __forceinline__ void warp_softmax_store(const WarpScratch& ws, int nsel,
                                                   int32_t* idx_out, float* wt_out,
                                                   int lane) {
  softmax_store(ws.out_v, ws.out_id, nsel, idx_out, wt_out, lane);
}

// ------------------------------------------------------------ warp groups
// The bucketed top-k above, shared by a group of NW consecutive warps that
// synchronise on named barrier `bar` (for latency-bound callers with idle
// warps: each phase then touches PL elements per thread instead of a warp's
// n / 32).  Same buckets, same exact ranks, so the same result as
// warp_topk_bucketed; returns false (group-uniform, nothing written) where
// that one would, and the caller falls back to the warp paths.
constexpr int kGTmpCap = 256;

struct GroupScratch {
  uint32_t hist[256];          // bucket counts, then scatter cursors
  uint32_t base[260];          // exclusive prefix of the counts
  float tmp_v[kGTmpCap];       // candidates in bucket order
  uint32_t tmp_id[kGTmpCap];
  float out_v[kMaxSel];
  uint32_t out_id[kMaxSel];
  float wmin[8], wmax[8];      // per-warp extremes
  uint32_t wsum[8];            // per-warp bucket totals (prefix scan)
  uint32_t bstar;
};

template <int NW, int PL, class Src>
__device__ bool group_topk_bucketed(const Src& src, int n, int k, GroupScratch& g, int gt,
                                    int bar) {
  constexpr int NT = 32 * NW;
  constexpr int BPT = 256 / NT;    // buckets per thread in the prefix scan
  static_assert(NT <= 256 && 256 % NT == 0, "group size");
  const int lane = gt & 31, w = gt >> 5;
  float v[PL];
  uint32_t id[PL];
  float vmax = -INFINITY, vmin = INFINITY;
#pragma unroll
  for (int i = 0; i < PL; ++i) {
    const int e = gt + NT * i;
    v[i] = 0.f;
    id[i] = 0u;
    if (e < n) {
      src.get(e, v[i], id[i]);
      vmax = fmaxf(vmax, v[i]);
      vmin = fminf(vmin, v[i]);
    }
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    vmax = fmaxf(vmax, __shfl_xor_sync(kFull, vmax, off));
    vmin = fminf(vmin, __shfl_xor_sync(kFull, vmin, off));
  }
  if (lane == 0) {
    g.wmax[w] = vmax;
    g.wmin[w] = vmin;
  }
#pragma unroll
  for (int i = 0; i < BPT; ++i) g.hist[gt * BPT + i] = 0u;
  named_bar_sync(bar, NT);
  vmax = g.wmax[0];
  vmin = g.wmin[0];
#pragma unroll
  for (int i = 1; i < NW; ++i) {
    vmax = fmaxf(vmax, g.wmax[i]);
    vmin = fminf(vmin, g.wmin[i]);
  }
  const float range = vmax - vmin;
  if (!(range > 0.f) || !(range < INFINITY)) return false;
  // Any positive scale keeps the map monotone (ranks are exact comparisons).
  const float scale = __fdividef(256.f, range);
  auto bucket = [&](float x) -> uint32_t {
    const float dd = (vmax - x) * scale;
    return min(255u, __float2uint_rz(dd));
  };
#pragma unroll
  for (int i = 0; i < PL; ++i)
    if (gt + NT * i < n) atomicAdd(&g.hist[bucket(v[i])], 1u);
  named_bar_sync(bar, NT);
  // Exclusive prefix over the buckets: thread gt owns BPT consecutive ones.
  uint32_t c[BPT], tot = 0;
#pragma unroll
  for (int i = 0; i < BPT; ++i) {
    c[i] = g.hist[gt * BPT + i];
    tot += c[i];
  }
  uint32_t inc = tot;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const uint32_t t = __shfl_up_sync(kFull, inc, off);
    if (lane >= off) inc += t;
  }
  if (lane == 31) g.wsum[w] = inc;
  named_bar_sync(bar, NT);
  uint32_t run = inc - tot;
  for (int i = 0; i < w; ++i) run += g.wsum[i];
#pragma unroll
  for (int i = 0; i < BPT; ++i) {
    const int b = gt * BPT + i;
    if (run < (uint32_t)k && (uint32_t)k <= run + c[i]) g.bstar = (uint32_t)b;
    g.base[b] = run;
    g.hist[b] = run;             // scatter cursor
    run += c[i];
  }
  if (gt == NT - 1) g.base[256] = run;
  named_bar_sync(bar, NT);
  const uint32_t bstar = g.bstar;
  const uint32_t ncand = g.base[bstar + 1];
  if (ncand > (uint32_t)kGTmpCap) return false;
#pragma unroll
  for (int i = 0; i < PL; ++i) {
    if (gt + NT * i < n) {
      const uint32_t b = bucket(v[i]);
      if (b <= bstar) {
        const uint32_t pos = atomicAdd(&g.hist[b], 1u);
        g.tmp_v[pos] = v[i];
        g.tmp_id[pos] = id[i];
      }
    }
  }
  named_bar_sync(bar, NT);
  for (uint32_t p = gt; p < ncand; p += NT) {
    const float pv = g.tmp_v[p];
    const uint32_t pid = g.tmp_id[p];
    const uint32_t b = bucket(pv);
    const uint32_t lo = g.base[b], hi = g.base[b + 1];
    uint32_t r = lo;
    for (uint32_t q = lo; q < hi; ++q) r += better(g.tmp_v[q], g.tmp_id[q], pv, pid) ? 1u : 0u;
    if (r < (uint32_t)k) {
      g.out_v[r] = pv;
      g.out_id[r] = pid;
    }
  }
  named_bar_sync(bar, NT);
  return true;
}

}  // namespace sdm
