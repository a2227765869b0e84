// address.cu -- product-key addressing on sm_103a.
//
// [SDM notes] "Sparse Delta Memory：中文精读笔记", 2.3: per token and head,
// two half-score vectors of length s = sqrt(N) per branch (write, read);
// [FwPKM notes] 2.2: those vectors as half-query x sub-key tables, and the
// inverse-distance score -log(eps + |q - K_j|^2).
//
// One CTA handles one head and a tile of 16 tokens x 2 branches = 32 score
// rows.  For each half p the 32 x s score tile is a small dense contraction
// (32 x d_h times d_h x s) done in fp32 FFMA from shared-memory tiles and
// kept on chip; warps then run the exact top-k of every row (select.cuh).
// After both halves, each row's two sorted lists are merged into the best W
// (R) slots with their softmax weights.
#include "common.cuh"
#include "internal.h"
#include "select.cuh"
#include "tcgen05.cuh"

namespace sdm {
namespace {

constexpr int kRows = 32;       // score rows per CTA
constexpr int kBK = 16;         // reduction chunk (d_h is a multiple of 16)
constexpr int kBN = 256;        // sub-key chunk
constexpr int kThreads = 256;   // 8 warps
constexpr int kWarps = kThreads / 32;
constexpr int kStairMax = 320;  // >= sum_{a<64} floor(64/(a+1)) = 280
// q tile row stride in (q, q) pairs: row r sits at r + 2 * (r / 16), so the
// four 8-row groups a warp reads at once start in distinct bank quarters.
constexpr int kQStride = kRows + 4;
__host__ __device__ constexpr int qpos(int r) { return r + 2 * (r >> 4); }

struct AddrArgs {
  Dims d;
  const void* q0;
  const void* q1;
  const void* K;
  const float* f0;
  const float* f1;
  int32_t* idx_w;
  float* wt_w;
  int32_t* idx_r;
  float* wt_r;
  float* S;
  unsigned* status;
};

struct SmemLayout {
  size_t qT, kT, sc, lv, lid, ws, stair, nst, total;
  int kst;                     // stride of one per-half list (>= k of both branches)
};

__host__ __device__ inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// The q / K tiles live only while scores are computed and the warps'
// selection scratch only while rows are selected (a block barrier separates
// the phases), so the two share one region; the per-half lists are as long
// as the larger k.  At s = 512 and k = 8 this keeps a CTA near 100 KB, two
// per SM.
__host__ __device__ inline SmemLayout smem_layout(int s, int kmax) {
  SmemLayout L;
  L.kst = kmax;
  L.qT = 0;
  L.kT = align_up(sizeof(float2) * kBK * kQStride, 16);  // (q, q) pairs
  const size_t tiles = L.kT + sizeof(float) * kBK * kBN;
  L.ws = 0;
  const size_t wsz = sizeof(WarpScratch) * kWarps;
  size_t o = align_up(tiles > wsz ? tiles : wsz, 16);
  L.sc = o;    o = align_up(o + sizeof(float) * kRows * (size_t)s, 16);
  L.lv = o;    o = align_up(o + sizeof(float) * kRows * 2 * (size_t)kmax, 16);
  L.lid = o;   o = align_up(o + sizeof(uint32_t) * kRows * 2 * (size_t)kmax, 16);
  L.stair = o; o = align_up(o + sizeof(uint16_t) * 2 * kStairMax, 16);
  L.nst = o;   o = align_up(o + sizeof(int) * 2, 16);
  L.total = o;
  return L;
}

__host__ __device__ inline int list_len(const Dims& d) { return d.kw > d.kr ? d.kw : d.kr; }

template <int MODE>
__device__ __forceinline__ void row_item(int r, int& sigma, long long& item) {
  if (MODE == kAddrScoresOnly) {
    sigma = 0;
    item = (long long)blockIdx.x * kRows + r;
  } else {
    sigma = r >> 4;
    item = (long long)blockIdx.x * (kRows / 2) + (r & 15);
  }
}

// Score tile of half p: rows x [j0, j0+kBN) accumulated over d_h.  The
// (sub-key chunk, d chunk) tiles are walked as one sequence; the global
// loads of the next tile are issued before the current tile's FMAs, so their
// latency hides behind the contraction (raw words are kept in registers and
// converted when they are stored to shared memory).
// Packed pairs of fp32 lanes (two IEEE round-to-nearest operations per
// instruction, each lane exactly what the scalar operation gives).
__device__ __forceinline__ uint64_t f32x2_sub(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ uint64_t f32x2_fma(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}
__device__ __forceinline__ uint64_t f32x2_pack(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ float2 f32x2_unpack(uint64_t v) {
  float2 f;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(f.x), "=f"(f.y) : "l"(v));
  return f;
}

template <bool BF16>
struct TileRegs {
  uint32_t q[2];             // this thread's two q elements (raw bits)
  uint32_t k[kBK];           // its sub-key row's kBK elements (raw bits; bf16: 2 per word)
};

template <int MODE, bool BF16, int KIND>
__device__ void score_half(const AddrArgs& A, int p, float2* qT, float* kT, float* sc) {
  const Dims& d = A.d;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int h = blockIdx.y;
  const long long BT = (long long)d.B * d.T;
  // Lane tile: 8 rows (group lane / 8) x 4 sub-keys; a warp covers all 32
  // rows x 32 sub-keys, so per d step it reads four q pairs (one address per
  // row group) and one 128-byte run of K.
  const int rb = 8 * (lane >> 3);
  const int cb = 32 * warp + 4 * (lane & 7);

  // Loader roles: q tile (row = tid/8, two d-elements), K tile (row jj = tid).
  const int lr = tid >> 3, lpart = tid & 7;
  int lsig;
  long long litem;
  row_item<MODE>(lr, lsig, litem);
  const bool lvalid = litem < BT;
  size_t qoff = 0;
  if (lvalid) {
    const long long b = litem / d.T, t = litem - b * d.T;
    const long long th = (b * d.H + h) * d.Ts + t;
    qoff = (size_t)(th * 2 + p) * d.dh;
  }
  const void* qbase = (lsig == 0) ? A.q0 : A.q1;
  const int nd = d.dh / kBK;
  const int ntiles = ((d.s + kBN - 1) / kBN) * nd;

  auto fetch = [&](int it, TileRegs<BF16>& g) {
    const int j0 = (it / nd) * kBN, d0 = (it % nd) * kBK;
    g.q[0] = g.q[1] = 0u;
    if (lvalid) {
      const size_t e = qoff + d0 + 2 * lpart;
      if (BF16) {
        const uint32_t w = __ldg(reinterpret_cast<const uint32_t*>(
            reinterpret_cast<const __nv_bfloat16*>(qbase) + e));
        g.q[0] = w & 0xffffu;
        g.q[1] = w >> 16;
      } else {
        const uint2 w = __ldg(reinterpret_cast<const uint2*>(
            reinterpret_cast<const float*>(qbase) + e));
        g.q[0] = w.x;
        g.q[1] = w.y;
      }
    }
    const int j = j0 + tid;
    if (j < d.s) {
      const size_t e = ((size_t)(h * 2 + p) * d.s + j) * d.dh + d0;
      if (BF16) {
        const uint4* src = reinterpret_cast<const uint4*>(
            reinterpret_cast<const __nv_bfloat16*>(A.K) + e);
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          const uint4 w = __ldg(src + u);
          g.k[4 * u + 0] = w.x; g.k[4 * u + 1] = w.y;
          g.k[4 * u + 2] = w.z; g.k[4 * u + 3] = w.w;
        }
      } else {
        const uint4* src = reinterpret_cast<const uint4*>(
            reinterpret_cast<const float*>(A.K) + e);
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const uint4 w = __ldg(src + u);
          g.k[4 * u + 0] = w.x; g.k[4 * u + 1] = w.y;
          g.k[4 * u + 2] = w.z; g.k[4 * u + 3] = w.w;
        }
      }
    } else {
#pragma unroll
      for (int c = 0; c < kBK; ++c) g.k[c] = 0u;
    }
  };
  // q tile: qT[dd][qpos(row)] as (q, q) pairs; K tile: kT[dd][jj].
  auto put = [&](const TileRegs<BF16>& g) {
    if (BF16) {
      const float x0 = bf16_bits_to_float(g.q[0]), x1 = bf16_bits_to_float(g.q[1]);
      qT[(2 * lpart) * kQStride + qpos(lr)] = make_float2(x0, x0);
      qT[(2 * lpart + 1) * kQStride + qpos(lr)] = make_float2(x1, x1);
#pragma unroll
      for (int c = 0; c < kBK / 2; ++c) {
        kT[(2 * c) * kBN + tid] = bf16_bits_to_float(g.k[c] & 0xffffu);
        kT[(2 * c + 1) * kBN + tid] = bf16_bits_to_float(g.k[c] >> 16);
      }
    } else {
      const float x0 = __uint_as_float(g.q[0]), x1 = __uint_as_float(g.q[1]);
      qT[(2 * lpart) * kQStride + qpos(lr)] = make_float2(x0, x0);
      qT[(2 * lpart + 1) * kQStride + qpos(lr)] = make_float2(x1, x1);
#pragma unroll
      for (int c = 0; c < kBK; ++c) kT[c * kBN + tid] = __uint_as_float(g.k[c]);
    }
  };

  // acc[r][cp]: rows rb + r, sub-key pair (cb + 2cp, cb + 2cp + 1), packed.
  uint64_t acc[8][2];
  TileRegs<BF16> g;
  if (ntiles > 0) fetch(0, g);
  for (int it = 0; it < ntiles; ++it) {
    const int j0 = (it / nd) * kBN;
    if (it % nd == 0) {
#pragma unroll
      for (int r = 0; r < 8; ++r) acc[r][0] = acc[r][1] = 0ull;
    }
    __syncthreads();            // every warp is done with the previous tile
    put(g);
    __syncthreads();
    if (it + 1 < ntiles) fetch(it + 1, g);   // in flight during the FMAs below
#pragma unroll
    for (int dd = 0; dd < kBK; ++dd) {
      uint64_t qv[8];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const float4 q2 = *reinterpret_cast<const float4*>(qT + dd * kQStride + qpos(rb) + 2 * u);
        qv[2 * u] = f32x2_pack(q2.x, q2.y);
        qv[2 * u + 1] = f32x2_pack(q2.z, q2.w);
      }
      const float4 kk = *reinterpret_cast<const float4*>(kT + dd * kBN + cb);
      const uint64_t kv[2] = {f32x2_pack(kk.x, kk.y), f32x2_pack(kk.z, kk.w)};
#pragma unroll
      for (int r = 0; r < 8; ++r)
#pragma unroll
        for (int cp = 0; cp < 2; ++cp) {
          if (KIND == SDM_SCORE_DOT) {
            acc[r][cp] = f32x2_fma(qv[r], kv[cp], acc[r][cp]);
          } else {
            const uint64_t df = f32x2_sub(qv[r], kv[cp]);
            acc[r][cp] = f32x2_fma(df, df, acc[r][cp]);
          }
        }
    }
    if (it % nd != nd - 1) continue;
    // Epilogue of sub-key chunk j0.
#pragma unroll
    for (int r = 0; r < 8; ++r) {
      const int row = rb + r;
      const float2 a01 = f32x2_unpack(acc[r][0]), a23 = f32x2_unpack(acc[r][1]);
      const float av[4] = {a01.x, a01.y, a23.x, a23.y};
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const int col = j0 + cb + c;
        if (col >= d.s) continue;
        const float val = (KIND == SDM_SCORE_DOT) ? av[c] : -logf(d.eps + av[c]);
        if (MODE == kAddrScoresOnly) {
          int sg;
          long long item;
          row_item<MODE>(row, sg, item);
          if (item < BT) {
            const long long b = item / d.T, t = item - b * d.T;
            const long long th = (b * d.H + h) * d.Ts + t;
            A.S[(size_t)(th * 2 + p) * d.s + col] = val;
          }
        } else {
          sc[(size_t)row * d.s + col] = val;
        }
      }
    }
  }
}

template <int MODE, bool BF16, int KIND>
__global__ void __launch_bounds__(kThreads) address_kernel(const AddrArgs A) {
  extern __shared__ __align__(16) unsigned char smem[];
  const Dims& d = A.d;
  const SmemLayout L = smem_layout(d.s, list_len(d));
  const int kst = L.kst;
  float2* qT = reinterpret_cast<float2*>(smem + L.qT);
  float* kT = reinterpret_cast<float*>(smem + L.kT);
  float* sc = reinterpret_cast<float*>(smem + L.sc);
  float* lv = reinterpret_cast<float*>(smem + L.lv);
  uint32_t* lid = reinterpret_cast<uint32_t*>(smem + L.lid);
  WarpScratch* wsa = reinterpret_cast<WarpScratch*>(smem + L.ws);
  uint16_t* stair = reinterpret_cast<uint16_t*>(smem + L.stair);
  int* nst = reinterpret_cast<int*>(smem + L.nst);

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int h = blockIdx.y;
  const long long BT = (long long)d.B * d.T;
  WarpScratch& ws = wsa[warp];

  if (MODE != kAddrScoresOnly) {
    if (warp == 0) {
      const int n = build_stair(d.W, d.kw, stair, lane);
      if (lane == 0) nst[0] = n;
    } else if (warp == 1) {
      const int n = build_stair(d.R, d.kr, stair + kStairMax, lane);
      if (lane == 0) nst[1] = n;
    }
  }

  for (int p = 0; p < 2; ++p) {
    if (MODE == kAddrSelectOnly) {
      __syncthreads();
      for (int e = tid; e < kRows * d.s; e += kThreads) {
        const int r = e / d.s, j = e - r * d.s;
        int sg;
        long long item;
        row_item<MODE>(r, sg, item);
        float val = 0.f;
        if (item < BT) {
          const long long b = item / d.T, t = item - b * d.T;
          const long long th = (b * d.H + h) * d.Ts + t;
          const float* f = sg == 0 ? A.f0 : A.f1;
          val = __ldg(f + (size_t)(th * 2 + p) * d.s + j);
        }
        sc[e] = val;
      }
    } else {
      score_half<MODE, BF16, KIND>(A, p, qT, kT, sc);
    }
    if (MODE == kAddrScoresOnly) continue;
    __syncthreads();
    for (int r = warp; r < kRows; r += kWarps) {
      int sg;
      long long item;
      row_item<MODE>(r, sg, item);
      if (item >= BT) continue;
      const int k = sg == 0 ? d.kw : d.kr;
      RowSrc src{sc + (size_t)r * d.s};
      warp_topk<16>(src, d.s, k, ws, lane);
      float* ov = lv + (r * 2 + p) * kst;
      uint32_t* oi = lid + (r * 2 + p) * kst;
      for (int e = lane; e < k; e += 32) {
        ov[e] = ws.out_v[e];
        oi[e] = ws.out_id[e];
      }
      __syncwarp();
    }
  }
  if (MODE == kAddrScoresOnly) return;
  __syncthreads();
  for (int r = warp; r < kRows; r += kWarps) {
    int sg;
    long long item;
    row_item<MODE>(r, sg, item);
    if (item >= BT) continue;
    const int k = sg == 0 ? d.kw : d.kr;
    const int nsel = sg == 0 ? d.W : d.R;
    warp_merge(lv + (r * 2 + 0) * kst, lid + (r * 2 + 0) * kst,
               lv + (r * 2 + 1) * kst, lid + (r * 2 + 1) * kst, k, nsel,
               (uint32_t)d.s, stair + sg * kStairMax, nst[sg], ws, lane);
    const long long b = item / d.T, t = item - b * d.T;
    const long long th = (b * d.H + h) * d.Ts + t;
    int32_t* io = (sg == 0 ? A.idx_w : A.idx_r) + (size_t)th * nsel;
    float* wo = (sg == 0 ? A.wt_w : A.wt_r) + (size_t)th * nsel;
    warp_softmax_store(ws, nsel, io, wo, lane);
    __syncwarp();
  }
}

template <int MODE, bool BF16, int KIND>
cudaError_t launch_t(const AddrArgs& A, cudaStream_t stream) {
  const SmemLayout L = smem_layout(A.d.s, list_len(A.d));
  auto kfn = address_kernel<MODE, BF16, KIND>;
  cudaError_t e = cudaFuncSetAttribute(kfn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)L.total);
  if (e != cudaSuccess) return e;
  const long long BT = (long long)A.d.B * A.d.T;
  const int per = MODE == kAddrScoresOnly ? kRows : kRows / 2;
  const long long tiles = (BT + per - 1) / per;
  if (tiles == 0 || A.d.H == 0) return cudaSuccess;
  dim3 grid((unsigned)tiles, (unsigned)A.d.H);
  kfn<<<grid, kThreads, L.total, stream>>>(A);
  return cudaGetLastError();
}

// ------------------------------------------------------------ tensor cores
// bf16 dot-product scores on the 5th-generation tensor cores.  One CTA =
// one head x 128 MMA rows (64 tokens x 2 branches when fused, 128 tokens of
// one branch for scores only).  Both halves' contractions (128 x d_h by
// d_h x s, fp32 accumulate) are issued by one thread into 2 x 256 tensor-
// memory columns; rows are then staged 32 at a time through padded shared
// memory for the warp selection and merge above.
constexpr int kTcRows = 128;
constexpr int kTcThreads = 1024;

struct TcLayout {
  size_t a, b, sc, lv, lid, ws, stair, nst, bar, tslot, th, cut, total;
  int spad, scs;
};

__host__ __device__ inline TcLayout tc_layout(int s, int dh) {
  TcLayout L;
  L.spad = (s + 15) & ~15;     // MMA N
  L.scs = L.spad + 4;          // staged row stride in floats (16-byte rows, no bank conflicts)
  // The MMA operands are dead once the MMA has completed, before any
  // selection starts: the warps' selection scratch overlays them.
  size_t o = 0;
  L.a = o;     o = align_up(o + (size_t)2 * kTcRows * dh * 2, 1024);
  L.b = o;     o = align_up(o + (size_t)2 * L.spad * dh * 2, 1024);
  L.ws = 0;
  o = align_up(o > sizeof(WarpScratch) * (kTcThreads / 32) ? o
                                                          : sizeof(WarpScratch) * (kTcThreads / 32),
               1024);
  L.sc = o;    o = align_up(o + sizeof(float) * 2 * 32 * (size_t)L.scs, 16);   // both halves
  L.lv = o;    o = align_up(o + sizeof(float) * 32 * 2 * kMaxSel, 16);
  L.lid = o;   o = align_up(o + sizeof(uint32_t) * 32 * 2 * kMaxSel, 16);
  L.stair = o; o = align_up(o + sizeof(uint16_t) * 2 * kStairMax, 16);
  L.nst = o;   o = align_up(o + sizeof(int) * 2, 16);
  L.bar = o;   o = align_up(o + sizeof(uint64_t), 16);
  L.tslot = o; o = align_up(o + sizeof(uint32_t), 16);
  L.th = o;    o = align_up(o + sizeof(long long) * kTcRows, 16);   // row -> token-head, -1 past the end
  L.cut = o;   o = align_up(o + sizeof(int) * 2 * kMaxSel, 16);     // nsel / (a + 1) per branch
  L.total = o;
  return L;
}

inline bool tc_eligible(const Dims& d) {
  return d.in_dtype == SDM_BF16 && d.score == SDM_SCORE_DOT && d.s <= 256 && d.dh <= 64 &&
         d.dh % 16 == 0 && (d.dh & (d.dh - 1)) == 0 &&
         tc_layout(d.s, d.dh).total <= device_limits().smem_per_cta;
}

template <int MODE>
__device__ __forceinline__ void tc_row_item(int r, int& sigma, long long& item) {
  if (MODE == kAddrScoresOnly) {
    sigma = 0;
    item = (long long)blockIdx.x * kTcRows + r;
  } else {
    sigma = r >> 6;
    item = (long long)blockIdx.x * (kTcRows / 2) + (r & 63);
  }
}

template <int MODE>
__global__ void __launch_bounds__(kTcThreads, 1) address_tc_kernel(const AddrArgs A) {
  extern __shared__ __align__(16) unsigned char smem[];
  const Dims& d = A.d;
  const TcLayout L = tc_layout(d.s, d.dh);
  unsigned char* sA = smem + L.a;
  unsigned char* sB = smem + L.b;
  float* sc = reinterpret_cast<float*>(smem + L.sc);
  float* lv = reinterpret_cast<float*>(smem + L.lv);
  uint32_t* lid = reinterpret_cast<uint32_t*>(smem + L.lid);
  WarpScratch* wsa = reinterpret_cast<WarpScratch*>(smem + L.ws);
  uint16_t* stair = reinterpret_cast<uint16_t*>(smem + L.stair);
  int* nst = reinterpret_cast<int*>(smem + L.nst);
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + L.bar);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(smem + L.tslot);
  long long* rth = reinterpret_cast<long long*>(smem + L.th);
  int* cut = reinterpret_cast<int*>(smem + L.cut);

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int h = blockIdx.y, dh = d.dh, spad = L.spad, scs = L.scs;
  const long long BT = (long long)d.B * d.T;
  const uint32_t ahalf = (uint32_t)kTcRows * dh * 2, bhalf = (uint32_t)spad * dh * 2;
  // Tensor-memory columns: half p's accumulators start at column p * cstride.
  const uint32_t cstride = spad <= 128 ? 128u : 256u, ncols = 2 * cstride;
  WarpScratch& ws = wsa[warp];

  if (warp == 0) tc::tmem_alloc(tslot, ncols);
  if (tid == 32) mbar_init(bar, 1);
  if (MODE != kAddrScoresOnly) {
    if (warp == 2) {
      const int n = build_stair(d.W, d.kw, stair, lane);
      if (lane == 0) nst[0] = n;
    } else if (warp == 3) {
      const int n = build_stair(d.R, d.kr, stair + kStairMax, lane);
      if (lane == 0) nst[1] = n;
    }
  }
  // Token-head of every MMA row (one 64-bit division per row, here only),
  // and the staircase's first excluded b per a for the merge's tie check.
  if (tid < kTcRows) {
    int sg;
    long long item;
    tc_row_item<MODE>(tid, sg, item);
    long long th = -1;
    if (item < BT) {
      const long long b = item / d.T, t = item - b * d.T;
      th = (b * d.H + h) * d.Ts + t;
    }
    rth[tid] = th;
  } else if (tid < kTcRows + 2 * kMaxSel) {
    const int a = tid - kTcRows;
    const int nsel = a < kMaxSel ? d.W : d.R;
    cut[a] = nsel / ((a & (kMaxSel - 1)) + 1);
  }
  __syncthreads();
  // Operands into the K-major core-matrix layout (16-byte chunks); d_h is a
  // power of two here, so the chunk index splits by shifts.
  const int kc = dh / 8, lkc = 31 - __clz(kc);
  for (int e = tid; e < 2 * kTcRows * kc; e += kTcThreads) {
    const int p = e >> (7 + lkc), rem = e & ((kTcRows << lkc) - 1);
    const int r = rem >> lkc, c = rem & (kc - 1);
    const long long th = rth[r];
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (th >= 0) {
      const __nv_bfloat16* q =
          reinterpret_cast<const __nv_bfloat16*>(MODE == kAddrScoresOnly || r < 64 ? A.q0 : A.q1);
      v = __ldg(reinterpret_cast<const uint4*>(q + (size_t)(th * 2 + p) * dh) + c);
    }
    *reinterpret_cast<uint4*>(sA + p * ahalf + tc::kmajor_off(r, 8 * c, dh)) = v;
  }
  for (int e = tid; e < 2 * spad * kc; e += kTcThreads) {
    const int p = e / (spad * kc), rem = e - p * spad * kc;
    const int j = rem >> lkc, c = rem & (kc - 1);
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (j < d.s) {
      const __nv_bfloat16* K = reinterpret_cast<const __nv_bfloat16*>(A.K);
      v = __ldg(reinterpret_cast<const uint4*>(K + ((size_t)(h * 2 + p) * d.s + j) * dh) + c);
    }
    *reinterpret_cast<uint4*>(sB + p * bhalf + tc::kmajor_off(j, 8 * c, dh)) = v;
  }
  tc::fence_smem_to_async();
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *tslot;
  if (tid == 0) {
    const uint32_t idesc = tc::idesc_bf16_f32(kTcRows, spad);
    const uint32_t sbo = (uint32_t)dh * 16;
    for (int p = 0; p < 2; ++p)
      for (int ks = 0; ks < dh / 16; ++ks)
        tc::mma_bf16(tmem + p * cstride,
                     tc::kmajor_desc(smem_u32(sA + p * ahalf) + ks * 256, 128, sbo),
                     tc::kmajor_desc(smem_u32(sB + p * bhalf) + ks * 256, 128, sbo), idesc,
                     ks > 0);
    tc::commit(bar);
  }
  if (!mbar_wait_bounded(bar, 0, 4000000000ull)) {
    record_status(A.status, SDM_ERR_TIMEOUT);
    mbar_wait_bounded(bar, 0, 1000000000ull);   // drain before the operands are reused
  }
  tc::fence_after_sync();
  tc::fence_smem_to_async();

  if (MODE == kAddrScoresOnly) {
    // Warps 0-3: half 0, warps 4-7: half 1; lane = row.
    const int g = warp & 3, p = (warp >> 2) & 1;
    const int r = 32 * g + lane;
    const long long th = rth[r];
    // Warps 8w .. 8w+7 take every (kTcThreads / 256)-th block of 16 columns.
    for (int c0 = 16 * (warp >> 3); c0 < spad; c0 += 16 * (kTcThreads / 256)) {
      float v[16];
      tc::ld16(tmem + ((uint32_t)(32 * g) << 16) + p * cstride + c0, v);
      if (th >= 0)
        for (int i = 0; i < 16; ++i)
          if (c0 + i < d.s) A.S[(size_t)(th * 2 + p) * d.s + c0 + i] = v[i];
    }
  } else {
    // Per group of 32 rows: the warps that own the group's tensor-memory lanes
    // stage both halves' scores, then every warp runs one row end to end (both
    // half top-k, merge, softmax) with no block barrier in between.
    const int nblk = spad / 16;
    for (int g = 0; g < 4; ++g) {
      if ((warp & 3) == g) {
        for (int e = warp >> 2; e < 2 * nblk; e += kTcThreads / 128) {
          const int p = e >= nblk, blk = e - p * nblk;
          float v[16];
          tc::ld16(tmem + ((uint32_t)(32 * g) << 16) + p * cstride + 16 * blk, v);
          float4* dst = reinterpret_cast<float4*>(sc + (size_t)(p * 32 + lane) * scs + 16 * blk);
          dst[0] = make_float4(v[0], v[1], v[2], v[3]);
          dst[1] = make_float4(v[4], v[5], v[6], v[7]);
          dst[2] = make_float4(v[8], v[9], v[10], v[11]);
          dst[3] = make_float4(v[12], v[13], v[14], v[15]);
        }
      }
      __syncthreads();
      for (int rr = warp; rr < 32; rr += kTcThreads / 32) {
        const long long th = rth[32 * g + rr];
        if (th < 0) continue;
        const int sg = g >> 1;                   // rows 0-63 write, 64-127 read
        const int k = sg == 0 ? d.kw : d.kr;
        const int nsel = sg == 0 ? d.W : d.R;
        float* ov = lv + rr * 2 * kMaxSel;
        uint32_t* oi = lid + rr * 2 * kMaxSel;
#pragma unroll 1
        for (int p = 0; p < 2; ++p) {
          RowSrc src{sc + (size_t)(p * 32 + rr) * scs};
          warp_topk<8>(src, d.s, k, ws, lane);   // s <= 256 here
          for (int e = lane; e < k; e += 32) {
            ov[p * kMaxSel + e] = ws.out_v[e];
            oi[p * kMaxSel + e] = ws.out_id[e];
          }
          __syncwarp();
        }
        warp_merge(ov, oi, ov + kMaxSel, oi + kMaxSel, k, nsel, (uint32_t)d.s,
                   stair + sg * kStairMax, nst[sg], ws, lane, cut + sg * kMaxSel);
        int32_t* io = (sg == 0 ? A.idx_w : A.idx_r) + (size_t)th * nsel;
        float* wo = (sg == 0 ? A.wt_w : A.wt_r) + (size_t)th * nsel;
        warp_softmax_store(ws, nsel, io, wo, lane);
        __syncwarp();
      }
      __syncthreads();
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 0) tc::tmem_dealloc(tmem, ncols);
}

template <int MODE>
cudaError_t launch_tc(const AddrArgs& A, cudaStream_t stream) {
  const TcLayout L = tc_layout(A.d.s, A.d.dh);
  auto kfn = address_tc_kernel<MODE>;
  cudaError_t e = cudaFuncSetAttribute(kfn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)L.total);
  if (e != cudaSuccess) return e;
  const long long BT = (long long)A.d.B * A.d.T;
  const int per = MODE == kAddrScoresOnly ? kTcRows : kTcRows / 2;
  const long long tiles = (BT + per - 1) / per;
  if (tiles == 0 || A.d.H == 0) return cudaSuccess;
  dim3 grid((unsigned)tiles, (unsigned)A.d.H);
  kfn<<<grid, kTcThreads, L.total, stream>>>(A);
  return cudaGetLastError();
}

template <int MODE>
cudaError_t launch_mode(const AddrArgs& A, cudaStream_t stream) {
  if (tc_eligible(A.d)) return launch_tc<MODE>(A, stream);
  const bool bf = A.d.in_dtype == SDM_BF16;
  if (A.d.score == SDM_SCORE_DOT)
    return bf ? launch_t<MODE, true, SDM_SCORE_DOT>(A, stream)
              : launch_t<MODE, false, SDM_SCORE_DOT>(A, stream);
  return bf ? launch_t<MODE, true, SDM_SCORE_IDW>(A, stream)
            : launch_t<MODE, false, SDM_SCORE_IDW>(A, stream);
}

}  // namespace

bool address_on_tensor_cores(const Dims& d) { return tc_eligible(d); }

cudaError_t launch_address(int mode, const Dims& d, const void* q0, const void* q1,
                           const void* K, const float* f0, const float* f1,
                           int32_t* idx_w, float* wt_w, int32_t* idx_r, float* wt_r,
                           float* S, unsigned* status, cudaStream_t stream) {
  AddrArgs A{d, q0, q1, K, f0, f1, idx_w, wt_w, idx_r, wt_r, S, status};
  switch (mode) {
    case kAddrFused: return launch_mode<kAddrFused>(A, stream);
    case kAddrSelectOnly:
      // Sub-scores are given: dtype and score kind do not matter.
      return launch_t<kAddrSelectOnly, false, SDM_SCORE_DOT>(A, stream);
    case kAddrScoresOnly: return launch_mode<kAddrScoresOnly>(A, stream);
  }
  return cudaErrorInvalidValue;
}

}  // namespace sdm
