// decode.cu -- one fused launch for short sequences (decode, T = 1).
//
// [SDM notes] "Sparse Delta Memory：中文精读笔记": 2.3 (product-key addressing),
// 2.4 Eq. (3)-(5) (gated delta write, read after the write; after Eq. (5) the
// per-head RMS-Norm and output gate), 2.5 (the Fig. 2 shared-residual form).
// The notes' section 3 reports decode speed as the inference number, and
// 2.8 gives the per-head shapes it runs at (sqrt N = 240 / 480, d_v = 960 /
// 1920 with 2 heads).
//
// A decode step has little work per chain but a long dependent path
// (scores -> top-k -> merge -> write -> read), so the tile kernels used for
// long sequences spend most of it waiting.  Here P CTAs own one (b, h)
// chain, each a 1/P range of its columns (P > 1 when there are too few
// chains to fill the GPU: the write and read act column by column, so the
// parts share nothing but the selection, which each part computes itself),
// and run its T steps in order, each step entirely on chip:
//   scores    FFMA (or inverse distance) of the four half-queries against
//             the two sub-key tables, into shared memory;
//   top-k     four groups of four warps, one half-row each, and
//   merge     two groups of eight warps, one branch each (staircase merge +
//             softmax): the bucketed exact selection of select.cuh shared by
//             a group's warps on a named barrier, with the warp paths as the
//             exact fallback;
//   write     every thread owns a 16-byte column chunk and a row group and
//             walks its W write rows in register batches, so the row loads
//             of a batch are in flight together; Fig. 2 form: a first pass
//             sums the shared prediction, a second writes;
//   read      after a block barrier (the CTA's own global writes are then
//             visible to all its threads) the R read rows, batched the same
//             way; optionally the RMS-Norm + gate epilogue, whose row sum of
//             squares is a block reduction, plus, for P > 1, a sum of the
//             parts' shares over distributed shared memory (the P CTAs of a
//             chain are one thread-block cluster).
// The table is read with plain (coherent) loads: the CTA rewrites it.
#include "common.cuh"
#include "internal.h"
#include "select.cuh"

namespace sdm {
namespace {

constexpr int kDecThreads = 512;
constexpr int kDecWarps = kDecThreads / 32;
constexpr int kStairCap = 320;   // >= sum_{a<64} floor(64/(a+1)) = 280
constexpr int kBatch = 8;        // table rows in flight per thread

struct DecArgs {
  Dims d;
  const void* q_w;
  const void* q_r;
  const void* K;
  const void* alpha;
  const void* beta;
  const void* v;
  float* M;
  float* y;
  int32_t* idx_w;
  float* wt_w;
  int32_t* idx_r;
  float* wt_r;
  const void* g;        // epilogue gate [B,H,T,d_v] (in_dtype) or null
  const float* gamma;   // [H,d_v] or null
  void* out;            // epilogue output or null (no epilogue)
  float eps;
  int out_dtype;
  int P;                // CTAs (column parts) per chain; a cluster when out != null
};

struct DecLayout {
  size_t q, S, lv, lid, ws, gs, stair, nst, sel, red, part, total;
};

__host__ __device__ inline size_t dl_align(size_t x) { return (x + 15) / 16 * 16; }

__host__ __device__ inline DecLayout dec_layout(int s, int dh) {
  DecLayout L;
  size_t o = 0;
  L.q = o;     o = dl_align(o + sizeof(float) * 4 * (size_t)dh);
  L.S = o;     o = dl_align(o + sizeof(float) * 4 * (size_t)s);
  L.lv = o;    o = dl_align(o + sizeof(float) * 4 * kMaxSel);
  L.lid = o;   o = dl_align(o + sizeof(uint32_t) * 4 * kMaxSel);
  L.ws = o;    o = dl_align(o + sizeof(WarpScratch) * 4);
  L.gs = o;    o = dl_align(o + sizeof(GroupScratch) * 4);
  L.stair = o; o = dl_align(o + sizeof(uint16_t) * 2 * kStairCap);
  L.nst = o;   o = dl_align(o + sizeof(int) * 2);
  L.sel = o;   o = dl_align(o + sizeof(float) * 4 * kMaxSel);   // idx_w, wt_w, idx_r, wt_r
  L.red = o;   o = dl_align(o + sizeof(float) * (kDecWarps + 1));   // + this part's share
  L.part = o;  o = dl_align(o + sizeof(float) * 4 * kDecThreads);   // row-group partials
  L.total = o;
  return L;
}

template <bool BF16>
__device__ __forceinline__ float4 ld_in4(const void* base, size_t i4) {
  if (BF16) {
    const uint2 w = __ldg(reinterpret_cast<const uint2*>(base) + i4);
    return make_float4(bf16_bits_to_float(w.x & 0xffffu), bf16_bits_to_float(w.x >> 16),
                       bf16_bits_to_float(w.y & 0xffffu), bf16_bits_to_float(w.y >> 16));
  }
  return __ldg(reinterpret_cast<const float4*>(base) + i4);
}

__device__ __forceinline__ void st_out4(void* base, size_t i4, int dt, float4 v) {
  if (dt == SDM_F32) {
    reinterpret_cast<float4*>(base)[i4] = v;
    return;
  }
  const __nv_bfloat162 a = __floats2bfloat162_rn(v.x, v.y);
  const __nv_bfloat162 b = __floats2bfloat162_rn(v.z, v.w);
  uint2 w;
  w.x = *reinterpret_cast<const uint32_t*>(&a);
  w.y = *reinterpret_cast<const uint32_t*>(&b);
  reinterpret_cast<uint2*>(base)[i4] = w;
}

// 16 consecutive input elements (bf16 or fp32) from element e (a multiple of
// 16), all loads issued before any is used.
template <bool BF16>
__device__ __forceinline__ void ld_in16(const void* base, size_t e, float (&k)[16]) {
  if (BF16) {
    const uint4* p = reinterpret_cast<const uint4*>(base) + e / 8;
    const uint4 a = __ldg(p), b = __ldg(p + 1);
    const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      k[2 * i] = bf16_bits_to_float(w[i] & 0xffffu);
      k[2 * i + 1] = bf16_bits_to_float(w[i] >> 16);
    }
  } else {
    const float4* p = reinterpret_cast<const float4*>(base) + e / 4;
    float4 v[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) v[i] = __ldg(p + i);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      k[4 * i] = v[i].x;
      k[4 * i + 1] = v[i].y;
      k[4 * i + 2] = v[i].z;
      k[4 * i + 3] = v[i].w;
    }
  }
}

// Element e of a dh-long input vector (bf16 or fp32) as float.
template <bool BF16>
__device__ __forceinline__ float ld_in1(const void* base, size_t e) {
  if (BF16) return bf16_bits_to_float(__ldg(reinterpret_cast<const unsigned short*>(base) + e));
  return __ldg(reinterpret_cast<const float*>(base) + e);
}

template <int PL, bool BF16, int KIND>
__global__ void __launch_bounds__(kDecThreads, 1) decode_kernel(const DecArgs A) {
  extern __shared__ __align__(16) unsigned char smem[];
  const Dims& d = A.d;
  const DecLayout L = dec_layout(d.s, d.dh);
  float* qs = reinterpret_cast<float*>(smem + L.q);
  float* S = reinterpret_cast<float*>(smem + L.S);
  float* lv = reinterpret_cast<float*>(smem + L.lv);
  uint32_t* lid = reinterpret_cast<uint32_t*>(smem + L.lid);
  WarpScratch* wsa = reinterpret_cast<WarpScratch*>(smem + L.ws);
  GroupScratch* gsa = reinterpret_cast<GroupScratch*>(smem + L.gs);
  uint16_t* stair = reinterpret_cast<uint16_t*>(smem + L.stair);
  int* nst = reinterpret_cast<int*>(smem + L.nst);
  int32_t* sidx = reinterpret_cast<int32_t*>(smem + L.sel);      // [2][64]
  float* swt = reinterpret_cast<float*>(smem + L.sel) + 2 * kMaxSel;
  float* red = reinterpret_cast<float*>(smem + L.red);
  float4* part = reinterpret_cast<float4*>(smem + L.part);

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int chain = blockIdx.x / A.P;        // b * H + h
  const int cpart = blockIdx.x - chain * A.P; // column part = rank in the chain's cluster
  const int h = chain % d.H;
  const int s = d.s, dh = d.dh, dv = d.dv, W = d.W, R = d.R;
  const int nc4 = dv / 4, ncp = nc4 / A.P;   // 16-byte chunks of a row, of this part
  // Write / read work items: (column chunk c4, row group rg); the G row
  // groups of a chunk split its rows and combine partial sums on chip.
  const int G = kDecThreads / ncp;           // >= 1 (d_v <= 2048)
  const int lc = tid % ncp, rg = tid / ncp;
  const int c4 = cpart * ncp + lc;
  const bool worker = rg < G;
  float* Mc = A.M + (size_t)chain * (size_t)d.N() * dv;
  const bool fig2 = d.update == SDM_UPDATE_SHARED_RESIDUAL;

  if (warp == 2) {
    const int n = build_stair(W, d.kw, stair, lane);
    if (lane == 0) nst[0] = n;
  } else if (warp == 3) {
    const int n = build_stair(R, d.kr, stair + kStairCap, lane);
    if (lane == 0) nst[1] = n;
  }

  {
    // The head's sub-key tables, line by line, into L2 for the first scores.
    const size_t kbytes = (size_t)2 * s * dh * (BF16 ? 2 : 4);
    const unsigned char* kb = static_cast<const unsigned char*>(A.K) + (size_t)h * kbytes;
    for (size_t o = (size_t)tid * 128; o < kbytes; o += (size_t)kDecThreads * 128)
      prefetch_l2(kb + o);
  }

  for (int t = 0; t < d.T; ++t) {
    const size_t th = (size_t)chain * d.T + t;
    // ---- half-queries: qs[(sigma * 2 + p) * dh + c]
    for (int e = tid; e < 4 * dh; e += kDecThreads) {
      const int sg = e / (2 * dh), rem = e - sg * 2 * dh;
      qs[e] = ld_in1<BF16>(sg == 0 ? A.q_w : A.q_r, th * 2 * dh + rem);
    }
    __syncthreads();
    // ---- sub-scores S[(sigma * 2 + p) * s + j]: one thread per (p, j) loads
    // sub-key K_p[j] once -- for d_h = 64 in bf16 the whole row in one round
    // trip -- and scores it against both branches' half-queries (read from
    // shared memory four floats at a time).
    for (int e = tid; e < 2 * s; e += kDecThreads) {
      const int p = e / s, j = e - p * s;
      const float* qw = qs + p * dh;           // write branch, half p
      const float* qr = qs + (2 + p) * dh;     // read branch, half p
      const size_t kb = ((size_t)(h * 2 + p) * s + j) * dh;
      float aw = 0.f, ar = 0.f;
      auto acc16 = [&](int c0, const float (&k)[16]) {
#pragma unroll
        for (int i = 0; i < 16; i += 4) {
          const float4 w4 = *reinterpret_cast<const float4*>(qw + c0 + i);
          const float4 r4 = *reinterpret_cast<const float4*>(qr + c0 + i);
          const float wq[4] = {w4.x, w4.y, w4.z, w4.w}, rq[4] = {r4.x, r4.y, r4.z, r4.w};
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            if (KIND == SDM_SCORE_DOT) {
              aw = fmaf(wq[u], k[i + u], aw);
              ar = fmaf(rq[u], k[i + u], ar);
            } else {
              const float dw = wq[u] - k[i + u], dr = rq[u] - k[i + u];
              aw = fmaf(dw, dw, aw);
              ar = fmaf(dr, dr, ar);
            }
          }
        }
      };
      if (BF16 && dh == 64) {
        float k0[16], k1[16], k2[16], k3[16];
        ld_in16<BF16>(A.K, kb, k0);
        ld_in16<BF16>(A.K, kb + 16, k1);
        ld_in16<BF16>(A.K, kb + 32, k2);
        ld_in16<BF16>(A.K, kb + 48, k3);
        acc16(0, k0);
        acc16(16, k1);
        acc16(32, k2);
        acc16(48, k3);
      } else {
#pragma unroll 2
        for (int c0 = 0; c0 < dh; c0 += 16) {
          float k[16];
          ld_in16<BF16>(A.K, kb + c0, k);
          acc16(c0, k);
        }
      }
      S[p * s + j] = KIND == SDM_SCORE_DOT ? aw : -logf(d.eps + aw);
      S[(2 + p) * s + j] = KIND == SDM_SCORE_DOT ? ar : -logf(d.eps + ar);
    }
    __syncthreads();
    // ---- per-half top-k: warps 4g .. 4g+3 take half-row g = sigma * 2 + p
    // together (named barrier 1 + g); the warp paths remain for the rows the
    // buckets cannot decide.
    {
      const int g = warp >> 2, gt = tid & 127;
      const int k = (g >> 1) == 0 ? d.kw : d.kr;
      RowSrc src{S + g * s};
      const float* ov = gsa[g].out_v;
      const uint32_t* oi = gsa[g].out_id;
      if (!group_topk_bucketed<4, PL / 4>(src, s, k, gsa[g], gt, 1 + g)) {
        if ((warp & 3) == 0) warp_topk_sorted(src, s, k, wsa[g], lane);
        named_bar_sync(1 + g, 128);
        ov = wsa[g].out_v;
        oi = wsa[g].out_id;
      }
      for (int e = gt; e < k; e += 128) {
        lv[g * kMaxSel + e] = ov[e];
        lid[g * kMaxSel + e] = oi[e];
      }
    }
    __syncthreads();
    // ---- merge + softmax: warps 8 sigma .. 8 sigma + 7 rank the staircase
    // pairs of branch sigma together (named barrier 5 + sigma); a tie at the
    // W-th sum, or rows the buckets cannot decide, take the warp merge.
    {
      const int sg = warp >> 3, gt = tid & 255;
      const int k = sg == 0 ? d.kw : d.kr, nsel = sg == 0 ? W : R;
      const float* v1 = lv + (2 * sg) * kMaxSel;
      const uint32_t* i1 = lid + (2 * sg) * kMaxSel;
      const float* v2 = lv + (2 * sg + 1) * kMaxSel;
      const uint32_t* i2 = lid + (2 * sg + 1) * kMaxSel;
      GroupScratch& gs = gsa[sg];
      PairSrc ps{v1, i1, v2, i2, stair + sg * kStairCap, (uint32_t)s};
      bool ok = group_topk_bucketed<8, 2>(ps, nst[sg], nsel, gs, gt, 5 + sg);
      bool tie = false;
      if (ok && gt < k) {
        const int b = nsel / (gt + 1);
        tie = b < k && __fadd_rn(v1[gt], v2[b]) >= gs.out_v[nsel - 1];
      }
      ok = !named_bar_or(5 + sg, 256, !ok || tie);
      if ((warp & 7) == 0) {
        const float* ov = gs.out_v;
        const uint32_t* oi = gs.out_id;
        if (!ok) {
          warp_merge(v1, i1, v2, i2, k, nsel, (uint32_t)s, stair + sg * kStairCap, nst[sg],
                     wsa[sg], lane);
          ov = wsa[sg].out_v;
          oi = wsa[sg].out_id;
        }
        softmax_store(ov, oi, nsel, sidx + sg * kMaxSel, swt + sg * kMaxSel, lane);
        __syncwarp();
        int32_t* io = (sg == 0 ? A.idx_w : A.idx_r) + th * nsel;
        float* wo = (sg == 0 ? A.wt_w : A.wt_r) + th * nsel;
        if (cpart == 0)
          for (int e = lane; e < nsel; e += 32) {
            io[e] = sidx[sg * kMaxSel + e];
            wo[e] = swt[sg * kMaxSel + e];
          }
      }
    }
    __syncthreads();

    // ---- write (Eq. (3)-(4), or the Fig. 2 form): group rg takes rows
    // j = rg, rg + G, ...; the Fig. 2 prediction is summed over the groups.
    const float a = load_scalar(A.alpha, th, d.in_dtype);
    const float bt = load_scalar(A.beta, th, d.in_dtype);
    float4 vv = make_float4(0.f, 0.f, 0.f, 0.f), res = vv;
    if (worker) {
      vv = ld_in4<BF16>(A.v, th * nc4 + c4);
      res = vv;
    }
    if (fig2) {
      float4 vh = make_float4(0.f, 0.f, 0.f, 0.f);
      if (worker) {
        for (int j0 = rg; j0 < W; j0 += kBatch * G) {
          float4 x[kBatch];
#pragma unroll
          for (int u = 0; u < kBatch; ++u)
            if (j0 + u * G < W)
              x[u] = reinterpret_cast<const float4*>(Mc + (size_t)sidx[j0 + u * G] * dv)[c4];
#pragma unroll
          for (int u = 0; u < kBatch; ++u)
            if (j0 + u * G < W) {
              const float wj = swt[j0 + u * G];
              vh.x = fmaf(wj, a * x[u].x, vh.x);
              vh.y = fmaf(wj, a * x[u].y, vh.y);
              vh.z = fmaf(wj, a * x[u].z, vh.z);
              vh.w = fmaf(wj, a * x[u].w, vh.w);
            }
        }
        part[rg * ncp + lc] = vh;
      }
      __syncthreads();
      if (worker) {
        vh = part[lc];
        for (int g2 = 1; g2 < G; ++g2) {
          const float4 p2 = part[g2 * ncp + lc];
          vh.x += p2.x;
          vh.y += p2.y;
          vh.z += p2.z;
          vh.w += p2.w;
        }
        res = make_float4(vv.x - vh.x, vv.y - vh.y, vv.z - vh.z, vv.w - vh.w);
      }
      __syncthreads();
    }
    if (worker) {
      for (int j0 = rg; j0 < W; j0 += kBatch * G) {
        float4 x[kBatch];
#pragma unroll
        for (int u = 0; u < kBatch; ++u)
          if (j0 + u * G < W)
            x[u] = reinterpret_cast<const float4*>(Mc + (size_t)sidx[j0 + u * G] * dv)[c4];
#pragma unroll
        for (int u = 0; u < kBatch; ++u)
          if (j0 + u * G < W) {
            const float cw = bt * swt[j0 + u * G];
            float4 o;
            float m;
            if (fig2) {
              m = a * x[u].x; o.x = fmaf(cw, res.x, m);
              m = a * x[u].y; o.y = fmaf(cw, res.y, m);
              m = a * x[u].z; o.z = fmaf(cw, res.z, m);
              m = a * x[u].w; o.w = fmaf(cw, res.w, m);
            } else {
              m = a * x[u].x; o.x = fmaf(cw, vv.x - m, m);
              m = a * x[u].y; o.y = fmaf(cw, vv.y - m, m);
              m = a * x[u].z; o.z = fmaf(cw, vv.z - m, m);
              m = a * x[u].w; o.w = fmaf(cw, vv.w - m, m);
            }
            reinterpret_cast<float4*>(Mc + (size_t)sidx[j0 + u * G] * dv)[c4] = o;
          }
      }
    }
    __syncthreads();

    // ---- read after the write (Eq. (5)): group partials, summed by group 0;
    // then the optional epilogue on the whole row.
    if (worker) {
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
      for (int q0 = rg; q0 < R; q0 += kBatch * G) {
        float4 x[kBatch];
#pragma unroll
        for (int u = 0; u < kBatch; ++u)
          if (q0 + u * G < R)
            x[u] = reinterpret_cast<const float4*>(
                Mc + (size_t)sidx[kMaxSel + q0 + u * G] * dv)[c4];
#pragma unroll
        for (int u = 0; u < kBatch; ++u)
          if (q0 + u * G < R) {
            const float w = swt[kMaxSel + q0 + u * G];
            acc.x = fmaf(w, x[u].x, acc.x);
            acc.y = fmaf(w, x[u].y, acc.y);
            acc.z = fmaf(w, x[u].z, acc.z);
            acc.w = fmaf(w, x[u].w, acc.w);
          }
      }
      part[rg * ncp + lc] = acc;
    }
    __syncthreads();
    float4 yv = make_float4(0.f, 0.f, 0.f, 0.f);
    float ss = 0.f;
    if (rg == 0) {
      yv = part[lc];
      for (int g2 = 1; g2 < G; ++g2) {
        const float4 p2 = part[g2 * ncp + lc];
        yv.x += p2.x;
        yv.y += p2.y;
        yv.z += p2.z;
        yv.w += p2.w;
      }
      reinterpret_cast<float4*>(A.y + th * dv)[c4] = yv;
      ss = fmaf(yv.x, yv.x, ss);
      ss = fmaf(yv.y, yv.y, ss);
      ss = fmaf(yv.z, yv.z, ss);
      ss = fmaf(yv.w, yv.w, ss);
    }
    if (A.out) {
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
      if (lane == 0) red[warp] = ss;
      __syncthreads();
      float tot = 0.f;
#pragma unroll
      for (int w = 0; w < kDecWarps; ++w) tot += red[w];
      if (A.P > 1) {
        // Sum the parts' shares: each part publishes its own, the cluster
        // barrier orders them, every thread reads all P from distributed
        // shared memory, and a second barrier keeps each share in place
        // until every part has read it.
        if (tid == 0) red[kDecWarps] = tot;
        cluster_sync();
        tot = 0.f;
        const uint32_t mine = smem_u32(red + kDecWarps);
        for (int r = 0; r < A.P; ++r) tot += ld_cluster_f32(map_cluster(mine, (uint32_t)r));
        cluster_sync();
      }
      const float inv = 1.f / sqrtf(tot / (float)dv + A.eps);
      if (rg == 0) {
        const float4 gt = ld_in4<BF16>(A.g, th * nc4 + c4);
        const float4 sc = A.gamma ? __ldg(reinterpret_cast<const float4*>(A.gamma) +
                                          (size_t)h * nc4 + c4)
                                  : make_float4(1.f, 1.f, 1.f, 1.f);
        st_out4(A.out, th * nc4 + c4, A.out_dtype,
                make_float4(yv.x * inv * sc.x * gt.x, yv.y * inv * sc.y * gt.y,
                            yv.z * inv * sc.z * gt.z, yv.w * inv * sc.w * gt.w));
      }
    }
    __syncthreads();
  }
}

template <int PL, bool BF16, int KIND>
cudaError_t launch_dec(const DecArgs& A, cudaStream_t stream) {
  const size_t smem = dec_layout(A.d.s, A.d.dh).total;
  auto kfn = decode_kernel<PL, BF16, KIND>;
  cudaError_t e =
      cudaFuncSetAttribute(kfn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const unsigned grid = (unsigned)(A.d.B * A.d.H * A.P);
  if (A.P > 1 && A.out) {
    // The epilogue's row norm spans the parts: they launch as one cluster.
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kDecThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = (unsigned)A.P;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, kfn, A);
    if (e != cudaSuccess) return e;
  } else {
    kfn<<<grid, kDecThreads, smem, stream>>>(A);
  }
  return cudaGetLastError();
}

template <int PL>
cudaError_t launch_pl(const DecArgs& A, cudaStream_t stream) {
  const bool bf = A.d.in_dtype == SDM_BF16;
  if (A.d.score == SDM_SCORE_DOT)
    return bf ? launch_dec<PL, true, SDM_SCORE_DOT>(A, stream)
              : launch_dec<PL, false, SDM_SCORE_DOT>(A, stream);
  return bf ? launch_dec<PL, true, SDM_SCORE_IDW>(A, stream)
            : launch_dec<PL, false, SDM_SCORE_IDW>(A, stream);
}

}  // namespace

cudaError_t launch_decode(const Dims& d, const void* q_w, const void* q_r, const void* K,
                          const void* alpha, const void* beta, const void* v, float* M, float* y,
                          int32_t* idx_w, float* wt_w, int32_t* idx_r, float* wt_r,
                          const void* g, const float* gamma, float eps, void* out,
                          int out_dtype, cudaStream_t stream) {
  const long long chains = (long long)d.B * d.H;
  if (chains == 0 || d.T == 0) return cudaSuccess;
  // Column parts per chain: as many as keep one CTA per SM busy (a CTA of
  // 512 threads at up to 128 registers is alone on its SM), each part at
  // least 32 chunks of 16 bytes wide.
  const long long sms = device_limits().sms;
  const int nc4 = d.dv / 4;
  int P = 1;
  for (int p = 2; p <= 8; p *= 2)
    if (chains * p <= sms && nc4 % p == 0 && nc4 / p >= 32) P = p;
  DecArgs A{d, q_w, q_r, K, alpha, beta, v, M, y, idx_w, wt_w, idx_r, wt_r,
            g, gamma, out, eps, out_dtype, P};
  return d.s <= 256 ? launch_pl<8>(A, stream) : launch_pl<16>(A, stream);
}

}  // namespace sdm
