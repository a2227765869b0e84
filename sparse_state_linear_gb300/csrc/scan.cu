// scan.cu -- the sparse gated delta write and the read, sequential in t.
//
// [SDM notes] "Sparse Delta Memory：中文精读笔记", 2.4, Eq. (3)-(5): for each
// selected write slot i, M~[i] = alpha_t M[i] and
// M[i] = M~[i] + beta_t w_i (v_t - M~[i]); other rows are untouched; then
// y_t = sum_{i in read set} q_i M_t[i] reads the table after the write.
//
// The Fig. 2 reading of the write ([SDM notes] 2.5) is the second update
// form: the decayed rows' weighted sum vhat = sum_j w_j M~[j] is one
// prediction shared by the write set, M[i] = M~[i] + beta_t w_i (v_t - vhat).
// It needs the whole write set before any row is written: on 32-float
// slices the consumers then own column chunks of every row (a warp
// reduction, see COL below), on other widths one more block reduction per
// step.
//
// With an undo log ([SDM notes] 2.9, appendix A.3: the backward pass
// restores earlier states by undoing the in-place sparse writes), the scan
// also stores each write row's value from just before its step's write;
// undo.cu puts a segment's logged rows back.
//
// Parallel units: (chain = (b,h), column slice of CW floats).  The update
// acts column by column with per-row scalars, so slices of one chain never
// communicate, and a step's write slots are distinct, so no atomics.
//
// launch_scan runs the hazard plan (plan.cu: for every row a step touches,
// whether its current value is the fetched copy or the on-chip copy a step
// still in flight left, and where) and then scan_kernel.  A unit has 8
// consumer warps, 1 producer warp and 4 loader warps (6 where each unit has
// an SM of its own).  Where two units share an SM, one CTA runs both units
// side by side (separate warps, shared-memory partitions and named
// barriers), so the launch occupies exactly units / 2 SMs and leaves the
// rest to concurrent work; otherwise one CTA per unit.
//  * The producer copies each step's slot lists, weights, plan codes and
//    value slice into a ring of metadata slots (cp.async, several steps
//    ahead) and adds the gates; it does nothing else, so its per-step work
//    stays short.
//  * The loaders fetch the rows of step u once its metadata is published and
//    the consumers have finished step u - depth (cp.async, 16 B per lane,
//    coalesced per row slice; only rows whose current value is in HBM), so
//    depth steps of row traffic are in flight per unit; completion is an
//    mbarrier arrive by the copies themselves.
//  * A consumer step: test the step's rows and metadata barriers (where two
//    units share an SM, one warp tests while the others sleep in a named
//    barrier; otherwise every warp tests, while the previous step's read sum
//    is reduced over the lanes), decay + delta on the write rows (kept on
//    chip for forwarding, stored to HBM), ONE block barrier, weighted read;
//    one warp sums the warps' partials of step t after the next barrier.
//  * Rings: write tiles 2 * depth - 1 (the oldest step a consumer may
//    forward from to the newest a loader may be filling), read tiles depth,
//    metadata depth + prefetch + batch + slack.
//  Every wait is bounded (seconds); a wait that runs out records
//  SDM_ERR_TIMEOUT in the status word and the CTA leaves cleanly.
#include "common.cuh"
#include "internal.h"

namespace sdm {
namespace {

// Consumer threads (the Fig. 2 column layout needs 8 warps: one per 16-byte
// chunk of a 32-float slice; it only runs in the MINB = 2 build).
template <int MINB>
__host__ __device__ constexpr int consumer_threads() { return 256; }
// Loader threads that fetch the rows: 4 warps where two CTAs share an SM
// (issue slots are scarce there), 6 where a unit has the SM to itself.
template <int MINB>
__host__ __device__ constexpr int loader_threads() { return MINB == 1 ? 192 : 128; }
template <int MINB>
__host__ __device__ constexpr int scan_threads() {
  return consumer_threads<MINB>() + 32 + loader_threads<MINB>();
}
// Producer's metadata prefetch distance (steps): the copies of a step are
// waited for kP steps after they were issued, so at most kP steps' metadata
// is in flight; their latency (microseconds under load) over kP bounds the
// step rate.  Deep where a CTA has an SM of its own (shared memory to
// spare), shallow where two CTAs share one.
template <int MINB>
__host__ __device__ constexpr int prefetch_steps() { return MINB == 1 ? 16 : 4; }
constexpr int kPrefetchBatch = 4;   // steps the producer handles per loop pass
constexpr int kSlack = 2;        // steps the producer may prepare beyond the need
constexpr uint64_t kTimeoutNs = 4000000000ull;

// One step's metadata.  Every array starts on a 16-byte boundary (16-byte
// cp.async destinations).
struct MetaSlot {
  int32_t idx_w[64];
  float wt_w[64];
  int32_t idx_r[64];
  float wt_r[64];
  int16_t code[128];      // plan codes: W write rows then R read rows
  unsigned char vraw[256];
  float alpha, beta, pad0, pad1;
};
static_assert(sizeof(MetaSlot) == 1552, "meta slot size");

struct ScanArgs {
  Dims d;
  const int32_t* idx_w;
  const float* wt_w;
  const int32_t* idx_r;
  const float* wt_r;
  const void* alpha;
  const void* beta;
  const void* v;
  const int16_t* codes;
  float* M;
  float* y;
  float* undo;      // optional log of the pre-write rows [B,H,T,W,d_v]
  int depth;
  unsigned* status;
};

struct ScanLayout {
  size_t meta, wtile, rtile, ypart, vpart, bars, total;
  int NS, MR;
};

__host__ __device__ inline ScanLayout scan_layout(int CW, int W, int R, int D, int kP,
                                                  bool fig2) {
  ScanLayout L;
  // Write tiles live from the oldest step a consumer may forward from
  // (t - D + 1) to the newest a loader may be filling (t + D - 1).
  L.NS = 2 * D - 1;
  L.MR = D + kP + kPrefetchBatch + kSlack;
  size_t o = 0;
  L.meta = o;  o += sizeof(MetaSlot) * L.MR;
  L.wtile = o; o += sizeof(float) * (size_t)L.NS * W * CW;
  L.rtile = o; o += sizeof(float) * (size_t)D * R * CW;
  L.ypart = o; o += sizeof(float) * 2 * 8 * CW;
  L.vpart = o;                                    // per-warp partials of vhat (Fig. 2 form)
  if (fig2) o += sizeof(float) * 8 * CW;
  L.bars = o;  o += sizeof(uint64_t) * (2 * L.MR + D);
  L.total = o;
  return L;
}


// Bytes between the shared-memory partitions of the units of one CTA.
__host__ __device__ inline size_t unit_smem_stride(size_t total) { return (total + 127) & ~(size_t)127; }

template <bool BF16>
__device__ __forceinline__ float4 load_v4(const unsigned char* vraw, int c) {
  if (BF16) {
    const uint2 w = *reinterpret_cast<const uint2*>(vraw + 8 * c);
    return make_float4(bf16_bits_to_float(w.x & 0xffffu), bf16_bits_to_float(w.x >> 16),
                       bf16_bits_to_float(w.y & 0xffffu), bf16_bits_to_float(w.y >> 16));
  }
  return *reinterpret_cast<const float4*>(vraw + 16 * c);
}

// Ring position that advances by one step at a time (no division).
struct Ring {
  int i, n;
  unsigned phase;
  __device__ __forceinline__ void next() {
    if (++i == n) {
      i = 0;
      phase ^= 1u;
    }
  }
};

// MINB: units per SM the build is sized for (2 on the bandwidth-bound
// workloads; 1 where every unit has an SM of its own and the per-step
// latency decides, which leaves the compiler twice the registers).
// PAIR: units per CTA.  With PAIR = 2 a CTA runs two independent units side
// by side (each with its own warps, shared-memory partition and named
// barriers), so a launch of U units occupies exactly U / 2 SMs and leaves
// the others free for concurrent work (the addressing of the next segment).
// WR: 0, or the write and read set size when both are that (64 on the
// GDN-matched shapes), fixed at compile time so the per-row bounds fold away.
template <int CW, bool BF16, bool FIG2, bool UNDO, int MINB, int PAIR, int WR = 0>
__global__ void __launch_bounds__(scan_threads<MINB>() * PAIR, PAIR == 2 ? 1 : MINB)
    scan_kernel(const ScanArgs A) {
  constexpr int kLoaders = loader_threads<MINB>();
  constexpr int kConsumers = consumer_threads<MINB>();
  constexpr int kCW = kConsumers / 32;     // consumer warps
  static_assert(!FIG2 || kCW == 8, "the Fig. 2 layouts assume 8 consumer warps");
  constexpr int CH = CW / 4;               // 16-byte chunks per row slice
  constexpr int RP = kConsumers / CH;      // rows per consumer pass
  constexpr int IB = BF16 ? 2 : 4;         // input element bytes
  // Fig. 2 form on 32-float slices: consumer warp c owns column chunk c of
  // every row (lanes = rows), so the shared prediction and the read are warp
  // reductions; tile row k keeps its chunk c at 16-byte position c ^ (k & 7)
  // (conflict-free when the lanes of a warp walk the rows of one chunk).
  constexpr bool COL = FIG2 && CW == 32;
  extern __shared__ __align__(128) unsigned char smem_all[];

  const Dims& d = A.d;
  const int D = A.depth;
  const int W = WR ? WR : d.W, R = WR ? WR : d.R, T = d.T, dv = d.dv;
  const ScanLayout L = scan_layout(CW, W, R, D, prefetch_steps<MINB>(), FIG2);
  const int NS = L.NS, MR = L.MR;
  const int nslice = dv / CW;
  // This unit: its threads, shared-memory partition and named barriers.
  const int sub = PAIR == 1 ? 0 : (int)(threadIdx.x / scan_threads<MINB>());
  const long long unit = (long long)blockIdx.x * PAIR + sub;
  unsigned char* const smem = smem_all + (size_t)sub * unit_smem_stride(L.total);
  const int bb = 4 * sub;                  // named barriers bb + 1 .. bb + 4
  const int chain = (int)(unit / nslice);
  const int c0 = (int)(unit - (long long)chain * nslice) * CW;
  const size_t th0 = (size_t)chain * d.Ts;  // flat (b,h,t=0) row
  float* Mc = A.M + (size_t)chain * (size_t)d.N() * dv + c0;
  const int CP = code_pitch(W, R);

  MetaSlot* meta = reinterpret_cast<MetaSlot*>(smem + L.meta);
  float* ypart = reinterpret_cast<float*>(smem + L.ypart);
  float* vpart = reinterpret_cast<float*>(smem + L.vpart);
  uint64_t* mfull = reinterpret_cast<uint64_t*>(smem + L.bars);
  uint64_t* mempty = mfull + MR;
  uint64_t* rfull = mempty + MR;     // rows of step u landed (ring of D)
  const uint32_t wslot = (uint32_t)(W * CW * 4), rslot = (uint32_t)(R * CW * 4);
  constexpr uint32_t rowb = (uint32_t)(CW * 4);

  const int tid = threadIdx.x - sub * scan_threads<MINB>(), lane = tid & 31, warp = tid >> 5;
  if (tid == 0) {
    for (int i = 0; i < MR; ++i) {
      mbar_init(&mfull[i], 32);
      mbar_init(&mempty[i], kConsumers / 32);
    }
    for (int i = 0; i < D; ++i) mbar_init(&rfull[i], kLoaders);
  }
  __syncthreads();
  if (unit >= (long long)d.B * d.H * nslice) return;   // odd unit count: idle half

  if (warp == kConsumers / 32) {
    // ------------------------------------------------------------ producer
    float ga_cur = 0.f, gb_cur = 0.f, ga_nxt = 0.f, gb_nxt = 0.f;
    if (lane < T) {
      ga_cur = load_scalar(A.alpha, th0 + lane, d.in_dtype);
      gb_cur = load_scalar(A.beta, th0 + lane, d.in_dtype);
    }
    if (32 + lane < T) {
      ga_nxt = load_scalar(A.alpha, th0 + 32 + lane, d.in_dtype);
      gb_nxt = load_scalar(A.beta, th0 + 32 + lane, d.in_dtype);
    }
    // Slot lists, weights, codes and the value slice of each step into its
    // metadata slot, kPS steps per iteration (one slot wait, one commit
    // group, one group wait and one loop pass per batch).  With every array
    // a whole number of 16-byte units each lane owns up to three fixed
    // (array, chunk) copy jobs whose source pointers just advance by the
    // array's step stride; otherwise 4-byte cp.async per element.
    constexpr int kP = prefetch_steps<MINB>();
    constexpr int kPS = kPrefetchBatch;
    constexpr int kPB = kP / kPS;                // batches of copies in flight
    static_assert(kP % kPS == 0 && 32 % kPS == 0, "prefetch batches");
    const bool vec = (W & 3) == 0 && (R & 3) == 0;
    const uint32_t vbytes = (uint32_t)(CW * IB);
    const unsigned char* jsrc[3];
    uint32_t jstride[3], jdst[3];
    bool jlive[3];
    {
      const int n0 = W / 4, n1 = n0 + W / 4, n2 = n1 + R / 4, n3 = n2 + R / 4;
      const int n4 = n3 + CP / 8, n5 = n4 + (int)vbytes / 16;
#pragma unroll
      for (int k = 0; k < 3; ++k) {
        const int j = lane + 32 * k;
        jlive[k] = vec && j < n5;
        const unsigned char* src = nullptr;
        uint32_t stride = 0, dst = 0;
        if (j < n0) {
          src = reinterpret_cast<const unsigned char*>(A.idx_w + th0 * W + 4 * j);
          stride = 4u * W;
          dst = (uint32_t)offsetof(MetaSlot, idx_w) + 16u * j;
        } else if (j < n1) {
          src = reinterpret_cast<const unsigned char*>(A.wt_w + th0 * W + 4 * (j - n0));
          stride = 4u * W;
          dst = (uint32_t)offsetof(MetaSlot, wt_w) + 16u * (j - n0);
        } else if (j < n2) {
          src = reinterpret_cast<const unsigned char*>(A.idx_r + th0 * R + 4 * (j - n1));
          stride = 4u * R;
          dst = (uint32_t)offsetof(MetaSlot, idx_r) + 16u * (j - n1);
        } else if (j < n3) {
          src = reinterpret_cast<const unsigned char*>(A.wt_r + th0 * R + 4 * (j - n2));
          stride = 4u * R;
          dst = (uint32_t)offsetof(MetaSlot, wt_r) + 16u * (j - n2);
        } else if (j < n4) {
          src = reinterpret_cast<const unsigned char*>(A.codes + th0 * CP + 8 * (j - n3));
          stride = 2u * CP;
          dst = (uint32_t)offsetof(MetaSlot, code) + 16u * (j - n3);
        } else if (j < n5) {
          src = reinterpret_cast<const unsigned char*>(A.v) + (th0 * dv + c0) * IB + 16 * (j - n4);
          stride = (uint32_t)(dv * IB);
          dst = (uint32_t)offsetof(MetaSlot, vraw) + 16u * (j - n4);
        }
        jsrc[k] = src;
        jstride[k] = stride;
        jdst[k] = dst;
      }
    }
    Ring mi{0, MR, 0u};         // slot of step u (copy stage)
    Ring mw{0, MR, 0u};         // slot of the batch's last step (slot-reuse wait)
    Ring mp{0, MR, 0u};         // slot of step up (publish stage)
    for (int i = 0; i < kPS - 1; ++i) mw.next();
    bool failed = false;
    for (int u0 = 0; u0 < T + kP && !failed; u0 += kPS) {
      if (u0 < T) {
        // Slot reuse: the batch's last step reuses the slot of step
        // u0 + kPS - 1 - MR; steps complete in order, so that one being
        // finished frees every slot of the batch.
        if (u0 + kPS - 1 >= MR) {
          bool ok = mbar_try_wait(&mempty[mw.i], mw.phase ^ 1u);
          if (!ok) {
            const uint64_t t0 = global_ns();
            while (!(ok = mbar_try_wait(&mempty[mw.i], mw.phase ^ 1u))) {
              __nanosleep(64);
              if (global_ns() - t0 > kTimeoutNs) break;
            }
          }
          if (!ok) {
            record_status(A.status, SDM_ERR_TIMEOUT);
            failed = true;
            break;
          }
        }
#pragma unroll
        for (int s = 0; s < kPS; ++s) {
          const int u = u0 + s;
          if (u < T) {
            unsigned char* m = reinterpret_cast<unsigned char*>(meta + mi.i);
            if (vec) {
#pragma unroll
              for (int k = 0; k < 3; ++k) {
                if (jlive[k]) cp_async16(m + jdst[k], jsrc[k]);
                jsrc[k] += jstride[k];
              }
            } else {
              MetaSlot* ms = meta + mi.i;
              const size_t th = th0 + u;
              for (int j = lane; j < W; j += 32) {
                cp_async4(&ms->idx_w[j], A.idx_w + th * W + j);
                cp_async4(&ms->wt_w[j], A.wt_w + th * W + j);
              }
              for (int j = lane; j < R; j += 32) {
                cp_async4(&ms->idx_r[j], A.idx_r + th * R + j);
                cp_async4(&ms->wt_r[j], A.wt_r + th * R + j);
              }
              if (lane < CP / 8) cp_async16(&ms->code[8 * lane], A.codes + th * CP + 8 * lane);
              if (lane < (int)vbytes / 16)
                cp_async16(ms->vraw + 16 * lane, reinterpret_cast<const unsigned char*>(A.v) +
                                                     (th * dv + c0) * IB + 16 * lane);
            }
            mi.next();
          }
        }
        for (int s = 0; s < kPS; ++s) mw.next();
      }
      cp_async_commit();
      if (u0 < kP) continue;

      // ---- batch up0 = u0 - kP: its metadata has landed; gates, publish.
      const int up0 = u0 - kP;
      cp_async_wait<kPB>();
      __syncwarp();
#pragma unroll
      for (int s = 0; s < kPS; ++s) {
        const int up = up0 + s;
        if (up >= T) break;
        if ((up & 31) == 0 && up > 0) {
          ga_cur = ga_nxt;
          gb_cur = gb_nxt;
          if (up + 32 + lane < T) {
            ga_nxt = load_scalar(A.alpha, th0 + up + 32 + lane, d.in_dtype);
            gb_nxt = load_scalar(A.beta, th0 + up + 32 + lane, d.in_dtype);
          }
        }
        const float ga = __shfl_sync(0xffffffffu, ga_cur, up & 31);
        const float gb = __shfl_sync(0xffffffffu, gb_cur, up & 31);
        MetaSlot* m = meta + mp.i;
        if (lane == 0) {
          m->alpha = ga;
          m->beta = gb;
        }
        __syncwarp();
        mbar_arrive(&mfull[mp.i]);
        mp.next();
      }
    }
    cp_async_wait_all();
    return;
  }

  if (warp > kConsumers / 32) {
    // -------------------------------------------------------------- loaders
    // Fetch the rows of step u once its metadata is decoded and the
    // consumers have finished step u - D (whose writes it must see, and whose
    // read tile it reuses).  Completion is signalled on rfull[u % D].
    const int lt = tid - (kConsumers + 32);
    const int lc = lt % CH, lr = lt / CH;
    constexpr int LRP = kLoaders / CH;       // rows per loader pass
    constexpr int kLoadRows = (128 + LRP - 1) / LRP;   // W + R <= 128 rows a step
    float* Ml = Mc + 4 * lc;
    unsigned char* sm_l = smem + 16 * lc;
    Ring mu{0, MR, 0u}, me{0, MR, 0u}, rf{0, D, 0u}, lw{0, NS, 0u};
    for (int u = 0; u < T; ++u) {
      // One thread waits for the step's metadata and for step u - D; the
      // other loaders sleep in a named barrier meanwhile (which also orders
      // their reads after that thread's acquire).  Waiting here is off the
      // critical path (the loaders run depth steps ahead), so it suspends.
      bool failed = false;
      if (lt == 0) {
        bool ok = u >= D ? mbar_wait2_bounded(&mfull[mu.i], mu.phase, &mempty[me.i], me.phase,
                                              kTimeoutNs)
                         : mbar_wait_bounded(&mfull[mu.i], mu.phase, kTimeoutNs);
        if (!ok) record_status(A.status, SDM_ERR_TIMEOUT);
        failed = !ok;
      }
      if (named_bar_or(bb + 3, kLoaders, failed)) break;
      const MetaSlot* m = meta + mu.i;
      // Only rows whose current value is in HBM (code -1) are fetched; a
      // forwarded (>= 0) or invalid (-2) row is not.
      // All of this thread's codes and slots are read before the first copy
      // is issued (a copy orders later shared-memory reads behind it).
      const uint32_t wb = (uint32_t)L.wtile + lw.i * wslot;
      const uint32_t rb = (uint32_t)L.rtile + rf.i * rslot;
      int code[kLoadRows], row[kLoadRows];
#pragma unroll
      for (int i = 0; i < kLoadRows; ++i) {
        const int k = lr + i * LRP;
        code[i] = -2;
        row[i] = 0;
        if (k < W + R) {
          code[i] = m->code[k];
          row[i] = k < W ? m->idx_w[k] : m->idx_r[k - W];
        }
      }
#pragma unroll
      for (int i = 0; i < kLoadRows; ++i) {
        const int k = lr + i * LRP;
        if (code[i] != -1) continue;
        const uint32_t off = k < W ? wb + k * rowb : rb + (k - W) * rowb;
        if constexpr (COL) {
          const int kk = k < W ? k : k - W;
          cp_async16(smem + off + 16 * (lc ^ (kk & 7)), Ml + (size_t)row[i] * dv);
        } else {
          cp_async16(sm_l + off, Ml + (size_t)row[i] * dv);
        }
      }
      cp_async_mbar_arrive_noinc(&rfull[rf.i]);
      mu.next();
      if (u >= D) me.next();
      rf.next();
      lw.next();
    }
    cp_async_wait_all();
    return;
  }

  // -------------------------------------------------------------- consumers
  if constexpr (COL) {
    // Warp cc: column chunk cc of every row; lane l: rows l and l + 32 of
    // the write and read sets.  A step: decay the write rows and reduce the
    // shared prediction over the lanes, write the rows' new values into the
    // tile, ONE block barrier, store the step's rows to HBM from the tile
    // (coalesced, 128 bytes per 8 lanes), weighted read reduced over the
    // lanes, y chunk stored by lane 0.
    const int cc = warp;
    unsigned char* tiles = smem + L.wtile;
    auto tile_chunk = [&](int slot, int k, int c) -> unsigned char* {
      return tiles + slot * wslot + k * rowb + 16 * (c ^ (k & 7));
    };
    bool aborted = false;
    Ring mt{0, MR, 0u}, wt{0, NS, 0u}, rf{0, D, 0u};
    for (int t = 0; t < T; ++t) {
      if (!aborted) {
        bool ok = true;
        if (lane == 0)
          ok = mbar_wait2_bounded(&rfull[rf.i], rf.phase, &mfull[mt.i], mt.phase, kTimeoutNs);
        __syncwarp();
        if (!__shfl_sync(0xffffffffu, ok, 0)) {
          if (lane == 0) record_status(A.status, SDM_ERR_TIMEOUT);
          aborted = true;
        }
      }
      const MetaSlot* m = meta + mt.i;
      if (!aborted) {
        const float a = m->alpha, b = m->beta;
        const float4 vv = load_v4<BF16>(m->vraw, cc);
        int code[2];
        float wj[2];
        float4 md[2];
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          const int j = lane + 32 * i;
          code[i] = -2;
          if (j < W) {
            code[i] = m->code[j];
            wj[i] = m->wt_w[j];
            md[i] = *reinterpret_cast<const float4*>(tile_chunk(wt.i, j, cc));   // fetched copy
          }
        }
        float4 part = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          const int j = lane + 32 * i;
          if (code[i] == -2) continue;
          if (code[i] >= 0) {
            const int dd = code[i] >> 6, p = code[i] & 63;
            const int sl = wt.i >= dd ? wt.i - dd : wt.i - dd + NS;
            md[i] = *reinterpret_cast<const float4*>(tile_chunk(sl, p, cc));
          }
          if constexpr (UNDO)
            *reinterpret_cast<float4*>(A.undo + ((th0 + t) * W + j) * dv + c0 + 4 * cc) = md[i];
          md[i] = make_float4(a * md[i].x, a * md[i].y, a * md[i].z, a * md[i].w);
          part.x = fmaf(wj[i], md[i].x, part.x);
          part.y = fmaf(wj[i], md[i].y, part.y);
          part.z = fmaf(wj[i], md[i].z, part.z);
          part.w = fmaf(wj[i], md[i].w, part.w);
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
          part.x += __shfl_xor_sync(0xffffffffu, part.x, off);
          part.y += __shfl_xor_sync(0xffffffffu, part.y, off);
          part.z += __shfl_xor_sync(0xffffffffu, part.z, off);
          part.w += __shfl_xor_sync(0xffffffffu, part.w, off);
        }
        const float4 res = make_float4(vv.x - part.x, vv.y - part.y, vv.z - part.z, vv.w - part.w);
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          if (code[i] == -2) continue;
          const float cw = b * wj[i];
          float4 o;
          o.x = fmaf(cw, res.x, md[i].x);
          o.y = fmaf(cw, res.y, md[i].y);
          o.z = fmaf(cw, res.z, md[i].z);
          o.w = fmaf(cw, res.w, md[i].w);
          *reinterpret_cast<float4*>(tile_chunk(wt.i, lane + 32 * i, cc)) = o;
        }
      }
      // The one block barrier of a step (a timeout becomes a uniform exit).
      if (named_bar_or(bb + 1, kConsumers, aborted)) {
        aborted = true;
        break;
      }
      // The step's rows to HBM from the tile: thread -> (row, chunk).
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const int j = (tid >> 3) + 32 * i, c = tid & 7;
        if (j < W && m->code[j] != -2)
          *reinterpret_cast<float4*>(Mc + (size_t)m->idx_w[j] * dv + 4 * c) =
              *reinterpret_cast<const float4*>(tile_chunk(wt.i, j, c));
      }
      // Read after the write (Eq. (5)), reduced over the lanes.
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
      {
        int code[2];
        float w[2];
        float4 x[2];
        const unsigned char* rsrc = smem + L.rtile + rf.i * rslot;
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          const int q = lane + 32 * i;
          code[i] = -2;
          if (q < R) {
            code[i] = m->code[W + q];
            w[i] = m->wt_r[q];
            x[i] = *reinterpret_cast<const float4*>(rsrc + q * rowb + 16 * (cc ^ (q & 7)));
          }
        }
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          if (code[i] == -2) continue;
          if (code[i] >= 0) {
            const int dd = code[i] >> 6, p = code[i] & 63;
            const int sl = wt.i >= dd ? wt.i - dd : wt.i - dd + NS;
            x[i] = *reinterpret_cast<const float4*>(tile_chunk(sl, p, cc));
          }
          acc.x = fmaf(w[i], x[i].x, acc.x);
          acc.y = fmaf(w[i], x[i].y, acc.y);
          acc.z = fmaf(w[i], x[i].z, acc.z);
          acc.w = fmaf(w[i], x[i].w, acc.w);
        }
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) {
        acc.x += __shfl_xor_sync(0xffffffffu, acc.x, off);
        acc.y += __shfl_xor_sync(0xffffffffu, acc.y, off);
        acc.z += __shfl_xor_sync(0xffffffffu, acc.z, off);
        acc.w += __shfl_xor_sync(0xffffffffu, acc.w, off);
      }
      if (lane == 0) *reinterpret_cast<float4*>(A.y + (th0 + t) * dv + c0 + 4 * cc) = acc;
      __syncwarp();
      if (lane == 0) mbar_arrive(&mempty[mt.i]);
      mt.next();
      wt.next();
      rf.next();
    }
    return;
  }

  const int myc = tid % CH, myr = tid / CH;
  constexpr int kMaxPW = (64 + RP - 1) / RP;   // write / read rows per thread (W, R <= 64)
  constexpr int kMaxPR = kMaxPW;
  float* Mt = Mc + 4 * myc;                  // this lane's column chunk of row 0
  unsigned char* sm_c = smem + 16 * myc;     // shared base shifted to the chunk
  bool aborted = false;

  // Shared-memory place of a forwarded row: position p of the write tile of
  // step t - dd, for plan code (dd << 6) | p; wcur is step t's write tile.
  auto fwd_place = [&](int code, int wcur) -> const unsigned char* {
    const int dd = code >> 6, p = code & 63;
    const int sl = wcur >= dd ? wcur - dd : wcur - dd + NS;
    return sm_c + L.wtile + sl * wslot + p * rowb;
  };

  auto finalize = [&](int t) {
    if (lane < CH) {
      const float* yp = ypart + (t & 1) * 8 * CW + 4 * lane;
      float4 s4 = *reinterpret_cast<const float4*>(yp);
#pragma unroll
      for (int w = 1; w < kCW; ++w) {
        const float4 p = *reinterpret_cast<const float4*>(yp + w * CW);
        s4.x += p.x;
        s4.y += p.y;
        s4.z += p.z;
        s4.w += p.w;
      }
      *reinterpret_cast<float4*>(A.y + (th0 + t) * dv + c0 + 4 * lane) = s4;
    }
  };

  Ring mt{0, MR, 0u};   // metadata slot of step t
  Ring wt{0, NS, 0u};   // write-tile slot of step t
  Ring rf{0, D, 0u};    // rows-landed barrier of step t

  // The read sum of step t is reduced over the lanes and stored to the
  // partials at the top of step t + 1, while that step's barrier tests are
  // in flight (the partials are read only after step t + 1's block barrier).
  float4 acc_prev = make_float4(0.f, 0.f, 0.f, 0.f);
  auto store_partial = [&](int tp, float4 acc) {
#pragma unroll
    for (int off = CH; off < 32; off <<= 1) {
      acc.x += __shfl_xor_sync(0xffffffffu, acc.x, off);
      acc.y += __shfl_xor_sync(0xffffffffu, acc.y, off);
      acc.z += __shfl_xor_sync(0xffffffffu, acc.z, off);
      acc.w += __shfl_xor_sync(0xffffffffu, acc.w, off);
    }
    if (lane < CH)
      *reinterpret_cast<float4*>(ypart + (tp & 1) * 8 * CW + warp * CW + 4 * lane) = acc;
  };

  if constexpr (!FIG2) {
    // Eq. (4).  The loop keeps its per-step work to the minimum: the ring
    // positions of the step advance as pointers, every per-thread offset is
    // computed once, and rows a thread does not hold are masked instead of
    // branched around.
    const MetaSlot* m = meta;                  // metadata slot of step t
    int mi = 0;
    unsigned mph = 0u;
    unsigned char* const wt0 = sm_c + L.wtile;
    unsigned char* wcur = wt0;                 // write tile of step t
    int wi = 0;                                // its slot
    const unsigned char* const rt0 = sm_c + L.rtile;
    const unsigned char* rcur = rt0;           // read tile of step t
    int ri = 0;
    unsigned rph = 0u;
    float* undo_p = nullptr;                   // log row of (t, j = myr)
    if constexpr (UNDO) undo_p = A.undo + (th0 * W + myr) * dv + c0 + 4 * myc;
    const size_t undo_step = (size_t)W * dv;
    // On-chip copy of a forwarded row: position p of the write tile of step
    // t - dd, for plan code (dd << 6) | p.
    // (Slot arithmetic on indices: a shared-memory pointer must not step
    // below the window even transiently.)
    auto fwd = [&](int code) -> const float4* {
      int sl = wi - (code >> 6);
      if (sl < 0) sl += NS;
      return reinterpret_cast<const float4*>(wt0 + sl * wslot + (code & 63) * rowb);
    };
    for (int t = 0; t < T; ++t) {
      // Rows and metadata of step t; the previous step's read sum is reduced
      // meanwhile.
      if constexpr (MINB == 2) {
        // Two CTAs share the SM and issue slots are the limit: one warp
        // tests the barriers, the other consumer warps sleep in a hardware
        // barrier meanwhile (which also orders their reads after its acquire).
        if (t > 0) store_partial(t - 1, acc_prev);
        bool bad = false;
        if (warp == 0) {
          const bool r0 = mbar_test_wait(&rfull[ri], rph);
          const bool m0 = mbar_test_wait(&mfull[mi], mph);
          if (!__all_sync(0xffffffffu, r0 && m0)) {
            bool ok = true;
            if (lane == 0) ok = mbar_wait2_bounded(&rfull[ri], rph, &mfull[mi], mph, kTimeoutNs);
            if (!__shfl_sync(0xffffffffu, ok, 0)) {
              if (lane == 0) record_status(A.status, SDM_ERR_TIMEOUT);
              bad = true;
            }
          }
        }
        if (named_bar_or(bb + 4, kConsumers, bad)) aborted = true;
      } else {
        const bool r0 = mbar_test_wait(&rfull[ri], rph);
        const bool m0 = mbar_test_wait(&mfull[mi], mph);
        if (t > 0) store_partial(t - 1, acc_prev);
        if (!__all_sync(0xffffffffu, r0 && m0)) {
          bool ok = true;
          if (lane == 0) ok = mbar_wait2_bounded(&rfull[ri], rph, &mfull[mi], mph, kTimeoutNs);
          if (!__shfl_sync(0xffffffffu, ok, 0)) {
            if (lane == 0) record_status(A.status, SDM_ERR_TIMEOUT);
            aborted = true;
          }
        }
      }
      if (!aborted) {
        // Write: decay + per-slot delta (Eq. (3)-(4)).  Every row this thread
        // writes is read first, so the rows' shared-memory latencies overlap.
        const float a = m->alpha, b = m->beta;
        const float4 vv = load_v4<BF16>(m->vraw, myc);
        int code[kMaxPW], row[kMaxPW];
        float wj[kMaxPW];
        float4 x[kMaxPW];
#pragma unroll
        for (int pw = 0; pw < kMaxPW; ++pw) {
          const int j = pw * RP + myr;
          code[pw] = -2;
          if (pw * RP < W - myr) {
            code[pw] = m->code[j];
            row[pw] = m->idx_w[j];
            wj[pw] = m->wt_w[j];
            x[pw] = *reinterpret_cast<const float4*>(wcur + j * rowb);   // fetched copy
          }
        }
#pragma unroll
        for (int pw = 0; pw < kMaxPW; ++pw) {
          const int j = pw * RP + myr;
          if (code[pw] >= 0) x[pw] = *fwd(code[pw]);
          const bool live = code[pw] != -2;                              // absent / invalid
          if constexpr (UNDO) {
            if (live) *reinterpret_cast<float4*>(undo_p + (size_t)pw * RP * dv) = x[pw];
          }
          const float cw = b * wj[pw];
          float4 o;
          float mt_;
          mt_ = a * x[pw].x; o.x = fmaf(cw, vv.x - mt_, mt_);
          mt_ = a * x[pw].y; o.y = fmaf(cw, vv.y - mt_, mt_);
          mt_ = a * x[pw].z; o.z = fmaf(cw, vv.z - mt_, mt_);
          mt_ = a * x[pw].w; o.w = fmaf(cw, vv.w - mt_, mt_);
          if (live) {
            *reinterpret_cast<float4*>(wcur + j * rowb) = o;
            *reinterpret_cast<float4*>(Mt + (size_t)row[pw] * dv) = o;
          }
        }
      }
      // The one block barrier of a step; it also turns a timeout anywhere
      // into a decision every consumer takes at the same point.
      if (named_bar_or(bb + 1, kConsumers, aborted)) {
        aborted = true;
        break;
      }
      if (t > 0 && warp == ((t - 1) & (kCW - 1))) finalize(t - 1);
      // Read after the write (Eq. (5)); all of this thread's rows are read first.
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
      {
        int code[kMaxPR];
        float w[kMaxPR];
        float4 xr[kMaxPR];
#pragma unroll
        for (int pr = 0; pr < kMaxPR; ++pr) {
          const int q = pr * RP + myr;
          code[pr] = -2;
          if (pr * RP < R - myr) {
            code[pr] = m->code[W + q];
            w[pr] = m->wt_r[q];
            xr[pr] = *reinterpret_cast<const float4*>(rcur + q * rowb);
          }
        }
#pragma unroll
        for (int pr = 0; pr < kMaxPR; ++pr) {
          if (code[pr] == -2) continue;                                  // absent / invalid
          if (code[pr] >= 0) xr[pr] = *fwd(code[pr]);
          acc.x = fmaf(w[pr], xr[pr].x, acc.x);
          acc.y = fmaf(w[pr], xr[pr].y, acc.y);
          acc.z = fmaf(w[pr], xr[pr].z, acc.z);
          acc.w = fmaf(w[pr], xr[pr].w, acc.w);
        }
      }
      acc_prev = acc;
      __syncwarp();
      if (lane == 0) mbar_arrive(&mempty[mi]);
      // Next step's ring positions.
      if (++mi == MR) {
        mi = 0;
        mph ^= 1u;
        m = meta;
      } else {
        ++m;
      }
      wcur += wslot;
      if (++wi == NS) {
        wi = 0;
        wcur = wt0;
      }
      rcur += rslot;
      if (++ri == D) {
        ri = 0;
        rph ^= 1u;
        rcur = rt0;
      }
      if constexpr (UNDO) undo_p += undo_step;
    }
    if (T > 0) store_partial(T - 1, acc_prev);
    named_bar_sync(bb + 1, kConsumers);
    if (!aborted && T > 0 && warp == ((T - 1) & (kCW - 1))) finalize(T - 1);
    return;
  }

  for (int t = 0; t < T; ++t) {
    // Rows of step t landed (and its metadata is decoded): every lane tests
    // both barriers; the previous step's read sum is reduced meanwhile.
    bool ok = true;
    if (!aborted) {
      const bool r0 = mbar_test_wait(&rfull[rf.i], rf.phase);
      const bool m0 = mbar_test_wait(&mfull[mt.i], mt.phase);
      if (t > 0) store_partial(t - 1, acc_prev);
      if (!__all_sync(0xffffffffu, r0 && m0)) {
        if (lane == 0)
          ok = mbar_wait2_bounded(&rfull[rf.i], rf.phase, &mfull[mt.i], mt.phase, kTimeoutNs);
        ok = __shfl_sync(0xffffffffu, ok, 0);
      }
      if (!ok) {
        if (lane == 0) record_status(A.status, SDM_ERR_TIMEOUT);
        aborted = true;
      }
    }
    const MetaSlot* m = meta + mt.i;
    if (!FIG2 && !aborted) {
      // Write: decay + per-slot delta (Eq. (3)-(4)).  Every row this thread
      // writes is read first, so the rows' shared-memory latencies overlap.
      const float a = m->alpha, b = m->beta;
      const float4 vv = load_v4<BF16>(m->vraw, myc);
      unsigned char* wdst = sm_c + L.wtile + wt.i * wslot;
      int code[kMaxPW], row[kMaxPW];
      float wj[kMaxPW];
      float4 x[kMaxPW];
#pragma unroll
      for (int pw = 0; pw < kMaxPW; ++pw) {
        const int j = pw * RP + myr;
        code[pw] = -2;
        if (j < W) {
          code[pw] = m->code[j];
          row[pw] = m->idx_w[j];
          wj[pw] = m->wt_w[j];
          x[pw] = *reinterpret_cast<const float4*>(wdst + j * rowb);   // fetched copy
        }
      }
#pragma unroll
      for (int pw = 0; pw < kMaxPW; ++pw) {
        const int j = pw * RP + myr;
        if (code[pw] == -2) continue;                                   // absent / invalid
        if (code[pw] >= 0) x[pw] = *reinterpret_cast<const float4*>(fwd_place(code[pw], wt.i));
        if constexpr (UNDO)
          *reinterpret_cast<float4*>(A.undo + ((th0 + t) * W + j) * dv + c0 + 4 * myc) = x[pw];
        const float cw = b * wj[pw];
        float4 o;
        float mt_;
        mt_ = a * x[pw].x; o.x = fmaf(cw, vv.x - mt_, mt_);
        mt_ = a * x[pw].y; o.y = fmaf(cw, vv.y - mt_, mt_);
        mt_ = a * x[pw].z; o.z = fmaf(cw, vv.z - mt_, mt_);
        mt_ = a * x[pw].w; o.w = fmaf(cw, vv.w - mt_, mt_);
        *reinterpret_cast<float4*>(wdst + j * rowb) = o;
        *reinterpret_cast<float4*>(Mt + (size_t)row[pw] * dv) = o;
      }
    }
    if (FIG2) {
      // Write, Fig. 2 form: decay every write row, reduce the shared
      // prediction vhat over the write set, then one residual for all rows.
      float4 md[kMaxPW];
      const float a = m->alpha;
      unsigned char* wdst = sm_c + L.wtile + wt.i * wslot;
      float4 part = make_float4(0.f, 0.f, 0.f, 0.f);
      if (!aborted) {
#pragma unroll
        for (int pw = 0; pw < kMaxPW; ++pw) {
          const int j = pw * RP + myr;
          md[pw] = make_float4(0.f, 0.f, 0.f, 0.f);
          if (j >= W) continue;
          const int code = m->code[j];
          float4 x = *reinterpret_cast<const float4*>(wdst + j * rowb);
          if (code == -2) continue;
          if (code >= 0) x = *reinterpret_cast<const float4*>(fwd_place(code, wt.i));
          if constexpr (UNDO)
            *reinterpret_cast<float4*>(A.undo + ((th0 + t) * W + j) * dv + c0 + 4 * myc) = x;
          const float wj = m->wt_w[j];
          md[pw] = make_float4(a * x.x, a * x.y, a * x.z, a * x.w);
          part.x = fmaf(wj, md[pw].x, part.x);
          part.y = fmaf(wj, md[pw].y, part.y);
          part.z = fmaf(wj, md[pw].z, part.z);
          part.w = fmaf(wj, md[pw].w, part.w);
        }
#pragma unroll
        for (int off = CH; off < 32; off <<= 1) {
          part.x += __shfl_xor_sync(0xffffffffu, part.x, off);
          part.y += __shfl_xor_sync(0xffffffffu, part.y, off);
          part.z += __shfl_xor_sync(0xffffffffu, part.z, off);
          part.w += __shfl_xor_sync(0xffffffffu, part.w, off);
        }
        if (lane < CH) *reinterpret_cast<float4*>(vpart + warp * CW + 4 * lane) = part;
      }
      // Every consumer reaches this barrier each step (a timeout becomes a
      // uniform exit here, as at the step barrier below).
      if (named_bar_or(bb + 2, kConsumers, aborted)) {
        aborted = true;
        break;
      }
      const float b = m->beta;
      const float4 vv = load_v4<BF16>(m->vraw, myc);
      float4 vh = *reinterpret_cast<const float4*>(vpart + 4 * myc);
#pragma unroll
      for (int w = 1; w < kCW; ++w) {
        const float4 p = *reinterpret_cast<const float4*>(vpart + w * CW + 4 * myc);
        vh.x += p.x;
        vh.y += p.y;
        vh.z += p.z;
        vh.w += p.w;
      }
      const float4 res = make_float4(vv.x - vh.x, vv.y - vh.y, vv.z - vh.z, vv.w - vh.w);
#pragma unroll
      for (int pw = 0; pw < kMaxPW; ++pw) {
        const int j = pw * RP + myr;
        if (j >= W) continue;
        if (m->code[j] == -2) continue;
        const int row = m->idx_w[j];
        const float cw = b * m->wt_w[j];
        float4 o;
        o.x = fmaf(cw, res.x, md[pw].x);
        o.y = fmaf(cw, res.y, md[pw].y);
        o.z = fmaf(cw, res.z, md[pw].z);
        o.w = fmaf(cw, res.w, md[pw].w);
        *reinterpret_cast<float4*>(wdst + j * rowb) = o;
        *reinterpret_cast<float4*>(Mt + (size_t)row * dv) = o;
      }
    }
    // The one block barrier of a step; it also turns a timeout anywhere
    // into a decision every consumer takes at the same point.
    if (named_bar_or(bb + 1, kConsumers, aborted)) {
      aborted = true;
      break;
    }
    if (t > 0 && warp == ((t - 1) & (kCW - 1))) finalize(t - 1);

    // Read after the write (Eq. (5)); all of this thread's rows are read first.
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    {
      int code[kMaxPR];
      float w[kMaxPR];
      float4 x[kMaxPR];
      const unsigned char* rsrc = sm_c + L.rtile + rf.i * rslot;
#pragma unroll
      for (int pr = 0; pr < kMaxPR; ++pr) {
        const int q = pr * RP + myr;
        code[pr] = -2;
        if (q < R) {
          code[pr] = m->code[W + q];
          w[pr] = m->wt_r[q];
          x[pr] = *reinterpret_cast<const float4*>(rsrc + q * rowb);
        }
      }
#pragma unroll
      for (int pr = 0; pr < kMaxPR; ++pr) {
        if (code[pr] == -2) continue;
        if (code[pr] >= 0) x[pr] = *reinterpret_cast<const float4*>(fwd_place(code[pr], wt.i));
        acc.x = fmaf(w[pr], x[pr].x, acc.x);
        acc.y = fmaf(w[pr], x[pr].y, acc.y);
        acc.z = fmaf(w[pr], x[pr].z, acc.z);
        acc.w = fmaf(w[pr], x[pr].w, acc.w);
      }
    }
    acc_prev = acc;
    __syncwarp();
    if (lane == 0) mbar_arrive(&mempty[mt.i]);
    mt.next();
    wt.next();
    rf.next();
  }
  if (T > 0) store_partial(T - 1, acc_prev);
  named_bar_sync(bb + 1, kConsumers);
  if (!aborted && T > 0 && warp == ((T - 1) & (kCW - 1))) finalize(T - 1);
}

template <int CW, bool BF16>
cudaError_t launch_t(const ScanArgs& A, bool one_per_sm, bool two_per_sm, cudaStream_t stream) {
  const bool fig2 = A.d.update == SDM_UPDATE_SHARED_RESIDUAL, logged = A.undo != nullptr;
  const bool one = !fig2 && !logged && one_per_sm;      // the MINB = 1 build
  // Two units per CTA for the Eq. (4) scan where exactly two units share an
  // SM (the Fig. 2 column path measured slower that way and keeps one per
  // CTA; with three per SM a CTA of two would not leave room for a second).
  const bool pair = !fig2 && !logged && two_per_sm;
  const bool w64 = A.d.W == 64 && A.d.R == 64;
  const int kp = one ? prefetch_steps<1>() : prefetch_steps<2>();
  const size_t total = scan_layout(CW, A.d.W, A.d.R, A.depth, kp, fig2).total;
  const size_t smem = pair ? 2 * unit_smem_stride(total) : total;
  auto kfn = fig2 ? (logged ? scan_kernel<CW, BF16, true, true, 2, 1>
                            : scan_kernel<CW, BF16, true, false, 2, 1>)
                  : (logged ? scan_kernel<CW, BF16, false, true, 2, 1>
                            : (one ? (w64 ? scan_kernel<CW, BF16, false, false, 1, 1, 64>
                                          : scan_kernel<CW, BF16, false, false, 1, 1>)
                                   : (pair ? (w64 ? scan_kernel<CW, BF16, false, false, 2, 2, 64>
                                                  : scan_kernel<CW, BF16, false, false, 2, 2>)
                                           : scan_kernel<CW, BF16, false, false, 2, 1>)));
  cudaError_t e =
      cudaFuncSetAttribute(kfn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const long long units = (long long)A.d.B * A.d.H * (A.d.dv / CW);
  if (units == 0 || A.d.T == 0) return cudaSuccess;
  const long long grid = pair ? (units + 1) / 2 : units;
  const int threads = one ? scan_threads<1>() : (pair ? 2 : 1) * scan_threads<2>();
  kfn<<<(unsigned)grid, threads, smem, stream>>>(A);
  return cudaGetLastError();
}


}  // namespace

size_t scan_workspace_bytes(const Dims& d) {
  return (size_t)d.B * d.H * d.T * code_pitch(d.W, d.R) * sizeof(int16_t);
}

cudaError_t scan_setup(const Dims& d, int depth, int col_slice, bool logged, ScanSetup* out) {
  const long long chains = (long long)d.B * d.H;
  const DeviceLimits lim = device_limits();
  const long long sms = lim.sms;
  int cw = col_slice;
  if (cw == 0) cw = (d.dv % 32 == 0 && chains * (d.dv / 32) >= sms) ? 32 : 16;
  if (d.dv % cw != 0) cw = 16;
  const long long units = chains * (d.dv / cw);
  // CTAs per SM needed to keep every unit resident, and the ring depth that fits.
  const long long per_sm = (units + sms - 1) / sms;
  // The build that runs (see launch_t) and its metadata prefetch distance.
  const bool one = per_sm <= 1;
  const bool fig2 = d.update == SDM_UPDATE_SHARED_RESIDUAL;
  const int kp = one && !fig2 && !logged ? prefetch_steps<1>() : prefetch_steps<2>();
  const size_t budget = per_sm <= 1    ? lim.smem_per_cta
                        : per_sm == 2 ? lim.smem_per_sm / 2 - 1024
                                      : lim.smem_per_sm / 3 - 1024;
  // (The pair build puts two such partitions, each rounded to 128 bytes, in
  // one CTA: 2 * (smem_per_sm / 2 - 1024) stays within smem_per_cta.)
  int D = depth;
  if (D == 0) {
    D = 1;
    for (int cand = 2; cand <= 16; ++cand)
      if (scan_layout(cw, d.W, d.R, cand, kp, fig2).total <= budget) D = cand;
  }
  if (D < 1 || D > 16) return cudaErrorInvalidValue;
  // A requested depth is a hint: shrink it until the ring fits on chip.
  while (D > 1 && scan_layout(cw, d.W, d.R, D, kp, fig2).total > lim.smem_per_cta) --D;
  *out = ScanSetup{cw, D, one, per_sm == 2};
  return cudaSuccess;
}

cudaError_t launch_scan_kernel(const Dims& d, const ScanSetup& c, const int32_t* idx_w,
                               const float* wt_w, const int32_t* idx_r, const float* wt_r,
                               const void* alpha, const void* beta, const void* v, float* M,
                               float* y, float* undo, const int16_t* codes, unsigned* status,
                               cudaStream_t stream) {
  if ((long long)d.B * d.H == 0 || d.T == 0) return cudaSuccess;
  ScanArgs A{d, idx_w, wt_w, idx_r, wt_r, alpha, beta, v, codes, M, y, undo, c.depth, status};
  const bool bf = d.in_dtype == SDM_BF16;
  const bool one = c.one_per_sm, two = c.pair;
  if (c.cw == 64)
    return bf ? launch_t<64, true>(A, one, two, stream) : launch_t<64, false>(A, one, two, stream);
  if (c.cw == 32)
    return bf ? launch_t<32, true>(A, one, two, stream) : launch_t<32, false>(A, one, two, stream);
  return bf ? launch_t<16, true>(A, one, two, stream) : launch_t<16, false>(A, one, two, stream);
}

cudaError_t launch_scan(const Dims& d, const int32_t* idx_w, const float* wt_w,
                        const int32_t* idx_r, const float* wt_r, const void* alpha,
                        const void* beta, const void* v, float* M, float* y, float* undo,
                        void* workspace, int depth, int col_slice, unsigned* status,
                        cudaStream_t stream) {
  if ((long long)d.B * d.H == 0 || d.T == 0) return cudaSuccess;
  ScanSetup c;
  cudaError_t e = scan_setup(d, depth, col_slice, undo != nullptr, &c);
  if (e != cudaSuccess) return e;
  int16_t* codes = static_cast<int16_t*>(workspace);
  e = launch_plan(d, idx_w, idx_r, codes, c.depth, status, stream);
  if (e != cudaSuccess) return e;
  return launch_scan_kernel(d, c, idx_w, wt_w, idx_r, wt_r, alpha, beta, v, M, y, undo, codes,
                            status, stream);
}

}  // namespace sdm
