// sv_rows.cuh -- the bandwidth-bound rows kernel (no top-k / top-p filter).
//
// One persistent cooperative grid, one CTA per SM, every SM busy.  Each
// logits row is cut into S slices of at most L elements; work unit
// u = (target row g, slice k), u = g * S + k, and CTA c handles units
// u = c, c + N, c + 2N, ... (N CTAs), so the S slices of a row are handled in
// the same round by S different CTAs.  A unit's slice pair (target slice and,
// when row g scores a drafted token, the draft partner's slice) is brought
// into one of NS shared-memory stages by bulk copies (cp.async.bulk) and
// stays there for both passes: each logit crosses HBM once.  The CTAs holding
// the slices of one row exchange their partial statistics through an
// L2-resident workspace slot per (row, slice) (all CTAs of a cooperative
// launch are co-resident; every wait is time-bounded).  Every published
// 32-bit word travels in a 64-bit word together with a per-call tag (relaxed
// 64-bit accesses are single-copy atomic), so a reader checks each word
// itself: no release/acquire pair, one L2 round trip per poll.
//
// Warp roles (mbarriers between them; no CTA-wide barrier in the loop):
//  * NCW consumer warps in two groups (labels on): one runs pass 1 of the
//    units, the other pass 2, each on its own stream of units, so that the
//    exchange of a unit's statistics overlaps pass 1 of later units;
//  * producer warp: refills a stage once every role has released it (row
//    metadata arrives by cp.async on the stage's `full` mbarrier) and writes
//    the unit's label partial;
//  * kPublishers publisher warps (unit i by warp i % kPublishers): merge the
//    consumer warps' pass-1 partials of a unit into the CTA partial and
//    publish it;
//  * kGatherers gatherer warps (unit j by warp j % kGatherers): wait for the
//    S partials of the unit's row, merge them into the row statistics for
//    pass 2, and for the row's first slice run the row epilogue (accept
//    decision, statistics).
//
// Per unit:
//  pass 1   sums kept as sum_v 2^(x_v * sc) = s * 2^h, sc = log2(e) / T: each
//           term is exp2(fma(x, sc, -h)) for a fixed reference h, so rounding
//           is relative to the (small) exponent itself, whatever T is.  The
//           running max / argmax is tracked only when needed (greedy
//           decisions, row statistics).  Partials merge as max h, one rescale
//           by exp2(h - H) per partial, then a plain sum.
//  pass 2   (labels only) c* = sum_v min(p_t(v), p_d(v)) = 1 - 1/2 ||p_t - p_d||_1
//           over the resident slice pair, one exp2 per element pair:
//           min(p_t, p_d) * s_t = exp2(min(a, b - delta)), a = fma(t, sc, -h_t),
//           b = fma(d, sc, -h_d), delta = log2(s_d / s_t).  One partial per
//           unit goes to the workspace; the finalize kernel sums a row's S
//           partials in slice order.
//  epilogue accept decision of the drafted token -- sampling:
//           u * p_d(x) < p_t(x), greedy: x == argmax_t -- and row statistics.
//
// Confidence label: DSpark tutorial, "置信度预测头".  Accept rule and the
// first-rejection structure: DSpark tutorial, "推测解码的两步流程"; DFlash /
// Spec V2 page, A3 (lossless rejection sampling after Leviathan et al.).
#pragma once

#include "sv_common.cuh"
#include "sv_finalize.cuh"

namespace sv {

constexpr int kMaxStages = 6;
// An mbarrier parity wait cannot tell "my phase completed" from "the barrier
// is still one phase behind me", so no warp may wait on a stage's barrier
// before the previous use of that stage has passed the same barrier.  Warps
// that handle every unit wait in order; a gatherer handles every kGatherers-th
// unit and a publisher every kPublishers-th, so their previous unit implies
// the stage's previous use is done only when stages >= both counts.
constexpr int kMinStages = 4;
constexpr int kMaxConsumerWarps = 24;
constexpr int kPublishers = 2;
constexpr int kGatherers = 4;
static_assert(kMinStages >= kGatherers && kMinStages >= kPublishers, "stage reuse order");
constexpr int kMaxSmemOffsets = 4096; // row_offsets entries kept in shared memory

// Shared-memory header layout of the rows kernel (bytes from the base).
constexpr int kOffFull = 0;                                   // kMaxStages mbarriers each
constexpr int kOffEmpty = kOffFull + 8 * kMaxStages;
constexpr int kOffPartBar = kOffEmpty + 8 * kMaxStages;
constexpr int kOffStatsBar = kOffPartBar + 8 * kMaxStages;
constexpr int kOffTailBar = kOffStatsBar + 8 * kMaxStages;   // slice copies of the tail
constexpr int kOffPart = 256;                                 // [stage][warp][16] words
constexpr int kOffCp = kOffPart + kMaxStages * kMaxConsumerWarps * 64;  // [stage][warp] floats
constexpr int kOffStats = kOffCp + kMaxStages * kMaxConsumerWarps * 4;  // [stage][8] words
constexpr int kOffInfo = kOffStats + kMaxStages * 32;                   // [stage] RowInfo
constexpr int kOffTail = kOffInfo + kMaxStages * 64;                    // DrawSel, then scratch
constexpr int kRowsHdrBytes = 12288;
static_assert(kOffTailBar + 8 <= kOffPart, "rows kernel barriers");
static_assert(sizeof(DrawSel) <= 64, "tail choice");
static_assert(kOffCp - kOffPart >= 4 * SV_MAX_LEN, "tail row marks");
static_assert(kOffTail + 64 + 4 * 32 <= kRowsHdrBytes, "rows kernel header");

struct RowInfo {
  int32_t g, k, r, off, off1, pair, gd;
  int32_t x;    // drafted token (cp.async)
  int32_t ell;  // l_r (cp.async)
  float u;      // uniform of the row (cp.async)
  int32_t tn, dn;        // bytes of the target / draft slice buffers (dn = 0: no draft row)
  int32_t thoff, dhoff;  // head offsets (elements) of the slices in them
  int32_t len, v0;       // slice length, vocabulary id of its first element
};
static_assert(sizeof(RowInfo) == 64, "RowInfo layout");

// The unit's slices as shared-memory buffer views (the global sources are
// not needed once the stage is filled).
__device__ __forceinline__ Slice slice_t(const RowInfo& i) {
  return Slice{nullptr, i.tn, i.thoff, i.len, i.v0};
}
__device__ __forceinline__ Slice slice_d(const RowInfo& i) {
  return Slice{nullptr, i.dn, i.dhoff, i.pair ? i.len : 0, i.v0};
}

// Position in a ring of n slots: the slot and the phase parity of its
// current use, advanced without a division (the ring size is a runtime
// value, and a division per step would sit on every role's critical path).
struct RingPos {
  int idx;
  uint32_t par;
  __device__ __forceinline__ void next(int n) {
    if (++idx == n) {
      idx = 0;
      par ^= 1u;
    }
  }
};

template <int VEC>
__device__ __forceinline__ float vmax_nan(const float* x) {
  float v = x[0];
#pragma unroll
  for (int l = 1; l < VEC; ++l) v = fmax_nan(v, x[l]);
  return v;
}

template <int VEC>
__device__ __forceinline__ float sum_exp2(const float* x, float sc, float h) {
  float e[VEC];
#pragma unroll
  for (int l = 0; l < VEC; ++l) e[l] = ex2(fmaf(x[l], sc, -h));
#pragma unroll
  for (int w = VEC / 2; w > 0; w >>= 1)
#pragma unroll
    for (int l = 0; l < w; ++l) e[l] += e[l + w];
  return e[0];
}

// Bound on a lane's sum in the passes whose reference is not the running
// maximum (2^24): larger sums mean a reference far below the maximum (low
// temperatures), where exponent arguments lose precision and the merge
// factors 2^(h - H) of such partials can flush to zero while the product
// does not; those lanes take the tracked variant instead.
constexpr float kFastSumMax = 16777216.f;

// Pass 1 of one consumer thread over its vectors k = ct, ct + NCT, ... of a
// slice.  TRACK: exact running max / argmax.  Otherwise the reference h is
// taken from the thread's first vector holding a finite value; a sum at or
// above kFastSumMax or a non-finite input sends the thread to the tracked
// variant (rare).
template <int ES, bool NEED_Z, bool TRACK>
__device__ __forceinline__ RStat pass1_thread(const unsigned char* buf, const Slice& s, float sc,
                                              int ct, int NCT, bool& bad) {
  constexpr int VEC = 16 / ES;
  const int32_t nv = s.nbytes >> 4;
  const int32_t idbase = s.v0 - s.hoff;
  RStat st = rstat_empty();
  int32_t k = ct;
  if (!TRACK) {
    for (; k < nv; k += NCT) {  // first vector with a finite maximum
      float x[VEC];
      load_vec<ES>(buf, s, k, x);
      const float vm = vmax_nan<VEC>(x);
      if (vm != vm || vm == INFINITY) break;  // non-finite: tracked variant below
      if (vm > -INFINITY) {
        st.h = vm * sc;
        break;
      }
    }
    if (st.h > -INFINITY) {
#pragma unroll 2
      for (; k < nv; k += NCT) {
        float x[VEC];
        load_vec<ES>(buf, s, k, x);
        st.s += sum_exp2<VEC>(x, sc, st.h);
      }
      if (st.s < kFastSumMax) return st;  // in range: done
    } else if (k >= nv) {
      return st;  // nothing but -inf in this thread's vectors
    }
    st = rstat_empty();  // overflow or non-finite input
  }
  for (k = ct; k < nv; k += NCT) {
    float x[VEC];
    load_vec<ES>(buf, s, k, x);
    const float vm = vmax_nan<VEC>(x);
    if (!(vm <= st.m)) {  // new maximum, or NaN
      if (vm != vm) {
        bad = true;
      } else {
        const float nh = vm * sc;
        if (NEED_Z && st.h > -INFINITY) st.s *= ex2(st.h - nh);
        st.h = nh;
        st.m = vm;
        int l0 = VEC - 1;
#pragma unroll
        for (int l = VEC - 2; l >= 0; --l)
          if (x[l] == vm) l0 = l;
        st.i = idbase + k * VEC + l0;
      }
    }
    if (NEED_Z && st.h > -INFINITY) st.s += sum_exp2<VEC>(x, sc, st.h);
  }
  if (st.m == INFINITY) bad = true;
  return st;
}

// sum_l exp2(x_l * sc - h) over one vector, as a packed pair of partial sums
// (fma / add on float2: two lanes per instruction on sm_100+).
template <int VEC>
__device__ __forceinline__ float2 sum_exp2_x2(const float* x, float2 sc2, float2 nh2) {
  float e[VEC];
#pragma unroll
  for (int l = 0; l < VEC; l += 2) {
    const float2 a = __ffma2_rn(make_float2(x[l], x[l + 1]), sc2, nh2);
    e[l] = ex2(a.x);
    e[l + 1] = ex2(a.y);
  }
  float2 acc = make_float2(e[0], e[1]);
#pragma unroll
  for (int l = 2; l < VEC; l += 2) acc = __fadd2_rn(acc, make_float2(e[l], e[l + 1]));
  return acc;
}

// Running maximum of one lane's vectors and the lowest id holding it.
template <int VEC>
__device__ __forceinline__ void track_max(const float* x, float vm, int32_t id0, float& m,
                                          int32_t& i) {
  if (vm > m) {  // vectors are visited in increasing id order: the first maximum wins
    int l0 = VEC - 1;
#pragma unroll
    for (int l = VEC - 2; l >= 0; --l)
      if (x[l] == vm) l0 = l;
    m = vm;
    i = id0 + l0;
  }
}

// Pass 1 fast path of one warp of the pass-1 group for a slice pair with no
// masked lanes, when the exact max is not needed: both rows in one loop,
// every lane of the warp using the same references (the warp maximum of the
// lanes' first vectors), so the warp's partials are plain sums.  Returns
// false, uniformly over the warp, on a non-finite input or a lane sum at or
// above kFastSumMax (the caller then runs the general path).  TRACKM: also
// the exact maximum of each row and the lowest id holding it (v0 =
// vocabulary id of vector 0's first element).
template <int ES, bool TRACKM>
__device__ __forceinline__ bool pass1_pair_fast(const unsigned char* bt, const unsigned char* bd,
                                                int32_t nv, float sc, int ct, int NT1, RStat& at,
                                                RStat& ad, int32_t v0) {
  constexpr int VEC = 16 / ES;
  float t[VEC], d[VEC];
  float mt = -INFINITY, md = -INFINITY;
  float rmt = -INFINITY, rmd = -INFINITY;  // running maxima (TRACKM)
  int32_t rit = 0x7fffffff, rid = 0x7fffffff;
  int32_t k = ct;
  if (k < nv) {
    load_vec_raw<ES>(bt, k, t);
    load_vec_raw<ES>(bd, k, d);
    mt = vmax_nan<VEC>(t);
    md = vmax_nan<VEC>(d);
    if (TRACKM) {
      track_max<VEC>(t, mt, v0 + k * VEC, rmt, rit);
      track_max<VEC>(d, md, v0 + k * VEC, rmd, rid);
    }
  }
  // NaN or +inf in a first vector: general path for the whole warp
  if (!__all_sync(0xffffffffu, !(mt != mt || md != md || mt == INFINITY || md == INFINITY)))
    return false;
  const float ht = warp_max_f32(mt) * sc, hd = warp_max_f32(md) * sc;
  const float2 sc2 = make_float2(sc, sc), nht = make_float2(-ht, -ht),
               nhd = make_float2(-hd, -hd);
  float2 at2 = make_float2(0.f, 0.f), ad2 = make_float2(0.f, 0.f);
  if (k < nv) {
    at2 = sum_exp2_x2<VEC>(t, sc2, nht);
    ad2 = sum_exp2_x2<VEC>(d, sc2, nhd);
#pragma unroll 2
    for (k += NT1; k < nv; k += NT1) {
      load_vec_raw<ES>(bt, k, t);
      load_vec_raw<ES>(bd, k, d);
      at2 = __fadd2_rn(at2, sum_exp2_x2<VEC>(t, sc2, nht));
      ad2 = __fadd2_rn(ad2, sum_exp2_x2<VEC>(d, sc2, nhd));
      if (TRACKM) {
        track_max<VEC>(t, vmax_nan<VEC>(t), v0 + k * VEC, rmt, rit);
        track_max<VEC>(d, vmax_nan<VEC>(d), v0 + k * VEC, rmd, rid);
      }
    }
  }
  float st = at2.x + at2.y, sd = ad2.x + ad2.y;
  // every lane's sum below 2^24 keeps each exponent argument <= 24 (full
  // fp32 precision of x sc - h) and the merged sums far from overflow, so a
  // partial whose merge factor flushes to zero holds < 2^-90 of the row
  if (!__all_sync(0xffffffffu, st < kFastSumMax && sd < kFastSumMax)) return false;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {  // two independent shuffle chains
    st += __shfl_xor_sync(0xffffffffu, st, off);
    sd += __shfl_xor_sync(0xffffffffu, sd, off);
  }
  at = RStat{ht, st, -INFINITY, 0x7fffffff};
  ad = RStat{hd, sd, -INFINITY, 0x7fffffff};
  if (TRACKM) {  // warp maximum, lowest id among the lanes holding it
    at.m = warp_max_f32(rmt);
    ad.m = warp_max_f32(rmd);
    at.i = __reduce_min_sync(0xffffffffu, rmt == at.m ? rit : 0x7fffffff);
    ad.i = __reduce_min_sync(0xffffffffu, rmd == ad.m ? rid : 0x7fffffff);
  }
  return true;
}

// Pass 2 of one thread of the pass-2 group: sum of exp2(min(a, b)) over its
// vectors, a = t sc - h_t, b = d sc - k_d with k_d = h_d + delta.  kd_hi +
// kd_lo represents k_d exactly; when kd_lo is 0 (FOLD) the subtraction
// disappears (the caller folds only when that costs at most ~2e-6 in c*).
template <int ES, bool FOLD>
__device__ __forceinline__ float pass2_aligned(const unsigned char* bt, const unsigned char* bd,
                                               int32_t nv, float sc, float ht, float kd_hi,
                                               float kd_lo, int ct, int NT2) {
  constexpr int VEC = 16 / ES;
  const float2 sc2 = make_float2(sc, sc), nht = make_float2(-ht, -ht),
               nkd = make_float2(-kd_hi, -kd_hi), nlo = make_float2(-kd_lo, -kd_lo);
  float2 acc = make_float2(0.f, 0.f);
#pragma unroll 2
  for (int32_t k = ct; k < nv; k += NT2) {
    float t[VEC], d[VEC];
    load_vec_raw<ES>(bt, k, t);
    load_vec_raw<ES>(bd, k, d);
    float e[VEC];
#pragma unroll
    for (int l = 0; l < VEC; l += 2) {
      const float2 a = __ffma2_rn(make_float2(t[l], t[l + 1]), sc2, nht);
      float2 b = __ffma2_rn(make_float2(d[l], d[l + 1]), sc2, nkd);
      if (!FOLD) b = __fadd2_rn(b, nlo);
      e[l] = ex2(fminf(a.x, b.x));
      e[l + 1] = ex2(fminf(a.y, b.y));
    }
#pragma unroll
    for (int l = 0; l < VEC; l += 2) acc = __fadd2_rn(acc, make_float2(e[l], e[l + 1]));
  }
  return acc.x + acc.y;
}

// Pass 2, general path (slices with masked ends or different 16-byte phases):
// sum of exp2(min(a, b - delta)) over the thread's elements.
template <int ES>
__device__ __forceinline__ float pass2_thread(const unsigned char* bt, const Slice& st_,
                                              const unsigned char* bd, const Slice& sd_, float sc,
                                              float ht, float hd, float delta, int ct, int NT2) {
  constexpr int VEC = 16 / ES;
  float acc = 0.f;
  if (st_.hoff == sd_.hoff) {  // same vector grid: vectorised, masked ends
    const int32_t nv = st_.nbytes >> 4;
    for (int32_t k = ct; k < nv; k += NT2) {
      float t[VEC], d[VEC];
      load_vec<ES>(bt, st_, k, t);
      load_vec<ES>(bd, sd_, k, d);
#pragma unroll
      for (int l = 0; l < VEC; ++l)
        acc += ex2(fminf(fmaf(t[l], sc, -ht), fmaf(d[l], sc, -hd) - delta));
    }
  } else {  // different 16-byte phases (V * esize not a multiple of 16)
    for (int32_t i = ct; i < st_.len; i += NT2) {
      const float t = slice_elem<ES>(bt, st_, i), d = slice_elem<ES>(bd, sd_, i);
      acc += ex2(fminf(fmaf(t, sc, -ht), fmaf(d, sc, -hd) - delta));
    }
  }
  return acc;
}

// Locate request r of target row g (largest r with offs[r] <= g) in the
// row_offsets array (a shared-memory copy when it fits).
__device__ __forceinline__ void locate_row(const Params& P, const int32_t* offs, int32_t g,
                                           RowInfo* info) {
  int32_t lo = 0, hi = P.B - 1;
  while (lo < hi) {
    const int32_t mid = (lo + hi + 1) >> 1;
    if (offs[mid] <= g) lo = mid; else hi = mid - 1;
  }
  info->g = g;
  info->r = lo;
  info->off = offs[lo];
  info->off1 = offs[lo + 1];
  info->gd = g - lo;
  info->pair = info->off <= g && g < info->off1 - 1 && info->gd >= 0 && info->gd < P.Nd;
  info->x = -1;
  info->ell = 0;
}

template <int ES>
__device__ __forceinline__ Slice target_slice(const Params& P, const RowInfo& info) {
  return make_slice<ES>(P.tgt + static_cast<size_t>(info.g) * P.V * ES, P.V, info.k, P.S);
}

template <int ES>
__device__ __forceinline__ Slice draft_slice(const Params& P, const RowInfo& info) {
  if (!info.pair) return Slice{nullptr, 0, 0, 0, info.k * P.S};
  return make_slice<ES>(P.drf + static_cast<size_t>(info.gd) * P.V * ES, P.V, info.k, P.S);
}

struct RowsSmem {
  unsigned char* base;
  int32_t rowbuf;
  __device__ __forceinline__ uint32_t full(int s) const { return smem_addr(base + kOffFull + 8 * s); }
  __device__ __forceinline__ uint32_t empty(int s) const { return smem_addr(base + kOffEmpty + 8 * s); }
  __device__ __forceinline__ uint32_t partbar(int s) const {
    return smem_addr(base + kOffPartBar + 8 * s);
  }
  __device__ __forceinline__ uint32_t statsbar(int s) const {
    return smem_addr(base + kOffStatsBar + 8 * s);
  }
  __device__ __forceinline__ float* part(int s, int w) const {
    return reinterpret_cast<float*>(base + kOffPart) + (s * kMaxConsumerWarps + w) * 16;
  }
  __device__ __forceinline__ float* cp(int s) const {
    return reinterpret_cast<float*>(base + kOffCp) + s * kMaxConsumerWarps;
  }
  __device__ __forceinline__ float* stats(int s) const {
    return reinterpret_cast<float*>(base + kOffStats) + s * 8;
  }
  __device__ __forceinline__ RowInfo* info(int s) const {
    return reinterpret_cast<RowInfo*>(base + kOffInfo) + s;
  }
  __device__ __forceinline__ unsigned char* tbuf(int s) const {
    return base + kRowsHdrBytes + s * 2 * rowbuf;
  }
  __device__ __forceinline__ unsigned char* dbuf(int s) const { return tbuf(s) + rowbuf; }
};

// What the producer needs to issue a unit, worked out ahead of time: the
// producer warp plans 32 units at once (one per lane) while it waits for
// stages, so that issuing a unit into a freed stage is a handful of
// instructions (the single-lane search and address arithmetic would
// otherwise delay every refill by a few thousand cycles).
struct UnitPlan {
  int32_t g, k, r, off, off1, pair, gd;
  int32_t tn, dn, thoff, dhoff, len, v0;  // slice buffers (RowInfo fields)
  const unsigned char* ts;                // 16-byte-aligned sources of the copies
  const unsigned char* ds;
};

template <int ES>
__device__ __forceinline__ UnitPlan plan_unit(const Params& P, const int32_t* offs, int32_t u) {
  RowInfo info;
  locate_row(P, offs, u / P.nslices, &info);
  info.k = u % P.nslices;
  const Slice st = target_slice<ES>(P, info);
  const Slice sd = draft_slice<ES>(P, info);
  return UnitPlan{info.g,  info.k,   info.r,  info.off, info.off1, info.pair, info.gd,
                  st.nbytes, sd.nbytes, st.hoff, sd.hoff, st.len,   st.v0,     st.gsrc, sd.gsrc};
}

// The plan held by lane `src` of the producer warp, on every lane.
__device__ __forceinline__ UnitPlan shfl_plan(const UnitPlan& p, int src) {
  constexpr unsigned F = 0xffffffffu;
  UnitPlan q;
  q.g = __shfl_sync(F, p.g, src);
  q.k = __shfl_sync(F, p.k, src);
  q.r = __shfl_sync(F, p.r, src);
  q.off = __shfl_sync(F, p.off, src);
  q.off1 = __shfl_sync(F, p.off1, src);
  q.pair = __shfl_sync(F, p.pair, src);
  q.gd = __shfl_sync(F, p.gd, src);
  q.tn = __shfl_sync(F, p.tn, src);
  q.dn = __shfl_sync(F, p.dn, src);
  q.thoff = __shfl_sync(F, p.thoff, src);
  q.dhoff = __shfl_sync(F, p.dhoff, src);
  q.len = __shfl_sync(F, p.len, src);
  q.v0 = __shfl_sync(F, p.v0, src);
  q.ts = reinterpret_cast<const unsigned char*>(
      __shfl_sync(F, reinterpret_cast<unsigned long long>(p.ts), src));
  q.ds = reinterpret_cast<const unsigned char*>(
      __shfl_sync(F, reinterpret_cast<unsigned long long>(p.ds), src));
  return q;
}

// Producer step (one lane): load the planned unit into stage s.  The stage's
// `full` barrier completes when the bulk copies' bytes have landed and the
// row metadata copied by cp.async has arrived.
__device__ __forceinline__ void issue_unit(const Params& P, const RowsSmem& sm, const UnitPlan& p,
                                           int s) {
  // the bulk copies go out first; the stage's `full` barrier completes once
  // their bytes have landed and three arrivals have happened: this
  // expect_tx, the plain arrival that releases the RowInfo writes, and the
  // completion of the cp.async copies of the row's token, length and uniform
  const uint32_t bar = sm.full(s);
  mbar_arrive_expect_tx(bar, static_cast<uint32_t>(p.tn + p.dn));
  if (p.tn) bulk_g2s(smem_addr(sm.tbuf(s)), p.ts, p.tn, bar);
  if (p.dn) bulk_g2s(smem_addr(sm.dbuf(s)), p.ds, p.dn, bar);
  RowInfo* info = sm.info(s);
  info->g = p.g;
  info->k = p.k;
  info->r = p.r;
  info->off = p.off;
  info->off1 = p.off1;
  info->pair = p.pair;
  info->gd = p.gd;
  info->x = -1;
  info->ell = 0;
  info->tn = p.tn;
  info->dn = p.dn;
  info->thoff = p.thoff;
  info->dhoff = p.dhoff;
  info->len = p.len;
  info->v0 = p.v0;
  mbar_arrive(bar);
  cp_async4(smem_addr(&info->u), P.uniforms + p.g);
  cp_async4(smem_addr(&info->ell), P.lens + p.r);
  if (p.pair) cp_async4(smem_addr(&info->x), P.draft_tokens + p.gd);
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ uint64_t ld_relaxed_u64(const uint64_t* p) {
  uint64_t v;
  asm volatile("ld.relaxed.gpu.global.b64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void st_relaxed_u64(uint64_t* p, uint64_t v) {
  asm volatile("st.relaxed.gpu.global.b64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}


// Threads of the rows kernel: NCW consumer warps, producer, publishers, gatherers.
__host__ __device__ constexpr int rows_threads(int ncw) { return (ncw + 1 + kPublishers + kGatherers) * 32; }

template <int ES, int NCW, bool NEED_Z, bool NEED_CONF, bool TRACK>
__global__ void __launch_bounds__(rows_threads(NCW), 1) rows_kernel(const Params P) {
  static_assert(NCW <= kMaxConsumerWarps, "consumer warps");
  // pass-1 warps [0, NW1), pass-2 warps [NW1, NCW) (labels on)
  const int NW1 = NEED_CONF ? P.nw1 : NCW;
  const int NW2 = NCW - NW1;
  const int NT1 = NW1 * 32, NT2 = NW2 > 0 ? NW2 * 32 : 32;
  constexpr int W_PROD = NCW, W_PUB = NCW + 1, W_GATH = NCW + 1 + kPublishers;
  extern __shared__ __align__(128) unsigned char smem_raw[];
  const RowsSmem sm{smem_raw, P.rowbuf};
  const int32_t N = static_cast<int32_t>(gridDim.x);
  const int32_t c = static_cast<int32_t>(blockIdx.x);
  const int32_t n_units = P.nunits > c ? (P.nunits - c + N - 1) / N : 0;
  const int NS = P.nstages;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const float sc = P.sc;
  uint64_t* parts = reinterpret_cast<uint64_t*>(P.parts);
  const uint64_t tagw = static_cast<uint64_t>(P.tag) << 32;
  grid_dep_launch_dependents();  // the finalize kernel may take SMs this grid leaves

  // ---- set-up: row_offsets into shared memory (when they fit), barriers,
  //      the first NS units in flight
  int32_t* offs_sm = reinterpret_cast<int32_t*>(smem_raw + kRowsHdrBytes + NS * 2 * P.rowbuf);
  const int32_t* offs = P.offs;
  if (P.offs_smem) {
    for (int32_t i = tid; i <= P.B; i += blockDim.x) offs_sm[i] = __ldg(P.offs + i);
    offs = offs_sm;
  }
  __syncthreads();
  // producer warp: plans of units [plan_base, plan_base + 32), one per lane
  UnitPlan plan{};
  int32_t plan_base = 0;
  if (warp == W_PROD) {
    if (lane == 0) {
      for (int s = 0; s < NS; ++s) {
        mbar_init(sm.full(s), 3);  // bulk-copy arm, RowInfo release, cp.async completion
        // pass-1 warps (labels off) or the pass-2 group, + publisher + gatherer
        mbar_init(sm.empty(s), (NEED_CONF ? 1 : NW1) + 2);
        mbar_init(sm.partbar(s), NW1);
        mbar_init(sm.statsbar(s), 1);
      }
      mbar_init(smem_addr(smem_raw + kOffTailBar), 1);
      fence_mbar_init();
    }
    if (lane < n_units) plan = plan_unit<ES>(P, offs, c + lane * N);
    for (int i = 0; i < NS && i < n_units; ++i) {
      const UnitPlan q = shfl_plan(plan, i);
      if (lane == 0) issue_unit(P, sm, q, i);
    }
  }
  __syncthreads();

  bool timeout = false;   // a wait on this CTA's own barriers gave up
  bool xtimeout = false;  // a wait on other CTAs' published words gave up
  if (warp < NCW) {
    // =============================== consumer warps
    // Labels on: warps [0, NW1) run pass 1, warps [NW1, NCW) pass 2, each
    // group on its own stream of units.  Labels off: all run pass 1.
    if (warp < NW1) {
      const int ct = tid;
      RingPos rp{0, 0u};
      for (int32_t i = 0; i < n_units; ++i, rp.next(NS)) {  // pass 1 of unit i
        const int s = rp.idx;
        mbar_wait(sm.full(s), rp.par, timeout);
        const RowInfo info = *sm.info(s);
        bool bad = false;
        const Slice s_t = slice_t(info), s_d = slice_d(info);
        RStat a_t, a_d;
        const bool fast = NEED_Z && info.pair && slice_aligned<ES>(s_t) &&
                          slice_aligned<ES>(s_d) &&
                          pass1_pair_fast<ES, TRACK>(sm.tbuf(s), sm.dbuf(s), s_t.nbytes >> 4, sc,
                                                     ct, NT1, a_t, a_d, s_t.v0);
        if (!fast) {  // general path: per-thread partials, then a warp merge
          a_t = pass1_thread<ES, NEED_Z, TRACK>(sm.tbuf(s), s_t, sc, ct, NT1, bad);
          a_d = info.pair ? pass1_thread<ES, NEED_Z, TRACK>(sm.dbuf(s), s_d, sc, ct, NT1, bad)
                          : rstat_empty();
          rstat_warp_reduce2<true>(a_t, a_d);
        }
        const unsigned badw = __ballot_sync(0xffffffffu, bad);
        if (lane == 0) {
          float* w = sm.part(s, warp);
          w[R_HT] = a_t.h; w[R_ST] = a_t.s; w[R_MT] = a_t.m; w[R_IT] = __int_as_float(a_t.i);
          w[R_HD] = a_d.h; w[R_SD] = a_d.s; w[R_MD] = a_d.m; w[R_ID] = __int_as_float(a_d.i);
          w[R_BAD] = __int_as_float((badw ? SV_DEVERR_NAN : 0) | (timeout ? SV_DEVERR_TIMEOUT : 0));
          mbar_arrive(sm.partbar(s));
          if (!NEED_CONF) mbar_arrive(sm.empty(s));  // no pass 2: release the stage
        }
      }
    } else {
      const int ct = tid - NT1;
      RingPos rp{0, 0u};
      for (int32_t j = 0; j < n_units; ++j, rp.next(NS)) {  // pass 2 of unit j, then release its stage
        const int s = rp.idx;
        mbar_wait(sm.full(s), rp.par, timeout);
        const RowInfo info = *sm.info(s);
        if (info.pair) {
          mbar_wait(sm.statsbar(s), rp.par, timeout);
          const float* st = sm.stats(s);
          const float ht = st[0], hd = st[4], delta = st[6];
          const Slice s_t = slice_t(info), s_d = slice_d(info);
          float part;
          if (slice_aligned<ES>(s_t) && slice_aligned<ES>(s_d)) {
            // k_d = h_d + delta as hi + lo (two-sum, exact)
            const float kd_hi = hd + delta;
            const float kd_lo = (hd - kd_hi) + delta;
            const int32_t nv = s_t.nbytes >> 4;
            if (fabsf(ht) < 64.f && fabsf(kd_hi) < 64.f)
              part = pass2_aligned<ES, true>(sm.tbuf(s), sm.dbuf(s), nv, sc, ht, kd_hi, 0.f, ct,
                                             NT2);
            else
              part = pass2_aligned<ES, false>(sm.tbuf(s), sm.dbuf(s), nv, sc, ht, kd_hi, kd_lo,
                                              ct, NT2);
          } else {
            part = pass2_thread<ES>(sm.tbuf(s), s_t, sm.dbuf(s), s_d, sc, ht, hd, delta, ct, NT2);
          }
          part = warp_sum_f32(part);
          if (lane == 0) sm.cp(s)[warp - NW1] = part;
        }
        // the whole group is done with the stage; its first warp writes the
        // unit's label partial (warp partials summed in order) and releases
        // the stage
        named_bar_sync(1, NT2);
        if (warp == NW1 && lane == 0) {
          if (info.pair) {
            float cs = 0.f;
            for (int w = 0; w < NW2; ++w) cs += sm.cp(s)[w];
            uint64_t* dst = parts + (static_cast<size_t>(info.g) * kMaxSlices + info.k) * kPartWords;
            st_relaxed_u64(dst + R_CP, tagw | __float_as_uint(cs / sm.stats(s)[1]));
          }
          mbar_arrive(sm.empty(s));
        }
      }
    }
  } else if (warp == W_PROD) {
    // =============================== producer warp
    // After unit j releases stage s, issue unit j + NS into it.  Plans for
    // the next 32 units are made (all lanes, one unit each) before waiting,
    // off the refill's path.
    RingPos rp{0, 0u};
    for (int32_t j = 0; j < n_units; ++j, rp.next(NS)) {
      const int s = rp.idx;
      const int32_t nxt = j + NS;
      if (nxt < n_units && nxt >= plan_base + 32) {
        plan_base += 32;
        if (plan_base + lane < n_units) plan = plan_unit<ES>(P, offs, c + (plan_base + lane) * N);
      }
      mbar_wait(sm.empty(s), rp.par, timeout);
      const UnitPlan q = shfl_plan(plan, (nxt - plan_base) & 31);
      if (lane == 0 && nxt < n_units) issue_unit(P, sm, q, s);
      __syncwarp();
    }
  } else if (warp < W_GATH) {
    // =============================== publisher warps (unit i by warp i % kPublishers)
    RingPos rp{0, 0u};
    for (int w = 0; w < warp - W_PUB; ++w) rp.next(NS);
    for (int32_t i = warp - W_PUB; i < n_units; i += kPublishers) {
      const int s = rp.idx;
      mbar_wait(sm.partbar(s), rp.par, timeout);
      mbar_wait(sm.full(s), rp.par, timeout);
      for (int w = 0; w < kPublishers; ++w) rp.next(NS);
      const RowInfo info = *sm.info(s);
      RStat b_t = rstat_empty(), b_d = rstat_empty();
      int flags = 0;
      if (lane < NW1) {
        const float* w = sm.part(s, lane);
        b_t = RStat{w[R_HT], w[R_ST], w[R_MT], __float_as_int(w[R_IT])};
        b_d = RStat{w[R_HD], w[R_SD], w[R_MD], __float_as_int(w[R_ID])};
        flags = __float_as_int(w[R_BAD]);
      }
      rstat_warp_reduce2<TRACK>(b_t, b_d);
      flags = __reduce_or_sync(0xffffffffu, flags);
      const Slice s_t = slice_t(info);
      const bool hasx = info.pair && info.x >= s_t.v0 && info.x < s_t.v0 + s_t.len;
      float xt = 0.f, xd = 0.f;
      if (hasx) {
        xt = slice_elem<ES>(sm.tbuf(s), s_t, info.x - s_t.v0);
        xd = slice_elem<ES>(sm.dbuf(s), slice_d(info), info.x - s_t.v0);
      }
      // lane w < R_NWORDS publishes word w of the partial, tagged (selects,
      // no divergent branches)
      uint32_t word = hasx ? 1u : 0u;
      word = lane == R_XD ? __float_as_uint(xd) : word;
      word = lane == R_XT ? __float_as_uint(xt) : word;
      word = lane == R_BAD ? static_cast<uint32_t>(flags) : word;
      word = lane == R_ID ? static_cast<uint32_t>(b_d.i) : word;
      word = lane == R_MD ? __float_as_uint(b_d.m) : word;
      word = lane == R_SD ? __float_as_uint(b_d.s) : word;
      word = lane == R_HD ? __float_as_uint(b_d.h) : word;
      word = lane == R_IT ? static_cast<uint32_t>(b_t.i) : word;
      word = lane == R_MT ? __float_as_uint(b_t.m) : word;
      word = lane == R_ST ? __float_as_uint(b_t.s) : word;
      word = lane == R_HT ? __float_as_uint(b_t.h) : word;
      if (lane < R_NWORDS) {
        uint64_t* dst = parts + (static_cast<size_t>(info.g) * kMaxSlices + info.k) * kPartWords;
        st_relaxed_u64(dst + lane, tagw | word);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(sm.empty(s));
    }
  } else {
    // =============================== gatherer warps (unit j by warp j % kGatherers)
    const int q = warp - W_GATH;
    RingPos rp{0, 0u};
    for (int w = 0; w < q; ++w) rp.next(NS);
    for (int32_t j = q; j < n_units; j += kGatherers) {
      const int s = rp.idx;
      const uint32_t par = rp.par;
      for (int w = 0; w < kGatherers; ++w) rp.next(NS);
      mbar_wait(sm.full(s), par, timeout);
      const RowInfo info = *sm.info(s);
      // start polling once this CTA has finished pass 1 of the unit (the
      // other slices of the row are handled in the same round elsewhere)
      mbar_wait(sm.partbar(s), par, timeout);
      // wait until the S partials of this row carry this call's tag (lane =
      // slice): poll one word per slice, then read all words and check each
      const uint64_t* row_parts = parts + static_cast<size_t>(info.g) * kMaxSlices * kPartWords;
      const bool mine = lane < P.nslices;
      const uint64_t* src = row_parts + (mine ? lane : 0) * kPartWords;
      uint32_t wv[R_NWORDS] = {};
      auto full_read = [&]() {
        bool ok = true;
        if (mine) {
#pragma unroll
          for (int w = 0; w < R_NWORDS; ++w) {
            const uint64_t v = ld_relaxed_u64(src + w);
            wv[w] = static_cast<uint32_t>(v);
            ok &= (v & 0xffffffff00000000ull) == tagw;
          }
        }
        return ok;
      };
      bool done = false;
      const uint64_t t0 = globaltimer_ns();
      for (uint32_t n = 0; !done; ++n) {
        const bool seen = !mine || (ld_relaxed_u64(src + R_BAD) & 0xffffffff00000000ull) == tagw;
        if (__all_sync(0xffffffffu, seen)) done = __all_sync(0xffffffffu, full_read());
        if (!done) {
          // a wait on other CTAs gives up after P.xwait_ns: the row's
          // statistics are then wrong and the call reports a timeout, but
          // this CTA's own pipeline (every wait below) runs on unchanged
          if (xtimeout || globaltimer_ns() - t0 >= P.xwait_ns) {
            xtimeout = true;
            break;
          }
          if (P.poll_ns > 0) __nanosleep(P.poll_ns);
        }
      }
      RStat gt = rstat_empty(), gdr = rstat_empty();
      int flags = 0;
      float xt = 0.f, xd = 0.f;
      bool hasx = false;
      if (mine) {
        gt = RStat{__uint_as_float(wv[R_HT]), __uint_as_float(wv[R_ST]), __uint_as_float(wv[R_MT]),
                   static_cast<int32_t>(wv[R_IT])};
        gdr = RStat{__uint_as_float(wv[R_HD]), __uint_as_float(wv[R_SD]),
                    __uint_as_float(wv[R_MD]), static_cast<int32_t>(wv[R_ID])};
        flags = static_cast<int>(wv[R_BAD]);
        xt = __uint_as_float(wv[R_XT]);
        xd = __uint_as_float(wv[R_XD]);
        hasx = wv[R_HASX] != 0;
      }
      rstat_warp_reduce2<TRACK>(gt, gdr);
      flags = __reduce_or_sync(0xffffffffu, flags) | (timeout || xtimeout ? SV_DEVERR_TIMEOUT : 0);
      const unsigned xl = __ballot_sync(0xffffffffu, hasx);
      if (xl) {
        xt = __shfl_sync(0xffffffffu, xt, __ffs(xl) - 1);
        xd = __shfl_sync(0xffffffffu, xd, __ffs(xl) - 1);
      }
      if (lane == 0) {
        float* st = sm.stats(s);
        st[0] = gt.h;
        st[1] = gt.s;
        st[4] = gdr.h;
        st[5] = gdr.s;
        st[6] = __log2f(gdr.s) - __log2f(gt.s);  // delta of pass 2
        mbar_arrive(sm.statsbar(s));
      }
      if (info.k == 0 && lane == 0) {  // row epilogue, once per row
        const int32_t g = info.g, ell = info.ell;
        const bool ok = info.off <= g && g < info.off1 && info.off1 - info.off == ell && ell >= 1 &&
                        ell <= P.max_len && info.off >= info.r;
        const bool tokok = info.x >= 0 && info.x < P.V;
        int fl = flags;
        if (NEED_Z && !(gt.s > 0.f && gt.s < INFINITY)) fl |= SV_DEVERR_NAN;
        if (NEED_Z && info.pair && !(gdr.s > 0.f && gdr.s < INFINITY)) fl |= SV_DEVERR_NAN;
        if (TRACK && !(gt.m > -INFINITY && gt.m < INFINITY)) fl |= SV_DEVERR_NAN;
        if (TRACK && info.pair && !(gdr.m > -INFINITY && gdr.m < INFINITY)) fl |= SV_DEVERR_NAN;
        if (!ok) fl |= SV_DEVERR_LEN;
        if (info.pair && !tokok) fl |= SV_DEVERR_TOKEN;
        int acc = 0;
        if (ok && info.pair && tokok) {
          if (P.mode == SV_GREEDY) {
            acc = info.x == gt.i;
          } else {
            // p_t(x) / p_d(x) = 2^(a - b) * s_d / s_t, a = x_t sc - h_t, b = x_d sc - h_d
            const float ratio =
                exp2f(fmaf(xt, sc, -gt.h) - fmaf(xd, sc, -gdr.h)) * (gdr.s / gt.s);
            acc = info.u < ratio;
          }
        }
        RowRec rr;
        rr.mt = gt.h; rr.zt = gt.s; rr.md = gdr.h; rr.zd = gdr.s;
        rr.argt = gt.i; rr.acc = acc; rr.pick = -1; rr.flags = fl;
        P.rec[g] = rr;
        st_relaxed_u64(parts + static_cast<size_t>(g) * kMaxSlices * kPartWords + R_REC,
                       tagw | rec_mark(acc != 0, fl));
        if (TRACK && P.out_row_stats != nullptr) {
          // Z relative to the true max: s * 2^(h - m sc)
          float* o = P.out_row_stats + 3 * static_cast<size_t>(g);
          o[0] = gt.m / P.T;
          o[1] = gt.s * exp2f(-fmaf(gt.m, sc, -gt.h));
          o[2] = __int_as_float(gt.i);
          if (info.pair) {
            float* o2 = P.out_row_stats + 3 * (static_cast<size_t>(P.Nt) + info.gd);
            o2[0] = gdr.m / P.T;
            o2[1] = gdr.s * exp2f(-fmaf(gdr.m, sc, -gdr.h));
            o2[2] = __int_as_float(gdr.i);
          }
        }
        if (fl) raise_error(P, fl);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(sm.empty(s));
    }
  }
  if ((timeout || xtimeout) && lane == 0) raise_error(P, SV_DEVERR_TIMEOUT);
  if (!P.fuse) return;
  // ---- tail: every role has left its loop and every copy has been consumed,
  //      so stage 0's buffers are free; this CTA finishes requests blockIdx.x,
  //      blockIdx.x + gridDim.x, ... as soon as their rows are done elsewhere
  //      (skipped after a timeout: the stages may still be in use, or the
  //      statistics are wrong)
  if (__syncthreads_or(timeout || xtimeout ? 1 : 0)) return;
  const FinishSmem fs{reinterpret_cast<DrawSel*>(smem_raw + kOffTail),
                      reinterpret_cast<float*>(smem_raw + kOffTail + 64),
                      reinterpret_cast<uint32_t*>(smem_raw + kOffPart),  // free after the loops
                      sm.tbuf(0), sm.dbuf(0), smem_addr(smem_raw + kOffTailBar)};
  uint32_t phase = 0;
  for (int32_t r = c; r < P.B; r += N)
    if (!finish_request<ES, rows_threads(NCW) / 32>(P, r, fs, true, phase)) break;
}

}  // namespace sv
