// sv_rows.cuh -- the bandwidth-bound rows kernel (no top-k / top-p filter).
//
// One thread-block cluster of C CTAs per target row g.  CTA `rank` owns the
// vocabulary slice [rank * S, rank * S + S) of target row g and, when row g
// scores a drafted token, of its draft partner row.  The slice pair is
// brought from HBM into the CTA's shared memory once, with bulk copies in
// kChunks pieces so that the statistics pass starts on the first piece
// while the rest is still in flight.
//
//  pass 1 (as pieces land): per-thread online max / sum exp / argmax of both
//         rows (log-sum-exp merge algebra), then a CTA merge;
//  exchange: every CTA stores its partial record into every other CTA's
//         shared memory (distributed shared memory), one cluster barrier,
//         then every CTA merges the C records in rank order;
//  pass 2 (only when labels are requested): c* = sum_v min(p_t(v), p_d(v))
//         = 1 - 1/2 ||p_t - p_d||_1 over the resident slice, one exp2 per
//         element pair: min(p_t, p_d) = exp2(min(log2 p_t, log2 p_d));
//         partial sums go to CTA 0 through distributed shared memory;
//  epilogue (CTA 0): row statistics, label, accept decision of the drafted
//         token -- sampling: u * p_d(x) < p_t(x), greedy: x == argmax_t.
//
// Confidence label: DSpark tutorial, "置信度预测头".  Accept rule and the
// first-rejection structure: DSpark tutorial, "推测解码的两步流程"; DFlash /
// Spec V2 page, A3 (lossless rejection sampling after Leviathan et al.).
#pragma once

#include "sv_common.cuh"

namespace sv {

// Shared-memory header layout of the rows kernel (bytes from the base).
constexpr int kOffBars = 0;                                   // kChunks mbarriers
constexpr int kOffRecs = 64;                                  // kMaxCluster records
constexpr int kOffCpart = kOffRecs + kMaxCluster * kRecWords * 4;  // kMaxCluster floats
constexpr int kOffScratch = kOffCpart + kMaxCluster * 4;      // reduction scratch
constexpr int kOffInfo = kOffScratch + 64 * 4;                // per-CTA row info
static_assert(kOffInfo + 64 <= kHdrBytes, "rows kernel header");

// Record word layout.
enum { R_MT = 0, R_ST, R_IT, R_MD, R_SD, R_ID, R_XT, R_XD, R_HASX, R_BAD };

struct RowInfo {
  int32_t r, j, pair, gd, x, ok, tokok, pad;
};

// Locate request r of target row g (largest r with offs[r] <= g) and check
// the request's layout.
__device__ __forceinline__ RowInfo locate_row(const Params& P, int32_t g) {
  RowInfo info{};
  int32_t lo = 0, hi = P.B - 1;
  while (lo < hi) {
    const int32_t mid = (lo + hi + 1) >> 1;
    if (__ldg(P.offs + mid) <= g) lo = mid; else hi = mid - 1;
  }
  const int32_t r = lo;
  const int32_t off = __ldg(P.offs + r), off1 = __ldg(P.offs + r + 1);
  const int32_t ell = __ldg(P.lens + r);
  info.r = r;
  info.j = g - off;
  info.ok = off <= g && g < off1 && off1 - off == ell && ell >= 1 && ell <= P.max_len && off >= r;
  info.gd = g - r;
  info.pair = info.ok && info.j < ell - 1 && info.gd >= 0 && info.gd < P.Nd;
  info.x = info.pair ? __ldg(P.draft_tokens + info.gd) : -1;
  info.tokok = info.x >= 0 && info.x < P.V;
  return info;
}

// Pass-1 update of one thread's statistics with VEC elements of one vector.
template <int VEC, bool NEED_Z>
__device__ __forceinline__ void stat_update(Stat& st, float& nm, const float* x, int32_t id0,
                                            float sc, bool& bad) {
  float vmax = x[0];
#pragma unroll
  for (int l = 1; l < VEC; ++l) vmax = fmax_nan(vmax, x[l]);
  bad |= (vmax != vmax);
  if (vmax > st.m) {
    if (NEED_Z) st.s *= ex2((st.m - vmax) * sc);
    st.m = vmax;
    nm = vmax * sc;
    int l0 = VEC - 1;
#pragma unroll
    for (int l = VEC - 2; l >= 0; --l)
      if (x[l] == vmax) l0 = l;
    st.i = id0 + l0;
  }
  if (NEED_Z && st.m > -INFINITY) {
    float e[VEC];
#pragma unroll
    for (int l = 0; l < VEC; ++l) e[l] = ex2(fmaf(x[l], sc, -nm));
#pragma unroll
    for (int w = VEC / 2; w > 0; w >>= 1)
#pragma unroll
      for (int l = 0; l < w; ++l) e[l] += e[l + w];
    st.s += e[0];
  }
}

// Pass 1 over the vectors [k0, k1) of a slice buffer, strided by the block.
template <int ES, bool NEED_Z>
__device__ __forceinline__ void stats_range(const unsigned char* buf, const Slice& s, int32_t k0,
                                            int32_t k1, float sc, Stat& st, float& nm, bool& bad) {
  constexpr int VEC = 16 / ES;
  for (int32_t k = k0 + threadIdx.x; k < k1; k += kThreads) {
    float x[VEC];
    load_vec<ES>(buf, s, k, x);
    stat_update<VEC, NEED_Z>(st, nm, x, s.v0 + k * VEC - s.hoff, sc, bad);
  }
}

// Pass 2: partial sum of exp2(min(t * sc - lt, d * sc - ld)) over the slice.
template <int ES>
__device__ __forceinline__ float overlap_range(const unsigned char* bt, const Slice& st_,
                                               const unsigned char* bd, const Slice& sd_,
                                               float sc, float lt, float ld) {
  constexpr int VEC = 16 / ES;
  float acc = 0.f;
  if (st_.hoff == sd_.hoff) {  // same vector grid: vectorised
    const int32_t nv = st_.nbytes >> 4;
    for (int32_t k = threadIdx.x; k < nv; k += kThreads) {
      float t[VEC], d[VEC];
      load_vec<ES>(bt, st_, k, t);
      load_vec<ES>(bd, sd_, k, d);
      float e[VEC];
#pragma unroll
      for (int l = 0; l < VEC; ++l) e[l] = ex2(fminf(fmaf(t[l], sc, -lt), fmaf(d[l], sc, -ld)));
#pragma unroll
      for (int w = VEC / 2; w > 0; w >>= 1)
#pragma unroll
        for (int l = 0; l < w; ++l) e[l] += e[l + w];
      acc += e[0];
    }
  } else {  // rows with different 16-byte phase (V * esize not a multiple of 16)
    for (int32_t i = threadIdx.x; i < st_.len; i += kThreads) {
      const float t = slice_elem<ES>(bt, st_, i), d = slice_elem<ES>(bd, sd_, i);
      acc += ex2(fminf(fmaf(t, sc, -lt), fmaf(d, sc, -ld)));
    }
  }
  return acc;
}

template <int ES, bool NEED_Z, bool NEED_CONF>
__global__ void __launch_bounds__(kThreads) rows_kernel(const Params P) {
  extern __shared__ __align__(128) unsigned char smem[];
  const uint32_t rank = cluster_ctarank();
  const uint32_t csize = cluster_nctarank();
  const int32_t g = static_cast<int32_t>(cluster_id_x());
  const int tid = threadIdx.x;
  float* recs = reinterpret_cast<float*>(smem + kOffRecs);
  float* cpart = reinterpret_cast<float*>(smem + kOffCpart);
  float* scratch = reinterpret_cast<float*>(smem + kOffScratch);
  RowInfo* sinfo = reinterpret_cast<RowInfo*>(smem + kOffInfo);
  unsigned char* buf_t = smem + kHdrBytes;
  unsigned char* buf_d = buf_t + P.rowbuf;
  const uint32_t bar0 = smem_addr(smem + kOffBars);

  cluster_arrive_relaxed();  // this CTA has started (completed before the first DSMEM store)

  if (tid == 0) {
    *sinfo = locate_row(P, g);
#pragma unroll
    for (int c = 0; c < kChunks; ++c) mbar_init(bar0 + 8 * c, 1);
    fence_mbar_init();
  }
  __syncthreads();
  const RowInfo info = *sinfo;

  const unsigned char* trow = P.tgt + static_cast<size_t>(g) * P.V * ES;
  const unsigned char* drow = P.drf + static_cast<size_t>(info.gd) * P.V * ES;
  const Slice s_t = make_slice<ES>(trow, P.V, rank, P.S);
  Slice s_d = make_slice<ES>(drow, P.V, rank, P.S);
  if (!info.pair) s_d.nbytes = 0, s_d.len = 0;

  if (tid == 0) {
    for (int c = 0; c < kChunks; ++c) {
      int32_t tlo, thi, dlo, dhi;
      chunk_range(s_t.nbytes, c, &tlo, &thi);
      chunk_range(s_d.nbytes, c, &dlo, &dhi);
      const uint32_t bar = bar0 + 8 * c;
      mbar_arrive_expect_tx(bar, static_cast<uint32_t>((thi - tlo) + (dhi - dlo)));
      if (thi > tlo) bulk_g2s(smem_addr(buf_t + tlo), s_t.gsrc + tlo, thi - tlo, bar);
      if (dhi > dlo) bulk_g2s(smem_addr(buf_d + dlo), s_d.gsrc + dlo, dhi - dlo, bar);
    }
  }

  // ---- pass 1: statistics while the pieces land
  const float sc = P.sc;
  Stat st_t = stat_empty(), st_d = stat_empty();
  float nm_t = 0.f, nm_d = 0.f;
  bool bad = false, timeout = false;
  for (int c = 0; c < kChunks; ++c) {
    if (!mbar_wait_bounded(bar0 + 8 * c, 0, kSpinLimit)) timeout = true;
    int32_t lo, hi;
    chunk_range(s_t.nbytes, c, &lo, &hi);
    stats_range<ES, NEED_Z>(buf_t, s_t, lo >> 4, hi >> 4, sc, st_t, nm_t, bad);
    if (info.pair) {
      chunk_range(s_d.nbytes, c, &lo, &hi);
      stats_range<ES, NEED_Z>(buf_d, s_d, lo >> 4, hi >> 4, sc, st_d, nm_d, bad);
    }
  }
  const bool any_bad = __syncthreads_or(bad ? 1 : 0) != 0;
  const bool any_timeout = __syncthreads_or(timeout ? 1 : 0) != 0;
  st_t = block_merge(st_t, sc, scratch);
  if (info.pair) st_d = block_merge(st_d, sc, scratch);

  // ---- exchange the CTA records through distributed shared memory
  if (tid == 0) {
    float* my = scratch + 32;  // staging of this CTA's record
    my[R_MT] = st_t.m; my[R_ST] = st_t.s; my[R_IT] = __int_as_float(st_t.i);
    my[R_MD] = st_d.m; my[R_SD] = st_d.s; my[R_ID] = __int_as_float(st_d.i);
    const bool hasx = info.pair && info.tokok && info.x >= s_t.v0 && info.x < s_t.v0 + s_t.len;
    my[R_XT] = hasx ? slice_elem<ES>(buf_t, s_t, info.x - s_t.v0) : 0.f;
    my[R_XD] = hasx ? slice_elem<ES>(buf_d, s_d, info.x - s_d.v0) : 0.f;
    my[R_HASX] = hasx ? 1.f : 0.f;
    my[R_BAD] = __int_as_float((any_bad ? SV_DEVERR_NAN : 0) | (any_timeout ? SV_DEVERR_TIMEOUT : 0));
  }
  __syncthreads();
  cluster_wait_acquire();  // every CTA of the cluster has started
  if (tid < static_cast<int>(csize) * kRecWords) {
    const int dst = tid / kRecWords, w = tid % kRecWords;
    const float* my = scratch + 32;
    const uint32_t a = smem_addr(recs + rank * kRecWords + w);
    st_cluster_u32(mapa(a, dst), __float_as_uint(w <= R_BAD ? my[w] : 0.f));
  }
  cluster_arrive_release();
  cluster_wait_acquire();

  // ---- merge the C records in rank order (identical in every thread)
  Stat gt = stat_empty(), gdr = stat_empty();
  float xt = 0.f, xd = 0.f;
  int flags = 0;
  for (uint32_t q = 0; q < csize; ++q) {
    const float* rq = recs + q * kRecWords;
    gt = stat_merge(gt, Stat{rq[R_MT], rq[R_ST], __float_as_int(rq[R_IT])}, sc);
    gdr = stat_merge(gdr, Stat{rq[R_MD], rq[R_SD], __float_as_int(rq[R_ID])}, sc);
    if (rq[R_HASX] != 0.f) { xt = rq[R_XT]; xd = rq[R_XD]; }
    flags |= __float_as_int(rq[R_BAD]);
  }
  if (!(gt.m > -INFINITY && gt.m < INFINITY)) flags |= SV_DEVERR_NAN;
  if (info.pair && !(gdr.m > -INFINITY && gdr.m < INFINITY)) flags |= SV_DEVERR_NAN;
  if (NEED_Z && !(gt.s > 0.f && gt.s < INFINITY)) flags |= SV_DEVERR_NAN;
  if (NEED_Z && info.pair && !(gdr.s > 0.f && gdr.s < INFINITY)) flags |= SV_DEVERR_NAN;

  // ---- pass 2: label c* over the resident slice pair
  float conf = 0.f;
  if (NEED_CONF && info.pair) {
    const float lt = fmaf(gt.m, sc, __log2f(gt.s));
    const float ld = fmaf(gdr.m, sc, __log2f(gdr.s));
    float part = overlap_range<ES>(buf_t, s_t, buf_d, s_d, sc, lt, ld);
    part = block_sum(part, scratch);
    if (tid == 0) st_cluster_u32(mapa(smem_addr(cpart + rank), 0), __float_as_uint(part));
    cluster_arrive_release();
    cluster_wait_acquire();
    if (rank == 0 && tid == 0)
      for (uint32_t q = 0; q < csize; ++q) conf += cpart[q];
  }

  // ---- epilogue in CTA 0
  if (rank == 0 && tid == 0) {
    if (!info.ok) flags |= SV_DEVERR_LEN;
    if (info.pair && !info.tokok) flags |= SV_DEVERR_TOKEN;
    int acc = 0;
    if (info.pair && info.tokok) {
      if (P.mode == SV_GREEDY) {
        acc = info.x == gt.i;
      } else {
        // ratio p_t(x) / p_d(x) = exp2(((xt - mt) - (xd - md)) * sc) * zd / zt
        const float delta = (xt - gt.m) - (xd - gdr.m);
        const float ratio = exp2f(delta * sc) * (gdr.s / gt.s);
        const float u = __ldg(P.uniforms + g);
        acc = u < ratio;
      }
    }
    RowRec rr;
    rr.mt = gt.m; rr.zt = gt.s; rr.md = gdr.m; rr.zd = gdr.s;
    rr.argt = gt.i; rr.acc = acc; rr.pick = -1; rr.flags = flags;
    P.rec[g] = rr;
    if (NEED_CONF && info.pair && P.out_conf != nullptr) P.out_conf[info.gd] = conf;
    if (P.out_row_stats != nullptr) {
      float* o = P.out_row_stats + 3 * static_cast<size_t>(g);
      o[0] = gt.m / P.T; o[1] = gt.s; o[2] = __int_as_float(gt.i);
      if (info.pair) {
        float* q = P.out_row_stats + 3 * (static_cast<size_t>(P.Nt) + info.gd);
        q[0] = gdr.m / P.T; q[1] = gdr.s; q[2] = __int_as_float(gdr.i);
      }
    }
    if (flags) raise_error(P, flags);
  }

  if (any_timeout) {  // never leave while a copy into this CTA may still land
    for (int c = 0; c < kChunks; ++c) mbar_wait_bounded(bar0 + 8 * c, 0, kSpinLimit);
  }
}

}  // namespace sv
