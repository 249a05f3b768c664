// sv_finalize.cuh -- per-request accept scan and final token.
//
// Per request r (DSpark tutorial, "推测解码的两步流程"; DSpine page, "原理"):
// a_r = index of the first rejected drafted position (l_r - 1 if none); the
// accepted drafts are emitted, then one final token:
//   greedy              argmax of target row a_r (rejected or bonus row);
//   filtered sampling   the draw the rows kernel already made for row a_r;
//   unfiltered sampling an inverse-CDF draw over ascending ids with the
//                       request's last uniform from max(0, p_t - p_d) of the
//                       rejected row pair, or from p_t of the bonus row after
//                       a fully accepted block (DFlash / Spec V2 page, A3 and
//                       its Leviathan et al. citation).
//
// The unfiltered draw runs on one CTA per request in two steps.  The slice
// is chosen first from per-slice masses the rows kernel left in the
// workspace: the target mass P_k of slice k from its pass-1 partial, and for
// a residual draw R_k = max(0, P_k - C_k) with C_k = sum of min(p_t, p_d)
// over the slice (the slice's label partial).  Only the chosen slice pair is
// then read again from HBM and walked element by element with the mass left
// over: running sums in (thread, element) order are sums in ascending token
// id.  fp32 slice masses differ from the exact ones by a few 1e-7 in
// probability, inside the near-tie margin the oracle reports.  A residual
// mass below kZeroResidual counts as zero: the draw then uses p_t, as the
// exact method does when max(0, p_t - p_d) vanishes.
#pragma once

#include "sv_common.cuh"

namespace sv {

// A residual mass sum max(0, p_t - p_d) below this is taken for zero (the
// draw then uses p_t): the fp32 slice masses of two equal distributions
// differ by rounding of order 1e-7, and a rejection with so little residual
// mass happens with probability below it (it needs p_d(x) = 0 or p_t within
// this of p_d everywhere).
constexpr float kZeroResidual = 7.62939453125e-06f;  // 2^-17

constexpr int kDrawThreads = 512;  // threads per CTA of the draw kernel
constexpr int kDrawWarps = kDrawThreads / 32;
constexpr int kD_OffBar = 0;    // mbarrier of the slice copies
constexpr int kD_OffSel = 64;   // DrawSel
constexpr int kD_OffRed = 128;  // [kDrawWarps] reduction scratch (floats / ints)
constexpr int kD_HdrBytes = 1024;
static_assert(kD_OffRed + 4 * kDrawWarps <= kD_HdrBytes, "draw header");

struct ReqInfo {
  int32_t ok, off, ell, a, residual, pad[3];
};

// Request r's layout and its first rejected position a_r, by one warp (every
// lane gets the result): lane j looks at drafted position j, so the accept
// flags are read in one round of independent loads instead of a dependent
// chain of l_r - 1.
__device__ __forceinline__ ReqInfo scan_request(const Params& P, int32_t r, int lane) {
  ReqInfo q{};
  const int32_t off = __ldg(P.offs + r), off1 = __ldg(P.offs + r + 1), ell = __ldg(P.lens + r);
  q.ok = ell >= 1 && ell <= P.max_len && off1 - off == ell && off >= r && off1 <= P.Nt &&
         (r != 0 || off == 0) && (r != P.B - 1 || off1 == P.Nt);
  q.off = off;
  q.ell = ell;
  int32_t a = 0;
  if (q.ok) {
    a = ell - 1;  // every drafted token accepted
    for (int32_t base = 0; base < ell - 1; base += 32) {
      const int32_t j = base + lane;
      const bool rejected = j < ell - 1 && !P.rec[off + j].acc;
      const unsigned m = __ballot_sync(0xffffffffu, rejected);
      if (m) {
        a = base + __ffs(m) - 1;
        break;
      }
    }
  }
  q.a = a;
  q.residual = a < ell - 1;
  // the draft partner of the stopping row must exist (guards corrupt offsets)
  if (q.residual && (off - r + a < 0 || off - r + a >= P.Nd)) q.ok = 0;
  return q;
}

// Weight of token v for the final draw, in units of 1 / z_t: the residual
// max(0, p_t - p_d) * z_t = max(0, 2^a - (z_t / z_d) 2^b), or p_t * z_t = 2^a,
// with a = t sc - h_t and b = d sc - h_d.
struct DrawRow {
  float ht, hd, ratio, sc;  // references and z_t / z_d
  bool residual;
  __device__ __forceinline__ float w(float t, float d) const {
    const float pt = ex2(fmaf(t, sc, -ht));
    if (!residual) return pt;
    return fmaxf(0.f, pt - ratio * ex2(fmaf(d, sc, -hd)));
  }
};

// c* of every drafted row of request r: the rows kernel's per-slice partials
// summed in slice order.  Lanes of one warp take one row each.
__device__ __forceinline__ void sum_labels(const Params& P, int32_t r, int32_t off, int32_t ell,
                                           int lane) {
  if (P.out_conf == nullptr) return;
  for (int32_t j = lane; j < ell - 1; j += 32) {
    const float* cp = P.cpart + static_cast<size_t>(off + j) * 32;
    float c = 0.f;
    for (int q = 0; q < P.nslices; ++q) c += cp[q];
    P.out_conf[off - r + j] = c;
  }
}

// Inclusive warp scan of v over lanes.
__device__ __forceinline__ float warp_incl_scan(float v) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const float n = __shfl_up_sync(0xffffffffu, v, off);
    if (lane >= off) v += n;
  }
  return v;
}

// Block-wide min of an int over NW warps; every thread gets the result.
template <int NW>
__device__ __forceinline__ int block_min_int(int v, int* scratch) {
  v = __reduce_min_sync(0xffffffffu, v);
  if ((threadIdx.x & 31) == 0) scratch[threadIdx.x >> 5] = v;
  __syncthreads();
  int r = scratch[0];
  for (int w = 1; w < NW; ++w) r = min(r, scratch[w]);
  __syncthreads();
  return r;
}

// Prefix bounds over the block of one float v >= 0 per thread, in thread
// order: thread t's interval [lo, hi) of the running sum, built so that hi
// of one thread and lo of the next are the same float (the intervals tile
// [0, total) with no gap or overlap whatever the rounding), and the total
// (equal to hi of the last thread).  Every thread gets its own bounds.
template <int NW>
__device__ __forceinline__ void block_scan_bounds(float v, float* scratch, float& lo, float& hi,
                                                  float& total) {
  const int lane = threadIdx.x & 31, w0 = threadIdx.x >> 5;
  const float incl = warp_incl_scan(v);
  const float prev = __shfl_up_sync(0xffffffffu, incl, 1);
  if (lane == 31) scratch[w0] = incl;
  __syncthreads();
  float base = 0.f, tot = 0.f;
  for (int w = 0; w < NW; ++w) {
    if (w < w0) base += scratch[w];
    tot += scratch[w];
  }
  __syncthreads();
  lo = lane == 0 ? base : base + prev;
  hi = base + incl;
  total = tot;
}

// The slice chosen for a draw: slice index (-1: no mass anywhere), the mass
// to pass inside it (probability units), the kind of draw and the stopping
// row's record.
struct DrawSel {
  int32_t k;
  int32_t residual;
  float need;
  int32_t pad;
  RowRec rec;  // record of the stopping row
};
static_assert(kD_OffSel + sizeof(DrawSel) <= kD_OffRed, "draw header");

__device__ __forceinline__ uint64_t ld_cg_u64(const uint64_t* p) {
  uint64_t v;
  asm volatile("ld.global.cg.b64 %0, [%1];" : "=l"(v) : "l"(p));
  return v;
}

// Unfiltered sampling: one CTA per request.  For requests of at most
// kDrawWarps rows warp j reads target row off + j as if it were the stopping
// row (its record and slice masses, one lane per slice) while thread j reads
// row j's accept flag, so the masses of the stopping row are in registers as
// soon as a_r is known (longer requests: warp 0 reads them afterwards); that
// warp picks the slice and the block walks it.  A slice whose recomputed
// weights turn out all zero (its fp32 mass was rounding only) is dropped and
// the choice repeated.
template <int ES>
__global__ void __launch_bounds__(kDrawThreads) finalize_draw_kernel(const Params P) {
  extern __shared__ __align__(128) unsigned char smem[];
  const int32_t r = static_cast<int32_t>(blockIdx.x);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  DrawSel* sel = reinterpret_cast<DrawSel*>(smem + kD_OffSel);
  float* fred = reinterpret_cast<float*>(smem + kD_OffRed);
  int* ired = reinterpret_cast<int*>(smem + kD_OffRed);
  unsigned char* buf_t = smem + kD_HdrBytes;
  unsigned char* buf_d = buf_t + P.rowbuf;
  const uint32_t bar = smem_addr(smem + kD_OffBar);
  const uint64_t* parts = reinterpret_cast<const uint64_t*>(P.parts);

  // ---- inputs only, before the rows kernel has finished
  const int32_t off = __ldg(P.offs + r), off1 = __ldg(P.offs + r + 1), ell = __ldg(P.lens + r);
  const bool ok = ell >= 1 && ell <= P.max_len && off1 - off == ell && off >= r &&
                  off1 <= P.Nt && (r != 0 || off == 0) && (r != P.B - 1 || off1 == P.Nt) &&
                  off - r + ell - 1 <= P.Nd;
  if (!ok) {  // uniform over the CTA
    if (tid == 0) raise_error(P, SV_DEVERR_LEN);
    return;
  }
  const float u = __ldg(P.uniforms + off + ell - 1);
  const int32_t xtok = tid < ell - 1 ? __ldg(P.draft_tokens + off - r + tid) : -1;
  if (tid == 0) {
    mbar_init(bar, 1);
    fence_mbar_init();
  }
  grid_dep_wait();  // row records, label partials and pass-1 partials from the rows kernel

  // slice masses of target row off + j as the stopping row, one lane per
  // slice: P_k, and for a drafted row the residual mass R_k (w)
  bool resid = false;
  float w = 0.f, pk = 0.f;
  RowRec rj{};
  auto load_masses = [&](int32_t j) {
    const int32_t g = off + j;
    resid = j < ell - 1;
    rj = P.rec[g];
    if (lane < P.nslices) {
      const uint64_t* pw = parts + (static_cast<size_t>(g) * kMaxSlices + lane) * kPartWords;
      const float h = __uint_as_float(static_cast<uint32_t>(ld_cg_u64(pw + R_HT)));
      const float s = __uint_as_float(static_cast<uint32_t>(ld_cg_u64(pw + R_ST)));
      pk = h > -INFINITY ? s * exp2f(h - rj.mt) / rj.zt : 0.f;
      w = pk;
      if (resid)
        w = fmaxf(0.f, pk - __ldcg(P.cpart + static_cast<size_t>(g) * kMaxSlices + lane));
    }
  };
  const bool spec = ell <= kDrawWarps;
  if (spec && warp < ell) load_masses(warp);
  if (warp == 1) sum_labels(P, r, off, ell, lane);
  // thread j: accept flag and error flags of row j (threads cover l_r <= SV_MAX_LEN)
  int32_t first = ell - 1, rflags = 0;
  if (tid < ell) {
    rflags = __ldcg(&P.rec[off + tid].flags);
    if (tid < ell - 1 && !__ldcg(&P.rec[off + tid].acc)) first = tid;
  }
  const int32_t a = block_min_int<kDrawWarps>(first, ired);  // first rejected position
  const int sw = spec ? a : 0;  // the warp that holds the stopping row's masses
  if (!spec && warp == 0) load_masses(a);
  const int32_t trow_i = off + a;
  // accepted drafts, -1 after the final token, flags of the rows up to a_r
  if (tid < ell) {
    if (tid < a) P.out_tokens[off + tid] = xtok;
    else if (tid > a) P.out_tokens[off + tid] = -1;
    if (tid <= a && rflags) raise_error(P, rflags);
  }

  bool timeout = false;
  bool picked = false;
  uint32_t phase = 0;  // parity of the copy barrier's current phase
  for (int attempt = 0; attempt <= P.nslices; ++attempt, phase ^= 1u) {
    if (warp == sw) {  // choose the slice: first whose interval passes u * total
      float incl = warp_incl_scan(w);
      float total = __shfl_sync(0xffffffffu, incl, 31);
      if (resid && !(total > kZeroResidual)) {  // no residual mass (rounding only): p_t
        resid = false;
        w = pk;
        incl = warp_incl_scan(w);
        total = __shfl_sync(0xffffffffu, incl, 31);
      }
      const float target = u * total;
      const unsigned hit = __ballot_sync(0xffffffffu, w > 0.f && target < incl);
      const unsigned pos = __ballot_sync(0xffffffffu, w > 0.f);
      const int k = hit ? __ffs(hit) - 1 : (pos ? 31 - __clz(pos) : -1);
      if (lane == 0) {
        sel->k = k;
        sel->residual = resid;
        sel->rec = rj;
      }
      if (lane == k) sel->need = fmaxf(0.f, target - (incl - w));
    }
    __syncthreads();
    const int32_t k = sel->k;
    const bool residual = sel->residual != 0;
    if (k < 0) break;  // no mass anywhere: non-finite statistics
    const Slice s_t = make_slice<ES>(P.tgt + static_cast<size_t>(trow_i) * P.V * ES, P.V, k, P.S);
    Slice s_d = make_slice<ES>(P.drf + static_cast<size_t>(off - r + a) * P.V * ES, P.V, k, P.S);
    if (!residual) s_d.nbytes = 0, s_d.len = 0;
    if (tid == 0) {
      mbar_arrive_expect_tx(bar, static_cast<uint32_t>(s_t.nbytes + s_d.nbytes));
      if (s_t.nbytes) bulk_g2s(smem_addr(buf_t), s_t.gsrc, s_t.nbytes, bar);
      if (s_d.nbytes) bulk_g2s(smem_addr(buf_d), s_d.gsrc, s_d.nbytes, bar);
    }
    mbar_wait(bar, phase, timeout);
    if (__syncthreads_or(timeout ? 1 : 0)) {
      timeout = true;
      break;
    }
    const RowRec rr = sel->rec;
    DrawRow dr;
    dr.sc = P.sc;
    dr.ht = rr.mt;
    dr.hd = rr.md;
    dr.ratio = rr.zt / rr.zd;
    dr.residual = residual;
    // weights in units of 1 / z_t: the mass to pass is need * z_t
    const float need = sel->need * rr.zt;
    const int32_t E = (s_t.len + kDrawThreads - 1) / kDrawThreads;  // elements per thread
    const int32_t i0 = min(s_t.len, tid * E), i1 = min(s_t.len, i0 + E);
    float wsum = 0.f;
#pragma unroll 4
    for (int32_t i = i0; i < i1; ++i) {
      const float t = slice_elem<ES>(buf_t, s_t, i);
      const float d = residual ? slice_elem<ES>(buf_d, s_d, i) : 0.f;
      wsum += dr.w(t, d);
    }
    float lo, hi, tot;
    block_scan_bounds<kDrawWarps>(wsum, fred, lo, hi, tot);
    if (tot > 0.f) {
      // the owner: the run whose interval holds `need`, or the last run with
      // positive weight when rounding left need >= tot
      const bool own = lo < hi && ((lo <= need && need < hi) || (need >= tot && hi == tot));
      if (own) {
        const float left = need - lo;  // mass to pass inside this run
        float run = 0.f;
        int32_t p = -1, last = -1;
        for (int32_t i = i0; i < i1; ++i) {
          const float t = slice_elem<ES>(buf_t, s_t, i);
          const float d = residual ? slice_elem<ES>(buf_d, s_d, i) : 0.f;
          const float wv = dr.w(t, d);
          run += wv;
          if (wv > 0.f) last = i;
          if (run > left) {
            p = i;
            break;
          }
        }
        if (p < 0) p = last;
        P.out_tokens[trow_i] = s_t.v0 + p;
      }
      picked = true;
      break;
    }
    // every weight of the slice is zero: drop it and choose again
    if (warp == sw && lane == k) w = 0.f;
    __syncthreads();  // the buffers are free again before the next copy
  }
  if (!picked && tid == 0) {  // no mass anywhere (or a wait gave up)
    raise_error(P, timeout ? SV_DEVERR_TIMEOUT : SV_DEVERR_NAN);
    P.out_tokens[trow_i] = P.rec[trow_i].argt;
  }
  if (warp == 0 && lane == 0) P.out_accept_len[r] = a;
  if (timeout) {  // one more bounded wait for a copy still in flight
    bool again = false;
    mbar_wait(bar, phase, again);
  }
}

// Greedy and filtered sampling: the final token is already known per row.
// One warp per request: lane 0 scans and writes, all lanes sum labels.
__global__ void __launch_bounds__(kThreads) finalize_select_kernel(const Params P) {
  const int32_t r = blockIdx.x * kWarps + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (r >= P.B) return;  // whole warps leave together
  grid_dep_wait();          // the row records come from the rows kernel
  const ReqInfo q = scan_request(P, r, lane);
  if (!q.ok) {
    if (lane == 0) raise_error(P, SV_DEVERR_LEN);
    return;
  }
  sum_labels(P, r, q.off, q.ell, lane);
  const RowRec& fr = P.rec[q.off + q.a];
  const int32_t final_tok = P.mode == SV_GREEDY ? fr.argt : fr.pick;
  if (lane == 0) P.out_accept_len[r] = q.a;
  int flags = 0;
  for (int32_t j = lane; j < q.ell; j += 32) {
    int32_t v = -1;
    if (j < q.a) v = __ldg(P.draft_tokens + q.off - r + j);
    else if (j == q.a) v = final_tok;
    P.out_tokens[q.off + j] = v;
    if (j <= q.a) flags |= P.rec[q.off + j].flags;
  }
  flags = __reduce_or_sync(0xffffffffu, flags);
  if (lane == 0 && flags) raise_error(P, flags);
}

}  // namespace sv
