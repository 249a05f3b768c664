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
// mass at or below kZeroResidual counts as zero: the draw then uses p_t, as
// the exact method does when max(0, p_t - p_d) vanishes.
#pragma once

#include "sv_common.cuh"

namespace sv {

// A residual mass sum max(0, p_t - p_d) at or below this is taken for zero
// (the draw then uses p_t).  The fp32 slice masses of two equal
// distributions differ by rounding of order 1e-7, so an exact zero is not
// seen as one.  The cutoff sits below the 1e-6 near-tie margin: a residual
// mass of 1e-6 or more is always drawn from (its fp32 estimate is off by far
// less than the 5e-7 between the two), and a smaller one is a near tie of
// the choice between the residual and p_t.  A slice whose mass was rounding
// only is found and dropped by the draw itself (its recomputed weights are
// all zero).
constexpr float kZeroResidual = 4.76837158203125e-07f;  // 2^-21

constexpr int kDrawThreads = 512;  // threads per CTA of the draw kernel
constexpr int kDrawWarps = kDrawThreads / 32;
constexpr int kD_OffBar = 0;     // mbarrier of the slice copies
constexpr int kD_OffSel = 64;    // DrawSel
constexpr int kD_OffRed = 128;   // [kDrawWarps] reduction scratch (floats / ints)
constexpr int kD_OffMarks = 1024;  // [SV_MAX_LEN] row marks
constexpr int kD_HdrBytes = kD_OffMarks + 4 * SV_MAX_LEN;
static_assert(kD_OffRed + 4 * kDrawWarps <= kD_OffMarks, "draw header");

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

__device__ __forceinline__ uint64_t ld_cg_u64(const uint64_t* p) {
  uint64_t v;
  asm volatile("ld.global.cg.b64 %0, [%1];" : "=l"(v) : "l"(p));
  return v;
}

// Two adjacent 64-bit words (16-byte aligned), each read whole.
__device__ __forceinline__ void ld_cg_u64x2(const uint64_t* p, uint64_t& a, uint64_t& b) {
  asm volatile("ld.global.cg.v2.b64 {%0, %1}, [%2];" : "=l"(a), "=l"(b) : "l"(p));
}

// Value of word w of the published record of (row g, slice k).
__device__ __forceinline__ float part_value(const Params& P, int32_t g, int32_t k, int w) {
  return __uint_as_float(static_cast<uint32_t>(ld_cg_u64(part_words(P.parts, g, k) + w)));
}

// c* of every drafted row of request r, by one warp: per row the slices'
// partials (lane = slice) summed in the warp's fixed tree order, eight rows'
// loads in flight at a time.
__device__ __forceinline__ void sum_labels(const Params& P, int32_t r, int32_t off, int32_t ell,
                                           int lane) {
  if (P.out_conf == nullptr) return;
  for (int32_t j0 = 0; j0 < ell - 1; j0 += 8) {
    float v[8];
#pragma unroll
    for (int q = 0; q < 8; ++q)
      v[q] = j0 + q < ell - 1 && lane < P.nslices ? part_value(P, off + j0 + q, lane, R_CP) : 0.f;
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const float c = warp_sum_f32(v[q]);
      if (lane == 0 && j0 + q < ell - 1) P.out_conf[off - r + j0 + q] = c;
    }
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

// Shared memory a CTA needs to finish requests: the slice choice, NW words
// of reduction scratch, SV_MAX_LEN accept marks, two slice buffers of
// P.rowbuf bytes and an mbarrier (count 1) for their copies.
struct FinishSmem {
  DrawSel* sel;
  float* red;
  uint32_t* marks;
  unsigned char* buf_t;
  unsigned char* buf_d;
  uint32_t bar;
};

// Label c* of row g: the slices' partials (lane = slice) summed over the
// warp in a fixed tree order; every lane gets it.
__device__ __forceinline__ float row_label(float cp_lane) { return warp_sum_f32(cp_lane); }

// What one warp reads of target row g (lane = slice k < nslices): the
// slice's pass-1 statistics of both rows, its label partial, and (lane 0)
// the row's mark.  Loads all go out before any is checked.
struct RowWords {
  uint64_t v[8];  // HT, ST, MT, IT, HD, SD, CP, REC
};

// Everything of request r after the rows kernel's passes, by one CTA of NW
// warps (all threads call it): the first-rejection scan, the labels, the
// accepted drafts, and the final token -- the argmax of the stopping row
// (greedy) or the inverse-CDF draw (unfiltered sampling).
//
// Warp j reads target row off + j, j = warp, warp + NW, ... in one round of
// loads (one lane per slice): its mark (accept decision, error bits), its
// label, and its statistics merged from the slices' partials exactly as the
// rows kernel merged them (same lanes, same order: the same bits).  When the
// request has at most NW rows, every warp keeps its row's slice masses P_k
// and residual masses R_k in registers, so the stopping row's warp can pick
// the slice as soon as a_r is known (longer requests: warp 0 reads row a_r
// again).  The block then walks the chosen slice pair.  A slice whose
// recomputed weights turn out all zero (its fp32 mass was rounding only) is
// dropped and the choice repeated.
//
// wait_ready: the rows kernel is still running elsewhere (its own tail);
// every published word is used only once it carries this call's tag.
// Returns false if a wait gave up (after raising the timeout flag).
template <int ES, int NW>
__device__ __forceinline__ bool finish_request(const Params& P, int32_t r, const FinishSmem& fs,
                                               bool wait_ready, uint32_t& phase) {
  constexpr int NT = NW * 32;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

  // ---- inputs only (before the rows kernel has finished, when launched as
  //      its dependent)
  const int32_t off = __ldg(P.offs + r), off1 = __ldg(P.offs + r + 1), ell = __ldg(P.lens + r);
  const bool ok = ell >= 1 && ell <= P.max_len && off1 - off == ell && off >= r &&
                  off1 <= P.Nt && (r != 0 || off == 0) && (r != P.B - 1 || off1 == P.Nt) &&
                  off - r + ell - 1 <= P.Nd;
  if (!ok) {  // uniform over the CTA
    if (tid == 0) raise_error(P, SV_DEVERR_LEN);
    return true;
  }
  const float u = __ldg(P.uniforms + off + ell - 1);
  const int32_t xtok = tid < ell - 1 ? __ldg(P.draft_tokens + off - r + tid) : -1;
  grid_dep_wait();  // published partials from the rows kernel
  const uint64_t tagw = static_cast<uint64_t>(P.tag) << 32;
  const bool sample = P.mode == SV_SAMPLE;
  const bool has_cp = sample || P.out_conf != nullptr;  // pass 2 ran
  const int S = P.nslices;

  // a published word v read from wp; while the rows kernel runs, taken only
  // once it carries this call's tag (bounded re-polls)
  bool stale = false;
  auto settle = [&](const uint64_t* wp, uint64_t v) {
    if (wait_ready && (v & 0xffffffff00000000ull) != tagw) {
      const uint64_t t0 = globaltimer_ns();
      while (((v = ld_cg_u64(wp)) & 0xffffffff00000000ull) != tagw) {
        if (globaltimer_ns() - t0 >= P.xwait_ns) {
          stale = true;
          break;
        }
        __nanosleep(128);
      }
    }
    return v;
  };
  // row j's words, settled: which ones exist depends on the row and mode
  auto read_row = [&](int32_t j) {
    const int32_t g = off + j;
    const bool drafted = j < ell - 1;
    RowWords rw{};
    if (lane < S) {
      const uint64_t* wp = part_words(P.parts, g, lane);
      const int at[8] = {R_HT, R_ST, R_MT, R_IT, R_HD, R_SD, R_CP, R_REC};
      static_assert(R_HT % 2 == 0 && R_ST == R_HT + 1 && R_MT % 2 == 0 && R_IT == R_MT + 1 &&
                        R_HD % 2 == 0 && R_SD == R_HD + 1 && R_CP % 2 == 0 && R_REC == R_CP + 1,
                    "record words read in aligned pairs");
#pragma unroll
      for (int q = 0; q < 8; q += 2) ld_cg_u64x2(wp + at[q], rw.v[q], rw.v[q + 1]);
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const bool need = q < 4 || (drafted && (q < 6 ? sample : q == 6 ? has_cp : false)) ||
                          (q == 7 && lane == 0);
        if (need) rw.v[q] = settle(wp + at[q], rw.v[q]);
      }
    }
    return rw;
  };
  const auto f32 = [](uint64_t v) { return __uint_as_float(static_cast<uint32_t>(v)); };

  // ---- one round of loads: marks, labels, statistics and slice masses
  bool resid = false;  // of the row this warp keeps
  float w = 0.f, pk = 0.f;
  RowRec rj{};
  auto masses = [&](int32_t j, const RowWords& rw) {
    resid = j < ell - 1;
    RStat t = rstat_empty(), d = rstat_empty();
    if (lane < S) {
      t = RStat{f32(rw.v[0]), f32(rw.v[1]), f32(rw.v[2]), static_cast<int32_t>(static_cast<uint32_t>(rw.v[3]))};
      if (resid) d = RStat{f32(rw.v[4]), f32(rw.v[5]), -INFINITY, 0x7fffffff};
    }
    rstat_warp_reduce2<true>(t, d);
    rj.mt = t.h; rj.zt = t.s; rj.md = d.h; rj.zd = d.s; rj.argt = t.i;
    w = pk = 0.f;
    if (sample && lane < S) {
      const float h = f32(rw.v[0]), s = f32(rw.v[1]);
      pk = h > -INFINITY ? s * exp2f(h - rj.mt) / rj.zt : 0.f;
      w = resid ? fmaxf(0.f, pk - f32(rw.v[6])) : pk;
    }
  };
  const bool spec = ell <= NW;
  for (int32_t j = warp; j < ell; j += NW) {
    const RowWords rw = read_row(j);
    if (lane == 0) fs.marks[j] = static_cast<uint32_t>(rw.v[7]);
    if (j < ell - 1 && P.out_conf != nullptr) {
      const float c = row_label(lane < S ? f32(rw.v[6]) : 0.f);
      if (lane == 0) P.out_conf[off - r + j] = c;
    }
    if (spec) masses(j, rw);
  }
  if (wait_ready && __syncthreads_or(stale ? 1 : 0)) {
    if (tid == 0) raise_error(P, SV_DEVERR_TIMEOUT);
    return false;
  }
  if (!wait_ready) __syncthreads();  // the marks
  int32_t a = ell - 1;  // first drafted position not accepted
  for (int32_t j = 0; j < ell - 1; ++j)
    if (!(fs.marks[j] >> 31)) {
      a = j;
      break;
    }
  const int sw = spec ? a : 0;  // the warp that holds the stopping row's masses
  if (!spec && warp == 0) masses(a, read_row(a));
  if (stale && lane == 0) raise_error(P, SV_DEVERR_TIMEOUT);
  const int32_t trow_i = off + a;
  // accepted drafts, -1 after the final token, error bits of the rows up to a_r
  for (int32_t j = tid; j < ell; j += NT) {
    if (j < a) P.out_tokens[off + j] = j == tid ? xtok : __ldg(P.draft_tokens + off - r + j);
    else if (j > a) P.out_tokens[off + j] = -1;
    const int fl = static_cast<int>(fs.marks[j] & 0x7fffffffu);
    if (j <= a && fl) raise_error(P, fl);
  }
  if (tid == 0) P.out_accept_len[r] = a;
  if (!sample) {  // greedy: the argmax of the stopping row
    if (warp == sw && lane == 0) P.out_tokens[trow_i] = rj.argt;
    __syncthreads();  // the marks are free for the next request
    return true;
  }

  bool timeout = false;
  bool picked = false;
  for (int attempt = 0; attempt <= S; ++attempt, phase ^= 1u) {
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
        fs.sel->k = k;
        fs.sel->residual = resid;
        fs.sel->rec = rj;
      }
      if (lane == k) fs.sel->need = fmaxf(0.f, target - (incl - w));
    }
    __syncthreads();
    const int32_t k = fs.sel->k;
    const bool residual = fs.sel->residual != 0;
    if (k < 0) break;  // no mass anywhere: non-finite statistics
    const Slice s_t = make_slice<ES>(P.tgt + static_cast<size_t>(trow_i) * P.V * ES, P.V, k, P.S);
    Slice s_d = make_slice<ES>(P.drf + static_cast<size_t>(off - r + a) * P.V * ES, P.V, k, P.S);
    if (!residual) s_d.nbytes = 0, s_d.len = 0;
    if (tid == 0) {
      mbar_arrive_expect_tx(fs.bar, static_cast<uint32_t>(s_t.nbytes + s_d.nbytes));
      if (s_t.nbytes) bulk_g2s(smem_addr(fs.buf_t), s_t.gsrc, s_t.nbytes, fs.bar);
      if (s_d.nbytes) bulk_g2s(smem_addr(fs.buf_d), s_d.gsrc, s_d.nbytes, fs.bar);
    }
    mbar_wait(fs.bar, phase, timeout);
    if (__syncthreads_or(timeout ? 1 : 0)) {
      timeout = true;
      break;
    }
    const RowRec rr = fs.sel->rec;
    DrawRow dr;
    dr.sc = P.sc;
    dr.ht = rr.mt;
    dr.hd = rr.md;
    dr.ratio = rr.zt / rr.zd;
    dr.residual = residual;
    // weights in units of 1 / z_t: the mass to pass is need * z_t
    const float need = fs.sel->need * rr.zt;
    const int32_t E = (s_t.len + NT - 1) / NT;  // elements per thread
    const int32_t i0 = min(s_t.len, tid * E), i1 = min(s_t.len, i0 + E);
    float wsum = 0.f;
#pragma unroll 4
    for (int32_t i = i0; i < i1; ++i) {
      const float t = slice_elem<ES>(fs.buf_t, s_t, i);
      const float d = residual ? slice_elem<ES>(fs.buf_d, s_d, i) : 0.f;
      wsum += dr.w(t, d);
    }
    float lo, hi, tot;
    block_scan_bounds<NW>(wsum, fs.red, lo, hi, tot);
    if (tot > 0.f) {
      // the owner: the run whose interval holds `need`, or the last run with
      // positive weight when rounding left need >= tot
      const bool own = lo < hi && ((lo <= need && need < hi) || (need >= tot && hi == tot));
      const unsigned ob = __ballot_sync(0xffffffffu, own);
      if (ob) {  // the owner's warp walks the owner's run, 32 elements a step
        const int ol = __ffs(ob) - 1;
        const int32_t oi0 = __shfl_sync(0xffffffffu, i0, ol), oi1 = __shfl_sync(0xffffffffu, i1, ol);
        const float left = __shfl_sync(0xffffffffu, need - lo, ol);  // mass to pass inside it
        float base = 0.f;
        int32_t p = -1, last = -1;
        for (int32_t b0 = oi0; b0 < oi1 && p < 0; b0 += 32) {
          const int32_t i = b0 + lane;
          float wv = 0.f;
          if (i < oi1) {
            const float t = slice_elem<ES>(fs.buf_t, s_t, i);
            const float d = residual ? slice_elem<ES>(fs.buf_d, s_d, i) : 0.f;
            wv = dr.w(t, d);
          }
          const float run = base + warp_incl_scan(wv);
          const unsigned hitm = __ballot_sync(0xffffffffu, wv > 0.f && run > left);
          const unsigned posm = __ballot_sync(0xffffffffu, wv > 0.f);
          if (posm) last = b0 + 31 - __clz(posm);
          if (hitm) p = b0 + __ffs(hitm) - 1;
          base = __shfl_sync(0xffffffffu, run, 31);
        }
        if (p < 0) p = last;
        if (lane == 0) P.out_tokens[trow_i] = s_t.v0 + p;
      }
      picked = true;
      phase ^= 1u;
      break;
    }
    // every weight of the slice is zero: drop it and choose again
    if (warp == sw && lane == k) w = 0.f;
    __syncthreads();  // the buffers are free again before the next copy
  }
  if (!picked && tid == 0) {  // no mass anywhere (or a wait gave up)
    raise_error(P, timeout ? SV_DEVERR_TIMEOUT : SV_DEVERR_NAN);
    P.out_tokens[trow_i] = fs.sel->rec.argt;
  }
  if (timeout) {  // one more bounded wait for the copy still in flight
    bool again = false;
    mbar_wait(fs.bar, phase, again);
    phase ^= 1u;
    return false;
  }
  __syncthreads();  // the buffers, the marks and the choice are free for the next request
  return true;
}

// Unfiltered sampling, as its own launch after the rows kernel: one CTA per
// request.
template <int ES>
__global__ void __launch_bounds__(kDrawThreads) finalize_draw_kernel(const Params P) {
  extern __shared__ __align__(128) unsigned char smem[];
  const FinishSmem fs{reinterpret_cast<DrawSel*>(smem + kD_OffSel),
                      reinterpret_cast<float*>(smem + kD_OffRed),
                      reinterpret_cast<uint32_t*>(smem + kD_OffMarks), smem + kD_HdrBytes,
                      smem + kD_HdrBytes + P.rowbuf, smem_addr(smem + kD_OffBar)};
  if (threadIdx.x == 0) {
    mbar_init(fs.bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  uint32_t phase = 0;
  finish_request<ES, kDrawWarps>(P, static_cast<int32_t>(blockIdx.x), fs, false, phase);
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
