// sv_gfilter.cuh -- the verify step under top-k / top-p filters whose kept
// set may be any size (top-p over the whole vocabulary, top_k above
// SV_MAX_FILTER_K).
//
// Filter order as in the other paths (DSpine page, "加速效果": temperature,
// top_p, top_k): z = logit / T; keep the top_k tokens by (z desc, id asc);
// renormalise; keep the shortest prefix of that order whose cumulative
// probability reaches top_p; renormalise.  A kept set is then a prefix of
// the (value desc, id asc) order, so one threshold describes it: a value key
// t and an id, the set being the tokens above t plus the tokens at t up to
// that id.
//
// The top-k threshold is found by bisection over the value key (16 bits for
// bf16, 32 for fp32), one counting pass per probe; the top-p threshold by a
// radix select, one pass per 8-bit digit: a histogram of counts and of
// weights w = exp2(x sc - h) (h = x_max sc) over the elements that match the
// digits chosen so far, then the bin where the cumulative mass from the top
// reaches the target.  Weights are summed as
// fixed-point integers of 2^-40, so every sum is exact and the same in any
// order.  Inside the tie class of the final value, the cut falls after c
// tokens of equal weight, c from integer arithmetic; a counting pass finds
// the id of the c-th.
//
//  gfilter_rows_kernel      one CTA per target row: the kept sets of the row
//                           and of its draft partner, the label
//                           sum_v min(p_t, p_d) over both kept sets (DSpark
//                           tutorial, "置信度预测头"), the accept test
//                           u * p_d(x) < p_t(x) (greedy: x is the argmax).
//  gfilter_requests_kernel  one CTA per request: the first rejection, the
//                           outputs, and the final token -- an inverse-CDF
//                           draw over ascending ids from max(0, p_t - p_d)
//                           on the kept sets of the rejected pair, or from p_t
//                           of the bonus row (DSpark tutorial,
//                           "推测解码的两步流程"; DFlash / Spec V2 page, A3).
#pragma once

#include "sv_common.cuh"
#include "sv_filter.cuh"
#include "sv_finalize.cuh"

namespace sv {

constexpr int kGThreads = 512;
constexpr int kGWarps = kGThreads / 32;
constexpr float kGFix = 1099511627776.f;  // 2^40: weight units of the exact sums

// A row's kept set and statistics (stored in the row's FiltRow slot of the
// workspace).
struct GRow {
  float h;           // reference x_max * sc
  float z;           // kept mass: sum over the kept set of exp2(x sc - h)
  float xmax;        // row maximum (raw logit)
  int32_t argmax;    // lowest id holding it
  uint32_t thr_key;  // kept: key > thr_key, or key == thr_key and id <= thr_id
  int32_t thr_id;
  int32_t n_kept;
  int32_t flags;
};
static_assert(sizeof(GRow) <= sizeof(FiltRow), "GRow in a FiltRow slot");

// Logit v of a row (read-only path).
template <int ES>
__device__ __forceinline__ float load_elem(const unsigned char* row, int32_t v) {
  if (ES == 2)
    return __uint_as_float(static_cast<uint32_t>(__ldg(reinterpret_cast<const uint16_t*>(row) + v))
                           << 16);
  return __ldg(reinterpret_cast<const float*>(row) + v);
}

// Value key of a logit: order_key's bits that tell bf16 values apart.
template <int ES>
__device__ __forceinline__ uint32_t gkey(float x) {
  return ES == 2 ? order_key(x) >> 16 : order_key(x);
}

__device__ __forceinline__ bool gkept(const GRow& g, uint32_t key, int32_t id) {
  return key > g.thr_key || (key == g.thr_key && id <= g.thr_id);
}

// Fixed-point weight of logit x (exact integer units of 2^-40).
__device__ __forceinline__ unsigned long long gweight(float x, float sc, float h) {
  return __float2ull_rn(ex2(fmaf(x, sc, -h)) * kGFix);
}

// ---- block reductions (all threads of the CTA call them; every thread gets
//      the result)
__device__ __forceinline__ unsigned long long g_sum_u64(unsigned long long v,
                                                        unsigned long long* red) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  __syncthreads();
  unsigned long long t = 0;
  for (int w = 0; w < kGWarps; ++w) t += red[w];
  __syncthreads();
  return t;
}

__device__ __forceinline__ unsigned long long g_max_u64(unsigned long long v,
                                                        unsigned long long* red) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v = max(v, __shfl_xor_sync(0xffffffffu, v, off));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  __syncthreads();
  unsigned long long t = 0;
  for (int w = 0; w < kGWarps; ++w) t = max(t, red[w]);
  __syncthreads();
  return t;
}

__device__ __forceinline__ float g_sum_f32(float v, float* red) {
  v = warp_sum_f32(v);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  __syncthreads();
  float t = 0.f;
  for (int w = 0; w < kGWarps; ++w) t += red[w];
  __syncthreads();
  return t;
}

// Visit every element (id, logit) of a row of V logits: thread t takes the
// 16-byte vectors t, t + NT, ... of the row's aligned cover.
template <int ES, typename F>
__device__ __forceinline__ void g_for_row(const unsigned char* row, int32_t V, F&& f) {
  constexpr int VEC = 16 / ES;
  const uintptr_t gs = reinterpret_cast<uintptr_t>(row);
  const uintptr_t as = gs & ~static_cast<uintptr_t>(15);
  const int32_t hoff = static_cast<int32_t>((gs - as) / ES);
  const int32_t nvec = (hoff + V + VEC - 1) / VEC;
  const unsigned char* base = reinterpret_cast<const unsigned char*>(as);
  for (int32_t k = threadIdx.x; k < nvec; k += kGThreads) {
    float x[VEC];
    load_vec_raw<ES>(base, k, x);  // 16 bytes of the cover (inside the allocation's 16-byte blocks)
#pragma unroll
    for (int l = 0; l < VEC; ++l) {
      const int32_t id = k * VEC - hoff + l;
      if (id >= 0 && id < V) f(id, x[l]);
    }
  }
}

// The c-th smallest id (c >= 1) among the elements with key == t: warps
// count the ties of contiguous ranges of the row, the warp whose range holds
// the c-th walks it 32 vectors a step.
template <int ES>
__device__ __forceinline__ int32_t g_tie_id(const unsigned char* row, int32_t V, uint32_t t,
                                            unsigned long long c, unsigned long long* red,
                                            int32_t* shared_id) {
  constexpr int VEC = 16 / ES;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const uintptr_t gs = reinterpret_cast<uintptr_t>(row);
  const uintptr_t as = gs & ~static_cast<uintptr_t>(15);
  const int32_t hoff = static_cast<int32_t>((gs - as) / ES);
  const int32_t nvec = (hoff + V + VEC - 1) / VEC;
  const unsigned char* base = reinterpret_cast<const unsigned char*>(as);
  const int32_t per = (nvec + kGWarps - 1) / kGWarps;  // vectors per warp range
  const int32_t k0 = min(nvec, warp * per), k1 = min(nvec, k0 + per);
  auto ties = [&](int32_t k) {  // ties in vector k, and their ids in order
    float x[VEC];
    load_vec_raw<ES>(base, k, x);
    unsigned m = 0;
#pragma unroll
    for (int l = 0; l < VEC; ++l) {
      const int32_t id = k * VEC - hoff + l;
      if (id >= 0 && id < V && gkey<ES>(x[l]) == t) m |= 1u << l;
    }
    return m;
  };
  unsigned long long n = 0;
  for (int32_t k = k0 + lane; k < k1; k += 32) n += __popc(ties(k));
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) n += __shfl_xor_sync(0xffffffffu, n, off);
  if (lane == 0) red[warp] = n;
  if (threadIdx.x == 0) *shared_id = -1;
  __syncthreads();
  unsigned long long before = 0;
  int owner = -1;
  for (int w = 0; w < kGWarps; ++w) {
    if (owner < 0 && before + red[w] >= c) owner = w;
    if (owner < 0) before += red[w];
  }
  __syncthreads();
  if (warp == owner) {
    unsigned long long left = c - before;  // >= 1
    for (int32_t kb = k0; kb < k1; kb += 32) {
      const int32_t k = kb + lane;
      const unsigned m = k < k1 ? ties(k) : 0u;
      unsigned cnt = __popc(m), incl = cnt;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const unsigned y = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += y;
      }
      const unsigned hit = __ballot_sync(0xffffffffu, incl >= left && incl - cnt < left);
      if (hit) {
        if (lane == __ffs(hit) - 1) {
          unsigned r = static_cast<unsigned>(left - (incl - cnt));  // r-th tie of this vector
          unsigned mm = m;
          for (unsigned i = 1; i < r; ++i) mm &= mm - 1;
          *shared_id = k * VEC - hoff + (__ffs(mm) - 1);
        }
        break;
      }
      left -= __shfl_sync(0xffffffffu, incl, 31);
    }
  }
  __syncthreads();
  const int32_t id = *shared_id;
  __syncthreads();
  return id;
}

constexpr int kHCopies = 8;  // histogram copies (two warps share one)

// Shared histograms of one radix level: per copy 256 bins of a count and a
// fixed-point mass.
struct GHist {
  uint32_t cnt[kHCopies][256];
  unsigned long long mass[kHCopies][256];
};

// The value key t of the first element, in (value desc, id asc) order, at
// which the cumulative count (by_mass false) or fixed-point mass reaches
// `target` (>= 1, at most the row's total), with the count and mass of the
// keys above t and the count and total weight of the keys equal to t (the
// top-p search; top-k counts by bisection, which needs no weights).  One
// pass per 8-bit digit of the key (two for bf16, four for fp32): a histogram
// of the elements that match the digits chosen so far, then the bin where
// the target falls.
struct GSel {
  uint32_t t;
  unsigned long long n_above, m_above, ties, m_ties;
};

template <int ES>
__device__ __forceinline__ GSel g_radix_select(const unsigned char* row, int32_t V, float sc, float h,
                                               unsigned long long target, bool by_mass,
                                               GHist* hist, unsigned long long* red) {
  constexpr int W = ES == 2 ? 16 : 32;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int copy = warp % kHCopies;
  uint32_t prefix = 0;
  unsigned long long n_above = 0, m_above = 0;
  GSel res{};
  for (int shift = W - 8; shift >= 0; shift -= 8) {
    for (int i = tid; i < kHCopies * 256; i += kGThreads) {
      (&hist->cnt[0][0])[i] = 0;
      (&hist->mass[0][0])[i] = 0;
    }
    __syncthreads();
    const bool top = shift + 8 >= W;
    g_for_row<ES>(row, V, [&](int32_t, float x) {
      const uint32_t k = gkey<ES>(x);
      if (top || (k >> (shift + 8)) == prefix) {
        const uint32_t d = (k >> shift) & 255u;
        atomicAdd(&hist->cnt[copy][d], 1u);
        atomicAdd(&hist->mass[copy][d], gweight(x, sc, h));
      }
    });
    __syncthreads();
    if (warp == 0) {  // lane l holds bins 255 - 8 l .. 248 - 8 l, highest first
      auto bin_n = [&](int b) {
        unsigned long long n = 0;
#pragma unroll
        for (int c = 0; c < kHCopies; ++c) n += hist->cnt[c][b];
        return n;
      };
      auto bin_m = [&](int b) {
        unsigned long long m = 0;
#pragma unroll
        for (int c = 0; c < kHCopies; ++c) m += hist->mass[c][b];
        return m;
      };
      unsigned long long ln = 0, lm = 0;
      for (int j = 0; j < 8; ++j) {
        ln += bin_n(255 - 8 * lane - j);
        lm += bin_m(255 - 8 * lane - j);
      }
      unsigned long long in = ln, im = lm;  // inclusive scans over lanes
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const unsigned long long yn = __shfl_up_sync(0xffffffffu, in, off);
        const unsigned long long ym = __shfl_up_sync(0xffffffffu, im, off);
        if (lane >= off) {
          in += yn;
          im += ym;
        }
      }
      const unsigned long long need = target - (by_mass ? m_above : n_above);
      const bool reach = (by_mass ? im : in) >= need;
      const unsigned rl = __ballot_sync(0xffffffffu, reach);
      const int L = rl ? __ffs(rl) - 1 : 31;  // the target is within the row's total
      if (lane == L) {
        unsigned long long an = in - ln, am = im - lm;  // bins of earlier lanes
        int bin = 255 - 8 * lane - 7;
        unsigned long long tn = 0, tm = 0;
        for (int j = 0; j < 8; ++j) {
          const int b = 255 - 8 * lane - j;
          tn = bin_n(b);
          tm = bin_m(b);
          bin = b;
          if ((by_mass ? am + tm : an + tn) >= need) break;
          an += tn;
          am += tm;
        }
        red[0] = static_cast<unsigned long long>(bin);
        red[1] = an;
        red[2] = am;
        red[3] = tn;
        red[4] = tm;
      }
    }
    __syncthreads();
    prefix = (prefix << 8) | static_cast<uint32_t>(red[0]);
    n_above += red[1];
    m_above += red[2];
    res.ties = red[3];
    res.m_ties = red[4];
    __syncthreads();
  }
  res.t = prefix;
  res.n_above = n_above;
  res.m_above = m_above;
  return res;
}

// Kept set and statistics of one row (all threads of the CTA).
template <int ES>
__device__ __forceinline__ GRow g_select_row(const Params& P, const unsigned char* row,
                                             unsigned long long* red, int32_t* sid, GHist* hist) {
  const int32_t V = P.V;
  const float sc = P.sc;
  GRow g{};
  // ---- maximum, its lowest id, non-finite inputs
  float mx = -INFINITY;
  int32_t arg = 0x7fffffff;
  bool bad = false;
  g_for_row<ES>(row, V, [&](int32_t id, float x) {
    if (x != x || x == INFINITY) bad = true;
    if (x > mx) { mx = x; arg = id; }
  });
  const float xmax = warp_max_f32(mx);
  float* fred = reinterpret_cast<float*>(red);
  if ((threadIdx.x & 31) == 0) fred[threadIdx.x >> 5] = xmax;
  __syncthreads();
  float gmx = -INFINITY;
  for (int w = 0; w < kGWarps; ++w) gmx = fmaxf(gmx, fred[w]);
  __syncthreads();
  const int32_t a_w = __reduce_min_sync(0xffffffffu, mx == gmx ? arg : 0x7fffffff);
  int* ired = reinterpret_cast<int*>(red);
  if ((threadIdx.x & 31) == 0) ired[threadIdx.x >> 5] = a_w;
  __syncthreads();
  int32_t gar = 0x7fffffff;
  for (int w = 0; w < kGWarps; ++w) gar = min(gar, ired[w]);
  __syncthreads();
  const bool any_bad = __syncthreads_or(bad ? 1 : 0) != 0;
  g.xmax = gmx;
  g.argmax = gar;
  g.h = gmx * sc;
  g.flags = (any_bad || !(gmx > -INFINITY)) ? SV_DEVERR_NAN : 0;
  if (g.flags) {  // no distribution: keep the argmax alone
    g.thr_key = 0xffffffffu;
    g.z = 1.f;
    g.n_kept = 1;
    return g;
  }
  const float h = g.h;
  const bool use_k = P.top_k > 0 && P.top_k < V;
  const bool use_p = P.top_p < 1.f;
  unsigned long long zk = 0;
  // ---- top-k: the k-th largest value key by bisection (counting passes, no
  //      weights), then the kept mass and the place in the tie class
  if (use_k) {
    constexpr int W = ES == 2 ? 16 : 32;
    const unsigned long long k = static_cast<unsigned long long>(P.top_k);
    uint32_t tk = 0;
    for (int bit = W - 1; bit >= 0; --bit) {
      const uint32_t cand = tk | (1u << bit);
      unsigned long long n = 0;
      g_for_row<ES>(row, V, [&](int32_t, float x) { n += gkey<ES>(x) >= cand; });
      if (g_sum_u64(n, red) >= k) tk = cand;
    }
    unsigned long long n = 0, m = 0, wt = 0;
    g_for_row<ES>(row, V, [&](int32_t, float x) {
      const uint32_t kx = gkey<ES>(x);
      if (kx > tk) {
        ++n;
        m += gweight(x, P.sc, h);
      } else if (kx == tk) {
        wt = gweight(x, P.sc, h);  // every tie weighs the same
      }
    });
    n = g_sum_u64(n, red);
    m = g_sum_u64(m, red);
    wt = g_max_u64(wt, red);
    const unsigned long long ck = k - n;  // 1 <= ck <= ties
    zk = m + ck * wt;
    g.thr_key = tk;
    g.thr_id = g_tie_id<ES>(row, V, tk, ck, red, sid);
    g.n_kept = static_cast<int32_t>(n + ck);
  } else {  // every token
    unsigned long long m = 0;
    g_for_row<ES>(row, V, [&](int32_t, float x) { m += gweight(x, P.sc, h); });
    zk = g_sum_u64(m, red);
  }
  // ---- top-p: the shortest prefix of the order whose mass reaches top_p *
  //      zk (integers: the first prefix with mass >= ceil(top_p * zk)); the
  //      top-k set is itself a prefix of the order holding zk >= that, so the
  //      search runs over the whole row and stops inside it
  if (use_p) {
    const unsigned long long target = max(1ull, static_cast<unsigned long long>(
        ceil(static_cast<double>(P.top_p) * static_cast<double>(zk))));
    const GSel sp = g_radix_select<ES>(row, V, P.sc, h, target, true, hist, red);
    const unsigned long long wt = sp.ties ? sp.m_ties / sp.ties : 0;
    unsigned long long cp = wt > 0 ? (target - sp.m_above + wt - 1) / wt : sp.ties;
    cp = max(1ull, min(cp, sp.ties));
    g.thr_key = sp.t;
    g.thr_id = g_tie_id<ES>(row, V, sp.t, cp, red, sid);
    g.n_kept = static_cast<int32_t>(sp.n_above + cp);
    zk = sp.m_above + cp * wt;
  }
  g.z = static_cast<float>(static_cast<double>(zk) / static_cast<double>(kGFix));
  return g;
}

// Weight of token id under a row's kept set, in units of 1 / z.
template <int ES>
__device__ __forceinline__ float g_p(const GRow& g, float x, int32_t id, float sc) {
  return gkept(g, gkey<ES>(x), id) ? ex2(fmaf(x, sc, -g.h)) / g.z : 0.f;
}

template <int ES>
__global__ void __launch_bounds__(kGThreads, 2) gfilter_rows_kernel(const Params P) {
  __shared__ unsigned long long red[kGWarps];
  __shared__ int32_t sid;
  __shared__ GHist hist;
  grid_dep_launch_dependents();
  auto slot = [&](int32_t i) {  // row i's record, at FiltRow stride
    return reinterpret_cast<GRow*>(reinterpret_cast<FiltRow*>(P.filt) + i);
  };
  const int32_t* offs = P.offs;
  for (int32_t g = blockIdx.x; g < P.Nt; g += gridDim.x) {
    // request of target row g (largest r with offs[r] <= g)
    int32_t lo = 0, hi = P.B - 1;
    while (lo < hi) {
      const int32_t mid = (lo + hi + 1) >> 1;
      if (__ldg(offs + mid) <= g) lo = mid; else hi = mid - 1;
    }
    const int32_t r = lo, off = __ldg(offs + r), off1 = __ldg(offs + r + 1);
    const int32_t gd = g - r;
    const bool pair = off <= g && g < off1 - 1 && gd >= 0 && gd < P.Nd;
    const unsigned char* trow = P.tgt + static_cast<size_t>(g) * P.V * ES;
    const GRow gt = g_select_row<ES>(P, trow, red, &sid, &hist);
    GRow gdr{};
    int fl = gt.flags;
    int acc = 0;
    if (pair) {
      const unsigned char* drow = P.drf + static_cast<size_t>(gd) * P.V * ES;
      gdr = g_select_row<ES>(P, drow, red, &sid, &hist);
      fl |= gdr.flags;
      // label: sum over both kept sets of min(p_t, p_d), element by element
      float part = 0.f;
      if (P.out_conf != nullptr && !fl) {
        for (int32_t v = threadIdx.x; v < P.V; v += kGThreads) {
          const float t = load_elem<ES>(trow, v), d = load_elem<ES>(drow, v);
          part += fminf(g_p<ES>(gt, t, v, P.sc), g_p<ES>(gdr, d, v, P.sc));
        }
      }
      const float label = g_sum_f32(part, reinterpret_cast<float*>(red));
      const int32_t x = __ldg(P.draft_tokens + gd);
      if (x < 0 || x >= P.V) {
        fl |= SV_DEVERR_TOKEN;
      } else if (!fl) {
        if (P.mode == SV_GREEDY) {
          acc = x == gt.argmax;
        } else {
          const float pt = g_p<ES>(gt, load_elem<ES>(trow, x), x, P.sc);
          const float pd = g_p<ES>(gdr, load_elem<ES>(drow, x), x, P.sc);
          acc = __ldg(P.uniforms + g) * pd < pt;
        }
      }
      if (threadIdx.x == 0 && P.out_conf != nullptr) P.out_conf[gd] = label;
    }
    if (threadIdx.x == 0) {
      *slot(g) = gt;
      if (pair) *slot(P.Nt + gd) = gdr;
      RowRec rr{};
      rr.mt = gt.h; rr.zt = gt.z; rr.md = gdr.h; rr.zd = gdr.z;
      rr.argt = gt.argmax; rr.acc = acc; rr.pick = -1; rr.flags = fl;
      P.rec[g] = rr;
      if (P.out_row_stats != nullptr) {
        float* o = P.out_row_stats + 3 * static_cast<size_t>(g);
        o[0] = gt.xmax / P.T; o[1] = gt.z; o[2] = __int_as_float(gt.argmax);
        if (pair) {
          float* o2 = P.out_row_stats + 3 * (static_cast<size_t>(P.Nt) + gd);
          o2[0] = gdr.xmax / P.T; o2[1] = gdr.z; o2[2] = __int_as_float(gdr.argmax);
        }
      }
      if (fl) raise_error(P, fl);
    }
    __syncthreads();
  }
}

// One request per CTA: first rejection, outputs, final token.
template <int ES>
__global__ void __launch_bounds__(kGThreads) gfilter_requests_kernel(const Params P) {
  __shared__ float fred[2 * kGWarps];
  __shared__ int ired[kGWarps];
  const int32_t r = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31;
  const int32_t off = __ldg(P.offs + r), off1 = __ldg(P.offs + r + 1), ell = __ldg(P.lens + r);
  const bool ok = ell >= 1 && ell <= P.max_len && off1 - off == ell && off >= r &&
                  off1 <= P.Nt && (r != 0 || off == 0) && (r != P.B - 1 || off1 == P.Nt) &&
                  off - r + ell - 1 <= P.Nd;
  if (!ok) {
    if (tid == 0) raise_error(P, SV_DEVERR_LEN);
    return;
  }
  const float u = __ldg(P.uniforms + off + ell - 1);
  grid_dep_wait();  // row records from gfilter_rows_kernel
  int32_t first = ell - 1;
  for (int32_t j = tid; j < ell - 1; j += kGThreads)
    if (!P.rec[off + j].acc && j < first) first = j;
  const int32_t a = block_min_int<kGWarps>(first, ired);
  for (int32_t j = tid; j < ell; j += kGThreads) {
    if (j < a) P.out_tokens[off + j] = __ldg(P.draft_tokens + off - r + j);
    else if (j > a) P.out_tokens[off + j] = -1;
  }
  if (tid == 0) P.out_accept_len[r] = a;
  const int32_t trow_i = off + a;
  const RowRec rr = P.rec[trow_i];
  if (P.mode == SV_GREEDY || rr.flags) {  // greedy, or no distribution
    if (tid == 0) P.out_tokens[trow_i] = rr.argt;
    return;
  }
  const FiltRow* slots = reinterpret_cast<const FiltRow*>(P.filt);
  const GRow gt = *reinterpret_cast<const GRow*>(slots + trow_i);
  bool residual = a < ell - 1;
  GRow gd{};
  if (residual) gd = *reinterpret_cast<const GRow*>(slots + P.Nt + off - r + a);
  const unsigned char* trow = P.tgt + static_cast<size_t>(trow_i) * P.V * ES;
  const unsigned char* drow = P.drf + static_cast<size_t>(off - r + a) * P.V * ES;
  const int32_t E = (P.V + kGThreads - 1) / kGThreads;  // ids per thread
  const int32_t i0 = min(P.V, tid * E), i1 = min(P.V, i0 + E);
  auto weight = [&](int32_t v, bool res) {
    const float pt = g_p<ES>(gt, load_elem<ES>(trow, v), v, P.sc);
    return res ? fmaxf(0.f, pt - g_p<ES>(gd, load_elem<ES>(drow, v), v, P.sc)) : pt;
  };
  for (int round = 0; round < 2; ++round) {
    float wsum = 0.f;
    for (int32_t v = i0; v < i1; ++v) wsum += weight(v, residual);
    float lo, hi, tot;
    block_scan_bounds<kGWarps>(wsum, fred, lo, hi, tot);
    if (residual && !(tot > kZeroResidual)) {  // no residual mass (rounding only): p_t
      residual = false;
      continue;
    }
    if (!(tot > 0.f)) {  // nothing to draw from
      if (tid == 0) {
        raise_error(P, SV_DEVERR_NAN);
        P.out_tokens[trow_i] = rr.argt;
      }
      return;
    }
    const float need = u * tot;
    const bool own = lo < hi && ((lo <= need && need < hi) || (need >= tot && hi == tot));
    const unsigned ob = __ballot_sync(0xffffffffu, own);
    if (ob) {  // the owner's warp walks the owner's run, 32 ids a step
      const int ol = __ffs(ob) - 1;
      const int32_t oi0 = __shfl_sync(0xffffffffu, i0, ol), oi1 = __shfl_sync(0xffffffffu, i1, ol);
      const float left = __shfl_sync(0xffffffffu, need - lo, ol);
      float base = 0.f;
      int32_t p = -1, last = -1;
      for (int32_t b0 = oi0; b0 < oi1 && p < 0; b0 += 32) {
        const int32_t v = b0 + lane;
        const float wv = v < oi1 ? weight(v, residual) : 0.f;
        const float run = base + warp_incl_scan(wv);
        const unsigned hitm = __ballot_sync(0xffffffffu, wv > 0.f && run > left);
        const unsigned posm = __ballot_sync(0xffffffffu, wv > 0.f);
        if (posm) last = b0 + 31 - __clz(posm);
        if (hitm) p = b0 + __ffs(hitm) - 1;
        base = __shfl_sync(0xffffffffu, run, 31);
      }
      if (p < 0) p = last;
      if (lane == 0) P.out_tokens[trow_i] = p;
    }
    return;
  }
}

}  // namespace sv
