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
// Both thresholds come from one search scheme along that order, exact and
// independent of the visiting order.  Weights w = exp2(x sc - h) (h = x_max
// sc) are fixed-point integers of 2^-40.  Level 1 is one pass: per weight
// bin (eighths of a binade of w; each bin a run of the order, and a row's
// tokens spread thinly over them) a count and a mass scaled down to 32 bits,
// which bound the bin's exact mass; the row's exact total comes from the
// threads' own sums.  The bin where the cumulative count reaches k, or the
// run of bins where the bounded cumulative mass reaches ceil(top_p * kept
// mass), is then searched by key digits over that run's tokens only (one
// pass for a bf16 run of at most 256 keys, else one per 8-bit digit), with
// warp-aggregated updates of per-warp histograms; the first of those passes
// also sums the exact mass before the run.  Inside the tie class of the
// final value every token weighs the same, so the cut falls after c of them,
// c from integer arithmetic; a counting pass finds the id of the c-th.
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
// 16-byte vectors in flight per thread in a row pass: 64 bytes, 16 logits
template <int ES>
__host__ __device__ constexpr int g_unroll() { return ES == 2 ? 2 : 4; }
constexpr int kGBins = 512;    // level-1 bins: eighths of a binade of the weight
constexpr int kL1Copies = 4;   // level-1 histogram copies
constexpr int kGMaxV = 1 << 21;  // largest V the 32-bit level-1 masses take (gshift)

// A row's kept set and statistics (stored in the row's FiltRow slot of the
// workspace).
struct GRow {
  float h;           // reference x_max * sc
  float z;           // kept mass: sum over the kept set of exp2(x sc - h)
  float xmax;        // row maximum (raw logit)
  int32_t argmax;    // lowest id holding it
  uint32_t thr_key;  // kept: key > thr_key, or key == thr_key and id <= thr_id
  int32_t thr_id;
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

// v * 2^40 rounded to the nearest integer (ties to even), v in [0, 2) and
// finite, in 32-bit integer and float-add operations: at 2^23 and above the
// product is already an integer, its 24-bit significand shifted left by the
// exponent less 23; below, F + 2^23 lands on the grid of 1, which rounds F.
// (A 64-bit conversion would run on the double-precision pipe.)
__device__ __forceinline__ unsigned long long gfix(float v) {
  const float F = v * kGFix;
  const uint32_t b = __float_as_uint(F);
  const unsigned long long big = static_cast<unsigned long long>((b & 0x7fffffu) | 0x800000u)
                                 << max(0, static_cast<int>(b >> 23) - 150);
  const uint32_t small = __float_as_uint(__fadd_rn(F, 8388608.f)) - 0x4b000000u;
  return F < 8388608.f ? static_cast<unsigned long long>(small) : big;
}

// Fixed-point weight of a logit from its log2 weight y = x sc - h (exact
// integer units of 2^-40).
__device__ __forceinline__ unsigned long long gweight_y(float y) { return gfix(ex2(y)); }

// Fixed-point weight of logit x.
__device__ __forceinline__ unsigned long long gweight(float x, float sc, float h) {
  return gweight_y(fmaf(x, sc, -h));
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

__device__ __forceinline__ float g_sum_f32(float v, float* red) {
  v = warp_sum_f32(v);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  __syncthreads();
  float t = 0.f;
  for (int w = 0; w < kGWarps; ++w) t += red[w];
  __syncthreads();
  return t;
}

// The 16-byte aligned cover of a row: its first vector, the elements of the
// cover before the row, and the number of vectors.
struct GCover {
  const unsigned char* base;
  int32_t hoff;
  int32_t nvec;
};

template <int ES>
__device__ __forceinline__ GCover g_cover(const unsigned char* row, int32_t V) {
  constexpr int VEC = 16 / ES;
  const uintptr_t gs = reinterpret_cast<uintptr_t>(row);
  const uintptr_t as = gs & ~static_cast<uintptr_t>(15);
  GCover c;
  c.base = reinterpret_cast<const unsigned char*>(as);
  c.hoff = static_cast<int32_t>((gs - as) / ES);
  c.nvec = (c.hoff + V + VEC - 1) / VEC;
  return c;
}

// 16 bytes of a cover (inside the allocation's 16-byte blocks), read-only path.
__device__ __forceinline__ uint4 g_ld16(const unsigned char* base, int32_t k) {
  return __ldg(reinterpret_cast<const uint4*>(base) + k);
}

template <int ES>
__device__ __forceinline__ void g_unpack(const uint4& w, float* x) {
  if (ES == 2) {
    x[0] = bf16lo(w.x); x[1] = bf16hi(w.x); x[2] = bf16lo(w.y); x[3] = bf16hi(w.y);
    x[4] = bf16lo(w.z); x[5] = bf16hi(w.z); x[6] = bf16lo(w.w); x[7] = bf16hi(w.w);
  } else {
    x[0] = __uint_as_float(w.x); x[1] = __uint_as_float(w.y);
    x[2] = __uint_as_float(w.z); x[3] = __uint_as_float(w.w);
  }
}

// Visit every element of a row of V logits.  Warp w takes the vectors
// 32 w + lane + 512 i of the row's cover, kGUnroll of them loaded before the
// first is used; f(id, x, ok) is called by the 32 lanes of a warp together,
// ok false for cover elements outside the row.  A thread meets its ids in
// ascending order.
template <int ES, typename F>
__device__ __forceinline__ void g_for_row(const unsigned char* row, int32_t V, F&& f) {
  constexpr int VEC = 16 / ES;
  constexpr int kGUnroll = g_unroll<ES>();
  const GCover c = g_cover<ES>(row, V);
  const int lane = threadIdx.x & 31;
  const int32_t kf0 = c.hoff > 0 ? 1 : 0, kf1 = (c.hoff + V) / VEC;  // vectors inside the row
  for (int32_t k0 = threadIdx.x - lane; k0 < c.nvec; k0 += kGUnroll * kGThreads) {
    uint4 w[kGUnroll];
#pragma unroll
    for (int u = 0; u < kGUnroll; ++u) {
      const int32_t k = k0 + u * kGThreads + lane;
      w[u] = k < c.nvec ? g_ld16(c.base, k) : make_uint4(0u, 0u, 0u, 0u);
    }
    if (k0 >= kf0 && k0 + (kGUnroll - 1) * kGThreads + 31 < kf1) {  // the warp's vectors are all inside
#pragma unroll
      for (int u = 0; u < kGUnroll; ++u) {
        const int32_t k = k0 + u * kGThreads + lane;
        float x[VEC];
        g_unpack<ES>(w[u], x);
#pragma unroll
        for (int l = 0; l < VEC; ++l) f(k * VEC - c.hoff + l, x[l], true);
      }
    } else {
#pragma unroll
      for (int u = 0; u < kGUnroll; ++u) {
        const int32_t k = k0 + u * kGThreads + lane;
        float x[VEC];
        g_unpack<ES>(w[u], x);
#pragma unroll
        for (int l = 0; l < VEC; ++l) {
          const int32_t id = k * VEC - c.hoff + l;
          f(id, x[l], k < c.nvec && id >= 0 && id < V);
        }
      }
    }
  }
}

// Visit every id of two rows of V logits together: f(id, a_id, b_id).  Rows
// with the same 16-byte phase go by vectors, two of each row in flight per
// thread; others element by element.
template <int ES, typename F>
__device__ __forceinline__ void g_for_pair(const unsigned char* a, const unsigned char* b,
                                           int32_t V, F&& f) {
  constexpr int VEC = 16 / ES;
  const GCover ca = g_cover<ES>(a, V), cb = g_cover<ES>(b, V);
  if (ca.hoff != cb.hoff) {
    for (int32_t v = threadIdx.x; v < V; v += kGThreads) f(v, load_elem<ES>(a, v), load_elem<ES>(b, v));
    return;
  }
  for (int32_t k0 = threadIdx.x; k0 < ca.nvec; k0 += 2 * kGThreads) {
    uint4 wa[2], wb[2];
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const int32_t k = k0 + u * kGThreads;
      if (k < ca.nvec) {
        wa[u] = g_ld16(ca.base, k);
        wb[u] = g_ld16(cb.base, k);
      }
    }
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const int32_t k = k0 + u * kGThreads;
      if (k < ca.nvec) {
        float xa[VEC], xb[VEC];
        g_unpack<ES>(wa[u], xa);
        g_unpack<ES>(wb[u], xb);
#pragma unroll
        for (int l = 0; l < VEC; ++l) {
          const int32_t id = k * VEC - ca.hoff + l;
          if (id >= 0 && id < V) f(id, xa[l], xb[l]);
        }
      }
    }
  }
}

// The logit whose value key is t (gkey inverted).
template <int ES>
__device__ __forceinline__ float gkey_value(uint32_t t) {
  const uint32_t k = ES == 2 ? t << 16 : t;
  const uint32_t u = (k & 0x80000000u) ? (k & 0x7fffffffu) : ~k;
  return __uint_as_float(ES == 2 ? (u & 0xffff0000u) : u);
}

// Level-1 bin of a logit from its log2 weight y = x sc - h (about 0 at the
// row maximum, below it elsewhere): floor(-8 y) clamped to [0, kGBins - 1],
// eighths of a binade of the weight.  It never falls along the (value desc,
// id asc) order, so each bin holds a run of that order (equal values share
// a bin); weights in the last bin are below 2^-63, 0 in fixed point.
__device__ __forceinline__ int gbin(float y) {
  const float t = fminf(fmaxf(-8.f * y, 0.f), static_cast<float>(kGBins - 1));
  return static_cast<int>(__float_as_uint(__fadd_rz(t, 8388608.f)) - 0x4b000000u);  // floor(t)
}

// Level-1 masses are kept in 32 bits, in units of 2^gshift(b) for bin b: a
// weight of bin b is below 2^(41 - floor(b / 8)), so w >> gshift(b) < 2^13
// and a copy's sum over at most V / kL1Copies tokens stays below 2^32 for
// V up to 2^21.  With the bin's count this bounds its exact mass:
// sum(w >> s) << s <= mass < (sum(w >> s) + count) << s.
__device__ __forceinline__ int gshift(int b) { return max(0, 28 - (b >> 3)); }

// The c-th smallest id (c >= 1) among the elements with key == t (all
// threads of the CTA; tb: 16 x 256 words of shared scratch).  Warps count
// the ties of each block of their contiguous ranges of the row (kGUnroll
// vectors a lane in flight); warp 0 finds the block holding the c-th along
// the id order, and the warp owning it walks just that block.
template <int ES>
__device__ __forceinline__ int32_t g_tie_id(const unsigned char* row, int32_t V, uint32_t t,
                                         unsigned long long c, unsigned long long* red,
                                         int32_t* shared_id, uint32_t (*tb)[256]) {
  constexpr int VEC = 16 / ES;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  constexpr int kGUnroll = g_unroll<ES>();
  constexpr int kStep = 32 * kGUnroll;  // vectors a warp reads per round
  const GCover cv = g_cover<ES>(row, V);
  const int32_t per = (cv.nvec + kGWarps - 1) / kGWarps;  // vectors per warp range
  const int32_t k0 = min(cv.nvec, warp * per), k1 = min(cv.nvec, k0 + per);
  // blocks of bstep vectors (a multiple of kStep), at most 256 a warp
  const int32_t bstep = kStep * ((per + kStep * 256 - 1) / (kStep * 256));
  auto scan = [&](const uint4& w, int32_t k) {  // tie mask of vector k
    float x[VEC];
    g_unpack<ES>(w, x);
    unsigned m = 0;
#pragma unroll
    for (int l = 0; l < VEC; ++l) {
      const int32_t id = k * VEC - cv.hoff + l;
      if (id >= 0 && id < V && gkey<ES>(x[l]) == t) m |= 1u << l;
    }
    return m;
  };
  // ---- every warp: the ties in each block of its range
  for (int i = lane; i < 256; i += 32) tb[warp][i] = 0u;
  __syncwarp();
  for (int32_t kb = k0; kb < k1; kb += kStep) {
    uint4 w[kGUnroll];
#pragma unroll
    for (int u = 0; u < kGUnroll; ++u) {
      const int32_t k = kb + 32 * u + lane;
      w[u] = k < k1 ? g_ld16(cv.base, k) : make_uint4(0u, 0u, 0u, 0u);
    }
    unsigned n = 0;
#pragma unroll
    for (int u = 0; u < kGUnroll; ++u) {
      const int32_t k = kb + 32 * u + lane;
      if (k < k1) n += __popc(scan(w[u], k));
    }
    n = __reduce_add_sync(0xffffffffu, n);
    if (lane == 0) tb[warp][(kb - k0) / bstep] += n;
  }
  if (threadIdx.x == 0) *shared_id = -1;
  __syncthreads();
  // ---- warp 0: the block holding the c-th tie along the id order (warp
  //      ranges in order, blocks in order inside each); lane l sums entries
  //      128 l .. 128 l + 127 of the flattened [warp][block] table
  if (warp == 0) {
    const uint32_t* flat = &tb[0][0];
    unsigned long long ls = 0;
    for (int i = 0; i < 128; ++i) ls += flat[128 * lane + i];
    unsigned long long incl = ls;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const unsigned long long y = __shfl_up_sync(0xffffffffu, incl, off);
      if (lane >= off) incl += y;
    }
    const unsigned hit = __ballot_sync(0xffffffffu, incl >= c && incl - ls < c);
    if (hit && lane == __ffs(hit) - 1) {
      unsigned long long before = incl - ls;
      int e = 128 * lane;
      while (before + flat[e] < c) before += flat[e++];
      red[0] = static_cast<unsigned long long>(e);
      red[1] = c - before;  // the tie's rank inside that block, >= 1
    }
    if (!hit && lane == 0) {  // fewer than c ties (no such row): no id
      red[0] = ~0ull;
      red[1] = 0ull;
    }
  }
  __syncthreads();
  const unsigned long long eb = red[0];
  unsigned long long left = red[1];
  __syncthreads();
  if (eb != ~0ull && warp == static_cast<int>(eb >> 8)) {
    // ---- the owner warp walks that one block
    const int32_t bk0 = k0 + static_cast<int32_t>(eb & 255u) * bstep;
    const int32_t bk1 = min(k1, bk0 + bstep);
    bool found = false;
    for (int32_t kb = bk0; kb < bk1 && !found; kb += kStep) {
      uint4 w[kGUnroll];
#pragma unroll
      for (int u = 0; u < kGUnroll; ++u) {
        const int32_t k = kb + 32 * u + lane;
        w[u] = k < bk1 ? g_ld16(cv.base, k) : make_uint4(0u, 0u, 0u, 0u);
      }
#pragma unroll
      for (int u = 0; u < kGUnroll; ++u) {
        if (found) break;
        const int32_t k = kb + 32 * u + lane;
        const unsigned m = k < bk1 ? scan(w[u], k) : 0u;
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
            *shared_id = k * VEC - cv.hoff + (__ffs(mm) - 1);
          }
          found = true;
        } else {
          left -= __shfl_sync(0xffffffffu, incl, 31);
        }
      }
    }
  }
  __syncthreads();
  const int32_t id = *shared_id;
  __syncthreads();
  return id;
}

// Shared histograms (dynamic shared memory): level 1 (kGBins weight bins,
// counts and scaled masses in 32 bits; kGWarps / kL1Copies warps share a
// copy) and the key-digit levels (256 bins, counts and exact fixed-point
// masses, one private copy per warp).
struct GHist {
  uint32_t l1n[kL1Copies][kGBins];
  uint32_t l1s[kL1Copies][kGBins];  // sum of w >> gshift(b)
  unsigned long long dm[kGWarps][256];
  uint32_t dn[kGWarps][256];
};

// Warp-aggregated update of the warp's own histogram: every lane with d >= 0
// adds one to count bin d and w to mass bin d; the lanes that share a bin
// add together, through one lane, so no other lane writes that bin meanwhile
// and plain stores suffice.  All 32 lanes of the warp call it.
__device__ __forceinline__ void g_add_agg(uint32_t* n, unsigned long long* m, int d,
                                          unsigned long long w) {
  const int lane = threadIdx.x & 31;
  unsigned todo = __ballot_sync(0xffffffffu, d >= 0);
  while (todo) {
    const int src = __ffs(todo) - 1;
    const int ds = __shfl_sync(0xffffffffu, d, src);
    const bool mine = d == ds;
    const unsigned grp = __ballot_sync(0xffffffffu, mine);
    unsigned long long s = mine ? w : 0ull;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
    if (lane == src) {
      n[ds] += static_cast<uint32_t>(__popc(grp));
      m[ds] += s;
    }
    __syncwarp();
    todo &= ~grp;
  }
}

// Warp 0 only: over NB bins in order (j = 0 first along the value-desc
// order; bin_n / bin_m give a bin's count and mass), the first bin at which
// the cumulative count (by_mass false) or mass reaches need (the last bin if
// none does), with the count and mass of the bins before it and its count;
// every lane of the warp gets the result.
struct GFound {
  int j;
  unsigned long long n_before, m_before, n_bin;
};

template <int NB, typename FN, typename FM>
__device__ __forceinline__ GFound g_find(FN&& bin_n, FM&& bin_m, bool by_mass,
                                         unsigned long long need) {
  constexpr int PER = NB / 32;
  const int lane = threadIdx.x & 31;
  unsigned long long ln = 0, lm = 0;
  for (int i = 0; i < PER; ++i) {  // the lane's bins in rotated order: few bank conflicts
    const int j = lane * PER + ((i + lane) & (PER - 1));
    ln += bin_n(j);
    lm += bin_m(j);
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
  const unsigned rl = __ballot_sync(0xffffffffu, (by_mass ? im : in) >= need);
  const int L = rl ? __ffs(rl) - 1 : 31;
  GFound f{L * PER + PER - 1, 0, 0, 0};
  if (lane == L) {
    unsigned long long an = in - ln, am = im - lm;  // bins of earlier lanes
    for (int i = 0; i < PER; ++i) {
      const int j = L * PER + i;
      const unsigned long long cn = bin_n(j), cm = bin_m(j);
      if ((by_mass ? am + cm : an + cn) >= need || i == PER - 1) {
        f = GFound{j, an, am, cn};
        break;
      }
      an += cn;
      am += cm;
    }
  }
  f.j = __shfl_sync(0xffffffffu, f.j, L);
  f.n_before = __shfl_sync(0xffffffffu, f.n_before, L);
  f.m_before = __shfl_sync(0xffffffffu, f.m_before, L);
  f.n_bin = __shfl_sync(0xffffffffu, f.n_bin, L);
  return f;
}

// Search along the (value desc, id asc) order inside the run of level-1 bins
// [ba, bb]: the value key t of the element at which the cumulative count
// (by_mass false) or mass reaches the target, the count and mass of the
// run's keys above t, the count of keys equal to t, and the exact mass of the
// bins before ba (summed in the first pass).  By count, need is the count
// still needed from the run; by mass, it is the target itself, reached
// inside the run.  One pass per 8-bit digit of the key (two for bf16, four
// for fp32; one for a bf16 run of at most 256 keys), each a histogram of the
// run's elements matching the digits chosen so far.
struct GSel {
  uint32_t t;
  unsigned long long n_above, m_above, ties, m_before;
};

template <int ES>
__device__ __forceinline__ GSel g_digits(const unsigned char* row, int32_t V, float sc, float h,
                                         int ba, int bb, unsigned long long need, bool by_mass,
                                         GHist* hist, unsigned long long* red) {
  constexpr int W = ES == 2 ? 16 : 32;
  constexpr int VEC = 16 / ES, kGUnroll = g_unroll<ES>(), NE = kGUnroll * VEC;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const GCover cv = g_cover<ES>(row, V);
  // bf16: the run's keys fill the interval [klo, khi] (the bin never rises
  // along the key order, from -inf to +inf); found by bisection over the
  // keys, and when it spans at most 256 keys one level with digit key - klo
  // replaces the two byte levels.  Digits are taken of key - base (base klo
  // for the one level, else 0; keys below base wrap and match no prefix).
  uint32_t klo = 0, khi = 0;
  bool single = false;
  if (ES == 2) {
    auto G = [&](uint32_t k) { return gbin(fmaf(gkey_value<ES>(k), sc, -h)); };
    uint32_t lo = 0x007fu, hi = 0xff80u;  // the smallest key with G <= bb
    while (lo < hi) {
      const uint32_t mid = (lo + hi) >> 1;
      if (G(mid) <= bb) hi = mid; else lo = mid + 1;
    }
    klo = lo;
    lo = 0x007fu;
    hi = 0xff80u;  // the largest key with G >= ba
    while (lo < hi) {
      const uint32_t mid = (lo + hi + 1) >> 1;
      if (G(mid) >= ba) lo = mid; else hi = mid - 1;
    }
    single = lo >= klo && lo - klo < 256u;
    khi = lo;
  }
  const uint32_t base = single ? klo : 0u;
  uint32_t prefix = 0;
  GSel res{};
  bool first = true;
  for (int shift = single ? 0 : W - 8; shift >= 0; shift -= 8) {
    for (int i = tid; i < kGWarps * 256; i += kGThreads) {
      (&hist->dn[0][0])[i] = 0;
      (&hist->dm[0][0])[i] = 0;
    }
    __syncthreads();
    // a round: kGUnroll vectors a lane (16 logits); the per-logit tests
    // first, the warp-aggregated updates only when some lane of the warp
    // holds a logit of the run
    unsigned long long mb = 0;  // the thread's share of the mass before the run
    if (ES == 2 && single) {
      // one level over a bf16 run of at most 256 keys [klo, khi]: the bins
      // never rise along the key order, so membership is a key comparison;
      // every element of a key has the same value and weight, so only the
      // count of each digit (key - klo) is kept, and its mass is count x
      // weight below
      g_for_row<ES>(row, V, [&](int32_t, float x, bool ok) {
        if (!ok) return;
        const uint32_t key = gkey<ES>(x);
        if (key > khi) mb += gweight(x, sc, h);
        else if (key >= klo) atomicAdd(&hist->dn[warp][key - klo], 1u);
      });
    } else
    for (int32_t k0 = tid - lane; k0 < cv.nvec; k0 += kGUnroll * kGThreads) {
      uint4 wv[kGUnroll];
#pragma unroll
      for (int u = 0; u < kGUnroll; ++u) {
        const int32_t k = k0 + u * kGThreads + lane;
        wv[u] = k < cv.nvec ? g_ld16(cv.base, k) : make_uint4(0u, 0u, 0u, 0u);
      }
      float x[NE];
#pragma unroll
      for (int u = 0; u < kGUnroll; ++u) g_unpack<ES>(wv[u], x + u * VEC);
      uint32_t inm = 0;
#pragma unroll
      for (int e = 0; e < NE; ++e) {
        const int32_t k = k0 + (e / VEC) * kGThreads + lane;
        const int32_t id = k * VEC - cv.hoff + e % VEC;
        const bool ok = k < cv.nvec && id >= 0 && id < V;
        const float y = fmaf(x[e], sc, -h);
        const int bx = gbin(y);
        if (ok && bx >= ba && bx <= bb && ((gkey<ES>(x[e]) - base) >> shift >> 8) == prefix)
          inm |= 1u << e;
        if (first && ok && bx < ba) mb += gweight_y(y);
      }
      if (__any_sync(0xffffffffu, inm != 0)) {
#pragma unroll
        for (int e = 0; e < NE; ++e) {
          const bool in = (inm >> e) & 1u;
          g_add_agg(hist->dn[warp], hist->dm[warp],
                    in ? static_cast<int>(((gkey<ES>(x[e]) - base) >> shift) & 255u) : -1,
                    in ? gweight_y(fmaf(x[e], sc, -h)) : 0ull);
        }
      }
    }
    __syncthreads();
    if (ES == 2 && single) {  // counts summed; a digit's mass is its count x its key's weight
      if (tid < 256) {
        uint32_t c = 0;
#pragma unroll
        for (int q = 0; q < kGWarps; ++q) c += hist->dn[q][tid];
        hist->dn[0][tid] = c;
        hist->dm[0][tid] = c ? static_cast<unsigned long long>(c) *
                                   gweight(gkey_value<ES>(klo + tid), sc, h)
                             : 0ull;
      }
    } else {  // the warps' histograms summed into warp 0's: counts by threads 0..255,
       // masses by threads 256..511, one bin each
      const int j = tid & 255;
      if (tid < 256) {
        uint32_t c = 0;
#pragma unroll
        for (int q = 0; q < kGWarps; ++q) c += hist->dn[q][j];
        hist->dn[0][j] = c;
      } else {
        unsigned long long m = 0;
#pragma unroll
        for (int q = 0; q < kGWarps; ++q) m += hist->dm[q][j];
        hist->dm[0][j] = m;
      }
    }
    if (first) {
      res.m_before = g_sum_u64(mb, red);  // its barriers also order the sums above
      if (by_mass) need -= res.m_before;  // >= 1: the bins before ba hold less than the target
    } else {
      __syncthreads();
    }
    if (warp == 0) {
      const GFound f = g_find<256>(
          [&](int j) { return static_cast<unsigned long long>(hist->dn[0][255 - j]); },
          [&](int j) { return hist->dm[0][255 - j]; },
          by_mass, need);
      if (lane == 0) {
        red[0] = static_cast<unsigned long long>(f.j);
        red[1] = f.n_before;
        red[2] = f.m_before;
        red[3] = f.n_bin;
      }
    }
    __syncthreads();
    prefix = (prefix << 8) | (255u - static_cast<uint32_t>(red[0]));
    res.n_above += red[1];
    res.m_above += red[2];
    res.ties = red[3];
    need -= by_mass ? red[2] : red[1];
    first = false;
    __syncthreads();
  }
  res.t = base + prefix;
  return res;
}

// Kept set and statistics of one row (all threads of the CTA).
template <int ES>
__device__ __forceinline__ GRow g_select_row(const Params& P, const unsigned char* row,
                                             unsigned long long* red, int32_t* sid, GHist* hist) {
  const int32_t V = P.V;
  const float sc = P.sc;
  const int tid = threadIdx.x, warp = tid >> 5;
  GRow g{};
  // ---- maximum, its lowest id, non-finite inputs
  float mx = -INFINITY;
  int32_t arg = 0x7fffffff;
  bool bad = false;
  g_for_row<ES>(row, V, [&](int32_t id, float x, bool ok) {
    if (!ok) return;
    if (x != x || x == INFINITY) bad = true;
    if (x > mx) { mx = x; arg = id; }
  });
  const float xmax = warp_max_f32(mx);
  float* fred = reinterpret_cast<float*>(red);
  if ((tid & 31) == 0) fred[warp] = xmax;
  __syncthreads();
  float gmx = -INFINITY;
  for (int w = 0; w < kGWarps; ++w) gmx = fmaxf(gmx, fred[w]);
  __syncthreads();
  const int32_t a_w = __reduce_min_sync(0xffffffffu, mx == gmx ? arg : 0x7fffffff);
  int* ired = reinterpret_cast<int*>(red);
  if ((tid & 31) == 0) ired[warp] = a_w;
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
    return g;
  }
  const float h = g.h;
  const bool use_k = P.top_k > 0 && P.top_k < V;
  const bool use_p = P.top_p < 1.f;
  const int lane = tid & 31;
  // ---- level 1, one pass: counts and scaled masses of the weight bins
  //      (32-bit shared atomics), and the row's exact mass from the threads'
  //      own sums
  const int c1 = warp % kL1Copies;
  for (int i = tid; i < kL1Copies * kGBins; i += kGThreads) {
    (&hist->l1n[0][0])[i] = 0;
    (&hist->l1s[0][0])[i] = 0;
  }
  __syncthreads();
  unsigned long long zs = 0;
  g_for_row<ES>(row, V, [&](int32_t, float x, bool ok) {
    if (!ok) return;
    const float y = fmaf(x, sc, -h);
    const int b = gbin(y);
    const unsigned long long w = gweight_y(y);
    zs += w;
    atomicAdd(&hist->l1n[c1][b], 1u);
    const uint32_t ws = static_cast<uint32_t>(w >> gshift(b));
    if (ws) atomicAdd(&hist->l1s[c1][b], ws);
  });
  __syncthreads();
  const unsigned long long zt = g_sum_u64(zs, red);  // the row's total mass
  auto l1n = [&](int j) {
    unsigned long long c = 0;
#pragma unroll
    for (int q = 0; q < kL1Copies; ++q) c += hist->l1n[q][j];
    return c;
  };
  auto l1lo = [&](int j) {  // lower bound of bin j's mass
    unsigned long long m = 0;
#pragma unroll
    for (int q = 0; q < kL1Copies; ++q) m += hist->l1s[q][j];
    return m << gshift(j);
  };
  auto l1hi = [&](int j) { return l1lo(j) + (l1n(j) << gshift(j)); };  // upper bound
  unsigned long long zk = zt;  // mass of the kept set
  if (use_k) {
    // ---- top-k: the bin holding the k-th element by count (exact), then its
    //      key digits; the kept mass from the mass before the bin, the
    //      digits above and the tie weight (every tie weighs the same)
    const unsigned long long k = static_cast<unsigned long long>(P.top_k);
    if (warp == 0) {
      const GFound f = g_find<kGBins>(l1n, l1lo, false, k);
      if (lane == 0) {
        red[0] = static_cast<unsigned long long>(f.j);
        red[1] = f.n_before;
      }
    }
    __syncthreads();
    const int bk = static_cast<int>(red[0]);
    const unsigned long long nb = red[1];
    __syncthreads();
    const GSel s = g_digits<ES>(row, V, sc, h, bk, bk, k - nb, false, hist, red);
    const unsigned long long ck = k - (nb + s.n_above);  // 1 <= ck <= ties
    const unsigned long long wt = gweight(gkey_value<ES>(s.t), sc, h);
    zk = s.m_before + s.m_above + ck * wt;
    g.thr_key = s.t;
    if (!use_p) g.thr_id = g_tie_id<ES>(row, V, s.t, ck, red, sid, hist->dn);
  }
  if (use_p) {
    // ---- top-p: the shortest prefix of the order whose mass reaches top_p *
    //      zk (integers: the first prefix with mass >= ceil(top_p * zk)); the
    //      top-k set is itself a prefix of the order holding zk >= that, so the
    //      search runs over the whole row and stops inside it.  The level-1
    //      bounds place the crossing inside the run of bins [ba, bb]: ba the
    //      first bin whose cumulative upper bound reaches the target, bb the
    //      first whose cumulative lower bound does (one bin but for targets
    //      within about 2^-13 of a bin edge).
    const unsigned long long target = max(1ull, static_cast<unsigned long long>(
        ceil(static_cast<double>(P.top_p) * static_cast<double>(zk))));
    if (warp == 0) {
      auto none = [](int) { return 0ull; };
      const GFound fa = g_find<kGBins>(none, l1hi, true, target);
      const GFound fb = g_find<kGBins>(none, l1lo, true, target);
      if (lane == 0) {
        red[0] = static_cast<unsigned long long>(fa.j);
        red[1] = static_cast<unsigned long long>(max(fa.j, fb.j));
      }
    }
    __syncthreads();
    const int ba = static_cast<int>(red[0]), bb = static_cast<int>(red[1]);
    __syncthreads();
    const GSel s = g_digits<ES>(row, V, sc, h, ba, bb, target, true, hist, red);
    const unsigned long long m_above = s.m_before + s.m_above;
    const unsigned long long wt = gweight(gkey_value<ES>(s.t), sc, h);
    unsigned long long cp = wt > 0 ? (target - m_above + wt - 1) / wt : s.ties;
    cp = max(1ull, min(cp, s.ties));
    g.thr_key = s.t;
    g.thr_id = g_tie_id<ES>(row, V, s.t, cp, red, sid, hist->dn);
    zk = m_above + cp * wt;
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
  extern __shared__ __align__(16) unsigned char g_dyn[];
  GHist& hist = *reinterpret_cast<GHist*>(g_dyn);  // sizeof(GHist) bytes of dynamic shared memory
  __shared__ GRow s_gt;  // the target row's record while its partner is selected
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
    {
      const GRow t = g_select_row<ES>(P, trow, red, &sid, &hist);
      if (threadIdx.x == 0) s_gt = t;
    }
    __syncthreads();
    GRow gdr{};
    int fl = s_gt.flags;
    int acc = 0;
    if (pair) {
      const unsigned char* drow = P.drf + static_cast<size_t>(gd) * P.V * ES;
      gdr = g_select_row<ES>(P, drow, red, &sid, &hist);
      const GRow gt = s_gt;
      fl |= gdr.flags;
      // label: sum over both kept sets of min(p_t, p_d), element by element
      float part = 0.f;
      if (P.out_conf != nullptr && !fl) {
        // min(p_t, p_d) is 0 unless both rows keep the token: keys first
        const float it = 1.f / gt.z, id = 1.f / gdr.z;
        g_for_pair<ES>(trow, drow, P.V, [&](int32_t v, float t, float d) {
          if (gkept(gt, gkey<ES>(t), v) && gkept(gdr, gkey<ES>(d), v))
            part += fminf(ex2(fmaf(t, P.sc, -gt.h)) * it, ex2(fmaf(d, P.sc, -gdr.h)) * id);
        });
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
      const GRow gt = s_gt;
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
  // thread t owns the ids of the row cover's vectors [t EV, t EV + EV), a run
  // of ascending ids read 16 bytes at a time
  constexpr int VEC = 16 / ES;
  const GCover ct = g_cover<ES>(trow, P.V), cd = g_cover<ES>(drow, P.V);
  const bool same_phase = ct.hoff == cd.hoff;
  const int32_t EV = (ct.nvec + kGThreads - 1) / kGThreads;
  const int32_t k0 = min(ct.nvec, tid * EV), k1 = min(ct.nvec, k0 + EV);
  const int32_t i0 = max(0, min(P.V, k0 * VEC - ct.hoff)), i1 = max(0, min(P.V, k1 * VEC - ct.hoff));
  auto wfun = [&](float xt, float xd, int32_t v, bool res) {
    const float pt = g_p<ES>(gt, xt, v, P.sc);
    return res ? fmaxf(0.f, pt - g_p<ES>(gd, xd, v, P.sc)) : pt;
  };
  auto weight = [&](int32_t v, bool res) {
    return wfun(load_elem<ES>(trow, v), res ? load_elem<ES>(drow, v) : 0.f, v, res);
  };
  for (int round = 0; round < 2; ++round) {
    float wsum = 0.f;
#pragma unroll 4
    for (int32_t k = k0; k < k1; ++k) {
      float xt[VEC], xd[VEC];
      g_unpack<ES>(g_ld16(ct.base, k), xt);
      if (residual && same_phase) {
        g_unpack<ES>(g_ld16(cd.base, k), xd);
      } else {
#pragma unroll
        for (int l = 0; l < VEC; ++l) {
          const int32_t v = k * VEC - ct.hoff + l;
          xd[l] = residual && v >= 0 && v < P.V ? load_elem<ES>(drow, v) : 0.f;
        }
      }
#pragma unroll
      for (int l = 0; l < VEC; ++l) {
        const int32_t v = k * VEC - ct.hoff + l;
        if (v >= 0 && v < P.V) wsum += wfun(xt[l], xd[l], v, residual);
      }
    }
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
