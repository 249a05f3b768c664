// sv_shard.cu -- the verify step over a vocabulary split across ranks
// (include/spec_verify_shard.h).
//
// A tensor-parallel LM head leaves rank q the columns [v_q, v_q + V_q) of
// every logits row (DFlash/Spec V2 page, section "A4 实验环境与运行配置":
// TP=8 serving).  Each step below is one launch on the caller's stream; the
// caller all-gathers the small per-row buffers between the steps:
//
//  stats   one CTA per target row: this rank's partial statistics of the
//          target row and its draft partner (sum 2^(x sc) = s 2^h, maximum,
//          lowest argmax id) and the two logits at the drafted token when
//          this rank holds it.  Reads the rank's columns once.
//  merge   one CTA per request: the ranks' partials merged in rank order
//          (one lane per rank, the same fixed tree on every rank, so every
//          rank gets the same bits), the accept test u * p_d(x) < p_t(x) or
//          x == argmax, the first rejection a_r and the accepted tokens.
//  masses  one CTA per target row (or per stopping row): this rank's shares
//          of sum min(p_t, p_d), sum max(0, p_t - p_d) and sum p_t under the
//          merged normalisers.  Reads the rank's columns a second time: the
//          normalisers are known only after the exchange.
//  draw    one CTA per request: labels from the shares in rank order; the
//          choice of the rank whose running mass passes u * total, and on
//          that rank the walk over its columns in ascending id.
//  finish  one thread per request: the owner's token.
//
// The residual and target weights of a token are formed by one function in
// both the masses and the draw kernels, with rounding fixed by explicit
// round-to-nearest operations, so a rank whose residual share is positive
// holds at least one token of positive weight in its walk.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <initializer_list>

#include "spec_verify_shard.h"
#include "sv_common.cuh"

namespace sv {
namespace shard {

constexpr int kShThreads = 256;
constexpr int kShWarps = kShThreads / 32;
// A residual mass at or below this counts as zero and the draw uses p_t
// (the same cutoff, 2^-21, as the unsplit path).
constexpr float kZeroResidualShard = 4.76837158203125e-07f;

__device__ __forceinline__ void flag_error(int32_t* dev_error, int bits) {
  if (dev_error != nullptr && bits) atomicOr(dev_error, bits);
}

__device__ __forceinline__ float f32w(int32_t w) { return __int_as_float(w); }

// Logit i of a row whose base is only element aligned.
template <int ES>
__device__ __forceinline__ float elem(const unsigned char* row, int32_t i) {
  if (ES == 2)
    return __uint_as_float(static_cast<uint32_t>(__ldg(reinterpret_cast<const uint16_t*>(row) + i))
                           << 16);
  return __ldg(reinterpret_cast<const float*>(row) + i);
}

template <int ES>
__device__ __forceinline__ void unpack16(const uint4 w, float* x) {
  if (ES == 2) {
    x[0] = bf16lo(w.x); x[1] = bf16hi(w.x); x[2] = bf16lo(w.y); x[3] = bf16hi(w.y);
    x[4] = bf16lo(w.z); x[5] = bf16hi(w.z); x[6] = bf16lo(w.w); x[7] = bf16hi(w.w);
  } else {
    x[0] = __uint_as_float(w.x); x[1] = __uint_as_float(w.y);
    x[2] = __uint_as_float(w.z); x[3] = __uint_as_float(w.w);
  }
}

// Visit elements [0, n) of row a, and of row b at the same indices when b is
// given, as f(i, a_i, b_i): the elements before the first 16-byte boundary
// and after the last one one at a time, the rest as 16-byte vectors of both
// rows when the two rows share their offset within 16 bytes, else all one
// at a time.  Each thread visits its indices in ascending order.
template <int ES, typename F>
__device__ __forceinline__ void for_elems(const unsigned char* a, const unsigned char* b, int32_t n,
                                          F&& f) {
  constexpr int VEC = 16 / ES;
  const int tid = threadIdx.x;
  const uintptr_t pa = reinterpret_cast<uintptr_t>(a);
  const bool vec = b == nullptr || ((pa ^ reinterpret_cast<uintptr_t>(b)) & 15u) == 0;
  if (!vec) {
    for (int32_t i = tid; i < n; i += kShThreads) f(i, elem<ES>(a, i), elem<ES>(b, i));
    return;
  }
  const int32_t head = min(n, static_cast<int32_t>(((16u - (pa & 15u)) & 15u) / ES));
  const int32_t nvec = (n - head) / VEC;
  const int32_t tail = head + nvec * VEC;
  if (tid < head) f(tid, elem<ES>(a, tid), b ? elem<ES>(b, tid) : 0.f);
  const uint4* va = reinterpret_cast<const uint4*>(a + head * ES);
  const uint4* vb = b ? reinterpret_cast<const uint4*>(b + head * ES) : nullptr;
#pragma unroll 2
  for (int32_t k = tid; k < nvec; k += kShThreads) {
    float x[VEC], y[VEC];
    unpack16<ES>(__ldg(va + k), x);
    if (vb) unpack16<ES>(__ldg(vb + k), y);
#pragma unroll
    for (int l = 0; l < VEC; ++l) f(head + k * VEC + l, x[l], vb ? y[l] : 0.f);
  }
  for (int32_t i = tail + tid; i < n; i += kShThreads)
    f(i, elem<ES>(a, i), b ? elem<ES>(b, i) : 0.f);
}

// Request layout, checked as the unsplit path checks it.
struct ReqLayout {
  int32_t off, ell;
  bool ok;
};

__device__ __forceinline__ ReqLayout req_layout(const int32_t* lens, const int32_t* offs, int32_t r,
                                                int32_t B, int32_t Nt, int32_t max_len) {
  ReqLayout L;
  L.off = __ldg(offs + r);
  const int32_t off1 = __ldg(offs + r + 1);
  L.ell = __ldg(lens + r);
  L.ok = L.ell >= 1 && L.ell <= max_len && off1 - L.off == L.ell && L.off >= r && off1 <= Nt &&
         (r != 0 || L.off == 0) && (r != B - 1 || off1 == Nt) && L.off - r + L.ell - 1 <= Nt - B;
  return L;
}

// The request holding target row g: the largest r with offs[r] <= g.
__device__ __forceinline__ int32_t find_request(const int32_t* offs, int32_t B, int32_t g) {
  int32_t lo = 0, hi = B - 1;
  while (lo < hi) {
    const int32_t mid = (lo + hi + 1) >> 1;
    if (__ldg(offs + mid) <= g) lo = mid;
    else hi = mid - 1;
  }
  return lo;
}

// Add logit x (id v) to running statistics s * 2^h = sum 2^(x sc) with
// h = m sc for the maximum m so far (lowest id on ties: ids arrive in
// ascending order per thread); NaN and +inf mark the row bad.
__device__ __forceinline__ void stat_add(RStat& st, float x, int32_t v, float sc, bool& bad) {
  if (x != x || x == INFINITY) {
    bad = true;
    return;
  }
  if (x > st.m) {
    const float nh = x * sc;
    if (!(fabsf(nh) < INFINITY)) bad = true;
    st.s = (st.h > -INFINITY ? st.s * ex2(st.h - nh) : 0.f) + 1.f;
    st.h = nh;
    st.m = x;
    st.i = v;
  } else if (st.h > -INFINITY) {
    st.s += ex2(fmaf(x, sc, -st.h));
  }
}

// Merge per-thread statistics of a target and a draft row over the CTA
// (fixed order: the warp tree, then warp 0 over the warps' results); the
// result is valid in warp 0.
__device__ __forceinline__ void block_reduce_stats(RStat& t, RStat& d, RStat* red_t, RStat* red_d) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  rstat_warp_reduce2<true>(t, d);
  if (lane == 0) {
    red_t[warp] = t;
    red_d[warp] = d;
  }
  __syncthreads();
  if (warp == 0) {
    t = lane < kShWarps ? red_t[lane] : rstat_empty();
    d = lane < kShWarps ? red_d[lane] : rstat_empty();
    rstat_warp_reduce2<true>(t, d);
  }
}

struct StatsArgs {
  const unsigned char* tgt;
  const unsigned char* drf;
  const int32_t* tokens;
  const int32_t* lens;
  const int32_t* offs;
  int32_t Vq, v0, B, Nt, max_len;
  float sc;
  int32_t* rec;
};

// Step 1: one CTA per target row g.
template <int ES>
__global__ void __launch_bounds__(kShThreads) shard_stats_kernel(const StatsArgs a) {
  __shared__ RStat red_t[kShWarps], red_d[kShWarps];
  const int32_t g = blockIdx.x;
  const int tid = threadIdx.x;
  const int32_t r = find_request(a.offs, a.B, g);
  const ReqLayout L = req_layout(a.lens, a.offs, r, a.B, a.Nt, a.max_len);
  const bool inrow = L.ok && g >= L.off && g < L.off + L.ell;
  const int32_t j = g - L.off;
  const bool pair = inrow && j < L.ell - 1;
  const int32_t gd = L.off - r + j;  // draft partner (pair only)
  const unsigned char* trow = a.tgt + static_cast<size_t>(g) * a.Vq * ES;
  const unsigned char* drow = pair ? a.drf + static_cast<size_t>(gd) * a.Vq * ES : nullptr;
  RStat t = rstat_empty(), d = rstat_empty();
  bool bad = false;
  for_elems<ES>(trow, nullptr, a.Vq, [&](int32_t i, float x, float) {
    stat_add(t, x, a.v0 + i, a.sc, bad);
  });
  if (pair)
    for_elems<ES>(drow, nullptr, a.Vq, [&](int32_t i, float x, float) {
      stat_add(d, x, a.v0 + i, a.sc, bad);
    });
  const bool anybad = __syncthreads_or(bad ? 1 : 0) != 0;
  block_reduce_stats(t, d, red_t, red_d);
  if (tid == 0) {
    int32_t* w = a.rec + static_cast<size_t>(g) * SV_SHARD_REC_WORDS;
    int flags = anybad ? SV_DEVERR_NAN : 0;
    if (!inrow) flags |= SV_DEVERR_LEN;
    float xt = 0.f, xd = 0.f;
    int32_t hasx = 0;
    if (pair) {
      const int32_t x = __ldg(a.tokens + gd);
      if (x >= a.v0 && x - a.v0 < a.Vq) {
        hasx = 1;
        xt = elem<ES>(trow, x - a.v0);
        xd = elem<ES>(drow, x - a.v0);
      }
    }
    w[SV_SREC_HT] = __float_as_int(t.h);
    w[SV_SREC_ST] = __float_as_int(t.s);
    w[SV_SREC_MT] = __float_as_int(t.m);
    w[SV_SREC_IT] = t.i;
    w[SV_SREC_HD] = __float_as_int(d.h);
    w[SV_SREC_SD] = __float_as_int(d.s);
    w[SV_SREC_MD] = __float_as_int(d.m);
    w[SV_SREC_ID] = d.i;
    w[SV_SREC_XT] = __float_as_int(xt);
    w[SV_SREC_XD] = __float_as_int(xd);
    w[SV_SREC_HASX] = hasx;
    w[SV_SREC_FLAGS] = flags;
  }
}

struct MergeArgs {
  const int32_t* recs;
  int32_t world;
  const int32_t* tokens;
  const float* uniforms;
  const int32_t* lens;
  const int32_t* offs;
  int32_t B, V, Nt, max_len;
  float T, sc;
  int32_t mode;
  int32_t* merged;
  int32_t* out_tokens;
  int32_t* accept_len;
  float* row_stats;
  int32_t* dev_error;
};

// Step 1 after the exchange: one CTA per request.  Warp w merges rows
// w, w + kShWarps, ... (lane q = rank q), then the CTA scans for the first
// rejection and writes the accepted tokens.
__global__ void __launch_bounds__(kShThreads) shard_merge_kernel(const MergeArgs a) {
  __shared__ uint32_t marks[SV_MAX_LEN];
  __shared__ int32_t argt[SV_MAX_LEN];
  __shared__ int32_t s_a;
  const int32_t r = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const ReqLayout L = req_layout(a.lens, a.offs, r, a.B, a.Nt, a.max_len);
  if (!L.ok) {  // uniform over the CTA
    if (tid == 0) {
      flag_error(a.dev_error, SV_DEVERR_LEN);
      a.accept_len[r] = -1;
    }
    return;
  }
  for (int32_t j = warp; j < L.ell; j += kShWarps) {
    const int32_t g = L.off + j;
    const bool pair = j < L.ell - 1;
    const int32_t gd = L.off - r + j;
    RStat t = rstat_empty(), d = rstat_empty();
    float xt = 0.f, xd = 0.f;
    bool hasx = false;
    int flags = 0;
    if (lane < a.world) {
      const int32_t* w = a.recs + (static_cast<size_t>(lane) * a.Nt + g) * SV_SHARD_REC_WORDS;
      t = RStat{f32w(w[SV_SREC_HT]), f32w(w[SV_SREC_ST]), f32w(w[SV_SREC_MT]), w[SV_SREC_IT]};
      if (pair) d = RStat{f32w(w[SV_SREC_HD]), f32w(w[SV_SREC_SD]), f32w(w[SV_SREC_MD]), w[SV_SREC_ID]};
      xt = f32w(w[SV_SREC_XT]);
      xd = f32w(w[SV_SREC_XD]);
      hasx = pair && w[SV_SREC_HASX] != 0;
      flags = w[SV_SREC_FLAGS];
    }
    rstat_warp_reduce2<true>(t, d);
    flags = __reduce_or_sync(0xffffffffu, flags);
    const unsigned xl = __ballot_sync(0xffffffffu, hasx);
    if (xl) {
      xt = __shfl_sync(0xffffffffu, xt, __ffs(xl) - 1);
      xd = __shfl_sync(0xffffffffu, xd, __ffs(xl) - 1);
    }
    if (lane == 0) {
      int fl = flags;
      if (!(t.s > 0.f && t.s < INFINITY) || !(t.m > -INFINITY && t.m < INFINITY)) fl |= SV_DEVERR_NAN;
      if (pair && (!(d.s > 0.f && d.s < INFINITY) || !(d.m > -INFINITY && d.m < INFINITY)))
        fl |= SV_DEVERR_NAN;
      int acc = 0;
      if (pair) {
        const int32_t x = __ldg(a.tokens + gd);
        if (!(x >= 0 && x < a.V && xl != 0)) {
          fl |= SV_DEVERR_TOKEN;
        } else if (a.mode == SV_GREEDY) {
          acc = x == t.i;
        } else {
          // p_t(x) / p_d(x) = 2^(a - b) * s_d / s_t, a = x_t sc - h_t, b = x_d sc - h_d
          const float ratio = exp2f(fmaf(xt, a.sc, -t.h) - fmaf(xd, a.sc, -d.h)) * (d.s / t.s);
          acc = __ldg(a.uniforms + g) < ratio;
        }
      }
      int32_t* m = a.merged + static_cast<size_t>(g) * SV_SHARD_ROW_WORDS;
      m[SV_SROW_HT] = __float_as_int(t.h);
      m[SV_SROW_ZT] = __float_as_int(t.s);
      m[SV_SROW_HD] = __float_as_int(d.h);
      m[SV_SROW_ZD] = __float_as_int(d.s);
      m[SV_SROW_ARGT] = t.i;
      m[SV_SROW_ACC] = acc;
      m[SV_SROW_FLAGS] = fl;
      m[SV_SROW_PAD] = 0;
      marks[j] = (acc ? 0x80000000u : 0u) | (static_cast<uint32_t>(fl) & 0x7fffffffu);
      argt[j] = t.i;
      if (a.row_stats != nullptr) {
        // Z relative to the true maximum: s * 2^(h - m sc)
        float* o = a.row_stats + 3 * static_cast<size_t>(g);
        o[0] = t.m / a.T;
        o[1] = t.s * exp2f(-fmaf(t.m, a.sc, -t.h));
        o[2] = __int_as_float(t.i);
        if (pair) {
          float* o2 = a.row_stats + 3 * (static_cast<size_t>(a.Nt) + gd);
          o2[0] = d.m / a.T;
          o2[1] = d.s * exp2f(-fmaf(d.m, a.sc, -d.h));
          o2[2] = __int_as_float(d.i);
        }
      }
    }
  }
  __syncthreads();
  if (tid == 0) {
    int32_t first = L.ell - 1;  // every drafted token accepted
    for (int32_t j = 0; j < L.ell - 1; ++j)
      if (!(marks[j] >> 31)) {
        first = j;
        break;
      }
    s_a = first;
    a.accept_len[r] = first;
  }
  __syncthreads();
  const int32_t ar = s_a;
  for (int32_t j = tid; j < L.ell; j += kShThreads) {
    int32_t v = -1;
    if (j < ar) v = __ldg(a.tokens + L.off - r + j);
    else if (j == ar && a.mode == SV_GREEDY) v = argt[j];
    a.out_tokens[L.off + j] = v;
    const int fl = static_cast<int>(marks[j] & 0x7fffffffu);
    if (j <= ar) flag_error(a.dev_error, fl);
  }
}

// Normalisers of a merged row: p_t(v) = 2^(x_v sc - h_t) / z_t, likewise
// p_d with the draft partner's.
struct Norm {
  float ht, izt, hd, izd, sc;
};

__device__ __forceinline__ Norm load_norm(const int32_t* merged, int32_t g, float sc) {
  const int32_t* m = merged + static_cast<size_t>(g) * SV_SHARD_ROW_WORDS;
  Norm n;
  n.ht = f32w(m[SV_SROW_HT]);
  n.izt = 1.f / f32w(m[SV_SROW_ZT]);
  n.hd = f32w(m[SV_SROW_HD]);
  n.izd = 1.f / f32w(m[SV_SROW_ZD]);
  n.sc = sc;
  return n;
}

// p_t and p_d of one token; the products are rounded on their own (no
// contraction into a later add), so every kernel forms the same values.
__device__ __forceinline__ float prob_t(float t, const Norm& n) {
  return __fmul_rn(ex2(fmaf(t, n.sc, -n.ht)), n.izt);
}
__device__ __forceinline__ float prob_d(float d, const Norm& n) {
  return __fmul_rn(ex2(fmaf(d, n.sc, -n.hd)), n.izd);
}
// Weight of a token in the final draw: max(0, p_t - p_d) or p_t.
__device__ __forceinline__ float draw_weight(float t, float d, const Norm& n, bool residual) {
  const float pt = prob_t(t, n);
  return residual ? fmaxf(0.f, __fsub_rn(pt, prob_d(d, n))) : pt;
}

// Sum over the CTA of one float per thread in a fixed order (the warp tree,
// then the warps' sums in warp order); the result is valid in thread 0.
__device__ __forceinline__ float block_sum(float v, float* red) {
  v = warp_sum_f32(v);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  __syncthreads();
  float s = 0.f;
  if (threadIdx.x == 0)
    for (int w = 0; w < kShWarps; ++w) s += red[w];
  __syncthreads();
  return s;
}

struct MassArgs {
  const unsigned char* tgt;
  const unsigned char* drf;
  int32_t Vq;
  const int32_t* merged;
  const int32_t* lens;
  const int32_t* offs;
  const int32_t* accept_len;
  int32_t B, Nt, max_len;
  float sc;
  int32_t all_rows;
  float* mass;
};

// Step 2: one CTA per target row (all_rows) or per request (its stopping
// row only).
template <int ES>
__global__ void __launch_bounds__(kShThreads) shard_masses_kernel(const MassArgs a) {
  __shared__ float red[kShWarps];
  int32_t r, g;
  if (a.all_rows) {
    g = blockIdx.x;
    r = find_request(a.offs, a.B, g);
  } else {
    r = blockIdx.x;
    g = -1;
  }
  const ReqLayout L = req_layout(a.lens, a.offs, r, a.B, a.Nt, a.max_len);
  if (!L.ok) return;  // uniform over the CTA; the merge raised the error
  if (!a.all_rows) {
    const int32_t ar = __ldg(a.accept_len + r);
    if (ar < 0 || ar >= L.ell) return;
    g = L.off + ar;
  } else if (g < L.off || g >= L.off + L.ell) {
    return;
  }
  const int32_t j = g - L.off;
  const bool pair = j < L.ell - 1;
  const Norm n = load_norm(a.merged, g, a.sc);
  const unsigned char* trow = a.tgt + static_cast<size_t>(g) * a.Vq * ES;
  const unsigned char* drow =
      pair ? a.drf + static_cast<size_t>(L.off - r + j) * a.Vq * ES : nullptr;
  float c = 0.f, res = 0.f, pm = 0.f;
  if (pair) {
    for_elems<ES>(trow, drow, a.Vq, [&](int32_t, float t, float d) {
      const float pt = prob_t(t, n), pd = prob_d(d, n);
      c += fminf(pt, pd);
      res += fmaxf(0.f, __fsub_rn(pt, pd));
      pm += pt;
    });
  } else {
    for_elems<ES>(trow, nullptr, a.Vq, [&](int32_t, float t, float) { pm += prob_t(t, n); });
  }
  c = block_sum(c, red);
  res = block_sum(res, red);
  pm = block_sum(pm, red);
  if (threadIdx.x == 0) {
    float* o = a.mass + static_cast<size_t>(g) * SV_SHARD_MASS_WORDS;
    o[SV_SMASS_C] = c;
    o[SV_SMASS_R] = res;
    o[SV_SMASS_P] = pm;
    o[SV_SMASS_PAD] = 0.f;
  }
}

// Inclusive scan of v over the warp's lanes.
__device__ __forceinline__ float lane_scan(float v) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const float o = __shfl_up_sync(0xffffffffu, v, d);
    if (lane >= d) v += o;
  }
  return v;
}

struct DrawArgs {
  const float* masses;
  int32_t world, rank;
  const unsigned char* tgt;
  const unsigned char* drf;
  int32_t Vq, v0;
  const int32_t* merged;
  const float* uniforms;
  const int32_t* lens;
  const int32_t* offs;
  const int32_t* accept_len;
  int32_t B, Nt, max_len;
  float sc;
  int32_t mode;
  float* conf;
  int32_t* cand;
  int32_t* dev_error;
};

// Step 3: one CTA per request.
template <int ES>
__global__ void __launch_bounds__(kShThreads) shard_draw_kernel(const DrawArgs a) {
  __shared__ float scan[kShWarps];
  __shared__ float s_need;
  __shared__ int32_t s_owner, s_resid, s_pick;
  const int32_t r = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const bool sample = a.mode == SV_SAMPLE;
  if (sample && tid == 0) a.cand[r] = -1;
  const ReqLayout L = req_layout(a.lens, a.offs, r, a.B, a.Nt, a.max_len);
  if (!L.ok) return;  // uniform; the merge raised the error
  const size_t plane = static_cast<size_t>(a.Nt) * SV_SHARD_MASS_WORDS;
  auto share = [&](int32_t q, int32_t g, int w) {
    return __ldg(a.masses + q * plane + static_cast<size_t>(g) * SV_SHARD_MASS_WORDS + w);
  };
  if (a.conf != nullptr)  // c* of every drafted row: the ranks' shares in rank order
    for (int32_t j = tid; j < L.ell - 1; j += kShThreads) {
      float c = 0.f;
      for (int32_t q = 0; q < a.world; ++q) c += share(q, L.off + j, SV_SMASS_C);
      a.conf[L.off - r + j] = c;
    }
  if (!sample) return;
  const int32_t ar = __ldg(a.accept_len + r);
  if (ar < 0 || ar >= L.ell) return;  // uniform
  const int32_t g = L.off + ar;
  if (tid == 0) {  // the rank that owns the draw, and the mass to pass inside its columns
    bool resid = ar < L.ell - 1;
    float rsum = 0.f;
    for (int32_t q = 0; q < a.world; ++q) rsum += share(q, g, SV_SMASS_R);
    if (resid && !(rsum > kZeroResidualShard)) resid = false;  // rounding only: p_t
    const int kind = resid ? SV_SMASS_R : SV_SMASS_P;
    float total = 0.f;
    for (int32_t q = 0; q < a.world; ++q) total += share(q, g, kind);
    const float target = __ldg(a.uniforms + L.off + L.ell - 1) * total;
    int32_t owner = -1, last = -1;
    float incl = 0.f, need = 0.f, need_last = 0.f;
    for (int32_t q = 0; q < a.world; ++q) {
      const float w = share(q, g, kind);
      const float before = incl;
      incl += w;
      if (w > 0.f) {
        last = q;
        need_last = target - before;
        if (owner < 0 && target < incl) {
          owner = q;
          need = target - before;
        }
      }
    }
    if (owner < 0) {  // rounding left the target at or past the total
      owner = last;
      need = need_last;
    }
    s_owner = owner;
    s_need = fmaxf(0.f, need);
    s_resid = resid;
    s_pick = -1;
  }
  __syncthreads();
  if (s_owner != a.rank) return;  // uniform; another rank draws (or none: no mass)
  const bool resid = s_resid != 0;
  const float need = s_need;
  const Norm n = load_norm(a.merged, g, a.sc);
  const unsigned char* trow = a.tgt + static_cast<size_t>(g) * a.Vq * ES;
  const unsigned char* drow =
      resid ? a.drf + static_cast<size_t>(L.off - r + ar) * a.Vq * ES : nullptr;
  auto weight = [&](int32_t i) {
    return draw_weight(elem<ES>(trow, i), resid ? elem<ES>(drow, i) : 0.f, n, resid);
  };
  // thread t owns the run [i0, i1) of ascending ids; runs tile the columns
  const int32_t E = (a.Vq + kShThreads - 1) / kShThreads;
  const int32_t i0 = min(a.Vq, tid * E), i1 = min(a.Vq, i0 + E);
  float wsum = 0.f;
  for (int32_t i = i0; i < i1; ++i) wsum += weight(i);
  // each thread's interval [lo, hi) of the running sum in thread order; hi
  // of one thread is lo of the next, so the intervals tile [0, total)
  const float incl = lane_scan(wsum);
  const float prev = __shfl_up_sync(0xffffffffu, incl, 1);
  if (lane == 31) scan[warp] = incl;
  __syncthreads();
  float base = 0.f, tot = 0.f;
  for (int w = 0; w < kShWarps; ++w) {
    if (w < warp) base += scan[w];
    tot += scan[w];
  }
  const float lo = lane == 0 ? base : base + prev;
  const float hi = base + incl;
  const bool own = tot > 0.f && lo < hi && ((lo <= need && need < hi) || (need >= tot && hi == tot));
  const unsigned ob = __ballot_sync(0xffffffffu, own);
  if (ob) {  // the owner's warp walks the owner's run, 32 ids a step
    const int ol = __ffs(ob) - 1;
    const int32_t o0 = __shfl_sync(0xffffffffu, i0, ol), o1 = __shfl_sync(0xffffffffu, i1, ol);
    const float left = __shfl_sync(0xffffffffu, need - lo, ol);
    float run_base = 0.f;
    int32_t p = -1, lastp = -1;
    for (int32_t b0 = o0; b0 < o1 && p < 0; b0 += 32) {
      const int32_t i = b0 + lane;
      const float wv = i < o1 ? weight(i) : 0.f;
      const float run = run_base + lane_scan(wv);
      const unsigned hit = __ballot_sync(0xffffffffu, wv > 0.f && run > left);
      const unsigned pos = __ballot_sync(0xffffffffu, wv > 0.f);
      if (pos) lastp = b0 + 31 - __clz(pos);
      if (hit) p = b0 + __ffs(hit) - 1;
      run_base = __shfl_sync(0xffffffffu, run, 31);
    }
    if (p < 0) p = lastp;
    if (lane == 0 && p >= 0) s_pick = a.v0 + p;
  }
  __syncthreads();
  if (tid == 0) a.cand[r] = s_pick;
}

struct FinishArgs {
  const int32_t* cands;
  int32_t world;
  const int32_t* merged;
  const int32_t* lens;
  const int32_t* offs;
  const int32_t* accept_len;
  int32_t B, Nt;
  int32_t* out_tokens;
  int32_t* dev_error;
};

// Step 3 after the exchange: one thread per request.
__global__ void __launch_bounds__(kShThreads) shard_finish_kernel(const FinishArgs a) {
  const int32_t r = blockIdx.x * kShThreads + threadIdx.x;
  if (r >= a.B) return;
  const ReqLayout L = req_layout(a.lens, a.offs, r, a.B, a.Nt, SV_MAX_LEN);
  if (!L.ok) return;
  const int32_t ar = __ldg(a.accept_len + r);
  if (ar < 0 || ar >= L.ell) return;
  int32_t tok = -1;
  for (int32_t q = 0; q < a.world && tok < 0; ++q) tok = __ldg(a.cands + static_cast<size_t>(q) * a.B + r);
  if (tok < 0) {  // no rank held any mass: non-finite statistics
    flag_error(a.dev_error, SV_DEVERR_NAN);
    tok = __ldg(a.merged + static_cast<size_t>(L.off + ar) * SV_SHARD_ROW_WORDS + SV_SROW_ARGT);
  }
  a.out_tokens[L.off + ar] = tok;
}

}  // namespace shard
}  // namespace sv

// ---------------------------------------------------------------------------
// Host side: argument checks (before anything is enqueued), then one launch.
namespace {

bool aligned_to(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int esize(int32_t dtype) { return dtype == SV_BF16 ? 2 : dtype == SV_FP32 ? 4 : 0; }

// Sizes shared by every step: B requests, N_t target rows, max_len.
int check_sizes(int32_t B, int32_t Nt, int32_t max_len) {
  if (B <= 0 || Nt < B) return SV_ERR_ARG;
  if (max_len < 1 || max_len > SV_MAX_LEN) return SV_ERR_ARG;
  if (static_cast<int64_t>(B) * max_len < Nt) return SV_ERR_ARG;
  return SV_OK;
}

// This rank's columns: V_shard >= 1 starting at v_begin inside [0, V).
int check_columns(const void* tgt, const void* drf, int32_t Vq, int32_t Nt, int32_t B,
                  int32_t dtype) {
  const int es = esize(dtype);
  if (es == 0) return SV_ERR_DTYPE;
  if (Vq < 1 || tgt == nullptr || !aligned_to(tgt, es)) return SV_ERR_ARG;
  if (Nt > B && (drf == nullptr || !aligned_to(drf, es))) return SV_ERR_ARG;
  if (static_cast<double>(Nt) * Vq * es > 9.0e18) return SV_ERR_ARG;
  return SV_OK;
}

bool temperature_ok(float T) { return T > 0.f && std::isfinite(T); }

bool ptrs4_ok(std::initializer_list<const void*> ps) {
  for (const void* p : ps)
    if (p != nullptr && !aligned_to(p, 4)) return false;
  return true;
}

int launched() { return cudaGetLastError() == cudaSuccess ? SV_OK : SV_ERR_CUDA; }

float scale_of(float T) { return 1.4426950408889634f / T; }  // log2(e) / T

}  // namespace

extern "C" {

int spec_verify_shard_stats(const void* target_shard, const void* draft_shard, int32_t V_shard,
                            int32_t v_begin, int32_t V, const int32_t* draft_tokens,
                            const int32_t* verify_lens, const int32_t* row_offsets, int32_t B,
                            int32_t n_target_rows, int32_t max_len, int32_t dtype,
                            float temperature, int32_t* out_rec, void* stream) {
  int rc = check_sizes(B, n_target_rows, max_len);
  if (rc == SV_OK) rc = check_columns(target_shard, draft_shard, V_shard, n_target_rows, B, dtype);
  if (rc != SV_OK) return rc;
  if (V <= 0 || v_begin < 0 || static_cast<int64_t>(v_begin) + V_shard > V) return SV_ERR_ARG;
  if (!temperature_ok(temperature)) return SV_ERR_ARG;
  if (verify_lens == nullptr || row_offsets == nullptr || out_rec == nullptr) return SV_ERR_ARG;
  if (n_target_rows > B && draft_tokens == nullptr) return SV_ERR_ARG;
  if (!ptrs4_ok({draft_tokens, verify_lens, row_offsets, out_rec})) return SV_ERR_ARG;
  sv::shard::StatsArgs a{static_cast<const unsigned char*>(target_shard),
                         static_cast<const unsigned char*>(draft_shard), draft_tokens, verify_lens,
                         row_offsets, V_shard, v_begin, B, n_target_rows, max_len,
                         scale_of(temperature), out_rec};
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (dtype == SV_BF16)
    sv::shard::shard_stats_kernel<2><<<n_target_rows, sv::shard::kShThreads, 0, s>>>(a);
  else
    sv::shard::shard_stats_kernel<4><<<n_target_rows, sv::shard::kShThreads, 0, s>>>(a);
  return launched();
}

int spec_verify_shard_merge(const int32_t* recs, int32_t world, const int32_t* draft_tokens,
                            const float* uniforms, const int32_t* verify_lens,
                            const int32_t* row_offsets, int32_t B, int32_t V,
                            int32_t n_target_rows, int32_t max_len, float temperature,
                            int32_t mode, int32_t* out_merged, int32_t* out_tokens,
                            int32_t* out_accept_len, float* out_row_stats, int32_t* dev_error,
                            void* stream) {
  const int rc = check_sizes(B, n_target_rows, max_len);
  if (rc != SV_OK) return rc;
  if (world < 1 || world > SV_SHARD_MAX_WORLD || V <= 0) return SV_ERR_ARG;
  if (mode != SV_GREEDY && mode != SV_SAMPLE) return SV_ERR_ARG;
  if (!temperature_ok(temperature)) return SV_ERR_ARG;
  if (recs == nullptr || uniforms == nullptr || verify_lens == nullptr ||
      row_offsets == nullptr || out_merged == nullptr || out_tokens == nullptr ||
      out_accept_len == nullptr)
    return SV_ERR_ARG;
  if (n_target_rows > B && draft_tokens == nullptr) return SV_ERR_ARG;
  if (!ptrs4_ok({recs, draft_tokens, uniforms, verify_lens, row_offsets, out_merged, out_tokens,
                 out_accept_len, out_row_stats, dev_error}))
    return SV_ERR_ARG;
  sv::shard::MergeArgs a{recs,         world,        draft_tokens,
                         uniforms,     verify_lens,  row_offsets,
                         B,            V,            n_target_rows,
                         max_len,      temperature,  scale_of(temperature),
                         mode,         out_merged,   out_tokens,
                         out_accept_len, out_row_stats, dev_error};
  sv::shard::shard_merge_kernel<<<B, sv::shard::kShThreads, 0, static_cast<cudaStream_t>(stream)>>>(a);
  return launched();
}

int spec_verify_shard_masses(const void* target_shard, const void* draft_shard, int32_t V_shard,
                             const int32_t* merged, const int32_t* verify_lens,
                             const int32_t* row_offsets, const int32_t* accept_len, int32_t B,
                             int32_t n_target_rows, int32_t max_len, int32_t dtype,
                             float temperature, int32_t all_rows, float* out_mass, void* stream) {
  int rc = check_sizes(B, n_target_rows, max_len);
  if (rc == SV_OK) rc = check_columns(target_shard, draft_shard, V_shard, n_target_rows, B, dtype);
  if (rc != SV_OK) return rc;
  if (!temperature_ok(temperature) || (all_rows != 0 && all_rows != 1)) return SV_ERR_ARG;
  if (merged == nullptr || verify_lens == nullptr || row_offsets == nullptr ||
      accept_len == nullptr || out_mass == nullptr)
    return SV_ERR_ARG;
  if (!ptrs4_ok({merged, verify_lens, row_offsets, accept_len, out_mass})) return SV_ERR_ARG;
  sv::shard::MassArgs a{static_cast<const unsigned char*>(target_shard),
                        static_cast<const unsigned char*>(draft_shard), V_shard, merged,
                        verify_lens, row_offsets, accept_len, B, n_target_rows, max_len,
                        scale_of(temperature), all_rows, out_mass};
  const int grid = all_rows ? n_target_rows : B;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (dtype == SV_BF16)
    sv::shard::shard_masses_kernel<2><<<grid, sv::shard::kShThreads, 0, s>>>(a);
  else
    sv::shard::shard_masses_kernel<4><<<grid, sv::shard::kShThreads, 0, s>>>(a);
  return launched();
}

int spec_verify_shard_draw(const float* masses, int32_t world, int32_t rank,
                           const void* target_shard, const void* draft_shard, int32_t V_shard,
                           int32_t v_begin, const int32_t* merged, const float* uniforms,
                           const int32_t* verify_lens, const int32_t* row_offsets,
                           const int32_t* accept_len, int32_t B, int32_t n_target_rows,
                           int32_t max_len, int32_t dtype, float temperature, int32_t mode,
                           float* out_conf, int32_t* out_cand, int32_t* dev_error, void* stream) {
  int rc = check_sizes(B, n_target_rows, max_len);
  if (rc == SV_OK) rc = check_columns(target_shard, draft_shard, V_shard, n_target_rows, B, dtype);
  if (rc != SV_OK) return rc;
  if (world < 1 || world > SV_SHARD_MAX_WORLD || rank < 0 || rank >= world || v_begin < 0)
    return SV_ERR_ARG;
  if (mode != SV_GREEDY && mode != SV_SAMPLE) return SV_ERR_ARG;
  if (!temperature_ok(temperature)) return SV_ERR_ARG;
  if (masses == nullptr || merged == nullptr || verify_lens == nullptr ||
      row_offsets == nullptr || accept_len == nullptr)
    return SV_ERR_ARG;
  if (mode == SV_SAMPLE && (uniforms == nullptr || out_cand == nullptr)) return SV_ERR_ARG;
  if (!ptrs4_ok({masses, merged, uniforms, verify_lens, row_offsets, accept_len, out_conf,
                 out_cand, dev_error}))
    return SV_ERR_ARG;
  sv::shard::DrawArgs a{masses,      world,       rank,
                        static_cast<const unsigned char*>(target_shard),
                        static_cast<const unsigned char*>(draft_shard),
                        V_shard,     v_begin,     merged,
                        uniforms,    verify_lens, row_offsets,
                        accept_len,  B,           n_target_rows,
                        max_len,     scale_of(temperature), mode,
                        out_conf,    out_cand,    dev_error};
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (dtype == SV_BF16)
    sv::shard::shard_draw_kernel<2><<<B, sv::shard::kShThreads, 0, s>>>(a);
  else
    sv::shard::shard_draw_kernel<4><<<B, sv::shard::kShThreads, 0, s>>>(a);
  return launched();
}

int spec_verify_shard_finish(const int32_t* cands, int32_t world, const int32_t* merged,
                             const int32_t* verify_lens, const int32_t* row_offsets,
                             const int32_t* accept_len, int32_t B, int32_t n_target_rows,
                             int32_t* out_tokens, int32_t* dev_error, void* stream) {
  if (B <= 0 || n_target_rows < B) return SV_ERR_ARG;
  if (world < 1 || world > SV_SHARD_MAX_WORLD) return SV_ERR_ARG;
  if (cands == nullptr || merged == nullptr || verify_lens == nullptr || row_offsets == nullptr ||
      accept_len == nullptr || out_tokens == nullptr)
    return SV_ERR_ARG;
  if (!ptrs4_ok({cands, merged, verify_lens, row_offsets, accept_len, out_tokens, dev_error}))
    return SV_ERR_ARG;
  sv::shard::FinishArgs a{cands, world, merged, verify_lens, row_offsets, accept_len,
                          B,     n_target_rows, out_tokens, dev_error};
  const int grid = (B + sv::shard::kShThreads - 1) / sv::shard::kShThreads;
  sv::shard::shard_finish_kernel<<<grid, sv::shard::kShThreads, 0,
                                   static_cast<cudaStream_t>(stream)>>>(a);
  return launched();
}

}  // extern "C"
