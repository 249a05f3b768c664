// sv_filter.cuh -- the verify step with top-k (k <= 64) and top-p filtering.
//
// Sampling parameters temperature, top_k and top_p (DSpine page, "加速效果":
// T 1.0, top_p 0.95, top_k 20) apply to the target and the draft rows alike.
// Every probability the verify step needs is then supported on at most k
// tokens per row, so the work splits in two:
//
//  filter_rows_kernel   one CTA per logits row, one streaming pass: the row's
//                       k largest logits by (value desc, id asc), exact; then
//                       the softmax weights of those k relative to the row
//                       maximum, renormalised, and the top-p cut (shortest
//                       prefix of that order whose cumulative probability
//                       reaches top_p), renormalised again.  The kept tokens
//                       and weights go to a FiltRow record in the workspace.
//  filter_requests_kernel  one warp per request, on the FiltRow records only:
//                       the accept chain u * p_d(x) < p_t(x) (greedy: x is
//                       the target argmax), the confidence labels
//                       c* = sum_v min(p_t, p_d) over the two kept sets
//                       (DSpark tutorial, "置信度预测头"), and the final token:
//                       an inverse-CDF draw over ascending ids from
//                       max(0, p_t - p_d) of the rejected pair, or from p_t
//                       of the bonus row (DFlash / Spec V2 page, A3; DSpark
//                       tutorial, "推测解码的两步流程").
//
// Selection keys: a logit's float bits mapped to an unsigned key that orders
// like the value, in the upper 32 bits, and the complement of the token id in
// the lower 32, so that a larger key means a larger logit or, for equal
// logits, a smaller id.  Keys are unique, so the selected set does not depend
// on the order in which the row is read.
#pragma once

#include "sv_common.cuh"

namespace sv {

constexpr int kMaxK = SV_MAX_FILTER_K;  // 64
constexpr int kCandCap = 288;           // per-warp candidate buffer (31 left over + 256 new)
constexpr int kFilterCtasPerSm = 5;

struct FiltRow {
  int32_t n;       // kept tokens (<= k)
  int32_t argmax;  // lowest id holding the row maximum
  float h;         // reference: x_max * sc
  float z;         // sum of the kept weights
  float xmax;      // row maximum (raw logit)
  int32_t flags;   // device error bits of this row
  int32_t pad[2];
  int32_t ids[kMaxK];  // kept tokens, by (value desc, id asc)
  float w[kMaxK];      // their weights exp2(x sc - h); p = w / z
};
static_assert(sizeof(FiltRow) == 544, "FiltRow layout");

// Order-preserving key of a logit: a larger key is a larger value.  -0 and
// +0 are one value (ties among them go by token id), so -0 is keyed as +0.
__device__ __forceinline__ uint32_t order_key(float x) {
  uint32_t u = __float_as_uint(x);
  u = u == 0x80000000u ? 0u : u;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ float key_value(uint64_t c) {
  const uint32_t k = static_cast<uint32_t>(c >> 32);
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

__device__ __forceinline__ int32_t key_id(uint64_t c) {
  return static_cast<int32_t>(~static_cast<uint32_t>(c));
}

// Sort n (a power of two, <= 2 * 32 * per) keys of a warp's shared buffer in
// descending order (bitonic network; entries >= count must already be 0).
__device__ __forceinline__ void warp_sort_desc(uint64_t* a, int n) {
  const int lane = threadIdx.x & 31;
  for (int k = 2; k <= n; k <<= 1) {
    for (int j = k >> 1; j > 0; j >>= 1) {
      __syncwarp();
      for (int i = lane; i < n; i += 32) {
        const int p = i ^ j;
        if (p > i) {
          const uint64_t x = a[i], y = a[p];
          const bool desc = (i & k) == 0;
          if (desc ? (x < y) : (x > y)) {
            a[i] = y;
            a[p] = x;
          }
        }
      }
    }
  }
  __syncwarp();
}

// Keep the kmax largest of the first `cap` keys of a warp's buffer (sorted,
// descending) and return the new count; entries beyond it are cleared.
__device__ __forceinline__ int warp_prune(uint64_t* cand, int cnt, int kmax, int cap) {
  const int lane = threadIdx.x & 31;
  __syncwarp();
  for (int i = cnt + lane; i < cap; i += 32) cand[i] = 0;
  warp_sort_desc(cand, cap);
  const int keep = min(cnt, kmax);
  for (int i = keep + lane; i < cap; i += 32) cand[i] = 0;
  __syncwarp();
  return keep;
}

// 16-byte read-only load that does not allocate in L1.
__device__ __forceinline__ uint4 ldg_nc_v4(const unsigned char* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// Descending bitonic sort of one key per lane across the warp.
__device__ __forceinline__ uint64_t warp_sort32_desc(uint64_t v) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int k = 2; k <= 32; k <<= 1)
#pragma unroll
    for (int j = k >> 1; j > 0; j >>= 1) {
      const uint64_t o = __shfl_xor_sync(0xffffffffu, v, j);
      const bool desc = (lane & k) == 0;  // every lane at k = 32
      v = (((lane & j) == 0) == desc) ? max(v, o) : min(v, o);
    }
  return v;
}

// The 32 largest keys of two descending lists (one key per lane), descending:
// the element-wise larger of one list and the other reversed is a bitonic
// sequence holding them, sorted by a bitonic merge.
__device__ __forceinline__ uint64_t warp_merge_top32(uint64_t a, uint64_t b) {
  const int lane = threadIdx.x & 31;
  uint64_t c = max(a, __shfl_sync(0xffffffffu, b, 31 - lane));
#pragma unroll
  for (int j = 16; j > 0; j >>= 1) {
    const uint64_t o = __shfl_xor_sync(0xffffffffu, c, j);
    c = (lane & j) == 0 ? max(c, o) : min(c, o);
  }
  return c;
}

// Keys of one queued 16-byte vector (vector index k of the row) that beat the
// bar `thr`, for one lane (valid: the lane holds an entry); NaN and +inf
// are flagged, not kept.  Returns how many of the VEC keys beat the bar.
template <int ES>
__device__ __forceinline__ int vector_keys(const uint4& raw, int32_t k, bool valid, const Slice& s,
                                           uint64_t thr, uint64_t* key, bool& bad) {
  constexpr int VEC = 16 / ES;
  const uint32_t wv[4] = {raw.x, raw.y, raw.z, raw.w};
  const int32_t i0 = k * VEC - s.hoff;
  int c = 0;
#pragma unroll
  for (int l = 0; l < VEC; ++l) {
    const float x = ES == 2 ? ((l & 1) ? bf16hi(wv[l >> 1]) : bf16lo(wv[l >> 1]))
                            : __uint_as_float(wv[l]);
    const int32_t id = i0 + l;
    const bool in = valid && id >= 0 && id < s.len;
    if (in && (x != x || x == INFINITY)) bad = true;
    key[l] = in && !(x != x)
                 ? (static_cast<uint64_t>(order_key(x)) << 32) | static_cast<uint32_t>(~id)
                 : 0ull;
    c += key[l] > thr;
  }
  return c;
}

constexpr int kQCap = 64;  // per-warp queue of vectors that passed the screen

template <int ES>
__global__ void __launch_bounds__(kThreads, kFilterCtasPerSm) filter_rows_kernel(const Params P) {
  constexpr int VEC = 16 / ES;
  __shared__ uint64_t cand[kWarps][kCandCap];
  __shared__ uint64_t merged[kWarps * kMaxK];
  __shared__ __align__(16) uint4 qraw[kWarps][kQCap];  // queued vectors
  __shared__ int32_t qidx[kWarps][kQCap];                // their vector indices
  __shared__ __align__(16) uint64_t bar_sh[kWarps];  // each warp's k-th best key
  __shared__ int bad_any;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const unsigned lt_mask = (1u << lane) - 1u;
  const int K = P.top_k;
  // buffer in use: the smallest power of two that holds k keys plus one
  // vote's worth (32), so that the bar is raised often and stays close to
  // the k-th best key seen so far
  int cap = 64;
  while (cap < K + 32) cap <<= 1;
  int kp = 32;  // the warps' best K, padded to a power of two, for the final merge
  while (kp < K) kp <<= 1;
  FiltRow* recs = reinterpret_cast<FiltRow*>(P.filt);
  const int32_t nrows = P.Nt + P.Nd;
  grid_dep_launch_dependents();

  for (int32_t row = blockIdx.x; row < nrows; row += gridDim.x) {
    const bool is_t = row < P.Nt;
    const unsigned char* base =
        is_t ? P.tgt + static_cast<size_t>(row) * P.V * ES
             : P.drf + static_cast<size_t>(row - P.Nt) * P.V * ES;
    const Slice s = make_slice<ES>(base, P.V, 0, P.V);  // the whole row
    const int32_t nv = s.nbytes >> 4;
    uint64_t* my = cand[warp];
    for (int i = lane; i < kCandCap; i += 32) my[i] = 0;
    if (tid == 0) bad_any = 0;
    if (tid < kWarps) bar_sh[tid] = 0ull;
    __syncthreads();
    int cnt = 0;        // warp-uniform
    uint64_t thr = 0;   // warp-uniform: only larger keys can still make the top k
    float thr_val = -INFINITY;  // the logit of that key (the screen's bar)
    bool bad = false;
    int qn = 0;         // warp-uniform: vectors waiting in the warp's queue
    // k <= 32: the warp's best 32 keys so far, one per lane, descending; new
    // candidates wait in the buffer and merge in 32 at a time
    uint64_t top = 0ull;
    const bool reg_list = K <= 32;

    // Insert the keys of the first n queued vectors (lane l takes entry l):
    // one scan when they all fit, else slot by slot, pruning (keep the best
    // K, raise the bar) whenever a slot would not fit.
    auto drain = [&](int n) {
      const bool valid = lane < n;
      const uint4 raw = valid ? qraw[warp][lane] : make_uint4(0, 0, 0, 0);
      const int32_t k = valid ? qidx[warp][lane] : 0;
      uint64_t key[VEC];
      const int c = vector_keys<ES>(raw, k, valid, s, thr, key, bad);
      const int total = __reduce_add_sync(0xffffffffu, c);
      if (total == 0) return;
      if (reg_list) {
        int pre = c;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int y = __shfl_up_sync(0xffffffffu, pre, o);
          if (lane >= o) pre += y;
        }
        int at = cnt + pre - c;
#pragma unroll
        for (int l = 0; l < VEC; ++l)
          if (key[l] > thr) my[at++] = key[l];
        cnt += total;
        __syncwarp();
        int base = 0;
        for (; cnt - base >= 32; base += 32)
          top = warp_merge_top32(top, warp_sort32_desc(my[base + lane]));
        if (base > 0) {
          // the bar: the k-th best key so far (it is in the list itself)
          const uint64_t kth = __shfl_sync(0xffffffffu, top, K - 1);
          if (kth > thr) {
            thr = kth;
            thr_val = key_value(thr);
            if (lane == 0) bar_sh[warp] = thr;
          }
          const int rest = cnt - base;  // the rest (< 32) to the front
          const uint64_t r = lane < rest ? my[base + lane] : 0ull;
          __syncwarp();
          if (lane < rest) my[lane] = r;
          __syncwarp();
          cnt = rest;
        }
        return;
      }
      if (cnt + total <= cap) {
        int pre = c;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int y = __shfl_up_sync(0xffffffffu, pre, o);
          if (lane >= o) pre += y;
        }
        int at = cnt + pre - c;
#pragma unroll
        for (int l = 0; l < VEC; ++l)
          if (key[l] > thr) my[at++] = key[l];
        cnt += total;
        return;
      }
#pragma unroll
      for (int l = 0; l < VEC; ++l) {
        bool take = key[l] > thr;
        unsigned m = __ballot_sync(0xffffffffu, take);
        if (!m) continue;
        if (cnt + __popc(m) > cap) {
          cnt = warp_prune(my, cnt, K, cap);
          if (cnt >= K && my[K - 1] > thr) {
            thr = my[K - 1];
            thr_val = key_value(thr);
            if (lane == 0) bar_sh[warp] = thr;
          }
          take = key[l] > thr;
          m = __ballot_sync(0xffffffffu, take);
        }
        if (take) my[cnt + __popc(m & lt_mask)] = key[l];
        cnt += __popc(m);
      }
    };

    // the loop runs on the warp's first vector, so that every lane takes
    // part in the warp-wide votes below; lanes past the end hold no element;
    // each step loads the next step's vector before screening its own
    int32_t kw = warp * 32;
    uint4 nxt = kw + lane < nv ? ldg_nc_v4(s.gsrc + 16 * static_cast<size_t>(kw + lane))
                               : make_uint4(0, 0, 0, 0);
    // a first bar before any prune (k <= 32): just below the k-th largest of
    // the lanes' first-vector maximum keys.  At least k keys of the row are
    // above it (those maxima), so no key at or below it can be among the
    // best k.
    if (K <= 32) {
      uint64_t key[VEC];
      bool seed_bad = false;
      vector_keys<ES>(nxt, kw + lane, kw + lane < nv, s, 0ull, key, seed_bad);
      uint64_t mk = key[0];
#pragma unroll
      for (int l = 1; l < VEC; ++l) mk = max(mk, key[l]);
      int above = 0;  // lanes whose maximum key is larger than this lane's
#pragma unroll 8
      for (int o = 0; o < 32; ++o) above += __shfl_sync(0xffffffffu, mk, o) > mk;
      // the lane of rank k - 1 holds the k-th largest (keys are unique; lanes
      // past the row hold 0, which never seeds)
      const unsigned r = __ballot_sync(0xffffffffu, above == K - 1 && mk != 0ull);
      if (r) {
        // one below that key, so that the maximum itself still enters the
        // buffer (the low half, a complemented id, is never zero: the value
        // half is unchanged)
        thr = __shfl_sync(0xffffffffu, mk, __ffs(r) - 1) - 1ull;
        thr_val = key_value(thr);
        if (lane == 0) bar_sh[warp] = thr;
      }
    }
    int step = 0;
    for (; kw < nv; kw += kThreads) {
      const int32_t k = kw + lane;
      const uint4 raw = nxt;
      if (kw + kThreads < nv)
        nxt = k + kThreads < nv ? ldg_nc_v4(s.gsrc + 16 * static_cast<size_t>(k + kThreads))
                                : make_uint4(0, 0, 0, 0);
      // any warp's k-th best key bars the whole CTA: an element below it
      // cannot be among the CTA's k best, so the highest of them is used
      // (read every eighth step: a stale bar only lets more vectors through)
      if ((++step & 7) == 0) {
        uint64_t b = thr;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) b = max(b, bar_sh[w]);
        if (b > thr) {
          thr = b;
          thr_val = key_value(b);
        }
      }
      // screen: a vector whose largest logit is below the bar holds no
      // candidate (a NaN maximum is queued and flagged); bf16 vectors take
      // their maximum on the packed pairs
      float vm;
      if (ES == 2) {
        const uint32_t m2 = bf16x2_max_nan(bf16x2_max_nan(raw.x, raw.y), bf16x2_max_nan(raw.z, raw.w));
        vm = fmax_nan(bf16lo(m2), bf16hi(m2));
      } else {
        vm = fmax_nan(fmax_nan(__uint_as_float(raw.x), __uint_as_float(raw.y)),
                      fmax_nan(__uint_as_float(raw.z), __uint_as_float(raw.w)));
      }
      const bool maybe = k < nv && !(vm < thr_val);
      const unsigned mq = __ballot_sync(0xffffffffu, maybe);
      if (mq == 0) continue;
      // queue the vectors that passed; keys are formed once 32 are waiting
      if (maybe) {
        const int at = qn + __popc(mq & lt_mask);
        qraw[warp][at] = raw;
        qidx[warp][at] = k;
      }
      qn += __popc(mq);
      __syncwarp();
      if (qn >= 32) {
        drain(32);
        // move the rest (at most 31) to the front
        const int rest = qn - 32;
        uint4 r4;
        int32_t ri = 0;
        if (lane < rest) {
          r4 = qraw[warp][32 + lane];
          ri = qidx[warp][32 + lane];
        }
        __syncwarp();
        if (lane < rest) {
          qraw[warp][lane] = r4;
          qidx[warp][lane] = ri;
        }
        __syncwarp();
        qn = rest;
      }
    }
    if (qn > 0) drain(qn);
    if (reg_list) {
      top = warp_merge_top32(top, warp_sort32_desc(lane < cnt ? my[lane] : 0ull));
      merged[warp * kp + lane] = lane < K ? top : 0ull;  // kp = 32
    } else {
      cnt = warp_prune(my, cnt, K, cap);
      for (int i = lane; i < kp; i += 32) merged[warp * kp + i] = i < K ? my[i] : 0ull;
    }
    if (__any_sync(0xffffffffu, bad) && lane == 0) atomicOr(&bad_any, 1);
    __syncthreads();
    if (reg_list) {
      // the CTA's best 32: warp 0 folds the warps' sorted lists together
      if (warp == 0) {
        uint64_t t = merged[lane];
#pragma unroll
        for (int w = 1; w < kWarps; ++w) t = warp_merge_top32(t, merged[w * 32 + lane]);
        merged[lane] = t;
        merged[32 + lane] = 0ull;
        __syncwarp();
      }
    } else {
    // the CTA's best K of the warps' best K: bitonic sort of kWarps * kp keys
      const int NM = kWarps * kp;
      for (int kk = 2; kk <= NM; kk <<= 1) {
        for (int j = kk >> 1; j > 0; j >>= 1) {
          for (int i = tid; i < NM; i += kThreads) {
            const int p = i ^ j;
            if (p > i) {
              const uint64_t a = merged[i], b = merged[p];
              const bool desc = (i & kk) == 0;
              if (desc ? (a < b) : (a > b)) {
                merged[i] = b;
                merged[p] = a;
              }
            }
          }
          __syncthreads();
        }
      }
    }
    if (warp == 0) {
      // weights of the k best relative to the maximum, then the top-p cut
      FiltRow* fr = recs + row;
      const float sc = P.sc;
      const uint64_t c0 = merged[lane], c1 = merged[lane + 32];
      const float xmax = key_value(merged[0]);
      const float h = xmax * sc;
      const bool v0 = lane < K && c0 != 0ull, v1 = lane + 32 < K && c1 != 0ull;
      const float x0 = v0 ? key_value(c0) : 0.f, x1 = v1 ? key_value(c1) : 0.f;
      const float w0 = v0 ? ex2(fmaf(x0, sc, -h)) : 0.f;
      const float w1 = v1 ? ex2(fmaf(x1, sc, -h)) : 0.f;
      const int navail = __popc(__ballot_sync(0xffffffffu, v0)) + __popc(__ballot_sync(0xffffffffu, v1));
      // inclusive prefix sums in (value desc, id asc) order: entries 0..31, then 32..63
      float p0 = w0, p1 = w1;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const float a = __shfl_up_sync(0xffffffffu, p0, off);
        const float b = __shfl_up_sync(0xffffffffu, p1, off);
        if (lane >= off) p0 += a, p1 += b;
      }
      const float half = __shfl_sync(0xffffffffu, p0, 31);
      p1 += half;
      const float zk = __shfl_sync(0xffffffffu, p1, 31);  // sum of the k weights
      int n = navail;
      if (P.top_p < 1.f) {
        // shortest prefix whose cumulative probability reaches top_p
        const unsigned r0 = __ballot_sync(0xffffffffu, v0 && p0 / zk >= P.top_p);
        const unsigned r1 = __ballot_sync(0xffffffffu, v1 && p1 / zk >= P.top_p);
        if (r0) n = __ffs(r0);
        else if (r1) n = 32 + __ffs(r1);
      }
      float z = n > 32 ? __shfl_sync(0xffffffffu, p1, (n - 33) & 31)
                       : __shfl_sync(0xffffffffu, p0, (n - 1) & 31);
      if (n == 0) z = 0.f;
      if (lane < n) {
        fr->ids[lane] = key_id(c0);
        fr->w[lane] = w0;
      }
      if (lane + 32 < n) {
        fr->ids[lane + 32] = key_id(c1);
        fr->w[lane + 32] = w1;
      }
      const bool row_bad = bad_any != 0 || !(xmax > -INFINITY);
      if (lane == 0) {
        fr->n = n;
        fr->argmax = key_id(merged[0]);
        fr->h = h;
        fr->z = z;
        fr->xmax = xmax;
        fr->flags = row_bad ? SV_DEVERR_NAN : 0;
        if (row_bad) raise_error(P, SV_DEVERR_NAN);
        if (P.out_row_stats != nullptr) {
          float* o = P.out_row_stats + 3 * static_cast<size_t>(row);  // targets, then drafts
          o[0] = xmax / P.T;
          o[1] = z * exp2f(h - xmax * sc);
          o[2] = __int_as_float(key_id(merged[0]));
        }
      }
    }
    __syncthreads();
  }
}

// Probability of token v in a kept set held in shared memory (0 if absent).
__device__ __forceinline__ float kept_prob(const FiltRow& r, int32_t v) {
  for (int i = 0; i < r.n; ++i)
    if (r.ids[i] == v) return r.w[i] / r.z;
  return 0.f;
}

__device__ __forceinline__ void copy_row(FiltRow& dst, const FiltRow* src, int lane) {
  const int4* s = reinterpret_cast<const int4*>(src);
  int4* d = reinterpret_cast<int4*>(&dst);
  for (int i = lane; i < static_cast<int>(sizeof(FiltRow) / 16); i += 32) d[i] = s[i];
  __syncwarp();
}

// One warp per request: accept chain, labels, final token, outputs.
__global__ void __launch_bounds__(kThreads) filter_requests_kernel(const Params P) {
  __shared__ FiltRow rows[kWarps][2];  // target row, draft row of the current position
  __shared__ int32_t draw_id[kWarps][kMaxK];
  __shared__ float draw_w[kWarps][kMaxK];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int32_t r = blockIdx.x * kWarps + warp;
  if (r >= P.B) return;  // whole warps leave together
  const FiltRow* recs = reinterpret_cast<const FiltRow*>(P.filt);
  FiltRow& T = rows[warp][0];
  FiltRow& D = rows[warp][1];
  const int32_t off = __ldg(P.offs + r), off1 = __ldg(P.offs + r + 1), ell = __ldg(P.lens + r);
  const bool ok = ell >= 1 && ell <= P.max_len && off1 - off == ell && off >= r && off1 <= P.Nt &&
                  (r != 0 || off == 0) && (r != P.B - 1 || off1 == P.Nt) &&
                  off - r + ell - 1 <= P.Nd;
  if (!ok) {
    if (lane == 0) raise_error(P, SV_DEVERR_LEN);
    return;
  }
  grid_dep_wait();  // the row records come from filter_rows_kernel
  int flags = 0;
  // labels of every drafted position, and the accept chain up to the first failure
  int32_t a = ell - 1;
  bool stopped = false;
  for (int32_t j = 0; j < ell - 1; ++j) {
    copy_row(T, recs + off + j, lane);
    copy_row(D, recs + P.Nt + off - r + j, lane);
    if (lane == 0) flags |= T.flags | D.flags;
    const int32_t x = __ldg(P.draft_tokens + off - r + j);
    if (P.out_conf != nullptr) {
      float c = 0.f;
      for (int i = lane; i < T.n; i += 32) c += fminf(T.w[i] / T.z, kept_prob(D, T.ids[i]));
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) c += __shfl_xor_sync(0xffffffffu, c, o);
      if (lane == 0) P.out_conf[off - r + j] = c;
    }
    if (stopped) continue;
    bool acc;
    if (x < 0 || x >= P.V) {
      flags |= SV_DEVERR_TOKEN;
      acc = false;
    } else if (P.mode == SV_GREEDY) {
      acc = x == T.argmax;
    } else {
      const float pt = kept_prob(T, x), pd = kept_prob(D, x);
      const float u = __ldg(P.uniforms + off + j);
      acc = pd > 0.f ? u * pd < pt : pt > 0.f;
    }
    if (!acc) {
      a = j;
      stopped = true;
      if (P.out_conf == nullptr) break;
    }
  }
  // final token from target row a (and its draft partner when a < l - 1)
  copy_row(T, recs + off + a, lane);
  if (lane == 0) flags |= T.flags;
  int32_t final_tok = T.argmax;
  if (P.mode == SV_SAMPLE) {
    const bool residual = a < ell - 1;
    if (residual) copy_row(D, recs + P.Nt + off - r + a, lane);
    // weights of the kept target tokens, then sorted by id (ascending)
    int32_t* sid = draw_id[warp];
    float* swt = draw_w[warp];
    float tot = 0.f;
    for (int q = 0; q < 2; ++q) {
      const int i = lane + 32 * q;
      const int32_t v = i < T.n ? T.ids[i] : 0x7fffffff;
      const float pt = i < T.n ? T.w[i] / T.z : 0.f;
      const float w = residual ? fmaxf(0.f, pt - kept_prob(D, v)) : pt;
      sid[i] = v;
      swt[i] = w;
      tot += w;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) tot += __shfl_xor_sync(0xffffffffu, tot, o);
    if (residual && !(tot > 0.f)) {  // no residual mass (rounding only): draw from p_t
      tot = 0.f;
      for (int q = 0; q < 2; ++q) {
        const int i = lane + 32 * q;
        swt[i] = i < T.n ? T.w[i] / T.z : 0.f;
        tot += swt[i];
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) tot += __shfl_xor_sync(0xffffffffu, tot, o);
    }
    for (int kk = 2; kk <= kMaxK; kk <<= 1) {  // bitonic, ascending ids
      for (int jj = kk >> 1; jj > 0; jj >>= 1) {
        __syncwarp();
        for (int i = lane; i < kMaxK; i += 32) {
          const int pj = i ^ jj;
          if (pj > i) {
            const bool up = (i & kk) == 0;
            if (up ? sid[i] > sid[pj] : sid[i] < sid[pj]) {
              const int32_t ti = sid[i]; sid[i] = sid[pj]; sid[pj] = ti;
              const float tw = swt[i]; swt[i] = swt[pj]; swt[pj] = tw;
            }
          }
        }
      }
    }
    __syncwarp();
    // inverse CDF over ascending ids: first token with cumsum > u * total
    // (lane l holds entries 2l and 2l + 1)
    const float w0 = swt[2 * lane], w1 = swt[2 * lane + 1];
    const float ls = w0 + w1;
    float incl = ls;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    const float c0 = incl - ls + w0, c1 = incl;
    const float target = __ldg(P.uniforms + off + ell - 1) * tot;
    const bool h0 = w0 > 0.f && c0 > target, h1 = w1 > 0.f && c1 > target;
    const unsigned hit = __ballot_sync(0xffffffffu, h0 || h1);
    const unsigned pos = __ballot_sync(0xffffffffu, w0 > 0.f || w1 > 0.f);
    int e = -1;
    if (hit) {
      const int L = __ffs(hit) - 1;
      e = 2 * L + (__shfl_sync(0xffffffffu, h0, L) ? 0 : 1);
    } else if (pos) {  // rounding: the last token with mass
      const int L = 31 - __clz(pos);
      e = 2 * L + (__shfl_sync(0xffffffffu, w1 > 0.f, L) ? 1 : 0);
    }
    if (e >= 0) final_tok = sid[e];
    else flags |= SV_DEVERR_NAN;
  }
  for (int32_t j = lane; j < ell; j += 32) {
    int32_t v = -1;
    if (j < a) v = __ldg(P.draft_tokens + off - r + j);
    else if (j == a) v = final_tok;
    P.out_tokens[off + j] = v;
  }
  flags = __reduce_or_sync(0xffffffffu, flags);
  if (lane == 0) {
    P.out_accept_len[r] = a;
    if (flags) raise_error(P, flags);
  }
}

}  // namespace sv
