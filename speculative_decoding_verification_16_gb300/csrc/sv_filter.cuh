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
//  filter_requests_kernel  one CTA per request, a warp per drafted
//                       position, on the FiltRow records only:
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
constexpr int kCandCap = 288;           // per-warp staged keys (31 left over + 256 new)
constexpr int kQCap = 64;               // per-warp queue of vectors that passed the screen
// The row streams through shared memory: each warp copies chunks of
// kFilterChunk 16-byte vectors (cp.async.bulk) into its own ring of
// kFilterStages stages, so the bytes in flight per SM are set by the ring,
// not by registers.
constexpr int kFilterChunk = 256;
constexpr int kFilterStages = 2;
constexpr int kFilterCtasPerSm = 2;
constexpr int kFilterRingBytes = kWarps * kFilterStages * kFilterChunk * 16;
// kWarps streaming warps and one finisher warp
constexpr int kFiltThreads = (kWarps + 1) * 32;
// named barriers (0 is __syncthreads): lists of row parity p complete, and
// the per-row state of parity p clear again
constexpr int kBarListsFull = 1;
constexpr int kBarSetFree = 3;

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

// Sort a bitonic sequence of keys (one per lane) into descending order.
__device__ __forceinline__ uint64_t warp_bitonic_desc(uint64_t c) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int j = 16; j > 0; j >>= 1) {
    const uint64_t o = __shfl_xor_sync(0xffffffffu, c, j);
    c = (lane & j) == 0 ? max(c, o) : min(c, o);
  }
  return c;
}

// The 32 largest keys of two descending lists (one key per lane), descending:
// the element-wise larger of one list and the other reversed is a bitonic
// sequence holding them.
__device__ __forceinline__ uint64_t warp_merge_top32(uint64_t a, uint64_t b) {
  return warp_bitonic_desc(max(a, __shfl_sync(0xffffffffu, b, 31 - (threadIdx.x & 31))));
}

// A warp's best keys so far, descending: ranks 0..31 in hi (lane i holds
// rank i) and, when more than 32 are kept (TWO), ranks 32..63 in lo.
// Empty ranks hold 0, which is below every key.
struct TopList {
  uint64_t hi, lo;
};

// Merge 32 keys (one per lane, descending) into the list.
template <bool TWO>
__device__ __forceinline__ void list_insert(TopList& t, uint64_t c) {
  const uint64_t cr = __shfl_sync(0xffffffffu, c, 31 - (threadIdx.x & 31));
  if (!TWO) {
    t.hi = warp_bitonic_desc(max(t.hi, cr));
    return;
  }
  // every lo key is below every hi key, so the best 32 of hi and c are the
  // best 32 overall; the other 32 of them compete with lo for ranks 32..63
  const uint64_t up = max(t.hi, cr), down = min(t.hi, cr);
  t.hi = warp_bitonic_desc(up);
  t.lo = warp_merge_top32(t.lo, warp_bitonic_desc(down));
}

// a := the best 32 (64 with TWO) keys of the lists a and b.
template <bool TWO>
__device__ __forceinline__ void list_merge(TopList& a, const TopList& b) {
  if (!TWO) {
    a.hi = warp_merge_top32(a.hi, b.hi);
    return;
  }
  // element i of a against element 63 - i of b: the larger ones form a
  // bitonic sequence of 64 holding the best 64; its first merge stage pairs
  // rank i with rank i + 32, then each half is bitonic
  const int rev = 31 - (threadIdx.x & 31);
  const uint64_t ch = max(a.hi, __shfl_sync(0xffffffffu, b.lo, rev));
  const uint64_t cl = max(a.lo, __shfl_sync(0xffffffffu, b.hi, rev));
  a.hi = warp_bitonic_desc(max(ch, cl));
  a.lo = warp_bitonic_desc(min(ch, cl));
}

// The key of rank j (0-based, warp-uniform, j < 32 or, with TWO, j < 64).
template <bool TWO>
__device__ __forceinline__ uint64_t list_rank(const TopList& t, int j) {
  if (TWO && j >= 32) return __shfl_sync(0xffffffffu, t.lo, j - 32);
  return __shfl_sync(0xffffffffu, t.hi, j & 31);
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

// Largest logit of one 16-byte vector, NaN if any element is NaN (bf16
// vectors take the maximum on the packed pairs first).
template <int ES>
__device__ __forceinline__ float vec_max(const uint4& v) {
  if (ES == 2) {
    const uint32_t m2 = bf16x2_max_nan(bf16x2_max_nan(v.x, v.y), bf16x2_max_nan(v.z, v.w));
    return fmax_nan(bf16lo(m2), bf16hi(m2));
  }
  return fmax_nan(fmax_nan(__uint_as_float(v.x), __uint_as_float(v.y)),
                  fmax_nan(__uint_as_float(v.z), __uint_as_float(v.w)));
}

// Largest logit of N vectors, NaN if any element is NaN.
template <int ES, int N>
__device__ __forceinline__ float vecs_max(const uint4 (&v)[N]) {
  if (ES == 2) {
    uint32_t m2 = bf16x2_max_nan(bf16x2_max_nan(v[0].x, v[0].y), bf16x2_max_nan(v[0].z, v[0].w));
#pragma unroll
    for (int i = 1; i < N; ++i)
      m2 = bf16x2_max_nan(m2, bf16x2_max_nan(bf16x2_max_nan(v[i].x, v[i].y),
                                             bf16x2_max_nan(v[i].z, v[i].w)));
    return fmax_nan(bf16lo(m2), bf16hi(m2));
  }
  float m = vec_max<ES>(v[0]);
#pragma unroll
  for (int i = 1; i < N; ++i) m = fmax_nan(m, vec_max<ES>(v[i]));
  return m;
}


// The finisher warp's part of a row: fold the streaming warps' lists into
// the CTA's best keys, then the weights of the k best relative to the
// maximum, the top-p cut and the row's FiltRow record.  flagged: a warp saw
// a NaN or +inf.
template <bool TWO>
__device__ __forceinline__ void finish_row(const Params& P, int32_t row, const uint64_t (*lists)[64],
                                           bool flagged) {
  const int lane = threadIdx.x & 31;
  const int K = P.top_k;
  FiltRow* recs = reinterpret_cast<FiltRow*>(P.filt);
  TopList t{lists[0][lane], TWO ? lists[0][32 + lane] : 0ull};
#pragma unroll 1
  for (int w = 1; w < kWarps; ++w)
    list_merge<TWO>(t, TopList{lists[w][lane], TWO ? lists[w][32 + lane] : 0ull});
  // weights of the k best relative to the maximum, then the top-p cut
  FiltRow* fr = recs + row;
  const float sc = P.sc;
  const uint64_t c0 = t.hi, c1 = TWO ? t.lo : 0ull;
  const uint64_t best = __shfl_sync(0xffffffffu, c0, 0);
  const float xmax = key_value(best);
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
  const bool row_bad = flagged || !(xmax > -INFINITY);
  if (lane == 0) {
    fr->n = n;
    fr->argmax = key_id(best);
    fr->h = h;
    fr->z = z;
    fr->xmax = xmax;
    fr->flags = row_bad ? SV_DEVERR_NAN : 0;
    if (row_bad) raise_error(P, SV_DEVERR_NAN);
    if (P.out_row_stats != nullptr) {
      float* o = P.out_row_stats + 3 * static_cast<size_t>(row);  // targets, then drafts
      o[0] = xmax / P.T;
      o[1] = z * exp2f(h - xmax * sc);
      o[2] = __int_as_float(key_id(best));
    }
  }
}

// filter_rows_kernel: the k best keys of each row, k <= 32 (TWO false) or
// k <= 64 (TWO true), one CTA per row at a time.
//
// Eight streaming warps each take chunks warp, warp + 8, ... of the row,
// copied into the warp's shared-memory ring, and screen them against a bar:
// a key at or below it cannot be among the row's k best.  Vectors that pass
// wait in a per-warp queue; 32 at a time become keys, those above the bar
// are staged, and staged keys merge 32 at a time (bitonic sort, then a
// bitonic merge) into the warp's register list of its best keys.  Every bar
// used is valid because at least k keys of the row lie above it:
//  - a warp's own k-th best key;
//  - the m-th largest of the warps' published rank-r keys (r = ceil(k / 8),
//    m = ceil(k / r)): m warps each hold r keys at or above it, m r >= k
//    keys in all, and the warps' keys are distinct elements of the row;
//  - from the first chunk on, the same two with the lanes' maxima over the
//    chunk standing in for the list (k-th largest: the warp's own, k <= 32;
//    r-th largest: the key it publishes).
// Bars are shared through a word in shared memory.  At the end of the row
// the streaming warps hand their lists to a ninth, finisher warp and go on
// with the next row while it folds them and writes the row's record.
template <int ES, bool TWO>
__global__ void __launch_bounds__(kFiltThreads, kFilterCtasPerSm) filter_rows_kernel(const Params P) {
  constexpr int VEC = 16 / ES;
  constexpr int CH = kFilterChunk, NS = kFilterStages, VPL = CH / 32;
  extern __shared__ __align__(128) unsigned char ring[];  // [kWarps][NS][CH * 16]: copies
  // per-row state, two sets (row parity): the streaming warps work on one
  // row while the finisher still reads the other
  __shared__ uint64_t lists[2][kWarps][64];  // the warps' lists, at the end of a row
  __shared__ uint64_t cand[kWarps][kCandCap];  // staged keys, per warp
  __shared__ __align__(16) uint4 qraw[kWarps][kQCap];  // queued vectors
  __shared__ int32_t qidx[kWarps][kQCap];                // their vector indices
  __shared__ __align__(8) uint64_t full_bar[kWarps][NS];  // one per copy stage
  __shared__ uint64_t pub[2][kWarps];  // each warp's key of rank r - 1 (0: fewer than r)
  __shared__ uint64_t cta_bar[2];      // the best bar any warp has found
  __shared__ int bad_any[2];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const unsigned lt_mask = (1u << lane) - 1u;
  const int K = P.top_k;
  const int r = (K + kWarps - 1) / kWarps;  // 1..8
  const int m = (K + r - 1) / r;            // <= kWarps
  const int32_t nrows = P.Nt + P.Nd;
  if (lane == 0 && warp < kWarps)
    for (int s = 0; s < NS; ++s) mbar_init(smem_addr(&full_bar[warp][s]), 1);
  if (tid < 2) {
    cta_bar[tid] = 0ull;
    bad_any[tid] = 0;
  }
  if (tid < 2 * kWarps) pub[tid / kWarps][tid % kWarps] = 0ull;
  fence_mbar_init();
  __syncthreads();
  grid_dep_launch_dependents();

  if (warp == kWarps) {
    // the finisher: row t's lists are complete once every streaming warp has
    // arrived on kBarListsFull + (t & 1); it then clears that set for the
    // CTA's row t + 2 and releases it on kBarSetFree + (t & 1)
    int t = 0;
    for (int32_t row = blockIdx.x; row < nrows; row += gridDim.x, ++t) {
      const int b = t & 1;
      named_bar_sync(kBarListsFull + b, kFiltThreads);
      finish_row<TWO>(P, row, lists[b], bad_any[b] != 0);
      if (row + 2 * static_cast<int32_t>(gridDim.x) < nrows) {
        if (lane < kWarps) pub[b][lane] = 0ull;
        if (lane == 0) {
          cta_bar[b] = 0ull;
          bad_any[b] = 0;
        }
        __threadfence_block();
        named_bar_arrive(kBarSetFree + b, kFiltThreads);
      }
    }
    return;
  }
  unsigned char* my_ring = ring + warp * NS * CH * 16;

  auto row_slice = [&](int32_t row) {
    const unsigned char* base = row < P.Nt ? P.tgt + static_cast<size_t>(row) * P.V * ES
                                           : P.drf + static_cast<size_t>(row - P.Nt) * P.V * ES;
    return make_slice<ES>(base, P.V, 0, P.V);  // the whole row
  };
  // chunks (CH vectors, the last one shorter) of a row of nv vectors that
  // this warp takes: warp, warp + kWarps, ...
  auto warp_chunks = [&](int32_t nv) {
    const int32_t nch = (nv + CH - 1) / CH;
    return nch > warp ? (nch - warp + kWarps - 1) / kWarps : 0;
  };

  // The warp's copies form one stream over the CTA's rows: lane 0 keeps NS
  // of them in flight and, each time the warp has read a stage, refills it
  // with the next chunk of the stream (the next row's, near a row's end).
  int32_t p_row = blockIdx.x, p_i = 0, p_nch = 0, p_nbytes = 0;
  const unsigned char* p_src = nullptr;
  uint32_t pseq = 0, cseq = 0;  // copies issued / consumed by this warp
  bool timed_out = false;       // a copy never arrived: stop issuing, skip work
  auto p_open = [&]() {         // the first row from p_row on with a chunk for this warp
    for (; p_row < nrows; p_row += gridDim.x) {
      const Slice ps = row_slice(p_row);
      p_nch = warp_chunks(ps.nbytes >> 4);
      if (p_nch > 0) {
        p_src = ps.gsrc;
        p_nbytes = ps.nbytes;
        p_i = 0;
        return;
      }
    }
  };
  auto issue = [&]() {
    if (p_row >= nrows || timed_out) return;
    const int32_t off = (warp + kWarps * p_i) * CH * 16;
    const uint32_t bytes = static_cast<uint32_t>(min(CH * 16, p_nbytes - off));  // 16 | bytes
    const int stg = static_cast<int>(pseq % NS);
    if (lane == 0) {
      const uint32_t bar = smem_addr(&full_bar[warp][stg]);
      mbar_arrive_expect_tx(bar, bytes);
      bulk_g2s(smem_addr(my_ring + stg * CH * 16), p_src + off, bytes, bar);
    }
    ++pseq;
    if (++p_i == p_nch) {
      p_row += gridDim.x;
      p_open();
    }
  };
  p_open();
  for (int s = 0; s < NS; ++s) issue();

  int t = 0;
  for (int32_t row = blockIdx.x; row < nrows; row += gridDim.x, ++t) {
    const int b = t & 1;
    if (t >= 2) named_bar_sync(kBarSetFree + b, kFiltThreads);  // set b is clear again
    const Slice s = row_slice(row);
    const int32_t nv = s.nbytes >> 4;
    uint64_t* my = cand[warp];
    int cnt = 0;                // warp-uniform: staged keys
    int qn = 0;                 // warp-uniform: vectors waiting in the warp's queue
    uint64_t pubv = 0;          // warp-uniform: this warp's published key
    uint64_t thr = 0;           // warp-uniform: the bar
    float thr_val = -INFINITY;  // the logit of that key (the screen's bar)
    bool bad = false;
    TopList top{0ull, 0ull};

    // adopt a bar (warp-uniform) and share it with the CTA
    auto raise_to = [&](uint64_t nb) {
      if (nb > thr) {
        thr = nb;
        thr_val = key_value(nb);
        if (lane == 0) atomicMax(reinterpret_cast<unsigned long long*>(&cta_bar[b]), nb);
      }
    };
    // publish a key with at least r of this warp's elements at or above it
    // (the largest so far: every one published stays true)
    auto publish = [&](uint64_t key) {
      if (key > pubv) {
        pubv = key;
        if (lane == 0) pub[b][warp] = key;
      }
    };
    // the m-th largest of the warps' published keys, less one
    auto cta_combined = [&]() {
      __syncwarp();
      const uint64_t v = lane < kWarps ? *reinterpret_cast<volatile uint64_t*>(&pub[b][lane]) : 0ull;
      int gt = 0, ge = 0;
#pragma unroll
      for (int j = 0; j < kWarps; ++j) {
        const uint64_t o = __shfl_sync(0xffffffffu, v, j);
        gt += o > v;
        ge += o >= v;
      }
      const unsigned sel = __ballot_sync(0xffffffffu, lane < kWarps && gt < m && m <= ge);
      const uint64_t q = sel ? __shfl_sync(0xffffffffu, v, __ffs(sel) - 1) : 0ull;
      if (q > 0ull) raise_to(q - 1ull);
    };
    // after the list changed: the warp's k-th best key, its rank-r key
    // published, and the combination
    auto list_bars = [&]() {
      raise_to(list_rank<TWO>(top, K - 1));
      publish(list_rank<TWO>(top, r - 1));
      cta_combined();
    };

    // Keys of the first n queued vectors (lane l takes entry l) that beat
    // the bar go to the staging buffer; full groups of 32 merge into the list.
    auto drain = [&](int n) {
      const bool valid = lane < n;
      const uint4 raw = valid ? qraw[warp][lane] : make_uint4(0, 0, 0, 0);
      const int32_t k = valid ? qidx[warp][lane] : 0;
      uint64_t key[VEC];
      const int c = vector_keys<ES>(raw, k, valid, s, thr, key, bad);
      const int total = __reduce_add_sync(0xffffffffu, c);
      if (total == 0) return;
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
      cnt += total;  // < 32 + 32 VEC <= kCandCap
      __syncwarp();
      if (cnt < 32) return;
      int done = 0;
      for (; cnt - done >= 32; done += 32) list_insert<TWO>(top, warp_sort32_desc(my[done + lane]));
      const int rest = cnt - done;  // the rest (< 32) to the front
      const uint64_t rk = lane < rest ? my[done + lane] : 0ull;
      __syncwarp();
      if (lane < rest) my[lane] = rk;
      __syncwarp();
      cnt = rest;
      list_bars();
    };

    const int32_t mych = timed_out ? 0 : warp_chunks(nv);
    for (int32_t i = 0; i < mych; ++i) {
      const int stg = static_cast<int>(cseq % NS);
      mbar_wait(smem_addr(&full_bar[warp][stg]), (cseq / NS) & 1u, timed_out);
      timed_out = __any_sync(0xffffffffu, timed_out);  // lanes may see the limit apart
      if (timed_out) break;
      const int32_t kbase = (warp + kWarps * i) * CH;  // the chunk's first vector
      const unsigned char* buf = my_ring + stg * CH * 16;
      uint4 v[VPL];  // lane's vectors kbase + lane + 32 t (stale past the row's end)
#pragma unroll
      for (int t = 0; t < VPL; ++t) v[t] = *reinterpret_cast<const uint4*>(buf + 16 * (lane + 32 * t));
      const float vm = vecs_max<ES, VPL>(v);
      if (i == 0 && kbase + CH <= nv) {
        // first bars from the lanes' maxima over this chunk (NaN maxima
        // count as -inf): with x the j-th largest of them, j distinct
        // elements have values at or above x, so their keys are at or above
        // order_key(x) << 32.  j = k gives this warp's own bar (k <= 32),
        // j = r the key it publishes.
        const float mx = vm == vm ? vm : -INFINITY;
        int gt = 0, ge = 0;
#pragma unroll 8
        for (int o = 0; o < 32; ++o) {
          const float y = __shfl_sync(0xffffffffu, mx, o);
          gt += y > mx;
          ge += y >= mx;
        }
        if (!TWO) {
          const unsigned sk = __ballot_sync(0xffffffffu, gt < K && K <= ge);
          const float x = __shfl_sync(0xffffffffu, mx, sk ? __ffs(sk) - 1 : 0);
          if (sk && x > -INFINITY) raise_to((static_cast<uint64_t>(order_key(x)) << 32) - 1ull);
        }
        const unsigned sr = __ballot_sync(0xffffffffu, gt < r && r <= ge);
        const float xr = __shfl_sync(0xffffffffu, mx, sr ? __ffs(sr) - 1 : 0);
        if (sr && xr > -INFINITY) publish(static_cast<uint64_t>(order_key(xr)) << 32);
      }
      // the best bar any warp has found (a stale one only lets more through)
      const uint64_t cb = *reinterpret_cast<volatile uint64_t*>(&cta_bar[b]);
      if (cb > thr) {
        thr = cb;
        thr_val = key_value(cb);
      }
      // screen: no logit of the chunk reaches the bar (stale entries past the
      // row's end only make the test pass more often)
      if (__ballot_sync(0xffffffffu, !(vm < thr_val)) != 0) {
        // queue each vector whose largest logit is not below the bar (a NaN
        // maximum is queued and flagged by the drain)
#pragma unroll 1
        for (int t = 0; t < VPL; ++t) {
          const int32_t k = kbase + lane + 32 * t;
          const uint4 raw = *reinterpret_cast<const uint4*>(buf + 16 * (lane + 32 * t));
          const bool maybe = k < nv && !(vec_max<ES>(raw) < thr_val);
          const unsigned mq = __ballot_sync(0xffffffffu, maybe);
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
      }
      __syncwarp();  // every lane has read the stage: refill it
      ++cseq;
      issue();
    }
    if (qn > 0) drain(qn);
    if (cnt > 0) list_insert<TWO>(top, warp_sort32_desc(lane < cnt ? my[lane] : 0ull));
    lists[b][warp][lane] = top.hi;
    if (TWO) lists[b][warp][32 + lane] = top.lo;
    if (__any_sync(0xffffffffu, bad) && lane == 0) atomicOr(&bad_any[b], 1);
    __threadfence_block();
    named_bar_arrive(kBarListsFull + b, kFiltThreads);  // the lists go to the finisher
  }
  if (timed_out) {
    // a copy did not arrive in time: report it, and before the CTA exits
    // wait (bounded) for every copy still in flight into its shared memory
    if (lane == 0) raise_error(P, SV_DEVERR_TIMEOUT);
    bool again = false;
    for (; cseq < pseq; ++cseq)
      mbar_wait(smem_addr(&full_bar[warp][cseq % NS]), (cseq / NS) & 1u, again);
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

// filter_requests_kernel: one CTA per request, kReqWarps warps.  Warp w
// takes drafted positions w, w + kReqWarps, ...: it copies the pair of row
// records, writes the label and records a rejection (the first one is
// kept); warp 0 then draws the final token from the rows of the first
// rejected position (or the bonus row) and writes the outputs.
constexpr int kReqWarps = 16;

__global__ void __launch_bounds__(kReqWarps * 32) filter_requests_kernel(const Params P) {
  __shared__ FiltRow rows[kReqWarps][2];  // per warp: target row, draft row of its position
  __shared__ int32_t draw_id[kMaxK];
  __shared__ float draw_w[kMaxK];
  __shared__ int32_t fail_pos;  // first rejected drafted position, or l - 1
  __shared__ int flags_sh;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int32_t r = blockIdx.x;
  const FiltRow* recs = reinterpret_cast<const FiltRow*>(P.filt);
  const int32_t off = __ldg(P.offs + r), off1 = __ldg(P.offs + r + 1), ell = __ldg(P.lens + r);
  const bool ok = ell >= 1 && ell <= P.max_len && off1 - off == ell && off >= r && off1 <= P.Nt &&
                  (r != 0 || off == 0) && (r != P.B - 1 || off1 == P.Nt) &&
                  off - r + ell - 1 <= P.Nd;
  if (!ok) {  // uniform over the CTA
    if (threadIdx.x == 0) raise_error(P, SV_DEVERR_LEN);
    return;
  }
  if (threadIdx.x == 0) {
    fail_pos = ell - 1;
    flags_sh = 0;
  }
  grid_dep_wait();  // the row records come from filter_rows_kernel
  __syncthreads();
  FiltRow& T = rows[warp][0];
  FiltRow& D = rows[warp][1];
  int flags = 0;
  // labels of every drafted position, and the accept tests
  for (int32_t j = warp; j < ell - 1; j += kReqWarps) {
    copy_row(T, recs + off + j, lane);
    copy_row(D, recs + P.Nt + off - r + j, lane);
    if (lane == 0) flags |= T.flags | D.flags;
    if (P.out_conf != nullptr) {
      float c = 0.f;
      for (int i = lane; i < T.n; i += 32) c += fminf(T.w[i] / T.z, kept_prob(D, T.ids[i]));
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) c += __shfl_xor_sync(0xffffffffu, c, o);
      if (lane == 0) P.out_conf[off - r + j] = c;
    }
    if (lane == 0) {
      const int32_t x = __ldg(P.draft_tokens + off - r + j);
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
      if (!acc) atomicMin(&fail_pos, j);
    }
    __syncwarp();  // the warp's row slots are reused for its next position
  }
  if (lane == 0 && flags) atomicOr(&flags_sh, flags);
  __syncthreads();
  if (warp != 0) return;
  const int32_t a = fail_pos;
  flags = 0;
  // final token from target row a (and its draft partner when a < l - 1)
  copy_row(T, recs + off + a, lane);
  if (lane == 0) flags |= T.flags;
  int32_t final_tok = T.argmax;
  if (P.mode == SV_SAMPLE) {
    const bool residual = a < ell - 1;
    if (residual) copy_row(D, recs + P.Nt + off - r + a, lane);
    // weights of the kept target tokens, then sorted by id (ascending)
    int32_t* sid = draw_id;
    float* swt = draw_w;
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
    flags |= flags_sh;
    if (flags) raise_error(P, flags);
  }
}

}  // namespace sv
