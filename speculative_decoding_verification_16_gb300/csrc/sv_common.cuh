// sv_common.cuh -- definitions shared by the verify kernels and the host code.
#pragma once

#include <cstdint>

#include "spec_verify.h"
#include "sv_ptx.cuh"

namespace sv {

constexpr int kThreads = 256;     // threads per CTA of the finalize kernels
constexpr int kWarps = kThreads / 32;
constexpr int kMaxCluster = 16;   // largest cluster (non-portable size 16)
constexpr int kRecWords = 16;     // words of one CTA's partial record

// Per-target-row result left in the workspace by the rows kernel.  The
// normalisers are kept as sum_v 2^(x_v * sc) = z * 2^h (sc = log2(e) / T) for
// a reference h of the row, so that p(v) = exp2(fma(x_v, sc, -h)) / z.
struct RowRec {
  float mt;   // target: reference h_t (scaled units)
  float zt;   // target: z_t
  float md;   // draft partner (pairs only): reference h_d
  float zd;   // draft partner: z_d
  int32_t argt;  // target argmax (lowest id; tracked only when needed)
  int32_t acc;   // 1 if the drafted token of this position is accepted
  int32_t pick;  // filtered sampling: final token if the chain stops here
  int32_t flags; // device error bits of this row
};
static_assert(sizeof(RowRec) == 32, "RowRec layout");

// Published pass-1 partials of the rows kernel, kept in the workspace for
// the rest of the call: per (target row g, slice k) kPartWords 64-bit words
// at parts + (g * kMaxSlices + k) * kPartWords; word w carries the call's
// tag in its upper and value w of the enum below in its lower 32 bits.
// Slice k covers vocabulary ids [k * L, min(V, (k + 1) * L)) for the slice
// length L of the call.  (h, s) pairs are partial statistics sum 2^(x sc) =
// s * 2^h over the slice; m / i the slice maximum and the lowest id holding
// it (greedy or statistics only); x the logits at the drafted token when the
// slice holds it.
constexpr int kMaxSlices = 32;  // slices per row
constexpr int kPartWords = 16;  // 64-bit words per published partial (14 used)
enum { R_HT = 0, R_ST, R_MT, R_IT, R_HD, R_SD, R_MD, R_ID, R_BAD, R_XT, R_XD, R_HASX, R_NWORDS };
// Words written after the exchange: the slice's label partial sum of
// min(p_t, p_d) (pass 2, pairs only), and in slice 0's record the row's
// accept decision and device error bits (rec_mark), written with its RowRec.
constexpr int R_CP = R_NWORDS;
constexpr int R_REC = R_NWORDS + 1;
static_assert(R_REC < kPartWords, "partial record");

__device__ __forceinline__ uint32_t rec_mark(bool acc, int flags) {
  return (acc ? 0x80000000u : 0u) | (static_cast<uint32_t>(flags) & 0x7fffffffu);
}

__device__ __forceinline__ const uint64_t* part_words(const void* parts, int32_t g, int32_t k) {
  return static_cast<const uint64_t*>(parts) + (static_cast<size_t>(g) * kMaxSlices + k) * kPartWords;
}

struct Params {
  const unsigned char* tgt;
  const unsigned char* drf;
  const int32_t* draft_tokens;
  const float* uniforms;
  const int32_t* lens;
  const int32_t* offs;
  int32_t B, V, Nt, Nd, max_len;
  float T;        // temperature
  float sc;       // log2(e) / T
  int32_t top_k;  // 0 = off
  float top_p;    // 1 = off
  int32_t gfilter;  // kept sets of any size (top_k above SV_MAX_FILTER_K, or full-vocabulary top_p)
  int32_t mode;
  int32_t* out_tokens;
  int32_t* out_accept_len;
  float* out_conf;
  float* out_row_stats;
  int32_t* dev_error;
  RowRec* rec;
  void* parts;       // [N_t][32][16] words: published pass-1 partials
  void* filt;        // filtered path: FiltRow per target row, then per draft row
  uint32_t tag;      // per-call tag of the published partials (never 0)
  int32_t nslices;   // slices per row of the rows kernel (<= 32)
  int32_t nunits;    // N_t * nslices
  int32_t S;         // slice length L (elements) of the rows kernel
  int32_t rowbuf;    // bytes of one slice buffer in shared memory
  int32_t nstages;   // shared-memory stages of the rows kernel
  int32_t offs_smem; // row_offsets copied into shared memory (B + 1 <= kMaxSmemOffsets)
  int32_t nw1;       // rows kernel, labels on: consumer warps running pass 1
  int32_t poll_ns;   // rows kernel: gatherer sleep between polls
  uint64_t xwait_ns; // limit of a wait on words published by other CTAs
  int32_t fuse;      // rows kernel: finish the requests in its tail (no finalize launch)
};

// Partial statistics of a row: sum_v 2^(x_v * sc) = s * 2^h; m = max raw
// logit and i = lowest id holding it (tracked variant only; m = -inf, i =
// INT_MAX otherwise).
struct RStat {
  float h, s, m;
  int32_t i;
};

__device__ __forceinline__ RStat rstat_empty() {
  return RStat{-INFINITY, 0.f, -INFINITY, 0x7fffffff};
}

__device__ __forceinline__ float warp_max_f32(float v) {
  float r;
  asm volatile("redux.sync.max.f32 %0, %1, 0xffffffff;" : "=f"(r) : "f"(v));
  return r;
}

__device__ __forceinline__ float warp_sum_f32(float v) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
  return v;
}

// Merge two statistics (a target and a draft row) over the 32 lanes'
// partials: max reference, one rescale each, plain sum (the two dependency
// chains interleaved); with TRACK also the max and the lowest id holding it
// (without TRACK those fields are unused and left as they are).  Every lane
// gets the same bits.
template <bool TRACK>
__device__ __forceinline__ void rstat_warp_reduce2(RStat& a, RStat& b) {
  const float ha = warp_max_f32(a.h), hb = warp_max_f32(b.h);
  float sa = a.h == -INFINITY ? 0.f : a.s * ex2(a.h - ha);
  float sb = b.h == -INFINITY ? 0.f : b.s * ex2(b.h - hb);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    sa += __shfl_xor_sync(0xffffffffu, sa, off);
    sb += __shfl_xor_sync(0xffffffffu, sb, off);
  }
  a.s = ha == -INFINITY ? 0.f : sa;
  b.s = hb == -INFINITY ? 0.f : sb;
  a.h = ha;
  b.h = hb;
  if (TRACK) {
    const float ma = warp_max_f32(a.m), mb = warp_max_f32(b.m);
    a.i = __reduce_min_sync(0xffffffffu, a.m == ma ? a.i : 0x7fffffff);
    b.i = __reduce_min_sync(0xffffffffu, b.m == mb ? b.i : 0x7fffffff);
    a.m = ma;
    b.m = mb;
  }
}

__device__ __forceinline__ void raise_error(const Params& P, int bits) {
  if (P.dev_error != nullptr) atomicOr(P.dev_error, bits);
}

// Geometry of one CTA's slice of one logits row in shared memory.  The
// copied byte range is the 16-byte-aligned cover [a_start, a_end) of the
// slice; element i of the slice sits at byte `head + i * esize` of the
// buffer.  16-byte vector k of the buffer holds slice elements
// k * VEC - hoff .. k * VEC - hoff + VEC - 1.
struct Slice {
  const unsigned char* gsrc;  // global address of the buffer's first byte (16-aligned)
  int32_t nbytes;             // bytes copied (multiple of 16; 0 when the slice is empty)
  int32_t hoff;               // head offset in elements
  int32_t len;                // valid elements
  int32_t v0;                 // vocabulary id of slice element 0
};

template <int ES>
__device__ __forceinline__ Slice make_slice(const unsigned char* row, int32_t V, int32_t rank,
                                            int32_t S) {
  Slice s;
  s.v0 = rank * S;
  s.len = max(0, min(S, V - s.v0));
  const uintptr_t gs = reinterpret_cast<uintptr_t>(row) + static_cast<uintptr_t>(s.v0) * ES;
  const uintptr_t as = gs & ~static_cast<uintptr_t>(15);
  const uintptr_t ae = (gs + static_cast<uintptr_t>(s.len) * ES + 15) & ~static_cast<uintptr_t>(15);
  s.gsrc = reinterpret_cast<const unsigned char*>(as);
  s.hoff = static_cast<int32_t>((gs - as) / ES);
  s.nbytes = s.len > 0 ? static_cast<int32_t>(ae - as) : 0;
  return s;
}

// Read slice element i (0 <= i < len) as float from the shared buffer.
template <int ES>
__device__ __forceinline__ float slice_elem(const unsigned char* buf, const Slice& s, int32_t i) {
  if (ES == 2) {
    const uint16_t b = *reinterpret_cast<const uint16_t*>(buf + (s.hoff + i) * 2);
    return __uint_as_float(static_cast<uint32_t>(b) << 16);
  }
  return *reinterpret_cast<const float*>(buf + (s.hoff + i) * 4);
}

// Unpack 16-byte vector k of a buffer into VEC floats (no masking).
template <int ES>
__device__ __forceinline__ void load_vec_raw(const unsigned char* buf, int32_t k, float* x) {
  const uint4 w = *reinterpret_cast<const uint4*>(buf + 16 * k);
  if (ES == 2) {
    x[0] = bf16lo(w.x); x[1] = bf16hi(w.x); x[2] = bf16lo(w.y); x[3] = bf16hi(w.y);
    x[4] = bf16lo(w.z); x[5] = bf16hi(w.z); x[6] = bf16lo(w.w); x[7] = bf16hi(w.w);
  } else {
    x[0] = __uint_as_float(w.x); x[1] = __uint_as_float(w.y);
    x[2] = __uint_as_float(w.z); x[3] = __uint_as_float(w.w);
  }
}

// True when every 16-byte vector of the slice buffer lies inside the slice.
template <int ES>
__device__ __forceinline__ bool slice_aligned(const Slice& s) {
  return s.hoff == 0 && (s.len % (16 / ES)) == 0;
}

// Unpack 16-byte vector k of a slice buffer into VEC floats; elements outside
// the slice read as -inf.
template <int ES>
__device__ __forceinline__ void load_vec(const unsigned char* buf, const Slice& s, int32_t k,
                                         float* x) {
  constexpr int VEC = 16 / ES;
  const uint4 w = *reinterpret_cast<const uint4*>(buf + 16 * k);
  if (ES == 2) {
    x[0] = bf16lo(w.x); x[1] = bf16hi(w.x); x[2] = bf16lo(w.y); x[3] = bf16hi(w.y);
    x[4] = bf16lo(w.z); x[5] = bf16hi(w.z); x[6] = bf16lo(w.w); x[7] = bf16hi(w.w);
  } else {
    x[0] = __uint_as_float(w.x); x[1] = __uint_as_float(w.y);
    x[2] = __uint_as_float(w.z); x[3] = __uint_as_float(w.w);
  }
  const int32_t i0 = k * VEC - s.hoff;  // slice index of lane 0
  if (i0 < 0 || i0 + VEC > s.len) {
#pragma unroll
    for (int l = 0; l < VEC; ++l)
      if (i0 + l < 0 || i0 + l >= s.len) x[l] = -INFINITY;
  }
}

}  // namespace sv
