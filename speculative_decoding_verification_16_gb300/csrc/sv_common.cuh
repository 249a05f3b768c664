// sv_common.cuh -- definitions shared by the verify kernels and the host code.
#pragma once

#include <cstdint>

#include "spec_verify.h"
#include "sv_ptx.cuh"

namespace sv {

constexpr int kThreads = 256;     // threads per CTA of every kernel
constexpr int kWarps = kThreads / 32;
constexpr int kChunks = 4;        // bulk-copy chunks (one mbarrier each) per CTA slice
constexpr int kMaxCluster = 16;   // largest cluster (non-portable size 16)
constexpr int kRecWords = 16;     // words of one CTA's partial record
constexpr int kHdrBytes = 4096;   // fixed shared-memory header of the rows kernel
constexpr uint32_t kSpinLimit = 1u << 22;  // polls before a bounded wait gives up

// Per-target-row result left in the workspace by the rows kernel.
struct RowRec {
  float mt;   // target: max raw logit over the row
  float zt;   // target: sum over the kept set of exp((x - mt) / T)
  float md;   // draft partner (pairs only): max raw logit
  float zd;   // draft partner: normaliser
  int32_t argt;  // target argmax (lowest id)
  int32_t acc;   // 1 if the drafted token of this position is accepted
  int32_t pick;  // filtered sampling: final token if the chain stops here
  int32_t flags; // device error bits of this row
};
static_assert(sizeof(RowRec) == 32, "RowRec layout");

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
  int32_t mode;
  int32_t* out_tokens;
  int32_t* out_accept_len;
  float* out_conf;
  float* out_row_stats;
  int32_t* dev_error;
  RowRec* rec;
  int32_t S;       // vocabulary slice (elements) per CTA of the rows kernel
  int32_t S4;      // vocabulary slice per CTA of the finalize kernel
  int32_t rowbuf;  // bytes of one row buffer in shared memory (rows kernel)
  int32_t rowbuf4; // bytes of one row buffer in shared memory (finalize kernel)
};

__device__ __forceinline__ void raise_error(const Params& P, int bits) {
  if (P.dev_error != nullptr) atomicOr(P.dev_error, bits);
}

// One thread's (or CTA's) running softmax statistics of a row:
// m = max raw logit, s = sum exp2((x - m) * sc), i = lowest id holding m.
struct Stat {
  float m;
  float s;
  int32_t i;
};

__device__ __forceinline__ Stat stat_empty() { return Stat{-INFINITY, 0.f, 0x7fffffff}; }

// Merge two partial statistics (log-sum-exp algebra, lowest id on ties).
__device__ __forceinline__ Stat stat_merge(Stat a, Stat b, float sc) {
  Stat r;
  r.m = fmaxf(a.m, b.m);
  if (r.m == -INFINITY) {
    r.s = 0.f;
  } else {
    r.s = (a.m == -INFINITY ? 0.f : a.s * ex2((a.m - r.m) * sc)) +
          (b.m == -INFINITY ? 0.f : b.s * ex2((b.m - r.m) * sc));
  }
  r.i = a.m > b.m ? a.i : (b.m > a.m ? b.i : min(a.i, b.i));
  return r;
}

__device__ __forceinline__ Stat stat_shfl_down(Stat a, int off) {
  Stat b;
  b.m = __shfl_down_sync(0xffffffffu, a.m, off);
  b.s = __shfl_down_sync(0xffffffffu, a.s, off);
  b.i = __shfl_down_sync(0xffffffffu, a.i, off);
  return b;
}

// Block-wide merge; the result is valid in thread 0.  `scratch` holds 3 *
// kWarps words.  Ends with a __syncthreads (scratch may be reused after).
__device__ __forceinline__ Stat block_merge(Stat a, float sc, float* scratch) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) a = stat_merge(a, stat_shfl_down(a, off), sc);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) {
    scratch[warp] = a.m;
    scratch[kWarps + warp] = a.s;
    scratch[2 * kWarps + warp] = __int_as_float(a.i);
  }
  __syncthreads();
  if (warp == 0) {
    Stat b = lane < kWarps ? Stat{scratch[lane], scratch[kWarps + lane],
                                  __float_as_int(scratch[2 * kWarps + lane])}
                           : stat_empty();
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) b = stat_merge(b, stat_shfl_down(b, off), sc);
    a = b;
  }
  __syncthreads();
  return a;
}

// Block-wide sum; valid in thread 0.  Fixed order (deterministic).
__device__ __forceinline__ float block_sum(float v, float* scratch) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v += __shfl_down_sync(0xffffffffu, v, off);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) scratch[warp] = v;
  __syncthreads();
  if (warp == 0) {
    float b = lane < kWarps ? scratch[lane] : 0.f;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) b += __shfl_down_sync(0xffffffffu, b, off);
    v = b;
  }
  __syncthreads();
  return v;
}

__device__ __forceinline__ bool block_any(bool v, int* scratch) {
  const int r = __syncthreads_or(v ? 1 : 0);
  (void)scratch;
  return r != 0;
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

// Byte range of chunk c (of kChunks) of a slice's copy, on the 16-byte grid.
__device__ __forceinline__ void chunk_range(int32_t nbytes, int c, int32_t* lo, int32_t* hi) {
  const int32_t nv = nbytes >> 4;
  *lo = (nv * c / kChunks) << 4;
  *hi = (nv * (c + 1) / kChunks) << 4;
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
