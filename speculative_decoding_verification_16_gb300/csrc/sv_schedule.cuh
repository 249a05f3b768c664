// sv_schedule.cuh -- DSpark hardware-aware prefix scheduler.
//
// "DeepSeek DSpark speculative decoding" tutorial: every drafted position k
// of request r carries a conditional survival probability c_{r,k} (section
// "置信度预测头"); the scheduler works on the prefix survival S_{r,k} =
// prod_{i<=k} c_{r,i} (section "时序温度缩放校准（STS）") and picks each
// request's verify length to maximise Theta = tau * SPS(B) greedily: all
// candidates sorted by S, descending, added one at a time while Theta still
// rises (section "硬件感知前缀调度器").
//
// tau = sum_r (1 + sum_{k < l_r - 1} S_{r,k}) (one token per request plus
// each verified draft with its survival probability), B = sum_r l_r, every
// request starting at l_r = 1.  Because c is clamped to [0, 1], S never
// rises along a request and the sorted order adds each request's positions
// as a prefix.  Adding the candidates best-first turns the greedy scan into
// a prefix-sum problem: after n additions tau_n = B_0 + (sum of the n best
// S) and B = B_0 + n, so one sort, one scan and one minimum (the first n
// whose next addition does not raise Theta) give the schedule.
//
// One CTA of kScheduleThreads threads per call; all in float64 (the pool is
// small: at most SV_SCHEDULE_MAX_CANDIDATES candidates).  The sort is a
// stable merge sort of the requests' runs (each already in order), so it
// takes log2(B) merge levels.
#pragma once

#include "sv_common.cuh"

namespace sv {

constexpr int kScheduleThreads = 1024;
constexpr int kScheduleWarps = kScheduleThreads / 32;

struct ScheduleArgs {
  const float* conf;  // [B][K]
  int32_t B, K;
  const double* sps;  // [n_sps]
  int32_t n_sps;
  int32_t* out_lens;  // [B]
  double* out_theta;  // [2] or null: Theta, candidates added
  int32_t npad;       // even, >= B * K (buffer length)
};

// Sort key of a candidate: larger S first (S >= +0, whose bits rise with
// the value, so the complement falls).  Equal keys keep their order: the
// merges below are stable and start from the candidates in index order.
__device__ __forceinline__ uint64_t schedule_key(double s) {
  return ~static_cast<uint64_t>(__double_as_longlong(s));
}

__device__ __forceinline__ double schedule_value(uint64_t key) {
  return __longlong_as_double(static_cast<long long>(~key));
}

// Inclusive float64 scan over the block, one value per thread, thread order
// (the warps' totals are prefixed once, by warp 0).
__device__ __forceinline__ double block_incl_scan_f64(double v, double* scratch) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const double n = __shfl_up_sync(0xffffffffu, v, off);
    if (lane >= off) v += n;
  }
  if (lane == 31) scratch[w] = v;
  __syncthreads();
  if (w == 0) {  // exclusive prefix of the warp totals, in warp order
    const double t = lane < kScheduleWarps ? scratch[lane] : 0.0;
    double x = t;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const double n = __shfl_up_sync(0xffffffffu, x, off);
      if (lane >= off) x += n;
    }
    if (lane < kScheduleWarps) scratch[kScheduleWarps + lane] = x - t;
  }
  __syncthreads();
  return scratch[kScheduleWarps + w] + v;
}

// One level of the stable merge sort: runs of R keys in src (the last one
// possibly short) merged pairwise into dst; thread t writes the outputs
// [t E, t E + E).  Equal keys: the earlier run first.
__device__ __forceinline__ void merge_level(const uint64_t* ks, const uint16_t* rs, uint64_t* kd,
                                            uint16_t* rd, int N, int R, int E) {
  int p = threadIdx.x * E;
  const int p1 = min(N, p + E);
  while (p < p1) {
    const int base = p / (2 * R) * (2 * R);
    const int alen = min(R, N - base), blen = max(0, min(R, N - base - R));
    const uint64_t* A = ks + base;
    const uint64_t* Bk = A + alen;
    const int q0 = p - base, q1 = min(p1, base + alen + blen) - base;
    // merge path: i = elements of A among the first q0 outputs
    int lo = max(0, q0 - blen), hi = min(q0, alen);
    while (lo < hi) {
      const int mid = (lo + hi) >> 1;
      if (A[mid] <= Bk[q0 - mid - 1]) lo = mid + 1; else hi = mid;
    }
    int i = lo, j = q0 - lo;
    for (int q = q0; q < q1; ++q) {
      const bool takeA = i < alen && (j >= blen || A[i] <= Bk[j]);
      kd[base + q] = takeA ? A[i] : Bk[j];
      rd[base + q] = takeA ? rs[base + i] : rs[base + alen + j];
      if (takeA) ++i; else ++j;
    }
    p = base + q1;
  }
}

__global__ void __launch_bounds__(kScheduleThreads) schedule_kernel(const ScheduleArgs A) {
  extern __shared__ __align__(128) unsigned char smem[];
  const int tid = threadIdx.x;
  const int N = A.B * A.K, NP = A.npad;
  uint64_t* key0 = reinterpret_cast<uint64_t*>(smem);
  uint64_t* key1 = key0 + NP;
  uint16_t* rid0 = reinterpret_cast<uint16_t*>(key1 + NP);
  uint16_t* rid1 = rid0 + NP;
  int32_t* cnt = reinterpret_cast<int32_t*>(rid1 + NP);  // NP even: 4-byte aligned
  double* red = reinterpret_cast<double*>(cnt + ((A.B + 1) & ~1));  // 8-byte aligned
  int* ired = reinterpret_cast<int*>(red + 2 * kScheduleWarps);

  // ---- prefix survival of every candidate (sequential product per request,
  //      as the definition reads); each request's run is already in order
  for (int32_t r = tid; r < A.B; r += kScheduleThreads) {
    double s = 1.0;
    for (int32_t k = 0; k < A.K; ++k) {
      const float c = __ldg(A.conf + static_cast<size_t>(r) * A.K + k);
      s *= c > 0.f ? fmin(static_cast<double>(c), 1.0) : 0.0;  // NaN, -0, < 0 -> +0
      key0[r * A.K + k] = schedule_key(s);
      rid0[r * A.K + k] = static_cast<uint16_t>(r);
    }
    cnt[r] = 1;
  }
  __syncthreads();
  // the best candidate overall is some request's first position (the
  // smallest key): when even it does not raise Theta, nothing is added and
  // the sort is skipped
  bool skip_sort = N == 0;
  if (N > 0) {
    unsigned long long kmin = ~0ull;
    for (int32_t r = tid; r < A.B; r += kScheduleThreads)
      kmin = min(kmin, static_cast<unsigned long long>(key0[r * A.K]));
    for (int off = 16; off > 0; off >>= 1) kmin = min(kmin, __shfl_xor_sync(0xffffffffu, kmin, off));
    uint64_t* wmin = reinterpret_cast<uint64_t*>(red);
    if ((tid & 31) == 0) wmin[tid >> 5] = kmin;
    __syncthreads();
    for (int w = 0; w < kScheduleWarps; ++w) kmin = min(kmin, static_cast<unsigned long long>(wmin[w]));
    const double B0 = static_cast<double>(A.B);
    skip_sort = A.B + 1 >= A.n_sps ||
                !((B0 + schedule_value(kmin)) * A.sps[A.B + 1] > B0 * A.sps[A.B]);
    __syncthreads();
  }
  if (skip_sort) {  // no candidate added: every l_r = 1
    for (int32_t r = tid; r < A.B; r += kScheduleThreads) A.out_lens[r] = 1;
    if (tid == 0 && A.out_theta != nullptr) {
      A.out_theta[0] = static_cast<double>(A.B) * A.sps[A.B];
      A.out_theta[1] = 0.0;
    }
    return;
  }

  // ---- stable merges of the per-request runs, ping-pong
  const int E = (N + kScheduleThreads - 1) / kScheduleThreads;  // outputs per thread
  uint64_t* ks = key0;
  uint16_t* rs = rid0;
  for (int R = max(A.K, 1); R < N; R *= 2) {
    uint64_t* kd = ks == key0 ? key1 : key0;
    uint16_t* rd = rs == rid0 ? rid1 : rid0;
    merge_level(ks, rs, kd, rd, N, R, E);
    __syncthreads();
    ks = kd;
    rs = rd;
  }

  // ---- tau after n additions: B + (sum of the n best S); thread t owns
  //      the contiguous candidates [t * E, t * E + E)
  const int i0 = min(N, tid * E), i1 = min(N, i0 + E);
  double run = 0.0;
  for (int i = i0; i < i1; ++i) run += schedule_value(ks[i]);
  const double incl = block_incl_scan_f64(run, red);
  // first n (candidates added) whose next addition does not raise Theta
  const double B0 = static_cast<double>(A.B);
  int stop = N;  // all candidates added
  {
    double pre = incl - run;  // sum of the candidates before i0
    for (int n = i0; n <= i1 && n <= N; ++n) {
      const int bn = A.B + n;
      bool halt = n == N || bn + 1 >= A.n_sps;
      if (!halt) {
        const double s_next = schedule_value(ks[n]);
        const double th = (B0 + pre) * A.sps[bn];
        const double th_next = (B0 + pre + s_next) * A.sps[bn + 1];
        halt = !(th_next > th);
        pre += s_next;
      }
      if (halt) {
        stop = n;
        break;
      }
    }
  }
  const int s_min = __reduce_min_sync(0xffffffffu, stop);
  if ((tid & 31) == 0) ired[tid >> 5] = s_min;
  __syncthreads();
  int nstar = ired[0];
  for (int w = 1; w < kScheduleWarps; ++w) nstar = min(nstar, ired[w]);

  // ---- lengths: one more verified row per added candidate
  for (int i = tid; i < nstar; i += kScheduleThreads) atomicAdd(&cnt[rs[i]], 1);
  __syncthreads();
  for (int32_t r = tid; r < A.B; r += kScheduleThreads) A.out_lens[r] = cnt[r];
  if (A.out_theta != nullptr) {
    // Theta of the schedule, by the thread whose run holds the last added
    // candidate (thread 0 when none was added), and the number added
    const bool owner = nstar == 0 ? tid == 0 : (i0 < nstar && nstar <= i1);
    if (owner) {
      double pre = nstar == 0 ? 0.0 : incl - run;
      for (int i = i0; i < nstar; ++i) pre += schedule_value(ks[i]);
      A.out_theta[0] = (B0 + pre) * A.sps[A.B + nstar];
      A.out_theta[1] = static_cast<double>(nstar);
    }
  }
}

}  // namespace sv
