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
//                       its Leviathan et al. citation).  Only that one row
//                       pair is read again from HBM.
//
// The unfiltered draw runs on a cluster of C4 CTAs per request: CTA `rank`
// owns a contiguous vocabulary slice, each thread a contiguous run of it, so
// that running sums in (CTA rank, thread, element) order are sums in
// ascending token id.  Partial masses are exchanged through distributed
// shared memory and the one thread whose run holds the target mass walks it.
#pragma once

#include "sv_common.cuh"

namespace sv {

constexpr int kF_OffBars = 0;
constexpr int kF_OffMass = 64;                                  // 2 rounds x kMaxCluster floats
constexpr int kF_OffScan = kF_OffMass + 2 * kMaxCluster * 4;    // kThreads floats
constexpr int kF_OffWarp = kF_OffScan + kThreads * 4;           // kWarps words
constexpr int kF_OffInfo = kF_OffWarp + 32 * 4;                 // request info
constexpr int kF_HdrBytes = 2048;
static_assert(kF_OffInfo + 64 <= kF_HdrBytes, "finalize header");

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

// Block-wide min / max of an int; every thread gets the result.
__device__ __forceinline__ int block_min_int(int v, int* scratch) {
  v = __reduce_min_sync(0xffffffffu, v);
  if ((threadIdx.x & 31) == 0) scratch[threadIdx.x >> 5] = v;
  __syncthreads();
  int r = scratch[0];
  for (int w = 1; w < kWarps; ++w) r = min(r, scratch[w]);
  __syncthreads();
  return r;
}

__device__ __forceinline__ int block_max_int(int v, int* scratch) {
  v = __reduce_max_sync(0xffffffffu, v);
  if ((threadIdx.x & 31) == 0) scratch[threadIdx.x >> 5] = v;
  __syncthreads();
  int r = scratch[0];
  for (int w = 1; w < kWarps; ++w) r = max(r, scratch[w]);
  __syncthreads();
  return r;
}

template <int ES>
__global__ void __launch_bounds__(kThreads) finalize_draw_kernel(const Params P) {
  extern __shared__ __align__(128) unsigned char smem[];
  const uint32_t rank = cluster_ctarank();
  const uint32_t csize = cluster_nctarank();
  const int32_t r = static_cast<int32_t>(cluster_id_x());
  const int tid = threadIdx.x;
  float* scan = reinterpret_cast<float*>(smem + kF_OffScan);
  int* wscr = reinterpret_cast<int*>(smem + kF_OffWarp);
  ReqInfo* sinfo = reinterpret_cast<ReqInfo*>(smem + kF_OffInfo);
  unsigned char* buf_t = smem + kF_HdrBytes;
  unsigned char* buf_d = buf_t + P.rowbuf4;
  const uint32_t bar = smem_addr(smem + kF_OffBars);

  cluster_arrive_relaxed();
  if (tid < 32) {
    const ReqInfo rq = scan_request(P, r, tid);
    if (tid == 0) {
      *sinfo = rq;
      mbar_init(bar, 1);
      fence_mbar_init();
    }
  }
  __syncthreads();
  const ReqInfo q = *sinfo;
  if (!q.ok) {  // uniform across the cluster: every CTA read the same request
    if (rank == 0 && tid == 0) raise_error(P, SV_DEVERR_LEN);
    cluster_wait_acquire();
    return;
  }
  const int32_t trow_i = q.off + q.a;
  const int32_t drow_i = q.off - r + q.a;
  const RowRec rr = P.rec[trow_i];
  const unsigned char* trow = P.tgt + static_cast<size_t>(trow_i) * P.V * ES;
  const unsigned char* drow = P.drf + static_cast<size_t>(drow_i) * P.V * ES;
  const Slice s_t = make_slice<ES>(trow, P.V, rank, P.S4);
  Slice s_d = make_slice<ES>(drow, P.V, rank, P.S4);
  if (!q.residual) s_d.nbytes = 0, s_d.len = 0;
  if (tid == 0) {
    mbar_arrive_expect_tx(bar, static_cast<uint32_t>(s_t.nbytes + s_d.nbytes));
    if (s_t.nbytes) bulk_g2s(smem_addr(buf_t), s_t.gsrc, s_t.nbytes, bar);
    if (s_d.nbytes) bulk_g2s(smem_addr(buf_d), s_d.gsrc, s_d.nbytes, bar);
  }
  bool timeout = false;
  mbar_wait(bar, 0, timeout);
  const bool any_timeout = __syncthreads_or(timeout ? 1 : 0) != 0;

  const float sc = P.sc;
  DrawRow dr;
  dr.sc = sc;
  dr.ht = rr.mt;
  dr.hd = rr.md;
  dr.ratio = rr.zt / rr.zd;
  dr.residual = q.residual;
  if (rank == 0 && (tid >> 5) == 1) sum_labels(P, r, q.off, q.ell, tid & 31);
  const int32_t E = (s_t.len + kThreads - 1) / kThreads;  // elements per thread
  const int32_t i0 = min(s_t.len, tid * E), i1 = min(s_t.len, i0 + E);
  const float u = __ldg(P.uniforms + q.off + q.ell - 1);

  cluster_wait_acquire();  // all CTAs started: DSMEM stores allowed from here
  // Two rounds at most: if the residual mass is zero the draw falls back to p_t.
  for (int round = 0; round < 2; ++round) {
    float* mass = reinterpret_cast<float*>(smem + kF_OffMass) + round * kMaxCluster;
    // this thread's run, summed in ascending id order
    float wsum = 0.f;
    for (int32_t i = i0; i < i1; ++i) {
      const float t = slice_elem<ES>(buf_t, s_t, i);
      const float d = dr.residual ? slice_elem<ES>(buf_d, s_d, i) : 0.f;
      wsum += dr.w(t, d);
    }
    // exclusive prefix of the per-thread sums inside the CTA (fixed order)
    const float incl = warp_incl_scan(wsum);
    float* wtot = reinterpret_cast<float*>(wscr);
    if ((tid & 31) == 31) wtot[tid >> 5] = incl;
    __syncthreads();
    float wbase = 0.f, cta_total = 0.f;
    for (int w = 0; w < kWarps; ++w) {
      if (w < (tid >> 5)) wbase += wtot[w];
      cta_total += wtot[w];
    }
    const float excl = wbase + (incl - wsum);
    scan[tid] = excl;
    __syncthreads();
    // CTA totals to every CTA of the cluster
    if (tid < static_cast<int>(csize))
      st_cluster_u32(mapa(smem_addr(mass + rank), tid), __float_as_uint(cta_total));
    cluster_arrive_release();
    cluster_wait_acquire();
    float total = 0.f, prefix = 0.f;
    for (uint32_t c = 0; c < csize; ++c) {
      if (c < rank) prefix += mass[c];
      total += mass[c];
    }
    if (round == 0 && dr.residual && !(total > 0.f)) {  // no residual mass: draw from p_t
      dr.residual = false;
      continue;
    }
    const float target = u * total;
    // owning CTA: first with positive mass whose range passes the target,
    // else the last with positive mass
    int owner = -1, last_pos = -1;
    float pc = 0.f;
    for (uint32_t c = 0; c < csize; ++c) {
      if (mass[c] > 0.f) {
        last_pos = static_cast<int>(c);
        if (owner < 0 && target < pc + mass[c]) owner = static_cast<int>(c);
      }
      pc += mass[c];
    }
    if (owner < 0) owner = last_pos;
    if (owner < 0) {  // no mass anywhere: non-finite statistics
      if (rank == 0 && tid == 0) {
        raise_error(P, SV_DEVERR_NAN);
        P.out_tokens[trow_i] = rr.argt;
      }
      break;
    }
    if (static_cast<int>(rank) == owner) {
      const float local = target - prefix;  // target mass inside this CTA
      const bool pos = wsum > 0.f;
      const bool hit = pos && local < excl + wsum;
      int own = block_min_int(hit ? tid : kThreads, wscr);
      const int lastp = block_max_int(pos ? tid : -1, wscr);
      if (own == kThreads) own = lastp;
      if (tid == own) {
        const float need = local - excl;  // mass to pass inside this run
        float run = 0.f;
        int32_t pick = -1, last = -1;
        for (int32_t i = i0; i < i1; ++i) {
          const float t = slice_elem<ES>(buf_t, s_t, i);
          const float d = dr.residual ? slice_elem<ES>(buf_d, s_d, i) : 0.f;
          const float wv = dr.w(t, d);
          run += wv;
          if (wv > 0.f) last = i;
          if (run > need) {
            pick = i;
            break;
          }
        }
        if (pick < 0) pick = last;
        P.out_tokens[trow_i] = s_t.v0 + pick;
      }
    }
    break;
  }

  if (rank == 0 && tid < 32) {  // accepted drafts, -1 after the final token, flags
    if (tid == 0) P.out_accept_len[r] = q.a;
    int flags = 0;
    for (int32_t j = tid; j < q.ell; j += 32) {
      if (j < q.a) P.out_tokens[q.off + j] = __ldg(P.draft_tokens + q.off - r + j);
      else if (j > q.a) P.out_tokens[q.off + j] = -1;
      if (j <= q.a) flags |= P.rec[q.off + j].flags;
    }
    flags = __reduce_or_sync(0xffffffffu, flags) | (any_timeout ? SV_DEVERR_TIMEOUT : 0);
    if (tid == 0 && flags) raise_error(P, flags);
  }
  if (any_timeout) {  // one more bounded wait for a copy still in flight
    bool again = false;
    mbar_wait(bar, 0, again);
  }
}

// Greedy and filtered sampling: the final token is already known per row.
// One warp per request: lane 0 scans and writes, all lanes sum labels.
__global__ void __launch_bounds__(kThreads) finalize_select_kernel(const Params P) {
  const int32_t r = blockIdx.x * kWarps + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (r >= P.B) return;  // whole warps leave together
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
