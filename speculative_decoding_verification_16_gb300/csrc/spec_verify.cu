// spec_verify.cu -- host side of the C ABI declared in include/spec_verify.h.
//
// Argument checks happen on the host before anything is enqueued; every
// entry point only enqueues kernels on the caller's stream and never
// synchronises.  Nothing here allocates device memory: all scratch comes
// from the caller's workspace.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <algorithm>
#include <atomic>
#include <mutex>
#include <unordered_map>

#include "spec_verify.h"
#include "sv_common.cuh"
#include "sv_filter.cuh"
#include "sv_finalize.cuh"
#include "sv_rows.cuh"
#include "sv_schedule.cuh"
#include "sv_gfilter.cuh"

namespace sv {
namespace {

constexpr int kMaxDevices = 64;

struct DeviceCache {
  bool init = false;
  int sms = 0;
  int max_smem_optin = 0;
};

std::mutex g_mu;
DeviceCache g_dev[kMaxDevices];

// Process-wide tuning of the rows kernel.  The defaults are the shipped
// configuration; only spec_verify_set_tuning changes them (tests and
// sweeps), so no call reads the environment.
struct Tuning {
  int slice = 0;            // target slice length in elements; 0: 22000 bytes' worth
  int stages = kMaxStages;  // most shared-memory stages
  int warps = 16;           // consumer warps (16 or 24)
  int pass1_warps = 0;      // consumer warps on pass 1 with labels on; 0: half
  int poll_ns = 64;         // sleep between polls of another CTA's words (64 ns: ~1 %
                            // faster than 128 on conc32 sampling, greedy unchanged)
  int64_t xwait_ns = static_cast<int64_t>(kWaitLimitNs);  // limit of a wait on other CTAs
};
std::mutex g_tune_mu;
Tuning g_tune;

Tuning tuning() {
  std::lock_guard<std::mutex> lock(g_tune_mu);
  return g_tune;
}

int device_info(DeviceCache* out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return SV_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceCache& c = g_dev[dev];
  if (!c.init) {
    if (cudaDeviceGetAttribute(&c.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&c.max_smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) !=
            cudaSuccess)
      return SV_ERR_CUDA;
    c.init = true;
  }
  *out = c;
  return SV_OK;
}

int round_up(int v, int m) { return (v + m - 1) / m * m; }

// Bytes of one row buffer for a slice of S elements (16-byte cover + slack).
int rowbuf_bytes(int S, int es) { return round_up(S * es + 32, 128); }

// Size k of the kept set under top-k / top-p filtering: 0 when unfiltered,
// -1 when the set can exceed SV_MAX_FILTER_K tokens (the general path).
int filter_k(int V, int top_k, float top_p) {
  const bool use_k = top_k > 0 && top_k < V;
  const bool use_p = top_p < 1.0f;
  if (!use_k && !use_p) return 0;
  const int k = use_k ? top_k : V;
  return k <= SV_MAX_FILTER_K ? k : -1;
}

// Geometry of the rows kernel: a row is cut into S <= kMaxSlices slices of
// L elements (L a multiple of the 16-byte vector; about 11000 bf16 / 5500
// fp32 elements by default, SV_TUNE_SLICE overrides) and as many stages
// (kMinStages .. kMaxStages, SV_TUNE_STAGES caps) as the shared memory
// allows next to the row_offsets copy (B + 1 entries when they fit).
struct RowsGeom {
  int L, S, stages, smem, offs_smem;
};

int rows_geometry(int V, int B, int es, const DeviceCache& dc, RowsGeom* g) {
  const int vec = 16 / es;
  const Tuning tu = tuning();
  const int target = tu.slice > 0 ? tu.slice : 22000 / es;
  int S = std::max(1, (V + target - 1) / target);
  S = std::min(S, kMaxSlices);
  const int L = round_up((V + S - 1) / S, vec);
  S = (V + L - 1) / L;  // no empty trailing slice
  const int offs = B + 1 <= kMaxSmemOffsets ? round_up((B + 1) * 4, 128) : 0;
  const int max_stages = std::min(kMaxStages, tu.stages);
  for (int ns = max_stages; ns >= kMinStages; --ns) {
    const int smem = kRowsHdrBytes + ns * 2 * rowbuf_bytes(L, es) + offs;
    if (smem <= dc.max_smem_optin) {
      *g = RowsGeom{L, S, ns, smem, offs > 0};
      return SV_OK;
    }
  }
  return SV_ERR_UNSUPPORTED;  // rows too long for kMaxSlices slices in shared memory
}

// Kernel attributes and the occupancy check are host calls that can cost
// microseconds; they run once per (device, kernel, smem, cluster size).
struct PreparedKey {
  int dev;
  const void* fn;
  int smem;
  int cluster;
  int status;
};
constexpr int kMaxPrepared = 256;
PreparedKey g_prepared[kMaxPrepared];
int g_nprepared = 0;

int find_prepared(int dev, const void* fn, int smem, int C) {
  std::lock_guard<std::mutex> lock(g_mu);
  for (int i = 0; i < g_nprepared; ++i) {
    const PreparedKey& k = g_prepared[i];
    if (k.dev == dev && k.fn == fn && k.smem == smem && k.cluster == C) return k.status;
  }
  return -1000;  // not prepared yet
}

void remember_prepared(int dev, const void* fn, int smem, int C, int status) {
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_nprepared < kMaxPrepared) g_prepared[g_nprepared++] = PreparedKey{dev, fn, smem, C, status};
}

// Launch `grid` CTAs of `threads` threads with `smem` bytes of dynamic
// shared memory.  Above the default 48 KB the kernel's dynamic limit is
// raised to the device maximum (not to this launch's size) once, so that one
// setting serves every configuration.  `dependent`: launch as a programmatic
// dependent of the previous kernel on the stream, which then must be this
// library's rows kernel of the same call (the kernel reads only the call's
// inputs before grid_dep_wait, and the rows kernel writes none of them).
template <typename K, typename Arg>
int launch_plain(K kernel, const Arg& P, int grid, int threads, int smem, int max_smem,
                 bool dependent, cudaStream_t stream) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return SV_ERR_CUDA;
  const void* fn = reinterpret_cast<const void*>(kernel);
  int status = find_prepared(dev, fn, smem, 1);
  if (status == -1000) {
    int n = 0;
    cudaFuncAttributes fa{};
    cudaError_t e = cudaFuncGetAttributes(&fa, kernel);
    // kernels that may need more than the default 48 KB (static and dynamic
    // together): the limit goes to the device maximum less the static part
    if (e == cudaSuccess && smem + static_cast<int>(fa.sharedSizeBytes) > 48 * 1024)
      e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               max_smem - static_cast<int>(fa.sharedSizeBytes));
    if (e != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, threads, smem) != cudaSuccess)
      status = SV_ERR_CUDA;
    else
      status = n > 0 ? n : SV_ERR_UNSUPPORTED;
    remember_prepared(dev, fn, smem, 1, status);
  }
  if (status <= 0) return status == 0 ? SV_ERR_UNSUPPORTED : status;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
  cfg.blockDim = dim3(static_cast<unsigned>(threads), 1, 1);
  cfg.dynamicSmemBytes = static_cast<size_t>(smem);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = dependent ? attr : nullptr;
  cfg.numAttrs = dependent ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, P) == cudaSuccess ? SV_OK : SV_ERR_CUDA;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

struct Args {
  const void* target_logits;
  const void* draft_logits;
  const int32_t* draft_tokens;
  const float* uniforms;
  const int32_t* verify_lens;
  const int32_t* row_offsets;
  int32_t B, V, n_target_rows, max_len, dtype;
  float temperature;
  int32_t top_k;
  float top_p;
  int32_t mode;
  int32_t* out_tokens;
  int32_t* out_accept_len;
  float* out_conf;
  float* out_row_stats;
  int32_t* dev_error;
  void* workspace;
  size_t workspace_bytes;
  void* stream;
};

// Host-visible checks shared by every entry point.
int check_args(const Args& a) {
  if (a.dtype != SV_BF16 && a.dtype != SV_FP32) return SV_ERR_DTYPE;
  if (a.B <= 0 || a.V <= 0 || a.n_target_rows < a.B) return SV_ERR_ARG;
  if (a.max_len < 1 || a.max_len > SV_MAX_LEN) return SV_ERR_ARG;
  if (static_cast<int64_t>(a.B) * a.max_len < a.n_target_rows) return SV_ERR_ARG;
  if (a.mode != SV_GREEDY && a.mode != SV_SAMPLE) return SV_ERR_ARG;
  const bool need_t = a.mode == SV_SAMPLE || a.out_conf != nullptr || a.out_row_stats != nullptr;
  if (need_t && !(a.temperature > 0.f && std::isfinite(a.temperature))) return SV_ERR_ARG;
  if (!(a.top_p > 0.f && a.top_p <= 1.f)) return SV_ERR_ARG;
  const int32_t n_draft = a.n_target_rows - a.B;
  if (a.target_logits == nullptr || a.verify_lens == nullptr || a.row_offsets == nullptr ||
      a.uniforms == nullptr || a.out_tokens == nullptr || a.out_accept_len == nullptr)
    return SV_ERR_ARG;
  if (n_draft > 0 && (a.draft_logits == nullptr || a.draft_tokens == nullptr)) return SV_ERR_ARG;
  if (!aligned(a.target_logits, 16) || (a.draft_logits && !aligned(a.draft_logits, 16)))
    return SV_ERR_ARG;
  const void* p4[] = {a.draft_tokens, a.uniforms, a.verify_lens, a.row_offsets, a.out_tokens,
                      a.out_accept_len, a.out_conf, a.out_row_stats, a.dev_error};
  for (const void* p : p4)
    if (p && !aligned(p, 4)) return SV_ERR_ARG;
  const int es = a.dtype == SV_BF16 ? 2 : 4;
  if (static_cast<double>(a.n_target_rows) * a.V * es > 9.0e18) return SV_ERR_ARG;
  // the general filter path sums level-1 masses in 32 bits, exact up to kGMaxV
  if (filter_k(a.V, a.top_k, a.top_p) < 0 && a.V > kGMaxV) return SV_ERR_UNSUPPORTED;
  if (a.workspace == nullptr || !aligned(a.workspace, 256) ||
      a.workspace_bytes < spec_verify_workspace_size(a.B, a.n_target_rows))
    return SV_ERR_WORKSPACE;
  return SV_OK;
}

// Workspace layout: RowRec[N_t] | published partials uint64[N_t][32][16]
// (tag in the upper half of every word; pass-1 statistics, the label partial
// and the row-record mark) | filtered-path row records FiltRow[2 N_t] (N_t
// target rows, then the draft rows).
size_t ws_parts_offset(int32_t n_target_rows) {
  return (static_cast<size_t>(n_target_rows) * sizeof(RowRec) + 255) / 256 * 256;
}

size_t ws_filt_offset(int32_t n_target_rows) {
  return ws_parts_offset(n_target_rows) +
         static_cast<size_t>(n_target_rows) * kMaxSlices * kPartWords * 8;
}

Params make_params(const Args& a) {
  Params P = {};
  P.tgt = static_cast<const unsigned char*>(a.target_logits);
  P.drf = static_cast<const unsigned char*>(a.draft_logits);
  P.draft_tokens = a.draft_tokens;
  P.uniforms = a.uniforms;
  P.lens = a.verify_lens;
  P.offs = a.row_offsets;
  P.B = a.B;
  P.V = a.V;
  P.Nt = a.n_target_rows;
  P.Nd = a.n_target_rows - a.B;
  P.max_len = a.max_len;
  const bool need_t = a.mode == SV_SAMPLE || a.out_conf != nullptr || a.out_row_stats != nullptr;
  P.T = need_t ? a.temperature : 1.f;
  P.sc = static_cast<float>(1.4426950408889634 / static_cast<double>(P.T));
  // the filtered paths: small kept sets (top_k = k <= SV_MAX_FILTER_K), or
  // any size (gfilter: top_k as given, 0 = off, with P.gfilter set)
  const int fk = filter_k(a.V, a.top_k, a.top_p);
  P.gfilter = fk < 0;
  P.top_k = fk >= 0 ? fk : (a.top_k > 0 && a.top_k < a.V ? a.top_k : 0);
  P.top_p = a.top_p;
  P.mode = a.mode;
  P.out_tokens = a.out_tokens;
  P.out_accept_len = a.out_accept_len;
  P.out_conf = a.out_conf;
  P.out_row_stats = a.out_row_stats;
  P.dev_error = a.dev_error;
  P.rec = static_cast<RowRec*>(a.workspace);
  P.parts = static_cast<unsigned char*>(a.workspace) + ws_parts_offset(a.n_target_rows);
  P.filt = static_cast<unsigned char*>(a.workspace) + ws_filt_offset(a.n_target_rows);
  return P;
}

// Per-call tag of the published partials: unique within the process, never 0.
std::atomic<uint32_t> g_tag{0};

uint32_t next_tag() {
  uint32_t t;
  do {
    t = g_tag.fetch_add(1, std::memory_order_relaxed) + 1;
  } while (t == 0);
  return t;
}

// Cooperative launch of one persistent wave: min(units, resident CTAs).
template <typename K>
int launch_coop(K kernel, const Params& P, int threads, int smem, const DeviceCache& dc,
                cudaStream_t stream) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return SV_ERR_CUDA;
  const void* fn = reinterpret_cast<const void*>(kernel);
  int per_sm = find_prepared(dev, fn, smem, 0);
  if (per_sm == -1000) {
    int n = 0;
    if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             dc.max_smem_optin) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, threads, smem) != cudaSuccess)
      per_sm = SV_ERR_CUDA;
    else
      per_sm = n > 0 ? n : SV_ERR_UNSUPPORTED;
    remember_prepared(dev, fn, smem, 0, per_sm);
  }
  if (per_sm <= 0) return per_sm == 0 ? SV_ERR_UNSUPPORTED : per_sm;
  const int grid = std::min(P.nunits, per_sm * dc.sms);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid, 1, 1);
  cfg.blockDim = dim3(threads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, kernel, P) != cudaSuccess) return SV_ERR_CUDA;
  return SV_OK;
}

template <int ES, int NCW>
int launch_rows(const Params& P, int smem, const DeviceCache& dc, bool need_z, bool need_conf,
                bool track, cudaStream_t st) {
#define SV_ROWS(Z, CF, TR) \
  launch_coop(rows_kernel<ES, NCW, Z, CF, TR>, P, rows_threads(NCW), smem, dc, st)
  if (need_conf) return track ? SV_ROWS(true, true, true) : SV_ROWS(true, true, false);
  if (need_z) return track ? SV_ROWS(true, false, true) : SV_ROWS(true, false, false);
  return SV_ROWS(false, false, true);
#undef SV_ROWS
}

// fuse: the rows kernel also finishes the requests in its tail (unfiltered
// path only; the caller then launches no finalize kernel).
int run_rows(const Args& a, bool fuse) {
  DeviceCache dc;
  int rc = device_info(&dc);
  if (rc != SV_OK) return rc;
  Params P = make_params(a);
  const int es = a.dtype == SV_BF16 ? 2 : 4;
  cudaStream_t st = static_cast<cudaStream_t>(a.stream);
  if (P.gfilter) {  // kept sets of any size: bisection on the value key per row
    const int rows = std::max(1, std::min(a.n_target_rows, dc.sms * 2));  // 2 CTAs per SM
    constexpr int hs = static_cast<int>(sizeof(GHist));
    if (es == 2) return launch_plain(gfilter_rows_kernel<2>, P, rows, kGThreads, hs, dc.max_smem_optin, false, st);
    return launch_plain(gfilter_rows_kernel<4>, P, rows, kGThreads, hs, dc.max_smem_optin, false, st);
  }
  if (P.top_k > 0) {  // top-k / top-p: one streaming pass per row, no exchange
    const int rows = P.Nt + P.Nd;
    const int grid = std::max(1, std::min(rows, dc.sms * kFilterCtasPerSm));
    const bool two = P.top_k > 32;  // kept lists of 64 keys per warp
    constexpr int rb = kFilterRingBytes;
    const int ms = dc.max_smem_optin;
    if (es == 2)
      return two ? launch_plain(filter_rows_kernel<2, true>, P, grid, kFiltThreads, rb, ms, false, st)
                 : launch_plain(filter_rows_kernel<2, false>, P, grid, kFiltThreads, rb, ms, false, st);
    return two ? launch_plain(filter_rows_kernel<4, true>, P, grid, kFiltThreads, rb, ms, false, st)
               : launch_plain(filter_rows_kernel<4, false>, P, grid, kFiltThreads, rb, ms, false, st);
  }
  RowsGeom geo;
  rc = rows_geometry(a.V, a.B, es, dc, &geo);
  if (rc != SV_OK) return rc;
  P.S = geo.L;
  P.nslices = geo.S;
  P.nunits = a.n_target_rows * geo.S;
  P.rowbuf = rowbuf_bytes(geo.L, es);
  P.nstages = geo.stages;
  P.tag = next_tag();
  P.offs_smem = geo.offs_smem;
  const Tuning tu = tuning();
  P.poll_ns = tu.poll_ns;
  P.xwait_ns = static_cast<uint64_t>(tu.xwait_ns);
  P.fuse = fuse ? 1 : 0;
  const int smem = geo.smem;
  // z is needed for sampling, labels and statistics; the exact max / argmax
  // only for greedy decisions and statistics
  const bool need_z = a.mode == SV_SAMPLE || a.out_conf != nullptr || a.out_row_stats != nullptr;
  // pass 2 (the per-slice sums of min(p_t, p_d)) for labels, and in sampling
  // mode for the residual masses of the slices that the final draw picks from
  const bool need_conf = a.out_conf != nullptr || a.mode == SV_SAMPLE;
  const bool track = a.mode == SV_GREEDY || a.out_row_stats != nullptr;
  // consumer warps (16 or 24) and, with labels, how many of them run pass 1
  // (SV_TUNE_WARPS, SV_TUNE_PASS1_WARPS)
  // Default split: half the warps on pass 1; with the exact max / argmax
  // tracked (greedy, statistics) pass 1 carries about a third more work, and
  // 11 of 16 warps on it measured fastest (conc32 greedy with labels: 97 us
  // against 106 us at 8).
  const int ncw = tu.warps >= 24 ? 24 : 16;
  const int dflt1 = track && ncw == 16 ? 11 : ncw / 2;
  P.nw1 = std::max(1, std::min(ncw - 1, tu.pass1_warps > 0 ? tu.pass1_warps : dflt1));
  if (es == 2)
    return ncw == 24 ? launch_rows<2, 24>(P, smem, dc, need_z, need_conf, track, st)
                     : launch_rows<2, 16>(P, smem, dc, need_z, need_conf, track, st);
  return ncw == 24 ? launch_rows<4, 24>(P, smem, dc, need_z, need_conf, track, st)
                   : launch_rows<4, 16>(P, smem, dc, need_z, need_conf, track, st);
}

// `after_rows`: the rows kernel of this same call was the last launch on the
// stream (the finalize kernel then overlaps its start with that kernel's end).
int run_finalize(const Args& a, bool after_rows) {
  DeviceCache dc;
  int rc = device_info(&dc);
  if (rc != SV_OK) return rc;
  Params P = make_params(a);
  const int es = a.dtype == SV_BF16 ? 2 : 4;
  cudaStream_t st = static_cast<cudaStream_t>(a.stream);
  const int per_warp_grid = (a.B + kWarps - 1) / kWarps;
  if (P.gfilter) {  // kept sets of any size: one CTA per request
    if (es == 2)
      return launch_plain(gfilter_requests_kernel<2>, P, a.B, kGThreads, 0, dc.max_smem_optin,
                          after_rows, st);
    return launch_plain(gfilter_requests_kernel<4>, P, a.B, kGThreads, 0, dc.max_smem_optin,
                        after_rows, st);
  }
  if (P.top_k > 0)  // top-k / top-p: decisions on the kept sets, one CTA per request
    return launch_plain(filter_requests_kernel, P, a.B, kReqWarps * 32, 0, dc.max_smem_optin,
                        after_rows, st);
  RowsGeom geo;
  rc = rows_geometry(a.V, a.B, es, dc, &geo);
  if (rc != SV_OK) return rc;
  P.nslices = geo.S;
  if (a.mode == SV_GREEDY)
    return launch_plain(finalize_select_kernel, P, per_warp_grid, kThreads, 0, dc.max_smem_optin,
                        after_rows, st);
  // unfiltered sampling: one CTA per request re-reads one slice pair
  P.S = geo.L;
  P.rowbuf = rowbuf_bytes(geo.L, es);
  const int smem = kD_HdrBytes + 2 * P.rowbuf;
  if (es == 2)
    return launch_plain(finalize_draw_kernel<2>, P, a.B, kDrawThreads, smem, dc.max_smem_optin,
                        after_rows, st);
  return launch_plain(finalize_draw_kernel<4>, P, a.B, kDrawThreads, smem, dc.max_smem_optin,
                      after_rows, st);
}

// The whole step: unfiltered, one launch (the rows kernel finishes the
// requests in its tail); filtered, the row kernel and then the request kernel
// as its programmatic dependent.
int run_call(const Args& a) {
  const bool fuse = filter_k(a.V, a.top_k, a.top_p) == 0;
  const int rc = run_rows(a, fuse);
  return rc != SV_OK || fuse ? rc : run_finalize(a, true);
}

// ---------------------------------------------------------------- static scratch
// Scratch of spec_verify_static: the same three workspace regions as a caller
// workspace (row records, label partials, published pass-1 partials), sized
// for SV_STATIC_MAX_ROWS target rows (about 21.9 MB), in a file-scope device
// array so that the call needs no allocation.  Some callers cannot allocate
// device memory at the point where they verify: a host loop in plain C with
// no caching allocator, where cudaMalloc / cudaFree would synchronise the
// whole device on every step, or a process whose memory is fully committed
// to a weight and KV-cache pool up front.  The array belongs to this module:
// two spec_verify_static calls that overlap on the GPU (different streams,
// or different host threads without ordering) share it and race.
constexpr size_t round256(size_t b) { return (b + 255) / 256 * 256; }
constexpr size_t kStaticBytes =
    round256(round256(static_cast<size_t>(SV_STATIC_MAX_ROWS) * sizeof(RowRec)) +
             static_cast<size_t>(SV_STATIC_MAX_ROWS) * kMaxSlices * kPartWords * 8 +
             static_cast<size_t>(SV_STATIC_MAX_ROWS) * 2 * sizeof(FiltRow)) +
    256;

__device__ __align__(256) unsigned char g_static_ws[kStaticBytes];

std::mutex g_static_mu;
std::unordered_map<int, void*> g_static_ptr;  // device ordinal -> address of g_static_ws

// Address of this device's static scratch.  The first call on a device looks
// the address up and clears the published-partials region (its words must
// not carry a live call tag; zero never is one) on `stream`, ahead of the
// kernels of the same call.
int static_workspace(void** out, cudaStream_t stream) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return SV_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_static_mu);
  auto it = g_static_ptr.find(dev);
  if (it == g_static_ptr.end()) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_static_ws) != cudaSuccess || p == nullptr) return SV_ERR_CUDA;
    if (cudaMemsetAsync(p, 0, kStaticBytes, stream) != cudaSuccess) return SV_ERR_CUDA;
    it = g_static_ptr.emplace(dev, p).first;
  }
  *out = it->second;
  return SV_OK;
}

}  // namespace
}  // namespace sv

#define SV_ARGS_DECL                                                                           \
  const void *target_logits, const void *draft_logits, const int32_t *draft_tokens,            \
      const float *uniforms, const int32_t *verify_lens, const int32_t *row_offsets, int32_t B, \
      int32_t V, int32_t n_target_rows, int32_t max_len, int32_t dtype, float temperature,     \
      int32_t top_k, float top_p, int32_t mode, int32_t *out_tokens, int32_t *out_accept_len,  \
      float *out_conf, float *out_row_stats, int32_t *dev_error, void *workspace,              \
      size_t workspace_bytes, void *stream
#define SV_ARGS_PACK                                                                           \
  sv::Args a{target_logits, draft_logits, draft_tokens, uniforms, verify_lens, row_offsets, B, \
             V, n_target_rows, max_len, dtype, temperature, top_k, top_p, mode, out_tokens,    \
             out_accept_len, out_conf, out_row_stats, dev_error, workspace, workspace_bytes,   \
             stream}

extern "C" {

size_t spec_verify_workspace_size(int32_t B, int32_t n_target_rows) {
  (void)B;
  const int32_t rows = n_target_rows > 0 ? n_target_rows : 0;
  const size_t bytes = sv::ws_filt_offset(rows) + static_cast<size_t>(rows) * 2 * sizeof(sv::FiltRow);
  return (bytes + 255) / 256 * 256 + 256;
}

int spec_verify_rows(SV_ARGS_DECL) {
  SV_ARGS_PACK;
  const int rc = sv::check_args(a);
  return rc != SV_OK ? rc : sv::run_rows(a, false);
}

int spec_verify_finalize(SV_ARGS_DECL) {
  SV_ARGS_PACK;
  const int rc = sv::check_args(a);
  return rc != SV_OK ? rc : sv::run_finalize(a, false);
}

int spec_verify(SV_ARGS_DECL) {
  SV_ARGS_PACK;
  int rc = sv::check_args(a);
  return rc != SV_OK ? rc : sv::run_call(a);
}

int spec_verify_static(const void* target_logits, const void* draft_logits,
                       const int32_t* draft_tokens, const float* uniforms,
                       const int32_t* verify_lens, const int32_t* row_offsets, int32_t B,
                       int32_t V, int32_t n_target_rows, int32_t max_len, int32_t dtype,
                       float temperature, int32_t top_k, float top_p, int32_t mode,
                       int32_t* out_tokens, int32_t* out_accept_len, float* out_conf,
                       float* out_row_stats, int32_t* dev_error, void* stream) {
  if (n_target_rows > SV_STATIC_MAX_ROWS ||
      spec_verify_workspace_size(B, n_target_rows) > sv::kStaticBytes)
    return SV_ERR_TOO_LARGE;
  // the host checks run first, against a stand-in for the array (aligned,
  // non-null, never dereferenced): a call with bad arguments enqueues nothing,
  // not even the first call's clear of the array
  const size_t workspace_bytes = sv::kStaticBytes;
  void* workspace = reinterpret_cast<void*>(static_cast<uintptr_t>(256));
  SV_ARGS_PACK;
  int rc = sv::check_args(a);
  if (rc != SV_OK) return rc;
  rc = sv::static_workspace(&a.workspace, static_cast<cudaStream_t>(stream));
  return rc != SV_OK ? rc : sv::run_call(a);
}

int spec_verify_schedule(const float* conf, int32_t B, int32_t K, const double* sps,
                         int32_t n_sps, int32_t* out_lens, double* out_theta, void* stream) {
  using sv::aligned;
  if (B < 1 || K < 0 || n_sps <= B || sps == nullptr || out_lens == nullptr ||
      (K > 0 && conf == nullptr))
    return SV_ERR_ARG;
  if ((conf != nullptr && !aligned(conf, 4)) || !aligned(sps, 8) || !aligned(out_lens, 4) ||
      (out_theta != nullptr && !aligned(out_theta, 8)))
    return SV_ERR_ARG;
  const int64_t n = static_cast<int64_t>(B) * K;
  if (n > SV_SCHEDULE_MAX_CANDIDATES || B > SV_SCHEDULE_MAX_CANDIDATES) return SV_ERR_UNSUPPORTED;
  sv::DeviceCache dc;
  const int rc = sv::device_info(&dc);
  if (rc != SV_OK) return rc;
  sv::ScheduleArgs A{conf, B, K, sps, n_sps, out_lens, out_theta,
                     static_cast<int32_t>(std::max<int64_t>(2, (n + 1) & ~int64_t{1}))};
  const int smem = A.npad * (2 * 8 + 2 * 2) + ((B + 1) & ~1) * 4 + sv::kScheduleWarps * (2 * 8 + 4);
  return sv::launch_plain(sv::schedule_kernel, A, 1, sv::kScheduleThreads, smem, dc.max_smem_optin,
                          false, static_cast<cudaStream_t>(stream));
}

const char* spec_verify_status_string(int status) {
  switch (status) {
    case SV_OK: return "ok";
    case SV_ERR_ARG: return "invalid argument (null or misaligned pointer, bad size or parameter)";
    case SV_ERR_DTYPE: return "unknown logits dtype";
    case SV_ERR_CUDA: return "CUDA runtime or launch failure";
    case SV_ERR_UNSUPPORTED:
      return "not served: a shape the kernels do not take";
    case SV_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
    case SV_ERR_TOO_LARGE:
      return "problem larger than the static scratch of spec_verify_static "
             "(more than SV_STATIC_MAX_ROWS target rows)";
    default: return "unknown status";
  }
}

int spec_verify_set_tuning(int32_t knob, int64_t value) {
  std::lock_guard<std::mutex> lock(sv::g_tune_mu);
  sv::Tuning& t = sv::g_tune;
  const sv::Tuning d{};
  const bool dflt = value < 0;
  switch (knob) {
    case SV_TUNE_SLICE:
      if (!dflt && value > (1 << 24)) return SV_ERR_ARG;
      t.slice = dflt ? d.slice : static_cast<int>(value);
      return SV_OK;
    case SV_TUNE_STAGES:
      if (!dflt && (value < sv::kMinStages || value > sv::kMaxStages)) return SV_ERR_ARG;
      t.stages = dflt ? d.stages : static_cast<int>(value);
      return SV_OK;
    case SV_TUNE_WARPS:
      if (!dflt && value != 16 && value != 24) return SV_ERR_ARG;
      t.warps = dflt ? d.warps : static_cast<int>(value);
      return SV_OK;
    case SV_TUNE_PASS1_WARPS:
      if (!dflt && value > 23) return SV_ERR_ARG;
      t.pass1_warps = dflt ? d.pass1_warps : static_cast<int>(value);
      return SV_OK;
    case SV_TUNE_POLL_NS:
      if (!dflt && value > 10000) return SV_ERR_ARG;
      t.poll_ns = dflt ? d.poll_ns : static_cast<int>(value);
      return SV_OK;
    case SV_TUNE_XWAIT_NS:
      if (!dflt && value > static_cast<int64_t>(sv::kWaitLimitNs)) return SV_ERR_ARG;
      t.xwait_ns = dflt ? d.xwait_ns : value;
      return SV_OK;
    default:
      return SV_ERR_ARG;
  }
}

int spec_verify_slices_per_row(int32_t V, int32_t dtype, int32_t top_k, float top_p) {
  (void)top_k;
  (void)top_p;
  if (V <= 0) return SV_ERR_ARG;
  if (dtype != SV_BF16 && dtype != SV_FP32) return SV_ERR_DTYPE;
  sv::DeviceCache dc;
  const int rc = sv::device_info(&dc);
  if (rc != SV_OK) return rc;
  sv::RowsGeom geo;
  const int g = sv::rows_geometry(V, 1, dtype == SV_BF16 ? 2 : 4, dc, &geo);
  return g != SV_OK ? g : geo.S;
}

}  // extern "C"
