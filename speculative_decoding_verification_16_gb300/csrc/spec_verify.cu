// spec_verify.cu -- host side of the C ABI declared in include/spec_verify.h.
//
// Argument checks happen on the host before anything is enqueued; every
// entry point only enqueues kernels on the caller's stream and never
// synchronises.  Nothing here allocates device memory: all scratch comes
// from the caller's workspace.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <mutex>

#include "spec_verify.h"
#include "sv_common.cuh"
#include "sv_finalize.cuh"
#include "sv_rows.cuh"

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

int env_int(const char* name, int dflt) {
  const char* v = std::getenv(name);
  return v ? std::atoi(v) : dflt;
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

int slice_len(int V, int C, int es) { return round_up((V + C - 1) / C, 16 / es); }

bool is_filtered(int V, int top_k, float top_p) {
  return (top_k > 0 && top_k < V) || top_p < 1.0f;
}

// Cluster size of the rows kernel: the smallest C in {1, 2, 4, 8, 16} whose
// slice pair fits the shared-memory budget (SPEC_VERIFY_SMEM_BUDGET bytes,
// default 80 KiB: two CTAs per SM); SPEC_VERIFY_CLUSTER forces a size.
int rows_cluster(int V, int es, const DeviceCache& dc, int* smem_out) {
  const int forced = env_int("SPEC_VERIFY_CLUSTER", 0);
  const int budget = env_int("SPEC_VERIFY_SMEM_BUDGET", 80 * 1024);
  if (forced > 0) {
    if (forced > kMaxCluster) return SV_ERR_UNSUPPORTED;
    const int smem = kHdrBytes + 2 * rowbuf_bytes(slice_len(V, forced, es), es);
    if (smem > dc.max_smem_optin) return SV_ERR_UNSUPPORTED;
    *smem_out = smem;
    return forced;
  }
  for (int C = 1; C <= kMaxCluster; C *= 2) {
    const int smem = kHdrBytes + 2 * rowbuf_bytes(slice_len(V, C, es), es);
    if (smem > dc.max_smem_optin) continue;
    if (smem <= budget || C == kMaxCluster) {
      *smem_out = smem;
      return C;
    }
  }
  return SV_ERR_UNSUPPORTED;
}

// Cluster size of the unfiltered final draw (one request per cluster).
int draw_cluster(int V, int es, const DeviceCache& dc, int* smem_out) {
  const int forced = env_int("SPEC_VERIFY_DRAW_CLUSTER", 0);
  for (int C = kMaxCluster; C >= 1; C /= 2) {
    if (forced > 0 && C != forced) continue;
    const int S = slice_len(V, C, es);
    const int smem = kF_HdrBytes + 2 * rowbuf_bytes(S, es);
    if (smem <= dc.max_smem_optin) {
      *smem_out = smem;
      return C;
    }
  }
  return SV_ERR_UNSUPPORTED;
}

template <typename K>
cudaError_t prepare_kernel(K kernel, int smem, int cluster) {
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e == cudaSuccess && cluster > 8)
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  return e;
}

template <typename K>
int launch_cluster(K kernel, const Params& P, int nclusters, int C, int smem, cudaStream_t stream) {
  if (prepare_kernel(kernel, smem, C) != cudaSuccess) return SV_ERR_CUDA;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(nclusters) * C, 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = C;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int active = 0;
  if (cudaOccupancyMaxActiveClusters(&active, kernel, &cfg) != cudaSuccess) return SV_ERR_CUDA;
  if (active <= 0) return SV_ERR_UNSUPPORTED;
  if (cudaLaunchKernelEx(&cfg, kernel, P) != cudaSuccess) return SV_ERR_CUDA;
  return SV_OK;
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
  if (a.workspace == nullptr || !aligned(a.workspace, 256) ||
      a.workspace_bytes < spec_verify_workspace_size(a.B, a.n_target_rows))
    return SV_ERR_WORKSPACE;
  if (is_filtered(a.V, a.top_k, a.top_p)) return SV_ERR_UNSUPPORTED;  // served by a later kernel
  return SV_OK;
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
  P.top_k = (a.top_k > 0 && a.top_k < a.V) ? a.top_k : 0;
  P.top_p = a.top_p;
  P.mode = a.mode;
  P.out_tokens = a.out_tokens;
  P.out_accept_len = a.out_accept_len;
  P.out_conf = a.out_conf;
  P.out_row_stats = a.out_row_stats;
  P.dev_error = a.dev_error;
  P.rec = static_cast<RowRec*>(a.workspace);
  return P;
}

int run_rows(const Args& a) {
  DeviceCache dc;
  int rc = device_info(&dc);
  if (rc != SV_OK) return rc;
  Params P = make_params(a);
  const int es = a.dtype == SV_BF16 ? 2 : 4;
  int smem = 0;
  const int C = rows_cluster(a.V, es, dc, &smem);
  if (C < 0) return C;
  P.S = slice_len(a.V, C, es);
  P.rowbuf = rowbuf_bytes(P.S, es);
  const bool need_z = a.mode == SV_SAMPLE || a.out_conf != nullptr || a.out_row_stats != nullptr;
  const bool need_conf = a.out_conf != nullptr;
  cudaStream_t st = static_cast<cudaStream_t>(a.stream);
#define SV_ROWS(ES, Z, CF) launch_cluster(rows_kernel<ES, Z, CF>, P, a.n_target_rows, C, smem, st)
  if (es == 2) {
    if (need_conf) rc = SV_ROWS(2, true, true);
    else if (need_z) rc = SV_ROWS(2, true, false);
    else rc = SV_ROWS(2, false, false);
  } else {
    if (need_conf) rc = SV_ROWS(4, true, true);
    else if (need_z) rc = SV_ROWS(4, true, false);
    else rc = SV_ROWS(4, false, false);
  }
#undef SV_ROWS
  return rc;
}

int run_finalize(const Args& a) {
  DeviceCache dc;
  int rc = device_info(&dc);
  if (rc != SV_OK) return rc;
  Params P = make_params(a);
  const int es = a.dtype == SV_BF16 ? 2 : 4;
  cudaStream_t st = static_cast<cudaStream_t>(a.stream);
  const bool filtered = P.top_k > 0 || P.top_p < 1.f;
  if (a.mode == SV_GREEDY || filtered) {
    finalize_select_kernel<<<(a.B + kThreads - 1) / kThreads, kThreads, 0, st>>>(P);
    return cudaGetLastError() == cudaSuccess ? SV_OK : SV_ERR_CUDA;
  }
  int smem = 0;
  const int C4 = draw_cluster(a.V, es, dc, &smem);
  if (C4 < 0) return C4;
  P.S4 = slice_len(a.V, C4, es);
  P.rowbuf4 = rowbuf_bytes(P.S4, es);
  if (es == 2) return launch_cluster(finalize_draw_kernel<2>, P, a.B, C4, smem, st);
  return launch_cluster(finalize_draw_kernel<4>, P, a.B, C4, smem, st);
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
  const size_t rows = n_target_rows > 0 ? static_cast<size_t>(n_target_rows) : 0;
  const size_t bytes = rows * sizeof(sv::RowRec);
  return (bytes + 255) / 256 * 256 + 256;
}

int spec_verify_rows(SV_ARGS_DECL) {
  SV_ARGS_PACK;
  const int rc = sv::check_args(a);
  return rc != SV_OK ? rc : sv::run_rows(a);
}

int spec_verify_finalize(SV_ARGS_DECL) {
  SV_ARGS_PACK;
  const int rc = sv::check_args(a);
  return rc != SV_OK ? rc : sv::run_finalize(a);
}

int spec_verify(SV_ARGS_DECL) {
  SV_ARGS_PACK;
  int rc = sv::check_args(a);
  if (rc == SV_OK) rc = sv::run_rows(a);
  if (rc == SV_OK) rc = sv::run_finalize(a);
  return rc;
}

const char* spec_verify_status_string(int status) {
  switch (status) {
    case SV_OK: return "ok";
    case SV_ERR_ARG: return "invalid argument (null or misaligned pointer, bad size or parameter)";
    case SV_ERR_DTYPE: return "unknown logits dtype";
    case SV_ERR_CUDA: return "CUDA runtime or launch failure";
    case SV_ERR_UNSUPPORTED: return "filter combination or cluster shape not supported";
    case SV_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
    default: return "unknown status";
  }
}

int spec_verify_cluster_size(int32_t V, int32_t dtype, int32_t top_k, float top_p) {
  (void)top_k;
  (void)top_p;
  if (V <= 0) return SV_ERR_ARG;
  if (dtype != SV_BF16 && dtype != SV_FP32) return SV_ERR_DTYPE;
  sv::DeviceCache dc;
  const int rc = sv::device_info(&dc);
  if (rc != SV_OK) return rc;
  int smem = 0;
  return sv::rows_cluster(V, dtype == SV_BF16 ? 2 : 4, dc, &smem);
}

}  // extern "C"
