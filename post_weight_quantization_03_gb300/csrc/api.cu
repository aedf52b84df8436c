// C ABI entry points: argument validation, workspace sizing, launch sequencing.
#include <atomic>
#include <mutex>
#include <vector>

#include "common.cuh"

namespace gptq {

static std::atomic<unsigned long long> g_launches{0};
void count_launch(unsigned n) { g_launches.fetch_add(n, std::memory_order_relaxed); }
unsigned long long launches_so_far() { return g_launches.load(); }

namespace {
struct AttrEntry {
  const void *func;
  int dev;
  int bytes;
};
std::mutex g_attr_mu;
std::vector<AttrEntry> g_attrs;            // (kernel, device) pairs already set
constexpr int kMaxSmDevices = 128;
std::atomic<int> g_sm_count[kMaxSmDevices];  // 0 = not yet queried
}  // namespace

gptq_status ensure_smem_attr(const void *func, int bytes) {
  int dev = -1;
  GPTQ_CUDA_CHECK(cudaGetDevice(&dev));
  std::lock_guard<std::mutex> lock(g_attr_mu);
  for (const AttrEntry &e : g_attrs)
    if (e.func == func && e.dev == dev && e.bytes >= bytes) return GPTQ_OK;
  GPTQ_CUDA_CHECK(cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes));
  g_attrs.push_back(AttrEntry{func, dev, bytes});
  return GPTQ_OK;
}

gptq_status device_sm_count(int *out) {
  int dev = -1;
  GPTQ_CUDA_CHECK(cudaGetDevice(&dev));
  if (dev < 0 || dev >= kMaxSmDevices) return GPTQ_ERR_UNSUPPORTED;
  int n = g_sm_count[dev].load(std::memory_order_relaxed);
  if (n == 0) {
    GPTQ_CUDA_CHECK(cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev));
    g_sm_count[dev].store(n, std::memory_order_relaxed);
  }
  *out = n;
  return GPTQ_OK;
}

static bool aligned(const void *p, size_t a) { return ((uintptr_t)p % a) == 0; }

static size_t elem_size(int dt) {
  switch (dt) {
    case GPTQ_F16:
    case GPTQ_BF16: return 2;
    case GPTQ_F32: return 4;
    default: return 0;
  }
}


gptq_status quantize_layer_checked(const void *W, int wdtype, int64_t d_out,
                                         int64_t d_in, int64_t ldw, const float *U,
                                         const uint8_t *dead_mask, int bits, int block,
                                         uint32_t *qpacked, float *scale, int32_t *zero,
                                         float *W_hat, void *ws, size_t ws_bytes,
                                         gptq_stream_t stream, bool allow_overlap) {
  const size_t es = elem_size(wdtype);
  if (es == 0 || !W || !U || !qpacked || !scale || !zero) return GPTQ_ERR_INVALID_ARG;
  if (d_out < 1 || d_in < 1 || ldw < d_in) return GPTQ_ERR_INVALID_ARG;
  if (!(bits == 2 || bits == 3 || bits == 4 || bits == 8)) return GPTQ_ERR_INVALID_ARG;
  if (block < 1 || block > 128) return GPTQ_ERR_INVALID_ARG;
  if (!aligned(W, es) || !aligned(U, 16) || !aligned(qpacked, 4) || !aligned(scale, 4) ||
      !aligned(zero, 4) || (W_hat && !aligned(W_hat, 4)))
    return GPTQ_ERR_INVALID_ARG;
  if (d_in > (int64_t)1 << 17 || d_out > (int64_t)1 << 24) return GPTQ_ERR_UNSUPPORTED;
  if (!ws || !aligned(ws, 256) || ws_bytes < quantize_ws_bytes(d_out, d_in, bits, block))
    return GPTQ_ERR_WORKSPACE;
  return launch_quantize(W, wdtype, d_out, d_in, ldw, U, dead_mask, bits, block, qpacked,
                         scale, zero, W_hat, ws, (cudaStream_t)stream, allow_overlap);
}

}  // namespace gptq

using namespace gptq;

extern "C" {

const char *gptq_status_str(int status) {
  switch (status) {
    case GPTQ_OK: return "GPTQ_OK";
    case GPTQ_ERR_INVALID_ARG: return "GPTQ_ERR_INVALID_ARG";
    case GPTQ_ERR_NOT_PD: return "GPTQ_ERR_NOT_PD";
    case GPTQ_ERR_NONFINITE: return "GPTQ_ERR_NONFINITE";
    case GPTQ_ERR_TIMEOUT: return "GPTQ_ERR_TIMEOUT";
    case GPTQ_ERR_CUDA: return "GPTQ_ERR_CUDA";
    case GPTQ_ERR_UNSUPPORTED: return "GPTQ_ERR_UNSUPPORTED";
    case GPTQ_ERR_WORKSPACE: return "GPTQ_ERR_WORKSPACE";
    default: return "GPTQ_ERR_UNKNOWN";
  }
}

int gptq_abi_version(void) { return GPTQ_ABI_VERSION; }

unsigned long long gptq_kernel_launches(void) { return g_launches.load(); }

gptq_status gptq_hessian_accumulate(const void *X, int xdtype, int64_t n_tok, int64_t d_in,
                                    int64_t ldx, float *H, int accumulate,
                                    gptq_stream_t stream) {
  const size_t es = elem_size(xdtype);
  if (es == 0 || n_tok < 0 || d_in < 1 || ldx < d_in || !H) return GPTQ_ERR_INVALID_ARG;
  if (n_tok > 0 && (!X || !aligned(X, 16) || (ldx * (int64_t)es) % 16 != 0))
    return GPTQ_ERR_INVALID_ARG;
  if (!aligned(H, 16)) return GPTQ_ERR_INVALID_ARG;
  if (d_in > (int64_t)1 << 20) return GPTQ_ERR_UNSUPPORTED;
  return launch_hessian(X, xdtype, n_tok, d_in, ldx, H, accumulate ? 1 : 0, nullptr,
                        (cudaStream_t)stream);
}

size_t gptq_hessian_host_workspace_bytes(int xdtype, int64_t d_in, int64_t chunk_tok) {
  const size_t es = elem_size(xdtype);
  if (es == 0 || d_in < 1 || chunk_tok < 0) return 0;
  return hessian_host_ws_bytes(d_in, es, chunk_tok);
}

gptq_status gptq_hessian_accumulate_host(const void *X_host, int xdtype, int64_t n_tok,
                                         int64_t d_in, int64_t ldx, float *H, int accumulate,
                                         int64_t chunk_tok, void *ws, size_t ws_bytes,
                                         gptq_stream_t stream) {
  const size_t es = elem_size(xdtype);
  if (es == 0 || n_tok < 0 || d_in < 1 || ldx < d_in || chunk_tok < 0 || !H)
    return GPTQ_ERR_INVALID_ARG;
  if (n_tok > 0 && !X_host) return GPTQ_ERR_INVALID_ARG;
  if (!aligned(H, 16) || (d_in * (int64_t)es) % 16 != 0) return GPTQ_ERR_INVALID_ARG;
  if (d_in > (int64_t)1 << 20) return GPTQ_ERR_UNSUPPORTED;
  if (!ws || !aligned(ws, 256) || ws_bytes < hessian_host_ws_bytes(d_in, es, chunk_tok))
    return GPTQ_ERR_WORKSPACE;
  return launch_hessian_host(X_host, xdtype, es, n_tok, d_in, ldx, H, accumulate ? 1 : 0,
                             chunk_tok, ws, (cudaStream_t)stream);
}

size_t gptq_prepare_workspace_bytes(int64_t d_in) {
  if (d_in < 1) return 0;
  return prepare_ws_bytes(d_in);
}

gptq_status gptq_prepare(float *H, int64_t d_in, float damp, float *U, uint8_t *dead_mask,
                         int32_t *n_dead, void *ws, size_t ws_bytes, gptq_stream_t stream) {
  if (!H || !U || d_in < 1 || !(damp >= 0.0f) || !aligned(H, 16) || !aligned(U, 16))
    return GPTQ_ERR_INVALID_ARG;
  if (d_in > (int64_t)1 << 17) return GPTQ_ERR_UNSUPPORTED;
  if (!ws || !aligned(ws, 256) || ws_bytes < prepare_ws_bytes(d_in)) return GPTQ_ERR_WORKSPACE;
  cudaStream_t s = (cudaStream_t)stream;
  GPTQ_TRY(launch_prepare(H, d_in, damp, U, dead_mask, ws, s));
  DevStatus st;
  GPTQ_CUDA_CHECK(cudaMemcpyAsync(&st, ws, sizeof(DevStatus), cudaMemcpyDeviceToHost, s));
  GPTQ_CUDA_CHECK(cudaStreamSynchronize(s));
  if (n_dead) *n_dead = st.n_dead;
  return (gptq_status)st.status;
}

size_t gptq_quantize_workspace_bytes(int64_t d_out, int64_t d_in, int bits, int block) {
  if (d_out < 1 || d_in < 1) return 0;
  return quantize_ws_bytes(d_out, d_in, bits, block);
}


size_t gptq_quantize_shared_workspace_bytes(int n_layers, const int64_t *d_out, int64_t d_in,
                                            int bits, int block) {
  if (n_layers < 1 || n_layers > GPTQ_MAX_SHARED_LAYERS || !d_out || d_in < 1) return 0;
  for (int i = 0; i < n_layers; ++i)
    if (d_out[i] < 1) return 0;
  return quantize_layers_ws_bytes(d_out, n_layers, d_in, bits, block);
}

gptq_status gptq_quantize_layers_shared(int n_layers, const void *const *W, const int *wdtype,
                                        const int64_t *d_out, const int64_t *ldw, int64_t d_in,
                                        const float *U, const uint8_t *dead_mask, int bits,
                                        int block, uint32_t *const *qpacked,
                                        float *const *scale, int32_t *const *zero,
                                        float *const *W_hat, void *ws, size_t ws_bytes,
                                        gptq_stream_t stream) {
  if (n_layers < 1 || n_layers > GPTQ_MAX_SHARED_LAYERS) return GPTQ_ERR_INVALID_ARG;
  if (!W || !wdtype || !d_out || !ldw || !qpacked || !scale || !zero || !U || d_in < 1)
    return GPTQ_ERR_INVALID_ARG;
  if (!(bits == 2 || bits == 3 || bits == 4 || bits == 8)) return GPTQ_ERR_INVALID_ARG;
  if (block < 1 || block > 128 || !aligned(U, 16)) return GPTQ_ERR_INVALID_ARG;
  QLayer L[GPTQ_MAX_SHARED_LAYERS];
  int64_t rows = 0;
  for (int i = 0; i < n_layers; ++i) {
    const size_t es = elem_size(wdtype[i]);
    float *wh = W_hat ? W_hat[i] : nullptr;
    if (es == 0 || !W[i] || !qpacked[i] || !scale[i] || !zero[i]) return GPTQ_ERR_INVALID_ARG;
    if (d_out[i] < 1 || ldw[i] < d_in) return GPTQ_ERR_INVALID_ARG;
    if (!aligned(W[i], es) || !aligned(qpacked[i], 4) || !aligned(scale[i], 4) ||
        !aligned(zero[i], 4) || (wh && !aligned(wh, 4)))
      return GPTQ_ERR_INVALID_ARG;
    rows += d_out[i];
    L[i] = QLayer{W[i], wdtype[i], d_out[i], ldw[i], qpacked[i], scale[i], zero[i], wh};
  }
  if (d_in > (int64_t)1 << 17 || rows > (int64_t)1 << 24) return GPTQ_ERR_UNSUPPORTED;
  if (!ws || !aligned(ws, 256) ||
      ws_bytes < quantize_layers_ws_bytes(d_out, n_layers, d_in, bits, block))
    return GPTQ_ERR_WORKSPACE;
  return launch_quantize_layers(L, n_layers, d_in, U, dead_mask, bits, block, ws,
                                (cudaStream_t)stream, true);
}

size_t gptq_recon_error_workspace_bytes(int xdtype, int64_t d_out, int64_t d_in,
                                        int64_t n_tok) {
  if (elem_size(xdtype) == 0 || d_out < 1 || d_in < 1 || n_tok < 0) return 0;
  return recon_ws_bytes(xdtype, d_out, d_in, n_tok);
}

gptq_status gptq_recon_error(const void *X, int xdtype, int64_t n_tok, int64_t d_in,
                             int64_t ldx, const void *W, int wdtype, int64_t d_out, int64_t ldw,
                             const uint32_t *qpacked, int bits, const float *scale,
                             const int32_t *zero, float *err, void *ws, size_t ws_bytes,
                             gptq_stream_t stream) {
  const size_t xes = elem_size(xdtype), wes = elem_size(wdtype);
  if (xes == 0 || wes == 0 || n_tok < 0 || d_in < 1 || d_out < 1 || ldx < d_in ||
      ldw < d_in || !W || !qpacked || !scale || !zero || !err)
    return GPTQ_ERR_INVALID_ARG;
  if (!(bits == 2 || bits == 3 || bits == 4 || bits == 8)) return GPTQ_ERR_INVALID_ARG;
  if (n_tok > 0 && (!X || !aligned(X, 16) || (ldx * (int64_t)xes) % 16 != 0))
    return GPTQ_ERR_INVALID_ARG;
  if (!aligned(W, wes) || !aligned(qpacked, 4) || !aligned(scale, 4) || !aligned(zero, 4) ||
      !aligned(err, 4))
    return GPTQ_ERR_INVALID_ARG;
  if (d_in > (int64_t)1 << 20 || d_out > (int64_t)1 << 24 || n_tok > (int64_t)1 << 31)
    return GPTQ_ERR_UNSUPPORTED;
  if (!ws || !aligned(ws, 256) || ws_bytes < recon_ws_bytes(xdtype, d_out, d_in, n_tok))
    return GPTQ_ERR_WORKSPACE;
  return launch_recon(X, xdtype, n_tok, d_in, ldx, W, wdtype, d_out, ldw, qpacked, bits, scale,
                      zero, err, ws, (cudaStream_t)stream);
}

size_t gptq_quantize_obq_workspace_bytes(int64_t d_out, int64_t d_in) {
  if (d_out < 1 || d_in < 1) return 0;
  return quantize_obq_ws_bytes(d_out, d_in);
}

gptq_status gptq_quantize_obq(const void *W, int wdtype, int64_t d_out, int64_t d_in,
                              int64_t ldw, const float *U, const uint8_t *dead_mask, int bits,
                              uint32_t *qpacked, float *scale, int32_t *zero, float *W_hat,
                              int32_t *order, void *ws, size_t ws_bytes, gptq_stream_t stream) {
  const size_t es = elem_size(wdtype);
  if (es == 0 || !W || !U || !qpacked || !scale || !zero) return GPTQ_ERR_INVALID_ARG;
  if (d_out < 1 || d_in < 1 || ldw < d_in) return GPTQ_ERR_INVALID_ARG;
  if (!(bits == 2 || bits == 3 || bits == 4 || bits == 8)) return GPTQ_ERR_INVALID_ARG;
  if (!aligned(W, es) || !aligned(U, 4) || !aligned(qpacked, 4) || !aligned(scale, 4) ||
      !aligned(zero, 4) || (W_hat && !aligned(W_hat, 4)) || (order && !aligned(order, 4)))
    return GPTQ_ERR_INVALID_ARG;
  if (d_in > GPTQ_OBQ_MAX_D_IN || d_out > (int64_t)1 << 24) return GPTQ_ERR_UNSUPPORTED;
  if (!ws || !aligned(ws, 256) || ws_bytes < quantize_obq_ws_bytes(d_out, d_in))
    return GPTQ_ERR_WORKSPACE;
  return launch_quantize_obq(W, wdtype, d_out, d_in, ldw, U, dead_mask, bits, qpacked, scale,
                             zero, W_hat, order, ws, (cudaStream_t)stream);
}

gptq_status gptq_quantize_layer(const void *W, int wdtype, int64_t d_out, int64_t d_in,
                                int64_t ldw, const float *U, const uint8_t *dead_mask,
                                int bits, int block, uint32_t *qpacked, float *scale,
                                int32_t *zero, float *W_hat, void *ws, size_t ws_bytes,
                                gptq_stream_t stream) {
  return gptq::quantize_layer_checked(W, wdtype, d_out, d_in, ldw, U, dead_mask, bits, block,
                                      qpacked, scale, zero, W_hat, ws, ws_bytes, stream, true);
}

gptq_status gptq_debug_hessian_lost_stage(const void *X, int xdtype, int64_t n_tok,
                                          int64_t d_in, int64_t ldx, float *H,
                                          int64_t lost_stage, uint64_t wait_ns, void *status_ws,
                                          gptq_stream_t stream) {
  const size_t es = elem_size(xdtype);
  if (es == 0 || n_tok < 1 || d_in < 1 || ldx < d_in || !X || !H || !status_ws)
    return GPTQ_ERR_INVALID_ARG;
  if (!aligned(X, 16) || (ldx * (int64_t)es) % 16 != 0 || !aligned(H, 16))
    return GPTQ_ERR_INVALID_ARG;
  if (!aligned(status_ws, 256)) return GPTQ_ERR_WORKSPACE;
  if (wait_ns < 1000 || wait_ns > 10000000000ull) return GPTQ_ERR_INVALID_ARG;
  cudaStream_t s = (cudaStream_t)stream;
  GPTQ_CUDA_CHECK(cudaMemsetAsync(status_ws, 0, sizeof(DevStatus), s));
  GPTQ_TRY(launch_hessian_lost_stage(X, xdtype, n_tok, d_in, ldx, H, lost_stage, wait_ns,
                                     (DevStatus *)status_ws, s));
  DevStatus st;
  GPTQ_CUDA_CHECK(cudaMemcpyAsync(&st, status_ws, sizeof(DevStatus), cudaMemcpyDeviceToHost, s));
  GPTQ_CUDA_CHECK(cudaStreamSynchronize(s));
  return (gptq_status)st.status;
}

gptq_status gptq_workspace_status(const void *ws, gptq_stream_t stream) {
  if (!ws || !aligned(ws, 256)) return GPTQ_ERR_WORKSPACE;
  cudaStream_t s = (cudaStream_t)stream;
  DevStatus st;
  GPTQ_CUDA_CHECK(cudaMemcpyAsync(&st, ws, sizeof(DevStatus), cudaMemcpyDeviceToHost, s));
  GPTQ_CUDA_CHECK(cudaStreamSynchronize(s));
  return (gptq_status)st.status;
}

}  // extern "C"
