// gptq_quantize_layer_noalloc: the layer sweep for callers that cannot allocate device
// memory themselves -- code that runs inside a host framework which owns the device
// memory pool and forbids allocations on its hot path, or code that must never trigger
// the device-wide synchronization that cudaMalloc/cudaFree can imply.  Instead of a
// caller workspace it uses a fixed scratch array that is part of this library's device
// image, so a call allocates nothing.
//
// The array is GPTQ_NOALLOC_SCRATCH_BYTES (32 MiB) on every GPU where the library's device
// code holding it has been loaded, and stays there until the process exits.  Under CUDA's
// default lazy module loading that happens at the first call on a device (the address
// look-up below loads it): that first call reserves the 32 MiB and may synchronize, so it
// belongs in the caller's set-up; later calls allocate nothing.  All calls on a device share
// the array, and it keeps the contents of the last call; the sweep overwrites every scratch
// byte it reads and clears its status block at the start of each call, so nothing needs to
// be zeroed beforehand.  Two calls whose work overlaps on the GPU (different streams, no
// ordering between them) race on the array and produce garbage: order them on one stream.
// The status block at the start of the array (non-finite weights, a bounded wait that gave
// up) is read back by gptq_noalloc_status.
#include <mutex>

#include "common.cuh"

namespace gptq {
namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[GPTQ_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 128;
std::mutex g_mu;
void *g_scratch_ptr[kMaxDevices];  // device address of g_noalloc_scratch, per device

// The array's name is only a host-side stand-in in host code; the device address must be
// looked up once per device, with that device current.
gptq_status scratch_address(void **out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    (void)cudaGetLastError();
    return GPTQ_ERR_CUDA;
  }
  if (dev < 0 || dev >= kMaxDevices) return GPTQ_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_ptr[dev]) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) {
      (void)cudaGetLastError();
      return GPTQ_ERR_CUDA;
    }
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return GPTQ_OK;
}

}  // namespace
}  // namespace gptq

extern "C" gptq_status gptq_quantize_layer_noalloc(
    const void *W, int wdtype, int64_t d_out, int64_t d_in, int64_t ldw, const float *U,
    const uint8_t *dead_mask, int bits, int block, uint32_t *qpacked, float *scale,
    int32_t *zero, float *W_hat, gptq_stream_t stream) {
  // Size check first: a layer whose scratch exceeds the fixed array is refused before
  // anything touches the GPU.
  if (d_out < 1 || d_in < 1) return GPTQ_ERR_INVALID_ARG;
  if (block < 1 || block > 128) return GPTQ_ERR_INVALID_ARG;
  const size_t need = gptq_quantize_workspace_bytes(d_out, d_in, bits, block);
  if (need == 0) return GPTQ_ERR_INVALID_ARG;
  if (need > (size_t)GPTQ_NOALLOC_SCRATCH_BYTES) return GPTQ_ERR_WORKSPACE;
  void *scratch = nullptr;
  const gptq_status st = gptq::scratch_address(&scratch);
  if (st != GPTQ_OK) return st;
  // one stream only: the two-stream schedule would create streams and events on first use
  return gptq::quantize_layer_checked(W, wdtype, d_out, d_in, ldw, U, dead_mask, bits, block,
                                      qpacked, scale, zero, W_hat, scratch,
                                      (size_t)GPTQ_NOALLOC_SCRATCH_BYTES, stream, false);
}

extern "C" gptq_status gptq_noalloc_status(gptq_stream_t stream) {
  void *scratch = nullptr;
  const gptq_status st = gptq::scratch_address(&scratch);
  if (st != GPTQ_OK) return st;
  cudaStream_t s = (cudaStream_t)stream;
  gptq::DevStatus ds;
  GPTQ_CUDA_CHECK(cudaMemcpyAsync(&ds, scratch, sizeof(ds), cudaMemcpyDeviceToHost, s));
  GPTQ_CUDA_CHECK(cudaStreamSynchronize(s));
  return (gptq_status)ds.status;
}
