// The Hessian accumulation with the activations in host memory: X is copied to the device
// chunk by chunk through two staging buffers, and the copy of the next chunk overlaps the
// Gram products of the current one ("tm_gptq_math", "Why it is second-order: the Hessian":
// H sums over the calibration tokens, so it can be built chunk by chunk).
//
// Copies run on a stream this library creates once per device; the products run on the
// caller's stream.  Per chunk c (staging buffer b = c % 2):
//   copy stream : [wait done[b], i.e. chunk c - 2 consumed] copy chunk c -> buf[b];
//                 record ready[b]
//   caller      : wait ready[b]; H += 2 X_c^T X_c; record done[b]
// The first copy waits for the caller's stream to reach the call, so staging buffers still
// read by earlier work are not overwritten.
#include <algorithm>
#include <mutex>

#include "common.cuh"

namespace gptq {
namespace {

constexpr size_t kChunkBytes = (size_t)64 << 20;

// Default chunk: about kChunkBytes of X, but at least kMinChunkTokens tokens, and at least
// kMinChunkTokensWide from d_in = kWideD on: every chunk's products read and write all of H
// and end in a partial round of tiles, so wide layers need long chunks (at d_in = 28672,
// 64 MiB would be 1024 tokens, and H's 6.6 GB of traffic per chunk would outweigh its
// products; measured there over 65,536 tokens: 69.3 ms with 8192-token chunks, 56.2 with
// 16384, 52.5 with 32768).  Narrower layers are bound by the copies, where a longer first
// chunk only delays the first product (10.45 against 10.65 ms at d_in = 4096).
constexpr int64_t kMinChunkTokens = 8192;
constexpr int64_t kMinChunkTokensWide = 32768;
constexpr int64_t kWideD = 16384;

int64_t chunk_tokens(int64_t d, size_t es, int64_t chunk_tok) {
  if (chunk_tok > 0) return chunk_tok;
  const int64_t t = (int64_t)(kChunkBytes / ((size_t)d * es)) / 512 * 512;
  const int64_t lo = d >= kWideD ? kMinChunkTokensWide : kMinChunkTokens;
  return t < lo ? lo : t;
}

struct CopyStream {
  std::mutex enqueue;  // one call at a time enqueues on these events
  cudaStream_t s = nullptr;
  cudaEvent_t start = nullptr, ready[2] = {nullptr, nullptr}, done[2] = {nullptr, nullptr};
};
constexpr int kMaxDevices = 128;
std::mutex g_mu;
CopyStream g_copy[kMaxDevices];

gptq_status copy_stream(CopyStream **out) {
  int dev = -1;
  GPTQ_CUDA_CHECK(cudaGetDevice(&dev));
  if (dev < 0 || dev >= kMaxDevices) return GPTQ_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_mu);
  CopyStream &cs = g_copy[dev];
  if (!cs.s) {
    GPTQ_CUDA_CHECK(cudaStreamCreateWithFlags(&cs.s, cudaStreamNonBlocking));
    GPTQ_CUDA_CHECK(cudaEventCreateWithFlags(&cs.start, cudaEventDisableTiming));
    for (int b = 0; b < 2; ++b) {
      GPTQ_CUDA_CHECK(cudaEventCreateWithFlags(&cs.ready[b], cudaEventDisableTiming));
      GPTQ_CUDA_CHECK(cudaEventCreateWithFlags(&cs.done[b], cudaEventDisableTiming));
    }
  }
  *out = &cs;
  return GPTQ_OK;
}

}  // namespace

size_t hessian_host_ws_bytes(int64_t d, size_t es, int64_t chunk_tok) {
  const int64_t ct = chunk_tokens(d, es, chunk_tok);
  return 2 * round_up((size_t)ct * (size_t)d * es, 256);
}

gptq_status launch_hessian_host(const void *X_host, int xdtype, size_t es, int64_t n_tok,
                                int64_t d, int64_t ldx, float *H, int accumulate,
                                int64_t chunk_tok, void *ws, cudaStream_t s) {
  if (n_tok == 0) return launch_hessian(nullptr, xdtype, 0, d, d, H, accumulate, nullptr, s);
  const size_t row = (size_t)d * es;
  const int64_t ct = chunk_tokens(d, es, chunk_tok);
  char *buf[2] = {(char *)ws, (char *)ws + round_up((size_t)ct * row, 256)};
  CopyStream *cs = nullptr;
  GPTQ_TRY(copy_stream(&cs));
  std::lock_guard<std::mutex> lock(cs->enqueue);
  GPTQ_CUDA_CHECK(cudaEventRecord(cs->start, s));
  GPTQ_CUDA_CHECK(cudaStreamWaitEvent(cs->s, cs->start, 0));
  int c = 0;
  for (int64_t t0 = 0; t0 < n_tok; t0 += ct, ++c) {
    const int64_t nt = std::min(ct, n_tok - t0);
    const int b = c & 1;
    if (c >= 2) GPTQ_CUDA_CHECK(cudaStreamWaitEvent(cs->s, cs->done[b], 0));
    const char *src = (const char *)X_host + (size_t)t0 * (size_t)ldx * es;
    if (ldx == d) {
      GPTQ_CUDA_CHECK(cudaMemcpyAsync(buf[b], src, (size_t)nt * row, cudaMemcpyHostToDevice,
                                      cs->s));
    } else {
      GPTQ_CUDA_CHECK(cudaMemcpy2DAsync(buf[b], row, src, (size_t)ldx * es, row, (size_t)nt,
                                        cudaMemcpyHostToDevice, cs->s));
    }
    GPTQ_CUDA_CHECK(cudaEventRecord(cs->ready[b], cs->s));
    GPTQ_CUDA_CHECK(cudaStreamWaitEvent(s, cs->ready[b], 0));
    GPTQ_TRY(launch_hessian(buf[b], xdtype, nt, d, d, H, c == 0 ? accumulate : 1, nullptr, s));
    GPTQ_CUDA_CHECK(cudaEventRecord(cs->done[b], s));
  }
  return GPTQ_OK;
}

}  // namespace gptq
