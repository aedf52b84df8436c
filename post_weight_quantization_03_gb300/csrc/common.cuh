// Internal definitions shared by the library's translation units.
#pragma once

#include <cuda_runtime.h>
#include <cuda_fp16.h>
#include <cuda_bf16.h>
#include <stdint.h>
#include <stddef.h>

#include "../../include/gptq.h"

namespace gptq {

// ----------------------------------------------------------------------------------------
// Host-side bookkeeping
// ----------------------------------------------------------------------------------------

// Counts every kernel this library launches (reported by gptq_kernel_launches()).
void count_launch(unsigned n = 1);

// The dynamic shared-memory limit of a kernel is an attribute of the (function, device)
// pair: sets it to at least `bytes` for `func` on the current device, once per pair, under
// a lock (so that calls from several host threads and on several devices are safe).
gptq_status ensure_smem_attr(const void *func, int bytes);

// Number of SMs of the current device (queried once per device).
gptq_status device_sm_count(int *out);

#define GPTQ_LAUNCH_CHECK()                                   \
  do {                                                        \
    ::gptq::count_launch();                                   \
    if (cudaPeekAtLastError() != cudaSuccess) {               \
      (void)cudaGetLastError();                               \
      return GPTQ_ERR_CUDA;                                   \
    }                                                         \
  } while (0)

#define GPTQ_CUDA_CHECK(call)                                 \
  do {                                                        \
    if ((call) != cudaSuccess) {                              \
      (void)cudaGetLastError();                               \
      return GPTQ_ERR_CUDA;                                   \
    }                                                         \
  } while (0)

#define GPTQ_TRY(expr)                                        \
  do {                                                        \
    gptq_status _s = (expr);                                  \
    if (_s != GPTQ_OK) return _s;                             \
  } while (0)

static inline size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Launches `kern` on `s` (arguments converted to the kernel's parameter types), counts the
// launch and maps a launch error to GPTQ_ERR_CUDA.
template <typename... KArgs, typename... Args>
gptq_status launch_kernel(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                          cudaStream_t s, Args &&...args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  count_launch();
  if (cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...) != cudaSuccess) {
    (void)cudaGetLastError();
    return GPTQ_ERR_CUDA;
  }
  return GPTQ_OK;
}
static inline int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Device-side status block at the start of every workspace.
struct DevStatus {
  int status;        // gptq_status recorded by kernels (0 = OK); first writer wins
  int info;          // NOT_PD: first failing pivot (global index) + 1
  int n_dead;        // number of dead columns
  int pad0;
  double lam;        // damping actually added
  double diag_sum;   // sum of the (dead-fixed) diagonal
  unsigned long long pad[4];
};
static_assert(sizeof(DevStatus) <= 256, "status block must fit in 256 bytes");

// Records `code` unless a status is already recorded.
__device__ __forceinline__ void set_status(DevStatus *st, int code) {
  atomicCAS(&st->status, 0, code);
}

// ----------------------------------------------------------------------------------------
// Element loads
// ----------------------------------------------------------------------------------------
__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__half x) { return __half2float(x); }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }

// Splits x into a TF32-representable head (low 13 mantissa bits cleared) and the exact
// remainder x - head, so that head*y_head + head*y_tail + tail*y_head reproduces a fp32
// product to about 2^-21 relative on a TF32 tensor core (the "3xTF32" scheme).
__device__ __forceinline__ float tf32_head(float x) {
  return __uint_as_float(__float_as_uint(x) & 0xFFFFE000u);
}

// ----------------------------------------------------------------------------------------
// Kernel launchers implemented in the .cu files (all enqueue on `s`, return a status)
// ----------------------------------------------------------------------------------------

// hessian.cu
// `st` (may be null) receives TIMEOUT if a bounded wait of the tensor-core kernel gives up.
gptq_status launch_hessian(const void *X, int xdtype, int64_t n_tok, int64_t d, int64_t ldx,
                           float *H, int accumulate, DevStatus *st, cudaStream_t s);

// Test hook of the bounded waits: the fp16/bf16 tensor-core Hessian with its producer
// skipping token stage `lost_stage` (no copy, no arrival) and every wait limited to wait_ns.
gptq_status launch_hessian_lost_stage(const void *X, int xdtype, int64_t n_tok, int64_t d,
                                      int64_t ldx, float *H, int64_t lost_stage,
                                      uint64_t wait_ns, DevStatus *st, cudaStream_t s);

// host_stream.cu: X streamed from host memory in chunks (see gptq_hessian_accumulate_host)
size_t hessian_host_ws_bytes(int64_t d, size_t es, int64_t chunk_tok);
gptq_status launch_hessian_host(const void *X_host, int xdtype, size_t es, int64_t n_tok,
                                int64_t d, int64_t ldx, float *H, int accumulate,
                                int64_t chunk_tok, void *ws, cudaStream_t s);

// recon.cu: per-row ||(W - W_hat) X^T||^2 on X (gptq_recon_error)
size_t recon_ws_bytes(int xdtype, int64_t m, int64_t d, int64_t n);
gptq_status launch_recon(const void *X, int xdtype, int64_t n, int64_t d, int64_t ldx,
                         const void *W, int wdtype, int64_t m, int64_t ldw, const uint32_t *qp,
                         int bits, const float *scale, const int32_t *zero, float *err,
                         void *ws, cudaStream_t s);

// gemm.cu: C[m, n] (+)= alpha * sum_k A[m, k] * B[n, k], operands given as a TF32 head
// and tail pair each (tail may be null = 0).  lower_only skips tiles strictly above the
// diagonal of C (C's row and column offsets equal, M >= N: a lower trapezoid; tiles on the
// diagonal are computed whole).  trans_c stores C(m, n) at C[n * ldc + m].
struct GemmArgs {
  const float *a_hi, *a_lo; int64_t lda;
  const float *b_hi, *b_lo; int64_t ldb;
  float *c; int64_t ldc;
  int64_t M, N, K;
  float alpha;
  int lower_only;
  int trans_c;
  int max_ctas;   // tensor-core path: at most this many persistent CTAs (0 = one per SM;
                  // -1 = one CTA per tile, so SMs free up tile by tile for other streams)
  int one_sum;    // tensor-core path: 1 = all three products of a tile in one TMEM sum
                  // (the sweep's updates); 0 = head products in sums of two 32-wide K
                  // stages and the cross products apart (the factorization's updates,
                  // whose accuracy needs the short sums)
  int wide;       // tensor-core path, one-sum products that are not triangles: 256-wide
                  // output tiles (fewer operand bytes per product; half the tiles)
};
gptq_status launch_gemm_nt(const GemmArgs &g, DevStatus *st, cudaStream_t s);
// tc_gemm.cu: the tcgen05 3xTF32 kernel; UNSUPPORTED when the operands do not meet its
// alignment requirements (launch_gemm_nt then takes the CUDA-core kernel).
gptq_status launch_gemm_nt_tc(const GemmArgs &g, DevStatus *st, cudaStream_t s);

// factor.cu
gptq_status launch_prepare(float *H, int64_t d, float damp, float *U, uint8_t *dead_mask,
                           void *ws, cudaStream_t s);
size_t prepare_ws_bytes(int64_t d);

// quantize.cu
// allow_overlap: the blocked sweep may run the far part of each trailing update on a
// second stream (same results bit for bit); false keeps every launch on `s`.
gptq_status launch_quantize(const void *W, int wdtype, int64_t m, int64_t d, int64_t ldw,
                            const float *U, const uint8_t *dead_mask, int bits, int block,
                            uint32_t *qpacked, float *scale, int32_t *zero, float *W_hat,
                            void *ws, cudaStream_t s, bool allow_overlap);
size_t quantize_ws_bytes(int64_t m, int64_t d, int bits, int block);
// api.cu: gptq_quantize_layer's validation + launch; allow_overlap as launch_quantize.
gptq_status quantize_layer_checked(const void *W, int wdtype, int64_t d_out, int64_t d_in,
                                   int64_t ldw, const float *U, const uint8_t *dead_mask,
                                   int bits, int block, uint32_t *qpacked, float *scale,
                                   int32_t *zero, float *W_hat, void *ws, size_t ws_bytes,
                                   gptq_stream_t stream, bool allow_overlap);
// Several layers sharing U, swept as one stack of rows (gptq_quantize_layers_shared).
struct QLayer {
  const void *W; int wdtype; int64_t m; int64_t ldw;
  uint32_t *qpacked; float *scale; int32_t *zero; float *W_hat;
};
gptq_status launch_quantize_layers(const QLayer *L, int n, int64_t d, const float *U,
                                   const uint8_t *dead_mask, int bits, int block, void *ws,
                                   cudaStream_t s, bool allow_overlap);
size_t quantize_layers_ws_bytes(const int64_t *m, int n, int64_t d, int bits, int block);
// OBQ greedy order, d <= 128 (gptq_quantize_obq)
gptq_status launch_quantize_obq(const void *W, int wdtype, int64_t m, int64_t d, int64_t ldw,
                                const float *U, const uint8_t *dead_mask, int bits,
                                uint32_t *qpacked, float *scale, int32_t *zero, float *W_hat,
                                int32_t *order, void *ws, cudaStream_t s);
size_t quantize_obq_ws_bytes(int64_t m, int64_t d);

}  // namespace gptq
