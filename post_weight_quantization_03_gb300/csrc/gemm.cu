// Rank-K updates C (+)= alpha * A * B^T with K-contiguous fp32 operands given as a
// TF32 head/tail pair.  Used by the lazy-batch trailing update of the column sweep and by
// the trailing updates of the blocked Cholesky factorization and inversion.
//
// launch_gemm_nt takes the tcgen05 kernel (tc_gemm.cu) whenever the operands meet its
// TMA alignment rules; this file's CUDA-core kernel (exact fp32 products of head + tail,
// fp32 accumulation) serves the remaining shapes (e.g. lazy-batch widths that are not a
// multiple of 4 columns).
#include "common.cuh"

namespace gptq {

namespace {

constexpr int TM = 64, TN = 64, TK = 16, NT = 256;

__global__ void __launch_bounds__(NT)
gemm_nt_simt_kernel(GemmArgs g, const DevStatus *st) {
  if (st && st->status != 0) return;
  const int tile_m = blockIdx.y, tile_n = blockIdx.x;
  if (g.lower_only && tile_m < tile_n) return;
  const int64_t m0 = (int64_t)tile_m * TM, n0 = (int64_t)tile_n * TN;

  __shared__ float As[TK][TM + 4];
  __shared__ float Bs[TK][TN + 4];

  const int tid = threadIdx.x;
  const int tr = tid / 16, tc = tid % 16;  // 16 x 16 threads, 4 x 4 outputs each
  float acc[4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;

  // loader mapping: 64 rows x 16 k = 1024 elements, 4 per thread along k
  const int lr = tid / 4, lk = (tid % 4) * 4;
  for (int64_t k0 = 0; k0 < g.K; k0 += TK) {
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int64_t k = k0 + lk + u;
      const int64_t am = m0 + lr, bn = n0 + lr;
      float a = 0.f, b = 0.f;
      if (k < g.K) {
        if (am < g.M) {
          a = g.a_hi[am * g.lda + k];
          if (g.a_lo) a += g.a_lo[am * g.lda + k];
        }
        if (bn < g.N) {
          b = g.b_hi[bn * g.ldb + k];
          if (g.b_lo) b += g.b_lo[bn * g.ldb + k];
        }
      }
      As[lk + u][lr] = a;
      Bs[lk + u][lr] = b;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < TK; ++kk) {
      float av[4], bv[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) av[i] = As[kk][tr * 4 + i];
#pragma unroll
      for (int j = 0; j < 4; ++j) bv[j] = Bs[kk][tc * 4 + j];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int64_t m = m0 + tr * 4 + i;
    if (m >= g.M) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int64_t n = n0 + tc * 4 + j;
      if (n >= g.N) continue;
      float *p = g.trans_c ? &g.c[n * g.ldc + m] : &g.c[m * g.ldc + n];
      *p = fmaf(g.alpha, acc[i][j], *p);
    }
  }
}

}  // namespace

gptq_status launch_gemm_nt(const GemmArgs &g, DevStatus *st, cudaStream_t s) {
  if (g.M <= 0 || g.N <= 0 || g.K <= 0) return GPTQ_OK;
  const gptq_status t = launch_gemm_nt_tc(g, st, s);
  if (t != GPTQ_ERR_UNSUPPORTED) return t;
  dim3 grid((unsigned)ceil_div(g.N, TN), (unsigned)ceil_div(g.M, TM));
  gemm_nt_simt_kernel<<<grid, NT, 0, s>>>(g, st);
  GPTQ_LAUNCH_CHECK();
  return GPTQ_OK;
}

}  // namespace gptq
