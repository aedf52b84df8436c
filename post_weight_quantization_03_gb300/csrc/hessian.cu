// Step 1 of the path: the layer Hessian H = 2 X^T X over token-major calibration inputs
// ("tm_gptq_math", "Why it is second-order: the Hessian"; "GPTQ Hessian").
//
// Only tiles on or below the diagonal are computed; each such tile writes its lower
// elements and their mirror images, so both triangles of H come out written exactly
// once.
#include "common.cuh"

namespace gptq {

namespace {

constexpr int HT = 64, HK = 16, HNT = 256;

// Maps a linear lower-triangle tile index to (ti, tj) with ti >= tj.
__device__ __forceinline__ void lower_tile(int64_t idx, int &ti, int &tj) {
  // ti = floor((sqrt(8 idx + 1) - 1) / 2), corrected for rounding
  int64_t r = (int64_t)((sqrt(8.0 * (double)idx + 1.0) - 1.0) * 0.5);
  while (r * (r + 1) / 2 > idx) --r;
  while ((r + 1) * (r + 2) / 2 <= idx) ++r;
  ti = (int)r;
  tj = (int)(idx - r * (r + 1) / 2);
}

template <typename T>
__global__ void __launch_bounds__(HNT)
hessian_simt_kernel(const T *__restrict__ X, int64_t n_tok, int64_t d, int64_t ldx,
                    float *__restrict__ H, int accumulate) {
  int ti, tj;
  lower_tile(blockIdx.x, ti, tj);
  const int64_t m0 = (int64_t)ti * HT, n0 = (int64_t)tj * HT;
  __shared__ float As[HK][HT + 4];
  __shared__ float Bs[HK][HT + 4];
  const int tid = threadIdx.x;
  const int tr = tid / 16, tc = tid % 16;
  float acc[4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;
  const int lt = tid / 16, lc = (tid % 16) * 4;  // token row, channel quad
  for (int64_t t0 = 0; t0 < n_tok; t0 += HK) {
    const int64_t t = t0 + lt;
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int64_t ca = m0 + lc + u, cb = n0 + lc + u;
      float a = 0.f, b = 0.f;
      if (t < n_tok) {
        if (ca < d) a = to_f32(X[t * ldx + ca]);
        if (cb < d) b = to_f32(X[t * ldx + cb]);
      }
      As[lt][lc + u] = a;
      Bs[lt][lc + u] = b;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < HK; ++kk) {
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
    if (m >= d) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int64_t n = n0 + tc * 4 + j;
      if (n >= d || n > m) continue;
      float v = 2.0f * acc[i][j];
      if (accumulate) v += H[m * d + n];
      H[m * d + n] = v;
      if (n != m) H[n * d + m] = v;
    }
  }
}

__global__ void zero_kernel(float *p, int64_t n) {
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x)
    p[i] = 0.f;
}

}  // namespace

gptq_status launch_hessian(const void *X, int xdtype, int64_t n_tok, int64_t d, int64_t ldx,
                           float *H, int accumulate, cudaStream_t s) {
  if (n_tok == 0) {
    if (!accumulate) {
      zero_kernel<<<1024, 256, 0, s>>>(H, d * d);
      GPTQ_LAUNCH_CHECK();
    }
    return GPTQ_OK;
  }
  const int64_t nt = ceil_div(d, HT);
  const int64_t tiles = nt * (nt + 1) / 2;
  switch (xdtype) {
    case GPTQ_F32:
      hessian_simt_kernel<float><<<(unsigned)tiles, HNT, 0, s>>>(
          (const float *)X, n_tok, d, ldx, H, accumulate);
      break;
    case GPTQ_F16:
      hessian_simt_kernel<__half><<<(unsigned)tiles, HNT, 0, s>>>(
          (const __half *)X, n_tok, d, ldx, H, accumulate);
      break;
    case GPTQ_BF16:
      hessian_simt_kernel<__nv_bfloat16><<<(unsigned)tiles, HNT, 0, s>>>(
          (const __nv_bfloat16 *)X, n_tok, d, ldx, H, accumulate);
      break;
    default:
      return GPTQ_ERR_INVALID_ARG;
  }
  GPTQ_LAUNCH_CHECK();
  return GPTQ_OK;
}

}  // namespace gptq
