// Step 1 of the path: the layer Hessian H = 2 X^T X over token-major calibration inputs
// ("tm_gptq_math", "Why it is second-order: the Hessian"; "GPTQ Hessian").
//
// Only tiles on or below the diagonal are computed; each such tile writes its lower
// elements and their mirror images, so both triangles of H come out written exactly
// once.
//
// fp16/bf16 inputs run on the tcgen05 tensor cores (kind::f16, fp32 accumulation in
// TMEM): the products of two 16-bit values are exact in fp32, and the accumulator is
// drained into fp32 registers every kSegTokens tokens so that no truncating tensor-core
// running sum spans more than one segment.  fp32 inputs (and tiny shapes) take a CUDA-core kernel.
#include <algorithm>

#include "tc.cuh"

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


// ---------------------------------------------------------------------------------------
// tcgen05 SYRK: one CTA per 128 x 256 tile of H on or below the diagonal.
//   operand tiles are token-major slices of X (MN-major for the MMA: channels contiguous)
//   warp 0      : TMA producer, 64 tokens per stage (2 + 4 boxes of 64 ch x 64 tok)
//   warp 1      : TMEM allocator (2 x 256 columns) + MMA issuer
//   warps 2..9  : drain TMEM segments into fp32 registers, then write H and its mirror
// ---------------------------------------------------------------------------------------
constexpr int TB_M = 128, TB_N = 256, TB_K = 64;
constexpr int T_STAGES = 4;
constexpr uint32_t T_BOX = 64 * TB_K * 2;                 // 8 KB
constexpr uint32_t T_TILE_A = 2 * T_BOX;                  // 16 KB
constexpr uint32_t T_TILE_B = 4 * T_BOX;                  // 32 KB
constexpr uint32_t T_STAGE = T_TILE_A + T_TILE_B;         // 48 KB
constexpr int T_EPI_WARPS = 8;
constexpr int T_THREADS = 64 + 32 * T_EPI_WARPS;          // 320
constexpr size_t T_SMEM = 1024 + T_STAGES * T_STAGE + 256;

struct HessTcParams {
  int64_t d, n_tok;
  int n_row_blocks;   // ceil(d / 128)
  int seg_stages;     // stages (of 64 tokens) per accumulation segment
  float *H;
  int accumulate;
};

template <int FMT>  // 0 = fp16, 1 = bf16
__global__ void __launch_bounds__(T_THREADS, 1)
hessian_tc_kernel(const __grid_constant__ CUtensorMap mx, HessTcParams p, DevStatus *st) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint64_t *full = (uint64_t *)(smem + T_STAGES * T_STAGE);
  uint64_t *empty = full + T_STAGES;
  uint64_t *tfull = empty + T_STAGES;   // [2]: accumulator buffer ready to drain
  uint64_t *tempty = tfull + 2;         // [2]: accumulator buffer drained
  uint32_t *tmem_slot = (uint32_t *)(tempty + 2);

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  // tile index -> (row block ib, column block jb): column blocks in order, rows 2jb..
  int ib = 0, jb = 0;
  {
    int idx = blockIdx.x;
    for (jb = 0;; ++jb) {
      const int cnt = p.n_row_blocks - 2 * jb;
      if (idx < cnt) { ib = 2 * jb + idx; break; }
      idx -= cnt;
    }
  }
  const int64_t m0 = (int64_t)ib * TB_M, n0 = (int64_t)jb * TB_N;
  const int total = (int)((p.n_tok + TB_K - 1) / TB_K);
  const int nseg = (total + p.seg_stages - 1) / p.seg_stages;

  if (threadIdx.x == 0) {
    for (int s = 0; s < T_STAGES; ++s) {
      tc::mbar_init(&full[s], 1);
      tc::mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      tc::mbar_init(&tfull[b], 1);
      tc::mbar_init(&tempty[b], T_EPI_WARPS);
    }
    tc::mbar_fence_init();
  }
  if (warp == 1) tc::tmem_alloc(tmem_slot, 512);
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0 && lane == 0) {
    tc::tma_prefetch_desc(&mx);
    for (int g = 0; g < total; ++g) {
      const int s = g % T_STAGES;
      if (g >= T_STAGES && !tc::mbar_wait(&empty[s], ((g / T_STAGES) - 1) & 1, st)) break;
      uint8_t *a = smem + s * T_STAGE;
      uint8_t *b = a + T_TILE_A;
      const int32_t t0 = g * TB_K;
      tc::mbar_arrive_expect_tx(&full[s], T_STAGE);
      tc::tma_load_2d(a, &mx, (int32_t)m0, t0, &full[s]);
      tc::tma_load_2d(a + T_BOX, &mx, (int32_t)m0 + 64, t0, &full[s]);
#pragma unroll
      for (int q = 0; q < 4; ++q)
        tc::tma_load_2d(b + q * T_BOX, &mx, (int32_t)n0 + 64 * q, t0, &full[s]);
    }
  } else if (warp == 1 && lane == 0) {
    constexpr uint32_t idesc = tc::instr_desc(FMT, FMT, TB_M, TB_N, 1, 1);
    int g = 0;
    bool ok = true;
    for (int sg = 0; sg < nseg && ok; ++sg) {
      const int buf = sg & 1;
      if (sg >= 2) {
        ok = tc::mbar_wait(&tempty[buf], ((sg / 2) - 1) & 1, st);
        if (!ok) break;
        tc::tc_fence_after();
      }
      const uint32_t dt = tmem + (uint32_t)(buf * TB_N);
      const int gend = min(total, (sg + 1) * p.seg_stages);
      for (int first = 1; g < gend; ++g, first = 0) {
        const int s = g % T_STAGES;
        ok = tc::mbar_wait(&full[s], (g / T_STAGES) & 1, st);
        if (!ok) break;
        tc::tc_fence_after();
        const uint32_t a = tc::smem_u32(smem + s * T_STAGE);
        const uint32_t b = a + T_TILE_A;
#pragma unroll
        for (int kk = 0; kk < TB_K / 16; ++kk) {  // 16 tokens = 2048 bytes per MMA
          const uint64_t da = tc::smem_desc_sw128(a + kk * 2048, T_BOX, 1024);
          const uint64_t db = tc::smem_desc_sw128(b + kk * 2048, T_BOX, 1024);
          tc::mma_f16(dt, da, db, idesc, (first && kk == 0) ? 0u : 1u);
        }
        tc::mma_commit(&empty[s]);
      }
      tc::mma_commit(&tfull[buf]);
    }
  } else if (warp >= 2) {
    const int e = warp - 2, q = warp & 3, h = e / 4;
    float acc[128];
#pragma unroll
    for (int i = 0; i < 128; ++i) acc[i] = 0.f;
    bool ok = true;
    for (int sg = 0; sg < nseg && ok; ++sg) {
      const int buf = sg & 1;
      int okl = 0;
      if (lane == 0) okl = tc::mbar_wait(&tfull[buf], (sg / 2) & 1, st) ? 1 : 0;
      ok = __shfl_sync(0xffffffffu, okl, 0) != 0;
      __syncwarp();
      if (!ok) break;
      tc::tc_fence_after();
      const uint32_t base = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(buf * TB_N + h * 128);
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t r[32];
        tc::tmem_ld32(base + (uint32_t)(c * 32), r);
        tc::tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 32; ++i) acc[c * 32 + i] += __uint_as_float(r[i]);
      }
      tc::tc_fence_before();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&tempty[buf]);
    }
    const int64_t r = m0 + q * 32 + lane;
    const int64_t d = p.d;
    if (ok && r < d) {
#pragma unroll
      for (int i = 0; i < 128; ++i) {
        const int64_t c = n0 + h * 128 + i;
        if (c < d && c <= r) {
          float v = 2.0f * acc[i];
          if (p.accumulate) v += p.H[r * d + c];
          p.H[r * d + c] = v;
          if (c != r) p.H[c * d + r] = v;
        }
      }
    }
  }
  tc::tc_fence_before();
  __syncthreads();
  if (warp == 1) tc::tmem_dealloc(tmem, 512);
}

__global__ void zero_kernel(float *p, int64_t n) {
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x)
    p[i] = 0.f;
}

// Tokens per TMEM accumulation segment (multiple of 64).  The tensor core's fp32
// accumulation rounds toward zero, so its relative bias grows with the number of MMAs
// summed in TMEM (measured: ~2e-5 after 256 MMAs of 16 tokens); 512 tokens (32 MMAs) keep
// it near 2e-6, and the segments are summed in round-to-nearest fp32 registers.
constexpr int kSegTokens = 512;

gptq_status launch_hessian_tc(const void *X, int xdtype, int64_t n_tok, int64_t d, int64_t ldx,
                              float *H, int accumulate, DevStatus *st, cudaStream_t s) {
  GPTQ_TRY(ensure_smem_attr((const void *)hessian_tc_kernel<0>, (int)T_SMEM));
  GPTQ_TRY(ensure_smem_attr((const void *)hessian_tc_kernel<1>, (int)T_SMEM));
  CUtensorMap mx;
  const CUtensorMapDataType dt =
      xdtype == GPTQ_F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  if (!tc::make_tmap_2d(&mx, dt, X, n_tok, d, ldx * 2, 64, TB_K)) return GPTQ_ERR_UNSUPPORTED;
  HessTcParams p{};
  p.d = d;
  p.n_tok = n_tok;
  p.n_row_blocks = (int)ceil_div(d, TB_M);
  p.seg_stages = kSegTokens / TB_K;
  p.H = H;
  p.accumulate = accumulate;
  const int ncb = (int)ceil_div(d, TB_N);
  int64_t tiles = 0;
  for (int j = 0; j < ncb; ++j) tiles += std::max(0, p.n_row_blocks - 2 * j);
  if (xdtype == GPTQ_F16)
    hessian_tc_kernel<0><<<(unsigned)tiles, T_THREADS, T_SMEM, s>>>(mx, p, st);
  else
    hessian_tc_kernel<1><<<(unsigned)tiles, T_THREADS, T_SMEM, s>>>(mx, p, st);
  GPTQ_LAUNCH_CHECK();
  return GPTQ_OK;
}

}  // namespace

gptq_status launch_hessian(const void *X, int xdtype, int64_t n_tok, int64_t d, int64_t ldx,
                           float *H, int accumulate, DevStatus *st, cudaStream_t s) {
  if (n_tok == 0) {
    if (!accumulate) {
      zero_kernel<<<1024, 256, 0, s>>>(H, d * d);
      GPTQ_LAUNCH_CHECK();
    }
    return GPTQ_OK;
  }
  if ((xdtype == GPTQ_F16 || xdtype == GPTQ_BF16) && d >= 64 && n_tok >= 64) {
    const gptq_status t = launch_hessian_tc(X, xdtype, n_tok, d, ldx, H, accumulate, st, s);
    if (t != GPTQ_ERR_UNSUPPORTED) return t;
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
