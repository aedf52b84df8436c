// The consumer of the quantized layer: its output error on the calibration inputs,
// ||W X^T - W_hat X^T||_F^2 per output row, evaluated on X itself ("tm_gptq_math", "The
// reconstruction objective, written out": the quantity GPTQ minimizes row by row).
//
//   1. diff_kernel  : Delta = W - W_hat, W_hat = scale * (code - zero) decoded from the
//                     packed codes, in fp32, stored in the activations' type
//   2. product      : E = Delta X^T with the row sums of E^2 taken in the epilogue, one
//                     partial per (row, token tile):
//                       fp16 / bf16 X : tcgen05 kind::f16, persistent, K-major operands
//                                       through 128-byte-swizzled TMA boxes, 4-stage ring,
//                                       M128 N256 K16, two TMEM accumulators
//                       fp32 X        : CUDA cores (64 x 64 tiles)
//   3. reduce_kernel: err[i] = sum over token tiles, in a fixed order (deterministic)
#include <cudaTypedefs.h>
#include <string.h>

#include <type_traits>

#include "tc.cuh"

namespace gptq {

namespace {

// ---------------------------------------------------------------------------------------
// Delta = W - scale * (code - zero), code c of a row at bits [c*bits, (c+1)*bits) of its
// little-endian packed bitstream.
// ---------------------------------------------------------------------------------------
template <typename TW, typename TD>
__global__ void diff_kernel(const TW *__restrict__ W, int64_t ldw, int64_t m, int64_t d,
                            const uint32_t *__restrict__ qp, int64_t words, int bits,
                            const float *__restrict__ scale, const int32_t *__restrict__ zero,
                            TD *__restrict__ D, int64_t ldd) {
  const int64_t total = m * ldd;
  for (int64_t idx = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; idx < total;
       idx += (int64_t)gridDim.x * blockDim.x) {
    const int64_t i = idx / ldd, k = idx % ldd;
    float v = 0.0f;
    if (k < d) {
      const int64_t bit = k * bits;
      const uint32_t *row = qp + i * words;
      uint64_t two = row[bit >> 5];
      if (((bit & 31) + bits) > 32) two |= (uint64_t)row[(bit >> 5) + 1] << 32;
      const uint32_t code = (uint32_t)(two >> (bit & 31)) & ((1u << bits) - 1u);
      const float what = scale[i] * ((float)code - (float)zero[i]);
      v = to_f32(W[i * ldw + k]) - what;
    }
    if constexpr (sizeof(TD) == 4) D[idx] = v;
    else if constexpr (std::is_same<TD, __half>::value) D[idx] = __float2half_rn(v);
    else D[idx] = __float2bfloat16_rn(v);
  }
}

// err[i] = sum_t partial[t][i] over the token tiles, accumulated in fp64.
__global__ void reduce_kernel(const float *__restrict__ part, int64_t ntiles, int64_t m,
                              float *__restrict__ err) {
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < m;
       i += (int64_t)gridDim.x * blockDim.x) {
    double s = 0.0;
    for (int64_t t = 0; t < ntiles; ++t) s += (double)part[t * m + i];
    err[i] = (float)s;
  }
}

// ---------------------------------------------------------------------------------------
// tcgen05 product: tiles of 128 rows of Delta x 256 tokens, persistent over tiles.
//   warp 0     : TMA producer (one lane), 4-stage ring of (Delta box, X box) per 64 k
//   warp 1     : TMEM allocator + MMA issuer (one lane), two 256-column accumulators
//   warps 2..5 : epilogue: each thread owns one row, sums the squares of its 256 outputs
//                and writes the partial; releases the accumulator after the reads
// ---------------------------------------------------------------------------------------
constexpr int RM = 128, RN = 256, RK = 64;   // RK 16-bit elements = 128 bytes
constexpr int kRStages = 4;
constexpr int kRThreads = 192;
constexpr uint32_t kRTileA = RM * RK * 2;    // 16 KB
constexpr uint32_t kRTileB = RN * RK * 2;    // 32 KB
constexpr uint32_t kRStage = kRTileA + kRTileB;
constexpr uint32_t kRTmemCols = 2 * RN;
constexpr size_t kRSmem = 1024 + kRStages * kRStage + 256;

struct ReconParams {
  int64_t m, n, k;
  int n_m, n_n, n_tiles;
  float *part;   // [n_n][m]
};

template <int FMT>
__global__ void __launch_bounds__(kRThreads, 1)
recon_tc_kernel(const __grid_constant__ CUtensorMap md, const __grid_constant__ CUtensorMap mx,
                ReconParams p, DevStatus *st) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint64_t *full = (uint64_t *)(smem + kRStages * kRStage);
  uint64_t *empty = full + kRStages;
  uint64_t *tfull = empty + kRStages;
  uint64_t *tempty = tfull + 2;
  uint32_t *tmem_slot = (uint32_t *)(tempty + 2);
  int *epi_ok = (int *)(tmem_slot + 1);

  __shared__ int s_skip;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  if (threadIdx.x == 0) s_skip = (st->status != 0);
  __syncthreads();
  if (s_skip) return;
  const int ktiles = (int)((p.k + RK - 1) / RK);

  if (threadIdx.x == 0) {
    for (int s = 0; s < kRStages; ++s) {
      tc::mbar_init(&full[s], 1);
      tc::mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      tc::mbar_init(&tfull[b], 1);
      tc::mbar_init(&tempty[b], 4);
    }
    tc::mbar_fence_init();
  }
  if (warp == 1) tc::tmem_alloc(tmem_slot, kRTmemCols);
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0 && lane == 0) {
    // ---------------- producer ----------------
    tc::tma_prefetch_desc(&md);
    tc::tma_prefetch_desc(&mx);
    int g = 0;
    bool ok = true;
    for (int t = blockIdx.x; t < p.n_tiles && ok; t += gridDim.x) {
      const int32_t m0 = (t % p.n_m) * RM, n0 = (t / p.n_m) * RN;
      for (int kt = 0; kt < ktiles; ++kt, ++g) {
        const int s = g % kRStages;
        if (g >= kRStages && !tc::mbar_wait(&empty[s], ((g / kRStages) - 1) & 1, st)) {
          ok = false;
          break;
        }
        uint8_t *base = smem + s * kRStage;
        tc::mbar_arrive_expect_tx(&full[s], kRStage);
        tc::tma_load_2d(base, &md, kt * RK, m0, &full[s]);
        tc::tma_load_2d(base + kRTileA, &mx, kt * RK, n0, &full[s]);
      }
    }
  } else if (warp == 1 && lane == 0) {
    // ---------------- MMA issuer ----------------
    constexpr uint32_t idesc = tc::instr_desc(FMT, FMT, RM, RN, 0, 0);
    int g = 0, it = 0;
    bool ok = true;
    for (int t = blockIdx.x; t < p.n_tiles && ok; t += gridDim.x, ++it) {
      const int b = it & 1;
      if (it >= 2) {
        ok = tc::mbar_wait(&tempty[b], ((it / 2) - 1) & 1, st);
        if (!ok) break;
        tc::tc_fence_after();
      }
      const uint32_t dt = tmem + (uint32_t)(b * RN);
      for (int kt = 0; kt < ktiles; ++kt, ++g) {
        const int s = g % kRStages;
        ok = tc::mbar_wait(&full[s], (g / kRStages) & 1, st);
        if (!ok) break;
        tc::tc_fence_after();
        const uint32_t a = tc::smem_u32(smem + s * kRStage);
        const uint32_t bb = a + kRTileA;
#pragma unroll
        for (int kk = 0; kk < RK / 16; ++kk) {  // 16 elements = 32 bytes per MMA
          const uint64_t da = tc::smem_desc_sw128(a + kk * 32, 16, 1024);
          const uint64_t db = tc::smem_desc_sw128(bb + kk * 32, 16, 1024);
          tc::mma_f16(dt, da, db, idesc, (kt > 0 || kk > 0) ? 1u : 0u);
        }
        tc::mma_commit(&empty[s]);
      }
      tc::mma_commit(&tfull[b]);
    }
  } else if (warp >= 2) {
    // ---------------- epilogue ----------------
    const int q = warp & 3;
    const int rl = q * 32 + lane;
    const bool leader = (warp == 2 && lane == 0);
    int it = 0;
    for (int t = blockIdx.x; t < p.n_tiles; t += gridDim.x, ++it) {
      const int b = it & 1;
      if (leader) *epi_ok = tc::mbar_wait(&tfull[b], (it / 2) & 1, st) ? 1 : 0;
      tc::named_barrier(1, 128);
      if (!*epi_ok) break;
      tc::tc_fence_after();
      const int tm = t % p.n_m, tn = t / p.n_m;
      float s0 = 0.f, s1 = 0.f;
#pragma unroll 1
      for (int c = 0; c < RN; c += 64) {
        uint32_t r0[32], r1[32];
        const uint32_t ta = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(b * RN + c);
        tc::tmem_ld32(ta, r0);
        tc::tmem_ld32(ta + 32, r1);
        tc::tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const float v0 = __uint_as_float(r0[i]), v1 = __uint_as_float(r1[i]);
          s0 = fmaf(v0, v0, s0);
          s1 = fmaf(v1, v1, s1);
        }
      }
      tc::tc_fence_before();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&tempty[b]);
      const int64_t row = (int64_t)tm * RM + rl;
      if (row < p.m) p.part[(int64_t)tn * p.m + row] = s0 + s1;
    }
  }
  tc::tc_fence_before();
  __syncthreads();
  if (warp == 1) tc::tmem_dealloc(tmem, kRTmemCols);
}

// ---------------------------------------------------------------------------------------
// CUDA-core product (fp32 X): 64 rows x 64 tokens per CTA, 4 x 4 outputs per thread; the
// 16 threads sharing a row group sit in one half-warp and reduce by shuffles.
// ---------------------------------------------------------------------------------------
__global__ void __launch_bounds__(256)
recon_simt_kernel(const float *__restrict__ D, int64_t ldd, const float *__restrict__ X,
                  int64_t ldx, int64_t m, int64_t n, int64_t k, float *__restrict__ part) {
  __shared__ float As[16][64 + 4], Bs[16][64 + 4];
  const int tx = threadIdx.x % 16, ty = threadIdx.x / 16;
  const int64_t r0 = (int64_t)blockIdx.y * 64, t0 = (int64_t)blockIdx.x * 64;
  float acc[4][4] = {};
  for (int64_t k0 = 0; k0 < k; k0 += 16) {
    for (int e = threadIdx.x; e < 16 * 64; e += 256) {
      const int kk = e % 16, rr = e / 16;
      As[kk][rr] = (r0 + rr < m && k0 + kk < k) ? D[(r0 + rr) * ldd + k0 + kk] : 0.f;
      Bs[kk][rr] = (t0 + rr < n && k0 + kk < k) ? X[(t0 + rr) * ldx + k0 + kk] : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < 16; ++kk) {
      float a[4], b[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] = As[kk][4 * ty + i];
#pragma unroll
      for (int j = 0; j < 4; ++j) b[j] = Bs[kk][4 * tx + j];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float s = 0.f;
#pragma unroll
    for (int j = 0; j < 4; ++j) s = fmaf(acc[i][j], acc[i][j], s);
#pragma unroll
    for (int o = 8; o; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    const int64_t row = r0 + 4 * ty + i;
    if (tx == 0 && row < m) part[(int64_t)blockIdx.x * m + row] = s;
  }
}

struct ReconWs {
  DevStatus *st;
  void *D; int64_t ldd;
  float *part;
};

ReconWs carve_recon(void *ws, int64_t m, int64_t d, size_t es) {
  ReconWs w;
  char *p = (char *)ws;
  w.st = (DevStatus *)p; p += 256;
  w.ldd = (int64_t)round_up((size_t)d, 8);
  w.D = p; p += round_up((size_t)m * w.ldd * es, 256);
  w.part = (float *)p;
  return w;
}

template <typename TW, typename TD>
void launch_diff(const void *W, int64_t ldw, int64_t m, int64_t d, const uint32_t *qp,
                 int bits, const float *scale, const int32_t *zero, const ReconWs &w,
                 cudaStream_t s) {
  const int64_t words = ceil_div(d, 32) * bits;
  diff_kernel<TW, TD><<<2048, 256, 0, s>>>((const TW *)W, ldw, m, d, qp, words, bits, scale,
                                           zero, (TD *)w.D, w.ldd);
}

template <typename TD>
gptq_status launch_diff_any(const void *W, int wdtype, int64_t ldw, int64_t m, int64_t d,
                            const uint32_t *qp, int bits, const float *scale,
                            const int32_t *zero, const ReconWs &w, cudaStream_t s) {
  switch (wdtype) {
    case GPTQ_F32: launch_diff<float, TD>(W, ldw, m, d, qp, bits, scale, zero, w, s); break;
    case GPTQ_F16: launch_diff<__half, TD>(W, ldw, m, d, qp, bits, scale, zero, w, s); break;
    case GPTQ_BF16:
      launch_diff<__nv_bfloat16, TD>(W, ldw, m, d, qp, bits, scale, zero, w, s);
      break;
    default: return GPTQ_ERR_INVALID_ARG;
  }
  GPTQ_LAUNCH_CHECK();
  return GPTQ_OK;
}

}  // namespace

size_t recon_ws_bytes(int xdtype, int64_t m, int64_t d, int64_t n) {
  const size_t es = xdtype == GPTQ_F32 ? 4 : 2;
  const int64_t tiles = xdtype == GPTQ_F32 ? ceil_div(n, 64) : ceil_div(n, RN);
  return 256 + round_up((size_t)m * round_up((size_t)d, 8) * es, 256) +
         round_up((size_t)(tiles > 0 ? tiles : 1) * m * 4, 256);
}

gptq_status launch_recon(const void *X, int xdtype, int64_t n, int64_t d, int64_t ldx,
                         const void *W, int wdtype, int64_t m, int64_t ldw, const uint32_t *qp,
                         int bits, const float *scale, const int32_t *zero, float *err,
                         void *ws, cudaStream_t s) {
  const size_t es = xdtype == GPTQ_F32 ? 4 : 2;
  ReconWs w = carve_recon(ws, m, d, es);
  GPTQ_CUDA_CHECK(cudaMemsetAsync(w.st, 0, sizeof(DevStatus), s));
  if (n == 0) {
    GPTQ_CUDA_CHECK(cudaMemsetAsync(err, 0, (size_t)m * 4, s));
    return GPTQ_OK;
  }
  int64_t ntiles = 0;
  if (xdtype == GPTQ_F32) {
    GPTQ_TRY(launch_diff_any<float>(W, wdtype, ldw, m, d, qp, bits, scale, zero, w, s));
    ntiles = ceil_div(n, 64);
    dim3 g((unsigned)ntiles, (unsigned)ceil_div(m, 64));
    recon_simt_kernel<<<g, 256, 0, s>>>((const float *)w.D, w.ldd, (const float *)X, ldx, m, n,
                                        d, w.part);
    GPTQ_LAUNCH_CHECK();
  } else {
    GPTQ_TRY(ensure_smem_attr((const void *)recon_tc_kernel<0>, (int)kRSmem));
    GPTQ_TRY(ensure_smem_attr((const void *)recon_tc_kernel<1>, (int)kRSmem));
    const CUtensorMapDataType dt =
        xdtype == GPTQ_F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    if (xdtype == GPTQ_F16)
      GPTQ_TRY(launch_diff_any<__half>(W, wdtype, ldw, m, d, qp, bits, scale, zero, w, s));
    else
      GPTQ_TRY(launch_diff_any<__nv_bfloat16>(W, wdtype, ldw, m, d, qp, bits, scale, zero, w,
                                              s));
    CUtensorMap md, mx;
    if (!tc::make_tmap_2d(&md, dt, w.D, m, d, w.ldd * 2, RK, RM) ||
        !tc::make_tmap_2d(&mx, dt, X, n, d, ldx * 2, RK, RN))
      return GPTQ_ERR_UNSUPPORTED;
    int num_sms = 0;
    GPTQ_TRY(device_sm_count(&num_sms));
    ReconParams p{};
    p.m = m; p.n = n; p.k = d;
    p.n_m = (int)ceil_div(m, RM);
    p.n_n = (int)ceil_div(n, RN);
    p.n_tiles = p.n_m * p.n_n;
    p.part = w.part;
    ntiles = p.n_n;
    const int grid = p.n_tiles < num_sms ? p.n_tiles : num_sms;
    if (xdtype == GPTQ_F16)
      recon_tc_kernel<0><<<grid, kRThreads, kRSmem, s>>>(md, mx, p, w.st);
    else
      recon_tc_kernel<1><<<grid, kRThreads, kRSmem, s>>>(md, mx, p, w.st);
    GPTQ_LAUNCH_CHECK();
  }
  reduce_kernel<<<(unsigned)ceil_div(m, 256), 256, 0, s>>>(w.part, ntiles, m, err);
  GPTQ_LAUNCH_CHECK();
  return GPTQ_OK;
}

}  // namespace gptq
