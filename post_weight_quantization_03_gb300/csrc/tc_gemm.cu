// Tensor-core rank-K update C (+)= alpha * A B^T in 3xTF32 on tcgen05.
//
// A [M, K] and B [N, K] are K-contiguous fp32 operands, each stored as a TF32 head and
// tail (x = head + tail exactly, head with its low 13 mantissa bits clear).  Per K step the
// tensor core accumulates head_A head_B^T + head_A tail_B^T + tail_A head_B^T into an fp32
// TMEM accumulator, which reproduces fp32 products to about 2^-21 relative.
//
// One CTA per 128 x 128 output tile; warp roles:
//   warp 0      : TMA producer (one lane): 4 operand tiles per 32-wide K stage
//   warp 1      : TMEM allocator + MMA issuer (one lane)
//   warps 2..5  : epilogue: TMEM -> registers -> alpha * acc staged in shared memory in
//                 the 128-byte-swizzled box layout -> TMA reduce-add into C (the add
//                 happens in L2); plain read-modify-write when C is not 16-byte aligned
// Stages live in a ring of kStages shared-memory buffers guarded by full/empty
// mbarriers; every wait is bounded (tc.cuh).
#include <cudaTypedefs.h>
#include <string.h>

#include "tc.cuh"

namespace gptq {

namespace {

constexpr int BM = 128, BN = 128, BK = 32;  // BK fp32 = 128 bytes = one swizzle row
constexpr int kStages = 3;
constexpr int kThreads = 192;
constexpr uint32_t kTileA = BM * BK * 4;  // 16 KB
constexpr uint32_t kTileB = BN * BK * 4;  // 16 KB
constexpr uint32_t kStageBytes = 2 * kTileA + 2 * kTileB;
constexpr uint32_t kTmemCols = BN;  // fp32 accumulator: one column per output column
constexpr size_t kSmemBytes = 1024 + kStages * kStageBytes + 256;

struct TcGemmParams {
  int32_t a_k0, a_m0;   // coordinates of A(0, 0) in its tensor map (x = k, y = row)
  int32_t b_k0, b_n0;   // coordinates of B(0, 0)
  int64_t M, N, K;
  float *c; int64_t ldc;
  float alpha;
  int lower_only, trans_c;
  int tma_c;            // 1: epilogue through the C tensor map (reduce-add)
};

__global__ void __launch_bounds__(kThreads, 1)
tc_gemm_3xtf32_kernel(const __grid_constant__ CUtensorMap ma_hi,
                      const __grid_constant__ CUtensorMap ma_lo,
                      const __grid_constant__ CUtensorMap mb_hi,
                      const __grid_constant__ CUtensorMap mb_lo,
                      const __grid_constant__ CUtensorMap mc, TcGemmParams p,
                      DevStatus *st) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint64_t *full = (uint64_t *)(smem + kStages * kStageBytes);
  uint64_t *empty = full + kStages;
  uint64_t *done = empty + kStages;
  uint32_t *tmem_slot = (uint32_t *)(done + 1);

  __shared__ int s_skip;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int tile_m = blockIdx.y, tile_n = blockIdx.x;
  if (threadIdx.x == 0)
    s_skip = (st && st->status != 0) || (p.lower_only && tile_m < tile_n);
  __syncthreads();
  if (s_skip) return;  // uniform for the whole CTA, before any barrier or TMEM use
  const int64_t m0 = (int64_t)tile_m * BM, n0 = (int64_t)tile_n * BN;
  const int ktiles = (int)((p.K + BK - 1) / BK);

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      tc::mbar_init(&full[s], 1);
      tc::mbar_init(&empty[s], 1);
    }
    tc::mbar_init(done, 1);
    tc::mbar_fence_init();
  }
  if (warp == 1) tc::tmem_alloc(tmem_slot, kTmemCols);
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0 && lane == 0) {
    // ---------------- producer ----------------
    tc::tma_prefetch_desc(&ma_hi);
    tc::tma_prefetch_desc(&ma_lo);
    tc::tma_prefetch_desc(&mb_hi);
    tc::tma_prefetch_desc(&mb_lo);
    for (int kt = 0; kt < ktiles; ++kt) {
      const int s = kt % kStages;
      if (kt >= kStages && !tc::mbar_wait(&empty[s], ((kt / kStages) - 1) & 1, st)) break;
      uint8_t *base = smem + s * kStageBytes;
      tc::mbar_arrive_expect_tx(&full[s], kStageBytes);
      const int32_t ka = p.a_k0 + kt * BK, kb = p.b_k0 + kt * BK;
      tc::tma_load_2d(base, &ma_hi, ka, p.a_m0 + (int32_t)m0, &full[s]);
      tc::tma_load_2d(base + kTileA, &ma_lo, ka, p.a_m0 + (int32_t)m0, &full[s]);
      tc::tma_load_2d(base + 2 * kTileA, &mb_hi, kb, p.b_n0 + (int32_t)n0, &full[s]);
      tc::tma_load_2d(base + 2 * kTileA + kTileB, &mb_lo, kb, p.b_n0 + (int32_t)n0, &full[s]);
    }
  } else if (warp == 1 && lane == 0) {
    // ---------------- MMA issuer ----------------
    constexpr uint32_t idesc = tc::instr_desc(2, 2, BM, BN, 0, 0);
    bool ok = true;
    for (int kt = 0; kt < ktiles && ok; ++kt) {
      const int s = kt % kStages;
      ok = tc::mbar_wait(&full[s], (kt / kStages) & 1, st);
      if (!ok) break;
      tc::tc_fence_after();
      const uint32_t a_hi = tc::smem_u32(smem + s * kStageBytes);
      const uint32_t a_lo = a_hi + kTileA;
      const uint32_t b_hi = a_hi + 2 * kTileA;
      const uint32_t b_lo = b_hi + kTileB;
#pragma unroll
      for (int kk = 0; kk < BK / 8; ++kk) {  // 8 tf32 = 32 bytes per MMA
        const uint32_t off = kk * 32;
        const uint64_t dah = tc::smem_desc_sw128(a_hi + off, 16, 1024);
        const uint64_t dal = tc::smem_desc_sw128(a_lo + off, 16, 1024);
        const uint64_t dbh = tc::smem_desc_sw128(b_hi + off, 16, 1024);
        const uint64_t dbl = tc::smem_desc_sw128(b_lo + off, 16, 1024);
        const uint32_t acc0 = (kt > 0 || kk > 0) ? 1u : 0u;
        tc::mma_tf32(tmem, dah, dbh, idesc, acc0);
        tc::mma_tf32(tmem, dah, dbl, idesc, 1u);
        tc::mma_tf32(tmem, dal, dbh, idesc, 1u);
      }
      tc::mma_commit(&empty[s]);  // frees the stage once these MMAs have read it
    }
    tc::mma_commit(done);  // accumulator complete (or abandoned after a timeout)
  } else if (warp >= 2) {
    // ---------------- epilogue ----------------
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    int okl = 0;
    if (lane == 0) okl = tc::mbar_wait(done, 0, st) ? 1 : 0;
    const bool ok = __shfl_sync(0xffffffffu, okl, 0) != 0;  // warp-uniform
    __syncwarp();
    tc::tc_fence_after();
    const int64_t row = m0 + q * 32 + lane;
    if (ok && ktiles > 0 && p.tma_c) {
      // every stage buffer is free once `done` fired: reuse stage 0 (4 boxes of 32 cols)
      const int rl = q * 32 + lane;
#pragma unroll 1
      for (int c0 = 0; c0 < BN; c0 += 32) {
        uint32_t r[32];
        tc::tmem_ld32(tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)c0, r);
        tc::tmem_ld_wait();
        uint8_t *rowp = smem + (c0 / 32) * (BM * 128) + rl * 128;
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const float4 v = make_float4(p.alpha * __uint_as_float(r[4 * u]),
                                       p.alpha * __uint_as_float(r[4 * u + 1]),
                                       p.alpha * __uint_as_float(r[4 * u + 2]),
                                       p.alpha * __uint_as_float(r[4 * u + 3]));
          *reinterpret_cast<float4 *>(rowp + ((u ^ (rl & 7)) * 16)) = v;
        }
      }
      tc::fence_proxy_async_smem();
      tc::named_barrier(1, 128);  // the four epilogue warps
      if (warp == 2 && lane == 0) {
#pragma unroll
        for (int c = 0; c < BN / 32; ++c)
          tc::tma_reduce_add_2d(&mc, (int32_t)(n0 + 32 * c), (int32_t)m0, smem + c * (BM * 128));
        tc::bulk_commit();
        tc::bulk_wait_read_all();
      }
    } else if (ok && ktiles > 0) {
#pragma unroll 1
      for (int c0 = 0; c0 < BN; c0 += 32) {
        uint32_t r[32];
        tc::tmem_ld32(tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)c0, r);
        tc::tmem_ld_wait();
        if (row < p.M) {
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const int64_t col = n0 + c0 + i;
            if (col < p.N) {
              float *ptr = p.trans_c ? &p.c[col * p.ldc + row] : &p.c[row * p.ldc + col];
              *ptr = fmaf(p.alpha, __uint_as_float(r[i]), *ptr);
            }
          }
        }
      }
    }
  }
  tc::tc_fence_before();
  __syncthreads();
  if (warp == 1) tc::tmem_dealloc(tmem, kTmemCols);
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = (PFN_cuTensorMapEncodeTiled_v12000)p;
  }
  return fn;
}

bool make_tmap_f32(CUtensorMap *m, const float *base, int64_t rows, int64_t cols, int64_t ld,
                   int box_rows) {
  return tc::make_tmap_2d(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, base, rows, cols, ld * 4, BK,
                          box_rows);
}

}  // namespace

bool tc::make_tmap_2d(CUtensorMap *m, CUtensorMapDataType dt, const void *base, int64_t rows,
                      int64_t cols, int64_t ld_bytes, int box_cols, int box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  if (((uintptr_t)base & 15) || (ld_bytes & 15) || rows < 1 || cols < 1) return false;
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)ld_bytes};
  cuuint32_t box[2] = {(cuuint32_t)box_cols, (cuuint32_t)box_rows};
  cuuint32_t es[2] = {1, 1};
  return fn(m, dt, 2, (void *)base, dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Tensor-core path of launch_gemm_nt.  Requirements (else returns UNSUPPORTED so the
// caller can take the CUDA-core kernel): both operands have head and tail, 16-byte
// aligned bases and row pitches, and K offsets that are multiples of 4 elements.
gptq_status launch_gemm_nt_tc(const GemmArgs &g, DevStatus *st, cudaStream_t s) {
  if (g.M <= 0 || g.N <= 0 || g.K <= 0) return GPTQ_OK;
  if (!g.a_lo || !g.b_lo) return GPTQ_ERR_UNSUPPORTED;
  static bool attr_done = false;
  if (!attr_done) {
    GPTQ_CUDA_CHECK(cudaFuncSetAttribute(tc_gemm_3xtf32_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)kSmemBytes));
    attr_done = true;
  }
  CUtensorMap mah, mal, mbh, mbl;
  // maps cover exactly the [M, K] / [N, K] operand windows: out-of-range reads are zero
  if (!make_tmap_f32(&mah, g.a_hi, g.M, g.K, g.lda, BM) ||
      !make_tmap_f32(&mal, g.a_lo, g.M, g.K, g.lda, BM) ||
      !make_tmap_f32(&mbh, g.b_hi, g.N, g.K, g.ldb, BN) ||
      !make_tmap_f32(&mbl, g.b_lo, g.N, g.K, g.ldb, BN))
    return GPTQ_ERR_UNSUPPORTED;
  CUtensorMap mc;
  memset(&mc, 0, sizeof(mc));
  const bool tma_c = !g.trans_c && make_tmap_f32(&mc, g.c, g.M, g.N, g.ldc, BM);
  TcGemmParams p{};
  p.tma_c = tma_c ? 1 : 0;
  p.a_k0 = 0; p.a_m0 = 0; p.b_k0 = 0; p.b_n0 = 0;
  p.M = g.M; p.N = g.N; p.K = g.K;
  p.c = g.c; p.ldc = g.ldc; p.alpha = g.alpha;
  p.lower_only = g.lower_only; p.trans_c = g.trans_c;
  dim3 grid((unsigned)ceil_div(g.N, BN), (unsigned)ceil_div(g.M, BM));
  tc_gemm_3xtf32_kernel<<<grid, kThreads, kSmemBytes, s>>>(mah, mal, mbh, mbl, mc, p, st);
  GPTQ_LAUNCH_CHECK();
  return GPTQ_OK;
}

}  // namespace gptq
