// Tensor-core rank-K update C (+)= alpha * A B^T in 3xTF32 on tcgen05.
//
// A [M, K] and B [N, K] are K-contiguous fp32 operands, each stored as a TF32 head and
// tail (x = head + tail exactly, head with its low 13 mantissa bits clear).  Per K step the
// tensor core accumulates head_A head_B^T + head_A tail_B^T + tail_A head_B^T, which
// reproduces fp32 products to about 2^-21 relative.
//
// The tensor core's fp32 accumulation truncates (rounds toward zero), so a long running
// sum in TMEM drifts.  Two kernels:
//   tc_gemm_short_sums_kernel (the factorization's updates, whose accuracy needs it): the
//     head products go to an accumulator of their own that the epilogue drains into
//     round-to-nearest fp32 registers every kHeadGroup K stages, and the two cross products
//     (about 2^-11 of the head product) to a second accumulator drained once per tile;
//   tc_gemm_one_sum_kernel (the sweep's updates, whose codes need no more): all three
//     products of a tile in one TMEM sum, drained once.  (One accumulator per 128-deep tile left the factor U of a 28672-wide layer
// with row errors up to 2e-4 against the fp64 oracle; short head sums bring it to the
// fp32 storage floor, about 7e-5.)
//
// Both are persistent: each CTA walks a static list of 128 x 128 output tiles; warp roles
// (short sums; the one-sum kernel alternates two 128-column tile accumulators instead):
//   warp 0      : TMA producer (one lane): 4 operand tiles per 32-wide K stage, running
//                 ahead across tile boundaries through a 3-stage ring
//   warp 1      : TMEM allocator + MMA issuer (one lane): head products into two alternating
//                 128-column accumulators (kHeadGroup stages each, or the whole tile), cross
//                 products into two more, alternating by tile (or with the head products)
//   warps 2..5  : epilogue: TMEM -> registers (the tile's running sum, one row per thread);
//                 per tile alpha * sum staged in shared memory in the 128-byte-swizzled box
//                 layout (two 64-column halves) -> TMA reduce-add into C (the add happens in
//                 L2, so concurrent updates of the same C are safe); plain
//                 read-modify-write when C is not 16-byte aligned
// Every mbarrier wait is bounded (tc.cuh); the epilogue warps agree on the outcome of their
// waits once per tile (a barrier with an AND vote), so all four leave their loops together.
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
constexpr uint32_t kStagingBytes = 2 * BM * 128;  // two 32-column boxes (one 64-col half)
constexpr uint32_t kTmemCols = 4 * BN;            // 3 head + 1 cross accumulators: 512
constexpr int kHeadGroup = 2;                     // K stages per head-product TMEM sum
constexpr int kHeadBufs = 3;                      // head-product accumulators used in turn
constexpr size_t kSmemBytes = 1024 + kStages * kStageBytes + kStagingBytes + 256;

struct TcGemmParams {
  int64_t M, N, K;
  float *c; int64_t ldc;
  float alpha;
  int lower_only;
  int tma_c;            // 1: epilogue through the C tensor map (reduce-add)
  int n_m, n_n;         // tile grid
  int n_tiles;          // tiles to process (lower ones only when lower_only)
};

// Linear tile index -> (tm, tn): row-major over the tile grid, or, when lower_only, over
// its lower trapezoid (tm >= tn): the triangle of the first n_n tile rows, then the whole
// tile rows below it.
__device__ __forceinline__ void tile_coords(const TcGemmParams &p, int t, int &tm, int &tn) {
  if (p.lower_only) {
    const int tri = p.n_n * (p.n_n + 1) / 2;
    if (t >= tri) {
      t -= tri;
      tm = p.n_n + t / p.n_n;
      tn = t % p.n_n;
      return;
    }
    int r = (int)((sqrtf(8.0f * (float)t + 1.0f) - 1.0f) * 0.5f);
    while (r * (r + 1) / 2 > t) --r;
    while ((r + 1) * (r + 2) / 2 <= t) ++r;
    tm = r;
    tn = t - r * (r + 1) / 2;
  } else {
    tm = t / p.n_n;
    tn = t % p.n_n;
  }
}

// TMA producer (one lane): 4 operand tiles per 32-wide K stage, running ahead across tile
// boundaries through the STAGES ring; output tiles BM x BNT.
template <int BNT, int STAGES>
__device__ __forceinline__ void produce(const CUtensorMap *ma_hi, const CUtensorMap *ma_lo,
                                        const CUtensorMap *mb_hi, const CUtensorMap *mb_lo,
                                        const TcGemmParams &p, uint8_t *smem, uint64_t *full,
                                        uint64_t *empty, int ktiles, DevStatus *st) {
  constexpr uint32_t tile_b = BNT * BK * 4, stage_bytes = 2 * kTileA + 2 * tile_b;
  tc::tma_prefetch_desc(ma_hi);
  tc::tma_prefetch_desc(ma_lo);
  tc::tma_prefetch_desc(mb_hi);
  tc::tma_prefetch_desc(mb_lo);
  int g = 0;
  for (int t = blockIdx.x; t < p.n_tiles; t += gridDim.x) {
    int tm, tn;
    tile_coords(p, t, tm, tn);
    const int32_t m0 = tm * BM, n0 = tn * BNT;
    for (int kt = 0; kt < ktiles; ++kt, ++g) {
      const int s = g % STAGES;
      if (g >= STAGES && !tc::mbar_wait(&empty[s], ((g / STAGES) - 1) & 1, st)) return;
      uint8_t *base = smem + s * stage_bytes;
      tc::mbar_arrive_expect_tx(&full[s], stage_bytes);
      const int32_t k0 = kt * BK;
      tc::tma_load_2d(base, ma_hi, k0, m0, &full[s]);
      tc::tma_load_2d(base + kTileA, ma_lo, k0, m0, &full[s]);
      tc::tma_load_2d(base + 2 * kTileA, mb_hi, k0, n0, &full[s]);
      tc::tma_load_2d(base + 2 * kTileA + tile_b, mb_lo, k0, n0, &full[s]);
    }
  }
}

// Epilogue of one 64-column half h of a tile (four warps, thread = row rl of the tile):
// alpha * (r0 | r1) into C, by TMA reduce-add through the 128-byte-swizzled staging boxes,
// or by read-modify-write when C has no tensor map.
__device__ __forceinline__ void store_half(const TcGemmParams &p, const CUtensorMap *mc,
                                           uint8_t *staging, const float *r0, const float *r1,
                                           int rl, int64_t row, int64_t m0, int64_t n0, int h,
                                           bool leader) {
  if (p.tma_c) {
    uint8_t *rowp0 = staging + rl * 128;
    uint8_t *rowp1 = staging + BM * 128 + rl * 128;
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int su = (u ^ (rl & 7)) * 16;
      *reinterpret_cast<float4 *>(rowp0 + su) =
          make_float4(p.alpha * r0[4 * u], p.alpha * r0[4 * u + 1], p.alpha * r0[4 * u + 2],
                      p.alpha * r0[4 * u + 3]);
      *reinterpret_cast<float4 *>(rowp1 + su) =
          make_float4(p.alpha * r1[4 * u], p.alpha * r1[4 * u + 1], p.alpha * r1[4 * u + 2],
                      p.alpha * r1[4 * u + 3]);
    }
    tc::fence_proxy_async_smem();
    tc::named_barrier(1, 128);
    if (leader) {
      tc::tma_reduce_add_2d(mc, (int32_t)(n0 + h * 64), (int32_t)m0, staging);
      tc::tma_reduce_add_2d(mc, (int32_t)(n0 + h * 64 + 32), (int32_t)m0, staging + BM * 128);
      tc::bulk_commit();
      tc::bulk_wait_read_all();  // staging may be overwritten after the next barrier
    }
    tc::named_barrier(1, 128);
  } else if (row < p.M) {
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      const int64_t c0 = n0 + h * 64 + i, c1 = c0 + 32;
      if (c0 < p.N) p.c[row * p.ldc + c0] = fmaf(p.alpha, r0[i], p.c[row * p.ldc + c0]);
      if (c1 < p.N) p.c[row * p.ldc + c1] = fmaf(p.alpha, r1[i], p.c[row * p.ldc + c1]);
    }
  }
}

__global__ void __launch_bounds__(kThreads, 1)
tc_gemm_short_sums_kernel(const __grid_constant__ CUtensorMap ma_hi,
                      const __grid_constant__ CUtensorMap ma_lo,
                      const __grid_constant__ CUtensorMap mb_hi,
                      const __grid_constant__ CUtensorMap mb_lo,
                      const __grid_constant__ CUtensorMap mc, TcGemmParams p,
                      DevStatus *st) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint8_t *staging = smem + kStages * kStageBytes;
  uint64_t *full = (uint64_t *)(staging + kStagingBytes);
  uint64_t *empty = full + kStages;
  uint64_t *hfull = empty + kStages;        // [3] head-product accumulator ready
  uint64_t *hempty = hfull + kHeadBufs;     // [3] head-product accumulator drained
  uint64_t *xfull = hempty + kHeadBufs;     // cross-product accumulator ready (per tile)
  uint64_t *xempty = xfull + 1;             // cross-product accumulator drained
  uint32_t *tmem_slot = (uint32_t *)(xempty + 1);

  __shared__ int s_skip;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  if (threadIdx.x == 0) s_skip = (st && st->status != 0);
  __syncthreads();
  if (s_skip) return;  // uniform for the whole CTA, before any barrier or TMEM use
  const int ktiles = (int)((p.K + BK - 1) / BK);

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      tc::mbar_init(&full[s], 1);
      tc::mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < kHeadBufs; ++b) {
      tc::mbar_init(&hfull[b], 1);
      tc::mbar_init(&hempty[b], 4);  // one arrival per epilogue warp
    }
    tc::mbar_init(xfull, 1);
    tc::mbar_init(xempty, 4);
    tc::mbar_fence_init();
  }
  if (warp == 1) tc::tmem_alloc(tmem_slot, kTmemCols);
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0 && lane == 0) {
    produce<BN, kStages>(&ma_hi, &ma_lo, &mb_hi, &mb_lo, p, smem, full, empty, ktiles, st);
  } else if (warp == 1 && lane == 0) {
    // ---------------- MMA issuer ----------------
    constexpr uint32_t idesc = tc::instr_desc(2, 2, BM, BN, 0, 0);
    int g = 0, hg = 0, it = 0, hb = 0;
    bool ok = true;
    for (int t = blockIdx.x; t < p.n_tiles && ok; t += gridDim.x, ++it) {
      if (it >= 1) {   // the previous tile's cross sum drained
        ok = tc::mbar_wait(xempty, (it - 1) & 1, st);
        if (!ok) break;
        tc::tc_fence_after();
      }
      const uint32_t dx = tmem + (uint32_t)(kHeadBufs * BN);
      for (int kt = 0; kt < ktiles; ++kt, ++g) {
        const int s = g % kStages;
        if (kt % kHeadGroup == 0) {
          hb = hg % kHeadBufs;
          if (hg >= kHeadBufs) {
            ok = tc::mbar_wait(&hempty[hb], ((hg / kHeadBufs) - 1) & 1, st);
            if (!ok) break;
            tc::tc_fence_after();
          }
        }
        ok = tc::mbar_wait(&full[s], (g / kStages) & 1, st);
        if (!ok) break;
        tc::tc_fence_after();
        const uint32_t dh = tmem + (uint32_t)(hb * BN);
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
          tc::mma_tf32(dh, dah, dbh, idesc, (kt % kHeadGroup != 0 || kk > 0) ? 1u : 0u);
          tc::mma_tf32(dx, dah, dbl, idesc, (kt > 0 || kk > 0) ? 1u : 0u);
          tc::mma_tf32(dx, dal, dbh, idesc, 1u);
        }
        tc::mma_commit(&empty[s]);   // frees the stage once these MMAs have read it
        if (kt % kHeadGroup == kHeadGroup - 1 || kt == ktiles - 1) {
          tc::mma_commit(&hfull[hb]);  // the head sum of this group is complete
          ++hg;
        }
      }
      if (!ok) break;
      tc::mma_commit(xfull);           // the tile's cross sum is complete
    }
  } else if (warp >= 2) {
    // ---------------- epilogue ----------------
    const int q = warp & 3;            // TMEM lane quarter this warp may access
    const int rl = q * 32 + lane;      // row within the tile
    const bool leader = (warp == 2 && lane == 0);
    const int ngroups = (ktiles + kHeadGroup - 1) / kHeadGroup;
    int hg = 0, it = 0;
    bool ok = true;
    for (int t = blockIdx.x; t < p.n_tiles && ok; t += gridDim.x, ++it) {
      float acc[BN];
#pragma unroll
      for (int i = 0; i < BN; ++i) acc[i] = 0.f;
      // this warp's lane quarter of an accumulator -> acc (two loads in flight per wait)
      auto drain = [&](uint32_t col) {
        const uint32_t ta = tmem + ((uint32_t)(q * 32) << 16) + col;
#pragma unroll
        for (int c = 0; c < BN / 32; c += 2) {
          uint32_t r0[32], r1[32];
          tc::tmem_ld32(ta + (uint32_t)(c * 32), r0);
          tc::tmem_ld32(ta + (uint32_t)(c * 32 + 32), r1);
          tc::tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            acc[c * 32 + i] += __uint_as_float(r0[i]);
            acc[c * 32 + 32 + i] += __uint_as_float(r1[i]);
          }
        }
        tc::tc_fence_before();
        __syncwarp();
      };
      // each warp drains its lane quarter on its own; the four agree once per tile.  The
      // cross sum is drained before the tile's last head sum (both are complete by then):
      // the next tile's first MMAs wait for the cross sum only, so they start one drain
      // earlier.
      auto drain_head = [&](int gi) -> bool {
        const int hb = (hg + gi) % kHeadBufs;
        int okl = 0;
        if (lane == 0) okl = tc::mbar_wait(&hfull[hb], ((hg + gi) / kHeadBufs) & 1, st) ? 1 : 0;
        if (!__shfl_sync(0xffffffffu, okl, 0)) return false;
        tc::tc_fence_after();
        drain((uint32_t)(hb * BN));
        if (lane == 0) tc::mbar_arrive(&hempty[hb]);
        return true;
      };
      for (int gi = 0; gi < ngroups - 1 && ok; ++gi) ok = drain_head(gi);
      if (ok) {
        int okl = 0;
        if (lane == 0) okl = tc::mbar_wait(xfull, it & 1, st) ? 1 : 0;
        if (__shfl_sync(0xffffffffu, okl, 0)) {
          tc::tc_fence_after();
          drain((uint32_t)(kHeadBufs * BN));
          if (lane == 0) tc::mbar_arrive(xempty);
        } else {
          ok = false;
        }
      }
      if (ok) ok = drain_head(ngroups - 1);
      hg += ngroups;
      ok = tc::named_barrier_and(1, 128, ok);   // uniform across the four warps
      if (!ok) break;
      int tm, tn;
      tile_coords(p, t, tm, tn);
      const int64_t m0 = (int64_t)tm * BM, n0 = (int64_t)tn * BN;
      const int64_t row = m0 + rl;
#pragma unroll
      for (int h = 0; h < 2; ++h)
        store_half(p, &mc, staging, acc + h * 64, acc + h * 64 + 32, rl, row, m0, n0, h, leader);
    }
    if (leader) tc::bulk_wait_all();
  }
  tc::tc_fence_before();
  __syncthreads();
  if (warp == 1) tc::tmem_dealloc(tmem, kTmemCols);
}

// One TMEM sum per tile (the sweep's updates): two BNT-column tile accumulators used in
// turn, so the next tile's MMAs overlap this tile's epilogue; the epilogue stages each
// 64-column part straight from its TMEM loads and releases the accumulator after the last.
// BNT = 128 (three stages of 64 KB) or 256 (two of 96 KB: per MMA the same A tile feeds
// twice the columns, so a quarter fewer operand bytes cross shared memory per product).
template <int BNT>
__global__ void __launch_bounds__(kThreads, 1)
tc_gemm_one_sum_kernel(const __grid_constant__ CUtensorMap ma_hi,
                       const __grid_constant__ CUtensorMap ma_lo,
                       const __grid_constant__ CUtensorMap mb_hi,
                       const __grid_constant__ CUtensorMap mb_lo,
                       const __grid_constant__ CUtensorMap mc, TcGemmParams p, DevStatus *st) {
  constexpr int STAGES = BNT == 256 ? 2 : kStages;
  constexpr uint32_t tile_b = BNT * BK * 4, stage_bytes = 2 * kTileA + 2 * tile_b;
  static_assert(1024 + STAGES * stage_bytes + kStagingBytes + 256 <= kSmemBytes, "smem");
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint8_t *staging = smem + STAGES * stage_bytes;
  uint64_t *full = (uint64_t *)(staging + kStagingBytes);
  uint64_t *empty = full + STAGES;
  uint64_t *tfull = empty + STAGES;    // [2] accumulator ready
  uint64_t *tempty = tfull + 2;        // [2] accumulator drained
  uint32_t *tmem_slot = (uint32_t *)(tempty + 2);
  int *epi_ok = (int *)(tmem_slot + 1);

  __shared__ int s_skip;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  if (threadIdx.x == 0) s_skip = (st && st->status != 0);
  __syncthreads();
  if (s_skip) return;  // uniform for the whole CTA, before any barrier or TMEM use
  const int ktiles = (int)((p.K + BK - 1) / BK);

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      tc::mbar_init(&full[s], 1);
      tc::mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      tc::mbar_init(&tfull[b], 1);
      tc::mbar_init(&tempty[b], 4);  // one arrival per epilogue warp
    }
    tc::mbar_fence_init();
  }
  if (warp == 1) tc::tmem_alloc(tmem_slot, 2 * BNT);
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0 && lane == 0) {
    produce<BNT, STAGES>(&ma_hi, &ma_lo, &mb_hi, &mb_lo, p, smem, full, empty, ktiles, st);
  } else if (warp == 1 && lane == 0) {
    // ---------------- MMA issuer ----------------
    constexpr uint32_t idesc = tc::instr_desc(2, 2, BM, BNT, 0, 0);
    int g = 0, it = 0;
    bool ok = true;
    for (int t = blockIdx.x; t < p.n_tiles && ok; t += gridDim.x, ++it) {
      const int b = it & 1;
      if (it >= 2) {
        ok = tc::mbar_wait(&tempty[b], ((it / 2) - 1) & 1, st);
        if (!ok) break;
        tc::tc_fence_after();
      }
      const uint32_t dt = tmem + (uint32_t)(b * BNT);
      for (int kt = 0; kt < ktiles; ++kt, ++g) {
        const int s = g % STAGES;
        ok = tc::mbar_wait(&full[s], (g / STAGES) & 1, st);
        if (!ok) break;
        tc::tc_fence_after();
        const uint32_t a_hi = tc::smem_u32(smem + s * stage_bytes);
        const uint32_t a_lo = a_hi + kTileA;
        const uint32_t b_hi = a_hi + 2 * kTileA;
        const uint32_t b_lo = b_hi + tile_b;
#pragma unroll
        for (int kk = 0; kk < BK / 8; ++kk) {  // 8 tf32 = 32 bytes per MMA
          const uint32_t off = kk * 32;
          const uint64_t dah = tc::smem_desc_sw128(a_hi + off, 16, 1024);
          const uint64_t dal = tc::smem_desc_sw128(a_lo + off, 16, 1024);
          const uint64_t dbh = tc::smem_desc_sw128(b_hi + off, 16, 1024);
          const uint64_t dbl = tc::smem_desc_sw128(b_lo + off, 16, 1024);
          tc::mma_tf32(dt, dah, dbh, idesc, (kt > 0 || kk > 0) ? 1u : 0u);
          tc::mma_tf32(dt, dah, dbl, idesc, 1u);
          tc::mma_tf32(dt, dal, dbh, idesc, 1u);
        }
        tc::mma_commit(&empty[s]);  // frees the stage once these MMAs have read it
      }
      tc::mma_commit(&tfull[b]);    // accumulator complete (or abandoned after a timeout)
    }
  } else if (warp >= 2) {
    // ---------------- epilogue ----------------
    const int q = warp & 3;            // TMEM lane quarter this warp may access
    const int rl = q * 32 + lane;      // row within the tile
    const bool leader = (warp == 2 && lane == 0);
    int it = 0;
    for (int t = blockIdx.x; t < p.n_tiles; t += gridDim.x, ++it) {
      const int b = it & 1;
      if (leader) *epi_ok = tc::mbar_wait(&tfull[b], (it / 2) & 1, st) ? 1 : 0;
      tc::named_barrier(1, 128);
      if (!*epi_ok) break;             // same value for all four warps
      tc::tc_fence_after();
      int tm, tn;
      tile_coords(p, t, tm, tn);
      const int64_t m0 = (int64_t)tm * BM, n0 = (int64_t)tn * BNT;
      const int64_t row = m0 + rl;
#pragma unroll 1
      for (int h = 0; h < BNT / 64; ++h) {
        uint32_t r0[32], r1[32];
        const uint32_t ta = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(b * BNT + h * 64);
        tc::tmem_ld32(ta, r0);
        tc::tmem_ld32(ta + 32, r1);
        tc::tmem_ld_wait();
        if (h == BNT / 64 - 1) {  // this warp's reads of the accumulator are done: release it
          tc::tc_fence_before();
          __syncwarp();
          if (lane == 0) tc::mbar_arrive(&tempty[b]);
        }
        float v0[32], v1[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          v0[i] = __uint_as_float(r0[i]);
          v1[i] = __uint_as_float(r1[i]);
        }
        store_half(p, &mc, staging, v0, v1, rl, row, m0, n0, h, leader);
      }
    }
    if (leader) tc::bulk_wait_all();
  }
  tc::tc_fence_before();
  __syncthreads();
  if (warp == 1) tc::tmem_dealloc(tmem, 2 * BNT);
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
  GPTQ_TRY(ensure_smem_attr((const void *)tc_gemm_short_sums_kernel, (int)kSmemBytes));
  GPTQ_TRY(ensure_smem_attr((const void *)tc_gemm_one_sum_kernel<BN>, (int)kSmemBytes));
  GPTQ_TRY(ensure_smem_attr((const void *)tc_gemm_one_sum_kernel<2 * BN>, (int)kSmemBytes));
  // 256-wide tiles for one-sum products that ask for them (not for triangles: their
  // diagonal tiles are square)
  const bool wide = g.one_sum && g.wide && !g.lower_only;
  const int bnt = wide ? 2 * BN : BN;
  CUtensorMap mah, mal, mbh, mbl;
  // maps cover exactly the [M, K] / [N, K] operand windows: out-of-range reads are zero
  if (!make_tmap_f32(&mah, g.a_hi, g.M, g.K, g.lda, BM) ||
      !make_tmap_f32(&mal, g.a_lo, g.M, g.K, g.lda, BM) ||
      !make_tmap_f32(&mbh, g.b_hi, g.N, g.K, g.ldb, bnt) ||
      !make_tmap_f32(&mbl, g.b_lo, g.N, g.K, g.ldb, bnt))
    return GPTQ_ERR_UNSUPPORTED;
  CUtensorMap mc;
  memset(&mc, 0, sizeof(mc));
  const bool tma_c = !g.trans_c && make_tmap_f32(&mc, g.c, g.M, g.N, g.ldc, BM);
  if (g.trans_c) return GPTQ_ERR_UNSUPPORTED;
  int num_sms = 0;
  GPTQ_TRY(device_sm_count(&num_sms));
  TcGemmParams p{};
  p.tma_c = tma_c ? 1 : 0;
  p.M = g.M; p.N = g.N; p.K = g.K;
  p.c = g.c; p.ldc = g.ldc; p.alpha = g.alpha;
  p.n_m = (int)ceil_div(g.M, BM);
  p.n_n = (int)ceil_div(g.N, bnt);
  p.lower_only = g.lower_only && g.M >= g.N;
  p.n_tiles = p.lower_only ? p.n_n * (p.n_n + 1) / 2 + (p.n_m - p.n_n) * p.n_n : p.n_m * p.n_n;
  const int cap = g.max_ctas < 0 ? p.n_tiles
                  : (g.max_ctas > 0 && g.max_ctas < num_sms) ? g.max_ctas : num_sms;
  const int grid = p.n_tiles < cap ? p.n_tiles : cap;
  GPTQ_TRY(launch_kernel(!g.one_sum ? tc_gemm_short_sums_kernel
                         : wide     ? tc_gemm_one_sum_kernel<2 * BN>
                                    : tc_gemm_one_sum_kernel<BN>,
                         grid, kThreads, kSmemBytes, s, mah, mal, mbh, mbl, mc, p, st));
  return GPTQ_OK;
}

}  // namespace gptq
