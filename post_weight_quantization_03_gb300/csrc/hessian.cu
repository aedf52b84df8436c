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
// running sum spans more than one segment.  fp32 inputs run on the tensor cores too, as
// kind::tf32 products of TF32 head/tail splits (3xTF32); tiny shapes take a CUDA-core
// kernel.
#include <algorithm>
#include <cstring>

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
// tcgen05 SYRK on CTA pairs: one cluster of two CTAs (two SMs) per 256 x 256 tile of H on
// or below the diagonal, one cta_group::2 MMA stream for the pair.  CTA r of the pair holds
// the tile's rows 128 r .. 128 r + 127 (its A half) and columns 128 r .. 128 r + 127 (its B
// half) of each 128-token stage, and its half of the accumulator (128 rows x 256 columns)
// in its own TMEM.  Per SM and 16 tokens that is 8 KB of X written into shared memory and
// 8 KB read by the tensor core, against 12 KB and 12 KB for a 128 x 256 tile on one SM
// with the same output per SM.
//   warp 0      : TMA producer of this CTA's halves; both CTAs' copies complete on the
//                 even CTA's stage barrier
//   warp 1      : TMEM allocator (2 x 256 columns, both SMs); in the even CTA the MMA
//                 issuer, whose commits arrive on the barriers of both CTAs
//   warps 2..9  : drain this SM's TMEM segments into fp32 registers (the accumulator
//                 buffer is free again once both CTAs' drains have arrived on the even
//                 CTA's barrier), then write H and its mirror
// All clusters of a wave walk the tokens in the same order, so each chunk of X is fetched
// from HBM about once per wave and served to the other tiles from L2.
//
// Balanced last round: when the tiles do not fill a whole number of rounds of the SM pairs,
// each tile of the last, partial round is cut at one token stage into a head and a tail.
// The heads run beside the first batch of tails on the pairs the partial round leaves idle,
// the later batches of tails follow on the same pairs, and the cut is placed so that the
// heads and the k batches of tails end together: a round of about k/(k+1) tile-times
// instead of one.  The heads walk the same tokens in step, and so does each batch of tails,
// so X stays shared through L2.  Head and tail add into H, which the launcher zeroes first
// (only calls that overwrite H are cut, so the sum 0 + head + tail is the same in either
// order).
// ---------------------------------------------------------------------------------------
// 128 tokens per stage (measured against 64: 2.64 against 2.99 ms at d_in = 4096, 42.5
// against 45.6 ms at 28672, the same at 11008; the same bytes in flight, half the barrier
// round trips per MMA)
constexpr int TB_M = 128, TB_N = 256, TB_K = 128;     // per-CTA rows, tile columns, tokens
constexpr int T_STAGES = 3;
constexpr uint32_t T_BOX = 64 * TB_K * 2;                 // 16 KB: 64 channels x 128 tokens
constexpr uint32_t T_HALF = 2 * T_BOX;                    // 32 KB: 128 channels
constexpr uint32_t T_STAGE = 2 * T_HALF;                  // A half + B half: 64 KB
constexpr int T_EPI_WARPS = 8;
constexpr int T_THREADS = 64 + 32 * T_EPI_WARPS;          // 320
constexpr size_t T_SMEM = 1024 + T_STAGES * T_STAGE + 256;

struct HessTcParams {
  int64_t d, n_tok;
  int n_blocks;       // ceil(d / 256)
  int seg_stages;     // stages (of TB_K tokens) per accumulation segment
  float *H;
  int accumulate;
  uint64_t wait_ns;   // budget of every mbarrier wait
  int lost_stage;     // test hook: the producers issue nothing for this stage (-1: none)
  int full_tiles;     // units [0, full_tiles): whole tiles, stored (added when accumulating)
  int cut_tiles;      // then cut_tiles heads and cut_tiles tails, added onto a zeroed H
  int cut_stage;      // first token stage of a tail
  int tma_h;          // 1: off-diagonal tiles leave through the H tensor map
};

template <int FMT>  // 0 = fp16, 1 = bf16
__global__ void __launch_bounds__(T_THREADS, 1)
hessian_tc_kernel(const __grid_constant__ CUtensorMap mx, const __grid_constant__ CUtensorMap mh,
                  HessTcParams p, DevStatus *st) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint64_t *full = (uint64_t *)(smem + T_STAGES * T_STAGE);   // even CTA's: both halves in
  uint64_t *empty = full + T_STAGES;    // each CTA's: stage consumed by the pair's MMAs
  uint64_t *tfull = empty + T_STAGES;   // [2] each CTA's: accumulator buffer ready to drain
  uint64_t *tempty = tfull + 2;         // [2] even CTA's: buffer drained by both CTAs
  uint64_t *mdone = tempty + 2;         // even CTA's: every MMA it issued has completed
  uint32_t *tmem_slot = (uint32_t *)(mdone + 1);

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const uint32_t rank = tc::cluster_ctarank();
  // unit -> tile and token stages [g0, g1)
  const int total_all = (int)((p.n_tok + TB_K - 1) / TB_K);
  int tile = blockIdx.x / 2, g0 = 0, g1 = total_all;
  bool add = false;
  if (tile >= p.full_tiles + p.cut_tiles) {
    tile -= p.cut_tiles;
    g0 = p.cut_stage;
    add = true;
  } else if (tile >= p.full_tiles) {
    g1 = p.cut_stage;
    add = true;
  }
  // tile index -> (row block I, column block J), I >= J: column blocks in order
  int I = 0, J = 0;
  {
    int idx = tile;
    for (J = 0;; ++J) {
      const int cnt = p.n_blocks - J;
      if (idx < cnt) { I = J + idx; break; }
      idx -= cnt;
    }
  }
  const int64_t m0 = (int64_t)I * 2 * TB_M + rank * TB_M;      // this CTA's rows
  const int64_t n0 = (int64_t)J * TB_N;                        // the tile's columns
  const int total = g1 - g0;   // stages of this unit
  const int nseg = (total + p.seg_stages - 1) / p.seg_stages;

  if (threadIdx.x == 0) {
    for (int s = 0; s < T_STAGES; ++s) {
      tc::mbar_init(&full[s], 1);
      tc::mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      tc::mbar_init(&tfull[b], 1);
      tc::mbar_init(&tempty[b], 2 * T_EPI_WARPS);
    }
    tc::mbar_init(mdone, 1);
    tc::mbar_fence_init();
  }
  if (warp == 1) tc::tmem_alloc_pair(tmem_slot, 512);
  tc::tc_fence_before();
  tc::cluster_sync();          // both CTAs' barriers initialised, TMEM allocated
  tc::tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0 && lane == 0) {
    tc::tma_prefetch_desc(&mx);
    const uint32_t full0 = tc::mapa_shared(tc::smem_u32(full), 0);
    for (int g = 0; g < total; ++g) {
      const int s = g % T_STAGES;
      if (g >= T_STAGES &&
          !tc::mbar_wait(&empty[s], ((g / T_STAGES) - 1) & 1, st, p.wait_ns))
        break;
      if (g == p.lost_stage) continue;   // test hook: no copy and no arrival for this stage
      uint8_t *a = smem + s * T_STAGE;
      uint8_t *b = a + T_HALF;
      const int32_t t0 = (g0 + g) * TB_K;
      const int32_t nb = (int32_t)(n0 + rank * TB_M);
      const uint32_t bar = full0 + (uint32_t)(s * sizeof(uint64_t));
      if (rank == 0) tc::mbar_arrive_expect_tx(&full[s], 2 * T_STAGE);
      tc::tma_load_2d_pair(a, &mx, (int32_t)m0, t0, bar);
      tc::tma_load_2d_pair(a + T_BOX, &mx, (int32_t)m0 + 64, t0, bar);
      tc::tma_load_2d_pair(b, &mx, nb, t0, bar);
      tc::tma_load_2d_pair(b + T_BOX, &mx, nb + 64, t0, bar);
    }
  } else if (warp == 1 && lane == 0 && rank == 0) {
    constexpr uint32_t idesc = tc::instr_desc(FMT, FMT, 2 * TB_M, TB_N, 1, 1);
    int g = 0;
    bool ok = true;
    for (int sg = 0; sg < nseg && ok; ++sg) {
      const int buf = sg & 1;
      if (sg >= 2) {
        ok = tc::mbar_wait_cluster(&tempty[buf], ((sg / 2) - 1) & 1, st, p.wait_ns);
        if (!ok) break;
        tc::tc_fence_after();
      }
      const uint32_t dt = tmem + (uint32_t)(buf * TB_N);
      const int gend = min(total, (sg + 1) * p.seg_stages);
      for (int first = 1; g < gend; ++g, first = 0) {
        const int s = g % T_STAGES;
        ok = tc::mbar_wait(&full[s], (g / T_STAGES) & 1, st, p.wait_ns);
        if (!ok) break;
        tc::tc_fence_after();
        const uint32_t a = tc::smem_u32(smem + s * T_STAGE);
        const uint32_t b = a + T_HALF;
#pragma unroll
        for (int kk = 0; kk < TB_K / 16; ++kk) {  // 16 tokens = 2048 bytes per MMA
          const uint64_t da = tc::smem_desc_sw128(a + kk * 2048, T_BOX, 1024);
          const uint64_t db = tc::smem_desc_sw128(b + kk * 2048, T_BOX, 1024);
          tc::mma_f16_pair(dt, da, db, idesc, (first && kk == 0) ? 0u : 1u);
        }
        tc::mma_commit_pair(&empty[s], 3);
      }
      tc::mma_commit_pair(&tfull[buf], 3);   // segment complete (or abandoned after a timeout)
    }
    // nothing of this CTA's MMAs may still be running when the pair's TMEM is released
    tc::mma_commit_pair(mdone, 1);
    tc::mbar_wait(mdone, 0, st, p.wait_ns);
  } else if (warp >= 2) {
    const int e = warp - 2, q = warp & 3, h = e / 4;
    const uint32_t tempty0 = tc::mapa_shared(tc::smem_u32(tempty), 0);
    float acc[128];
#pragma unroll
    for (int i = 0; i < 128; ++i) acc[i] = 0.f;
    bool ok = true;
    for (int sg = 0; sg < nseg && ok; ++sg) {
      const int buf = sg & 1;
      int okl = 0;
      if (lane == 0) okl = tc::mbar_wait(&tfull[buf], (sg / 2) & 1, st, p.wait_ns) ? 1 : 0;
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
      if (lane == 0) tc::mbar_arrive_cluster(tempty0 + (uint32_t)(buf * sizeof(uint64_t)));
    }
    const int64_t rl = q * 32 + lane;   // row within this CTA's 128
    const int64_t r = m0 + rl;
    const int64_t d = p.d;
    if (p.tma_h && I != J) {
      // Off-diagonal tile: the operand ring is free now (the last MMA has completed), so the
      // tile goes out through it by TMA, first as it is (H rows m0.., columns n0..), then
      // transposed (H rows n0.., columns m0..): eight boxes of 32 columns x 128 rows, with
      // the 128-byte swizzle, each time.  A store overwrites H; an accumulating call or a cut
      // tile's part adds in L2 instead.  All eight warps agree on `ok` first.
      ok = tc::named_barrier_and(1, 32 * T_EPI_WARPS, ok);
      const bool lead = warp == 2 && lane == 0;
      const bool red = add || p.accumulate;
      if (ok && m0 < d) {
        uint8_t *stg = smem;
        // as it is: column c of this thread's half -> box (h * 128 + c) / 32, row rl
#pragma unroll
        for (int u = 0; u < 32; ++u) {
          const int c = 4 * u, b = h * 4 + c / 32, ch = (c % 32) / 4;
          *reinterpret_cast<float4 *>(stg + b * 16384 + rl * 128 + ((ch ^ (rl & 7)) * 16)) =
              make_float4(2.0f * acc[c], 2.0f * acc[c + 1], 2.0f * acc[c + 2], 2.0f * acc[c + 3]);
        }
        tc::fence_proxy_async_smem();
        tc::named_barrier(2, 32 * T_EPI_WARPS);
        if (lead) {
          for (int b = 0; b < 8; ++b) {
            const int32_t x = (int32_t)(n0 + 32 * b);
            if (x >= d) continue;     // boxes wholly past the last column are not issued
            if (red) tc::tma_reduce_add_2d(&mh, x, (int32_t)m0, stg + b * 16384);
            else tc::tma_store_2d(&mh, x, (int32_t)m0, stg + b * 16384);
          }
          tc::bulk_commit();
          tc::bulk_wait_read_all();   // the staging is rewritten next
        }
        tc::named_barrier(2, 32 * T_EPI_WARPS);
        // transposed: tile column h * 128 + i -> H row n0 + h * 128 + i, this thread's row
        // rl -> H column m0 + rl; box (rl / 32) + 4 h, row i, column rl % 32
#pragma unroll
        for (int i = 0; i < 128; ++i) {
          const int b = (int)(rl / 32) + 4 * h, cc = (int)(rl % 32);
          *reinterpret_cast<float *>(stg + b * 16384 + i * 128 + (((cc / 4) ^ (i & 7)) * 16) +
                                     (cc % 4) * 4) = 2.0f * acc[i];
        }
        tc::fence_proxy_async_smem();
        tc::named_barrier(2, 32 * T_EPI_WARPS);
        if (lead) {
          for (int hh = 0; hh < 2; ++hh)
            for (int b = 0; b < 4; ++b) {
              uint8_t *src = stg + (b + 4 * hh) * 16384;
              const int32_t x = (int32_t)(m0 + 32 * b), y = (int32_t)(n0 + 128 * hh);
              if (x >= d || y >= d) continue;
              if (red) tc::tma_reduce_add_2d(&mh, x, y, src);
              else tc::tma_store_2d(&mh, x, y, src);
            }
          tc::bulk_commit();
          tc::bulk_wait_all();
        }
      }
    } else if (ok && r < d && add) {
#pragma unroll
      for (int i = 0; i < 128; ++i) {
        const int64_t c = n0 + h * 128 + i;
        if (c < d && c <= r) {
          const float v = 2.0f * acc[i];
          atomicAdd(&p.H[r * d + c], v);
          if (c != r) atomicAdd(&p.H[c * d + r], v);
        }
      }
    } else if (ok && r < d) {
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
  __syncwarp();
  tc::tc_fence_before();
  tc::cluster_sync();          // neither CTA leaves while the other may still signal it
  tc::tc_fence_after();
  if (warp == 1) tc::tmem_dealloc_pair(tmem, 512);
}

// ---------------------------------------------------------------------------------------
// fp32 inputs on the tensor cores: tcgen05 kind::tf32 in the 3xTF32 scheme.  One CTA per
// 128 x 128 tile of H on or below the diagonal.  Per stage, 32 tokens of the tile's two
// channel ranges arrive by TMA as token-major boxes (channels contiguous, 128-byte
// swizzle); four converter warps transpose them into the K-major layout the MMA reads
// (rows = channels, 32 tokens = one 128-byte swizzled row) while splitting every element
// into its TF32 head (low 13 mantissa bits cleared) and the exact remainder; the MMA warp
// accumulates head head^T + head tail^T + tail head^T, which reproduces the fp32 products
// to about 2^-21 relative.
//   warp 0      : TMA producer (raw ring of F_RAW stages)
//   warp 1      : TMEM allocator (2 x 128 columns) + MMA issuer (converted ring of F_CONV)
//   warps 2..5  : drain the accumulator every kSegTokensTf32 tokens into fp32 registers,
//                 then write H and its mirror
//   warps 6..9  : transpose + head/tail split, raw stage -> converted stage
// ---------------------------------------------------------------------------------------
constexpr int F_M = 128, F_K = 32;               // tile edge (channels), tokens per stage
constexpr int F_RAW = 2, F_CONV = 2;
constexpr uint32_t F_BOX = 32 * F_K * 4;         // 32 channels x 32 tokens of fp32: 4 KB
constexpr uint32_t F_TILE = F_M * F_K * 4;       // 128 channels x 32 tokens: 16 KB
constexpr uint32_t F_RAW_STAGE = 2 * F_TILE;     // the two channel ranges, token-major
constexpr uint32_t F_CONV_STAGE = 4 * F_TILE;    // A, B heads then A, B tails, K-major
constexpr int F_CONV_WARPS = 4;
constexpr int F_THREADS = 64 + 32 * 4 + 32 * F_CONV_WARPS;   // 320
constexpr size_t F_SMEM = 1024 + F_RAW * F_RAW_STAGE + F_CONV * F_CONV_STAGE + 256;

struct HessF32Params {
  int64_t d, n_tok;
  int seg_stages;     // stages (of F_K tokens) per accumulation segment
  float *H;
  int accumulate;
};

__global__ void __launch_bounds__(F_THREADS, 1)
hessian_tf32_kernel(const __grid_constant__ CUtensorMap mx, HessF32Params p, DevStatus *st) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint8_t *raw = smem;                                   // F_RAW x F_RAW_STAGE
  uint8_t *cvt = smem + F_RAW * F_RAW_STAGE;             // F_CONV x F_CONV_STAGE
  uint64_t *rfull = (uint64_t *)(cvt + F_CONV * F_CONV_STAGE);
  uint64_t *rempty = rfull + F_RAW;     // raw stage read by all converter warps
  uint64_t *cfull = rempty + F_RAW;     // converted stage written by all converter warps
  uint64_t *cempty = cfull + F_CONV;    // converted stage consumed by the MMAs
  uint64_t *tfull = cempty + F_CONV;    // [2]: accumulator buffer ready to drain
  uint64_t *tempty = tfull + 2;         // [2]: accumulator buffer drained
  uint32_t *tmem_slot = (uint32_t *)(tempty + 2);

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  int ti, tj;
  lower_tile(blockIdx.x, ti, tj);
  const int64_t m0 = (int64_t)ti * F_M, n0 = (int64_t)tj * F_M;
  const int total = (int)((p.n_tok + F_K - 1) / F_K);
  const int nseg = (total + p.seg_stages - 1) / p.seg_stages;

  if (threadIdx.x == 0) {
    for (int s = 0; s < F_RAW; ++s) {
      tc::mbar_init(&rfull[s], 1);
      tc::mbar_init(&rempty[s], F_CONV_WARPS);
    }
    for (int s = 0; s < F_CONV; ++s) {
      tc::mbar_init(&cfull[s], F_CONV_WARPS);
      tc::mbar_init(&cempty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      tc::mbar_init(&tfull[b], 1);
      tc::mbar_init(&tempty[b], 4);
    }
    tc::mbar_fence_init();
  }
  if (warp == 1) tc::tmem_alloc(tmem_slot, 2 * F_M);
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      tc::tma_prefetch_desc(&mx);
      for (int g = 0; g < total; ++g) {
        const int s = g % F_RAW;
        if (g >= F_RAW && !tc::mbar_wait(&rempty[s], ((g / F_RAW) - 1) & 1, st)) break;
        uint8_t *a = raw + s * F_RAW_STAGE;
        const int32_t t0 = g * F_K;
        tc::mbar_arrive_expect_tx(&rfull[s], F_RAW_STAGE);
#pragma unroll
        for (int q = 0; q < F_M / 32; ++q) {
          tc::tma_load_2d(a + q * F_BOX, &mx, (int32_t)m0 + 32 * q, t0, &rfull[s]);
          tc::tma_load_2d(a + F_TILE + q * F_BOX, &mx, (int32_t)n0 + 32 * q, t0, &rfull[s]);
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc = tc::instr_desc(2, 2, F_M, F_M, 0, 0);
      int g = 0;
      bool ok = true;
      for (int sg = 0; sg < nseg && ok; ++sg) {
        const int buf = sg & 1;
        if (sg >= 2) {
          ok = tc::mbar_wait(&tempty[buf], ((sg / 2) - 1) & 1, st);
          if (!ok) break;
          tc::tc_fence_after();
        }
        const uint32_t dt = tmem + (uint32_t)(buf * F_M);
        const int gend = min(total, (sg + 1) * p.seg_stages);
        for (int first = 1; g < gend; ++g, first = 0) {
          const int s = g % F_CONV;
          ok = tc::mbar_wait(&cfull[s], (g / F_CONV) & 1, st);
          if (!ok) break;
          tc::tc_fence_after();
          const uint32_t ah = tc::smem_u32(cvt + s * F_CONV_STAGE);
          const uint32_t bh = ah + F_TILE, al = ah + 2 * F_TILE, bl = ah + 3 * F_TILE;
#pragma unroll
          for (int kk = 0; kk < F_K / 8; ++kk) {   // 8 tf32 = 32 bytes of each row per MMA
            const uint32_t off = kk * 32;
            const uint64_t dah = tc::smem_desc_sw128(ah + off, 16, 1024);
            const uint64_t dbh = tc::smem_desc_sw128(bh + off, 16, 1024);
            const uint64_t dal = tc::smem_desc_sw128(al + off, 16, 1024);
            const uint64_t dbl = tc::smem_desc_sw128(bl + off, 16, 1024);
            tc::mma_tf32(dt, dah, dbh, idesc, (first && kk == 0) ? 0u : 1u);
            tc::mma_tf32(dt, dah, dbl, idesc, 1u);
            tc::mma_tf32(dt, dal, dbh, idesc, 1u);
          }
          tc::mma_commit(&cempty[s]);
        }
        tc::mma_commit(&tfull[buf]);
      }
    }
  } else if (warp >= 6) {
    // Raw stage: per channel range, four boxes of 32 channels; in box q token t's 128-byte
    // row holds its 32 channels with 16-byte chunk c stored at chunk c ^ (t % 8).  Output:
    // per channel r a 128-byte row of 32 tokens, chunk c (tokens 4c .. 4c + 3) stored at
    // chunk c ^ (r % 8) -- the layout a K-major 128-byte-swizzled TMA box has.
    const int ct = threadIdx.x - 32 * 6;
    for (int g = 0; g < total; ++g) {
      const int rs = g % F_RAW, cs = g % F_CONV;
      int okl = 0;
      if (lane == 0)
        okl = tc::mbar_wait(&rfull[rs], (g / F_RAW) & 1, st) &&
              (g < F_CONV || tc::mbar_wait(&cempty[cs], ((g / F_CONV) - 1) & 1, st));
      if (!__shfl_sync(0xffffffffu, okl, 0)) break;
      const uint8_t *rb = raw + rs * F_RAW_STAGE;
      uint8_t *cb = cvt + cs * F_CONV_STAGE;
#pragma unroll 4
      for (int i = 0; i < 2 * F_M * (F_K / 4) / (32 * F_CONV_WARPS); ++i) {
        const int idx = i * 32 * F_CONV_WARPS + ct;    // (tile, chunk, row), row fastest
        const int tile = idx / (F_M * (F_K / 4));
        const int rem = idx % (F_M * (F_K / 4));
        const int c = rem / F_M, r = rem % F_M;
        const uint8_t *box = rb + tile * F_TILE + (r / 32) * F_BOX;
        const int rc = r % 32;
        float v[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int t = 4 * c + j;
          v[j] = *reinterpret_cast<const float *>(box + t * 128 + (((rc / 4) ^ (t & 7)) * 16) +
                                                  (rc % 4) * 4);
        }
        const float4 h = make_float4(tf32_head(v[0]), tf32_head(v[1]), tf32_head(v[2]),
                                     tf32_head(v[3]));
        const uint32_t o = tile * F_TILE + r * 128 + ((c ^ (r & 7)) * 16);
        *reinterpret_cast<float4 *>(cb + o) = h;
        *reinterpret_cast<float4 *>(cb + 2 * F_TILE + o) =
            make_float4(v[0] - h.x, v[1] - h.y, v[2] - h.z, v[3] - h.w);
      }
      tc::fence_proxy_async_smem();   // the tensor core reads these through the async proxy
      __syncwarp();
      if (lane == 0) {
        tc::mbar_arrive(&rempty[rs]);
        tc::mbar_arrive(&cfull[cs]);
      }
    }
  } else {
    // warps 2..5: drain and write
    const int q = warp & 3;
    float acc[F_M];
#pragma unroll
    for (int i = 0; i < F_M; ++i) acc[i] = 0.f;
    bool ok = true;
    for (int sg = 0; sg < nseg && ok; ++sg) {
      const int buf = sg & 1;
      int okl = 0;
      if (lane == 0) okl = tc::mbar_wait(&tfull[buf], (sg / 2) & 1, st) ? 1 : 0;
      ok = __shfl_sync(0xffffffffu, okl, 0) != 0;
      __syncwarp();
      if (!ok) break;
      tc::tc_fence_after();
      const uint32_t base = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(buf * F_M);
#pragma unroll
      for (int c = 0; c < F_M / 32; ++c) {
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
      for (int i = 0; i < F_M; ++i) {
        const int64_t c = n0 + i;
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
  if (warp == 1) tc::tmem_dealloc(tmem, 2 * F_M);
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
// The 3xTF32 kernel issues 12 MMAs per 32 tokens (three products of four 8-wide steps), so
// its segments are shorter: 64 tokens, 24 MMAs per TMEM running sum (512-token segments,
// 192 MMAs, left H about 1e-5 low).
constexpr int kSegTokensTf32 = 64;

gptq_status launch_hessian_tc(const void *X, int xdtype, int64_t n_tok, int64_t d, int64_t ldx,
                              float *H, int accumulate, DevStatus *st, cudaStream_t s,
                              uint64_t wait_ns = tc::kWaitNs, int lost_stage = -1) {
  GPTQ_TRY(ensure_smem_attr((const void *)hessian_tc_kernel<0>, (int)T_SMEM));
  GPTQ_TRY(ensure_smem_attr((const void *)hessian_tc_kernel<1>, (int)T_SMEM));
  CUtensorMap mx;
  const CUtensorMapDataType dt =
      xdtype == GPTQ_F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  if (!tc::make_tmap_2d(&mx, dt, X, n_tok, d, ldx * 2, 64, TB_K)) return GPTQ_ERR_UNSUPPORTED;
  HessTcParams p{};
  p.d = d;
  p.n_tok = n_tok;
  p.n_blocks = (int)ceil_div(d, TB_N);
  p.seg_stages = kSegTokens / TB_K;
  p.H = H;
  p.accumulate = accumulate;
  p.wait_ns = wait_ns;
  p.lost_stage = lost_stage;
  const int64_t tiles = (int64_t)p.n_blocks * (p.n_blocks + 1) / 2;
  const int total = (int)ceil_div(n_tok, TB_K);
  // H as a tensor map (32-column x 128-row boxes, 128-byte swizzle) when its rows start on
  // 16-byte boundaries: off-diagonal tiles then leave through TMA stores
  CUtensorMap mh;
  memset(&mh, 0, sizeof(mh));
  p.tma_h = (d % 4 == 0) &&
            tc::make_tmap_2d(&mh, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, H, d, d, d * 4, 32, 128) ? 1 : 0;
  p.full_tiles = (int)tiles;
  p.cut_tiles = 0;
  p.cut_stage = total;
  if (!accumulate && lost_stage < 0) {
    int nsm = 0;
    GPTQ_TRY(device_sm_count(&nsm));
    const int64_t pairs = nsm / 2;
    const int64_t r = tiles % pairs, rounds = tiles / pairs + (r ? 1 : 0);
    if (r > 0 && pairs > r) {
      const int64_t k = ceil_div(r, pairs - r);     // batches of tails per idle pair
      // heads and k batches of tails end together: head = k rho / (1 + k rho) of the tokens,
      // in whole accumulation segments, where rho = 1.05 is the time of a tail's token stage
      // relative to a head's (measured at d = 4096: 816 against 791 ns per 128 tokens; the
      // tails share their tokens through L2 with fewer tiles)
      const int64_t nsegs = ceil_div(total, p.seg_stages);
      const int64_t head_segs = (nsegs * 21 * k + (20 + 21 * k) / 2) / (20 + 21 * k);
      // worth it when the last round shrinks by at least 2 % of the whole call
      if (head_segs >= 1 && head_segs < nsegs && nsegs >= 8 &&
          50 * (nsegs - head_segs) >= rounds * nsegs) {
        p.full_tiles = (int)(tiles - r);
        p.cut_tiles = (int)r;
        p.cut_stage = (int)(head_segs * p.seg_stages);
        GPTQ_CUDA_CHECK(cudaMemsetAsync(H, 0, (size_t)(d * d) * sizeof(float), s));
      }
    }
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(2 * (tiles + p.cut_tiles)));
  cfg.blockDim = dim3(T_THREADS);
  cfg.dynamicSmemBytes = T_SMEM;
  cfg.stream = s;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = 2;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  const cudaError_t e = xdtype == GPTQ_F16
                            ? cudaLaunchKernelEx(&cfg, hessian_tc_kernel<0>, mx, mh, p, st)
                            : cudaLaunchKernelEx(&cfg, hessian_tc_kernel<1>, mx, mh, p, st);
  count_launch();
  if (e != cudaSuccess) {
    (void)cudaGetLastError();
    return GPTQ_ERR_CUDA;
  }
  return GPTQ_OK;
}

gptq_status launch_hessian_tf32(const void *X, int64_t n_tok, int64_t d, int64_t ldx, float *H,
                                int accumulate, DevStatus *st, cudaStream_t s) {
  GPTQ_TRY(ensure_smem_attr((const void *)hessian_tf32_kernel, (int)F_SMEM));
  CUtensorMap mx;
  if (!tc::make_tmap_2d(&mx, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, X, n_tok, d, ldx * 4, 32, F_K))
    return GPTQ_ERR_UNSUPPORTED;
  HessF32Params p{};
  p.d = d;
  p.n_tok = n_tok;
  p.seg_stages = kSegTokensTf32 / F_K;
  p.H = H;
  p.accumulate = accumulate;
  const int64_t nb = ceil_div(d, F_M);
  hessian_tf32_kernel<<<(unsigned)(nb * (nb + 1) / 2), F_THREADS, F_SMEM, s>>>(mx, p, st);
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
  if (xdtype == GPTQ_F32 && d >= 32 && n_tok >= 32) {
    const gptq_status t = launch_hessian_tf32(X, n_tok, d, ldx, H, accumulate, st, s);
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

gptq_status launch_hessian_lost_stage(const void *X, int xdtype, int64_t n_tok, int64_t d,
                                      int64_t ldx, float *H, int64_t lost_stage,
                                      uint64_t wait_ns, DevStatus *st, cudaStream_t s) {
  if (!((xdtype == GPTQ_F16 || xdtype == GPTQ_BF16) && d >= 64 && n_tok >= 64))
    return GPTQ_ERR_UNSUPPORTED;
  if (lost_stage < 0 || lost_stage >= ceil_div(n_tok, TB_K)) return GPTQ_ERR_INVALID_ARG;
  return launch_hessian_tc(X, xdtype, n_tok, d, ldx, H, 0, st, s, wait_ns, (int)lost_stage);
}

}  // namespace gptq
