// Steps 4 and 5 of the path: the GPTQ column sweep of one layer ("tm_gptq_math",
// "Greedy quantization with error compensation" and "GPTQ's speedups: fixed order and
// lazy batches"; "GPTQ Hessian", "GPTQ: Block Structure in Quantization").
//
// Per pair of blocks of B columns [b0, b1) and [b1, b2):
//   sweep    : every row (one thread each, the row's working weights in registers)
//              quantizes columns b0..b2-1 in order, spreading each column's scaled error
//              e_j = (w_j - q_j) / U_jj along row j of U inside the pair at once (the
//              first block's errors reach the second through U[b0:b1, b1:b2]);
//              writes the codes and E = [e_b0 .. e_b2-1] (as a TF32 head/tail pair)
//   trailing : W[:, b2:] -= E U[b0:b2, b2:]   (the deferred lazy-batch product, run as
//              C -= A B^T with B = U^T rows, i.e. Lt = U^T split into head/tail)
// then one pass packs the codes and writes W_hat.
#include <algorithm>
#include <cfloat>
#include <mutex>

#include "graph_cache.cuh"
#include "tc.cuh"

namespace gptq {

namespace {

constexpr int SB = 128;          // maximum block width held by one thread
constexpr int SW_ROWS = 64;      // rows per sweep CTA
constexpr int LDU = SB + 4;      // leading dimension of a packed U block
constexpr int LDW = 2 * SB + 4;  // smem leading dimension of the staging tile (a pair of
                                 // blocks; float4 rows of consecutive threads fall in
                                 // distinct bank groups)
// One packed diagonal block: U[b0:b0+nb, b0:b0+nb] upper part in SB x LDU (identity
// padding), then the SB reciprocal pivots 1 / U_jj.
constexpr int UD_FLOATS = SB * LDU + SB;
// One packed off-diagonal block of a pair: U[b0:b1, b1:b2] in SB x LDU (zero padding).
constexpr int UO_FLOATS = SB * LDU;

// ---------------------------------------------------------------------------------------
// Grid: per-row asymmetric min-max with 0 in the range; fp32 working copy of W with dead
// columns zeroed.  One warp per row; with `vec` (rows 16-byte aligned) W is read 16 bytes
// and the copy written 4 floats at a time.
// ---------------------------------------------------------------------------------------
template <typename T>
__global__ void grid_kernel(const T *__restrict__ W, int64_t m, int64_t d, int64_t ldw,
                            const uint8_t *__restrict__ dead, float maxq,
                            float *__restrict__ scale, int32_t *__restrict__ zero,
                            float *__restrict__ Wf, int64_t ldwf, int vec, DevStatus *st) {
  constexpr int VE = 16 / sizeof(T);   // elements per 16-byte load
  const int64_t row = (int64_t)blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  if (row >= m) return;
  const T *w = W + row * ldw;
  const int64_t dv = vec ? (d / VE) * VE : 0;   // the 16-byte part of the row
  float lo = 0.f, hi = 0.f;
  int bad = 0;
#pragma unroll 4
  for (int64_t j = (int64_t)lane * VE; j < dv; j += 32 * VE) {
    const uint4 u = *reinterpret_cast<const uint4 *>(w + j);
    const T *e = reinterpret_cast<const T *>(&u);
#pragma unroll
    for (int k = 0; k < VE; ++k) {
      const float v = to_f32(e[k]);
      bad |= !isfinite(v);
      lo = fminf(lo, v);
      hi = fmaxf(hi, v);
    }
  }
  for (int64_t j = dv + lane; j < d; j += 32) {
    const float v = to_f32(w[j]);
    bad |= !isfinite(v);
    lo = fminf(lo, v);
    hi = fmaxf(hi, v);
  }
  for (int o = 16; o; o >>= 1) {
    lo = fminf(lo, __shfl_xor_sync(0xffffffffu, lo, o));
    hi = fmaxf(hi, __shfl_xor_sync(0xffffffffu, hi, o));
    bad |= __shfl_xor_sync(0xffffffffu, bad, o);
  }
  const float width = __fsub_rn(hi, lo);
  const float s = (width == 0.0f) ? 1.0f : __fdiv_rn(width, maxq);
  const float z = rintf(__fdiv_rn(-lo, s));
  if (lane == 0) {
    scale[row] = s;
    zero[row] = (int32_t)z;
    if (bad) set_status(st, GPTQ_ERR_NONFINITE);
  }
  float *wf = Wf + row * ldwf;
#pragma unroll 2
  for (int64_t j = (int64_t)lane * VE; j < dv; j += 32 * VE) {
    const uint4 u = *reinterpret_cast<const uint4 *>(w + j);
    const T *e = reinterpret_cast<const T *>(&u);
    float v[VE];
#pragma unroll
    for (int k = 0; k < VE; ++k) v[k] = (dead && dead[j + k]) ? 0.0f : to_f32(e[k]);
#pragma unroll
    for (int k = 0; k < VE; k += 4)
      *reinterpret_cast<float4 *>(wf + j + k) = make_float4(v[k], v[k + 1], v[k + 2], v[k + 3]);
  }
  for (int64_t j = dv + lane; j < d; j += 32) wf[j] = (dead && dead[j]) ? 0.0f : to_f32(w[j]);
}

// ---------------------------------------------------------------------------------------
// Lt = U^T (lower part only: Lt[i][j] = U[j][i], j <= i) as a TF32 head/tail pair, in 64 x 64
// tiles through shared memory (U rows read, Lt rows written; float4 with VEC: d % 4 == 0
// and U 16-byte aligned).  Tiles wholly above the diagonal are never read and not written.
// ---------------------------------------------------------------------------------------
constexpr int LT_T = 64;

template <bool VEC>
__global__ void __launch_bounds__(256)
lt_split_kernel(const float *__restrict__ U, int64_t d, float *__restrict__ hi,
                float *__restrict__ lo, int64_t ld) {
  __shared__ float tile[LT_T][LT_T + 1];   // tile[cc][rr] = U[c0 + cc][r0 + rr]
  const int64_t r0 = (int64_t)blockIdx.y * LT_T, c0 = (int64_t)blockIdx.x * LT_T;
  if (r0 + LT_T - 1 < c0) return;
  const int tid = threadIdx.x, c4 = 4 * (tid % 16), t16 = tid / 16;
#pragma unroll
  for (int p = 0; p < LT_T / 16; ++p) {
    const int cc = t16 + 16 * p;
    const int64_t c = c0 + cc, r = r0 + c4;
    float v[4] = {0.f, 0.f, 0.f, 0.f};
    if (c < d) {
      if (VEC && r + 4 <= d) {
        const float4 u = *reinterpret_cast<const float4 *>(U + c * d + r);
        v[0] = u.x; v[1] = u.y; v[2] = u.z; v[3] = u.w;
      } else {
#pragma unroll
        for (int e = 0; e < 4; ++e)
          if (r + e < d) v[e] = U[c * d + r + e];
      }
    }
#pragma unroll
    for (int e = 0; e < 4; ++e) tile[cc][c4 + e] = (c <= r + e) ? v[e] : 0.f;
  }
  __syncthreads();
#pragma unroll
  for (int p = 0; p < LT_T / 16; ++p) {
    const int rr = t16 + 16 * p;
    const int64_t r = r0 + rr, c = c0 + c4;
    if (r >= d) continue;
    float h[4], l[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float v = tile[c4 + e][rr];
      h[e] = tf32_head(v);
      l[e] = v - h[e];
    }
    if (VEC && c + 4 <= d) {
      *reinterpret_cast<float4 *>(hi + r * ld + c) = make_float4(h[0], h[1], h[2], h[3]);
      *reinterpret_cast<float4 *>(lo + r * ld + c) = make_float4(l[0], l[1], l[2], l[3]);
    } else {
#pragma unroll
      for (int e = 0; e < 4; ++e)
        if (c + e < d) {
          hi[r * ld + c + e] = h[e];
          lo[r * ld + c + e] = l[e];
        }
    }
  }
}

// ---------------------------------------------------------------------------------------
// Packs the diagonal blocks of U for the sweep: upper triangle of U[b0:b0+nb, b0:b0+nb],
// identity padding to SB x SB (zero columns up to LDU), then 1 / U_jj.  CTA (x, y) writes
// rows [DB_ROWS y, DB_ROWS (y + 1)) of block x, 4 floats per store; y = 0 also the pivots.
// ---------------------------------------------------------------------------------------
constexpr int DB_ROWS = 16;

__global__ void __launch_bounds__(256)
diag_blocks_kernel(const float *__restrict__ U, int64_t d, int block, float *__restrict__ Ud) {
  const int64_t b0 = (int64_t)blockIdx.x * block;
  const int nb = (int)((d - b0) < block ? (d - b0) : block);
  float *out = Ud + (int64_t)blockIdx.x * UD_FLOATS;
  constexpr int Q = LDU / 4;   // float4 per packed row
  for (int t = threadIdx.x; t < DB_ROWS * Q; t += 256) {
    const int i = DB_ROWS * blockIdx.y + t / Q, j4 = 4 * (t % Q);
    float v[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int j = j4 + e;
      if (i < nb && j < nb) v[e] = i <= j ? U[(b0 + i) * d + (b0 + j)] : 0.f;
      else v[e] = (i == j && j < SB) ? 1.f : 0.f;
    }
    *reinterpret_cast<float4 *>(out + i * LDU + j4) = make_float4(v[0], v[1], v[2], v[3]);
  }
  if (blockIdx.y == 0)
    for (int j = threadIdx.x; j < SB; j += 256)
      out[SB * LDU + j] = (j < nb) ? 1.0f / U[(b0 + j) * d + (b0 + j)] : 1.0f;
}

// Packs the off-diagonal block of each pair of blocks (2p, 2p + 1) that has a second block:
// U[a0 + i][b0 + j] for i < block, j < nbB (a0 = 2p block, b0 = a0 + block), zero
// elsewhere in SB x LDU.  Same CTA layout as diag_blocks_kernel.
__global__ void __launch_bounds__(256)
offdiag_blocks_kernel(const float *__restrict__ U, int64_t d, int block, float *__restrict__ Uo) {
  const int64_t a0 = (int64_t)blockIdx.x * 2 * block, b0 = a0 + block;
  const int nbB = (int)((d - b0) < block ? (d - b0) : block);
  float *out = Uo + (int64_t)blockIdx.x * UO_FLOATS;
  constexpr int Q = LDU / 4;
  for (int t = threadIdx.x; t < DB_ROWS * Q; t += 256) {
    const int i = DB_ROWS * blockIdx.y + t / Q, j4 = 4 * (t % Q);
    float v[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int j = j4 + e;
      v[e] = (i < block && j < nbB) ? U[(a0 + i) * d + (b0 + j)] : 0.f;
    }
    *reinterpret_cast<float4 *>(out + i * LDU + j4) = make_float4(v[0], v[1], v[2], v[3]);
  }
}

// ---------------------------------------------------------------------------------------
// One column step of the in-block sweep within a 32-column sub-block, unrolled at compile
// time over the sub-block so its working weights stay in registers:
//   code = clamp(rint(w_J / s) + z, 0, maxq);  q = s (code - z);  e = (w_J - q) / U_JJ
//   w_k -= e U_Jk  for the later columns k of the sub-block.
// The same 32-step code serves all four sub-blocks of a block (runtime loop), which keeps
// the kernel inside the instruction cache.
// ---------------------------------------------------------------------------------------
constexpr int SUB = 32;

// k-th working weight of the sub-block, held as float2 pairs (k/2).(x|y)
#define W_AT(wp, k) (((k) & 1) ? (wp)[(k) >> 1].y : (wp)[(k) >> 1].x)

template <int J>
struct SweepStep {
  static __device__ __forceinline__ void run(float2 (&wp)[SUB / 2], uint32_t (&cw)[SUB / 4],
                                             const float *Ub, const float *rd, float s,
                                             float z, float maxq) {
    const float wj = W_AT(wp, J);
    const float x = __fdiv_rn(wj, s);
    const float c = fminf(fmaxf(rintf(x) + z, 0.0f), maxq);
    const float q = s * (c - z);
    const float e = (wj - q) * rd[J];
    cw[J / 4] |= (uint32_t)c << (8 * (J % 4));
    if (J & 1) wp[J >> 1].y = e; else wp[J >> 1].x = e;  // now the scaled error of column J
    // w_k -= e U_Jk for k > J in the sub-block: a lone odd column, then pairs
    constexpr int K0 = J + 1;
    if (K0 < SUB && (K0 & 1)) wp[K0 >> 1].y = fmaf(-e, Ub[J * LDU + K0], wp[K0 >> 1].y);
    const float2 ne = make_float2(-e, -e);
#pragma unroll
    for (int k = (K0 + 1) & ~1; k < SUB; k += 2)
      wp[k >> 1] = __ffma2_rn(ne, *reinterpret_cast<const float2 *>(Ub + J * LDU + k), wp[k >> 1]);
    SweepStep<J + 1>::run(wp, cw, Ub, rd, s, z, maxq);
  }
};
template <>
struct SweepStep<SUB> {
  static __device__ __forceinline__ void run(float2 (&)[SUB / 2], uint32_t (&)[SUB / 4],
                                             const float *, const float *, float, float,
                                             float) {}
};

// ---------------------------------------------------------------------------------------
// In-block sweep over a pair of blocks, A = columns [a0, a0 + nbA) and B = [a0 + block,
// a0 + block + nbB) (nbB = 0: A alone), for SW_ROWS rows per CTA:
//   chain  (warps 0-1, one thread per row): quantizes one 32-column sub-block at a time, A's
//          then B's, its working weights in registers, and leaves the sub-block's errors
//          and codes in the row.  Then, while the update threads already take those errors
//          on, it applies them to the next sub-block itself, as a register delta added when
//          it loads that sub-block: the next sub-block is ready as soon as the errors two
//          and more sub-blocks back have reached it.
//   update (warps 2, 3, 6, 7, 10, 11, 14, 15, four threads per row, all on the two
//          schedulers that the chain warps do not use): apply each sub-block's errors to
//          the sub-blocks two and more ahead, the nearest first (then signal it ready), and
//          store the sub-block's E and codes.  Errors of A reach B through the off-diagonal
//          block U[A, B], so B is swept in the same launch with no trailing product in
//          between.  Thread u of a row owns float4 columns u and u + 4 of every sub-block,
//          so each column receives its updates in one fixed order.
// The other six warps only help stage the tile.  Hand-offs are named barriers, each an arrive on
// one side and a sync on the other; every role alternates between two ids, so the chain,
// which may run a sub-block ahead, never arrives at an instance that is still open:
//   1 + S % 2: errors of sub-block S ready        3 + T % 2: sub-block T has the errors of
//                                                            all sub-blocks before T - 1
//   5: the chain's last read of the rows of A's block that B's first copy replaces
// A's diagonal block and the off-diagonal block arrive by bulk copies while the threads
// stage the tile.  B's diagonal block replaces A's in two bulk copies: its leading rows once
// only the chain's last sub-block of A still reads A's block, the rest once that is done.
// ---------------------------------------------------------------------------------------
constexpr int SW_THREADS = 8 * SW_ROWS;   // 16 warps: 2 chain, 8 update, 6 staging only
constexpr int SW_BAR = 5 * SW_ROWS;       // threads in each named barrier (chain + update)
constexpr int CW = 2 * SB / 4 + 1;        // staged code words per row

__device__ __forceinline__ void bar_arrive(int id, int n) {
  asm volatile("bar.arrive %0, %1;" ::"r"(id), "r"(n) : "memory");
}

// Two float4s of a row's working weights, wa and wb: w -= sum_{k < SUB} e_k U[k][.], the U
// rows at stride LDU from ua and ub (the float4s' columns); paired fp32 FMAs in k order.
__device__ __forceinline__ void update2(float *wa, float *wb, const float *ua, const float *ub,
                                        const float (&e)[SUB]) {
  const float4 a = *reinterpret_cast<const float4 *>(wa);
  const float4 b = *reinterpret_cast<const float4 *>(wb);
  float2 a0 = make_float2(a.x, a.y), a1 = make_float2(a.z, a.w);
  float2 b0 = make_float2(b.x, b.y), b1 = make_float2(b.z, b.w);
#pragma unroll
  for (int k = 0; k < SUB; ++k) {
    const float4 x = *reinterpret_cast<const float4 *>(ua + k * LDU);
    const float4 y = *reinterpret_cast<const float4 *>(ub + k * LDU);
    const float2 ne = make_float2(-e[k], -e[k]);
    a0 = __ffma2_rn(ne, make_float2(x.x, x.y), a0);
    a1 = __ffma2_rn(ne, make_float2(x.z, x.w), a1);
    b0 = __ffma2_rn(ne, make_float2(y.x, y.y), b0);
    b1 = __ffma2_rn(ne, make_float2(y.z, y.w), b1);
  }
  *reinterpret_cast<float4 *>(wa) = make_float4(a0.x, a0.y, a1.x, a1.y);
  *reinterpret_cast<float4 *>(wb) = make_float4(b0.x, b0.y, b1.x, b1.y);
}

__global__ void __launch_bounds__(SW_THREADS, 1)
sweep_pair_kernel(const float *__restrict__ Wf, int64_t ldwf, int64_t m, int64_t a0, int nbA,
                  int nbB, int block, const float *__restrict__ UdA,
                  const float *__restrict__ UdB, const float *__restrict__ Uo,
                  const float *__restrict__ scale, const int32_t *__restrict__ zero,
                  float maxq, float *__restrict__ Ehi, float *__restrict__ Elo, int64_t lde,
                  uint8_t *__restrict__ codes, int64_t ldc, DevStatus *st) {
  extern __shared__ __align__(16) float sm[];
  float *Us = sm;                        // SB x LDU: A's diagonal block, then B's
  float *rdA = sm + SB * LDU;            // A's SB reciprocal pivots
  float *Uos = sm + UD_FLOATS;           // SB x LDU: U[A, B]
  float *stage = Uos + UO_FLOATS;        // SW_ROWS x LDW: A from column 0, B from column SB
  uint32_t *cstage = (uint32_t *)(stage + SW_ROWS * LDW);  // SW_ROWS x CW words
  float *rdB = (float *)(cstage + SW_ROWS * CW);           // B's SB reciprocal pivots
  __shared__ __align__(8) uint64_t bar[3];   // A's blocks; B's leading rows; B's other rows
  const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
  const int64_t r0 = (int64_t)blockIdx.x * SW_ROWS;
  const int nsA = (nbA + SUB - 1) / SUB, nsB = (nbB + SUB - 1) / SUB, nS = nsA + nsB;
  const int R1 = (nsA - 1) * SUB;        // B's leading rows: those the first copy brings
  if (tid == 0) {
    for (int i = 0; i < 3; ++i) tc::mbar_init(&bar[i], 1);
    tc::mbar_fence_init();
    tc::mbar_arrive_expect_tx(&bar[0], (UD_FLOATS + (nsB ? UO_FLOATS : 0)) * 4);
    tc::bulk_load(Us, UdA, UD_FLOATS * 4, &bar[0]);
    if (nsB) tc::bulk_load(Uos, Uo, UO_FLOATS * 4, &bar[0]);
  }
  __syncthreads();
  // working weights, coalesced, zero beyond each block's width; float4 when the tile rows
  // and both blocks start on 16-byte boundaries
  if ((a0 % 4) == 0 && (ldwf % 4) == 0 && (block % 4) == 0) {
#pragma unroll 4
    for (int e = tid; e < SW_ROWS * (2 * SB / 4); e += SW_THREADS) {
      const int r = e / (2 * SB / 4), q = e % (2 * SB / 4);
      const int h = q / (SB / 4), c = 4 * (q % (SB / 4));   // block of the pair, column
      const int nb = h ? nbB : nbA;
      const int64_t gr = r0 + r;
      float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
      if (gr < m && c < nb) {
        v = *reinterpret_cast<const float4 *>(Wf + gr * ldwf + a0 + h * block + c);
        if (c + 1 >= nb) v.y = 0.f;
        if (c + 2 >= nb) v.z = 0.f;
        if (c + 3 >= nb) v.w = 0.f;
      }
      *reinterpret_cast<float4 *>(stage + r * LDW + h * SB + c) = v;
    }
  } else {
#pragma unroll 4
    for (int e = tid; e < SW_ROWS * 2 * SB; e += SW_THREADS) {
      const int r = e / (2 * SB), q = e % (2 * SB);
      const int h = q / SB, j = q % SB;
      const int64_t gr = r0 + r;
      stage[r * LDW + q] =
          (gr < m && j < (h ? nbB : nbA)) ? Wf[gr * ldwf + a0 + h * block + j] : 0.f;
    }
  }
  const int got = tc::mbar_wait(&bar[0], 0, st) ? 1 : 0;
  if (!__syncthreads_and(got)) return;  // CTA-uniform: later barriers stay matched
  int ok = 1;                           // every wait for B's diagonal block succeeded
  if (warp < 2) {
    // ---------------- chain ----------------
    float *my = stage + tid * LDW;      // this row of the pair
    const int64_t row = r0 + tid;
    const float s = row < m ? scale[row] : 1.f;
    const float z = row < m ? (float)zero[row] : 0.f;
    float2 wp[SUB / 2], dn[SUB / 2];
#pragma unroll
    for (int i = 0; i < SUB / 2; ++i) wp[i] = *reinterpret_cast<const float2 *>(my + 2 * i);
#pragma unroll 1
    for (int S = 0; S < nS; ++S) {
      const int h = S >= nsA, sb = h ? S - nsA : S, c0 = sb * SUB;
      float *w = my + h * SB + c0;
      if (S > 0) {
        if (S >= 2) tc::named_barrier(3 + S % 2, SW_BAR);   // errors up to S - 2 applied
        if (h && sb == 0 && nsA >= 2) ok &= tc::mbar_wait(&bar[1], 0, st) ? 1 : 0;
        if (h && (sb == nsA - 1 || sb == nsB - 1)) ok &= tc::mbar_wait(&bar[2], 0, st) ? 1 : 0;
        // the stage's sub-block plus the delta of the errors of sub-block S - 1
#pragma unroll
        for (int i = 0; i < SUB / 2; ++i) {
          const float2 v = *reinterpret_cast<const float2 *>(w + 2 * i);
          wp[i] = make_float2(v.x + dn[i].x, v.y + dn[i].y);
        }
      }
      uint32_t cw[SUB / 4];
#pragma unroll
      for (int i = 0; i < SUB / 4; ++i) cw[i] = 0u;
      SweepStep<0>::run(wp, cw, Us + c0 * LDU + c0, (h ? rdB : rdA) + c0, s, z, maxq);
#pragma unroll
      for (int i = 0; i < SUB / 2; ++i) *reinterpret_cast<float2 *>(w + 2 * i) = wp[i];
#pragma unroll
      for (int i = 0; i < SUB / 4; ++i) cstage[tid * CW + h * (SB / 4) + c0 / 4 + i] = cw[i];
      bar_arrive(1 + S % 2, SW_BAR);                 // errors of sub-block S ready
      if (S + 1 < nS) {
        // the next sub-block's delta: dn_k = -sum_J e_J U[J][k], J in order
        const int hn = (S + 1) >= nsA, cn = (hn ? S + 1 - nsA : S + 1) * SUB;
        const float *Un = (hn == h ? Us : Uos) + c0 * LDU + cn;
#pragma unroll
        for (int i = 0; i < SUB / 2; ++i) dn[i] = make_float2(0.f, 0.f);
#pragma unroll 4
        for (int J = 0; J < SUB; ++J) {
          const float e = w[J];                       // the error just stored
          const float2 ne = make_float2(-e, -e);
#pragma unroll
          for (int k = 0; k < SUB; k += 4) {
            const float4 x = *reinterpret_cast<const float4 *>(Un + J * LDU + k);
            dn[k >> 1] = __ffma2_rn(ne, make_float2(x.x, x.y), dn[k >> 1]);
            dn[(k >> 1) + 1] = __ffma2_rn(ne, make_float2(x.z, x.w), dn[(k >> 1) + 1]);
          }
        }
        // that delta read the last rows of A's block that B's first copy replaces
        if (nsB && S == nsA - 2) bar_arrive(5, SW_ROWS + 32);
      }
    }
  } else if ((warp & 3) >= 2) {
    // ---------------- update ----------------
    const int v = 2 * (warp >> 2) + (warp & 1);      // 0 .. 7
    const int rl = 32 * (v & 1) + lane, u = v >> 1, ut = 32 * v + lane;
    float *my = stage + rl * LDW;
    const bool evec = ((uintptr_t)Ehi % 16) == 0 && ((uintptr_t)Elo % 16) == 0 &&
                      (lde % 4) == 0 && (block % 4) == 0;
    const bool cvec = (a0 % 4) == 0 && (ldc % 4) == 0 && (block % 4) == 0;
    bool waited = false;
#pragma unroll 1
    for (int S = 0; S < nS; ++S) {
      tc::named_barrier(1 + S % 2, SW_BAR);          // errors of sub-block S ready
      const int h = S >= nsA, sb = h ? S - nsA : S, c0 = sb * SUB, nb = h ? nbB : nbA;
      if (nsB && S == nsA - 2 && warp == 2) tc::named_barrier(5, SW_ROWS + 32);  // chain's delta
      if (nsB && ut == 0 && (S == nsA - 2 || S == nsA - 1)) {
        // every read of these rows of A's diagonal block is done: B's replace them
        tc::fence_proxy_async_smem();
        if (S == nsA - 2) {
          tc::mbar_arrive_expect_tx(&bar[1], (R1 * LDU + SB) * 4);
          tc::bulk_load(Us, UdB, R1 * LDU * 4, &bar[1]);
          tc::bulk_load(rdB, UdB + SB * LDU, SB * 4, &bar[1]);
        } else {
          tc::mbar_arrive_expect_tx(&bar[2], ((SB - R1) * LDU + (nsA == 1 ? SB : 0)) * 4);
          tc::bulk_load(Us + R1 * LDU, UdB + R1 * LDU, (SB - R1) * LDU * 4, &bar[2]);
          if (nsA == 1) tc::bulk_load(rdB, UdB + SB * LDU, SB * 4, &bar[2]);
        }
      }
      if (S + 2 < nS) {
        if (h && !waited) {                          // B's leading rows of its block
          ok &= tc::mbar_wait(&bar[1], 0, st) ? 1 : 0;
          waited = true;
        }
        float e[SUB];
#pragma unroll
        for (int q = 0; q < SUB / 4; ++q) {
          const float4 x = *reinterpret_cast<const float4 *>(my + h * SB + c0 + 4 * q);
          e[4 * q] = x.x; e[4 * q + 1] = x.y; e[4 * q + 2] = x.z; e[4 * q + 3] = x.w;
        }
#pragma unroll 1
        for (int T = S + 2; T < nS; ++T) {
          const int ht = T >= nsA, t0 = (ht ? T - nsA : T) * SUB;
          const float *Ub = (ht == h ? Us : Uos) + c0 * LDU + t0;
          float *wt = my + ht * SB + t0;
          update2(wt + 4 * u, wt + 4 * (u + 4), Ub + 4 * u, Ub + 4 * (u + 4), e);
          if (T == S + 2) bar_arrive(3 + S % 2, SW_BAR);   // sub-block S + 2 ready
        }
      }
      // sub-block S's E (a TF32 head/tail pair, at column h * block + c0 of the pair
      // buffer) and codes, coalesced: float4 / whole words when aligned
      if (evec) {
#pragma unroll
        for (int i = 0; i < SW_ROWS * (SUB / 4) / 256; ++i) {
          const int qi = ut + 256 * i, r = qi / (SUB / 4), c = c0 + 4 * (qi % (SUB / 4));
          const int64_t gr = r0 + r;
          if (gr < m && c < nb) {
            float4 x = *reinterpret_cast<const float4 *>(stage + r * LDW + h * SB + c);
            if (c + 1 >= nb) x.y = 0.f;
            if (c + 2 >= nb) x.z = 0.f;
            if (c + 3 >= nb) x.w = 0.f;
            const float4 hd = make_float4(tf32_head(x.x), tf32_head(x.y), tf32_head(x.z), tf32_head(x.w));
            *reinterpret_cast<float4 *>(Ehi + gr * lde + h * block + c) = hd;
            *reinterpret_cast<float4 *>(Elo + gr * lde + h * block + c) =
                make_float4(x.x - hd.x, x.y - hd.y, x.z - hd.z, x.w - hd.w);
          }
        }
      } else {
        for (int i = ut; i < SW_ROWS * SUB; i += 256) {
          const int r = i / SUB, c = c0 + i % SUB;
          const int64_t gr = r0 + r;
          if (gr < m && c < nb) {
            const float x = stage[r * LDW + h * SB + c], hd = tf32_head(x);
            Ehi[gr * lde + h * block + c] = hd;
            Elo[gr * lde + h * block + c] = x - hd;
          }
        }
      }
      if (cvec) {
#pragma unroll
        for (int i = 0; i < SW_ROWS * (SUB / 4) / 256; ++i) {
          const int wi = ut + 256 * i, r = wi / (SUB / 4), wq = wi % (SUB / 4), c = c0 + 4 * wq;
          const int64_t gr = r0 + r;
          if (gr < m && c < nb) {
            uint32_t x = cstage[r * CW + h * (SB / 4) + c / 4];
            if (c + 4 > nb) x &= (1u << (8 * (nb - c))) - 1u;   // ragged block end
            *reinterpret_cast<uint32_t *>(codes + gr * ldc + a0 + h * block + c) = x;
          }
        }
      } else {
        const uint8_t *cb = (const uint8_t *)cstage;
        for (int i = ut; i < SW_ROWS * SUB; i += 256) {
          const int r = i / SUB, c = c0 + i % SUB;
          const int64_t gr = r0 + r;
          if (gr < m && c < nb) codes[gr * ldc + a0 + h * block + c] = cb[r * CW * 4 + h * SB + c];
        }
      }
    }
  }
  if (!__syncthreads_and(ok) && tid == 0 && nsB) {
    // a wait ran out (TIMEOUT recorded): give the copies in flight one more bounded wait
    if (nsA >= 2) tc::mbar_wait(&bar[1], 0, nullptr);
    tc::mbar_wait(&bar[2], 0, nullptr);
  }
}

// ---------------------------------------------------------------------------------------
// Eager sweep (B = 1, "tm_gptq_math", "GPTQ's speedups: fixed order and lazy batches": the
// column-at-a-time form whose per-column update of every later column the pages call
// memory-bandwidth-bound).  One launch per column j: each CTA takes ER rows x EC later
// columns; every thread quantizes its row's column j itself (the threads of a row reach
// the same code) and applies w_k -= e U_jk to its four columns, so the later columns
// stream through memory once per column.  Same arithmetic as the blocked sweep.
// ---------------------------------------------------------------------------------------
constexpr int EC = 256, ER = 32, E_THREADS = 256;  // 64 column threads (float4) x 4 rows

__global__ void __launch_bounds__(E_THREADS)
eager_column_kernel(float *__restrict__ Wf, int64_t ldwf, int64_t m, int64_t d, int64_t j,
                    const float *__restrict__ U, const float *__restrict__ scale,
                    const int32_t *__restrict__ zero, float maxq, uint8_t *__restrict__ codes,
                    int64_t ldc) {
  const int tx = threadIdx.x % 64, ty = threadIdx.x / 64;
  const int64_t c = (((j + 1) >> 2) << 2) + (int64_t)blockIdx.x * EC + 4 * tx;
  const float rd = 1.0f / U[j * d + j];
  float u[4];
  if ((d % 4) == 0 && c + 4 <= d) {
    const float4 v = *reinterpret_cast<const float4 *>(U + j * d + c);
    u[0] = v.x; u[1] = v.y; u[2] = v.z; u[3] = v.w;
  } else {
#pragma unroll
    for (int q = 0; q < 4; ++q) u[q] = (c + q < d) ? U[j * d + c + q] : 0.0f;
  }
#pragma unroll 2
  for (int rr = ty; rr < ER; rr += E_THREADS / 64) {
    const int64_t r = (int64_t)blockIdx.y * ER + rr;
    if (r >= m) break;
    float *wr = Wf + r * ldwf;
    const float wj = wr[j];
    const float s = scale[r], z = (float)zero[r];
    const float cd = fminf(fmaxf(rintf(__fdiv_rn(wj, s)) + z, 0.0f), maxq);
    const float e = (wj - s * (cd - z)) * rd;
    if (blockIdx.x == 0 && tx == 0) codes[r * ldc + j] = (uint8_t)cd;
    if (c > j && c + 4 <= d) {
      float4 w = *reinterpret_cast<float4 *>(wr + c);
      w.x = fmaf(-e, u[0], w.x);
      w.y = fmaf(-e, u[1], w.y);
      w.z = fmaf(-e, u[2], w.z);
      w.w = fmaf(-e, u[3], w.w);
      *reinterpret_cast<float4 *>(wr + c) = w;
    } else {
#pragma unroll
      for (int q = 0; q < 4; ++q)   // the float4 holding column j (never written) or the end
        if (c + q > j && c + q < d) wr[c + q] = fmaf(-e, u[q], wr[c + q]);
    }
  }
}

// ---------------------------------------------------------------------------------------
// OBQ greedy order ("tm_gptq_math", "Greedy quantization with error compensation"; the
// Schur downdate of "GPTQ › Mathematical Details of the Update"), for d_in <= OBQ_MAX_D:
// one CTA per row, thread j owns column j; the row's inverse Hessian of the free weights
// lives in shared memory.  Per step: every free column's cost (w - quant(w))^2 / [H_F^-1]_jj
// in fp32, an argmin over the CTA (lowest index on ties), then the chosen thread stores its
// code and scaled error, the free threads compensate their weights and downdate their own
// column of H_F^-1.  Only uniform barriers; no waits on other CTAs.
// ---------------------------------------------------------------------------------------
constexpr int OBQ_MAX_D = 128;

// Hinv = U^T U (U upper): Hinv[i][j] = sum_{k <= min(i, j)} U[k][i] U[k][j].
__global__ void hinv_kernel(const float *__restrict__ U, int64_t d, float *__restrict__ Hinv) {
  for (int64_t e = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; e < d * d;
       e += (int64_t)gridDim.x * blockDim.x) {
    const int64_t i = e / d, j = e % d, kmax = i < j ? i : j;
    float acc = 0.f;
    for (int64_t k = 0; k <= kmax; ++k) acc = fmaf(U[k * d + i], U[k * d + j], acc);
    Hinv[e] = acc;
  }
}

__global__ void __launch_bounds__(OBQ_MAX_D)
obq_kernel(const float *__restrict__ Wf, int64_t ldwf, int d, const float *__restrict__ Hinv,
           const float *__restrict__ scale, const int32_t *__restrict__ zero, float maxq,
           uint8_t *__restrict__ codes, int64_t ldc, int32_t *__restrict__ order) {
  // R = the transpose of H_F^-1 as downdated column by column: thread j owns row j of R, so
  // its update is a float4 sweep along its own row against row q (a broadcast).  R starts
  // as H^-1 itself (bitwise symmetric), and each step computes exactly the transpose of the
  // column-wise downdate H_ij -= H_iq (H_qj / H_qq):  R_ji -= R_qi (R_jq / R_qq).
  extern __shared__ __align__(16) float Rs[];  // d x LH
  __shared__ float s_val[OBQ_MAX_D / 32];
  __shared__ int s_idx[OBQ_MAX_D / 32];
  __shared__ float s_e;
  const int j = threadIdx.x, lane = j % 32, wid = j / 32;
  const int64_t row = blockIdx.x;
  const int LH = ((d + 3) / 4) * 4 + 4;
  for (int e = j; e < d * LH; e += OBQ_MAX_D) {
    const int i = e / LH, c = e % LH;
    Rs[e] = c < d ? Hinv[i * d + c] : 0.f;
  }
  bool free = j < d;
  uint32_t fm[OBQ_MAX_D / 32];   // free columns, the same in every thread
#pragma unroll
  for (int k = 0; k < OBQ_MAX_D / 32; ++k) {
    const int lo = 32 * k;
    fm[k] = d >= lo + 32 ? 0xffffffffu : (d > lo ? (1u << (d - lo)) - 1u : 0u);
  }
  float w = free ? Wf[row * ldwf + j] : 0.f;
  const float sc_row = scale[row], z = (float)zero[row];
  __syncthreads();
#pragma unroll 1
  for (int step = 0; step < d; ++step) {
    float cd = 0.f, qv = 0.f, key = INFINITY;   // non-free columns never win
    if (free) {
      cd = fminf(fmaxf(rintf(__fdiv_rn(w, sc_row)) + z, 0.f), maxq);
      qv = sc_row * (cd - z);
      const float er = w - qv;
      const float cost = __fdiv_rn(er * er, Rs[j * LH + j]);
      key = (cost >= 0.f && cost <= FLT_MAX) ? cost : FLT_MAX;  // NaN/inf: last among free
    }
    int idx = free ? j : OBQ_MAX_D;
#pragma unroll
    for (int o = 16; o; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, key, o);
      const int oi = __shfl_xor_sync(0xffffffffu, idx, o);
      if (ov < key || (ov == key && oi < idx)) { key = ov; idx = oi; }
    }
    if (lane == 0) { s_val[wid] = key; s_idx[wid] = idx; }
    __syncthreads();
    float best = s_val[0];
    int q = s_idx[0];
#pragma unroll
    for (int k = 1; k < OBQ_MAX_D / 32; ++k)
      if (s_val[k] < best || (s_val[k] == best && s_idx[k] < q)) { best = s_val[k]; q = s_idx[k]; }
    // a free column always exists while step < d, so q < d; the clamp only keeps every
    // index inside the tile should that ever fail
    q = q < d ? q : d - 1;
    fm[q / 32] &= ~(1u << (q % 32));
    if (j == q) {
      codes[row * ldc + q] = (uint8_t)cd;
      if (order) order[row * d + step] = q;
      s_e = __fdiv_rn(w - qv, Rs[q * LH + q]);
      w = qv;
      free = false;
    }
    __syncthreads();
    if (free) {
      w = fmaf(-s_e, Rs[q * LH + j], w);                 // H_jq = R_qj
      const float f = __fdiv_rn(Rs[j * LH + q], Rs[q * LH + q]);   // H_qj / H_qq
      // row q is not written in this step (its thread has left the free set): each batch of
      // sixteen columns is read before any of it is written
      float *rj = Rs + j * LH;
      const float *rq = Rs + q * LH;
#pragma unroll 1
      for (int i0 = 0; i0 < d; i0 += 16) {
        float4 hq[4], hj[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          if (i0 + 4 * u < d) {
            hq[u] = *reinterpret_cast<const float4 *>(rq + i0 + 4 * u);
            hj[u] = *reinterpret_cast<const float4 *>(rj + i0 + 4 * u);
          }
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int i = i0 + 4 * u;
          if (i < d) {
            const uint32_t bits = (fm[i / 32] >> (i % 32)) & 0xfu;   // i % 4 == 0: one word
            float4 v = hj[u];
            if (bits & 1u) v.x = fmaf(-hq[u].x, f, v.x);
            if (bits & 2u) v.y = fmaf(-hq[u].y, f, v.y);
            if (bits & 4u) v.z = fmaf(-hq[u].z, f, v.z);
            if (bits & 8u) v.w = fmaf(-hq[u].w, f, v.w);
            *reinterpret_cast<float4 *>(rj + i) = v;
          }
        }
      }
    }
    __syncthreads();
  }
}

// ---------------------------------------------------------------------------------------
// Pack codes into the row bitstream: the 32 codes of group g fill exactly words
// [BITS g, BITS (g + 1)) of the row, so one thread packs one group (two 16-byte loads for a
// whole group: the code rows are 16-byte aligned).  Rows are strided over CTAs.
// ---------------------------------------------------------------------------------------
template <int BITS>
__global__ void __launch_bounds__(128)
pack_kernel(const uint8_t *__restrict__ codes, int64_t ldc, int64_t m, int64_t d,
            int64_t words, uint32_t *__restrict__ qp) {
  const int64_t ng = (d + 31) / 32;
  for (int64_t row = blockIdx.x; row < m; row += gridDim.x) {
    const uint8_t *cr = codes + row * ldc;
    uint32_t *out = qp + row * words;
    for (int64_t g = threadIdx.x; g < ng; g += blockDim.x) {
      uint8_t c[32];
      if (32 * g + 32 <= d) {
        const uint4 u0 = *reinterpret_cast<const uint4 *>(cr + 32 * g);
        const uint4 u1 = *reinterpret_cast<const uint4 *>(cr + 32 * g + 16);
        memcpy(c, &u0, 16);
        memcpy(c + 16, &u1, 16);
      } else {
#pragma unroll
        for (int k = 0; k < 32; ++k) c[k] = 32 * g + k < d ? cr[32 * g + k] : 0;
      }
      uint64_t acc = 0;
      int nacc = 0, wo = 0;
#pragma unroll
      for (int k = 0; k < 32; ++k) {
        acc |= (uint64_t)c[k] << nacc;
        nacc += BITS;
        if (nacc >= 32) {
          out[BITS * g + wo++] = (uint32_t)acc;
          acc >>= 32;
          nacc -= 32;
        }
      }
    }
  }
}

// W_hat = scale * (code - zero), rows strided over CTAs, 4 columns per thread (float4 stores
// with VEC: d % 4 == 0 and W_hat 16-byte aligned).
template <bool VEC>
__global__ void __launch_bounds__(256)
dequant_kernel(const uint8_t *__restrict__ codes, int64_t ldc, int64_t m, int64_t d,
               const float *__restrict__ scale, const int32_t *__restrict__ zero,
               float *__restrict__ Wh) {
  for (int64_t row = blockIdx.x; row < m; row += gridDim.x) {
    const float s = scale[row], z = (float)zero[row];
    const uint8_t *cr = codes + row * ldc;
    float *wr = Wh + row * d;
    for (int64_t c = 4 * (int64_t)threadIdx.x; c < d; c += 4 * blockDim.x) {
      const uchar4 u = *reinterpret_cast<const uchar4 *>(cr + c);   // ldc % 16 == 0
      const float v[4] = {s * ((float)u.x - z), s * ((float)u.y - z), s * ((float)u.z - z),
                          s * ((float)u.w - z)};
      if (VEC) {
        *reinterpret_cast<float4 *>(wr + c) = make_float4(v[0], v[1], v[2], v[3]);
      } else {
#pragma unroll
        for (int e = 0; e < 4; ++e)
          if (c + e < d) wr[c + e] = v[e];
      }
    }
  }
}

// The sweep's views of U: Lt = U^T as head/tail (the trailing updates) and the packed
// diagonal blocks (the sweep).
gptq_status launch_lt_split(const float *U, int64_t d, float *hi, float *lo, int64_t ld,
                            cudaStream_t s) {
  dim3 tg((unsigned)ceil_div(d, LT_T), (unsigned)ceil_div(d, LT_T));
  if ((d % 4) == 0) lt_split_kernel<true><<<tg, 256, 0, s>>>(U, d, hi, lo, ld);   // U: 16 B
  else lt_split_kernel<false><<<tg, 256, 0, s>>>(U, d, hi, lo, ld);
  GPTQ_LAUNCH_CHECK();
  return GPTQ_OK;
}

gptq_status launch_diag_blocks(const float *U, int64_t d, int block, float *Ud, float *Uo,
                               cudaStream_t s) {
  const int64_t nblk = ceil_div(d, block);
  diag_blocks_kernel<<<dim3((unsigned)nblk, SB / DB_ROWS), 256, 0, s>>>(U, d, block, Ud);
  GPTQ_LAUNCH_CHECK();
  if (nblk >= 2) {
    offdiag_blocks_kernel<<<dim3((unsigned)(nblk / 2), SB / DB_ROWS), 256, 0, s>>>(U, d, block, Uo);
    GPTQ_LAUNCH_CHECK();
  }
  return GPTQ_OK;
}

gptq_status launch_pack(const uint8_t *codes, int64_t ldc, int64_t m, int64_t d, int bits,
                        int64_t words, uint32_t *qp, cudaStream_t s) {
  const unsigned g = (unsigned)std::min<int64_t>(std::max<int64_t>(m, 1), 8192);
  switch (bits) {
    case 2: pack_kernel<2><<<g, 128, 0, s>>>(codes, ldc, m, d, words, qp); break;
    case 3: pack_kernel<3><<<g, 128, 0, s>>>(codes, ldc, m, d, words, qp); break;
    case 4: pack_kernel<4><<<g, 128, 0, s>>>(codes, ldc, m, d, words, qp); break;
    case 8: pack_kernel<8><<<g, 128, 0, s>>>(codes, ldc, m, d, words, qp); break;
    default: return GPTQ_ERR_INVALID_ARG;
  }
  GPTQ_LAUNCH_CHECK();
  return GPTQ_OK;
}

gptq_status launch_dequant(const uint8_t *codes, int64_t ldc, int64_t m, int64_t d,
                           const float *scale, const int32_t *zero, float *Wh, cudaStream_t s) {
  const unsigned g = (unsigned)std::min<int64_t>(std::max<int64_t>(m, 1), 8192);
  if ((d % 4) == 0 && ((uintptr_t)Wh % 16) == 0)
    dequant_kernel<true><<<g, 256, 0, s>>>(codes, ldc, m, d, scale, zero, Wh);
  else
    dequant_kernel<false><<<g, 256, 0, s>>>(codes, ldc, m, d, scale, zero, Wh);
  GPTQ_LAUNCH_CHECK();
  return GPTQ_OK;
}

struct QuantWs {
  DevStatus *st;
  float *Wf; int64_t ldwf;
  float *Ehi, *Elo;
  float *Lhi, *Llo; int64_t ldl;
  uint8_t *codes; int64_t ldc;
  float *Ud, *Uo;       // packed diagonal blocks; off-diagonal block of each pair
  float *Ehi2, *Elo2;   // second E buffer
  int64_t lde;          // E row stride: a pair of blocks side by side, or a group of two pairs
};

// On wide layers the far part of the blocked sweep's trailing update is most of its work; it
// is then applied once per group of two pairs of blocks, as one product of depth up to 4B
// (measured faster per flop than two of depth 2B), and each E buffer holds a group.
constexpr int64_t kGroupedMinD = 8192;
inline bool sweep_grouped(int64_t d, int block) { return block > 1 && d >= kGroupedMinD; }
inline int64_t sweep_lde(int64_t d, int block) {
  return block > 1 ? (sweep_grouped(d, block) ? 4 : 2) * SB : SB;
}

QuantWs carve_quantize(void *ws, int64_t m, int64_t d, int block) {
  QuantWs q;
  char *p = (char *)ws;
  q.st = (DevStatus *)p; p += 256;
  q.ldwf = (int64_t)round_up((size_t)d, 4);
  q.Wf = (float *)p; p += round_up((size_t)m * q.ldwf * 4, 256);
  q.lde = sweep_lde(d, block);
  q.Ehi = (float *)p; p += round_up((size_t)m * q.lde * 4, 256);
  q.Elo = (float *)p; p += round_up((size_t)m * q.lde * 4, 256);
  q.ldl = (int64_t)round_up((size_t)d, 4);
  q.Lhi = (float *)p; p += round_up((size_t)d * q.ldl * 4, 256);
  q.Llo = (float *)p; p += round_up((size_t)d * q.ldl * 4, 256);
  q.ldc = (int64_t)round_up((size_t)d, 16);
  q.codes = (uint8_t *)p; p += round_up((size_t)m * q.ldc, 256);
  q.Ud = (float *)p;
  const size_t nblk = (size_t)ceil_div(d, block < 1 ? 1 : block);
  p += block > 1 ? nblk * UD_FLOATS * 4 : 0;
  q.Uo = (float *)p;
  p += block > 1 ? (nblk / 2) * UO_FLOATS * 4 : 0;
  q.Ehi2 = (float *)p; p += round_up((size_t)m * q.lde * 4, 256);
  q.Elo2 = (float *)p;
  return q;
}

}  // namespace

size_t quantize_ws_bytes(int64_t m, int64_t d, int bits, int block) {
  (void)bits;
  const size_t ldwf = round_up((size_t)d, 4), ldl = round_up((size_t)d, 4);
  const size_t ldc = round_up((size_t)d, 16);
  const size_t nblk = (size_t)ceil_div(d, block < 1 ? 1 : block);
  const size_t lde = (size_t)sweep_lde(d, block);
  return 256 + round_up((size_t)m * ldwf * 4, 256) + 2 * round_up((size_t)m * lde * 4, 256) +
         2 * round_up((size_t)d * ldl * 4, 256) + round_up((size_t)m * ldc, 256) +
         (block > 1 ? nblk * UD_FLOATS * 4 + (nblk / 2) * UO_FLOATS * 4 +
                          2 * round_up((size_t)m * lde * 4, 256)
                    : 0);   // B = 1 needs neither packed U blocks nor a second E pair
}

namespace {

// The blocked sweep's two streams per device, created once and kept for the process:
// `crit` (highest priority) runs the sweeps and each block's update of the next block's
// columns; `side` (lowest priority) runs the far part of each block's trailing update.
struct QuantStreams {
  std::mutex enqueue;  // one call at a time enqueues on these events
  cudaStream_t crit = nullptr, side = nullptr;
  cudaEvent_t start = nullptr, crit_done = nullptr, side_done = nullptr;
  cudaEvent_t e_ready[2] = {nullptr, nullptr};   // E of a block written (by parity)
  cudaEvent_t far_done[2] = {nullptr, nullptr};  // that block's far update finished
  cudaEvent_t g_in = nullptr, g_out = nullptr;   // joins of a graph replay
  cudaEvent_t fork = nullptr, ud_done = nullptr, lt_done = nullptr;  // U views beside the grid
  GraphCache graphs;                             // the sweep captured per argument set
};
constexpr int kMaxDevices = 128;
std::mutex g_qs_mu;
QuantStreams g_qs[kMaxDevices];

gptq_status quant_streams(QuantStreams **out) {
  int dev = -1;
  GPTQ_CUDA_CHECK(cudaGetDevice(&dev));
  if (dev < 0 || dev >= kMaxDevices) return GPTQ_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_qs_mu);
  QuantStreams &q = g_qs[dev];
  if (!q.crit) {
    int lo = 0, hi = 0;
    GPTQ_CUDA_CHECK(cudaDeviceGetStreamPriorityRange(&lo, &hi));
    GPTQ_CUDA_CHECK(cudaStreamCreateWithPriority(&q.crit, cudaStreamNonBlocking, hi));
    GPTQ_CUDA_CHECK(cudaStreamCreateWithPriority(&q.side, cudaStreamNonBlocking, lo));
    cudaEvent_t *evs[] = {&q.start, &q.crit_done, &q.side_done, &q.e_ready[0], &q.e_ready[1],
                          &q.far_done[0], &q.far_done[1], &q.g_in, &q.g_out, &q.fork,
                          &q.ud_done, &q.lt_done};
    for (cudaEvent_t *e : evs) GPTQ_CUDA_CHECK(cudaEventCreateWithFlags(e, cudaEventDisableTiming));
  }
  *out = &q;
  return GPTQ_OK;
}

gptq_status launch_grid(const void *W, int wdtype, int64_t m, int64_t d, int64_t ldw,
                        const uint8_t *dead_mask, float maxq, float *scale, int32_t *zero,
                        float *Wf, int64_t ldwf, DevStatus *st, cudaStream_t s) {
  const int warps = 8;
  const unsigned g = (unsigned)ceil_div(m, warps);
  const int es = wdtype == GPTQ_F32 ? 4 : 2;
  const int vec = ((uintptr_t)W % 16) == 0 && (ldw * es) % 16 == 0;
  switch (wdtype) {
    case GPTQ_F32:
      grid_kernel<float><<<g, warps * 32, 0, s>>>((const float *)W, m, d, ldw, dead_mask, maxq,
                                                  scale, zero, Wf, ldwf, vec, st);
      break;
    case GPTQ_F16:
      grid_kernel<__half><<<g, warps * 32, 0, s>>>((const __half *)W, m, d, ldw, dead_mask,
                                                   maxq, scale, zero, Wf, ldwf, vec, st);
      break;
    case GPTQ_BF16:
      grid_kernel<__nv_bfloat16><<<g, warps * 32, 0, s>>>((const __nv_bfloat16 *)W, m, d, ldw,
                                                          dead_mask, maxq, scale, zero, Wf, ldwf,
                                                          vec, st);
      break;
    default:
      return GPTQ_ERR_INVALID_ARG;
  }
  GPTQ_LAUNCH_CHECK();
  return GPTQ_OK;
}

}  // namespace

size_t quantize_layers_ws_bytes(const int64_t *m, int n, int64_t d, int bits, int block) {
  int64_t mt = 0;
  for (int i = 0; i < n; ++i) mt += m[i];
  const size_t base = quantize_ws_bytes(mt, d, bits, block);
  return n == 1 ? base : base + 2 * round_up((size_t)mt * 4, 256);
}

// Layers that share U are swept as one matrix of their stacked rows (rows decouple:
// "GPTQ Hessian"): one grid pass per layer into the shared fp32 working copy, one sweep and
// one trailing update per block over all rows, then each layer's rows packed into its own
// outputs.  With one layer the per-row scale and zero are written in place.
namespace {

constexpr size_t kSweepSmem = (UD_FLOATS + UO_FLOATS + SW_ROWS * LDW + SW_ROWS * CW + SB) * sizeof(float);

// The sweep's launches (no set-up, no locking): on `s`, and with `qs` the blocked sweep's
// far updates on qs->side and the rest on qs->crit (which is `s` itself when the whole
// routine is captured on it).
gptq_status enqueue_quantize_layers(const QLayer *L, int n, int64_t d, const float *U,
                                    const uint8_t *dead_mask, int bits, int block, void *ws,
                                    cudaStream_t s, QuantStreams *qs) {
  const size_t sweep_smem = kSweepSmem;
  int64_t m = 0;
  for (int i = 0; i < n; ++i) m += L[i].m;
  QuantWs q = carve_quantize(ws, m, d, block);
  float *scale = L[0].scale;
  int32_t *zero = L[0].zero;
  if (n > 1) {
    char *p = (char *)ws + quantize_ws_bytes(m, d, bits, block);
    scale = (float *)p;
    zero = (int32_t *)(p + round_up((size_t)m * 4, 256));
  }
  const float maxq = (float)((1 << bits) - 1);
  GPTQ_CUDA_CHECK(cudaMemsetAsync(q.st, 0, sizeof(DevStatus), s));
  // blocked with the side stream: the U views (which need only U) beside the grid pass
  const bool overlap = qs != nullptr && block > 1;
  if (overlap) {
    GPTQ_CUDA_CHECK(cudaEventRecord(qs->fork, s));
    GPTQ_CUDA_CHECK(cudaStreamWaitEvent(qs->side, qs->fork, 0));
    GPTQ_TRY(launch_diag_blocks(U, d, block, q.Ud, q.Uo, qs->side));
    GPTQ_CUDA_CHECK(cudaEventRecord(qs->ud_done, qs->side));
    GPTQ_TRY(launch_lt_split(U, d, q.Lhi, q.Llo, q.ldl, qs->side));
    GPTQ_CUDA_CHECK(cudaEventRecord(qs->lt_done, qs->side));
  }
  for (int64_t i = 0, off = 0; i < n; off += L[i].m, ++i)
    GPTQ_TRY(launch_grid(L[i].W, L[i].wdtype, L[i].m, d, L[i].ldw, dead_mask, maxq,
                         scale + off, zero + off, q.Wf + off * q.ldwf, q.ldwf, q.st, s));
  if (block == 1) {
    // eager: one launch per column, U read in place
    for (int64_t j = 0; j < d; ++j) {
      const int64_t first = ((j + 1) >> 2) << 2;
      dim3 eg((unsigned)(ceil_div(d - first, EC) > 0 ? ceil_div(d - first, EC) : 1),
              (unsigned)ceil_div(m, ER));
      eager_column_kernel<<<eg, E_THREADS, 0, s>>>(q.Wf, q.ldwf, m, d, j, U, scale, zero, maxq,
                                                   q.codes, q.ldc);
      GPTQ_LAUNCH_CHECK();
    }
  } else {
    // blocked: the pairs of blocks, each swept in one launch, then one trailing update of
    // depth up to 2B per pair
    if (!overlap) {
      GPTQ_TRY(launch_lt_split(U, d, q.Lhi, q.Llo, q.ldl, s));
      GPTQ_TRY(launch_diag_blocks(U, d, block, q.Ud, q.Uo, s));
    }
    const unsigned sweep_grid = (unsigned)ceil_div(m, SW_ROWS);
    // The E of both blocks of pair p sit side by side in buffer p % 2 (block 2p + h at
    // column h * block), so one product of depth up to 2B applies the pair to the columns
    // past it: the next two blocks' columns in 128-wide tiles, the rest in 256-wide ones.
    // Every column thus receives the contributions of earlier pairs in the same order,
    // grouping and kernel in both schedules below (the results are bit for bit the same).
    // On wide layers (grouped) pair p writes its E into buffer (p / 2) % 2 at column
    // (p % 2) 2B, so that a group's two pairs sit side by side; otherwise into buffer p % 2.
    const bool grouped = sweep_grouped(d, block);
    auto e_col = [&](int64_t p) -> int64_t { return grouped ? (p & 1) * 2 * block : 0; };
    auto e_buf = [&](int64_t p) -> int { return (int)((grouped ? p >> 1 : p) & 1); };
    // W[:, c0:c1] -= E U[kb0:kb0+K, c0:c1] with E the K columns of buffer e from column ec
    auto update = [&](int e, int64_t ec, int64_t kb0, int K, int64_t c0, int64_t c1,
                      int max_ctas, cudaStream_t st, int wide) -> gptq_status {
      GemmArgs g{};
      g.a_hi = (e ? q.Ehi2 : q.Ehi) + ec; g.a_lo = (e ? q.Elo2 : q.Elo) + ec; g.lda = q.lde;
      g.b_hi = q.Lhi + c0 * q.ldl + kb0; g.b_lo = q.Llo + c0 * q.ldl + kb0; g.ldb = q.ldl;
      g.c = q.Wf + c0; g.ldc = q.ldwf;
      g.M = m; g.N = c1 - c0; g.K = K;
      g.alpha = -1.0f; g.lower_only = 0; g.trans_c = 0; g.max_ctas = max_ctas;
      g.one_sum = 1;   // one TMEM sum per tile: the codes need no shorter sums
      g.wide = wide;
      return launch_gemm_nt(g, q.st, st);
    };
    // pair p: blocks 2p ([a0, a0 + nbA)) and 2p + 1 ([a0 + block, + nbB), nbB = 0 if none)
    auto sweep = [&](int64_t p, int nbA, int nbB, cudaStream_t st) -> gptq_status {
      const int64_t a0 = 2 * p * block;
      const int e = e_buf(p);
      const int64_t ec = e_col(p);
      return launch_kernel(sweep_pair_kernel, sweep_grid, SW_THREADS, sweep_smem, st,
                           (const float *)q.Wf, q.ldwf, m, a0, nbA, nbB, block,
                           (const float *)(q.Ud + 2 * p * UD_FLOATS),
                           (const float *)(q.Ud + (nbB ? 2 * p + 1 : 2 * p) * UD_FLOATS),
                           (const float *)(q.Uo + (nbB ? p : 0) * UO_FLOATS),
                           (const float *)scale, (const int32_t *)zero, maxq,
                           (e ? q.Ehi2 : q.Ehi) + ec, (e ? q.Elo2 : q.Elo) + ec, q.lde, q.codes,
                           q.ldc, q.st);
    };
    auto widths = [&](int64_t p, int &nbA, int &nbB) {
      const int64_t a0 = 2 * p * block, b0 = a0 + block;
      nbA = (int)std::min<int64_t>(block, d - a0);
      nbB = b0 < d ? (int)std::min<int64_t>(block, d - b0) : 0;
    };
    const int64_t npairs = ceil_div(d, 2 * (int64_t)block);
    // The trailing update after pair p (group g = p / 2 when grouped), its columns split by
    // where they are needed next:
    //   near: [pe, ne), ne = the end of group g + 1 (grouped) or of the layer, depth = the
    //         pair: the next pair's columns first (the sweep after waits for them), then the
    //         rest of the near columns in 256-wide tiles;
    //   far:  grouped, after a group's last pair, [ne, d) once for the whole group, depth up
    //         to 4B, in 256-wide tiles.
    // Every column thus receives the contributions of earlier pairs and groups in one order,
    // grouping and kernel in both schedules below (the results are bit for bit the same).
    struct Split {
      int64_t a0, pe, f0, ne;   // pair start and end; next pair's end; near end
      bool far;                 // a group's far product follows this pair
      int64_t g0;               // the group's first column
    };
    auto split = [&](int64_t p, int nbA, int nbB) {
      Split t;
      t.a0 = 2 * p * block;
      t.pe = t.a0 + (nbB ? block + nbB : nbA);
      t.f0 = std::min<int64_t>(t.pe + 2 * block, d);
      t.g0 = grouped ? (p & ~int64_t(1)) * 2 * block : t.a0;
      t.ne = grouped ? std::min<int64_t>(t.g0 + 8 * block, d) : d;
      t.far = grouped && ((p & 1) || p + 1 == npairs) && t.ne < d;
      return t;
    };
    if (!overlap) {
      for (int64_t p = 0; p < npairs; ++p) {
        int nbA, nbB;
        widths(p, nbA, nbB);
        const Split t = split(p, nbA, nbB);
        GPTQ_TRY(sweep(p, nbA, nbB, s));
        if (t.pe >= d) break;
        // the same column split and kernels as the two-stream schedule below
        const int e = e_buf(p), K = (int)(t.pe - t.a0);
        GPTQ_TRY(update(e, e_col(p), t.a0, K, t.pe, std::min(t.f0, t.ne), 0, s, 0));
        if (t.f0 < t.ne) GPTQ_TRY(update(e, e_col(p), t.a0, K, t.f0, t.ne, 0, s, 1));
        if (t.far) GPTQ_TRY(update(e, 0, t.g0, (int)(t.pe - t.g0), t.ne, d, 0, s, 1));
      }
    } else {
      // After pair p: the next pair's columns on the critical stream right after the sweep,
      // the rest of its near columns and a group's far product on the side stream, where
      // they have at least a pair sweep and a near update's time before the sweep that needs
      // them.  Pair p's update on the critical stream waits for the side stream's work of
      // pair p - 1, which keeps each column's contributions in the single-stream order and
      // frees the E buffer that the next pair or group reuses.
      cudaStream_t c = qs->crit, sd = qs->side;
      int nsm = 0;
      GPTQ_TRY(device_sm_count(&nsm));
      // the far update (persistent): up to d_in = 4096 it leaves one SM per sweep CTA, which
      // measured better than sharing SMs two sweep CTAs each and than one CTA per tile over
      // all SMs; on wide layers the far products are most of the work and take every SM
      // (measured at d_in = 28672: 35.9 against 56.9 ms; 11008: 3.83 against 3.95 ms)
      const int far_ctas = d >= 8192 ? 0
                                     : std::max(1, nsm - (int)std::min<unsigned>(sweep_grid, nsm / 2));
      GPTQ_CUDA_CHECK(cudaEventRecord(qs->start, s));
      GPTQ_CUDA_CHECK(cudaStreamWaitEvent(c, qs->start, 0));
      GPTQ_CUDA_CHECK(cudaStreamWaitEvent(sd, qs->start, 0));
      GPTQ_CUDA_CHECK(cudaStreamWaitEvent(c, qs->ud_done, 0));   // the first sweep
      bool lt_waited = false;                                     // the first update on c
      for (int64_t p = 0; p < npairs; ++p) {
        int nbA, nbB;
        widths(p, nbA, nbB);
        const Split t = split(p, nbA, nbB);
        const int pb = (int)(p & 1);                              // event parity
        GPTQ_TRY(sweep(p, nbA, nbB, c));
        if (t.pe >= d) break;
        if (!lt_waited) GPTQ_CUDA_CHECK(cudaStreamWaitEvent(c, qs->lt_done, 0));
        lt_waited = true;
        const int e = e_buf(p), K = (int)(t.pe - t.a0);
        GPTQ_CUDA_CHECK(cudaEventRecord(qs->e_ready[pb], c));
        if (p > 0) GPTQ_CUDA_CHECK(cudaStreamWaitEvent(c, qs->far_done[pb ^ 1], 0));
        GPTQ_TRY(update(e, e_col(p), t.a0, K, t.pe, std::min(t.f0, t.ne), 0, c, 0));
        GPTQ_CUDA_CHECK(cudaStreamWaitEvent(sd, qs->e_ready[pb], 0));
        if (t.f0 < t.ne) GPTQ_TRY(update(e, e_col(p), t.a0, K, t.f0, t.ne, far_ctas, sd, 1));
        if (t.far) GPTQ_TRY(update(e, 0, t.g0, (int)(t.pe - t.g0), t.ne, d, far_ctas, sd, 1));
        GPTQ_CUDA_CHECK(cudaEventRecord(qs->far_done[pb], sd));
      }
      GPTQ_CUDA_CHECK(cudaEventRecord(qs->crit_done, c));
      GPTQ_CUDA_CHECK(cudaEventRecord(qs->side_done, sd));
      GPTQ_CUDA_CHECK(cudaStreamWaitEvent(s, qs->crit_done, 0));
      GPTQ_CUDA_CHECK(cudaStreamWaitEvent(s, qs->side_done, 0));
    }
  }
  const int64_t words = ceil_div(d, 32) * bits;
  for (int64_t i = 0, off = 0; i < n; off += L[i].m, ++i) {
    const uint8_t *codes = q.codes + off * q.ldc;
    GPTQ_TRY(launch_pack(codes, q.ldc, L[i].m, d, bits, words, L[i].qpacked, s));
    if (L[i].W_hat)
      GPTQ_TRY(launch_dequant(codes, q.ldc, L[i].m, d, scale + off, zero + off, L[i].W_hat, s));
    if (n > 1) {
      GPTQ_CUDA_CHECK(cudaMemcpyAsync(L[i].scale, scale + off, L[i].m * 4,
                                      cudaMemcpyDeviceToDevice, s));
      GPTQ_CUDA_CHECK(cudaMemcpyAsync(L[i].zero, zero + off, L[i].m * 4,
                                      cudaMemcpyDeviceToDevice, s));
    }
  }
  return GPTQ_OK;
}

}  // namespace

gptq_status launch_quantize_layers(const QLayer *L, int n, int64_t d, const float *U,
                                   const uint8_t *dead_mask, int bits, int block, void *ws,
                                   cudaStream_t s, bool allow_overlap) {
  GPTQ_TRY(ensure_smem_attr((const void *)sweep_pair_kernel, (int)kSweepSmem));
  if (!allow_overlap || block == 1 || d <= 2 * (int64_t)block)
    return enqueue_quantize_layers(L, n, d, U, dead_mask, bits, block, ws, s, nullptr);
  QuantStreams *qs = nullptr;
  GPTQ_TRY(quant_streams(&qs));
  std::lock_guard<std::mutex> lock(qs->enqueue);
  if (caller_capturing(s))
    return enqueue_quantize_layers(L, n, d, U, dead_mask, bits, block, ws, s, qs);
  // Graph replay (graph_cache.cuh), captured on the critical stream
  GPTQ_CUDA_CHECK(cudaEventRecord(qs->g_in, s));
  GPTQ_CUDA_CHECK(cudaStreamWaitEvent(qs->crit, qs->g_in, 0));
  std::vector<uint64_t> key = {(uint64_t)n, (uint64_t)d, (uint64_t)U, (uint64_t)dead_mask,
                               (uint64_t)bits, (uint64_t)block, (uint64_t)ws};
  for (int i = 0; i < n; ++i) {
    const uint64_t f[] = {(uint64_t)L[i].W, (uint64_t)L[i].wdtype, (uint64_t)L[i].m,
                          (uint64_t)L[i].ldw, (uint64_t)L[i].qpacked, (uint64_t)L[i].scale,
                          (uint64_t)L[i].zero, (uint64_t)L[i].W_hat};
    key.insert(key.end(), f, f + 8);
  }
  gptq_status st = GPTQ_OK;
  if (!qs->graphs.run(key, qs->crit, [&](cudaStream_t o) {
        return enqueue_quantize_layers(L, n, d, U, dead_mask, bits, block, ws, o, qs);
      }, &st))
    return enqueue_quantize_layers(L, n, d, U, dead_mask, bits, block, ws, s, qs);
  GPTQ_CUDA_CHECK(cudaEventRecord(qs->g_out, qs->crit));
  GPTQ_CUDA_CHECK(cudaStreamWaitEvent(s, qs->g_out, 0));
  return GPTQ_OK;
}

size_t quantize_obq_ws_bytes(int64_t m, int64_t d) {
  return 256 + round_up((size_t)m * round_up((size_t)d, 4) * 4, 256) +
         round_up((size_t)m * round_up((size_t)d, 16), 256) + round_up((size_t)d * d * 4, 256);
}

gptq_status launch_quantize_obq(const void *W, int wdtype, int64_t m, int64_t d, int64_t ldw,
                                const float *U, const uint8_t *dead_mask, int bits,
                                uint32_t *qpacked, float *scale, int32_t *zero, float *W_hat,
                                int32_t *order, void *ws, cudaStream_t s) {
  GPTQ_TRY(ensure_smem_attr((const void *)obq_kernel,
                            (int)(OBQ_MAX_D * (OBQ_MAX_D + 4) * sizeof(float))));
  char *p = (char *)ws;
  DevStatus *st = (DevStatus *)p; p += 256;
  const int64_t ldwf = (int64_t)round_up((size_t)d, 4), ldc = (int64_t)round_up((size_t)d, 16);
  float *Wf = (float *)p; p += round_up((size_t)m * ldwf * 4, 256);
  uint8_t *codes = (uint8_t *)p; p += round_up((size_t)m * ldc, 256);
  float *Hinv = (float *)p;
  const float maxq = (float)((1 << bits) - 1);
  GPTQ_CUDA_CHECK(cudaMemsetAsync(st, 0, sizeof(DevStatus), s));
  GPTQ_TRY(launch_grid(W, wdtype, m, d, ldw, dead_mask, maxq, scale, zero, Wf, ldwf, st, s));
  hinv_kernel<<<(unsigned)ceil_div(d * d, 256), 256, 0, s>>>(U, d, Hinv);
  GPTQ_LAUNCH_CHECK();
  obq_kernel<<<(unsigned)m, OBQ_MAX_D, (size_t)d * (((d + 3) / 4) * 4 + 4) * sizeof(float), s>>>(
      Wf, ldwf, (int)d, Hinv, scale, zero, maxq, codes, ldc, order);
  GPTQ_LAUNCH_CHECK();
  const int64_t words = ceil_div(d, 32) * bits;
  GPTQ_TRY(launch_pack(codes, ldc, m, d, bits, words, qpacked, s));
  if (W_hat) GPTQ_TRY(launch_dequant(codes, ldc, m, d, scale, zero, W_hat, s));
  return GPTQ_OK;
}

gptq_status launch_quantize(const void *W, int wdtype, int64_t m, int64_t d, int64_t ldw,
                            const float *U, const uint8_t *dead_mask, int bits, int block,
                            uint32_t *qpacked, float *scale, int32_t *zero, float *W_hat,
                            void *ws, cudaStream_t s, bool allow_overlap) {
  const QLayer one{W, wdtype, m, ldw, qpacked, scale, zero, W_hat};
  return launch_quantize_layers(&one, 1, d, U, dead_mask, bits, block, ws, s, allow_overlap);
}


}  // namespace gptq
