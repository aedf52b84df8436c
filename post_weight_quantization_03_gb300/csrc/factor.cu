// Steps 2 and 3 of the path: dead columns, damping, and the upper Cholesky factor U of
// the inverse damped Hessian ("tm_gptq_math", "The Cholesky trick for the inverse
// Hessian"; "GPTQ Hessian": H^-1 = U^T U).
//
// Route (same U, half the work of inverting then factoring): with P the index reversal,
// A = P H P = L L^T (lower Cholesky), Y = L^-1, and U = P Y P is upper with
// U^T U = P (L L^T)^-1 P = H^-1; the Cholesky factor with positive diagonal is unique.
//
// Blocked right-looking algorithm over panels of NB columns of A, interleaving the
// forward substitution Y = L^-1 (kept transposed: Yt = Y^T, upper):
//   potrf  : factor the diagonal block A_kk = L_kk L_kk^T and invert it (one CTA)
//   trsm   : L_ik = A_ik Linv_kk^T for the rows below              (row-panel product)
//   inv-a  : Yt[c, k] = Bt[c, k] Linv_kk^T for columns c < (k+1)NB (row-panel product)
//   syrk   : A_ij -= L_ik L_jk^T on the lower trailing tiles           (rank-NB update)
//   inv-b  : Bt[c, r] -= Yt[c, k] L_rk^T for c < (k+1)NB <= r          (rank-NB update)
// where Bt is the transposed right-hand side of L Y = I, updated in place into Yt.
// Finally U[i][j] = Yt[d-1-j][d-1-i] for i <= j.
#include <algorithm>
#include <cstring>
#include <mutex>

#include "graph_cache.cuh"

namespace gptq {

namespace {

constexpr int NB = 128;            // panel width
constexpr int kGroup = 4;          // panels per group (the deferred updates' K = 512)
constexpr int64_t GW = kGroup * NB;

// ---------------------------------------------------------------------------------------
// Dead columns and damping (one CTA): dead = {i : H_ii == 0}; H_ii <- 1 for dead i;
// lambda = damp * mean(diag); H_ii += lambda.  The damped diagonal is written reversed
// (A_ii = damped H_{d-1-i, d-1-i}): thread t swaps the pair (t, d-1-t), so no entry is
// read after another thread wrote it.
// ---------------------------------------------------------------------------------------
__global__ void dead_damp_kernel(float *H, int64_t d, float damp, uint8_t *dead_mask,
                                 DevStatus *st) {
  __shared__ double red[32];
  __shared__ int s_ndead, s_bad;
  if (threadIdx.x == 0) { s_ndead = 0; s_bad = 0; }
  __syncthreads();
  double sum = 0.0;
  int ndead = 0, bad = 0;
  // the diagonal entries lie in distinct lines: four loads in flight per thread and round trip
#pragma unroll 4
  for (int64_t i = threadIdx.x; i < d; i += blockDim.x) {
    const float h = H[i * d + i];
    if (!isfinite(h)) bad = 1;
    const bool dead = (h == 0.0f);
    ndead += dead;
    sum += dead ? 1.0 : (double)h;
  }
  for (int o = 16; o; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
  const int w = threadIdx.x / 32, l = threadIdx.x % 32;
  if (l == 0) red[w] = sum;
  if (ndead) atomicAdd(&s_ndead, ndead);
  if (bad) atomicOr(&s_bad, 1);
  __syncthreads();
  if (threadIdx.x < 32) {
    const int nw = blockDim.x / 32;
    double t = threadIdx.x < nw ? red[threadIdx.x] : 0.0;
    for (int o = 16; o; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
    if (threadIdx.x == 0) red[0] = t;
  }
  __syncthreads();
  const double diag_sum = red[0];
  const float lam = (float)((double)damp * (diag_sum / (double)d));
  if (threadIdx.x == 0) {
    st->n_dead = s_ndead;
    st->lam = (double)lam;
    st->diag_sum = diag_sum;
    if (s_bad) set_status(st, GPTQ_ERR_NONFINITE);
  }
  // pairs (i, d-1-i), two per thread and round trip (all four loads before the stores)
  const int64_t half = (d + 1) / 2;
  for (int64_t i0 = threadIdx.x; i0 < half; i0 += 2 * (int64_t)blockDim.x) {
    const int64_t i1 = i0 + blockDim.x;
    const bool two = i1 < half;
    const int64_t j0 = d - 1 - i0, j1 = d - 1 - i1;
    const float h0 = H[i0 * d + i0], g0 = H[j0 * d + j0];
    const float h1 = two ? H[i1 * d + i1] : 0.0f, g1 = two ? H[j1 * d + j1] : 0.0f;
    if (dead_mask) {
      dead_mask[i0] = h0 == 0.0f;
      dead_mask[j0] = g0 == 0.0f;
      if (two) {
        dead_mask[i1] = h1 == 0.0f;
        dead_mask[j1] = g1 == 0.0f;
      }
    }
    H[i0 * d + i0] = (g0 == 0.0f ? 1.0f : g0) + lam;
    H[j0 * d + j0] = (h0 == 0.0f ? 1.0f : h0) + lam;
    if (two) {
      H[i1 * d + i1] = (g1 == 0.0f ? 1.0f : g1) + lam;
      H[j1 * d + j1] = (h1 == 0.0f ? 1.0f : h1) + lam;
    }
  }
}

// ---------------------------------------------------------------------------------------
// A = P H P below the diagonal (P the order reversal): A_ij = H_{d-1-i, d-1-j} for i > j,
// read from H's strict upper triangle, which no thread writes (only the upper triangle of
// the symmetric H is read, with a finiteness check).  The same pass sets Yt to the
// identity on every block row's diagonal block and the blocks right of it: the only part of
// Yt that the panel loop reads.  One CTA per row i; VEC moves float4s (d % 4 == 0, H and
// Yt 16-byte aligned), each thread issuing its loads before its stores.
// ---------------------------------------------------------------------------------------
constexpr int RV_THREADS = 256, RV_UNROLL = 4;

template <bool VEC>
__global__ void __launch_bounds__(RV_THREADS)
reverse_lower_kernel(float *H, int64_t d, float *Yt, DevStatus *st) {
  const int64_t i = blockIdx.x, r = d - 1 - i;
  const float *src = H + r * d;   // source row: A_ij = src[d - 1 - j]
  float *dst = H + i * d;
  const int tid = threadIdx.x;
  int bad = 0;
  if (VEC) {
    // float4 q covers j = 4q .. 4q+3 < i, i.e. q < i / 4: source columns d-4-4q .. d-1-4q
    const int64_t nq = i / 4;
    for (int64_t q0 = tid; q0 < nq; q0 += (int64_t)RV_THREADS * RV_UNROLL) {
      float4 v[RV_UNROLL];
#pragma unroll
      for (int u = 0; u < RV_UNROLL; ++u) {
        const int64_t q = q0 + (int64_t)u * RV_THREADS;
        if (q < nq) v[u] = *reinterpret_cast<const float4 *>(src + d - 4 - 4 * q);
      }
#pragma unroll
      for (int u = 0; u < RV_UNROLL; ++u) {
        const int64_t q = q0 + (int64_t)u * RV_THREADS;
        if (q < nq) {
          bad |= !isfinite(v[u].x) | !isfinite(v[u].y) | !isfinite(v[u].z) | !isfinite(v[u].w);
          *reinterpret_cast<float4 *>(dst + 4 * q) = make_float4(v[u].w, v[u].z, v[u].y, v[u].x);
        }
      }
    }
    const int64_t j = 4 * nq + tid;   // the last i % 4 entries left of the diagonal
    if (j < i) {
      const float v = src[d - 1 - j];
      bad |= !isfinite(v);
      dst[j] = v;
    }
    // Yt row i from column (i / NB) * NB: identity
    const int64_t c0 = (i / NB) * NB;
    for (int64_t c = c0 + 4 * tid; c < d; c += 4 * RV_THREADS)
      *reinterpret_cast<float4 *>(Yt + i * d + c) =
          make_float4(c == i ? 1.f : 0.f, c + 1 == i ? 1.f : 0.f, c + 2 == i ? 1.f : 0.f,
                      c + 3 == i ? 1.f : 0.f);
  } else {
    for (int64_t j = tid; j < i; j += RV_THREADS) {
      const float v = src[d - 1 - j];
      bad |= !isfinite(v);
      dst[j] = v;
    }
    for (int64_t c = (i / NB) * NB + tid; c < d; c += RV_THREADS) Yt[i * d + c] = c == i ? 1.f : 0.f;
  }
  if (__syncthreads_or(bad) && tid == 0) set_status(st, GPTQ_ERR_NONFINITE);
}

// ---------------------------------------------------------------------------------------
// potrf: Cholesky factor L of the n x n diagonal block at (k0, k0) of A (n <= NB) and its
// inverse Linv.  Only Linv leaves the kernel (NB x NB, lower, zero padded): the panel below
// is L_ik = A_ik Linv^T and the inversion needs Linv only.
//
// Recursive over eight PW-column sub-panels p (P0 = PW p, R0 = P0 + PW), in shared memory,
// with the inverse built alongside in transposed form (Bt = right-hand side of L Y = I,
// transposed, which becomes Yt = Linv^T), exactly like the panel loop of the whole
// factorization:
//   leaf   : one warp factors the PW x PW tile (lane i holds row i; four columns per
//            step, each lane factoring the step's 4 x 4 diagonal block itself) and writes the
//            scaled transpose M[j][i] = L_ij / L_jj and the reciprocal pivots rd
//   phase 1: L_ip  L_pp^T = A_ip                  rows i >= R0      (trsm)
//            Yt_cp L_pp^T = Bt_cp                  rows c <  R0      (inverse, step a)
//            one thread per row, forward substitution against M
//   phase 2: A_il -= L_ip L_lp^T                  R0 <= l <= i      (syrk)
//            Bt_cr -= Yt_cp L_rp^T                c < R0 <= r       (inverse, step b)
// Phase 2 is a product over PW k in tiles of 8 rows x 64 columns per warp (A read by
// broadcast, B as float4 along k at row stride 132: eight consecutive rows fall in distinct
// bank groups).  The leaf runs one sub-panel ahead: after phase 1 of sub-panel p, warp 0
// applies phase 2 to the next leaf's tile alone and factors it, while the other fifteen
// warps run the rest of phase 2 and write the next identity rows of Bt (untouched until
// then), so one barrier per sub-panel orders both; the warps that share warp 0's scheduler
// (4, 8, 12) stay out of phase 2 so that the leaf's serial chain is not slowed.  The rows
// of Linv that phase 1 finishes are stored before the split.  A non-positive pivot records
// NOT_PD with its global index.
// ---------------------------------------------------------------------------------------
constexpr int PF_THREADS = 512;
constexpr int PF_WARPS = PF_THREADS / 32;
constexpr int PW = 16;             // sub-panel width
constexpr int PL = NB + 4;         // smem leading dimension (16-byte rows)
// Shared memory the kernel uses, and what it requests: enough that no other kernel's CTA
// (the row-panel products of the concurrent streams need 34 KB or more) fits on its SM, so
// that no foreign warps compete with the leaf's serial chain for issue slots.
constexpr size_t kPotrfSmemUsed = (2 * NB * PL + PW * PL + PW) * sizeof(float);
constexpr size_t kPotrfSmem = 200 * 1024;
static_assert(kPotrfSmemUsed <= kPotrfSmem, "potrf shared memory");

// Columns JB .. JB + 3 of the leaf at once.  Lane i holds row i of the tile in a[] (its
// diagonal entry included, updated like the others).  Every lane takes the block's 4 x 4
// lower part from lanes JB .. JB + 3 by shuffles and factors it itself (the same values in
// every lane), then solves its own row against it, L[i][JB + c] = x_c, and subtracts the
// rank-4 product of the block's columns from its later entries, with the rows' x exchanged
// through shared memory (two buffers by block parity).  Per entry the operations and their
// order are those of eliminating the four columns one after another.  What lands above the
// diagonal is never read and is cleared at the end.
template <int JB>
struct LeafBlock {
  static __device__ __forceinline__ void run(float (&a)[PW], float &rdl, float &pvl, float4 *xb,
                                             float *M, int lane) {
    constexpr unsigned F = 0xffffffffu;
    const float b00 = __shfl_sync(F, a[JB], JB);
    const float b10 = __shfl_sync(F, a[JB], JB + 1), b11 = __shfl_sync(F, a[JB + 1], JB + 1);
    const float b20 = __shfl_sync(F, a[JB], JB + 2), b21 = __shfl_sync(F, a[JB + 1], JB + 2);
    const float b22 = __shfl_sync(F, a[JB + 2], JB + 2);
    const float b30 = __shfl_sync(F, a[JB], JB + 3), b31 = __shfl_sync(F, a[JB + 1], JB + 3);
    const float b32 = __shfl_sync(F, a[JB + 2], JB + 3), b33 = __shfl_sync(F, a[JB + 3], JB + 3);
    // the block's factor, with no test on the chain: a non-positive pivot gives an infinite
    // or NaN r (the factor is then discarded; the pivot itself is recorded below)
    const float r0 = rsqrtf(b00);
    const float l10 = b10 * r0, l20 = b20 * r0, l30 = b30 * r0;
    const float t11 = fmaf(-l10, l10, b11);
    const float r1 = rsqrtf(t11);
    const float l21 = fmaf(-l20, l10, b21) * r1, l31 = fmaf(-l30, l10, b31) * r1;
    const float t22 = fmaf(-l21, l21, fmaf(-l20, l20, b22));
    const float r2 = rsqrtf(t22);
    const float l32 = fmaf(-l31, l21, fmaf(-l30, l20, b32)) * r2;
    const float t33 = fmaf(-l32, l32, fmaf(-l31, l31, fmaf(-l30, l30, b33)));
    const float r3 = rsqrtf(t33);
    // this lane's row in the block's columns, without branches (a divergent chain of cases
    // costs hundreds of cycles per block): the general solve gives, in the block's own rows
    // rr = 0..3, exactly the block factor's operations (x_j = l_rr,j for j < rr and
    // x_rr = t_rr,rr r_rr), and entries right of the diagonal (j > rr) are set to zero
    const int rr = lane - JB;
    float x0 = a[JB] * r0;
    float x1 = fmaf(-x0, l10, a[JB + 1]) * r1;
    float x2 = fmaf(-x1, l21, fmaf(-x0, l20, a[JB + 2])) * r2;
    float x3 = fmaf(-x2, l32, fmaf(-x1, l31, fmaf(-x0, l30, a[JB + 3]))) * r3;
    x0 = rr >= 0 ? x0 : 0.0f;
    x1 = rr >= 1 ? x1 : 0.0f;
    x2 = rr >= 2 ? x2 : 0.0f;
    x3 = rr >= 3 ? x3 : 0.0f;
    rdl = rr == 0 ? r0 : rr == 1 ? r1 : rr == 2 ? r2 : rr == 3 ? r3 : rdl;
    pvl = rr == 0 ? b00 : rr == 1 ? t11 : rr == 2 ? t22 : rr == 3 ? t33 : pvl;
    M[(JB + 0) * PL + lane] = x0 * r0;   // L[i][j] / L[j][j]
    M[(JB + 1) * PL + lane] = x1 * r1;
    M[(JB + 2) * PL + lane] = x2 * r2;
    M[(JB + 3) * PL + lane] = x3 * r3;
    a[JB] = x0; a[JB + 1] = x1; a[JB + 2] = x2; a[JB + 3] = x3;
    if (JB + 4 < PW) {
      float4 *xs = xb + ((JB / 4) & 1) * 32;
      xs[lane] = make_float4(x0, x1, x2, x3);
      __syncwarp();
#pragma unroll
      for (int k = JB + 4; k < PW; ++k) {
        const float4 v = xs[k];          // L[k][JB .. JB + 3]
        a[k] = fmaf(-x0, v.x, a[k]);
        a[k] = fmaf(-x1, v.y, a[k]);
        a[k] = fmaf(-x2, v.z, a[k]);
        a[k] = fmaf(-x3, v.w, a[k]);
      }
    }
    LeafBlock<JB + 4>::run(a, rdl, pvl, xb, M, lane);
  }
};
template <>
struct LeafBlock<PW> {
  static __device__ __forceinline__ void run(float (&)[PW], float &, float &, float4 *, float *,
                                             int) {}
};
static_assert(PW % 4 == 0, "the leaf eliminates four columns at a time");

// Factor the PW x PW tile at (t0, t0) of S in place (lower part; lanes >= PW carry zeros).
// Returns the first column with a non-positive (or NaN) pivot, or -1.
__device__ __forceinline__ int leaf_factor(float *S, float *M, float *rd, float4 *xb, int t0,
                                           int lane) {
  const bool own = lane < PW;
  float *row = S + (t0 + (own ? lane : 0)) * PL + t0;
  float a[PW];
#pragma unroll
  for (int q = 0; q < PW / 4; ++q) {
    const float4 v = *reinterpret_cast<const float4 *>(row + 4 * q);
    a[4 * q] = v.x; a[4 * q + 1] = v.y; a[4 * q + 2] = v.z; a[4 * q + 3] = v.w;
  }
#pragma unroll
  for (int l = 0; l < PW; ++l)
    if (l > lane || !own) a[l] = 0.0f;
  float rdl = 0.0f, pvl = 1.0f;   // this lane's reciprocal pivot and its pivot
  LeafBlock<0>::run(a, rdl, pvl, xb, M, lane);
  if (own) {
#pragma unroll
    for (int q = 0; q < PW / 4; ++q)
      *reinterpret_cast<float4 *>(row + 4 * q) =
          make_float4(4 * q + 0 <= lane ? a[4 * q + 0] : 0.0f, 4 * q + 1 <= lane ? a[4 * q + 1] : 0.0f,
                      4 * q + 2 <= lane ? a[4 * q + 2] : 0.0f, 4 * q + 3 <= lane ? a[4 * q + 3] : 0.0f);
    rd[lane] = rdl;
  }
  // a pivot that is not positive (or is NaN) fails in its lane
  const unsigned badm = __ballot_sync(0xffffffffu, own && !(pvl > 0.0f));
  return badm ? t0 + __ffs((int)badm) - 1 : -1;
}

// The next leaf's tile (rows and columns t0..t0+PW-1 of S) minus its product over the
// sub-panel just solved (columns c0..c0+PW-1): the part of phase 2 that the next leaf
// waits for.  Lane (i, h) = (lane % PW, lane / PW) owns row t0 + i, columns t0 + 8h .. +7;
// the whole tile is written (the leaf reads its lower part only and clears the rest).
__device__ __forceinline__ void leaf_tile_update(float *S, int t0, int c0, int lane) {
  const int i = lane % PW, h = lane / PW;
  float x[PW];
#pragma unroll
  for (int q = 0; q < PW / 4; ++q) {
    const float4 v = *reinterpret_cast<const float4 *>(S + (t0 + i) * PL + c0 + 4 * q);
    x[4 * q] = v.x; x[4 * q + 1] = v.y; x[4 * q + 2] = v.z; x[4 * q + 3] = v.w;
  }
  float2 acc[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    acc[j] = make_float2(0.f, 0.f);
    const float *yj = S + (t0 + 8 * h + j) * PL + c0;
#pragma unroll
    for (int q = 0; q < PW / 4; ++q) {
      const float4 v = *reinterpret_cast<const float4 *>(yj + 4 * q);
      acc[j] = __ffma2_rn(make_float2(x[4 * q], x[4 * q + 1]), make_float2(v.x, v.y), acc[j]);
      acc[j] = __ffma2_rn(make_float2(x[4 * q + 2], x[4 * q + 3]), make_float2(v.z, v.w), acc[j]);
    }
  }
  float *ci = S + (t0 + i) * PL + t0 + 8 * h;
#pragma unroll
  for (int q = 0; q < 2; ++q) {
    float4 c = *reinterpret_cast<float4 *>(ci + 4 * q);
    c.x -= acc[4 * q].x + acc[4 * q].y;
    c.y -= acc[4 * q + 1].x + acc[4 * q + 1].y;
    c.z -= acc[4 * q + 2].x + acc[4 * q + 2].y;
    c.w -= acc[4 * q + 3].x + acc[4 * q + 3].y;
    *reinterpret_cast<float4 *>(ci + 4 * q) = c;
  }
}

// x L_pp^T = c for one row, in place: z_l -= z_j M[j][l] (l > j), then x_j = z_j / L_jj.
template <int J>
struct RowSolve {
  static __device__ __forceinline__ void run(float (&x)[PW], const float *M) {
#pragma unroll
    for (int l4 = (J + 1) / 4; l4 < PW / 4; ++l4) {
      const float4 v = *reinterpret_cast<const float4 *>(M + J * PL + 4 * l4);
      if (4 * l4 + 0 > J) x[4 * l4 + 0] = fmaf(-x[J], v.x, x[4 * l4 + 0]);
      if (4 * l4 + 1 > J) x[4 * l4 + 1] = fmaf(-x[J], v.y, x[4 * l4 + 1]);
      if (4 * l4 + 2 > J) x[4 * l4 + 2] = fmaf(-x[J], v.z, x[4 * l4 + 2]);
      if (4 * l4 + 3 > J) x[4 * l4 + 3] = fmaf(-x[J], v.w, x[4 * l4 + 3]);
    }
    RowSolve<J + 1>::run(x, M);
  }
};
template <>
struct RowSolve<PW> {
  static __device__ __forceinline__ void run(float (&)[PW], const float *) {}
};

// Phase-2 tile: C rows m0..m0+7 (Cm), columns n0 + lane + 32q (q < 2), minus
// sum_{k < PW} A(m, k) B(n, k) with A(m, k) = Am[m * PL + k], B(n, k) = Bm[n * PL + k];
// columns >= NB skipped, and with `lower` also columns above the row.
__device__ __forceinline__ void update_tile(float *Cm, const float *Am, const float *Bm,
                                            int m0, int n0, int lane, bool lower) {
  float2 c2[8][2];
#pragma unroll
  for (int i = 0; i < 8; ++i) c2[i][0] = c2[i][1] = make_float2(0.f, 0.f);
  const int nb0 = min(n0 + lane, NB - 1), nb1 = min(n0 + 32 + lane, NB - 1);
#pragma unroll
  for (int k = 0; k < PW; k += 4) {
    const float4 b0 = *reinterpret_cast<const float4 *>(Bm + nb0 * PL + k);
    const float4 b1 = *reinterpret_cast<const float4 *>(Bm + nb1 * PL + k);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float4 a = *reinterpret_cast<const float4 *>(Am + (m0 + i) * PL + k);
      c2[i][0] = __ffma2_rn(make_float2(a.x, a.y), make_float2(b0.x, b0.y), c2[i][0]);
      c2[i][0] = __ffma2_rn(make_float2(a.z, a.w), make_float2(b0.z, b0.w), c2[i][0]);
      c2[i][1] = __ffma2_rn(make_float2(a.x, a.y), make_float2(b1.x, b1.y), c2[i][1]);
      c2[i][1] = __ffma2_rn(make_float2(a.z, a.w), make_float2(b1.z, b1.w), c2[i][1]);
    }
  }
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      const int col = n0 + lane + 32 * q;
      if (col < NB && (!lower || col <= m0 + i)) Cm[(m0 + i) * PL + col] -= c2[i][q].x + c2[i][q].y;
    }
}

__global__ void __launch_bounds__(PF_THREADS, 1)
potrf_kernel(const float *A, int64_t d, int64_t k0, int n, float *Linv, DevStatus *st) {
  extern __shared__ __align__(16) float psm[];
  float *S = psm;                // NB x PL: working block, becomes L (lower)
  float *Bt = psm + NB * PL;     // NB x PL: transposed right-hand side -> Linv^T
  float *M = Bt + NB * PL;       // PW x PL: scaled transpose of the current leaf
  float *rd = M + PW * PL;       // PW reciprocal pivots of the current leaf
  __shared__ __align__(16) float4 cb[64];   // the leaf's row exchange (two buffers)
  __shared__ int s_skip, s_bad;
  const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
  if (tid == 0) { s_skip = st->status != 0; s_bad = -1; }
  __syncthreads();
  if (s_skip) return;
  // the block, padded with the identity beyond n; float4 index e = (row i, columns l4..l4+3)
  auto load4 = [&](int e) {
    const int i = e / (NB / 4), l4 = 4 * (e % (NB / 4));
    float v[4];
    if (i < n && (d % 4) == 0 && l4 + 4 <= n) {
      const float4 u = *reinterpret_cast<const float4 *>(A + (k0 + i) * d + k0 + l4);
      v[0] = u.x; v[1] = u.y; v[2] = u.z; v[3] = u.w;
    } else {
#pragma unroll
      for (int q = 0; q < 4; ++q) v[q] = (i < n && l4 + q < n) ? A[(k0 + i) * d + k0 + l4 + q] : 0.f;
    }
    float sv[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int l = l4 + q;
      sv[q] = (i < n && l < n) ? v[q] : (i == l ? 1.0f : 0.0f);
    }
    *reinterpret_cast<float4 *>(S + i * PL + l4) = make_float4(sv[0], sv[1], sv[2], sv[3]);
  };
  // identity rows R0..R0+PW-1 of Bt, first read by the phase 1 of sub-panel R0 / PW
  auto identity_rows = [&](int R0) {
    for (int e = tid - 32; e < PW * NB / 4; e += PF_THREADS - 32) {
      const int r = R0 + e / (NB / 4), c4 = 4 * (e % (NB / 4));
      *reinterpret_cast<float4 *>(Bt + r * PL + c4) =
          make_float4(r == c4 ? 1.f : 0.f, r == c4 + 1 ? 1.f : 0.f, r == c4 + 2 ? 1.f : 0.f,
                      r == c4 + 3 ? 1.f : 0.f);
    }
  };
  // the same rows written by warps 4, 8 and 12 alone (96 threads)
  auto identity_rows4 = [&](int R0) {
    for (int e = 32 * (warp / 4 - 1) + lane; e < PW * NB / 4; e += 96) {
      const int r = R0 + e / (NB / 4), c4 = 4 * (e % (NB / 4));
      *reinterpret_cast<float4 *>(Bt + r * PL + c4) =
          make_float4(r == c4 ? 1.f : 0.f, r == c4 + 1 ? 1.f : 0.f, r == c4 + 2 ? 1.f : 0.f,
                      r == c4 + 3 ? 1.f : 0.f);
    }
  };
  // warp 0 loads the first leaf's PW x PW tile and factors it at once; the other warps load
  // the rest of the block and the first identity rows meanwhile
  if (warp == 0) {
    for (int t = lane; t < PW * PW / 4; t += 32) load4((t / (PW / 4)) * (NB / 4) + t % (PW / 4));
    __syncwarp();
    const int bad = leaf_factor(S, M, rd, cb, 0, lane);
    if (lane == 0 && bad >= 0) s_bad = bad;
  } else {
#pragma unroll 4
    for (int e = tid - 32; e < NB * NB / 4; e += PF_THREADS - 32)
      if (e / (NB / 4) >= PW || e % (NB / 4) >= PW / 4) load4(e);
    identity_rows(0);
  }
  __syncthreads();
#pragma unroll 1
  for (int p = 0; p < NB / PW; ++p) {
    const int P0 = p * PW, R0 = P0 + PW;
    // phase 1: row r < R0 of Bt or row r >= R0 of S, columns P0..R0-1, one thread each
    if (tid < NB) {
      float *xr = (tid < R0 ? Bt : S) + tid * PL + P0;
      float x[PW];
#pragma unroll
      for (int q = 0; q < PW / 4; ++q) {
        const float4 v = *reinterpret_cast<const float4 *>(xr + 4 * q);
        x[4 * q] = v.x; x[4 * q + 1] = v.y; x[4 * q + 2] = v.z; x[4 * q + 3] = v.w;
      }
      RowSolve<0>::run(x, M);
#pragma unroll
      for (int q = 0; q < PW / 4; ++q) {
        const float4 r = *reinterpret_cast<const float4 *>(rd + 4 * q);
        *reinterpret_cast<float4 *>(xr + 4 * q) =
            make_float4(x[4 * q] * r.x, x[4 * q + 1] * r.y, x[4 * q + 2] * r.z, x[4 * q + 3] * r.w);
      }
    }
    __syncthreads();
    // rows P0..R0-1 of Linv are final: Linv[i][c] = Yt[c][i] for c < R0, zero beyond
    {
      const int i4 = P0 + 4 * (tid / NB), c = tid % NB;   // PW * NB / 4 == PF_THREADS
      const float4 v = c < R0 ? *reinterpret_cast<const float4 *>(Bt + c * PL + i4)
                              : make_float4(0.f, 0.f, 0.f, 0.f);
      const bool cc = c < n;
      Linv[(i4 + 0) * NB + c] = (cc && i4 + 0 < n) ? v.x : 0.0f;
      Linv[(i4 + 1) * NB + c] = (cc && i4 + 1 < n) ? v.y : 0.0f;
      Linv[(i4 + 2) * NB + c] = (cc && i4 + 2 < n) ? v.z : 0.0f;
      Linv[(i4 + 3) * NB + c] = (cc && i4 + 3 < n) ? v.w : 0.0f;
    }
    if (R0 == NB) break;
    if (warp == 0) {
      // the next leaf: its tile's share of phase 2, then its factorization
      leaf_tile_update(S, R0, P0, lane);
      __syncwarp();
      const int bad = leaf_factor(S, M, rd, cb, R0, lane);
      if (lane == 0 && bad >= 0 && s_bad < 0) s_bad = bad;
    } else if (warp % 4 == 0) {
      // warps 4, 8, 12 share warp 0's scheduler: they take only the next identity rows
      identity_rows4(R0);
    } else {
      // phase 2 over 8-row tiles of [Bt rows < R0 ; S rows >= R0] x 64-column tiles from R0,
      // without S rows R0..R0+PW-1 (their lower part is the next leaf's tile), on the twelve
      // warps of the other three schedulers
      const int nct = (NB - R0 + 63) / 64;
      const int wi = 3 * (warp / 4) + warp % 4 - 1;
#pragma unroll 1
      for (int t = wi; t < (NB / 8) * nct; t += PF_WARPS - PF_WARPS / 4) {
        const int m0 = 8 * (t / nct), n0 = R0 + 64 * (t % nct);
        if (m0 < R0) {
          update_tile(Bt, Bt + P0, S + P0, m0, n0, lane, false);
        } else if (m0 >= R0 + PW && n0 <= m0 + 7) {
          update_tile(S, S + P0, S + P0, m0, n0, lane, true);
        }
      }
    }
    __syncthreads();
  }
  if (s_bad >= 0 && tid == 0 && s_bad < n &&
      atomicCAS(&st->status, 0, (int)GPTQ_ERR_NOT_PD) == 0)
    st->info = (int)(k0 + s_bad) + 1;
}

// ---------------------------------------------------------------------------------------
// Row-panel product: P[r][j] = sum_{t<n} In[r][t] * Bm[j][t] for rows r in [r0, r1),
// j < nj, with In and Bm optionally given as TF32 head + tail pairs (In_lo, Bm_lo summed on
// load: the exact fp32 value).  Out[r][j] = P (sub = 0) or Out[r][j] -= P by atomic adds
// (sub = 1: another stream may be adding into the same block).  Optionally also writes the
// TF32 head/tail split of P into (hi, lo) panels (row r -> hi[r * ldh + j]).  A CTA takes
// RM_ROWS rows and NCQ of the four 32-column quarters of the output (blockIdx.y selects
// which); with NCQ = 4 a CTA owns whole rows, stages its input rows before writing, and
// Out may alias In.
// ---------------------------------------------------------------------------------------
constexpr int RM_ROWS = 32, RM_THREADS = 256;
constexpr int RML = NB + 4;  // smem leading dimension: float4 rows of 8 consecutive
                             // threads fall in distinct bank groups

// Thread (rg, cg) computes rows 4rg..4rg+3 x columns 32(q0 + q) + cg (q < NCQ): per 4-wide
// K step, 4 broadcast + NCQ float4 shared loads feed 8 NCQ paired FMAs.  With KS > 1 the CTA
// takes only K chunk blockIdx.z of NB / KS (a quarter of the loads and of the dependent
// product); its partial sums are subtracted by atomic adds, so KS > 1 needs sub and no
// head/tail output.
template <int NCQ, int KS = 1>
__global__ void __launch_bounds__(RM_THREADS)
rowmul_kernel(const float *In, const float *In_lo, int64_t ldi, float *Out, int64_t ldo,
              int64_t r0, int64_t r1, const float *Bm, const float *Bm_lo, int64_t ldb, int n,
              int nj, int sub, float *hi, float *lo, int64_t ldh, const DevStatus *st) {
  constexpr int KC = NB / KS, LD = KC + 4;   // K chunk and its shared row stride
  extern __shared__ __align__(16) float sm[];
  float *Bs = sm;                    // 32 NCQ x LD: the CTA's Bm rows (output columns, K)
  float *Is = sm + 32 * NCQ * LD;    // RM_ROWS x LD: the CTA's input rows
  if (st->status != 0) return;
  const int kz = KS > 1 ? KC * (int)blockIdx.z : 0;   // first K of the chunk
  const int tid = threadIdx.x;
  const int64_t rb = r0 + (int64_t)blockIdx.x * RM_ROWS;
  const int q0 = blockIdx.y * NCQ;
  // every global load of the CTA is issued before the first shared store (one round trip)
  constexpr int NBI = 32 * NCQ * KC / 4 / RM_THREADS, NII = RM_ROWS * KC / 4 / RM_THREADS;
  float4 bv[NBI], iv[NII];
#pragma unroll
  for (int it = 0; it < NBI; ++it) {
    const int e = it * RM_THREADS + tid;  // float4 index within the CTA's Bm rows
    const int j = e / (KC / 4), t4 = kz + 4 * (e % (KC / 4));
    const int64_t bo = (int64_t)(32 * q0 + j) * ldb + t4;
    bv[it] = make_float4(0.f, 0.f, 0.f, 0.f);
    if (32 * q0 + j < nj) {
      bv[it] = *reinterpret_cast<const float4 *>(Bm + bo);
      if (Bm_lo) {
        const float4 u = *reinterpret_cast<const float4 *>(Bm_lo + bo);
        bv[it] = make_float4(bv[it].x + u.x, bv[it].y + u.y, bv[it].z + u.z, bv[it].w + u.w);
      }
    }
  }
  const bool vec = (ldi % 4) == 0 && (((uintptr_t)In) % 16) == 0;
#pragma unroll
  for (int it = 0; it < NII; ++it) {
    const int e = it * RM_THREADS + tid;
    const int r = e / (KC / 4), t4 = kz + 4 * (e % (KC / 4));
    const int64_t gr = rb + r;
    iv[it] = make_float4(0.f, 0.f, 0.f, 0.f);
    if (gr < r1) {
      if (vec && t4 + 4 <= n) {
        iv[it] = *reinterpret_cast<const float4 *>(In + gr * ldi + t4);
        if (In_lo) {
          const float4 u = *reinterpret_cast<const float4 *>(In_lo + gr * ldi + t4);
          iv[it] = make_float4(iv[it].x + u.x, iv[it].y + u.y, iv[it].z + u.z, iv[it].w + u.w);
        }
      } else {
#define RM_IN(q) ((t4 + q < n) ? In[gr * ldi + t4 + q] + (In_lo ? In_lo[gr * ldi + t4 + q] : 0.f) : 0.f)
        iv[it] = make_float4(RM_IN(0), RM_IN(1), RM_IN(2), RM_IN(3));
#undef RM_IN
      }
    }
  }
#pragma unroll
  for (int it = 0; it < NBI; ++it) {
    const int e = it * RM_THREADS + tid;
    *reinterpret_cast<float4 *>(Bs + (e / (KC / 4)) * LD + 4 * (e % (KC / 4))) = bv[it];
  }
#pragma unroll
  for (int it = 0; it < NII; ++it) {
    const int e = it * RM_THREADS + tid;
    *reinterpret_cast<float4 *>(Is + (e / (KC / 4)) * LD + 4 * (e % (KC / 4))) = iv[it];
  }
  __syncthreads();
  const int rg = tid / 32, cg = tid % 32;
  float2 acc[4][NCQ];   // even and odd k summed apart
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int q = 0; q < NCQ; ++q) acc[i][q] = make_float2(0.f, 0.f);
#pragma unroll 2
  for (int t = 0; t < KC; t += 4) {
    float4 a[4], b[NCQ];
#pragma unroll
    for (int i = 0; i < 4; ++i) a[i] = *reinterpret_cast<const float4 *>(Is + (4 * rg + i) * LD + t);
#pragma unroll
    for (int q = 0; q < NCQ; ++q) b[q] = *reinterpret_cast<const float4 *>(Bs + (32 * q + cg) * LD + t);
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int q = 0; q < NCQ; ++q) {
        acc[i][q] = __ffma2_rn(make_float2(a[i].x, a[i].y), make_float2(b[q].x, b[q].y), acc[i][q]);
        acc[i][q] = __ffma2_rn(make_float2(a[i].z, a[i].w), make_float2(b[q].z, b[q].w), acc[i][q]);
      }
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int64_t gr = rb + 4 * rg + i;
    if (gr >= r1) continue;
#pragma unroll
    for (int q = 0; q < NCQ; ++q) {
      const int j = 32 * (q0 + q) + cg;
      const float v = (j < nj) ? acc[i][q].x + acc[i][q].y : 0.f;
      if (Out && j < nj) {
        if (sub) atomicAdd(Out + gr * ldo + j, -v);
        else Out[gr * ldo + j] = v;
      }
      if (hi) {
        const float h = tf32_head(v);
        hi[gr * ldh + j] = h;
        lo[gr * ldh + j] = v - h;
      }
    }
  }
}

// U[i][j] = Yt[d-1-j][d-1-i] for i <= j, 0 below the diagonal: 64 x 64 tiles through shared
// memory (Yt rows read forwards and stored reversed, U rows written), float4 with VEC
// (d % 4 == 0, both 16-byte aligned).  Tiles wholly below the diagonal only write zeros.
constexpr int AU_T = 64;

template <bool VEC>
__global__ void __launch_bounds__(256) assemble_u_kernel(const float *Yt, float *U, int64_t d) {
  __shared__ float tile[AU_T][AU_T + 1];   // tile[jj][ii] = Yt[d-1-j][d-1-i]
  const int64_t i0 = (int64_t)blockIdx.y * AU_T, j0 = (int64_t)blockIdx.x * AU_T;
  const int tid = threadIdx.x, c4 = 4 * (tid % 16), rr = tid / 16;
  const bool any = i0 <= j0 + AU_T - 1;
  if (any) {
    // Yt row y = d-1-(j0+jj), columns x = xs + c4 + e hold ii = AU_T-1-c4-e (xs = d-AU_T-i0)
    const int64_t xs = d - AU_T - i0;
#pragma unroll
    for (int p = 0; p < AU_T / 16; ++p) {
      const int jj = rr + 16 * p;
      const int64_t y = d - 1 - (j0 + jj);
      float v[4] = {0.f, 0.f, 0.f, 0.f};
      if (y >= 0) {
        const int64_t x = xs + c4;
        if (VEC && x >= 0) {
          const float4 u = *reinterpret_cast<const float4 *>(Yt + y * d + x);
          v[0] = u.x; v[1] = u.y; v[2] = u.z; v[3] = u.w;
        } else {
#pragma unroll
          for (int e = 0; e < 4; ++e)
            if (x + e >= 0) v[e] = Yt[y * d + x + e];
        }
      }
#pragma unroll
      for (int e = 0; e < 4; ++e) tile[jj][AU_T - 1 - c4 - e] = v[e];
    }
  }
  __syncthreads();
#pragma unroll
  for (int p = 0; p < AU_T / 16; ++p) {
    const int ii = rr + 16 * p;
    const int64_t i = i0 + ii;
    if (i >= d) continue;
    float v[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int64_t j = j0 + c4 + e;
      v[e] = (any && i <= j) ? tile[c4 + e][ii] : 0.f;
    }
    const int64_t j = j0 + c4;
    if (VEC && j + 4 <= d) {
      *reinterpret_cast<float4 *>(U + i * d + j) = make_float4(v[0], v[1], v[2], v[3]);
    } else {
#pragma unroll
      for (int e = 0; e < 4; ++e)
        if (j + e < d) U[i * d + j + e] = v[e];
    }
  }
}

// A group's L panels (rows of L, TF32 head + tail) and inverse panels (rows c of Yt) side by
// side, d x GW each, panel k in columns (k % kGroup) NB; both double buffered by group
// parity.  Linv (the inverted diagonal block) by panel parity.
struct PrepWs {
  DevStatus *st;
  float *Yt;
  float *Yhi[2], *Ylo[2], *Lhi[2], *Llo[2];
  float *Linv[2];
};

PrepWs carve_prepare(void *ws, int64_t d) {
  char *p = (char *)ws;
  PrepWs w;
  w.st = (DevStatus *)p;
  p += 256;
  w.Yt = (float *)p;  p += round_up((size_t)d * d * 4, 256);
  for (int b = 0; b < 2; ++b) {
    w.Yhi[b] = (float *)p; p += round_up((size_t)d * GW * 4, 256);
    w.Ylo[b] = (float *)p; p += round_up((size_t)d * GW * 4, 256);
    w.Lhi[b] = (float *)p; p += round_up((size_t)d * GW * 4, 256);
    w.Llo[b] = (float *)p; p += round_up((size_t)d * GW * 4, 256);
    w.Linv[b] = (float *)p; p += round_up((size_t)NB * NB * 4, 256);
  }
  return w;
}

// Rows [S + NB, E) of a group's inverse panels are zero in the columns of the group's
// panels that end at or above the row (panel p covers rows c < S + (p + 1) NB only), so the
// group's deferred product can take all its panels over rows [0, E).
__global__ void __launch_bounds__(128) zero_group_tail_kernel(float *hi, float *lo, int64_t S,
                                                              int64_t E) {
  const int64_t r = S + NB + blockIdx.x;
  if (r >= E) return;
  const int ncols = (int)(NB * ((r - S) / NB));
  float4 *h = reinterpret_cast<float4 *>(hi + r * GW), *l = reinterpret_cast<float4 *>(lo + r * GW);
  for (int c = threadIdx.x; c < ncols / 4; c += blockDim.x) {
    h[c] = make_float4(0.f, 0.f, 0.f, 0.f);
    l[c] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
}

// Four streams and their events per device, created once and kept for the process: the
// panel loop runs its critical chain on `crit` (the device's highest stream priority, so its
// blocks are dispatched first whenever an SM has room) and `crit2`, the panels' near updates
// beside it on `s`, and the groups' deferred far updates on `far` (the lowest priority).
struct SideStream {
  std::mutex enqueue;  // one panel loop at a time enqueues on these events
  cudaStream_t s = nullptr, crit = nullptr, crit2 = nullptr, far = nullptr;
  cudaEvent_t ea[2] = {nullptr, nullptr}, eb[2] = {nullptr, nullptr}, en[2] = {nullptr, nullptr},
              ep[2] = {nullptr, nullptr}, ed[2] = {nullptr, nullptr}, eg[2] = {nullptr, nullptr},
              ef[2] = {nullptr, nullptr}, e0 = nullptr, e1 = nullptr, e_in = nullptr,
              e_out = nullptr;
  int num_sms = 0;
  GraphCache graphs;   // the panel loop captured per buffer set
};
constexpr int kMaxDevices = 128;
std::mutex g_side_mu;
SideStream g_side[kMaxDevices];

gptq_status side_stream(SideStream **out) {
  int dev = -1;
  GPTQ_CUDA_CHECK(cudaGetDevice(&dev));
  if (dev < 0 || dev >= kMaxDevices) return GPTQ_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_side_mu);
  SideStream &ss = g_side[dev];
  if (!ss.s) {
    int lo = 0, hi = 0;
    GPTQ_CUDA_CHECK(cudaDeviceGetStreamPriorityRange(&lo, &hi));
    // priorities run from lo down to hi: crit, then crit2 one level below it, then the near
    // updates, then the far updates at the lowest
    const int p2 = hi < lo ? hi + 1 : hi, p3 = p2 < lo ? p2 + 1 : p2;
    GPTQ_CUDA_CHECK(cudaStreamCreateWithPriority(&ss.crit, cudaStreamNonBlocking, hi));
    GPTQ_CUDA_CHECK(cudaStreamCreateWithPriority(&ss.crit2, cudaStreamNonBlocking, p2));
    GPTQ_CUDA_CHECK(cudaStreamCreateWithPriority(&ss.s, cudaStreamNonBlocking, p3));
    GPTQ_CUDA_CHECK(cudaStreamCreateWithPriority(&ss.far, cudaStreamNonBlocking, lo));
    GPTQ_CUDA_CHECK(cudaDeviceGetAttribute(&ss.num_sms, cudaDevAttrMultiProcessorCount, dev));
    for (int b = 0; b < 2; ++b) {
      GPTQ_CUDA_CHECK(cudaEventCreateWithFlags(&ss.ea[b], cudaEventDisableTiming));
      GPTQ_CUDA_CHECK(cudaEventCreateWithFlags(&ss.eb[b], cudaEventDisableTiming));
      GPTQ_CUDA_CHECK(cudaEventCreateWithFlags(&ss.en[b], cudaEventDisableTiming));
      GPTQ_CUDA_CHECK(cudaEventCreateWithFlags(&ss.ep[b], cudaEventDisableTiming));
      GPTQ_CUDA_CHECK(cudaEventCreateWithFlags(&ss.ed[b], cudaEventDisableTiming));
      GPTQ_CUDA_CHECK(cudaEventCreateWithFlags(&ss.eg[b], cudaEventDisableTiming));
      GPTQ_CUDA_CHECK(cudaEventCreateWithFlags(&ss.ef[b], cudaEventDisableTiming));
    }
    GPTQ_CUDA_CHECK(cudaEventCreateWithFlags(&ss.e0, cudaEventDisableTiming));
    GPTQ_CUDA_CHECK(cudaEventCreateWithFlags(&ss.e1, cudaEventDisableTiming));
    GPTQ_CUDA_CHECK(cudaEventCreateWithFlags(&ss.e_in, cudaEventDisableTiming));
    GPTQ_CUDA_CHECK(cudaEventCreateWithFlags(&ss.e_out, cudaEventDisableTiming));
  }
  *out = &ss;
  return GPTQ_OK;
}

}  // namespace

size_t prepare_ws_bytes(int64_t d) {
  return 256 + round_up((size_t)d * d * 4, 256) + 8 * round_up((size_t)d * GW * 4, 256) +
         2 * round_up((size_t)NB * NB * 4, 256);
}

// Panel loop.  On the critical stream (highest priority; the caller's stream when the
// side streams cannot be used):
//   potrf(k) -> trsm(k) for the next NB rows -> the next panel column's update on its
//   diagonal block (rows [k1, k1 + NB)) -> potrf(k + 1) ...
// On a second critical stream, once potrf(k) is done: trsm(k) for the rows below, then (once
// the critical stream's NB rows of L exist) the next column's update for those rows (a
// tensor-core product), beside potrf(k + 1), which leaves all but one SM idle; trsm(k + 1)
// waits for it.  On the side
// stream, once panel k's factor and L panel exist:
//   inverse step a(k) -> the rest of the trailing update (the lower trapezoid from
//   k1 + NB) -> inverse step b(k),
// both updates over the columns up to the end of the next group of kGroup panels only (the
// near columns).  Once a group's last inverse panel exists, the far stream applies the
// group's updates to the columns beyond (the far columns) as two K = GW products: the
// output is read and written once per group instead of once per panel.  potrf(k) waits for
// the side stream's panel k - 2, which last wrote its diagonal block and read the panel
// buffers it is about to overwrite; a group's first potrf also waits for the far update of
// the group two before it, the last to write its columns and to read the group buffers it
// is about to overwrite.  Updates of one column block by several streams are atomic adds
// (L2 reduce-adds in the tensor-core epilogue, red.add in the next-column update); where C
// is not 16-byte aligned everything runs on the caller's stream, without deferral.  The
// caller's stream waits for all of them at the end.
namespace {

// The panel loop's launches (no set-up, no locking): on `s`, and with `ss` on its four
// streams as well.
gptq_status enqueue_prepare(float *H, int64_t d, float damp, float *U, uint8_t *dead_mask,
                            void *ws, cudaStream_t s, SideStream *ss) {
  const size_t rm_smem = (NB + RM_ROWS) * RML * sizeof(float);       // whole rows
  const size_t rmq_smem = (32 + RM_ROWS) * RML * sizeof(float);       // one column quarter
  const size_t rmk_smem = (32 + RM_ROWS) * (NB / 4 + 4) * sizeof(float);   // and a K quarter
  const size_t potrf_smem = kPotrfSmem;
  PrepWs w = carve_prepare(ws, d);
  const bool overlap = ss != nullptr;
  const bool defer = overlap;
  cudaStream_t b = overlap ? ss->s : s;
  cudaStream_t f = overlap ? ss->far : s;
  // the side stream's persistent GEMMs leave 16 SMs to the critical chain (measured: better
  // than all SMs, than one CTA per tile, and the same as 32)
  const int side_ctas = overlap ? std::max(1, ss->num_sms - 16) : 0;
  // the far products are persistent too (measured: 95 against 116 ms for one CTA per tile
  // on a 28672-wide layer, 8.3 against 9.0 ms at 11008).  On narrower layers they are a
  // smaller part of the work and leave more SMs to the chain and the near products
  // (measured, prepare: 1.221 against 1.248 ms at 4096 leaving 76, 7.53 against 7.74 ms at
  // 11008 leaving 48; at 28672 leaving 32 or more costs 1.5 % to 50 %)
  const int far_left = d <= 6144 ? 76 : d <= 16384 ? 48 : 16;
  const int far_ctas = overlap ? std::max(1, ss->num_sms - far_left) : 0;
  GPTQ_CUDA_CHECK(cudaMemsetAsync(w.st, 0, sizeof(DevStatus), s));
  // vector path: rows of H, Yt and U start 16-byte aligned (the workspace is)
  const bool vec = (d % 4) == 0 && (((uintptr_t)H) % 16) == 0 && (((uintptr_t)U) % 16) == 0;
  dead_damp_kernel<<<1, 1024, 0, s>>>(H, d, damp, dead_mask, w.st);
  GPTQ_LAUNCH_CHECK();
  if (vec) reverse_lower_kernel<true><<<(unsigned)d, RV_THREADS, 0, s>>>(H, d, w.Yt, w.st);
  else reverse_lower_kernel<false><<<(unsigned)d, RV_THREADS, 0, s>>>(H, d, w.Yt, w.st);
  GPTQ_LAUNCH_CHECK();
  cudaStream_t c = overlap ? ss->crit : s;  // the critical chain
  if (overlap) {
    GPTQ_CUDA_CHECK(cudaEventRecord(ss->e0, s));
    GPTQ_CUDA_CHECK(cudaStreamWaitEvent(b, ss->e0, 0));
    GPTQ_CUDA_CHECK(cudaStreamWaitEvent(c, ss->e0, 0));
  }
  float *A = H;  // reversed, damped Hessian; lower triangle is the Cholesky workspace
  int k = 0;
  bool next_rest = false;   // the last panel's column update left rows to the second stream
  bool far_pending[2] = {false, false};   // by group parity: ef recorded, not yet waited on
  bool far_any[2] = {false, false};       // by group parity: ef recorded in this call
  for (int64_t k0 = 0; k0 < d; k0 += NB, ++k) {
    const int par = k & 1;
    const int n = (int)std::min<int64_t>(NB, d - k0);
    const int64_t k1 = k0 + n;
    const int64_t grp = k / kGroup, S = grp * GW;
    const int gp = (int)(grp & 1), slot = k % kGroup;
    // the near columns end with the next group; with deferral off, all columns are near
    const int64_t near_end = defer ? std::min(d, S + 2 * GW) : d;
    const bool far_after = defer && slot == kGroup - 1 && S + 2 * GW < d;
    float *lhi = w.Lhi[gp] + slot * NB, *llo = w.Llo[gp] + slot * NB;
    float *yhi = w.Yhi[gp] + slot * NB, *ylo = w.Ylo[gp] + slot * NB;
    if (overlap && k >= 2) GPTQ_CUDA_CHECK(cudaStreamWaitEvent(c, ss->eb[par], 0));
    if (slot == 0 && far_pending[gp]) {
      GPTQ_CUDA_CHECK(cudaStreamWaitEvent(c, ss->ef[gp], 0));
      far_pending[gp] = false;
    }
    GPTQ_TRY(launch_kernel(potrf_kernel, 1, PF_THREADS, potrf_smem, c, A, d, k0, n,
                           w.Linv[par], w.st));
    if (overlap) GPTQ_CUDA_CHECK(cudaEventRecord(ss->ep[par], c));
    // the previous column update's rows below the diagonal block (second critical stream)
    if (overlap && next_rest) GPTQ_CUDA_CHECK(cudaStreamWaitEvent(c, ss->en[par ^ 1], 0));
    next_rest = false;
    if (k1 < d) {
      const int nn = (int)std::min<int64_t>(NB, d - k1);
      // trsm: rows [r0, r1) of panel k -> L panel (hi/lo)
      auto trsm = [&](int64_t r0, int64_t r1, cudaStream_t st) {
        dim3 g((unsigned)ceil_div(r1 - r0, RM_ROWS), 4);
        return launch_kernel(rowmul_kernel<1>, g, RM_THREADS, rmq_smem, st, A + k0,
                             (const float *)nullptr, d, (float *)nullptr, (int64_t)0, r0, r1,
                             w.Linv[par], (const float *)nullptr, (int64_t)NB, n, n, 0, lhi,
                             llo, GW, w.st);
      };
      // next panel column, rows k1 + [r0, r1): A[., k1:k1+NB] -= L[.] L[k1:k1+NB]^T (fp32
      // from the head + tail panels; atomic adds: the side stream's previous trailing update
      // adds here too)
      auto next_col = [&](int64_t r0, int64_t r1, cudaStream_t st) {
        dim3 g2((unsigned)ceil_div(r1 - r0, RM_ROWS), (unsigned)ceil_div(nn, 32));
        return launch_kernel(rowmul_kernel<1>, g2, RM_THREADS, rmq_smem, st, lhi + k1 * GW,
                             llo + k1 * GW, GW, A + k1 * d + k1, d, r0, r1, lhi + k1 * GW,
                             llo + k1 * GW, GW, n, nn, 1, (float *)nullptr, (float *)nullptr,
                             (int64_t)0, w.st);
      };
      if (overlap && d - k1 > nn) {
        cudaStream_t c2 = ss->crit2;
        GPTQ_CUDA_CHECK(cudaStreamWaitEvent(c2, ss->ep[par], 0));
        GPTQ_TRY(trsm(k1 + nn, d, c2));           // the rows below, beside the chain
        GPTQ_CUDA_CHECK(cudaEventRecord(ss->ea[par], c2));
        GPTQ_TRY(trsm(k1, k1 + nn, c));           // the next potrf's rows
        GPTQ_CUDA_CHECK(cudaEventRecord(ss->ed[par], c));
        GPTQ_CUDA_CHECK(cudaStreamWaitEvent(c2, ss->ed[par], 0));
        {
          // the rows below, beside the next potrf: a tensor-core product of the L panel's
          // head/tail rows (measured: prepare 1.28 against 1.35 ms at d = 4096, 7.8 against
          // 8.3 ms at 11008, 92 against 95 ms at 28672, than the CUDA-core row product)
          GemmArgs t{};
          t.a_hi = lhi + (k1 + nn) * GW; t.a_lo = llo + (k1 + nn) * GW; t.lda = GW;
          t.b_hi = lhi + k1 * GW; t.b_lo = llo + k1 * GW; t.ldb = GW;
          t.c = A + (k1 + nn) * d + k1; t.ldc = d;
          t.M = d - k1 - nn; t.N = nn; t.K = n;
          t.alpha = -1.0f; t.lower_only = 0; t.trans_c = 0; t.max_ctas = -1;
          GPTQ_TRY(launch_gemm_nt(t, w.st, c2));
        }
        GPTQ_CUDA_CHECK(cudaEventRecord(ss->en[par], c2));
        next_rest = true;
        {
          // the next potrf's block, in four K chunks (64 CTAs; atomic adds)
          dim3 g2((unsigned)ceil_div(nn, RM_ROWS), (unsigned)ceil_div(nn, 32), 4);
          GPTQ_TRY(launch_kernel(rowmul_kernel<1, 4>, g2, RM_THREADS, rmk_smem, c,
                                 lhi + k1 * GW, llo + k1 * GW, GW, A + k1 * d + k1, d,
                                 (int64_t)0, (int64_t)nn, lhi + k1 * GW, llo + k1 * GW, GW, n,
                                 nn, 1, (float *)nullptr, (float *)nullptr, (int64_t)0, w.st));
        }
        GPTQ_CUDA_CHECK(cudaStreamWaitEvent(b, ss->ea[par], 0));
        GPTQ_CUDA_CHECK(cudaStreamWaitEvent(b, ss->ed[par], 0));
      } else {
        GPTQ_TRY(trsm(k1, d, c));
        GPTQ_TRY(next_col(0, d - k1, c));
        if (overlap) {
          GPTQ_CUDA_CHECK(cudaEventRecord(ss->ea[par], c));
          GPTQ_CUDA_CHECK(cudaStreamWaitEvent(b, ss->ea[par], 0));
        }
      }
    } else if (overlap) {
      GPTQ_CUDA_CHECK(cudaEventRecord(ss->ea[par], c));
      GPTQ_CUDA_CHECK(cudaStreamWaitEvent(b, ss->ea[par], 0));
    }
    if (slot == 0 && defer && S + 2 * GW < d) {
      // this group will have a far update: its inverse panels' rows below each panel are zero
      const int64_t E = std::min(d, S + GW);
      if (E > S + NB)
        GPTQ_TRY(launch_kernel(zero_group_tail_kernel, (unsigned)(E - S - NB), 128, 0, b,
                               w.Yhi[gp], w.Ylo[gp], S, E));
    }
    // inverse step a: Yt[c][k0:k1] = Bt[c][k0:k1] Linv^T for c in [0, k1), in place
    {
      const unsigned g = (unsigned)ceil_div(k1, RM_ROWS);
      GPTQ_TRY(launch_kernel(rowmul_kernel<4>, g, RM_THREADS, rm_smem, b,
                             (const float *)(w.Yt + k0), (const float *)nullptr, d, w.Yt + k0, d,
                             (int64_t)0, k1, (const float *)w.Linv[par], (const float *)nullptr,
                             (int64_t)NB, n, n, 0, yhi, ylo, GW, w.st));
    }
    if (far_after) {
      // the group's far columns [S + 2 GW, d): the rest of its trailing update (lower
      // square) and of its inverse step b (rows c < S + GW), K = GW
      const int64_t r0 = S + 2 * GW;
      GPTQ_CUDA_CHECK(cudaEventRecord(ss->eg[gp], b));
      GPTQ_CUDA_CHECK(cudaStreamWaitEvent(f, ss->eg[gp], 0));
      GemmArgs t{};
      t.a_hi = w.Lhi[gp] + r0 * GW; t.a_lo = w.Llo[gp] + r0 * GW; t.lda = GW;
      t.b_hi = w.Lhi[gp] + r0 * GW; t.b_lo = w.Llo[gp] + r0 * GW; t.ldb = GW;
      t.c = A + r0 * d + r0; t.ldc = d;
      t.M = d - r0; t.N = d - r0; t.K = GW;
      t.alpha = -1.0f; t.lower_only = 1; t.trans_c = 0; t.max_ctas = far_ctas;
      GPTQ_TRY(launch_gemm_nt(t, w.st, f));
      GemmArgs v{};
      v.a_hi = w.Yhi[gp]; v.a_lo = w.Ylo[gp]; v.lda = GW;
      v.b_hi = w.Lhi[gp] + r0 * GW; v.b_lo = w.Llo[gp] + r0 * GW; v.ldb = GW;
      v.c = w.Yt + r0; v.ldc = d;
      v.M = S + GW; v.N = d - r0; v.K = GW;
      v.alpha = -1.0f; v.lower_only = 0; v.trans_c = 0; v.max_ctas = far_ctas;
      GPTQ_TRY(launch_gemm_nt(v, w.st, f));
      GPTQ_CUDA_CHECK(cudaEventRecord(ss->ef[gp], f));
      far_pending[gp] = far_any[gp] = true;
    }
    if (k1 < d) {
      if (near_end - k1 > NB) {
        // the rest of the trailing update: lower trapezoid from (k1 + NB, k1 + NB), near
        // columns
        const int64_t r0 = k1 + NB;
        GemmArgs g2{};
        g2.a_hi = lhi + r0 * GW; g2.a_lo = llo + r0 * GW; g2.lda = GW;
        g2.b_hi = lhi + r0 * GW; g2.b_lo = llo + r0 * GW; g2.ldb = GW;
        g2.c = A + r0 * d + r0; g2.ldc = d;
        g2.M = d - r0; g2.N = near_end - r0; g2.K = n;
        g2.alpha = -1.0f; g2.lower_only = 1; g2.trans_c = 0; g2.max_ctas = side_ctas;
        GPTQ_TRY(launch_gemm_nt(g2, w.st, b));
      }
      // inverse step b: Bt[c][k1:near_end] -= Yp[c] Lp[k1:near_end]^T for c < k1
      GemmArgs h{};
      h.a_hi = yhi; h.a_lo = ylo; h.lda = GW;
      h.b_hi = lhi + k1 * GW; h.b_lo = llo + k1 * GW; h.ldb = GW;
      h.c = w.Yt + k1; h.ldc = d;
      h.M = k1; h.N = near_end - k1; h.K = n;
      h.alpha = -1.0f; h.lower_only = 0; h.trans_c = 0; h.max_ctas = side_ctas;
      GPTQ_TRY(launch_gemm_nt(h, w.st, b));
    }
    if (overlap) GPTQ_CUDA_CHECK(cudaEventRecord(ss->eb[par], b));
  }
  if (overlap) {
    // join only what this call recorded (one panel records eb[0] only): waiting on an event
    // recorded elsewhere is not allowed inside a graph capture
    GPTQ_CUDA_CHECK(cudaEventRecord(ss->e1, c));
    GPTQ_CUDA_CHECK(cudaStreamWaitEvent(s, ss->e1, 0));
    for (int p = 0; p < std::min(k, 2); ++p) GPTQ_CUDA_CHECK(cudaStreamWaitEvent(s, ss->eb[p], 0));
    for (int p = 0; p < 2; ++p)
      if (far_any[p]) GPTQ_CUDA_CHECK(cudaStreamWaitEvent(s, ss->ef[p], 0));
  }
  dim3 tg((unsigned)ceil_div(d, AU_T), (unsigned)ceil_div(d, AU_T));
  if (vec) assemble_u_kernel<true><<<tg, 256, 0, s>>>(w.Yt, U, d);
  else assemble_u_kernel<false><<<tg, 256, 0, s>>>(w.Yt, U, d);
  GPTQ_LAUNCH_CHECK();
  return GPTQ_OK;
}

}  // namespace

gptq_status launch_prepare(float *H, int64_t d, float damp, float *U, uint8_t *dead_mask,
                           void *ws, cudaStream_t s) {
  GPTQ_TRY(ensure_smem_attr((const void *)potrf_kernel, (int)kPotrfSmem));
  GPTQ_TRY(ensure_smem_attr((const void *)rowmul_kernel<4>,
                            (int)((NB + RM_ROWS) * RML * sizeof(float))));
  const bool overlap = (d % 4) == 0 && (((uintptr_t)H) % 16) == 0;
  if (!overlap) return enqueue_prepare(H, d, damp, U, dead_mask, ws, s, nullptr);
  SideStream *ss = nullptr;
  GPTQ_TRY(side_stream(&ss));
  std::lock_guard<std::mutex> lock(ss->enqueue);
  // Graph replay (graph_cache.cuh): the loop is ~200 dependent launches on three streams.
  if (caller_capturing(s)) return enqueue_prepare(H, d, damp, U, dead_mask, ws, s, ss);
  GPTQ_CUDA_CHECK(cudaEventRecord(ss->e_in, s));
  GPTQ_CUDA_CHECK(cudaStreamWaitEvent(ss->crit, ss->e_in, 0));
  uint32_t damp_bits = 0;
  memcpy(&damp_bits, &damp, 4);
  const std::vector<uint64_t> key = {(uint64_t)H, (uint64_t)U, (uint64_t)dead_mask,
                                     (uint64_t)ws, (uint64_t)d, (uint64_t)damp_bits};
  gptq_status st = GPTQ_OK;
  if (!ss->graphs.run(key, ss->crit, [&](cudaStream_t o) {
        return enqueue_prepare(H, d, damp, U, dead_mask, ws, o, ss);
      }, &st))
    return enqueue_prepare(H, d, damp, U, dead_mask, ws, s, ss);  // after the join above
  GPTQ_CUDA_CHECK(cudaEventRecord(ss->e_out, ss->crit));
  GPTQ_CUDA_CHECK(cudaStreamWaitEvent(s, ss->e_out, 0));
  return GPTQ_OK;
}

}  // namespace gptq
