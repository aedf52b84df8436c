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

#include "common.cuh"

namespace gptq {

namespace {

constexpr int NB = 128;            // panel width
constexpr int LDS = NB + 1;        // padded smem leading dimension

// ---------------------------------------------------------------------------------------
// Dead columns and damping (one CTA): dead = {i : H_ii == 0}; H_ii <- 1 for dead i;
// lambda = damp * mean(diag); H_ii += lambda.
// ---------------------------------------------------------------------------------------
__global__ void dead_damp_kernel(float *H, int64_t d, float damp, uint8_t *dead_mask,
                                 DevStatus *st) {
  __shared__ double red[32];
  __shared__ int s_ndead, s_bad;
  if (threadIdx.x == 0) { s_ndead = 0; s_bad = 0; }
  __syncthreads();
  double sum = 0.0;
  int ndead = 0, bad = 0;
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
  for (int64_t i = threadIdx.x; i < d; i += blockDim.x) {
    const float h = H[i * d + i];
    const bool dead = (h == 0.0f);
    if (dead_mask) dead_mask[i] = dead ? 1 : 0;
    H[i * d + i] = (dead ? 1.0f : h) + lam;
  }
}

// In-place reversal of the d*d array (A = P H P) with a finiteness check.
__global__ void reverse_kernel(float *H, int64_t n, DevStatus *st) {
  int bad = 0;
  for (int64_t k = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; k < n / 2;
       k += (int64_t)gridDim.x * blockDim.x) {
    const float a = H[k], b = H[n - 1 - k];
    bad |= !isfinite(a) | !isfinite(b);
    H[k] = b;
    H[n - 1 - k] = a;
  }
  if (bad) set_status(st, GPTQ_ERR_NONFINITE);
}

// Yt = identity.
__global__ void identity_kernel(float *Y, int64_t d) {
  for (int64_t k = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; k < d * d;
       k += (int64_t)gridDim.x * blockDim.x)
    Y[k] = (k / d == k % d) ? 1.0f : 0.0f;
}

// ---------------------------------------------------------------------------------------
// potrf: Cholesky factor of the n x n diagonal block at (k0, k0) of A (n <= NB) and, in
// the same pass, its inverse Linv (the forward substitution L X = I run alongside).  Only
// Linv leaves the kernel (NB x NB, lower, zero padded): the panel below is L_ik = A_ik
// Linv^T and the inversion needs Linv only.
//
// Register blocked, 16 warps: warp w owns columns [8w, 8w+8), lane owns rows lane + 32a,
// of both the working block S and the right-hand side B (identity at start).  Column j:
//   publish S[:, j] and B[j, :]; one barrier; then with p = S[j][j] (pivot):
//   S[i][l] -= S[i][j] S[l][j] / p          for i >= l > j      (outer-product Cholesky)
//   B[i][c] -= S[i][j] B[j][c] / p  (i > j), B[j][c] /= sqrt(p)  (forward substitution)
// which leaves B = L^-1.  Warps whose columns are finished (or not yet reached, for B)
// skip their update; column buffers are double buffered so one barrier per column suffices.
// A non-positive pivot records NOT_PD with its global index.
// ---------------------------------------------------------------------------------------
constexpr int PF_THREADS = 512;

template <int J>
struct PotrfStep {
  static __device__ __forceinline__ void run(float (&s)[4][8], float (&x)[4][8],
                                             float *colbuf, float *rowbuf, int warp, int lane,
                                             int &bad) {
    constexpr int BJ = J % 8, AJ = J / 32, LJ = J % 32;
    float *cb = colbuf + (J & 1) * NB;
    float *rb = rowbuf + (J & 1) * NB;
    if (warp == J / 8) {
#pragma unroll
      for (int a = 0; a < 4; ++a) cb[lane + 32 * a] = s[a][BJ];
    }
    if (lane == LJ) {
#pragma unroll
      for (int b = 0; b < 8; ++b) rb[8 * warp + b] = x[AJ][b];
    }
    __syncthreads();
    const float piv = cb[J];
    const bool okp = piv > 0.0f;  // false for NaN as well
    if (!okp && bad < 0) bad = J;
    const float rp = okp ? 1.0f / piv : 0.0f;
    const float rl = okp ? 1.0f / sqrtf(piv) : 0.0f;
    float ci[4];
#pragma unroll
    for (int a = 0; a < 4; ++a) ci[a] = cb[lane + 32 * a] * rp;
    if (8 * warp + 7 > J) {  // this warp still has unfinished columns l > J
      float cl[8];
#pragma unroll
      for (int b = 0; b < 8; ++b) cl[b] = cb[8 * warp + b];
#pragma unroll
      for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int b = 0; b < 8; ++b) {
          const int i = lane + 32 * a, l = 8 * warp + b;
          if (l > J && i >= l) s[a][b] = fmaf(-ci[a], cl[b], s[a][b]);
        }
    }
    if (8 * warp <= J) {  // B row J is zero beyond column J
      float rc[8];
#pragma unroll
      for (int b = 0; b < 8; ++b) rc[b] = rb[8 * warp + b];
#pragma unroll
      for (int a = 0; a < 4; ++a) {
        const int i = lane + 32 * a;
#pragma unroll
        for (int b = 0; b < 8; ++b) {
          if (i > J) x[a][b] = fmaf(-ci[a], rc[b], x[a][b]);
          else if (i == J) x[a][b] = rc[b] * rl;
        }
      }
    }
    PotrfStep<J + 1>::run(s, x, colbuf, rowbuf, warp, lane, bad);
  }
};
template <>
struct PotrfStep<NB> {
  static __device__ __forceinline__ void run(float (&)[4][8], float (&)[4][8], float *, float *,
                                             int, int, int &) {}
};

__global__ void __launch_bounds__(PF_THREADS)
potrf_kernel(const float *A, int64_t d, int64_t k0, int n, float *Linv, DevStatus *st) {
  __shared__ float colbuf[2 * NB], rowbuf[2 * NB];
  __shared__ int s_skip;
  if (threadIdx.x == 0) s_skip = st->status != 0;
  __syncthreads();
  if (s_skip) return;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  float s[4][8], x[4][8];
  const bool vec = (d % 4 == 0);
#pragma unroll
  for (int a = 0; a < 4; ++a) {
    const int i = lane + 32 * a;
    const float *row = A + (k0 + i) * d + k0 + 8 * warp;
    if (i < n && vec && 8 * warp + 8 <= n) {
      const float4 u = *reinterpret_cast<const float4 *>(row);
      const float4 v = *reinterpret_cast<const float4 *>(row + 4);
      s[a][0] = u.x; s[a][1] = u.y; s[a][2] = u.z; s[a][3] = u.w;
      s[a][4] = v.x; s[a][5] = v.y; s[a][6] = v.z; s[a][7] = v.w;
    } else {
#pragma unroll
      for (int b = 0; b < 8; ++b) s[a][b] = (i < n && 8 * warp + b < n) ? row[b] : 0.0f;
    }
#pragma unroll
    for (int b = 0; b < 8; ++b) {
      const int l = 8 * warp + b;
      if (i >= n || l >= n) s[a][b] = (i == l) ? 1.0f : 0.0f;  // identity padding
      x[a][b] = (i == l) ? 1.0f : 0.0f;
    }
  }
  int bad = -1;
  PotrfStep<0>::run(s, x, colbuf, rowbuf, warp, lane, bad);
  if (bad >= 0) {
    if (threadIdx.x == 0 && bad < n &&
        atomicCAS(&st->status, 0, (int)GPTQ_ERR_NOT_PD) == 0)
      st->info = (int)(k0 + bad) + 1;
    return;
  }
#pragma unroll
  for (int a = 0; a < 4; ++a) {
    const int i = lane + 32 * a;
#pragma unroll
    for (int b = 0; b < 8; ++b) {
      const int c = 8 * warp + b;
      Linv[i * NB + c] = (i < n && c < n) ? x[a][b] : 0.0f;
    }
  }
}

// ---------------------------------------------------------------------------------------
// Row-panel product: Out[r][j] = sum_{t<n} In[r][t] * Bm[j][t] for rows r in [r0, r1),
// j < n.  Each CTA owns whole rows, so Out may alias In.  Optionally also writes the
// TF32 head/tail split of Out into (hi, lo) panels (row r -> hi[r * NB + j]).
// ---------------------------------------------------------------------------------------
constexpr int RM_ROWS = 32, RM_THREADS = 256;

__global__ void __launch_bounds__(RM_THREADS)
rowmul_kernel(const float *In, int64_t ldi, float *Out, int64_t ldo, int64_t r0, int64_t r1,
              const float *Bm, int n, float *hi, float *lo, const DevStatus *st) {
  extern __shared__ float sm[];
  float *Bs = sm;                 // NB x LDS
  float *Is = sm + NB * LDS;      // RM_ROWS x LDS
  if (st->status != 0) return;
  const int tid = threadIdx.x;
  const int64_t rb = r0 + (int64_t)blockIdx.x * RM_ROWS;
#pragma unroll 16
  for (int it = 0; it < NB * NB / RM_THREADS; ++it) {
    const int e = it * RM_THREADS + tid;
    Bs[(e / NB) * LDS + e % NB] = Bm[e];
  }
#pragma unroll 16
  for (int it = 0; it < RM_ROWS * NB / RM_THREADS; ++it) {
    const int e = it * RM_THREADS + tid;
    const int r = e / NB, t = e % NB;
    const int64_t gr = rb + r;
    Is[r * LDS + t] = (gr < r1 && t < n) ? In[gr * ldi + t] : 0.0f;
  }
  __syncthreads();
  // thread -> row (tid / 8), 16 columns j = (tid % 8) + 8 * u
  const int r = tid / 8, jb = tid % 8;
  float acc[16];
#pragma unroll
  for (int u = 0; u < 16; ++u) acc[u] = 0.f;
  for (int t = 0; t < NB; ++t) {
    const float a = Is[r * LDS + t];
#pragma unroll
    for (int u = 0; u < 16; ++u) acc[u] = fmaf(a, Bs[(jb + 8 * u) * LDS + t], acc[u]);
  }
  const int64_t gr = rb + r;
  if (gr < r1) {
#pragma unroll
    for (int u = 0; u < 16; ++u) {
      const int j = jb + 8 * u;
      if (j < n) {
        if (Out) Out[gr * ldo + j] = acc[u];
        if (hi) {
          const float h = tf32_head(acc[u]);
          hi[gr * NB + j] = h;
          lo[gr * NB + j] = acc[u] - h;
        }
      } else if (hi) {
        hi[gr * NB + j] = 0.f;
        lo[gr * NB + j] = 0.f;
      }
    }
  }
}

// U[i][j] = Yt[d-1-j][d-1-i] for i <= j, 0 below the diagonal (32 x 32 smem tiles).
__global__ void assemble_u_kernel(const float *Yt, float *U, int64_t d) {
  __shared__ float tile[32][33];
  const int64_t i0 = (int64_t)blockIdx.y * 32, j0 = (int64_t)blockIdx.x * 32;
  const int tx = threadIdx.x, ty = threadIdx.y;  // 32 x 8
  // Tile of U rows [i0, i0+32), cols [j0, j0+32) reads Yt rows d-1-j, cols d-1-i.
  for (int yy = ty; yy < 32; yy += 8) {
    const int64_t j = j0 + yy, i = i0 + tx;
    float v = 0.f;
    if (i < d && j < d && i <= j) v = Yt[(d - 1 - j) * d + (d - 1 - i)];
    tile[yy][tx] = v;
  }
  __syncthreads();
  for (int yy = ty; yy < 32; yy += 8) {
    const int64_t i = i0 + yy, j = j0 + tx;
    if (i < d && j < d) U[i * d + j] = tile[tx][yy];
  }
}

struct PrepWs {
  DevStatus *st;
  float *Yt, *Lhi, *Llo, *Yhi, *Ylo, *Linv;
};

PrepWs carve_prepare(void *ws, int64_t d) {
  char *p = (char *)ws;
  PrepWs w;
  w.st = (DevStatus *)p;
  p += 256;
  w.Yt = (float *)p;  p += round_up((size_t)d * d * 4, 256);
  w.Lhi = (float *)p; p += round_up((size_t)d * NB * 4, 256);
  w.Llo = (float *)p; p += round_up((size_t)d * NB * 4, 256);
  w.Yhi = (float *)p; p += round_up((size_t)d * NB * 4, 256);
  w.Ylo = (float *)p; p += round_up((size_t)d * NB * 4, 256);
  w.Linv = (float *)p;
  return w;
}

}  // namespace

size_t prepare_ws_bytes(int64_t d) {
  return 256 + round_up((size_t)d * d * 4, 256) + 4 * round_up((size_t)d * NB * 4, 256) +
         round_up((size_t)NB * NB * 4, 256);
}

gptq_status launch_prepare(float *H, int64_t d, float damp, float *U, uint8_t *dead_mask,
                           void *ws, cudaStream_t s) {
  static bool attr_done = false;
  const size_t rm_smem = (NB + RM_ROWS) * LDS * sizeof(float);
  if (!attr_done) {
    GPTQ_CUDA_CHECK(cudaFuncSetAttribute(rowmul_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)rm_smem));
    attr_done = true;
  }
  PrepWs w = carve_prepare(ws, d);
  GPTQ_CUDA_CHECK(cudaMemsetAsync(w.st, 0, sizeof(DevStatus), s));
  dead_damp_kernel<<<1, 1024, 0, s>>>(H, d, damp, dead_mask, w.st);
  GPTQ_LAUNCH_CHECK();
  reverse_kernel<<<1024, 256, 0, s>>>(H, d * d, w.st);
  GPTQ_LAUNCH_CHECK();
  identity_kernel<<<1024, 256, 0, s>>>(w.Yt, d);
  GPTQ_LAUNCH_CHECK();
  float *A = H;  // reversed, damped Hessian; lower triangle is the Cholesky workspace
  for (int64_t k0 = 0; k0 < d; k0 += NB) {
    const int n = (int)std::min<int64_t>(NB, d - k0);
    const int64_t k1 = k0 + n;
    potrf_kernel<<<1, PF_THREADS, 0, s>>>(A, d, k0, n, w.Linv, w.st);
    GPTQ_LAUNCH_CHECK();
    // trsm: rows [k1, d) of panel k -> L panel (hi/lo) only (A's panel is not reused)
    if (k1 < d) {
      const unsigned g = (unsigned)ceil_div(d - k1, RM_ROWS);
      rowmul_kernel<<<g, RM_THREADS, rm_smem, s>>>(A + k0, d, nullptr, 0, k1, d, w.Linv, n,
                                                  w.Lhi, w.Llo, w.st);
      GPTQ_LAUNCH_CHECK();
    }
    // inv-a: Yt[c][k0:k1] = Bt[c][k0:k1] Linv^T for c in [0, k1), in place
    {
      const unsigned g = (unsigned)ceil_div(k1, RM_ROWS);
      rowmul_kernel<<<g, RM_THREADS, rm_smem, s>>>(w.Yt + k0, d, w.Yt + k0, d, 0, k1, w.Linv,
                                                  n, w.Yhi, w.Ylo, w.st);
      GPTQ_LAUNCH_CHECK();
    }
    if (k1 < d) {
      // syrk: A[k1:, k1:] -= Lp Lp^T (lower tiles)
      GemmArgs g{};
      g.a_hi = w.Lhi + k1 * NB; g.a_lo = w.Llo + k1 * NB; g.lda = NB;
      g.b_hi = w.Lhi + k1 * NB; g.b_lo = w.Llo + k1 * NB; g.ldb = NB;
      g.c = A + k1 * d + k1; g.ldc = d;
      g.M = d - k1; g.N = d - k1; g.K = n;
      g.alpha = -1.0f; g.lower_only = 1; g.trans_c = 0;
      GPTQ_TRY(launch_gemm_nt(g, w.st, s));
      // inv-b: Bt[c][k1:] -= Yp[c] Lp[k1:]^T for c < k1
      GemmArgs h{};
      h.a_hi = w.Yhi; h.a_lo = w.Ylo; h.lda = NB;
      h.b_hi = w.Lhi + k1 * NB; h.b_lo = w.Llo + k1 * NB; h.ldb = NB;
      h.c = w.Yt + k1; h.ldc = d;
      h.M = k1; h.N = d - k1; h.K = n;
      h.alpha = -1.0f; h.lower_only = 0; h.trans_c = 0;
      GPTQ_TRY(launch_gemm_nt(h, w.st, s));
    }
  }
  dim3 tg((unsigned)ceil_div(d, 32), (unsigned)ceil_div(d, 32));
  assemble_u_kernel<<<tg, dim3(32, 8), 0, s>>>(w.Yt, U, d);
  GPTQ_LAUNCH_CHECK();
  return GPTQ_OK;
}

}  // namespace gptq
