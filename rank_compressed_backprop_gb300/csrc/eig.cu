// eig.cu -- calibration solve of INSTANT (page "INSTANT: Compressing Gradients
// and Activations for Resource-Efficient Training", 关键设计 1 and 2):
//   C/n = U Sigma U^T (symmetric PSD: the SVD is the eigendecomposition),
//   E = ||C/n||_F^2, k = min{k : sum_{i<=k} sigma_i^2 >= eps E}, R = k + p,
//   rows = (sum_{i<=R} sigma_i^2)^(-1/2) U_R^T.
//
// Only the top R eigenpairs are needed.  L <= 128: one CTA runs a cyclic
// (round-robin parallel) Jacobi method on the whole matrix in shared memory.
// Larger L: block subspace iteration with a Rayleigh-Ritz step every
// iteration, as one cluster launch where the rows fit (k_solve_cluster below),
// otherwise as a host loop whose iterations are five launches:
//   orth   (1 CTA)  T = D W_G Lambda_G^(-1/2) from the Gram matrix of Z
//   apply  (grid)   V = Z T                         (orthonormal basis)
//   cv     (grid)   Y = C V / n,  H += V^T Y
//   rr     (1 CTA)  H = W Theta W^T  (Jacobi, sorted descending)
//   ritz   (grid)   U = V W, Z = Y W = C U / n, G += Z^T Z, res_j += |Z_j - theta_j U_j|^2
// Because U holds Ritz vectors, the columns of Z are nearly orthogonal with
// norms ~theta_j; normalising them with D before the Gram eigensolve keeps the
// fp32 orthonormalisation well conditioned.  The energy E is a fp64 sum over
// C itself (the iteration never sees the spectrum's tail), and the k rule runs
// in fp64.  Every loop is bounded; a Jacobi solve that hits its sweep cap
// records that in the result block instead of spinning.
#include <math.h>

#include "kernels.h"
#include "tc.cuh"

namespace instant {

namespace {

constexpr int kMaxBlock = 128;
constexpr int kJacThreads = 512;
constexpr int kRows = 32;  // rows of the tall matrices per CTA in grid kernels

__device__ __forceinline__ double warp_sum_d(double v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ float warp_sum_f(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// block-wide sum (blockDim.x a multiple of 32, <= 1024); every thread gets it
__device__ float block_sum_f(float v, float* red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  v = warp_sum_f(v);
  __syncthreads();
  if (lane == 0) red[warp] = v;
  __syncthreads();
  float t = 0.f;
  const int nw = blockDim.x >> 5;
  for (int i = 0; i < nw; ++i) t += red[i];
  return t;
}

// ---------------------------------------------------------------------------
// reset + energy
// ---------------------------------------------------------------------------
__global__ void k_solver_reset(SolverResult* r) {
  double* d = reinterpret_cast<double*>(r);
  for (int i = threadIdx.x; i < static_cast<int>(sizeof(SolverResult) / sizeof(double)); i += blockDim.x)
    d[i] = 0.0;
}

__global__ void k_solver_energy(const float* __restrict__ C, size_t count, SolverResult* r) {
  double acc = 0.0;
  int bad = 0;
  for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < count;
       i += static_cast<size_t>(gridDim.x) * blockDim.x) {
    const float v = C[i];
    if (!isfinite(v)) bad = 1;
    acc += static_cast<double>(v) * static_cast<double>(v);
  }
  acc = warp_sum_d(acc);
  __shared__ double red[32];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (lane == 0) red[warp] = acc;
  if (bad) r->nonfinite = 1;
  __syncthreads();
  if (threadIdx.x == 0) {
    double t = 0.0;
    for (int i = 0; i < static_cast<int>(blockDim.x >> 5); ++i) t += red[i];
    atomicAdd(&r->energy_sum, t);
  }
}

// ---------------------------------------------------------------------------
// cyclic Jacobi on a symmetric n x n matrix in shared memory (n <= 128).
// A[i*ld + j] with ld >= N = n rounded up to even; an odd n is padded with a
// zero row/column that never rotates.  V accumulates the rotations.
// Round-robin ordering: in each of the N-1 rounds the N/2 disjoint pairs are
// rotated together, and because the pairs are disjoint every 2x2 block
// A[{p,q},{p',q'}] <- J_k^T A J_k' is updated by one thread with no ordering
// between blocks (one barrier per round).  Rotation angle as in the classical
// symmetric 2x2 Schur decomposition (Golub & Van Loan, Matrix Computations,
// sec. 8.5): tau = (a_qq - a_pp) / (2 a_pq), t = sign(tau) /
// (|tau| + sqrt(1 + tau^2)), c = 1/sqrt(1 + t^2), s = t c.
// Stops when the off-diagonal mass falls below tol * ||A||_F, or when it
// stops shrinking (the fp32 rounding floor) below 1e-4 * ||A||_F; returns
// false when neither happens within max_sweeps.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void jac_pair(int r, int k, int N, int& p, int& q) {
  if (k == 0) {
    p = r;
    q = N - 1;
  } else {
    int a = r + k;
    if (a >= N - 1) a -= N - 1;
    int b = r - k;
    if (b < 0) b += N - 1;
    p = a < b ? a : b;
    q = a < b ? b : a;
  }
  if (p > q) {
    const int t = p;
    p = q;
    q = t;
  }
}

__device__ __forceinline__ void jac_rot(const float* A, int ld, int p, int q, float& c, float& s) {
  c = 1.f;
  s = 0.f;
  const float apq = A[p * ld + q];
  if (fabsf(apq) > 1e-30f) {
    const float app = A[p * ld + p], aqq = A[q * ld + q];
    const float tau = __fdividef(aqq - app, 2.f * apq);
    float t;
    if (fabsf(tau) > 1e18f) {
      t = __fdividef(0.5f, tau);
    } else {
      const float u = 1.f + tau * tau;
      t = copysignf(1.f, tau) * __fdividef(1.f, fabsf(tau) + u * rsqrtf(u));
    }
    c = rsqrtf(1.f + t * t);
    s = t * c;
  }
}

__device__ bool block_jacobi(float* A, float* A2, float* V, int n, int ld, float tol,
                             int max_sweeps, float* cs, int* pairs, float* red) {
  const int N = n + (n & 1);
  const int half = N / 2;
  for (int idx = threadIdx.x; idx < N * N; idx += blockDim.x) {
    const int i = idx / N, j = idx - (idx / N) * N;
    V[i * ld + j] = (i == j) ? 1.f : 0.f;
    if (i >= n || j >= n) A[i * ld + j] = 0.f;
  }
  __syncthreads();
  float* Ao = A;   // current matrix
  float* An = A2;  // next matrix
  bool converged = false;
  float prev = 0.f;
  for (int sweep = 0; sweep <= max_sweeps; ++sweep) {
    float off = 0.f, tot = 0.f;
    for (int idx = threadIdx.x; idx < n * n; idx += blockDim.x) {
      const int i = idx / n, j = idx - (idx / n) * n;
      const float v = Ao[i * ld + j];
      tot += v * v;
      if (i != j) off += v * v;
    }
    off = block_sum_f(off, red);
    tot = block_sum_f(tot, red);
    if (off <= tol * tol * tot || tot == 0.f) {
      converged = true;
      break;
    }
    if (sweep >= 3 && off > 0.25f * prev && off <= 1e-8f * tot) {
      converged = true;  // stagnating at the rounding floor
      break;
    }
    prev = off;
    if (sweep == max_sweeps) break;
    for (int r = 0; r < N - 1; ++r) {
      for (int k = threadIdx.x; k < half; k += blockDim.x) {
        int p, q;
        jac_pair(r, k, N, p, q);
        float c, sn;
        jac_rot(Ao, ld, p, q, c, sn);
        pairs[2 * k] = p;
        pairs[2 * k + 1] = q;
        cs[2 * k] = c;
        cs[2 * k + 1] = sn;
      }
      __syncthreads();
      // A' = J^T A J: disjoint 2x2 blocks, read from Ao, written to An
      for (int idx = threadIdx.x; idx < half * half; idx += blockDim.x) {
        const int k = idx / half, k2 = idx - (idx / half) * half;
        const int p = pairs[2 * k], q = pairs[2 * k + 1];
        const int p2 = pairs[2 * k2], q2 = pairs[2 * k2 + 1];
        const float c1 = cs[2 * k], s1 = cs[2 * k + 1];
        const float c2 = cs[2 * k2], s2 = cs[2 * k2 + 1];
        const float a = Ao[p * ld + p2], b = Ao[p * ld + q2];
        const float c = Ao[q * ld + p2], d = Ao[q * ld + q2];
        const float y00 = c1 * a - s1 * c, y01 = c1 * b - s1 * d;
        const float y10 = s1 * a + c1 * c, y11 = s1 * b + c1 * d;
        An[p * ld + p2] = c2 * y00 - s2 * y01;
        An[p * ld + q2] = s2 * y00 + c2 * y01;
        An[q * ld + p2] = c2 * y10 - s2 * y11;
        An[q * ld + q2] = s2 * y10 + c2 * y11;
      }
      // V <- V J (each item owns its two entries)
      for (int idx = threadIdx.x; idx < N * half; idx += blockDim.x) {
        const int k = idx / N, i = idx - (idx / N) * N;
        const float c = cs[2 * k], sn = cs[2 * k + 1];
        if (sn == 0.f) continue;
        const int p = pairs[2 * k], q = pairs[2 * k + 1];
        const float vp = V[i * ld + p], vq = V[i * ld + q];
        V[i * ld + p] = c * vp - sn * vq;
        V[i * ld + q] = sn * vp + c * vq;
      }
      __syncthreads();
      float* t = Ao;
      Ao = An;
      An = t;
    }
  }
  if (Ao != A) {
    for (int idx = threadIdx.x; idx < N * N; idx += blockDim.x) {
      const int i = idx / N, j = idx - (idx / N) * N;
      A[i * ld + j] = Ao[i * ld + j];
    }
  }
  __syncthreads();
  return converged;
}

// threads for a one-CTA Jacobi of order n: barriers are nearly free for a
// single warp, so small problems run on one warp
// threads of a full-Jacobi CTA: a round updates (N/2)^2 2x2 blocks and N^2/2
// entries of V, about 15 dependent shared-memory items a thread at 128 threads
// for N = 50; with 512 the round is shorter (the ViT-MLP statistics, L = 49:
// see the calibration notes)
__host__ __device__ inline int jac_threads(int n) {
  return n <= 24 ? 128 : 512;
}

// rank of diagonal entry i in descending order (ties: lower index first)
__device__ __forceinline__ int desc_rank(const float* A, int ld, int n, int i) {
  const float v = A[i * ld + i];
  int r = 0;
  for (int j = 0; j < n; ++j) {
    const float u = A[j * ld + j];
    r += (u > v) || (u == v && j < i);
  }
  return r;
}

struct JacSmem {
  float* A;
  float* A2;
  float* V;
  float* cs;
  int* pairs;
  float* red;
  int* rank;
};

__device__ JacSmem jac_carve(uint8_t* smem, int n) {
  JacSmem s;
  const int ld = n + 1;
  const int N = n + (n & 1);
  s.A = reinterpret_cast<float*>(smem);
  s.A2 = s.A + N * ld;
  s.V = s.A2 + N * ld;
  s.cs = s.V + N * ld;
  s.pairs = reinterpret_cast<int*>(s.cs + kMaxBlock + 2);
  s.red = reinterpret_cast<float*>(s.pairs + kMaxBlock + 2);
  s.rank = reinterpret_cast<int*>(s.red + 32);
  return s;
}

__host__ __device__ inline size_t jac_smem_bytes(int n) {
  const int ld = n + 1;
  const int N = n + (n & 1);
  return sizeof(float) * (3 * N * ld + kMaxBlock + 2 + 32) + sizeof(int) * (kMaxBlock + 2 + kMaxBlock);
}

// ---------------------------------------------------------------------------
// full Jacobi (L <= 128): theta (desc) -> res->theta, vectors -> U[:, rank]
// ---------------------------------------------------------------------------
__device__ __forceinline__ void jacobi_full(const float* __restrict__ C, int L, float inv_n,
                                            int max_sweeps, SolverWs w);

__global__ void __launch_bounds__(kJacThreads) k_jacobi_full(const float* __restrict__ C, int L,
                                                             float inv_n, int max_sweeps,
                                                             SolverWs w) {
  jacobi_full(C, L, inv_n, max_sweeps, w);
}

// one statistic per CTA
__global__ void __launch_bounds__(kJacThreads) k_jacobi_full_batch(const __grid_constant__ JacobiBatch b) {
  const int i = blockIdx.x;
  jacobi_full(b.C[i], b.L, b.inv_n[i], b.max_sweeps, b.w[i]);
}

__device__ __forceinline__ void jacobi_full(const float* __restrict__ C, int L, float inv_n,
                                            int max_sweeps, SolverWs w) {
  extern __shared__ uint8_t smem[];
  JacSmem s = jac_carve(smem, L);
  const int ld = L + 1;
  // a statistic whose energy is not finite and positive is not solved (the
  // caller reports it from the result block)
  __shared__ int s_skip;
  if (threadIdx.x == 0) s_skip = w.res->nonfinite || !(w.res->energy_sum > 0.0);
  __syncthreads();
  if (s_skip) return;
  for (int idx = threadIdx.x; idx < L * L; idx += blockDim.x) {
    const int i = idx / L, j = idx - (idx / L) * L;
    s.A[i * ld + j] = 0.5f * (C[i * L + j] + C[j * L + i]) * inv_n;
  }
  __syncthreads();
  const bool ok = block_jacobi(s.A, s.A2, s.V, L, ld, 3e-6f, max_sweeps, s.cs, s.pairs, s.red);
  for (int i = threadIdx.x; i < L; i += blockDim.x) s.rank[i] = desc_rank(s.A, ld, L, i);
  __syncthreads();
  for (int i = threadIdx.x; i < L; i += blockDim.x)
    w.res->theta[s.rank[i]] = static_cast<double>(s.A[i * ld + i]);
  for (int idx = threadIdx.x; idx < L * L; idx += blockDim.x) {
    const int row = idx / L, col = idx - (idx / L) * L;
    w.U[row * L + s.rank[col]] = s.V[row * ld + col];
  }
  if (threadIdx.x == 0) {
    if (!ok) w.res->jacobi_failed = 1;
    w.res->converged = ok ? 1 : 0;
  }
}

// ---------------------------------------------------------------------------
// subspace iteration kernels
// ---------------------------------------------------------------------------
__device__ __forceinline__ float hash_uniform(uint32_t i, uint32_t j) {
  // integer hash -> [-1, 1): deterministic starting block
  uint32_t h = i * 0x9E3779B1u ^ (j + 0x7F4A7C15u) * 0x85EBCA77u;
  h ^= h >> 15;
  h *= 0x2C1B3C6Du;
  h ^= h >> 12;
  h *= 0x297A2D39u;
  h ^= h >> 15;
  return static_cast<float>(h) * (2.0f / 4294967296.0f) - 1.0f;
}

// starting block: columns j < n_seed are the seed rows (a previous projector,
// row j = column j), the rest deterministic pseudo-random
__global__ void k_sub_init(int L, int m, const void* seed, int n_seed, int seed_bf16, SolverWs w) {
  if (blockIdx.x == 0)
    for (int i = threadIdx.x; i < 128; i += blockDim.x) w.res->res2_prev[i] = __int_as_float(0x7f800000);
  for (int idx = blockIdx.x * blockDim.x + threadIdx.x; idx < L * m; idx += gridDim.x * blockDim.x) {
    const int i = idx / m, j = idx - (idx / m) * m;
    float v = hash_uniform(i, j);
    if (j < n_seed) {
      const size_t o = static_cast<size_t>(j) * L + i;
      v = seed_bf16 ? bf16_to_f32(static_cast<const uint16_t*>(seed)[o])
                    : static_cast<const float*>(seed)[o];
    }
    w.Z[idx] = v;
  }
  for (int idx = blockIdx.x * blockDim.x + threadIdx.x; idx < m * m; idx += gridDim.x * blockDim.x) {
    w.G[idx] = 0.f;
    w.H[idx] = 0.f;
  }
}

// G += Z[rows]^T Z[rows]
__global__ void k_sub_gram(int L, int m, SolverWs w) {
  extern __shared__ float zs[];  // [kRows][m]
  const int i0 = blockIdx.x * kRows;
  const int nr = min(kRows, L - i0);
  for (int idx = threadIdx.x; idx < kRows * m; idx += blockDim.x) {
    const int r = idx / m;
    zs[idx] = r < nr ? w.Z[(i0 + r) * m + (idx - r * m)] : 0.f;
  }
  __syncthreads();
  for (int idx = threadIdx.x; idx < m * m; idx += blockDim.x) {
    const int a = idx / m, b = idx - (idx / m) * m;
    if (b < a) continue;
    float acc = 0.f;
    for (int r = 0; r < nr; ++r) acc = fmaf(zs[r * m + a], zs[r * m + b], acc);
    atomicAdd(&w.G[a * m + b], acc);
    if (a != b) atomicAdd(&w.G[b * m + a], acc);
  }
}

// T with Z T orthonormal, from the Gram matrix G = Z^T Z (m x m, row stride
// ldg), written to T (row stride ldt); the whole CTA takes part.
// Columns are first normalised (D = diag(G)^(-1/2)); the normalised Gram
// matrix of near-orthogonal Ritz directions is close to I, so a Cholesky
// factorisation D G D = L L^T is stable and T = D L^(-T).  When a pivot
// vanishes (Z rank deficient) the symmetric (Lowdin) form T = D W Lambda^(-1/2)
// from a Jacobi eigensolve is used instead; it zeroes the null directions.
// Returns false when that Jacobi solve hit its sweep cap.  G before the first Cholesky step and T is written last, so G and
// T may share storage.
__device__ bool orth_core(const float* G, int ldg, int m, int max_sweeps, JacSmem s, float* T,
                          int ldt, float* dsc, float* pv, int* deficient) {
  const int ld = m + 1;
  for (int i = threadIdx.x; i < m; i += blockDim.x) {
    const float g = G[i * ldg + i];
    dsc[i] = g > 0.f ? 1.f / sqrtf(g) : 0.f;
  }
  if (threadIdx.x == 0) *deficient = 0;
  __syncthreads();
  for (int idx = threadIdx.x; idx < m * m; idx += blockDim.x) {
    const int i = idx / m, j = idx - (idx / m) * m;
    s.A[i * ld + j] = 0.5f * (G[i * ldg + j] + G[j * ldg + i]) * dsc[i] * dsc[j];
  }
  __syncthreads();
  // ---- Cholesky (elimination form in V, so that A survives for the fallback):
  // step k subtracts a_ik a_jk / a_kk from the trailing block; column k is then
  // final and L = (column k) / sqrt(a_kk).  One barrier per step.
  float* Lc = s.V;
  for (int idx = threadIdx.x; idx < m * m; idx += blockDim.x) {
    const int i = idx / m, j = idx - (idx / m) * m;
    Lc[i * ld + j] = j <= i ? s.A[i * ld + j] : 0.f;
  }
  __syncthreads();
  for (int k = 0; k < m; ++k) {
    const float d = Lc[k * ld + k];
    if (!(d > 1e-6f)) {
      if (threadIdx.x == 0) *deficient = 1;
      break;
    }
    const int rem = m - k - 1;
    const float inv = 1.f / d;
    for (int idx = threadIdx.x; idx < rem * rem; idx += blockDim.x) {
      const int i = k + 1 + idx / rem, j = k + 1 + idx % rem;
      if (j <= i) Lc[i * ld + j] -= Lc[i * ld + k] * Lc[j * ld + k] * inv;
    }
    __syncthreads();
  }
  __syncthreads();
  if (!*deficient) {
    for (int j = threadIdx.x; j < m; j += blockDim.x) pv[j] = rsqrtf(Lc[j * ld + j]);
    __syncthreads();
    for (int idx = threadIdx.x; idx < m * m; idx += blockDim.x) {
      const int i = idx / m, j = idx - (idx / m) * m;
      if (j <= i) Lc[i * ld + j] *= pv[j];
    }
  }
  __syncthreads();
  if (!*deficient) {
    // T = D L^-T.  s.A is free now: X = L^-1 by forward substitution, one
    // thread per column j (each thread reads only the entries it wrote)
    for (int j = threadIdx.x; j < m; j += blockDim.x) {
      for (int i = 0; i < m; ++i) {
        float acc = i == j ? 1.f : 0.f;
        for (int k = j; k < i; ++k) acc -= Lc[i * ld + k] * s.A[k * ld + j];
        s.A[i * ld + j] = i < j ? 0.f : acc / Lc[i * ld + i];
      }
    }
    __syncthreads();
    // T[a][c] = D_a * (L^-T)[a][c] = D_a * X[c][a]
    for (int idx = threadIdx.x; idx < m * m; idx += blockDim.x) {
      const int a = idx / m, c = idx - (idx / m) * m;
      T[a * ldt + c] = dsc[a] * s.A[c * ld + a];
    }
    __syncthreads();
    return true;
  }
  // ---- fallback: symmetric orthonormalisation (A still holds D G D) ----
  const bool ok = block_jacobi(s.A, s.A2, s.V, m, ld, 1e-5f, max_sweeps, s.cs, s.pairs, s.red);
  float lmax = 0.f;
  for (int j = 0; j < m; ++j) lmax = fmaxf(lmax, s.A[j * ld + j]);
  for (int idx = threadIdx.x; idx < m * m; idx += blockDim.x) {
    const int a = idx / m, j = idx - (idx / m) * m;
    const float lam = s.A[j * ld + j];
    const float f = lam > 1e-10f * lmax ? 1.f / sqrtf(lam) : 0.f;
    T[a * ldt + j] = dsc[a] * s.V[a * ld + j] * f;
  }
  __syncthreads();
  return ok;
}

// 1 CTA: T from the Gram matrix G (see orth_core); zeroes G for the next step
__global__ void __launch_bounds__(kJacThreads) k_sub_orth(int m, int max_sweeps, SolverWs w) {
  pdl_launch_dependents();
  pdl_wait();
  extern __shared__ uint8_t smem[];
  JacSmem s = jac_carve(smem, m);
  __shared__ float dsc[kMaxBlock];
  __shared__ float pv[kMaxBlock];
  __shared__ int deficient;
  const bool ok = orth_core(w.G, m, m, max_sweeps, s, w.T, m, dsc, pv, &deficient);
  for (int idx = threadIdx.x; idx < m * m; idx += blockDim.x) w.G[idx] = 0.f;
  if (threadIdx.x == 0 && !ok) w.res->jacobi_failed = 1;
}

// out[rows] = in[rows] * M   (M m x m), rows of kRows per CTA
__global__ void k_sub_apply(const float* __restrict__ in, const float* __restrict__ M, float* out,
                            float* zero_rows, int L, int m) {
  pdl_launch_dependents();
  pdl_wait();
  extern __shared__ float sm[];
  float* Ms = sm;            // [m][m]
  float* rs = sm + m * m;    // [kRows][m]
  const int i0 = blockIdx.x * kRows;
  const int nr = min(kRows, L - i0);
  for (int idx = threadIdx.x; idx < m * m; idx += blockDim.x) Ms[idx] = M[idx];
  for (int idx = threadIdx.x; idx < kRows * m; idx += blockDim.x) {
    const int r = idx / m;
    rs[idx] = r < nr ? in[(i0 + r) * m + (idx - r * m)] : 0.f;
  }
  __syncthreads();
  for (int idx = threadIdx.x; idx < nr * m; idx += blockDim.x) {
    const int r = idx / m, j = idx - (idx / m) * m;
    float acc = 0.f;
    for (int k = 0; k < m; ++k) acc = fmaf(rs[r * m + k], Ms[k * m + j], acc);
    out[(i0 + r) * m + j] = acc;
    if (zero_rows) zero_rows[(i0 + r) * m + j] = 0.f;
  }
}

// Y += C[rows, js] V[js, :] / n over a (32-row x JB-column) block of C per
// CTA: one global round trip stages the C block and the matching V rows in
// shared memory, then each thread accumulates its outputs and adds them to Y
// (zeroed by the preceding apply step) with atomics.
constexpr int kCvRows = 32;
__global__ void __launch_bounds__(128) k_sub_cv(const float* __restrict__ C, int L, int m, int JB,
                                                float inv_n, SolverWs w) {
  pdl_launch_dependents();
  pdl_wait();
  extern __shared__ float sm[];
  const int ldc = JB + 1;
  float* cs = sm;                   // [kCvRows][JB + 1]
  float* vs = cs + kCvRows * ldc;   // [JB][m]
  const int i0 = blockIdx.x * kCvRows;
  const int j0 = blockIdx.y * JB;
  const int nr = min(kCvRows, L - i0);
  const int nj = min(JB, L - j0);
  for (int idx = threadIdx.x; idx < kCvRows * JB; idx += blockDim.x) {
    const int r = idx / JB, j = idx - (idx / JB) * JB;
    cs[r * ldc + j] = (r < nr && j < nj) ? C[static_cast<size_t>(i0 + r) * L + j0 + j] : 0.f;
  }
  for (int idx = threadIdx.x; idx < JB * m; idx += blockDim.x) {
    const int j = idx / m;
    vs[idx] = j < nj ? w.V[static_cast<size_t>(j0 + j) * m + (idx - j * m)] : 0.f;
  }
  __syncthreads();
  for (int o = threadIdx.x; o < nr * m; o += blockDim.x) {
    const int r = o / m, col = o - (o / m) * m;
    const float* crow = cs + r * ldc;
    float acc0 = 0.f, acc1 = 0.f;
    int j = 0;
    for (; j + 1 < nj; j += 2) {
      acc0 = fmaf(crow[j], vs[j * m + col], acc0);
      acc1 = fmaf(crow[j + 1], vs[(j + 1) * m + col], acc1);
    }
    if (j < nj) acc0 = fmaf(crow[j], vs[j * m + col], acc0);
    atomicAdd(&w.Y[static_cast<size_t>(i0 + r) * m + col], (acc0 + acc1) * inv_n);
  }
}

// H += V[rows]^T Y[rows] over chunks of 64 rows (H is zeroed by the previous
// Rayleigh-Ritz step and by the start of the iteration)
constexpr int kHRows = 64;
__global__ void __launch_bounds__(256) k_sub_h(int L, int m, SolverWs w) {
  pdl_launch_dependents();
  pdl_wait();
  extern __shared__ float sm[];
  float* vr = sm;               // [kHRows][m]
  float* yr = vr + kHRows * m;  // [kHRows][m]
  const int i0 = blockIdx.x * kHRows;
  const int nr = min(kHRows, L - i0);
  for (int idx = threadIdx.x; idx < kHRows * m; idx += blockDim.x) {
    const int r = idx / m, c = idx - (idx / m) * m;
    vr[idx] = r < nr ? w.V[static_cast<size_t>(i0 + r) * m + c] : 0.f;
    yr[idx] = r < nr ? w.Y[static_cast<size_t>(i0 + r) * m + c] : 0.f;
  }
  __syncthreads();
  for (int idx = threadIdx.x; idx < m * m; idx += blockDim.x) {
    const int a = idx / m, b = idx - (idx / m) * m;
    float h = 0.f;
#pragma unroll 8
    for (int r = 0; r < kHRows; ++r) h = fmaf(vr[r * m + a], yr[r * m + b], h);
    atomicAdd(&w.H[a * m + b], h);
  }
}

// 1 CTA: Rayleigh-Ritz on H -> W (columns sorted by descending theta), theta;
// zeroes H and the residual accumulators
__global__ void __launch_bounds__(kJacThreads) k_sub_rr(int m, int max_sweeps, float tol, SolverWs w) {
  pdl_launch_dependents();
  pdl_wait();
  extern __shared__ uint8_t smem[];
  JacSmem s = jac_carve(smem, m);
  const int ld = m + 1;
  for (int idx = threadIdx.x; idx < m * m; idx += blockDim.x) {
    const int i = idx / m, j = idx - (idx / m) * m;
    s.A[i * ld + j] = 0.5f * (w.H[i * m + j] + w.H[j * m + i]);
  }
  __syncthreads();
  for (int idx = threadIdx.x; idx < m * m; idx += blockDim.x) w.H[idx] = 0.f;
  const bool ok = block_jacobi(s.A, s.A2, s.V, m, ld, tol, max_sweeps, s.cs, s.pairs, s.red);
  for (int i = threadIdx.x; i < m; i += blockDim.x) s.rank[i] = desc_rank(s.A, ld, m, i);
  __syncthreads();
  for (int i = threadIdx.x; i < m; i += blockDim.x) {
    w.res->theta[s.rank[i]] = static_cast<double>(s.A[i * ld + i]);
    w.res->res2[i] = 0.f;
  }
  for (int idx = threadIdx.x; idx < m * m; idx += blockDim.x) {
    const int row = idx / m, col = idx - (idx / m) * m;
    w.W[row * m + s.rank[col]] = s.V[row * ld + col];
  }
  if (threadIdx.x == 0 && !ok) w.res->jacobi_failed = 1;
}

// U = V W, Z = Y W; G += Z^T Z; res2_j += |Z_j - theta_j U_j|^2 over this block's rows
__global__ void k_sub_ritz(int L, int m, SolverWs w) {
  pdl_launch_dependents();
  pdl_wait();
  extern __shared__ float sm[];
  float* Ws = sm;                 // [m][m]
  float* vs = Ws + m * m;         // [kRows][m]
  float* ys = vs + kRows * m;     // [kRows][m]
  float* us = ys + kRows * m;     // [kRows][m]
  float* zs = us + kRows * m;     // [kRows][m]
  __shared__ float th[kMaxBlock];
  const int i0 = blockIdx.x * kRows;
  const int nr = min(kRows, L - i0);
  for (int idx = threadIdx.x; idx < m * m; idx += blockDim.x) Ws[idx] = w.W[idx];
  for (int idx = threadIdx.x; idx < kRows * m; idx += blockDim.x) {
    const int r = idx / m, c = idx - (idx / m) * m;
    vs[idx] = r < nr ? w.V[(i0 + r) * m + c] : 0.f;
    ys[idx] = r < nr ? w.Y[(i0 + r) * m + c] : 0.f;
  }
  for (int j = threadIdx.x; j < m; j += blockDim.x) th[j] = static_cast<float>(w.res->theta[j]);
  __syncthreads();
  for (int idx = threadIdx.x; idx < kRows * m; idx += blockDim.x) {
    const int r = idx / m, j = idx - (idx / m) * m;
    float u = 0.f, z = 0.f;
    for (int k = 0; k < m; ++k) {
      const float wk = Ws[k * m + j];
      u = fmaf(vs[r * m + k], wk, u);
      z = fmaf(ys[r * m + k], wk, z);
    }
    us[idx] = u;
    zs[idx] = z;
    if (r < nr) {
      w.U[(i0 + r) * m + j] = u;
      w.Z[(i0 + r) * m + j] = z;
    }
  }
  __syncthreads();
  for (int j = threadIdx.x; j < m; j += blockDim.x) {
    float acc = 0.f;
    for (int r = 0; r < nr; ++r) {
      const float d = zs[r * m + j] - th[j] * us[r * m + j];
      acc = fmaf(d, d, acc);
    }
    atomicAdd(&w.res->res2[j], acc);
  }
  for (int idx = threadIdx.x; idx < m * m; idx += blockDim.x) {
    const int a = idx / m, b = idx - (idx / m) * m;
    if (b < a) continue;
    float acc = 0.f;
    for (int r = 0; r < nr; ++r) acc = fmaf(zs[r * m + a], zs[r * m + b], acc);
    atomicAdd(&w.G[a * m + b], acc);
    if (a != b) atomicAdd(&w.G[b * m + a], acc);
  }
}

// k rule in fp64: smallest k with sum_{i<=k} theta_i^2 >= eps * E; m + 1 if none
__device__ int k_rule(const double* theta, int m, double target) {
  double cum = 0.0;
  for (int i = 0; i < m; ++i) {
    cum += theta[i] * theta[i];
    if (cum >= target) return i + 1;
  }
  return m + 1;
}

// Convergence of Ritz pair i (used by both subspace-iteration paths).  Its
// eigenvector error is about residual / gap, so a residual that is small only
// against the largest Ritz value theta_1 leaves the trailing vectors of a
// decaying spectrum inaccurate.  A pair is converged when its residual is
// below kRitzRelTol * theta_i, or -- at the rounding floor of the fp32 C V
// product, which can lie above that for small theta_i -- when it is below
// tol * theta_1 and no longer shrinking (at least half the previous check's
// squared residual).
constexpr double kRitzRelTol = 1e-3;

__host__ __device__ inline bool ritz_converged(double r2, double r2_prev, double th_i, double th_1,
                                               double tol) {
  if (r2 <= kRitzRelTol * kRitzRelTol * th_i * th_i) return true;
  return r2 <= tol * tol * th_1 * th_1 && r2 >= 0.5 * r2_prev;
}

__global__ void k_sub_check(int L, int m, double eps, int p, int r_override, double tol,
                            double inv_n2, SolverWs w) {
  if (threadIdx.x != 0) return;
  SolverResult* r = w.res;
  const double E = r->energy_sum * inv_n2;
  const int k = k_rule(r->theta, m, eps * E);
  int R = r_override > 0 ? r_override : k + p;
  if (R > L) R = L;
  r->k = k;
  r->R = R;
  const bool fits = k <= m && R <= m - 1;
  r->block_short = fits ? 0 : 1;
  int conv = fits ? 1 : 0;
  const double th1 = r->theta[0];
  for (int i = 0; i < R && i < m && conv; ++i)
    if (!ritz_converged(r->res2[i], r->res2_prev[i], r->theta[i], th1, tol)) conv = 0;
  for (int i = 0; i < m; ++i) r->res2_prev[i] = r->res2[i];
  r->converged = conv;
}

__global__ void k_finalize(int L, int m, double eps, int p, int r_override, int scale_on,
                           void* rows_out, int r_cap, int out_bf16, double inv_n2, SolverWs w) {
  __shared__ int sR;
  __shared__ float ss;
  SolverResult* r = w.res;
  // no projector from a statistic whose energy is not finite and positive
  if (r->nonfinite || !(r->energy_sum > 0.0)) return;
  if (threadIdx.x == 0) {
    const double E = r->energy_sum * inv_n2;
    int k = k_rule(r->theta, m, eps * E);
    if (k > L) k = L;
    int R = r_override > 0 ? r_override : k + p;
    if (R > L) R = L;
    if (R > m) R = m;
    double cum = 0.0;
    for (int i = 0; i < R; ++i) cum += r->theta[i] * r->theta[i];
    const double s = scale_on ? 1.0 / sqrt(cum) : 1.0;
    r->k = k;
    r->R = R;
    r->scale = static_cast<float>(s);
    sR = R;
    ss = static_cast<float>(s);
  }
  __syncthreads();
  const int R = sR;
  const float s = ss;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  for (int i = warp; i < r_cap; i += nw) {
    float sign = 1.f;
    if (i < R) {
      // argmax |u_j| with the lowest index on ties
      float best = -1.f;
      int bidx = 0x7fffffff;
      for (int j = lane; j < L; j += 32) {
        const float a = fabsf(w.U[j * m + i]);
        if (a > best || (a == best && j < bidx)) {
          best = a;
          bidx = j;
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float ob = __shfl_xor_sync(0xffffffffu, best, o);
        const int oi = __shfl_xor_sync(0xffffffffu, bidx, o);
        if (ob > best || (ob == best && oi < bidx)) {
          best = ob;
          bidx = oi;
        }
      }
      sign = w.U[bidx * m + i] < 0.f ? -1.f : 1.f;
    }
    for (int j = lane; j < L; j += 32) {
      const float v = i < R ? s * sign * w.U[j * m + i] : 0.f;
      if (out_bf16)
        static_cast<uint16_t*>(rows_out)[static_cast<size_t>(i) * L + j] = bf16_bits(v);
      else
        static_cast<float*>(rows_out)[static_cast<size_t>(i) * L + j] = v;
    }
  }
}

// ---------------------------------------------------------------------------
// whole subspace iteration in one launch: a cluster of 8 CTAs (128 < L, block
// m <= 32, while the CTA's rows fit in shared memory: L <= 2048 for m = 32).
// CTA q owns rows [q*rp, (q+1)*rp) of every tall matrix and streams the same
// rows of C for Y = C V / n.  Up to L = 512 it gathers the rest of V from its
// peers' shared memory; beyond that the basis no longer fits next to the
// CTA's rows, so every CTA publishes its rows of V in the solver workspace and
// streams V tiles from L2 along with the C tiles.  The m x m steps (Rayleigh-Ritz Jacobi, Cholesky-QR,
// convergence test) run in every CTA on partial sums that each CTA adds in
// rank order, so all CTAs hold identical copies; the decision to stop is
// still taken from rank 0 so that every CTA leaves the loop together.
// ---------------------------------------------------------------------------
__device__ __forceinline__ float dsmem_ld_f32(uint32_t addr) {
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
  return v;
}
__device__ __forceinline__ double dsmem_ld_f64(uint32_t addr) {
  double v;
  asm volatile("ld.shared::cluster.f64 %0, [%1];" : "=d"(v) : "r"(addr) : "memory");
  return v;
}
__device__ __forceinline__ int dsmem_ld_s32(uint32_t addr) {
  int v;
  asm volatile("ld.shared::cluster.s32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
  return v;
}

// Rotation annihilating a_pq of a symmetric 2x2 block, branch-free:
// theta = a_qq - a_pp, t = sign(theta) 2 a_pq / (|theta| + sqrt(theta^2 + 4 a_pq^2))
// (the smaller root of the classical tangent equation, Golub & Van Loan
// sec. 8.5, multiplied through by |2 a_pq|), c = 1 / sqrt(1 + t^2), s = t c.
__device__ __forceinline__ void jac_rot_bf(float app, float aqq, float apq, float& c, float& s) {
  const float th = aqq - app;
  const float two = 2.f * apq;
  const float r2 = fmaf(th, th, two * two);
  const float r = r2 * rsqrtf(fmaxf(r2, 1e-38f));
  float t = __fdividef(copysignf(1.f, th) * two, fabsf(th) + r);
  t = fabsf(apq) > 1e-30f ? t : 0.f;
  c = rsqrtf(fmaf(t, t, 1.f));
  s = t * c;
}

// Jacobi of order M (even, <= 32) for the whole CTA: per round, the M/2
// rotations are computed once (one thread each), then the disjoint 2x2 blocks
// of A' = J^T A J (double-buffered in A/A2) and the pairs of columns of V J
// are updated.  Round-robin ordering and stopping rule as block_jacobi.
template <int M>
__device__ bool jacobi_fast(float* A, float* A2, float* V, int ld, float tol, int max_sweeps,
                            float* red, float* cs) {
  constexpr int H = M / 2;
  const int tid = threadIdx.x, nthr = blockDim.x;
  for (int idx = tid; idx < M * M; idx += nthr) {
    const int i = idx / M, j = idx % M;
    V[i * ld + j] = (i == j) ? 1.f : 0.f;
  }
  __syncthreads();
  float* Ao = A;
  float* An = A2;
  bool converged = false;
  float prev = 0.f;
  for (int sweep = 0; sweep <= max_sweeps; ++sweep) {
    float off = 0.f, tot = 0.f;
    for (int idx = tid; idx < M * M; idx += nthr) {
      const int i = idx / M, j = idx % M;
      const float v = Ao[i * ld + j];
      tot += v * v;
      if (i != j) off += v * v;
    }
    off = block_sum_f(off, red);
    tot = block_sum_f(tot, red);
    if (off <= tol * tol * tot || tot == 0.f) {
      converged = true;
      break;
    }
    if (sweep >= 3 && off > 0.25f * prev && off <= 1e-8f * tot) {
      converged = true;
      break;
    }
    prev = off;
    if (sweep == max_sweeps) break;
    for (int r = 0; r < M - 1; ++r) {
      if (tid < H) {
        int p, q;
        jac_pair(r, tid, M, p, q);
        float c, sn;
        jac_rot_bf(Ao[p * ld + p], Ao[q * ld + q], Ao[p * ld + q], c, sn);
        cs[2 * tid] = c;
        cs[2 * tid + 1] = sn;
      }
      __syncthreads();
      for (int idx = tid; idx < H * H; idx += nthr) {
        const int k = idx / H, k2 = idx % H;
        int p, q, p2, q2;
        jac_pair(r, k, M, p, q);
        jac_pair(r, k2, M, p2, q2);
        const float c1 = cs[2 * k], s1 = cs[2 * k + 1];
        const float c2 = cs[2 * k2], s2 = cs[2 * k2 + 1];
        const float a = Ao[p * ld + p2], b = Ao[p * ld + q2];
        const float c = Ao[q * ld + p2], d = Ao[q * ld + q2];
        const float y00 = c1 * a - s1 * c, y01 = c1 * b - s1 * d;
        const float y10 = s1 * a + c1 * c, y11 = s1 * b + c1 * d;
        An[p * ld + p2] = c2 * y00 - s2 * y01;
        An[p * ld + q2] = s2 * y00 + c2 * y01;
        An[q * ld + p2] = c2 * y10 - s2 * y11;
        An[q * ld + q2] = s2 * y10 + c2 * y11;
      }
      for (int idx = tid; idx < M * H; idx += nthr) {
        const int k = idx / M, i = idx % M;
        const float c = cs[2 * k], sn = cs[2 * k + 1];
        if (sn == 0.f) continue;
        int p, q;
        jac_pair(r, k, M, p, q);
        const float vp = V[i * ld + p], vq = V[i * ld + q];
        V[i * ld + p] = c * vp - sn * vq;
        V[i * ld + q] = sn * vp + c * vq;
      }
      __syncthreads();
      float* t = Ao;
      Ao = An;
      An = t;
    }
  }
  if (Ao != A) {
    for (int idx = tid; idx < M * M; idx += nthr) {
      const int i = idx / M, j = idx % M;
      A[i * ld + j] = Ao[i * ld + j];
    }
  }
  __syncthreads();
  return converged;
}

// Cholesky factor of the column-normalised Gram matrix: D = diag(G)^(-1/2)
// into dsc, L (lower, D G D = L L^T) into Lf.  Whole CTA, one barrier per
// column.  Returns false (uniformly) when a pivot vanishes; G is only read.
template <int M>
__device__ bool chol_block(const float* G, int ld, float* Lf, float* dsc, float* pv, int* flag) {
  const int tid = threadIdx.x, nthr = blockDim.x;
  for (int i = tid; i < M; i += nthr) {
    const float g = G[i * ld + i];
    dsc[i] = g > 0.f ? 1.f / sqrtf(g) : 0.f;
  }
  if (tid == 0) *flag = 0;
  __syncthreads();
  for (int idx = tid; idx < M * M; idx += nthr) {
    const int i = idx / M, j = idx % M;
    Lf[i * ld + j] = j <= i ? 0.5f * (G[i * ld + j] + G[j * ld + i]) * dsc[i] * dsc[j] : 0.f;
  }
  __syncthreads();
  for (int k = 0; k < M; ++k) {
    const float d = Lf[k * ld + k];
    if (!(d > 1e-6f)) {
      if (tid == 0) *flag = 1;
      break;
    }
    const float inv = 1.f / d;
    for (int idx = tid; idx < M * M; idx += nthr) {
      const int i = idx / M, j = idx % M;
      if (k < j && j <= i) Lf[i * ld + j] -= Lf[i * ld + k] * Lf[j * ld + k] * inv;
    }
    __syncthreads();
  }
  __syncthreads();
  if (*flag) return false;
  for (int j = tid; j < M; j += nthr) pv[j] = rsqrtf(Lf[j * ld + j]);
  __syncthreads();
  for (int idx = tid; idx < M * M; idx += nthr) {
    const int i = idx / M, j = idx % M;
    if (j <= i) Lf[i * ld + j] *= pv[j];
  }
  __syncthreads();
  return true;
}

// error-free sum of two floats (Knuth's two-sum): a + b = s + e exactly
__device__ __forceinline__ void two_sum(float a, float b, float& s, float& e) {
  s = a + b;
  const float bb = s - a;
  e = (a - (s - bb)) + (b - bb);
}

// one exact square added to a double-float (hi, lo) accumulator
__device__ __forceinline__ void add_square(float v, float& hi, float& lo, int& bad) {
  if (!isfinite(v)) bad = 1;
  const float sq = v * v;
  const float sq_err = fmaf(v, v, -sq);
  float sum, err;
  two_sum(hi, sq, sum, err);
  hi = sum;
  lo += err + sq_err;
}

constexpr int kCvTileRows = 64;  // rows of C per staged tile
constexpr int kCvTileL = 64;     // columns of C per staged tile
constexpr int kCvTileLd = 68;    // padded row stride: 16-byte rows, conflict-free column reads

// stage columns [t * 64, t * 64 + 64) of the CTA's rows of C into a tile
__device__ __forceinline__ void stage_c_tile(float* dst, const float* Cown, int nr, int L, int t,
                                             bool vec) {
  const int l0 = t * kCvTileL;
  for (int i = threadIdx.x; i < kCvTileRows * (kCvTileL / 4); i += blockDim.x) {
    const int rr = i / (kCvTileL / 4), c4 = (i - rr * (kCvTileL / 4)) * 4;
    float* d = dst + rr * kCvTileLd + c4;
    if (vec && rr < nr && l0 + c4 + 4 <= L) {
      cp_async16(d, Cown + static_cast<size_t>(rr) * L + l0 + c4);
    } else {
      for (int e = 0; e < 4; ++e)
        d[e] = (rr < nr && l0 + c4 + e < L) ? Cown[static_cast<size_t>(rr) * L + l0 + c4 + e] : 0.f;
    }
  }
  cp_async_commit();
}

constexpr int kClusterCtas = 8;  // CTAs of a solver cluster (16 above 1024 tokens)
constexpr int kClusterThreads = 256;

// cluster size of the one-launch solver: 16 CTAs (a non-portable cluster) for
// long token axes, where the row-parallel steps dominate (a warm two-iteration
// solve at L = 2048 took 0.51 ms against 0.63 ms with 8); 8 below, where the
// replicated m x m steps and the cluster barriers dominate (L = 300: 0.28 ms
// with 8 against 0.34 ms with 16)
__host__ __device__ inline int cluster_ctas(int L) { return L > 1024 ? 16 : kClusterCtas; }

// Long token axes: Y = C V over all of the CTA's rows at once (see cv_big);
// C and V arrive in 16-token chunks through a 4-deep cp.async ring.
constexpr int kCvBigK = 16;       // tokens per chunk
constexpr int kCvBigLd = 20;      // padded row stride of a C chunk: 16-byte rows, conflict-free
constexpr int kCvBigStages = 4;
constexpr int kCvBigRows = 256;   // rows of a C chunk: the CTA's rows (L <= 8 * 256)

// stage tokens [t * 16, t * 16 + 16) of the CTA's nr rows of C and of V [L, m]
// into one ring slot; tokens past L are zero in both (an empty group past the end)
__device__ __forceinline__ void stage_cv_chunk(float* cdst, float* vdst, const float* Cown, int nr,
                                               const float* V, int L, int m, int t, bool vec) {
  const int l0 = t * kCvBigK;
  if (l0 < L) {
    constexpr int q = kCvBigK / 4;
    for (int i = threadIdx.x; i < nr * q; i += blockDim.x) {
      const int rr = i / q, c4 = (i - rr * q) * 4;
      float* d = cdst + rr * kCvBigLd + c4;
      const float* s = Cown + static_cast<size_t>(rr) * L + l0 + c4;
      if (vec && l0 + c4 + 4 <= L) {
        cp_async16(d, s);
      } else {
        for (int e = 0; e < 4; ++e) d[e] = l0 + c4 + e < L ? s[e] : 0.f;
      }
    }
    const int q4 = m / 4;
    for (int i = threadIdx.x; i < kCvBigK * q4; i += blockDim.x) {
      const int rr = i / q4, c4 = (i - rr * q4) * 4;
      float* d = vdst + rr * m + c4;
      if (l0 + rr < L) {
        cp_async16(d, V + static_cast<size_t>(l0 + rr) * m + c4);
      } else {
        d[0] = d[1] = d[2] = d[3] = 0.f;
      }
    }
  }
  cp_async_commit();
}

// Y[r, :] = C[own row r, :] V / n for the CTA's nr rows.  The CTA's threads
// form two halves, each taking 8 of a chunk's 16 tokens; thread (slot, cg) of
// a half owns rows slot + i * slots (i < RB) and columns [8 cg, 8 cg + 8), so
// per 4 tokens RB 16-byte loads of C and 8 of V feed 32 RB FMAs.  The halves'
// sums meet in the idle ring at the end.  V is read from the workspace where
// every CTA of the cluster published its rows.
template <int M, int RB>
__device__ __forceinline__ void cv_big(const float* Cown, int nr, const float* Vg, int L, bool vec,
                                       float* Cs, float* Vs, float* Y, float inv_n) {
  constexpr int NH = kClusterThreads / 2;  // threads of a half
  constexpr int ncg = M / 8;
  constexpr int slots = NH / ncg;
  constexpr int cstage = kCvBigRows * kCvBigLd, vstage = kCvBigK * M;
  const int half = threadIdx.x / NH;
  const int t = threadIdx.x - half * NH;
  const int cg = t % ncg, slot = t / ncg;
  float acc[RB][8];
#pragma unroll
  for (int i = 0; i < RB; ++i)
#pragma unroll
    for (int c = 0; c < 8; ++c) acc[i][c] = 0.f;
  const int nch = (L + kCvBigK - 1) / kCvBigK;
  for (int s = 0; s < kCvBigStages - 1; ++s)
    stage_cv_chunk(Cs + s * cstage, Vs + s * vstage, Cown, nr, Vg, L, M, s, vec);
  for (int t2 = 0; t2 < nch; ++t2) {
    cp_async_wait<kCvBigStages - 2>();  // chunk t2's group (this thread's copies) has landed
    __syncthreads();                    // ... everyone's; the slot of chunk t2 - 1 is free
    {
      const int s = t2 + kCvBigStages - 1;
      const int b = s % kCvBigStages;
      stage_cv_chunk(Cs + b * cstage, Vs + b * vstage, Cown, nr, Vg, L, M, s, vec);
    }
    const int b = t2 % kCvBigStages;
    const float* cb = Cs + b * cstage + slot * kCvBigLd + half * (kCvBigK / 2);
    const float* vb = Vs + b * vstage + half * (kCvBigK / 2) * M + cg * 8;
#pragma unroll
    for (int k4 = 0; k4 < kCvBigK / 2; k4 += 4) {
      float4 c[RB];
#pragma unroll
      for (int i = 0; i < RB; ++i) c[i] = *reinterpret_cast<const float4*>(cb + i * slots * kCvBigLd + k4);
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        const float4 v0 = *reinterpret_cast<const float4*>(vb + (k4 + kk) * M);
        const float4 v1 = *reinterpret_cast<const float4*>(vb + (k4 + kk) * M + 4);
#pragma unroll
        for (int i = 0; i < RB; ++i) {
          const float cv = kk == 0 ? c[i].x : (kk == 1 ? c[i].y : (kk == 2 ? c[i].z : c[i].w));
          acc[i][0] = fmaf(cv, v0.x, acc[i][0]);
          acc[i][1] = fmaf(cv, v0.y, acc[i][1]);
          acc[i][2] = fmaf(cv, v0.z, acc[i][2]);
          acc[i][3] = fmaf(cv, v0.w, acc[i][3]);
          acc[i][4] = fmaf(cv, v1.x, acc[i][4]);
          acc[i][5] = fmaf(cv, v1.y, acc[i][5]);
          acc[i][6] = fmaf(cv, v1.z, acc[i][6]);
          acc[i][7] = fmaf(cv, v1.w, acc[i][7]);
        }
      }
    }
  }
  cp_async_wait<0>();  // the empty groups past the end
  __syncthreads();     // the ring is idle: the second half parks its sums there
  float* red = Cs;     // [RB * 8][NH]
  if (half == 1) {
#pragma unroll
    for (int i = 0; i < RB; ++i)
#pragma unroll
      for (int c = 0; c < 8; ++c) red[(i * 8 + c) * NH + t] = acc[i][c];
  }
  __syncthreads();
  if (half == 0) {
#pragma unroll
    for (int i = 0; i < RB; ++i) {
      const int r = slot + i * slots;
      if (r < nr)
#pragma unroll
        for (int c = 0; c < 8; ++c) Y[r * M + cg * 8 + c] = (acc[i][c] + red[(i * 8 + c) * NH + t]) * inv_n;
    }
  }
  __syncthreads();  // the ring is free for the next iteration's prologue
}

// row stride of the resident C rows: 4 mod 32 words, so that the eight rows a
// warp reads at one column fall in distinct banks; rows stay 16-byte aligned
__host__ __device__ inline int cres_ld(int L) { return (L + 31) / 32 * 32 + 4; }

// sum over the CTAS CTAs of the cluster of the float at `p` (the same shared
// address in every CTA), in rank order; every load is issued before the adds
template <int CTAS>
__device__ __forceinline__ float cluster_sum(const float* p) {
  float v[CTAS];
#pragma unroll
  for (int q = 0; q < CTAS; ++q) v[q] = dsmem_ld_f32(dsmem_addr(p, q));
  float t = v[0];
#pragma unroll
  for (int q = 1; q < CTAS; ++q) t += v[q];
  return t;
}

struct ClusterLay {
  uint32_t V, Y, Hp, Gp, resp, r2, W, T, Lf, th, dpart, ipart, aval, aidx, flag, dsc, pv, jac,
      vt, ct, total;
};

__host__ __device__ inline uint32_t lay_take(uint32_t& o, size_t bytes) {
  const uint32_t r = o;
  o = static_cast<uint32_t>((o + bytes + 15u) & ~static_cast<size_t>(15u));
  return r;
}

// Above this token length the whole basis no longer fits next to the CTA's
// rows: each CTA keeps only its own rows of V and publishes them through the
// solver workspace, and C V streams tiles of C and of V from L2.
constexpr int kClusterGatherMaxL = 512;

__host__ __device__ inline ClusterLay cluster_layout(int L, int m, int rp) {
  ClusterLay c;
  uint32_t o = 0;
  const bool big = L > kClusterGatherMaxL;
  // the whole basis, gathered each iteration (own rows only for long L)
  c.V = lay_take(o, 4u * (big ? rp : L) * m);
  // own rows of Y = C V / n, overwritten in place by Z = Y W (the next block);
  // the Ritz vectors U = V W overwrite the own rows of V in the same way
  c.Y = lay_take(o, 4u * rp * m);
  c.Hp = lay_take(o, 4u * m * m);      // partial V^T Y (read by the peers)
  c.Gp = lay_take(o, 4u * m * m);      // partial Z^T Z (read by the peers)
  c.resp = lay_take(o, 4u * m);        // partial residual norms (read by the peers)
  c.r2 = lay_take(o, 4u * m);          // summed residual norms
  c.W = lay_take(o, 4u * m * (m + 1)); // Ritz rotation, columns by descending theta
  c.T = lay_take(o, 4u * m * (m + 1)); // summed Gram matrix; Z -> V transform on the fallback
  c.Lf = lay_take(o, 4u * m * (m + 1)); // Cholesky factor of the normalised Gram matrix
  c.th = lay_take(o, 8u * m);          // Ritz values (descending)
  c.dpart = lay_take(o, 8u);           // partial energy (read by the peers)
  c.ipart = lay_take(o, 16u);          // partial non-finite flag (read by the peers)
  c.aval = lay_take(o, 4u * m);        // per column: entry of largest magnitude (peers)
  c.aidx = lay_take(o, 4u * m);        // ... and its row (peers)
  c.flag = lay_take(o, 16u);           // rank 0's decision (read by the peers)
  c.dsc = lay_take(o, 4u * kMaxBlock);
  c.pv = lay_take(o, 4u * kMaxBlock);
  c.jac = lay_take(o, jac_smem_bytes(m));
  if (big) {
    // the ring of C and V chunks for Y = C V
    c.ct = lay_take(o, 4u * kCvBigStages * kCvBigRows * kCvBigLd);
    c.vt = lay_take(o, 4u * kCvBigStages * kCvBigK * m);
  } else if (m == 16) {
    // the CTA's rows of C stay in shared memory for the whole solve
    c.ct = lay_take(o, 4u * rp * cres_ld(L));
  } else {
    c.ct = lay_take(o, 4u * 2 * kCvTileRows * kCvTileLd);  // two C tiles for Y = C V
  }
  if (!big) c.vt = o;
  c.total = o;
  return c;
}

template <int M, int CTAS>
__global__ void __launch_bounds__(kClusterThreads, 1)
    k_solve_cluster(const __grid_constant__ ClusterSolveBatch batch) {
  extern __shared__ __align__(16) uint8_t csm[];
  const ClusterSolveArgs& a = batch.s[blockIdx.y];  // one statistic per cluster
  constexpr int m = M;
  const int L = a.L, rp = a.rp;
  const ClusterLay lay = cluster_layout(L, m, rp);
  float* Vall = reinterpret_cast<float*>(csm + lay.V);
  float* Y = reinterpret_cast<float*>(csm + lay.Y);
  float* Z = Y;  // Z = Y W replaces Y in place
  float* Hp = reinterpret_cast<float*>(csm + lay.Hp);
  float* Gp = reinterpret_cast<float*>(csm + lay.Gp);
  float* resp = reinterpret_cast<float*>(csm + lay.resp);
  float* r2 = reinterpret_cast<float*>(csm + lay.r2);
  float* W = reinterpret_cast<float*>(csm + lay.W);
  float* T = reinterpret_cast<float*>(csm + lay.T);
  float* Lf = reinterpret_cast<float*>(csm + lay.Lf);
  double* th = reinterpret_cast<double*>(csm + lay.th);
  double* dpart = reinterpret_cast<double*>(csm + lay.dpart);
  int* ipart = reinterpret_cast<int*>(csm + lay.ipart);
  float* aval = reinterpret_cast<float*>(csm + lay.aval);
  int* aidx = reinterpret_cast<int*>(csm + lay.aidx);
  int* flag = reinterpret_cast<int*>(csm + lay.flag);
  float* dsc = reinterpret_cast<float*>(csm + lay.dsc);
  float* pv = reinterpret_cast<float*>(csm + lay.pv);
  JacSmem js = jac_carve(csm + lay.jac, m);
  float* Ct = reinterpret_cast<float*>(csm + lay.ct);
  float* Vt = reinterpret_cast<float*>(csm + lay.vt);
  const bool big = L > kClusterGatherMaxL;
  __shared__ double s_E;
  __shared__ int s_bad, s_dec, s_jfail, s_deficient, s_cflag, s_useT, s_k, s_R;
  __shared__ float s_scale;
  __shared__ double wred[kClusterThreads / 32];
  __shared__ float s_r2prev[M];  // rank 0: squared residuals at the previous check
  for (int i = threadIdx.x; i < M; i += blockDim.x) s_r2prev[i] = __int_as_float(0x7f800000);

  const int tid = threadIdx.x;
  const int nthr = blockDim.x;
  const int rank = blockIdx.z;  // == rank in the cluster (dims 1 x 1 x 8)
  const int r0 = rank * rp;
  const int nr = min(rp, L - r0);  // >= 1 for 128 < L (host guarantees rp * 7 < L)
  constexpr int ld = m + 1;
  const float* Cown = a.C + static_cast<size_t>(r0) * L;

  const bool kResident = (M == 16) && !big;
  const bool vecC = (L & 3) == 0 && (reinterpret_cast<uintptr_t>(a.C) & 15) == 0;
  if (kResident) {
    // load the own rows of C once (cp.async when rows are 16-byte aligned)
    const int ldc = cres_ld(L);
    const int l4 = (L + 3) / 4;
    for (int i = tid; i < nr * l4; i += nthr) {
      const int r = i / l4, c4 = (i - r * l4) * 4;
      float* d = Ct + r * ldc + c4;
      if (vecC && c4 + 4 <= L) {
        cp_async16(d, Cown + static_cast<size_t>(r) * L + c4);
      } else {
        for (int e = 0; e < 4; ++e) d[e] = c4 + e < L ? Cown[static_cast<size_t>(r) * L + c4 + e] : 0.f;
      }
    }
    cp_async_commit();
    cp_async_wait<0>();
    __syncthreads();
  }
  // ---- energy ||C||_F^2 and finiteness, summed over the cluster ----
  if (kResident) {
    float hi = 0.f, lo = 0.f;
    int bad = 0;
    const int ldc = cres_ld(L);
    // warp w takes rows w, w + 8, ...; its lanes stride along the row
    for (int r = tid >> 5; r < nr; r += nthr >> 5)
#pragma unroll 4
      for (int l = tid & 31; l < L; l += 32) add_square(Ct[r * ldc + l], hi, lo, bad);
    double acc = static_cast<double>(hi) + static_cast<double>(lo);
    acc = warp_sum_d(acc);
    bad = __syncthreads_or(bad);
    if ((tid & 31) == 0) wred[tid >> 5] = acc;
    __syncthreads();
    if (tid == 0) {
      double t = 0.0;
      for (int i = 0; i < nthr / 32; ++i) t += wred[i];
      dpart[0] = t;
      ipart[0] = bad;
      s_jfail = 0;
    }
  } else {
    // per thread a double-float (hi, lo) sum of exact squares: fp32 arithmetic
    // only (fp64 units are scarce), about fp64 accuracy
    float hi = 0.f, lo = 0.f;
    int bad = 0;
    const int count = nr * L;
    if ((count & 3) == 0 && (reinterpret_cast<uintptr_t>(Cown) & 15) == 0) {
      const float4* c4 = reinterpret_cast<const float4*>(Cown);
#pragma unroll 8
      for (int i = tid; i < count / 4; i += nthr) {
        const float4 v = __ldg(c4 + i);
        add_square(v.x, hi, lo, bad);
        add_square(v.y, hi, lo, bad);
        add_square(v.z, hi, lo, bad);
        add_square(v.w, hi, lo, bad);
      }
    } else {
#pragma unroll 8
      for (int i = tid; i < count; i += nthr) add_square(__ldg(Cown + i), hi, lo, bad);
    }
    double acc = static_cast<double>(hi) + static_cast<double>(lo);
    acc = warp_sum_d(acc);
    bad = __syncthreads_or(bad);
    if ((tid & 31) == 0) wred[tid >> 5] = acc;
    __syncthreads();
    if (tid == 0) {
      double t = 0.0;
      for (int i = 0; i < nthr / 32; ++i) t += wred[i];
      dpart[0] = t;
      ipart[0] = bad;
      s_jfail = 0;
    }
  }
  cluster_sync();
  if (tid == 0) {
    double t = 0.0;
    int bad = 0;
    for (int q = 0; q < CTAS; ++q) {
      t += dsmem_ld_f64(dsmem_addr(dpart, q));
      bad |= dsmem_ld_s32(dsmem_addr(ipart, q));
    }
    s_E = t;
    s_bad = bad;
  }
  __syncthreads();
  const double E = s_E * a.inv_n2;
  if (rank == 0 && tid == 0) {
    a.res->energy_sum = s_E;
    a.res->nonfinite = s_bad;
  }
  if (s_bad || !isfinite(E) || !(E > 0.0)) {
    cluster_sync();
    return;
  }

  // ---- starting block (own rows): seed rows first, then pseudo-random ----
  for (int idx = tid; idx < nr * m; idx += nthr) {
    const int r = idx / m, j = idx % m;
    const int i = r0 + r;
    float v = hash_uniform(i, j);
    if (j < a.n_seed) {
      const size_t o = static_cast<size_t>(j) * L + i;
      v = a.seed_bf16 ? bf16_to_f32(static_cast<const uint16_t*>(a.seed)[o])
                      : static_cast<const float*>(a.seed)[o];
    }
    Z[idx] = v;
  }
  __syncthreads();
  for (int idx = tid; idx < m * m; idx += nthr) {
    const int p = idx / m, q = idx % m;
    float g = 0.f;
    for (int r = 0; r < nr; ++r) g = fmaf(Z[r * m + p], Z[r * m + q], g);
    Gp[idx] = g;
  }

  int dec = 0;  // 1 converged, 2 block too short, 3 iteration cap
  constexpr int cpg = m / 4;  // columns per thread group in C V
  float* Vown = big ? Vall : Vall + static_cast<size_t>(r0) * m;
  float* U = Vown;  // U = V W replaces the own rows of V in place
  for (int it = 0;; ++it) {
    // ---- orthonormalise Z (Gram partials in Gp): V = Z D L^-T ----
    cluster_sync();
    for (int idx = tid; idx < m * m; idx += nthr) {
      float g = 0.f;
      g = cluster_sum<CTAS>(Gp + idx);
      T[(idx / m) * ld + idx % m] = g;
    }
    __syncthreads();
    if (chol_block<M>(T, ld, Lf, dsc, pv, &s_cflag)) {
      // each row v of V solves v L^T = z D by forward substitution
      for (int r = tid; r < nr; r += nthr) {
        float v[M];
#pragma unroll
        for (int j = 0; j < M; ++j) {
          float acc = Z[r * m + j] * dsc[j];
#pragma unroll
          for (int k = 0; k < j; ++k) acc = fmaf(-v[k], Lf[j * ld + k], acc);
          v[j] = acc / Lf[j * ld + j];
        }
#pragma unroll
        for (int j = 0; j < M; ++j) Vown[r * m + j] = v[j];
      }
    } else {
      // rank-deficient block: symmetric orthonormalisation with Jacobi
      if (!orth_core(T, ld, m, a.max_sweeps, js, T, ld, dsc, pv, &s_deficient) && tid == 0)
        s_jfail = 1;
      for (int idx = tid; idx < nr * m; idx += nthr) {
        const int r = idx / m, j = idx % m;
        float v = 0.f;
        for (int k = 0; k < m; ++k) v = fmaf(Z[r * m + k], T[k * ld + j], v);
        Vown[idx] = v;
      }
    }
    if (big) {
      // ---- publish the own rows of V in the workspace (read back by every CTA) ----
      __syncthreads();
      float* vg = a.Vg + static_cast<size_t>(r0) * m;
      for (int i4 = tid; i4 < nr * m / 4; i4 += nthr)
        reinterpret_cast<float4*>(vg)[i4] = reinterpret_cast<const float4*>(Vown)[i4];
      __threadfence();
      cluster_sync();
    } else {
      // ---- gather the other rows of V from the peers ----
      cluster_sync();
      for (int q = 0; q < CTAS; ++q) {
        if (q == rank) continue;
        const int q0 = q * rp;
        const int nq = min(rp, L - q0);
        float* dst = Vall + static_cast<size_t>(q0) * m;
        for (int i4 = tid; i4 < nq * m / 4; i4 += nthr)
          reinterpret_cast<float4*>(dst)[i4] = dsmem_ld_f4(dsmem_addr(dst + 4 * i4, q));
      }
    }
    __syncthreads();
    // ---- Y = C[own rows, :] V / n ----
    if (kResident) {
      const int r = tid >> 2, cg = tid & 3;
      const float* crow = Ct + r * cres_ld(L);
      const float* vb = Vall + cg * cpg;
      float acc[cpg];
#pragma unroll
      for (int c = 0; c < cpg; ++c) acc[c] = 0.f;
      if (r < nr) {
#pragma unroll 4
        for (int l = 0; l < L; ++l) {
          const float cv = crow[l];
#pragma unroll
          for (int c4 = 0; c4 < cpg; c4 += 4) {
            const float4 v = *reinterpret_cast<const float4*>(vb + l * m + c4);
            acc[c4] = fmaf(cv, v.x, acc[c4]);
            acc[c4 + 1] = fmaf(cv, v.y, acc[c4 + 1]);
            acc[c4 + 2] = fmaf(cv, v.z, acc[c4 + 2]);
            acc[c4 + 3] = fmaf(cv, v.w, acc[c4 + 3]);
          }
        }
#pragma unroll
        for (int c = 0; c < cpg; ++c) Y[r * m + cg * cpg + c] = acc[c] * a.inv_n;
      }
    } else if (big) {
      constexpr int slots = (kClusterThreads / 2) / (M / 8);
      switch ((nr + slots - 1) / slots) {
        case 1: cv_big<M, 1>(Cown, nr, a.Vg, L, vecC, Ct, Vt, Y, a.inv_n); break;
        case 2: cv_big<M, 2>(Cown, nr, a.Vg, L, vecC, Ct, Vt, Y, a.inv_n); break;
        case 3: cv_big<M, 3>(Cown, nr, a.Vg, L, vecC, Ct, Vt, Y, a.inv_n); break;
        case 4: cv_big<M, 4>(Cown, nr, a.Vg, L, vecC, Ct, Vt, Y, a.inv_n); break;
        case 5: cv_big<M, 5>(Cown, nr, a.Vg, L, vecC, Ct, Vt, Y, a.inv_n); break;
        case 6: cv_big<M, 6>(Cown, nr, a.Vg, L, vecC, Ct, Vt, Y, a.inv_n); break;
        case 7: cv_big<M, 7>(Cown, nr, a.Vg, L, vecC, Ct, Vt, Y, a.inv_n); break;
        default: cv_big<M, 8>(Cown, nr, a.Vg, L, vecC, Ct, Vt, Y, a.inv_n); break;
      }
    } else {
      // C streamed through double-buffered cp.async tiles
      const int r = tid >> 2, cg = tid & 3;
      const int ntile = (L + kCvTileL - 1) / kCvTileL;
      const bool vec = vecC;
      float acc[cpg];
#pragma unroll
      for (int c = 0; c < cpg; ++c) acc[c] = 0.f;
      stage_c_tile(Ct, Cown, nr, L, 0, vec);
      for (int t = 0; t < ntile; ++t) {
        if (t + 1 < ntile) {
          stage_c_tile(Ct + ((t + 1) & 1) * kCvTileRows * kCvTileLd, Cown, nr, L, t + 1, vec);
          cp_async_wait<1>();
        } else {
          cp_async_wait<0>();
        }
        __syncthreads();
        const float* crow = Ct + (t & 1) * kCvTileRows * kCvTileLd + r * kCvTileLd;
        const int l0 = t * kCvTileL;
        const int nl = min(kCvTileL, L - l0);
        const float* vb = Vall + static_cast<size_t>(l0) * m + cg * cpg;
        for (int l = 0; l < nl; ++l) {
          const float cv = crow[l];
#pragma unroll
          for (int c4 = 0; c4 < cpg; c4 += 4) {
            const float4 v = *reinterpret_cast<const float4*>(vb + l * m + c4);
            acc[c4] = fmaf(cv, v.x, acc[c4]);
            acc[c4 + 1] = fmaf(cv, v.y, acc[c4 + 1]);
            acc[c4 + 2] = fmaf(cv, v.z, acc[c4 + 2]);
            acc[c4 + 3] = fmaf(cv, v.w, acc[c4 + 3]);
          }
        }
        __syncthreads();  // the buffer is refilled two tiles later
      }
      if (r < nr)
#pragma unroll
        for (int c = 0; c < cpg; ++c) Y[r * m + cg * cpg + c] = acc[c] * a.inv_n;
    }
    __syncthreads();
    // ---- H = V^T Y summed over the cluster, symmetrised, into the Jacobi matrix ----
    for (int idx = tid; idx < m * m; idx += nthr) {
      const int p = idx / m, q = idx % m;
      float h = 0.f;
      for (int r = 0; r < nr; ++r) h = fmaf(Vown[r * m + p], Y[r * m + q], h);
      Hp[idx] = h;
    }
    cluster_sync();
    for (int idx = tid; idx < m * m; idx += nthr) {
      const int i = idx / m, j = idx % m;
      const float hij = cluster_sum<CTAS>(Hp + i * m + j);
      const float hji = cluster_sum<CTAS>(Hp + j * m + i);
      js.A[i * ld + j] = 0.5f * (hij + hji);
    }
    __syncthreads();
    // ---- Rayleigh-Ritz: H = W Theta W^T, columns by descending theta ----
    if (!jacobi_fast<M>(js.A, js.A2, js.V, ld, a.rr_tol, a.max_sweeps, js.red, js.cs) && tid == 0)
      s_jfail = 1;
    for (int i = tid; i < m; i += nthr) js.rank[i] = desc_rank(js.A, ld, m, i);
    __syncthreads();
    for (int i = tid; i < m; i += nthr) th[js.rank[i]] = static_cast<double>(js.A[i * ld + i]);
    for (int idx = tid; idx < m * m; idx += nthr) {
      const int row = idx / m, col = idx % m;
      W[row * ld + js.rank[col]] = js.V[row * ld + col];
    }
    __syncthreads();
    // ---- U = V W and Z = Y W in place (own rows); residual and Gram partials ----
    {
      // the M lanes of a row hold its entries; lane j forms column j from the
      // row read through shuffles, so the row is read before it is overwritten
      constexpr int rows_per_warp = 32 / M;
      const int lane = tid & 31, sub = lane / M, j = lane % M;
      for (int rb = (tid >> 5) * rows_per_warp; rb < nr; rb += (nthr >> 5) * rows_per_warp) {
        const int r = rb + sub;
        const bool ok = r < nr;
        const float v = ok ? Vown[r * m + j] : 0.f;
        const float y = ok ? Y[r * m + j] : 0.f;
        float u = 0.f, z = 0.f;
#pragma unroll
        for (int k = 0; k < M; ++k) {
          const float wk = W[k * ld + j];
          u = fmaf(__shfl_sync(0xffffffffu, v, sub * M + k), wk, u);
          z = fmaf(__shfl_sync(0xffffffffu, y, sub * M + k), wk, z);
        }
        if (ok) {
          U[r * m + j] = u;
          Z[r * m + j] = z;
        }
      }
    }
    __syncthreads();
    for (int j = tid; j < m; j += nthr) {
      const float t = static_cast<float>(th[j]);
      float acc = 0.f;
      for (int r = 0; r < nr; ++r) {
        const float d = Z[r * m + j] - t * U[r * m + j];
        acc = fmaf(d, d, acc);
      }
      resp[j] = acc;
    }
    for (int idx = tid; idx < m * m; idx += nthr) {
      const int p = idx / m, q = idx % m;
      float g = 0.f;
      for (int r = 0; r < nr; ++r) g = fmaf(Z[r * m + p], Z[r * m + q], g);
      Gp[idx] = g;
    }
    cluster_sync();
    for (int j = tid; j < m; j += nthr) {
      float t = 0.f;
      t = cluster_sum<CTAS>(resp + j);
      r2[j] = t;
    }
    __syncthreads();
    // ---- convergence test (as in the multi-launch path), decided by rank 0 ----
    if (rank == 0 && tid == 0) {
      const int k = k_rule(th, m, a.eps * E);
      int R = a.r_override > 0 ? a.r_override : k + a.p;
      if (R > L) R = L;
      const bool fits = k <= m && R <= m - 1;
      int conv = fits ? 1 : 0;
      for (int i = 0; i < R && i < m && conv; ++i)
        if (!ritz_converged(r2[i], s_r2prev[i], th[i], th[0], a.tol)) conv = 0;
      for (int i = 0; i < m; ++i) s_r2prev[i] = r2[i];
      int d = conv ? 1 : 0;
      if (!d && !fits && it >= 15) d = 2;
      if (!d && it >= a.max_iter - 1) d = 3;
      flag[0] = d;
    }
    cluster_sync();
    if (tid == 0) s_dec = dsmem_ld_s32(dsmem_addr(flag, 0));
    __syncthreads();
    dec = s_dec;
    if (dec != 0) break;
  }

  // ---- projector rows: sign-canonical, scaled Ritz vectors ----
  if (tid == 0) {
    int k = k_rule(th, m, a.eps * E);
    if (k > L) k = L;
    int R = a.r_override > 0 ? a.r_override : k + a.p;
    if (R > L) R = L;
    if (R > m) R = m;
    double cum = 0.0;
    for (int i = 0; i < R; ++i) cum += th[i] * th[i];
    s_k = k;
    s_R = R;
    s_scale = static_cast<float>(a.scale_on ? 1.0 / sqrt(cum) : 1.0);
  }
  // largest-magnitude entry of each column over the own rows (lowest row on ties)
  for (int j = tid; j < m; j += nthr) {
    float best = -1.f, val = 0.f;
    int bi = 0x7fffffff;
    for (int r = 0; r < nr; ++r) {
      const float u = U[r * m + j];
      if (fabsf(u) > best) {
        best = fabsf(u);
        val = u;
        bi = r0 + r;
      }
    }
    aval[j] = val;
    aidx[j] = bi;
  }
  cluster_sync();
  const int R = s_R;
  const float sc = s_scale;
  if (dec != 2) {
    for (int j = tid; j < m; j += nthr) {
      float best = -1.f, val = 0.f;
      int bi = 0x7fffffff;
      for (int q = 0; q < CTAS; ++q) {
        const float v = dsmem_ld_f32(dsmem_addr(aval + j, q));
        const int ix = dsmem_ld_s32(dsmem_addr(aidx + j, q));
        if (fabsf(v) > best || (fabsf(v) == best && ix < bi)) {
          best = fabsf(v);
          val = v;
          bi = ix;
        }
      }
      pv[j] = val < 0.f ? -sc : sc;
    }
    __syncthreads();
    for (int idx = tid; idx < a.r_cap * nr; idx += nthr) {
      const int i = idx / nr, r = idx - (idx / nr) * nr;
      const float v = i < R ? pv[i] * U[r * m + i] : 0.f;
      const size_t o = static_cast<size_t>(i) * L + r0 + r;
      if (a.out_bf16)
        static_cast<uint16_t*>(a.rows_out)[o] = bf16_bits(v);
      else
        static_cast<float*>(a.rows_out)[o] = v;
    }
  }
  if (rank == 0 && tid == 0) {
    SolverResult* res = a.res;
    res->k = s_k;
    res->R = R;
    res->scale = sc;
    res->converged = dec == 1 ? 1 : 0;
    res->block_short = dec == 2 ? 1 : 0;
    res->jacobi_failed = s_jfail;
    for (int i = 0; i < m; ++i) {
      res->theta[i] = th[i];
      res->res2[i] = r2[i];
    }
  }
  cluster_sync();  // no CTA leaves while a peer may still read its shared memory
}

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

}  // namespace

size_t solver_workspace_bytes(int L) {
  const size_t tall = align256(sizeof(float) * static_cast<size_t>(L) * kMaxBlock);
  const size_t ufull = align256(sizeof(float) * static_cast<size_t>(L) * (L > kMaxBlock ? kMaxBlock : L));
  const size_t sq = align256(sizeof(float) * kMaxBlock * kMaxBlock);
  return align256(sizeof(SolverResult)) + 3 * tall + (ufull > tall ? ufull : tall) + 4 * sq;
}

SolverWs solver_carve(void* ws, int L) {
  uint8_t* p = static_cast<uint8_t*>(ws);
  const size_t tall = align256(sizeof(float) * static_cast<size_t>(L) * kMaxBlock);
  const size_t ufull = align256(sizeof(float) * static_cast<size_t>(L) * (L > kMaxBlock ? kMaxBlock : L));
  const size_t sq = align256(sizeof(float) * kMaxBlock * kMaxBlock);
  SolverWs w;
  w.res = reinterpret_cast<SolverResult*>(p);
  p += align256(sizeof(SolverResult));
  w.V = reinterpret_cast<float*>(p); p += tall;
  w.Y = reinterpret_cast<float*>(p); p += tall;
  w.Z = reinterpret_cast<float*>(p); p += tall;
  w.U = reinterpret_cast<float*>(p); p += (ufull > tall ? ufull : tall);
  w.H = reinterpret_cast<float*>(p); p += sq;
  w.G = reinterpret_cast<float*>(p); p += sq;
  w.W = reinterpret_cast<float*>(p); p += sq;
  w.T = reinterpret_cast<float*>(p);
  return w;
}

cudaError_t launch_solver_energy(const float* C, int L, SolverWs w, cudaStream_t st) {
  k_solver_reset<<<1, 256, 0, st>>>(w.res);
  const size_t count = static_cast<size_t>(L) * L;
  int blocks = static_cast<int>((count + 255) / 256);
  if (blocks > 1024) blocks = 1024;
  // up to L = 128 one block: the same sum, in the same order, on every call
  if (L <= 128) blocks = 1;
  k_solver_energy<<<blocks, 256, 0, st>>>(C, count, w.res);
  count_launches(2);
  return cudaGetLastError();
}

static cudaError_t set_smem(const void* f, size_t bytes) {
  // 200 KB up front for every solver kernel: one attribute call per kernel and device
  (void)bytes;
  return raise_smem_limit(f, 200 * 1024);
}

cudaError_t launch_jacobi_full_batch(const JacobiBatch& b, cudaStream_t st) {
  if (b.count < 1 || b.count > kMaxJacobiBatch || b.L < 1 || b.L > 128) return cudaErrorInvalidValue;
  const size_t bytes = jac_smem_bytes(b.L);
  cudaError_t e = set_smem(reinterpret_cast<const void*>(k_jacobi_full_batch), bytes);
  if (e != cudaSuccess) return e;
  k_jacobi_full_batch<<<b.count, jac_threads(b.L), bytes, st>>>(b);
  count_launches(1);
  return cudaGetLastError();
}

cudaError_t launch_jacobi_full(const float* C, int L, double inv_n, int max_sweeps, SolverWs w,
                               cudaStream_t st) {
  const size_t bytes = jac_smem_bytes(L);
  cudaError_t e = set_smem(reinterpret_cast<const void*>(k_jacobi_full), bytes);
  if (e != cudaSuccess) return e;
  const int jt = jac_threads(L);
  k_jacobi_full<<<1, jt, bytes, st>>>(C, L, static_cast<float>(inv_n), max_sweeps, w);
  count_launches(1);
  return cudaGetLastError();
}

cudaError_t launch_subspace_init(int L, int m, const void* seed, int n_seed, int seed_bf16,
                                 SolverWs w, cudaStream_t st) {
  k_sub_init<<<64, 256, 0, st>>>(L, m, seed, n_seed, seed_bf16, w);
  const size_t gb = sizeof(float) * kRows * m;
  k_sub_gram<<<(L + kRows - 1) / kRows, 256, gb, st>>>(L, m, w);
  count_launches(2);
  return cudaGetLastError();
}

cudaError_t launch_subspace_iteration(const float* C, int L, int m, double inv_n, int max_sweeps,
                                      float rr_tol, SolverWs w, cudaStream_t st) {
  const int nb = (L + kRows - 1) / kRows;
  const size_t jb = jac_smem_bytes(m);
  const size_t ab = sizeof(float) * (m * m + kRows * m);
  const size_t hb = sizeof(float) * (2 * kHRows * m);
  const size_t rb = sizeof(float) * (m * m + 4 * kRows * m);
  cudaError_t e;
  if ((e = set_smem(reinterpret_cast<const void*>(k_sub_orth), jb)) != cudaSuccess) return e;
  if ((e = set_smem(reinterpret_cast<const void*>(k_sub_rr), jb)) != cudaSuccess) return e;
  if ((e = set_smem(reinterpret_cast<const void*>(k_sub_apply), ab)) != cudaSuccess) return e;
  if ((e = set_smem(reinterpret_cast<const void*>(k_sub_h), hb)) != cudaSuccess) return e;
  if ((e = set_smem(reinterpret_cast<const void*>(k_sub_ritz), rb)) != cudaSuccess) return e;
  const int jt = jac_threads(m);
  const bool pdl = pdl_enabled();
  const float fn = static_cast<float>(inv_n);
  if ((e = launch_ex(k_sub_orth, dim3(1), dim3(jt), jb, st, 1, pdl, m, max_sweeps, w)) != cudaSuccess)
    return e;
  if ((e = launch_ex(k_sub_apply, dim3(nb), dim3(256), ab, st, 1, pdl,
                     static_cast<const float*>(w.Z), static_cast<const float*>(w.T), w.V, w.Y, L,
                     m)) != cudaSuccess)
    return e;
  {
    const int JB = L >= 1024 ? 256 : (L >= 256 ? 64 : 32);
    const size_t cvb = sizeof(float) * (kCvRows * (JB + 1) + JB * m);
    if ((e = set_smem(reinterpret_cast<const void*>(k_sub_cv), cvb)) != cudaSuccess) return e;
    e = launch_ex(k_sub_cv, dim3((L + kCvRows - 1) / kCvRows, (L + JB - 1) / JB), dim3(128), cvb, st,
                  1, pdl, C, L, m, JB, fn, w);
    if (e != cudaSuccess) return e;
  }
  if ((e = launch_ex(k_sub_h, dim3((L + kHRows - 1) / kHRows), dim3(256), hb, st, 1, pdl, L, m, w)) !=
      cudaSuccess)
    return e;
  if ((e = launch_ex(k_sub_rr, dim3(1), dim3(jt), jb, st, 1, pdl, m, max_sweeps, rr_tol, w)) !=
      cudaSuccess)
    return e;
  return launch_ex(k_sub_ritz, dim3(nb), dim3(256), rb, st, 1, pdl, L, m, w);
}

cudaError_t launch_subspace_check(int L, int m, double eps, int p, int r_override, double tol,
                                  double inv_n2, SolverWs w, cudaStream_t st) {
  k_sub_check<<<1, 32, 0, st>>>(L, m, eps, p, r_override, tol, inv_n2, w);
  count_launches(1);
  return cudaGetLastError();
}

cudaError_t launch_solver_finalize(int L, int m, double eps, int p, int r_override, int scale_on,
                                   void* rows_out, int r_cap, int out_bf16, double inv_n2,
                                   SolverWs w, cudaStream_t st) {
  k_finalize<<<1, 256, 0, st>>>(L, m, eps, p, r_override, scale_on, rows_out, r_cap, out_bf16,
                                inv_n2, w);
  count_launches(1);
  return cudaGetLastError();
}

bool cluster_solve_fits(int L, int m) {
  if (L <= 128 || L > kClusterCtas * kCvBigRows || (m != 16 && m != 32)) return false;
  const int rp = (L + kClusterCtas - 1) / kClusterCtas;
  // (the static shared arrays of the kernel take about 2 KB more)
  return cluster_layout(L, m, rp).total <= (L > kClusterGatherMaxL ? 216 : 200) * 1024;
}

cudaError_t launch_cluster_solve_batch(ClusterSolveBatch& b, int count, cudaStream_t st) {
  if (count < 1 || count > kMaxSolveBatch) return cudaErrorInvalidValue;
  const int L = b.s[0].L, m = b.s[0].m;
  if (!cluster_solve_fits(L, m)) return cudaErrorInvalidValue;
  int ctas = cluster_ctas(L);
  if (ctas > kClusterCtas) {
    // clusters above 8 CTAs are opt-in, and need 16 SMs of one GPC: where no
    // GPC of the device can hold one (the cluster occupancy query) the
    // cluster stays at 8
    auto k16 = m == 16 ? k_solve_cluster<16, 16> : k_solve_cluster<32, 16>;
    const size_t bytes16 = cluster_layout(L, m, (L + 15) / 16).total;
    int fit = 0;
    if (raise_smem_limit(reinterpret_cast<const void*>(k16), 216 * 1024) == cudaSuccess &&
        cudaFuncSetAttribute(k16, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) == cudaSuccess) {
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3(1, 1, 16);
      cfg.blockDim = dim3(kClusterThreads);
      cfg.dynamicSmemBytes = bytes16;
      cudaLaunchAttribute at[1];
      at[0].id = cudaLaunchAttributeClusterDimension;
      at[0].val.clusterDim.x = 1;
      at[0].val.clusterDim.y = 1;
      at[0].val.clusterDim.z = 16;
      cfg.attrs = at;
      cfg.numAttrs = 1;
      if (cudaOccupancyMaxActiveClusters(&fit, k16, &cfg) != cudaSuccess) fit = 0;
    }
    if (fit < 1) ctas = kClusterCtas;
  }
  const int rp = (L + ctas - 1) / ctas;
  for (int i = 0; i < count; ++i) {
    if (b.s[i].L != L || b.s[i].m != m) return cudaErrorInvalidValue;
    b.s[i].rp = rp;
  }
  const size_t bytes = cluster_layout(L, m, rp).total;
  auto kern = ctas == 16 ? (m == 16 ? k_solve_cluster<16, 16> : k_solve_cluster<32, 16>)
                         : (m == 16 ? k_solve_cluster<16, kClusterCtas> : k_solve_cluster<32, kClusterCtas>);
  cudaError_t e = raise_smem_limit(reinterpret_cast<const void*>(kern), 216 * 1024);
  if (e != cudaSuccess) return e;
  return launch_ex(kern, dim3(1, count, ctas), dim3(kClusterThreads), bytes, st, ctas, false, b);
}

cudaError_t launch_cluster_solve(ClusterSolveArgs a, cudaStream_t st) {
  ClusterSolveBatch b;
  b.s[0] = a;
  return launch_cluster_solve_batch(b, 1, st);
}

INSTANT_FAULT_READER(read_fault_eig)

}  // namespace instant
