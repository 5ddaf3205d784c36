// kernels.h -- launch interfaces between the C-ABI layer and the kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace instant {

// ---------------------------------------------------------------------------
// projection along the token axis: out_r[b, c] = sum_l PQ[r, l] t[b, l, c]
// (compress_act with Ry = 0; project_grad with both planes)
// ---------------------------------------------------------------------------
struct ProjectArgs {
  int B, L, C;       // t is [B, L, C]
  int Rx, Ry;        // rows 0..Rx-1 -> out0, rows Rx..Rx+Ry-1 -> out1
  int NT;            // MMA N: Rx + Ry rounded up to a multiple of 16
  int nk;            // ceil(L / 64)
  int pq_tma;        // 1: PQ tiles arrive by TMA; 0: threads fill all of PQ up front
  int pf_chunks;     // leading 64-token chunks of its tile a CTA prefetches into L2
  int split;         // CTAs sharing a tile's token axis (1..4, a cluster along grid z);
                     // their fp32 partial sums are reduced through DSMEM
  int spb;           // samples per CTA (1 with a split): short token axes share a CTA
  int stages;        // A ring depth: kProjectStages, or 2 (at most two chunks, no split)
  const void* pq;    // [Rx+Ry, L]
  void* out0;        // [B*Rx, C]
  void* out1;        // [B*Ry, C] or null
};

constexpr int kProjectStages = 4;  // 2 and 3 stages measured slower on GB300
size_t project_bf16_smem_bytes(const ProjectArgs& a);
int project_bf16_ctas_per_sm(const ProjectArgs& a);  // 0 if a query fails
cudaError_t launch_project_bf16(const CUtensorMap& tmap_t, const CUtensorMap& tmap_pq,
                                const ProjectArgs& a, cudaStream_t st);
cudaError_t launch_project_f32(const ProjectArgs& a, const float* t, cudaStream_t st);

// ---------------------------------------------------------------------------
// dense GEMM D[M, N] = sum_k A[m, k] B[k, n] with fp32 output
// ---------------------------------------------------------------------------
struct GemmArgs {
  int M, N, K;
  int a_mn_major;    // 1: A stored [K, M]; 0: A stored [M, K]
  int b_mn_major;    // 1: B stored [K, N]; 0: B stored [N, K]
  int BN;            // N tile (64, 128 or 256)
  int nk;            // ceil(K / 64)
  int splits;        // split-K factor = cluster size along grid z (1..8);
                     // partial tiles are reduced through distributed shared memory
  int chunks_per_split;
  int stages;        // TMA ring depth, 1..kGemmStages
  int accumulate;    // fp32 output only: out += D
  int out_bf16;      // 1: bf16 output (round to nearest even); 0: fp32
  int short_a;       // 1: A stored [M, K] with M <= 64, loaded as a 64-row box
  void* out;         // [M][N]
};

constexpr int kGemmStages = 4;
size_t gemm_bf16_smem_bytes(const GemmArgs& g);
int gemm_bf16_ctas_per_sm(const GemmArgs& g);  // resident CTAs on one SM
int gemm_bf16_max_clusters(const GemmArgs& g);  // co-resident clusters of g.splits CTAs
cudaError_t launch_gemm_bf16(const CUtensorMap& tmap_a, const CUtensorMap& tmap_b,
                             const GemmArgs& g, cudaStream_t st);
cudaError_t launch_gemm_f32(const GemmArgs& g, const float* A, const float* Bm, cudaStream_t st);

// ---------------------------------------------------------------------------
// weight gradient with a short contraction, streamed to HBM:
// gw[m, n] (+)= sum_k Sx[k, m] xh[k, n], K = B * Rx <= 64 * kGradWMaxChunks
// ---------------------------------------------------------------------------
struct GradWStreamArgs {
  int M, N, K;       // gw [M = Cy, N = Cx] fp32; Sx [K, M], xh [K, N] bf16
  int nkc;           // ceil(K / 64)
  int mt, nt;        // ceil(M / 128) row tiles, ceil(N / 64) column strips
  int stages;        // Sx chunk ring depth, 2..kGradWStages
  int accumulate;    // 1: gw += result
};

constexpr int kGradWStages = 4;
constexpr int kGradWMaxChunks = 4;
size_t gradw_stream_smem_bytes(const GradWStreamArgs& g);
cudaError_t launch_gradw_stream(const CUtensorMap& tmap_sx, const CUtensorMap& tmap_xh,
                                const CUtensorMap& tmap_gw, const GradWStreamArgs& g, int ctas,
                                cudaStream_t st);

// ---------------------------------------------------------------------------
// forward y = x w^T (bf16, fp32 accumulation) with the optional side output
// x_hat = P x computed from the staged x tiles
// ---------------------------------------------------------------------------
constexpr int kForwardBN = 192;    // output tile: 128 tokens x 192 columns of y
constexpr int kForwardStages = 4;  // 40 KB each
struct ForwardArgs {
  int M, N, K;       // y [M = B*L, N = Cy], x [M, K = Cx], w [N, K]
  int mt, nt, nkc;   // ceil(M / 128), ceil(N / 192), ceil(K / 64)
  int group;         // m tiles per rasterization group
  int Rx;            // rows of P (0: no side output; else <= 32, L % 128 == 0)
  int L;             // tokens per sample
  float* xh32;       // [B, Rx, K] fp32 accumulation, zero before and after a launch
  void* xh;          // [B, Rx, K] bf16 x_hat
  unsigned int* cnt; // [B] finished tiles per sample, zero before and after a launch
};
size_t forward_bf16_smem_bytes();
cudaError_t launch_forward_bf16(const CUtensorMap& tmap_x, const CUtensorMap& tmap_w,
                                const CUtensorMap& tmap_y, const CUtensorMap& tmap_p,
                                const ForwardArgs& a, int ctas, cudaStream_t st);
cudaError_t launch_forward_f32(const float* x, const float* w, float* y, int M, int N, int K,
                               cudaStream_t st);

// ---------------------------------------------------------------------------
// rank-R expansion: out[b, l, c] = sum_r Q[r, l] * (sum_s gxh[s][b*Ry + r, c])
// ---------------------------------------------------------------------------
struct ExpandArgs {
  int B, L, Cx, Ry;
  int KR;            // Ry rounded up to a multiple of 16
  int BN;            // column tile (64 or 128)
  int nlt;           // ceil(L / 128) token tiles
  int q_tma;         // 1: Q tiles arrive by TMA (L % 8 == 0); 0: threads fill them
  int qres;          // 1: all nlt (<= kExpandMaxQRes) Q^T tiles stay resident
  int nb;            // g_hat_x blocks in flight (1..kExpandMaxBRing)
  int total;         // jobs: ceil(Cx / BN) * B * nlt
  int ctas;          // grid size (1..total); each CTA takes an equal run of jobs
  const void* gxh;   // [B*Ry][Cx], same dtype as out (fp32 path: fp32)
  const void* Q;     // [Ry, L]
  void* out;         // [B, L, Cx]
};

constexpr int kExpandStages = 2;    // Q^T ring (more than kExpandMaxQRes token tiles)
constexpr int kExpandMaxBRing = 4;
constexpr int kExpandMaxQRes = 4;
size_t expand_bf16_smem_bytes(const ExpandArgs& e);
int expand_bf16_ctas_per_sm(const ExpandArgs& e);  // 0 if the configuration cannot launch
cudaError_t launch_expand_bf16(const CUtensorMap& tmap_q, const CUtensorMap& tmap_g,
                               const CUtensorMap& tmap_out, const ExpandArgs& e, cudaStream_t st);
cudaError_t launch_expand_f32(const ExpandArgs& e, cudaStream_t st);

// ---------------------------------------------------------------------------
// fused input gradient: out[b] = Q^T (Sq[b] w) with g_hat_x kept on chip
// ---------------------------------------------------------------------------
struct FusedArgs {
  int B, L, Cx, Cy, Ry;
  int KR;            // Ry rounded up to a multiple of 16
  int spt;           // samples per g_hat_x tile (spt * Ry <= 128)
  int BN;            // column strip (64 or 128)
  int nk;            // ceil(Cy / 64)
  int stages;        // phase-1 TMA ring depth (1..6)
  int nlt;           // ceil(L / 128)
  int lt_per;        // token tiles per CTA
  int cl;            // cluster size along the token axis (1, 2, 4, 8): phase 1's K
                     // range is split across the cluster and reduced through DSMEM
  int kfull;         // 1: every CTA of the cluster runs phase 1 over the whole K
                     // (no exchange; the cluster only splits the token range)
  int q_tma;         // 1: Q^T tiles by TMA (L % 8 == 0); 0: threads fill them
  int a_rows;        // Sq rows per phase-1 TMA box (spt * Ry rounded up to 8, <= 128):
                     // the MMA still reads 128 rows, the ones past the box are unused
  const void* Q;     // [Ry, L]
  // weight gradient in the same launch (gw_mt > 0): grid rows gw_y0.. run the
  // 128 x 64 tiles of g_w[Cy, Cx] = Sx^T x_hat over K = B * Rx
  int gw_y0;         // first weight-gradient grid row (= ceil(B / spt))
  int gw_mt;         // ceil(Cy / 128) row tiles, 0: none
  int gw_nk;         // ceil(B * Rx / 64)
  int gw_acc;        // 1: g_w += result
  float* gw;         // [Cy, Cx] fp32
  // projection of g_y in the same launch (proj = 1): the input-gradient CTAs
  // of a sample group first compute the group's (sample, 128-column) tiles of
  // Sx and Sq, each tile followed by a signal; phase 1 of the group waits for
  // its own tiles, the weight-gradient CTAs for all of them
  int proj;
  int nct;           // ceil(Cy / 128): projection tiles per sample
  ProjectArgs pa;    // the projection of g_y [B, L, Cy] by [P; Q]
  unsigned int* sync;  // [gw_y0] per-group tile counts, total, finished CTAs,
                       // next ticket; zero before the launch, zeroed again by
                       // its last CTA
};

size_t gradx_fused_smem_bytes(const FusedArgs& f);
cudaError_t launch_gradx_fused(const CUtensorMap& tmap_sq, const CUtensorMap& tmap_w,
                               const CUtensorMap& tmap_q, const CUtensorMap& tmap_out,
                               const CUtensorMap& tmap_sx, const CUtensorMap& tmap_xh,
                               const CUtensorMap& tmap_gy, const CUtensorMap& tmap_pq,
                               const FusedArgs& f, cudaStream_t st);


// ---------------------------------------------------------------------------
// autocorrelation accumulation: Cout[i, j] += sum_b sum_c t[b,i,c] t[b,j,c]
// ---------------------------------------------------------------------------
struct SyrkArgs {
  int B, L, C;
  int nblk;          // ceil(L / 128)
  int ntiles;        // upper-triangle tiles: nblk * (nblk + 1) / 2 of 128 x 128, or
                     // sum_i ceil((nblk - i) / 2) of 128 x 256
  int splits;        // CTAs per tile (grid y) = cs * bs
  int cs;            // channel ranges per tile (each CTA walks all of its samples)
  int bs;            // sample ranges per tile (small statistics only)
  int nkc;           // ceil(C / 64)
  float* Cout;       // [L, L]
};

constexpr int kSyrkStages = 3;      // narrow tiles: 96 KB of stages, two CTAs per SM
constexpr int kSyrkWideStages = 4;  // wide tiles: 192 KB of stages, one CTA per SM
size_t syrk_bf16_smem_bytes(bool wide);
cudaError_t launch_syrk_bf16(const CUtensorMap& tmap_t, const SyrkArgs& s, cudaStream_t st);
// up to kMaxSyrkBatch statistics of one token length in one launch: problem p
// owns grid rows [split0[p], split0[p + 1])
constexpr int kMaxSyrkBatch = 4;
struct SyrkBatch {
  SyrkArgs s[kMaxSyrkBatch];
  int split0[kMaxSyrkBatch + 1];
  int count;
  int wide;  // 1: 128 x 256 tiles (ntiles counts them), 0: 128 x 128
};
cudaError_t launch_syrk_bf16_batch(const CUtensorMap* tmaps, const SyrkBatch& b, cudaStream_t st);
cudaError_t launch_syrk_f32(const SyrkArgs& s, const float* t, cudaStream_t st);

// ---------------------------------------------------------------------------
// symmetric eigensolver for calibration
// ---------------------------------------------------------------------------
struct SolverResult {      // lives at the start of the solver workspace
  double energy_sum;       // sum_ij C_sum[i,j]^2 (fp64)
  int nonfinite;           // any non-finite entry in C_sum
  int converged;           // set by the check step
  int k, R;
  float scale;
  int jacobi_failed;       // a Jacobi solve hit its sweep cap
  int block_short;         // k + p does not fit the block
  int pad_;
  double theta[128];       // Ritz values (descending)
  float res2[128];         // squared residual norms of the Ritz vectors
  float res2_prev[128];    // the same at the previous convergence check
};

struct SolverWs {
  SolverResult* res;
  float* V;      // [L, m] orthonormal basis
  float* Y;      // [L, m] C V
  float* Z;      // [L, m]
  float* U;      // [L, m] Ritz vectors  (full path: [L, L] eigenvectors)
  float* H;      // [m, m]
  float* G;      // [m, m]
  float* W;      // [m, m]
  float* T;      // [m, m]
};

size_t solver_workspace_bytes(int L);
SolverWs solver_carve(void* ws, int L);

cudaError_t launch_solver_energy(const float* C, int L, SolverWs w, cudaStream_t st);
constexpr int kMaxJacobiBatch = 16;
// full Jacobi of C/n (L <= 128): eigenvalues -> res->theta, vectors -> U columns
// several statistics of one L <= 128 in one launch, one CTA each
struct JacobiBatch {
  const float* C[kMaxJacobiBatch];
  float inv_n[kMaxJacobiBatch];
  SolverWs w[kMaxJacobiBatch];
  int L, max_sweeps, count;
};
cudaError_t launch_jacobi_full_batch(const JacobiBatch& b, cudaStream_t st);
cudaError_t launch_jacobi_full(const float* C, int L, double inv_n, int max_sweeps, SolverWs w,
                               cudaStream_t st);
// subspace iteration building blocks
// seed: optional [n_seed, L] rows (bf16 when seed_bf16) used as the first
// block columns; the rest is pseudo-random
cudaError_t launch_subspace_init(int L, int m, const void* seed, int n_seed, int seed_bf16,
                                 SolverWs w, cudaStream_t st);
// rr_tol: Jacobi tolerance of the Rayleigh-Ritz step (loose between
// convergence checks, tight right before one)
cudaError_t launch_subspace_iteration(const float* C, int L, int m, double inv_n, int max_sweeps,
                                      float rr_tol, SolverWs w, cudaStream_t st);
cudaError_t launch_subspace_check(int L, int m, double eps, int p, int r_override,
                                  double tol, double inv_n2, SolverWs w, cudaStream_t st);
// k, R, s and the projector rows from theta and U (sign-canonical)
cudaError_t launch_solver_finalize(int L, int m, double eps, int p, int r_override,
                                   int scale_on, void* rows_out, int r_cap, int out_bf16,
                                   double inv_n2, SolverWs w, cudaStream_t st);

// the whole subspace iteration + projector rows in one launch of an 8-CTA
// cluster (128 < L, block m of 16 or 32, while cluster_solve_fits); rp is set
// by the launcher
struct ClusterSolveArgs {
  const float* C;
  int L, m, rp;
  float inv_n;
  double inv_n2;
  double eps;
  int p, r_override, scale_on;
  double tol;
  int max_iter, max_sweeps;
  float rr_tol;
  const void* seed;      // [n_seed, L] rows seeding the block (bf16 when seed_bf16)
  int n_seed, seed_bf16;
  void* rows_out;        // [r_cap, L]; written unless the block proved too short
  int r_cap, out_bf16;
  SolverResult* res;
  float* Vg;             // [L, m] scratch: the basis exchanged through L2 (L > 512)
};
bool cluster_solve_fits(int L, int m);
cudaError_t launch_cluster_solve(ClusterSolveArgs a, cudaStream_t st);
// up to kMaxSolveBatch statistics of one size (same L and m) in one launch,
// one cluster each (grid 1 x count x 8); rp is set by the launcher
constexpr int kMaxSolveBatch = 16;
struct ClusterSolveBatch {
  ClusterSolveArgs s[kMaxSolveBatch];
};
cudaError_t launch_cluster_solve_batch(ClusterSolveBatch& b, int count, cudaStream_t st);

// ||t - Q^T S||^2 and ||t||^2 over a batch (S = Q t per sample, [B*R, C]) into
// totals[0..1] (fp64 device, zeroed by the launch)
cudaError_t launch_recon(const void* t, const void* Q, const void* S, int B, int L, int C, int R,
                         int bf16, double* totals, cudaStream_t st);

// host-side count of kernel launches issued by the library
void count_launches(unsigned int n);

// streaming multiprocessors of the current device (queried once per device)
int sm_count();

// Raises `kernel`'s dynamic shared memory limit on the current device to at
// least `bytes`.  It never lowers it, so configurations launched later with
// less still fit; with max_shared the unified L1 goes to shared memory first
// (so that as many CTAs as the shared memory allows share an SM).  Thread-safe;
// one attribute call per new maximum per (kernel, device).
cudaError_t raise_smem_limit(const void* kernel, size_t bytes, bool max_shared = false);

// CTAs of `kernel` (launched with `threads` threads and `smem` bytes of dynamic
// shared memory, allocating `tmem_cols` TMEM columns) that one SM holds at
// once: shared memory, threads, TMEM, and registers per SM sub-partition (each
// of the four holds a quarter of the register file and of the CTA's warps;
// the occupancy query does not model this split).  0 if a query fails.
int resident_ctas_per_sm(const void* kernel, int threads, size_t smem, int tmem_cols);

}  // namespace instant

#include "instant.h"

namespace instant {

// g_tilde_x = Q^T (Sq w) as two launches (g_hat_x in `ws`): every argument is
// checked and both launches are planned before the first one is issued
instant_status grad_x_two_kernels(const void* Sq, const void* w, const void* Q, void* gx, void* ws,
                                  size_t ws_bytes, int B, int L, int Cx, int Cy, int Ry,
                                  instant_dtype dt, cudaStream_t st);

// programmatic dependent launch on/off (INSTANT_NO_PDL=1 turns it off)
bool pdl_enabled();

// cudaLaunchKernelEx with an optional 1 x 1 x cluster_z cluster and optional
// programmatic stream serialization (the kernel must call pdl_wait() before
// its first global-memory access when pdl is set)
template <typename... KArgs, typename... Args>
inline cudaError_t launch_ex(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                             cudaStream_t st, int cluster_z, bool pdl, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  int na = 0;
  if (cluster_z > 1) {
    attr[na].id = cudaLaunchAttributeClusterDimension;
    attr[na].val.clusterDim.x = 1;
    attr[na].val.clusterDim.y = 1;
    attr[na].val.clusterDim.z = static_cast<unsigned>(cluster_z);
    ++na;
  }
  if (pdl) {
    attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
  }
  cfg.attrs = attr;
  cfg.numAttrs = na;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, args...);
  count_launches(1);
  return e != cudaSuccess ? e : cudaGetLastError();
}

// sticky device status words, one per translation unit
cudaError_t read_fault_project(unsigned int* out, int clear);
cudaError_t read_fault_gemm(unsigned int* out, int clear);
cudaError_t read_fault_expand(unsigned int* out, int clear);
cudaError_t read_fault_syrk(unsigned int* out, int clear);
cudaError_t read_fault_eig(unsigned int* out, int clear);
cudaError_t read_fault_fused(unsigned int* out, int clear);
cudaError_t read_fault_gradw(unsigned int* out, int clear);
cudaError_t read_fault_forward(unsigned int* out, int clear);

}  // namespace instant
