// project.cu -- projection of a [B, L, C] tensor along its token axis L by a
// small stacked projector:  out_r[b, c] = sum_l PQ[r, l] * t[b, l, c].
//
// It serves two steps of INSTANT (page "INSTANT: Compressing Gradients and
// Activations for Resource-Efficient Training"):
//   * 整体框架 -- the forward stores x_hat = P x (compress_act, Ry = 0);
//   * 关键设计 3 -- g_hat_y1 = g_y^T P^T and g_hat_y2 = Q g_y are both read off
//     one pass over g_y with the stacked [P; Q] (project_grad).
//
// bf16 design (sm_103a): the contraction runs on the tensor cores as
// D[c, r] = sum_l t[l, c] * PQ[r, l], i.e. M = 128 columns of t per CTA,
// N = Rx + Ry (padded to 16), K = L streamed in 64-token chunks.  t is the
// MN-major A operand, read exactly once from HBM by TMA through a 4-stage
// mbarrier ring; PQ is the K-major B operand.  The fp32 accumulator lives in
// TMEM and the epilogue writes both planes as bf16 (the tile itself is in
// project_tile.cuh).  One CTA per (128-column tile, sample) over the whole
// token axis; a 4-stage ring (73 KB of shared memory) lets three CTAs share
// an SM.  Before waiting for its predecessor, each CTA prefetches its tile
// into L2, so the ring mostly refills from L2.  (A token split over a 2-CTA
// cluster with a DSMEM reduction measured slower at every batch from 2 to 64
// samples of a BERT-base block: its two cluster barriers cost more than the
// balance it bought.)
#include "kernels.h"
#include "project_tile.cuh"
#include "tc.cuh"

namespace instant {

namespace {

__host__ __device__ inline uint32_t project_smem_bytes(int NT, int nk, int pq_tma) {
  return proj_layout(NT, nk, pq_tma).bytes + 128;  // + barriers and the TMEM slot
}

__global__ void __launch_bounds__(128, 1)
    k_project_bf16(const __grid_constant__ CUtensorMap tmap_t,
                   const __grid_constant__ CUtensorMap tmap_pq, ProjectArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const int NT = a.NT;
  const ProjLayout lay = proj_layout(NT, a.nk, a.pq_tma);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + lay.bytes);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + kProjBarriers);
  const uint32_t tmem_cols = NT <= 32 ? 32 : (NT <= 64 ? 64 : 128);

  ProjPipe pipe = proj_pipe(smem, bars, NT, a.nk, a.pq_tma, 0);
  if (threadIdx.x == 0) {
    proj_init_barriers(pipe);
    fence_barrier_init();
    prefetch_tmap(&tmap_t);
    if (a.pq_tma) prefetch_tmap(&tmap_pq);
    // the input tile streams into L2 while the predecessor finishes (issued
    // before the TMEM allocation, which may wait for TMEM the predecessor's
    // CTAs on this SM still hold)
    proj_prefetch(&tmap_t, a, blockIdx.y, blockIdx.x * kProjBM);
  }
  if (threadIdx.x < 32) {
    tmem_alloc(tmem_slot, tmem_cols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  pdl_launch_dependents();  // after the allocation
  pdl_wait();
  if (!a.pq_tma) {
    proj_fill_pq(a, pipe, NT, threadIdx.x, blockDim.x);
    __syncthreads();
  }
  pipe.tmem = *tmem_slot;
  proj_tile<1>(&tmap_t, &tmap_pq, a, NT, blockIdx.y, blockIdx.x * kProjBM, pipe);
  tc_fence_before();
  __syncthreads();
  if (threadIdx.x < 32) tmem_dealloc(pipe.tmem, tmem_cols);
}

// fp32 path (no tensor cores, no TF32): one thread per output element.
__global__ void k_project_f32(const float* __restrict__ t, ProjectArgs a) {
  const int c = blockIdx.x * blockDim.x + threadIdx.x;
  const int r = blockIdx.y;
  const int b = blockIdx.z;
  if (c >= a.C) return;
  const float* pq = static_cast<const float*>(a.pq);
  const float* tb = t + static_cast<size_t>(b) * a.L * a.C + c;
  float acc = 0.f;
  for (int l = 0; l < a.L; ++l) acc = fmaf(pq[static_cast<size_t>(r) * a.L + l], tb[static_cast<size_t>(l) * a.C], acc);
  if (r < a.Rx)
    static_cast<float*>(a.out0)[(static_cast<size_t>(b) * a.Rx + r) * a.C + c] = acc;
  else
    static_cast<float*>(a.out1)[(static_cast<size_t>(b) * a.Ry + (r - a.Rx)) * a.C + c] = acc;
}

}  // namespace

size_t project_bf16_smem_bytes(const ProjectArgs& a) {
  return project_smem_bytes(a.NT, a.nk, a.pq_tma) + 1024;
}

cudaError_t launch_project_bf16(const CUtensorMap& tmap_t, const CUtensorMap& tmap_pq,
                                const ProjectArgs& a, cudaStream_t st) {
  if (a.NT < 16 || a.NT > 128 || a.NT % 16 != 0) return cudaErrorInvalidValue;
  const size_t bytes = project_bf16_smem_bytes(a);
  static size_t configured_ = 0;
  if (bytes > configured_) {
    cudaError_t e = cudaFuncSetAttribute(k_project_bf16, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(bytes));
    if (e != cudaSuccess) return e;
    configured_ = bytes;
  }
  return launch_ex(k_project_bf16, dim3((a.C + kProjBM - 1) / kProjBM, a.B, 1), dim3(128), bytes,
                   st, 1, pdl_enabled(), tmap_t, tmap_pq, a);
}

cudaError_t launch_project_f32(const ProjectArgs& a, const float* t, cudaStream_t st) {
  dim3 grid((a.C + 127) / 128, a.Rx + a.Ry, a.B);
  k_project_f32<<<grid, 128, 0, st>>>(t, a);
  count_launches(1);
  return cudaGetLastError();
}

INSTANT_FAULT_READER(read_fault_project)

}  // namespace instant
