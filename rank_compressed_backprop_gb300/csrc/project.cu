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
// into L2, so the ring mostly refills from L2.  When those tiles would leave
// SMs idle (few samples, e.g. four 2048-token samples of 4096 channels: 128
// tiles for 152 SMs), two to four CTAs of a cluster share each tile's token
// axis and sum their fp32 partials through distributed shared memory; with
// short token axes (a BERT-base batch: 8 chunks per tile) the two cluster
// barriers cost more than the balance buys, so the split is kept for shares
// of at least 8 chunks.
#include <map>
#include <mutex>
#include <tuple>

#include "kernels.h"
#include "project_tile.cuh"
#include "tc.cuh"

namespace instant {

namespace {

__host__ __device__ inline uint32_t project_smem_bytes(int NT, int nk, int pq_tma, int ns) {
  return proj_layout(NT, nk, pq_tma, ns).bytes + 128;  // + barriers and the TMEM slot
}

// NS: ring depth (kProjectStages; 2 for tiles of at most two chunks, so that
// twice the CTAs share an SM and hide each other's per-sample latency)
template <int NS>
__global__ void __launch_bounds__(128, 1)
    k_project_bf16(const __grid_constant__ CUtensorMap tmap_t,
                   const __grid_constant__ CUtensorMap tmap_pq, ProjectArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const int NT = a.NT;
  const ProjLayout lay = proj_layout(NT, a.nk, a.pq_tma, NS);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + lay.bytes);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + kProjBarriers);
  const uint32_t tmem_cols = NT <= 32 ? 32 : (NT <= 64 ? 64 : 128);

  ProjPipe pipe = proj_pipe(smem, bars, NT, a.nk, a.pq_tma, 0, NS);
  // token share of this CTA: the split CTAs of a tile form one cluster along z
  const int S = a.split;
  const int rank = blockIdx.z;
  const int k0 = static_cast<int>(static_cast<long long>(a.nk) * rank / S);
  const int nkl = static_cast<int>(static_cast<long long>(a.nk) * (rank + 1) / S) - k0;
  if (threadIdx.x == 0) {
    proj_init_barriers(pipe, NS);
    fence_barrier_init();
    prefetch_tmap(&tmap_t);
    if (a.pq_tma) prefetch_tmap(&tmap_pq);
    // the input tile streams into L2 while the predecessor finishes (issued
    // before the TMEM allocation, which may wait for TMEM the predecessor's
    // CTAs on this SM still hold)
    proj_prefetch(&tmap_t, a, blockIdx.y * a.spb, blockIdx.x * kProjBM, k0, nkl);
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
  if (S == 1) {
    // a.spb consecutive samples of the same column tile (short token axes:
    // one launch's fixed costs and the projector in shared memory are shared)
    const int b0 = blockIdx.y * a.spb;
    const int b1 = min(a.B, b0 + a.spb);
    for (int b = b0; b < b1; ++b) {
      if (threadIdx.x == 0 && b + 1 < b1) proj_prefetch(&tmap_t, a, b + 1, blockIdx.x * kProjBM);
      proj_tile<1, NS>(&tmap_t, &tmap_pq, a, NT, b, blockIdx.x * kProjBM, pipe);
    }
    tc_fence_before();
    __syncthreads();
    if (threadIdx.x < 32) tmem_dealloc(pipe.tmem, tmem_cols);
    return;
  }
  // ---- token split: partial sums in the idle ring, reduced across the cluster ----
  float* part = reinterpret_cast<float*>(pipe.sA);  // [NT][128] fp32
  proj_tile<1, NS>(&tmap_t, &tmap_pq, a, NT, blockIdx.y, blockIdx.x * kProjBM, pipe, k0, nkl, part);
  tc_fence_before();
  __syncthreads();
  if (threadIdx.x < 32) tmem_dealloc(pipe.tmem, tmem_cols);
  cluster_sync();
  {
    // rank z writes columns [z * 128 / S, (z + 1) * 128 / S) of every row, in
    // pieces of 8 columns (16 bytes of bf16), summing the S partials in rank order
    const int b = blockIdx.y;  // spb == 1 with a split
    const int c_tile = blockIdx.x * kProjBM;
    const int Rt = a.Rx + a.Ry;
    const int p0 = kProjBM / 8 * rank / S, p1 = kProjBM / 8 * (rank + 1) / S;
    const int np = p1 - p0;
    uint16_t* out0 = static_cast<uint16_t*>(a.out0);
    uint16_t* out1 = static_cast<uint16_t*>(a.out1);
    for (int idx = threadIdx.x; idx < Rt * np; idx += blockDim.x) {
      const int r = idx / np;
      const int piece = p0 + (idx - r * np);
      const float* src = part + r * kProjBM + piece * 8;
      float4 lo[4], hi[4];
#pragma unroll
      for (int q = 0; q < 4; ++q)
        if (q < S) {
          lo[q] = dsmem_ld_f4(dsmem_addr(src, q));
          hi[q] = dsmem_ld_f4(dsmem_addr(src + 4, q));
        }
      float4 l = lo[0], h = hi[0];
#pragma unroll
      for (int q = 1; q < 4; ++q)
        if (q < S) {
          l.x += lo[q].x; l.y += lo[q].y; l.z += lo[q].z; l.w += lo[q].w;
          h.x += hi[q].x; h.y += hi[q].y; h.z += hi[q].z; h.w += hi[q].w;
        }
      const int c = c_tile + piece * 8;
      uint16_t* dst = r < a.Rx ? out0 + (static_cast<size_t>(b) * a.Rx + r) * a.C + c
                               : out1 + (static_cast<size_t>(b) * a.Ry + (r - a.Rx)) * a.C + c;
      const uint4 v = make_uint4(pack_bf16x2(l.x, l.y), pack_bf16x2(l.z, l.w), pack_bf16x2(h.x, h.y),
                                 pack_bf16x2(h.z, h.w));
      if (c + 8 <= a.C) {
        *reinterpret_cast<uint4*>(dst) = v;
      } else {
        const uint16_t e[8] = {static_cast<uint16_t>(v.x & 0xffffu), static_cast<uint16_t>(v.x >> 16),
                               static_cast<uint16_t>(v.y & 0xffffu), static_cast<uint16_t>(v.y >> 16),
                               static_cast<uint16_t>(v.z & 0xffffu), static_cast<uint16_t>(v.z >> 16),
                               static_cast<uint16_t>(v.w & 0xffffu), static_cast<uint16_t>(v.w >> 16)};
        for (int j = 0; c + j < a.C; ++j) dst[j] = e[j];
      }
    }
  }
  cluster_sync();  // peers may still read this CTA's partial sums
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
  return project_smem_bytes(a.NT, a.nk, a.pq_tma, a.stages) + 1024;
}

namespace {

template <int NS>
cudaError_t ensure_project_smem(size_t bytes) {
  return raise_smem_limit(reinterpret_cast<const void*>(k_project_bf16<NS>), bytes);
}

template <int NS>
int resident_project(size_t bytes, int cols) {
  if (ensure_project_smem<NS>(bytes) != cudaSuccess) return 0;
  return resident_ctas_per_sm(reinterpret_cast<const void*>(k_project_bf16<NS>), 128, bytes, cols);
}

template <int NS>
cudaError_t launch_ns(const CUtensorMap& tmap_t, const CUtensorMap& tmap_pq, const ProjectArgs& a,
                      cudaStream_t st) {
  const size_t bytes = project_bf16_smem_bytes(a);
  const cudaError_t err = ensure_project_smem<NS>(bytes);
  if (err != cudaSuccess) return err;
  return launch_ex(k_project_bf16<NS>, dim3((a.C + kProjBM - 1) / kProjBM, (a.B + a.spb - 1) / a.spb, a.split),
                   dim3(128), bytes, st, a.split, pdl_enabled(), tmap_t, tmap_pq, a);
}

}  // namespace

int project_bf16_ctas_per_sm(const ProjectArgs& a) {
  // one residency count per (device, shared-memory size, TMEM width, ring depth)
  static std::mutex mu;
  static std::map<std::tuple<int, size_t, int, int>, int> counts;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  const size_t bytes = project_bf16_smem_bytes(a);
  const int cols = a.NT <= 32 ? 32 : (a.NT <= 64 ? 64 : 128);
  const auto key = std::make_tuple(dev, bytes, cols, a.stages);
  {
    std::lock_guard<std::mutex> lock(mu);
    const auto it = counts.find(key);
    if (it != counts.end()) return it->second;
  }
  const int n = a.stages == 2 ? resident_project<2>(bytes, cols) : resident_project<kProjectStages>(bytes, cols);
  std::lock_guard<std::mutex> lock(mu);
  if (n > 0) counts[key] = n;
  return n;
}

cudaError_t launch_project_bf16(const CUtensorMap& tmap_t, const CUtensorMap& tmap_pq,
                                const ProjectArgs& a, cudaStream_t st) {
  if (a.NT < 16 || a.NT > 128 || a.NT % 16 != 0) return cudaErrorInvalidValue;
  if (a.split < 1 || a.split > 4) return cudaErrorInvalidValue;
  if (a.spb < 1 || (a.split > 1 && a.spb != 1)) return cudaErrorInvalidValue;
  // a split parks NT x 128 fp32 partials in the idle ring: the two-stage ring
  // (32 KB) holds them up to NT = 64
  if (a.stages == 2 && (a.split == 1 || a.NT <= 64)) return launch_ns<2>(tmap_t, tmap_pq, a, st);
  if (a.stages != kProjectStages) return cudaErrorInvalidValue;
  return launch_ns<kProjectStages>(tmap_t, tmap_pq, a, st);
}

cudaError_t launch_project_f32(const ProjectArgs& a, const float* t, cudaStream_t st) {
  dim3 grid((a.C + 127) / 128, a.Rx + a.Ry, a.B);
  k_project_f32<<<grid, 128, 0, st>>>(t, a);
  count_launches(1);
  return cudaGetLastError();
}

INSTANT_FAULT_READER(read_fault_project)

}  // namespace instant
