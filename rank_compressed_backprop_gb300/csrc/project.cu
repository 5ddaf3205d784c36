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
// TMEM and the epilogue writes both planes as bf16.  One CTA per
// (128-column tile, sample); 72 KB of shared memory lets three CTAs share an
// SM so that the HBM stream stays busy while other CTAs drain.
#include "kernels.h"
#include "tc.cuh"

namespace instant {

namespace {

constexpr int BM = 128;                 // columns of t per CTA (MMA M)
constexpr int BK = 64;                  // tokens per stage
constexpr int A_BYTES = BM * BK * 2;    // 16 KB: two 64-column boxes
constexpr int HALF_A = A_BYTES / 2;     // byte distance between the two boxes

struct Smem {
  uint32_t a_off, b_off, bar_off, b_stage_bytes, total;
};

__host__ __device__ inline Smem project_layout(int NT, int nk, int pq_tma) {
  Smem s;
  s.a_off = 0;
  s.b_off = kProjectStages * A_BYTES;
  s.b_stage_bytes = NT * 128;
  const uint32_t b_total = pq_tma ? kProjectStages * s.b_stage_bytes : nk * s.b_stage_bytes;
  s.bar_off = s.b_off + ((b_total + 1023u) & ~1023u);
  s.total = s.bar_off + 256;
  return s;
}

template <int NT>
__global__ void __launch_bounds__(128, 1)
    k_project_bf16(const __grid_constant__ CUtensorMap tmap_t,
                   const __grid_constant__ CUtensorMap tmap_pq, ProjectArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const Smem lay = project_layout(NT, a.nk, a.pq_tma);
  uint8_t* sA = smem + lay.a_off;
  uint8_t* sB = smem + lay.b_off;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + lay.bar_off);
  uint64_t* empty = full + kProjectStages;
  uint64_t* done = empty + kProjectStages;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int c0 = blockIdx.x * BM;
  const int b = blockIdx.y;
  const int split = blockIdx.z;  // == rank in the cluster (cluster dims 1 x 1 x splits)
  const int per = (a.nk + a.splits - 1) / a.splits;
  const int kc_begin = split * per;
  const int kc_end = kc_begin + per < a.nk ? kc_begin + per : a.nk;
  const int nkc = kc_end > kc_begin ? kc_end - kc_begin : 0;
  constexpr uint32_t kTmemCols = NT <= 32 ? 32 : (NT <= 64 ? 64 : 128);

  if (threadIdx.x == 0) {
    for (int s = 0; s < kProjectStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(done, 1);
    fence_barrier_init();
    prefetch_tmap(&tmap_t);
    if (a.pq_tma) prefetch_tmap(&tmap_pq);
  }
  if (warp == 0) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  pdl_launch_dependents();
  pdl_wait();
  if (!a.pq_tma) {
    // whole projector into shared memory, K-major with the 128-byte swizzle
    const int Rt = a.Rx + a.Ry;
    const uint16_t* pq = static_cast<const uint16_t*>(a.pq);
    const int per_chunk = NT * BK;
    for (int idx = threadIdx.x; idx < a.nk * per_chunk; idx += blockDim.x) {
      const int kc = idx / per_chunk;
      const int rem = idx - kc * per_chunk;
      const int r = rem / BK;
      const int col = rem - r * BK;
      const int l = kc * BK + col;
      const uint16_t v = (r < Rt && l < a.L) ? pq[static_cast<size_t>(r) * a.L + l] : 0;
      *reinterpret_cast<uint16_t*>(sB + kc * lay.b_stage_bytes + sw128_offset(r, col)) = v;
    }
    fence_proxy_async_smem();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0 && lane == 0) {
    // ---------------- TMA producer ----------------
    const uint32_t bytes = A_BYTES + (a.pq_tma ? lay.b_stage_bytes : 0);
    int issued = 0;
    for (int i = 0; i < nkc; ++i) {
      const int kc = kc_begin + i;
      const int s = i % kProjectStages;
      if (i >= kProjectStages &&
          !mbar_wait(&empty[s], ((i / kProjectStages) - 1) & 1)) {
        raise_fault(FAULT_WAIT_EMPTY);
        break;
      }
      mbar_arrive_expect_tx(&full[s], bytes);
      uint8_t* dst = sA + s * A_BYTES;
      tma_load_3d(dst, &tmap_t, &full[s], c0, kc * BK, b);
      tma_load_3d(dst + HALF_A, &tmap_t, &full[s], c0 + 64, kc * BK, b);
      if (a.pq_tma) tma_load_2d(sB + s * lay.b_stage_bytes, &tmap_pq, &full[s], kc * BK, 0);
      ++issued;
    }
    // drain: every copy this thread issued has landed before the CTA moves on
    for (int i = issued - kProjectStages < 0 ? 0 : issued - kProjectStages; i < issued; ++i)
      if (!mbar_wait(&full[i % kProjectStages], (i / kProjectStages) & 1))
        raise_fault(FAULT_WAIT_FULL);
  } else if (warp == 1 && lane == 0) {
    // ---------------- MMA issuer ----------------
    constexpr uint32_t idesc = idesc_bf16_f32(128, NT, /*a_mn=*/1, /*b_mn=*/0);
    bool ok = true;
    for (int i = 0; i < nkc; ++i) {
      const int kc = kc_begin + i;
      const int s = i % kProjectStages;
      if (!mbar_wait(&full[s], (i / kProjectStages) & 1)) {
        raise_fault(FAULT_WAIT_FULL);
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t a_base = smem_u32(sA + s * A_BYTES);
      const uint32_t b_base =
          smem_u32(sB + (a.pq_tma ? s : kc) * lay.b_stage_bytes);
#pragma unroll
      for (int kk = 0; kk < BK / 16; ++kk) {
        // A (MN-major): 16 tokens = 2 groups of 8 rows of 128 B; the second
        // 64-column box is HALF_A bytes away.  B (K-major): +32 B per 16 tokens.
        const uint64_t ad = sdesc_sw128(a_base + kk * 2048, HALF_A, 1024);
        const uint64_t bd = sdesc_sw128(b_base + kk * 32, 16, 1024);
        umma_bf16(tmem, ad, bd, idesc, (i | kk) != 0);
      }
      umma_commit(&empty[s]);
    }
    if (ok && nkc > 0) umma_commit(done);
  }
  __syncwarp();

  // ---------------- epilogue: TMEM -> bf16 planes ----------------
  const bool have = nkc > 0;
  if (have && !mbar_wait(done, 0)) raise_fault(FAULT_WAIT_DONE);
  tc_fence_after();
  const int row = warp * 32 + lane;
  const uint32_t taddr = tmem + (static_cast<uint32_t>(warp * 32) << 16);
  uint16_t* out0 = static_cast<uint16_t*>(a.out0);
  uint16_t* out1 = static_cast<uint16_t*>(a.out1);
  if (a.splits == 1) {
    const int c = c0 + row;
#pragma unroll
    for (int j0 = 0; j0 < NT; j0 += 16) {
      float v[16];
      tmem_ld16(taddr + j0, v);
      if (c < a.C) {
#pragma unroll
        for (int jj = 0; jj < 16; ++jj) {
          const int r = j0 + jj;
          if (r < a.Rx) {
            out0[(static_cast<size_t>(b) * a.Rx + r) * a.C + c] = bf16_bits(v[jj]);
          } else if (r < a.Rx + a.Ry) {
            out1[(static_cast<size_t>(b) * a.Ry + (r - a.Rx)) * a.C + c] = bf16_bits(v[jj]);
          }
        }
      }
    }
  } else {
    // split over tokens: park the fp32 partial, then each CTA of the cluster
    // sums a slice of the columns over all partials (distributed shared memory)
    constexpr int LDR = NT + 4;
    float* red = reinterpret_cast<float*>(sA);  // the ring is idle after the MMAs
    fence_proxy_async_smem();
    __syncthreads();
#pragma unroll
    for (int j0 = 0; j0 < NT; j0 += 16) {
      float v[16];
      if (have) {
        tmem_ld16(taddr + j0, v);
      } else {
#pragma unroll
        for (int q = 0; q < 16; ++q) v[q] = 0.f;
      }
#pragma unroll
      for (int q = 0; q < 4; ++q)
        *reinterpret_cast<float4*>(red + row * LDR + j0 + 4 * q) =
            make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
    }
    tc_fence_before();
    cluster_sync();
    const int cols = BM / a.splits;
    const int Rt = a.Rx + a.Ry;
    for (int idx = threadIdx.x; idx < (NT / 4) * cols; idx += blockDim.x) {
      const int q4 = idx / cols;
      const int cl = split * cols + (idx - q4 * cols);
      const float* src = red + cl * LDR + q4 * 4;
      float4 acc = *reinterpret_cast<const float4*>(src);
      float4 part[2];
#pragma unroll
      for (int q = 0; q < 2; ++q)
        if (q < a.splits && q != split) part[q] = dsmem_ld_f4(dsmem_addr(src, q));
#pragma unroll
      for (int q = 0; q < 2; ++q)
        if (q < a.splits && q != split) {
          acc.x += part[q].x; acc.y += part[q].y; acc.z += part[q].z; acc.w += part[q].w;
        }
      const float vals[4] = {acc.x, acc.y, acc.z, acc.w};
      const int c = c0 + cl;
      if (c < a.C) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int r = q4 * 4 + e;
          if (r < a.Rx)
            out0[(static_cast<size_t>(b) * a.Rx + r) * a.C + c] = bf16_bits(vals[e]);
          else if (r < Rt)
            out1[(static_cast<size_t>(b) * a.Ry + (r - a.Rx)) * a.C + c] = bf16_bits(vals[e]);
        }
      }
    }
    cluster_sync();
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, kTmemCols);
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

template <int NT>
cudaError_t launch_nt(const CUtensorMap& tt, const CUtensorMap& tpq, const ProjectArgs& a,
                      cudaStream_t st) {
  const Smem lay = project_layout(NT, a.nk, a.pq_tma);
  const size_t bytes = lay.total + 1024;
  static size_t configured_ = 0;
  if (bytes > configured_) {
    cudaError_t e = cudaFuncSetAttribute(k_project_bf16<NT>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(bytes));
    if (e != cudaSuccess) return e;
    configured_ = bytes;
  }
  return launch_ex(k_project_bf16<NT>, dim3((a.C + BM - 1) / BM, a.B, a.splits), dim3(128), bytes,
                   st, a.splits, pdl_enabled(), tt, tpq, a);
}

}  // namespace

size_t project_bf16_smem_bytes(const ProjectArgs& a) {
  return project_layout(a.NT, a.nk, a.pq_tma).total + 1024;
}

cudaError_t launch_project_bf16(const CUtensorMap& tmap_t, const CUtensorMap& tmap_pq,
                                const ProjectArgs& a, cudaStream_t st) {
  switch (a.NT) {
    case 16: return launch_nt<16>(tmap_t, tmap_pq, a, st);
    case 32: return launch_nt<32>(tmap_t, tmap_pq, a, st);
    case 48: return launch_nt<48>(tmap_t, tmap_pq, a, st);
    case 64: return launch_nt<64>(tmap_t, tmap_pq, a, st);
    case 80: return launch_nt<80>(tmap_t, tmap_pq, a, st);
    case 96: return launch_nt<96>(tmap_t, tmap_pq, a, st);
    case 112: return launch_nt<112>(tmap_t, tmap_pq, a, st);
    case 128: return launch_nt<128>(tmap_t, tmap_pq, a, st);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_project_f32(const ProjectArgs& a, const float* t, cudaStream_t st) {
  dim3 grid((a.C + 127) / 128, a.Rx + a.Ry, a.B);
  k_project_f32<<<grid, 128, 0, st>>>(t, a);
  count_launches(1);
  return cudaGetLastError();
}

INSTANT_FAULT_READER(read_fault_project)

}  // namespace instant
