// gemm.cu -- the two dense low-rank products of INSTANT's backward (page
// "INSTANT: Compressing Gradients and Activations for Resource-Efficient
// Training", 关键设计 3):
//   g_w      = g_hat_y1 x_hat = Sx^T x_hat    (M = Cy, N = Cx, K = B*Rx)
//   g_hat_x  = g_hat_y2 w     = Sq w          (M = B*Ry, N = Cx, K = Cy)
//
// bf16 design: a tcgen05 GEMM with a 128 x BN fp32 accumulator in TMEM.  Both
// operands stream through a 4-stage TMA/mbarrier ring; either operand may be
// K-major or MN-major (Sx, x_hat and w are contracted over their row index,
// so they are MN-major operands read straight from their natural layout).
// One elected thread issues the MMAs; all four warps run the epilogue, which
// writes (or accumulates into) fp32 rows with 16-byte stores.  Split-K over
// grid z writes separate fp32 partial planes that the consumer sums.
#include "kernels.h"
#include "tc.cuh"

namespace instant {

namespace {

constexpr int BM = 128;
constexpr int BK = 64;
constexpr int A_BYTES = BM * BK * 2;  // 16 KB

__host__ __device__ inline uint32_t b_bytes(int BN) { return BN * BK * 2; }

template <int BN, int A_MN, int B_MN>
__global__ void __launch_bounds__(128, 1)
    k_gemm_bf16(const __grid_constant__ CUtensorMap tmap_a,
                const __grid_constant__ CUtensorMap tmap_b, GemmArgs g) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  constexpr uint32_t STAGE = A_BYTES + BN * BK * 2;
  uint8_t* sbase = smem;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kGemmStages * STAGE);
  uint64_t* empty = full + kGemmStages;
  uint64_t* done = empty + kGemmStages;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int n0 = blockIdx.x * BN;
  const int m0 = blockIdx.y * BM;
  const int split = blockIdx.z;
  const int kc_begin = split * g.chunks_per_split;
  int kc_end = kc_begin + g.chunks_per_split;
  if (kc_end > g.nk) kc_end = g.nk;
  const int nkc = kc_end > kc_begin ? kc_end - kc_begin : 0;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kGemmStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(done, 1);
    fence_barrier_init();
    prefetch_tmap(&tmap_a);
    prefetch_tmap(&tmap_b);
  }
  if (warp == 0) {
    tmem_alloc(tmem_slot, BN);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0 && lane == 0) {
    // ---------------- TMA producer ----------------
    int issued = 0;
    for (int i = 0; i < nkc; ++i) {
      const int s = i % kGemmStages;
      if (i >= kGemmStages && !mbar_wait(&empty[s], ((i / kGemmStages) - 1) & 1)) {
        raise_fault(FAULT_WAIT_EMPTY);
        break;
      }
      const int k0 = (kc_begin + i) * BK;
      uint8_t* sa = sbase + s * STAGE;
      uint8_t* sb = sa + A_BYTES;
      mbar_arrive_expect_tx(&full[s], STAGE);
      if (A_MN) {  // A stored [K, M]: two 64-wide M boxes of 64 K-rows
        tma_load_2d(sa, &tmap_a, &full[s], m0, k0);
        tma_load_2d(sa + A_BYTES / 2, &tmap_a, &full[s], m0 + 64, k0);
      } else {     // A stored [M, K]: one box of 64 K x 128 rows
        tma_load_2d(sa, &tmap_a, &full[s], k0, m0);
      }
      if (B_MN) {  // B stored [K, N]: BN/64 boxes of 64 N x 64 K-rows
#pragma unroll
        for (int h = 0; h < BN / 64; ++h)
          tma_load_2d(sb + h * (64 * BK * 2), &tmap_b, &full[s], n0 + 64 * h, k0);
      } else {     // B stored [N, K]: one box of 64 K x BN rows
        tma_load_2d(sb, &tmap_b, &full[s], k0, n0);
      }
      ++issued;
    }
    for (int i = issued - kGemmStages < 0 ? 0 : issued - kGemmStages; i < issued; ++i)
      if (!mbar_wait(&full[i % kGemmStages], (i / kGemmStages) & 1)) raise_fault(FAULT_WAIT_FULL);
  } else if (warp == 1 && lane == 0) {
    // ---------------- MMA issuer ----------------
    constexpr uint32_t idesc = idesc_bf16_f32(128, BN, A_MN, B_MN);
    bool ok = true;
    for (int i = 0; i < nkc; ++i) {
      const int s = i % kGemmStages;
      if (!mbar_wait(&full[s], (i / kGemmStages) & 1)) {
        raise_fault(FAULT_WAIT_FULL);
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t a_base = smem_u32(sbase + s * STAGE);
      const uint32_t b_base = a_base + A_BYTES;
#pragma unroll
      for (int kk = 0; kk < BK / 16; ++kk) {
        const uint64_t ad = A_MN ? sdesc_sw128(a_base + kk * 2048, A_BYTES / 2, 1024)
                                 : sdesc_sw128(a_base + kk * 32, 16, 1024);
        const uint64_t bd = B_MN ? sdesc_sw128(b_base + kk * 2048, 64 * BK * 2, 1024)
                                 : sdesc_sw128(b_base + kk * 32, 16, 1024);
        umma_bf16(tmem, ad, bd, idesc, (i | kk) != 0);
      }
      umma_commit(&empty[s]);
    }
    if (ok && nkc > 0) umma_commit(done);
  }
  __syncwarp();

  // ---------------- epilogue: TMEM -> fp32 rows ----------------
  const bool have = nkc > 0;
  if (have && !mbar_wait(done, 0)) raise_fault(FAULT_WAIT_DONE);
  tc_fence_after();
  const int m = m0 + warp * 32 + lane;
  const uint32_t taddr = tmem + (static_cast<uint32_t>(warp * 32) << 16);
  float* out = g.out + static_cast<size_t>(split) * g.M * g.N;
#pragma unroll 1
  for (int j0 = 0; j0 < BN; j0 += 16) {
    float v[16];
    if (have) {
      tmem_ld16(taddr + j0, v);
    } else {
#pragma unroll
      for (int q = 0; q < 16; ++q) v[q] = 0.f;
    }
    if (m < g.M) {
      float* row = out + static_cast<size_t>(m) * g.N;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int n = n0 + j0 + 4 * q;
        if (n + 3 < g.N) {
          float4 val = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
          float4* dst = reinterpret_cast<float4*>(row + n);
          if (g.accumulate) {
            const float4 o = *dst;
            val.x += o.x; val.y += o.y; val.z += o.z; val.w += o.w;
          }
          *dst = val;
        } else {
#pragma unroll
          for (int e = 0; e < 4; ++e)
            if (n + e < g.N) row[n + e] = g.accumulate ? row[n + e] + v[4 * q + e] : v[4 * q + e];
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, BN);
}

// fp32 path: one thread per output element, plain FFMA.
__global__ void k_gemm_f32(const float* __restrict__ A, const float* __restrict__ Bm, GemmArgs g) {
  const int n = blockIdx.x * blockDim.x + threadIdx.x;
  const int m = blockIdx.y;
  if (n >= g.N) return;
  float acc = 0.f;
  for (int k = 0; k < g.K; ++k) {
    const float av = g.a_mn_major ? A[static_cast<size_t>(k) * g.M + m] : A[static_cast<size_t>(m) * g.K + k];
    const float bv = g.b_mn_major ? Bm[static_cast<size_t>(k) * g.N + n] : Bm[static_cast<size_t>(n) * g.K + k];
    acc = fmaf(av, bv, acc);
  }
  float* dst = g.out + static_cast<size_t>(m) * g.N + n;
  *dst = g.accumulate ? *dst + acc : acc;
}

template <int BN, int A_MN, int B_MN>
cudaError_t launch_cfg(const CUtensorMap& ta, const CUtensorMap& tb, const GemmArgs& g,
                       cudaStream_t st) {
  const size_t bytes = gemm_bf16_smem_bytes(g);
  static size_t configured_ = 0;
  if (bytes > configured_) {
    cudaError_t e = cudaFuncSetAttribute(k_gemm_bf16<BN, A_MN, B_MN>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(bytes));
    if (e != cudaSuccess) return e;
    configured_ = bytes;
  }
  dim3 grid((g.N + BN - 1) / BN, (g.M + BM - 1) / BM, g.splits);
  k_gemm_bf16<BN, A_MN, B_MN><<<grid, 128, bytes, st>>>(ta, tb, g);
  count_launches(1);
  return cudaGetLastError();
}

template <int A_MN, int B_MN>
cudaError_t launch_bn(const CUtensorMap& ta, const CUtensorMap& tb, const GemmArgs& g,
                      cudaStream_t st) {
  switch (g.BN) {
    case 64: return launch_cfg<64, A_MN, B_MN>(ta, tb, g, st);
    case 128: return launch_cfg<128, A_MN, B_MN>(ta, tb, g, st);
    case 256: return launch_cfg<256, A_MN, B_MN>(ta, tb, g, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

size_t gemm_bf16_smem_bytes(const GemmArgs& g) {
  return kGemmStages * (A_BYTES + b_bytes(g.BN)) + 256 + 1024;
}

cudaError_t launch_gemm_bf16(const CUtensorMap& ta, const CUtensorMap& tb, const GemmArgs& g,
                             cudaStream_t st) {
  if (g.a_mn_major && g.b_mn_major) return launch_bn<1, 1>(ta, tb, g, st);
  if (!g.a_mn_major && g.b_mn_major) return launch_bn<0, 1>(ta, tb, g, st);
  if (g.a_mn_major && !g.b_mn_major) return launch_bn<1, 0>(ta, tb, g, st);
  return launch_bn<0, 0>(ta, tb, g, st);
}

cudaError_t launch_gemm_f32(const GemmArgs& g, const float* A, const float* Bm, cudaStream_t st) {
  dim3 grid((g.N + 127) / 128, g.M);
  k_gemm_f32<<<grid, 128, 0, st>>>(A, Bm, g);
  count_launches(1);
  return cudaGetLastError();
}

INSTANT_FAULT_READER(read_fault_gemm)

}  // namespace instant
