// syrk.cu -- calibration statistic of INSTANT (page "INSTANT: Compressing
// Gradients and Activations for Resource-Efficient Training", 关键设计 1):
//   C[i, j] += sum_b sum_c t[b, i, c] * t[b, j, c]      (t = x or g_y)
// i.e. the token-by-token autocorrelation accumulated over a batch without
// storing the batch.  This is the one truly tensor-bound step (2L flops per
// byte of t), so it is a tcgen05 GEMM over the upper-triangle 128x128 tiles of
// C: both operands are K-major row blocks of the same sample (K = channels),
// streamed by TMA; the sum over samples continues the K loop.  Grid y splits
// each tile's work into channel ranges (every CTA walks all of its samples in
// order, so the CTAs running at one time read the same sample and its tiles
// meet in L2) and, for small statistics only, sample ranges; the host sizes
// the splits so that the CTAs carry equal work and fill whole waves of two
// CTAs per SM.  Every CTA adds its tile (and, off the diagonal, the mirrored
// tile) into C with fp32 atomics.
#include "kernels.h"
#include "tc.cuh"

namespace instant {

namespace {

constexpr int BT = 128;                  // tile edge
constexpr int BK = 64;                   // channels per stage
constexpr int TILE_BYTES = BT * BK * 2;  // 16 KB
constexpr int STAGE = 2 * TILE_BYTES;

__device__ __forceinline__ void tile_coords(int t, int nblk, int& bi, int& bj) {
  // t enumerates (bi, bj), bi <= bj, row by row
  int i = 0;
  int rem = t;
  while (rem >= nblk - i) {
    rem -= nblk - i;
    ++i;
  }
  bi = i;
  bj = i + rem;
}

__global__ void __launch_bounds__(128, 1)
    k_syrk_bf16(const __grid_constant__ CUtensorMap tmap0, const __grid_constant__ CUtensorMap tmap1,
                const __grid_constant__ CUtensorMap tmap2, const __grid_constant__ CUtensorMap tmap3,
                const __grid_constant__ SyrkBatch batch) {
  // the problem of this grid row
  int p = 0;
  while (p + 1 < batch.count && static_cast<int>(blockIdx.y) >= batch.split0[p + 1]) ++p;
  const SyrkArgs& a = batch.s[p];
  const CUtensorMap& tmap_t = p == 0 ? tmap0 : (p == 1 ? tmap1 : (p == 2 ? tmap2 : tmap3));
  // split index -> (channel range, sample range): every CTA walks its samples
  // in order, each over its own channel chunks
  const int split = static_cast<int>(blockIdx.y) - batch.split0[p];
  const int ks = split % a.cs;
  const int bsx = split / a.cs;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kSyrkStages * STAGE);
  uint64_t* empty = full + kSyrkStages;
  uint64_t* done = empty + kSyrkStages;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  int bi, bj;
  tile_coords(blockIdx.x, a.nblk, bi, bj);
  const bool diag = bi == bj;
  const int i0 = bi * BT;
  const int j0 = bj * BT;
  const int kc_lo = static_cast<int>(static_cast<long long>(a.nkc) * ks / a.cs);
  const int kc_hi = static_cast<int>(static_cast<long long>(a.nkc) * (ks + 1) / a.cs);
  const int b_lo = static_cast<int>(static_cast<long long>(a.B) * bsx / a.bs);
  const int b_hi = static_cast<int>(static_cast<long long>(a.B) * (bsx + 1) / a.bs);
  const int niter = (kc_hi - kc_lo) * (b_hi - b_lo);

  if (threadIdx.x == 0) {
    for (int s = 0; s < kSyrkStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(done, 1);
    fence_barrier_init();
    prefetch_tmap(&tmap_t);
  }
  if (warp == 0) {
    tmem_alloc(tmem_slot, BT);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  pdl_launch_dependents();
  pdl_wait();

  if (warp == 0 && lane == 0) {
    const uint32_t bytes = diag ? TILE_BYTES : STAGE;
    int issued = 0;
    // (sample, channel chunk) of iteration it, kept without divisions
    int b = b_lo, kc = kc_lo;
    for (int it = 0; it < niter; ++it) {
      const int s = it % kSyrkStages;
      if (it >= kSyrkStages && !mbar_wait(&empty[s], ((it / kSyrkStages) - 1) & 1)) {
        raise_fault(FAULT_WAIT_EMPTY);
        break;
      }
      const int c0 = kc * BK;
      uint8_t* dst = smem + s * STAGE;
      mbar_arrive_expect_tx(&full[s], bytes);
      tma_load_3d(dst, &tmap_t, &full[s], c0, i0, b);
      if (!diag) tma_load_3d(dst + TILE_BYTES, &tmap_t, &full[s], c0, j0, b);
      ++issued;
      if (++kc == kc_hi) {
        kc = kc_lo;
        ++b;
      }
    }
    for (int it = issued - kSyrkStages < 0 ? 0 : issued - kSyrkStages; it < issued; ++it)
      if (!mbar_wait(&full[it % kSyrkStages], (it / kSyrkStages) & 1)) raise_fault(FAULT_WAIT_FULL);
  } else if (warp == 1 && lane == 0) {
    constexpr uint32_t idesc = idesc_bf16_f32(128, 128, 0, 0);
    bool ok = true;
    for (int it = 0; it < niter; ++it) {
      const int s = it % kSyrkStages;
      if (!mbar_wait(&full[s], (it / kSyrkStages) & 1)) {
        raise_fault(FAULT_WAIT_FULL);
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t a_base = smem_u32(smem + s * STAGE);
      const uint32_t b_base = diag ? a_base : a_base + TILE_BYTES;
#pragma unroll
      for (int kk = 0; kk < BK / 16; ++kk) {
        const uint64_t ad = sdesc_sw128(a_base + kk * 32, 16, 1024);
        const uint64_t bd = sdesc_sw128(b_base + kk * 32, 16, 1024);
        umma_bf16(tmem, ad, bd, idesc, (it | kk) != 0);
      }
      umma_commit(&empty[s]);
    }
    if (ok && niter > 0) umma_commit(done);
  }
  __syncwarp();

  if (niter > 0) {
    if (!mbar_wait(done, 0)) raise_fault(FAULT_WAIT_DONE);
    tc_fence_after();
    const int i = i0 + warp * 32 + lane;
    const uint32_t taddr = tmem + (static_cast<uint32_t>(warp * 32) << 16);
    const bool vec_ok = (a.L & 3) == 0;
#pragma unroll 1
    for (int jc = 0; jc < BT; jc += 16) {
      float v[16];
      tmem_ld16(taddr + jc, v);
      const int j = j0 + jc;
      if (i < a.L) {
        float* row = a.Cout + static_cast<size_t>(i) * a.L;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int jj = j + 4 * q;
          if (vec_ok && jj + 3 < a.L) {
            atomicAdd(reinterpret_cast<float4*>(row + jj),
                      make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]));
          } else {
#pragma unroll
            for (int e2 = 0; e2 < 4; ++e2)
              if (jj + e2 < a.L) atomicAdd(row + jj + e2, v[4 * q + e2]);
          }
        }
        if (!diag) {
          // mirrored tile: C[j, i] += D[i, j]; lanes write consecutive i
#pragma unroll
          for (int q = 0; q < 16; ++q)
            if (j + q < a.L) atomicAdd(a.Cout + static_cast<size_t>(j + q) * a.L + i, v[q]);
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, BT);
}

// fp32 path: one thread per (i, j), full matrix.
__global__ void k_syrk_f32(const float* __restrict__ t, SyrkArgs a) {
  const int j = blockIdx.x * blockDim.x + threadIdx.x;
  const int i = blockIdx.y;
  if (j >= a.L) return;
  float acc = 0.f;
  for (int b = 0; b < a.B; ++b) {
    const float* ti = t + (static_cast<size_t>(b) * a.L + i) * a.C;
    const float* tj = t + (static_cast<size_t>(b) * a.L + j) * a.C;
    for (int c = 0; c < a.C; ++c) acc = fmaf(ti[c], tj[c], acc);
  }
  a.Cout[static_cast<size_t>(i) * a.L + j] += acc;
}

}  // namespace

size_t syrk_bf16_smem_bytes() { return kSyrkStages * STAGE + 256 + 1024; }

cudaError_t launch_syrk_bf16_batch(const CUtensorMap* tmaps, const SyrkBatch& b, cudaStream_t st) {
  if (b.count < 1 || b.count > kMaxSyrkBatch || b.split0[0] != 0) return cudaErrorInvalidValue;
  for (int p = 0; p < b.count; ++p)
    if (b.s[p].L != b.s[0].L || b.split0[p + 1] != b.split0[p] + b.s[p].splits || b.s[p].splits < 1 ||
        b.s[p].cs < 1 || b.s[p].bs < 1 || b.s[p].cs * b.s[p].bs != b.s[p].splits)
      return cudaErrorInvalidValue;
  const size_t bytes = syrk_bf16_smem_bytes();
  static size_t configured_ = 0;
  if (bytes > configured_) {
    cudaError_t e = cudaFuncSetAttribute(k_syrk_bf16, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(bytes));
    if (e != cudaSuccess) return e;
    configured_ = bytes;
  }
  const CUtensorMap& m0 = tmaps[0];
  const CUtensorMap& m1 = tmaps[b.count > 1 ? 1 : 0];
  const CUtensorMap& m2 = tmaps[b.count > 2 ? 2 : 0];
  const CUtensorMap& m3 = tmaps[b.count > 3 ? 3 : 0];
  return launch_ex(k_syrk_bf16, dim3(b.s[0].ntiles, b.split0[b.count]), dim3(128), bytes, st, 1,
                   pdl_enabled(), m0, m1, m2, m3, b);
}

cudaError_t launch_syrk_bf16(const CUtensorMap& tmap_t, const SyrkArgs& s, cudaStream_t st) {
  SyrkBatch b;
  b.s[0] = s;
  b.split0[0] = 0;
  b.split0[1] = s.splits;
  b.count = 1;
  return launch_syrk_bf16_batch(&tmap_t, b, st);
}

cudaError_t launch_syrk_f32(const SyrkArgs& s, const float* t, cudaStream_t st) {
  dim3 grid((s.L + 127) / 128, s.L);
  k_syrk_f32<<<grid, 128, 0, st>>>(t, s);
  count_launches(1);
  return cudaGetLastError();
}

INSTANT_FAULT_READER(read_fault_syrk)

}  // namespace instant
