// syrk.cu -- calibration statistic of INSTANT (page "INSTANT: Compressing
// Gradients and Activations for Resource-Efficient Training", 关键设计 1):
//   C[i, j] += sum_b sum_c t[b, i, c] * t[b, j, c]      (t = x or g_y)
// i.e. the token-by-token autocorrelation accumulated over a batch without
// storing the batch.  This is the one truly tensor-bound step (2L flops per
// byte of t), so it is a tcgen05 GEMM over the upper triangle of C: both
// operands are K-major row blocks of the same sample (K = channels), streamed
// by TMA; the sum over samples continues the K loop.  Two tile shapes:
//   * wide (the default): 128 x 256 tiles -- row block bi against the column
//     blocks bj, bj + 1 (bj = bi + 2p) -- one CTA per SM with a 4-stage ring of
//     48 KB.  Per 64-channel chunk it reads 48 KB for 4.2 MFLOP (a 128 x 128
//     tile reads 32 KB for 2.1 MFLOP): with 128 x 128 tiles every SM needs
//     ~96 B/clk of operands at the tensor peak, more than L2 delivers to all
//     SMs at once.  A pair on the diagonal (bj = bi) loads its 256 rows once
//     and takes the first 128 as the A operand;
//   * narrow: 128 x 128 tiles, two CTAs per SM with a 3-stage ring of 32 KB.  Grid y splits
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

constexpr int BT = 128;                  // tile edge (rows; columns of a narrow tile)
constexpr int BK = 64;                   // channels per stage
constexpr int TILE_BYTES = BT * BK * 2;  // 16 KB

template <bool WIDE>
struct SyrkShape {
  static constexpr int BN = WIDE ? 2 * BT : BT;                  // tile columns
  static constexpr int STAGE = TILE_BYTES + BN * BK * 2;         // A rows + B rows
  static constexpr int STAGES = WIDE ? kSyrkWideStages : kSyrkStages;
};

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

// wide tiles: t enumerates (bi, bj = bi + 2p), row by row; bj + 1 may be past
// the last block (its rows load as zeros and are not stored)
__device__ __forceinline__ void pair_coords(int t, int nblk, int& bi, int& bj) {
  int i = 0;
  int rem = t;
  while (rem >= (nblk - i + 1) / 2) {
    rem -= (nblk - i + 1) / 2;
    ++i;
  }
  bi = i;
  bj = i + 2 * rem;
}

template <bool WIDE>
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
  using SH = SyrkShape<WIDE>;
  constexpr int STAGE = SH::STAGE;
  constexpr int NS = SH::STAGES;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + NS * STAGE);
  uint64_t* empty = full + NS;
  uint64_t* done = empty + NS;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  int bi, bj;
  if (WIDE)
    pair_coords(blockIdx.x, a.nblk, bi, bj);
  else
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
    for (int s = 0; s < NS; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(done, 1);
    fence_barrier_init();
    prefetch_tmap(&tmap_t);
  }
  if (warp == 0) {
    tmem_alloc(tmem_slot, SH::BN);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  pdl_launch_dependents();
  pdl_wait();

  if (warp == 0 && lane == 0) {
    // narrow: A rows at the stage start, B rows after them (none on the
    // diagonal); wide: B's 256 rows after the A slot, A's own rows only off
    // the diagonal (on it, A is B's first half)
    const uint32_t bytes = diag ? (WIDE ? 2 * TILE_BYTES : TILE_BYTES) : STAGE;
    int issued = 0;
    // (sample, channel chunk) of iteration it, kept without divisions
    int b = b_lo, kc = kc_lo;
    int s = 0;
    for (int it = 0; it < niter; ++it) {
      if (it >= NS && !mbar_wait(&empty[s], ((it / NS) - 1) & 1)) {
        raise_fault(FAULT_WAIT_EMPTY);
        break;
      }
      const int c0 = kc * BK;
      uint8_t* dst = smem + s * STAGE;
      mbar_arrive_expect_tx(&full[s], bytes);
      if (WIDE) {
        if (!diag) tma_load_3d(dst, &tmap_t, &full[s], c0, i0, b);
        tma_load_3d(dst + TILE_BYTES, &tmap_t, &full[s], c0, j0, b);
        tma_load_3d(dst + 2 * TILE_BYTES, &tmap_t, &full[s], c0, j0 + BT, b);
      } else {
        tma_load_3d(dst, &tmap_t, &full[s], c0, i0, b);
        if (!diag) tma_load_3d(dst + TILE_BYTES, &tmap_t, &full[s], c0, j0, b);
      }
      ++issued;
      if (++kc == kc_hi) {
        kc = kc_lo;
        ++b;
      }
      if (++s == NS) s = 0;
    }
    for (int it = issued - NS < 0 ? 0 : issued - NS; it < issued; ++it)
      if (!mbar_wait(&full[it % NS], (it / NS) & 1)) raise_fault(FAULT_WAIT_FULL);
  } else if (warp == 1 && lane == 0) {
    constexpr uint32_t idesc = idesc_bf16_f32(128, SH::BN, 0, 0);
    bool ok = true;
    int s = 0, par = 0;
    for (int it = 0; it < niter; ++it) {
      if (!mbar_wait(&full[s], par)) {
        raise_fault(FAULT_WAIT_FULL);
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t stage = smem_u32(smem + s * STAGE);
      const uint32_t b_base = (WIDE || !diag) ? stage + TILE_BYTES : stage;
      const uint32_t a_base = (WIDE && diag) ? b_base : stage;
#pragma unroll
      for (int kk = 0; kk < BK / 16; ++kk) {
        const uint64_t ad = sdesc_sw128(a_base + kk * 32, 16, 1024);
        const uint64_t bd = sdesc_sw128(b_base + kk * 32, 16, 1024);
        umma_bf16(tmem, ad, bd, idesc, (it | kk) != 0);
      }
      umma_commit(&empty[s]);
      if (++s == NS) {
        s = 0;
        par ^= 1;
      }
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
    for (int jc = 0; jc < SH::BN; jc += 16) {
      float v[16];
      tmem_ld16(taddr + jc, v);
      const int j = j0 + jc;
      // a column block other than the row block also lands mirrored
      const bool mirror = !diag || jc >= BT;
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
        if (mirror) {
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
  if (warp == 0) tmem_dealloc(tmem, SH::BN);
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

template <bool WIDE>
size_t syrk_smem_bytes() {
  return SyrkShape<WIDE>::STAGES * SyrkShape<WIDE>::STAGE + 256 + 1024;
}

template <bool WIDE>
cudaError_t configure_syrk() {
  return raise_smem_limit(reinterpret_cast<const void*>(k_syrk_bf16<WIDE>), syrk_smem_bytes<WIDE>());
}

}  // namespace

size_t syrk_bf16_smem_bytes(bool wide) { return wide ? syrk_smem_bytes<true>() : syrk_smem_bytes<false>(); }

cudaError_t launch_syrk_bf16_batch(const CUtensorMap* tmaps, const SyrkBatch& b, cudaStream_t st) {
  if (b.count < 1 || b.count > kMaxSyrkBatch || b.split0[0] != 0) return cudaErrorInvalidValue;
  for (int p = 0; p < b.count; ++p)
    if (b.s[p].L != b.s[0].L || b.split0[p + 1] != b.split0[p] + b.s[p].splits || b.s[p].splits < 1 ||
        b.s[p].cs < 1 || b.s[p].bs < 1 || b.s[p].cs * b.s[p].bs != b.s[p].splits)
      return cudaErrorInvalidValue;
  const cudaError_t e = b.wide ? configure_syrk<true>() : configure_syrk<false>();
  if (e != cudaSuccess) return e;
  const CUtensorMap& m0 = tmaps[0];
  const CUtensorMap& m1 = tmaps[b.count > 1 ? 1 : 0];
  const CUtensorMap& m2 = tmaps[b.count > 2 ? 2 : 0];
  const CUtensorMap& m3 = tmaps[b.count > 3 ? 3 : 0];
  const dim3 grid(b.s[0].ntiles, b.split0[b.count]);
  if (b.wide)
    return launch_ex(k_syrk_bf16<true>, grid, dim3(128), syrk_smem_bytes<true>(), st, 1, pdl_enabled(),
                     m0, m1, m2, m3, b);
  return launch_ex(k_syrk_bf16<false>, grid, dim3(128), syrk_smem_bytes<false>(), st, 1, pdl_enabled(),
                   m0, m1, m2, m3, b);
}

cudaError_t launch_syrk_bf16(const CUtensorMap& tmap_t, const SyrkArgs& s, cudaStream_t st) {
  SyrkBatch b;
  b.s[0] = s;
  b.split0[0] = 0;
  b.split0[1] = s.splits;
  b.count = 1;
  b.wide = 0;
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
