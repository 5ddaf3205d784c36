// expand.cu -- rank-R expansion of the input gradient (page "INSTANT:
// Compressing Gradients and Activations for Resource-Efficient Training",
// 关键设计 3):  g_tilde_x,b = Q^T g_hat_x,b,   [L, Ry] x [Ry, Cx] per sample.
//
// The step writes the full [B, L, Cx] gradient while reading only Q and the
// small g_hat_x, so it is bound by HBM writes.  With 2*Ry flops per output
// element the FFMA pipes cannot keep up with the write stream at Ry >= 8, so
// the contraction runs on the tensor cores.
//
// One CTA owns one BN-column strip of the output for one sample (or a few
// consecutive samples when the token axis is short) and walks its 128-token
// tiles:
//   warp 0  TMA producer: the strip's g_hat_x block once per sample (MN-major
//           B operand, two buffers), then Q^T tiles (MN-major A operand, read
//           straight from Q [Ry, L]) through a ring;
//   warp 1  MMA issuer: one K = Ry (padded to 16) tcgen05 MMA chain per tile
//           into one of two TMEM accumulators (double buffered);
//   warps 2-9  epilogue (two warps per TMEM lane quarter, split by columns):
//           TMEM -> bf16 -> 128-byte-swizzled staging tile -> TMA bulk store,
//           two staging buffers in flight, so the MMA of tile t+1 and the
//           store of tile t overlap.
// Full 128-byte lines leave the SM through the TMA engine; rows past L are
// clipped by the tensor map.
#include "kernels.h"
#include "tc.cuh"

namespace instant {

namespace {

constexpr int BM = 128;
constexpr int BOX = BM * 128;  // one staging box: 128 rows x 64 bf16

struct Lay {
  uint32_t stg, b, a, bar, a_stage, b_bytes, total;
};

__host__ __device__ inline Lay expand_layout(int BN, int KR) {
  Lay l;
  l.stg = 0;
  l.b = 4 * (BN / 64) * BOX;
  l.b_bytes = (BN / 64) * KR * 128;
  l.a = l.b + 2 * l.b_bytes;  // two g_hat_x strips: the next sample's loads early
  l.a_stage = 2 * KR * 128;
  l.bar = l.a + kExpandStages * l.a_stage;
  l.total = l.bar + 256;
  return l;
}

template <int BN>
// two CTAs per SM: at most 102 registers a thread (with more, as an
// instrumented build once had, the SM held one CTA and the grid ran in two waves)
__global__ void __launch_bounds__(320, 2)
    k_expand_bf16(const __grid_constant__ CUtensorMap tmap_q,
                  const __grid_constant__ CUtensorMap tmap_g,
                  const __grid_constant__ CUtensorMap tmap_out, ExpandArgs e) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const Lay lay = expand_layout(BN, e.KR);
  uint8_t* stg = smem + lay.stg;
  uint8_t* sB = smem + lay.b;
  uint8_t* sA = smem + lay.a;
  uint64_t* a_full = reinterpret_cast<uint64_t*>(smem + lay.bar);
  uint64_t* a_empty = a_full + kExpandStages;
  uint64_t* b_full = a_empty + kExpandStages;   // [2]
  uint64_t* b_empty = b_full + 2;               // [2]
  uint64_t* t_full = b_empty + 2;
  uint64_t* t_empty = t_full + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(t_empty + 2);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int n0 = blockIdx.x * BN;
  // samples b0 .. b1-1 of this CTA, each walked over its token tiles: job j is
  // (sample b0 + j / nlt, token tile j % nlt)
  const int b0 = blockIdx.y * e.spb;
  const int b1 = min(e.B, b0 + e.spb);
  const int njobs = (b1 - b0) * e.nlt;
  const int KR = e.KR;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kExpandStages; ++s) {
      mbar_init(&a_full[s], 1);
      mbar_init(&a_empty[s], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&b_full[i], 1);
      mbar_init(&b_empty[i], 1);
      mbar_init(&t_full[i], 1);
      mbar_init(&t_empty[i], 4);  // one arrival per warp of the epilogue group
    }
    fence_barrier_init();
    if (e.q_tma) prefetch_tmap(&tmap_q);
    prefetch_tmap(&tmap_g);
    prefetch_tmap(&tmap_out);
  }
  if (warp == 0) {
    tmem_alloc(tmem_slot, 2 * BN);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  pdl_launch_dependents();
  pdl_wait();
  // Q^T tiles filled by threads (no TMA: L % 8 != 0) stay resident when they
  // all fit the ring: every sample of the CTA reuses them
  const bool res = !e.q_tma && e.nlt <= kExpandStages;
  if (res) {
    const uint16_t* Q = static_cast<const uint16_t*>(e.Q);
    for (int idx = threadIdx.x; idx < e.nlt * KR * BM; idx += blockDim.x) {
      const int t = idx / (KR * BM);
      const int rem = idx - t * (KR * BM);
      const int r = rem / BM;
      const int ll = rem - r * BM;
      const int l = t * BM + ll;
      const uint16_t v = (r < e.Ry && l < e.L) ? Q[static_cast<size_t>(r) * e.L + l] : 0;
      *reinterpret_cast<uint16_t*>(sA + t * lay.a_stage + (ll >> 6) * KR * 128 + sw128_offset(r, ll & 63)) = v;
    }
    fence_proxy_async_smem();
    __syncthreads();
  }

  if (warp == 0) {
    // ---------------- producer ----------------
    const uint16_t* Q = static_cast<const uint16_t*>(e.Q);
    int issued = 0, nb = 0;
    int s = 0, par = 0;     // ring slot and round parity of job j
    int lt = 0, sj = 0;     // token tile and sample index (within the CTA) of job j
    bool ok = true;
    for (int j = 0; ok && j < njobs; ++j) {
      if (lt == 0) {
        // the g_hat_x strip of sample b0 + sj into buffer sj & 1
        if (lane == 0) {
          const int bi = sj & 1;
          if (sj >= 2 && !mbar_wait(&b_empty[bi], ((sj >> 1) - 1) & 1)) {
            raise_fault(FAULT_WAIT_EMPTY);
            ok = false;
          } else {
            mbar_arrive_expect_tx(&b_full[bi], lay.b_bytes);
            for (int h = 0; h < BN / 64; ++h)
              tma_load_3d(sB + bi * lay.b_bytes + h * KR * 128, &tmap_g, &b_full[bi], n0 + 64 * h, 0,
                          b0 + sj);
            ++nb;
          }
        }
        ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
        if (!ok) break;
      }
      if (res) {
        if (++lt == e.nlt) {
          lt = 0;
          ++sj;
        }
        continue;
      }
      if (lane == 0 && j >= kExpandStages && !mbar_wait(&a_empty[s], par ^ 1)) {
        raise_fault(FAULT_WAIT_EMPTY);
        ok = false;
      }
      ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
      if (!ok) break;
      uint8_t* dst = sA + s * lay.a_stage;
      const int l0 = lt * BM;
      if (e.q_tma) {
        if (lane == 0) {
          mbar_arrive_expect_tx(&a_full[s], lay.a_stage);
          tma_load_2d(dst, &tmap_q, &a_full[s], l0, 0);
          tma_load_2d(dst + KR * 128, &tmap_q, &a_full[s], l0 + 64, 0);
        }
      } else {
        // A[k][l] MN-major: two 64-token atoms, KR rows of 128 B each
        for (int idx = lane; idx < KR * BM; idx += 32) {
          const int r = idx / BM;
          const int ll = idx - r * BM;
          const int l = l0 + ll;
          const uint16_t v = (r < e.Ry && l < e.L) ? Q[static_cast<size_t>(r) * e.L + l] : 0;
          *reinterpret_cast<uint16_t*>(dst + (ll >> 6) * KR * 128 + sw128_offset(r, ll & 63)) = v;
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&a_full[s]);
      }
      ++issued;
      if (++s == kExpandStages) {
        s = 0;
        par ^= 1;
      }
      if (++lt == e.nlt) {
        lt = 0;
        ++sj;
      }
    }
    if (lane == 0) {
      for (int k = 0; k < kExpandStages && k < issued; ++k) {
        if (--s < 0) {
          s = kExpandStages - 1;
          par ^= 1;
        }
        if (!mbar_wait(&a_full[s], par)) raise_fault(FAULT_WAIT_FULL);
      }
      if (nb > 0 && !mbar_wait(&b_full[(nb - 1) & 1], ((nb - 1) >> 1) & 1)) raise_fault(FAULT_WAIT_FULL);
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(128, BN, /*a_mn=*/1, /*b_mn=*/1);
      int s = 0, par = 0, lt = 0, sj = 0;
      for (int j = 0; j < njobs; ++j) {
        const int bi = sj & 1;
        if (lt == 0 && !mbar_wait(&b_full[bi], (sj >> 1) & 1)) {
          raise_fault(FAULT_WAIT_FULL);
          break;
        }
        const int buf = j & 1;
        if (j >= 2 && !mbar_wait(&t_empty[buf], ((j >> 1) - 1) & 1)) {
          raise_fault(FAULT_WAIT_EMPTY);
          break;
        }
        if (!res && !mbar_wait(&a_full[s], par)) {
          raise_fault(FAULT_WAIT_FULL);
          break;
        }
        tc_fence_after();
        const uint32_t a_base = smem_u32(sA + (res ? lt : s) * lay.a_stage);
        const uint32_t b_base = smem_u32(sB + bi * lay.b_bytes);
        for (int kk = 0; kk < KR / 16; ++kk) {
          const uint64_t ad = sdesc_sw128(a_base + kk * 2048, KR * 128, 1024);
          const uint64_t bd = sdesc_sw128(b_base + kk * 2048, KR * 128, 1024);
          umma_bf16(tmem + buf * BN, ad, bd, idesc, kk != 0);
        }
        if (!res) umma_commit(&a_empty[s]);
        umma_commit(&t_full[buf]);
        if (++s == kExpandStages) {
          s = 0;
          par ^= 1;
        }
        if (++lt == e.nlt) {
          lt = 0;
          ++sj;
          if (j + 1 < njobs) umma_commit(&b_empty[bi]);  // this strip may be replaced
        }
      }
    }
  } else {
    // ---------------- epilogue (warps 2..9) ----------------
    // two groups of four warps (one per TMEM lane quarter); group g handles
    // jobs g, g+2, ... from accumulator g, so two tiles are converted at once.
    // Each group double-buffers its staging and tracks its own store groups.
    const int grp = (warp - 2) >> 2;       // 0 or 1
    const int gt = (threadIdx.x - 64) & 127;  // thread index within the group
    const int quarter = warp & 3;          // TMEM lanes this warp may read
    const int row = quarter * 32 + lane;   // token row within the tile
    int it = 0;
    for (int j = grp; j < njobs; j += 2, ++it) {
      const int sj = j / e.nlt;
      const int lt = j - sj * e.nlt;
      uint8_t* st = stg + (2 * grp + (it & 1)) * (BN / 64) * BOX;
      if (gt == 0 && it >= 2) tma_store_wait_read<1>();
      if (grp == 0) named_barrier<1>(128); else named_barrier<2>(128);
      if (!mbar_wait(&t_full[grp], it & 1)) raise_fault(FAULT_WAIT_DONE);
      tc_fence_after();
      const uint32_t taddr = tmem + grp * BN + (static_cast<uint32_t>(quarter * 32) << 16);
#pragma unroll 1
      for (int h = 0; h < BN / 64; ++h) {
        float v[64];
        tmem_ld64(taddr + 64 * h, v);
        if (h == BN / 64 - 1) {
          // this warp has read its lanes of the accumulator: hand it back to
          // the MMA issuer before converting
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&t_empty[grp]);
        }
        uint8_t* box = st + h * BOX + row * 128;
#pragma unroll
        for (int q = 0; q < 8; ++q)
          *reinterpret_cast<uint4*>(box + ((q ^ (row & 7)) << 4)) =
              make_uint4(pack_bf16x2(v[8 * q], v[8 * q + 1]), pack_bf16x2(v[8 * q + 2], v[8 * q + 3]),
                         pack_bf16x2(v[8 * q + 4], v[8 * q + 5]),
                         pack_bf16x2(v[8 * q + 6], v[8 * q + 7]));
      }
      fence_proxy_async_smem();
      if (grp == 0) named_barrier<1>(128); else named_barrier<2>(128);
      if (gt == 0) {
        for (int h = 0; h < BN / 64; ++h)
          if (n0 + 64 * h < e.Cx) tma_store_3d(&tmap_out, st + h * BOX, n0 + 64 * h, lt * BM, b0 + sj);
        tma_store_commit();
      }
    }
    const int et = gt;
    if (et == 0) tma_store_wait_all();
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, 2 * BN);
}

// fp32 path: one thread per output element.
__global__ void k_expand_f32(ExpandArgs e) {
  const int c = blockIdx.x * blockDim.x + threadIdx.x;
  const int l = blockIdx.y;
  const int b = blockIdx.z;
  if (c >= e.Cx) return;
  const float* Q = static_cast<const float*>(e.Q);
  const float* g = static_cast<const float*>(e.gxh);
  float acc = 0.f;
  for (int r = 0; r < e.Ry; ++r)
    acc = fmaf(Q[static_cast<size_t>(r) * e.L + l], g[(static_cast<size_t>(b) * e.Ry + r) * e.Cx + c],
               acc);
  static_cast<float*>(e.out)[(static_cast<size_t>(b) * e.L + l) * e.Cx + c] = acc;
}

template <int BN>
cudaError_t launch_bn(const CUtensorMap& tq, const CUtensorMap& tg, const CUtensorMap& to,
                      const ExpandArgs& e, cudaStream_t st) {
  const size_t bytes = expand_bf16_smem_bytes(e);
  static size_t configured_ = 0;
  if (bytes > configured_) {
    cudaError_t err = cudaFuncSetAttribute(k_expand_bf16<BN>,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           static_cast<int>(bytes));
    if (err != cudaSuccess) return err;
    configured_ = bytes;
  }
  if (e.spb < 1) return cudaErrorInvalidValue;
  return launch_ex(k_expand_bf16<BN>, dim3((e.Cx + BN - 1) / BN, (e.B + e.spb - 1) / e.spb), dim3(320),
                   bytes, st, 1, pdl_enabled(), tq, tg, to, e);
}

}  // namespace

size_t expand_bf16_smem_bytes(const ExpandArgs& e) { return expand_layout(e.BN, e.KR).total + 1024; }

cudaError_t launch_expand_bf16(const CUtensorMap& tmap_q, const CUtensorMap& tmap_g,
                               const CUtensorMap& tmap_out, const ExpandArgs& e, cudaStream_t st) {
  switch (e.BN) {
    case 64: return launch_bn<64>(tmap_q, tmap_g, tmap_out, e, st);
    case 128: return launch_bn<128>(tmap_q, tmap_g, tmap_out, e, st);
    case 256: return launch_bn<256>(tmap_q, tmap_g, tmap_out, e, st);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_expand_f32(const ExpandArgs& e, cudaStream_t st) {
  dim3 grid((e.Cx + 127) / 128, e.L, e.B);
  k_expand_f32<<<grid, 128, 0, st>>>(e);
  count_launches(1);
  return cudaGetLastError();
}

INSTANT_FAULT_READER(read_fault_expand)

}  // namespace instant
