// expand.cu -- rank-R expansion of the input gradient (page "INSTANT:
// Compressing Gradients and Activations for Resource-Efficient Training",
// 关键设计 3):  g_tilde_x,b = Q^T g_hat_x,b,   [L, Ry] x [Ry, Cx] per sample.
//
// The step writes the full [B, L, Cx] gradient while reading only Q and the
// small g_hat_x, so it is bound by HBM writes.  With 2*Ry flops per output
// element the FFMA pipes cannot keep up with the write stream at Ry >= 8, so
// the contraction runs on the tensor cores.
//
// The work is a list of jobs, one per (BN-column strip, sample, 128-token
// tile), strip-major; the grid holds as many CTAs as fit on the GPU at once
// and each takes an equal run of consecutive jobs, so the whole expansion is
// one wave whatever B, L and Cx are:
//   warp 0  TMA producer: each (strip, sample) g_hat_x block once (MN-major B
//           operand) through a ring of up to four, then Q^T tiles (MN-major
//           A operand, read straight from Q [Ry, L]) through a ring -- or, for
//           at most four token tiles, all of them once;
//   warp 1  MMA issuer: one K = Ry (padded to 16) tcgen05 MMA chain per job
//           into one of two TMEM accumulators (double buffered);
//   warps 2-9  epilogue (two groups of four warps, one warp per TMEM lane
//           quarter, alternate jobs): TMEM -> bf16 -> 128-byte-swizzled staging
//           tile -> TMA bulk store, two staging buffers per group in flight,
//           so the MMA of job t+1 and the store of job t overlap.
// Full 128-byte lines leave the SM through the TMA engine; rows past L are
// clipped by the tensor map (and lane quarters wholly past L skip their TMEM
// reads).
#include <map>
#include <mutex>
#include <tuple>

#include "kernels.h"
#include "tc.cuh"

namespace instant {

namespace {

constexpr int BM = 128;
constexpr int BOX = BM * 128;  // one staging box: 128 rows x 64 bf16

struct Lay {
  uint32_t stg, b, a, bar, a_stage, b_bytes, total;
};

// nb g_hat_x slots; na Q^T slots (the ring, or the nlt resident tiles)
__host__ __device__ inline Lay expand_layout(int BN, int KR, int nb, int na) {
  Lay l;
  l.stg = 0;
  l.b = 4 * (BN / 64) * BOX;
  l.b_bytes = (BN / 64) * KR * 128;
  l.a = l.b + nb * l.b_bytes;
  l.a_stage = 2 * KR * 128;
  l.bar = l.a + na * l.a_stage;
  l.total = l.bar + 256;
  return l;
}

__host__ __device__ inline int expand_a_slots(const ExpandArgs& e) {
  return (e.qres && e.nlt > kExpandStages) ? e.nlt : kExpandStages;
}

template <int BN>
// two CTAs per SM where shared memory allows: at most 102 registers a thread
__global__ void __launch_bounds__(320, 2)
    k_expand_bf16(const __grid_constant__ CUtensorMap tmap_q,
                  const __grid_constant__ CUtensorMap tmap_g,
                  const __grid_constant__ CUtensorMap tmap_out, ExpandArgs e) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const Lay lay = expand_layout(BN, e.KR, e.nb, expand_a_slots(e));
  uint8_t* stg = smem + lay.stg;
  uint8_t* sB = smem + lay.b;
  uint8_t* sA = smem + lay.a;
  uint64_t* a_full = reinterpret_cast<uint64_t*>(smem + lay.bar);
  uint64_t* a_empty = a_full + kExpandStages;
  uint64_t* b_full = a_empty + kExpandStages;   // [kExpandMaxBRing]
  uint64_t* b_empty = b_full + kExpandMaxBRing;  // [kExpandMaxBRing]
  uint64_t* t_full = b_empty + kExpandMaxBRing;
  uint64_t* t_empty = t_full + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(t_empty + 2);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // this CTA's run of jobs [J0, J1); job J = ((strip * B) + sample) * nlt + lt
  const int J0 = static_cast<int>(static_cast<long long>(blockIdx.x) * e.total / gridDim.x);
  const int J1 = static_cast<int>(static_cast<long long>(blockIdx.x + 1) * e.total / gridDim.x);
  const int njobs = J1 - J0;
  const int lt0 = J0 % e.nlt;
  const int smp0 = (J0 / e.nlt) % e.B;
  const int strip0 = (J0 / e.nlt) / e.B;
  const int KR = e.KR;
  const int nb = e.nb;
  const bool res = e.qres != 0;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kExpandStages; ++s) {
      mbar_init(&a_full[s], 1);
      mbar_init(&a_empty[s], 1);
    }
    for (int i = 0; i < kExpandMaxBRing; ++i) {
      mbar_init(&b_full[i], 1);
      mbar_init(&b_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
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
  // resident Q^T tiles filled by threads (no TMA: L % 8 != 0); every job of
  // the CTA reuses them
  if (res && !e.q_tma) {
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
    int issued = 0, ng = 0;  // Q^T ring loads and g_hat_x blocks issued
    int s = 0, par = 0;      // Q^T ring slot and round parity of job j
    int bs = 0, bpar = 0;    // g_hat_x slot and round parity of the next block
    int lt = lt0, smp = smp0, strip = strip0;
    bool ok = true;
    if (res && e.q_tma && njobs > 0 && lane == 0) {
      // every token tile of Q^T at once, on a_full[0]
      mbar_arrive_expect_tx(&a_full[0], e.nlt * lay.a_stage);
      for (int t = 0; t < e.nlt; ++t) {
        tma_load_2d(sA + t * lay.a_stage, &tmap_q, &a_full[0], t * BM, 0);
        tma_load_2d(sA + t * lay.a_stage + KR * 128, &tmap_q, &a_full[0], t * BM + 64, 0);
      }
    }
    for (int j = 0; ok && j < njobs; ++j) {
      if (j == 0 || lt == 0) {
        // the g_hat_x block of (strip, sample) into slot bs
        if (lane == 0) {
          if (ng >= nb && !mbar_wait(&b_empty[bs], bpar ^ 1)) {
            raise_fault(FAULT_WAIT_EMPTY);
            ok = false;
          } else {
            mbar_arrive_expect_tx(&b_full[bs], lay.b_bytes);
            for (int h = 0; h < BN / 64; ++h)
              tma_load_3d(sB + bs * lay.b_bytes + h * KR * 128, &tmap_g, &b_full[bs],
                          strip * BN + 64 * h, 0, smp);
          }
        }
        ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
        if (!ok) break;
        ++ng;
        if (++bs == nb) {
          bs = 0;
          bpar ^= 1;
        }
      }
      if (!res) {
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
      }
      if (++lt == e.nlt) {
        lt = 0;
        if (++smp == e.B) {
          smp = 0;
          ++strip;
        }
      }
    }
    if (lane == 0) {
      // every copy this CTA issued has landed before it may exit
      for (int k = 0; k < kExpandStages && k < issued; ++k) {
        if (--s < 0) {
          s = kExpandStages - 1;
          par ^= 1;
        }
        if (!mbar_wait(&a_full[s], par)) raise_fault(FAULT_WAIT_FULL);
      }
      for (int k = 0; k < nb && k < ng; ++k) {
        if (--bs < 0) {
          bs = nb - 1;
          bpar ^= 1;
        }
        if (!mbar_wait(&b_full[bs], bpar)) raise_fault(FAULT_WAIT_FULL);
      }
      if (res && e.q_tma && njobs > 0 && !mbar_wait(&a_full[0], 0)) raise_fault(FAULT_WAIT_FULL);
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(128, BN, /*a_mn=*/1, /*b_mn=*/1);
      int s = 0, par = 0, bs = 0, bpar = 0, lt = lt0;
      bool ok = true;
      if (res && e.q_tma && njobs > 0 && !mbar_wait(&a_full[0], 0)) {
        raise_fault(FAULT_WAIT_FULL);
        ok = false;
      }
      for (int j = 0; ok && j < njobs; ++j) {
        if ((j == 0 || lt == 0) && !mbar_wait(&b_full[bs], bpar)) {
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
        const uint32_t b_base = smem_u32(sB + bs * lay.b_bytes);
        for (int kk = 0; kk < KR / 16; ++kk) {
          const uint64_t ad = sdesc_sw128(a_base + kk * 2048, KR * 128, 1024);
          const uint64_t bd = sdesc_sw128(b_base + kk * 2048, KR * 128, 1024);
          umma_bf16(tmem + buf * BN, ad, bd, idesc, kk != 0);
        }
        if (!res) {
          umma_commit(&a_empty[s]);
          if (++s == kExpandStages) {
            s = 0;
            par ^= 1;
          }
        }
        if (++lt == e.nlt) {
          lt = 0;
          if (j + 1 < njobs) umma_commit(&b_empty[bs]);  // this block's slot may be refilled
          if (++bs == nb) {
            bs = 0;
            bpar ^= 1;
          }
        }
        umma_commit(&t_full[buf]);
      }
    }
  } else {
    // ---------------- epilogue (warps 2..9) ----------------
    // two groups of four warps (one per TMEM lane quarter); group g handles
    // jobs g, g+2, ... from accumulator g, so two tiles are converted at once.
    // Each group double-buffers its staging and tracks its own store groups.
    const int grp = (warp - 2) >> 2;          // 0 or 1
    const int gt = (threadIdx.x - 64) & 127;  // thread index within the group
    const int quarter = warp & 3;             // TMEM lanes this warp may read
    const int row = quarter * 32 + lane;      // token row within the tile
    int it = 0;
    int lt = lt0, smp = smp0, strip = strip0;
    for (int j = 0; j < njobs; ++j) {
      if ((j & 1) == grp) {
        uint8_t* st = stg + (2 * grp + (it & 1)) * (BN / 64) * BOX;
        if (gt == 0 && it >= 2) tma_store_wait_read<1>();
        if (grp == 0) named_barrier<1>(128); else named_barrier<2>(128);
        if (!mbar_wait(&t_full[grp], it & 1)) raise_fault(FAULT_WAIT_DONE);
        tc_fence_after();
        const uint32_t taddr = tmem + grp * BN + (static_cast<uint32_t>(quarter * 32) << 16);
        // a lane quarter wholly past the token axis holds only clipped rows
        const bool live = lt * BM + quarter * 32 < e.L;
#pragma unroll 1
        for (int h = 0; h < BN / 64; ++h) {
          float v[64];
          if (live) tmem_ld64(taddr + 64 * h, v);
          if (h == BN / 64 - 1) {
            // this warp has read its lanes of the accumulator: hand it back to
            // the MMA issuer before converting
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&t_empty[grp]);
          }
          if (live) {
            uint8_t* box = st + h * BOX + row * 128;
#pragma unroll
            for (int q = 0; q < 8; ++q)
              *reinterpret_cast<uint4*>(box + ((q ^ (row & 7)) << 4)) =
                  make_uint4(pack_bf16x2(v[8 * q], v[8 * q + 1]), pack_bf16x2(v[8 * q + 2], v[8 * q + 3]),
                             pack_bf16x2(v[8 * q + 4], v[8 * q + 5]),
                             pack_bf16x2(v[8 * q + 6], v[8 * q + 7]));
          }
        }
        fence_proxy_async_smem();
        if (grp == 0) named_barrier<1>(128); else named_barrier<2>(128);
        if (gt == 0) {
          for (int h = 0; h < BN / 64; ++h)
            if (strip * BN + 64 * h < e.Cx)
              tma_store_3d(&tmap_out, st + h * BOX, strip * BN + 64 * h, lt * BM, smp);
          tma_store_commit();
        }
        ++it;
      }
      if (++lt == e.nlt) {
        lt = 0;
        if (++smp == e.B) {
          smp = 0;
          ++strip;
        }
      }
    }
    if (gt == 0) tma_store_wait_all();
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
cudaError_t ensure_smem(size_t bytes) {
  // two CTAs per SM need the whole unified L1 as shared memory
  return raise_smem_limit(reinterpret_cast<const void*>(k_expand_bf16<BN>), bytes, true);
}

template <int BN>
cudaError_t launch_bn(const CUtensorMap& tq, const CUtensorMap& tg, const CUtensorMap& to,
                      const ExpandArgs& e, cudaStream_t st) {
  const size_t bytes = expand_bf16_smem_bytes(e);
  const cudaError_t err = ensure_smem<BN>(bytes);
  if (err != cudaSuccess) return err;
  if (e.ctas < 1 || e.ctas > e.total || e.nb < 1 || e.nb > kExpandMaxBRing ||
      (e.qres && e.nlt > kExpandMaxQRes))
    return cudaErrorInvalidValue;
  return launch_ex(k_expand_bf16<BN>, dim3(e.ctas), dim3(320), bytes, st, 1, pdl_enabled(), tq, tg,
                   to, e);
}

template <int BN>
int resident_bn(const ExpandArgs& e) {
  const size_t bytes = expand_bf16_smem_bytes(e);
  if (ensure_smem<BN>(bytes) != cudaSuccess) return 0;
  return resident_ctas_per_sm(reinterpret_cast<const void*>(k_expand_bf16<BN>), 320, bytes, 2 * BN);
}

}  // namespace

size_t expand_bf16_smem_bytes(const ExpandArgs& e) {
  return expand_layout(e.BN, e.KR, e.nb, expand_a_slots(e)).total + 1024;
}

int expand_bf16_ctas_per_sm(const ExpandArgs& e) {
  // one residency count per (device, BN, shared-memory size)
  static std::mutex mu;
  static std::map<std::tuple<int, int, size_t>, int> counts;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  const size_t bytes = expand_bf16_smem_bytes(e);
  const auto key = std::make_tuple(dev, e.BN, bytes);
  {
    std::lock_guard<std::mutex> lock(mu);
    const auto it = counts.find(key);
    if (it != counts.end()) return it->second;
  }
  const int n = e.BN == 128 ? resident_bn<128>(e) : resident_bn<64>(e);
  std::lock_guard<std::mutex> lock(mu);
  if (n > 0) counts[key] = n;
  return n;
}

cudaError_t launch_expand_bf16(const CUtensorMap& tmap_q, const CUtensorMap& tmap_g,
                               const CUtensorMap& tmap_out, const ExpandArgs& e, cudaStream_t st) {
  switch (e.BN) {
    case 64: return launch_bn<64>(tmap_q, tmap_g, tmap_out, e, st);
    case 128: return launch_bn<128>(tmap_q, tmap_g, tmap_out, e, st);
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
