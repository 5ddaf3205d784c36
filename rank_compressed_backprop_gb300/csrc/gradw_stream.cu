// gradw_stream.cu -- the weight gradient of INSTANT's backward when its
// contraction is short (page "INSTANT: Compressing Gradients and Activations
// for Resource-Efficient Training", 关键设计 3):
//   g_w = g_hat_y1 x_hat = Sx^T x_hat,   [Cy, K] x [K, Cx],   K = B * Rx.
//
// With K = 64 (a long-sequence layer: four samples of rank 16) the product
// costs 2K = 128 flops per output element, while every element is a 4-byte
// fp32 write: the step is bound by HBM writes of the [Cy, Cx] result (180 MB
// for a 4096 -> 11008 layer), like the input-gradient expansion.  So it is
// built the same way: a persistent grid, one CTA per SM, each CTA walking a
// contiguous range of 128 x 64 output tiles (column strip major, so the
// x_hat strip -- the B operand -- stays resident while the CTA walks down
// its rows):
//   warp 0  TMA producer: the x_hat strip (K x 64, MN-major B operand) once
//           per strip, then the Sx tiles (K x 128, MN-major A operand) through
//           a ring of 64-deep K chunks;
//   warp 1  MMA issuer: K/16 tcgen05 MMAs per tile into one of two TMEM
//           accumulators (double buffered);
//   warps 2-9  epilogue, two groups of four warps taking alternate tiles:
//           TMEM -> registers (+ the old tile, read by TMA, when
//           accumulating) -> 128-byte-swizzled fp32 staging -> TMA bulk
//           store; two staging buffers per group, so the stores of one tile
//           overlap the conversion of the next.
// Rows past Cy and columns past Cx are zero-filled on load and clipped on
// store by the tensor maps.
#include "kernels.h"
#include "tc.cuh"

namespace instant {

namespace {

constexpr int BM = 128;
constexpr int BN = 64;
constexpr int BK = 64;
constexpr uint32_t A_CHUNK = BM * BK * 2;        // 16 KB: 64 K-rows x 128 rows of Cy
constexpr uint32_t B_CHUNK = BN * BK * 2;        // 8 KB: 64 K-rows x 64 columns of Cx
constexpr uint32_t OUT_BOX = BM * 32 * 4;        // 16 KB: 128 rows x 32 fp32 (128 B)
constexpr uint32_t OUT_TILE = 2 * OUT_BOX;       // 128 x 64 fp32

struct Lay {
  uint32_t stg, b, a, bar, total;
};

__host__ __device__ inline Lay gradw_layout(int nkc, int stages) {
  Lay l;
  l.stg = 0;                                     // 4 staging tiles: 2 groups x 2
  l.b = 4 * OUT_TILE;
  l.a = l.b + nkc * B_CHUNK;
  l.bar = l.a + stages * A_CHUNK;
  l.total = l.bar + 256;
  return l;
}

__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, const void* src, int c0, int c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.global.shared::cta.tile.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
          reinterpret_cast<uint64_t>(map)),
      "r"(smem_u32(src)), "r"(c0), "r"(c1)
      : "memory");
}

__global__ void __launch_bounds__(320, 1)
    k_gradw_stream(const __grid_constant__ CUtensorMap tmap_sx,
                   const __grid_constant__ CUtensorMap tmap_xh,
                   const __grid_constant__ CUtensorMap tmap_gw, GradWStreamArgs g) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const int NS = g.stages;
  const int nkc = g.nkc;
  const Lay lay = gradw_layout(nkc, NS);
  uint8_t* stg = smem + lay.stg;
  uint8_t* sB = smem + lay.b;
  uint8_t* sA = smem + lay.a;
  uint64_t* a_full = reinterpret_cast<uint64_t*>(smem + lay.bar);
  uint64_t* a_empty = a_full + kGradWStages;
  uint64_t* b_full = a_empty + kGradWStages;
  uint64_t* b_empty = b_full + 1;
  uint64_t* t_full = b_empty + 1;
  uint64_t* t_empty = t_full + 2;
  uint64_t* o_full = t_empty + 2;                // old tile in staging buffer (accumulate)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(o_full + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // this CTA's tiles: [t0, t1) of the strip-major tile order
  const long long T = static_cast<long long>(g.mt) * g.nt;
  const int t0 = static_cast<int>(T * blockIdx.x / gridDim.x);
  const int t1 = static_cast<int>(T * (blockIdx.x + 1) / gridDim.x);
  const int ntile = t1 - t0;

  if (threadIdx.x == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(&a_full[s], 1);
      mbar_init(&a_empty[s], 1);
    }
    mbar_init(b_full, 1);
    mbar_init(b_empty, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&t_full[i], 1);
      mbar_init(&t_empty[i], 4);  // one arrival per warp of the epilogue group
    }
    for (int i = 0; i < 4; ++i) mbar_init(&o_full[i], 1);
    fence_barrier_init();
    prefetch_tmap(&tmap_sx);
    prefetch_tmap(&tmap_xh);
    prefetch_tmap(&tmap_gw);
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

  if (warp == 0) {
    // ---------------- producer ----------------
    if (lane == 0) {
      int s = 0, par = 0, issued = 0;
      int strip = -1, seg = -1;
      int row = 0, cur = t0 / g.mt;
      row = t0 - cur * g.mt;
      bool ok = true;
      for (int i = 0; ok && i < ntile; ++i) {
        if (cur != strip) {
          // the previous strip's B is free once its last MMA has completed
          if (seg >= 0 && !mbar_wait(b_empty, seg & 1)) {
            raise_fault(FAULT_WAIT_EMPTY);
            break;
          }
          strip = cur;
          ++seg;
          mbar_arrive_expect_tx(b_full, nkc * B_CHUNK);
          for (int c = 0; c < nkc; ++c)
            tma_load_2d(sB + c * B_CHUNK, &tmap_xh, b_full, strip * BN, c * BK);
        }
        for (int c = 0; c < nkc; ++c) {
          if (issued >= NS && !mbar_wait(&a_empty[s], par ^ 1)) {
            raise_fault(FAULT_WAIT_EMPTY);
            ok = false;
            break;
          }
          uint8_t* dst = sA + s * A_CHUNK;
          mbar_arrive_expect_tx(&a_full[s], A_CHUNK);
          tma_load_2d(dst, &tmap_sx, &a_full[s], row * BM, c * BK);
          tma_load_2d(dst + A_CHUNK / 2, &tmap_sx, &a_full[s], row * BM + 64, c * BK);
          ++issued;
          if (++s == NS) {
            s = 0;
            par ^= 1;
          }
        }
        if (++row == g.mt) {
          row = 0;
          ++cur;
        }
      }
      // leave only after every copy issued into this CTA's shared memory landed
      for (int k = 0; k < NS && k < issued; ++k) {
        if (--s < 0) {
          s = NS - 1;
          par ^= 1;
        }
        if (!mbar_wait(&a_full[s], par)) raise_fault(FAULT_WAIT_FULL);
      }
      if (seg >= 0 && !mbar_wait(b_full, seg & 1)) raise_fault(FAULT_WAIT_FULL);
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(BM, BN, /*a_mn=*/1, /*b_mn=*/1);
      const uint32_t b_base = smem_u32(sB);
      int s = 0, par = 0;
      int strip = -1, seg = -1;
      int row = 0, cur = t0 / g.mt;
      row = t0 - cur * g.mt;
      bool ok = true;
      for (int i = 0; ok && i < ntile; ++i) {
        const int buf = i & 1;
        if (cur != strip) {
          strip = cur;
          ++seg;
          if (!mbar_wait(b_full, seg & 1)) {
            raise_fault(FAULT_WAIT_FULL);
            break;
          }
        }
        if (i >= 2 && !mbar_wait(&t_empty[buf], ((i >> 1) - 1) & 1)) {
          raise_fault(FAULT_WAIT_EMPTY);
          break;
        }
        for (int c = 0; c < nkc; ++c) {
          if (!mbar_wait(&a_full[s], par)) {
            raise_fault(FAULT_WAIT_FULL);
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_base = smem_u32(sA + s * A_CHUNK);
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk) {
            const uint64_t ad = sdesc_sw128(a_base + kk * 2048, A_CHUNK / 2, 1024);
            const uint64_t bd = sdesc_sw128(b_base + c * B_CHUNK + kk * 2048, B_CHUNK, 1024);
            umma_bf16(tmem + buf * BN, ad, bd, idesc, (c | kk) != 0);
          }
          umma_commit(&a_empty[s]);
          if (++s == NS) {
            s = 0;
            par ^= 1;
          }
        }
        if (!ok) break;
        umma_commit(&t_full[buf]);
        if (++row == g.mt) {
          row = 0;
          ++cur;
        }
        // last tile of this strip with more tiles to come: B may be replaced
        if (cur != strip && i + 1 < ntile) umma_commit(b_empty);
      }
    }
  } else {
    // ---------------- epilogue (warps 2..9) ----------------
    const int grp = (warp - 2) >> 2;          // 0 or 1: takes local tiles grp, grp+2, ...
    const int gt = (threadIdx.x - 64) & 127;  // thread index within the group
    const int quarter = warp & 3;             // TMEM lanes this warp may read
    const int r = quarter * 32 + lane;        // row within the tile
    int it = 0;
    for (int i = grp; i < ntile; i += 2, ++it) {
      const int t = t0 + i;
      const int strip = t / g.mt;
      const int row = t - strip * g.mt;
      const int bi = 2 * grp + (it & 1);
      uint8_t* st = stg + bi * OUT_TILE;
      if (gt == 0) {
        // this buffer's store from two tiles ago has finished reading it
        if (it >= 2) tma_store_wait_read<1>();
        if (g.accumulate) {
          mbar_arrive_expect_tx(&o_full[bi], OUT_TILE);
          for (int h = 0; h < 2; ++h)
            tma_load_2d(st + h * OUT_BOX, &tmap_gw, &o_full[bi], strip * BN + 32 * h, row * BM);
        }
      }
      if (grp == 0) named_barrier<1>(128); else named_barrier<2>(128);
      if (!mbar_wait(&t_full[grp], it & 1)) raise_fault(FAULT_WAIT_DONE);
      tc_fence_after();
      float v[64];
      tmem_ld64(tmem + grp * BN + (static_cast<uint32_t>(quarter * 32) << 16), v);
      // this warp has read its lanes of the accumulator: hand it back
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&t_empty[grp]);
      if (g.accumulate && !mbar_wait(&o_full[bi], (it >> 1) & 1)) raise_fault(FAULT_WAIT_FULL);
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        uint8_t* line = st + h * OUT_BOX + r * 128;
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          float4* p = reinterpret_cast<float4*>(line + ((q ^ (r & 7)) << 4));
          float4 x = make_float4(v[32 * h + 4 * q], v[32 * h + 4 * q + 1], v[32 * h + 4 * q + 2],
                                 v[32 * h + 4 * q + 3]);
          if (g.accumulate) {
            const float4 o = *p;
            x.x += o.x;
            x.y += o.y;
            x.z += o.z;
            x.w += o.w;
          }
          *p = x;
        }
      }
      fence_proxy_async_smem();
      if (grp == 0) named_barrier<1>(128); else named_barrier<2>(128);
      if (gt == 0) {
        for (int h = 0; h < 2; ++h)
          if (strip * BN + 32 * h < g.N) tma_store_2d(&tmap_gw, st + h * OUT_BOX, strip * BN + 32 * h, row * BM);
        tma_store_commit();
      }
    }
    if (gt == 0) tma_store_wait_all();
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, 2 * BN);
}

}  // namespace

size_t gradw_stream_smem_bytes(const GradWStreamArgs& g) {
  return gradw_layout(g.nkc, g.stages).total + 1024;
}

cudaError_t launch_gradw_stream(const CUtensorMap& tmap_sx, const CUtensorMap& tmap_xh,
                                const CUtensorMap& tmap_gw, const GradWStreamArgs& g, int ctas,
                                cudaStream_t st) {
  if (g.nkc < 1 || g.nkc > kGradWMaxChunks || g.stages < 2 || g.stages > kGradWStages || ctas < 1)
    return cudaErrorInvalidValue;
  const size_t bytes = gradw_stream_smem_bytes(g);
  const cudaError_t e = raise_smem_limit(reinterpret_cast<const void*>(k_gradw_stream), bytes);
  if (e != cudaSuccess) return e;
  return launch_ex(k_gradw_stream, dim3(ctas), dim3(320), bytes, st, 1, pdl_enabled(), tmap_sx,
                   tmap_xh, tmap_gw, g);
}

INSTANT_FAULT_READER(read_fault_gradw)

}  // namespace instant
