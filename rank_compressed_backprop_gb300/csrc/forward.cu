// forward.cu -- the layer's forward y = x w^T with the stored activation
// x_hat = P x computed from the same x tiles (page "INSTANT: Compressing
// Gradients and Activations for Resource-Efficient Training", 整体框架: the
// forward product is unchanged, and the compressed activation is what the
// layer keeps for its backward instead of x).
//
// A persistent tcgen05 GEMM, one CTA per SM walking 128 x 192 output tiles
// (grouped so that the CTAs running at one time share w tiles in L2):
//   warp 0  TMA producer: per 64-channel chunk the x tile [128 tokens x 64]
//           (K-major A operand) and the w tile [192 rows x 64] (K-major B);
//           for the tiles of the first column strip also the P columns of
//           the tile's 128 tokens, once per tile;
//   warp 1  MMA issuer: four K = 16 MMAs per chunk into one of two TMEM
//           accumulators (192 columns each, double buffered); on the first
//           column strip, for x_hat, after every second chunk eight more MMAs
//           that reuse the two staged x tiles of the chunk pair as one
//           MN-major A operand of 128 channels:
//             D[c, r] = sum_{l in tile} x[l, c] P[r, l]   (M = the 128
//             channels, N = Rx rounded up to 16, K = the 128 tokens),
//           into one of two small TMEM buffers (the same contraction as the
//           projection kernel's, so it costs a few percent of the chunk's
//           MMA time);
//   warps 2-5  epilogue: TMEM -> bf16 -> 128-byte-swizzled staging box ->
//           TMA bulk store, two staging boxes in flight;
//   warps 6-9  x_hat flush: each thread holds one channel of the pair and adds
//           its Rx values into an fp32 accumulation buffer [B, Rx, Cx] with
//           atomics (coalesced along the channels); the tile that completes a
//           sample's token range converts that sample's rows to bf16 x_hat and
//           clears them (a counter per sample), so the buffer and the
//           counters are zero again after every launch.
// Only the first column strip computes x_hat: each x tile is on chip once per
// strip, and one strip suffices.  A 128-token tile never straddles two
// samples, and the chunk pairs sit in adjacent ring stages (the side output
// requires L % 128 == 0 and Cx % 128 == 0).
#include "kernels.h"
#include "tc.cuh"

namespace instant {

namespace {

constexpr int BM = 128;
constexpr int BN = kForwardBN;                  // 192
constexpr int BK = 64;
constexpr uint32_t A_BYTES = BM * BK * 2;       // 16 KB
constexpr uint32_t B_BYTES = BN * BK * 2;       // 24 KB
constexpr uint32_t STAGE = A_BYTES + B_BYTES;   // 40 KB
constexpr uint32_t P_ATOM = 32 * 128;           // 64 tokens x up to 32 rows of P
constexpr uint32_t P_BYTES = 2 * P_ATOM;        // the tile's 128 tokens: 8 KB
constexpr uint32_t BOX = BM * 128;              // staging box: 128 rows x 64 bf16
constexpr int NS = kForwardStages;
constexpr int XH_COLS = 32;                     // x_hat accumulator columns (>= Rx rounded to 16)
static_assert(NS % 2 == 0, "chunk pairs must sit in adjacent ring stages");

struct Lay {
  uint32_t stage, p, stg, bar, total;
};

__host__ __device__ inline Lay fwd_layout() {
  Lay l;
  l.stage = 0;
  l.p = NS * STAGE;
  l.stg = l.p + P_BYTES;
  l.bar = l.stg + 2 * BOX;
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

// output tile t of the grouped order -> (m, n)
__device__ __forceinline__ void fwd_tile(const ForwardArgs& a, int t, int& m, int& n) {
  const int per_group = a.group * a.nt;
  const int gid = t / per_group;
  const int first = gid * a.group;
  const int gsz = min(a.mt - first, a.group);
  const int r = t - gid * per_group;
  m = first + r % gsz;
  n = r / gsz;
}

__global__ void __launch_bounds__(320, 1)
    k_forward_bf16(const __grid_constant__ CUtensorMap tmap_x, const __grid_constant__ CUtensorMap tmap_w,
                   const __grid_constant__ CUtensorMap tmap_y, const __grid_constant__ CUtensorMap tmap_p,
                   ForwardArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const Lay lay = fwd_layout();
  uint8_t* sP = smem + lay.p;
  uint8_t* stg = smem + lay.stg;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + lay.bar);
  uint64_t* empty = full + NS;
  uint64_t* t_full = empty + NS;     // [2]
  uint64_t* t_empty = t_full + 2;    // [2]
  uint64_t* p_full = t_empty + 2;
  uint64_t* p_empty = p_full + 1;
  uint64_t* x_full = p_empty + 1;    // [2]
  uint64_t* x_empty = x_full + 2;    // [2] (one arrival per flush warp)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(x_empty + 2);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const bool side = a.Rx > 0;

  if (threadIdx.x == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&t_full[i], 1);
      mbar_init(&t_empty[i], 4);  // one arrival per epilogue warp
      mbar_init(&x_full[i], 1);
      mbar_init(&x_empty[i], 4);  // one arrival per flush warp
    }
    mbar_init(p_full, 1);
    mbar_init(p_empty, 1);
    fence_barrier_init();
    prefetch_tmap(&tmap_x);
    prefetch_tmap(&tmap_w);
    prefetch_tmap(&tmap_y);
    if (side) prefetch_tmap(&tmap_p);
  }
  const int NP = a.Rx <= 16 ? 16 : 32;  // x_hat MMA N: rows of P, rounded up
  if (side) {
    // rows Rx..NP-1 of both P atoms stay zero: the x_hat MMA reads NP rows
    for (int i = threadIdx.x; i < static_cast<int>(P_BYTES / 16); i += blockDim.x)
      reinterpret_cast<uint4*>(sP)[i] = make_uint4(0, 0, 0, 0);
    fence_proxy_async_smem();
  }
  if (warp == 0) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  pdl_launch_dependents();
  pdl_wait();

  const int tiles = a.mt * a.nt;
  if (warp == 0) {
    // ---------------- producer ----------------
    if (lane == 0) {
      int s = 0, par = 0, issued = 0, np = 0;
      bool ok = true;
      for (int t = blockIdx.x; ok && t < tiles; t += gridDim.x) {
        int m, n;
        fwd_tile(a, t, m, n);
        if (side && n == 0) {
          // the P columns of this tile's tokens (rows 0..Rx-1 of both atoms)
          if (np > 0 && !mbar_wait(p_empty, (np - 1) & 1)) {
            raise_fault(FAULT_WAIT_EMPTY);
            break;
          }
          const int l0 = m * BM - (m * BM / a.L) * a.L;
          mbar_arrive_expect_tx(p_full, 2 * a.Rx * 128);
          tma_load_2d(sP, &tmap_p, p_full, l0, 0);
          tma_load_2d(sP + NP * 128, &tmap_p, p_full, l0 + 64, 0);
          ++np;
        }
        for (int kc = 0; kc < a.nkc; ++kc) {
          if (issued >= NS && !mbar_wait(&empty[s], par ^ 1)) {
            raise_fault(FAULT_WAIT_EMPTY);
            ok = false;
            break;
          }
          uint8_t* st = smem + s * STAGE;
          mbar_arrive_expect_tx(&full[s], STAGE);
          tma_load_2d(st, &tmap_x, &full[s], kc * BK, m * BM);
          tma_load_2d(st + A_BYTES, &tmap_w, &full[s], kc * BK, n * BN);
          ++issued;
          if (++s == NS) {
            s = 0;
            par ^= 1;
          }
        }
      }
      for (int k = 0; k < NS && k < issued; ++k) {
        if (--s < 0) {
          s = NS - 1;
          par ^= 1;
        }
        if (!mbar_wait(&full[s], par)) raise_fault(FAULT_WAIT_FULL);
      }
      if (np > 0 && !mbar_wait(p_full, (np - 1) & 1)) raise_fault(FAULT_WAIT_FULL);
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(BM, BN, 0, 0);
      const uint32_t idesc_x = NP == 16 ? idesc_bf16_f32(128, 16, /*a_mn=*/1, /*b_mn=*/0)
                                        : idesc_bf16_f32(128, 32, /*a_mn=*/1, /*b_mn=*/0);
      int s = 0, par = 0, q = 0, np = 0, xc = 0;
      bool ok = true;
      for (int t = blockIdx.x; ok && t < tiles; t += gridDim.x, ++q) {
        int m, n;
        fwd_tile(a, t, m, n);
        const bool xh = side && n == 0;
        const int acc = q & 1;
        if (q >= 2 && !mbar_wait(&t_empty[acc], ((q >> 1) - 1) & 1)) {
          raise_fault(FAULT_WAIT_EMPTY);
          break;
        }
        if (xh && !mbar_wait(p_full, np & 1)) {
          raise_fault(FAULT_WAIT_FULL);
          break;
        }
        for (int kc = 0; kc < a.nkc; ++kc) {
          if (!mbar_wait(&full[s], par)) {
            raise_fault(FAULT_WAIT_FULL);
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_base = smem_u32(smem + s * STAGE);
          const uint32_t b_base = a_base + A_BYTES;
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk) {
            const uint64_t ad = sdesc_sw128(a_base + kk * 32, 16, 1024);
            const uint64_t bd = sdesc_sw128(b_base + kk * 32, 16, 1024);
            umma_bf16(tmem + acc * BN, ad, bd, idesc, (kc | kk) != 0);
          }
          if (xh && (kc & 1)) {
            // x_hat partial of the chunk pair's 128 channels over the tile's
            // tokens: A = the two x tiles (stages s-1 and s, STAGE bytes apart:
            // an even number of chunks precede every pair), B = the P tile
            const int xb = xc & 1;
            if (xc >= 2 && !mbar_wait(&x_empty[xb], ((xc >> 1) - 1) & 1)) {
              raise_fault(FAULT_WAIT_EMPTY);
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t x_base = a_base - STAGE;
            const uint32_t p_base = smem_u32(sP);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
              const uint64_t ad = sdesc_sw128(x_base + kk * 2048, STAGE, 1024);
              const uint64_t bd = sdesc_sw128(p_base + (kk >> 2) * (NP * 128) + (kk & 3) * 32, 16, 1024);
              umma_bf16(tmem + 2 * BN + xb * XH_COLS, ad, bd, idesc_x, kk != 0);
            }
            umma_commit(&x_full[xb]);
            ++xc;
            umma_commit(&empty[s - 1]);  // the pair's first stage, read by these MMAs too
          }
          if (!(xh && !(kc & 1))) umma_commit(&empty[s]);
          if (++s == NS) {
            s = 0;
            par ^= 1;
          }
        }
        if (!ok) break;
        umma_commit(&t_full[acc]);
        if (xh) {
          umma_commit(p_empty);  // the P buffer may be refilled
          ++np;
        }
      }
    }
  } else if (warp >= 2 && warp <= 5) {
    // ---------------- epilogue: y tiles ----------------
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;
    const int gt = threadIdx.x - 64;   // 0..127
    int q = 0, boxes = 0;
    for (int t = blockIdx.x; t < tiles; t += gridDim.x, ++q) {
      int m, n;
      fwd_tile(a, t, m, n);
      const int acc = q & 1;
      if (!mbar_wait(&t_full[acc], (q >> 1) & 1)) {
        raise_fault(FAULT_WAIT_DONE);
        break;
      }
      tc_fence_after();
      const uint32_t taddr = tmem + acc * BN + (static_cast<uint32_t>(quarter * 32) << 16);
      for (int h = 0; h < BN / 64; ++h, ++boxes) {
        uint8_t* box = stg + (boxes & 1) * BOX;
        if (gt == 0 && boxes >= 2) tma_store_wait_read<1>();
        named_barrier<1>(128);
        float v[64];
        tmem_ld64(taddr + 64 * h, v);
        if (h == BN / 64 - 1) {
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&t_empty[acc]);
        }
        uint8_t* row = box + r * 128;
#pragma unroll
        for (int c = 0; c < 8; ++c)
          *reinterpret_cast<uint4*>(row + ((c ^ (r & 7)) << 4)) =
              make_uint4(pack_bf16x2(v[8 * c], v[8 * c + 1]), pack_bf16x2(v[8 * c + 2], v[8 * c + 3]),
                         pack_bf16x2(v[8 * c + 4], v[8 * c + 5]), pack_bf16x2(v[8 * c + 6], v[8 * c + 7]));
        fence_proxy_async_smem();
        named_barrier<1>(128);
        if (gt == 0) {
          if (n * BN + 64 * h < a.N) tma_store_2d(&tmap_y, box, n * BN + 64 * h, m * BM);
          tma_store_commit();
        }
      }
    }
    if (gt == 0) tma_store_wait_all();
  } else if (warp >= 6 && side) {
    // ---------------- x_hat flush (warps 6-9) ----------------
    const int quarter = warp & 3;
    const int ch = quarter * 32 + lane;   // channel within the chunk pair (TMEM lane)
    const int ft = threadIdx.x - 192;     // 0..127
    int xc = 0;
    const int per_sample = a.L / BM;
    for (int t = blockIdx.x; t < tiles; t += gridDim.x) {
      int m, n;
      fwd_tile(a, t, m, n);
      if (n != 0) continue;
      const int b = m * BM / a.L;
      float* dst = a.xh32 + static_cast<size_t>(b) * a.Rx * a.K;
      bool ok = true;
      for (int kp = 0; kp < a.nkc / 2; ++kp, ++xc) {
        const int xb = xc & 1;
        if (!mbar_wait(&x_full[xb], (xc >> 1) & 1)) {
          raise_fault(FAULT_WAIT_DONE);
          ok = false;
          break;
        }
        tc_fence_after();
        float v[32];
        tmem_ld32(tmem + 2 * BN + xb * XH_COLS + (static_cast<uint32_t>(quarter * 32) << 16), v);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&x_empty[xb]);
        const int c = kp * 2 * BK + ch;
#pragma unroll
        for (int r = 0; r < 32; ++r)
          if (r < a.Rx) atomicAdd(dst + static_cast<size_t>(r) * a.K + c, v[r]);
      }
      if (!ok) break;
      // the tile that completes sample b converts its rows and clears them
      __threadfence();
      named_barrier<2>(128);
      __shared__ unsigned s_prev;
      if (ft == 0) s_prev = atomicAdd(a.cnt + b, 1u);
      named_barrier<2>(128);
      if (s_prev == static_cast<unsigned>(per_sample - 1)) {
        __threadfence();
        float* src = dst;
        uint16_t* out = static_cast<uint16_t*>(a.xh) + static_cast<size_t>(b) * a.Rx * a.K;
        // 8 loads in flight per thread: the conversion is latency-bound otherwise
        const int n4 = a.Rx * a.K / 4;
        constexpr int kBatch = 8;
        for (int i0 = 0; i0 < n4; i0 += 128 * kBatch) {
          float4 f[kBatch];
#pragma unroll
          for (int j = 0; j < kBatch; ++j) {
            const int i = i0 + j * 128 + ft;
            f[j] = i < n4 ? __ldcg(reinterpret_cast<const float4*>(src) + i) : make_float4(0.f, 0.f, 0.f, 0.f);
          }
#pragma unroll
          for (int j = 0; j < kBatch; ++j) {
            const int i = i0 + j * 128 + ft;
            if (i < n4) {
              reinterpret_cast<uint2*>(out)[i] =
                  make_uint2(pack_bf16x2(f[j].x, f[j].y), pack_bf16x2(f[j].z, f[j].w));
              reinterpret_cast<float4*>(src)[i] = make_float4(0.f, 0.f, 0.f, 0.f);
            }
          }
        }
        if (ft == 0) a.cnt[b] = 0u;
      }
      named_barrier<2>(128);  // s_prev is rewritten by the next tile
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, 512);
}

// fp32 path (no tensor cores): one thread per output element
__global__ void k_forward_f32(const float* __restrict__ x, const float* __restrict__ w,
                              float* __restrict__ y, int M, int N, int K) {
  const int n = blockIdx.x * blockDim.x + threadIdx.x;
  const int m = blockIdx.y;
  if (n >= N) return;
  const float* xr = x + static_cast<size_t>(m) * K;
  const float* wr = w + static_cast<size_t>(n) * K;
  float acc = 0.f;
  for (int k = 0; k < K; ++k) acc = fmaf(xr[k], wr[k], acc);
  y[static_cast<size_t>(m) * N + n] = acc;
}

}  // namespace

cudaError_t launch_forward_f32(const float* x, const float* w, float* y, int M, int N, int K,
                               cudaStream_t st) {
  dim3 grid((N + 127) / 128, M);
  k_forward_f32<<<grid, 128, 0, st>>>(x, w, y, M, N, K);
  count_launches(1);
  return cudaGetLastError();
}

size_t forward_bf16_smem_bytes() { return fwd_layout().total + 1024; }

cudaError_t launch_forward_bf16(const CUtensorMap& tmap_x, const CUtensorMap& tmap_w,
                                const CUtensorMap& tmap_y, const CUtensorMap& tmap_p,
                                const ForwardArgs& a, int ctas, cudaStream_t st) {
  if (ctas < 1 || a.mt < 1 || a.nt < 1 || a.nkc < 1 || a.group < 1) return cudaErrorInvalidValue;
  if (a.Rx < 0 || a.Rx > 32 || (a.Rx > 0 && (a.L % BM != 0 || a.K % 128 != 0)))
    return cudaErrorInvalidValue;
  const size_t bytes = forward_bf16_smem_bytes();
  const cudaError_t e = raise_smem_limit(reinterpret_cast<const void*>(k_forward_bf16), bytes);
  if (e != cudaSuccess) return e;
  return launch_ex(k_forward_bf16, dim3(ctas), dim3(320), bytes, st, 1, pdl_enabled(), tmap_x,
                   tmap_w, tmap_y, tmap_p, a);
}

INSTANT_FAULT_READER(read_fault_forward)

}  // namespace instant
