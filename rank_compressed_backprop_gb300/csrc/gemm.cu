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
// One elected thread issues the MMAs.  These products are small (a few MB), so
// the grid is widened by splitting K across the CTAs of a thread-block
// cluster: every CTA parks its fp32 partial tile in its own shared memory, and
// after a cluster barrier each CTA sums a slice of the tile's rows over all S
// partials through distributed shared memory and writes it with coalesced
// stores (fp32, fp32 accumulate, or bf16).  No global scratch.
// A short K-major A (M <= 64, g_hat_x for a few samples) takes a 64-row box:
// the stage is 8 KB smaller, so more CTAs share an SM, and the M = 128 MMA
// reads rows 64..127 from the B slot after it (results never used).
#include <map>
#include <mutex>
#include <tuple>

#include "kernels.h"
#include "tc.cuh"

namespace instant {

namespace {

constexpr int BM = 128;
constexpr int BK = 64;
constexpr int A_BYTES = BM * BK * 2;  // 16 KB

__host__ __device__ inline uint32_t a_bytes(int short_a) { return short_a ? A_BYTES / 2 : A_BYTES; }
__host__ __device__ inline uint32_t stage_bytes(int BN, int short_a) {
  return a_bytes(short_a) + BN * BK * 2;
}
__host__ __device__ inline int tile_rows(int short_a) { return short_a ? BM / 2 : BM; }

template <int BN, int A_MN, int B_MN>
__global__ void __launch_bounds__(128, 1)
    k_gemm_bf16(const __grid_constant__ CUtensorMap tmap_a,
                const __grid_constant__ CUtensorMap tmap_b, GemmArgs g) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t ABYTES = a_bytes(g.short_a);
  const uint32_t STAGE = stage_bytes(BN, g.short_a);
  const int ROWS = tile_rows(g.short_a);  // rows of the tile that can hold results
  constexpr int RED_LD = BN + 4;  // fp32 reduction tile row pitch (bank spread)
  const int NS = g.stages;  // ring depth: min(4, chunks per CTA)
  const uint32_t RING = NS * STAGE;
  const uint32_t REDB = ROWS * RED_LD * 4;
  const uint32_t BAR_OFF = RING > REDB ? RING : REDB;
  uint8_t* sbase = smem;
  float* red = reinterpret_cast<float*>(smem);  // reuses the stages after the K loop
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + BAR_OFF);
  uint64_t* empty = full + NS;
  uint64_t* done = empty + NS;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int n0 = blockIdx.x * BN;
  const int m0 = blockIdx.y * BM;
  const int split = blockIdx.z;  // == rank in the cluster (cluster dims 1 x 1 x splits)
  const int kc_begin = split * g.chunks_per_split;
  int kc_end = kc_begin + g.chunks_per_split;
  if (kc_end > g.nk) kc_end = g.nk;
  const int nkc = kc_end > kc_begin ? kc_end - kc_begin : 0;

  if (threadIdx.x == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(done, 1);
    fence_barrier_init();
    prefetch_tmap(&tmap_a);
    prefetch_tmap(&tmap_b);
    // the ring's first chunks into L2 while the predecessor finishes (w for
    // g_hat_x comes from HBM; L2 is the point of coherence, so a line fetched
    // early is still updated by the predecessor's writes); at most 32 MB over
    // the grid
    const long long ctas = static_cast<long long>(gridDim.x) * gridDim.y * gridDim.z;
    const long long cap = (32ll << 20) / (ctas * STAGE);
    const int npf = static_cast<int>(cap < nkc ? (cap < NS ? cap : NS) : (nkc < NS ? nkc : NS));
    for (int i = 0; i < npf; ++i) {
      const int k0 = (kc_begin + i) * BK;
      if (A_MN) {
        tma_prefetch_l2_2d(&tmap_a, m0, k0);
        tma_prefetch_l2_2d(&tmap_a, m0 + 64, k0);
      } else {
        tma_prefetch_l2_2d(&tmap_a, k0, m0);
      }
      if (B_MN) {
#pragma unroll
        for (int h = 0; h < BN / 64; ++h) tma_prefetch_l2_2d(&tmap_b, n0 + 64 * h, k0);
      } else {
        tma_prefetch_l2_2d(&tmap_b, k0, n0);
      }
    }
  }
  if (warp == 0) {
    tmem_alloc(tmem_slot, BN);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  pdl_launch_dependents();
  pdl_wait();

  if (warp == 0 && lane == 0) {
    // ---------------- TMA producer ----------------
    int issued = 0;
    int s = 0, par = 0;  // ring slot and round parity of chunk i, kept without divisions
    for (int i = 0; i < nkc; ++i) {
      if (i >= NS && !mbar_wait(&empty[s], par ^ 1)) {
        raise_fault(FAULT_WAIT_EMPTY);
        break;
      }
      const int k0 = (kc_begin + i) * BK;
      uint8_t* sa = sbase + s * STAGE;
      uint8_t* sb = sa + ABYTES;
      mbar_arrive_expect_tx(&full[s], STAGE);
      if (A_MN) {  // A stored [K, M]: two 64-wide M boxes of 64 K-rows
        tma_load_2d(sa, &tmap_a, &full[s], m0, k0);
        tma_load_2d(sa + A_BYTES / 2, &tmap_a, &full[s], m0 + 64, k0);
      } else {     // A stored [M, K]: one box of 64 K x 128 (short: 64) rows
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
      if (++s == NS) {
        s = 0;
        par ^= 1;
      }
    }
    for (int i = issued - NS < 0 ? 0 : issued - NS; i < issued; ++i)
      if (!mbar_wait(&full[i % NS], (i / NS) & 1)) raise_fault(FAULT_WAIT_FULL);
  } else if (warp == 1 && lane == 0) {
    // ---------------- MMA issuer ----------------
    constexpr uint32_t idesc = idesc_bf16_f32(128, BN, A_MN, B_MN);
    bool ok = true;
    int s = 0, par = 0;
    for (int i = 0; i < nkc; ++i) {
      if (!mbar_wait(&full[s], par)) {
        raise_fault(FAULT_WAIT_FULL);
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t a_base = smem_u32(sbase + s * STAGE);
      const uint32_t b_base = a_base + ABYTES;
#pragma unroll
      for (int kk = 0; kk < BK / 16; ++kk) {
        const uint64_t ad = A_MN ? sdesc_sw128(a_base + kk * 2048, A_BYTES / 2, 1024)
                                 : sdesc_sw128(a_base + kk * 32, 16, 1024);
        const uint64_t bd = B_MN ? sdesc_sw128(b_base + kk * 2048, 64 * BK * 2, 1024)
                                 : sdesc_sw128(b_base + kk * 32, 16, 1024);
        umma_bf16(tmem, ad, bd, idesc, (i | kk) != 0);
      }
      umma_commit(&empty[s]);
      if (++s == NS) {
        s = 0;
        par ^= 1;
      }
    }
    if (ok && nkc > 0) umma_commit(done);
  }
  __syncwarp();

  // ---------------- epilogue 1: TMEM -> fp32 partial tile in shared memory ----------------
  const bool have = nkc > 0;
  if (have && !mbar_wait(done, 0)) raise_fault(FAULT_WAIT_DONE);
  tc_fence_after();
  fence_proxy_async_smem();
  __syncthreads();  // every stage is consumed: the ring becomes the reduction tile
  if (warp * 32 < ROWS) {
    const int row = warp * 32 + lane;
    const uint32_t taddr = tmem + (static_cast<uint32_t>(warp * 32) << 16);
    float* dst = red + row * RED_LD;
#pragma unroll 1
    for (int j0 = 0; j0 < BN; j0 += 16) {
      float v[16];
      if (have) {
        tmem_ld16(taddr + j0, v);
      } else {
#pragma unroll
        for (int q = 0; q < 16; ++q) v[q] = 0.f;
      }
#pragma unroll
      for (int q = 0; q < 4; ++q)
        *reinterpret_cast<float4*>(dst + j0 + 4 * q) =
            make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
    }
  }
  tc_fence_before();
  if (g.splits > 1) cluster_sync(); else __syncthreads();

  // ---------------- epilogue 2: reduce a row slice over the cluster, store ----------------
  {
    const int per = (ROWS + g.splits - 1) / g.splits;
    const int r0 = split * per;
    const int rows = r0 >= ROWS ? 0 : (ROWS - r0 < per ? ROWS - r0 : per);
    constexpr int C4 = BN / 4;
    for (int idx = threadIdx.x; idx < rows * C4; idx += blockDim.x) {
      const int rr = r0 + idx / C4;
      const int c = (idx % C4) * 4;
      const float* src = red + rr * RED_LD + c;
      float4 acc = *reinterpret_cast<const float4*>(src);
      // issue every peer load before the first add (in-order issue would
      // otherwise stall on each remote round trip)
      float4 part[8];
#pragma unroll
      for (int q = 0; q < 8; ++q)
        if (q < g.splits && q != split) part[q] = dsmem_ld_f4(dsmem_addr(src, q));
#pragma unroll
      for (int q = 0; q < 8; ++q)
        if (q < g.splits && q != split) {
          acc.x += part[q].x; acc.y += part[q].y; acc.z += part[q].z; acc.w += part[q].w;
        }
      const int m = m0 + rr;
      const int n = n0 + c;
      if (m < g.M && n < g.N) {
        const size_t off = static_cast<size_t>(m) * g.N + n;
        if (g.out_bf16) {
          uint2 p;
          p.x = static_cast<uint32_t>(bf16_bits(acc.x)) | (static_cast<uint32_t>(bf16_bits(acc.y)) << 16);
          p.y = static_cast<uint32_t>(bf16_bits(acc.z)) | (static_cast<uint32_t>(bf16_bits(acc.w)) << 16);
          *reinterpret_cast<uint2*>(static_cast<uint16_t*>(g.out) + off) = p;
        } else {
          float4* dstp = reinterpret_cast<float4*>(static_cast<float*>(g.out) + off);
          if (g.accumulate) {
            const float4 o = *dstp;
            acc.x += o.x; acc.y += o.y; acc.z += o.z; acc.w += o.w;
          }
          *dstp = acc;
        }
      }
    }
  }
  // peers may still read this CTA's tile: leave together
  if (g.splits > 1) cluster_sync(); else __syncthreads();
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
  float* dst = static_cast<float*>(g.out) + static_cast<size_t>(m) * g.N + n;
  *dst = g.accumulate ? *dst + acc : acc;
}

template <int BN, int A_MN, int B_MN>
cudaError_t launch_cfg(const CUtensorMap& ta, const CUtensorMap& tb, const GemmArgs& g,
                       cudaStream_t st) {
  const size_t bytes = gemm_bf16_smem_bytes(g);
  const cudaError_t e = raise_smem_limit(reinterpret_cast<const void*>(k_gemm_bf16<BN, A_MN, B_MN>), bytes);
  if (e != cudaSuccess) return e;
  return launch_ex(k_gemm_bf16<BN, A_MN, B_MN>, dim3((g.N + BN - 1) / BN, (g.M + BM - 1) / BM, g.splits),
                   dim3(128), bytes, st, g.splits, pdl_enabled(), ta, tb, g);
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

template <int A_MN, int B_MN>
const void* kernel_bn(int BN) {
  switch (BN) {
    case 64: return reinterpret_cast<const void*>(k_gemm_bf16<64, A_MN, B_MN>);
    case 128: return reinterpret_cast<const void*>(k_gemm_bf16<128, A_MN, B_MN>);
    case 256: return reinterpret_cast<const void*>(k_gemm_bf16<256, A_MN, B_MN>);
    default: return nullptr;
  }
}

const void* kernel_for(const GemmArgs& g) {
  if (g.a_mn_major && g.b_mn_major) return kernel_bn<1, 1>(g.BN);
  if (!g.a_mn_major && g.b_mn_major) return kernel_bn<0, 1>(g.BN);
  if (g.a_mn_major && !g.b_mn_major) return kernel_bn<1, 0>(g.BN);
  return kernel_bn<0, 0>(g.BN);
}

}  // namespace

size_t gemm_bf16_smem_bytes(const GemmArgs& g) {
  const size_t ring = static_cast<size_t>(g.stages) * stage_bytes(g.BN, g.short_a);
  const size_t red = static_cast<size_t>(tile_rows(g.short_a)) * (g.BN + 4) * sizeof(float);
  return (ring > red ? ring : red) + 256 + 1024;
}

int gemm_bf16_ctas_per_sm(const GemmArgs& g) {
  // one residency count per (device, shared-memory size, kernel)
  static std::mutex mu;
  static std::map<std::tuple<int, size_t, int, int, int>, int> counts;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  const size_t bytes = gemm_bf16_smem_bytes(g);
  const auto key = std::make_tuple(dev, bytes, g.BN, g.a_mn_major, g.b_mn_major);
  {
    std::lock_guard<std::mutex> lock(mu);
    const auto it = counts.find(key);
    if (it != counts.end()) return it->second;
  }
  const void* k = kernel_for(g);
  const int n = k ? resident_ctas_per_sm(k, 128, bytes, g.BN) : 0;
  std::lock_guard<std::mutex> lock(mu);
  if (n > 0) counts[key] = n;
  return n;
}

// Stand-in for the cluster occupancy query: asked about the GEMM kernel itself
// (66 KB form, GB300) the driver answers 76 clusters of two CTAs and 46 of
// three, as if one CTA filled an SM, against 228 and 148 for an empty kernel
// with the same block size and shared memory; so the query runs on that
// empty kernel, and registers and TMEM are counted separately by the caller.
__global__ void __launch_bounds__(128, 1) k_cluster_fit(int* p) {
  extern __shared__ int fit_smem[];
  if (p) p[threadIdx.x] = fit_smem[threadIdx.x];
}

int gemm_bf16_max_clusters(const GemmArgs& g) {
  static std::mutex mu;
  static std::map<std::tuple<int, size_t, int, int, int, int, int, int>, int> counts;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  const size_t bytes = gemm_bf16_smem_bytes(g);
  const dim3 grid((g.N + g.BN - 1) / g.BN, (g.M + BM - 1) / BM, g.splits);
  const auto key = std::make_tuple(dev, bytes, g.BN, g.a_mn_major, g.b_mn_major, g.splits,
                                   static_cast<int>(grid.x), static_cast<int>(grid.y));
  {
    std::lock_guard<std::mutex> lock(mu);
    const auto it = counts.find(key);
    if (it != counts.end()) return it->second;
  }
  const void* k = reinterpret_cast<const void*>(k_cluster_fit);
  if (raise_smem_limit(k, bytes) != cudaSuccess) return 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(128);
  cfg.dynamicSmemBytes = bytes;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = 1;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = g.splits;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, k, &cfg) != cudaSuccess) {
    (void)cudaGetLastError();
    n = 0;
  }
  std::lock_guard<std::mutex> lock(mu);
  if (n > 0) counts[key] = n;
  return n;
}

cudaError_t launch_gemm_bf16(const CUtensorMap& ta, const CUtensorMap& tb, const GemmArgs& g,
                             cudaStream_t st) {
  if (g.splits < 1 || g.splits > 8) return cudaErrorInvalidValue;
  if (g.stages < 1 || g.stages > kGemmStages) return cudaErrorInvalidValue;
  if (g.short_a && (g.a_mn_major || g.M > BM / 2)) return cudaErrorInvalidValue;
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
