// gradx_fused.cu -- input gradient in one kernel (page "INSTANT: Compressing
// Gradients and Activations for Resource-Efficient Training", 关键设计 3:
// g_hat_x = g_hat_y2 w, g_tilde_x = Q^T g_hat_x), so that g_hat_x never
// leaves the SM.
//
// A CTA owns a tile of `spt` whole samples (spt * Ry <= 128 rows of g_hat_x),
// a BN-column strip of the output, and a range of 128-token tiles:
//   phase 1  TMEM acc1[128 x BN] = Sq[tile rows, :] w[:, strip]  (tcgen05, K = Cy
//            streamed through a TMA ring: Sq K-major, w MN-major; only the
//            tile's spt * Ry rows of Sq are copied, the MMA rows past them read
//            whatever the stage holds and are never used);
//   phase 2  the epilogue warps turn acc1 into bf16 and write, per sample, the
//            MN-major B operand [Ry (padded to 16) x BN] of the expansion
//            straight into shared memory.  When the token range is split over
//            a cluster (dims 1 x 1 x cl), each CTA's phase 1 covers only a
//            slice of K = Cy; the slices are summed through DSMEM (each CTA
//            reduces a share of the rows from all peers' fp32 partials, then
//            writes the bf16 rows into every CTA's operands: two cluster
//            barriers);
//   phase 3  for every (sample, token tile): TMEM acc2 = Q^T[tile] B_s (one
//            K = Ry MMA chain, two accumulators in flight) -> bf16 -> swizzled
//            staging (reusing the phase-1 ring) -> TMA bulk store.
// Used when the K-slice of Cy per cluster CTA stays short (at most 16 chunks
// of 64); the token range is split across the cluster for parallelism.
//
// The same launch can also compute the weight gradient g_w = Sx^T x_hat
// (关键设计 3): extra grid rows of CTAs (clusters of their own, no cluster
// barrier) each produce one 128 x 64 fp32 tile of g_w, so that both products
// of the backward pass share one launch and fill the SMs the input gradient
// leaves free.
//
// And it can start one step earlier, from g_y itself (the whole backward of
// the layer in one launch): clusters take tickets as they start; the first
// tickets are projection tiles (sample, 128 columns of g_y -> Sx, Sq, one per
// CTA), then the input-gradient items of the sample groups in order, then the
// weight-gradient tiles.  Each projection tile adds to its group's counter and
// to a total (release); phase 1 of a group waits for its group's count, the
// weight-gradient tiles for the total (acquire, bounded).  A consumer only
// waits for smaller tickets, held by clusters that are running and never
// wait themselves, so the waits end whatever the scheduling; the last CTA
// zeroes the counters for the next launch.
#include <mutex>

#include "kernels.h"
#include "project_tile.cuh"
#include "tc.cuh"

namespace instant {

namespace {

constexpr int BM = 128;
constexpr int BK = 64;
constexpr int A_BYTES = BM * BK * 2;  // 16 KB
constexpr int BOX = BM * 128;         // staging box: 128 rows x 64 bf16

struct FLay {
  uint32_t ring, stage, qt, qt_tile, bs, bs_sample, stg, bar, pbar, total;
};

// gw: the launch also runs weight-gradient tiles, whose 3-stage ring needs 72 KB;
// proj_bytes: the projection phase's ring (0: none), also at the start
// A slot of a phase-1 stage: with at most 64 rows of Sq (and 64-column strips)
// only 8 KB are loaded; the M = 128 MMA then reads rows 64..127 from the B
// slot after it, results that are never used.  The smaller stage lets the
// ring run deeper.
__host__ __device__ inline uint32_t fused_a_bytes(int a_rows, int BN) {
  return (a_rows <= 64 && BN == 64) ? A_BYTES / 2 : A_BYTES;
}

__host__ __device__ inline FLay fused_layout(int BN, int KR, int stages, int lt_per, int spt,
                                             bool gw, uint32_t proj_bytes, uint32_t a_bytes) {
  FLay l;
  l.stage = a_bytes + BN * BK * 2;
  l.ring = 0;
  const uint32_t ring_bytes = stages * l.stage;
  const uint32_t stg_bytes = 4 * (BN / 64) * BOX;  // staging reuses the ring after phase 1
  const uint32_t red_bytes = BM * (BN + 4) * 4;     // so does the cluster reduction tile
  uint32_t first = ring_bytes > stg_bytes ? ring_bytes : stg_bytes;
  if (red_bytes > first) first = red_bytes;
  if (gw && first < 3u * (A_BYTES + 64 * BK * 2)) first = 3u * (A_BYTES + 64 * BK * 2);
  if (first < proj_bytes) first = proj_bytes;
  first = (first + 1023u) & ~1023u;
  l.stg = 0;
  l.qt = first;
  l.qt_tile = 2 * KR * 128;
  l.bs = l.qt + lt_per * l.qt_tile;
  l.bs_sample = (BN / 64) * KR * 128;
  l.bar = l.bs + spt * l.bs_sample;
  l.pbar = l.bar + 256;
  l.total = l.pbar + 128;
  return l;
}

__host__ __device__ inline uint32_t fused_proj_bytes(const FusedArgs& f) {
  return f.proj ? proj_layout(f.pa.NT, f.pa.nk, f.pa.pq_tma).bytes : 0u;
}

// last action of every CTA of a launch with the projection phase: the CTA
// that finishes last (all others are past all their waits) zeroes the
// counters for the next launch
__device__ __forceinline__ void proj_launch_done(const FusedArgs& f) {
  if (threadIdx.x != 0) return;
  unsigned int* done = f.sync + f.gw_y0 + 1;
  const unsigned int ctas = gridDim.x * gridDim.y * gridDim.z;
  if (atomicAdd(done, 1u) == ctas - 1) {
    for (int i = 0; i < f.gw_y0 + 3; ++i) f.sync[i] = 0u;
  }
}

// Work items of a launch with the projection phase, in ticket order: first
// the projection tiles (cl per cluster), then the input-gradient items (one
// (sample group, column strip) per cluster, groups in order), then the
// weight-gradient tiles (cl per cluster).  Consumers only wait for items with
// smaller tickets, which running clusters hold and finish without waiting.
struct ProjItems {
  int nstrips, n_tiles, n_pc, n_xc, n_gc;
};

__host__ __device__ inline ProjItems proj_items(const FusedArgs& f) {
  ProjItems w;
  w.nstrips = (f.Cx + f.BN - 1) / f.BN;
  w.n_tiles = f.B * f.nct;
  w.n_pc = (w.n_tiles + f.cl - 1) / f.cl;
  w.n_xc = f.gw_y0 * w.nstrips;
  w.n_gc = (f.gw_mt * w.nstrips + f.cl - 1) / f.cl;
  return w;
}

// one projection tile of g_y (u = sample * nct + column tile; none when u is
// past the last tile) into Sx and Sq, then its signals: one for the sample's
// group and one in total
__device__ __forceinline__ void proj_item(const CUtensorMap* tmap_gy, const CUtensorMap* tmap_pq,
                                          const FusedArgs& f, uint8_t* smem, uint32_t pbar_off,
                                          int u) {
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + pbar_off);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + kProjBarriers);
  const uint32_t cols = f.pa.NT <= 32 ? 32 : (f.pa.NT <= 64 ? 64 : 128);
  ProjPipe pipe = proj_pipe(smem, bars, f.pa.NT, f.pa.nk, f.pa.pq_tma, 0);
  if (threadIdx.x == 0) {
    proj_init_barriers(pipe);
    fence_barrier_init();
    prefetch_tmap(tmap_gy);
    if (f.pa.pq_tma) prefetch_tmap(tmap_pq);
  }
  if (threadIdx.x < 32) {
    tmem_alloc(tmem_slot, cols);
    tmem_relinquish();
  }
  if (!f.pa.pq_tma) proj_fill_pq(f.pa, pipe, f.pa.NT, threadIdx.x, blockDim.x);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  pdl_launch_dependents();  // after the allocation
  pipe.tmem = *tmem_slot;
  if (u < f.B * f.nct && threadIdx.x < 128) {
    const int b = u / f.nct;
    proj_tile<2>(tmap_gy, tmap_pq, f.pa, f.pa.NT, b, (u % f.nct) * kProjBM, pipe);
    // publish: the tile's stores, then the signals
    __threadfence();
    fence_proxy_async_global();
    named_barrier<3>(128);
    if (threadIdx.x == 0) {
      signal_add(f.sync + b / f.spt, 1u);
      signal_add(f.sync + f.gw_y0, 1u);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (threadIdx.x < 32) tmem_dealloc(pipe.tmem, cols);
}

// One 128 x 64 tile of g_w[Cy, Cx] = Sx^T x_hat (K = B * Rx): Sx [K, Cy] and
// x_hat [K, Cx] both arrive MN-major by TMA through a 3-stage ring (the first
// 72 KB of shared memory); warps 2..9 store the fp32 tile (or add it to g_w).
__device__ __forceinline__ void grad_w_tile(const CUtensorMap* tmap_sx, const CUtensorMap* tmap_xh,
                                            const FusedArgs& f, uint8_t* smem, uint32_t bar_off,
                                            int m0, int n0) {
  constexpr uint32_t STAGE = A_BYTES + 64 * BK * 2;  // 24 KB
  const int nk = f.gw_nk;
  const int NS = nk < 3 ? (nk < 1 ? 1 : nk) : 3;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + bar_off);
  uint64_t* empty = full + 3;
  uint64_t* done = empty + 3;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done + 1);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < 3; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(done, 1);
    fence_barrier_init();
    prefetch_tmap(tmap_sx);
    prefetch_tmap(tmap_xh);
  }
  if (warp == 0) {
    tmem_alloc(tmem_slot, 64);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  pdl_launch_dependents();
  pdl_wait();
  if (warp == 0 && lane == 0) {
    if (f.proj) {
      // Sx comes from the projection phase of this launch: all of its tiles
      if (!wait_signal(f.sync + f.gw_y0, static_cast<unsigned>(f.B * f.nct)))
        raise_fault(FAULT_WAIT_SIGNAL);
      fence_proxy_async_global();
    }
    int issued = 0;
    int s = 0, par = 0;  // ring slot and round parity of chunk i, kept without divisions
    for (int i = 0; i < nk; ++i) {
      if (i >= NS && !mbar_wait(&empty[s], par ^ 1)) {
        raise_fault(FAULT_WAIT_EMPTY);
        break;
      }
      uint8_t* sa = smem + s * STAGE;
      const int k0 = i * BK;
      mbar_arrive_expect_tx(&full[s], STAGE);
      tma_load_2d(sa, tmap_sx, &full[s], m0, k0);
      tma_load_2d(sa + A_BYTES / 2, tmap_sx, &full[s], m0 + 64, k0);
      tma_load_2d(sa + A_BYTES, tmap_xh, &full[s], n0, k0);
      ++issued;
      if (++s == NS) {
        s = 0;
        par ^= 1;
      }
    }
    for (int i = issued - NS < 0 ? 0 : issued - NS; i < issued; ++i)
      if (!mbar_wait(&full[i % NS], (i / NS) & 1)) raise_fault(FAULT_WAIT_FULL);
  } else if (warp == 1 && lane == 0) {
    constexpr uint32_t idesc = idesc_bf16_f32(128, 64, /*a_mn=*/1, /*b_mn=*/1);
    bool ok = true;
    int s = 0, par = 0;
    for (int i = 0; i < nk; ++i) {
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
        const uint64_t ad = sdesc_sw128(a_base + kk * 2048, A_BYTES / 2, 1024);
        const uint64_t bd = sdesc_sw128(b_base + kk * 2048, 64 * BK * 2, 1024);
        umma_bf16(tmem, ad, bd, idesc, (i | kk) != 0);
      }
      umma_commit(&empty[s]);
      if (++s == NS) {
        s = 0;
        par ^= 1;
      }
    }
    if (ok && nk > 0) umma_commit(done);
  }
  __syncwarp();
  if (warp >= 2) {
    if (nk > 0 && !mbar_wait(done, 0)) raise_fault(FAULT_WAIT_DONE);
    tc_fence_after();
    const int quarter = warp & 3;
    const int c0 = ((warp - 2) >> 2) * 32;
    float v[32];
    if (nk > 0) {
      tmem_ld32(tmem + (static_cast<uint32_t>(quarter * 32) << 16) + c0, v);
    } else {
#pragma unroll
      for (int q = 0; q < 32; ++q) v[q] = 0.f;
    }
    const int m = m0 + quarter * 32 + lane;
    if (m < f.Cy) {
      float* dst = f.gw + static_cast<size_t>(m) * f.Cx + n0 + c0;
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        if (n0 + c0 + 4 * q < f.Cx) {
          float4 o = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
          if (f.gw_acc) {
            const float4 p = *reinterpret_cast<const float4*>(dst + 4 * q);
            o.x += p.x; o.y += p.y; o.z += p.z; o.w += p.w;
          }
          *reinterpret_cast<float4*>(dst + 4 * q) = o;
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, 64);
}

template <int BN>
// two CTAs per SM: at most 102 registers a thread (with more, as an
// instrumented build once had, the SM held one CTA and the grid ran in two waves)
__global__ void __launch_bounds__(320, 2)
    k_gradx_fused(const __grid_constant__ CUtensorMap tmap_sq,
                  const __grid_constant__ CUtensorMap tmap_w,
                  const __grid_constant__ CUtensorMap tmap_q,
                  const __grid_constant__ CUtensorMap tmap_out,
                  const __grid_constant__ CUtensorMap tmap_sx,
                  const __grid_constant__ CUtensorMap tmap_xh,
                  const __grid_constant__ CUtensorMap tmap_gy,
                  const __grid_constant__ CUtensorMap tmap_pq, FusedArgs f) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const int KR = f.KR;
  const int NS = f.stages;
  const uint32_t a_bytes = fused_a_bytes(f.a_rows, BN);
  const FLay lay = fused_layout(BN, KR, NS, f.lt_per, f.spt, f.gw_mt > 0, fused_proj_bytes(f), a_bytes);
  uint8_t* ring = smem + lay.ring;
  uint8_t* stg = smem + lay.stg;
  uint8_t* sQ = smem + lay.qt;
  uint8_t* sB = smem + lay.bs;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + lay.bar);
  uint64_t* empty = full + NS;
  uint64_t* acc1_full = empty + NS;
  uint64_t* b_ready = acc1_full + 1;
  uint64_t* q_full = b_ready + 1;
  uint64_t* t_full = q_full + 1;
  uint64_t* t_empty = t_full + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(t_empty + 2);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int crank = blockIdx.z;                  // rank in the cluster (dims 1 x 1 x cl)
  int item_x = blockIdx.x;                       // column strip
  int item_y = blockIdx.y;                       // sample group
  __shared__ unsigned int s_ticket;
  if (f.proj) {
    // (every path below lets the next kernel launch only after its own TMEM
    // allocation: a CTA of the next kernel holding TMEM while it waits for
    // this grid must never be what an allocation here waits for)
    pdl_wait();  // the counters are this launch's only once its predecessor has finished
    if (crank == 0 && threadIdx.x == 0) {
      const unsigned int t = atomicAdd(f.sync + f.gw_y0 + 2, 1u);
      for (int q = 0; q < f.cl; ++q) dsmem_st_u32(dsmem_addr(&s_ticket, q), t);
    }
    cluster_sync();
    const int T = static_cast<int>(s_ticket);
    const ProjItems w = proj_items(f);
    if (T < w.n_pc) {
      proj_item(&tmap_gy, &tmap_pq, f, smem, lay.pbar, T * f.cl + crank);
      proj_launch_done(f);
      return;
    }
    if (T >= w.n_pc + w.n_xc) {
      const int u = (T - w.n_pc - w.n_xc) * f.cl + crank;  // weight-gradient tile
      if (BN == 64 && u < f.gw_mt * w.nstrips) {
        grad_w_tile(&tmap_sx, &tmap_xh, f, smem, lay.bar, (u / w.nstrips) * BM,
                    (u % w.nstrips) * BN);
      } else {
        pdl_launch_dependents();
        __syncthreads();
      }
      proj_launch_done(f);
      return;
    }
    item_y = (T - w.n_pc) / w.nstrips;
    item_x = (T - w.n_pc) % w.nstrips;
  } else if (BN == 64 && static_cast<int>(blockIdx.y) >= f.gw_y0) {
    // weight-gradient rows of the grid (clusters of their own)
    const int mt = (static_cast<int>(blockIdx.y) - f.gw_y0) * f.cl + static_cast<int>(blockIdx.z);
    if (mt < f.gw_mt) grad_w_tile(&tmap_sx, &tmap_xh, f, smem, lay.bar, mt * BM, blockIdx.x * BN);
    return;
  }
  const int n0 = item_x * BN;
  const int s0 = item_y * f.spt;                 // first sample of the tile
  const int m0 = s0 * f.Ry;                      // first g_hat_x row of the tile
  const int lt0 = crank * f.lt_per;              // first token tile
  const int kper = f.kfull ? f.nk : (f.nk + f.cl - 1) / f.cl;  // phase-1 chunks per rank
  const int kc0 = f.kfull ? 0 : crank * kper;
  int nkc = f.nk - kc0;
  if (nkc > kper) nkc = kper;
  if (nkc < 0) nkc = 0;
  int nlt = f.nlt - lt0;
  if (nlt > f.lt_per) nlt = f.lt_per;
  if (nlt < 0) nlt = 0;
  int nsamp = f.B - s0;
  if (nsamp > f.spt) nsamp = f.spt;
  const int njobs = nsamp * (nlt > 0 ? nlt : 0);
  constexpr uint32_t kCols = BN == 64 ? 256 : 512;  // acc1 + two acc2 buffers

  if (threadIdx.x == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(acc1_full, 1);
    mbar_init(b_ready, 1);
    mbar_init(q_full, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&t_full[i], 1);
      mbar_init(&t_empty[i], 4);  // one arrival per warp of the epilogue group
    }
    fence_barrier_init();
    prefetch_tmap(&tmap_sq);
    prefetch_tmap(&tmap_w);
    if (f.q_tma) prefetch_tmap(&tmap_q);
    prefetch_tmap(&tmap_out);
    // this CTA's K-slice of the w strip into L2 while the predecessor finishes
    for (int i = 0; i < nkc; ++i)
      for (int h = 0; h < BN / 64; ++h)
        if (n0 + 64 * h < f.Cx) tma_prefetch_l2_2d(&tmap_w, n0 + 64 * h, (kc0 + i) * BK);
  }
  if (warp == 0) {
    tmem_alloc(tmem_slot, kCols);
    tmem_relinquish();
  }
  // zero the expansion operands: rows Ry..KR-1 of every sample stay zero
  for (uint32_t i = threadIdx.x * 16; i < static_cast<uint32_t>(f.spt) * lay.bs_sample;
       i += blockDim.x * 16)
    *reinterpret_cast<uint4*>(sB + i) = make_uint4(0, 0, 0, 0);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t acc1 = tmem;
  pdl_launch_dependents();
  pdl_wait();

  if (warp == 0) {
    // ---------------- producer ----------------
    const uint16_t* Q = static_cast<const uint16_t*>(f.Q);
    if (f.q_tma) {
      if (lane == 0) {
        mbar_arrive_expect_tx(q_full, nlt * lay.qt_tile);
        for (int t = 0; t < nlt; ++t) {
          uint8_t* dst = sQ + t * lay.qt_tile;
          tma_load_2d(dst, &tmap_q, q_full, (lt0 + t) * BM, 0);
          tma_load_2d(dst + KR * 128, &tmap_q, q_full, (lt0 + t) * BM + 64, 0);
        }
      }
    } else {
      for (int t = 0; t < nlt; ++t) {
        uint8_t* dst = sQ + t * lay.qt_tile;
        for (int idx = lane; idx < KR * BM; idx += 32) {
          const int r = idx / BM;
          const int ll = idx - r * BM;
          const int l = (lt0 + t) * BM + ll;
          const uint16_t v = (r < f.Ry && l < f.L) ? Q[static_cast<size_t>(r) * f.L + l] : 0;
          *reinterpret_cast<uint16_t*>(dst + (ll >> 6) * KR * 128 + sw128_offset(r, ll & 63)) = v;
        }
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(q_full);
    }
    if (lane == 0) {
      if (f.proj) {
        // the group's Sq rows come from the projection phase of its CTAs
        if (!wait_signal(f.sync + item_y, static_cast<unsigned>(nsamp * f.nct)))
          raise_fault(FAULT_WAIT_SIGNAL);
        fence_proxy_async_global();
      }
      int issued = 0;
      int s = 0, par = 0;  // ring slot and round parity of chunk i, kept without divisions
      for (int i = 0; i < nkc; ++i) {
        if (i >= NS && !mbar_wait(&empty[s], par ^ 1)) {
          raise_fault(FAULT_WAIT_EMPTY);
          break;
        }
        uint8_t* sa = ring + s * lay.stage;
        uint8_t* sb = sa + a_bytes;
        const int k0 = (kc0 + i) * BK;
        mbar_arrive_expect_tx(&full[s], f.a_rows * BK * 2 + BN * BK * 2);
        tma_load_2d(sa, &tmap_sq, &full[s], k0, m0);
#pragma unroll
        for (int h = 0; h < BN / 64; ++h)
          tma_load_2d(sb + h * (64 * BK * 2), &tmap_w, &full[s], n0 + 64 * h, k0);
        ++issued;
        if (++s == NS) {
          s = 0;
          par ^= 1;
        }
      }
      for (int i = issued - NS < 0 ? 0 : issued - NS; i < issued; ++i)
        if (!mbar_wait(&full[i % NS], (i / NS) & 1)) raise_fault(FAULT_WAIT_FULL);
      if (!mbar_wait(q_full, 0)) raise_fault(FAULT_WAIT_FULL);
    }
  }
  if (warp == 1) {
    // ---------------- MMA issuer, phase 1 ----------------
    if (lane == 0) {
      constexpr uint32_t idesc1 = idesc_bf16_f32(128, BN, /*a_mn=*/0, /*b_mn=*/1);
      bool ok = true;
      int s = 0, par = 0;
      for (int i = 0; i < nkc; ++i) {
        if (!mbar_wait(&full[s], par)) {
          raise_fault(FAULT_WAIT_FULL);
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t a_base = smem_u32(ring + s * lay.stage);
        const uint32_t b_base = a_base + a_bytes;
#pragma unroll
        for (int kk = 0; kk < BK / 16; ++kk) {
          const uint64_t ad = sdesc_sw128(a_base + kk * 32, 16, 1024);
          const uint64_t bd = sdesc_sw128(b_base + kk * 2048, 64 * BK * 2, 1024);
          umma_bf16(acc1, ad, bd, idesc1, (i | kk) != 0);
        }
        umma_commit(&empty[s]);
        if (++s == NS) {
          s = 0;
          par ^= 1;
        }
      }
      if (ok) umma_commit(acc1_full);
    }
  }
  __syncwarp();

  // ---------------- phase 2: g_hat_x tile -> bf16 expansion operands ----------------
  // epilogue warps 2..9: two per TMEM lane quarter, each owning half the columns
  const bool epi = warp >= 2;
  const int et = threadIdx.x - 64;   // 0..255 for the epilogue warps
  const int quarter = warp & 3;
  const int row = quarter * 32 + lane;
  const int c_lo = ((warp - 2) >> 2) * (BN / 2);
  const uint32_t t1 = acc1 + (static_cast<uint32_t>(quarter * 32) << 16);
  const int real_rows = f.spt * f.Ry;
  constexpr int LDR = BN + 4;
  float* red = reinterpret_cast<float*>(ring);  // the ring is idle once acc1 is complete
  if (epi) {
    if (nkc > 0 && !mbar_wait(acc1_full, 0)) raise_fault(FAULT_WAIT_DONE);
    tc_fence_after();
    fence_proxy_async_smem();
  }
  if (f.cl > 1 && !f.kfull) {
    // every CTA of the cluster holds a K-slice of the tile.  Reduce-scatter:
    // CTA r sums rows [r*rows_per, ...) over all slices; all-gather: it writes
    // the bf16 result into the expansion operands of every CTA of the cluster.
    if (epi) {
#pragma unroll 1
      for (int j0 = c_lo; j0 < c_lo + BN / 2; j0 += 32) {
        float v[32];
        if (nkc > 0) {
          tmem_ld32(t1 + j0, v);
        } else {
#pragma unroll
          for (int q = 0; q < 32; ++q) v[q] = 0.f;
        }
#pragma unroll
        for (int q = 0; q < 8; ++q)
          *reinterpret_cast<float4*>(red + row * LDR + j0 + 4 * q) =
              make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
      }
      tc_fence_before();
    }
    cluster_sync();
    if (epi) {
      const int rows_per = (real_rows + f.cl - 1) / f.cl;
      const int r_begin = crank * rows_per;
      constexpr int C4 = BN / 4;
      for (int idx = et; idx < rows_per * C4; idx += 256) {
        const int rr = r_begin + idx / C4;
        if (rr >= real_rows) break;
        const int c4 = (idx % C4) * 4;
        const float* src = red + rr * LDR + c4;
        float4 acc = *reinterpret_cast<const float4*>(src);
        float4 part[8];
#pragma unroll
        for (int q = 0; q < 8; ++q)
          if (q < f.cl && q != crank) part[q] = dsmem_ld_f4(dsmem_addr(src, q));
#pragma unroll
        for (int q = 0; q < 8; ++q)
          if (q < f.cl && q != crank) {
            acc.x += part[q].x; acc.y += part[q].y; acc.z += part[q].z; acc.w += part[q].w;
          }
        const uint2 pk = make_uint2(pack_bf16x2(acc.x, acc.y), pack_bf16x2(acc.z, acc.w));
        const int s_r = rr / f.Ry;
        const int r_r = rr - s_r * f.Ry;
        uint8_t* dst = sB + s_r * lay.bs_sample + (c4 >> 6) * KR * 128 + sw128_offset(r_r, c4 & 63);
        *reinterpret_cast<uint2*>(dst) = pk;
#pragma unroll
        for (int q = 0; q < 8; ++q)
          if (q < f.cl && q != crank) dsmem_st_u2(dsmem_addr(dst, q), pk);
      }
      fence_proxy_async_cluster();  // the operands feed the tensor cores of every CTA
    }
    cluster_sync();  // operands gathered everywhere; peers are done with this CTA's slice
  } else if (epi) {
    const int s_row = row / f.Ry;
    const int r_row = row - s_row * f.Ry;
    {
#pragma unroll 1
      for (int j0 = c_lo; j0 < c_lo + BN / 2; j0 += 32) {
        float v[32];
        tmem_ld32(t1 + j0, v);
        if (row < real_rows) {
          uint8_t* base = sB + s_row * lay.bs_sample + (j0 >> 6) * KR * 128;
          const int c = j0 & 63;
#pragma unroll
          for (int q = 0; q < 4; ++q)
            *reinterpret_cast<uint4*>(base + sw128_offset(r_row, c + 8 * q)) =
                make_uint4(pack_bf16x2(v[8 * q], v[8 * q + 1]), pack_bf16x2(v[8 * q + 2], v[8 * q + 3]),
                           pack_bf16x2(v[8 * q + 4], v[8 * q + 5]),
                           pack_bf16x2(v[8 * q + 6], v[8 * q + 7]));
        }
      }
    }
    tc_fence_before();
  }
  if (epi) {
    fence_proxy_async_smem();
    named_barrier<1>(256);
    if (et == 0) mbar_arrive(b_ready);
  }

  if (warp == 1) {
    // ---------------- MMA issuer, phase 3 ----------------
    if (lane == 0) {
      constexpr uint32_t idesc2 = idesc_bf16_f32(128, BN, /*a_mn=*/1, /*b_mn=*/1);
      bool ok = mbar_wait(b_ready, 0);
      if (!ok) raise_fault(FAULT_WAIT_DONE);
      if (ok && !mbar_wait(q_full, 0)) {
        raise_fault(FAULT_WAIT_FULL);
        ok = false;
      }
      tc_fence_after();
      const uint32_t q_base = smem_u32(sQ);
      const uint32_t b_base = smem_u32(sB);
      int s = 0, t = 0;  // (sample, token tile) of job j, kept without divisions
      for (int j = 0; ok && j < njobs; ++j) {
        const int buf = j & 1;
        if (j >= 2 && !mbar_wait(&t_empty[buf], ((j >> 1) - 1) & 1)) {
          raise_fault(FAULT_WAIT_EMPTY);
          break;
        }
        tc_fence_after();
        const uint32_t ab = q_base + t * lay.qt_tile;
        const uint32_t bb = b_base + s * lay.bs_sample;
        for (int kk = 0; kk < KR / 16; ++kk) {
          const uint64_t ad = sdesc_sw128(ab + kk * 2048, KR * 128, 1024);
          const uint64_t bd = sdesc_sw128(bb + kk * 2048, KR * 128, 1024);
          umma_bf16(tmem + BN + buf * BN, ad, bd, idesc2, kk != 0);
        }
        umma_commit(&t_full[buf]);
        if (++t == nlt) {
          t = 0;
          ++s;
        }
      }
    }
  } else if (epi) {
    // phase 3: expansion tiles -> TMA stores (staging reuses the phase-1 ring,
    // whose TMA writes all completed before acc1 did).  Two groups of four
    // warps: group g converts jobs g, g+2, ... from accumulator g into its own
    // two staging buffers and tracks its own store groups.
    fence_proxy_async_smem();
    const int grp = (warp - 2) >> 2;
    const int gt = et & 127;
    int it = 0;
    int s = grp / nlt, t = grp - (grp / nlt) * nlt;  // (sample, token tile) of job j
    for (int j = grp; j < njobs; j += 2, ++it) {
      uint8_t* st = stg + (2 * grp + (it & 1)) * (BN / 64) * BOX;
      if (gt == 0 && it >= 2) tma_store_wait_read<1>();
      if (grp == 0) named_barrier<2>(128); else named_barrier<3>(128);
      if (!mbar_wait(&t_full[grp], it & 1)) raise_fault(FAULT_WAIT_DONE);
      tc_fence_after();
      const uint32_t taddr = tmem + BN + grp * BN + (static_cast<uint32_t>(quarter * 32) << 16);
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
      if (grp == 0) named_barrier<2>(128); else named_barrier<3>(128);
      if (gt == 0) {
        for (int h = 0; h < BN / 64; ++h)
          if (n0 + 64 * h < f.Cx)
            tma_store_3d(&tmap_out, st + h * BOX, n0 + 64 * h, (lt0 + t) * BM, s0 + s);
        tma_store_commit();
      }
      t += 2;
      while (t >= nlt) {
        t -= nlt;
        ++s;
      }
    }
    if (gt == 0) tma_store_wait_all();
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, kCols);
  if (f.proj) proj_launch_done(f);
}

dim3 fused_grid(const FusedArgs& f) {
  if (f.proj) {
    const ProjItems w = proj_items(f);
    return dim3(w.n_pc + w.n_xc + w.n_gc, 1, f.cl);
  }
  const int gw_rows = f.gw_mt > 0 ? (f.gw_mt + f.cl - 1) / f.cl : 0;
  return dim3((f.Cx + f.BN - 1) / f.BN, f.gw_y0 + gw_rows, f.cl);
}

size_t fused_smem_bytes(const FusedArgs& f) {
  size_t b = fused_layout(f.BN, f.KR, f.stages, f.lt_per, f.spt, f.gw_mt > 0, fused_proj_bytes(f),
                          fused_a_bytes(f.a_rows, f.BN))
                 .total +
             1024;
  // with the projection phase at most two CTAs share an SM, so that two
  // CTAs' TMEM (256 columns each) always fits and no allocation waits on a
  // CTA that waits for a signal
  if (f.proj && b < 80 * 1024) b = 80 * 1024;
  return b;
}

template <int BN>
cudaError_t configure_smem(size_t bytes) {
  return raise_smem_limit(reinterpret_cast<const void*>(k_gradx_fused<BN>), bytes);
}

template <int BN>
cudaError_t launch_bn(const CUtensorMap& ts, const CUtensorMap& tw, const CUtensorMap& tq,
                      const CUtensorMap& to, const CUtensorMap& tsx, const CUtensorMap& txh,
                      const CUtensorMap& tgy, const CUtensorMap& tpq, const FusedArgs& f,
                      cudaStream_t st) {
  const size_t bytes = fused_smem_bytes(f);
  const cudaError_t e = configure_smem<BN>(bytes);
  if (e != cudaSuccess) return e;
  const dim3 grid = fused_grid(f);
  return launch_ex(k_gradx_fused<BN>, grid, dim3(320), bytes, st, f.cl, pdl_enabled(), ts, tw, tq,
                   to, tsx, txh, tgy, tpq, f);
}


}  // namespace

size_t gradx_fused_smem_bytes(const FusedArgs& f) { return fused_smem_bytes(f); }

cudaError_t launch_gradx_fused(const CUtensorMap& tmap_sq, const CUtensorMap& tmap_w,
                               const CUtensorMap& tmap_q, const CUtensorMap& tmap_out,
                               const CUtensorMap& tmap_sx, const CUtensorMap& tmap_xh,
                               const CUtensorMap& tmap_gy, const CUtensorMap& tmap_pq,
                               const FusedArgs& f, cudaStream_t st) {
  if (f.stages < 1 || f.stages > 6 || f.spt < 1 || f.spt * f.Ry > 128) return cudaErrorInvalidValue;
  if (f.a_rows < f.spt * f.Ry || f.a_rows > BM || f.a_rows % 8 != 0) return cudaErrorInvalidValue;
  if (f.cl != 1 && f.cl != 2 && f.cl != 4 && f.cl != 8) return cudaErrorInvalidValue;
  if (f.lt_per * f.cl < f.nlt) return cudaErrorInvalidValue;
  if (f.gw_y0 != (f.B + f.spt - 1) / f.spt) return cudaErrorInvalidValue;
  if (f.gw_mt > 0 && (f.BN != 64 || !f.gw || f.gw_nk < 1)) return cudaErrorInvalidValue;
  if (f.proj && (!f.sync || f.BN != 64 || f.nct != (f.Cy + kProjBM - 1) / kProjBM ||
                 f.pa.C != f.Cy || f.pa.B != f.B || f.pa.NT < 16 || f.pa.NT > 128 ||
                 f.pa.NT % 16 != 0))
    return cudaErrorInvalidValue;
  switch (f.BN) {
    case 64:
      return launch_bn<64>(tmap_sq, tmap_w, tmap_q, tmap_out, tmap_sx, tmap_xh, tmap_gy, tmap_pq,
                           f, st);
    case 128:
      return launch_bn<128>(tmap_sq, tmap_w, tmap_q, tmap_out, tmap_sx, tmap_xh, tmap_gy, tmap_pq,
                            f, st);
    default: return cudaErrorInvalidValue;
  }
}

INSTANT_FAULT_READER(read_fault_fused)

}  // namespace instant
