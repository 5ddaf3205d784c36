// project_tile.cuh -- one tile of the token-axis projection
//   out_r[b, c] = sum_l PQ[r, l] * t[b, l, c]     (c in a 128-column tile)
// on the tensor cores, shared by the projection kernel (one tile per CTA) and
// the fused backward kernel (the projection of g_y as the first phase of the
// CTAs that then consume it).
//
// Page "INSTANT: Compressing Gradients and Activations for Resource-Efficient
// Training": 整体框架 (x_hat = P x) and 关键设计 3 (g_hat_y1 = g_y^T P^T and
// g_hat_y2 = Q g_y read off one pass over g_y with the stacked [P; Q]).
//
// D[c, r] = sum_l t[l, c] PQ[r, l]: M = 128 columns of t, N = Rx + Ry padded
// to 16 (NT), K = L streamed in 64-token chunks.  t is the MN-major A operand
// (two 64-column TMA boxes per chunk), PQ the K-major B operand (by TMA per
// chunk when L % 8 == 0, else filled into shared memory once by the threads).
// Thread roles within threads 0..127: warp 0 lane 0 issues the TMA copies,
// warp 1 lane 0 the MMAs, warps 0-3 read the accumulator (one column of t per
// TMEM lane), stage it as bf16 rows in the idle ring and write both planes in
// 16-byte pieces (2-byte stores per row and column cost ~1 us per step graph
// of a BERT-base block on GB300).
#pragma once

#include "kernels.h"
#include "tc.cuh"

namespace instant {

constexpr int kProjBM = 128;                    // columns of t per tile (MMA M)
constexpr int kProjBK = 64;                     // tokens per chunk
constexpr int kProjABytes = kProjBM * kProjBK * 2;  // 16 KB: two 64-column boxes
constexpr int kProjHalfA = kProjABytes / 2;

// ring of ns (kProjectStages, or 2 for tiles of at most two chunks) A stages,
// then the PQ stages (or all of PQ)
struct ProjLayout {
  uint32_t a_off, b_off, b_stage_bytes, bytes;
};

__host__ __device__ inline ProjLayout proj_layout(int NT, int nk, int pq_tma, int ns = kProjectStages) {
  ProjLayout l;
  l.a_off = 0;
  l.b_off = ns * kProjABytes;
  l.b_stage_bytes = NT * 128;
  const uint32_t b_total = pq_tma ? ns * l.b_stage_bytes : nk * l.b_stage_bytes;
  l.bytes = l.b_off + ((b_total + 1023u) & ~1023u);
  return l;
}

// per-CTA pipeline state; every role thread advances its own copy identically
struct ProjPipe {
  uint64_t* full;    // [ns]
  uint64_t* empty;   // [ns]
  uint64_t* done;    // accumulator complete
  uint8_t* sA;
  uint8_t* sB;
  uint32_t b_stage_bytes;
  uint32_t tmem;     // accumulator: NT fp32 columns
  int chunk;         // chunks that have gone through the ring
  int tiles;         // tiles finished
};

__device__ __forceinline__ ProjPipe proj_pipe(uint8_t* region, uint64_t* bars, int NT, int nk,
                                              int pq_tma, uint32_t tmem, int ns = kProjectStages) {
  const ProjLayout l = proj_layout(NT, nk, pq_tma, ns);
  ProjPipe p;
  p.full = bars;
  p.empty = bars + ns;
  p.done = bars + 2 * ns;
  p.sA = region + l.a_off;
  p.sB = region + l.b_off;
  p.b_stage_bytes = l.b_stage_bytes;
  p.tmem = tmem;
  p.chunk = 0;
  p.tiles = 0;
  return p;
}

constexpr int kProjBarriers = 2 * kProjectStages + 1;  // room for the deepest ring

// one thread, before the CTA-wide barrier that publishes the initialisation
__device__ __forceinline__ void proj_init_barriers(const ProjPipe& p, int ns = kProjectStages) {
  for (int s = 0; s < ns; ++s) {
    mbar_init(&p.full[s], 1);
    mbar_init(&p.empty[s], 1);
  }
  mbar_init(p.done, 1);
}

// whole projector into shared memory, K-major with the 128-byte swizzle (when
// PQ does not arrive by TMA); any number of threads, before a CTA barrier
__device__ __forceinline__ void proj_fill_pq(const ProjectArgs& a, const ProjPipe& p, int NT,
                                             int tid, int nthreads) {
  const int Rt = a.Rx + a.Ry;
  const uint16_t* pq = static_cast<const uint16_t*>(a.pq);
  const int per_chunk = NT * kProjBK;
  for (int idx = tid; idx < a.nk * per_chunk; idx += nthreads) {
    const int kc = idx / per_chunk;
    const int rem = idx - kc * per_chunk;
    const int r = rem / kProjBK;
    const int col = rem - r * kProjBK;
    const int l = kc * kProjBK + col;
    const uint16_t v = (r < Rt && l < a.L) ? pq[static_cast<size_t>(r) * a.L + l] : 0;
    *reinterpret_cast<uint16_t*>(p.sB + kc * p.b_stage_bytes + sw128_offset(r, col)) = v;
  }
  fence_proxy_async_smem();
}

// The leading a.pf_chunks chunks of the t tile of (sample b, columns c0 ..)
// into L2, by one thread, before the wait for the predecessor (the CTA is
// resident early under programmatic dependent launch, and its first loads
// then hit L2).
__device__ __forceinline__ void proj_prefetch(const CUtensorMap* tmap_t, const ProjectArgs& a, int b,
                                              int c0, int k0 = 0, int nkl = -1) {
  const int nk = nkl < 0 ? a.nk : nkl;
  for (int i = 0; i < a.pf_chunks && i < nk; ++i) {
    tma_prefetch_l2_3d(tmap_t, c0, (k0 + i) * kProjBK, b);
    if (c0 + 64 < a.C) tma_prefetch_l2_3d(tmap_t, c0 + 64, (k0 + i) * kProjBK, b);
  }
}

// One tile (sample b, columns c0 .. c0+127), run by threads 0..127 (the other
// threads of the CTA must not touch the ring meanwhile).  On return every
// store of the tile has been issued by its thread and the accumulator is free
// for the next tile (named barrier BAR over the 128 threads).
// With part != nullptr the tile covers only the 64-token chunks k0 .. k0+nkl-1
// (one share of a token split) and, instead of writing the planes, leaves
// its fp32 partial sums in part[r * 128 + column], r < NT (shared memory of
// this CTA, e.g. the idle ring), for the caller to reduce.
template <int BAR, int NS = kProjectStages>
__device__ __forceinline__ void proj_tile(const CUtensorMap* tmap_t, const CUtensorMap* tmap_pq,
                                          const ProjectArgs& a, int NT, int b, int c0,
                                          ProjPipe& p, int k0 = 0, int nkl = -1,
                                          float* part = nullptr) {
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int nk = nkl < 0 ? a.nk : nkl;
  if (warp == 0 && lane == 0) {
    // ---------------- TMA producer ----------------
    const uint32_t bytes = kProjABytes + (a.pq_tma ? p.b_stage_bytes : 0);
    int issued = 0;
    for (int i = 0; i < nk; ++i) {
      const int g = p.chunk + i;
      const int s = g % NS;
      if (g >= NS && !mbar_wait(&p.empty[s], ((g / NS) - 1) & 1)) {
        raise_fault(FAULT_WAIT_EMPTY);
        break;
      }
      mbar_arrive_expect_tx(&p.full[s], bytes);
      uint8_t* dst = p.sA + s * kProjABytes;
      const int l0 = (k0 + i) * kProjBK;
      tma_load_3d(dst, tmap_t, &p.full[s], c0, l0, b);
      tma_load_3d(dst + kProjHalfA, tmap_t, &p.full[s], c0 + 64, l0, b);
      if (a.pq_tma) tma_load_2d(p.sB + s * p.b_stage_bytes, tmap_pq, &p.full[s], l0, 0);
      ++issued;
    }
    // every copy this thread issued has landed before it moves on (the ring is
    // reused by whatever follows, also when the MMA side gave up)
    for (int i = issued - NS < 0 ? 0 : issued - NS; i < issued; ++i) {
      const int g = p.chunk + i;
      if (!mbar_wait(&p.full[g % NS], (g / NS) & 1))
        raise_fault(FAULT_WAIT_FULL);
    }
  } else if (warp == 1 && lane == 0) {
    // ---------------- MMA issuer ----------------
    const uint32_t idesc = idesc_bf16_f32(128, NT, /*a_mn=*/1, /*b_mn=*/0);
    bool ok = true;
    for (int i = 0; i < nk; ++i) {
      const int g = p.chunk + i;
      const int s = g % NS;
      if (!mbar_wait(&p.full[s], (g / NS) & 1)) {
        raise_fault(FAULT_WAIT_FULL);
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t a_base = smem_u32(p.sA + s * kProjABytes);
      const uint32_t b_base = smem_u32(p.sB + (a.pq_tma ? s : k0 + i) * p.b_stage_bytes);
#pragma unroll
      for (int kk = 0; kk < kProjBK / 16; ++kk) {
        // A (MN-major): 16 tokens = 2 groups of 8 rows of 128 B; the second
        // 64-column box is kProjHalfA bytes away.  B (K-major): +32 B per 16 tokens.
        const uint64_t ad = sdesc_sw128(a_base + kk * 2048, kProjHalfA, 1024);
        const uint64_t bd = sdesc_sw128(b_base + kk * 32, 16, 1024);
        umma_bf16(p.tmem, ad, bd, idesc, (i | kk) != 0);
      }
      umma_commit(&p.empty[s]);
    }
    if (ok && nk > 0) umma_commit(p.done);
  }
  __syncwarp();

  // ---------------- epilogue: TMEM -> bf16 planes ----------------
  if (nk > 0 && !mbar_wait(p.done, p.tiles & 1)) raise_fault(FAULT_WAIT_DONE);
  tc_fence_after();
  const int row = warp * 32 + lane;
  const uint32_t taddr = p.tmem + (static_cast<uint32_t>(warp * 32) << 16);
  uint16_t* out0 = static_cast<uint16_t*>(a.out0);
  uint16_t* out1 = static_cast<uint16_t*>(a.out1);
  const int Rt = a.Rx + a.Ry;
  if (part != nullptr) {
    // one share of a token split: the fp32 partial sums, for the caller
    for (int j0 = 0; j0 < NT; j0 += 16) {
      float v[16];
      if (nk > 0) {
        tmem_ld16(taddr + j0, v);
      } else {
#pragma unroll
        for (int jj = 0; jj < 16; ++jj) v[jj] = 0.f;
      }
#pragma unroll
      for (int jj = 0; jj < 16; ++jj) part[(j0 + jj) * kProjBM + row] = v[jj];
    }
    tc_fence_before();
    named_barrier<BAR>(128);  // accumulator read by all four warps
    tc_fence_after();
    p.chunk += nk;
    p.tiles += 1;
    return;
  }
  // the bf16 tile [Rt rows][128 columns] staged in the ring (idle: every MMA
  // has completed, so every copy into it has landed), then written back in
  // 16-byte pieces of the output rows
  uint16_t* stage = reinterpret_cast<uint16_t*>(p.sA);
  for (int j0 = 0; j0 < NT; j0 += 16) {
    float v[16];
    tmem_ld16(taddr + j0, v);
#pragma unroll
    for (int jj = 0; jj < 16; ++jj)
      if (j0 + jj < Rt) stage[(j0 + jj) * kProjBM + row] = bf16_bits(v[jj]);
  }
  tc_fence_before();
  named_barrier<BAR>(128);
  for (int idx = threadIdx.x; idx < Rt * (kProjBM / 8); idx += 128) {
    const int r = idx / (kProjBM / 8);
    const int piece = idx - r * (kProjBM / 8);
    const int c = c0 + piece * 8;
    uint16_t* dst = r < a.Rx ? out0 + (static_cast<size_t>(b) * a.Rx + r) * a.C + c
                             : out1 + (static_cast<size_t>(b) * a.Ry + (r - a.Rx)) * a.C + c;
    const uint16_t* src = stage + r * kProjBM + piece * 8;
    if (c + 8 <= a.C) {
      *reinterpret_cast<uint4*>(dst) = *reinterpret_cast<const uint4*>(src);
    } else {
      for (int e = 0; c + e < a.C; ++e) dst[e] = src[e];
    }
  }
  tc_fence_before();
  named_barrier<BAR>(128);  // accumulator read by all four warps
  tc_fence_after();
  p.chunk += nk;
  p.tiles += 1;
}

}  // namespace instant
