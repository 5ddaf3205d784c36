// expand.cu -- rank-R expansion of the input gradient (page "INSTANT:
// Compressing Gradients and Activations for Resource-Efficient Training",
// 关键设计 3):  g_tilde_x,b = Q^T g_hat_x,b,   [L, Ry] x [Ry, Cx] per sample.
//
// The step writes the full [B, L, Cx] gradient while reading only Q and the
// small g_hat_x, so it is bound by HBM writes.  With 2*Ry flops per output
// element the FFMA pipes cannot keep up with the write stream at Ry >= 8, so
// the contraction runs on the tensor cores: one CTA computes a 128-token x BN
// tile as a single K = Ry (padded to 16) tcgen05 MMA.  Both operands are tiny
// and are built by the threads directly in the K-major 128-byte-swizzle layout
// (Q^T from Q, g_hat_x by summing the split-K partial planes of the previous
// GEMM and rounding to bf16).  The epilogue converts the fp32 TMEM tile to bf16
// and writes 32-byte runs per row.
#include "kernels.h"
#include "tc.cuh"

namespace instant {

namespace {

constexpr int BM = 128;

template <int BN>
__global__ void __launch_bounds__(128, 1) k_expand_bf16(ExpandArgs e) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* sA = smem;                       // [128 tokens][128 B]: Q^T, K-major
  uint8_t* sB = smem + BM * 128;            // [BN cols][128 B]: g_hat_x^T, K-major
  uint64_t* done = reinterpret_cast<uint64_t*>(sB + BN * 128);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int n0 = blockIdx.x * BN;
  const int l0 = blockIdx.y * BM;
  const int b = blockIdx.z;

  if (threadIdx.x == 0) {
    mbar_init(done, 1);
    fence_barrier_init();
  }
  if (warp == 0) {
    tmem_alloc(tmem_slot, BN);
    tmem_relinquish();
  }

  // A[m, k] = Q[k, l0 + m]  (zero past Ry or past L)
  const uint16_t* Q = static_cast<const uint16_t*>(e.Q);
  for (int idx = threadIdx.x; idx < e.KR * BM; idx += blockDim.x) {
    const int k = idx / BM;
    const int m = idx - k * BM;
    const int l = l0 + m;
    const uint16_t v = (k < e.Ry && l < e.L) ? Q[static_cast<size_t>(k) * e.L + l] : 0;
    *reinterpret_cast<uint16_t*>(sA + sw128_offset(m, k)) = v;
  }
  // B[n, k] = sum_s gxh[s][b*Ry + k, n0 + n]  (zero past Ry or past Cx)
  const size_t plane = static_cast<size_t>(e.B) * e.Ry * e.Cx;
  for (int idx = threadIdx.x; idx < e.KR * BN; idx += blockDim.x) {
    const int k = idx / BN;
    const int n = idx - k * BN;
    const int c = n0 + n;
    float acc = 0.f;
    if (k < e.Ry && c < e.Cx) {
      const float* src = e.gxh + (static_cast<size_t>(b) * e.Ry + k) * e.Cx + c;
      for (int s = 0; s < e.splits; ++s) acc += src[s * plane];
    }
    *reinterpret_cast<uint16_t*>(sB + sw128_offset(n, k)) = bf16_bits(acc);
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 1 && lane == 0) {
    constexpr uint32_t idesc = idesc_bf16_f32(128, BN, 0, 0);
    const uint32_t a_base = smem_u32(sA);
    const uint32_t b_base = smem_u32(sB);
    for (int kk = 0; kk < e.KR / 16; ++kk) {
      const uint64_t ad = sdesc_sw128(a_base + kk * 32, 16, 1024);
      const uint64_t bd = sdesc_sw128(b_base + kk * 32, 16, 1024);
      umma_bf16(tmem, ad, bd, idesc, kk != 0);
    }
    umma_commit(done);
  }
  __syncwarp();
  if (!mbar_wait(done, 0)) raise_fault(FAULT_WAIT_DONE);
  tc_fence_after();

  const int l = l0 + warp * 32 + lane;
  const uint32_t taddr = tmem + (static_cast<uint32_t>(warp * 32) << 16);
  uint16_t* orow = static_cast<uint16_t*>(e.out) + (static_cast<size_t>(b) * e.L + l) * e.Cx;
#pragma unroll 1
  for (int j0 = 0; j0 < BN; j0 += 16) {
    float v[16];
    tmem_ld16(taddr + j0, v);
    const int c = n0 + j0;
    if (l < e.L) {
      if (c + 16 <= e.Cx) {
        uint32_t p[8];
#pragma unroll
        for (int q = 0; q < 8; ++q)
          p[q] = static_cast<uint32_t>(bf16_bits(v[2 * q])) |
                 (static_cast<uint32_t>(bf16_bits(v[2 * q + 1])) << 16);
        uint4* dst = reinterpret_cast<uint4*>(orow + c);
        dst[0] = make_uint4(p[0], p[1], p[2], p[3]);
        dst[1] = make_uint4(p[4], p[5], p[6], p[7]);
      } else {
#pragma unroll
        for (int q = 0; q < 16; ++q)
          if (c + q < e.Cx) orow[c + q] = bf16_bits(v[q]);
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, BN);
}

// fp32 path: one thread per output element.
__global__ void k_expand_f32(ExpandArgs e) {
  const int c = blockIdx.x * blockDim.x + threadIdx.x;
  const int l = blockIdx.y;
  const int b = blockIdx.z;
  if (c >= e.Cx) return;
  const float* Q = static_cast<const float*>(e.Q);
  const size_t plane = static_cast<size_t>(e.B) * e.Ry * e.Cx;
  float acc = 0.f;
  for (int r = 0; r < e.Ry; ++r) {
    const float* src = e.gxh + (static_cast<size_t>(b) * e.Ry + r) * e.Cx + c;
    float g = 0.f;
    for (int s = 0; s < e.splits; ++s) g += src[s * plane];
    acc = fmaf(Q[static_cast<size_t>(r) * e.L + l], g, acc);
  }
  static_cast<float*>(e.out)[(static_cast<size_t>(b) * e.L + l) * e.Cx + c] = acc;
}

template <int BN>
cudaError_t launch_bn(const ExpandArgs& e, cudaStream_t st) {
  const size_t bytes = expand_bf16_smem_bytes(e);
  static size_t configured_ = 0;
  if (bytes > configured_) {
    cudaError_t err = cudaFuncSetAttribute(k_expand_bf16<BN>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(bytes));
    if (err != cudaSuccess) return err;
    configured_ = bytes;
  }
  dim3 grid((e.Cx + BN - 1) / BN, (e.L + BM - 1) / BM, e.B);
  k_expand_bf16<BN><<<grid, 128, bytes, st>>>(e);
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace

size_t expand_bf16_smem_bytes(const ExpandArgs& e) {
  return BM * 128 + static_cast<size_t>(e.BN) * 128 + 64 + 1024;
}

cudaError_t launch_expand_bf16(const ExpandArgs& e, cudaStream_t st) {
  switch (e.BN) {
    case 128: return launch_bn<128>(e, st);
    case 256: return launch_bn<256>(e, st);
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
