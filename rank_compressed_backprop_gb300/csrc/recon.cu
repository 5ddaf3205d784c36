// recon.cu -- how much of a tensor a projector keeps: ||t - Q^T Q t||_F^2 and
// ||t||_F^2 over a batch, with Q t already computed (the output of the
// projection kernel).  This is the error that the oversampling p of page
// "INSTANT: Compressing Gradients and Activations for Resource-Efficient
// Training", 关键设计 2, is meant to keep small while the subspace drifts
// between recalibrations.
//
// Memory-bound: t is read once, 16 bytes per thread and step; the projected
// rows S_b = Q t_b [R, C] of a sample stay in L1/L2 while its L token rows
// stream by; Q [R, L] is staged in shared memory.  Squares are summed in fp32
// per thread, then per block, and added to two fp64 totals.
#include "kernels.h"
#include "tc.cuh"

namespace instant {

namespace {

template <typename T>
__device__ __forceinline__ float to_f(T v);
template <>
__device__ __forceinline__ float to_f<float>(float v) { return v; }
template <>
__device__ __forceinline__ float to_f<uint16_t>(uint16_t v) { return bf16_to_f32(v); }

// eight consecutive elements from a 16-byte aligned address
__device__ __forceinline__ void load8(const uint16_t* p, float (&v)[8]) {
  const uint4 u = __ldg(reinterpret_cast<const uint4*>(p));
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    v[2 * k] = __uint_as_float(w[k] << 16);
    v[2 * k + 1] = __uint_as_float(w[k] & 0xffff0000u);
  }
}
__device__ __forceinline__ void load8(const float* p, float (&v)[8]) {
  const float4 a = __ldg(reinterpret_cast<const float4*>(p));
  const float4 b = __ldg(reinterpret_cast<const float4*>(p + 4));
  v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
  v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}

constexpr int kReconThreads = 256;
constexpr int kMaxR = 64;

// one (sample, token) row of C elements per loop trip; each thread owns
// columns [8 i, 8 i + 8) of that row
template <typename T>
__global__ void __launch_bounds__(kReconThreads)
    k_recon(const T* __restrict__ t, const T* __restrict__ Q, const T* __restrict__ S, int B, int L,
            int C, int R, int vec, double* totals) {
  extern __shared__ float qs[];  // [R][L]
  for (int i = threadIdx.x; i < R * L; i += blockDim.x) qs[i] = to_f(Q[i]);
  __syncthreads();
  float err = 0.f, en = 0.f;
  const int c8 = (C + 7) / 8;
  const long long rows = static_cast<long long>(B) * L;
  for (long long row = blockIdx.x; row < rows; row += gridDim.x) {
    const int b = static_cast<int>(row / L);
    const int l = static_cast<int>(row - static_cast<long long>(b) * L);
    const T* trow = t + row * C;
    const T* Sb = S + static_cast<size_t>(b) * R * C;
    for (int i = threadIdx.x; i < c8; i += blockDim.x) {
      const int c0 = 8 * i;
      float v[8], rec[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) rec[e] = 0.f;
      if (vec) {
        // 8 consecutive elements in one or two 16-byte loads
        load8(trow + c0, v);
        for (int r = 0; r < R; ++r) {
          const float q = qs[r * L + l];
          float sv[8];
          load8(Sb + static_cast<size_t>(r) * C + c0, sv);
#pragma unroll
          for (int e = 0; e < 8; ++e) rec[e] = fmaf(q, sv[e], rec[e]);
        }
      } else {
#pragma unroll
        for (int e = 0; e < 8; ++e) v[e] = c0 + e < C ? to_f(trow[c0 + e]) : 0.f;
        for (int r = 0; r < R; ++r) {
          const float q = qs[r * L + l];
          const T* srow = Sb + static_cast<size_t>(r) * C;
#pragma unroll
          for (int e = 0; e < 8; ++e)
            if (c0 + e < C) rec[e] = fmaf(q, to_f(srow[c0 + e]), rec[e]);
        }
      }
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const float d = v[e] - rec[e];
        err = fmaf(d, d, err);
        en = fmaf(v[e], v[e], en);
      }
    }
  }
  // block sums, then one fp64 atomic per total and block
  __shared__ float red[2][kReconThreads / 32];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    err += __shfl_xor_sync(0xffffffffu, err, o);
    en += __shfl_xor_sync(0xffffffffu, en, o);
  }
  if ((threadIdx.x & 31) == 0) {
    red[0][threadIdx.x >> 5] = err;
    red[1][threadIdx.x >> 5] = en;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    double e2 = 0.0, n2 = 0.0;
    for (int w = 0; w < static_cast<int>(blockDim.x >> 5); ++w) {
      e2 += red[0][w];
      n2 += red[1][w];
    }
    atomicAdd(&totals[0], e2);
    atomicAdd(&totals[1], n2);
  }
}

}  // namespace

cudaError_t launch_recon(const void* t, const void* Q, const void* S, int B, int L, int C, int R,
                         int bf16, double* totals, cudaStream_t st) {
  if (R < 1 || R > kMaxR || L < 1 || static_cast<size_t>(R) * L * sizeof(float) > 48 * 1024)
    return cudaErrorInvalidValue;
  cudaError_t e = cudaMemsetAsync(totals, 0, 2 * sizeof(double), st);
  if (e != cudaSuccess) return e;
  const long long rows = static_cast<long long>(B) * L;
  const long long cap = 4ll * sm_count();
  const int grid = static_cast<int>(rows < cap ? rows : cap);
  const size_t smem = sizeof(float) * R * L;
  // 16-byte loads when every row of t and S starts on a 16-byte boundary
  const int vec = (C % 8 == 0 && (reinterpret_cast<uintptr_t>(t) & 15) == 0 &&
                   (reinterpret_cast<uintptr_t>(S) & 15) == 0) ? 1 : 0;
  if (bf16)
    k_recon<uint16_t><<<grid, kReconThreads, smem, st>>>(
        static_cast<const uint16_t*>(t), static_cast<const uint16_t*>(Q),
        static_cast<const uint16_t*>(S), B, L, C, R, vec, totals);
  else
    k_recon<float><<<grid, kReconThreads, smem, st>>>(static_cast<const float*>(t),
                                                      static_cast<const float*>(Q),
                                                      static_cast<const float*>(S), B, L, C, R,
                                                      vec, totals);
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace instant
