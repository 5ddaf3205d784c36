// static_scratch.cu -- input gradient with the g_hat_x intermediate held in a
// fixed, module-scope device buffer instead of caller-provided workspace.
//
// Some callers cannot hand the library a workspace: a plain C host that links
// only this library has no device allocator of its own, and a training loop
// whose device memory is planned once at start-up must not allocate after the
// steady state has begun (a cudaMalloc there synchronises the device and
// breaks the plan).  instant_grad_x_static serves them.  It runs the two-kernel
// form of the input gradient (g_hat_x = Sq w, then g_tilde_x = Q^T g_hat_x,
// page "INSTANT: Compressing Gradients and Activations for Resource-Efficient
// Training", 关键设计 3) with g_hat_x parked in `g_gxh_scratch` below, whose
// storage the CUDA module reserves when it loads.  Nothing here calls
// cudaMalloc, cudaFree or any routine that allocates device memory.
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

#include "instant.h"
#include "kernels.h"

namespace {

constexpr size_t kScratchBytes = INSTANT_GRAD_X_STATIC_SCRATCH_BYTES;

// g_hat_x of one call: [B*Ry, Cx] in the call's dtype.  The first kernel
// overwrites every element the second one reads (no accumulation, and rows
// past Ry in a tile come from the TMA zero fill, not from memory), so the
// buffer never needs clearing.
__device__ __align__(256) unsigned char g_gxh_scratch[kScratchBytes];

// Device address of the scratch array in the current device's context.  It
// is looked up on every call rather than cached: a cached address would go
// stale if the context were destroyed and recreated (cudaDeviceReset), and the
// lookup is cheap once the module is loaded.  The first lookup on a device
// may load the module there, which is why the first call on a device has to
// happen outside any stream capture.
cudaError_t scratch_address(void** out) {
  void* p = nullptr;
  const cudaError_t e = cudaGetSymbolAddress(&p, g_gxh_scratch);
  if (e != cudaSuccess) return e;
  if (!p) return cudaErrorInvalidSymbol;
  *out = p;
  return cudaSuccess;
}

}  // namespace

extern "C" instant_status instant_grad_x_static(const void* Sq, const void* w, const void* Q,
                                                void* gx, int B, int L, int Cx, int Cy, int Ry,
                                                instant_dtype dt, void* stream) {
  if (dt != INSTANT_F32 && dt != INSTANT_BF16) return INSTANT_ERR_DTYPE;
  if (!Sq || !w || !Q || !gx) return INSTANT_ERR_ARG;
  if (B < 1 || L < 1 || Cx < 1 || Cy < 1 || Ry < 1 || Ry > 64) return INSTANT_ERR_SHAPE;
  const size_t need = instant_grad_x_workspace_bytes(B, L, Cx, Cy, Ry, dt);
  if (need == 0 || need > kScratchBytes) return INSTANT_ERR_WORKSPACE;
  // the layout rules of the bf16 path, checked before any CUDA call (the
  // array itself is 256-byte aligned)
  const auto aligned16 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
  if (dt == INSTANT_BF16 && (!aligned16(Sq) || !aligned16(w) || !aligned16(gx) || Cx % 8 != 0 ||
                             Cy % 8 != 0))
    return INSTANT_ERR_ALIGN;
  void* ws = nullptr;
  if (scratch_address(&ws) != cudaSuccess) return INSTANT_ERR_CUDA;
  // both launches are checked and planned before the first is issued
  return instant::grad_x_two_kernels(Sq, w, Q, gx, ws, kScratchBytes, B, L, Cx, Cy, Ry, dt,
                                     static_cast<cudaStream_t>(stream));
}
