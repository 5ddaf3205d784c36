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
#include <mutex>

#include "instant.h"

namespace {

constexpr size_t kScratchBytes = INSTANT_GRAD_X_STATIC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

// g_hat_x of one call: [B*Ry, Cx] in the call's dtype.  The first kernel
// overwrites every element the second one reads (no accumulation, and rows
// past Ry in a tile come from the TMA zero fill, not from memory), so the
// buffer never needs clearing.
__device__ __align__(256) unsigned char g_gxh_scratch[kScratchBytes];

std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device, looked up once
// per device with that device current.  The lookup may load the module on
// that device, which is why the first call on a device has to happen outside
// any stream capture.
cudaError_t scratch_address(void** out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_gxh_scratch);
    if (e != cudaSuccess) return e;
    if (!p) return cudaErrorInvalidSymbol;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
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
  void* ws = nullptr;
  if (scratch_address(&ws) != cudaSuccess) return INSTANT_ERR_CUDA;
  const instant_status s = instant_grad_x_core(Sq, w, ws, kScratchBytes, B, Cx, Cy, Ry, dt, stream);
  if (s != INSTANT_OK) return s;
  return instant_expand(Q, gx, ws, kScratchBytes, B, L, Cx, Cy, Ry, dt, stream);
}
