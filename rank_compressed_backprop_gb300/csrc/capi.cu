// capi.cu -- the extern "C" boundary declared in include/instant.h: argument
// validation, tensor-map encoding, launch planning and the host loop of the
// calibration solve.  No device memory is allocated here.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <vector>
#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <cstdio>
#include <cstring>
#include <atomic>
#include <map>
#include <mutex>
#include <utility>

#include "instant.h"
#include "kernels.h"

using namespace instant;

namespace {
std::atomic<unsigned long long> g_launches{0};
}  // namespace

void instant::count_launches(unsigned int n) { g_launches.fetch_add(n, std::memory_order_relaxed); }

bool instant::pdl_enabled() {
  static const bool on = [] {
    const char* v = std::getenv("INSTANT_NO_PDL");
    return !(v && v[0] == '1');
  }();
  return on;
}

int instant::sm_count() {
  // queried once per device (the grids below are sized in multiples of it)
  static std::atomic<int> cache[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 1;
  int n = cache[dev].load(std::memory_order_relaxed);
  if (n > 0) return n;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1)
    return 1;
  cache[dev].store(n, std::memory_order_relaxed);
  return n;
}

cudaError_t instant::raise_smem_limit(const void* kernel, size_t bytes, bool max_shared) {
  static std::mutex mu;
  static std::map<std::pair<const void*, int>, size_t> configured;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(mu);
  size_t& have = configured[std::make_pair(kernel, dev)];
  if (bytes <= have) return cudaSuccess;
  if (max_shared) {
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                             static_cast<int>(cudaSharedmemCarveoutMaxShared));
    if (e != cudaSuccess) return e;
  }
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(bytes));
  if (e == cudaSuccess) have = bytes;
  return e;
}

int instant::resident_ctas_per_sm(const void* kernel, int threads, size_t smem, int tmem_cols) {
  cudaFuncAttributes fa;
  int dev = 0, smem_sm = 0, reserved = 0, regs_sm = 0, threads_sm = 0;
  if (cudaFuncGetAttributes(&fa, kernel) != cudaSuccess || cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&reserved, cudaDevAttrReservedSharedMemoryPerBlock, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&regs_sm, cudaDevAttrMaxRegistersPerMultiprocessor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&threads_sm, cudaDevAttrMaxThreadsPerMultiProcessor, dev) != cudaSuccess)
    return 0;
  const int warps = (threads + 31) / 32;
  const int regs_warp = (fa.numRegs * 32 + 255) / 256 * 256;
  const size_t per_cta = smem + fa.sharedSizeBytes + static_cast<size_t>(reserved);
  int n = 0;
  for (;;) {
    const int m = n + 1;
    const bool fits = static_cast<size_t>(m) * per_cta <= static_cast<size_t>(smem_sm) &&
                      m * threads <= threads_sm && (m * warps + 3) / 4 * regs_warp <= regs_sm / 4 &&
                      m * tmem_cols <= 512 && m <= 32;
    if (!fits) break;
    n = m;
  }
  return n;
}

namespace {

// ---------------------------------------------------------------------------
// tensor maps (driver entry point fetched through the runtime; no -lcuda)
// ---------------------------------------------------------------------------
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encoder() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// tiled map with the 128-byte swizzle (bf16 unless stated); dims/strides
// innermost first
bool make_map(CUtensorMap* m, const void* base, int rank, const uint64_t* dims,
              const uint64_t* strides_bytes, const uint32_t* box,
              CUtensorMapDataType type = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16) {
  EncodeTiledFn f = encoder();
  if (!f) return false;
  cuuint64_t d[5], s[5];
  cuuint32_t b[5], e[5];
  for (int i = 0; i < rank; ++i) {
    d[i] = dims[i];
    b[i] = box[i];
    e[i] = 1;
    if (i < rank - 1) s[i] = strides_bytes[i];
  }
  return f(m, type, rank, const_cast<void*>(base), d, s, b, e,
           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
int round_up(int x, int m) { return (x + m - 1) / m * m; }
int cdiv(int a, int b) { return (a + b - 1) / b; }

// INSTANT_ERR_CUDA for a failed CUDA call; with INSTANT_VERBOSE_ERRORS set the
// runtime's error string goes to stderr as well
instant_status from_cuda(cudaError_t e) {
  if (e == cudaSuccess) return INSTANT_OK;
  if (std::getenv("INSTANT_VERBOSE_ERRORS")) std::fprintf(stderr, "instant: %s\n", cudaGetErrorString(e));
  return INSTANT_ERR_CUDA;
}

bool dtype_ok(instant_dtype dt) { return dt == INSTANT_F32 || dt == INSTANT_BF16; }

bool fault_injected(const char* what) {
  const char* v = std::getenv("INSTANT_FAULT");
  return v && std::strcmp(v, what) == 0;
}

// ---------------------------------------------------------------------------
// projection (shared by compress_act and project_grad)
// ---------------------------------------------------------------------------
instant_status project(const void* t, const void* pq, void* out0, void* out1, int B, int L, int C,
                       int Rx, int Ry, instant_dtype dt, cudaStream_t st) {
  ProjectArgs a;
  a.B = B;
  a.L = L;
  a.C = C;
  a.Rx = Rx;
  a.Ry = Ry;
  a.NT = round_up(Rx + Ry, 16);
  a.nk = cdiv(L, 64);
  a.pq = pq;
  a.out0 = out0;
  a.out1 = out1;
  a.stages = kProjectStages;
  // token split: when the (sample, 128-column) tiles leave SMs idle or
  // unevenly loaded, up to four CTAs of a cluster share each tile's token axis
  // (every share at least 8 chunks of 64 tokens) and reduce their fp32 partial
  // sums through distributed shared memory.  INSTANT_PROJ_SPLIT=S forces S.
  {
    const long long tiles = static_cast<long long>(B) * cdiv(C, 128);
    a.split = 1;
    while (a.split < 4 && tiles * a.split < 2ll * sm_count() && a.nk / (a.split + 1) >= 8) ++a.split;
    if (const char* v = std::getenv("INSTANT_PROJ_SPLIT")) {
      const int f = std::atoi(v);
      if (f >= 1 && f <= 4) a.split = std::min(f, std::max(1, a.nk));
    }
    a.spb = 1;
  }
  // L2 prefetch: the whole tile while the grid's prefetches stay within a
  // quarter of L2 (all of a BERT-base batch), else the ring's worth.  The
  // count is taken before the plan below may split the token axis in two
  // with the two-stage ring; a split's shares then prefetch up to about half
  // of L2 (the long-sequence project_grad: 30.9 us, against 31.8 us with the
  // count taken after the split)
  {
    const long long ctas = static_cast<long long>(B) * cdiv(C, 128) * a.split;
    const long long budget = (32ll << 20) / std::max(1ll, ctas) / (128 * 64 * 2);
    a.pf_chunks = static_cast<int>(std::min<long long>(a.nk, std::max<long long>(kProjectStages, budget)));
  }
  if (dt == INSTANT_F32) {
    a.pq_tma = 0;
    return from_cuda(launch_project_f32(a, static_cast<const float*>(t), st));
  }
  a.pq_tma = (L % 8 == 0 && aligned16(pq)) ? 1 : 0;
  if (!a.pq_tma && static_cast<size_t>(a.nk) * a.NT * 128 > 96 * 1024) return INSTANT_ERR_SHAPE;
  // tiles of at most two chunks need no deeper ring: with two stages twice as
  // many CTAs share an SM and hide each other's per-sample latency.
  if (a.split == 1 && a.nk <= 2) a.stages = 2;
  // A streaming SM reads HBM at a fixed rate, so the launch lasts as long as
  // the SM with the most bytes streams.  Where halving the token axis (a
  // 2-CTA cluster, shares of at least 8 chunks) lowers the most tiles an SM
  // holds, and the halves all fit at once with the two-stage ring, split:
  // the long-sequence layer's 344 tiles put three on 40 SMs, 688 halves at
  // most five (2.5 tiles): project_grad 37.2 -> 30.9 us.  (Shorter token axes
  // lost more to the cluster's barriers: BERT-base 6.2 -> 7.9 us.)
  if (a.split == 1 && a.spb == 1 && a.nk >= 16 && a.NT <= 64 && !std::getenv("INSTANT_PROJ_SPLIT")) {
    const long long nsm = sm_count();
    const long long T = static_cast<long long>(B) * cdiv(C, 128);
    ProjectArgs h = a;
    h.split = 2;
    h.stages = 2;
    const int per_sm = project_bf16_ctas_per_sm(h);
    if (per_sm < 1) return INSTANT_ERR_CUDA;
    const long long most_whole = 2 * ((T + nsm - 1) / nsm);  // in half tiles
    const long long most_half = (2 * T + nsm - 1) / nsm;
    if (2 * T <= per_sm * nsm && most_half < most_whole) {
      a.split = 2;
      a.stages = 2;
    }
  }
  // INSTANT_PROJ_STAGES=2|4 forces the depth (2 with a split only up to NT = 64)
  if (const char* v = std::getenv("INSTANT_PROJ_STAGES")) {
    const int f = std::atoi(v);
    if (f == kProjectStages || (f == 2 && (a.split == 1 || a.NT <= 64))) a.stages = f;
  }
  // short token axes (at most 4 chunks): each CTA takes several consecutive
  // samples of its column tile, the fewest that still make the grid one wave
  // of resident CTAs (49-token ViT-MLP batches of 256: 7.0 / 17.6 us for
  // 1,024 / 3,584 tiles against 11.4 / 35.7 us at one sample per CTA and
  // 21.2 us for the latter at four, which took two waves).
  // INSTANT_PROJ_SPB=n forces n.
  if (a.split == 1) {
    if (a.nk <= 4) {
      const int per_sm = project_bf16_ctas_per_sm(a);
      if (per_sm < 1) return INSTANT_ERR_CUDA;
      const long long slots = static_cast<long long>(per_sm) * sm_count();
      const long long ct = cdiv(C, 128);
      long long s = std::max(1ll, (ct * B + slots - 1) / slots);
      while (s < B && ct * ((B + s - 1) / s) > slots) ++s;
      a.spb = static_cast<int>(std::min<long long>(s, B));
    }
    if (const char* v = std::getenv("INSTANT_PROJ_SPB")) {
      const int f = std::atoi(v);
      if (f >= 1) a.spb = std::min(f, B);
    }
  }
  CUtensorMap mt, mpq;
  std::memset(&mpq, 0, sizeof(mpq));
  const uint64_t dt3[3] = {static_cast<uint64_t>(C), static_cast<uint64_t>(L), static_cast<uint64_t>(B)};
  const uint64_t st3[2] = {static_cast<uint64_t>(C) * 2, static_cast<uint64_t>(L) * C * 2};
  const uint32_t bx3[3] = {64, 64, 1};
  if (!make_map(&mt, t, 3, dt3, st3, bx3)) return INSTANT_ERR_CUDA;
  if (a.pq_tma) {
    const uint64_t d2[2] = {static_cast<uint64_t>(L), static_cast<uint64_t>(Rx + Ry)};
    const uint64_t s2[1] = {static_cast<uint64_t>(L) * 2};
    const uint32_t b2[2] = {64, static_cast<uint32_t>(a.NT)};
    if (!make_map(&mpq, pq, 2, d2, s2, b2)) return INSTANT_ERR_CUDA;
  }
  return from_cuda(launch_project_bf16(mt, mpq, a, st));
}

// ---------------------------------------------------------------------------
// GEMM plan: N tile and split-K cluster size for an M x N x K product
// ---------------------------------------------------------------------------
struct GemmPlan {
  int BN, splits, cps, nk, stages, short_a;
};

// short_ok: A is K-major, so M <= 64 may take the 64-row A box (three CTAs
// share an SM instead of two).  With it K takes the most cluster shares (up to
// 8) whose CTAs and clusters all fit on the device at once: the long-sequence
// g_hat_x (64 x 4096, K = 11008, 64 column tiles) at 2 / 4 / 5 / 6 shares
// took 34 / 23 / 20 / 20 us, and at 7 shares (448 CTAs, not all placeable as
// 7-CTA clusters) 29 us.  Otherwise the largest split that keeps two waves'
// worth of work.
GemmPlan plan_gemm(int M, int N, int K, bool short_ok) {
  GemmPlan p;
  p.nk = cdiv(K, 64);
  p.short_a = short_ok && M <= 64 && !std::getenv("INSTANT_GEMM_LONG_A");
  const int tm = cdiv(M, 128);
  p.BN = 64;
  const int nsm = sm_count();
  for (int bn : {256, 128}) {
    if (tm * cdiv(N, bn) >= nsm) {
      p.BN = bn;
      break;
    }
  }
  if (const char* v = std::getenv("INSTANT_GEMM_BN")) {
    const int f = std::atoi(v);
    if (f == 64 || f == 128 || f == 256) p.BN = f;
  }
  const int tiles = tm * cdiv(N, p.BN);
  p.stages = 4;
  p.splits = 1;
  if (p.short_a) {
    GemmArgs g{};
    g.M = M;
    g.N = N;
    g.K = K;
    g.b_mn_major = 1;
    g.BN = p.BN;
    g.stages = p.stages;
    g.short_a = 1;
    const long long slots = static_cast<long long>(gemm_bf16_ctas_per_sm(g)) * nsm;
    for (int s = 2; s <= 8 && s <= p.nk; ++s) {
      g.splits = s;
      if (static_cast<long long>(tiles) * s > slots) break;
      if (gemm_bf16_max_clusters(g) >= tiles) p.splits = s;
    }
  } else {
    for (int s : {8, 4, 2}) {
      if (s <= p.nk && tiles * s <= 2 * nsm) {  // two waves' worth of work
        p.splits = s;
        break;
      }
    }
  }
  if (const char* v = std::getenv("INSTANT_GEMM_SPLITS")) {
    const int f = std::atoi(v);
    if (f >= 1 && f <= 8 && f <= p.nk) p.splits = f;
  }
  p.cps = cdiv(p.nk, p.splits);
  return p;
}

// weight gradient: the write-streaming kernel when the contraction fits its
// resident x_hat strip (K <= 256) and the output has several tiles per SM;
// else the split-K GEMM.  INSTANT_GRADW_PATH=gemm|stream forces one.
bool use_gradw_stream(int M, int N, int K) {
  if (K > 64 * kGradWMaxChunks) return false;
  const char* v = std::getenv("INSTANT_GRADW_PATH");
  if (v && std::strcmp(v, "gemm") == 0) return false;
  if (v && std::strcmp(v, "stream") == 0) return true;
  return static_cast<long long>(cdiv(M, 128)) * cdiv(N, 64) >= 4ll * sm_count();
}

// Split of the autocorrelation work (statistic p: B[p] samples of nkc[p]
// 64-channel chunks on each of `ntiles` tiles): cs[p] channel ranges per tile,
// each CTA walking all its samples in order (so the CTAs running at one time
// read the same sample and its tiles meet in L2), and bs[p] sample ranges only
// when the channel ranges alone cannot fill the GPU.  Among grids of w whole
// waves of two CTAs per SM (w = 1..8) it takes the one whose slowest CTA
// finishes first, counting a CTA's set-up and atomic flush as 12 iterations;
// a CTA keeps at least 4 iterations and a tile at most 64 CTAs (more
// concurrent atomic adds into one tile cost more than they save: 256 samples
// of 197 tokens on GB300).
void plan_syrk(int n, const int* B, const int* nkc, int ntiles, int per_sm, int* cs, int* bs) {
  const long long slots = static_cast<long long>(per_sm) * sm_count();
  double total = 0.0;
  for (int p = 0; p < n; ++p) total += static_cast<double>(B[p]) * nkc[p] * ntiles;
  double best = 1e300;
  for (int w = 1; w <= 8; ++w) {
    int c[kMaxSyrkBatch], s[kMaxSyrkBatch];
    long long ctas = 0;
    long long maxw = 0;
    for (int p = 0; p < n; ++p) {
      const double work = static_cast<double>(B[p]) * nkc[p] * ntiles;
      int per_tile = static_cast<int>(std::lround(w * slots * work / total / ntiles));
      per_tile = std::max(1, std::min(per_tile, 64));
      c[p] = std::min(per_tile, nkc[p]);
      s[p] = std::max(1, std::min(B[p], per_tile / c[p]));
      // at least 4 iterations per CTA
      while (c[p] * s[p] > 1 && static_cast<long long>(cdiv(nkc[p], c[p])) * cdiv(B[p], s[p]) < 4) {
        if (s[p] > 1) --s[p]; else --c[p];
      }
      ctas += static_cast<long long>(ntiles) * c[p] * s[p];
      maxw = std::max<long long>(maxw, static_cast<long long>(cdiv(nkc[p], c[p])) * cdiv(B[p], s[p]));
    }
    const long long waves = (ctas + slots - 1) / slots;
    const double cost = static_cast<double>(waves) * (maxw + 12);
    if (cost < best) {
      best = cost;
      for (int p = 0; p < n; ++p) {
        cs[p] = c[p];
        bs[p] = s[p];
      }
    }
  }
}

size_t grad_x_ws(int B, int Cx, int Cy, int Ry, instant_dtype dt) {
  (void)Cy;
  return static_cast<size_t>(B) * Ry * Cx * (dt == INSTANT_F32 ? sizeof(float) : 2);
}

}  // namespace

// ===========================================================================
// C ABI
// ===========================================================================
namespace {

// fused single-kernel input gradient when every CTA can afford to recompute
// its g_hat_x tile (small Cy); otherwise grad_x_core + expand
// token-axis cluster of the fused kernel: up to 8 CTAs, a power of two
int fused_cluster(int L) {
  const int nlt = cdiv(L, 128);
  int cl = 1;
  while (cl * 2 <= nlt && cl < 8) cl *= 2;
  return cl;
}

bool use_fused_grad_x(int B, int L, int Cx, int Cy, int Ry, instant_dtype dt) {
  if (dt != INSTANT_BF16 || Ry > 64) return false;
  if (std::getenv("INSTANT_NO_FUSED_GRAD_X")) return false;
  // a large g_tilde_x on 128-token tiles streams out faster from the
  // standalone expansion (one wave of equal job runs): on a 3072 -> 768 FFN
  // layer (B = 32, L = 512, 100 MB) g_hat_x, the expansion and g_w took
  // 36.6 us in three launches against 41.2 us fused, while the BERT-base
  // block (25 MB) stays fused (11.5 against 19.2 us), as do 49-token tiles
  if (L >= 128 && static_cast<long long>(B) * L * Cx * 2 > (64ll << 20)) return false;
  // each CTA recomputes a K-slice of its g_hat_x tile: keep that slice short
  return cdiv(cdiv(Cy, 64), fused_cluster(L)) <= 16;
}

// weight-gradient operands riding along in the fused launch (Sx == nullptr: none)
struct GradWPart {
  const void* Sx;
  const void* xhat;
  float* gw;
  int accumulate;
  int Rx;
};

// projection of g_y riding along in the fused launch (instant_backward)
struct ProjPart {
  const void* gy;    // [B, L, Cy]
  const void* PQ;    // [Rx + Ry, L]
  void* Sx;          // [B * Rx, Cy]
  int Rx;
  unsigned int* sync;  // zeroed counters, at least B + 3
};

// *no_room: the projector does not fit the projection phase's shared memory
// (nothing launched; the caller takes two launches)
instant_status grad_x_fused(const void* Sq, const void* w, const void* Q, void* gx, int B, int L,
                            int Cx, int Cy, int Ry, const GradWPart& gwp, cudaStream_t st,
                            const ProjPart* pp = nullptr, bool* no_room = nullptr) {
  FusedArgs f;
  f.B = B;
  f.L = L;
  f.Cx = Cx;
  f.Cy = Cy;
  f.Ry = Ry;
  f.KR = round_up(Ry, 16);
  f.spt = 128 / Ry;
  f.BN = 64;
  f.nk = cdiv(Cy, 64);
  f.nlt = cdiv(L, 128);
  f.cl = fused_cluster(L);
  f.lt_per = cdiv(f.nlt, f.cl);
  // a short K (at most 12 chunks) is cheaper to run whole in every CTA of the
  // cluster than to split and exchange: the FFN's 3072 -> 768 layer (B = 32,
  // L = 512) measured 41.7 us against 44.7 us, a BERT-base block the same
  // (11.5 against 11.6 us), the 768 -> 3072 layer (48 chunks) 28.0 against
  // 22.1 us split.  INSTANT_FUSED_KFULL=0/1 forces either form.
  f.kfull = (f.cl > 1 && f.nk <= 12) ? 1 : 0;
  if (const char* v = std::getenv("INSTANT_FUSED_KFULL")) f.kfull = (f.cl > 1 && std::atoi(v) != 0) ? 1 : 0;
  const int kper = f.kfull ? f.nk : cdiv(f.nk, f.cl);
  f.stages = kper < 3 ? (kper < 1 ? 1 : kper) : 3;  // deepened below for compact stages
  // smaller sample tiles when the grid would not cover the SMs
  while (f.spt > 2 && cdiv(Cx, f.BN) * cdiv(B, f.spt) * f.cl < sm_count()) f.spt /= 2;
  f.a_rows = std::min(128, round_up(f.spt * Ry, 8));
  f.q_tma = (L % 8 == 0 && aligned16(Q)) ? 1 : 0;
  f.Q = Q;
  f.gw_y0 = cdiv(B, f.spt);
  f.gw_mt = gwp.Sx ? cdiv(Cy, 128) : 0;
  f.gw_nk = gwp.Sx ? cdiv(B * gwp.Rx, 64) : 0;
  f.gw_acc = gwp.accumulate ? 1 : 0;
  f.gw = gwp.gw;
  CUtensorMap ms, mw, mq, mo, msx, mxh;
  std::memset(&mq, 0, sizeof(mq));
  std::memset(&msx, 0, sizeof(msx));
  std::memset(&mxh, 0, sizeof(mxh));
  if (gwp.Sx) {
    // Sx [B*Rx, Cy] and x_hat [B*Rx, Cx], both read MN-major in 64 x 64 boxes
    const uint64_t K = static_cast<uint64_t>(B) * gwp.Rx;
    const uint64_t da[2] = {static_cast<uint64_t>(Cy), K};
    const uint64_t sa[1] = {static_cast<uint64_t>(Cy) * 2};
    const uint64_t db[2] = {static_cast<uint64_t>(Cx), K};
    const uint64_t sb[1] = {static_cast<uint64_t>(Cx) * 2};
    const uint32_t bx[2] = {64, 64};
    if (!make_map(&msx, gwp.Sx, 2, da, sa, bx) || !make_map(&mxh, gwp.xhat, 2, db, sb, bx))
      return INSTANT_ERR_CUDA;
  }
  const uint64_t ds[2] = {static_cast<uint64_t>(Cy), static_cast<uint64_t>(B) * Ry};
  const uint64_t ss[1] = {static_cast<uint64_t>(Cy) * 2};
  const uint32_t bs[2] = {64, static_cast<uint32_t>(f.a_rows)};
  const uint64_t dw[2] = {static_cast<uint64_t>(Cx), static_cast<uint64_t>(Cy)};
  const uint64_t sw[1] = {static_cast<uint64_t>(Cx) * 2};
  const uint32_t bw[2] = {64, 64};
  const uint64_t dout[3] = {static_cast<uint64_t>(Cx), static_cast<uint64_t>(L), static_cast<uint64_t>(B)};
  const uint64_t sout[2] = {static_cast<uint64_t>(Cx) * 2, static_cast<uint64_t>(L) * Cx * 2};
  const uint32_t bout[3] = {64, 128, 1};
  if (!make_map(&ms, Sq, 2, ds, ss, bs) || !make_map(&mw, w, 2, dw, sw, bw) ||
      !make_map(&mo, gx, 3, dout, sout, bout))
    return INSTANT_ERR_CUDA;
  if (f.q_tma) {
    const uint64_t d2[2] = {static_cast<uint64_t>(L), static_cast<uint64_t>(Ry)};
    const uint64_t s2[1] = {static_cast<uint64_t>(L) * 2};
    const uint32_t b2[2] = {64, static_cast<uint32_t>(f.KR)};
    if (!make_map(&mq, Q, 2, d2, s2, b2)) return INSTANT_ERR_CUDA;
  }
  CUtensorMap mgy, mpq;
  std::memset(&mgy, 0, sizeof(mgy));
  std::memset(&mpq, 0, sizeof(mpq));
  f.proj = pp ? 1 : 0;
  f.nct = cdiv(Cy, 128);
  f.sync = pp ? pp->sync : nullptr;
  std::memset(&f.pa, 0, sizeof(f.pa));
  if (pp) {
    ProjectArgs& a = f.pa;
    a.B = B;
    a.L = L;
    a.C = Cy;
    a.Rx = pp->Rx;
    a.Ry = Ry;
    a.NT = round_up(pp->Rx + Ry, 16);
    a.nk = cdiv(L, 64);
    a.pq = pp->PQ;
    a.out0 = pp->Sx;
    a.out1 = const_cast<void*>(Sq);
    a.pq_tma = (L % 8 == 0 && aligned16(pp->PQ)) ? 1 : 0;
    a.pf_chunks = 0;  // its tiles start after the wait
    a.split = 1;
    a.spb = 1;
    a.stages = kProjectStages;
    if (!a.pq_tma && static_cast<size_t>(a.nk) * a.NT * 128 > 96 * 1024) {
      if (no_room) *no_room = true;
      return INSTANT_ERR_SHAPE;
    }
    const uint64_t dt3[3] = {static_cast<uint64_t>(Cy), static_cast<uint64_t>(L), static_cast<uint64_t>(B)};
    const uint64_t st3[2] = {static_cast<uint64_t>(Cy) * 2, static_cast<uint64_t>(L) * Cy * 2};
    const uint32_t bx3[3] = {64, 64, 1};
    if (!make_map(&mgy, pp->gy, 3, dt3, st3, bx3)) return INSTANT_ERR_CUDA;
    if (a.pq_tma) {
      const uint64_t d2[2] = {static_cast<uint64_t>(L), static_cast<uint64_t>(pp->Rx + Ry)};
      const uint64_t s2[1] = {static_cast<uint64_t>(L) * 2};
      const uint32_t b2[2] = {64, static_cast<uint32_t>(a.NT)};
      if (!make_map(&mpq, pp->PQ, 2, d2, s2, b2)) return INSTANT_ERR_CUDA;
    }
  }
  // at most 64 rows of Sq: 16 KB phase-1 stages, so up to 5 of them while two
  // CTAs still share an SM (a BERT-base block's phase 1 streams 12 chunks per
  // CTA against L2 latency: the deeper ring keeps more of them in flight)
  if (f.a_rows <= 64 && f.BN == 64 && kper > 3) {
    f.stages = std::min(kper, 5);
    while (f.stages > 3 && gradx_fused_smem_bytes(f) > 113 * 1024) --f.stages;
  }
  return from_cuda(launch_gradx_fused(ms, mw, mq, mo, msx, mxh, mgy, mpq, f, st));
}

// counters of the fused backward: per sample group (at most B), total, done, ticket
size_t backward_sync_bytes(int B) { return (static_cast<size_t>(B + 3) * 4 + 255) & ~static_cast<size_t>(255); }

// ---------------------------------------------------------------------------
// calibration solve of one statistic (instant_calib_solve and the batch call)
// ---------------------------------------------------------------------------
struct SolveJob {
  const float* C;
  int L;
  instant_calib_params prm;
  void* rows_out;
  int r_cap;
  int out_bf16;
  int max_iter, max_sweeps;
  double tol, inv_n, inv_n2;
  int m_block;  // subspace block of the first attempt
  bool warm;
  SolverWs w;
};

struct SolveOut {
  int k = 0, R = 0;
  float scale = 0.f;
  double energy = 0.0;
};

size_t solve_ws_stride(int L) { return (solver_workspace_bytes(L) + 255) & ~static_cast<size_t>(255); }

instant_status solve_prepare(const float* C, long long n_samples, int L,
                             const instant_calib_params* prm, void* rows_out, int r_cap,
                             instant_dtype dt, void* ws, size_t ws_bytes, SolveJob* j) {
  if (!dtype_ok(dt)) return INSTANT_ERR_DTYPE;
  if (!C || !prm || !rows_out) return INSTANT_ERR_ARG;
  if (n_samples < 1 || !(prm->eps > 0.0 && prm->eps <= 1.0) || prm->p < 0 || prm->r_override < 0)
    return INSTANT_ERR_ARG;
  if (L < 1 || L > 8192 || r_cap < 1 || r_cap > 128 || r_cap > L) return INSTANT_ERR_SHAPE;
  if (prm->r_override > r_cap) return INSTANT_ERR_SHAPE;
  if (!ws || ws_bytes < solver_workspace_bytes(L)) return INSTANT_ERR_WORKSPACE;
  if (!aligned16(ws)) return INSTANT_ERR_ALIGN;
  const bool noconv = fault_injected("solve_noconv");
  j->C = C;
  j->L = L;
  j->prm = *prm;
  j->rows_out = rows_out;
  j->r_cap = r_cap;
  j->out_bf16 = dt == INSTANT_BF16 ? 1 : 0;
  j->max_iter = noconv ? 1 : (prm->max_iter > 0 ? prm->max_iter : 300);
  j->max_sweeps = noconv ? 0 : 60;
  j->tol = prm->tol > 0.0 ? prm->tol : 2e-5;
  j->inv_n = 1.0 / static_cast<double>(n_samples);
  j->inv_n2 = j->inv_n * j->inv_n;
  // block: the needed rank plus a margin for the convergence rate
  const int r_guess = prm->r_override > 0 ? prm->r_override : prm->p + 8;
  j->m_block = std::min(128, std::max(16, round_up(std::max(2 * r_guess, r_guess + 8), 16)));
  j->warm = prm->warm_start != 0;
  j->w = solver_carve(ws, L);
  return INSTANT_OK;
}

// the whole iteration in one launch of an 8-CTA cluster, checked on the device
bool solve_uses_cluster(const SolveJob& j) {
  return j.L > 128 && cluster_solve_fits(j.L, j.m_block) && !std::getenv("INSTANT_SOLVER_MULTI");
}

ClusterSolveArgs cluster_args(const SolveJob& j) {
  ClusterSolveArgs ca;
  ca.C = j.C;
  ca.L = j.L;
  ca.m = j.m_block;
  ca.rp = 0;
  ca.inv_n = static_cast<float>(j.inv_n);
  ca.inv_n2 = j.inv_n2;
  ca.eps = j.prm.eps;
  ca.p = j.prm.p;
  ca.r_override = j.prm.r_override;
  ca.scale_on = j.prm.scale_on ? 1 : 0;
  ca.tol = j.tol;
  ca.max_iter = j.max_iter;
  ca.max_sweeps = j.max_sweeps;
  ca.rr_tol = 1e-5f;
  ca.seed = j.rows_out;
  ca.n_seed = j.warm ? std::min(j.r_cap, j.m_block) : 0;
  ca.seed_bf16 = j.out_bf16;
  ca.rows_out = j.rows_out;
  ca.r_cap = j.r_cap;
  ca.out_bf16 = j.out_bf16;
  ca.res = j.w.res;
  ca.Vg = j.w.V;
  return ca;
}

// outcome of a one-launch solve; false: k + p did not fit the block, and the
// multi-launch loop continues with twice the columns (rows_out still holds
// the caller's seed)
bool cluster_finish(SolveJob& j, const SolverResult& res, SolveOut* o, double* eig_out,
                    instant_status* status) {
  const double E = res.energy_sum * j.inv_n2;
  if (res.nonfinite || !std::isfinite(E) || !(E > 0.0)) {
    *status = INSTANT_ERR_NONFINITE;
    return true;
  }
  if (res.block_short) {
    j.m_block = std::min(128, 2 * j.m_block);
    return false;
  }
  instant_status st1 = res.converged ? INSTANT_OK : INSTANT_ERR_NOT_CONVERGED;
  if (res.jacobi_failed) st1 = INSTANT_ERR_NOT_CONVERGED;
  if (res.R > j.r_cap) st1 = INSTANT_ERR_SHAPE;
  o->k = res.k;
  o->R = res.R < j.r_cap ? res.R : j.r_cap;
  o->scale = res.scale;
  o->energy = E;
  if (eig_out)
    for (int i = 0; i < j.r_cap; ++i) eig_out[i] = i < j.m_block ? res.theta[i] : 0.0;
  *status = st1;
  return true;
}

// L <= 128 without host round trips: the energies, one full-Jacobi launch
// for all the statistics (one CTA each; a statistic whose energy is not
// finite and positive is skipped) and the projector rows, all queued on the
// stream; small_finish reads each result block afterwards
instant_status solve_small_async(std::vector<SolveJob*>& js, cudaStream_t st) {
  for (size_t i0 = 0; i0 < js.size(); i0 += kMaxJacobiBatch) {
    const size_t n = std::min<size_t>(kMaxJacobiBatch, js.size() - i0);
    JacobiBatch b;
    b.L = js[i0]->L;
    b.max_sweeps = js[i0]->max_sweeps;
    b.count = static_cast<int>(n);
    for (size_t u = 0; u < n; ++u) {
      SolveJob& j = *js[i0 + u];
      if (launch_solver_energy(j.C, j.L, j.w, st) != cudaSuccess) return INSTANT_ERR_CUDA;
      b.C[u] = j.C;
      b.inv_n[u] = static_cast<float>(j.inv_n);
      b.w[u] = j.w;
      b.max_sweeps = std::max(b.max_sweeps, j.max_sweeps);
    }
    if (launch_jacobi_full_batch(b, st) != cudaSuccess) return INSTANT_ERR_CUDA;
    for (size_t u = 0; u < n; ++u) {
      SolveJob& j = *js[i0 + u];
      if (launch_solver_finalize(j.L, j.L, j.prm.eps, j.prm.p, j.prm.r_override,
                                 j.prm.scale_on ? 1 : 0, j.rows_out, j.r_cap, j.out_bf16, j.inv_n2,
                                 j.w, st) != cudaSuccess)
        return INSTANT_ERR_CUDA;
    }
  }
  return INSTANT_OK;
}

void small_finish(const SolveJob& j, const SolverResult& res, SolveOut* o, double* eig_out,
                  instant_status* status) {
  const double E = res.energy_sum * j.inv_n2;
  if (res.nonfinite || !std::isfinite(E) || !(E > 0.0)) {
    *status = INSTANT_ERR_NONFINITE;
    return;
  }
  instant_status st1 = res.jacobi_failed ? INSTANT_ERR_NOT_CONVERGED : INSTANT_OK;
  if (res.R > j.r_cap && st1 == INSTANT_OK) st1 = INSTANT_ERR_SHAPE;
  o->k = res.k;
  o->R = res.R < j.r_cap ? res.R : j.r_cap;
  o->scale = res.scale;
  o->energy = E;
  if (eig_out)
    for (int i = 0; i < j.r_cap; ++i) eig_out[i] = i < j.L ? res.theta[i] : 0.0;
  *status = st1;
}

// energy, then full Jacobi (L <= 128) or the multi-launch subspace iteration
// with host-side convergence checks, then the projector rows
instant_status solve_multi(SolveJob& j, SolveOut* o, double* eig_out, cudaStream_t st) {
  const int L = j.L;
  SolverWs& w = j.w;
  SolverResult res;
  if (launch_solver_energy(j.C, L, w, st) != cudaSuccess) return INSTANT_ERR_CUDA;
  if (cudaMemcpyAsync(&res, w.res, sizeof(res), cudaMemcpyDeviceToHost, st) != cudaSuccess ||
      cudaStreamSynchronize(st) != cudaSuccess)
    return INSTANT_ERR_CUDA;
  const double E = res.energy_sum * j.inv_n2;
  if (res.nonfinite || !std::isfinite(E) || !(E > 0.0)) return INSTANT_ERR_NONFINITE;

  instant_status status = INSTANT_OK;
  int m = L;
  if (L <= 128) {
    if (launch_jacobi_full(j.C, L, j.inv_n, j.max_sweeps, w, st) != cudaSuccess)
      return INSTANT_ERR_CUDA;
  } else {
    m = j.m_block;
    bool converged = false;
    // warm start: the previous projector rows seed the block; the subspace has
    // usually moved little, so convergence is checked early and often
    for (;;) {
      const int n_seed = j.warm ? std::min(j.r_cap, m) : 0;
      if (launch_subspace_init(L, m, j.rows_out, n_seed, j.out_bf16, w, st) != cudaSuccess)
        return INSTANT_ERR_CUDA;
      bool grow = false;
      for (int it = 0; it < j.max_iter; ++it) {
        const bool check =
            (j.warm ? (it + 1) % 2 == 1 : (it + 1) % 4 == 0) || it == j.max_iter - 1;
        if (launch_subspace_iteration(j.C, L, m, j.inv_n, j.max_sweeps, check ? 1e-5f : 1e-3f, w,
                                      st) != cudaSuccess)
          return INSTANT_ERR_CUDA;
        if (!check) continue;
        if (launch_subspace_check(L, m, j.prm.eps, j.prm.p, j.prm.r_override, j.tol, j.inv_n2, w,
                                  st) != cudaSuccess)
          return INSTANT_ERR_CUDA;
        if (cudaMemcpyAsync(&res, w.res, sizeof(res), cudaMemcpyDeviceToHost, st) != cudaSuccess ||
            cudaStreamSynchronize(st) != cudaSuccess)
          return INSTANT_ERR_CUDA;
        if (res.converged) {
          converged = true;
          break;
        }
        if (res.block_short && it >= 15 && m < 128) {
          grow = true;
          break;
        }
      }
      if (grow) {
        m = std::min(128, 2 * m);
        continue;
      }
      break;
    }
    if (!converged) status = INSTANT_ERR_NOT_CONVERGED;
  }
  if (launch_solver_finalize(L, m, j.prm.eps, j.prm.p, j.prm.r_override, j.prm.scale_on ? 1 : 0,
                             j.rows_out, j.r_cap, j.out_bf16, j.inv_n2, w, st) != cudaSuccess)
    return INSTANT_ERR_CUDA;
  if (cudaMemcpyAsync(&res, w.res, sizeof(res), cudaMemcpyDeviceToHost, st) != cudaSuccess ||
      cudaStreamSynchronize(st) != cudaSuccess)
    return INSTANT_ERR_CUDA;
  if (res.jacobi_failed) status = INSTANT_ERR_NOT_CONVERGED;
  if (L > 128 && res.R > j.r_cap) status = INSTANT_ERR_SHAPE;
  o->k = res.k;
  o->R = res.R < j.r_cap ? res.R : j.r_cap;
  o->scale = res.scale;
  o->energy = E;
  if (eig_out)
    for (int i = 0; i < j.r_cap; ++i) eig_out[i] = i < m ? res.theta[i] : 0.0;
  if (L <= 128 && res.R > j.r_cap && status == INSTANT_OK) status = INSTANT_ERR_SHAPE;
  return status;
}

}  // namespace

extern "C" {

const char* instant_status_string(instant_status s) {
  switch (s) {
    case INSTANT_OK: return "ok";
    case INSTANT_ERR_ARG: return "invalid argument";
    case INSTANT_ERR_SHAPE: return "unsupported or inconsistent shape";
    case INSTANT_ERR_DTYPE: return "unsupported dtype";
    case INSTANT_ERR_ALIGN: return "misaligned pointer or row pitch";
    case INSTANT_ERR_WORKSPACE: return "workspace missing or too small";
    case INSTANT_ERR_CUDA: return "CUDA error";
    case INSTANT_ERR_NOT_CONVERGED: return "eigensolver did not converge";
    case INSTANT_ERR_NONFINITE: return "autocorrelation energy not finite and positive";
    case INSTANT_ERR_DEVICE: return "a device-side wait ran out of time";
  }
  return "unknown status";
}

int instant_version(void) { return 100; }

unsigned long long instant_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

instant_status instant_compress_act(const void* x, const void* P, void* xhat, int B, int L, int Cx,
                                    int Rx, instant_dtype dt, void* stream) {
  if (!dtype_ok(dt)) return INSTANT_ERR_DTYPE;
  if (!x || !P || !xhat) return INSTANT_ERR_ARG;
  if (B < 1 || L < 1 || Cx < 1 || Rx < 1 || Rx > 64) return INSTANT_ERR_SHAPE;
  if (dt == INSTANT_BF16 && (!aligned16(x) || !aligned16(xhat) || Cx % 8 != 0))
    return INSTANT_ERR_ALIGN;
  return project(x, P, xhat, nullptr, B, L, Cx, Rx, 0, dt, static_cast<cudaStream_t>(stream));
}

instant_status instant_project_grad(const void* gy, const void* PQ, void* Sx, void* Sq, int B,
                                    int L, int Cy, int Rx, int Ry, instant_dtype dt, void* stream) {
  if (!dtype_ok(dt)) return INSTANT_ERR_DTYPE;
  if (!gy || !PQ || !Sx || !Sq) return INSTANT_ERR_ARG;
  if (B < 1 || L < 1 || Cy < 1 || Rx < 1 || Ry < 1 || Rx + Ry > 128) return INSTANT_ERR_SHAPE;
  if (dt == INSTANT_BF16 && (!aligned16(gy) || !aligned16(Sx) || !aligned16(Sq) || Cy % 8 != 0))
    return INSTANT_ERR_ALIGN;
  return project(gy, PQ, Sx, Sq, B, L, Cy, Rx, Ry, dt, static_cast<cudaStream_t>(stream));
}

instant_status instant_grad_w(const void* Sx, const void* xhat, float* gw, int accumulate, int B,
                              int Rx, int Cx, int Cy, instant_dtype dt, void* stream) {
  if (!dtype_ok(dt)) return INSTANT_ERR_DTYPE;
  if (!Sx || !xhat || !gw) return INSTANT_ERR_ARG;
  if (B < 1 || Rx < 1 || Cx < 1 || Cy < 1) return INSTANT_ERR_SHAPE;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  GemmArgs g{};
  g.M = Cy;
  g.N = Cx;
  g.K = B * Rx;
  g.a_mn_major = 1;
  g.b_mn_major = 1;
  g.accumulate = accumulate ? 1 : 0;
  g.out_bf16 = 0;
  g.out = gw;
  if (dt == INSTANT_F32) {
    g.BN = 128;
    g.nk = cdiv(g.K, 64);
    g.splits = 1;
    g.chunks_per_split = g.nk;
    g.stages = 1;
    return from_cuda(launch_gemm_f32(g, static_cast<const float*>(Sx),
                                     static_cast<const float*>(xhat), st));
  }
  if (!aligned16(Sx) || !aligned16(xhat) || !aligned16(gw) || Cx % 8 != 0 || Cy % 8 != 0)
    return INSTANT_ERR_ALIGN;
  CUtensorMap ma, mb;
  const uint64_t da[2] = {static_cast<uint64_t>(Cy), static_cast<uint64_t>(g.K)};
  const uint64_t sa[1] = {static_cast<uint64_t>(Cy) * 2};
  const uint32_t ba[2] = {64, 64};
  const uint64_t db[2] = {static_cast<uint64_t>(Cx), static_cast<uint64_t>(g.K)};
  const uint64_t sb[1] = {static_cast<uint64_t>(Cx) * 2};
  const uint32_t bb[2] = {64, 64};
  if (!make_map(&ma, Sx, 2, da, sa, ba) || !make_map(&mb, xhat, 2, db, sb, bb))
    return INSTANT_ERR_CUDA;
  if (use_gradw_stream(g.M, g.N, g.K)) {
    // short contraction, large output: the persistent write-streaming kernel
    GradWStreamArgs a;
    a.M = g.M;
    a.N = g.N;
    a.K = g.K;
    a.nkc = cdiv(g.K, 64);
    a.mt = cdiv(g.M, 128);
    a.nt = cdiv(g.N, 64);
    a.stages = a.nkc == 1 ? kGradWStages : 3;
    a.accumulate = g.accumulate;
    CUtensorMap mo;
    const uint64_t dout[2] = {static_cast<uint64_t>(Cx), static_cast<uint64_t>(Cy)};
    const uint64_t sout[1] = {static_cast<uint64_t>(Cx) * 4};
    const uint32_t bout[2] = {32, 128};
    if (!make_map(&mo, gw, 2, dout, sout, bout, CU_TENSOR_MAP_DATA_TYPE_FLOAT32))
      return INSTANT_ERR_CUDA;
    const long long tiles = static_cast<long long>(a.mt) * a.nt;
    const int ctas = static_cast<int>(std::min<long long>(tiles, sm_count()));
    return from_cuda(launch_gradw_stream(ma, mb, mo, a, ctas, st));
  }
  const GemmPlan p = plan_gemm(g.M, g.N, g.K, false);
  g.BN = p.BN;
  g.nk = p.nk;
  g.splits = p.splits;
  g.chunks_per_split = p.cps;
  g.stages = p.stages;
  g.short_a = 0;
  return from_cuda(launch_gemm_bf16(ma, mb, g, st));
}

size_t instant_forward_workspace_bytes(int B, int L, int Cx, int Rx, instant_dtype dt) {
  (void)L;
  if (B < 1 || Cx < 1 || Rx < 0 || !dtype_ok(dt)) return 0;
  if (dt == INSTANT_F32 || Rx == 0) return 16;
  // fp32 x_hat accumulation [B, Rx, Cx], then one counter per sample
  return ((static_cast<size_t>(B) * Rx * Cx * 4 + 255) & ~static_cast<size_t>(255)) +
         ((static_cast<size_t>(B) * 4 + 255) & ~static_cast<size_t>(255));
}

instant_status instant_forward(const void* x, const void* w, const void* P, void* y, void* xhat,
                               void* ws, size_t ws_bytes, int B, int L, int Cx, int Cy, int Rx,
                               instant_dtype dt, void* stream) {
  if (!dtype_ok(dt)) return INSTANT_ERR_DTYPE;
  if (!x || !w || !y || (Rx > 0 && (!P || !xhat))) return INSTANT_ERR_ARG;
  if (B < 1 || L < 1 || Cx < 1 || Cy < 1 || Rx < 0 || Rx > 64) return INSTANT_ERR_SHAPE;
  if (Rx > 0 && (!ws || ws_bytes < instant_forward_workspace_bytes(B, L, Cx, Rx, dt)))
    return INSTANT_ERR_WORKSPACE;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const long long M = static_cast<long long>(B) * L;
  if (M > 0x7fffffffll) return INSTANT_ERR_SHAPE;
  if (dt == INSTANT_F32) {
    if (launch_forward_f32(static_cast<const float*>(x), static_cast<const float*>(w),
                           static_cast<float*>(y), static_cast<int>(M), Cy, Cx, st) != cudaSuccess)
      return INSTANT_ERR_CUDA;
    return Rx > 0 ? project(x, P, xhat, nullptr, B, L, Cx, Rx, 0, dt, st) : INSTANT_OK;
  }
  if (!aligned16(x) || !aligned16(w) || !aligned16(y) || Cx % 8 != 0 || Cy % 8 != 0 ||
      (Rx > 0 && (!aligned16(xhat) || !aligned16(ws))))
    return INSTANT_ERR_ALIGN;
  // x_hat from the GEMM's own x tiles when a 128-token tile never straddles
  // two samples, the channels come in pairs of 64-channel chunks and the rows
  // fit the small accumulator; otherwise the forward GEMM and then the
  // projection kernel
  const bool side = Rx > 0 && L % 128 == 0 && Cx % 128 == 0 && Rx <= 32 && aligned16(P) &&
                    !std::getenv("INSTANT_NO_FUSED_FORWARD");
  ForwardArgs a;
  a.M = static_cast<int>(M);
  a.N = Cy;
  a.K = Cx;
  a.mt = cdiv(a.M, 128);
  a.nt = cdiv(Cy, kForwardBN);
  a.nkc = cdiv(Cx, 64);
  a.group = 16;
  a.Rx = side ? Rx : 0;
  a.L = L;
  a.xh32 = side ? static_cast<float*>(ws) : nullptr;
  a.xh = side ? xhat : nullptr;
  a.cnt = side ? reinterpret_cast<unsigned int*>(
                     static_cast<uint8_t*>(ws) +
                     ((static_cast<size_t>(B) * Rx * Cx * 4 + 255) & ~static_cast<size_t>(255)))
               : nullptr;
  CUtensorMap mx, mw, my, mp;
  std::memset(&mp, 0, sizeof(mp));
  const uint64_t dx[2] = {static_cast<uint64_t>(Cx), static_cast<uint64_t>(M)};
  const uint64_t sx[1] = {static_cast<uint64_t>(Cx) * 2};
  const uint32_t bx[2] = {64, 128};
  const uint64_t dw[2] = {static_cast<uint64_t>(Cx), static_cast<uint64_t>(Cy)};
  const uint64_t sw[1] = {static_cast<uint64_t>(Cx) * 2};
  const uint32_t bw[2] = {64, static_cast<uint32_t>(kForwardBN)};
  const uint64_t dy[2] = {static_cast<uint64_t>(Cy), static_cast<uint64_t>(M)};
  const uint64_t sy[1] = {static_cast<uint64_t>(Cy) * 2};
  const uint32_t by[2] = {64, 128};
  if (!make_map(&mx, x, 2, dx, sx, bx) || !make_map(&mw, w, 2, dw, sw, bw) ||
      !make_map(&my, y, 2, dy, sy, by))
    return INSTANT_ERR_CUDA;
  if (side) {
    const uint64_t dp[2] = {static_cast<uint64_t>(L), static_cast<uint64_t>(Rx)};
    const uint64_t sp[1] = {static_cast<uint64_t>(L) * 2};
    const uint32_t bp[2] = {64, static_cast<uint32_t>(Rx)};
    if (!make_map(&mp, P, 2, dp, sp, bp)) return INSTANT_ERR_CUDA;
  }
  const long long tiles = static_cast<long long>(a.mt) * a.nt;
  const int ctas = static_cast<int>(std::min<long long>(tiles, sm_count()));
  if (launch_forward_bf16(mx, mw, my, mp, a, ctas, st) != cudaSuccess) return INSTANT_ERR_CUDA;
  if (Rx > 0 && !side) return project(x, P, xhat, nullptr, B, L, Cx, Rx, 0, dt, st);
  return INSTANT_OK;
}

size_t instant_grad_x_workspace_bytes(int B, int L, int Cx, int Cy, int Ry, instant_dtype dt) {
  (void)L;
  if (B < 1 || Cx < 1 || Cy < 1 || Ry < 1 || !dtype_ok(dt)) return 0;
  return grad_x_ws(B, Cx, Cy, Ry, dt);
}

}  // extern "C"

namespace {

// The two halves of the two-kernel input gradient, each split into a plan
// (every argument checked, every tensor map encoded) and its launch, so that
// a caller running both can report any error before either launches.
struct CorePlan {
  GemmArgs g{};
  CUtensorMap ma, mb;
  const void* Sq;
  const void* w;
};

instant_status plan_grad_x_core(const void* Sq, const void* w, void* ws, size_t ws_bytes, int B,
                                int Cx, int Cy, int Ry, instant_dtype dt, CorePlan* pl) {
  if (!dtype_ok(dt)) return INSTANT_ERR_DTYPE;
  if (!Sq || !w) return INSTANT_ERR_ARG;
  if (B < 1 || Cx < 1 || Cy < 1 || Ry < 1 || Ry > 64) return INSTANT_ERR_SHAPE;
  if (!ws || ws_bytes < grad_x_ws(B, Cx, Cy, Ry, dt)) return INSTANT_ERR_WORKSPACE;
  GemmArgs& g = pl->g;
  pl->Sq = Sq;
  pl->w = w;
  g.M = B * Ry;
  g.N = Cx;
  g.K = Cy;
  g.a_mn_major = 0;
  g.b_mn_major = 1;
  g.accumulate = 0;
  g.out = ws;
  if (dt == INSTANT_F32) {
    g.out_bf16 = 0;
    g.BN = 128;
    g.nk = cdiv(g.K, 64);
    g.splits = 1;
    g.chunks_per_split = g.nk;
    g.stages = 1;
    return INSTANT_OK;
  }
  if (!aligned16(Sq) || !aligned16(w) || !aligned16(ws) || Cx % 8 != 0 || Cy % 8 != 0)
    return INSTANT_ERR_ALIGN;
  const GemmPlan p = plan_gemm(g.M, g.N, g.K, true);
  g.out_bf16 = 1;
  g.BN = p.BN;
  g.nk = p.nk;
  g.splits = p.splits;
  g.chunks_per_split = p.cps;
  g.stages = p.stages;
  g.short_a = p.short_a;
  const uint64_t da[2] = {static_cast<uint64_t>(Cy), static_cast<uint64_t>(g.M)};
  const uint64_t sa[1] = {static_cast<uint64_t>(Cy) * 2};
  const uint32_t ba[2] = {64, static_cast<uint32_t>(p.short_a ? 64 : 128)};
  const uint64_t db[2] = {static_cast<uint64_t>(Cx), static_cast<uint64_t>(Cy)};
  const uint64_t sb[1] = {static_cast<uint64_t>(Cx) * 2};
  const uint32_t bb[2] = {64, 64};
  if (!make_map(&pl->ma, Sq, 2, da, sa, ba) || !make_map(&pl->mb, w, 2, db, sb, bb))
    return INSTANT_ERR_CUDA;
  return INSTANT_OK;
}

instant_status run_grad_x_core(const CorePlan& pl, cudaStream_t st) {
  if (!pl.g.out_bf16)
    return from_cuda(launch_gemm_f32(pl.g, static_cast<const float*>(pl.Sq),
                                     static_cast<const float*>(pl.w), st));
  return from_cuda(launch_gemm_bf16(pl.ma, pl.mb, pl.g, st));
}

struct ExpandPlan {
  ExpandArgs e;
  bool f32;
  CUtensorMap mq, mg, mo;
};

instant_status plan_expand(const void* Q, void* gx, const void* ws, size_t ws_bytes, int B, int L,
                           int Cx, int Cy, int Ry, instant_dtype dt, ExpandPlan* pl) {
  if (!dtype_ok(dt)) return INSTANT_ERR_DTYPE;
  if (!Q || !gx) return INSTANT_ERR_ARG;
  if (B < 1 || L < 1 || Cx < 1 || Cy < 1 || Ry < 1 || Ry > 64) return INSTANT_ERR_SHAPE;
  if (!ws || ws_bytes < grad_x_ws(B, Cx, Cy, Ry, dt)) return INSTANT_ERR_WORKSPACE;
  ExpandArgs& e = pl->e;
  e.B = B;
  e.L = L;
  e.Cx = Cx;
  e.Ry = Ry;
  e.KR = round_up(Ry, 16);
  e.nlt = cdiv(L, 128);
  e.gxh = ws;
  e.Q = Q;
  e.out = gx;
  e.q_tma = 0;
  e.BN = 128;
  e.qres = 0;
  e.nb = 1;
  e.total = 0;
  e.ctas = 0;
  pl->f32 = dt == INSTANT_F32;
  if (pl->f32) return INSTANT_OK;
  if (!aligned16(gx) || !aligned16(ws) || Cx % 8 != 0) return INSTANT_ERR_ALIGN;
  // 64-column strips: two CTAs share an SM (128 columns hold one)
  e.BN = 64;
  if (const char* v = std::getenv("INSTANT_EXPAND_BN")) {
    const int f = std::atoi(v);
    if (f == 64 || f == 128) e.BN = f;
  }
  e.q_tma = (L % 8 == 0 && aligned16(Q)) ? 1 : 0;
  // Q^T resident for short token axes, a ring of four g_hat_x blocks: each
  // only while the shared memory still fits
  constexpr size_t kSmemMax = 227 * 1024;
  e.qres = e.nlt <= kExpandMaxQRes ? 1 : 0;
  e.nb = kExpandMaxBRing;
  if (expand_bf16_smem_bytes(e) > kSmemMax) e.nb = 2;
  if (expand_bf16_smem_bytes(e) > kSmemMax) e.qres = 0;
  if (expand_bf16_smem_bytes(e) > kSmemMax) return INSTANT_ERR_SHAPE;
  const long long total = static_cast<long long>(cdiv(Cx, e.BN)) * B * e.nlt;
  if (total > (1ll << 30)) return INSTANT_ERR_SHAPE;
  e.total = static_cast<int>(total);
  // one wave.  When the (strip, sample) groups fill at least half of the
  // resident slots, one CTA per group walks the group's token tiles: the CTAs
  // then write the same token rows of every strip together (on the
  // long-sequence layer 12.8 us against 13.3 us with equal runs).  Otherwise as
  // many CTAs as fit take equal runs of jobs (groups are split where runs
  // meet).  INSTANT_EXPAND_CTAS=n forces the grid size.
  const int per_sm = expand_bf16_ctas_per_sm(e);
  if (per_sm < 1) return INSTANT_ERR_CUDA;
  const long long slots = static_cast<long long>(per_sm) * sm_count();
  const long long groups = total / e.nlt;
  e.ctas = static_cast<int>((groups <= slots && 2 * groups >= slots) ? groups : std::min(total, slots));
  if (const char* v = std::getenv("INSTANT_EXPAND_CTAS")) {
    const int f = std::atoi(v);
    if (f >= 1) e.ctas = static_cast<int>(std::min<long long>(f, total));
  }
  std::memset(&pl->mq, 0, sizeof(pl->mq));
  if (e.q_tma) {
    const uint64_t d2[2] = {static_cast<uint64_t>(L), static_cast<uint64_t>(Ry)};
    const uint64_t s2[1] = {static_cast<uint64_t>(L) * 2};
    const uint32_t b2[2] = {64, static_cast<uint32_t>(e.KR)};
    if (!make_map(&pl->mq, Q, 2, d2, s2, b2)) return INSTANT_ERR_CUDA;
  }
  const uint64_t dg[3] = {static_cast<uint64_t>(Cx), static_cast<uint64_t>(Ry), static_cast<uint64_t>(B)};
  const uint64_t sg[2] = {static_cast<uint64_t>(Cx) * 2, static_cast<uint64_t>(Ry) * Cx * 2};
  const uint32_t bg[3] = {64, static_cast<uint32_t>(e.KR), 1};
  const uint64_t dout[3] = {static_cast<uint64_t>(Cx), static_cast<uint64_t>(L), static_cast<uint64_t>(B)};
  const uint64_t sout[2] = {static_cast<uint64_t>(Cx) * 2, static_cast<uint64_t>(L) * Cx * 2};
  const uint32_t bout[3] = {64, 128, 1};
  if (!make_map(&pl->mg, ws, 3, dg, sg, bg) || !make_map(&pl->mo, gx, 3, dout, sout, bout))
    return INSTANT_ERR_CUDA;
  return INSTANT_OK;
}

instant_status run_expand(const ExpandPlan& pl, cudaStream_t st) {
  if (pl.f32) return from_cuda(launch_expand_f32(pl.e, st));
  return from_cuda(launch_expand_bf16(pl.mq, pl.mg, pl.mo, pl.e, st));
}

}  // namespace

instant_status instant::grad_x_two_kernels(const void* Sq, const void* w, const void* Q, void* gx,
                                           void* ws, size_t ws_bytes, int B, int L, int Cx,
                                           int Cy, int Ry, instant_dtype dt, cudaStream_t st) {
  CorePlan cp;
  ExpandPlan ep;
  instant_status s = plan_grad_x_core(Sq, w, ws, ws_bytes, B, Cx, Cy, Ry, dt, &cp);
  if (s != INSTANT_OK) return s;
  s = plan_expand(Q, gx, ws, ws_bytes, B, L, Cx, Cy, Ry, dt, &ep);
  if (s != INSTANT_OK) return s;
  s = run_grad_x_core(cp, st);
  if (s != INSTANT_OK) return s;
  return run_expand(ep, st);
}

extern "C" {

instant_status instant_grad_x_core(const void* Sq, const void* w, void* ws, size_t ws_bytes, int B,
                                   int Cx, int Cy, int Ry, instant_dtype dt, void* stream) {
  CorePlan cp;
  const instant_status s = plan_grad_x_core(Sq, w, ws, ws_bytes, B, Cx, Cy, Ry, dt, &cp);
  return s != INSTANT_OK ? s : run_grad_x_core(cp, static_cast<cudaStream_t>(stream));
}

instant_status instant_expand(const void* Q, void* gx, const void* ws, size_t ws_bytes, int B, int L,
                              int Cx, int Cy, int Ry, instant_dtype dt, void* stream) {
  ExpandPlan ep;
  const instant_status s = plan_expand(Q, gx, ws, ws_bytes, B, L, Cx, Cy, Ry, dt, &ep);
  return s != INSTANT_OK ? s : run_expand(ep, static_cast<cudaStream_t>(stream));
}

instant_status instant_grad_x(const void* Sq, const void* w, const void* Q, void* gx, void* ws,
                              size_t ws_bytes, int B, int L, int Cx, int Cy, int Ry,
                              instant_dtype dt, void* stream) {
  if (!dtype_ok(dt)) return INSTANT_ERR_DTYPE;
  if (!Sq || !w || !Q || !gx) return INSTANT_ERR_ARG;
  if (B < 1 || L < 1 || Cx < 1 || Cy < 1 || Ry < 1 || Ry > 64) return INSTANT_ERR_SHAPE;
  if (!ws || ws_bytes < grad_x_ws(B, Cx, Cy, Ry, dt)) return INSTANT_ERR_WORKSPACE;
  if (dt == INSTANT_BF16 && (!aligned16(Sq) || !aligned16(w) || !aligned16(gx) || !aligned16(ws) ||
                             Cx % 8 != 0 || Cy % 8 != 0))
    return INSTANT_ERR_ALIGN;
  if (use_fused_grad_x(B, L, Cx, Cy, Ry, dt))
    return grad_x_fused(Sq, w, Q, gx, B, L, Cx, Cy, Ry, GradWPart{nullptr, nullptr, nullptr, 0, 0},
                        static_cast<cudaStream_t>(stream));
  return grad_x_two_kernels(Sq, w, Q, gx, ws, ws_bytes, B, L, Cx, Cy, Ry, dt,
                            static_cast<cudaStream_t>(stream));
}

instant_status instant_grad_w_x(const void* Sx, const void* xhat, float* gw, int accumulate,
                                const void* Sq, const void* w, const void* Q, void* gx, void* ws,
                                size_t ws_bytes, int B, int L, int Cx, int Cy, int Rx, int Ry,
                                instant_dtype dt, void* stream) {
  if (!dtype_ok(dt)) return INSTANT_ERR_DTYPE;
  if (!Sx || !xhat || !gw || !Sq || !w || !Q || !gx) return INSTANT_ERR_ARG;
  if (B < 1 || L < 1 || Cx < 1 || Cy < 1 || Rx < 1 || Ry < 1 || Ry > 64) return INSTANT_ERR_SHAPE;
  if (!ws || ws_bytes < grad_x_ws(B, Cx, Cy, Ry, dt)) return INSTANT_ERR_WORKSPACE;
  if (dt == INSTANT_BF16 &&
      (!aligned16(Sx) || !aligned16(xhat) || !aligned16(gw) || !aligned16(Sq) || !aligned16(w) ||
       !aligned16(gx) || !aligned16(ws) || Cx % 8 != 0 || Cy % 8 != 0))
    return INSTANT_ERR_ALIGN;
  if (use_fused_grad_x(B, L, Cx, Cy, Ry, dt))
    return grad_x_fused(Sq, w, Q, gx, B, L, Cx, Cy, Ry, GradWPart{Sx, xhat, gw, accumulate, Rx},
                        static_cast<cudaStream_t>(stream));
  // g_tilde_x first, g_w last: g_w depends on neither of g_tilde_x's two
  // launches, and in this order a step of a 4096 -> 11008 layer (with the two
  // projections before it) measured 124.5 us against 129.3 us with g_w first
  const instant_status s = instant_grad_x(Sq, w, Q, gx, ws, ws_bytes, B, L, Cx, Cy, Ry, dt, stream);
  if (s != INSTANT_OK) return s;
  return instant_grad_w(Sx, xhat, gw, accumulate, B, Rx, Cx, Cy, dt, stream);
}

size_t instant_backward_workspace_bytes(int B, int L, int Cx, int Cy, int Ry, instant_dtype dt) {
  (void)L;
  if (B < 1 || Cx < 1 || Cy < 1 || Ry < 1 || !dtype_ok(dt)) return 0;
  return backward_sync_bytes(B) + grad_x_ws(B, Cx, Cy, Ry, dt);
}

instant_status instant_backward(const void* gy, const void* PQ, const void* xhat, const void* w,
                                void* Sx, void* Sq, float* gw, int accumulate, void* gx, void* ws,
                                size_t ws_bytes, int B, int L, int Cx, int Cy, int Rx, int Ry,
                                instant_dtype dt, void* stream) {
  if (!dtype_ok(dt)) return INSTANT_ERR_DTYPE;
  if (!gy || !PQ || !xhat || !w || !Sx || !Sq || !gw || !gx) return INSTANT_ERR_ARG;
  if (B < 1 || L < 1 || Cx < 1 || Cy < 1 || Rx < 1 || Ry < 1 || Ry > 64 || Rx + Ry > 128)
    return INSTANT_ERR_SHAPE;
  if (!ws || ws_bytes < instant_backward_workspace_bytes(B, L, Cx, Cy, Ry, dt))
    return INSTANT_ERR_WORKSPACE;
  if (!aligned16(ws)) return INSTANT_ERR_ALIGN;
  if (dt == INSTANT_BF16 &&
      (!aligned16(gy) || !aligned16(xhat) || !aligned16(w) || !aligned16(Sx) || !aligned16(Sq) ||
       !aligned16(gw) || !aligned16(gx) || Cx % 8 != 0 || Cy % 8 != 0))
    return INSTANT_ERR_ALIGN;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const size_t elt = dt == INSTANT_BF16 ? 2 : 4;
  const void* Q = static_cast<const uint8_t*>(PQ) + static_cast<size_t>(Rx) * L * elt;
  const size_t sync_bytes = backward_sync_bytes(B);
  void* ws_gx = static_cast<uint8_t*>(ws) + sync_bytes;
  // one launch on request: correct, but measured slower than the two launches
  // below on a BERT-base block (23.9 against 18.9 us: the projection tiles
  // finish late and the input-gradient items still take ~9 us after their signal)
  if (use_fused_grad_x(B, L, Cx, Cy, Ry, dt) && std::getenv("INSTANT_ONE_LAUNCH_BACKWARD")) {
    const ProjPart pp{gy, PQ, Sx, Rx, static_cast<unsigned int*>(ws)};
    bool no_room = false;
    const instant_status s = grad_x_fused(Sq, w, Q, gx, B, L, Cx, Cy, Ry,
                                          GradWPart{Sx, xhat, gw, accumulate, Rx}, st, &pp, &no_room);
    if (!no_room) return s;
  }
  // two launches: the projection, then the weight and input gradients
  const instant_status s = project(gy, PQ, Sx, Sq, B, L, Cy, Rx, Ry, dt, st);
  if (s != INSTANT_OK) return s;
  return instant_grad_w_x(Sx, xhat, gw, accumulate, Sq, w, Q, gx, ws_gx, ws_bytes - sync_bytes, B, L,
                          Cx, Cy, Rx, Ry, dt, stream);
}

instant_status instant_calib_accumulate(const void* t, float* C, int B, int L, int Cdim,
                                        instant_dtype dt, void* stream) {
  const instant_accumulate_item item{t, C, B, Cdim};
  return instant_calib_accumulate_batch(&item, 1, L, dt, stream);
}

instant_status instant_calib_accumulate_batch(const instant_accumulate_item* items, int count, int L,
                                              instant_dtype dt, void* stream) {
  if (!dtype_ok(dt)) return INSTANT_ERR_DTYPE;
  if (!items || count < 1) return INSTANT_ERR_ARG;
  if (L < 1 || L > 8192) return INSTANT_ERR_SHAPE;
  for (int i = 0; i < count; ++i) {
    const instant_accumulate_item& it = items[i];
    if (!it.t || !it.C) return INSTANT_ERR_ARG;
    if (it.B < 1 || it.Cdim < 1) return INSTANT_ERR_SHAPE;
    if (dt == INSTANT_BF16 && (!aligned16(it.t) || !aligned16(it.C) || it.Cdim % 8 != 0))
      return INSTANT_ERR_ALIGN;
  }
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int nblk = cdiv(L, 128);
  const int ntiles = nblk * (nblk + 1) / 2;
  if (dt == INSTANT_F32) {
    for (int i = 0; i < count; ++i) {
      SyrkArgs s;
      s.B = items[i].B;
      s.L = L;
      s.C = items[i].Cdim;
      s.nblk = nblk;
      s.ntiles = ntiles;
      s.nkc = cdiv(s.C, 64);
      s.Cout = items[i].C;
      s.splits = s.cs = s.bs = 1;
      if (launch_syrk_f32(s, static_cast<const float*>(items[i].t), st) != cudaSuccess)
        return INSTANT_ERR_CUDA;
    }
    return INSTANT_OK;
  }
  // groups of up to kMaxSyrkBatch statistics per launch
  for (int g0 = 0; g0 < count; g0 += kMaxSyrkBatch) {
    const int n = std::min(kMaxSyrkBatch, count - g0);
    SyrkBatch b;
    CUtensorMap maps[kMaxSyrkBatch];
    b.count = n;
    b.split0[0] = 0;
    // 128 x 256 tiles, one CTA per SM, from 8 row blocks (L > 896) on
    // (INSTANT_SYRK_NARROW: 128 x 128, two per SM).  With fewer blocks the
    // pairs that run past the last block waste more (1/6 of the work at 4
    // blocks): the FFN's L = 512 statistics measured 174 us wide against 150
    // us narrow, the long-sequence L = 2048 ones 2.59 ms against 3.05 ms.
    // INSTANT_SYRK_WIDE forces wide tiles for any L above 128.
    b.wide = (nblk >= 8 && !std::getenv("INSTANT_SYRK_NARROW")) ? 1 : 0;
    if (nblk >= 2 && std::getenv("INSTANT_SYRK_WIDE")) b.wide = 1;
    int ntiles_b = ntiles;
    if (b.wide) {
      ntiles_b = 0;
      for (int i = 0; i < nblk; ++i) ntiles_b += (nblk - i + 1) / 2;
    }
    int Bs[kMaxSyrkBatch], nkcs[kMaxSyrkBatch], cs[kMaxSyrkBatch], bs[kMaxSyrkBatch];
    for (int i = 0; i < n; ++i) {
      Bs[i] = items[g0 + i].B;
      nkcs[i] = cdiv(items[g0 + i].Cdim, 64);
    }
    plan_syrk(n, Bs, nkcs, ntiles_b, b.wide ? 1 : 2, cs, bs);
    for (int i = 0; i < n; ++i) {
      const instant_accumulate_item& it = items[g0 + i];
      SyrkArgs& s = b.s[i];
      s.B = it.B;
      s.L = L;
      s.C = it.Cdim;
      s.nblk = nblk;
      s.ntiles = ntiles_b;
      s.nkc = nkcs[i];
      s.Cout = it.C;
      s.cs = cs[i];
      s.bs = bs[i];
      s.splits = s.cs * s.bs;
      b.split0[i + 1] = b.split0[i] + s.splits;
      const uint64_t d3[3] = {static_cast<uint64_t>(it.Cdim), static_cast<uint64_t>(L),
                              static_cast<uint64_t>(it.B)};
      const uint64_t s3[2] = {static_cast<uint64_t>(it.Cdim) * 2, static_cast<uint64_t>(L) * it.Cdim * 2};
      const uint32_t b3[3] = {64, 128, 1};
      if (!make_map(&maps[i], it.t, 3, d3, s3, b3)) return INSTANT_ERR_CUDA;
    }
    if (launch_syrk_bf16_batch(maps, b, st) != cudaSuccess) return INSTANT_ERR_CUDA;
  }
  return INSTANT_OK;
}

size_t instant_calib_workspace_bytes(int L, int r_cap) {
  (void)r_cap;
  if (L < 1) return 0;
  return solver_workspace_bytes(L);
}

// batch workspace: the one-launch results of all problems side by side (one
// copy to the host), then one solver workspace per problem
size_t batch_results_bytes(int count) {
  return (static_cast<size_t>(count) * sizeof(SolverResult) + 255) & ~static_cast<size_t>(255);
}

size_t instant_calib_batch_workspace_bytes(int L, int count) {
  if (L < 1 || count < 1) return 0;
  return batch_results_bytes(count) + static_cast<size_t>(count) * solve_ws_stride(L);
}

instant_status instant_calib_solve(const float* C, long long n_samples, int L,
                                   const instant_calib_params* prm, void* rows_out, int r_cap,
                                   instant_dtype dt, int* k_out, int* r_out, float* scale_out,
                                   double* energy_out, double* eig_out, void* ws, size_t ws_bytes,
                                   void* stream) {
  if (!dtype_ok(dt)) return INSTANT_ERR_DTYPE;
  if (!k_out || !r_out || !scale_out) return INSTANT_ERR_ARG;
  SolveJob j;
  const instant_status v = solve_prepare(C, n_samples, L, prm, rows_out, r_cap, dt, ws, ws_bytes, &j);
  if (v != INSTANT_OK) return v;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  SolveOut o;
  instant_status status = INSTANT_OK;
  bool done = false;
  if (solve_uses_cluster(j)) {
    if (launch_cluster_solve(cluster_args(j), st) != cudaSuccess) return INSTANT_ERR_CUDA;
    SolverResult res;
    if (cudaMemcpyAsync(&res, j.w.res, sizeof(res), cudaMemcpyDeviceToHost, st) != cudaSuccess ||
        cudaStreamSynchronize(st) != cudaSuccess)
      return INSTANT_ERR_CUDA;
    done = cluster_finish(j, res, &o, eig_out, &status);
  }
  if (!done) status = solve_multi(j, &o, eig_out, st);
  *k_out = o.k;
  *r_out = o.R;
  *scale_out = o.scale;
  if (energy_out) *energy_out = o.energy;
  return status;
}

instant_status instant_calib_solve_batch(instant_calib_problem* problems, int count, int L,
                                         instant_dtype dt, void* ws, size_t ws_bytes,
                                         void* stream) {
  if (!problems || count < 1) return INSTANT_ERR_ARG;
  if (L < 1 || L > 8192) return INSTANT_ERR_SHAPE;
  const size_t stride = solve_ws_stride(L);
  const size_t res_bytes = batch_results_bytes(count);
  instant_status v = INSTANT_OK;
  if (!ws || ws_bytes < res_bytes + static_cast<size_t>(count) * stride) v = INSTANT_ERR_WORKSPACE;
  std::vector<SolveJob> jobs(count);
  for (int i = 0; i < count && v == INSTANT_OK; ++i) {
    const instant_calib_problem& q = problems[i];
    v = solve_prepare(q.C, q.n_samples, L, &q.prm, q.rows_out, q.r_cap, dt,
                      static_cast<uint8_t*>(ws) + res_bytes + i * stride, stride, &jobs[i]);
  }
  SolverResult* res_dev = static_cast<SolverResult*>(ws);
  if (v != INSTANT_OK) {
    for (int i = 0; i < count; ++i) problems[i].status = v;
    return v;
  }
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // every problem that the one-launch solver takes: one cluster each, all in
  // as few launches as the block sizes allow, one synchronisation
  std::vector<SolverResult> res(count);
  std::vector<char> launched(count, 0);
  for (int m : {16, 32}) {
    ClusterSolveBatch batch;
    int idx[kMaxSolveBatch];
    int n = 0;
    for (int i = 0; i <= count; ++i) {
      const bool take = i < count && solve_uses_cluster(jobs[i]) && jobs[i].m_block == m;
      if (take) {
        batch.s[n] = cluster_args(jobs[i]);
        batch.s[n].res = res_dev + i;  // results side by side
        idx[n++] = i;
      }
      if (n == kMaxSolveBatch || (i == count && n > 0)) {
        if (launch_cluster_solve_batch(batch, n, st) != cudaSuccess) return INSTANT_ERR_CUDA;
        for (int u = 0; u < n; ++u) launched[idx[u]] = 1;
        n = 0;
      }
    }
  }
  // the small statistics (L <= 128): queued too, results in the same block
  std::vector<char> small(count, 0);
  std::vector<SolveJob*> sj;
  for (int i = 0; i < count; ++i) {
    if (launched[i] || jobs[i].L > 128 || std::getenv("INSTANT_SOLVER_MULTI")) continue;
    jobs[i].w.res = res_dev + i;
    sj.push_back(&jobs[i]);
    small[i] = 1;
  }
  if (!sj.empty() && solve_small_async(sj, st) != INSTANT_OK) return INSTANT_ERR_CUDA;
  bool any = false;
  for (int i = 0; i < count; ++i) any = any || launched[i] || small[i];
  if (any && cudaMemcpyAsync(res.data(), res_dev, sizeof(SolverResult) * count,
                             cudaMemcpyDeviceToHost, st) != cudaSuccess)
    return INSTANT_ERR_CUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return INSTANT_ERR_CUDA;
  instant_status first = INSTANT_OK;
  for (int i = 0; i < count; ++i) {
    instant_calib_problem& q = problems[i];
    SolveOut o;
    instant_status s1 = INSTANT_OK;
    bool done = false;
    if (small[i]) {
      small_finish(jobs[i], res[i], &o, q.eig_out, &s1);
      done = true;
    } else if (launched[i]) {
      done = cluster_finish(jobs[i], res[i], &o, q.eig_out, &s1);
    }
    if (!done) s1 = solve_multi(jobs[i], &o, q.eig_out, st);
    q.k = o.k;
    q.R = o.R;
    q.scale = o.scale;
    q.energy = o.energy;
    q.status = s1;
    if (first == INSTANT_OK) first = s1;
  }
  return first;
}

instant_status instant_reconstruction_error(const void* t, const void* Q, const void* S, int B,
                                           int L, int C, int R, instant_dtype dt,
                                           double* err2_out, double* energy_out, void* ws,
                                           size_t ws_bytes, void* stream) {
  if (!dtype_ok(dt)) return INSTANT_ERR_DTYPE;
  if (!t || !Q || !S || !err2_out || !energy_out) return INSTANT_ERR_ARG;
  if (B < 1 || L < 1 || C < 1 || R < 1 || R > 64 || static_cast<long long>(R) * L > 12288)
    return INSTANT_ERR_SHAPE;
  if (!ws || ws_bytes < 2 * sizeof(double)) return INSTANT_ERR_WORKSPACE;
  if (reinterpret_cast<uintptr_t>(ws) & 7u) return INSTANT_ERR_ALIGN;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  double* totals = static_cast<double*>(ws);
  if (launch_recon(t, Q, S, B, L, C, R, dt == INSTANT_BF16 ? 1 : 0, totals, st) != cudaSuccess)
    return INSTANT_ERR_CUDA;
  double h[2];
  if (cudaMemcpyAsync(h, totals, sizeof(h), cudaMemcpyDeviceToHost, st) != cudaSuccess ||
      cudaStreamSynchronize(st) != cudaSuccess)
    return INSTANT_ERR_CUDA;
  *err2_out = h[0];
  *energy_out = h[1];
  return INSTANT_OK;
}

instant_status instant_device_status(int clear, void* stream) {
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return INSTANT_ERR_CUDA;
  unsigned int total = 0, v = 0;
  if (read_fault_project(&v, clear) != cudaSuccess) return INSTANT_ERR_CUDA;
  total |= v;
  if (read_fault_gemm(&v, clear) != cudaSuccess) return INSTANT_ERR_CUDA;
  total |= v;
  if (read_fault_expand(&v, clear) != cudaSuccess) return INSTANT_ERR_CUDA;
  total |= v;
  if (read_fault_syrk(&v, clear) != cudaSuccess) return INSTANT_ERR_CUDA;
  total |= v;
  if (read_fault_eig(&v, clear) != cudaSuccess) return INSTANT_ERR_CUDA;
  total |= v;
  if (read_fault_fused(&v, clear) != cudaSuccess) return INSTANT_ERR_CUDA;
  total |= v;
  if (read_fault_gradw(&v, clear) != cudaSuccess) return INSTANT_ERR_CUDA;
  total |= v;
  if (read_fault_forward(&v, clear) != cudaSuccess) return INSTANT_ERR_CUDA;
  total |= v;
  return total ? INSTANT_ERR_DEVICE : INSTANT_OK;
}

}  // extern "C"
