// mlora_linear_noalloc: the multi-adapter linear layer for callers that
// cannot allocate device memory.
//
// Some callers of this library have no way to obtain a device buffer for the
// workspace: a plugin running inside a host framework that owns every device
// allocation, or code that must not call cudaMalloc because an allocation
// would synchronise the device or break a memory budget fixed at start-up.
// This entry point keeps its scratch (segment plan, low-rank activations T
// and the device status word) in one array compiled into the library, so the
// caller passes only inputs and outputs.
//
// The array is a file-scope __device__ variable of NOALLOC_SCRATCH_BYTES; every
// GPU that loads the library holds it until the process exits.  Host code
// cannot use the array's name as a device address (in host code it names a
// host-side stand-in), so the first call on each device looks up the device
// address with cudaGetSymbolAddress while that device is current and keeps
// it for later calls.  Make that first call on a device before any stream
// capture begins.
//
// All calls share the array.  Nothing in it needs to start at zero: each call
// rewrites the plan and T before reading them.  The device status bits this
// variant accumulates are not reported.  Two calls whose work overlaps on the
// GPU (for example on two streams) race on the array.
#include <mutex>

#include "common.cuh"
#include "launch.h"

namespace mlora {

constexpr int NOALLOC_MAX_ROWS = 1024;
constexpr int NOALLOC_MAX_ADAPTERS = 256;
constexpr size_t NOALLOC_SCRATCH_BYTES = 512 * 1024;
constexpr int NOALLOC_MAX_DEVICES = 64;

static __device__ __align__(256) uint8_t g_noalloc_scratch[NOALLOC_SCRATCH_BYTES];

static std::mutex g_noalloc_mutex;
static void *g_noalloc_base[NOALLOC_MAX_DEVICES];

// Device address of the scratch array on the current device (set-up on the
// first call per device).
static cudaError_t noalloc_base(void **out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= NOALLOC_MAX_DEVICES) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_noalloc_mutex);
  if (!g_noalloc_base[dev]) {
    void *p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    g_noalloc_base[dev] = p;
  }
  *out = g_noalloc_base[dev];
  return cudaSuccess;
}

}  // namespace mlora

using namespace mlora;

extern "C" MLORA_API mlora_status mlora_linear_noalloc(const mlora_bf16 *x, int M, int K, const mlora_bf16 *W, int N,
                                                       const mlora_bf16 *A_stack, const mlora_bf16 *B_stack,
                                                       int n_adapters, int r_max, const int32_t *rank_of,
                                                       const int32_t *adapter_idx, float scale, int mode,
                                                       mlora_bf16 *y, mlora_stream stream) {
  if (!x || !W || !y) return MLORA_ERR_ARG;
  const int prefetch_w = (mode & MLORA_PREFETCH_WEIGHTS) ? 1 : 0;
  const int base_mode = mode & ~MLORA_PREFETCH_WEIGHTS;
  if (base_mode != MLORA_DRAFT && base_mode != MLORA_VERIFY) return MLORA_ERR_ARG;
  const bool verify = base_mode == MLORA_VERIFY;
  if (verify && (!A_stack || !B_stack || !rank_of || !adapter_idx)) return MLORA_ERR_ARG;
  if (M < 1 || N < 1 || K < 8 || (K % 8) != 0) return MLORA_ERR_SHAPE;
  // Sizes beyond the fixed scratch array are refused, never truncated.
  if (M > NOALLOC_MAX_ROWS) return MLORA_ERR_SHAPE;
  const int n_ad = verify ? n_adapters : 0;
  if (verify && (n_adapters < 1 || n_adapters > NOALLOC_MAX_ADAPTERS)) return MLORA_ERR_SHAPE;
  if (verify && (r_max < 8 || r_max > MLORA_MAX_RANK || (r_max % 8) != 0)) return MLORA_ERR_SHAPE;
  if ((reinterpret_cast<uintptr_t>(x) & 15) || (reinterpret_cast<uintptr_t>(W) & 15)) return MLORA_ERR_ARG;
  if (verify && ((reinterpret_cast<uintptr_t>(A_stack) & 15) || (reinterpret_cast<uintptr_t>(B_stack) & 15)))
    return MLORA_ERR_ARG;
  const PlanLayout P = plan_layout(M, n_ad);
  const size_t plan_off = 256;
  const size_t t_off = align_up(plan_off + P.words * 4, 256);
  if (t_off + (size_t)M * T_STRIDE * 4 > NOALLOC_SCRATCH_BYTES) return MLORA_ERR_SHAPE;

  void *base = nullptr;
  if (noalloc_base(&base) != cudaSuccess) return MLORA_ERR_CUDA;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MLORA_ERR_CUDA;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
    return MLORA_ERR_CUDA;

  cudaStream_t s = (cudaStream_t)stream;
  uint8_t *scratch = static_cast<uint8_t *>(base);
  uint32_t *status = reinterpret_cast<uint32_t *>(scratch);
  int32_t *plan = reinterpret_cast<int32_t *>(scratch + plan_off);
  float *T = reinterpret_cast<float *>(scratch + t_off);
  if (verify) {
    if (launch_plan(adapter_idx, M, rank_of, n_ad, r_max, plan, status, s) != cudaSuccess)
      return MLORA_ERR_CUDA;
    if (launch_shrink(x, M, K, A_stack, n_ad, r_max, plan, T, T_STRIDE, false, sms, nullptr, 1.f, 1, status, s) !=
        cudaSuccess)
      return MLORA_ERR_CUDA;
  }
  GemmLaunch g;
  g.x = x;
  g.W = W;
  g.M = M;
  g.N = N;
  g.K = K;
  g.n_slices = 1;
  for (int i = 0; i < MLORA_MAX_SLICES; ++i) g.slice_end[i] = N;
  g.mode = base_mode;
  g.prefetch_w = prefetch_w;
  g.after_shrink = verify ? 1 : 0;
  g.scale = scale;
  g.y = y;
  g.B_stack = B_stack;
  g.r_max = r_max;
  g.n_ad = n_ad;
  g.T = T;
  g.plan = plan;
  g.status = status;
  g.tw = nullptr;
  g.test_flag_wait_ns = 0;
  int err = 0;
  const cudaError_t e = launch_gemm(g, gemm_shape(M, N, K, sms), s, &err);
  if (err) return MLORA_ERR_ARG;
  return e == cudaSuccess ? MLORA_OK : MLORA_ERR_CUDA;
}
