// GroupNorm (+ optional SiLU) that allocates no device memory.
//
// Some callers cannot call cudaMalloc while they run this op: plugin hosts and
// inference servers that hand a plugin only its input/output buffers and forbid
// allocation inside their enqueue callback, real-time pipelines whose memory is
// fixed at start-up, and code running under another allocator that must not see
// raw device allocations.  For them this entry point keeps its scratch (the
// per-chunk moments and the merged per-channel scale/shift) in one fixed array
// inside this library instead of the decoder handle's workspace.
//
// The array below is a device symbol: in host code its name is only a host-side
// stand-in, so the host asks the runtime for its device address once per device
// context (cudaGetSymbolAddress, with that device current) and passes that address
// to the kernels.  The address is cached under the context's unique id, so a new
// context on the same device (after cudaDeviceReset, or a caller's own driver-API
// context) gets its own look-up instead of a stale address.  Every GPU that loads
// this library holds the array until the process exits.  All calls share it: two
// calls whose kernels overlap on the GPU (for example on two streams) race on it
// and must be ordered by the caller.
#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>
#include <string>

#include "vaedec.h"
#include "kernels.h"

using namespace vd;

namespace {

// Scratch limits: B * rows * G chunk moments and B * C scale/shift pairs.
constexpr size_t kMaxPartials = 131072;          // 16 B each: 2 MiB
constexpr size_t kMaxScaleShift = 32768;         // floats each for scale and shift: 256 KiB
constexpr size_t kScratchBytes = kMaxPartials * sizeof(GnPartial) + 2 * kMaxScaleShift * sizeof(float);

static __device__ __align__(256) unsigned char g_gn_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mu;
struct ScratchAddr {
  unsigned long long ctx_id = 0;   // unique id of the context the address belongs to (0: none yet)
  void* ptr = nullptr;
};
ScratchAddr g_scratch_dev[kMaxDevices];

using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);

// Unique id of the calling thread's current context (0 when there is none or the driver
// cannot say).  The driver entry points are resolved once through the runtime.
unsigned long long current_ctx_id() {
  static CtxGetCurrentFn get_cur = nullptr;
  static CtxGetIdFn get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_cur = reinterpret_cast<CtxGetCurrentFn>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<CtxGetIdFn>(p);
  });
  if (get_cur == nullptr || get_id == nullptr) return 0;
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (get_cur(&ctx) != CUDA_SUCCESS || ctx == nullptr) return 0;
  if (get_id(ctx, &id) != CUDA_SUCCESS) return 0;
  return id;
}

vaedec_status noalloc_fail(vaedec_status s, const std::string& m) {
  record_last_error(m);
  return s;
}

}  // namespace

extern "C" vaedec_status vaedec_groupnorm_noalloc(int in_dtype, int out_dtype, const void* x, void* y, int B,
                                                  int rows, int W, int C, int G, const float* gamma,
                                                  const float* beta, float eps, int silu, void* stream) {
  if (x == nullptr || y == nullptr || gamma == nullptr || beta == nullptr)
    return noalloc_fail(VAEDEC_ERR_INVALID_ARG, "NULL pointer argument");
  if (B < 1 || rows < 1 || W < 1 || C < 1 || G < 1)
    return noalloc_fail(VAEDEC_ERR_INVALID_ARG, "sizes must be positive");
  if (C % 8 != 0 || C / 8 > 256 || C % G != 0)
    return noalloc_fail(VAEDEC_ERR_INVALID_ARG, "C must be a multiple of 8, at most 2048, and divisible by G");
  const bool types_ok = (in_dtype == VAEDEC_DTYPE_F32 && (out_dtype == VAEDEC_DTYPE_BF16 || out_dtype == VAEDEC_DTYPE_F32)) ||
                        (in_dtype == VAEDEC_DTYPE_BF16 && out_dtype == VAEDEC_DTYPE_BF16);
  if (!types_ok) return noalloc_fail(VAEDEC_ERR_INVALID_ARG, "unsupported dtype pair");
  if ((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(y)) & 15)
    return noalloc_fail(VAEDEC_ERR_INVALID_ARG, "x and y must be 16-byte aligned");
  if (!(eps > 0.f)) return noalloc_fail(VAEDEC_ERR_INVALID_ARG, "eps must be positive");
  const size_t n_part = (size_t)B * rows * G;
  if (n_part > kMaxPartials)
    return noalloc_fail(VAEDEC_ERR_INVALID_ARG, "B * rows * G = " + std::to_string(n_part) +
                                                     " exceeds the fixed scratch limit of " +
                                                     std::to_string(kMaxPartials));
  if ((size_t)B * C > kMaxScaleShift)
    return noalloc_fail(VAEDEC_ERR_INVALID_ARG, "B * C = " + std::to_string((size_t)B * C) +
                                                     " exceeds the fixed scratch limit of " +
                                                     std::to_string(kMaxScaleShift));

  // Set-up once per device context: the device address of the scratch array.
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return noalloc_fail(VAEDEC_ERR_CUDA, std::string("cudaGetDevice: ") + cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices) return noalloc_fail(VAEDEC_ERR_UNSUPPORTED, "device index out of range");
  void* base = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_setup_mu);
    ScratchAddr& a = g_scratch_dev[dev];
    const unsigned long long id = current_ctx_id();
    if (a.ptr == nullptr || id == 0 || id != a.ctx_id) {
      void* p = nullptr;
      e = cudaGetSymbolAddress(&p, g_gn_scratch);
      if (e != cudaSuccess || p == nullptr)
        return noalloc_fail(VAEDEC_ERR_CUDA, std::string("cudaGetSymbolAddress: ") + cudaGetErrorString(e));
      a.ptr = p;
      a.ctx_id = current_ctx_id();   // the look-up made the device's context current if none was
    }
    base = a.ptr;
  }
  GnPartial* part = static_cast<GnPartial*>(base);
  float* scale = reinterpret_cast<float*>(static_cast<unsigned char*>(base) + kMaxPartials * sizeof(GnPartial));
  float* shift = scale + kMaxScaleShift;

  // Every scratch word that is read is first written by this call (partials by
  // phase 1, scale/shift by phase 2), so nothing needs clearing between calls.
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int idt = in_dtype == VAEDEC_DTYPE_BF16 ? kBF16 : kF32;
  const int odt = out_dtype == VAEDEC_DTYPE_BF16 ? kBF16 : kF32;
  e = launch_gn_partials(idt, x, B, rows, W, C, G, 1, part, st);
  if (e == cudaSuccess) e = launch_gn_finalize(part, B, rows, C, G, gamma, beta, eps, scale, shift, st);
  if (e == cudaSuccess)
    e = launch_gn_apply(idt, odt, x, y, nullptr, (long long)rows * W, B, C, scale, shift, silu ? 1 : 0, st);
  if (e != cudaSuccess) return noalloc_fail(VAEDEC_ERR_CUDA, std::string("groupnorm launch: ") + cudaGetErrorString(e));
  return VAEDEC_OK;
}
