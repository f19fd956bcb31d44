// fp8_quantize_absmax_noalloc: per-tensor absmax quantization for callers that
// cannot allocate device memory.
//
// The regular fp8_quantize_absmax asks its caller for a small workspace (the
// per-block absmax partials of the first pass).  Some callers have no way to
// provide one: code inside a framework that owns every device allocation
// through its own pool and hands out none to plug-ins, and latency-critical
// loops that must not call cudaMalloc/cudaFree because those synchronize the
// device and can stall every stream.
// This entry point keeps its scratch in a fixed array that lives in the
// library's own device memory, so the caller passes only the input and the
// outputs.
//
// The array is a file-scope __device__ variable: it exists once per GPU that
// loads the library and stays allocated until the process exits.  Host code
// must not use the array's name as a device address (on the host it is only a
// stand-in symbol); the device address is obtained once per device with
// cudaGetSymbolAddress, with that device current, and handed to the kernels.
#include "fp8q.h"
#include "fp8q_internal.h"

#include <mutex>

namespace {

using namespace fp8q;

// Capacity of the scratch array: one absmax partial per block of the first
// pass.  The first pass never launches more than kMaxPartials blocks, so this
// covers every tensor size.
constexpr int kNoallocPartials = kMaxPartials;  // 1024 x 4 bytes = 4 KiB

static __device__ __align__(256) uint32_t g_noalloc_partials[kNoallocPartials];
static_assert(kNoallocPartials >= kMaxPartials, "the first pass may write up to kMaxPartials partials");

struct NoallocDevice {
  uint32_t* partials = nullptr;
  unsigned* status = nullptr;
  int num_sms = 0;
};

// Looks up (and on the first call for the current device, resolves) the device
// address of the scratch array, plus the library's status word and SM count.
int noalloc_device(NoallocDevice* out) {
  static std::mutex mu;
  static NoallocDevice cache[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return FP8Q_ERR_CUDA;
  std::lock_guard<std::mutex> lock(mu);
  NoallocDevice& d = cache[dev];
  if (!d.partials) {
    void* part = nullptr;
    unsigned* st = nullptr;
    int sms = 0;
    if (cudaGetSymbolAddress(&part, g_noalloc_partials) != cudaSuccess) return FP8Q_ERR_CUDA;
    if (device_status_and_sms(&st, &sms) != 0) return FP8Q_ERR_CUDA;
    d.partials = static_cast<uint32_t*>(part);
    d.status = st;
    d.num_sms = sms;
  }
  *out = d;
  return FP8Q_OK;
}

}  // namespace

extern "C" {

int fp8_quantize_absmax_noalloc(const void* x, fp8q_dtype x_dtype, int64_t n, fp8q_fmt fmt, uint8_t* q,
                                float* scal, fp8q_stream stream) {
  if (n < 1 || !x || !q || ((uintptr_t)x & 15u) || ((uintptr_t)q & 15u) || !scal || ((uintptr_t)scal & 3u))
    return FP8Q_ERR_INVALID_ARG;
  if ((x_dtype != FP8Q_BF16 && x_dtype != FP8Q_F32) || (fmt != FP8Q_E4M3 && fmt != FP8Q_E5M2))
    return FP8Q_ERR_INVALID_ARG;
  // the first pass's own grid size (one partial per block) must fit the array
  if (absmax_partial_blocks((int)x_dtype, n) > kNoallocPartials) return FP8Q_ERR_INVALID_ARG;
  NoallocDevice d;
  int e = noalloc_device(&d);
  if (e) return e;
  Launch L;
  L.stream = static_cast<cudaStream_t>(stream);
  L.status = d.status;
  L.num_sms = d.num_sms;
  int launches = 0;
  L.launches = &launches;
  // The first pass overwrites partials [0, P) before the second pass reads
  // exactly those, so nothing left from an earlier call needs clearing.
  int P = 0;
  bool traced = trace_step_begin(L.stream, kTraceAbsmaxPartial);
  cudaError_t e1 = launch_absmax_partial(x, (int)x_dtype, n, d.partials, &P, L);
  trace_step_end(L.stream, traced);
  if (e1 != cudaSuccess) return FP8Q_ERR_CUDA;
  traced = trace_step_begin(L.stream, kTraceQuantCast);
  cudaError_t e2 = launch_quant_cast(x, (int)x_dtype, n, (int)fmt, d.partials, P, q, scal, L);
  trace_step_end(L.stream, traced);
  if (e2 != cudaSuccess) return FP8Q_ERR_CUDA;
  set_last_launch_count(launches);
  return FP8Q_OK;
}

}  // extern "C"
