// Decode entry point that allocates nothing.
//
// pa_decode needs a workspace the caller allocates once (partials, arrival
// counters, a status word). Some callers cannot call cudaMalloc at all: a
// plugin or extension running inside a host framework that owns every device
// allocation and hands out none, or a latency-critical path where cudaMalloc
// may synchronise the device and stall other streams. pa_decode_noalloc serves
// them: it runs the same dense decode kernel on a fixed scratch buffer that is
// compiled into this library as a file-scope __device__ array, so the caller
// passes only inputs, outputs and a plan.
//
// Costs and limits:
//  * every GPU that loads this library holds kNoAllocScratchBytes (32 MiB) of
//    device memory for this array until the process exits;
//  * a plan whose workspace exceeds that size is rejected with
//    PA_ERR_WORKSPACE;
//  * all calls share the one array, so calls that can overlap on the GPU (on
//    different streams, or on the same plan from several threads) race and
//    corrupt each other's partials; serialise them.
#include <mutex>

#include "pa_decode.h"
#include "pa_internal.h"

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(32) << 20;
constexpr int kMaxDevices = 64;

// Zero-initialised at module load; holds partials, counters and the status word.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_scratch_mutex;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of the scratch array on `device` (looked up once per device,
// with that device current). Host code cannot use the array's name as an
// address: it is a host-side stand-in for the symbol.
pa_status scratch_address(int device, void** out) {
  if (device < 0 || device >= kMaxDevices) return pa::set_error(PA_ERR_INVALID_ARG, "device ordinal out of range");
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  if (!g_scratch_addr[device]) {
    pa::DeviceGuard guard(device);  // restores the caller's current device on return
    cudaError_t e = guard.error();
    if (e != cudaSuccess) return pa::set_error(PA_ERR_CUDA, cudaGetErrorString(e));
    void* ptr = nullptr;
    e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
    if (e != cudaSuccess || ptr == nullptr)
      return pa::set_error(PA_ERR_CUDA, e != cudaSuccess ? cudaGetErrorString(e) : "null scratch address");
    g_scratch_addr[device] = ptr;
  }
  *out = g_scratch_addr[device];
  return PA_OK;
}

}  // namespace

extern "C" pa_status pa_decode_noalloc(void* out, const void* q, const void* k_cache, const void* v_cache,
                                       const int32_t* block_table, const int32_t* ctx_lens, const float* k_scale,
                                       const float* v_scale, int window, const float* sinks, const pa_plan_t* plan,
                                       void* stream) {
  if (!plan) return pa::set_error(PA_ERR_INVALID_ARG, "null plan");
  size_t zero_from = 0;
  int device = 0, sparse = 0;
  const size_t need = pa::plan_workspace_layout(plan, &zero_from, &device, &sparse);
  if (sparse) return pa::set_error(PA_ERR_INVALID_ARG, "pa_decode_noalloc takes dense-decode plans only");
  if (need > kNoAllocScratchBytes)
    return pa::set_error(PA_ERR_WORKSPACE,
                         "plan needs more workspace than the 32 MiB built-in scratch of pa_decode_noalloc");
  void* scratch = nullptr;
  pa_status st = scratch_address(device, &scratch);
  if (st != PA_OK) return st;
  // Counters, reducer descriptors and the status word must start at zero; the
  // previous call may have left them otherwise (e.g. after a reported timeout).
  cudaError_t e = cudaMemsetAsync(static_cast<unsigned char*>(scratch) + zero_from, 0, need - zero_from,
                                  static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return pa::set_error(PA_ERR_CUDA, cudaGetErrorString(e));
  return pa::launch_on_workspace(plan, scratch, kNoAllocScratchBytes, out, q, k_cache, v_cache, block_table, ctx_lens,
                                 k_scale, v_scale, window, sinks, stream);
}
