// route_noalloc.cu -- moe_route_noalloc: the router + top-k for callers that
// cannot hand the library any workspace.
//
// moe_route needs scratch device memory (the C x E router logits and a
// completion counter) that the caller normally allocates as "workspace".  Some
// callers cannot allocate: code that runs while a stream is being captured in
// a mode that forbids cudaMalloc, plug-ins whose host framework owns every
// device buffer through its own allocator, and latency-critical loops that
// must not pay cudaMalloc's implicit device synchronisation.  This entry
// point keeps that scratch in a fixed array that lives in the library itself
// (a file-scope __device__ array, 32 KiB + 256 bytes; every GPU that loads
// the library holds it until the process exits), so such a caller passes only
// its inputs and outputs.
//
// Limits and rules of use:
//   - C * E must fit the array: C <= 8 tokens and C * E <= 8192 logits;
//     larger calls return MOE_ERR_WORKSPACE_TOO_SMALL before queuing anything.
//   - The array's device address is looked up once per device
//     (cudaGetSymbolAddress) by the first call made on that device; make that
//     first call outside any stream capture.
//   - Every call shares the one array: calls whose work overlaps on the GPU
//     (different streams, or different host threads) race on it.  Serialise
//     them on one stream.
//   - Each call clears the completion counters before its kernel, so the
//     contents a previous call left behind do not matter.
//   - No device flags reach the caller (the flag word lives in the array and
//     no entry point reads it); a call whose bounded router wait ran out
//     writes every id as -1 and every weight as 0 instead.
//   - The cached device address is invalid after cudaDeviceReset.
#include <mutex>

#include "kernels.h"
#include "moe_internal.cuh"

namespace {

constexpr int kNoAllocTokens = 8;
constexpr int kNoAllocLogits = 8192;                 // floats: C * E limit
constexpr size_t kNoAllocBytes = 256 + sizeof(float) * kNoAllocLogits;

// [0, 256): uint32 completion counter, flag word, reserved word (+ padding);
// [256, ...): logits.
static __device__ __align__(256) unsigned char g_route_scratch[kNoAllocBytes];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mutex;
void *g_scratch_ptr[kMaxDevices] = {};

// Device address of g_route_scratch on the current device (set-up on first use).
cudaError_t scratch_address(int device, unsigned char **out) {
  if (device < 0 || device >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  if (!g_scratch_ptr[device]) {
    void *p = nullptr;
    const cudaError_t err = cudaGetSymbolAddress(&p, g_route_scratch);
    if (err != cudaSuccess) return err;
    g_scratch_ptr[device] = p;
  }
  *out = static_cast<unsigned char *>(g_scratch_ptr[device]);
  return cudaSuccess;
}

bool aligned16(const void *p) { return ((uintptr_t)p & 15u) == 0; }

}  // namespace

extern "C" moe_status moe_route_noalloc(moe_layer_t L, const uint16_t *x, int C,
                                        const float *w_router, const float *bias, int32_t *ids,
                                        float *weights, cudaStream_t stream) {
  if (!L || !x || !w_router || !ids || !weights) return MOE_ERR_INVALID_ARG;
  if (C < 1 || C > L->cfg.max_tokens) return MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(w_router)) return MOE_ERR_INVALID_ARG;
  if (C > kNoAllocTokens || (long long)C * L->cfg.num_experts > kNoAllocLogits)
    return MOE_ERR_WORKSPACE_TOO_SMALL;
  int prev = -1;
  if (cudaGetDevice(&prev) != cudaSuccess) return MOE_ERR_CUDA;
  if (prev != L->device && cudaSetDevice(L->device) != cudaSuccess) return MOE_ERR_CUDA;
  unsigned char *scratch = nullptr;
  cudaError_t err = scratch_address(L->device, &scratch);
  if (err == cudaSuccess) err = cudaMemsetAsync(scratch, 0, 3 * sizeof(uint32_t), stream);
  if (err == cudaSuccess) {
    moe::RouteArgs a = {};
    a.x = x; a.w_router = w_router; a.bias = bias; a.ids = ids; a.weights = weights;
    a.logits = reinterpret_cast<float *>(scratch + 256);
    a.ticket = reinterpret_cast<uint32_t *>(scratch);
    a.flags = reinterpret_cast<int32_t *>(scratch + sizeof(uint32_t));
    a.C = C; a.E = L->cfg.num_experts; a.H = L->cfg.hidden; a.k = L->cfg.top_k;
    moe::route_wait_policy(L->cfg.flags, &a);
    const int grid = a.E < L->num_sms ? a.E : L->num_sms;
    err = moe::launch_route_fused(a, grid, stream);
  }
  if (prev != L->device) cudaSetDevice(prev);
  return err == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
