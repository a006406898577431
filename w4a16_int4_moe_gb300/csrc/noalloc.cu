// noalloc.cu -- the indexed GEMM for callers that cannot allocate device
// memory.
//
// Some callers have no way to obtain a scratch buffer at call time: a host
// whose caching allocator owns every byte of device memory and hands out no
// raw allocations, a runtime that forbids allocation after start-up
// (cudaMalloc and cudaFree can synchronise the whole device and take a global
// lock, which latency-critical or certified code paths must not do), or a
// plugin ABI that passes only the tensors of the operation. For them this
// file keeps the GEMM's workspace in a fixed array of device memory that is
// part of the library image: it exists on every GPU that loads the library
// and stays allocated until the process exits.

#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>

#include "internal.h"

namespace {

// Largest workspace the no-allocation entry point can provide: the status
// block plus the routed activation rows of, e.g., a gate_up call with
// capacity 2048 and k 7168 (28 MiB).
constexpr size_t kNoAllocScratchBytes = 32u << 20;

// File-scope scratch: zero at module load, shared by every call on a device.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

// Device address of the scratch array, looked up once per device (and again
// when the device's context changes, e.g. after cudaDeviceReset) with that
// device current. In host code the symbol itself is only a host-side
// stand-in and must never be passed to a kernel.
using CtxGetCurrentFn = CUresult (*)(CUcontext*);

CtxGetCurrentFn ctx_get_current() {
  static CtxGetCurrentFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<CtxGetCurrentFn>(f);
  });
  return fn;
}

void* scratch_address(int device) {
  static std::mutex mu;
  static void* cache[64] = {nullptr};
  static CUcontext cache_ctx[64] = {nullptr};
  if (device < 0 || device >= 64) return nullptr;
  CUcontext ctx = nullptr;
  const CtxGetCurrentFn get = ctx_get_current();
  if (get == nullptr || get(&ctx) != CUDA_SUCCESS) ctx = nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (cache[device] == nullptr || ctx == nullptr || cache_ctx[device] != ctx) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess) return nullptr;
    cache[device] = ptr;
    cache_ctx[device] = ctx;
  }
  return cache[device];
}

}  // namespace

void* w4a16::noalloc_scratch_address() {
  int device = 0;
  if (cudaGetDevice(&device) != cudaSuccess) return nullptr;
  return scratch_address(device);
}

extern "C" w4a16_status w4a16_moe_indexed_gemm_noalloc(
    int mode, const void* packed, int num_experts, int n, int k, const uint16_t* a, int tokens,
    int topk, const int32_t* sorted_ids, const int32_t* expert_ids,
    const int32_t* num_tokens_padded, int capacity, const float* topk_weights, void* out,
    int flags, const w4a16_plan_t* plan, void* stream) {
  if (plan == nullptr) return W4A16_ERR_INVALID_ARG;
  if ((flags & ~(W4A16_FLAG_VALIDATE_ROUTING | W4A16_FLAG_ACCUMULATE |
                 W4A16_FLAG_SYNC_STATUS)) != 0)
    return W4A16_ERR_INVALID_ARG;
  if (tokens < 0 || topk <= 0 || k <= 0 || capacity < 0) return W4A16_ERR_INVALID_ARG;
  if (w4a16_workspace_size(plan, capacity, k) > kNoAllocScratchBytes) return W4A16_ERR_WORKSPACE;
  // every other check, then the scratch address, the status clear and the
  // launches, in that order
  const w4a16_status st = w4a16::indexed_gemm(
      mode, packed, num_experts, n, k, a, tokens, topk, sorted_ids, expert_ids,
      num_tokens_padded, capacity, topk_weights, out, flags & ~W4A16_FLAG_SYNC_STATUS, plan,
      nullptr, kNoAllocScratchBytes, stream, true);
  if (st != W4A16_OK) return st;
  if (flags & W4A16_FLAG_SYNC_STATUS)
    return w4a16_read_device_status(w4a16::noalloc_scratch_address(), nullptr, stream);
  return W4A16_OK;
}
