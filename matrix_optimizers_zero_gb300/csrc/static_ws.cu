// muon_owner_step_noalloc: the Muon step with its scratch in a fixed device
// array owned by this library, for callers that cannot allocate device memory.
//
// Who needs it: code that runs where cudaMalloc is unavailable or forbidden --
// for example a host that has handed the whole device to another memory
// manager (a framework's caching allocator that must see every allocation),
// plugin or callback contexts that may not allocate, or startup paths that
// want a step without first sizing and obtaining a workspace.
//
// The scratch is the array below: kStaticScratchBytes (64 MiB) of device
// memory in every process that loads this code, on every device it is used
// on, held until the process exits. Tables whose workspace
// (mo_muon_workspace_bytes) exceeds it are rejected with
// MO_ERR_SCRATCH_LIMIT before anything is enqueued.
#include <cuda_runtime.h>

#include <array>
#include <cstdint>
#include <mutex>

#include "mo.h"

namespace mo {
struct StepHooks;
void note_cuda_error(int e);   // records the code returned by mo_last_cuda_error()
// The Muon step of abi.cu; allow_pinned = false keeps every host upload in
// pageable memory, so this path allocates no pinned or device memory.
int muon_step_impl(const mo_matrix* tbl, int32_t n, const mo_muon_params* prm, void* ws, size_t ws_bytes,
                   cudaStream_t stream, cudaEvent_t ev_begin, cudaEvent_t ev_end, bool allow_pinned,
                   const StepHooks* hooks);
}

namespace {

constexpr size_t kStaticScratchBytes = size_t(64) << 20;

static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

// Device address of g_static_scratch per device. In host code the array's
// name is only a host-side stand-in, so the address must come from
// cudaGetSymbolAddress with the device current. It is looked up on the first
// call on each device and kept for the life of the process (a
// cudaDeviceReset, after which the array may move, is not supported).
struct ScratchAddr {
  bool ready = false;
  void* ptr = nullptr;
};
std::array<ScratchAddr, 64> g_addr;
std::mutex g_addr_mu;

int scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    mo::note_cuda_error(int(e));
    return MO_ERR_CUDA;
  }
  if (dev < 0 || dev >= int(g_addr.size())) return MO_ERR_UNSUPPORTED_DEVICE;
  std::lock_guard<std::mutex> lock(g_addr_mu);
  ScratchAddr& a = g_addr[size_t(dev)];
  if (!a.ready) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_static_scratch);
    if (e != cudaSuccess || p == nullptr) {
      mo::note_cuda_error(int(e == cudaSuccess ? cudaErrorInvalidSymbol : e));
      return MO_ERR_CUDA;
    }
    a.ptr = p;
    a.ready = true;
  }
  *out = a.ptr;
  return MO_OK;
}

}  // namespace

extern "C" {

size_t mo_static_scratch_bytes(void) { return kStaticScratchBytes; }

int muon_owner_step_noalloc(const mo_matrix* tbl, int32_t n, const mo_muon_params* params, cudaStream_t stream) {
  if (n == 0) return muon_owner_step(tbl, n, params, nullptr, 0, stream);
  const size_t need = mo_muon_workspace_bytes(tbl, n, params);
  if (need == 0) {
    // invalid table or parameters: let the regular entry point report which
    return muon_owner_step(tbl, n, params, nullptr, 0, stream);
  }
  if (need > kStaticScratchBytes) return MO_ERR_SCRATCH_LIMIT;
  void* scratch = nullptr;
  const int st = scratch_address(&scratch);
  if (st != MO_OK) return st;
  // The per-call header written at the start of the scratch resets every
  // counter the step relies on; all other scratch is written before it is read.
  return mo::muon_step_impl(tbl, n, params, scratch, kStaticScratchBytes, stream, nullptr, nullptr, false, nullptr);
}

}  // extern "C"
