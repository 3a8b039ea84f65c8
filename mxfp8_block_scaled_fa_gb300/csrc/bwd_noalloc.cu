// bwd_noalloc.cu -- mxfa_bwd_noalloc: the dense backward pass for callers that
// cannot allocate device memory.
//
// mxfa_bwd needs a caller-provided workspace (Delta and the dQ accumulator).
// Some callers have no way to provide one: code that runs where cudaMalloc is
// not allowed or not wanted (inside another library's allocator or memory
// pool hooks, real-time or embedded runtimes that forbid device allocation
// after start-up, or bindings that have no device allocator at all).  For
// them this entry point uses a scratch array that lives in the library's own
// device image instead, so the call itself allocates nothing.
//
// The array is file-scope, 256-byte aligned and kNoAllocScratchBytes long.
// Every GPU that loads the library holds it until the process exits.  In host
// code the array's name is only a host-side stand-in for the symbol, so its
// device address is looked up once per device (with that device current) by
// cudaGetSymbolAddress and cached; the first call on each device does this
// lookup, so make that first call before any stream capture.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "../../include/mxfa.h"

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(32) << 20;  // 32 MiB
constexpr int kMaxDevices = 64;

__device__ __align__(256) unsigned char g_bwd_scratch[kNoAllocScratchBytes];

std::mutex g_mu;

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of g_bwd_scratch on the current device (nullptr on error).
void* scratch_on_current_device() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_bwd_scratch) != cudaSuccess || !p) {
      (void)cudaGetLastError();  // leave no stale error for the caller's next runtime call
      return nullptr;
    }
    g_scratch_ptr[dev] = p;
  }
  return g_scratch_ptr[dev];
}

}  // namespace

extern "C" size_t mxfa_bwd_noalloc_scratch_bytes(void) { return kNoAllocScratchBytes; }

extern "C" mxfa_status mxfa_bwd_noalloc(const mxfa_mx* q, const mxfa_mx* k, const mxfa_mx* v,
                                        const mxfa_mx* dout_mx, const void* o, const void* dout,
                                        const float* lse, int B, int S, int H, int D,
                                        float softmax_scale, int causal, int dq_mode,
                                        float dq_static_scale, void* dq, void* dk, void* dv,
                                        mxfa_stream_t stream) {
  if (B <= 0 || S <= 0 || H <= 0 || D <= 0) return MXFA_ERR_INVALID_ARG;
  // the argument checks that need no workspace come first, so that a bad
  // call is reported the same way mxfa_bwd reports it
  for (const mxfa_mx* m : {q, k, v, dout_mx}) {
    if (!m || !m->data || !m->sf) return MXFA_ERR_INVALID_ARG;
    if (!aligned16(m->data) || !aligned16(m->sf)) return MXFA_ERR_MISALIGNED;
  }
  if (!o || !dout || !lse || !dq || !dk || !dv) return MXFA_ERR_INVALID_ARG;
  if (D != 128) return MXFA_ERR_UNSUPPORTED;
  if (!aligned16(o) || !aligned16(dout) || !aligned16(dq) || !aligned16(dk) || !aligned16(dv))
    return MXFA_ERR_MISALIGNED;
  const size_t need = mxfa_bwd_workspace_size(int64_t(B) * S, B, H, D, dq_mode);
  if (need == 0) return MXFA_ERR_INVALID_ARG;
  if (need > kNoAllocScratchBytes) return MXFA_ERR_WORKSPACE_TOO_SMALL;
  void* ws = scratch_on_current_device();
  if (!ws) return MXFA_ERR_CUDA;
  return mxfa_bwd(q, k, v, dout_mx, o, dout, lse, B, S, H, D, softmax_scale, causal, dq_mode,
                  dq_static_scale, dq, dk, dv, ws, kNoAllocScratchBytes, stream);
}
