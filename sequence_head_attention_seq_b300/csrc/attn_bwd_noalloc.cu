// attn_bwd_noalloc.cu -- the attention backward for callers that cannot allocate.
//
// sp_attn_bwd needs a device workspace (the fp32 dQ accumulator and per-row
// statistics) that the caller allocates.  Some callers cannot: code running
// inside a framework or runtime that owns all device memory and forbids
// cudaMalloc/cudaFree on its threads, or code whose allocations would break a
// fixed memory plan.  For them this file keeps the workspace in a fixed-size
// array of device memory that is part of the library image itself, so the entry
// point below allocates nothing.  The array is created when the library's
// device code is loaded on a GPU and stays there until the process exits.
//
// None of the cited pages has a counterpart: this is a packaging variant of sp_attn_bwd.
#include "internal.h"

// Scratch for sp_attn_bwd_noalloc.  In host code this name is only a host-side
// handle, not a device address: its device address comes from cudaGetSymbolAddress
// (below) and is what the kernels receive.
static __device__ __align__(256) uint8_t g_bwd_scratch[SP_NOALLOC_SCRATCH_BYTES];

namespace sp {
namespace {

ContextAddressCache g_scratch_addr;

// Device address of g_bwd_scratch in the current CUDA context.  The first call in a
// context (normally the device's primary context; a caller's own driver-API context gets
// its own copy of the array) looks it up with cudaGetSymbolAddress, with that context
// current; later calls reuse the cached address.
void* scratch_address() {
  return g_scratch_addr.get([]() -> void* {
    void* p = nullptr;
    return cudaGetSymbolAddress(&p, g_bwd_scratch) == cudaSuccess ? p : nullptr;
  });
}

}  // namespace
}  // namespace sp

extern "C" sp_status sp_attn_bwd_noalloc(const sp_attn_params* p, const void* o,
                                         const float* lse, const void* dout, void* dq, void* dk,
                                         void* dv, void* stream) {
  // the shared scratch carries no accumulation from one call to the next
  if (p != nullptr && p->dq_accumulate != 0) return SP_ERR_INVALID_ARG;
  const size_t need = sp_attn_bwd_workspace_size(p);
  if (need == 0) {
    // invalid parameters, or a problem that needs no workspace: the regular entry
    // point validates first; it only asks for a workspace pointer once all is valid
    const sp_status st = sp_attn_bwd(p, o, lse, dout, dq, dk, dv, nullptr, 0, stream);
    if (st != SP_ERR_WORKSPACE) return st;
  }
  if (need > SP_NOALLOC_SCRATCH_BYTES) return SP_ERR_WORKSPACE;
  void* scratch = sp::scratch_address();
  if (scratch == nullptr) return SP_ERR_CUDA;
  // sp_attn_bwd rewrites every workspace byte it reads before reading it, so the
  // previous call's leftovers need no clearing.
  return sp_attn_bwd(p, o, lse, dout, dq, dk, dv, scratch, SP_NOALLOC_SCRATCH_BYTES, stream);
}
