// dflash_noalloc.cu -- dflash_verify for callers that cannot allocate device
// memory.
//
// Some callers have no way to hand the library a workspace: code running
// inside another framework's memory pool that forbids foreign cudaMalloc
// calls, plugins loaded into a process whose allocator they do not own, or
// latency-critical paths where an allocation (and the implicit device
// synchronisation cudaFree can cause) is not allowed. For them this file keeps
// the verification scratch in a fixed, file-scope device array that exists on
// every GPU that loads the library, from module load until process exit.
//
// The array holds kNoAllocScratchBytes (4 MiB): enough for the batched step at
// B = 32, block 8, V = 248320 in bf16 (about 3.6 MB). Shapes whose workspace
// would not fit are rejected with DFLASH_ERR_INVALID_ARG.

#include <cuda_runtime.h>

#include <cstdio>
#include <cstring>
#include <mutex>

#include "../../include/dflash_verify.h"
#include "dflash_internal.h"

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(4) << 20;

// The scratch itself. Host code may not use this name as a pointer: on the
// host it is only a stand-in symbol, so its device address is looked up below.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {nullptr};

int noalloc_fail(int code, const char* msg) {
  dflash::set_last_error(msg);
  return code;
}

// Device address of the scratch on the current device, looked up once per
// device (with that device current) and cached.
int scratch_address(void** out) {
  char msg[256];
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    snprintf(msg, sizeof msg, "dflash_verify_noalloc: cudaGetDevice: %s", cudaGetErrorString(e));
    return noalloc_fail(DFLASH_ERR_CUDA, msg);
  }
  if (dev < 0 || dev >= kMaxDevices) {
    snprintf(msg, sizeof msg, "dflash_verify_noalloc: device %d beyond the supported %d", dev, kMaxDevices);
    return noalloc_fail(DFLASH_ERR_INVALID_ARG, msg);
  }
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || p == nullptr) {
      snprintf(msg, sizeof msg, "dflash_verify_noalloc: cudaGetSymbolAddress of the scratch: %s",
               cudaGetErrorString(e));
      return noalloc_fail(DFLASH_ERR_CUDA, msg);
    }
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return DFLASH_OK;
}

}  // namespace

extern "C" {

size_t dflash_noalloc_scratch_bytes(void) { return kNoAllocScratchBytes; }

int dflash_verify_noalloc(const void* target_logits, const void* draft_logits, const int32_t* draft_tokens,
                          int B, int gamma, int V, int dtype, const float* temperature, int top_k, float top_p,
                          uint64_t seed, int32_t* out_tokens, int32_t* out_accept_len, uint32_t* status,
                          void* stream) {
  const size_t need = dflash_workspace_bytes(B, gamma, V, dtype, top_k, top_p);
  if (need == 0) {
    // Invalid or unsupported shape / filter: the main entry point says which,
    // with the same code and message (DFLASH_ERR_UNSUPPORTED for a filter
    // outside the supported set). It rejects such a call before it looks at
    // its workspace, so a non-null stand-in is passed where the workspace
    // goes: a null one would be reported as a null pointer first.
    static unsigned char stand_in[16];
    return dflash_verify(target_logits, draft_logits, draft_tokens, B, gamma, V, dtype, temperature, top_k,
                         top_p, seed, out_tokens, out_accept_len, stand_in, 0, status, stream);
  }
  char msg[256];
  if (need > kNoAllocScratchBytes) {
    snprintf(msg, sizeof msg,
             "dflash_verify_noalloc: B=%d gamma=%d V=%d needs %zu bytes of scratch, more than the "
             "fixed %zu; use dflash_verify with a caller-provided workspace",
             B, gamma, V, need, kNoAllocScratchBytes);
    return noalloc_fail(DFLASH_ERR_INVALID_ARG, msg);
  }
  void* scratch = nullptr;
  int rc = scratch_address(&scratch);
  if (rc) return rc;
  // The scratch keeps whatever the previous call left. Its counters and tile
  // keys must be zero when the kernel starts (a call that timed out leaves
  // them dirty), so the part this call uses is cleared on the call's stream
  // before every launch.
  cudaError_t e = cudaMemsetAsync(scratch, 0, need, (cudaStream_t)stream);
  if (e != cudaSuccess) {
    snprintf(msg, sizeof msg, "dflash_verify_noalloc: clearing the scratch: %s", cudaGetErrorString(e));
    return noalloc_fail(DFLASH_ERR_CUDA, msg);
  }
  return dflash_verify(target_logits, draft_logits, draft_tokens, B, gamma, V, dtype, temperature, top_k, top_p,
                       seed, out_tokens, out_accept_len, scratch, kNoAllocScratchBytes, status, stream);
}

}  // extern "C"
