// cpa_chunk_prefill_attn_noalloc: the chunk-prefill attention entry point for
// callers that cannot allocate device memory.
//
// Some callers have no way to obtain a workspace: code running while a CUDA
// graph is being captured (an allocation would break or be baked into the
// capture), runtimes whose device memory is planned once up front from static
// shapes (the exported-graph deployments this library serves pre-plan every
// buffer), and plugins embedded in a host framework that owns the allocator
// and exposes none to them.  For them this entry point keeps the split-KV
// partial results in a fixed array compiled into the library instead of in
// caller memory.  It is the regular cpa_chunk_prefill_attn, pointed at that
// array; it allocates nothing.
#include <mutex>

#include "common.cuh"
#include "kernels.h"

namespace {

// 16 MiB of split-KV partials; every GPU that loads this library's device code
// holds it until the process exits.
constexpr size_t kStaticScratchBytes = size_t(16) << 20;
static __device__ __align__(256) unsigned char g_split_scratch[kStaticScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_addr[kMaxDevices] = {};

// Device address of g_split_scratch on the current device, looked up once per
// device (with that device current).  Returns nullptr on failure.
void* scratch_address() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_addr[dev]) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_split_scratch) != cudaSuccess) return nullptr;
    g_addr[dev] = ptr;
  }
  return g_addr[dev];
}

}  // namespace

extern "C" cpa_status cpa_chunk_prefill_attn_noalloc(const cpa_attn_args* args, cpa_stream stream) {
  if (!args) return CPA_ERR_NULL;
  // sized for the call's own SM budget (a partial budget needs fewer partial slots)
  const size_t need = cpa::attn_workspace_need(args);
  if (need > kStaticScratchBytes) return CPA_ERR_WORKSPACE;
  cpa_attn_args a = *args;
  a.workspace = nullptr;
  a.workspace_bytes = 0;
  if (need > 0) {
    void* ptr = scratch_address();
    if (!ptr) return CPA_ERR_CUDA;
    a.workspace = ptr;
    a.workspace_bytes = kStaticScratchBytes;
  }
  return cpa_chunk_prefill_attn(&a, stream);
}
