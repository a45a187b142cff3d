// noalloc.cu -- spec_verify_chain for callers that cannot allocate device
// memory.
//
// Some callers have no way to provide the scratch workspace: a plain-C host
// that owns no device allocator and only receives the input and output
// buffers from its embedding application, or a serving runtime that has
// already reserved all device memory (for its KV cache) and forbids further
// allocation, or a decode loop that avoids cudaMalloc because it synchronises
// the device. This entry point needs nothing beyond the inputs and outputs:
// its scratch lives in a fixed array in this library's device memory.
//
// The array is kNoAllocScratchBytes long and exists once per GPU that loads
// the library, for as long as the process lives. Every call on a device uses
// the same array and leaves its contents behind. Nothing carries over from
// one call to the next: each kernel of a call writes every scratch word it
// later reads within that call (no kernel keeps a counter or any other
// state that must start at zero), and the streaming pass, the call's first
// kernel, waits at griddepcontrol.wait until the previous kernel on the same
// stream (the previous call's last one) has completed before it writes. Two
// calls whose work overlaps on the GPU (different streams, or different host
// threads on the same device) share the array and race: the caller must
// order them.
#include <mutex>

#include "internal.h"

namespace {

constexpr size_t kNoAllocScratchBytes = 8u << 20;  // 8 MiB
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_setup_mutex;
void* g_scratch_addr[kMaxDevices] = {nullptr};

// Device address of the scratch array on the current device, looked up once
// per device (the host-side name of the array is not a device address).
int scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return SPEC_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return SPEC_ERR_CUDA;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return SPEC_OK;
}

}  // namespace

extern "C" {

int spec_verify_chain_noalloc(const void* target_logits, const void* draft_logits, int dtype,
                              const int32_t* draft_tokens, const float* u_accept, const float* u_resample,
                              float temperature, int B, int K, int V, int32_t* accept_len, int32_t* out_tokens,
                              float* lse_target, float* lse_draft, float* p_at_x, float* q_at_x,
                              int32_t* row_status, void* stream) {
  const size_t need = spec_workspace_bytes(B, K, V, dtype);
  if (need == 0) return SPEC_ERR_ARG;
  if (need > kNoAllocScratchBytes) return SPEC_ERR_UNSUPPORTED;
  void* scratch = nullptr;
  int e = scratch_address(&scratch);
  if (e) return e;
  return spec_verify_chain(target_logits, draft_logits, dtype, draft_tokens, u_accept, u_resample, temperature, B, K,
                           V, accept_len, out_tokens, lse_target, lse_draft, p_at_x, q_at_x, row_status, scratch,
                           kNoAllocScratchBytes, stream);
}

}  // extern "C"
