// Sampling verification for callers that cannot allocate device memory.
//
// dflash_verify in sampling mode needs a small scratch buffer (per-row
// softmax statistics) that the caller normally allocates and passes in. Some
// callers cannot do that: code that runs inside a host framework which owns
// every device allocation through its own pool, plugins loaded into another
// runtime that forbids raw cudaMalloc, and serving loops that must not call
// the allocator once they are running (cudaMalloc and cudaFree may
// synchronise the whole device). This entry point runs the same two kernels
// with their scratch in a file-scope device array instead, so it allocates
// nothing.
#include <mutex>

#include "internal.h"

namespace {

// Statistics of up to kNoAllocMaxStreams streams: 31 rows (16 target, 15
// draft) x (max, sum) floats each, 248 KiB. Every GPU that loads the library
// holds this array until the process exits. The limit is the one the header
// documents, so the refusal below and the documented maximum cannot diverge.
constexpr int kNoAllocMaxStreams = DFLASH_NOALLOC_MAX_STREAMS;
static_assert(kNoAllocMaxStreams > 0, "the no-allocation stream limit must be positive");
static __device__ __align__(256) float g_sample_scratch[kNoAllocMaxStreams * 31 * 2];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
float* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device, looked up once
// per device (the array's name is only a host-side stand-in in host code).
int scratch_for_current_device(float** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return DFLASH_E_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return DFLASH_E_UNSUPPORTED;
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_sample_scratch) != cudaSuccess || p == nullptr) return DFLASH_E_CUDA;
    g_scratch_ptr[dev] = static_cast<float*>(p);
  }
  *out = g_scratch_ptr[dev];
  return DFLASH_OK;
}

}  // namespace

extern "C" int dflash_verify_sample_noalloc(int streams, int vocab, const int32_t* draft_ids, int draft_ld,
                                            const void* target_logits, const void* draft_logits,
                                            const float* uniforms, float temperature, int32_t* accept_len,
                                            int32_t* out_tokens, dflash_stream_t stream) {
  if (streams < 0 || vocab < 8 || vocab % 8 || !draft_ids || draft_ld < 1 || !target_logits || !draft_logits ||
      !uniforms || !accept_len || !out_tokens || !(temperature > 0.f))
    return DFLASH_E_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(target_logits) & 15u) || (reinterpret_cast<uintptr_t>(draft_logits) & 15u))
    return DFLASH_E_INVALID_ARG;
  if (streams > kNoAllocMaxStreams) return DFLASH_E_WORKSPACE;
  if (streams == 0) return DFLASH_OK;
  float* scratch = nullptr;
  const int rc = scratch_for_current_device(&scratch);
  if (rc) return rc;
  return dfl::launch_verify_sample(streams, vocab, draft_ids, draft_ld,
                                   static_cast<const __nv_bfloat16*>(target_logits),
                                   static_cast<const __nv_bfloat16*>(draft_logits), uniforms, temperature,
                                   accept_len, out_tokens, scratch, reinterpret_cast<cudaStream_t>(stream));
}
