// noalloc.cu -- flint_decode_tokens_noalloc: the persistent decode without a
// caller-provided workspace.
//
// Some callers cannot hand the library scratch memory: a host that reserves the whole
// device up front and gives its extensions no allocator, or a serving loop that must
// never call cudaMalloc (it can block, and it can synchronise the device).  For them
// the decode's scratch (the abort word and the tagged boards through which the
// clusters swap residual partial sums and the head's per-CTA maxima) lives in the fixed
// device array below.
// It is part of the loaded module, so every GPU that loads the library holds it until
// the process exits.
#include <mutex>

namespace flint {

// Device-side scratch of the no-allocation decode entry point.
constexpr size_t kNoAllocScratchBytes = FLINT_NOALLOC_SCRATCH_BYTES;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

// In host code g_noalloc_scratch names a host-side shadow, not device memory: the
// device address is looked up once per device with cudaGetSymbolAddress.
static void* g_noalloc_ptr[64];
static std::mutex g_noalloc_mu;

static cudaError_t noalloc_scratch(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (!g_noalloc_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    g_noalloc_ptr[dev] = p;
  }
  *out = g_noalloc_ptr[dev];
  return cudaSuccess;
}

}  // namespace flint

extern "C" flint_status flint_decode_tokens_noalloc(
    const flint_moe_layer* layers, int n_layers, const flint_nvfp4* head, const void* x_bf16,
    const float* residual, int T, float rms_eps, float* out, void* x_out_bf16, float* logits,
    int32_t* argmax, int32_t* topk_idx, float* topk_w, flint_stream stream) {
  if (!layers || n_layers <= 0) return FLINT_ERR_INVALID_ARG;
  if (flint::decode_workspace_bytes(layers[0].hidden) > flint::kNoAllocScratchBytes)
    return FLINT_ERR_UNSUPPORTED;
  void* scratch = nullptr;
  if (flint::noalloc_scratch(&scratch) != cudaSuccess) return FLINT_ERR_CUDA;
  // Every launch clears the scratch it uses (sync words and the tagged exchange
  // boards) before the kernel starts, so what an earlier call left there is harmless.
  return decode_tokens_impl(layers, n_layers, head, x_bf16, residual, T, rms_eps, out,
                            x_out_bf16, logits, argmax, topk_idx, topk_w, nullptr, nullptr,
                            scratch, flint::kNoAllocScratchBytes, stream);
}
