// Prefill entry point that allocates no device memory.
//
// The ordinary csa_compress_prefill grows its scratch (the pooled values of the tensor-core
// kernel) with cudaMalloc on first use.  Some callers cannot
// allow that: serving runtimes that reserve the whole device memory up front for their own
// pool (a later cudaMalloc fails, or fragments memory the runtime has already planned), and
// code that enqueues work while a CUDA graph is being captured on another thread, where
// cudaMalloc is not a permitted call.  This entry point runs the same kernel with its scratch
// in a fixed file-scope device array instead.
#include <mutex>

#include "csa_internal.cuh"
#include "kernels.h"

namespace {

// Largest scratch this entry point can use.  Every GPU that loads the library holds these
// arrays until the process exits.
constexpr size_t kPooledBytes = 16u << 20;  // pooled bf16 values: B * token tiles * groups * H * 2

static __device__ __align__(256) uint8_t g_noalloc_scratch[kPooledBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_addr[kMaxDevices];  // device address of g_noalloc_scratch, per device

}  // namespace

// Defined in api.cu: records the message returned by csa_last_error on this thread.
int csa_internal_fail(int code, const char* msg);

extern "C" int csa_compress_prefill_noalloc(csa_compressor* c, const uint16_t* x, int B, int N, int start_pos,
                                            int slot_offset, const csa_out* out, csa_stream_t stream) {
  if (!c) return csa_internal_fail(CSA_ERR_ARG, "handle is NULL");
  if (!c->weights_set) return csa_internal_fail(CSA_ERR_STATE, "weights not set");
  if (start_pos != 0) return csa_internal_fail(CSA_ERR_ARG, "prefill needs start_pos 0");
  if (B < 1 || N < 1) return csa_internal_fail(CSA_ERR_ARG, "B and N must be >= 1");
  if (slot_offset < 0 || (long long)slot_offset + B > c->opt.max_batch)
    return csa_internal_fail(CSA_ERR_ARG, "state slots exceed max_batch");
  if (!x) return csa_internal_fail(CSA_ERR_ARG, "x is NULL");
  const int G = N / c->ratio;
  if (G > 0 && (!out || !out->latent)) return csa_internal_fail(CSA_ERR_ARG, "out->latent is required");
  if (G > 0 && c->opt.rope_dim > 0 && (long long)c->ratio * (G - 1) >= c->opt.max_pos)
    return csa_internal_fail(CSA_ERR_ARG, "entry position exceeds the RoPE table (max_pos)");
  if (!csa::prefill_tc_supported(c, x))
    return csa_internal_fail(CSA_ERR_ARG,
                             "csa_compress_prefill_noalloc: this shape runs the CUDA-core projection, whose "
                             "scratch is not preallocated (needs 128-row packed tiles, ratio <= 256, 16-byte "
                             "aligned x)");
  const size_t bytes = csa::prefill_tc_scratch_bytes(c, B, N);
  if (bytes > kPooledBytes)
    return csa_internal_fail(CSA_ERR_ARG,
                             "csa_compress_prefill_noalloc: B x N too large for the preallocated scratch "
                             "(limit: 16 MiB of pooled values)");
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
    return csa_internal_fail(CSA_ERR_CUDA, "csa_compress_prefill_noalloc: no current device");
  void* base = nullptr;
  {
    // set-up, once per device, with that device current: the device address of the array
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_addr[dev]) {
      void* p = nullptr;
      cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
      if (e != cudaSuccess || !p)
        return csa_internal_fail(CSA_ERR_CUDA, "csa_compress_prefill_noalloc: cudaGetSymbolAddress failed");
      g_addr[dev] = p;
    }
    base = g_addr[dev];
  }
  cudaStream_t s = (cudaStream_t)stream;
  if (csa::invalidate_decode_acc(c, slot_offset, B, s) != cudaSuccess)
    return csa_internal_fail(CSA_ERR_CUDA, "csa_compress_prefill_noalloc: marking the decode running values failed");
  csa_out o = out ? *out : csa_out{nullptr, nullptr, nullptr, nullptr};
  if (csa::launch_prefill_tc(c, x, B, N, slot_offset, o, base, s) != cudaSuccess)
    return csa_internal_fail(CSA_ERR_CUDA, "csa_compress_prefill_noalloc: kernel launch failed");
  c->launches += G > 0 ? 2 : 1;
  return G;
}
