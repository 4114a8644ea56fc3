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

#include <nvtx3/nvToolsExt.h>

#include "csa_internal.cuh"
#include "kernels.h"

namespace {

// Largest scratch this entry point can use: the pooled bf16 values (B * token tiles * groups *
// H * 2 bytes).  Every GPU that loads the library holds the
// array until the process exits.
constexpr size_t kScratchBytes = 16u << 20;

static __device__ __align__(256) uint8_t g_noalloc_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_addr[kMaxDevices];  // device address of g_noalloc_scratch, per device

}  // namespace

// Defined in api.cu: records the message returned by csa_last_error on this thread.
int csa_internal_fail(int code, const char* msg);

// Defined in api.cu: the argument checks of csa_compress_prefill, and the call geometry.
int csa_internal_check_prefill(const csa_compressor* c, const uint16_t* x, int B, int N, int start_pos,
                               int slot_offset, const csa_out* out, const char* what, csa::Chunk* ck);

namespace {
int noalloc_call(csa_compressor* c, const uint16_t* x, int B, int N, int start_pos, int slot_offset,
                 const csa_out* out, csa_stream_t stream);
}  // namespace

extern "C" int csa_compress_prefill_noalloc(csa_compressor* c, const uint16_t* x, int B, int N, int start_pos,
                                            int slot_offset, const csa_out* out, csa_stream_t stream) {
  nvtxRangePushA("csa_compress_prefill_noalloc");
  const int rc = noalloc_call(c, x, B, N, start_pos, slot_offset, out, stream);
  nvtxRangePop();
  return rc;
}

namespace {

int noalloc_call(csa_compressor* c, const uint16_t* x, int B, int N, int start_pos, int slot_offset,
                 const csa_out* out, csa_stream_t stream) {
  try {
    csa::Chunk ck;
    // also checks that the handle's device is the current one: the array used below is that
    // device's copy
    const int rc =
        csa_internal_check_prefill(c, x, B, N, start_pos, slot_offset, out, "csa_compress_prefill_noalloc", &ck);
    if (rc) return rc;
    if (!csa::prefill_tc_supported(c, x))
      return csa_internal_fail(CSA_ERR_ARG,
                               "csa_compress_prefill_noalloc: this shape runs the CUDA-core projection, whose "
                               "scratch is not preallocated (needs 128-row packed tiles, ratio <= 256, 16-byte "
                               "aligned x)");
    // the one launch geometry used both for this size check and for the launch below
    const csa::PrefillPlan plan = csa::prefill_tc_plan(c, B, N, ck);
    if (plan.bytes > kScratchBytes)
      return csa_internal_fail(CSA_ERR_ARG,
                               "csa_compress_prefill_noalloc: B x N too large for the preallocated scratch "
                               "(limit: 16 MiB of pooled values)");
    const int dev = c->device;
    if (dev < 0 || dev >= kMaxDevices)
      return csa_internal_fail(CSA_ERR_CUDA, "csa_compress_prefill_noalloc: device index out of range");
    void* base = nullptr;
    {
      // set-up, once per device, with that device current (the check above): the device address
      // of the array
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
    cudaStream_t s = (cudaStream_t)stream;  // the kernel marks the sequences' decode running values invalid
    csa_out o = out ? *out : csa_out{nullptr, nullptr, nullptr, nullptr};
    // the array's capacity is the extent the bounds-checked build checks the scratch stores against
    if (csa::launch_prefill_tc(c, x, B, N, slot_offset, ck, plan, o, base, kScratchBytes, s) != cudaSuccess)
      return csa_internal_fail(CSA_ERR_CUDA, "csa_compress_prefill_noalloc: kernel launch failed");
    c->launches += plan.kernels;
    return ck.G;
  } catch (...) {
    return csa_internal_fail(CSA_ERR_INTERNAL, "csa_compress_prefill_noalloc: unexpected exception");
  }
}

}  // namespace
