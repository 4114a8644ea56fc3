// C ABI of the compressor: argument checks, ownership of device buffers, the host-built
// YaRN RoPE table, and the launch sequence of each call.  Declared in include/csa.h.
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <new>
#include <string>
#include <vector>

#include <nvtx3/nvToolsExt.h>

#include "csa_internal.cuh"
#include "kernels.h"

namespace {

// An NVTX range around an ABI call, for timelines taken with the CUDA tools (a no-op otherwise).
struct NvtxRange {
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
};

thread_local std::string g_last_error;

int fail(int code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return code;
}

int cuda_fail(cudaError_t e, const char* what) {
  return fail(CSA_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

#define CSA_CUDA(call, what)                  \
  do {                                        \
    cudaError_t e_ = (call);                  \
    if (e_ != cudaSuccess) return cuda_fail(e_, what); \
  } while (0)

// YaRN NTK-by-parts frequency correction (Peng et al., 2023), as used by the compressed
// layers' RoPE table ("Module compress", yarn_freqs_cis, built from compress_rope_theta):
// dims whose wavelength turns more than beta_fast times over the original context keep
// their frequency, dims turning fewer than beta_slow times are divided by the factor,
// with a linear ramp between the two correction dims.
void yarn_inv_freq(const csa_options& o, std::vector<double>& f) {
  const int d = o.rope_dim;
  const double base = o.rope_base;
  auto corr = [&](double turns) {
    return d * std::log((double)o.rope_orig_len / (turns * 2.0 * M_PI)) / (2.0 * std::log(base));
  };
  double lo = std::floor(corr(o.beta_fast)), hi = std::ceil(corr(o.beta_slow));
  lo = std::max(lo, 0.0);
  hi = std::min(hi, (double)(d - 1));
  if (hi == lo) hi += 0.001;
  f.resize(d / 2);
  for (int i = 0; i < d / 2; ++i) {
    const double f0 = std::pow(base, -2.0 * i / d);
    const double t = std::min(std::max((i - lo) / (hi - lo), 0.0), 1.0);
    f[i] = f0 / o.rope_factor * t + f0 * (1.0 - t);
  }
}

void rope_rows(const csa_options& o, const std::vector<double>& f, int pos0, int npos, float* cs, float* sn) {
  const int hr = o.rope_dim / 2;
  for (int p = 0; p < npos; ++p)
    for (int i = 0; i < hr; ++i) {
      const double th = (double)(pos0 + p) * f[i];  // angle in double: pos * f reaches ~1e5 rad
      cs[(size_t)p * hr + i] = (float)std::cos(th);
      sn[(size_t)p * hr + i] = (float)std::sin(th);
    }
}

bool check_options(const csa_options& o, int H, std::string& why) {
  char buf[256];
  if (o.max_batch < 1) why = "max_batch must be >= 1";
  else if (o.rope_dim < 0 || o.rope_dim % 2 || o.rope_dim > H) {
    snprintf(buf, sizeof buf, "rope_dim %d must be even and in [0, head_dim=%d]", o.rope_dim, H);
    why = buf;
  } else if (o.rope_dim > 0 && (o.max_pos < 1 || !(o.rope_base > 1.0f) || !(o.rope_factor > 0.0f) ||
                                o.rope_orig_len < 1 || !(o.beta_fast > 0.0f) || !(o.beta_slow > 0.0f)))
    why = "invalid RoPE options (max_pos, rope_base, rope_factor, rope_orig_len, beta_fast, beta_slow)";
  else if (o.fp4 < 0 || o.fp4 > 2) why = "fp4 must be 0 (off), 1 (e4m3 scales, block 16) or 2 (power-of-two scales, block 32)";
  else if (o.fp4 == 2 && H % 32) {
    snprintf(buf, sizeof buf, "fp4 = 2 quantises blocks of 32 features: head_dim %d must be a multiple of 32", H);
    why = buf;
  }
  else if (!(o.eps >= 0.0f)) why = "eps must be >= 0";
  else if (o.prefill_split < 0 || o.prefill_split > 2) why = "prefill_split must be 0 (chosen per call), 1 or 2";
  else if (o.prefill_pair != 0 && o.prefill_pair != 2) why = "prefill_pair must be 0 (one CTA per packed tile) or 2";
  else return true;
  return false;
}

void free_all(csa_compressor* c) {
  cudaFree(c->w_packed);
  cudaFree(c->w_planes);
  cudaFree(c->gain);
  cudaFree(c->ape);
  cudaFree(c->rope_cos);
  cudaFree(c->rope_sin);
  cudaFree(c->state);
  cudaFree(c->dev_flag);
  cudaFree(c->scratch);
  cudaFree(c->dec_part);
  cudaFree(c->dec_acc);
  cudaFree(c->dec_acc_pos);
  cudaFree(c->prefill_order);
  cudaFree(c->dec_pos);
}

int ensure_scratch(csa_compressor* c, size_t bytes, cudaStream_t s) {
  if (c->scratch_bytes >= bytes) return CSA_OK;
  // failure injection on the host, for tests of the error path: CSA_TEST_FAIL_ALLOC set makes
  // growing the scratch fail as a cudaMalloc failure would (nothing is freed or enqueued)
  if (getenv("CSA_TEST_FAIL_ALLOC"))
    return fail(CSA_ERR_CUDA, "cudaMalloc(scratch): forced failure (CSA_TEST_FAIL_ALLOC is set)");
  CSA_CUDA(cudaStreamSynchronize(s), "cudaStreamSynchronize");
  cudaFree(c->scratch);
  c->scratch = nullptr;
  c->scratch_bytes = 0;
  CSA_CUDA(cudaMalloc(&c->scratch, bytes), "cudaMalloc(scratch)");
  c->scratch_bytes = bytes;
  return CSA_OK;
}

// Every call on a handle launches on the current device with pointers into the handle's device
// memory: a call made while another device is current would use them on the wrong GPU.
int check_device(const csa_compressor* c, const char* what) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev != c->device)
    return fail(CSA_ERR_ARG, "%s: the handle lives on device %d but device %d is current", what, c->device, dev);
  return CSA_OK;
}

// Checks shared by the prefill entry points; on success fills the call geometry.  cache_rows < 0:
// entries go to out [B][G][..]; else to rows start_pos / ratio .. of a cache [B][cache_rows][..].
int check_prefill(const csa_compressor* c, const uint16_t* x, int B, int N, int start_pos, int slot_offset,
                  const csa_out* out, int cache_rows, const char* what, csa::Chunk* ck) {
  if (!c) return fail(CSA_ERR_ARG, "%s: handle is NULL", what);
  if (!c->weights_set) return fail(CSA_ERR_STATE, "%s: weights not set", what);
  if (int rc = check_device(c, what)) return rc;
  if (B < 1 || N < 1) return fail(CSA_ERR_ARG, "%s: B (%d) and N (%d) must be >= 1", what, B, N);
  if (start_pos < 0 || (long long)start_pos + N > 0x7fffffffLL)
    return fail(CSA_ERR_ARG, "%s: start_pos %d must be >= 0 and start_pos + N must fit in int32", what, start_pos);
  if (slot_offset < 0 || (long long)slot_offset + B > c->opt.max_batch)
    return fail(CSA_ERR_ARG, "%s: slots [%d, %d) exceed max_batch %d", what, slot_offset, slot_offset + B,
                c->opt.max_batch);
  if (!x) return fail(CSA_ERR_ARG, "%s: x is NULL", what);
  if ((long long)B * N > 0x7fffffffLL) return fail(CSA_ERR_ARG, "%s: B * N too large", what);
  const int r = c->ratio;
  const int gend = (int)(((long long)start_pos + N) / r);
  if (cache_rows >= 0 && gend > cache_rows)
    return fail(CSA_ERR_ARG, "%s: group %d does not fit a cache of %d rows", what, gend - 1, cache_rows);
  *ck = csa::make_chunk(start_pos, N, r);
  if (cache_rows >= 0) {
    ck->bstride = cache_rows;
    ck->row0 = ck->g0;
  }
  if (ck->G > 0 && (!out || !out->latent)) return fail(CSA_ERR_ARG, "%s: out->latent is required", what);
  if (ck->G > 0 && c->opt.rope_dim > 0 && (long long)r * (gend - 1) >= c->opt.max_pos)
    return fail(CSA_ERR_ARG, "%s: entry position %lld exceeds the RoPE table (max_pos %d)", what,
                (long long)r * (gend - 1), c->opt.max_pos);
  return CSA_OK;
}

int prefill_call(csa_compressor* c, const uint16_t* x, int B, int N, int start_pos, int slot_offset,
                 const csa_out* out, int cache_rows, csa_stream_t stream, const char* what) {
  NvtxRange range(what);
  try {
    csa::Chunk ck;
    int rc = check_prefill(c, x, B, N, start_pos, slot_offset, out, cache_rows, what, &ck);
    if (rc) return rc;
    cudaStream_t s = (cudaStream_t)stream;
    const long long M = (long long)B * N;
    const csa_out o = out ? *out : csa_out{nullptr, nullptr, nullptr, nullptr};
    if (csa::prefill_tc_supported(c, x)) {  // the kernel marks the decode running values invalid
      const csa::PrefillPlan plan = csa::prefill_tc_plan(c, B, N, ck);
      rc = ensure_scratch(c, plan.bytes, s);
      if (rc) return rc;
      if (c->prof_start) CSA_CUDA(cudaEventRecord(c->prof_start, s), "cudaEventRecord");
      CSA_CUDA(csa::launch_prefill_tc(c, x, B, N, slot_offset, ck, plan, o, c->scratch, c->scratch_bytes, s),
               "tensor-core prefill launch");
      if (c->prof_stop) CSA_CUDA(cudaEventRecord(c->prof_stop, s), "cudaEventRecord");
      c->launches += plan.kernels;
      return ck.G;
    }
    CSA_CUDA(csa::invalidate_decode_acc(c, slot_offset, B, s), "invalidate decode running values");
    rc = ensure_scratch(c, (size_t)M * c->pk.cols() * sizeof(float), s);
    if (rc) return rc;
    if (c->prof_start) CSA_CUDA(cudaEventRecord(c->prof_start, s), "cudaEventRecord");
    CSA_CUDA(csa::launch_projection_ffma(c, x, (int)M, c->scratch, 0, nullptr, N, start_pos, s), "projection launch");
    if (c->prof_stop) CSA_CUDA(cudaEventRecord(c->prof_stop, s), "cudaEventRecord");
    c->launches += 1;
    if (ck.G > 0) {
      CSA_CUDA(csa::launch_prefill_pool(c, c->scratch, B, N, slot_offset, ck, o, s), "pool launch");
      c->launches += 1;
    }
    CSA_CUDA(csa::launch_prefill_state(c, c->scratch, B, N, slot_offset, ck, s), "state launch");
    c->launches += 1;
    return ck.G;
  } catch (...) {
    return fail(CSA_ERR_INTERNAL, "%s: unexpected exception", what);
  }
}

int check_decode(const csa_compressor* c, const uint16_t* x_tok, int B, const csa_out* out, const char* what) {
  if (!c) return fail(CSA_ERR_ARG, "%s: handle is NULL", what);
  if (!c->weights_set) return fail(CSA_ERR_STATE, "%s: weights not set", what);
  if (int rc = check_device(c, what)) return rc;
  if (B < 1 || B > c->opt.max_batch)
    return fail(CSA_ERR_ARG, "%s: B %d must be in [1, max_batch=%d]", what, B, c->opt.max_batch);
  if (!x_tok || !out || !out->latent) return fail(CSA_ERR_ARG, "%s: x_tok and out->latent are required", what);
  return CSA_OK;
}

// The decode kernels of one step, positions and emission flags in device memory (emitted may be
// null: the host form fills its own).
int decode_call(csa_compressor* c, const uint16_t* x_tok, int B, const int32_t* start_pos, const csa_out& out,
                uint8_t* emitted, cudaStream_t s) {
  if (csa::decode_tc_supported(c, x_tok, B)) {
    // split-K partial sums: [slices][B][2C] f32, grown on first use (a later call of the same or
    // smaller B allocates nothing)
    const size_t bytes = csa::decode_tc_part_bytes(c, B);
    if (c->dec_part_bytes < bytes) {
      CSA_CUDA(cudaStreamSynchronize(s), "cudaStreamSynchronize");
      cudaFree(c->dec_part);
      c->dec_part = nullptr;
      c->dec_part_bytes = 0;
      CSA_CUDA(cudaMalloc(&c->dec_part, bytes), "cudaMalloc(decode partial sums)");
      c->dec_part_bytes = bytes;
    }
    if (c->prof_start) CSA_CUDA(cudaEventRecord(c->prof_start, s), "cudaEventRecord");
    CSA_CUDA(csa::launch_decode_tc(c, x_tok, B, start_pos, c->dec_part, out, emitted, c->dec_early_start, s),
             "tensor-core decode launch");
    if (c->prof_stop) CSA_CUDA(cudaEventRecord(c->prof_stop, s), "cudaEventRecord");
    c->dec_early_start = true;
    c->launches += csa::decode_tc_kernels_per_call();
    return CSA_OK;
  }
  CSA_CUDA(csa::invalidate_decode_acc(c, 0, B, s), "invalidate decode running values");
  if (c->prof_start) CSA_CUDA(cudaEventRecord(c->prof_start, s), "cudaEventRecord");
  CSA_CUDA(csa::launch_projection_ffma(c, x_tok, B, c->state, 1, start_pos, 0, 0, s), "decode projection launch");
  if (c->prof_stop) CSA_CUDA(cudaEventRecord(c->prof_stop, s), "cudaEventRecord");
  CSA_CUDA(csa::launch_decode_emit(c, start_pos, B, out, emitted, s), "decode emit launch");
  c->launches += 2;
  return CSA_OK;
}

}  // namespace

// Argument checks of a prefill call, shared with the no-alloc entry point (not part of the C ABI).
__attribute__((visibility("hidden"))) int csa_internal_check_prefill(const csa_compressor* c, const uint16_t* x, int B,
                                                                  int N, int start_pos, int slot_offset,
                                                                  const csa_out* out, const char* what,
                                                                  csa::Chunk* ck) {
  return check_prefill(c, x, B, N, start_pos, slot_offset, out, -1, what, ck);
}

// Used by other translation units of the library to report a failure through
// csa_last_error (not part of the C ABI).
__attribute__((visibility("hidden"))) int csa_internal_fail(int code, const char* msg) { return fail(code, "%s", msg); }

extern "C" {

void csa_options_default(csa_options* o) {
  if (!o) return;
  o->max_batch = 128;
  o->rope_dim = 64;
  o->rope_base = 160000.0f;
  o->rope_factor = 16.0f;
  o->rope_orig_len = 4096;
  o->beta_fast = 32.0f;
  o->beta_slow = 1.0f;
  o->max_pos = 262144;
  o->fp4 = 1;
  o->eps = 1e-6f;
  o->prefill_split = 0;
  o->prefill_pair = 0;
}

const char* csa_last_error(void) { return g_last_error.c_str(); }

int csa_rope_table(const csa_options* opt, int pos0, int npos, float* cos_out, float* sin_out) {
  if (!opt || !cos_out || !sin_out || pos0 < 0 || npos < 0 || opt->rope_dim <= 0 || opt->rope_dim % 2)
    return fail(CSA_ERR_ARG, "csa_rope_table: bad arguments");
  std::vector<double> f;
  yarn_inv_freq(*opt, f);
  rope_rows(*opt, f, pos0, npos, cos_out, sin_out);
  return CSA_OK;
}

int csa_compressor_create(int dim, int H, int ratio, int overlap, csa_compressor** out) {
  return csa_compressor_create_ex(dim, H, ratio, overlap, nullptr, out);
}

int csa_compressor_create_ex(int dim, int H, int ratio, int overlap, const csa_options* opt, csa_compressor** out) {
  try {
    if (!out) return fail(CSA_ERR_ARG, "csa_compressor_create: out is NULL");
    *out = nullptr;
    if (dim <= 0 || dim % 64) return fail(CSA_ERR_ARG, "dim %d must be a positive multiple of 64", dim);
    if (H < 16 || H > 512 || H % 16) return fail(CSA_ERR_ARG, "head_dim %d must be a multiple of 16 in [16, 512]", H);
    if (ratio < 1) return fail(CSA_ERR_ARG, "ratio %d must be >= 1", ratio);
    if (overlap != 0 && overlap != 1) return fail(CSA_ERR_ARG, "overlap must be 0 or 1");
    if (overlap && ratio != 4) return fail(CSA_ERR_ARG, "the overlapped form exists only at ratio 4 (got %d)", ratio);
    csa_options o;
    csa_options_default(&o);
    if (opt) o = *opt;
    std::string why;
    if (!check_options(o, H, why)) return fail(CSA_ERR_ARG, "%s", why.c_str());
    csa::Packing pk = csa::make_packing(H, overlap);
    if (H % pk.ft) return fail(CSA_ERR_ARG, "head_dim %d must be a multiple of %d", H, pk.ft);

    auto* c = new (std::nothrow) csa_compressor();
    if (!c) return fail(CSA_ERR_INTERNAL, "out of host memory");
    c->dim = dim;
    c->H = H;
    c->ratio = ratio;
    c->overlap = overlap;
    c->width = (1 + overlap) * H;
    c->opt = o;
    c->pk = pk;
    c->slots = overlap ? 8 : ratio;
    c->weights_set = false;
    if (cudaError_t ed = cudaGetDevice(&c->device); ed != cudaSuccess) {
      delete c;
      return cuda_fail(ed, "cudaGetDevice");
    }
    const size_t ncol = pk.cols();
    cudaError_t e = cudaSuccess;
    auto alloc = [&](void** p, size_t bytes) {
      if (e == cudaSuccess) e = cudaMalloc(p, bytes);
    };
    alloc((void**)&c->w_packed, ncol * dim * sizeof(float));
    alloc((void**)&c->w_planes, 3 * ncol * dim * sizeof(__nv_bfloat16));
    alloc((void**)&c->gain, H * sizeof(float));
    alloc((void**)&c->state, (size_t)o.max_batch * c->slots * ncol * sizeof(float));
    alloc((void**)&c->dev_flag, sizeof(int));
    alloc((void**)&c->dec_acc, (size_t)o.max_batch * 3 * H * sizeof(float));
    alloc((void**)&c->dec_acc_pos, (size_t)o.max_batch * pk.ntiles * sizeof(int));
    alloc((void**)&c->prefill_order, (size_t)o.max_batch * pk.ntiles * 2 * sizeof(int));
    alloc((void**)&c->dec_pos, (size_t)o.max_batch * sizeof(int32_t));
    if (o.rope_dim > 0) {
      const size_t n = (size_t)o.max_pos * (o.rope_dim / 2);
      alloc((void**)&c->rope_cos, n * sizeof(float));
      alloc((void**)&c->rope_sin, n * sizeof(float));
      if (e == cudaSuccess) {
        std::vector<double> f;
        yarn_inv_freq(o, f);
        std::vector<float> cs(n), sn(n);
        rope_rows(o, f, 0, o.max_pos, cs.data(), sn.data());
        e = cudaMemcpy(c->rope_cos, cs.data(), n * sizeof(float), cudaMemcpyHostToDevice);
        if (e == cudaSuccess) e = cudaMemcpy(c->rope_sin, sn.data(), n * sizeof(float), cudaMemcpyHostToDevice);
      }
    }
    if (e == cudaSuccess) e = cudaMemset(c->dev_flag, 0, sizeof(int));
    if (e == cudaSuccess) e = cudaMemset(c->dec_acc_pos, 0xFF, (size_t)o.max_batch * pk.ntiles * sizeof(int));
    if (e == cudaSuccess) e = cudaMemset(c->prefill_order, 0, (size_t)o.max_batch * pk.ntiles * 2 * sizeof(int));
    if (e == cudaSuccess && csa::launch_state_reset(c, 0, o.max_batch, 0) != cudaSuccess) e = cudaGetLastError();
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    if (e != cudaSuccess) {
      free_all(c);
      delete c;
      return cuda_fail(e, "csa_compressor_create");
    }
    *out = c;
    return CSA_OK;
  } catch (...) {
    return fail(CSA_ERR_INTERNAL, "csa_compressor_create: unexpected exception");
  }
}

int csa_compressor_set_weights(csa_compressor* c, const float* wkv, const float* wgate, const float* gain,
                               csa_stream_t stream) {
  NvtxRange range("csa_compressor_set_weights");
  if (!c) return fail(CSA_ERR_ARG, "handle is NULL");
  if (!wkv || !gain) return fail(CSA_ERR_ARG, "wkv and norm_gain are required");
  if (!wgate && c->ratio > 1) return fail(CSA_ERR_ARG, "wgate is required at ratio > 1");
  if (int rc = check_device(c, "csa_compressor_set_weights")) return rc;
  cudaStream_t s = (cudaStream_t)stream;
  CSA_CUDA(csa::launch_pack_weights(c, wkv, wgate, s), "pack_weights launch");
  c->launches += 1;
  CSA_CUDA(cudaMemcpyAsync(c->gain, gain, c->H * sizeof(float), cudaMemcpyDeviceToDevice, s), "copy gain");
  c->weights_set = true;
  c->dec_early_start = false;  // the next decode reads the new planes only after this stream's work
  return CSA_OK;
}

int csa_compressor_set_gate_bias(csa_compressor* c, const float* ape, csa_stream_t stream) {
  if (!c) return fail(CSA_ERR_ARG, "handle is NULL");
  if (int rc = check_device(c, "csa_compressor_set_gate_bias")) return rc;
  if (!ape) {
    c->ape_set = false;
    return CSA_OK;
  }
  cudaStream_t s = (cudaStream_t)stream;
  if (!c->ape) CSA_CUDA(cudaMalloc(&c->ape, (size_t)c->ratio * c->pk.cols() * sizeof(float)), "cudaMalloc(gate bias)");
  CSA_CUDA(csa::launch_pack_ape(c, ape, s), "gate bias launch");
  c->launches += 1;
  c->ape_set = true;
  return CSA_OK;
}

int csa_compress_prefill(csa_compressor* c, const uint16_t* x, int B, int N, int start_pos, int slot_offset,
                         const csa_out* out, csa_stream_t stream) {
  return prefill_call(c, x, B, N, start_pos, slot_offset, out, -1, stream, "csa_compress_prefill");
}

int csa_compress_prefill_into(csa_compressor* c, const uint16_t* x, int B, int N, int start_pos, int slot_offset,
                              const csa_out* cache, int cache_rows, csa_stream_t stream) {
  if (cache_rows < 1) return fail(CSA_ERR_ARG, "csa_compress_prefill_into: cache_rows %d must be >= 1", cache_rows);
  return prefill_call(c, x, B, N, start_pos, slot_offset, cache, cache_rows, stream, "csa_compress_prefill_into");
}

int csa_compress_decode(csa_compressor* c, const uint16_t* x_tok, int B, const int32_t* start_pos,
                        const csa_out* out, uint8_t* emitted, csa_stream_t stream) {
  NvtxRange range("csa_compress_decode");
  try {
    if (int rc = check_decode(c, x_tok, B, out, "csa_compress_decode")) return rc;
    if (!start_pos) return fail(CSA_ERR_ARG, "csa_compress_decode: start_pos (host) is required");
    // the positions are on the host: validate them here, count the emitting sequences ("None"
    // for the others) and fill a host emitted array; a device emitted array is left to the kernels
    int count = 0;
    const int r = c->ratio;
    for (int b = 0; b < B; ++b) {
      const long long p = start_pos[b];
      if (p < 0) return fail(CSA_ERR_ARG, "csa_compress_decode: start_pos[%d] = %lld is negative", b, p);
      if ((p + 1) % r == 0) {
        if (c->opt.rope_dim > 0 && p + 1 - r >= c->opt.max_pos)
          return fail(CSA_ERR_ARG, "csa_compress_decode: entry position %lld of sequence %d exceeds the RoPE table (max_pos %d)",
                      p + 1 - r, b, c->opt.max_pos);
        ++count;
      }
    }
    uint8_t* emitted_dev = nullptr;
    if (emitted) {
      cudaPointerAttributes pa;
      if (cudaPointerGetAttributes(&pa, emitted) == cudaSuccess &&
          (pa.type == cudaMemoryTypeDevice || pa.type == cudaMemoryTypeManaged)) {
        emitted_dev = emitted;
      } else {
        cudaGetLastError();  // an unregistered host pointer may leave an error behind on old drivers
        for (int b = 0; b < B; ++b) emitted[b] = (start_pos[b] + 1) % r == 0 ? 1 : 0;
      }
    }
    cudaStream_t s = (cudaStream_t)stream;
    // a copy from ordinary host memory is staged before cudaMemcpyAsync returns: the caller may
    // reuse start_pos at once, and this call's copy is ordered before its kernels
    CSA_CUDA(cudaMemcpyAsync(c->dec_pos, start_pos, (size_t)B * sizeof(int32_t), cudaMemcpyHostToDevice, s),
             "copy start_pos to the device");
    int rc = decode_call(c, x_tok, B, c->dec_pos, *out, emitted_dev, s);
    return rc ? rc : count;
  } catch (...) {
    return fail(CSA_ERR_INTERNAL, "csa_compress_decode: unexpected exception");
  }
}

int csa_compress_decode_dev(csa_compressor* c, const uint16_t* x_tok, int B, const int32_t* start_pos,
                            const csa_out* out, uint8_t* emitted, csa_stream_t stream) {
  NvtxRange range("csa_compress_decode_dev");
  try {
    if (int rc = check_decode(c, x_tok, B, out, "csa_compress_decode_dev")) return rc;
    if (!start_pos || !emitted) return fail(CSA_ERR_ARG, "csa_compress_decode_dev: start_pos and emitted are required");
    return decode_call(c, x_tok, B, start_pos, *out, emitted, (cudaStream_t)stream);
  } catch (...) {
    return fail(CSA_ERR_INTERNAL, "csa_compress_decode_dev: unexpected exception");
  }
}

int csa_state_reset(csa_compressor* c, int slot_begin, int slot_count, csa_stream_t stream) {
  NvtxRange range("csa_state_reset");
  if (!c) return fail(CSA_ERR_ARG, "handle is NULL");
  if (int rc = check_device(c, "csa_state_reset")) return rc;
  if (slot_begin < 0 || slot_count < 0 || (long long)slot_begin + slot_count > c->opt.max_batch)
    return fail(CSA_ERR_ARG, "slots [%d, %d) outside [0, %d)", slot_begin, slot_begin + slot_count, c->opt.max_batch);
  CSA_CUDA(csa::invalidate_decode_acc(c, slot_begin, slot_count, (cudaStream_t)stream),
           "invalidate decode running values");
  CSA_CUDA(csa::launch_state_reset(c, slot_begin, slot_count, (cudaStream_t)stream), "state reset launch");
  // the chunk ordering counters are zero after every call that completed; a call that timed out
  // may have left one set
  CSA_CUDA(cudaMemsetAsync(c->prefill_order + (size_t)slot_begin * c->pk.ntiles * 2, 0,
                           (size_t)slot_count * c->pk.ntiles * 2 * sizeof(int), (cudaStream_t)stream),
           "reset chunk ordering counters");
  c->launches += slot_count > 0;
  return CSA_OK;
}

int64_t csa_state_elems(const csa_compressor* c) {
  if (!c) return fail(CSA_ERR_ARG, "handle is NULL");
  return (int64_t)c->opt.max_batch * c->slots * c->width;
}

int csa_state_export(const csa_compressor* c, float* kv, float* score, csa_stream_t stream) {
  if (!c) return fail(CSA_ERR_ARG, "handle is NULL");
  if (!kv || !score) return fail(CSA_ERR_ARG, "kv and score are required");
  if (int rc = check_device(c, "csa_state_export")) return rc;
  CSA_CUDA(csa::launch_state_export(c, kv, score, (cudaStream_t)stream), "state export launch");
  const_cast<csa_compressor*>(c)->launches += 1;
  return CSA_OK;
}

int csa_state_import(csa_compressor* c, const float* kv, const float* score, csa_stream_t stream) {
  if (!c) return fail(CSA_ERR_ARG, "handle is NULL");
  if (!kv || !score) return fail(CSA_ERR_ARG, "kv and score are required");
  if (int rc = check_device(c, "csa_state_import")) return rc;
  cudaStream_t s = (cudaStream_t)stream;
  const int mb = c->opt.max_batch;
  CSA_CUDA(csa::launch_state_import(c, kv, score, s), "state import launch");
  CSA_CUDA(csa::invalidate_decode_acc(c, 0, mb, s), "invalidate decode running values");
  CSA_CUDA(cudaMemsetAsync(c->prefill_order, 0, (size_t)mb * c->pk.ntiles * 2 * sizeof(int), s),
           "reset chunk ordering counters");
  c->launches += 1;
  return CSA_OK;
}

int csa_set_profile_events(csa_compressor* c, csa_event_t start, csa_event_t stop) {
  if (!c) return fail(CSA_ERR_ARG, "handle is NULL");
  if ((start == nullptr) != (stop == nullptr)) return fail(CSA_ERR_ARG, "set both events or neither");
  c->prof_start = (cudaEvent_t)start;
  c->prof_stop = (cudaEvent_t)stop;
  return CSA_OK;
}

int csa_uses_tensor_cores(const csa_compressor* c) {
  if (!c) return fail(CSA_ERR_ARG, "handle is NULL");
  static const uint16_t aligned[8] = {};
  return csa::prefill_tc_supported(c, aligned) ? 1 : 0;
}

int64_t csa_kernel_launches(const csa_compressor* c) {
  if (!c) return fail(CSA_ERR_ARG, "handle is NULL");
  return c->launches;
}

int csa_prefill_geometry(const csa_compressor* c, int B, int N, int start_pos, int* token_tile, int* k_split,
                         int* cta_pair) {
  try {
    if (!c || !token_tile || !k_split) return fail(CSA_ERR_ARG, "csa_prefill_geometry: NULL argument");
    if (B < 1 || N < 1 || start_pos < 0) return fail(CSA_ERR_ARG, "csa_prefill_geometry: bad shape");
    if (int rc = check_device(c, "csa_prefill_geometry")) return rc;
    static const uint16_t aligned[8] = {};
    if (!csa::prefill_tc_supported(c, aligned))
      return fail(CSA_ERR_STATE, "csa_prefill_geometry: this compressor runs the CUDA-core projection");
    const csa::PrefillPlan plan = csa::prefill_tc_plan(c, B, N, csa::make_chunk(start_pos, N, c->ratio));
    *token_tile = plan.tok;
    *k_split = plan.split;
    if (cta_pair) *cta_pair = plan.pair;
    return CSA_OK;
  } catch (...) {
    return fail(CSA_ERR_INTERNAL, "csa_prefill_geometry: unexpected exception");
  }
}

int csa_device_status(csa_compressor* c, csa_stream_t stream) {
  if (!c) return fail(CSA_ERR_ARG, "handle is NULL");
  if (int rc = check_device(c, "csa_device_status")) return rc;
  cudaStream_t s = (cudaStream_t)stream;
  int flag = 0;
  CSA_CUDA(cudaMemcpyAsync(&flag, c->dev_flag, sizeof(int), cudaMemcpyDeviceToHost, s), "read device flag");
  CSA_CUDA(cudaStreamSynchronize(s), "cudaStreamSynchronize");
  if (!flag) return CSA_OK;
  CSA_CUDA(cudaMemsetAsync(c->dev_flag, 0, sizeof(int), s), "clear device flag");
  return fail((flag & 4) ? CSA_ERR_TIMEOUT : CSA_ERR_DEVICE, "device flag 0x%x:%s%s%s%s%s", flag,
              (flag & 1) ? " negative start_pos;" : "", (flag & 2) ? " entry position beyond the RoPE table;" : "",
              (flag & 4) ? " wait budget exhausted;" : "", (flag & 8) ? " index out of bounds (bounds-checked build);" : "",
              (flag & 16) ? " chunk ordering counters left set (bounds-checked build);" : "");
}

void csa_compressor_destroy(csa_compressor* c) {
  if (!c) return;
  cudaDeviceSynchronize();
  free_all(c);
  delete c;
}

int csa_fp4_e4m3_roundtrip(const uint16_t* in, int64_t n_blocks, uint8_t* codes, uint8_t* scales, uint16_t* out,
                           csa_stream_t stream) {
  if (n_blocks < 0 || (n_blocks > 0 && (!in || !scales || !out))) return fail(CSA_ERR_ARG, "bad arguments");
  if (n_blocks == 0) return CSA_OK;  // nothing to do, nothing enqueued
  CSA_CUDA(csa::launch_fp4_roundtrip(in, n_blocks, codes, scales, out, (cudaStream_t)stream), "fp4 launch");
  return CSA_OK;
}

int csa_fp4_e8m0_roundtrip(const uint16_t* in, int64_t n_blocks, uint8_t* codes, uint8_t* scales, uint16_t* out,
                           csa_stream_t stream) {
  if (n_blocks < 0 || (n_blocks > 0 && (!in || !scales || !out))) return fail(CSA_ERR_ARG, "bad arguments");
  if (n_blocks == 0) return CSA_OK;  // nothing to do, nothing enqueued
  CSA_CUDA(csa::launch_fp4_e8m0_roundtrip(in, n_blocks, codes, scales, out, (cudaStream_t)stream), "fp4 launch");
  return CSA_OK;
}

}  // extern "C"
