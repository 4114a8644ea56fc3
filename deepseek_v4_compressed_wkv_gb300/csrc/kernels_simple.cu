// Kernels of the compressor other than the fused tensor-core prefill: weight re-layout,
// the decode path (projection of one token per sequence into its state slot, then the
// pool + epilogue of the sequences whose group completed), state maintenance, the
// standalone fp4 round trip, and the CUDA-core prefill used for shapes the tensor-core
// kernel does not take.
#include "csa_internal.cuh"
#include "kernels.h"

namespace csa {

// ---------------------------------------------------------------------------------------
// Weight re-layout: logical wkv/wgate [C][dim] -> packed f32 [2C][dim] and three bf16
// planes whose sum is exactly the f32 weight (each plane takes the next 8 significant bits:
// w - p0 and w - p0 - p1 are exact in f32, and the last remainder fits a bf16), in the tiled
// layout of plane_tile_elem (only where the tensor-core kernels can run: 128-row packed tiles
// and dim a multiple of 32).
__global__ void pack_weights_kernel(const float* __restrict__ wkv, const float* __restrict__ wgate, Packing pk,
                                    int overlap, int dim, float* __restrict__ w_packed,
                                    __nv_bfloat16* __restrict__ planes) {
  const bool tiled = pk.tw == kPlaneTileRows && dim % kPlaneTileK == 0;
  const int nkb = dim / kPlaneTileK;
  const int pr = blockIdx.y;  // packed row
  const int tile = pr / pk.tw, within = pr % pk.tw;
  const int kind = within / pk.ft, f = tile * pk.ft + within % pk.ft;
  const float* src;
  if (overlap)
    src = (kind == KV_A || kind == KV_B) ? wkv : wgate;
  else
    src = kind == KV ? wkv : wgate;
  const int row = overlap ? ((kind == KV_B || kind == S_B) ? pk.H + f : f) : f;
  for (int k = blockIdx.x * blockDim.x + threadIdx.x; k < dim; k += gridDim.x * blockDim.x) {
    const float w = src ? src[(size_t)row * dim + k] : 0.0f;
    const __nv_bfloat16 p0 = __float2bfloat16_rn(w);
    const float r1 = w - __bfloat162float(p0);
    const __nv_bfloat16 p1 = __float2bfloat16_rn(r1);
    const float r2 = r1 - __bfloat162float(p1);
    const size_t o = (size_t)pr * dim + k;
    w_packed[o] = w;
    if (tiled) {
      planes[plane_tile_elem(nkb, pr, k, 0)] = p0;
      planes[plane_tile_elem(nkb, pr, k, 1)] = p1;
      planes[plane_tile_elem(nkb, pr, k, 2)] = __float2bfloat16_rn(r2);
    }
  }
}

// Gate positional bias: logical ape [ratio][C] (the gate's columns, branch A then B) -> packed
// [ratio][2C] with the bias at the score columns and zero at the kv columns.
__global__ void pack_ape_kernel(const float* __restrict__ src, Packing pk, int overlap, int ratio,
                                float* __restrict__ dst) {
  const int ncol = pk.cols(), C = (1 + overlap) * pk.H;
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < ratio * ncol; i += gridDim.x * blockDim.x) {
    const int r = i / ncol, pc = i % ncol;
    const int within = pc % pk.tw, kind = within / pk.ft, f = (pc / pk.tw) * pk.ft + within % pk.ft;
    float v = 0.0f;
    if (kind >= pk.nk / 2) v = src[(size_t)r * C + ((overlap && kind == S_B) ? pk.H + f : f)];
    dst[i] = v;
  }
}

// ---------------------------------------------------------------------------------------
// CUDA-core projection: out[m][n] = sum_k x[m][k] * w[n][k], f32 accumulation in k order.
// Rows go to out + m*ncol (prefill) or, for decode, to the state slot of sequence m.
constexpr int GM = 64, GN = 64, GK = 16;

struct RowMap {
  int mode;  // 0: dense rows; 1: decode state slots
  const int32_t* start_pos;
  int slots, ratio, overlap;
  const float* ape;  // packed gate positional bias [ratio][2C], or null
  int N, p0;         // dense rows: row m is token m % N of its sequence, at position p0 + m % N
  long long extent;  // elements of the destination (checked by the bounds-checked build)
  int* flag;
  // position of the token of row m (for the bias)
  __device__ long long pos(int m) const { return mode == 0 ? (long long)p0 + m % N : (long long)max(start_pos[m], 0); }
  __device__ size_t row(int m, int ncol) const {
    if (mode == 0) return (size_t)m * ncol;
    const int slot = state_slot(max(start_pos[m], 0), ratio, overlap);
    return ((size_t)m * slots + slot) * ncol;
  }
};

__global__ __launch_bounds__(256) void gemm_ffma_kernel(const uint16_t* __restrict__ x, const float* __restrict__ w,
                                                        int M, int ncol, int K, float* __restrict__ out, RowMap map) {
  __shared__ float As[GK][GM + 4];
  __shared__ float Bs[GK][GN + 4];
  const int tx = threadIdx.x % 16, ty = threadIdx.x / 16;
  const int m0 = blockIdx.y * GM, n0 = blockIdx.x * GN;
  float acc[4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = 0.0f;
  for (int k0 = 0; k0 < K; k0 += GK) {
    for (int i = threadIdx.x; i < GM * GK; i += 256) {
      const int r = i / GK, kk = i % GK, m = m0 + r;
      As[kk][r] = m < M ? __uint_as_float((uint32_t)x[(size_t)m * K + k0 + kk] << 16) : 0.0f;
    }
    for (int i = threadIdx.x; i < GN * GK; i += 256) {
      const int r = i / GK, kk = i % GK, n = n0 + r;
      Bs[kk][r] = n < ncol ? w[(size_t)n * K + k0 + kk] : 0.0f;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < GK; ++kk) {
      float a[4], b[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] = As[kk][ty * 4 + i];
#pragma unroll
      for (int j = 0; j < 4; ++j) b[j] = Bs[kk][tx * 4 + j];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int m = m0 + ty * 4 + i;
    if (m >= M) continue;
    float* dst = out + map.row(m, ncol);
    const float* ab = map.ape ? map.ape + (size_t)(map.pos(m) % map.ratio) * ncol : nullptr;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int n = n0 + tx * 4 + j;
      // wgate(x) + bias at the score columns ("Compressed Sparse Attention": positional bias);
      // the packed bias is zero at the kv columns, where nothing is added
      if (n < ncol && in_bounds((long long)((dst - out) + n), map.extent, map.flag))
        dst[n] = (ab && ab[n] != 0.0f) ? acc[i][j] + ab[n] : acc[i][j];
    }
  }
}

// ---------------------------------------------------------------------------------------
// Softmax pool of one lane's 16 features over a candidate list ("Pool token pairs":
// (kv * score.softmax(dim)).sum(dim)): max, then exp(s - max) sums, then num / den.
template <class Cand>
__device__ __forceinline__ void pool16(int ncand, Cand cand, float out[16]) {
  float m[16], den[16], num[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    m[i] = -INFINITY;
    den[i] = 0.0f;
    num[i] = 0.0f;
  }
  for (int c = 0; c < ncand; ++c) {
    const float* kvp;
    const float* sp;
    if (!cand(c, kvp, sp)) continue;  // padded candidate: weight 0
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const float4 s4 = *reinterpret_cast<const float4*>(sp + 4 * q);
      m[4 * q] = fmaxf(m[4 * q], s4.x);
      m[4 * q + 1] = fmaxf(m[4 * q + 1], s4.y);
      m[4 * q + 2] = fmaxf(m[4 * q + 2], s4.z);
      m[4 * q + 3] = fmaxf(m[4 * q + 3], s4.w);
    }
  }
  for (int c = 0; c < ncand; ++c) {
    const float* kvp;
    const float* sp;
    if (!cand(c, kvp, sp)) continue;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const float4 s4 = *reinterpret_cast<const float4*>(sp + 4 * q);
      const float4 k4 = *reinterpret_cast<const float4*>(kvp + 4 * q);
      const float s[4] = {s4.x, s4.y, s4.z, s4.w}, k[4] = {k4.x, k4.y, k4.z, k4.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float ex = expf(s[e] - m[4 * q + e]);
        den[4 * q + e] += ex;
        num[4 * q + e] = fmaf(ex, k[e], num[4 * q + e]);
      }
    }
  }
#pragma unroll
  for (int i = 0; i < 16; ++i) out[i] = __fdiv_rn(num[i], den[i]);
}

// Prefill pool + epilogue from the projection scratch, one warp per entry (b, j): entry j of
// the call is absolute group g0 + j; a candidate token before the call's first position p0
// (a chunk) is read from its state slot, which prefill_state_kernel rewrites only after this
// kernel.
__global__ __launch_bounds__(128) void prefill_pool_kernel(const float* __restrict__ proj, int B, int N, Chunk ck,
                                                           int ratio, int overlap, Packing pk,
                                                           const float* __restrict__ state, int slots,
                                                           int slot_offset, EpiParams ep, csa_out out, int* flag) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = ck.G;
  const long long e = (long long)blockIdx.x * 4 + warp;
  if (e >= (long long)B * G) return;
  const int b = (int)(e / G), j = (int)(e % G);
  const long long g = (long long)ck.g0 + j;
  const int ncol = pk.cols();
  const float* seq = proj + (size_t)b * N * ncol;
  const float* st = state + (size_t)(slot_offset + b) * slots * ncol;
  auto row_of = [&](long long p) {  // projected row of the token at position p
    return p >= ck.p0 ? seq + (size_t)(p - ck.p0) * ncol : st + (size_t)state_slot(p, ratio, overlap) * ncol;
  };
  const int f0 = min(lane, (pk.H >> 4) - 1) * 16;
  float v[16];
  if (overlap) {
    pool16(8, [&](int c, const float*& kvp, const float*& sp) {
      if (c < 4) {
        if (g == 0) return false;
        const float* row = row_of(4 * g - 4 + c);
        kvp = row + pk.col(KV_B, f0);
        sp = row + pk.col(S_B, f0);
      } else {
        const float* row = row_of(4 * g + c - 4);
        kvp = row + pk.col(KV_A, f0);
        sp = row + pk.col(S_A, f0);
      }
      return true;
    }, v);
  } else {
    pool16(ratio, [&](int c, const float*& kvp, const float*& sp) {
      const float* row = row_of(ratio * g + c);
      kvp = row + pk.col(KV, f0);
      sp = row + pk.col(S, f0);
      return true;
    }, v);
  }
  const size_t H = pk.H;
  const size_t o = (size_t)ck.row(b, j);
  if (!in_bounds((long long)o, (long long)B * ck.bstride, flag)) return;  // the same for the whole warp
  entry_epilogue(v, lane, (long long)ratio * g, ep, out.latent + o * H, out.codes ? out.codes + o * (H / 2) : nullptr,
                 out.scales ? out.scales + o * (H / fp4_scale_block(ep.fp4)) : nullptr,
                 out.prequant ? out.prequant + o * H : nullptr);
}

__device__ __forceinline__ float padded_value(const Packing& pk, int col) {
  const int kind = (col % pk.tw) / pk.ft;
  return kind < pk.nk / 2 ? 0.0f : -INFINITY;  // kv kinds first, score kinds second
}

// Prefill state update ("Pool token pairs": the trailing partial group waits in the state;
// at ratio 4 overlapped also the last complete group, whose branch B the next entry pools):
// the call's tokens of those groups go to their slots (a chunk's earlier tokens are there
// already).
__global__ void prefill_state_kernel(const float* __restrict__ proj, int N, Chunk ck, int ratio, int overlap,
                                     Packing pk, float* __restrict__ state, int slots, int slot_offset,
                                     long long state_elems, int* flag) {
  const int b = blockIdx.x;
  const int ncol = pk.cols();
  const float* seq = proj + (size_t)b * N * ncol;
  float* st = state + (size_t)(slot_offset + b) * slots * ncol;
  const long long p1 = (long long)ck.p0 + N;
  const long long keep = max((long long)ck.p0, ((long long)ck.gend - overlap) * ratio);
  for (long long p = keep; p < p1; ++p) {
    const float* src = seq + (size_t)(p - ck.p0) * ncol;
    float* dst = st + (size_t)state_slot(p, ratio, overlap) * ncol;
    if (!in_bounds((long long)((dst - state) + ncol - 1), state_elems, flag)) continue;
    for (int c = threadIdx.x; c < ncol; c += blockDim.x) dst[c] = src[c];
  }
  if (overlap && ck.gend == 0 && in_bounds((long long)((st - state) + 8 * ncol - 1), state_elems, flag))
    for (int c = threadIdx.x; c < 4 * ncol; c += blockDim.x) st[(size_t)4 * ncol + c] = padded_value(pk, c % ncol);
}

// Decode: pool + epilogue for the sequences whose token completed a group; one warp per
// sequence.  The projection of this step's tokens is already in their state slots.  emitted may
// be null (the caller learns the emissions on the host).
__global__ __launch_bounds__(128) void decode_emit_kernel(const int32_t* __restrict__ start_pos, int B, int ratio,
                                                          int overlap, Packing pk, float* __restrict__ state, int slots,
                                                          EpiParams ep, csa_out out, uint8_t* __restrict__ emitted,
                                                          int* __restrict__ flag) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int b = blockIdx.x * 4 + warp;
  if (b >= B) return;
  const int ncol = pk.cols();
  const int p = start_pos[b];
  float* st = state + (size_t)b * slots * ncol;
  if (p < 0) {
    if (lane == 0) {
      if (emitted) emitted[b] = 0;
      atomicOr(flag, 1);
    }
    return;
  }
  if (p == 0 && overlap) {  // restart: the previous group's branch is the padded one
    for (int c = lane; c < 4 * ncol; c += 32) st[(size_t)4 * ncol + c] = padded_value(pk, c % ncol);
  }
  const bool emit = (p + 1) % ratio == 0;
  const long long pos = (long long)p + 1 - ratio;
  const bool pos_ok = ep.rope_dim == 0 || pos < ep.max_pos;
  if (lane == 0) {
    if (emitted) emitted[b] = (emit && pos_ok) ? 1 : 0;
    if (emit && !pos_ok) atomicOr(flag, 2);
  }
  if (!emit || !pos_ok) return;
  const int f0 = min(lane, (pk.H >> 4) - 1) * 16;
  float v[16];
  if (overlap) {
    const int q = (p >> 2) & 1;
    pool16(8, [&](int c, const float*& kvp, const float*& sp) {
      const float* row = st + (size_t)(c < 4 ? 4 * (1 - q) + c : 4 * q + c - 4) * ncol;
      kvp = row + pk.col(c < 4 ? KV_B : KV_A, f0);
      sp = row + pk.col(c < 4 ? S_B : S_A, f0);
      return true;
    }, v);
  } else {
    pool16(ratio, [&](int c, const float*& kvp, const float*& sp) {
      const float* row = st + (size_t)c * ncol;
      kvp = row + pk.col(KV, f0);
      sp = row + pk.col(S, f0);
      return true;
    }, v);
  }
  const size_t H = pk.H;
  entry_epilogue(v, lane, pos, ep, out.latent + b * H, out.codes ? out.codes + b * (H / 2) : nullptr,
                 out.scales ? out.scales + b * (H / fp4_scale_block(ep.fp4)) : nullptr,
                 out.prequant ? out.prequant + b * H : nullptr);
}

__global__ void state_reset_kernel(float* __restrict__ state, Packing pk, size_t first, size_t count) {
  const int ncol = pk.cols();
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < count; i += (size_t)gridDim.x * blockDim.x)
    state[first + i] = padded_value(pk, (int)((first + i) % ncol));
}

// Packed state rows -> logical kv / score rows (branch A then B when overlapped).
__global__ void state_export_kernel(const float* __restrict__ state, Packing pk, int overlap, size_t rows,
                                    float* __restrict__ kv, float* __restrict__ score) {
  const int W = (1 + overlap) * pk.H, ncol = pk.cols();
  const size_t n = rows * W;
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x) {
    const size_t r = i / W;
    const int c = (int)(i % W);
    const int br = c / pk.H, f = c % pk.H;
    const float* row = state + r * ncol;
    kv[i] = row[pk.col(overlap ? (br ? KV_B : KV_A) : KV, f)];
    score[i] = row[pk.col(overlap ? (br ? S_B : S_A) : S, f)];
  }
}

// The inverse of state_export_kernel: the logical arrays written back into the packed state.
__global__ void state_import_kernel(float* __restrict__ state, Packing pk, int overlap, size_t rows,
                                    const float* __restrict__ kv, const float* __restrict__ score) {
  const int W = (1 + overlap) * pk.H, ncol = pk.cols();
  const size_t n = rows * W;
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x) {
    const size_t r = i / W;
    const int c = (int)(i % W);
    const int br = c / pk.H, f = c % pk.H;
    float* row = state + r * ncol;
    row[pk.col(overlap ? (br ? KV_B : KV_A) : KV, f)] = kv[i];
    row[pk.col(overlap ? (br ? S_B : S_A) : S, f)] = score[i];
  }
}

__global__ void fp4_roundtrip_kernel(const uint16_t* __restrict__ in, long long nb, uint8_t* __restrict__ codes,
                                     uint8_t* __restrict__ scales, uint16_t* __restrict__ out) {
  for (long long b = blockIdx.x * (long long)blockDim.x + threadIdx.x; b < nb; b += (long long)gridDim.x * blockDim.x) {
    float y[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) y[i] = __uint_as_float((uint32_t)in[b * 16 + i] << 16);
    uint8_t cd[8], sb;
    fp4_block16(y, cd, &sb);
    scales[b] = sb;
    if (codes)
#pragma unroll
      for (int i = 0; i < 8; ++i) codes[b * 8 + i] = cd[i];
#pragma unroll
    for (int i = 0; i < 16; ++i) out[b * 16 + i] = bf16_bits(y[i]);
  }
}

// The indexer's fp4 round trip alone: one thread per block of 32 values.
__global__ void fp4_e8m0_roundtrip_kernel(const uint16_t* __restrict__ in, long long nb, uint8_t* __restrict__ codes,
                                          uint8_t* __restrict__ scales, uint16_t* __restrict__ out) {
  for (long long b = blockIdx.x * (long long)blockDim.x + threadIdx.x; b < nb; b += (long long)gridDim.x * blockDim.x) {
    float y[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) y[i] = __uint_as_float((uint32_t)in[b * 32 + i] << 16);
    uint8_t cd[16], sb;
    fp4_block32_e8m0(y, cd, &sb);
    scales[b] = sb;
    if (codes)
#pragma unroll
      for (int i = 0; i < 16; ++i) codes[b * 16 + i] = cd[i];
#pragma unroll
    for (int i = 0; i < 32; ++i) out[b * 32 + i] = bf16_bits(y[i]);
  }
}

// ---------------------------------------------------------------------------------------
// Host-side launchers.

static int grid_cap(size_t n, int per) {
  size_t g = (n + per - 1) / per;
  return (int)(g > 152 * 32 ? 152 * 32 : (g < 1 ? 1 : g));
}

cudaError_t launch_pack_weights(const csa_compressor* c, const float* wkv, const float* wgate, cudaStream_t s) {
  dim3 grid((c->dim + 255) / 256, c->pk.cols());
  pack_weights_kernel<<<grid, 256, 0, s>>>(wkv, wgate, c->pk, c->overlap, c->dim, c->w_packed, c->w_planes);
  return cudaGetLastError();
}

cudaError_t launch_pack_ape(const csa_compressor* c, const float* ape, cudaStream_t s) {
  const int n = c->ratio * c->pk.cols();
  pack_ape_kernel<<<grid_cap((size_t)n, 256), 256, 0, s>>>(ape, c->pk, c->overlap, c->ratio, c->ape);
  return cudaGetLastError();
}

cudaError_t launch_projection_ffma(const csa_compressor* c, const uint16_t* x, int M, float* out, int mode,
                                   const int32_t* start_pos, int N, int p0, cudaStream_t s) {
  const long long extent = mode == 0 ? (long long)M * c->pk.cols() : (long long)c->opt.max_batch * c->slots * c->pk.cols();
  RowMap map{mode, start_pos, c->slots, c->ratio, c->overlap, c->ape_set ? c->ape : nullptr, N, p0, extent, c->dev_flag};
  const int ncol = c->pk.cols();
  dim3 grid((ncol + GN - 1) / GN, (M + GM - 1) / GM);
  gemm_ffma_kernel<<<grid, 256, 0, s>>>(x, c->w_packed, M, ncol, c->dim, out, map);
  return cudaGetLastError();
}

EpiParams epi_params(const csa_compressor* c) {
  EpiParams ep;
  ep.gain = c->gain;
  ep.rope_cos = c->rope_cos;
  ep.rope_sin = c->rope_sin;
  ep.H = c->H;
  ep.rope_dim = c->opt.rope_dim;
  ep.fp4 = c->opt.fp4;
  ep.max_pos = c->opt.max_pos;
  ep.eps = c->opt.eps;
  return ep;
}

cudaError_t launch_prefill_pool(const csa_compressor* c, const float* proj, int B, int N, int slot_offset,
                                const Chunk& ck, const csa_out& out, cudaStream_t s) {
  const long long E = (long long)B * ck.G;
  if (E > 0)
    prefill_pool_kernel<<<(unsigned)((E + 3) / 4), 128, 0, s>>>(proj, B, N, ck, c->ratio, c->overlap, c->pk, c->state,
                                                              c->slots, slot_offset, epi_params(c), out, c->dev_flag);
  return cudaGetLastError();
}

cudaError_t launch_prefill_state(const csa_compressor* c, const float* proj, int B, int N, int slot_offset,
                                 const Chunk& ck, cudaStream_t s) {
  prefill_state_kernel<<<B, 256, 0, s>>>(proj, N, ck, c->ratio, c->overlap, c->pk, c->state, c->slots, slot_offset,
                                         (long long)c->opt.max_batch * c->slots * c->pk.cols(), c->dev_flag);
  return cudaGetLastError();
}

cudaError_t launch_decode_emit(const csa_compressor* c, const int32_t* start_pos, int B, const csa_out& out,
                               uint8_t* emitted, cudaStream_t s) {
  decode_emit_kernel<<<(B + 3) / 4, 128, 0, s>>>(start_pos, B, c->ratio, c->overlap, c->pk, c->state, c->slots,
                                                 epi_params(c), out, emitted, c->dev_flag);
  return cudaGetLastError();
}

cudaError_t launch_state_reset(const csa_compressor* c, int slot_begin, int count, cudaStream_t s) {
  const size_t row = (size_t)c->slots * c->pk.cols();
  const size_t n = row * count;
  if (n) state_reset_kernel<<<grid_cap(n, 256), 256, 0, s>>>(c->state, c->pk, row * slot_begin, n);
  return cudaGetLastError();
}

cudaError_t launch_state_export(const csa_compressor* c, float* kv, float* score, cudaStream_t s) {
  const size_t rows = (size_t)c->opt.max_batch * c->slots;
  state_export_kernel<<<grid_cap(rows * c->width, 256), 256, 0, s>>>(c->state, c->pk, c->overlap, rows, kv, score);
  return cudaGetLastError();
}

cudaError_t launch_state_import(const csa_compressor* c, const float* kv, const float* score, cudaStream_t s) {
  const size_t rows = (size_t)c->opt.max_batch * c->slots;
  state_import_kernel<<<grid_cap(rows * c->width, 256), 256, 0, s>>>(c->state, c->pk, c->overlap, rows, kv, score);
  return cudaGetLastError();
}

cudaError_t launch_fp4_roundtrip(const uint16_t* in, long long nb, uint8_t* codes, uint8_t* scales, uint16_t* out,
                                 cudaStream_t s) {
  if (nb > 0) fp4_roundtrip_kernel<<<grid_cap((size_t)nb, 256), 256, 0, s>>>(in, nb, codes, scales, out);
  return cudaGetLastError();
}

cudaError_t launch_fp4_e8m0_roundtrip(const uint16_t* in, long long nb, uint8_t* codes, uint8_t* scales,
                                      uint16_t* out, cudaStream_t s) {
  if (nb > 0) fp4_e8m0_roundtrip_kernel<<<grid_cap((size_t)nb, 128), 128, 0, s>>>(in, nb, codes, scales, out);
  return cudaGetLastError();
}

}  // namespace csa
