// Internal declarations of the CSA KV compressor library: the handle, the packed weight
// layout, and the device routines shared by the kernels (bf16 rounding, the fp4 round
// trip, the per-entry epilogue).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "csa.h"  // include/ is on the include path (see build.py)

namespace csa {

// ---------------------------------------------------------------------------------------
// Packed column order.
//
// The projection's 2C output columns (kv and score; at ratio 4 overlapped each has branch
// A and branch B) are stored tile by tile: a tile holds `nk` kinds x `ft` features, kind
// major.  Kinds: overlapped (kvA, kvB, sA, sB); otherwise (kv, s).  Tile t covers features
// [t*ft, (t+1)*ft).  All kinds of a feature therefore sit in the same tile, which is what a
// GEMM tile needs to pool without leaving the chip.  The same order is used for the packed
// f32 weights, the bf16 weight planes, the projection scratch and the state rows.
struct Packing {
  int H, nk, ft, tw, ntiles;  // tw = nk * ft columns per tile
  __host__ __device__ int col(int kind, int f) const { return (f / ft) * tw + kind * ft + (f % ft); }
  __host__ __device__ int cols() const { return ntiles * tw; }
};

enum Kind { KV_A = 0, KV_B = 1, S_A = 2, S_B = 3 };  // overlapped
enum KindN { KV = 0, S = 1 };                        // non-overlapped

inline __host__ __device__ Packing make_packing(int H, int overlap) {
  Packing p;
  p.H = H;
  p.nk = overlap ? 4 : 2;
  p.ft = 128 / p.nk;
  if (p.ft > H) p.ft = H;
  p.tw = p.nk * p.ft;
  p.ntiles = H / p.ft;
  return p;
}

// Tiled layout of the three bf16 weight planes used by the tensor-core kernels.  For packed
// tile t (128 rows) and K block kb (32 columns) the three planes' 128 x 32 blocks follow each
// other (24 KB, plane-major), each stored as the image a 64-byte-swizzled shared-memory tile
// has: row r at byte 64 r, its 16-byte chunk c at chunk position c ^ ((r >> 1) & 3).  One
// contiguous copy of 24 KB then fills a pipeline stage with operands the MMA reads directly.
constexpr int kPlaneTileRows = 128, kPlaneTileK = 32;
__host__ __device__ inline size_t plane_tile_elem(int nkb, int pr, int k, int p) {
  const int t = pr / kPlaneTileRows, r = pr % kPlaneTileRows, kb = k / kPlaneTileK, kk = k % kPlaneTileK;
  const int c = kk >> 3, e = kk & 7;
  const size_t block = ((size_t)t * nkb + kb) * 3 + p;
  return block * (kPlaneTileRows * kPlaneTileK) + r * kPlaneTileK + ((c ^ ((r >> 1) & 3)) << 3) + e;
}
// The stage of (tile t, K block kb): 3 planes x 128 x 32 bf16.
__host__ __device__ inline size_t plane_stage_elem(int nkb, int t, int kb) {
  return ((size_t)t * nkb + kb) * 3 * (kPlaneTileRows * kPlaneTileK);
}

// State slot of the token at position p of a sequence ("Pool token pairs", decode branch:
// p % ratio; ratio 4 overlapped: group p / 4 lives in parity (p / 4) % 2, slot p % 4 of it).
__host__ __device__ inline int state_slot(long long p, int ratio, int overlap) {
  return overlap ? (int)(((p >> 2) & 1) * 4 + (p & 3)) : (int)(p % ratio);
}

// Geometry of one prefill call over tokens [p0, p0 + N) of each sequence (all sequences at the
// same position).  p0 = 0 is the whole-sequence prefill of the pages; p0 > 0 a chunk that
// continues sequences whose earlier tokens are in the state (the same rule as decode, token by
// token).  The kernels index tokens from the start of the open group: virtual token v is
// position p0 - a + v, so v < a are the open group's earlier tokens, read from the state.
struct Chunk {
  int p0;              // position of the call's first token
  int a;               // p0 % ratio
  int g0;              // p0 / ratio: absolute index of the first group the call can complete
  int G;               // groups completing in the call: (p0 + N) / ratio - g0
  int gend;            // (p0 + N) / ratio: the group left unfinished
  long long bstride;   // output rows per sequence
  long long row0;      // output row of the call's first entry
  // entry j of sequence b goes to output row b * bstride + row0 + j
  __host__ __device__ long long row(int b, int j) const { return (long long)b * bstride + row0 + j; }
};

// Entries to out [B][G][..] (set bstride and row0 for other layouts).
inline Chunk make_chunk(int p0, int N, int ratio) {
  Chunk k;
  k.p0 = p0;
  k.a = p0 % ratio;
  k.g0 = p0 / ratio;
  k.gend = (int)(((long long)p0 + N) / ratio);
  k.G = k.gend - k.g0;
  k.bstride = k.G;
  k.row0 = 0;
  return k;
}

// The earlier candidates a chunk's first group pools besides its new tokens (the open group's
// tokens before p0 and, overlapped, branch B of the previous group; overlapped, the second
// group's branch B of those same tokens) are reduced by chunk_carry_kernel to running softmax
// values (max, denominator, numerator) per feature, [B][1 + overlap][3][H] f32, before the
// projection kernel overwrites any state slot.
inline bool chunk_needs_carry(const Chunk& k, int overlap) { return k.G > 0 && (k.a > 0 || (overlap && k.g0 > 0)); }

// SMs of the current device, the one a launch goes to (152 on a GB300, used if the query fails).
inline int current_sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
      n <= 0)
    return 152;
  return n;
}

// Kernel-side view of the epilogue parameters.
struct EpiParams {
  const float* gain;      // [H]
  const float* rope_cos;  // [max_pos][rope_dim/2]
  const float* rope_sin;
  int H, rope_dim, fp4, max_pos;  // fp4: 0 off, 1 e4m3 scale per 16, 2 power-of-two scale per 32
  float eps;
};

// ---------------------------------------------------------------------------------------
// Index checks of the bounds-checked build (compiled with -DCSA_DEBUG_BOUNDS): a store whose
// element index falls outside its buffer's extent [0, n) is skipped and raises bit 8 of the
// handle's device flag, instead of writing out of bounds.  Compiled out otherwise.
#ifdef CSA_DEBUG_BOUNDS
__device__ __forceinline__ bool in_bounds(long long i, long long n, int* flag) {
  if (i >= 0 && i < n) return true;
  atomicOr(flag, 8);
  return false;
}
#else
__device__ __forceinline__ bool in_bounds(long long, long long, int*) { return true; }
#endif

// ---------------------------------------------------------------------------------------
// Device number formats.

__device__ __forceinline__ float bf16_round(float v) { return __bfloat162float(__float2bfloat16_rn(v)); }

__device__ __forceinline__ uint16_t bf16_bits(float v) {
  __nv_bfloat16 b = __float2bfloat16_rn(v);
  return *reinterpret_cast<uint16_t*>(&b);
}

// e4m3 bit pattern -> value (exact).  1 sign, 4 exponent bits (bias 7), 3 mantissa bits.
__device__ __forceinline__ float e4m3_value(uint32_t b) {
  uint32_t e = (b >> 3) & 15u, m = b & 7u;
  float mag = e == 0 ? (float)m * 0.001953125f /* 2^-9 */ : __uint_as_float(((e + 120u) << 23) | (m << 20));
  return (b & 0x80u) ? -mag : mag;
}

// Two float32 -> two e2m1 codes packed in one byte, `lo` in bits 0..3, round to nearest
// even, saturating to +-6 (PTX cvt with .satfinite; the first source goes to the upper
// nibble).
__device__ __forceinline__ uint32_t e2m1x2(float lo, float hi) {
  uint16_t r;
  asm("{\n\t.reg .b8 t;\n\tcvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n\tcvt.u16.u8 %0, t;\n\t}"
      : "=h"(r)
      : "f"(hi), "f"(lo));
  return r;
}

__device__ __forceinline__ float e2m1_value(uint32_t code) {
  // magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6 by code: exponent field e = code>>1, mantissa m
  uint32_t e = (code >> 1) & 3u, m = code & 1u;
  float mag = e == 0 ? 0.5f * (float)m : (1.0f + 0.5f * (float)m) * (float)(1u << (e - 1));
  return (code & 8u) ? -mag : mag;
}

// fp4 round trip of one block of 16 bf16 values held by one thread ("Module compress",
// fp4_quant_e4m3_inplace): amax floored at 6*2^-9, scale = e4m3(amax / 6) with the
// division in IEEE f32, values divided by the scale (IEEE f32) to e2m1, dequantised
// exactly and rounded to bf16.  y[] holds bf16 values (as float); replaced in place by
// the dequantised values.
__device__ __forceinline__ void fp4_block16(float y[16], uint8_t codes[8], uint8_t* scale_bits) {
  float amax = 0.0f;
#pragma unroll
  for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(y[i]));
  const float sq = __fdiv_rn(fmaxf(amax, 0.01171875f /* 6 * 2^-9 */), 6.0f);
  const __nv_fp8_storage_t sb = __nv_cvt_float_to_fp8(sq, __NV_SATFINITE, __NV_E4M3);
  const float s = e4m3_value(sb);
  *scale_bits = sb;
#pragma unroll
  for (int i = 0; i < 16; i += 2) {
    uint32_t c2 = e2m1x2(__fdiv_rn(y[i], s), __fdiv_rn(y[i + 1], s));
    codes[i / 2] = (uint8_t)c2;
    y[i] = bf16_round(e2m1_value(c2 & 15u) * s);
    y[i + 1] = bf16_round(e2m1_value(c2 >> 4) * s);
  }
}

// Power-of-two scale of the indexer's fp4 round trip ("Module compress", fp4_quant_e8m0_inplace):
// the smallest power of two >= max(amax, 6 * 2^-126) / 6, the division in IEEE f32.  The
// quotient is a normal float (>= 2^-126), so the ceiling is its exponent, plus one unless the
// mantissa is zero.  *byte receives the e8m0 encoding (the biased exponent, value 2^(byte-127)).
__device__ __forceinline__ float e8m0_scale(float amax, uint32_t* byte) {
  const float q = __fdiv_rn(fmaxf(amax, 6.0f * 1.17549435082228750797e-38f /* 6 * 2^-126 */), 6.0f);
  const uint32_t u = __float_as_uint(q);
  const uint32_t e = (u >> 23) + ((u & 0x7FFFFFu) != 0u ? 1u : 0u);
  *byte = e;
  return __uint_as_float(e << 23);
}

// fp4 round trip of one block of 32 bf16 values with a power-of-two scale ("Module compress",
// fp4_quant_e8m0_inplace, FP4_BLOCK = 32): values divided by the scale (exact) to e2m1,
// dequantised and rounded to bf16 in place.
__device__ __forceinline__ void fp4_block32_e8m0(float y[32], uint8_t codes[16], uint8_t* scale_byte) {
  float amax = 0.0f;
#pragma unroll
  for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(y[i]));
  uint32_t sb;
  const float s = e8m0_scale(amax, &sb);
  *scale_byte = (uint8_t)sb;
#pragma unroll
  for (int i = 0; i < 32; i += 2) {
    const uint32_t c2 = e2m1x2(__fdiv_rn(y[i], s), __fdiv_rn(y[i + 1], s));
    codes[i / 2] = (uint8_t)c2;
    y[i] = bf16_round(e2m1_value(c2 & 15u) * s);
    y[i + 1] = bf16_round(e2m1_value(c2 >> 4) * s);
  }
}

// Values per fp4 scale of the compressor's output: 16 (e4m3 scales, the latent) or 32
// (power-of-two scales, the indexer's keys).
__host__ __device__ inline int fp4_scale_block(int fp4) { return fp4 == 2 ? 32 : 16; }

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Epilogue of one block of 16 features f0..f0+15 of an entry, after the RMSNorm factor `inv`
// is known: v[] holds the bf16-rounded pooled values.  RMSNorm in f32 with the f32 gain and one
// bf16 rounding, YaRN RoPE on the trailing rope_dim features (adjacent pairs, angle pos * f_i
// from the host-built table), then the fp4 round trip; stores the block's outputs.  gain points
// at the gain of feature f0; cs / sn at the table row of the entry's position (global or shared
// memory).
__device__ __forceinline__ void entry_epilogue_block(float v[16], int f0, float inv, const float* gain,
                                                     const float* cs, const float* sn, const EpiParams& ep,
                                                     uint16_t* latent, uint8_t* codes, uint8_t* scales,
                                                     uint16_t* prequant, unsigned lanes) {
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = bf16_round(v[i] * inv * gain[i]);
  const int r0 = ep.H - ep.rope_dim;
  if (ep.rope_dim > 0 && f0 + 16 > r0) {
#pragma unroll
    for (int i = 0; i < 16; i += 2) {
      const int f = f0 + i;
      if (f >= r0) {
        const int k = (f - r0) >> 1;
        const float c = cs[k], s = sn[k];
        const float a = v[i], b = v[i + 1];
        v[i] = bf16_round(a * c - b * s);
        v[i + 1] = bf16_round(a * s + b * c);
      }
    }
  }
  if (prequant) {
    uint32_t w[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) w[i] = (uint32_t)bf16_bits(v[2 * i]) | ((uint32_t)bf16_bits(v[2 * i + 1]) << 16);
    uint4* dst = reinterpret_cast<uint4*>(prequant + f0);
    dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
    dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
  }
  if (ep.fp4 == 2) {  // power-of-two scale over 32 features: this lane and its neighbour
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(v[i]));
    amax = fmaxf(amax, __shfl_xor_sync(lanes, amax, 1));
    uint32_t sb;
    const float s = e8m0_scale(amax, &sb);
    uint8_t cd[8];
#pragma unroll
    for (int i = 0; i < 16; i += 2) {
      const uint32_t c2 = e2m1x2(__fdiv_rn(v[i], s), __fdiv_rn(v[i + 1], s));
      cd[i / 2] = (uint8_t)c2;
      v[i] = bf16_round(e2m1_value(c2 & 15u) * s);
      v[i + 1] = bf16_round(e2m1_value(c2 >> 4) * s);
    }
    if (codes) {
      uint2 pk;
      pk.x = cd[0] | (cd[1] << 8) | (cd[2] << 16) | ((uint32_t)cd[3] << 24);
      pk.y = cd[4] | (cd[5] << 8) | (cd[6] << 16) | ((uint32_t)cd[7] << 24);
      *reinterpret_cast<uint2*>(codes + f0 / 2) = pk;
    }
    if (scales && (f0 & 31) == 0) scales[f0 >> 5] = (uint8_t)sb;
  } else if (ep.fp4) {
    uint8_t cd[8], sb;
    fp4_block16(v, cd, &sb);
    if (codes) {
      uint2 pk;
      pk.x = cd[0] | (cd[1] << 8) | (cd[2] << 16) | ((uint32_t)cd[3] << 24);
      pk.y = cd[4] | (cd[5] << 8) | (cd[6] << 16) | ((uint32_t)cd[7] << 24);
      *reinterpret_cast<uint2*>(codes + f0 / 2) = pk;
    }
    if (scales) scales[f0 >> 4] = sb;
  }
  uint32_t w[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) w[i] = (uint32_t)bf16_bits(v[2 * i]) | ((uint32_t)bf16_bits(v[2 * i + 1]) << 16);
  uint4* dst = reinterpret_cast<uint4*>(latent + f0);
  dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
  dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
}

// Epilogue of four adjacent features f..f+3 of entry row `e`, held by one thread, once the
// RMSNorm factor `inv` is known: v[] holds the bf16-rounded pooled values, gn[] the gain,
// rc/rs the RoPE cos/sin of the pairs (f, f+1) and (f+2, f+3) (used for pairs at or past
// H - rope_dim).  RMSNorm with one bf16 rounding, RoPE, then the fp4 round trip, whose block
// is four adjacent lanes (16 features, e4m3 scale) or eight (32 features, power-of-two scale)
// (all 32 lanes of the warp must call it; `act` is the same for the lanes of a block), and the
// stores.
__device__ __forceinline__ void entry_epilogue_quad(const float v[4], bool act, int f, int lane, float inv,
                                                   const float gn[4], const float rc[2], const float rs[2],
                                                   const EpiParams& ep, size_t e, const csa_out& out) {
  const size_t H = ep.H;
  float y[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) y[i] = bf16_round(v[i] * inv * gn[i]);
  if (act && ep.rope_dim > 0) {
    const int r0 = ep.H - ep.rope_dim;
#pragma unroll
    for (int u = 0; u < 2; ++u)
      if (f + 2 * u >= r0) {
        const float a = y[2 * u], b = y[2 * u + 1];
        y[2 * u] = bf16_round(a * rc[u] - b * rs[u]);
        y[2 * u + 1] = bf16_round(a * rs[u] + b * rc[u]);
      }
  }
  if (act && out.prequant)
    *reinterpret_cast<uint2*>(out.prequant + e * H + f) =
        make_uint2((uint32_t)bf16_bits(y[0]) | ((uint32_t)bf16_bits(y[1]) << 16),
                   (uint32_t)bf16_bits(y[2]) | ((uint32_t)bf16_bits(y[3]) << 16));
  if (ep.fp4) {
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 4; ++i) amax = fmaxf(amax, fabsf(y[i]));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
    uint32_t sb;
    float scl;
    if (ep.fp4 == 2) {  // power-of-two scale over 32 features: eight lanes
      amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 4));
      scl = e8m0_scale(amax, &sb);
    } else {  // e4m3 scale over 16 features: four lanes
      const float sq = __fdiv_rn(fmaxf(amax, 0.01171875f /* 6 * 2^-9 */), 6.0f);
      sb = __nv_cvt_float_to_fp8(sq, __NV_SATFINITE, __NV_E4M3);
      scl = e4m3_value(sb);
    }
    const uint32_t c0 = e2m1x2(__fdiv_rn(y[0], scl), __fdiv_rn(y[1], scl));  // element 2i in the low nibble
    const uint32_t c1 = e2m1x2(__fdiv_rn(y[2], scl), __fdiv_rn(y[3], scl));
    y[0] = bf16_round(e2m1_value(c0 & 15u) * scl);
    y[1] = bf16_round(e2m1_value(c0 >> 4) * scl);
    y[2] = bf16_round(e2m1_value(c1 & 15u) * scl);
    y[3] = bf16_round(e2m1_value(c1 >> 4) * scl);
    if (act && out.codes) *reinterpret_cast<uint16_t*>(out.codes + e * (H / 2) + f / 2) = (uint16_t)(c0 | (c1 << 8));
    const int blk = fp4_scale_block(ep.fp4);
    if (act && out.scales && (lane & (blk / 4 - 1)) == 0) out.scales[e * (H / blk) + f / blk] = (uint8_t)sb;
  }
  if (act)
    *reinterpret_cast<uint2*>(out.latent + e * H + f) =
        make_uint2((uint32_t)bf16_bits(y[0]) | ((uint32_t)bf16_bits(y[1]) << 16),
                   (uint32_t)bf16_bits(y[2]) | ((uint32_t)bf16_bits(y[3]) << 16));
}

// RMSNorm factor from the sum of squares of the bf16-rounded pooled values.
__device__ __forceinline__ float rms_inv(float ss, const EpiParams& ep) {
  return 1.0f / sqrtf(ss / (float)ep.H + ep.eps);
}

// Epilogue of one entry, one warp per entry: lane l (< H/16) holds pooled features
// 16l..16l+15 in v[].  bf16 round ("norm(kv.to(bf16))"), the sum of squares over the warp,
// then entry_epilogue_block.  All 32 lanes must call it (the RMSNorm sum is a warp
// reduction); lanes >= H/16 pass zeros and store nothing.
__device__ __forceinline__ void entry_epilogue(float v[16], int lane, long long pos, const EpiParams& ep,
                                               uint16_t* latent, uint8_t* codes, uint8_t* scales,
                                               uint16_t* prequant) {
  const int nl = ep.H >> 4;
  const bool act = lane < nl;
  float ss = 0.0f;
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    v[i] = act ? bf16_round(v[i]) : 0.0f;
    ss = fmaf(v[i], v[i], ss);
  }
  ss = warp_sum(ss);
  const float inv = rms_inv(ss, ep);
  if (!act) return;
  const int hr = ep.rope_dim >> 1;
  const unsigned lanes = nl >= 32 ? 0xffffffffu : (1u << nl) - 1u;  // the lanes that reach here
  entry_epilogue_block(v, lane * 16, inv, ep.gain + lane * 16, hr ? ep.rope_cos + pos * hr : nullptr,
                       hr ? ep.rope_sin + pos * hr : nullptr, ep, latent, codes, scales, prequant, lanes);
}

}  // namespace csa

// ---------------------------------------------------------------------------------------
// The handle (host side).
struct csa_compressor {
  int dim, H, ratio, overlap, width;  // width = (1 + overlap) * H rows per weight matrix
  csa_options opt;
  csa::Packing pk;
  int slots;        // state slots per sequence: ratio, or 8 (2 parities x 4) overlapped
  int device;
  bool weights_set;
  float* w_packed;  // [2C][dim] f32, packed column order
  __nv_bfloat16* w_planes;  // 3 bf16 split planes (w = p0 + p1 + p2), tiled (plane_tile_elem)
  float* gain;              // [H]
  float* ape;               // gate positional bias [ratio][2C] f32, packed order, zero at the kv
                            // columns (allocated by the first csa_compressor_set_gate_bias)
  bool ape_set;             // the bias is in use
  float* rope_cos;          // [max_pos][rope_dim/2]
  float* rope_sin;
  float* state;             // [max_batch][slots][2C] f32, packed column order
  int* dev_flag;            // device-side error flag
  float* scratch;           // projection scratch [rows][2C] f32 (grown on demand)
  size_t scratch_bytes;
  float* dec_part;          // decode split-K partial sums [slices][B][2C] (grown on demand)
  size_t dec_part_bytes;
  float* dec_acc;           // decode, non-overlapped: running softmax max / denominator / numerator
                            // of each sequence's open group [max_batch][3][H]
  int* dec_acc_pos;         //   position of the last token folded in [max_batch][ntiles] (-1: not
                            //   valid); prefill invalidates every entry of its sequences, the
                            //   decode keeps a sequence's in its first entry
  int32_t* dec_pos;         // [max_batch] device copy of the positions of a host-array decode call
  int* prefill_order;       // [max_batch][ntiles][2] counters ordering a chunk's state read before
                            // its later tiles' state writes (zero between calls)
  bool dec_early_start;     // the next decode may start its weight loads before the preceding
                            // kernel ends (false right after set_weights rewrote the planes)
  cudaEvent_t prof_start, prof_stop;  // optional events around the dominant kernel
  long long launches;                 // kernels enqueued so far
};
