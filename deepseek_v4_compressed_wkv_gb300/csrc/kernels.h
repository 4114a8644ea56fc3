// Launchers of the compressor's kernels (host side, enqueue only).
#pragma once

#include "csa_internal.cuh"

namespace csa {

EpiParams epi_params(const csa_compressor* c);
cudaError_t launch_pack_weights(const csa_compressor* c, const float* wkv, const float* wgate, cudaStream_t s);
// Dense rows (mode 0, prefill: row m is token m % N at position p0 + m % N) or decode state
// slots (mode 1, positions start_pos); the gate positional bias, if set, is added.
cudaError_t launch_projection_ffma(const csa_compressor* c, const uint16_t* x, int M, float* out, int mode,
                                   const int32_t* start_pos, int N, int p0, cudaStream_t s);
cudaError_t launch_pack_ape(const csa_compressor* c, const float* ape, cudaStream_t s);
cudaError_t launch_prefill_pool(const csa_compressor* c, const float* proj, int B, int N, int slot_offset,
                                const Chunk& ck, const csa_out& out, cudaStream_t s);
cudaError_t launch_prefill_state(const csa_compressor* c, const float* proj, int B, int N, int slot_offset,
                                 const Chunk& ck, cudaStream_t s);
cudaError_t launch_decode_emit(const csa_compressor* c, const int32_t* start_pos, int B, const csa_out& out,
                               uint8_t* emitted, cudaStream_t s);
cudaError_t launch_state_reset(const csa_compressor* c, int slot_begin, int count, cudaStream_t s);
cudaError_t launch_state_export(const csa_compressor* c, float* kv, float* score, cudaStream_t s);
cudaError_t launch_state_import(const csa_compressor* c, const float* kv, const float* score, cudaStream_t s);
cudaError_t launch_fp4_roundtrip(const uint16_t* in, long long nb, uint8_t* codes, uint8_t* scales, uint16_t* out,
                                 cudaStream_t s);
cudaError_t launch_fp4_e8m0_roundtrip(const uint16_t* in, long long nb, uint8_t* codes, uint8_t* scales,
                                      uint16_t* out, cudaStream_t s);

// Tensor-core prefill (prefill_tc.cu): projection + pool + norm + RoPE + fp4 + state update.
bool prefill_tc_supported(const csa_compressor* c, const void* x);
// The launch geometry of one call, fixed once so that the scratch it is given and the launch
// agree: the token tile, the K split and the scratch bytes it needs (the pooled values [B][token
// tiles][groups per tile][H] bf16 and, for a chunk whose first group has earlier candidates, their
// running softmax values [B][1 + overlap][3][H] f32 after them).
struct PrefillPlan {
  int tok;       // token tile: 256, 224 or 128
  int split;     // 1: one CTA per tile; 2: a cluster of two CTAs per tile, each half of K
  size_t bytes;  // scratch bytes
  int kernels;   // kernels the call launches
  int pair = 1;  // split 1: 2 when two CTAs (two packed tiles) share one MMA of M = 256 and the
                 // token tile, each loading half of its tokens
};
PrefillPlan prefill_tc_plan(const csa_compressor* c, int B, int N, const Chunk& ck);
// scratch_bytes: the capacity of `scratch` (>= plan.bytes), the extent the bounds-checked build
// checks the kernels' scratch stores against.
cudaError_t launch_prefill_tc(const csa_compressor* c, const uint16_t* x, int B, int N, int slot_offset,
                              const Chunk& ck, const PrefillPlan& plan, const csa_out& out, void* scratch,
                              size_t scratch_bytes, cudaStream_t s);

// Tensor-core decode (decode_tc.cu): two launches per call, the projection of one token per
// sequence (split over K, partial sums to `part`), then one CTA per sequence for the reduction into
// its state slot, the pool and the epilogue.  `early_start` lets the projection fetch its weights
// before the preceding kernel in the stream has finished.
bool decode_tc_supported(const csa_compressor* c, const void* x, int B);
// Marks the decode running values of sequences [first, first + count) as not valid (their state
// slots were rewritten by something other than the tensor-core decode).
cudaError_t invalidate_decode_acc(const csa_compressor* c, int first, int count, cudaStream_t s);
int decode_tc_slices(const csa_compressor* c);
// Bytes of the split-K partial sums of a call of B sequences; kernels a call launches.
size_t decode_tc_part_bytes(const csa_compressor* c, int B);
int decode_tc_kernels_per_call();
cudaError_t launch_decode_tc(csa_compressor* c, const uint16_t* x, int B, const int32_t* start_pos, float* part,
                             const csa_out& out, uint8_t* emitted, bool early_start, cudaStream_t s);

}  // namespace csa
