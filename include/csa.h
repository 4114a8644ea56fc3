/*
 * csa.h - C ABI of the GB300 (sm_103a) compressed-sparse-attention KV Compressor.
 *
 * What it computes (per compressor instance, i.e. per attention layer):
 *
 *   kv, score = x . wkv^T, x . wgate^T        f32, x is bf16 promoted to f32
 *       ("DeepSeek V4.1 - Pool token pairs", Compressor excerpt, forward: x.float(),
 *        wkv(x), wgate(x); "Module compress", linear_f32: w is [out_dim][in_dim])
 *   k^p_j = sum_i softmax_i(score_i) (.) kv_i  per feature, over the candidates of group j
 *       (same page, pooling formula; "Compressed Sparse Attention - ratio m = 4":
 *        at ratio 4 overlapped, 8 candidates = branch B of the previous group's 4 tokens
 *        + branch A of the current group's 4 tokens, the first entry's previous branch
 *        padded)
 *   latent = fp4( RoPE( RMSNorm( bf16(k^p_j) ) ) )
 *       (Pool token pairs: norm(kv.to(bf16)); ratio-4 page: "normalized, rotary position
 *        is applied"; "Module compress": yarn_freqs_cis with compress_rope_theta, and
 *        fp4_quant_e4m3_inplace with LATENT_BLOCK = 16: e2m1 values, e4m3 scales)
 *
 * Prefill (start_pos 0) emits N / ratio entries per sequence and leaves the trailing
 * partial group in the per-sequence state; decode (one token per sequence) writes a state
 * slot and emits an entry when its group completes, (start_pos + 1) % ratio == 0
 * (Pool token pairs, forward; ratio-4 page, "Prefill and decode use the same rule").
 *
 * Conventions
 *  - All pointers marked "dev" are CUDA device pointers on the current device; "host"
 *    pointers are ordinary host memory.  The caller owns every buffer it passes in.
 *    The library owns its weights (copied and re-laid out by set_weights), the state,
 *    the RoPE table and its scratch memory.
 *  - Layouts are row-major and dense.  bf16 values are passed as uint16_t bit patterns.
 *  - Work is enqueued on the given stream and is asynchronous unless stated otherwise.
 *    A NULL stream is the legacy default stream.
 *  - Every function returns a status (CSA_OK = 0, or a negative csa_status) unless it
 *    states otherwise; csa_last_error() then describes the failure (per host thread).
 *    Nothing aborts and no C++ exception crosses this boundary.
 *  - A handle is not thread-safe: calls on one handle must be serialised by the caller,
 *    and work on one handle's state must be ordered on the device (one stream, or
 *    events), since decode and prefill read and write the state.
 */
#ifndef CSA_H
#define CSA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* csa_stream_t; /* the same type as cudaStream_t */
typedef struct CUevent_st* csa_event_t;   /* the same type as cudaEvent_t */
typedef struct csa_compressor csa_compressor;

typedef enum {
  CSA_OK = 0,
  CSA_ERR_ARG = -1,      /* invalid argument or shape */
  CSA_ERR_CUDA = -2,     /* a CUDA call failed (launch, allocation, copy) */
  CSA_ERR_STATE = -3,    /* call out of order (weights not set) */
  CSA_ERR_TIMEOUT = -4,  /* a device-side wait ran out of its iteration budget */
  CSA_ERR_DEVICE = -5,   /* a kernel reported an input it could not handle (see csa_device_status) */
  CSA_ERR_INTERNAL = -6
} csa_status;

/* Options of a compressor instance.  csa_options_default() gives the released Flash
 * configuration of the ratio-4 page ("Released Flash configuration": RoPE sub-dimension
 * 64) with compress_rope_theta 160000, YaRN factor 16 over an original length of 4096. */
typedef struct {
  int max_batch;       /* state slots (sequences); default 128 */
  int rope_dim;        /* rotary slice at the end of the latent; 0 disables RoPE; default 64 */
  float rope_base;     /* compress_rope_theta; default 160000 */
  float rope_factor;   /* YaRN scaling factor; default 16 */
  int rope_orig_len;   /* YaRN original context length; default 4096 */
  float beta_fast;     /* YaRN ramp: dims turning more often than this keep their frequency; 32 */
  float beta_slow;     /* YaRN ramp: dims turning less often than this are interpolated; 1 */
  int max_pos;         /* RoPE table length (largest position + 1); default 262144 */
  int fp4;             /* fp4 round trip of the output: 1 = e2m1 values with an e4m3 scale per 16
                          features, the latent's (default); 2 = e2m1 values with a power-of-two
                          (e8m0) scale per 32 features, the indexer's keys (head_dim % 32 == 0);
                          0 = off */
  float eps;           /* RMSNorm epsilon; default 1e-6 */
  int prefill_split;   /* launch geometry of the tensor-core prefill: 0 = chosen per call from a
                          model of its time (default); 1 = one CTA per (packed tile, token tile);
                          2 = a cluster of two CTAs per tile, each taking half of K (dim), the two
                          partial sums added on chip.  The outputs agree within the rounding of
                          that addition; a tuning knob, not a change of the method. */
  int prefill_pair;    /* 0 = one CTA per packed tile (default); 2 = where a tile is not split
                          over K and the packed tiles pair up, two CTAs (a cluster of two) share
                          one tcgen05 MMA of M = 256 rows, each holding its packed tile's weights
                          and half of the token tile.  The same products and additions; a tuning
                          knob (on GB300 it measured 2-3 % slower at the configurations here). */
} csa_options;

/* Output buffers of one call (dev).  Rows are entries: prefill [B][G][..], decode [B][..].
 *  latent   [.., H] bf16, required: the final latent (dequantised fp4 values if fp4 is on)
 *  codes    [.., H/2] u8 or NULL: e2m1 codes, element 2i in the low nibble, sign in bit 3
 *  scales   [.., H/16] u8 or NULL: e4m3 bit patterns, one per block of 16 features (fp4 = 1);
 *           [.., H/32] u8: e8m0 bytes (2^(byte - 127)), one per block of 32 features (fp4 = 2)
 *  prequant [.., H] bf16 or NULL: the latent after RMSNorm and RoPE, before fp4 */
typedef struct {
  uint16_t* latent;
  uint8_t* codes;
  uint8_t* scales;
  uint16_t* prequant;
} csa_out;

/* Fills *opt with the defaults above. */
void csa_options_default(csa_options* opt);

/* Creates a compressor with the default options (csa_options_default) for x of width dim,
 * latent width head_dim, group size ratio ("Pool token pairs", Compressor(dim, head_dim,
 * ratio); "Compressed Sparse Attention - ratio m = 4": the overlapped form).  overlap = 1
 * selects the ratio-4 overlapped form (two branches of head_dim each) and requires ratio == 4.
 * Requirements: dim % 64 == 0, head_dim % 16 == 0 and 16 <= head_dim <= 512, ratio >= 1.
 * Allocates device memory on the current device (weights, state, RoPE table), which becomes the
 * handle's device: every later call on the handle must be made with that device current
 * (otherwise it returns CSA_ERR_ARG).  Builds the YaRN table on the host in double precision.
 * On success *out receives the handle; on failure *out is NULL and nothing stays allocated. */
int csa_compressor_create(int dim, int head_dim, int ratio, int overlap, csa_compressor** out);

/* The same with explicit options; opt may be NULL (defaults).  Further requirements: rope_dim
 * even and <= head_dim, max_batch >= 1, fp4 in {0, 1, 2} (2: head_dim % 32 == 0), eps >= 0,
 * valid RoPE constants when rope_dim > 0. */
int csa_compressor_create_ex(int dim, int head_dim, int ratio, int overlap, const csa_options* opt,
                             csa_compressor** out);

/* Copies the weights into library-owned, re-laid-out buffers.
 *  wkv   [C][dim] f32 dev, C = (1 + overlap) * head_dim ("Module compress" linear_f32 layout);
 *        rows 0..head_dim-1 are branch A (or the only branch), rows head_dim.. branch B
 *  wgate [C][dim] f32 dev, same layout; may be NULL only at ratio 1 (softmax over one
 *        candidate is 1, so the gate has no effect)
 *  norm_gain [head_dim] f32 dev: RMSNorm weight
 * Returns after the re-layout kernels are enqueued; the caller's buffers may be freed once
 * the stream reaches that point. */
int csa_compressor_set_weights(csa_compressor* c, const float* wkv, const float* wgate, const float* norm_gain,
                               csa_stream_t stream);

/* Gate positional bias ("Compressed Sparse Attention": the pooling logits are "wgate(x) +
 * positional bias"; the pages give neither its shape nor its values).  ape [ratio][C] f32 dev,
 * C = (1 + overlap) * head_dim (the gate's columns, branch A then B): a token at position p
 * gets score = wgate(x) + ape[p % ratio], one f32 addition, before it is pooled or stored in
 * the state.  The library keeps its own re-laid-out copy (the caller's buffer may be freed once
 * the stream reaches this call); NULL removes the bias (the default: none).  Applies to calls
 * enqueued after this one; tokens already in the state keep the bias they were given. */
int csa_compressor_set_gate_bias(csa_compressor* c, const float* ape, csa_stream_t stream);

/* Prefill of B sequences, tokens start_pos .. start_pos + N - 1 of each ("Pool token pairs",
 * Compressor forward, prefill branch).  x [B][N][dim] bf16 dev.  Sequence b uses state slot
 * slot_offset + b; needs B >= 1, N >= 1 and slot_offset + B <= max_batch (an empty call returns
 * CSA_ERR_ARG and enqueues nothing).
 *  - start_pos 0: the whole-sequence prefill of the pages.  Writes G = N / ratio entries per
 *    sequence and leaves the trailing N % ratio tokens in the state (at ratio 4 overlapped, also
 *    the last complete group's tokens, whose branch B the next entry pools).
 *  - start_pos > 0: a chunk continuing sequences whose earlier tokens went through prefill,
 *    chunks or decode (all B at the same position).  The pages define this only one token at a
 *    time (the decode branch); a chunk gives the results of N such steps ("Compressed Sparse
 *    Attention", "prefill and decode use the same rule"): the entries of the groups that
 *    complete inside the chunk, G = (start_pos + N) / ratio - start_pos / ratio, their earlier
 *    candidates read from the state, and a state holding the chunk's tokens of the unfinished
 *    group (and, overlapped, of the last complete group).
 * Entry j of sequence b (group start_pos / ratio + j, RoPE position ratio * that group) goes to
 * row b * G + j of out ([B][G][..]).  Returns G (0 means "no entry", the pages' None) or a
 * negative csa_status.  Requires ratio * (last group) < max_pos when RoPE is on.
 * The launch geometry (token tile, K split; csa_prefill_geometry) is chosen per call on the host.
 * The first prefill on a device also sets the kernels' shared-memory attribute and asks the
 * device how many two-CTA clusters it holds; make it before capturing prefill calls into a CUDA
 * graph. */
int csa_compress_prefill(csa_compressor* c, const uint16_t* x, int B, int N, int start_pos, int slot_offset,
                         const csa_out* out, csa_stream_t stream);

/* The same prefill (whole sequence or chunk), writing each entry straight into the caller's
 * compressed-KV cache at its group index: group g of sequence b goes to row b * cache_rows + g
 * of each array of *cache ([B][cache_rows][..], same element layouts as csa_out; codes, scales
 * and prequant may be NULL).  The pages have no such call; it saves the copy from out into a
 * cache.  Needs (start_pos + N) / ratio <= cache_rows; rows of other groups are not touched.
 * Returns the number of entries written per sequence, or a negative csa_status. */
int csa_compress_prefill_into(csa_compressor* c, const uint16_t* x, int B, int N, int start_pos, int slot_offset,
                              const csa_out* cache, int cache_rows, csa_stream_t stream);

/* Prefill that allocates no device memory.  The pages have no counterpart: this exists for
 * callers that cannot let the library call cudaMalloc, such as serving runtimes that reserve
 * all device memory for their own pool up front, or code that enqueues work while a CUDA
 * graph is being captured.  Same arguments, results and return value as
 * csa_compress_prefill, but the tensor-core kernel's scratch lives in a device array built
 * into the library (16 MiB, held by every GPU that loads the library until the process
 * exits).  It therefore needs:
 *  - a shape that runs the tensor-core kernel (csa_uses_tensor_cores(c) == 1, x 16-byte
 *    aligned); other shapes return CSA_ERR_ARG;
 *  - scratch of at most 16 MiB: B * ceil((a + N) / T) * (T / ratio) * head_dim * 2 bytes of
 *    pooled values, with a = start_pos % ratio and T the tokens a tile owns (the launch takes a
 *    tile of 256, 224 or 128 tokens, chosen from the number of SMs of the device: at ratio 4
 *    overlapped T = 252, 220 or 124, else the largest multiple of ratio <= the tile).  Because T
 *    depends on the device, the CSA_ERR_ARG "too large" return is the authoritative check:
 *    larger calls return it without launching anything.
 * The first call on each device looks up the array's device address (with that device
 * current); make that first call before any stream capture.  Every call shares the one
 * array: calls that overlap on the GPU (other streams, other handles) race, so serialise
 * them. */
int csa_compress_prefill_noalloc(csa_compressor* c, const uint16_t* x, int B, int N, int start_pos,
                                 int slot_offset, const csa_out* out, csa_stream_t stream);

/* One decode step for sequences 0..B-1 (state slots 0..B-1), one token each ("Pool token
 * pairs", Compressor forward, decode branch: the token goes to state slot start_pos % ratio, and
 * when (start_pos + 1) % ratio == 0 the group is pooled and emitted, otherwise the module returns
 * None; "Module compress", compressor: "or None while a group is still filling").
 *  x_tok     [B][dim] bf16 dev
 *  start_pos [B] int32 HOST: position of this token in its sequence (per sequence); 0 restarts
 *            the sequence (the pages' prefill branch with one token).  The library copies the
 *            array before returning, so the caller may reuse it at once.
 *  out       rows [B][..] (dev); row b is written only where sequence b emits
 *  emitted   [B] u8, HOST or dev, or NULL: 1 where the token completed a group, else 0 (a host
 *            array is filled before the call returns; a device array is written by the kernels)
 * Returns the number of emitting sequences (0 is the pages' None for every sequence), or a
 * negative csa_status.  1 <= B <= max_batch; positions must be >= 0 and, for emitting
 * sequences, the entry position start_pos + 1 - ratio must be < max_pos when RoPE is on:
 * violations return CSA_ERR_ARG and enqueue nothing.  The copy of start_pos to the device is
 * a host-to-device copy from ordinary host memory, which cannot be captured into a CUDA graph:
 * graphs use csa_compress_decode_dev. */
int csa_compress_decode(csa_compressor* c, const uint16_t* x_tok, int B, const int32_t* start_pos,
                        const csa_out* out, uint8_t* emitted, csa_stream_t stream);

/* The same decode step with the positions in device memory, for callers whose positions live on
 * the device and for CUDA-graph capture (a replayed graph reads positions that device work has
 * advanced between replays).  The pages have only the host form above; this one cannot return
 * the count, because the positions are not known on the host when the call is enqueued.
 *  start_pos [B] int32 dev
 *  emitted   [B] u8 dev (required)
 * Returns CSA_OK or a negative csa_status.  A position the kernels cannot handle (negative, or
 * an entry position beyond the RoPE table) leaves its row unwritten, sets emitted[b] = 0 and
 * raises the flag read by csa_device_status. */
int csa_compress_decode_dev(csa_compressor* c, const uint16_t* x_tok, int B, const int32_t* start_pos,
                            const csa_out* out, uint8_t* emitted, csa_stream_t stream);

/* Resets state slots [slot_begin, slot_begin + slot_count): kv 0, score -inf.  It also clears,
 * for those sequences, the library's own per-call bookkeeping (the decode running values, and
 * the counters that order a chunk's state read before its state writes, which a call that
 * returned CSA_ERR_TIMEOUT may have left set). */
int csa_state_reset(csa_compressor* c, int slot_begin, int slot_count, csa_stream_t stream);

/* Number of float elements of each of the two exported state arrays. */
int64_t csa_state_elems(const csa_compressor* c);

/* Copies the state into kv and score (dev, csa_state_elems floats each), in the logical
 * layout: non-overlapped [max_batch][ratio][head_dim]; ratio 4 overlapped
 * [max_batch][2 parities][4 slots][2 * head_dim] (branch A then B; group g of a sequence
 * lives in parity g % 2).  For tests and for moving a session, not for checkpoints (the
 * pages keep the state out of checkpoints). */
int csa_state_export(const csa_compressor* c, float* kv, float* score, csa_stream_t stream);

/* The inverse of csa_state_export: replaces the whole state (every sequence's slots) with kv and
 * score (dev, csa_state_elems floats each, the logical layout above), e.g. a session moved from
 * another handle of the same shape and options.  The decode running values kept between calls
 * are marked stale (the next decode rebuilds them from the slots, as after a prefill), and the
 * chunk ordering counters are cleared.  Returns CSA_OK or a negative csa_status. */
int csa_state_import(csa_compressor* c, const float* kv, const float* score, csa_stream_t stream);

/* Reads and clears the device-side error flag of the handle (synchronises the stream).
 * Returns CSA_OK if no kernel flagged anything since the last call; CSA_ERR_TIMEOUT if a
 * device-side wait ran out of its time budget (flag bit 4: the kernel stopped its work, let its
 * copies and tensor-core operations in flight finish and returned, leaving that call's outputs
 * and state slots undefined; the handle stays usable); else CSA_ERR_DEVICE: bit 1 a negative
 * start_pos, bit 2 an entry position beyond the RoPE table, bit 8 (only in the bounds-checked
 * build of the library) a store outside its buffer, skipped, bit 16 (that build only) a counter
 * ordering a prefill chunk's state read before its state writes not back at zero after the call.
 * A time-out (bit 4) is also raised when a chunk's later token tile waited in vain for its first
 * tile's state read; it then leaves the state unwritten. */
int csa_device_status(csa_compressor* c, csa_stream_t stream);

/* Frees the handle and its device memory (synchronises the device first). NULL is a no-op. */
void csa_compressor_destroy(csa_compressor* c);

/* Description of the last failure on this host thread ("" if none). */
const char* csa_last_error(void);

/* The latent's fp4 round trip alone ("Module compress", fp4_quant_e4m3_inplace, block 16):
 * in [n_blocks][16] bf16 dev -> codes [n_blocks][8] u8 dev (may be NULL),
 * scales [n_blocks] u8 dev (e4m3 bits), out [n_blocks][16] bf16 dev (dequantised).
 * Runs the same device routine as the compressor's epilogue. */
int csa_fp4_e4m3_roundtrip(const uint16_t* in, int64_t n_blocks, uint8_t* codes, uint8_t* scales, uint16_t* out,
                           csa_stream_t stream);

/* The indexer's fp4 round trip alone ("Module compress", fp4_quant_e8m0_inplace, FP4_BLOCK 32:
 * scale = the power-of-two ceiling of max(amax, 6 * 2^-126) / 6, values to e2m1, dequantised
 * and rounded to bf16): in [n_blocks][32] bf16 dev -> codes [n_blocks][16] u8 dev (may be
 * NULL), scales [n_blocks] u8 dev (e8m0 bytes), out [n_blocks][32] bf16 dev.  Runs the same
 * device routine as the compressor's epilogue with fp4 = 2. */
int csa_fp4_e8m0_roundtrip(const uint16_t* in, int64_t n_blocks, uint8_t* codes, uint8_t* scales, uint16_t* out,
                           csa_stream_t stream);

/* Measurement hook (the pages have no counterpart): while start and stop are set, every
 * prefill or decode call on this handle records `start` on its stream just before its
 * dominant kernel (the projection GEMM with its fused epilogue) and `stop` just after it,
 * so the caller can time that kernel alone with cudaEventElapsedTime.  NULL, NULL turns it
 * off.  The events stay owned by the caller and must outlive their use. */
int csa_set_profile_events(csa_compressor* c, csa_event_t start, csa_event_t stop);

/* 1 if csa_compress_prefill on this handle runs the tensor-core kernel (for a 16-byte
 * aligned x), 0 if it runs the CUDA-core projection (packed tiles narrower than 128 rows,
 * ratio above 256, or no tensor-map encoder in the driver), or a negative csa_status. */
int csa_uses_tensor_cores(const csa_compressor* c);

/* Number of kernels this handle has enqueued since it was created (all calls). */
int64_t csa_kernel_launches(const csa_compressor* c);

/* The launch geometry a tensor-core prefill of B sequences of N tokens at start_pos would use on
 * the current device (no counterpart on the pages; for tuning and measurement): *token_tile = the
 * tokens per tile including the overlapped halo (256, 224 or 128), *k_split = 1 (one CTA per tile)
 * or 2 (a cluster of two CTAs per tile, each half of dim), *cta_pair (may be NULL) = 1, or 2 when
 * two CTAs share one MMA of 256 rows (option prefill_pair).  Returns CSA_OK, CSA_ERR_ARG for a
 * NULL pointer or a bad shape, or CSA_ERR_STATE when the shape runs the CUDA-core projection
 * (csa_uses_tensor_cores(c) == 0).  Host only: nothing is enqueued. */
int csa_prefill_geometry(const csa_compressor* c, int B, int N, int start_pos, int* token_tile, int* k_split,
                         int* cta_pair);

/* Host-only: the YaRN RoPE table the library uploads ("Module compress", yarn_freqs_cis):
 * cos_out, sin_out [npos][rope_dim/2] f32 host for positions pos0..pos0+npos-1, computed in
 * double precision and rounded once to f32. */
int csa_rope_table(const csa_options* opt, int pos0, int npos, float* cos_out, float* sin_out);

#ifdef __cplusplus
}
#endif
#endif /* CSA_H */
