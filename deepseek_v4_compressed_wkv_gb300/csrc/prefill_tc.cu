// Fused prefill on the 5th-generation tensor cores (sm_103a): the projection GEMM with the
// group softmax pool, bf16 rounding, RMSNorm, YaRN RoPE and the fp4 round trip in its
// epilogue.  The pre-pool kv / score values live only in TMEM and shared memory.
//
// GEMM orientation: the packed weight rows are the MMA's M side (128 rows = one packed tile:
// ft features x nk kinds), the tokens its N side (a tile of 256, 224 or 128), K = dim; a tile is
// one CTA, or for compressors with few packed tiles a cluster of two CTAs that each take half of
// K (the launch geometry with the least modelled time, prefill_shape).  The f32 weights
// enter as three bf16 planes whose sum is exact (w = p0 + p1 + p2), so three bf16 MMAs into
// one f32 accumulator give the f32 product (x is bf16, so every partial product is exact):
// the f32 projection of "Pool token pairs" (x.float(), wkv(x), wgate(x)) and the f32 x . w^T
// of "Module compress" (linear_f32).
//
// Accumulation: the tensor cores' f32 accumulator is not IEEE round-to-nearest (truncation per
// MMA leaves ~2^-16 relative error after 768 steps of K=16), so the MMAs of each K chunk of 256
// go into a fresh TMEM accumulator (two, alternating) and the epilogue warps add each chunk into
// f32 registers with ordinary round-to-nearest additions, in chunk order (the promotion to CUDA
// cores used for low-precision accumulators).  Chunks of 128 measured a mean projection error of
// half that of an f32 FMA GEMM; chunks of 256 are 4% faster (chunks of 512: another 2%).
//
// Roles (320 threads): warp 0 issues the TMA loads (x tile shared by all three planes, one
// tile per plane), warp 1 owns TMEM and issues tcgen05.mma, warps 2-9 drain the chunk
// accumulators (warps w and w+4 share TMEM lane quarter w%4 and split the token columns) and
// stage the sums in the idle stage buffers; once the TMEM is freed all ten warps write the state
// tokens and pool.  A tile's CTA (or pair) leaves its pooled values in scratch; the entries are
// then normalised, rotated and quantised by prefill_entry_kernel over all SMs (the RMSNorm needs
// all H features, and one SM finishing a token tile's 63 entries alone took about as long as a
// quarter of the projection).
//
// A chunk at position p0 > 0 (Chunk) tiles the tokens from the start of the open group: the
// first tile's leading a = p0 % ratio token columns (and the overlapped halo) are earlier
// tokens, whose contribution to the first group (overlapped: the first two groups) the first
// tile's CTAs read from the state as running softmax values, before any CTA of the call rewrites
// those slots (a later tile that writes the state waits for that read: a counter per sequence,
// packed tile and K half); their x rows read as zeros and their columns are not pooled.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstdlib>

#include "csa_internal.cuh"
#include "kernels.h"
#include "tc_common.cuh"

namespace csa {
namespace tc {

using namespace tcx;

constexpr int kRows = 128;           // packed rows per tile (MMA M)
constexpr int kTokMax = 256;         // tokens per tile including the halo (MMA N): 256, 224 or 128
constexpr int kKb = 32;              // K elements per stage (one 64-byte swizzle row of bf16)
constexpr int kPlaneBytes = kRows * kKb * 2;          // 8 KB
static_assert(kRows == kPlaneTileRows && kKb == kPlaneTileK, "a stage is one tile of the plane layout");
constexpr int kChunkKb = 8;         // K blocks per accumulator chunk (K = 256)
constexpr int kEpiThreads = 256;
constexpr int kThreads = 64 + kEpiThreads;
constexpr int kTmemCols = 512;      // two chunk accumulators of up to 256 columns (a power of two)

// The sizes that follow from the token tile and from whether a pair of CTAs shares it (PAIR = 2:
// one MMA of M = 256 over two packed tiles, each CTA loading half of the tile's tokens, so that a
// stage is smaller and more of them are in flight).  Epilogue warp half h drains token columns
// [128 h, min(128 h + 128, TOK)).
template <int TOK, int PAIR = 1>
struct Tile {
  static_assert(TOK == 256 || TOK == 224 || TOK == 128, "token tile");
  static_assert(PAIR == 1 || PAIR == 2, "CTA pair");
  static constexpr int kXBytes = TOK / PAIR * kKb * 2;           // 16 / 14 / 8 KB (a pair: half)
  static constexpr int kStageBytes = 3 * kPlaneBytes + kXBytes;  // 40 / 38 / 32 KB (a pair: 32 / 31 / 28)
  static constexpr int kStages = PAIR > 1 ? 6 : 5;               // up to 200 KB
  // f32 staging row stride: a multiple of 4 floats, so that the epilogue moves 16-byte vectors,
  // and an odd number of 16-byte units, so that the vectors of 8 consecutive rows (a quarter-warp)
  // fall in distinct banks
  static constexpr int kSmemStride = TOK + 4;
  static_assert(kSmemStride % 8 == 4, "16-byte rows, odd in 16-byte units");
  static_assert(kRows * kSmemStride * 4 <= kStages * kStageBytes, "staging must fit in the stage buffers");
  static_assert(kStageBytes % 1024 == 0, "stages keep the 1 KB alignment of the swizzled tiles");
};

struct EntryParams {
  int B, G, GT, ntt, ratio;
  int tpe;                 // threads per entry: H / 4 rounded up to a power of two
  Chunk ck;
  const uint16_t* pooled;  // [B][ntt][GT][H] bf16 bits
  EpiParams ep;
  csa_out out;
  long long out_rows;      // rows of the outputs (checked by the bounds-checked build)
  int* flag;
  const int* order;        // a chunk with carried candidates: the call's ordering counters (the
  int order_n;             // bounds-checked build checks that each is back at zero), else null
};

struct Params {
  int N, K, ratio, overlap, T, GT, halo, ntt, G, ncol, slots, slot_offset;
  int a, g0, gend;         // chunk geometry (Chunk): all 0 / G for a prefill from position 0
  const float* ape;        // packed gate positional bias [ratio][ncol] (zero at kv columns), or null
  const __nv_bfloat16* w;  // weight planes, tiled (plane_tile_elem)
  Packing pk;
  float* state;
  uint16_t* pooled;        // [B][ntt][GT][H] bf16 bits
  int carry;               // the first groups have candidates earlier than the chunk (in the state)
  int order_writers;       // carry: later token tiles of a sequence that write the state
  int* order;              // carry: [max_batch][ntiles][2] counters, the first tile's state read done
  int* flag;
  int* acc_pos;            // [max_batch][ntiles] decode running values: marked invalid for the call's sequences
  long long state_elems, pooled_elems;  // extents checked by the bounds-checked build
  unsigned long long wait_ns;           // budget of each device-side wait
  int test_stall;          // bounds-checked build only: the producer never issues the last stage
                           // (a test of the time-out path); 0 otherwise
};

// ---- one entry's epilogue ---------------------------------------------------------------------
//
// The entries (b, j) take H / 4 threads each (rounded up to a power of two, `tpe`, an aligned
// segment of lanes or whole warps); thread te of an entry takes features 4te..4te+3 of its pooled
// values, then bf16, RMSNorm (the sum of squares over the entry's lanes, and over its warps in
// order when it spans several), RoPE and the fp4 round trip (entry_epilogue_quad, whose fp4 blocks
// are aligned groups of four or eight lanes).  entry_prepare reads what does not depend on the
// projection (gain, RoPE factors), entry_finish the rest.

struct EntryPrep {
  int b, j, f;
  bool live, act;
  float gn[4], rc[2], rs[2];
};

__device__ __forceinline__ EntryPrep entry_prepare(const EntryParams& P, int e, int te) {
  EntryPrep q;
  const int H = P.ep.H, hr = P.ep.rope_dim >> 1, r0 = H - P.ep.rope_dim;
  q.f = 4 * te;
  q.live = e < P.B * P.G;
  q.act = q.f < H;
  q.b = q.live ? e / P.G : 0;
  q.j = q.live ? e % P.G : 0;
  const long long pos = (long long)P.ratio * (P.ck.g0 + q.j);
#pragma unroll
  for (int i = 0; i < 4; ++i) q.gn[i] = 0.0f;
#pragma unroll
  for (int u = 0; u < 2; ++u) {
    q.rc[u] = 1.0f;
    q.rs[u] = 0.0f;
  }
  if (q.live && q.act) {
    const float4 gg = __ldg(reinterpret_cast<const float4*>(P.ep.gain + q.f));
    q.gn[0] = gg.x;
    q.gn[1] = gg.y;
    q.gn[2] = gg.z;
    q.gn[3] = gg.w;
#pragma unroll
    for (int u = 0; u < 2; ++u)
      if (hr > 0 && q.f + 2 * u >= r0) {
        q.rc[u] = __ldg(P.ep.rope_cos + pos * hr + ((q.f + 2 * u - r0) >> 1));
        q.rs[u] = __ldg(P.ep.rope_sin + pos * hr + ((q.f + 2 * u - r0) >> 1));
      }
  }
  return q;
}

// t: the thread's index in its CTA; wss: 4 floats of shared memory when tpe > 32 (then every thread
// of the CTA calls this, it synchronises the CTA), else unused.  All 32 lanes of a warp call it.
__device__ __forceinline__ void entry_finish(const EntryParams& P, const EntryPrep& q, int t, float* wss) {
  const int H = P.ep.H, tpe = P.tpe, lane = t & 31;
  const int tt = q.j / P.GT, g = q.j % P.GT;
  float v[4] = {0.0f, 0.0f, 0.0f, 0.0f};
  if (q.live && q.act) {
    const uint2 u = __ldcg(reinterpret_cast<const uint2*>(P.pooled + (((size_t)q.b * P.ntt + tt) * P.GT + g) * H + q.f));
    v[0] = __uint_as_float(u.x << 16);
    v[1] = __uint_as_float(u.x & 0xFFFF0000u);
    v[2] = __uint_as_float(u.y << 16);
    v[3] = __uint_as_float(u.y & 0xFFFF0000u);
  }
  float ss = 0.0f;
#pragma unroll
  for (int i = 0; i < 4; ++i) ss = fmaf(v[i], v[i], ss);
#pragma unroll
  for (int o = 1; o < 32; o <<= 1)
    if (o < tpe) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  if (tpe > 32) {
    if (lane == 0) wss[t >> 5] = ss;
    __syncthreads();
    const int w0 = ((t / tpe) * tpe) >> 5;
    ss = wss[w0];
    for (int w = 1; w < tpe / 32; ++w) ss += wss[w0 + w];
  }
  const float inv = rms_inv(ss, P.ep);
  const long long row = P.ck.row(q.b, q.j);
  const bool ok = q.live && in_bounds(row, P.out_rows, P.flag);
  entry_epilogue_quad(v, q.act && ok, q.f, lane, inv, q.gn, q.rc, q.rs, P.ep, ok ? (size_t)row : 0, P.out);
}

// ---- the kernel ----------------------------------------------------------------------------
//
// kSplit = 2 (a cluster of two CTAs per tile, the narrow compressors' grid): CTA r of the cluster
// runs the K blocks [r K / 2, (r + 1) K / 2) and owns features [r F / 2, (r + 1) F / 2) of the
// tile (F features per kind).  Each CTA stages its partial sums, copies the rows of the other
// CTA's features into that CTA's shared memory (a bulk copy between the two CTAs), adds the
// received half-K sums to its own (the lower K half first) and pools its features: a tile of
// 128 x TOK outputs is then computed at the wide token tile by twice the CTAs.

template <int kTok, int kSplit, int kPair>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_tc_kernel(const __grid_constant__ CUtensorMap map_x, const __grid_constant__ CUtensorMap map_w,
                      const Params P) {
  static_assert(kSplit == 1 || kSplit == 2, "K split");
  static_assert(kSplit == 1 || kPair == 1, "a K split or a CTA pair, not both");
  constexpr bool kP = kPair > 1;
  constexpr int kStages = Tile<kTok, kPair>::kStages;
  constexpr int kStageBytes = Tile<kTok, kPair>::kStageBytes;
  constexpr int kSmemStride = Tile<kTok, kPair>::kSmemStride;
  constexpr int kRecvRows = kSplit > 1 ? kRows / kSplit : 0;  // rows received from the other CTA
  static_assert((kRows + kRecvRows) * kSmemStride * 4 <= kStages * kStageBytes,
                "the staged and the received sums fit in the stage buffers");
  extern __shared__ uint8_t smem_raw[];
  // 1 KB aligned (the swizzled tiles), offset from the shared array itself so that the compiler
  // keeps the accesses through it in the shared state space
  uint8_t* smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
  uint64_t* full = (uint64_t*)(smem + kStages * kStageBytes);
  uint64_t* empty = full + kStages;
  uint64_t* chunk_full = empty + kStages;  // [2]: chunk accumulator ready for the epilogue
  uint64_t* chunk_empty = chunk_full + 2;  // [2]: chunk accumulator drained, free for the MMAs
  uint64_t* mma_done = chunk_empty + 2;    // clean-up after an abort: the issued MMAs have completed
  uint64_t* recv_bar = mma_done + 1;       // kSplit 2: the other CTA's sums of this CTA's rows landed
  uint32_t* tmem_slot = (uint32_t*)(recv_bar + 1);
  volatile int* abort_flag = (volatile int*)(tmem_slot + 1);
  int* issued_s = (int*)(tmem_slot + 2);  // stages the producer issued (read by the clean-up)
  int* order_seen = (int*)(tmem_slot + 3);  // a chunk's later tile: the first tile's state read was
                                            // already done when the stages started
  // a chunk's first tile: the running softmax values (max, denominator, numerator) of the carried
  // candidates of group j and feature f0 + i at [3 * (j * hf + i)], at most 2 x 32 or 64 values
  float* carried = (float*)(tmem_slot + 4);
  static_assert((2 * kStages + 6) * 8 + 16 + 3 * 64 * 4 <= 1024, "barriers, flags and carried values fit their region");

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int ftile = blockIdx.x / kSplit, rank = blockIdx.x % kSplit, tt = blockIdx.y, b = blockIdx.z;
  const int nloc = P.K / kKb / kSplit;  // K blocks of this CTA: kb0 .. kb0 + nloc - 1
  const int kb0 = rank * nloc;
  const int nch = (nloc + kChunkKb - 1) / kChunkKb;
  const int t0 = tt * P.T - P.halo;  // virtual index (from the open group's start) of the tile's token 0
  // a CTA pair: the even CTA (the leader) issues the MMAs for both; each loads its packed tile's
  // weight planes and half of the token tile (the leader the first half)
  const int prank = kP ? (int)(blockIdx.x & 1) : 0;
  const bool leader = prank == 0;
#ifdef CSA_DEBUG_BOUNDS
  const uint64_t kWait = P.wait_ns;  // the time-out test shortens the waits
#else
  constexpr uint64_t kWait = kWaitNs;
#endif

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&chunk_full[i], 1);
      mbar_init(&chunk_empty[i], kPair * kEpiThreads / 32);  // a pair: the leader's counts both CTAs' warps
    }
    mbar_init(mma_done, 1);
    mbar_init(recv_bar, 1);
    *abort_flag = 0;
    *order_seen = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    prefetch_map(&map_x);
    if constexpr (kP) prefetch_map(&map_w);
  }
  if (warp == 1) {
    if constexpr (kP)
      tmem_alloc_pair(tmem_slot, kTmemCols);
    else
      tmem_alloc(tmem_slot, kTmemCols);
  }
  griddep_launch_dependents();  // the entry kernel may be scheduled; it waits for this grid
  tc_fence_before();
  __syncthreads();
  if constexpr (kP) {
    cluster_arrive();
    cluster_wait();  // both CTAs' barriers are initialised before either's copies complete on them
  }
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;


  if (warp == 0) {
    // ---- producer: one x tile and three weight-plane tiles per stage
    if (lane == 0) {
      int issued = 0;
      for (int i = 0; i < nloc; ++i) {
        const int s = i % kStages, kb = kb0 + i;
        if (i >= kStages && !mbar_wait(&empty[s], ((i / kStages) & 1) ^ 1, abort_flag, kWait)) break;
#ifdef CSA_DEBUG_BOUNDS
        if (P.test_stall && i == nloc - 1) break;  // test of the time-out path: the last stage never comes
#endif
        uint8_t* st = smem + s * kStageBytes;
        if constexpr (kP) {
          // both CTAs' copies complete on the leader's barrier, which expects the bytes of both
          const uint32_t fb = cluster_map(&full[s], 0);
          if (leader) mbar_arrive_expect_tx(&full[s], 2 * kStageBytes);
          tma_load_3d_pair(st, &map_w, 0, (3 * kPlaneBytes / 512) * (ftile * (P.K / kKb) + kb), 0, fb);
          tma_load_3d_pair(st + 3 * kPlaneBytes, &map_x, kb * kKb, t0 - P.a + prank * (kTok / 2), b, fb);
        } else {
          mbar_arrive_expect_tx(&full[s], kStageBytes);
          bulk_load(st, P.w + plane_stage_elem(P.K / kKb, ftile, kb), 3 * kPlaneBytes, &full[s]);
          tma_load_3d(st + 3 * kPlaneBytes, &map_x, kb * kKb, t0 - P.a, b, &full[s]);
        }
        ++issued;
      }
      *issued_s = issued;
    }
  } else if (warp == 1) {
    // ---- MMA issuer (a pair: the leader's, for both CTAs)
    if (lane == 0 && leader) {
      constexpr uint32_t idesc = idesc_bf16(kRows * kPair, kTok);
      bool ok = true;
      for (int c = 0; c < nch && ok; ++c) {
        const int buf = c & 1;
        if (c >= 2 && !mbar_wait<kP>(&chunk_empty[buf], ((c >> 1) - 1) & 1, abort_flag, kWait)) break;
        tc_fence_after();
        const uint32_t d = tmem + (uint32_t)(buf * kTok);
        const int i0 = c * kChunkKb, i1 = min(nloc, i0 + kChunkKb);
        for (int i = i0; i < i1; ++i) {
          const int s = i % kStages;
          if (!mbar_wait<kP>(&full[s], (i / kStages) & 1, abort_flag, kWait)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t st = smem_addr(smem + s * kStageBytes);
          const uint32_t xs = st + 3 * kPlaneBytes;
          for (int p = 0; p < 3; ++p)
            for (int k = 0; k < kKb / 16; ++k) {
              const uint64_t a = sw64_desc(st + p * kPlaneBytes + k * 32), bd = sw64_desc(xs + k * 32);
              const uint32_t en = (i != i0 || p != 0 || k != 0) ? 1u : 0u;
              if constexpr (kP)
                mma_bf16_pair(d, a, bd, idesc, en);
              else
                mma_bf16(d, a, bd, idesc, en);
            }
          if constexpr (kP)
            mma_commit_pair_multicast(&empty[s], 0x3);  // both CTAs' producers may refill the stage
          else
            mma_commit(&empty[s]);
        }
        if (ok) {  // arrives once this chunk's MMAs have completed
          if constexpr (kP)
            mma_commit_pair_multicast(&chunk_full[buf], 0x3);
          else
            mma_commit(&chunk_full[buf]);
        }
      }
    }
  } else {
    // ---- epilogue (warps 2..9; warp w reads TMEM lanes 32*(w%4) .. +31, its packed row, and
    //      columns 128*h .. up to 128 columns): the chunk accumulators into registers in chunk
    //      order, then staged as [packed row][token] f32 in the stage buffers (idle once the last
    //      chunk has completed)
    if (P.carry) {
      // idle until the first chunk completes: the first tile reads the candidates it carries
      // from the state (their running values, for the pool), then lets the later tiles of the
      // sequence rewrite it; a later tile looks whether that read is already done (then its state
      // writes need not wait)
      const int e = (int)threadIdx.x - 64;
      if (tt == 0) {
        const int F = P.pk.ft, hf = F / kSplit, f0 = rank * hf, j = e / hf;
        if (j < 1 + P.overlap) {
          const int f = f0 + e % hf;
          const float* sq = P.state + (size_t)(P.slot_offset + b) * P.slots * P.ncol + ftile * kRows + f;
          // candidate i of group j: group 0 takes, overlapped, branch B of group g0 - 1 (parity
          // (g0 - 1) % 2; none for g0 = 0, the padded branch) and branch A of the open group's
          // tokens before p0 (parity g0 % 2, slots 0 .. a - 1), non-overlapped those tokens;
          // overlapped group 1 takes branch B of those tokens
          const int open = 4 * (P.g0 & 1), prev = 4 * ((P.g0 + 1) & 1);
          const int nprev = P.overlap && j == 0 && P.g0 > 0 ? 4 : 0, n = nprev + P.a;
          auto cand = [&](int i, bool score) -> float {
            int slot, kind;
            if (!P.overlap) {
              slot = i;
              kind = score ? S : KV;
            } else if (i < nprev) {
              slot = prev + i;
              kind = score ? S_B : KV_B;
            } else {
              slot = open + i - nprev;
              kind = j == 0 ? (score ? S_A : KV_A) : (score ? S_B : KV_B);
            }
            return sq[(size_t)slot * P.ncol + kind * F];
          };
          float m = -INFINITY, den = 0.0f, num = 0.0f;
          for (int i = 0; i < n; ++i) m = fmaxf(m, cand(i, true));
          if (m > -INFINITY)
            for (int i = 0; i < n; ++i) {
              const float x = expf(cand(i, true) - m);
              den += x;
              num = fmaf(x, cand(i, false), num);
            }
          carried[3 * e] = m;
          carried[3 * e + 1] = den;
          carried[3 * e + 2] = num;
        }
        // every value read (and used) before the later tiles may write: the epilogue warps meet,
        // then one thread signals
        asm volatile("bar.sync 1, %0;" ::"n"(kEpiThreads) : "memory");
        if (e == 0 && P.order_writers > 0)
          counter_release_add(P.order + ((size_t)(P.slot_offset + b) * P.pk.ntiles + ftile) * 2 + rank,
                              P.order_writers);
      } else if (e == 0) {
        *order_seen = counter_ready(P.order + ((size_t)(P.slot_offset + b) * P.pk.ntiles + ftile) * 2 + rank);
      }
    }
    const int q = warp & 3, h = (warp - 2) >> 2;
    const int row = 32 * q + lane;
    const int hcols = h ? kTok - 128 : 128;  // a multiple of 32 (0: the 128-token tile's second half idles)
    float acc[128];
#pragma unroll
    for (int i = 0; i < 128; ++i) acc[i] = 0.0f;
    bool ok = true;
    for (int c = 0; c < nch; ++c) {
      const int buf = c & 1;
      if (!mbar_wait(&chunk_full[buf], (c >> 1) & 1, abort_flag, kWait)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t base = tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(buf * kTok + 128 * h);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        if (32 * j < hcols) {  // the same for the whole warp
          uint32_t r[32];
          tmem_ld32(base + 32 * j, r);
#pragma unroll
          for (int i = 0; i < 32; i += 2)
            fadd2(acc[32 * j + i], acc[32 * j + i + 1], __uint_as_float(r[i]), __uint_as_float(r[i + 1]));
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if constexpr (kP)
          mbar_arrive_remote(cluster_map(&chunk_empty[buf], 0));  // the leader's MMAs may reuse it
        else
          mbar_arrive(&chunk_empty[buf]);
      }
    }
    if (ok && !*abort_flag) {
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      float* stg = (float*)smem;
#pragma unroll
      for (int i = 0; i < 128; i += 4)
        if (i < hcols)
          *reinterpret_cast<float4*>(stg + row * kSmemStride + 128 * h + i) =
              make_float4(acc[i], acc[i + 1], acc[i + 2], acc[i + 3]);
    }
  }

  tc_fence_before();
  __syncthreads();  // every role has left its loop; the flag no longer changes
  const bool aborted = *abort_flag != 0;
  if (aborted) {
    // a wait ran out: the copies in flight land and the issued MMAs complete before the TMEM is
    // freed and the CTA leaves (this call's outputs are undefined; the flag says so)
    if constexpr (kP) {
      // the leader's barriers count both CTAs' copies of the stages it expected, and only it
      // issued MMAs; the other CTA's copies of stages the leader never expected are given time
      // to land (a bounded pause: nothing waits for them)
      if (warp == 0 && lane == 0) {
        if (leader) {
          for (int t = max(0, *issued_s - kStages); t < *issued_s; ++t)
            mbar_wait_bounded(&full[t % kStages], (t / kStages) & 1);
        } else {
          const uint64_t t0 = globaltimer();
          while (globaltimer() - t0 < 50000ull) __nanosleep(1000);
        }
      }
      if (warp == 1 && lane == 0 && leader) {
        mma_commit_pair(mma_done);
        mbar_wait_bounded(mma_done, 0);
      }
    } else {
      drain_after_abort(warp == 0 && lane == 0, warp == 1 && lane == 0, full, kStages, *issued_s, mma_done);
    }
    tc_fence_before();
    __syncthreads();
    if (threadIdx.x == 0) atomicOr(P.flag, 4);
  }
  if (warp == 1 && !kP) {  // a pair frees its TMEM at the end, after both CTAs are done with it
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }

  // ---- the pool, by all warps
  const Packing& pk = P.pk;
  const int F = pk.ft, hf = F / kSplit, f0 = rank * hf;  // this CTA's features of the tile
  float* stg = (float*)smem;
  // the state slots of the sequence's unfinished group (and, overlapped, of the last complete
  // group) that this tile rewrites: virtual tokens [max(own0, s_lo), own1)
  const int own0 = max(tt * P.T, P.a), own1 = min(tt * P.T + P.T, P.a + P.N);
  const int s_lo = P.overlap ? 4 * P.G - (P.G >= 1 ? 4 : 0) : P.ratio * P.G;
  int* order = P.carry ? P.order + ((size_t)(P.slot_offset + b) * pk.ntiles + ftile) * 2 + rank : nullptr;
  if (!aborted) {
    // the prefill rewrites the sequence's state: its decode running values (kept per packed
    // tile) are no longer valid
    if (rank == 0 && tt == 0 && threadIdx.x == 0) P.acc_pos[(size_t)(P.slot_offset + b) * pk.ntiles + ftile] = -1;
  }
  bool lost = false;  // the other CTA's sums never arrived
  if constexpr (kSplit > 1) {
    // the rows of the other CTA's features go to its shared memory (kind k's rows in a block of
    // hf rows), its sums of this CTA's rows come back into `recv`; every CTA takes part whatever
    // its state, so that neither waits on a barrier the other never reaches
    constexpr uint32_t kRunBytesPerRow = kSmemStride * 4;
    float* recv = stg + kRows * kSmemStride;
    if (threadIdx.x == 0) mbar_arrive_expect_tx(recv_bar, (uint32_t)(pk.nk * hf) * kRunBytesPerRow);
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // the staged sums, for the copy
    cluster_arrive();
    cluster_wait();  // both CTAs have staged their sums; neither uses its stage buffers any more
    if (threadIdx.x == 0) {
      const uint32_t peer = (uint32_t)(rank ^ 1);
      const uint32_t peer_bar = cluster_map(recv_bar, peer);
      for (int k = 0; k < pk.nk; ++k)
        bulk_push_cluster(cluster_map(recv + k * hf * kSmemStride, peer),
                          stg + (k * F + (int)peer * hf) * kSmemStride, (uint32_t)hf * kRunBytesPerRow, peer_bar);
    }
    lost = __syncthreads_or(!mbar_wait_bounded(recv_bar, 0, kWait));
    if (lost && threadIdx.x == 0) atomicOr(P.flag, 4);
  }
  // Split without a gate bias, the received half-K sums are added where the state writes and the
  // pool read them (`fold`); unsplit and overlapped, so is the gate bias (`fold_bias`: the token in
  // tile column c has group position c % 4, as the tile starts on a group); otherwise the pass
  // below leaves this CTA's final values in stg.
  const float* recv = stg + kRows * kSmemStride;
  const bool fold = kSplit > 1 && !P.ape;
  const bool fold_bias = kSplit == 1 && P.ape && P.overlap;
  if (!aborted && !lost && (kSplit > 1 || P.ape) && !fold && !fold_bias) {
    // this CTA's rows: the two half-K sums added (the same sum in either order), then wgate(x) +
    // the positional bias of each token's place in its group (score rows; column c holds the
    // token at position ratio * g0 + t0 + c, halo columns wrap harmlessly).  Unsplit, only the
    // score rows of a layer with the bias are visited.  Warp w takes rows w, w + 10, ..., its
    // lanes the columns.
    const int kind0 = kSplit > 1 ? 0 : pk.nk / 2;
    const int r = P.ratio, step = 32 % r;
    const int sl0 = ((P.ratio * P.g0 + t0 + lane) % r + r) % r;
    for (int rr = kind0 * hf + warp; rr < pk.nk * hf; rr += kThreads / 32) {
      const int kind = rr / hf;
      const int prow = kind * F + f0 + (rr - kind * hf);
      float* srow = stg + prow * kSmemStride;
      const float* rrow = recv + rr * kSmemStride;
      const float* ab = P.ape && kind >= pk.nk / 2 ? P.ape + ftile * kRows + prow : nullptr;
      // every load of the row before any store (the stores could otherwise alias the next loads)
      constexpr int kCol = kTok / 32;
      float v[kCol], w[kCol];
#pragma unroll
      for (int i = 0; i < kCol; ++i) {
        v[i] = srow[lane + 32 * i];
        w[i] = kSplit > 1 ? rrow[lane + 32 * i] : 0.0f;
      }
      if (ab) {
        int sl = sl0;
#pragma unroll
        for (int i = 0; i < kCol; ++i) {
          w[i] = kSplit > 1 ? v[i] + w[i] : v[i];
          v[i] = __ldg(ab + (size_t)sl * P.ncol);
          sl += step;
          sl = sl >= r ? sl - r : sl;
        }
      }
#pragma unroll
      for (int i = 0; i < kCol; ++i) srow[lane + 32 * i] = v[i] + w[i];
    }
  }
  __syncthreads();

  // the final sum of packed row (kind, f) of this CTA's features at tile column col, one value or
  // the four from col (col a multiple of 4)
  // the bias of packed row prow at group position sl (zero at the kv rows)
  auto bias = [&](int prow, int sl) { return __ldg(P.ape + (size_t)sl * P.ncol + ftile * kRows + prow); };
  auto at = [&](int kind, int f, int col) -> float {
    float v = stg[(kind * F + f) * kSmemStride + col];
    if (fold) v += recv[(kind * hf + f - f0) * kSmemStride + col];
    if (fold_bias && kind >= pk.nk / 2) v += bias(kind * F + f, (t0 + col) & 3);
    return v;
  };
  // the four group positions' biases of this thread's pool feature (col is a multiple of 4, so
  // position i is element i), for the score kinds
  const int fpool = f0 + (int)threadIdx.x % hf;
  float4 bias4[2] = {make_float4(0.f, 0.f, 0.f, 0.f), make_float4(0.f, 0.f, 0.f, 0.f)};
  if (fold_bias)
    for (int u = 0; u < 2; ++u)
      bias4[u] = make_float4(bias((S_A + u) * F + fpool, 0), bias((S_A + u) * F + fpool, 1),
                             bias((S_A + u) * F + fpool, 2), bias((S_A + u) * F + fpool, 3));
  auto at4 = [&](int kind, int f, int col) -> float4 {
    float4 v = *reinterpret_cast<const float4*>(stg + (kind * F + f) * kSmemStride + col);
    if (fold) {
      const float4 w = *reinterpret_cast<const float4*>(recv + (kind * hf + f - f0) * kSmemStride + col);
      v.x += w.x;
      v.y += w.y;
      v.z += w.z;
      v.w += w.w;
    }
    if (fold_bias && kind >= S_A) {  // f is this thread's pool feature
      const float4 w = bias4[kind - S_A];
      v.x += w.x;
      v.y += w.y;
      v.z += w.z;
      v.w += w.w;
    }
    return v;
  };

  // a later tile that rewrites state slots waits until the first tile has read its carried
  // candidates (also when aborted, so that the counter returns to zero); a wait that runs out
  // leaves the state unwritten and raises the time-out bit
  bool late = false;
  if (P.carry && tt > 0 && max(own0, s_lo) < own1) {
    late = __syncthreads_or(threadIdx.x == 0 && !(*order_seen ? (atomicSub(order, 1), true) : counter_take(order, kWait)));
    if (late && threadIdx.x == 0) atomicOr(P.flag, 4);
  }
  if (!aborted) {
    const int r = P.ratio, G = P.G;
    const int col0 = ftile * kRows;  // first packed column of this tile
    // -- state: the new tokens (virtual index >= a) of the unfinished group and, overlapped,
    //    of the last complete group that this tile owns; thread et < nk * hf writes one packed
    //    column of this CTA's features.  Virtual group G is absolute group gend.
    const int et = threadIdx.x;
    if (et < pk.nk * hf && !late) {
      const int kind = et / hf, prow = kind * F + f0 + et % hf;
      const size_t st0 = (size_t)(P.slot_offset + b) * P.slots * P.ncol + col0 + prow;
      float* st = P.state + st0;
      auto put = [&](int tok, int slot) {  // token tok is the tile's column tok - t0
        if (in_bounds((long long)st0 + (long long)slot * P.ncol, P.state_elems, P.flag))
          st[slot * P.ncol] = at(kind, f0 + et % hf, tok - t0);
      };
      if (!P.overlap) {
        for (int tok = max(own0, r * G); tok < own1; ++tok) put(tok, tok - r * G);
      } else {
        const int qp = P.gend & 1;
        for (int tok = max(own0, 4 * G); tok < own1; ++tok) put(tok, 4 * qp + tok - 4 * G);
        if (G >= 1)
          for (int tok = max(own0, 4 * G - 4); tok < min(own1, 4 * G); ++tok)
            put(tok, 4 * (1 - qp) + tok - (4 * G - 4));
        if (P.gend == 0 && tt == 0) {
          const float pad = kind < pk.nk / 2 ? 0.0f : -INFINITY;  // padded previous branch: kv 0, score -inf
          for (int i = 0; i < 4; ++i)
            if (in_bounds((long long)st0 + (long long)(4 + i) * P.ncol, P.state_elems, P.flag)) st[(4 + i) * P.ncol] = pad;
        }
      }
    }
    // -- pool every (feature, group) pair of this CTA's features into bf16 scratch: thread t
    //    takes feature f0 + t % hf and groups t / hf, t / hf + kThreads / hf, ... (hf divides the
    //    320 threads: 16, 32 or 64), two groups per step whose chains are independent
    uint16_t* pooled_tile = P.pooled + ((size_t)b * P.ntt + tt) * P.GT * pk.H;
    const int f = f0 + (int)threadIdx.x % hf;
    // a group all of whose candidates are this tile's columns
    auto pool_tile = [&](int g, int j) -> float {
      float m = -INFINITY, den = 0.0f, num = 0.0f;
      if (P.overlap) {
        // branch A: tokens 4g + 4 .. 4g + 7 of the tile, branch B: tokens 4g .. 4g + 3 (one
        // 16-byte vector each)
        const float4 a4 = at4(KV_A, f, 4 * g + 4), p4 = at4(S_A, f, 4 * g + 4);
        const float4 b4 = at4(KV_B, f, 4 * g), q4 = at4(S_B, f, 4 * g);
        const float kA[4] = {a4.x, a4.y, a4.z, a4.w}, sA[4] = {p4.x, p4.y, p4.z, p4.w};
        const float kB[4] = {b4.x, b4.y, b4.z, b4.w}, sB[4] = {q4.x, q4.y, q4.z, q4.w};
        const bool padB = P.g0 + j == 0;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          m = fmaxf(m, sA[i]);
          if (!padB) m = fmaxf(m, sB[i]);
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float ea = expf(sA[i] - m);
          den += ea;
          num = fmaf(ea, kA[i], num);
          if (!padB) {
            const float eb = expf(sB[i] - m);
            den += eb;
            num = fmaf(eb, kB[i], num);
          }
        }
      } else if (r % 2 == 0) {
        // the group's ratio tokens as 8-byte pairs (and the received half-K sums beside them)
        const float2* kv = reinterpret_cast<const float2*>(stg + (KV * F + f) * kSmemStride + r * g);
        const float2* sc = reinterpret_cast<const float2*>(stg + (S * F + f) * kSmemStride + r * g);
        const float2* kv2 = reinterpret_cast<const float2*>(recv + (KV * hf + f - f0) * kSmemStride + r * g);
        const float2* sc2 = reinterpret_cast<const float2*>(recv + (S * hf + f - f0) * kSmemStride + r * g);
        auto pair = [&](const float2* own, const float2* got, int i) {
          float2 v = own[i];
          if (fold) {
            const float2 w = got[i];
            v.x += w.x;
            v.y += w.y;
          }
          return v;
        };
        for (int i = 0; i < r / 2; ++i) {
          const float2 s2 = pair(sc, sc2, i);
          m = fmaxf(m, fmaxf(s2.x, s2.y));
        }
        for (int i = 0; i < r / 2; ++i) {
          const float2 s2 = pair(sc, sc2, i), k2 = pair(kv, kv2, i);
          const float e0 = expf(s2.x - m), e1 = expf(s2.y - m);
          den += e0;
          num = fmaf(e0, k2.x, num);
          den += e1;
          num = fmaf(e1, k2.y, num);
        }
      } else {
        for (int i = 0; i < r; ++i) m = fmaxf(m, at(S, f, r * g + i));
        for (int i = 0; i < r; ++i) {
          const float e = expf(at(S, f, r * g + i) - m);
          den += e;
          num = fmaf(e, at(KV, f, r * g + i), num);
        }
      }
      return __fdiv_rn(num, den);
    };
    // a chunk's first groups hold tokens earlier than the chunk (virtual index < a, or the halo):
    // those arrive as the running values read while the stages streamed; the rest are this tile's columns.  Group 0:
    // branch A of tokens a..3 (non-overlapped: tokens a..ratio-1); overlapped group 1: branch B
    // of tokens a..3 and branch A of tokens 4..7.
    auto pool_carried = [&](int j) -> float {
      const float* cv = carried + 3 * (j * hf + f - f0);
      const float mc = cv[0], dc = cv[1], nc = cv[2];  // max, denominator, numerator
      const int kk = P.overlap ? KV_A : KV, ks = P.overlap ? S_A : S;
      const int c0 = P.halo + 4 * j;  // this group's first column (branch A when overlapped)
      const int n = P.overlap ? 4 : r, i0 = j == 0 ? P.a : 0, iB = j == 1 ? P.a : 4;
      float m = mc;
      for (int i = i0; i < n; ++i) m = fmaxf(m, at(ks, f, c0 + i));
      for (int i = iB; i < 4; ++i) m = fmaxf(m, at(S_B, f, P.halo + i));
      const float rs = expf(mc - m);  // 0 when nothing was carried (mc = -inf)
      float den = dc * rs, num = nc * rs;
      for (int i = iB; i < 4; ++i) {
        const float e = expf(at(S_B, f, P.halo + i) - m);
        den += e;
        num = fmaf(e, at(KV_B, f, P.halo + i), num);
      }
      for (int i = i0; i < n; ++i) {
        const float e = expf(at(ks, f, c0 + i) - m);
        den += e;
        num = fmaf(e, at(kk, f, c0 + i), num);
      }
      return __fdiv_rn(num, den);
    };
    auto put_pooled = [&](int g, float v) {
      const size_t pi = (size_t)g * pk.H + ftile * F + f;
      if (in_bounds((long long)((pooled_tile - P.pooled) + pi), P.pooled_elems, P.flag)) pooled_tile[pi] = bf16_bits(v);
    };
    const int gstep = kThreads / hf;
    if (!P.overlap && r == 2 && !P.carry) {
      // pairs of tokens ("Pool token pairs"): one 16-byte load holds groups 2p and 2p + 1, the
      // additions in the order of the general loop below
      for (int p = (int)threadIdx.x / hf; 2 * p < P.GT; p += gstep) {
        const int g = 2 * p, j = tt * P.GT + g;
        if (j >= G) break;
        const float4 s4 = at4(S, f, 4 * p), k4 = at4(KV, f, 4 * p);
        const float m0 = fmaxf(s4.x, s4.y), m1 = fmaxf(s4.z, s4.w);
        const float a0 = expf(s4.x - m0), b0 = expf(s4.y - m0), a1 = expf(s4.z - m1), b1 = expf(s4.w - m1);
        put_pooled(g, __fdiv_rn(fmaf(b0, k4.y, fmaf(a0, k4.x, 0.0f)), (0.0f + a0) + b0));
        if (g + 1 < P.GT && j + 1 < G)
          put_pooled(g + 1, __fdiv_rn(fmaf(b1, k4.w, fmaf(a1, k4.z, 0.0f)), (0.0f + a1) + b1));
      }
    } else if (!P.overlap && r >= 64 && r % 8 == 0 && !P.carry && hf % 16 == 0) {
      // long groups (ratio 128: two per 256-token tile): two adjacent threads per (feature, group),
      // each over half of the group's tokens from the group's maximum (the pair's), the two
      // halves' sums added once.  The 16 pairs of a warp share their group (16 divides hf), so whole
      // warps iterate together and the pair exchanges are full-warp shuffles.
      const int q = (int)threadIdx.x >> 1, part = (int)threadIdx.x & 1;
      const int qstep = (kThreads / 2) / hf;  // groups per step: 2 (hf 64) or 5 (hf 32)
      const int fq = f0 + q % hf, half = r / 2;
      if (q < qstep * hf) {
        for (int g = q / hf; g < P.GT; g += qstep) {
          const int j = tt * P.GT + g;
          if (j >= G) break;
          const int c0 = r * g + half * part;  // this thread's first column
          float m = -INFINITY;
          for (int i = 0; i < half; i += 4) {
            const float4 v = at4(S, fq, c0 + i);
            m = fmaxf(m, fmaxf(fmaxf(v.x, v.y), fmaxf(v.z, v.w)));
          }
          m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
          float den = 0.0f, num = 0.0f;
          for (int i = 0; i < half; i += 4) {
            const float4 sv = at4(S, fq, c0 + i), kv = at4(KV, fq, c0 + i);
            const float e0 = expf(sv.x - m), e1 = expf(sv.y - m), e2 = expf(sv.z - m), e3 = expf(sv.w - m);
            den += e0;
            num = fmaf(e0, kv.x, num);
            den += e1;
            num = fmaf(e1, kv.y, num);
            den += e2;
            num = fmaf(e2, kv.z, num);
            den += e3;
            num = fmaf(e3, kv.w, num);
          }
          den += __shfl_xor_sync(0xffffffffu, den, 1);  // the same sum in both threads of the pair
          num += __shfl_xor_sync(0xffffffffu, num, 1);
          if (part == 0) {
            const size_t pi = (size_t)g * pk.H + ftile * F + fq;
            if (in_bounds((long long)((pooled_tile - P.pooled) + pi), P.pooled_elems, P.flag))
              pooled_tile[pi] = bf16_bits(__fdiv_rn(num, den));
          }
        }
      }
    } else {
      for (int g = (int)threadIdx.x / hf; g < P.GT; g += 2 * gstep) {
        const int j = tt * P.GT + g;
        if (j >= G) break;  // groups are visited in order
        // the second group (never a carried one: gstep >= 5), or the first again when there is none
        const bool two = g + gstep < P.GT && j + gstep < G;
        const float v2 = two ? pool_tile(g + gstep, j + gstep) : 0.0f;
        const float v1 = P.carry && j < 1 + P.overlap ? pool_carried(j) : pool_tile(g, j);
        put_pooled(g, v1);
        if (two) put_pooled(g + gstep, v2);
      }
    }
  }
  if constexpr (kSplit > 1) {
    cluster_arrive();
    cluster_wait();  // the other CTA has received this CTA's copy: its source may go
  }
  if constexpr (kP) {
    tc_fence_before();
    cluster_arrive();
    cluster_wait();  // the leader's MMAs into this CTA's TMEM and its arrivals on this CTA's barriers are over
    if (warp == 1) {
      tc_fence_after();
      tmem_dealloc_pair(tmem, kTmemCols);
    }
  }
}

// The entries in their own kernel: a CTA of 128 threads takes 128 / tpe consecutive entries (one
// CTA per entry at H = 512); the gain and RoPE factors (written before this launch's predecessor
// started) are read before the wait for the projection kernel.
__global__ void __launch_bounds__(128) prefill_entry_kernel(const EntryParams P) {
  __shared__ float wss[4];
  const int t = threadIdx.x;
  const EntryPrep q = entry_prepare(P, blockIdx.x * (128 / P.tpe) + t / P.tpe, t % P.tpe);
  griddep_wait();  // the pooled values of the projection kernel
#ifdef CSA_DEBUG_BOUNDS
  // the projection grid has completed: every counter that ordered the first tile's state read
  // before a later tile's state writes was taken as often as it was released
  if (P.order && blockIdx.x == 0)
    for (int i = t; i < P.order_n; i += 128)
      if (P.order[i] != 0) atomicOr(P.flag, 16);
#endif
  entry_finish(P, q, t, wss);
}

}  // namespace tc

// ---- host side ------------------------------------------------------------------------------

bool prefill_tc_supported(const csa_compressor* c, const void* x) {
  return c->pk.tw == tc::kRows && c->dim % tc::kKb == 0 && (c->overlap || c->ratio <= tc::kTokMax) &&
         ((uintptr_t)x & 15) == 0 && tcx::get_encode() != nullptr;
}

namespace {

// The token tiles after the first that rewrite state slots of a chunk whose first tile reads
// candidates from the state (the kernel's own test, for tiles 1 .. ntt - 1).
int order_writers(const csa_compressor* c, const tc::Params& P, int N) {
  const int s_lo = c->overlap ? 4 * P.G - (P.G >= 1 ? 4 : 0) : c->ratio * P.G;
  int n = 0;
  for (int tt = 1; tt < P.ntt; ++tt)
    n += std::max(std::max(tt * P.T, P.a), s_lo) < std::min(tt * P.T + P.T, P.a + N);
  return n;
}

// Tokens of a tile owned by it (the overlapped tile also loads the 4 tokens before it).
int owned_tokens(const csa_compressor* c, int tok) {
  return c->overlap ? tok - 4 : (tok / c->ratio) * c->ratio;
}

// Time of one K stage of a CTA, in cycles: the six MMAs of 64-cycle units per 128 tokens, or the
// round trip of the 5-stage ring (a stage's copy issued when its slot is freed, landed, consumed
// by the MMAs, freed again), which measured about 750 cycles whatever the tile: the 128- and
// 224-token tiles ran at that floor (0.46 and 0.86 of the MMA rate), the 256-token tile at its
// 768 cycles of MMA (0.98-0.99).
long long stage_cycles(int tok) { return std::max(3LL * tok, 750LL); }
// Per CTA besides its K stages (from per-CTA timestamps at about 1.9 GHz): the first stage landing,
// the last chunk drained, the staging and the pool, about 3.5 us; a K-split CTA adds the cluster
// barrier, the copy between the two CTAs and the received sums it reads, about 2.6 us.
constexpr long long kTileCycles = 6700;
constexpr long long kSplitCycles = 5000;

template <int TOK, int SPLIT, int PAIR>
size_t smem_bytes() {
  using T = tc::Tile<TOK, PAIR>;
  return (size_t)T::kStages * T::kStageBytes + 1024 /* barriers */ + 1024 /* alignment */;
}

template <int TOK, int SPLIT, int PAIR>
cudaError_t set_smem_attr() {
  static std::atomic<unsigned long long> attr_set{0};
  return tcx::once_per_device(attr_set, [] {
    return cudaFuncSetAttribute(tc::prefill_tc_kernel<TOK, SPLIT, PAIR>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)smem_bytes<TOK, SPLIT, PAIR>());
  });
}

// Clusters of two CTAs of the K-split kernel that the device holds at once (0 if it cannot say),
// asked once per device and tile.
template <int TOK>
int split_clusters() {
  static std::atomic<int> known[64];  // clusters + 1 per device; 0: not asked yet
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  const int k = known[dev & 63].load();
  if (k > 0) return k - 1;
  int n = 0;
  if (set_smem_attr<TOK, 2, 1>() == cudaSuccess) {
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = 2;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * current_sm_count(), 1, 1);
    cfg.blockDim = dim3(tc::kThreads, 1, 1);
    cfg.dynamicSmemBytes = smem_bytes<TOK, 2, 1>();
    cfg.attrs = at;
    cfg.numAttrs = 1;
    if (cudaOccupancyMaxActiveClusters(&n, (const void*)tc::prefill_tc_kernel<TOK, 2, 1>, &cfg) != cudaSuccess) {
      (void)cudaGetLastError();
      n = 0;
    }
  } else {
    (void)cudaGetLastError();
  }
  known[dev & 63].store(n + 1);
  return n;
}

int split_clusters_of(int tok) {
  switch (tok) {
    case 224:
      return split_clusters<224>();
    case 128:
      return split_clusters<128>();
    default:
      return split_clusters<256>();
  }
}

// The launch geometry with the least modelled time: waves (CTAs over the SMs, or clusters of two
// over the clusters the device holds) x the time of a CTA (its K stages x the stage time, plus the
// rest of a tile and the exchange of a split tile); the larger tile, then the unsplit grid, on a
// tie.  At the Flash CSA shape the
// 224-token tile makes 16 x 19 = 304 CTAs, exactly two waves of 152 SMs; the indexer's 128-wide
// compressor (4 packed tiles) takes the 224-token tile split over K, 4 x 19 clusters of two in one
// wave; one long sequence through the ratio-128 compressor takes the 256-token tile.
PrefillPlan prefill_shape(const csa_compressor* c, int B, int N) {
  const int sms = current_sm_count();
  const int nkb = c->dim / tc::kKb;
  const int force = c->opt.prefill_split;
  PrefillPlan best{tc::kTokMax, 1, 0, 0};
  long long best_cost = -1;
  for (int split : {1, 2}) {
    if (force && split != force) continue;
    if (split == 2 && (nkb % 2 != 0 || c->pk.ft % 2 != 0)) continue;
    for (int tok : {256, 224, 128}) {
      const int T = owned_tokens(c, tok);
      if (T < 1) continue;
      const long long ctas = (long long)c->pk.ntiles * ((N + T - 1) / T) * B * split;
      const long long slots = split == 1 ? sms : 2LL * split_clusters_of(tok);
      if (slots <= 0) continue;
      const long long cost =
          (ctas + slots - 1) / slots * (nkb / split * stage_cycles(tok) + kTileCycles + (split > 1 ? kSplitCycles : 0));
      if (best_cost < 0 || cost < best_cost) {
        best = PrefillPlan{tok, split, 0, 0};
        best_cost = cost;
      }
    }
  }
  // asked for, unsplit tiles run as CTA pairs wherever the packed tiles pair up
  if (c->opt.prefill_pair == 2 && best.split == 1 && c->pk.ntiles % 2 == 0) best.pair = 2;
  return best;
}

template <int TOK, int SPLIT, int PAIR>
cudaError_t launch_tok(const csa_compressor* c, const uint16_t* x, int B, int N, int slot_offset, const Chunk& ck,
                       const csa_out& out, void* scratch, size_t scratch_bytes, cudaStream_t s) {
  using namespace tc;
  auto encode = tcx::get_encode();
  if (!encode) return cudaErrorNotSupported;
  Params P;
  P.N = N;
  P.K = c->dim;
  P.ratio = c->ratio;
  P.overlap = c->overlap;
  P.halo = c->overlap ? 4 : 0;
  P.T = owned_tokens(c, TOK);
  P.GT = P.T / c->ratio;
  P.ntt = (ck.a + N + P.T - 1) / P.T;
  P.G = ck.G;
  P.a = ck.a;
  P.g0 = ck.g0;
  P.gend = ck.gend;
  P.ncol = c->pk.cols();
  P.slots = c->slots;
  P.slot_offset = slot_offset;
  P.pk = c->pk;
  P.state = c->state;
  P.pooled = (uint16_t*)scratch;
  P.carry = chunk_needs_carry(ck, c->overlap);
  P.order_writers = P.carry ? order_writers(c, P, N) : 0;
  P.order = c->prefill_order;
  P.ape = c->ape_set ? c->ape : nullptr;
  P.flag = c->dev_flag;
  P.acc_pos = c->dec_acc_pos;
  P.state_elems = (long long)c->opt.max_batch * c->slots * P.ncol;
  // the pooled values' extent, for the bounds-checked build: what this launch writes, but never
  // past the scratch it was given
  const size_t pooled_bytes = (size_t)B * P.ntt * P.GT * c->H * sizeof(uint16_t);
  P.pooled_elems = (long long)(std::min(pooled_bytes, scratch_bytes) / sizeof(uint16_t));
  P.w = c->w_planes;
  P.wait_ns = tcx::kWaitNs;
  P.test_stall = 0;
#ifdef CSA_DEBUG_BOUNDS
  // the time-out test: the producer leaves out the last stage, and the waits give up sooner
  if (getenv("CSA_TEST_STALL_LAST_STAGE")) {
    P.test_stall = 1;
    P.wait_ns = 200000000ull;
  }
#endif
  CUtensorMap mx;
  {
    // x: [B][N][dim] bf16; out-of-range tokens (the halo before token 0, the tail past N) read as 0
    cuuint64_t dims[3] = {(cuuint64_t)c->dim, (cuuint64_t)N, (cuuint64_t)B};
    cuuint64_t strides[2] = {(cuuint64_t)c->dim * 2, (cuuint64_t)N * c->dim * 2};
    cuuint32_t box[3] = {kKb, TOK / PAIR, 1};  // a pair: each CTA loads half of the tile's tokens
    cuuint32_t es[3] = {1, 1, 1};
    if (encode(&mx, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, (void*)x, dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  CUtensorMap mw = mx;  // read only by a CTA pair
  if (PAIR > 1) {
    // the weight planes as the contiguous 24 KB stages they are stored in (already the swizzled
    // image a stage holds, so copied as they are), seen as rows of 512 bytes: a stage (the three
    // planes of one tile and K block) is 48 rows
    const int nkb = c->dim / kKb;
    constexpr int kW = 256, kWRows = 3 * kPlaneBytes / (2 * kW);
    cuuint64_t dims[3] = {(cuuint64_t)kW, (cuuint64_t)c->pk.ntiles * nkb * kWRows, 1};
    cuuint64_t strides[2] = {(cuuint64_t)kW * 2, (cuuint64_t)c->pk.ntiles * nkb * kWRows * kW * 2};
    cuuint32_t box[3] = {kW, kWRows, 1};
    cuuint32_t es[3] = {1, 1, 1};
    if (encode(&mw, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, (void*)c->w_planes, dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  // the entries: RMSNorm, RoPE and fp4, in their own kernel, started early by programmatic
  // dependent launch (the pooled values are read after its wait)
  EntryParams Q;
  Q.B = B;
  Q.G = P.G;
  Q.GT = P.GT;
  Q.ntt = P.ntt;
  Q.ratio = c->ratio;
  Q.tpe = 4;
  while (Q.tpe < c->H / 4) Q.tpe *= 2;
  Q.ck = ck;
  Q.pooled = P.pooled;
  Q.out_rows = (long long)B * ck.bstride;
  Q.flag = c->dev_flag;
  Q.order = P.carry ? c->prefill_order + (size_t)slot_offset * c->pk.ntiles * 2 : nullptr;
  Q.order_n = B * c->pk.ntiles * 2;
  Q.ep = epi_params(c);
  Q.out = out;
  cudaError_t ea = set_smem_attr<TOK, SPLIT, PAIR>();
  if (ea != cudaSuccess) return ea;
  cudaLaunchAttribute pat[1];
  int npat = 0;
  if (SPLIT > 1 || PAIR > 1) {  // the two K halves of a tile, or two packed tiles sharing the MMA: one cluster
    pat[npat].id = cudaLaunchAttributeClusterDimension;
    pat[npat].val.clusterDim.x = SPLIT * PAIR;
    pat[npat].val.clusterDim.y = 1;
    pat[npat].val.clusterDim.z = 1;
    ++npat;
  }
  cudaLaunchConfig_t pc = {};
  pc.gridDim = dim3(c->pk.ntiles * SPLIT, P.ntt, B);
  pc.blockDim = dim3(kThreads, 1, 1);
  pc.dynamicSmemBytes = smem_bytes<TOK, SPLIT, PAIR>();
  pc.stream = s;
  pc.attrs = pat;
  pc.numAttrs = npat;
  cudaError_t e = cudaLaunchKernelEx(&pc, prefill_tc_kernel<TOK, SPLIT, PAIR>, mx, mw, P);
  if (e != cudaSuccess || P.G == 0) return e;
  const long long ctas = ((long long)B * P.G + 128 / Q.tpe - 1) / (128 / Q.tpe);
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)ctas, 1, 1);
  cfg.blockDim = dim3(128, 1, 1);
  cfg.stream = s;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, prefill_entry_kernel, Q);
}

}  // namespace

PrefillPlan prefill_tc_plan(const csa_compressor* c, int B, int N, const Chunk& ck) {
  PrefillPlan plan = prefill_shape(c, B, ck.a + N);
  const int T = owned_tokens(c, plan.tok);
  const int GT = T / c->ratio;
  const int ntt = (ck.a + N + T - 1) / T;
  plan.bytes = (size_t)B * ntt * GT * c->H * sizeof(uint16_t);
  // the projection kernel, the entry kernel
  plan.kernels = 1 + (ck.G > 0);
  return plan;
}

cudaError_t launch_prefill_tc(const csa_compressor* c, const uint16_t* x, int B, int N, int slot_offset,
                              const Chunk& ck, const PrefillPlan& plan, const csa_out& out, void* scratch,
                              size_t scratch_bytes, cudaStream_t s) {
  if (scratch_bytes < plan.bytes) return cudaErrorInvalidValue;
  if (plan.pair == 2 && (plan.split != 1 || c->pk.ntiles % 2 != 0)) return cudaErrorInvalidValue;
  const int kind = plan.split == 2 ? 2 : plan.pair == 2 ? 1 : 0;  // split, pair, one CTA per tile
#define CSA_LAUNCH_TOK(T)                                                                                         \
  return kind == 2   ? launch_tok<T, 2, 1>(c, x, B, N, slot_offset, ck, out, scratch, scratch_bytes, s)          \
         : kind == 1 ? launch_tok<T, 1, 2>(c, x, B, N, slot_offset, ck, out, scratch, scratch_bytes, s)          \
                     : launch_tok<T, 1, 1>(c, x, B, N, slot_offset, ck, out, scratch, scratch_bytes, s)
  switch (plan.tok) {
    case 224:
      CSA_LAUNCH_TOK(224);
    case 128:
      CSA_LAUNCH_TOK(128);
    default:
      CSA_LAUNCH_TOK(256);
  }
#undef CSA_LAUNCH_TOK
}

}  // namespace csa
