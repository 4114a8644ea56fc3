// Decode on the tensor cores (sm_103a): one token per sequence, into each sequence's state slot
// ("Pool token pairs", decode branch: kv_state[:, slot] = kv, score_state[:, slot] = score),
// then the pool and epilogue of the sequences whose group completes.
//
// Decode streams every weight once per step for only B tokens, so it is bound by HBM.  The
// projection streams the three exact bf16 planes of the weights that set_weights prepared (w =
// p0 + p1 + p2; 6 bytes per weight, 1.5x the f32 weights) straight into the tensor cores.
//
// Two launches per call, chained by programmatic dependent launch so that neither waits for
// the other to be scheduled:
//
//  * decode_proj_kernel, grid (packed tile, K slice, 128-token block): accumulates the slice in
//    K chunks of 128 (TMEM, promoted to f32 registers as in the prefill kernel) and writes its
//    partial sums.  Roles (320 threads): warp 0 issues the loads (one bulk copy of the three
//    pre-swizzled plane tiles and one TMA token tile of K = 32 per stage, 6 stages), warp 1 owns
//    TMEM and issues tcgen05.mma, warps 2-9 drain the chunk accumulators, the cluster of 4 K
//    slices adds its sums through distributed shared memory and stores them with TMA.  The
//    weights are not written by any kernel that can precede a decode launch in early-start
//    mode, so warp 0 fetches the first stages' weight tiles (and prefetches the next stages into
//    L2) before it waits for the preceding kernel; the tokens, and every write, come after
//    that wait.
//
//  * decode_finish_kernel, one CTA per sequence: adds the K slices' partial sums in slice order
//    (a deterministic split-K reduction) into the token's state slot, applies the restart at
//    position 0, and where the token completed a group pools every feature over the group's
//    candidates ("Pool token pairs", decode branch; "Compressed Sparse Attention - ratio m =
//    4", decode rule) and runs the entry epilogue (bf16, RMSNorm, RoPE, fp4).  The candidates
//    from earlier calls are combined before the wait for the projection, while it still runs;
//    non-overlapped groups keep running softmax values from call to call instead of re-reading
//    their earlier tokens.  One CTA per sequence fits on an SM beside a projection CTA.
//
// Each launch lets the next one start as soon as all of its CTAs have begun: the finish kernel
// at once, the projection right after its own wait.  A CTA only ever waits for a launch whose
// CTAs have all started, so the chain cannot deadlock whatever the occupancy.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "csa_internal.cuh"
#include "kernels.h"
#include "tc_common.cuh"

namespace csa {
namespace dtc {

using namespace tcx;

constexpr int kRows = 128;                              // packed rows per tile (MMA M)
constexpr int kTok = 128;                               // tokens per CTA (MMA N)
constexpr int kKb = 64;                                 // K granularity of the slice split
constexpr int kKs = 32;                                 // K per stage (one 64-byte swizzle row of bf16)
constexpr int kStages = 6;
constexpr int kPrefetchStages = 2;                     // weight stages fetched into L2 beyond the ring
constexpr int kChunkSteps = 4;                          // stages per accumulator chunk (K = 128)
constexpr int kPlaneBytes = kRows * kKs * 2;            // 8 KB
static_assert(kRows == kPlaneTileRows && kKs == kPlaneTileK, "a stage is one tile of the plane layout");
constexpr int kXBytes = kTok * kKs * 2;                 // 8 KB
constexpr int kStageBytes = 3 * kPlaneBytes + kXBytes;  // 32 KB
constexpr int kRingBytes = kStages * kStageBytes;       // 192 KB
constexpr int kPartBytes = kTok * kRows * 4;            // one CTA's partial sums, staged in the ring
static_assert(kPartBytes <= kRingBytes, "the partial tile is staged in the free ring");
constexpr int kEpiThreads = 256;
constexpr int kThreads = 64 + kEpiThreads;
constexpr int kTmemCols = 2 * kTok;
// One warp per SM sub-partition: fits beside a projection CTA, whose three warps on a sub-partition
// (135 registers each) leave room for one finish warp (87 registers).  More registers in either kernel
// break that overlap: at 142 projection registers a decode step measured 0.254 of HBM instead of 0.29.
constexpr int kFinThreads = 128;

__device__ __forceinline__ void add4(float4& a, const float4& v) {
  a.x += v.x;
  a.y += v.y;
  a.z += v.z;
  a.w += v.w;
}

struct ProjParams {
  const __nv_bfloat16* w;  // weight planes, tiled (plane_tile_elem)
  int nkb_total, ks;  // K blocks (of 64) of dim, number of K slices
  int cs;             // K slices per cluster, added on chip: 1, 2 or 4 (divides ks and the 128 tokens)
  int B;              // tokens of the call
  int ncol;           // packed columns (rows of one weight plane)
  float* part;        // [ks][B][ncol] partial sums
  int* flag;
};

__global__ void __launch_bounds__(kThreads, 1)
    decode_proj_kernel(const __grid_constant__ CUtensorMap map_x, const __grid_constant__ CUtensorMap map_p,
                       const ProjParams P) {
  extern __shared__ uint8_t smem_raw[];
  // 1 KB aligned (the swizzled tiles), offset from the shared array itself so that the compiler
  // keeps the accesses through it in the shared state space
  uint8_t* smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
  uint64_t* full = (uint64_t*)(smem + kRingBytes);
  uint64_t* empty = full + kStages;
  uint64_t* c_full = empty + kStages;
  uint64_t* c_empty = c_full + 2;
  uint64_t* mma_done = c_empty + 2;  // clean-up after an abort: the issued MMAs have completed
  uint32_t* tmem_slot = (uint32_t*)(mma_done + 1);
  volatile int* abort_flag = (volatile int*)(tmem_slot + 1);
  int* issued_s = (int*)(tmem_slot + 2);  // stages the producer issued (read by the clean-up)

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int tile = blockIdx.x, ks = blockIdx.y, tb = blockIdx.z * kTok;
  const int kb_base = (int)((long long)ks * P.nkb_total / P.ks);
  const int nkb = (int)((long long)(ks + 1) * P.nkb_total / P.ks) - kb_base;
  const int nstep = nkb * (kKb / kKs);
  const int nch = (nstep + kChunkSteps - 1) / kChunkSteps;
  const int k0 = kb_base * kKb;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&c_full[i], 1);
      mbar_init(&c_empty[i], kEpiThreads / 32);
    }
    mbar_init(mma_done, 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    prefetch_map(&map_x);
    prefetch_map(&map_p);
  }
  if (warp == 1) tmem_alloc(tmem_slot, kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  float acc[kTok / 2];  // epilogue warps: this thread's row over half of the token columns
#pragma unroll
  for (int i = 0; i < kTok / 2; ++i) acc[i] = 0.0f;

  if (warp == 0) {
    if (lane == 0) {
      const int npre = min(nstep, kStages);
      const uint64_t stream_pol = l2_evict_first();  // every weight is read once per call
      const int nkb32 = P.nkb_total * (kKb / kKs), kb0 = k0 / kKs;
      const __nv_bfloat16* wt = P.w + plane_stage_elem(nkb32, tile, kb0);  // this slice's stages, contiguous
      constexpr int kW = 3 * kPlaneBytes;
      // weights of the first stages into the ring and of the next kPrefetchStages into L2.  A
      // longer L2 prefetch was slower: the copy engine works through the queued prefetches
      // before the token tiles that the MMAs wait for after the wait below
      for (int t = 0; t < npre; ++t) {
        mbar_arrive_expect_tx(&full[t], kStageBytes);
        bulk_load_hint(smem + t * kStageBytes, wt + (size_t)t * (kW / 2), kW, &full[t], stream_pol);
      }
      for (int t = npre; t < min(nstep, npre + kPrefetchStages); ++t)
        bulk_prefetch_l2_hint(wt + (size_t)t * (kW / 2), kW, stream_pol);
      griddep_wait();  // the tokens may come from the preceding kernel
      griddep_launch_dependents();
      for (int t = 0; t < npre; ++t)
        tma_load_2d(smem + t * kStageBytes + 3 * kPlaneBytes, &map_x, k0 + t * kKs, tb, &full[t]);
      int issued = npre;
      for (int t = npre; t < nstep; ++t) {
        const int s = t % kStages;
        if (!mbar_wait(&empty[s], ((t / kStages) - 1) & 1, abort_flag)) break;
        uint8_t* st = smem + s * kStageBytes;
        mbar_arrive_expect_tx(&full[s], kStageBytes);
        bulk_load_hint(st, wt + (size_t)t * (kW / 2), kW, &full[s], stream_pol);
        tma_load_2d(st + 3 * kPlaneBytes, &map_x, k0 + t * kKs, tb, &full[s]);
        ++issued;
      }
      *issued_s = issued;
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16(kRows, kTok);
      bool ok = true;
      for (int c = 0; c < nch && ok; ++c) {
        const int buf = c & 1;
        if (c >= 2 && !mbar_wait(&c_empty[buf], ((c >> 1) - 1) & 1, abort_flag)) break;
        tc_fence_after();
        const uint32_t d = tmem + (uint32_t)(buf * kTok);
        const int t0 = c * kChunkSteps, t1 = min(nstep, t0 + kChunkSteps);
        for (int t = t0; t < t1; ++t) {
          const int s = t % kStages;
          if (!mbar_wait(&full[s], (t / kStages) & 1, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t st = smem_addr(smem + s * kStageBytes);
          const uint32_t xa = st + 3 * kPlaneBytes;
          for (int p = 0; p < 3; ++p)
            for (int k = 0; k < kKs / 16; ++k)
              mma_bf16(d, sw64_desc(st + p * kPlaneBytes + k * 32), sw64_desc(xa + k * 32), idesc,
                       (t != t0 || p != 0 || k != 0) ? 1u : 0u);
          mma_commit(&empty[s]);
        }
        if (ok) mma_commit(&c_full[buf]);
      }
    }
  } else {
    // drain each chunk into f32 registers, in chunk order (staged for the reduction below)
    const int q = warp & 3, h = (warp - 2) >> 2;
    bool ok = true;
    for (int c = 0; c < nch; ++c) {
      const int buf = c & 1;
      if (!mbar_wait(&c_full[buf], (c >> 1) & 1, abort_flag)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t base = tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(buf * kTok + (kTok / 2) * h);
#pragma unroll
      for (int j = 0; j < kTok / 64; ++j) {
        uint32_t r[32];
        tmem_ld32(base + 32 * j, r);
#pragma unroll
        for (int i = 0; i < 32; ++i) acc[32 * j + i] += __uint_as_float(r[i]);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&c_empty[buf]);
    }
    (void)ok;  // a failed wait has raised the abort flag
  }

  tc_fence_before();
  __syncthreads();  // every role has left its loop; the flag no longer changes
  if (*abort_flag) {
    // a wait ran out: the copies in flight land and the issued MMAs complete before the TMEM is
    // freed and the ring is reused (this call's results are undefined; the flag says so)
    drain_after_abort(warp == 0 && lane == 0, warp == 1 && lane == 0, full, kStages, *issued_s, mma_done);
    tc_fence_before();
    __syncthreads();
    if (threadIdx.x == 0) atomicOr(P.flag, 4);
  }
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
  if (warp >= 2) {
    // every MMA has completed and every load has landed: the ring is free.  Stage the partial
    // sums as [token][packed row]
    const int h = (warp - 2) >> 2, row = 32 * (warp & 3) + lane;
    float* stg = reinterpret_cast<float*>(smem);
#pragma unroll
    for (int i = 0; i < kTok / 2; ++i) stg[((kTok / 2) * h + i) * kRows + row] = acc[i];
  }
  // The cs K slices of the cluster are added on chip: CTA r adds tokens [r * 128 / cs, ...) of
  // the cs staged tiles in slice order (distributed shared memory) and stores that part of the
  // cluster's partial sums with one TMA store (tokens past B are clipped)
  const int cs = P.cs, tr = kTok / cs;
  const int crank = cs > 1 ? (int)cluster_rank() : 0;
  float* stg = reinterpret_cast<float*>(smem);
  float* red = cs > 1 ? stg + kTok * kRows : stg + crank * tr * kRows;
  if (cs > 1) {
    cluster_arrive();
    cluster_wait();  // every CTA of the cluster has staged its tile
    // up to kRedItems items of four floats per thread, every load issued before the additions
    constexpr int kRedItems = (kTok / 2) * (kRows / 4) / kThreads + 1;  // covers cs >= 2
    float4 v[kRedItems][4];
#pragma unroll
    for (int it = 0; it < kRedItems; ++it) {
      const int idx = threadIdx.x + it * kThreads;
      if (idx < tr * (kRows / 4)) {
        const float* src = stg + (crank * tr + idx / (kRows / 4)) * kRows + 4 * (idx % (kRows / 4));
#pragma unroll
        for (int q = 0; q < 4; ++q)
          if (q < cs) v[it][q] = ld_cluster_f4(cluster_map(src, q));
      }
    }
#pragma unroll
    for (int it = 0; it < kRedItems; ++it) {
      const int idx = threadIdx.x + it * kThreads;
      if (idx < tr * (kRows / 4)) {
        float4 a = v[it][0];
#pragma unroll
        for (int q = 1; q < 4; ++q)
          if (q < cs) add4(a, v[it][q]);
        *reinterpret_cast<float4*>(red + (idx / (kRows / 4)) * kRows + 4 * (idx % (kRows / 4))) = a;
      }
    }
  }
  fence_async_shared();
  __syncthreads();
  if (threadIdx.x == 64) {
    griddep_wait();  // the preceding finish kernel may still be reading this scratch
    // read back by the finish kernel
    tma_store_3d_hint(&map_p, red, tile * kRows, tb + crank * tr, ks / cs, l2_evict_last());
    bulk_commit();
    bulk_wait_read();
  }
  if (cs > 1) {
    cluster_arrive();
    cluster_wait();  // no CTA leaves while another may still read its staged tile
  }
}

struct FinParams {
  int B, ks, ncol;
  int order;                 // 1: CTAs take the sequences emitting ones first (more CTAs than SMs)
  int stage_floats;          // partial-sum rows staged per round (a multiple of ncol)
  const float* part;         // [ks][B][ncol]
  int* flag;
  const int32_t* start_pos;  // [B]
  float* state;              // [max_batch][slots][ncol]
  int slots, ratio, overlap;
  Packing pk;
  EpiParams ep;
  csa_out out;               // rows indexed by sequence
  uint8_t* emitted;          // [B], or null (the caller learns the emissions on the host)
  float* acc;                // non-overlapped: [max_batch][3][H] running max, denominator and
                             // numerator of the open group over its tokens so far
  int* acc_pos;              // [max_batch][ntiles] position of the last token in acc (-1: not valid);
                             // this kernel keeps a sequence's in its first entry
  const float* ape;          // packed gate positional bias [ratio][ncol] (zero at kv columns), or null
  long long state_elems, acc_elems;  // extents checked by the bounds-checked build
};

__device__ __forceinline__ float padded_kind_value(const Packing& pk, int col) {
  return ((col % pk.tw) / pk.ft) < pk.nk / 2 ? 0.0f : -INFINITY;  // kv kinds first, then scores
}

__device__ __forceinline__ float comp(const float4& v, int e) {
  return e == 0 ? v.x : e == 1 ? v.y : e == 2 ? v.z : v.w;
}

constexpr int kPoolUnroll = 4;          // candidates in flight per thread
constexpr int kMaxFinB = 4096;          // sequences per call (the emitting-first order is built in shared memory)
constexpr int kFinGroups = 1;           // feature groups of four per thread: H <= 4 * kFinThreads (head_dim <= 512)
constexpr int kFinColGroups = 4;        // column groups of four per thread: ncol <= 4 * 4 * kFinThreads
constexpr int kFinSmemFloats = 22528;   // dynamic shared memory (88 KB): staged partial sums + the token's row

// Waits for the phase of `parity` at most kWaitNs; false on time-out.
__device__ __forceinline__ bool wait_bounded(uint64_t* bar, uint32_t parity) {
  const uint64_t t0 = globaltimer();
  while (!mbar_try_wait(bar, parity))
    if (globaltimer() - t0 > kWaitNs) return false;
  return true;
}

// Whether the token at position p completes a group that is emitted (a position the RoPE
// table covers).
__device__ __forceinline__ bool emits(const FinParams& P, int p) {
  if (p < 0 || (p + 1) % P.ratio != 0) return false;
  return P.ep.rope_dim == 0 || (long long)p + 1 - P.ratio < P.ep.max_pos;
}

// The t-th sequence in the order "emitting sequences, then the others", each by index.  CTAs
// start in index order, so with more sequences than SMs the ones with pooling to do start
// first, beside the projection that is still running.  All threads call it; ew is shared
// scratch of (B + 31) / 32 words.
__device__ int nth_in_emit_order(const FinParams& P, int t, unsigned* ew, int* s_b) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nwarp = blockDim.x >> 5;
  const int nw = (P.B + 31) >> 5;
  for (int w = warp; w < nw; w += nwarp) {
    const int b = 32 * w + lane;
    const unsigned bal = __ballot_sync(0xffffffffu, b < P.B && emits(P, P.start_pos[b]));
    if (lane == 0) ew[w] = bal;
  }
  __syncthreads();
  if (warp == 0) {
    auto valid = [&](int w) -> unsigned {
      const int n = P.B - 32 * w;
      return n >= 32 ? 0xffffffffu : ((1u << n) - 1u);
    };
    int cnt = 0;
    for (int w = lane; w < nw; w += 32) cnt += __popc(ew[w] & valid(w));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) cnt += __shfl_xor_sync(0xffffffffu, cnt, o);
    const bool want = t < cnt;
    int r = want ? t : t - cnt;
    int found = 0;
    for (int w0 = 0; w0 < nw; w0 += 32) {
      const int w = w0 + lane;
      const unsigned bits = w < nw ? (want ? ew[w] : ~ew[w]) & valid(w) : 0u;
      const int c = __popc(bits);
      int inc = c;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, inc, o);
        if (lane >= o) inc += y;
      }
      const int tot = __shfl_sync(0xffffffffu, inc, 31);
      if (r < tot) {
        const int L = __ffs(__ballot_sync(0xffffffffu, r >= inc - c && r < inc)) - 1;
        const int rr = r - __shfl_sync(0xffffffffu, inc - c, L);
        const unsigned wb = __shfl_sync(0xffffffffu, bits, L);
        const bool mb = ((wb >> lane) & 1u) && __popc(wb & ((1u << lane) - 1u)) == rr;
        found = 32 * (w0 + L) + __ffs(__ballot_sync(0xffffffffu, mb)) - 1;
        break;
      }
      r -= tot;
    }
    if (lane == 0) *s_b = found;
  }
  __syncthreads();
  return *s_b;
}

// Pools candidates [i0, i1) for features f .. f+3 with a running maximum, into (m, den, num).
// cand(i) gives the state row and the score and kv columns of candidate i.
template <class Cand>
__device__ __forceinline__ void pool_range(const float* st, int ncol, int i0, int i1, Cand cand, float m[4],
                                           float den[4], float num[4]) {
  for (int ib = i0; ib < i1; ib += kPoolUnroll) {
    float4 sv[kPoolUnroll], kv[kPoolUnroll];
#pragma unroll
    for (int u = 0; u < kPoolUnroll; ++u) {
      const int i = ib + u;
      sv[u] = make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
      kv[u] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
      if (i < i1) {
        int srow, cs, ck;
        cand(i, srow, cs, ck);
        const float* row = st + (size_t)srow * ncol;
        sv[u] = __ldcg(reinterpret_cast<const float4*>(row + cs));
        kv[u] = __ldcg(reinterpret_cast<const float4*>(row + ck));
      }
    }
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      float cm = m[e];
#pragma unroll
      for (int u = 0; u < kPoolUnroll; ++u) cm = fmaxf(cm, comp(sv[u], e));
      if (cm == -INFINITY) continue;  // padded candidates only, so far
      const float sc = expf(m[e] - cm);  // 0 while m was -inf, 1 when the maximum is unchanged
      den[e] *= sc;
      num[e] *= sc;
#pragma unroll
      for (int u = 0; u < kPoolUnroll; ++u) {
        const float ex = expf(comp(sv[u], e) - cm);
        den[e] += ex;
        num[e] = fmaf(ex, comp(kv[u], e), num[e]);
      }
      m[e] = cm;
    }
  }
}

// One CTA per sequence; thread t takes the features of groups t, t + 128 (four adjacent
// features, i.e. four adjacent packed columns of each kind).
//
// The token of this call always completes the open group last, so every other candidate sits in
// a state slot written by work that completed before this launch could start (the projection
// before it only lets it start once its own wait has returned).  Before its wait a CTA
// therefore combines them into a running (maximum, denominator, numerator) per feature:
// overlapped (8 candidates) it pools the 7 earlier ones when the token completes a group;
// otherwise it takes the open group's running values kept from the previous call (acc), or
// rebuilds them from the state slots when they are not for the previous position.  It also
// loads the gain and RoPE factors of an emitted entry.  After the wait the sequence's rows of
// the K slices' partial sums arrive by bulk copy and are added in slice order into its state
// slot; the token is folded in, and the running values are kept (open group) or the entry
// epilogue runs (completed group: bf16, RMSNorm, RoPE, fp4).
__global__ void __launch_bounds__(kFinThreads, 5) decode_finish_kernel(const FinParams P) {
  extern __shared__ __align__(16) float fsm[];  // [stage_floats] staged rows, then [ncol] the token's row
  __shared__ __align__(8) uint64_t rbar_s;
  __shared__ float wss[kFinThreads / 32];
  __shared__ unsigned ew[kMaxFinB / 32];
  __shared__ int s_b;
  float* pst = fsm;
  float* cur = fsm + P.stage_floats;
  uint64_t* rbar = &rbar_s;

  griddep_launch_dependents();  // the next launch may take the SMs this grid leaves free
  const Packing& pk = P.pk;
  const int tid = threadIdx.x, nthr = blockDim.x, lane = tid & 31, warp = tid >> 5;
  const int ncol = P.ncol, H = pk.H, nfg = H / 4;
  if (tid == 0) {
    mbar_init(rbar, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  int b;
  if (P.order) {
    b = nth_in_emit_order(P, blockIdx.x, ew, &s_b);
  } else {
    b = blockIdx.x;
    __syncthreads();
  }
  const int p = P.start_pos[b];
  const int pp = max(p, 0);
  const int slot = P.overlap ? ((pp >> 2) & 1) * 4 + (pp & 3) : pp % P.ratio;
  const int q = (pp >> 2) & 1;
  float* st = P.state + (size_t)b * P.slots * ncol;
  const bool emit = p >= 0 && (p + 1) % P.ratio == 0;
  const long long pos = (long long)p + 1 - P.ratio;
  const bool pool = emits(P, p);
  float* acc = P.acc + (size_t)b * 3 * H;
  const int hr = P.ep.rope_dim >> 1;
  const int r0 = H - P.ep.rope_dim;  // even: H is a multiple of 16 and rope_dim is even

  // -- before the wait: the earlier candidates, as running values per feature
  float m[kFinGroups][4], den[kFinGroups][4], num[kFinGroups][4];
  float gn[kFinGroups][4], rc[kFinGroups][2], rs[kFinGroups][2];
#pragma unroll
  for (int gi = 0; gi < kFinGroups; ++gi)
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      m[gi][e] = -INFINITY;
      den[gi][e] = 0.0f;
      num[gi][e] = 0.0f;
    }
  const bool open = !P.overlap && pp % P.ratio != 0;  // running values of an open group to continue
  const bool use_acc = open && P.acc_pos[(size_t)b * pk.ntiles] == p - 1;
#pragma unroll
  for (int gi = 0; gi < kFinGroups; ++gi) {
    const int g = tid + gi * nthr;
    if (g >= nfg) continue;
    const int f = 4 * g;
    if (P.overlap) {
      if (pool)
        pool_range(st, ncol, 0, 7,
                   [&](int i, int& srow, int& cs, int& ck) {
                     const bool prevB = i < 4;  // the previous group's branch B, then this group's A
                     srow = prevB ? 4 * (1 - q) + i : 4 * q + i - 4;
                     cs = pk.col(prevB ? S_B : S_A, f);
                     ck = pk.col(prevB ? KV_B : KV_A, f);
                   },
                   m[gi], den[gi], num[gi]);
    } else if (use_acc) {
      const float4 a0 = __ldcg(reinterpret_cast<const float4*>(acc + f));
      const float4 a1 = __ldcg(reinterpret_cast<const float4*>(acc + H + f));
      const float4 a2 = __ldcg(reinterpret_cast<const float4*>(acc + 2 * H + f));
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        m[gi][e] = comp(a0, e);
        den[gi][e] = comp(a1, e);
        num[gi][e] = comp(a2, e);
      }
    } else if (open) {  // rebuild from the state slots of the open group
      pool_range(st, ncol, 0, pp % P.ratio,
                 [&](int i, int& srow, int& cs, int& ck) {
                   srow = i;
                   cs = pk.col(S, f);
                   ck = pk.col(KV, f);
                 },
                 m[gi], den[gi], num[gi]);
    }
    if (pool) {  // the epilogue's gain and RoPE factors
      const float4 gg = __ldg(reinterpret_cast<const float4*>(P.ep.gain + f));
      gn[gi][0] = gg.x;
      gn[gi][1] = gg.y;
      gn[gi][2] = gg.z;
      gn[gi][3] = gg.w;
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const int k = (f + 2 * u - r0) >> 1;
        rc[gi][u] = (hr > 0 && f + 2 * u >= r0) ? __ldg(P.ep.rope_cos + pos * hr + k) : 1.0f;
        rs[gi][u] = (hr > 0 && f + 2 * u >= r0) ? __ldg(P.ep.rope_sin + pos * hr + k) : 0.0f;
      }
    }
  }

  griddep_wait();  // the partial sums of the projection are complete

  // -- the K-slice partial sums: the sequence's row of every slice arrives by bulk copy (all in
  //    flight at once, as many slices per round as the staging holds), then thread t adds
  //    column groups t, t + 128, ... over the slices in order
  {
    const int ncg = ncol / 4;
    const int per_round = P.stage_floats / ncol;
    const float* src = P.part + (size_t)b * ncol;
    const size_t kstride = (size_t)P.B * ncol;
    float4 a[kFinColGroups];
#pragma unroll
    for (int i = 0; i < kFinColGroups; ++i) a[i] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    int round = 0;
    for (int k0 = 0; k0 < P.ks; k0 += per_round, ++round) {
      const int nr = min(per_round, P.ks - k0);
      if (tid == 0) {
        mbar_arrive_expect_tx(rbar, (uint32_t)(nr * ncol * 4));
        const uint64_t once = l2_evict_first();  // the partial sums are dead once read
        for (int r = 0; r < nr; ++r)
          bulk_load_hint(pst + r * ncol, src + (size_t)(k0 + r) * kstride, ncol * 4, rbar, once);
      }
      if (!wait_bounded(rbar, round & 1)) atomicOr(P.flag, 4);
      const float4* pst4 = reinterpret_cast<const float4*>(pst);
#pragma unroll
      for (int i = 0; i < kFinColGroups; ++i) {
        const int cg = tid + i * nthr;
        if (cg >= ncg) continue;
        for (int r0 = 0; r0 < nr; r0 += 8) {  // eight rows in flight, added in order
          float4 v[8];
#pragma unroll
          for (int u = 0; u < 8; ++u) v[u] = r0 + u < nr ? pst4[(r0 + u) * ncg + cg] : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
#pragma unroll
          for (int u = 0; u < 8; ++u) add4(a[i], v[u]);
        }
      }
      __syncthreads();  // the staging is free for the next round
    }
#pragma unroll
    for (int i = 0; i < kFinColGroups; ++i) {
      const int cg = tid + i * nthr;
      if (cg < ncg) {
        // wgate(x) + the positional bias of the token's place in its group, at the score columns
        // (a float4 never straddles two kinds: a kind spans ft >= 16 columns)
        if (P.ape && ((4 * cg) % pk.tw) / pk.ft >= pk.nk / 2)
          add4(a[i], __ldg(reinterpret_cast<const float4*>(P.ape + (size_t)(pp % P.ratio) * ncol) + cg));
        reinterpret_cast<float4*>(cur)[cg] = a[i];
        if (in_bounds((long long)((st - P.state) + (size_t)slot * ncol + 4 * cg + 3), P.state_elems, P.flag))
          reinterpret_cast<float4*>(st + (size_t)slot * ncol)[cg] = a[i];
      }
    }
  }
  // -- restart at position 0: the previous group's branch is the padded one
  if (p == 0 && P.overlap)
    for (int i = tid; i < 4 * ncol; i += nthr)
      if (in_bounds((long long)((st - P.state) + (size_t)4 * ncol + i), P.state_elems, P.flag))
        st[(size_t)4 * ncol + i] = padded_kind_value(pk, i % ncol);
  if (tid == 0) {
    if (P.emitted) P.emitted[b] = pool ? 1 : 0;
    if (p < 0) atomicOr(P.flag, 1);
    if (emit && !pool) atomicOr(P.flag, 2);
    if (!P.overlap) P.acc_pos[(size_t)b * pk.ntiles] = p >= 0 ? p : -1;
  }
  if (P.overlap && !pool) return;
  __syncthreads();  // the token's row is complete in shared memory

  // -- fold the token itself in (the last candidate); keep the running values of an open group,
  //    or finish the entry
  float pv[kFinGroups][4];
#pragma unroll
  for (int gi = 0; gi < kFinGroups; ++gi) {
    const int g = tid + gi * nthr;
    if (g >= nfg) continue;
    const int f = 4 * g;
    const float4 sc4 = *reinterpret_cast<const float4*>(cur + pk.col(P.overlap ? S_A : S, f));
    const float4 kc4 = *reinterpret_cast<const float4*>(cur + pk.col(P.overlap ? KV_A : KV, f));
    float M[4], D[4], Nn[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float sc = comp(sc4, e), kc = comp(kc4, e), mk = m[gi][e];
      M[e] = fmaxf(mk, sc);
      const float w = mk == -INFINITY ? 0.0f : expf(mk - M[e]);  // earlier candidates, rescaled
      const float ex = expf(sc - M[e]);
      D[e] = fmaf(den[gi][e], w, ex);
      Nn[e] = fmaf(num[gi][e], w, ex * kc);
      pv[gi][e] = __fdiv_rn(Nn[e], D[e]);
    }
    if (!pool && !P.overlap &&
        in_bounds((long long)((acc - P.acc) + 2 * H + f + 3), P.acc_elems, P.flag)) {  // running values for the next call
      reinterpret_cast<float4*>(acc + f)[0] = make_float4(M[0], M[1], M[2], M[3]);
      reinterpret_cast<float4*>(acc + H + f)[0] = make_float4(D[0], D[1], D[2], D[3]);
      reinterpret_cast<float4*>(acc + 2 * H + f)[0] = make_float4(Nn[0], Nn[1], Nn[2], Nn[3]);
    }
  }
  if (!pool) return;

  // -- the entry epilogue: bf16, the sum of squares over the CTA (warps, then in warp order),
  //    RMSNorm, RoPE (pairs within a thread), the fp4 round trip (a block of 16 features is
  //    four adjacent threads)
  float v[kFinGroups][4];
  float ss = 0.0f;
#pragma unroll
  for (int gi = 0; gi < kFinGroups; ++gi)
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      v[gi][e] = (tid + gi * nthr < nfg) ? bf16_round(pv[gi][e]) : 0.0f;
      ss = fmaf(v[gi][e], v[gi][e], ss);
    }
  ss = warp_sum(ss);
  if (lane == 0) wss[warp] = ss;
  __syncthreads();
  float tot = 0.0f;
  for (int w = 0; w < (nthr >> 5); ++w) tot += wss[w];
  const float inv = rms_inv(tot, P.ep);
#pragma unroll
  for (int gi = 0; gi < kFinGroups; ++gi) {
    const int g = tid + gi * nthr;
    entry_epilogue_quad(v[gi], g < nfg, 4 * g, lane, inv, gn[gi], rc[gi], rs[gi], P.ep, (size_t)b, P.out);
  }
}

}  // namespace dtc

// ---- host side ------------------------------------------------------------------------------

// Number of K slices: about one CTA per SM for a 128-token block, at least one K block per CTA.
int decode_tc_slices(const csa_compressor* c) {
  const int sms = current_sm_count();
  const int nkb = c->dim / dtc::kKb;
  int ks = sms / c->pk.ntiles;
  if (ks > nkb) ks = nkb;
  if (ks < 1) ks = 1;
  ks -= ks >= 4 ? ks % 4 : ks % 2;  // whole clusters of K slices (decode_tc_cluster)
  return ks;
}

// K slices added on chip per cluster: 4 or 2 where they divide the slices, else 1.
static int decode_tc_cluster(int ks) { return ks % 4 == 0 ? 4 : ks % 2 == 0 ? 2 : 1; }

bool decode_tc_supported(const csa_compressor* c, const void* x, int B) {
  using namespace dtc;
  return B <= kMaxFinB && c->pk.tw == kRows && c->dim % kKb == 0 && ((uintptr_t)x & 15) == 0 && c->H % 16 == 0 &&
         c->H <= 4 * kFinGroups * kFinThreads && c->pk.cols() <= 4 * kFinColGroups * kFinThreads &&
         2 * c->pk.cols() <= kFinSmemFloats && tcx::get_encode() != nullptr;
}

cudaError_t invalidate_decode_acc(const csa_compressor* c, int first, int count, cudaStream_t s) {
  if (count <= 0) return cudaSuccess;
  return cudaMemsetAsync(c->dec_acc_pos + (size_t)first * c->pk.ntiles, 0xFF,
                         (size_t)count * c->pk.ntiles * sizeof(int), s);
}

size_t decode_tc_part_bytes(const csa_compressor* c, int B) {
  return (size_t)decode_tc_slices(c) * B * c->pk.cols() * sizeof(float);
}

int decode_tc_kernels_per_call() { return 2; }

cudaError_t launch_decode_tc(csa_compressor* c, const uint16_t* x, int B, const int32_t* start_pos, float* part,
                             const csa_out& out, uint8_t* emitted, bool early_start, cudaStream_t s) {
  using namespace dtc;
  const int ks = decode_tc_slices(c);
  auto encode = tcx::get_encode();
  if (!encode) return cudaErrorNotSupported;
  const size_t smem = (size_t)kRingBytes + 1024 + 1024;
  static std::atomic<unsigned long long> attr{0};
  cudaError_t ea = tcx::once_per_device(attr, [] {
    cudaError_t e = cudaFuncSetAttribute(decode_proj_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)((size_t)kRingBytes + 1024 + 1024));
    // both kernels ask for the largest shared-memory carveout, so that finish CTAs can share an
    // SM with a projection CTA
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(decode_proj_kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                               cudaSharedmemCarveoutMaxShared);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(decode_finish_kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                               cudaSharedmemCarveoutMaxShared);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(decode_finish_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               kFinSmemFloats * (int)sizeof(float));
    return e;
  });
  if (ea != cudaSuccess) return ea;
  CUtensorMap mx;
  {
    // the tokens: [B rows][dim]; rows past B in the last 128-token block read as zeros
    cuuint64_t dims[2] = {(cuuint64_t)c->dim, (cuuint64_t)B};
    cuuint64_t strides[1] = {(cuuint64_t)c->dim * 2};
    cuuint32_t box[2] = {kKs, kTok};
    cuuint32_t es[2] = {1, 1};
    if (encode(&mx, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, (void*)x, dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  CUtensorMap mp;
  {
    // the partial sums of each cluster of K slices: [ks / cs][B][ncol] f32, stored as boxes of
    // 128 columns x 128 / cs tokens
    cuuint64_t dims[3] = {(cuuint64_t)c->pk.cols(), (cuuint64_t)B, (cuuint64_t)(ks / decode_tc_cluster(ks))};
    cuuint64_t strides[2] = {(cuuint64_t)c->pk.cols() * 4, (cuuint64_t)B * c->pk.cols() * 4};
    cuuint32_t box[3] = {kRows, (cuuint32_t)(kTok / decode_tc_cluster(ks)), 1};
    cuuint32_t es[3] = {1, 1, 1};
    if (encode(&mp, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, (void*)part, dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  cudaLaunchAttribute at[2];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  {
    ProjParams P;
    P.w = c->w_planes;
    P.nkb_total = c->dim / kKb;
    P.ks = ks;
    P.cs = decode_tc_cluster(ks);
    P.B = B;
    P.ncol = c->pk.cols();
    P.part = part;
    P.flag = c->dev_flag;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(c->pk.ntiles, ks, (B + kTok - 1) / kTok);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    at[0].val.programmaticStreamSerializationAllowed = early_start ? 1 : 0;
    at[1].id = cudaLaunchAttributeClusterDimension;
    at[1].val.clusterDim.x = 1;
    at[1].val.clusterDim.y = P.cs;
    at[1].val.clusterDim.z = 1;
    cfg.attrs = at;
    cfg.numAttrs = 2;
    cudaError_t e = cudaLaunchKernelEx(&cfg, decode_proj_kernel, mx, mp, P);
    if (e != cudaSuccess) return e;
  }
  {
    FinParams P;
    const int sms = current_sm_count();
    P.B = B;
    P.ks = ks / decode_tc_cluster(ks);  // partial sums left after the on-chip additions
    P.ncol = c->pk.cols();
    P.order = B > sms;
    P.stage_floats = min(P.ks, max(1, (kFinSmemFloats - P.ncol) / P.ncol)) * P.ncol;
    P.part = part;
    P.flag = c->dev_flag;
    P.start_pos = start_pos;
    P.state = c->state;
    P.slots = c->slots;
    P.ratio = c->ratio;
    P.overlap = c->overlap;
    P.pk = c->pk;
    P.ep = epi_params(c);
    P.out = out;
    P.emitted = emitted;
    P.acc = c->dec_acc;
    P.acc_pos = c->dec_acc_pos;
    P.ape = c->ape_set ? c->ape : nullptr;
    P.state_elems = (long long)c->opt.max_batch * c->slots * P.ncol;
    P.acc_elems = (long long)c->opt.max_batch * 3 * c->H;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(B, 1, 1);
    cfg.blockDim = dim3(kFinThreads, 1, 1);
    cfg.dynamicSmemBytes = (size_t)(P.stage_floats + P.ncol) * sizeof(float);
    cfg.stream = s;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, decode_finish_kernel, P);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace csa
