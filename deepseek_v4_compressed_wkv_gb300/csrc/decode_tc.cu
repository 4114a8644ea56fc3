// Decode on the tensor cores (sm_103a): one token per sequence, into each sequence's state slot
// ("Pool token pairs", decode branch: kv_state[:, slot] = kv, score_state[:, slot] = score),
// then the pool and epilogue of the sequences whose group completes, in one launch.
//
// Decode streams every weight once per step for only B tokens, so it is bound by HBM.  The
// kernel streams the three exact bf16 planes of the weights that set_weights prepared (w = p0 +
// p1 + p2; 6 bytes per weight, 1.5x the f32 weights) straight into the tensor cores: splitting
// the f32 weights on the CUDA cores instead (4 bytes per weight) made the kernel bound by
// instruction issue at a quarter of the HBM bandwidth.
//
// Work split: packed tile t (128 rows) x K slice, at most one CTA per SM, launched cooperatively
// so that all CTAs are resident together.  Each CTA accumulates its slice in K chunks of 128
// (TMEM, promoted to f32 registers as in the prefill kernel) and writes its partial sums to
// scratch.  The K slices of a tile then meet at a self-resetting counter barrier (a bounded
// wait), and each of them finishes a share of the tokens: it adds the slices' partials in a
// fixed order into the token's state slot (a deterministic split-K reduction), applies the
// restart at position 0, and, where the token completed a group, pools the tile's features
// ("Pool token pairs", decode branch; "Compressed Sparse Attention - ratio m = 4", decode
// rule).  The last tile to finish a sequence (a completion counter, no waiting) runs the
// entry epilogue, which needs all H features for the RMSNorm.
//
// Roles (320 threads) in the projection: warp 0 issues the TMA loads (three plane tiles and one
// token tile of K = 32 per stage, 64-byte swizzle, 6 stages), warp 1 owns TMEM and issues
// tcgen05.mma, warps 2-9 drain the chunk accumulators and store the partial sums.  All warps
// take part in the reduction and pooling.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "csa_internal.cuh"
#include "kernels.h"
#include "tc_common.cuh"

namespace csa {
namespace dtc {

using namespace tcx;

constexpr int kRows = 128;                              // packed rows per tile (MMA M)
constexpr int kTok = 128;                               // tokens per launch (MMA N)
constexpr int kKb = 64;                                 // K granularity of the slice split
constexpr int kKs = 32;                                 // K per stage (one 64-byte swizzle row of bf16)
constexpr int kStages = 6;
constexpr int kChunkSteps = 4;                          // stages per accumulator chunk (K = 128)
constexpr int kPlaneBytes = kRows * kKs * 2;            // 8 KB
constexpr int kXBytes = kTok * kKs * 2;                 // 8 KB
constexpr int kStageBytes = 3 * kPlaneBytes + kXBytes;  // 32 KB
constexpr int kRingBytes = kStages * kStageBytes;       // 192 KB
constexpr int kEpiThreads = 256;
constexpr int kThreads = 64 + kEpiThreads;
constexpr int kTmemCols = 2 * kTok;

struct Params {
  int nkb_total, ks;         // K blocks (of 64) of dim, number of K slices
  int B, b_total, b0;        // tokens in this launch, in the call, first token of this launch
  int ncol;                  // packed columns (rows of one weight plane)
  float* part;               // [ks][b_total][ncol] partial sums
  int* flag;
  const int32_t* start_pos;  // [b_total]
  float* state;              // [max_batch][slots][ncol]
  int slots, ratio, overlap;
  Packing pk;
  EpiParams ep;
  csa_out out;               // rows indexed by sequence
  uint8_t* emitted;          // [b_total]
  uint16_t* pooled;          // [b_total][H] bf16 scratch
  int* seq_ctr;              // [b_total] per-sequence tile counters (kept at zero between calls)
  unsigned* tile_ctr;        // [ntiles] barrier arrivals (kept at zero between calls)
  unsigned* tile_gen;        // [ntiles] barrier generations
};

__device__ __forceinline__ float padded_kind_value(const Packing& pk, int col) {
  return ((col % pk.tw) / pk.ft) < pk.nk / 2 ? 0.0f : -INFINITY;  // kv kinds first, then scores
}

// After the projection: meet the other K slices of this tile, then reduce, update the state and
// pool for tokens [ks*B/KS, (ks+1)*B/KS) of this launch.  `scr` is free shared memory.
__device__ void finish_tokens(const Params& P, int tile, int ks, float* scr) {
  __shared__ unsigned gen0;
  __shared__ int go;
  __threadfence();  // this CTA's partial sums are visible before it arrives
  __syncthreads();
  if (threadIdx.x == 0) {
    volatile unsigned* gen = P.tile_gen + tile;
    gen0 = *gen;
    __threadfence();
    go = 1;
    if (atomicAdd(P.tile_ctr + tile, 1u) == (unsigned)P.ks - 1) {
      P.tile_ctr[tile] = 0;  // every slice has arrived: reset for the next call, then release
      __threadfence();
      atomicAdd(P.tile_gen + tile, 1u);
    } else {
      const uint64_t t0 = globaltimer();
      while (*gen == gen0) {
        if (globaltimer() - t0 > kWaitNs) {
          atomicOr(P.flag, 4);
          go = 0;
          break;
        }
        __nanosleep(64);
      }
    }
    __threadfence();
  }
  __syncthreads();
  if (!go) return;

  const Packing& pk = P.pk;
  const int ncol = pk.cols(), c0 = tile * kRows, f0 = tile * pk.ft;
  const int tb0 = (int)((long long)ks * P.B / P.ks), tb1 = (int)((long long)(ks + 1) * P.B / P.ks);
  const int nt = tb1 - tb0;
  // -- the K-slice partials of each token into its state slot, in slice order
  for (int it = threadIdx.x; it < nt * (kRows / 4); it += blockDim.x) {
    const int b = P.b0 + tb0 + it / (kRows / 4), c = c0 + 4 * (it % (kRows / 4));
    const float* src = P.part + (size_t)b * ncol + c;
    const size_t stride = (size_t)P.b_total * ncol;
    float4 a = __ldcg(reinterpret_cast<const float4*>(src));
    for (int k = 1; k < P.ks; ++k) {
      const float4 v = __ldcg(reinterpret_cast<const float4*>(src + k * stride));
      a.x += v.x;
      a.y += v.y;
      a.z += v.z;
      a.w += v.w;
    }
    const int pp = max(P.start_pos[b], 0);
    const int slot = P.overlap ? ((pp >> 2) & 1) * 4 + (pp & 3) : pp % P.ratio;
    *reinterpret_cast<float4*>(P.state + ((size_t)b * P.slots + slot) * ncol + c) = a;
  }
  // -- restart padding, emission flags, position checks
  for (int it = threadIdx.x; it < nt; it += blockDim.x) {
    const int b = P.b0 + tb0 + it;
    const int p = P.start_pos[b];
    if (p == 0 && P.overlap)  // the previous group's branch is the padded one
      for (int i = 0; i < 4; ++i)
        for (int c = c0; c < c0 + kRows; ++c)
          P.state[((size_t)b * P.slots + 4 + i) * ncol + c] = padded_kind_value(pk, c);
    if (tile == 0) {
      const bool emit = p >= 0 && (p + 1) % P.ratio == 0;
      const long long pos = (long long)p + 1 - P.ratio;
      const bool pos_ok = P.ep.rope_dim == 0 || pos < P.ep.max_pos;
      P.emitted[b] = (emit && pos_ok) ? 1 : 0;
      if (p < 0) atomicOr(P.flag, 1);
      if (emit && !pos_ok) atomicOr(P.flag, 2);
    }
  }
  __syncthreads();  // the slots written above are read below by other threads
  // -- pool the tile's features for the tokens of this share that completed a group, in batches
  //    of up to blockDim / ft tokens at once; within a token, groups of threads split the
  //    candidates (max, then exp sums) and the group partials are merged in a fixed order
  __shared__ int elist[kTok];
  __shared__ int ne;
  __shared__ int lastv[kThreads / 32];
  if (threadIdx.x == 0) {
    int n = 0;
    for (int it = 0; it < nt; ++it) {
      const int b = P.b0 + tb0 + it;
      const int p = P.start_pos[b];
      const long long pos = (long long)p + 1 - P.ratio;
      if (p >= 0 && (p + 1) % P.ratio == 0 && (P.ep.rope_dim == 0 || pos < P.ep.max_pos)) elist[n++] = b;
    }
    ne = n;
  }
  __syncthreads();
  const int ncand = P.overlap ? 8 : P.ratio;
  const int nthr = (int)blockDim.x;
  const int epb = min(nthr / pk.ft, nthr / 32);  // tokens per batch (one epilogue warp each)
  float* sm_m = scr;
  float* sm_d = scr + nthr;
  float* sm_n = scr + 2 * nthr;
  for (int e0 = 0; e0 < ne; e0 += epb) {
    const int nbe = min(epb, ne - e0);
    const int ng = max(1, nthr / (nbe * pk.ft));  // candidate groups per token
    const int per_tok = ng * pk.ft;
    const int e = (int)threadIdx.x / per_tok, r = (int)threadIdx.x % per_tok;
    const int f = f0 + r % pk.ft, g = r / pk.ft;
    float m = -INFINITY, den = 0.0f, num = 0.0f;
    if (e < nbe) {
      const int b = elist[e0 + e];
      const int q = (P.start_pos[b] >> 2) & 1;
      const float* st = P.state + (size_t)b * P.slots * ncol;
      auto row_of = [&](int i, int& cs, int& ck) -> const float* {
        if (P.overlap) {
          const bool prevB = i < 4;
          cs = pk.col(prevB ? S_B : S_A, f);
          ck = pk.col(prevB ? KV_B : KV_A, f);
          return st + (size_t)(prevB ? 4 * (1 - q) + i : 4 * q + i - 4) * ncol;
        }
        cs = pk.col(S, f);
        ck = pk.col(KV, f);
        return st + (size_t)i * ncol;
      };
#pragma unroll 8
      for (int i = g; i < ncand; i += ng) {
        int cs, ck;
        const float* row = row_of(i, cs, ck);
        m = fmaxf(m, row[cs]);
      }
      if (m != -INFINITY) {  // a group of padded slots adds nothing
#pragma unroll 8
        for (int i = g; i < ncand; i += ng) {
          int cs, ck;
          const float* row = row_of(i, cs, ck);
          const float ex = expf(row[cs] - m);
          den += ex;
          num = fmaf(ex, row[ck], num);
        }
      }
    }
    sm_m[threadIdx.x] = m;
    sm_d[threadIdx.x] = den;
    sm_n[threadIdx.x] = num;
    __syncthreads();
    if (e < nbe && g == 0) {
      const int base = e * per_tok + r;
      float M = -INFINITY;
      for (int k = 0; k < ng; ++k) M = fmaxf(M, sm_m[base + k * pk.ft]);
      float D = 0.0f, Nn = 0.0f;
      for (int k = 0; k < ng; ++k) {
        const int t = base + k * pk.ft;
        if (sm_m[t] == -INFINITY) continue;
        const float w = expf(sm_m[t] - M);
        D = fmaf(sm_d[t], w, D);
        Nn = fmaf(sm_n[t], w, Nn);
      }
      P.pooled[(size_t)elist[e0 + e] * pk.H + f] = bf16_bits(__fdiv_rn(Nn, D));
    }
    __threadfence();
    __syncthreads();
    if ((int)threadIdx.x < nbe)
      lastv[threadIdx.x] = atomicAdd(&P.seq_ctr[elist[e0 + threadIdx.x]], 1) == pk.ntiles - 1;
    __syncthreads();
    // the last tile of a sequence runs its RMSNorm, RoPE and fp4: warp w takes token e0 + w
    const int w = (int)threadIdx.x >> 5, lane = (int)threadIdx.x & 31;
    if (w < nbe && lastv[w]) {
      __threadfence();
      const int b = elist[e0 + w];
      const long long pos = (long long)P.start_pos[b] + 1 - P.ratio;
      const int l = min(lane, (pk.H >> 4) - 1);
      const uint4* src = reinterpret_cast<const uint4*>(P.pooled + (size_t)b * pk.H + 16 * l);
      const uint4 a = __ldcg(src), c = __ldcg(src + 1);
      const uint32_t wd[8] = {a.x, a.y, a.z, a.w, c.x, c.y, c.z, c.w};
      float v[16];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        v[2 * i] = __uint_as_float(wd[i] << 16);
        v[2 * i + 1] = __uint_as_float(wd[i] & 0xFFFF0000u);
      }
      const size_t H = pk.H;
      entry_epilogue(v, lane, pos, P.ep, P.out.latent + b * H, P.out.codes ? P.out.codes + b * (H / 2) : nullptr,
                     P.out.scales ? P.out.scales + b * (H / 16) : nullptr,
                     P.out.prequant ? P.out.prequant + b * H : nullptr);
      if (lane == 0) P.seq_ctr[b] = 0;  // ready for the next call
    }
    __syncthreads();
  }
}

__global__ void __launch_bounds__(kThreads, 1)
    decode_tc_kernel(const __grid_constant__ CUtensorMap map_w, const __grid_constant__ CUtensorMap map_x,
                     const Params P) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint64_t* full = (uint64_t*)(smem + kRingBytes);
  uint64_t* empty = full + kStages;
  uint64_t* c_full = empty + kStages;
  uint64_t* c_empty = c_full + 2;
  uint32_t* tmem_slot = (uint32_t*)(c_empty + 2);
  volatile int* abort_flag = (volatile int*)(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int tile = blockIdx.x, ks = blockIdx.y;
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
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    prefetch_map(&map_w);
    prefetch_map(&map_x);
  }
  if (warp == 1) tmem_alloc(tmem_slot, kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      for (int t = 0; t < nstep; ++t) {
        const int s = t % kStages;
        if (t >= kStages && !mbar_wait(&empty[s], ((t / kStages) - 1) & 1, abort_flag)) break;
        uint8_t* st = smem + s * kStageBytes;
        mbar_arrive_expect_tx(&full[s], kStageBytes);
        for (int p = 0; p < 3; ++p)
          tma_load_2d(st + p * kPlaneBytes, &map_w, k0 + t * kKs, p * P.ncol + tile * kRows, &full[s]);
        tma_load_2d(st + 3 * kPlaneBytes, &map_x, k0 + t * kKs, 0, &full[s]);
      }
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
    // drain each chunk into f32 registers, in chunk order; then store the partial sums
    const int q = warp & 3, h = (warp - 2) >> 2;
    const int row = 32 * q + lane;
    float acc[kTok / 2];
#pragma unroll
    for (int i = 0; i < kTok / 2; ++i) acc[i] = 0.0f;
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
    if (!ok && threadIdx.x == 64) atomicOr(P.flag, 4);
    float* dst = P.part + ((size_t)ks * P.b_total + P.b0) * P.ncol + tile * kRows + row;
#pragma unroll
    for (int i = 0; i < kTok / 2; ++i) {
      const int b = (kTok / 2) * h + i;
      if (b < P.B) dst[(size_t)b * P.ncol] = acc[i];
    }
  }

  tc_fence_before();
  __syncthreads();
  if (*abort_flag && threadIdx.x == 0) atomicOr(P.flag, 4);
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
  // the ring is free: every stage was consumed by MMAs that completed before the last chunk
  finish_tokens(P, tile, ks, (float*)smem);
}

}  // namespace dtc

// ---- host side ------------------------------------------------------------------------------

// Number of K slices: at most one CTA per SM (the launch is cooperative), at least one K block
// per CTA.
int decode_tc_slices(const csa_compressor* c) {
  static int sms = 0;
  if (!sms) {
    int dev = 0;
    cudaGetDevice(&dev);
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0) sms = 148;
  }
  const int nkb = c->dim / dtc::kKb;
  int ks = sms / c->pk.ntiles;
  if (ks < 1) ks = 1;
  if (ks > nkb) ks = nkb;
  return ks;
}

bool decode_tc_supported(const csa_compressor* c, const void* x) {
  return c->pk.tw == dtc::kRows && c->dim % dtc::kKb == 0 && ((uintptr_t)x & 15) == 0 &&
         c->pk.ntiles <= 148 && tcx::get_encode() != nullptr;
}

cudaError_t launch_decode_tc(const csa_compressor* c, const uint16_t* x, int B, const int32_t* start_pos,
                             float* part, int ks, const csa_out& out, uint8_t* emitted, cudaStream_t s) {
  using namespace dtc;
  auto encode = tcx::get_encode();
  if (!encode) return cudaErrorNotSupported;
  const size_t smem = (size_t)kRingBytes + 1024 + 1024;
  static bool attr = false;
  if (!attr) {
    cudaError_t e = cudaFuncSetAttribute(decode_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    attr = true;
  }
  CUtensorMap mw;
  {
    // the three bf16 weight planes: [3 * ncol rows][dim], K innermost
    cuuint64_t dims[2] = {(cuuint64_t)c->dim, (cuuint64_t)3 * c->pk.cols()};
    cuuint64_t strides[1] = {(cuuint64_t)c->dim * 2};
    cuuint32_t box[2] = {kKs, kRows};
    cuuint32_t es[2] = {1, 1};
    if (encode(&mw, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, (void*)c->w_planes, dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  for (int b0 = 0; b0 < B; b0 += kTok) {
    const int nb = min(kTok, B - b0);
    CUtensorMap mx;
    cuuint64_t dims[2] = {(cuuint64_t)c->dim, (cuuint64_t)nb};
    cuuint64_t strides[1] = {(cuuint64_t)c->dim * 2};
    cuuint32_t box[2] = {kKs, kTok};
    cuuint32_t es[2] = {1, 1};
    if (encode(&mx, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, (void*)(x + (size_t)b0 * c->dim), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
    Params P;
    P.nkb_total = c->dim / kKb;
    P.ks = ks;
    P.B = nb;
    P.b_total = B;
    P.b0 = b0;
    P.ncol = c->pk.cols();
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
    P.pooled = c->dec_pooled;
    P.seq_ctr = c->dec_counters;
    P.tile_ctr = c->dec_tile_ctr;
    P.tile_gen = c->dec_tile_gen;
    // the K slices of a tile wait for each other: a cooperative launch keeps the grid resident
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(c->pk.ntiles, ks, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeCooperative;
    at[0].val.cooperative = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, decode_tc_kernel, mw, mx, P);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace csa
