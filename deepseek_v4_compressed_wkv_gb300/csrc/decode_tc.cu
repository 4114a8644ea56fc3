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
//    partial sums.  Roles (320 threads): warp 0 issues the TMA loads (three plane tiles and one
//    token tile of K = 32 per stage, 64-byte swizzle, 6 stages), warp 1 owns TMEM and issues
//    tcgen05.mma, warps 2-9 drain the chunk accumulators and store the partial sums.  The
//    weights are not written by any kernel that can precede a decode launch in early-start
//    mode, so warp 0 fetches the first stages' weight tiles (and prefetches the rest of the
//    slice into L2) before it waits for the preceding kernel; the tokens, and every write,
//    come after that wait.
//
//  * decode_finish_kernel, one CTA per (sequence, chunk of 128 features): adds the K slices'
//    partial sums in slice order (a deterministic split-K reduction) into the token's state
//    slot, applies the restart at position 0, and where the token completed a group pools the
//    chunk's features over the group's candidates ("Pool token pairs", decode branch;
//    "Compressed Sparse Attention - ratio m = 4", decode rule).  The last chunk of a token to
//    finish (a completion counter; nothing waits) runs the entry epilogue (bf16, RMSNorm, RoPE,
//    fp4), which needs all features.
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
constexpr int kChunkSteps = 4;                          // stages per accumulator chunk (K = 128)
constexpr int kPlaneBytes = kRows * kKs * 2;            // 8 KB
constexpr int kXBytes = kTok * kKs * 2;                 // 8 KB
constexpr int kStageBytes = 3 * kPlaneBytes + kXBytes;  // 32 KB
constexpr int kRingBytes = kStages * kStageBytes;       // 192 KB
constexpr int kEpiThreads = 256;
constexpr int kThreads = 64 + kEpiThreads;
constexpr int kTmemCols = 2 * kTok;
constexpr int kFinThreads = 256;

struct ProjParams {
  int nkb_total, ks;  // K blocks (of 64) of dim, number of K slices
  int B;              // tokens of the call
  int ncol;           // packed columns (rows of one weight plane)
  float* part;        // [ks][B][ncol] partial sums
  int* flag;
};

__global__ void __launch_bounds__(kThreads, 1)
    decode_proj_kernel(const __grid_constant__ CUtensorMap map_w, const __grid_constant__ CUtensorMap map_x,
                       const ProjParams P) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint64_t* full = (uint64_t*)(smem + kRingBytes);
  uint64_t* empty = full + kStages;
  uint64_t* c_full = empty + kStages;
  uint64_t* c_empty = c_full + 2;
  uint32_t* tmem_slot = (uint32_t*)(c_empty + 2);
  volatile int* abort_flag = (volatile int*)(tmem_slot + 1);

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
      const int npre = min(nstep, kStages);
      const int wrow = tile * kRows;
      // weights of the first stages into the ring, the rest of the slice into L2
      for (int t = 0; t < npre; ++t) {
        uint8_t* st = smem + t * kStageBytes;
        mbar_arrive_expect_tx(&full[t], kStageBytes);
        for (int p = 0; p < 3; ++p)
          tma_load_2d(st + p * kPlaneBytes, &map_w, k0 + t * kKs, p * P.ncol + wrow, &full[t]);
      }
      for (int t = npre; t < nstep; ++t)
        for (int p = 0; p < 3; ++p) tma_prefetch_l2_2d(&map_w, k0 + t * kKs, p * P.ncol + wrow);
      griddep_wait();  // the tokens may come from the preceding kernel
      griddep_launch_dependents();
      for (int t = 0; t < npre; ++t)
        tma_load_2d(smem + t * kStageBytes + 3 * kPlaneBytes, &map_x, k0 + t * kKs, tb, &full[t]);
      for (int t = npre; t < nstep; ++t) {
        const int s = t % kStages;
        if (!mbar_wait(&empty[s], ((t / kStages) - 1) & 1, abort_flag)) break;
        uint8_t* st = smem + s * kStageBytes;
        mbar_arrive_expect_tx(&full[s], kStageBytes);
        for (int p = 0; p < 3; ++p)
          tma_load_2d(st + p * kPlaneBytes, &map_w, k0 + t * kKs, p * P.ncol + wrow, &full[s]);
        tma_load_2d(st + 3 * kPlaneBytes, &map_x, k0 + t * kKs, tb, &full[s]);
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
    griddep_wait();  // the preceding finish kernel may still be reading this scratch
    float* dst = P.part + ((size_t)ks * P.B + tb) * P.ncol + tile * kRows + row;
    const int nb = min(kTok, P.B - tb);
#pragma unroll
    for (int i = 0; i < kTok / 2; ++i) {
      const int b = (kTok / 2) * h + i;
      if (b < nb) dst[(size_t)b * P.ncol] = acc[i];
    }
  }

  tc_fence_before();
  __syncthreads();
  if (*abort_flag && threadIdx.x == 0) atomicOr(P.flag, 4);
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

struct FinParams {
  int B, ks, ncol;
  int fc, nchunk;            // features per chunk (whole tiles), chunks per token
  const float* part;         // [ks][B][ncol]
  int* flag;
  const int32_t* start_pos;  // [B]
  float* state;              // [max_batch][slots][ncol]
  int slots, ratio, overlap;
  Packing pk;
  EpiParams ep;
  csa_out out;               // rows indexed by sequence
  uint8_t* emitted;          // [B]
  float* pooled;             // [B][H] pooled values of the emitting tokens
  int* seq_ctr;              // [B] chunks done (kept at zero between calls)
};

__device__ __forceinline__ float padded_kind_value(const Packing& pk, int col) {
  return ((col % pk.tw) / pk.ft) < pk.nk / 2 ? 0.0f : -INFINITY;  // kv kinds first, then scores
}

__device__ __forceinline__ void add4(float4& a, const float4& v) {
  a.x += v.x;
  a.y += v.y;
  a.z += v.z;
  a.w += v.w;
}

__device__ __forceinline__ float comp(const float4& v, int e) {
  return e == 0 ? v.x : e == 1 ? v.y : e == 2 ? v.z : v.w;
}

constexpr int kFinChunk = 128;  // features per finish CTA (a whole number of packed tiles)
constexpr int kPoolUnroll = 4;  // candidates in flight per thread

// One CTA per (sequence b, chunk j of kFinChunk features): the chunk's packed columns are the
// contiguous range [j * cw, (j + 1) * cw), cw = fc * nk.
__global__ void __launch_bounds__(kFinThreads, 4) decode_finish_kernel(const FinParams P) {
  __shared__ float sm_m[8 * kFinChunk], sm_d[8 * kFinChunk], sm_n[8 * kFinChunk];
  __shared__ int last;
  griddep_launch_dependents();  // the next launch may take the SMs this grid leaves free
  griddep_wait();               // the partial sums of the projection are complete

  const Packing& pk = P.pk;
  const int b = blockIdx.x, j = blockIdx.y, tid = threadIdx.x, nthr = blockDim.x;
  const int ncol = P.ncol, cw = P.fc * pk.nk, c0 = j * cw;
  const int p = P.start_pos[b];
  const int pp = max(p, 0);
  const int slot = P.overlap ? ((pp >> 2) & 1) * 4 + (pp & 3) : pp % P.ratio;
  float* st = P.state + (size_t)b * P.slots * ncol;

  // -- the K-slice partial sums, in slice order, into the state slot
  {
    const float* src = P.part + (size_t)b * ncol + c0;
    const size_t kstride = (size_t)P.B * ncol;
    for (int i = tid; i < cw / 4; i += nthr) {
      const float* s0 = src + 4 * i;
      float4 a = __ldcg(reinterpret_cast<const float4*>(s0));
      int k = 1;
      for (; k + 4 <= P.ks; k += 4) {
        float4 v[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) v[u] = __ldcg(reinterpret_cast<const float4*>(s0 + (k + u) * kstride));
#pragma unroll
        for (int u = 0; u < 4; ++u) add4(a, v[u]);
      }
      for (; k < P.ks; ++k) add4(a, __ldcg(reinterpret_cast<const float4*>(s0 + k * kstride)));
      *reinterpret_cast<float4*>(st + (size_t)slot * ncol + c0 + 4 * i) = a;
    }
  }
  // -- restart at position 0: the previous group's branch is the padded one
  if (p == 0 && P.overlap)
    for (int i = tid; i < 4 * cw; i += nthr) {
      const int r = i / cw, c = c0 + i % cw;
      st[(size_t)(4 + r) * ncol + c] = padded_kind_value(pk, c);
    }
  const bool emit = p >= 0 && (p + 1) % P.ratio == 0;
  const long long pos = (long long)p + 1 - P.ratio;
  const bool pos_ok = P.ep.rope_dim == 0 || pos < P.ep.max_pos;
  if (tid == 0 && j == 0) {
    P.emitted[b] = (emit && pos_ok) ? 1 : 0;
    if (p < 0) atomicOr(P.flag, 1);
    if (emit && !pos_ok) atomicOr(P.flag, 2);
  }
  if (!(emit && pos_ok)) return;
  __threadfence();
  __syncthreads();  // the slot written above is one of the candidates

  // -- pool: thread (g, fg) takes features f0 + 4fg .. +3 (four adjacent columns of one kind)
  //    over its contiguous share of the candidates with a running maximum; the shares are
  //    merged in a fixed order
  const int fc = P.fc, nfg = fc / 4, f0 = j * fc;
  const int ncand = P.overlap ? 8 : P.ratio;
  const int ng = max(1, min(min(nthr / nfg, 8), ncand));
  const int g = tid / nfg, f = f0 + 4 * (tid % nfg);
  if (g < ng) {
    const int i0 = (int)((long long)g * ncand / ng), i1 = (int)((long long)(g + 1) * ncand / ng);
    const int q = (pp >> 2) & 1;
    float m[4], den[4], num[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      m[e] = -INFINITY;
      den[e] = 0.0f;
      num[e] = 0.0f;
    }
    for (int ib = i0; ib < i1; ib += kPoolUnroll) {
      float4 sv[kPoolUnroll], kv[kPoolUnroll];
#pragma unroll
      for (int u = 0; u < kPoolUnroll; ++u) {
        const int i = ib + u;
        sv[u] = make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
        kv[u] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        if (i < i1) {
          int srow, cs, ck;
          if (P.overlap) {
            const bool prevB = i < 4;  // the previous group's branch B, then this group's branch A
            srow = prevB ? 4 * (1 - q) + i : 4 * q + i - 4;
            cs = pk.col(prevB ? S_B : S_A, f);
            ck = pk.col(prevB ? KV_B : KV_A, f);
          } else {
            srow = i;
            cs = pk.col(S, f);
            ck = pk.col(KV, f);
          }
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
    const int o = g * fc + (f - f0);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      sm_m[o + e] = m[e];
      sm_d[o + e] = den[e];
      sm_n[o + e] = num[e];
    }
  }
  __syncthreads();
  for (int ff = tid; ff < fc; ff += nthr) {
    float M = -INFINITY;
    for (int k = 0; k < ng; ++k) M = fmaxf(M, sm_m[k * fc + ff]);
    float D = 0.0f, Nn = 0.0f;
    for (int k = 0; k < ng; ++k) {
      const float mk = sm_m[k * fc + ff];
      if (mk == -INFINITY) continue;  // a share of padded candidates adds nothing
      const float w = expf(mk - M);
      D = fmaf(sm_d[k * fc + ff], w, D);
      Nn = fmaf(sm_n[k * fc + ff], w, Nn);
    }
    P.pooled[(size_t)b * pk.H + f0 + ff] = __fdiv_rn(Nn, D);
  }
  __threadfence();
  __syncthreads();
  if (tid == 0) last = atomicAdd(P.seq_ctr + b, 1) == P.nchunk - 1;
  __syncthreads();
  // -- the last chunk of the token runs the entry epilogue, one warp: lane l holds features
  //    16l..16l+15
  if (last && tid < 32) {
    __threadfence();
    const int H = pk.H;
    const int l = min(tid, (H >> 4) - 1);
    const float4* src = reinterpret_cast<const float4*>(P.pooled + (size_t)b * H + 16 * l);
    float v[16];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const float4 a = __ldcg(src + u);
      v[4 * u] = a.x;
      v[4 * u + 1] = a.y;
      v[4 * u + 2] = a.z;
      v[4 * u + 3] = a.w;
    }
    const size_t Hs = H;
    entry_epilogue(v, tid, pos, P.ep, P.out.latent + b * Hs, P.out.codes ? P.out.codes + b * (Hs / 2) : nullptr,
                   P.out.scales ? P.out.scales + b * (Hs / 16) : nullptr,
                   P.out.prequant ? P.out.prequant + b * Hs : nullptr);
    if (tid == 0) P.seq_ctr[b] = 0;  // ready for the next call
  }
}

}  // namespace dtc

// ---- host side ------------------------------------------------------------------------------

// Number of K slices: about one CTA per SM for a 128-token block, at least one K block per CTA.
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
  const int fc = c->H < dtc::kFinChunk ? c->H : dtc::kFinChunk;
  return c->pk.tw == dtc::kRows && c->dim % dtc::kKb == 0 && ((uintptr_t)x & 15) == 0 && c->H % 16 == 0 &&
         c->H % fc == 0 && fc % c->pk.ft == 0 && tcx::get_encode() != nullptr;
}

cudaError_t launch_decode_tc(const csa_compressor* c, const uint16_t* x, int B, const int32_t* start_pos,
                             float* part, int ks, const csa_out& out, uint8_t* emitted, bool early_start,
                             cudaStream_t s) {
  using namespace dtc;
  auto encode = tcx::get_encode();
  if (!encode) return cudaErrorNotSupported;
  const size_t smem = (size_t)kRingBytes + 1024 + 1024;
  static bool attr = false;
  if (!attr) {
    cudaError_t e = cudaFuncSetAttribute(decode_proj_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    attr = true;
  }
  CUtensorMap mw, mx;
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
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  {
    ProjParams P;
    P.nkb_total = c->dim / kKb;
    P.ks = ks;
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
    cfg.attrs = at;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, decode_proj_kernel, mw, mx, P);
    if (e != cudaSuccess) return e;
  }
  {
    FinParams P;
    P.B = B;
    P.ks = ks;
    P.ncol = c->pk.cols();
    P.fc = c->H < kFinChunk ? c->H : kFinChunk;
    P.nchunk = c->H / P.fc;
    P.pooled = c->dec_pooled;
    P.seq_ctr = c->dec_counters;
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
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(B, P.nchunk, 1);
    cfg.blockDim = dim3(kFinThreads, 1, 1);
    cfg.dynamicSmemBytes = 0;
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
