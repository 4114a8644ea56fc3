// Decode projection on the tensor cores (sm_103a): one token per sequence, written straight
// into each sequence's state slot ("Pool token pairs", decode branch: kv_state[:, slot] =
// kv, score_state[:, slot] = score).  The pool and epilogue of the sequences whose group
// completes run afterwards in decode_emit_kernel.
//
// Decode streams every weight once per step for only B tokens, so it is bound by HBM: the
// f32 weights are read once (4 bytes each) and split into three exact bf16 planes in shared
// memory by the CUDA cores, which the tensor cores then multiply with the bf16 tokens.
//
// Work split: packed tile t (128 rows) x K slice.  The K slices of one tile form a thread-block
// cluster; each CTA accumulates its slice in K chunks of 128 (TMEM, promoted to f32 registers
// as in the prefill kernel), then the cluster reduces the partial sums through distributed
// shared memory in a fixed order, each CTA owning 128 / cluster-size tokens, and writes them
// to the state.
//
// Roles (320 threads): warp 0 lane 0 streams weight tiles (TMA, 3-stage ring), warp 0 lane 1
// streams token tiles, warp 1 owns TMEM and issues tcgen05.mma, warps 2-9 split the weights
// into bf16 planes, drain the chunk accumulators and run the reduction.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "csa_internal.cuh"
#include "kernels.h"
#include "tc_common.cuh"

namespace csa {
namespace dtc {

using namespace tcx;

constexpr int kRows = 128;                       // packed rows per tile (MMA M)
constexpr int kTok = 128;                        // tokens per launch (MMA N)
constexpr int kKb = 64;                          // K per block
constexpr int kWStages = 3;                      // f32 weight ring
constexpr int kMStages = 2;                      // bf16 planes + token ring
constexpr int kChunkKb = 2;                      // K blocks per accumulator chunk
constexpr int kWBytes = kRows * kKb * 4;         // 32 KB
constexpr int kPlaneBytes = kRows * kKb * 2;     // 16 KB
constexpr int kXBytes = kTok * kKb * 2;          // 16 KB
constexpr int kMBytes = 3 * kPlaneBytes + kXBytes;  // 64 KB
constexpr int kRingBytes = kWStages * kWBytes + kMStages * kMBytes;  // 224 KB
constexpr int kEpiThreads = 256;
constexpr int kThreads = 64 + kEpiThreads;
constexpr int kTmemCols = 2 * kTok;
constexpr int kMaxCluster = 16;

struct Params {
  int K, ks_kb;          // dim, K blocks per CTA
  int B, ncol, slots, ratio, overlap;
  const int32_t* start_pos;
  float* state;
  int* flag;
};

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

__device__ __forceinline__ uint32_t cluster_size() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
  return r;
}

__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ uint32_t mapa(uint32_t saddr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
  return r;
}

__device__ __forceinline__ void st_cluster_v4(uint32_t addr, float a, float b, float c, float d) {
  asm volatile("st.shared::cluster.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "f"(a), "f"(b), "f"(c), "f"(d)
               : "memory");
}

__device__ __forceinline__ uint32_t bf16x2_bits(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

__global__ void __launch_bounds__(kThreads, 1)
    decode_tc_kernel(const __grid_constant__ CUtensorMap map_w, const __grid_constant__ CUtensorMap map_x,
                     const Params P) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint8_t* wring = smem;                               // [kWStages][128 rows][64] f32, row-major
  uint8_t* mring = smem + kWStages * kWBytes;          // [kMStages]{3 planes, x}, 128-byte swizzle
  uint64_t* w_full = (uint64_t*)(smem + kRingBytes);
  uint64_t* w_empty = w_full + kWStages;
  uint64_t* m_full = w_empty + kWStages;
  uint64_t* m_empty = m_full + kMStages;
  uint64_t* c_full = m_empty + kMStages;
  uint64_t* c_empty = c_full + 2;
  uint32_t* tmem_slot = (uint32_t*)(c_empty + 2);
  volatile int* abort_flag = (volatile int*)(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int tile = blockIdx.x;
  const uint32_t crank = cluster_rank(), csize = cluster_size();
  const int kb_base = (int)crank * P.ks_kb;
  const int nkb = P.ks_kb;
  const int nch = (nkb + kChunkKb - 1) / kChunkKb;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kWStages; ++s) {
      mbar_init(&w_full[s], 1);
      mbar_init(&w_empty[s], kEpiThreads / 32);
    }
    for (int m = 0; m < kMStages; ++m) {
      mbar_init(&m_full[m], kEpiThreads / 32 + 1);
      mbar_init(&m_empty[m], 1);
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

  float acc[kTok / 2];
#pragma unroll
  for (int i = 0; i < kTok / 2; ++i) acc[i] = 0.0f;

  if (warp == 0) {
    if (lane == 0) {  // weights: HBM -> f32 ring
      for (int kb = 0; kb < nkb; ++kb) {
        const int s = kb % kWStages;
        if (kb >= kWStages && !mbar_wait(&w_empty[s], ((kb / kWStages) - 1) & 1, abort_flag)) break;
        mbar_arrive_expect_tx(&w_full[s], kWBytes);
        tma_load_2d(wring + s * kWBytes, &map_w, (kb_base + kb) * kKb, tile * kRows, &w_full[s]);
      }
    } else if (lane == 1) {  // tokens: -> x slot of the MMA ring
      for (int kb = 0; kb < nkb; ++kb) {
        const int m = kb % kMStages;
        if (kb >= kMStages && !mbar_wait(&m_empty[m], ((kb / kMStages) - 1) & 1, abort_flag)) break;
        mbar_arrive_expect_tx(&m_full[m], kXBytes);
        tma_load_2d(mring + m * kMBytes + 3 * kPlaneBytes, &map_x, (kb_base + kb) * kKb, 0, &m_full[m]);
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
        const int kb0 = c * kChunkKb, kb1 = min(nkb, kb0 + kChunkKb);
        for (int kb = kb0; kb < kb1; ++kb) {
          const int m = kb % kMStages;
          if (!mbar_wait(&m_full[m], (kb / kMStages) & 1, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t st = smem_addr(mring + m * kMBytes);
          const uint32_t xs = st + 3 * kPlaneBytes;
          for (int p = 0; p < 3; ++p)
            for (int k = 0; k < kKb / 16; ++k)
              mma_bf16(d, sw128_desc(st + p * kPlaneBytes + k * 32), sw128_desc(xs + k * 32), idesc,
                       (kb != kb0 || p != 0 || k != 0) ? 1u : 0u);
          mma_commit(&m_empty[m]);
        }
        if (ok) mma_commit(&c_full[buf]);
      }
    }
  } else {
    const int et = threadIdx.x - 64;  // 0..255
    const int q = warp & 3, h = (warp - 2) >> 2;
    bool ok = true;
    int drained = 0;
    auto drain = [&](int c) {  // add chunk c into the f32 registers
      const int buf = c & 1;
      if (!mbar_wait(&c_full[buf], (c >> 1) & 1, abort_flag)) return false;
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
      return true;
    };
    for (int kb = 0; kb < nkb && ok; ++kb) {
      const int s = kb % kWStages, m = kb % kMStages;
      if (!mbar_wait(&w_full[s], (kb / kWStages) & 1, abort_flag)) {
        ok = false;
        break;
      }
      if (kb >= kMStages && !mbar_wait(&m_empty[m], ((kb / kMStages) - 1) & 1, abort_flag)) {
        ok = false;
        break;
      }
      // split 128 x 64 f32 weights into three bf16 planes, K-major with the 128-byte swizzle:
      // element (r, k) at r*128 + ((k/8) ^ (r%8))*16 + (k%8)*2
      const float4* src = (const float4*)(wring + s * kWBytes);
      uint8_t* planes = mring + m * kMBytes;
#pragma unroll 4
      for (int it = 0; it < kWBytes / 16 / kEpiThreads; ++it) {
        const int idx = it * kEpiThreads + et;  // float4 index: row idx/16, k 4*(idx%16)
        const float4 w = src[idx];
        const int r = idx >> 4, k = (idx & 15) * 4;
        const float wv[4] = {w.x, w.y, w.z, w.w};
        float r1[4], r2[4];
        uint32_t p0[2], p1[2], p2[2];
#pragma unroll
        for (int e = 0; e < 4; e += 2) {
          p0[e / 2] = bf16x2_bits(wv[e], wv[e + 1]);
          r1[e] = wv[e] - __uint_as_float(p0[e / 2] << 16);
          r1[e + 1] = wv[e + 1] - __uint_as_float(p0[e / 2] & 0xFFFF0000u);
          p1[e / 2] = bf16x2_bits(r1[e], r1[e + 1]);
          r2[e] = r1[e] - __uint_as_float(p1[e / 2] << 16);
          r2[e + 1] = r1[e + 1] - __uint_as_float(p1[e / 2] & 0xFFFF0000u);
          p2[e / 2] = bf16x2_bits(r2[e], r2[e + 1]);
        }
        const int off = r * 128 + ((((k >> 3) ^ (r & 7))) << 4) + (k & 7) * 2;
        *(uint2*)(planes + off) = make_uint2(p0[0], p0[1]);
        *(uint2*)(planes + kPlaneBytes + off) = make_uint2(p1[0], p1[1]);
        *(uint2*)(planes + 2 * kPlaneBytes + off) = make_uint2(p2[0], p2[1]);
      }
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&w_empty[s]);
        mbar_arrive(&m_full[m]);
      }
      // drain chunk c once the chunk after it has been fed (keeps one chunk of slack)
      if ((kb % kChunkKb) == kChunkKb - 1 && kb >= 2 * kChunkKb - 1) {
        if (!drain(drained)) ok = false;
        ++drained;
      }
    }
    while (ok && drained < nch) {
      if (!drain(drained)) ok = false;
      ++drained;
    }
    if (!ok && threadIdx.x == 64) atomicOr(P.flag, 4);
  }

  // ---- cluster reduction of the K-slice partial sums (every thread of every CTA takes part)
  tc_fence_before();
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  __syncthreads();
  cluster_sync();  // all CTAs of the cluster are past their main loops: ring memory is free
  const int w = kTok / (int)csize;  // tokens owned per CTA
  float* recv = (float*)smem;       // [csize][128 rows][w]
  if (warp >= 2) {
    const int q = warp & 3, h = (warp - 2) >> 2;
    const int row = 32 * q + lane;
    const uint32_t base = smem_addr(recv);
#pragma unroll
    for (int i = 0; i < kTok / 2; i += 4) {
      const int t = (kTok / 2) * h + i;  // first of 4 tokens; w >= 8 keeps them in one owner
      const uint32_t dst = (uint32_t)(t / w);
      const uint32_t off = (uint32_t)(((crank * kRows + row) * w + (t % w)) * 4);
      st_cluster_v4(mapa(base + off, dst), acc[i], acc[i + 1], acc[i + 2], acc[i + 3]);
    }
  }
  cluster_sync();
  // each CTA sums its w tokens over the cluster (in rank order) and writes the state slots
  for (int o = threadIdx.x; o < kRows * w; o += kThreads) {
    const int row = o % kRows, tl = o / kRows;
    const int b = (int)crank * w + tl;
    if (b >= P.B) continue;
    float v = 0.0f;
    for (uint32_t src = 0; src < csize; ++src) v += recv[((int)src * kRows + row) * w + tl];
    const int p = max(P.start_pos[b], 0);
    const int slot = P.overlap ? ((p >> 2) & 1) * 4 + (p & 3) : p % P.ratio;
    P.state[((size_t)b * P.slots + slot) * P.ncol + tile * kRows + row] = v;
  }
  tc_fence_before();
  __syncthreads();
  if (*abort_flag && threadIdx.x == 0) atomicOr(P.flag, 4);
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace dtc

// ---- host side ------------------------------------------------------------------------------

// Cluster size (K slices per packed tile) for a launch: a power of two that divides the K
// blocks, keeps at least 2 K blocks per CTA, and brings the CTA count near the SM count.
static int pick_cluster(const csa_compressor* c) {
  const int nkb = c->dim / dtc::kKb;
  int ks = 1;
  while (ks * 2 <= dtc::kMaxCluster && nkb % (ks * 2) == 0 && nkb / (ks * 2) >= 2 && c->pk.ntiles * ks * 2 <= 160)
    ks *= 2;
  return ks;
}

bool decode_tc_supported(const csa_compressor* c, const void* x) {
  return c->pk.tw == dtc::kRows && c->dim % dtc::kKb == 0 && ((uintptr_t)x & 15) == 0 &&
         tcx::get_encode() != nullptr;
}

cudaError_t launch_decode_tc(const csa_compressor* c, const uint16_t* x, int B, const int32_t* start_pos,
                             cudaStream_t s) {
  using namespace dtc;
  auto encode = tcx::get_encode();
  if (!encode) return cudaErrorNotSupported;
  static int ks_cached = 0;
  const size_t smem = (size_t)kRingBytes + 1024 + 1024;
  static bool attr = false;
  if (!attr) {
    cudaError_t e = cudaFuncSetAttribute(decode_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(decode_tc_kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
    attr = true;
  }
  int ks = pick_cluster(c);
  // a cluster of 16 is beyond the portable size: use it only if the GPU can place one
  while (ks > 8) {
    cudaLaunchConfig_t q = {};
    q.gridDim = dim3(c->pk.ntiles, ks, 1);
    q.blockDim = dim3(kThreads, 1, 1);
    q.dynamicSmemBytes = smem;
    cudaLaunchAttribute a;
    a.id = cudaLaunchAttributeClusterDimension;
    a.val.clusterDim.x = 1;
    a.val.clusterDim.y = ks;
    a.val.clusterDim.z = 1;
    q.attrs = &a;
    q.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, decode_tc_kernel, &q) == cudaSuccess && n > 0) break;
    cudaGetLastError();
    ks /= 2;
  }
  (void)ks_cached;
  CUtensorMap mw;
  {
    cuuint64_t dims[2] = {(cuuint64_t)c->dim, (cuuint64_t)c->pk.cols()};
    cuuint64_t strides[1] = {(cuuint64_t)c->dim * 4};
    cuuint32_t box[2] = {kKb, kRows};
    cuuint32_t es[2] = {1, 1};
    if (encode(&mw, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, (void*)c->w_packed, dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  for (int b0 = 0; b0 < B; b0 += kTok) {
    const int nb = min(kTok, B - b0);
    CUtensorMap mx;
    cuuint64_t dims[2] = {(cuuint64_t)c->dim, (cuuint64_t)nb};
    cuuint64_t strides[1] = {(cuuint64_t)c->dim * 2};
    cuuint32_t box[2] = {kKb, kTok};
    cuuint32_t es[2] = {1, 1};
    if (encode(&mx, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, (void*)(x + (size_t)b0 * c->dim), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
    Params P;
    P.K = c->dim;
    P.ks_kb = c->dim / kKb / ks;
    P.B = nb;
    P.ncol = c->pk.cols();
    P.slots = c->slots;
    P.ratio = c->ratio;
    P.overlap = c->overlap;
    P.start_pos = start_pos + b0;
    P.state = c->state + (size_t)b0 * c->slots * c->pk.cols();
    P.flag = c->dev_flag;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(c->pk.ntiles, ks, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr_c[1];
    attr_c[0].id = cudaLaunchAttributeClusterDimension;
    attr_c[0].val.clusterDim.x = 1;
    attr_c[0].val.clusterDim.y = ks;
    attr_c[0].val.clusterDim.z = 1;
    cfg.attrs = attr_c;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, decode_tc_kernel, mw, mx, P);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace csa
