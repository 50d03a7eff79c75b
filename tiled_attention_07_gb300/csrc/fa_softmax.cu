// fa_softmax.cu -- row-wise softmax with the online max / sum recurrence.
//
// "Puzzles 8 Long Softmax": z_ij = softmax_j(x_i1, ..., x_iT), stabilised by
// subtracting the row max; the loop that finds the max and the loop that sums
// the exponentials are merged by rescaling the running sum when the running
// max grows: for a running max m1 with sum s and a new max m2 > m1,
// sum' = sum * exp(m1 - m2) + sum_j exp(x_j - m2).  exp is taken as exp2 of
// log2(e) x, as the puzzle recommends.
//
// GB300 design: the row is cut into C <= 16 slices of about 64 KB, one CTA
// each, launched as one thread-block cluster per row.  A CTA brings its slice
// into shared memory with one bulk asynchronous copy (cp.async.bulk on an
// mbarrier), keeps a running (max, sum) per thread over it, merges the
// threads' pairs with the same rescaling, then merges the CTAs' pairs through
// distributed shared memory.  It writes z over its slice in shared memory and
// stores it with one bulk copy back to global memory, so every element crosses
// HBM once in and once out.  Slices longer than the on-chip limit are streamed
// from global memory: one pass for the (max, sum), a second read for z.
#include "../../include/fa.h"
#include "ptx.cuh"

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <math_constants.h>

#include <algorithm>
#include <limits>

namespace fa {
namespace {

constexpr int kThreads = 256;
constexpr int kTargetSliceBytes = 64 * 1024;   // slice size aimed at: three CTAs per SM
constexpr int kMaxSliceBytes = 192 * 1024;     // the most one CTA holds on chip
constexpr int kMaxCluster = 16;                // 8 is portable; 16 where the GPU can schedule it
constexpr uint32_t kBulkChunk = 32768;         // bytes per bulk copy instruction
constexpr float kLog2e = 1.4426950408889634f;

struct SoftmaxParams {
  const void* x;
  void* z;
  float* lse;
  int rows, T;
  int64_t xs, zs;   // row strides, elements
  int C;            // CTAs (cluster size) per row
  int per;          // elements per slice, a multiple of 8
  bool resident;    // slice fits the shared-memory buffer
};

// Running (max, sum of exp(x - max)) pair and the rescaling merge of two of
// them.  An empty pair is (-inf, 0).
struct Stat {
  float m, s;
};

__device__ __forceinline__ Stat merge_stat(Stat a, Stat b) {
  const float m = fmaxf(a.m, b.m);
  if (m == -CUDART_INF_F) return Stat{m, 0.f};
  const float sa = a.m == -CUDART_INF_F ? 0.f : a.s * ex2_approx((a.m - m) * kLog2e);
  const float sb = b.m == -CUDART_INF_F ? 0.f : b.s * ex2_approx((b.m - m) * kLog2e);
  return Stat{m, sa + sb};
}

// Folds n values into a running pair: the rescaling step once per group.
template <int N>
__device__ __forceinline__ Stat fold(Stat st, const float (&v)[N]) {
  float vm = v[0];
#pragma unroll
  for (int i = 1; i < N; ++i) vm = fmaxf(vm, v[i]);
  const float m = fmaxf(st.m, vm);
  if (m == -CUDART_INF_F) return st;
  float s = st.m == -CUDART_INF_F ? 0.f : st.s * ex2_approx((st.m - m) * kLog2e);
  // (x - m) first: exact for x near m, so large logits keep their precision
#pragma unroll
  for (int i = 0; i < N; ++i) s += ex2_approx((v[i] - m) * kLog2e);
  return Stat{m, s};
}

// 16-byte vectors of the element type, widened to / narrowed from float32.
template <typename E>
struct Vec;
template <>
struct Vec<float> {
  static constexpr int N = 4;
  static __device__ __forceinline__ void load(const void* p, float (&v)[4]) {
    const float4 w = *reinterpret_cast<const float4*>(p);
    v[0] = w.x;
    v[1] = w.y;
    v[2] = w.z;
    v[3] = w.w;
  }
  static __device__ __forceinline__ void store(void* p, const float (&v)[4]) {
    *reinterpret_cast<float4*>(p) = make_float4(v[0], v[1], v[2], v[3]);
  }
  static __device__ __forceinline__ float get(const void* p, int i) { return reinterpret_cast<const float*>(p)[i]; }
  static __device__ __forceinline__ void put(void* p, int i, float x) { reinterpret_cast<float*>(p)[i] = x; }
};
template <bool BF16>
struct Vec16 {
  static constexpr int N = 8;
  static __device__ __forceinline__ float widen(uint16_t h) {
    if constexpr (BF16) {
      return __uint_as_float(static_cast<uint32_t>(h) << 16);
    } else {
      return __half2float(__ushort_as_half(h));
    }
  }
  static __device__ __forceinline__ void load(const void* p, float (&v)[8]) {
    const uint4 w = *reinterpret_cast<const uint4*>(p);
    const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      v[2 * i] = widen(static_cast<uint16_t>(u[i] & 0xffffu));
      v[2 * i + 1] = widen(static_cast<uint16_t>(u[i] >> 16));
    }
  }
  static __device__ __forceinline__ void store(void* p, const float (&v)[8]) {
    uint4 w;
    w.x = pack2<BF16>(v[0], v[1]);
    w.y = pack2<BF16>(v[2], v[3]);
    w.z = pack2<BF16>(v[4], v[5]);
    w.w = pack2<BF16>(v[6], v[7]);
    *reinterpret_cast<uint4*>(p) = w;
  }
  static __device__ __forceinline__ float get(const void* p, int i) {
    return widen(reinterpret_cast<const uint16_t*>(p)[i]);
  }
  static __device__ __forceinline__ void put(void* p, int i, float x) {
    const uint32_t w = pack2<BF16>(x, 0.f);
    reinterpret_cast<uint16_t*>(p)[i] = static_cast<uint16_t>(w & 0xffffu);
  }
};
template <>
struct Vec<__half> : Vec16<false> {};
template <>
struct Vec<__nv_bfloat16> : Vec16<true> {};

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_arrive() { asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory"); }
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory"); }
// A float2 from the shared memory of CTA `rank` of this cluster.
__device__ __forceinline__ float2 ld_cluster_f2(const void* local, uint32_t rank) {
  uint32_t remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_u32(local)), "r"(rank));
  float2 v;
  asm volatile("ld.shared::cluster.v2.f32 {%0, %1}, [%2];" : "=f"(v.x), "=f"(v.y) : "r"(remote) : "memory");
  return v;
}

// (max, sum) of the whole CTA from each thread's pair.
template <int THREADS>
__device__ __forceinline__ Stat block_stat(Stat st, Stat* red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    Stat o;
    o.m = __shfl_xor_sync(0xffffffffu, st.m, off);
    o.s = __shfl_xor_sync(0xffffffffu, st.s, off);
    st = merge_stat(st, o);
  }
  if (lane == 0) red[warp] = st;
  __syncthreads();
  Stat r = red[0];
  for (int w = 1; w < THREADS / 32; ++w) r = merge_stat(r, red[w]);
  __syncthreads();
  return r;
}

template <typename E, int THREADS>
__global__ void __launch_bounds__(THREADS) softmax_rows_kernel(const SoftmaxParams p) {
  using V = Vec<E>;
  constexpr int N = V::N;
  extern __shared__ __align__(128) uint8_t sm[];   // the slice, in the input type
  __shared__ uint64_t bar;
  __shared__ Stat red[THREADS / 32];
  __shared__ float2 cta_stat;   // this CTA's (max, sum), read by the rest of the cluster

  const int rank = p.C > 1 ? static_cast<int>(cluster_rank()) : 0;
  const int row = static_cast<int>(blockIdx.x) / p.C;
  const int c0 = rank * p.per;
  const int c1 = min(p.T, c0 + p.per);
  const int n = max(0, c1 - c0);
  const int nv = n / N;   // whole 16-byte vectors; only the last slice has a tail
  const uint8_t* xr = reinterpret_cast<const uint8_t*>(p.x) + (static_cast<int64_t>(row) * p.xs + c0) * sizeof(E);
  uint8_t* zr = reinterpret_cast<uint8_t*>(p.z) + (static_cast<int64_t>(row) * p.zs + c0) * sizeof(E);

  // The slice in bytes: a 16-byte multiple by bulk copy, the rest (the last
  // slice's < 16-byte tail) through registers.
  const uint32_t nbytes = static_cast<uint32_t>(n) * sizeof(E);
  const uint32_t bulk = nbytes & ~15u;
  const int t0 = static_cast<int>(bulk / sizeof(E));
  if (p.resident) {
    if (threadIdx.x == 0) {
      mbar_init(&bar, 1);
      fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x == 0 && bulk > 0) {
      mbar_arrive_expect_tx(&bar, bulk);
      for (uint32_t off = 0; off < bulk; off += kBulkChunk)
        bulk_load(sm + off, xr + off, min(kBulkChunk, bulk - off), &bar);
    }
    for (int e = t0 + threadIdx.x; e < n; e += THREADS)
      reinterpret_cast<E*>(sm)[e] = reinterpret_cast<const E*>(xr)[e];
    if (bulk > 0) mbar_wait_drain(&bar, 0);   // the copy always completes
    __syncthreads();
  }
  const uint8_t* src = p.resident ? sm : xr;

  // pass 1: running (max, sum) per thread
  Stat st{-CUDART_INF_F, 0.f};
  for (int i = threadIdx.x; i < nv; i += THREADS) {
    float v[N];
    V::load(src + static_cast<size_t>(i) * 16, v);
    st = fold<N>(st, v);
  }
  for (int e = nv * N + threadIdx.x; e < n; e += THREADS) {
    const float v1[1] = {V::get(src, e)};
    st = fold<1>(st, v1);
  }
  Stat tot = block_stat<THREADS>(st, red);
  if (p.C > 1) {
    if (threadIdx.x == 0) cta_stat = make_float2(tot.m, tot.s);
    cluster_arrive();
    cluster_wait();
    Stat all{-CUDART_INF_F, 0.f};
    for (int r = 0; r < p.C; ++r) {
      const float2 o = ld_cluster_f2(&cta_stat, static_cast<uint32_t>(r));
      all = merge_stat(all, Stat{o.x, o.y});
    }
    tot = all;
    cluster_arrive();   // this CTA is done reading the others' statistics
  }
  if (rank == 0 && threadIdx.x == 0 && p.lse != nullptr) p.lse[row] = tot.m + logf(tot.s);

  // pass 2: z = exp(x - max) / sum, over the slice in shared memory (then one
  // bulk store) or straight to global memory when streaming
  const float inv = 1.f / tot.s;
  const float mx = tot.m;
  uint8_t* dst = p.resident ? sm : zr;
  for (int i = threadIdx.x; i < nv; i += THREADS) {
    float v[N];
    V::load(src + static_cast<size_t>(i) * 16, v);
#pragma unroll
    for (int e = 0; e < N; ++e) v[e] = ex2_approx((v[e] - mx) * kLog2e) * inv;
    V::store(dst + static_cast<size_t>(i) * 16, v);
  }
  for (int e = nv * N + threadIdx.x; e < n; e += THREADS) V::put(dst, e, ex2_approx((V::get(src, e) - mx) * kLog2e) * inv);
  if (p.resident) {
    fence_proxy_async_smem();   // z in shared memory, visible to the bulk copy
    __syncthreads();
    if (threadIdx.x == 0 && bulk > 0) {
      for (uint32_t off = 0; off < bulk; off += kBulkChunk) bulk_store(zr + off, sm + off, min(kBulkChunk, bulk - off));
      bulk_commit_group();
    }
    for (int e = t0 + threadIdx.x; e < n; e += THREADS)
      reinterpret_cast<E*>(zr)[e] = reinterpret_cast<const E*>(sm)[e];
    if (threadIdx.x == 0 && bulk > 0) bulk_wait_group0();   // shared memory is read before the CTA exits
  }
  // No CTA may exit while another still reads its shared memory.
  if (p.C > 1) cluster_wait();
}

template <typename E, int THREADS>
cudaError_t launch_softmax_t(SoftmaxParams p, cudaStream_t stream) {
  auto kern = softmax_rows_kernel<E, THREADS>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kMaxSliceBytes);
  if (e != cudaSuccess) return e;
  const int C = p.C;
  auto slice = [&](int c) {
    const int64_t per = (static_cast<int64_t>(p.T) + c - 1) / c;
    p.C = c;
    p.per = static_cast<int>((per + 7) / 8 * 8);
    p.resident = static_cast<int64_t>(p.per) * sizeof(E) <= kMaxSliceBytes;
  };
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  auto config = [&]() {
    cfg.gridDim = dim3(static_cast<unsigned>(static_cast<long long>(p.rows) * p.C));
    cfg.blockDim = dim3(THREADS);
    cfg.dynamicSmemBytes = p.resident ? static_cast<size_t>(p.per) * sizeof(E) : 0;
    cfg.stream = stream;
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(p.C);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
  };
  slice(C);
  if (C > 8) {
    // A cluster of more than 8 CTAs is not portable: use it only where this
    // GPU can schedule one with this much shared memory.
    int n_clusters = 0;
    config();
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess ||
        cudaOccupancyMaxActiveClusters(&n_clusters, kern, &cfg) != cudaSuccess || n_clusters < 1) {
      (void)cudaGetLastError();
      slice(8);
    }
  }
  config();
  return cudaLaunchKernelEx(&cfg, kern, p);
}

// Slices of about kTargetSliceBytes over a cluster of up to kMaxCluster CTAs.
template <typename E>
cudaError_t launch_softmax(SoftmaxParams p, cudaStream_t stream) {
  const int64_t row_bytes = static_cast<int64_t>(p.T) * sizeof(E);
  p.C = static_cast<int>(std::min<int64_t>(kMaxCluster, (row_bytes + kTargetSliceBytes - 1) / kTargetSliceBytes));
  // 256 threads measured fastest for both 64 KB and 128 KB slices (512 and
  // 1024 were slower on GB300).
  return launch_softmax_t<E, kThreads>(p, stream);
}

}  // namespace
}  // namespace fa

extern "C" fa_status fa_softmax_rows(const void* x, void* z, float* lse, int rows, int T, int64_t x_row_stride,
                                     int64_t z_row_stride, fa_dtype dtype, void* stream) {
  using namespace fa;
  if (dtype != FA_FP32 && dtype != FA_FP16 && dtype != FA_BF16) return FA_ERR_UNSUPPORTED;
  if (rows < 0 || T < 1) return FA_ERR_INVALID_ARG;
  if (rows == 0) return FA_OK;
  const int64_t esz = dtype == FA_FP32 ? 4 : 2;
  auto aligned = [](const void* ptr) { return ptr != nullptr && (reinterpret_cast<uintptr_t>(ptr) & 15u) == 0; };
  if (!aligned(x) || !aligned(z)) return FA_ERR_INVALID_ARG;
  if (lse != nullptr && (reinterpret_cast<uintptr_t>(lse) & 3u) != 0) return FA_ERR_INVALID_ARG;
  if (x_row_stride < T || z_row_stride < T) return FA_ERR_INVALID_ARG;
  // Each tensor's byte span, (rows - 1) * stride + T elements, must fit in int64.
  const int64_t max_stride = (std::numeric_limits<int64_t>::max() / esz - T) / std::max(rows - 1, 1);
  if (x_row_stride > max_stride || z_row_stride > max_stride) return FA_ERR_INVALID_ARG;
  if ((x_row_stride * esz) % 16 != 0 || (z_row_stride * esz) % 16 != 0) return FA_ERR_INVALID_ARG;
  if (static_cast<int64_t>(rows) * kMaxCluster > 0x7fffffffLL) return FA_ERR_INVALID_ARG;
  // z may only alias x exactly (in place): every element is read before the
  // same thread writes it, and no thread reads another's elements.
  const uintptr_t xb = reinterpret_cast<uintptr_t>(x);
  const uintptr_t zb = reinterpret_cast<uintptr_t>(z);
  const int64_t xspan = ((static_cast<int64_t>(rows) - 1) * x_row_stride + T) * esz;
  const int64_t zspan = ((static_cast<int64_t>(rows) - 1) * z_row_stride + T) * esz;
  const bool overlap = xb < zb + static_cast<uintptr_t>(zspan) && zb < xb + static_cast<uintptr_t>(xspan);
  if (overlap && !(xb == zb && x_row_stride == z_row_stride)) return FA_ERR_INVALID_ARG;

  SoftmaxParams p;
  p.x = x;
  p.z = z;
  p.lse = lse;
  p.rows = rows;
  p.T = T;
  p.xs = x_row_stride;
  p.zs = z_row_stride;
  cudaError_t e;
  switch (dtype) {
    case FA_FP32: e = launch_softmax<float>(p, static_cast<cudaStream_t>(stream)); break;
    case FA_FP16: e = launch_softmax<__half>(p, static_cast<cudaStream_t>(stream)); break;
    default: e = launch_softmax<__nv_bfloat16>(p, static_cast<cudaStream_t>(stream)); break;
  }
  return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}
