// fa_bwd.cu -- recompute-based FlashAttention-2 backward for sm_103a.
//
// "[CS336] Assignment 2: Systems", "FlashAttention V2 / High level" and
// "Backward Pass": with the saved LSE L and D = rowsum(O o dO) precomputed in
// global memory, the backward needs no stored P:
//   P_ij = exp(S_ij - L_i),  dV = P^T dO,  dP = dO V^T,  dS = P o (dP - D),
//   dQ = sm_scale dS K,  dK = sm_scale dS^T Q.
// dQ accumulates along key tiles and dK/dV along query tiles, so (as on that
// page) the work is split into two passes that each recompute P:
//   bwd_pre_kernel   D_i and -L_i * log2(e) per query row into the workspace
//                    (padded to whole 128-row tiles: D = 0, -L = -inf)
//   dkdv_kernel      one CTA per 128-key tile, loop over query tiles:
//                    S^T = K Q_i^T, dP^T = V dO_i^T (TMEM), P^T and dS^T by
//                    sixteen elementwise warps, dV += P^T dO_i, dK += dS^T Q_i
//   dq_kernel        one CTA per 128-query tile, loop over key tiles:
//                    S = Q K_j^T, dP = dO V_j^T, dS, dQ += dS K_j
// At d = 64 the library also has a single-pass form (the "fused" backward):
//   dkdv_kernel<.., FUSED>  as dkdv_kernel, and besides dK and dV it forms
//                    each query tile's share of dQ, dQ_i += dS_i K (dS_i
//                    written to shared memory by the elementwise warps, the
//                    product into TMEM), and adds it into a float32 dQ
//                    accumulator in the workspace with vector reductions;
//   dq_convert_kernel  dQ = sm_scale * accumulator, in the input type.
// It computes the five products of the recompute equations instead of the
// two passes' seven, at the cost of the reductions into L2; the order of the
// float32 additions into dQ then varies from run to run (dQ is not bitwise
// deterministic, dK and dV are).
// P is exp2(c S - L log2 e) with c = sm_scale log2(e) ("Fused Attention 2":
// exp2 with the scale folded by log2 e).  P^T and dS^T (dS) are rounded to the
// input type and written back into the TMEM columns they were computed from,
// where they are the A operand of the next tcgen05.mma.
// Causal: only query/key tile pairs on or below the diagonal are visited; only
// the diagonal tile is masked.
#include "fa_internal.h"
#include "ptx.cuh"

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <math_constants.h>

namespace fa {
namespace {

constexpr int kT = 128;                  // rows per query / key tile
constexpr float kLog2e = 1.4426950408889634f;

__device__ __forceinline__ const uint8_t* row_ptr(const void* base, int64_t sb, int64_t sh, int64_t ss, int b,
                                                  int h, int r) {
  return reinterpret_cast<const uint8_t*>(base) +
         2 * (static_cast<int64_t>(b) * sb + static_cast<int64_t>(h) * sh + static_cast<int64_t>(r) * ss);
}

// 16-bit pair -> two fp32
template <bool BF16>
__device__ __forceinline__ float2 unpack2(uint32_t w) {
  float2 f;
  if constexpr (BF16) {
    f.x = __uint_as_float(w << 16);
    f.y = __uint_as_float(w & 0xffff0000u);
  } else {
    __half2 hh = *reinterpret_cast<__half2*>(&w);
    f = __half22float2(hh);
  }
  return f;
}

// ---------------------------------------------------------------------------
// D = rowsum(O o dO), nL = -LSE * log2(e), padded per (b, h) to Nqp rows
// ---------------------------------------------------------------------------
struct PreParams {
  const void* o;
  int64_t o_sb, o_sh, o_ss;
  const void* dout;
  int64_t d_sb, d_sh, d_ss;
  const float* lse;
  float* wsD;
  float* wsL;
  float* dqacc;   // fused backward: float32 dQ accumulator rows, zeroed here (else null)
  int B, H, Nq, Nqp, d;
};

template <bool BF16>
__global__ void __launch_bounds__(256) bwd_pre_kernel(const PreParams p) {
  const long long gid = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 3;
  const int sub = threadIdx.x & 7;
  const long long total = static_cast<long long>(p.B) * p.H * p.Nqp;
  const bool active = gid < total;
  const long long row = active ? gid : 0;
  const int bh = static_cast<int>(row / p.Nqp);
  const int q = static_cast<int>(row % p.Nqp);
  const int b = bh / p.H;
  const int h = bh % p.H;
  const bool valid = active && q < p.Nq;
  float acc = 0.f;
  if (valid) {
    // 16-byte vectors of the row, at most two per lane (d <= 128), all
    // loaded before the first product so that a row costs one round trip
    const int nv = p.d / 8;
    const uint4* po = reinterpret_cast<const uint4*>(row_ptr(p.o, p.o_sb, p.o_sh, p.o_ss, b, h, q));
    const uint4* pd = reinterpret_cast<const uint4*>(row_ptr(p.dout, p.d_sb, p.d_sh, p.d_ss, b, h, q));
    uint4 a[2] = {}, g[2] = {};
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      if (sub + 8 * i < nv) {
        a[i] = __ldg(po + sub + 8 * i);
        g[i] = __ldg(pd + sub + 8 * i);
      }
    }
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const uint32_t aw[4] = {a[i].x, a[i].y, a[i].z, a[i].w};
      const uint32_t gw[4] = {g[i].x, g[i].y, g[i].z, g[i].w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 fa = unpack2<BF16>(aw[e]);
        const float2 fg = unpack2<BF16>(gw[e]);
        acc = fmaf(fa.x, fg.x, acc);
        acc = fmaf(fa.y, fg.y, acc);
      }
    }
  }
  acc += __shfl_xor_sync(0xffffffffu, acc, 4);
  acc += __shfl_xor_sync(0xffffffffu, acc, 2);
  acc += __shfl_xor_sync(0xffffffffu, acc, 1);
  if (active && sub == 0) {
    p.wsD[row] = valid ? acc : 0.f;
    p.wsL[row] = valid ? -p.lse[static_cast<long long>(bh) * p.Nq + q] * kLog2e : -CUDART_INF_F;
  }
  if (active && p.dqacc != nullptr) {
    float4* z = reinterpret_cast<float4*>(p.dqacc + row * p.d);
    for (int c = sub; c < p.d / 4; c += 8) z[c] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
}

// zero dK and dV when there are no queries
template <int D>
__global__ void zero_rows_kernel(void* x, int64_t sb, int64_t sh, int64_t ss, int B, int H, int N) {
  const long long r = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (r >= static_cast<long long>(B) * H * N) return;
  const int n = static_cast<int>(r % N);
  const int bh = static_cast<int>(r / N);
  uint4* dst = reinterpret_cast<uint4*>(const_cast<uint8_t*>(row_ptr(x, sb, sh, ss, bh / H, bh % H, n)));
#pragma unroll
  for (int c = 0; c < D / 8; ++c) dst[c] = make_uint4(0, 0, 0, 0);
}

// ---------------------------------------------------------------------------
// shared pieces of the two main kernels
// ---------------------------------------------------------------------------
template <int D>
struct BwdCfg {
  using G = TileGeo<D>;
  static constexpr int TILE = G::TILE;
  static constexpr int EW_WARPS = 16;   // 4 warpgroups x 32 columns of the 128-wide tile
  static constexpr int THREADS = EW_WARPS * 32 + 96;   // + producer + 2 MMA issuers
  static constexpr int PROD_WARP = EW_WARPS;
  static constexpr int MMA_WARP = EW_WARPS + 1;   // issuer A (also allocates TMEM); issuer B follows
  // dK/dV: K, V resident; ring of (Q_i, dO_i, L_i, D_i)
  static constexpr int KV_NSTAGE = D == 64 ? 5 : (D == 80 ? 3 : 2);
  static constexpr int KV_STAGE = 2 * TILE + 2 * 512;
  static constexpr int KV_SMEM = 1024 + 2 * TILE + KV_NSTAGE * KV_STAGE + 512;
  // fused dK/dV/dQ (d = 64): two ring stages less than dK/dV alone, to make
  // room for the 128 x 128 16-bit dS tile and the 128 x 64 float32 dQ tile
  static constexpr int KVQ_NSTAGE = KV_NSTAGE - 2;
  static constexpr int DS_TILE = 128 * 128 * 2;
  static constexpr int DQ_TILE = 128 * D * 4;
  static constexpr int KVQ_SMEM = 1024 + 2 * TILE + KVQ_NSTAGE * KV_STAGE + DS_TILE + DQ_TILE + 512;
  static_assert(D != 64 || KVQ_SMEM <= 227 * 1024, "the fused layout's shared memory");
  // dQ: Q, dO resident; ring of (K_j, V_j)
  static constexpr int Q_NSTAGE = D == 64 ? 5 : (D == 80 ? 3 : 2);
  static constexpr int Q_STAGE = 2 * TILE;
  static constexpr int Q_SMEM = 1024 + 2 * TILE + Q_NSTAGE * Q_STAGE + 512;
};

// TMEM column of the A operand for K-step ks (16 elements) when the 16-bit
// matrix was written by four warpgroups, each packing its 32 columns into the
// first 16 columns of its own 32-column quarter.
__device__ __forceinline__ uint32_t split_a_col(int ks) { return (ks >> 1) * 32 + (ks & 1) * 8; }

// M = 128 x N = 128 x K = 16 KS (default: D), both operands K-major in
// swizzled tiles.  KS > D / 16 takes in the tiles' padding columns too.
template <int D, int KS = D / 16>
__device__ __forceinline__ void mma_nt(uint32_t d_tmem, uint32_t a_addr, uint32_t b_addr, uint32_t idesc) {
  using G = TileGeo<D>;
  static_assert(16 * KS <= G::NCH * G::CC, "K-steps beyond the tile");
  const uint64_t ad0 = make_sdesc(a_addr, 16, G::SBO, G::LAYOUT);
  const uint64_t bd0 = make_sdesc(b_addr, 16, G::SBO, G::LAYOUT);
#pragma unroll
  for (int ks = 0; ks < KS; ++ks) {
    const uint32_t off = (ks / G::KPC) * G::CHB + (ks % G::KPC) * 32;
    if (elect_one()) umma_ss(d_tmem, desc_add(ad0, off), desc_add(bd0, off), idesc, ks > 0);
  }
}

// D(128 x D) (+)= A(TMEM, 128 x 128) * B(128 x D, MN-major tile of 128 rows).
// A is either split over four 32-column quarters (split_a_col) or packed
// contiguously (8 columns per K-step).
template <int D, bool kContiguousA = false>
__device__ __forceinline__ void mma_tn(uint32_t d_tmem, uint32_t a_tmem, uint32_t b_addr, uint32_t idesc,
                                       bool acc) {
  using G = TileGeo<D>;
  const uint64_t bd0 = make_sdesc(b_addr, G::CHB, G::SBO, G::LAYOUT);
#pragma unroll
  for (int ks = 0; ks < 8; ++ks) {
    const uint32_t acol = kContiguousA ? static_cast<uint32_t>(ks * 8) : split_a_col(ks);
    if (elect_one()) umma_ts(d_tmem, a_tmem + acol, desc_add(bd0, ks * 16 * G::ROWB), idesc, (acc || ks > 0) ? 1u : 0u);
  }
}

// D(128 x D) = A(128 x 128) * B(128 x D), both MN-major tiles in shared
// memory: A a 128-column tile (two 64-column chunks; M along its columns, K
// along its rows), B a tile of D columns (N along its columns, K along its
// rows).  Used for dQ_i = dS_i K with dS_i stored keys x queries.
template <int D>
__device__ __forceinline__ void mma_mn_mn(uint32_t d_tmem, uint32_t a_addr, uint32_t b_addr, uint32_t idesc) {
  using GA = TileGeo<128>;
  using G = TileGeo<D>;
  const uint64_t ad0 = make_sdesc(a_addr, GA::CHB, GA::SBO, GA::LAYOUT);
  const uint64_t bd0 = make_sdesc(b_addr, G::CHB, G::SBO, G::LAYOUT);
#pragma unroll
  for (int ks = 0; ks < 8; ++ks)
    if (elect_one()) umma_ss(d_tmem, desc_add(ad0, ks * 16 * GA::ROWB), desc_add(bd0, ks * 16 * G::ROWB), idesc, ks > 0);
}

// Folding L and D into the GEMMs (bf16, d = 80): the tiles of d = 80 carry
// 16 zero-filled padding columns [80, 96).  With 1 in columns 80 and 81 of K
// and V, and a two-term bf16 split of -L log2(e) / c and of -D in columns 80
// and 81 of Q_i and dO_i, the padded GEMMs give
//   K Q_i^T (96 columns) = S^T - L log2(e) / c,   V dO_i^T = dP^T - D,
// so that P^T = exp2(c (S^T)') and dS^T = P^T o (dP^T)': the elementwise
// warps read no L or D.  The split a = bf16(v), b = bf16(v - a) keeps v to
// about 2^-16 relatively; v = -inf (padded query rows) gives a = -inf, b = 0.
// The write goes to (row r, columns 80-81) of a tile stored as 32-column
// chunks with 64-byte rows and the 64-byte swizzle: chunk 2, 16-byte granule
// 2 ^ ((r / 2) % 4) of row r.
constexpr int kFoldKSteps = 6;

__device__ __forceinline__ uint32_t* fold_slot(uint8_t* tile, int r) {
  using G = TileGeo<80>;
  return reinterpret_cast<uint32_t*>(tile + 2 * G::CHB + r * G::ROWB + ((2 ^ ((r >> 1) & 3)) << 4));
}

__device__ __forceinline__ uint32_t bf16_split(float v) {
  if (!(v > -CUDART_INF_F)) return pack2<true>(v, 0.f);   // -inf: (-inf, 0)
  const float a = __bfloat162float(__float2bfloat16_rn(v));
  return pack2<true>(a, v - a);
}

struct MainParams {
  int B, H, Nq, Nk, Nqp;
  int causal;
  float scale_log2;   // sm_scale * log2(e)
  float sm_scale;
  const float* wsD;
  const float* wsL;
  void* out0;         // dkdv: dV   dq: dQ
  int64_t o0_sb, o0_sh, o0_ss;
  void* out1;         // dkdv: dK
  int64_t o1_sb, o1_sh, o1_ss;
  float* dqacc;       // fused dkdv: float32 dQ accumulator [B*H][Nqp][D]
  int* err;
};

// Store 16 fp32 TMEM columns of this thread's row, times `scale`, as 16-bit.
template <bool BF16>
__device__ __forceinline__ void store16(uint8_t* dst, const uint32_t (&v)[16], float scale) {
  uint4 w0, w1;
  w0.x = pack2<BF16>(__uint_as_float(v[0]) * scale, __uint_as_float(v[1]) * scale);
  w0.y = pack2<BF16>(__uint_as_float(v[2]) * scale, __uint_as_float(v[3]) * scale);
  w0.z = pack2<BF16>(__uint_as_float(v[4]) * scale, __uint_as_float(v[5]) * scale);
  w0.w = pack2<BF16>(__uint_as_float(v[6]) * scale, __uint_as_float(v[7]) * scale);
  w1.x = pack2<BF16>(__uint_as_float(v[8]) * scale, __uint_as_float(v[9]) * scale);
  w1.y = pack2<BF16>(__uint_as_float(v[10]) * scale, __uint_as_float(v[11]) * scale);
  w1.z = pack2<BF16>(__uint_as_float(v[12]) * scale, __uint_as_float(v[13]) * scale);
  w1.w = pack2<BF16>(__uint_as_float(v[14]) * scale, __uint_as_float(v[15]) * scale);
  reinterpret_cast<uint4*>(dst)[0] = w0;
  reinterpret_cast<uint4*>(dst)[1] = w1;
}

// ---------------------------------------------------------------------------
// dK / dV: one CTA per (key tile, b, h)
// ---------------------------------------------------------------------------
// TMEM columns: [0,128) S^T, [128,256) dP^T -> dS^T, then dV and dK (D
// columns each).  With d <= 96 a 64-column region after dK holds the 16-bit
// P^T, so S^T_{i+1} is computed while the elementwise warps still work on
// tile i; with d = 128 there is no room and P^T overwrites S^T.  Elementwise warps:
// warpgroup g = warp / 4 owns query columns [32 g, 32 g + 32); warp % 4
// selects the 32 key rows.
// FUSED (d = 64): also dQ.  The elementwise warps write dS_i = (dS^T_i)^T
// into a shared-memory tile (keys x queries) besides the 16-bit dS^T in
// TMEM; issuer B computes dQ_i = dS_i K into the last 64 TMEM columns (lanes
// = queries).  At the end of the next step the elementwise warps copy dQ_i
// into a float32 tile of its own as two 32-column boxes in the 128-byte
// swizzle, and one more warp adds them into the float32 accumulator with TMA
// tensor reductions (cp.reduce.async.bulk.tensor .add).
template <int D, bool BF16, bool FUSED = false>
__global__ void __launch_bounds__(BwdCfg<D>::THREADS + (FUSED ? 32 : 0), 1)
    dkdv_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmdO,
                const __grid_constant__ CUtensorMap tmAcc, const MainParams p) {
  using C = BwdCfg<D>;
  constexpr int NS = FUSED ? C::KVQ_NSTAGE : C::KV_NSTAGE;
  // kSepP: P^T has a 64-column region of its own (see above).
  constexpr bool kSepP = 256 + 2 * D + 64 <= 512;
  // kFold: L and D folded into the padded GEMMs (see fold_slot).
  constexpr bool kFold = BF16 && D == 80 && kSepP;
  constexpr int KS = kFold ? kFoldKSteps : D / 16;
  constexpr uint32_t kColDV = 256;
  constexpr uint32_t kColDK = kSepP ? 256 + D : 384;
  constexpr uint32_t kColP = kSepP ? 256 + 2 * D : 0;
  constexpr uint32_t kColDQ = kColP + 64;   // FUSED: dQ_i, D columns
  static_assert(!FUSED || (kSepP && !kFold && kColDQ + D <= 512), "the fused layout fits d = 64 only");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sK = smem;
  uint8_t* sV = smem + C::TILE;
  uint8_t* sStage = smem + 2 * C::TILE;   // per stage: Q, dO, L[128], D[128]
  uint8_t* sDS = sStage + NS * C::KV_STAGE;   // FUSED: dS_i, 128 keys x 128 queries, two 64-query chunks
  uint8_t* sDQ = sDS + C::DS_TILE;            // FUSED: dQ_i, float32, two 32-column boxes
  uint64_t* bars = reinterpret_cast<uint64_t*>(sDS + (FUSED ? C::DS_TILE + C::DQ_TILE : 0));
  uint64_t* bar_kv = bars;            // K, V loaded
  uint64_t* bar_full = bars + 1;      // [NS]
  uint64_t* bar_empty = bar_full + NS;
  uint64_t* bar_s = bar_empty + NS;   // S^T ready
  uint64_t* bar_dp = bar_s + 1;       // dP^T ready
  uint64_t* bar_pt = bar_dp + 1;      // P^T written (one arrival per elementwise warp)
  uint64_t* bar_ds = bar_pt + 1;      // dS^T written
  uint64_t* bar_acc = bar_ds + 1;     // dV, dK complete (one commit per issuer)
  uint64_t* bar_drain = bar_acc + 1;  // every MMA of both issuers complete
  uint64_t* bar_sfree = bar_drain + 1;  // S^T read into registers (separate-P^T layout)
  uint64_t* bar_dvd = bar_sfree + 1;    // dV_i complete: P^T_i consumed
  uint64_t* bar_ext = bar_dvd + 1;      // folded columns of K, V, Q_0, dO_0 written (kFold)
  uint64_t* bar_dq = bar_ext + 1;       // FUSED: dQ_i complete
  uint64_t* bar_dqfree = bar_dq + 1;    // FUSED: dQ_i read out of TMEM (one arrival per elementwise warp)
  uint64_t* bar_stage = bar_dqfree + 1;  // FUSED: dQ_i staged in its shared tile (one arrival per elementwise warp)
  uint64_t* bar_dsfree = bar_stage + 1;  // FUSED: the TMA has read the staged dQ_i (the tile may be reused)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar_dsfree + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int BH = p.B * p.H;
  // Heads in chunks sharing Q/dO through L2; inside a chunk the heaviest key
  // tiles first (for causal the first key tile sees every query).
  int kt, bh;
  chunked_order(static_cast<int>(blockIdx.x), (p.Nk + kT - 1) / kT, BH, &kt, &bh);
  const int b = bh / p.H;
  const int h = bh % p.H;
  const int k0 = kt * kT;
  const int nqt = (p.Nq + kT - 1) / kT;
  const int i_first = p.causal ? min(k0 / kT, nqt) : 0;
  const int n_it = nqt - i_first;   // query tiles this key tile meets

  if (threadIdx.x == 0) {
    mbar_init(bar_kv, 1);
    for (int s = 0; s < NS; ++s) {
      mbar_init(&bar_full[s], 1);
      mbar_init(&bar_empty[s], 2);   // one release per issuer
    }
    mbar_init(bar_s, 1);
    mbar_init(bar_dp, 1);
    mbar_init(bar_pt, C::EW_WARPS);   // one arrival per elementwise warp
    mbar_init(bar_ds, C::EW_WARPS);
    mbar_init(bar_acc, 2);
    mbar_init(bar_drain, 2);
    mbar_init(bar_sfree, C::EW_WARPS);
    mbar_init(bar_dvd, 1);
    mbar_init(bar_ext, C::EW_WARPS);
    mbar_init(bar_dq, 1);
    mbar_init(bar_dqfree, C::EW_WARPS);
    mbar_init(bar_stage, C::EW_WARPS);
    mbar_init(bar_dsfree, 1);
    fence_mbar_init();
  }
  if (warp == C::MMA_WARP) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == C::PROD_WARP) {
    if (lane == 0 && n_it > 0) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmdO);
      mbar_arrive_expect_tx(bar_kv, 2 * C::TILE);
      for (int c = 0; c < C::G::NCH; ++c) {
        tma_load_4d(sK + c * C::G::CHB, &tmK, bar_kv, c * C::G::CC, k0, h, b);
        tma_load_4d(sV + c * C::G::CHB, &tmV, bar_kv, c * C::G::CC, k0, h, b);
      }
      int n_issued = n_it;   // one copy in flight per slot; a give-up stops the fills
      for (int it = 0; it < n_it; ++it) {
        const int s = it % NS;
        const int use = it / NS;
        if (use > 0 && (!mbar_wait(&bar_empty[s], (use - 1) & 1, p.err, 21) ||
                        !mbar_wait_drain(&bar_full[s], (use - 1) & 1))) {
          n_issued = it;
          break;
        }
        uint8_t* st = sStage + s * C::KV_STAGE;
        const int q0 = (i_first + it) * kT;
        mbar_arrive_expect_tx(&bar_full[s], 2 * C::TILE + 1024);
        for (int c = 0; c < C::G::NCH; ++c) {
          tma_load_4d(st + c * C::G::CHB, &tmQ, &bar_full[s], c * C::G::CC, q0, h, b);
          tma_load_4d(st + C::TILE + c * C::G::CHB, &tmdO, &bar_full[s], c * C::G::CC, q0, h, b);
        }
        const int64_t off = static_cast<int64_t>(bh) * p.Nqp + q0;
        bulk_load(st + 2 * C::TILE, p.wsL + off, 512, &bar_full[s]);
        bulk_load(st + 2 * C::TILE + 512, p.wsD + off, 512, &bar_full[s]);
      }
      for (int it = max(0, n_issued - NS); it < n_issued; ++it) mbar_wait_drain(&bar_full[it % NS], (it / NS) & 1);
      mbar_wait_drain(bar_kv, 0);
    }
  } else if (FUSED && warp == C::MMA_WARP + 2) {
    // FUSED: the accumulator's reductions.  For each query tile, once the
    // elementwise warps have staged dQ_i, add its two 32-column boxes into
    // rows [bh Nqp + q0_i, + 128) of the accumulator; when the TMA has read
    // them, hand the tile back for dQ_{i+1}.  Every reduction has completed
    // before the warp leaves.
    const int row0 = bh * p.Nqp + i_first * kT;
    for (int it = 0; it < n_it; ++it) {
      mbar_wait(bar_stage, it & 1, p.err, 54);
      if (elect_one()) {
        tma_reduce_add_2d(&tmAcc, sDQ, 0, row0 + it * kT);
        tma_reduce_add_2d(&tmAcc, sDQ + 128 * 128, 32, row0 + it * kT);
        bulk_commit_group();
        bulk_wait_group_read0();
        mbar_arrive(bar_dsfree);
      }
      __syncwarp();
    }
    if (elect_one()) bulk_wait_group0();
    __syncwarp();
  } else if (warp >= C::MMA_WARP) {
    // Two issuers: A (warp 9) computes S^T_i and dV, B (warp 10) dP^T_i and
    // dK, so that one issuer's barrier polls are covered by the other's MMAs.
    // Each releases every stage once (the empty barriers count two).
    const bool issuer_a = warp == C::MMA_WARP;
    if (n_it > 0) {
      constexpr uint32_t idesc_nt = make_idesc_f16(BF16, kT, kT, false, false);
      constexpr uint32_t idesc_tn = make_idesc_f16(BF16, kT, D, false, true);
      const uint32_t sk = smem_u32(sK);
      const uint32_t sv = smem_u32(sV);
      const uint32_t sst = smem_u32(sStage);
      mbar_wait(bar_kv, 0, p.err, 22);
      if (kFold) mbar_wait(bar_ext, 0, p.err, 36);
      __syncwarp();
      for (int it = 0; it < n_it; ++it) {
        const int s = it % NS;
        const uint32_t sq = sst + s * C::KV_STAGE;
        const uint32_t sdo = sq + C::TILE;
        mbar_wait(&bar_full[s], (it / NS) & 1, p.err, 23);
        __syncwarp();
        tc_fence_after();
        if (issuer_a) {
          if (kSepP) {
            // S^T_i was issued one step ahead (below); issue S^T_{i+1} as soon
            // as the elementwise warps hold S^T_i in registers.
            if (it == 0) {
              mma_nt<D, KS>(tmem, sk, sq, idesc_nt);      // S^T_0 = K Q_0^T
              if (elect_one()) umma_commit(bar_s);
            }
            if (it + 1 < n_it) {
              const int s1 = (it + 1) % NS;
              mbar_wait(&bar_full[s1], ((it + 1) / NS) & 1, p.err, 25);
              mbar_wait(bar_sfree, it & 1, p.err, 31);
              __syncwarp();
              tc_fence_after();
              mma_nt<D, KS>(tmem, sk, sst + s1 * C::KV_STAGE, idesc_nt);   // S^T_{i+1}
              if (elect_one()) umma_commit(bar_s);
            }
            mbar_wait(bar_pt, it & 1, p.err, 24);
            __syncwarp();
            tc_fence_after();
            mma_tn<D, true>(tmem + kColDV, tmem + kColP, sdo, idesc_tn, it > 0);  // dV += P^T_i dO_i
            if (elect_one()) umma_commit(bar_dvd);
          } else {
            mma_nt<D>(tmem, sk, sq, idesc_nt);            // S^T_i = K Q_i^T
            if (elect_one()) umma_commit(bar_s);
            mbar_wait(bar_pt, it & 1, p.err, 24);
            __syncwarp();
            tc_fence_after();
            mma_tn<D>(tmem + kColDV, tmem, sdo, idesc_tn, it > 0);  // dV += P^T_i dO_i
          }
        } else {
          mma_nt<D, KS>(tmem + 128, sv, sdo, idesc_nt);   // dP^T_i = V dO_i^T
          if (elect_one()) umma_commit(bar_dp);
          mbar_wait(bar_ds, it & 1, p.err, 26);
          __syncwarp();
          tc_fence_after();
          mma_tn<D>(tmem + kColDK, tmem + 128, sq, idesc_tn, it > 0);  // dK += dS^T_i Q_i
          if constexpr (FUSED) {
            constexpr uint32_t idesc_dq = make_idesc_f16(BF16, kT, D, true, true);
            if (it > 0) {
              mbar_wait(bar_dqfree, (it - 1) & 1, p.err, 52);   // dQ_{i-1} read out of TMEM
              __syncwarp();
              tc_fence_after();
            }
            mma_mn_mn<D>(tmem + kColDQ, smem_u32(sDS), sk, idesc_dq);   // dQ_i = dS_i K
            if (elect_one()) umma_commit(bar_dq);
          }
        }
        if (elect_one()) umma_commit(&bar_empty[s]);
      }
      if (elect_one()) umma_commit(bar_acc);
    }
    if (elect_one()) umma_commit(bar_drain);
    __syncwarp();
    mbar_wait_drain(bar_drain, 0);
  } else {
    // ------------------------------------------------------- elementwise
    // Warpgroup g owns query columns [32 g, 32 g + 32) of S^T / dP^T; warp % 4
    // selects the 32 key rows (TMEM lanes) of its thread.
    const int g = warp >> 2;
    const int quad = warp & 3;
    const int krow = k0 + quad * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
    const uint32_t tS = tmem + lane_off + g * 32;
    const uint32_t tdP = tmem + lane_off + 128 + g * 32;
    const uint32_t tP = tmem + lane_off + kColP + g * (kSepP ? 16 : 32);
    const uint64_t cs2 = f2pack(p.scale_log2, p.scale_log2);
    const int kr = quad * 32 + lane;   // this thread's row of the K/V tile and of the stage rows it folds

    // FUSED: stage dQ_j (TMEM lanes = the 128 queries of query tile j) in
    // its shared tile once the TMA has read dQ_{j-1} from it: row r of box b
    // (columns [32 b, 32 b + 32)) at b * 16 KB + r * 128 bytes, 16-byte
    // granule x at x ^ (r % 8) (the 128-byte swizzle of the accumulator's
    // tensor map).  Warp (g, quad) writes rows [32 quad, + 32), columns
    // [16 g, + 16): box g / 2, granules 4 (g % 2) .. + 3.
    auto stage_dq = [&](int j) {
      mbar_wait(bar_dq, j & 1, p.err, 53);
      tc_fence_after();
      uint32_t v[16];
      tmem_ld16(tmem + lane_off + kColDQ + g * 16, v);
      tmem_wait_ld();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_dqfree);
      if (j > 0) mbar_wait(bar_dsfree, (j - 1) & 1, p.err, 55);
      const int r = quad * 32 + lane;
      uint8_t* row = sDQ + (g >> 1) * (128 * 128) + r * 128;
#pragma unroll
      for (int c = 0; c < 4; ++c)
        *reinterpret_cast<uint4*>(row + ((((g & 1) * 4 + c) ^ (r & 7)) << 4)) =
            make_uint4(v[4 * c], v[4 * c + 1], v[4 * c + 2], v[4 * c + 3]);
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_stage);
    };
    // Folded columns of stage s: Q rows by warpgroup 2 (-L log2 e / c), dO
    // rows by warpgroup 3 (-D); L and D come with the stage.
    auto fold_stage = [&](int s) {
      uint8_t* st = sStage + s * C::KV_STAGE;
      const float* l = reinterpret_cast<const float*>(st + 2 * C::TILE);
      if (g == 2) *fold_slot(st, kr) = bf16_split(l[kr] / p.scale_log2);
      if (g == 3) *fold_slot(st + C::TILE, kr) = bf16_split(-l[128 + kr]);
    };
    if (kFold) {
      if (n_it > 0) {
        mbar_wait(bar_kv, 0, p.err, 37);
        mbar_wait(&bar_full[0], 0, p.err, 38);
        if (g == 0) *fold_slot(sK, kr) = 0x3F803F80u;   // bf16 (1, 1)
        if (g == 1) *fold_slot(sV, kr) = 0x3F803F80u;
        fold_stage(0);
        fence_proxy_async_smem();
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_ext);
    }

    for (int it = 0; it < n_it; ++it) {
      const int s = it % NS;
      const float* sL = reinterpret_cast<const float*>(sStage + s * C::KV_STAGE + 2 * C::TILE) + g * 32;
      const float* sD = sL + 128;
      const int q0 = (i_first + it) * kT + g * 32;   // first query of this quarter
      const bool diag = p.causal && (q0 < k0 + kT - 1);   // some column q < some row k

      mbar_wait(bar_s, it & 1, p.err, 27);
      // L and D of this stage are in shared memory once its copy landed.
      mbar_wait(&bar_full[s], (it / NS) & 1, p.err, 28);
      tc_fence_after();
      float pt[32];
      {
        uint32_t r[32];
        tmem_ld32(tS, r);
        tmem_wait_ld();
#pragma unroll
        for (int e = 0; e < 32; ++e) pt[e] = __uint_as_float(r[e]);
      }
      if (kSepP) {
        if (kFold && it + 1 < n_it) {
          // stage i+1's folded columns, before S^T_{i+1} may be issued
          const int s1 = (it + 1) % NS;
          mbar_wait(&bar_full[s1], ((it + 1) / NS) & 1, p.err, 39);
          fold_stage(s1);
          fence_proxy_async_smem();
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_sfree);   // S^T_i is in registers
      }
      // P^T = exp2(c S^T - L log2 e); sL holds -L log2 e
#pragma unroll
      for (int e = 0; e < 32; e += 4) {
        float x0, x1, x2, x3;
        if (kFold) {   // -L log2 e is already in S^T
          f2unpack(fmul2(f2pack(pt[e], pt[e + 1]), cs2), x0, x1);
          f2unpack(fmul2(f2pack(pt[e + 2], pt[e + 3]), cs2), x2, x3);
        } else {
          const float4 nl = *reinterpret_cast<const float4*>(sL + e);
          f2unpack(ffma2(f2pack(pt[e], pt[e + 1]), cs2, f2pack(nl.x, nl.y)), x0, x1);
          f2unpack(ffma2(f2pack(pt[e + 2], pt[e + 3]), cs2, f2pack(nl.z, nl.w)), x2, x3);
        }
        pt[e] = ex2_approx(x0);
        pt[e + 1] = ex2_approx(x1);
        pt[e + 2] = ex2_approx(x2);
        pt[e + 3] = ex2_approx(x3);
      }
      if (diag) {
#pragma unroll
        for (int e = 0; e < 32; ++e)
          if (q0 + e < krow) pt[e] = 0.f;
      }
      if (FUSED && krow >= p.Nk) {
        // keys past Nk (zero-filled K, V rows) must add nothing to dQ
#pragma unroll
        for (int e = 0; e < 32; ++e) pt[e] = 0.f;
      }
      {
        uint32_t pk[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) pk[e] = pack2<BF16>(pt[2 * e], pt[2 * e + 1]);
        if (kSepP && it > 0) {
          mbar_wait(bar_dvd, (it - 1) & 1, p.err, 32);   // dV_{i-1} has read P^T_{i-1}
          tc_fence_after();
        }
        tmem_st16(tP, pk);
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_pt);

      mbar_wait(bar_dp, it & 1, p.err, 29);
      tc_fence_after();
      {
        uint32_t r[32];
        tmem_ld32(tdP, r);
        tmem_wait_ld();
        // dS^T = P^T o (dP^T - D)
        uint32_t pk[16];
#pragma unroll
        for (int e = 0; e < 32; e += 4) {
          float a0, a1, a2, a3;
          if (kFold) {   // -D is already in dP^T
            f2unpack(fmul2(f2pack(__uint_as_float(r[e]), __uint_as_float(r[e + 1])), f2pack(pt[e], pt[e + 1])),
                     a0, a1);
            f2unpack(fmul2(f2pack(__uint_as_float(r[e + 2]), __uint_as_float(r[e + 3])), f2pack(pt[e + 2], pt[e + 3])),
                     a2, a3);
          } else {
            const float4 dd = *reinterpret_cast<const float4*>(sD + e);
            f2unpack(fmul2(fsub2(f2pack(__uint_as_float(r[e]), __uint_as_float(r[e + 1])), f2pack(dd.x, dd.y)),
                           f2pack(pt[e], pt[e + 1])),
                     a0, a1);
            f2unpack(fmul2(fsub2(f2pack(__uint_as_float(r[e + 2]), __uint_as_float(r[e + 3])), f2pack(dd.z, dd.w)),
                           f2pack(pt[e + 2], pt[e + 3])),
                     a2, a3);
          }
          pk[e / 2] = pack2<BF16>(a0, a1);
          pk[e / 2 + 1] = pack2<BF16>(a2, a3);
        }
        tmem_st16(tdP, pk);
        if constexpr (FUSED) {
          // dS_i row kr (this thread's key), queries [32 g, 32 g + 32): 64
          // bytes of 64-query chunk g / 2, 16-byte granules 4 (g % 2) .. + 3,
          // 128-byte swizzle.  The tile's last reader was dQ_{i-1}.
          if (it > 0) {
            mbar_wait(bar_dq, (it - 1) & 1, p.err, 56);
            tc_fence_after();
          }
          uint8_t* row = sDS + (g >> 1) * TileGeo<128>::CHB + kr * 128;
#pragma unroll
          for (int c = 0; c < 4; ++c)
            *reinterpret_cast<uint4*>(row + ((((g & 1) * 4 + c) ^ (kr & 7)) << 4)) =
                make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
          fence_proxy_async_smem();
        }
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_ds);
      if (FUSED && it > 0) stage_dq(it - 1);
    }
    if (FUSED && n_it > 0) stage_dq(n_it - 1);

    // epilogue: warpgroups 0-1 write dV, 2-3 write dK * sm_scale (16-column
    // chunks alternate between the two warpgroups of each)
    if (n_it > 0) {
      mbar_wait(bar_acc, 0, p.err, 30);
      tc_fence_after();
    }
    const bool is_dk = g >= 2;
    const bool valid = krow < p.Nk;
    void* outp = is_dk ? p.out1 : p.out0;
    const int64_t sb = is_dk ? p.o1_sb : p.o0_sb;
    const int64_t sh = is_dk ? p.o1_sh : p.o0_sh;
    const int64_t ss = is_dk ? p.o1_ss : p.o0_ss;
    const float scale = is_dk ? p.sm_scale : 1.f;
    uint8_t* dst = const_cast<uint8_t*>(row_ptr(outp, sb, sh, ss, b, h, krow));
    const uint32_t tacc = tmem + lane_off + (is_dk ? kColDK : kColDV);
#pragma unroll
    for (int c = 0; c < D / 16; ++c) {
      if ((c & 1) != (g & 1)) continue;
      uint32_t v[16];
      if (n_it > 0) {
        tmem_ld16(tacc + c * 16, v);
        tmem_wait_ld();
      } else {
#pragma unroll
        for (int e = 0; e < 16; ++e) v[e] = 0u;
      }
      if (valid) store16<BF16>(dst + c * 32, v, scale);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == C::MMA_WARP) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ---------------------------------------------------------------------------
// dQ: one CTA per (query tile, b, h)
// ---------------------------------------------------------------------------
// TMEM columns: [0,128) S, [128,256) dP, [256,256+D) dQ, then 64 columns
// for the 16-bit dS (A operand of the dQ MMA).  dS having columns of its own,
// dP_{j+1} is issued as soon as dP_j is in registers.  Elementwise warps:
// warpgroup g owns key columns [32 g, 32 g + 32); warp % 4 selects the 32
// query rows.
template <int D, bool BF16>
__global__ void __launch_bounds__(BwdCfg<D>::THREADS, 1)
    dq_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
              const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmdO,
              const MainParams p) {
  using C = BwdCfg<D>;
  constexpr int NS = C::Q_NSTAGE;
  constexpr uint32_t kColDQ = 256;
  constexpr uint32_t kColDS = 256 + (D + 31) / 32 * 32;
  static_assert(kColDS + 64 <= 512, "TMEM budget");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem;
  uint8_t* sdO = smem + C::TILE;
  uint8_t* sStage = smem + 2 * C::TILE;   // per stage: K_j, V_j
  uint64_t* bars = reinterpret_cast<uint64_t*>(sStage + NS * C::Q_STAGE);
  uint64_t* bar_q = bars;
  uint64_t* bar_full = bars + 1;
  uint64_t* bar_empty = bar_full + NS;
  uint64_t* bar_s = bar_empty + NS;
  uint64_t* bar_dp = bar_s + 1;
  uint64_t* bar_sfree = bar_dp + 1;   // S read into registers (one arrival per elementwise warp)
  uint64_t* bar_ds = bar_sfree + 1;   // dS written
  uint64_t* bar_acc = bar_ds + 1;     // dQ complete (one commit per issuer)
  uint64_t* bar_drain = bar_acc + 1;  // every MMA of both issuers complete
  uint64_t* bar_dpfree = bar_drain + 1;  // dP_j read into registers
  uint64_t* bar_dqd = bar_dpfree + 1;    // dQ += dS_j K_j complete: dS_j consumed
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar_dqd + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int BH = p.B * p.H;
  const int nqt = (p.Nq + kT - 1) / kT;
  // Heads in chunks sharing K/V through L2; inside a chunk the heaviest query
  // tiles first (for causal the last query tile sees every key).
  int rank, bh;
  chunked_order(static_cast<int>(blockIdx.x), nqt, BH, &rank, &bh);
  const int qt = nqt - 1 - rank;
  const int b = bh / p.H;
  const int h = bh % p.H;
  const int q0 = qt * kT;
  int n_jt = (p.Nk + kT - 1) / kT;
  if (p.causal) n_jt = min(n_jt, min(q0 + kT - 1, p.Nq - 1) / kT + 1);

  if (threadIdx.x == 0) {
    mbar_init(bar_q, 1);
    for (int s = 0; s < NS; ++s) {
      mbar_init(&bar_full[s], 1);
      mbar_init(&bar_empty[s], 2);   // one release per issuer
    }
    mbar_init(bar_s, 1);
    mbar_init(bar_dp, 1);
    mbar_init(bar_sfree, C::EW_WARPS);
    mbar_init(bar_ds, C::EW_WARPS);
    mbar_init(bar_acc, 2);
    mbar_init(bar_drain, 2);
    mbar_init(bar_dpfree, C::EW_WARPS);
    mbar_init(bar_dqd, 1);
    fence_mbar_init();
  }
  if (warp == C::MMA_WARP) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == C::PROD_WARP) {
    if (lane == 0) {
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      mbar_arrive_expect_tx(bar_q, 2 * C::TILE);
      for (int c = 0; c < C::G::NCH; ++c) {
        tma_load_4d(sQ + c * C::G::CHB, &tmQ, bar_q, c * C::G::CC, q0, h, b);
        tma_load_4d(sdO + c * C::G::CHB, &tmdO, bar_q, c * C::G::CC, q0, h, b);
      }
      int n_issued = n_jt;   // one copy in flight per slot; a give-up stops the fills
      for (int jt = 0; jt < n_jt; ++jt) {
        const int s = jt % NS;
        const int use = jt / NS;
        if (use > 0 && (!mbar_wait(&bar_empty[s], (use - 1) & 1, p.err, 41) ||
                        !mbar_wait_drain(&bar_full[s], (use - 1) & 1))) {
          n_issued = jt;
          break;
        }
        uint8_t* st = sStage + s * C::Q_STAGE;
        mbar_arrive_expect_tx(&bar_full[s], 2 * C::TILE);
        for (int c = 0; c < C::G::NCH; ++c) {
          tma_load_4d(st + c * C::G::CHB, &tmK, &bar_full[s], c * C::G::CC, jt * kT, h, b);
          tma_load_4d(st + C::TILE + c * C::G::CHB, &tmV, &bar_full[s], c * C::G::CC, jt * kT, h, b);
        }
      }
      for (int jt = max(0, n_issued - NS); jt < n_issued; ++jt) mbar_wait_drain(&bar_full[jt % NS], (jt / NS) & 1);
      mbar_wait_drain(bar_q, 0);
    }
  } else if (warp >= C::MMA_WARP) {
    // Two issuers: A (warp 9) computes S_j, B (warp 10) dP_j and dQ; each
    // releases every stage once (the empty barriers count two).
    const bool issuer_a = warp == C::MMA_WARP;
    if (n_jt > 0) {
      constexpr uint32_t idesc_nt = make_idesc_f16(BF16, kT, kT, false, false);
      constexpr uint32_t idesc_tn = make_idesc_f16(BF16, kT, D, false, true);
      const uint32_t sq = smem_u32(sQ);
      const uint32_t sdo = smem_u32(sdO);
      const uint32_t sst = smem_u32(sStage);
      mbar_wait(bar_q, 0, p.err, 42);
      for (int jt = 0; jt < n_jt; ++jt) {
        const int s = jt % NS;
        const uint32_t sk = sst + s * C::Q_STAGE;
        mbar_wait(&bar_full[s], (jt / NS) & 1, p.err, 43);
        __syncwarp();
        if (issuer_a) {
          if (jt > 0) mbar_wait(bar_sfree, (jt - 1) & 1, p.err, 45);   // S_{j-1} read
          __syncwarp();
          tc_fence_after();
          mma_nt<D>(tmem, sq, sk, idesc_nt);                // S_j = Q K_j^T
          if (elect_one()) umma_commit(bar_s);
        } else {
          if (jt == 0) {
            tc_fence_after();
            mma_nt<D>(tmem + 128, sdo, sk + C::TILE, idesc_nt);   // dP_0 = dO V_0^T
            if (elect_one()) umma_commit(bar_dp);
          }
          if (jt + 1 < n_jt) {
            const int s1 = (jt + 1) % NS;
            mbar_wait(&bar_full[s1], ((jt + 1) / NS) & 1, p.err, 44);
            mbar_wait(bar_dpfree, jt & 1, p.err, 50);   // dP_j read
            __syncwarp();
            tc_fence_after();
            mma_nt<D>(tmem + 128, sdo, sst + s1 * C::Q_STAGE + C::TILE, idesc_nt);   // dP_{j+1}
            if (elect_one()) umma_commit(bar_dp);
          }
          mbar_wait(bar_ds, jt & 1, p.err, 46);
          __syncwarp();
          tc_fence_after();
          mma_tn<D, true>(tmem + kColDQ, tmem + kColDS, sk, idesc_tn, jt > 0);  // dQ += dS_j K_j
          if (elect_one()) umma_commit(bar_dqd);
        }
        if (elect_one()) umma_commit(&bar_empty[s]);
      }
      if (elect_one()) umma_commit(bar_acc);
    }
    if (elect_one()) umma_commit(bar_drain);
    __syncwarp();
    mbar_wait_drain(bar_drain, 0);
  } else {
    // Warpgroup g owns key columns [32 g, 32 g + 32) of S / dP; warp % 4
    // selects the 32 query rows (TMEM lanes) of its thread.
    const int g = warp >> 2;
    const int quad = warp & 3;
    const int qrow = q0 + quad * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
    const uint32_t tS = tmem + lane_off + g * 32;
    const uint32_t tdP = tmem + lane_off + 128 + g * 32;
    const uint32_t tdS = tmem + lane_off + kColDS + g * 16;
    const int64_t wrow = static_cast<int64_t>(bh) * p.Nqp + qrow;
    const float nLr = p.wsL[wrow];   // -L log2 e; -inf on padded rows
    const float Dr = p.wsD[wrow];
    const uint64_t cs2 = f2pack(p.scale_log2, p.scale_log2);
    const uint64_t nl2 = f2pack(nLr, nLr);
    const uint64_t d2 = f2pack(Dr, Dr);
    const int lim = p.causal ? min(p.Nk, qrow + 1) : p.Nk;   // keys < lim are visible

    for (int jt = 0; jt < n_jt; ++jt) {
      const int kb = jt * kT + g * 32;   // first key of this quarter
      const bool need_mask = (kb + 32 > p.Nk) || (p.causal && kb + 31 > q0);

      mbar_wait(bar_s, jt & 1, p.err, 47);
      tc_fence_after();
      float pr[32];
      {
        uint32_t r[32];
        tmem_ld32(tS, r);
        tmem_wait_ld();
#pragma unroll
        for (int e = 0; e < 32; ++e) pr[e] = __uint_as_float(r[e]);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_sfree);
#pragma unroll
      for (int e = 0; e < 32; e += 2) {
        float x0, x1;
        f2unpack(ffma2(f2pack(pr[e], pr[e + 1]), cs2, nl2), x0, x1);
        pr[e] = ex2_approx(x0);
        pr[e + 1] = ex2_approx(x1);
      }
      if (need_mask) {
#pragma unroll
        for (int e = 0; e < 32; ++e)
          if (kb + e >= lim) pr[e] = 0.f;
      }
      mbar_wait(bar_dp, jt & 1, p.err, 48);
      tc_fence_after();
      {
        uint32_t r[32];
        tmem_ld32(tdP, r);
        tmem_wait_ld();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_dpfree);   // dP_j is in registers
        // dS = P o (dP - D)
        uint32_t pk[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          float a0, a1;
          f2unpack(fmul2(fsub2(f2pack(__uint_as_float(r[2 * e]), __uint_as_float(r[2 * e + 1])), d2),
                         f2pack(pr[2 * e], pr[2 * e + 1])),
                   a0, a1);
          pk[e] = pack2<BF16>(a0, a1);
        }
        if (jt > 0) {
          mbar_wait(bar_dqd, (jt - 1) & 1, p.err, 51);   // dS_{j-1} consumed
          tc_fence_after();
        }
        tmem_st16(tdS, pk);
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_ds);
    }

    // epilogue: dQ * sm_scale; 16-column chunk c is written by warpgroup c % 4
    if (n_jt > 0) {
      mbar_wait(bar_acc, 0, p.err, 49);
      tc_fence_after();
    }
    const bool valid = qrow < p.Nq;
    uint8_t* dst = const_cast<uint8_t*>(row_ptr(p.out0, p.o0_sb, p.o0_sh, p.o0_ss, b, h, qrow));
    const uint32_t tacc = tmem + lane_off + kColDQ;
#pragma unroll
    for (int c = 0; c < D / 16; ++c) {
      if ((c & 3) != g) continue;
      uint32_t v[16];
      if (n_jt > 0) {
        tmem_ld16(tacc + c * 16, v);
        tmem_wait_ld();
      } else {
#pragma unroll
        for (int e = 0; e < 16; ++e) v[e] = 0u;
      }
      if (valid) store16<BF16>(dst + c * 32, v, p.sm_scale);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == C::MMA_WARP) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// dQ = sm_scale * accumulator, in the input type: one thread per 8 columns of
// a row (two 16-byte loads, one 16-byte store); padded rows are not stored.
struct ConvertParams {
  const float* acc;   // [B*H][Nqp][D]
  void* dq;
  int64_t sb, sh, ss;
  int H, Nq, Nqp;
  long long rows;     // B*H*Nq
  float scale;
};

template <int D, bool BF16>
__global__ void __launch_bounds__(256) dq_convert_kernel(const ConvertParams p) {
  constexpr int kGroups = D / 8;
  const long long t = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (t >= p.rows * kGroups) return;
  const int c = static_cast<int>(t % kGroups);
  const long long r = t / kGroups;
  const int q = static_cast<int>(r % p.Nq);
  const int bh = static_cast<int>(r / p.Nq);
  const float4* src = reinterpret_cast<const float4*>(p.acc + (static_cast<size_t>(bh) * p.Nqp + q) * D + 8 * c);
  const float4 a = src[0], b = src[1];
  const float s = p.scale;
  uint4 w;
  w.x = pack2<BF16>(a.x * s, a.y * s);
  w.y = pack2<BF16>(a.z * s, a.w * s);
  w.z = pack2<BF16>(b.x * s, b.y * s);
  w.w = pack2<BF16>(b.z * s, b.w * s);
  uint8_t* dst = const_cast<uint8_t*>(row_ptr(p.dq, p.sb, p.sh, p.ss, bh / p.H, bh % p.H, q));
  reinterpret_cast<uint4*>(dst)[c] = w;
}

template <int D, bool BF16>
cudaError_t launch_bwd_t(const BwdArgs& a, int phase, cudaStream_t stream) {
  using C = BwdCfg<D>;
  const int BH = a.B * a.H;
  cudaError_t e;
  if (a.Nq == 0) {
    if (phase == 1 || phase == 3) return cudaSuccess;
    const long long rows = static_cast<long long>(BH) * a.Nk;
    const unsigned blocks = static_cast<unsigned>((rows + 255) / 256);
    zero_rows_kernel<D><<<blocks, 256, 0, stream>>>(const_cast<void*>(a.dk.ptr), a.dk.sb, a.dk.sh, a.dk.ss, a.B,
                                                     a.H, a.Nk);
    zero_rows_kernel<D><<<blocks, 256, 0, stream>>>(const_cast<void*>(a.dv.ptr), a.dv.sb, a.dv.sh, a.dv.ss, a.B,
                                                     a.H, a.Nk);
    return cudaGetLastError();
  }
  const int Nqp = nq_pad(a.Nq);
  float* wsD = a.ws;
  float* wsL = a.ws + static_cast<size_t>(BH) * Nqp;

  PreParams pp;
  pp.o = a.o.ptr;
  pp.o_sb = a.o.sb;
  pp.o_sh = a.o.sh;
  pp.o_ss = a.o.ss;
  pp.dout = a.dout.ptr;
  pp.d_sb = a.dout.sb;
  pp.d_sh = a.dout.sh;
  pp.d_ss = a.dout.ss;
  pp.lse = a.lse;
  pp.wsD = wsD;
  pp.wsL = wsL;
  float* dqacc = a.fused ? a.ws + 2 * static_cast<size_t>(BH) * Nqp : nullptr;
  pp.dqacc = dqacc;
  pp.B = a.B;
  pp.H = a.H;
  pp.Nq = a.Nq;
  pp.Nqp = Nqp;
  pp.d = D;
  if (phase == 0 || phase == 1) {
    const long long rows = static_cast<long long>(BH) * Nqp;
    const long long blocks = (rows * 8 + 255) / 256;
    bwd_pre_kernel<BF16><<<static_cast<unsigned>(blocks), 256, 0, stream>>>(pp);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }

  if (phase == 1) return cudaSuccess;
  CUtensorMap tq, tk, tv, tdo, tacc = {};
  if (!make_tile_map(&tq, a.q, D, a.Nq, a.H, a.B, BF16) || !make_tile_map(&tk, a.k, D, a.Nk, a.H, a.B, BF16) ||
      !make_tile_map(&tv, a.v, D, a.Nk, a.H, a.B, BF16) || !make_tile_map(&tdo, a.dout, D, a.Nq, a.H, a.B, BF16))
    return cudaErrorInvalidValue;
  if (a.fused && !make_f32_rows_map(&tacc, dqacc, static_cast<int64_t>(BH) * Nqp, D)) return cudaErrorInvalidValue;

  MainParams mp;
  mp.B = a.B;
  mp.H = a.H;
  mp.Nq = a.Nq;
  mp.Nk = a.Nk;
  mp.Nqp = Nqp;
  mp.causal = a.causal;
  mp.scale_log2 = a.sm_scale * kLog2e;
  mp.sm_scale = a.sm_scale;
  mp.wsD = wsD;
  mp.wsL = wsL;
  mp.dqacc = dqacc;
  mp.err = a.err;

  // dK, dV
  mp.out0 = const_cast<void*>(a.dv.ptr);
  mp.o0_sb = a.dv.sb;
  mp.o0_sh = a.dv.sh;
  mp.o0_ss = a.dv.ss;
  mp.out1 = const_cast<void*>(a.dk.ptr);
  mp.o1_sb = a.dk.sb;
  mp.o1_sh = a.dk.sh;
  mp.o1_ss = a.dk.ss;
  if (a.fused) {
    if constexpr (D == 64) {
      if (phase == 0 || phase == 2) {
        auto kern = dkdv_kernel<D, BF16, true>;
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::KVQ_SMEM);
        if (e != cudaSuccess) return e;
        const long long blocks = static_cast<long long>((a.Nk + kT - 1) / kT) * BH;
        kern<<<static_cast<unsigned>(blocks), C::THREADS + 32, C::KVQ_SMEM, stream>>>(tq, tk, tv, tdo, tacc, mp);
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
      }
      if (phase == 0 || phase == 3) {
        ConvertParams cp;
        cp.acc = dqacc;
        cp.dq = const_cast<void*>(a.dq.ptr);
        cp.sb = a.dq.sb;
        cp.sh = a.dq.sh;
        cp.ss = a.dq.ss;
        cp.H = a.H;
        cp.Nq = a.Nq;
        cp.Nqp = Nqp;
        cp.rows = static_cast<long long>(BH) * a.Nq;
        cp.scale = a.sm_scale;
        const long long threads = cp.rows * (D / 8);
        dq_convert_kernel<D, BF16><<<static_cast<unsigned>((threads + 255) / 256), 256, 0, stream>>>(cp);
        e = cudaGetLastError();
      }
      return e;
    } else {
      return cudaErrorInvalidValue;
    }
  }
  if (phase == 0 || phase == 2) {
    auto kern = dkdv_kernel<D, BF16>;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::KV_SMEM);
    if (e != cudaSuccess) return e;
    const long long blocks = static_cast<long long>((a.Nk + kT - 1) / kT) * BH;
    kern<<<static_cast<unsigned>(blocks), C::THREADS, C::KV_SMEM, stream>>>(tq, tk, tv, tdo, tacc, mp);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  // dQ
  mp.out0 = const_cast<void*>(a.dq.ptr);
  mp.o0_sb = a.dq.sb;
  mp.o0_sh = a.dq.sh;
  mp.o0_ss = a.dq.ss;
  mp.out1 = nullptr;
  if (phase == 0 || phase == 3) {
    auto kern = dq_kernel<D, BF16>;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::Q_SMEM);
    if (e != cudaSuccess) return e;
    const long long blocks = static_cast<long long>((a.Nq + kT - 1) / kT) * BH;
    kern<<<static_cast<unsigned>(blocks), C::THREADS, C::Q_SMEM, stream>>>(tq, tk, tv, tdo, mp);
    e = cudaGetLastError();
  }
  return e;
}

}  // namespace

cudaError_t launch_bwd(const BwdArgs& a, int phase, cudaStream_t stream) {
  switch (a.d) {
    case 64: return a.bf16 ? launch_bwd_t<64, true>(a, phase, stream) : launch_bwd_t<64, false>(a, phase, stream);
    case 80: return a.bf16 ? launch_bwd_t<80, true>(a, phase, stream) : launch_bwd_t<80, false>(a, phase, stream);
    case 128:
      return a.bf16 ? launch_bwd_t<128, true>(a, phase, stream) : launch_bwd_t<128, false>(a, phase, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace fa
