// fa_fwd.cu -- FlashAttention-2 forward for sm_103a (tcgen05 + TMA).
//
// Computes O = softmax(sm_scale * Q K^T [+ causal mask]) V and the per-row
// natural-log LSE with the online-softmax recurrences of "[CS336] Assignment 2:
// Systems", "FlashAttention V2 / Forward Pass" (running max m, running sum l,
// one query tile against all key tiles, no tiling over d), evaluated in the
// exp2 domain with sm_scale folded by log2(e) as in "Understanding Triton
// Tutorials Part 2", "Fused Attention 2" (_attn_fwd_inner: qk_scale =
// sm_scale * 1.44269504, p = exp2(qk - m), alpha = exp2(m_old - m_new)), and the
// delayed normalisation of FA-2 (O divided by the final l only).
//
// Two kernels.  fwd_sp_kernel (d <= 96, further below) gives P TMEM columns
// of its own, splits the issuers by MMA kind (one warp every S, one every PV),
// lets blocks walk several work units, and has an e5m2-V variant; at d = 64
// it also has a one-query-tile build that runs two blocks per SM.
// fwd_kernel (d = 128, next) is described here.
//
// GB300 design (one CTA = two 128-row query tiles of one (b, h)):
//   warps 0-3  softmax / correction / epilogue of query tile 0 (one row each)
//   warps 4-7  the same for query tile 1
//   warp  8    TMA producer: Q tiles once, then K_j, V_j through an
//              mbarrier ring of NSTAGE shared-memory slots
//   warps 9-10 tcgen05.mma issuers, one warp per query tile (warp 9 also
//              allocates TMEM).  Two issuers keep the tensor pipe fed: the
//              issue of tcgen05.mma runs at most about one MMA ahead of its
//              execution, so every barrier poll by an issuer leaves a bubble
//              that only the other issuer's MMAs can fill.  The whole warp
//              runs the issue loop (descriptors are warp-uniform) and one
//              elected lane issues each MMA: an issuing warp shares its
//              sub-partition's issue slots with two busy softmax warps, and
//              in this form it keeps the MMA rate they would otherwise cut
//              by a third.
// Tensor memory (512 columns x 128 lanes): S_t at column 128*t (fp32 scores,
// overwritten in place by the 16-bit P_t that feeds the PV MMA as its A
// operand), O_t at column 256 + 128*t (fp32 accumulator).  While tile 0's
// softmax runs on S_0 the tensor cores compute PV and the next S of tile 1,
// and the other way round.
// O is rescaled in TMEM only when a row's running max grows by more than
// 2^8 (the stale max stays exact because l uses the same max); in the common
// case the exponentials are taken against the running max in the same pass
// that finds the tile max, and the tile is redone only when a max jumped.
// Causal: tiles above the diagonal are never loaded or computed; only the
// diagonal tile and the ragged key tail are masked.
#include "fa_internal.h"
#include "ptx.cuh"

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <math_constants.h>

namespace fa {
namespace {

constexpr int kBM = 128;          // query rows per tile
constexpr int kBN = 128;          // keys per tile
constexpr int kNQT = 2;           // query tiles per CTA
constexpr float kRescaleLog2 = 8.0f;
// A row sum of p = exp2(c s - m) at most 2^kRescaleLog2 bounds every p of the
// row by the same, i.e. its max grew by at most kRescaleLog2.
constexpr float kFastSumBound = 256.0f;
static_assert(kFastSumBound == (1 << static_cast<int>(kRescaleLog2)), "keep the two bounds in step");
// How far a row's max may grow before the running max is moved: 2^8 with
// 16-bit P (the stale max is exact, as O / l and LSE use the same one), and
// with e5m2 P under the lazy rule (LAZY8); 0 with e5m2 P otherwise.  The
// e5m2 cast of p depends on the scale p is taken at, and "Fused Attention 2"
// takes p against the running max of the blocks so far, moved at every
// block; the kernels do the same by default, so that they cast the same
// values (O is then rescaled whenever a row's max grows).
template <bool FP8V, bool LAZY8>
constexpr float kMaxGrowth = FP8V && !LAZY8 ? 0.0f : kRescaleLog2;

template <int D>
struct FwdCfg {
  using G = TileGeo<D>;
  static constexpr int TILE = G::TILE;                  // one 128-row tile of Q, K or V
  static constexpr int NSTAGE = D == 64 ? 8 : (D == 80 ? 6 : 4);   // K/V ring depth
  static constexpr int SMEM_DATA = kNQT * TILE + NSTAGE * TILE;
  static constexpr int NBARS = kNQT + 2 * NSTAGE + 4 * kNQT + 1;
  static constexpr int SMEM = 1024 + SMEM_DATA + NBARS * 8 + 16;
  static constexpr int THREADS = kNQT * 128 + 32 + kNQT * 32;
  static constexpr int PROD_WARP = kNQT * 4;
  static constexpr int MMA_WARP = kNQT * 4 + 1;   // first of kNQT issuer warps (also allocates TMEM)
};

// Programmatic dependent launch.  launch_dependents: once every block of
// this grid has issued it (or exited), the grid launched after it on the
// stream with the programmatic-serialization attribute may start.  wait:
// blocks until the grids this one depends on have completed and their memory
// operations are visible to it.
__device__ __forceinline__ void griddep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

struct FwdParams {
  int B, H, Nq, Nk;
  int n_pairs;          // ceil(Nq / 256)
  int causal;
  float scale_log2;     // sm_scale * log2(e)
  void* o;
  int64_t o_sb, o_sh, o_ss;
  float* lse;
  int* err;
  // Split-KV: block b works on split b % n_splits, key tiles
  // [split * tiles_per_split, (split + 1) * tiles_per_split).
  int n_splits;
  int tiles_per_split;
  int Nqp;              // query rows padded to whole tiles (partial buffers)
  float* part_o;        // [n_splits][B*H][Nqp][d]
  float* part_lse;      // [n_splits][B*H][Nqp]
  // Work split of the separate-P forward (n_splits == 1 only): blocks
  // [0, grid_p) each walk units b, b + grid_p, ... below persist_units; the
  // other blocks take one item each of the remaining units (see sp_next).
  int grid_p = 0;
  int persist_units = 0;
  // Separate-P forward on a grid under one wave: one 128-row query tile per
  // block (tile 1 of every item empty), so that twice as many SMs work.
  int single_tile = 0;
};

// Number of key tiles query tile t (rows r0 .. r0+127) needs.
__device__ __forceinline__ int key_tiles(int r0, int Nq, int Nk, int causal) {
  if (r0 >= Nq) return 0;
  int n = (Nk + kBN - 1) / kBN;
  if (causal) {
    const int last = min(r0 + kBM - 1, Nq - 1);
    n = min(n, last / kBN + 1);
  }
  return n;
}

// Epilogue of one query row: O = O_acc / l to 16-bit (16-byte stores) and
// LSE = ln(sum_j exp(sm_scale q.k_j)) = ln 2 * (m + log2 l); rows >= Nq
// store nothing.
template <int D, bool BF16>
__device__ __forceinline__ void store_o_lse(const FwdParams& p, uint32_t tO, int b, int h, int qrow, float m,
                                            float l) {
  const float inv_l = 1.f / l;
  const bool valid = qrow < p.Nq;
  uint8_t* orow = reinterpret_cast<uint8_t*>(p.o) +
                  2 * (static_cast<int64_t>(b) * p.o_sb + static_cast<int64_t>(h) * p.o_sh +
                       static_cast<int64_t>(qrow) * p.o_ss);
#pragma unroll
  for (int c = 0; c < D / 16; ++c) {
    uint32_t o[16];
    tmem_ld16(tO + c * 16, o);
    tmem_wait_ld();
    uint4 w0, w1;
    w0.x = pack2<BF16>(__uint_as_float(o[0]) * inv_l, __uint_as_float(o[1]) * inv_l);
    w0.y = pack2<BF16>(__uint_as_float(o[2]) * inv_l, __uint_as_float(o[3]) * inv_l);
    w0.z = pack2<BF16>(__uint_as_float(o[4]) * inv_l, __uint_as_float(o[5]) * inv_l);
    w0.w = pack2<BF16>(__uint_as_float(o[6]) * inv_l, __uint_as_float(o[7]) * inv_l);
    w1.x = pack2<BF16>(__uint_as_float(o[8]) * inv_l, __uint_as_float(o[9]) * inv_l);
    w1.y = pack2<BF16>(__uint_as_float(o[10]) * inv_l, __uint_as_float(o[11]) * inv_l);
    w1.z = pack2<BF16>(__uint_as_float(o[12]) * inv_l, __uint_as_float(o[13]) * inv_l);
    w1.w = pack2<BF16>(__uint_as_float(o[14]) * inv_l, __uint_as_float(o[15]) * inv_l);
    if (valid) {
      reinterpret_cast<uint4*>(orow + c * 32)[0] = w0;
      reinterpret_cast<uint4*>(orow + c * 32)[1] = w1;
    }
  }
  if (valid) p.lse[(static_cast<int64_t>(b) * p.H + h) * p.Nq + qrow] = (m + log2f(l)) * 0.69314718055994531f;
}

// store_o_lse with every O column read out of TMEM before one wait (the
// separate-P forward's epilogue, where the softmax warps' score and P
// registers are free by then).
template <int D, bool BF16>
__device__ __forceinline__ void store_o_lse_batched(const FwdParams& p, uint32_t tO, int b, int h, int qrow, float m,
                                                    float l) {
  uint32_t o[D / 16][16];
#pragma unroll
  for (int c = 0; c < D / 16; ++c) tmem_ld16(tO + c * 16, o[c]);
  tmem_wait_ld();
  const float inv_l = 1.f / l;
  const bool valid = qrow < p.Nq;
  uint8_t* orow = reinterpret_cast<uint8_t*>(p.o) +
                  2 * (static_cast<int64_t>(b) * p.o_sb + static_cast<int64_t>(h) * p.o_sh +
                       static_cast<int64_t>(qrow) * p.o_ss);
#pragma unroll
  for (int c = 0; c < D / 16; ++c) {
    uint4 w0, w1;
    w0.x = pack2<BF16>(__uint_as_float(o[c][0]) * inv_l, __uint_as_float(o[c][1]) * inv_l);
    w0.y = pack2<BF16>(__uint_as_float(o[c][2]) * inv_l, __uint_as_float(o[c][3]) * inv_l);
    w0.z = pack2<BF16>(__uint_as_float(o[c][4]) * inv_l, __uint_as_float(o[c][5]) * inv_l);
    w0.w = pack2<BF16>(__uint_as_float(o[c][6]) * inv_l, __uint_as_float(o[c][7]) * inv_l);
    w1.x = pack2<BF16>(__uint_as_float(o[c][8]) * inv_l, __uint_as_float(o[c][9]) * inv_l);
    w1.y = pack2<BF16>(__uint_as_float(o[c][10]) * inv_l, __uint_as_float(o[c][11]) * inv_l);
    w1.z = pack2<BF16>(__uint_as_float(o[c][12]) * inv_l, __uint_as_float(o[c][13]) * inv_l);
    w1.w = pack2<BF16>(__uint_as_float(o[c][14]) * inv_l, __uint_as_float(o[c][15]) * inv_l);
    if (valid) {
      reinterpret_cast<uint4*>(orow + c * 32)[0] = w0;
      reinterpret_cast<uint4*>(orow + c * 32)[1] = w1;
    }
  }
  if (valid) p.lse[(static_cast<int64_t>(b) * p.H + h) * p.Nq + qrow] = (m + log2f(l)) * 0.69314718055994531f;
}

// Epilogue of one query row in split mode: the split's own softmax output
// O_s = O_acc / l and lse_s = ln 2 * (m + log2 l) in float32, or O_s = 0 and
// lse_s = -inf when the row saw no key of the split (have == false).
template <int D>
__device__ __forceinline__ void store_partial(const FwdParams& p, uint32_t tO, int bh, int split, int qrow,
                                              float m, float l, bool have) {
  const bool valid = qrow < p.Nq;
  const size_t row = (static_cast<size_t>(split) * p.B * p.H + bh) * p.Nqp + qrow;
  float4* dst = reinterpret_cast<float4*>(p.part_o + row * D);
  const float inv_l = have ? 1.f / l : 0.f;
#pragma unroll
  for (int c = 0; c < D / 16; ++c) {
    uint32_t o[16];
    if (have) {
      tmem_ld16(tO + c * 16, o);
      tmem_wait_ld();
    } else {
#pragma unroll
      for (int e = 0; e < 16; ++e) o[e] = 0u;
    }
    if (valid) {
#pragma unroll
      for (int i = 0; i < 4; ++i)
        dst[c * 4 + i] = make_float4(__uint_as_float(o[4 * i]) * inv_l, __uint_as_float(o[4 * i + 1]) * inv_l,
                                     __uint_as_float(o[4 * i + 2]) * inv_l, __uint_as_float(o[4 * i + 3]) * inv_l);
    }
  }
  if (valid) p.part_lse[row] = have ? (m + log2f(l)) * 0.69314718055994531f : -CUDART_INF_F;
}

// S = Q_t K_j^T into TMEM columns [d_tmem, d_tmem + 128): M = 128 queries,
// N = 128 keys, K = D (16 per MMA), both operands K-major in shared memory.
template <int D, bool BF16>
__device__ __forceinline__ void issue_s(uint32_t d_tmem, uint32_t q_addr, uint32_t k_addr) {
  using G = TileGeo<D>;
  constexpr uint32_t idesc = make_idesc_f16(BF16, kBM, kBN, false, false);
  const uint64_t ad0 = make_sdesc(q_addr, 16, G::SBO, G::LAYOUT);
  const uint64_t bd0 = make_sdesc(k_addr, 16, G::SBO, G::LAYOUT);
#pragma unroll
  for (int ks = 0; ks < D / 16; ++ks) {
    const uint32_t off = (ks / G::KPC) * G::CHB + (ks % G::KPC) * 32;
    if (elect_one()) umma_ss(d_tmem, desc_add(ad0, off), desc_add(bd0, off), idesc, ks > 0);
  }
}

// O_t (+)= P V_j : M = 128 queries, N = D, K = 128 keys (16 per MMA).  P is
// 16-bit, two per TMEM column, in columns [p_tmem, p_tmem + 64); V is the
// MN-major B operand in shared memory.
template <int D, bool BF16>
__device__ __forceinline__ void issue_pv(uint32_t o_tmem, uint32_t p_tmem, uint32_t v_addr, bool acc) {
  using G = TileGeo<D>;
  constexpr uint32_t idesc = make_idesc_f16(BF16, kBM, D, false, true);
  const uint64_t bd0 = make_sdesc(v_addr, G::CHB, G::SBO, G::LAYOUT);
#pragma unroll
  for (int ks = 0; ks < kBN / 16; ++ks)
    if (elect_one()) umma_ts(o_tmem, p_tmem + ks * 8, desc_add(bd0, ks * 16 * G::ROWB), idesc, (acc || ks > 0) ? 1u : 0u);
}

// O_t (+)= P V_j with P in e5m2, four per TMEM column (32 columns at p_tmem),
// and V_j^T an e5m2 tile of D rows x 128 keys (K-major: 128-byte rows, the
// 128-byte swizzle, 8-row groups 1024 bytes apart); K = 32 keys per MMA.
template <int D>
__device__ __forceinline__ void issue_pv_f8(uint32_t o_tmem, uint32_t p_tmem, uint32_t vt_addr, bool acc) {
  constexpr uint32_t idesc = make_idesc_f8(kFmtE5M2, kFmtE5M2, kBM, D);
  const uint64_t bd0 = make_sdesc(vt_addr, 16, 1024, 2);
#pragma unroll
  for (int ks = 0; ks < kBN / 32; ++ks)
    if (elect_one()) umma_ts_f8(o_tmem, p_tmem + ks * 8, desc_add(bd0, ks * 32), idesc, (acc || ks > 0) ? 1u : 0u);
}

// p = exp2(c s - m) over the 128 scores of this thread's row (cs2 = (c, c),
// nm2 = (-m, -m)), packed as the A operand of the PV product: two 16-bit
// values per register, or four e5m2 values (FP8V: the cast of "Fused
// Attention 2" before the product with V).  Returns the sum of the unrounded
// p.
template <bool BF16, bool FP8V>
__device__ __forceinline__ float exp_pack(const float (&s)[kBN], uint64_t cs2, uint64_t nm2,
                                          uint32_t (&pk)[FP8V ? kBN / 4 : kBN / 2]) {
  uint64_t acc[4] = {0ull, 0ull, 0ull, 0ull};
  float q0 = 0.f, q1 = 0.f;   // FP8V: the previous pair, waiting for its partner
#pragma unroll
  for (int e = 0; e < kBN / 2; ++e) {
    float x0, x1;
    f2unpack(ffma2(f2pack(s[2 * e], s[2 * e + 1]), cs2, nm2), x0, x1);
    const float p0 = ex2_approx(x0);
    const float p1 = ex2_approx(x1);
    acc[e & 3] = fadd2(acc[e & 3], f2pack(p0, p1));
    if constexpr (FP8V) {
      if (e & 1) {
        pk[e >> 1] = pack4_e5m2(q0, q1, p0, p1);
      } else {
        q0 = p0;
        q1 = p1;
      }
    } else {
      pk[e] = pack2<BF16>(p0, p1);
    }
  }
  float a0, a1;
  f2unpack(fadd2(fadd2(acc[0], acc[1]), fadd2(acc[2], acc[3])), a0, a1);
  return a0 + a1;
}

// LAZY8 (e5m2 P only): the running max moves only when it grows by more
// than 2^8, as with 16-bit P (faster; p's e5m2 cast can then differ from the
// page's steps by one rounding step), instead of at every block.
template <int D, bool BF16, bool FP8V, bool LAZY8 = false>
__global__ void __launch_bounds__(FwdCfg<D>::THREADS, 1)
    fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
               const __grid_constant__ CUtensorMap tmV, const FwdParams p) {
  using C = FwdCfg<D>;
  if (p.n_splits > 1) griddep_launch_dependents();   // the merge may take SMs as blocks of this grid finish
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem;
  uint8_t* sKV = smem + kNQT * C::TILE;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sKV + C::NSTAGE * C::TILE);
  uint64_t* bar_q = bars;                           // [kNQT]
  uint64_t* bar_full = bar_q + kNQT;                // [NSTAGE]
  uint64_t* bar_empty = bar_full + C::NSTAGE;       // [NSTAGE]
  uint64_t* bar_s = bar_empty + C::NSTAGE;          // [kNQT] S_t ready
  uint64_t* bar_p = bar_s + kNQT;                   // [kNQT] P_t written (one arrival per softmax warp)
  uint64_t* bar_o = bar_p + kNQT;                   // [kNQT] PV_t complete
  uint64_t* bar_turn = bar_o + kNQT;                // [kNQT] issuer t may issue its next group
  uint64_t* bar_drain = bar_turn + kNQT;            // [1]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar_drain + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // Work decode: heads in chunks sharing K/V through L2; inside a chunk the
  // heaviest query-tile pairs first (longest-processing-time order for causal).
  const int BH = p.B * p.H;
  const int split = static_cast<int>(blockIdx.x) % p.n_splits;
  int rank, bh;
  chunked_order(static_cast<int>(blockIdx.x) / p.n_splits, p.n_pairs, BH, &rank, &bh);
  const int pair = p.n_pairs - 1 - rank;
  const int b = bh / p.H;
  const int h = bh % p.H;
  const int q0 = pair * (kNQT * kBM);
  const int kt0 = split * p.tiles_per_split;   // first key tile of this block

  // Key tiles of query tile t in this block: [kt0, kt0 + nkt[t]).
  int nkt[kNQT];
  int n_max = 0;
#pragma unroll
  for (int t = 0; t < kNQT; ++t) {
    nkt[t] = max(0, min(key_tiles(q0 + t * kBM, p.Nq, p.Nk, p.causal), kt0 + p.tiles_per_split) - kt0);
    n_max = max(n_max, nkt[t]);
  }

  if (threadIdx.x == 0) {
    for (int t = 0; t < kNQT; ++t) {
      mbar_init(&bar_q[t], 1);
      mbar_init(&bar_s[t], 1);
      mbar_init(&bar_p[t], 4);
      mbar_init(&bar_o[t], 1);
      mbar_init(&bar_turn[t], 1);
    }
    for (int s = 0; s < C::NSTAGE; ++s) {
      mbar_init(&bar_full[s], 1);
      mbar_init(&bar_empty[s], kNQT);   // one release per issuer
    }
    mbar_init(bar_drain, kNQT);
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
    // ------------------------------------------------------------------ TMA
    if (lane == 0) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
#pragma unroll
      for (int t = 0; t < kNQT; ++t) {
        if (nkt[t] == 0) continue;
        mbar_arrive_expect_tx(&bar_q[t], C::TILE);
        for (int c = 0; c < C::G::NCH; ++c)
          tma_load_4d(sQ + t * C::TILE + c * C::G::CHB, &tmQ, &bar_q[t], c * C::G::CC, q0 + t * kBM, h, b);
      }
      // K_0, V_0, K_1, V_1, ... : the order the MMA issuers consume them in.
      // A slot is refilled only after its previous fill has landed (even if
      // a consumer that gave up released it early), so each slot has at most
      // one copy in flight and one pending expect-tx phase.  A give-up stops
      // the fills; only the fills actually issued are drained.
      int nfill = 2 * n_max;
      for (int f = 0; f < nfill; ++f) {
        const int s = f % C::NSTAGE;
        const int use = f / C::NSTAGE;
        if (use > 0 && (!mbar_wait(&bar_empty[s], (use - 1) & 1, p.err, 1) ||
                        !mbar_wait_drain(&bar_full[s], (use - 1) & 1))) {
          nfill = f;
          break;
        }
        const int j = kt0 + (f >> 1);
        if (FP8V && (f & 1)) {
          // V_j^T: D rows of 128 keys, one box
          mbar_arrive_expect_tx(&bar_full[s], D * kBN);
          tma_load_4d(sKV + s * C::TILE, &tmV, &bar_full[s], j * kBN, 0, h, b);
        } else {
          mbar_arrive_expect_tx(&bar_full[s], C::TILE);
          const CUtensorMap* map = (f & 1) ? &tmV : &tmK;
          for (int c = 0; c < C::G::NCH; ++c)
            tma_load_4d(sKV + s * C::TILE + c * C::G::CHB, map, &bar_full[s], c * C::G::CC, j * kBN, h, b);
        }
      }
      // Drain: the last fill of every slot has landed before the CTA exits.
      for (int f = max(0, nfill - C::NSTAGE); f < nfill; ++f)
        mbar_wait_drain(&bar_full[f % C::NSTAGE], (f / C::NSTAGE) & 1);
#pragma unroll
      for (int t = 0; t < kNQT; ++t)
        if (nkt[t] > 0) mbar_wait_drain(&bar_q[t], 0);
    }
  } else if (warp >= C::MMA_WARP) {
    // ------------------------------------------------------------ MMA issue
    // Issuer t drives query tile t.  Its groups are G(t,-1) = S_t,0 and
    // G(t,j) = PV_t,j + S_t,j+1; the two issuers take turns in the order
    // G(0,-1) G(1,-1) G(0,0) G(1,0) G(0,1) ..., handing over through
    // bar_turn, which keeps the two tiles half a step apart (one tile's
    // softmax runs while the tensor cores work for the other).  An issuer
    // does its barrier polls for the next group before it waits for its
    // turn, i.e. while the other issuer's MMAs execute.
    // Every K/V fill is released by one commit of each issuer, also fills
    // its own tile does not need, and only after the fill has landed, so
    // both releases of one use of a slot come before any release of its next
    // use (the empty barriers count two).
    const int t = warp - C::MMA_WARP;
    if (n_max > 0) {
      const uint32_t sq_addr = smem_u32(sQ);
      const uint32_t skv_addr = smem_u32(sKV);
      const int nt = nkt[t];
      // G(t,-1)
      if (nt > 0) mbar_wait(&bar_q[t], 0, p.err, 2);
      mbar_wait(&bar_full[0], 0, p.err, 3);
      if (t == 1) mbar_wait(&bar_turn[1], 0, p.err, 11);
      __syncwarp();
      if (nt > 0) {
        tc_fence_after();
        issue_s<D, BF16>(tmem + t * 128, sq_addr + t * C::TILE, skv_addr);
      }
      if (elect_one()) {
        mbar_arrive(&bar_turn[1 - t]);
        if (nt > 0) umma_commit(&bar_s[t]);
        umma_commit(&bar_empty[0]);
      }
      for (int j = 0; j < n_max; ++j) {
        const int fv = 2 * j + 1;            // fill index of V_j
        const int fk = 2 * j + 2;            // fill index of K_{j+1}
        const bool pv = j < nt;
        const bool sn = j + 1 < nt;
        mbar_wait(&bar_full[fv % C::NSTAGE], (fv / C::NSTAGE) & 1, p.err, 4);
        if (j + 1 < n_max) mbar_wait(&bar_full[fk % C::NSTAGE], (fk / C::NSTAGE) & 1, p.err, 6);
        if (pv) mbar_wait(&bar_p[t], j & 1, p.err, 5);
        // turn: G(0,j) follows G(1,j-1), G(1,j) follows G(0,j)
        mbar_wait(&bar_turn[t], (t == 0 ? j : j + 1) & 1, p.err, 12);
        __syncwarp();
        tc_fence_after();
        if (pv) {
          if constexpr (FP8V)
            issue_pv_f8<D>(tmem + 256 + t * 128, tmem + t * 128, skv_addr + (fv % C::NSTAGE) * C::TILE, j > 0);
          else
            issue_pv<D, BF16>(tmem + 256 + t * 128, tmem + t * 128, skv_addr + (fv % C::NSTAGE) * C::TILE, j > 0);
        }
        if (sn) issue_s<D, BF16>(tmem + t * 128, sq_addr + t * C::TILE, skv_addr + (fk % C::NSTAGE) * C::TILE);
        if (elect_one()) {
          mbar_arrive(&bar_turn[1 - t]);
          if (pv && !sn) umma_commit(&bar_o[t]);   // last PV of this tile
          if (sn) umma_commit(&bar_s[t]);
          umma_commit(&bar_empty[fv % C::NSTAGE]);
          if (j + 1 < n_max) umma_commit(&bar_empty[fk % C::NSTAGE]);
        }
      }
      // Drain: every MMA of both issuers has completed before TMEM is freed.
      if (elect_one()) umma_commit(bar_drain);
      __syncwarp();
      mbar_wait_drain(bar_drain, 0);
    }
  } else {
    // ------------------------------------------------- softmax / epilogue
    const int t = warp >> 2;
    const int quad = warp & 3;
    const int row = quad * 32 + lane;
    const int r0 = q0 + t * kBM;
    const int qrow = r0 + row;
    const int n = nkt[t];
    const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
    const uint32_t tS = tmem + lane_off + t * 128;
    const uint32_t tO = tmem + lane_off + 256 + t * 128;
    const float cs = p.scale_log2;
    // scores per 16-column P store: 32 as 16-bit pairs, 64 as e5m2 quads
    constexpr int kPChunk = FP8V ? 64 : 32;

    float m = -CUDART_INF_F;  // running max of the scaled scores (log2 domain)
    float l = 0.f;            // running sum of exp2(score - m)

    for (int j = 0; j < n; ++j) {
      // S_t,j complete implies PV_t,j-1 complete (one issuer, and a commit
      // tracks every earlier MMA of its thread), so O_t may be rescaled.
      mbar_wait(&bar_s[t], j & 1, p.err, 8);
      tc_fence_after();

      float s[kBN];
#pragma unroll
      for (int i = 0; i < kBN / 32; ++i) {
        uint32_t r[32];
        tmem_ld32(tS + i * 32, r);
#pragma unroll
        for (int e = 0; e < 32; ++e) s[i * 32 + e] = __uint_as_float(r[e]);
      }
      tmem_wait_ld();

      const int kbase = (kt0 + j) * kBN;
      const bool tail = kbase + kBN > p.Nk;
      const bool diag = p.causal && (kbase + kBN - 1 > r0);
      if (tail || diag) {
        const int lim = p.causal ? min(p.Nk, qrow + 1) : p.Nk;  // keys < lim are visible
#pragma unroll
        for (int c = 0; c < kBN; ++c)
          if (kbase + c >= lim) s[c] = -CUDART_INF_F;
      }
      const uint64_t cs2 = f2pack(cs, cs);
      bool done = false;
      if (j > 0) {
        // Common case: exp2 against the running max m (any score up to
        // m + 8 gives p <= 2^8), finding the tile max in the same pass.  If a
        // row's max grew by more than 8, the tile is redone below with a new
        // max; otherwise this is exactly the result of the redo.
        const uint64_t nm2 = f2pack(-m, -m);
        uint64_t acc[4] = {0ull, 0ull, 0ull, 0ull};
        float mc[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) mc[i] = -CUDART_INF_F;
#pragma unroll
        for (int i = 0; i < kBN / kPChunk; ++i) {
          uint32_t pk[16];
          float q0 = 0.f, q1 = 0.f;   // e5m2: the previous pair, waiting for its partner
#pragma unroll
          for (int e = 0; e < kPChunk / 2; ++e) {
            const int c = i * kPChunk + 2 * e;
            mc[e & 7] = fmax3(mc[e & 7], s[c], s[c + 1]);
            float x0, x1;
            f2unpack(ffma2(f2pack(s[c], s[c + 1]), cs2, nm2), x0, x1);
            const float p0 = ex2_approx(x0);
            const float p1 = ex2_approx(x1);
            acc[e & 3] = fadd2(acc[e & 3], f2pack(p0, p1));
            if constexpr (FP8V) {
              if (e & 1) {
                pk[e >> 1] = pack4_e5m2(q0, q1, p0, p1);
              } else {
                q0 = p0;
                q1 = p1;
              }
            } else {
              pk[e] = pack2<BF16>(p0, p1);
            }
          }
          tmem_st16(tS + i * 16, pk);
        }
        const float mx = fmax3(fmax3(mc[0], mc[1], mc[2]), fmax3(mc[3], mc[4], mc[5]), fmaxf(mc[6], mc[7]));
        const bool need = mx * cs > m + kMaxGrowth<FP8V, LAZY8>;
        if (!__any_sync(0xffffffffu, need)) {
          float a0, a1;
          f2unpack(fadd2(fadd2(acc[0], acc[1]), fadd2(acc[2], acc[3])), a0, a1);
          l += a0 + a1;
          done = true;
        }
      }
      if (!done) {
        // First tile, or a running max grew by more than 2^8 in this warp:
        // new max, O and l rescaled, p recomputed.
        // row max: eight independent chains of 3-input max
        float mc[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) mc[i] = fmaxf(s[2 * i], s[2 * i + 1]);
#pragma unroll
        for (int c = 16; c < kBN; c += 16) {
#pragma unroll
          for (int i = 0; i < 8; ++i) mc[i] = fmax3(mc[i], s[c + 2 * i], s[c + 2 * i + 1]);
        }
        const float mx = fmax3(fmax3(mc[0], mc[1], mc[2]), fmax3(mc[3], mc[4], mc[5]), fmaxf(mc[6], mc[7]));
        const float m_tile = mx * cs;
        if (j == 0) {
          m = m_tile;
        } else {
          const bool need = m_tile > m + kMaxGrowth<FP8V, LAZY8>;
          const float m_new = need ? m_tile : m;
          const float alpha = ex2_approx(m - m_new);
          m = m_new;
          l *= alpha;
          const uint64_t a2 = f2pack(alpha, alpha);
#pragma unroll
          for (int c = 0; c < D / 16; ++c) {
            uint32_t o[16];
            tmem_ld16(tO + c * 16, o);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 16; e += 2) {
              float lo, hi;
              f2unpack(fmul2(f2pack(__uint_as_float(o[e]), __uint_as_float(o[e + 1])), a2), lo, hi);
              o[e] = __float_as_uint(lo);
              o[e + 1] = __float_as_uint(hi);
            }
            tmem_st16(tO + c * 16, o);
          }
        }
        const float mb = (m == -CUDART_INF_F) ? 0.f : m;

        // p = exp2(c s - m) two at a time (packed FFMA), row sum in four
        // independent packed accumulators
        const uint64_t nm2 = f2pack(-mb, -mb);
        uint64_t acc[4] = {0ull, 0ull, 0ull, 0ull};
#pragma unroll
        for (int i = 0; i < kBN / kPChunk; ++i) {
          uint32_t pk[16];
          float q0 = 0.f, q1 = 0.f;
#pragma unroll
          for (int e = 0; e < kPChunk / 2; ++e) {
            const int c = i * kPChunk + 2 * e;
            float x0, x1;
            f2unpack(ffma2(f2pack(s[c], s[c + 1]), cs2, nm2), x0, x1);
            const float p0 = ex2_approx(x0);
            const float p1 = ex2_approx(x1);
            acc[e & 3] = fadd2(acc[e & 3], f2pack(p0, p1));
            if constexpr (FP8V) {
              if (e & 1) {
                pk[e >> 1] = pack4_e5m2(q0, q1, p0, p1);
              } else {
                q0 = p0;
                q1 = p1;
              }
            } else {
              pk[e] = pack2<BF16>(p0, p1);
            }
          }
          tmem_st16(tS + i * 16, pk);
        }
        float a0, a1;
        f2unpack(fadd2(fadd2(acc[0], acc[1]), fadd2(acc[2], acc[3])), a0, a1);
        l += a0 + a1;
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar_p[t]);
    }

    if (p.n_splits > 1) {
      if (n > 0) {
        mbar_wait(&bar_o[t], 0, p.err, 10);
        tc_fence_after();
      }
      store_partial<D>(p, tO, bh, split, qrow, m, l, n > 0);
    } else if (n > 0) {
      mbar_wait(&bar_o[t], 0, p.err, 10);   // committed once, after the last PV
      tc_fence_after();
      store_o_lse<D, BF16>(p, tO, b, h, qrow, m, l);
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
// Forward with P in TMEM columns of its own (d <= 96)
// ---------------------------------------------------------------------------
// Tensor memory: S_0 [0, 128), S_1 [128, 256), O_0 [256, 256 + D),
// O_1 [256 + D, 256 + 2 D), and one 64-column P buffer after them that the two
// query tiles take turns on.  Because P no longer overwrites S, a softmax
// warp releases S_t,j as soon as it holds it in registers and S_t,j+1 is
// computed while it works; the tensor cores then wait on a tile's softmax
// only through its PV.
//   warps 0-7   softmax / correction / epilogue (tile t = warp / 4, one row
//               per thread), 224 registers each
//   warp  8     TMA producer: Q tiles, then K_j (even ring slots) and V_j
//               (odd ring slots)
//   warp  9     issuer A: S_t,j = Q_t K_j^T (also allocates TMEM)
//   warp  10    issuer B: O_t += P V_j
//   warp  11    idle (completes the third warpgroup for the register split)
// Writes to the P buffer go in the order (j, t): P_0,0, P_1,0, P_0,1, ...
// (tiles without key tile j skipped); issuer B issues the PVs in the same
// order.  A write waits for the PV of the write before it, through that
// tile's PV barrier at that tile's step: then the buffer is free and, since
// one issuer's MMAs complete in order, the writer's own PV_t,j-1 is done and
// O_t may be rescaled.  Per-tile barriers keep every parity wait at most one
// phase behind its barrier (a single barrier counting all PVs could be two
// phases behind a softmax warp that ran ahead).
// P gets TMEM columns of its own when S_0, S_1, O_0, O_1 and a 64-column P
// buffer fit in 512 columns (d <= 96).
template <int D>
constexpr bool kSepP = 256 + 2 * D + 64 <= 512;

// One work item of the separate-P forward: the key tiles of split `split` for
// the query-tile pair of rank `rank` (0 = the heaviest) of head bh.  An item
// with n_max == 0 has no work.
struct SpItem {
  int b, h, bh, split, q0, kt0, n_max;
  int nkt[kNQT];   // key tiles of query tile t: [kt0, kt0 + nkt[t])
};

__device__ __forceinline__ SpItem sp_item(const FwdParams& p, int rank, int bh, int split) {
  SpItem it;
  it.split = split;
  it.bh = bh;
  const int pair = p.n_pairs - 1 - rank;
  it.b = bh / p.H;
  it.h = bh % p.H;
  it.q0 = pair * (p.single_tile ? kBM : kNQT * kBM);
  it.kt0 = split * p.tiles_per_split;
  it.n_max = 0;
#pragma unroll
  for (int t = 0; t < kNQT; ++t) {
    it.nkt[t] = t > 0 && p.single_tile
                    ? 0
                    : max(0, min(key_tiles(it.q0 + t * kBM, p.Nq, p.Nk, p.causal), it.kt0 + p.tiles_per_split) - it.kt0);
    it.n_max = max(it.n_max, it.nkt[t]);
  }
  return it;
}

// The q-th work item of this block; false past its last one.
// Without persistent blocks (grid_p == 0) block w takes the single item w:
// split w % n_splits of the pair of rank w / n_splits in chunked_order.
// Otherwise the work is cut into units: unit u of head bh holds the pairs of
// ranks r and n_pairs - 1 - r (the heaviest with the lightest, so that under
// the causal mask every unit has the same number of key tiles; an odd middle
// pair is alone), units in chunked_order.  Block b < grid_p walks the units
// b, b + grid_p, ... below persist_units, two items each; each later block
// takes one item of the remaining units, first items (heavy) in unit order,
// then second items (light) in reverse, so that the hardware hands the
// leftover work out heaviest first.
__device__ __forceinline__ bool sp_next(const FwdParams& p, int q, SpItem* it) {
  const int BH = p.B * p.H;
  const int bid = static_cast<int>(blockIdx.x);
  int r, bh;
  if (p.grid_p == 0) {
    if (q > 0) return false;
    chunked_order(bid / p.n_splits, p.n_pairs, BH, &r, &bh);
    *it = sp_item(p, r, bh, bid % p.n_splits);
    return true;
  }
  const int units = (p.n_pairs + 1) / 2;
  int u, second;
  if (bid < p.grid_p) {
    u = bid + (q >> 1) * p.grid_p;
    if (u >= p.persist_units) return false;
    second = q & 1;
  } else {
    if (q > 0) return false;
    const int n_tail = units * BH - p.persist_units;
    const int ti = bid - p.grid_p;
    second = ti >= n_tail ? 1 : 0;
    u = p.persist_units + (second ? 2 * n_tail - 1 - ti : ti);
  }
  chunked_order(u, units, BH, &r, &bh);
  const int rank = second ? p.n_pairs - 1 - r : r;
  if (second && rank == r) {   // the odd middle pair: no second item
    it->n_max = 0;
    it->nkt[0] = it->nkt[1] = 0;
    it->b = it->h = it->bh = it->split = it->q0 = it->kt0 = 0;
    return true;
  }
  *it = sp_item(p, rank, bh, 0);
  return true;
}

// SMALL: the one-query-tile build (d = 64): one softmax
// warpgroup, 256 TMEM columns, a 4-slot ring and a 128-register launch, so
// that two blocks share an SM; each tile's K/V stream is its own, and the two
// blocks of an SM run out of step with each other.
template <int D, bool SMALL = false>
struct FwdSpCfg {
  using G = TileGeo<D>;
  static constexpr int TILE = G::TILE;
  static constexpr int NT = SMALL ? 1 : kNQT;        // query tiles with softmax warps
  static constexpr int NSTAGE = SMALL ? 4 : (D == 64 ? 8 : 6);   // even: K_j in even slots, V_j in odd
  static constexpr int SMEM_DATA = NT * TILE + NSTAGE * TILE;
  static constexpr int NBARS = 2 * kNQT + 2 * NSTAGE + 4 * kNQT + 3;
  static constexpr int SMEM = 1024 + SMEM_DATA + NBARS * 8 + 16;
  static constexpr int THREADS = NT * 128 + 128;
  static constexpr int BLOCKS_PER_SM = SMALL ? 2 : 1;
  static constexpr int LAUNCH_REGS = SMALL ? 128 : 168;   // registers a thread launches with
  static constexpr int PROD_WARP = NT * 4;
  static constexpr int MMA_WARP = NT * 4 + 1;   // issuer A; issuer B is the warp after it
  static constexpr uint32_t TMEM_COLS = SMALL ? 256 : 512;
  static constexpr uint32_t kColO = NT * 128;   // O_t at kColO + t * D (S_t at t * 128)
  static constexpr uint32_t kColP = kColO + NT * D;
  // Register split: the softmax warpgroups grow, the last warpgroup
  // (producer, issuers) shrinks, within the block's launch registers:
  // 384 x 168 = 64,512 >= 2 * 128 * 224 + 128 * 56; SMALL: 256 x 128 =
  // 32,768 >= 128 * 208 + 128 * 48.
  static constexpr uint32_t kRegSoftmax = SMALL ? 208 : 224;
  static constexpr uint32_t kRegOther = SMALL ? 48 : 56;
  static_assert(!SMALL || D == 64, "the one-tile build fits d = 64");
  static_assert(NSTAGE % 2 == 0, "K and V alternate between even and odd slots");
  static_assert(kColP + 64 <= TMEM_COLS, "TMEM budget");
  static_assert(NT * 128 * kRegSoftmax + 128 * kRegOther <= THREADS * LAUNCH_REGS,
                "register split exceeds the launch");
  static_assert(SMEM * BLOCKS_PER_SM <= 227 * 1024, "shared memory budget");
};

template <int D, bool BF16, bool FP8V, bool LAZY8 = false, bool SMALL = false>
__global__ void __launch_bounds__(FwdSpCfg<D, SMALL>::THREADS, FwdSpCfg<D, SMALL>::BLOCKS_PER_SM)
    fwd_sp_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                  const __grid_constant__ CUtensorMap tmV, const FwdParams p) {
  using C = FwdSpCfg<D, SMALL>;
  if (p.n_splits > 1) griddep_launch_dependents();   // the merge may take SMs as blocks of this grid finish
  constexpr int NS = C::NSTAGE;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem;
  uint8_t* sKV = smem + C::NT * C::TILE;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sKV + NS * C::TILE);
  uint64_t* bar_q = bars;                      // [kNQT] Q_t landed
  uint64_t* bar_qfree = bar_q + kNQT;          // [kNQT] last S_t of an item complete: Q_t may be replaced
  uint64_t* bar_full = bar_qfree + kNQT;       // [NS]
  uint64_t* bar_empty = bar_full + NS;         // [NS] one release by the issuer that read the slot
  uint64_t* bar_s = bar_empty + NS;            // [kNQT] S_t,j complete
  uint64_t* bar_sfree = bar_s + kNQT;          // [kNQT] S_t,j in registers (one arrival per warp)
  uint64_t* bar_o = bar_sfree + kNQT;          // [kNQT] last PV of tile t complete
  uint64_t* bar_pv = bar_o + kNQT;             // [kNQT] PV_t,j complete (phase j)
  uint64_t* bar_pready = bar_pv + kNQT;        // next P write done (one arrival per warp of the writer)
  uint64_t* bar_item = bar_pready + 1;         // every PV of an item (with work) complete
  uint64_t* bar_drain = bar_item + 1;          // every MMA of both issuers complete
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar_drain + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int t = 0; t < kNQT; ++t) {
      mbar_init(&bar_q[t], 1);
      mbar_init(&bar_qfree[t], 1);
      mbar_init(&bar_s[t], 1);
      mbar_init(&bar_sfree[t], 4);
      mbar_init(&bar_o[t], 1);
      mbar_init(&bar_pv[t], 1);
    }
    for (int s = 0; s < NS; ++s) {
      mbar_init(&bar_full[s], 1);
      mbar_init(&bar_empty[s], 1);
    }
    mbar_init(bar_pready, 4);
    mbar_init(bar_item, 1);
    mbar_init(bar_drain, 2);
    fence_mbar_init();
  }
  if (warp == C::MMA_WARP) {
    tmem_alloc(tmem_slot, C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp >= C::PROD_WARP) {
   setmaxnreg_dec<C::kRegOther>();
   if (warp == C::PROD_WARP && lane == 0) {
      // ---------------------------------------------------------------- TMA
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      // Fill g (counted over all items of the block) of slot g % NS: fill
      // 2 j of an item holds its K_j, fill 2 j + 1 its V_j.  A slot is
      // refilled only after its previous fill has landed, so each slot has
      // at most one copy in flight; a give-up stops the fills and only the
      // fills issued are drained.
      int F = 0;                  // fills issued
      int qn[kNQT] = {0, 0};      // Q_t loads issued
      bool stop = false;
      for (int r = 0; !stop; ++r) {
        SpItem it;
        if (!sp_next(p, r, &it)) break;
#pragma unroll
        for (int t = 0; t < kNQT; ++t) {
          if (it.nkt[t] == 0 || stop) continue;
          // Q_t of the previous item is no longer read by its S MMAs.
          if (qn[t] > 0 && !mbar_wait(&bar_qfree[t], (qn[t] - 1) & 1, p.err, 14)) {
            stop = true;
            continue;
          }
          mbar_arrive_expect_tx(&bar_q[t], C::TILE);
          for (int c = 0; c < C::G::NCH; ++c)
            tma_load_4d(sQ + t * C::TILE + c * C::G::CHB, &tmQ, &bar_q[t], c * C::G::CC, it.q0 + t * kBM, it.h, it.b);
          ++qn[t];
        }
        for (int f = 0; f < 2 * it.n_max && !stop; ++f) {
          const int g = F;
          const int s = g % NS;
          const int use = g / NS;
          if (use > 0 && (!mbar_wait(&bar_empty[s], (use - 1) & 1, p.err, 1) ||
                          !mbar_wait_drain(&bar_full[s], (use - 1) & 1))) {
            stop = true;
            break;
          }
          const int kt = it.kt0 + (f >> 1);
          if (FP8V && (f & 1)) {
            // V_j^T: D rows of 128 keys, one box
            mbar_arrive_expect_tx(&bar_full[s], D * kBN);
            tma_load_4d(sKV + s * C::TILE, &tmV, &bar_full[s], kt * kBN, 0, it.h, it.b);
          } else {
            mbar_arrive_expect_tx(&bar_full[s], C::TILE);
            const CUtensorMap* map = (f & 1) ? &tmV : &tmK;
            for (int c = 0; c < C::G::NCH; ++c)
              tma_load_4d(sKV + s * C::TILE + c * C::G::CHB, map, &bar_full[s], c * C::G::CC, kt * kBN, it.h, it.b);
          }
          ++F;
        }
      }
      for (int g = max(0, F - NS); g < F; ++g) mbar_wait_drain(&bar_full[g % NS], (g / NS) & 1);
#pragma unroll
      for (int t = 0; t < kNQT; ++t)
        if (qn[t] > 0) mbar_wait_drain(&bar_q[t], (qn[t] - 1) & 1);
   } else if (warp == C::MMA_WARP) {
    // ------------------------------------------------------ issuer A: S MMAs
    const uint32_t sq_addr = smem_u32(sQ);
    const uint32_t skv_addr = smem_u32(sKV);
    int F = 0;                  // fills of the items before this one
    int sc[kNQT] = {0, 0};      // S_t issued
    int qn[kNQT] = {0, 0};      // items before this one that had tile t
    for (int r = 0;; ++r) {
      SpItem it;
      if (!sp_next(p, r, &it)) break;
      for (int j = 0; j < it.n_max; ++j) {
        const int g = F + 2 * j;
        mbar_wait(&bar_full[g % NS], (g / NS) & 1, p.err, 3);
#pragma unroll
        for (int t = 0; t < kNQT; ++t) {
          if (j >= it.nkt[t]) continue;
          if (j == 0) mbar_wait(&bar_q[t], qn[t] & 1, p.err, 2);
          if (sc[t] > 0) mbar_wait(&bar_sfree[t], (sc[t] - 1) & 1, p.err, 13);   // S_t before this one read
          __syncwarp();
          tc_fence_after();
          issue_s<D, BF16>(tmem + t * 128, sq_addr + t * C::TILE, skv_addr + (g % NS) * C::TILE);
          if (elect_one()) {
            umma_commit(&bar_s[t]);
            if (j == it.nkt[t] - 1) umma_commit(&bar_qfree[t]);   // last S_t of the item: Q_t free
          }
          ++sc[t];
        }
        if (elect_one()) umma_commit(&bar_empty[g % NS]);   // K_j read by every S of step j
      }
      F += 2 * it.n_max;
#pragma unroll
      for (int t = 0; t < kNQT; ++t) qn[t] += it.nkt[t] > 0 ? 1 : 0;
    }
    if (elect_one()) umma_commit(bar_drain);
    __syncwarp();
    mbar_wait_drain(bar_drain, 0);
   } else if (warp == C::MMA_WARP + 1) {
    // ----------------------------------------------------- issuer B: PV MMAs
    const uint32_t skv_addr = smem_u32(sKV);
    int F = 0;   // fills of the items before this one
    int k = 0;   // number of the next P write
    for (int r = 0;; ++r) {
      SpItem it;
      if (!sp_next(p, r, &it)) break;
      for (int j = 0; j < it.n_max; ++j) {
        const int g = F + 2 * j + 1;
        mbar_wait(&bar_full[g % NS], (g / NS) & 1, p.err, 4);
#pragma unroll
        for (int t = 0; t < kNQT; ++t) {
          if (j >= it.nkt[t]) continue;
          mbar_wait(bar_pready, k & 1, p.err, 5);
          __syncwarp();
          tc_fence_after();
          if constexpr (FP8V)
            issue_pv_f8<D>(tmem + C::kColO + t * D, tmem + C::kColP, skv_addr + (g % NS) * C::TILE, j > 0);
          else
            issue_pv<D, BF16>(tmem + C::kColO + t * D, tmem + C::kColP, skv_addr + (g % NS) * C::TILE, j > 0);
          if (elect_one()) {
            umma_commit(&bar_pv[t]);
            if (j == it.nkt[t] - 1) umma_commit(&bar_o[t]);
          }
          ++k;
        }
        if (elect_one()) umma_commit(&bar_empty[g % NS]);   // V_j read by every PV of step j
      }
      if (it.n_max > 0 && elect_one()) umma_commit(bar_item);
      F += 2 * it.n_max;
    }
    if (elect_one()) umma_commit(bar_drain);
    __syncwarp();
    mbar_wait_drain(bar_drain, 0);
   }
  } else {
    setmaxnreg_inc<C::kRegSoftmax>();
    // ------------------------------------------------- softmax / epilogue
    const int t = warp >> 2;
    const int quad = warp & 3;
    const int row = quad * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
    const uint32_t tS = tmem + lane_off + t * 128;
    const uint32_t tO = tmem + lane_off + C::kColO + t * D;
    const uint32_t tP = tmem + lane_off + C::kColP;
    const float cs = p.scale_log2;
    const uint64_t cs2 = f2pack(cs, cs);
    int sc = 0;                 // S_t read (phase of bar_s[t])
    int on = 0;                 // items before this one with keys for tile t (phase of bar_o[t])
    int pvb[kNQT] = {0, 0};     // PVs of each tile in the items before this one
    int ni = 0;                 // items before this one with work (phase of bar_item)

    for (int r = 0;; ++r) {
      SpItem it;
      if (!sp_next(p, r, &it)) break;
      const int r0 = it.q0 + t * kBM;
      const int qrow = r0 + row;
      const int n = it.nkt[t];

      float m = -CUDART_INF_F;  // running max of the scaled scores (log2 domain)
      float l = 0.f;            // running sum of exp2(score - m)

      for (int j = 0; j < n; ++j) {
        mbar_wait(&bar_s[t], sc & 1, p.err, 8);
        ++sc;
        tc_fence_after();
        float s[kBN];
        {
          uint32_t r0_[32], r1_[32], r2_[32], r3_[32];
          tmem_ld32(tS, r0_);
          tmem_ld32(tS + 32, r1_);
          tmem_ld32(tS + 64, r2_);
          tmem_ld32(tS + 96, r3_);
          tmem_wait_ld(r3_);
          tmem_reg_tie(r0_);
          tmem_reg_tie(r1_);
          tmem_reg_tie(r2_);
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            s[e] = __uint_as_float(r0_[e]);
            s[32 + e] = __uint_as_float(r1_[e]);
            s[64 + e] = __uint_as_float(r2_[e]);
            s[96 + e] = __uint_as_float(r3_[e]);
          }
        }
        // S_t,j is in registers: the tensor cores may overwrite it with S_t,j+1.
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bar_sfree[t]);

        const int kbase = (it.kt0 + j) * kBN;
        if (kbase + kBN > p.Nk || (p.causal && kbase + kBN - 1 > r0)) {
          const int lim = p.causal ? min(p.Nk, qrow + 1) : p.Nk;  // keys < lim are visible
#pragma unroll
          for (int c = 0; c < kBN; ++c)
            if (kbase + c >= lim) s[c] = -CUDART_INF_F;
        }
        // The write before this one in this item (tile pt, that tile's PV
        // number pn), or none: the item's first write, by tile 0, which
        // instead waits for every PV of the items before (bar_item).  A
        // parity wait must be at most one phase behind its barrier; tile 0
        // waits on bar_item at every item and, with every item giving tile
        // 0 keys and tile 1 at least as many (the launcher only walks
        // several items per block then), no other wait of this loop can fall
        // two phases behind either.
        int pt = -1, pn = 0;
        if (t == 1 && j < it.nkt[0]) {
          pt = 0;
          pn = pvb[0] + j;
        } else if (j > 0) {
          pt = (t == 0 && j - 1 < it.nkt[1]) ? 1 : t;
          pn = pvb[pt] + j - 1;
        }

        constexpr int NPK = FP8V ? kBN / 4 : kBN / 2;   // P registers (and TMEM columns) per row
        uint32_t pk[NPK];
        bool done = false;
        bool grew = false;   // FP8V: some row of this warp has a new max (O must be rescaled)
        float alpha8 = 1.f;
        if (FP8V && !LAZY8 && j > 0) {
          // e5m2 P: the max first, then one pass against the new running max
          // (the scale the page's steps take p at), O rescaled below if a
          // row of this warp grew.
          float mc[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) mc[i] = fmaxf(s[2 * i], s[2 * i + 1]);
#pragma unroll
          for (int c = 16; c < kBN; c += 16) {
#pragma unroll
            for (int i = 0; i < 8; ++i) mc[i] = fmax3(mc[i], s[c + 2 * i], s[c + 2 * i + 1]);
          }
          const float mx = fmax3(fmax3(mc[0], mc[1], mc[2]), fmax3(mc[3], mc[4], mc[5]), fmaxf(mc[6], mc[7]));
          const float m_new = fmaxf(m, mx * cs);
          alpha8 = m == -CUDART_INF_F ? 0.f : ex2_approx(m - m_new);
          grew = __any_sync(0xffffffffu, m_new > m);
          m = m_new;
          const float mb = (m == -CUDART_INF_F) ? 0.f : m;
          l = l * alpha8 + exp_pack<BF16, FP8V>(s, cs2, f2pack(-mb, -mb), pk);
#pragma unroll
          for (int i = 0; i < NPK / 32; ++i) tmem_reg_tie(*reinterpret_cast<uint32_t(*)[32]>(&pk[32 * i]));
          done = true;
        } else if (j > 0) {
          // Common case: p = exp2(c s - m) against the running max m.  A row
          // sum <= 2^8 bounds every p of the row by 2^8, i.e. its max grew by
          // at most 8 and the exact path below would keep m: this P is its
          // result.
          const float sum = exp_pack<BF16, FP8V>(s, cs2, f2pack(-m, -m), pk);
          // P complete before the wait for the buffer: the compiler may
          // otherwise sink its conversions past the wait.
#pragma unroll
          for (int i = 0; i < NPK / 32; ++i) tmem_reg_tie(*reinterpret_cast<uint32_t(*)[32]>(&pk[32 * i]));
          if (!__any_sync(0xffffffffu, !(sum <= kFastSumBound))) {
            l += sum;
            done = true;
          }
        }
        if (pt >= 0)
          mbar_wait(&bar_pv[pt], pn & 1, p.err, 9);
        else if (ni > 0)
          mbar_wait(bar_item, (ni - 1) & 1, p.err, 15);
        tc_fence_after();
        if (FP8V && grew) {
          // this tile's previous PV has completed (the wait above): O_t *= alpha
          const uint64_t a2 = f2pack(alpha8, alpha8);
#pragma unroll
          for (int c = 0; c < D / 16; ++c) {
            uint32_t o[16];
            tmem_ld16(tO + c * 16, o);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 16; e += 2) {
              float lo, hi;
              f2unpack(fmul2(f2pack(__uint_as_float(o[e]), __uint_as_float(o[e + 1])), a2), lo, hi);
              o[e] = __float_as_uint(lo);
              o[e + 1] = __float_as_uint(hi);
            }
            tmem_st16(tO + c * 16, o);
          }
        }
        if (!done) {
          // First tile, or a row of this warp may have grown by more than 2^8:
          // tile max, O_t and l rescaled if the max grew by more than 2^8, p.
          float mc[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) mc[i] = fmaxf(s[2 * i], s[2 * i + 1]);
#pragma unroll
          for (int c = 16; c < kBN; c += 16) {
#pragma unroll
            for (int i = 0; i < 8; ++i) mc[i] = fmax3(mc[i], s[c + 2 * i], s[c + 2 * i + 1]);
          }
          const float mx = fmax3(fmax3(mc[0], mc[1], mc[2]), fmax3(mc[3], mc[4], mc[5]), fmaxf(mc[6], mc[7]));
          const float m_tile = mx * cs;
          if (j == 0) {
            m = m_tile;
          } else {
            const bool need = m_tile > m + kMaxGrowth<FP8V, LAZY8>;
            const float m_new = need ? m_tile : m;
            const float alpha = ex2_approx(m - m_new);
            m = m_new;
            l *= alpha;
            const uint64_t a2 = f2pack(alpha, alpha);
#pragma unroll
            for (int c = 0; c < D / 16; ++c) {
              uint32_t o[16];
              tmem_ld16(tO + c * 16, o);
              tmem_wait_ld();
#pragma unroll
              for (int e = 0; e < 16; e += 2) {
                float lo, hi;
                f2unpack(fmul2(f2pack(__uint_as_float(o[e]), __uint_as_float(o[e + 1])), a2), lo, hi);
                o[e] = __float_as_uint(lo);
                o[e + 1] = __float_as_uint(hi);
              }
              tmem_st16(tO + c * 16, o);
            }
          }
          const float mb = (m == -CUDART_INF_F) ? 0.f : m;
          l += exp_pack<BF16, FP8V>(s, cs2, f2pack(-mb, -mb), pk);
        }
#pragma unroll
        for (int i = 0; i < NPK / 16; ++i) tmem_st16(tP + i * 16, *reinterpret_cast<uint32_t(*)[16]>(&pk[i * 16]));
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_pready);
      }

      // Epilogue.  O_t is read before this warp's next P write, so the
      // next item's first PV (which overwrites O_t) cannot start earlier.
      if (n > 0) {
        mbar_wait(&bar_o[t], on & 1, p.err, 10);
        ++on;
        tc_fence_after();
      }
      if (p.n_splits > 1) {
        // (with one query tile per block, tile 1's rows belong to the next block)
        if (t == 0 || !p.single_tile) store_partial<D>(p, tO, it.bh, it.split, qrow, m, l, n > 0);
      } else if (n > 0) {
        store_o_lse_batched<D, BF16>(p, tO, it.b, it.h, qrow, m, l);
      }

      ni += it.n_max > 0 ? 1 : 0;
#pragma unroll
      for (int u = 0; u < kNQT; ++u) pvb[u] += it.nkt[u];
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == C::MMA_WARP) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

// ---------------------------------------------------------------------------
// Split-KV merge: one warp per query row
// ---------------------------------------------------------------------------
// lse = log sum_s exp(lse_s) and O = sum_s exp(lse_s - lse) O_s: the
// rescaling step of the online softmax applied to whole key ranges.
struct MergeParams {
  const float* part_o;
  const float* part_lse;
  int n_splits, BH, H, Nq, Nqp;
  void* o;
  int64_t o_sb, o_sh, o_ss;
  float* lse;
};

template <int D, bool BF16>
__global__ void __launch_bounds__(128) fwd_merge_kernel(const MergeParams mp) {
  // Launched as a programmatic dependent of the partial forward: its blocks
  // may start before that grid ends, and wait here for its partials.
  griddep_wait();
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const long long r = static_cast<long long>(blockIdx.x) * 4 + warp;
  if (r >= static_cast<long long>(mp.BH) * mp.Nq) return;
  const int bh = static_cast<int>(r / mp.Nq);
  const int q = static_cast<int>(r % mp.Nq);
  const size_t stride = static_cast<size_t>(mp.BH) * mp.Nqp;   // rows between splits
  const size_t row0 = static_cast<size_t>(bh) * mp.Nqp + q;
  float mx = -CUDART_INF_F;
  for (int s = 0; s < mp.n_splits; ++s) mx = fmaxf(mx, mp.part_lse[row0 + s * stride]);
  float wsum = 0.f;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  const bool col = lane < D / 4;   // this lane's 4 columns
  if (mx != -CUDART_INF_F) {
    for (int s = 0; s < mp.n_splits; ++s) {
      const size_t row = row0 + s * stride;
      const float w = expf(mp.part_lse[row] - mx);
      wsum += w;
      if (col && w != 0.f) {
        const float4 v = reinterpret_cast<const float4*>(mp.part_o + row * D)[lane];
        acc.x += w * v.x;
        acc.y += w * v.y;
        acc.z += w * v.z;
        acc.w += w * v.w;
      }
    }
  }
  const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
  const int b = bh / mp.H;
  const int h = bh % mp.H;
  if (col) {
    uint8_t* orow = reinterpret_cast<uint8_t*>(mp.o) +
                    2 * (static_cast<int64_t>(b) * mp.o_sb + static_cast<int64_t>(h) * mp.o_sh +
                         static_cast<int64_t>(q) * mp.o_ss);
    uint2 w2;
    w2.x = pack2<BF16>(acc.x * inv, acc.y * inv);
    w2.y = pack2<BF16>(acc.z * inv, acc.w * inv);
    reinterpret_cast<uint2*>(orow)[lane] = w2;
  }
  if (lane == 0) mp.lse[static_cast<size_t>(bh) * mp.Nq + q] = wsum > 0.f ? mx + logf(wsum) : -CUDART_INF_F;
}

template <int D, bool BF16, bool FP8V, bool LAZY8 = false>
cudaError_t launch_fwd_t(const FwdArgs& a, cudaStream_t stream) {
  using C = FwdCfg<D>;
  CUtensorMap tq, tk, tv;
  const bool v_ok = FP8V ? make_vt_map(&tv, a.v.ptr, a.vt_ld, a.Nk, D, a.H, a.B)
                         : make_tile_map(&tv, a.v, D, a.Nk, a.H, a.B, BF16);
  if (!make_tile_map(&tq, a.q, D, a.Nq, a.H, a.B, BF16) || !make_tile_map(&tk, a.k, D, a.Nk, a.H, a.B, BF16) || !v_ok)
    return cudaErrorInvalidValue;
  FwdParams p;
  p.B = a.B;
  p.H = a.H;
  p.Nq = a.Nq;
  p.Nk = a.Nk;
  p.n_pairs = (a.Nq + kNQT * kBM - 1) / (kNQT * kBM);
  p.causal = a.causal;
  p.scale_log2 = a.sm_scale * 1.4426950408889634f;
  p.o = const_cast<void*>(a.o.ptr);
  p.o_sb = a.o.sb;
  p.o_sh = a.o.sh;
  p.o_ss = a.o.ss;
  p.lse = a.lse;
  p.err = a.err;
  const int n_kt = (a.Nk + kBN - 1) / kBN;
  const int n_splits = a.n_splits > 1 ? a.n_splits : 1;
  p.n_splits = n_splits;
  p.tiles_per_split = (n_kt + n_splits - 1) / n_splits;
  p.Nqp = nq_pad(a.Nq);
  p.part_o = n_splits > 1 ? a.part : nullptr;
  p.part_lse = n_splits > 1 ? a.part + static_cast<size_t>(n_splits) * a.B * a.H * p.Nqp * D : nullptr;
  const long long blocks = static_cast<long long>(p.n_pairs) * a.B * a.H * n_splits;
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidValue;
  if constexpr (kSepP<D>) {
    using CS = FwdSpCfg<D>;
    auto kern = fwd_sp_kernel<D, BF16, FP8V, LAZY8>;
    // setmaxnreg.inc waits until the block's launch registers cover the
    // split: never launch a build whose register count would not.
    static const int num_regs = [&] {
      cudaFuncAttributes fattr{};
      return cudaFuncGetAttributes(&fattr, kern) == cudaSuccess ? fattr.numRegs : 0;
    }();
    if (num_regs * CS::THREADS < 2 * 128 * static_cast<int>(CS::kRegSoftmax) + 128 * static_cast<int>(CS::kRegOther))
      return cudaErrorInvalidConfiguration;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, CS::SMEM);
    if (e != cudaSuccess) return e;
    int dev = 0, sms = 0;
    e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    long long grid = blocks;
    const int pair_rows = kNQT * kBM;
    const int n_tiles = (a.Nq + kBM - 1) / kBM;
    const long long tile_blocks = static_cast<long long>(n_tiles) * a.B * a.H * n_splits;
    bool small = false;
    if constexpr (D == 64) {
      // The one-tile build, two blocks per SM, whenever one-tile blocks
      // outnumber the SMs: unsplit, or split with the two-tile grid under one
      // wave and the one-tile grid within two blocks per SM.  Only if this
      // build's launch registers cover its register split.
      using CM = FwdSpCfg<D, true>;
      auto km = fwd_sp_kernel<D, BF16, FP8V, LAZY8, true>;
      static const int m_regs = [&] {
        cudaFuncAttributes fattr{};
        return cudaFuncGetAttributes(&fattr, km) == cudaSuccess ? fattr.numRegs : 0;
      }();
      const long long slots = 2LL * sms;   // resident one-tile blocks
      if (tile_blocks > sms && (n_splits == 1 || (blocks < sms && tile_blocks <= slots)) &&
          m_regs * CM::THREADS >= 128 * static_cast<int>(CM::kRegSoftmax) + 128 * static_cast<int>(CM::kRegOther)) {
        e = cudaFuncSetAttribute(km, cudaFuncAttributeMaxDynamicSharedMemorySize, CM::SMEM);
        if (e != cudaSuccess) return e;
        p.single_tile = 1;
        p.n_pairs = n_tiles;
        long long grid_m = tile_blocks;
        if (n_splits == 1) {
          // Walking blocks, two per SM, for all but about one round of the
          // units (a unit: the query tiles of ranks r and n_tiles - 1 - r of
          // one head; see sp_next).  With one tile per item every non-empty
          // item has tile 0 keys, so no shape condition is needed.
          const long long units = static_cast<long long>((n_tiles + 1) / 2) * a.B * a.H;
          const long long rounds = units / slots - 1;
          if (rounds >= 1) {
            p.grid_p = static_cast<int>(slots);
            p.persist_units = static_cast<int>(rounds * slots);
            grid_m = slots + 2 * (units - p.persist_units);
          }
        }
        km<<<static_cast<unsigned>(grid_m), CM::THREADS, CM::SMEM, stream>>>(tq, tk, tv, p);
        small = true;
      }
    }
    if (!small) {
      if (blocks < sms && tile_blocks > blocks && tile_blocks <= sms) {
        // Under one wave: one query tile per block still fits in one wave.
        p.single_tile = 1;
        p.n_pairs = n_tiles;
        grid = tile_blocks;
      } else if (n_splits == 1 && (a.Nq % pair_rows == 0 || a.Nq % pair_rows > kBM)) {
        // Persistent blocks for all but about one round of the units (see
        // sp_next), when every item gives tile 0 keys and tile 1 at least as
        // many: no split, and no pair whose second tile lies wholly past Nq.
        const long long units = static_cast<long long>((p.n_pairs + 1) / 2) * a.B * a.H;
        const long long rounds = sms > 0 ? units / sms - 1 : 0;
        if (rounds >= 1) {
          p.grid_p = sms;
          p.persist_units = static_cast<int>(rounds * sms);
          grid = sms + 2 * (units - p.persist_units);
        }
      }
      kern<<<static_cast<unsigned>(grid), CS::THREADS, CS::SMEM, stream>>>(tq, tk, tv, p);
    }
  } else {
    auto kern = fwd_kernel<D, BF16, FP8V, LAZY8>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) return e;
    kern<<<static_cast<unsigned>(blocks), C::THREADS, C::SMEM, stream>>>(tq, tk, tv, p);
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess || n_splits == 1) return e;
  MergeParams mp;
  mp.part_o = p.part_o;
  mp.part_lse = p.part_lse;
  mp.n_splits = n_splits;
  mp.BH = a.B * a.H;
  mp.H = a.H;
  mp.Nq = a.Nq;
  mp.Nqp = p.Nqp;
  mp.o = p.o;
  mp.o_sb = p.o_sb;
  mp.o_sh = p.o_sh;
  mp.o_ss = p.o_ss;
  mp.lse = a.lse;
  const long long rows = static_cast<long long>(mp.BH) * a.Nq;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>((rows + 3) / 4));
  cfg.blockDim = dim3(128);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, fwd_merge_kernel<D, BF16>, mp);
}

}  // namespace

cudaError_t launch_fwd(const FwdArgs& a, cudaStream_t stream) {
  if (a.fp8v && a.fp8_lazy) {
    if (a.n_splits > 1) return cudaErrorInvalidValue;
    switch (a.d) {
      case 64:
        return a.bf16 ? launch_fwd_t<64, true, true, true>(a, stream) : launch_fwd_t<64, false, true, true>(a, stream);
      case 80:
        return a.bf16 ? launch_fwd_t<80, true, true, true>(a, stream) : launch_fwd_t<80, false, true, true>(a, stream);
      case 128:
        return a.bf16 ? launch_fwd_t<128, true, true, true>(a, stream)
                      : launch_fwd_t<128, false, true, true>(a, stream);
      default: return cudaErrorInvalidValue;
    }
  }
  if (a.fp8v) {
    if (a.n_splits > 1) return cudaErrorInvalidValue;
    switch (a.d) {
      case 64: return a.bf16 ? launch_fwd_t<64, true, true>(a, stream) : launch_fwd_t<64, false, true>(a, stream);
      case 80: return a.bf16 ? launch_fwd_t<80, true, true>(a, stream) : launch_fwd_t<80, false, true>(a, stream);
      case 128:
        return a.bf16 ? launch_fwd_t<128, true, true>(a, stream) : launch_fwd_t<128, false, true>(a, stream);
      default: return cudaErrorInvalidValue;
    }
  }
  switch (a.d) {
    case 64: return a.bf16 ? launch_fwd_t<64, true, false>(a, stream) : launch_fwd_t<64, false, false>(a, stream);
    case 80: return a.bf16 ? launch_fwd_t<80, true, false>(a, stream) : launch_fwd_t<80, false, false>(a, stream);
    case 128:
      return a.bf16 ? launch_fwd_t<128, true, false>(a, stream) : launch_fwd_t<128, false, false>(a, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace fa
