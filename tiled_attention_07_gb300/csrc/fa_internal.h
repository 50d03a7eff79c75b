// fa_internal.h -- host-side interface between the C ABI layer (fa_api.cu)
// and the kernel translation units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace fa {

// One [B, H, seq, d] tensor: base pointer and element strides (d stride 1).
struct Tensor4 {
  const void* ptr;
  int64_t sb, sh, ss;
};

struct FwdArgs {
  Tensor4 q, k, v, o;
  float* lse;  // [B, H, Nq] fp32
  int B, H, Nq, Nk, d;
  float sm_scale;
  int causal;
  bool bf16;
  int* err;  // device error word
  // Split-KV (n_splits > 1): partial O_s then lse_s of every split, float32,
  // [n_splits][B*H][nq_pad(Nq)][d] and [n_splits][B*H][nq_pad(Nq)].
  int n_splits = 1;
  float* part = nullptr;
  // V in float8 e5m2, transposed: v.ptr is [B][H][d][vt_ld] bytes (key j of
  // head dim c at byte ((b H + h) d + c) vt_ld + j); P is cast to e5m2 for
  // the PV product.
  bool fp8v = false;
  int64_t vt_ld = 0;
  // e5m2 P under the lazy running-max rule instead of the page's steps
  bool fp8_lazy = false;
};

struct BwdArgs {
  Tensor4 q, k, v, o, dout, dq, dk, dv;
  const float* lse;  // [B, H, Nq] fp32
  float* ws;         // workspace: D and log2-domain LSE, [B*H][Nq_pad] each;
                     // fused: then the float32 dQ accumulator [B*H][Nq_pad][d]
  int B, H, Nq, Nk, d;
  float sm_scale;
  int causal;
  bool bf16;
  int* err;
  bool fused = false;   // one pass over key tiles for dK, dV and dQ (d = 64)
};

// Rows per query / key tile of every kernel (one TMEM lane per row).
constexpr int kTileRows = 128;

inline int nq_pad(int Nq) { return (Nq + kTileRows - 1) / kTileRows * kTileRows; }

// Columns per swizzle chunk of a 128-row shared-memory tile: 64 (128-byte
// rows, 128-byte swizzle) when d is a multiple of 64, else 32 (64-byte rows,
// 64-byte swizzle), so that d = 80 pads to 96 columns instead of 128.
__host__ __device__ constexpr int chunk_cols(int d) { return d % 64 == 0 ? 64 : 32; }

// Shared-memory geometry of one 128-row tile of a [.., d] tensor as TMA
// writes it: NCH chunks of 128 rows x CC columns, each chunk row-major with
// ROWB-byte rows, swizzled in 8-row atoms.
template <int D>
struct TileGeo {
  static constexpr int CC = chunk_cols(D);
  static constexpr int NCH = (D + CC - 1) / CC;
  static constexpr int ROWB = CC * 2;
  static constexpr int CHB = kTileRows * ROWB;
  static constexpr int TILE = NCH * CHB;
  static constexpr int SBO = 8 * ROWB;                // bytes between 8-row groups
  static constexpr uint32_t LAYOUT = CC == 64 ? 2u : 4u;   // UMMA descriptor: 128B / 64B swizzle
  static constexpr int KPC = CC / 16;                 // 16-wide K-steps per chunk
};

// Work order of the attention kernels: one block per (tile, head).  Heads
// are taken in chunks of kHeadChunk so that the blocks that run at the same
// time share K/V (or Q/dO) tiles through L2; inside a chunk the tiles go in
// the order 0, 1, 2, ... of `rank` (the caller maps rank 0 to its heaviest
// tile), with all heads of the chunk at one rank next to each other.
constexpr int kHeadChunk = 8;

__host__ __device__ inline void chunked_order(int lin, int n_tiles, int BH, int* rank, int* bh) {
  const int per_chunk = kHeadChunk * n_tiles;
  const int chunk = lin / per_chunk;
  const int heads = BH - chunk * kHeadChunk < kHeadChunk ? BH - chunk * kHeadChunk : kHeadChunk;
  const int r = lin - chunk * per_chunk;
  *rank = r / heads;
  *bh = chunk * kHeadChunk + r % heads;
}

// Encodes a 4-D TMA map {d, rows, H, B} with a {chunk_cols(d), 128, 1, 1}
// box and the matching swizzle.  Returns false if the driver rejects it.
bool make_tile_map(CUtensorMap* map, const Tensor4& t, int d, int rows, int H, int B, bool bf16);
// Tensor map of a transposed e5m2 V: boxes of 128 keys (one 128-byte row,
// 128-byte swizzle) by d rows.
bool make_vt_map(CUtensorMap* map, const void* vt, int64_t ld, int Nk, int d, int H, int B);

// Tensor map of a float32 [rows, cols] row-major matrix (cols * 4 bytes a
// multiple of 16) with 32-column x 128-row boxes and the 128-byte swizzle.
bool make_f32_rows_map(CUtensorMap* map, const float* base, int64_t rows, int cols);

cudaError_t launch_fwd(const FwdArgs& a, cudaStream_t stream);
// phase: 0 = all three launches; 1 = D / log2-LSE preprocess; 2 = dK, dV;
// 3 = dQ (phases 2 and 3 read what phase 1 wrote to the workspace).  With
// a.fused: 1 also zeroes the dQ accumulator, 2 = dK, dV and dQ's partial
// sums (added into the accumulator), 3 = dQ from the accumulator.
cudaError_t launch_bwd(const BwdArgs& a, int phase, cudaStream_t stream);
// Head dims the fused backward is built for.
inline bool bwd_fused_supported(int d) { return d == 64; }

}  // namespace fa
