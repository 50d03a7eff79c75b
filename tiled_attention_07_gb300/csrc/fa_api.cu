// fa_api.cu -- the C ABI of libfa.so: argument validation, TMA map encoding,
// the per-device error word, and dispatch to the forward / backward launchers.
// Declarations and the contract of every entry point are in include/fa.h.
#include "../../include/fa.h"
#include "fa_internal.h"

#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <limits>
#include <mutex>

namespace fa {

// Device error word: written by kernels whose bounded waits gave up.
__device__ int g_err_word;

namespace {

constexpr int kMaxDevices = 64;

std::mutex g_mu;
int* g_err_ptr[kMaxDevices];   // device address of g_err_word per device
bool g_err_init[kMaxDevices];

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;
bool g_encode_tried = false;

EncodeTiledFn get_encode() {
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_encode_tried) {
    g_encode_tried = true;
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<EncodeTiledFn>(fn);
  }
  return g_encode;
}

// Address of this device's error word (looked up once per device).
int* err_word(cudaError_t* e) {
  int dev = 0;
  *e = cudaGetDevice(&dev);
  if (*e != cudaSuccess) return nullptr;
  if (dev < 0 || dev >= kMaxDevices) {
    *e = cudaErrorInvalidDevice;
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_err_init[dev]) {
    void* ptr = nullptr;
    *e = cudaGetSymbolAddress(&ptr, g_err_word);
    if (*e != cudaSuccess) return nullptr;
    g_err_ptr[dev] = static_cast<int*>(ptr);
    g_err_init[dev] = true;
  }
  return g_err_ptr[dev];
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// a * b for a, b >= 0; -1 (an invalid stride) when either is negative or the
// product does not fit in int64.
int64_t mul_nonneg(int64_t a, int64_t b) {
  if (a < 0 || b < 0) return -1;
  if (a != 0 && b > std::numeric_limits<int64_t>::max() / a) return -1;
  return a * b;
}

// a * b saturated at SIZE_MAX, a size no buffer has.
size_t mul_sat(size_t a, size_t b) {
  return a != 0 && b > std::numeric_limits<size_t>::max() / a ? std::numeric_limits<size_t>::max() : a * b;
}

// TMA takes strides below 2^40 bytes.
constexpr int64_t kMaxStrideBytes = int64_t(1) << 40;

// A [B, H, rows, d] tensor view is valid for TMA and 16-byte vector access.
bool valid_tensor(const Tensor4& t) {
  if (t.ptr == nullptr || !aligned16(t.ptr)) return false;
  const int64_t st[3] = {t.sb, t.sh, t.ss};
  for (int64_t s : st) {
    if (s <= 0 || s >= kMaxStrideBytes / 2) return false;
    if ((s * 2) % 16 != 0) return false;
  }
  return true;
}

fa_status check_common(int B, int H, int Nq, int Nk, int d, float sm_scale, int causal, fa_dtype dtype) {
  if (B < 0 || H < 0 || Nq < 0 || Nk < 1) return FA_ERR_INVALID_ARG;
  if (Nq > FA_MAX_SEQLEN || Nk > FA_MAX_SEQLEN) return FA_ERR_INVALID_ARG;
  if (!(std::isfinite(sm_scale)) || !(sm_scale > 0.f)) return FA_ERR_INVALID_ARG;
  if (causal != 0 && causal != 1) return FA_ERR_INVALID_ARG;
  if (dtype != FA_FP16 && dtype != FA_BF16) return FA_ERR_UNSUPPORTED;
  if (d != 64 && d != 80 && d != 128) return FA_ERR_UNSUPPORTED;
  if (static_cast<int64_t>(B) * H > 0x7fffffffLL) return FA_ERR_INVALID_ARG;
  return FA_OK;
}

// Strides of a contiguous [B, H, n, d] tensor; one that overflows comes out
// negative, which valid_tensor rejects.
Tensor4 contiguous(const void* p, int H, int n, int d) {
  Tensor4 t;
  t.ptr = p;
  t.ss = d;
  t.sh = mul_nonneg(n, d);
  t.sb = mul_nonneg(mul_nonneg(H, n), d);
  return t;
}

Tensor4 strided(const void* p, const fa_strides& s) {
  Tensor4 t;
  t.ptr = p;
  t.sb = s.b;
  t.sh = s.h;
  t.ss = s.s;
  return t;
}

size_t split_ws_bytes(int B, int H, int Nq, int d, int n_splits) {
  if (n_splits < 2 || B <= 0 || H <= 0 || Nq <= 0 || d <= 0) return 0;
  size_t n = sizeof(float) * static_cast<size_t>(n_splits);
  n = mul_sat(n, static_cast<size_t>(B) * static_cast<size_t>(H));
  n = mul_sat(n, static_cast<size_t>(nq_pad(Nq)));
  return mul_sat(n, static_cast<size_t>(d) + 1);
}

fa_status fwd_impl(const Tensor4& q, const Tensor4& k, const Tensor4& v, const Tensor4& o, float* lse, int B, int H,
                   int Nq, int Nk, int d, float sm_scale, int causal, fa_dtype dtype, void* stream,
                   int n_splits = 1, void* workspace = nullptr, size_t workspace_bytes = 0) {
  if (n_splits < 1 || n_splits > FA_MAX_SPLITS) return FA_ERR_INVALID_ARG;
  fa_status st = check_common(B, H, Nq, Nk, d, sm_scale, causal, dtype);
  if (st != FA_OK) return st;
  if (B == 0 || H == 0 || Nq == 0) return FA_OK;
  if (!valid_tensor(q) || !valid_tensor(k) || !valid_tensor(v) || !valid_tensor(o)) return FA_ERR_INVALID_ARG;
  if (lse == nullptr || !aligned16(lse)) return FA_ERR_INVALID_ARG;
  if (n_splits > 1 && (workspace == nullptr || !aligned16(workspace) ||
                       workspace_bytes < split_ws_bytes(B, H, Nq, d, n_splits)))
    return FA_ERR_WORKSPACE;
  if (get_encode() == nullptr) return FA_ERR_CUDA;
  cudaError_t e;
  int* err = err_word(&e);
  if (err == nullptr) return FA_ERR_CUDA;
  FwdArgs a;
  a.q = q;
  a.k = k;
  a.v = v;
  a.o = o;
  a.lse = lse;
  a.B = B;
  a.H = H;
  a.Nq = Nq;
  a.Nk = Nk;
  a.d = d;
  a.sm_scale = sm_scale;
  a.causal = causal;
  a.bf16 = dtype == FA_BF16;
  a.err = err;
  a.n_splits = n_splits;
  a.part = static_cast<float*>(workspace);
  e = launch_fwd(a, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

fa_status fwd_fp8v_impl(const void* q, const void* k, const void* vt, void* o, float* lse, int B, int H, int Nq,
                        int Nk, int d, int64_t ld, float sm_scale, int causal, fa_dtype dtype, void* stream,
                        int mode = FA_FP8V_PAGE_STEPS) {
  fa_status st = check_common(B, H, Nq, Nk, d, sm_scale, causal, dtype);
  if (st != FA_OK) return st;
  if (mode != FA_FP8V_PAGE_STEPS && mode != FA_FP8V_LAZY_MAX) return FA_ERR_INVALID_ARG;
  if (ld < Nk || ld % 16 != 0 || ld >= (int64_t(1) << 32)) return FA_ERR_INVALID_ARG;
  if (B == 0 || H == 0 || Nq == 0) return FA_OK;
  const Tensor4 tq = contiguous(q, H, Nq, d), tk = contiguous(k, H, Nk, d), to = contiguous(o, H, Nq, d);
  if (!valid_tensor(tq) || !valid_tensor(tk) || !valid_tensor(to)) return FA_ERR_INVALID_ARG;
  if (vt == nullptr || !aligned16(vt)) return FA_ERR_INVALID_ARG;
  const int64_t vt_sb = mul_nonneg(ld * d, H);   // ld < 2^32 and d <= 128: ld * d fits
  if (vt_sb < 0 || vt_sb >= kMaxStrideBytes) return FA_ERR_INVALID_ARG;
  if (lse == nullptr || !aligned16(lse)) return FA_ERR_INVALID_ARG;
  if (get_encode() == nullptr) return FA_ERR_CUDA;
  cudaError_t e;
  int* err = err_word(&e);
  if (err == nullptr) return FA_ERR_CUDA;
  FwdArgs a;
  a.q = tq;
  a.k = tk;
  a.v.ptr = vt;
  a.v.ss = ld;
  a.v.sh = ld * d;
  a.v.sb = vt_sb;
  a.o = to;
  a.lse = lse;
  a.B = B;
  a.H = H;
  a.Nq = Nq;
  a.Nk = Nk;
  a.d = d;
  a.sm_scale = sm_scale;
  a.causal = causal;
  a.bf16 = dtype == FA_BF16;
  a.err = err;
  a.fp8v = true;
  a.vt_ld = ld;
  a.fp8_lazy = mode == FA_FP8V_LAZY_MAX;
  e = launch_fwd(a, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

// Workspace of the two-pass backward: D and log2-LSE, float32, per padded row.
size_t ws_bytes(int B, int H, int Nq) {
  if (B <= 0 || H <= 0 || Nq <= 0) return 0;
  const size_t rows = mul_sat(static_cast<size_t>(B) * static_cast<size_t>(H), static_cast<size_t>(nq_pad(Nq)));
  return mul_sat(2 * sizeof(float), rows);
}

// Workspace of the fused backward: D, log2-LSE and a float32 dQ row each.
size_t ws_bytes_fused(int B, int H, int Nq, int d) {
  if (B <= 0 || H <= 0 || Nq <= 0 || d <= 0) return 0;
  const size_t rows = mul_sat(static_cast<size_t>(B) * static_cast<size_t>(H), static_cast<size_t>(nq_pad(Nq)));
  return mul_sat(sizeof(float) * (2 + static_cast<size_t>(d)), rows);
}

// The path FA_BWD_PATH_AUTO prefers at head dim d: the fused backward
// wherever it is built (d = 64), where it was measured faster than the two
// passes on the bf16 causal B4 H20 N4096 backward (0.663 ms against 0.707).
bool fused_preferred(int d) { return bwd_fused_supported(d); }

size_t ws_bytes_path(int B, int H, int Nq, int d, fa_bwd_path path) {
  switch (path) {
    case FA_BWD_PATH_TWO_PASS: return ws_bytes(B, H, Nq);
    case FA_BWD_PATH_FUSED: return bwd_fused_supported(d) ? ws_bytes_fused(B, H, Nq, d) : 0;
    case FA_BWD_PATH_AUTO: return fused_preferred(d) ? ws_bytes_fused(B, H, Nq, d) : ws_bytes(B, H, Nq);
  }
  return 0;
}

fa_status bwd_impl(const Tensor4& q, const Tensor4& k, const Tensor4& v, const Tensor4& o, const Tensor4& dout,
                   const float* lse, const Tensor4& dq, const Tensor4& dk, const Tensor4& dv, int B, int H, int Nq,
                   int Nk, int d, float sm_scale, int causal, fa_dtype dtype, void* workspace,
                   size_t workspace_bytes, int phase, void* stream, fa_bwd_path path = FA_BWD_PATH_AUTO) {
  if (phase < 0 || phase > 3) return FA_ERR_INVALID_ARG;
  if (path != FA_BWD_PATH_AUTO && path != FA_BWD_PATH_TWO_PASS && path != FA_BWD_PATH_FUSED)
    return FA_ERR_INVALID_ARG;
  fa_status st = check_common(B, H, Nq, Nk, d, sm_scale, causal, dtype);
  if (st != FA_OK) return st;
  if (path == FA_BWD_PATH_FUSED && !bwd_fused_supported(d)) return FA_ERR_UNSUPPORTED;
  if (B == 0 || H == 0) return FA_OK;
  // AUTO takes the preferred path when the workspace holds it, else the
  // two-pass path.
  const bool fused = path == FA_BWD_PATH_FUSED ||
                     (path == FA_BWD_PATH_AUTO && fused_preferred(d) &&
                      workspace_bytes >= ws_bytes_fused(B, H, Nq, d));
  // With no queries only dK = dV = 0 is written; the query-side tensors, lse
  // and the workspace are not touched.
  if (!valid_tensor(k) || !valid_tensor(v) || !valid_tensor(dk) || !valid_tensor(dv)) return FA_ERR_INVALID_ARG;
  if (Nq > 0) {
    if (!valid_tensor(q) || !valid_tensor(o) || !valid_tensor(dout) || !valid_tensor(dq))
      return FA_ERR_INVALID_ARG;
    if (lse == nullptr || !aligned16(lse)) return FA_ERR_INVALID_ARG;
    const size_t need = fused ? ws_bytes_fused(B, H, Nq, d) : ws_bytes(B, H, Nq);
    if (workspace == nullptr || !aligned16(workspace) || workspace_bytes < need) return FA_ERR_WORKSPACE;
  }
  if (get_encode() == nullptr) return FA_ERR_CUDA;
  cudaError_t e;
  int* err = err_word(&e);
  if (err == nullptr) return FA_ERR_CUDA;
  BwdArgs a;
  a.q = q;
  a.k = k;
  a.v = v;
  a.o = o;
  a.dout = dout;
  a.dq = dq;
  a.dk = dk;
  a.dv = dv;
  a.lse = lse;
  a.ws = static_cast<float*>(workspace);
  a.B = B;
  a.H = H;
  a.Nq = Nq;
  a.Nk = Nk;
  a.d = d;
  a.sm_scale = sm_scale;
  a.causal = causal;
  a.bf16 = dtype == FA_BF16;
  a.err = err;
  a.fused = fused;
  e = launch_bwd(a, phase, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

}  // namespace

bool make_tile_map(CUtensorMap* map, const Tensor4& t, int d, int rows, int H, int B, bool bf16) {
  EncodeTiledFn enc = get_encode();
  if (enc == nullptr) return false;
  const cuuint64_t dims[4] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(rows),
                              static_cast<cuuint64_t>(H), static_cast<cuuint64_t>(B)};
  const cuuint64_t strides[3] = {static_cast<cuuint64_t>(t.ss * 2), static_cast<cuuint64_t>(t.sh * 2),
                                 static_cast<cuuint64_t>(t.sb * 2)};
  const int cc = chunk_cols(d);
  const cuuint32_t box[4] = {static_cast<cuuint32_t>(cc), static_cast<cuuint32_t>(kTileRows), 1, 1};
  const cuuint32_t estride[4] = {1, 1, 1, 1};
  CUresult r = enc(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 4,
                   const_cast<void*>(t.ptr), dims, strides, box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   cc == 64 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool make_f32_rows_map(CUtensorMap* map, const float* base, int64_t rows, int cols) {
  EncodeTiledFn enc = get_encode();
  if (enc == nullptr || rows <= 0 || cols <= 0 || (cols * 4) % 16 != 0) return false;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols) * 4};
  const cuuint32_t box[2] = {32, static_cast<cuuint32_t>(kTileRows)};
  const cuuint32_t estride[2] = {1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float*>(base), dims, strides, box, estride,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool make_vt_map(CUtensorMap* map, const void* vt, int64_t ld, int Nk, int d, int H, int B) {
  EncodeTiledFn enc = get_encode();
  if (enc == nullptr) return false;
  const cuuint64_t dims[4] = {static_cast<cuuint64_t>(Nk), static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(H),
                              static_cast<cuuint64_t>(B)};
  const cuuint64_t strides[3] = {static_cast<cuuint64_t>(ld), static_cast<cuuint64_t>(ld * d),
                                 static_cast<cuuint64_t>(ld * d * H)};
  const cuuint32_t box[4] = {static_cast<cuuint32_t>(kTileRows), static_cast<cuuint32_t>(d), 1, 1};
  const cuuint32_t estride[4] = {1, 1, 1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, const_cast<void*>(vt), dims, strides, box, estride,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

}  // namespace fa

using fa::Tensor4;

extern "C" {

fa_status fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int Nq, int Nk,
                 int d, float sm_scale, int causal, fa_dtype dtype, void* stream) {
  return fa::fwd_impl(fa::contiguous(q, H, Nq, d), fa::contiguous(k, H, Nk, d), fa::contiguous(v, H, Nk, d),
                      fa::contiguous(o, H, Nq, d), lse, B, H, Nq, Nk, d, sm_scale, causal, dtype, stream);
}

fa_status fa_fwd_fp8v(const void* q, const void* k, const void* vt, void* o, float* lse, int B, int H, int Nq,
                      int Nk, int d, int64_t vt_ld, float sm_scale, int causal, fa_dtype dtype, void* stream) {
  return fa::fwd_fp8v_impl(q, k, vt, o, lse, B, H, Nq, Nk, d, vt_ld, sm_scale, causal, dtype, stream);
}

fa_status fa_fwd_fp8v_ex(const void* q, const void* k, const void* vt, void* o, float* lse, int B, int H, int Nq,
                         int Nk, int d, int64_t vt_ld, float sm_scale, int causal, fa_dtype dtype, int mode,
                         void* stream) {
  return fa::fwd_fp8v_impl(q, k, vt, o, lse, B, H, Nq, Nk, d, vt_ld, sm_scale, causal, dtype, stream, mode);
}

fa_status fa_fwd_strided(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int Nq,
                         int Nk, int d, float sm_scale, int causal, fa_dtype dtype, const fa_layout* layout,
                         void* stream) {
  if (layout == nullptr) return FA_ERR_INVALID_ARG;
  return fa::fwd_impl(fa::strided(q, layout->q), fa::strided(k, layout->k), fa::strided(v, layout->v),
                      fa::strided(o, layout->o), lse, B, H, Nq, Nk, d, sm_scale, causal, dtype, stream);
}

size_t fa_fwd_split_workspace_bytes(int B, int H, int Nq, int d, int n_splits) {
  return fa::split_ws_bytes(B, H, Nq, d, n_splits);
}

int fa_fwd_split_count(int B, int H, int Nq, int Nk, int d, int causal) {
  (void)d;
  (void)causal;
  if (B <= 0 || H <= 0 || Nq <= 0 || Nk <= 0) return 1;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
      sms <= 0)
    return 1;
  // Every CTA pays a fixed start-up and drain time of a few key tiles' work,
  // so a split only pays while the split grid still runs in one wave and
  // every split keeps at least kMinTilesPerSplit key tiles.  Under one wave
  // the forward runs one 128-row query tile per CTA, so the unsplit grid to
  // beat is that one.
  constexpr long long kMinTilesPerSplit = 4;
  const long long ctas = static_cast<long long>((Nq + 127) / 128) * B * H;   // one query tile per CTA
  const long long n_kt = (Nk + 127) / 128;
  long long s = sms / ctas;
  if (s > n_kt / kMinTilesPerSplit) s = n_kt / kMinTilesPerSplit;
  if (s > FA_MAX_SPLITS) s = FA_MAX_SPLITS;
  return s < 1 ? 1 : static_cast<int>(s);
}

fa_status fa_fwd_split(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int Nq,
                       int Nk, int d, float sm_scale, int causal, fa_dtype dtype, const fa_layout* layout,
                       int n_splits, void* workspace, size_t workspace_bytes, void* stream) {
  if (layout == nullptr)
    return fa::fwd_impl(fa::contiguous(q, H, Nq, d), fa::contiguous(k, H, Nk, d), fa::contiguous(v, H, Nk, d),
                        fa::contiguous(o, H, Nq, d), lse, B, H, Nq, Nk, d, sm_scale, causal, dtype, stream, n_splits,
                        workspace, workspace_bytes);
  return fa::fwd_impl(fa::strided(q, layout->q), fa::strided(k, layout->k), fa::strided(v, layout->v),
                      fa::strided(o, layout->o), lse, B, H, Nq, Nk, d, sm_scale, causal, dtype, stream, n_splits,
                      workspace, workspace_bytes);
}

size_t fa_bwd_workspace_bytes(int B, int H, int Nq, int Nk, int d) {
  (void)Nk;
  return fa::ws_bytes_path(B, H, Nq, d, FA_BWD_PATH_AUTO);
}

size_t fa_bwd_workspace_bytes_path(int B, int H, int Nq, int Nk, int d, fa_bwd_path path) {
  (void)Nk;
  return fa::ws_bytes_path(B, H, Nq, d, path);
}

fa_status fa_bwd(const void* q, const void* k, const void* v, const void* o, const void* dout, const float* lse,
                 void* dq, void* dk, void* dv, int B, int H, int Nq, int Nk, int d, float sm_scale, int causal,
                 fa_dtype dtype, void* workspace, size_t workspace_bytes, void* stream) {
  return fa::bwd_impl(fa::contiguous(q, H, Nq, d), fa::contiguous(k, H, Nk, d), fa::contiguous(v, H, Nk, d),
                      fa::contiguous(o, H, Nq, d), fa::contiguous(dout, H, Nq, d), lse,
                      fa::contiguous(dq, H, Nq, d), fa::contiguous(dk, H, Nk, d), fa::contiguous(dv, H, Nk, d), B,
                      H, Nq, Nk, d, sm_scale, causal, dtype, workspace, workspace_bytes, 0, stream);
}

fa_status fa_bwd_strided(const void* q, const void* k, const void* v, const void* o, const void* dout,
                         const float* lse, void* dq, void* dk, void* dv, int B, int H, int Nq, int Nk, int d,
                         float sm_scale, int causal, fa_dtype dtype, const fa_layout* layout, void* workspace,
                         size_t workspace_bytes, void* stream) {
  if (layout == nullptr) return FA_ERR_INVALID_ARG;
  return fa::bwd_impl(fa::strided(q, layout->q), fa::strided(k, layout->k), fa::strided(v, layout->v),
                      fa::strided(o, layout->o), fa::strided(dout, layout->dout), lse,
                      fa::strided(dq, layout->dq), fa::strided(dk, layout->dk), fa::strided(dv, layout->dv), B, H,
                      Nq, Nk, d, sm_scale, causal, dtype, workspace, workspace_bytes, 0, stream);
}

fa_status fa_bwd_phase(int phase, const void* q, const void* k, const void* v, const void* o, const void* dout,
                       const float* lse, void* dq, void* dk, void* dv, int B, int H, int Nq, int Nk, int d,
                       float sm_scale, int causal, fa_dtype dtype, const fa_layout* layout, void* workspace,
                       size_t workspace_bytes, void* stream) {
  if (phase < 1 || phase > 3) return FA_ERR_INVALID_ARG;
  if (layout == nullptr)
    return fa::bwd_impl(fa::contiguous(q, H, Nq, d), fa::contiguous(k, H, Nk, d), fa::contiguous(v, H, Nk, d),
                        fa::contiguous(o, H, Nq, d), fa::contiguous(dout, H, Nq, d), lse,
                        fa::contiguous(dq, H, Nq, d), fa::contiguous(dk, H, Nk, d), fa::contiguous(dv, H, Nk, d),
                        B, H, Nq, Nk, d, sm_scale, causal, dtype, workspace, workspace_bytes, phase, stream);
  return fa::bwd_impl(fa::strided(q, layout->q), fa::strided(k, layout->k), fa::strided(v, layout->v),
                      fa::strided(o, layout->o), fa::strided(dout, layout->dout), lse,
                      fa::strided(dq, layout->dq), fa::strided(dk, layout->dk), fa::strided(dv, layout->dv), B, H,
                      Nq, Nk, d, sm_scale, causal, dtype, workspace, workspace_bytes, phase, stream);
}

fa_status fa_bwd_ex(fa_bwd_path path, int phase, const void* q, const void* k, const void* v, const void* o,
                    const void* dout, const float* lse, void* dq, void* dk, void* dv, int B, int H, int Nq, int Nk,
                    int d, float sm_scale, int causal, fa_dtype dtype, const fa_layout* layout, void* workspace,
                    size_t workspace_bytes, void* stream) {
  if (phase < 0 || phase > 3) return FA_ERR_INVALID_ARG;
  if (layout == nullptr)
    return fa::bwd_impl(fa::contiguous(q, H, Nq, d), fa::contiguous(k, H, Nk, d), fa::contiguous(v, H, Nk, d),
                        fa::contiguous(o, H, Nq, d), fa::contiguous(dout, H, Nq, d), lse,
                        fa::contiguous(dq, H, Nq, d), fa::contiguous(dk, H, Nk, d), fa::contiguous(dv, H, Nk, d),
                        B, H, Nq, Nk, d, sm_scale, causal, dtype, workspace, workspace_bytes, phase, stream, path);
  return fa::bwd_impl(fa::strided(q, layout->q), fa::strided(k, layout->k), fa::strided(v, layout->v),
                      fa::strided(o, layout->o), fa::strided(dout, layout->dout), lse,
                      fa::strided(dq, layout->dq), fa::strided(dk, layout->dk), fa::strided(dv, layout->dv), B, H,
                      Nq, Nk, d, sm_scale, causal, dtype, workspace, workspace_bytes, phase, stream, path);
}

const char* fa_status_string(fa_status s) {
  switch (s) {
    case FA_OK: return "FA_OK";
    case FA_ERR_INVALID_ARG: return "FA_ERR_INVALID_ARG: bad pointer, size, stride, alignment or scale";
    case FA_ERR_UNSUPPORTED: return "FA_ERR_UNSUPPORTED: head dim or dtype not supported";
    case FA_ERR_CUDA: return "FA_ERR_CUDA: a CUDA call failed";
    case FA_ERR_TIMEOUT: return "FA_ERR_TIMEOUT: a bounded device-side wait ran out";
    case FA_ERR_WORKSPACE: return "FA_ERR_WORKSPACE: backward workspace missing or too small";
  }
  return "unknown fa_status";
}

fa_status fa_last_device_error(void* stream, int* detail) {
  if (detail) *detail = 0;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return FA_ERR_CUDA;
  int v = 0;
  if (cudaMemcpyFromSymbol(&v, fa::g_err_word, sizeof(int)) != cudaSuccess) return FA_ERR_CUDA;
  if (v != 0) {
    const int zero = 0;
    if (cudaMemcpyToSymbol(fa::g_err_word, &zero, sizeof(int)) != cudaSuccess) return FA_ERR_CUDA;
  }
  if (detail) *detail = v;
  return v != 0 ? FA_ERR_TIMEOUT : FA_OK;
}

fa_status fa_inject_device_error(int code) {
  if (code == 0) return FA_ERR_INVALID_ARG;
  if (cudaMemcpyToSymbol(fa::g_err_word, &code, sizeof(int)) != cudaSuccess) return FA_ERR_CUDA;
  return FA_OK;
}

const char* fa_version(void) { return "0.1.0"; }

}  // extern "C"
