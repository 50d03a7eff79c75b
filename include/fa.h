/*
 * fa.h -- C ABI of the GB300 (sm_103a) FlashAttention-2 library (libfa.so).
 *
 * Exact attention, forward and recompute-based backward:
 *
 *   S = sm_scale * Q K^T  [+ causal mask],  P = softmax_row(S),  O = P V,
 *   LSE_i = log sum_j exp(S_ij),
 *   dV = P^T dO,  dP = dO V^T,  D = rowsum(O o dO),  dS = P o (dP - D),
 *   dQ = sm_scale dS K,  dK = sm_scale dS^T Q.
 *
 * Sources: "[CS336] Assignment 2: Systems", section "FlashAttention V2"
 * (High level: the forward and backward equations, the logsumexp L and the
 * precomputed D; Forward Pass: the online running max / running sum over key
 * tiles; Backward Pass: the two accumulation directions).  "Understanding
 * Triton Tutorials Part 2", section "Fused Attention 2" (exp2 with sm_scale
 * folded by log2(e), causal block skipping, the [Z, H, N_CTX, HEAD_DIM]
 * layout).  "BUG in flash attention kernel" (triton issue 2626): the
 * [seq, heads, d] layout with Nq != Nk, and per-tensor strides.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - All tensor pointers are DEVICE pointers owned by the caller.  The library
 *   never allocates or frees device memory.  It keeps two statically sized
 *   device arrays in every GPU that loads it: one 4-byte error word, and the
 *   16 MiB scratch array that only fa_bwd_noalloc uses (below).  Outputs are
 *   fully overwritten (no accumulate-into semantics), so they need no zeroing.
 * - The device addresses of those arrays are looked up once per device, on
 *   the first call that needs them, and kept for the life of the process:
 *   resetting a device (cudaDeviceReset) after that first call is not
 *   supported.
 * - Element type: FA_FP16 or FA_BF16 for Q, K, V, O, dO, dQ, dK, dV; the
 *   log-sum-exp is always float32.  Arithmetic is fp32 accumulation on the
 *   tensor cores, P and dS are rounded to the input type before their GEMMs.
 * - Layout: each Q/K/V/O-like tensor is addressed as x[b, h, s, 0..d-1] at
 *   element offset b*stride_b + h*stride_h + s*stride_s, with the head
 *   dimension contiguous (stride 1).  fa_fwd / fa_bwd assume contiguous
 *   [B, H, seq, d]; the *_strided variants take explicit strides (e.g.
 *   [seq, heads, d] is B = 1, stride_h = d, stride_s = H*d).
 * - lse (and the backward's lse input) is float32 [B, H, Nq] contiguous, the
 *   natural log of sum_j exp(sm_scale * q_i . k_j) over the visible keys.
 * - Causal masking is top-left aligned: key j is visible to query i iff
 *   j <= i, also when Nq != Nk.
 * - Requirements (checked before any launch): B, H, Nq >= 0; Nk >= 1;
 *   Nq, Nk <= FA_MAX_SEQLEN; B*H < 2^31; d in {64, 80, 128}; pointers
 *   non-null and 16-byte aligned; strides positive, in bytes multiples of 16
 *   and below 2^40 (the TMA limit); sm_scale finite and > 0.  B*H == 0 or
 *   Nq == 0 is a no-op returning FA_OK.  Other d give FA_ERR_UNSUPPORTED.
 * - Calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy
 *   default stream) and never synchronise.  The return value reports
 *   argument errors (nothing launched) and launch errors (FA_ERR_CUDA).
 * - Every device-side wait is bounded.  A wait that runs out records a code in
 *   the per-device error word and the kernel finishes without hanging;
 *   fa_last_device_error() reports it.
 * - Thread safety: entry points may be called from several host threads.
 */
#ifndef TILED_ATTENTION_07_GB300_FA_H
#define TILED_ATTENTION_07_GB300_FA_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define FA_API __attribute__((visibility("default")))
#else
#define FA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    FA_OK = 0,
    FA_ERR_INVALID_ARG = 1,   /* bad pointer, size, stride, alignment or scale */
    FA_ERR_UNSUPPORTED = 2,   /* valid but not implemented (head dim, dtype)   */
    FA_ERR_CUDA = 3,          /* a CUDA runtime/driver call failed             */
    FA_ERR_TIMEOUT = 4,       /* a bounded device-side wait ran out            */
    FA_ERR_WORKSPACE = 5      /* backward workspace missing or too small       */
} fa_status;

/* Element types.  The attention entry points take FA_FP16 and FA_BF16 (other
 * values give FA_ERR_UNSUPPORTED); fa_softmax_rows also takes FA_FP32. */
typedef enum { FA_FP16 = 0, FA_BF16 = 1, FA_FP32 = 2 } fa_dtype;

/* Longest Nq or Nk the attention entry points take (2^30).  A longer
 * sequence does not fit the device's memory at any supported head dim, and
 * the bound keeps every row index and tile count in int arithmetic. */
#define FA_MAX_SEQLEN (1 << 30)

/* Element strides of one [B, H, seq, d] tensor; the d stride is always 1. */
typedef struct {
    int64_t b, h, s;
} fa_strides;

/* Strides of every tensor an entry point touches; entries it does not use are
 * ignored. */
typedef struct {
    fa_strides q, k, v, o, dout, dq, dk, dv;
} fa_layout;

/*
 * fa_fwd -- FlashAttention-2 forward ("[CS336]", "FlashAttention V2 /
 * Forward Pass"; "Fused Attention 2", _attn_fwd).
 *   q   [B, H, Nq, d]   in          k, v [B, H, Nk, d]  in
 *   o   [B, H, Nq, d]   out         lse  [B, H, Nq] float32 out
 *   sm_scale: multiplies q.k before the softmax; causal: 0 or 1.
 * Returns FA_OK or an error code (see the conventions above).
 */
FA_API fa_status fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
                 int B, int H, int Nq, int Nk, int d, float sm_scale, int causal,
                 fa_dtype dtype, void* stream);

/* fa_fwd with explicit strides for q, k, v and o (layout->q, ->k, ->v, ->o);
 * e.g. the [seq, heads, d] layout of "BUG in flash attention kernel"
 * (B = 1, stride_h = d, stride_s = heads*d).  lse stays [B, H, Nq]. */
FA_API fa_status fa_fwd_strided(const void* q, const void* k, const void* v, void* o, float* lse,
                         int B, int H, int Nq, int Nk, int d, float sm_scale, int causal,
                         fa_dtype dtype, const fa_layout* layout, void* stream);

/*
 * Split-KV forward: the key tiles of every query tile are divided into
 * n_splits contiguous ranges handled by different CTAs, so that problems with
 * few query tiles still fill the GPU.  Split s covers key tiles
 * [s*T, min((s+1)*T, nk)) with nk = ceil(Nk/128), T = ceil(nk/n_splits).
 * Each split writes, per query row, its own softmax over its keys: O_s (the
 * partial output already divided by its own row sum) and lse_s (its own
 * log-sum-exp; -inf and O_s = 0 when the row sees none of its keys).  A merge
 * kernel then combines them with the rescaling of the online softmax
 * ("[CS336]", "FlashAttention V2 / Forward Pass": m' = max, l' = e^(m-m') l
 * + ...; "Puzzles 8 Long Softmax": sum' = sum * exp(m1 - m2) + ...):
 *     lse = log sum_s exp(lse_s),   O = sum_s exp(lse_s - lse) O_s,
 * which equals the one-pass result up to rounding.
 *
 * fa_fwd_split_workspace_bytes -- scratch for the partial results: float32
 * O_s and lse_s of every split, query rows padded to whole 128-row tiles:
 * 4 * n_splits * B*H*ceil(Nq/128)*128 * (d + 1) bytes.  0 for n_splits < 2.
 */
FA_API size_t fa_fwd_split_workspace_bytes(int B, int H, int Nq, int d, int n_splits);

/*
 * fa_fwd_split_count -- a split count for this problem on the current device:
 * the most splits for which the split grid still fits in one wave (one CTA
 * per 128-row query tile and split, one CTA per SM) while every split keeps
 * at least 4 of the 128-key tiles, capped at FA_MAX_SPLITS; 1 when the
 * unsplit grid already fills the SMs.  (Each CTA
 * has a fixed start-up and drain cost of a few key tiles' work, so more
 * splits than that are slower.)  Returns 1 for invalid or empty problems.
 */
#define FA_MAX_SPLITS 64
FA_API int fa_fwd_split_count(int B, int H, int Nq, int Nk, int d, int causal);

/*
 * fa_fwd_split -- fa_fwd / fa_fwd_strided over n_splits key ranges (1 <=
 * n_splits <= FA_MAX_SPLITS).  layout: strides of q, k, v, o, or NULL for
 * contiguous [B, H, seq, d].  n_splits == 1 runs the one-pass forward and
 * needs no workspace; otherwise workspace (device, 16-byte aligned, owned by
 * the caller, contents on entry ignored) must hold
 * fa_fwd_split_workspace_bytes(B, H, Nq, d, n_splits) bytes, else
 * FA_ERR_WORKSPACE.  Two launches on `stream`: the partial forward, and the
 * merge as its programmatic dependent (its blocks start as the forward's
 * finish and wait for the forward's results).
 */
FA_API fa_status fa_fwd_split(const void* q, const void* k, const void* v, void* o, float* lse,
                       int B, int H, int Nq, int Nk, int d, float sm_scale, int causal,
                       fa_dtype dtype, const fa_layout* layout, int n_splits, void* workspace,
                       size_t workspace_bytes, void* stream);

/*
 * fa_fwd_fp8v -- the forward with V in float8 e5m2 ("Understanding Triton
 * Tutorials Part 2", "Fused Attention 2": when V is float8_e5m2 it is stored
 * transposed, and the probabilities of each key block are cast to float8 e5m2
 * before the product with V; the row sum l takes the unrounded p).
 *   q   [B, H, Nq, d]  in  (dtype)       k  [B, H, Nk, d]  in  (dtype)
 *   vt  [B, H, d, vt_ld] e5m2 codes (one byte each), in: key j of head
 *       dimension c of head (b, h) at byte ((b*H + h)*d + c)*vt_ld + j;
 *       vt_ld >= Nk, vt_ld % 16 == 0, vt 16-byte aligned; bytes j >= Nk of a
 *       row are not read.
 *   o   [B, H, Nq, d]  out (dtype)       lse [B, H, Nq] float32 out
 * q, k and o are contiguous; dtype (FA_FP16 or FA_BF16) is theirs.  S = q k^T
 * runs on the 16-bit tensor-core path; P is rounded to e5m2 (to nearest
 * even, saturating) and O += P V runs on the 8-bit path (kind::f8f6f4) with
 * float32 accumulation.  p is taken, per block of 128 keys, against the
 * running max of the blocks so far, moved at every block as in the page's
 * steps (O is rescaled in tensor memory whenever a row's max grows), so the
 * kernel casts the same p as those steps; the float32 arithmetic that forms
 * p can only move an element lying within about 1e-6 of an e5m2 rounding
 * midpoint to the other side.  LSE is exact, as in fa_fwd; O differs from
 * the exact result by at most about 2^-3 * max |v| over the row's keys (the
 * rounding of P, relative 2^-3) plus the 16-bit rounding of O.
 * d in {64, 80, 128} (at d = 128 the 8-bit P is written over the first 32
 * columns of its tile's S in tensor memory, as the 16-bit P is there).
 * Errors as fa_fwd; vt_ld out of range gives FA_ERR_INVALID_ARG.  One launch
 * on `stream`.
 */
FA_API fa_status fa_fwd_fp8v(const void* q, const void* k, const void* vt, void* o, float* lse,
                      int B, int H, int Nq, int Nk, int d, int64_t vt_ld, float sm_scale,
                      int causal, fa_dtype dtype, void* stream);

/*
 * fa_fwd_fp8v_ex -- fa_fwd_fp8v with a choice of running-max rule:
 *   FA_FP8V_PAGE_STEPS (0): as fa_fwd_fp8v (the page's steps).
 *   FA_FP8V_LAZY_MAX (1): the running max moves only when a row's max grows
 *     by more than 2^8 (in log2 units), as in the 16-bit forward, so O is
 *     rarely rescaled.  This departs from the page's steps: p is taken at a
 *     scale up to 2^8 larger than theirs and its e5m2 rounding can differ by
 *     one step, so O differs from theirs by up to about 2^-2 * max |v| over
 *     the row's keys (and from the exact result by the same 2^-3 bound as
 *     above).  Faster: the per-block rescale of O costs the page's rule
 *     about 20 % of the forward on causal shapes.
 * Other values of mode give FA_ERR_INVALID_ARG.
 */
enum { FA_FP8V_PAGE_STEPS = 0, FA_FP8V_LAZY_MAX = 1 };
FA_API fa_status fa_fwd_fp8v_ex(const void* q, const void* k, const void* vt, void* o, float* lse,
                         int B, int H, int Nq, int Nk, int d, int64_t vt_ld, float sm_scale,
                         int causal, fa_dtype dtype, int mode, void* stream);

/*
 * fa_bwd_workspace_bytes -- size of the scratch buffer fa_bwd needs: the
 * per-row D = rowsum(O o dO) and the log2-domain LSE, float32, padded to
 * whole 128-row query tiles: 2 * 4 * B*H*ceil(Nq/128)*128 bytes, plus a
 * float32 dQ accumulator row per query where the fused path is the faster
 * one (see fa_bwd_path below).  ("[CS336]", "FlashAttention V2 / Backward
 * Pass": D is computed once, before the passes, and kept in global memory.)
 */
FA_API size_t fa_bwd_workspace_bytes(int B, int H, int Nq, int Nk, int d);

/*
 * fa_bwd -- recompute-based backward ("[CS336]", "FlashAttention V2 /
 * Backward Pass": P_ij = exp(S_ij - L_i), dS = P o (dP - D), the two passes
 * over K tiles (dQ) and Q tiles (dK, dV)).
 *   q, k, v, o, dout: as produced/consumed by fa_fwd (o is fa_fwd's output)
 *   lse: float32 [B, H, Nq] from fa_fwd
 *   dq [B, H, Nq, d], dk, dv [B, H, Nk, d]: out, input dtype
 *   workspace: device buffer of at least fa_bwd_workspace_bytes() bytes,
 *   16-byte aligned, owned by the caller; its contents on entry are ignored.
 *   (A workspace of only the two-pass size selects the two-pass path.)
 * Returns FA_ERR_WORKSPACE if the workspace is NULL or too small.
 */
FA_API fa_status fa_bwd(const void* q, const void* k, const void* v, const void* o, const void* dout,
                 const float* lse, void* dq, void* dk, void* dv,
                 int B, int H, int Nq, int Nk, int d, float sm_scale, int causal,
                 fa_dtype dtype, void* workspace, size_t workspace_bytes, void* stream);

/* fa_bwd with explicit strides (layout->q, k, v, o, dout, dq, dk, dv), e.g.
 * the [seq, heads, d] layout of "BUG in flash attention kernel".  Every
 * tensor is addressed with its own strides: the kernel in that issue offset
 * K and V by Q's head stride, which is wrong once Nq != Nk. */
FA_API fa_status fa_bwd_strided(const void* q, const void* k, const void* v, const void* o, const void* dout,
                         const float* lse, void* dq, void* dk, void* dv,
                         int B, int H, int Nq, int Nk, int d, float sm_scale, int causal,
                         fa_dtype dtype, const fa_layout* layout,
                         void* workspace, size_t workspace_bytes, void* stream);

/*
 * fa_bwd_phase -- one of the three launches fa_bwd makes, for callers that
 * schedule or time them separately ("[CS336]", "FlashAttention V2 / Backward
 * Pass": D precomputed in global memory before the backward, then the dQ pass
 * over key tiles and the dK/dV pass over query tiles):
 *   phase FA_BWD_PREPROCESS (1): D = rowsum(O o dO) and LSE*log2(e) into the
 *                                workspace (reads o, dout, lse)
 *   phase FA_BWD_DKDV (2):       dk, dv (reads q, k, v, dout, workspace)
 *   phase FA_BWD_DQ (3):         dq (reads q, k, v, dout, workspace)
 * Calling phases 1, 2, 3 in order on one stream, with the same workspace, is
 * exactly fa_bwd.  layout == NULL means contiguous [B, H, seq, d] tensors.
 * Other arguments, requirements and errors as fa_bwd / fa_bwd_strided; an
 * unknown phase gives FA_ERR_INVALID_ARG.
 */
enum { FA_BWD_PREPROCESS = 1, FA_BWD_DKDV = 2, FA_BWD_DQ = 3 };
FA_API fa_status fa_bwd_phase(int phase, const void* q, const void* k, const void* v, const void* o,
                       const void* dout, const float* lse, void* dq, void* dk, void* dv,
                       int B, int H, int Nq, int Nk, int d, float sm_scale, int causal,
                       fa_dtype dtype, const fa_layout* layout,
                       void* workspace, size_t workspace_bytes, void* stream);

/*
 * Backward paths.
 *   FA_BWD_PATH_TWO_PASS: the scheme of "[CS336]", "FlashAttention V2 /
 *     Backward Pass": dK and dV accumulate along query tiles and dQ along key
 *     tiles, so one pass over query tiles forms dK, dV and one over key tiles
 *     forms dQ, each recomputing P (seven products per tile pair).  Every
 *     output is bitwise reproducible.  Any d.
 *   FA_BWD_PATH_FUSED (d = 64 only): one pass over key tiles.  Besides dK and
 *     dV it forms each query tile's share of dQ and adds it into a float32
 *     accumulator in the workspace (reductions performed in L2), then a
 *     short launch converts the accumulator to dQ.  That is the five products
 *     of the recompute equations.  The order of the float32 additions into dQ
 *     varies from run to run, so dQ (not dK, dV) may differ in the last bits
 *     between runs.
 *   FA_BWD_PATH_AUTO: the path measured faster at this head dim, when the
 *     workspace holds it; otherwise the two-pass path.  This is what fa_bwd,
 *     fa_bwd_strided and fa_bwd_phase do, and fa_bwd_workspace_bytes gives
 *     the size of the path AUTO prefers.
 */
typedef enum { FA_BWD_PATH_AUTO = 0, FA_BWD_PATH_TWO_PASS = 1, FA_BWD_PATH_FUSED = 2 } fa_bwd_path;

/*
 * fa_bwd_workspace_bytes_path -- workspace bytes of one path: two-pass
 * 2 * 4 * B*H*ceil(Nq/128)*128 (D and the log2-domain LSE); fused
 * (2 + d) * 4 * B*H*ceil(Nq/128)*128 (the same, then a float32 dQ row per
 * query); AUTO as fa_bwd_workspace_bytes.  0 for the fused path at a head dim
 * it does not support, and for empty problems.
 */
FA_API size_t fa_bwd_workspace_bytes_path(int B, int H, int Nq, int Nk, int d, fa_bwd_path path);

/*
 * fa_bwd_ex -- the backward on a chosen path, whole (phase 0) or one launch
 * at a time (phases 1-3 as fa_bwd_phase: on the fused path 1 also zeroes the
 * dQ accumulator, 2 forms dK, dV and adds dQ's partial sums into the
 * accumulator, 3 writes dQ from it).  layout == NULL means contiguous
 * [B, H, seq, d].  The workspace must hold fa_bwd_workspace_bytes_path() of
 * the path taken, else FA_ERR_WORKSPACE.  FA_BWD_PATH_FUSED at a head dim
 * other than 64 gives FA_ERR_UNSUPPORTED; an unknown path or phase
 * FA_ERR_INVALID_ARG.  Other arguments and errors as fa_bwd_strided.
 */
FA_API fa_status fa_bwd_ex(fa_bwd_path path, int phase, const void* q, const void* k, const void* v,
                    const void* o, const void* dout, const float* lse, void* dq, void* dk, void* dv,
                    int B, int H, int Nq, int Nk, int d, float sm_scale, int causal,
                    fa_dtype dtype, const fa_layout* layout,
                    void* workspace, size_t workspace_bytes, void* stream);

/*
 * fa_bwd_noalloc -- fa_bwd for callers that cannot allocate device memory.
 * The pages have no counterpart to it.  It serves callers that are handed
 * only their input and output buffers and may not allocate on their own, for
 * example plugins inside an inference engine that plans every buffer in
 * advance, or code that must not call cudaMalloc while it submits work.
 * Instead of a caller workspace it uses a fixed scratch array of
 * FA_NOALLOC_SCRATCH_BYTES that the library keeps in every GPU that loads
 * it, until the process exits.
 *   Arguments: as fa_bwd (contiguous [B, H, seq, d]), without the workspace.
 *   Path: always the two-pass backward (its scratch needs 8 bytes per row).
 *   Limit: B*H*ceil(Nq/128)*128 <= FA_NOALLOC_SCRATCH_BYTES / 8 query rows
 *   (2,097,152; e.g. B=4, H=32, Nq=16384).  Larger problems return
 *   FA_ERR_WORKSPACE before anything is launched.
 *   Allocation: none (no cudaMalloc, cudaFree or allocating library call).
 *   Set-up: the first call on a device looks up the scratch array's device
 *   address (cudaGetSymbolAddress) with that device current; make that first
 *   call before any stream capture.
 *   Sharing: every call on a device uses the same scratch array, which keeps
 *   the previous call's contents (each call's first launch overwrites every
 *   entry its later launches read, so nothing needs clearing).  Calls whose
 *   work can overlap on the GPU (other streams, or host threads without
 *   ordering between them) race on the array: serialise them.
 */
#define FA_NOALLOC_SCRATCH_BYTES (16u << 20)
FA_API fa_status fa_bwd_noalloc(const void* q, const void* k, const void* v, const void* o,
                         const void* dout, const float* lse, void* dq, void* dk, void* dv,
                         int B, int H, int Nq, int Nk, int d, float sm_scale, int causal,
                         fa_dtype dtype, void* stream);

/*
 * fa_softmax_rows -- row-wise softmax of a [rows, T] matrix with the online
 * max/sum recurrence ("Puzzles 8 Long Softmax": z_ij = softmax_j(x_i1..x_iT),
 * stabilised by the row max; the max and sum loops merged by rescaling the
 * running sum, sum' = sum * exp(m_old - m_new) + ..., exp taken as exp2 of
 * log2(e) x).
 *   x    [rows, T] in, row r at element offset r * x_row_stride
 *   z    [rows, T] out (same dtype as x), row r at r * z_row_stride
 *   lse  float32 [rows] out, natural log of sum_j exp(x_rj), or NULL
 *   dtype: FA_FP32, FA_FP16 or FA_BF16; arithmetic is float32 (exp2 of
 *          the hardware approximation), z is rounded to dtype.
 * Every x_rj takes part (nothing is padded into the sum, also when T is not
 * a multiple of any tile).  A row of -inf gives NaN, like the definition.
 * Requirements: rows >= 0, T >= 1; x, z non-null and 16-byte aligned; row
 * strides >= T, in bytes multiples of 16; z must not overlap x unless
 * z == x with equal strides (in place).  rows == 0 is a no-op.
 * A row is split over a cluster of up to 16 CTAs (8 where the GPU cannot
 * schedule 16) of at most 192 KB each: rows of up to 3 MB (1.5 MB) are held
 * on chip, one read and one write of every element; longer rows are read
 * twice.  Asynchronous on `stream`.
 */
FA_API fa_status fa_softmax_rows(const void* x, void* z, float* lse, int rows, int T, int64_t x_row_stride,
                          int64_t z_row_stride, fa_dtype dtype, void* stream);

/* Human-readable name of a status code (static string, never NULL); codes
 * outside fa_status give "unknown fa_status".  Library plumbing: the pages
 * have no counterpart. */
FA_API const char* fa_status_string(fa_status status);

/*
 * fa_last_device_error -- (library plumbing; the pages have no counterpart)
 * synchronises `stream`, then reads and clears the
 * current device's error word.  Returns FA_ERR_TIMEOUT if a kernel gave up a
 * bounded wait since the last call, FA_ERR_CUDA if the synchronisation
 * failed, else FA_OK.  *detail (if non-NULL) receives the raw device code
 * (which wait gave up), 0 if none.
 */
FA_API fa_status fa_last_device_error(void* stream, int* detail);

/*
 * fa_inject_device_error -- test hook for failure handling.  Writes `code`
 * (non-zero) into the current device's error word, as if a kernel's bounded
 * wait had given up.  Kernels launched afterwards see the word set and make
 * every wait give up at once: they finish quickly with undefined output
 * values (never touching memory outside their arguments), and the next
 * fa_last_device_error() reports FA_ERR_TIMEOUT with `code` as detail and
 * clears the word.  Nothing faults or hangs on the device.  Returns
 * FA_ERR_INVALID_ARG for code == 0, FA_ERR_CUDA if the write fails.
 */
FA_API fa_status fa_inject_device_error(int code);

/* Library version string, e.g. "0.1.0". */
FA_API const char* fa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* TILED_ATTENTION_07_GB300_FA_H */
