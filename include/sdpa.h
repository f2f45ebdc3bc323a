/*
 * sdpa.h — C ABI of the GB300 fused scaled-dot-product attention library
 * (libsdpa.so, sm_103a only).
 *
 * What is computed is the equation block that opens CK tile's
 * fmha_bwd_kernel.hpp (page "Composable Kernel: fmha_bwd_kernel.hpp Source
 * File", header comment):
 *     S = Q K^T,  S' = S * scale,  S'' = S' + Bias,  P = softmax(S''),  O = P V
 *     dV = P^T dO,  dP = dO V^T,  D = rowsum(dO * O),  dS = P * (dP - D),
 *     dBias = dS,  dK = dS^T Q * scale,  dQ = dS K * scale
 * with the parameter set of PyTorch's cuDNN attention glue
 * (page "aten/src/ATen/native/cudnn/MHA.cpp", run_cudnn_SDP_fprop and
 * run_cudnn_SDP_bprop): b, h, s_q, s_kv, d_qk, d_v, a scale passed by value,
 * a causal flag, a dropout probability with seed and offset, an optional
 * bias, and an fp32 per-row softmax statistic of shape [b, h, s_q].
 *
 * Conventions shared by every entry point
 *   Layout      Contiguous BHSD: Q [b,h,s_q,d_qk], K [b,h,s_kv,d_qk],
 *               V [b,h,s_kv,d_v], O and dO [b,h,s_q,d_v], LSE [b,h,s_q] fp32,
 *               Bias and dBias [1,h,s_q,s_kv] fp32 (one bias shared by the
 *               batch; dBias is the sum over the batch of dS).
 *   Types       Q, K, V, O, dO, dQ, dK, dV are bf16 or fp16 (dtype argument);
 *               accumulation and softmax are fp32.
 *   Head sizes  (d_qk, d_v) in {(64,64), (128,128), (192,128)}.
 *   Scale       Any float whose product with log2(e) is finite, of either
 *               sign or zero; a NaN or infinite one is SDPA_ERR_INVALID_ARG.
 *   Causal      Top-left: key j is visible to query i iff j <= i.
 *   LSE         Natural-log logsumexp of the scaled, biased, masked scores
 *               before dropout; -inf for a row that sees no key (its O row
 *               is 0 and it adds nothing to any gradient).
 *   Dropout     p in [0, 1); p == 0 disables it and seed/offset are ignored.
 *               Element (b,h,i,j) has linear index L = ((b*h_n+h)*s_q+i)*s_kv+j;
 *               its 32-bit draw r is word L%4 of Philox4x32-10 with key
 *               (lo32 seed, hi32 seed) and counter (lo32 offset, hi32 offset,
 *               lo32 L/4, hi32 L/4); it is kept iff r >= floor(p * 2^32), and
 *               kept values of P are scaled by 1/(1-p). Needs s_kv % 4 == 0.
 *   Pointers    Device pointers, 16-byte aligned, owned by the caller; the
 *               library never allocates, frees or retains them.
 *   Streams     `stream` is a cudaStream_t (NULL = legacy default stream).
 *               Every call is asynchronous on that stream; nothing is
 *               synchronised unless stated.
 *   Errors      Every call returns a status and never throws or aborts.
 *               Arguments are validated before any CUDA call; a rejected call
 *               launches nothing. Zero-sized problems (any of b, h, s_q, s_kv
 *               equal to 0) return SDPA_OK and launch nothing, as the cuDNN
 *               glue does for 0-element tensors.
 *   Devices     The current CUDA device must be a compute capability 10.3
 *               GPU (GB300); the library holds one 4-byte error word per
 *               device in its static device memory.
 */
#ifndef SDPA_H_
#define SDPA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  SDPA_OK = 0,
  SDPA_ERR_INVALID_ARG = 1,   /* null pointer, negative size, p outside [0,1) */
  SDPA_ERR_UNSUPPORTED = 2,   /* head sizes, dtype, or dropout with s_kv % 4 != 0 */
  SDPA_ERR_MISALIGNED = 3,    /* a pointer that is not 16-byte aligned */
  SDPA_ERR_WORKSPACE = 4,     /* workspace null or smaller than sdpa_bwd_workspace_size */
  SDPA_ERR_CUDA = 5,          /* a CUDA runtime / driver call failed */
  SDPA_ERR_DEVICE_TIMEOUT = 6 /* a kernel gave up waiting (see sdpa_device_error) */
} sdpa_status_t;

typedef enum { SDPA_BF16 = 0, SDPA_FP16 = 1 } sdpa_dtype_t;

/*
 * Forward pass (the S .. O lines of the CK header equations; output set of
 * run_cudnn_SDP_fprop with the softmax statistics requested).
 *   q, k, v   inputs (dtype), BHSD.
 *   bias      optional fp32 [1,h,s_q,s_kv] added after scaling; NULL for none.
 *   o         output [b,h,s_q,d_v] (dtype), O = (P * Z) V with Z the dropout
 *             factor (1 without dropout).
 *   lse       output fp32 [b,h,s_q].
 */
sdpa_status_t sdpa_fwd(int64_t b, int64_t h, int64_t s_q, int64_t s_kv, int64_t d_qk,
                       int64_t d_v, float scale, int is_causal, float dropout_p, uint64_t seed,
                       uint64_t offset, sdpa_dtype_t dtype, const void* q, const void* k,
                       const void* v, const float* bias, void* o, float* lse, void* stream);

/*
 * Bytes of device workspace sdpa_bwd needs. Every backward keeps two fp32 row
 * statistics per query row, D = rowsum(dO * O) (oneDNN's sdpa micro.cpp books
 * the same buffer in its scratchpad) and -LSE * log2(e), with s_q padded up
 * to a multiple of 128 for each (b, h): 8 * b * h * ceil(s_q / 128) * 128
 * bytes, rounded up to 256. The default backward at d_qk <= 128 also keeps
 * its fp32 dQ accumulator there (CK tile fmha_bwd_kernel.hpp's dq_acc,
 * oneDNN's f32 dQ scratchpad): 4 * b * h * ceil(s_q / 128) * 128 * d_qk bytes
 * more. Returns 0 for invalid sizes.
 */
size_t sdpa_bwd_workspace_size(int64_t b, int64_t h, int64_t s_q, int64_t s_kv, int64_t d_qk,
                               int64_t d_v);

/*
 * The workspace of any batch-mode backward: h_kv K/V heads (h_kv = h when
 * they are not grouped; see the grouped calls), and deterministic != 0 for
 * the deterministic backward (SDPA_BWD_DETERMINISTIC), which needs only the
 * row statistics. With grouped heads the room for splitting large groups is
 * included (see sdpa_bwd_workspace_size_gqa). 0 for invalid sizes.
 */
size_t sdpa_bwd_workspace_size_ex(int64_t b, int64_t h, int64_t h_kv, int64_t s_q, int64_t s_kv,
                                  int64_t d_qk, int64_t d_v, int deterministic);

/*
 * Backward pass (the dV .. dQ lines of the CK header equations; argument set
 * of run_cudnn_SDP_bprop plus the bias gradient).
 *   o, lse    the forward outputs for the same inputs and parameters.
 *   dout      upstream gradient dO [b,h,s_q,d_v] (dtype).
 *   dq, dk, dv  outputs (dtype), shapes of q, k, v.
 *   dbias     fp32 [1,h,s_q,s_kv] output (overwritten with sum_b dS); must be
 *             non-NULL iff bias is non-NULL.
 *   workspace caller-owned device memory of at least
 *             sdpa_bwd_workspace_size(...) bytes, 256-byte aligned; its
 *             contents on entry are ignored and on exit are unspecified.
 * Runs up to three kernels on `stream`. At d_qk <= 128 (the default backward):
 * preprocess (row statistics; zero dBias and the dQ accumulator), one
 * key/value-stationary kernel that forms every product of each (query tile,
 * key tile) pair once (dK, dV, dBias, and dQ added into the fp32 accumulator
 * with fp32 reductions, as CK tile's FmhaBwdDQDKDVKernel and oneDNN's backward
 * kernel do), and a convert pass dQ = scale * dQacc (with s_kv <= 128 under a
 * mask where every query tile meets the one key tile, and no split of
 * grouped heads, the kernel writes dQ itself: two kernels, dQ reproducible
 * too). dK and dV are bitwise
 * reproducible; dQ's fp32 sums depend on the order the reductions arrive in
 * (results of two calls may differ in the last bits), as does dBias for
 * b > 2. At d_qk = 192, and with SDPA_BWD_DETERMINISTIC, the deterministic
 * backward instead: preprocess, the key/value-stationary kernel (dK, dV,
 * dBias) and a query-stationary kernel that sums dQ over the key tiles inside
 * one CTA (recomputing S and dP), so dQ, dK and dV are bitwise reproducible.
 */
sdpa_status_t sdpa_bwd(int64_t b, int64_t h, int64_t s_q, int64_t s_kv, int64_t d_qk,
                       int64_t d_v, float scale, int is_causal, float dropout_p, uint64_t seed,
                       uint64_t offset, sdpa_dtype_t dtype, const void* q, const void* k,
                       const void* v, const float* bias, const void* o, const void* dout,
                       const float* lse, void* dq, void* dk, void* dv, float* dbias,
                       void* workspace, size_t workspace_bytes, void* stream);

/* Phases of the backward pass, in the order they must run, and the flag that
 * selects the deterministic backward. */
typedef enum {
  SDPA_BWD_PREPROCESS = 1, /* D = rowsum(dO * O) and -LSE*log2e; zero dQacc (and dBias,
                              for the fused backward) */
  SDPA_BWD_DKDV = 2,       /* key/value-stationary kernel: dK, dV, dBias (the deterministic
                              backward zeroes dBias first) (and dQacc, or dQ itself where
                              each dQ row has one key tile) */
  SDPA_BWD_DQ = 4,         /* dQ: convert dQacc (nothing left to do when the fused
                              kernel wrote dQ), or the query-stationary kernel */
  SDPA_BWD_ALL = 7,
  SDPA_BWD_DETERMINISTIC = 8 /* flag: the deterministic backward (no dQ accumulator) */
} sdpa_bwd_phase_t;

/*
 * sdpa_bwd restricted to the phases set in `phases` (a non-empty subset of
 * SDPA_BWD_ALL, optionally with SDPA_BWD_DETERMINISTIC), with identical
 * arguments and validation. Issuing the three phases in order, with the same
 * arguments and flag, on one stream is exactly sdpa_bwd (or its
 * deterministic form); they are separate so a caller can time them one by
 * one (the CK page also splits its backward into three kernels:
 * FmhaBwdOGradDotOKernel, FmhaBwdDQDKDVKernel, FmhaBwdConvertQGradKernel).
 * The later phases read the row statistics (and the zeroed dQ accumulator)
 * the preprocess phase leaves in `workspace`, and the dK/dV phase adds into
 * `dbias`, so the preprocess phase must run first. With the flag the
 * workspace need only hold sdpa_bwd_workspace_size_ex(..., 1) bytes.
 */
sdpa_status_t sdpa_bwd_phases(int phases, int64_t b, int64_t h, int64_t s_q, int64_t s_kv,
                              int64_t d_qk, int64_t d_v, float scale, int is_causal,
                              float dropout_p, uint64_t seed, uint64_t offset, sdpa_dtype_t dtype,
                              const void* q, const void* k, const void* v, const float* bias,
                              const void* o, const void* dout, const float* lse, void* dq, void* dk,
                              void* dv, float* dbias, void* workspace, size_t workspace_bytes,
                              void* stream);

/*
 * Grouped K/V heads (GQA; MQA when h_kv = 1): the same three calls with an
 * h_kv argument. q, o, dout, dq and lse have h query heads; k, v, dk and dv
 * have h_kv heads, [b, h_kv, s_kv, d]; query head i reads K/V head
 * i / (h / h_kv), so consecutive query heads share a K/V head (CK tile
 * fmha_bwd_kernel.hpp: K and V taken at i_nhead / nhead_ratio_qk; oneDNN sdpa
 * micro.cpp: kv_group_size = query heads / KV heads). dK and dV are the sums
 * over each group, formed inside the key/value-stationary kernel without
 * atomics, so they stay bitwise reproducible. Bias, dBias, the dropout bits
 * and the workspace are per query head, as in the ungrouped calls.
 * Requires 1 <= h_kv <= h with h_kv dividing h (SDPA_ERR_INVALID_ARG
 * otherwise); with h_kv = h these are exactly sdpa_fwd / sdpa_bwd /
 * sdpa_bwd_phases.
 */
/*
 * Workspace for the grouped backward: sdpa_bwd_workspace_size's bytes plus,
 * when the group is large for the number of key tiles (e.g. MQA at a small
 * batch), room for splitting each group's query heads over several CTAs per
 * key tile (fp32 partial dK / dV rows and one counter per key tile; the last
 * CTA of a tile adds the partials in a fixed order, so results stay bitwise
 * reproducible). sdpa_bwd_gqa / sdpa_bwd_phases_gqa split only when given
 * at least this many bytes and run one CTA per key tile with the smaller
 * workspace. 0 for invalid sizes.
 */
size_t sdpa_bwd_workspace_size_gqa(int64_t b, int64_t h, int64_t h_kv, int64_t s_q, int64_t s_kv,
                                   int64_t d_qk, int64_t d_v);
sdpa_status_t sdpa_fwd_gqa(int64_t b, int64_t h, int64_t h_kv, int64_t s_q, int64_t s_kv,
                           int64_t d_qk, int64_t d_v, float scale, int is_causal, float dropout_p,
                           uint64_t seed, uint64_t offset, sdpa_dtype_t dtype, const void* q,
                           const void* k, const void* v, const float* bias, void* o, float* lse,
                           void* stream);
sdpa_status_t sdpa_bwd_gqa(int64_t b, int64_t h, int64_t h_kv, int64_t s_q, int64_t s_kv,
                           int64_t d_qk, int64_t d_v, float scale, int is_causal, float dropout_p,
                           uint64_t seed, uint64_t offset, sdpa_dtype_t dtype, const void* q,
                           const void* k, const void* v, const float* bias, const void* o,
                           const void* dout, const float* lse, void* dq, void* dk, void* dv,
                           float* dbias, void* workspace, size_t workspace_bytes, void* stream);
sdpa_status_t sdpa_bwd_phases_gqa(int phases, int64_t b, int64_t h, int64_t h_kv, int64_t s_q,
                                  int64_t s_kv, int64_t d_qk, int64_t d_v, float scale,
                                  int is_causal, float dropout_p, uint64_t seed, uint64_t offset,
                                  sdpa_dtype_t dtype, const void* q, const void* k, const void* v,
                                  const float* bias, const void* o, const void* dout,
                                  const float* lse, void* dq, void* dk, void* dv, float* dbias,
                                  void* workspace, size_t workspace_bytes, void* stream);

/*
 * Packed variable-length sequences (CK tile fmha_bwd_kernel.hpp group mode:
 * seqstart_q_ptr / seqstart_k_ptr give each sequence's first row, and the
 * batch offsets become query_start / key_start times the row stride).
 *   Layout   q, o, dout, dq [h, total_q, d]; k, v, dk, dv [h_kv, total_k, d];
 *            lse [h, total_q] fp32: every head holds all sequences' rows one
 *            after another (BHSD with the batch folded into the rows).
 *   Sequences  b of them. seqstart_q / seqstart_k are DEVICE arrays of b + 1
 *            int32 (4-byte aligned): sequence i owns query rows
 *            [seqstart_q[i], seqstart_q[i+1]) and key rows [seqstart_k[i],
 *            seqstart_k[i+1]), non-decreasing, seqstart[b] <= total. They are
 *            read on the device only; the kernels clamp them into [0, total)
 *            so that no content makes them access memory out of range (out-of-
 *            order entries give wrong results, never a fault).
 *   max_seqlen_q / max_seqlen_k  at least every sequence's length (rows past
 *            them are neither read nor written); they size the grid and take
 *            the place of s_q / s_kv in every rule above.
 *   Masks    each sequence is its own problem: causal is top-left within the
 *            sequence (local key j visible to local query i iff j <= i); keys
 *            of other sequences are never visible. A query row whose sequence
 *            has no key gets O = 0, LSE = -inf and dQ = 0; a key whose
 *            sequence has no query gets dK = dV = 0.
 *   Dropout  the keep bit of (sequence i, head hh, local query r, local key c)
 *            is the batch-mode bit of element (i, hh, r, c) of a
 *            [b, h, max_seqlen_q, max_seqlen_k] problem (see "Dropout"), so
 *            max_seqlen_k % 4 == 0 is required when dropout_p > 0.
 *   Inputs   K/V rows of the neighbouring sequence can enter a tile before
 *            their scores are masked: inputs must be finite.
 *   Bias     not supported with packed sequences (no bias argument).
 *   Workspace  256-byte aligned. sdpa_bwd_varlen_workspace_size_ex(b, h,
 *            total_q, d_qk, 0) bytes run the default backward (at d_qk <= 128
 *            the fused one, with its fp32 dQ accumulator over the packed rows:
 *            4 * h * ceil(total_q / 128) * 128 * d_qk bytes after the
 *            statistics); a workspace of fewer bytes but at least
 *            sdpa_bwd_varlen_workspace_size(b, h, total_q) (the row statistics
 *            alone, = the _ex size with deterministic != 0) runs the
 *            deterministic backward. The fused backward's convert pass writes
 *            every row of dq: rows of no sequence get dQ = 0. Both sizes are 0
 *            for invalid sizes.
 * h_kv as in the grouped calls. Zero b, h, total_q, total_k, max_seqlen_q or
 * max_seqlen_k is a no-op returning SDPA_OK.
 */
size_t sdpa_bwd_varlen_workspace_size(int64_t b, int64_t h, int64_t total_q);
size_t sdpa_bwd_varlen_workspace_size_ex(int64_t b, int64_t h, int64_t total_q, int64_t d_qk,
                                         int deterministic);
sdpa_status_t sdpa_fwd_varlen(int64_t b, int64_t h, int64_t h_kv, int64_t total_q, int64_t total_k,
                              int64_t max_seqlen_q, int64_t max_seqlen_k, int64_t d_qk, int64_t d_v,
                              float scale, int is_causal, float dropout_p, uint64_t seed,
                              uint64_t offset, sdpa_dtype_t dtype, const int32_t* seqstart_q,
                              const int32_t* seqstart_k, const void* q, const void* k, const void* v,
                              void* o, float* lse, void* stream);
sdpa_status_t sdpa_bwd_varlen(int64_t b, int64_t h, int64_t h_kv, int64_t total_q, int64_t total_k,
                              int64_t max_seqlen_q, int64_t max_seqlen_k, int64_t d_qk, int64_t d_v,
                              float scale, int is_causal, float dropout_p, uint64_t seed,
                              uint64_t offset, sdpa_dtype_t dtype, const int32_t* seqstart_q,
                              const int32_t* seqstart_k, const void* q, const void* k, const void* v,
                              const void* o, const void* dout, const float* lse, void* dq, void* dk,
                              void* dv, void* workspace, size_t workspace_bytes, void* stream);
sdpa_status_t sdpa_bwd_phases_varlen(int phases, int64_t b, int64_t h, int64_t h_kv, int64_t total_q,
                                     int64_t total_k, int64_t max_seqlen_q, int64_t max_seqlen_k,
                                     int64_t d_qk, int64_t d_v, float scale, int is_causal,
                                     float dropout_p, uint64_t seed, uint64_t offset,
                                     sdpa_dtype_t dtype, const int32_t* seqstart_q,
                                     const int32_t* seqstart_k, const void* q, const void* k,
                                     const void* v, const void* o, const void* dout,
                                     const float* lse, void* dq, void* dk, void* dv,
                                     void* workspace, size_t workspace_bytes, void* stream);

/*
 * Local windows, the bottom-right alignment, ALiBi and dropout bits drawn
 * beforehand (CK tile
 * fmha_bwd_kernel.hpp mask arguments window_size_left, window_size_right and
 * mask_type, and its ALiBi slopes alibi_slope_ptr / alibi_slope_stride;
 * oneDNN sdpa micro.cpp's top_left and bottom_right attention masks). The
 * grouped and packed calls with is_causal replaced by:
 *   window_left, window_right  key j is visible to query i iff
 *            i + off - window_left <= j <= i + off + window_right; a negative
 *            size leaves that side unbounded (so does one of s_q + s_kv or
 *            more).
 *   bottom_right  0: off = 0 (diagonal through (0, 0)); 1: off = s_kv - s_q
 *            (diagonal through (s_q - 1, s_kv - 1)), per sequence when packed.
 *   alibi_slopes  null, or a DEVICE fp32 array: the score of (i, j) in batch
 *            entry (or sequence) bb and query head hh gets
 *            -alibi_slopes[bb * alibi_stride + hh] * |j - i - off_a| added
 *            after the scale (the slopes are constants, with no gradient);
 *            off_a = 0 when a window size is given (>= 0) and bottom_right is
 *            0, else s_kv - s_q. 4-byte aligned (SDPA_ERR_MISALIGNED).
 *   alibi_stride  0 (one slope per head for every batch entry) or >= h
 *            (SDPA_ERR_INVALID_ARG otherwise).
 *   keep_bits  null, or the dropout keep bits of the whole problem drawn
 *            beforehand by sdpa_dropout_mask with the same b, h, s_q, s_kv (the
 *            max lengths when packed), p, seed and offset (DEVICE, 4-byte
 *            aligned), or recorded by a forward call (keep_bits_out): the
 *            kernels then read them instead of drawing Philox numbers, with
 *            identical results. Ignored when dropout_p is 0.
 *   keep_bits_out  (forward calls) null, or DEVICE memory of
 *            ceil(b*h*s_q*s_kv / 32) words (4-byte aligned) where the forward
 *            records the keep bits it draws, in sdpa_dropout_mask's packing,
 *            so that the backward can take them as keep_bits instead of
 *            drawing them again (CK tile's kIsStoreRandval keeps its random
 *            values for the same reason). Only the words of (query row, key
 *            tile) pairs the forward visits are written; a backward with the
 *            same mask reads no other. With no mask (window (-1, -1), batch
 *            mode) every word is written, by sdpa_dropout_mask's kernel on the
 *            same stream before the forward, which then reads them. Requires s_kv % 32 == 0
 *            (SDPA_ERR_UNSUPPORTED) and keep_bits null (SDPA_ERR_INVALID_ARG);
 *            ignored when dropout_p is 0.
 * Causal is (-1, 0, 0), bottom-right causal (-1, 0, 1), a sliding window of
 * w keys back (w, 0, 0), no mask (-1, -1, 0). A query row that sees no key
 * gets O = 0, LSE = -inf and dQ = 0; a key no query sees gets dK = dV = 0.
 * Key tiles outside every window of a tile's rows are skipped, so a window of
 * w keys costs about (w + 128) / s_kv of the unmasked work.
 */
sdpa_status_t sdpa_fwd_ex(int64_t b, int64_t h, int64_t h_kv, int64_t s_q, int64_t s_kv,
                              int64_t d_qk, int64_t d_v, float scale, int64_t window_left,
                              int64_t window_right, int bottom_right, const float* alibi_slopes,
                              int64_t alibi_stride, const uint32_t* keep_bits, uint32_t* keep_bits_out,
                              float dropout_p, uint64_t seed,
                              uint64_t offset, sdpa_dtype_t dtype, const void* q, const void* k,
                              const void* v, const float* bias, void* o, float* lse, void* stream);
sdpa_status_t sdpa_bwd_ex(int64_t b, int64_t h, int64_t h_kv, int64_t s_q, int64_t s_kv,
                              int64_t d_qk, int64_t d_v, float scale, int64_t window_left,
                              int64_t window_right, int bottom_right, const float* alibi_slopes,
                              int64_t alibi_stride, const uint32_t* keep_bits, float dropout_p, uint64_t seed,
                              uint64_t offset, sdpa_dtype_t dtype, const void* q, const void* k,
                              const void* v, const float* bias, const void* o, const void* dout,
                              const float* lse, void* dq, void* dk, void* dv, float* dbias,
                              void* workspace, size_t workspace_bytes, void* stream);
sdpa_status_t sdpa_bwd_phases_ex(int phases, int64_t b, int64_t h, int64_t h_kv, int64_t s_q,
                                     int64_t s_kv, int64_t d_qk, int64_t d_v, float scale,
                                     int64_t window_left, int64_t window_right, int bottom_right,
                                     const float* alibi_slopes, int64_t alibi_stride, const uint32_t* keep_bits,
                                     float dropout_p, uint64_t seed, uint64_t offset,
                                     sdpa_dtype_t dtype, const void* q, const void* k, const void* v,
                                     const float* bias, const void* o, const void* dout,
                                     const float* lse, void* dq, void* dk, void* dv, float* dbias,
                                     void* workspace, size_t workspace_bytes, void* stream);
sdpa_status_t sdpa_fwd_varlen_ex(int64_t b, int64_t h, int64_t h_kv, int64_t total_q,
                                     int64_t total_k, int64_t max_seqlen_q, int64_t max_seqlen_k,
                                     int64_t d_qk, int64_t d_v, float scale, int64_t window_left,
                                     int64_t window_right, int bottom_right,
                                     const float* alibi_slopes, int64_t alibi_stride, const uint32_t* keep_bits,
                                     uint32_t* keep_bits_out, float dropout_p, uint64_t seed,
                                     uint64_t offset, sdpa_dtype_t dtype, const int32_t* seqstart_q,
                                     const int32_t* seqstart_k, const void* q, const void* k,
                                     const void* v, void* o, float* lse, void* stream);
sdpa_status_t sdpa_bwd_varlen_ex(int64_t b, int64_t h, int64_t h_kv, int64_t total_q,
                                     int64_t total_k, int64_t max_seqlen_q, int64_t max_seqlen_k,
                                     int64_t d_qk, int64_t d_v, float scale, int64_t window_left,
                                     int64_t window_right, int bottom_right,
                                     const float* alibi_slopes, int64_t alibi_stride, const uint32_t* keep_bits,
                                     float dropout_p, uint64_t seed, uint64_t offset,
                                     sdpa_dtype_t dtype, const int32_t* seqstart_q,
                                     const int32_t* seqstart_k, const void* q, const void* k,
                                     const void* v, const void* o, const void* dout,
                                     const float* lse, void* dq, void* dk, void* dv,
                                     void* workspace, size_t workspace_bytes, void* stream);
sdpa_status_t sdpa_bwd_phases_varlen_ex(
    int phases, int64_t b, int64_t h, int64_t h_kv, int64_t total_q, int64_t total_k,
    int64_t max_seqlen_q, int64_t max_seqlen_k, int64_t d_qk, int64_t d_v, float scale,
    int64_t window_left, int64_t window_right, int bottom_right, const float* alibi_slopes,
    int64_t alibi_stride, const uint32_t* keep_bits, float dropout_p, uint64_t seed, uint64_t offset, sdpa_dtype_t dtype,
    const int32_t* seqstart_q, const int32_t* seqstart_k, const void* q, const void* k,
    const void* v, const void* o, const void* dout, const float* lse, void* dq, void* dk, void* dv,
    void* workspace, size_t workspace_bytes, void* stream);

/*
 * The backward pass for callers that cannot allocate device memory when they
 * run it (a host framework that owns all GPU memory through its own pool, or
 * a latency-critical loop that cannot afford cudaMalloc's implicit
 * synchronisation). There is no counterpart on the pages; it exists for such
 * callers. Same arguments as sdpa_bwd minus the workspace, and the results of
 * the deterministic backward (sdpa_bwd_phases with SDPA_BWD_ALL |
 * SDPA_BWD_DETERMINISTIC): its scratch, the per-row statistics, lives in a
 * 16 MiB static device array inside the library, which every GPU that loads
 * the library holds until the process exits. The call allocates nothing.
 *   Limit    problems whose sdpa_bwd_workspace_size_ex(b, h, h, s_q, s_kv,
 *            d_qk, d_v, 1) exceeds 16 MiB are rejected with
 *            SDPA_ERR_WORKSPACE before any device work (detail in
 *            sdpa_last_error).
 *   Sharing  all calls on a device use the same array and leave their data in
 *            it; each call rewrites what it reads, but calls whose kernels
 *            overlap on the GPU (e.g. on two streams) race: serialise them.
 *   Set-up   the first call on each device looks up the array's device
 *            address (cudaGetSymbolAddress) with that device current; make
 *            that first call before any stream capture begins.
 */
sdpa_status_t sdpa_bwd_noalloc(int64_t b, int64_t h, int64_t s_q, int64_t s_kv, int64_t d_qk,
                               int64_t d_v, float scale, int is_causal, float dropout_p,
                               uint64_t seed, uint64_t offset, sdpa_dtype_t dtype, const void* q,
                               const void* k, const void* v, const float* bias, const void* o,
                               const void* dout, const float* lse, void* dq, void* dk, void* dv,
                               float* dbias, void* stream);

/*
 * Test hook: the packed dropout keep bits of a whole problem, drawn by the
 * same device Philox function the fused kernels use. Bit (L % 32) of word
 * bits[L / 32] is element L's keep flag (L as in "Dropout" above); bits past
 * the last element of the final word are 0. bits must hold
 * ceil(b*h*s_q*s_kv / 32) words. p == 0 gives all ones.
 */
sdpa_status_t sdpa_dropout_mask(int64_t b, int64_t h, int64_t s_q, int64_t s_kv, float dropout_p,
                                uint64_t seed, uint64_t offset, uint32_t* bits, void* stream);

/*
 * Reads the current device's error word (synchronising the device) and, when
 * `clear` is non-zero, resets it. A non-zero word means a kernel's bounded
 * wait ran out: the kernel recorded which role gave up (bit mask), released
 * its resources and returned without completing its outputs. Returns
 * SDPA_ERR_DEVICE_TIMEOUT when the word is non-zero, SDPA_OK otherwise.
 */
sdpa_status_t sdpa_device_error(uint32_t* word, int clear);

/*
 * Test hook for the bounded-wait path (no counterpart on the pages; it exists
 * so the hang-safety machinery can be exercised without faulting a GPU).
 * Applies to sdpa_fwd calls made after it, on any thread, until reset:
 *   fault 0  normal operation (the default)
 *   fault 1  the forward kernel's producer warp issues no K/V loads, so the
 *            MMA issuer's bounded wait runs out: every role leaves its loop,
 *            drains what is in flight, frees tensor memory and returns; the
 *            error word gets the MMA site bit, sdpa_device_error then reports
 *            SDPA_ERR_DEVICE_TIMEOUT, and O / LSE are left unwritten.
 *   wait_limit_ns  wall-clock limit of each device wait in those forward
 *            launches; 0 restores the default (2 s).
 * Returns SDPA_ERR_INVALID_ARG for an unknown fault. Call sdpa_debug_fault(0, 0)
 * to restore normal operation.
 */
sdpa_status_t sdpa_debug_fault(int fault, uint64_t wait_limit_ns);

/*
 * Test hook, host only (no device work, no CUDA call): the (query tile, key
 * tile) pairs a kernel of this library processes for one sequence of s_q
 * query rows and s_kv keys under a mask given as for sdpa_fwd_ex (window
 * (-1, 0) is the plain causal mask, (-1, -1) none), computed by the functions
 * the kernels themselves call, so that a host test can check them against
 * the visibility rule. The kernels' other cases (packed sequences, grouped
 * heads) walk the same ranges per sequence and head.
 *   kernel      0 the forward, 1 the key/value-stationary backward kernels
 *               (dK/dV and the fused one), 2 the query-stationary dQ kernel
 *   windowed    nonzero: the band arithmetic the kernels use for any
 *               window that is not plain (and, with ALiBi, for the plain ones
 *               too); zero: the mask decides, as without ALiBi
 *   query_rows  the kernel's query tile height: 128, or 64 for the dK/dV
 *               kernel at d_qk = 192
 *   out         HOST memory for up to cap triples (first query row of the
 *               tile, query rows of the tile, key tile index of 128 keys),
 *               in the order the kernels' CTAs walk them
 * Returns the number of triples (written up to cap), or -1 for an invalid
 * argument (kernel, query_rows, negative or out-of-range sizes, out null with
 * cap > 0).
 */
int64_t sdpa_tile_ranges(int kernel, int64_t s_q, int64_t s_kv, int64_t window_left,
                         int64_t window_right, int bottom_right, int windowed, int query_rows,
                         int32_t* out, int64_t cap);

/* Detail of the calling thread's most recent failure (the step and, for
 * SDPA_ERR_CUDA, the CUDA error string); "" if none. Valid until the thread's
 * next call into the library. */
const char* sdpa_last_error(void);

/* Static, human-readable name of a status code. */
const char* sdpa_status_string(sdpa_status_t status);

/* Library version as MAJOR*10000 + MINOR*100 + PATCH. */
int sdpa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* SDPA_H_ */
