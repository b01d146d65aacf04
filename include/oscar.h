/*
 * oscar.h -- C ABI of liboscar.so: OSCAR-style rotated INT2 KV cache on GB300.
 *
 * Sources (web pages, cited by title and section):
 *  [OSCAR news]  "Together AI、OSCARをオープンソース化：長コンテキストLLMサービング
 *                のためのアテンション認識2ビットKVキャッシュ量子化システム"
 *                sections "OSCARの違い" (C_Q, C_S, R = U·H_Had·P_br, logit-error
 *                identity) and "サービングシステム：混合精度キャッシュレイアウト"
 *                (64 BF16 sink tokens, 256 BF16 recent tokens, INT2 history
 *                after rotation and clipping, paged attention).
 *  [Escha log]   "RTX 5070×2(12GB×2)でQwen3.8-27B-Escha-W2を動かす", part 2
 *                "KVキャッシュも2bitにして長コンテキストにする": fix 1 (0.25 byte
 *                per INT2 element), fix 3 (Hadamard / sqrt(head_dim)), fix 4
 *                (query head -> KV head mapping), settings table (group size 64).
 *  [Scheduler log] sglang scheduler article on 12 GB / 27B: page_size 1.
 *  [Prefix log]  "KVプールが上限だった — hybrid GDN の長文キャッシュ…": the INT2
 *                prefill path expands the cached prefix to fp16 before attention.
 *
 * Conventions shared by every entry point
 *  - Return value: OSCAR_OK (0) or a negative OSCAR_ERR_* code.  Nothing
 *    aborts, throws or traps.  oscar_last_error() returns a message for the
 *    last failing call on the calling thread.
 *  - Arguments are validated on the host before anything is launched; a
 *    failed validation launches nothing and leaves every buffer untouched.
 *  - Device pointers are CUDA device (or managed) memory owned by the caller;
 *    the library never frees or keeps them.  Host pointers are marked "host".
 *  - `stream` is a cudaStream_t (NULL = the legacy default stream).  Device
 *    work is enqueued asynchronously on it; the library allocates no device
 *    memory on the append and decode paths.
 *  - Row-vector convention: a head vector x is rotated as x·R (R row-major).
 *  - Device-side checks (slot ids, positions, request rows, sequence
 *    lengths) never trap: an offending access is skipped and a bit is set in
 *    a per-device status word read by oscar_device_status().
 */
#ifndef OSCAR_H
#define OSCAR_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes ------------------------------------------------------ */
#define OSCAR_OK               0
#define OSCAR_ERR_ARG         -1  /* bad shape, dtype or parameter            */
#define OSCAR_ERR_NULL        -2  /* a required pointer is NULL               */
#define OSCAR_ERR_WORKSPACE   -3  /* workspace missing or too small           */
#define OSCAR_ERR_CUDA        -4  /* a CUDA runtime call or launch failed     */
#define OSCAR_ERR_NUMERIC     -5  /* eigensolver did not converge             */

/* bits of the device status word (oscar_device_status) */
#define OSCAR_DEV_BAD_SLOT     1  /* page-table slot outside [0, num_slots)   */
#define OSCAR_DEV_BAD_LEN      2  /* seq_len outside [1, max_seq_len] or a
                                     position beyond the page-table row       */
#define OSCAR_DEV_BAD_REQ      4  /* req_idx outside [0, max_reqs)            */
#define OSCAR_DEV_TIMEOUT      8  /* a bounded pipeline wait gave up          */

/* ---- element types ------------------------------------------------------ */
#define OSCAR_DTYPE_BF16       0
#define OSCAR_DTYPE_F32        1

/* storage of a group's (scale, zero) pair in the INT2 records */
#define OSCAR_SCALE_F16        0  /* two fp16 values (4 bytes per group)       */
#define OSCAR_SCALE_E4M3       1  /* two float8 E4M3 values (2 bytes per group):
                                     2 + 16/G bits per INT2 element, the 2.28
                                     bits per element of [OSCAR news] at G = 64
                                     and 128K context                         */

/* Shape and quantisation parameters of one attention layer.
 *  head_dim      d: 64, 128 or 256.
 *  num_q_heads   Hq; num_kv_heads Hkv; Hq % Hkv == 0, 1 <= Hq/Hkv <= 16,
 *                Hkv <= 64.  Query head h reads KV head h / (Hq/Hkv)
 *                ([Escha log] fix 4).
 *  group_size    G: channels sharing one fp16 (scale, zero); 32, 64, 128 or
 *                256, dividing d ([Escha log] settings table uses 64).
 *  sink, recent  BF16 window sizes S and W ([OSCAR news]: 64 and 256);
 *                0 <= S <= 4096, 1 <= W <= 4096.
 *  clip_ratio    r in (0, 1]: a group's quantisation range is
 *                [r·min, r·max] of its rotated values.
 *  kv_dtype      element type of the K/V rows handed to oscar_quantize_append.
 *  q_dtype       element type of q handed to oscar_decode_attention.
 *  scale_dtype   OSCAR_SCALE_F16 (zero-initialised default) or
 *                OSCAR_SCALE_E4M3: s = rnd((hi - lo)/3) and z = rnd(lo) are
 *                rounded to fp16, or to E4M3 (nearest, ties to even, finite
 *                values beyond ±448 saturate to ±448); codes are decided
 *                against the rounded pair either way.                      */
typedef struct {
    int32_t head_dim;
    int32_t num_q_heads;
    int32_t num_kv_heads;
    int32_t group_size;
    int32_t sink;
    int32_t recent;
    float   clip_ratio;
    int32_t kv_dtype;
    int32_t q_dtype;
    int32_t scale_dtype;
} oscar_config;

/* Device buffers of one layer's cache (all owned by the caller).
 *  records   INT2 pool, uint8 [num_slots][slot_bytes]: slot i holds the
 *            records of all KV heads, head h at byte h·rec_bytes, padded
 *            with zeros to slot_bytes (oscar_slot_bytes(), a multiple of 16;
 *            rec_bytes from oscar_record_bytes()).  One (slot, KV head)
 *            record is
 *              [K codes d/4 B][V codes d/4 B][K (s,z) × d/G][V (s,z) × d/G]
 *            padded with zeros: to a multiple of 16 bytes with fp16 pairs
 *            (4 bytes each), so that slot_bytes = Hkv·rec_bytes, or to a
 *            multiple of 8 bytes with E4M3 pairs (2 bytes each).  Channel j's
 *            2-bit code sits at bits 2·(j%4) of byte j/4; each pair is scale
 *            first.  Base address 16-byte aligned.
 *  sink      bf16 [max_reqs][S][Hkv][2][d]   (index 0 = K, 1 = V)
 *  recent    bf16 [max_reqs][W][Hkv][2][d]   ring: position p at p % W
 *  rot_k     fp32 [d][d] row-major R_K; rot_v likewise R_V (both orthogonal).
 *            The append reads them before waiting for the stream's previous
 *            kernel to finish (programmatic dependent launch), so write them
 *            with a copy or with a kernel that does not signal its dependents
 *            early.
 *  num_slots number of records in the pool; max_reqs rows of the windows.  */
typedef struct {
    uint8_t*     records;
    uint16_t*    sink;
    uint16_t*    recent;
    const float* rot_k;
    const float* rot_v;
    int64_t      num_slots;
    int32_t      max_reqs;
} oscar_layer_cache;

/* ---- information ------------------------------------------------------- */

/* Version string of the library (static storage). */
const char* oscar_version(void);

/* Message of the last failing call on this thread ("" if none). */
const char* oscar_last_error(void);

/* Bytes of one (slot, KV head) record: d/2 + 8·d/G rounded up to 16 with fp16
 * (s, z), d/2 + 4·d/G rounded up to 8 with E4M3.  80 / 72 at d=128, G=64;
 * 144 / 136 at d=256, G=128. */
int oscar_record_bytes(const oscar_config* cfg, int64_t* out /*host*/);

/* Bytes of one slot of the pool (the records of all KV heads): Hkv·rec_bytes
 * rounded up to 16.  640 (fp16) / 576 (E4M3) at d=128, G=64, 8 KV heads. */
int oscar_slot_bytes(const oscar_config* cfg, int64_t* out /*host*/);

/* Storage per cached token of one layer, all KV heads:
 *  int2_bytes  INT2 slot bytes (codes + scales + padding) per history token
 *  bf16_bytes  BF16 bytes per sink/recent token (2·Hkv·d·2).
 * The code share alone is Hkv·d·2·0.25 bytes ([Escha log] fix 1). */
int oscar_cache_bytes_per_token(const oscar_config* cfg, int64_t* int2_bytes /*host*/,
                                int64_t* bf16_bytes /*host*/);

/* ---- rotation construction (host, fp64) -------------------------------- */

/* C = (1/n) Σ_i x_iᵀ x_i over the rows of samples (host, row-major n×d, fp64):
 * the empirical query covariance C_Q of [OSCAR news] "OSCARの違い".
 * cov: host, d×d fp64 output.  n >= 1, 1 <= d <= 4096. */
int oscar_covariance(const double* samples, int64_t n, int32_t d, double* cov);

/* C_S = (1/n_q) Vᵀ Sᵀ S V, the score-weighted value covariance of
 * [OSCAR news] "OSCARの違い".  scores: host n_q×n_k fp64 (row-major);
 * values: host n_k×d fp64; cov: host d×d fp64 output. */
int oscar_value_covariance(const double* scores, const double* values, int64_t n_q,
                           int64_t n_k, int32_t d, double* cov);

/* ---- calibration statistics on the device ------------------------------ */

/* Workspace bytes of oscar_covariance_device for n rows of width d (host output). */
int oscar_covariance_workspace_bytes(int64_t n, int32_t d, size_t* bytes);

/* C = (1/n) Σ_i x_iᵀ x_i over the rows of x, the query covariance C_Q of
 * [OSCAR news] "OSCARの違い", on the device.
 *  x          device, row-major n×d in x_dtype (OSCAR_DTYPE_BF16 or _F32)
 *  cov        device, d×d fp64 output (symmetric, both triangles written)
 *  workspace  device, >= oscar_covariance_workspace_bytes(n, d), 256-byte aligned
 * Accumulated in fp64 (every product of bf16 or fp32 inputs is exact; the
 * additions round) over row slices added in a fixed order, so repeated calls
 * give identical results.  n >= 1, 1 <= d <= 4096.  Asynchronous on stream. */
int oscar_covariance_device(const void* x, int32_t x_dtype, int64_t n, int32_t d, double* cov,
                            void* workspace, size_t workspace_bytes, void* stream);

/* Workspace bytes of oscar_value_covariance_device (host output). */
int oscar_value_covariance_workspace_bytes(int64_t n_q, int64_t n_k, int32_t d, size_t* bytes);

/* C_S = (1/n_q) Vᵀ Sᵀ S V, the score-weighted value covariance of
 * [OSCAR news] "OSCARの違い", on the device: Y = S·V (fp64 accumulation),
 * then C_S = (1/n_q) YᵀY as in oscar_covariance_device.
 *  scores     device fp32 n_q×n_k (row-major attention scores of the calibration queries)
 *  values     device n_k×d in v_dtype (OSCAR_DTYPE_BF16 or _F32)
 *  cov        device d×d fp64 output
 *  workspace  device, >= oscar_value_covariance_workspace_bytes(n_q, n_k, d), 256-byte aligned
 * 1 <= n_q <= 4,194,240, n_k >= 1, 1 <= d <= 4096.  Asynchronous on stream. */
int oscar_value_covariance_device(const float* scores, const void* values, int32_t v_dtype, int64_t n_q,
                                  int64_t n_k, int32_t d, double* cov, void* workspace,
                                  size_t workspace_bytes, void* stream);

/* R = U · (H_d/√d) · P_br  ([OSCAR news] "OSCARの違い"; [Escha log] fix 3).
 *  cov       host d×d fp64 symmetric covariance, or NULL for U = I (the
 *            calibration-free Hadamard rotation, identical in every layer).
 *  d         power of two, 2..256.
 *  use_bitrev  0: leave out P_br (cov = NULL then gives exactly H/√d).
 *  R_f32     host d×d fp32 output (row-major), required.
 *  R_f64     host d×d fp64 output, optional (NULL).
 *  eigvals   host d fp64 output, optional; descending eigenvalues of cov.
 * U holds the eigenvectors of cov (cyclic Jacobi, fp64) in descending
 * eigenvalue order, each signed so that its largest-magnitude entry is
 * positive (lowest index on a tie).  P_br maps column j to column bitrev(j).
 * Returns OSCAR_ERR_NUMERIC if the eigensolver does not converge. */
int oscar_build_rotation(const double* cov, int32_t d, int32_t use_bitrev,
                         float* R_f32, double* R_f64, double* eigvals);

/* As oscar_build_rotation, with the Hadamard factor block-diagonal: d/B copies
 * of H_B/√B along the diagonal (B = hadamard_block, a power of two in [1, d];
 * B = d is oscar_build_rotation).  [OSCAR news] "OSCARの違い" names the
 * Hadamard factor without a size; with B < d each block mixes only B
 * consecutive eigen-directions (channels of similar importance), and P_br then
 * places every block's channels evenly over the quantisation groups: a group
 * of G consecutive output channels takes G·B/d channels of each block. */
int oscar_build_rotation_ex(const double* cov, int32_t d, int32_t use_bitrev, int32_t hadamard_block,
                            float* R_f32, double* R_f64, double* eigvals);

/* ---- append: rotate, clip, quantise, pack (device) ---------------------- */

/* Append new K/V tokens for a batch of requests ([OSCAR news] serving-system
 * section).  For batch row b, the new rows are k/v[cu_new[b] .. cu_new[b+1])
 * at positions L0 .. L1-1 with L0 = start_pos[b], L1 = L0 + (cu_new[b+1] -
 * cu_new[b]).  Every input vector is first rounded to bf16.  Then:
 *   1. each position in [max(S, L0-W), max(S, L1-W)) enters the history:
 *      positions below L0 are read from the recent ring, the others from
 *      k/v; each K (V) head vector x is rotated y = x·R_K (x·R_V) in fp32,
 *      and per group of G channels: lo = r·min y, hi = r·max y,
 *      s = fp16((hi-lo)/3), z = fp16(lo), c = clamp(rint((y - z)/s), 0, 3)
 *      (fp32, from the fp16-rounded s and z; s == 0 gives c = 0); the codes
 *      and (s, z) are written to record page_table[b][p];
 *   2. new positions p < S are written to sink[req_idx[b]][p]; new positions
 *      p >= max(S, L1-W) to recent[req_idx[b]][p % W].
 * Arguments (device unless marked):
 *  k, v             [total_new][Hkv][d] in cfg->kv_dtype
 *  total_new        host: rows of k and v (may be 0)
 *  cu_new           int32 [batch+1], cu_new[0] = 0, non-decreasing,
 *                   cu_new[batch] = total_new (rows beyond total_new are
 *                   skipped and flagged OSCAR_DEV_BAD_LEN)
 *  start_pos        int32 [batch], tokens already cached per row
 *  req_idx          int32 [batch] window row per batch row, or NULL for b
 *  page_table       int32 [batch][pt_stride]; must cover every position
 *                   that enters the history in this call
 *  batch            host, >= 0
 * Concurrent appends to the same request, or an append racing a decode of
 * the same layer, are the caller's to order (use one stream). */
int oscar_quantize_append(const oscar_config* cfg, const oscar_layer_cache* cache,
                          const void* k, const void* v, int64_t total_new,
                          const int32_t* cu_new, const int32_t* start_pos,
                          const int32_t* req_idx, const int32_t* page_table,
                          int64_t pt_stride, int32_t batch, void* stream);

/* ---- decode attention (device) ----------------------------------------- */

/* Workspace bytes oscar_decode_attention needs for up to `batch` requests of
 * at most `max_seq_len` tokens (host output).  The workspace holds the
 * rotated queries and the per-split (m, l, o) partials. */
int oscar_decode_workspace_bytes(const oscar_config* cfg, int32_t batch,
                                 int32_t max_seq_len, size_t* bytes);

/* One decode step of attention over the mixed cache.
 * For batch row b holding L = seq_lens[b] tokens (the current token
 * included, already appended) and every query head h (KV head h/(Hq/Hkv)):
 *   sink [0, min(S,L)) and recent [max(S,L-W), L): logit = q·k/√d on the
 *     BF16 vectors;
 *   history [S, max(S,L-W)): logit = (q·R_K)·k̂/√d, k̂ = s·c + z;
 *   one softmax over all L logits (split-K over the history with a
 *   log-sum-exp combine), and
 *   out = Σ_bf16 p·v + (Σ_hist p·v̂)·R_Vᵀ.
 * Arguments (device unless marked):
 *  q            [batch][Hq][d] in cfg->q_dtype
 *  page_table   int32 [batch][pt_stride]
 *  seq_lens     int32 [batch], 1 <= L <= max_seq_len
 *  req_idx      int32 [batch] window row, or NULL for b
 *  batch        host, 0 <= batch <= 4096; max_seq_len host, >= 1, <= pt_stride
 *  out          fp32 [batch][Hq][d]
 *  workspace    device, >= oscar_decode_workspace_bytes(cfg, batch,
 *               max_seq_len) bytes, 256-byte aligned; the library writes it
 *               and reads it back within the call's stream order.
 * Returns OSCAR_ERR_ARG if batch or max_seq_len is out of range or
 * num_q_heads·head_dim exceeds 16384 (one request's rotated queries are
 * staged in shared memory), OSCAR_ERR_WORKSPACE if workspace is NULL, too
 * small or misaligned. */
int oscar_decode_attention(const oscar_config* cfg, const oscar_layer_cache* cache,
                           const void* q, const int32_t* page_table, int64_t pt_stride,
                           const int32_t* seq_lens, const int32_t* req_idx,
                           int32_t batch, int32_t max_seq_len, float* out,
                           void* workspace, size_t workspace_bytes, void* stream);

/* One fused decode step: the append of one new token per request followed
 * by attention over the cache that includes it.  The result (out, and every
 * byte written to the cache) is that of
 *   oscar_quantize_append(k_new, v_new, cu_new = 0, 1, .., batch,
 *                         start_pos = seq_lens - 1, req_idx, page_table)
 *   oscar_decode_attention(q, page_table, seq_lens, req_idx, ...)
 * on the same stream, in three launches instead of four: the append, the
 * query preparation and the BF16 window tiles run in one grid (the window
 * tiles read the new token from k_new / v_new, the append writes it to its
 * window row and quantises the token leaving the recent window), then the
 * history kernel and the combine.
 * Arguments (device unless marked): as oscar_decode_attention, plus
 *  k_new, v_new  [batch][Hkv][d] in cfg->kv_dtype: request b's new token,
 *                position seq_lens[b] - 1.
 * seq_lens counts the new token.  A request whose length or window row is
 * invalid is flagged as by oscar_decode_attention and appends nothing. */
int oscar_decode_step(const oscar_config* cfg, const oscar_layer_cache* cache,
                      const void* k_new, const void* v_new, const void* q,
                      const int32_t* page_table, int64_t pt_stride,
                      const int32_t* seq_lens, const int32_t* req_idx,
                      int32_t batch, int32_t max_seq_len, float* out,
                      void* workspace, size_t workspace_bytes, void* stream);

/* Same contract and arguments as oscar_decode_attention, but the history is
 * always processed by the CUDA-core (fp32 FFMA) kernel instead of the
 * tensor-core one.  Kept as the measured baseline for the choice of tensor
 * cores on the QK/PV tiles; results agree with oscar_decode_attention within
 * the attention tolerance. */
int oscar_decode_attention_simt(const oscar_config* cfg, const oscar_layer_cache* cache,
                                const void* q, const int32_t* page_table, int64_t pt_stride,
                                const int32_t* seq_lens, const int32_t* req_idx,
                                int32_t batch, int32_t max_seq_len, float* out,
                                void* workspace, size_t workspace_bytes, void* stream);

/* Allocation-free variant of oscar_decode_attention (no counterpart on the
 * pages: an interface addition of this library).  Same arguments and result
 * minus the workspace: the scratch lives in a 16 MiB array compiled into the
 * library, which every GPU that loads the library holds until the process
 * exits.  It serves callers that cannot allocate device memory -- host
 * runtimes that reserve almost all of the GPU for their own pool and give
 * plug-in kernels no allocation rights, or code paths where a cudaMalloc
 * (which may synchronise the device) is not allowed.  This call allocates
 * nothing: no cudaMalloc, no cudaFree, no allocating library routine.
 *  - Sizes whose scratch need (oscar_decode_workspace_bytes) exceeds 16 MiB
 *    are rejected with OSCAR_ERR_WORKSPACE before anything is launched.
 *  - Every call looks up the array's device address in the current context
 *    (cudaGetSymbolAddress, with the caller's device current), which
 *    allocates nothing; the first call on a device may also load the
 *    library's module there, so make it before any stream capture.
 *  - All calls on a device share the one array and it keeps the previous
 *    call's contents; every byte a call reads is written earlier in the same
 *    call, so nothing needs clearing.  Calls that overlap on the GPU (e.g.
 *    on two streams) race on the array: order them on one stream. */
int oscar_decode_attention_noalloc(const oscar_config* cfg, const oscar_layer_cache* cache,
                                   const void* q, const int32_t* page_table, int64_t pt_stride,
                                   const int32_t* seq_lens, const int32_t* req_idx,
                                   int32_t batch, int32_t max_seq_len, float* out, void* stream);

/* ---- prefill attention over the cached prefix (device) ------------------ */

/* Workspace bytes of oscar_prefill_attention for `batch` requests and
 * `total_q` chunk tokens in all (host output). */
int oscar_prefill_workspace_bytes(const oscar_config* cfg, int32_t batch, int64_t total_q, size_t* bytes);

/* Attention of prefill chunks over the mixed cache, reading the INT2 history
 * directly: [Prefix log] "KVプールが上限だった — hybrid GDN の長文キャッシュ…"
 * describes the prefill path that first expands the cached INT2 prefix into
 * an fp16 workspace growing with the sequence; this call needs no such copy.
 * Request b holds L0 = start_pos[b] tokens in the cache (sink and recent
 * windows in BF16, history in INT2, page_table row b covering positions < L0)
 * and brings chunk rows cu_q[b] .. cu_q[b+1] (positions L0, L0+1, ...).  For
 * every chunk query i and query head h (KV head h/(Hq/Hkv)):
 *   out = softmax over { the prefix as stored: logit q·k/√d against BF16 keys,
 *         (q·R_K)·k̂/√d against INT2 keys } ∪ { the chunk's own keys at
 *         positions L0 .. L0+i, at bf16 } of the values, the INT2 values
 *         mapped back by R_Vᵀ.
 * The chunk's keys and values are not written to the cache by this call;
 * append them with oscar_quantize_append afterwards.
 * Arguments (device unless marked):
 *  q            [total_q][Hq][d] in cfg->q_dtype
 *  k, v         [total_q][Hkv][d] in cfg->kv_dtype (the chunk's own keys / values)
 *  total_q      host: rows of q, k, v
 *  cu_q         int32 [batch+1], cu_q[0] = 0, non-decreasing, cu_q[batch] = total_q
 *  start_pos    int32 [batch] prefix length L0 (0 <= L0 <= pt_stride)
 *  req_idx      int32 [batch] window row, or NULL for b
 *  page_table   int32 [batch][pt_stride]
 *  batch        host, 0..4096; max_chunk host, the largest cu_q[b+1] - cu_q[b]
 *  out          fp32 [total_q][Hq][d]
 *  workspace    device, >= oscar_prefill_workspace_bytes(cfg, batch, total_q), 256-byte aligned
 * Invalid prefix lengths or rows set OSCAR_DEV_BAD_LEN / _BAD_REQ and attend
 * over the chunk alone; out-of-pool slots set OSCAR_DEV_BAD_SLOT and are skipped. */
int oscar_prefill_attention(const oscar_config* cfg, const oscar_layer_cache* cache, const void* q,
                            const void* k, const void* v, int64_t total_q, const int32_t* cu_q,
                            const int32_t* start_pos, const int32_t* req_idx, const int32_t* page_table,
                            int64_t pt_stride, int32_t batch, int32_t max_chunk, float* out,
                            void* workspace, size_t workspace_bytes, void* stream);

/* ---- kernel timing (benchmarks) ----------------------------------------- */

/* Event timing of the kernels: `enable` is a bit mask of kinds (bit k times
 * kind k; 0 disables) and earlier records are forgotten.  Kinds: 0 the
 * history kernel, 4 the window kernel (which also prepares the rotated
 * queries) and 5 the combine kernel of oscar_decode_attention; 1 the quantise
 * kernel (for appends of at most W tokens it also writes the window rows) and
 * 2 the window-copy kernel (larger appends) of oscar_quantize_append; 6 the
 * attention kernel of oscar_prefill_attention; 7 the first launch of
 * oscar_decode_step (append, query preparation and window tiles; its history
 * kernel and combine are kinds 0 and 5).  Kind 3 is reserved and never
 * recorded.  A timed launch gets a CUDA event pair on
 * the call's stream (two cudaEventRecord, which also separate it from its
 * neighbours). */
int oscar_profile_enable(int32_t enable);

/* Waits for the recorded events of `kind` and returns their summed duration
 * in milliseconds and the number of timed launches (host outputs). */
int oscar_profile_read(int32_t kind, double* total_ms, int64_t* launches);

/* ---- device status ------------------------------------------------------ */

/* Waits for the current device, reads the OR of OSCAR_DEV_* bits set by the
 * kernels since the last clear into *flags (host), and clears the word if
 * `clear` is non-zero.  Returns OSCAR_ERR_CUDA if the device cannot be read. */
int oscar_device_status(int32_t* flags, int32_t clear);

/* Self-test of the bounded pipeline wait that the kernels use on their
 * mbarriers.  One warp waits for phase 0 of a shared-memory mbarrier for at
 * most `budget_cycles` SM clock cycles (clamped to [1,000, 4e9]).  With
 * `complete` = 0 nothing ever arrives, so the wait runs out: it sets
 * OSCAR_DEV_TIMEOUT in the device status word and the kernel returns, leaving
 * the context usable.  With `complete` = 1 the barrier is completed first and
 * no bit is set.  Asynchronous on `stream`; read the result with
 * oscar_device_status. */
int oscar_selftest_bounded_wait(int64_t budget_cycles, int32_t complete, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* OSCAR_H */
