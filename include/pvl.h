/*
 * pvl.h — packed variable-length masked attention for GB300 (sm_103a).
 *
 * C ABI of libpvl.so.  Several variable-length episodes share one [B, L]
 * token grid, either zero-padded to a common frame count (one episode per
 * batch row) or concatenated along the sequence axis; every token carries a
 * seq_id, and query i may attend key j iff seq_id[i] == seq_id[j] >= 0.
 * Sources: "lingbot_va_packing" §2.1 (pad-collate, valid_frames, seq_id -1
 * for padding frames in FlexAttnFunc.init_mask), "furniture_packing_variable_
 * length" (seq_id -1 keeps padding out of attention on the query and key side
 * and blocks leaks between episodes), "lingbot_va_attn_profiling" (packing
 * proposal: per-token document id and the mask condition doc_id[q] ==
 * doc_id[k]).
 *
 * Conventions for every call:
 *  - Tensors are dense and contiguous.  Q, K, V, O, dO, dQ, dK, dV are bf16
 *    [B, L, H, D] (D fastest).  LSE is fp32 [B, H, L].  seq_id is int32 [B, L].
 *  - Pointers marked "dev" are device pointers of the current CUDA device;
 *    "host" pointers are ordinary host memory read before the call returns.
 *  - The caller owns and allocates every buffer and the stream.  The library
 *    allocates no device memory at run time.  Its static device globals, held
 *    by every GPU that loads it until the process exits, are: a 16-byte error
 *    record, the PVL_NO_ALLOC_SCRATCH_BYTES scratch array of
 *    masked_attn_bwd_no_alloc, 256 32-bit work-item counters of the forward
 *    (one per (device, stream) in use; when all are taken the forward shares
 *    its items out in fixed turns instead), and two 32-bit result words of
 *    pvl_selftest_wait_timeout.  Calls are asynchronous on `stream` (NULL =
 *    legacy default stream) and return after enqueueing.
 *  - Arguments are validated on the host before anything is launched; a
 *    failed check returns a status and launches nothing.  Device-side
 *    failures (a bounded wait that ran out, a tile map built for another
 *    shape) are recorded in the device error record and surface through
 *    pvl_device_error().  No kernel traps or spins without bound.
 *  - pvl_last_error_message() describes the most recent non-OK status of the
 *    calling thread.
 */
#ifndef PVL_H_
#define PVL_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define PVL_API __attribute__((visibility("default")))
#else
#define PVL_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum pvl_status {
  PVL_OK = 0,
  PVL_ERR_INVALID_ARG = 1, /* null pointer, negative size, inconsistent table, short workspace */
  PVL_ERR_UNSUPPORTED = 2, /* valid but outside what the kernels implement (D, alignment, limits) */
  PVL_ERR_CUDA = 3,        /* a CUDA runtime/driver call failed (launch, attribute, tensor map) */
  PVL_ERR_TIMEOUT = 4      /* a device-side bounded wait ran out (reported by pvl_device_error) */
} pvl_status;

/* Same type as cudaStream_t / CUstream. */
typedef struct CUstream_st* pvl_stream_t;

/* Raw bfloat16 bits. */
typedef uint16_t pvl_bf16;

/* Limits (UNSUPPORTED beyond them). */
#define PVL_MAX_SEGMENTS 2048     /* B * K of pack_build_seq_ids */
#define PVL_MAX_L (1 << 19)       /* sequence length */
#define PVL_MAX_ORDER_TILES 16384 /* B * ceil(L / block) of tile_map_build */

/* ------------------------------------------------------------------------
 * pack_build_seq_ids — per-token episode id from a segment table.
 * Defines: "lingbot_va_packing" §2.1 (seq_id of frames >= valid_frames[b]
 * becomes -1) and "lingbot_va_attn_profiling" (per-token document id of
 * concatenated episodes).
 *
 * seg_frames, seg_valid: host int32 [B * K], row-major [B][K].  Row b holds K
 *   segments laid end to end; segment k spans seg_frames[b,k] frames of
 *   tokens_per_frame tokens, of which the first seg_valid[b,k] frames are real.
 * seq_id: dev int32 [B * L], written completely: id b*K + k on the real
 *   frames of segment k, -1 on padding frames and past the last segment.
 * Errors: INVALID_ARG for null pointers, B/K/L/tokens_per_frame < 1, any
 *   negative entry, seg_valid > seg_frames, or a row needing more than L
 *   tokens; UNSUPPORTED for B*K > PVL_MAX_SEGMENTS or L > PVL_MAX_L.
 * ---------------------------------------------------------------------- */
PVL_API pvl_status pack_build_seq_ids(const int32_t* seg_frames, const int32_t* seg_valid, int B, int K,
                              int tokens_per_frame, int L, int32_t* seq_id, pvl_stream_t stream);

/* ------------------------------------------------------------------------
 * Tile map — which (query tile, key tile) pairs can hold an admissible pair.
 * Defines: "lingbot_va_packing" §2.1-§2.2 (FlexAttention block mask built from
 * the seq_ids; the same mask must be seen by forward and backward, so here it
 * is an explicit argument of both instead of hidden state).
 *
 * Rule.  A position p < L with seq_id >= 0 is valid.  Per tile: nv = number
 * of valid positions, lo/hi = min/max id over them.  A pair is EMPTY (0) if
 * either nv is 0 or the id ranges do not overlap, FULL (2) if both tiles are
 * wholly valid and carry one and the same id, PARTIAL (1) otherwise.  EMPTY
 * pairs hold no admissible pair; FULL pairs hold only admissible pairs.
 *
 * Workspace (dev, caller-allocated, tile_map_ws_bytes() bytes, 256-byte
 * aligned) holds, at the byte offsets tile_map_layout() returns:
 *   HEADER      int32[16]  magic, version, B, Lq, block_m, block_n, nTq, nTk, Lk
 *   Q_NV/LO/HI  int32[B*nTq]      K_NV/LO/HI int32[B*nTk]
 *   CLS         uint8[B*nTq*nTk]  class of (b, qt, kt)
 *   ROW_COUNT   int32[B*nTq]  non-empty key tiles per query tile
 *   ROW_FULL    int32[B*nTq]  how many of them are FULL
 *   ROW_LIST    int32[B*nTq*nTk]  their indices: FULL first, then PARTIAL,
 *                              each ascending; unused slots -1
 *   COL_COUNT/COL_FULL int32[B*nTk], COL_LIST int32[B*nTk*nTq]: the same per
 *                              key tile over query tiles
 *   Q_ORDER     int32[B*nTq]  b*nTq+qt sorted by descending ROW_COUNT, ties
 *                              by ascending index (longest work first)
 *   K_ORDER     int32[B*nTk]  the same over key tiles by COL_COUNT
 * nTq = ceil(Lq / block_m), nTk = ceil(Lk / block_n); Lq = Lk = L for the
 * self-attention map of tile_map_build.
 *
 * The workspace holds PVL_TM_LEVELS such maps built from the same seq_ids:
 * level 0 at (block_m, block_n) and level 1 at (2*block_m, block_n), whose
 * query tiles are pairs of level-0 query tiles (the forward processes a pair
 * of query tiles against one stream of key tiles).
 * ---------------------------------------------------------------------- */
enum {
  PVL_TM_HEADER = 0,
  PVL_TM_Q_NV, PVL_TM_Q_LO, PVL_TM_Q_HI,
  PVL_TM_K_NV, PVL_TM_K_LO, PVL_TM_K_HI,
  PVL_TM_CLS,
  PVL_TM_ROW_COUNT, PVL_TM_ROW_FULL, PVL_TM_ROW_LIST,
  PVL_TM_COL_COUNT, PVL_TM_COL_FULL, PVL_TM_COL_LIST,
  PVL_TM_Q_ORDER, PVL_TM_K_ORDER,
  PVL_TM_NFIELDS
};
#define PVL_TM_LEVELS 2

/* Bytes of workspace for tile_map_build (both levels); 0 if the arguments
 * are invalid. */
PVL_API size_t tile_map_ws_bytes(int B, int L, int block_m, int block_n);

/* Byte offsets of the arrays inside the workspace (host call, no device
 * work).  offsets: host size_t[PVL_TM_LEVELS * PVL_TM_NFIELDS]; entry
 * level * PVL_TM_NFIELDS + field. */
PVL_API pvl_status tile_map_layout(int B, int L, int block_m, int block_n, size_t* offsets);

/* seq_id: dev int32 [B * L].  block_m, block_n in 1..1024 (the attention
 * calls need 128 and 128).  tile_ws: dev, ws_bytes >= tile_map_ws_bytes().
 * Errors: INVALID_ARG for null pointers, sizes < 1, a short or misaligned
 * workspace; UNSUPPORTED for L > PVL_MAX_L or B*nT > PVL_MAX_ORDER_TILES. */
PVL_API pvl_status tile_map_build(const int32_t* seq_id, int B, int L, int block_m, int block_n, void* tile_ws,
                          size_t ws_bytes, pvl_stream_t stream);

/* Cross-attention tile map ("lingbot_va_packing" §2.1: the latent and the
 * action tokens carry their own seq_ids, both dropping invalid frames from
 * the self and cross attention masks): query tiles over q_seq_id (dev int32
 * [B * Lq]), key tiles over k_seq_id (dev int32 [B * Lk]); the pair rule,
 * lists, orders and errors are those of tile_map_build, with "valid" read on
 * each side over its own ids and length.  tile_map_build(seq_id, B, L, ...)
 * is tile_map_build_cross(seq_id, seq_id, B, L, L, ...). */
PVL_API size_t tile_map_ws_bytes_cross(int B, int Lq, int Lk, int block_m, int block_n);
PVL_API pvl_status tile_map_layout_cross(int B, int Lq, int Lk, int block_m, int block_n, size_t* offsets);
PVL_API pvl_status tile_map_build_cross(const int32_t* q_seq_id, const int32_t* k_seq_id, int B, int Lq, int Lk,
                                        int block_m, int block_n, void* tile_ws, size_t ws_bytes,
                                        pvl_stream_t stream);

/* ------------------------------------------------------------------------
 * masked_attn_fwd — O = softmax(scale * Q K^T restricted to admissible keys) V.
 * Defines: "furniture_packing_variable_length" (attention masking by seq_id)
 * and "lingbot_va_attn_profiling" (FlexAttention forward, doc_id mask).
 *
 * q, k, v: dev bf16 [B, L, H, D], 16-byte aligned.  seq_id: dev int32 [B, L].
 * tile_ws: a tile map built from this seq_id with block_m = block_n = 128.
 * D in {64, 128}; H >= 1; scale > 0 (1/sqrt(D) is the usual choice).
 * o: dev bf16 [B, L, H, D].  lse: dev fp32 [B, H, L], natural-log
 *   log-sum-exp of the admissible scaled scores.
 * Rows with no admissible key (seq_id -1) get O = 0 exactly and LSE = -inf.
 * Errors: INVALID_ARG for null pointers or sizes < 1; UNSUPPORTED for other
 *   D, misaligned pointers or L > PVL_MAX_L; CUDA for launch failures.  A
 *   tile map of another shape is detected on the device (INVALID_ARG from
 *   pvl_device_error, outputs untouched).
 * ---------------------------------------------------------------------- */
PVL_API pvl_status masked_attn_fwd(const pvl_bf16* q, const pvl_bf16* k, const pvl_bf16* v, const int32_t* seq_id,
                           const void* tile_ws, int B, int L, int H, int D, float scale, pvl_bf16* o,
                           float* lse, pvl_stream_t stream);

/* Cross attention: q dev bf16 [B, Lq, H, D] with ids q_seq_id [B, Lq]; k, v
 * dev bf16 [B, Lk, H, D] with ids k_seq_id [B, Lk]; query i attends key j iff
 * q_seq_id[i] == k_seq_id[j] >= 0.  tile_ws: tile_map_build_cross of these
 * ids at 128 x 128.  o: dev bf16 [B, Lq, H, D]; lse: dev fp32 [B, H, Lq].  A
 * query with no admissible key (seq_id -1, or an id no key carries) gets
 * O = 0 and LSE = -inf.  Errors as masked_attn_fwd, lengths checked each on
 * its side.  masked_attn_fwd is the case k_seq_id = seq_id, Lk = Lq = L. */
PVL_API pvl_status masked_attn_fwd_cross(const pvl_bf16* q, const pvl_bf16* k, const pvl_bf16* v,
                                         const int32_t* q_seq_id, const int32_t* k_seq_id, const void* tile_ws,
                                         int B, int Lq, int Lk, int H, int D, float scale, pvl_bf16* o, float* lse,
                                         pvl_stream_t stream);

/* ------------------------------------------------------------------------
 * masked_attn_bwd — gradients of the masked attention from the saved LSE.
 * Defines: the backward of the FlexAttention template the pages run
 * ("lingbot_va_attn_profiling", kernel table); P is recomputed from LSE and
 * the score matrix is never stored.
 *   Delta_i = <dO_i, O_i>,  dS = P * (dO V^T - Delta),
 *   dQ = scale dS K,  dK = scale dS^T Q,  dV = P^T dO.
 *
 * q, k, v, o, dO: dev bf16 [B, L, H, D] (o as written by masked_attn_fwd);
 * lse: dev fp32 [B, H, L] from masked_attn_fwd; seq_id, tile_ws as for the
 * forward.  dq, dk, dv: dev bf16 [B, L, H, D], fully written; rows with
 * seq_id -1 get exact zeros.
 * ws: dev scratch of masked_attn_bwd_ws_bytes(B, L, H, D) bytes, 256-byte
 *   aligned (fp32 dQ accumulator; Delta, LSE*log2(e) and query seq_ids padded
 *   to whole 128-row tiles; the counter that hands out work items); contents
 *   on entry are ignored.  A workspace serves one call at a time.
 * Errors: as masked_attn_fwd, plus INVALID_ARG for a short workspace.
 * ---------------------------------------------------------------------- */
PVL_API size_t masked_attn_bwd_ws_bytes(int B, int L, int H, int D);

PVL_API pvl_status masked_attn_bwd(const pvl_bf16* q, const pvl_bf16* k, const pvl_bf16* v, const pvl_bf16* o,
                           const pvl_bf16* dO, const float* lse, const int32_t* seq_id, const void* tile_ws,
                           int B, int L, int H, int D, float scale, pvl_bf16* dq, pvl_bf16* dk, pvl_bf16* dv,
                           void* ws, size_t ws_bytes, pvl_stream_t stream);

/* Cross attention backward: q, o, dO, dq [B, Lq, H, D] and lse [B, H, Lq]
 * on the query side, k, v, dk, dv [B, Lk, H, D] on the key side, ids and
 * tile map as for masked_attn_fwd_cross.  Keys with seq_id -1 or an id no
 * query carries get dK = dV = 0; queries without an admissible key get
 * dQ = 0.  ws: masked_attn_bwd_ws_bytes_cross(B, Lq, Lk, H, D) bytes (the
 * query-side arrays of masked_attn_bwd's workspace, over Lq). */
PVL_API size_t masked_attn_bwd_ws_bytes_cross(int B, int Lq, int Lk, int H, int D);

PVL_API pvl_status masked_attn_bwd_cross(const pvl_bf16* q, const pvl_bf16* k, const pvl_bf16* v, const pvl_bf16* o,
                                         const pvl_bf16* dO, const float* lse, const int32_t* q_seq_id,
                                         const int32_t* k_seq_id, const void* tile_ws, int B, int Lq, int Lk, int H,
                                         int D, float scale, pvl_bf16* dq, pvl_bf16* dk, pvl_bf16* dv, void* ws,
                                         size_t ws_bytes, pvl_stream_t stream);

/* ------------------------------------------------------------------------
 * masked_attn_bwd_no_alloc — masked_attn_bwd for callers that cannot
 * allocate device memory.  The pages have no counterpart: this entry point
 * exists for the caller, not for the method.
 *
 * Some callers are handed only their input and output buffers and may not
 * call cudaMalloc: a plug-in inside a framework that has reserved the whole
 * device memory pool for its own allocator, or a latency-bound loop where an
 * allocation (which can synchronise the device) is not allowed.  This call
 * computes exactly what masked_attn_bwd computes, with the same arguments
 * minus the workspace: its scratch (fp32 dQ accumulator and Delta) lives in
 * one static device array of PVL_NO_ALLOC_SCRATCH_BYTES inside the library,
 * which every GPU that loads the library holds until the process exits.  It
 * calls no allocating routine.
 *
 * Limit: masked_attn_bwd_ws_bytes(B, L, H, D) (about B*L*H*(D+2)*4 bytes)
 *   must not exceed PVL_NO_ALLOC_SCRATCH_BYTES; larger shapes return
 *   PVL_ERR_UNSUPPORTED without launching anything.
 * Set-up: the first call on a device looks up the array's device address
 *   (cudaGetSymbolAddress) with that device current; make that first call
 *   before any stream capture.  The address is kept for the rest of the
 *   process: it assumes the device keeps one CUDA context (the runtime's
 *   primary context) for the life of the process; after a cudaDeviceReset
 *   the kept address is stale and this call must not be used again.  The
 *   error record that every call uses is located the same way.
 * Sharing: all calls on a device use the same array.  Each call clears what
 *   must start at zero, so earlier contents do not matter, but calls whose
 *   work overlaps on the GPU (other streams, other threads) race on the
 *   scratch and give wrong gradients: serialise them.
 * Errors: as masked_attn_bwd.
 * ---------------------------------------------------------------------- */
#define PVL_NO_ALLOC_SCRATCH_BYTES (32u << 20) /* 32 MiB */

PVL_API pvl_status masked_attn_bwd_no_alloc(const pvl_bf16* q, const pvl_bf16* k, const pvl_bf16* v,
                                            const pvl_bf16* o, const pvl_bf16* dO, const float* lse,
                                            const int32_t* seq_id, const void* tile_ws, int B, int L, int H, int D,
                                            float scale, pvl_bf16* dq, pvl_bf16* dk, pvl_bf16* dv,
                                            pvl_stream_t stream);

/* ------------------------------------------------------------------------
 * adaln_fwd / adaln_bwd — layer norm over the feature dimension followed by
 * the AdaLN modulation, fused ("AdaptiveLoad" §2.B, the fused
 * LayerNorm-Modulate kernel of a DiT / MMDiT block; the page gives no
 * formulas, the plain reading is the adaptive layer norm of DiT):
 *   mu = mean_d x,  r = 1 / sqrt(mean_d (x - mu)^2 + eps),
 *   y = (x - mu) r (1 + scale_b) + shift_b           (no affine of its own)
 *   backward, g = dy (1 + scale_b), xh = (x - mu) r:
 *   dx = r (g - mean_d g - xh mean_d(g xh)),
 *   dshift_b = sum_n dy,  dscale_b = sum_n dy xh.
 *
 * x, y, dy, dx: dev bf16 [B, N, D]; shift, scale, dshift, dscale: dev fp32
 * [B, D] (one modulation vector per batch row, shared by its N tokens).
 * D a multiple of 8, at most 8192; eps >= 0 (1e-6 is the usual choice).
 * mean, rstd: optional (null allowed) dev fp32 [B, N] row statistics the
 * forward can write; the backward recomputes them from x and needs neither.
 * adaln_bwd ws: dev scratch of adaln_bwd_ws_bytes(B, N, D) bytes (partial
 * sums of dshift / dscale, one per (CTA, batch row): 2 * (min(B N, 2048) +
 * B - 1) * D fp32); contents on entry are ignored.  The partials are added
 * in a fixed order: repeated calls on one GPU give the same bits.
 * All pointers 16-byte aligned (mean / rstd 4-byte).  Errors: INVALID_ARG
 * for null pointers, sizes < 1, a negative eps or a short workspace;
 * UNSUPPORTED for other D or misaligned pointers; CUDA for launch failures;
 * a device-side bounded wait that runs out surfaces through pvl_device_error.
 * ---------------------------------------------------------------------- */
PVL_API pvl_status adaln_fwd(const pvl_bf16* x, const float* shift, const float* scale, int B, int N, int D,
                             float eps, pvl_bf16* y, float* mean, float* rstd, pvl_stream_t stream);

PVL_API size_t adaln_bwd_ws_bytes(int B, int N, int D);

PVL_API pvl_status adaln_bwd(const pvl_bf16* x, const float* scale, const pvl_bf16* dy, int B, int N, int D,
                             float eps, pvl_bf16* dx, float* dshift, float* dscale, void* ws, size_t ws_bytes,
                             pvl_stream_t stream);

/* ------------------------------------------------------------------------
 * masked_mse_loss / masked_mse_loss_bwd — the squared-error loss averaged
 * over valid frames only, and its gradient ("lingbot_va_packing" §2.1,
 * compute_loss: frame_valid = f < valid_frames[b], latent and action
 * losses averaged over the valid frames; "furniture_packing_variable_length",
 * the loss paragraph).  Per stream (latent or action tokens):
 *   valid token  = seq_id >= 0 (the attention's mask; on pad-collated rows
 *                  it is frame_valid spread over the frame's tokens)
 *   loss         = sum_{valid} sum_c (pred - target)^2 / (C n_valid)
 *   grad         = dloss 2 (pred - target) / (C n_valid) on valid tokens,
 *                  0 on the others; loss = 0 and grad = 0 if n_valid = 0.
 *
 * pred, target, grad: dev bf16 [B, L, C] (token-major, C fastest); seq_id:
 * dev int32 [B, L]; loss: dev fp32 [1].  C a multiple of 8; B * L < 2^31.
 * masked_mse_loss writes the loss and, when grad is not null, the gradient
 * scaled by the host value grad_scale in the same pass (the fused form for
 * a loss that is the objective: grad_scale = its weight).
 * masked_mse_loss_bwd writes only the gradient, scaled by the device value
 * dloss[0] (the autograd form).  Padding tokens' pred and target are never
 * read.  One cooperative launch (with the gradient, its CTAs meet at a
 * bounded grid barrier once the valid tokens are counted).  ws: dev scratch of
 * masked_mse_ws_bytes(B, L, C) bytes, contents on entry ignored, one per
 * call in flight.  The loss is deterministic for a
 * given GPU model (fixed grid, fixed summation order).  pred, target,
 * seq_id, grad, ws 16-byte aligned; loss, dloss 4-byte.  Errors:
 * INVALID_ARG for null pointers, sizes < 1, a non-finite grad_scale or a
 * short workspace; UNSUPPORTED for other C, sizes or alignment; CUDA for
 * launch failures.
 * ---------------------------------------------------------------------- */
PVL_API size_t masked_mse_ws_bytes(int B, int L, int C);

PVL_API pvl_status masked_mse_loss(const pvl_bf16* pred, const pvl_bf16* target, const int32_t* seq_id, int B, int L,
                                   int C, float* loss, pvl_bf16* grad, float grad_scale, void* ws, size_t ws_bytes,
                                   pvl_stream_t stream);

PVL_API pvl_status masked_mse_loss_bwd(const pvl_bf16* pred, const pvl_bf16* target, const int32_t* seq_id, int B,
                                       int L, int C, const float* dloss, pvl_bf16* grad, void* ws, size_t ws_bytes,
                                       pvl_stream_t stream);

/* ------------------------------------------------------------------------
 * Device error record.  Synchronises `stream`, reads and clears the current
 * device's error record.  Returns PVL_OK, PVL_ERR_TIMEOUT (a bounded wait ran
 * out; the kernel released its resources and returned), PVL_ERR_INVALID_ARG
 * (tile map of another shape) or PVL_ERR_CUDA (the synchronisation failed).
 * info (optional, host int32[4]): code, where, block, thread of the first
 * failure.
 * ---------------------------------------------------------------------- */
PVL_API pvl_status pvl_device_error(pvl_stream_t stream);
PVL_API pvl_status pvl_device_error_detail(pvl_stream_t stream, int32_t* info);

/* pvl_selftest_wait_timeout — exercises the bounded waits every kernel uses,
 * without a fault: one CTA in which warp 0 waits short_ns on an mbarrier
 * that nothing arrives on (and records a timeout) while warp 1 waits up to
 * long_ns on another and leaves through the CTA's abort flag.  Synchronises
 * `stream`; out (host int32[2]) receives each warp's wait result (1 = the
 * barrier completed, 0 = gave up: both 0 when the path works).  The timeout
 * itself is then read with pvl_device_error (PVL_ERR_TIMEOUT, site 91).
 * Errors: INVALID_ARG for a null out or limits outside 0 < short_ns <=
 * long_ns, short_ns <= 10 s, long_ns <= 60 s; CUDA for launch failures. */
PVL_API pvl_status pvl_selftest_wait_timeout(uint64_t short_ns, uint64_t long_ns, int32_t* out, pvl_stream_t stream);

/* pvl_set_attn_wait_timeout_ns — the bound on any single device-side wait of
 * the attention kernels (masked_attn_fwd*, masked_attn_bwd*) launched after
 * this call, process-wide.  ns = 0 restores the default of 2 s; at most 60 s.
 * A wait that runs out records PVL_ERR_TIMEOUT (read by pvl_device_error)
 * and the kernel leaves through its abort path: every role stops, copies
 * and MMAs in flight are drained, tensor memory is released and the kernel
 * returns, so the context stays usable.  The outputs of such a call are
 * undefined.  A bound far below the time a tile load takes (a few
 * nanoseconds) makes the kernels' first waits run out: this is how the
 * abort path is tested on a working GPU.  Errors: INVALID_ARG above 60 s. */
PVL_API pvl_status pvl_set_attn_wait_timeout_ns(uint64_t ns);

/* pvl_mark_next_bwd_main — for measurement: `before` and `after` (cudaEvent_t
 * handles, created by the caller) are recorded on the call's stream just
 * before and just after the launch of the main backward kernel of the calling
 * thread's next masked_attn_bwd, masked_attn_bwd_cross or
 * masked_attn_bwd_no_alloc call (the Delta / dQ-accumulator preprocess and
 * the dQ conversion launches stay outside the pair), so that the main kernel
 * can be timed alone.  One-shot: that call consumes and clears both; either
 * may be null; null / null clears a pending pair.  Always PVL_OK. */
PVL_API pvl_status pvl_mark_next_bwd_main(void* before, void* after);

/* Human-readable text of the calling thread's last non-OK status. */
PVL_API const char* pvl_last_error_message(void);

/* Library version, e.g. 0x000100 for 0.1.0. */
PVL_API int pvl_version(void);

#ifdef __cplusplus
}
#endif

#endif /* PVL_H_ */
