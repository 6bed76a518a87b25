/*
 * attn.h — C ABI of the GB300 (sm_103a) fused RoPE + causal attention forward.
 *
 * One operation: the prefill attention forward of a decoder layer,
 *
 *   O = softmax(mask(RoPE(Q) RoPE(K)^T / sqrt(D))) V,   LSE_i = m_i + ln l_i,
 *
 * with RoPE applied to Q and K pair by pair as their tiles are loaded
 * ("AttnFuse: A Composable DSL for Compiling Attentions to Fused GPU Kernels",
 * sec. 4.1 Fused RoPE), the causal mask applied before the softmax, an exp2
 * online softmax with scale log2(e)/sqrt(D) ("Flash Attention: Causal Prefill
 * D=128", Online softmax: what must remain invariant), P.V accumulated in fp32
 * with P rounded to bf16, and one LSE value per query row ("AttnFuse", sec. 4.4
 * Backward Pass: the forward keeps L = m + log l).  An optional per-RoPE-pair
 * distance window drops pair r's QK terms beyond w_r = k * 2*pi/theta_r
 * ("ATFlash — Per-RoPE-Wavelength Attention Windows", The idea).
 *
 * Conventions shared by every entry point:
 *   - Tensors are BSHD: q and o are [B][S][Hq][D], k and v are [B][S][Hkv][D],
 *     contiguous, bfloat16, device pointers, 16-byte aligned.
 *   - lse is float32 [B][Hq][S] (natural log), device pointer, or NULL.
 *   - Query head h reads KV head h / (Hq / Hkv) (grouped-query attention).
 *   - RoPE pairs dimension r with r + D/2 (NeoX half split), theta_r =
 *     base^(-2r/D), positions 0..S-1 for both Q and K.
 *   - The caller owns every buffer it passes.  The library owns only cached
 *     device tables (cos/sin, tile schedules) that it builds on the first call
 *     for a given shape and frees in attn_release_cache().
 *   - stream is a cudaStream_t passed as void*; NULL is the legacy default
 *     stream.  attn_fwd is asynchronous on that stream.
 *   - Return values are attn_status codes; attn_error_string() names them.
 */
#ifndef ATTN_H_
#define ATTN_H_

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    ATTN_OK = 0,
    ATTN_ERR_NULL = -1,        /* a required pointer is NULL */
    ATTN_ERR_SHAPE = -2,       /* B, S, H or D out of range, or Hq not a multiple of Hkv */
    ATTN_ERR_ALIGN = -3,       /* a tensor pointer is not 16-byte aligned */
    ATTN_ERR_UNSUPPORTED = -4, /* a combination the kernel does not implement */
    ATTN_ERR_CUDA = -5,        /* a CUDA runtime or driver call failed */
    ATTN_ERR_TIMEOUT = -6,     /* a bounded in-kernel wait ran out (see attn_check) */
    ATTN_ERR_OOM = -7,         /* the library could not allocate its cached tables */
    ATTN_ERR_NO_DEVICE = -8,   /* no sm_103 device is current */
    ATTN_ERR_SCRATCH = -9,     /* attn_fwd_noalloc: tables exceed its static scratch */
    ATTN_ERR_NONFINITE = -10   /* a forward row's result was not finite (see attn_check) */
} attn_status;

/*
 * attn_fwd — fused RoPE + causal attention forward (prefill).
 *
 *   q, k, v     bf16 device tensors, BSHD, see above.
 *   o           bf16 device output [B][S][Hq][D]; rows are O_i / l_i rounded to bf16.
 *   lse         float32 device output [B][Hq][S], ln(sum_j exp(s_ij)) over the
 *               kept keys, or NULL to skip it.
 *   B, S        batch and sequence length, 1 <= B <= 65535, 1 <= S <= 2^22.
 *   Hq, Hkv     query and key/value heads, 1 <= Hkv <= Hq <= 255, Hq % Hkv == 0.
 *   D           head dimension, 64 or 128.
 *   causal      1: key j is excluded for query i when j > i; 0: full attention.
 *   rope_base   theta base (e.g. 10000, 500000); <= 0 turns RoPE off.
 *   window_k    per-pair window multiplier k > 0 (pair r keeps distances
 *               i - j <= floor(k * 2*pi / theta_r)); <= 0 or +inf turns it off.
 *               The window needs RoPE on and causal = 1, else ATTN_ERR_UNSUPPORTED.
 *   stream      cudaStream_t (as void*).
 *
 * Returns ATTN_OK once the kernel is enqueued.  Argument errors are found on
 * the host before anything is launched.  The first call for a new (device,
 * S, D, rope_base, window_k, B, Hq, Hkv) builds and uploads tables
 * synchronously; later calls only launch.  Precision: with RoPE on, the
 * rotated Q and K are rounded to fp16 for the QK^T product (inputs must keep
 * |x| < 46000 so the rotated values stay finite: a rotation keeps each pair's
 * norm, and sqrt(2) * 46000 < 65504); with RoPE off, Q and K go to the tensor
 * cores as the given bf16 values.  A row whose LSE comes out non-finite (an
 * input past that bound or not finite) raises a bit in the device status
 * word, and the next attn_check reports ATTN_ERR_NONFINITE.
 */
int attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
             int B, int Hq, int Hkv, int S, int D, int causal,
             double rope_base, double window_k, void* stream);

/*
 * attn_fwd_noalloc — attn_fwd for callers that must not allocate device memory.
 *
 * The source pages have no counterpart to this entry point.  It exists for
 * callers that cannot call cudaMalloc: code running where an allocation would
 * break a memory budget fixed up front, allocators that own every device byte
 * (a framework's caching allocator, an inference server's arena), or code that
 * must not add allocator traffic to a hot loop.
 *
 * Arguments, results and precision are those of attn_fwd.  Instead of cached
 * cudaMalloc'd buffers, the RoPE factor tables (about (S/128 + 17) * D * 4
 * bytes) and the tile schedule (8 bytes per work unit of up to 256 query rows)
 * live in one 16 MiB array in device global memory that is part of the
 * library: every GPU that loads libattn.so holds those 16 MiB until the
 * process exits.  The call allocates no device memory and calls no
 * allocating CUDA or PyTorch routine.
 *   - Limit: tables plus schedule must fit in 16 MiB, about two million work
 *     units (B * Hq * S up to roughly 5e8); larger requests return
 *     ATTN_ERR_SCRATCH before anything is enqueued.  The window must be off.
 *   - The first call on a device looks up the array's device address
 *     (cudaGetSymbolAddress, with that device current) and creates one event
 *     (no device memory); make that first call before any stream capture.
 *   - The array keeps the last call's contents.  A call whose shape, RoPE base
 *     and causal flag differ from the previous call on the device re-uploads
 *     the tables with cudaMemcpyAsync on `stream` (from pageable host memory,
 *     so the host waits for the staging) and records the event there;
 *     otherwise it only launches.  A call of the same shape on another stream
 *     waits for that event (cudaStreamWaitEvent) until the upload has been
 *     seen complete, so it never reads tables still in flight.
 *   - While `stream` is being captured, a call that would upload, or that
 *     would have to wait for an upload enqueued on another stream, returns
 *     ATTN_ERR_UNSUPPORTED and enqueues nothing.
 *   - All calls share the one array: a call whose shape or options differ
 *     overwrites the tables that a call still running on another stream
 *     reads (a race).  Keep such calls on one stream, or synchronise between
 *     them.
 */
int attn_fwd_noalloc(const void* q, const void* k, const void* v, void* o, float* lse,
                     int B, int Hq, int Hkv, int S, int D, int causal,
                     double rope_base, double window_k, void* stream);

/*
 * attn_fwd_host — attn_fwd with host buffers: copies in, computes, copies out.
 *
 * The source pages have no counterpart to this entry point.  It is for callers
 * whose tensors live in host memory (a CPU-resident KV store, an offload
 * path, an end-to-end measurement): it overlaps the host-device transfers
 * with the compute instead of leaving them to run one after another.
 *
 *   q, k, v, o, lse  HOST pointers with the layouts of attn_fwd (lse may be
 *                    NULL).  Page-locked memory (cudaHostAlloc / pinned torch
 *                    tensors) lets the copies run asynchronously; pageable
 *                    memory works, with the copies then staged by the driver.
 *   other arguments  as attn_fwd; the device is the current one.
 *
 * The work is cut into chunks of one batch element and a group of KV heads
 * (with their query heads): about four chunks per call.  Two device staging
 * slots cycle through three library-owned streams: the next chunk's Q/K/V go
 * host-to-device while the current chunk runs through attn_fwd and the
 * previous chunk's O/LSE go device-to-host.  Each head's arithmetic is that
 * of attn_fwd, so the results are bitwise those of attn_fwd on the same data.
 *   - Synchronous: returns after every output is in host memory, with
 *     ATTN_ERR_TIMEOUT if a bounded in-kernel wait ran out (as attn_check).
 *   - The library keeps the staging slots (2 x the largest chunk's Q, K, V,
 *     O and LSE) and the streams until attn_release_cache().
 *   - One call at a time per device (calls are serialised by a lock).
 */
int attn_fwd_host(const void* q, const void* k, const void* v, void* o, float* lse,
                  int B, int Hq, int Hkv, int S, int D, int causal,
                  double rope_base, double window_k);

/*
 * attn_rope_rotate — RoPE applied to a whole BSHD tensor in one pass.
 *
 * The pre-rotation side of "AttnFuse: A Composable DSL for Compiling
 * Attentions to Fused GPU Kernels", sec. 5.3 The Rotation Calculus: rotate Q
 * and K once, in a memory-bound sweep, then run the attention without in-loop
 * rotation (attn_fwd_rotated), against attn_fwd's rotation of K tiles inside
 * the loop each time a query tile visits them.  Same pairing, angles and
 * positions (0..S-1) as attn_fwd.
 *   x          bf16 device tensor [B][S][H][D], 16-byte aligned.
 *   y          fp16 device output of the same shape (must not overlap x): the
 *              rotation in fp32, rounded to fp16 as attn_fwd rounds its rotated
 *              operands.  Angles are products of two factors computed in
 *              float64 (tile base and row offset), accurate to a few fp32 ulps.
 *   B, S, H, D as attn_fwd (H for the tensor's own heads); rope_base > 0.
 *   stream     cudaStream_t (as void*); asynchronous.
 * The first call for a (device, S, D, rope_base) builds and caches a factor
 * table of (S/128 + 128) * D * 4 bytes.
 */
int attn_rope_rotate(const void* x, void* y, int B, int S, int H, int D, double rope_base, void* stream);

/*
 * attn_fwd_rotated — the forward on Q and K rotated beforehand.
 *
 *   q_rot, k_rot   fp16 device tensors, BSHD, as written by attn_rope_rotate.
 *   v, o, lse, B, Hq, Hkv, S, D, causal, stream   as attn_fwd.
 * Runs attn_fwd's kernel without in-loop rotation, with QK^T on the fp16
 * operands (the window is not available here).  With attn_rope_rotate on Q
 * and K first, the result equals attn_fwd's with RoPE up to the rounding of
 * the angles (both paths round the rotated values to fp16).
 */
int attn_fwd_rotated(const void* q_rot, const void* k_rot, const void* v, void* o, float* lse,
                     int B, int Hq, int Hkv, int S, int D, int causal, void* stream);

/*
 * attn_decode — one decode step: each sequence's newest token against its KV cache.
 *
 * The query of each sequence sits at position S-1 and attends to keys
 * 0..S-1 (its own K/V are the cache's last rows), with the conventions of
 * attn_fwd: RoPE applied to q and to K as it is loaded, scale 1/sqrt(D),
 * bf16 output, natural-log LSE.  The key range is split across CTAs and the
 * partial results merge through their log-sum-exp ("AttnFuse: A Composable
 * DSL for Compiling Attentions to Fused GPU Kernels", sec. 4.2 Decode).
 * With window_k > 0 the per-RoPE-pair window of "ATFlash — Per-RoPE-Wavelength
 * Attention Windows" (decode) applies: pair r of key j is dropped when
 * S-1-j > W_r, and those K components are not loaded.
 *   q       bf16 device [B][Hq][D].
 *   k, v    bf16 device caches [B][S][Hkv][D] (K not rotated).
 *   o       bf16 device output [B][Hq][D];  lse float32 [B][Hq] or NULL.
 *   B, Hq, Hkv, S, D, rope_base, window_k   as attn_fwd; Hq / Hkv <= 32.
 * Decode reads each K/V byte once: it is bound by HBM bandwidth.  Q K^T and
 * P V run as warp-level mma.sync over 32-key tiles (rotated q and K rounded to
 * fp16, P to bf16, fp32 accumulation, as in attn_fwd); the number of splits
 * (multiples of 128 keys) is chosen for about one or two waves of resident
 * CTAs.  Asynchronous on `stream`; the library keeps a partial-result scratch
 * of B * Hq * splits * (D + 2) floats and a rotation-factor table of
 * (ceil(S/32) + 32) * D/2 (cos, sin) pairs per (S, D, rope_base) until
 * attn_release_cache().  Errors: as attn_fwd, and ATTN_ERR_UNSUPPORTED when
 * Hq / Hkv > 32.
 */
int attn_decode(const void* q, const void* k, const void* v, void* o, float* lse,
                int B, int Hq, int Hkv, int S, int D, double rope_base, double window_k, void* stream);

/*
 * attn_bwd — gradients of the attention forward: dQ, dK, dV for an upstream
 * gradient dO ("AttnFuse: A Composable DSL for Compiling Attentions to Fused
 * GPU Kernels", sec. 4.4 Backward Pass: a row-reduction kernel, a dK/dV
 * kernel and a dQ kernel, each writing its own output tiles, with the
 * probabilities re-derived from the forward's per-row LSE).
 *   q, k, v  bf16 device, the forward's inputs (BSHD, K and V not rotated).
 *   o, lse   the forward's outputs: o bf16 [B][S][Hq][D], lse float32
 *            [B][Hq][S] (natural log), both required.
 *   dO       bf16 device [B][S][Hq][D].
 *   dq       bf16 device output [B][S][Hq][D]; dk, dv bf16 [B][S][Hkv][D]
 *            (a KV head's gradients sum over its query heads).
 *   B, Hq, Hkv, S, D, causal, rope_base   as attn_fwd; the window is not
 *            supported here.
 * P is rounded to bf16 (for dV, and as the P of dS = P (dP - dO.O)); dS is
 * rounded to fp16 for the products with the rotated fp16 Q and K (bf16
 * without RoPE); accumulation in fp32.  With RoPE, Q and K are rotated once
 * by the rotation pass (as attn_rope_rotate) into library-owned fp16 buffers
 * before the tile kernels, which then rotate nothing inside their loops.
 * Asynchronous on `stream`.  The library keeps a scratch of B*Hq*S floats
 * (dO.O per row), with RoPE B*S*(Hq+Hkv)*D fp16 values (the rotated Q and
 * K), and the rotation tables until attn_release_cache().
 * Errors: as attn_fwd (ATTN_ERR_NULL also for dO, lse, dq, dk, dv).
 */
int attn_bwd(const void* q, const void* k, const void* v, const void* o, const void* dO, const float* lse,
             void* dq, void* dk, void* dv, int B, int Hq, int Hkv, int S, int D, int causal, double rope_base,
             void* stream);

/*
 * attn_fwd_blocksparse — the forward over a block-sparse mask ("AttnFuse: A
 * Composable DSL for Compiling Attentions to Fused GPU Kernels", sec. 4.3
 * Block-Sparse Attention: a CSR BlockMask lists each row's active key
 * blocks, and the kernel visits only those).
 *   Blocks are 128 x 128 (query tile x key tile), shared by every batch
 *   element and head: key j is visible to query i iff block (i/128, j/128) is
 *   listed, and j <= i when causal.
 *   row_ptr  host int32 [ceil(S/128) + 1], row_ptr[0] = 0, non-decreasing.
 *   col_idx  host int32 [row_ptr[last]]: each row's key tiles, strictly
 *            ascending, in [0, ceil(S/128)); with causal, at most the row.
 *   q, k, v, o, lse, B, Hq, Hkv, S, D, causal, rope_base   as attn_fwd (no
 *            window).  A query row that sees no key gets O = 0, LSE = -inf.
 * The library keeps a device copy of each distinct mask, and the task
 * schedule of each (mask, B * Hq) (see attn_mask_schedule), until
 * attn_release_cache(); the first call with a new mask or shape uploads them
 * synchronously.  Asynchronous on `stream` after that.
 * Errors: as attn_fwd; ATTN_ERR_SHAPE for a malformed mask.
 */
int attn_fwd_blocksparse(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq, int Hkv,
                         int S, int D, int causal, double rope_base, const int* row_ptr, const int* col_idx,
                         void* stream);

/*
 * attn_bwd_blocksparse — attn_bwd under the block mask of
 * attn_fwd_blocksparse ("AttnFuse", sec. 4.3: the backward also iterates
 * only over active blocks).  The dQ kernel walks each row's listed key
 * tiles, the dK/dV kernel each key tile's listing rows (the library builds
 * that column-major copy with the device copy of the mask).  o and lse are
 * attn_fwd_blocksparse's outputs.  A query row that sees no key gets dQ = 0
 * and passes nothing to dK, dV; a key tile no row lists gets dK = dV = 0.
 * Arguments and errors: as attn_bwd, plus the mask of attn_fwd_blocksparse
 * (ATTN_ERR_NULL without row_ptr, ATTN_ERR_SHAPE for a malformed mask).
 */
int attn_bwd_blocksparse(const void* q, const void* k, const void* v, const void* o, const void* dO,
                         const float* lse, void* dq, void* dk, void* dv, int B, int Hq, int Hkv, int S, int D,
                         int causal, double rope_base, const int* row_ptr, const int* col_idx, void* stream);

/*
 * attn_fwd_local — the forward with the sliding_window and alibi combinators
 * of "AttnFuse: A Composable DSL for Compiling Attentions to Fused GPU
 * Kernels" (sec. 3; sliding windows and linear biases after its refs. 6, 7).
 *   window > 0: key j is visible to query i only when |i - j| < window
 *               (with causal: the last `window` keys up to and including i).
 *   alibi = 1:  the score gains -m_h |i - j|, m_h = 2^(-8 (h+1) / Hq).
 * The library lists the 128 x 128 tiles the window reaches and runs the
 * block-sparse kernel over them, masking and biasing cell by cell.
 * q, k, v, o, lse, B, Hq, Hkv, S, D, causal, rope_base: as attn_fwd.
 * A window of S or more keys is no window (every distance is below S).
 * Errors: as attn_fwd; ATTN_ERR_UNSUPPORTED for window < 0 or alibi not 0/1.
 */
int attn_fwd_local(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq, int Hkv, int S,
                   int D, int causal, double rope_base, int window, int alibi, void* stream);

/*
 * attn_bwd_local — attn_bwd for attn_fwd_local's attention ("AttnFuse",
 * sec. 3 sliding_window and alibi combinators; sec. 4.4: the backward
 * re-derives P from the forward's LSE and visits only the active blocks).
 * The library lists the window's tiles as attn_fwd_local does and runs the
 * block-sparse backward over them; each cell's P is exp(s + bias - LSE),
 * 0 outside the window, with the same bias -m_h |i - j| (alibi = 1), so
 * dS = P (dP - Dlt) keeps its form.  o and lse are attn_fwd_local's outputs
 * for the same window and alibi.
 * Arguments: as attn_bwd, plus window and alibi as attn_fwd_local.
 * Errors: as attn_bwd; ATTN_ERR_UNSUPPORTED for window < 0 or alibi not 0/1.
 */
int attn_bwd_local(const void* q, const void* k, const void* v, const void* o, const void* dO, const float* lse,
                   void* dq, void* dk, void* dv, int B, int Hq, int Hkv, int S, int D, int causal, double rope_base,
                   int window, int alibi, void* stream);

/*
 * attn_mask_schedule — the static task schedule attn_fwd_blocksparse and
 * attn_fwd_local launch with, for inspection and tests (host only).
 * A task is one 128-row query tile i of one (batch, head) x, encoded
 * i * bh + x; its cost is the number of key tiles row i lists plus one.
 * Each of `ctas` = min(num_ctas, ceil(nrows * bh / 2)) CTAs runs two task
 * streams; stream s of CTA c runs tasks_out[offsets_out[2c+s] ..
 * offsets_out[2c+s+1]).  Heaviest tasks go first into the least loaded
 * stream ("AttnFuse", sec. 4.3 visits only the listed blocks; the balance is
 * the prefill's longest-first rule, "Flash Attention: Causal Prefill D=128",
 * Step 4); each stream's list is then ordered by (batch-head, descending
 * query tile).
 *   row_ptr      host int32 [nrows + 1], a CSR block mask's row pointers
 *                (non-decreasing, row_ptr[0] = 0)
 *   bh           batch x heads, >= 1;  num_ctas >= 1
 *   tasks_out    host int32 [nrows * bh], or NULL
 *   offsets_out  host int32 [2 * ctas + 1], or NULL
 *   ctas_out     host int32, or NULL: receives ctas
 * Returns ATTN_ERR_NULL without row_ptr, ATTN_ERR_SHAPE for a bad argument
 * or more than 2^31 - 1 tasks.  Pure host computation.
 */
int attn_mask_schedule(const int* row_ptr, int nrows, long long bh, int num_ctas, int* tasks_out, int* offsets_out,
                       int* ctas_out);

/*
 * attn_fwd_schedule — the static tile schedule attn_fwd launches with, for
 * inspection and tests (host only).
 * A work unit is two 128-row query tiles that share one KV head: two
 * consecutive tiles of one head (Hq == Hkv), or two query heads of one KV
 * group at the same tile (Hq > Hkv; a group of odd size ends with a unit of
 * one head).  Unit word pair: x = qtile0 | qtile1 << 16 (0xFFFF: no second
 * tile), y = h0 | h1 << 8 | b << 16.  Its estimated cost is 2(bm + 1) + 4 per
 * query tile bm ("Flash Attention: Causal Prefill D=128", Step 4).
 * The KV heads, in (batch, KV head) order, are cut into windows whose K and
 * V take at most kv_window_bytes (at least one KV head each; <= 0: one
 * window); window by window, the heaviest units go first into the CTA with
 * the least load accumulated so far, and each CTA runs its units in that
 * order, so the CTAs move through the windows together and share K/V tiles
 * in L2.  attn_fwd uses 64 MiB, or ATTN_SCHEDULE_WINDOW_MB from the
 * environment when it is set.
 *   num_ctas     >= 1 (attn_fwd passes the device's SM count);
 *                ctas = min(num_ctas, units)
 *   words_out    host uint32 [2 * units], or NULL
 *   offsets_out  host int32 [ctas + 1], or NULL: CTA c runs units
 *                offsets_out[c] .. offsets_out[c+1]
 *   ctas_out     host int32, or NULL: receives ctas
 * Returns ATTN_ERR_SHAPE / ATTN_ERR_UNSUPPORTED on bad arguments.  Pure host
 * computation.
 */
int attn_fwd_schedule(int B, int Hq, int Hkv, int S, int D, int causal, int num_ctas, double kv_window_bytes,
                      unsigned* words_out, int* offsets_out, int* ctas_out);

/*
 * attn_build_tables — the host-side RoPE angles and window widths.
 *
 * The kernel derives the same angles on the device by complex multiplication
 * of per-tile, per-row and per-step factors computed from the same float64
 * values, so its rotated operands agree with these tables to a few float32 ulps.
 *   cos_out, sin_out  host float32 [S][D/2]: cos and sin of (p + pos_offset) *
 *                     theta_r for p = 0..S-1, computed in float64 and rounded.
 *                     Either may be NULL.  Requires rope_base > 0.
 *   win_out           host int32 [D/2]: W_r = floor(k * 2*pi / theta_r),
 *                     clamped to [0, 2^31-1]; 2^31-1 when the window is off.
 *                     May be NULL.
 * Pure host computation; returns ATTN_ERR_SHAPE / ATTN_ERR_UNSUPPORTED on bad
 * arguments.  ("ATFlash", The idea: w_r = k * lambda_r, lambda_r = 2*pi/theta_r.)
 */
int attn_build_tables(int S, int D, double rope_base, double window_k, long long pos_offset,
                      float* cos_out, float* sin_out, int* win_out);

/*
 * attn_selftest_wait_timeout — a check of the kernels' bounded waits, for tests.
 *
 * The source pages have no counterpart: this is failure detection.  It
 * enqueues the attn_fwd kernel for the given arguments (as attn_fwd, window
 * off) in a mode in which its TMA producer issues no load at all, with each
 * in-kernel wait limited to wait_limit_ns.  Every role's first wait then runs
 * out: the CTAs raise the status word and leave (no load or tensor-core work
 * is in flight), and attn_check(stream) returns ATTN_ERR_TIMEOUT.  Nothing is
 * read from q, k, v or written to o and lse; the device stays usable.
 *   wait_limit_ns  100000 (0.1 ms) .. 2000000000 (the limit of real launches),
 *                  else ATTN_ERR_UNSUPPORTED.
 */
int attn_selftest_wait_timeout(const void* q, const void* k, const void* v, void* o, float* lse,
                               int B, int Hq, int Hkv, int S, int D, int causal,
                               double rope_base, unsigned long long wait_limit_ns, void* stream);

/*
 * attn_check — synchronise `stream`, then read and clear the device status
 * word that the kernels raise when a bounded wait inside them runs out, or
 * when a row of the forward (attn_fwd and the entries built on it) came out
 * non-finite.  Returns ATTN_OK, ATTN_ERR_TIMEOUT (which takes precedence),
 * ATTN_ERR_NONFINITE, or ATTN_ERR_CUDA if the stream failed.
 */
int attn_check(void* stream);

/* attn_error_string — a static, human-readable name for an attn_status code. */
const char* attn_error_string(int status);

/*
 * attn_release_cache — free every cached device table on every device the
 * library has used.  No attn_fwd call may be in flight.
 */
void attn_release_cache(void);

#ifdef __cplusplus
}
#endif

#endif /* ATTN_H_ */
