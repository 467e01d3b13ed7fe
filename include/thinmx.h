/*
 * thinmx — weight-only low-bit decode matvecs for GB300 (sm_103a).
 *
 * A C ABI over hand-written CUDA kernels for the batch-1 (small-M) matvecs
 * of a weight-only quantised decoder:
 *   - MXFP4 gate/up matvec fused into SwiGLU (h = silu(g) * u);
 *   - the MoE variant: router, top-k, softmax and only the selected
 *     experts' gate/up/down;
 *   - grouped affine INT4 matvec for the dense Q/K/V/O projections;
 *   - bf16 gate/up SwiGLU matvec for the layers kept in bf16;
 *   - FP8 (E4M3, one scale per row) matvec and gate/up SwiGLU matvec;
 *   - single-token grouped-query attention over a bf16 KV cache;
 *   - the MoE layer with Q1 / Q2 packed low-bit experts.
 *
 * Sources.  The method is the ThinTensor decode runtime's:
 *   [DL4]  kerbin.cskartikey.dev/@satvikhardat, "Dev Log #4 — 91–96 tok/s
 *          with Selective MXFP4": MXFP4 on gate/up of layers 0:24 with an
 *          fp32 row postscale, the rest bf16 ("Why this was not just normal
 *          quantization"); MXFP4 as an execution format — read fewer bytes,
 *          block scales, bf16 activations, safe accumulation, then the row
 *          postscale ("Where Blackwell helps"); decode is a weight-read
 *          problem ("Why gate/up was the right target").
 *   [DL2]  same feed, "Dev Log #2": the gated_activation, router and expert
 *          operators of the execution tape.
 *   [DL3]  same feed, "Dev Log #3 — SmolLM3-3B Results": the quality FP8
 *          profile and its per-row-scaled matvec; its single-token GQA
 *          attention kernel over a bf16 KV cache.
 *   [SHIP] stardance.hackclub.com/projects/29750, "Hitting 100hrs and final
 *          ship" (production MXFP4/INT4 quantizers, exact routing, expert
 *          routing on the decode hot path), the MoE drift devlog (block-
 *          scaled matvec over the selected experts; fast_math lost accuracy),
 *          the 97.87 tok/s notes (dense_int4_layers for Q/K/V/O), the fixes
 *          list (affine INT4 with a partial last group; no allocations on
 *          the hot path; device given by the caller), the wide-matvec
 *          devlog (always loop over K with a bounded tile) and the graph-mode
 *          devlog's "What I've Done" (attention over a token bucket).
 *
 * Formats (canonical layouts; the parity surface):
 *   E2M1 code: bit 3 sign, bits 2..1 exponent (bias 1), bit 0 mantissa:
 *     +-{0, 0.5, 1, 1.5, 2, 3, 4, 6}.  E8M0 scale byte b: 2^(b-127), 255=NaN.
 *   MXFP4 matrix W [n][k] (row n = output, k = reduction), k % 32 == 0:
 *     codes  uint8 [n][k/2]  — byte j holds k=2j (low nibble), 2j+1 (high);
 *     scales uint8 [n][k/32] — one E8M0 byte per 32 consecutive k;
 *     postscale fp32 [n] (optional; absent = 1), applied after the sum.
 *   INT4 matrix [n][k], group G along k (last group may be partial):
 *     codes uint8 [n][k/2] (low nibble = even k), scales fp16 [n][ceil(k/G)],
 *     zero points uint8 [n][ceil(ceil(k/G)/2)] (low nibble = even group);
 *     w = (q - zp) * s.
 *   Activations x: bf16 [m][k] row-major; outputs bf16 [m][n] row-major.
 *
 * Conventions for every entry point:
 *   - Pointers are DEVICE pointers owned by the caller, on the current
 *     device; the library never allocates, frees or synchronises
 *     (tt_device_error_read is the one synchronising diagnostic).
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy stream).
 *   - Arguments are validated on the host before any launch; a non-OK
 *     status means nothing was launched.  TT_ERR_CUDA reports a launch
 *     error (cudaGetLastError) after the launch.
 *   - Asynchronous faults inside a kernel (a bounded wait that gave up)
 *     are recorded in a library-wide device error word, read and cleared by
 *     tt_device_error_read.
 *   - Alignment: every device pointer 16 bytes, except the per-row vectors
 *     (postscales, scales_f16, zero points, status words) which need their
 *     natural alignment.
 *   - Weights (and the MoE expert tables) are read before a call waits for
 *     the preceding kernel on its stream (programmatic dependent launch), so
 *     that their streaming overlaps that kernel's tail: the kernel launched
 *     just before a call must not write them.  Activations and outputs are
 *     touched only after the wait.
 *   - The library caches per-device state on first use (the device error
 *     word's address, the fixed MoE scratch's address, kernel attributes).
 *     A device reset (cudaDeviceReset) invalidates it: do not call the
 *     library on a device after resetting that device in the same process.
 */
#ifndef THINMX_H
#define THINMX_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    TT_OK = 0,
    TT_ERR_NULL = 1,        /* a required pointer is NULL                     */
    TT_ERR_SHAPE = 2,       /* a size is negative, zero where not allowed,
                               or breaks a divisibility rule                  */
    TT_ERR_ALIGN = 3,       /* a pointer is not aligned as documented         */
    TT_ERR_NONFINITE = 4,   /* NaN/Inf met by a quantiser (reported through
                               its device status word)                        */
    TT_ERR_UNSUPPORTED = 5, /* valid request outside what is implemented      */
    TT_ERR_CUDA = 6,        /* the CUDA runtime reported an error             */
    TT_ERR_TIMEOUT = 7,     /* a bounded device-side wait gave up             */
    TT_ERR_SIZE = 8         /* a caller buffer is smaller than required       */
} tt_status;

/* Human-readable name of a status.  Never NULL. */
const char* tt_status_str(int status);

/* ABI version: major*10000 + minor*100 + patch. */
int tt_version(void);

/* Reads the library's device error word (TT_OK, TT_ERR_TIMEOUT, ...) into
   *out and clears it.  Synchronises the device.  A diagnostic, not for the
   hot path. */
tt_status tt_device_error_read(int32_t* out);

/* ------------------------------------------------------------------------
 * MXFP4 quantiser  [SHIP "final ship": production MXFP4 quantizers]
 *
 * Per row and per block of 32 consecutive k:
 *   amax = max|w|; X = floor(log2 amax) - 2, read from the fp32 exponent
 *   field, clamped to [-127, 127] (X = -127 when amax = 0); scale byte
 *   X + 127; code = E2M1 round-to-nearest-even of w / 2^X, saturating at
 *   +-6, the sign bit kept on zero (a negative value that rounds to 0 gives
 *   code 0x8).  A block holding NaN/Inf gets scale 0xFF and zero codes, and
 *   TT_ERR_NONFINITE is OR-ed into *status_dev.
 * w: fp32 [n][k] device; codes [n][k/2]; scales [n][k/32];
 * status_dev: device int32 (may be NULL); the caller zeroes it beforehand.
 * Requires n >= 0, k >= 0, k % 32 == 0.  Setup step, not on the hot path.
 * --------------------------------------------------------------------- */
tt_status tt_quantize_mxfp4(const float* w, int64_t n, int64_t k,
                            uint8_t* codes, uint8_t* scales,
                            int32_t* status_dev, void* stream);

/* Test aid: out[n][k] fp32 = E2M1(code) * 2^(scale-127), exact (scale 0xFF
   gives NaN).  Canonical inputs. */
tt_status tt_mxfp4_dequantize(const uint8_t* codes, const uint8_t* scales,
                              int64_t n, int64_t k, float* out, void* stream);

/* ------------------------------------------------------------------------
 * Packed gate/up layout and loader  [DL4 "Where Blackwell helps": read
 * fewer bytes; the packed layout keeps the source encoding bit-exact]
 *
 * The packed buffer holds, for each output row r, one record with gate row
 * r's codes, up row r's codes and both rows' scales, contiguous and padded
 * to 16 bytes, followed by the two fp32 postscale vectors.  The exact
 * record layout is private; only its size is part of the ABI.  Packing is
 * a byte-for-byte rearrangement (no rounding).
 * --------------------------------------------------------------------- */
size_t tt_mxfp4_swiglu_packed_bytes(int64_t n, int64_t k);

/* gate_*, up_*: canonical MXFP4 [n][k]; postscales may be NULL (= 1).
   packed: device buffer of at least tt_mxfp4_swiglu_packed_bytes(n, k)
   bytes, 16-byte aligned.  Requires n >= 1, k >= 32, k % 32 == 0. */
tt_status tt_mxfp4_pack_swiglu(const uint8_t* gate_codes,
                               const uint8_t* gate_scales,
                               const float* gate_postscale,
                               const uint8_t* up_codes,
                               const uint8_t* up_scales,
                               const float* up_postscale, int64_t n,
                               int64_t k, void* packed, size_t packed_bytes,
                               void* stream);

/* ------------------------------------------------------------------------
 * MXFP4 gate/up SwiGLU matvec  [DL4 "Where Blackwell helps"; DL2
 * gated_activation]
 *
 *   g[i][r] = post_g[r] * sum_k Wg[r][k] * x[i][k]
 *   u[i][r] = post_u[r] * sum_k Wu[r][k] * x[i][k]
 *   h[i][r] = bf16_rne( silu(g) * u ),  silu(g) = g / (1 + exp(-g))
 * with fp32 accumulation.  packed: from tt_mxfp4_pack_swiglu(n, k).
 * x_bf16 [m][k], h_bf16 [m][n]; 1 <= m <= 64.  m = 1 streams the packed
 * records on CUDA cores; m = 2..8 runs a tile kernel whose multiply-adds go
 * to the warp-level tensor-core instruction (k <= 5120); the tcgen05
 * tensor-core kernel serves m >= 9, and m = 4..8 beyond k = 5120, when
 * k % 64 == 0; the CUDA-core kernels serve the rest of m <= 8.  m > 8 with
 * k % 64 != 0, or a tensor-core plan that does not fit, returns
 * TT_ERR_UNSUPPORTED before any launch.  Every kernel multiplies x in f16
 * after an exact power-of-two prescale (per 32-block and batch row, or on
 * the tensor-core kernel per batch row from its largest value over all of
 * k), so every finite bf16 input is served.
 * Requires n >= 1, 32 <= k <= 16384, k % 32 == 0.
 * --------------------------------------------------------------------- */
tt_status tt_mxfp4_swiglu_matvec(const void* packed, int64_t n, int64_t k,
                                 const uint16_t* x_bf16, int64_t m,
                                 uint16_t* h_bf16, void* stream);

/* bf16 gate/up SwiGLU matvec (the layers a selective profile keeps in
   bf16) [DL4 "Why this was not just normal quantization"].
   wg, wu: bf16 [n][k]; x [m][k]; h [m][n]; 1 <= m <= 8; k % 8 == 0. */
tt_status tt_bf16_swiglu_matvec(const uint16_t* wg, const uint16_t* wu,
                                int64_t n, int64_t k, const uint16_t* x_bf16,
                                int64_t m, uint16_t* h_bf16, void* stream);

/* ------------------------------------------------------------------------
 * Down projection of a dense decode MLP: single-matrix matvecs.  [DL4 "Why
 * this was not just normal quantization": the MLP block is gate/up SwiGLU
 * then the down projection, each projection in the precision its profile
 * gives it; SHIP 97.87 tok/s notes: layer stacks run as captured CUDA
 * graphs]  Like the gate/up calls they start streaming weights before
 * waiting for the preceding kernel (programmatic dependent launch), so a
 * gate/up -> down pair on one stream overlaps the two.
 * --------------------------------------------------------------------- */

/* y[i][r] = bf16_rne( post[r] * sum_k W[r][k] * x[i][k] ) on the canonical
   MXFP4 buffers (codes [n][k/2], scales [n][k/32], postscale [n] or NULL),
   fp32 accumulation.  x [m][k], y [m][n].  Requires n >= 1,
   32 <= k <= 16384, k % 32 == 0, 1 <= m <= 8; codes and x 16-byte aligned.
   A batch whose x does not fit the kernel's shared-memory staging
   (m * (2k + k/8) bytes) returns TT_ERR_UNSUPPORTED before any launch. */
tt_status tt_mxfp4_matvec(const uint8_t* codes, const uint8_t* scales, const float* postscale,
                          int64_t n, int64_t k, const uint16_t* x_bf16, int64_t m,
                          uint16_t* y_bf16, void* stream);

/* y[i][r] = bf16_rne( sum_k W[r][k] * x[i][k] ), W bf16 [n][k], fp32
   accumulation.  Requires n >= 1, k % 8 == 0, 1 <= m <= 8; w and x 16-byte
   aligned. */
tt_status tt_bf16_matvec(const uint16_t* w, int64_t n, int64_t k, const uint16_t* x_bf16,
                         int64_t m, uint16_t* y_bf16, void* stream);

/* ------------------------------------------------------------------------
 * Packed single-matrix layout (MoE down projections), sliced by columns:
 * for each 16-wide slice of k, the 8 code bytes of every row in row order,
 * then for each 32-block the E8M0 byte of every row; each part padded to 16
 * bytes.  A kernel that owns one slice of the reduction index reads it as
 * one contiguous run.  Byte-for-byte rearrangement of canonical MXFP4;
 * layout private, size public.
 * Requires n >= 1, 32 <= k <= 16384, k % 32 == 0; packed 16-byte aligned.
 * --------------------------------------------------------------------- */
size_t tt_mxfp4_rows_packed_bytes(int64_t n, int64_t k);
tt_status tt_mxfp4_pack_rows(const uint8_t* codes, const uint8_t* scales, int64_t n, int64_t k,
                             void* packed, size_t packed_bytes, void* stream);

/* ------------------------------------------------------------------------
 * MoE MLP at batch 1  [DL2 router/expert operators; SHIP MoE drift devlog
 * (block-scaled matvec over the selected experts), "final ship" (exact
 * routing; expert routing on the decode hot path)]
 *
 *   logit[e] = x . W_r[e]            (bf16 inputs; the fp32 logit is the
 *                                     rounding of the exact dot product)
 *   idx      = the top_k experts by logit, descending, ties to the lower
 *              index; p = softmax of their logits
 *   h_j      = silu(Wg[idx_j] x) * (Wu[idx_j] x)          (fp32, inter)
 *   out      = bf16_rne( sum_j p_j * Wd[idx_j] h_j )      (hidden)
 * Experts live in buffers of their own: gate_up_packed and down_packed are
 * DEVICE arrays of n_experts DEVICE pointers (8-byte aligned arrays), entry
 * e pointing to expert e's tt_mxfp4_swiglu_packed_bytes(inter, hidden)-byte
 * gate/up buffer (gate = the swiglu gate rows, packed without postscales)
 * and its tt_mxfp4_rows_packed_bytes(hidden, inter)-byte down buffer, each
 * 16-byte aligned.  Only the selected experts' entries are read; a selected
 * entry that is NULL or misaligned is reported through the device error
 * word (TT_ERR_NULL / TT_ERR_ALIGN, tt_device_error_read) and nothing is
 * read from it or written to out.  The tables, like every weight buffer of
 * this library, are read before the call waits for the preceding kernel on
 * the stream (programmatic dependent launch): that kernel must not write
 * them.  router_w_bf16 [E][hidden].
 * out_idx int32 [top_k], out_prob fp32 [top_k] (device).  workspace: device,
 * >= tt_moe_workspace_bytes(...) bytes, 16-byte aligned, ZERO-FILLED before
 * its first use (e.g. cudaMemsetAsync once after allocating it); the call
 * owns it until the stream reaches the end of the call and leaves it ready
 * for the next call.  Its first 64 bytes hold the kernel's grid-wide counter
 * (64-bit), which each call advances by the number of CTAs and never resets;
 * the router partial replicas that follow are left cleared.  After a call
 * that reported TT_ERR_TIMEOUT through tt_device_error_read, zero the
 * workspace again before reusing it.
 * The layer runs as one cooperative kernel of one CTA per SM: router
 * partial sums, expert choice in every CTA, each CTA computing a 16-wide
 * slice range of the selected experts' h and multiplying it into the
 * matching down columns, then a fixed-order sum of the per-CTA partial
 * outputs (a grid-wide counter and self-marking partial slots in the
 * workspace).  A shape whose
 * shared-memory plan does not fit one CTA per SM returns TT_ERR_UNSUPPORTED
 * before any launch.
 * Requires hidden, inter multiples of 32, hidden <= 8192, inter <= 8192,
 * 1 <= top_k <= min(E, 8), E <= 256.  Router logits must be finite.
 * --------------------------------------------------------------------- */
size_t tt_moe_workspace_bytes(int64_t hidden, int64_t inter, int32_t n_experts, int32_t top_k);
tt_status tt_moe_mxfp4_topk_mlp(const uint16_t* x_bf16, int64_t hidden, int64_t inter,
                                const uint16_t* router_w_bf16, int32_t n_experts, int32_t top_k,
                                const void* const* gate_up_packed, const void* const* down_packed,
                                uint16_t* out_bf16, int32_t* out_idx, float* out_prob,
                                void* workspace, size_t workspace_bytes, void* stream);

/* ------------------------------------------------------------------------
 * MoE MLP without a caller workspace.  (No counterpart on the ThinTensor
 * pages: an addition of this library.)
 *
 * Same computation, arguments and requirements as tt_moe_mxfp4_topk_mlp,
 * minus the workspace.  It is for callers that cannot give the library
 * device memory: plugins inside a host that owns the device pool and offers
 * no allocator, real-time loops that forbid allocator calls (an allocation
 * can synchronise the device or fragment the pool), or bindings without a
 * CUDA allocator.  The call allocates nothing; it runs on a fixed array
 * inside the library (static device memory, held by every GPU that loads
 * the library until the process exits, zero at load: 524,352 bytes of
 * counter and router partials + 256 * 4 * TT_MOE_STATIC_MAX_HIDDEN bytes
 * of partial outputs) sized for hidden <= TT_MOE_STATIC_MAX_HIDDEN; larger
 * requests return TT_ERR_SIZE before any launch.  After a TT_ERR_TIMEOUT
 * from this entry point its counters may be left set: the process must not
 * reuse it.  The first call on each device looks the array's address up
 * (cudaGetSymbolAddress), so make it before any stream capture.  All calls
 * share the array: two calls that can overlap on the GPU (different
 * streams without ordering between them) race and give wrong results.
 * --------------------------------------------------------------------- */
#define TT_MOE_STATIC_MAX_HIDDEN 4096
tt_status tt_moe_mxfp4_topk_mlp_static(const uint16_t* x_bf16, int64_t hidden, int64_t inter,
                                       const uint16_t* router_w_bf16, int32_t n_experts,
                                       int32_t top_k, const void* const* gate_up_packed,
                                       const void* const* down_packed, uint16_t* out_bf16,
                                       int32_t* out_idx, float* out_prob, void* stream);

/* ------------------------------------------------------------------------
 * FP8 (E4M3) weights with one fp32 scale per row  [DL3 "Dev Log #3 —
 * SmolLM3-3B Results": the quality FP8 profile keeps gate/up and the middle
 * down projections in FP8; its scaled matvec sums code value times x along
 * the row, then multiplies by the row's scale]
 *
 * E4M3 code: bit 7 sign, bits 6..3 exponent (bias 7), bits 2..0 mantissa;
 * exponent 0 is subnormal (m/8 * 2^-6); 0x7F/0xFF are NaN; no infinities;
 * largest magnitude 448.  Canonical matrix [n][k]: codes uint8 [n][k] (row
 * major), scales fp32 [n].
 *
 * Quantiser, per row: amax = max |w|; scale = fp32 round-to-nearest of
 * amax / 448 (computed in fp64); code = E4M3 round-to-nearest-even of
 * w / scale (the division in fp64), saturating at +-448, the sign kept on a
 * zero result (0x80).  A row with scale 0 (amax = 0, or below fp32's range)
 * gets zero codes; a row holding NaN/Inf gets scale NaN, zero codes, and
 * TT_ERR_NONFINITE OR-ed into *status_dev (device int32, may be NULL, zeroed
 * by the caller).  Setup step.  Requires n >= 0, k >= 0.
 * --------------------------------------------------------------------- */
tt_status tt_quantize_fp8(const float* w, int64_t n, int64_t k, uint8_t* codes, float* scales,
                          int32_t* status_dev, void* stream);

/* y[i][r] = bf16_rne( scale[r] * sum_k E4M3(codes[r][k]) * x[i][k] ), fp32
   accumulation (the down projection of the FP8 profile).  x [m][k], y [m][n].
   Requires n >= 1, 16 <= k <= 16384, k % 16 == 0, 1 <= m <= 8; codes and x
   16-byte aligned.  A batch whose x does not fit the kernel's shared-memory
   staging (m * k f16 values, at most the device's per-block limit) returns
   TT_ERR_UNSUPPORTED before any launch. */
tt_status tt_fp8_matvec(const uint8_t* codes, const float* scales, int64_t n, int64_t k,
                        const uint16_t* x_bf16, int64_t m, uint16_t* y_bf16, void* stream);

/* h[i][r] = bf16_rne( silu(g) * u ) with g, u the FP8 matvecs of the gate and
   up matrices (same shapes and rules as tt_fp8_matvec). */
tt_status tt_fp8_swiglu_matvec(const uint8_t* gate_codes, const float* gate_scales,
                               const uint8_t* up_codes, const float* up_scales, int64_t n,
                               int64_t k, const uint16_t* x_bf16, int64_t m, uint16_t* h_bf16,
                               void* stream);

/* ------------------------------------------------------------------------
 * Grouped affine INT4  [SHIP 97.87 tok/s notes: dense_int4_layers="all" for
 * Q/K/V/O; fixes list: "correct affine INT4 partial-group quantization"]
 *
 * Quantiser, per row and group [g*G, min((g+1)*G, k)) (the last group may be
 * partial and uses only its own elements):
 *   s  = fp16 round-to-nearest-even of (max - min) / 15, computed in fp64;
 *   zp = clamp(rint(-min / s), 0, 15);  q = clamp(rint(w / s) + zp, 0, 15)
 *   (rint = nearest, ties to even).  A group with s == 0 stores zp = q = 0.
 *   A group holding NaN/Inf (scale 0x7E00), or whose scale overflows fp16,
 *   stores zp = q = 0 and OR-s TT_ERR_NONFINITE into *status_dev.
 * w fp32 [n][k]; codes [n][k/2] (low nibble = even k); scales_f16
 * [n][ceil(k/G)]; zp_u4 [n][ceil(ceil(k/G)/2)] (low nibble = even group).
 * Requires k even, G even >= 2.  Setup step.
 * --------------------------------------------------------------------- */
tt_status tt_quantize_int4_grouped(const float* w, int64_t n, int64_t k, int32_t group,
                                   uint8_t* codes, uint16_t* scales_f16, uint8_t* zp_u4,
                                   int32_t* status_dev, void* stream);

/* y[i][r] = bf16_rne( sum_g s[r][g] * sum_{k in g} (q[r][k] - zp[r][g]) * x[i][k] )
   with fp32 accumulation; canonical INT4 buffers as above; x [m][k],
   y [m][n].  Requires 32 <= k <= 8192, k % 32 == 0, G % 32 == 0, 1 <= m <= 8;
   codes and x 16-byte aligned. */
tt_status tt_int4_grouped_matvec(const uint8_t* codes, const uint16_t* scales_f16,
                                 const uint8_t* zp_u4, int64_t n, int64_t k, int32_t group,
                                 const uint16_t* x_bf16, int64_t m, uint16_t* y_bf16,
                                 void* stream);

/* ------------------------------------------------------------------------
 * Single-token GQA attention  [DL3 "Dev Log #3 — SmolLM3-3B Results": the
 * attention path is single-token GQA, query head h reads kv head
 * h // (heads // kv_heads), scores = sum(key * q) * scale, KV cache bf16;
 * SHIP graph-mode devlog, "What I've Done" item 3: the same kernel over a
 * context of up to a fixed token bucket]
 *
 *   G = heads / kv_heads,  j = h / G,  for t < len:
 *   s[h][t] = scale * sum_i q[h][i] * k[j][t][i]
 *   o[h][i] = bf16_rne( sum_t softmax_t(s[h][.]) * v[j][t][i] )
 *
 * q_bf16 [heads][head_dim]; k_cache, v_cache bf16 [kv_heads][cap][head_dim]
 * (token t of kv head j at (j * cap + t) * head_dim; only t < len is read);
 * out_bf16 [heads][head_dim].  Scores are exact bf16 products summed in
 * fp32; the softmax and the weighted sum are fp32 (the weights carried as
 * two bf16 terms into the tensor-core product).
 * Requires heads >= 1, kv_heads >= 1, heads % kv_heads == 0, 1 <= len <= cap,
 * scale finite (else TT_ERR_SHAPE / TT_ERR_NONFINITE); head_dim 64 or 128,
 * G <= 16, kv_heads <= 64 and cap <= 2^31 (else TT_ERR_UNSUPPORTED).  q, k_cache,
 * v_cache, out and workspace 16-byte aligned.
 * workspace: device, >= tt_gqa_decode_workspace_bytes(...) bytes: scratch for
 * the per-split partial results (no initial contents needed).  Calls that
 * share a workspace must be ordered on one stream.  The call is two kernels:
 * the split kernel (token ranges of each kv head, one CTA per SM) and the
 * merge kernel, launched programmatically behind it.  q and the cache are
 * read after the call waits for the preceding kernel on the stream (that
 * kernel may append the newest token).
 * --------------------------------------------------------------------- */
size_t tt_gqa_decode_workspace_bytes(int32_t heads, int32_t kv_heads, int32_t head_dim);
tt_status tt_gqa_decode_attention(const uint16_t* q_bf16, const uint16_t* k_cache,
                                  const uint16_t* v_cache, int32_t heads, int32_t kv_heads,
                                  int32_t head_dim, int64_t cap, int64_t len, float scale,
                                  uint16_t* out_bf16, void* workspace, size_t workspace_bytes,
                                  void* stream);

/* ------------------------------------------------------------------------
 * Q1 / Q2 packed low-bit experts  [SHIP 97.87 tok/s notes:
 * packed_expert_q1_layers="0:24", the MoE experts packed as 1-bit "Q1"
 * structures, 9.52 GB of MXFP4 experts becoming 2.38 GB; final devlog: Q2
 * and Q1 quantizers, the low-bit selected-expert SwiGLU kernel]
 *
 * The pages do not print the encoding.  Reading taken (the one the 4x
 * footprint fixes for an MX-style format): bits = 1 (Q1) or 2 (Q2) per
 * weight and one E8M0 step 2^X per block of 128 weights along k (the last
 * block may be partial).
 *   X: m = (sum of |w| over the block, in k order, in fp64) / count;
 *      2^X = the power of two nearest m (ties to the lower), clamped to
 *      [2^-127, 2^127]; an all-zero block has X = -127.
 *   Q1: code c = 1 if w < 0 else 0; value (1 - 2c) 2^X.
 *   Q2: code q = clamp(floor(w / 2^X) + 2, 0, 3); value (q - 1.5) 2^X.
 *   A block holding NaN/Inf: scale byte 0xFF, zero codes, TT_ERR_NONFINITE
 *   OR-ed into *status_dev.
 * Matrix buffer [n][k]: plane 0 [n][P] (and, for Q2, plane 1 [n][P]) then
 * the scales [n][S]; P = 16 * ceil(k/128), S = ceil(k/128) rounded up to
 * 16; bit (kk % 8) of byte kk / 8 of a row's plane p is bit p of element
 * kk's code; padding is zero.  tt_lowbit_matrix_bytes gives the size.
 * --------------------------------------------------------------------- */
size_t tt_lowbit_matrix_bytes(int32_t bits, int64_t n, int64_t k);

/* Quantise w fp32 [n][k] (device) into buf (device, >= the matrix bytes,
   16-byte aligned).  status_dev: device int32, may be NULL.  Setup step. */
tt_status tt_quantize_lowbit(int32_t bits, const float* w, int64_t n, int64_t k, void* buf,
                             size_t buf_bytes, int32_t* status_dev, void* stream);

/* The MoE layer with low-bit experts:
 *   logits = fp32(Wr x) (exact products, compensated sums, rounded once),
 *   idx = the top_k largest (ties to the lower index, descending), p =
 *   softmax over them; for each selected expert j
 *   h_j = silu(G_j x) * (U_j x) (fp32), out = bf16_rne( sum_j p_j D_j h_j ).
 * gate_up: device array of E pointers, expert e's gate/up matrix buffer
 * ([2 inter][hidden]: gate rows first, then up rows); down: device array of
 * E pointers, expert e's down matrix buffer ([hidden][inter]); each buffer
 * 16-byte aligned, only the selected experts' entries are read (a NULL or
 * misaligned one is reported through tt_device_error_read and its expert
 * contributes nothing).  router_w_bf16 [E][hidden].  out_idx int32
 * [top_k], out_prob fp32 [top_k] (device).  workspace: device, >=
 * tt_moe_lowbit_workspace_bytes(...) bytes, 16-byte aligned, no initial
 * contents needed; after the call (in stream order) it holds h, fp32
 * [top_k][inter], at its start.  Requires bits 1 or 2, hidden and inter
 * multiples of 32 in [32, 8192], 1 <= top_k <= min(8, E), E <= 256.  Three
 * kernels (router; selected-expert SwiGLU; weighted down projection).
 * --------------------------------------------------------------------- */
size_t tt_moe_lowbit_workspace_bytes(int64_t inter, int32_t n_experts, int32_t top_k);
tt_status tt_moe_lowbit_topk_mlp(int32_t bits, const uint16_t* x_bf16, int64_t hidden,
                                 int64_t inter, const uint16_t* router_w_bf16, int32_t n_experts,
                                 int32_t top_k, const void* const* gate_up,
                                 const void* const* down, uint16_t* out_bf16, int32_t* out_idx,
                                 float* out_prob, void* workspace, size_t workspace_bytes,
                                 void* stream);

#ifdef __cplusplus
}
#endif
#endif /* THINMX_H */
