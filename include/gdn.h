/*
 * gdn.h -- C-ABI of libgdn, the GB300 (sm_103a) gated delta rule library.
 *
 * The method (logicaffeine_compile/codegen_cuda/gdn.rs, kernel `gdn_step`):
 * for every sequence b and value head h, with key/query head g = h mod NK
 * (heads are tiled, not repeat-interleaved), the D x D state S of (b, h)
 * takes one token as
 *
 *     u[a]    = S[a] . k_g                    (row a of S against the key)
 *     coef[a] = beta_h * (v_h[a] - alpha_h * u[a])
 *     S[a][c] = alpha_h * S[a][c] + coef[a] * k_g[c]
 *     o[a]    = (S_new[a] . q_g) / sqrt(D)
 *
 * i.e. S <- alpha S + beta (v - alpha S k) k^T and o = S q / sqrt(D).  The
 * gated RMS norm that follows (same page, kernel `gdn_gate_norm`) is
 *
 *     out[a]  = gn[a] * o[a] / sqrt(mean_a(o^2) + eps) * z[a] * sigmoid(z[a])
 *
 * (normalise first, then gate).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - Memory: every pointer is a DEVICE pointer to memory the caller owns.  The
 *   library allocates nothing, keeps no per-call state, and updates the state
 *   in place.  Calls are asynchronous on `stream` (a cudaStream_t passed as
 *   void*; NULL is the legacy default stream); the caller synchronises.  The
 *   outputs of the gdn_decode* calls (o, out, and the int8 codes, scales and
 *   y) may also be pinned host memory, which the kernels then write directly
 *   over the host link (the same results; complete, like any output, when the
 *   call's work in the stream is); everything else should be device memory.
 * - State layout: sequence b's slot starts `b * state_pitch` ELEMENTS after
 *   `state`; inside a slot, head h is a contiguous D x D row-major block at
 *   `h * D * D`, row a = value index, column c = key index.  state_pitch >=
 *   NV * D * D; a pitch larger than that leaves padding the library never
 *   reads or writes.  (metrale_model_layers/layers/ops/ssm_gdn_a.rs,
 *   `gdn_decode_f16_strided_norm`, passes the slot pitch the same way: in
 *   elements, set by how the pool was sized.)
 * - Token rows: q and k rows hold NK * D floats, v, z, o and out rows NV * D,
 *   alpha and beta rows NV.  Row i (sequence b for decode; token (b, t) at
 *   i = b * seq_len + t for prefill) starts `i * <x>_stride` ELEMENTS after its
 *   base pointer; a stride must be at least the row length.
 * - Return value: GDN_OK, or a GDN_ERR_* code.  Arguments are checked on the
 *   host before anything is launched; a rejected call touches no memory.
 *   GDN_ERR_CUDA means the launch itself failed; gdn_last_cuda_error() gives
 *   the cudaError_t.  A batch, seq_len or n of 0 is a valid empty call.
 * - Fast paths (D == 128, 16-byte aligned base pointers, strides and pitch
 *   that keep every row 16-byte aligned) are taken automatically; any other
 *   1 <= D <= 256 runs a general kernel with the same results up to fp32
 *   summation order.
 * - Ordering: results are those of plain stream order.  When their grid is
 *   a few waves at most (e.g. one layer at batch 32), the D == 128 kernels of
 *   gdn_decode*, gdn_decode_chunk2 and (fp32 states) gdn_decode_conv_norm*,
 *   and the general gdn_decode* kernel on grids of one wave, are launched
 *   with CUDA's programmatic stream serialisation: such a kernel may become
 *   resident while the kernel before it in the stream is still running, but
 *   reads and writes no memory until that kernel has completed
 *   (meanwhile it only asks the L2 for part of its state, a hint), and it lets
 *   the kernel after it start the same way.  A caller's kernel that follows
 *   in the stream sees the outputs as usual; if it is itself launched with
 *   that attribute it must wait for its grid dependency (griddepcontrol.wait)
 *   before reading them, as that attribute always requires.
 */
#ifndef GDN_H
#define GDN_H

#include <stdint.h>

#if defined(_WIN32)
#define GDN_API __declspec(dllexport)
#else
#define GDN_API __attribute__((visibility("default")))
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Status codes. */
#define GDN_OK 0
#define GDN_ERR_ARG 1          /* null pointer, negative or zero dims, short stride/pitch, bad eps */
#define GDN_ERR_UNSUPPORTED 2  /* D > 256, unknown state dtype */
#define GDN_ERR_ALIGN 3        /* a pointer not aligned to its element size */
#define GDN_ERR_ALIAS 4        /* an output overlaps another operand */
#define GDN_ERR_CUDA 5         /* the CUDA launch failed (see gdn_last_cuda_error) */
/* There is no timeout status: no kernel of the library waits on a flag, a
 * counter or another block (only on its own barriers, copy groups and, in
 * gdn_prefill_chunked, the completion of its own MMAs and tensor copies,
 * bounded waits counted by gdn_device_wait_timeouts).  A
 * base, stride or pitch that rules out the 16-byte vector kernels is not an
 * error either: the general kernel runs instead (GDN_ERR_ALIGN is only for a
 * pointer not aligned to its own element size). */

/* Storage type of the h-state. */
typedef enum {
    GDN_STATE_F32 = 0,
    GDN_STATE_F16 = 1,
    GDN_STATE_DTYPE_MAX_ENUM = 0x7fffffff   /* not a dtype: keeps the type int-sized on every ABI */
} gdn_state_dtype;

/*
 * gdn_decode -- one token through the recurrence for `batch` sequences,
 * raw fp32 output.
 *   Defined by: gdn.rs, kernel `gdn_step` (the step, g = h mod NK, the
 *   1/sqrt(D) output scale); ssm_gdn_a.rs, launchers `gdn_decode` and
 *   `gdn_decode_f32_strided` (batched, per-sequence row strides).
 *   state        [batch] slots, dtype `state_dtype` (fp32, or fp16 that is
 *                read to fp32, updated in fp32 and stored back
 *                round-to-nearest-even), updated in place.
 *   q, k         [batch] rows of NK*D fp32 (already L2-normalised upstream).
 *   v            [batch] rows of NV*D fp32.
 *   alpha, beta  [batch] rows of NV fp32: linear decay in (0,1] and write
 *                strength.
 *   o            [batch] rows of NV*D fp32, written.
 *   Errors: GDN_ERR_ARG, GDN_ERR_UNSUPPORTED, GDN_ERR_ALIGN, GDN_ERR_ALIAS
 *   (state or o overlapping any operand), GDN_ERR_CUDA.
 */
GDN_API int gdn_decode(void *state, gdn_state_dtype state_dtype, int64_t state_pitch,
                       const float *q, const float *k, const float *v,
                       const float *alpha, const float *beta, float *o,
                       int batch, int nk, int nv, int d,
                       int64_t qk_stride, int64_t v_stride, int64_t gb_stride,
                       int64_t o_stride, void *stream);

/*
 * gdn_decode_norm -- gdn_decode with the gated RMS norm fused in the same
 * kernel; writes bf16 and no fp32 output.
 *   Defined by: gdn.rs, kernels `gdn_step` and `gdn_gate_norm` (norm over
 *   the D outputs of a head, mean of squares plus eps under the root, weight
 *   gn shared by all heads, then the silu(z) gate); ssm_gdn_a.rs,
 *   `gdn_decode_f32_norm` / `gdn_decode_f32_strided_norm` (fused, bf16 out)
 *   and `gdn_decode_f16_strided_norm` (fp16 h-state pool with a slot pitch).
 *   z            [batch] rows of NV*D fp32 gate input.
 *   gn           [D] fp32 norm weight.
 *   eps          >= 0, finite.
 *   out          [batch] rows of NV*D bf16 (raw uint16 bits), written,
 *                rounded to nearest even.
 *   Other arguments and errors as gdn_decode.
 */
GDN_API int gdn_decode_norm(void *state, gdn_state_dtype state_dtype, int64_t state_pitch,
                            const float *q, const float *k, const float *v,
                            const float *alpha, const float *beta,
                            const float *z, const float *gn, float eps,
                            uint16_t *out,
                            int batch, int nk, int nv, int d,
                            int64_t qk_stride, int64_t v_stride, int64_t gb_stride,
                            int64_t z_stride, int64_t out_stride, void *stream);

/*
 * gdn_decode_norm_q8 -- gdn_decode_norm with the activation quantisation of
 * the o-projection's input fused in: the normed output leaves as int8 codes
 * in groups of 32 with one fp32 scale per group.
 *   Defined by: gdn.rs, kernel `gdn_gate_norm_q` (the gate norm, then per
 *   32-value group: scale = max |y| / 127, or 1 when the group is all zero;
 *   code = y / scale rounded to the nearest integer, ties to even; computed in
 *   fp32); the step and the norm as gdn_decode_norm.
 *   Groups are 32 consecutive values of a token's NV*D output vector, so a
 *   head holds D/32 of them; D must be a multiple of 32
 *   (GDN_ERR_UNSUPPORTED otherwise).
 *   xq           [batch] rows of NV*D int8 codes, written; row stride
 *                xq_stride elements (bytes).
 *   xs           [batch] rows of NV*D/32 fp32 scales, written; row stride
 *                xs_stride elements.
 *   y            NULL, or [batch] rows of NV*D fp32: the normed values the
 *                codes were taken from, written; row stride y_stride.
 *   Other arguments and errors as gdn_decode_norm (xq, xs and y overlapping
 *   any operand: GDN_ERR_ALIAS).
 */
GDN_API int gdn_decode_norm_q8(void *state, gdn_state_dtype state_dtype, int64_t state_pitch,
                               const float *q, const float *k, const float *v,
                               const float *alpha, const float *beta,
                               const float *z, const float *gn, float eps,
                               int8_t *xq, float *xs, float *y,
                               int batch, int nk, int nv, int d,
                               int64_t qk_stride, int64_t v_stride, int64_t gb_stride,
                               int64_t z_stride, int64_t xq_stride, int64_t xs_stride,
                               int64_t y_stride, void *stream);

/*
 * gdn_gate_norm -- the gated RMS norm as its own call, over rows of raw
 * outputs o (for instance every token of gdn_prefill_seq), bf16 out.
 *   Defined by: gdn.rs, kernel `gdn_gate_norm` (per head of D values:
 *   out = gn * o / sqrt(mean o^2 + eps) * silu(z); the norm first, then the
 *   gate; gn shared by all heads).
 *   o, z         [rows] rows of NV*D fp32, row strides o_stride, z_stride.
 *   gn           [D] fp32.  eps >= 0, finite.  1 <= D <= 256.
 *   out          [rows] rows of NV*D bf16 (raw uint16 bits, round to nearest
 *                even), written; row stride out_stride.
 *   rows = 0 is a valid empty call.  Errors: GDN_ERR_ARG, GDN_ERR_UNSUPPORTED
 *   (D > 256), GDN_ERR_ALIGN, GDN_ERR_ALIAS (out overlapping any operand),
 *   GDN_ERR_CUDA.
 */
GDN_API int gdn_gate_norm(const float *o, const float *z, const float *gn, float eps, uint16_t *out,
                          int64_t rows, int nv, int d, int64_t o_stride, int64_t z_stride,
                          int64_t out_stride, void *stream);

/*
 * gdn_gate_norm_q8 -- gdn_gate_norm with the int8 epilogue of
 * gdn_decode_norm_q8 (gdn.rs `gdn_gate_norm_q`): groups of 32 consecutive
 * values of a row, scale = max |y| / 127 (1 for an all-zero group), code =
 * y / scale rounded to nearest even, in fp32.  D must be a multiple of 32.
 *   xq           [rows] rows of NV*D int8 codes, row stride xq_stride.
 *   xs           [rows] rows of NV*D/32 fp32 scales, row stride xs_stride.
 *   y            NULL, or [rows] rows of NV*D fp32 normed values, y_stride.
 *   Other arguments and errors as gdn_gate_norm.
 */
GDN_API int gdn_gate_norm_q8(const float *o, const float *z, const float *gn, float eps,
                             int8_t *xq, float *xs, float *y, int64_t rows, int nv, int d,
                             int64_t o_stride, int64_t z_stride, int64_t xq_stride, int64_t xs_stride,
                             int64_t y_stride, void *stream);

/*
 * gdn_decode_conv_norm -- one token from the projection outputs to the normed
 * bf16 output in one launch: the depthwise causal conv ring update with silu
 * on q, k and v, the per-head L2 normalisation of q and k, the gates from
 * their logits, the recurrence and the gated RMS norm.
 *   Defined by: ssm_gdn_a.rs, launcher `gdn_decode_f32_conv_norm` (conv
 *   update, L2 norm, recurrence and gated norm in one decode launch);
 *   gdn.rs `gk_conv_silu_l2` (ring shifted by one, the token appended,
 *   reduced with the taps, silu; q/k heads divided by sqrt(sum y^2 +
 *   l2_eps)), `gk_gdn_gates` (beta = sigmoid(br), alpha = (1 + e^(ar +
 *   dt))^rate, rate the stored negative decay rate), `gdn_step`,
 *   `gdn_gate_norm`.
 *   C            conv channels = 2*NK*D + NV*D, ordered [q heads | k heads |
 *                v heads] (value head h's v channels at 2*NK*D + h*D).
 *   conv_state   [batch] slots of taps*C fp32, slot pitch conv_pitch >= taps*C
 *                elements, [tap][channel] with tap taps-1 the newest; updated
 *                in place (shifted by one, this token appended).
 *   taps         1..8.
 *   x            [batch] rows of C fp32: this token's projection.
 *   conv_w       [taps][C] fp32 conv taps.
 *   br, ar       [batch] rows of NV gate logits.  dt, rate: [NV].
 *   z, gn, eps, out as gdn_decode_norm; l2_eps >= 0 for the q/k norm.
 *   workspace    [batch*NK] int32 counters owned by the caller: zero before
 *                the first call (e.g. cudaMemsetAsync); every call leaves
 *                them zero.  Where the kernel gives each value head its own
 *                block (fp32 states, or NV/NK > 8), the value heads of a key
 *                head each read its q/k ring rows and the counters let the
 *                last reader write them; the fp16 kernel (one block per key
 *                head) does not touch them.  Always required.  Calls that can
 *                overlap on the GPU need separate workspaces (and separate
 *                conv states).
 *   NV must be a multiple of NK (the value heads of a key head are h = kh +
 *   r*NK, r < NV/NK).  State and output as gdn_decode_norm.
 *   Errors as gdn_decode_norm; GDN_ERR_UNSUPPORTED if NV % NK != 0.
 */
GDN_API int gdn_decode_conv_norm(void *state, gdn_state_dtype state_dtype, int64_t state_pitch,
                                 float *conv_state, int64_t conv_pitch, int taps,
                                 const float *x, const float *conv_w,
                                 const float *br, const float *ar, const float *dt, const float *rate,
                                 const float *z, const float *gn, float l2_eps, float eps,
                                 uint16_t *out, int32_t *workspace,
                                 int batch, int nk, int nv, int d,
                                 int64_t x_stride, int64_t gate_stride, int64_t z_stride,
                                 int64_t out_stride, void *stream);

/*
 * gdn_decode_conv_norm_noalloc -- gdn_decode_conv_norm without a workspace
 * argument, for callers that cannot provide device memory beyond the inputs
 * and outputs (no allocator of their own, a fixed memory plan, or no device
 * synchronisation allowed on the decode path).  None of the source pages has
 * a counterpart: it is an addition of this library.
 *   The counters live in a static array inside the library, one copy per
 *   device, GDN_NOALLOC_MAX_KEY_HEADS int32 long.  The first call on a device
 *   (with that device current) looks up its address once; make that first
 *   call before any stream capture begins.  The array is zero when the
 *   library is loaded and every completed call leaves it zero; nothing needs
 *   clearing by the caller.  The call allocates and frees nothing.
 *   Calls that can run on the GPU at the same time on one device (streams
 *   with no ordering between them) share the array and race: results are
 *   then undefined.  Calls ordered on one stream are fine.
 *   Arguments, layouts and results as gdn_decode_conv_norm (without
 *   workspace).
 *   Calls after cudaDeviceReset of a device are not supported: the address
 *   looked up before the reset belongs to the old context.
 *   Errors as gdn_decode_conv_norm; GDN_ERR_UNSUPPORTED if batch * NK >
 *   GDN_NOALLOC_MAX_KEY_HEADS (checked first); then every argument check of
 *   gdn_decode_conv_norm, before any CUDA call (batch 0 returns GDN_OK with
 *   no CUDA call); GDN_ERR_CUDA if the address lookup fails.
 */
#define GDN_NOALLOC_MAX_KEY_HEADS 16384
GDN_API int gdn_decode_conv_norm_noalloc(void *state, gdn_state_dtype state_dtype, int64_t state_pitch,
                                         float *conv_state, int64_t conv_pitch, int taps,
                                         const float *x, const float *conv_w,
                                         const float *br, const float *ar, const float *dt, const float *rate,
                                         const float *z, const float *gn, float l2_eps, float eps,
                                         uint16_t *out,
                                         int batch, int nk, int nv, int d,
                                         int64_t x_stride, int64_t gate_stride, int64_t z_stride,
                                         int64_t out_stride, void *stream);

/*
 * gdn_decode_chunk2 -- two tokens per sequence through the recurrence in one
 * launch (the verify step of speculative decoding), keeping the state after
 * the first token so that a rejected draft token can be rolled back.
 *   Defined by: ssm_gdn_a.rs, launcher `gdn_decode_chunk2` (two tokens per
 *   launch, the intermediate state written for rollback, strides in
 *   elements); the step is gdn.rs `gdn_step`.
 *   state        as gdn_decode; on return it holds the state after BOTH
 *                tokens.
 *   state_mid    [batch] slots of the same dtype, slot pitch mid_pitch >=
 *                NV*D*D elements: written with the state after the FIRST
 *                token (fp16: rounded, as it would be stored between two
 *                calls).
 *   q, k         [2*batch] rows of NK*D; token t of sequence b is row 2b+t.
 *   v            [2*batch] rows of NV*D.  alpha, beta: [2*batch] rows of NV.
 *   o            [2*batch] rows of NV*D fp32 (raw o of each token, no norm).
 *   The result equals two gdn_decode calls on the same kernel path, bit for
 *   bit, while the state is read once instead of twice.
 *   Errors as gdn_decode (state_mid overlapping any operand: GDN_ERR_ALIAS).
 */
GDN_API int gdn_decode_chunk2(void *state, gdn_state_dtype state_dtype, int64_t state_pitch,
                              void *state_mid, int64_t mid_pitch,
                              const float *q, const float *k, const float *v,
                              const float *alpha, const float *beta, float *o,
                              int batch, int nk, int nv, int d,
                              int64_t qk_stride, int64_t v_stride, int64_t gb_stride,
                              int64_t o_stride, void *stream);

/*
 * gdn_prefill_seq -- seq_len tokens per sequence through the recurrence in
 * one launch, token by token in order, the state held on chip between
 * tokens; writes the raw fp32 o of every token (no norm).
 *   Defined by: ssm_gdn_a.rs, launcher `gdn_prefill_regresident`
 *   (token-sequential prefill with the state in registers); the step is
 *   gdn.rs `gdn_step`.
 *   state        as gdn_decode.  An fp16 state is widened to fp32 once when
 *                loaded, carried in fp32 across the tokens and rounded to
 *                fp16 (nearest even) once when stored.
 *   q, k         [batch * seq_len] rows of NK*D, row b*seq_len + t.
 *   v            [batch * seq_len] rows of NV*D.
 *   alpha, beta  [batch * seq_len] rows of NV.
 *   o            [batch * seq_len] rows of NV*D, written.
 *   Splitting seq_len into consecutive calls gives the same result as one
 *   call, up to fp32 rounding order.
 *   Errors as gdn_decode.
 */
GDN_API int gdn_prefill_seq(void *state, gdn_state_dtype state_dtype, int64_t state_pitch,
                            const float *q, const float *k, const float *v,
                            const float *alpha, const float *beta, float *o,
                            int batch, int seq_len, int nk, int nv, int d,
                            int64_t qk_stride, int64_t v_stride, int64_t gb_stride,
                            int64_t o_stride, void *stream);

/*
 * gdn_prefill_chunked -- gdn_prefill_seq computed in chunks of 64 tokens with
 * the chunk's matrix products on the tensor cores.
 *   Defined by: the same recurrence as gdn_prefill_seq (gdn.rs `gdn_step`,
 *   token by token as ssm_gdn_a.rs `gdn_prefill_regresident`), unrolled over
 *   a chunk from the state at its start: with gamma_t the product of the
 *   chunk's alphas up to t and rho(t,i) = gamma_t / gamma_i, the chunk's
 *   deltas solve (I + A) Delta = R, A[t][i] = beta_t rho(t,i) k_t.k_i (i < t),
 *   R[t] = beta_t (v_t - gamma_t S k_t); o_t = (gamma_t S q_t + sum_{i<=t}
 *   rho(t,i) q_t.k_i delta_i) / sqrt(D); at the chunk's end S <- gamma_C S +
 *   sum_t rho(C,t) delta_t k_t^T.  Equal to the token loop in exact
 *   arithmetic; in floating point every product is taken from operands split
 *   into two TF32 parts (three MMAs: about 22 significant bits, 20 where k or
 *   q is an operand), accumulated in fp32, and the state itself is carried
 *   in fp32.
 *   Taken for D == 128 with k and q rows 16-byte aligned (base and stride);
 *   any other call runs gdn_prefill_seq's kernels.  Arguments, layouts,
 *   results (up to fp32 rounding) and errors as gdn_prefill_seq.
 *   The kernel's only waits are on the completion of its own MMAs and of its
 *   own tensor copies (k, q), each bounded; see gdn_device_wait_timeouts.
 */
GDN_API int gdn_prefill_chunked(void *state, gdn_state_dtype state_dtype, int64_t state_pitch,
                                const float *q, const float *k, const float *v,
                                const float *alpha, const float *beta, float *o,
                                int batch, int seq_len, int nk, int nv, int d,
                                int64_t qk_stride, int64_t v_stride, int64_t gb_stride,
                                int64_t o_stride, void *stream);

/*
 * gdn_device_wait_timeouts -- how many times, on the current device since
 * the library was loaded, a tensor-core kernel's bounded wait for its own
 * MMAs or tensor copies ran out (the kernel then stops and writes NaN to its
 * state; 0 in every healthy run).  Synchronises the current device first.  No
 * counterpart on the source pages: a health check of this library's kernels.
 *   count        host pointer, written.
 *   Errors: GDN_ERR_ARG (count NULL), GDN_ERR_CUDA.
 */
GDN_API int gdn_device_wait_timeouts(unsigned *count);

/*
 * gdn_set_wait_polls -- how many times a tensor-core kernel launched after
 * this call polls for the completion of its own MMAs or tensor copies before
 * it gives up (default GDN_DEFAULT_WAIT_POLLS, a second or more).  0 makes
 * every such wait give up at once: the kernel then lets the MMAs and copies
 * it issued finish (bounded by the default), writes NaN to its state, counts
 * the event for gdn_device_wait_timeouts and returns, so the timeout path can
 * be tested without any fault and the context stays usable.  Process-wide; calls that
 * are already launched keep their value.  No counterpart on the source
 * pages.
 */
#define GDN_DEFAULT_WAIT_POLLS 4194304u
GDN_API void gdn_set_wait_polls(unsigned polls);

/*
 * gdn_set_mma_wait_polls -- as gdn_set_wait_polls for the waits on the
 * kernel's own MMAs only; the waits on its tensor copies keep their bound.
 * With 0 here (and the copies' default) the first wait to give up is one for
 * MMAs in flight, so that path can be tested apart from the copies'.  No
 * counterpart on the source pages.
 */
GDN_API void gdn_set_mma_wait_polls(unsigned polls);

/*
 * gdn_h_f32_to_f16 -- n h-state elements binary32 -> binary16, round to
 * nearest, ties to even (overflow to +-inf, subnormals kept, NaN stays NaN).
 *   Defined by: ssm_gdn_a.rs, launcher `ssm_h_state_f32_to_f16`.
 *   src [n] fp32, dst [n] fp16 bits.  src and dst must not overlap
 *   (GDN_ERR_ALIAS): an in-place narrowing conversion would race.
 */
GDN_API int gdn_h_f32_to_f16(const float *src, uint16_t *dst, uint64_t n, void *stream);

/*
 * gdn_h_f16_to_f32 -- n h-state elements binary16 -> binary32, exact.
 *   Defined by: ssm_gdn_a.rs, launcher `ssm_h_state_f16_to_f32`.
 *   src [n] fp16 bits, dst [n] fp32; no overlap (GDN_ERR_ALIAS).
 */
GDN_API int gdn_h_f16_to_f32(const uint16_t *src, float *dst, uint64_t n, void *stream);

/* Human-readable name of a status code (static string, never NULL). */
GDN_API const char *gdn_status_str(int status);

/* The cudaError_t of the last GDN_ERR_CUDA returned on the calling host
 * thread (0 if none). */
GDN_API int gdn_last_cuda_error(void);

#ifdef __cplusplus
}
#endif

#endif /* GDN_H */
