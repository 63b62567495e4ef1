/*
 * gdn.h -- C ABI of libgdn.so, the GB300 (sm_103a) Gated DeltaNet layer hot path.
 *
 * The layer (Qwen3.5-style hybrid models) is a width-4 causal depthwise conv1d with SiLU
 * over the packed q||k||v channels, followed by the gated delta rule
 *
 *     S_t = exp(g_t) S_{t-1} (I - beta_t k_t k_t^T) + beta_t v_t k_t^T,   o_t = scale * S_t q_t
 *
 * ("Qwen3.5-27B GPTQ Garbage Inference -- Root Cause Analysis", "Why abliteration failed
 * on Qwen3.5", item 3), run as a chunked prefill over packed variable-length sequences and
 * as a one-token recurrent decode step on fp32 state ("[Feature] Add batch invariance
 * support to GDN_ATTN backend - #45819", Birol's comment, parts 1 and 3).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  * Activations are token-major: [T, H, D] (or [1, T, H, D]); head_first layouts are
 *    rejected by an explicit stride check, never by a "T < H" heuristic ("Fix [Bug]:
 *    Qwen3.5 ... FLA linear attention tensor format mismatch causes gibberish output",
 *    Root Cause).  T = 1 and T < H are legal.
 *  * The recurrent state is fp32 with layout [.., Hv, dk, dv]; element [i][j] is S[j][i]
 *    (S is dv x dk), so o[j] = scale * sum_i state[i][j] q[i].
 *  * The conv state is the three conv inputs that precede the next token, [.., 3, C],
 *    oldest first, in the activation dtype (bf16).
 *  * v-head h reads q/k head h / (Hv / Hk).  g and beta are per v-head, fp32 [T, Hv].
 *  * Every device pointer and stream is owned by the caller.  The library allocates no
 *    device or pinned memory and keeps no global state beyond per-device cached
 *    properties (SM count, kernel attributes set once), driver entry points and the
 *    NVTX function table that the first range resolves.  Inputs are read-only; only the
 *    documented outputs are written.  All calls are asynchronous on `stream` (a
 *    cudaStream_t; NULL = legacy default stream) and may be issued from several host
 *    threads.
 *  * Validation failures return before anything is launched.  Launch failures return
 *    GDN_ERR_CUDA.  Errors found on the device (an out-of-range state index) are
 *    written to the optional device int `status_dev` (0 untouched = OK), which the
 *    caller reads after synchronising; the offending item is skipped, nothing faults.
 *  * Each entry point that validates or launches holds an NVTX range named after itself
 *    (gdn_chunk_prefill, ...) for the duration of the host call, so timeline tools show
 *    every call with the kernels it launched.  With no tool attached a range is a call
 *    through a resolved pointer.
 *  * Results are batch-invariant: each sequence's outputs and states are bit-identical
 *    whatever other sequences share the launch (the reduction order of every value
 *    depends only on that sequence's own data and its position relative to its start).
 */
#ifndef GDN_H_
#define GDN_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    GDN_OK = 0,
    GDN_ERR_NULL = 1,        /* a required pointer is NULL */
    GDN_ERR_SHAPE = 2,       /* inconsistent sizes */
    GDN_ERR_LAYOUT = 3,      /* head-first or otherwise unsupported strides/alignment */
    GDN_ERR_DTYPE = 4,       /* unsupported or mismatched element type */
    GDN_ERR_SEQLENS = 5,     /* cu_seqlens not 0 = c0 <= c1 <= ... <= cN = T */
    GDN_ERR_UNSUPPORTED = 6, /* shape combination without a kernel */
    GDN_ERR_CUDA = 7,        /* a CUDA runtime call failed */
    GDN_ERR_TIMEOUT = 8,     /* a bounded device-side wait gave up (device status) */
    GDN_ERR_WORKSPACE = 9,   /* workspace missing, too small or misaligned */
    GDN_ERR_INDEX = 10,      /* a state index outside [0, P) (device status) */
    GDN_ERR_NONFINITE = 11   /* GDN_CHECK_INPUTS: a gate input is a NaN or an infinity */
} gdn_status_t;

typedef enum { GDN_BF16 = 0, GDN_F32 = 1, GDN_I32 = 2 } gdn_dtype_t;

/* Strided view of an activation tensor.  Strides are in elements.  q/k/v/o must have a
 * unit element stride, a head stride equal to D, a token stride >= H*D that is a multiple
 * of 16 bytes, and a 16-byte aligned base pointer. */
typedef struct {
    void *ptr;
    int32_t ndim;       /* 3: [T,H,D]   4: [1,T,H,D] */
    int32_t dtype;      /* gdn_dtype_t */
    int64_t shape[4];
    int64_t stride[4];
} gdn_tensor_t;

/* Flags */
#define GDN_QK_L2NORM 0x1u /* normalise q and k per head: x / sqrt(sum x^2 + 1e-6) */
/* Debug checks of the inputs (the entries that take flags: the prefills, the decodes and
 * the layer entry), run on the host before anything is launched, waiting for `stream`:
 *  - the gate inputs (g and beta; for gdn_fused_decode the logits a_raw and b_raw) are
 *    copied to pageable host memory, and a NaN or an infinity returns GDN_ERR_NONFINITE.
 *    The recurrence multiplies the state by e^g at every token, so one bad gate ruins
 *    every later state of its sequence ("Qwen3.5-27B GPTQ Garbage Inference -- Root Cause
 *    Analysis", "Why abliteration failed on Qwen3.5", item 3);
 *  - the prefills' device cu_seqlens is copied back and must equal the host copy, else
 *    GDN_ERR_SEQLENS (the kernels index the packed batch by the device copy).
 * It synchronises the stream: not for use under stream capture or on a latency-critical
 * path. */
#define GDN_CHECK_INPUTS 0x1000u

/* Human-readable name of a status code (static storage, never NULL). */
const char *gdn_status_string(gdn_status_t s);

/* Library ABI version (major * 10000 + minor * 100 + patch). */
int32_t gdn_version(void);

/*
 * gdn_conv1d_fwd -- prefill conv over packed sequences.
 * Source: "[Feature] Add batch invariance support to GDN_ATTN backend - #45819", Birol's
 * comment, part 3(a): conv over cat(conv_state, x) with padding 0 and groups = channels,
 * SiLU of the last seq_len outputs, new conv state = last three conv inputs.
 *
 *   y[t,c] = silu(bias[c] + sum_{j=0..3} w[c][j] * xs[t+j][c]),  xs = [state(3) ; x_seq]
 *
 * x [T, C] bf16 contiguous (device); w [C, 4] bf16; bias [C] bf16 or NULL;
 * cu_seqlens_dev / cu_seqlens_host: the same int32 [N+1] offsets on device and host;
 * conv_state_in [N, 3, C] bf16 or NULL (zeros: fresh prefill);
 * conv_state_out [N, 3, C] bf16 or NULL (may equal conv_state_in: updated in place);
 * y [T, C] bf16 contiguous.  C must be a multiple of 8; pointers 16-byte aligned.
 * Sequences with length 0 pass their conv state through unchanged.
 */
gdn_status_t gdn_conv1d_fwd(const void *x, int64_t T, int32_t C, const void *w,
                            const void *bias, const int32_t *cu_seqlens_dev,
                            const int32_t *cu_seqlens_host, int32_t N,
                            const void *conv_state_in, void *conv_state_out, void *y,
                            void *stream);

/*
 * gdn_conv1d_update -- decode conv: one new token per sequence, conv state shifted in
 * place.  Same arithmetic (and the same fp32 operation order) as gdn_conv1d_fwd for that
 * token.  Source: the decode conv update of the same PR comment (causal_conv1d_update).
 *
 * x [N, C] bf16; w [C, 4]; bias [C] or NULL; conv_state [P, 3, C] bf16, in place;
 * state_idx [N] int32 (device) or NULL for identity (then P >= N); y [N, C] bf16.
 * Indices outside [0, P) set *status_dev = GDN_ERR_INDEX and skip that sequence.
 */
gdn_status_t gdn_conv1d_update(const void *x, int32_t N, int32_t C, const void *w,
                               const void *bias, void *conv_state, int32_t P,
                               const int32_t *state_idx, void *y, int32_t *status_dev,
                               void *stream);

/*
 * gdn_chunk_prefill -- chunked gated delta rule over packed variable-length sequences.
 * Source: "[Feature] Add batch invariance support to GDN_ATTN backend - #45819", Birol's
 * comment, part 3(a) (chunk_gated_delta_rule with initial_state, output_final_state and
 * use_qk_l2norm_in_kernel; chunk boundaries on multiples of the 64-token block) and the
 * PR's commit message "Fixes: 2." (per-sequence chunking independent of batch geometry).
 *
 * q, k [T, Hk, dk]; v [T, Hv, dv]; o [T, Hv, dv] (views as described for gdn_tensor_t);
 * g, beta [T, Hv] fp32 contiguous; cu_seqlens_dev / cu_seqlens_host int32 [N+1];
 * initial_state [N, Hv, dk, dv] fp32 or NULL (zeros); final_state [N, Hv, dk, dv] fp32 or
 * NULL (not written).  initial_state == final_state is allowed (updated in place).
 * chunk: the chunk length; chunks are anchored at every sequence start, so a sequence's
 * result never depends on its neighbours, and a continuation split at a multiple of
 * `chunk` reproduces the unsplit run bit for bit.  Zero-length sequences keep their
 * initial state; with T = 0 the views may have no storage and final_state is a copy of
 * initial_state (zeros without one).
 * Kernels: q/k/v bf16 with dk = dv = 128 and chunk = 64 run on the tensor cores
 * (tcgen05, TMEM, TMA); q/k/v bf16 or fp32 with dk = dv in {16, 32, 64, 128} and chunk in
 * {16, 32, 64} run on a CUDA-core fp32 kernel when flags has GDN_PREFILL_SIMT or the
 * shape has no tensor-core kernel.  Anything else returns GDN_ERR_UNSUPPORTED.
 * workspace: device scratch of gdn_chunk_prefill_workspace_size() bytes, 256-byte
 * aligned (may be NULL when that size is 0).
 */
#define GDN_PREFILL_SIMT 0x100u /* force the CUDA-core kernel */
/* Tensor-core kernel only: the state pass splits each head's 128 dv columns into tiles,
 * three (48 + 48 + 32) when 3 * Hv * N CTAs fit the device's SMs in one wave, else two of
 * 64.  These flags force one tiling (tests and tuning); results are bit-identical under
 * either, since no column's arithmetic depends on its tile. */
#define GDN_PREFILL_TILES2 0x200u
#define GDN_PREFILL_TILES3 0x400u
/* gdn_layer_prefill only: fuse the v channels' conv into the scan's state pass. */
#define GDN_LAYER_FUSED_VCONV 0x800u

size_t gdn_chunk_prefill_workspace_size(int32_t N, int64_t T, int32_t Hk, int32_t Hv,
                                        int32_t dk, int32_t dv, int32_t chunk,
                                        uint32_t flags);

gdn_status_t gdn_chunk_prefill(const gdn_tensor_t *q, const gdn_tensor_t *k,
                               const gdn_tensor_t *v, const float *g, const float *beta,
                               const int32_t *cu_seqlens_dev,
                               const int32_t *cu_seqlens_host, int32_t N, int32_t chunk,
                               float scale, uint32_t flags, const float *initial_state,
                               const gdn_tensor_t *o, float *final_state, void *workspace,
                               size_t workspace_bytes, int32_t *status_dev, void *stream);

/*
 * gdn_chunk_prefill_cp -- gdn_chunk_prefill with each sequence split into ranges of
 * range_chunks chunks (64 tokens each) that run side by side: a context-parallel scan
 * for long sequences whose heads alone leave SMs idle.
 * Sources: the recurrence of gdn_chunk_prefill ("Qwen3.5-27B GPTQ Garbage Inference --
 * Root Cause Analysis", "Why abliteration failed on Qwen3.5", item 3).  The per-token
 * update h <- e^g (I - beta k k^T) h + beta k v^T is affine in the state, so a range's end
 * state is P h_start + R; "[Feature] Add batch invariance support to GDN_ATTN backend -
 * #45819" (its commit adding use_cp=False) records that a context-parallel variant chosen
 * by batch composition breaks batch invariance, so here the split is the caller's
 * explicit choice and depends only on each sequence's own length.
 * Method: one prep pass over the ranges; a state pass that gives every range's end state
 * from its first state (the sequence's initial state for a first range, zero otherwise)
 * and every middle range's P (V taken as zero, start = identity); the start states in
 * order (S_{r+1} = P_r S_r + R_r, fp32); a second state pass from those starts, which
 * writes o and the final states.  A sequence of at most range_chunks chunks is one range
 * and gives exactly the bits of gdn_chunk_prefill.  Longer ones match the oracle within
 * the same tolerances but are not bit-identical to gdn_chunk_prefill (the starts come
 * from composed maps); they are bit-identical alone and in any batch, for a given
 * range_chunks.
 * Arguments are those of gdn_chunk_prefill plus range_chunks >= 1; the tensor-core path
 * only (bf16, dk = dv = 128, chunk 64), else GDN_ERR_UNSUPPORTED.  workspace: device
 * scratch of gdn_chunk_prefill_cp_workspace_size() bytes, 256-byte aligned.  A device
 * cu_seqlens that disagrees with the host copy is reported in *status_dev as
 * GDN_ERR_SEQLENS.
 */
size_t gdn_chunk_prefill_cp_workspace_size(const int32_t *cu_seqlens_host, int32_t N,
                                           int64_t T, int32_t Hk, int32_t Hv, int32_t dk,
                                           int32_t dv, int32_t chunk, int32_t range_chunks);

/*
 * gdn_chunk_prefill_cp_range_hint -- a range_chunks for one sequence of seq_len tokens
 * over Hv v-heads run alone on the current device, or 0 when the plain gdn_chunk_prefill
 * is expected to be at least as fast.  A host-side estimate (no launch, no allocation):
 * each state pass is counted as its waves of CTAs (one per SM, the dv tiling of the
 * kernels) times the range length, plus a fixed allowance for the composition; the
 * range length with the lowest count wins.  It depends on seq_len, Hv and the device's
 * SM count only, never on other sequences, so passing it keeps a sequence's bits the
 * same in any batch on that device (a value chosen from a whole batch would not: see
 * gdn_chunk_prefill_cp).  0 also when there is no current device or an argument is not
 * positive.
 */
int32_t gdn_chunk_prefill_cp_range_hint(int64_t seq_len, int32_t Hv);

/* The same estimate for a device with sm_count SMs (e.g. planning for another GPU); no
 * CUDA call is made.  0 when an argument is not positive. */
int32_t gdn_chunk_prefill_cp_range_hint_for(int64_t seq_len, int32_t Hv, int32_t sm_count);

gdn_status_t gdn_chunk_prefill_cp(const gdn_tensor_t *q, const gdn_tensor_t *k,
                                  const gdn_tensor_t *v, const float *g, const float *beta,
                                  const int32_t *cu_seqlens_dev,
                                  const int32_t *cu_seqlens_host, int32_t N, int32_t chunk,
                                  float scale, uint32_t flags, int32_t range_chunks,
                                  const float *initial_state, const gdn_tensor_t *o,
                                  float *final_state, void *workspace, size_t workspace_bytes,
                                  int32_t *status_dev, void *stream);

/*
 * gdn_chunk_prefill_noalloc -- gdn_chunk_prefill without a caller-provided workspace.
 * The pages have no counterpart to this entry point; it exists for callers that cannot
 * call cudaMalloc (an engine whose allocator owns all device memory, a latency-critical
 * loop that must not allocate, a host program with no device allocator of its own).
 *
 * Arguments, results, kernels and errors are those of gdn_chunk_prefill, except that the
 * scratch comes from a fixed array of GDN_NOALLOC_SCRATCH_BYTES inside the library's
 * device image, which every GPU that loads the library holds until the process exits.
 * A tensor-core call needs (ceil(T / 64) + N + 1) * Hv * 17408 bytes (one 17408-byte tile
 * per chunk slot and v-head); one whose size exceeds the array returns GDN_ERR_WORKSPACE
 * before launching anything.  With 48 v-heads that admits up to 160 slots, e.g. one
 * 10112-token sequence or 8 sequences totalling 9664 tokens; fp32 activations (CUDA-core
 * kernel) need no scratch at any size.  The call allocates nothing (no cudaMalloc or
 * cudaFree, no allocating library routine).
 * The first call on a device (with that device current) looks up the array's device
 * address once and caches it; make that first call before any stream capture.
 * Every call shares the one array: calls that overlap on the GPU (on different streams,
 * or from several threads without ordering) race on it and must be serialised by the
 * caller.  Each call writes every scratch byte it later reads, so stale contents from an
 * earlier call do not matter.
 */
#define GDN_NOALLOC_SCRATCH_BYTES (128u << 20)

gdn_status_t gdn_chunk_prefill_noalloc(const gdn_tensor_t *q, const gdn_tensor_t *k,
                                       const gdn_tensor_t *v, const float *g,
                                       const float *beta, const int32_t *cu_seqlens_dev,
                                       const int32_t *cu_seqlens_host, int32_t N,
                                       int32_t chunk, float scale, uint32_t flags,
                                       const float *initial_state, const gdn_tensor_t *o,
                                       float *final_state, int32_t *status_dev,
                                       void *stream);

/*
 * gdn_recurrent_decode -- one token per sequence on a pool of fp32 states, in place.
 * Source: the decode path of "[Feature] Add batch invariance support to GDN_ATTN
 * backend - #45819" (fused_sigmoid_gating_delta_rule_update with ssm_state_indices into
 * the state pool; fp32 recurrent state from Birol's comment, part 1).
 *
 *   h <- exp(g) h;  u = beta (v - h^T k);  h <- h + k u^T;  o = scale * h^T q
 *
 * q, k [N, Hk, dk]; v [N, Hv, dv]; o [N, Hv, dv] (gdn_tensor_t views, T = N);
 * g, beta [N, Hv] fp32; state [P, Hv, dk, dv] fp32, read once and written once;
 * state_idx [N] int32 (device) or NULL for identity (then P >= N).  dk = dv = 128.
 * Indices outside [0, P) set *status_dev = GDN_ERR_INDEX and skip that sequence.
 */
gdn_status_t gdn_recurrent_decode(const gdn_tensor_t *q, const gdn_tensor_t *k,
                                  const gdn_tensor_t *v, const float *g,
                                  const float *beta, float *state, int32_t P,
                                  const int32_t *state_idx, float scale, uint32_t flags,
                                  const gdn_tensor_t *o, int32_t *status_dev,
                                  void *stream);

/*
 * gdn_layer_prefill -- the layer's prefill in one call: gdn_conv1d_fwd over the packed
 * q | k | v channels, then gdn_chunk_prefill on q, k, v as strided views of its output.
 * Sources: those of the two entries it chains; the fused conv follows "[Feature] Add
 * batch invariance support to GDN_ATTN backend - #45819", Birol's comment, part 3(a)
 * (the conv output feeds the scan directly).
 * side_stream: NULL, or a second cudaStream_t of the caller's (it must differ from
 * `stream`).  With NULL everything runs on `stream` in order.
 * With a side stream the conv of the v channels runs on it while the q/k channels' conv
 * and the chunk preparation, which reads only q and k, run on `stream`; the state pass
 * waits for v, and `stream` waits for the side stream before the call returns, so the
 * caller sees one ordered stream (CUDA-graph capture included).  The library owns no
 * stream: the fork and join use two events that this call creates and destroys.  Calls
 * that share a side stream are ordered on it.
 * GDN_LAYER_FUSED_VCONV (tensor-core shapes only, else GDN_ERR_UNSUPPORTED; side_stream
 * is then unused): the conv kernel runs over the q/k channels only, and the scan's state
 * pass convolves each V tile from x itself one chunk ahead, writing it to y and, at the
 * end, the v channels' conv states.  It saves the v channels' round trip through memory
 * but adds its arithmetic to the latency-bound state pass, which makes the call slower
 * on the 27B shapes, so it is not the default.
 * Every path gives exactly the bits of calling the two entries in sequence (y, o,
 * final_state and conv_state_out alike).
 *
 * x [T, C] bf16, C = 2*Hk*dk + Hv*dv, rows contiguous; y [T, C] bf16 receives the conv
 * output; o [T, Hv, dv] bf16 contiguous; everything else as in gdn_conv1d_fwd and
 * gdn_chunk_prefill with chunk = 64 (flags may hold GDN_QK_L2NORM, GDN_PREFILL_SIMT and
 * the tiling flags).
 */
gdn_status_t gdn_layer_prefill(const void *x, int64_t T, int32_t Hk, int32_t Hv,
                               int32_t dk, int32_t dv, const void *conv_w,
                               const void *conv_bias, const int32_t *cu_seqlens_dev,
                               const int32_t *cu_seqlens_host, int32_t N,
                               const void *conv_state_in, void *conv_state_out, void *y,
                               const float *g, const float *beta, float scale, uint32_t flags,
                               const float *initial_state, void *o, float *final_state,
                               void *workspace, size_t workspace_bytes, int32_t *status_dev,
                               void *side_stream, void *stream);

/*
 * gdn_fused_decode -- the whole decode step of one token per sequence in one call:
 * conv update, q/k/v split, optional q/k L2 norm, gates from raw logits, recurrent step.
 * One kernel does all of it per (sequence, v-head); a second, small one then shifts the
 * conv-state rows of the q and k channels, which several v-heads read.
 * Source: the decode path of "[Feature] Add batch invariance support to GDN_ATTN
 * backend - #45819", which names the fused_sigmoid_gating_delta_rule_update entry
 * and the state pool indexed by ssm_state_indices; the pages give the name only, so the
 * gates are taken in their plainest form:
 *
 *   beta = sigmoid(b_raw),   g = -softplus(a_raw)   (so exp(g) = 1 / (1 + exp(a_raw)))
 *
 * followed by exactly gdn_conv1d_update and gdn_recurrent_decode (same conv bits, the
 * conv output rounded to bf16 before use).
 *
 * x [N, C] bf16 with C = 2*Hk*dk + Hv*dv channels in the order q | k | v, rows contiguous;
 * conv_w [C, 4] bf16; conv_bias [C] bf16 or NULL; conv_state [P, 3, C] bf16, shifted in
 * place; a_raw, b_raw [N, Hv] fp32; state [P, Hv, dk, dv] fp32, read once and written
 * once; state_idx [N] int32 (device, one slot for both pools) or NULL for identity (then
 * P >= N); o [N, Hv, dv] bf16, rows contiguous.  dk = dv = 128 and Hv % Hk == 0.  All
 * pointers 16-byte aligned.  Two tokens of one call must not share a slot.  Indices
 * outside [0, P) set *status_dev = GDN_ERR_INDEX and skip that sequence.
 */
gdn_status_t gdn_fused_decode(const void *x, int32_t N, int32_t Hk, int32_t Hv, int32_t dk,
                              int32_t dv, const void *conv_w, const void *conv_bias,
                              void *conv_state, const float *a_raw, const float *b_raw,
                              float *state, int32_t P, const int32_t *state_idx, float scale,
                              uint32_t flags, void *o, int32_t *status_dev, void *stream);

/* gdn_selftest_bounded_wait -- checks the failure path of the bounded waits.  Every wait
 * of the tensor-core kernels on an mbarrier (a TMA copy or an MMA completing) gives up
 * after 2 s; the CTA then records GDN_ERR_TIMEOUT in the status word, stops issuing work,
 * frees its TMEM and returns, so the context stays usable.  This entry launches one CTA
 * that waits, with the same helper, on a barrier phase that nothing completes: about 2 s
 * later it sets *status_dev = GDN_ERR_TIMEOUT (first writer wins) and exits.
 * status_dev: device int32, required (NULL: GDN_ERR_NULL, nothing launched).
 */
gdn_status_t gdn_selftest_bounded_wait(int32_t *status_dev, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* GDN_H_ */
