/*
 * gdn.h -- C ABI of the gated delta-rule (GDN) library for NVIDIA GB300 (sm_103a).
 *
 * The library computes the gated delta-rule linear-attention recurrence named
 * in the "Background" section of the "GDN CTE Kernel API Reference" page:
 * for every batch b, value head h (reading query/key head h / (Hv/Hk)) and
 * token t,
 *
 *     S_t = exp(g_t) S_{t-1} + beta_t k_t (v_t - exp(g_t) S_{t-1}^T k_t)^T
 *     o_t = scale * S_t^T q_t
 *
 * with an fp32 state S of shape [Dk, Dv].  Two entry points compute it:
 * a chunk-parallel prefill over a whole sequence (gdn_prefill) and one
 * single-token step (gdn_decode_step).
 *
 * Conventions shared by every call:
 *   - All tensor pointers are DEVICE pointers to contiguous row-major memory
 *     owned by the caller; the library never allocates, frees or keeps them.
 *   - Work is enqueued on `stream`; calls return before the GPU finishes.
 *     Host-side argument checks run first: when one fails, nothing is launched
 *     and the error code is returned.  Asynchronous kernel faults surface at
 *     the caller's next synchronisation; kernel-side wait timeouts are recorded
 *     in a per-device status word read by gdn_device_status().
 *   - Preconditions the library does NOT check: q and k are L2-normalised per
 *     token ("GDN CTE Kernel API Reference", Notes), g_log <= 0 (Parameters /
 *     g_log), beta in (0, 1) (Parameters / beta), and the buffers do not overlap
 *     except state_inout with itself.
 */
#ifndef GDN_H
#define GDN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same handle as cudaStream_t / CUstream; NULL is the legacy default stream. */
typedef struct CUstream_st* gdn_stream_t;

typedef enum {
    GDN_OK = 0,
    GDN_ERR_NULL = 1,        /* a required pointer is NULL                                  */
    GDN_ERR_DIMS = 2,        /* dims inconsistent with the pages' constraints (see gdn_dims) */
    GDN_ERR_UNSUPPORTED = 3, /* allowed by the pages but not implemented by this build      */
    GDN_ERR_ALIGN = 4,       /* a tensor pointer is not 16-byte aligned                     */
    GDN_ERR_CUDA = 5,        /* a CUDA call (launch, attribute, tensor-map encode) failed    */
    GDN_ERR_TIMEOUT = 6,     /* a kernel wait ran past its bound (device status only)        */
    GDN_ERR_WORKSPACE = 7    /* a caller workspace smaller than the call needs              */
} gdn_status;

/* Compute dtype = dtype of q, k, v and out ("GDN CTE Kernel API Reference",
 * Parameters / query: the query's dtype sets the compute dtype).  g_log, beta
 * and the state are always fp32. */
typedef enum { GDN_F32 = 0, GDN_BF16 = 1 } gdn_dtype;

enum {
    /* The "omitted" recurrent_state form (Parameters / recurrent_state): start
     * from a zero state and emit no load.  state_inout is still required and
     * receives the final state. */
    GDN_ZERO_INITIAL_STATE = 1u << 0,
    /* Run the prefill on the fp32 FFMA kernel even where the tensor-core kernel
     * applies (a cross-check path; same results within fp32 rounding). */
    GDN_FORCE_FFMA = 1u << 1,
    /* Never split a sequence into segments (see gdn_prefill): one pass over
     * every sequence, whatever the SM count, so results do not depend on it. */
    GDN_SINGLE_PASS = 1u << 2
};

/*
 * Problem sizes ("GDN CTE Kernel API Reference", Dimensions and Notes):
 *   B  >= 0 batch (0: nothing to do);  Hk >= 1 key/query heads;
 *   Hv >= 1 value heads with Hv % Hk == 0;
 *   S  >= 0 tokens for the prefill (0: no tokens, the state is left as it is,
 *      or zeroed under GDN_ZERO_INITIAL_STATE); the decode step requires S == 1;
 *   Dk, Dv in [1, 128] head dims (Dq == Dk: q and k share Dk).
 * Violations return GDN_ERR_DIMS.  The pages' S % 128 rule belongs to their
 * Trainium algorithm choice; this library accepts any S.  When B == 0 or
 * S == 0, q, k, v, g_log, beta and out may be NULL.
 */
typedef struct {
    int64_t B, Hk, Hv, S, Dk, Dv;
    int32_t dtype;   /* gdn_dtype */
    uint32_t flags;  /* GDN_ZERO_INITIAL_STATE | GDN_FORCE_FFMA | GDN_SINGLE_PASS */
} gdn_dims;

/*
 * gdn_prefill -- chunk-parallel prefill of the recurrence over S tokens.
 * ("GDN CTE Kernel API Reference", API Reference / gdn_cte: Parameters, Returns.)
 *
 *   q           [B, Hk, S, Dk]  compute dtype, token-major, L2-normalised rows
 *   k           [B, Hk, S, Dk]  compute dtype, token-major, L2-normalised rows
 *   v           [B, Hv, S, Dv]  compute dtype
 *   g_log       [B, Hv, S]      fp32 per-token log-decay (negative)
 *   beta        [B, Hv, S]      fp32 per-token update strength in (0, 1)
 *   scale       query scale, applied on the device (typically 1/sqrt(Dk))
 *   state_inout [B, Hv, Dk, Dv] fp32, Dv contiguous.  Read as the initial state
 *               (unless GDN_ZERO_INITIAL_STATE) and overwritten in place with the
 *               final state (the page's aliased in/out recurrent_state).
 *   out         [B, Hv, S, Dv]  compute dtype, head-major, un-normalised
 *
 * Every pointer must be non-NULL and 16-byte aligned.  Returns GDN_OK once the
 * work is enqueued.  Implementation: Dk = Dv = 128 with bf16 runs on the
 * tcgen05 tensor-core kernel; every other supported shape and fp32 compute run
 * on the FFMA kernel.
 *
 * Few long sequences (on the tensor-core path) are split into P >= 2 segments
 * unless GDN_SINGLE_PASS is set, when a host-side model of the launch (one CTA
 * per SM, CTAs dispatched in order) predicts that it saves at least a tenth of
 * one pass; gdn_prefill_segment_starts reports the split.  The recurrence is
 * affine in its start state: a later segment's end state is M S0 + X and its
 * output at token t is out_0[t] + C[t] S0, with X and out_0 its end state and
 * outputs from a zero start and M and C (C[t]: 1 x Dk per token) its end state
 * and outputs from S0 = I with v = 0.  Four kernel launches and a memset: an
 * identity matrix and a zero v tile; one launch of segment 0 from the real
 * start state and both runs of every later
 * segment (out_0 is written to out, C to the scratch); a combine step that
 * chains the maps into every segment's start state and the final state
 * (fp32); a correction that adds C[t] S0 to the later segments' outputs
 * (tcgen05, S0 rounded to bf16; the sum rounded once to bf16).  The scratch
 * (gdn_prefill_workspace_bytes: 3 (P - 1) states per sequence, one identity,
 * and C for every token after segment 0) is allocated with cudaMallocAsync on
 * `stream` and freed there; if that allocation fails, the call runs one pass
 * instead.  The results agree with the one-pass form to within rounding (a
 * similar error against an fp64 reference, from strong decay to none), not bit
 * for bit; segment 0's outputs are those of one pass.
 */
gdn_status gdn_prefill(const void* q, const void* k, const void* v,
                       const float* g_log, const float* beta, float scale,
                       float* state_inout, void* out,
                       const gdn_dims* dims, gdn_stream_t stream);

/*
 * gdn_decode_step -- one token of the recurrence (the prefill at S = 1), the
 * core of the single-token step of the "GDN Block TKG Kernel API Reference"
 * page (its recurrent_state [B, num_v_heads, head_k_dim, head_v_dim] fp32).
 * Same arguments and layouts as gdn_prefill with dims->S == 1 (else
 * GDN_ERR_DIMS).  The state is updated in place: each fp32 state element is
 * read once and written once.
 */
gdn_status gdn_decode_step(const void* q, const void* k, const void* v,
                           const float* g_log, const float* beta, float scale,
                           float* state_inout, void* out,
                           const gdn_dims* dims, gdn_stream_t stream);

/*
 * gdn_decode_gated -- the gated single-token step of the decode block: the
 * decode prologue, one token of the recurrence, and the RMSNormGated output
 * epilogue ("GDN Block TKG Kernel API Reference": gdn_block_tkg Parameters
 * A_log, dt_bias, norm_weight and the z / a / b in_proj outputs; Returns
 * "RMSNormGated decode output").  The page names these inputs but prints no
 * formulas; this library reads them as (eps_l2 = eps_rms = 1e-6):
 *
 *     q^ = q / sqrt(|q|^2 + eps_l2),  k^ likewise (q and k need NOT be normalised)
 *     g  = -exp(A_log[h]) * softplus(a[b, h] + dt_bias[h]),   beta = sigmoid(b[b, h])
 *     (o, S') = the recurrence step of gdn_decode_step on q^, k^, v, g, beta, scale
 *     y  = o / sqrt(mean over Dv of o^2 + eps_rms) * norm_weight * silu(z)
 *
 *   qkv          [B, 2*Hk*Dk + Hv*Dv]  compute dtype: the post-conv q | k | v row
 *                (q [Hk, Dk] head-major, then k [Hk, Dk], then v [Hv, Dv])
 *   z            [B, Hv*Dv]  compute dtype, output gate
 *   a, b         [B, Hv]     compute dtype, raw decay-gate and beta inputs
 *   A_log, dt_bias [Hv] fp32;  norm_weight [Dv] fp32
 *   state_inout  [B, Hv, Dk, Dv] fp32, updated in place (GDN_ZERO_INITIAL_STATE
 *                starts from zeros)
 *   out          [B, Hv*Dv]  compute dtype, y
 * dims as for gdn_decode_step (S == 1, Dk, Dv <= 128, Hv % Hk == 0).  Pointers
 * must be non-NULL and aligned to their element size; the state takes 128-bit
 * accesses when it is 16-byte aligned and Dv % 4 == 0.
 */
#define GDN_L2NORM_EPS 1e-6f
#define GDN_RMSNORM_EPS 1e-6f
gdn_status gdn_decode_gated(const void* qkv, const void* z, const void* a, const void* b,
                            const float* A_log, const float* dt_bias, const float* norm_weight,
                            float scale, float* state_inout, void* out,
                            const gdn_dims* dims, gdn_stream_t stream);

/*
 * Depthwise causal conv1d + SiLU in front of the recurrence, with its conv_state
 * ("GDN Conv1D Kernel API Reference": gdn_conv1d_prefill, gdn_conv1d_decode;
 * Parameters, Returns, Notes).  Every channel is an independent K-tap FIR over
 * the raw (pre-convolution) q|k|v activations:
 *
 *     out[b, c, t] = silu( sum_{m=0}^{K-1} w[c, K-1-m] x[b, c, t-m] ),   silu(z) = z / (1 + e^-z)
 *
 * (weight[c, K-1] multiplies the current token, as in a depthwise Conv1d).
 *
 *   B >= 0 batch (0: nothing to do);  C >= 1 channels;  T >= 0 tokens for the
 *   prefill, T == 1 for the decode step;  K in [1, 8] taps (more returns
 *   GDN_ERR_UNSUPPORTED);  dtype = gdn_dtype of x, out and conv_state; the
 *   weights are fp32.  flags must be 0.
 */
typedef struct {
    int64_t B, C, T, K;
    int32_t dtype;   /* gdn_dtype */
    uint32_t flags;  /* 0 */
} gdn_conv_dims;

/*
 * gdn_conv1d_prefill -- the whole sequence, starting from zeros (the prefill
 * takes no previous window).
 *   mixed           [B, C, T]  dtype, raw input, tokens contiguous per channel
 *   conv_weight     [C, K]     fp32
 *   out             [B, C, T]  dtype, silu(causal conv)
 *   conv_state_out  [B, C, K]  dtype, the last K raw tokens of mixed,
 *                   right-aligned behind zeros when T < K (written when T == 0 too)
 * Pointers must be non-NULL (x and out may be NULL when T == 0 or B == 0) and
 * aligned to their element size (else GDN_ERR_ALIGN).  bf16 rows with T % 8 == 0
 * and 16-byte aligned x / out take the vectorised path.
 */
gdn_status gdn_conv1d_prefill(const void* mixed, const float* conv_weight, void* out, void* conv_state_out,
                              const gdn_conv_dims* dims, gdn_stream_t stream);

/*
 * gdn_conv1d_decode -- one token.
 *   x                 [B, C, 1]  dtype, the current raw token
 *   conv_weight       [C, K]     fp32
 *   conv_state_inout  [B, C, K]  dtype, the previous window; overwritten in place
 *                     with the shifted window (the previous one without its
 *                     oldest token, then x)
 *   out               [B, C, 1]  dtype, silu(sum_k w[c, k] window[k])
 * dims->T must be 1 (else GDN_ERR_DIMS).
 */
gdn_status gdn_conv1d_decode(const void* x, const float* conv_weight, void* conv_state_inout, void* out,
                             const gdn_conv_dims* dims, gdn_stream_t stream);

/*
 * The decode block without its output projection ("GDN Block TKG Kernel API
 * Reference": gdn_block_tkg Parameters, Returns, Notes; the data flow "in_proj
 * matmuls -> gdn_conv1d_decode -> split conv_out + GQA-repeat q,k -> gdn_tkg"):
 * the four input projections of one token's hidden state, the conv1d decode step
 * on the q|k|v channels, and the gated single-token step (gdn_decode_gated, with
 * the query scale 1/sqrt(Dk), the page having no scale argument).
 *
 *   B in [0, 256]; H (hidden size) a multiple of 64; Hk, Hv, Dk, Dv as for
 *   gdn_decode_step; K in [1, 8] conv taps; dtype GDN_BF16 (the page's bf16
 *   weights and activations; others return GDN_ERR_UNSUPPORTED); flags 0.
 *   conv_dim C = 2*Hk*Dk + Hv*Dv; value_dim = Hv*Dv; C, value_dim and Hv must be
 *   multiples of 8 (row pitches of 16 bytes).
 */
typedef struct {
    int64_t B, H, Hk, Hv, Dk, Dv, K;
    int32_t dtype;   /* GDN_BF16 */
    uint32_t flags;  /* 0 */
} gdn_block_dims;

/* Size of the fixed scratch array that gdn_decode_block_noalloc uses (4 MiB). */
#define GDN_NOALLOC_SCRATCH_BYTES ((size_t)4 << 20)

/* Device workspace bytes gdn_decode_block needs (the inter-stage activations z,
 * a, b in bf16, and a work counter of the gated step); 0 for invalid dims. */
size_t gdn_decode_block_workspace_bytes(const gdn_block_dims* dims);

/*
 * gdn_decode_block -- one token through the block.
 *   hidden            [B, 1, H] bf16
 *   W_qkv             [H, C] bf16, W_z [H, value_dim] bf16, W_a, W_b [H, Hv] bf16
 *                     (each == nn.Linear.weight.T)
 *   conv_weight       [C, K] fp32;  conv_state_inout [B, C, K] bf16, shifted in place
 *   A_log, dt_bias    [Hv] fp32;    norm_weight [Dv] fp32
 *   state_inout       [B, Hv, Dk, Dv] fp32, updated in place
 *   out               [B, 1, value_dim] bf16, the RMSNormGated output
 *   workspace         device memory of at least gdn_decode_block_workspace_bytes,
 *                     16-byte aligned, owned by the caller (else GDN_ERR_DIMS)
 * hidden, the weights and the workspace must be 16-byte aligned, every other
 * pointer aligned to its element (GDN_ERR_ALIGN); all checks run before the
 * first launch.  Launches two kernels on `stream`: the projections (whose
 * q|k|v epilogue shifts the conv windows in place), then the gated step, which
 * takes the conv1d output from the shifted windows and starts loading the state
 * while the projections run (programmatic dependent launch).
 */
gdn_status gdn_decode_block(const void* hidden, const void* W_qkv, const void* W_z, const void* W_a,
                            const void* W_b, const float* conv_weight, void* conv_state_inout,
                            const float* A_log, const float* dt_bias, const float* norm_weight,
                            float* state_inout, void* out, void* workspace, size_t workspace_bytes,
                            const gdn_block_dims* dims, gdn_stream_t stream);

/*
 * gdn_decode_block_noalloc -- gdn_decode_block for callers that cannot allocate
 * device memory: a runtime that owns every byte of the device and hands out no
 * buffers to kernels it does not know, a plugin whose host code must not call the
 * CUDA allocator, or a serving loop that may not risk an allocation (which can
 * synchronise the device or fail under memory pressure) while it runs.  The
 * pages' block kernel has no such variant; it exists for this library's callers.
 *
 * Arguments and results are those of gdn_decode_block without the workspace: the
 * inter-stage scratch (z, a, b in bf16 and the gated step's head counter) lives
 * in a fixed array inside the library, GDN_NOALLOC_SCRATCH_BYTES bytes, of which
 * every CUDA device that loads the library keeps one copy until the process
 * exits.  Dims whose scratch, gdn_decode_block_workspace_bytes, exceeds that size
 * return GDN_ERR_UNSUPPORTED and launch nothing (for the workloads here, B = 64
 * and value_dim = 4096 need 0.5 MiB; B = 256 with value_dim = 4096 about 2 MiB).
 * The call allocates nothing: no cudaMalloc, cudaFree or allocating library
 * routine.
 *
 * The first call on a device looks up the array's device address
 * (cudaGetSymbolAddress, with that device current) and caches it; make that first
 * call before any stream capture on the device.  Every call on a device shares
 * the one array, and the array keeps the previous call's contents: each call
 * rewrites z, a and b and clears the counter before reading them, so results do
 * not depend on earlier calls, but two calls whose kernels overlap on the GPU
 * (different streams, or different host threads, without ordering between them)
 * race on the array and give wrong results.  Serialise such calls on one stream.
 */
gdn_status gdn_decode_block_noalloc(const void* hidden, const void* W_qkv, const void* W_z, const void* W_a,
                                    const void* W_b, const float* conv_weight, void* conv_state_inout,
                                    const float* A_log, const float* dt_bias, const float* norm_weight,
                                    float* state_inout, void* out, const gdn_block_dims* dims, gdn_stream_t stream);

/*
 * gdn_rmsnorm_gated -- the RMSNormGated output epilogue ("GDN Block TKG Kernel
 * API Reference": Returns, "RMSNormGated decode output"; norm_weight, the
 * "RMSNormGated weight") over `rows` rows of D elements:
 *     out[r, :] = x[r, :] / sqrt(mean(x[r, :]^2) + GDN_RMSNORM_EPS) * norm_weight * silu(z[r, :])
 *   x, z, out   [rows, D] in `dtype` (GDN_BF16 or GDN_F32), element-aligned;
 *               out may be x (in place)
 *   norm_weight [D] fp32
 * rows >= 0, 1 <= D <= 4096.  One launch on `stream`.
 */
gdn_status gdn_rmsnorm_gated(const void* x, const void* z, const float* norm_weight, void* out, int64_t rows,
                             int64_t D, int32_t dtype, gdn_stream_t stream);

/*
 * gdn_prefill_gated -- gdn_prefill followed by gdn_rmsnorm_gated on its output,
 * per token and value head over Dv (the decode block's RMSNormGated applied to
 * every token of a prefill):
 *   z           [B, Hv, S, Dv] in the compute dtype (head-major, like out)
 *   norm_weight [Dv] fp32
 *   the other arguments as gdn_prefill; out receives the gated output.
 * Every check of both steps runs before the first launch.  Launches the
 * prefill's kernel, then one normalisation pass that reads the output and z
 * and rewrites the output in place.
 */
gdn_status gdn_prefill_gated(const void* q, const void* k, const void* v, const float* g_log, const float* beta,
                             const void* z, const float* norm_weight, float scale, float* state_inout, void* out,
                             const gdn_dims* dims, gdn_stream_t stream);

/* Device scratch a prefill with these dims needs on the current device: the
 * segment states, maps and identity-start outputs of a split (see gdn_prefill;
 * the split depends on the device's SM count), 0 when the call runs one pass.  0 as well for
 * invalid dims or when no CUDA device can be queried.  Host only. */
size_t gdn_prefill_workspace_bytes(const gdn_dims* dims);

/*
 * gdn_prefill_ws -- gdn_prefill with the scratch of a split supplied by the
 * caller.  No counterpart on the pages (their kernels allocate nothing the
 * caller sees); it exists so that a split prefill need not allocate.
 *   workspace        device memory of workspace_bytes >= gdn_prefill_workspace_bytes(dims)
 *                    bytes on the current device, 16-byte aligned, owned by the caller
 *                    and not touched by anything else until the call's work on `stream`
 *                    has finished; NULL: the call behaves exactly like gdn_prefill
 *                    (stream-ordered scratch of its own)
 * A non-NULL workspace that is too small returns GDN_ERR_WORKSPACE (misaligned:
 * GDN_ERR_ALIGN) and launches nothing.  Results are bit-identical to gdn_prefill's.
 */
gdn_status gdn_prefill_ws(const void* q, const void* k, const void* v,
                          const float* g_log, const float* beta, float scale,
                          float* state_inout, void* out, const gdn_dims* dims,
                          void* workspace, size_t workspace_bytes, gdn_stream_t stream);

/* Segments gdn_prefill splits each sequence into for these dims on a device
 * with sm_count SMs (see gdn_prefill): 1 for one pass (every shape off the
 * tensor-core path, GDN_FORCE_FFMA, GDN_SINGLE_PASS, B == 0 or S == 0),
 * otherwise 2 .. 16.  0 for invalid dims or sm_count < 1.  Host only. */
int32_t gdn_prefill_segments(const gdn_dims* dims, int32_t sm_count);

/* gdn_prefill_segments, and where the segments start: with starts != NULL and
 * capacity >= P + 1 (P the return value), starts[j] is the first token of
 * segment j (starts[0] = 0) and starts[P] = S.  Segment 0 may be longer than
 * the others; segments 1 .. P - 2 have the same multiple of 128 tokens and the
 * last one ends at S.  No counterpart on the pages.  Host only. */
int32_t gdn_prefill_segment_starts(const gdn_dims* dims, int32_t sm_count, int64_t* starts, int32_t capacity);

/* Static, NUL-terminated description of a status code. */
const char* gdn_status_string(gdn_status s);

/*
 * gdn_device_status -- read (and, when clear != 0, reset to 0) the kernel-side
 * status word of CUDA device `device`.  0 means no kernel reported a problem;
 * otherwise the value is a gdn_status (GDN_ERR_TIMEOUT).  Synchronises the
 * device.  Returns GDN_ERR_NULL if code is NULL, GDN_ERR_CUDA if the copy fails.
 */
gdn_status gdn_device_status(int device, int clear, int32_t* code);

/*
 * gdn_set_wait_limit_ns -- the time after which a wait inside the tensor-core
 * prefill (gdn_prefill on bf16 with Dk = Dv = 128) gives up, on CUDA device
 * `device`: ns > 0 sets it, 0 restores the default of one second.  A wait that
 * gives up records GDN_ERR_TIMEOUT in the status word (gdn_device_status), the
 * CTA's roles stop, every copy and product already in flight is drained (those
 * drains keep their own one-second bound) and the CTA frees its tensor memory
 * and exits; the outputs of such a call are undefined.  This exists to exercise
 * that path without a GPU fault (a limit of a few microseconds makes ordinary
 * waits run out); it synchronises the device.  The pages define no such knob.
 * Returns GDN_ERR_CUDA if the device cannot be selected or the value not set.
 */
gdn_status gdn_set_wait_limit_ns(int device, uint64_t ns);

/*
 * gdn_test_stall_prefill -- test hook for the path above, on CUDA device `device`:
 * while on != 0, every CTA of the tensor-core prefill first waits on a barrier
 * that nothing arrives at, so that the wait runs out after the wait limit (set
 * it low with gdn_set_wait_limit_ns) and the call takes its give-up path:
 * GDN_ERR_TIMEOUT in the status word, nothing computed.  No GPU fault is
 * involved.  Synchronises the device.  Off by default; the pages define no
 * such hook.  Returns GDN_ERR_CUDA if the device cannot be selected or the
 * value not set.
 */
gdn_status gdn_test_stall_prefill(int device, int on);

/* Number of kernels one call of gdn_prefill (in one pass), gdn_decode_step,
 * gdn_decode_gated or the conv1d entry points launches: one.  A split prefill
 * launches four, gdn_decode_block and gdn_prefill_gated two. */
int gdn_kernels_per_call(void);

#ifdef __cplusplus
}
#endif

#endif /* GDN_H */
