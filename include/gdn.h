/*
 * gdn.h -- C ABI of the GB300 (sm_103a) GatedDeltaNet mixer library.
 *
 * The mixer (haskell-infer-demo README, "Highlights": "GatedDeltaNet layers
 * (causal conv1d, gated delta rule, gated RMSNorm)"; "Architecture":
 * kernels/gdn_conv.cu, kernels/fla_gdn.cu, kernels/gdn_norm.cu) is, per token
 * t of a sequence and per v-head h (q/k head kh = h / (HV/HK)):
 *
 *   x^_t   = SiLU( sum_{j=0..3} w[c][j] * x_{t-3+j}[c] )        width-4 causal conv
 *   q, k   = q_scale * q / |q|, k / |k|   (|x| = sqrt(sum x^2 + l2_eps))
 *   g_t    = -exp(A_log[h]) * softplus(u_t + dt_bias[h]),  a_t = exp(g_t)
 *   b_t    = sigmoid(b_logit_t)
 *   S_t    = a_t S_{t-1} (I - b_t k_t k_t^T) + b_t v_t k_t^T,   o_t = S_t q_t
 *   y_t    = o_t / sqrt(mean(o_t^2) + norm_eps) * norm_w * SiLU(z_t)
 *
 * The pages name these steps without printing their formulas; the forms above
 * are the standard statements, and the readings taken where the pages are
 * silent (L2 eps placement, q_scale = 1, norm weight used as w and not 1+w,
 * GQA grouping by consecutive v-heads) are listed in the design notes.
 *
 * Interface properties (hyperflare core-design, prepared short-convolution
 * interface list: packed prefill and single-token decode, caller-owned state,
 * explicit request-to-slot mapping, fixed capacities, inactive lanes write no
 * state, capture-safe with no host read of sequence lengths; negative slot
 * mappings suppress writes; "Main KV / GDN recurrence: BF16 / FP32";
 * steady-state serving performs no CUDA allocations):
 *
 *  - Every pointer argument is a DEVICE pointer unless its comment says HOST.
 *    The caller owns all buffers, the workspace and the stream.  The library
 *    allocates no device memory in any call, never synchronises the stream
 *    (except gdn_device_error) and never reads device data on the host, so
 *    every call may be captured into a CUDA graph.
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).
 *  - Packed tokens: cu_seqlens is int32 [n_seqs + 1], cu_seqlens[0] = 0,
 *    non-decreasing, cu_seqlens[n_seqs] = T.  Sequences may be empty.
 *  - state_idx (nullable, int32 [n_seqs]) maps sequence n to a state slot;
 *    NULL means slot n.  A negative entry marks a padding lane: no state or
 *    conv history of it is read or written, and its outputs are zero.
 *  - Recurrent state: fp32 [slots][HV][dk][dv]; element (i, j) of head h holds
 *    S[j][i] (S is dv x dk; the buffer stores S transposed, so the dk index is
 *    the slow one).  Conv history: act dtype [slots][CH][3], oldest tap first.
 *  - Channels of the raw projection x: [q (HK*dk) | k (HK*dk) | v (HV*dv)],
 *    head-major, CH = 2*HK*dk + HV*dv.  Row strides (ld_*) are in ELEMENTS.
 *    Wide views (x, z, q, k, v) need 16-byte aligned bases and strides that
 *    are multiples of 8 elements; the narrow [T][HV] views u and b_logit need
 *    only element alignment and ld >= HV.  Conv weights, the norm weight,
 *    states, histories, workspaces and outputs need 16-byte aligned bases.
 *  - The live (non-negative) entries of state_idx must be distinct within a
 *    call: two sequences writing one slot race.
 *  - Outputs never alias inputs, except state_out == state_in (in place).
 *
 * Errors: every entry point validates its arguments on the host BEFORE any
 * launch and returns GDN_ERR_INVALID_ARG / GDN_ERR_UNSUPPORTED /
 * GDN_ERR_WORKSPACE without touching the GPU.  A failed launch returns
 * GDN_ERR_CUDA.  Faults the kernels detect on the device (cu_seqlens that are
 * not monotone or exceed T, a state slot index >= n_slots, a bounded wait that
 * ran out) never trap: the kernel records a code in a device error word, skips
 * the affected work and returns; gdn_device_error() reads and clears it.
 */
#ifndef GDN_GB300_H
#define GDN_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum gdn_status {
    GDN_OK = 0,
    GDN_ERR_INVALID_ARG = 1, /* null required pointer, bad size, bad stride or alignment */
    GDN_ERR_UNSUPPORTED = 2, /* valid but not built: head dims, chunk, GQA ratio */
    GDN_ERR_WORKSPACE = 3,   /* workspace missing or smaller than gdn_workspace_size() */
    GDN_ERR_CUDA = 4,        /* a CUDA runtime call or launch failed */
    GDN_ERR_DEVICE = 5       /* a kernel reported a device-side fault (gdn_device_error) */
} gdn_status;

typedef enum gdn_dtype { GDN_BF16 = 0, GDN_FP32 = 1 } gdn_dtype;

/* Device error codes reported through gdn_device_error(). */
#define GDN_DEVERR_NONE 0u
#define GDN_DEVERR_CU_SEQLENS 1u   /* cu_seqlens not monotone or beyond T */
#define GDN_DEVERR_SLOT 2u         /* state_idx entry >= n_slots */
#define GDN_DEVERR_TIMEOUT 4u      /* a bounded device wait gave up */

/* Flags for gdn_chunk_prefill / gdn_recurrent_decode. */
#define GDN_FLAG_L2NORM_QK 1u      /* normalise q and k in the kernel (and apply q_scale) */

typedef struct gdn_config {
    int32_t hk, hv;      /* q/k heads, v heads; hv % hk == 0, hv/hk in {1,2,4} */
    int32_t dk, dv;      /* head dims; dk == dv in {32, 64, 128} */
    int32_t chunk;       /* prefill chunk length: 16 or 64 */
    gdn_dtype act;       /* dtype of x, z, u, b_logit, conv weights and conv history */
    int32_t n_slots;     /* number of state / conv-history slots (capacity) */
    float q_scale;       /* multiplies q after its L2 norm (1.0 = plain rule) */
    float l2_eps;        /* 1e-6 */
    float norm_eps;      /* 1e-6 */
} gdn_config;

/* Arguments of the fused mixer entry points (one struct so that the C ABI
 * stays stable as layouts grow). */
typedef struct gdn_mixer_io {
    const void *x;            /* [T][ld_x] act: raw projected q|k|v channels */
    int64_t ld_x;
    const void *z;            /* [T][ld_z] act: gate input of the norm, HV*dv channels */
    int64_t ld_z;
    const void *u;            /* [T][ld_ub] act: decay projection, HV channels */
    const void *b_logit;      /* [T][ld_ub] act: beta projection, HV channels */
    int64_t ld_ub;
    const void *conv_w;       /* [CH][4] act: conv taps, w[c][3] multiplies the current token */
    const float *A_log;       /* [HV] */
    const float *dt_bias;     /* [HV] */
    const float *norm_w;      /* [dv] */
    const int32_t *cu_seqlens;/* [n_seqs+1]; ignored (may be NULL) by gdn_mixer_decode */
    int32_t n_seqs;
    int64_t T;                /* packed tokens (decode: T == n_seqs) */
    const int32_t *state_idx; /* [n_seqs] or NULL */
    const float *state_in;    /* [n_slots][HV][dk][dv] or NULL = zero initial state */
    float *state_out;         /* [n_slots][HV][dk][dv] or NULL = not written; may == state_in */
    void *conv_state;         /* [n_slots][CH][3] act, in/out, or NULL = zero history, not written */
    void *y;                  /* [T][HV*dv] y_dtype */
    gdn_dtype y_dtype;
} gdn_mixer_io;

/* Bytes of workspace any entry point needs for up to max_tokens packed tokens
 * and max_seqs sequences under cfg (0 when cfg is invalid).  HOST only. */
size_t gdn_workspace_size(const gdn_config *cfg, int64_t max_tokens, int32_t max_seqs);

/* a1 gate prep: g = -exp(A_log[h]) * softplus(u + dt_bias[h]), beta =
 * sigmoid(b_logit), per token and v-head.  u, b_logit: [T][ld_ub] act;
 * g, beta: [T][HV] fp32. */
gdn_status gdn_gate_prep(const gdn_config *cfg, const void *u, const void *b_logit, int64_t ld_ub,
                         int64_t T, const float *A_log, const float *dt_bias, float *g,
                         float *beta, void *stream);

/* a2/a3 causal conv1d prefill + SiLU over a packed batch (haskell-infer-demo
 * README, "Architecture", kernels/gdn_conv.cu; hyperflare core-design, the
 * short-convolution paragraph).  x: [T][ld_x] act; w: [CH][4] act;
 * conv_state: [n_slots][CH][3] act in/out (NULL = zero history, not
 * written): the history of sequence n is read at its first token and replaced
 * by its last three raw inputs.  out: [T][CH] out_dtype, SiLU applied, no L2. */
gdn_status gdn_conv1d_prefill(const gdn_config *cfg, const void *x, int64_t ld_x,
                              const int32_t *cu_seqlens, int32_t n_seqs, int64_t T,
                              const void *w, void *conv_state, const int32_t *state_idx,
                              void *out, gdn_dtype out_dtype, void *stream);

/* a8 conv part: one token for each of n sequences; x: [n][ld_x] act.  Shifts
 * each history in place (requires conv_state).  out: [n][CH] out_dtype. */
gdn_status gdn_conv1d_step(const gdn_config *cfg, const void *x, int64_t ld_x, int32_t n,
                           const void *w, void *conv_state, const int32_t *state_idx, void *out,
                           gdn_dtype out_dtype, void *stream);

/* a4/a5/a7 chunked gated delta rule over a packed batch (haskell-infer-demo
 * README, kernels/fla_gdn.cu "chunked prefill"; hyperflare core-design, GDN
 * numerics paragraph: chunks restart at each sequence's first token in the
 * call, FP32 state).  q, k: [T][ld_qk] in_dtype, head kh at column kh*dk;
 * v: [T][ld_v] in_dtype, head h at column h*dv; g, beta: [T][HV] fp32.
 * state_in may be NULL (zero state); state_out may be NULL or == state_in.
 * o: [T][HV*dv] o_dtype.  flags: GDN_FLAG_L2NORM_QK.
 * workspace: DEVICE, caller-owned, 16-byte aligned.  The tensor-core path
 * (bf16 activations, dk = dv = 128, chunk 64) keeps per-(chunk, v-head)
 * operands there and needs gdn_workspace_size(cfg, T, n_seqs) bytes, else
 * GDN_ERR_WORKSPACE; the fp32 path needs none (NULL, 0 accepted). */
gdn_status gdn_chunk_prefill(const gdn_config *cfg, const void *q, const void *k, int64_t ld_qk,
                             const void *v, int64_t ld_v, gdn_dtype in_dtype, const float *g,
                             const float *beta, const int32_t *cu_seqlens, int32_t n_seqs,
                             int64_t T, const float *state_in, float *state_out,
                             const int32_t *state_idx, void *o, gdn_dtype o_dtype, uint32_t flags,
                             void *workspace, size_t workspace_bytes, void *stream);

/* a8 one-token recurrent update for n sequences, state in place (haskell-
 * infer-demo README, kernels/fla_gdn.cu "recurrent decode").  q, k: [n][ld_qk];
 * v: [n][ld_v] in_dtype; g, beta: [n][HV] fp32; state: [n_slots][HV][dk][dv]
 * read once and written once; o: [n][HV*dv] o_dtype. */
gdn_status gdn_recurrent_decode(const gdn_config *cfg, const void *q, const void *k, int64_t ld_qk,
                                const void *v, int64_t ld_v, gdn_dtype in_dtype, const float *g,
                                const float *beta, int32_t n, float *state,
                                const int32_t *state_idx, void *o, gdn_dtype o_dtype,
                                uint32_t flags, void *stream);

/* a6 gated RMSNorm per token and v-head (haskell-infer-demo README,
 * kernels/gdn_norm.cu "model-specific gated norm"): y = o * rsqrt(mean(o^2) +
 * norm_eps) * w * SiLU(z).  o: [T][HV*dv] o_dtype; z: [T][ld_z] act;
 * w: [dv] fp32; y: [T][HV*dv] y_dtype. */
gdn_status gdn_gated_rmsnorm(const gdn_config *cfg, const void *o, gdn_dtype o_dtype,
                             const void *z, int64_t ld_z, const float *w, int64_t T, void *y,
                             gdn_dtype y_dtype, void *stream);

/* Fused prefill, a1..a7: raw projections in, y, final state and new conv
 * history out.  Needs gdn_workspace_size(cfg, T, n_seqs) bytes of workspace. */
gdn_status gdn_mixer_prefill(const gdn_config *cfg, const gdn_mixer_io *io, void *workspace,
                             size_t workspace_bytes, void *stream);

/* Size of the library-owned scratch array used by gdn_mixer_prefill_static. */
#define GDN_STATIC_SCRATCH_BYTES (64u << 20)

/* Fused prefill for callers that cannot allocate device memory (the pages
 * have no counterpart: it exists for callers such as allocation-free step
 * loops or plugins that receive only a stream and their tensors).  Same
 * arguments and results as gdn_mixer_prefill, without the workspace: the
 * intermediates live in a GDN_STATIC_SCRATCH_BYTES array compiled into the
 * library, which every GPU that loads the library keeps until exit.
 *  - Allocates nothing.  Returns GDN_ERR_WORKSPACE when the prefill's own
 *    intermediates for (io->T, io->n_seqs) exceed the array (this is at most
 *    gdn_workspace_size, which covers every mode).  At HK=16, HV=32,
 *    dk=dv=128 that is more than about 700 packed tokens for one sequence,
 *    575 for four and 121 for sixteen on the tensor-core (bf16, chunk 64)
 *    path, whose per-chunk operands dominate, and more than 1,358 tokens
 *    whatever the sequence count in fp32 mode.
 *  - The cached array address belongs to the device's context: after
 *    cudaDeviceReset it is stale, so do not call this again on that device.
 *  - The first call on a device looks up the array's device address (with
 *    that device current); make it before any stream capture.
 *  - All calls share the one array and it keeps the last call's contents:
 *    calls whose GPU work overlaps (other streams, other host threads) race
 *    and must be serialised by the caller. */
gdn_status gdn_mixer_prefill_static(const gdn_config *cfg, const gdn_mixer_io *io, void *stream);

/* Fused decode, a8: one token per sequence (io->T == io->n_seqs), conv history
 * and state updated in place (io->state_out must equal io->state_in and be
 * non-NULL; io->conv_state must be non-NULL).  Two launches: a per-(sequence,
 * q/k head) prep kernel (conv step, SiLU, L2, gates, SiLU(z)) writes a small
 * record per unit to `workspace` (DEVICE, caller-owned, 16-byte aligned, at
 * least gdn_workspace_size(cfg, n_seqs, n_seqs) bytes, else GDN_ERR_WORKSPACE);
 * a persistent kernel then streams every head state through shared memory
 * once.  The workspace holds nothing between calls. */
gdn_status gdn_mixer_decode(const gdn_config *cfg, const gdn_mixer_io *io, void *workspace,
                            size_t workspace_bytes, void *stream);

/* Q8 recurrent state: int8 codes [n_slots][HV][dk][dv] with one fp32 scale
 * per state row, [n_slots][HV][dk] (the row of dk index i holds M[i][0..dv)),
 * so M[i][j] = code[i][j] * scale[i]: about 4x fewer state bytes per decode
 * step (warpfront/hipfire PR #527 thread, STEP-004 note: a DeltaNet Q8 state
 * requantised stochastically, with an error-feedback residual; issue #588: the
 * dither is keyed by a frame counter).  The value x of a row is encoded with
 * stochastic rounding: scale = max_j |x_ij| / 127, code = clamp(floor(x_ij *
 * (127 / max) + u), -127, 127), every step an fp32 operation rounded to
 * nearest, a zero row giving scale 0 and codes 0.  Every code draws its own
 * dither u = (r >> 8) * 2^-24, r = pcg_hash(e ^ pcg_hash(frame)), e = ((slot *
 * HV + head) * dk + i) * dv + j (uint32), pcg_hash being the PCG hash of
 * Jarzynski and Olano (JCGT 2020).  The expected code is then exact, so the
 * rounding adds no bias.  The caller passes a new frame every step.
 *
 * Error feedback (optional): `residual` (bf16 [n_slots][HV][dk][dv], 16-byte
 * aligned, NULL = off) holds the rounding error the last encode left.  With
 * it, the value encoded is x = M_new + residual and the residual becomes
 * bf16(x - code * scale).  The running sum of the decoded states then tracks
 * the running sum of the exact ones to within one residual, instead of
 * drifting like a random walk.  The recurrence itself reads only the codes.
 * It costs 2 more bytes per element in each direction.
 *
 * gdn_state_to_q8 / gdn_state_from_q8: convert the whole pool (cfg->n_slots
 * slots) between fp32 [n_slots][HV][dk][dv] and Q8; with a residual, to_q8
 * is the first encode of an error-feedback pool (residual in = 0) and
 * writes the residual.
 * gdn_mixer_decode_q8: gdn_mixer_decode on a Q8 pool; io->state_in and
 * io->state_out must be NULL; io->conv_state is required; same workspace as
 * gdn_mixer_decode.  A non-NULL residual turns error feedback on: it is read
 * and rewritten for the active slots. */
gdn_status gdn_state_to_q8(const gdn_config *cfg, const float *state, int8_t *codes, float *scales,
                           void *residual, uint32_t frame, void *stream);
gdn_status gdn_state_from_q8(const gdn_config *cfg, const int8_t *codes, const float *scales,
                             float *state, void *stream);
gdn_status gdn_mixer_decode_q8(const gdn_config *cfg, const gdn_mixer_io *io, int8_t *codes,
                               float *scales, void *residual, uint32_t frame, void *workspace,
                               size_t workspace_bytes, void *stream);

/* Backward of the gated delta rule core from retained chunk-boundary states
 * (hyperflare core-design, training plan: a training step retains
 * activations and GDN chunk-boundary states; the backward has one entry per
 * region, the GDN core among them).  The core is the rule of
 * gdn_chunk_prefill on q, k, v as given (no in-kernel L2 norm: q and k are
 * the normalised vectors; the norm's own backward is outside the core).
 * Chunks are cfg->chunk tokens from each sequence's first token; sequence n
 * has ceil(len_n / chunk) of them and its chunk c is boundary index
 * (sum over m < n of ceil(len_m / chunk)) + c.
 *
 * gdn_chunk_states: the state before the first token of every chunk, fp32
 * [n_chunks][HV][dk][dv] (the layout of the recurrent state), from state_in
 * (NULL: zero) of slot state_idx[n] (NULL: slot n; a negative entry is a
 * padding lane and gets no entries written).  k: [T][ld_qk], v: [T][ld_v]
 * in_dtype; g, beta: [T][HV] fp32.  token_pw (NULL: not written): fp32
 * [T][HV][2][dv], 16-byte aligned, caller-owned; for every token of every
 * sequence that is not a padding lane, row 0 gets p = M^T k (the state before
 * the token read at k) and row 1 gets w = beta (v - a p), the row the token
 * adds to the state (M <- a M + k w^T).  workspace: at least
 * gdn_backward_workspace_size(cfg, T, n_seqs) bytes (this call uses 256 plus
 * 4 * (n_seqs + 1) of them).
 *
 * gdn_chunk_backward: for the loss sum(d_o * o) + sum(d_state_out * S_final)
 * (d_state_out NULL: no final-state term), writes dq, dk ([T][ld_dqk] fp32, the
 * v-heads of each q/k head summed: head kh at column kh*dk), dv ([T][HV*dv]
 * fp32), dg and dbeta ([T][HV] fp32; dg is the gradient with respect to the
 * log-decay g, a = exp(g)) and, when non-NULL, d_state_in ([n_slots][HV][dk]
 * [dv] fp32, the gradient with respect to the initial state of each
 * sequence's slot).  boundary_states as written by gdn_chunk_states for the
 * same batch; token_pw either NULL (the walk recomputes p and w from the
 * boundary states) or as written by that same call (the walk reads them and
 * skips the recomputation: the same result up to rounding, faster).  Padding lanes get zero gradients.  workspace: at least
 * gdn_backward_workspace_size(cfg, T, n_seqs) bytes (the replayed states of
 * one chunk and the gradients entering the segments each sequence is walked
 * in, per (sequence, v-head), and the per-slice parts of dq, dk, dg and dbeta
 * per token). */
size_t gdn_backward_workspace_size(const gdn_config *cfg, int64_t max_tokens, int32_t max_seqs);
gdn_status gdn_chunk_states(const gdn_config *cfg, const void *k, int64_t ld_qk, const void *v,
                            int64_t ld_v, gdn_dtype in_dtype, const float *g, const float *beta,
                            const int32_t *cu_seqlens, int32_t n_seqs, int64_t T,
                            const float *state_in, const int32_t *state_idx, float *boundary_states,
                            float *token_pw, void *workspace, size_t workspace_bytes, void *stream);
gdn_status gdn_chunk_backward(const gdn_config *cfg, const void *q, const void *k, int64_t ld_qk,
                              const void *v, int64_t ld_v, gdn_dtype in_dtype, const float *g,
                              const float *beta, const int32_t *cu_seqlens, int32_t n_seqs, int64_t T,
                              const int32_t *state_idx, const float *boundary_states,
                              const float *token_pw, const float *d_o, const float *d_state_out,
                              float *dq, float *dk,
                              int64_t ld_dqk, float *dv, float *dg, float *dbeta, float *d_state_in,
                              void *workspace, size_t workspace_bytes, void *stream);

/* Multi-token verification decode (hyperflare core-design, speculative
 * target state: each request reserves eight recurrent checkpoint columns, a
 * verification round writes the columns of its inputs, and the round after
 * continues from the column of the last accepted input, whose three-token
 * conv window goes with it).  k (1..8) tokens for each of io->n_seqs
 * sequences, packed sequence-major: rows n*k .. n*k+k-1 of io->x, io->z,
 * io->u, io->b_logit and io->y (io->T == n_seqs * k; cu_seqlens unused).
 * Sequence n starts from the state and conv history of slot
 * io->state_idx[n] (NULL: slot n), which are read and not modified; the
 * one-token rule of gdn_mixer_decode is applied to its k tokens in order,
 * y row n*k+j is token j's output, and the state and conv history after
 * token j are written to slot ckpt_idx[n] + j (ckpt_idx: int32 [n_seqs],
 * DEVICE).  io->state_out must equal io->state_in (one pool, non-NULL) and
 * io->conv_state must be non-NULL.  To commit `a` accepted tokens, continue
 * from slot ckpt_idx[n] + a - 1 (as the next call's state_idx, or copy it to
 * a live slot with gdn_state_copy).  The columns of different sequences must
 * not overlap one another or another sequence's source slot; a sequence's
 * own source slot may be its column 0 (it is read before it is written).
 * A negative state_idx[n] is a padding lane (zero outputs, nothing written);
 * columns reaching past n_slots are reported as GDN_DEVERR_SLOT and that
 * sequence is skipped.  One launch; the per-token intermediates stay in
 * shared memory, so `workspace` / `workspace_bytes` are not used (NULL and 0
 * are accepted; the arguments keep the signature of the other fused entry
 * points). */
gdn_status gdn_mixer_verify(const gdn_config *cfg, const gdn_mixer_io *io, int32_t k,
                            const int32_t *ckpt_idx, void *workspace, size_t workspace_bytes,
                            void *stream);

/* State maintenance: snapshot, restore, initialise and reset of state slots
 * as one indirect copy driven by device-resident slot-index buffers
 * (hyperflare core-design: the "State operations" row of the native model
 * contract, the state-maintenance graph entries, and the speculative-state
 * section: a snapshot selects one recurrent state column and copies its
 * three-token conv window; snapshot and restore preserve committed state
 * exactly and allocate nothing).  For each pair i < n, with s = src_idx[i]
 * and t = dst_idx[i] (int32, DEVICE):
 *   t < 0          nothing (an inactive lane);
 *   s >= 0, t >= 0 slot s of (src_state, src_conv) is copied to slot t of
 *                  (dst_state, dst_conv) bit for bit;
 *   s < 0,  t >= 0 slot t is reset to zeros (the initial state and history).
 * src_state / dst_state: fp32 [slots][HV][dk][dv]; src_conv / dst_conv: act
 * [slots][CH][3].  dst_state == NULL leaves states untouched (and src_state
 * is not read); likewise dst_conv.  A NULL source with a non-NULL
 * destination resets.  n_src_slots / n_dst_slots bound the indices: a pair
 * with t >= n_dst_slots, or s >= n_src_slots while a source pool is given,
 * is skipped and reported as GDN_DEVERR_SLOT.  Source and destination may be the same pool (a pool
 * holding live and snapshot rows); then the live destination slots of one
 * call must be distinct and must not be read as a source by another pair of
 * the same call (the indices are device data and are not checked on the
 * host).  n == 0 launches nothing. */
gdn_status gdn_state_copy(const gdn_config *cfg, const float *src_state, const void *src_conv,
                          int32_t n_src_slots, float *dst_state, void *dst_conv,
                          int32_t n_dst_slots, const int32_t *src_idx, const int32_t *dst_idx,
                          int32_t n, void *stream);

/* Bounded waits (no page counterpart: it makes the device-side timeout
 * testable without a GPU fault).  Every wait of a kernel on another part of
 * the kernel (an mbarrier, a copy, a peer CTA's flag) gives up after wait_ns
 * nanoseconds (default 2 s), records GDN_DEVERR_TIMEOUT, skips the rest of
 * its work and returns; the caller reads the bit with gdn_device_error().
 * `lose` (tests only; 0 in normal use) makes the calls that follow drop one
 * operand copy so that such a wait really runs out: bit 0 the first head
 * state of a gdn_mixer_decode / gdn_mixer_decode_q8 launch, bit 1 the first
 * chunk operand of the tensor-core state chain (gdn_chunk_prefill,
 * gdn_mixer_prefill).  A call that timed out writes no state.  Process-wide,
 * read at each call; GDN_ERR_INVALID_ARG for wait_ns = 0, above 60 s, or an
 * unknown bit. */
gdn_status gdn_debug_set_wait(uint64_t wait_ns, uint32_t lose);

/* Synchronises `stream`, then reads and clears the device error word of the
 * current device into *code (HOST pointer; GDN_DEVERR_* bits).  Returns
 * GDN_ERR_DEVICE when a code was set, GDN_OK otherwise. */
gdn_status gdn_device_error(void *stream, uint32_t *code);

/* Static description of a status code (HOST). */
const char *gdn_status_string(gdn_status s);

#ifdef __cplusplus
}
#endif

#endif /* GDN_GB300_H */
