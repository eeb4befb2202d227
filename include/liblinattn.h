/*
 * liblinattn.h -- C ABI of the GB300 (sm_103a) chunked Gated DeltaNet forward.
 *
 * The operation is defined on the cuDNN "Linear Attention" operations page
 * (docs.nvidia.com/cudnn/operations/LinearAttention): for every sequence of a
 * packed THD batch and every output head, a recurrent matrix state
 * S[K][V] evolves token by token as
 *
 *     S_t = exp(g_t) (I - beta_t k_t k_t^T) S_{t-1} + beta_t k_t v_t^T
 *     o_t = scale * S_t^T q_t
 *
 * (the page's Householder-product family with one update per token), with the
 * options of its worked example and of its "Semantics worth knowing" section:
 * in-kernel L2 normalisation of q and k, an initial state, the final state,
 * state checkpoints every n tokens, and the span summary.
 *
 * Conventions shared by every entry point
 *   - Layout is packed THD ("Layout" section): tokens of all N sequences are
 *     concatenated on axis 0; cu_seqlens[N+1] (int32 or int64, device memory)
 *     gives the boundaries and must start at 0, be nondecreasing and end at T.
 *   - Operands are rank-3 [T, heads, dim] views given by a device pointer and
 *     two strides in ELEMENTS (token stride, head stride); the innermost (dim)
 *     axis must be contiguous.  Base addresses must be 16-byte aligned and
 *     the token/head strides of bf16 operands multiples of 8 elements (the
 *     kernels read q/k/v through TMA descriptors built from these strides,
 *     "Layout" section: column slices of a fused projection are accepted).
 *   - Dtypes are fixed, as on the page's support matrix (callers convert):
 *     q, k, v and o are bf16; g and beta are fp32 [T, HO]; states are fp32 (an
 *     initial state may also be bf16).  K and V must be 64 or 128.
 *   - Heads: HK q/k heads, HV value heads, HO = HV output heads; HV must be a
 *     multiple of HK and output head h reads q/k head h / (HV / HK).
 *   - Every pointer is device memory unless stated.  The caller owns every
 *     buffer; the library never frees caller memory.
 *   - Calls are asynchronous on `stream` (a cudaStream_t passed as void*;
 *     NULL is the legacy default stream) and never synchronise the host.
 *   - Errors: argument problems found on the host are returned synchronously
 *     and nothing is launched.  Problems only the device can see (bad
 *     cu_seqlens values, a bounded wait that ran out) are written to the
 *     device status word; the outputs are then unspecified.
 *   - Batch invariance (batch_invariant, same section): a sequence's results
 *     are bitwise identical whatever else is in the batch.
 */
#ifndef LIBLINATTN_H
#define LIBLINATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum la_status {
    LA_OK = 0,
    LA_ERR_INVALID_ARG = 1,  /* null pointer, bad shape/stride/alignment, N < 0, ... */
    LA_ERR_UNSUPPORTED = 2,  /* K or V not in {64,128}, HV % HK != 0, HK > HV, dtype */
    LA_ERR_CUDA = 3,         /* a CUDA runtime or driver call failed (launch, encode) */
    LA_ERR_BAD_SEQLENS = 4,  /* cu_seqlens not 0-based, decreasing or != T at N (device-side; returned by gdn_fwd_host) */
    LA_ERR_TIMEOUT = 5,      /* device-side: a bounded wait in a kernel gave up */
    LA_ERR_WORKSPACE = 6,    /* workspace smaller than la_gdn_workspace_bytes() */
    LA_ERR_BAD_STATE_INDEX = 7 /* device-side: a state_indices entry outside [0, state_pool_size) */
} la_status;

typedef enum la_dtype { LA_DTYPE_BF16 = 0, LA_DTYPE_F32 = 1 } la_dtype;

/*
 * How the kernel reads g (cudnn-frontend PR #616: in-kernel gate fusion, used
 * by the FLA GatedDeltaNet layer).  a_log and dt_bias are per output head.
 *   LA_GATE_LOG           g is the natural-log decay itself (default).
 *   LA_GATE_SOFTPLUS      log decay = -exp(a_log[h]) * softplus(g[t,h] + dt_bias[h]),
 *                         softplus(x) = log(1 + e^x) (taken as x above 20).
 *   LA_GATE_SIGMOID_BOUND log decay = gate_lower_bound * sigmoid(g[t,h]), bounded
 *                         below by gate_lower_bound (< 0; PR #616 uses -5 by default).
 */
typedef enum la_gate_mode { LA_GATE_LOG = 0, LA_GATE_SOFTPLUS = 1, LA_GATE_SIGMOID_BOUND = 2 } la_gate_mode;

/* Parameters of gdn_fwd.  Strides are in elements. */
typedef struct la_gdn_fwd_params {
    /* ---- inputs ---- */
    const void* q;    int64_t q_stride_t, q_stride_h;       /* [T, HK, K] bf16 */
    const void* k;    int64_t k_stride_t, k_stride_h;       /* [T, HK, K] bf16 */
    const void* v;    int64_t v_stride_t, v_stride_h;       /* [T, HV, V] bf16 */
    const float* g;   int64_t g_stride_t, g_stride_h;       /* [T, HO] fp32, natural-log decay */
    const float* beta; int64_t beta_stride_t, beta_stride_h; /* [T, HO] fp32 */
    const void* cu_seqlens;                                 /* [N + 1] */
    int32_t cu_seqlens_bits;                                /* 32 or 64 */
    int64_t T;
    int32_t N, HK, HV, K, V;
    float scale;              /* multiplies the (normalised) query; <= 0 selects 1/sqrt(K) */
    int32_t use_qk_l2norm;    /* q, k <- x / sqrt(sum x^2 + 1e-6) before the recurrence */
    const void* initial_state;  /* [N, HO, K, V] contiguous, or NULL for a zero start */
    int32_t initial_state_dtype; /* la_dtype */
    /* ---- outputs ---- */
    void* o;          int64_t o_stride_t, o_stride_h;       /* [T, HO, V] bf16 */
    float* final_state;       /* [N, HO, K, V] fp32 contiguous, or NULL (output_final_state=False) */
    void* checkpoints;        /* [R, HO, K, V] contiguous, or NULL; R = la_checkpoint_rows() */
    int32_t checkpoint_dtype; /* la_dtype of the checkpoint rows */
    int64_t checkpoint_every_n; /* > 0 and a multiple of 64 when checkpoints != NULL */
    /* ---- scratch and status ---- */
    void* workspace;          /* >= la_gdn_workspace_bytes(N, 0) bytes, 256-byte aligned, or NULL;
                                 >= la_gdn_fwd_split_workspace_bytes(T, N, HV) allows two passes */
    size_t workspace_bytes;
    int32_t* status;          /* optional device int32; receives LA_OK or a device-side error */
    /* ---- optional input transforms (all zero = off; PR #616 in-kernel fusions) ---- */
    int32_t gate_mode;        /* la_gate_mode */
    const float* a_log;       /* [HO] fp32 (LA_GATE_SOFTPLUS) */
    const float* dt_bias;     /* [HO] fp32 (LA_GATE_SOFTPLUS) */
    float gate_lower_bound;   /* < 0 (LA_GATE_SIGMOID_BOUND) */
    int32_t beta_sigmoid;     /* beta holds logits: beta <- 1 / (1 + exp(-beta)) */
    int32_t beta_bf16;        /* beta is bf16 (same strides) instead of fp32 */
    /* ---- optional state pool (page: "States and checkpoints", state_indices) ----
     * When state_indices ([N] int32, device) is set, initial_state is a pool
     * [state_pool_size, HO, K, V] (contiguous, fp32 or bf16): sequence i starts
     * from slot state_indices[i] and its end state is written back to that slot
     * in place, in the pool's dtype.  final_state and checkpoints must be NULL.
     * Two sequences of one call must not name the same slot (their write-backs
     * would race).  An index outside the pool sets LA_ERR_BAD_STATE_INDEX in the
     * status word and that sequence is skipped. */
    const int32_t* state_indices;
    int64_t state_pool_size;
    /* ---- Gated DeltaProduct (page: GDP runs on two timelines) ----
     * num_householder n > 1: k, v and beta hold n rows per token, update-major (the n updates
     * of token t are rows t*n .. t*n+n-1; a contiguous token-major [T, n, H, D] view is the same
     * memory), and their row strides above are per update row; q, g and o keep one row per
     * token and T counts tokens.  Per token the state decays once (exp(g_t)), takes the n delta
     * updates in order, and o_t reads the state after the last.  checkpoint_every_n counts
     * tokens (n * checkpoint_every_n must be a multiple of 64).  0 or 1: GDN. */
    int32_t num_householder;
} la_gdn_fwd_params;

/*
 * gdn_fwd -- the chunked GDN forward over a packed THD batch.
 *
 * Page: "Example" (gated_delta_net(q, k, v, g, beta, cu_seqlens,
 * output_final_state, use_qk_l2norm_in_kernel)) and "States and checkpoints".
 *   o[t, h, :]       = scale * S_t^T q_hat_t for every token (inclusive of t).
 *   final_state      = the state after each sequence's last token (an empty
 *                      sequence returns its initial state, or zeros).
 *   checkpoints      = the state entering token offsets 0, n, 2n, ... < L of
 *                      each sequence (entry 0 is the initial state), packed in
 *                      sequence order: sequence i owns ceil(L_i / n) rows
 *                      starting at sum_{j<i} ceil(L_j / n).
 * Workspace: if `workspace` is NULL an internal per-device buffer is used;
 * overlapping calls on different streams must then each pass their own.  That
 * buffer grows on demand (every entry point that takes a workspace shares it)
 * without any synchronisation: a larger buffer replaces it and the old one
 * stays allocated until the process exits, since earlier kernels may still
 * read it (sizes at least double, so the kept buffers total less than the
 * current one).  Growth allocates, which stream capture forbids: a call on a
 * capturing stream that would need to grow the buffer returns
 * LA_ERR_WORKSPACE and launches nothing (pass a workspace, or make a call of
 * that size before capturing).
 * Two passes: half of each chunk's work does not depend on the state (the
 * gates' cumulative sums, the row norms, A, P and T = (I + A)^{-1}).  When the
 * workspace has room for it (la_gdn_fwd_split_workspace_bytes; with workspace
 * = NULL the internal buffer grows to that size, and a failed allocation or a
 * capturing stream falls back), gdn_fwd first forms that half for every
 * (chunk, head) of the batch at once, then walks each sequence with only the
 * state-dependent products on its serial chain; otherwise one fused kernel
 * does both on the chain.  The two compute the same bits.
 * Scheduling: each (sequence, head) is one serial walk over its chunks.  When
 * the walks fill between one and four waves of the CTAs the GPU holds at once
 * and final_state is fp32 (or the state pool is), the call may instead enqueue
 * several launches that walk every sequence in 2 to 8 chunk ranges, handing the
 * exact fp32 state from range to range through final_state (each walk reads
 * and writes only its own rows there, and a range ending on a checkpoint
 * boundary writes that row): the results are the same bits as one walk, with
 * a shorter tail when the last wave would be partly empty.
 * Returns LA_OK once the work is enqueued.
 */
la_status gdn_fwd(const la_gdn_fwd_params* p, void* stream);

/*
 * gdn_fwd_static_workspace -- gdn_fwd for callers that cannot allocate device memory.
 *
 * The pages have no counterpart to this entry point; it exists for callers
 * that are not allowed to call cudaMalloc (a process whose allocator owns all
 * device memory, or one that must not allocate once it is serving).  It runs
 * exactly the gdn_fwd computation with the same parameters, but takes its
 * scratch from a fixed array compiled into the library (about 96 KB per GPU,
 * held from library load to process exit) instead of a workspace:
 *   - p->workspace must be NULL (LA_ERR_INVALID_ARG otherwise);
 *   - N may be at most 8192 sequences; larger batches return LA_ERR_WORKSPACE
 *     and launch nothing;
 *   - Gated DeltaProduct with num_householder > 64 is not available here (its
 *     timeline scratch grows with T): LA_ERR_UNSUPPORTED, nothing launched;
 *   - no call allocates or frees device memory.  The first call on a device
 *     looks up the array's device address (once, with that device current);
 *     make that first call before any stream capture.  The address is kept
 *     for the life of the process: after the application resets a device
 *     (cudaDeviceReset) it is stale, and this entry point must not be used
 *     on that device again.
 *   - every call on a device shares the one array.  Each call re-initialises
 *     what must start at zero (status word, unit ticket) in its own prologue
 *     kernel, so leftovers from an earlier call are harmless, but calls whose
 *     kernels overlap on the GPU (different streams, no ordering between them)
 *     race on the array and give undefined results.
 */
la_status gdn_fwd_static_workspace(const la_gdn_fwd_params* p, void* stream);

/*
 * gdn_fwd_host -- gdn_fwd on HOST buffers: copy in, forward, copy out, pipelined.
 *
 * Computes exactly what gdn_fwd computes (bitwise the same o, final state and
 * checkpoints) for inputs and outputs that live in host memory.  The packed
 * batch is cut into about `ranges` token ranges (la_gdn_fwd_host_plan): runs
 * of whole sequences, and sequences longer than a range cut into pieces at
 * multiples of the range length P (a multiple of the 64-token chunk and of
 * checkpoint_every_n), each piece starting from the exact fp32 state the
 * previous piece ended in.  A range's host-to-device copies, its forward and
 * its device-to-host copies are chained by events across one copy-in stream,
 * eight compute streams (the pieces of one sequence share one) and one
 * copy-out stream, owned by the library per device, so copies of some ranges
 * overlap the forwards of others.
 *
 *   fwd: the gdn_fwd parameters with HOST pointers for q, k, v, g, beta,
 *     cu_seqlens, initial_state, a_log, dt_bias, o, final_state and
 *     checkpoints.  q, k, v, g, beta and o must be contiguous ([T, H, D] with
 *     token stride H * D and head stride D; [T, HO] with stride HO, 1).
 *     Page-locked (pinned) host memory lets the copies run asynchronously;
 *     pageable memory is accepted but serialises the copies with the host.
 *     fwd.status, if set, is a DEVICE int32 as in gdn_fwd; fwd.workspace is
 *     ignored; state_indices must be NULL and num_householder <= 1.
 *   staging: DEVICE memory of at least la_gdn_fwd_host_staging_bytes(p)
 *     bytes, 256-byte aligned, owned by the caller (the device copies of every
 *     input and output plus per-stream scratch).
 *   ranges: >= 1.
 * Ordering: the first call with a given staging buffer is ordered after the
 * work already enqueued on `stream`; a later call with the same buffer is
 * ordered after the previous call that used it (not after `stream`: its
 * inputs are host memory), so a caller that alternates two staging buffers
 * lets the copies of one call run under the last forwards of the one before.
 * `stream` is made to wait for the call's last copy out.  The call returns
 * once everything is enqueued (host buffers must stay valid and the outputs
 * must not be read until `stream` has been synchronised).
 * The host may block while the previous call's small metadata copy is still
 * pending.  Not capturable in a CUDA graph (use gdn_fwd on device buffers).
 * Errors: argument checks as gdn_fwd, plus LA_ERR_BAD_SEQLENS for a host
 * cu_seqlens that is not 0, nondecreasing, T; LA_ERR_WORKSPACE for a staging
 * buffer that is too small or misaligned; LA_ERR_UNSUPPORTED for a state pool
 * or Gated DeltaProduct.
 */
typedef struct la_gdn_fwd_host_params {
    la_gdn_fwd_params fwd;
    void* staging;
    size_t staging_bytes;
    int32_t ranges;
} la_gdn_fwd_host_params;

la_status gdn_fwd_host(const la_gdn_fwd_host_params* p, void* stream);

/* Device staging bytes gdn_fwd_host needs for these parameters (reads the host
 * cu_seqlens); 0 if the parameters are invalid. */
size_t la_gdn_fwd_host_staging_bytes(const la_gdn_fwd_host_params* p);

/* The token ranges of gdn_fwd_host for a host cu_seqlens [N + 1] (idx_bits 32 or
 * 64), `ranges` and the checkpoint cadence n (0: none).  Writes up to
 * max_ranges rows of six int64 (t_a, t_b, a, b, piece, last) into out: tokens
 * t_a .. t_b of the packed batch; a run of whole sequences a .. b-1 has
 * piece = -1 and last = 1; a piece of sequence a (b = a + 1) has its index
 * within the sequence and last = 1 when it ends the sequence.  *piece_tokens
 * receives P.  Returns the number of ranges (which may exceed max_ranges: call
 * again with room), or -1 for invalid arguments. */
int32_t la_gdn_fwd_host_plan(const void* cu_seqlens_host, int32_t idx_bits, int32_t N, int32_t ranges,
                             int64_t checkpoint_every_n, int64_t* out, int32_t max_ranges, int64_t* piece_tokens);

/* Parameters of gdn_summary.  Strides are in elements. */
typedef struct la_gdn_summary_params {
    const void* k;    int64_t k_stride_t, k_stride_h;       /* [T, HK, K] bf16 */
    const void* v;    int64_t v_stride_t, v_stride_h;       /* [T, HV, V] bf16 */
    const float* g;   int64_t g_stride_t, g_stride_h;       /* [T, HO] fp32 */
    const float* beta; int64_t beta_stride_t, beta_stride_h; /* [T, HO] fp32 */
    const void* cu_seqlens;                                 /* [N + 1]: the spans */
    int32_t cu_seqlens_bits;
    int64_t T;
    int32_t N, HK, HV, K, V;
    int32_t use_qk_l2norm;
    const void* start_state;  /* [N, HO, K, V] contiguous, or NULL for a zero start */
    int32_t start_state_dtype;
    float* end_state;         /* [N, HO, K, V] fp32: S_H, the end state from start_state */
    float* transition;        /* [N, HO, K, K] fp32 */
    void* workspace;          /* >= la_gdn_workspace_bytes(N, 1) bytes, or NULL */
    size_t workspace_bytes;
    int32_t* status;
    /* optional input transforms, as in la_gdn_fwd_params */
    int32_t gate_mode;
    const float* a_log;
    const float* dt_bias;
    float gate_lower_bound;
    int32_t beta_sigmoid;
    int32_t beta_bf16;
} la_gdn_summary_params;

/*
 * gdn_summary -- per-span end state and state-transition operator.
 *
 * Page: "Summaries" (for the delta-rule variants the transition is a
 * [N, HO, K, K] fp32 matrix: the span's decayed erase factors multiplied
 * together, composed across spans as S_final = S_init * transition + S_H).
 * With P = prod_{t = L-1 .. 0} exp(g_t)(I - beta_t k_hat_t k_hat_t^T), later
 * steps on the left, the library stores transition = P^T, i.e.
 *     S_final[b][v] = sum_a transition[a][b] * S_init[a][v] + S_H[b][v]
 * which is the page's S_init * transition with states read V-major, and the
 * orientation a backward applies (dS_0 = P^T dS_L).  An empty span returns the
 * identity and its start state.
 * Two passes as in gdn_fwd ("Two passes"), when the workspace has room for them
 * (la_gdn_fwd_split_workspace_bytes; with workspace = NULL the internal buffer
 * grows to that size): the WY pass forms each (chunk, head)'s T once for both
 * tiles, and the state pass, which then needs less shared memory, runs two
 * units per SM; the same bits as the fused kernel.
 * When the (span, head, tile) units outnumber the CTAs the GPU holds at once,
 * the call enqueues several launches that walk each span in four chunk ranges
 * and keep the state between ranges in end_state and transition themselves
 * (each unit reads only its own rows there); the results are the same bits as
 * one walk.
 */
la_status gdn_summary(const la_gdn_summary_params* p, void* stream);

/* ---- composition of span summaries ---------------------------------------------------- */
typedef struct la_gdn_compose_params {
    int32_t R;                /* spans, >= 0 */
    int32_t HO, K, V;         /* heads (>= 1); K, V in {64, 128} */
    const float* transitions; /* [R, HO, K, K] fp32 contiguous: gdn_summary's transition per span */
    const float* terms;       /* [R, HO, K, V] fp32 contiguous: forward, each span's end state from a
                                 zero start; backward, each span's own entering-state gradient */
    const float* start;       /* [HO, K, V] fp32 contiguous, or NULL for zeros: forward, the state
                                 entering span 0; backward, the cotangent of the state after span R-1 */
    float* out;               /* [R + 1, HO, K, V] fp32 contiguous, written */
    int32_t backward;         /* 0 forward, 1 backward */
} la_gdn_compose_params;

/*
 * gdn_compose_spans -- context parallelism over sequence spans: compose span summaries.
 *
 * Page: "Summaries" (the end state and the transition of consecutive spans compose as
 * S_final = S_init * transition + S_H, which is how the summaries give context
 * parallelism).  In the library's orientation (states [K][V], transition = P^T):
 *   forward:  out[0] = start; out[r + 1][b][v] = sum_a transitions[r][a][b] out[r][a][v]
 *             + terms[r][b][v]: the state entering span r + 1, out[R] the final state;
 *   backward: d = start; for r = R - 1 down to 0: out[r] = d (the cotangent of the state
 *             leaving span r), d[a][v] <- terms[r][a][v] + sum_b transitions[r][a][b] d[b][v];
 *             out[R] = d, the gradient of the state entering span 0.
 * fp32 throughout; each output is a K-term dot product in ascending order (no dependence on
 * the launch shape).  out must not overlap the inputs.  Asynchronous on `stream`; no
 * workspace, no synchronisation.  Errors: LA_ERR_INVALID_ARG (null params or out, null
 * transitions or terms with R > 0, R < 0, HO < 1, pointers not 4-byte aligned),
 * LA_ERR_UNSUPPORTED (K or V not in {64, 128}), LA_ERR_CUDA (launch failure).
 */
la_status gdn_compose_spans(const la_gdn_compose_params* p, void* stream);

/* Parameters of gdn_decode: one new token for each of N sequences.  Strides are in elements. */
typedef struct la_gdn_decode_params {
    const void* q;    int64_t q_stride_n, q_stride_h;       /* [N, HK, K] bf16 */
    const void* k;    int64_t k_stride_n, k_stride_h;       /* [N, HK, K] bf16 */
    const void* v;    int64_t v_stride_n, v_stride_h;       /* [N, HV, V] bf16 */
    const float* g;   int64_t g_stride_n, g_stride_h;       /* [N, HO] fp32 (raw gate if gate_mode != 0) */
    const float* beta; int64_t beta_stride_n, beta_stride_h; /* [N, HO] fp32 (or bf16 logits, see beta_bf16) */
    int32_t N, HK, HV, K, V;
    float scale;              /* <= 0 selects 1/sqrt(K) */
    int32_t use_qk_l2norm;
    void* state_pool;         /* [state_pool_size, HO, K, V] contiguous, updated in place */
    int32_t state_dtype;      /* la_dtype of the pool */
    int64_t state_pool_size;
    const int32_t* state_indices; /* [N] int32, or NULL: sequence i uses slot i (state_pool_size >= N) */
    void* o;          int64_t o_stride_n, o_stride_h;       /* [N, HO, V] bf16 */
    int32_t* status;          /* optional; LA_ERR_BAD_STATE_INDEX for an index outside the pool */
    int32_t gate_mode;        /* as in la_gdn_fwd_params */
    const float* a_log;
    const float* dt_bias;
    float gate_lower_bound;
    int32_t beta_sigmoid;
    int32_t beta_bf16;
} la_gdn_decode_params;

/*
 * gdn_decode -- one recurrence step per sequence against a state pool.
 *
 * Page: "States and checkpoints" (state_indices turns initial_state into a pool
 * addressed per sequence and written back in place), for the serving case where
 * every sequence brings exactly one token: for each sequence i and head h, with
 * S = pool[state_indices[i], h],
 *     S <- exp(g) (I - beta k_hat k_hat^T) S + beta k_hat v^T,   o = scale S^T q_hat
 * and S is stored back into the same slot.  Equal to gdn_fwd over
 * cu_seqlens = [0, 1, ..., N] with the same pool.  No workspace; never syncs.
 * Two sequences must not name the same slot.
 */
la_status gdn_decode(const la_gdn_decode_params* p, void* stream);

/* Parameters of gdn_bwd.  Strides are in elements. */
typedef struct la_gdn_bwd_params {
    /* ---- the forward's inputs (natural-log gate, beta as given: no input transforms) ---- */
    const void* q;    int64_t q_stride_t, q_stride_h;       /* [T, HK, K] bf16 */
    const void* k;    int64_t k_stride_t, k_stride_h;       /* [T, HK, K] bf16 */
    const void* v;    int64_t v_stride_t, v_stride_h;       /* [T, HV, V] bf16 */
    const float* g;   int64_t g_stride_t, g_stride_h;       /* [T, HO] fp32 */
    const float* beta; int64_t beta_stride_t, beta_stride_h; /* [T, HO] fp32 */
    const void* cu_seqlens;
    int32_t cu_seqlens_bits;
    int64_t T;
    int32_t N, HK, HV, K, V;
    float scale;
    int32_t use_qk_l2norm;
    const void* initial_state;   /* [N, HO, K, V] or NULL */
    int32_t initial_state_dtype;
    /* the forward's checkpoints, as gdn_fwd writes them ([sum ceil(L_i / n), HO, K, V]: the
       states entering offsets 0, n, 2n, ... of each sequence), with n = checkpoint_every_n and the
       dtype of checkpoint_bf16 below; NULL: regenerated by a forward pass */
    const void* checkpoints;
    /* ---- incoming gradients ---- */
    const void* d_o;  int64_t d_o_stride_t, d_o_stride_h;   /* [T, HO, V] bf16 */
    const float* d_final_state;  /* [N, HO, K, V] fp32 or NULL (zero) */
    /* ---- gradients (every one in its input's dtype; dg, dbeta fp32) ---- */
    void* dq;         int64_t dq_stride_t, dq_stride_h;     /* [T, HK, K] bf16 */
    void* dk;         int64_t dk_stride_t, dk_stride_h;     /* [T, HK, K] bf16 */
    void* dv;         int64_t dv_stride_t, dv_stride_h;     /* [T, HV, V] bf16 */
    float* dg;        int64_t dg_stride_t, dg_stride_h;     /* [T, HO] fp32 */
    float* dbeta;     int64_t dbeta_stride_t, dbeta_stride_h; /* [T, HO] fp32 */
    float* d_initial_state;      /* [N, HO, K, V] fp32 or NULL */
    void* workspace;             /* >= la_gdn_bwd_workspace_bytes_min(...), 256-byte aligned, or NULL
                                    (then a per-device buffer, the tensor-core size when possible) */
    size_t workspace_bytes;
    int32_t* status;
    /* ---- optional input transforms, as in gdn_fwd (zero-initialised: none) ---- */
    int32_t gate_mode;           /* la_gate_mode */
    const float* a_log;          /* [HO] fp32 (LA_GATE_SOFTPLUS) */
    const float* dt_bias;        /* [HO] fp32 (LA_GATE_SOFTPLUS) */
    float gate_lower_bound;      /* < 0 (LA_GATE_SIGMOID_BOUND) */
    int32_t beta_sigmoid;        /* beta holds logits */
    int32_t beta_bf16;           /* beta is bf16 (values, or logits with beta_sigmoid) */
    float* d_a_log;              /* [HO] fp32 out (LA_GATE_SOFTPLUS), or NULL */
    float* d_dt_bias;            /* [HO] fp32 out (LA_GATE_SOFTPLUS), or NULL */
    /* ---- the given checkpoints' cadence and dtype (zero-initialised: every 64 tokens, fp32) ---- */
    int64_t checkpoint_every_n;  /* 0 or 64: the chunk cadence; else a multiple of 64 */
    int32_t checkpoint_bf16;     /* the rows are bf16 (as gdn_fwd writes with checkpoint_dtype bf16) */
} la_gdn_bwd_params;

/*
 * gdn_bwd -- the backward of gdn_fwd.
 *
 * Page: every variant has "a full backward", which reuses the forward's checkpoints at the
 * chunk cadence.  Gradients of L = sum(d_o * o) + sum(d_final_state * final_state) with
 * respect to q, k, v, g, beta and the initial state; grouped heads: dq and dk of a q/k head
 * sum the contributions of its value heads.  The backward walks each chunk from the state
 * entering it (page, "States and checkpoints": it reuses rows at the chunk cadence and
 * regenerates the dense series from any other rows):
 *   - fp32 rows every 64 tokens are read as they are;
 *   - bf16 rows every 64 tokens are widened to fp32 in the workspace;
 *   - rows every n > 64 tokens (fp32 or bf16): every sequence is cut at multiples of n into
 *     segments that each start from their row, and one forward launch over all the segments
 *     (independent, so they run side by side) regenerates the states entering every chunk.
 *     From fp32 rows these are bitwise the states the full forward produced;
 *   - no rows: the library re-runs the forward with fp32 checkpoints every 64 tokens.
 * Two schedules, the same mathematics:
 *   - tensor cores (K = V = 128, d_o 16-byte aligned with strides in 8-element units, fp32
 *     states 16-byte aligned, and a workspace of la_gdn_bwd_workspace_bytes_ckpt): the
 *     forward's WY pass over every (chunk, head), which also keeps T's bf16 residual; the
 *     state-gradient pass (as gdn_summary_bwd's), which walks each (sequence, head) backwards
 *     and stores the gradient leaving every chunk; then a chunk-parallel pass that forms every
 *     (chunk, head)'s gradients from its entering state, that stored gradient and its WY
 *     record with tcgen05 products (bf16 hi + lo splits where fp32 gradients depend on them).
 *     Full chunks of dq, dk, dv leave by TMA when their rows are 16-byte aligned;
 *   - otherwise (other head sizes, a workspace of at least la_gdn_bwd_workspace_bytes_min but
 *     less than the above) the tile kernel: one CTA per (sequence, head) walks the chunks in
 *     reverse with warp-level tensor-core MMAs, in four chunk ranges launched one after the
 *     other when the units outnumber the CTAs the GPU holds at once (the state gradient handed
 *     from range to range exactly, the same bits as one walk).
 * Every (sequence, head) runs in a fixed order on either schedule, so results do not depend on
 * the batch around a sequence.  With gdn_fwd's input
 * transforms (cudnn-frontend PR #616 fusions) dg and dbeta are the gradients of the raw inputs
 * (the gate input, the beta logits), and the softplus gate also gives d_a_log and d_dt_bias,
 * summed over the batch in a fixed order (deterministic).
 */
la_status gdn_bwd(const la_gdn_bwd_params* p, void* stream);

/* Bytes of device workspace gdn_bwd needs (checkpoints_given = 0 when they are regenerated,
   1 for fp32 rows every 64 tokens), with room for the tensor-core schedule when K = V = 128. */
size_t la_gdn_bwd_workspace_bytes(int64_t T, int32_t N, int32_t HK, int32_t HV, int32_t K, int32_t V,
                                  int32_t checkpoints_given);

/* Bytes of device workspace gdn_bwd needs with given checkpoint rows every checkpoint_every_n
   tokens (0: none given), fp32 or bf16 (checkpoint_bf16): room for the tensor-core schedule
   when K = V = 128 (the split layout's WY records, T's residual and the gradient leaving every
   (chunk, head), about 90 KB per chunk and head more than the tile kernel needs). */
size_t la_gdn_bwd_workspace_bytes_ckpt(int64_t T, int32_t N, int32_t HK, int32_t HV, int32_t K, int32_t V,
                                       int64_t checkpoint_every_n, int32_t checkpoint_bf16);

/* The least workspace gdn_bwd accepts for the same call: the tile kernel's (a smaller one
   gives LA_ERR_WORKSPACE; one between this and la_gdn_bwd_workspace_bytes_ckpt selects the
   tile kernel).  0 for invalid arguments. */
size_t la_gdn_bwd_workspace_bytes_min(int64_t T, int32_t N, int32_t HK, int32_t HV, int32_t K, int32_t V,
                                      int64_t checkpoint_every_n, int32_t checkpoint_bf16);

/* Parameters of gdn_summary_bwd.  Strides are in elements. */
typedef struct la_gdn_summary_bwd_params {
    const void* q;    int64_t q_stride_t, q_stride_h;       /* [T, HK, K] bf16 */
    const void* k;    int64_t k_stride_t, k_stride_h;       /* [T, HK, K] bf16 */
    const float* g;   int64_t g_stride_t, g_stride_h;       /* [T, HO] fp32, natural-log gate */
    const float* beta; int64_t beta_stride_t, beta_stride_h; /* [T, HO] fp32 */
    const void* cu_seqlens;                                 /* [N + 1]: one span per entry */
    int32_t cu_seqlens_bits;
    int64_t T;
    int32_t N, HK, HV, K, V;
    float scale;                 /* <= 0: 1 / sqrt(K) */
    int32_t use_qk_l2norm;
    const void* d_o;  int64_t d_o_stride_t, d_o_stride_h;   /* [T, HO, V] bf16: the outputs' cotangent */
    const float* d_final_state;  /* [N, HO, K, V] fp32 cotangent of each span's end state, or NULL (zero) */
    float* d_state;              /* [N, HO, K, V] fp32 out: gradient w.r.t. the state entering each span */
    void* workspace;             /* >= la_gdn_summary_bwd_workspace_bytes(...), 256-byte aligned, or NULL */
    size_t workspace_bytes;
    int32_t* status;
    /* ---- optional input transforms, as in gdn_fwd / gdn_summary (zero-initialised: none) ---- */
    int32_t gate_mode;
    const float* a_log;
    const float* dt_bias;
    float gate_lower_bound;
    int32_t beta_sigmoid;
    int32_t beta_bf16;
} la_gdn_summary_bwd_params;

/*
 * gdn_summary_bwd -- the state-gradient mirror of gdn_summary.
 *
 * Page (cuDNN Linear Attention, "Summaries"): the summary ops come in pairs, <op>_summary and
 * <op>_summary_bwd, the second being the first's counterpart on the state gradient; the pair
 * gives context parallelism over spans.  Read here as: for each span (sequence) and head, the gradient of L = sum(d_o * o) +
 * sum(d_final_state * S_end) with respect to the state entering the span,
 *
 *   d_state = transition applied to d_final_state + dS_H,   dS_H = the same with d_final_state = 0,
 *
 * i.e. dS_enter[a][v] = sum_b transition[a][b] dS_exit[b][v] + dS_H[a][v] with gdn_summary's
 * transition.  That gradient does not depend on the entering state or on v (the map from the
 * state to the outputs is affine), so neither is an input and no forward pass runs.  Errors and
 * ownership as gdn_summary; g and beta go through gdn_fwd's input transforms when named.
 * Two paths: when the workspace has room for the forward's WY records
 * (la_gdn_fwd_split_workspace_bytes(T, N, HV); with workspace = NULL the internal buffer grows to
 * it) and d_o is 16-byte aligned with strides in 16-byte units, the WY pass and a state-gradient
 * pass on the tensor cores (the state gradient in TMEM, bf16 hi + lo operands); otherwise a tile
 * kernel on warp-level MMAs (split tf32 operands), whose result equals gdn_bwd's d_initial_state
 * bit for bit.  The two agree to fp32-level tolerance; each is bitwise independent of the batch.
 */
la_status gdn_summary_bwd(const la_gdn_summary_bwd_params* p, void* stream);

/* Bytes of device workspace gdn_summary_bwd needs (the tile kernel's path; the tensor-core path
   needs la_gdn_fwd_split_workspace_bytes(T, N, HV)). */
size_t la_gdn_summary_bwd_workspace_bytes(int32_t N, int32_t HV, int32_t K, int32_t V);

/* Bytes of device workspace gdn_fwd needs with num_householder = n > 1: for n <= 64 (run
   natively on the update timeline) the two-pass workspace of that timeline (T * n rows; a
   smaller workspace of at least la_gdn_workspace_bytes(N, 0) takes the fused kernel, the same
   bits); for n > 64 the timeline's query, gate and output rows plus the chunk kernel's scratch.
   n <= 1: la_gdn_workspace_bytes. */
size_t la_gdp_workspace_bytes(int64_t T, int32_t N, int32_t HK, int32_t HV, int32_t K, int32_t V, int32_t n);

/* Bytes of device workspace gdn_fwd (summary = 0) or gdn_summary (summary = 1) needs. */
size_t la_gdn_workspace_bytes(int32_t N, int32_t summary);

/* Bytes of device workspace with which gdn_fwd (num_householder <= 1) or gdn_summary may run
   as two passes (see gdn_fwd, "Two passes"; N counts the spans for gdn_summary):
   la_gdn_workspace_bytes(N, 0) plus per-chunk tables and one 17408-byte record per
   (chunk, head), at most (T / 64 + N) * HV of them (0.57 GB for T = 65536, N = 8, HV = 32). */
size_t la_gdn_fwd_split_workspace_bytes(int64_t T, int32_t N, int32_t HV);

/*
 * Host helper: total checkpoint rows R = sum_i ceil(L_i / n) for a HOST copy of
 * cu_seqlens (idx_bits 32 or 64).  Returns LA_ERR_INVALID_ARG for n <= 0 or a
 * decreasing cu_seqlens.
 */
la_status la_checkpoint_rows(const void* cu_seqlens_host, int32_t idx_bits, int32_t N, int64_t n,
                             int64_t* rows_out);

/*
 * Reads a device status word written by gdn_fwd / gdn_summary.  Synchronises
 * `stream` first, so it belongs in tests and error paths, not in a hot loop.
 */
la_status la_read_status(const int32_t* device_status, void* stream, int32_t* out);

/*
 * Profiling hook: record `start_event` and `stop_event` (cudaEvent_t handles) on
 * the launch stream immediately before and after the fused chunk kernel of the
 * next gdn_fwd / gdn_summary call (the decode kernel of the next gdn_decode call,
 * the backward kernels of the next gdn_bwd / gdn_summary_bwd call) made by this
 * host thread, so a caller can time
 * that kernel alone with CUDA events.  The hook is consumed by that one call;
 * pass NULL, NULL to clear it.  Not part of the computation; no citation.
 */
la_status la_set_kernel_timing_events(void* start_event, void* stop_event);

/*
 * Failure-path test hook, not for production use (no counterpart on the pages).
 * skip_tile_load != 0 makes the forward's chunk kernel issue no K/Q tile loads,
 * so its first bounded wait can never complete and it reports LA_ERR_TIMEOUT in
 * the status word; wait_budget_ns > 0 replaces the 1 s budget of every bounded
 * wait of the forward.  The settings are process-wide and apply to every later
 * gdn_fwd call from any thread until cleared with (0, 0); nothing else sets
 * them (the library reads no environment variables).
 */
la_status la_test_set_wait_hooks(int32_t skip_tile_load, uint64_t wait_budget_ns);

/*
 * Scheduling test hook, not for production use (no counterpart on the pages).
 * pieces = 0 restores the automatic choice of gdn_fwd's chunk ranges (see
 * gdn_fwd, "Scheduling"); 1 makes every later gdn_fwd call walk whole
 * sequences; 2..16 makes it walk every sequence in that many ranges whenever
 * the walks outnumber one wave and final_state is fp32 (or the pool is), so
 * that tests can compare ranged and whole walks bitwise on any batch.
 * Process-wide, like la_test_set_wait_hooks.  LA_ERR_INVALID_ARG for pieces
 * outside 0..16.
 */
la_status la_test_set_fwd_pieces(int32_t pieces);

/*
 * Scheduling test hook, not for production use (no counterpart on the pages).
 * passes = 0 restores the automatic choice between the fused and the two-pass
 * forward and summary (see gdn_fwd, "Two passes"); 1 makes every later
 * gdn_fwd and gdn_summary call use the fused kernel; 2 the two passes wherever
 * the workspace allows them.
 * Process-wide.  LA_ERR_INVALID_ARG for passes outside 0..2.
 */
la_status la_test_set_fwd_passes(int32_t passes);

/* Static description of a status code. */
const char* la_status_string(la_status s);

/* Library version, major * 10000 + minor * 100 + patch. */
int32_t la_version(void);

#ifdef __cplusplus
}
#endif

#endif /* LIBLINATTN_H */
