/*
 * gdn_scan.h - C ABI of the GB300 (sm_103a) Gated DeltaNet state-scan library.
 *
 * The operation (notes page "Tail-Replay: Escaping the Curse of Linear
 * Attention in Prefix Caching for Hybrid LLMs", section 2.3, equation (1),
 * in the right-multiplied layout the same section requires for a state
 * S in R^{d_v x d_k}):
 *
 *     S_t = alpha_t * S_{t-1} (I - beta_t k_t k_t^T) + beta_t v_t k_t^T,
 *     o_t = S_t q_t                      (readout of the post-update state)
 *
 * run independently for every (sequence, head) of a ragged batch.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Token streams are packed over the batch: q, k are [T, H, d_k], v is
 *    [T, H, d_v], alpha and beta are [T, H] fp32, all row-major (last index
 *    fastest), where T = cu_seqlens[B] and sequence b owns rows
 *    [cu_seqlens[b], cu_seqlens[b+1]).  q/k/v are fp32 or bf16 (qkv_dtype);
 *    bf16 values are widened exactly to fp32.
 *  - States are fp32 [d_v, d_k] row-major (key index fastest), stacked as
 *    [.., H, d_v, d_k].  All arithmetic is fp32.
 *  - Positions are 1-based as on the pages: "token t" is row t-1 of its
 *    sequence; "the state at c" is the state after token c.
 *  - Device pointers must be 16-byte aligned (q, k, v, states) or aligned
 *    to their element size (alpha, beta, o).  Host arrays are read before the
 *    call returns.  Device work is enqueued on `stream` (NULL = the legacy
 *    default stream) and is complete when the stream is; outputs are valid
 *    only then.
 *  - The caller owns every buffer.  The library allocates no device memory;
 *    it needs a small caller-provided workspace (gdn_workspace_size bytes,
 *    16-byte aligned) that carries a sticky device status word.  A larger
 *    workspace (gdn_workspace_size_two_pass bytes) lets the chunked scan
 *    precompute the per-chunk matrices of every chunk in parallel first
 *    (GDN_ALGO_CHUNKED_TWO_PASS), which AUTO then prefers.
 *  - Errors: a non-GDN_OK status.  Invalid arguments are detected on the
 *    host before anything is enqueued; outputs are then untouched.  A
 *    kernel-side failure (a bounded wait that ran out) is reported later by
 *    gdn_read_status on the same workspace.
 *  - Supported sizes: d_k, d_v in {32, 64, 128}; T < 2^31; H * d_v * d_k
 *    state elements per sequence fit in 2^40.  alpha must lie in (0, 1]
 *    (results are exact to fp32 rounding for alpha >= 1e-30), beta is any
 *    finite value.
 */
#ifndef GDN_SCAN_H
#define GDN_SCAN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t. */
typedef struct CUstream_st* gdn_stream_t;

typedef enum gdn_status {
    GDN_OK = 0,
    GDN_ERR_INVALID_ARG = 1,    /* bad pointer, size, position or alignment      */
    GDN_ERR_UNSUPPORTED = 2,    /* valid but not supported (e.g. d_k = 96)        */
    GDN_ERR_CUDA = 3,           /* a CUDA runtime / driver call failed            */
    GDN_ERR_DEVICE_TIMEOUT = 4  /* a kernel's bounded wait ran out (see read_status) */
} gdn_status;

typedef enum gdn_dtype { GDN_F32 = 0, GDN_BF16 = 1 } gdn_dtype;

/* Which kernel runs the scan.  All compute the same recurrence in fp32 state
 * precision; they differ in rounding order only.
 *  GDN_ALGO_AUTO         when supported (d_k = d_v = 128, bf16 q/k/v)
 *                        GDN_ALGO_CHUNKED_TWO_PASS if the workspace is large
 *                        enough for it, else GDN_ALGO_CHUNKED; otherwise per-token
 *  GDN_ALGO_PER_TOKEN    token by token on the FP32 pipes (any supported size)
 *  GDN_ALGO_CHUNKED      chunks of up to 64 tokens (WY / UT-transform form) on the
 *                        5th-generation tensor cores (tcgen05, accumulators and
 *                        state in tensor memory); non-exact operands are split into
 *                        two bf16 halves with fp32 accumulation.  A chunk also ends
 *                        where the decay product within it would fall below 2^-32,
 *                        so every alpha in (0, 1] is handled.
 *  GDN_ALGO_CHUNKED_MMA  the same chunkwise form on warp-level mma.sync, 64-token
 *                        chunks only: the decay product over one chunk must stay
 *                        above 2^-126 (alpha^64 > 1.2e-38), else results are not
 *                        finite.
 *  GDN_ALGO_CHUNKED_TWO_PASS  the chunks of GDN_ALGO_CHUNKED (same chunk ends), in
 *                        three launches: the chunk schedule of every (range, head),
 *                        T = (I + L)^-1 of every chunk at once on every SM, then the
 *                        tcgen05 state scan, which no longer waits for T.  Needs a
 *                        workspace of gdn_workspace_size_two_pass bytes for the
 *                        call (GDN_ERR_INVALID_ARG with a smaller one).
 * The chunked algorithms return GDN_ERR_UNSUPPORTED for other sizes.  Calls whose
 * results are compared bit for bit (a resume against its prefill) must use the
 * same algorithm: the chunked ones differ from each other in rounding order. */
typedef enum gdn_algo {
    GDN_ALGO_AUTO = 0,
    GDN_ALGO_PER_TOKEN = 1,
    GDN_ALGO_CHUNKED = 2,
    GDN_ALGO_CHUNKED_MMA = 3,
    GDN_ALGO_CHUNKED_TWO_PASS = 4
} gdn_algo;

typedef struct gdn_problem {
    int32_t num_seqs;            /* B >= 1                                           */
    int32_t num_heads;           /* H >= 1                                           */
    int32_t d_k;                 /* key / query width                                */
    int32_t d_v;                 /* value width = rows of the state                  */
    const int64_t* cu_seqlens;   /* host [B+1]: 0 = cu[0] <= cu[1] <= ... = T        */
    gdn_dtype qkv_dtype;         /* dtype of q, k, v                                 */
    gdn_dtype out_dtype;         /* dtype of the readout o (rounded to nearest even) */
    gdn_algo algo;               /* kernel choice (GDN_ALGO_AUTO by default)          */
} gdn_problem;

/*
 * Prefill with sparse exact checkpoints.
 * ("Sparse prefix caching in hybrid and recurrent LLM serving", section 3:
 * exact recurrent states are stored at positions 1 <= c_1 < ... < c_M <= N.)
 *
 * For every sequence b and head h, scan tokens 1..N_b from S0[b, h] (zeros
 * when S0 is NULL), write the readout of every token to o (skipped when o is
 * NULL), dump the state after each checkpoint position and write the state
 * after token N_b to S_final.
 *
 *  q            device [T, H, d_k]   (may be NULL when o is NULL)
 *  k            device [T, H, d_k]
 *  v            device [T, H, d_v]
 *  alpha, beta  device [T, H] fp32
 *  S0           device [B, H, d_v, d_k] fp32, or NULL for zero initial states
 *  o            device [T, H, d_v] out_dtype, or NULL
 *  S_final      device [B, H, d_v, d_k] fp32
 *  ckpt_pos     host, concatenated per sequence: the M_b positions of sequence
 *               b are ckpt_pos[cu_ckpt[b] .. cu_ckpt[b+1]), strictly
 *               increasing, each in [1, N_b]
 *  cu_ckpt      host [B+1], cu_ckpt[0] = 0, non-decreasing (NULL = no checkpoints)
 *  ckpt_states  device [cu_ckpt[B], H, d_v, d_k] fp32: slot cu_ckpt[b] + i
 *               receives the state after token ckpt_pos[cu_ckpt[b] + i]
 */
gdn_status gdn_prefill_ckpt(const gdn_problem* p, const void* q, const void* k, const void* v,
                            const float* alpha, const float* beta, const float* S0, void* o,
                            float* S_final, const int64_t* ckpt_pos, const int64_t* cu_ckpt,
                            float* ckpt_states, void* workspace, size_t ws_bytes,
                            gdn_stream_t stream);

/*
 * Resume from the deepest stored checkpoint.
 * ("Sparse prefix caching ...", section 3: for overlap depth d take
 * j = argmax{c_i <= d}, restore S_{c_j}, recompute tokens c_j+1 .. d; nothing
 * to recompute when c_j = d.)  With no checkpoint at or below d the scan
 * starts from the initial state S0[s] (zeros when S0 is NULL), i.e. c_0 = 0.
 *
 *  q, k, v, alpha, beta   the packed streams of gdn_prefill_ckpt
 *  S0           device [B, H, d_v, d_k] or NULL (the c_0 = 0 state)
 *  ckpt_states, ckpt_pos, cu_ckpt   as written / read by gdn_prefill_ckpt
 *  num_probes   P >= 0
 *  probe_seq    host [P]: sequence of each probe, in [0, B)
 *  probe_depth  host [P]: overlap depth d in [0, N_seq]
 *  S_out        device [P, H, d_v, d_k]: state after token d
 *  o_out        device [R, H, d_v] out_dtype or NULL: readout of the
 *               recomputed tokens, probe p's tokens c_j+1..d packed at rows
 *               [o_offsets[p], o_offsets[p+1]) in probe order,
 *               R = sum_p (d_p - c_jp)
 *  chosen_pos   host [P] out (nullable): c_j of each probe (0 = initial state)
 *  o_offsets    host [P+1] out (nullable): the packing offsets above
 */
gdn_status gdn_resume_from_ckpt(const gdn_problem* p, const void* q, const void* k, const void* v,
                                const float* alpha, const float* beta, const float* S0,
                                const float* ckpt_states, const int64_t* ckpt_pos,
                                const int64_t* cu_ckpt, int32_t num_probes,
                                const int32_t* probe_seq, const int64_t* probe_depth, float* S_out,
                                void* o_out, int64_t* chosen_pos, int64_t* o_offsets,
                                void* workspace, size_t ws_bytes, gdn_stream_t stream);

/*
 * Tail-Replay state recovery.
 * (Tail-Replay notes page, section 2.1 table: k = ceil(r m), a = m - k;
 * section 2.2 steps 2-3: set the state to zero at the tail start and run the
 * k tail tokens, i.e. positions a+1 .. m, giving the approximation S_hat_m.)
 *
 *  q, k, v, alpha, beta   full prefix streams; only rows [cu[b]+a_b, cu[b]+m_b) are read
 *                         (q only when o is non-NULL)
 *  m            host [B]: matched prefix length, 0 <= m_b <= N_b
 *  r_num/r_den  the replay ratio r = r_num / r_den, 0 <= r_num <= r_den, r_den > 0;
 *               k_b = ceil(r m_b) is computed exactly in integers
 *  S_a          device [B, H, d_v, d_k] or NULL: the exact state at a_b.  When
 *               given, the same tokens are also run from S_a ("exact twin"),
 *               giving S_m, so that E_m = S_m - S_hat_m can be formed
 *  S_hat        device [B, H, d_v, d_k]: the replayed state (zeros when k_b = 0)
 *  S_exact      device [B, H, d_v, d_k]: required iff S_a is given
 *  o            device [T, H, d_v] out_dtype or NULL: readout of S_hat over the
 *               replayed tokens, written at their own stream rows
 *  a_out, k_out host [B] out (nullable): a_b and k_b
 */
gdn_status gdn_tail_replay(const gdn_problem* p, const void* q, const void* k, const void* v,
                           const float* alpha, const float* beta, const int64_t* m, int32_t r_num,
                           int32_t r_den, const float* S_a, float* S_hat, float* S_exact, void* o,
                           int64_t* a_out, int64_t* k_out, void* workspace, size_t ws_bytes,
                           gdn_stream_t stream);

/*
 * Tail replay with a caller-chosen tail length per sequence: rows [m_b - k_b, m_b)
 * of sequence b from a zero state (and the exact twin from S_a when given).  Same
 * buffers and rules as gdn_tail_replay; k_replay host int64 [B] with
 * 0 <= k_b <= m_b (e.g. from gdn_adaptive_replay_plan).
 */
gdn_status gdn_tail_replay_k(const gdn_problem* p, const void* q, const void* k, const void* v,
                             const float* alpha, const float* beta, const int64_t* m, const int64_t* k_replay,
                             const float* S_a, float* S_hat, float* S_exact, void* o, void* workspace,
                             size_t ws_bytes, gdn_stream_t stream);

/*
 * One serving step's scans in a single launch: the prefills of gdn_prefill_ckpt,
 * the resumes of gdn_resume_from_ckpt and the tail replays of gdn_tail_replay over
 * the same packed streams, as one job list ordered longest first.  The short
 * resume and replay jobs then run on the multiprocessors that the long prefills
 * leave free, instead of after them.  The setting is the pages' serving step: the
 * "Sparse prefix caching ..." page (section 3) serves new prompts that store
 * checkpoints beside requests resumed from checkpoints stored earlier, and the
 * "Tail-Replay" notes page (section 2.2) recovers the states of cache hits by
 * replay.
 *
 * Each part is optional (NULL skips it) and takes the arguments of its own entry
 * point, with the same meaning, index plan and checks; every state and output
 * equals, bit for bit, what that entry point gives for the same part on its own.
 * The exact twin of a replay (S_a given) runs as jobs of its own; on the
 * token-by-token kernel (sizes other than d_k = d_v = 128 with bf16 q/k/v), whose
 * replay entry point runs the twin beside the replay in one block, S_exact then
 * agrees with it to rounding rather than bit for bit.
 *
 * On the tensor-core path, when a few long scans come with many scans at most a
 * quarter of their length (and the long ones fit on the GPU's multiprocessors at
 * once), the two groups run as two launches side by side on streams of the
 * library's own (the long one of the highest priority, so that its blocks are
 * placed first), forked from `stream` and joined back to it with events: work
 * enqueued on `stream` before the call is waited for, and work enqueued after it
 * waits for both launches.  The first such call on a device creates those two
 * streams and three events (kept until the process exits; make the first call
 * before any stream capture); calls from several host threads share them.
 *
 * The parts of one call run at the same time, so none may read what another
 * writes: the resumes read checkpoints stored by earlier calls, and
 * resume->ckpt_states overlapping prefill->ckpt_states is GDN_ERR_INVALID_ARG;
 * no output may alias an input or another output (not checked).  q may be NULL
 * only when no part has a readout.  The per-part host outputs (chosen_pos,
 * o_offsets, a_out, k_out) are written once every check has passed.
 */
typedef struct gdn_prefill_args {
    const float* S0;            /* as gdn_prefill_ckpt                              */
    void* o;
    float* S_final;
    const int64_t* ckpt_pos;
    const int64_t* cu_ckpt;
    float* ckpt_states;         /* written by this call                             */
} gdn_prefill_args;

typedef struct gdn_resume_args {
    const float* S0;            /* as gdn_resume_from_ckpt                          */
    const float* ckpt_states;   /* read by this call: stored by an earlier one      */
    const int64_t* ckpt_pos;
    const int64_t* cu_ckpt;
    int32_t num_probes;
    const int32_t* probe_seq;
    const int64_t* probe_depth;
    float* S_out;
    void* o_out;
    int64_t* chosen_pos;
    int64_t* o_offsets;
} gdn_resume_args;

typedef struct gdn_replay_args {
    const int64_t* m;           /* as gdn_tail_replay                               */
    int32_t r_num;
    int32_t r_den;
    const float* S_a;
    float* S_hat;
    float* S_exact;
    void* o;
    int64_t* a_out;
    int64_t* k_out;
} gdn_replay_args;

gdn_status gdn_step(const gdn_problem* p, const void* q, const void* k, const void* v,
                    const float* alpha, const float* beta, const gdn_prefill_args* prefill,
                    const gdn_resume_args* resume, const gdn_replay_args* replay, void* workspace,
                    size_t ws_bytes, gdn_stream_t stream);

/*
 * Tail replay with the prefix's cached attention KV copied to the device at the
 * same time ("Tail-Replay" notes page, section 2.5, transfer / replay overlap:
 * the replay needs only the tail's inputs, not the KV, so the two run on
 * different streams and join before the new suffix is processed; the page's
 * latency model T_overlap ~ max(T_KV, T_replay) + T_other against
 * T_serial ~ T_KV + T_replay + T_other).
 *  Arguments as gdn_tail_replay, plus:
 *  kv_host     host buffer of kv_bytes (pinned memory for a truly asynchronous copy)
 *  kv_dev      device buffer of kv_bytes
 *  copy_stream stream for the copy.  The copy starts after the work already
 *              enqueued on `stream` (which may still use kv_dev), runs beside the
 *              replay, and `stream` waits for it after the replay, so work enqueued
 *              on `stream` afterwards sees the copied KV.  kv_bytes = 0 copies nothing.
 *  Every argument is checked before anything is enqueued (GDN_ERR_INVALID_ARG);
 *  GDN_ERR_CUDA if enqueueing the copy or its events fails.
 */
gdn_status gdn_tail_replay_overlap(const gdn_problem* p, const void* q, const void* k, const void* v,
                                   const float* alpha, const float* beta, const int64_t* m, int32_t r_num,
                                   int32_t r_den, const float* S_a, float* S_hat, float* S_exact, void* o,
                                   int64_t* a_out, int64_t* k_out, const void* kv_host, void* kv_dev,
                                   size_t kv_bytes, void* workspace, size_t ws_bytes, gdn_stream_t stream,
                                   gdn_stream_t copy_stream);

/*
 * Adaptive tail length per request ("Tail-Replay" notes page, section 5, the
 * proposed extension: shorter tails where the state forgets fast, longer ones or
 * exact recovery where it does not).  With unit keys and beta in [0, 2] the
 * replay error obeys ||E_m||_F <= (alpha_{a+1} ... alpha_m) ||S_a||_F (section 2.3),
 * so for each sequence b: k_b = the least k <= ceil(rmax_num m_b / rmax_den) with
 * alpha_m alpha_{m-1} ... alpha_{m-k+1} <= eps for every head (the product taken in
 * fp32, newest gate first), and exact_out[b] = 0; when the budget is too short for
 * some head, k_b is the budget and exact_out[b] = 1 (recover that request exactly,
 * e.g. from a checkpoint).
 *  alpha     device [T, H] fp32 (only the budget's tail rows are read; they are
 *            copied to the host on `stream`, which the call then synchronises: work
 *            enqueued on `stream` before the call, e.g. what writes the gates, is
 *            complete before they are read)
 *  m         host int64 [B]; eps in [0, 1); rmax_num / rmax_den as in gdn_replay_plan
 *  k_out     host int64 [B]; exact_out host int32 [B]
 */
gdn_status gdn_adaptive_replay_plan(const gdn_problem* p, const float* alpha, const int64_t* m, float eps,
                                    int32_t rmax_num, int32_t rmax_den, int64_t* k_out, int32_t* exact_out,
                                    gdn_stream_t stream);

/*
 * In-group chained replay ("Tail-Replay" notes page, section 2.2 step 3 and
 * section 2.4): the linear-attention layers of one group are replayed one after
 * the other from zero states over the tail a+1..m (k = ceil(r m) exact, a = m - k),
 * the first layer reading the group's exact cached input hidden states h and every
 * later layer the previous layer's replayed outputs; the last layer needs only its
 * state (its output feeds nothing the recovery uses).  With S_exact the same
 * chain also runs over 1..m (the full prefill) for comparison.
 *
 * The pages fix no model, so the group is synthetic, with weights given per layer
 * l (fp32, contiguous, layer after layer; D = d_model, Hd = heads * d_head):
 *   W_q [Hd, D], W_k [Hd, D], W_v [Hd, D], w_a [heads, D], w_b [heads, D], W_o [D, Hd]
 * and, per token t and head: q = W_q h / |W_q h|, k = W_k h / |W_k h|, v = W_v h,
 * alpha = 1 - 0.1 sigmoid(w_a . h), beta = sigmoid(w_b . h); next layer's input
 * h + W_o [o_1; ...; o_heads] (o_t = S_t q_t per head).
 *
 *  g          layers 1..64, heads 1..1024, d_model 1..8192, d_head in {32, 64, 128},
 *             heads * d_head <= 8192
 *  h          device [m, d_model] fp32 (one request's rows)
 *  weights    device, layers * (4 Hd + 2 heads) * d_model floats
 *  S_hat      device [layers, heads, d_head, d_head] fp32 out (replayed states at m)
 *  S_exact    device, same shape, or null (skip the full chain)
 *  a_out, k_out  host int64 out (nullable)
 *  scratch    device, 16-byte aligned, at least gdn_group_scratch_bytes(g, rows)
 *             bytes with rows = m when S_exact is given, else k
 *  workspace  as for the other device entry points
 * Invalid arguments: GDN_ERR_INVALID_ARG before anything is enqueued.
 */
typedef struct gdn_group {
    int32_t layers;
    int32_t heads;
    int32_t d_model;
    int32_t d_head;
} gdn_group;

size_t gdn_group_scratch_bytes(const gdn_group* g, int64_t rows);

gdn_status gdn_group_replay(const gdn_group* g, const float* h, int64_t m, int32_t r_num, int32_t r_den,
                            const float* weights, float* S_hat, float* S_exact, int64_t* a_out, int64_t* k_out,
                            void* scratch, size_t scratch_bytes, void* workspace, size_t ws_bytes,
                            gdn_stream_t stream);

/*
 * Prefill with sparse checkpoints for callers that cannot allocate device memory.
 * (No counterpart on the pages: this is a calling convention of this library.)
 *
 * Same arguments and results as gdn_prefill_ckpt, without the workspace. It is
 * meant for callers that are handed their input and output buffers but have
 * no device allocator of their own -- for instance a plugin inside a serving
 * engine whose memory pool owns all of HBM, or a latency-critical loop that
 * cannot afford cudaMalloc's implicit synchronisation. Neither this call nor
 * anything it calls allocates device memory.
 *
 * Instead of a workspace it uses a 256-byte static device array inside the
 * library (the maximum scratch it can hold; a build whose scan needs more
 * returns GDN_ERR_UNSUPPORTED). Every GPU that loads the library keeps that
 * array until the process exits.
 *  - The first call on each device looks up the array's device address (with
 *    that device current) and caches it for the rest of the process; make that
 *    first call before any stream capture.  The cached address does not survive
 *    cudaDeviceReset (which unloads the library's device code): do not call this
 *    entry point on a device after resetting it.
 *  - Every call on a device shares the one array. The call clears it on
 *    `stream` before launching, so calls whose work overlaps on the GPU (e.g.
 *    from several host threads on different streams) race on it; serialise them.
 *  - The call synchronises `stream` before returning, so that it can report a
 *    device-side wait expiry (GDN_ERR_DEVICE_TIMEOUT) without a workspace.
 *  - Invalid arguments are rejected exactly as by gdn_prefill_ckpt; only the
 *    library's own array has been cleared by then.
 */
gdn_status gdn_prefill_ckpt_noalloc(const gdn_problem* p, const void* q, const void* k, const void* v,
                                    const float* alpha, const float* beta, const float* S0, void* o,
                                    float* S_final, const int64_t* ckpt_pos, const int64_t* cu_ckpt,
                                    float* ckpt_states, gdn_stream_t stream);

/* --- host-only helpers (no GPU needed) ------------------------------------------------ */

/* Tail-Replay notes page, section 2.1 table: k = ceil(r_num * m / r_den), a = m - k.
 * GDN_ERR_INVALID_ARG when m < 0, m > 2^40, r_den <= 0 or r_num outside [0, r_den]. */
gdn_status gdn_replay_plan(int64_t m, int32_t r_num, int32_t r_den, int64_t* a, int64_t* k);

/* "Sparse prefix caching ...", section 3: *j = 0-based index of the deepest
 * c_i <= d in the strictly increasing c[0..M), or -1 when none (resume from
 * the initial state).  GDN_ERR_INVALID_ARG when c is not strictly increasing. */
gdn_status gdn_select_ckpt(const int64_t* c, int32_t M, int64_t d, int32_t* j);

/* --- checkpoint placement (host only) -------------------------------------------------
 * "Sparse prefix caching in hybrid and recurrent LLM serving", sections 3-5.  A
 * cached prefix of N tokens keeps states at 1 <= c_1 < ... < c_M <= N; a request
 * overlapping it to depth d recomputes f(d) = d - max{c_i <= d} tokens (the start,
 * c_0 = 0, when no c_i <= d; f(0) = 0).  The depth distribution is given as integer
 * weights w[0..N] (host array, w[d] >= 0, e.g. counts of observed depths), so the
 * expected recompute is the exact integer numerator R = sum_d w[d] f(d) (divide by
 * sum_d w[d] for tokens per request).  Inputs must satisfy 1 <= N < 2^31 and
 * sum_d d w[d] < 2^60 and N sum_d w[d] < 2^60 (else GDN_ERR_UNSUPPORTED). */
typedef enum gdn_placement {
    GDN_PLACE_DP = 0,        /* optimal: dynamic programme of Theorem 2 in O(N M)
                                (monotone convex-hull trick); needs (M+1)(N+1) <= 2^26 */
    GDN_PLACE_BALANCED = 1,  /* Theorem 1: M+1 gaps summing to N+1 that differ by at
                                most one, the larger ones first (optimal for uniform d) */
    GDN_PLACE_BLOCK = 2,     /* block boundaries b, 2b, ... <= N, at most M of them;
                                b = `block`, or floor(N/M) when block = 0 */
    GDN_PLACE_RANDOM = 3,    /* M distinct positions: the first M draws of a Fisher-Yates
                                shuffle of 1..N driven by splitmix64(seed), sorted; N <= 2^24 */
    GDN_PLACE_GREEDY = 4     /* M times the free position that lowers R most (the
                                shallowest on ties); N <= 2^24 */
} gdn_placement;

/* Choose checkpoint positions.  M >= 0 is the budget; when M > N every position is
 * taken.  positions: host int64 [M], written strictly increasing in [1, N]; *count:
 * how many were written (M, or min(M, N), or fewer for GDN_PLACE_BLOCK); *cost: R of
 * the written placement.  GDN_ERR_INVALID_ARG on a null pointer, negative weight,
 * M < 0, block < 0 or an unknown strategy; nothing is written then. */
gdn_status gdn_ckpt_placement(const int64_t* weights, int64_t N, int32_t M, gdn_placement strategy,
                              uint64_t seed, int64_t block, int64_t* positions, int32_t* count,
                              int64_t* cost);

/* R = sum_d w[d] f(d) of a given placement positions[0..M) (host, strictly
 * increasing in [1, N]); GDN_ERR_INVALID_ARG otherwise. */
gdn_status gdn_expected_recompute(const int64_t* weights, int64_t N, const int64_t* positions, int32_t M,
                                  int64_t* cost);

/* Bytes of workspace every device entry point needs. */
size_t gdn_workspace_size(void);

/* Bytes of workspace with which a call can use GDN_ALGO_CHUNKED_TWO_PASS:
 * `tokens` = tokens scanned by the call summed over its ranges (prefill: T;
 * resume: the sum of the probe depths bounds it; tail replay: the sum of the
 * tails, plus the sum of m when S_a is given), `num_ranges` = ranges scanned
 * (sequences, probes; twice the sequences for a replay with S_a).  It holds
 * the status word, the chunk schedule and the T = (I + L)^-1 operands (256
 * bf16 per token and head).  0 for negative arguments or 2^29 - 64 token-heads
 * or more. */
size_t gdn_workspace_size_two_pass(int64_t tokens, int32_t num_heads, int32_t num_ranges);

/* Zero the sticky status word of a workspace (enqueued on stream). */
gdn_status gdn_clear_status(void* workspace, size_t ws_bytes, gdn_stream_t stream);

/* Synchronise `stream` and report the workspace's sticky device status:
 * GDN_OK, or GDN_ERR_DEVICE_TIMEOUT if any kernel that used it gave up on a wait. */
gdn_status gdn_read_status(const void* workspace, size_t ws_bytes, gdn_stream_t stream);

/* Time limit, in nanoseconds, of every device-side wait of later launches
 * from this process (default 2 s; 0 restores the default). */
void gdn_set_wait_limit_ns(uint64_t ns);

/* Testing hook for failure detection: kernels launched afterwards from this
 * process stop issuing their input copies after `chunks` chunks (of 32 tokens
 * per-token, 64 chunked), so the next wait of each CTA can only run out; the
 * CTA then drains its own copies, records GDN_ERR_DEVICE_TIMEOUT in the
 * workspace and returns (outputs are incomplete).  Negative disables (the
 * default).  Pair it with a short gdn_set_wait_limit_ns. */
void gdn_debug_stall_after(int32_t chunks);

/* Human-readable name of a status code. */
const char* gdn_status_string(gdn_status s);

#ifdef __cplusplus
}
#endif

#endif /* GDN_SCAN_H */
