/*
 * wf.h - C ABI of the GB300 (sm_103a) verify-and-route library for WhiFlash
 * token-level cross-paradigm speculative decoding.
 *
 * One speculation round of WhiFlash (WhiFlash paper, arXiv 2606.07710,
 * Sec. 3.2 "Proposed Architecture"): the target model verifies the drafted
 * candidates in parallel, decoding resumes from the last accepted token, and
 * the token-level router picks the drafter for the next round (Sec. 3.3).
 * This library covers the data-parallel arithmetic of that step once the
 * target's final hidden states exist:
 *
 *   wf_lmhead_argmax  target LM head + greedy choice at every verified row
 *   wf_verify_chain   DFlash block acceptance (longest matched prefix) + bonus
 *   wf_verify_tree    EAGLE-3 tree acceptance (deepest matched root path) + bonus
 *   wf_router_mlp     neural router f_theta and the threshold decision
 *   wf_draft_topk     EAGLE-3 draft head, top-k, draft-to-target id map
 *   wf_lmhead_draft_topk  the target and draft heads in one weight sweep
 *   wf_round          all of the above as one stream-ordered round
 *   wf_catchup        KV-only catch-up of the EAGLE-3 drafter after a switch
 *
 * Conventions shared by every call
 * - Pointers named as device buffers must be device (or managed) memory
 *   allocated by the caller; the library allocates nothing and keeps no
 *   per-call state outside the caller's workspace.  Operands the kernels copy
 *   with the tensor-memory accelerator or bulk copies (weight matrices,
 *   hidden states, backlog rows, the key / value caches) must be memory of
 *   the current device: a host pointer or another GPU's memory there returns
 *   WF_ERR_INVALID_ARG.
 * - bf16 tensors are passed as raw uint16 bit patterns, row-major, densely
 *   packed (row stride = number of columns), 16-byte aligned.
 * - Every call is asynchronous on `stream`: it validates its arguments on the
 *   host, enqueues kernels and returns.  Host-detectable errors (NULL
 *   pointers, sizes, alignment, workspace too small) are returned at once and
 *   nothing is enqueued.
 * - Data errors that only the device can see (a parent index outside
 *   [-1, node), a sequence longer than WF_MAX_SEQ_NODES, a draft id with no
 *   valid target id) set a sticky error word in the workspace and turn the
 *   affected outputs into -1.  The device never traps; read the word with
 *   wf_read_device_error.  Every wait inside a kernel is bounded
 *   (wf_set_wait_timeout_ns); a wait that gives up records WF_ERR_TIMEOUT.
 * - Stream order: a call reads its per-call inputs (hidden states, drafts,
 *   parents, offsets, rows, backlog) only after everything enqueued before it
 *   on `stream` has finished.  Model state — weight matrices, biases, gains,
 *   the draft-to-target map — may be fetched as soon as a kernel of the call
 *   starts, which can be while the previous kernel on the stream is still
 *   running (programmatic dependent launch): do not have work that is still
 *   in flight on the stream write it.
 * - Workspace: caller-owned device memory of at least wf_workspace_bytes()
 *   bytes, zeroed once with wf_workspace_init() before first use.  Calls
 *   leave it zeroed where that matters, so it can be reused without
 *   re-initialisation.  Calls that share a workspace must not overlap in time
 *   (use one stream, or one workspace per stream).
 */
#ifndef WF_H
#define WF_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define WF_API __attribute__((visibility("default")))
#else
#define WF_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t; NULL = the legacy default stream. */
struct CUstream_st;
typedef struct CUstream_st* wf_stream_t;

typedef enum wf_status {
    WF_OK = 0,
    WF_ERR_INVALID_ARG = 1,   /* NULL pointer, bad size or alignment; nothing enqueued */
    WF_ERR_WORKSPACE = 2,     /* workspace NULL, misaligned or below wf_workspace_bytes() */
    WF_ERR_CUDA = 3,          /* a CUDA runtime call or kernel launch failed */
    WF_ERR_UNSUPPORTED = 4,   /* device is not sm_103 (GB300) or shape outside the kernels' range */
    WF_ERR_BAD_DATA = 5,      /* device-side: malformed tree / id data (see above) */
    WF_ERR_TIMEOUT = 6        /* device-side: a bounded wait gave up */
} wf_status;

/* Longest drafted sequence (nodes, not rows) a single sequence may carry. */
#define WF_MAX_SEQ_NODES 256
/* Largest k of wf_draft_topk. */
#define WF_MAX_TOPK 16

/* Human-readable name of a status code (static storage). */
WF_API const char* wf_status_string(int status);

/* Library ABI version (major * 100 + minor). */
WF_API int wf_version(void);

/*
 * Workspace size (bytes) sufficient for every call below with at most
 * P verified rows, B sequences, hidden size d, router width m, draft
 * vocabulary Vd and top-k k (pass 0 for Vd / k when the draft head is not
 * used).
 */
WF_API size_t wf_workspace_bytes(int P, int B, int d, int m, int Vd, int k);

/* Zero a workspace (asynchronously on `stream`).  Needed once before first use. */
WF_API wf_status wf_workspace_init(void* ws, size_t ws_bytes, wf_stream_t stream);

/*
 * Copy the sticky device error word out of the workspace (synchronises
 * `stream`).  *code is a wf_status (WF_OK if none), *info a call-specific
 * detail (the offending sequence index for WF_ERR_BAD_DATA).  clear != 0
 * resets the word afterwards.
 */
WF_API wf_status wf_read_device_error(void* ws, int* code, int* info, int clear, wf_stream_t stream);

/*
 * Upper bound (ns) on any single wait inside a kernel before it gives up with
 * WF_ERR_TIMEOUT (process-wide; default 2e9 = 2 s; 0 restores the default).
 * Applies to launches made after the call.
 */
WF_API void wf_set_wait_timeout_ns(uint64_t ns);

/*
 * Diagnostic for the failure path: enqueues one kernel whose single wait (an
 * mbarrier nothing ever arrives on, the same bounded wait the pipelined
 * kernels use) gives up after timeout_ns (<= 1e10) and records WF_ERR_TIMEOUT
 * in the workspace error word; the context stays usable.  No passage of the
 * pages corresponds to it.
 */
WF_API wf_status wf_probe_bounded_wait(uint64_t timeout_ns, void* ws, size_t ws_bytes, wf_stream_t stream);

/*
 * Target LM head fused with the greedy choice (WhiFlash paper Sec. 3.3.1:
 * under greedy decoding the target's next token at a verified position is
 * the argmax of its next-token distribution; Sec. 4 "Evaluation": greedy
 * decoding; vocabulary 151,936 and hidden size 2560 for Qwen3-4B per the
 * Qwen3-4B-EAGLE3 card, "Technical Specifications").
 *
 *   ids[p]      = argmax_v sum_k hidden[p,k] * W[v,k]   (lowest v on a tie)
 *   maxlogit[p] = that maximum logit (fp32), optional (NULL = not written)
 *
 * hidden   device, [P, d] bf16 bits, the target's final hidden states
 * W        device, [V, d] bf16 bits, LM-head weight (out x in)
 * P        rows, 1 <= P;  d % 8 == 0, 8 <= d <= 16384;  1 <= V < 2^31
 * ids      device, [P] int32 out
 * Logits are accumulated in fp32 on the tensor cores and never stored.
 */
WF_API wf_status wf_lmhead_argmax(const uint16_t* hidden, const uint16_t* W, int P, int d, int V,
                           int32_t* ids, float* maxlogit, void* ws, size_t ws_bytes,
                           wf_stream_t stream);

/*
 * wf_lmhead_argmax without a workspace: same inputs, outputs and result as
 * wf_lmhead_argmax, but the scratch lives in a fixed array inside the
 * library, for callers that cannot allocate device memory (a plug-in that a
 * host engine calls with only its input and output buffers, or a decode loop
 * that may not call cudaMalloc because it synchronises the device).  The
 * pages have no counterpart to this entry point; it exists for those callers.
 *
 * Limits: P <= WF_NOALLOC_MAX_ROWS (else WF_ERR_INVALID_ARG, nothing
 * enqueued).  Every loaded GPU holds the array (about 128 KB) until the
 * process exits.  All calls on a device share it: calls that overlap on the
 * GPU race, so serialise them (one stream).  The first call on a device looks
 * up the array's address and should come before any stream capture.  It
 * allocates nothing; each call clears the part of the array it uses,
 * including the array's error word: read a call's device-side status with
 * wf_noalloc_read_device_error before the next call on that device.
 */
#define WF_NOALLOC_MAX_ROWS 16384
WF_API wf_status wf_lmhead_argmax_noalloc(const uint16_t* hidden, const uint16_t* W, int P, int d, int V,
                                          int32_t* ids, float* maxlogit, wf_stream_t stream);

/*
 * The device-side status left by the last wf_lmhead_argmax_noalloc call on the
 * current device (0, or WF_ERR_TIMEOUT if one of its bounded waits gave up;
 * *info as in wf_read_device_error).  Synchronises `stream` first; clear != 0
 * resets the word.  Like the entry point above, this has no counterpart on the
 * pages.
 */
WF_API wf_status wf_noalloc_read_device_error(int* code, int* info, int clear, wf_stream_t stream);

/*
 * Runtime-informed router, WhiFlash-Entropy (paper Sec. 3.3.1): at each
 * selected row the entropy of the target's next-token distribution,
 *   H[b]     = - sum_v p_v log p_v,  p = softmax(<hidden[row_b], W_v>) (natural log)
 *   route[b] = 1 (autoregressive drafter) if H[b] > tau, else 0 (diffusion drafter)
 * computed in the same weight sweep as an LM-head argmax (the logits stay in
 * TMEM), with fp32 online softmax statistics.
 *
 * hidden device [P, d] bf16 bits; rows device [B] int32 rows of hidden, or
 * NULL for rows 0 .. B-1 (then B <= P); 1 <= B <= 256; W as for
 * wf_lmhead_argmax.  H device [B] fp32; route device [B] int32 or NULL.  A
 * row outside [0, P) sets WF_ERR_BAD_DATA and writes NaN / -1 for it.
 */
WF_API wf_status wf_lmhead_entropy(const uint16_t* hidden, int P, int d, const int32_t* rows, int B,
                                   const uint16_t* W, int V, float tau, float* H, int32_t* route, void* ws,
                                   size_t ws_bytes, wf_stream_t stream);

/*
 * DFlash block verification (paper Sec. 3.2: the parallel block returns to
 * the target for parallel verification; App. A: block size 16 for Qwen3).
 * Sequence b owns verified rows pos_off[b] .. pos_off[b+1]-1; row pos_off[b]
 * holds the last committed token, row pos_off[b]+1+j draft token j.  Its
 * drafts are draft[node_off[b] .. node_off[b+1]-1]; node count = rows - 1.
 *
 *   n_accept[b] = largest n with draft[j] == g[pos_off[b]+j] for all j < n
 *   last_pos[b] = pos_off[b] + n_accept[b]   (global row, feeds the router)
 *   bonus[b]    = g[last_pos[b]]              (the target's own next token)
 *   path[b*path_stride + j] = j for j < n, -1 otherwise (NULL = not written)
 * Tokens committed this round (the paper's acceptance length, Sec. 4
 * "Metrics") = n_accept + 1.
 *
 * g, draft, pos_off [B+1], node_off [B+1]: device int32.  Outputs: device int32 [B].
 */
WF_API wf_status wf_verify_chain(const int32_t* g, const int32_t* draft, const int32_t* pos_off,
                          const int32_t* node_off, int B, int path_stride, int32_t* n_accept,
                          int32_t* bonus, int32_t* last_pos, int32_t* path, void* ws,
                          size_t ws_bytes, wf_stream_t stream);

/*
 * EAGLE-3 tree verification (paper Sec. 3.2: the autoregressive drafter
 * produces a tree of candidates; App. A / Table 7: depth 8, top-k 10, 60
 * draft tokens).  Same row / node layout as wf_verify_chain; parent[] holds
 * sequence-local parent indices, -1 = the root, and parent[i] < i.
 *
 *   node i is accepted iff tok[i] == g[row of parent(i)] and parent(i) is
 *   accepted (the root always is); n_accept = depth of the deepest accepted
 *   node (lowest index on a tie; 0 if none); last_pos = its row (the root row
 *   if none); bonus = g[last_pos]; path = its ancestors' node ids from depth 1
 *   down, -1 padded, truncated at path_stride.
 * A parent outside [-1, i) or more than WF_MAX_SEQ_NODES nodes sets
 * WF_ERR_BAD_DATA (info = b) and writes -1 to that sequence's outputs.
 */
WF_API wf_status wf_verify_tree(const int32_t* g, const int32_t* tok, const int32_t* parent,
                         const int32_t* node_off, const int32_t* pos_off, int B, int path_stride,
                         int32_t* n_accept, int32_t* bonus, int32_t* last_pos, int32_t* path,
                         void* ws, size_t ws_bytes, wf_stream_t stream);

/*
 * Rows kept after a round (paper Sec. 3.2: decoding continues from the last
 * accepted token, so the committed positions - the root and the accepted
 * path - keep their target states and every other drafted row is dropped):
 *   acc_rows[b*(path_stride+1) + 0] = pos_off[b]                      (root)
 *   acc_rows[b*(path_stride+1) + j] = pos_off[b] + 1 + path[b*path_stride + j-1], j = 1..n_accept[b]
 *   acc_rows[...]                   = -1 after that
 *   acc_off[0] = 0, acc_off[b+1] = acc_off[b] + n_accept[b] + 1      (packed order)
 * and, if hidden_out != NULL, hidden_out[acc_off[b] + j] = hidden[acc_rows[b][j]]
 * (the hidden states the next drafting step conditions on, packed).
 * n_accept, path as returned by wf_verify_* / wf_round with the same
 * path_stride (n_accept[b] <= path_stride; a larger value is taken as
 * path_stride, -1 keeps no row); pos_off [B+1]; all device int32.
 * acc_rows [B, path_stride+1], acc_off [B+1] device int32 out; hidden [*, d],
 * hidden_out [sum(n_accept+1), d] device bf16 bits (both NULL to skip).
 */
WF_API wf_status wf_accepted_rows(const int32_t* n_accept, const int32_t* path, int path_stride,
                                  const int32_t* pos_off, int B, int32_t* acc_rows, int32_t* acc_off,
                                  const uint16_t* hidden, int d, uint16_t* hidden_out, wf_stream_t stream);

/*
 * EAGLE-3 draft-tree construction (the context-aware dynamic tree the
 * autoregressive drafter proposes; paper App. A / Table 7: depth 8, top-k 10,
 * 60 draft tokens).  Step s = 0 .. D-1 expands the frontier: frontier slot j
 * (only slot 0, the root, at s = 0) proposes k children, target ids
 * tid[b][s][j][c] and draft log-probabilities lp[b][s][j][c] <= 0 (e.g. the
 * top-k of wf_draft_topk, shifted by its log-sum-exp).  A child's score is
 * its parent's (0 at the root) plus its lp, summed in fp32.  The k best
 * children of a step (score desc, creation order asc) form the next
 * frontier, best first; the N best of all children created form the tree,
 * listed depth by depth (rank order within a depth), so parent[i] < i.
 *
 * tid device [B, D, k, k] int32, lp device [B, D, k, k] fp32 (entries of
 * unused slots at s = 0 are ignored); 1 <= k <= 16, 1 <= D <= 16,
 * 1 <= N <= k + (D-1) k^2.  Out (device, [B, N]): parent int32 (-1 = root),
 * token int32, score fp32 and depth int32 (score / depth may be NULL).  An lp
 * above 0 or not finite sets WF_ERR_BAD_DATA and writes -1 for that sequence.
 */
WF_API wf_status wf_build_tree(const int32_t* tid, const float* lp, int B, int D, int k, int N, int32_t* parent,
                               int32_t* token, float* score, int32_t* depth, void* ws, size_t ws_bytes,
                               wf_stream_t stream);

/*
 * Neural router and hardware-aware routing decision (paper Sec. 3.3.2; App. A
 * "Neural Router Architecture": h -> Linear(d, m) -> GELU -> dropout ->
 * Linear(m, 1), m = d/8 in the paper; route to the autoregressive drafter iff
 * the predicted gain exceeds tau_neural).  Dropout is the identity at
 * inference; GELU is the exact erf form.
 *
 *   z_j         = b1[j] + sum_k W1[j,k] * hidden[rows[b], k]
 *   delta_al[b] = b2 + sum_j w2[j] * GELU(z_j)
 *   route[b]    = 1 (EAGLE-3, autoregressive) if delta_al[b] > tau, else 0 (DFlash)
 *
 * hidden device [*, d] bf16 bits; rows device [B] int32 (row of each sequence,
 * e.g. last_pos of a verify call); W1 device [m, d] fp32 row-major; b1, w2
 * device [m] fp32; b2, tau host scalars.  d % 8 == 0; 1 <= m <= 65536.
 * Outputs: delta_al device [B] fp32, route device [B] int32 (either may be NULL).
 * fp32 arithmetic; the sum over j is taken in a fixed order (deterministic).
 */
WF_API wf_status wf_router_mlp(const uint16_t* hidden, const int32_t* rows, int B, int d, int m,
                        const float* W1, const float* b1, const float* w2, float b2, float tau,
                        float* delta_al, int32_t* route, void* ws, size_t ws_bytes,
                        wf_stream_t stream);

/*
 * EAGLE-3 draft head with top-k and the draft-to-target id map (Qwen3-4B-EAGLE3
 * card: fixed 32,000-id draft vocabulary, "top-k 10"; the draft vocabulary
 * cannot propose target ids outside it).
 *
 *   logits L[b,v] = sum_k x[b,k] * Wd[v,k], v < Vd
 *   for each b the k largest (logit desc, draft id asc):
 *   draft_ids[b,j] (optional), tids[b,j] = d2t[draft id], vals[b,j] = logit (fp32)
 *   lse[b] = log sum_v exp(L[b,v]) over all Vd draft ids (optional)
 *
 * lse turns the top-k logits into the draft distribution's log-probabilities,
 * vals[b,j] - lse[b], which EAGLE-3 tree construction accumulates along a
 * branch (WhiFlash paper App. A "Drafter Hyperparameters", Table 7: depth 8,
 * top-k 10, 60 draft tokens; see wf_build_tree).
 *
 * x device [B, d] bf16 bits (drafter hidden state); Wd device [Vd, d] bf16 bits;
 * d2t device [Vd] int32 absolute target ids; 1 <= k <= WF_MAX_TOPK, k <= Vd.
 * Outputs device: draft_ids / tids [B, k] int32, vals [B, k] fp32, lse [B]
 * fp32; each may be NULL, not all.  lse is fp32 (per-tile sums of e^(L - max)
 * merged in a fixed order).
 * A d2t entry < 0 sets WF_ERR_BAD_DATA (info = b) and writes -1 for that id.
 */
WF_API wf_status wf_draft_topk(const uint16_t* x, const uint16_t* Wd, const int32_t* d2t, int B, int d,
                        int Vd, int k, int32_t* draft_ids, int32_t* tids, float* vals, float* lse,
                        void* ws, size_t ws_bytes, wf_stream_t stream);

/*
 * Both heads of a round in one weight sweep: the results of wf_lmhead_argmax
 * over the P rows of hidden and of wf_draft_topk over the B rows of x (ids and
 * logits bit for bit; the log-sum-exp to fp32 rounding, its per-tile partials
 * being summed over this sweep's tiles), from one persistent launch that
 * streams Wd and W through the same pipeline (plus a small merge of the draft
 * candidates).  The pages
 * describe the two heads as separate steps (target verification, WhiFlash
 * paper Sec. 3.2; EAGLE-3 drafting, Qwen3-4B-EAGLE3 card); reading both
 * matrices in one pass is this library's scheduling, so that the smaller
 * draft matrix streams at full bandwidth instead of as a second sweep that
 * fills the GPU poorly.  No passage corresponds to the fused call itself.
 *
 * Arguments as in wf_lmhead_argmax (hidden, W, P, d, V, ids, maxlogit) and
 * wf_draft_topk (x, Wd, d2t, B, Vd, k, draft_ids, tids, vals, lse), one shared d.
 * P <= 128 and B <= 128 (one activation tile each), or P > 128 and B <= 256
 * (the paired-CTA sweep of several activation tiles, the draft rows in one
 * tile pair), else WF_ERR_UNSUPPORTED: call the two entry points.
 * Workspace: wf_workspace_bytes(P, B, d, 0, Vd, k).
 */
WF_API wf_status wf_lmhead_draft_topk(const uint16_t* hidden, const uint16_t* W, int P, int d, int V,
                               int32_t* ids, float* maxlogit, const uint16_t* x, const uint16_t* Wd,
                               const int32_t* d2t, int B, int Vd, int k, int32_t* draft_ids,
                               int32_t* tids, float* vals, float* lse, void* ws, size_t ws_bytes,
                               wf_stream_t stream);

/*
 * One whole verify-and-route round (paper Sec. 3.2 - 3.3): LM-head argmax at
 * every verified row -> per-sequence acceptance (chain or tree by kind[b])
 * -> router on each sequence's last accepted row -> route for the next round;
 * plus, if Wd != NULL, the draft head's top-k for every sequence.  All stages
 * are stream-ordered on `stream` with no host synchronisation.  The draft
 * head shares the LM head's weight sweep (as in wf_lmhead_draft_topk) when
 * P <= 128 and B <= 128, or P > 128 and B <= 256.
 */
typedef struct wf_round_args {
    /* verified rows */
    const uint16_t* hidden;    /* [P, d] bf16 bits */
    const uint16_t* W;         /* [V, d] bf16 bits */
    int P, d, V;
    /* sequences */
    int B;
    const int32_t* pos_off;    /* [B+1] */
    const int32_t* node_off;   /* [B+1] */
    const int32_t* kind;       /* [B] 0 = DFlash chain, 1 = EAGLE-3 tree; NULL = all trees */
    const int32_t* tok;        /* [N] drafted target ids */
    const int32_t* parent;     /* [N] tree parents; ignored for chains; NULL only if kind marks all chains */
    int path_stride;           /* columns of path (0 = path not written) */
    /* router */
    int m;
    const float* W1;           /* [m, d] */
    const float* b1;           /* [m] */
    const float* w2;           /* [m] */
    float b2, tau;
    /* draft head (optional: Wd == NULL skips it) */
    const uint16_t* x;         /* [B, d] bf16 bits */
    const uint16_t* Wd;        /* [Vd, d] bf16 bits */
    const int32_t* d2t;        /* [Vd] */
    int Vd, k;
    /* outputs (device) */
    int32_t* ids;              /* [P] target argmax at every row */
    float* maxlogit;           /* [P] or NULL */
    int32_t* n_accept;         /* [B] */
    int32_t* bonus;            /* [B] */
    int32_t* last_pos;         /* [B] */
    int32_t* path;             /* [B, path_stride] or NULL */
    float* delta_al;           /* [B] */
    int32_t* route;            /* [B] */
    int32_t* draft_ids;        /* [B, k] or NULL */
    int32_t* tids;             /* [B, k] (needed if Wd != NULL) */
    float* vals;               /* [B, k] or NULL */
    /* routing policy: WF_ROUTER_NEURAL (the MLP above) or WF_ROUTER_ENTROPY
     * (WhiFlash-Entropy: route = H > tau on the target's next-token
     * distribution at the last accepted row; delta_al then receives H and
     * W1 / b1 / w2 / m are not read).  The entropy policy needs P <= 128 or
     * B <= 256. */
    int router_kind;
    float* lse;                /* [B] draft head's log-sum-exp (as in wf_draft_topk) or NULL */
} wf_round_args;

#define WF_ROUTER_NEURAL 0
#define WF_ROUTER_ENTROPY 1

WF_API wf_status wf_round(const wf_round_args* args, void* ws, size_t ws_bytes, wf_stream_t stream);

/*
 * KV-only catch-up of the autoregressive drafter (paper Sec. 3.4, "Lazy
 * Catch-up" and "KV-only Prefill"): after a switch to the EAGLE-3 drafter,
 * the tokens accepted while it was idle (its backlog) enter its KV cache in
 * one batch.  For every backlog token only the keys and values of the
 * drafter's attention layer are computed; only the final backlog token runs
 * through the attention sublayer in full, so that its state can feed the
 * next draft round.  The drafter is one Llama-style decoder layer (EAGLE3
 * card, "Technical Specifications": hidden 2560, 32 attention heads, 8 KV
 * heads; head size D = 2560 / 32 = 80).  Per backlog token j of sequence b,
 * at position pos = cache_len[b] + j:
 *   a      = u / sqrt(mean(u^2) + eps) * gamma                 (RMSNorm)
 *   Kc[b, pos] = rope(Wk a, pos),  Vc[b, pos] = Wv a            (bf16)
 * rope turns each pair (x[i], x[i + D/2]) of a head by pos * theta^(-2i/D).
 * For the final token f of each sequence (wf_catchup only):
 *   q      = rope(Wq a_f, pos_f)
 *   attn_h = softmax_t(<q_h, Kc[b, t, g]> / sqrt D) Vc[b, t, g],
 *            t < cache_len[b] + n_b, KV head g = h / (H / G)
 *   out[b] = u_f + Wo attn                                      (residual)
 * The MLP of the final token is the drafter's ordinary decode step and is not
 * part of this call.
 */
typedef struct wf_catchup_args {
    const uint16_t* u;         /* [N, din] bf16: the backlog tokens' layer inputs, sequences packed */
    const int32_t* bl_off;     /* [B+1] backlog offsets: bl_off[0] = 0, bl_off[B] = N, n_b >= 1 */
    const int32_t* cache_len;  /* [B] entries already in each sequence's caches */
    int B, N, din;             /* din % 8 == 0, 8 <= din <= 16384 */
    int H, G, D;               /* query heads, KV heads (H % G == 0, H / G <= 16), head size (D % 16 == 0, <= 128) */
    const uint16_t* gamma;     /* [din] bf16 RMSNorm gain */
    float eps, theta;          /* RMSNorm epsilon (>= 0), rotary base (> 0) */
    const uint16_t* Wq;        /* [H*D, din] bf16 (out x in) */
    const uint16_t* Wk;        /* [G*D, din] bf16 */
    const uint16_t* Wv;        /* [G*D, din] bf16 */
    const uint16_t* Wo;        /* [din, H*D] bf16 */
    uint16_t* Kc;              /* [B, cap, G*D] bf16 key cache (rotated keys), in/out */
    uint16_t* Vc;              /* [B, cap, G*D] bf16 value cache, in/out */
    int cap;                   /* cache rows per sequence; B * cap < 2^31 - 4096 */
    float* out;                /* [B, din] fp32 out (wf_catchup) */
    float* attn;               /* [B, H*D] fp32 out or NULL: the final token's attention output */
} wf_catchup_args;

/* Workspace (bytes) for wf_catchup / wf_catchup_kv with these shapes. */
WF_API size_t wf_catchup_workspace_bytes(int B, int N, int din, int H, int G, int D);

/*
 * The KV-only part alone: writes cache rows cache_len[b] .. cache_len[b] + n_b - 1
 * of every sequence and nothing else (Wq, Wo, out, attn unused).  A sequence
 * with no backlog or a backlog past `cap` sets WF_ERR_BAD_DATA (info = b)
 * and its rows past the cache are not written.
 */
WF_API wf_status wf_catchup_kv(const wf_catchup_args* args, void* ws, size_t ws_bytes, wf_stream_t stream);

/* The whole catch-up: wf_catchup_kv, then the final token's attention sublayer. */
WF_API wf_status wf_catchup(const wf_catchup_args* args, void* ws, size_t ws_bytes, wf_stream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* WF_H */
