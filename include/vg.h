/*
 * vg.h — C ABI of the Vegas hot path on one GB300 (sm_103a).
 *
 * Verification-guided sparse self-speculative decoding, as described on the page
 * "Resumo Técnico: Vegas – Decodificação Auto-Especulativa com Atenção Esparsa
 * Guiada por Verificação" (gist.science summary of paper 2602.07223), cited below
 * as "Vegas §<section>".  One iteration has three device steps:
 *
 *   vg_verify_attn        full attention of the gamma+1 verify rows over the KV cache
 *                         (Vegas §2 step 1), which also sums the pre-softmax logits of
 *                         every prefix entry over the chosen rows and all query heads
 *                         (Vegas §2.A formula, §2.B Collect-2-Query, §3 instrumentation);
 *   vg_topk_select        the k prefix entries with the largest summed logit
 *                         (Vegas §2 step 2, the argmax of §2.A);
 *   vg_sparse_draft_attn  one draft step's attention over the selected entries plus the
 *                         draft tokens appended so far, gathered token by token
 *                         (Vegas §2 step 3; §3 sparse execution, page size one).
 *   vg_iteration          verify -> select -> gamma draft steps, in stream order.
 *   vg_iteration_plan_*   the same iteration captured once as a CUDA graph and
 *                         launched step after step.
 *
 * Conventions shared by every call
 *   - All tensor arguments are DEVICE pointers to caller-owned memory, unless a
 *     comment says "host".  The library never allocates, frees or synchronises,
 *     and never keeps a pointer after a call returns (except the plans of
 *     vg_iteration_plan_create, which allocate and keep theirs).
 *   - bf16 is IEEE bfloat16 (uint16 storage); fp32 is IEEE binary32.
 *   - Every call only enqueues work on `stream` (0 = legacy default stream) and
 *     returns.  Arguments are validated on the host before anything is enqueued;
 *     a call that returns an error has enqueued nothing.
 *   - Device-side checks (a prefix length above max_len, an index outside the
 *     allowed range, a bounded wait that ran out) never fault: the kernel skips the
 *     offending item and writes a VG_ERR_* code into *dev_status (if dev_status is
 *     non-NULL; the first error wins, the caller zeroes it).  Results for a sequence
 *     whose inputs failed a device check are unspecified.
 *   - Alignment: every device pointer must be 16-byte aligned (dev_status: 4-byte).
 *   - Workspace: `ws` is caller-owned device scratch of at least
 *     vg_workspace_size(...) bytes, 256-byte aligned.  Its contents need no
 *     initialisation and are garbage after a call.  Calls that share a workspace
 *     must be ordered on one stream.
 *   - Thread safety: calls may be made from several host threads; vg_last_error()
 *     is per thread.
 *
 * KV cache (Vegas §1: one K and one V entry per token, growing with the context)
 *   Token-granular slot pool: K and V are bf16 [capacity_slots][H_kv][d], one slot
 *   per token holding all KV heads contiguously (the "page size of one token" of
 *   Vegas §3).  Sequence b's token i lives in slot seq_offset[b] + i.  The caller
 *   reserves, after each prefix, room for the gamma+1 verify rows.
 *
 * Shapes supported by this build: d in {64, 128}; H_kv in [1, 16]; H_q = G * H_kv
 * with G in [1, 16]; gamma in [0, 15]; G * (gamma+1) <= 64; 1 <= B <= 1024;
 * max_len <= 262144 for vg_topk_select; k >= 1; H_kv * d <= 1024 for
 * vg_sparse_draft_attn (one token's page of K and of V is staged whole).
 */
#ifndef VG_H
#define VG_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef int32_t vg_status;

#define VG_OK 0
#define VG_ERR_INVALID_ARG (-1)        /* null pointer, bad value, misalignment      */
#define VG_ERR_UNSUPPORTED_SHAPE (-2)  /* outside the shapes listed above             */
#define VG_ERR_WORKSPACE (-3)          /* ws NULL or smaller than vg_workspace_size  */
#define VG_ERR_CUDA (-4)               /* a CUDA runtime call failed                 */
#define VG_ERR_DEVICE_TIMEOUT (-5)     /* device: a bounded wait ran out             */
#define VG_ERR_DEVICE_BOUNDS (-6)      /* device: length or index out of range       */

/* Problem dimensions (host struct). */
typedef struct vg_dims {
  int32_t B;       /* sequences in the batch                                          */
  int32_t H_q;     /* query heads                                                     */
  int32_t H_kv;    /* key/value heads; query head h reads KV head h / (H_q/H_kv)      */
  int32_t d;       /* head dimension                                                  */
  int32_t gamma;   /* draft tokens per iteration; verification has gamma+1 rows,     */
                   /* row gamma being the bonus token (Vegas §2.B)                    */
  int32_t max_len; /* host-side upper bound on every prefix length (sizes grids and  */
                   /* the workspace; longer device lengths are reported, not read)   */
  float scale;     /* logit scale; 0 means 1/sqrt(d)                                  */
} vg_dims;

/* The KV cache of one layer (host struct holding device pointers).
 *
 * Two layouts of the same slot pool (one slot = one token's keys of every KV head):
 *   page_table == NULL: sequence b's token i lives in slot seq_offset[b] + i;
 *   page_table != NULL: the vLLM-style block table of Vegas §3 (the draft runs as a
 *     paged attention whose pages are tokens): the pool is cut into pages of page_size
 *     slots (page p = slots p * page_size .. p * page_size + page_size - 1) and token i
 *     of sequence b lives in row i % page_size of page page_table[b][i / page_size].
 *     seq_offset is then unused (may be NULL).  Page entries outside the pool are
 *     reported on the device as VG_ERR_DEVICE_BOUNDS and their tokens skipped.
 *     vg_sparse_draft_attn reads any page_size >= 1; vg_verify_attn and vg_iteration
 *     need page_size 8, 16, 32 or a multiple of 64 (VG_ERR_UNSUPPORTED_SHAPE otherwise).
 *     pages_per_seq (>= 1) is the row stride of page_table; a sequence's prefix plus
 *     its gamma+1 verify rows must fit pages_per_seq * page_size tokens. */
typedef struct vg_kv_cache {
  void* K;                    /* bf16 [capacity_slots][H_kv][d]                       */
  void* V;                    /* bf16 [capacity_slots][H_kv][d]                       */
  const int64_t* seq_offset;  /* device int64 [B]: slot of token 0 of sequence b      */
  int64_t capacity_slots;     /* slots in K and V                                     */
  const int32_t* page_table;  /* device int32 [B][pages_per_seq], or NULL             */
  int32_t page_size;          /* tokens per page (page_table only)                    */
  int32_t pages_per_seq;      /* row stride of page_table (page_table only)          */
} vg_kv_cache;

/*
 * Verification attention with fused logit aggregation (Vegas §2 step 1; §2.A; §2.B; §3).
 *
 * For sequence b with prefix length n_b = prefix_len[b], verify row t in [0, gamma]
 * and query head h (KV head g = h / G):
 *   out[b][t][h] = softmax_j(l_j) . V_j over j in {prefix 0..n_b-1} U {verify rows u <= t},
 *   l_j = scale * q[b][t][h] . K_j   (causal among the verify rows, itself included);
 * and for every prefix entry i < n_b and each enabled mask (row_mask0, row_mask1):
 *   scores[b][i] = sum over rows t with bit t set, over all H_q heads, of
 *                  scale * q[b][t][h] . K[seq_offset[b] + i][h / G]
 * i.e. the objective of the Vegas §2.A selection formula, before any softmax.  The
 * verify rows' own keys are not scored (T is a subset of the prefix P).
 *
 *   q        bf16 [B][gamma+1][H_q][d]
 *   k_new    bf16 [B][gamma+1][H_kv][d] — the verify rows' keys and values.  They are
 *   v_new        appended to the cache at slots seq_offset[b] + n_b + t.  Pass both
 *                NULL when those slots already hold them.
 *   prefix_len  device int32 [B], each in [0, max_len]
 *   row_mask0/1 bit t selects verify row t; 0 disables that output.  Collect-2-Query
 *               is (1 | 1 << gamma); all rows is (1 << (gamma+1)) - 1.
 *   scores0/1   fp32 [B][score_stride] (score_stride >= max_len); NULL iff its mask is 0.
 *               Entries at positions >= n_b are left untouched.
 *   out      bf16 [B][gamma+1][H_q][d]
 */
vg_status vg_verify_attn(const vg_dims* dims, const vg_kv_cache* cache, const void* q,
                         const void* k_new, const void* v_new, const int32_t* prefix_len,
                         uint32_t row_mask0, uint32_t row_mask1, float* scores0, float* scores1,
                         int64_t score_stride, void* out, void* ws, size_t ws_bytes,
                         int32_t* dev_status, void* stream);

/*
 * Per-sequence top-k of the aggregated scores (Vegas §2 step 2, the argmax of §2.A).
 *
 * T_b = the k positions i < len[b] with the largest scores[b][i]; equal scores
 * prefer the lower position; -0.0 equals +0.0 (NaN scores: unspecified order).
 *   idx[b][0..count_b) = T_b in ascending order, count_b = min(k, len[b]);
 *   idx[b][count_b..k) = -1;  count[b] = count_b.
 *
 *   scores  fp32 [B][score_stride];  len  device int32 [B], each in [0, max_len]
 *   idx     int32 [B][k];            count  int32 [B]
 * Uses no workspace (ws may be NULL).
 */
vg_status vg_topk_select(const float* scores, int64_t score_stride, const int32_t* len, int32_t B,
                         int32_t max_len, int32_t k, int32_t* idx, int32_t* count, void* ws,
                         size_t ws_bytes, int32_t* dev_status, void* stream);

/*
 * Sliding-window selection: the query-agnostic comparison policy of Vegas §1 (simple
 * query-agnostic methods such as sliding windows select cheaply but draft poorly).
 * No counterpart in the Vegas method itself; it gives drafts a baseline selection in
 * the same form as vg_topk_select, whose overlap with the verification-guided one can
 * be measured.
 *
 *   T_b = the last min(k, len[b]) prefix positions, len[b] - count_b .. len[b] - 1,
 *   idx[b][0..count_b) = T_b ascending, idx[b][count_b..k) = -1, count[b] = count_b.
 *
 *   len  device int32 [B], each in [0, max_len] (others: VG_ERR_DEVICE_BOUNDS, count 0)
 *   idx  int32 [B][k];  count  int32 [B];  1 <= k <= 2^24
 */
vg_status vg_window_select(const int32_t* len, int32_t B, int32_t max_len, int32_t k, int32_t* idx,
                           int32_t* count, int32_t* dev_status, void* stream);

/*
 * One sparse draft step (Vegas §2 step 3; §3 sparse execution with page size one).
 *
 * For sequence b the attended set is
 *   A_b = { idx[b][j] : j < count[b] }  U  { tail_start[b] + u : u < tail_len[b] },
 * positions relative to seq_offset[b].  out[b][h] = softmax over A_b of
 * scale * q[b][h] . K_j, applied to V_j, on KV head h / G.
 * If k_new / v_new (bf16 [B][H_kv][d]) are non-NULL they are the current draft
 * token's key and value: they are appended at slot tail_start[b] + tail_len[b] - 1
 * (tail_len[b] >= 1 is then required) and attended from the inputs directly.
 * tail_len[b] <= 16 (a draft phase appends at most gamma + 1 <= 16 tokens); a longer
 * tail is reported as VG_ERR_DEVICE_BOUNDS.  k_stride <= 2^24.
 * Selected positions must be < tail_start[b]; entries outside [0, tail_start[b]) are
 * skipped and reported as VG_ERR_DEVICE_BOUNDS.
 *
 *   q      bf16 [B][H_q][d]             idx  int32 [B][k_stride], count int32 [B] (<= k_stride)
 *   tail_start, tail_len  device int32 [B]   out  bf16 [B][H_q][d]
 *   flags  0, or VG_DRAFT_SELECTION_SETTLED (below); other bits are VG_ERR_INVALID_ARG.
 */
/* The caller vouches that idx, count, seq_offset, tail_start, tail_len and the cache
 * entries at the selected positions were all written before the kernel that precedes
 * this call in the stream began.  That holds for every draft step of a phase after the
 * first: the selection is made once per verification and the steps in between only
 * append draft tokens (Vegas §2 step 3).  The call then starts gathering the selected
 * entries before its dependency on that preceding kernel resolves, overlapping the
 * end of the previous step; the draft-token tail still waits for it.  Results are
 * unspecified if the promise does not hold. */
#define VG_DRAFT_SELECTION_SETTLED 1u

vg_status vg_sparse_draft_attn(const vg_dims* dims, const vg_kv_cache* cache, const void* q,
                               const void* k_new, const void* v_new, const int32_t* idx,
                               const int32_t* count, int32_t k_stride, const int32_t* tail_start,
                               const int32_t* tail_len, uint32_t flags, void* out, void* ws,
                               size_t ws_bytes, int32_t* dev_status, void* stream);

/* Inputs of one iteration (host struct of device pointers). */
typedef struct vg_iter_inputs {
  const void* q_verify;        /* bf16 [B][gamma+1][H_q][d]                              */
  const void* k_verify;        /* bf16 [B][gamma+1][H_kv][d], appended at n_b + t         */
  const void* v_verify;
  const void* q_draft;         /* bf16 [gamma][B][H_q][d]                                */
  const void* k_draft;         /* bf16 [gamma][B][H_kv][d]; step s appended at n_b + s    */
  const void* v_draft;
  const int32_t* prefix_len;   /* device int32 [B]                                       */
} vg_iter_inputs;

/* Outputs of one iteration (host struct of device pointers). */
typedef struct vg_iter_outputs {
  void* out_verify;            /* bf16 [B][gamma+1][H_q][d]                              */
  float* scores0;              /* fp32 [B][score_stride], rows of row_mask0 (selection)   */
  float* scores1;              /* fp32 [B][score_stride] or NULL (row_mask1 == 0)         */
  int64_t score_stride;
  int32_t* idx;                /* int32 [B][k]: selection on scores0                      */
  int32_t* count;              /* int32 [B]                                              */
  int32_t* idx1;               /* int32 [B][k] selection on scores1, or NULL              */
  int32_t* count1;             /* int32 [B], or NULL                                     */
  void* out_draft;             /* bf16 [gamma][B][H_q][d]                                */
} vg_iter_outputs;

/*
 * One Vegas round (Vegas §2 steps 1-3), enqueued in order on `stream`:
 *   vg_verify_attn (appends k_verify/v_verify) -> vg_topk_select on scores0
 *   (and on scores1 if idx1 != NULL) -> for s = 0..gamma-1: vg_sparse_draft_attn
 *   with q_draft[s], appending k_draft[s] at slot n_b + s and attending
 *   T_b U {n_b .. n_b + s} (the draft tokens so far, the current one included).
 * Draft tokens reuse the verify rows' slots.  k >= 1.
 */
vg_status vg_iteration(const vg_dims* dims, const vg_kv_cache* cache, const vg_iter_inputs* in,
                       int32_t k, uint32_t row_mask0, uint32_t row_mask1, vg_iter_outputs* out,
                       void* ws, size_t ws_bytes, int32_t* dev_status, void* stream);

/*
 * vg_iteration (Vegas §2 steps 1-3), captured once and launched many times.  This
 * has no counterpart in the paper, which runs inside a serving framework's loop.  A
 * decode loop calls the same iteration with the same buffers step after step;
 * launching its ~3 + 2*gamma kernels one by one costs the GPU a fraction of a
 * microsecond each.  A plan records the launch sequence of one argument set as a CUDA
 * graph, and each launch replays it in a single call, with the same results as
 * vg_iteration on the buffers' contents at launch time.
 *
 * vg_iteration_plan_create: same arguments and validation as vg_iteration (returns
 *   the same codes, enqueues nothing, writes *plan = NULL on error) plus
 *   plan (out): receives an opaque handle owned by the caller.
 *   The plan keeps every pointer it was given, and the values of *dims, *cache, *in
 *   and *out at creation: each launch reads and writes those same buffers, which
 *   must stay allocated, at the same addresses, until vg_iteration_plan_destroy.
 *   Put new inputs in those buffers between launches.  Unlike every other call,
 *   creating a plan allocates: host memory and the CUDA graph's resources
 *   (VG_ERR_CUDA if the CUDA runtime refuses).  Do not call it while this
 *   thread is capturing a stream.  The plan belongs to the current device.
 * vg_iteration_plan_launch: enqueues one iteration on `stream`, in stream order
 *   with the work before and after it.  VG_ERR_INVALID_ARG for a NULL plan or a
 *   current device other than the plan's; VG_ERR_CUDA if the launch fails.  Launches
 *   of one plan on different streams race on its buffers: order them.
 * vg_iteration_plan_destroy: frees the plan (NULL is a no-op).  Launches already
 *   enqueued still complete.
 */
typedef struct vg_iteration_plan vg_iteration_plan;
vg_status vg_iteration_plan_create(const vg_dims* dims, const vg_kv_cache* cache, const vg_iter_inputs* in,
                                   int32_t k, uint32_t row_mask0, uint32_t row_mask1,
                                   const vg_iter_outputs* out, void* ws, size_t ws_bytes,
                                   int32_t* dev_status, vg_iteration_plan** plan);
vg_status vg_iteration_plan_launch(const vg_iteration_plan* plan, void* stream);
vg_status vg_iteration_plan_destroy(vg_iteration_plan* plan);

/*
 * vg_sparse_draft_attn without a workspace argument.  This entry point has no
 * counterpart in the paper; it exists for callers that cannot hand the library
 * device memory, for example a host that must not call cudaMalloc during decoding
 * (the call can synchronise the device and stall other streams) or that has no
 * workspace to offer.  Same computation, arguments and results as
 * vg_sparse_draft_attn with flags 0; the scratch space comes from an 8 MiB area
 * inside the library that every GPU using the library keeps until the process exits.
 *   - It allocates and frees nothing.
 *   - Dimensions whose draft scratch exceeds 8 MiB are rejected with
 *     VG_ERR_WORKSPACE (for 152 SMs: about H_q * (152 + B) * (d + 2) * 4 bytes).
 *   - The first call on each device looks up the area's device address and keeps
 *     it for the life of the process; make that first call before any stream
 *     capture, and do not reset a device (cudaDeviceReset) while the library is
 *     loaded, since the kept address would then be stale.
 *   - All calls share the one area, which keeps the last call's contents (nothing
 *     in it needs to start at zero).  Calls that may overlap on the GPU - on
 *     different streams, or from different host threads - race on it; order them.
 */
vg_status vg_sparse_draft_attn_noalloc(const vg_dims* dims, const vg_kv_cache* cache, const void* q,
                                       const void* k_new, const void* v_new, const int32_t* idx,
                                       const int32_t* count, int32_t k_stride, const int32_t* tail_start,
                                       const int32_t* tail_len, void* out, int32_t* dev_status, void* stream);

/*
 * Acceptance of the draft chain (Vegas §2 step 1: the verification pass accepts or
 * rejects the draft tokens; §5: lossless, what is committed follows the target model).
 * The page leaves the rule to standard speculative decoding; this is that rule on
 * given logits.  For sequence b:
 *   p_logits  fp32 [B][gamma+1][V]  row t: the target's logits for the token after t
 *                                     accepted drafts (row gamma: the bonus position)
 *   q_logits  fp32 [B][gamma][V]    the draft's logits of draft token t (sampling only)
 *   draft_tokens  int32 [B][gamma]  in [0, V) (others: rejected, VG_ERR_DEVICE_BOUNDS)
 *   mode VG_ACCEPT_GREEDY: draft t survives while it is the most likely token of row t
 *     (ties: lowest token); the next token is the most likely token of row a.
 *   mode VG_ACCEPT_SAMPLE: draft t survives iff u_accept[b][t] * q_t(x_t) < p_t(x_t), p and
 *     q the softmax of the rows; at the first rejection a the next token is drawn from
 *     max(0, p_a - q_a) (from p_a if that is zero everywhere), after gamma acceptances
 *     from p_gamma.  A draw with weights w takes the smallest v whose running sum of
 *     weights exceeds u_resample[b] times their total.  u values in [0, 1), fp32.
 *   n_accept  int32 [B]: a, the drafts accepted (0 .. gamma);  next_token int32 [B].
 *   advance_len  int32 [B] or NULL: if given, increased by a + 1 (the verified row before
 *     the drafts and the a accepted drafts join the prefix; their keys and values are
 *     already in the cache).
 * Computed in fp32 with fixed summation orders (deterministic).  B <= 1024, gamma <= 15,
 * V <= 2^20; V % 4 == 0 reads the rows with 16-byte loads.  Workspace: at least
 * vg_accept_workspace_size(B, gamma, V) bytes, 256-byte aligned, no initialisation.
 */
#define VG_ACCEPT_GREEDY 0u
#define VG_ACCEPT_SAMPLE 1u
size_t vg_accept_workspace_size(int32_t B, int32_t gamma, int32_t V);
vg_status vg_accept(int32_t B, int32_t gamma, int32_t V, const float* p_logits, const float* q_logits,
                    const int32_t* draft_tokens, const float* u_accept, const float* u_resample,
                    uint32_t mode, int32_t* n_accept, int32_t* next_token, int32_t* advance_len,
                    void* ws, size_t ws_bytes, int32_t* dev_status, void* stream);

/* Bytes of workspace any call above needs for these dimensions on the current
 * device (0 on invalid dims or no device; see vg_last_error()). */
size_t vg_workspace_size(const vg_dims* dims, int32_t k);

/* Kernels one vg_sparse_draft_attn call with these dimensions enqueues on the current
 * device: 1 when every sequence's entries fall to a single CTA of the step's grid
 * (that CTA finishes the sequence), else 2 (a second kernel merges the partials).  tail_len_max is the
 * longest tail the call may attend, 0 for the bound of a device tail_len array (16).
 * Returns 0 on invalid arguments or when no device is present (see vg_last_error()).
 * vg_iteration enqueues 3 (verify, its merge, the selection; 4 with a second
 * selection) plus gamma times this number for tail_len_max = 1 .. gamma. */
int32_t vg_sparse_draft_launches(const vg_dims* dims, int32_t k_stride, int32_t tail_len_max);

/* Human-readable description of the last error on this host thread ("" if none). */
const char* vg_last_error(void);

/* Library version, as major * 10000 + minor * 100 + patch. */
int32_t vg_version(void);

/* Self-test of the device-side failure path (no part of the method): launches one
 * CTA of two warps on `stream`; each waits on an mbarrier that nothing arrives on.
 * The first wait gives up after limit_us microseconds (1 .. 1000000), writes
 * VG_ERR_DEVICE_TIMEOUT into *dev_status (if it holds 0) and raises the CTA's abort
 * flag, on which the second wait (whose own limit is the library's 2 s) gives up at
 * once.  *elapsed_ns (device memory, may be NULL) receives the time from the start
 * of the waits to the end of both, so a caller can check that neither a lost wait
 * nor its abort leaves a kernel running.  No copy or tensor-core operation is
 * involved.  Returns VG_ERR_INVALID_ARG for a limit out of range or a NULL or
 * misaligned dev_status / elapsed_ns, VG_ERR_CUDA if the launch fails. */
vg_status vg_selftest_lost_wait(uint32_t limit_us, int32_t* dev_status, uint64_t* elapsed_ns, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* VG_H */
