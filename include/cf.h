/*
 * cf.h — C ABI of libcf: one co-batched transformer layer step on one GB300.
 *
 * The method (ConfluxServe: Reconciling Resource Utilization and Parallelism
 * Efficiency across Prefill and Decode in LLM Serving, §4 and Fig. 7): the
 * tokens of a prefill chunk and the single tokens of many decode requests are
 * stacked into one matrix [prefill rows; decode rows] so that every dense
 * projection (fused QKV, O-proj, SwiGLU FFN) reads its weights once for both
 * phases; attention then forks into decode attention over each request's own
 * paged KV and causal chunked-prefill attention over the chunk's cached
 * prefix, the two running concurrently on disjoint SM partitions (§6.1,
 * "Coordinated attention overlap"), and the paths rejoin before O-proj.
 *
 * Conventions shared by every call
 * --------------------------------
 * - All tensors are DEVICE memory owned by the caller; they must stay valid
 *   until the work queued on the given stream has finished.  Weights must
 *   outlive the engine.  The engine owns only its workspace.
 * - bf16 means IEEE bfloat16 stored as uint16; row-major unless stated.
 * - Paged KV pool (one for K, one for V): bf16 [num_pages][Hkv][page_size][d].
 *   Each (page, kv head) is one contiguous page_size x d tile.  The slot of
 *   token position p of a request with page table pt is
 *   pt[p / page_size] * page_size + p % page_size (ConfluxServe §7: paged
 *   blocks addressed through per-request block tables).
 * - `stream` is a cudaStream_t passed as void*; NULL means the legacy default
 *   stream.  Every call is asynchronous on it.
 * - Argument and shape checks are synchronous: a failing call returns a
 *   status and launches nothing.  Problems only the device can see (a page id
 *   outside the pool, a context longer than its page table, a bounded wait
 *   that expired) set the engine's device error word; the kernels skip the
 *   offending access instead of trapping.  cf_get_error() reports and clears
 *   it.  No call traps or aborts.
 * - An engine is not thread-safe.
 */
#ifndef CF_H
#define CF_H

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    CF_OK = 0,
    CF_ERR_INVALID_ARG = 1,   /* bad pointer, size or shape; nothing launched   */
    CF_ERR_UNSUPPORTED = 2,   /* valid but not implemented (e.g. head_dim 96)    */
    CF_ERR_CUDA = 3,          /* a CUDA runtime/driver call failed               */
    CF_ERR_TIMEOUT = 4,       /* a device-side bounded wait expired              */
    CF_ERR_OOM = 5,           /* workspace allocation failed in cf_create        */
    CF_ERR_DEVICE = 6         /* device error word set (bad page id, ...)        */
} cf_status;

/* Device error word bits (cf_get_error). */
#define CF_DEVERR_PAGE     0x1   /* a page id outside [0, num_pages) was skipped */
#define CF_DEVERR_CONTEXT  0x2   /* a context needs more pages than its table has */
#define CF_DEVERR_TIMEOUT  0x4   /* a bounded mbarrier wait gave up              */
#define CF_DEVERR_INTERNAL 0x8   /* a kernel refused to run (e.g. misaligned shared memory) */

typedef struct cf_engine cf_engine;

/* Layer shape and engine limits. */
typedef struct {
    int hidden;          /* H                                                    */
    int n_q_heads;       /* Hq                                                   */
    int n_kv_heads;      /* Hkv; Hq % Hkv == 0, G = Hq / Hkv <= 16               */
    int head_dim;        /* d: 64 or 128                                         */
    int ffn_dim;         /* F (SwiGLU width); multiple of 128                    */
    int page_size;       /* tokens per KV page: 16                               */
    float rope_theta;    /* RoPE base                                            */
    float rms_eps;       /* RMSNorm epsilon (also used by QK-norm)               */
    int qk_norm;         /* 1: per-head RMSNorm of q and k over d before RoPE    */
    int max_tokens;      /* largest T = l + n_decode of any step                 */
    int max_decode;      /* largest n_decode of any step (<= 2048)               */
    int decode_sms;      /* SMs given to decode attention in the fork; 0 = auto:
                            the ConfluxServe §6.1 rule, measured per decode-batch
                            bucket (see cf_calibrate_decode_sms)                 */
} cf_config;

/* Weights, nn.Linear layout [out_features][in_features], bf16, device. */
typedef struct {
    const void* w_qkv;   /* [(Hq + 2 Hkv) d][H]: Q heads, then K heads, then V
                            heads (Decode Token Parallelism §4.4, Eq. 1)         */
    const void* w_o;     /* [H][Hq d]                                            */
    const void* w_gate;  /* [F][H]                                               */
    const void* w_up;    /* [F][H]                                               */
    const void* w_down;  /* [H][F]                                               */
    const void* g_attn;  /* [H] RMSNorm gain before QKV                          */
    const void* g_ffn;   /* [H] RMSNorm gain before the FFN                      */
    const void* g_q;     /* [d] QK-norm gain of q (NULL unless qk_norm)          */
    const void* g_k;     /* [d] QK-norm gain of k (NULL unless qk_norm)          */
} cf_weights;

typedef struct {
    void* k;             /* bf16 [num_pages][Hkv][page_size][d]                  */
    void* v;             /* bf16 [num_pages][Hkv][page_size][d]                  */
    int num_pages;
} cf_kv_pool;

/* One iteration's batch: prefill chunks and n_decode resident decodes
 * (ConfluxServe §6.2: the scheduled prefill batch P, chunk l_i of a request
 * with processed context c_i; decode requests with context c_i).  Rows of x
 * are [chunk rows; n_decode decode rows], the chunks one after another.
 * One chunk can be given in prefill_len / prefill_prefix / pre_pages; any
 * number up to 32 in the n_chunks arrays (then prefill_len must be 0).
 * Fields a caller leaves zero mean "none". */
typedef struct {
    int n_decode;
    const int* dec_ctx;    /* device int32 [n_decode]: c_j, tokens cached before
                              this step; the new token sits at position c_j and
                              attends to c_j + 1 keys                           */
    const int* dec_pages;  /* device int32 [n_decode][dec_stride] page ids;
                              needs ceil((c_j + 1) / page_size) valid entries   */
    int dec_stride;
    int prefill_len;       /* l, 0 = no chunk                                   */
    int prefill_prefix;    /* c_p: chunk token i sits at position c_p + i       */
    const int* pre_pages;  /* device int32 [ceil((c_p + l) / page_size)]       */
    int n_chunks;          /* 0: the chunk above (or none); 1..32: these chunks */
    const int* chunk_len;  /* HOST int32 [n_chunks]: l_i >= 1                   */
    const int* chunk_prefix; /* HOST int32 [n_chunks]: c_i >= 0; row r of chunk
                              i sits at position c_i + r of its own request     */
    const int* chunk_pages;  /* device int32 [n_chunks][chunk_stride]: chunk i's
                              page table, ceil((c_i + l_i) / page_size) valid
                              entries (chunk_stride or fewer)                   */
    int chunk_stride;
} cf_batch;

/* Piecewise CUDA graphs (ConfluxServe §6.1, Fig. 10), off by default.  When
 * on, cf_layer_step captures its two shared linear segments (RMSNorm + fused
 * QKV; O-proj + RMSNorm + gate/up + down) as CUDA graphs on first use and
 * replays them, while the attention fork between them is launched eagerly.
 * The graphs depend on T and on the buffers (x_in, x_out, pool, page tables):
 * a batch with the same T and buffers but another split into chunk and
 * decode rows, other prefix or other context lengths reuses them (the chunk
 * length and prefix reach the captured kernels through device memory).  Up
 * to 16 keys are cached; steps with profiling on run eagerly.  Outputs are
 * the same bits as eager steps. */
cf_status cf_set_graphs(cf_engine* e, int enable);
/* Number of graph pairs this engine has captured so far. */
long long cf_graph_captures(cf_engine* e);

/* The work plan of one decode launch (host only; needs no GPU), as the
 * decode kernels compute it on the device from the key counts n_keys[j]
 * (page table width page_stride pages) for a plan sized to plan_ctas CTAs:
 * each request's pages are cut into chunks of *chunk pages, one work item
 * per (request, KV head, chunk); *items is their count and *max_items the
 * bound the engine's partial-output workspace is sized for (n decodes on
 * plan_ctas CTAs).  Any output may be NULL. */
cf_status cf_decode_plan(int n, const int* n_keys, int page_stride, int n_kv_heads, int plan_ctas, int* chunk,
                         int* items, long long* max_items);

/* The work plan of one prefill launch (host only; needs no GPU), as the
 * layer step and cf_prefill_attn_varlen make it for n chunks (len[i],
 * prefix[i]) given in stacked-row order on `sms` SMs.  *kind: the work unit,
 * 0 single 128-row query tiles, 1 pairs of consecutive query tiles of one
 * head, 2 pairs of query heads of one KV head on one query tile (used when
 * Hq / Hkv is even); pairing_mode 0 chooses it as the engine does, 1..3 force
 * kind 0..2.  splits[i]: the key ranges each cut unit of chunk i is cut into
 * (1: none cut; see cf_set_prefill_split for split_mode); cut_from[i]: the
 * chunk's units in queue order before this index run whole, the rest are cut
 * (units_i when none is, 0 when all are); *items: the queue length,
 * sum_i cut_from[i] + (units_i - cut_from[i]) * splits[i].  Any output may be
 * NULL.  Returns CF_ERR_INVALID_ARG for bad sizes, CF_ERR_UNSUPPORTED for head
 * pairs with an odd group. */
cf_status cf_prefill_plan(int n, const int* len, const int* prefix, int n_q_heads, int n_kv_heads, int sms,
                          int split_mode, int pairing_mode, int* kind, int* splits, int* cut_from, int* items);

/* Work items of prefill attention.  Each item runs two 128-row query tiles
 * that share every K/V tile it loads, or one:
 *   1 single tiles;
 *   2 two consecutive query tiles of one head;
 *   3 one query tile of two heads of the same KV head (GQA groups of even
 *     size only; CF_ERR_UNSUPPORTED otherwise);
 *   0 (default) 3 when the group size is even, else 2 when the chunks have
 *     at least one tile pair per SM, else 1.
 * A query tile is computed the same way in every mode (same key order, same
 * products), so outputs are the same bits in every mode. */
cf_status cf_set_prefill_pairing(cf_engine* e, int mode);
/* Key-range cuts of prefill items (flash-decoding style, for items that
 * would otherwise be the critical path of a launch: a short chunk after a
 * long prefix gives few, long items).  A cut item covers a range of key
 * tiles and writes its unnormalised output, running max and sum (fp32) to
 * engine workspace; a merge kernel combines the ranges in order, so results
 * are deterministic.  0 (default): cut a chunk's items into
 * ceil(reach / w) ranges when its longest item reaches more than 1.25 w key
 * tiles, w the launch's average key tiles per SM (at least 8), or into up to
 * 4 when the launch has fewer than 4 units per SM; when neither applies and
 * the units make more than two waves, cut the last wave's worth of units of
 * the queue (one per SM) into 4 ranges of at least 8 key tiles, so that the
 * SMs finish close together; 1 never; n in 2..16 cut every chunk into n
 * ranges where possible.  A chunk is cut into at most as many ranges as its
 * shortest item has key tiles, and cut items use at most 2048 partial query
 * tiles per launch (128 MB at d = 128).  Cut rows agree with uncut ones
 * within fp32 rounding. */
cf_status cf_set_prefill_split(cf_engine* e, int mode);

/* How cf_layer_step runs decode and prefill attention:
 *   0 (default) concurrently, on disjoint SM partitions, each side's SMs
 *     taking over the other side's remaining work items once their own are
 *     done (ConfluxServe §6.1, "Coordinated attention overlap");
 *   1 serially, decode alone on all SMs and then prefill alone on all SMs,
 *     on the caller's stream, with the same kernels and work items: the
 *     serialized execution that §8.3 (Fig. 14a) measures the overlap
 *     against.  Its per-phase times (cf_get_phase_times) give each path's
 *     isolated time ("decode": decode kernel and merge; "prefill": prefill
 *     kernel and merge), whose larger one is the contention-free bound.
 * Outputs are the same bits in both modes: the work items, and the order in
 * which the partials of a cut item are combined, depend neither on the mode
 * nor on the SM share. */
cf_status cf_set_fork_mode(cf_engine* e, int mode);

/* Failure-detection self-test (no counterpart on the pages): launches one
 * 128 x 256 GEMM tile on the engine's own buffers whose MMA-issuing thread
 * first waits on an mbarrier that nothing arrives at.  The wait is bounded
 * by wait_ns (1 ns .. 2 s); when it runs out the kernel sets the timeout bit
 * of the device error word, lets its own TMA copies land, frees its tensor
 * memory and returns, as any kernel here does after an expired wait.  The
 * next cf_get_error reports CF_ERR_TIMEOUT and clears the word;
 * the engine stays usable.  Overwrites workspace Q rows: do not run it
 * during a layer step on another stream. */
cf_status cf_selftest_timeout(cf_engine* e, unsigned long long wait_ns, void* stream);

/* Largest number of SMs the device offers (0 if unknown).  No engine needed. */
int cf_device_sm_count(void);

/* Create an engine on the current device: checks the configuration, keeps
 * the weight pointers, builds TMA descriptors and allocates the workspace
 * (activations for max_tokens rows, split-K partials for max_decode
 * requests), two streams' worth of events and the device error word.
 * Returns CF_ERR_INVALID_ARG / CF_ERR_UNSUPPORTED for a bad configuration,
 * CF_ERR_OOM if the workspace cannot be allocated. */
cf_status cf_create(const cf_config* cfg, const cf_weights* w, cf_engine** out);

/* Frees the workspace (synchronises the engine's streams first). NULL is ok. */
void cf_destroy(cf_engine* e);

/* One co-batched layer step (ConfluxServe Fig. 1, Fig. 7, §6.1):
 *   xn = RMSNorm(x) g_attn; qkv = xn W_qkv^T; [QK-norm]; RoPE at each row's
 *   position; K, V appended to the pool at slot(position) (Decode Token
 *   Parallelism §4.3: rotary embeddings, append, attention);
 *   fork: decode attention (rows l..T-1) on a second stream with decode_sms
 *   SMs || causal prefill attention (rows 0..l-1) on `stream` with the rest;
 *   each path's SMs take over the other path's remaining work items once
 *   their own path is done; join; h = x + O W_o^T (fp32); hn = RMSNorm(h) g_ffn;
 *   x_out = h + (silu(hn W_gate^T) * (hn W_up^T)) W_down^T.
 * x_in, x_out: bf16 [T][H], T = l + n_decode <= max_tokens; they must not
 * overlap.  The pool is modified (T new K/V rows).  The cached slots that
 * the step reads must not be written by other work in flight. */
cf_status cf_layer_step(cf_engine* e, const cf_batch* b, const void* x_in, void* x_out,
                        const cf_kv_pool* pool, void* stream);

/* Split-K decode attention (ConfluxServe App. B, Table 7, "Decode
 * Attention"; partial results merged with fp32 log-sum-exp as in Decode
 * Token Parallelism §4.4, Eq. 4).  For request j and query head h:
 *   out[j][h] = softmax(q[j][h] . K_j^T / sqrt(d)) V_j over the n_keys[j]
 *   keys at positions 0..n_keys[j]-1 of the request, KV head h / G.
 * q: bf16, row j at q + j * q_row_stride (elements), [Hq][d] inside the row.
 * n_keys: device int32 [n] (>= 1).  pages: device int32 [n][page_stride].
 * out: bf16, row j at out + j * out_row_stride, [Hq][d].
 * num_sms: CTAs of the persistent grid (0 = all SMs).  The keys are cut
 * into chunks planned for the device's full SM count, whatever num_sms is,
 * so the output is bit-identical for every num_sms.
 * Uses the engine's workspace for the partials; n <= max_decode. */
cf_status cf_decode_attn(cf_engine* e, const void* q, long long q_row_stride,
                         const cf_kv_pool* pool, int n, const int* n_keys,
                         const int* pages, int page_stride, void* out,
                         long long out_row_stride, int num_sms, void* stream);

/* Causal chunked-prefill attention over a cached prefix (Adaptive Context
 * Parallelism §2.1 mask M_ij = 0 iff j <= i; §2.2 Eq. 1 workload
 * W(l, c_p) = l c_p + l(l+1)/2).  Chunk query i (position prefix + i) and
 * head h attends to keys 0..prefix+i of the request, whose K/V (prefix and
 * chunk) are already in the pool at the slots of `pages`.
 * q: bf16 [l][Hq][d]; out: bf16 [l][Hq][d]; pages: device int32
 * [ceil((prefix + l) / page_size)].  num_sms as above. */
cf_status cf_prefill_attn(cf_engine* e, const void* q, const cf_kv_pool* pool, int l,
                          int prefix, const int* pages, void* out, int num_sms,
                          void* stream);

/* Several chunks of different requests in one launch (ConfluxServe §6.2
 * Eq. 6: the scheduled prefill batch P), each as in cf_prefill_attn: chunk
 * i's queries are rows [r_i, r_i + l_i) of q and of out, r_i the sum of the
 * earlier chunks' lengths, and attend to their own request's keys
 * 0..c_i + row through chunk i's page table.  chunk_len, chunk_prefix: HOST
 * int32 [n_chunks] (1 <= n_chunks <= 32, l_i >= 1, c_i >= 0); chunk_pages:
 * device int32 [n_chunks][chunk_stride].  The items of all chunks share one
 * work queue.  CF_ERR_INVALID_ARG for a bad length, prefix or stride,
 * CF_ERR_UNSUPPORTED for more than 32 chunks. */
cf_status cf_prefill_attn_varlen(cf_engine* e, const void* q, const cf_kv_pool* pool, int n_chunks,
                                 const int* chunk_len, const int* chunk_prefix, const int* chunk_pages,
                                 int chunk_stride, void* out, int num_sms, void* stream);

/* RMSNorm of T rows of width H (the engine's hidden size): out = x /
 * sqrt(mean(x^2) + eps) * gain, fp32 reduction (the pre-attention and
 * pre-FFN norms of the layer; Decode Token Parallelism §4.3 "residual and
 * normalization").  x: bf16 [T][H] (x_is_f32 = 0) or fp32 [T][H]; gain:
 * bf16 [H]; out: bf16 [T][H]. */
cf_status cf_rmsnorm(cf_engine* e, const void* x, int x_is_f32, const void* gain, void* out, int T,
                     void* stream);

/* The fused QKV stage of the layer on an already normalised input:
 * qkv = xn W_qkv^T on the tensor cores; per head [QK-norm]; RoPE at each
 * row's position (chunk row i: c_p + i; decode row j: c_j); q written to
 * q_out (bf16 [T][Hq][d]); k and v appended to the pool at the slot of the
 * row's position (Decode Token Parallelism §4.3: rotary embeddings, then the
 * append).  xn: bf16 [T][H], T = l + n_decode <= max_tokens. */
cf_status cf_qkv(cf_engine* e, const cf_batch* b, const void* xn, const cf_kv_pool* pool, void* q_out,
                 void* stream);

/* Epilogues of cf_gemm. */
#define CF_EPI_NONE        0  /* C bf16 [M][N] = A B^T                               */
#define CF_EPI_RESID_F32   1  /* C fp32 [M][N] = aux (bf16 [M][N]) + A B^T           */
#define CF_EPI_RESID_BF16  2  /* C bf16 [M][N] = aux (fp32 [M][N]) + A B^T           */
#define CF_EPI_SWIGLU      3  /* C bf16 [M][N] = silu(A B^T) * (A aux^T),
                                 B = gate and aux = up, both bf16 [N][K]          */

/* Dense GEMM on the tcgen05 tensor cores: A bf16 [M][K] (row stride lda
 * elements), B bf16 [N][K] (row stride ldb), fp32 accumulation, epilogue
 * as above (C row stride ldc elements; aux uses ldc for the residual
 * epilogues and ldb for SwiGLU).  K % 64 == 0; N % 256 == 0 (N % 128 == 0
 * for SwiGLU); all strides multiples of 8 and pointers 16-byte aligned.  The
 * co-batched rows of A are independent: any row of C equals the same row
 * computed alone (ConfluxServe §4: co-batching needs only a shared weight
 * matrix and feature dimension). */
cf_status cf_gemm(cf_engine* e, const void* A, int lda, const void* B, int ldb,
                  void* C, int ldc, int M, int N, int K, int epilogue,
                  const void* aux, void* stream);

/* Work split of a GEMM over `ctas` persistent CTAs, as cf_gemm and the
 * layer step's GEMMs use it (host only; needs no GPU).  Tiles are 128 x 256
 * outputs (128 x 128 of the result for SwiGLU), numbered m-fastest; K is cut
 * into 64-wide k-blocks.  Tiles [0, *dp_tiles) fill whole waves, one tile
 * per CTA per wave.  The *tiles - *dp_tiles tiles of a partial last wave are
 * each cut into *split equal k-chunks (1: not cut), run one chunk per CTA,
 * so the last wave does not leave SMs idle; a cut tile is summed in k order
 * by the CTA that finishes last, so results are deterministic.  split_mode:
 * 0 chooses the cut from a cost model, 1 never cuts, n >= 2 cuts into n
 * chunks (at most what fits in one wave).  A row's rounding depends on
 * whether its tile was cut, i.e. on M: with split_mode 1 every output row is
 * bit-identical however many other rows share the batch (ConfluxServe §4:
 * co-batched rows are independent).  Returns CF_ERR_INVALID_ARG for
 * non-positive sizes or ctas. */
cf_status cf_gemm_schedule(int M, int N, int K, int epilogue, int ctas, int split_mode, int* grid, int* tiles,
                           int* dp_tiles, int* split);

/* Split-K mode of this engine's GEMMs (see cf_gemm_schedule); default 0.
 * With 1 the GEMM rows of a layer step are bit-identical to the same rows
 * run in any other batch. */
cf_status cf_set_split_k(cf_engine* e, int split_mode);

/* Decode attention that allocates nothing.  The paper has no counterpart:
 * this entry point exists for callers that cannot allocate device memory --
 * a serving runtime whose own pool already holds all free device memory, a
 * plugin inside a framework whose allocator owns the device, or a loop that
 * must never pay for cudaMalloc's device-wide synchronisation -- and so can
 * create no engine.  It computes exactly what cf_decode_attn computes (same
 * kernel, same arguments, shape passed explicitly) but keeps its split-K
 * scratch in a 16 MiB array compiled into the library, which every GPU that
 * loads the library holds until the process exits.
 * - The first call on each device looks up that array's device address
 *   (with that device current); make that first call before any stream
 *   capture.
 * - The keys are cut into chunks planned for the num_sms CTAs the call
 *   launches (0 = all SMs).  With all SMs the output is bit-identical to
 *   cf_decode_attn's; with fewer it differs from it only in fp32 rounding.
 * - Batches whose scratch would exceed 16 MiB are rejected with
 *   CF_ERR_INVALID_ARG.  The need grows with n * Hkv * G * d and with the
 *   CTAs launched, so a batch rejected on all SMs may fit with a smaller
 *   num_sms (e.g. 32 Qwen3-32B-shaped requests need about 22 MB on 152 SMs,
 *   but fit on up to 116).
 * - All calls share the one array, which keeps the last call's contents.
 *   Each call first clears the words that must start at zero (the work-queue
 *   counter, the error word) on its own stream, so it does not depend on how
 *   an earlier call ended; calls that may overlap on the GPU, e.g. on two
 *   streams, race on the array and must be serialised by the caller.
 * - Device-side problems are not reported, since there is no engine error
 *   word: a page id outside the pool is skipped (its keys read as zeros) as
 *   in cf_decode_attn, and a bounded wait that expires ends the kernel with
 *   part of the output unwritten.  Either way the call returns CF_OK.
 * It calls no cudaMalloc, cudaFree or allocating library routine. */
cf_status cf_decode_attn_noalloc(int n_q_heads, int n_kv_heads, int head_dim, int page_size,
                                 const void* q, long long q_row_stride, const cf_kv_pool* pool, int n,
                                 const int* n_keys, const int* pages, int page_stride, void* out,
                                 long long out_row_stride, int num_sms, void* stream);

/* Paged KV append (ConfluxServe §4, Fig. 8: each request extends its own KV
 * cache with its new tokens).  k, v: bf16 [n][Hkv][d]; slots: device int32
 * [n] = page * page_size + offset.  Row r is copied bit for bit to
 * pool.k[slot / ps][:, slot % ps, :] (and v).  Slots outside the pool are
 * skipped and set CF_DEVERR_PAGE in the engine's error word (if e != NULL). */
cf_status cf_kv_append(cf_engine* e, const void* k, const void* v, int n, const int* slots,
                       const cf_kv_pool* pool, int n_kv_heads, int head_dim, int page_size,
                       void* stream);

/* Waits for the engine's streams, reads and clears the device error word.
 * Returns CF_OK, CF_ERR_DEVICE or CF_ERR_TIMEOUT; writes a message to buf. */
cf_status cf_get_error(cf_engine* e, char* buf, int len);

/* Introspection for tests and benchmarks.
 * cf_engine_buffer: device pointer of a workspace tensor of the last step:
 *   "xn" bf16 [T][H], "q" bf16 [T][Hq][d], "attn" bf16 [T][Hq d],
 *   "h" fp32 [T][H], "hn" bf16 [T][H], "act" bf16 [T][F]; NULL otherwise.
 * cf_engine_decode_sms: SMs the fork gives decode attention for n_sms total.
 * cf_set_profiling: 1 = record CUDA events around every phase of each step.
 * cf_get_phase_times: accumulated milliseconds per phase since the last
 *   reset (order: rmsnorm, qkv, decode, prefill, fork, oproj, rmsnorm2,
 *   gateup, down, step, fork_in = fork start to the decode grid's start,
 *   fork_out = the decode grid's end to the join) and the number of steps;
 *   resets the counters.
 * cf_launch_count: kernels this engine launched since creation. */
void* cf_engine_buffer(cf_engine* e, const char* name);
int cf_engine_decode_sms(cf_engine* e);
cf_status cf_set_decode_sms(cf_engine* e, int n);
cf_status cf_set_profiling(cf_engine* e, int on);
/* The decode SM share by the ConfluxServe §6.1 rule: "the minimum number of
 * SMs needed to sustain 90% of its standalone peak HBM bandwidth".  Times the
 * decode attention of batch b (on the Q rows the engine's last cf_layer_step
 * produced, over `pool`) alone on 8, 12, 16, ... and all SMs, each point the
 * median of three launches, picks the smallest count whose time is within
 * 1/frac of the fastest, stores it as the automatic share of b's decode-batch
 * bucket (ceil(log2 n_decode)) and returns it in *chosen.  Synchronous;
 * overwrites the engine's attention buffer.  cf_calibration_points copies
 * the measured (CTAs, ms) pairs (returns how many there are).
 *
 * With decode_sms = 0 (config) and no cf_set_decode_sms override, the first
 * concurrent cf_layer_step of each bucket that has both decodes and prefill
 * rows runs this measurement itself, with frac = 0.9, on its own batch after
 * its QKV stage: that one call blocks the host until the measurement is done
 * (tens of ms) and its phase times include it.  Make it before any stream
 * capture: a step on a capturing stream skips the measurement and uses the
 * bucket's share if known, else a third of the SMs.  The fork is
 * work-conserving (each side's SMs take the other side's remaining items),
 * so the rule sets where the two partitions start, not what each may use.
 * cf_engine_decode_sms reports the share of the last step's bucket. */
cf_status cf_calibrate_decode_sms(cf_engine* e, const cf_batch* b, const cf_kv_pool* pool, float frac,
                                  void* stream, int* chosen);
int cf_calibration_points(cf_engine* e, int* sms, float* ms, int cap);
cf_status cf_get_phase_times(cf_engine* e, float* ms, int n, int* steps);
long long cf_launch_count(cf_engine* e);

/* ---- Iteration-latency estimator --------------------------------------
 * ConfluxServe §6.2 "Latency Modeling and Estimation" (Eq. 2-6) with the
 * base latency functions of App. D (Eq. 7-11).  Host code only: these calls
 * touch no GPU, hold no state and are safe from any thread.  Times come out
 * in the unit the coefficients were fitted in.
 *
 * Per iteration over L layers and N ranks:
 *   T_iter = L (T_GEMM + T_ATTN)                                  (Eq. 2)
 *   T_GEMM = f_GEMM(max_r (n_p^r + n_d^r))                        (Eq. 3)
 *   T_ATTN = max{beta T_P, alpha T_D}                             (Eq. 4)
 *   T_D    = max over ranks holding decodes of f_D(sum_i c_i)     (Eq. 5)
 *   T_P    = f_comm(max_r n_p^r) + f_P((1/N) sum_i W_i)           (Eq. 6)
 *   W_i    = l_i (c_i + (l_i + 1) / 2)                            (Eq. 9)
 * with every f linear (Eq. 7, 8, 10, 11).  A path with no work takes no
 * time (T_D = 0 without decodes, T_P = 0 without chunks, T_GEMM = 0 without
 * tokens); f_comm is added only when N > 1. */
typedef struct {
  double gamma, gamma0;     /* f_GEMM(n) = gamma n + gamma0, n rank-local tokens (Eq. 7) */
  double a_d, a_d0;         /* f_D(W) = a_d W + a_d0, W = sum of decode contexts (Eq. 8) */
  double a_p, a_p0;         /* f_P(W) = a_p W + a_p0, W per-rank chunk workload (Eq. 10) */
  double a_comm, a_comm0;   /* f_comm(n) = a_comm n + a_comm0, n largest shard (Eq. 11)  */
  double alpha, beta;       /* contention factors of the decode / prefill path (Eq. 4)  */
} cf_latency_model;

typedef struct {
  long long n_prefill;      /* n_p^r: prefill tokens assigned to rank r                 */
  long long n_decode;       /* n_d^r: decode requests resident on rank r                */
  double ctx_sum;           /* sum of c_i over rank r's resident decodes                */
} cf_rank_load;

typedef struct {
  double t_iter, t_gemm, t_attn, t_prefill, t_decode;
} cf_latency_parts;

/* Predicts one iteration.  ranks: host [n_ranks]; chunk_len / chunk_ctx:
 * host [n_chunks], the scheduled chunks' l_i and processed context c_i
 * (chunks of length 0 are ignored).  Returns CF_ERR_INVALID_ARG for a null
 * pointer, n_ranks < 1, a negative count or length, or a non-finite
 * coefficient or context sum; *out is then left untouched. */
cf_status cf_latency_predict(const cf_latency_model* m, int n_ranks, const cf_rank_load* ranks, int n_chunks,
                             const long long* chunk_len, const long long* chunk_ctx, int n_layers,
                             cf_latency_parts* out);

/* Ordinary least-squares line y ~ slope x + intercept over n host points
 * (App. D: each base function is fitted from offline profiles).
 * CF_ERR_INVALID_ARG if n < 2, all x are equal or a value is not finite. */
cf_status cf_latency_fit_line(const double* x, const double* y, int n, double* slope, double* intercept);

/* Calibrates the contention factors of Eq. 4 on n co-batched profiles
 * (App. D "Fitting"): for every pair (alpha, beta) on the grid
 * {1, 1 + step, 1 + 2 step, ...} <= f_max, scores the mean absolute
 * percentage error of t_gemm[i] + max(beta t_prefill[i], alpha t_decode[i])
 * against t_meas[i] (the accuracy measure of ConfluxServe §8.4), and keeps
 * the first minimum in (alpha, beta) order.  The inputs are host [n]:
 * the fitted f_GEMM, f_P and f_D of each batch (0 for an absent path) and
 * its measured time.  Writes m->alpha, m->beta and, if mape != NULL, the
 * minimum in percent; the other fields of *m are left as they are.
 * CF_ERR_INVALID_ARG for n < 1, step <= 0, f_max < 1, more than 100001 grid
 * points per factor, a zero measured time or a non-finite value. */
cf_status cf_latency_calibrate(cf_latency_model* m, int n, const double* t_gemm, const double* t_prefill,
                               const double* t_decode, const double* t_meas, double f_max, double step,
                               double* mape);

/* ---- Waterfill prefill dispatch ----------------------------------------
 * ConfluxServe §6.3 "Prefill: waterfill dispatch" and App. E Algorithm 2.
 * Host code only (no GPU, no state).  Given the decode state and the prefill
 * already assigned this iteration, finds the largest combined-load level
 * n_target (a multiple of the alignment quantum q) whose estimated
 * iteration latency (cf_latency_predict) stays within the TBT SLO, the
 * budget B = sum_r max{0, n_target - n_d^r - n_p^r}, and for a request
 * with m_i prefill tokens left the chunk l_i = min{m_i, B} and its per-rank
 * split A_i.
 *
 * Readings of what the pages leave open:
 * - A level n is feasible if the iteration it would run is within the SLO:
 *   with a request, rank r carries n_p^r + A_i^r(n) prefill tokens and the
 *   chunk (l_i(n), c_i) joins the scheduled chunks; without one, every rank
 *   is filled to n by tokens that count for Eq. 3 and f_comm but carry no
 *   attention workload.
 * - Search: level 0 first (if even that is over the SLO, nothing fits:
 *   feasible = 0, B = 0).  With a request the search range ends at the
 *   first level whose budget covers m_i; without one its end is found by
 *   doubling (capped at 2^40 tokens).  Bisection then finds the largest
 *   feasible multiple of q.
 * - Water-filling (cf_waterfill_assign): the tokens raise the lowest loads
 *   first to a common level w <= n_target; tokens left over after the last
 *   whole level go one each to the ranks standing at w, lowest rank index
 *   first. */
typedef struct {
  int n_ranks;
  const long long* n_decode;    /* host [n_ranks]: n_d^r                                 */
  const double* ctx_sum;        /* host [n_ranks]: sum of the resident decodes' c_i      */
  const long long* n_prefill;   /* host [n_ranks]: n_p^r of the existing assignment A_p  */
  int n_chunks;                 /* prefill chunks P already scheduled this iteration     */
  const long long* chunk_len;   /* host [n_chunks]: their l_j                            */
  const long long* chunk_ctx;   /* host [n_chunks]: their processed context c_j          */
} cf_dispatch_state;

typedef struct {
  long long n_target;           /* the level (0 when nothing fits)                       */
  long long budget;             /* B at that level                                       */
  long long chunk;              /* l_i (0 without a request)                             */
  int feasible;                 /* 0: even level 0 exceeds the SLO                       */
  double t_iter;                /* estimated latency of the iteration at n_target        */
} cf_dispatch_result;

/* remaining < 0 asks for the budget only (Algorithm 2 with no request);
 * otherwise remaining = m_i and context = c_i of the request.  assign:
 * host [n_ranks] receives A_i (zeros without a request) or may be NULL.
 * CF_ERR_INVALID_ARG for a null pointer, n_ranks < 1, quantum < 1, a
 * negative count, a NaN SLO or an invalid model (as cf_latency_predict). */
cf_status cf_waterfill_dispatch(const cf_latency_model* m, int n_layers, double tbt_slo, long long quantum,
                                const cf_dispatch_state* s, long long remaining, long long context,
                                cf_dispatch_result* out, long long* assign);

/* WaterfillAssign alone: splits `tokens` over ranks with combined loads
 * loads[n_ranks] toward n_target; give: host [n_ranks].
 * CF_ERR_INVALID_ARG if tokens exceed sum_r max{0, n_target - loads[r]} or a
 * load or tokens is negative. */
cf_status cf_waterfill_assign(const long long* loads, int n_ranks, long long tokens, long long n_target,
                              long long* give);

#ifdef __cplusplus
}
#endif
#endif /* CF_H */
