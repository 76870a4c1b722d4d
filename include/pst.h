/*
 * pst.h -- C ABI of libpst: decode-phase attention over a prefix-shared,
 * tree-structured, paged KV cache on one GPU (sm_103a).
 *
 * Method: CoDec: Prefix-Shared Decoding Kernel for LLMs (papercache.org,
 * 2026-06): the KV cache is a forest of nodes (a virtual root joins unrelated
 * prefixes, "KV cache management"); each node's K/V is read from HBM once for
 * all the queries that share it (KV-guided grouping, DEFT section 3.3); a
 * partial attention computation (PAC) per node chunk emits a partial output
 * with its log-sum-exp, and the partial output reduction (POR) merges them per
 * query ("intra-block primitives", "inter-block launch and tree reduction");
 * a cost-model partitioner splits long nodes along the KV axis ("workload
 * balancing").
 *
 * Conventions for every call:
 *   - Return value 0 (PST_OK) on success, a negative PST_E* code on failure.
 *     No exception crosses the ABI. pst_last_error() gives a message for the
 *     last failure on the calling thread.
 *   - Host arrays passed in are read during the call only (copied); the caller
 *     keeps ownership.
 *   - Device buffers (Q, pools, O, LSE, workspace) are owned by the caller.
 *   - A `stream` argument is a cudaStream_t passed as void* (NULL = legacy
 *     default stream). Device work is asynchronous on that stream; no call
 *     synchronises the host unless it says so.
 */
#ifndef PST_H
#define PST_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---------------------------------------------------------------- errors */
#define PST_OK            0
#define PST_EINVAL       -1   /* malformed argument (null, negative size, query sees no token) */
#define PST_ECYCLE       -2   /* parent array has a cycle */
#define PST_ERANGE       -3   /* parent / page id / offset out of range */
#define PST_EUNSUPPORTED -4   /* shape the kernels do not cover (d, page size, Hq % Hkv) */
#define PST_EWORKSPACE   -5   /* workspace missing, too small or misaligned */
#define PST_ECUDA        -6   /* a CUDA runtime call failed (message has the CUDA error) */
#define PST_EDEVICE      -7   /* a kernel reported a fault in the device status word */
#define PST_ENOMEM       -8   /* host allocation failed */

typedef struct pst_tree pst_tree;
typedef struct pst_plan pst_plan;
typedef struct pst_timer pst_timer;

typedef enum { PST_BF16 = 0, PST_F32 = 1 } pst_dtype;

/* Split policies of the partitioner (CoDec "workload balancing"). */
typedef enum {
    PST_SPLIT_COST_MODEL = 0, /* binary search on the max-block cost + greedy b_k  */
    PST_SPLIT_NONE       = 1, /* b_k = 1: one chunk per node (DEFT-Node)            */
    PST_SPLIT_UNIFORM    = 2, /* every node cut into chunks of `fixed_chunk` tokens */
    PST_SPLIT_FLATTEN    = 3  /* DEFT-Flatten (DEFT A.9): the tokens of every node a
                                 query sees, in depth-first order, cut into chunks
                                 of at most `fixed_chunk` (1..64, default 64)
                                 tokens that cross node boundaries; a chunk also
                                 ends where its tokens stop being consecutive page
                                 rows. Each chunk is one task with the union of its
                                 nodes' queries and a 64-bit bit causal mask per
                                 query (bit j: chunk token j is on its path).    */
} pst_split_policy;

typedef struct {
    int32_t split_policy;   /* pst_split_policy; default PST_SPLIT_COST_MODEL          */
    int32_t fixed_chunk;    /* tokens per chunk for PST_SPLIT_UNIFORM (multiple of 64);
                               at most this many per chunk for PST_SPLIT_FLATTEN    */
    int32_t tc_min_rows;    /* rows (queries x GQA group) from which a node runs on the
                               tensor-core PAC; default 16; fp32 inputs never do      */
    int32_t pack_masks;     /* 1 (default): pack a page-contiguous subtree of <= 64
                               tokens into one chunk with a 64-bit causal mask per
                               query (DEFT bit causal mask); 0: one chunk per node  */
    int32_t num_sms;        /* 0: ask the current device                              */
    int32_t slots_per_sm;   /* concurrent PAC thread blocks per SM assumed by the
                               list schedule; 0: default (1)                         */
    int32_t tc_engine;      /* tensor-core PAC: 0 (default) tcgen05 + tensor memory,
                               1 legacy mma.sync (kept for comparison)               */
    int32_t tc_block_rows;  /* tcgen05 PAC rows per thread block: 256 (default; two
                               128-row halves share each K/V tile) or 128            */
    int32_t p_bf16_min_tokens; /* tcgen05 PAC: chunks of nodes of at least this many
                               tokens multiply V by the softmax weights P rounded
                               once to bf16; chunks of shorter nodes (and packed
                               draft subtrees) split P into bf16 hi + lo parts,
                               which keeps P V as accurate as an fp32 product.
                               0: default (1024); -1: always split               */
    int32_t thin_engine;    /* chunks below tc_min_rows rows ("thin" chunks): 0
                               (default) the tcgen05 thin PAC, tokens on the MMA's
                               M side and query rows (at most 16 per block) on N;
                               bf16 with d = 128 only, other shapes take the
                               CUDA-core PAC; 1 the CUDA-core PAC always         */
    int32_t debug_stall;    /* test only; 0 (default) off. 1: the tcgen05 PAC's MMA
                               thread first waits on a barrier nothing arrives on,
                               so that bounded wait runs out; every role of the
                               block then leaves through its error path (bounded
                               waits, TMA loads drained) and the device status word
                               is set. The outputs of such a call are undefined;
                               pst_plan_check_status reports PST_EDEVICE.        */
    int32_t side_streams;   /* how the PAC launch groups of one call share the GPU.
                               0 (default): all on the caller's stream, each
                               launch after the first with a programmatic
                               dependency on the one before (it starts once every
                               block of that one has started; POR waits for all
                               on the device). 1: each group on its own stream
                               forked from the caller's and joined before POR.
                               pst_decode_attn_timed always uses 1; the
                               no-allocation entry point runs the groups one
                               after the other with 1.                        */
    int32_t flatten_candidates; /* PST_SPLIT_COST_MODEL only. 0 (default): also
                               score DEFT-Flatten chunkings (PST_SPLIT_FLATTEN)
                               of 1024 and 2048 tokens with the same cost model
                               and keep one whose predicted makespan is at
                               least 3 % below the node partition's (the plan's
                               policy then reads PST_SPLIT_FLATTEN); -1: the
                               node partition only.                           */
} pst_plan_opts;

/* Fill `o` with the defaults above. */
void pst_plan_opts_default(pst_plan_opts* o);

/* --------------------------------------------------------------- tree_build
 * Set up the KV forest (CoDec "KV cache management"; block tables as in the
 * shared-prefix techniques blog, section 4.3).
 *
 *   n_nodes        number of KV nodes N (>= 1)
 *   node_len[N]    tokens held by each node (>= 0; 0-length nodes are skipped)
 *   parent[N]      parent node id, or -1 for a child of the virtual root; the
 *                  edge p -> c means "p is a prefix of c"
 *   page_ptr[N+1]  CSR offsets into page_ids (page_ptr[0] == 0, non-decreasing)
 *   page_ids[..]   physical page ids, each in [0, num_pages)
 *   first_offset   nullable (= all 0): row of the node's first token inside its
 *                  first listed page; token t of node n lives in page
 *                  page_ids[page_ptr[n] + (first_offset[n]+t)/page_size], row
 *                  (first_offset[n]+t) % page_size
 *   page_size      tokens per page: 16 or 32
 *   num_pages      pages in the pool
 *   out            receives the tree handle (free with pst_tree_destroy)
 *
 * Errors: PST_EINVAL (null/negative), PST_ECYCLE, PST_ERANGE (parent, page id,
 * first_offset >= page_size, or a node's tokens overrun its listed pages),
 * PST_EUNSUPPORTED (page_size).
 */
int pst_tree_build(int32_t n_nodes, const int32_t* node_len, const int32_t* parent,
                   const int64_t* page_ptr, const int32_t* page_ids,
                   const int32_t* first_offset, int32_t page_size, int64_t num_pages,
                   pst_tree** out);
void pst_tree_destroy(pst_tree* t);

/* ---------------------------------------------------------------- plan
 * KV-guided grouping + partition plan (CoDec "workload balancing"; DEFT
 * Algorithm 1).
 *
 *   tree           from pst_tree_build (not retained: the plan copies what it needs)
 *   n_queries      decode queries B (>= 1)
 *   query_node[B]  node each query sits on; it attends every token on the path
 *                  from the top of its tree down to that node, inclusive
 *   n_q_heads, n_kv_heads   Hq, Hkv with Hq % Hkv == 0; q-head h reads kv head
 *                  h / (Hq/Hkv)
 *   d              head dimension: 64 or 128
 *   dtype          element type of Q, K_pool and V_pool
 *   opts           nullable: defaults
 *   out            receives the plan (free with pst_plan_destroy)
 *
 * The plan is immutable and reusable for any number of pst_decode_attn calls
 * while the tree topology, node lengths and page tables stay unchanged.
 * Errors: PST_EINVAL (query out of range, a query that sees no token),
 * PST_EUNSUPPORTED (d, Hq % Hkv), PST_ECUDA (device query when num_sms == 0).
 */
int pst_plan_create(const pst_tree* tree, int32_t n_queries, const int32_t* query_node,
                    int32_t n_q_heads, int32_t n_kv_heads, int32_t d, pst_dtype dtype,
                    const pst_plan_opts* opts, pst_plan** out);
void pst_plan_destroy(pst_plan* p);

/* Incremental plan for the next decode step (CoDec, "workload balancing": the
 * plan is reused across decode steps while the tree keeps its shape). `tree`
 * has prev's node count and parents (leaves may have grown or shrunk, pages
 * may have been added); queries stay on the nodes they sat on in prev, with
 * prev's heads, d, dtype and options. The grouping, packing, chunks, items and
 * metadata are rebuilt for the new lengths, but each node keeps prev's KV-axis
 * split b_k (bounded by its tiles) instead of a new partition search; a task
 * that did not exist in prev (a packing that changed) takes ceil(C_est /
 * cost_l) under prev's cost_l. The new plan is independent of prev (upload it
 * to a workspace of its own size). Errors: PST_EINVAL (null, node count or
 * parents differ), and those of pst_plan_create. */
int pst_plan_update(const pst_plan* prev, const pst_tree* tree, pst_plan** out);

/* Incremental plan for a decode step whose tree changed shape, e.g. after the
 * verification of a speculative decoding step (CoDec, "workload balancing":
 * the plan is reused across steps; DEFT section 3.3: the accepted drafts stay,
 * the rejected ones are pruned and a new draft tree grows). `tree` is the new
 * tree, n_queries / query_node its queries (as for pst_plan_create), and
 * prev_node[N] (N = the new tree's node count) gives for each node the id of
 * the same node in prev's tree (its tokens may have grown or shrunk), or -1
 * for a node that is new. Heads, d, dtype and options come from prev. The
 * grouping, packing (bit causal masks of the new draft chunks), chunks, items
 * and metadata are built for the new tree, but a node mapped to prev keeps
 * prev's KV-axis split b_k (bounded by its tiles), and a new node takes
 * ceil(C_est / cost_l) under prev's cost bound cost_l, with no partition
 * search. The new plan is independent of prev (upload it to a workspace of its
 * own size). Errors: PST_EINVAL (null argument), PST_ERANGE (a prev_node entry
 * outside [-1, prev's node count)), and those of pst_plan_create. */
int pst_plan_update_tree(const pst_plan* prev, const pst_tree* tree, int32_t n_queries, const int32_t* query_node,
                         const int32_t* prev_node, pst_plan** out);

/* Bytes of device workspace the plan needs: its metadata plus the partial
 * output scratch (fp32 partial outputs and log-sum-exps). */
int64_t pst_plan_workspace_bytes(const pst_plan* p);

/* Copy the plan's metadata into the caller-owned device workspace (one
 * host-to-device copy on `stream`) and bind the workspace to the plan. The
 * workspace must stay allocated and unused by anything else while the plan
 * is used. d_workspace must be 256-byte aligned.
 * Errors: PST_EWORKSPACE (null, too small, misaligned), PST_ECUDA. */
int pst_plan_upload(pst_plan* p, void* d_workspace, int64_t bytes, void* stream);

/* ---------------------------------------------------------------- decode_attn
 * Tree decode attention on `stream` (asynchronous):
 *   O[b][h][:] = softmax(q_{b,h} K_b^T / sqrt(d)) V_b,
 *   LSE[b][h]  = ln sum_j exp(q_{b,h} . k_j / sqrt(d)),
 * where K_b, V_b are the tokens on query b's path (CoDec "background"; DEFT
 * section 3.2 for the LSE).
 *
 *   Q       device [B][Hq][d], dtype of the plan
 *   K_pool  device [num_pages][Hkv][page_size][d], dtype of the plan, 16-byte aligned
 *   V_pool  same layout as K_pool
 *   O       device fp32 [B][Hq][d]
 *   LSE     device fp32 [B][Hq], natural log
 *
 * Page rows not covered by any node may hold any finite or non-finite values;
 * they are never read into the result. Requires a prior pst_plan_upload.
 * Launches (opts.side_streams = 0): the PAC launch groups and POR on `stream`
 * only, each after the first with a programmatic dependency on the one
 * before (programmatic dependent launch); work queued on `stream` after the
 * call starts when all of it has finished. The call can be captured into a
 * CUDA graph after one ordinary call (which sets up the kernels).
 * Errors: PST_EWORKSPACE (no upload), PST_EINVAL (null pointer), PST_ECUDA
 * (launch failure). Device-side faults detected by the kernels' own checks
 * are reported by pst_plan_check_status().
 */
int pst_decode_attn(const pst_plan* p, const void* Q, const void* K_pool, const void* V_pool,
                    float* O, float* LSE, void* stream);

/* Read and clear the device status word written by the kernels' bounds and
 * wait-limit checks (synchronises `stream`). 0 = clean, PST_EDEVICE = a
 * kernel gave up; *code (nullable) receives the raw word. */
int pst_plan_check_status(const pst_plan* p, void* stream, int32_t* code);

/* ---------------------------------------------------------------- timing
 * Per-kernel device times of pst_decode_attn, for roofline accounting. A timer
 * holds CUDA events for up to `max_calls` calls; pst_decode_attn_timed records
 * an event at the start of the call, after each PAC launch group that has
 * work (on the stream that ran it) and around POR. It always runs the groups
 * on side streams forked from `stream` (opts.side_streams = 1), since events
 * between chained launches would serialise them. The events themselves add
 * to the call's time: time steps for throughput with pst_decode_attn.
 * Slots (pst_timer_kernel_name):
 *   0 "pac_tc"        tensor-core PAC that rounds P once to bf16 (every
 *                     tensor-core item of the mma.sync engine)
 *   1 "pac_tc_exact"  tensor-core PAC with P split into bf16 hi + lo
 *   2 "pac_thin"      PAC of the thin chunks (below tc_min_rows rows): the
 *                     tcgen05 thin PAC, or every CUDA-core row-tile launch
 *   3 "por"           partial-output reduction
 * The PAC groups run side by side on forked streams, so slots 0-2 give the
 * time from the call's start to the end of that group (overlapping
 * intervals, not shares of the call; 0 for a call in which the slot's groups
 * had no work); slot 3 is POR alone.
 * pst_timer_read synchronises on the last event, writes the summed
 * milliseconds per slot into ms[0..n-1], the number of timed calls into
 * *calls, and resets the timer. */
int pst_timer_create(int32_t max_calls, pst_timer** out);
void pst_timer_destroy(pst_timer* t);
int pst_decode_attn_timed(const pst_plan* p, const void* Q, const void* K_pool,
                          const void* V_pool, float* O, float* LSE, void* stream,
                          pst_timer* timer);
int pst_timer_read(pst_timer* t, float* ms, int32_t n, int32_t* calls);
const char* pst_timer_kernel_name(int32_t slot);

/* ---------------------------------------------------------------- no-allocation variant
 * No counterpart in the papers: this is a convenience of this library.
 *
 * Same computation and arguments as pst_decode_attn, but it needs no
 * workspace: not from the caller and not from the library at call time. It is
 * meant for callers that cannot allocate device memory where they run
 * attention -- e.g. a plug-in inside an engine whose framework owns and
 * pre-plans all device memory, or code that must avoid the device-wide
 * synchronisation of cudaFree. Its scratch (the plan's metadata and partial
 * outputs) lives in one fixed array of PST_NOALLOC_WORKSPACE_BYTES inside the
 * library's device image; every GPU on which the library is loaded holds that
 * array until the process exits.
 *
 *   - The plan need not be uploaded; plans whose pst_plan_workspace_bytes()
 *     exceeds PST_NOALLOC_WORKSPACE_BYTES are rejected with PST_EWORKSPACE.
 *   - Each call copies the plan's metadata into the array (one host-to-device
 *     copy on `stream`) before its kernels run; no allocation of any kind.
 *   - The first call on a device looks up the array's device address (with
 *     that device current) and caches it; make that first call before any
 *     CUDA stream capture.
 *   - All calls share the one array: calls whose work overlaps on the GPU (on
 *     different streams, or from different threads) race and corrupt each
 *     other. Serialise them.
 *   - The device status word used by the kernels' bounded waits lives in the
 *     array too; pst_noalloc_check_status reads it.
 */
#define PST_NOALLOC_WORKSPACE_BYTES (32ll << 20)
int pst_decode_attn_noalloc(const pst_plan* p, const void* Q, const void* K_pool, const void* V_pool,
                            float* O, float* LSE, void* stream);

/* Reads and clears the device status word in the built-in scratch of
 * pst_decode_attn_noalloc on the current device (synchronises `stream`):
 * 0 = clean, PST_EDEVICE = a kernel of the last calls gave up (a bounded wait
 * ran out or an index check failed; those calls' outputs are undefined);
 * *code (nullable) receives the raw word. Allocates nothing. */
int pst_noalloc_check_status(void* stream, int32_t* code);

/* ---------------------------------------------------------------- MLA
 * Multi-head latent attention: rebuild the per-head K/V blocks of the tree's
 * pages from a latent KV cache, after which pst_decode_attn runs the same
 * prefix-aware pipeline on them (CoDec "supplementary details", the kernel
 * module paragraph on MLA models). Every token j has a latent c_j of d_c
 * channels; kv head h has up-projections W_UK[h], W_UV[h] (d x d_c):
 *   K_pool[page][h][row][:] = bf16( W_UK[h] c_j ),  V likewise with W_UV,
 * accumulated in fp32 on the tensor cores and rounded once to bf16. Each page
 * some node of the plan's tree uses is rebuilt once (all its rows), however
 * many queries share it; other pages of K_pool / V_pool are left as they are.
 *
 *   C_pool  device bf16 [num_pages][page_size][d_c], the tree's page ids
 *   d_c     128, 256, 384 or 512
 *   W_uk    device bf16 [Hkv][d][d_c] (row e of head h: the weights of output
 *           channel e), W_uv likewise
 *   K_pool, V_pool  device bf16 [num_pages][Hkv][page_size][d] (caller-owned
 *           scratch in the layout pst_decode_attn reads)
 * All pointers 16-byte aligned. Requires a bf16 plan with page size 16 and a
 * prior pst_plan_upload (the page list lives in the workspace). Asynchronous
 * on `stream`; the kernel's bounded waits report through
 * pst_plan_check_status. Errors: PST_EINVAL, PST_EUNSUPPORTED (dtype, d_c,
 * page size), PST_EWORKSPACE (no upload), PST_ECUDA. */
int pst_mla_reconstruct(const pst_plan* p, const void* C_pool, int32_t d_c, const void* W_uk, const void* W_uv,
                        void* K_pool, void* V_pool, void* stream);

/* ---------------------------------------------------------------- introspection */
typedef struct {
    double  plan_us;              /* host time of pst_plan_create                    */
    double  predicted_makespan_us;/* list-schedule makespan under the cost model     */
    double  cost_lower_bound_us;  /* binary-searched lower bound cost_l              */
    int64_t n_chunks;             /* KV chunks (a node part or a packed subtree)     */
    int64_t n_items;              /* PAC thread blocks: chunk x kv head x row block  */
    int64_t n_tc_items;           /* ... on the tensor-core PAC                      */
    int64_t n_cc_items;           /* ... on the thin-chunk PAC (tcgen05 thin or CUDA core) */
    int64_t n_partial_rows;       /* partial outputs written per call                */
    int64_t unique_kv_tokens;     /* sum of node lengths                             */
    int64_t kv_tokens_read;       /* tokens loaded per kv head (chunks' page span)   */
    int64_t workspace_bytes;
    int32_t num_slots;            /* m: concurrent PAC blocks the schedule assumes    */
    int32_t n_launches;           /* kernels per pst_decode_attn                      */
    int32_t split_policy;         /* the plan's pst_split_policy (after the choice
                                     between node partition and DEFT-Flatten)      */
    int32_t fixed_chunk;          /* its fixed_chunk (S_t for PST_SPLIT_FLATTEN)     */
} pst_plan_stats;
int pst_plan_stats_get(const pst_plan* p, pst_plan_stats* s);

/* Plan export for exact (integer) checks. pst_plan_export_sizes fills the
 * array lengths; pst_plan_export fills every non-null pointer of `e`, each of
 * the length given by the sizes.
 *   qpath:  per query, its nodes root first (QMapKV)
 *   nodeq:  per node, ascending ids of queries sharing it (KVMapQ)
 *   chunk_q / chunk_q_mask: per chunk, its queries and, per query, a 64-bit
 *           visibility mask over the chunk's first 64 tokens (all ones when
 *           the chunk has no mask)
 *   chunk_tok_node / chunk_tok_t: per chunk, the (node, token) it covers in
 *           chunk order
 *   chunk_kind: 0 thin chunk (tcgen05 thin PAC or CUDA-core PAC), 1 tensor-core PAC
 *   merge: per query, the partial-row bases merged by POR */
typedef struct {
    int64_t n_queries, n_nodes, n_chunks;
    int64_t n_qpath, n_nodeq, n_chunk_q, n_chunk_tok, n_merge;
} pst_export_sizes;

typedef struct {
    int32_t*  qpath_ptr;      /* n_queries + 1 */
    int32_t*  qpath_node;     /* n_qpath       */
    int32_t*  nodeq_ptr;      /* n_nodes + 1   */
    int32_t*  nodeq;          /* n_nodeq       */
    int32_t*  chunk_q_ptr;    /* n_chunks + 1  */
    int32_t*  chunk_q;        /* n_chunk_q     */
    uint64_t* chunk_q_mask;   /* n_chunk_q     */
    int32_t*  chunk_tok_ptr;  /* n_chunks + 1  */
    int32_t*  chunk_tok_node; /* n_chunk_tok   */
    int32_t*  chunk_tok_t;    /* n_chunk_tok   */
    int32_t*  chunk_kind;     /* n_chunks      */
    int32_t*  merge_ptr;      /* n_queries + 1 */
    int32_t*  merge_row;      /* n_merge       */
} pst_export;

int pst_plan_export_sizes(const pst_plan* p, pst_export_sizes* s);
int pst_plan_export(const pst_plan* p, pst_export* e);

/* Cost model C_est(rows, tokens) in microseconds for one PAC thread block
 * with every SM busy (CoDec "profile-based cost estimation"), per PAC kind:
 * 0 = CUDA-core PAC, 1 = tcgen05 PAC with P rounded once to bf16, 2 = tcgen05
 * PAC with exact (hi + lo) P, 3 = tcgen05 thin PAC. Tables measured on a GB300 are built in (see
 * the package's cost_fit.py); pst_cost_set_table replaces the table of one
 * kind: n_r row grid points x n_n token grid points, values row-major
 * [n_r][n_n]; n_r == 0 selects the analytic model for that kind and n_r < 0
 * restores the built-in table. Between grid
 * points the estimate is bilinear in (log rows, log tokens), past the last
 * token point it grows linearly with tokens. The tables cover d = 128 bf16;
 * other shapes and the mma.sync engine use the analytic model. For the thin
 * PAC (one block per SM) C_est is the block's wall time. Process-wide;
 * plans created afterwards use it. pst_cost_estimate returns -1 for an
 * unknown kind. */
int pst_cost_set_table(int32_t kind, int32_t n_r, const float* rows, int32_t n_n,
                       const float* tokens, const float* us);
double pst_cost_estimate(int32_t kind, double rows, double tokens);

/* The partitioner's list schedule, exported for checks (host only): CoDec,
 * "workload balancing", assigns the sub-tasks to the m thread-block slots
 * largest first, each to the least-loaded slot (Graham's list scheduling,
 * whose makespan is at most (2 - 1/m) times the optimum; largest-first order
 * tightens that to 4/3 - 1/(3m)). n costs (>= 0) go onto m slots; slot[i]
 * (nullable) receives task i's slot in [0, m), ties going to the lowest slot
 * index and equal costs to the lower task index first; *makespan (nullable)
 * the largest slot load. Errors: PST_EINVAL (n < 0, m <= 0, a negative or
 * NaN cost). */
int pst_list_schedule(int32_t n, const double* cost, int32_t m, int32_t* slot, double* makespan);

const char* pst_last_error(void);

#ifdef __cplusplus
}
#endif
#endif /* PST_H */
