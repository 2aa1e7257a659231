/*
 * vas.h -- C ABI of libvas.so: the data-parallel hot path of one continuous-batching
 * iteration on one NVIDIA GB300 (sm_103a).
 *
 *   paged_attn_fwd  : attention of a ragged batch of decode (1 query token) and
 *                     speculative-verify (k+1 query tokens) sequences over a KV cache
 *                     held in fixed-size pages addressed through per-sequence block
 *                     tables (split-KV with a log-sum-exp merge).
 *   paged_attn_fwd_tree, paged_attn_fwd_quant, paged_attn_fwd_static : the same
 *                     attention with draft-tree masks, over FP8 / INT8 pages, and
 *                     without a caller workspace.
 *   spec_verify     : speculative-decoding modified rejection sampling with an
 *                     in-kernel Philox4x32-10 stream; spec_verify_tree, the same rule
 *                     over a draft tree.
 *   vas_last_device_error, vas_philox4x32_10 : the device error word, and the device
 *                     Philox stream on caller counters.
 *   vas_pool_*      : host-side page allocator and block-table builder that models
 *                     admission, growth, rollback of rejected drafts, eviction.
 *
 * Conventions shared by every entry point
 *  - Plain C types only.  Device pointers belong to the caller and no call allocates
 *    device memory.  Scratch space (paged_attn_fwd's workspace) is caller-owned and
 *    sized by the matching *_workspace_size query; paged_attn_fwd_static instead uses a
 *    fixed array the library reserves once per GPU when its device code is loaded.
 *  - Device calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy default
 *    stream).  They validate their arguments on the host and return a status code
 *    immediately; nothing synchronises except vas_last_device_error.
 *  - Problems that only the device can see (a bad block-table entry, inconsistent
 *    lengths, an out-of-range draft token) never trap: the kernel sets a bit in a
 *    per-device error word (read with vas_last_device_error) and poisons the affected
 *    outputs (NaN for attention rows, -1 for tokens).
 *  - Every device entry point runs on the device current for the calling thread.
 */
#ifndef VAS_H
#define VAS_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* vas_stream_t; /* identical to cudaStream_t */

/* ---- status codes (return values) ---------------------------------------------- */
#define VAS_OK 0
#define VAS_E_INVALID_ARG (-1) /* null pointer, bad size, misaligned buffer          */
#define VAS_E_UNSUPPORTED (-2) /* dtype / head_dim / page_size this build lacks      */
#define VAS_E_WORKSPACE (-3)   /* workspace smaller than the minimum for these dims   */
#define VAS_E_CUDA (-4)        /* a CUDA runtime or driver call failed                */
#define VAS_E_NOMEM (-5)       /* page pool: not enough free pages                    */
#define VAS_E_NOT_FOUND (-6)   /* page pool: unknown sequence id                      */
#define VAS_E_EXISTS (-7)      /* page pool: sequence id already admitted             */

/* ---- device error bits (vas_last_device_error) --------------------------------- */
#define VAS_DEV_BAD_PAGE 0x1       /* block-table entry outside [0, num_pages)         */
#define VAS_DEV_BAD_LENGTHS 0x2    /* query_len > seq_len, seq_len > max_pages*page,   */
                                   /* negative length, or sum(query_lens) differs from */
                                   /* total_q_tokens                                   */
#define VAS_DEV_BAD_TOKEN 0x4      /* draft token outside [0, V)                       */
#define VAS_DEV_EMPTY_ROW 0x8      /* the row to draw from has no positive mass        */
#define VAS_DEV_TIMEOUT 0x10       /* a bounded in-kernel wait gave up                 */
#define VAS_DEV_BAD_TREE 0x20      /* spec_verify_tree: a parent outside 0..node - 1     */
#define VAS_DEV_RESIDUAL_FALLBACK 0x100 /* informational: a zero residual after a       */
                                        /* rejection; the token was drawn from p_j      */

/* Storage types of k_pages and v_pages (and of q and out for VAS_F32 / VAS_BF16; with
 * the quantised types q and out are bf16). */
#define VAS_F32 0
#define VAS_BF16 1
#define VAS_FP8_E4M3 2 /* FP8 E4M3 codes + fp32 scales, paged_attn_fwd_quant only */
#define VAS_INT8 3     /* INT8 codes + fp32 scales, paged_attn_fwd_quant only     */

/* ==================================================================================
 * Paged decode / verify attention
 *
 * Defined by: "Continuous Batching and Speculative Decoding: How Modern LLM Serving
 * Engines Actually Work" (syslabs.in), section "PagedAttention: making the KV cache
 * schedulable" -- fixed-size KV blocks, a per-sequence block table mapping logical
 * positions to physical blocks, and kernels that read through that indirection; and
 * section "The core idea" -- the target verifies k proposals in one pass over
 * context + proposals.  Pool layout from "llm-inference-optimization-batching"
 * (tempatgunting.com), section "Anatomy of the KV Cache": [num_blocks, block_size,
 * num_heads, head_dim].  Ragged batches without padding: same page, section
 * "Implementation Details That Affect Tail Latency" (cu_seqlens-style packing).
 *
 * For sequence i (length L_i = seq_lens[i] KV tokens, this step's query tokens
 * included) with ql_i = query_lens[i] query tokens, query token j (0 <= j < ql_i) sits
 * at position pos = L_i - ql_i + j and attends to KV positions 0..pos (causal inside
 * the draft window).  Query head h reads KV head h / (num_q_heads / num_kv_heads).
 * KV position t lives in page block_table[i][t / page_size], slot t % page_size.
 *     s_t = scale * <q, k_t>,   lse = ln sum_t exp(s_t),   out = sum_t exp(s_t - lse) v_t
 * ================================================================================== */
typedef struct {
  int32_t num_seqs;          /* B, number of sequences in the batch                   */
  int32_t total_q_tokens;    /* T = sum of query_lens (rows of q / out / lse)         */
  int32_t num_q_heads;       /* Hq                                                    */
  int32_t num_kv_heads;      /* Hkv; Hq % Hkv == 0                                    */
  int32_t head_dim;          /* D: 64 or 128                                          */
  int32_t page_size;         /* P: 16 or 32 tokens per page                           */
  int32_t num_pages;         /* physical pages in the pool                            */
  int32_t max_pages_per_seq; /* columns of block_table                                */
  int32_t kv_dtype;          /* VAS_BF16 or VAS_F32 (q and out share it), or          */
                             /* VAS_FP8_E4M3 / VAS_INT8 (q and out bf16)              */
  float scale;               /* softmax scale; 0 selects 1/sqrt(head_dim)             */
} vas_attn_dims;

/* Bytes of workspace paged_attn_fwd should be given for these dimensions (a
 * recommendation: any size >= paged_attn_workspace_min works; a smaller workspace
 * only limits how finely long sequences are split across SMs).  Returns 0 for
 * invalid dims. */
size_t paged_attn_workspace_size(const vas_attn_dims* dims);

/* Smallest workspace paged_attn_fwd accepts for these dimensions. */
size_t paged_attn_workspace_min(const vas_attn_dims* dims);

/*
 * q           [T, Hq, D]            device, kv_dtype, 16-byte aligned.  Rows packed by
 *                                   sequence in batch order (row of token j of sequence
 *                                   i = sum_{i'<i} query_lens[i'] + j).
 * k_pages     [num_pages, P, Hkv, D] device, kv_dtype, 16-byte aligned.
 * v_pages     [num_pages, P, Hkv, D] device, same layout as k_pages.
 * block_table [B, max_pages_per_seq] device int32; entries past ceil(L_i / P) are not
 *                                   read (pad with -1).  Tables may share pages.
 * seq_lens    [B] device int32, L_i >= query_lens[i] >= 0.
 * query_lens  [B] device int32: 1 for decode, k+1 for verify (0 skips the sequence).
 * out         [T, Hq, D]            device, kv_dtype, 16-byte aligned; fully written.
 * lse         [T, Hq]               device fp32, natural log; fully written.
 * workspace   device scratch, 256-byte aligned, at least paged_attn_workspace_min
 *             bytes; contents need no initialisation and are overwritten.
 * Errors: VAS_E_INVALID_ARG / VAS_E_UNSUPPORTED / VAS_E_WORKSPACE on the host;
 * VAS_E_CUDA if a launch fails.  Device-detected problems set VAS_DEV_BAD_PAGE or
 * VAS_DEV_BAD_LENGTHS and write NaN to the affected rows of out and lse.
 * Two calls sharing one workspace must be ordered on the device (same stream).
 */
int paged_attn_fwd(const void* q, const void* k_pages, const void* v_pages,
                   const int32_t* block_table, const int32_t* seq_lens,
                   const int32_t* query_lens, void* out, float* lse,
                   const vas_attn_dims* dims, void* workspace, size_t workspace_bytes,
                   vas_stream_t stream);

/* paged_attn_fwd for draft trees.
 *
 * Defined by: "Continuous Batching & Speculative Decoding" (neuralmasteryai.com),
 * section "4. Tree Attention & Medusa Heads" -- the draft is a tree of candidate
 * tokens, verified in one pass under a tree attention mask; and
 * "llm-inference-optimization-batching" (tempatgunting.com), section "Draft Model
 * Selection and Tree-Style Variants" -- verifying a tree of drafts masks attention by
 * the tree's shape.
 *
 * tree_mask   [T] device uint64, 8-byte aligned, one word per query token (the rows of
 *             q).  For query token j of sequence i, bit a (a < j) set means draft token a
 *             of the same sequence (position L_i - ql_i + a) is an ancestor of j in the
 *             tree.  Token j then attends to every context position (0 .. L_i - ql_i - 1),
 *             to the draft tokens whose bits are set, and to itself (its own bit is
 *             implied).  Bits a >= j are ignored: a parent precedes its children in the
 *             packing, so a chain (bits 0 .. j-1 set) is exactly paged_attn_fwd.
 *             Sequences with ql_i == 1 or ql_i > 64 ignore their words and use the
 *             causal window of paged_attn_fwd (64 draft tokens at most per tree).
 * Other arguments, results and errors: those of paged_attn_fwd; a null tree_mask is
 * VAS_E_INVALID_ARG.
 */
int paged_attn_fwd_tree(const void* q, const void* k_pages, const void* v_pages,
                        const int32_t* block_table, const int32_t* seq_lens,
                        const int32_t* query_lens, const uint64_t* tree_mask, void* out,
                        float* lse, const vas_attn_dims* dims, void* workspace,
                        size_t workspace_bytes, vas_stream_t stream);

/* paged_attn_fwd over a quantised KV cache.
 *
 * Defined by: "llm-inference-optimization-batching" (tempatgunting.com), section
 * "Quantization and Precision Choices for KV" -- INT8 or FP8 KV pages with per-head or
 * per-token scaling factors, separate for K and V, dequantised inside the attention
 * kernel; "Continuous Batching and Speculative Decoding..." (syslabs.in), section "A
 * tuning framework" (an FP8 KV cache to fit more blocks).
 *
 * dims->kv_dtype is VAS_FP8_E4M3 (OCP E4M3: bias 7, 3 mantissa bits, subnormals, no
 * infinities, max 448) or VAS_INT8 (two's complement).  Element d of token slot t of
 * page p, KV head h, stands for
 *     k = k_scale[(p * num_kv_heads + h) * page_size + t] * code(k_pages[p][t][h][d])
 * and likewise for v with v_scale: one scale per token and KV head, no zero point.
 * k_pages     [num_pages, P, Hkv, D] device bytes (the pool layout), 16-byte aligned.
 * v_pages     the same for V.
 * k_scale     [num_pages, Hkv, P] device fp32, 16-byte aligned.
 * v_scale     the same for V.  Scales of slots past a sequence's end are not used.
 * q, out      [T, Hq, D] bf16.  lse, block_table, seq_lens, query_lens, workspace: as for
 *             paged_attn_fwd (the workspace queries are the same for every kv_dtype).
 * tree_mask   null (the causal window) or the draft-tree masks of paged_attn_fwd_tree.
 * Arithmetic: the codes are exact in f16; Q is taken to f16 (scaled by a power of two
 * when its magnitude nears the f16 range), products accumulate in fp32, and P enters
 * the PV product as f16 after multiplication by the V scale of its token, so
 * |v_scale| * 256 must stay within the f16 range (|v| up to about 1e5).
 * Errors: those of paged_attn_fwd; a kv_dtype that is not quantised, or a null scale
 * array, is VAS_E_INVALID_ARG.  paged_attn_fwd and paged_attn_fwd_tree reject the
 * quantised kv_dtypes with VAS_E_INVALID_ARG.
 */
int paged_attn_fwd_quant(const void* q, const void* k_pages, const void* v_pages,
                         const float* k_scale, const float* v_scale, const int32_t* block_table,
                         const int32_t* seq_lens, const int32_t* query_lens,
                         const uint64_t* tree_mask, void* out, float* lse,
                         const vas_attn_dims* dims, void* workspace, size_t workspace_bytes,
                         vas_stream_t stream);

/* paged_attn_fwd without a workspace argument, for callers that cannot allocate device
 * memory: code being captured into a CUDA graph (where cudaMalloc is not allowed), hosts
 * that hand a plug-in only the tensors of a call, or callers whose allocator is out of
 * memory.  The web pages have no counterpart; this is a property of the library.
 * Scratch space is a 32 MiB array in device global memory that the library reserves on
 * every GPU where its device code is loaded, held until the process exits; the call
 * itself allocates nothing.  The first call on a device looks up that array's address
 * (and so does the first call after the device's context has been created anew, e.g.
 * after cudaDeviceReset); make that first call before any stream capture.  Arguments and results are those of
 * paged_attn_fwd.  Returns VAS_E_WORKSPACE when the batch needs more than 32 MiB of plan
 * space (paged_attn_workspace_min(dims) > 32 MiB; thousands of sequences fit); a batch
 * whose split partials would not fit is split less finely instead.  Every call on a
 * device shares the one array, and each call rewrites all of it that it reads, so no
 * clearing is needed between calls -- but calls whose kernels may overlap on the GPU
 * (different streams without ordering between them) race on it: order them. */
int paged_attn_fwd_static(const void* q, const void* k_pages, const void* v_pages,
                          const int32_t* block_table, const int32_t* seq_lens,
                          const int32_t* query_lens, void* out, float* lse,
                          const vas_attn_dims* dims, vas_stream_t stream);

/* ==================================================================================
 * Speculative verification: modified rejection sampling
 *
 * Defined by: "Continuous Batching & Speculative Decoding" (neuralmasteryai.com),
 * section "3. Mathematical Proof: Exact Distributional Match" / "The Modified
 * Rejection Sampling Algorithm" -- accept x_i when r <= min(1, p(x_i)/q(x_i)), halt
 * at the first rejection, resample from max(0, p - q) / sum_y max(0, p(y) - q(y));
 * "Continuous Batching and Speculative Decoding..." (syslabs.in), section "The core
 * idea" -- a bonus token from the last target row when all k drafts are accepted.
 *
 * For sequence b: for i = 0..k-1 accept draft x_i iff r_i * q_i(x_i) <= p_i(x_i)
 * (evaluated in double); j = first rejected position, or k.  The token at position j
 * is drawn by inverse CDF (smallest x whose inclusive prefix sum exceeds s_j * S)
 * from w = max(0, p_j - q_j) when j < k, else from w = p_k; S = sum w.  A zero
 * residual after a rejection (impossible in exact arithmetic) draws from p_j instead
 * and sets VAS_DEV_RESIDUAL_FALLBACK.
 * Uniforms: Philox4x32-10 (Salmon et al., SC'11) with key (seed low 32 bits, seed
 * high 32 bits) and counter (position, b, 0, 0); r_i = (word0 + 0.5) * 2^-32 of
 * position i, s_j = (word1 + 0.5) * 2^-32 of position j.
 *
 * p            [B, k+1, V] device fp32 target probabilities (row k: bonus row).
 * q            [B, k, V]   device fp32 draft probabilities (may be NULL when k == 0).
 * draft_tokens [B, k]      device int32 (may be NULL when k == 0).
 * accepted_len [B]         device int32 out: j (number of accepted drafts); -1 for a
 *                          sequence with an out-of-range draft token.
 * out_tokens   [B, k+1]    device int32 out: x_0..x_{j-1}, the drawn token, then -1.
 * Rows need no alignment.  k == 0 is plain sampling from p_0.  k < 256 and
 * V <= 1048576 (VAS_E_INVALID_ARG / VAS_E_UNSUPPORTED beyond).
 * Errors: VAS_E_INVALID_ARG on the host; device: VAS_DEV_BAD_TOKEN (sequence emits
 * -1s), VAS_DEV_EMPTY_ROW (position j emits -1).
 */
int spec_verify(const float* p, const float* q, const int32_t* draft_tokens, uint64_t seed,
                int32_t* accepted_len, int32_t* out_tokens, int32_t B, int32_t k, int32_t V,
                vas_stream_t stream);

/* Synchronises `stream`, then returns (and clears) the device error word of the
 * current device in *bits.  Returns VAS_OK or VAS_E_CUDA. */
int vas_last_device_error(int32_t* bits, vas_stream_t stream);

/* Verification of a draft tree.
 *
 * Defined by: "Continuous Batching & Speculative Decoding" (neuralmasteryai.com),
 * section "4. Tree Attention & Medusa Heads" -- candidate paths verified in one pass --
 * and section "The Modified Rejection Sampling Algorithm", applied to a node's
 * children in turn (the pages give no rule for several candidates; this reading keeps
 * the output distribution equal to p when each child of a node was drawn
 * independently from that node's q row).
 *
 * Per sequence b: nodes 1..n are draft tokens, node 0 is the root (the last context
 * token).  parents[b][i] is the parent of node i + 1, in 0..i; draft_tokens[b][i] its
 * token.  p[b][u] ([B, n+1, V] fp32) is the target's distribution after node u;
 * q[b][u] ([B, n, V] fp32) the distribution node u's children were drawn from.
 * Walk: at node u the children are tried in node order against a residual R (first
 * p_u) with total S (first 1): child c with token x is accepted iff
 * r_c * S * q_u(x) <= R(x), r_c = (word 0 of Philox(c - 1, b)) per spec_verify; a
 * rejection makes R = max(0, R - S * q_u) and S its sum.  An accepted child becomes u.
 * When a node's children are all rejected, or it has none, one token is drawn from R
 * by inverse CDF with word 1 of Philox(u, b) (from p_u when a rejection leaves a zero
 * residual: VAS_DEV_RESIDUAL_FALLBACK) and the walk ends.  For a chain (parents[b][i]
 * = i) this is exactly spec_verify.
 * Outputs: accepted_len[b] (accepted draft tokens), out_tokens[b] ([n+1]: the accepted
 * tokens, the drawn token, then -1), path[b] ([n]: the accepted nodes, then -1).
 * n in 1..255.  Errors: VAS_E_INVALID_ARG on the host; device: VAS_DEV_BAD_TOKEN or
 * VAS_DEV_BAD_TREE (the sequence emits accepted_len = -1 and all -1), VAS_DEV_EMPTY_ROW.
 */
int spec_verify_tree(const float* p, const float* q, const int32_t* draft_tokens,
                     const int32_t* parents, uint64_t seed, int32_t* accepted_len,
                     int32_t* out_tokens, int32_t* path, int32_t B, int32_t n, int32_t V,
                     vas_stream_t stream);

/* Diagnostic: the device Philox4x32-10 used by spec_verify, exposed for testing.
 * counters [n, 4] and out [n, 4] are device uint32 arrays; key = (key0, key1). */
int vas_philox4x32_10(const uint32_t* counters, uint32_t key0, uint32_t key1, uint32_t* out,
                      int64_t n, vas_stream_t stream);

/* Human-readable name of a status code (static string). */
const char* vas_status_string(int status);

/* ==================================================================================
 * Host page allocator and block-table builder
 *
 * Models the KV block manager of the pages: fixed-size blocks handed out on demand
 * from a free list, a block table per sequence, blocks returned on finish
 * (syslabs.in "PagedAttention"; martinuke0.github.io "PagedAttention: The Other Half
 * of the Story"), admission gated on can_allocate and preemption of the newest
 * sequence when the pool is exhausted (syslabs.in "Continuous batching: scheduling
 * per iteration"), speculative reservation of k+1 slots and rollback of rejected
 * drafts (tempatgunting.com "Speculative Decoding..."; mohashari.github.io
 * "Speculative Decoding: Draft Fast, Verify Cheap"), and prefix sharing with
 * reference counts (tempatgunting.com "Anatomy of the KV Cache").
 * Waste is at most one partially filled page per sequence.  Host memory only; not
 * thread-safe (one pool per scheduler thread).
 * ================================================================================== */
typedef struct vas_pool vas_pool;

/* A pool of num_pages pages of page_size tokens.  The free list starts as a seeded
 * random permutation of the page ids (seed 0: ascending).  NULL on bad arguments. */
vas_pool* vas_pool_create(int32_t num_pages, int32_t page_size, uint64_t seed);
void vas_pool_destroy(vas_pool* pool);

int32_t vas_pool_free_pages(const vas_pool* pool);
int32_t vas_pool_num_seqs(const vas_pool* pool);
/* 1 if a new sequence of n_tokens tokens fits in the free pages, else 0. */
int vas_pool_can_allocate(const vas_pool* pool, int32_t n_tokens);
/* Pages sequence seq_id would need to grow by n_tokens (0 if its last page has room);
 * negative status for an unknown id. */
int32_t vas_seq_pages_needed(const vas_pool* pool, int64_t seq_id, int32_t n_tokens);
/* Current length (tokens) of seq_id, or a negative status. */
int32_t vas_seq_len(const vas_pool* pool, int64_t seq_id);

/* Admit a new sequence holding n_tokens tokens (its prompt).  VAS_E_NOMEM leaves the
 * pool unchanged. */
int vas_seq_admit(vas_pool* pool, int64_t seq_id, int32_t n_tokens);
/* Append n_tokens (1 for decode, k+1 for a verify step).  All-or-nothing. */
int vas_seq_grow(vas_pool* pool, int64_t seq_id, int32_t n_tokens);
/* Drop the last n_tokens (rejected drafts) and free pages past the new end. */
int vas_seq_rollback(vas_pool* pool, int64_t seq_id, int32_t n_tokens);
/* Retire a sequence and return its pages (shared pages when their count drops to 0). */
int vas_seq_free(vas_pool* pool, int64_t seq_id);
/* Evict the most recently admitted sequence; its id is stored in *victim. */
int vas_pool_preempt_newest(vas_pool* pool, int64_t* victim);
/* New sequence child_id sharing every full page of parent_id's first n_tokens tokens
 * (a common prefix) by reference; the remainder is copied into fresh pages by the
 * caller (the copies' ids are in the child's block table).  n_tokens <= parent length. */
int vas_seq_fork(vas_pool* pool, int64_t parent_id, int64_t child_id, int32_t n_tokens);
/* Reference count of a page (0 = free). */
int32_t vas_page_refcount(const vas_pool* pool, int32_t page);

/* Dense block table for n sequences: block_table [n, max_pages] row r lists the page
 * ids of seq_ids[r] in logical order, padded with -1; seq_lens[r] receives its length.
 * VAS_E_INVALID_ARG if a sequence needs more than max_pages pages. */
int vas_build_block_table(const vas_pool* pool, const int64_t* seq_ids, int32_t n,
                          int32_t* block_table, int32_t max_pages, int32_t* seq_lens);

#ifdef __cplusplus
}
#endif

#endif /* VAS_H */
