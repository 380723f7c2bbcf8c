/*
 * spec_verify.h -- C ABI of libspecverify, the batched speculative-decoding
 * verification step over a paged KV cache, for NVIDIA GB300 (sm_103a).
 *
 * One verify step for a continuous batch is four calls on one CUDA stream:
 *
 *   sv_kv_append              write the K_b+1 new K/V rows of every sequence
 *                             into its blocks, taking blocks from the free list
 *   sv_spec_verify_attn       (K_b+1)-query GQA attention over the paged cache,
 *                             causal or tree mask
 *   sv_spec_rejection_sample  vocab-wide softmax of target and draft logits,
 *                             accept test, first-reject scan and residual
 *                             resample (or greedy / tree-greedy acceptance)
 *   sv_kv_rollback            truncate every sequence at its accepted length
 *
 * Between steps, on the host, sv_adaptive_k_update turns the accept counts
 * into each sequence's draft length for the next step. sv_kv_fork lets new
 * sequences share a parent's blocks (copy-on-write, with kv->ref_count) and
 * sv_kv_release gives a finished sequence's blocks back.
 *
 * Conventions shared by every call:
 *  - Pointers are DEVICE pointers owned by the caller, unless stated. The
 *    library never allocates, frees or keeps a pointer after a call returns.
 *  - Calls are asynchronous on `stream` (a cudaStream_t passed as void*;
 *    NULL = the legacy default stream). Nothing synchronises with the host.
 *  - The return value reports what the host can see: argument errors
 *    (SV_ERR_INVALID_ARG / SV_ERR_UNSUPPORTED / SV_ERR_WORKSPACE, nothing is
 *    launched) and launch errors (SV_ERR_CUDA).
 *  - Errors found on the device go to `status_dev`, one int32 in device
 *    memory. A kernel records its error only if the word still holds SV_OK
 *    (the first error wins). sv_kv_append and sv_kv_rollback do nothing at all
 *    while the word holds an error, so a failed step leaves the cache as it
 *    was; the caller clears the word (writes 0) to go on.
 *  - No C++ exception crosses this ABI.
 *
 * Query rows are ragged: sequence b owns rows cu_q[b] .. cu_q[b+1]-1 (n_b of
 * them, 1 <= n_b <= max_q_per_seq <= 64). Row 0 of a sequence is the last
 * emitted token; rows 1..n_b-1 are its draft tokens (chain) or its draft-tree
 * nodes in BFS order (tree). Arrays on the draft side (draft logits, draft
 * tokens, accept uniforms) have one entry per row except row 0: the entry of
 * row i >= 1 sits at index cu_q[b] - b + i - 1.
 *
 * The method (pages on speculative decoding, cited by title and section):
 *  - the target scores the K drafts plus one bonus position in one pass
 *    ("Speculative decoding and continuous batching in practice", sec. 1.2);
 *  - accept x with probability min(1, p(x)/q(x)); on the first rejection draw
 *    from norm(max(0, p - q)) and drop the rest of the draft ("Speculative
 *    decoding principles and a vLLM production setup", sec. 2.1-2.2);
 *  - a block table maps each sequence's logical KV blocks to physical ones,
 *    and blocks are taken only when the current one is full ("LLM serving:
 *    speculative decoding and PagedAttention memory management",
 *    PagedAttention section);
 *  - on rejection only whole blocks of rejected positions go back, accepted
 *    entries stay in place (vLLM page, sec. 3.1); tree drafts are verified in
 *    one pass under a tree mask (vLLM page, sec. 3.2 and 5.2).
 */
#ifndef SPEC_VERIFY_H
#define SPEC_VERIFY_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum sv_status {
  SV_OK = 0,
  SV_ERR_INVALID_ARG = 1,   /* host: a pointer, size or enum is invalid */
  SV_ERR_UNSUPPORTED = 2,   /* host: valid but not built (e.g. head_dim > 256) */
  SV_ERR_CUDA = 3,          /* host: a CUDA launch or attribute call failed */
  SV_ERR_OUT_OF_BLOCKS = 4, /* device: the free list holds too few blocks */
  SV_ERR_TIMEOUT = 5,       /* device: a bounded wait inside a kernel gave up */
  SV_ERR_BAD_BLOCK_ID = 6,  /* device: a block id outside [0, num_blocks) */
  SV_ERR_BAD_LENGTH = 7,    /* device: a length, accept count or path entry out of range */
  SV_ERR_BAD_TOKEN = 8,     /* device: a token id outside [0, vocab) */
  SV_ERR_NONFINITE = 9,     /* device: a NaN or +inf logit, a row without finite logits, or a
                               query beyond fp16 range on the E4M3 tensor-core path */
  SV_ERR_WORKSPACE = 10     /* host: workspace missing or smaller than required */
} sv_status;

/* SV_DTYPE_E4M3 (8-bit floating point: sign, 4 exponent bits with bias 7, 3
 * mantissa bits, no infinity, largest finite 448) is a KV-pool type only. */
typedef enum sv_dtype { SV_DTYPE_BF16 = 0, SV_DTYPE_F32 = 1, SV_DTYPE_E4M3 = 2 } sv_dtype;

typedef enum sv_mask_kind { SV_MASK_CAUSAL = 0, SV_MASK_TREE = 1 } sv_mask_kind;

/*
 * One layer's paged KV cache. Every pointer is a caller-owned device pointer.
 *   k_pool, v_pool   [num_blocks, num_kv_heads, block_size, head_dim] of dtype,
 *                    head-major inside a block: the rows of one (block, head)
 *                    are contiguous (block_size * head_dim elements)
 *   block_table      int32 [batch, max_blocks_per_seq]: logical -> physical
 *                    block; -1 marks "no block"
 *   seq_lens         int32 [batch]: committed tokens c_b (KV rows kept)
 *   free_list        int32 [num_blocks]: a stack of free physical ids; entries
 *                    [0, *free_top) are valid, entry *free_top-1 is the top
 *   free_top         int32 [1]
 *   ref_count        int32 [num_blocks], or NULL: no block is shared. With it,
 *                    sequences may share physical blocks copy-on-write ("LLM
 *                    serving: speculative decoding and PagedAttention memory
 *                    management", PagedAttention section: parent and child
 *                    sequences of beam search or parallel sampling share
 *                    blocks): ref_count[x] is the number of block-table
 *                    entries, over all sequences, that hold block x (0 for a
 *                    free block). The caller sets it up to match the tables
 *                    (1 per held block when nothing is shared yet); the calls
 *                    below keep it so.
 *   k_scale, v_scale dequantisation scales of an SV_DTYPE_E4M3 pool (the value
 *                    of a stored code is its E4M3 value times the scale);
 *                    finite and > 0; ignored for the other types.
 * block_size: a power of two in [1, 256]; head_dim: a multiple of 8 in
 * [8, 256] (of 16 for E4M3); dtype: SV_DTYPE_BF16, SV_DTYPE_F32 or
 * SV_DTYPE_E4M3.
 *
 * fp8 pools (SV_DTYPE_E4M3; the pages mention KV-cache quantisation without a
 * format, "LLM serving: speculative decoding and PagedAttention memory
 * management", TensorRT-LLM section; the reading taken: E4M3 codes with one
 * scale per pool): the new rows given to sv_kv_append and the queries and
 * outputs of sv_spec_verify_attn are bf16. Append stores each new element x as
 * the E4M3 code nearest to x / scale (fp32 division; ties to the even
 * mantissa; saturating at +-448), so it never writes the NaN codes 0x7F and
 * 0xFF; a pool must not hold them. Attention reads code * scale: the CUDA-core
 * kernel in fp32; the tcgen05 kernel (head_dim 128) widens the codes to fp16
 * exactly, rounds the queries and the softmax weights to fp16 and applies the
 * scales to the scores and the outputs in fp32, so a query element beyond the
 * fp16 range (|q| > 65504) records SV_ERR_NONFINITE there.
 */
typedef struct sv_paged_kv {
  void *k_pool;
  void *v_pool;
  int32_t *block_table;
  int32_t *seq_lens;
  int32_t *free_list;
  int32_t *free_top;
  int32_t num_blocks;
  int32_t block_size;
  int32_t max_blocks_per_seq;
  int32_t num_kv_heads;
  int32_t head_dim;
  int32_t batch;
  int32_t dtype;
  int32_t *ref_count;
  float k_scale;
  float v_scale;
} sv_paged_kv;

/*
 * sv_kv_append -- write the new K/V rows of every sequence into the cache.
 *
 * Sequence b needs ceil((c_b + n_b) / bs) - ceil(c_b / bs) new blocks (a block
 * is taken only when the current one is full). They are popped from the free
 * list in (sequence, logical block) order: the top entry goes to sequence 0's
 * first new block. Row j of sequence b (new_k[cu_q[b] + j]) is then written at
 * logical position c_b + j: physical block block_table[b][(c_b+j) / bs], slot
 * (c_b+j) % bs, for every KV head. seq_lens is not changed (the new rows are
 * pending until sv_kv_rollback).
 * With ref_count: a sequence whose first new row lands in a partly filled
 * block that is still shared when its turn comes (sequences in order; a block
 * held by r sequences) first takes a private copy: one more block, popped just
 * before its new blocks, that receives the block's c_b % bs rows (every KV
 * head) and replaces it in the table; the shared block's count drops by one.
 * So of w writers into a block held by r, the first min(w, r - 1) copy and a
 * last writer that holds the only remaining reference writes in place. New
 * blocks get count 1.
 *   new_k, new_v  [total_q, num_kv_heads, head_dim] of kv->dtype (bf16 for an E4M3 pool)
 *   cu_q          int32 [batch + 1], cu_q[0] = 0, cu_q[batch] = total_q
 *   status_dev    int32 [1], required
 * All or nothing: if the blocks would not fit the block table
 * (SV_ERR_BAD_LENGTH), the free list is too short (SV_ERR_OUT_OF_BLOCKS), or a
 * popped id is out of range (SV_ERR_BAD_BLOCK_ID), nothing is written.
 * Popped free-list entries are overwritten with -1.
 */
sv_status sv_kv_append(const sv_paged_kv *kv, const void *new_k, const void *new_v, const int32_t *cu_q,
                       int32_t total_q, int32_t *status_dev, void *stream);

/*
 * Workspace bytes sv_spec_verify_attn needs for these sizes: the split-KV
 * partial results (head_dim floats plus one log-sum-exp per partial row) of
 * whichever kernel the call may select, and for the tcgen05 kernel the
 * per-sequence tile prefix. max_seq_len bounds c_b + n_b over the batch;
 * max_q_per_seq bounds n_b. Returns 0 for invalid sizes.
 */
size_t sv_spec_verify_attn_workspace_bytes(const sv_paged_kv *kv, int32_t num_q_heads, int32_t total_q,
                                           int32_t max_q_per_seq, int32_t max_seq_len);

/*
 * sv_spec_verify_attn -- (K+1)-query grouped-query attention over the paged
 * cache, after sv_kv_append has written the step's rows.
 *
 * For sequence b with L_b = c_b + n_b tokens (c_b = seq_lens[b]), query row i
 * (0 <= i < n_b) and query head h (KV head h / (num_q_heads / num_kv_heads)):
 *   out[row][h] = sum_t softmax_t(scale * <q[row][h], k_t>) v_t
 * over the visible t < L_b: all committed t < c_b, plus new row j = t - c_b
 * when j <= i (SV_MASK_CAUSAL) or when bit j of tree_mask[row] is set
 * (SV_MASK_TREE: the row's ancestors and itself; the caller sets the bits).
 * Softmax and accumulation are fp32; a row that sees no key gets zeros.
 *   q, out      [total_q, num_q_heads, head_dim] of kv->dtype
 *   cu_q        int32 [batch + 1]
 *   tree_mask   uint64 [total_q] for SV_MASK_TREE, else NULL
 *   max_seq_len an upper bound of c_b + n_b (sizes the launch; a longer
 *               sequence sets SV_ERR_BAD_LENGTH and its rows are not written)
 *   workspace   device scratch of at least sv_spec_verify_attn_workspace_bytes,
 *               256-byte aligned; its contents need no initialisation
 *   status_dev  int32 [1] or NULL
 * Block ids outside [0, num_blocks) set SV_ERR_BAD_BLOCK_ID; the rows of that
 * sequence are then undefined, no out-of-bounds memory is touched.
 */
sv_status sv_spec_verify_attn(const sv_paged_kv *kv, const void *q, void *out, const int32_t *cu_q,
                              int32_t num_q_heads, int32_t total_q, int32_t max_q_per_seq,
                              int32_t max_seq_len, float scale, int32_t mask_kind, const uint64_t *tree_mask,
                              void *workspace, size_t workspace_bytes, int32_t *status_dev, void *stream);

/*
 * sv_spec_verify_attn_no_alloc -- sv_spec_verify_attn without a caller
 * workspace. The pages have no counterpart to this entry point; it exists for
 * callers that cannot allocate device memory around the attention call: an
 * engine that hands all free HBM to its KV block pool at start-up and has none
 * left to lend, or a host framework that owns the device allocator and
 * forbids a plug-in from calling cudaMalloc (which may also synchronise the
 * device in the middle of a step).
 *
 * Same arguments, semantics and status codes as sv_spec_verify_attn, minus
 * the workspace. The scratch is a static device array of
 * SV_ATTN_NO_ALLOC_SCRATCH_BYTES that every device loading the library holds
 * until the process exits. Sizes whose sv_spec_verify_attn_workspace_bytes
 * exceeds it return SV_ERR_WORKSPACE and launch nothing; that check comes
 * before any other CUDA runtime call of this entry point.
 *   - The first call on each device that launches work looks up the array's
 *     device address (with that device current; this may load the library's
 *     module there); make that first call before any stream capture.
 *   - Every call on a device uses the same array and leaves its contents
 *     behind; nothing in it needs to start at zero, since each value the
 *     kernels read was written earlier in the same call.
 *   - Calls whose kernels overlap on the GPU (other streams, other host
 *     threads) race on the array: order them on one stream or with events.
 * It allocates nothing: no cudaMalloc, no cudaFree, no allocating library call.
 */
#define SV_ATTN_NO_ALLOC_SCRATCH_BYTES ((size_t)16 << 20)
sv_status sv_spec_verify_attn_no_alloc(const sv_paged_kv *kv, const void *q, void *out, const int32_t *cu_q,
                                       int32_t num_q_heads, int32_t total_q, int32_t max_q_per_seq,
                                       int32_t max_seq_len, float scale, int32_t mask_kind,
                                       const uint64_t *tree_mask, int32_t *status_dev, void *stream);

/*
 * sv_spec_rejection_sample -- lossless verification of chain drafts.
 *
 * Target row cu_q[b] + i holds the logits of the position that draft token
 * x_{i+1} fills (row 0 scores x_1; row n_b-1 is the bonus position). With
 * temperature T > 0: p = softmax(l_target / T), q = softmax(l_draft / T) over
 * the vocabulary; for i = 0..K_b-1 (K_b = n_b - 1) x is accepted iff
 * u_accept < min(1, p(x)/q(x)) (q(x) == 0 counts as accept); a_b is the first
 * rejected i, or K_b. Then one token y is drawn by inverse CDF with
 * u_resample[b]: from norm(max(0, p_a - q_a)) when a_b < K_b (from p_a if that
 * residual has no mass), from p_K when every draft was accepted: y is the
 * smallest index whose inclusive prefix sum exceeds u_resample[b] times the
 * total mass. With T == 0 (greedy): x is accepted while it equals the target
 * argmax (lowest index on ties) and y is the argmax of row a_b; draft_logits,
 * u_accept and u_resample are not read and may be NULL.
 *   target_logits  [total_q, vocab] of logits_dtype (bf16 or f32)
 *   draft_logits   [total_q - batch, vocab]
 *   draft_tokens   int32 [total_q - batch]
 *   u_accept       float [total_q - batch], in [0, 1)
 *   u_resample     float [batch], in [0, 1)
 *   accept_count   int32 [batch] out: a_b
 *   out_tokens     int32 [batch, max_q_per_seq] out: x_1..x_a, y, then -1
 *   num_out        int32 [batch] out: a_b + 1
 *   margin         float [batch] out, or NULL: the smallest distance, over
 *                  the comparisons that decided the sequence, between a
 *                  uniform and the threshold it was compared with:
 *                  |u - min(1, p/q)| for each draft tested, and for the draw
 *                  the distance of u' from the chosen token's interval edges
 *                  on the normalised CDF (from the fixed-point sums; 0 when
 *                  rounding left no crossing); +inf at T = 0. Below 1e-4 it
 *                  marks a near-tie, where the fp32 decision may differ from
 *                  an exact one.
 *   workspace      device scratch of at least
 *                  sv_spec_rejection_sample_workspace_bytes(...) bytes,
 *                  256-byte aligned, owned by the caller; its contents need no
 *                  initialisation and are not kept between calls (per-row
 *                  partial softmax statistics: the statistics kernel writes
 *                  them, the decision kernel reads them). SV_ERR_WORKSPACE if
 *                  it is NULL, unaligned or too small.
 *   status_dev     int32 [1] or NULL: SV_ERR_NONFINITE for NaN/+inf logits,
 *                  SV_ERR_BAD_TOKEN for a draft token outside the vocabulary
 * Arithmetic is fp32; decisions equal the exact ones except when a uniform
 * lies within about 1e-6 of its threshold.
 */
sv_status sv_spec_rejection_sample(const void *target_logits, const void *draft_logits, int32_t logits_dtype,
                                   int32_t vocab, int32_t batch, const int32_t *cu_q, int32_t total_q,
                                   int32_t max_q_per_seq, const int32_t *draft_tokens, const float *u_accept,
                                   const float *u_resample, float temperature, int32_t *accept_count,
                                   int32_t *out_tokens, int32_t *num_out, float *margin, void *workspace,
                                   size_t workspace_bytes, int32_t *status_dev, void *stream);

/*
 * Workspace bytes of sv_spec_rejection_sample for these sizes (temperature 0:
 * greedy, target rows only; also the size for sv_tree_greedy_accept). It is
 * (rows) x ceil(vocab x element size / 32 KB) x 64 bytes, rows = total_q, plus
 * total_q - batch draft rows when temperature > 0. Returns 0 for invalid sizes
 * or types.
 */
size_t sv_spec_rejection_sample_workspace_bytes(int32_t logits_dtype, int32_t vocab, int32_t batch, int32_t total_q,
                                                float temperature);

/*
 * sv_tree_greedy_accept -- greedy verification of a draft tree (the tree mode
 * of the sampler). Row 0 of a sequence is the root; node row j >= 1 has parent
 * row parent[cu_q[b] + j] and token node_tokens[cu_q[b] - b + j - 1]. From the
 * root, move to the child (lowest row first) whose token equals the argmax of
 * the current node's target row, while there is one; y = argmax of the last
 * node's row.
 *   parent        int32 [total_q]: parent row within the sequence, -1 for row 0
 *   accept_count  int32 [batch] out: a_b, the accepted path length
 *   path_nodes    int32 [batch, max_q_per_seq] out: rows of the accepted
 *                 nodes in path order, then -1 (input of sv_kv_rollback)
 *   out_tokens    int32 [batch, max_q_per_seq] out: path tokens, y, then -1
 *   num_out       int32 [batch] out: a_b + 1
 *   workspace     as for sv_spec_rejection_sample, sized with temperature 0
 */
sv_status sv_tree_greedy_accept(const void *target_logits, int32_t logits_dtype, int32_t vocab, int32_t batch,
                                const int32_t *cu_q, int32_t total_q, int32_t max_q_per_seq,
                                const int32_t *node_tokens, const int32_t *parent, int32_t *accept_count,
                                int32_t *path_nodes, int32_t *out_tokens, int32_t *num_out, void *workspace,
                                size_t workspace_bytes, int32_t *status_dev, void *stream);

/*
 * sv_tree_rejection_sample -- lossless verification of a draft tree at
 * temperature T > 0 (T == 0: sv_tree_greedy_accept). The pages fix only the
 * greedy tree rule; the reading implemented: a node's children carry distinct
 * candidate tokens picked without sampling (the top-k of the draft at that
 * node), so each child is a proposal with all its mass on its token, which the
 * rejection rule accepts with probability p(x), leaving on rejection p with x
 * removed, renormalised. From the root, at node v (p_v = softmax(row v / T)):
 * children in row order; child c with token x is accepted iff
 * u_accept[cu_q[b] - b + c - 1] < p'(x), p' being p_v without the tokens of
 * the siblings rejected before (0 for a token already rejected); the first
 * accepted child becomes the current node. When no child is accepted, or v has
 * none, y is drawn by inverse CDF with u_resample[b] from p' (from p_v if the
 * rejected tokens held all its mass). Every emitted token is then distributed
 * as p at its position. Node rows are in BFS order (parent row < row), else
 * SV_ERR_BAD_LENGTH.
 *   arguments and outputs as sv_tree_greedy_accept, plus u_accept (float
 *   [total_q - batch]) and u_resample (float [batch]) in [0, 1), and margin
 *   (float [batch] out, or NULL) as for sv_spec_rejection_sample (each child
 *   tested against p'(x), then the draw; +inf at T = 0); the workspace is
 *   sized with sv_spec_rejection_sample_workspace_bytes(..., temperature 0)
 *   (target rows only); no draft logits are read.
 * Arithmetic as sv_spec_rejection_sample: p'(x) in fp32 from the row
 * statistics, the draw exact in 64-bit fixed point.
 */
sv_status sv_tree_rejection_sample(const void *target_logits, int32_t logits_dtype, int32_t vocab, int32_t batch,
                                   const int32_t *cu_q, int32_t total_q, int32_t max_q_per_seq,
                                   const int32_t *node_tokens, const int32_t *parent, const float *u_accept,
                                   const float *u_resample, float temperature, int32_t *accept_count,
                                   int32_t *path_nodes, int32_t *out_tokens, int32_t *num_out, float *margin,
                                   void *workspace, size_t workspace_bytes, int32_t *status_dev, void *stream);

/*
 * sv_kv_rollback -- keep each sequence's accepted prefix, give back the rest.
 *
 * The new length is c_b + a_b + 1: the last emitted token and the a_b
 * accepted rows keep their KV where it is; the resampled token has no KV yet.
 * With path_nodes (tree drafts), the accepted path's rows are first copied, in
 * path order, to logical positions c_b + 1 .. c_b + a_b. Blocks with logical
 * index >= ceil(new_len / bs) that held this step's rows are pushed on the
 * free list in sequence order, highest logical block first, and their block
 * table entries set to -1. seq_lens[b] becomes the new length.
 *   cu_q          int32 [batch + 1] (the step's rows, as given to sv_kv_append)
 *   accept_count  int32 [batch]: 0 <= a_b <= n_b - 1
 *   path_nodes    int32 [batch, max_q_per_seq] or NULL (chain drafts)
 *   status_dev    int32 [1], required
 * With ref_count, the count of each block given back drops by one and the
 * block is pushed only when it reaches zero (the blocks past the new end were
 * taken by this step's append, so they are the sequence's own).
 * All or nothing: an accept count or path entry out of range sets
 * SV_ERR_BAD_LENGTH and changes nothing.
 */
sv_status sv_kv_rollback(const sv_paged_kv *kv, const int32_t *cu_q, const int32_t *accept_count,
                         const int32_t *path_nodes, int32_t max_q_per_seq, int32_t *status_dev, void *stream);

/*
 * sv_kv_fork -- children share their parents' blocks (copy-on-write; requires
 * kv->ref_count).
 *
 * For pair k, sequence children[k] (an empty slot: length 0, no table entry)
 * takes the length of parents[k] and the ids of its ceil(len / bs) blocks; each
 * of those blocks' count goes up by one. Every pair sees the cache as it was
 * before the call: children are distinct and none is also a parent.
 *   parents, children  int32 [n_pairs], device
 *   status_dev         int32 [1], required; nothing happens while it holds an error
 * All or nothing: an id out of [0, batch), a child that is not empty, a
 * repeated child or a child that is also a parent sets SV_ERR_BAD_LENGTH; a
 * parent's block id out of range or with count < 1 sets SV_ERR_BAD_BLOCK_ID.
 * batch <= 65536.
 */
sv_status sv_kv_fork(const sv_paged_kv *kv, const int32_t *parents, const int32_t *children, int32_t n_pairs,
                     int32_t *status_dev, void *stream);

/*
 * sv_kv_release -- finished sequences give their blocks back.
 *
 * In the order listed, each sequence's blocks, highest logical block first,
 * lose one reference (without ref_count: every block) and are pushed on the
 * free list when their count reaches zero; the sequence's table entries become
 * -1 and its length 0. A block held only by listed sequences is therefore
 * pushed once, at the last listed sequence that holds it.
 *   seqs        int32 [n], device: distinct sequence ids
 *   status_dev  int32 [1], required; nothing happens while it holds an error
 * All or nothing: an id out of range or repeated sets SV_ERR_BAD_LENGTH; a
 * block id out of range or a count below the references being dropped sets
 * SV_ERR_BAD_BLOCK_ID; a free list that would overflow, SV_ERR_OUT_OF_BLOCKS.
 * batch <= 65536.
 */
sv_status sv_kv_release(const sv_paged_kv *kv, const int32_t *seqs, int32_t n, int32_t *status_dev, void *stream);

/*
 * Adaptive draft length: the host-side controller that picks each sequence's
 * K for the next step from its observed acceptance ("Speculative decoding
 * principles and a vLLM production setup", sec. 4.3, the sliding-window
 * controller; the same rule with a 10-step window and 80% / 50% thresholds is
 * the tuning advice of "LLM inference optimisation: speculative decoding and
 * dynamic batching", engineering parameters).
 *
 * Per sequence b the state holds K_b and the last `window` acceptance rates
 * alpha = accepted / max(drafted, 1). An update appends the step's alpha
 * (dropping the oldest once the window is full); when the window then holds
 * at least `min_samples` rates, their mean (summed oldest first, in double)
 * moves K_b up by one if it is above up_threshold, down by one if it is below
 * down_threshold, within [k_min, k_max]. K_b starts at k_init.
 *
 * Every pointer here is a HOST pointer; nothing touches the GPU. The state is
 * caller-owned memory of sv_adaptive_k_state_bytes bytes, 8-byte aligned,
 * opaque, written only by these calls; one state must not be used by two host
 * threads at once.
 *   params        k_min >= 0, k_min <= k_init <= k_max <= 63 (K + 1 rows must
 *                 fit max_q_per_seq <= 64), window >= 1, min_samples >= 1
 *                 (a min_samples above window never moves K, as the sample
 *                 controller's rule gives), finite thresholds
 *   accepted      int32 [batch]: a_b of the step, 0 <= a_b <= drafted_b
 *   drafted       int32 [batch]: K_b of the step, >= 0
 *   k_next        int32 [batch] out (may be NULL): K_b for the next step
 * All or nothing: invalid arguments return SV_ERR_INVALID_ARG and leave the
 * state unchanged.
 */
typedef struct sv_adaptive_k_params {
  int32_t k_min, k_max, k_init;
  int32_t window, min_samples;
  double up_threshold, down_threshold;
} sv_adaptive_k_params;

/* Bytes of state for `batch` sequences and this window; 0 for invalid sizes. */
size_t sv_adaptive_k_state_bytes(int32_t batch, int32_t window);
sv_status sv_adaptive_k_init(void *state, size_t state_bytes, int32_t batch, const sv_adaptive_k_params *params);
sv_status sv_adaptive_k_update(void *state, const int32_t *accepted, const int32_t *drafted, int32_t *k_next);
/* Sequence slot `seq` starts over (a new request took it): K = k_init, empty window. */
sv_status sv_adaptive_k_reset(void *state, int32_t seq);
/* The current K of every sequence into k (int32 [batch]). */
sv_status sv_adaptive_k_current(const void *state, int32_t *k);

/*
 * Process-wide options (no counterpart on the pages; they select between
 * complete implementations of the same operation, for measurement, and set
 * the failure-detection limits).
 *   SV_OPT_ATTN_PATH:
 *     SV_ATTN_AUTO (default): 5th-generation tensor cores (tcgen05, TMEM) for
 *       bf16 and E4M3 caches with head_dim 128 and blocks of 16..256 tokens
 *       (the query-major kernel), CUDA cores for every other shape;
 *     SV_ATTN_CUDA_CORES: the CUDA-core kernel for every shape;
 *     SV_ATTN_TENSOR_CORES: tcgen05 (an unsupported shape then returns
 *       SV_ERR_UNSUPPORTED from sv_spec_verify_attn);
 *     SV_ATTN_WARP_MMA: warp-level mma.sync tensor-core kernel (the bf16
 *       shapes of tcgen05);
 *     SV_ATTN_KEYS_MAJOR: the keys-major tcgen05 kernel (S^T = K Q^T with keys
 *       on the MMA's M dimension; units of at most 32 query rows, i.e. query
 *       heads per KV head x max_q_per_seq <= 32; bf16 caches), else
 *       SV_ERR_UNSUPPORTED. SV_ATTN_TENSOR_CORES is the query-major one.
 *   SV_OPT_WAIT_BUDGET_US (value in microseconds, 1000 .. 2000000; default
 *     500000): how long a pipeline wait (a consumer waiting for the data its
 *     producer brings, a producer waiting for a free stage) of the tcgen05
 *     attention kernels and of the sampler's statistics kernel may take before
 *     the kernel gives up, records SV_ERR_TIMEOUT in the status word and ends.
 *     A kernel that gives up still waits for the copies and matrix operations
 *     it has issued (at most 0.5 s each, whatever this option says) before it
 *     releases its shared memory and tensor memory, so that nothing lands in
 *     memory it no longer owns. The mma.sync attention kernel
 *     (SV_ATTN_WARP_MMA) keeps 0.5 s for every wait. A budget shorter than the
 *     time the memory system needs to deliver a stage makes healthy calls
 *     fail, hence the 1 ms floor.
 *   SV_OPT_STALL_FOR_TEST (SV_STALL_NONE, the default; SV_STALL_ATTENTION;
 *     SV_STALL_SAMPLER): for tests of the failure path only. The producer warp
 *     of the tensor-core attention kernel, or of the sampler's statistics
 *     kernel, first waits on a barrier that nothing ever completes, as a
 *     producer whose data never arrives would; that wait runs out after the
 *     wait budget, the producer issues nothing, and every pipeline wait of its
 *     consumers runs out in turn. The call then records SV_ERR_TIMEOUT and its
 *     outputs are undefined; it faults and traps nothing.
 * Returns SV_ERR_INVALID_ARG for an unknown option or value. Not thread-safe
 * with respect to calls in flight on other host threads.
 */
typedef enum sv_option { SV_OPT_ATTN_PATH = 1, SV_OPT_WAIT_BUDGET_US = 2, SV_OPT_STALL_FOR_TEST = 3 } sv_option;
typedef enum sv_stall { SV_STALL_NONE = 0, SV_STALL_ATTENTION = 1, SV_STALL_SAMPLER = 2 } sv_stall;
typedef enum sv_attn_path {
  SV_ATTN_AUTO = 0,
  SV_ATTN_CUDA_CORES = 1,
  SV_ATTN_TENSOR_CORES = 2,
  SV_ATTN_WARP_MMA = 3,
  SV_ATTN_KEYS_MAJOR = 4
} sv_attn_path;
sv_status sv_set_option(int32_t option, int32_t value);

/* A static, human-readable name of a status code. */
const char *sv_status_string(int32_t status);

/* Version of this ABI (major * 10000 + minor * 100 + patch). */
int32_t sv_version(void);

#ifdef __cplusplus
}
#endif

#endif /* SPEC_VERIFY_H */
