/*
 * dcp.h -- C ABI of libdcp.so, the GB300 (sm_103a) hot path of Decode
 * Context Parallelism (DCP): the KV cache of every request is sharded along
 * the sequence over dcp_size ranks with the interleaved layout, each rank
 * attends its own shard and emits a partial output plus a log-sum-exp
 * (LSE), and the partials are merged exactly by LSE.
 *
 * All dcp_size ranks are "virtual": they are separate per-rank buffers on
 * the one GPU the caller's stream runs on.  No call communicates.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Every pointer is DEVICE memory owned by the caller, unless a comment
 *    says otherwise.  The library allocates no device memory and keeps no
 *    state between calls except a per-device cache of the SM count and of
 *    driver entry points.
 *  - Every call is asynchronous on `stream` (NULL = legacy default stream)
 *    and never synchronises.  Results are valid once the stream reaches
 *    the call.
 *  - Return value: DCP_OK, or a negative code (see dcp_strerror):
 *      DCP_EINVAL       bad layout or argument (checked on the host before
 *                       anything is launched; nothing is written);
 *      DCP_EWORKSPACE   workspace pointer NULL or smaller than
 *                       dcp_decode_workspace_size() asks for;
 *      DCP_EUNSUPPORTED a shape or dtype this build has no kernel for;
 *      DCP_ECUDA        a launch or driver call failed (cudaGetLastError).
 *  - Data errors found on the device (an index out of range, a block-table
 *    entry outside [0, num_blocks), a virtual block beyond max_vblocks)
 *    never trap: the offending entry becomes -1 or is skipped, and if
 *    `err_count` is not NULL the kernel atomically adds 1 to *err_count per
 *    bad entry.
 *  - Layouts are row-major, dimensions listed outermost first.
 *
 * KV-cache layout -- page "Decode Context Parallel (DCP)" (docs.vllm.ai,
 * vLLM Ascend design documents), section "KV-cache layout": a virtual
 * block holds block_size*dcp_size tokens and token x goes to
 *     virtual_block_index     = x / (block_size*dcp_size)
 *     offset_in_virtual_block = x % (block_size*dcp_size)
 *     local_block_index       = offset_in_virtual_block / interleave
 *     target_rank             = local_block_index % dcp_size
 * with block_size % interleave == 0.  The pages do not print where inside
 * the rank's block the token lands; this library reads it as
 *     local_offset = (local_block_index / dcp_size)*interleave
 *                    + offset_in_virtual_block % interleave
 * so each rank fills one block_size-token physical block per virtual block,
 * in increasing token order, and the token's slot on its rank is
 *     slot = block_table[rank][req][virtual_block_index]*block_size + local_offset.
 */
#ifndef DCP_H_
#define DCP_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st;
/* Same type as cudaStream_t. */
typedef struct CUstream_st* dcp_stream_t;

#define DCP_MAX_RANKS 16

enum {
  DCP_OK = 0,
  DCP_EINVAL = -1,
  DCP_EWORKSPACE = -2,
  DCP_ECUDA = -3,
  DCP_EUNSUPPORTED = -4
};

typedef enum { DCP_F32 = 0, DCP_BF16 = 1 } dcp_dtype_t;

/* Attention family, for dcp_decode_workspace_size. */
typedef enum { DCP_KIND_GQA = 0, DCP_KIND_MLA = 1, DCP_KIND_SFA = 2 } dcp_kind_t;

typedef struct {
  int32_t dcp_size;   /* ranks, 1..DCP_MAX_RANKS                          */
  int32_t block_size; /* tokens per physical KV block, >= 1               */
  int32_t interleave; /* cp_kv_cache_interleave_size, >= 1, divides block_size */
} dcp_layout_t;

/* One device pointer per rank; entries >= dcp_size are ignored. */
typedef struct {
  void* ptr[DCP_MAX_RANKS];
} dcp_rank_ptrs_t;

/*
 * The paged, sequence-sharded KV cache as the decode kernels read it.
 *  k, v        per-rank pools.  GQA: k and v are [num_blocks][num_kv_heads]
 *              [block_size][head_dim] ("HND": one (block, head) page is
 *              contiguous).  MLA / SFA: k is the latent pool
 *              [num_blocks][block_size][kv_dim]; v is ignored (the value is
 *              the first v_dim entries of each latent row).
 *  num_blocks  physical blocks in each rank's pool.
 *  block_table [dcp_size][num_reqs][max_vblocks] int32 physical block of
 *              virtual block vb of request b on rank r, at
 *              block_table[r*bt_rank_stride + b*max_vblocks + vb];
 *              bt_rank_stride == 0 means every rank uses the same table.
 */
typedef struct {
  dcp_rank_ptrs_t k;
  dcp_rank_ptrs_t v;
  int64_t num_blocks;
  const int32_t* block_table;
  int32_t max_vblocks;
  int64_t bt_rank_stride;
} dcp_paged_kv_t;

/* Text for a return code (static storage; never NULL). */
const char* dcp_strerror(int code);

/* Library version, e.g. 100 for 0.1.0. */
int dcp_version(void);

/*
 * dcp_local_seq_lens -- the per-rank context-length matrix that the page
 * "Decode Context Parallel (DCP)", section "Backend structure", assigns to
 * the DCP metadata builder: local_lens[b][r] = number of tokens x <
 * seq_lens[b] with target_rank(x) == r.
 *  seq_lens   [num_reqs] int32, each >= 0 (negative counts as 0 and bumps
 *             err_count).  A length counts the decode token itself.
 *  local_lens [num_reqs][dcp_size] int32 output.
 */
int dcp_local_seq_lens(dcp_layout_t layout, const int32_t* seq_lens, int32_t num_reqs,
                       int32_t* local_lens, int32_t* err_count, dcp_stream_t stream);

/*
 * dcp_slot_mapping -- token -> (owner rank, slot on every rank), page
 * "Decode Context Parallel (DCP)", section "KV-cache layout" (the slot
 * mapping uses the layout so each rank stores only its local shard) and
 * page "DeepSeek V4.1 context parallelism" (lightseek.org), section "Cache
 * ownership" (writes translate virtual slots to local slots and mask
 * non-owners).
 *  req_idx   [num_tokens] int32 request of each token.
 *  positions [num_tokens] int64 global position x of each token.
 *  out_rank  [num_tokens] int32 owner rank, -1 for an invalid token.
 *  out_slot  [dcp_size][num_tokens] int64 slot of the token on rank r if r
 *            owns it, else -1.
 * A token is invalid (rank -1, all slots -1, err_count += 1) when its
 * request is outside [0, num_reqs), its position is negative, its virtual
 * block is >= max_vblocks or its block-table entry is outside
 * [0, num_blocks).
 */
int dcp_slot_mapping(dcp_layout_t layout, const int32_t* req_idx, const int64_t* positions,
                     int64_t num_tokens, const int32_t* block_table, int32_t num_reqs,
                     int32_t max_vblocks, int64_t bt_rank_stride, int64_t num_blocks,
                     int32_t* out_rank, int64_t* out_slot, int32_t* err_count,
                     dcp_stream_t stream);

/*
 * dcp_cache_write_gqa -- owner-masked reshape-and-cache (page "DeepSeek
 * V4.1 context parallelism", section "Cache ownership"): every rank sees
 * every token's write; only the owner (slot[r][t] >= 0) stores it.
 *  k, v      [num_tokens][num_kv_heads][head_dim] of `dtype`.
 *  slot      [dcp_size][num_tokens] int64 from dcp_slot_mapping.
 *  k_cache, v_cache per-rank pools [num_blocks][num_kv_heads][block_size][head_dim].
 * Bytes are copied unchanged.  A slot outside [-1, num_blocks*block_size)
 * is skipped and counted in err_count.
 */
int dcp_cache_write_gqa(dcp_layout_t layout, const void* k, const void* v, int64_t num_tokens,
                        int32_t num_kv_heads, int32_t head_dim, dcp_dtype_t dtype,
                        const int64_t* slot, int64_t num_blocks, dcp_rank_ptrs_t k_cache,
                        dcp_rank_ptrs_t v_cache, int32_t* err_count, dcp_stream_t stream);

/*
 * dcp_cache_write_mla -- the same for a latent cache: kv [num_tokens][kv_dim]
 * (for MLA the 512 latent entries followed by the 64 rope entries) into the
 * per-rank pools [num_blocks][block_size][kv_dim].  kv_dim*element size must
 * be a multiple of 16 bytes.
 */
int dcp_cache_write_mla(dcp_layout_t layout, const void* kv, int64_t num_tokens, int32_t kv_dim,
                        dcp_dtype_t dtype, const int64_t* slot, int64_t num_blocks,
                        dcp_rank_ptrs_t cache, int32_t* err_count, dcp_stream_t stream);

/*
 * dcp_gather_context_mla -- read tokens back out of the sharded latent cache
 * in the order given, page "Decode Context Parallel (DCP)", section "Prefill
 * and chunked prefill" (MLA gathers the context KV cache and restores
 * request-contiguous order before attending it).  Passing every position
 * 0..L_b-1 of request b, in order, restores that request's contiguous
 * context.
 *  kv          latent pools [num_blocks][block_size][kv_dim] + block table
 *              (kv.v is ignored).
 *  req_idx     [num_tokens] int32, positions [num_tokens] int64.
 *  out         [num_tokens][kv_dim] of dtype: bytes copied unchanged.
 * A token that does not resolve to a stored slot (request outside
 * [0, num_reqs), negative position, virtual block beyond the table, table
 * entry outside [0, num_blocks)) gets a zero row and bumps err_count.
 * kv_dim * element size must be a multiple of 16 bytes.
 */
int dcp_gather_context_mla(dcp_layout_t layout, dcp_paged_kv_t kv, int32_t num_reqs,
                           int32_t kv_dim, dcp_dtype_t dtype, const int32_t* req_idx,
                           const int64_t* positions, int64_t num_tokens, void* out,
                           int32_t* err_count, dcp_stream_t stream);

/*
 * dcp_decode_workspace_size -- bytes of device workspace the decode calls
 * below need for a batch of this shape (an upper bound that holds for any
 * context lengths).  The caller allocates it; its contents need not be
 * initialised and are garbage afterwards.
 *  head_dim_v  value width (GQA head_dim; 512 for MLA / SFA).
 * For DCP_KIND_SFA this includes 16 KB per request for the remapped
 * (rank, slot) pairs of up to 2048 selected tokens.
 */
int dcp_decode_workspace_size(dcp_layout_t layout, dcp_kind_t kind, int32_t num_reqs,
                              int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim_v,
                              size_t* bytes);

/*
 * dcp_decode_partial_gqa -- per-rank partial decode attention for GQA,
 * pages "Decode Context Parallel (DCP)", section "Decode" (each rank
 * attends its local KV shard and produces partial outputs and LSE values)
 * and the vLLM DCP blog post, section 5.4 (KV heads broadcast to their
 * query heads).  One decode query per request; query head h reads KV head
 * h / (num_q_heads / num_kv_heads).
 *  q          [num_reqs][num_q_heads][head_dim] of `dtype` (shared by all
 *             ranks: the Q-head gather is one buffer on one GPU).
 *  local_lens [num_reqs][dcp_size] int32 (dcp_local_seq_lens): rank r
 *             attends local positions [0, local_lens[b][r]) of request b.
 *  part_o     [dcp_size][num_reqs][num_q_heads][head_dim] float32:
 *             o_r = sum_j exp(s_j - lse_r) v_j over rank r's tokens.
 *  part_lse   [dcp_size][num_reqs][num_q_heads] float32:
 *             lse_r = ln sum_j exp(s_j), s_j = scale * q.k_j.
 *             A rank with no tokens gives lse_r = -inf and o_r = 0.
 * Long shards are split into chunks internally (split-KV) and combined
 * before the call returns its per-rank result.
 * Supported: dtype F32 or BF16, head_dim a multiple of 32 up to 256,
 * num_q_heads % num_kv_heads == 0, num_q_heads/num_kv_heads <= 16.
 */
int dcp_decode_partial_gqa(dcp_layout_t layout, const void* q, int32_t num_reqs,
                           int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                           float scale, dcp_dtype_t dtype, dcp_paged_kv_t kv,
                           const int32_t* local_lens, float* part_o, float* part_lse,
                           void* workspace, size_t workspace_bytes, int32_t* err_count,
                           dcp_stream_t stream);

/*
 * dcp_lse_merge -- exact merge of partial attention results, pages
 * "Decode Context Parallel (DCP)", section "Backend structure" (the common
 * partial-output/LSE merge) and "DeepSeek V4.1 context parallelism",
 * section "Decode computation" (the attention sink is applied once when
 * the partials are merged by log-sum-exp):
 *     lse = ln( sum_i exp(lse_i) + exp(sink[h]) ),
 *     o   = sum_i exp(lse_i - lse) * o_i.
 *  part_o   [num_parts][num_reqs][num_heads][head_dim_v] float32.
 *  part_lse [num_parts][num_reqs][num_heads] float32 (-inf = empty part).
 *  sink     [num_heads] float32 logits in scaled-score units, or NULL.
 *  out      [num_reqs][num_heads][head_dim_v] of out_dtype (bf16 is
 *           rounded to nearest even from float32).
 *  out_lse  [num_reqs][num_heads] float32, or NULL.
 * If every part is empty and there is no sink, o = 0 and lse = -inf.
 * head_dim_v must be a multiple of 4, at most 1024.
 */
int dcp_lse_merge(int32_t num_parts, const float* part_o, const float* part_lse,
                  int32_t num_reqs, int32_t num_heads, int32_t head_dim_v, const float* sink,
                  void* out, dcp_dtype_t out_dtype, float* out_lse, dcp_stream_t stream);

/*
 * dcp_lse_merge_swa -- dcp_lse_merge with one more part: the partial of a
 * sliding-window (SWA) KV set that every rank holds in full.  Page
 * "DeepSeek V4.1 context parallelism", section "Decode computation":
 * replicated SWA contributes on one rank, and the sink is applied once when
 * the partials are merged by log-sum-exp.  The window partial is therefore
 * merged exactly once, next to the num_parts per-rank partials:
 *     lse = ln( sum_i exp(lse_i) + exp(swa_lse) + exp(sink[h]) ).
 *  swa_o   [num_reqs][num_heads][head_dim_v] float32, swa_lse
 *          [num_reqs][num_heads] float32 (-inf = empty window), e.g. from
 *          dcp_decode_partial_gqa with dcp_size 1 over the window cache.
 * Other arguments as for dcp_lse_merge.
 */
int dcp_lse_merge_swa(int32_t num_parts, const float* part_o, const float* part_lse,
                      const float* swa_o, const float* swa_lse, int32_t num_reqs,
                      int32_t num_heads, int32_t head_dim_v, const float* sink, void* out,
                      dcp_dtype_t out_dtype, float* out_lse, dcp_stream_t stream);

/*
 * dcp_decode_gqa -- the fused decode step: per-rank split-KV partials and
 * one merge over (rank x split) with the optional sink, giving the same
 * result as dcp_decode_partial_gqa followed by dcp_lse_merge.
 * Arguments as in those two calls; out is [num_reqs][num_q_heads][head_dim]
 * of out_dtype, out_lse [num_reqs][num_q_heads] float32 or NULL.
 */
int dcp_decode_gqa(dcp_layout_t layout, const void* q, int32_t num_reqs, int32_t num_q_heads,
                   int32_t num_kv_heads, int32_t head_dim, float scale, dcp_dtype_t dtype,
                   dcp_paged_kv_t kv, const int32_t* local_lens, const float* sink, void* out,
                   dcp_dtype_t out_dtype, float* out_lse, void* workspace,
                   size_t workspace_bytes, int32_t* err_count, dcp_stream_t stream);

/*
 * dcp_decode_gqa_noalloc -- dcp_decode_gqa without a caller workspace.  The
 * pages have no counterpart: this entry point exists for callers that cannot
 * allocate device memory when they decode (a runtime that owns all device
 * memory and gives the library none, code running under a fixed memory
 * budget, or a C caller with no device allocator).  The split-KV workspace
 * comes from a fixed 16 MiB array inside the library's own device memory.
 * Arguments and results are those of dcp_decode_gqa.
 *  - Returns DCP_EWORKSPACE, launching nothing, when the batch needs more
 *    than 16 MiB of workspace (dcp_decode_workspace_size tells in advance).
 *  - The array is reserved on a device by the first call made there (the
 *    library's device code loads lazily); the device then holds it until the
 *    process exits.  That first call returns DCP_ECUDA if the 16 MiB cannot
 *    be reserved.  Make it before any stream capture, as a warm-up.
 *  - The array's device address is looked up with that device current and
 *    cached with the id of the CUDA context it was found in; a call made in
 *    another context (after cudaDeviceReset, or under a context the caller
 *    created) looks it up again.
 *  - Every call on a device uses the same array: calls that overlap on the
 *    GPU (different streams, concurrent graphs) race and corrupt each
 *    other's results.  Calls in one stream order are safe.  The array keeps
 *    the last call's contents; each call rewrites every counter it reads
 *    (in stream order, before its kernels use them), so nothing needs
 *    clearing between calls.
 *  - Allocates nothing: no cudaMalloc, no cudaFree.
 */
int dcp_decode_gqa_noalloc(dcp_layout_t layout, const void* q, int32_t num_reqs,
                           int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                           float scale, dcp_dtype_t dtype, dcp_paged_kv_t kv,
                           const int32_t* local_lens, const float* sink, void* out,
                           dcp_dtype_t out_dtype, float* out_lse, int32_t* err_count,
                           dcp_stream_t stream);

/*
 * dcp_decode_partial_mla -- per-rank partial decode attention for MLA
 * (vLLM DCP blog post, section 1: one latent KV head shared by every query
 * head, which tensor parallelism cannot split, so DCP splits it by
 * sequence).  Key = the whole latent row (kv_dim = 512 + 64 rope),
 * value = its first v_dim (512) entries.
 *  q        [num_reqs][num_q_heads][kv_dim] of dtype (the query already
 *           projected into the latent space).
 *  part_o   [dcp_size][num_reqs][num_q_heads][v_dim] float32, part_lse
 *           [dcp_size][num_reqs][num_q_heads] float32, as for GQA.
 * Supported: BF16 or F32 latent with kv_dim a multiple of 32 up to 1024 and
 * v_dim <= kv_dim, a multiple of 32.  BF16 with kv_dim 576, v_dim 512 and
 * num_q_heads 128 runs on the tcgen05 tensor-core kernel; other shapes run
 * a CUDA-core kernel.
 */
int dcp_decode_partial_mla(dcp_layout_t layout, const void* q, int32_t num_reqs,
                           int32_t num_q_heads, int32_t kv_dim, int32_t v_dim, float scale,
                           dcp_dtype_t dtype, dcp_paged_kv_t kv, const int32_t* local_lens,
                           float* part_o, float* part_lse, void* workspace,
                           size_t workspace_bytes, int32_t* err_count, dcp_stream_t stream);

/* dcp_decode_mla -- fused MLA decode step (partials + merge + optional sink). */
int dcp_decode_mla(dcp_layout_t layout, const void* q, int32_t num_reqs, int32_t num_q_heads,
                   int32_t kv_dim, int32_t v_dim, float scale, dcp_dtype_t dtype,
                   dcp_paged_kv_t kv, const int32_t* local_lens, const float* sink, void* out,
                   dcp_dtype_t out_dtype, float* out_lse, void* workspace,
                   size_t workspace_bytes, int32_t* err_count, dcp_stream_t stream);

/*
 * dcp_sfa_remap -- page "Decode Context Parallel (DCP)", section "GLM-5.2
 * SFA DCP replicated indexer": top-k token indices chosen on the
 * replicated full-sequence indexer view are remapped to local KV indices
 * before sparse attention runs.
 *  topk     [num_reqs][topk_len] int32 global token indices.
 *  seq_lens [num_reqs] int32.
 *  out_rank [num_reqs][topk_len] int32 owner rank of each index.
 *  out_slot [num_reqs][topk_len] int32 slot on that rank.
 * An index < 0 or >= seq_lens[b] gives (-1, -1) (not an error: padding);
 * a virtual block beyond max_vblocks or a table entry outside
 * [0, num_blocks) gives (-1, -1) and bumps err_count.
 * num_blocks*block_size must be < 2^31.
 */
int dcp_sfa_remap(dcp_layout_t layout, const int32_t* topk, int32_t num_reqs, int32_t topk_len,
                  const int32_t* seq_lens, const int32_t* block_table, int32_t max_vblocks,
                  int64_t bt_rank_stride, int64_t num_blocks, int32_t* out_rank,
                  int32_t* out_slot, int32_t* err_count, dcp_stream_t stream);

/*
 * Exact distributed top-k -- page "DeepSeek V4.1 context parallelism",
 * section "Decode computation": every rank computes local top-k candidates
 * over the tokens it owns and the scores and logical ids are merged across
 * ranks, which selects exactly the global top-k.  Rule (the page names
 * none): a higher score ranks first, equal scores rank the smaller logical
 * (global) token id first, NaN counts as -inf, -0 equals +0 (reported
 * scores: NaN as -inf, -0 as +0).
 *
 * dcp_topk_local
 *  local_scores [dcp_size][num_reqs][max_local] float32: score of local
 *               position p of request b on rank r (read for p < local_lens[b][r]).
 *  local_lens   [num_reqs][dcp_size] int32 (dcp_local_seq_lens).
 *  cand_keys    [dcp_size][num_reqs][k] uint64 candidates, best first:
 *               key = (order(score) << 32) | (0xFFFFFFFF - id) with order()
 *               the monotone map of float32 onto uint32; 0 = no candidate.
 * dcp_topk_merge
 *  out_ids      [num_reqs][k] int32 global token ids, best first (-1 when a
 *               request has fewer than k tokens).
 *  out_scores   [num_reqs][k] float32 (NULL allowed; -inf past the end).
 *  workspace    num_reqs*k*8 bytes.
 * dcp_topk     both steps; workspace dcp_topk_workspace_size bytes.
 * 1 <= k <= 4096.
 */
int dcp_topk_workspace_size(dcp_layout_t layout, int32_t num_reqs, int32_t k, size_t* bytes);
int dcp_topk_local(dcp_layout_t layout, const float* local_scores, int32_t num_reqs,
                   int32_t max_local, const int32_t* local_lens, int32_t k, uint64_t* cand_keys,
                   dcp_stream_t stream);
int dcp_topk_merge(int32_t dcp_size, const uint64_t* cand_keys, int32_t num_reqs, int32_t k,
                   void* workspace, size_t workspace_bytes, int32_t* out_ids, float* out_scores,
                   dcp_stream_t stream);
int dcp_topk(dcp_layout_t layout, const float* local_scores, int32_t num_reqs, int32_t max_local,
             const int32_t* local_lens, int32_t k, int32_t* out_ids, float* out_scores,
             void* workspace, size_t workspace_bytes, dcp_stream_t stream);

/*
 * dcp_sfa_compact_workspace_size -- bytes of workspace dcp_sfa_compact_blocks
 * needs for pools of num_blocks physical blocks per rank.
 */
int dcp_sfa_compact_workspace_size(dcp_layout_t layout, int64_t num_blocks, size_t* bytes);

/*
 * dcp_sfa_compact_blocks -- page "Decode Context Parallel (DCP)", section
 * "GLM-5.2 SFA DCP replicated indexer": during prefill or a mixed batch only
 * the KV blocks referenced by the sparse block table are compacted (and then
 * all-gathered after the layer writes its KV cache).  This is the one-GPU
 * part: every rank's physical blocks that some selected token of some query
 * refers to are numbered (ranks in order, increasing block id within a
 * rank), copied into one buffer, and every selected token is rewritten as a
 * row of that buffer.
 *  topk       [num_queries][topk_len] int32 global token ids (index < 0 or
 *             >= seq_lens[q_req[q]] is padding: skipped, index -1).
 *  q_req      [num_queries] int32 request of each query.
 *  kv         latent pools [num_blocks][block_size][kv_dim] + block table.
 *  out_blocks [max_blocks][block_size][kv_dim] of dtype: the compacted blocks.
 *  out_block_ids [max_blocks] int32 physical id of each compacted block.
 *  out_counts [dcp_size] int32 compacted blocks of each rank (their sum may
 *             exceed max_blocks: blocks past the capacity are not stored and
 *             the tokens in them get index -1 and bump err_count).
 *  out_index  [num_queries][topk_len] int64 row of each selected token in
 *             out_blocks viewed as [max_blocks*block_size][kv_dim], or -1.
 *  workspace  dcp_sfa_compact_workspace_size bytes (contents not needed).
 * A table entry outside [0, num_blocks) gives -1 and bumps err_count.
 */
int dcp_sfa_compact_blocks(dcp_layout_t layout, const int32_t* topk, const int32_t* q_req,
                           int32_t num_queries, int32_t topk_len, const int32_t* seq_lens,
                           int32_t num_reqs, dcp_paged_kv_t kv, int32_t kv_dim, dcp_dtype_t dtype,
                           int64_t max_blocks, void* out_blocks, int32_t* out_block_ids,
                           int32_t* out_counts, int64_t* out_index, void* workspace,
                           size_t workspace_bytes, int32_t* err_count, dcp_stream_t stream);

/*
 * dcp_sfa_decode_partial -- per-rank sparse attention over the selected
 * tokens each rank owns (section "GLM-5.2 SFA DCP replicated indexer":
 * decode-only batches keep the Q-gather and result-merge path).  Latent
 * cache as for MLA (kv.k, kv.num_blocks; the block table is not read).
 *  sel_rank, sel_slot [num_reqs][topk_len] from dcp_sfa_remap; entries
 *           with rank -1 are skipped.
 *  part_o   [dcp_size][num_reqs][num_q_heads][v_dim] float32, part_lse
 *           [dcp_size][num_reqs][num_q_heads] float32 (rank with no
 *           selected token: -inf and 0).
 * Supported: dtype BF16 or F32, kv_dim/v_dim multiples of 32 up to 1024.
 */
int dcp_sfa_decode_partial(dcp_layout_t layout, const void* q, int32_t num_reqs,
                           int32_t num_q_heads, int32_t kv_dim, int32_t v_dim, float scale,
                           dcp_dtype_t dtype, dcp_paged_kv_t kv, const int32_t* sel_rank,
                           const int32_t* sel_slot, int32_t topk_len, float* part_o,
                           float* part_lse, int32_t* err_count, dcp_stream_t stream);

/*
 * dcp_sfa_decode -- the fused SFA decode step: remap, per-rank sparse
 * partials and the merge with the optional sink applied once.
 *  topk, seq_lens as for dcp_sfa_remap; the block table is kv.block_table.
 *  out [num_reqs][num_q_heads][v_dim] of out_dtype; out_lse may be NULL.
 */
int dcp_sfa_decode(dcp_layout_t layout, const void* q, int32_t num_reqs, int32_t num_q_heads,
                   int32_t kv_dim, int32_t v_dim, float scale, dcp_dtype_t dtype,
                   dcp_paged_kv_t kv, const int32_t* topk, int32_t topk_len,
                   const int32_t* seq_lens, const float* sink, void* out,
                   dcp_dtype_t out_dtype, float* out_lse, void* workspace,
                   size_t workspace_bytes, int32_t* err_count, dcp_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* DCP_H_ */
