/*
 * pa.h: C ABI of the paged KV-cache hot path (store, paged decode, varlen prefill) for one
 * NVIDIA GB300 (sm_103a).
 *
 * The three operations are the attention layer's GPU work in the engines that the
 * "nano-vLLM Part 4" page (section 3, the prefill/decode table and the per-rank tensor list)
 * and the smzdm nano-vLLM deep dive ("模型实现细节": store_kvcache, flash_attn_varlen_func,
 * flash_attn_with_kvcache, the prefix-cache rule) describe, and that the "mini-vLLM" page
 * describes for its 16-token paged pool with grouped-query attention.
 *
 * Conventions shared by every call
 * --------------------------------
 * - Pointers are DEVICE pointers unless a comment says otherwise. The caller owns every
 *   buffer. The library allocates nothing that outlives a call. Nothing is freed by the library.
 * - Every call is asynchronous on `stream`; it returns after the launch. Errors that the host
 *   can see are returned before anything is launched, and nothing is written then.
 * - Element types: `pa_dtype` selects fp16 or bf16 for q, k, v, the pools and the output.
 *   Scores, softmax and accumulation run in fp32; the output is rounded once (to nearest even).
 * - Pools: `k_cache` and `v_cache` are each [num_blocks, block_size, Hkv, D], contiguous.
 *   Token slot `s` (0 <= s < num_blocks * block_size) is block `s / block_size`, offset
 *   `s % block_size`; its K row for kv head g starts at element (s * Hkv + g) * D.
 * - Block tables: int32 [rows, max_blocks_per_seq], row-major; entry b of a row is the physical
 *   block holding that sequence's positions b*block_size .. b*block_size + block_size - 1.
 *   Only the first ceil(length / block_size) entries of a row are read; the rest may hold
 *   anything (the workloads use -1).
 * - Grouped-query heads: query head h reads kv head h / (Hq / Hkv).
 * - Alignment: every tensor pointer must be 16-byte aligned (torch allocations are).
 * - Supported: D = 64 or 128 (pa_store_kv: any D with D % 8 == 0); 1 <= Hq / Hkv <= 8 with
 *   Hq % Hkv == 0; any block_size >= 1.
 * - `err` (nullable, device int32): data-dependent problems that only the GPU sees are OR-ed
 *   into *err as PA_DEVERR_* bits and the offending item is skipped, with every memory
 *   access kept in bounds. The library never traps and never clears *err: zero it before the call if you
 *   want to read it afterwards.
 */
#ifndef PA_H
#define PA_H

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    PA_OK = 0,
    PA_ERR_NULL = 1,        /* a required pointer is NULL */
    PA_ERR_SHAPE = 2,       /* a size is negative, zero where it must not be, or inconsistent */
    PA_ERR_DTYPE = 3,       /* dtype is not PA_F16 or PA_BF16 */
    PA_ERR_UNSUPPORTED = 4, /* a shape outside the supported set (D, group size, alignment) */
    PA_ERR_WORKSPACE = 5,   /* workspace missing or smaller than pa_decode_workspace_size() */
    PA_ERR_CUDA = 6         /* a CUDA runtime call failed (e.g. the launch) */
} pa_status;

typedef enum { PA_F16 = 0, PA_BF16 = 1 } pa_dtype;

/* Bits OR-ed into *err by the kernels. */
#define PA_DEVERR_SLOT 1   /* slot_mapping entry >= num_blocks * block_size: token not stored */
#define PA_DEVERR_TABLE 2  /* a block-table entry that must be read lies outside [0, num_blocks):
                              the positions of that block are left out of the softmax */
#define PA_DEVERR_LENGTH 4 /* a context length or cu_seqlens span outside its contract
                              (negative, longer than the block table covers, k_len < q_len,
                              q_len > max_seqlen_q): the sequence's output rows are zero */
#define PA_DEVERR_TIMEOUT 8 /* an internal wait (on an asynchronous copy or on another warp)
                               gave up after about half a second: the kernel stopped early and
                               its outputs are incomplete */

/*
 * pa_store_kv: scatter this step's new K and V rows into the pools.
 *
 * Source: "nano-vLLM Part 4" section 3 (table row "K/V work": K/V written for every new prompt
 * token in prefill, for one input token per sequence in decode; step 3: per-rank slot
 * mappings); smzdm deep dive "模型实现细节" (store_kvcache writes newly computed K and V rows
 * to their physical positions).
 *
 *   for t in [0, T): s = slot_mapping[t]; if s < 0 skip (padding token)
 *       k_cache row s = k[t]  (Hkv * D elements, bit copy);  v_cache row s = v[t]
 *
 * k, v          [T, Hkv, D] contiguous, the new rows.
 * k_cache/v_cache  pools (see above), written in place.
 * slot_mapping  int32 [T]; entries must be unique among the non-negative ones (two tokens in
 *               one slot leave either row there). An entry >= num_blocks * block_size sets
 *               PA_DEVERR_SLOT and that token is not stored.
 * T == 0 is a no-op. Bytes moved: 4 * T * Hkv * D * 2 (read k, v; write both pools).
 */
pa_status pa_store_kv(const void *k, const void *v, void *k_cache, void *v_cache,
                      const int32_t *slot_mapping, int T, int num_blocks, int block_size, int Hkv,
                      int D, pa_dtype dtype, int32_t *err, cudaStream_t stream);

/*
 * pa_decode_workspace_size: bytes of scratch pa_decode needs for these sizes on the current
 * device. The work is cut into units: one per CTA (one or two CTAs per SM), and, for group sizes
 * up to 3 and batches of at most 9216 sequences whose tables could hold at least 16 tiles of 64
 * positions per CTA, up to eight more per CTA that CTAs take as they finish.
 * Each unit has two partial results (G query heads x (D + 2) fp32: output, running max, sum) for
 * the at most two context pieces it shares with a neighbour, plus a 64-byte record; the launch a
 * 16-byte counter. It depends on the group size G = Hq / Hkv, D, the batch size, the table's
 * width and the SM count (about 12 MB at most on a GB300), not on the context lengths. Never
 * fails; returns 0 for sizes that pa_decode would reject.
 */
size_t pa_decode_workspace_size(int B, int Hq, int Hkv, int D, int max_blocks_per_seq,
                                int block_size);

/*
 * pa_decode_debug_tail_units: diagnostics (the pages have no counterpart). Once the last
 * pa_decode or pa_store_decode launch that used `workspace` (with these sizes) has completed, the
 * number of dynamic-tail units that launch ran: 0 when it kept one equal share per CTA. Read from
 * the launch's own record in the workspace with a synchronous 64-byte device-to-host copy.
 * Returns -1 for sizes pa_decode would reject, a NULL workspace or a failed copy. Launches whose
 * table holds at most 256 positions per sequence run the short-context kernel, which writes no
 * record: for those the value read is whatever an earlier launch left.
 */
int pa_decode_debug_tail_units(const void *workspace, int B, int Hq, int Hkv, int D,
                               int max_blocks_per_seq, int block_size);

/*
 * pa_decode: paged grouped-query decode attention, one query token per sequence.
 *
 * Source: "nano-vLLM Part 4" section 3 (decode: one already-sampled token per sequence;
 * attention over cached history through a block table, flash_attn_with_kvcache); "mini-vLLM"
 * (one token per sequence attending to that sequence's cached keys and values; grouped-query
 * attention).
 *
 *   for sequence i, query head h, kv head g = h / (Hq / Hkv), n = context_lens[i]:
 *       s_j = scale * q[i,h,:] . K_j,   K_j, V_j = row j of sequence i (0 <= j < n) via its table
 *       out[i,h,:] = sum_j softmax(s)_j V_j         (zeros when n == 0)
 *
 * The step's own token must already be in the pool (pa_store_kv first) and counted in n.
 *
 * out           [B, Hq, D], written.
 * q             [B, Hq, D].
 * block_tables  int32 [B, max_blocks_per_seq].
 * context_lens  int32 [B]; 0 <= n <= max_blocks_per_seq * block_size, else PA_DEVERR_LENGTH.
 * scale         softmax scale (1/sqrt(D) in the usual case).
 * workspace     device scratch of at least pa_decode_workspace_size(B, Hq, Hkv, D,
 *               max_blocks_per_seq, block_size) bytes, or NULL when that size is 0. Its
 *               contents on entry do not matter; calls that share a workspace must not overlap
 *               on the GPU.
 * B == 0 is a no-op.
 */
pa_status pa_decode(void *out, const void *q, const void *k_cache, const void *v_cache,
                    const int32_t *block_tables, int max_blocks_per_seq,
                    const int32_t *context_lens, int B, int Hq, int Hkv, int D, int block_size,
                    int num_blocks, float scale, pa_dtype dtype, void *workspace,
                    size_t workspace_bytes, int32_t *err, cudaStream_t stream);

/*
 * pa_store_decode: the decode layer step (store the new token's K/V, then decode) in one launch.
 *
 * Source: "nano-vLLM Part 4" section 3 (each decode step writes the new token's key and value into
 * the cache through the slot mapping, then attends over the cached history); "mini-vLLM" (one
 * token per sequence attending to that sequence's cached keys and values).
 *
 * For sequence i with n = context_lens[i] > 0 the new token is position n - 1: its rows k_new[i],
 * v_new[i] are written to the slot of that position, block_tables[i][(n-1) / block_size] *
 * block_size + (n-1) % block_size, and the attention uses them for that position directly (the
 * launch does not read them back from the pool). The result, pools included, equals pa_store_kv
 * with slot_mapping[i] = that slot (or -1 when n == 0) followed by pa_decode.
 *
 * k_new, v_new  [B, Hkv, D], 16-byte aligned. Rows of sequences with n == 0 are not stored.
 * Other arguments, the workspace and the errors as pa_decode. The new token's slot must not be
 * read by another sequence of the same call (a block with free slots belongs to one sequence).
 */
pa_status pa_store_decode(void *out, const void *q, const void *k_new, const void *v_new,
                          void *k_cache, void *v_cache, const int32_t *block_tables,
                          int max_blocks_per_seq, const int32_t *context_lens, int B, int Hq,
                          int Hkv, int D, int block_size, int num_blocks, float scale,
                          pa_dtype dtype, void *workspace, size_t workspace_bytes, int32_t *err,
                          cudaStream_t stream);

/*
 * pa_store_decode_host: pa_store_decode for a step whose inputs and output live in host memory
 * (the pools stay on the device, as in an engine). On `stream`, in order: one copy host -> device
 * of each input (q, k_new, v_new, block_tables, context_lens) into the device workspace, the
 * store + decode launches, and one copy device -> host of the output. The call returns once these
 * are queued; the host buffers must stay valid and unchanged until the stream has passed them
 * (synchronise the stream before reading out_host). Page-locked host memory lets the copies run
 * asynchronously; pageable memory works too, with copies that block.
 *
 * Source: as pa_store_decode ("nano-vLLM Part 4" section 3: the engine moves each step's inputs
 * to the device and reads the sampled result back).
 *
 * out_host, q_host               [B, Hq, D] (fp16/bf16 bits), host
 * k_new_host, v_new_host         [B, Hkv, D], host
 * block_tables_host              int32 [B, max_blocks_per_seq], host
 * context_lens_host              int32 [B], host
 * k_cache, v_cache               device pools, as pa_store_decode
 * workspace                      device memory of at least pa_store_decode_host_workspace_size()
 *                                bytes, 256-byte aligned: the staged inputs and output, then
 *                                pa_decode's workspace
 * Inputs packed in one host buffer at the offsets pa_store_decode_host_layout() gives (q_host at
 * offset 0 of the buffer, the others after it) travel in one copy instead of five. When that
 * buffer (or out_host) is page-locked memory registered with CUDA and mapped into the device's
 * address space, 16-byte aligned, the copy is done by a kernel whose SMs load (store) the host
 * bytes directly; otherwise by cudaMemcpyAsync.
 * Errors: as pa_store_decode; PA_ERR_NULL for a missing host pointer; PA_ERR_WORKSPACE when the
 * workspace is missing, too small or unaligned; PA_ERR_CUDA when a copy cannot be queued.
 */
size_t pa_store_decode_host_workspace_size(int B, int Hq, int Hkv, int D, int max_blocks_per_seq,
                                           int block_size);
/*
 * pa_store_decode_host_layout: the packed host layout of a step's inputs. Writes the byte offsets
 * of q, k_new, v_new, block_tables and context_lens (in that order, 256-byte aligned, q at 0) to
 * offsets[0..4] and returns the bytes a buffer holding all five needs; returns 0 (offsets
 * untouched) for an empty batch or invalid sizes. offsets may be NULL to query the size alone.
 */
size_t pa_store_decode_host_layout(int B, int Hq, int Hkv, int D, int max_blocks_per_seq,
                                   size_t *offsets);
pa_status pa_store_decode_host(void *out_host, const void *q_host, const void *k_new_host,
                               const void *v_new_host, void *k_cache, void *v_cache,
                               const int32_t *block_tables_host, int max_blocks_per_seq,
                               const int32_t *context_lens_host, int B, int Hq, int Hkv, int D,
                               int block_size, int num_blocks, float scale, pa_dtype dtype,
                               void *workspace, size_t workspace_bytes, int32_t *err,
                               cudaStream_t stream);

/*
 * pa_prefill_varlen: variable-length (causal) prefill attention over packed prompts, with a
 * cached prefix read from the pool.
 *
 * Source: "nano-vLLM Part 4" section 3 (prefill: packed tokens, variable-length attention,
 * optional prefix block table); smzdm deep dive "GPU执行优化" (cu_seqlens mark sequence
 * boundaries) and "模型实现细节" (the prefix cache is used when cu_seqlens_k > cu_seqlens_q);
 * "mini-vLLM" (concatenated prompts, each attending causally to itself).
 *
 *   for sequence s: q_len = cu_seqlens_q[s+1] - cu_seqlens_q[s],
 *                   k_len = cu_seqlens_k[s+1] - cu_seqlens_k[s],  P = k_len - q_len >= 0
 *   new row r (0 <= r < q_len) sits at position P + r and, with `causal`, sees keys 0 .. P + r
 *   (without it, all k_len keys):
 *       out[cu_seqlens_q[s] + r, h, :] = sum_j softmax_j(scale * q . K_j) V_j
 *
 * Key/value source:
 *   block_tables != NULL: every key (prefix and new) is read from k_cache / v_cache through
 *       block_tables[s]; call pa_store_kv for the new rows first. k and v are not read (may
 *       be NULL).
 *   block_tables == NULL: keys are the packed rows k[cu_seqlens_k[s] + j], v[...] ([Tk, Hkv, D],
 *       Tk = cu_seqlens_k[S]); k_cache, v_cache are not read (may be NULL).
 *
 * out           [Tq, Hq, D], Tq = cu_seqlens_q[S], written (rows of sequences flagged with
 *               PA_DEVERR_LENGTH are zero).
 * q             [Tq, Hq, D].
 * cu_seqlens_q, cu_seqlens_k  int32 [S+1], non-decreasing, starting at 0.
 * total_q       host int: rows of q and out (= cu_seqlens_q[S]); bounds every read of q.
 * total_k       host int: rows of the packed k, v (= cu_seqlens_k[S]) when block_tables is NULL;
 *               ignored otherwise.
 * max_seqlen_q  host int >= every q_len (sizes the grid).
 * max_seqlen_k  host int, a bound on k_len used only to order the work (how many prompts run
 *               together so that their keys stay in L2); any value gives the same result.
 * S == 0 is a no-op.
 */
pa_status pa_prefill_varlen(void *out, const void *q, const void *k, const void *v,
                            const void *k_cache, const void *v_cache,
                            const int32_t *cu_seqlens_q, const int32_t *cu_seqlens_k, int S,
                            int total_q, int total_k, int max_seqlen_q, int max_seqlen_k,
                            const int32_t *block_tables, int max_blocks_per_seq, int Hq, int Hkv,
                            int D, int block_size, int num_blocks, float scale, int causal,
                            pa_dtype dtype, int32_t *err, cudaStream_t stream);

/*
 * pa_decode_noalloc: pa_decode for callers that cannot allocate device memory.
 *
 * The pages have no counterpart to this call; it exists for users of the library that cannot
 * provide pa_decode's workspace: a host framework that owns every device allocation and gives
 * its plugins none, a process whose device memory is already fully reserved by another
 * allocator, or a step loop that cannot afford cudaMalloc's implicit device synchronisation.
 *
 * It computes exactly what pa_decode computes, with the same arguments minus the workspace. Its
 * split-K scratch is one file-scope device array of PA_DECODE_NOALLOC_SCRATCH_BYTES (1 MiB),
 * which every GPU that loads this library holds until the process exits. The call itself
 * allocates nothing (no cudaMalloc, no cudaFree, no allocating library routine).
 *
 * - Limit: it always cuts the work into one unit per CTA (no units taken as CTAs finish), so it
 *   needs the partials of those units only; sizes for which they exceed
 *   PA_DECODE_NOALLOC_SCRATCH_BYTES (GQA groups of 8 at D = 128, for instance) are rejected with
 *   PA_ERR_WORKSPACE before anything is launched (use pa_decode for them).
 * - Set-up: the first call on each device looks up the array's device address
 *   (cudaGetSymbolAddress) with that device current and keeps it for the life of the process;
 *   make that first call before any stream capture. A failed lookup returns PA_ERR_CUDA. A
 *   cudaDeviceReset (or any reset of the device's primary context) invalidates the kept address:
 *   do not call pa_decode_noalloc on a device after resetting it.
 * - Sharing: every call on a device uses the same array and leaves the last call's partial
 *   results in it. Nothing in it needs to start at zero, but calls that overlap on the GPU
 *   (on different streams, or from different host threads) race on it: serialise them.
 */
#define PA_DECODE_NOALLOC_SCRATCH_BYTES (1u << 20)
pa_status pa_decode_noalloc(void *out, const void *q, const void *k_cache, const void *v_cache,
                            const int32_t *block_tables, int max_blocks_per_seq,
                            const int32_t *context_lens, int B, int Hq, int Hkv, int D,
                            int block_size, int num_blocks, float scale, pa_dtype dtype,
                            int32_t *err, cudaStream_t stream);

/*
 * Host block manager: block ids, reference counts and an exact full-block prefix cache for the
 * pool, with one block table per sequence. Host code only; nothing here touches the GPU.
 *
 * Source: "nano-vLLM Part 4", sections 2 and 3 (the BlockManager's ids, reference counts and
 * prefix-hash metadata, the exact full-block prefix cache, complete blocks hashed after each step,
 * blocks freed when a sequence finishes); smzdm nano-vLLM deep dive "调度与内存" (fixed-size blocks,
 * reference counts, the prefix cache shared by requests with a common system prompt, preemption
 * that frees blocks and keeps the tokens); "mini-vLLM" (a preallocated pool, an O(1) free-list
 * allocator, a block table per sequence). The pages give no API; this one is:
 *
 *   pa_bm_create        a pool of num_blocks blocks of block_size slots; all free, queued in id
 *                       order. flags: 0, or PA_BM_DEGENERATE_HASH (every token hash equal, for
 *                       tests of the collision path). NULL on bad arguments or no memory.
 *   pa_bm_allocate      blocks for a new sequence `seq` with tokens[0..n): the longest run of
 *                       cached full blocks that starts it is reused, except a block holding its
 *                       last token (at least one token is always computed); the other blocks come
 *                       from the front of the free queue (a free block taken for new content is
 *                       no longer findable, nor is any block cached after it); the sequence's full
 *                       blocks are cached at once. Returns the number of tokens already cached (a
 *                       multiple of block_size, < n), or PA_BM_ERR_NO_BLOCKS with nothing changed.
 *   pa_bm_can_allocate  1 if pa_bm_allocate would succeed now, else 0.
 *   pa_bm_append        one more token for `seq`: a new block from the free queue when its last
 *                       block is full (PA_BM_ERR_NO_BLOCKS with nothing changed if none is free);
 *                       a block that becomes full is cached. Returns the token's slot
 *                       (block * block_size + offset), the value pa_store_kv's slot_mapping takes.
 *   pa_bm_release       the sequence finishes (or is preempted): one reference less on each of
 *                       its blocks, last block first; blocks left with none join the back of the
 *                       free queue and stay findable by the cache until taken for new content.
 *   pa_bm_block_table   writes min(cap, blocks) entries of the sequence's table, returns blocks.
 *   pa_bm_num_tokens, pa_bm_num_free, pa_bm_refcount: state queries.
 *
 * A cached full block is identified by its own tokens and by its parent (the block before it when
 * it was filled, and that block's content generation), so a hit is a match on the whole prefix;
 * hits are checked token by token, so a hash collision can cost a hit but never give a wrong one.
 * Not thread-safe: one host thread (the scheduler) owns a manager.
 */
#define PA_BM_DEGENERATE_HASH 1
#define PA_BM_ERR_ARG (-1)        /* null manager / tokens, n < 1, bad block id */
#define PA_BM_ERR_NO_BLOCKS (-2)  /* not enough free blocks: nothing changed */
#define PA_BM_ERR_NO_SEQ (-3)     /* unknown sequence id */
#define PA_BM_ERR_SEQ_EXISTS (-4) /* pa_bm_allocate on a live sequence id */
typedef struct pa_block_manager pa_block_manager;
pa_block_manager *pa_bm_create(int num_blocks, int block_size, int flags);
void pa_bm_destroy(pa_block_manager *bm);
int pa_bm_allocate(pa_block_manager *bm, int64_t seq, const int32_t *tokens, int n);
int pa_bm_can_allocate(const pa_block_manager *bm, const int32_t *tokens, int n);
int64_t pa_bm_append(pa_block_manager *bm, int64_t seq, int32_t token);
int pa_bm_release(pa_block_manager *bm, int64_t seq);
int pa_bm_block_table(const pa_block_manager *bm, int64_t seq, int32_t *out, int cap);
int pa_bm_num_tokens(const pa_block_manager *bm, int64_t seq);
int pa_bm_num_free(const pa_block_manager *bm);
int pa_bm_refcount(const pa_block_manager *bm, int block);

/* A static, human-readable name for a status code. */
const char *pa_status_string(pa_status status);

#ifdef __cplusplus
}
#endif

#endif /* PA_H */
