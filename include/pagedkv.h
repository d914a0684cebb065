/*
 * pagedkv.h -- C ABI of a GB300 (sm_103a) paged KV cache: block manager,
 * slot write, copy-on-write block copy, split-K decode attention and
 * chunked-prefill attention.
 *
 * Pages followed (cited by title and section):
 *   [BT] "KV Cache 还有空间为何新请求却进不来？PagedAttention 的块表与碎片控制"
 *        (zwjcode.cn), sections 03-13.
 *   [KC] "KV 缓存管理" (gptbert.com, mlsys vol. 3), sections "PagedAttention
 *        虚拟内存模型" and "通过写时复制分支实现零复制审慎推理", and the
 *        chunked-prefill section (online-softmax merge).
 *   [IO] "第 8 章 推理优化" (bojieli.github.io), sections 8.2.3 and 8.3.1-8.3.2.
 *
 * Layout ([BT] §06):
 *   K_cache, V_cache : [N_layers][N_blocks][B][H_kv][D_h], row-major, dtype
 *                      float32 or bfloat16, owned by the caller (device).
 *   block_table      : int32 [N_seq][max_blocks], -1 past ceil(ctx / B).
 *   context_lens     : int32 [N_seq].
 *   slot             : int64 p * B + o for physical block p, offset o.
 * Token t of a sequence lives at (block_table[seq][t / B], t % B) ([BT] §03).
 *
 * Conventions
 *   - Every function returns a kvStatus.  Arguments are checked before any
 *     state changes: a call that fails changes nothing ([BT] §10).
 *   - Host functions (block_*, seq_*, kv_pool_stats/check) never touch the
 *     device and are synchronous.  A pool is not thread safe.
 *   - Device functions enqueue work on the given stream (a cudaStream_t passed
 *     as void*; NULL is the legacy default stream) and return after the
 *     launch; they report launch errors only.  Bad block ids or slots met on
 *     the device are skipped and recorded in the pool's device status word;
 *     kv_pool_device_status() reads it.
 *   - The library allocates no device memory.  Device buffers (pools, the
 *     status word, decode workspaces) come from the caller.
 *   - A freed block may be handed out again by the next allocation; device
 *     readers stay safe because later writers are ordered after them on the
 *     same stream ([IO] §8.3.2: free only once the accelerator is done).
 *     Callers that use several streams must order them themselves.
 */
#ifndef PAGEDKV_H
#define PAGEDKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef int kvStatus;
enum {
  KV_OK = 0,
  KV_ERR_NO_FREE_BLOCK = 1, /* free list empty ([BT] §05 "no free KV block") */
  KV_ERR_INVALID_ARG = 2,   /* bad shape, id, size or unknown sequence      */
  KV_ERR_REFCOUNT = 3,      /* handle not held, double free, broken counts   */
  KV_ERR_CUDA = 4,          /* a CUDA runtime call failed                   */
  KV_ERR_DEVICE_CHECK = 5,  /* a kernel recorded a bad id / slot / timeout  */
  KV_ERR_UNSUPPORTED = 6,   /* shape outside the compiled kernel set        */
  KV_ERR_SCRATCH_TOO_SMALL = 7 /* request exceeds the static scratch array    */
};

/* KV_DTYPE_FP8_E4M3: a quantized pool ("第 8 章 推理优化" §8.4.2): each K or V
 * element is one E4M3 code (sign, 4 exponent bits with bias 7, 3 mantissa
 * bits, no infinities, NaN = all exponent and mantissa bits set) of
 * x / scale, with one float32 scale per pool for K and one for V
 * (kv_pool_set_fp8_scales); half the bytes of BF16.  Its q, new K/V rows and
 * outputs are bfloat16 (outputs may also be float32).
 * KV_DTYPE_Q8_0: the pages' q8_0 ([IO] §8.4.2, Fig. 8-23): every group of 32
 * consecutive values of a (slot, head) row shares one fp16 scale d and keeps
 * one int8 code each, x ~ code * d (34 bytes per 32 values, against 64 for
 * BF16).  The codes fill K_cache / V_cache ([N_layers][N_blocks][B][H_kv]
 * [D_h], one byte each); the scales live in two more arrays given by
 * kv_pool_set_q8_scales.  A written group's scale is the fp16 nearest to
 * max |x| / 127 (float32 division), each code the integer nearest to x / d
 * (float32 division, ties to even) clamped to [-127, 127], an all-zero group
 * having d = 0 and zero codes.  q, new K/V rows and outputs as for FP8.
 * D_h a multiple of 32; device work needs the scale arrays. */
enum { KV_DTYPE_F32 = 0, KV_DTYPE_BF16 = 1, KV_DTYPE_FP8_E4M3 = 2, KV_DTYPE_Q8_0 = 3 };

/* bits of the device status word */
enum {
  KV_DEV_BAD_BLOCK_ID = 1, /* block_table entry outside [0, N_blocks)  */
  KV_DEV_BAD_SLOT = 2,     /* slot_mapping entry >= N_blocks * B       */
  KV_DEV_BAD_COW_PAIR = 4, /* copy pair id outside [0, N_blocks)       */
  KV_DEV_WAIT_TIMEOUT = 8, /* a pipeline wait gave up (never expected;
                              kv_device_wait_selftest sets it on purpose) */
  KV_DEV_BAD_CONTEXT = 16, /* context_lens entry < 0 or > max_blocks * B */
  KV_DEV_SMEM_ALIGN = 32   /* shared staging not 1 KiB aligned: pass skipped */
};

typedef struct kvPool kvPool;

const char* kv_status_string(kvStatus s);

/* ---------------------------------------------------------------- pool -- */

/* Create a pool over caller-owned device caches.
 *   k_cache, v_cache: device pointers, layout above, 16-byte aligned; may be
 *     NULL for a host-only manager (device functions then fail with
 *     KV_ERR_INVALID_ARG).
 *   d_status: device int32 the kernels OR error bits into; may be NULL.
 *   free_order: host array of n_blocks ids, a permutation of 0..n_blocks-1
 *     giving the initial FIFO free list ([BT] §05); NULL means 0..n_blocks-1.
 * Supported: block_size 1..256, head_dim 64 or 128, dtype F32 or BF16;
 * FP8_E4M3 with head_dim 128 and block_size a multiple of 8 that divides 64
 * or is a multiple of it (decode on either tensor-core pass); Q8_0 with
 * FP8's shapes (decode on the warp-level pass).  Creation itself fails with
 * KV_ERR_INVALID_ARG only for non-positive sizes, block_size > 256, an
 * unknown dtype, or (Q8_0) a head_dim not a multiple of 32 or H_kv *
 * block_size * head_dim / 16 scale bytes per block not a multiple of 16;
 * device calls on other unsupported shapes return KV_ERR_UNSUPPORTED. */
kvStatus kv_pool_create(int n_layers, int n_blocks, int block_size, int n_kv_heads,
                        int head_dim, int dtype, void* k_cache, void* v_cache,
                        int32_t* d_status, const int32_t* free_order, kvPool** out);
void kv_pool_destroy(kvPool* pool);

/* Free / allocated / shared (count > 1) block counts; [KC] Eq. 8 U_KV is
 * n_allocated / (n_free + n_allocated). */
kvStatus kv_pool_stats(const kvPool* pool, int* n_free, int* n_allocated, int* n_shared);

/* Conservation checks of [BT] §13: N_free + N_alloc = N_total, the set of
 * blocks with a positive count is exactly the allocated set, each count
 * equals the table entries naming the block plus the caller-held handles,
 * and every table holds ceil(len / B) entries.  KV_ERR_REFCOUNT if broken. */
kvStatus kv_pool_check(const kvPool* pool);

/* Reference count of one block (debugging aid). */
kvStatus kv_block_refcount(const kvPool* pool, int32_t id, int* out);

/* Pool options.  KV_OPT_DECODE_PATH selects the split-pass kernel:
 * 0 = automatic (warp-level tensor-core pass for bfloat16 pools whose block
 * size is a multiple of 8 and for FP8 and q8_0 pools, CUDA-core pass
 * otherwise), 1 = always the CUDA-core pass (not for FP8 or q8_0 pools), 2 =
 * the warp-level tensor-core pass (mma.sync) where the pool allows it, 3 =
 * the tcgen05 pass (tensor-memory accumulators; bfloat16 or FP8, D_h = 128)
 * where the pool allows it, else as 2.  A plan (paged_decode_plan)
 * records the kernel it was built for and the planned calls run that kernel;
 * in automatic mode the plan takes the tcgen05 pass when segments wider than
 * 16 query columns hold at least half of the blocks it reads, else the
 * warp-level pass.  Changing the option invalidates partials of earlier split
 * passes.  KV_OPT_PDL: 1 (default) =
 * launch kernels with a programmatic dependency on the previous grid in the
 * stream (each kernel waits for its predecessors before reading their
 * results, but is scheduled while they finish), 0 = plain launches.
 * KV_OPT_PLAN_GRID: the CTA count for which paged_decode_plan writes its
 * per-CTA start records (value in 1 .. 1024; 0, the default = the split
 * pass's own count once the device is known).  Records built for another
 * count than the launch's are ignored (the kernel then searches the plan);
 * results are the same either way. */
enum { KV_OPT_DECODE_PATH = 1, KV_OPT_PDL = 2, KV_OPT_PLAN_GRID = 3 };
kvStatus kv_pool_set_option(kvPool* pool, int option, int value);

/* Scales of an FP8_E4M3 pool (default 1, 1): a written value x is stored as
 * the E4M3 code nearest to x / scale in float32 (IEEE division), ties to the
 * even mantissa, magnitudes beyond 448 (infinities too) saturating to 448;
 * attention reads code * scale.  Both must be positive and finite; other
 * dtypes: KV_ERR_INVALID_ARG.  Codes already written keep their meaning only
 * under the scales they were written with. */
kvStatus kv_pool_set_fp8_scales(kvPool* pool, float k_scale, float v_scale);

/* Scale arrays of a Q8_0 pool: fp16, [N_layers][N_blocks][H_kv][B][D_h / 32]
 * each (the scales of one block and head side by side, B * D_h / 16 bytes),
 * 16-byte aligned device memory owned by the caller.  The pool's copy-on-write
 * copies them with the codes.  Other dtypes or null / misaligned pointers:
 * KV_ERR_INVALID_ARG. */
kvStatus kv_pool_set_q8_scales(kvPool* pool, void* k_scales, void* v_scales);

/* Synchronise `stream`, copy the device status word to *out_bits and clear
 * it.  Returns KV_ERR_DEVICE_CHECK when any bit was set. */
kvStatus kv_pool_device_status(kvPool* pool, void* stream, int* out_bits);

/* Health check of the device's bounded waits (no counterpart on the pages):
 * enqueues on `stream` a one-thread kernel that waits on a barrier nothing
 * completes, with the helper every pipeline wait of the library uses; after
 * limit_us microseconds (1 .. 1,000,000) the wait gives up and
 * KV_DEV_WAIT_TIMEOUT is set in the pool's status word, read with
 * kv_pool_device_status.  No copy or other work is in flight while it waits,
 * and the device stays usable.  Returns launch errors only. */
kvStatus kv_device_wait_selftest(kvPool* pool, int limit_us, void* stream);

/* ---------------------------------------------------------- block level --
 * Caller-held handles on blocks, sharing the pool's free list and counts
 * ([KC] zero-copy branching section).                                     */

/* Pop n ids from the head of the free list (all or nothing), count 1 each. */
kvStatus block_alloc(kvPool* pool, int n, int32_t* out_ids);
/* Drop one handle per listed id; a count reaching 0 returns the block to the
 * tail of the free list.  KV_ERR_REFCOUNT if a handle is not held. */
kvStatus block_free(kvPool* pool, const int32_t* ids, int n);
/* Add one handle per listed id (share).  KV_ERR_REFCOUNT if a block is free. */
kvStatus block_fork(kvPool* pool, const int32_t* ids, int n);
/* Copy-on-write for a held handle on `id`: if the block is shared, take a new
 * block from the free list, move the handle to it and return it in *out_id
 * (the caller then copies id -> *out_id with cow_copy); otherwise return id. */
kvStatus block_cow(kvPool* pool, int32_t id, int32_t* out_id);

/* ------------------------------------------------------- sequence level --
 * The teaching BlockManager of [BT] §05 with the counts, fork and CoW of
 * [KC].  A sequence is created by its first append.                       */

/* One slot for each listed sequence, in the listed order, all or nothing
 * ([BT] §10).  For sequence i, out_slots[i] = p * B + o where (p, o) is the
 * new token's position ([BT] §03-§04).  When a token lands in a shared,
 * partly filled tail block, a fresh block replaces it in that sequence's
 * table and the pair (old, new) is appended to out_cow_pairs (capacity
 * n_seq pairs, int32 [n][2]); *out_n_cow gets the number of pairs.  The
 * first sharer to write copies; the last one writes in place.  A sequence
 * listed twice is KV_ERR_INVALID_ARG. */
kvStatus seq_append_slots(kvPool* pool, const int32_t* seq_ids, int n_seq, int64_t* out_slots,
                          int32_t* out_cow_pairs, int* out_n_cow);
/* n_tokens consecutive slots for one sequence (a prefill chunk), all or
 * nothing; at most one copy pair (capacity 1 pair). */
kvStatus seq_append_tokens(kvPool* pool, int32_t seq, int n_tokens, int64_t* out_slots,
                           int32_t* out_cow_pair, int* out_n_cow);
/* Child gets a copy of the parent's table, one more count on each block and
 * the parent's length ([KC] fork steps 1-3).  No device work. */
kvStatus seq_fork(kvPool* pool, int32_t parent, int32_t child);
/* Drop one count per table entry, in table order; blocks reaching 0 go to the
 * free-list tail ([KC] release_sequence_blocks).  No device work. */
kvStatus seq_release(kvPool* pool, int32_t seq);
kvStatus seq_length(const kvPool* pool, int32_t seq, int* out_len);
/* Rows of the listed sequences' tables, padded with -1 to max_blocks, and
 * their context lengths.  KV_ERR_INVALID_ARG if a table is wider. */
kvStatus seq_block_table(const kvPool* pool, const int32_t* seq_ids, int n_seq, int max_blocks,
                         int32_t* out_table, int32_t* out_context_lens);

/* ------------------------------------------------------- prefix cache -- */
/* Full-block prefix reuse across requests ("KV 缓存管理", radix-tree section:
 * longest prefix match, block-aligned truncation, leaf-first LRU eviction;
 * "第 11 章 KV Cache 内存管理" §11.5: block-level hashing, a key that covers
 * everything changing the KV numbers).  Host only, no device work.
 *
 * With the cache on, a full block is identified by the salt and every token
 * of its sequence up to the block's end (a chained 64-bit hash finds it; the
 * block's tokens and its parent are compared, so no hash collision can alias
 * two prefixes).  A block joins the cache when it fills (at the end of the
 * append call), if its tokens are known, its key is not cached yet and the
 * block before it in the same table is cached (or it is the first).  A
 * cached block whose count drops to 0 stays allocated but dormant; when a
 * block is needed and the free list is empty, the dormant leaf (no cached
 * block after it) with the oldest access is evicted to the free list, and
 * its parent may become such a leaf.  Accesses are stamped by a logical
 * clock: the blocks a match takes, a block joining the cache, a block turning
 * dormant, in table order.  kv_pool_check also checks the cache's tree,
 * counts and eviction set; kv_pool_stats counts dormant blocks as allocated.
 */
/* Turn the cache on with a salt standing for the model, template, adapters
 * and anything else that changes the KV numbers; again with the same salt:
 * KV_OK; with another: KV_ERR_INVALID_ARG.  Positions written before are
 * unknown tokens (their blocks never join). */
kvStatus kv_prefix_cache_enable(kvPool* pool, uint64_t salt);
/* A new sequence (KV_ERR_INVALID_ARG if it exists, or the cache is off)
 * starts with the longest chain of cached full blocks matching its prompt
 * tokens[0 .. n_tokens): *out_matched = that many tokens, a multiple of B
 * (the tail of a partly matching block counts as a miss and is prefilled
 * with the rest).  One more count on each taken block. */
kvStatus seq_match_prefix(kvPool* pool, int32_t seq, const int32_t* tokens, int n_tokens,
                          int* out_matched);
/* seq_append_slots / seq_append_tokens with the token ids of the appended
 * positions (token_ids: one per listed sequence / n_tokens; NULL: unknown).
 * Blocks may be evicted from the cache to make room. */
kvStatus seq_append_slots_ids(kvPool* pool, const int32_t* seq_ids, int n_seq,
                              const int32_t* token_ids, int64_t* out_slots,
                              int32_t* out_cow_pairs, int* out_n_cow);
kvStatus seq_append_tokens_ids(kvPool* pool, int32_t seq, int n_tokens, const int32_t* token_ids,
                               int64_t* out_slots, int32_t* out_cow_pair, int* out_n_cow);
/* Evict dormant leaves, oldest access first, until the free list holds
 * target_free blocks or none is left (the pages' low-water-mark round). */
kvStatus kv_prefix_evict(kvPool* pool, int target_free, int* out_n_evicted);
kvStatus kv_prefix_stats(const kvPool* pool, int* n_cached, int* n_dormant);

/* ------------------------------------------------------------- device --
 * All pointers below are device pointers.                                */

/* Copy-on-write copy ([KC] CoW paragraph; [IO] §8.3.2): for each pair
 * d_pairs[i] = (src, dst) copy every slot of block src into block dst, K and
 * V, in every layer.  No dst may be another pair's src in the same call. */
kvStatus cow_copy(kvPool* pool, const int32_t* d_pairs, int n_pairs, void* stream);

/* Slot write ("reshape_and_cache"; [KC] paging section, [BT] §04): token i's
 * K and V rows [H_kv][D_h] go to slot d_slot_mapping[i] of `layer`; a
 * negative slot skips the token.  layer == -1 writes every layer at once,
 * with k_new / v_new laid out [N_layers][n_tokens][H_kv][D_h]. */
kvStatus reshape_and_cache(kvPool* pool, int layer, const void* d_k_new, const void* d_v_new,
                           const int64_t* d_slot_mapping, int n_tokens, void* stream);

/* Bytes of decode workspace for n_seq sequences with n_q_heads query heads.
 * Independent of the context lengths. */
size_t paged_decode_workspace_bytes(const kvPool* pool, int n_seq, int n_q_heads);

/* Split-K partial pass of decode attention ([BT] §07; [KC] online softmax).
 * q: [n_seq][n_q_heads][D_h] in the pool dtype.  Query head h reads K/V head
 * h / (n_q_heads / H_kv).  The work (all sequences x K/V heads x blocks) is
 * cut into equal contiguous block ranges, one per CTA; each CTA writes the
 * running max m, normaliser l and unnormalised output O of every range it
 * covers into the workspace.  scale <= 0 means 1 / sqrt(D_h). */
kvStatus paged_decode_partials(kvPool* pool, int layer, const void* d_q, int n_q_heads,
                               const int32_t* d_block_table, int max_blocks,
                               const int32_t* d_context_lens, int n_seq, float scale,
                               void* d_workspace, size_t workspace_bytes, void* stream);

/* Merge pass: m = max m_i, l = sum l_i e^(m_i - m), out = sum O_i e^(m_i - m)
 * / l per (sequence, query head); out [n_seq][n_q_heads][D_h] as float32
 * (out_dtype F32) or bfloat16 (BF16).  A sequence with context 0 gets zeros.
 * Must follow paged_decode_partials on the same stream with the same
 * arguments. */
kvStatus paged_decode_merge(kvPool* pool, int n_q_heads, const int32_t* d_context_lens,
                            int n_seq, void* d_out, int out_dtype, const void* d_workspace,
                            size_t workspace_bytes, void* stream);

/* Both passes: decode attention of one layer for every listed sequence. */
kvStatus paged_decode_attention(kvPool* pool, int layer, const void* d_q, int n_q_heads,
                                const int32_t* d_block_table, int max_blocks,
                                const int32_t* d_context_lens, int n_seq, float scale,
                                void* d_out, int out_dtype, void* d_workspace,
                                size_t workspace_bytes, void* stream);

/* ------------------------------------------- sharing-aware decode plan --
 * Sequences that share physical blocks (after seq_fork, or a shared prompt;
 * [KC] zero-copy branching, [IO] §8.3.2) can have each shared block read
 * once for all of them.  paged_decode_plan builds, on the host, from the
 * pool's tables, a work list for the listed sequences (in their current
 * state, after the step's seq_append_slots): sequences whose tables start
 * with the same run of full blocks (at least min_shared_tokens tokens; 0
 * means 128) form groups of at most 32 / G members, whose shared prefix is one
 * segment per K/V head carrying all members' query heads; the rest of each
 * sequence is a segment of its own.  The plan is a flat byte buffer to copy
 * to the device as-is.  *out_workspace_bytes gets the decode workspace size
 * the plan needs.  Once the pool's device is known the plan also carries, per
 * CTA of the split pass, the CTA's first piece of work and the physical ids
 * of its first blocks (taken from the tables as they are now: the plan goes
 * with the block table of the same state), so that the CTA's first copies
 * start without searching the plan or reading the table; a buffer sized by
 * paged_decode_plan_bytes before the device was known has no room for them,
 * and the plan is then built without. */
size_t paged_decode_plan_bytes(const kvPool* pool, int n_seq, int n_q_heads);
kvStatus paged_decode_plan(const kvPool* pool, const int32_t* seq_ids, int n_seq, int n_q_heads,
                           int max_blocks, int min_shared_tokens, void* h_plan, size_t plan_bytes,
                           size_t* out_workspace_bytes);

/* The two passes of a planned decode, separately (same arguments as
 * paged_decode_attention_planned; the merge must follow the partials on the
 * same stream with the same plan and workspace). */
kvStatus paged_decode_partials_planned(kvPool* pool, int layer, const void* d_q, int n_q_heads,
                                       const int32_t* d_block_table, int max_blocks,
                                       const void* d_plan, const void* h_plan, float scale,
                                       void* d_workspace, size_t workspace_bytes, void* stream);
kvStatus paged_decode_merge_planned(kvPool* pool, int n_q_heads, const void* d_plan,
                                    const void* h_plan, void* d_out, int out_dtype,
                                    const void* d_workspace, size_t workspace_bytes, void* stream);

/* The planned split pass with the step's slot write of `layer` fused in
 * ([BT] §10's reserve -> write -> attend, the write done by the CTA that
 * reads the block it lands in, just before that read): the same pool
 * contents and partials as reshape_and_cache(layer, rows, slots) followed by
 * paged_decode_partials_planned.  Every listed sequence must have its
 * newest token, the one this step reserved, at its last context position
 * (context_len - 1) of the tables the plan was built from, with any
 * copy-on-write of the step already enqueued (cow_copy).
 *   d_k_new, d_v_new: [n_seq][H_kv][D_h] bfloat16 rows of this layer, in
 *                     plan order (FP8 pools quantize them as the slot write
 *                     does), 16-byte aligned
 * bfloat16 and FP8 pools only (KV_ERR_UNSUPPORTED otherwise); other
 * arguments as paged_decode_partials_planned.  A bad block id met while
 * writing skips the write (the read records KV_DEV_BAD_BLOCK_ID). */
kvStatus paged_decode_partials_planned_write(kvPool* pool, int layer, const void* d_q,
                                             int n_q_heads, const void* d_k_new,
                                             const void* d_v_new, const int32_t* d_block_table,
                                             int max_blocks, const void* d_plan,
                                             const void* h_plan, float scale, void* d_workspace,
                                             size_t workspace_bytes, void* stream);

/* Decode attention of one layer following a plan: d_block_table and d_q hold
 * the listed sequences' rows in plan order; d_plan is the device copy of
 * h_plan (both are read: the host copy for sizes, the device copy by the
 * kernels).  Tensor-core path only (bfloat16 pool, B a multiple of 8):
 * KV_ERR_UNSUPPORTED otherwise.  Output as paged_decode_attention. */
kvStatus paged_decode_attention_planned(kvPool* pool, int layer, const void* d_q, int n_q_heads,
                                        const int32_t* d_block_table, int max_blocks,
                                        const void* d_plan, const void* h_plan, float scale,
                                        void* d_out, int out_dtype, void* d_workspace,
                                        size_t workspace_bytes, void* stream);

/* Same as paged_decode_attention, without a caller workspace, for callers
 * that cannot allocate device memory (under an allocator that has reserved
 * all device memory; plain C hosts with no allocator).  The workspace is a
 * 16 MiB array in the library's static device memory, one per GPU, held
 * until the process exits.  Requests whose paged_decode_workspace_bytes()
 * exceed 16 MiB (about 880 sequences at G = 4, D_h = 128, H_kv = 8) fail with
 * KV_ERR_SCRATCH_TOO_SMALL before any device work.  Every call looks the
 * array's device address up on the current device (no allocation, no device
 * work), so no address is kept across a reset of the device's context.
 * Calls on one GPU share the array: calls that overlap on the GPU race.  The
 * pages have no counterpart of this call. */
kvStatus paged_decode_attention_noalloc(kvPool* pool, int layer, const void* d_q, int n_q_heads,
                                        const int32_t* d_block_table, int max_blocks,
                                        const int32_t* d_context_lens, int n_seq, float scale,
                                        void* d_out, int out_dtype, void* stream);

/* ------------------------------------------------- chunked prefill --
 * Attention of prompt chunks over the paged cache ([KC] chunked-prefill
 * section; [IO] §8.2.3).  For each listed sequence s, the chunk's queries
 * are rows d_chunk_start[s] .. d_chunk_start[s + 1] - 1 of d_q; the chunk's
 * K and V must already be in the pool (reserve the chunk with
 * seq_append_tokens, write it with reshape_and_cache), as the last
 * c = d_chunk_start[s + 1] - d_chunk_start[s] of d_context_lens[s] positions.
 * The chunk's token i (position h + i, h = context - c) attends to positions
 * 0 .. h + i: the whole history and the chunk up to its own token.
 *   d_q          : [n_tok][n_q_heads][D_h] bfloat16, 16-byte aligned
 *   d_block_table: [n_seq][max_blocks] int32
 *   d_chunk_start: [n_seq + 1] int32, non-decreasing query-row offsets
 *   d_context_lens: [n_seq] int32, context after the chunk
 *   max_chunk    : an upper bound on every chunk's length (sizes the grid; a
 *                  longer chunk, or a chunk longer than its context, is
 *                  skipped and flagged KV_DEV_BAD_CONTEXT)
 *   d_out        : [n_tok][n_q_heads][D_h] float32 or bfloat16 (out_dtype)
 * Runs on the tcgen05 tensor cores: bfloat16 pools with D_h = 128 and B a
 * multiple of 8 (whole 64-row boxes), H_q / H_kv in {1, 2, 4, 8}; other
 * pools get KV_ERR_UNSUPPORTED.  Allocates nothing; enqueues one kernel on
 * `stream`. */
kvStatus paged_prefill_attention(kvPool* pool, int layer, const void* d_q, int n_q_heads,
                                 const int32_t* d_block_table, int max_blocks,
                                 const int32_t* d_chunk_start, const int32_t* d_context_lens,
                                 int n_seq, int max_chunk, float scale, void* d_out,
                                 int out_dtype, void* stream);

/* Heaviest-first work order for chunked prefill.  A work item is one tile
 * of 128 / G query tokens (G = n_q_heads / H_kv) of one sequence's chunk;
 * its work is the number of 128-key blocks its queries read,
 * ceil((h + min(c, (t + 1) * 128 / G)) / 128) for history h = context - c,
 * chunk length c and tile t ([KC] chunked-prefill section: a chunk's token
 * attends to the whole history and the chunk up to itself).  The natural
 * grid starts the items of later sequences last, whatever their length;
 * launching the longest items first lets the SMs finish together.
 * paged_prefill_schedule builds the order on the host from host copies of
 * the chunk geometry that paged_prefill_attention_scheduled will get:
 *   h_chunk_start : [n_seq + 1] int32, h_context_lens: [n_seq] int32
 *   h_sched       : caller buffer of at least
 *                   paged_prefill_schedule_bytes(pool, n_seq, n_q_heads,
 *                   max_chunk) bytes (max_chunk bounds every chunk), filled
 *                   with *out_n_items records of four int32: (sequence,
 *                   tile, chunk length, blocks), blocks non-increasing,
 *                   equal blocks in (sequence, tile) order.
 * Empty chunks have no items.  KV_ERR_INVALID_ARG for a negative chunk, a
 * chunk longer than its context, or a buffer too small;
 * paged_prefill_schedule_bytes returns 0 for invalid arguments. */
size_t paged_prefill_schedule_bytes(const kvPool* pool, int n_seq, int n_q_heads, int max_chunk);
kvStatus paged_prefill_schedule(const kvPool* pool, const int32_t* h_chunk_start,
                                const int32_t* h_context_lens, int n_seq, int n_q_heads,
                                void* h_sched, size_t sched_bytes, int* out_n_items);

/* paged_prefill_attention over the work order d_sched (the device copy of
 * h_sched, 16-byte aligned, n_items records; not written by a kernel on the
 * stream since the previous kernel began): the same results, bit for bit,
 * as the natural grid, one CTA per (item, K/V head) in the order's order.
 * A sequence whose chunk length differs from the one its items were built
 * for is skipped and flagged KV_DEV_BAD_CONTEXT; so is an item naming no
 * listed sequence. */
kvStatus paged_prefill_attention_scheduled(kvPool* pool, int layer, const void* d_q, int n_q_heads,
                                           const int32_t* d_block_table, int max_blocks,
                                           const int32_t* d_chunk_start,
                                           const int32_t* d_context_lens, int n_seq,
                                           const void* d_sched, int n_items, float scale,
                                           void* d_out, int out_dtype, void* stream);

/* Chunked prefill for any pool dtype.  A bfloat16 pool is read in place, as
 * by paged_prefill_attention (d_sched null: the natural grid over max_chunk)
 * or paged_prefill_attention_scheduled (d_sched, n_items), and the
 * workspace is not used.  An FP8 (E4M3) pool (D_h = 128, the tensor-core
 * block shapes) is read through a bfloat16 copy in the caller's workspace:
 * a first kernel turns the codes of every block each listed sequence reads
 * (its first ceil(context_lens[s] / B) table entries of layer `layer`) into
 * their exact bfloat16 values, then the same tcgen05 pass attends over the
 * copy with the K scale folded into the score scale and the outputs
 * multiplied by the V scale, so the results are those of attention over the
 * pool's dequantized values ([IO] §8.4.2: narrower KV read, wider
 * arithmetic).  Slots past a context are copied as zeros.
 *   d_workspace : device buffer, 256-byte aligned, of at least
 *                 paged_prefill_staging_bytes(pool, n_seq, max_blocks)
 *                 bytes (0 for a bfloat16 pool); reused across calls, it
 *                 must not be written while a call on it is in flight.
 * Errors as paged_prefill_attention; KV_ERR_UNSUPPORTED for other dtypes
 * or shapes; an out-of-range table entry is flagged KV_DEV_BAD_BLOCK_ID and
 * its block copied as zeros. */
size_t paged_prefill_staging_bytes(const kvPool* pool, int n_seq, int max_blocks);
kvStatus paged_prefill_attention_staged(kvPool* pool, int layer, const void* d_q, int n_q_heads,
                                        const int32_t* d_block_table, int max_blocks,
                                        const int32_t* d_chunk_start,
                                        const int32_t* d_context_lens, int n_seq, int max_chunk,
                                        const void* d_sched, int n_items, float scale,
                                        void* d_out, int out_dtype, void* d_workspace,
                                        size_t workspace_bytes, void* stream);

/* --------------------------------------------------- whole decode step --
 * One decode step through host buffers ([BT] §10 order: reserve, upload,
 * launch, read back): reserve a slot per listed sequence on the host, build
 * the tables (and, on the tensor-core passes, the sharing-aware plan), copy
 * them with the slots and copy pairs to the device in one copy, run
 * cow_copy, write the new token of every layer, attend per layer, and
 * synchronise the stream.
 *   h_q     : [N_layers][n_seq][n_q_heads][D_h]  (pool dtype; bf16 for FP8)
 *   h_k_new : [N_layers][n_seq][H_kv][D_h]        same dtype, same h_v_new
 *   h_out   : [N_layers][n_seq][n_q_heads][D_h]  float32
 *   d_staging: caller device buffer of kv_decode_step_staging_bytes() bytes.
 * Page-locked host buffers that are mapped into the device's address space
 * (cudaMallocHost / cudaHostAlloc, a mapped cudaHostRegister, or torch's
 * pin_memory, under unified addressing) are used in place: the kernels read
 * q and the new rows and the merge writes the outputs through the mapping.
 * Other host buffers go through d_staging with copies.  With a plan on a
 * bfloat16 or FP8 pool the split pass writes the new rows itself (the
 * fused slot write); otherwise reshape_and_cache does.  In-place and
 * staged buffers give the same outputs and pools, bit for bit.  A step
 * that fails after issuing copies synchronises before returning; a failure
 * after the reservation leaves the reservation in place.  max_blocks bounds
 * every listed table after the step. */
size_t kv_decode_step_staging_bytes(const kvPool* pool, int n_seq, int n_q_heads, int max_blocks);
kvStatus kv_decode_step_host(kvPool* pool, const int32_t* seq_ids, int n_seq, int n_q_heads,
                             int max_blocks, const void* h_q, const void* h_k_new,
                             const void* h_v_new, float scale, float* h_out, void* d_staging,
                             size_t staging_bytes, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* PAGEDKV_H */
