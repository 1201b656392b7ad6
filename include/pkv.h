/*
 * pkv.h -- C ABI of the paged KV-cache attention library (GB300, sm_103a).
 *
 * The operations are those of a nano-vllm style engine's attention layer:
 *   - the KV-cache store through a slot mapping, which nano-vllm performs with
 *     a Triton kernel (nano-vllm hub page, pomoai.com, "core tech 2:
 *     Attention + Triton kernel");
 *   - attention over the paged cache, with fixed 256-token blocks managed by a
 *     block manager (same page, "core tech 4: KV Cache block manager") and a
 *     per-sequence block table mapping logical to physical blocks (CSDN essay
 *     "from nanoVLLM to vLLM", Mountain 1: KV cache);
 *   - separate kernels for the compute-dense prefill phase and the
 *     memory-bound decode phase (same essay, Mountain 3 and the study route's
 *     attention/ module notes).
 * The result of both attention calls is that of standard attention,
 * softmax(q K^T * scale) V: FlashAttention-style tiling only reorders the
 * computation (same essay, Mountain 3).
 *
 * Conventions shared by every call
 * --------------------------------
 *  - bf16 tensors are passed as pointers to their 16-bit patterns.
 *  - Every pointer argument except `dev_status` and `stream` is a DEVICE
 *    pointer owned by the caller; no call allocates memory or keeps a
 *    reference after it returns.  The library caches small per-device tables
 *    (the SM count) and, loaded on a GPU, holds one fixed 16 MiB device array
 *    (the scratch of pkv_paged_decode_attn_noalloc).
 *  - Layouts (all row-major, contiguous):
 *      q             [T_q, Hq, D]
 *      k, v          [T_new, Hkv, D]   (token stride configurable in kv_store)
 *      k_cache       [num_blocks, block_size, Hkv, D]; one slot = Hkv*D values
 *      v_cache       same as k_cache
 *      out           [T_q, Hq, D]
 *      block_tables  int32 [num_seqs, max_blocks_per_seq], unused entries -1
 *      slot_mapping  int32 [T_new]; slot = block * block_size + offset; -1 = skip
 *      context_lens  int32 [num_seqs]; keys visible, INCLUDING the tokens just
 *                    stored
 *      cu_seqlens_q  int32 [num_seqs+1], prefix sums of new-token counts
 *      cu_seqlens_k  int32 [num_seqs+1], prefix sums of (cached + new) counts
 *  - GQA: query head h reads kv head h / (Hq / Hkv).
 *  - Pointers to bf16 data must be 16-byte aligned.
 *  - Every call is asynchronous on `stream` (a cudaStream_t; NULL = the
 *    legacy default stream).  Host-side argument checks run before any
 *    launch: a failed check returns a status and launches nothing.
 *  - Data-dependent faults (a slot or block id out of range, an empty or
 *    oversize context) are caught by bounds checks on the device: the kernel
 *    skips the access, ORs a PKV_DEV_* bit into *dev_status (when dev_status is
 *    not NULL; it is a device int32) and finishes.  Nothing traps or spins
 *    without a limit; a wait that exceeds its limit sets PKV_DEV_TIMEOUT.
 */
#ifndef PKV_H_
#define PKV_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum pkv_status {
  PKV_OK = 0,
  PKV_ERR_INVALID_ARG = 1, /* null pointer, bad size, misaligned pointer */
  PKV_ERR_UNSUPPORTED = 2, /* head_dim, group size or block_size not built */
  PKV_ERR_WORKSPACE = 3,   /* workspace missing or too small */
  PKV_ERR_CUDA = 4,        /* a CUDA runtime/driver call or launch failed */
  PKV_ERR_OUT_OF_BLOCKS = 5 /* block manager: not enough free blocks (nothing changed) */
} pkv_status;

/* Bits OR-ed into *dev_status by the kernels. */
#define PKV_DEV_BAD_SLOT 0x1    /* slot_mapping entry outside [-1, NB*BS) */
#define PKV_DEV_BAD_BLOCK 0x2   /* block_tables entry outside [0, NB) */
#define PKV_DEV_BAD_CONTEXT 0x4 /* context length <= 0 or > max_blocks*BS */
#define PKV_DEV_TIMEOUT 0x8     /* a bounded wait ran out */
#define PKV_DEV_WORKSPACE 0x10  /* decode: more blocks than max_total_blocks */
#define PKV_DEV_BAD_SEQLEN 0x20 /* prefill: bad cu_seqlens (n > len_k, n > max_seqlen_q) */

/* Human-readable name of a pkv_status value (static string). */
const char *pkv_status_string(int status);

/* ABI revision of this header; bumped on any signature change. */
int pkv_abi_version(void);

/*
 * kv_store -- write this step's new K and V rows into the paged cache.
 *
 * For every token t in [0, num_tokens) with s = slot_mapping[t] >= 0:
 *   k_cache slot s (Hkv*D values) <- k row t,  v_cache slot s <- v row t.
 * A bit copy: no arithmetic touches the values.  Slots equal to -1 are
 * skipped (padding); any other slot outside [0, num_blocks*block_size) sets
 * PKV_DEV_BAD_SLOT and is skipped.  Slots >= 0 must be unique.
 *
 * k_token_stride / v_token_stride: elements between consecutive tokens of k
 * and v (0 = Hkv*D, i.e. contiguous); must keep rows 16-byte aligned.
 * Requires (Hkv*D) % 8 == 0.
 */
pkv_status pkv_kv_store(const uint16_t *k, const uint16_t *v, uint16_t *k_cache,
                        uint16_t *v_cache, const int32_t *slot_mapping, int64_t num_tokens,
                        int num_kv_heads, int head_dim, int64_t k_token_stride,
                        int64_t v_token_stride, int64_t num_blocks, int block_size,
                        int32_t *dev_status, void *stream);

/*
 * Bytes of device workspace paged_decode_attn needs: a 256-byte work counter,
 * then the split-K scratch.  max_total_blocks is an upper bound the caller
 * guarantees on sum_s ceil(context_lens[s]/block_size) (num_seqs *
 * max_blocks_per_seq always works).  Returns 0 for invalid sizes
 * and for sizes whose workspace would not fit a size_t.
 */
size_t pkv_decode_workspace_size(int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                                 int64_t max_total_blocks);

/*
 * paged_decode_attn -- one query token per sequence against its paged K/V.
 *
 * out[s, h, :] = softmax_p(scale * <q[s,h,:], K_s[p, h/g, :]>) V_s[p, h/g, :]
 * over p in [0, context_lens[s]), where K_s[p] is the cache slot
 * block_tables[s][p / block_size] * block_size + p % block_size and
 * g = Hq / Hkv.  bf16 in, fp32 accumulation, bf16 out (round to nearest even).
 *
 * Split-K flash-decoding: each (sequence, kv head, block) is one work item
 * (two consecutive blocks per item when the batch has very many of them)
 * whose partial (max, sum, unnormalised output) goes to the workspace; the
 * persistent CTAs take items from a counter in the workspace as they become
 * free.  A second kernel, launched as a programmatic dependent of the first,
 * merges the partials of every sequence that spans more than one item.  Two
 * kernel launches per call (one when max_blocks_per_seq == 1).
 *
 * workspace: device buffer of at least pkv_decode_workspace_size(...) bytes,
 * 256-byte aligned, zero-filled once before its first use.  Its first 256
 * bytes hold the work counter, which every call leaves at zero (also a call
 * whose waits ran out); the rest needs no initialisation (each call writes
 * every entry before reading it).  Calls that overlap on the device must not
 * share a workspace.
 *
 * scale: any finite value (zero averages the context's values; a NaN or
 * infinite scale returns PKV_ERR_INVALID_ARG and launches nothing).
 *
 * Supported: head_dim in {64, 128}; Hq/Hkv in {1, 2, 4, 8}; block_size in
 * {64, 128, 256, 512}; num_seqs <= 16384, and the kernel's per-CTA shared
 * memory (which holds every sequence's block offset and length) must fit in
 * 227 KiB: only head_dim 128 with Hq/Hkv 8 and block_size 512 reaches that
 * limit first, at 16093 sequences.  A batch beyond either limit returns
 * PKV_ERR_UNSUPPORTED; sizes whose workspace cannot be addressed return
 * PKV_ERR_INVALID_ARG.  Both launch nothing.
 */
pkv_status pkv_paged_decode_attn(uint16_t *out, const uint16_t *q, const uint16_t *k_cache,
                                 const uint16_t *v_cache, const int32_t *block_tables,
                                 const int32_t *context_lens, int num_seqs, int num_q_heads,
                                 int num_kv_heads, int head_dim, int block_size,
                                 int max_blocks_per_seq, int64_t num_blocks,
                                 int64_t max_total_blocks, float scale, void *workspace,
                                 size_t workspace_bytes, int32_t *dev_status, void *stream);

/*
 * paged_decode_store_attn -- kv_store of this step's tokens fused with
 * paged_decode_attn, in the same launches as paged_decode_attn alone.
 *
 * A decode step stores one new token per sequence and then attends over the
 * whole context including it (nano-vllm hub page, "core tech 2": the layer
 * writes K/V through the slot mapping, then runs attention; CSDN essay
 * "from nanoVLLM to vLLM", Mountain 3).  Here new_k / new_v [num_seqs, Hkv, D]
 * (contiguous) hold, in row s, the token at position context_lens[s] - 1 of
 * sequence s, and slot_mapping[s] is its slot (-1: attend to it but do not
 * store it).  The result and the cache afterwards are bit-identical to
 * pkv_kv_store followed by pkv_paged_decode_attn: the work item that holds
 * the newest token takes that token's row from new_k / new_v and, after using
 * it, writes it to the cache; no other work item of the call reads that slot.
 *
 * Arguments, workspace and errors as for paged_decode_attn and kv_store
 * (slots out of range set PKV_DEV_BAD_SLOT and are not written).
 */
pkv_status pkv_paged_decode_store_attn(uint16_t *out, const uint16_t *q, const uint16_t *new_k,
                                       const uint16_t *new_v, const int32_t *slot_mapping,
                                       uint16_t *k_cache, uint16_t *v_cache,
                                       const int32_t *block_tables, const int32_t *context_lens,
                                       int num_seqs, int num_q_heads, int num_kv_heads,
                                       int head_dim, int block_size, int max_blocks_per_seq,
                                       int64_t num_blocks, int64_t max_total_blocks, float scale,
                                       void *workspace, size_t workspace_bytes,
                                       int32_t *dev_status, void *stream);

/*
 * paged_decode_attn_noalloc -- paged_decode_attn without a caller workspace.
 *
 * The pages have no counterpart to this call; it exists for callers of this
 * library that cannot allocate device memory for a workspace: code running
 * under a host framework whose allocator owns all device memory and offers no
 * hook, a plugin that may not allocate inside its host process, or a serving
 * loop that must keep cudaMalloc/cudaFree (which synchronise the device) off
 * its latency path.
 *
 * The split-K scratch lives in a fixed 16 MiB array in the library's own
 * device memory, which every GPU that loads the library holds until the
 * process exits.  A call whose workspace need,
 * pkv_decode_workspace_size(num_seqs, num_q_heads, num_kv_heads, head_dim,
 * max_total_blocks), exceeds 16 MiB returns PKV_ERR_WORKSPACE and launches
 * nothing.  The call itself allocates nothing.
 *
 * The first call on each device looks up the array's device address
 * (cudaGetSymbolAddress) with that device current; make that first call
 * before any stream capture.  Each call then runs the same kernels as
 * pkv_paged_decode_attn on that array.  The array is zero when the library
 * loads and keeps the previous call's contents: its work counter (the first
 * 256 bytes) is left at zero by every call, and the rest is written before it
 * is read.  All calls on a device share the one array, so
 * calls that overlap on the GPU (other streams, other host threads) race and
 * corrupt each other's results: serialise them.
 *
 * Arguments, layouts, results and errors are those of pkv_paged_decode_attn.
 */
pkv_status pkv_paged_decode_attn_noalloc(uint16_t *out, const uint16_t *q,
                                         const uint16_t *k_cache, const uint16_t *v_cache,
                                         const int32_t *block_tables,
                                         const int32_t *context_lens, int num_seqs,
                                         int num_q_heads, int num_kv_heads, int head_dim,
                                         int block_size, int max_blocks_per_seq,
                                         int64_t num_blocks, int64_t max_total_blocks,
                                         float scale, int32_t *dev_status, void *stream);

/*
 * test_decode_fault -- TEST-ONLY fault injection for the decode kernels'
 * bounded waits (the pages have no counterpart; it exists so that tests can
 * make a wait run out without faulting or hanging the GPU).
 *
 * Sets, for the current device, the wall-clock limit of every wait in the
 * decode kernels (default 1 s) and a tile number that every decode CTA's
 * producer then skips instead of loading (-1: none, the default).  A decode
 * call made while a tile is withheld waits out the limit, flags
 * PKV_DEV_TIMEOUT in *dev_status, leaves its output undefined and returns;
 * the device stays usable.  Restore with pkv_test_decode_fault(1000000000, -1).
 * Synchronous (it copies to device memory).  Returns PKV_ERR_INVALID_ARG for
 * wait_limit_ns <= 0 or withhold_tile < -1.
 */
pkv_status pkv_test_decode_fault(int64_t wait_limit_ns, int withhold_tile);

/*
 * paged_prefill_attn -- causal attention of packed variable-length prompts
 * over the paged cache, including an already-cached prefix.
 *
 * For sequence s: n = cu_seqlens_q[s+1] - cu_seqlens_q[s] new queries and
 * len_k = cu_seqlens_k[s+1] - cu_seqlens_k[s] keys, of which c = len_k - n
 * were cached before this step (their K/V, and the new tokens' K/V, must
 * already be in the cache: call kv_store first).  Query i sits at absolute
 * position c + i and attends to keys 0 .. c + i:
 *   out[cu_q[s]+i, h, :] = softmax_{p <= c+i}(scale * <q, K_s[p, h/g]>) V_s[p, h/g]
 * bf16 operands on the tcgen05 tensor cores, fp32 accumulation in tensor
 * memory, bf16 out.
 *
 * total_q = cu_seqlens_q[num_seqs]; max_seqlen_q bounds every n (a larger n
 * sets PKV_DEV_BAD_SEQLEN and its excess rows are not written).  A sequence
 * with n = 0 has no rows.  A sequence's rows do not depend on the other
 * sequences of the call or on their order (the kernel schedules the longest
 * contexts first; the result is the same bit for bit).
 *
 * workspace: device memory of at least pkv_prefill_workspace_size() bytes,
 * 256-byte aligned, zero-filled before its first use.  It holds the counter
 * from which the kernel's CTAs take their work; every call leaves it zeroed
 * again, so one zero-fill at allocation is enough.  Calls that may run at the
 * same time on the GPU (other streams, other host threads) need workspaces
 * of their own.  Missing, short or misaligned: PKV_ERR_WORKSPACE.
 *
 * scale: any finite value (a NaN or infinite scale returns
 * PKV_ERR_INVALID_ARG and launches nothing).
 *
 * Supported: head_dim in {64, 128}; Hq/Hkv in {1, 2, 4, 8};
 * block_size in {64, 128, 256, 512}.
 */
pkv_status pkv_paged_prefill_attn(uint16_t *out, const uint16_t *q, const uint16_t *k_cache,
                                  const uint16_t *v_cache, const int32_t *block_tables,
                                  const int32_t *cu_seqlens_q, const int32_t *cu_seqlens_k,
                                  int num_seqs, int64_t total_q, int max_seqlen_q,
                                  int num_q_heads, int num_kv_heads, int head_dim,
                                  int block_size, int max_blocks_per_seq, int64_t num_blocks,
                                  float scale, void *workspace, size_t workspace_bytes,
                                  int32_t *dev_status, void *stream);

/* Bytes of device workspace pkv_paged_prefill_attn needs (any shape). */
size_t pkv_prefill_workspace_size(void);

/*
 * w4a16_dequant -- W4A16-G128 weight dequantisation (s1nh.org post on
 * upgrading nano-vllm to big-vLLM, section on quantisation: every int32 of
 * weight_packed holds eight 4-bit values; int32 -> u4 unpack -> s4
 * reconstruct -> float x weight_scale, one scale per 128 weights).
 *
 *   out[n, j] = bf16( (u4(packed[n, j / 8], j % 8) - 8) * scales[n, j / 128] )
 *
 * where u4(w, i) = (w >> 4i) & 15 (the lowest nibble is the first value).
 * packed [n_rows, k/8] int32, scales [n_rows, k/128] bf16, out [n_rows, k]
 * bf16, all row-major and contiguous, device memory owned by the caller.
 * The product is exact in fp32 and rounded once (nearest even) to bf16.
 *
 * k must be a multiple of 128 and group_size 128 (PKV_ERR_INVALID_ARG /
 * PKV_ERR_UNSUPPORTED otherwise); out and packed 16-byte aligned, scales
 * 2-byte aligned.  n_rows == 0 or k == 0: nothing to do.
 */
pkv_status pkv_w4a16_dequant(uint16_t *out, const int32_t *packed, const uint16_t *scales,
                             int64_t n_rows, int64_t k, int group_size, void *stream);

/*
 * Block manager -- host-side allocator of the cache's blocks (no GPU work).
 *
 * The cache is a pool of fixed-size blocks handed out and released by
 * reference counting (nano-vllm hub page, "core tech 4: KV Cache block
 * manager"); a sequence takes a new block when its length reaches a multiple
 * of the block size plus one (CSDN essay "from nanoVLLM to vLLM", Mountain
 * 1).  Prefix sharing: every full block gets a content key, a 64-bit FNV-1a
 * hash chained over the key of the block before it and the block's token
 * ids; a new sequence whose prompt begins with full blocks whose keys (and
 * tokens) match reuses those blocks, reference count + 1, and only the rest
 * of the prompt needs kv_store and its own prefill rows.  Freed blocks keep
 * their content and key, and stay reusable, until they are handed out again
 * (oldest freed first; a sequence's tail is freed before its prefix).
 *
 * The outputs feed the kernels directly: pkv_bm_block_table gives a row of
 * block_tables (padded with -1), pkv_bm_slots the slot_mapping of a token
 * range, and pkv_bm_allocate the cached length c (cu_seqlens_k - cu_seqlens_q).
 * Not thread-safe: one manager per host thread.
 */
typedef struct pkv_block_manager pkv_block_manager;

/* num_blocks > 0 blocks of block_size tokens; NULL on bad arguments or no memory. */
pkv_block_manager *pkv_bm_create(int num_blocks, int block_size);
void pkv_bm_destroy(pkv_block_manager *m);
int pkv_bm_num_free_blocks(const pkv_block_manager *m);

/* Admit sequence seq_id (not yet present) with its num_tokens > 0 prompt
 * tokens: reuses the cached leading full blocks, takes fresh ones for the
 * rest (all or nothing: PKV_ERR_OUT_OF_BLOCKS leaves the manager unchanged).
 * *num_cached_tokens = tokens whose K/V are already in reused blocks, at most
 * num_tokens - 1 (the last prompt token is always computed). */
pkv_status pkv_bm_allocate(pkv_block_manager *m, int64_t seq_id, const int32_t *tokens,
                           int num_tokens, int *num_cached_tokens);
/* Append one generated token (a fresh block when it starts a new one). */
pkv_status pkv_bm_append(pkv_block_manager *m, int64_t seq_id, int32_t token);
/* Release the sequence's blocks (reference count - 1 each). */
pkv_status pkv_bm_free(pkv_block_manager *m, int64_t seq_id);

/* Tokens held by the sequence, or -1 if unknown. */
int pkv_bm_num_tokens(const pkv_block_manager *m, int64_t seq_id);
/* Writes max_blocks entries of the sequence's block table (-1 past its
 * blocks) when out != NULL; returns its block count, -1 if unknown. */
int pkv_bm_block_table(const pkv_block_manager *m, int64_t seq_id, int32_t *out,
                       int max_blocks);
/* slots[i] = block_table[p / bs] * bs + p % bs for p = first .. first+count-1. */
pkv_status pkv_bm_slots(const pkv_block_manager *m, int64_t seq_id, int first, int count,
                        int32_t *slots);
/* Reference count of a block (0 = free), -1 on a bad index. */
int pkv_bm_ref_count(const pkv_block_manager *m, int block);

#ifdef __cplusplus
}
#endif

#endif /* PKV_H_ */
