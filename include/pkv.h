/*
 * pkv.h -- C ABI of the GB300 (sm_103a) paged KV-cache attention library.
 *
 * Decode-phase attention over a paged KV cache, plus the cache writes that feed it:
 *
 *   pkv_kv_append               scatter new tokens' K/V into cache slots (slot_mapping)
 *   pkv_kv_block_copy           copy whole blocks (copy-on-write of shared blocks)
 *   pkv_paged_decode_attention  one query per sequence against its paged cache,
 *                               GQA groups sharing each K/V tile, split-K with a
 *                               log-sum-exp merge for long contexts
 *   pkv_decode_step             a decode step: each sequence's new token appended, then
 *                               attended (one launch where the plan allows)
 *   pkv_decode_step_fp8         the same over an FP8 (E4M3) cache, the new rows quantised
 *   pkv_prefill_attention       varlen causal attention over cu_seqlens that also
 *                               writes the cache
 *
 * Conventions shared by every call
 * --------------------------------
 * Cache layout: k_cache and v_cache are each [NB][Hkv][bs][d] row-major (NB physical
 *   blocks, Hkv KV heads, bs tokens per block, head_dim d).  The K (or V) row of the
 *   token stored in slot s for KV head h starts at element
 *   ((s / bs) * Hkv + h) * bs * d + (s % bs) * d.
 *   A slot is a physical block id times bs plus the offset inside the block: logical
 *   position pos of a sequence lives in slot block_table[pos / bs] * bs + pos % bs
 *   (plumephp.com "KV Cache 优化与注意力机制加速：FlashAttention / PagedAttention"
 *   §4.2-§4.3, BlockTable.get_kv).
 * Element types: PKV_F32 (fp32) or PKV_BF16 (bf16).  Queries of decode are fp32;
 *   outputs and lse are fp32.
 * GQA: query head i reads KV head floor(i / m), m = Hq / Hkv consecutive query heads per
 *   group (limoncc.com "大语言模型研究15——注意力机制优化之KV缓存" §3.3).  MHA is
 *   Hkv == Hq, MQA is Hkv == 1.
 * Pointers: every array argument is a DEVICE pointer on the current CUDA device unless
 *   stated otherwise.  The caller owns all memory; the library allocates no device
 *   memory in any call (split-K scratch is the caller's workspace).  The only library
 *   state is one device error word per device (a static device variable).
 * Streams: every call only enqueues work on `stream` and returns; nothing is
 *   synchronised except in pkv_get_device_error.  NULL is the legacy default stream.
 * Errors: arguments are validated on the host before any launch; a bad argument
 *   returns PKV_ERR_INVALID_ARG (or PKV_ERR_UNSUPPORTED / PKV_ERR_WORKSPACE) and
 *   enqueues nothing.  A failed launch returns PKV_ERR_CUDA.  Values that live in
 *   device memory (slots, block ids, lengths, cu_seqlens) are checked by the kernels:
 *   an out-of-range value skips the access it would make and sets a bit of the device
 *   error word (PKV_DEVERR_*), read with pkv_get_device_error.  No kernel traps or
 *   waits without a bound.  pkv_last_error() gives a message for the last failing call
 *   of the calling thread.
 */
#ifndef PKV_H_
#define PKV_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t. */
typedef struct CUstream_st *pkv_stream_t;

typedef enum {
    PKV_OK = 0,
    PKV_ERR_INVALID_ARG = 1,  /* null pointer, bad size, Hq % Hkv != 0, ... */
    PKV_ERR_UNSUPPORTED = 2,  /* valid but not implemented (e.g. an element type) */
    PKV_ERR_WORKSPACE = 3,    /* split-K workspace missing or too small */
    PKV_ERR_CUDA = 4          /* a CUDA runtime call or kernel launch failed */
} pkv_status;

/* Element types of caches and inputs.  PKV_FP8_E4M3 is a one-byte E4M3 code (1 sign, 4
 * exponent bits with bias 7, 3 mantissa bits; no infinities, S.1111.111 is NaN, largest
 * finite 448): kv_append and kv_block_copy move such codes as bytes, and the _fp8 entry
 * points read them with their per-row scales. */
typedef enum { PKV_F32 = 0, PKV_BF16 = 1, PKV_FP8_E4M3 = 2 } pkv_dtype;

/* Bits of the device error word. */
#define PKV_DEVERR_SLOT        1u   /* slot_mapping entry >= NB * bs (write skipped) */
#define PKV_DEVERR_BLOCK       2u   /* block_table entry outside [0, NB) (block read as zeros) */
#define PKV_DEVERR_LEN         4u   /* context length < 0 or > MBS * bs (sequence treated as empty) */
#define PKV_DEVERR_CU_SEQLENS  8u   /* cu_seqlens decreasing, > T, or a sequence > max_seqlen */
#define PKV_DEVERR_PAIR       16u   /* kv_block_copy pair outside [0, NB) (pair skipped) */
#define PKV_DEVERR_TIMEOUT    32u   /* a bounded wait for an asynchronous copy gave up */
#define PKV_DEVERR_LAYOUT     64u   /* a kernel found its shared memory misaligned and did nothing */
#define PKV_DEVERR_PREFIX    128u   /* a shared-prefix group whose members' prefixes differ (length, blocks) */

/* Static description of a status code. */
const char *pkv_status_string(pkv_status status);

/* Message describing the last failing call on the calling thread ("" if none). */
const char *pkv_last_error(void);

/* Library version, major * 10000 + minor * 100 + patch. */
int pkv_version(void);

/*
 * pkv_kv_append -- write T new tokens' K and V rows into the cache.
 *
 * For every token t with slot_mapping[t] >= 0 and every KV head h:
 *   K row of (slot_mapping[t], h) = k_new[t][h][:],  V row likewise from v_new.
 * Compute only the new token's K/V and add it to the cache (limoncc.com
 * "大语言模型研究15——注意力机制优化之KV缓存" §2; zwjcode.cn "KV Cache 的增量解码" §04,
 * §10: write into a preallocated slot instead of concatenating).
 *
 *   k_new, v_new   [T][Hkv][d], element type dt (the cache's; the copy is bit-exact)
 *   k_cache, v_cache  [NB][Hkv][bs][d] of type dt
 *   slot_mapping   int64 [T]; a negative entry is padding (token skipped); an entry
 *                  >= NB * bs sets PKV_DEVERR_SLOT and is skipped
 *   T >= 0 (T == 0 enqueues nothing), Hkv >= 1, d >= 1, bs >= 1, NB >= 1.
 * Two tokens naming the same slot race (the result is one of them).
 */
pkv_status pkv_kv_append(const void *k_new, const void *v_new, void *k_cache, void *v_cache,
                         pkv_dtype dt, const int64_t *slot_mapping, int T, int Hkv, int d,
                         int bs, int NB, pkv_stream_t stream);

/*
 * pkv_kv_block_copy -- copy-on-write support: copy whole physical blocks.
 *
 * For each pair p: block pairs[p][1] of k_cache (all Hkv heads, all bs slots) becomes
 * a copy of block pairs[p][0]; the same for v_cache.  Before a sequence writes into a
 * block whose reference count is above one, the block is copied and the writer gets
 * the copy (plumephp.com "KV Cache 优化与注意力机制加速" §4.3; 0539edu.com
 * "从KV cache共享到批量调度…" §3.2, §5.2: check the count before the write).
 *
 *   pairs  int32 [n][2] (src, dst), device memory.  The copies run concurrently: a
 *          block may not be the dst of two pairs, nor both a src and a dst.  A
 *          block id outside [0, NB) sets PKV_DEVERR_PAIR and the pair is skipped.
 *   n >= 0 (0 enqueues nothing).
 */
pkv_status pkv_kv_block_copy(void *k_cache, void *v_cache, pkv_dtype dt, const int32_t *pairs,
                             int n, int Hkv, int d, int bs, int NB, pkv_stream_t stream);

/*
 * Bytes of split-K workspace pkv_paged_decode_attention needs for these sizes and
 * num_splits on the current device (0 when the call runs in one pass).  The split
 * count chosen for num_splits == 0 depends on the device's SM count.  The workspace
 * starts with PKV_DECODE_COUNTER_BYTES of arrival counters, then the chunk partials.
 */
#define PKV_DECODE_COUNTER_BYTES (256u << 10)

size_t pkv_decode_workspace_bytes(int B, int Hq, int Hkv, int d, int bs, int MBS, int num_splits);

/*
 * Kernels one pkv_paged_decode_attention call with these arguments enqueues on the
 * current device, for q and caches whose base addresses are 16-byte aligned: 0 for B == 0,
 * 1 when the call runs in one pass or the last chunk of each sequence merges in place,
 * 2 when a separate log-sum-exp merge kernel follows the split-K kernel.  Returns -1
 * for arguments pkv_paged_decode_attention rejects.  Enqueues nothing.
 */
int pkv_decode_kernel_launches(int B, int Hq, int Hkv, int d, int bs, int MBS, int NB, pkv_dtype dt,
                               int num_splits);

/* The same count for a pkv_paged_attention call with these arguments. */
int pkv_paged_attention_kernel_launches(int B, int Tq, int max_q, int Hq, int Hkv, int d, int bs,
                                        int MBS, int NB, pkv_dtype dt, int window, int num_splits);

/*
 * pkv_paged_decode_attention -- one new query per sequence against its cached K/V.
 *
 * For sequence b, query head i, KV head j = floor(i / m), len = context_lens[b]:
 *   s_t = scale * q[b][i] . K_t      for the len tokens t of sequence b, K_t read
 *                                   from slot block_table[b][t / bs] * bs + t % bs
 *   out[b][i] = sum_t softmax(s)_t V_t,   lse[b][i] = log sum_t exp(s_t)
 * (softmax(qK^T/sqrt(d))V: limoncc.com §3.1, §3.3; online softmax and the statistic
 * L = m + log l: plumephp.com §2.2-§2.3).  Long contexts are split into chunks of
 * whole blocks whose partial results merge by log-sum-exp.
 *
 *   out          fp32 [B][Hq][d]
 *   lse          fp32 [B][Hq] (natural log) or NULL
 *   q            fp32 [B][Hq][d]
 *   k_cache, v_cache  [NB][Hkv][bs][d], element type dt
 *   block_table  int32 [B][MBS]; entries past a sequence's last block are not read
 *   context_lens int32 [B]: tokens in the cache, counting the token just appended;
 *                0 gives out = 0 and lse = -inf
 *   scale        score scale (1/sqrt(d) for a standard layer)
 *   num_splits   0: chosen by the library; 1: one pass; k > 1: at most k chunks per
 *                sequence (chunk = ceil(MBS / k) blocks)
 *   workspace    device scratch of at least pkv_decode_workspace_bytes(...) bytes
 *                (may be NULL when that is 0).  Zero it once after allocating it:
 *                its first PKV_DECODE_COUNTER_BYTES hold arrival counters that must
 *                be zero when a call starts, and every call that completes leaves
 *                them zero again (the rest is overwritten), so one zeroed workspace
 *                serves any sequence of calls and shapes.  After a call that raised
 *                PKV_DEVERR_TIMEOUT, zero it again.  Calls that share a workspace
 *                must not overlap.
 *   Requires Hq % Hkv == 0, B >= 0, d >= 1, bs >= 1, MBS >= 1.
 *   bf16 caches with d in {64, 128, 256}, bs in {16, 32}, 16-byte aligned caches use
 *   the tensor-core path; other shapes use a CUDA-core path with the same results.
 */
pkv_status pkv_paged_decode_attention(float *out, float *lse, const float *q, const void *k_cache,
                                      const void *v_cache, pkv_dtype dt,
                                      const int32_t *block_table, const int32_t *context_lens,
                                      int B, int Hq, int Hkv, int d, int bs, int MBS, int NB,
                                      float scale, int num_splits, void *workspace,
                                      size_t workspace_bytes, pkv_stream_t stream);

/*
 * pkv_decode_step -- one decode step: the new token of each sequence is appended to the
 * cache, then attended with the rest of the sequence.
 *
 * The same results as pkv_kv_append(k_new, v_new, ..., slot_mapping, T = B) followed by
 * pkv_paged_decode_attention(...) on the same arguments (the new K/V are written into the
 * cache once, zwjcode.cn "KV Cache 的增量解码" §04, §10; the attention as in
 * pkv_paged_decode_attention).  Where the plan allows it (bf16 caches on a tensor-core
 * path -- the chunked kernel with at most 8 query heads per KV head, or the tcgen05
 * kernel -- with 16-byte aligned k_new and v_new) the append runs inside the attention
 * launch: the block that reads a sequence's last page writes the new rows there first,
 * so the step is one launch instead of two.
 *
 *   k_new, v_new  [B][Hkv][d], element type dt: the new token of sequence b is row b
 *   slot_mapping  int64 [B]: its slot, which must be that of position
 *                 context_lens[b] - 1 (block_table[b][(len-1)/bs] * bs + (len-1) % bs);
 *                 < 0: sequence b has no new token this step.  Its block must belong to
 *                 sequence b alone (copy-on-write before the step when it is shared).
 *                 When the append runs inside the attention launch, a slot other than the
 *                 last position's (or any slot for an empty sequence) sets
 *                 PKV_DEVERR_SLOT and is not written; otherwise kv_append's rules apply.
 *   the other arguments as pkv_paged_decode_attention (k_cache, v_cache are written).
 */
pkv_status pkv_decode_step(float *out, float *lse, const float *q, const void *k_new, const void *v_new,
                           const int64_t *slot_mapping, void *k_cache, void *v_cache, pkv_dtype dt,
                           const int32_t *block_table, const int32_t *context_lens, int B, int Hq,
                           int Hkv, int d, int bs, int MBS, int NB, float scale, int num_splits,
                           void *workspace, size_t workspace_bytes, pkv_stream_t stream);

/* Kernels one pkv_decode_step call with these sizes enqueues (16-byte aligned new rows and
 * caches assumed), or -1 when the call would be rejected; 0 for B == 0. */
int pkv_decode_step_kernel_launches(int B, int Hq, int Hkv, int d, int bs, int MBS, int NB, pkv_dtype dt,
                                    int num_splits);

/*
 * pkv_decode_step_shared_prefix -- pkv_decode_step for a batch in which groups of sequences
 * share a prefix through the same physical blocks (forks and a common prompt share their
 * blocks by reference count: 0539edu.com "从KV cache共享到批量调度…" §3, plumephp.com
 * "KV Cache 优化与注意力机制加速" §4.3).  The results are those of pkv_decode_step on the
 * same arguments (caches bit-identical; outputs and lse equal to rounding): the attention
 * over a sequence's keys is the log-sum-exp merge of the attention over its shared prefix
 * and over the keys after it (plumephp.com §2.2-§2.3).  What changes is the work: the
 * prefix of a group is read once, by a tensor-core kernel that attends every member's
 * query heads to it at once, and the decode reads each sequence from the end of its prefix.
 *
 *   prefix_tokens  int32 [B] (device): the number of leading tokens of sequence b that are
 *                  its group's shared prefix -- a multiple of bs, at most context_lens[b] - 1
 *                  (the step's new token is never in it); 0 for a sequence in no group
 *   group_start    int32 [n_groups + 1] (device): the members of group g are
 *                  group_seqs[group_start[g] .. group_start[g+1]), group_start[0] = 0 and
 *                  group_start[n_groups] = n_members
 *   group_seqs     int32 [n_members] (device): sequence indices, each in at most one group;
 *                  every member of a group has the same prefix_tokens and the same first
 *                  prefix_tokens / bs block-table entries (otherwise PKV_DEVERR_PREFIX is set
 *                  and that group's outputs are not to be trusted)
 *   n_groups, n_members, max_group_size, max_prefix_tokens: host-side sizes (max_prefix_tokens
 *                  bounds every prefix_tokens[b]); they size the grids and the workspace
 *   workspace      at least pkv_decode_step_shared_prefix_workspace_bytes(...) bytes, 16-byte
 *                  aligned, its first PKV_DECODE_COUNTER_BYTES zeroed once (as the decode's)
 *   the other arguments as pkv_decode_step.
 * The prefix path is taken for bf16 caches with d in {64, 128}, bs in {16, 32}, 16-byte aligned
 * caches and q, and at most 64 query heads per KV head; otherwise (or with n_groups = 0) the call
 * is exactly pkv_decode_step.
 */
pkv_status pkv_decode_step_shared_prefix(float *out, float *lse, const float *q, const void *k_new,
                                         const void *v_new, const int64_t *slot_mapping, void *k_cache,
                                         void *v_cache, pkv_dtype dt, const int32_t *block_table,
                                         const int32_t *context_lens, const int32_t *prefix_tokens,
                                         const int32_t *group_start, const int32_t *group_seqs, int n_groups,
                                         int n_members, int max_group_size, int max_prefix_tokens, int B, int Hq,
                                         int Hkv, int d, int bs, int MBS, int NB, float scale, int num_splits,
                                         void *workspace, size_t workspace_bytes, pkv_stream_t stream);

/* Workspace bytes of pkv_decode_step_shared_prefix for these sizes on the current device. */
size_t pkv_decode_step_shared_prefix_workspace_bytes(int B, int Hq, int Hkv, int d, int bs, int MBS, int num_splits,
                                                     int n_groups, int n_members, int max_group_size,
                                                     int max_prefix_tokens);

/* Kernels one pkv_decode_step_shared_prefix call with these sizes enqueues (aligned pointers
 * assumed), or -1 when the call would be rejected; 0 for B == 0. */
int pkv_decode_step_shared_prefix_kernel_launches(int B, int Hq, int Hkv, int d, int bs, int MBS, int NB,
                                                  pkv_dtype dt, int num_splits, int n_groups, int n_members,
                                                  int max_group_size, int max_prefix_tokens);

/*
 * pkv_paged_attention -- queries at the end of each cached sequence: several per
 * sequence, causal, with an optional sliding window.
 *
 * Sequence b holds L = context_lens[b] tokens in the cache, its queries' own K/V among
 * them (append first), and owns query rows cu_q[b] .. cu_q[b+1]-1.  Its i-th row, of
 * nq = cu_q[b+1] - cu_q[b], is the token at position p = L - nq + i and attends the keys
 * lo .. p: a query sees itself and the tokens before it, not the later new tokens
 * (zwjcode.cn "KV Cache 的增量解码" §13).  lo = 0 without a window; with window W > 0,
 * lo = max(0, p - W + 1), the most recent W positions (zwjcode.cn §10, §15;
 * plumephp.com "KV Cache 优化与注意力机制加速" §5.2).  One query per sequence and
 * W = 0 is pkv_paged_decode_attention; nq = k new tokens is a k-token verification
 * step; a long nq is a prefill of new tokens on top of a cached prefix.
 *
 *   out, lse     fp32 [Tq][Hq][d] and [Tq][Hq] (lse may be NULL), row-major by query row
 *   q            fp32 [Tq][Hq][d]
 *   cu_q         int32 [B+1], non-decreasing, cu_q[0] = 0, cu_q[B] = Tq, each count
 *                <= max_q and <= context_lens[b].  When Tq == B and max_q == 1 every
 *                sequence has exactly one query and cu_q is not read (may be NULL).
 *   window       0: none; W > 0: sliding window of W tokens.  Blocks before a row's
 *                window are never read, so a caller may free them.
 *   caches, block_table, context_lens, scale, num_splits: as pkv_paged_decode_attention
 *   workspace    pkv_paged_attention_workspace_bytes(...) bytes, zeroed once, same
 *                rules as pkv_paged_decode_attention.
 * One query per sequence runs the decode kernels (tensor cores where they apply);
 * several run a CUDA-core kernel, one warp per (query row, head, chunk).  An
 * inconsistent cu_q or a row count above its sequence length sets
 * PKV_DEVERR_CU_SEQLENS and those rows get out = 0, lse = -inf.  Requires
 * Tq <= B * max_q and Tq * Hq < 2^31.
 */
size_t pkv_paged_attention_workspace_bytes(int B, int Tq, int max_q, int Hq, int Hkv, int d, int bs,
                                           int MBS, int window, int num_splits);

pkv_status pkv_paged_attention(float *out, float *lse, const float *q, const void *k_cache,
                               const void *v_cache, pkv_dtype dt, const int32_t *block_table,
                               const int32_t *context_lens, const int32_t *cu_q, int B, int Tq,
                               int max_q, int Hq, int Hkv, int d, int bs, int MBS, int NB, float scale,
                               int window, int num_splits, void *workspace, size_t workspace_bytes,
                               pkv_stream_t stream);

/*
 * FP8 KV cache.  The pages leave the low-bit format open (zwjcode.cn "KV Cache 的增量解码"
 * §14: low-bit K/V lowers memory and bandwidth, and its error reaches every later query;
 * plumephp.com "KV Cache 优化与注意力机制加速" §2.5: FP8 attention).  This library stores
 * E4M3 codes [NB][Hkv][bs][d] (uint8) with one fp32 scale per row (token slot x KV head)
 * in k_scale / v_scale [NB][Hkv][bs]; the cached value is code * scale.  Blocks move with
 * pkv_kv_block_copy: the codes with dt = PKV_FP8_E4M3, the scales as an fp32 "cache" with
 * d = 1.
 *
 * pkv_kv_append_fp8 -- quantise and scatter new rows.  For each token t with
 * slot_mapping[t] >= 0 and each KV head h, the rows k_new[t][h][:], v_new[t][h][:]
 * (element type new_dt: PKV_BF16 or PKV_F32) are written as
 *   scale = amax(row) / 448,  code_e = E4M3(x_e / scale)  (fp32 divisions; round to
 *   nearest, ties to even, saturating at +-448), a row of zeros as scale 0 and codes 0,
 * into row (slot / bs, h, slot % bs).  Slot errors as pkv_kv_append.
 */
pkv_status pkv_kv_append_fp8(const void *k_new, const void *v_new, pkv_dtype new_dt, uint8_t *k_codes,
                             uint8_t *v_codes, float *k_scale, float *v_scale, const int64_t *slot_mapping,
                             int T, int Hkv, int d, int bs, int NB, pkv_stream_t stream);

/*
 * pkv_paged_decode_attention_fp8 -- pkv_paged_attention with one query per sequence over
 * an FP8 cache: the attention of the cached values code * scale, exactly as if they had
 * been stored in a wider type (scores scale * k_scale[t] * (q . codes_t); weights times
 * v_scale[t] against the codes).  window: 0 or a sliding window of that many tokens.
 * Workspace: pkv_decode_workspace_bytes(B, Hq, Hkv, d, bs, MBS, num_splits) bytes, same
 * rules.  d = 128, bs in {16, 32}, up to 8 query heads per KV head and 16-byte aligned
 * codes and scales use tensor cores; other shapes a CUDA-core path with the same results.
 */
pkv_status pkv_paged_decode_attention_fp8(float *out, float *lse, const float *q, const uint8_t *k_codes,
                                          const uint8_t *v_codes, const float *k_scale, const float *v_scale,
                                          const int32_t *block_table, const int32_t *context_lens, int B,
                                          int Hq, int Hkv, int d, int bs, int MBS, int NB, float scale,
                                          int window, int num_splits, void *workspace,
                                          size_t workspace_bytes, pkv_stream_t stream);

/*
 * pkv_decode_step_fp8 -- pkv_decode_step over an FP8 cache: the same results as
 * pkv_kv_append_fp8(k_new, v_new, new_dt, ..., slot_mapping, T = B) followed by
 * pkv_paged_decode_attention_fp8(..., window = 0, ...) on the same arguments (codes,
 * scales, outputs and lse bit-identical).  With bf16 new rows, at most 8 query heads per
 * KV head and 16-byte aligned codes and scales (the tensor-core path) the quantising
 * append runs inside the attention launch, with pkv_decode_step's slot rules (the slot of
 * position context_lens[b] - 1, or < 0; another slot, or one for an empty sequence, sets
 * PKV_DEVERR_SLOT and is not written); otherwise kv_append_fp8 runs first, with its rules.
 *
 *   k_new, v_new  [B][Hkv][d], element type new_dt (PKV_BF16 or PKV_F32)
 *   k_codes, v_codes, k_scale, v_scale  written as well as read
 *   the other arguments as pkv_decode_step and pkv_paged_decode_attention_fp8.
 */
pkv_status pkv_decode_step_fp8(float *out, float *lse, const float *q, const void *k_new, const void *v_new,
                               pkv_dtype new_dt, const int64_t *slot_mapping, uint8_t *k_codes, uint8_t *v_codes,
                               float *k_scale, float *v_scale, const int32_t *block_table,
                               const int32_t *context_lens, int B, int Hq, int Hkv, int d, int bs, int MBS,
                               int NB, float scale, int num_splits, void *workspace, size_t workspace_bytes,
                               pkv_stream_t stream);

/* Kernels one pkv_decode_step_fp8 call with these sizes enqueues (aligned codes, scales and
 * new rows assumed), or -1 when the call would be rejected; 0 for B == 0. */
int pkv_decode_step_fp8_kernel_launches(int B, int Hq, int Hkv, int d, int bs, int MBS, int NB, pkv_dtype new_dt,
                                        int num_splits);

/*
 * pkv_paged_decode_attention_noalloc -- pkv_paged_decode_attention without a workspace.
 *
 * The pages this library follows (the paper) have no counterpart for this entry point:
 * it exists for callers that cannot call cudaMalloc -- a plugin or extension running
 * inside a host application that owns every byte of device memory and hands out none, or
 * a latency-critical decode loop that must not allocate or free device memory in the
 * middle of a step because cudaFree (and often cudaMalloc) synchronises the whole device.
 *
 * Arguments, layouts and results are those of pkv_paged_decode_attention, minus
 * `workspace` and `workspace_bytes`.  The split-K partials go to a scratch array built
 * into the library: a static device array of PKV_NOALLOC_SCRATCH_BYTES bytes that every
 * GPU which loads the library holds until the process exits.
 *   - Sizes whose partials need more than PKV_NOALLOC_SCRATCH_BYTES (the value
 *     pkv_decode_workspace_bytes returns for the same arguments) are rejected with
 *     PKV_ERR_WORKSPACE before anything is enqueued; num_splits = 1 needs no scratch.
 *   - The first call in each CUDA context (once per device for the runtime's primary
 *     context) looks up the array's device address with that device current; make that
 *     first call before any stream capture.
 *   - Every call shares the one array, which keeps the last call's contents.  Calls
 *     that overlap on the GPU (other streams, other host threads) race on it: the
 *     caller must order them.  Its first PKV_DECODE_COUNTER_BYTES hold the arrival
 *     counters of the split-K chunks that merge in place; a call that uses them first
 *     clears the ones it uses (one cudaMemsetAsync on the stream, no allocation), so a
 *     call that gave up on a wait (PKV_DEVERR_TIMEOUT) leaves nothing behind that
 *     spoils a later call.  The rest of the array need not start at zero.
 *   - No call allocates or frees device memory.
 */
#define PKV_NOALLOC_SCRATCH_BYTES (16u << 20)

pkv_status pkv_paged_decode_attention_noalloc(float *out, float *lse, const float *q,
                                              const void *k_cache, const void *v_cache,
                                              pkv_dtype dt, const int32_t *block_table,
                                              const int32_t *context_lens, int B, int Hq, int Hkv,
                                              int d, int bs, int MBS, int NB, float scale,
                                              int num_splits, pkv_stream_t stream);

/*
 * pkv_prefill_attention -- varlen causal attention of whole prompts, writing the cache.
 *
 * Sequences are packed: sequence b owns tokens [cu_seqlens[b], cu_seqlens[b+1]) of
 * q/k/v (0539edu.com "从KV cache共享到批量调度…" §3.3).  Token t of a sequence (0-based)
 * attends to tokens 0..t of the same sequence with the GQA head mapping:
 *   out[tok][i] = softmax_{u <= t}(scale * q[tok][i] . k[u][j]) v[u][j],  j = floor(i/m)
 * (causal prefill: zwjcode.cn "KV Cache 的增量解码" §05, §13).  When slot_mapping is not
 * NULL, every token's k/v rows are also written to the cache exactly as pkv_kv_append
 * does with the same slot_mapping.
 *
 *   out         fp32 [T][Hq][d];  lse fp32 [T][Hq] or NULL
 *   q           [T][Hq][d];  k, v [T][Hkv][d]; all of element type dt
 *   cu_seqlens  int32 [B+1], non-decreasing, cu_seqlens[0] = 0, cu_seqlens[B] = T;
 *               zero-length sequences are allowed.  Violations set
 *               PKV_DEVERR_CU_SEQLENS and the offending sequence is skipped.
 *   max_seqlen  host-side upper bound of every sequence length (sizes the grid); a
 *               longer sequence sets PKV_DEVERR_CU_SEQLENS and its rows past
 *               max_seqlen are not computed
 *   k_cache, v_cache, slot_mapping, bs, NB: as pkv_kv_append; the caches may be NULL
 *               when slot_mapping is NULL
 *   bf16 with d in {64, 128} uses the tensor-core path; other inputs a CUDA-core path.
 */
pkv_status pkv_prefill_attention(float *out, float *lse, const void *q, const void *k,
                                 const void *v, pkv_dtype dt, const int32_t *cu_seqlens, int B,
                                 int T, int max_seqlen, int Hq, int Hkv, int d, float scale,
                                 void *k_cache, void *v_cache, const int64_t *slot_mapping,
                                 int bs, int NB, pkv_stream_t stream);

/*
 * pkv_selftest_bounded_wait -- runs the kernels' failure path on purpose, for tests.
 *
 * Not part of the attention path, and without a counterpart on the pages: every wait of
 * the library's kernels for an asynchronous copy or tensor-core operation is bounded
 * (about 2 s), and a wait that runs out raises PKV_DEVERR_TIMEOUT and makes its block
 * release what it holds and return, so that the context stays usable.  No correct call
 * ever gets there, so this entry point launches `blocks` blocks of 128 threads that
 * each arm an mbarrier for bytes no copy will deliver (none is issued), wait on it
 * through the kernels' own bounded wait with a limit of `limit_ns` nanoseconds, and tear
 * down as the attention kernels do (with `hold_tmem` != 0, holding all 512 tensor-memory
 * columns of their SM while they wait, freed afterwards).
 *
 *   limit_ns  0 < limit_ns <= 1e9
 *   blocks    1 .. 1024
 *   gave_up   device counter (one unsigned) that every thread whose wait ran out
 *             increments, or NULL
 * On return of the kernel the device error word holds PKV_DEVERR_TIMEOUT
 * (pkv_get_device_error reads and clears it).
 */
pkv_status pkv_selftest_bounded_wait(unsigned long long limit_ns, int blocks, int hold_tmem,
                                     unsigned *gave_up, pkv_stream_t stream);

/*
 * pkv_get_device_error -- synchronise `stream`, then read and clear the device error
 * word of the current device.  *code receives the OR of the PKV_DEVERR_* bits raised
 * since the last clear (0: none).  code is a HOST pointer.
 */
pkv_status pkv_get_device_error(int *code, pkv_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* PKV_H_ */
