// internal.h -- declarations shared by the library's translation units (not the ABI).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "pkv.h"

namespace pkv {

// ------------------------------------------------------------- host helpers

// Encode a 2-D / 3-D bf16 tiled tensor map with 128-byte swizzle.  dims[0] is the
// innermost (contiguous) dimension; strides are the byte strides of dims 1.. .
bool encode_map_bf16(CUtensorMap *map, const void *base, int rank, const uint64_t *dims,
                     const uint64_t *strides_bytes, const uint32_t *box);
// The same for a byte array (FP8 codes).
bool encode_map_u8(CUtensorMap *map, const void *base, int rank, const uint64_t *dims,
                   const uint64_t *strides_bytes, const uint32_t *box);

// Per-device state of the current device (SM count, device error word), set up on
// first use; and recording of the calling thread's pkv_last_error() message.
pkv_status current_device_info(int *sm_count, unsigned **err);
pkv_status record_error(pkv_status status, const char *message);

// ---------------------------------------------------------------- cache ops

cudaError_t launch_kv_append(const void *k_new, const void *v_new, void *k_cache, void *v_cache,
                             int elem_bytes, const int64_t *slot_mapping, int T, int Hkv, int d,
                             int bs, int NB, unsigned *err, cudaStream_t stream);

// FP8 append: new rows (dt PKV_BF16 or PKV_F32) quantised to E4M3 codes + fp32 row scales.
cudaError_t launch_kv_append_fp8(const void *k_new, const void *v_new, pkv_dtype new_dt, uint8_t *k_codes,
                                 uint8_t *v_codes, float *k_scale, float *v_scale,
                                 const int64_t *slot_mapping, int T, int Hkv, int d, int bs, int NB,
                                 unsigned *err, cudaStream_t stream);

cudaError_t launch_kv_block_copy(void *k_cache, void *v_cache, int elem_bytes,
                                 const int32_t *pairs, int n, int Hkv, int d, int bs, int NB,
                                 unsigned *err, cudaStream_t stream);

// ------------------------------------------------------------------ decode

struct DecodePlan {
    bool tensor_core;   // bf16 TMA + mma path; otherwise the CUDA-core path
    bool group;         // tensor-core path with 9..64 query heads per KV head: all head
                        // tiles of a KV head in one CTA sharing each page
    bool umma;          // the large-group case on tcgen05 (d in {64, 128})
    int splits;         // chunks per sequence at most (1: one pass, no workspace)
    int chunk_pages;    // blocks per chunk
    bool fused_merge;   // the last chunk of each unit merges (counters in the workspace)
    size_t counter_bytes = 0;  // bytes of arrival counters a call uses (from the start)
    int sm_count = 0;          // the device's SMs the plan was made for
    size_t workspace_bytes;
    int q_per_tile = 1; // tcgen05 kernel: query rows per block (several queries per sequence)
    int qtiles = 1;     // tcgen05 kernel: query tiles per sequence
    bool paged_prefill = false;   // many query rows per sequence: the chunked-prefill kernel
                                  // (128 rows of one head per block, all keys, no split)
};

// caches_aligned: both cache bases 16-byte aligned; q_aligned: q 16-byte aligned (the
// tcgen05 large-group kernel copies the group's queries in one bulk copy).
DecodePlan plan_decode(int B, int Hq, int Hkv, int d, int bs, int MBS, int NB, pkv_dtype dt,
                       int num_splits, int sm_count, bool caches_aligned, bool q_aligned);

// Several query rows per sequence (pkv_paged_attention with cu_q): Tq rows, at most max_q
// per sequence.  bf16 caches with d in {64, 128}, bs in {16, 32}, aligned caches and q:
// without a window and with at least kPagedPrefillMinRows rows in some sequence, the
// chunked-prefill kernel (paged_prefill.cu); otherwise, with up to 64 heads per KV head,
// the tcgen05 kernel with tiles of floor(64 / m) query rows; other shapes the CUDA-core
// path.  MBS: the blocks any row can see.
constexpr int kPagedPrefillMinRows = 64;
DecodePlan plan_attention_rows(int B, int Tq, int max_q, int Hq, int Hkv, int d, int bs, int MBS, int NB,
                               pkv_dtype dt, int window, int num_splits, int sm_count, bool caches_aligned,
                               bool q_aligned);

// Workspace that covers every plan these shapes can take (element type and alignment
// unknown).
size_t decode_workspace_upper_bound(int B, int Hq, int Hkv, int d, int bs, int MBS,
                                    int num_splits, int sm_count);

struct DecodeArgs {
    float *out;
    float *lse;
    const float *q;
    const void *k_cache;
    const void *v_cache;
    const int32_t *block_table;
    const int32_t *context_lens;
    int B, Hq, Hkv, d, bs, MBS, NB;
    float scale;
    void *workspace;
    unsigned *err;
    int window = 0;                  // > 0: sliding window of this many tokens
    const float *k_scale = nullptr;  // FP8 caches: per-row scales [NB][Hkv][bs]
    const float *v_scale = nullptr;
    const int32_t *cu_q = nullptr;   // query rows per sequence; nullptr: one per sequence
    int rows = -1;                   // query rows (B when cu_q is nullptr)
    // the step's new tokens, appended inside the decode launch (decode_fuses_append)
    const void *k_new = nullptr, *v_new = nullptr;   // [B][Hkv][d], bf16
    const int64_t *new_slots = nullptr;              // [B]; < 0: no new token
    const int32_t *kv_start = nullptr;               // [B]: keys read from this token on (a shared
                                                     // prefix attended elsewhere); nullptr: 0
};

// Whether launch_decode can write the step's new tokens (one per sequence, at its last
// position; rows of type new_dt) inside the decode launch for this plan over a cache of
// type dt; otherwise kv_append (kv_append_fp8) runs first.
bool decode_fuses_append(const DecodePlan &plan, pkv_dtype dt, pkv_dtype new_dt, int Hq, int Hkv,
                         const void *k_new, const void *v_new);

// Blocks a query row can see: all of MBS, or with a window of W tokens at most
// ceil(W / bs) + 1 (the window may start inside a block).
inline int visible_blocks(int MBS, int bs, int window) {
    if (window <= 0) return MBS;
    const long long w = (static_cast<long long>(window) + bs - 1) / bs + 1;
    return static_cast<int>(w < MBS ? w : MBS);
}

cudaError_t launch_decode(const DecodeArgs &a, const DecodePlan &plan, pkv_dtype dt,
                          cudaStream_t stream);

// ----------------------------------------------------------------- prefill

struct PrefillArgs {
    float *out;
    float *lse;
    const void *q, *k, *v;
    const int32_t *cu_seqlens;
    int B, T, max_seqlen, Hq, Hkv, d;
    float scale;
    unsigned *err;
};

bool prefill_tensor_core_ok(pkv_dtype dt, int d, const void *q, const void *k, const void *v,
                            int T, int Hq, int Hkv);

cudaError_t launch_prefill(const PrefillArgs &a, pkv_dtype dt, cudaStream_t stream);

}  // namespace pkv
