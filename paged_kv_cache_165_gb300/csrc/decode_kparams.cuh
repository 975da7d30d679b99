// decode_kparams.cuh -- kernel parameters and helpers shared by the decode kernels of
// decode.cu and decode_umma.cu (not part of the ABI).
#pragma once

#include "common.cuh"
#include "internal.h"

namespace pkv {

constexpr float kDecLog2e = 1.4426950408889634f;
constexpr float kDecLn2 = 0.6931471805599453f;

struct DecodeKParams {
    float *out;
    float *lse;
    float *ws_o;         // partial outputs [B*Hq][splits][d], normalised
    float *ws_lse;       // partial log-sum-exp [B*Hq][splits], base 2
    unsigned *counters;  // arrival counters, one per (sequence, KV head, head tile) unit
    const float *q;
    const int32_t *block_table;
    const int32_t *context_lens;
    unsigned *err;
    int B, Hq, Hkv, m, MBS, NB;
    int head_tiles;   // ceil(m / 8): head groups per KV head
    int chunk_pages;  // blocks per chunk
    int splits;       // chunks per sequence at most (partial slots per sequence)
    float scale_log2; // scale * log2(e): scores are kept in the base-2 domain
    int window;       // > 0: only the most recent `window` tokens are visible
    const int32_t *cu_q;   // query rows per sequence [B+1]; nullptr: row b = sequence b
    const float *k_scale, *v_scale;   // FP8 caches: fp32 scale per row [NB][Hkv][bs]
    int q_per_tile;   // tcgen05 kernel: query rows of a sequence per block (1 for decode)
    int qtiles;       // tcgen05 kernel: query tiles per sequence (grid z = B * qtiles)
    int longest_first;   // tcgen05 kernel: grid z ranks the sequences by length, longest first
    // the step's new tokens written inside the chunked kernel (nullptr: appended before)
    const void *k_new, *v_new;   // [B][Hkv][d] (bf16)
    const int64_t *new_slots;    // [B]; < 0: no new token
    void *k_cache_w, *v_cache_w; // the caches (FP8: the codes), for those writes
    float *k_scale_w, *v_scale_w;   // FP8 caches: the row scales, for those writes
    // shared prefixes (pkv_decode_step_shared_prefix): sequence b's first kv_start[b] tokens
    // are its group's shared prefix, attended by the prefix kernel; the decode kernels read
    // keys from kv_start[b] on (nullptr: from 0)
    const int32_t *kv_start;
    const int32_t *group_seqs;   // prefix kernel: the member sequences of each group (cu_q: offsets)
    int prefix_splits;           // prefix kernel: key splits of a group's prefix
    int prefix_rtiles;           // prefix kernel: 128-row tiles of (member, head) rows per group
    int n_members;               // prefix kernel: entries of group_seqs (group offsets must stay within)
};

// The step's new token, written by one warp of the block that reads sequence b's last page
// (pkv_decode_step with the append inside the decode launch): K and V rows of KV head kvh
// from k_new/v_new [B][Hkv][D] (bf16, 16-byte aligned) into the slot of position len - 1.
// A slot that is not that position's is flagged and not written.  The caller fences the
// writes for the asynchronous proxy and syncs the block before the page's TMA copies.
template <int D, int BS>
__device__ __forceinline__ void write_new_token(const DecodeKParams &p, int b, int kvh, int len, int lane) {
    const long long slot = __ldg(p.new_slots + b);
    if (slot < 0) return;                                  // no new token this step
    const int pos = len - 1;
    const int phys = pos >= 0 ? __ldg(p.block_table + static_cast<size_t>(b) * p.MBS + pos / BS) : -1;
    if (phys < 0 || phys >= p.NB || slot != static_cast<long long>(phys) * BS + pos % BS) {
        if (lane == 0) raise_error(p.err, PKV_DEVERR_SLOT);
        return;
    }
    const size_t src = (static_cast<size_t>(b) * p.Hkv + kvh) * D;
    const size_t dst = ((static_cast<size_t>(phys) * p.Hkv + kvh) * BS + pos % BS) * D;
    const uint4 *kn = reinterpret_cast<const uint4 *>(static_cast<const uint16_t *>(p.k_new) + src);
    const uint4 *vn = reinterpret_cast<const uint4 *>(static_cast<const uint16_t *>(p.v_new) + src);
    uint4 *kd = reinterpret_cast<uint4 *>(static_cast<uint16_t *>(p.k_cache_w) + dst);
    uint4 *vd = reinterpret_cast<uint4 *>(static_cast<uint16_t *>(p.v_cache_w) + dst);
    for (int u = lane; u < D / 8; u += 32) {
        kd[u] = __ldg(kn + u);
        vd[u] = __ldg(vn + u);
    }
}

// Sequence length after validation; an invalid length counts as empty.
__device__ __forceinline__ int checked_len(const DecodeKParams &p, int b, int bs, bool report) {
    int len = __ldg(p.context_lens + b);
    if (len < 0 || (long long)len > (long long)p.MBS * bs) {
        if (report) raise_error(p.err, PKV_DEVERR_LEN);
        len = 0;
    }
    return len;
}

// The keys a query row sees: tokens [lo, len) of sequence b, on pages [pfirst, pfirst +
// npages).  A row is the token at position len - 1 of its sequence (the decode query,
// row b = sequence b), or with query rows cu_q the i-th of the nq rows of sequence b,
// at position L - nq + i: `len` is then that position + 1 (causal, aligned to the end
// of the cache).  With a sliding window of W tokens, lo = max(0, len - W), the most
// recent W positions; blocks before pfirst are never read and may have been freed.
// Chunks of a sequence cover the pages [cpfirst, cpfirst + cnpages) that any of its query
// rows sees (the same boundaries for every row, so that chunk partials line up); a row
// whose own keys miss a chunk writes an empty partial there.
struct SeqSpan {
    int b, len, lo, pfirst, npages;
    int cpfirst, cnpages;
};

__device__ __forceinline__ SeqSpan span_of(const DecodeKParams &p, int b, int len, int bs) {
    SeqSpan s;
    s.b = b;
    s.len = len;
    s.lo = p.window > 0 ? max(0, len - p.window) : 0;
    // a shared prefix read elsewhere: keys from kv_start[b] on, the last token always kept
    if (p.kv_start != nullptr && len > 0) s.lo = max(s.lo, min(__ldg(p.kv_start + b), len - 1));
    s.pfirst = s.lo / bs;
    s.npages = len > 0 ? (len + bs - 1) / bs - s.pfirst : 0;
    s.cpfirst = s.pfirst;
    s.cnpages = s.npages;
    return s;
}

__device__ __forceinline__ SeqSpan seq_span(const DecodeKParams &p, int b, int bs, bool report) {
    return span_of(p, b, checked_len(p, b, bs, report), bs);
}

// Query row r (cu_q != nullptr): its sequence by binary search over cu_q, its position,
// its span.  An inconsistent cu_q or a row count above the sequence length raises
// PKV_DEVERR_CU_SEQLENS and the row sees nothing (out = 0, lse = -inf).
__device__ __forceinline__ SeqSpan row_span(const DecodeKParams &p, int r, int bs, bool report) {
    if (p.cu_q == nullptr) return seq_span(p, r, bs, report);
    int lo = 0, hi = p.B;   // find b with cu_q[b] <= r < cu_q[b+1]
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (__ldg(p.cu_q + mid) <= r) lo = mid;
        else hi = mid;
    }
    const int b = lo;
    const int c0 = __ldg(p.cu_q + b), c1 = __ldg(p.cu_q + b + 1);
    const int L = checked_len(p, b, bs, report);
    const int nq = c1 - c0;
    if (r < c0 || r >= c1 || nq > L) {
        if (report) raise_error(p.err, PKV_DEVERR_CU_SEQLENS);
        return span_of(p, b, 0, bs);
    }
    SeqSpan s = span_of(p, b, L - nq + (r - c0) + 1, bs);
    // the sequence's chunk range: from the first row's window start to the last key
    const SeqSpan first = span_of(p, b, L - nq + 1, bs);
    s.cpfirst = first.pfirst;
    s.cnpages = (L + bs - 1) / bs - first.pfirst;
    return s;
}

// Large-group decode on tcgen05 (decode_umma.cu): d in {64, 128}, bs in {16, 32},
// grid (chunks, Hkv, B).  Key tiles hold this many tokens.
constexpr int kUmmaDecodeKeys = 128;

cudaError_t launch_decode_umma(const DecodeKParams &kp, const CUtensorMap &tk, const CUtensorMap &tv,
                               int d, int bs, dim3 grid, cudaStream_t stream);

// Chunked prefill over a paged cache (paged_prefill.cu): bf16 caches, d in {64, 128}, bs in
// {16, 32}, query rows cu_q; grid (query tiles of 128 rows, Hq, B); one pass, no workspace.
cudaError_t launch_paged_prefill(const DecodeKParams &kp, const CUtensorMap &tk, const CUtensorMap &tv, int d,
                                 int bs, dim3 grid, cudaStream_t stream);

// Shared prefixes (paged_prefill.cu): the attention of every member's query heads over its
// group's prefix, one partial per key split into ws_o / ws_lse indexed by member (cu_q:
// group offsets, group_seqs: members, kv_start: prefix tokens); grid (prefix_splits, Hkv,
// groups * prefix_rtiles).  Then the merge of each member's partials with its suffix result
// (out / lse as the decode wrote them, lse in natural log in suffix_lse), one warp per
// (member, head), in place into out (and lse when not null; suffix_lse may be lse itself).
cudaError_t launch_shared_prefix(const DecodeKParams &kp, const CUtensorMap &tk, const CUtensorMap &tv, int d,
                                 int bs, dim3 grid, cudaStream_t stream);
cudaError_t launch_shared_prefix_merge(const DecodeKParams &kp, const float *suffix_lse, int d, int bs,
                                       int n_groups, int n_members, cudaStream_t stream);

// FP8 (E4M3) decode (decode_fp8.cu): d = 128, bs in {16, 32}, up to 8 query heads per KV
// head; grid (chunks x head tiles, Hkv, B).  tk / tv are uint8 maps with {128, bs} boxes.
cudaError_t launch_decode_fp8(const DecodeKParams &kp, const CUtensorMap &tk, const CUtensorMap &tv, int bs,
                              dim3 grid, cudaStream_t stream);

}  // namespace pkv
