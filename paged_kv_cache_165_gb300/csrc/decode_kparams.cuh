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
};

// Sequence length after validation; an invalid length counts as empty.
__device__ __forceinline__ int checked_len(const DecodeKParams &p, int b, int bs, bool report) {
    int len = __ldg(p.context_lens + b);
    if (len < 0 || (long long)len > (long long)p.MBS * bs) {
        if (report) raise_error(p.err, PKV_DEVERR_LEN);
        len = 0;
    }
    return len;
}

// Large-group decode on tcgen05 (decode_umma.cu): d in {64, 128}, bs in {16, 32},
// grid (chunks, Hkv, B).  Key tiles hold this many tokens.
constexpr int kUmmaDecodeKeys = 64;

cudaError_t launch_decode_umma(const DecodeKParams &kp, const CUtensorMap &tk, const CUtensorMap &tv,
                               int d, int bs, dim3 grid, cudaStream_t stream);

}  // namespace pkv
