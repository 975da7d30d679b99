// api.cu -- the extern "C" entry points declared in include/pkv.h.
//
// Every entry point validates its host-side arguments before enqueueing anything,
// maps CUDA failures to PKV_ERR_CUDA, and records a message for pkv_last_error().
// Per-device state is limited to the SM count and the address of the device error
// word (a static __device__ variable: nothing is allocated).
#include <algorithm>
#include <cudaTypedefs.h>

#include <cstdarg>
#include <cstdio>
#include <mutex>

#include "common.cuh"
#include "decode_kparams.cuh"
#include "internal.h"

namespace pkv {
namespace {

__device__ unsigned g_device_error;   // OR of PKV_DEVERR_* bits, one word per device

thread_local char t_last_error[256] = "";

pkv_status fail(pkv_status s, const char *fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(t_last_error, sizeof t_last_error, fmt, ap);
    va_end(ap);
    return s;
}

pkv_status cuda_fail(cudaError_t e, const char *where) {
    return fail(PKV_ERR_CUDA, "%s: %s", where, cudaGetErrorString(e));
}

struct DeviceState {
    bool ready = false;
    int sm_count = 0;
    unsigned *err = nullptr;
};

constexpr int kMaxDevices = 64;
DeviceState g_devices[kMaxDevices];
std::mutex g_mutex;

// State of the current device, set up on first use.
pkv_status device_state(DeviceState **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices) return fail(PKV_ERR_UNSUPPORTED, "device ordinal %d", dev);
    DeviceState &st = g_devices[dev];
    std::lock_guard<std::mutex> lock(g_mutex);
    if (!st.ready) {
        e = cudaDeviceGetAttribute(&st.sm_count, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute");
        e = cudaGetSymbolAddress(reinterpret_cast<void **>(&st.err), g_device_error);
        if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(device error word)");
        st.ready = true;
    }
    *out = &st;
    return PKV_OK;
}

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

bool elem_size(pkv_dtype dt, int *bytes) {
    if (dt == PKV_F32) { *bytes = 4; return true; }
    if (dt == PKV_BF16) { *bytes = 2; return true; }
    if (dt == PKV_FP8_E4M3) { *bytes = 1; return true; }
    return false;
}

// Attention over values of the cache's own type (FP8 needs its scales: the _fp8 entry).
bool attention_dtype(pkv_dtype dt) { return dt == PKV_F32 || dt == PKV_BF16; }

bool aligned16(const void *p) { return reinterpret_cast<uintptr_t>(p) % 16 == 0; }

}  // namespace

namespace {

bool encode_map(CUtensorMapDataType type, CUtensorMap *map, const void *base, int rank,
                const uint64_t *dims, const uint64_t *strides_bytes, const uint32_t *box) {
    std::call_once(g_encode_once, [] {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    });
    if (g_encode == nullptr) return false;
    cuuint64_t gdim[5];
    cuuint64_t gstride[4];
    cuuint32_t bdim[5], estride[5];
    for (int r = 0; r < rank; ++r) {
        gdim[r] = dims[r];
        bdim[r] = box[r];
        estride[r] = 1;
        if (r + 1 < rank) gstride[r] = strides_bytes[r];
    }
    const CUresult res = g_encode(map, type, rank, const_cast<void *>(base), gdim, gstride, bdim,
                                  estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return res == CUDA_SUCCESS;
}

}  // namespace

bool encode_map_bf16(CUtensorMap *map, const void *base, int rank, const uint64_t *dims,
                     const uint64_t *strides_bytes, const uint32_t *box) {
    return encode_map(CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, map, base, rank, dims, strides_bytes, box);
}

bool encode_map_u8(CUtensorMap *map, const void *base, int rank, const uint64_t *dims,
                   const uint64_t *strides_bytes, const uint32_t *box) {
    return encode_map(CU_TENSOR_MAP_DATA_TYPE_UINT8, map, base, rank, dims, strides_bytes, box);
}

pkv_status current_device_info(int *sm_count, unsigned **err) {
    DeviceState *st = nullptr;
    const pkv_status s = device_state(&st);
    if (s != PKV_OK) return s;
    *sm_count = st->sm_count;
    *err = st->err;
    return PKV_OK;
}

pkv_status record_error(pkv_status status, const char *message) {
    return fail(status, "%s", message);
}

}  // namespace pkv

using namespace pkv;

extern "C" {

const char *pkv_status_string(pkv_status status) {
    switch (status) {
        case PKV_OK: return "ok";
        case PKV_ERR_INVALID_ARG: return "invalid argument";
        case PKV_ERR_UNSUPPORTED: return "unsupported";
        case PKV_ERR_WORKSPACE: return "workspace missing or too small";
        case PKV_ERR_CUDA: return "CUDA error";
    }
    return "unknown status";
}

const char *pkv_last_error(void) { return t_last_error; }

int pkv_version(void) { return 10000; }

pkv_status pkv_kv_append(const void *k_new, const void *v_new, void *k_cache, void *v_cache,
                         pkv_dtype dt, const int64_t *slot_mapping, int T, int Hkv, int d, int bs,
                         int NB, pkv_stream_t stream) {
    int eb = 0;
    if (!elem_size(dt, &eb)) return fail(PKV_ERR_UNSUPPORTED, "kv_append: element type %d", dt);
    if (T < 0 || Hkv < 1 || d < 1 || bs < 1 || NB < 1)
        return fail(PKV_ERR_INVALID_ARG, "kv_append: T=%d Hkv=%d d=%d bs=%d NB=%d", T, Hkv, d, bs, NB);
    if (T == 0) return PKV_OK;
    if (!k_new || !v_new || !k_cache || !v_cache || !slot_mapping)
        return fail(PKV_ERR_INVALID_ARG, "kv_append: null pointer");
    DeviceState *st = nullptr;
    pkv_status s = device_state(&st);
    if (s != PKV_OK) return s;
    cudaError_t e = launch_kv_append(k_new, v_new, k_cache, v_cache, eb, slot_mapping, T, Hkv, d,
                                     bs, NB, st->err, stream);
    return e == cudaSuccess ? PKV_OK : cuda_fail(e, "kv_append launch");
}

pkv_status pkv_kv_block_copy(void *k_cache, void *v_cache, pkv_dtype dt, const int32_t *pairs,
                             int n, int Hkv, int d, int bs, int NB, pkv_stream_t stream) {
    int eb = 0;
    if (!elem_size(dt, &eb)) return fail(PKV_ERR_UNSUPPORTED, "kv_block_copy: element type %d", dt);
    if (n < 0 || Hkv < 1 || d < 1 || bs < 1 || NB < 1)
        return fail(PKV_ERR_INVALID_ARG, "kv_block_copy: n=%d Hkv=%d d=%d bs=%d NB=%d", n, Hkv, d, bs, NB);
    if (n == 0) return PKV_OK;
    if (!k_cache || !v_cache || !pairs) return fail(PKV_ERR_INVALID_ARG, "kv_block_copy: null pointer");
    DeviceState *st = nullptr;
    pkv_status s = device_state(&st);
    if (s != PKV_OK) return s;
    cudaError_t e = launch_kv_block_copy(k_cache, v_cache, eb, pairs, n, Hkv, d, bs, NB, st->err, stream);
    return e == cudaSuccess ? PKV_OK : cuda_fail(e, "kv_block_copy launch");
}

static pkv_status check_decode_sizes(int B, int Hq, int Hkv, int d, int bs, int MBS) {
    if (B < 0 || B > 65535 || Hq < 1 || Hq > 65535 || Hkv < 1 || Hq % Hkv != 0 || d < 1 ||
        d > 256 || bs < 1 || MBS < 1)
        return fail(PKV_ERR_INVALID_ARG,
                    "paged_decode_attention: B=%d Hq=%d Hkv=%d d=%d bs=%d MBS=%d (need 0<=B<=65535, "
                    "Hq %% Hkv == 0, 1<=d<=256, bs>=1, MBS>=1)",
                    B, Hq, Hkv, d, bs, MBS);
    return PKV_OK;
}

size_t pkv_decode_workspace_bytes(int B, int Hq, int Hkv, int d, int bs, int MBS, int num_splits) {
    if (check_decode_sizes(B, Hq, Hkv, d, bs, MBS) != PKV_OK || num_splits < 0) return 0;
    DeviceState *st = nullptr;
    if (device_state(&st) != PKV_OK) return 0;
    return decode_workspace_upper_bound(B, Hq, Hkv, d, bs, MBS, num_splits, st->sm_count);
}

int pkv_decode_kernel_launches(int B, int Hq, int Hkv, int d, int bs, int MBS, int NB, pkv_dtype dt,
                               int num_splits) {
    int eb = 0;
    if (!elem_size(dt, &eb) || check_decode_sizes(B, Hq, Hkv, d, bs, MBS) != PKV_OK || NB < 1 ||
        num_splits < 0)
        return -1;
    if (B == 0) return 0;
    DeviceState *st = nullptr;
    if (device_state(&st) != PKV_OK) return -1;
    const DecodePlan plan = plan_decode(B, Hq, Hkv, d, bs, MBS, NB, dt, num_splits, st->sm_count, true, true);
    return plan.splits > 1 && !plan.fused_merge ? 2 : 1;
}

int pkv_paged_attention_kernel_launches(int B, int Tq, int max_q, int Hq, int Hkv, int d, int bs,
                                        int MBS, int NB, pkv_dtype dt, int window, int num_splits) {
    int eb = 0;
    if (!elem_size(dt, &eb) || check_decode_sizes(B, Hq, Hkv, d, bs, MBS) != PKV_OK || NB < 1 ||
        num_splits < 0 || window < 0 || Tq < 0 || max_q < 0 ||
        static_cast<long long>(Tq) > static_cast<long long>(B) * max_q)
        return -1;
    if (B == 0 || Tq == 0) return 0;
    DeviceState *st = nullptr;
    if (device_state(&st) != PKV_OK) return -1;
    const bool one_per_seq = Tq == B && max_q == 1;
    const DecodePlan plan =
        one_per_seq
            ? plan_decode(B, Hq, Hkv, d, bs, visible_blocks(MBS, bs, window), NB, dt, num_splits, st->sm_count,
                          true, true)
            : plan_attention_rows(B, Tq, max_q, Hq, Hkv, d, bs,
                                  visible_blocks(MBS, bs, window > 0 ? window + max_q - 1 : 0), NB, dt, window,
                                  num_splits, st->sm_count, true, true);
    return plan.splits > 1 && !plan.fused_merge ? 2 : 1;
}

pkv_status pkv_paged_decode_attention(float *out, float *lse, const float *q, const void *k_cache,
                                      const void *v_cache, pkv_dtype dt, const int32_t *block_table,
                                      const int32_t *context_lens, int B, int Hq, int Hkv, int d,
                                      int bs, int MBS, int NB, float scale, int num_splits,
                                      void *workspace, size_t workspace_bytes, pkv_stream_t stream) {
    int eb = 0;
    if (!elem_size(dt, &eb) || !attention_dtype(dt))
        return fail(PKV_ERR_UNSUPPORTED, "paged_decode_attention: element type %d", dt);
    pkv_status s = check_decode_sizes(B, Hq, Hkv, d, bs, MBS);
    if (s != PKV_OK) return s;
    if (NB < 1 || num_splits < 0)
        return fail(PKV_ERR_INVALID_ARG, "paged_decode_attention: NB=%d num_splits=%d", NB, num_splits);
    if (B == 0) return PKV_OK;
    if (!out || !q || !k_cache || !v_cache || !block_table || !context_lens)
        return fail(PKV_ERR_INVALID_ARG, "paged_decode_attention: null pointer");
    if (reinterpret_cast<uintptr_t>(q) % 8 != 0)
        return fail(PKV_ERR_INVALID_ARG, "paged_decode_attention: q must be 8-byte aligned");
    DeviceState *st = nullptr;
    s = device_state(&st);
    if (s != PKV_OK) return s;
    const DecodePlan plan = plan_decode(B, Hq, Hkv, d, bs, MBS, NB, dt, num_splits, st->sm_count,
                                        aligned16(k_cache) && aligned16(v_cache), aligned16(q));
    if (plan.workspace_bytes > 0 &&
        (workspace == nullptr || workspace_bytes < plan.workspace_bytes ||
         reinterpret_cast<uintptr_t>(workspace) % 16 != 0))
        return fail(PKV_ERR_WORKSPACE,
                    "paged_decode_attention: needs %zu bytes of 16-byte aligned workspace, got %zu",
                    plan.workspace_bytes, workspace == nullptr ? size_t(0) : workspace_bytes);
    DecodeArgs a{out, lse, q, k_cache, v_cache, block_table, context_lens,
                 B, Hq, Hkv, d, bs, MBS, NB, scale, workspace, st->err};
    cudaError_t e = launch_decode(a, plan, dt, stream);
    return e == cudaSuccess ? PKV_OK : cuda_fail(e, "paged_decode_attention launch");
}

pkv_status pkv_decode_step(float *out, float *lse, const float *q, const void *k_new, const void *v_new,
                           const int64_t *slot_mapping, void *k_cache, void *v_cache, pkv_dtype dt,
                           const int32_t *block_table, const int32_t *context_lens, int B, int Hq,
                           int Hkv, int d, int bs, int MBS, int NB, float scale, int num_splits,
                           void *workspace, size_t workspace_bytes, pkv_stream_t stream) {
    int eb = 0;
    if (!elem_size(dt, &eb) || !attention_dtype(dt))
        return fail(PKV_ERR_UNSUPPORTED, "decode_step: element type %d", dt);
    pkv_status s = check_decode_sizes(B, Hq, Hkv, d, bs, MBS);
    if (s != PKV_OK) return s;
    if (NB < 1 || num_splits < 0)
        return fail(PKV_ERR_INVALID_ARG, "decode_step: NB=%d num_splits=%d", NB, num_splits);
    if (B == 0) return PKV_OK;
    if (!out || !q || !k_new || !v_new || !slot_mapping || !k_cache || !v_cache || !block_table ||
        !context_lens)
        return fail(PKV_ERR_INVALID_ARG, "decode_step: null pointer");
    if (reinterpret_cast<uintptr_t>(q) % 8 != 0)
        return fail(PKV_ERR_INVALID_ARG, "decode_step: q must be 8-byte aligned");
    DeviceState *st = nullptr;
    s = device_state(&st);
    if (s != PKV_OK) return s;
    const DecodePlan plan = plan_decode(B, Hq, Hkv, d, bs, MBS, NB, dt, num_splits, st->sm_count,
                                        aligned16(k_cache) && aligned16(v_cache), aligned16(q));
    if (plan.workspace_bytes > 0 &&
        (workspace == nullptr || workspace_bytes < plan.workspace_bytes ||
         reinterpret_cast<uintptr_t>(workspace) % 16 != 0))
        return fail(PKV_ERR_WORKSPACE, "decode_step: needs %zu bytes of 16-byte aligned workspace, got %zu",
                    plan.workspace_bytes, workspace == nullptr ? size_t(0) : workspace_bytes);
    DecodeArgs a{out, lse, q, k_cache, v_cache, block_table, context_lens,
                 B, Hq, Hkv, d, bs, MBS, NB, scale, workspace, st->err};
    cudaError_t e = cudaSuccess;
    if (decode_fuses_append(plan, dt, dt, Hq, Hkv, k_new, v_new)) {
        a.k_new = k_new;
        a.v_new = v_new;
        a.new_slots = slot_mapping;
    } else {
        e = launch_kv_append(k_new, v_new, k_cache, v_cache, eb, slot_mapping, B, Hkv, d, bs, NB, st->err,
                             stream);
        if (e != cudaSuccess) return cuda_fail(e, "decode_step append launch");
    }
    e = launch_decode(a, plan, dt, stream);
    return e == cudaSuccess ? PKV_OK : cuda_fail(e, "decode_step launch");
}

int pkv_decode_step_kernel_launches(int B, int Hq, int Hkv, int d, int bs, int MBS, int NB, pkv_dtype dt,
                                    int num_splits) {
    const int n = pkv_decode_kernel_launches(B, Hq, Hkv, d, bs, MBS, NB, dt, num_splits);
    if (n <= 0) return n;
    DeviceState *st = nullptr;
    if (device_state(&st) != PKV_OK) return -1;
    const DecodePlan plan = plan_decode(B, Hq, Hkv, d, bs, MBS, NB, dt, num_splits, st->sm_count, true, true);
    // new rows from a 16-byte aligned allocation (as tensors are)
    static const uint4 aligned{};
    return n + (decode_fuses_append(plan, dt, dt, Hq, Hkv, &aligned, &aligned) ? 0 : 1);
}

size_t pkv_paged_attention_workspace_bytes(int B, int Tq, int max_q, int Hq, int Hkv, int d, int bs,
                                           int MBS, int window, int num_splits) {
    if (check_decode_sizes(B, Hq, Hkv, d, bs, MBS) != PKV_OK || Tq < 0 || max_q < 0 || window < 0 ||
        num_splits < 0)
        return 0;
    DeviceState *st = nullptr;
    if (device_state(&st) != PKV_OK) return 0;
    if (Tq == B && max_q <= 1)
        return decode_workspace_upper_bound(B, Hq, Hkv, d, bs, visible_blocks(MBS, bs, window), num_splits,
                                            st->sm_count);
    // query rows: cover the tcgen05 and the CUDA-core plans
    const int vis = visible_blocks(MBS, bs, window > 0 ? window + max_q - 1 : 0);
    return std::max(plan_attention_rows(B, Tq, max_q, Hq, Hkv, d, bs, vis, 1, PKV_BF16, window, num_splits,
                                        st->sm_count, true, true).workspace_bytes,
                    plan_attention_rows(B, Tq, max_q, Hq, Hkv, d, bs, vis, 1, PKV_F32, window, num_splits,
                                        st->sm_count, false, false).workspace_bytes);
}

pkv_status pkv_paged_attention(float *out, float *lse, const float *q, const void *k_cache,
                               const void *v_cache, pkv_dtype dt, const int32_t *block_table,
                               const int32_t *context_lens, const int32_t *cu_q, int B, int Tq,
                               int max_q, int Hq, int Hkv, int d, int bs, int MBS, int NB, float scale,
                               int window, int num_splits, void *workspace, size_t workspace_bytes,
                               pkv_stream_t stream) {
    int eb = 0;
    if (!elem_size(dt, &eb) || !attention_dtype(dt))
        return fail(PKV_ERR_UNSUPPORTED, "paged_attention: element type %d", dt);
    pkv_status s = check_decode_sizes(B, Hq, Hkv, d, bs, MBS);
    if (s != PKV_OK) return s;
    if (NB < 1 || num_splits < 0 || window < 0 || Tq < 0 || max_q < 0 ||
        static_cast<long long>(Tq) > static_cast<long long>(B) * max_q ||
        static_cast<long long>(Tq) * Hq > 0x7fffffffll)
        return fail(PKV_ERR_INVALID_ARG, "paged_attention: NB=%d num_splits=%d window=%d Tq=%d max_q=%d",
                    NB, num_splits, window, Tq, max_q);
    if (B == 0 || Tq == 0) return PKV_OK;
    const bool one_per_seq = Tq == B && max_q == 1;
    if (!out || !q || !k_cache || !v_cache || !block_table || !context_lens || (!one_per_seq && !cu_q))
        return fail(PKV_ERR_INVALID_ARG, "paged_attention: null pointer");
    if (reinterpret_cast<uintptr_t>(q) % 8 != 0)
        return fail(PKV_ERR_INVALID_ARG, "paged_attention: q must be 8-byte aligned");
    DeviceState *st = nullptr;
    s = device_state(&st);
    if (s != PKV_OK) return s;
    const bool caches_aligned = aligned16(k_cache) && aligned16(v_cache);
    const DecodePlan plan =
        one_per_seq
            ? plan_decode(B, Hq, Hkv, d, bs, visible_blocks(MBS, bs, window), NB, dt, num_splits, st->sm_count,
                          caches_aligned, aligned16(q))
            : plan_attention_rows(B, Tq, max_q, Hq, Hkv, d, bs,
                                  visible_blocks(MBS, bs, window > 0 ? window + max_q - 1 : 0), NB, dt, window,
                                  num_splits, st->sm_count, caches_aligned, aligned16(q));
    if (plan.workspace_bytes > 0 &&
        (workspace == nullptr || workspace_bytes < plan.workspace_bytes ||
         reinterpret_cast<uintptr_t>(workspace) % 16 != 0))
        return fail(PKV_ERR_WORKSPACE,
                    "paged_attention: needs %zu bytes of 16-byte aligned workspace, got %zu",
                    plan.workspace_bytes, workspace == nullptr ? size_t(0) : workspace_bytes);
    DecodeArgs a{out, lse, q, k_cache, v_cache, block_table, context_lens,
                 B, Hq, Hkv, d, bs, MBS, NB, scale, workspace, st->err};
    a.window = window;
    a.cu_q = one_per_seq ? nullptr : cu_q;
    a.rows = one_per_seq ? B : Tq;
    cudaError_t e = launch_decode(a, plan, dt, stream);
    return e == cudaSuccess ? PKV_OK : cuda_fail(e, "paged_attention launch");
}

pkv_status pkv_kv_append_fp8(const void *k_new, const void *v_new, pkv_dtype new_dt, uint8_t *k_codes,
                             uint8_t *v_codes, float *k_scale, float *v_scale, const int64_t *slot_mapping,
                             int T, int Hkv, int d, int bs, int NB, pkv_stream_t stream) {
    if (!attention_dtype(new_dt)) return fail(PKV_ERR_UNSUPPORTED, "kv_append_fp8: input type %d", new_dt);
    if (T < 0 || Hkv < 1 || d < 1 || d > 256 || bs < 1 || NB < 1)
        return fail(PKV_ERR_INVALID_ARG, "kv_append_fp8: T=%d Hkv=%d d=%d bs=%d NB=%d", T, Hkv, d, bs, NB);
    if (T == 0) return PKV_OK;
    if (!k_new || !v_new || !k_codes || !v_codes || !k_scale || !v_scale || !slot_mapping)
        return fail(PKV_ERR_INVALID_ARG, "kv_append_fp8: null pointer");
    DeviceState *st = nullptr;
    pkv_status s = device_state(&st);
    if (s != PKV_OK) return s;
    const cudaError_t e = launch_kv_append_fp8(k_new, v_new, new_dt, k_codes, v_codes, k_scale, v_scale,
                                               slot_mapping, T, Hkv, d, bs, NB, st->err, stream);
    return e == cudaSuccess ? PKV_OK : cuda_fail(e, "kv_append_fp8 launch");
}

pkv_status pkv_paged_decode_attention_fp8(float *out, float *lse, const float *q, const uint8_t *k_codes,
                                          const uint8_t *v_codes, const float *k_scale, const float *v_scale,
                                          const int32_t *block_table, const int32_t *context_lens, int B,
                                          int Hq, int Hkv, int d, int bs, int MBS, int NB, float scale,
                                          int window, int num_splits, void *workspace,
                                          size_t workspace_bytes, pkv_stream_t stream) {
    pkv_status s = check_decode_sizes(B, Hq, Hkv, d, bs, MBS);
    if (s != PKV_OK) return s;
    if (NB < 1 || num_splits < 0 || window < 0)
        return fail(PKV_ERR_INVALID_ARG, "paged_decode_attention_fp8: NB=%d num_splits=%d window=%d", NB,
                    num_splits, window);
    if (B == 0) return PKV_OK;
    if (!out || !q || !k_codes || !v_codes || !k_scale || !v_scale || !block_table || !context_lens)
        return fail(PKV_ERR_INVALID_ARG, "paged_decode_attention_fp8: null pointer");
    if (reinterpret_cast<uintptr_t>(q) % 8 != 0)
        return fail(PKV_ERR_INVALID_ARG, "paged_decode_attention_fp8: q must be 8-byte aligned");
    DeviceState *st = nullptr;
    s = device_state(&st);
    if (s != PKV_OK) return s;
    const bool aligned = aligned16(k_codes) && aligned16(v_codes) && aligned16(k_scale) && aligned16(v_scale);
    const DecodePlan plan = plan_decode(B, Hq, Hkv, d, bs, visible_blocks(MBS, bs, window), NB, PKV_FP8_E4M3,
                                        num_splits, st->sm_count, aligned, aligned16(q));
    if (plan.workspace_bytes > 0 &&
        (workspace == nullptr || workspace_bytes < plan.workspace_bytes ||
         reinterpret_cast<uintptr_t>(workspace) % 16 != 0))
        return fail(PKV_ERR_WORKSPACE,
                    "paged_decode_attention_fp8: needs %zu bytes of 16-byte aligned workspace, got %zu",
                    plan.workspace_bytes, workspace == nullptr ? size_t(0) : workspace_bytes);
    DecodeArgs a{out, lse, q, k_codes, v_codes, block_table, context_lens,
                 B, Hq, Hkv, d, bs, MBS, NB, scale, workspace, st->err};
    a.window = window;
    a.k_scale = k_scale;
    a.v_scale = v_scale;
    cudaError_t e = launch_decode(a, plan, PKV_FP8_E4M3, stream);
    return e == cudaSuccess ? PKV_OK : cuda_fail(e, "paged_decode_attention_fp8 launch");
}

pkv_status pkv_decode_step_fp8(float *out, float *lse, const float *q, const void *k_new, const void *v_new,
                               pkv_dtype new_dt, const int64_t *slot_mapping, uint8_t *k_codes, uint8_t *v_codes,
                               float *k_scale, float *v_scale, const int32_t *block_table,
                               const int32_t *context_lens, int B, int Hq, int Hkv, int d, int bs, int MBS,
                               int NB, float scale, int num_splits, void *workspace, size_t workspace_bytes,
                               pkv_stream_t stream) {
    if (!attention_dtype(new_dt)) return fail(PKV_ERR_UNSUPPORTED, "decode_step_fp8: input type %d", new_dt);
    pkv_status s = check_decode_sizes(B, Hq, Hkv, d, bs, MBS);
    if (s != PKV_OK) return s;
    if (NB < 1 || num_splits < 0)
        return fail(PKV_ERR_INVALID_ARG, "decode_step_fp8: NB=%d num_splits=%d", NB, num_splits);
    if (B == 0) return PKV_OK;
    if (!out || !q || !k_new || !v_new || !slot_mapping || !k_codes || !v_codes || !k_scale || !v_scale ||
        !block_table || !context_lens)
        return fail(PKV_ERR_INVALID_ARG, "decode_step_fp8: null pointer");
    if (reinterpret_cast<uintptr_t>(q) % 8 != 0)
        return fail(PKV_ERR_INVALID_ARG, "decode_step_fp8: q must be 8-byte aligned");
    DeviceState *st = nullptr;
    s = device_state(&st);
    if (s != PKV_OK) return s;
    const bool aligned = aligned16(k_codes) && aligned16(v_codes) && aligned16(k_scale) && aligned16(v_scale);
    const DecodePlan plan = plan_decode(B, Hq, Hkv, d, bs, MBS, NB, PKV_FP8_E4M3, num_splits, st->sm_count,
                                        aligned, aligned16(q));
    if (plan.workspace_bytes > 0 &&
        (workspace == nullptr || workspace_bytes < plan.workspace_bytes ||
         reinterpret_cast<uintptr_t>(workspace) % 16 != 0))
        return fail(PKV_ERR_WORKSPACE, "decode_step_fp8: needs %zu bytes of 16-byte aligned workspace, got %zu",
                    plan.workspace_bytes, workspace == nullptr ? size_t(0) : workspace_bytes);
    DecodeArgs a{out, lse, q, k_codes, v_codes, block_table, context_lens,
                 B, Hq, Hkv, d, bs, MBS, NB, scale, workspace, st->err};
    a.k_scale = k_scale;
    a.v_scale = v_scale;
    cudaError_t e = cudaSuccess;
    if (decode_fuses_append(plan, PKV_FP8_E4M3, new_dt, Hq, Hkv, k_new, v_new)) {
        a.k_new = k_new;
        a.v_new = v_new;
        a.new_slots = slot_mapping;
    } else {
        e = launch_kv_append_fp8(k_new, v_new, new_dt, k_codes, v_codes, k_scale, v_scale, slot_mapping, B, Hkv, d,
                                 bs, NB, st->err, stream);
        if (e != cudaSuccess) return cuda_fail(e, "decode_step_fp8 append launch");
    }
    e = launch_decode(a, plan, PKV_FP8_E4M3, stream);
    return e == cudaSuccess ? PKV_OK : cuda_fail(e, "decode_step_fp8 launch");
}

int pkv_decode_step_fp8_kernel_launches(int B, int Hq, int Hkv, int d, int bs, int MBS, int NB, pkv_dtype new_dt,
                                        int num_splits) {
    if (!attention_dtype(new_dt)) return -1;
    const int n = pkv_decode_kernel_launches(B, Hq, Hkv, d, bs, MBS, NB, PKV_FP8_E4M3, num_splits);
    if (n <= 0) return n;
    DeviceState *st = nullptr;
    if (device_state(&st) != PKV_OK) return -1;
    const DecodePlan plan =
        plan_decode(B, Hq, Hkv, d, bs, MBS, NB, PKV_FP8_E4M3, num_splits, st->sm_count, true, true);
    static const uint4 aligned{};
    return n + (decode_fuses_append(plan, PKV_FP8_E4M3, new_dt, Hq, Hkv, &aligned, &aligned) ? 0 : 1);
}

}  // extern "C"

namespace {

// The shared-prefix decode step's layout: key splits of the prefix and 128-row tiles of a
// group's (member, head) pairs for the prefix kernel, and the workspace after the decode's
// own: prefix partials o [members][Hq][splits][d], their lse [members][Hq][splits], the
// suffix lse [B][Hq].
struct SharedPrefixLayout {
    bool ok = false;   // the cascade applies (otherwise the call is a plain decode step)
    int splits = 1, rtiles = 1;
    size_t decode_bytes = 0, o_off = 0, lse_off = 0, suffix_off = 0, total = 0;
};

SharedPrefixLayout shared_prefix_layout(const DecodePlan &plan, pkv_dtype dt, int B, int Hq, int Hkv, int d, int bs,
                                        int n_groups, int n_members, int max_group_size, int max_prefix_tokens,
                                        int sm_count, bool aligned) {
    SharedPrefixLayout L;
    L.decode_bytes = (plan.workspace_bytes + 255) / 256 * 256;
    L.total = plan.workspace_bytes;
    L.ok = n_groups > 0 && n_members > 0 && max_group_size > 0 && max_prefix_tokens > 0 && dt == PKV_BF16 &&
           (d == 64 || d == 128) && (bs == 16 || bs == 32) && aligned && plan.tensor_core &&
           (!plan.group || plan.umma) && Hq / Hkv <= 64;
    if (!L.ok) return L;
    const int m = Hq / Hkv;
    L.rtiles = static_cast<int>((static_cast<long long>(max_group_size) * m + 127) / 128);
    const long long units = static_cast<long long>(n_groups) * Hkv * L.rtiles;
    const int max_tiles = (max_prefix_tokens + 127) / 128;
    // the prefix kernel runs beside the decode: about a quarter of the SMs, with whole
    // equal key splits (each split a few thousand cycles of start-up, then 16+ key tiles)
    const long long want = std::max<long long>(1, (sm_count / 4 + units - 1) / units);
    const int per = static_cast<int>(std::max<long long>(1, (max_tiles + want - 1) / want));
    L.splits = std::min((max_tiles + per - 1) / per, 256);
    const size_t parts = static_cast<size_t>(n_members) * Hq * L.splits;
    L.o_off = L.decode_bytes;
    L.lse_off = L.o_off + (parts * d * sizeof(float) + 255) / 256 * 256;
    L.suffix_off = L.lse_off + (parts * sizeof(float) + 255) / 256 * 256;
    L.total = L.suffix_off + static_cast<size_t>(B) * Hq * sizeof(float);
    return L;
}

// A non-blocking stream and two events per device for work that runs beside a call's
// stream (created on first use in each CUDA context, kept until the process exits).  The
// mutex keeps one call's record / wait / launch / record sequence whole when several host
// threads call at once.
struct SideStream {
    unsigned long long ctx_id = 0;   // the CUDA context they belong to (cuCtxGetId)
    cudaStream_t stream = nullptr;
    cudaEvent_t fork = nullptr, join = nullptr;
};
SideStream g_side[kMaxDevices];
std::mutex g_side_mutex;
PFN_cuCtxGetCurrent_v4000 g_ctx_current = nullptr;
PFN_cuCtxGetId_v12000 g_ctx_id = nullptr;
std::once_flag g_ctx_fn_once;

// Id of the current CUDA context (0 when none is current).  A stream or event created in a
// context that has since been destroyed (cudaDeviceReset) must not be used again.
unsigned long long current_ctx_id() {
    std::call_once(g_ctx_fn_once, [] {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &fn, 4000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_ctx_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(fn);
        fn = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &fn, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_ctx_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(fn);
    });
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    if (g_ctx_current != nullptr && g_ctx_id != nullptr && g_ctx_current(&ctx) == CUDA_SUCCESS && ctx != nullptr)
        g_ctx_id(ctx, &id);
    return id;
}

pkv_status side_stream(cudaStream_t *stream, cudaEvent_t *fork, cudaEvent_t *join) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices) return fail(PKV_ERR_UNSUPPORTED, "device ordinal %d", dev);
    const unsigned long long ctx = current_ctx_id();
    std::lock_guard<std::mutex> lock(g_side_mutex);
    SideStream &s = g_side[dev];
    if (s.stream != nullptr && s.ctx_id != ctx) s = SideStream{};   // made in a context since destroyed
    if (s.stream == nullptr) {
        s.ctx_id = ctx;
        e = cudaStreamCreateWithFlags(&s.stream, cudaStreamNonBlocking);
        if (e == cudaSuccess) e = cudaEventCreateWithFlags(&s.fork, cudaEventDisableTiming);
        if (e == cudaSuccess) e = cudaEventCreateWithFlags(&s.join, cudaEventDisableTiming);
        if (e != cudaSuccess) {
            s = SideStream{};
            return cuda_fail(e, "side stream");
        }
    }
    *stream = s.stream;
    *fork = s.fork;
    *join = s.join;
    return PKV_OK;
}

}  // namespace

extern "C" {

size_t pkv_decode_step_shared_prefix_workspace_bytes(int B, int Hq, int Hkv, int d, int bs, int MBS, int num_splits,
                                                     int n_groups, int n_members, int max_group_size,
                                                     int max_prefix_tokens) {
    if (check_decode_sizes(B, Hq, Hkv, d, bs, MBS) != PKV_OK || num_splits < 0 || n_groups < 0 || n_members < 0 ||
        max_group_size < 0 || max_prefix_tokens < 0)
        return 0;
    DeviceState *st = nullptr;
    if (device_state(&st) != PKV_OK) return 0;
    const size_t plain = decode_workspace_upper_bound(B, Hq, Hkv, d, bs, MBS, num_splits, st->sm_count);
    const DecodePlan plan = plan_decode(B, Hq, Hkv, d, bs, MBS, 1, PKV_BF16, num_splits, st->sm_count, true, true);
    const SharedPrefixLayout L = shared_prefix_layout(plan, PKV_BF16, B, Hq, Hkv, d, bs, n_groups, n_members,
                                                      max_group_size, max_prefix_tokens, st->sm_count, true);
    return std::max(plain, L.total);
}

int pkv_decode_step_shared_prefix_kernel_launches(int B, int Hq, int Hkv, int d, int bs, int MBS, int NB,
                                                  pkv_dtype dt, int num_splits, int n_groups, int n_members,
                                                  int max_group_size, int max_prefix_tokens) {
    const int n = pkv_decode_step_kernel_launches(B, Hq, Hkv, d, bs, MBS, NB, dt, num_splits);
    if (n <= 0 || n_groups < 0 || n_members < 0 || max_group_size < 0 || max_prefix_tokens < 0) return n;
    DeviceState *st = nullptr;
    if (device_state(&st) != PKV_OK) return -1;
    const DecodePlan plan = plan_decode(B, Hq, Hkv, d, bs, MBS, NB, dt, num_splits, st->sm_count, true, true);
    const SharedPrefixLayout L = shared_prefix_layout(plan, dt, B, Hq, Hkv, d, bs, n_groups, n_members,
                                                      max_group_size, max_prefix_tokens, st->sm_count, true);
    return n + (L.ok ? 2 : 0);   // the prefix kernel and the merge around the decode
}

pkv_status pkv_decode_step_shared_prefix(float *out, float *lse, const float *q, const void *k_new,
                                         const void *v_new, const int64_t *slot_mapping, void *k_cache,
                                         void *v_cache, pkv_dtype dt, const int32_t *block_table,
                                         const int32_t *context_lens, const int32_t *prefix_tokens,
                                         const int32_t *group_start, const int32_t *group_seqs, int n_groups,
                                         int n_members, int max_group_size, int max_prefix_tokens, int B, int Hq,
                                         int Hkv, int d, int bs, int MBS, int NB, float scale, int num_splits,
                                         void *workspace, size_t workspace_bytes, pkv_stream_t stream) {
    int eb = 0;
    if (!elem_size(dt, &eb) || !attention_dtype(dt))
        return fail(PKV_ERR_UNSUPPORTED, "decode_step_shared_prefix: element type %d", dt);
    pkv_status s = check_decode_sizes(B, Hq, Hkv, d, bs, MBS);
    if (s != PKV_OK) return s;
    if (NB < 1 || num_splits < 0 || n_groups < 0 || n_members < 0 || max_group_size < 0 || max_prefix_tokens < 0 ||
        max_prefix_tokens > MBS * bs || max_group_size > n_members)
        return fail(PKV_ERR_INVALID_ARG,
                    "decode_step_shared_prefix: NB=%d num_splits=%d groups=%d members=%d max_group=%d "
                    "max_prefix=%d",
                    NB, num_splits, n_groups, n_members, max_group_size, max_prefix_tokens);
    if (B == 0) return PKV_OK;
    if (!out || !q || !k_new || !v_new || !slot_mapping || !k_cache || !v_cache || !block_table ||
        !context_lens || (n_groups > 0 && (!prefix_tokens || !group_start || !group_seqs)))
        return fail(PKV_ERR_INVALID_ARG, "decode_step_shared_prefix: null pointer");
    if (reinterpret_cast<uintptr_t>(q) % 8 != 0)
        return fail(PKV_ERR_INVALID_ARG, "decode_step_shared_prefix: q must be 8-byte aligned");
    DeviceState *st = nullptr;
    s = device_state(&st);
    if (s != PKV_OK) return s;
    const bool aligned = aligned16(k_cache) && aligned16(v_cache) && aligned16(q);
    const DecodePlan plan = plan_decode(B, Hq, Hkv, d, bs, MBS, NB, dt, num_splits, st->sm_count,
                                        aligned16(k_cache) && aligned16(v_cache), aligned16(q));
    const SharedPrefixLayout L = shared_prefix_layout(plan, dt, B, Hq, Hkv, d, bs, n_groups, n_members,
                                                      max_group_size, max_prefix_tokens, st->sm_count, aligned);
    if (L.total > 0 && (workspace == nullptr || workspace_bytes < L.total ||
                        reinterpret_cast<uintptr_t>(workspace) % 16 != 0))
        return fail(PKV_ERR_WORKSPACE,
                    "decode_step_shared_prefix: needs %zu bytes of 16-byte aligned workspace, got %zu", L.total,
                    workspace == nullptr ? size_t(0) : workspace_bytes);
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    cudaError_t e = cudaSuccess;
    cudaEvent_t joined = nullptr;
    std::unique_lock<std::mutex> side_lock(g_side_mutex, std::defer_lock);   // fork .. join enqueued
    DecodeArgs a{out, lse, q, k_cache, v_cache, block_table, context_lens,
                 B, Hq, Hkv, d, bs, MBS, NB, scale, workspace, st->err};
    if (L.ok) {
        // the attention of every member over its group's prefix, read once per group
        DecodeKParams kp{};
        kp.q = q;
        kp.block_table = block_table;
        kp.context_lens = context_lens;
        kp.err = st->err;
        kp.B = B;
        kp.Hq = Hq;
        kp.Hkv = Hkv;
        kp.m = Hq / Hkv;
        kp.MBS = MBS;
        kp.NB = NB;
        kp.scale_log2 = scale * 1.4426950408889634f;
        kp.cu_q = group_start;
        kp.group_seqs = group_seqs;
        kp.kv_start = prefix_tokens;
        kp.prefix_splits = L.splits;
        kp.prefix_rtiles = L.rtiles;
        kp.n_members = n_members;
        kp.ws_o = reinterpret_cast<float *>(ws + L.o_off);
        kp.ws_lse = reinterpret_cast<float *>(ws + L.lse_off);
        CUtensorMap tk, tv;
        const uint64_t dims[2] = {static_cast<uint64_t>(d), static_cast<uint64_t>(NB) * Hkv * bs};
        const uint64_t strides[1] = {static_cast<uint64_t>(d) * 2};
        const uint32_t box[2] = {64, static_cast<uint32_t>(bs)};
        if (!encode_map_bf16(&tk, k_cache, 2, dims, strides, box) || !encode_map_bf16(&tv, v_cache, 2, dims, strides, box))
            return fail(PKV_ERR_CUDA, "decode_step_shared_prefix: tensor map");
        // on the device's side stream, beside the decode (which reads other pages and writes
        // none of the prefix kernel's); joined back to `stream` before the merge
        cudaStream_t side = nullptr;
        cudaEvent_t fork = nullptr, join = nullptr;
        s = side_stream(&side, &fork, &join);
        if (s != PKV_OK) return s;
        side_lock.lock();
        e = cudaEventRecord(fork, stream);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(side, fork, 0);
        if (e == cudaSuccess) e = launch_shared_prefix(kp, tk, tv, d, bs, dim3(L.splits, Hkv, n_groups * L.rtiles), side);
        if (e == cudaSuccess) e = cudaEventRecord(join, side);
        if (e != cudaSuccess) return cuda_fail(e, "decode_step_shared_prefix prefix launch");
        joined = join;
        // the decode reads each sequence's keys after its prefix; its lse (the caller's array,
        // or the workspace's) feeds the merge, which rewrites the members' entries in place
        a.kv_start = prefix_tokens;
        a.lse = lse != nullptr ? lse : reinterpret_cast<float *>(ws + L.suffix_off);
    }
    if (decode_fuses_append(plan, dt, dt, Hq, Hkv, k_new, v_new)) {
        a.k_new = k_new;
        a.v_new = v_new;
        a.new_slots = slot_mapping;
    } else {
        e = launch_kv_append(k_new, v_new, k_cache, v_cache, eb, slot_mapping, B, Hkv, d, bs, NB, st->err, stream);
        if (e != cudaSuccess) return cuda_fail(e, "decode_step_shared_prefix append launch");
    }
    e = launch_decode(a, plan, dt, stream);
    if (e != cudaSuccess) return cuda_fail(e, "decode_step_shared_prefix decode launch");
    if (L.ok) {
        e = cudaStreamWaitEvent(stream, joined, 0);   // the prefix partials are complete
        side_lock.unlock();
        if (e != cudaSuccess) return cuda_fail(e, "decode_step_shared_prefix join");
        DecodeKParams kp{};
        kp.out = out;
        kp.lse = lse;
        kp.block_table = block_table;
        kp.context_lens = context_lens;
        kp.err = st->err;
        kp.B = B;
        kp.Hq = Hq;
        kp.MBS = MBS;
        kp.cu_q = group_start;
        kp.group_seqs = group_seqs;
        kp.kv_start = prefix_tokens;
        kp.prefix_splits = L.splits;
        kp.ws_o = reinterpret_cast<float *>(ws + L.o_off);
        kp.ws_lse = reinterpret_cast<float *>(ws + L.lse_off);
        e = launch_shared_prefix_merge(kp, a.lse, d, bs, n_groups, n_members, stream);
        if (e != cudaSuccess) return cuda_fail(e, "decode_step_shared_prefix merge launch");
    }
    return PKV_OK;
}

pkv_status pkv_prefill_attention(float *out, float *lse, const void *q, const void *k, const void *v,
                                 pkv_dtype dt, const int32_t *cu_seqlens, int B, int T,
                                 int max_seqlen, int Hq, int Hkv, int d, float scale,
                                 void *k_cache, void *v_cache, const int64_t *slot_mapping, int bs,
                                 int NB, pkv_stream_t stream) {
    int eb = 0;
    if (!elem_size(dt, &eb) || !attention_dtype(dt))
        return fail(PKV_ERR_UNSUPPORTED, "prefill_attention: element type %d", dt);
    if (B < 0 || B > 65535 || T < 0 || max_seqlen < 0 || Hq < 1 || Hq > 65535 || Hkv < 1 ||
        Hq % Hkv != 0 || d < 1 || d > 256)
        return fail(PKV_ERR_INVALID_ARG,
                    "prefill_attention: B=%d T=%d max_seqlen=%d Hq=%d Hkv=%d d=%d", B, T, max_seqlen,
                    Hq, Hkv, d);
    if (slot_mapping != nullptr && (bs < 1 || NB < 1 || !k_cache || !v_cache))
        return fail(PKV_ERR_INVALID_ARG, "prefill_attention: cache write needs caches, bs and NB");
    if (B == 0 || T == 0) return PKV_OK;
    if (!out || !q || !k || !v || !cu_seqlens)
        return fail(PKV_ERR_INVALID_ARG, "prefill_attention: null pointer");
    DeviceState *st = nullptr;
    pkv_status s = device_state(&st);
    if (s != PKV_OK) return s;
    cudaError_t e;
    if (slot_mapping != nullptr) {
        e = launch_kv_append(k, v, k_cache, v_cache, eb, slot_mapping, T, Hkv, d, bs, NB, st->err,
                             stream);
        if (e != cudaSuccess) return cuda_fail(e, "prefill_attention cache write");
    }
    PrefillArgs a{out, lse, q, k, v, cu_seqlens, B, T, max_seqlen, Hq, Hkv, d, scale, st->err};
    e = launch_prefill(a, dt, stream);
    return e == cudaSuccess ? PKV_OK : cuda_fail(e, "prefill_attention launch");
}

pkv_status pkv_get_device_error(int *code, pkv_stream_t stream) {
    if (code == nullptr) return fail(PKV_ERR_INVALID_ARG, "get_device_error: null code");
    DeviceState *st = nullptr;
    pkv_status s = device_state(&st);
    if (s != PKV_OK) return s;
    unsigned host = 0;
    cudaError_t e = cudaStreamSynchronize(stream);
    if (e == cudaSuccess) e = cudaMemcpyAsync(&host, st->err, sizeof host, cudaMemcpyDeviceToHost, stream);
    if (e == cudaSuccess) e = cudaMemsetAsync(st->err, 0, sizeof host, stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return cuda_fail(e, "get_device_error");
    *code = static_cast<int>(host);
    return PKV_OK;
}

}  // extern "C"
