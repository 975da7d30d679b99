// decode_noalloc.cu -- paged decode attention whose split-K scratch is built into the
// library, for callers that cannot call cudaMalloc.
//
// Who needs it: an extension running inside a host application that owns all device
// memory and gives its plugins none to allocate, and latency-critical decode loops that
// must not allocate or free in the middle of a step (cudaFree, and often cudaMalloc,
// synchronise the whole device).  The pages this library follows (the paper) have no
// counterpart for this entry point.
//
// How: the split-K partials live in g_decode_scratch, a file-scope static device array
// of PKV_NOALLOC_SCRATCH_BYTES bytes.  Each GPU that loads the library holds one copy
// until the process exits.  Host code cannot pass the array's name to a kernel (on the
// host it is only a stand-in symbol), so the first call in each CUDA context, with that
// context's device current, looks up its device address with cudaGetSymbolAddress and
// caches it under the context's id (a module's device symbols belong to the context that
// loaded it: after cudaDeviceReset, or under a context the host application made
// current itself, the address is looked up again).  The kernels and the launch sequence
// are those of pkv_paged_decode_attention: this file only supplies the scratch pointer
// in place of a caller workspace, and clears the arrival counters a call will use.
#include <cudaTypedefs.h>

#include <cstdio>
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace pkv {
namespace {

static __device__ __align__(256) unsigned char g_decode_scratch[PKV_NOALLOC_SCRATCH_BYTES];

struct ScratchEntry {
    unsigned long long ctx_id;   // cuCtxGetId: unique for the process's lifetime
    void *addr;
};
constexpr int kMaxScratchContexts = 64;
ScratchEntry g_scratch[kMaxScratchContexts] = {};
int g_scratch_used = 0;
std::mutex g_scratch_mutex;
PFN_cuCtxGetCurrent_v4000 g_ctx_get_current = nullptr;
PFN_cuCtxGetId_v12000 g_ctx_get_id = nullptr;
std::once_flag g_ctx_once;

// Id of the current context; false when no context is current (or the driver calls are
// missing).
bool current_context_id(unsigned long long *id) {
    std::call_once(g_ctx_once, [] {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &fn, 4000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_ctx_get_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(fn);
        fn = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &fn, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_ctx_get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(fn);
    });
    CUcontext ctx = nullptr;
    return g_ctx_get_current != nullptr && g_ctx_get_id != nullptr && g_ctx_get_current(&ctx) == CUDA_SUCCESS &&
           ctx != nullptr && g_ctx_get_id(ctx, id) == CUDA_SUCCESS;
}

// Device address of g_decode_scratch in the current context: looked up once per context
// (keyed by the context's id, which a later context never reuses), or on every call with
// more than kMaxScratchContexts contexts.
pkv_status scratch_address(void **addr) {
    unsigned long long id = 0;
    bool have_id = current_context_id(&id);
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    if (have_id)
        for (int i = 0; i < g_scratch_used; ++i)
            if (g_scratch[i].ctx_id == id) {
                *addr = g_scratch[i].addr;
                return PKV_OK;
            }
    // with no context current yet, this makes the device's primary context current
    void *p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_decode_scratch);
    if (e != cudaSuccess || p == nullptr)
        return record_error(PKV_ERR_CUDA, "decode_noalloc: cudaGetSymbolAddress(scratch) failed");
    if (!have_id) have_id = current_context_id(&id);
    if (have_id && g_scratch_used < kMaxScratchContexts) g_scratch[g_scratch_used++] = {id, p};
    *addr = p;
    return PKV_OK;
}

}  // namespace
}  // namespace pkv

using namespace pkv;

extern "C" pkv_status pkv_paged_decode_attention_noalloc(
    float *out, float *lse, const float *q, const void *k_cache, const void *v_cache, pkv_dtype dt,
    const int32_t *block_table, const int32_t *context_lens, int B, int Hq, int Hkv, int d, int bs,
    int MBS, int NB, float scale, int num_splits, pkv_stream_t stream) {
    if (dt != PKV_F32 && dt != PKV_BF16)
        return record_error(PKV_ERR_UNSUPPORTED, "decode_noalloc: element type");
    if (B < 0 || B > 65535 || Hq < 1 || Hq > 65535 || Hkv < 1 || Hq % Hkv != 0 || d < 1 ||
        d > 256 || bs < 1 || MBS < 1 || NB < 1 || num_splits < 0)
        return record_error(PKV_ERR_INVALID_ARG,
                            "decode_noalloc: bad sizes (need 0<=B<=65535, Hq % Hkv == 0, "
                            "1<=d<=256, bs>=1, MBS>=1, NB>=1, num_splits>=0)");
    if (B == 0) return PKV_OK;
    if (!out || !q || !k_cache || !v_cache || !block_table || !context_lens)
        return record_error(PKV_ERR_INVALID_ARG, "decode_noalloc: null pointer");
    if (reinterpret_cast<uintptr_t>(q) % 8 != 0)
        return record_error(PKV_ERR_INVALID_ARG, "decode_noalloc: q must be 8-byte aligned");
    int sm_count = 0;
    unsigned *err = nullptr;
    pkv_status s = current_device_info(&sm_count, &err);
    if (s != PKV_OK) return s;
    const bool aligned = reinterpret_cast<uintptr_t>(k_cache) % 16 == 0 &&
                         reinterpret_cast<uintptr_t>(v_cache) % 16 == 0;
    const DecodePlan plan =
        plan_decode(B, Hq, Hkv, d, bs, MBS, NB, dt, num_splits, sm_count, aligned,
                    reinterpret_cast<uintptr_t>(q) % 16 == 0);
    if (plan.workspace_bytes > PKV_NOALLOC_SCRATCH_BYTES) {
        char msg[200];
        snprintf(msg, sizeof msg,
                 "decode_noalloc: split-K partials need %zu bytes, more than the built-in "
                 "scratch of %u bytes (use fewer splits or the workspace entry point)",
                 plan.workspace_bytes, static_cast<unsigned>(PKV_NOALLOC_SCRATCH_BYTES));
        return record_error(PKV_ERR_WORKSPACE, msg);
    }
    void *scratch = nullptr;
    s = scratch_address(&scratch);   // the first call in this context looks it up
    if (s != PKV_OK) return s;
    cudaError_t e = cudaSuccess;
    if (plan.counter_bytes > 0) {
        // the counters this call uses (arrivals of the chunks that merge in place, tiles
        // taken): cleared here, so that a call that gave up on a wait (and left its
        // counters behind) cannot spoil this one
        e = cudaMemsetAsync(scratch, 0, plan.counter_bytes, stream);
        if (e != cudaSuccess) return record_error(PKV_ERR_CUDA, cudaGetErrorString(e));
    }
    DecodeArgs a{out, lse, q, k_cache, v_cache, block_table, context_lens,
                 B, Hq, Hkv, d, bs, MBS, NB, scale, scratch, err};
    e = launch_decode(a, plan, dt, stream);
    if (e != cudaSuccess) return record_error(PKV_ERR_CUDA, cudaGetErrorString(e));
    return PKV_OK;
}
