// selftest.cu -- a self-test of the kernels' failure path: a bounded wait that runs out.
//
// Every wait of the attention kernels on an mbarrier (a TMA copy landing, an MMA group
// completing) goes through wait_or_abort with a limit of kWaitLimitNs; the first thread to
// give up raises PKV_DEVERR_TIMEOUT and sets the block's abort flag, the other threads see
// the flag and give up too, and the block frees its tensor memory and returns.  Nothing in
// a correct attention call makes a wait run out, so this file gives the path its own
// kernel: the barrier's phase is armed for bytes that no copy will ever deliver (no copy
// is issued at all, so nothing can land after the block has exited), every thread waits
// on it through the same wait_or_abort with a short limit, and the block tears down the
// way the attention kernels do.
#include "common.cuh"
#include "internal.h"

namespace pkv {
namespace {

constexpr int kSelftestThreads = 128;
constexpr uint32_t kSelftestTmemCols = 512;

__global__ void __launch_bounds__(kSelftestThreads)
    bounded_wait_selftest_kernel(unsigned long long limit_ns, int hold_tmem, unsigned *err,
                                 unsigned *gave_up) {
    __shared__ __align__(8) uint64_t bar;
    __shared__ uint32_t tslot;
    __shared__ int abort_flag;
    const int warp = threadIdx.x >> 5;
    const uint32_t b = smem_addr(&bar);
    if (threadIdx.x == 0) {
        mbar_init(b, 1);
        abort_flag = 0;
        fence_barrier_init();
    }
    // the attention kernels hold all 512 tensor-memory columns while they wait
    if (hold_tmem && warp == 0) tmem_alloc(smem_addr(&tslot), kSelftestTmemCols);
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    // the single expected arrival, with 1024 bytes of transactions that never come: the
    // barrier's phase 0 cannot complete
    if (threadIdx.x == 0) mbar_arrive_expect_tx(b, 1024);
    __syncthreads();
    const bool ok = wait_or_abort(b, 0, reinterpret_cast<volatile int *>(&abort_flag), err, limit_ns);
    if (!ok && gave_up != nullptr) atomicAdd(gave_up, 1u);
    // teardown as in the attention kernels: every thread has left its wait, then the
    // allocating warp frees tensor memory
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    if (hold_tmem && warp == 0) tmem_dealloc(tslot, kSelftestTmemCols);
}

}  // namespace
}  // namespace pkv

using namespace pkv;

extern "C" pkv_status pkv_selftest_bounded_wait(unsigned long long limit_ns, int blocks, int hold_tmem,
                                                unsigned *gave_up, pkv_stream_t stream) {
    if (limit_ns == 0 || limit_ns > 1000000000ull || blocks < 1 || blocks > 1024)
        return record_error(PKV_ERR_INVALID_ARG,
                            "selftest_bounded_wait: need 0 < limit_ns <= 1e9 and 1 <= blocks <= 1024");
    int sm_count = 0;
    unsigned *err = nullptr;
    const pkv_status s = current_device_info(&sm_count, &err);
    if (s != PKV_OK) return s;
    bounded_wait_selftest_kernel<<<blocks, kSelftestThreads, 0, stream>>>(limit_ns, hold_tmem ? 1 : 0, err,
                                                                           gave_up);
    const cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? PKV_OK : record_error(PKV_ERR_CUDA, cudaGetErrorString(e));
}
