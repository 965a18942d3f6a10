// Check of the kernels' failure detection: a bounded wait that runs out.
//
// Every decode kernel waits on mbarriers that asynchronous copies complete.
// Such a wait is bounded: past its limit the kernel records PA_ERR_TIMEOUT in
// the device status word, stops its loop, drains what it issued and returns,
// so the context stays usable and the host learns of it through
// pa_device_status. Nothing in a correct run lets a wait run out, so this
// file gives that path a run of its own. One CTA is laid out as the decode
// kernels are (a producer warp that arms a ring stage, a consumer warp that
// waits for it), except that the producer arms the stage for a copy it never
// issues: the phase cannot complete, the consumer's wait gives up after the
// caller's limit, records the timeout and raises the abort flag; the producer,
// seeing it, stops; the drain's own bounded wait gives up too (it records
// the same code), and the CTA returns. No copy is in flight at any point,
// so nothing lands in shared memory after the CTA has gone.
#include "../../include/pa.h"
#include "device_common.cuh"
#include "internal.h"

namespace pa {

namespace {

__global__ void __launch_bounds__(64, 1) wait_timeout_check_kernel(int *status, unsigned long long limit_ns) {
    __shared__ __align__(8) uint64_t bars[2];   // the stage's full and empty barriers
    __shared__ int s_abort;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t full = smem_addr(&bars[0]), empty = smem_addr(&bars[1]);
    if (threadIdx.x == 0) {
        mbar_init(full, 1);
        mbar_init(empty, 1);
        s_abort = 0;
        mbar_fence_init();
    }
    __syncthreads();
    if (warp == 1) {
        // producer: arm stage 0 for 1 KiB of copies, then (as for a second
        // round of the ring) wait for the consumer to release it
        if (lane == 0) {
            mbar_arrive_expect_tx(full, 1024u);   // no copy is ever issued
            while (!*reinterpret_cast<volatile int *>(&s_abort)) {
                if (mbar_wait_for(empty, 0, limit_ns)) break;   // (never: the consumer does not release)
                record_status(status, kStatusTimeout);
                s_abort = 1;
            }
        }
    } else if (lane == 0) {
        // consumer: the decode kernels' wait for a stage to fill
        if (!mbar_wait_for(full, 0, limit_ns)) {
            record_status(status, kStatusTimeout);
            s_abort = 1;
        } else {
            mbar_arrive(empty);
        }
    }
    __syncthreads();
    // drain: the last phase the producer armed (bounded as well)
    if (threadIdx.x == 0 && !mbar_wait_for(full, 0, limit_ns)) record_status(status, kStatusTimeout);
}

}  // namespace

cudaError_t launch_wait_timeout_check(int *status, unsigned long long limit_ns, cudaStream_t stream) {
    wait_timeout_check_kernel<<<1, 64, 0, stream>>>(status, limit_ns);
    return cudaGetLastError();
}

}  // namespace pa

extern "C" PA_API pa_status pa_check_wait_timeout(unsigned timeout_us, void *stream) {
    if (timeout_us == 0 || timeout_us > 2000000u) return PA_ERR_INVALID_ARG;
    int *status = pa::device_status_word();
    if (!status) return PA_ERR_CUDA;
    const cudaError_t e = pa::launch_wait_timeout_check(status, 1000ull * timeout_us,
                                                        reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}
