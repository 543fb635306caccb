// Check of the device-side failure path: a kernel whose one wait can never be
// satisfied gives up after the bounded wait's limit and latches the time-out
// in the handle's error word, as any kernel of the layer would; nothing
// faults, traps or hangs, and the context stays usable.
#include "k3moe_internal.cuh"

namespace k3 {

__global__ void k_wait_check(int *err)
{
    __shared__ uint64_t bar;
    mbar_init(&bar, 1);    // one arrival completes the phase; none is made
    fence_mbar_init();
    mbar_wait(&bar, 0u, err, kWaitCheckWhere);
}

cudaError_t launch_wait_check(const k3moe &h, cudaStream_t s)
{
    k_wait_check<<<1, 1, 0, s>>>(h.ws.err);
    return cudaGetLastError();
}

}  // namespace k3
