// The expired-wait path, exercised on purpose: one thread runs the bounded
// waits the warp-MMA kernels use (a completion counter that must reach a
// target, an mbarrier phase) on a counter nothing increments and an mbarrier
// nothing arrives at.  Each wait gives up after its time limit and the thread
// ORs a status bit into the library's device status word, the same report an
// expired wait in a production kernel makes; nothing faults, traps or hangs,
// and the context stays usable.  Given an arrival counter, the probe first
// increments it: what a split-K launch cut short by an expired wait can leave
// behind (an arrival counted, its block never reduced), so that a test can
// check that the report of the expiry also clears such counters.
#include <cuda.h>

#include "w4a16_internal.h"
#include "w4a16_mma_common.cuh"

namespace w4a16 {
namespace {

using namespace warp_mma;

__device__ unsigned g_never_incremented;  // zero for the life of the module

__global__ void wait_probe_kernel(int *status, unsigned *stale) {
    __shared__ __align__(8) uint64_t bar;
    if (stale) atomicAdd(stale, 1u);
    const uint32_t b = dev::smem_u32(&bar);
    mbar_init(b, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    if (!wait_counter(&g_never_incremented, 1u)) atomicOr(status, kErrProbeCounterWait);
    if (!mbar_wait(b, 0)) atomicOr(status, kErrProbeBarrierWait);
}

}  // namespace

cudaError_t launch_wait_probe(int *status, unsigned *stale, cudaStream_t stream) {
    wait_probe_kernel<<<1, 1, 0, stream>>>(status, stale);
    return cudaGetLastError();
}

}  // namespace w4a16
