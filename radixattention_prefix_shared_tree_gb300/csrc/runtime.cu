// Host runtime pieces of the device half: status strings, stream sync with the
// device error word, and the cached SM count used to size grids.

#include "common.cuh"
#include "tc.cuh"

namespace rc_host {

int sm_count() {
    static int cached[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
    if (!cached[dev]) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
        cached[dev] = n;
    }
    return cached[dev];
}

}  // namespace rc_host

namespace {

// One warp waits, with the bounded mbarrier wait every kernel here uses, on a
// barrier that no thread ever arrives at.  When the wait gives up (about a
// second) the warp ORs the timeout bit into the error word and leaves.
__global__ void __launch_bounds__(32) wait_probe_kernel(int32_t* err) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x == 0) {
        tc::mbar_init(&bar, 1);
        tc::fence_mbar_init();
    }
    __syncwarp();
    const bool ok = __all_sync(0xffffffffu, tc::mbar_wait(&bar, 0, 1u << 24));
    if (!ok && threadIdx.x == 0) rc::flag_error(err, rc::kErrTimeout);
}

}  // namespace

extern "C" rc_status rc_probe_wait_timeout(int32_t* err, rc_stream_t stream) {
    if (!err) return RC_ERR_ARG;
    wait_probe_kernel<<<1, 32, 0, (cudaStream_t)stream>>>(err);
    return rc_host::launch_status(cudaGetLastError());
}

extern "C" rc_status rc_sync(rc_stream_t stream, int32_t* err) {
    cudaError_t e = cudaStreamSynchronize((cudaStream_t)stream);
    if (e != cudaSuccess) return RC_ERR_CUDA;
    if (!err) return RC_OK;
    int32_t h = 0;
    e = cudaMemcpyAsync(&h, err, sizeof h, cudaMemcpyDeviceToHost, (cudaStream_t)stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize((cudaStream_t)stream);
    if (e != cudaSuccess) return RC_ERR_CUDA;
    if (!h) return RC_OK;
    const int32_t zero = 0;
    e = cudaMemcpyAsync(err, &zero, sizeof zero, cudaMemcpyHostToDevice, (cudaStream_t)stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize((cudaStream_t)stream);
    if (e != cudaSuccess) return RC_ERR_CUDA;
    if (h & rc::kErrBadSlot) return RC_ERR_DEVICE;
    return RC_ERR_TIMEOUT;
}

extern "C" const char* rc_strerror(rc_status s) {
    switch (s) {
        case RC_OK: return "ok";
        case RC_ERR_ARG: return "invalid argument";
        case RC_ERR_NOMEM: return "not enough free slots";
        case RC_ERR_STATE: return "invalid state (unknown or unpinned node, slot not held by the caller)";
        case RC_ERR_CUDA: return "CUDA runtime error";
        case RC_ERR_TIMEOUT: return "bounded device wait gave up";
        case RC_ERR_DEVICE: return "kernel found a slot index outside the pool";
        case RC_ERR_UNSUPPORTED: return "head layout not supported by this build";
        case RC_ERR_SCRATCH: return "batch needs more split scratch than the library's fixed area holds";
        default: return "unknown status";
    }
}
