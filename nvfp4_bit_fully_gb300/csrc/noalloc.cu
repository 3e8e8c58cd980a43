// noalloc.cu - the input-gradient backward (tj_linear_bwd_dx) for callers that
// cannot allocate device memory.
//
// tj_linear_bwd_dx needs a scratch workspace for the quantized backward operands,
// and the caller normally passes one in.  Some callers have no way to obtain one
// when the backward runs: code that lives below the framework's allocator (a custom
// allocator hook or a runtime that must not re-enter it), embedded or
// pre-provisioned deployments that hand out only buffers registered up front, or
// host code that is not allowed to call cudaMalloc at that point.  For them this
// file holds a fixed scratch array inside the library, so the call needs nothing
// beyond its inputs and outputs.
//
// The scratch is a file-scope __device__ array of kNoAllocScratchBytes.  Every GPU
// that loads the library keeps it resident until the process exits.  In host code
// the array's name is only a host-side stand-in, not a device address, so every call
// looks the device address up with cudaGetSymbolAddress in the current context (a host
// call of a few microseconds).  Nothing is cached, so the address stays right after a
// cudaDeviceReset and under any context.  No cudaMalloc, cudaFree or allocating
// library routine is called.
#include "tj_common.cuh"
#include "tj_internal.h"

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(16) << 20;      // 16 MiB
static __device__ __align__(256) uint8_t g_bwd_dx_scratch[kNoAllocScratchBytes];

// Device address of the scratch array in the current context (nullptr on failure).
void *scratch_on_current_device() {
    void *p = nullptr;
    return cudaGetSymbolAddress(&p, g_bwd_dx_scratch) == cudaSuccess ? p : nullptr;
}

}  // namespace

extern "C" size_t tj_noalloc_scratch_bytes(void) { return kNoAllocScratchBytes; }

extern "C" tj_status tj_linear_bwd_dx_noalloc(const void *dy, int64_t M, int64_t N, int64_t lddy,
                                              const tj_nvfp4 *wq, const tj_mxfp8 *w8, const int32_t *normal_idx,
                                              const int32_t *outlier_idx, int64_t k, uint64_t seed, void *dx,
                                              int out_dtype, int64_t lddx, void *stream) {
    if (wq == nullptr || M < 0 || N < 0 || k < 0) return TJ_ERR_INVALID_ARG;
    const size_t need = tj_workspace_size(TJ_OP_BWD_DX, M, N, wq->cols + k, k);
    if (need > kNoAllocScratchBytes) return TJ_ERR_WORKSPACE;       // problem too large for the fixed scratch
    void *scratch = scratch_on_current_device();
    if (scratch == nullptr) return TJ_ERR_CUDA;
    // Every byte of the scratch that the backward reads is written earlier in the same
    // call (the quantize kernels fill the padded operands completely), so the previous
    // call's contents never leak into the result and nothing needs clearing.
    return tj_linear_bwd_dx(dy, M, N, lddy, wq, w8, normal_idx, outlier_idx, k, seed, dx, out_dtype, lddx, scratch,
                            kNoAllocScratchBytes, stream);
}
