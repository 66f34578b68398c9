// Persistent decode step, Q4_0 weights (instantiations of kernels_step.cuh).
#include "kernels_step.cuh"

namespace er {

template <int HD, int G>
static cudaError_t q4_launch(const StepArgs &a, int num_sms, size_t smem, cudaStream_t st) {
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    cfg.gridDim = dim3(num_sms);
    cfg.blockDim = dim3(GV_WARPS * 32);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, step_kernel<Q4_0, HD, G>, a);
}

template <int HD, int G>
static cudaError_t q4_attr() {
    // dynamic + static shared memory may not exceed the 227 KB per-block limit
    cudaFuncAttributes fa;
    cudaError_t e = cudaFuncGetAttributes(&fa, step_kernel<Q4_0, HD, G>);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(step_kernel<Q4_0, HD, G>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)(227 * 1024 - fa.sharedSizeBytes));
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(step_kernel<Q4_0, HD, G>, cudaFuncAttributePreferredSharedMemoryCarveout,
                                 cudaSharedmemCarveoutMaxShared);
    return e;
}

cudaError_t step_prepare_q4() {
    cudaError_t r[8] = {q4_attr<64, 1>(),  q4_attr<64, 2>(),  q4_attr<64, 3>(),  q4_attr<64, 4>(),
                        q4_attr<128, 1>(), q4_attr<128, 2>(), q4_attr<128, 3>(), q4_attr<128, 4>()};
    for (cudaError_t x : r)
        if (x != cudaSuccess) return x;
    return cudaSuccess;
}

// blocks of the step kernel that fit on one SM with `smem` bytes of dynamic shared memory
int step_occupancy_q4(int hd, size_t smem) {
    int per_sm = 0;
    cudaError_t e = hd == 64 ? cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, step_kernel<Q4_0, 64, 4>, GV_WARPS * 32, smem)
                             : cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, step_kernel<Q4_0, 128, 4>, GV_WARPS * 32, smem);
    return e == cudaSuccess ? per_sm : 0;
}

cudaError_t launch_step_q4(const StepArgs &a, int num_sms, size_t smem, cudaStream_t st) {
    const int G = a.H / a.KV;
    if (a.hd == 64) {
        switch (G) {
            case 1: return q4_launch<64, 1>(a, num_sms, smem, st);
            case 2: return q4_launch<64, 2>(a, num_sms, smem, st);
            case 3: return q4_launch<64, 3>(a, num_sms, smem, st);
            case 4: return q4_launch<64, 4>(a, num_sms, smem, st);
        }
    } else if (a.hd == 128) {
        switch (G) {
            case 1: return q4_launch<128, 1>(a, num_sms, smem, st);
            case 2: return q4_launch<128, 2>(a, num_sms, smem, st);
            case 3: return q4_launch<128, 3>(a, num_sms, smem, st);
            case 4: return q4_launch<128, 4>(a, num_sms, smem, st);
        }
    }
    return cudaErrorInvalidValue;
}

// this translation unit's copy of the bounded-wait limit
cudaError_t set_wait_limit_step_q4(unsigned long long ns) { return set_wait_limit_here(ns); }

}  // namespace er
