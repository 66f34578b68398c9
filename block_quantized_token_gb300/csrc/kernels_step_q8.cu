// Persistent decode step, Q8_0 weights (instantiations of kernels_step.cuh).
#include "kernels_step.cuh"

namespace er {

template <int HD, int G>
static cudaError_t q8_launch(const StepArgs &a, int num_sms, size_t smem, cudaStream_t st) {
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
    return cudaLaunchKernelEx(&cfg, step_kernel<Q8_0, HD, G>, a);
}

template <int HD, int G>
static cudaError_t q8_attr() {
    // dynamic + static shared memory may not exceed the 227 KB per-block limit
    cudaFuncAttributes fa;
    cudaError_t e = cudaFuncGetAttributes(&fa, step_kernel<Q8_0, HD, G>);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(step_kernel<Q8_0, HD, G>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)(227 * 1024 - fa.sharedSizeBytes));
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(step_kernel<Q8_0, HD, G>, cudaFuncAttributePreferredSharedMemoryCarveout,
                                 cudaSharedmemCarveoutMaxShared);
    return e;
}

cudaError_t step_prepare_q8() {
    cudaError_t r[8] = {q8_attr<64, 1>(),  q8_attr<64, 2>(),  q8_attr<64, 3>(),  q8_attr<64, 4>(),
                        q8_attr<128, 1>(), q8_attr<128, 2>(), q8_attr<128, 3>(), q8_attr<128, 4>()};
    for (cudaError_t x : r)
        if (x != cudaSuccess) return x;
    return cudaSuccess;
}

// blocks of the step kernel that fit on one SM with `smem` bytes of dynamic shared memory
int step_occupancy_q8(int hd, size_t smem) {
    int per_sm = 0;
    cudaError_t e = hd == 64 ? cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, step_kernel<Q8_0, 64, 4>, GV_WARPS * 32, smem)
                             : cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, step_kernel<Q8_0, 128, 4>, GV_WARPS * 32, smem);
    return e == cudaSuccess ? per_sm : 0;
}

cudaError_t launch_step_q8(const StepArgs &a, int num_sms, size_t smem, cudaStream_t st) {
    const int G = a.H / a.KV;
    if (a.hd == 64) {
        switch (G) {
            case 1: return q8_launch<64, 1>(a, num_sms, smem, st);
            case 2: return q8_launch<64, 2>(a, num_sms, smem, st);
            case 3: return q8_launch<64, 3>(a, num_sms, smem, st);
            case 4: return q8_launch<64, 4>(a, num_sms, smem, st);
        }
    } else if (a.hd == 128) {
        switch (G) {
            case 1: return q8_launch<128, 1>(a, num_sms, smem, st);
            case 2: return q8_launch<128, 2>(a, num_sms, smem, st);
            case 3: return q8_launch<128, 3>(a, num_sms, smem, st);
            case 4: return q8_launch<128, 4>(a, num_sms, smem, st);
        }
    }
    return cudaErrorInvalidValue;
}

}  // namespace er

// ---------------------------------------------------------------------------
// dispatch shared by both weight types
// ---------------------------------------------------------------------------
namespace er {

cudaError_t step_prepare_q4();
int step_occupancy_q4(int hd, size_t smem);
cudaError_t launch_step_q4(const StepArgs &a, int num_sms, size_t smem, cudaStream_t st);

cudaError_t step_prepare() {
    cudaError_t e = step_prepare_q8();
    return e == cudaSuccess ? step_prepare_q4() : e;
}

static size_t step_smem(int qt, int max_k, int B, int hd, int G) {
    return qt == Q8_0 ? mk_smem_bytes<Q8_0>(max_k, B, hd, G) : mk_smem_bytes<Q4_0>(max_k, B, hd, G);
}
// static shared memory of the step kernel (barrier flag, warp ranges, per-step tables)
constexpr size_t STEP_STATIC_SMEM = 12288;

bool step_supported(int qt, int hd, int G, int B, int KV, int cap, int max_k, const int R[5], const int UPR[5],
                    int num_sms) {
    if (B < 1 || B > ER_MK_MAXB || G < 1 || G > ER_MK_MAXG || (hd != 64 && hd != 128)) return false;
    // 32-bit row and unit indices, byte-sized CTA indices in the segment table
    if (num_sms > 255 || B * KV > MK_MAX_SEGS) return false;
    if ((long long)B * KV * cap * (num_sms + 1) >= (1ll << 31)) return false;
    for (int i = 0; i < 5; ++i)
        if (!gv_index_ok(R[i], UPR[i], num_sms)) return false;
    if (step_smem(qt, max_k, B, hd, G) + STEP_STATIC_SMEM > 227 * 1024) return false;
    // cooperative launch: one CTA of the kernel must fit on every SM (each
    // weight type's kernels are instantiated, and configured, in their own file)
    const size_t smem = step_smem(qt, max_k, B, hd, G);
    const int per_sm = qt == Q8_0 ? step_occupancy_q8(hd, smem) : step_occupancy_q4(hd, smem);
    return per_sm >= 1;
}

size_t step_apart_floats(int num_sms, int hd) { return (size_t)num_sms * 2 * ER_MK_MAXG * (hd + 4); }

cudaError_t launch_step(int qt, const StepArgs &a, int num_sms, cudaStream_t st) {
    const int max_k = a.D > a.qd ? (a.D > a.F ? a.D : a.F) : (a.qd > a.F ? a.qd : a.F);
    const size_t smem = step_smem(qt, max_k, a.B, a.hd, a.H / a.KV);
    return qt == Q8_0 ? launch_step_q8(a, num_sms, smem, st) : launch_step_q4(a, num_sms, smem, st);
}

// this translation unit's copy of the bounded-wait limit
cudaError_t set_wait_limit_step_q8(unsigned long long ns) { return set_wait_limit_here(ns); }

}  // namespace er
