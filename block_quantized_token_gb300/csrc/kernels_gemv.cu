// Stand-alone block-quantized GEMV kernel (batch 1..4) with the fused
// epilogues; the arithmetic lives in gemv_core.cuh.
//
// Streaming: each warp owns a ring of shared-memory slots filled by bulk async
// copies (cp.async.bulk, completion on an mbarrier).  The first slots are
// requested before griddepcontrol.wait, so the weight traffic of this kernel
// overlaps the tail of the previous one.
#include <mutex>

#include "gemv_core.cuh"

namespace er {

// shared-memory map: [mbarriers 512][rings][scratch][operand]
constexpr int GV_OFF_RING = 512;
template <int QT>
constexpr int gv_off_scratch() { return GV_OFF_RING + GvCfg<QT>::RING; }

template <int QT, int EPI>
__global__ void __launch_bounds__(GV_WARPS * 32, 1) gemv_kernel(const GemvArgs a, int max_ctas) {
    using C = GvCfg<QT>;
    extern __shared__ __align__(128) uint8_t smem[];
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem);
    const GvScratch s = gv_scratch(smem + gv_off_scratch<QT>());

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const GvRange r = gv_range(a.R, a.UPR, blockIdx.x, max_ctas, warp);
    const int nunits = r.wb - r.wa;
    const int nslots = (nunits + C::SU - 1) / C::SU;
    uint64_t *wbar = bars + warp * GV_SLOTS;
    uint8_t *ring = smem + GV_OFF_RING + warp * GV_SLOTS * C::SLOT;
    const uint8_t *wsrc = a.W + (size_t)r.wa * C::UB;

    auto issue = [&](int k) {  // lane 0 only
        int sidx = k % GV_SLOTS;
        int cnt = min(C::SU, nunits - k * C::SU);
        uint32_t bytes = (uint32_t)cnt * C::UB;
        mbar_arrive_expect_tx(wbar + sidx, bytes);
        bulk_g2s(ring + sidx * C::SLOT, wsrc + (size_t)k * C::SLOT, bytes, wbar + sidx);
    };

    int issued = min(GV_SLOTS, nslots);
    if (lane == 0) {
        for (int i = 0; i < GV_SLOTS; ++i) mbar_init(wbar + i, 1);
        fence_mbar_init();
        for (int k = 0; k < issued; ++k) issue(k);
        s.wrg[warp * 2] = s.wrg[warp * 2 + 1] = -1;
    }
    __syncwarp();

    // ---- everything above touches only constant weights; now wait for inputs
    pdl_wait();
    int flag_wait = 0;
    if (tid == 0) flag_wait = *reinterpret_cast<volatile int *>(a.flags) & ER_FLAG_WAIT;
    gv_operand(a, s, tid, blockDim.x);
    if (tid == 0) s.fac[8] = flag_wait ? 1.f : 0.f;
    __syncthreads();
    // a kernel earlier in the stream gave up on a wait: the state is already
    // invalid, so drain this warp's copies and stop (one read, shared by the CTA)
    if (s.fac[8] != 0.f) {
        if (lane == 0)
            for (int k = 0; k < issued; ++k) mbar_wait(wbar + k % GV_SLOTS, (k / GV_SLOTS) & 1);
        return;
    }
    pdl_launch_dependents();

    auto refill = [&](unsigned k) {
        if ((int)k + GV_SLOTS < nslots) {
            if (lane == 0) {
                fence_proxy_async_smem();
                issue((int)k + GV_SLOTS);
            }
            ++issued;
        }
    };
    const int done = gv_consume<QT, EPI>(a, s, r, ring, wbar, 0, refill, lane, warp);
    if (done < 0 && lane == 0) {
        // wait (bounded) for this warp's copies still in flight before the CTA exits
        for (int k = 0; k < issued; ++k) mbar_wait(wbar + k % GV_SLOTS, (k / GV_SLOTS) & 1);
    }
    __syncthreads();
    int stop = 0;  // read once per warp: the shared-row-group sums below are warp-synchronous
    if (lane == 0) stop = *reinterpret_cast<volatile int *>(a.flags) & ER_FLAG_WAIT;
    if (__shfl_sync(0xffffffffu, stop, 0)) return;
    gv_finish_shared<EPI>(a, s, r, blockIdx.x, max_ctas, lane, warp);
}

// ---------------------------------------------------------------------------
size_t gemv_part_floats(int num_sms) { return (size_t)num_sms * 2 * 64; }

template <int QT>
static size_t gv_smem(int K, int B) { return gv_off_scratch<QT>() + GV_SCRATCH_BYTES + gv_xs_bytes(K, B); }

template <int QT, int EPI>
static cudaError_t gv_attr() {
    cudaError_t e = cudaFuncSetAttribute(gemv_kernel<QT, EPI>, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
    // one shared-memory carveout for every kernel of the step: no L1/shared
    // reconfiguration between consecutive launches
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(gemv_kernel<QT, EPI>, cudaFuncAttributePreferredSharedMemoryCarveout,
                                 cudaSharedmemCarveoutMaxShared);
    return e;
}

cudaError_t gemv_prepare() {
    cudaError_t e = cudaSuccess;
    cudaError_t r[10] = {gv_attr<Q8_0, EPI_STORE>(), gv_attr<Q8_0, EPI_RESID>(), gv_attr<Q8_0, EPI_QKV>(),
                         gv_attr<Q8_0, EPI_SWIGLU>(), gv_attr<Q8_0, EPI_LOGITS>(), gv_attr<Q4_0, EPI_STORE>(),
                         gv_attr<Q4_0, EPI_RESID>(), gv_attr<Q4_0, EPI_QKV>(), gv_attr<Q4_0, EPI_SWIGLU>(),
                         gv_attr<Q4_0, EPI_LOGITS>()};
    for (cudaError_t x : r)
        if (x != cudaSuccess) e = x;
    if (e == cudaSuccess) e = gemv_wide_prepare();
    if (e == cudaSuccess) e = attention_prepare();
    if (e == cudaSuccess) e = step_prepare();
    return e;
}

bool gemv_fits(int qt, int K, int B) {
    if (B < 1 || B > GV_MAXB || K % 32) return false;
    size_t need = qt == Q8_0 ? gv_smem<Q8_0>(K, B) : gv_smem<Q4_0>(K, B);
    return need <= 227 * 1024;
}

int gemv_max_cols(int qt, int K) {
    for (int b = GV_MAXB; b >= 1; --b)
        if (gemv_fits(qt, K, b)) return b;
    return 0;
}

template <int QT, int EPI>
static cudaError_t gv_launch(const GemvArgs &a, int num_sms, cudaStream_t st, bool pdl) {
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    cfg.gridDim = dim3((unsigned)gv_ctas(a.R, a.UPR, num_sms));
    cfg.blockDim = dim3(GV_WARPS * 32);
    cfg.dynamicSmemBytes = gv_smem<QT>(a.K, a.B);
    cfg.stream = st;
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, gemv_kernel<QT, EPI>, a, num_sms);
}

cudaError_t launch_gemv(int epi, const GemvArgs &a, int num_sms, cudaStream_t st, bool pdl) {
    if (!gemv_fits(a.qt, a.K, a.B) || !gv_index_ok(a.R, a.UPR, num_sms)) return cudaErrorInvalidValue;
    if (a.qt == Q8_0) {
        switch (epi) {
            case EPI_STORE: return gv_launch<Q8_0, EPI_STORE>(a, num_sms, st, pdl);
            case EPI_RESID: return gv_launch<Q8_0, EPI_RESID>(a, num_sms, st, pdl);
            case EPI_QKV: return gv_launch<Q8_0, EPI_QKV>(a, num_sms, st, pdl);
            case EPI_SWIGLU: return gv_launch<Q8_0, EPI_SWIGLU>(a, num_sms, st, pdl);
            case EPI_LOGITS: return gv_launch<Q8_0, EPI_LOGITS>(a, num_sms, st, pdl);
        }
    } else {
        switch (epi) {
            case EPI_STORE: return gv_launch<Q4_0, EPI_STORE>(a, num_sms, st, pdl);
            case EPI_RESID: return gv_launch<Q4_0, EPI_RESID>(a, num_sms, st, pdl);
            case EPI_QKV: return gv_launch<Q4_0, EPI_QKV>(a, num_sms, st, pdl);
            case EPI_SWIGLU: return gv_launch<Q4_0, EPI_SWIGLU>(a, num_sms, st, pdl);
            case EPI_LOGITS: return gv_launch<Q4_0, EPI_LOGITS>(a, num_sms, st, pdl);
        }
    }
    return cudaErrorInvalidValue;
}

// this translation unit's copy of the bounded-wait limit
cudaError_t set_wait_limit_gemv(unsigned long long ns) { return set_wait_limit_here(ns); }

}  // namespace er

// ---------------------------------------------------------------------------
// er_matrix_gemv_noalloc: the stand-alone GEMV with its scratch in a fixed array
// ---------------------------------------------------------------------------
namespace er {

// Scratch of the allocation-free GEMV, compiled into the library (every GPU that
// loads the library holds it until the process exits):
//   [partials: NOALLOC_MAX_SMS * 2 * 64 floats][counters: NOALLOC_MAX_RG ints][flag: 64 ints]
constexpr int NOALLOC_MAX_SMS = 256;
constexpr int NOALLOC_MAX_RG = 16384;  // row groups of 16 rows: up to 262144 rows
constexpr size_t NOALLOC_PART_BYTES = (size_t)NOALLOC_MAX_SMS * 2 * 64 * sizeof(float);
constexpr size_t NOALLOC_CNT_BYTES = (size_t)NOALLOC_MAX_RG * sizeof(int);
constexpr size_t NOALLOC_BYTES = NOALLOC_PART_BYTES + NOALLOC_CNT_BYTES + 64 * sizeof(int);

static __device__ __align__(256) unsigned char noalloc_scratch[NOALLOC_BYTES];

// Device address of noalloc_scratch on each device, looked up once per device
// (with that device current) on the first call there.  The name of the array
// in host code is only a host-side stand-in, so kernels get this address.
static unsigned char *noalloc_addr[64];
static std::mutex noalloc_mutex;

static cudaError_t noalloc_scratch_for(int device, unsigned char **out) {
    if (device < 0 || device >= 64) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(noalloc_mutex);
    if (!noalloc_addr[device]) {
        void *p = nullptr;
        cudaError_t e = cudaGetSymbolAddress(&p, noalloc_scratch);
        if (e != cudaSuccess) return e;
        noalloc_addr[device] = static_cast<unsigned char *>(p);
    }
    *out = noalloc_addr[device];
    return cudaSuccess;
}

}  // namespace er

extern "C" er_status er_matrix_gemv_noalloc(const er_matrix *x, const float *xin, int32_t batch, float *y,
                                           void *stream) {
    using namespace er;
    if (!x || !xin || !y) return er_fail_status(ER_EINVAL, "NULL argument");
    if (batch < 1 || batch > 16) return er_fail_status(ER_EINVAL, "batch must be in 1..16");
    if (x->m.R > NOALLOC_MAX_RG) return er_fail_status(ER_EINVAL, "matrix has more rows than the fixed scratch holds");
    if (x->num_sms > NOALLOC_MAX_SMS) return er_fail_status(ER_EUNSUPPORTED, "more SMs than the fixed scratch holds");
    int device = 0;
    cudaError_t e = cudaGetDevice(&device);
    if (e != cudaSuccess) return er_fail_cuda(e, "er_matrix_gemv_noalloc set-up");
    // the array used is the current device's; the matrix (and its SM count) must belong to that device
    if (device != x->device) return er_fail_status(ER_EINVAL, "the matrix belongs to another device than the current one");
    unsigned char *base = nullptr;
    e = noalloc_scratch_for(device, &base);
    if (e != cudaSuccess) return er_fail_cuda(e, "er_matrix_gemv_noalloc set-up");
    cudaStream_t st = (cudaStream_t)stream;
    GemvArgs a = {};
    a.W = x->m.d;
    a.R = x->m.R;
    a.UPR = x->m.UPR;
    a.N = x->m.N;
    a.K = x->m.K;
    a.qt = x->m.qt;
    a.x = xin;
    a.y = y;
    a.part = reinterpret_cast<float *>(base);
    a.cnt = reinterpret_cast<int *>(base + NOALLOC_PART_BYTES);
    a.flags = reinterpret_cast<int *>(base + NOALLOC_PART_BYTES + NOALLOC_CNT_BYTES);
    // the array keeps the last call's contents: counters and the flag start at zero
    e = cudaMemsetAsync(a.cnt, 0, (size_t)a.R * sizeof(int), st);
    if (e == cudaSuccess) e = cudaMemsetAsync(a.flags, 0, sizeof(int), st);
    const int per = gemv_max_cols(a.qt, a.K);
    for (int b0 = 0; b0 < batch && e == cudaSuccess; b0 += per) {
        a.b0 = b0;
        a.B = batch - b0 < per ? batch - b0 : per;
        e = launch_gemv(EPI_STORE, a, x->num_sms, st, false);
    }
    if (e != cudaSuccess) return er_fail_cuda(e, "er_matrix_gemv_noalloc");
    return ER_OK;
}

extern "C" er_status er_matrix_gemv_noalloc_error(int32_t *code) {
    using namespace er;
    if (!code) return er_fail_status(ER_EINVAL, "NULL argument");
    int device = 0;
    cudaError_t e = cudaGetDevice(&device);
    unsigned char *base = nullptr;
    if (e == cudaSuccess) e = noalloc_scratch_for(device, &base);
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    int *flag = reinterpret_cast<int *>(base + NOALLOC_PART_BYTES + NOALLOC_CNT_BYTES);
    int f = 0;
    if (e == cudaSuccess) e = cudaMemcpy(&f, flag, sizeof(int), cudaMemcpyDeviceToHost);
    if (e == cudaSuccess) e = cudaMemset(flag, 0, sizeof(int));
    if (e != cudaSuccess) return er_fail_cuda(e, "er_matrix_gemv_noalloc_error");
    *code = f & ER_FLAG_WAIT;
    return *code ? er_fail_status(ER_EDEVICE, "a wait in er_matrix_gemv_noalloc gave up") : ER_OK;
}
