// gate.cu -- stream gate for pipelined input staging: one warp waits for
// flags that a copy stream sets after a step's inputs have landed, clears
// them, and then lets the next kernel launch under programmatic dependent
// launch, so a decode loop can stage its inputs on another stream without an
// event wait between two kernels (which would break their launch link).
#include "dsv4_common.cuh"
#include "tc_common.cuh"

namespace dsv4 {

struct GateParams {
    int* f[4];
    unsigned long long limit_ns;
    int* status;
};

__device__ __forceinline__ int ld_acquire_gpu(const int* p)
{
    int v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__global__ void __launch_bounds__(32) stream_gate_kernel(GateParams G)
{
    const int lane = threadIdx.x;
    int* f = lane < 4 ? G.f[lane] : nullptr;
    bool ok = true;
    if (f != nullptr && ld_acquire_gpu(f) == 0) {
        const uint64_t t0 = tc::global_timer_ns();
        while (ld_acquire_gpu(f) == 0) {
            if (tc::global_timer_ns() - t0 > G.limit_ns) {
                ok = false;
                break;
            }
            __nanosleep(64);
        }
    }
    ok = __all_sync(0xffffffffu, ok);
    if (!ok) {
        if (lane == 0) flag(G.status, DSV4_DEV_TIMEOUT);
    } else if (f != nullptr) {
        *f = 0;                                      // consumed: the next set guards later inputs
    }
    __syncwarp();
    // the step's kernels may launch now; this grid completes after its
    // predecessor, so their dependency waits still order them after it
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

}  // namespace dsv4

using namespace dsv4;

extern "C" dsv4_status dsv4_stream_gate(const dsv4_gate_args* a, dsv4_stream_t stream)
{
    if (a == nullptr || a->timeout_us < 0) return DSV4_ERR_INVALID;
    GateParams G;
    int n = 0;
    for (int i = 0; i < 4; ++i) {
        G.f[i] = a->flags_dev[i];
        if (G.f[i] == nullptr) continue;
        if (reinterpret_cast<uintptr_t>(G.f[i]) & 3) return DSV4_ERR_SHAPE;
        ++n;
    }
    if (n == 0) return DSV4_ERR_INVALID;
    G.limit_ns = a->timeout_us > 0 ? static_cast<unsigned long long>(a->timeout_us) * 1000ull : tc::kWaitNs;
    G.status = a->status_dev;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(1, 1, 1);
    cfg.blockDim = dim3(32, 1, 1);
    cfg.stream = reinterpret_cast<cudaStream_t>(stream);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, stream_gate_kernel, G) == cudaSuccess ? DSV4_OK : DSV4_ERR_CUDA;
}
