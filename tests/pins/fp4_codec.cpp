// Host-side E2M1 codec from CUDA's cuda_fp4.h (a library routine), built by
// the FP4 oracle tests to pin the oracle's own codec against.
#include <cuda_fp4.h>

extern "C" float pin_e2m1_decode(int code)
{
    const __half_raw h = __nv_cvt_fp4_to_halfraw(static_cast<__nv_fp4_storage_t>(code), __NV_E2M1);
    return __half2float(__half(h));
}

extern "C" int pin_e2m1_encode(float x)
{
    return static_cast<int>(__nv_cvt_float_to_fp4(x, __NV_E2M1, cudaRoundNearest));
}
