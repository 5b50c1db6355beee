// Device side of the synthetic input generator (see gen.h).  Produces the
// same bits as synth_host.c: integer hashing, one double multiply
// (__dmul_rn, never contracted) and __double2float_rn.
#include <cuda_runtime.h>
#include <stdint.h>

#include "gen.h"

namespace {

__device__ __forceinline__ float dev_value_f32(const syn_stream_t& st, uint64_t n) {
    double z = syn_normal(st.key, n);
    double s = syn_is_outlier(st.key_out, n, st.thr) ? st.sigma_out : st.sigma;
    return __double2float_rn(__dmul_rn(z, s));
}

// KIND 0: fp32, 1: bf16, 2: fp16
template <int KIND>
__global__ void fill_kernel(syn_stream_t st, int64_t start, int64_t n, void* out) {
    int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride) {
        float f = dev_value_f32(st, (uint64_t)(start + i));
        if (KIND == 1)
            static_cast<uint16_t*>(out)[i] = syn_f32bits_to_bf16(__float_as_uint(f));
        else if (KIND == 2)
            static_cast<uint16_t*>(out)[i] = syn_f32bits_to_f16(__float_as_uint(f));
        else
            static_cast<float*>(out)[i] = f;
    }
}

int launch(const syn_stream_t* st, int64_t start, int64_t n, void* out, int kind, void* stream) {
    if (n <= 0) return 0;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return -1;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return -1;
    int64_t want = (n + 255) / 256;
    int64_t cap = (int64_t)sms * 16;
    unsigned grid = (unsigned)(want < cap ? want : cap);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (kind == 1)
        fill_kernel<1><<<grid, 256, 0, s>>>(*st, start, n, out);
    else if (kind == 2)
        fill_kernel<2><<<grid, 256, 0, s>>>(*st, start, n, out);
    else
        fill_kernel<0><<<grid, 256, 0, s>>>(*st, start, n, out);
    return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

}  // namespace

extern "C" int synth_dev_fill_bf16(const syn_stream_t* st, int64_t start, int64_t n, uint16_t* out, void* stream) {
    return launch(st, start, n, out, 1, stream);
}

extern "C" int synth_dev_fill_f32(const syn_stream_t* st, int64_t start, int64_t n, float* out, void* stream) {
    return launch(st, start, n, out, 0, stream);
}

extern "C" int synth_dev_fill_f16(const syn_stream_t* st, int64_t start, int64_t n, uint16_t* out, void* stream) {
    return launch(st, start, n, out, 2, stream);
}
