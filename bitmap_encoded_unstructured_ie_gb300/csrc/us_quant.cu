// us_quant.cu -- per-token int4 quantisation of fp16 activations.
//
// "UnionSparse: An Index-Efficient Sparsity Framework for Low-Bit Sparse LLM
// Inference on Edge", Fig. 2: FP16 X -> Quant -> INT4 X with one scale per
// token, ahead of the INT4 x INT4 SpMM.  s = fp16_rn(amax / 7) (1 if that is 0),
// code = clamp(rint(x / s), -8, 7), both divisions in fp32, ties to even.
//
// One CTA per token: 16-byte loads of eight fp16 values, a block maximum, then a
// second pass over the (cached) row that writes eight packed codes per thread.
#include "us_common.cuh"
#include "us_internal.h"

namespace {

constexpr int kThreads = 256;

__global__ void __launch_bounds__(kThreads)
quantize_x_kernel(const uint16_t* __restrict__ X, int K, uint8_t* __restrict__ Xq, uint16_t* __restrict__ s_x) {
    __shared__ float wmax[kThreads / 32];
    const int n = blockIdx.x;
    const uint4* xv = reinterpret_cast<const uint4*>(X + (int64_t)n * K);
    const int chunks = K / 8;
    us::pdl_wait();
    float amax = 0.f;
    for (int c = threadIdx.x; c < chunks; c += kThreads) {
        const uint4 v = xv[c];
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            amax = fmaxf(amax, fabsf(us::half_bits_to_float((uint16_t)(w[i] & 0xFFFFu))));   // NaN ignored
            amax = fmaxf(amax, fabsf(us::half_bits_to_float((uint16_t)(w[i] >> 16))));
        }
    }
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, d));
    if ((threadIdx.x & 31) == 0) wmax[threadIdx.x >> 5] = amax;
    __syncthreads();
    amax = wmax[0];
#pragma unroll
    for (int i = 1; i < kThreads / 32; ++i) amax = fmaxf(amax, wmax[i]);
    uint16_t s16 = us::float_to_half_bits(amax / 7.0f);
    if ((s16 & 0x7FFFu) == 0) s16 = 0x3C00u;                  // 1.0
    const float s = us::half_bits_to_float(s16);
    if (threadIdx.x == 0) s_x[n] = s16;
    uint32_t* out = reinterpret_cast<uint32_t*>(Xq + (int64_t)n * (K / 2));
    for (int c = threadIdx.x; c < chunks; c += kThreads) {
        const uint4 v = xv[c];
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
        uint32_t packed = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const uint16_t h = (uint16_t)(w[i >> 1] >> (16 * (i & 1)));
            float q = rintf(us::half_bits_to_float(h) / s);
            if (!(q == q)) q = 0.f;
            q = fminf(fmaxf(q, -8.f), 7.f);
            packed |= ((uint32_t)(int)q & 0xFu) << (4 * i);   // element 2j low nibble, 2j+1 high
        }
        out[c] = packed;
    }
    us::pdl_launch_dependents();
}

}  // namespace

namespace us {

us_status launch_quantize_x(const uint16_t* X, int N, int K, uint8_t* Xq, uint16_t* s_x, cudaStream_t st) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)N);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, quantize_x_kernel, X, K, Xq, s_x) == cudaSuccess ? US_OK : US_ERR_CUDA;
}

}  // namespace us
