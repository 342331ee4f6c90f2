// gelu.cu -- the MLP activation of the transformer layer around the
// attention core, for the layer-level measurement of selective activation
// recomputation ("Reducing Activation Recomputation in Large Transformer
// Models", Key takeaways, fourth bullet: recomputing the whole layer against
// only the attention core).  GeLU in its tanh form,
//     y = x / 2 * (1 + tanh(c (x + a x^3))),  c = sqrt(2 / pi), a = 0.044715,
//     dy/dx = (1 + t) / 2 + x / 2 * (1 - t^2) * c * (1 + 3 a x^2),  t = tanh(...),
// elementwise on bf16 (fp32 arithmetic).  HBM-bound: 16-byte vectors,
// grid-stride over a grid of 4 CTAs per SM.
#include "kernels.h"
#include "ptx.cuh"

namespace ac {

namespace {

constexpr float kGeluC = 0.7978845608028654f;   // sqrt(2 / pi)
constexpr float kGeluA = 0.044715f;

__device__ __forceinline__ float gelu_f(float x)
{
    const float t = tanhf(kGeluC * fmaf(kGeluA * x * x, x, x));
    return 0.5f * x * (1.0f + t);
}

__device__ __forceinline__ float gelu_grad(float x)
{
    const float t = tanhf(kGeluC * fmaf(kGeluA * x * x, x, x));
    return 0.5f * (1.0f + t) + 0.5f * x * (1.0f - t * t) * kGeluC * fmaf(3.0f * kGeluA, x * x, 1.0f);
}

__device__ __forceinline__ void unpack8(const uint4 v, float (&f)[8])
{
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        f[2 * e] = __uint_as_float(w[e] << 16);
        f[2 * e + 1] = __uint_as_float(w[e] & 0xFFFF0000u);
    }
}

__device__ __forceinline__ uint4 pack8(const float (&f)[8])
{
    return make_uint4(pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]), pack_bf16x2(f[4], f[5]),
                      pack_bf16x2(f[6], f[7]));
}

}  // namespace

__global__ void __launch_bounds__(256) gelu_fwd_kernel(const uint16_t* x, uint16_t* y, int64_t n8)
{
    for (int64_t i = blockIdx.x * 256ll + threadIdx.x; i < n8; i += (int64_t)gridDim.x * 256) {
        float f[8];
        unpack8(reinterpret_cast<const uint4*>(x)[i], f);
#pragma unroll
        for (int e = 0; e < 8; ++e) f[e] = gelu_f(f[e]);
        reinterpret_cast<uint4*>(y)[i] = pack8(f);
    }
}

__global__ void __launch_bounds__(256) gelu_bwd_kernel(const uint16_t* x, const uint16_t* dy, uint16_t* dx,
                                                       int64_t n8)
{
    for (int64_t i = blockIdx.x * 256ll + threadIdx.x; i < n8; i += (int64_t)gridDim.x * 256) {
        float f[8], g[8];
        unpack8(reinterpret_cast<const uint4*>(x)[i], f);
        unpack8(reinterpret_cast<const uint4*>(dy)[i], g);
#pragma unroll
        for (int e = 0; e < 8; ++e) g[e] *= gelu_grad(f[e]);
        reinterpret_cast<uint4*>(dx)[i] = pack8(g);
    }
}

int launch_gelu_fwd(const uint16_t* x, uint16_t* y, int64_t n, int sms, cudaStream_t st)
{
    const int64_t n8 = n / 8;
    const int64_t want = (n8 + 255) / 256;
    const int grid = (int)(want < 4ll * sms ? want : 4ll * sms);
    gelu_fwd_kernel<<<grid > 0 ? grid : 1, 256, 0, st>>>(x, y, n8);
    return (int)cudaGetLastError();
}

int launch_gelu_bwd(const uint16_t* x, const uint16_t* dy, uint16_t* dx, int64_t n, int sms, cudaStream_t st)
{
    const int64_t n8 = n / 8;
    const int64_t want = (n8 + 255) / 256;
    const int grid = (int)(want < 4ll * sms ? want : 4ll * sms);
    gelu_bwd_kernel<<<grid > 0 ? grid : 1, 256, 0, st>>>(x, dy, dx, n8);
    return (int)cudaGetLastError();
}

}  // namespace ac
