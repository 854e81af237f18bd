// The pre-attention LayerNorm (sm_103a): h = (x - mean) / sqrt(var + eps) * w
// per row of 768, the mean and the population variance over the row, a
// learned weight and no bias ("ModernBERT-base Architecture Teardown", "What
// Does LayerNorm Do?"; every norm of the checkpoint is weight-only,
// "ModernBERT" (candding), "The pre-norm layer and the final norm").
//
// HBM-bound: each row is read once (1536 B) and written once.  One warp per
// row; lane l holds the 16-byte chunks l, l + 32 and l + 64 of the row, so a
// warp's load or store instruction moves 512 contiguous bytes.  Statistics in
// fp32, two passes over the registers (mean, then squared deviations), each
// reduced across the warp with shuffles; the weight is loaded once per warp.
#include "common.cuh"
#include "internal.h"

namespace mbert {
namespace {

constexpr int kRowChunks = kHidden / 8;         // 96 chunks of 8 bf16
constexpr int kChunksPerLane = kRowChunks / 32; // 3
constexpr int kWarpsPerBlock = 8;

__device__ __forceinline__ void unpack8(const uint4 &u, float (&f)[8])
{
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        f[2 * e] = bf16lo_to_f32(w[e]);
        f[2 * e + 1] = bf16hi_to_f32(w[e]);
    }
}

__device__ __forceinline__ float warp_sum(float v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

__global__ void __launch_bounds__(32 * kWarpsPerBlock)
layernorm_kernel(const __nv_bfloat16 *__restrict__ x, const __nv_bfloat16 *__restrict__ w,
                 long long T, float eps, __nv_bfloat16 *__restrict__ h)
{
    pdl_wait();
    const int lane = threadIdx.x & 31;
    const long long first = static_cast<long long>(blockIdx.x) * kWarpsPerBlock + (threadIdx.x >> 5);
    const long long stride = static_cast<long long>(gridDim.x) * kWarpsPerBlock;
    float wv[kChunksPerLane][8];
#pragma unroll
    for (int j = 0; j < kChunksPerLane; ++j)
        unpack8(reinterpret_cast<const uint4 *>(w)[lane + 32 * j], wv[j]);
    constexpr float kInvD = 1.0f / kHidden;
    for (long long row = first; row < T; row += stride) {
        const uint4 *xr = reinterpret_cast<const uint4 *>(x + row * kHidden);
        float v[kChunksPerLane][8];
#pragma unroll
        for (int j = 0; j < kChunksPerLane; ++j)
            unpack8(xr[lane + 32 * j], v[j]);
        float s = 0.f;
#pragma unroll
        for (int j = 0; j < kChunksPerLane; ++j)
#pragma unroll
            for (int e = 0; e < 8; ++e)
                s += v[j][e];
        const float mean = warp_sum(s) * kInvD;
        float q = 0.f;
#pragma unroll
        for (int j = 0; j < kChunksPerLane; ++j)
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                v[j][e] -= mean;
                q += v[j][e] * v[j][e];
            }
        const float rstd = rsqrtf(warp_sum(q) * kInvD + eps);
        uint4 *hr = reinterpret_cast<uint4 *>(h + row * kHidden);
#pragma unroll
        for (int j = 0; j < kChunksPerLane; ++j) {
            uint4 o;
            o.x = pack_bf16x2(v[j][0] * rstd * wv[j][0], v[j][1] * rstd * wv[j][1]);
            o.y = pack_bf16x2(v[j][2] * rstd * wv[j][2], v[j][3] * rstd * wv[j][3]);
            o.z = pack_bf16x2(v[j][4] * rstd * wv[j][4], v[j][5] * rstd * wv[j][5]);
            o.w = pack_bf16x2(v[j][6] * rstd * wv[j][6], v[j][7] * rstd * wv[j][7]);
            hr[lane + 32 * j] = o;
        }
    }
    pdl_trigger();
}

}  // namespace

cudaError_t launch_layernorm(const __nv_bfloat16 *x, const __nv_bfloat16 *w, long long T,
                             float eps, __nv_bfloat16 *h, int num_sms, cudaStream_t stream)
{
    if (T <= 0)
        return cudaSuccess;
    const long long need = (T + kWarpsPerBlock - 1) / kWarpsPerBlock;
    const long long cap = static_cast<long long>(num_sms) * 8;      // 64 resident warps per SM
    const int grid = static_cast<int>(need < cap ? need : cap);
    return launch_chained(layernorm_kernel, dim3(grid), dim3(32 * kWarpsPerBlock), 0, stream, x, w, T,
                          eps, h);
}

}  // namespace mbert
