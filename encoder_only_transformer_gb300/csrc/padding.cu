// The padded-batch form to and from the packed form (sm_103a).
//
// A padded batch holds B rows of S tokens with an attention mask of 1 for a
// real token and 0 for a pad ("ModernBERT-base Architecture Teardown", the
// tokenizer with padding=True: the mask marks the [PAD] tokens, which no
// real token may take information from; "Encoder-only models", "Padding and
// the key padding mask": pad keys get -inf, so real outputs do not depend on
// how long the batch-mates were).  Packing each row's real tokens, in order,
// into one sequence of the packed form gives exactly that: every key of a
// row's sequence is a real token of the row.  A real token's position is its
// rank among the row's real tokens, which for a right-padded row (the
// tokenizer's form) is its index in the row.
//
// mask_rows_kernel: one block per row, a block-wide exclusive scan of
// (mask != 0).  mask_offsets_kernel: one block, the exclusive scan of the
// row counts.  gather / scatter: one warp per padded row, 16-byte vectors.
#include "common.cuh"
#include "internal.h"

namespace mbert {
namespace {

constexpr int kScanThreads = 1024;

// Exclusive block-wide sum of one int per thread; *total gets the sum.
__device__ int block_exclusive_scan(int v, int *total)
{
    __shared__ int s_warp[kScanThreads / 32];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o)
            x += y;
    }
    if (lane == 31)
        s_warp[warp] = x;
    __syncthreads();
    if (warp == 0) {
        int w = lane < (blockDim.x >> 5) ? s_warp[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o)
                w += y;
        }
        s_warp[lane] = w;                       // inclusive sums of the warps
    }
    __syncthreads();
    const int before = (warp > 0 ? s_warp[warp - 1] : 0) + x - v;
    *total = s_warp[(blockDim.x >> 5) - 1];
    __syncthreads();                            // s_warp is reused by the next call
    return before;
}

__global__ void __launch_bounds__(kScanThreads)
mask_rows_kernel(const int32_t *__restrict__ mask, int S, int32_t *__restrict__ rank,
                 int32_t *__restrict__ len)
{
    pdl_wait();
    const int b = blockIdx.x;
    const int32_t *m = mask + static_cast<size_t>(b) * S;
    int32_t *rk = rank + static_cast<size_t>(b) * S;
    int carry = 0;
    for (int s0 = 0; s0 < S; s0 += kScanThreads) {
        const int s = s0 + threadIdx.x;
        const int real = s < S && m[s] != 0 ? 1 : 0;
        int total;
        const int before = block_exclusive_scan(real, &total);
        if (s < S)
            rk[s] = real ? carry + before : -1;
        carry += total;
    }
    if (threadIdx.x == 0)
        len[b] = carry;
    pdl_trigger();
}

__global__ void __launch_bounds__(kScanThreads)
mask_offsets_kernel(const int32_t *__restrict__ len, int B, int32_t *__restrict__ cu)
{
    pdl_wait();
    int carry = 0;
    for (int b0 = 0; b0 < B; b0 += kScanThreads) {
        const int b = b0 + threadIdx.x;
        const int v = b < B ? len[b] : 0;
        int total;
        const int before = block_exclusive_scan(v, &total);
        if (b < B)
            cu[b] = carry + before;
        carry += total;
    }
    if (threadIdx.x == 0)
        cu[B] = carry;
    pdl_trigger();
}

// One warp per padded row: a real row moves between padded row b S + s and
// packed row cu[b] + rank; with kScatter a pad row of dst is zeroed.
template <bool kScatter>
__global__ void __launch_bounds__(256)
move_rows_kernel(const __nv_bfloat16 *__restrict__ src, const int32_t *__restrict__ rank,
                 const int32_t *__restrict__ cu, int B, int S, int width,
                 __nv_bfloat16 *__restrict__ dst)
{
    pdl_wait();
    const int lane = threadIdx.x & 31;
    const long long rows = static_cast<long long>(B) * S;
    const long long stride = static_cast<long long>(gridDim.x) * (blockDim.x >> 5);
    const int vecs = width / 8;                           // 16-byte vectors per row
    for (long long pr = static_cast<long long>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
         pr < rows; pr += stride) {
        const int rk = rank[pr];
        const long long b = pr / S;
        if (rk < 0) {
            if (kScatter) {
                uint4 *d = reinterpret_cast<uint4 *>(dst + pr * width);
                for (int v = lane; v < vecs; v += 32)
                    d[v] = make_uint4(0u, 0u, 0u, 0u);
            }
            continue;
        }
        const long long packed = static_cast<long long>(cu[b]) + rk;
        const uint4 *s = reinterpret_cast<const uint4 *>(src + (kScatter ? packed : pr) * width);
        uint4 *d = reinterpret_cast<uint4 *>(dst + (kScatter ? pr : packed) * width);
        for (int v = lane; v < vecs; v += 32)
            d[v] = s[v];
    }
    if (!kScatter) {
        // packed rows past the last sequence hold no token; the attention
        // kernels load the first of them inside the last sequence's last
        // tiles (as keys they are masked, as values they meet a zero weight,
        // so they must be finite): zero the 256 rows that a tile of 256
        // query rows or a key tile with the band's reach can touch
        const long long used = cu[B];
        const long long end = used + 256 < rows ? used + 256 : rows;
        for (long long r = used + static_cast<long long>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
             r < end; r += stride) {
            uint4 *d = reinterpret_cast<uint4 *>(dst + r * width);
            for (int v = lane; v < vecs; v += 32)
                d[v] = make_uint4(0u, 0u, 0u, 0u);
        }
    }
    pdl_trigger();
}

int move_grid(int B, int S, int num_sms)
{
    const long long rows = static_cast<long long>(B) * S;
    const long long need = (rows + 7) / 8;
    const long long cap = static_cast<long long>(num_sms) * 8;
    return static_cast<int>(need < cap ? need : cap);
}

}  // namespace

cudaError_t launch_mask_scan(const int32_t *mask, int B, int S, int32_t *rank, int32_t *len,
                             int32_t *cu, cudaStream_t stream)
{
    if (B <= 0)
        return cudaSuccess;
    cudaError_t e = launch_chained(mask_rows_kernel, dim3(B), dim3(kScanThreads), 0, stream, mask,
                                   S, rank, len);
    if (e == cudaSuccess)
        e = launch_chained(mask_offsets_kernel, dim3(1), dim3(kScanThreads), 0, stream, len, B, cu);
    return e;
}

cudaError_t launch_gather_rows(const __nv_bfloat16 *src, const int32_t *rank, const int32_t *cu,
                               int B, int S, int width, __nv_bfloat16 *dst, int num_sms,
                               cudaStream_t stream)
{
    if (B <= 0 || S <= 0)
        return cudaSuccess;
    return launch_chained(move_rows_kernel<false>, dim3(move_grid(B, S, num_sms)), dim3(256), 0,
                          stream, src, rank, cu, B, S, width, dst);
}

cudaError_t launch_scatter_rows(const __nv_bfloat16 *src, const int32_t *rank, const int32_t *cu,
                                int B, int S, int width, __nv_bfloat16 *dst, int num_sms,
                                cudaStream_t stream)
{
    if (B <= 0 || S <= 0)
        return cudaSuccess;
    return launch_chained(move_rows_kernel<true>, dim3(move_grid(B, S, num_sms)), dim3(256), 0,
                          stream, src, rank, cu, B, S, width, dst);
}

}  // namespace mbert
