// Preparatory kernels of the attention block: the device-side plan (checks
// cu_seqlens and writes the work list), the RoPE pass over Q and K, and the
// admitted-key count used to verify the schedule.
#include "common.cuh"
#include "internal.h"

namespace mbert {
namespace {

constexpr int kPlanThreads = 1024;
constexpr int kMaxBins = 1024;   // 128-query blocks per sequence: max_seqlen <= 131072

// Inclusive block-wide scan of one int per thread (blockDim.x == 1024).
__device__ int block_inclusive_scan(int v, int *warp_sums)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        int n = __shfl_up_sync(0xffffffffu, v, d);
        if (lane >= d)
            v += n;
    }
    if (lane == 31)
        warp_sums[warp] = v;
    __syncthreads();
    if (warp == 0) {
        int w = warp_sums[lane];
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            int n = __shfl_up_sync(0xffffffffu, w, d);
            if (lane >= d)
                w += n;
        }
        warp_sums[lane] = w;
    }
    __syncthreads();
    if (warp > 0)
        v += warp_sums[warp - 1];
    return v;
}

// One block.  Checks cu_seqlens (cu[0] == 0, non-decreasing, cu[n] == T --
// or cu[n] <= T with cu_short_ok, when rows past the last sequence belong to
// none -- every length <= max_seqlen) and writes the work list: for each sequence,
// its ceil(L/blk) query blocks of blk rows, sequences ordered by decreasing block count
// (longest-processing-time first; the order inside a bin is arbitrary and
// does not affect any result).
__device__ void plan_block(const int32_t *__restrict__ cu, int n_seqs, long long T, int max_seqlen, int blk,
                           int cu_short_ok, int32_t *err, int2 *__restrict__ work,
                           int32_t *__restrict__ work_count, int32_t *__restrict__ tile_start,
                           int32_t *__restrict__ unit_cnt)
{
    __shared__ int s_bad;
    __shared__ int s_hist[kMaxBins + 1];
    __shared__ int s_off[kMaxBins + 1];
    __shared__ int s_warp[32];
    const int tid = threadIdx.x;
    const int nbmax = (max_seqlen + blk - 1) / blk;   // <= kMaxBins (host-checked)

    if (tid == 0)
        s_bad = 0;
    for (int i = tid; i <= kMaxBins; i += kPlanThreads)
        s_hist[i] = 0;
    __syncthreads();
    if (tid == 0 && (cu[0] != 0 || (cu_short_ok ? static_cast<long long>(cu[n_seqs]) > T
                                                : static_cast<long long>(cu[n_seqs]) != T)))
        atomicOr(&s_bad, kErrBadCu);
    for (int s = tid; s < n_seqs; s += kPlanThreads) {
        const int L = cu[s + 1] - cu[s];
        if (L < 0)
            atomicOr(&s_bad, kErrBadCu);
        else if (L > max_seqlen)
            atomicOr(&s_bad, kErrTooLong);
        else
            atomicAdd(&s_hist[(L + blk - 1) / blk], 1);
    }
    __syncthreads();
    if (s_bad) {
        if (tid == 0) {
            atomicOr(err, s_bad);
            *work_count = 0;
        }
        return;
    }
    // Entries of bin b (sequences with b blocks) start after every bin with
    // more blocks: off[b] = sum over b' > b of hist[b'] * b'.  Thread t owns
    // bin nbmax - t, so an inclusive scan in thread order is a suffix sum.
    const int b = nbmax - tid;
    const int mine = (b >= 1) ? s_hist[b] * b : 0;
    const int incl = block_inclusive_scan(mine, s_warp);
    if (b >= 1)
        s_off[b] = incl - mine;
    if (tid == kPlanThreads - 1)
        *work_count = incl;
    __syncthreads();
    // reuse s_hist as the per-bin cursor
    for (int i = tid; i <= kMaxBins; i += kPlanThreads)
        s_hist[i] = 0;
    __syncthreads();
    for (int s = tid; s < n_seqs; s += kPlanThreads) {
        const int L = cu[s + 1] - cu[s];
        const int nb = (L + blk - 1) / blk;
        if (nb == 0)
            continue;
        const int slot = atomicAdd(&s_hist[nb], 1);
        int2 *dst = work + s_off[nb] + slot * nb;
        for (int q = 0; q < nb; ++q)
            dst[q] = make_int2(s, q);
    }
    if (tile_start == nullptr)
        return;
    // Iteration offsets of the entries, in list order: an exclusive scan of
    // heads * ceil(L/128) (one iteration per head and key tile).
    __syncthreads();
    __shared__ int s_carry;
    const int total = *work_count;
    if (tid == 0)
        s_carry = 0;
    __syncthreads();
    for (int b = 0; b < total; b += kPlanThreads) {
        const int e = b + tid;
        int v = 0;
        if (e < total) {
            const int2 w = work[e];
            const int L = cu[w.x + 1] - cu[w.x];
            v = kHeads * ((L + kBlockN - 1) / kBlockN);
        }
        const int incl = block_inclusive_scan(v, s_warp);
        if (e < total)
            tile_start[e] = s_carry + incl - v;
        __syncthreads();
        if (tid == kPlanThreads - 1)
            s_carry += incl;
        __syncthreads();
    }
    if (tid == 0)
        tile_start[total] = s_carry;
    for (int i = tid; i < total * kHeads; i += kPlanThreads)
        unit_cnt[i] = 0;
}

__global__ void __launch_bounds__(kPlanThreads)
plan_kernel(const int32_t *__restrict__ cu, int n_seqs, long long T, int max_seqlen, int blk,
            int cu_short_ok, int32_t *err, int2 *__restrict__ work, int32_t *__restrict__ work_count,
            int32_t *__restrict__ tile_start, int32_t *__restrict__ unit_cnt)
{
    pdl_wait();
    plan_block(cu, n_seqs, T, max_seqlen, blk, cu_short_ok, err, work, work_count, tile_start, unit_cnt);
    pdl_trigger();
}

// Sequence index of packed row `row` (cu validated, non-decreasing).
__device__ __forceinline__ int seq_of_row(const int32_t *__restrict__ cu, int n_seqs, long long row)
{
    int lo = 0, hi = n_seqs;
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (static_cast<long long>(__ldg(cu + mid)) <= row)
            lo = mid;
        else
            hi = mid;
    }
    return lo;
}

constexpr int kRopeThreadsPerRow = 2 * kHeads * (kPairs / 8);   // 96: 24 head blocks x 4 chunks
constexpr int kRopeRowsPerCta = kPlanThreads / kRopeThreadsPerRow;   // 10 rows of a 1024-thread block

// Rotate-half RoPE of Q and K ("ModernBERT" (candding), "The two rope
// tables"): for pair m = (x[m], x[m+32]) at position p,
//   y[m] = x[m] cos - x[m+32] sin,  y[m+32] = x[m+32] cos + x[m] sin,
// with (cos, sin) of p * base^(-2m/64) from the fp32 table.  Each thread
// rotates 8 pairs of one head of Q or K, rows 10 b .. 10 b + 9 for block b;
// the result is rounded to bf16.  Positions come from cu_seqlens by binary
// search; with cu_seqlens the plan rejects, the rows still land in rot[T]
// (and the table index is clamped), and the attention kernel reads none.
//
// With `norms` set, the pass also records the Euclidean norm of every
// rounded row and head: Q head h in norms[h][row] (fp32), K head h in
// knorm[h][row] as fp16 rounded up (an upper bound: +inf past the fp16
// range), rows `norm_pitch` apart.  By Cauchy-Schwarz |q . k| <= |q| |k|,
// so these bound every score.
__device__ void rope_block(long long b, const __nv_bfloat16 *__restrict__ qkv,
                           const int32_t *__restrict__ cu, int n_seqs, long long T,
                           const float2 *__restrict__ table, int table_rows, __nv_bfloat16 *__restrict__ rot,
                           float *__restrict__ norms, uint16_t *__restrict__ knorm, long long norm_pitch)
{
    const long long row = b * kRopeRowsPerCta + threadIdx.x / kRopeThreadsPerRow;
    // whole warps drop out here: a row is three full warps
    if (threadIdx.x < kRopeRowsPerCta * kRopeThreadsPerRow && row < T) {
        const int sub = threadIdx.x % kRopeThreadsPerRow;
        const int blk = sub >> 2;          // 0..11 Q heads, 12..23 K heads
        const int chunk = sub & 3;         // pairs chunk*8 .. chunk*8+7
        const int s = seq_of_row(cu, n_seqs, row);
        int pos = static_cast<int>(row - __ldg(cu + s));
        pos = min(max(pos, 0), table_rows - 1);
        const int col = blk * kHeadDim + chunk * 8;

        const uint4 a = __ldg(reinterpret_cast<const uint4 *>(qkv + row * kQKVWidth + col));
        const uint4 bb = __ldg(reinterpret_cast<const uint4 *>(qkv + row * kQKVWidth + col + kPairs));
        const float4 *cs = reinterpret_cast<const float4 *>(table + static_cast<long long>(pos) * kPairs + chunk * 8);
        const uint32_t av[4] = {a.x, a.y, a.z, a.w};
        const uint32_t bv[4] = {bb.x, bb.y, bb.z, bb.w};
        uint32_t ya[4], yb[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float4 t = __ldg(cs + i);          // (cos, sin) of pairs 2i, 2i+1
            const float x0 = bf16lo_to_f32(av[i]), x1 = bf16hi_to_f32(av[i]);
            const float z0 = bf16lo_to_f32(bv[i]), z1 = bf16hi_to_f32(bv[i]);
            const float y0 = x0 * t.x - z0 * t.y;
            const float y1 = x1 * t.z - z1 * t.w;
            const float w0 = z0 * t.x + x0 * t.y;
            const float w1 = z1 * t.z + x1 * t.w;
            ya[i] = pack_bf16x2(y0, y1);
            yb[i] = pack_bf16x2(w0, w1);
        }
        constexpr int kRotWidth = 2 * kHidden;
        *reinterpret_cast<uint4 *>(rot + row * kRotWidth + col) = make_uint4(ya[0], ya[1], ya[2], ya[3]);
        *reinterpret_cast<uint4 *>(rot + row * kRotWidth + col + kPairs) = make_uint4(yb[0], yb[1], yb[2], yb[3]);
        if (norms) {
            // squared norm of the 16 rounded values, then of the head's 64
            // (the four chunk threads of a (row, head) are neighbouring lanes)
            float sq = 0.f;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float y0 = bf16lo_to_f32(ya[i]), y1 = bf16hi_to_f32(ya[i]);
                const float w0 = bf16lo_to_f32(yb[i]), w1 = bf16hi_to_f32(yb[i]);
                sq = fmaf(y0, y0, sq);
                sq = fmaf(y1, y1, sq);
                sq = fmaf(w0, w0, sq);
                sq = fmaf(w1, w1, sq);
            }
            sq += __shfl_xor_sync(0xffffffffu, sq, 1);
            sq += __shfl_xor_sync(0xffffffffu, sq, 2);
            if (chunk == 0) {
                const float nrm = sqrtf(sq);
                if (blk < kHeads)
                    norms[blk * norm_pitch + row] = nrm;
                else
                    knorm[(blk - kHeads) * norm_pitch + row] = __half_as_ushort(__float2half_ru(nrm));
            }
        }
    }
}

// The plan and the RoPE pass in one launch: block 0 builds the plan, blocks
// 1.. rotate rows.  The RoPE pass does not read the plan.
__global__ void __launch_bounds__(kPlanThreads)
plan_rope_kernel(const int32_t *__restrict__ cu, int n_seqs, long long T, int max_seqlen, int blk,
                 int cu_short_ok, int32_t *err, int2 *__restrict__ work, int32_t *__restrict__ work_count,
                 int32_t *__restrict__ tile_start, int32_t *__restrict__ unit_cnt,
                 const __nv_bfloat16 *__restrict__ qkv, const float2 *__restrict__ table, int table_rows,
                 __nv_bfloat16 *__restrict__ rot, float *__restrict__ norms, uint16_t *__restrict__ knorm,
                 long long norm_pitch)
{
    pdl_wait();
    if (blockIdx.x == 0)
        plan_block(cu, n_seqs, T, max_seqlen, blk, cu_short_ok, err, work, work_count, tile_start, unit_cnt);
    else
        rope_block(blockIdx.x - 1, qkv, cu, n_seqs, T, table, table_rows, rot, norms, knorm, norm_pitch);
    pdl_trigger();
}

// One CTA of 128 threads per work entry; thread r is query position
// q0 + r.  Walks exactly the key tiles the attention kernels visit and
// counts the keys they let into the softmax: all 128 of a tile that needs
// no mask, else the admitted ones.
__global__ void __launch_bounds__(kBlockM)
key_count_kernel(const int32_t *__restrict__ cu, const int2 *__restrict__ work,
                 const int32_t *__restrict__ work_count, int hw, int32_t *__restrict__ counts)
{
    pdl_wait();
    if (static_cast<int>(blockIdx.x) >= *work_count)
        return;
    const int2 e = work[blockIdx.x];
    const int row0 = cu[e.x];
    const int L = cu[e.x + 1] - row0;
    const int q0 = e.y * kBlockM;
    const int qpos = q0 + threadIdx.x;
    int cnt = 0;
    if (hw >= 0 && hw <= kBandReach) {
        // the local kernel: two band tiles, chunks chosen per warp
        const int w = threadIdx.x >> 5;
        for (int t = 0; t < 2; ++t) {
            const int key0 = band_tile_key0(q0, t);
            for (int c = band_chunk_begin(t, w); c < band_chunk_end(t, w); ++c) {
                if (!band_chunk_needs_mask(q0, L, hw, t, w, c)) {
                    cnt += 32;
                    continue;
                }
                for (int k = 0; k < 32; ++k) {
                    const int kp = key0 + 32 * c + k;
                    cnt += (kp >= 0 && kp < L && abs(qpos - kp) <= hw) ? 1 : 0;
                }
            }
        }
    } else {
        int kt0, kt1;
        key_tile_range(q0, L, hw, kt0, kt1);
        for (int kt = kt0; kt < kt1; ++kt) {
            if (!tile_needs_mask(q0, L, hw, kt)) {
                cnt += kBlockN;
                continue;
            }
            for (int c = 0; c < kBlockN; ++c)
                cnt += admitted(qpos, kt * kBlockN + c, L, hw) ? 1 : 0;
        }
    }
    if (qpos < L)
        counts[row0 + qpos] = cnt;
    pdl_trigger();
}

// Self-test of the bounded wait: one thread initialises an mbarrier that
// nothing ever arrives on and waits for it with a short limit.  The wait must
// give up, set kErrTimeout in the error word and let the kernel return.
__global__ void wait_timeout_selftest_kernel(int32_t *err, unsigned long long limit_ns)
{
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x != 0)
        return;
    const uint32_t b = smem_u32(&bar);
    mbar_init(b, 1);
    fence_mbar_init();
    mbar_wait(b, 0, err, limit_ns);
}

}  // namespace

cudaError_t launch_wait_timeout_selftest(int32_t *err, unsigned long long limit_ns,
                                         cudaStream_t stream)
{
    wait_timeout_selftest_kernel<<<1, 32, 0, stream>>>(err, limit_ns);
    return cudaGetLastError();
}

cudaError_t launch_plan(const Plan &p, cudaStream_t stream)
{
    return launch_chained(plan_kernel, dim3(1), dim3(kPlanThreads), 0, stream, p.cu, p.n_seqs, p.T,
                          p.max_seqlen, p.block, p.cu_short_ok ? 1 : 0, p.err, p.work,
                          p.work_count, p.tile_start, p.unit_cnt);
}

cudaError_t launch_plan_rope(const Plan &p, const __nv_bfloat16 *qkv, const float2 *table,
                             int table_rows, __nv_bfloat16 *rot, float *norms, uint16_t *knorm,
                             long long norm_pitch, cudaStream_t stream)
{
    const long long blocks = 1 + (p.T + kRopeRowsPerCta - 1) / kRopeRowsPerCta;
    return launch_chained(plan_rope_kernel, dim3(static_cast<unsigned>(blocks)), dim3(kPlanThreads), 0, stream,
                          p.cu, p.n_seqs, p.T, p.max_seqlen, p.block, p.cu_short_ok ? 1 : 0, p.err, p.work,
                          p.work_count, p.tile_start, p.unit_cnt, qkv, table, table_rows, rot, norms,
                          knorm, norm_pitch);
}

cudaError_t launch_key_count(const Plan &p, int half_window, int32_t *counts, cudaStream_t stream)
{
    return launch_chained(key_count_kernel, dim3(p.entry_bound), dim3(kBlockM), 0, stream, p.cu,
                          p.work, p.work_count, half_window, counts);
}

}  // namespace mbert
