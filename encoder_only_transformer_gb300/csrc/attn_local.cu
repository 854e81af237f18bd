// Local-layer attention with RoPE fused into the prologue (tcgen05 + TMA,
// sm_103a).
//
// One CTA per (128-query block, head): 4 compute warps (thread r owns query
// row q0 + r, TMEM lane r) and one issuer warp (TMA and MMA, one elected
// lane).  A local layer keeps key j for query i when |i - j| <= 64 ("ModernBERT"
// (candding), "The alternating attention"), so two 128-key tiles offset by
// -64 and +64 from the block hold every visible key; warps skip the 32-key
// chunks their rows cannot see (see the band helpers in common.cuh).
//
//   TMA   raw Q, K0, K1, V0, V1 tiles (5 x 16 KB, 128-byte swizzle) straight
//         from the fused qkv rows
//   RoPE  in shared memory, rotate-half, base 10000, positions restarting
//         per sequence ("ModernBERT-base Architecture Teardown", "How Does
//         RoPE Work With Two Bases?"); each thread rotates one K row of each
//         tile and the Q row at the same position with the same cos/sin,
//         which it computes itself from the frequencies
//   S0 = Q K0^T -> softmax -> P0, O = P0 V0, S1 = Q K1^T -> softmax -> P1,
//   O += P1 V1  (fp32 online softmax over the two tiles, base 2; the
//         reference maximum moves only when tile 1's maximum exceeds it by
//         more than 8)
//   out = O / l in bf16.
// TMEM (256 columns, two CTAs per SM): S [0,128) P [128,192) O [192,256).
//
// The block is found from cu_seqlens by the CTA itself (no plan kernel) when
// the work list is null; then every CTA also checks the whole cu_seqlens
// array, so a bad array makes every CTA exit without writing.
#include "common.cuh"
#include "internal.h"

namespace mbert {
namespace {

constexpr int kThreads = 160;
constexpr int kCompute = 128;
constexpr uint32_t kOffQ = 0;
constexpr uint32_t kOffK = 16384;       // K0, K1
constexpr uint32_t kOffV = 49152;       // V0, V1
constexpr uint32_t kOffBar = 81920;
constexpr uint32_t kSmemBytes = kOffBar + 128 + 1024;
constexpr uint32_t kTmemCols = 256;
constexpr uint32_t kColS = 0, kColP = 128, kColO = 192;

constexpr int kBarQK = 0, kBarV = 1, kBarRope = 2, kBarS = 3, kBarP = 4, kBarO = 5;

constexpr uint32_t kIdescS = make_idesc_bf16(128, 128, false);
constexpr uint32_t kIdescO = make_idesc_bf16(128, 64, true);
constexpr float kScaleLog2 = 0.125f * 1.4426950408889634f;
constexpr float kRescaleThreshold = 8.0f;

__device__ __forceinline__ uint32_t barp(uint32_t base, int i) { return base + kOffBar + 8u * i; }

// Rotate one 128-byte swizzled row (64 bf16) in place, 8 pairs (one chunk
// pair j, j+4) at a time: pair m = (x[m], x[m+32]) turns by the angle whose
// cosine and sine are c[m - 8j], s[m - 8j].  16-byte chunk j of row r sits
// at chunk j ^ (r % 8).
__device__ __forceinline__ void rope_chunk(uint32_t row_addr, int r, int j, const float (&c)[8],
                                           const float (&s)[8])
{
    const uint32_t a = row_addr + ((j ^ (r & 7)) << 4);
    const uint32_t b = row_addr + (((j + 4) ^ (r & 7)) << 4);
    uint32_t x[4], z[4];
    asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];" : "=r"(x[0]), "=r"(x[1]), "=r"(x[2]), "=r"(x[3]) : "r"(a));
    asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];" : "=r"(z[0]), "=r"(z[1]), "=r"(z[2]), "=r"(z[3]) : "r"(b));
    uint32_t ya[4], yb[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float x0 = bf16lo_to_f32(x[i]), x1 = bf16hi_to_f32(x[i]);
        const float z0 = bf16lo_to_f32(z[i]), z1 = bf16hi_to_f32(z[i]);
        ya[i] = pack_bf16x2(x0 * c[2 * i] - z0 * s[2 * i], x1 * c[2 * i + 1] - z1 * s[2 * i + 1]);
        yb[i] = pack_bf16x2(z0 * c[2 * i] + x0 * s[2 * i], z1 * c[2 * i + 1] + x1 * s[2 * i + 1]);
    }
    asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" :: "r"(a), "r"(ya[0]), "r"(ya[1]), "r"(ya[2]), "r"(ya[3]) : "memory");
    asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" :: "r"(b), "r"(yb[0]), "r"(yb[1]), "r"(yb[2]), "r"(yb[3]) : "memory");
}

// cos and sin of 2 pi * pos * (hi + lo) turns, for |pos| < 2^13: pos * hi is
// exact (hi has at most 11 significant bits), its integer part is removed
// exactly (round to nearest by adding and subtracting 1.5 * 2^23), the small
// pos * lo is added, and the reduced angle in [-pi, pi] goes to the fast
// sine and cosine (additive range reduction in the manner of Cody and Waite).
__device__ __forceinline__ void angle_cos_sin(float pos, float hi, float lo, float &c, float &s)
{
    const float t = pos * hi;
    const float n = (t + 12582912.0f) - 12582912.0f;
    const float f = fmaf(pos, lo, t - n);
    const float phi = f * 6.283185307179586f;
    __sincosf(phi, &s, &c);
}

// Find this CTA's (sequence, block) from cu_seqlens with one warp, and check
// the whole array.  Returns false (and sets *err on CTA 0) if the array is
// invalid, or if the block index is past the last block.
__device__ bool find_block(const int32_t *__restrict__ cu, int n_seqs, long long T, int max_seqlen,
                           int g, int32_t *err, int &seq, int &qb)
{
    const int lane = threadIdx.x & 31;
    int bad = 0;
    int base = 0;         // blocks before the current chunk of sequences
    int found_seq = -1, found_qb = 0;
    if (lane == 0 && (cu[0] != 0 || static_cast<long long>(cu[n_seqs]) != T))
        bad |= kErrBadCu;
    for (int s0 = 0; s0 < n_seqs; s0 += 32) {
        const int s = s0 + lane;
        int nb = 0;
        if (s < n_seqs) {
            const int L = cu[s + 1] - cu[s];
            if (L < 0)
                bad |= kErrBadCu;
            else if (L > max_seqlen)
                bad |= kErrTooLong;
            else
                nb = (L + kBlockM - 1) / kBlockM;
        }
        int incl = nb;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, incl, d);
            if (lane >= d)
                incl += v;
        }
        const int excl = base + incl - nb;
        if (found_seq < 0) {
            const unsigned hit = __ballot_sync(0xffffffffu, nb > 0 && g >= excl && g < excl + nb);
            if (hit) {
                const int src = __ffs(hit) - 1;
                found_seq = s0 + src;
                found_qb = g - __shfl_sync(0xffffffffu, excl, src);
            }
        }
        base += __shfl_sync(0xffffffffu, incl, 31);
    }
#pragma unroll
    for (int d = 16; d > 0; d >>= 1)
        bad |= __shfl_xor_sync(0xffffffffu, bad, d);
    if (bad) {
        if (blockIdx.x == 0 && lane == 0)
            atomicOr(err, bad);
        return false;
    }
    seq = found_seq;
    qb = found_qb;
    return found_seq >= 0;
}

__global__ void __launch_bounds__(kThreads, 2)
attn_local_kernel(const __grid_constant__ CUtensorMap tm_qkv, const __grid_constant__ RopeConsts rope,
                  const int32_t *__restrict__ cu, int n_seqs, long long T, int max_seqlen,
                  const int2 *__restrict__ work, const int32_t *__restrict__ work_count, int hw,
                  __nv_bfloat16 *__restrict__ out, int32_t *err)
{
    extern __shared__ uint8_t smem_raw[];
    __shared__ int s_unit[2];
    __shared__ uint32_t s_tmem;
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    const int g = blockIdx.x / kHeads;
    const int head = blockIdx.x % kHeads;
    if (work) {
        if (g >= *work_count)
            return;
        if (tid == 0) {
            const int2 e = work[g];
            s_unit[0] = e.x;
            s_unit[1] = e.y;
        }
    } else if (warp == 0) {
        int seq = -1, qb = 0;
        if (!find_block(cu, n_seqs, T, max_seqlen, g, err, seq, qb))
            seq = -1;
        if (lane == 0) {
            s_unit[0] = seq;
            s_unit[1] = qb;
        }
    }
    if (warp == 0) {
        tmem_alloc(smem_u32(&s_tmem), kTmemCols);
        tmem_relinquish();
    }
    if (tid == 0) {
        tma_prefetch_desc(&tm_qkv);
        for (int i = 0; i < 6; ++i)
            mbar_init(barp(base, i), i == kBarRope || i == kBarP ? kCompute : 1);
        fence_mbar_init();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = s_tmem;
    const int seq = s_unit[0];
    if (seq >= 0) {
        const int row0 = cu[seq];
        const int L = cu[seq + 1] - row0;
        const int q0 = s_unit[1] * kBlockM;

        if (warp == 4) {
            // ------------------------------------------------ issuer warp
            const uint64_t once = l2_policy_evict_first();
            const uint64_t keep = l2_policy_evict_last();    // K/V rows: re-read by the neighbour block
            const int colQ = head * kHeadDim, colK = kHidden + colQ, colV = 2 * kHidden + colQ;
            if (elect_one_sync()) {
                mbar_arrive_expect_tx(barp(base, kBarQK), 3 * kTileBytes);
                tma_load_2d_hint(base + kOffQ, &tm_qkv, colQ, row0 + q0, barp(base, kBarQK), once);
                tma_load_2d_hint(base + kOffK, &tm_qkv, colK, row0 + q0 - 64, barp(base, kBarQK), keep);
                tma_load_2d_hint(base + kOffK + kTileBytes, &tm_qkv, colK, row0 + q0 + 64, barp(base, kBarQK), keep);
                mbar_arrive_expect_tx(barp(base, kBarV), 2 * kTileBytes);
                tma_load_2d_hint(base + kOffV, &tm_qkv, colV, row0 + q0 - 64, barp(base, kBarV), keep);
                tma_load_2d_hint(base + kOffV + kTileBytes, &tm_qkv, colV, row0 + q0 + 64, barp(base, kBarV), keep);
            }
            __syncwarp();
            // S0 = Q K0^T; once softmax has turned S0 into P0, S1 = Q K1^T
            // (into the same columns) and then O = P0 V0, so that the second
            // softmax starts as early as possible; O += P1 V1 last.
            auto issue_s = [&](int t) {
                const uint32_t q = base + kOffQ, k = base + kOffK + t * kTileBytes;
#pragma unroll
                for (int kk = 0; kk < kHeadDim / 16; ++kk)
                    mma_bf16_ss_warp(tmem + kColS, make_sdesc_sw128(q + 32 * kk, 16, 1024),
                                     make_sdesc_sw128(k + 32 * kk, 16, 1024), kIdescS, kk > 0);
                mma_commit_warp(barp(base, kBarS));
            };
            auto issue_o = [&](int t) {
                const uint32_t v = base + kOffV + t * kTileBytes;
#pragma unroll
                for (int kk = 0; kk < kBlockN / 16; ++kk)
                    mma_bf16_ts_warp(tmem + kColO, tmem + kColP + 8 * kk,
                                     make_sdesc_sw128(v + 2048 * kk, 1024, 1024), kIdescO,
                                     (t > 0 || kk > 0) ? 1u : 0u);
                mma_commit_warp(barp(base, kBarO));
            };
            if (mbar_wait(barp(base, kBarRope), 0, err)) {
                __syncwarp();
                tc_fence_after();
                issue_s(0);
                if (mbar_wait(barp(base, kBarP), 0, err)) {
                    __syncwarp();
                    tc_fence_after();
                    issue_s(1);
                    if (mbar_wait(barp(base, kBarV), 0, err)) {
                        __syncwarp();
                        issue_o(0);
                        if (mbar_wait(barp(base, kBarP), 1, err)) {
                            __syncwarp();
                            tc_fence_after();
                            issue_o(1);
                        }
                    }
                }
            }
            __syncwarp();
        } else {
            // ------------------------------------------------ compute warps
            const int r = tid;                 // row in the block, TMEM lane
            const int i = q0 + r;              // query position in the sequence
            const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
            // RoPE: position q0 - 64 + r is K row r of tile 0 (and Q row
            // r - 64), position q0 + 64 + r is K row r of tile 1 (and Q row
            // r + 64).  cos/sin are computed here (no table): for the first
            // position from the split frequencies, for the second by one
            // more rotation of 128 positions.
            bool ok = mbar_wait(barp(base, kBarQK), 0, err);
            if (ok) {
                const float pos0 = static_cast<float>(q0 - 64 + r);
                const int qr0 = r - 64, qr1 = r + 64;
#pragma unroll 1
                for (int j = 0; j < 4; ++j) {
                    float c0[8], s0[8], c1[8], s1[8];
#pragma unroll
                    for (int k = 0; k < 8; ++k) {
                        const int mm = 8 * j + k;
                        angle_cos_sin(pos0, rope.turns_hi[mm], rope.turns_lo[mm], c0[k], s0[k]);
                        c1[k] = c0[k] * rope.cos128[mm] - s0[k] * rope.sin128[mm];
                        s1[k] = s0[k] * rope.cos128[mm] + c0[k] * rope.sin128[mm];
                    }
                    rope_chunk(base + kOffK + r * 128, r, j, c0, s0);
                    if (qr0 >= 0)
                        rope_chunk(base + kOffQ + qr0 * 128, qr0, j, c0, s0);
                    rope_chunk(base + kOffK + kTileBytes + r * 128, r, j, c1, s1);
                    if (qr1 < kBlockM)
                        rope_chunk(base + kOffQ + qr1 * 128, qr1, j, c1, s1);
                }
                fence_proxy_async_smem();
            }
            mbar_arrive(barp(base, kBarRope));

            // admitted keys of this row: positions [klo, khi]
            const int klo = max(0, i - hw), khi = min(L - 1, i + hw);
            float m = -INFINITY, l = 0.f;
            for (int t = 0; t < 2 && ok; ++t) {
                if (!(ok = mbar_wait(barp(base, kBarS), t, err)))
                    break;
                __syncwarp();
                tc_fence_after();
                const int c0 = band_chunk_begin(t, warp), c1 = band_chunk_end(t, warp);
                const int key0 = band_tile_key0(q0, t);
                // pass 1: row maximum over the visited chunks
                float mx = -INFINITY;
#pragma unroll 1
                for (int c = c0; c < c1; ++c) {
                    uint32_t v[32];
                    tmem_ld32(tmem + kColS + lane_off + 32 * c, v);
                    tmem_wait_ld();
                    const bool masked = band_chunk_needs_mask(q0, L, hw, t, warp, c);
                    const int lo = klo - key0 - 32 * c, hi = khi - key0 - 32 * c;
                    float mp[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
                    for (int k = 0; k < 32; ++k) {
                        float x = __uint_as_float(v[k]);
                        if (masked && (k < lo || k > hi))
                            x = -INFINITY;
                        mp[k & 3] = fmaxf(mp[k & 3], x);
                    }
                    mx = fmaxf(mx, fmaxf(fmaxf(mp[0], mp[1]), fmaxf(mp[2], mp[3])));
                }
                const float mc = mx * kScaleLog2;
                const bool need = mc > m + kRescaleThreshold;
                const float mn = need ? mc : m;
                const float m_use = mn == -INFINITY ? 0.f : mn;
                const float alpha = need ? ex2_approx(m - m_use) : 1.f;
                if (t > 0) {
                    // P and O are free once P0 V0 has completed
                    if (!(ok = mbar_wait(barp(base, kBarO), 0, err)))
                        break;
                    __syncwarp();
                    tc_fence_after();
                    if (__any_sync(0xffffffffu, need)) {
#pragma unroll 1
                        for (int h = 0; h < 2; ++h) {
                            uint32_t o[32];
                            tmem_ld32(tmem + kColO + lane_off + 32 * h, o);
                            tmem_wait_ld();
#pragma unroll
                            for (int k = 0; k < 32; ++k)
                                o[k] = __float_as_uint(__uint_as_float(o[k]) * alpha);
                            tmem_st32(tmem + kColO + lane_off + 32 * h, o);
                        }
                    }
                }
                // pass 2: p = 2^(s * scale - m) -> bf16 P, chunk by chunk;
                // chunks the warp does not visit get P = 0
                float sum = 0.f;
#pragma unroll 1
                for (int c = 0; c < 4; ++c) {
                    uint32_t pk[16];
                    if (c >= c0 && c < c1) {
                        uint32_t v[32];
                        tmem_ld32(tmem + kColS + lane_off + 32 * c, v);
                        tmem_wait_ld();
                        const bool masked = band_chunk_needs_mask(q0, L, hw, t, warp, c);
                        const int lo = klo - key0 - 32 * c, hi = khi - key0 - 32 * c;
                        float a0 = 0.f, a1 = 0.f;
#pragma unroll
                        for (int k = 0; k < 16; ++k) {
                            float x0 = fmaf(__uint_as_float(v[2 * k]), kScaleLog2, -m_use);
                            float x1 = fmaf(__uint_as_float(v[2 * k + 1]), kScaleLog2, -m_use);
                            if (masked && (2 * k < lo || 2 * k > hi))
                                x0 = -INFINITY;
                            if (masked && (2 * k + 1 < lo || 2 * k + 1 > hi))
                                x1 = -INFINITY;
                            const float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
                            a0 += p0;
                            a1 += p1;
                            pk[k] = pack_bf16x2(p0, p1);
                        }
                        sum += a0 + a1;
                    } else {
#pragma unroll
                        for (int k = 0; k < 16; ++k)
                            pk[k] = 0u;
                    }
                    tmem_st16(tmem + kColP + lane_off + 16 * c, pk);
                }
                l = l * alpha + sum;
                m = mn;
                tmem_wait_st();
                tc_fence_before();
                mbar_arrive(barp(base, kBarP));
            }
            if (ok && mbar_wait(barp(base, kBarO), 1, err)) {
                __syncwarp();
                tc_fence_after();
                const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll 1
                for (int h = 0; h < 2; ++h) {
                    uint32_t o[32];
                    tmem_ld32(tmem + kColO + lane_off + 32 * h, o);
                    tmem_wait_ld();
                    if (i < L) {
                        uint4 *dst = reinterpret_cast<uint4 *>(out + static_cast<long long>(row0 + i) * kHidden
                                                               + head * kHeadDim + 32 * h);
#pragma unroll
                        for (int k = 0; k < 4; ++k)
                            dst[k] = make_uint4(
                                pack_bf16x2(__uint_as_float(o[8 * k]) * inv, __uint_as_float(o[8 * k + 1]) * inv),
                                pack_bf16x2(__uint_as_float(o[8 * k + 2]) * inv, __uint_as_float(o[8 * k + 3]) * inv),
                                pack_bf16x2(__uint_as_float(o[8 * k + 4]) * inv, __uint_as_float(o[8 * k + 5]) * inv),
                                pack_bf16x2(__uint_as_float(o[8 * k + 6]) * inv, __uint_as_float(o[8 * k + 7]) * inv));
                    }
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

}  // namespace

cudaError_t launch_attn_local(const LocalArgs &a, cudaStream_t stream)
{
    static bool configured[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 0 && dev < 64 && !configured[dev]) {
        cudaError_t e = cudaFuncSetAttribute(attn_local_kernel,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(kSmemBytes));
        if (e != cudaSuccess)
            return e;
        configured[dev] = true;
    }
    const long long grid = static_cast<long long>(a.block_bound) * kHeads;
    attn_local_kernel<<<static_cast<unsigned>(grid), kThreads, kSmemBytes, stream>>>(
        a.tm_qkv, a.rope, a.cu, a.n_seqs, a.T, a.max_seqlen, a.work, a.work_count,
        a.half_window, a.out, a.err);
    return cudaGetLastError();
}

}  // namespace mbert
