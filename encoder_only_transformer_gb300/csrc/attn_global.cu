// Global-layer attention over pre-rotated Q/K: a warp-specialised tcgen05
// pipeline for sm_103a.
//
// One CTA (12 warps) per (work entry, head); an entry is 256 query rows of
// one sequence, split into two 128-row tiles that share every K/V tile:
//   warps 0-3  softmax group 0 (query tile 0, TMEM lanes 0..127)
//   warps 4-7  softmax group 1 (query tile 1)
//   warp  8    TMA producer: Q0, Q1 once, then K and V through 3-stage rings
//   warp  9    MMA issuer (the whole warp runs the loop; one elected lane
//              issues): S_w = Q_w K_j^T and O_w += P_w V_j
//   warps 10-11 idle (they complete the third warpgroup, whose registers
//              go to the softmax groups)
// TMEM (512 columns): S0 [0,128) S1 [128,256) P0 [256,320) P1 [320,384)
// O0 [384,448) O1 [448,512), all fp32 except P (bf16 pairs).  The issue
// order S0(j+1), S1(j+1), PV0(j), PV1(j) keeps the tensor core fed while
// each softmax group works on its previous tile.
//
// Arithmetic ("ModernBERT-base Architecture Teardown", "How Does
// Self-Attention Work?"): scores q.k / 8, softmax over every key of the
// sequence (a global layer, "What Are Local and Global Attention?"), output
// the weighted blend of V.  The softmax is online in base 2; the running
// maximum is only raised (and O rescaled) when a tile's maximum exceeds it
// by more than 8, so the unnormalised weights stay below 2^8 and O and the
// row sum always use the same reference.
#include "common.cuh"
#include "internal.h"

namespace mbert {
namespace {

constexpr int kThreads = 384;      // 3 warpgroups
// Registers per thread after the split: the producer/MMA warpgroup gives up
// registers to the two softmax warpgroups (4 x 88 + 8 x 208 = 12 x 168, the
// launch budget).
constexpr int kRegsSoftmax = 208;
constexpr int kRegsControl = 88;
constexpr int kStages = 3;
constexpr uint32_t kOffQ = 0;                                  // Q0, Q1
constexpr uint32_t kOffK = 2 * kTileBytes;                     // K ring
constexpr uint32_t kOffV = kOffK + kStages * kTileBytes;       // V ring
constexpr uint32_t kOffBar = kOffV + kStages * kTileBytes;     // 131072
constexpr uint32_t kSmemBytes = kOffBar + 256 + 1024;

// barrier slots (8 bytes each) from kOffBar
constexpr int kBarQ = 0;
constexpr int kBarKFull = 1;      // + stage
constexpr int kBarKEmpty = 4;     // + stage
constexpr int kBarVFull = 7;      // + stage
constexpr int kBarVEmpty = 10;    // + stage
constexpr int kBarSFull = 13;     // + group
constexpr int kBarSEmpty = 15;    // + group
constexpr int kBarPFull = 17;     // + group
constexpr int kBarODone = 19;     // + group
constexpr int kNumBars = 21;
constexpr uint32_t kOffSlot = kOffBar + 8 * kNumBars;

constexpr uint32_t kTmemCols = 512;
__host__ __device__ constexpr uint32_t col_s(int w) { return 128u * w; }
__host__ __device__ constexpr uint32_t col_p(int w) { return 256u + 64u * w; }
__host__ __device__ constexpr uint32_t col_o(int w) { return 384u + 64u * w; }

constexpr uint32_t kIdescS = make_idesc_bf16(128, 128, false);
constexpr uint32_t kIdescO = make_idesc_bf16(128, 64, true);
constexpr float kScaleLog2 = 0.125f * 1.4426950408889634f;
constexpr float kRescaleThreshold = 8.0f;

__device__ __forceinline__ float fmax3(float a, float b, float c)
{
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

// (a0, a1) * (b, b) + (c, c) on the packed fp32x2 path
__device__ __forceinline__ void ffma2_bc(float &x0, float &x1, float b, float c)
{
    uint64_t a, bb, cc, d;
    asm("mov.b64 %0, {%1, %2};" : "=l"(a) : "f"(x0), "f"(x1));
    asm("mov.b64 %0, {%1, %1};" : "=l"(bb) : "f"(b));
    asm("mov.b64 %0, {%1, %1};" : "=l"(cc) : "f"(c));
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(bb), "l"(cc));
    asm("mov.b64 {%0, %1}, %2;" : "=f"(x0), "=f"(x1) : "l"(d));
}

__device__ __forceinline__ void fadd2(float &a0, float &a1, float b0, float b1)
{
    uint64_t a, b, d;
    asm("mov.b64 %0, {%1, %2};" : "=l"(a) : "f"(a0), "f"(a1));
    asm("mov.b64 %0, {%1, %2};" : "=l"(b) : "f"(b0), "f"(b1));
    asm("add.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    asm("mov.b64 {%0, %1}, %2;" : "=f"(a0), "=f"(a1) : "l"(d));
}

struct Ctx {
    uint32_t base;          // 1024-aligned shared address
    uint32_t tmem;
    int row0, L, q0, head, ntiles;
};

__device__ __forceinline__ uint32_t bar(const Ctx &c, int i) { return c.base + kOffBar + 8u * i; }

// ---------------------------------------------------------------- producer
__device__ void producer(const Ctx &c, const CUtensorMap *tm_rot, const CUtensorMap *tm_qkv,
                         int *err)
{
    const uint64_t keep = l2_policy_evict_last();    // K/V: re-read by every query block
    const uint64_t once = l2_policy_evict_first();   // Q: read once
    const int colQ = c.head * kHeadDim;
    const int colK = kHidden + c.head * kHeadDim;
    const int colV = 2 * kHidden + c.head * kHeadDim;
    mbar_arrive_expect_tx(bar(c, kBarQ), 2 * kTileBytes);
    tma_load_2d_hint(c.base + kOffQ, tm_rot, colQ, c.row0 + c.q0, bar(c, kBarQ), once);
    tma_load_2d_hint(c.base + kOffQ + kTileBytes, tm_rot, colQ, c.row0 + c.q0 + kBlockM,
                     bar(c, kBarQ), once);
    for (int j = 0; j < c.ntiles; ++j) {
        const int s = j % kStages;
        const uint32_t u = j / kStages;
        const int krow = c.row0 + j * kBlockN;
        if (u > 0 && !mbar_wait(bar(c, kBarKEmpty + s), (u - 1) & 1, err))
            return;
        mbar_arrive_expect_tx(bar(c, kBarKFull + s), kTileBytes);
        tma_load_2d_hint(c.base + kOffK + s * kTileBytes, tm_rot, colK, krow, bar(c, kBarKFull + s), keep);
        if (u > 0 && !mbar_wait(bar(c, kBarVEmpty + s), (u - 1) & 1, err))
            return;
        mbar_arrive_expect_tx(bar(c, kBarVFull + s), kTileBytes);
        tma_load_2d_hint(c.base + kOffV + s * kTileBytes, tm_qkv, colV, krow, bar(c, kBarVFull + s), keep);
    }
}

// ---------------------------------------------------------------- MMA issuer
// The MMA issuer runs on the whole (converged) warp 9: descriptors are
// computed by every lane, and the *_warp wrappers let one elected lane issue.
__device__ __forceinline__ void issue_s(const Ctx &c, int w, int s)
{
    const uint32_t q = c.base + kOffQ + w * kTileBytes;
    const uint32_t k = c.base + kOffK + s * kTileBytes;
#pragma unroll
    for (int kk = 0; kk < kHeadDim / 16; ++kk)
        mma_bf16_ss_warp(c.tmem + col_s(w), make_sdesc_sw128(q + 32 * kk, 16, 1024),
                         make_sdesc_sw128(k + 32 * kk, 16, 1024), kIdescS, kk > 0);
}

__device__ __forceinline__ void issue_o(const Ctx &c, int w, int s, bool accumulate)
{
    const uint32_t v = c.base + kOffV + s * kTileBytes;
#pragma unroll
    for (int kk = 0; kk < kBlockN / 16; ++kk)
        mma_bf16_ts_warp(c.tmem + col_o(w), c.tmem + col_p(w) + 8 * kk,
                         make_sdesc_sw128(v + 2048 * kk, 1024, 1024), kIdescO,
                         (accumulate || kk > 0) ? 1u : 0u);
}

__device__ void mma_issuer(const Ctx &c, int *err)
{
    if (!mbar_wait(bar(c, kBarQ), 0, err) || !mbar_wait(bar(c, kBarKFull), 0, err))
        return;
    __syncwarp();
    tc_fence_after();
    issue_s(c, 0, 0);
    mma_commit_warp(bar(c, kBarSFull + 0));
    issue_s(c, 1, 0);
    mma_commit_warp(bar(c, kBarSFull + 1));
    mma_commit_warp(bar(c, kBarKEmpty + 0));
    for (int j = 0; j < c.ntiles; ++j) {
        const uint32_t ph = j & 1;
        if (j + 1 < c.ntiles) {
            const int s1 = (j + 1) % kStages;
            const uint32_t u1 = (j + 1) / kStages;
            if (!mbar_wait(bar(c, kBarKFull + s1), u1 & 1, err))
                return;
            if (!mbar_wait(bar(c, kBarSEmpty + 0), ph, err))
                return;
            __syncwarp();
            tc_fence_after();
            issue_s(c, 0, s1);
            mma_commit_warp(bar(c, kBarSFull + 0));
            if (!mbar_wait(bar(c, kBarSEmpty + 1), ph, err))
                return;
            __syncwarp();
            tc_fence_after();
            issue_s(c, 1, s1);
            mma_commit_warp(bar(c, kBarSFull + 1));
            mma_commit_warp(bar(c, kBarKEmpty + s1));
        }
        const int s = j % kStages;
        const uint32_t u = j / kStages;
        if (!mbar_wait(bar(c, kBarVFull + s), u & 1, err))
            return;
        if (!mbar_wait(bar(c, kBarPFull + 0), ph, err))
            return;
        __syncwarp();
        tc_fence_after();
        issue_o(c, 0, s, j > 0);
        mma_commit_warp(bar(c, kBarODone + 0));
        if (!mbar_wait(bar(c, kBarPFull + 1), ph, err))
            return;
        __syncwarp();
        tc_fence_after();
        issue_o(c, 1, s, j > 0);
        mma_commit_warp(bar(c, kBarODone + 1));
        mma_commit_warp(bar(c, kBarVEmpty + s));
    }
}

// ---------------------------------------------------------------- softmax
__device__ void softmax_group(const Ctx &c, int w, int warp_in_group, int lane,
                              __nv_bfloat16 *__restrict__ out, int *err)
{
    const uint32_t lane_off = static_cast<uint32_t>(32 * warp_in_group) << 16;
    const uint32_t tS = c.tmem + col_s(w) + lane_off;
    const uint32_t tP = c.tmem + col_p(w) + lane_off;
    const uint32_t tO = c.tmem + col_o(w) + lane_off;
    const int qpos = c.q0 + kBlockM * w + 32 * warp_in_group + lane;
    float m = -INFINITY;    // running reference maximum (scaled, base 2)
    float l = 0.f;          // running sum of exp2(score - m)
    bool ok = true;

    for (int j = 0; j < c.ntiles; ++j) {
        if (!(ok = mbar_wait(bar(c, kBarSFull + w), j & 1, err)))
            break;
        __syncwarp();
        tc_fence_after();
        float s[kBlockN];
        {
            uint32_t r0[32], r1[32], r2[32], r3[32];
            tmem_ld32(tS, r0);
            tmem_ld32(tS + 32, r1);
            tmem_ld32(tS + 64, r2);
            tmem_ld32(tS + 96, r3);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                s[i] = __uint_as_float(r0[i]);
                s[32 + i] = __uint_as_float(r1[i]);
                s[64 + i] = __uint_as_float(r2[i]);
                s[96 + i] = __uint_as_float(r3[i]);
            }
        }
        tc_fence_before();
        mbar_arrive(bar(c, kBarSEmpty + w));   // S may be overwritten now

        const int kvalid = c.L - j * kBlockN;   // keys of this tile inside the sequence
        if (kvalid < kBlockN) {
#pragma unroll
            for (int i = 0; i < kBlockN; ++i)
                if (i >= kvalid)
                    s[i] = -INFINITY;
        }
        // row maximum: 8 independent chains of 3-input max, then combine
        float mp[8];
#pragma unroll
        for (int k = 0; k < 8; ++k)
            mp[k] = fmax3(s[k], s[8 + k], s[16 + k]);
#pragma unroll
        for (int i = 24; i < kBlockN; i += 16)
#pragma unroll
            for (int k = 0; k < 8; ++k)
                mp[k] = fmax3(mp[k], s[i + k], s[i + 8 + k]);
        const float mx = fmaxf(fmax3(mp[0], mp[1], mp[2]),
                               fmaxf(fmax3(mp[3], mp[4], mp[5]), fmax3(mp[6], mp[7], mp[7])));
        const float mc = mx * kScaleLog2;
        const bool need = mc > m + kRescaleThreshold;
        const float mn = need ? mc : m;
        const float alpha = need ? ex2_approx(m - mn) : 1.f;
        const float neg = -mn;

        // p = 2^(s * scale - m), packed to bf16 pairs; row sum in 4
        // independent fp32x2 accumulators
        uint32_t pk[kBlockN / 2];
        float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int i = 0; i < kBlockN / 2; ++i) {
            float x0 = s[2 * i], x1 = s[2 * i + 1];
            ffma2_bc(x0, x1, kScaleLog2, neg);
            const float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
            const int a = 2 * (i & 3);
            fadd2(acc[a], acc[a + 1], p0, p1);
            pk[i] = pack_bf16x2(p0, p1);
        }
        fadd2(acc[0], acc[1], acc[2], acc[3]);
        fadd2(acc[4], acc[5], acc[6], acc[7]);
        fadd2(acc[0], acc[1], acc[4], acc[5]);
        const float a0 = acc[0], a1 = acc[1];

        if (j > 0) {
            // P_w and O_w are free once the previous P V has completed
            if (!(ok = mbar_wait(bar(c, kBarODone + w), (j - 1) & 1, err)))
                break;
            __syncwarp();
            tc_fence_after();
            if (__any_sync(0xffffffffu, need)) {
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    uint32_t o[32];
                    tmem_ld32(tO + 32 * h, o);
                    tmem_wait_ld();
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
                    tmem_st32(tO + 32 * h, o);
                }
            }
        }
        l = l * alpha + (a0 + a1);
        m = mn;
        tmem_st64(tP, pk);
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(bar(c, kBarPFull + w));
    }
    if (!ok || !mbar_wait(bar(c, kBarODone + w), (c.ntiles - 1) & 1, err))
        return;
    __syncwarp();
    tc_fence_after();
    const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        uint32_t o[32];
        tmem_ld32(tO + 32 * h, o);
        tmem_wait_ld();
        uint32_t wv[16];
#pragma unroll
        for (int i = 0; i < 16; ++i)
            wv[i] = pack_bf16x2(__uint_as_float(o[2 * i]) * inv, __uint_as_float(o[2 * i + 1]) * inv);
        if (qpos < c.L) {
            uint4 *dst = reinterpret_cast<uint4 *>(out + static_cast<long long>(c.row0 + qpos) * kHidden
                                                   + c.head * kHeadDim + 32 * h);
#pragma unroll
            for (int i = 0; i < 4; ++i)
                dst[i] = make_uint4(wv[4 * i], wv[4 * i + 1], wv[4 * i + 2], wv[4 * i + 3]);
        }
    }
}

__global__ void __launch_bounds__(kThreads, 1)
attn_global_kernel(const __grid_constant__ CUtensorMap tm_rot,
                   const __grid_constant__ CUtensorMap tm_qkv,
                   const int32_t *__restrict__ cu, const int2 *__restrict__ work,
                   const int32_t *__restrict__ work_count, __nv_bfloat16 *__restrict__ out,
                   int32_t *err)
{
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    Ctx c;
    c.base = (raw + 1023u) & ~1023u;
    uint32_t *slot = reinterpret_cast<uint32_t *>(smem_raw + (c.base - raw) + kOffSlot);

    const int entry = blockIdx.x / kHeads;
    c.head = blockIdx.x % kHeads;
    if (entry >= *work_count)
        return;
    const int2 e = work[entry];
    c.row0 = cu[e.x];
    c.L = cu[e.x + 1] - c.row0;
    c.q0 = e.y * 2 * kBlockM;
    c.ntiles = (c.L + kBlockN - 1) / kBlockN;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        tma_prefetch_desc(&tm_rot);
        tma_prefetch_desc(&tm_qkv);
        mbar_init(bar(c, kBarQ), 1);
        for (int s = 0; s < kStages; ++s) {
            mbar_init(bar(c, kBarKFull + s), 1);
            mbar_init(bar(c, kBarKEmpty + s), 1);
            mbar_init(bar(c, kBarVFull + s), 1);
            mbar_init(bar(c, kBarVEmpty + s), 1);
        }
        for (int w = 0; w < 2; ++w) {
            mbar_init(bar(c, kBarSFull + w), 1);
            mbar_init(bar(c, kBarSEmpty + w), kBlockM);
            mbar_init(bar(c, kBarPFull + w), kBlockM);
            mbar_init(bar(c, kBarODone + w), 1);
        }
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(smem_u32(slot), kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    c.tmem = *slot;

    if (warp >= 8) {
        asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" :: "n"(kRegsControl));
        if (warp == 8) {
            if (lane == 0)
                producer(c, &tm_rot, &tm_qkv, err);
            __syncwarp();
        } else if (warp == 9) {
            mma_issuer(c, err);
            __syncwarp();
        }
    } else {
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" :: "n"(kRegsSoftmax));
        softmax_group(c, warp >> 2, warp & 3, lane, out, err);
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(c.tmem, kTmemCols);
    }
}

}  // namespace

cudaError_t launch_attn_global(const AttnArgs &a, cudaStream_t stream)
{
    static bool configured[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 0 && dev < 64 && !configured[dev]) {
        cudaError_t e = cudaFuncSetAttribute(attn_global_kernel,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(kSmemBytes));
        if (e != cudaSuccess)
            return e;
        configured[dev] = true;
    }
    const long long grid = static_cast<long long>(a.entry_bound) * kHeads;
    attn_global_kernel<<<static_cast<unsigned>(grid), kThreads, kSmemBytes, stream>>>(
        a.tm_rot, a.tm_qkv, a.cu, a.work, a.work_count, a.out, a.err);
    return cudaGetLastError();
}

}  // namespace mbert
