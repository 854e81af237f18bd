// Generic flash attention over pre-rotated Q/K (tcgen05 + TMA, sm_103a).
//
// One CTA of 128 threads per (work entry, head): a block of 128 query rows
// of one sequence against every key tile the schedule admits.  Thread r
// owns query row r (TMEM lane r).  Thread 0 issues the TMA loads and the
// MMAs; the whole CTA runs the softmax.
//
//   S = Q K^T          tcgen05.mma M=128 N=128 K=16 x4, fp32 in TMEM cols [0,128)
//   online softmax     fp32 row max / sum in registers, P -> bf16 in smem
//   O = a*O + P V      tcgen05.mma M=128 N=64 K=16 x8, fp32 in TMEM cols [128,192)
//
// Scores are q.k / 8, softmax along the keys, output the blend of V
// ("ModernBERT-base Architecture Teardown", "How Does Self-Attention
// Work?"); keys outside the sequence or, on local layers, further than
// half_window away are masked ("What Are Local and Global Attention?").
#include "common.cuh"
#include "internal.h"

namespace mbert {
namespace {

constexpr int kThreads = 128;
constexpr uint32_t kOffQ = 0;
constexpr uint32_t kOffK = 16384;          // 2 stages of 16 KB
constexpr uint32_t kOffV = 49152;          // 2 stages of 16 KB
constexpr uint32_t kOffP = 81920;          // 128 x 128 bf16 = 2 column blocks of 16 KB
constexpr uint32_t kOffBar = 114688;
constexpr uint32_t kSmemBytes = kOffBar + 128 + 1024;   // + 1024 for base alignment
constexpr uint32_t kTmemCols = 256;
constexpr uint32_t kColS = 0;
constexpr uint32_t kColO = 128;

constexpr uint32_t kIdescS = make_idesc_bf16(128, 128, false);   // Q (K-major) x K (K-major)
constexpr uint32_t kIdescO = make_idesc_bf16(128, 64, true);     // P (K-major) x V (MN-major)

// log2(e) / sqrt(64): softmax in base 2
constexpr float kScaleLog2 = 0.125f * 1.4426950408889634f;

__global__ void __launch_bounds__(kThreads, 1)
attn_generic_kernel(const __grid_constant__ CUtensorMap tm_rot,
                    const __grid_constant__ CUtensorMap tm_qkv,
                    const int32_t *__restrict__ cu, const int2 *__restrict__ work,
                    const int32_t *__restrict__ work_count, int hw,
                    __nv_bfloat16 *__restrict__ out, int32_t *err)
{
    pdl_wait();
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *sbase = smem_raw + (base - raw);

    const int entry = blockIdx.x / kHeads;
    const int head = blockIdx.x % kHeads;
    if (entry >= *work_count)
        return;
    const int2 e = work[entry];
    const int row0 = cu[e.x];
    const int L = cu[e.x + 1] - row0;
    const int q0 = e.y * kBlockM;
    int kt0, kt1;
    key_tile_range(q0, L, hw, kt0, kt1);
    const int ntiles = kt1 - kt0;

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const uint32_t sQ = base + kOffQ;
    const uint32_t sP = base + kOffP;
    const uint32_t bar_q = base + kOffBar;
    const uint32_t bar_kv0 = bar_q + 8;      // + 8 * stage
    const uint32_t bar_s = bar_q + 24;
    const uint32_t bar_o = bar_q + 32;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sbase + kOffBar + 64);

    if (tid == 0) {
        tma_prefetch_desc(&tm_rot);
        tma_prefetch_desc(&tm_qkv);
        mbar_init(bar_q, 1);
        mbar_init(bar_kv0, 1);
        mbar_init(bar_kv0 + 8, 1);
        mbar_init(bar_s, 1);
        mbar_init(bar_o, 1);
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(smem_u32(tmem_slot), kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t tS = tmem + kColS;
    const uint32_t tO = tmem + kColO;
    const uint32_t lane = static_cast<uint32_t>(warp * 32) << 16;   // this warp's TMEM lanes

    const int colQ = head * kHeadDim;
    const int colK = kHidden + head * kHeadDim;
    const int colV = 2 * kHidden + head * kHeadDim;
    if (tid == 0) {
        mbar_arrive_expect_tx(bar_q, kTileBytes);
        tma_load_2d(sQ, &tm_rot, colQ, row0 + q0, bar_q);
        for (int st = 0; st < 2 && st < ntiles; ++st) {
            const int krow = row0 + (kt0 + st) * kBlockN;
            mbar_arrive_expect_tx(bar_kv0 + 8 * st, 2 * kTileBytes);
            tma_load_2d(base + kOffK + st * kTileBytes, &tm_rot, colK, krow, bar_kv0 + 8 * st);
            tma_load_2d(base + kOffV + st * kTileBytes, &tm_qkv, colV, krow, bar_kv0 + 8 * st);
        }
    }

    const int qpos = q0 + tid;
    float m_run = -INFINITY;   // running max of the scaled scores (base-2 units)
    float l_run = 0.f;         // running sum of exp2(score - m_run)
    bool ok = mbar_wait(bar_q, 0, err);

    for (int t = 0; t < ntiles && ok; ++t) {
        const int st = t & 1;
        const uint32_t bar_kv = bar_kv0 + 8 * st;
        if (!(ok = mbar_wait(bar_kv, (t >> 1) & 1, err)))
            break;
        if (tid == 0) {
            tc_fence_after();
            const uint32_t sK = base + kOffK + st * kTileBytes;
#pragma unroll
            for (int k = 0; k < kHeadDim / 16; ++k)
                mma_bf16_ss(tS, make_sdesc_sw128(sQ + 32 * k, 16, 1024),
                            make_sdesc_sw128(sK + 32 * k, 16, 1024), kIdescS, k > 0);
            mma_commit(bar_s);
        }
        if (!(ok = mbar_wait(bar_s, t & 1, err)))
            break;
        __syncwarp();
        tc_fence_after();

        float s[kBlockN];
#pragma unroll
        for (int c = 0; c < kBlockN / 32; ++c) {
            uint32_t r[32];
            tmem_ld32(tS + lane + 32 * c, r);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 32; ++i)
                s[32 * c + i] = __uint_as_float(r[i]);
        }
        const int kt = kt0 + t;
        if (tile_needs_mask(q0, L, hw, kt)) {
            const int kb = kt * kBlockN;
#pragma unroll
            for (int c = 0; c < kBlockN; ++c)
                if (!admitted(qpos, kb + c, L, hw))
                    s[c] = -INFINITY;
        }
        float mx = -INFINITY;
#pragma unroll
        for (int c = 0; c < kBlockN; ++c)
            mx = fmaxf(mx, s[c]);
        const float m_new = fmaxf(m_run, mx * kScaleLog2);
        const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
        const float alpha = ex2_approx(m_run - m_use);
        float sum = 0.f;
        uint32_t pk[kBlockN / 2];
#pragma unroll
        for (int c = 0; c < kBlockN / 2; ++c) {
            const float p0 = ex2_approx(fmaf(s[2 * c], kScaleLog2, -m_use));
            const float p1 = ex2_approx(fmaf(s[2 * c + 1], kScaleLog2, -m_use));
            sum += p0 + p1;
            pk[c] = pack_bf16x2(p0, p1);
        }
        l_run = l_run * alpha + sum;
        m_run = m_new;

        // P row -> shared memory, K-major with the 128-byte swizzle: keys
        // 0..63 in column block 0, 64..127 in block 1; 16-byte chunk j of
        // row r sits at chunk j ^ (r % 8) of its 128-byte line.
#pragma unroll
        for (int ch = 0; ch < kBlockN / 8; ++ch) {
            const uint32_t addr = sP + (ch >> 3) * 16384 + (tid >> 3) * 1024 + (tid & 7) * 128
                                  + (((ch & 7) ^ (tid & 7)) << 4);
            asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};"
                         :: "r"(addr), "r"(pk[4 * ch]), "r"(pk[4 * ch + 1]), "r"(pk[4 * ch + 2]),
                            "r"(pk[4 * ch + 3]) : "memory");
        }
        // O *= alpha (the previous P V has completed: bar_o was waited on)
        if (t > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll
            for (int h = 0; h < kHeadDim / 32; ++h) {
                uint32_t o[32];
                tmem_ld32(tO + lane + 32 * h, o);
                tmem_wait_ld();
#pragma unroll
                for (int i = 0; i < 32; ++i)
                    o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
                tmem_st32(tO + lane + 32 * h, o);
            }
            tmem_wait_st();
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();
        if (tid == 0) {
            tc_fence_after();
            const uint32_t sV = base + kOffV + st * kTileBytes;
#pragma unroll
            for (int k = 0; k < kBlockN / 16; ++k)
                mma_bf16_ss(tO, make_sdesc_sw128(sP + (k >> 2) * 16384 + (k & 3) * 32, 16, 1024),
                            make_sdesc_sw128(sV + k * 2048, 1024, 1024), kIdescO,
                            (t > 0 || k > 0) ? 1u : 0u);
            mma_commit(bar_o);
        }
        if (!(ok = mbar_wait(bar_o, t & 1, err)))
            break;
        tc_fence_after();
        // stage st is free again: fetch tile t + 2 into it
        if (tid == 0 && t + 2 < ntiles) {
            const int krow = row0 + (kt0 + t + 2) * kBlockN;
            mbar_arrive_expect_tx(bar_kv, 2 * kTileBytes);
            tma_load_2d(base + kOffK + st * kTileBytes, &tm_rot, colK, krow, bar_kv);
            tma_load_2d(base + kOffV + st * kTileBytes, &tm_qkv, colV, krow, bar_kv);
        }
    }

    if (ok) {
        // out[row, head*64 + d] = O / l, rounded to bf16; rows past the end
        // of the sequence are not written.
        const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
#pragma unroll
        for (int h = 0; h < kHeadDim / 32; ++h) {
            uint32_t o[32];
            tmem_ld32(tO + lane + 32 * h, o);
            tmem_wait_ld();
            uint32_t w[16];
#pragma unroll
            for (int i = 0; i < 16; ++i)
                w[i] = pack_bf16x2(__uint_as_float(o[2 * i]) * inv, __uint_as_float(o[2 * i + 1]) * inv);
            if (qpos < L) {
                uint4 *dst = reinterpret_cast<uint4 *>(out + static_cast<long long>(row0 + qpos) * kHidden
                                                       + head * kHeadDim + h * 32);
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    dst[i] = make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
    pdl_trigger();
}

}  // namespace

cudaError_t launch_attn_generic(const AttnArgs &a, cudaStream_t stream)
{
    static PerDeviceOnce smem_once;
    cudaError_t e = smem_opt_in(smem_once, attn_generic_kernel, kSmemBytes);
    if (e != cudaSuccess)
        return e;
    const long long grid = static_cast<long long>(a.entry_bound) * kHeads;
    return launch_chained(attn_generic_kernel, dim3(static_cast<unsigned>(grid)), dim3(kThreads), kSmemBytes, stream,
        a.tm_rot, a.tm_qkv, a.cu, a.work, a.work_count, a.half_window, a.out, a.err);
}

}  // namespace mbert
