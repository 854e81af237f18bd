// The block's two projections, as paired-SM GEMMs (tcgen05 + TMA, sm_103a):
//
//  * qkv_proj_kernel: qkv = h Wqkv^T, h bf16 [T][768] (the pre-attention
//    LayerNorm's output, or x itself on layer 0), Wqkv bf16 [2304][768]
//    stored [out][in] ("ModernBERT-base Architecture Teardown", "How Does
//    ModernBERT Make Q, K and V?": Wqkv turns 768 numbers into 2304; the
//    norm's output times Wqkv^T, "ModernBertModel", "Implementing it");
//    qkv bf16 [T][2304].
//  * out_proj_kernel: y = x + a Wo^T, a the joined head outputs bf16
//    [T][768], Wo bf16 [768][768] stored [out][in] (same section: Wo maps
//    the joined heads back from 768 to 768), x the residual stream bf16
//    [T][768] ("Implementing it": x = x + a Wo^T); y bf16 [T][768].
//  * mlp_up_kernel: m = GELU(g) * u with g, u the first and second halves of
//    h Wi^T, h bf16 [T][768] (the MLP's LayerNorm output), Wi bf16
//    [2304][768] ("ModernBERT-base Architecture Teardown", "What Does the
//    GeGLU MLP Do?"; the first half is the GELU branch, "modernbert-base",
//    "The fused projections"), GELU in the exact erf form ("ModernBERT"
//    (candding), "The feed-forward halves"); m bf16 [T][1152].
//  * mlp_down_kernel: y = x + m Wo^T, Wo bf16 [768][1152] (K = 1152).
// All accumulate in fp32 and round once to bf16.
//
// The tensor pipe of one SM takes 128 x N x 16 per 64 clocks at N = 128,
// and an SM's copy engine delivers about 64 bytes per clock, which feeds a
// 128 x 128 tile at only half that rate.  So the kernel pairs SMs: a cluster
// of two CTAs issues tcgen05.mma.cta_group::2 with M = 256 and N = 256, each
// CTA holding 128 rows of a and 128 rows of Wo (half of B) per K step, which
// is 32 KB per 512 clocks of MMA.
//
// Persistent pairs: each takes a contiguous run of units, a unit being 256
// rows x 256 output columns (row-major over the units); CTA r of the pair
// owns rows 128 r .. 128 r + 127 of the unit.  K = 768 is walked in 12 steps
// of 64 (A = the activations, B = the weight):
//   warp 0      producer (both CTAs): TMA of the CTA's A box and B box
//               (128 x 64 each, 128-byte swizzle) into a 5-stage ring, both
//               completing the leader CTA's stage barrier
//   warp 1      MMA issuer (leader CTA only): D (+)= A B^T over the pair
//               into one of two 256-column TMEM accumulators per CTA; each
//               stage's commit frees the stage in both CTAs
//   warps 2-9   epilogue (both CTAs): warp w takes TMEM lane quadrant w % 4
//               and column half (w - 2) / 4, one row per thread; the output
//               goes through a staging tile and TMA stores that clip rows
//               past T.  With the residual, the unit's x first arrives in the
//               staging tile by TMA (fetched into L2 a unit ahead) and
//               y = D + x is written over it; the lead thread loads the next
//               unit's x once the store has read the tile.
// y may be x itself: a unit reads its x before its y is stored, and no other
// unit touches those elements.
#include "common.cuh"
#include "internal.h"

namespace mbert {
namespace {

constexpr int kThreads = 320;
constexpr int kEpiWarps = 8;
constexpr int kBM = 128;                // rows per CTA
constexpr int kUnitM = 2 * kBM;         // rows per unit (the pair)
constexpr int kBN = 256;                // output columns per unit (MMA N)
constexpr int kBK = 64;
constexpr int kInner = kInnerMlp;       // the MLP's inner width
constexpr int kStages = 5;
constexpr uint32_t kStageBytes = 2 * kTileBytes;             // A box + B box (this CTA's half)
constexpr uint32_t kOffRing = 0;
constexpr uint32_t kOffY = kStages * kStageBytes;            // staging tile: 128 rows x 256 columns
constexpr int kYBoxes = kBN / 64;
constexpr uint32_t kYBytes = kYBoxes * kTileBytes;
constexpr uint32_t kOffBar = kOffY + kYBytes;
constexpr uint32_t kSmemBytes = kOffBar + 256 + 1024;
constexpr uint32_t kTmemCols = 2 * kBN; // two fp32 accumulators of 256 columns
constexpr uint16_t kPairMask = 0x3;
static_assert(kSmemBytes + 16 <= 227 * 1024, "shared memory");

enum : int {
    kBarFull = 0, kBarEmpty = kStages, kBarAccFull = 2 * kStages, kBarAccEmpty = kBarAccFull + 2,
    kBarXFull = kBarAccEmpty + 2,  // residual: x landed; otherwise: the staging tile is free
    kBarYReady, kBarDrain,
    kNumBars
};

constexpr uint32_t kIdesc = make_idesc_bf16(kUnitM, kBN, false);
constexpr unsigned long long kDrainLimitNs = 100000000ull;

__device__ __forceinline__ uint32_t barp(uint32_t base, int i) { return base + kOffBar + 8u * i; }

// ---- the pair forms of the tcgen05 and TMA wrappers ----

// the address of the same shared-memory offset in CTA `rank` of the cluster
__device__ __forceinline__ uint32_t map_to_rank(uint32_t addr, uint32_t rank)
{
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
    return r;
}

__device__ __forceinline__ uint32_t ld_shared_cluster_u32(uint32_t addr)
{
    uint32_t v;
    asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
    return v;
}

__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr)
{
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];"
                 :: "r"(cluster_addr) : "memory");
}

__device__ __forceinline__ void tmem_alloc_pair(uint32_t dst_smem, uint32_t ncols)
{
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;"
                 :: "r"(dst_smem), "r"(ncols) : "memory");
}

__device__ __forceinline__ void tmem_relinquish_pair()
{
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols)
{
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;"
                 :: "r"(taddr), "r"(ncols) : "memory");
}

// D (+)= A B over the pair: A rows 0..127 and B rows 0..N/2-1 from the
// leader's shared memory, the rest from the peer's at the same offsets.
__device__ __forceinline__ void mma_pair_warp(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                              uint32_t idesc, uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p, e;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "@e tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}"
        :: "r"(d_tmem), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// arrive once on the mbarrier at offset `bar` of each CTA in `cta_mask` when
// the pair MMAs issued so far are complete
__device__ __forceinline__ void mma_commit_pair_warp(uint32_t bar, uint16_t cta_mask)
{
    asm volatile(
        "{\n\t.reg .pred e;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "@e tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
        " [%0], %1;\n\t}"
        :: "r"(bar), "h"(cta_mask) : "memory");
}

// tma_load_2d_hint into this CTA's shared memory, completing an mbarrier
// that may sit in the peer CTA (cluster address)
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const CUtensorMap *tm, int x, int y,
                                                 uint32_t bar_cluster, uint64_t policy)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        ".cta_group::2.L2::cache_hint [%0], [%1, {%2, %3}], [%4], %5;"
        :: "r"(dst), "l"(reinterpret_cast<uint64_t>(tm)), "r"(x), "r"(y), "r"(bar_cluster),
           "l"(policy)
        : "memory");
}

// y = v + x for one 64-column box row: x read from the swizzled staging
// row (16-byte chunk c at c ^ (r % 8)), bf16 y written over it.
__device__ __forceinline__ void add_x_row(uint32_t rowp, int r, const uint32_t (&v)[2][32])
{
    uint32_t xw[8][4];
#pragma unroll
    for (int c = 0; c < 8; ++c)
        asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];"
                     : "=r"(xw[c][0]), "=r"(xw[c][1]), "=r"(xw[c][2]), "=r"(xw[c][3])
                     : "r"(rowp + ((c ^ (r & 7)) << 4)));
#pragma unroll
    for (int c = 0; c < 8; ++c) {
        uint32_t yw[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const uint32_t a0 = v[c / 4][8 * (c % 4) + 2 * e], a1 = v[c / 4][8 * (c % 4) + 2 * e + 1];
            yw[e] = pack_bf16x2(__uint_as_float(a0) + bf16lo_to_f32(xw[c][e]),
                                __uint_as_float(a1) + bf16hi_to_f32(xw[c][e]));
        }
        asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};"
                     :: "r"(rowp + ((c ^ (r & 7)) << 4)), "r"(yw[0]), "r"(yw[1]), "r"(yw[2]), "r"(yw[3])
                     : "memory");
    }
}

// bf16(v) for one 64-column box row into the swizzled staging row.
__device__ __forceinline__ void store_row(uint32_t rowp, int r, const uint32_t (&v)[2][32])
{
#pragma unroll
    for (int c = 0; c < 8; ++c) {
        uint32_t yw[4];
#pragma unroll
        for (int e = 0; e < 4; ++e)
            yw[e] = pack_bf16x2(__uint_as_float(v[c / 4][8 * (c % 4) + 2 * e]),
                                __uint_as_float(v[c / 4][8 * (c % 4) + 2 * e + 1]));
        asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};"
                     :: "r"(rowp + ((c ^ (r & 7)) << 4)), "r"(yw[0]), "r"(yw[1]), "r"(yw[2]), "r"(yw[3])
                     : "memory");
    }
}

// What the epilogue makes of the accumulator D of a unit.
enum class Epi {
    kPlain,      // y = D (256 output columns per unit)
    kResidual,   // y = x + D (256 output columns per unit)
    kGeglu       // y = GELU(g) * u (128 output columns per unit; D holds g, then u)
};

// GELU(g) * u for 64 output columns of one row into the swizzled staging
// row, GELU in its exact erf form: z / 2 * (1 + erf(z / sqrt 2)).
__device__ __forceinline__ void geglu_row(uint32_t rowp, int r, const uint32_t (&g)[2][32],
                                          const uint32_t (&u)[2][32])
{
    constexpr float kRsqrt2 = 0.70710678118654752f;
#pragma unroll
    for (int c = 0; c < 8; ++c) {
        uint32_t yw[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            float m[2];
#pragma unroll
            for (int k = 0; k < 2; ++k) {
                const int col = 8 * (c % 4) + 2 * e + k;
                const float z = __uint_as_float(g[c / 4][col]);
                m[k] = 0.5f * z * (1.0f + erff(z * kRsqrt2)) * __uint_as_float(u[c / 4][col]);
            }
            yw[e] = pack_bf16x2(m[0], m[1]);
        }
        asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};"
                     :: "r"(rowp + ((c ^ (r & 7)) << 4)), "r"(yw[0]), "r"(yw[1]), "r"(yw[2]), "r"(yw[3])
                     : "memory");
    }
}

// The kernel body: K = 64 kKSteps; kColBlocks column blocks per row block of
// 256 rows.  kPlain / kResidual: block j is output columns 256 j .. + 255,
// weight rows the same.  kGeglu: block j is output columns 128 j .. + 127,
// from weight rows 128 j .. + 127 (g, the leader CTA's half of B) and
// kInner + 128 j .. + 127 (u, the peer's half).
template <int kKSteps, int kColBlocks, Epi kEpi>
__device__ __forceinline__ void pair_gemm(const CUtensorMap &tm_a, const CUtensorMap &tm_w,
                                          const CUtensorMap &tm_x, const CUtensorMap &tm_y,
                                          const __nv_bfloat16 *x, long long T, int n_units,
                                          int32_t *err)
{
    extern __shared__ uint8_t smem_raw[];
    __shared__ uint32_t s_tmem;
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;     // the same offset in both CTAs
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int rank = static_cast<int>(cluster_ctarank());
    const bool leader = rank == 0;
    const int cluster = blockIdx.x >> 1, n_clusters = gridDim.x >> 1;
    // units [u_begin, u_begin + my_units), the same for both CTAs of the pair
    const int u_begin = static_cast<int>(static_cast<long long>(cluster) * n_units / n_clusters);
    int my_units =
        static_cast<int>(static_cast<long long>(cluster + 1) * n_units / n_clusters) - u_begin;
    if (my_units <= 0)
        return;

    if (warp == 1) {
        tmem_alloc_pair(smem_u32(&s_tmem), kTmemCols);
        tmem_relinquish_pair();
    } else if (tid == 0) {
        tma_prefetch_desc(&tm_a);
        tma_prefetch_desc(&tm_w);
        if constexpr (kEpi == Epi::kResidual)
            tma_prefetch_desc(&tm_x);
        tma_prefetch_desc(&tm_y);
        for (int i = 0; i < kNumBars; ++i) {
            uint32_t count = 1;
            if (i == kBarAccEmpty || i == kBarAccEmpty + 1)
                count = 2 * kEpiWarps;                   // the epilogue warps of both CTAs
            if (i == kBarYReady)
                count = 32 * kEpiWarps;
            mbar_init(barp(base, i), count);
        }
        fence_mbar_init();
    }
    tc_fence_before();
    cluster_sync();                                      // both CTAs' barriers and TMEM exist
    tc_fence_after();
    const uint32_t tmem = s_tmem;
    // The pair's accumulators must sit at the same TMEM address in both CTAs.
    if (ld_shared_cluster_u32(map_to_rank(smem_u32(&s_tmem), rank ^ 1)) != tmem) {
        if (tid == 0)
            atomicOr(err, kErrPairTmem);
        my_units = 0;
    }

    if (warp == 0) {
        // ------------------------------------------------------ producer
        const uint64_t keep = l2_policy_evict_last();    // a rows and Wo: re-read by other units
        bool ok = true;
        int g = 0;
        for (int i = 0; i < my_units && ok; ++i) {
            const int u = u_begin + i;
            const int m0 = (u / kColBlocks) * kUnitM + rank * kBM;
            const int w0 = kEpi == Epi::kGeglu ? rank * kInner + (u % kColBlocks) * (kBN / 2)
                                               : (u % kColBlocks) * kBN + rank * (kBN / 2);
            for (int k = 0; k < kKSteps && ok; ++k, ++g) {
                const int st = g % kStages;
                if (!(ok = mbar_wait(barp(base, kBarEmpty + st), ((g / kStages) & 1) ^ 1u, err)))
                    break;
                if (elect_one_sync()) {
                    const uint32_t dst = base + kOffRing + st * kStageBytes;
                    const uint32_t full = map_to_rank(barp(base, kBarFull + st), 0);
                    if (leader)                          // both CTAs' boxes land on the leader's barrier
                        mbar_arrive_expect_tx(barp(base, kBarFull + st), 2 * kStageBytes);
                    tma_load_2d_pair(dst, &tm_a, k * kBK, m0, full, keep);
                    tma_load_2d_pair(dst + kTileBytes, &tm_w, k * kBK, w0, full, keep);
                }
                __syncwarp();
            }
        }
        // every stage this CTA loaded has been read by the pair's MMAs
        for (int t = max(0, g - kStages); t < g; ++t)
            mbar_wait(barp(base, kBarEmpty + t % kStages), (t / kStages) & 1, err, kDrainLimitNs);
    } else if (warp == 1) {
        // ------------------------------------------------------ MMA issuer
        if (leader) {
            bool ok = true;
            int g = 0;
            for (int i = 0; i < my_units && ok; ++i) {
                const int acc = i & 1;
                const uint32_t d = tmem + acc * kBN;
                if (!(ok = mbar_wait(barp(base, kBarAccEmpty + acc), ((i >> 1) & 1) ^ 1u, err)))
                    break;
                __syncwarp();
                tc_fence_after();
                for (int k = 0; k < kKSteps && ok; ++k, ++g) {
                    const int st = g % kStages;
                    if (!(ok = mbar_wait(barp(base, kBarFull + st), (g / kStages) & 1, err)))
                        break;
                    __syncwarp();
                    tc_fence_after();
                    const uint32_t sa = base + kOffRing + st * kStageBytes;
                    const uint32_t sb = sa + kTileBytes;
#pragma unroll
                    for (int kk = 0; kk < kBK / 16; ++kk)
                        mma_pair_warp(d, make_sdesc_sw128(sa + 32 * kk, 16, 1024),
                                      make_sdesc_sw128(sb + 32 * kk, 16, 1024), kIdesc,
                                      (k > 0 || kk > 0) ? 1u : 0u);
                    mma_commit_pair_warp(barp(base, kBarEmpty + st), kPairMask);
                }
                if (ok)
                    mma_commit_pair_warp(barp(base, kBarAccFull + acc), kPairMask);
            }
            // every MMA issued has completed before TMEM is released
            mma_commit_pair_warp(barp(base, kBarDrain), 0x1);
            mbar_wait(barp(base, kBarDrain), 0, err, kDrainLimitNs);
        }
    } else {
        // ------------------------------------------------------ epilogue
        constexpr bool kRes = kEpi == Epi::kResidual;
        constexpr int kOutCols = kEpi == Epi::kGeglu ? kBN / 2 : kBN;   // output columns per unit
        constexpr int kOutBoxes = kOutCols / 64;
        constexpr int kOutWidth = kColBlocks * kOutCols;               // row length of y (and x)
        const int q = warp & 3;                        // TMEM lane quadrant: rows 32 q .. 32 q + 31
        const int hf = (warp - 2) >> 2;                // column half of the unit's output
        const int r = 32 * q + lane;                   // row in the tile, TMEM lane
        const bool lead = warp == 2 && lane == 0;      // x loads and y stores
        const uint32_t lane_off = static_cast<uint32_t>(32 * q) << 16;
        const uint64_t once = l2_policy_evict_first(); // x: read once
        auto unit_m0 = [&](int i) { return ((u_begin + i) / kColBlocks) * kUnitM + rank * kBM; };
        auto unit_n0 = [&](int i) { return ((u_begin + i) % kColBlocks) * kOutCols; };
        // this thread's half row of unit i's x into L2
        auto prefetch_x = [&](int i) {
            const long long row = static_cast<long long>(unit_m0(i)) + r;
            if (row < T)
                l2_prefetch_bytes(x + static_cast<size_t>(row) * kOutWidth + unit_n0(i) + 128 * hf, 256);
        };
        auto load_x = [&](int i) {                     // unit i's x into the staging tile
            const uint32_t bar = barp(base, kBarXFull);
            mbar_arrive_expect_tx(bar, kYBytes);
            for (int b = 0; b < kYBoxes; ++b)
                tma_load_2d_hint(base + kOffY + b * kTileBytes, &tm_x, unit_n0(i) + 64 * b, unit_m0(i), bar, once);
        };
        int x_issued = 0, x_done = 0;
        if constexpr (kRes) {
            if (lead && my_units > 0) {
                load_x(0);
                x_issued = 1;
            }
        }
        bool ok = true;
        for (int i = 0; i < my_units && ok; ++i) {
            if constexpr (kRes) {
                if (i + 1 < my_units)
                    prefetch_x(i + 1);                 // a unit ahead of its load
            }
            const int acc = i & 1;
            // the accumulator is complete; with the residual the unit's x has
            // landed, otherwise the previous unit's store has read the tile
            bool ready = mbar_wait(barp(base, kBarAccFull + acc), static_cast<uint32_t>(i >> 1) & 1u, err);
            if constexpr (kRes)
                ready = ready && mbar_wait(barp(base, kBarXFull), static_cast<uint32_t>(i & 1), err);
            else
                ready = ready && (i == 0 || mbar_wait(barp(base, kBarXFull), static_cast<uint32_t>((i - 1) & 1), err));
            if (!(ok = ready))
                break;
            x_done = i + 1;
            __syncwarp();
            tc_fence_after();
            const uint32_t dacc = tmem + acc * kBN + lane_off;
            if constexpr (kEpi == Epi::kGeglu) {
                // output columns 64 hf .. + 63: g at accumulator columns
                // 64 hf .., u at 128 + 64 hf ..
                uint32_t vg[2][32], vu[2][32];
                tmem_ld32(dacc + 64 * hf, vg[0]);
                tmem_ld32(dacc + 64 * hf + 32, vg[1]);
                tmem_ld32(dacc + 128 + 64 * hf, vu[0]);
                tmem_ld32(dacc + 128 + 64 * hf + 32, vu[1]);
                tmem_wait_ld();
                reg_fence32(vg[0]);
                reg_fence32(vg[1]);
                reg_fence32(vu[0]);
                reg_fence32(vu[1]);
                geglu_row(base + kOffY + hf * kTileBytes + r * 128, r, vg, vu);
            } else {
                // box 2 hf + bb holds columns 64 (2 hf + bb) .. + 63; the
                // second box's accumulator loads while the first is written
                uint32_t va[2][32], vb[2][32];
                tmem_ld32(dacc + 128 * hf, va[0]);
                tmem_ld32(dacc + 128 * hf + 32, va[1]);
                tmem_wait_ld();
                reg_fence32(va[0]);
                reg_fence32(va[1]);
                tmem_ld32(dacc + 128 * hf + 64, vb[0]);
                tmem_ld32(dacc + 128 * hf + 96, vb[1]);
                if constexpr (kRes)
                    add_x_row(base + kOffY + (2 * hf) * kTileBytes + r * 128, r, va);
                else
                    store_row(base + kOffY + (2 * hf) * kTileBytes + r * 128, r, va);
                tmem_wait_ld();
                reg_fence32(vb[0]);
                reg_fence32(vb[1]);
                if constexpr (kRes)
                    add_x_row(base + kOffY + (2 * hf + 1) * kTileBytes + r * 128, r, vb);
                else
                    store_row(base + kOffY + (2 * hf + 1) * kTileBytes + r * 128, r, vb);
            }
            // the accumulator may be reused: one arrival per warp at the leader
            tc_fence_before();
            __syncwarp();
            if (lane == 0)
                mbar_arrive_cluster(map_to_rank(barp(base, kBarAccEmpty + acc), 0));
            fence_proxy_async_smem();
            mbar_arrive(barp(base, kBarYReady));
            if (lead) {
                if (!(ok = mbar_wait(barp(base, kBarYReady), static_cast<uint32_t>(i & 1), err)))
                    break;
                const int m0 = unit_m0(i);
                if (m0 < T) {                            // rows past T are not stored
                    for (int b = 0; b < kOutBoxes; ++b)
                        tma_store_2d(&tm_y, base + kOffY + b * kTileBytes, unit_n0(i) + 64 * b, m0);
                    bulk_commit();
                }
                if constexpr (kRes) {
                    if (i + 1 < my_units) {
                        bulk_wait_read0();               // the store has read the staging tile
                        load_x(i + 1);
                        x_issued = i + 2;
                    }
                } else {
                    bulk_wait_read0();
                    mbar_arrive(barp(base, kBarXFull));  // the staging tile may be rewritten
                }
            }
        }
        if (lead) {
            // an x load still in flight after a timeout lands before the exit
            if (kRes && x_done < x_issued)
                mbar_wait(barp(base, kBarXFull), static_cast<uint32_t>((x_issued - 1) & 1), err, kDrainLimitNs);
            bulk_wait0();                                // the stores have completed
        }
    }

    tc_fence_before();
    cluster_sync();                   // neither CTA exits while the other may still signal it
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc_pair(tmem, kTmemCols);
    }
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
out_proj_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_w,
                const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_y,
                const __nv_bfloat16 *x, long long T, int n_units, int32_t *err)
{
    pdl_wait();
    pair_gemm<kHidden / kBK, kHidden / kBN, Epi::kResidual>(tm_a, tm_w, tm_x, tm_y, x, T, n_units, err);
    pdl_trigger();
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
qkv_proj_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_w,
                const __grid_constant__ CUtensorMap tm_y, long long T, int n_units, int32_t *err)
{
    pdl_wait();
    pair_gemm<kHidden / kBK, kQKVWidth / kBN, Epi::kPlain>(tm_a, tm_w, tm_y, tm_y, nullptr, T, n_units, err);
    pdl_trigger();
}

// The MLP's first GEMM with its GeGLU: m = GELU(h Wi_g^T) * (h Wi_u^T),
// [T][1152] from h [T][768] and Wi [2304][768].
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
mlp_up_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_w,
              const __grid_constant__ CUtensorMap tm_y, long long T, int n_units, int32_t *err)
{
    pdl_wait();
    pair_gemm<kHidden / kBK, kInner / (kBN / 2), Epi::kGeglu>(tm_a, tm_w, tm_y, tm_y, nullptr, T, n_units, err);
    pdl_trigger();
}

// The MLP's second GEMM with the residual: y = x + m Wo^T, K = 1152.
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
mlp_down_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_w,
                const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_y,
                const __nv_bfloat16 *x, long long T, int n_units, int32_t *err)
{
    pdl_wait();
    pair_gemm<kInner / kBK, kHidden / kBN, Epi::kResidual>(tm_a, tm_w, tm_x, tm_y, x, T, n_units, err);
    pdl_trigger();
}

// Pairs of CTAs to launch for `kernel`: as many as fit at once (per device,
// found once, with the shared-memory opt-in set first), at most one per unit.
template <typename Kernel>
cudaError_t pair_count(Kernel kernel, PerDeviceOnce &once, int num_ctas, long long n_units, int *pairs)
{
    int fit = 0;
    cudaError_t e = per_device_once(once, &fit, [&](int *out) {
        cudaError_t r = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(kSmemBytes));
        if (r != cudaSuccess)
            return r;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(2 * (num_ctas / 2));
        cfg.blockDim = dim3(kThreads);
        cfg.dynamicSmemBytes = kSmemBytes;
        int n = 0;
        r = cudaOccupancyMaxActiveClusters(&n, kernel, &cfg);
        *out = n > 0 ? n : 1;
        return r;
    });
    if (e != cudaSuccess)
        return e;
    *pairs = static_cast<int>(n_units < fit ? n_units : fit);   // >= 1 unit each
    return cudaSuccess;
}

}  // namespace

cudaError_t launch_out_proj(const OutProjArgs &a, cudaStream_t stream)
{
    static PerDeviceOnce max_pairs;
    const long long n_units = ((a.T + kUnitM - 1) / kUnitM) * (kHidden / kBN);
    if (n_units <= 0)
        return cudaSuccess;
    int pairs = 0;
    cudaError_t e = pair_count(out_proj_kernel, max_pairs, a.num_ctas, n_units, &pairs);
    if (e != cudaSuccess)
        return e;
    return launch_chained(out_proj_kernel, dim3(2 * pairs), dim3(kThreads), kSmemBytes, stream,
        a.tm_a, a.tm_w, a.tm_x, a.tm_y, a.x, a.T, static_cast<int>(n_units), a.err);
}

cudaError_t launch_mlp_down(const OutProjArgs &a, cudaStream_t stream)
{
    static PerDeviceOnce max_pairs;
    const long long n_units = ((a.T + kUnitM - 1) / kUnitM) * (kHidden / kBN);
    if (n_units <= 0)
        return cudaSuccess;
    int pairs = 0;
    cudaError_t e = pair_count(mlp_down_kernel, max_pairs, a.num_ctas, n_units, &pairs);
    if (e != cudaSuccess)
        return e;
    return launch_chained(mlp_down_kernel, dim3(2 * pairs), dim3(kThreads), kSmemBytes, stream,
        a.tm_a, a.tm_w, a.tm_x, a.tm_y, a.x, a.T, static_cast<int>(n_units), a.err);
}

cudaError_t launch_qkv_proj(const QkvProjArgs &a, cudaStream_t stream)
{
    static PerDeviceOnce max_pairs;
    const long long n_units = ((a.T + kUnitM - 1) / kUnitM) * (kQKVWidth / kBN);
    if (n_units <= 0)
        return cudaSuccess;
    int pairs = 0;
    cudaError_t e = pair_count(qkv_proj_kernel, max_pairs, a.num_ctas, n_units, &pairs);
    if (e != cudaSuccess)
        return e;
    return launch_chained(qkv_proj_kernel, dim3(2 * pairs), dim3(kThreads), kSmemBytes, stream,
        a.tm_a, a.tm_w, a.tm_y, a.T, static_cast<int>(n_units), a.err);
}

cudaError_t launch_mlp_up(const QkvProjArgs &a, cudaStream_t stream)
{
    static PerDeviceOnce max_pairs;
    const long long n_units = ((a.T + kUnitM - 1) / kUnitM) * (kInner / (kBN / 2));
    if (n_units <= 0)
        return cudaSuccess;
    int pairs = 0;
    cudaError_t e = pair_count(mlp_up_kernel, max_pairs, a.num_ctas, n_units, &pairs);
    if (e != cudaSuccess)
        return e;
    return launch_chained(mlp_up_kernel, dim3(2 * pairs), dim3(kThreads), kSmemBytes, stream,
        a.tm_a, a.tm_w, a.tm_y, a.T, static_cast<int>(n_units), a.err);
}

}  // namespace mbert
