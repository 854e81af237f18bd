// Device-side building blocks for the sm_103a attention kernels: constants of
// the block, the tile schedule and mask predicate, and thin inline-PTX
// wrappers for mbarrier, TMA (cp.async.bulk.tensor), and tcgen05 (TMEM
// allocation, MMA, loads and stores).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

namespace mbert {

// ---------------------------------------------------------------------------
// shape of the block ("ModernBERT-base Architecture Teardown", "How Does
// ModernBERT Make Q, K and V?": 12 heads of 64; Wqkv output 2304 = 3 x 768)
// ---------------------------------------------------------------------------
constexpr int kHeads = 12;
constexpr int kHeadDim = 64;
constexpr int kHidden = kHeads * kHeadDim;      // 768
constexpr int kQKVWidth = 3 * kHidden;          // 2304
constexpr int kPairs = kHeadDim / 2;            // 32 RoPE pairs per head
constexpr int kInnerMlp = 1152;                 // the GeGLU MLP's inner width (Wi: 2 x 1152)

constexpr int kBlockM = 128;                    // query rows per tile
constexpr int kBlockN = 128;                    // key rows per tile
constexpr int kTileBytes = kBlockM * kHeadDim * 2;  // 16 KB bf16 tile

// device error word bits
constexpr int kErrBadCu = 1;
constexpr int kErrTooLong = 2;
constexpr int kErrTimeout = 4;
constexpr int kErrPairTmem = 8;   // a CTA pair's TMEM allocations disagree

// bounded waits give up after this long (ns) and report kErrTimeout
constexpr unsigned long long kWaitLimitNs = 2000000000ull;

// ---------------------------------------------------------------------------
// tile schedule and mask (shared by the attention and key-count kernels)
// ---------------------------------------------------------------------------

// Key tiles [kt0, kt1) of 128 keys, aligned to the sequence start, that hold
// at least one key admitted for some valid query of the block starting at
// position q0 of a sequence of length L.  hw < 0: global layer.
__device__ __forceinline__ void key_tile_range(int q0, int L, int hw, int &kt0, int &kt1)
{
    if (hw < 0) {
        kt0 = 0;
        kt1 = (L + kBlockN - 1) / kBlockN;
        return;
    }
    const int qlast = min(q0 + kBlockM - 1, L - 1);
    const int lo = max(0, q0 - hw);
    const int hi = min(L - 1, qlast + hw);
    kt0 = lo / kBlockN;
    kt1 = hi / kBlockN + 1;
}

// Does key tile kt need the per-element mask for the query block at q0?
// False only when every key of the tile lies in the sequence and is
// admitted for every valid query of the block.
__device__ __forceinline__ bool tile_needs_mask(int q0, int L, int hw, int kt)
{
    const int k0 = kt * kBlockN, k1 = k0 + kBlockN - 1;
    if (k1 >= L)
        return true;
    if (hw < 0)
        return false;
    const int qlast = min(q0 + kBlockM - 1, L - 1);
    return !(k1 - q0 <= hw && qlast - k0 <= hw);
}

// Key position j is visible to query position i (both in one sequence of
// length L): inside the sequence and, on a local layer, |i - j| <= hw.
__device__ __forceinline__ bool admitted(int i, int j, int L, int hw)
{
    return j < L && (hw < 0 || abs(i - j) <= hw);
}

// ---------------------------------------------------------------------------
// local-band schedule (shared by the local attention and key-count kernels)
//
// A block of 128 queries at position q0 sees keys in [q0 - hw, q0 + 127 + hw];
// for hw <= 64 two 128-key tiles cover that: tile 0 = keys q0 - 64 .. q0 + 63,
// tile 1 = keys q0 + 64 .. q0 + 191.  Warp w (queries q0 + 32w .. + 31)
// visits only the 32-key chunks of a tile that can hold a key within 64 of
// one of its queries: chunks w..3 of tile 0 and chunks 0..w of tile 1
// (5 chunks, 160 keys, per row instead of 256).
// ---------------------------------------------------------------------------
constexpr int kBandReach = 64;   // tile geometry supports half windows up to this

__device__ __forceinline__ int band_tile_key0(int q0, int tile) { return q0 - 64 + 128 * tile; }
__device__ __forceinline__ int band_chunk_begin(int tile, int w) { return tile == 0 ? w : 0; }
__device__ __forceinline__ int band_chunk_end(int tile, int w) { return tile == 0 ? 4 : w + 1; }

// Must chunk c of `tile` be masked element by element for warp w?  Not when
// every key of the chunk lies in the sequence and within hw (= 64) of every
// query of the warp: off-diagonal chunks of interior blocks.
__device__ __forceinline__ bool band_chunk_needs_mask(int q0, int L, int hw, int tile, int w, int c)
{
    const int k0 = band_tile_key0(q0, tile) + 32 * c;
    if (k0 < 0 || k0 + 31 >= L || hw != kBandReach)
        return true;
    return c == w;
}

// ---------------------------------------------------------------------------
// small PTX helpers
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ unsigned long long globaltimer_ns()
{
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ uint32_t elect_one_sync()
{
    uint32_t pred = 0;
    asm volatile(
        "{\n\t.reg .b32 rx;\n\t.reg .pred px;\n\t"
        "elect.sync rx|px, %1;\n\t"
        "@px mov.s32 %0, 1;\n\t}"
        : "+r"(pred) : "r"(0xffffffffu));
    return pred;
}

// ---- programmatic dependent launch ----
// Every kernel is launched so that its launch may overlap the end of the
// kernel before it in the stream.  A kernel calls pdl_wait() before its
// first global-memory access (it returns once the previous kernel has
// completed and its writes are visible; at once if there is none), and
// pdl_trigger() when its own work is done, which lets the next kernel's
// launch begin before this grid has fully retired.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// ---- thread-block clusters ----
__device__ __forceinline__ uint32_t cluster_ctarank()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// Every thread of every CTA in the cluster arrives (release) and waits
// (acquire).
__device__ __forceinline__ void cluster_sync()
{
    asm volatile("barrier.cluster.arrive.release;\n\t"
                 "barrier.cluster.wait.acquire;" ::: "memory");
}

// ---- mbarrier ----
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" :: "r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;"
                 :: "r"(bar), "r"(bytes) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" :: "r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok) : "r"(bar), "r"(parity) : "memory");
    return ok != 0;
}

// try_wait with a suspend-time hint: a waiting warp sleeps in hardware until
// the phase completes (or about `hint_ns` pass) instead of re-polling, so it
// takes no issue slots from the warps that share its SM sub-partition.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint32_t bar, uint32_t parity, uint32_t hint_ns)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok) : "r"(bar), "r"(parity), "r"(hint_ns) : "memory");
    return ok != 0;
}

// Wait for the phase with the given parity to complete.  Gives up once
// `limit_ns` of global time or 2.5 * limit_ns SM cycles have passed
// (whichever comes first, so that the wait ends even if one clock stalls),
// then sets kErrTimeout in *err and returns false.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, int *err,
                                          unsigned long long limit_ns = kWaitLimitNs)
{
    if (mbar_try_wait(bar, parity))
        return true;
    const unsigned long long t0 = globaltimer_ns();
    const long long c0 = clock64();
    const long long climit = static_cast<long long>(limit_ns) * 5 / 2;
    for (;;) {
        if (mbar_try_wait_sleep(bar, parity, 1000000u))
            return true;
        if (globaltimer_ns() - t0 > limit_ns || clock64() - c0 > climit)
            break;
    }
    atomicOr(err, kErrTimeout);
    return false;
}

// ---- TMA ----
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap *tm)
{
    asm volatile("prefetch.tensormap [%0];" :: "l"(reinterpret_cast<uint64_t>(tm)) : "memory");
}

// 2-D tiled load of the box at (x = column, y = row) into shared memory;
// completes `bar` with the box's byte count.  Rows outside the tensor read 0.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *tm, int x, int y,
                                            uint32_t bar)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];"
        :: "r"(dst), "l"(reinterpret_cast<uint64_t>(tm)), "r"(x), "r"(y), "r"(bar)
        : "memory");
}

__device__ __forceinline__ void tma_load_2d_hint(uint32_t dst, const CUtensorMap *tm, int x,
                                                 int y, uint32_t bar, uint64_t policy)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        ".L2::cache_hint [%0], [%1, {%2, %3}], [%4], %5;"
        :: "r"(dst), "l"(reinterpret_cast<uint64_t>(tm)), "r"(x), "r"(y), "r"(bar),
           "l"(policy)
        : "memory");
}

// Fetch `bytes` (a multiple of 16) from a 16-byte aligned global address
// into L2, with no completion to wait for.
__device__ __forceinline__ void l2_prefetch_bytes(const void *p, uint32_t bytes)
{
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;"
                 :: "l"(reinterpret_cast<uint64_t>(p)), "r"(bytes) : "memory");
}

// 2-D tiled store of the box at (x = column, y = row) from shared memory
// (bulk async-group of the issuing thread); x, y >= 0.
__device__ __forceinline__ void tma_store_2d(const CUtensorMap *tm, uint32_t src, int x, int y)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.global.shared::cta.tile.bulk_group [%0, {%1, %2}], [%3];"
        :: "l"(reinterpret_cast<uint64_t>(tm)), "r"(x), "r"(y), "r"(src)
        : "memory");
}

__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }

// the issuing thread's bulk stores have finished reading shared memory
__device__ __forceinline__ void bulk_wait_read0() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }

// the issuing thread's bulk stores have completed
__device__ __forceinline__ void bulk_wait0() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

__device__ __forceinline__ uint64_t l2_policy_evict_last()
{
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ uint64_t l2_policy_evict_first()
{
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// generic-proxy shared-memory writes -> visible to the async proxy (MMA, TMA)
__device__ __forceinline__ void fence_proxy_async_smem()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---- tcgen05: TMEM allocation ----
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols)
{
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                 :: "r"(dst_smem), "r"(ncols) : "memory");
}

__device__ __forceinline__ void tmem_relinquish()
{
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols)
{
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;"
                 :: "r"(taddr), "r"(ncols) : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// ---- tcgen05: descriptors ----

// Instruction descriptor for kind::f16 with bf16 A and B and an fp32
// accumulator: D format at bits [4,6), A/B formats at [7,10) and [10,13),
// A/B major-ness at bits 15/16 (0 = K-major, 1 = MN-major), N>>3 at
// [17,23), M>>4 at [24,29).
__host__ __device__ constexpr uint32_t make_idesc_bf16(int M, int N, bool b_mn_major)
{
    return (1u << 4) | (1u << 7) | (1u << 10) | ((b_mn_major ? 1u : 0u) << 16) |
           (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}

// Shared-memory matrix descriptor, 128-byte swizzle: start address >> 4 at
// [0,14), leading-dimension byte offset >> 4 at [16,30), stride-dimension
// byte offset >> 4 at [32,46), descriptor version 1 at [46,48), base offset 0
// (tiles are 1024-byte aligned), layout type 2 (SWIZZLE_128B) at [61,64).
__device__ __forceinline__ uint64_t make_sdesc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo)
{
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
    d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
    d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
    d |= static_cast<uint64_t>(1) << 46;
    d |= static_cast<uint64_t>(2) << 61;
    return d;
}

// ---- tcgen05: MMA ----
// D[tmem] (+)= A[smem] * B[smem]; issued by a single thread.
__device__ __forceinline__ void mma_bf16_ss(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                            uint32_t idesc, uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}"
        :: "r"(d_tmem), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// D[tmem] (+)= A[tmem] * B[smem]; issued by a single thread.
__device__ __forceinline__ void mma_bf16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc,
                                            uint32_t idesc, uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}"
        :: "r"(d_tmem), "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Warp-wide variants: called by all 32 lanes of a converged warp (so the
// descriptors stay warp-uniform); one lane, chosen by elect.sync, issues.
__device__ __forceinline__ void mma_bf16_ss_warp(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                                 uint32_t idesc, uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p, e;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}"
        :: "r"(d_tmem), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void mma_bf16_ts_warp(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc,
                                                 uint32_t idesc, uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p, e;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}"
        :: "r"(d_tmem), "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void mma_commit_warp(uint32_t bar)
{
    asm volatile(
        "{\n\t.reg .pred e;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}"
        :: "r"(bar) : "memory");
}

// Arrive once on `bar` when every MMA this thread issued so far is complete.
__device__ __forceinline__ void mma_commit(uint32_t bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
                 :: "r"(bar) : "memory");
}

// ---- tcgen05: TMEM <-> registers (32 lanes x 32-bit, one lane per thread) ----
#define MBERT_R8(i) "=r"(r[i]), "=r"(r[i + 1]), "=r"(r[i + 2]), "=r"(r[i + 3]), \
                    "=r"(r[i + 4]), "=r"(r[i + 5]), "=r"(r[i + 6]), "=r"(r[i + 7])

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32])
{
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : MBERT_R8(0), MBERT_R8(8), MBERT_R8(16), MBERT_R8(24)
        : "r"(taddr));
}

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16])
{
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : MBERT_R8(0), MBERT_R8(8)
        : "r"(taddr));
}
#undef MBERT_R8

#define MBERT_W8(i) "r"(r[i]), "r"(r[i + 1]), "r"(r[i + 2]), "r"(r[i + 3]), \
                    "r"(r[i + 4]), "r"(r[i + 5]), "r"(r[i + 6]), "r"(r[i + 7])

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32])
{
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
        "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
        "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};"
        :: "r"(taddr), MBERT_W8(0), MBERT_W8(8), MBERT_W8(16), MBERT_W8(24)
        : "memory");
}

__device__ __forceinline__ void tmem_st64(uint32_t taddr, const uint32_t (&r)[64])
{
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x64.b32 [%0], "
        "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
        "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32,"
        "%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,%48,"
        "%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63,%64};"
        :: "r"(taddr), MBERT_W8(0), MBERT_W8(8), MBERT_W8(16), MBERT_W8(24),
           MBERT_W8(32), MBERT_W8(40), MBERT_W8(48), MBERT_W8(56)
        : "memory");
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16])
{
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
        "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};"
        :: "r"(taddr), MBERT_W8(0), MBERT_W8(8)
        : "memory");
}
#undef MBERT_W8

// Ties 32 registers to this point of the program: code that reads them is not
// scheduled above an earlier tcgen05.wait::ld (the load's destination
// registers are only valid after that wait).
#define MBERT_RW8(i) "+r"(r[i]), "+r"(r[i + 1]), "+r"(r[i + 2]), "+r"(r[i + 3]), \
                     "+r"(r[i + 4]), "+r"(r[i + 5]), "+r"(r[i + 6]), "+r"(r[i + 7])
__device__ __forceinline__ void reg_fence32(uint32_t (&r)[32])
{
    asm volatile("" : MBERT_RW8(0), MBERT_RW8(8), MBERT_RW8(16), MBERT_RW8(24));
}
#undef MBERT_RW8

// ---- math ----
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

// packed fp32x2 values (lo, hi) in one 64-bit register pair
__device__ __forceinline__ uint64_t f2(float lo, float hi)
{
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}

__device__ __forceinline__ void f2_split(uint64_t v, float &lo, float &hi)
{
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}

__device__ __forceinline__ uint64_t fmul2(uint64_t a, uint64_t b)
{
    uint64_t d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

__device__ __forceinline__ uint64_t ffma2(uint64_t a, uint64_t b, uint64_t c)
{
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}

// bf16x2 word -> fp32x2 (exact)
__device__ __forceinline__ uint64_t bf16x2_to_f2(uint32_t v)
{
    return f2(__uint_as_float(v << 16), __uint_as_float(v & 0xFFFF0000u));
}

// fp32x2 -> bf16x2 word, round to nearest even
__device__ __forceinline__ uint32_t f2_to_bf16x2(uint64_t v)
{
    float lo, hi;
    f2_split(v, lo, hi);
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

__device__ __forceinline__ float fmax3(float a, float b, float c)
{
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

__device__ __forceinline__ float ex2_approx(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// two floats -> packed bf16x2 (lo in bits 0..15), round to nearest even
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi)
{
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

__device__ __forceinline__ float bf16lo_to_f32(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16hi_to_f32(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }

}  // namespace mbert
