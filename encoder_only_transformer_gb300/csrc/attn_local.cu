// Local-layer attention with RoPE fused into the prologue (tcgen05 + TMA,
// sm_103a).
//
// A local layer keeps key j for query i when |i - j| <= 64 ("ModernBERT"
// (candding), "The alternating attention"), so for a block of 128 queries
// starting at q0 every visible key lies in the 256-key window [q0 - 64,
// q0 + 192), two 128-key tiles.  Query row r sees window columns
// [r, r + 128]; warp w (rows 32w .. 32w + 31) therefore only ever needs the
// five 32-key chunks starting at window column 32w, and never rescales: the
// softmax of a row is taken in one go over its five chunks.
//
// Persistent: one CTA per SM walks a contiguous range of units (sequence,
// 128-query block, head) in the order head, then work entry.  Consecutive
// blocks of one sequence share a key tile (tile 1 of block b is tile 0 of
// block b + 1), so a unit that continues its predecessor loads and rotates
// only Q and one new K/V tile.
//
//   warp 8      producer: TMA of raw Q, K, V tiles (16 KB, 128-byte swizzle)
//               straight from the fused qkv rows into 4-deep rings
//   warp 9      MMA issuer: S = Q [K0 K1]^T (256 TMEM columns), then, once
//               softmax has written P, O = P0 V0 + P1 V1
//   warps 0-3,  two compute groups taking alternate units: RoPE in shared
//   warps 4-7   memory (rotate-half, positions restarting per sequence;
//               "ModernBERT-base Architecture Teardown", "How Does RoPE Work
//               With Two Bases?"), softmax (fp32, base 2) writing bf16 P over
//               the S columns it has read, and the epilogue out = O / l
//
// TMEM: 512 columns, 256 per group: S over the window [0, 256); P0 packed
// into [0, 64), P1 into [128, 192); O into [64, 128).
//
// Work split: with a null work list the CTA finds the blocks from cu_seqlens
// itself (and checks the whole array first, so a bad array makes every CTA
// exit without writing); otherwise it walks the plan kernel's entries.
#include "common.cuh"
#include "internal.h"

namespace mbert {
namespace {

constexpr int kThreads = 320;
constexpr int kGroupThreads = 128;
constexpr int kWarpProducer = 8;
constexpr int kWarpMma = 9;
constexpr int kRing = 4;
constexpr uint32_t kOffQ = 0;
constexpr uint32_t kOffK = kRing * kTileBytes;
constexpr uint32_t kOffV = 2 * kRing * kTileBytes;
constexpr uint32_t kOffBar = 3 * kRing * kTileBytes;
constexpr uint32_t kSmemBytes = kOffBar + 512 + 1024;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kGroupCols = 256;
constexpr uint32_t kColO = 64;

enum : int {
    kBarQF = 0, kBarQE = 4, kBarKF = 8, kBarKE = 12, kBarVF = 16, kBarVE = 20,
    kBarRope = 24, kBarS = 26, kBarP = 28, kBarO = 30, kBarFree = 32, kBarDrain = 34,
    kNumBars = 35
};

constexpr uint32_t kIdescS = make_idesc_bf16(128, 128, false);
constexpr uint32_t kIdescO = make_idesc_bf16(128, 64, true);
constexpr float kScaleLog2 = 0.125f * 1.4426950408889634f;
constexpr float kSlack = 64.0f;     // reference maximum may sit this far (base 2) below the row maximum
constexpr unsigned long long kDrainLimitNs = 100000000ull;

__device__ __forceinline__ uint32_t barp(uint32_t base, int i) { return base + kOffBar + 8u * i; }
__device__ __forceinline__ uint32_t ring_parity(int t) { return static_cast<uint32_t>(t / kRing) & 1u; }

// Chunks j and j + 4 (elements 8j .. 8j + 7 and 32 + 8j .. 32 + 8j + 7, the
// pairs m = 8j .. 8j + 7) of one 128-byte swizzled row (64 bf16): 16-byte
// chunk c of row r sits at chunk c ^ (r % 8).
struct PairChunks {
    uint32_t x[4], z[4];
};

__device__ __forceinline__ void pair_load(uint32_t row_addr, int r, int j, PairChunks &v)
{
    const uint32_t a = row_addr + ((j ^ (r & 7)) << 4);
    const uint32_t b = row_addr + (((j + 4) ^ (r & 7)) << 4);
    asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x[0]), "=r"(v.x[1]), "=r"(v.x[2]), "=r"(v.x[3]) : "r"(a));
    asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];" : "=r"(v.z[0]), "=r"(v.z[1]), "=r"(v.z[2]), "=r"(v.z[3]) : "r"(b));
}

// Rotate the pairs (x[m], x[m + 32]) by the angles whose cosines and sines
// are c[m - 8j], s[m - 8j] and store the two chunks back.
__device__ __forceinline__ void pair_rotate_store(uint32_t row_addr, int r, int j, const PairChunks &v,
                                                  const float (&c)[8], const float (&s)[8])
{
    uint32_t ya[4], yb[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float x0 = bf16lo_to_f32(v.x[i]), x1 = bf16hi_to_f32(v.x[i]);
        const float z0 = bf16lo_to_f32(v.z[i]), z1 = bf16hi_to_f32(v.z[i]);
        ya[i] = pack_bf16x2(x0 * c[2 * i] - z0 * s[2 * i], x1 * c[2 * i + 1] - z1 * s[2 * i + 1]);
        yb[i] = pack_bf16x2(z0 * c[2 * i] + x0 * s[2 * i], z1 * c[2 * i + 1] + x1 * s[2 * i + 1]);
    }
    const uint32_t a = row_addr + ((j ^ (r & 7)) << 4);
    const uint32_t b = row_addr + (((j + 4) ^ (r & 7)) << 4);
    asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" :: "r"(a), "r"(ya[0]), "r"(ya[1]), "r"(ya[2]), "r"(ya[3]) : "memory");
    asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" :: "r"(b), "r"(yb[0]), "r"(yb[1]), "r"(yb[2]), "r"(yb[3]) : "memory");
}

// cos and sin of the RoPE angle pos * w for one frequency w, given as turns
// per position in 64-bit fixed point (fhi, flo = 2^-32 and 2^-64 turns).
// The fractional turns of pos * w are formed exactly modulo 1 in integer
// arithmetic (the top 32 bits of pos * (fhi.flo) mod 2^32), read as a signed
// fraction in [-1/2, 1/2), and the angle in [-pi, pi) goes to the fast sine
// and cosine.
__device__ __forceinline__ void pos_cos_sin(uint32_t pos, uint32_t fhi, uint32_t flo, float &c,
                                            float &s)
{
    const uint32_t ph = __umulhi(pos, flo) + pos * fhi;
    const float phi = static_cast<float>(static_cast<int32_t>(ph)) * 1.4629180792671596e-9f;  // 2 pi / 2^32
    __sincosf(phi, &s, &c);
}

__device__ __forceinline__ float max32(const uint32_t (&x)[32])
{
    float t[8];
#pragma unroll
    for (int k = 0; k < 8; ++k)
        t[k] = fmax3(__uint_as_float(x[k]), __uint_as_float(x[k + 8]),
                     fmaxf(__uint_as_float(x[k + 16]), __uint_as_float(x[k + 24])));
    return fmaxf(fmax3(t[0], t[1], t[2]), fmaxf(fmax3(t[3], t[4], t[5]), fmaxf(t[6], t[7])));
}

// ---------------------------------------------------------------------------
// the unit walk
// ---------------------------------------------------------------------------

// Number of 128-query blocks over all sequences, with the whole of
// cu_seqlens checked (one warp).  Returns -1 if the array is invalid (CTA 0
// records why in *err).
__device__ int count_blocks(const int32_t *__restrict__ cu, int n_seqs, long long T, int max_seqlen,
                            int32_t *err)
{
    const int lane = threadIdx.x & 31;
    int bad = 0, total = 0;
    if (lane == 0 && (cu[0] != 0 || static_cast<long long>(cu[n_seqs]) != T))
        bad |= kErrBadCu;
#pragma unroll 4
    for (int s = lane; s < n_seqs; s += 32) {
        const int L = cu[s + 1] - cu[s];
        if (L < 0)
            bad |= kErrBadCu;
        else if (L > max_seqlen)
            bad |= kErrTooLong;
        else
            total += (L + kBlockM - 1) / kBlockM;
    }
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) {
        bad |= __shfl_xor_sync(0xffffffffu, bad, d);
        total += __shfl_xor_sync(0xffffffffu, total, d);
    }
    if (bad) {
        if (blockIdx.x == 0 && lane == 0)
            atomicOr(err, bad);
        return -1;
    }
    return total;
}

// Sequence and block of block number e (0 <= e < the count above), blocks
// numbered sequence by sequence (one warp; cu_seqlens already checked).
__device__ void locate_block(const int32_t *__restrict__ cu, int n_seqs, int e, int &seq, int &qb)
{
    const int lane = threadIdx.x & 31;
    int base = 0;
    seq = -1;
    qb = 0;
    for (int s0 = 0; s0 < n_seqs && seq < 0; s0 += 32) {
        const int s = s0 + lane;
        const int nb = s < n_seqs ? (cu[s + 1] - cu[s] + kBlockM - 1) / kBlockM : 0;
        int incl = nb;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, incl, d);
            if (lane >= d)
                incl += v;
        }
        const int excl = base + incl - nb;
        const unsigned hit = __ballot_sync(0xffffffffu, nb > 0 && e >= excl && e < excl + nb);
        if (hit) {
            const int src = __ffs(hit) - 1;
            seq = s0 + src;
            qb = e - __shfl_sync(0xffffffffu, excl, src);
        }
        base += __shfl_sync(0xffffffffu, incl, 31);
    }
}

// Walks the CTA's units in order.  Every role runs its own copy; all copies
// see the same sequence.  `fresh` is set when a unit does not continue its
// predecessor (first unit, new head, new sequence, or a gap in the work
// list): then its key tile 0 must be loaded and rotated too.
struct Walker {
    const int32_t *cu;
    const int2 *work;   // null: blocks sequence by sequence
    int G;              // entries per head
    int e, head, seq, qb;
    int row0, L;
    bool fresh;

    __device__ void start(const int32_t *cu_, const int2 *work_, int G_, long long u, int seq0, int qb0)
    {
        cu = cu_;
        work = work_;
        G = G_;
        head = static_cast<int>(u / G);
        e = static_cast<int>(u % G);
        if (work) {
            const int2 w = work[e];
            seq = w.x;
            qb = w.y;
        } else {
            seq = seq0;
            qb = qb0;
        }
        row0 = cu[seq];
        L = cu[seq + 1] - row0;
        fresh = true;
    }

    __device__ void next()
    {
        const int pseq = seq, pqb = qb, phead = head;
        if (++e == G) {
            e = 0;
            ++head;
        }
        if (work) {
            const int2 w = work[e];
            seq = w.x;
            qb = w.y;
        } else if (e == 0) {
            seq = 0;
            while (cu[seq + 1] == cu[seq])
                ++seq;
            qb = 0;
        } else if ((qb + 1) * kBlockM < L) {
            ++qb;
        } else {
            ++seq;
            while (cu[seq + 1] == cu[seq])
                ++seq;
            qb = 0;
        }
        if (seq != pseq) {
            row0 = cu[seq];
            L = cu[seq + 1] - row0;
        }
        fresh = !(head == phead && seq == pseq && qb == pqb + 1);
    }
};

__global__ void __launch_bounds__(kThreads, 1)
attn_local_kernel(const __grid_constant__ CUtensorMap tm_qkv, const __grid_constant__ RopeConsts rope,
                  const int32_t *__restrict__ cu, int n_seqs, long long T, int max_seqlen,
                  const int2 *__restrict__ work, const int32_t *__restrict__ work_count, int hw,
                  __nv_bfloat16 *__restrict__ out, int32_t *err)
{
    extern __shared__ uint8_t smem_raw[];
    __shared__ long long s_range[2];
    __shared__ int s_first[3];
    __shared__ uint32_t s_tmem;
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    // ---- this CTA's range of units [u_lo, u_hi) of heads x G
    if (warp == 0) {
        int G = work ? *work_count : count_blocks(cu, n_seqs, T, max_seqlen, err);
        long long lo = 0, hi = 0;
        if (G > 0) {
            const long long U = static_cast<long long>(kHeads) * G;
            lo = U * blockIdx.x / gridDim.x;
            hi = U * (blockIdx.x + 1) / gridDim.x;
        }
        int seq0 = 0, qb0 = 0;
        if (lo < hi && !work)
            locate_block(cu, n_seqs, static_cast<int>(lo % G), seq0, qb0);
        if (lane == 0) {
            s_range[0] = lo;
            s_range[1] = hi;
            s_first[0] = G;
            s_first[1] = seq0;
            s_first[2] = qb0;
        }
    }
    __syncthreads();
    const long long u_lo = s_range[0];
    const int nunits = static_cast<int>(s_range[1] - u_lo);
    if (nunits <= 0)
        return;
    const int G = s_first[0];

    if (warp == 0) {
        tmem_alloc(smem_u32(&s_tmem), kTmemCols);
        tmem_relinquish();
    }
    if (tid == 32) {
        tma_prefetch_desc(&tm_qkv);
        for (int i = 0; i < kNumBars; ++i) {
            uint32_t count = 1;
            if (i == kBarRope || i == kBarRope + 1 || i == kBarP || i == kBarP + 1 ||
                i == kBarFree || i == kBarFree + 1)
                count = kGroupThreads;
            mbar_init(barp(base, i), count);
        }
        fence_mbar_init();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = s_tmem;

    Walker w;
    w.start(cu, work, G, u_lo, s_first[1], s_first[2]);

    if (warp == kWarpProducer) {
        // ------------------------------------------------------ producer
        const uint64_t once = l2_policy_evict_first();
        int nq = 0, tk = 0, tv = 0;   // tiles issued per ring (issued in index order)
        bool ok = true;
        // wait for the ring slot of tile t, then TMA the 128 x 64 box at
        // (column x, row y) into it
        auto load = [&](uint32_t ring_off, int bar_full, int bar_empty, int t, int x, int y,
                        int &issued) {
            if (!ok)
                return;
            if (!(ok = mbar_wait(barp(base, bar_empty + t % kRing), ring_parity(t) ^ 1u, err)))
                return;
            if (elect_one_sync()) {
                mbar_arrive_expect_tx(barp(base, bar_full + t % kRing), kTileBytes);
                tma_load_2d_hint(base + ring_off + (t % kRing) * kTileBytes, &tm_qkv, x, y,
                                 barp(base, bar_full + t % kRing), once);
            }
            __syncwarp();
            issued = t + 1;
        };
        int tc = 0;
        for (int k = 0; k < nunits && ok; ++k) {
            const int a = w.fresh ? tc : tc - 1;
            tc = a + 2;
            const int colQ = w.head * kHeadDim, colK = kHidden + colQ, colV = 2 * kHidden + colQ;
            const int r0 = w.row0 + w.qb * kBlockM;
            if (w.fresh)
                load(kOffK, kBarKF, kBarKE, a, colK, r0 - 64, tk);
            load(kOffQ, kBarQF, kBarQE, k, colQ, r0, nq);
            load(kOffK, kBarKF, kBarKE, a + 1, colK, r0 + 64, tk);
            if (w.fresh)
                load(kOffV, kBarVF, kBarVE, a, colV, r0 - 64, tv);
            load(kOffV, kBarVF, kBarVE, a + 1, colV, r0 + 64, tv);
            if (k + 1 < nunits)
                w.next();
        }
        // every copy issued has landed before the CTA can exit
        for (int t = max(0, nq - kRing); t < nq; ++t)
            mbar_wait(barp(base, kBarQF + t % kRing), ring_parity(t), err, kDrainLimitNs);
        for (int t = max(0, tk - kRing); t < tk; ++t)
            mbar_wait(barp(base, kBarKF + t % kRing), ring_parity(t), err, kDrainLimitNs);
        for (int t = max(0, tv - kRing); t < tv; ++t)
            mbar_wait(barp(base, kBarVF + t % kRing), ring_parity(t), err, kDrainLimitNs);
    } else if (warp == kWarpMma) {
        // ------------------------------------------------------ MMA issuer
        bool ok = true;
        int tc = 0;
        int a_prev = 0, a_prev2 = 0;
        bool fresh_prev = true;
        // O = P0 V0 + P1 V1 of unit kp (tiles ap, ap + 1); a fresh unit that
        // follows another also retires its predecessor's V tile 1.
        auto issue_pv = [&](int kp, int ap, bool fresh_p, int ap_before) -> bool {
            const int g = kp & 1;
            const uint32_t tm = tmem + g * kGroupCols;
            if (!(mbar_wait(barp(base, kBarP + g), static_cast<uint32_t>(kp >> 1) & 1u, err) &&
                  mbar_wait(barp(base, kBarVF + ap % kRing), ring_parity(ap), err) &&
                  mbar_wait(barp(base, kBarVF + (ap + 1) % kRing), ring_parity(ap + 1), err)))
                return false;
            __syncwarp();
            tc_fence_after();
#pragma unroll
            for (int t = 0; t < 2; ++t) {
                const uint32_t v = base + kOffV + ((ap + t) % kRing) * kTileBytes;
#pragma unroll
                for (int kk = 0; kk < kBlockN / 16; ++kk)
                    mma_bf16_ts_warp(tm + kColO, tm + 128 * t + 8 * kk,
                                     make_sdesc_sw128(v + 2048 * kk, 1024, 1024), kIdescO,
                                     (t > 0 || kk > 0) ? 1u : 0u);
            }
            mma_commit_warp(barp(base, kBarO + g));
            mma_commit_warp(barp(base, kBarVE + ap % kRing));
            if (fresh_p && kp > 0)
                mma_commit_warp(barp(base, kBarVE + (ap_before + 1) % kRing));
            return true;
        };
        for (int k = 0; k < nunits && ok; ++k) {
            const bool fresh = w.fresh;
            const int a = fresh ? tc : tc - 1;
            tc = a + 2;
            const int g = k & 1, j = k >> 1;
            const uint32_t tm = tmem + g * kGroupCols;
            ok = mbar_wait(barp(base, kBarRope + g), static_cast<uint32_t>(j) & 1u, err) &&
                 (j == 0 || mbar_wait(barp(base, kBarFree + g), static_cast<uint32_t>(j - 1) & 1u, err));
            if (!ok)
                break;
            __syncwarp();
            tc_fence_after();
            const uint32_t q = base + kOffQ + (k % kRing) * kTileBytes;
#pragma unroll
            for (int t = 0; t < 2; ++t) {
                const uint32_t kt = base + kOffK + ((a + t) % kRing) * kTileBytes;
#pragma unroll
                for (int kk = 0; kk < kHeadDim / 16; ++kk)
                    mma_bf16_ss_warp(tm + 128 * t, make_sdesc_sw128(q + 32 * kk, 16, 1024),
                                     make_sdesc_sw128(kt + 32 * kk, 16, 1024), kIdescS, kk > 0);
            }
            mma_commit_warp(barp(base, kBarS + g));
            mma_commit_warp(barp(base, kBarQE + k % kRing));
            mma_commit_warp(barp(base, kBarKE + a % kRing));
            if (fresh && k > 0)
                mma_commit_warp(barp(base, kBarKE + (a_prev + 1) % kRing));
            if (k > 0)
                ok = issue_pv(k - 1, a_prev, fresh_prev, a_prev2);
            a_prev2 = a_prev;
            a_prev = a;
            fresh_prev = fresh;
            if (k + 1 < nunits)
                w.next();
        }
        if (ok)
            issue_pv(nunits - 1, a_prev, fresh_prev, a_prev2);
        // every MMA issued has completed before TMEM is released
        mma_commit_warp(barp(base, kBarDrain));
        mbar_wait(barp(base, kBarDrain), 0, err, kDrainLimitNs);
    } else if (warp < 8) {
        // ------------------------------------------------------ compute groups
        const int g = warp >> 2, wq = warp & 3;
        const int r = 32 * wq + lane;                 // row in the block, TMEM lane
        const uint32_t tm = tmem + g * kGroupCols + (static_cast<uint32_t>(32 * wq) << 16);
        bool ok = true;
        int tc = 0, j = 0;
        // the group's previous unit, whose epilogue runs after the next
        // unit's RoPE (while its P V product is on the tensor cores)
        int p_row = -1, p_col = 0;
        float p_inv = 0.f;

        auto epilogue = [&](int jp) -> bool {
            if (!mbar_wait(barp(base, kBarO + g), static_cast<uint32_t>(jp) & 1u, err))
                return false;
            __syncwarp();
            tc_fence_after();
            uint32_t o[2][32];
            tmem_ld32(tm + kColO, o[0]);
            tmem_ld32(tm + kColO + 32, o[1]);
            tmem_wait_ld();
            reg_fence32(o[0]);
            reg_fence32(o[1]);
            if (p_row >= 0) {
                uint4 *dst = reinterpret_cast<uint4 *>(out + static_cast<long long>(p_row) * kHidden + p_col);
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    const uint32_t *x = o[k / 4] + 8 * (k % 4);
                    dst[k] = make_uint4(
                        pack_bf16x2(__uint_as_float(x[0]) * p_inv, __uint_as_float(x[1]) * p_inv),
                        pack_bf16x2(__uint_as_float(x[2]) * p_inv, __uint_as_float(x[3]) * p_inv),
                        pack_bf16x2(__uint_as_float(x[4]) * p_inv, __uint_as_float(x[5]) * p_inv),
                        pack_bf16x2(__uint_as_float(x[6]) * p_inv, __uint_as_float(x[7]) * p_inv));
                }
            }
            tc_fence_before();
            mbar_arrive(barp(base, kBarFree + g));
            return true;
        };

        for (int k = 0; k < nunits && ok; ++k) {
            const bool fresh = w.fresh;
            const int a = fresh ? tc : tc - 1;
            tc = a + 2;
            if ((k & 1) == g) {
                const int q0 = w.qb * kBlockM, L = w.L;
                // ---- RoPE.  Thread r takes position p = q0 + 64 + r: K
                // tile 1 row r, and the Q row at p (r + 64, for r < 64) or
                // at p - 128 (r - 64, for r >= 64), and on a fresh unit K
                // tile 0 row r (at p - 128).  cos/sin at p - 128 come from
                // those at p by one rotation of -128 positions.
                ok = mbar_wait(barp(base, kBarQF + k % kRing), ring_parity(k), err) &&
                     mbar_wait(barp(base, kBarKF + (a + 1) % kRing), ring_parity(a + 1), err) &&
                     (!fresh || mbar_wait(barp(base, kBarKF + a % kRing), ring_parity(a), err));
                if (ok) {
                    const uint32_t qs = base + kOffQ + (k % kRing) * kTileBytes;
                    const uint32_t k0s = base + kOffK + (a % kRing) * kTileBytes;
                    const uint32_t k1s = base + kOffK + ((a + 1) % kRing) * kTileBytes;
                    const uint32_t p = static_cast<uint32_t>(q0 + 64 + r);
                    const bool q_at_p = r < 64;          // warp-uniform
                    const int qr = q_at_p ? r + 64 : r - 64;
#pragma unroll 1
                    for (int jj = 0; jj < 4; ++jj) {
                        // the rows' chunks first (one shared-memory round
                        // trip), then the angles, then rotate and store
                        PairChunks vk1, vq, vk0;
                        pair_load(k1s + r * 128, r, jj, vk1);
                        pair_load(qs + qr * 128, qr, jj, vq);
                        if (fresh)
                            pair_load(k0s + r * 128, r, jj, vk0);
                        float c[8], s[8], cm[8], sm[8], cq[8], sq[8];
#pragma unroll
                        for (int kx = 0; kx < 8; ++kx) {
                            const int m = 8 * jj + kx;
                            pos_cos_sin(p, rope.frac_hi[m], rope.frac_lo[m], c[kx], s[kx]);
                            cm[kx] = c[kx] * rope.cos128[m] + s[kx] * rope.sin128[m];
                            sm[kx] = s[kx] * rope.cos128[m] - c[kx] * rope.sin128[m];
                            cq[kx] = q_at_p ? c[kx] : cm[kx];
                            sq[kx] = q_at_p ? s[kx] : sm[kx];
                        }
                        pair_rotate_store(k1s + r * 128, r, jj, vk1, c, s);
                        pair_rotate_store(qs + qr * 128, qr, jj, vq, cq, sq);
                        if (fresh)
                            pair_rotate_store(k0s + r * 128, r, jj, vk0, cm, sm);
                    }
                    fence_proxy_async_smem();
                }
                mbar_arrive(barp(base, kBarRope + g));
                if (!ok)
                    break;

                if (j > 0 && !(ok = epilogue(j - 1)))
                    break;

                // ---- softmax over the window chunks 32 wq .. 32 wq + 159
                const int i = q0 + r;
                // admitted keys [klo, khi]; none for rows past the sequence
                const int klo = i < L ? max(0, i - hw) : L, khi = min(L - 1, i + hw);
                if (!(ok = mbar_wait(barp(base, kBarS + g), static_cast<uint32_t>(j) & 1u, err)))
                    break;
                __syncwarp();
                tc_fence_after();
                // masked keys of chunk e (window columns 32 (wq + e) ..) ->
                // -inf; only the edge chunks, chunks at a sequence edge or a
                // narrower band have any
                auto mask = [&](uint32_t (&x)[32], int e) {
                    const int key0 = q0 - 64 + 32 * (wq + e);
                    if (e == 0 || e == 4 || hw != kBandReach || key0 < 0 || key0 + 31 >= L) {
                        const int lo = klo - key0, hi = khi - key0;
#pragma unroll
                        for (int kx = 0; kx < 32; ++kx)
                            if (kx < lo || kx > hi)
                                x[kx] = __float_as_uint(-INFINITY);
                    }
                };
                // The reference maximum m (base 2, scaled) is taken from
                // window chunk 2, which holds the diagonal key i of every
                // row; p = 2^(s * scale - m) is then written chunk by chunk
                // in one pass.  Any reference within 2^kSlack of the row
                // maximum gives the same softmax up to rounding; a chunk
                // whose maximum exceeds m by more than that raises m and
                // rescales the P already written (exact powers of two).
                uint32_t cur[32], nxt[32];
                tmem_ld32(tm + 32 * wq, cur);
                tmem_ld32(tm + 32 * (wq + 2), nxt);
                tmem_wait_ld();
                reg_fence32(cur);
                reg_fence32(nxt);
                mask(nxt, 2);
                float m = max32(nxt) * kScaleLog2;
                float sum = 0.f;
#pragma unroll 1
                for (int e = 0; e < 5; ++e) {
                    if (e < 4)
                        tmem_ld32(tm + 32 * (wq + e + 1), nxt);
                    mask(cur, e);
                    const float cmax = max32(cur) * kScaleLog2;
                    if (__any_sync(0xffffffffu, cmax > m + kSlack)) {
                        const float mn = fmaxf(m, cmax);
                        const float f = m == -INFINITY ? 0.f : ex2_approx(m - mn);
                        tmem_wait_st();
#pragma unroll 1
                        for (int e2 = 0; e2 < e; ++e2) {
                            const int col2 = 32 * (wq + e2);
                            const uint32_t pa = tm + col2 / 2 + (col2 >= 128 ? 64 : 0);
                            uint32_t pv[16];
                            tmem_ld16(pa, pv);
                            tmem_wait_ld();
#pragma unroll
                            for (int kx = 0; kx < 16; ++kx)
                                pv[kx] = pack_bf16x2(bf16lo_to_f32(pv[kx]) * f, bf16hi_to_f32(pv[kx]) * f);
                            tmem_st16(pa, pv);
                        }
                        sum *= f;
                        m = mn;
                    }
                    const float m_use = m == -INFINITY ? 0.f : m;
                    uint32_t pk[16];
                    float a0 = 0.f, a1 = 0.f;
#pragma unroll
                    for (int kx = 0; kx < 16; ++kx) {
                        const float p0 = ex2_approx(fmaf(__uint_as_float(cur[2 * kx]), kScaleLog2, -m_use));
                        const float p1 = ex2_approx(fmaf(__uint_as_float(cur[2 * kx + 1]), kScaleLog2, -m_use));
                        a0 += p0;
                        a1 += p1;
                        pk[kx] = pack_bf16x2(p0, p1);
                    }
                    sum += a0 + a1;
                    // P chunk of window column c sits at c / 2 (+ 64 in tile
                    // 1): below every S column not yet read
                    const int col = 32 * (wq + e);
                    tmem_st16(tm + col / 2 + (col >= 128 ? 64 : 0), pk);
                    if (e < 4) {
                        tmem_wait_ld();
                        reg_fence32(nxt);
#pragma unroll
                        for (int kx = 0; kx < 32; ++kx)
                            cur[kx] = nxt[kx];
                    }
                }
                {
                    uint32_t z[16];
#pragma unroll
                    for (int kx = 0; kx < 16; ++kx)
                        z[kx] = 0u;
                    for (int c = 0; c < wq; ++c)
                        tmem_st16(tm + 16 * c, z);
                    for (int c = wq + 1; c < 4; ++c)
                        tmem_st16(tm + 128 + 16 * c, z);
                }
                tmem_wait_st();
                tc_fence_before();
                mbar_arrive(barp(base, kBarP + g));
                p_row = i < L ? w.row0 + i : -1;
                p_col = w.head * kHeadDim;
                p_inv = sum > 0.f ? 1.f / sum : 0.f;
                ++j;
            }
            if (k + 1 < nunits)
                w.next();
        }
        if (ok && j > 0)
            epilogue(j - 1);
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
    const long long units = static_cast<long long>(a.block_bound) * kHeads;
    const long long grid = units < a.num_ctas ? units : a.num_ctas;
    if (grid <= 0)
        return cudaSuccess;
    attn_local_kernel<<<static_cast<unsigned>(grid), kThreads, kSmemBytes, stream>>>(
        a.tm_qkv, a.rope, a.cu, a.n_seqs, a.T, a.max_seqlen, a.work, a.work_count,
        a.half_window, a.out, a.err);
    return cudaGetLastError();
}

}  // namespace mbert
