// Local-layer attention with RoPE fused into the prologue (tcgen05 + TMA,
// sm_103a).
//
// A local layer keeps key j for query i when |i - j| <= 64 ("ModernBERT"
// (candding), "The alternating attention"), so for a block of 128 queries
// starting at q0 every visible key lies in the 256-key window [q0 - 64,
// q0 + 192), two 128-key tiles.  Query row r sees window columns
// [r, r + 128]; the rows 32w .. 32w + 31 therefore only ever need the five
// 32-key chunks starting at window column 32w, and the softmax of a row is
// taken in one pass over them.
//
// Persistent: one CTA per SM walks a contiguous range of units (sequence,
// 128-query block, head) in the order head, then work entry.  Consecutive
// blocks of one sequence share a key tile (tile 1 of block b is tile 0 of
// block b + 1), so a unit that continues its predecessor loads and rotates
// only Q and one new K/V tile.
//
//   warp 8      producer: TMA of raw Q, K, V tiles (16 KB, 128-byte swizzle)
//               straight from the fused qkv rows into rings (3 Q, 4 K, 4 V),
//               and each unit's record (rows, block, head) beside its Q tile
//   warps 9, 10 MMA issuers, one per compute group: S = Q [K0 K1]^T (256
//               TMEM columns), then, once softmax has written P,
//               O = P0 V0 + P1 V1
//   warps 0-3,  two compute groups taking alternate units, one thread per
//   warps 4-7   row: RoPE in shared memory (rotate-half, positions restarting
//               per sequence; "ModernBERT-base Architecture Teardown", "How
//               Does RoPE Work With Two Bases?"), softmax (fp32, base 2)
//               writing bf16 P over the S columns already read, and the
//               epilogue out = O / l through a staging tile and a TMA store
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

constexpr int kThreads = 352;
constexpr int kGroupThreads = 128;     // 4 warps, one per TMEM lane quadrant
constexpr int kWarpProducer = 8;
constexpr int kWarpMma = 9;            // + group: one MMA issuer per compute group
constexpr int kQRing = 3;              // Q tiles
constexpr int kRing = 4;               // K and V tiles
constexpr uint32_t kOffQ = 0;
constexpr uint32_t kOffK = kQRing * kTileBytes;
constexpr uint32_t kOffV = kOffK + kRing * kTileBytes;
constexpr uint32_t kOffStage = kOffV + kRing * kTileBytes;   // per group: O tile (bf16) for the TMA store
constexpr uint32_t kOffBias = kOffStage + 2 * kTileBytes;   // band edge masks: [2 chunks][32 lanes][32] fp32
constexpr uint32_t kOffRec = kOffBias + 8192;               // per Q slot: the unit's record (32 bytes)
constexpr uint32_t kOffPrev = kOffRec + kQRing * 32;         // per group: the unit awaiting its epilogue (16 bytes)
constexpr uint32_t kOffBar = kOffRec + 128;
constexpr uint32_t kSmemBytes = kOffBar + 512 + 1024;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kGroupCols = 256;
constexpr uint32_t kColO = 64;

// Ring barriers (one per slot): full (TMA landed), empty (consumers done;
// K and V take two arrivals per tile: one from each unit using it, or two
// from a tile's only user), rotated (RoPE done; Q and K).  Per group: S
// ready, P written, O ready, TMEM free (epilogue done), drain, staging tile
// written (all rows), staging tile free (the previous TMA store has read
// it).
enum : int {
    kBarQF = 0, kBarQE = 3, kBarKF = 6, kBarKE = 10, kBarVF = 14, kBarVE = 18,
    kBarQR = 22, kBarKR = 25,
    kBarS = 29, kBarP = 31, kBarO = 33, kBarFree = 35, kBarDrain = 37,
    kBarStg = 39, kBarStgFree = 41,
    kNumBars = 43
};

constexpr uint32_t kIdescS = make_idesc_bf16(128, 128, false);
constexpr uint32_t kIdescO = make_idesc_bf16(128, 64, true);
constexpr float kScaleLog2 = 0.125f * 1.4426950408889634f;
constexpr float kSlack = 64.0f;     // reference maximum may sit this far (base 2) below the row maximum
constexpr unsigned long long kDrainLimitNs = 100000000ull;

__device__ __forceinline__ uint32_t barp(uint32_t base, int i) { return base + kOffBar + 8u * i; }
__device__ __forceinline__ uint32_t ring_parity(int t) { return static_cast<uint32_t>(t / kRing) & 1u; }
__device__ __forceinline__ uint32_t qring_parity(int k) { return static_cast<uint32_t>(k / kQRing) & 1u; }

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

// Cosines and sines of eight pairs' angles, packed two pairs per register:
// c[i] = (cos, cos) of pairs 2i, 2i + 1; s[i] the sines; ns[i] = -s[i].
struct Angles8 {
    uint64_t c[4], s[4], ns[4];
};

// Rotate the pairs (x[m], x[m + 32]) of the chunk pair j by the angles in
// `an`: x' = x cos - z sin, z' = z cos + x sin (fp32), and store the two
// chunks back.
__device__ __forceinline__ void pair_rotate_store(uint32_t row_addr, int r, int j, const PairChunks &v,
                                                  const Angles8 &an)
{
    uint32_t ya[4], yb[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint64_t x = bf16x2_to_f2(v.x[i]), z = bf16x2_to_f2(v.z[i]);
        ya[i] = f2_to_bf16x2(ffma2(z, an.ns[i], fmul2(x, an.c[i])));
        yb[i] = f2_to_bf16x2(ffma2(z, an.c[i], fmul2(x, an.s[i])));
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

    // First unit u; without a work list its sequence, block, first row and
    // length are given (found by the range search).
    __device__ void start(const int32_t *cu_, const int2 *work_, int G_, long long u, const int (&first)[4])
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
            row0 = cu[seq];
            L = cu[seq + 1] - row0;
        } else {
            seq = first[0];
            qb = first[1];
            row0 = first[2];
            L = first[3];
        }
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
attn_local_kernel(const __grid_constant__ CUtensorMap tm_qkv, const __grid_constant__ CUtensorMap tm_out,
                  const __grid_constant__ RopeConsts rope,
                  const int32_t *__restrict__ cu, int n_seqs, long long T, int max_seqlen,
                  const int2 *__restrict__ work, const int32_t *__restrict__ work_count, int hw,
                  __nv_bfloat16 *__restrict__ out, int32_t *err)
{
    pdl_wait();
    extern __shared__ uint8_t smem_raw[];
    __shared__ long long s_range[2];
    __shared__ int s_g;
    __shared__ int s_first[4];       // first unit: sequence, block, first row, length
    __shared__ uint32_t s_tmem;
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    // ---- setup, in parallel: warp 0 finds this CTA's range [u_lo, u_hi) of
    // the heads x G units; warp 1 allocates TMEM and writes the band mask
    // tables; warp 2 initialises the barriers.
    if (warp == 0) {
        int G = 0, seq0 = 0, qb0 = 0, row00 = 0, L0 = 0;
        long long lo = 0, hi = 0;
        if (work) {
            G = *work_count;
        } else if (n_seqs <= 32) {
            // one sequence per lane: check, count and locate in one pass
            int c0 = 0, c1 = 0;
            if (lane < n_seqs) {
                c0 = cu[lane];
                c1 = cu[lane + 1];
            }
            const int Ls = c1 - c0;
            int bad = 0;
            if (lane < n_seqs) {
                if (Ls < 0)
                    bad |= kErrBadCu;
                else if (Ls > max_seqlen)
                    bad |= kErrTooLong;
            }
            if ((lane == 0 && c0 != 0) || (lane == n_seqs - 1 && static_cast<long long>(c1) != T))
                bad |= kErrBadCu;
            const int nb = (lane < n_seqs && Ls > 0) ? (Ls + kBlockM - 1) / kBlockM : 0;
            int incl = nb;
#pragma unroll
            for (int d = 1; d < 32; d <<= 1) {
                const int v = __shfl_up_sync(0xffffffffu, incl, d);
                if (lane >= d)
                    incl += v;
            }
#pragma unroll
            for (int d = 16; d > 0; d >>= 1)
                bad |= __shfl_xor_sync(0xffffffffu, bad, d);
            G = __shfl_sync(0xffffffffu, incl, 31);
            if (bad) {
                if (blockIdx.x == 0 && lane == 0)
                    atomicOr(err, bad);
                G = -1;
            } else if (G > 0) {
                const long long U = static_cast<long long>(kHeads) * G;
                lo = U * blockIdx.x / gridDim.x;
                hi = U * (blockIdx.x + 1) / gridDim.x;
                const int e0 = static_cast<int>(lo % G), excl = incl - nb;
                const unsigned hit = __ballot_sync(0xffffffffu, nb > 0 && e0 >= excl && e0 < excl + nb);
                const int src = hit ? __ffs(hit) - 1 : 0;
                seq0 = src;
                qb0 = e0 - __shfl_sync(0xffffffffu, excl, src);
                row00 = __shfl_sync(0xffffffffu, c0, src);
                L0 = __shfl_sync(0xffffffffu, Ls, src);
            }
        } else {
            G = count_blocks(cu, n_seqs, T, max_seqlen, err);
            if (G > 0) {
                const long long U = static_cast<long long>(kHeads) * G;
                lo = U * blockIdx.x / gridDim.x;
                hi = U * (blockIdx.x + 1) / gridDim.x;
                if (lo < hi) {
                    locate_block(cu, n_seqs, static_cast<int>(lo % G), seq0, qb0);
                    row00 = cu[seq0];
                    L0 = cu[seq0 + 1] - row00;
                }
            }
        }
        if (work && G > 0) {
            const long long U = static_cast<long long>(kHeads) * G;
            lo = U * blockIdx.x / gridDim.x;
            hi = U * (blockIdx.x + 1) / gridDim.x;
        }
        if (lane == 0) {
            s_range[0] = lo;
            s_range[1] = hi;
            s_g = G;
            s_first[0] = seq0;
            s_first[1] = qb0;
            s_first[2] = row00;
            s_first[3] = L0;
        }
    } else if (warp == 1) {
        tmem_alloc(smem_u32(&s_tmem), kTmemCols);
        tmem_relinquish();
        // The band's edge chunks: in the first window chunk of its rows,
        // lane l keeps keys k >= l; in the last, k <= l.  As additive masks
        // (0 keeps, -inf drops), row l of each table, 16-byte chunk c at
        // c ^ (l % 8).
        const float ninf = -INFINITY;
#pragma unroll
        for (int t = 0; t < 2; ++t)
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                float b[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int kx = 4 * c + e;
                    b[e] = (t == 0 ? kx >= lane : kx <= lane) ? 0.f : ninf;
                }
                asm volatile("st.shared.v4.f32 [%0], {%1,%2,%3,%4};"
                             :: "r"(base + kOffBias + t * 4096 + lane * 128 + ((c ^ (lane & 7)) << 4)),
                                "f"(b[0]), "f"(b[1]), "f"(b[2]), "f"(b[3]) : "memory");
            }
    } else if (tid == 64) {
        tma_prefetch_desc(&tm_qkv);
        tma_prefetch_desc(&tm_out);
        for (int i = 0; i < kNumBars; ++i) {
            uint32_t count = 1;
            if ((i >= kBarKE && i < kBarKE + kRing) || (i >= kBarVE && i < kBarVE + kRing))
                count = 2;
            if ((i >= kBarQR && i < kBarKR + kRing) || i == kBarP || i == kBarP + 1 ||
                i == kBarFree || i == kBarFree + 1 || i == kBarStg || i == kBarStg + 1)
                count = kGroupThreads;
            mbar_init(barp(base, i), count);
        }
        fence_mbar_init();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const long long u_lo = s_range[0];
    const int nunits = static_cast<int>(s_range[1] - u_lo);
    if (nunits <= 0) {
        if (warp == 1)
            tmem_dealloc(s_tmem, kTmemCols);
        return;
    }
    const int G = s_g;
    int first[4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
        first[i] = s_first[i];
    const uint32_t tmem = s_tmem;

    if (warp >= kWarpProducer) {
        if (warp == kWarpProducer) {
            // ------------------------------------------------------ producer
            Walker w;
            w.start(cu, work, G, u_lo, first);
            const uint64_t once = l2_policy_evict_first();
            int nq = 0, tk = 0, tv = 0;   // tiles issued per ring (issued in index order)
            bool ok = true;
            // wait for the ring slot of tile t, then TMA the 128 x 64 box at
            // (column x, row y) into it
            auto load = [&](uint32_t ring_off, int nslots, int bar_full, int bar_empty, int t, int x, int y,
                            int &issued) {
                if (!ok)
                    return;
                const int sl = t % nslots;
                const uint32_t par = static_cast<uint32_t>(t / nslots) & 1u;
                if (!(ok = mbar_wait(barp(base, bar_empty + sl), par ^ 1u, err)))
                    return;
                if (elect_one_sync()) {
                    mbar_arrive_expect_tx(barp(base, bar_full + sl), kTileBytes);
                    tma_load_2d_hint(base + ring_off + sl * kTileBytes, &tm_qkv, x, y,
                                     barp(base, bar_full + sl), once);
                }
                __syncwarp();
                issued = t + 1;
            };
            // Q and K of unit k (needed first, by RoPE), then the V tiles of
            // unit k - 1 (needed last, by P V); unit k is only started once the
            // Q tile of unit k - 2 has landed, so that at the start every SM's
            // first tiles are not queued behind a burst of prefetches.
            int tc = 0, a_prev = 0, colV_prev = 0, r0_prev = 0;
            bool fresh_prev = false;
            for (int k = 0; k < nunits && ok; ++k) {
                const int a = w.fresh ? tc : tc - 1;
                tc = a + 2;
                const int colQ = w.head * kHeadDim, colK = kHidden + colQ, colV = 2 * kHidden + colQ;
                const int r0 = w.row0 + w.qb * kBlockM;
                if (k >= 2)
                    ok = mbar_wait(barp(base, kBarQF + (k - 2) % kQRing), qring_parity(k - 2), err);
                if (w.fresh)
                    load(kOffK, kRing, kBarKF, kBarKE, a, colK, r0 - 64, tk);
                // the unit's record for the compute group, published with its Q
                // tile (the slot is free once the Q slot is: S of unit k - 3 done)
                if (ok && mbar_wait(barp(base, kBarQE + k % kQRing), qring_parity(k) ^ 1u, err)) {
                    if (lane == 0) {
                        const uint32_t rec = base + kOffRec + (k % kQRing) * 32;
                        asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};"
                                     :: "r"(rec), "r"(w.row0), "r"(w.L), "r"(w.qb * kBlockM), "r"(w.head) : "memory");
                        asm volatile("st.shared.v2.b32 [%0], {%1,%2};"
                                     :: "r"(rec + 16), "r"(w.fresh ? 1 : 0), "r"(a) : "memory");
                    }
                    __syncwarp();
                } else {
                    ok = false;
                }
                load(kOffQ, kQRing, kBarQF, kBarQE, k, colQ, r0, nq);
                load(kOffK, kRing, kBarKF, kBarKE, a + 1, colK, r0 + 64, tk);
                if (k >= 1) {
                    if (fresh_prev)
                        load(kOffV, kRing, kBarVF, kBarVE, a_prev, colV_prev, r0_prev - 64, tv);
                    load(kOffV, kRing, kBarVF, kBarVE, a_prev + 1, colV_prev, r0_prev + 64, tv);
                }
                a_prev = a;
                fresh_prev = w.fresh;
                colV_prev = colV;
                r0_prev = r0;
                if (k + 1 < nunits)
                    w.next();
            }
            if (fresh_prev)
                load(kOffV, kRing, kBarVF, kBarVE, a_prev, colV_prev, r0_prev - 64, tv);
            load(kOffV, kRing, kBarVF, kBarVE, a_prev + 1, colV_prev, r0_prev + 64, tv);
            // every copy issued has landed before the CTA can exit
            for (int t = max(0, nq - kQRing); t < nq; ++t)
                mbar_wait(barp(base, kBarQF + t % kQRing), qring_parity(t), err, kDrainLimitNs);
            for (int t = max(0, tk - kRing); t < tk; ++t)
                mbar_wait(barp(base, kBarKF + t % kRing), ring_parity(t), err, kDrainLimitNs);
            for (int t = max(0, tv - kRing); t < tv; ++t)
                mbar_wait(barp(base, kBarVF + t % kRing), ring_parity(t), err, kDrainLimitNs);
        } else if (warp == kWarpMma || warp == kWarpMma + 1) {
            // ------------------------------------------------------ MMA issuers
            Walker w;
            w.start(cu, work, G, u_lo, first);
            const int g = warp - kWarpMma;
            const uint32_t tm = tmem + g * kGroupCols;
            bool ok = true;
            int tc = 0;
            bool fresh = w.fresh;
            // Each unit gives every K and V tile it uses one release; a tile that
            // has no second user (tile 0 of a fresh unit, tile 1 when the next
            // unit is fresh or there is none) gets both releases from it.
            for (int k = 0; k < nunits && ok; ++k) {
                const int a = fresh ? tc : tc - 1;
                tc = a + 2;
                bool fresh_next = true;
                if (k + 1 < nunits) {
                    w.next();
                    fresh_next = w.fresh;
                }
                if ((k & 1) == g) {
                    const int j = k >> 1;
                    ok = mbar_wait(barp(base, kBarQR + k % kQRing), qring_parity(k), err) &&
                         mbar_wait(barp(base, kBarKR + a % kRing), ring_parity(a), err) &&
                         mbar_wait(barp(base, kBarKR + (a + 1) % kRing), ring_parity(a + 1), err) &&
                         (j == 0 || mbar_wait(barp(base, kBarFree + g), static_cast<uint32_t>(j - 1) & 1u, err));
                    if (!ok)
                        break;
                    __syncwarp();
                    tc_fence_after();
                    const uint32_t q = base + kOffQ + (k % kQRing) * kTileBytes;
    #pragma unroll
                    for (int t = 0; t < 2; ++t) {
                        const uint32_t kt = base + kOffK + ((a + t) % kRing) * kTileBytes;
    #pragma unroll
                        for (int kk = 0; kk < kHeadDim / 16; ++kk)
                            mma_bf16_ss_warp(tm + 128 * t, make_sdesc_sw128(q + 32 * kk, 16, 1024),
                                             make_sdesc_sw128(kt + 32 * kk, 16, 1024), kIdescS, kk > 0);
                    }
                    mma_commit_warp(barp(base, kBarS + g));
                    mma_commit_warp(barp(base, kBarQE + k % kQRing));
                    mma_commit_warp(barp(base, kBarKE + a % kRing));
                    mma_commit_warp(barp(base, kBarKE + (a + 1) % kRing));
                    if (fresh)
                        mma_commit_warp(barp(base, kBarKE + a % kRing));
                    if (fresh_next)
                        mma_commit_warp(barp(base, kBarKE + (a + 1) % kRing));

                    ok = mbar_wait(barp(base, kBarP + g), static_cast<uint32_t>(j) & 1u, err) &&
                         mbar_wait(barp(base, kBarVF + a % kRing), ring_parity(a), err) &&
                         mbar_wait(barp(base, kBarVF + (a + 1) % kRing), ring_parity(a + 1), err);
                    if (!ok)
                        break;
                    __syncwarp();
                    tc_fence_after();
    #pragma unroll
                    for (int t = 0; t < 2; ++t) {
                        const uint32_t v = base + kOffV + ((a + t) % kRing) * kTileBytes;
    #pragma unroll
                        for (int kk = 0; kk < kBlockN / 16; ++kk)
                            mma_bf16_ts_warp(tm + kColO, tm + 128 * t + 8 * kk,
                                             make_sdesc_sw128(v + 2048 * kk, 1024, 1024), kIdescO,
                                             (t > 0 || kk > 0) ? 1u : 0u);
                    }
                    mma_commit_warp(barp(base, kBarO + g));
                    mma_commit_warp(barp(base, kBarVE + a % kRing));
                    mma_commit_warp(barp(base, kBarVE + (a + 1) % kRing));
                    if (fresh)
                        mma_commit_warp(barp(base, kBarVE + a % kRing));
                    if (fresh_next)
                        mma_commit_warp(barp(base, kBarVE + (a + 1) % kRing));
                }
                fresh = fresh_next;
            }
            // every MMA issued has completed before TMEM is released
            mma_commit_warp(barp(base, kBarDrain + g));
            mbar_wait(barp(base, kBarDrain + g), 0, err, kDrainLimitNs);
        }
    } else {
        // ------------------------------------------------------ compute groups
        // Warp q of group g (warp 4g + q): TMEM lane quadrant q, rows
        // 32q .. 32q + 31, one row per thread.
        const int g = warp >> 2, q = warp & 3;
        const int r = 32 * q + lane;                  // row in the block, TMEM lane
        const uint32_t tm = tmem + g * kGroupCols + (static_cast<uint32_t>(32 * q) << 16);
        const uint32_t stage = base + kOffStage + g * kTileBytes;
        // the group's previous unit, whose epilogue runs after the next
        // unit's RoPE (while its P V product is on the tensor cores): its
        // rows, block and head in shared memory, its row sum in p_sum
        const uint32_t prev = base + kOffPrev + g * 16;
        const bool lead = r == 0;                     // issues the group's TMA stores
        bool ok = true;
        int j = 0, nst = 0;                           // units done; staged (TMA-stored) epilogues
        float p_sum = 0.f;

        // out = O / l.  A full block goes through the group's staging tile
        // and one TMA store; a block that runs past its sequence end stores
        // its rows directly (rows past the end are not written).
        auto epilogue = [&](int jp) -> bool {
            // P of the unit complete (its record is visible) and O = P V ready
            if (!(mbar_wait(barp(base, kBarP + g), static_cast<uint32_t>(jp) & 1u, err) &&
                  mbar_wait(barp(base, kBarO + g), static_cast<uint32_t>(jp) & 1u, err)))
                return false;
            __syncwarp();
            tc_fence_after();
            uint32_t o[2][32];
            tmem_ld32(tm + kColO, o[0]);
            tmem_ld32(tm + kColO + 32, o[1]);
            int row0, q0, L, head;
            asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];"
                         : "=r"(row0), "=r"(q0), "=r"(L), "=r"(head) : "r"(prev) : "memory");
            tmem_wait_ld();
            reg_fence32(o[0]);
            reg_fence32(o[1]);
            tc_fence_before();
            mbar_arrive(barp(base, kBarFree + g));     // the group's TMEM may be reused
            const int p_row = q0 + r < L ? row0 + q0 + r : -1;
            const int p_col = head * kHeadDim;
            const int p_blk = q0 + kBlockM <= L ? row0 + q0 : -1;     // a full block
            const float inv = p_sum > 0.f ? 1.f / p_sum : 0.f;
            uint32_t w4[8][4];
#pragma unroll
            for (int c = 0; c < 8; ++c)
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    w4[c][e] = pack_bf16x2(__uint_as_float(o[c / 4][8 * (c % 4) + 2 * e]) * inv,
                                           __uint_as_float(o[c / 4][8 * (c % 4) + 2 * e + 1]) * inv);
            if (p_blk >= 0) {
                const uint32_t par = static_cast<uint32_t>(nst) & 1u;
                ++nst;
                if (lead) {
                    bulk_wait_read0();                  // the previous store has left the tile
                    mbar_arrive(barp(base, kBarStgFree + g));
                }
                if (!mbar_wait(barp(base, kBarStgFree + g), par, err))
                    return false;
#pragma unroll
                for (int c = 0; c < 8; ++c)
                    asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};"
                                 :: "r"(stage + r * 128 + ((c ^ (r & 7)) << 4)),
                                    "r"(w4[c][0]), "r"(w4[c][1]), "r"(w4[c][2]), "r"(w4[c][3]) : "memory");
                fence_proxy_async_smem();
                mbar_arrive(barp(base, kBarStg + g));
                if (lead) {
                    if (!mbar_wait(barp(base, kBarStg + g), par, err))
                        return false;
                    tma_store_2d(&tm_out, stage, p_col, p_blk);
                    bulk_commit();
                }
            } else if (p_row >= 0) {
                uint4 *dst = reinterpret_cast<uint4 *>(out + static_cast<long long>(p_row) * kHidden + p_col);
#pragma unroll
                for (int c = 0; c < 8; ++c)
                    dst[c] = make_uint4(w4[c][0], w4[c][1], w4[c][2], w4[c][3]);
            }
            return true;
        };

#pragma unroll 1
        for (int k = g; k < nunits && ok; k += 2) {
            // ---- the unit's record (published with its Q tile)
            if (!(ok = mbar_wait(barp(base, kBarQF + k % kQRing), qring_parity(k), err)))
                break;
            const uint32_t rec = base + kOffRec + (k % kQRing) * 32;
            int row0, L, q0, head, fresh_i, a;
            asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];"
                         : "=r"(row0), "=r"(L), "=r"(q0), "=r"(head) : "r"(rec) : "memory");
            asm volatile("ld.shared.v2.b32 {%0,%1}, [%2];" : "=r"(fresh_i), "=r"(a) : "r"(rec + 16) : "memory");
            const bool fresh = fresh_i != 0;

            // ---- RoPE.  Thread r takes position p = q0 + 64 + r: K tile 1
            // row r, and the Q row at p (r + 64, for r < 64) or at p - 128
            // (r - 64, for r >= 64), and on a fresh unit K tile 0 row r (at
            // p - 128).  cos/sin at p - 128 come from those at p by one
            // rotation of -128 positions.
            ok = mbar_wait(barp(base, kBarKF + (a + 1) % kRing), ring_parity(a + 1), err) &&
                 (!fresh || mbar_wait(barp(base, kBarKF + a % kRing), ring_parity(a), err));
            if (ok) {
                const uint32_t qs = base + kOffQ + (k % kQRing) * kTileBytes;
                const uint32_t k0s = base + kOffK + (a % kRing) * kTileBytes;
                const uint32_t k1s = base + kOffK + ((a + 1) % kRing) * kTileBytes;
                const uint32_t p = static_cast<uint32_t>(q0 + 64 + r);
                const bool q_at_p = r < 64;          // warp-uniform
                const int qr = q_at_p ? r + 64 : r - 64;
#pragma unroll 1
                for (int jj = 0; jj < 4; ++jj) {
                    // the rows' chunks first (one shared-memory round trip),
                    // then the angles, then rotate and store
                    PairChunks vk1, vq, vk0;
                    pair_load(k1s + r * 128, r, jj, vk1);
                    pair_load(qs + qr * 128, qr, jj, vq);
                    if (fresh)
                        pair_load(k0s + r * 128, r, jj, vk0);
                    Angles8 an;                       // at p
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        float c0, s0, c1, s1;
                        pos_cos_sin(p, rope.frac_hi[8 * jj + 2 * i], rope.frac_lo[8 * jj + 2 * i], c0, s0);
                        pos_cos_sin(p, rope.frac_hi[8 * jj + 2 * i + 1], rope.frac_lo[8 * jj + 2 * i + 1], c1, s1);
                        an.c[i] = f2(c0, c1);
                        an.s[i] = f2(s0, s1);
                        an.ns[i] = f2(-s0, -s1);
                    }
                    pair_rotate_store(k1s + r * 128, r, jj, vk1, an);
                    if (q_at_p)
                        pair_rotate_store(qs + qr * 128, qr, jj, vq, an);
                    if (fresh || !q_at_p) {
                        // now at p - 128 (one rotation by -128 w):
                        // c' = c cos + s sin, s' = s cos - c sin
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            const int m = 8 * jj + 2 * i;
                            const uint64_t c128 = f2(rope.cos128[m], rope.cos128[m + 1]);
                            const uint64_t s128 = f2(rope.sin128[m], rope.sin128[m + 1]);
                            const uint64_t c1 = ffma2(an.s[i], s128, fmul2(an.c[i], c128));
                            const uint64_t s1 = ffma2(an.c[i], f2(-rope.sin128[m], -rope.sin128[m + 1]),
                                                      fmul2(an.s[i], c128));
                            an.c[i] = c1;
                            an.s[i] = s1;
                            an.ns[i] = fmul2(s1, f2(-1.f, -1.f));
                        }
                        if (!q_at_p)
                            pair_rotate_store(qs + qr * 128, qr, jj, vq, an);
                        if (fresh)
                            pair_rotate_store(k0s + r * 128, r, jj, vk0, an);
                    }
                }
                fence_proxy_async_smem();
            }
            mbar_arrive(barp(base, kBarQR + k % kQRing));
            mbar_arrive(barp(base, kBarKR + (a + 1) % kRing));
            if (fresh)
                mbar_arrive(barp(base, kBarKR + a % kRing));
            if (!ok)
                break;

            if (j > 0 && !(ok = epilogue(j - 1)))
                break;

            // ---- softmax of the rows over the window chunks 32q .. 32q + 159
            const int i = q0 + r;
            // admitted keys [klo, khi]; none for rows past the sequence
            const int klo = i < L ? max(0, i - hw) : L, khi = min(L - 1, i + hw);
            // Keys outside [klo, khi] of window chunk e -> -inf, from a bit
            // mask of the admitted keys; needed only where a chunk meets a
            // sequence edge or the band is narrower.  The band's own edge
            // chunks (e = 0 and 4) take their masks from the lane tables.
            auto general = [&](int e) {
                const int key0 = q0 - 64 + 32 * (q + e);
                return hw != kBandReach || key0 < 0 || key0 + 31 >= L;
            };
            auto mask_bits = [&](uint32_t (&x)[32], int e) {
                const int key0 = q0 - 64 + 32 * (q + e);
                const int lo = klo - key0, hi = khi - key0;
                const uint32_t keep = (lo > 31 || hi < 0 || lo > hi) ? 0u
                    : ((0xFFFFFFFFu >> (31 - min(hi, 31))) & (0xFFFFFFFFu << max(lo, 0)));
#pragma unroll
                for (int kx = 0; kx < 32; ++kx)
                    x[kx] = (keep & (1u << kx)) ? x[kx] : __float_as_uint(-INFINITY);
            };
            if (!(ok = mbar_wait(barp(base, kBarS + g), static_cast<uint32_t>(j) & 1u, err)))
                break;
            __syncwarp();
            tc_fence_after();
            // The reference maximum m (base 2, scaled) is taken from window
            // chunk 2, which holds the diagonal key i of every row; p =
            // 2^(s * scale - m) is then written chunk by chunk in one pass.
            // Any reference within 2^kSlack of the row maximum gives the
            // same softmax up to rounding; a chunk whose exponents exceed
            // kSlack raises m by an integer and rescales the P already
            // written by that power of two (exact in bf16).
            uint32_t v[32];
            tmem_ld32(tm + 32 * (q + 2), v);
            tmem_wait_ld();
            reg_fence32(v);
            if (general(2))
                mask_bits(v, 2);
            float m = max32(v) * kScaleLog2;
            float s0 = 0.f, s1 = 0.f;
#pragma unroll 1
            for (int e = 0; e < 5; ++e) {
                tmem_ld32(tm + 32 * (q + e), v);
                tmem_wait_ld();
                reg_fence32(v);
                const float m_use = m == -INFINITY ? 0.f : m;
                // exponents y = s * scale - m (+ the lane's edge mask)
                if (general(e)) {
                    mask_bits(v, e);
#pragma unroll
                    for (int kx = 0; kx < 16; ++kx) {
                        float x0 = __uint_as_float(v[2 * kx]), x1 = __uint_as_float(v[2 * kx + 1]);
                        ffma2_bc(x0, x1, kScaleLog2, -m_use);
                        v[2 * kx] = __float_as_uint(x0);
                        v[2 * kx + 1] = __float_as_uint(x1);
                    }
                } else if (e == 0 || e == 4) {
                    const uint32_t tab = base + kOffBias + (e == 4 ? 4096 : 0) + lane * 128;
#pragma unroll
                    for (int c = 0; c < 8; ++c) {
                        float b[4];
                        asm volatile("ld.shared.v4.f32 {%0,%1,%2,%3}, [%4];"
                                     : "=f"(b[0]), "=f"(b[1]), "=f"(b[2]), "=f"(b[3])
                                     : "r"(tab + ((c ^ (lane & 7)) << 4)));
#pragma unroll
                        for (int t = 0; t < 2; ++t) {
                            const uint64_t y = ffma2(f2(__uint_as_float(v[4 * c + 2 * t]), __uint_as_float(v[4 * c + 2 * t + 1])),
                                                     f2(kScaleLog2, kScaleLog2),
                                                     f2(b[2 * t] - m_use, b[2 * t + 1] - m_use));
                            float y0, y1;
                            f2_split(y, y0, y1);
                            v[4 * c + 2 * t] = __float_as_uint(y0);
                            v[4 * c + 2 * t + 1] = __float_as_uint(y1);
                        }
                    }
                } else {
#pragma unroll
                    for (int kx = 0; kx < 16; ++kx) {
                        float x0 = __uint_as_float(v[2 * kx]), x1 = __uint_as_float(v[2 * kx + 1]);
                        ffma2_bc(x0, x1, kScaleLog2, -m_use);
                        v[2 * kx] = __float_as_uint(x0);
                        v[2 * kx + 1] = __float_as_uint(x1);
                    }
                }
                const float ymax = max32(v);
                if (__any_sync(0xffffffffu, ymax > kSlack)) {
                    // raise m by the integer d = ceil(ymax) (0 in lanes that
                    // need no change) and rescale this chunk's exponents, the
                    // P already written and the sums by f = 2^-d, built from
                    // its exponent bits: multiplying a bf16 P by f is exact,
                    // so nothing already written is rounded again.  Past
                    // d = 126 the scaled P would be below 2^-62 of the new
                    // maximum; it is flushed to 0.
                    const float d = ymax > kSlack ? fminf(ceilf(ymax), 1024.f) : 0.f;
                    const int di = static_cast<int>(d);
                    const float f = di <= 126 ? __int_as_float((127 - di) << 23) : 0.f;
                    tmem_wait_st();
#pragma unroll 1
                    for (int e2 = 0; e2 < e; ++e2) {
                        const int col2 = 32 * (q + e2);
                        const uint32_t pa = tm + col2 / 2 + (col2 >= 128 ? 64 : 0);
                        uint32_t pv[16];
                        tmem_ld16(pa, pv);
                        tmem_wait_ld();
#pragma unroll
                        for (int kx = 0; kx < 16; ++kx)
                            pv[kx] = pack_bf16x2(bf16lo_to_f32(pv[kx]) * f, bf16hi_to_f32(pv[kx]) * f);
                        tmem_st16(pa, pv);
                    }
#pragma unroll
                    for (int kx = 0; kx < 32; ++kx)
                        v[kx] = __float_as_uint(__uint_as_float(v[kx]) - d);
                    s0 *= f;
                    s1 *= f;
                    m = m_use + d;
                }
                uint32_t pk[16];
#pragma unroll
                for (int kx = 0; kx < 16; ++kx) {
                    const float p0 = ex2_approx(__uint_as_float(v[2 * kx]));
                    const float p1 = ex2_approx(__uint_as_float(v[2 * kx + 1]));
                    fadd2(s0, s1, p0, p1);
                    pk[kx] = pack_bf16x2(p0, p1);
                }
                // P chunk of window column c sits at c / 2 (+ 64 in tile 1):
                // below every S column not yet read
                const int col = 32 * (q + e);
                tmem_st16(tm + col / 2 + (col >= 128 ? 64 : 0), pk);
            }
            {
                uint32_t z[16];
#pragma unroll
                for (int kx = 0; kx < 16; ++kx)
                    z[kx] = 0u;
                // P = 0 over tile 0's chunks left of the rows' window and
                // tile 1's chunks right of it
                for (int c = 0; c < q; ++c)
                    tmem_st16(tm + 16 * c, z);
                for (int c = q + 1; c < 4; ++c)
                    tmem_st16(tm + 128 + 16 * c, z);
            }
            p_sum = s0 + s1;
            if (lead)
                asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};"
                             :: "r"(prev), "r"(row0), "r"(q0), "r"(L), "r"(head) : "memory");
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(barp(base, kBarP + g));
            ++j;
        }
        if (ok && j > 0)
            epilogue(j - 1);
        if (lead)
            bulk_wait0();                               // this group's stores have completed
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
    pdl_trigger();
}

}  // namespace

cudaError_t launch_attn_local(const LocalArgs &a, cudaStream_t stream)
{
    static PerDeviceOnce smem_once;
    cudaError_t e = smem_opt_in(smem_once, attn_local_kernel, kSmemBytes);
    if (e != cudaSuccess)
        return e;
    const long long units = static_cast<long long>(a.block_bound) * kHeads;
    const long long grid = units < a.num_ctas ? units : a.num_ctas;
    if (grid <= 0)
        return cudaSuccess;
    return launch_chained(attn_local_kernel, dim3(static_cast<unsigned>(grid)), dim3(kThreads), kSmemBytes, stream,
        a.tm_qkv, a.tm_out, a.rope, a.cu, a.n_seqs, a.T, a.max_seqlen, a.work, a.work_count,
        a.half_window, a.out, a.err);
}

}  // namespace mbert
