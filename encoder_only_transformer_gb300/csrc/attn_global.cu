// Global-layer attention over pre-rotated Q/K: a persistent, warp-specialised
// tcgen05 pipeline for sm_103a.
//
// Work: a unit is (work entry, head), an entry being 256 query rows of one
// sequence; a unit needs ceil(L/128) key tiles.  All (unit, key tile)
// iterations, in work-list order, are split into contiguous ranges, one per
// persistent CTA (one CTA per SM), of equal cost whatever the number of
// units: a range's cost is its iterations plus kSegCost for each unit that
// starts inside it (each extra segment costs a Q load, an epilogue and a
// pipeline refill).  A CTA walks its range as a
// sequence of segments (a unit and a run of its key tiles).  A segment that
// covers its whole unit writes the output directly; a unit cut between CTAs
// leaves one partial state (unnormalised O, row maximum, row sum) per
// segment in a workspace, and whichever CTA completes the unit's last
// segment (an atomic counter per unit decides) merges them, always in CTA
// order, so results are reproducible run to run.  No CTA ever waits for
// another.  (Where a unit is cut depends on the whole batch, so adding a
// sequence to a pack can change another sequence's outputs by rounding.)
//
// CTA (12 warps):
//   warps 0-3   softmax group 0 (query tile 0 of the entry, TMEM lanes 0..127)
//   warps 4-7   softmax group 1 (query tile 1)
//   warp  8     TMA producer: Q tiles (double-buffered per segment), K and V
//               through 3-stage rings
//   warps 9,10  MMA issuers, one per query tile (whole warp runs the loop;
//               one elected lane issues): S_w = Q_w K^T, O_w += P_w V
//   warp  11    per segment, stages the score bound's inputs in shared
//               memory: the norms of the segment's 256 rotated Q rows and the
//               largest rotated K row norm of the head over the sequence
// TMEM (512 columns): S0 [0,128) S1 [128,256) P0 [256,320) P1 [320,384)
// O0 [384,448) O1 [448,512); fp32 except P (bf16 pairs).
//
// Arithmetic ("ModernBERT-base Architecture Teardown", "How Does
// Self-Attention Work?"): scores q.k / 8, softmax over every key of the
// sequence (a global layer, "What Are Local and Global Attention?"), output
// the weighted blend of V.  The softmax is online in base 2; the reference
// maximum only moves (and O is rescaled) when a tile's maximum exceeds it by
// more than 8, so O and the row sum always share one reference.  Partial
// states over disjoint key ranges are merged exactly:
// m = max(m_a, m_b), O = O_a 2^(m_a - m) + O_b 2^(m_b - m), likewise l.
// The reference may sit below a row's true maximum by any amount for which
// 2^(score - reference) stays finite in the fp32 sums.  By Cauchy-Schwarz
// every score of a row is at most |q| max|k| / 8 (norms of the rotated
// rows, from the RoPE pass; the key maximum over the sequence).  After a
// segment's second tile, a warp whose 32 rows all have that bound within
// kSkipSlack (base 2) of their reference runs the segment's later tiles
// without a row maximum and keeps its reference (weights up to 2^32).
#include <type_traits>

#include "common.cuh"
#include "internal.h"

namespace mbert {
namespace {

constexpr int kThreads = 384;
constexpr int kRegsSoftmax = 216;   // 4 x 72 + 8 x 216 = 12 x 168 (the launch budget)
constexpr int kRegsControl = 72;
constexpr int kStages = 3;

constexpr uint32_t kOffQ = 0;                                  // 2 sets of (Q0, Q1)
constexpr uint32_t kOffK = 4 * kTileBytes;                     // K ring
constexpr uint32_t kOffV = kOffK + kStages * kTileBytes;       // V ring
constexpr uint32_t kOffBar = kOffV + kStages * kTileBytes;     // 163840
constexpr uint32_t kNormSlotBytes = 4 * (2 * kBlockM + 4);    // 256 Q norms, max |k|, padding
constexpr uint32_t kOffNorm = kOffBar + 512;                   // 2 slots of the score bound's inputs
constexpr uint32_t kSmemBytes = kOffNorm + 2 * kNormSlotBytes + 1024;

// barrier slots (8 bytes each) from kOffBar
constexpr int kBarQFull = 0;      // + set (2)
constexpr int kBarQEmpty = 2;     // + set
constexpr int kBarKFull = 4;      // + stage (3)
constexpr int kBarKEmpty = 7;
constexpr int kBarVFull = 10;
constexpr int kBarVEmpty = 13;
constexpr int kBarSFull = 16;     // + group (2)
constexpr int kBarSEmpty = 18;
constexpr int kBarPFull = 20;
constexpr int kBarODone = 22;
constexpr int kBarOFree = 24;
constexpr int kBarSegSync = 26;   // all 256 softmax threads wrote their partial rows
constexpr int kBarSegFlag = 27;   // the counter result is in shared memory
constexpr int kBarEarly = 28;     // the early look at the last segment's unit is in shared memory
constexpr int kBarNormFull = 29;  // + slot (2): a segment's bound inputs staged
constexpr int kBarNormEmpty = 31; // + slot: read by all 256 softmax threads
constexpr int kNumBars = 33;
constexpr uint32_t kOffSlot = kOffBar + 8 * kNumBars;          // TMEM address
constexpr uint32_t kOffFlag = kOffSlot + 8;                    // "I merge" flag
constexpr uint32_t kOffEarly = kOffFlag + 4;                   // early-look result

constexpr uint32_t kTmemCols = 512;
__host__ __device__ constexpr uint32_t col_s(int w) { return 128u * w; }
__host__ __device__ constexpr uint32_t col_p(int w) { return 256u + 64u * w; }
__host__ __device__ constexpr uint32_t col_o(int w) { return 384u + 64u * w; }

constexpr uint32_t kIdescS = make_idesc_bf16(128, 128, false);
constexpr uint32_t kIdescO = make_idesc_bf16(128, 64, true);
constexpr float kScaleLog2 = 0.125f * 1.4426950408889634f;
constexpr float kRescaleThreshold = 8.0f;
// Largest exponent (base 2) a weight may take when the row maximum is
// skipped: weights up to 2^32 keep the row sums of 2^31 keys (2^63) and the
// P V sums of values below 2^60 finite in fp32.
constexpr float kSkipSlack = 32.0f;
// Relative margin on the bound for the fp32 rounding of the norms and of the
// tensor-core sums (each far below 2^-16 relative).
constexpr float kBoundMargin = 1.0f + 1.0f / 1024.0f;
// Cost of a segment's fixed work (Q load, epilogue, pipeline refill) in key
// tile iterations, for the split of the iterations among CTAs.
constexpr int kSegCost = 4;

// ---------------------------------------------------------------- schedule
struct Params {
    const int32_t *cu;
    const int2 *work;
    const int32_t *tile_start;   // [entries + 1]
    int32_t *unit_cnt;
    float *partials;
    __nv_bfloat16 *out;
    int32_t *err;
    const float *norms;          // [12][norm_pitch]: rotated Q row norms per head
    const uint16_t *knorm;       // [12][norm_pitch]: rotated K row norms, fp16 rounded up
    long long norm_pitch;        // a multiple of 8
    long long rows;              // rows of qkv (norms exist for rows below)
    int entries;
    long long total;             // iterations of all units
    int ctas;
    int alpha;                   // cost of a unit start inside a range (kSegCost or 0)
    long long cost;              // total + alpha * (units - 1)
};

// The split is made in cost coordinates: iteration `it` of unit u sits at
// x = it + alpha * u, so each unit start adds alpha.  CTA c owns the
// iterations whose x lies in [x_lo(c), x_lo(c + 1)).
__device__ __forceinline__ long long x_lo(const Params &p, int c)
{
    return static_cast<long long>(c) * p.cost / p.ctas;
}

// The CTA whose range contains iteration `it` of unit `u`: the largest c
// with floor(c * cost / ctas) <= x.
__device__ __forceinline__ int cta_of(const Params &p, long long it, int u)
{
    const long long x = it + static_cast<long long>(p.alpha) * u;
    const long long c = ((x + 1) * p.ctas - 1) / p.cost;
    return c < p.ctas - 1 ? static_cast<int>(c) : p.ctas - 1;
}

// The first iteration at or after cost coordinate x, and the entry holding it
// (p.entries for x = cost, the end).  Entry e starts at x = tile_start[e] +
// alpha * heads * e; x values between two units map to the later unit's start.
__device__ long long iter_at(const Params &p, long long x, int &entry)
{
    const long long per = static_cast<long long>(p.alpha) * kHeads;
    // a guess as if all entries cost the same (exact for one sequence; two
    // independent loads), then a binary search on the side it missed
    int e = min(static_cast<int>((x * p.entries) / p.cost), p.entries - 1);
    long long t0 = p.tile_start[e], t1 = p.tile_start[e + 1];
    if (!(t0 + per * e <= x && x < t1 + per * (e + 1))) {
        int lo = 0, h = p.entries;
        while (h - lo > 1) {
            const int mid = (lo + h) >> 1;
            if (p.tile_start[mid] + per * mid <= x)
                lo = mid;
            else
                h = mid;
        }
        e = lo;
        t0 = p.tile_start[e];
        t1 = p.tile_start[e + 1];
    }
    const long long n = (t1 - t0) / kHeads;           // iterations of each unit of the entry
    const long long d = x - t0 - per * e;
    const long long h = min(static_cast<long long>(kHeads - 1), d / (n + p.alpha));
    const long long r = d - h * (n + p.alpha);
    entry = (r >= n && h == kHeads - 1) ? e + 1 : e;
    return t0 + h * n + (r < n ? r : n);
}

// A run of key tiles [kb, ke) of one unit.
struct Seg {
    int entry, head, kb, ke, ntiles;
    int row0, L, q0;
    long long ua;              // first iteration of the unit
};

// Walks the segments of one CTA's range [it, hi).
struct SegIter {
    long long it, hi;
    int entry;

    __device__ void init(const Params &p, int c)
    {
        int e_hi;
        it = iter_at(p, x_lo(p, c), entry);
        hi = iter_at(p, x_lo(p, c + 1), e_hi);
    }

    __device__ bool next(const Params &p, Seg &s)
    {
        if (it >= hi)
            return false;
        while (entry + 1 < p.entries && p.tile_start[entry + 1] <= it)
            ++entry;
        const int2 w = p.work[entry];
        s.entry = entry;
        s.row0 = p.cu[w.x];
        s.L = p.cu[w.x + 1] - s.row0;
        s.q0 = w.y * 2 * kBlockM;
        s.ntiles = (s.L + kBlockN - 1) / kBlockN;
        const long long off = it - p.tile_start[entry];
        s.head = static_cast<int>(off / s.ntiles);
        s.kb = static_cast<int>(off % s.ntiles);
        const long long left = hi - it;
        s.ke = static_cast<int>(left < s.ntiles - s.kb ? s.kb + left : s.ntiles);
        s.ua = p.tile_start[entry] + static_cast<long long>(s.head) * s.ntiles;
        it += s.ke - s.kb;
        return true;
    }
};

struct Ctx {
    uint32_t base;          // 1024-aligned shared address
    uint32_t tmem;
    uint8_t *sbase;         // generic pointer to the same address
};

__device__ __forceinline__ uint32_t bar(const Ctx &c, int i) { return c.base + kOffBar + 8u * i; }

// ---------------------------------------------------------------- producer
__device__ void producer(const Ctx &c, const Params &p, const CUtensorMap *tm_rot,
                         const CUtensorMap *tm_qkv, int cta)
{
    const uint64_t keep = l2_policy_evict_last();    // K/V: re-read by every query block
    const uint64_t once = l2_policy_evict_first();   // Q: read once
    SegIter si;
    si.init(p, cta);
    Seg s;
    uint32_t g = 0;          // key tiles issued by this CTA so far
    for (uint32_t sg = 0; si.next(p, s); ++sg) {
        const int qs = sg & 1;
        if (sg >= 2 && !mbar_wait(bar(c, kBarQEmpty + qs), ((sg >> 1) - 1) & 1, p.err))
            return;
        const int colQ = s.head * kHeadDim;
        const int colK = kHidden + s.head * kHeadDim;
        const int colV = 2 * kHidden + s.head * kHeadDim;
        const uint32_t qdst = c.base + kOffQ + qs * 2 * kTileBytes;
        mbar_arrive_expect_tx(bar(c, kBarQFull + qs), 2 * kTileBytes);
        tma_load_2d_hint(qdst, tm_rot, colQ, s.row0 + s.q0, bar(c, kBarQFull + qs), once);
        tma_load_2d_hint(qdst + kTileBytes, tm_rot, colQ, s.row0 + s.q0 + kBlockM,
                         bar(c, kBarQFull + qs), once);
        for (int k = s.kb; k < s.ke; ++k, ++g) {
            const int st = g % kStages;
            const uint32_t u = g / kStages;
            const int krow = s.row0 + k * kBlockN;
            if (u > 0 && !mbar_wait(bar(c, kBarKEmpty + st), (u - 1) & 1, p.err))
                return;
            mbar_arrive_expect_tx(bar(c, kBarKFull + st), kTileBytes);
            tma_load_2d_hint(c.base + kOffK + st * kTileBytes, tm_rot, colK, krow,
                             bar(c, kBarKFull + st), keep);
            if (u > 0 && !mbar_wait(bar(c, kBarVEmpty + st), (u - 1) & 1, p.err))
                return;
            mbar_arrive_expect_tx(bar(c, kBarVFull + st), kTileBytes);
            tma_load_2d_hint(c.base + kOffV + st * kTileBytes, tm_qkv, colV, krow,
                             bar(c, kBarVFull + st), keep);
        }
    }
}

// ---------------------------------------------------------------- MMA issuers
__device__ __forceinline__ void issue_s(const Ctx &c, int w, int qs, int st)
{
    const uint32_t q = c.base + kOffQ + (qs * 2 + w) * kTileBytes;
    const uint32_t k = c.base + kOffK + st * kTileBytes;
#pragma unroll
    for (int kk = 0; kk < kHeadDim / 16; ++kk)
        mma_bf16_ss_warp(c.tmem + col_s(w), make_sdesc_sw128(q + 32 * kk, 16, 1024),
                         make_sdesc_sw128(k + 32 * kk, 16, 1024), kIdescS, kk > 0);
}

__device__ __forceinline__ void issue_o(const Ctx &c, int w, int st, bool accumulate)
{
    const uint32_t v = c.base + kOffV + st * kTileBytes;
#pragma unroll
    for (int kk = 0; kk < kBlockN / 16; ++kk)
        mma_bf16_ts_warp(c.tmem + col_o(w), c.tmem + col_p(w) + 8 * kk,
                         make_sdesc_sw128(v + 2048 * kk, 1024, 1024), kIdescO,
                         (accumulate || kk > 0) ? 1u : 0u);
}

// Issuer for query tile w: per segment, S_w(t) for each key tile t, and
// O_w += P_w(t-1) V(t-1) one tile behind, so that S of the next tile is
// computed while the softmax group works on the current one.
__device__ void mma_issuer(const Ctx &c, const Params &p, int w, int cta)
{
    SegIter si;
    si.init(p, cta);
    Seg s;
    uint32_t g0 = 0;
    for (uint32_t sg = 0; si.next(p, s); ++sg) {
        const int qs = sg & 1;
        const int n = s.ke - s.kb;
        if (!mbar_wait(bar(c, kBarQFull + qs), (sg >> 1) & 1, p.err))
            return;
        for (int t = 0; t <= n; ++t) {
            if (t < n) {
                const uint32_t g = g0 + t;
                const int st = g % kStages;
                if (!mbar_wait(bar(c, kBarKFull + st), (g / kStages) & 1, p.err))
                    return;
                if (g > 0 && !mbar_wait(bar(c, kBarSEmpty + w), (g - 1) & 1, p.err))
                    return;
                // Query tile 1's S of a key tile only once group 0 has
                // loaded its own S of it: group 1 then trails group 0 by
                // about one TMEM load, so that their exponential loops
                // overlap less on the shared MUFU pipe than in lockstep.  Only
                // where the tile and the two after it belong to this segment:
                // group 0 may be up to two loads ahead (the K ring of 3 waits
                // for group 1's S), and the parity wait then stands for the
                // later phase, which group 0 reaches within the segment
                // without anything from group 1.  Across a segment end it
                // would wait on group 0's next segment, which waits on
                // group 1.
                if (w == 1 && t + 2 < n && !mbar_wait(bar(c, kBarSEmpty + 0), g & 1, p.err))
                    return;
                __syncwarp();
                tc_fence_after();
                issue_s(c, w, qs, st);
                mma_commit_warp(bar(c, kBarSFull + w));
                mma_commit_warp(bar(c, kBarKEmpty + st));
                if (t == n - 1)
                    mma_commit_warp(bar(c, kBarQEmpty + qs));
            }
            if (t > 0) {
                const uint32_t g = g0 + t - 1;
                const int st = g % kStages;
                if (!mbar_wait(bar(c, kBarVFull + st), (g / kStages) & 1, p.err))
                    return;
                if (!mbar_wait(bar(c, kBarPFull + w), g & 1, p.err))
                    return;
                if (t == 1 && sg > 0 && !mbar_wait(bar(c, kBarOFree + w), (sg - 1) & 1, p.err))
                    return;
                __syncwarp();
                tc_fence_after();
                issue_o(c, w, st, t > 1);
                mma_commit_warp(bar(c, kBarODone + w));
                mma_commit_warp(bar(c, kBarVEmpty + st));
            }
        }
        g0 += n;
    }
}

// ---------------------------------------------------------------- bound inputs
// Non-blocking look at a barrier phase (acquire when it is complete).
__device__ __forceinline__ bool mbar_test(uint32_t bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok) : "r"(bar), "r"(parity) : "memory");
    return ok != 0;
}
// The bounded wait out of line: the hot loop only calls it when the staged
// bound is late.
__device__ __noinline__ bool slow_wait(uint32_t bar, uint32_t parity, int *err)
{
    return mbar_wait(bar, parity, err);
}

// Warp 11: for each segment, into shared-memory slot sg % 2, the norms of
// the segment's 256 rotated Q rows (0 past the end of qkv, whose rows the
// tensor map fills with zeros) and the largest rotated K row norm of its
// head over the sequence (from fp16 norms rounded up; non-negative fp16
// values order like their bits, +inf and NaN above all finite ones).
__device__ void norm_stager(const Ctx &c, const Params &p, int lane, int cta)
{
    SegIter si;
    si.init(p, cta);
    Seg s;
    for (uint32_t sg = 0; si.next(p, s); ++sg) {
        const uint32_t slot = sg & 1;
        if (sg >= 2 && !mbar_wait(bar(c, kBarNormEmpty + slot), ((sg >> 1) - 1) & 1, p.err))
            return;
        float *dst = reinterpret_cast<float *>(c.sbase + kOffNorm + slot * kNormSlotBytes);
        const float *src = p.norms + s.head * p.norm_pitch;
        const long long r0 = static_cast<long long>(s.row0) + s.q0;
        float v[2 * kBlockM / 32];
#pragma unroll
        for (int j = 0; j < 2 * kBlockM / 32; ++j) {
            const long long r = r0 + lane + 32 * j;
            v[j] = r < p.rows ? src[r] : 0.f;
        }
        // K rows [lo, hi): the unaligned ends one by one, the rest 8 at a time
        // (pairs of fp16 bit patterns, maxima taken two at a time)
        const uint16_t *kn = p.knorm + s.head * p.norm_pitch;
        const long long lo = s.row0, hi = static_cast<long long>(s.row0) + s.L;
        const long long a0 = min((lo + 7) & ~7ll, hi), a1 = max(hi & ~7ll, a0);
        uint32_t k0 = 0u, k1 = 0u;
        if (lo + lane < a0)
            k0 = kn[lo + lane];
        if (a1 + lane < hi)
            k1 = kn[a1 + lane];
        const uint4 *kv = reinterpret_cast<const uint4 *>(kn + a0);
        const int nv = static_cast<int>((a1 - a0) >> 3);
#pragma unroll 8
        for (int i = lane; i < nv; i += 32) {
            const uint4 q8 = kv[i];
            k0 = __vmaxu2(k0, __vmaxu2(q8.x, q8.y));
            k1 = __vmaxu2(k1, __vmaxu2(q8.z, q8.w));
        }
        const uint32_t k2 = __vmaxu2(k0, k1);
        const uint32_t kh = __reduce_max_sync(0xffffffffu, max(k2 & 0xFFFFu, k2 >> 16));
        const float kmx = __half2float(__ushort_as_half(static_cast<unsigned short>(kh)));
#pragma unroll
        for (int j = 0; j < 2 * kBlockM / 32; ++j)
            dst[lane + 32 * j] = v[j];
        if (lane == 0)
            dst[2 * kBlockM] = kmx;
        __syncwarp();
        if (lane == 0)
            mbar_arrive(bar(c, kBarNormFull + slot));
    }
}

// ---------------------------------------------------------------- softmax
__device__ __forceinline__ float *partial_slot(const Params &p, int slot)
{
    return p.partials + static_cast<size_t>(slot) * kPartialFloats;
}

// Slot used by CTA cc for unit u, starting at iteration ua: its first slot
// when the unit is (or starts) its first segment, else its second.  CTA cc's
// range starts at or after ua when x_lo(cc) lies past the last iteration
// before the unit (ua - 1, of unit u - 1).
__device__ __forceinline__ int slot_of(const Params &p, int cc, long long ua, int u)
{
    return (ua == 0 || x_lo(p, cc) >= ua + static_cast<long long>(p.alpha) * (u - 1)) ? 2 * cc : 2 * cc + 1;
}

__device__ void softmax_group(const Ctx &c, const Params &p, int w, int warp_in_group,
                              int lane, int cta)
{
    const uint32_t lane_off = static_cast<uint32_t>(32 * warp_in_group) << 16;
    const uint32_t tS = c.tmem + col_s(w) + lane_off;
    const uint32_t tP = c.tmem + col_p(w) + lane_off;
    const uint32_t tO = c.tmem + col_o(w) + lane_off;
    const int r = 32 * warp_in_group + lane;          // row within the query tile
    const int rr = kBlockM * w + r;                   // row within the entry
    volatile int *flag = reinterpret_cast<volatile int *>(c.sbase + kOffFlag);
    SegIter si;
    si.init(p, cta);
    Seg s;
    uint32_t g0 = 0, npartial = 0;
    for (uint32_t sg = 0; si.next(p, s); ++sg) {
        const int n = s.ke - s.kb;
        // The CTA's last segment, when it is the first of a unit cut between
        // CTAs (the usual case at the end of a range): the unit's other
        // segments ran at the start of the next CTAs' ranges.  One thread
        // reads the unit's counter now (acquire), while the segment runs; if
        // they are all in, this segment merges at its end without leaving
        // its own state in the workspace.
        const bool early = si.it >= si.hi && s.kb == 0 && n != s.ntiles;
        const bool looker = early && w == 0 && r == 0;
        int early_done = -1;
        if (looker)
            asm volatile("ld.acquire.gpu.global.b32 %0, [%1];"
                         : "=r"(early_done) : "l"(p.unit_cnt + s.entry * kHeads + s.head) : "memory");
        float m = -INFINITY;    // running reference maximum (scaled, base 2)
        float l = 0.f;          // running sum of exp2(score - m)
        // One key tile; with_max false leaves out the row maximum (the
        // reference stays).  False when a wait gave up.
        auto tile = [&](int t, auto with_max) -> bool {
            const uint32_t g = g0 + t;
            if (!mbar_wait(bar(c, kBarSFull + w), g & 1, p.err))
                return false;
            __syncwarp();
            tc_fence_after();
            float sc[kBlockN];
            {
                uint32_t r0[32], r1[32], r2[32], r3[32];
                tmem_ld32(tS, r0);
                tmem_ld32(tS + 32, r1);
                tmem_ld32(tS + 64, r2);
                tmem_ld32(tS + 96, r3);
                tmem_wait_ld();
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    sc[i] = __uint_as_float(r0[i]);
                    sc[32 + i] = __uint_as_float(r1[i]);
                    sc[64 + i] = __uint_as_float(r2[i]);
                    sc[96 + i] = __uint_as_float(r3[i]);
                }
            }
            tc_fence_before();
            mbar_arrive(bar(c, kBarSEmpty + w));   // S may be overwritten now

            const int kvalid = s.L - (s.kb + t) * kBlockN;   // keys of this tile in the sequence
            if (kvalid < kBlockN) {
#pragma unroll
                for (int i = 0; i < kBlockN; ++i)
                    if (i >= kvalid)
                        sc[i] = -INFINITY;
            }
            // row maximum: 8 independent chains (columns 0-15 by 2-input
            // max, then 16 columns per step by 3-input max), then combine
            float mc = m;
            if constexpr (decltype(with_max)::value) {
                float mp[8];
#pragma unroll
                for (int k = 0; k < 8; ++k)
                    mp[k] = fmaxf(sc[k], sc[8 + k]);
#pragma unroll
                for (int i = 16; i < kBlockN; i += 16)
#pragma unroll
                    for (int k = 0; k < 8; ++k)
                        mp[k] = fmax3(mp[k], sc[i + k], sc[i + 8 + k]);
                const float mx = fmaxf(fmax3(mp[0], mp[1], mp[2]),
                                       fmaxf(fmax3(mp[3], mp[4], mp[5]), fmax3(mp[6], mp[7], mp[7])));
                mc = mx * kScaleLog2;
            }
            // (without the maximum the reference stays: no rescale at all)
            const bool need = decltype(with_max)::value && mc > m + kRescaleThreshold;
            const float mn = need ? mc : m;
            const float alpha = need ? ex2_approx(m - mn) : 1.f;
            const float neg = -mn;

            // p = 2^(s * scale - m), packed to bf16 pairs; row sum in 4
            // independent packed fp32x2 accumulators
            uint32_t pk[kBlockN / 2];
            // one asm block per score pair: the exponent on the packed
            // fp32x2 path, the two exponentials, the pair added to one of four
            // packed row-sum accumulators, and the bf16 pack of P
            uint64_t acc2[4] = {0ull, 0ull, 0ull, 0ull};
            const uint64_t sc2 = f2(kScaleLog2, kScaleLog2), nm2 = f2(neg, neg);
#pragma unroll
            for (int i = 0; i < kBlockN / 2; ++i) {
                asm("{\n\t.reg .b64 y, pp;\n\t.reg .f32 y0, y1, p0, p1;\n\t"
                    "mov.b64 y, {%2, %3};\n\t"
                    "fma.rn.f32x2 y, y, %4, %5;\n\t"
                    "mov.b64 {y0, y1}, y;\n\t"
                    "ex2.approx.ftz.f32 p0, y0;\n\t"
                    "ex2.approx.ftz.f32 p1, y1;\n\t"
                    "mov.b64 pp, {p0, p1};\n\t"
                    "add.f32x2 %1, %1, pp;\n\t"
                    "cvt.rn.bf16x2.f32 %0, p1, p0;\n\t}"
                    : "=r"(pk[i]), "+l"(acc2[i & 3])
                    : "f"(sc[2 * i]), "f"(sc[2 * i + 1]), "l"(sc2), "l"(nm2));
            }
            uint64_t accs = acc2[0];
            asm("add.f32x2 %0, %0, %1;" : "+l"(accs) : "l"(acc2[1]));
            asm("add.f32x2 %0, %0, %1;" : "+l"(accs) : "l"(acc2[2]));
            asm("add.f32x2 %0, %0, %1;" : "+l"(accs) : "l"(acc2[3]));
            float acc0, acc1;
            f2_split(accs, acc0, acc1);

            if (t > 0) {
                // P_w and O_w are free once the previous P V has completed
                if (!mbar_wait(bar(c, kBarODone + w), (g - 1) & 1, p.err))
                    return false;
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
            l = l * alpha + (acc0 + acc1);
            m = mn;
            tmem_st64(tP, pk);
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(bar(c, kBarPFull + w));
            return true;
        };
        // Tiles with the row maximum up to the segment's second tile; then,
        // when a later tile follows, the rows' score bound (staged by warp 11)
        // decides whether the remaining tiles need a maximum.  The decision
        // always falls at that tile, so the result does not depend on timing.
        const uint32_t nslot = sg & 1, npar = (sg >> 1) & 1;
        const float *nv = reinterpret_cast<const float *>(c.sbase + kOffNorm + nslot * kNormSlotBytes);
        bool decided = false, skip = false;
        int t = 0;
        for (; t < n; ++t) {
            if (!tile(t, std::true_type{}))
                return;
            if (!decided && t >= 1 && t + 1 < n) {
                if (!__all_sync(0xffffffffu, mbar_test(bar(c, kBarNormFull + nslot), npar)) &&
                    !slow_wait(bar(c, kBarNormFull + nslot), npar, p.err))
                    return;
                const float bound = nv[rr] * nv[2 * kBlockM] * (kScaleLog2 * kBoundMargin);
                mbar_arrive(bar(c, kBarNormEmpty + nslot));
                decided = true;
                skip = __all_sync(0xffffffffu, bound <= m + kSkipSlack);
                if (skip) {
                    ++t;
                    break;
                }
            }
        }
        for (; t < n; ++t)
            if (!tile(t, std::false_type{}))
                return;
        if (!decided) {
            if (!mbar_wait(bar(c, kBarNormFull + nslot), npar, p.err))
                return;
            mbar_arrive(bar(c, kBarNormEmpty + nslot));
        }
        g0 += n;

        // ---- end of the segment: O of this segment in registers
        if (!mbar_wait(bar(c, kBarODone + w), (g0 - 1) & 1, p.err))
            return;
        __syncwarp();
        tc_fence_after();
        float o[kHeadDim];
        {
            uint32_t a[32], b[32];
            tmem_ld32(tO, a);
            tmem_ld32(tO + 32, b);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                o[i] = __uint_as_float(a[i]);
                o[32 + i] = __uint_as_float(b[i]);
            }
        }
        tc_fence_before();
        mbar_arrive(bar(c, kBarOFree + w));   // the next segment may reset O

        bool write = true;
        bool merge_now = false;
        if (early) {
            if (looker) {
                *reinterpret_cast<volatile int *>(c.sbase + kOffEarly) =
                    early_done == cta_of(p, s.ua + s.ntiles - 1, s.entry * kHeads + s.head) - cta;
                mbar_arrive(bar(c, kBarEarly));
            }
            if (!mbar_wait(bar(c, kBarEarly), 0, p.err))
                return;
            merge_now = *reinterpret_cast<volatile int *>(c.sbase + kOffEarly) != 0;
        }
        if (n != s.ntiles) {
            // The unit is split between CTAs: leave this segment's state in
            // the workspace, and merge if this is the unit's last segment
            // (known from the early look, or from the unit's counter).
            const long long ua = s.ua, ub = s.ua + s.ntiles;
            const int unit = s.entry * kHeads + s.head;
            if (!merge_now) {
                float *mine = partial_slot(p, slot_of(p, cta, ua, unit));
                float4 *dst = reinterpret_cast<float4 *>(mine + rr * kHeadDim);
#pragma unroll
                for (int i = 0; i < kHeadDim / 4; ++i)
                    dst[i] = make_float4(o[4 * i], o[4 * i + 1], o[4 * i + 2], o[4 * i + 3]);
                reinterpret_cast<float2 *>(mine + kPartialRows * kHeadDim)[rr] = make_float2(m, l);
                __threadfence();
                mbar_arrive(bar(c, kBarSegSync));
            }
            if (w == 0 && r == 0) {
                int last = 1;
                if (!merge_now) {
                    last = 0;
                    if (mbar_wait(bar(c, kBarSegSync), npartial & 1, p.err)) {
                        const int c_first = cta_of(p, ua, unit), c_last = cta_of(p, ub - 1, unit);
                        const int nseg = c_last - c_first + 1;
                        last = atomicAdd(p.unit_cnt + unit, 1) == nseg - 1;
                        __threadfence();
                    }
                }
                *flag = last;
                mbar_arrive(bar(c, kBarSegFlag));
            }
            if (!mbar_wait(bar(c, kBarSegFlag), npartial & 1, p.err))
                return;
            ++npartial;                                  // (SegSync is not used when merge_now: last segment)
            write = *flag != 0;
            if (write) {
                // Merge every segment's state (this CTA's included) in CTA
                // order, so that the result does not depend on which CTA
                // finished last.  When this CTA holds the first segment (the
                // usual case: its last segment is the unit's first), its own
                // state is already the running state; the first merge step
                // would reproduce it exactly (weights 0 and 1).
                const int c_first = cta_of(p, ua, unit), c_last = cta_of(p, ub - 1, unit);
                int cc = c_first;
                if (c_first == cta) {
                    ++cc;
                } else {
                    m = -INFINITY;
                    l = 0.f;
#pragma unroll
                    for (int i = 0; i < kHeadDim; ++i)
                        o[i] = 0.f;
                }
                for (; cc <= c_last; ++cc) {
                    const float *part = partial_slot(p, slot_of(p, cc, ua, unit));
                    const float2 ml = __ldcg(reinterpret_cast<const float2 *>(part + kPartialRows * kHeadDim) + rr);
                    const float mnew = fmaxf(m, ml.x);
                    const float a = cc == c_first ? 0.f : ex2_approx(m - mnew);
                    const float b = ex2_approx(ml.x - mnew);
                    const float4 *src = reinterpret_cast<const float4 *>(part + rr * kHeadDim);
#pragma unroll
                    for (int i = 0; i < kHeadDim / 4; ++i) {
                        const float4 v = __ldcg(src + i);
                        o[4 * i] = o[4 * i] * a + v.x * b;
                        o[4 * i + 1] = o[4 * i + 1] * a + v.y * b;
                        o[4 * i + 2] = o[4 * i + 2] * a + v.z * b;
                        o[4 * i + 3] = o[4 * i + 3] * a + v.w * b;
                    }
                    l = l * a + ml.y * b;
                    m = mnew;
                }
            }
        }
        if (write) {
            // out[row, head*64 + d] = O / l, rounded to bf16; rows past the
            // end of the sequence are not written
            const int qpos = s.q0 + rr;
            if (qpos < s.L) {
                const float inv = l > 0.f ? 1.f / l : 0.f;
                uint4 *dst = reinterpret_cast<uint4 *>(p.out + static_cast<long long>(s.row0 + qpos) * kHidden
                                                       + s.head * kHeadDim);
#pragma unroll
                for (int i = 0; i < kHeadDim / 8; ++i)
                    dst[i] = make_uint4(pack_bf16x2(o[8 * i] * inv, o[8 * i + 1] * inv),
                                        pack_bf16x2(o[8 * i + 2] * inv, o[8 * i + 3] * inv),
                                        pack_bf16x2(o[8 * i + 4] * inv, o[8 * i + 5] * inv),
                                        pack_bf16x2(o[8 * i + 6] * inv, o[8 * i + 7] * inv));
            }
        }
    }
}

__global__ void __launch_bounds__(kThreads, 1)
attn_global_kernel(const __grid_constant__ CUtensorMap tm_rot,
                   const __grid_constant__ CUtensorMap tm_qkv,
                   const int32_t *__restrict__ cu, const int2 *__restrict__ work,
                   const int32_t *__restrict__ work_count, const int32_t *__restrict__ tile_start,
                   int32_t *__restrict__ unit_cnt, float *__restrict__ partials,
                   __nv_bfloat16 *__restrict__ out, int32_t *err, const float *__restrict__ norms,
                   const uint16_t *__restrict__ knorm, long long norm_pitch, long long rows)
{
    pdl_wait();
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    Ctx c;
    c.base = (raw + 1023u) & ~1023u;
    c.sbase = smem_raw + (c.base - raw);
    uint32_t *slot = reinterpret_cast<uint32_t *>(c.sbase + kOffSlot);

    Params p;
    p.entries = *work_count;
    if (p.entries <= 0)
        return;
    p.cu = cu;
    p.work = work;
    p.tile_start = tile_start;
    p.unit_cnt = unit_cnt;
    p.partials = partials;
    p.out = out;
    p.err = err;
    p.norms = norms;
    p.knorm = knorm;
    p.norm_pitch = norm_pitch;
    p.rows = rows;
    p.total = tile_start[p.entries];
    // split among at most `total` CTAs, so that every range is non-empty
    p.ctas = p.total < gridDim.x ? static_cast<int>(p.total) : static_cast<int>(gridDim.x);
    // weigh unit starts only where every range stays non-empty: with
    // cost >= (alpha + 1) * ctas consecutive range starts lie more than one
    // inter-unit gap apart in cost coordinates
    {
        const long long extra = static_cast<long long>(kSegCost) * (static_cast<long long>(kHeads) * p.entries - 1);
        const bool weigh = p.total + extra >= static_cast<long long>(kSegCost + 1) * p.ctas;
        p.alpha = weigh ? kSegCost : 0;
        p.cost = p.total + (weigh ? extra : 0);
    }
    const int cta = blockIdx.x;
    if (cta >= p.ctas)
        return;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        tma_prefetch_desc(&tm_rot);
        tma_prefetch_desc(&tm_qkv);
        for (int q = 0; q < 2; ++q) {
            mbar_init(bar(c, kBarQFull + q), 1);
            mbar_init(bar(c, kBarQEmpty + q), 2);   // one commit per issuer
        }
        for (int s = 0; s < kStages; ++s) {
            mbar_init(bar(c, kBarKFull + s), 1);
            mbar_init(bar(c, kBarKEmpty + s), 2);
            mbar_init(bar(c, kBarVFull + s), 1);
            mbar_init(bar(c, kBarVEmpty + s), 2);
        }
        for (int w = 0; w < 2; ++w) {
            mbar_init(bar(c, kBarSFull + w), 1);
            mbar_init(bar(c, kBarSEmpty + w), kBlockM);
            mbar_init(bar(c, kBarPFull + w), kBlockM);
            mbar_init(bar(c, kBarODone + w), 1);
            mbar_init(bar(c, kBarOFree + w), kBlockM);
        }
        mbar_init(bar(c, kBarSegSync), 2 * kBlockM);
        mbar_init(bar(c, kBarSegFlag), 1);
        mbar_init(bar(c, kBarEarly), 1);
        for (int q = 0; q < 2; ++q) {
            mbar_init(bar(c, kBarNormFull + q), 1);
            mbar_init(bar(c, kBarNormEmpty + q), 2 * kBlockM);
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
                producer(c, p, &tm_rot, &tm_qkv, cta);
            __syncwarp();
        } else if (warp == 9 || warp == 10) {
            mma_issuer(c, p, warp - 9, cta);
            __syncwarp();
        } else {
            norm_stager(c, p, lane, cta);
            __syncwarp();
        }
    } else {
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" :: "n"(kRegsSoftmax));
        softmax_group(c, p, warp >> 2, warp & 3, lane, cta);
        __syncwarp();
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(c.tmem, kTmemCols);
    }
    pdl_trigger();
}

}  // namespace

cudaError_t launch_attn_global(const AttnArgs &a, cudaStream_t stream)
{
    static PerDeviceOnce smem_once;
    cudaError_t e = smem_opt_in(smem_once, attn_global_kernel, kSmemBytes);
    if (e != cudaSuccess)
        return e;
    return launch_chained(attn_global_kernel, dim3(a.num_ctas), dim3(kThreads), kSmemBytes, stream,
        a.tm_rot, a.tm_qkv, a.cu, a.work, a.work_count, a.tile_start, a.unit_cnt, a.partials,
        a.out, a.err, a.norms, a.knorm, a.norm_pitch, a.rows);
}

}  // namespace mbert
