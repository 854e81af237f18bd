// Launch interface between the host library (host.cu) and the kernel
// translation units.  Not part of the public C ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include <atomic>
#include <mutex>

namespace mbert {

constexpr int kMaxDevices = 64;

// Per-device set-up of one kernel that must happen once in each device
// context before its first launch there (a shared-memory opt-in, an
// occupancy query).  Safe to use from several host threads: the first
// caller on a device runs the set-up under the lock, later callers read the
// published value without locking.
struct PerDeviceOnce {
    std::mutex mu;
    std::atomic<int> value[kMaxDevices] = {};   // 0: not set up yet
};

// Returns in *value the set-up result for the current device (a positive
// int), running `setup(&v)` on the first call there.
template <typename Setup>
cudaError_t per_device_once(PerDeviceOnce &once, int *value, Setup setup)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    if (dev < 0 || dev >= kMaxDevices)
        return cudaErrorInvalidDevice;
    int v = once.value[dev].load(std::memory_order_acquire);
    if (v == 0) {
        std::lock_guard<std::mutex> lock(once.mu);
        v = once.value[dev].load(std::memory_order_relaxed);
        if (v == 0) {
            e = setup(&v);
            if (e != cudaSuccess)
                return e;
            once.value[dev].store(v, std::memory_order_release);
        }
    }
    *value = v;
    return cudaSuccess;
}

// Raise `kernel`'s dynamic shared-memory limit to `bytes` on the current
// device (once per device).
template <typename Kernel>
cudaError_t smem_opt_in(PerDeviceOnce &once, Kernel kernel, size_t bytes)
{
    int v = 0;
    return per_device_once(once, &v, [&](int *out) {
        cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(bytes));
        *out = 1;
        return e;
    });
}

// Launch `kernel` on `stream` with programmatic stream serialization: its
// launch may overlap the tail of the previous kernel in the stream, which
// it waits for in-kernel (pdl_wait) before touching memory.
template <typename... KArgs, typename... Args>
cudaError_t launch_chained(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                           cudaStream_t stream, Args &&...args)
{
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

constexpr int kPairsConst = 32;

// Work list written by the plan kernel: one entry per (sequence, 128-query
// block), longest sequences first; the attention grid covers entries x heads.
struct Plan {
    int block = 128;        // query rows per work entry (128 or 256)
    const int32_t *cu;      // device [n_seqs + 1]
    int n_seqs;
    int64_t T;
    int max_seqlen;         // longest sequence accepted by the device check
    int2 *work;             // device [entry_bound]
    int32_t *work_count;    // device scalar: entries written (0 if the checks failed)
    int entry_bound;        // host-side upper bound on the entry count
    int32_t *err;           // device error word (sticky, bit mask)
    bool cu_short_ok = false;   // accept cu[n] <= T: rows past cu[n] belong to no sequence
    // Optional (global layers): tile_start[e] = sum over entries before e of
    // heads * ceil(L/128) (the entry's first iteration in the split of all
    // (entry, head, key tile) iterations among persistent CTAs), with
    // tile_start[count] = the total; unit_cnt[entry * heads + head] zeroed.
    int32_t *tile_start = nullptr;   // device [entry_bound + 1]
    int32_t *unit_cnt = nullptr;     // device [entry_bound * heads]
};

cudaError_t launch_plan(const Plan &p, cudaStream_t stream);

// The plan and, in the same launch, the RoPE of Q and K of every row (all
// heads) into rot[T][1536] bf16.  With norms set (global layers), also the
// Euclidean norm of every rotated row and head: Q head h in norms[h][row]
// (fp32), K head h in knorm[h][row] (fp16 bits, rounded up), rows
// `norm_pitch` apart (a multiple of 8).
cudaError_t launch_plan_rope(const Plan &p, const __nv_bfloat16 *qkv, const float2 *table,
                             int table_rows, __nv_bfloat16 *rot, float *norms, uint16_t *knorm,
                             long long norm_pitch, cudaStream_t stream);

// Admitted-key count per query row, from the attention kernels' tile
// schedule and mask.
cudaError_t launch_key_count(const Plan &p, int half_window, int32_t *counts,
                             cudaStream_t stream);

struct AttnArgs {
    CUtensorMap tm_rot;     // rotated Q/K [T][1536], box 64 x 128, 128B swizzle
    CUtensorMap tm_qkv;     // qkv [T][2304], box 64 x 128, 128B swizzle
    const int32_t *cu;
    const int2 *work;
    const int32_t *work_count;
    int entry_bound;
    int half_window;        // < 0: global layer
    __nv_bfloat16 *out;     // [T][768]
    int32_t *err;
    // global layers: persistent CTAs and the split of iterations
    int num_ctas = 0;
    const int32_t *tile_start = nullptr;
    int32_t *unit_cnt = nullptr;
    float *partials = nullptr;   // [2 * num_ctas][kPartialFloats]
    const float *norms = nullptr;     // [12][norm_pitch]: rotated Q row norms per head
    const uint16_t *knorm = nullptr;  // [12][norm_pitch]: rotated K row norms, fp16 rounded up
    long long norm_pitch = 0;         // a multiple of 8
    long long rows = 0;               // rows of qkv
};

// One partial state of a query block split across CTAs: O (unnormalised,
// fp32) for 256 rows x 64, then (m, l) for the 256 rows.
constexpr int kPartialRows = 256;
constexpr int kPartialFloats = kPartialRows * 64 + kPartialRows * 2;

// RoPE constants for computing cos/sin in the local kernel: for pair m the
// frequency in turns per position as a 64-bit binary fraction (frac_hi holds
// 2^-1 .. 2^-32, frac_lo 2^-33 .. 2^-64), so that the turns of any position
// are exact modulo 1 in integer arithmetic, and the rotation by 128
// positions (cos, sin of 128 w, fp64 values rounded to fp32).
struct RopeConsts {
    uint32_t frac_hi[kPairsConst];
    uint32_t frac_lo[kPairsConst];
    float cos128[kPairsConst];
    float sin128[kPairsConst];
};

struct LocalArgs {
    RopeConsts rope;
    CUtensorMap tm_qkv;          // qkv [T][2304], box 64 x 128, 128B swizzle
    CUtensorMap tm_out;          // out [T][768], box 64 x 128, 128B swizzle
    const int32_t *cu;
    int n_seqs;
    long long T;
    int max_seqlen;
    const int2 *work;            // null: each CTA finds its block from cu_seqlens
    const int32_t *work_count;
    int half_window;             // <= kBandReach
    int block_bound;             // upper bound on 128-query blocks over all sequences
    int num_ctas;                // persistent CTAs (one per SM)
    __nv_bfloat16 *out;
    int32_t *err;
};

// Local-layer attention with RoPE in the prologue: persistent CTAs, each
// walking a contiguous range of (128-query block, head) units, two band
// tiles of keys per unit.
cudaError_t launch_attn_local(const LocalArgs &a, cudaStream_t stream);

// Output projection with the residual add, y = x + a Wo^T: persistent pairs
// of CTAs over 256 x 256 output blocks.
struct OutProjArgs {
    CUtensorMap tm_a;            // a  [T][768], box 64 x 128, 128B swizzle
    CUtensorMap tm_w;            // Wo [768][768] ([out][in]), box 64 x 128, 128B swizzle
    CUtensorMap tm_x;            // x  [T][768], box 64 x 128, 128B swizzle
    CUtensorMap tm_y;            // y  [T][768] (may be x), box 64 x 128, 128B swizzle
    const __nv_bfloat16 *x;      // x itself, for L2 prefetches
    long long T;
    int num_ctas;                // SMs: the launch sizes its pairs by occupancy
    int32_t *err;
};

cudaError_t launch_out_proj(const OutProjArgs &a, cudaStream_t stream);

// The fused Wqkv projection, qkv = h Wqkv^T: the same paired GEMM over
// 256 x 256 output blocks, 2304 output columns, no residual.
struct QkvProjArgs {
    CUtensorMap tm_a;            // h    [T][768], box 64 x 128, 128B swizzle
    CUtensorMap tm_w;            // Wqkv [2304][768] ([out][in]), box 64 x 128, 128B swizzle
    CUtensorMap tm_y;            // qkv  [T][2304], box 64 x 128, 128B swizzle
    long long T;
    int num_ctas;
    int32_t *err;
};

cudaError_t launch_qkv_proj(const QkvProjArgs &a, cudaStream_t stream);

// The GeGLU MLP's two GEMMs, on the same paired body: m = GELU(g) * u from
// h [T][768] and Wi [2304][768] into m [T][1152] (tm_a over h with width
// 768, tm_w over Wi, tm_y over m), then y = x + m Wo^T with Wo [768][1152]
// (tm_a over m and tm_w over Wo, both width 1152).
cudaError_t launch_mlp_up(const QkvProjArgs &a, cudaStream_t stream);
cudaError_t launch_mlp_down(const OutProjArgs &a, cudaStream_t stream);

// Bias-free LayerNorm of each row of x [T][768] (bf16) with weight w [768]
// into h [T][768] (bf16): one warp per row, fp32 statistics.
cudaError_t launch_layernorm(const __nv_bfloat16 *x, const __nv_bfloat16 *w, long long T,
                             float eps, __nv_bfloat16 *h, int num_sms, cudaStream_t stream);

// The padded-batch form [B][S] with a 0/1 attention mask, to and from the
// packed form: mask_scan writes, per row b, each real token's rank among the
// row's real tokens (-1 for a pad) and the row's count, then the exclusive
// prefix sum of the counts as cu_seqlens[0..B]; gather copies every real
// token's qkv row to packed row cu[b] + rank; scatter writes every padded
// row of out from its packed row, zeros for pads.
cudaError_t launch_mask_scan(const int32_t *mask, int B, int S, int32_t *rank, int32_t *len,
                             int32_t *cu, cudaStream_t stream);
cudaError_t launch_gather_rows(const __nv_bfloat16 *src, const int32_t *rank, const int32_t *cu,
                               int B, int S, int width, __nv_bfloat16 *dst, int num_sms,
                               cudaStream_t stream);
cudaError_t launch_scatter_rows(const __nv_bfloat16 *src, const int32_t *rank, const int32_t *cu,
                                int B, int S, int width, __nv_bfloat16 *dst, int num_sms,
                                cudaStream_t stream);

// Number of sequences up to which the local kernel finds its blocks itself
// (above it the plan kernel writes a work list first).
constexpr int kLocalSelfScheduleMaxSeqs = 256;

// One bounded mbarrier wait that nothing completes (exercises kErrTimeout).
cudaError_t launch_wait_timeout_selftest(int32_t *err, unsigned long long limit_ns,
                                         cudaStream_t stream);

// Generic flash attention over pre-rotated Q/K: one CTA per (entry, head),
// entries of 128 query rows.
cudaError_t launch_attn_generic(const AttnArgs &a, cudaStream_t stream);

// Global-layer attention over pre-rotated Q/K: one CTA per (entry, head),
// entries of 256 query rows, warp-specialised tcgen05 pipeline.
cudaError_t launch_attn_global(const AttnArgs &a, cudaStream_t stream);

}  // namespace mbert
