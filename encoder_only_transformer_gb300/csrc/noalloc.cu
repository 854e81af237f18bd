// A forward entry point that allocates no device memory.
//
// Some callers cannot call cudaMalloc: a plugin loaded into a host
// framework that owns all device memory through its own pool, a serving
// process whose memory is reserved up front and must not grow afterwards,
// or a real-time loop that cannot afford the device-wide synchronisation a
// cudaMalloc or cudaFree may cause.  They cannot create a handle (creating
// one allocates the RoPE tables and the workspace), so this entry point
// takes every piece of scratch memory (work list, work count, error word,
// rotated Q/K rows and the two RoPE tables) from one file-scope static
// __device__ array.
//
// It is not the benchmarked path: for both layer kinds it runs the plan and
// the RoPE pass into the static rotated-Q/K rows (one launch), then the generic
// attention kernel (one CTA per 128-query block and head), not the
// persistent global and local kernels of mbert_attn_forward.  Its results
// agree with the oracle within the same bounds; its speed and its fp32
// summation order differ.
//
// That array lives in every GPU context that loads this part of the
// library, from the first call on that device until the process exits.
// All calls share it and it keeps the last call's contents: each call
// clears the words that must start at zero, and two calls whose work
// overlaps on the GPU (for example on two streams) race on it.
//
// The first call on a device sets up that device: it looks up the array's
// device address and fills the RoPE tables with a blocking copy, which
// synchronises with other work on the device.  Make that first call before
// any stream capture and outside any loop that must not block; later calls
// only enqueue work on the caller's stream.
#include <cmath>
#include <mutex>

#include "mbert_attn.h"
#include "common.cuh"
#include "internal.h"

#define MBERT_API extern "C" __attribute__((visibility("default")))

using namespace mbert;

namespace {

constexpr int64_t kMaxTokens = MBERT_NOALLOC_MAX_TOKENS;
constexpr int64_t kMaxSeqs = MBERT_NOALLOC_MAX_TOKENS;
constexpr int64_t kMaxEntries = (kMaxTokens + (kBlockM - 1) * kMaxSeqs) / kBlockM;
constexpr int kTableRows = static_cast<int>(kMaxTokens);

constexpr size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

// layout of the scratch array (every region 256-byte aligned)
constexpr size_t kOffRot = 0;
constexpr size_t kRotBytes = static_cast<size_t>(kMaxTokens) * 2 * kHidden * sizeof(__nv_bfloat16);
constexpr size_t kOffWork = align256(kOffRot + kRotBytes);
constexpr size_t kWorkBytes = static_cast<size_t>(kMaxEntries) * sizeof(int2);
constexpr size_t kOffWords = align256(kOffWork + kWorkBytes);   // [0] work count, [1] error word
constexpr size_t kOffRope = align256(kOffWords + 2 * sizeof(int32_t));
constexpr size_t kRopeBytes = static_cast<size_t>(kTableRows) * kPairs * sizeof(float2);
constexpr size_t kScratchBytes = align256(kOffRope + 2 * kRopeBytes);

static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

struct DeviceState {
    bool ready = false;
    unsigned char *base = nullptr;   // device address of g_scratch on this device
};
DeviceState g_dev[kMaxDevices];
EncodeTiledFn g_encode = nullptr;
std::mutex g_mu;

// host staging for one RoPE table (static storage: no allocation call)
float2 g_host_table[static_cast<size_t>(kTableRows) * kPairs];

// One-time set-up on the current device: find the device address of the
// scratch array and fill its two RoPE tables (cos, sin of
// pos * base^(-2m/64), evaluated in fp64, stored as fp32).
int setup(int device)
{
    std::lock_guard<std::mutex> lock(g_mu);
    if (g_dev[device].ready)
        return MBERT_OK;
    if (!g_encode) {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                             cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess || !fn)
            return MBERT_ERR_CUDA;
        g_encode = reinterpret_cast<EncodeTiledFn>(fn);
    }
    void *ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_scratch) != cudaSuccess || !ptr) {
        cudaGetLastError();
        return MBERT_ERR_CUDA;
    }
    unsigned char *base = static_cast<unsigned char *>(ptr);
    mbert_attn_config c;
    mbert_attn_default_config(&c);
    const double thetas[2] = {c.theta_global, c.theta_local};
    for (int k = 0; k < 2; ++k) {
        double inv[kPairs];
        for (int m = 0; m < kPairs; ++m)
            inv[m] = std::pow(thetas[k], -2.0 * m / kHeadDim);
        for (int p = 0; p < kTableRows; ++p)
            for (int m = 0; m < kPairs; ++m) {
                const double a = static_cast<double>(p) * inv[m];
                g_host_table[static_cast<size_t>(p) * kPairs + m] =
                    make_float2(static_cast<float>(std::cos(a)), static_cast<float>(std::sin(a)));
            }
        if (cudaMemcpy(base + kOffRope + k * kRopeBytes, g_host_table, kRopeBytes,
                       cudaMemcpyHostToDevice) != cudaSuccess)
            return MBERT_ERR_CUDA;
    }
    g_dev[device].base = base;
    g_dev[device].ready = true;
    return MBERT_OK;
}

int encode_map(CUtensorMap *tm, const void *ptr, int width, int64_t rows)
{
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(width), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(width) * 2};
    cuuint32_t box[2] = {static_cast<cuuint32_t>(kHeadDim), static_cast<cuuint32_t>(kBlockM)};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = g_encode(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(ptr), dims,
                          strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? MBERT_OK : MBERT_ERR_CUDA;
}

}  // namespace

MBERT_API int mbert_attn_forward_noalloc(const void *qkv, const int32_t *cu_seqlens, int n_seqs,
                                         int64_t total_tokens, int max_seqlen, int layer_kind,
                                         void *out, int32_t *device_status, void *stream)
{
    const int64_t T = total_tokens;
    if (n_seqs < 0 || T < 0 || max_seqlen < 0)
        return MBERT_ERR_BAD_ARG;
    if (T > kMaxTokens || n_seqs > kMaxSeqs)
        return MBERT_ERR_BAD_ARG;               // beyond the static scratch
    if (layer_kind != MBERT_GLOBAL && layer_kind != MBERT_LOCAL)
        return MBERT_ERR_BAD_ARG;
    if (max_seqlen > kTableRows)
        return MBERT_ERR_SEQ_TOO_LONG;
    if (T == 0)
        return MBERT_OK;
    if (!qkv || !out || !cu_seqlens || n_seqs == 0)
        return MBERT_ERR_BAD_ARG;
    if ((reinterpret_cast<uintptr_t>(qkv) & 15) || (reinterpret_cast<uintptr_t>(out) & 15) ||
        (reinterpret_cast<uintptr_t>(device_status) & 3))
        return MBERT_ERR_BAD_ARG;
    const char *q0 = static_cast<const char *>(qkv), *o0 = static_cast<const char *>(out);
    if (q0 < o0 + T * kHidden * 2 && o0 < q0 + T * kQKVWidth * 2)
        return MBERT_ERR_BAD_ARG;

    int device = 0;
    if (cudaGetDevice(&device) != cudaSuccess || device < 0 || device >= kMaxDevices)
        return MBERT_ERR_CUDA;
    int rc = setup(device);
    if (rc != MBERT_OK)
        return rc;
    unsigned char *base = g_dev[device].base;
    int32_t *words = reinterpret_cast<int32_t *>(base + kOffWords);
    __nv_bfloat16 *rot = reinterpret_cast<__nv_bfloat16 *>(base + kOffRot);
    const float2 *table = reinterpret_cast<const float2 *>(base + kOffRope + layer_kind * kRopeBytes);
    cudaStream_t st = static_cast<cudaStream_t>(stream);

    Plan p;
    p.cu = cu_seqlens;
    p.n_seqs = n_seqs;
    p.T = T;
    p.max_seqlen = max_seqlen > 0 ? max_seqlen : kTableRows;
    p.work = reinterpret_cast<int2 *>(base + kOffWork);
    p.work_count = words;
    p.entry_bound = static_cast<int>((T + (kBlockM - 1) * static_cast<int64_t>(n_seqs)) / kBlockM);
    p.err = words + 1;

    AttnArgs a;
    if (encode_map(&a.tm_rot, rot, 2 * kHidden, T) != MBERT_OK ||
        encode_map(&a.tm_qkv, qkv, kQKVWidth, T) != MBERT_OK)
        return MBERT_ERR_CUDA;
    a.cu = cu_seqlens;
    a.work = p.work;
    a.work_count = p.work_count;
    a.entry_bound = p.entry_bound;
    mbert_attn_config c;
    mbert_attn_default_config(&c);
    a.half_window = layer_kind == MBERT_GLOBAL ? -1 : c.half_window;
    a.out = static_cast<__nv_bfloat16 *>(out);
    a.err = p.err;

    // the work count and the error word must start at zero on every call
    cudaError_t e = cudaMemsetAsync(words, 0, 2 * sizeof(int32_t), st);
    if (e == cudaSuccess)
        e = launch_plan_rope(p, static_cast<const __nv_bfloat16 *>(qkv), table, kTableRows, rot, nullptr,
                             nullptr, 0, st);
    if (e == cudaSuccess)
        e = launch_attn_generic(a, st);
    if (e == cudaSuccess && device_status)
        e = cudaMemcpyAsync(device_status, p.err, sizeof(int32_t), cudaMemcpyDeviceToDevice, st);
    return e == cudaSuccess ? MBERT_OK : MBERT_ERR_CUDA;
}
