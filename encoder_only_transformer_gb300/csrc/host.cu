// Host side of the mbert_attn C ABI: argument checks, the handle's device
// memory (RoPE tables, work list, rotated-operand scratch, error word),
// tensor-map encoding and kernel launches.
#include <cmath>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <new>
#include <vector>

#include "mbert_attn.h"
#include "common.cuh"
#include "internal.h"

#define MBERT_API extern "C" __attribute__((visibility("default")))

using namespace mbert;

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

struct mbert_attn {
    int device = 0;
    RopeConsts rope_consts[2];              // per layer kind, for in-kernel cos/sin
    int num_sms = 0;
    mbert_attn_config cfg{};
    float2 *rope[2] = {nullptr, nullptr};   // [MBERT_GLOBAL], [MBERT_LOCAL]: [max_seqlen][32]
    int32_t *err = nullptr;                 // sticky device error word
    int32_t *work_count = nullptr;
    int2 *work = nullptr;
    int64_t work_cap = 0;                   // entries
    __nv_bfloat16 *rot = nullptr;           // rotated Q/K scratch [rows][1536]
    int64_t rot_cap = 0;                    // rows
    __nv_bfloat16 *ln = nullptr;            // normalised rows [ln_cap][768] (ln_qkv, mlp)
    int64_t ln_cap = 0;                     // rows
    __nv_bfloat16 *mid = nullptr;           // GELU(g) * u rows [mid_cap][1152] (mlp)
    int64_t mid_cap = 0;                    // rows
    // the padded-batch call: packed qkv and out, each padded token's rank
    // among its row's real tokens, the row lengths and their cu_seqlens
    __nv_bfloat16 *pad_qkv = nullptr, *pad_out = nullptr;
    int64_t pad_qkv_cap = 0, pad_out_cap = 0;
    int32_t *pad_idx = nullptr, *pad_len = nullptr, *pad_cu = nullptr;
    int64_t pad_idx_cap = 0, pad_seq_cap = 0;
    // global layers: split of the (entry, head, key tile) iterations among
    // one persistent CTA per SM
    int32_t *tile_start = nullptr;          // [entries + 1]
    int32_t *unit_cnt = nullptr;            // [entries * heads]
    int64_t sk_cap = 0;                     // entries
    float *partials = nullptr;              // [2 * num_sms][kPartialFloats]
    // global layers: norms of the rotated rows, for the score bound that
    // lets the softmax skip its row maximum: Q fp32 [12][rot_cap], then K
    // fp16 [12][rot_cap] (rot_cap a multiple of 8)
    float *norms = nullptr;
    cudaStream_t last_stream = nullptr;
    EncodeTiledFn encode = nullptr;
    // measurement: event pairs around the attention kernel, per layer kind
    bool profiling = false;
    // start, end, start, end, ... per profile slot (global, local, projection)
    std::vector<cudaEvent_t> ev[MBERT_PROFILE_SLOTS];
    size_t ev_used[MBERT_PROFILE_SLOTS] = {};
    int64_t launches = 0;                   // every kernel this handle enqueued
    // recently encoded tensor maps, by (address, width, rows): encoding one
    // costs microseconds of host time, as much as a short kernel
    struct MapEntry {
        const void *ptr = nullptr;
        int width = 0;
        int64_t rows = -1;
        uint64_t used = 0;
        CUtensorMap map;
    };
    MapEntry maps[32];
    uint64_t map_clock = 0;
};

namespace {

struct DeviceGuard {
    int prev = -1;
    bool changed = false;
    explicit DeviceGuard(int dev)
    {
        if (cudaGetDevice(&prev) == cudaSuccess && prev != dev) {
            changed = cudaSetDevice(dev) == cudaSuccess;
        }
    }
    ~DeviceGuard()
    {
        if (changed)
            cudaSetDevice(prev);
    }
};

int fail_cuda(cudaError_t e)
{
    (void)e;
    return MBERT_ERR_CUDA;
}

// Upper bound on the number of (sequence, 128-query block) entries:
// sum ceil(L/128) <= (T + 127 n) / 128.
int64_t entry_bound(int64_t T, int64_t n)
{
    return (T + (kBlockM - 1) * n) / kBlockM;
}

int grow_workspace(mbert_attn *h, int64_t entries, int64_t rot_rows)
{
    if (entries > h->work_cap) {
        int64_t cap = entries < 1024 ? 1024 : entries;
        int2 *w = nullptr;
        if (cudaMalloc(&w, sizeof(int2) * cap) != cudaSuccess) {
            cudaGetLastError();
            return MBERT_ERR_OOM;
        }
        if (h->work) {
            cudaDeviceSynchronize();
            cudaFree(h->work);
        }
        h->work = w;
        h->work_cap = cap;
    }
    // global-layer split bookkeeping, sized for 256-row entries (at most
    // `entries` of them: (T + 255 n) / 256 <= the 128-row bound)
    if (entries > h->sk_cap) {
        int64_t cap = entries < 1024 ? 1024 : entries;
        int32_t *ts = nullptr, *uc = nullptr;
        if (cudaMalloc(&ts, sizeof(int32_t) * (cap + 1)) != cudaSuccess ||
            cudaMalloc(&uc, sizeof(int32_t) * cap * kHeads) != cudaSuccess) {
            cudaGetLastError();
            cudaFree(ts);
            return MBERT_ERR_OOM;
        }
        if (h->tile_start) {
            cudaDeviceSynchronize();
            cudaFree(h->tile_start);
            cudaFree(h->unit_cnt);
        }
        h->tile_start = ts;
        h->unit_cnt = uc;
        h->sk_cap = cap;
    }
    if (!h->partials) {
        if (cudaMalloc(&h->partials, sizeof(float) * 2 * h->num_sms * kPartialFloats) != cudaSuccess) {
            cudaGetLastError();
            h->partials = nullptr;
            return MBERT_ERR_OOM;
        }
    }
    if (rot_rows > h->rot_cap) {
        int64_t cap = rot_rows < 8192 ? 8192 : (rot_rows + 7) & ~static_cast<int64_t>(7);
        __nv_bfloat16 *r = nullptr;
        float *nr = nullptr;
        if (cudaMalloc(&r, sizeof(__nv_bfloat16) * 2 * kHidden * cap) != cudaSuccess ||
            cudaMalloc(&nr, (sizeof(float) + sizeof(uint16_t)) * kHeads * cap) != cudaSuccess) {
            cudaGetLastError();
            cudaFree(r);
            return MBERT_ERR_OOM;
        }
        if (h->rot) {
            cudaDeviceSynchronize();
            cudaFree(h->rot);
            cudaFree(h->norms);
        }
        h->rot = r;
        h->norms = nr;
        h->rot_cap = cap;
    }
    return MBERT_OK;
}

// 2-D bf16 tensor map over [rows][width] (row pitch = width * 2 bytes),
// box 64 columns x 128 rows, 128-byte swizzle, out-of-range reads give 0.
// Grow a handle-owned bf16 buffer of `width` columns to at least `rows` rows
// (at least 8192); the old buffer is freed after the device is idle.
int grow_rows(__nv_bfloat16 **buf, int64_t *cap, int64_t rows, int width)
{
    if (rows <= *cap)
        return MBERT_OK;
    const int64_t n = rows < 8192 ? 8192 : rows;
    __nv_bfloat16 *p = nullptr;
    if (cudaMalloc(&p, sizeof(__nv_bfloat16) * static_cast<size_t>(width) * n) != cudaSuccess) {
        cudaGetLastError();
        return MBERT_ERR_OOM;
    }
    if (*buf) {
        cudaDeviceSynchronize();
        cudaFree(*buf);
    }
    *buf = p;
    *cap = n;
    return MBERT_OK;
}

// The next event pair of a profile slot (both null while profiling is off).
int profile_events(mbert_attn *h, int slot, cudaEvent_t *ev0, cudaEvent_t *ev1)
{
    *ev0 = *ev1 = nullptr;
    if (!h->profiling)
        return MBERT_OK;
    std::vector<cudaEvent_t> &v = h->ev[slot];
    while (v.size() < h->ev_used[slot] + 2) {
        cudaEvent_t x;
        if (cudaEventCreate(&x) != cudaSuccess)
            return MBERT_ERR_CUDA;
        v.push_back(x);
    }
    *ev0 = v[h->ev_used[slot]];
    *ev1 = v[h->ev_used[slot] + 1];
    h->ev_used[slot] += 2;
    return MBERT_OK;
}

int encode_map(mbert_attn *h, CUtensorMap *tm, const void *ptr, int width, int64_t rows)
{
    mbert_attn::MapEntry *victim = &h->maps[0];
    for (auto &m : h->maps) {
        if (m.ptr == ptr && m.width == width && m.rows == rows) {
            m.used = ++h->map_clock;
            *tm = m.map;
            return MBERT_OK;
        }
        if (m.used < victim->used)
            victim = &m;
    }
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(width), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(width) * 2};
    cuuint32_t box[2] = {static_cast<cuuint32_t>(kHeadDim), static_cast<cuuint32_t>(kBlockM)};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = h->encode(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(ptr), dims,
                           strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                           CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        return MBERT_ERR_CUDA;
    victim->ptr = ptr;
    victim->width = width;
    victim->rows = rows;
    victim->used = ++h->map_clock;
    victim->map = *tm;
    return MBERT_OK;
}

bool ranges_overlap(const void *a, size_t na, const void *b, size_t nb)
{
    const char *pa = static_cast<const char *>(a), *pb = static_cast<const char *>(b);
    return pa < pb + nb && pb < pa + na;
}

// Common argument checks of forward / key_counts.
int check_common(const mbert_attn *h, const int32_t *cu, int n_seqs, int64_t T, int max_seqlen,
                 int layer_kind)
{
    if (!h)
        return MBERT_ERR_BAD_ARG;
    if (n_seqs < 0 || T < 0 || T > INT32_MAX || max_seqlen < 0)
        return MBERT_ERR_BAD_ARG;
    if (layer_kind != MBERT_GLOBAL && layer_kind != MBERT_LOCAL)
        return MBERT_ERR_BAD_ARG;
    if (T > 0 && (n_seqs == 0 || !cu))
        return MBERT_ERR_BAD_ARG;
    if (max_seqlen > h->cfg.max_seqlen)
        return MBERT_ERR_SEQ_TOO_LONG;
    return MBERT_OK;
}

Plan make_plan(mbert_attn *h, const int32_t *cu, int n_seqs, int64_t T, int max_seqlen)
{
    Plan p;
    p.cu = cu;
    p.n_seqs = n_seqs;
    p.T = T;
    p.max_seqlen = max_seqlen > 0 ? max_seqlen : h->cfg.max_seqlen;
    p.work = h->work;
    p.work_count = h->work_count;
    p.entry_bound = static_cast<int>(entry_bound(T, n_seqs));
    p.err = h->err;
    return p;
}

}  // namespace

MBERT_API int mbert_attn_default_config(mbert_attn_config *cfg)
{
    if (!cfg)
        return MBERT_ERR_BAD_ARG;
    cfg->heads = kHeads;
    cfg->head_dim = kHeadDim;
    cfg->half_window = 64;
    cfg->max_seqlen = 8192;
    cfg->theta_global = 160000.0;
    cfg->theta_local = 10000.0;
    return MBERT_OK;
}

MBERT_API const char *mbert_attn_strerror(int status)
{
    switch (status) {
    case MBERT_OK: return "success";
    case MBERT_ERR_BAD_ARG: return "invalid argument";
    case MBERT_ERR_UNSUPPORTED: return "unsupported configuration or device";
    case MBERT_ERR_SEQ_TOO_LONG: return "sequence longer than max_seqlen";
    case MBERT_ERR_BAD_CU_SEQLENS: return "invalid cu_seqlens";
    case MBERT_ERR_TIMEOUT: return "device wait timed out";
    case MBERT_ERR_CUDA: return "CUDA runtime error";
    case MBERT_ERR_OOM: return "out of device memory";
    default: return "unknown status";
    }
}

MBERT_API void mbert_attn_destroy(mbert_attn *h)
{
    if (!h)
        return;
    {
        DeviceGuard g(h->device);
        for (int k = 0; k < MBERT_PROFILE_SLOTS; ++k)
            for (cudaEvent_t e : h->ev[k])
                cudaEventDestroy(e);
        cudaFree(h->rope[0]);
        cudaFree(h->rope[1]);
        cudaFree(h->err);
        cudaFree(h->work_count);
        cudaFree(h->work);
        cudaFree(h->rot);
        cudaFree(h->norms);
        cudaFree(h->tile_start);
        cudaFree(h->unit_cnt);
        cudaFree(h->partials);
        cudaFree(h->ln);
        cudaFree(h->mid);
        cudaFree(h->pad_qkv);
        cudaFree(h->pad_out);
        cudaFree(h->pad_idx);
        cudaFree(h->pad_len);
        cudaFree(h->pad_cu);
    }
    delete h;
}

MBERT_API int mbert_attn_create(mbert_attn **out, const mbert_attn_config *cfg, int device)
{
    if (!out)
        return MBERT_ERR_BAD_ARG;
    *out = nullptr;
    mbert_attn_config c;
    if (cfg)
        c = *cfg;
    else
        mbert_attn_default_config(&c);
    if (c.heads != kHeads || c.head_dim != kHeadDim)
        return MBERT_ERR_UNSUPPORTED;
    if (c.half_window < 0 || c.half_window > 128 || c.max_seqlen < 1 ||
        c.max_seqlen > 1024 * kBlockM || !(c.theta_global > 1.0) || !(c.theta_local > 1.0))
        return MBERT_ERR_BAD_ARG;

    int ndev = 0;
    if (cudaGetDeviceCount(&ndev) != cudaSuccess) {
        cudaGetLastError();
        return MBERT_ERR_UNSUPPORTED;
    }
    if (device < 0 || device >= ndev)
        return MBERT_ERR_BAD_ARG;
    cudaDeviceProp prop;
    if (cudaGetDeviceProperties(&prop, device) != cudaSuccess)
        return MBERT_ERR_CUDA;
    if (prop.major != 10 || prop.minor != 3)
        return MBERT_ERR_UNSUPPORTED;   // the kernels are built for sm_103a only

    mbert_attn *h = new (std::nothrow) mbert_attn;
    if (!h)
        return MBERT_ERR_OOM;
    h->device = device;
    h->num_sms = prop.multiProcessorCount;
    h->cfg = c;
    DeviceGuard g(device);

    void *fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q)
            != cudaSuccess || q != cudaDriverEntryPointSuccess || !fn) {
        delete h;
        return MBERT_ERR_CUDA;
    }
    h->encode = reinterpret_cast<EncodeTiledFn>(fn);

    // RoPE tables: cos and sin of pos * base^(-2m/64), evaluated in fp64 and
    // stored as fp32 ("ModernBERT-base Architecture Teardown", "How Does
    // RoPE Work With Two Bases?"; "ModernBERT" (candding), "The two rope
    // tables": both tables are built once, up to the longest sequence).
    const size_t n = static_cast<size_t>(c.max_seqlen) * kPairs;
    float2 *host = static_cast<float2 *>(std::malloc(sizeof(float2) * n));
    if (!host) {
        delete h;
        return MBERT_ERR_OOM;
    }
    int rc = MBERT_OK;
    const double thetas[2] = {c.theta_global, c.theta_local};
    for (int k = 0; k < 2 && rc == MBERT_OK; ++k) {
        double inv[kPairs];
        for (int m = 0; m < kPairs; ++m)
            inv[m] = std::pow(thetas[k], -2.0 * m / kHeadDim);
        for (int p = 0; p < c.max_seqlen; ++p)
            for (int m = 0; m < kPairs; ++m) {
                const double a = static_cast<double>(p) * inv[m];
                host[static_cast<size_t>(p) * kPairs + m] =
                    make_float2(static_cast<float>(std::cos(a)), static_cast<float>(std::sin(a)));
            }
        if (cudaMalloc(&h->rope[k], sizeof(float2) * n) != cudaSuccess)
            rc = MBERT_ERR_OOM;
        else if (cudaMemcpy(h->rope[k], host, sizeof(float2) * n, cudaMemcpyHostToDevice) != cudaSuccess)
            rc = MBERT_ERR_CUDA;
    }
    std::free(host);
    // Constants for the kernels that compute cos/sin themselves: turns per
    // position, 1/(2 pi) base^(-2m/64), as a 64-bit binary fraction, and the
    // rotation by 128 positions.
    for (int k = 0; k < 2; ++k) {
        for (int m = 0; m < kPairs; ++m) {
            const double w = std::pow(thetas[k], -2.0 * m / kHeadDim);
            const double turns = w / (2.0 * 3.14159265358979323846);   // in (0, 1)
            const double t32 = std::ldexp(turns, 32);
            const double hi = std::floor(t32);
            const double lo = std::floor(std::ldexp(t32 - hi, 32));
            h->rope_consts[k].frac_hi[m] = static_cast<uint32_t>(hi);
            h->rope_consts[k].frac_lo[m] = static_cast<uint32_t>(lo);
            h->rope_consts[k].cos128[m] = static_cast<float>(std::cos(128.0 * w));
            h->rope_consts[k].sin128[m] = static_cast<float>(std::sin(128.0 * w));
        }
    }
    if (rc == MBERT_OK) {
        if (cudaMalloc(&h->err, sizeof(int32_t)) != cudaSuccess ||
            cudaMalloc(&h->work_count, sizeof(int32_t)) != cudaSuccess)
            rc = MBERT_ERR_OOM;
        else if (cudaMemset(h->err, 0, sizeof(int32_t)) != cudaSuccess ||
                 cudaMemset(h->work_count, 0, sizeof(int32_t)) != cudaSuccess)
            rc = MBERT_ERR_CUDA;
    }
    if (rc == MBERT_OK)
        rc = grow_workspace(h, entry_bound(c.max_seqlen, 1), 0);
    if (rc != MBERT_OK) {
        cudaGetLastError();
        mbert_attn_destroy(h);
        return rc;
    }
    *out = h;
    return MBERT_OK;
}

MBERT_API int mbert_attn_reserve(mbert_attn *h, int64_t max_tokens, int64_t max_seqs)
{
    if (!h || max_tokens < 0 || max_seqs < 0 || max_tokens > INT32_MAX)
        return MBERT_ERR_BAD_ARG;
    DeviceGuard g(h->device);
    return grow_workspace(h, entry_bound(max_tokens, max_seqs), max_tokens);
}

namespace {

// The attention call.  cu_short: the packed rows past cu[n_seqs] belong to
// no sequence (cu[n_seqs] <= total_tokens, checked on the device); the plan
// kernel then schedules local layers too.
int forward_impl(mbert_attn *h, const void *qkv, const int32_t *cu_seqlens, int n_seqs,
                 int64_t total_tokens, int max_seqlen, int layer_kind, void *out, void *stream,
                 bool cu_short)
{
    int rc = check_common(h, cu_seqlens, n_seqs, total_tokens, max_seqlen, layer_kind);
    if (rc != MBERT_OK)
        return rc;
    const int64_t T = total_tokens;
    if (T == 0)
        return MBERT_OK;
    if (!qkv || !out)
        return MBERT_ERR_BAD_ARG;
    if ((reinterpret_cast<uintptr_t>(qkv) & 15) || (reinterpret_cast<uintptr_t>(out) & 15))
        return MBERT_ERR_BAD_ARG;
    if (ranges_overlap(qkv, static_cast<size_t>(T) * kQKVWidth * 2, out,
                       static_cast<size_t>(T) * kHidden * 2))
        return MBERT_ERR_BAD_ARG;

    DeviceGuard g(h->device);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    rc = grow_workspace(h, entry_bound(T, n_seqs), T);
    if (rc != MBERT_OK)
        return rc;
    Plan p = make_plan(h, cu_seqlens, n_seqs, T, max_seqlen);
    p.cu_short_ok = cu_short;
    if (layer_kind == MBERT_GLOBAL) {
        // the global kernel takes 256 query rows (two 128-row tiles) per
        // entry and splits all iterations among one CTA per SM into
        // ranges of equal cost
        p.block = 2 * kBlockM;
        p.entry_bound = static_cast<int>((T + (p.block - 1) * static_cast<int64_t>(n_seqs)) / p.block);
        p.tile_start = h->tile_start;
        p.unit_cnt = h->unit_cnt;
    }

    AttnArgs a;
    if (encode_map(h, &a.tm_rot, h->rot, 2 * kHidden, T) != MBERT_OK ||
        encode_map(h, &a.tm_qkv, qkv, kQKVWidth, T) != MBERT_OK)
        return MBERT_ERR_CUDA;
    a.cu = cu_seqlens;
    a.work = h->work;
    a.work_count = h->work_count;
    a.entry_bound = p.entry_bound;
    a.half_window = layer_kind == MBERT_GLOBAL ? -1 : h->cfg.half_window;
    a.out = static_cast<__nv_bfloat16 *>(out);
    a.err = h->err;
    a.num_ctas = h->num_sms;
    a.tile_start = h->tile_start;
    a.unit_cnt = h->unit_cnt;
    a.partials = h->partials;

    cudaEvent_t ev0 = nullptr, ev1 = nullptr;
    if (profile_events(h, layer_kind, &ev0, &ev1) != MBERT_OK)
        return MBERT_ERR_CUDA;
    cudaError_t e = cudaSuccess;
    if (layer_kind == MBERT_LOCAL && h->cfg.half_window <= kBandReach) {
        // RoPE inside the attention kernel; with few sequences each CTA finds
        // its block itself and no plan kernel runs.
        LocalArgs la;
        la.rope = h->rope_consts[MBERT_LOCAL];
        la.tm_qkv = a.tm_qkv;
        if (encode_map(h, &la.tm_out, out, kHidden, T) != MBERT_OK)
            return MBERT_ERR_CUDA;
        la.cu = cu_seqlens;
        la.n_seqs = n_seqs;
        la.T = T;
        la.max_seqlen = p.max_seqlen;
        la.half_window = h->cfg.half_window;
        la.out = a.out;
        la.err = h->err;
        la.work = nullptr;
        la.work_count = nullptr;
        la.block_bound = p.entry_bound;
        la.num_ctas = h->num_sms;
        if (n_seqs > kLocalSelfScheduleMaxSeqs || cu_short) {
            e = launch_plan(p, st);
            la.work = h->work;
            la.work_count = h->work_count;
            h->launches += 1;
        }
        if (e == cudaSuccess && ev0)
            e = cudaEventRecord(ev0, st);
        if (e == cudaSuccess)
            e = launch_attn_local(la, st);
        if (e == cudaSuccess && ev1)
            e = cudaEventRecord(ev1, st);
        h->launches += 1;
        h->last_stream = st;
        return e == cudaSuccess ? MBERT_OK : fail_cuda(e);
    }
    float *norms = nullptr;
    uint16_t *knorm = nullptr;
    if (layer_kind == MBERT_GLOBAL) {
        norms = h->norms;
        knorm = reinterpret_cast<uint16_t *>(h->norms + kHeads * h->rot_cap);
        a.norms = norms;
        a.knorm = knorm;
        a.norm_pitch = h->rot_cap;
        a.rows = T;
    }
    e = launch_plan_rope(p, static_cast<const __nv_bfloat16 *>(qkv), h->rope[layer_kind],
                         h->cfg.max_seqlen, h->rot, norms, knorm, h->rot_cap, st);
    if (e == cudaSuccess && ev0)
        e = cudaEventRecord(ev0, st);
    if (e == cudaSuccess)
        e = layer_kind == MBERT_GLOBAL ? launch_attn_global(a, st) : launch_attn_generic(a, st);
    if (e == cudaSuccess && ev1)
        e = cudaEventRecord(ev1, st);
    h->launches += 2;
    h->last_stream = st;
    return e == cudaSuccess ? MBERT_OK : fail_cuda(e);
}

}  // namespace

MBERT_API int mbert_attn_forward(mbert_attn *h, const void *qkv, const int32_t *cu_seqlens,
                                 int n_seqs, int64_t total_tokens, int max_seqlen,
                                 int layer_kind, void *out, void *stream)
{
    return forward_impl(h, qkv, cu_seqlens, n_seqs, total_tokens, max_seqlen, layer_kind, out,
                        stream, false);
}

MBERT_API int mbert_attn_forward_padded(mbert_attn *h, const void *qkv, const int32_t *attention_mask,
                                        int batch, int seq_len, int layer_kind, void *out,
                                        void *stream)
{
    if (!h || batch < 0 || seq_len < 0 || (layer_kind != MBERT_GLOBAL && layer_kind != MBERT_LOCAL))
        return MBERT_ERR_BAD_ARG;
    if (seq_len > h->cfg.max_seqlen)
        return MBERT_ERR_SEQ_TOO_LONG;
    const int64_t rows = static_cast<int64_t>(batch) * seq_len;
    if (rows > INT32_MAX)
        return MBERT_ERR_BAD_ARG;
    if (rows == 0)
        return MBERT_OK;
    if (!qkv || !attention_mask || !out)
        return MBERT_ERR_BAD_ARG;
    if ((reinterpret_cast<uintptr_t>(qkv) & 15) || (reinterpret_cast<uintptr_t>(out) & 15) ||
        (reinterpret_cast<uintptr_t>(attention_mask) & 3))
        return MBERT_ERR_BAD_ARG;
    if (ranges_overlap(qkv, static_cast<size_t>(rows) * kQKVWidth * 2, out,
                       static_cast<size_t>(rows) * kHidden * 2) ||
        ranges_overlap(attention_mask, static_cast<size_t>(rows) * 4, out,
                       static_cast<size_t>(rows) * kHidden * 2))
        return MBERT_ERR_BAD_ARG;
    DeviceGuard g(h->device);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    int rc = grow_rows(&h->pad_qkv, &h->pad_qkv_cap, rows, kQKVWidth);
    if (rc == MBERT_OK)
        rc = grow_rows(&h->pad_out, &h->pad_out_cap, rows, kHidden);
    if (rc == MBERT_OK && (rows > h->pad_idx_cap || batch + 1 > h->pad_seq_cap)) {
        const int64_t ri = rows > h->pad_idx_cap ? (rows < 8192 ? 8192 : rows) : h->pad_idx_cap;
        const int64_t si = batch + 1 > h->pad_seq_cap ? (batch + 1 < 1024 ? 1024 : batch + 1)
                                                       : h->pad_seq_cap;
        int32_t *idx = nullptr, *len = nullptr, *cu = nullptr;
        if (cudaMalloc(&idx, sizeof(int32_t) * ri) != cudaSuccess ||
            cudaMalloc(&len, sizeof(int32_t) * si) != cudaSuccess ||
            cudaMalloc(&cu, sizeof(int32_t) * si) != cudaSuccess) {
            cudaGetLastError();
            cudaFree(idx);
            cudaFree(len);
            return MBERT_ERR_OOM;
        }
        if (h->pad_idx) {
            cudaDeviceSynchronize();
            cudaFree(h->pad_idx);
            cudaFree(h->pad_len);
            cudaFree(h->pad_cu);
        }
        h->pad_idx = idx;
        h->pad_len = len;
        h->pad_cu = cu;
        h->pad_idx_cap = ri;
        h->pad_seq_cap = si;
    }
    if (rc != MBERT_OK)
        return rc;
    cudaError_t e = launch_mask_scan(attention_mask, batch, seq_len, h->pad_idx, h->pad_len,
                                     h->pad_cu, st);
    if (e == cudaSuccess)
        e = launch_gather_rows(static_cast<const __nv_bfloat16 *>(qkv), h->pad_idx, h->pad_cu,
                               batch, seq_len, kQKVWidth, h->pad_qkv, h->num_sms, st);
    h->launches += 3;
    if (e != cudaSuccess)
        return fail_cuda(e);
    rc = forward_impl(h, h->pad_qkv, h->pad_cu, batch, rows, seq_len, layer_kind, h->pad_out,
                      stream, true);
    if (rc != MBERT_OK)
        return rc;
    e = launch_scatter_rows(h->pad_out, h->pad_idx, h->pad_cu, batch, seq_len, kHidden,
                            static_cast<__nv_bfloat16 *>(out), h->num_sms, st);
    h->launches += 1;
    h->last_stream = st;
    return e == cudaSuccess ? MBERT_OK : fail_cuda(e);
}

MBERT_API int mbert_attn_key_counts(mbert_attn *h, const int32_t *cu_seqlens, int n_seqs,
                                    int64_t total_tokens, int max_seqlen, int layer_kind,
                                    int32_t *counts, void *stream)
{
    int rc = check_common(h, cu_seqlens, n_seqs, total_tokens, max_seqlen, layer_kind);
    if (rc != MBERT_OK)
        return rc;
    if (total_tokens == 0)
        return MBERT_OK;
    if (!counts)
        return MBERT_ERR_BAD_ARG;
    DeviceGuard g(h->device);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    rc = grow_workspace(h, entry_bound(total_tokens, n_seqs), 0);
    if (rc != MBERT_OK)
        return rc;
    Plan p = make_plan(h, cu_seqlens, n_seqs, total_tokens, max_seqlen);
    h->launches += 2;
    cudaError_t e = launch_plan(p, st);
    if (e == cudaSuccess)
        e = launch_key_count(p, layer_kind == MBERT_GLOBAL ? -1 : h->cfg.half_window, counts, st);
    h->last_stream = st;
    return e == cudaSuccess ? MBERT_OK : fail_cuda(e);
}

MBERT_API int mbert_attn_out_proj(mbert_attn *h, const void *a, const void *wo, const void *x,
                                  int64_t total_tokens, void *y, void *stream)
{
    if (!h || total_tokens < 0 || total_tokens > INT32_MAX)
        return MBERT_ERR_BAD_ARG;
    const int64_t T = total_tokens;
    if (T == 0)
        return MBERT_OK;
    if (!a || !wo || !x || !y)
        return MBERT_ERR_BAD_ARG;
    for (const void *ptr : {a, wo, x, static_cast<const void *>(y)})
        if (reinterpret_cast<uintptr_t>(ptr) & 15)
            return MBERT_ERR_BAD_ARG;
    const size_t act = static_cast<size_t>(T) * kHidden * 2;
    const size_t wbytes = static_cast<size_t>(kHidden) * kHidden * 2;
    if (ranges_overlap(a, act, y, act) || ranges_overlap(wo, wbytes, y, act) ||
        (x != y && ranges_overlap(x, act, y, act)))
        return MBERT_ERR_BAD_ARG;
    DeviceGuard g(h->device);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    OutProjArgs o;
    if (encode_map(h, &o.tm_a, a, kHidden, T) != MBERT_OK ||
        encode_map(h, &o.tm_w, wo, kHidden, kHidden) != MBERT_OK ||
        encode_map(h, &o.tm_x, x, kHidden, T) != MBERT_OK ||
        encode_map(h, &o.tm_y, y, kHidden, T) != MBERT_OK)
        return MBERT_ERR_CUDA;
    o.x = static_cast<const __nv_bfloat16 *>(x);
    o.T = T;
    o.num_ctas = h->num_sms;
    o.err = h->err;
    cudaEvent_t ev0, ev1;
    if (profile_events(h, MBERT_PROFILE_OUT_PROJ, &ev0, &ev1) != MBERT_OK)
        return MBERT_ERR_CUDA;
    cudaError_t e = ev0 ? cudaEventRecord(ev0, st) : cudaSuccess;
    if (e == cudaSuccess)
        e = launch_out_proj(o, st);
    if (e == cudaSuccess && ev1)
        e = cudaEventRecord(ev1, st);
    h->launches += 1;
    h->last_stream = st;
    return e == cudaSuccess ? MBERT_OK : fail_cuda(e);
}

MBERT_API int mbert_attn_ln_qkv(mbert_attn *h, const void *x, const void *norm_w, const void *wqkv,
                                int64_t total_tokens, float eps, void *qkv, void *stream)
{
    if (!h || total_tokens < 0 || total_tokens > INT32_MAX || !(eps >= 0.f) || eps > 1.f)
        return MBERT_ERR_BAD_ARG;
    const int64_t T = total_tokens;
    if (T == 0)
        return MBERT_OK;
    if (!x || !wqkv || !qkv)
        return MBERT_ERR_BAD_ARG;
    for (const void *ptr : {x, norm_w, wqkv, static_cast<const void *>(qkv)})
        if (reinterpret_cast<uintptr_t>(ptr) & 15)
            return MBERT_ERR_BAD_ARG;
    const size_t xbytes = static_cast<size_t>(T) * kHidden * 2;
    const size_t qbytes = static_cast<size_t>(T) * kQKVWidth * 2;
    const size_t wbytes = static_cast<size_t>(kQKVWidth) * kHidden * 2;
    if (ranges_overlap(x, xbytes, qkv, qbytes) || ranges_overlap(wqkv, wbytes, qkv, qbytes) ||
        (norm_w && ranges_overlap(norm_w, kHidden * 2, qkv, qbytes)))
        return MBERT_ERR_BAD_ARG;
    DeviceGuard g(h->device);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const void *a = x;
    if (norm_w) {
        const int rc = grow_rows(&h->ln, &h->ln_cap, T, kHidden);
        if (rc != MBERT_OK)
            return rc;
        a = h->ln;
    }
    QkvProjArgs q;
    if (encode_map(h, &q.tm_a, a, kHidden, T) != MBERT_OK ||
        encode_map(h, &q.tm_w, wqkv, kHidden, kQKVWidth) != MBERT_OK ||
        encode_map(h, &q.tm_y, qkv, kQKVWidth, T) != MBERT_OK)
        return MBERT_ERR_CUDA;
    q.T = T;
    q.num_ctas = h->num_sms;
    q.err = h->err;
    cudaError_t e = cudaSuccess;
    if (norm_w) {
        cudaEvent_t l0, l1;
        if (profile_events(h, MBERT_PROFILE_LAYERNORM, &l0, &l1) != MBERT_OK)
            return MBERT_ERR_CUDA;
        if (l0)
            e = cudaEventRecord(l0, st);
        if (e == cudaSuccess)
            e = launch_layernorm(static_cast<const __nv_bfloat16 *>(x),
                                 static_cast<const __nv_bfloat16 *>(norm_w), T, eps, h->ln,
                                 h->num_sms, st);
        if (e == cudaSuccess && l1)
            e = cudaEventRecord(l1, st);
        h->launches += 1;
    }
    cudaEvent_t ev0, ev1;
    if (e == cudaSuccess && profile_events(h, MBERT_PROFILE_QKV_PROJ, &ev0, &ev1) != MBERT_OK)
        return MBERT_ERR_CUDA;
    if (e == cudaSuccess && ev0)
        e = cudaEventRecord(ev0, st);
    if (e == cudaSuccess)
        e = launch_qkv_proj(q, st);
    if (e == cudaSuccess && ev1)
        e = cudaEventRecord(ev1, st);
    h->launches += 1;
    h->last_stream = st;
    return e == cudaSuccess ? MBERT_OK : fail_cuda(e);
}

MBERT_API int mbert_attn_mlp(mbert_attn *h, const void *x, const void *norm_w, const void *wi,
                             const void *wo, int64_t total_tokens, float eps, void *y, void *stream)
{
    if (!h || total_tokens < 0 || total_tokens > INT32_MAX || !(eps >= 0.f) || eps > 1.f)
        return MBERT_ERR_BAD_ARG;
    const int64_t T = total_tokens;
    if (T == 0)
        return MBERT_OK;
    if (!x || !norm_w || !wi || !wo || !y)
        return MBERT_ERR_BAD_ARG;
    for (const void *ptr : {x, norm_w, wi, wo, static_cast<const void *>(y)})
        if (reinterpret_cast<uintptr_t>(ptr) & 15)
            return MBERT_ERR_BAD_ARG;
    const size_t act = static_cast<size_t>(T) * kHidden * 2;
    const size_t wib = static_cast<size_t>(2 * kInnerMlp) * kHidden * 2;
    const size_t wob = static_cast<size_t>(kHidden) * kInnerMlp * 2;
    if (ranges_overlap(wi, wib, y, act) || ranges_overlap(wo, wob, y, act) ||
        ranges_overlap(norm_w, kHidden * 2, y, act) || (x != y && ranges_overlap(x, act, y, act)))
        return MBERT_ERR_BAD_ARG;
    DeviceGuard g(h->device);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    int rc = grow_rows(&h->ln, &h->ln_cap, T, kHidden);
    if (rc == MBERT_OK)
        rc = grow_rows(&h->mid, &h->mid_cap, T, kInnerMlp);
    if (rc != MBERT_OK)
        return rc;
    QkvProjArgs up;
    OutProjArgs down;
    if (encode_map(h, &up.tm_a, h->ln, kHidden, T) != MBERT_OK ||
        encode_map(h, &up.tm_w, wi, kHidden, 2 * kInnerMlp) != MBERT_OK ||
        encode_map(h, &up.tm_y, h->mid, kInnerMlp, T) != MBERT_OK ||
        encode_map(h, &down.tm_a, h->mid, kInnerMlp, T) != MBERT_OK ||
        encode_map(h, &down.tm_w, wo, kInnerMlp, kHidden) != MBERT_OK ||
        encode_map(h, &down.tm_x, x, kHidden, T) != MBERT_OK ||
        encode_map(h, &down.tm_y, y, kHidden, T) != MBERT_OK)
        return MBERT_ERR_CUDA;
    up.T = down.T = T;
    up.num_ctas = down.num_ctas = h->num_sms;
    up.err = down.err = h->err;
    down.x = static_cast<const __nv_bfloat16 *>(x);
    cudaError_t e = cudaSuccess;
    // one event pair per kernel while profiling
    auto timed = [&](int slot, auto &&launch) {
        cudaEvent_t e0, e1;
        if (e != cudaSuccess)
            return;
        if (profile_events(h, slot, &e0, &e1) != MBERT_OK) {
            e = cudaErrorMemoryAllocation;
            return;
        }
        if (e0)
            e = cudaEventRecord(e0, st);
        if (e == cudaSuccess)
            e = launch();
        if (e == cudaSuccess && e1)
            e = cudaEventRecord(e1, st);
        h->launches += 1;
    };
    timed(MBERT_PROFILE_LAYERNORM, [&] {
        return launch_layernorm(static_cast<const __nv_bfloat16 *>(x),
                                static_cast<const __nv_bfloat16 *>(norm_w), T, eps, h->ln,
                                h->num_sms, st);
    });
    timed(MBERT_PROFILE_MLP_UP, [&] { return launch_mlp_up(up, st); });
    timed(MBERT_PROFILE_MLP_DOWN, [&] { return launch_mlp_down(down, st); });
    h->last_stream = st;
    return e == cudaSuccess ? MBERT_OK : fail_cuda(e);
}

MBERT_API int mbert_attn_get_error(mbert_attn *h)
{
    if (!h)
        return MBERT_ERR_BAD_ARG;
    DeviceGuard g(h->device);
    if (cudaStreamSynchronize(h->last_stream) != cudaSuccess)
        return MBERT_ERR_CUDA;
    int32_t word = 0;
    if (cudaMemcpy(&word, h->err, sizeof word, cudaMemcpyDeviceToHost) != cudaSuccess ||
        cudaMemset(h->err, 0, sizeof(int32_t)) != cudaSuccess)
        return MBERT_ERR_CUDA;
    if (word & kErrTimeout)
        return MBERT_ERR_TIMEOUT;
    if (word & kErrPairTmem)
        return MBERT_ERR_CUDA;
    if (word & kErrBadCu)
        return MBERT_ERR_BAD_CU_SEQLENS;
    if (word & kErrTooLong)
        return MBERT_ERR_SEQ_TOO_LONG;
    return MBERT_OK;
}

MBERT_API int mbert_attn_selftest_timeout(mbert_attn *h, int64_t limit_us, void *stream)
{
    if (!h || limit_us <= 0 || limit_us > 2000000)
        return MBERT_ERR_BAD_ARG;
    DeviceGuard g(h->device);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaError_t e = launch_wait_timeout_selftest(
        h->err, static_cast<unsigned long long>(limit_us) * 1000ull, st);
    h->last_stream = st;
    return e == cudaSuccess ? MBERT_OK : fail_cuda(e);
}

MBERT_API int mbert_attn_profile_enable(mbert_attn *h, int enable)
{
    if (!h)
        return MBERT_ERR_BAD_ARG;
    h->profiling = enable != 0;
    return MBERT_OK;
}

MBERT_API int mbert_attn_profile_read(mbert_attn *h, double *kernel_ms, int64_t *kernel_launches,
                                      int64_t *total_launches)
{
    if (!h)
        return MBERT_ERR_BAD_ARG;
    DeviceGuard g(h->device);
    for (int k = 0; k < MBERT_PROFILE_SLOTS; ++k) {
        double ms = 0.0;
        for (size_t i = 0; i + 1 < h->ev_used[k]; i += 2) {
            float x = 0.f;
            if (cudaEventSynchronize(h->ev[k][i + 1]) != cudaSuccess ||
                cudaEventElapsedTime(&x, h->ev[k][i], h->ev[k][i + 1]) != cudaSuccess)
                return MBERT_ERR_CUDA;
            ms += x;
        }
        if (kernel_ms)
            kernel_ms[k] = ms;
        if (kernel_launches)
            kernel_launches[k] = static_cast<int64_t>(h->ev_used[k] / 2);
        h->ev_used[k] = 0;
    }
    if (total_launches)
        *total_launches = h->launches;
    h->launches = 0;
    return MBERT_OK;
}
