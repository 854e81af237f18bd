/*
 * mbert_attn: the bidirectional self-attention block of ModernBERT-base as a
 * C-ABI library for NVIDIA GB300 (sm_103a).
 *
 * What one call computes (page title, section):
 *  - Input: the fused Wqkv output, one row of 2304 bf16 numbers per token,
 *    cut as (3, 12, 64): columns 0..767 are Q, 768..1535 K, 1536..2303 V,
 *    head h at columns h*64 .. h*64+63 of each block ("ModernBERT-base
 *    Architecture Teardown", "How Does ModernBERT Make Q, K and V?";
 *    "ModernBERT" (candding), "The tensors").
 *  - RoPE, rotate-half over the full 64-wide head, on Q and K only; pair m
 *    turns by pos * base^(-2m/64); base 160000 on global layers, 10000 on
 *    local layers (teardown, "How Does RoPE Work With Two Bases?"; candding,
 *    "The two rope tables").  Positions restart at 0 in every sequence.
 *  - Scores q.k / sqrt(64), softmax along the keys, weighted blend of V, no
 *    causal mask (teardown, "How Does Self-Attention Work?").
 *  - Local layers keep key j for query i when |i - j| <= 64; global layers
 *    keep every key of the sequence (teardown, "What Are Local and Global
 *    Attention?"; candding, "The alternating attention").
 *  - Sequences are unpadded and packed back to back; cu_seqlens holds their
 *    offsets.  A query never sees keys of another sequence, which is what a
 *    padding mask achieves for a padded batch ("Encoder-only models"
 *    (rayaq), padding mask; teardown, "What Is ModernBERT-base?", unpadding).
 *  - Output: out[t, h*64 + d], 768 bf16 per token, heads in input order,
 *    ready for Wo (teardown, "How Does ModernBERT Make Q, K and V?").
 *
 * Conventions for every entry point:
 *  - Status: 0 on success, a negative MBERT_ERR_* code otherwise.  Host-side
 *    argument checks are synchronous and enqueue nothing when they fail.
 *    Checks that need device data (cu_seqlens contents) run on the GPU and
 *    are reported later by mbert_attn_get_error().
 *  - Pointers marked "device" must be CUDA device (or managed) memory on the
 *    handle's device; "host" pointers are ordinary host memory.
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *    stream).  All device work is enqueued asynchronously on it; the caller
 *    keeps ownership of the stream and of every buffer it passes.
 *  - A handle may be used from one host thread at a time.
 */
#ifndef MBERT_ATTN_H
#define MBERT_ATTN_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Opaque handle: owns the two RoPE cos/sin tables, the device work-list
 * workspace, the rotated-operand scratch (with the rotated rows' norms that
 * global layers use to bound their scores) and the device error word. */
typedef struct mbert_attn mbert_attn;

/* Layer kinds.  Layer i of the 22-layer stack is global iff i % 3 == 0
 * (teardown, "What Are Local and Global Attention?"). */
enum {
    MBERT_GLOBAL = 0,
    MBERT_LOCAL = 1
};

/* Status codes. */
enum {
    MBERT_OK = 0,
    MBERT_ERR_BAD_ARG = -1,        /* null/misaligned/aliased pointer, bad size or kind */
    MBERT_ERR_UNSUPPORTED = -2,    /* config other than 12 heads x 64, or no sm_103 device */
    MBERT_ERR_SEQ_TOO_LONG = -3,   /* a sequence longer than the handle's max_seqlen */
    MBERT_ERR_BAD_CU_SEQLENS = -4, /* cu_seqlens[0] != 0, decreasing, or cu[n] != T (device-detected) */
    MBERT_ERR_TIMEOUT = -5,        /* a kernel's bounded wait ran out; results are invalid */
    MBERT_ERR_CUDA = -6,           /* a CUDA runtime call failed */
    MBERT_ERR_OOM = -7             /* device allocation failed */
};

/* Create-time configuration. */
typedef struct {
    int heads;            /* must be 12 */
    int head_dim;         /* must be 64 */
    int half_window;      /* local band half-width, |i - j| <= half_window (64), 0..128 */
    int max_seqlen;       /* longest sequence accepted; sizes the RoPE tables (8192) */
    double theta_global;  /* RoPE base of global layers (160000) */
    double theta_local;   /* RoPE base of local layers (10000) */
} mbert_attn_config;

/* Fill *cfg with ModernBERT-base's values: 12, 64, 64, 8192, 160000, 10000. */
int mbert_attn_default_config(mbert_attn_config *cfg);

/* Create a handle on CUDA device `device` (host pointer out, host pointer
 * cfg; cfg == NULL means the defaults).  Allocates the RoPE tables
 * (2 x max_seqlen x 32 x (cos, sin) fp32, computed in fp64 on the host) and a
 * small workspace.  Synchronous.  On failure *out is NULL. */
int mbert_attn_create(mbert_attn **out, const mbert_attn_config *cfg, int device);

/* Grow the workspace so that later forward calls with up to `max_tokens`
 * packed tokens in up to `max_seqs` sequences allocate nothing.  Optional:
 * mbert_attn_forward grows it on demand (a synchronous cudaMalloc). */
int mbert_attn_reserve(mbert_attn *h, int64_t max_tokens, int64_t max_seqs);

/* The attention block for one layer.
 *   qkv          device, bf16 [total_tokens][2304] row-major, 16-byte aligned.
 *   cu_seqlens   device, int32 [n_seqs + 1]; cu[0] = 0, non-decreasing,
 *                cu[n_seqs] = total_tokens.  Empty sequences are allowed.
 *   n_seqs       >= 0; total_tokens >= 0 (0 enqueues nothing).
 *   max_seqlen   caller's bound on the longest sequence (<= the handle's
 *                max_seqlen, else MBERT_ERR_SEQ_TOO_LONG); a longer sequence
 *                found on the device sets MBERT_ERR_SEQ_TOO_LONG.
 *   layer_kind   MBERT_GLOBAL or MBERT_LOCAL.
 *   out          device, bf16 [total_tokens][768], 16-byte aligned, must not
 *                overlap qkv.  Every row of every sequence is written.
 * Enqueues a few kernels on `stream`; when the device-side checks fail the
 * attention kernels write nothing and the error is reported by
 * mbert_attn_get_error(). */
int mbert_attn_forward(mbert_attn *h, const void *qkv, const int32_t *cu_seqlens,
                       int n_seqs, int64_t total_tokens, int max_seqlen,
                       int layer_kind, void *out, void *stream);

/* The attention block for a padded batch: B rows of S tokens with an
 * attention mask of 1 for a real token and 0 for a pad ("ModernBERT-base
 * Architecture Teardown", the tokenizer with padding=True: the 0s of the
 * mask become a mask inside attention, so no real token takes information
 * from a pad; "Encoder-only models", "Padding and the key padding mask").
 * Each row's real tokens, in order, are one sequence: a real token's
 * position is its rank among its row's real tokens (its index for a
 * right-padded row), and only real tokens of the same row are keys.
 *   qkv             device bf16 [batch][seq_len][2304], 16-byte aligned.
 *   attention_mask  device int32 [batch][seq_len]: non-zero = real token.
 *   seq_len         <= the handle's max_seqlen (else MBERT_ERR_SEQ_TOO_LONG);
 *                   batch * seq_len < 2^31.
 *   out             device bf16 [batch][seq_len][768], 16-byte aligned, must
 *                   not overlap qkv or the mask.  Every row is written: a
 *                   real token's attention output, zeros for a pad.
 * The call packs the real rows into handle-owned buffers (grown with
 * cudaMalloc when needed), runs mbert_attn_forward's kernels on them and
 * unpacks the result, all on `stream`; calls sharing a handle must not
 * overlap on the GPU.  Returns as mbert_attn_forward. */
int mbert_attn_forward_padded(mbert_attn *h, const void *qkv, const int32_t *attention_mask,
                              int batch, int seq_len, int layer_kind, void *out, void *stream);

/* Debug/verification entry: for every packed row, the number of keys the
 * attention kernel's tile schedule and mask admit for that query (the size
 * of its admitted set), computed by the same device code the forward pass
 * uses to choose and mask key tiles.  counts: device int32 [total_tokens].
 * Other arguments as for mbert_attn_forward. */
int mbert_attn_key_counts(mbert_attn *h, const int32_t *cu_seqlens, int n_seqs,
                          int64_t total_tokens, int max_seqlen, int layer_kind,
                          int32_t *counts, void *stream);

/* The step before the attention block: its input qkv from the residual
 * stream x, qkv = LayerNorm(x) Wqkv^T.  The LayerNorm is bias-free: each
 * row minus its mean, divided by sqrt(population variance + eps), times the
 * weight ("ModernBERT-base Architecture Teardown", "What Does LayerNorm
 * Do?"); layer 0 has no norm before attention ("ModernBERT" (candding), "The
 * pre-norm layer and the final norm").  Wqkv turns 768 numbers into 2304 =
 * (3, 12, 64), Q, K, V head by head (teardown, "How Does ModernBERT Make Q,
 * K and V?"), the layout mbert_attn_forward reads.
 *   x       device bf16 [total_tokens][768], row-major.
 *   norm_w  device bf16 [768], the norm's weight; NULL for no norm
 *           (layer 0: qkv = x Wqkv^T).
 *   wqkv    device bf16 [2304][768], row-major, [out][in].
 *   eps     added to the variance under the square root (1e-5 in
 *           ModernBERT-base); 0 <= eps <= 1.
 *   qkv     device bf16 [total_tokens][2304], row-major: written; must not
 *           overlap x, norm_w or wqkv.
 * The norm runs in fp32 and its output is rounded to bf16 (the GEMM's
 * operand) in a handle-owned buffer of total_tokens x 768 (grown with
 * cudaMalloc when a call needs more; mbert_attn_reserve does not size it);
 * the products accumulate in fp32 and qkv is rounded to bf16 once.  All
 * pointers 16-byte aligned; the caller owns every buffer.  Returns MBERT_OK;
 * MBERT_ERR_BAD_ARG for a null handle or buffer, a misaligned or overlapping
 * buffer, a bad eps or total_tokens outside [0, 2^31); MBERT_ERR_OOM if the
 * buffer cannot grow; MBERT_ERR_CUDA on a launch failure.  Calls that share
 * a handle must not overlap on the GPU (they share the buffer).  Device
 * timeouts are reported by mbert_attn_get_error(). */
int mbert_attn_ln_qkv(mbert_attn *h, const void *x, const void *norm_w, const void *wqkv,
                      int64_t total_tokens, float eps, void *qkv, void *stream);

/* The layer's second block, the GeGLU MLP with its pre-norm and residual:
 * y = x + (GELU(g) * u) Wo^T with g, u the first and second halves of
 * LayerNorm(x) Wi^T ("ModernBERT-base Architecture Teardown", "What Does
 * the GeGLU MLP Do?": Wi makes two vectors of 1152, the first goes through
 * GELU and the second multiplies it, Wo brings 1152 back to 768;
 * "modernbert-base" (nest.franknoh), "The fused projections": the first
 * half of Wi's output is the GELU branch).  GELU is the exact erf form
 * ("ModernBERT" (candding), "The feed-forward halves"); the LayerNorm is as
 * in mbert_attn_ln_qkv.
 *   x       device bf16 [total_tokens][768]: the residual stream.
 *   norm_w  device bf16 [768]: the MLP norm's weight (not NULL).
 *   wi      device bf16 [2304][768], [out][in].
 *   wo      device bf16 [768][1152], [out][in].
 *   eps     as in mbert_attn_ln_qkv.
 *   y       device bf16 [total_tokens][768]: written.  y may be x itself
 *           (in-place update); it must not overlap the weights, and must
 *           overlap x either exactly or not at all.
 * Three kernels: the norm (fp32, bf16 result), Wi with the GeGLU in its
 * epilogue (fp32 accumulation, GELU(g) * u rounded to bf16), Wo with the
 * residual (fp32, y rounded to bf16 once).  The norm's output and the
 * [total_tokens][1152] intermediate live in handle-owned buffers (grown
 * with cudaMalloc when needed); calls sharing a handle must not overlap on
 * the GPU.  All pointers 16-byte aligned.  Returns as mbert_attn_ln_qkv. */
int mbert_attn_mlp(mbert_attn *h, const void *x, const void *norm_w, const void *wi,
                   const void *wo, int64_t total_tokens, float eps, void *y, void *stream);

/* The step after the attention block: the output projection with the
 * residual add, y = x + a Wo^T ("ModernBERT-base Architecture Teardown",
 * "How Does ModernBERT Make Q, K and V?": Wo maps the joined heads back from
 * 768 to 768, stored [out, in]; "ModernBertModel", "Implementing it":
 * x = x + a Wo^T).
 *   a   device bf16 [total_tokens][768], row-major: the attention block's out.
 *   wo  device bf16 [768][768], row-major, [out][in].
 *   x   device bf16 [total_tokens][768], row-major: the residual stream.
 *   y   device bf16 [total_tokens][768], row-major: written.  y may be x
 *       itself (in-place update); it must not overlap a or wo, and must
 *       overlap x either exactly or not at all.
 * Products accumulate in fp32; y is rounded to bf16 (nearest even) once.
 * All pointers 16-byte aligned; the caller owns every buffer.  Returns
 * MBERT_OK; MBERT_ERR_BAD_ARG for a null handle or buffer, a misaligned or
 * overlapping buffer, or total_tokens outside [0, 2^31); MBERT_ERR_CUDA on a
 * launch failure.  Device timeouts are reported by mbert_attn_get_error(). */
int mbert_attn_out_proj(mbert_attn *h, const void *a, const void *wo, const void *x,
                        int64_t total_tokens, void *y, void *stream);

/* Wait for the handle's most recent stream, then return (and clear) the
 * device error word as a status: MBERT_OK, MBERT_ERR_BAD_CU_SEQLENS,
 * MBERT_ERR_SEQ_TOO_LONG or MBERT_ERR_TIMEOUT; MBERT_ERR_CUDA if the wait
 * itself fails. */
int mbert_attn_get_error(mbert_attn *h);

/* Diagnostic: enqueue one kernel whose bounded wait on a barrier that
 * nothing completes gives up after limit_us microseconds (1 .. 2000000),
 * exactly as the attention kernels' waits do if a transfer or an MMA never
 * completes.  Afterwards mbert_attn_get_error() returns MBERT_ERR_TIMEOUT.
 * Nothing faults or traps; the context stays usable. */
int mbert_attn_selftest_timeout(mbert_attn *h, int64_t limit_us, void *stream);

/* Largest batch the allocation-free entry point below accepts: total
 * tokens, and also sequences, per call. */
#define MBERT_NOALLOC_MAX_TOKENS 8192

/* The attention block without any device allocation.  The pages have no
 * counterpart: this exists for callers that cannot call cudaMalloc -- a
 * plugin inside a framework that owns all device memory through its own
 * pool, a service whose memory is reserved once at start-up, or a loop that
 * cannot take the device-wide synchronisation cudaMalloc/cudaFree may
 * cause.  Such callers cannot create a handle, so this call needs none.
 *   Arguments as for mbert_attn_forward, on the current CUDA device, with
 *   the ModernBERT-base defaults (half window 64, bases 160000 / 10000).
 *   device_status  device int32 or NULL: receives the device-side error bits
 *                  of this call (0 = ok, 1 = bad cu_seqlens, 2 = a sequence
 *                  longer than max_seqlen, 4 = a bounded wait timed out),
 *                  written on `stream` after the kernels.
 * Scratch memory (work list, rotated Q/K rows, RoPE tables: about 28 MiB)
 * is one static device array that every GPU that loads this part of the
 * library holds until the process exits.  total_tokens or n_seqs above
 * MBERT_NOALLOC_MAX_TOKENS, or max_seqlen above it, are rejected
 * (MBERT_ERR_BAD_ARG / MBERT_ERR_SEQ_TOO_LONG) before anything is enqueued.
 * The first call on a device does a one-time set-up (it looks up the
 * array's device address and fills the RoPE tables with blocking copies,
 * which synchronise with other work on that device); make that first call
 * before any stream capture and outside any loop that must not block.
 * Every call shares the array and overwrites what the previous call left
 * there, so two calls whose work overlaps on the GPU (e.g. on different
 * streams) race.
 * This is not the benchmarked path: for both layer kinds it runs the plan
 * and a RoPE pass into the static rotated-Q/K rows (one launch), then the generic
 * attention kernel (one CTA per 128-query block and head), not the
 * persistent kernels of mbert_attn_forward, so its speed and its fp32
 * summation order differ; its results meet the same bounds against the
 * oracle. */
int mbert_attn_forward_noalloc(const void *qkv, const int32_t *cu_seqlens, int n_seqs,
                               int64_t total_tokens, int max_seqlen, int layer_kind,
                               void *out, int32_t *device_status, void *stream);

/* Measurement.  While enabled, every mbert_attn_forward also records a
 * CUDA event pair on its stream around its attention kernel (the plan and
 * RoPE kernels before it are outside the pair), every mbert_attn_out_proj
 * one around its kernel, and every mbert_attn_ln_qkv and mbert_attn_mlp one
 * around each of their kernels.  The handle always counts the kernels it enqueues. */
int mbert_attn_profile_enable(mbert_attn *h, int enable);

/* Profile slots: the two layer kinds, the output projection, the Wqkv
 * projection, the LayerNorm (before attention or before the MLP) and the
 * MLP's two GEMMs. */
enum {
    MBERT_PROFILE_OUT_PROJ = 2,
    MBERT_PROFILE_QKV_PROJ = 3,
    MBERT_PROFILE_LAYERNORM = 4,
    MBERT_PROFILE_MLP_UP = 5,
    MBERT_PROFILE_MLP_DOWN = 6,
    MBERT_PROFILE_SLOTS = 7
};

/* Synchronise on the recorded events and return, per profile slot (index
 * MBERT_GLOBAL, MBERT_LOCAL or MBERT_PROFILE_* of the host arrays
 * kernel_ms[MBERT_PROFILE_SLOTS] and kernel_launches[MBERT_PROFILE_SLOTS]),
 * the summed kernel milliseconds and
 * the number of recorded kernels, plus the number of kernels enqueued by
 * every entry point (*total_launches).  Clears all three.  Any output
 * pointer may be NULL. */
int mbert_attn_profile_read(mbert_attn *h, double *kernel_ms, int64_t *kernel_launches,
                            int64_t *total_launches);

/* Release the handle's device memory.  NULL is allowed.  The caller must
 * make sure no enqueued work still uses the handle. */
void mbert_attn_destroy(mbert_attn *h);

/* Static, human-readable text for a status code. */
const char *mbert_attn_strerror(int status);

#ifdef __cplusplus
}
#endif

#endif /* MBERT_ATTN_H */
