/*
 * mla_decode.h — C ABI of the GB300 (sm_103a) absorbed Multi-head Latent Attention decode
 * library (libmla_decode.so).
 *
 * The operation ("MLA 在极长上下文下的显存带宽突围", run-time matrix absorption;
 * "MLA & DSA 推理性能优化指南" §1.1 and §4.1): every query step of request b has H heads.
 * Head h carries an absorbed query q~ = q^C W^UK (512 values) and a decoupled-RoPE query
 * q_R (64 values).  All heads attend over one shared paged cache whose per-token entry is
 * the 512-d latent c_KV followed by the 64-d RoPE key k_R (576 values, 1152 B in bf16):
 *
 *     s_t      = softmax_scale * (q~ . c_t + q_R . k_R,t)
 *     out[b,h] = sum_t softmax(s)_t * c_t             (512 fp32 values, still latent)
 *     lse[b,h] = ln sum_t exp(s_t)                    (natural log of the scaled scores)
 *
 * W^UV is applied by the caller afterwards.  A request with no tokens gets out = 0 and
 * lse = -inf.
 *
 * Memory: every pointer argument is caller-owned DEVICE memory unless stated otherwise.
 * The library allocates nothing per call.  All calls are asynchronous on `stream`
 * (a cudaStream_t; NULL means the legacy default stream) and return as soon as the work
 * is enqueued.  Host-detectable argument errors are returned immediately and nothing is
 * enqueued.  Errors that only the GPU can see (a page id outside [0, num_pages), a token
 * index outside [-1, seq_len), a length beyond the block table, a pipeline wait that
 * exceeded its iteration limit) are recorded in a status word inside the workspace; the
 * offending access is skipped, nothing traps, and mla_decode_status() reports the code.
 *
 * Layouts (row-major, no padding):
 *   q_nope        bf16  [B][H][512]     absorbed queries
 *   q_rope        bf16  [B][H][64]      RoPE queries
 *   cache (bf16)  bf16  [num_pages][64][576]   row = latent[512] | k_rope[64]
 *   cache (fp8)   u8    [num_pages][64][656]   row = 512 e4m3 "fn" codes |
 *                                              4 fp32 scales (channel block c/128) |
 *                                              64 bf16 k_rope; latent = e4m3 * scale
 *   block_table   int32 [B][max_pages]  physical page of logical page j of request b
 *   seq_lens      int32 [B]             tokens of request b (0 allowed)
 *   indices       int32 [B][topk]       sparse: logical positions in [0, seq_len), -1 pad
 *   out           fp32  [B][H][512]
 *   lse           fp32  [B][H]
 * Token t of request b lives in page block_table[b][t / 64], row t % 64.  Rows of a
 * request's last page at or beyond seq_len are never attended and may hold anything.
 * Base pointers of q_nope, q_rope and cache must be 16-byte aligned.
 */
#ifndef MLA_DECODE_H
#define MLA_DECODE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    MLA_OK = 0,
    MLA_ERR_INVALID_ARG = 1, /* null pointer, bad size or alignment, scale not in (0,inf) */
    MLA_ERR_UNSUPPORTED = 2, /* H > 128, no sm_103a device, ...                          */
    MLA_ERR_WORKSPACE = 3,   /* workspace too small, or it does not hold a matching plan */
    MLA_ERR_CUDA = 4,        /* a CUDA runtime call failed                               */
    MLA_ERR_INDEX = 5,       /* device: page id, token index or length out of range      */
    MLA_ERR_TIMEOUT = 6,     /* device: a pipeline wait exceeded its iteration limit     */
    MLA_ERR_RANGE = 7        /* device: FP8-record decode met a value outside the fp16
                                range of its operands (|query| or 448 x scale > 65504)   */
} mla_status;

typedef enum { MLA_KV_BF16 = 0, MLA_KV_FP8_E4M3 = 1 } mla_kv_dtype;

/* Bytes of device workspace a plan for B requests of H heads needs on a GPU with
 * `num_sms` SMs (pass 0 for the current device's count).  The workspace holds the plan,
 * the split-KV partial results and the status word.  Returns 0 for invalid arguments. */
size_t mla_decode_workspace_size(int B, int H, int num_sms);

/* Split-KV planner ("Fused Reduction" of weight-absorbed decode, "MLA 最佳算子全景调研"
 * §3; variable-length paged batches, same page §2).  Reads the device array seq_lens[B]
 * on the GPU (no host synchronisation; capturable in a CUDA graph) and writes into
 * `workspace` a list of (request, token range) work items balanced over the persistent
 * decode workers, the number of splits of each request and where its partial results go.
 * With topk > 0 the plan is for mla_decode_sparse: every request is planned over its
 * topk index slots and seq_lens may be NULL.  The plan stays valid until seq_lens changes.
 * kv_dtype: the cache layout the decode will read (it sets the cost the planner charges per
 * piece; a plan of either layout is correct for both); top-k plans take MLA_KV_BF16.
 * num_sms: SMs the decode may use (0 = all SMs of the current device). */
mla_status mla_decode_plan(const int32_t *seq_lens, int B, int H, int topk, mla_kv_dtype kv_dtype,
                           int num_sms, void *workspace, size_t ws_bytes, void *stream);

/* Dense decode over the paged cache with the plan in `workspace` (built by
 * mla_decode_plan with topk = 0 for the same B, H and seq_lens).  Writes out and lse.
 * kv_dtype selects the cache layout above.  softmax_scale must be finite and > 0. */
mla_status mla_decode(const void *workspace, size_t ws_bytes, const void *q_nope,
                      const void *q_rope, const void *cache, mla_kv_dtype kv_dtype,
                      int64_t num_pages, const int32_t *block_table, int max_pages,
                      const int32_t *seq_lens, int B, int H, float softmax_scale, float *out,
                      float *lse, void *stream);

/* Token-sparse (DSA top-k) decode ("MLA & DSA 推理性能优化指南" §1.2, §4.2): request b
 * attends only over the logical positions indices[b][0..topk) that are >= 0; -1 is
 * padding.  A repeated index is attended once per occurrence.  bf16 cache only.  Needs
 * a plan built with the same topk. */
mla_status mla_decode_sparse(const void *workspace, size_t ws_bytes, const void *q_nope,
                             const void *q_rope, const void *cache, int64_t num_pages,
                             const int32_t *block_table, int max_pages,
                             const int32_t *seq_lens, const int32_t *indices, int topk, int B,
                             int H, float softmax_scale, float *out, float *lse,
                             void *stream);

/* Synchronises `stream`, returns the first device-side error recorded in the workspace
 * since the last call (MLA_OK if none) and clears it. */
mla_status mla_decode_status(void *workspace, size_t ws_bytes, void *stream);

/* Static description of a status code. */
const char *mla_status_string(mla_status status);

/* Limit, in SM clock cycles, of every pipeline wait inside the decode kernel, for the
 * mla_decode / mla_decode_sparse / mla_decode_static calls made after it in this process
 * (0 restores the default, about two seconds).  A wait that runs out records
 * MLA_ERR_TIMEOUT in the status word; the kernel then stops issuing work, gives copies and
 * tensor-core operations already in flight a bounded time to land, releases its tensor
 * memory and returns, so the device and the workspace stay usable (the call's out and lse
 * are then undefined).  The default is far above any healthy wait; a tiny limit makes
 * waits run out on purpose, which is how the timeout path is tested.  Returns
 * MLA_ERR_INVALID_ARG for a negative limit. */
mla_status mla_decode_set_wait_limit(int64_t cycles);

/* Test hook for the timeout path: while enabled (enable != 0), every decode call made
 * afterwards in this process has its tensor-core issuer wait, before it issues anything,
 * on a barrier that nothing ever completes.  That wait runs out after the wait limit
 * above, the call records MLA_ERR_TIMEOUT and winds down as described there, and the
 * device stays usable.  It exists so that tests can make a wait run out on purpose without
 * any fault; production code leaves it disabled (the default). */
mla_status mla_decode_inject_stall(int enable);

/* Dense decode (plan + decode + split merge) that allocates nothing and takes no
 * workspace.  It is for callers that cannot allocate device memory at decode time: all
 * memory handed to an arena up front, a real-time loop that must not call cudaMalloc
 * (it may synchronise the device), or a plugin whose host application owns every
 * allocation.  The pages have no counterpart; this is a usage variant of mla_decode.
 * The workspace is a fixed 48 MiB array in the library's device image, held on every
 * GPU that uses this call until the process exits.  B x H beyond what the array holds
 * (mla_decode_workspace_size(B, H, 0) > 48 MiB, e.g. more than about 110 requests of 128
 * heads on a 152-SM GB300) returns MLA_ERR_WORKSPACE and enqueues nothing.
 * All calls on one device share the array: calls whose work overlaps on the GPU (two
 * streams) race; calls on one stream are safe.  The first call on a device does a
 * one-time set-up (it looks up the array's device address); make it before any stream
 * capture.  Arguments are those of mla_decode; device_status (optional, device int32)
 * receives this call's status word (MLA_OK or a device-side error code) in stream order. */
mla_status mla_decode_static(const void *q_nope, const void *q_rope, const void *cache,
                             mla_kv_dtype kv_dtype, int64_t num_pages,
                             const int32_t *block_table, int max_pages,
                             const int32_t *seq_lens, int B, int H, float softmax_scale,
                             float *out, float *lse, int32_t *device_status, void *stream);

/* Cache append, the step after each decode step ("MLA & DSA 推理性能优化指南", §4: the
 * decode figure appends each step's output token to the cache): request b's new token —
 * c_kv[b][0..512) (its latent) and k_rope[b][0..64) (its RoPE key), bf16 — goes to logical
 * position positions[b]: page block_table[b][positions[b] / 64], row positions[b] % 64.
 * A bf16 cache receives the 576 values.  An FP8 cache (§5.3; the record layout above)
 * receives, per block of 128 latent channels, scale = max|x| / 448 computed in binary32
 * (1 for an all-zero block) and each code the e4m3 "fn" value nearest to x / scale (binary32
 * division; clamped to +-448; ties to the even code), then the four scales and the 64 RoPE
 * values as given.  positions[b] < 0 skips request b.  A position beyond the block table
 * or a page id outside [0, num_pages) skips the request and records MLA_ERR_INDEX in
 * *device_status (optional, device int32; the first error wins, nothing is cleared).
 * cache, c_kv and k_rope must be 16-byte aligned device pointers; block_table, positions
 * device int32; c_kv finite.  Rows of different requests must differ (each request
 * writes one row). */
mla_status mla_cache_append(void *cache, mla_kv_dtype kv_dtype, int64_t num_pages,
                            const int32_t *block_table, int max_pages, const int32_t *positions,
                            const void *c_kv, const void *k_rope, int B, int32_t *device_status,
                            void *stream);

/* Query absorption before the decode ("MLA 在极长上下文下的显存带宽突围", run-time matrix
 * absorption: q~ = q^C W^UK, the up-projection folded into the query so that the score is
 * taken against the 512-d latent): for every request b and head h,
 *   q_nope[b][h][c] = bf16_rne( sum_k q_c[b][h][k] * w_uk[h][k][c] ),  c < 512, k < 128,
 * with bf16 inputs, fp32 accumulation (tensor cores) and one rounding to bf16, ready for
 * mla_decode.  q_c bf16 [B][H][128] (the per-head nope query, d_h = 128 of the guide's
 * §5.1), w_uk bf16 [H][128][512], q_nope bf16 [B][H][512]; all device pointers, 16-byte
 * aligned, caller-owned.  Launched as a programmatic dependent of the previous kernel on
 * `stream` (it waits for that kernel before reading q_c).  *device_status (optional,
 * device int32) receives MLA_ERR_TIMEOUT if an internal wait gives up. */
mla_status mla_absorb_query(const void *q_c, const void *w_uk, int B, int H, void *q_nope,
                            int32_t *device_status, void *stream);

/* Value up-projection after the decode ("MLA & DSA 推理性能优化指南", §1.1: the absorbed
 * path attends in latent space and W^UV maps the result back to each head's value space):
 *   y[b][h][j] = sum_c bf16_rne(out[b][h][c]) * w_uv[h][j][c],  j < 128, c < 512,
 * fp32 accumulation (tensor cores; the latent output is rounded to bf16, the operand type of
 * the bf16 MMA), y fp32.  out fp32 [B][H][512] (mla_decode's output), w_uv bf16
 * [H][128][512], y fp32 [B][H][128]; device pointers, 16-byte aligned, caller-owned.
 * Launched as a programmatic dependent of the previous kernel on `stream` (it waits for
 * that kernel before reading out).  device_status as for mla_absorb_query. */
mla_status mla_project_output(const float *out, const void *w_uv, int B, int H, float *y,
                              int32_t *device_status, void *stream);

/* DSA token selection ("MLA & DSA 推理性能优化指南" §1.2: a lightweight indexer scores every
 * earlier token and only the top-k join the sparse attention; "GPU partial sort").  For each
 * request b with L = seq_lens[b] (0 <= L <= Lmax), keeps the min(k, L) positions of [0, L)
 * with the highest scores[b * row_stride + t] (fp32; equal scores go to the lower position;
 * -0.0 equals +0.0) and writes them to indices[b][0..k) in ascending position order, padded
 * with -1 — the index list mla_decode_sparse takes.  Scores must not be NaN.  A length
 * outside [0, Lmax] writes k times -1 for that request and records MLA_ERR_INDEX in
 * *device_status (optional, device int32).  scores: device fp32, 16-byte aligned, row_stride
 * a multiple of 4 and >= Lmax; seq_lens, indices: device int32 ([B], [B][k]).  k >= 1. */
mla_status mla_topk_select(const float *scores, int64_t row_stride, int Lmax,
                           const int32_t *seq_lens, int B, int k, int32_t *indices,
                           int32_t *device_status, void *stream);

/* Non-absorbed prefill, step 1 ("MLA & DSA 推理性能优化指南" §3.1 and §1.1: the latents are
 * decompressed before standard attention): for a sequence of L tokens whose entries
 * [L][576] (latent c_t | RoPE key, bf16, the cache entry layout, contiguous) are given,
 *   k_nope[h][t][j] = bf16_rne( sum_c w_uk[h][j][c] c_t[c] ),
 *   v[h][t][j]      = bf16_rne( sum_c w_uv[h][j][c] c_t[c] ),   j < 128, c < 512,
 * fp32 accumulation on the tensor cores.  w_uk, w_uv bf16 [H][128][512]; k_nope, v bf16
 * [H][L][128].  Device pointers, 16-byte aligned, caller-owned; a programmatic dependent of
 * the previous kernel on `stream`.  *device_status (optional) gets MLA_ERR_TIMEOUT if an
 * internal wait gives up. */
mla_status mla_prefill_decompress(const void *entries, int L, const void *w_uk, const void *w_uv,
                                  int H, void *k_nope, void *v, int32_t *device_status,
                                  void *stream);

/* Non-absorbed prefill, step 2 ("MLA 最佳算子全景调研" §4: a FlashAttention variant with
 * 192-wide keys and 128-wide values): causal multi-head attention of query i over keys
 * t <= i of the same sequence,
 *   s_t = softmax_scale * (q_nope[i][h] . k_nope[h][t] + q_rope[i][h] . k_R[t]),
 *   out[i][h] = sum_t softmax(s)_t v[h][t]  (fp32),  lse[i][h] = ln sum_t e^{s_t},
 * with k_R[t] = entries[t][512..576).  q_nope bf16 [L][H][128], q_rope bf16 [L][H][64],
 * k_nope and v as mla_prefill_decompress writes them, out fp32 [L][H][128], lse fp32
 * [L][H].  Scores and the softmax in fp32, probabilities rounded to bf16 for the
 * probability x value product, fp32 accumulation.  softmax_scale finite and > 0.  Pointers
 * as above; a programmatic dependent of the previous kernel on `stream`. */
mla_status mla_prefill_attention(const void *q_nope, const void *q_rope, const void *entries,
                                 const void *k_nope, const void *v, int L, int H,
                                 float softmax_scale, float *out, float *lse,
                                 int32_t *device_status, void *stream);

/* Host twin of mla_decode_plan for tests and tooling: plans from a HOST array
 * seq_lens[B] (NULL with topk > 0) into a HOST buffer of mla_decode_workspace_size()
 * bytes, producing exactly the bytes the device planner writes into the plan region.
 * num_sms must be > 0. */
mla_status mla_decode_plan_host(const int32_t *seq_lens, int B, int H, int topk, mla_kv_dtype kv_dtype,
                                int num_sms, void *workspace_host, size_t ws_bytes);

#ifdef __cplusplus
}
#endif
#endif /* MLA_DECODE_H */
