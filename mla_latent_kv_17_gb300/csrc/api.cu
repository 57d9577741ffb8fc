// C ABI of libmla_decode: argument checks, the device planner, the split-KV merge kernel
// and the launches of the decode kernels.
#include <cuda_runtime.h>
#include <math.h>
#include <string.h>

#include <atomic>

#include "common.cuh"
#include "launch.h"
#include "mla_decode.h"

namespace mla {
namespace {

// ---------------------------------------------------------------------------------
// Device planner: one CTA.  Each thread owns a contiguous slice of requests; block-wide
// exclusive scans give every request its budget position, item offset and first partial
// slot, then each thread writes its requests' pieces, and one pass over the items marks
// where each unit's items begin.  Same per-request functions as the host twin, so the
// two produce identical plans.
// ---------------------------------------------------------------------------------
constexpr int kPlanThreads = 256;
constexpr int kPlanWarps = kPlanThreads / 32;

// Exclusive prefix sum of v over the block (shuffles within each warp, then one warp over
// the warp totals); *total receives the sum over the block.  sh holds kPlanWarps values.
__device__ int64_t block_exclusive_scan(int64_t v, int64_t *total, int64_t *sh) {
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    int64_t x = v;
    for (int off = 1; off < 32; off <<= 1) {
        const int64_t y = __shfl_up_sync(0xffffffffu, x, off);
        if (lane >= off) x += y;
    }
    if (lane == 31) sh[wid] = x;
    __syncthreads();
    if (wid == 0) {
        int64_t t = lane < kPlanWarps ? sh[lane] : 0;
        for (int off = 1; off < 32; off <<= 1) {
            const int64_t y = __shfl_up_sync(0xffffffffu, t, off);
            if (lane >= off) t += y;
        }
        if (lane < kPlanWarps) sh[lane] = t;
    }
    __syncthreads();
    const int64_t r = (wid > 0 ? sh[wid - 1] : 0) + x - v;
    *total = sh[kPlanWarps - 1];
    __syncthreads();  // sh is reused by the next scan
    return r;
}

// The same for three values at once (one pass of barriers for the three).
struct Sum3 {
    int64_t v[3];
};
__device__ Sum3 block_exclusive_scan3(Sum3 v, Sum3 *total, Sum3 *sh) {
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    Sum3 x = v;
    for (int off = 1; off < 32; off <<= 1) {
#pragma unroll
        for (int k = 0; k < 3; ++k) {
            const int64_t y = __shfl_up_sync(0xffffffffu, x.v[k], off);
            if (lane >= off) x.v[k] += y;
        }
    }
    if (lane == 31) sh[wid] = x;
    __syncthreads();
    if (wid == 0) {
        Sum3 t;
#pragma unroll
        for (int k = 0; k < 3; ++k) t.v[k] = lane < kPlanWarps ? sh[lane].v[k] : 0;
        for (int off = 1; off < 32; off <<= 1) {
#pragma unroll
            for (int k = 0; k < 3; ++k) {
                const int64_t y = __shfl_up_sync(0xffffffffu, t.v[k], off);
                if (lane >= off) t.v[k] += y;
            }
        }
        if (lane < kPlanWarps) sh[lane] = t;
    }
    __syncthreads();
    Sum3 r;
#pragma unroll
    for (int k = 0; k < 3; ++k) r.v[k] = (wid > 0 ? sh[wid - 1].v[k] : 0) + x.v[k] - v.v[k];
    *total = sh[kPlanWarps - 1];
    __syncthreads();
    return r;
}

__global__ void __launch_bounds__(kPlanThreads)
plan_kernel(const int32_t *seq_lens, int B, int H, int topk, int units, int ovh, unsigned char *ws, int iu_in_smem) {
    __shared__ int64_t sh[kPlanWarps];
    __shared__ Sum3 sh3[kPlanWarps];
    extern __shared__ int32_t s_iu[];  // items' units (when max_items of them fit)
    grid_dep_wait();    // seq_lens may come from the kernel before this one on the stream
    grid_dep_launch();  // the decode kernel may launch now; it waits for this plan to complete
    const WsLayout L = ws_layout(B, H, units);
    int64_t *req_start = reinterpret_cast<int64_t *>(ws + L.req_start);
    int32_t *num_splits = reinterpret_cast<int32_t *>(ws + L.num_splits);
    int32_t *split_base = reinterpret_cast<int32_t *>(ws + L.split_base);
    int32_t *unit_begin = reinterpret_cast<int32_t *>(ws + L.unit_begin);
    const int32_t *item_unit = iu_in_smem ? s_iu : reinterpret_cast<const int32_t *>(ws + L.item_unit);
    const int chunk = (B + kPlanThreads - 1) / kPlanThreads;
    const int b0 = min(B, (int)threadIdx.x * chunk), b1 = min(B, b0 + chunk);

    // budget positions: the running position stays in a register (req_start is only written)
    int64_t local = 0;
    for (int b = b0; b < b1; ++b) local += req_cost(req_tiles(seq_lens, topk, b), ovh);
    int64_t total;
    const int64_t pos0 = block_exclusive_scan(local, &total, sh);
    const int64_t per = plan_budget(total, units, topk > 0 ? req_cost(req_tiles(seq_lens, topk, 0), ovh) : 0, B, ovh);

    // With at most one request per thread, its cut stays in a register and every thread then
    // emits one work item at a time (a request cut into many pieces is not left to one thread);
    // otherwise each thread emits its requests' items itself.
    const bool one_each = B <= kPlanThreads;
    __shared__ int32_t s_off[kPlanThreads + 1], s_len[kPlanThreads], s_slot[kPlanThreads];
    __shared__ ReqSplit s_rs[kPlanThreads];
    ReqSplit r_one{};
    int64_t n_local = 0, s_local = 0, r_local = 0;
    {
        int64_t pos = pos0;
        for (int b = b0; b < b1; ++b) {
            const int32_t tiles = req_tiles(seq_lens, topk, b);
            const ReqSplit r = req_split(pos, tiles, per, units, ovh);
            r_one = r;
            req_start[b] = pos;
            n_local += r.n;
            if (r.n > 1) {
                s_local += r.n;
                ++r_local;
            }
            pos += req_cost(tiles, ovh);
        }
    }
    Sum3 tot;
    const Sum3 ex = block_exclusive_scan3(Sum3{{n_local, s_local, r_local}}, &tot, sh3);
    const int64_t n_total = tot.v[0], s_total = tot.v[1], r_total = tot.v[2];
    int64_t off = ex.v[0], slot = ex.v[1], rpos = ex.v[2];
    int32_t *split_list = reinterpret_cast<int32_t *>(ws + L.split_list);
    int32_t *iu_copy = iu_in_smem ? s_iu : nullptr;
    {
        int64_t pos = pos0;
        for (int b = b0; b < b1; ++b) {
            const int32_t tiles = req_tiles(seq_lens, topk, b);
            const ReqSplit r = one_each ? r_one : req_split(pos, tiles, per, units, ovh);
            const int32_t sb = r.n > 1 ? (int32_t)slot : -1;
            num_splits[b] = r.n;
            split_base[b] = sb;
            if (one_each) {
                s_off[b] = (int32_t)off;
                s_rs[b] = r;
                s_len[b] = req_len(seq_lens, topk, b);
                s_slot[b] = sb;
            } else {
                emit_request(ws, L, seq_lens, topk, b, pos, per, units, ovh, (int32_t)off, sb, iu_copy);
            }
            off += r.n;
            if (r.n > 1) {
                slot += r.n;
                split_list[rpos++] = b;
            }
            pos += req_cost(tiles, ovh);
        }
    }
    if (one_each) {
        __syncthreads();  // s_off, s_rs, s_len, s_slot are complete
        for (int32_t i = threadIdx.x; i < (int32_t)n_total; i += kPlanThreads) {
            // the request holding item i: the last b with s_off[b] <= i (every request has an item)
            int lo = 0, hi = B - 1;
            while (lo < hi) {
                const int mid = (lo + hi + 1) >> 1;
                if (s_off[mid] <= i) lo = mid;
                else hi = mid - 1;
            }
            emit_piece(ws, L, lo, s_len[lo], s_rs[lo], i - s_off[lo], per, units, i, s_slot[lo], iu_copy);
        }
    }
    __syncthreads();  // item_unit is complete (shared, or global writes of this block)
    // unit_begin[u] = first item whose unit is >= u (items are grouped by unit in order):
    // item i starts the units (unit of item i-1, unit of item i]
    const int32_t n = (int32_t)n_total;
    for (int32_t i = threadIdx.x; i < n; i += kPlanThreads) {
        const int32_t uc = item_unit[i], up = i == 0 ? -1 : item_unit[i - 1];
        for (int32_t u = up + 1; u <= uc; ++u) unit_begin[u] = i;
    }
    const int32_t last = n > 0 ? item_unit[n - 1] : -1;
    for (int u = threadIdx.x; u <= units; u += kPlanThreads)
        if (u > last) unit_begin[u] = n;
    if (threadIdx.x == 0) {
        write_header(ws, L, B, H, topk, units, n, per, (int32_t)s_total, (int32_t)r_total, ovh);
        *reinterpret_cast<int *>(ws + L.status) = 0;
    }
}

// ---------------------------------------------------------------------------------
// Merge of split-KV partial results through their log-sum-exp:
//   lse = ln sum_i exp(lse_i),  out = sum_i exp(lse_i - lse) * out_i,
// taken online over groups of four pieces (running maximum M and sum Z of exp(lse_i - M)),
// so that a group's loads (its lse_i and rows) are in flight together.  A persistent grid
// (kCombineCtasPerSm CTAs per SM): warp w of the grid merges the (request, head) tasks
// w, w + warps, ... over the split requests the plan lists; a lane covers 16 of the 512
// columns, so every load and store of a warp spans 512 contiguous bytes.  Requests with a
// single piece were written directly by the decode kernel.  Launched as a programmatic
// dependent of the decode kernel: it waits for it before reading anything.
// ---------------------------------------------------------------------------------
constexpr int kCombineThreads = 256;
constexpr int kCombineCtasPerSm = 2;
constexpr int kCombineSmemReqs = 1024;  // split requests whose (b, n, s0) are staged in shared memory

__global__ void __launch_bounds__(kCombineThreads, kCombineCtasPerSm)
combine_kernel(DecodeArgs a) {
    __shared__ int32_t s_b[kCombineSmemReqs], s_n[kCombineSmemReqs], s_s0[kCombineSmemReqs];
    grid_dep_wait();
    grid_dep_launch();  // the next kernel on the stream may launch (it waits for this one)
    if (!plan_matches(a)) return;
    const unsigned char *ws = a.ws;
    const int H = a.H;
    const PlanHeader *hd = reinterpret_cast<const PlanHeader *>(ws);
    const WsLayout L = ws_layout(hd->B, hd->H, hd->num_units);
    const int nsr = hd->num_split_reqs;
    if (nsr <= 0) return;
    const int32_t *split_list = reinterpret_cast<const int32_t *>(ws + L.split_list);
    const int32_t *num_splits = reinterpret_cast<const int32_t *>(ws + L.num_splits);
    const int32_t *split_base = reinterpret_cast<const int32_t *>(ws + L.split_base);
    for (int k = threadIdx.x; k < nsr && k < kCombineSmemReqs; k += kCombineThreads) {
        const int b = split_list[k];
        s_b[k] = b;
        s_n[k] = num_splits[b];
        s_s0[k] = split_base[b];
    }
    __syncthreads();
    const float *part_lse = reinterpret_cast<const float *>(ws + L.part_lse);
    const float4 *part_o = reinterpret_cast<const float4 *>(ws + L.part_o);
    const int64_t ostep = (int64_t)H * (kDLatent / 4);  // one piece to the next, in float4
    const int lane = threadIdx.x & 31;
    const int64_t nw = (int64_t)gridDim.x * (kCombineThreads / 32);
    const int64_t ntasks = (int64_t)nsr * H;
    for (int64_t t = (int64_t)blockIdx.x * (kCombineThreads / 32) + (threadIdx.x >> 5); t < ntasks; t += nw) {
        const int k = (int)(t / H), h = (int)(t % H);
        int b, n, s0;
        if (k < kCombineSmemReqs) {
            b = s_b[k];
            n = s_n[k];
            s0 = s_s0[k];
        } else {
            b = split_list[k];
            n = num_splits[b];
            s0 = split_base[b];
        }
        const float *plse = part_lse + (int64_t)s0 * H + h;
        const float4 *po = part_o + ((int64_t)s0 * H + h) * (kDLatent / 4);
        float M = -INFINITY, Z = 0.f;
        float4 acc[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) acc[q] = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int i0 = 0; i0 < n; i0 += 4) {
            float li[4];
            float4 v[4][4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int i = i0 + j;
                li[j] = i < n ? plse[(int64_t)i * H] : -INFINITY;
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    v[j][q] = i < n ? po[i * ostep + lane + 32 * q] : make_float4(0.f, 0.f, 0.f, 0.f);
            }
            float mn = M;
#pragma unroll
            for (int j = 0; j < 4; ++j) mn = fmaxf(mn, li[j]);
            if (mn == -INFINITY) continue;  // every piece so far is empty
            const float r = exp2f((M - mn) * kLog2e);  // 0 while M is -inf
            Z *= r;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                acc[q].x *= r;
                acc[q].y *= r;
                acc[q].z *= r;
                acc[q].w *= r;
            }
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const float wt = exp2f((li[j] - mn) * kLog2e);  // 0 for an empty or absent piece
                Z += wt;
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    acc[q].x = fmaf(wt, v[j][q].x, acc[q].x);
                    acc[q].y = fmaf(wt, v[j][q].y, acc[q].y);
                    acc[q].z = fmaf(wt, v[j][q].z, acc[q].z);
                    acc[q].w = fmaf(wt, v[j][q].w, acc[q].w);
                }
            }
            M = mn;
        }
        const float inv = Z > 0.f ? 1.f / Z : 0.f;
        float4 *dst = reinterpret_cast<float4 *>(a.out + ((int64_t)b * H + h) * kDLatent);
#pragma unroll
        for (int q = 0; q < 4; ++q)
            dst[lane + 32 * q] = make_float4(acc[q].x * inv, acc[q].y * inv, acc[q].z * inv, acc[q].w * inv);
        if (lane == 0) a.lse[(int64_t)b * H + h] = M == -INFINITY ? -INFINITY : M + logf(Z);
    }
}

int device_sm_count() {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    return sms;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Limit of one pipeline wait in the decode kernel (SM clock cycles), for calls made from now on.
std::atomic<long long> g_wait_cycles{kDefaultWaitCycles};
// Injected stall for tests of the timeout path (mla_decode_inject_stall).
std::atomic<int> g_stall_test{0};

mla_status check_common(const void *ws, size_t ws_bytes, const void *q_nope, const void *q_rope,
                        const void *cache, int64_t num_pages, const int32_t *block_table,
                        int max_pages, const int32_t *seq_lens, int B, int H, float scale,
                        const float *out, const float *lse) {
    if (!ws || !q_nope || !q_rope || !cache || !block_table || !seq_lens || !out || !lse)
        return MLA_ERR_INVALID_ARG;
    if (B < 1 || H < 1 || max_pages < 1 || num_pages < 1) return MLA_ERR_INVALID_ARG;
    if (H > kMaxHeads) return MLA_ERR_UNSUPPORTED;
    if (num_pages > (int64_t)(INT32_MAX / kPageRows)) return MLA_ERR_UNSUPPORTED;
    if (!isfinite(scale) || !(scale > 0.f)) return MLA_ERR_INVALID_ARG;
    if (!aligned16(q_nope) || !aligned16(q_rope) || !aligned16(cache) || !aligned16(out))
        return MLA_ERR_INVALID_ARG;
    if (ws_bytes < ws_layout(B, H, 1).plan_end) return MLA_ERR_WORKSPACE;
    return MLA_OK;
}

// Work units for `num_sms` SMs: one per SM pair, capped by the clusters that fit at once.
int units_for(int num_sms) {
    int u = num_units_for(num_sms);
    const int mc = sm103_max_units();
    if (mc > 0 && u > mc) u = mc;
    return u;
}

mla_status run_decode(const DecodeArgs &a, cudaStream_t stream) {
    int sms = device_sm_count();
    if (sms <= 0) return MLA_ERR_CUDA;
    const int units = units_for(sms);
    cudaError_t e;
    e = launch_decode_sm103(a, units, stream);  // dense bf16, DSA sparse, or FP8 records
    if (e != cudaSuccess) return MLA_ERR_CUDA;
    // the merge: a programmatic dependent of the decode kernel (it may launch while the
    // decode's last CTAs finish, and waits for them before it reads anything)
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(kCombineCtasPerSm * sms, 1, 1);
    cfg.blockDim = dim3(kCombineThreads, 1, 1);
    cfg.stream = stream;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr.val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, combine_kernel, a) != cudaSuccess) return MLA_ERR_CUDA;
    return MLA_OK;
}

}  // namespace
}  // namespace mla

using namespace mla;

extern "C" {

size_t mla_decode_workspace_size(int B, int H, int num_sms) {
    if (B < 1 || H < 1 || H > kMaxHeads || num_sms < 0) return 0;
    if (num_sms == 0) num_sms = device_sm_count();
    if (num_sms <= 0) return 0;
    return ws_layout(B, H, units_for(num_sms)).total;
}

mla_status mla_decode_plan(const int32_t *seq_lens, int B, int H, int topk, mla_kv_dtype kv_dtype,
                           int num_sms, void *workspace, size_t ws_bytes, void *stream) {
    if (!workspace || B < 1 || H < 1 || topk < 0 || num_sms < 0) return MLA_ERR_INVALID_ARG;
    if (kv_dtype != MLA_KV_BF16 && kv_dtype != MLA_KV_FP8_E4M3) return MLA_ERR_INVALID_ARG;
    if (topk > 0 && kv_dtype != MLA_KV_BF16) return MLA_ERR_UNSUPPORTED;
    if (H > kMaxHeads) return MLA_ERR_UNSUPPORTED;
    if (topk == 0 && !seq_lens) return MLA_ERR_INVALID_ARG;
    if (num_sms == 0) num_sms = device_sm_count();
    if (num_sms <= 0) return MLA_ERR_CUDA;
    const int units = units_for(num_sms);
    if (ws_bytes < ws_layout(B, H, units).total) return MLA_ERR_WORKSPACE;
    // a programmatic dependent of whatever ran before on the stream (it waits for it before
    // reading seq_lens); the items' units stay in shared memory when they fit
    const size_t iu_bytes = sizeof(int32_t) * (size_t)ws_layout(B, H, units).max_items;
    const int iu_in_smem = iu_bytes <= 32 * 1024 ? 1 : 0;  // beside the kernel's ~12 KB of static shared memory
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(1, 1, 1);
    cfg.blockDim = dim3(kPlanThreads, 1, 1);
    cfg.dynamicSmemBytes = iu_in_smem ? iu_bytes : 0;
    cfg.stream = (cudaStream_t)stream;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr.val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    const int ovh = piece_overhead(kv_dtype == MLA_KV_FP8_E4M3);
    return cudaLaunchKernelEx(&cfg, plan_kernel, seq_lens, B, H, topk, units, ovh, (unsigned char *)workspace,
                              iu_in_smem) == cudaSuccess
               ? MLA_OK
               : MLA_ERR_CUDA;
}

mla_status mla_decode_plan_host(const int32_t *seq_lens, int B, int H, int topk, mla_kv_dtype kv_dtype,
                                int num_sms, void *workspace_host, size_t ws_bytes) {
    if (!workspace_host || B < 1 || H < 1 || topk < 0 || num_sms < 1) return MLA_ERR_INVALID_ARG;
    if (kv_dtype != MLA_KV_BF16 && kv_dtype != MLA_KV_FP8_E4M3) return MLA_ERR_INVALID_ARG;
    if (topk > 0 && kv_dtype != MLA_KV_BF16) return MLA_ERR_UNSUPPORTED;
    if (H > kMaxHeads) return MLA_ERR_UNSUPPORTED;
    if (topk == 0 && !seq_lens) return MLA_ERR_INVALID_ARG;
    const int units = num_units_for(num_sms);
    const WsLayout L = ws_layout(B, H, units);
    if (ws_bytes < L.plan_end) return MLA_ERR_WORKSPACE;
    build_plan_serial(seq_lens, B, H, topk, units, piece_overhead(kv_dtype == MLA_KV_FP8_E4M3),
                      (unsigned char *)workspace_host);
    *reinterpret_cast<int *>((unsigned char *)workspace_host + L.status) = 0;
    return MLA_OK;
}

mla_status mla_decode(const void *workspace, size_t ws_bytes, const void *q_nope,
                      const void *q_rope, const void *cache, mla_kv_dtype kv_dtype,
                      int64_t num_pages, const int32_t *block_table, int max_pages,
                      const int32_t *seq_lens, int B, int H, float softmax_scale, float *out,
                      float *lse, void *stream) {
    mla_status st = check_common(workspace, ws_bytes, q_nope, q_rope, cache, num_pages,
                                 block_table, max_pages, seq_lens, B, H, softmax_scale, out, lse);
    if (st != MLA_OK) return st;
    if (kv_dtype != MLA_KV_BF16 && kv_dtype != MLA_KV_FP8_E4M3) return MLA_ERR_INVALID_ARG;
    DecodeArgs a;
    memset(&a, 0, sizeof a);
    a.ws = (const unsigned char *)workspace;
    a.status = (int *)((unsigned char *)workspace + ws_layout(B, H, 1).status);
    a.q_nope = (const uint16_t *)q_nope;
    a.q_rope = (const uint16_t *)q_rope;
    a.cache = (const unsigned char *)cache;
    a.num_pages = num_pages;
    a.block_table = block_table;
    a.max_pages = max_pages;
    a.seq_lens = seq_lens;
    a.indices = nullptr;
    a.topk = 0;
    a.B = B;
    a.H = H;
    a.scale_log2 = softmax_scale * kLog2e;
    a.out = out;
    a.lse = lse;
    a.kv_fp8 = kv_dtype == MLA_KV_FP8_E4M3;
    a.ws_bytes = ws_bytes;
    a.wait_cycles = g_wait_cycles.load();
    a.stall_test = g_stall_test.load();
    return run_decode(a, (cudaStream_t)stream);
}

mla_status mla_decode_sparse(const void *workspace, size_t ws_bytes, const void *q_nope,
                             const void *q_rope, const void *cache, int64_t num_pages,
                             const int32_t *block_table, int max_pages,
                             const int32_t *seq_lens, const int32_t *indices, int topk, int B,
                             int H, float softmax_scale, float *out, float *lse,
                             void *stream) {
    mla_status st = check_common(workspace, ws_bytes, q_nope, q_rope, cache, num_pages,
                                 block_table, max_pages, seq_lens, B, H, softmax_scale, out, lse);
    if (st != MLA_OK) return st;
    if (!indices || topk < 1) return MLA_ERR_INVALID_ARG;
    DecodeArgs a;
    memset(&a, 0, sizeof a);
    a.ws = (const unsigned char *)workspace;
    a.status = (int *)((unsigned char *)workspace + ws_layout(B, H, 1).status);
    a.q_nope = (const uint16_t *)q_nope;
    a.q_rope = (const uint16_t *)q_rope;
    a.cache = (const unsigned char *)cache;
    a.num_pages = num_pages;
    a.block_table = block_table;
    a.max_pages = max_pages;
    a.seq_lens = seq_lens;
    a.indices = indices;
    a.topk = topk;
    a.B = B;
    a.H = H;
    a.scale_log2 = softmax_scale * kLog2e;
    a.out = out;
    a.lse = lse;
    a.kv_fp8 = 0;
    a.ws_bytes = ws_bytes;
    a.wait_cycles = g_wait_cycles.load();
    a.stall_test = g_stall_test.load();
    return run_decode(a, (cudaStream_t)stream);
}

mla_status mla_decode_status(void *workspace, size_t ws_bytes, void *stream) {
    if (!workspace || ws_bytes < 256) return MLA_ERR_INVALID_ARG;
    cudaStream_t s = (cudaStream_t)stream;
    if (cudaStreamSynchronize(s) != cudaSuccess) return MLA_ERR_CUDA;
    int *dev_status = (int *)((unsigned char *)workspace + ws_layout(1, 1, 1).status);
    int host = 0;
    if (cudaMemcpy(&host, dev_status, sizeof host, cudaMemcpyDeviceToHost) != cudaSuccess)
        return MLA_ERR_CUDA;
    if (host != 0 && cudaMemset(dev_status, 0, sizeof(int)) != cudaSuccess) return MLA_ERR_CUDA;
    return (mla_status)host;
}

mla_status mla_decode_inject_stall(int enable) {
    g_stall_test.store(enable ? 1 : 0);
    return MLA_OK;
}

mla_status mla_decode_set_wait_limit(int64_t cycles) {
    if (cycles < 0) return MLA_ERR_INVALID_ARG;
    g_wait_cycles.store(cycles == 0 ? kDefaultWaitCycles : (long long)cycles);
    return MLA_OK;
}

const char *mla_status_string(mla_status s) {
    switch (s) {
        case MLA_OK: return "ok";
        case MLA_ERR_INVALID_ARG: return "invalid argument";
        case MLA_ERR_UNSUPPORTED: return "unsupported configuration";
        case MLA_ERR_WORKSPACE: return "workspace too small or holds no matching plan";
        case MLA_ERR_CUDA: return "CUDA runtime error";
        case MLA_ERR_INDEX: return "page id, token index or length out of range";
        case MLA_ERR_TIMEOUT: return "pipeline wait exceeded its iteration limit";
        case MLA_ERR_RANGE: return "value outside the fp16 operand range of the FP8-record decode";
    }
    return "unknown status";
}

}  // extern "C"
