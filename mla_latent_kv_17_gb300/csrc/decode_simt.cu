// Straightforward CUDA-core decode kernel (no tensor cores).  One CTA handles one unit's
// work items for 16 heads; the 32-token tile is staged in shared memory as fp32 and each
// warp runs an online softmax for two heads.  Covers the bf16 cache, the FP8-record cache
// and token-sparse index lists.
#include <cuda_fp8.h>

#include "common.cuh"
#include "launch.h"

namespace mla {
namespace {

constexpr int kSimtHeads = 16;
constexpr int kSimtTile = 32;
constexpr int kSimtThreads = 256;
constexpr int kRowPitch = kDEntry + 1;  // fp32 words; the +1 keeps lanes on distinct banks

__device__ __forceinline__ float e4m3_to_f32(unsigned char code) {
    __half_raw h = __nv_cvt_fp8_to_halfraw((__nv_fp8_storage_t)code, __NV_E4M3);
    return __half2float(__half(h));
}

// Physical cache row of logical token t of request b, or -1 (error recorded) when the
// block table or page id is out of range.
__device__ __forceinline__ int64_t cache_row(const DecodeArgs &a, int b, int t) {
    int lp = t / kPageRows;
    if (lp >= a.max_pages) {
        record_error(a.status, MLA_ERR_INDEX);
        return -1;
    }
    int64_t page = a.block_table[(int64_t)b * a.max_pages + lp];
    if (page < 0 || page >= a.num_pages) {
        record_error(a.status, MLA_ERR_INDEX);
        return -1;
    }
    return page * kPageRows + (t % kPageRows);
}

__global__ void __launch_bounds__(kSimtThreads)
decode_simt_kernel(DecodeArgs a) {
    extern __shared__ float smem[];
    float *qs = smem;                                // [16][577]
    float *cs = qs + kSimtHeads * kRowPitch;         // [32][577]
    int *valid = reinterpret_cast<int *>(cs + kSimtTile * kRowPitch);  // [32]

    if (!plan_matches(a)) {
        if (threadIdx.x == 0 && blockIdx.x == 0 && blockIdx.y == 0)
            record_error(a.status, MLA_ERR_WORKSPACE);
        return;
    }
    const PlanHeader *hd = reinterpret_cast<const PlanHeader *>(a.ws);
    const WsLayout L = ws_layout(hd->B, hd->H, hd->num_units);
    const int32_t *unit_begin = reinterpret_cast<const int32_t *>(a.ws + L.unit_begin);
    const WorkItem *items = reinterpret_cast<const WorkItem *>(a.ws + L.items);
    float *part_lse = reinterpret_cast<float *>(const_cast<unsigned char *>(a.ws) + L.part_lse);
    float *part_o = reinterpret_cast<float *>(const_cast<unsigned char *>(a.ws) + L.part_o);

    const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
    const int h_base = blockIdx.y * kSimtHeads;
    const int num_units = hd->num_units;

    for (int u = blockIdx.x; u < num_units; u += gridDim.x) {
        for (int it = unit_begin[u]; it < unit_begin[u + 1]; ++it) {
            const WorkItem w = items[it];
            const int b = w.b;
            int seq_len = a.seq_lens[b];
            if (seq_len < 0) seq_len = 0;
            __syncthreads();
            for (int i = tid; i < kSimtHeads * kDEntry; i += kSimtThreads) {
                int hh = i / kDEntry, c = i % kDEntry, h = h_base + hh;
                float v = 0.f;
                if (h < a.H)
                    v = c < kDLatent
                            ? bf16_to_f32(a.q_nope[((int64_t)b * a.H + h) * kDLatent + c])
                            : bf16_to_f32(a.q_rope[((int64_t)b * a.H + h) * kDRope + c - kDLatent]);
                qs[hh * kRowPitch + c] = v;
            }
            float m[2], l[2], acc[2][16];
            for (int j = 0; j < 2; ++j) {
                m[j] = -INFINITY;
                l[j] = 0.f;
                for (int k = 0; k < 16; ++k) acc[j][k] = 0.f;
            }
            for (int ts = w.t0; ts < w.t1; ts += kSimtTile) {
                __syncthreads();
                if (tid < kSimtTile) {
                    int r = tid, slot = ts + r;
                    int64_t row = -1;
                    if (slot < w.t1) {
                        int t = slot;
                        if (a.indices) {
                            t = a.indices[(int64_t)b * a.topk + slot];
                            if (t < -1 || t >= seq_len) {
                                record_error(a.status, MLA_ERR_INDEX);
                                t = -1;
                            }
                        } else if (t >= seq_len) {
                            t = -1;
                        }
                        if (t >= 0) row = cache_row(a, b, t);
                    }
                    valid[r] = row >= 0;
                    reinterpret_cast<long long *>(valid + kSimtTile)[r] = row;
                }
                __syncthreads();
                const long long *rows = reinterpret_cast<const long long *>(valid + kSimtTile);
                for (int i = tid; i < kSimtTile * kDEntry; i += kSimtThreads) {
                    int r = i / kDEntry, c = i % kDEntry;
                    long long row = rows[r];
                    float v = 0.f;
                    if (row >= 0) {
                        if (!a.kv_fp8) {
                            v = bf16_to_f32(reinterpret_cast<const uint16_t *>(a.cache)[row * kDEntry + c]);
                        } else {
                            const unsigned char *rec = a.cache + row * kFp8RecordBytes;
                            if (c < kDLatent) {
                                float s = *reinterpret_cast<const float *>(rec + 512 + 4 * (c / 128));
                                v = e4m3_to_f32(rec[c]) * s;
                            } else {
                                v = bf16_to_f32(reinterpret_cast<const uint16_t *>(rec + 528)[c - kDLatent]);
                            }
                        }
                    }
                    cs[r * kRowPitch + c] = v;
                }
                __syncthreads();
                for (int j = 0; j < 2; ++j) {
                    const int hh = warp * 2 + j;
                    const float *q = qs + hh * kRowPitch;
                    const float *crow = cs + lane * kRowPitch;
                    float s = 0.f;
                    for (int c = 0; c < kDEntry; ++c) s = fmaf(q[c], crow[c], s);
                    s = valid[lane] ? s * a.scale_log2 : -INFINITY;
                    float mt = s;
                    for (int o = 16; o > 0; o >>= 1) mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, o));
                    float mn = fmaxf(m[j], mt);
                    if (mn == -INFINITY) continue;  // nothing attended yet
                    float p = exp2f(s - mn);
                    float alpha = exp2f(m[j] - mn);
                    float ps = p;
                    for (int o = 16; o > 0; o >>= 1) ps += __shfl_xor_sync(0xffffffffu, ps, o);
                    l[j] = l[j] * alpha + ps;
                    for (int k = 0; k < 16; ++k) acc[j][k] *= alpha;
                    for (int r = 0; r < kSimtTile; ++r) {
                        float pr = __shfl_sync(0xffffffffu, p, r);
                        const float *cr = cs + r * kRowPitch;
                        for (int k = 0; k < 16; ++k) acc[j][k] = fmaf(pr, cr[lane + 32 * k], acc[j][k]);
                    }
                    m[j] = mn;
                }
            }
            for (int j = 0; j < 2; ++j) {
                const int h = h_base + warp * 2 + j;
                if (h >= a.H) continue;
                float inv = l[j] > 0.f ? 1.f / l[j] : 0.f;
                float lse = l[j] > 0.f ? (m[j] + log2f(l[j])) * kLn2 : -INFINITY;
                float *o;
                if (w.slot < 0) {
                    o = a.out + ((int64_t)b * a.H + h) * kDLatent;
                    if (lane == 0) a.lse[(int64_t)b * a.H + h] = lse;
                } else {
                    o = part_o + ((int64_t)w.slot * a.H + h) * kDLatent;
                    if (lane == 0) part_lse[(int64_t)w.slot * a.H + h] = lse;
                }
                for (int k = 0; k < 16; ++k) o[lane + 32 * k] = acc[j][k] * inv;
            }
        }
    }
}

}  // namespace

cudaError_t launch_decode_simt(const DecodeArgs &a, int num_units, cudaStream_t stream) {
    size_t smem = sizeof(float) * (kSimtHeads + kSimtTile) * kRowPitch + kSimtTile * 4 +
                  kSimtTile * 8;
    static bool attr_set = false;
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(decode_simt_kernel,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    dim3 grid(num_units, (a.H + kSimtHeads - 1) / kSimtHeads);
    decode_simt_kernel<<<grid, kSimtThreads, smem, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace mla
