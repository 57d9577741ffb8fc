// DSA token selection ("MLA & DSA 推理性能优化指南" §1.2: an indexer scores every earlier token
// and only the top-k take part in the sparse attention; "GPU partial sort"): per request, the
// k positions of [0, seq_len) with the highest scores, equal scores to the lower position,
// written as ascending positions padded with -1.  The definition is in include/mla_decode.h
// (mla_topk_select).
//
// One CTA of 1024 threads per request.  Scores map to order-preserving 32-bit keys; three
// histogram passes (11, 11 and 10 key bits) narrow down the key of the k-th best position
// (radix select), then one ordered pass writes every position above that key and the
// first `need` positions equal to it, in position order, through block-wide prefix sums.
// Loads are batched (several 16-B loads per thread in flight) so that one CTA streams its
// request's scores at more than one load per thread per memory latency.  Requests of up to
// kCacheKeys positions keep their keys in shared memory after the first pass, so the later
// passes read shared memory instead of the scores again; longer ones read the scores once
// more after the first pass to list, in position order, the positions whose key's top 11 bits
// reach the selected bin (the only ones that can be selected), and run the rest on that list
// when it fits in kListCap entries.
#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"
#include "mla_decode.h"

namespace mla {
namespace {

constexpr int kTkThreads = 1024;
constexpr int kTkWarps = kTkThreads / 32;
constexpr int kBins = 2048;
constexpr int kHistCopies = 8;  // warp w adds into copy w % 8 (fewer collisions on hot bins)
constexpr uint32_t kTkHistBytes = kHistCopies * kBins * 4;
constexpr int kCacheKeys = 32768;  // keys of a request kept in shared memory (128 KB)
constexpr int kListCap = 16384;    // candidates (position, key) of a longer request (128 KB)
constexpr int kLoadsInFlight = 8;  // float4 loads per thread per histogram iteration
constexpr int kPerThread = 16;     // consecutive positions per thread per ordered-write round

// Larger key <=> larger score; -0.0 and +0.0 share a key.
__device__ __forceinline__ uint32_t order_key(float f) {
    uint32_t u = __float_as_uint(f);
    if (u == 0x80000000u) u = 0u;
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ float4 ld4(const float *p) { return __ldg(reinterpret_cast<const float4 *>(p)); }

// Inclusive prefix sum of v over the block in thread order; `total` gets the block's sum.
__device__ __forceinline__ uint32_t block_scan(uint32_t v, uint32_t *warp_sums, uint32_t &total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    uint32_t x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) warp_sums[warp] = x;
    __syncthreads();
    if (warp == 0) {
        uint32_t w = warp_sums[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t y = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += y;
        }
        warp_sums[lane] = w;
    }
    __syncthreads();
    const uint32_t before = warp ? warp_sums[warp - 1] : 0u;
    total = warp_sums[kTkWarps - 1];
    __syncthreads();  // warp_sums is reused by the next scan
    return x + before;
}

__global__ void __launch_bounds__(kTkThreads) topk_kernel(const float *__restrict__ scores, int64_t stride, int Lmax,
                                                          const int32_t *__restrict__ seq_lens, int k,
                                                          int32_t *indices, int cache_keys, int list_cap, int *status) {
    // [kHistCopies][kBins] histograms, then either cache_keys keys (every position of a short
    // request) or list_cap (position, key) pairs (the candidates of a long one)
    extern __shared__ uint32_t hist[];
    __shared__ uint32_t warp_sums[kTkWarps];
    __shared__ uint32_t sel_bin, sel_above, sel_count;
    const int b = blockIdx.x;
    const int L = seq_lens[b];
    int32_t *out = indices + (int64_t)b * k;
    if (L < 0 || L > Lmax) {
        if (threadIdx.x == 0 && status) record_error(status, MLA_ERR_INDEX);
        for (int i = threadIdx.x; i < k; i += kTkThreads) out[i] = -1;
        return;
    }
    const int K = min(k, L);
    if (K == L) {  // every position is kept
        for (int i = threadIdx.x; i < k; i += kTkThreads) out[i] = i < L ? i : -1;
        return;
    }
    const float *s = scores + (int64_t)b * stride;
    const int n4 = (L + 3) >> 2;
    uint32_t *cache = hist + kHistCopies * kBins;                     // keys of positions [0, L)
    uint32_t *list_key = cache, *list_pos = cache + list_cap;          // candidates in position order
    // where the passes after the first read their keys: 0 the scores again, 1 the key cache
    // (filled by the first pass), 2 the candidate list (built after the first pass: the
    // positions whose key's top 11 bits are at least the selected bin's, when they fit)
    int mode = L <= cache_keys ? 1 : 0;
    int ncand = 0;

    // ---- radix select: key of the K-th best position, and how many of its ties to keep
    uint32_t prefix = 0u, pmask = 0u, need = (uint32_t)K;
    uint32_t *hmine = hist + ((threadIdx.x >> 5) & (kHistCopies - 1)) * kBins;
#pragma unroll 1
    for (int pass = 0; pass < 3; ++pass) {
        const int shift = pass == 0 ? 21 : pass == 1 ? 10 : 0;
        const uint32_t bmask = pass == 2 ? 1023u : 2047u;
        for (int i = threadIdx.x; i < kHistCopies * kBins; i += kTkThreads) hist[i] = 0u;
        __syncthreads();
        if (pass > 0 && mode == 1) {
            // the keys from shared memory, four per thread and step
            for (int i = threadIdx.x; i < n4; i += kTkThreads) {
                const uint4 kv = reinterpret_cast<const uint4 *>(cache)[i];
                const uint32_t kk[4] = {kv.x, kv.y, kv.z, kv.w};
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    if (4 * i + j < L && (kk[j] & pmask) == prefix) atomicAdd(&hmine[(kk[j] >> shift) & bmask], 1u);
            }
        } else if (pass > 0 && mode == 2) {
            for (int i = threadIdx.x; i < ncand; i += kTkThreads) {
                const uint32_t kk = list_key[i];
                if ((kk & pmask) == prefix) atomicAdd(&hmine[(kk >> shift) & bmask], 1u);
            }
        } else {
            // kLoadsInFlight float4 loads per thread are issued before any of them is used
            for (int i0 = threadIdx.x; i0 < n4; i0 += kLoadsInFlight * kTkThreads) {
                float4 v[kLoadsInFlight];
#pragma unroll
                for (int u = 0; u < kLoadsInFlight; ++u) v[u] = ld4(s + 4 * min(i0 + u * kTkThreads, n4 - 1));
#pragma unroll
                for (int u = 0; u < kLoadsInFlight; ++u) {
                    const int i = i0 + u * kTkThreads;
                    const float f[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
                    uint32_t kk[4];
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        kk[j] = order_key(f[j]);
                        if (i < n4 && 4 * i + j < L && (kk[j] & pmask) == prefix)
                            atomicAdd(&hmine[(kk[j] >> shift) & bmask], 1u);
                    }
                    if (mode == 1 && i < n4) reinterpret_cast<uint4 *>(cache)[i] = make_uint4(kk[0], kk[1], kk[2], kk[3]);
                }
            }
        }
        __syncthreads();
        // thread t holds bins hi = 2047 - 2t and lo = hi - 1, so thread order is descending key
        const int hi = kBins - 1 - 2 * (int)threadIdx.x, lo = hi - 1;
        uint32_t ch = 0u, cl = 0u;
#pragma unroll
        for (int c = 0; c < kHistCopies; ++c) {
            ch += hist[c * kBins + hi];
            cl += hist[c * kBins + lo];
        }
        uint32_t total;
        const uint32_t incl = block_scan(ch + cl, warp_sums, total);
        const uint32_t above = incl - ch - cl;  // keys (with this prefix) in bins above hi
        if (above < need && need <= above + ch) {
            sel_bin = (uint32_t)hi;
            sel_above = above;
            sel_count = ch;
        } else if (above + ch < need && need <= incl) {
            sel_bin = (uint32_t)lo;
            sel_above = above + ch;
            sel_count = cl;
        }
        __syncthreads();
        prefix |= sel_bin << shift;
        pmask |= bmask << shift;
        need -= sel_above;
        const uint32_t candidates = sel_above + sel_count;  // keys at or above the selected bin
        __syncthreads();  // sel_bin / sel_above / sel_count and hist are rewritten by the next pass
        if (pass == 0 && mode == 0 && candidates <= (uint32_t)list_cap) {
            // one more read of the scores: the candidates, in position order (16 consecutive
            // positions per thread and round, placed by a block-wide prefix sum)
            const uint32_t lo_key = prefix;  // smallest key with the selected top bits
            uint32_t base = 0u;
#pragma unroll 1
            for (int r0 = 0; r0 < L; r0 += kPerThread * kTkThreads) {
                const int p0 = r0 + kPerThread * (int)threadIdx.x;
                float4 v[kPerThread / 4];
#pragma unroll
                for (int u = 0; u < kPerThread / 4; ++u) v[u] = ld4(s + min(p0 + 4 * u, 4 * (n4 - 1)));
                uint32_t keys[kPerThread], bits = 0u;
#pragma unroll
                for (int u = 0; u < kPerThread / 4; ++u) {
                    keys[4 * u] = order_key(v[u].x);
                    keys[4 * u + 1] = order_key(v[u].y);
                    keys[4 * u + 2] = order_key(v[u].z);
                    keys[4 * u + 3] = order_key(v[u].w);
                }
#pragma unroll
                for (int j = 0; j < kPerThread; ++j)
                    if (p0 + j < L && keys[j] >= lo_key) bits |= 1u << j;
                uint32_t tot;
                const uint32_t mine = (uint32_t)__popc(bits);
                uint32_t at = base + block_scan(mine, warp_sums, tot) - mine;
#pragma unroll
                for (int j = 0; j < kPerThread; ++j) {
                    if (bits & (1u << j)) {
                        if (at < (uint32_t)list_cap) {  // always: the count was taken from the histogram
                            list_key[at] = keys[j];
                            list_pos[at] = (uint32_t)(p0 + j);
                        }
                        ++at;
                    }
                }
                base += tot;
            }
            ncand = (int)min(base, (uint32_t)list_cap);
            mode = 2;
            __syncthreads();  // the list is complete
        }
    }
    const uint32_t kstar = prefix;

    // ---- ordered write: positions above kstar, and the first `need` positions equal to it.
    // A round covers kPerThread consecutive positions (mode 2: candidates) per thread,
    // 16,384 per round.
    uint32_t base_gt = 0u, base_eq = 0u;
    const int nitems = mode == 2 ? ncand : L;
#pragma unroll 1
    for (int r0 = 0; r0 < nitems; r0 += kPerThread * kTkThreads) {
        const int p0 = r0 + kPerThread * (int)threadIdx.x;
        uint32_t keys[kPerThread];
        if (mode == 1) {
#pragma unroll
            for (int u = 0; u < kPerThread / 4; ++u) {
                const uint4 kv = reinterpret_cast<const uint4 *>(cache)[min(p0 / 4 + u, n4 - 1)];
                keys[4 * u] = kv.x;
                keys[4 * u + 1] = kv.y;
                keys[4 * u + 2] = kv.z;
                keys[4 * u + 3] = kv.w;
            }
        } else if (mode == 2) {
#pragma unroll
            for (int j = 0; j < kPerThread; ++j) keys[j] = list_key[min(p0 + j, ncand - 1)];
        } else {
            float4 v[kPerThread / 4];
#pragma unroll
            for (int u = 0; u < kPerThread / 4; ++u) v[u] = ld4(s + min(p0 + 4 * u, 4 * (n4 - 1)));
#pragma unroll
            for (int u = 0; u < kPerThread / 4; ++u) {
                keys[4 * u] = order_key(v[u].x);
                keys[4 * u + 1] = order_key(v[u].y);
                keys[4 * u + 2] = order_key(v[u].z);
                keys[4 * u + 3] = order_key(v[u].w);
            }
        }
        uint32_t gt = 0u, eq = 0u;  // bit j: item p0 + j
#pragma unroll
        for (int j = 0; j < kPerThread; ++j) {
            const bool ok = p0 + j < nitems;
            if (ok && keys[j] > kstar) gt |= 1u << j;
            if (ok && keys[j] == kstar) eq |= 1u << j;
        }
        uint32_t total;
        const uint32_t mine = ((uint32_t)__popc(gt) << 16) | (uint32_t)__popc(eq);  // < 2^16 of each per round
        const uint32_t excl = block_scan(mine, warp_sums, total) - mine;
        const uint32_t gt_before = base_gt + (excl >> 16);
        uint32_t eq_seen = base_eq + (excl & 0xFFFFu);
        uint32_t slot = gt_before + min(need, eq_seen);
#pragma unroll
        for (int j = 0; j < kPerThread; ++j) {  // slot < K always holds; the check keeps writes in the row
            const int pos = mode == 2 ? (int)list_pos[min(p0 + j, ncand - 1)] : p0 + j;
            if (gt & (1u << j)) {
                if (slot < (uint32_t)K) out[slot] = pos;
                ++slot;
            } else if (eq & (1u << j)) {
                if (eq_seen < need) {
                    if (slot < (uint32_t)K) out[slot] = pos;
                    ++slot;
                }
                ++eq_seen;
            }
        }
        base_gt += total >> 16;
        base_eq += total & 0xFFFFu;
    }
    for (int i = K + (int)threadIdx.x; i < k; i += kTkThreads) out[i] = -1;
}

bool set_topk_attr() {
    static bool done[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return false;
    if (done[dev]) return true;
    if (cudaFuncSetAttribute(topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)(kTkHistBytes + (4u * kCacheKeys > 8u * kListCap ? 4u * kCacheKeys : 8u * kListCap))) !=
        cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    done[dev] = true;
    return true;
}

}  // namespace
}  // namespace mla

using namespace mla;

extern "C" mla_status mla_topk_select(const float *scores, int64_t row_stride, int Lmax, const int32_t *seq_lens,
                                      int B, int k, int32_t *indices, int32_t *device_status, void *stream) {
    if (!scores || !seq_lens || !indices || B < 1 || k < 1 || Lmax < 0 || row_stride < Lmax ||
        (row_stride & 3) != 0 || (reinterpret_cast<uintptr_t>(scores) & 15u) != 0)
        return MLA_ERR_INVALID_ARG;
    if (!set_topk_attr()) return MLA_ERR_CUDA;
    // the key cache holds the longest request when it fits (positions rounded up to 4);
    // otherwise the same space holds a candidate list
    const int cache_keys = Lmax <= kCacheKeys ? ((Lmax + 3) & ~3) : 0;
    const int list_cap = cache_keys ? 0 : kListCap;
    const size_t smem = kTkHistBytes + 4u * (size_t)cache_keys + 8u * (size_t)list_cap;
    topk_kernel<<<B, kTkThreads, smem, (cudaStream_t)stream>>>(scores, row_stride, Lmax, seq_lens, k, indices,
                                                              cache_keys, list_cap, (int *)device_status);
    return cudaGetLastError() == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}
