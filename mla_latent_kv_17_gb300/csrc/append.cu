// Cache append: one new token per request written into its page (bf16 entry or FP8
// record).  The definition is in include/mla_decode.h (mla_cache_append).
#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"
#include "mla_decode.h"

namespace mla {
namespace {

constexpr int kAppendWarps = 8;

// e4m3 "fn" codes of two binary32 values (round to nearest even, saturated to +-448);
// the first value in the low byte
__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi) {
    uint16_t d;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(d) : "f"(hi), "f"(lo));
    return d;
}

// One warp per request.  Lane l handles latent channels 16 l .. 16 l + 15 (so lanes 8k ..
// 8k + 7 hold channel block k of 128) and, for l < 8, RoPE values 8 l .. 8 l + 7.
__global__ void __launch_bounds__(32 * kAppendWarps)
append_kernel(unsigned char *cache, int fp8, int64_t num_pages, const int32_t *block_table, int max_pages,
              const int32_t *positions, const uint16_t *c_kv, const uint16_t *k_rope, int B, int *status) {
    const int lane = threadIdx.x & 31;
    const int b = blockIdx.x * kAppendWarps + (threadIdx.x >> 5);
    if (b >= B) return;
    // the token's values and its position are read together, then the page id
    const uint4 *src = reinterpret_cast<const uint4 *>(c_kv + (int64_t)b * kDLatent + 16 * lane);
    const uint4 v0 = src[0], v1 = src[1];
    const uint4 rp = lane < 8 ? reinterpret_cast<const uint4 *>(k_rope + (int64_t)b * kDRope)[lane]
                              : make_uint4(0u, 0u, 0u, 0u);
    const int32_t pos = positions[b];
    if (pos < 0) return;
    const int32_t lp = pos / kPageRows;
    const int64_t page = lp < max_pages ? (int64_t)block_table[(int64_t)b * max_pages + lp] : -1;
    if (page < 0 || page >= num_pages) {
        if (lane == 0 && status) record_error(status, MLA_ERR_INDEX);
        return;
    }
    const int64_t row = page * kPageRows + pos % kPageRows;
    if (!fp8) {
        uint4 *dst = reinterpret_cast<uint4 *>(cache + row * (kDEntry * 2));
        dst[2 * lane] = v0;
        dst[2 * lane + 1] = v1;
        if (lane < 8) dst[kDLatent * 2 / 16 + lane] = rp;
        return;
    }
    // FP8 record: block scale from the 8 lanes of the block, then 16 codes per lane
    const uint32_t w[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
    float x[16];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        x[2 * i] = __uint_as_float(w[i] << 16);
        x[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(x[i]));
#pragma unroll
    for (int o = 1; o < 8; o <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    const float s = amax > 0.f ? __fdiv_rn(amax, 448.f) : 1.f;
    uint32_t codes[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        float q[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) q[i] = fminf(fmaxf(__fdiv_rn(x[4 * k + i], s), -448.f), 448.f);
        codes[k] = e4m3x2(q[0], q[1]) | (e4m3x2(q[2], q[3]) << 16);
    }
    unsigned char *rec = cache + row * kFp8RecordBytes;
    reinterpret_cast<uint4 *>(rec)[lane] = make_uint4(codes[0], codes[1], codes[2], codes[3]);
    if ((lane & 7) == 0) reinterpret_cast<float *>(rec + kDLatent)[lane >> 3] = s;
    if (lane < 8) reinterpret_cast<uint4 *>(rec + kDLatent + 16)[lane] = rp;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace
}  // namespace mla

using namespace mla;

extern "C" mla_status mla_cache_append(void *cache, mla_kv_dtype kv_dtype, int64_t num_pages,
                                       const int32_t *block_table, int max_pages, const int32_t *positions,
                                       const void *c_kv, const void *k_rope, int B, int32_t *device_status,
                                       void *stream) {
    if (!cache || !block_table || !positions || !c_kv || !k_rope || B < 1 || max_pages < 1 || num_pages < 1)
        return MLA_ERR_INVALID_ARG;
    if (kv_dtype != MLA_KV_BF16 && kv_dtype != MLA_KV_FP8_E4M3) return MLA_ERR_INVALID_ARG;
    if (!aligned16(cache) || !aligned16(c_kv) || !aligned16(k_rope)) return MLA_ERR_INVALID_ARG;
    const int grid = (B + kAppendWarps - 1) / kAppendWarps;
    append_kernel<<<grid, 32 * kAppendWarps, 0, (cudaStream_t)stream>>>(
        (unsigned char *)cache, kv_dtype == MLA_KV_FP8_E4M3 ? 1 : 0, num_pages, block_table, max_pages, positions,
        (const uint16_t *)c_kv, (const uint16_t *)k_rope, B, (int *)device_status);
    return cudaGetLastError() == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}
