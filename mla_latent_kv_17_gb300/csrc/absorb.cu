// Query absorption before the absorbed decode and the value up-projection after it, one bf16
// matrix per head ("MLA 在极长上下文下的显存带宽突围", run-time matrix absorption: q~ = q^C W^UK;
// "MLA & DSA 推理性能优化指南" §1.1: W^UV is applied to the latent output afterwards).  The
// definitions are in include/mla_decode.h (mla_absorb_query, mla_project_output).
//
// Both are batched over the requests of one head, so the request index is the MMA's N side
// (up to 64 requests per tile) and the weight matrix its M side:
//   absorb : D[c][b] = sum_k W^UK[h][k][c] q^C[b][h][k]    M = 128 latent columns, K = d_h
//   project: D[j][b] = sum_c W^UV[h][j][c] out[b][h][c]    M = d_h = 128, K = 512
// so that one TMEM lane holds one output channel of every request in the tile.  The
// projection's warps store y straight from TMEM (32 consecutive channels of one request per
// store); the absorption transposes q~ through shared memory and stores it by the TMA.  The
// projection streams K in 64-column chunks (weights and the fp32 output by the TMA, the
// output rounded to bf16 in shared memory by eight warps).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"
#include "mla_decode.h"
#include "sm103_ptx.cuh"
#include "tc_util.cuh"

namespace mla {
namespace {

using namespace ptx;

constexpr int kDh = 128;     // per-head nope / value width d_h
constexpr int kNb = 64;      // requests per tile (MMA N, TMEM columns)
constexpr uint32_t kWBox = 128 * 128;       // 128 rows x 64 bf16 of a weight matrix, 128-B swizzle
constexpr uint32_t kRBox = kNb * 128;       // 64 requests x 64 bf16, 128-B swizzle

// absorb: A = W^UK[h][0:128][c0 : c0 + 128] as two MN-major boxes, B = q^C of the tile as two
// K-major boxes; then three mbarriers and the TMEM address
constexpr uint32_t kAbsBar = 2 * kWBox + 2 * kRBox;
constexpr uint32_t kAbsSmem = kAbsBar + 32 + 1024;
// project: a ring of four stages, each one 64-column chunk of K: the W^UV box (bf16, 16 KB),
// the tile's fp32 output (two 32-column boxes, 16 KB) and its bf16 copy (the B operand, 8 KB)
constexpr int kPrjStages = 4;
constexpr uint32_t kPrjF = kNb * 64 * 4;                 // fp32 output chunk: 64 requests x 64 columns
constexpr uint32_t kPrjStage = kWBox + kPrjF + kRBox;    // 40 KB
constexpr uint32_t kPrjBar = kPrjStages * kPrjStage;
constexpr uint32_t kPrjSmem = kPrjBar + 128 + 1024;
constexpr int kPrjConvWarps = 8;                         // convert, then store y
constexpr int kPrjThreads = 32 * (kPrjConvWarps + 2);    // + one loading warp, one MMA warp

// One CTA per (latent tile ct of 128 columns, head h, request tile bt): four warps.
__global__ void __launch_bounds__(128) absorb_kernel(const __grid_constant__ CUtensorMap tm_w,
                                                     const __grid_constant__ CUtensorMap tm_q,
                                                     const __grid_constant__ CUtensorMap tm_o, int H,
                                                     int *status) {
    extern __shared__ unsigned char smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    unsigned char *gbase = smem_raw + (base - raw);
    const uint32_t sA = base, sB = base + 2 * kWBox;
    const uint32_t bar_full = base + kAbsBar, bar_done = bar_full + 8;
    volatile uint32_t *tslot = reinterpret_cast<volatile uint32_t *>(gbase + kAbsBar + 16);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int ct = blockIdx.x & 3;
    const int h = (blockIdx.x >> 2) % H;
    const int bt = (blockIdx.x >> 2) / H;

    if (warp == 0) {
        if (lane == 0) {
            mbar_init(bar_full, 1);
            mbar_init(bar_done, 1);
            fence_mbar_init();
        }
        __syncwarp();
        tmem_alloc(smem_u32(const_cast<uint32_t *>(tslot)), kNb);
        tmem_relinquish();
    }
    grid_dep_wait();  // q^C may come from the previous kernel of the stream
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;

    bool ok = true;
    if (threadIdx.x == 0) {
        mbar_arrive_expect_tx(bar_full, 2 * kWBox + 2 * kRBox);
        for (int i = 0; i < 2; ++i) tma_load_3d(sA + i * kWBox, &tm_w, 128 * ct + 64 * i, 0, h, bar_full);
        for (int i = 0; i < 2; ++i) tma_load_3d(sB + i * kRBox, &tm_q, 64 * i, h, kNb * bt, bar_full);
        ok = wait_bounded(bar_full, 0);
        if (ok) {
            tc_fence_after();
            constexpr uint32_t idesc = idesc_bf16_major(128, kNb, true, false);
            for (int k = 0; k < kDh / 16; ++k) {
                // A: 16 k-rows of both 64-column boxes; B: 16 k of the request rows
                const uint64_t ad = smem_desc_sw128(sA + k * 2048u, kWBox, 1024u);
                const uint64_t bd = smem_desc_sw128(sB + (k >> 2) * kRBox + (k & 3) * 32u, 16u, 1024u);
                mma_ss(tmem, ad, bd, idesc, k > 0 ? 1u : 0u);
            }
            mma_commit(bar_done);
        }
    }
    grid_dep_launch();
    if (__syncthreads_and(ok ? 1 : 0)) {
        ok = wait_bounded(bar_done, 0);
        tc_fence_after();
        if (ok) {
            // q~ of the tile, transposed into two 64-column boxes [64 requests][64 bf16] (128-B
            // swizzle) over the weight boxes (the MMAs have read them), then stored by the TMA;
            // rows past B fall outside the tensor and are not written
            const int cc = 32 * (warp & 1) + lane;  // column within box warp / 2
            const uint32_t box = sA + (warp >> 1) * kRBox;
            const uint32_t taddr = tmem + ((uint32_t)(32 * warp) << 16);
#pragma unroll 1
            for (int ch = 0; ch < kNb / 32; ++ch) {
                uint32_t r[32];
                tmem_ld32(taddr + 32u * ch, r);
                tmem_wait_ld();
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    const int b = 32 * ch + i;
                    st_shared_u16(box + b * 128 + ((((cc >> 3) ^ (b & 7))) << 4) + (cc & 7) * 2,
                                  bf16_bits(__uint_as_float(r[i])));
                }
            }
            fence_proxy_async_smem();
        }
    }
    if (__syncthreads_and(ok ? 1 : 0) && threadIdx.x == 0) {
        for (int q = 0; q < 2; ++q) tma_store_3d(&tm_o, sA + q * kRBox, 128 * ct + 64 * q, h, kNb * bt);
        bulk_commit_group();
        bulk_wait_group0();
    }
    if (!ok) {
        if (status) record_error(status, MLA_ERR_TIMEOUT);
        drain_pause();
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, kNb);
    }
}

// One CTA per (head h, request tile bt).  K = 512 latent columns in eight chunks of 64 through
// a four-stage ring: one thread loads each chunk's W^UV box (bf16) and the tile's fp32 output
// (two 32-column boxes, 128-B swizzle) by the TMA; eight warps round the fp32 values to the
// swizzled bf16 B operand; one thread issues the chunk's four MMAs; the eight warps store y.
__global__ void __launch_bounds__(kPrjThreads, 1) project_kernel(const __grid_constant__ CUtensorMap tm_v,
                                                                 const __grid_constant__ CUtensorMap tm_f, float *y,
                                                                 int B, int H, int *status) {
    extern __shared__ unsigned char smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    unsigned char *gbase = smem_raw + (base - raw);
    const uint32_t bars = base + kPrjBar;  // full[4], conv[4], empty[4], done
    auto full = [&](int st) { return bars + 8u * st; };
    auto conv = [&](int st) { return bars + 32u + 8u * st; };
    auto empty = [&](int st) { return bars + 64u + 8u * st; };
    const uint32_t done = bars + 96u;
    volatile uint32_t *tslot = reinterpret_cast<volatile uint32_t *>(gbase + kPrjBar + 104);
    int *abort_flag = reinterpret_cast<int *>(gbase + kPrjBar + 112);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int h = blockIdx.x % H;
    const int bt = blockIdx.x / H;
    const int b0 = kNb * bt;

    if (warp == 0) {
        if (lane == 0) {
            for (int st = 0; st < kPrjStages; ++st) {
                mbar_init(full(st), 1);
                mbar_init(conv(st), kPrjConvWarps);
                mbar_init(empty(st), 1);
            }
            mbar_init(done, 1);
            *abort_flag = 0;
            fence_mbar_init();
        }
        __syncwarp();
        tmem_alloc(smem_u32(const_cast<uint32_t *>(tslot)), kNb);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;
    bool ok = true;
    auto wait = [&](uint32_t bar, uint32_t parity) { return wait_bounded(bar, parity, abort_flag); };
    constexpr int kChunks = kDLatent / 64;
    if (warp == kPrjConvWarps) {
        // loads: the weights do not depend on the previous kernel, the output does
        if (lane == 0) {
            bool waited = false;
            for (int c = 0; c < kChunks && ok; ++c) {
                const int st = c % kPrjStages;
                if (c >= kPrjStages) ok = wait(empty(st), ((c / kPrjStages) - 1) & 1);
                if (!ok) break;
                const uint32_t sd = base + st * kPrjStage;
                mbar_arrive_expect_tx(full(st), kWBox + kPrjF);
                tma_load_3d(sd, &tm_v, 64 * c, 0, h, full(st));
                if (!waited) {
                    grid_dep_wait();
                    waited = true;
                }
                tma_load_3d(sd + kWBox, &tm_f, 64 * c, h, b0, full(st));
                tma_load_3d(sd + kWBox + kPrjF / 2, &tm_f, 64 * c + 32, h, b0, full(st));
            }
        }
    } else if (warp == kPrjConvWarps + 1) {
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_bf16_major(128, kNb, false, false);
            for (int c = 0; c < kChunks && ok; ++c) {
                const int st = c % kPrjStages;
                ok = wait(conv(st), (c / kPrjStages) & 1);
                if (!ok) break;
                tc_fence_after();
                const uint32_t sd = base + st * kPrjStage;
                for (int k = 0; k < 4; ++k)
                    mma_ss(tmem, smem_desc_sw128(sd + k * 32u, 16u, 1024u),
                           smem_desc_sw128(sd + kWBox + kPrjF + k * 32u, 16u, 1024u), idesc, (c | k) ? 1u : 0u);
                mma_commit(empty(st));
            }
            if (ok) mma_commit(done);
        }
    } else {
        // thread t: request row r = t / 4 of the tile, 16 columns (quarter qd) of each chunk
        const int r = threadIdx.x >> 2, qd = threadIdx.x & 3;
        for (int c = 0; c < kChunks && ok; ++c) {
            const int st = c % kPrjStages;
            ok = wait(full(st), (c / kPrjStages) & 1);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            const uint32_t sd = base + st * kPrjStage;
            // fp32 box qd / 2 (32 columns, 128-B rows, 16-B unit u at u ^ (r % 8)); units
            // 4 (qd % 2) .. + 3 hold this thread's 16 values
            const uint32_t fbox = sd + kWBox + (qd >> 1) * (kPrjF / 2) + r * 128;
            uint32_t w[8];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int u = 4 * (qd & 1) + i;
                float4 f;
                asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                             : "=f"(f.x), "=f"(f.y), "=f"(f.z), "=f"(f.w)
                             : "r"(fbox + ((u ^ (r & 7)) << 4)));
                w[2 * i] = bf16x2_bits(f.x, f.y);
                w[2 * i + 1] = bf16x2_bits(f.z, f.w);
            }
            // bf16 B operand row r: 16-B units 2 qd and 2 qd + 1, swizzled
            const uint32_t brow = sd + kWBox + kPrjF + r * 128;
            asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(brow + (((2 * qd) ^ (r & 7)) << 4)),
                         "r"(w[0]), "r"(w[1]), "r"(w[2]), "r"(w[3])
                         : "memory");
            asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(brow + (((2 * qd + 1) ^ (r & 7)) << 4)),
                         "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7])
                         : "memory");
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(conv(st));
        }
        if (ok) {
            ok = wait(done, 0);
            ok = __all_sync(0xffffffffu, ok);
        }
        if (ok) {
            tc_fence_after();
            // warp w: TMEM lanes 32 (w % 4) .. (output channels j), requests 32 (w / 4) ..
            const int j = 32 * (warp & 3) + lane;
            const int half = warp >> 2;
            uint32_t rr[32];
            tmem_ld32(tmem + ((uint32_t)(32 * (warp & 3)) << 16) + 32u * half, rr);
            tmem_wait_ld();
            const int bb = b0 + 32 * half;
#pragma unroll
            for (int i = 0; i < 32; ++i)
                if (bb + i < B) y[((int64_t)(bb + i) * H + h) * kDh + j] = __uint_as_float(rr[i]);
        }
    }
    grid_dep_launch();
    if (!__syncthreads_and(ok ? 1 : 0)) {
        if (threadIdx.x == 0 && status) record_error(status, MLA_ERR_TIMEOUT);
        drain_pause();
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, kNb);
    }
}

// 3-D bf16 / fp32 tensors (d0 innermost, d1, d2) with byte strides s1, s2 and boxes b0 x b1 x b2.
bool tmap_3d(CUtensorMap *m, const void *p, uint64_t d0, uint64_t d1, uint64_t d2, uint64_t s1, uint64_t s2,
             uint32_t b0, uint32_t b1, uint32_t b2) {
    const uint64_t d[3] = {d0, d1, d2}, st[2] = {s1, s2};
    const uint32_t b[3] = {b0, b1, b2};
    return tmap_tiled(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, p, 3, d, st, b);
}
bool tmap_3d_f32(CUtensorMap *m, const void *p, uint64_t d0, uint64_t d1, uint64_t d2, uint64_t s1, uint64_t s2,
                 uint32_t b0, uint32_t b1, uint32_t b2) {
    const uint64_t d[3] = {d0, d1, d2}, st[2] = {s1, s2};
    const uint32_t b[3] = {b0, b1, b2};
    return tmap_tiled(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, p, 3, d, st, b);
}

bool set_attrs() {
    static bool done[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return false;
    if (done[dev]) return true;
    if (cudaFuncSetAttribute(absorb_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kAbsSmem) !=
            cudaSuccess ||
        cudaFuncSetAttribute(project_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kPrjSmem) !=
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

extern "C" mla_status mla_absorb_query(const void *q_c, const void *w_uk, int B, int H, void *q_nope,
                                       int32_t *device_status, void *stream) {
    if (!q_c || !w_uk || !q_nope || B < 1 || H < 1) return MLA_ERR_INVALID_ARG;
    if (!aligned16(q_c) || !aligned16(w_uk) || !aligned16(q_nope)) return MLA_ERR_INVALID_ARG;
    const int64_t tiles = (int64_t)4 * H * ((B + kNb - 1) / kNb);
    if (tiles > 0x7FFFFFFF) return MLA_ERR_UNSUPPORTED;
    if (!set_attrs()) return MLA_ERR_CUDA;
    CUtensorMap tw, tq, to;
    // W^UK [H][128][512]: (c, k, h); q^C [B][H][128]: (k, h, b); q~ [B][H][512]: (c, h, b)
    if (!tmap_3d(&tw, w_uk, kDLatent, kDh, H, kDLatent * 2, (uint64_t)kDh * kDLatent * 2, 64, 128, 1) ||
        !tmap_3d(&tq, q_c, kDh, H, B, kDh * 2, (uint64_t)kDh * 2 * H, 64, 1, kNb) ||
        !tmap_3d(&to, q_nope, kDLatent, H, B, kDLatent * 2, (uint64_t)kDLatent * 2 * H, 64, 1, kNb))
        return MLA_ERR_CUDA;
    return launch_pdl(absorb_kernel, (int)tiles, 128, kAbsSmem, (cudaStream_t)stream, tw, tq, to, H,
                      (int *)device_status) == cudaSuccess
               ? MLA_OK
               : MLA_ERR_CUDA;
}

extern "C" mla_status mla_project_output(const float *out, const void *w_uv, int B, int H, float *y,
                                         int32_t *device_status, void *stream) {
    if (!out || !w_uv || !y || B < 1 || H < 1) return MLA_ERR_INVALID_ARG;
    if (!aligned16(out) || !aligned16(w_uv) || !aligned16(y)) return MLA_ERR_INVALID_ARG;
    const int64_t tiles = (int64_t)H * ((B + kNb - 1) / kNb);
    if (tiles > 0x7FFFFFFF) return MLA_ERR_UNSUPPORTED;
    if (!set_attrs()) return MLA_ERR_CUDA;
    CUtensorMap tv, tf;
    // W^UV [H][128][512]: (c, j, h); the latent output [B][H][512] fp32: (c, h, b), boxes of
    // 32 columns x 64 requests
    if (!tmap_3d(&tv, w_uv, kDLatent, kDh, H, kDLatent * 2, (uint64_t)kDh * kDLatent * 2, 64, 128, 1) ||
        !tmap_3d_f32(&tf, out, kDLatent, H, B, kDLatent * 4, (uint64_t)kDLatent * 4 * H, 32, 1, kNb))
        return MLA_ERR_CUDA;
    return launch_pdl(project_kernel, (int)tiles, kPrjThreads, kPrjSmem, (cudaStream_t)stream, tv, tf, y, B, H,
                      (int *)device_status) == cudaSuccess
               ? MLA_OK
               : MLA_ERR_CUDA;
}
