// Non-absorbed (MHA-mode) prefill of one sequence ("MLA & DSA 推理性能优化指南" §3.1 and §1.1:
// the latents are decompressed into per-head keys and values, then standard causal
// attention runs; "MLA 最佳算子全景调研" §4: a FlashAttention variant with 192-wide keys and
// 128-wide values).  The definitions are in include/mla_decode.h (mla_prefill_decompress,
// mla_prefill_attention).
//
// decompress_kernel: per (head, tile of 256 tokens) D[j][t] = sum_c W[h][j][c] c_t[c] for
// W = W^UK and W^UV at once (two TMEM accumulators of 256 columns), K = 512 streamed in
// 64-column chunks through a three-stage TMA ring; the results are transposed through
// shared memory and written by TMA tile stores as K_h, V_h [H][L][128] bf16.
//
// attention_kernel: per (head, two adjacent tiles of 128 queries) a loop over the causal key
// tiles of 128: S = Q K^T on tcgen05 (K = 128 nope + 64 RoPE) into TMEM, online softmax by
// four warps per query tile (one thread per query row, all 128 keys of the tile), P as bf16
// over the first half of that tile's S in TMEM, O += P V on tcgen05 into TMEM (rescaled in
// place only when a row's maximum exceeds its reference by 2^8).  The two query tiles take
// turns on the tensor pipe: while one tile's softmax runs, the other tile's PV and next
// scores run.  Keys are double-buffered in shared memory and shared by both tiles' QK.
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

constexpr int kDh = 128;

// ------------------------------------------------------------------ decompression
constexpr int kDcTok = 256;                       // tokens per CTA (MMA N)
constexpr uint32_t kDcW = 128 * 128;              // 128 rows x 64 bf16 of W^UK or W^UV
constexpr uint32_t kDcC = kDcTok * 128;           // 256 tokens x 64 bf16 of the latent
constexpr uint32_t kDcStage = 2 * kDcW + kDcC;    // 64 KB
constexpr int kDcStages = 3;
constexpr uint32_t kDcBar = kDcStages * kDcStage;
constexpr uint32_t kDcSmem = kDcBar + 128 + 1024;
constexpr int kDcThreads = 192;                   // warps 0-3 epilogue, 4 loads, 5 MMAs

__global__ void __launch_bounds__(kDcThreads, 1) decompress_kernel(const __grid_constant__ CUtensorMap tm_uk,
                                                                   const __grid_constant__ CUtensorMap tm_uv,
                                                                   const __grid_constant__ CUtensorMap tm_c,
                                                                   const __grid_constant__ CUtensorMap tm_k,
                                                                   const __grid_constant__ CUtensorMap tm_v,
                                                                   int H, int *status) {
    extern __shared__ unsigned char smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    unsigned char *gbase = smem_raw + (base - raw);
    const uint32_t bars = base + kDcBar;  // full[3], empty[3], done
    int *abort_flag = reinterpret_cast<int *>(gbase + kDcBar + 64);
    volatile uint32_t *tslot = reinterpret_cast<volatile uint32_t *>(gbase + kDcBar + 72);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int h = blockIdx.x % H;
    const int t0 = (blockIdx.x / H) * kDcTok;
    auto full = [&](int s) { return bars + 8u * s; };
    auto empty = [&](int s) { return bars + 24u + 8u * s; };
    const uint32_t done = bars + 48u;

    if (warp == 0) {
        if (lane == 0) {
            for (int s = 0; s < kDcStages; ++s) {
                mbar_init(full(s), 1);
                mbar_init(empty(s), 1);
            }
            mbar_init(done, 1);
            *abort_flag = 0;
            fence_mbar_init();
        }
        __syncwarp();
        tmem_alloc(smem_u32(const_cast<uint32_t *>(tslot)), 512);
        tmem_relinquish();
    }
    grid_dep_wait();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;  // K accumulator at column 0, V at 256
    bool ok = true;
    constexpr int kChunks = kDLatent / 64;
    if (warp == 4 && lane == 0) {
        for (int c = 0; c < kChunks && ok; ++c) {
            const int s = c % kDcStages;
            if (c >= kDcStages) ok = wait_bounded(empty(s), ((c / kDcStages) - 1) & 1, abort_flag);
            if (!ok) break;
            const uint32_t st = base + s * kDcStage;
            mbar_arrive_expect_tx(full(s), kDcStage);
            tma_load_3d(st, &tm_uk, 64 * c, 0, h, full(s));
            tma_load_3d(st + kDcW, &tm_uv, 64 * c, 0, h, full(s));
            tma_load_2d(st + 2 * kDcW, &tm_c, 64 * c, t0, full(s));
        }
    } else if (warp == 5 && lane == 0) {
        constexpr uint32_t idesc = idesc_bf16_major(128, kDcTok, false, false);
        for (int c = 0; c < kChunks && ok; ++c) {
            const int s = c % kDcStages;
            ok = wait_bounded(full(s), (c / kDcStages) & 1, abort_flag);
            if (!ok) break;
            tc_fence_after();
            const uint32_t st = base + s * kDcStage;
            for (int k = 0; k < 4; ++k) {
                const uint64_t bd = smem_desc_sw128(st + 2 * kDcW + k * 32u, 16u, 1024u);
                mma_ss(tmem, smem_desc_sw128(st + k * 32u, 16u, 1024u), bd, idesc, (c | k) ? 1u : 0u);
                mma_ss(tmem + 256u, smem_desc_sw128(st + kDcW + k * 32u, 16u, 1024u), bd, idesc, (c | k) ? 1u : 0u);
            }
            mma_commit(empty(s));
        }
        if (ok) mma_commit(done);
    }
    grid_dep_launch();
    if (warp < 4) {
        ok = wait_bounded(done, 0, abort_flag);
        tc_fence_after();
        if (ok) {
            // both results transposed into [256 tokens][64 bf16] boxes over the (finished)
            // ring: K in boxes 0-1, V in boxes 2-3 (32 KB each)
            const int j = 32 * warp + lane;
            const uint32_t taddr = tmem + ((uint32_t)(32 * warp) << 16);
            for (int m = 0; m < 2; ++m) {
                const uint32_t box = base + (2 * m + (j >> 6)) * (kDcTok * 128);
                const int jj = j & 63;
#pragma unroll 1
                for (int ch = 0; ch < kDcTok / 32; ++ch) {
                    uint32_t r[32];
                    tmem_ld32(taddr + 256u * m + 32u * ch, r);
                    tmem_wait_ld();
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        const int t = 32 * ch + i;
                        st_shared_u16(box + t * 128 + (((jj >> 3) ^ (t & 7)) << 4) + (jj & 7) * 2,
                                      bf16_bits(__uint_as_float(r[i])));
                    }
                }
            }
            fence_proxy_async_smem();
        }
    }
    if (__syncthreads_and(ok ? 1 : 0) && threadIdx.x == 0) {
        for (int q = 0; q < 2; ++q) {
            tma_store_3d(&tm_k, base + q * (kDcTok * 128), 64 * q, t0, h);
            tma_store_3d(&tm_v, base + (2 + q) * (kDcTok * 128), 64 * q, t0, h);
        }
        bulk_commit_group();
        bulk_wait_group0();
    }
    if (!ok) {
        if (threadIdx.x == 0 && status) record_error(status, MLA_ERR_TIMEOUT);
        drain_pause();
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

// ------------------------------------------------------------------ attention
// Two query tiles per CTA (tiles 2p and 2p + 1 of a head, "A" and "B"): while one tile's
// softmax runs, the tensor pipe works on the other tile's PV and next scores.  Each tile has
// its scores S and its accumulator O in TMEM; P (bf16) overwrites the first 64 columns of its
// S once the scores are read (the next S of that tile is issued after its PV, and the tensor
// pipe runs them in order).  A key tile is read by both query tiles' QK; B, one tile further
// down the diagonal, takes one key tile more.
constexpr int kAtQ = 128;                  // queries per tile (MMA M)
constexpr int kAtK = 128;                  // keys per tile (MMA N of the scores, K of PV)
constexpr uint32_t kAtBox = 128 * 128;     // 128 rows x 64 bf16
constexpr uint32_t kOffQ = 0;              // per query tile: q nope (2 boxes) + q rope (1 box)
constexpr uint32_t kOffK = 6 * kAtBox;     // two key buffers: k nope (2 boxes) + k rope (1 box)
constexpr uint32_t kOffV = 12 * kAtBox;    // one value buffer (2 boxes: 128 keys x 64 value columns)
constexpr uint32_t kAtBar = 14 * kAtBox;
constexpr uint32_t kAtSmem = kAtBar + 256 + 1024;
// warps 0-3 softmax of tile A, 4-7 of tile B (one thread per query row), 8 query/key loads,
// 9 MMAs, 10 value loads
constexpr int kAtThreads = 32 * 11;
constexpr float kRescaleLog2 = 8.0f;       // a row's reference maximum moves only when exceeded by 2^8
// TMEM: tile X (0 = A, 1 = B) has S at 256 X, O at 256 X + 128; P at 256 X (bf16 pairs)
constexpr uint32_t kColS = 0, kColO = 128;
constexpr int kAtHeadGroup = 8;         // heads whose pairs are ordered together

__global__ void __launch_bounds__(kAtThreads, 1) attention_kernel(
    const __grid_constant__ CUtensorMap tm_qn, const __grid_constant__ CUtensorMap tm_qr,
    const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_kr,
    const __grid_constant__ CUtensorMap tm_v, int L, int H, float scale_log2, float *out, float *lse, int *status) {
    extern __shared__ unsigned char smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    unsigned char *gbase = smem_raw + (base - raw);
    const uint32_t bars = base + kAtBar;
    // barriers: q_full; per key buffer b: k_full, k_empty; the value buffer: v_full, v_empty;
    // per query tile X: s_full (its scores are in TMEM), p_full (its P is, one arrival per
    // softmax warp), pv_done (its PV has finished)
    const uint32_t q_full = bars;
    auto k_full = [&](int b) { return bars + 8u + 8u * b; };
    auto k_empty = [&](int b) { return bars + 24u + 8u * b; };
    const uint32_t v_full = bars + 40, v_empty = bars + 48;
    auto s_full = [&](int x) { return bars + 56u + 8u * x; };
    auto p_full = [&](int x) { return bars + 72u + 8u * x; };
    auto pv_done = [&](int x) { return bars + 88u + 8u * x; };
    int *abort_flag = reinterpret_cast<int *>(gbase + kAtBar + 128);
    volatile uint32_t *tslot = reinterpret_cast<volatile uint32_t *>(gbase + kAtBar + 136);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nqt = (L + kAtQ - 1) / kAtQ;
    const int npair = (nqt + 1) / 2;
    // Groups of kAtHeadGroup heads in turn: the CTAs resident at once share a few heads' keys
    // and values (2 MB a head at 4,096 tokens), which then stay in L2; within a group the
    // longest pairs of all its heads first, so that every group, the last one too, ends on
    // its shortest pairs.
    const int g0 = (int)(blockIdx.x / (kAtHeadGroup * npair)) * kAtHeadGroup;
    const int hg = min(kAtHeadGroup, H - g0);        // heads in this group
    const int r = (int)blockIdx.x - g0 * npair;
    const int h = g0 + r % hg;
    const int pr = npair - 1 - r / hg;
    const int qa = 2 * pr;                           // query tile A; B = qa + 1 if it exists
    const bool has_b = qa + 1 < nqt;
    const int nt_b = has_b ? qa + 2 : 0;             // causal: key tiles 0 .. q tile (A: qa + 1)
    const int ntot = has_b ? qa + 2 : qa + 1;        // key tiles loaded
    auto ntiles = [&](int x) { return x == 0 ? qa + 1 : nt_b; };

    if (warp == 0) {
        if (lane == 0) {
            mbar_init(q_full, 1);
            for (int b = 0; b < 2; ++b) {
                mbar_init(k_full(b), 1);
                mbar_init(k_empty(b), 1);
                mbar_init(s_full(b), 1);
                mbar_init(p_full(b), 4);
                mbar_init(pv_done(b), 1);
            }
            mbar_init(v_full, 1);
            mbar_init(v_empty, 1);
            *abort_flag = 0;
            fence_mbar_init();
        }
        __syncwarp();
        tmem_alloc(smem_u32(const_cast<uint32_t *>(tslot)), 512);
        tmem_relinquish();
    }
    grid_dep_wait();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;
    bool ok = true;

    if (warp == 8) {
        // both query tiles once, then the keys of tile g into buffer g % 2 once the last QK of
        // tile g - 2 has read it
        if (lane == 0) {
            mbar_arrive_expect_tx(q_full, (has_b ? 6 : 3) * kAtBox);
            for (int x = 0; x < (has_b ? 2 : 1); ++x) {
                const int q0 = (qa + x) * kAtQ;
                const uint32_t qd = base + kOffQ + 3 * kAtBox * x;
                tma_load_3d(qd, &tm_qn, 0, h, q0, q_full);
                tma_load_3d(qd + kAtBox, &tm_qn, 64, h, q0, q_full);
                tma_load_3d(qd + 2 * kAtBox, &tm_qr, 0, h, q0, q_full);
            }
            for (int g = 0; g < ntot && ok; ++g) {
                const int k0 = g * kAtK, kb = g & 1;
                if (g >= 2) ok = wait_bounded(k_empty(kb), ((g >> 1) - 1) & 1, abort_flag);
                if (!ok) break;
                const uint32_t kd = base + kOffK + kb * 3 * kAtBox;
                mbar_arrive_expect_tx(k_full(kb), 3 * kAtBox);
                tma_load_3d(kd, &tm_k, 0, k0, h, k_full(kb));
                tma_load_3d(kd + kAtBox, &tm_k, 64, k0, h, k_full(kb));
                tma_load_2d(kd + 2 * kAtBox, &tm_kr, kDLatent, k0, k_full(kb));
            }
        }
    } else if (warp == 10) {
        // the values of tile g once the last PV of tile g - 1 has read the buffer
        if (lane == 0) {
            for (int g = 0; g < ntot && ok; ++g) {
                if (g >= 1) ok = wait_bounded(v_empty, (g - 1) & 1, abort_flag);
                if (!ok) break;
                mbar_arrive_expect_tx(v_full, 2 * kAtBox);
                tma_load_3d(base + kOffV, &tm_v, 0, g * kAtK, h, v_full);
                tma_load_3d(base + kOffV + kAtBox, &tm_v, 64, g * kAtK, h, v_full);
            }
        }
    } else if (warp == 9) {
        // the whole warp runs the issue loop (its waits made warp-uniform); one elected lane
        // issues each MMA and commit
        auto wait_w = [&](uint32_t bar, uint32_t parity) {
            return __all_sync(0xffffffffu, wait_quick(bar, parity, abort_flag));
        };
        {
            constexpr uint32_t idesc_s = idesc_bf16_major(128, kAtK, false, false);
            constexpr uint32_t idesc_o = idesc_bf16_major(128, kDh, false, true);
            // S_x(g): 8 steps over the 128 nope columns, 4 over RoPE; the key buffer goes back
            // after the last query tile that reads it
            auto qk = [&](int x, int g) -> bool {
                const int b = g & 1;
                if (!wait_w(k_full(b), (g >> 1) & 1)) return false;
                tc_fence_after();
                const uint32_t kd = base + kOffK + b * 3 * kAtBox, qd = base + kOffQ + 3 * kAtBox * x;
                for (int k = 0; k < 12; ++k) {
                    const uint32_t off = (k >> 2) * kAtBox + (k & 3) * 32u;
                    mma_ss_warp(tmem + 256u * x + kColS, smem_desc_sw128(qd + off, 16u, 1024u),
                                smem_desc_sw128(kd + off, 16u, 1024u), idesc_s, k > 0 ? 1u : 0u);
                }
                mma_commit_warp(s_full(x));
                if (x == 1 || g >= nt_b) mma_commit_warp(k_empty(b));
                return true;
            };
            // O_x += P_x(g) V(g); the value buffer goes back after the last query tile's PV
            auto pv = [&](int x, int g) -> bool {
                if (!wait_w(p_full(x), g & 1) || !wait_w(v_full, g & 1))
                    return false;
                tc_fence_after();
                for (int k = 0; k < kAtK / 16; ++k) {
                    // A: P in TMEM, 16 keys = 8 columns of bf16 pairs; B: 16 key rows of V
                    const uint64_t bd = smem_desc_sw128(base + kOffV + k * 2048u, kAtBox, 1024u);
                    mma_ts_warp(tmem + 256u * x + kColO, tmem + 256u * x + kColS + 8u * k, bd, idesc_o,
                                (g > 0 || k > 0) ? 1u : 0u);
                }
                mma_commit_warp(pv_done(x));
                if (x == 1 || g >= nt_b) mma_commit_warp(v_empty);
                return true;
            };
            ok = wait_w(q_full, 0) && qk(0, 0) && (!has_b || qk(1, 0));
            for (int g = 0; g < ntot && ok; ++g) {
                for (int x = 0; x < 2 && ok; ++x) {
                    if (g >= ntiles(x)) continue;
                    ok = pv(x, g) && (g + 1 >= ntiles(x) || qk(x, g + 1));
                }
            }
        }
    } else {
        // ---------------------------------------------------------------- softmax
        // warps 4x .. 4x + 3: query tile x, rows 32 (w % 4) .. (its TMEM lanes), one thread per
        // row over the tile's 128 keys
        const int x = warp >> 2, quad = warp & 3;
        const int row = 32 * quad + lane;
        const int qi = (qa + x) * kAtQ + row;
        const uint32_t lane_base = (uint32_t)(32 * quad) << 16;
        const uint32_t cS = tmem + lane_base + 256u * x + kColS, cO = tmem + lane_base + 256u * x + kColO;
        const int nt = ntiles(x);
        float m = -INFINITY, l = 0.f;  // reference maximum (log2 units), running sum
        for (int g = 0; g < nt && ok; ++g) {
            const int k0 = g * kAtK;
            ok = wait_bounded(s_full(x), g & 1, abort_flag);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            tc_fence_after();
            float s[kAtK];
#pragma unroll
            for (int c = 0; c < kAtK / 32; ++c) {
                uint32_t r[32];
                tmem_ld32(cS + 32u * c, r);
                tmem_wait_ld();
#pragma unroll
                for (int i = 0; i < 32; ++i) s[32 * c + i] = __uint_as_float(r[i]);
            }
            // causal mask (and keys past the sequence) on the diagonal tiles
            const int lim = min(qi, L - 1) - k0;  // columns c <= lim are seen
            if (__any_sync(0xffffffffu, lim < kAtK - 1)) {
#pragma unroll
                for (int c = 0; c < kAtK; ++c) s[c] = c <= lim ? s[c] : -INFINITY;
            }
            // the row maximum over the raw scores (the scale is positive, so the order is
            // theirs), in eight independent chains
            float mxs[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) mxs[j] = s[j];
#pragma unroll
            for (int c = 8; c < kAtK; ++c) mxs[c & 7] = fmaxf(mxs[c & 7], s[c]);
            const float mx = fmaxf(m, scale_log2 * fmaxf(fmaxf(fmaxf(mxs[0], mxs[1]), fmaxf(mxs[2], mxs[3])),
                                                         fmaxf(fmaxf(mxs[4], mxs[5]), fmaxf(mxs[6], mxs[7]))));
            // the reference maximum moves only when the row maximum exceeds it by 2^8, so most
            // tiles keep it and leave O alone (probabilities stay <= 2^8); key 0 is always seen,
            // so mx is finite
            const float mref = (m == -INFINITY || mx > m + kRescaleLog2) ? mx : m;
            const float alpha = (m == -INFINITY) ? 0.f : ex2_approx(m - mref);
            // p = 2^(s scale_log2 - mref), the scale folded into the exponent's FMA; the P row as
            // bf16 pairs (lower key in the low half) over the first 64 columns of this tile's S
            // (read above): the A operand of PV
            float sums[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                uint32_t pv[32];
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    const float p0 = ex2_approx(fmaf(s[64 * c + 2 * i], scale_log2, -mref));
                    const float p1 = ex2_approx(fmaf(s[64 * c + 2 * i + 1], scale_log2, -mref));
                    sums[i & 3] += p0 + p1;
                    pv[i] = bf16x2_bits(p0, p1);
                }
                tmem_st32(cS + 32u * c, pv);
            }
            const float sum = (sums[0] + sums[1]) + (sums[2] + sums[3]);
            l = l * alpha + sum;
            m = mref;
            // O is rescaled (rarely) once the previous PV of this tile has finished; the next
            // PV waits for this tile's P
            if (g > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
                ok = wait_bounded(pv_done(x), (g - 1) & 1, abort_flag);
                ok = __all_sync(0xffffffffu, ok);
                if (!ok) break;
                tc_fence_after();
#pragma unroll 1
                for (int c = 0; c < kDh / 32; ++c) {
                    uint32_t r[32];
                    tmem_ld32(cO + 32u * c, r);
                    tmem_wait_ld();
#pragma unroll
                    for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * alpha);
                    tmem_st32(cO + 32u * c, r);
                }
            }
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(p_full(x));
        }
        if (ok && nt > 0) {
            ok = wait_bounded(pv_done(x), (nt - 1) & 1, abort_flag);
            ok = __all_sync(0xffffffffu, ok);
        }
        if (ok && nt > 0) {
            tc_fence_after();
            const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll 1
            for (int c = 0; c < kDh / 32; ++c) {
                uint32_t r[32];
                tmem_ld32(cO + 32u * c, r);
                tmem_wait_ld();
                if (qi < L) {
                    float4 *dst = reinterpret_cast<float4 *>(out + ((int64_t)qi * H + h) * kDh + 32 * c);
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        dst[i] = make_float4(__uint_as_float(r[4 * i]) * inv, __uint_as_float(r[4 * i + 1]) * inv,
                                             __uint_as_float(r[4 * i + 2]) * inv, __uint_as_float(r[4 * i + 3]) * inv);
                }
            }
            if (qi < L) lse[(int64_t)qi * H + h] = (m + log2f(l)) * kLn2;
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
        tmem_dealloc(tmem, 512);
    }
}

bool tmap_bf16(CUtensorMap *m, const void *p, int rank, const uint64_t *d, const uint64_t *s, const uint32_t *b) {
    return tmap_tiled(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, p, rank, d, s, b);
}

bool set_prefill_attrs() {
    static bool done[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return false;
    if (done[dev]) return true;
    if (cudaFuncSetAttribute(decompress_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kDcSmem) !=
            cudaSuccess ||
        cudaFuncSetAttribute(attention_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kAtSmem) !=
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

extern "C" mla_status mla_prefill_decompress(const void *entries, int L, const void *w_uk, const void *w_uv, int H,
                                             void *k_nope, void *v, int32_t *device_status, void *stream) {
    if (!entries || !w_uk || !w_uv || !k_nope || !v || L < 1 || H < 1) return MLA_ERR_INVALID_ARG;
    if (!aligned16(entries) || !aligned16(w_uk) || !aligned16(w_uv) || !aligned16(k_nope) || !aligned16(v))
        return MLA_ERR_INVALID_ARG;
    const int64_t grid = (int64_t)H * ((L + kDcTok - 1) / kDcTok);
    if (grid > 0x7FFFFFFF) return MLA_ERR_UNSUPPORTED;
    if (!set_prefill_attrs()) return MLA_ERR_CUDA;
    CUtensorMap tuk, tuv, tc, tk, tv;
    const uint64_t dw[3] = {kDLatent, kDh, (uint64_t)H}, sw[2] = {kDLatent * 2, (uint64_t)kDh * kDLatent * 2};
    const uint32_t bw[3] = {64, 128, 1};
    const uint64_t dc[2] = {kDEntry, (uint64_t)L}, sc[1] = {kDEntry * 2};
    const uint32_t bc[2] = {64, kDcTok};
    const uint64_t dkv[3] = {kDh, (uint64_t)L, (uint64_t)H}, skv[2] = {kDh * 2, (uint64_t)kDh * 2 * L};
    const uint32_t bkv[3] = {64, kDcTok, 1};
    if (!tmap_bf16(&tuk, w_uk, 3, dw, sw, bw) || !tmap_bf16(&tuv, w_uv, 3, dw, sw, bw) ||
        !tmap_bf16(&tc, entries, 2, dc, sc, bc) || !tmap_bf16(&tk, k_nope, 3, dkv, skv, bkv) ||
        !tmap_bf16(&tv, v, 3, dkv, skv, bkv))
        return MLA_ERR_CUDA;
    return launch_pdl(decompress_kernel, (int)grid, kDcThreads, kDcSmem, (cudaStream_t)stream, tuk, tuv, tc, tk, tv,
                      H, (int *)device_status) == cudaSuccess
               ? MLA_OK
               : MLA_ERR_CUDA;
}

extern "C" mla_status mla_prefill_attention(const void *q_nope, const void *q_rope, const void *entries,
                                            const void *k_nope, const void *v, int L, int H, float softmax_scale,
                                            float *out, float *lse, int32_t *device_status, void *stream) {
    if (!q_nope || !q_rope || !entries || !k_nope || !v || !out || !lse || L < 1 || H < 1)
        return MLA_ERR_INVALID_ARG;
    if (!(softmax_scale > 0.f) || softmax_scale == INFINITY) return MLA_ERR_INVALID_ARG;
    if (!aligned16(q_nope) || !aligned16(q_rope) || !aligned16(entries) || !aligned16(k_nope) || !aligned16(v) ||
        !aligned16(out))
        return MLA_ERR_INVALID_ARG;
    const int64_t grid = (int64_t)H * (((L + kAtQ - 1) / kAtQ + 1) / 2);
    if (grid > 0x7FFFFFFF) return MLA_ERR_UNSUPPORTED;
    if (!set_prefill_attrs()) return MLA_ERR_CUDA;
    CUtensorMap tqn, tqr, tk, tkr, tv;
    // q nope [L][H][128], q rope [L][H][64]: (cols, h, query); boxes of 64 columns x 128 queries
    const uint64_t dqn[3] = {kDh, (uint64_t)H, (uint64_t)L}, sqn[2] = {kDh * 2, (uint64_t)kDh * 2 * H};
    const uint64_t dqr[3] = {kDRope, (uint64_t)H, (uint64_t)L}, sqr[2] = {kDRope * 2, (uint64_t)kDRope * 2 * H};
    const uint32_t bq[3] = {64, 1, kAtQ};
    // k nope, v [H][L][128]: (cols, key, h); boxes of 64 columns x 128 keys
    const uint64_t dkv[3] = {kDh, (uint64_t)L, (uint64_t)H}, skv[2] = {kDh * 2, (uint64_t)kDh * 2 * L};
    const uint32_t bkv[3] = {64, kAtK, 1};
    // RoPE keys: columns 512 .. 575 of the [L][576] entries
    const uint64_t de[2] = {kDEntry, (uint64_t)L}, se[1] = {kDEntry * 2};
    const uint32_t be[2] = {64, kAtK};
    if (!tmap_bf16(&tqn, q_nope, 3, dqn, sqn, bq) || !tmap_bf16(&tqr, q_rope, 3, dqr, sqr, bq) ||
        !tmap_bf16(&tk, k_nope, 3, dkv, skv, bkv) || !tmap_bf16(&tkr, entries, 2, de, se, be) ||
        !tmap_bf16(&tv, v, 3, dkv, skv, bkv))
        return MLA_ERR_CUDA;
    const float scale_log2 = softmax_scale * kLog2e;
    return launch_pdl(attention_kernel, (int)grid, kAtThreads, kAtSmem, (cudaStream_t)stream, tqn, tqr, tk, tkr, tv, L,
                      H, scale_log2, out, lse, (int *)device_status) == cudaSuccess
               ? MLA_OK
               : MLA_ERR_CUDA;
}
