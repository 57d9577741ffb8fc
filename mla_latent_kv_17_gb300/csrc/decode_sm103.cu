// Tensor-core decode kernel for sm_103a (bf16 paged cache).
//
// One work unit = a cluster of two CTAs on two SMs.  Both CTAs walk the same work items
// (request b, token range) tile by tile, one 64-token page per tile; CTA r owns output
// latent columns [256 r, 256 r + 256).
//
//   cache tile (TMA, 128-B swizzle)   CTA 0: latent 0..255          (4 boxes of 64 columns)
//                                     CTA 1: latent 256..511 + RoPE (5 boxes)
//   QK^T  S_r[h, t] = Q_r[h, :] . C_r[t, :]   tcgen05.mma M=128 (heads), N=64 (tokens),
//         A = the CTA's query slice held in TMEM, B = the cache tile (K-major)
//   S exchange: each CTA sends its fp32 partial scores to the peer through distributed
//         shared memory; both then hold S = S_0 + S_1 (the full 576-wide score), bitwise
//         identical, so both take identical softmax decisions.
//   softmax: one thread per head; online maximum with lazy rescaling (O is rescaled only
//         when the running maximum grows by more than 2^8), p = 2^(s*scale*log2e - m)
//         rounded to bf16 into TMEM.
//   PV    O_r[h, :] += P[h, :] . C_r[:, latent half]   M=128, N=256, K=64 tokens,
//         A = P in TMEM, B = the same cache tile (MN-major); O_r (128 x 256 fp32) in TMEM.
//   epilogue: out = O / l, lse = (m + log2 l) ln 2, or a partial result for the merge.
//
// TMEM columns: O [0,256)  S [256,320)  P [320,352)  Q [352,512).
// Warp roles: warps 0-3 softmax/epilogue (thread = head, warp w reads TMEM lanes
// 32w..32w+31), warp 4 TMA producer, warp 5 MMA issuer (and TMEM owner).
// Every wait is bounded: on timeout the kernel records MLA_ERR_TIMEOUT, stops issuing,
// and all roles fall through to a clean exit.
#include <cuda.h>
#include <cuda_bf16.h>

#include "common.cuh"
#include "launch.h"
#include "sm103_ptx.cuh"

namespace mla {
namespace {

using namespace ptx;

constexpr int kStages = 3;
constexpr uint32_t kBoxBytes = 64 * 128;            // 64 rows x 64 bf16 (128 B), SW128
constexpr uint32_t kStageBytes = 5 * kBoxBytes;      // 4 latent boxes + the RoPE box
constexpr uint32_t kXBytes = 128 * 64 * 4;           // one exchange buffer: 128 heads x 64 fp32
constexpr int kThreads = 192;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColO = 0, kColS = 256, kColP = 320, kColQ = 352;
constexpr float kRescaleLog2 = 8.0f;
constexpr long long kSpinCycles = 4000000000LL;      // about two seconds

constexpr uint32_t kOffStages = 0;
constexpr uint32_t kOffX = kStages * kStageBytes;
constexpr uint32_t kOffBar = kOffX + 2 * kXBytes;
constexpr uint32_t kOffMisc = kOffBar + 8 * 32;
constexpr uint32_t kSmemBytes = kOffMisc + 64 + 1024;  // + slack for 1024-B alignment

enum {
    B_KV_FULL = 0,
    B_KV_EMPTY = kStages,
    B_S_FULL = 2 * kStages,
    B_S_FREE,
    B_P_FULL,
    B_O_DONE,
    B_Q_READY,
    B_X_FULL0,
    B_X_FULL1,
    B_X_EMPTY0,
    B_X_EMPTY1,
    B_COUNT
};
static_assert(B_COUNT <= 32, "barrier area");

struct Ctx {
    uint32_t base;
    int *status;
    volatile uint32_t *abort;
};

__device__ __forceinline__ uint32_t bar(uint32_t base, int i) { return base + kOffBar + 8u * i; }

// Bounded wait by the calling thread.  False on timeout (recorded) or when another role
// has already given up.
__device__ bool wait_bar(const Ctx &c, uint32_t b, uint32_t parity, bool cluster_scope) {
    const long long t0 = (long long)clock64_now();
    for (uint32_t i = 0;; ++i) {
        const bool ok = cluster_scope ? mbar_try_wait_cluster(b, parity) : mbar_try_wait(b, parity);
        if (ok) return true;
        if ((i & 63u) == 63u) {
            if (*c.abort) return false;
            if ((long long)clock64_now() - t0 > kSpinCycles) {
                *c.abort = 1u;
                record_error(c.status, MLA_ERR_TIMEOUT);
                return false;
            }
        }
    }
}

// All lanes of a warp wait; the outcome is made warp-uniform.
__device__ __forceinline__ bool warp_wait(const Ctx &c, uint32_t b, uint32_t parity,
                                          bool cluster_scope) {
    const bool ok = wait_bar(c, b, parity, cluster_scope);
    return __all_sync(0xffffffffu, ok);
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
decode_sm103_kernel(const __grid_constant__ CUtensorMap tmap, DecodeArgs a) {
    extern __shared__ uint8_t smem_raw[];
    if (!plan_matches(a)) {
        if (threadIdx.x == 0 && blockIdx.x == 0) record_error(a.status, MLA_ERR_WORKSPACE);
        return;
    }
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *gbase = smem_raw + (base - raw);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank(), peer = rank ^ 1u;
    volatile uint32_t *misc = reinterpret_cast<volatile uint32_t *>(gbase + kOffMisc);
    // misc[0]: TMEM base address, misc[1]: abort flag, misc[2 + s]: stage s holds no data
    Ctx c{base, a.status, misc + 1};

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(bar(base, B_KV_FULL + s), 1);
            mbar_init(bar(base, B_KV_EMPTY + s), 1);
        }
        mbar_init(bar(base, B_S_FULL), 1);
        mbar_init(bar(base, B_S_FREE), 4);
        mbar_init(bar(base, B_P_FULL), 4);
        mbar_init(bar(base, B_O_DONE), 1);
        mbar_init(bar(base, B_Q_READY), 4);
        for (int k = 0; k < 2; ++k) {
            mbar_init(bar(base, B_X_FULL0 + k), 4);
            mbar_init(bar(base, B_X_EMPTY0 + k), 4);
        }
        misc[1] = 0u;
        fence_mbar_init();
    }
    if (warp == 5) {
        tmem_alloc(smem_u32(const_cast<uint32_t *>(misc)), kTmemCols);
        tmem_relinquish();
    }
    if (warp == 4 && lane == 0) prefetch_tmap(&tmap);
    tc_fence_before();
    cluster_sync();
    tc_fence_after();
    const uint32_t tmem = misc[0];

    const PlanHeader *hd = reinterpret_cast<const PlanHeader *>(a.ws);
    const WsLayout L = ws_layout(hd->B, hd->H, hd->num_units);
    const int32_t *unit_begin = reinterpret_cast<const int32_t *>(a.ws + L.unit_begin);
    const WorkItem *items = reinterpret_cast<const WorkItem *>(a.ws + L.items);
    float *part_lse = reinterpret_cast<float *>(const_cast<unsigned char *>(a.ws) + L.part_lse);
    float *part_o = reinterpret_cast<float *>(const_cast<unsigned char *>(a.ws) + L.part_o);
    const int units = hd->num_units;
    const int cl = (int)cluster_id_x(), ncl = (int)nclusters_x();

    if (warp == 4) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            const int nbox = 4 + (int)rank;
            const int x0 = rank == 0 ? 0 : 256;
            uint32_t kv_it = 0;
            bool ok = true;
            for (int u = cl; u < units && ok; u += ncl) {
                for (int it = unit_begin[u]; it < unit_begin[u + 1] && ok; ++it) {
                    const WorkItem w = items[it];
                    for (int t = w.t0; t < w.t1; t += kTileTokens, ++kv_it) {
                        const int st = (int)(kv_it % kStages);
                        const uint32_t ph = (kv_it / kStages) & 1u;
                        if (!wait_bar(c, bar(base, B_KV_EMPTY + st), ph ^ 1u, false)) {
                            ok = false;
                            break;
                        }
                        const int lp = t / kPageRows;
                        const int64_t page =
                            lp < a.max_pages ? (int64_t)a.block_table[(int64_t)w.b * a.max_pages + lp] : -1;
                        const uint32_t dst = base + kOffStages + st * kStageBytes;
                        const uint32_t fb = bar(base, B_KV_FULL + st);
                        if (page >= 0 && page < a.num_pages) {
                            misc[2 + st] = 0u;
                            mbar_arrive_expect_tx(fb, nbox * kBoxBytes);
                            for (int i = 0; i < nbox; ++i)
                                tma_load_2d(dst + i * kBoxBytes, &tmap, x0 + 64 * i,
                                            (int32_t)(page * kPageRows), fb);
                        } else {
                            record_error(a.status, MLA_ERR_INDEX);
                            misc[2 + st] = 1u;
                            mbar_arrive(fb);
                        }
                    }
                }
            }
            if (!ok) {
                // give loads already in flight a bounded time to land before exit
                const long long t0 = (long long)clock64_now();
                while ((long long)clock64_now() - t0 < 20000000LL) {
                }
            }
        }
    } else if (warp == 5) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            const int nk = 16 + 4 * (int)rank;  // QK^T K-steps of 16
            constexpr uint32_t idesc_qk = idesc_bf16(128, 64, false);
            constexpr uint32_t idesc_pv = idesc_bf16(128, 256, true);
            uint32_t kv_it = 0, g = 0, nitem = 0;
            bool ok = true;
            auto issue_pv = [&](int stage, uint32_t gp, bool first) -> bool {
                if (!wait_bar(c, bar(base, B_P_FULL), gp & 1u, false)) return false;
                tc_fence_after();
                const uint32_t sb = base + kOffStages + stage * kStageBytes;
                for (int kk = 0; kk < 4; ++kk) {
                    const uint64_t bd = smem_desc_sw128(sb + kk * 2048u, kBoxBytes, 1024u);
                    mma_ts(tmem + kColO, tmem + kColP + 8u * kk, bd, idesc_pv,
                           (first && kk == 0) ? 0u : 1u);
                }
                mma_commit(bar(base, B_O_DONE));
                mma_commit(bar(base, B_KV_EMPTY + stage));
                return true;
            };
            for (int u = cl; u < units && ok; u += ncl) {
                for (int it = unit_begin[u]; it < unit_begin[u + 1] && ok; ++it) {
                    const WorkItem w = items[it];
                    const int ntiles = (w.t1 - w.t0 + kTileTokens - 1) / kTileTokens;
                    if (ntiles <= 0) continue;
                    if (!wait_bar(c, bar(base, B_Q_READY), nitem & 1u, false)) {
                        ok = false;
                        break;
                    }
                    ++nitem;
                    tc_fence_after();
                    int prev = 0;
                    for (int j = 0; j < ntiles; ++j, ++kv_it, ++g) {
                        const int st = (int)(kv_it % kStages);
                        const uint32_t ph = (kv_it / kStages) & 1u;
                        if (!wait_bar(c, bar(base, B_KV_FULL + st), ph, false) ||
                            (g > 0 && !wait_bar(c, bar(base, B_S_FREE), (g - 1) & 1u, false))) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const uint32_t sb = base + kOffStages + st * kStageBytes;
                        for (int k = 0; k < nk; ++k) {
                            const uint64_t bd = smem_desc_sw128(sb + (k >> 2) * kBoxBytes + (k & 3) * 32u,
                                                                16u, 1024u);
                            mma_ts(tmem + kColS, tmem + kColQ + 8u * k, bd, idesc_qk, k > 0 ? 1u : 0u);
                        }
                        mma_commit(bar(base, B_S_FULL));
                        if (j > 0 && !issue_pv(prev, g - 1, j == 1)) {
                            ok = false;
                            break;
                        }
                        prev = st;
                    }
                    if (ok && !issue_pv(prev, g - 1, ntiles == 1)) ok = false;
                }
            }
            if (!ok) {
                // let issued MMAs drain before TMEM is released
                const long long t0 = (long long)clock64_now();
                while ((long long)clock64_now() - t0 < 20000000LL) {
                }
            }
        }
    } else {
        // ------------------------------------------------------------ softmax + epilogue
        const int h = threadIdx.x;  // head row = TMEM lane
        const uint32_t trow = tmem + ((uint32_t)(warp * 32) << 16);
        const uint32_t xbase = base + kOffX;
        const uint32_t peer_x = mapa(xbase, peer);
        uint32_t kv_it = 0, g = 0, nitem = 0;
        bool ok = true;
        for (int u = cl; u < units && ok; u += ncl) {
            for (int it = unit_begin[u]; it < unit_begin[u + 1] && ok; ++it) {
                const WorkItem w = items[it];
                const int b = w.b;
                const int ntiles = (w.t1 - w.t0 + kTileTokens - 1) / kTileTokens;
                float *orow;
                float *lrow;
                if (w.slot < 0) {
                    orow = a.out + ((int64_t)b * a.H + h) * kDLatent + rank * 256;
                    lrow = a.lse + (int64_t)b * a.H + h;
                } else {
                    orow = part_o + ((int64_t)w.slot * a.H + h) * kDLatent + rank * 256;
                    lrow = part_lse + (int64_t)w.slot * a.H + h;
                }
                if (ntiles <= 0) {
                    if (h < a.H) {
                        for (int q = 0; q < 64; ++q)
                            reinterpret_cast<float4 *>(orow)[q] = make_float4(0.f, 0.f, 0.f, 0.f);
                        if (rank == 0) *lrow = -INFINITY;
                    }
                    continue;
                }
                // query slice -> TMEM (K-major bf16 pairs, one head per lane)
                {
                    const uint16_t *qn = a.q_nope + ((int64_t)b * a.H + h) * kDLatent + rank * 256;
                    const uint16_t *qr = a.q_rope + ((int64_t)b * a.H + h) * kDRope;
                    const int nch = 4 + (int)rank;
                    for (int cb = 0; cb < nch; ++cb) {
                        uint32_t v[32];
                        const uint4 *src = reinterpret_cast<const uint4 *>(cb < 4 ? qn + cb * 64 : qr);
                        for (int q = 0; q < 8; ++q) {
                            uint4 x = make_uint4(0u, 0u, 0u, 0u);
                            if (h < a.H) x = src[q];
                            v[4 * q] = x.x;
                            v[4 * q + 1] = x.y;
                            v[4 * q + 2] = x.z;
                            v[4 * q + 3] = x.w;
                        }
                        tmem_st32(trow + kColQ + 32u * cb, v);
                    }
                    tmem_wait_st();
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(bar(base, B_Q_READY));
                    ++nitem;
                }
                float m = -INFINITY, l = 0.f;
                for (int j = 0; j < ntiles; ++j, ++kv_it, ++g) {
                    const int t = w.t0 + kTileTokens * j;
                    const int st = (int)(kv_it % kStages);
                    const uint32_t ph = (kv_it / kStages) & 1u;
                    if (!warp_wait(c, bar(base, B_S_FULL), g & 1u, false)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    uint32_t sr[64];
                    {
                        uint32_t (&lo)[32] = *reinterpret_cast<uint32_t (*)[32]>(&sr[0]);
                        uint32_t (&hi)[32] = *reinterpret_cast<uint32_t (*)[32]>(&sr[32]);
                        tmem_ld32(trow + kColS, lo);
                        tmem_ld32(trow + kColS + 32u, hi);
                    }
                    tmem_wait_ld();
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(bar(base, B_S_FREE));

                    // ---- exchange partial scores with the peer CTA
                    const uint32_t xb = g & 1u, xu = g >> 1;
                    if (g >= 2 && !warp_wait(c, bar(base, B_X_EMPTY0 + xb), (xu - 1u) & 1u, true)) {
                        ok = false;
                        break;
                    }
                    const uint32_t rdst = peer_x + xb * kXBytes + (uint32_t)h * 256u;
                    for (int q = 0; q < 16; ++q) {
                        const uint32_t pos = (uint32_t)(q ^ (h & 7));
                        st_cluster_v4(rdst + pos * 16u, sr[4 * q], sr[4 * q + 1], sr[4 * q + 2],
                                      sr[4 * q + 3]);
                    }
                    __syncwarp();
                    if (lane == 0) mbar_arrive_cluster(mapa(bar(base, B_X_FULL0 + xb), peer));
                    if (!warp_wait(c, bar(base, B_X_FULL0 + xb), xu & 1u, true)) {
                        ok = false;
                        break;
                    }
                    float s[64];
                    {
                        const float4 *xs = reinterpret_cast<const float4 *>(gbase + kOffX + xb * kXBytes +
                                                                            (uint32_t)h * 256u);
                        for (int q = 0; q < 16; ++q) {
                            const float4 v = xs[q ^ (h & 7)];
                            s[4 * q] = __uint_as_float(sr[4 * q]) + v.x;
                            s[4 * q + 1] = __uint_as_float(sr[4 * q + 1]) + v.y;
                            s[4 * q + 2] = __uint_as_float(sr[4 * q + 2]) + v.z;
                            s[4 * q + 3] = __uint_as_float(sr[4 * q + 3]) + v.w;
                        }
                    }
                    __syncwarp();
                    if (lane == 0) mbar_arrive_cluster(mapa(bar(base, B_X_EMPTY0 + xb), peer));

                    // ---- online softmax (identical decisions in both CTAs)
                    if (!warp_wait(c, bar(base, B_KV_FULL + st), ph, false)) {
                        ok = false;
                        break;
                    }
                    const bool bad = misc[2 + st] != 0u;
                    const int nvalid = bad ? 0 : min(kTileTokens, w.t1 - t);
                    float mt = -INFINITY;
#pragma unroll
                    for (int i = 0; i < 64; ++i) {
                        s[i] = i < nvalid ? s[i] * a.scale_log2 : -INFINITY;
                        mt = fmaxf(mt, s[i]);
                    }
                    float alpha = 1.f;
                    bool resc = false;
                    if (mt > m + kRescaleLog2) {
                        alpha = exp2f(m - mt);
                        l *= alpha;
                        m = mt;
                        resc = true;
                    }
                    const float mref = m == -INFINITY ? 0.f : m;
                    uint32_t pk[32];
                    float psum = 0.f;
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        const float p0 = exp2f(s[2 * i] - mref), p1 = exp2f(s[2 * i + 1] - mref);
                        psum += p0 + p1;
                        __nv_bfloat162 v = __floats2bfloat162_rn(p0, p1);
                        pk[i] = *reinterpret_cast<uint32_t *>(&v);
                    }
                    l += psum;

                    // ---- P buffer and O belong to PV of the previous tile until it completes
                    if (j > 0) {
                        if (!warp_wait(c, bar(base, B_O_DONE), (g - 1) & 1u, false)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        if (__any_sync(0xffffffffu, resc)) {
                            const float al = resc ? alpha : 1.f;
                            for (int cb = 0; cb < 256; cb += 32) {
                                uint32_t o[32];
                                tmem_ld32(trow + kColO + cb, o);
                                tmem_wait_ld();
#pragma unroll
                                for (int q = 0; q < 32; ++q) o[q] = __float_as_uint(__uint_as_float(o[q]) * al);
                                tmem_st32(trow + kColO + cb, o);
                            }
                        }
                    }
                    // ---- cache rows this tile must not contribute (page tail, missing page)
                    if (nvalid < kTileTokens) {
                        const uint32_t sb = kOffStages + st * kStageBytes;
                        const int nz = (kTileTokens - nvalid) * 32;  // 16-B chunks in 4 boxes
                        for (int i = h; i < nz; i += 128) {
                            const int row = nvalid + i / 32, ch = i % 32;
                            *reinterpret_cast<uint4 *>(gbase + sb + (ch / 8) * kBoxBytes + row * 128 + (ch % 8) * 16) =
                                make_uint4(0u, 0u, 0u, 0u);
                        }
                        fence_proxy_async_smem();
                    }
                    tmem_st32(trow + kColP, pk);
                    tmem_wait_st();
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(bar(base, B_P_FULL));
                }
                if (!ok) break;
                // ---- epilogue: wait for the last PV, normalise, store
                if (!warp_wait(c, bar(base, B_O_DONE), (g - 1) & 1u, false)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const float inv = l > 0.f ? 1.f / l : 0.f;
                for (int cb = 0; cb < 256; cb += 32) {
                    uint32_t o[32];
                    tmem_ld32(trow + kColO + cb, o);
                    tmem_wait_ld();
                    if (h < a.H) {
                        float4 *dst = reinterpret_cast<float4 *>(orow + cb);
#pragma unroll
                        for (int q = 0; q < 8; ++q)
                            dst[q] = make_float4(__uint_as_float(o[4 * q]) * inv, __uint_as_float(o[4 * q + 1]) * inv,
                                                 __uint_as_float(o[4 * q + 2]) * inv,
                                                 __uint_as_float(o[4 * q + 3]) * inv);
                    }
                }
                if (rank == 0 && h < a.H) *lrow = l > 0.f ? (m + log2f(l)) * kLn2 : -INFINITY;
                tc_fence_before();
            }
        }
    }

    // ---------------------------------------------------------------- teardown
    tc_fence_before();
    __syncthreads();
    cluster_sync();  // the peer may still have been writing into this CTA's shared memory
    if (warp == 5) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

// cuTensorMapEncodeTiled from the driver, looked up once through the runtime.
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    if (!fn) {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    }
    return fn;
}

}  // namespace

int sm103_max_units() {
    static int cached = -1;
    static int cached_dev = -1;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (cached >= 0 && cached_dev == dev) return cached;
    if (cudaFuncSetAttribute(decode_sm103_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)kSmemBytes) != cudaSuccess)
        return 0;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2, 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = kSmemBytes;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeClusterDimension;
    attr.val.clusterDim.x = 2;
    attr.val.clusterDim.y = 1;
    attr.val.clusterDim.z = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, decode_sm103_kernel, &cfg) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    cached = n;
    cached_dev = dev;
    return n;
}

cudaError_t launch_decode_sm103(const DecodeArgs &a, int num_clusters, cudaStream_t stream) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return cudaErrorNotSupported;
    CUtensorMap tmap;
    const cuuint64_t dims[2] = {(cuuint64_t)kDEntry, (cuuint64_t)a.num_pages * kPageRows};
    const cuuint64_t strides[1] = {(cuuint64_t)kDEntry * 2};
    const cuuint32_t box[2] = {64, 64};
    const cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(&tmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<unsigned char *>(a.cache),
                     dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                     CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
    static bool attr_set = false;
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(decode_sm103_kernel,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    decode_sm103_kernel<<<dim3(2 * num_clusters), dim3(kThreads), kSmemBytes, stream>>>(tmap, a);
    return cudaGetLastError();
}

}  // namespace mla
