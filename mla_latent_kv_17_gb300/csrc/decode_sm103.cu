// Tensor-core decode kernel for sm_103a (bf16 paged cache).
//
// One work unit = a cluster of two CTAs on two SMs.  Both CTAs walk the same work items
// (request b, token range) tile by tile, one 64-token page per tile.  CTA r owns
//   * the scores of the page's tokens [32 r, 32 r + 32) — full 576-wide dot products, so no
//     partial score ever crosses between the SMs, and
//   * the output latent columns [256 r, 256 r + 256) of every head (its O half, 128 x 256
//     fp32 in TMEM; the full 128 x 512 accumulator does not fit one SM's TMEM).
// Per tile:
//   TMA (128-B swizzle)  own-half latent of all 64 tokens (PV operand, kept until PV) and
//                        the other 320 columns (other latent half + RoPE) of its own 32
//                        tokens (QK operand only, released after QK).
//   QK^T  S[h, i] = q[h, :] . entry[own token i, :]   tcgen05.mma M=128 heads, N=32,
//         K=576: 448 K from the query slice held in TMEM, 128 K from shared memory.
//   softmax (one thread per head): x = s * scale * log2(e); reference r = the running
//         maximum m, or the tile's own maximum if that exceeds m by more than 8; own
//         weights p = 2^(x - r) in bf16 go to a shared-memory tile, followed by r and the
//         fp32 sum of p; each warp bulk-copies its 32 rows of that (2.25 KB) into the peer's
//         copy of the tile, completing on the peer's mbarrier (9 KB per tile in all).
//   merge: with both CTAs' (r, sum) both compute the same new maximum m', rescale a half
//         whose reference was below m' (2^(r - m')), the sum l and — when m' > m — O, so
//         both hold bitwise identical weights for all 64 tokens.
//   PV    O_r[h, :] += P[h, 0:64] . C[0:64, own latent half]   M=128, N=256, K=64,
//         A = the probability tile (64-B swizzle), B = the own-half cache tile (MN-major).
//   epilogue: out = O / l, lse = (m + log2 l) ln 2, or a partial result for the merge.
//
// TMEM columns: O [0,256)  S [256,288)  query [288,512) (own latent half, RoPE, first 128
// columns of the other half; the last 128 columns of the other half sit in shared memory).
// Warp roles: warps 0-3 softmax/epilogue (thread = head, warp w reads TMEM lanes
// 32w..32w+31), warp 4 TMA producer, warp 5 issues QK^T (and owns TMEM), warp 6 issues
// PV.  Two issuing threads let the tensor pipe take a tile's PV as soon as its weights
// are ready instead of after the next tile's QK^T has been queued.
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

constexpr int kDhStages = 3;   // own-half latent tiles (live until PV)
constexpr int kOthStages = 2;  // other-columns tiles (live until QK)
constexpr int kPSlots = 3;     // probability tiles (live until both CTAs' PV)
constexpr uint32_t kHalfBox = 32 * 128;          // 32 rows x 64 bf16, 128-B swizzle
constexpr uint32_t kDhBlock = 2 * kHalfBox;      // 64 token rows x 64 columns
constexpr uint32_t kDhBytes = 4 * kDhBlock;      // 256 columns
constexpr uint32_t kOthBytes = 5 * kHalfBox;     // 4 x 64 latent columns + RoPE, 32 rows
constexpr uint32_t kQsBox = 128 * 128;           // 128 heads x 64 bf16
constexpr uint32_t kQsBytes = 2 * kQsBox;
constexpr uint32_t kPHalf = 128 * 64;            // 128 heads x 32 tokens bf16, 64-B swizzle
constexpr uint32_t kRlBytes = 1024;              // r[128] and sum[128], fp32
constexpr uint32_t kPSlotBytes = 2 * kPHalf + 2 * kRlBytes;
constexpr uint32_t kMsgBytes = kPHalf + kRlBytes;
constexpr int kThreads = 224;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColO = 0, kColS = 256, kColQ = 288;
constexpr uint32_t kColQRope = kColQ + 128, kColQOther = kColQ + 160;
constexpr float kRescaleLog2 = 8.0f;
constexpr long long kSpinCycles = 4000000000LL;  // about two seconds

constexpr uint32_t kOffDh = 0;
constexpr uint32_t kOffOth = kOffDh + kDhStages * kDhBytes;
constexpr uint32_t kOffQs = kOffOth + kOthStages * kOthBytes;
constexpr uint32_t kOffP = kOffQs + kQsBytes;
constexpr uint32_t kOffBar = kOffP + kPSlots * kPSlotBytes;
constexpr uint32_t kOffMisc = kOffBar + 8 * 32;
constexpr uint32_t kSmemBytes = kOffMisc + 64 + 1024;  // + slack for 1024-B alignment
static_assert(kSmemBytes <= 232448, "shared memory");

enum {
    B_DH_FULL = 0,
    B_DH_EMPTY = B_DH_FULL + kDhStages,
    B_OTH_FULL = B_DH_EMPTY + kDhStages,
    B_OTH_EMPTY = B_OTH_FULL + kOthStages,
    B_S_FULL = B_OTH_EMPTY + kOthStages,
    B_S_FREE,
    B_O_FINAL,                    // the last PV of a work item (waited by the epilogue)
    B_Q_READY,
    B_RFULL,                      // peer's message for probability slot s has landed
    B_PFREE = B_RFULL + kPSlots,  // both CTAs' PV have finished reading slot s
    B_P_FULL = B_PFREE + kPSlots, // slot s holds the merged weights of its tile
    B_COUNT = B_P_FULL + kPSlots
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

__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}
__device__ __forceinline__ void scale_row16(uint4 *prow, float f) {
    for (int q = 0; q < 4; ++q) {
        uint4 v = prow[q];
        v.x = pack_bf16(bf16lo(v.x) * f, bf16hi(v.x) * f);
        v.y = pack_bf16(bf16lo(v.y) * f, bf16hi(v.y) * f);
        v.z = pack_bf16(bf16lo(v.z) * f, bf16hi(v.z) * f);
        v.w = pack_bf16(bf16lo(v.w) * f, bf16hi(v.w) * f);
        prow[q] = v;
    }
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
    // misc[0]: TMEM base address, misc[1]: abort flag, misc[2 + s]: own-half tile s holds
    // no data (its page id was out of range)
    Ctx c{base, a.status, misc + 1};

    if (threadIdx.x == 0) {
        for (int s = 0; s < kDhStages; ++s) {
            mbar_init(bar(base, B_DH_FULL + s), 1);
            mbar_init(bar(base, B_DH_EMPTY + s), 1);
        }
        for (int s = 0; s < kOthStages; ++s) {
            mbar_init(bar(base, B_OTH_FULL + s), 1);
            mbar_init(bar(base, B_OTH_EMPTY + s), 1);
        }
        mbar_init(bar(base, B_S_FULL), 1);
        mbar_init(bar(base, B_S_FREE), 4);
        mbar_init(bar(base, B_O_FINAL), 1);
        mbar_init(bar(base, B_Q_READY), 4);
        for (int s = 0; s < kPSlots; ++s) {
            mbar_init(bar(base, B_RFULL + s), 1);  // + the message bytes
            mbar_init(bar(base, B_PFREE + s), 2);  // one commit from each CTA's PV
            mbar_init(bar(base, B_P_FULL + s), 4);
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
            const int xown = 256 * (int)rank, xoth = 256 * (int)peer;
            uint32_t g = 0;
            bool ok = true;
            for (int u = cl; u < units && ok; u += ncl) {
                for (int it = unit_begin[u]; it < unit_begin[u + 1] && ok; ++it) {
                    const WorkItem w = items[it];
                    for (int t = w.t0; t < w.t1; t += kTileTokens, ++g) {
                        const int ds = (int)(g % kDhStages), os = (int)(g % kOthStages);
                        const uint32_t dph = (g / kDhStages) & 1u, oph = (g / kOthStages) & 1u;
                        if (!wait_bar(c, bar(base, B_DH_EMPTY + ds), dph ^ 1u, false) ||
                            !wait_bar(c, bar(base, B_OTH_EMPTY + os), oph ^ 1u, false)) {
                            ok = false;
                            break;
                        }
                        const int lp = t / kPageRows;
                        const int64_t page =
                            lp < a.max_pages ? (int64_t)a.block_table[(int64_t)w.b * a.max_pages + lp] : -1;
                        const uint32_t dfb = bar(base, B_DH_FULL + ds), ofb = bar(base, B_OTH_FULL + os);
                        if (page >= 0 && page < a.num_pages) {
                            misc[2 + ds] = 0u;
                            const int32_t y = (int32_t)(page * kPageRows);
                            const uint32_t dst_dh = base + kOffDh + ds * kDhBytes;
                            const uint32_t dst_ot = base + kOffOth + os * kOthBytes;
                            mbar_arrive_expect_tx(dfb, kDhBytes);
                            for (int i = 0; i < 4; ++i)
                                for (int hf = 0; hf < 2; ++hf)
                                    tma_load_2d(dst_dh + i * kDhBlock + hf * kHalfBox, &tmap, xown + 64 * i,
                                                y + 32 * hf, dfb);
                            mbar_arrive_expect_tx(ofb, kOthBytes);
                            const int yo = y + 32 * (int)rank;
                            for (int i = 0; i < 4; ++i)
                                tma_load_2d(dst_ot + i * kHalfBox, &tmap, xoth + 64 * i, yo, ofb);
                            tma_load_2d(dst_ot + 4 * kHalfBox, &tmap, kDLatent, yo, ofb);
                        } else {
                            record_error(a.status, MLA_ERR_INDEX);
                            misc[2 + ds] = 1u;
                            mbar_arrive(dfb);
                            mbar_arrive(ofb);
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
        // ------------------------------------------------------------ QK^T issuer
        if (lane == 0) {
            constexpr uint32_t idesc_qk = idesc_bf16(128, 32, false);
            uint32_t g = 0, nitem = 0;
            bool ok = true;
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
                    for (int j = 0; j < ntiles; ++j, ++g) {
                        const int ds = (int)(g % kDhStages), os = (int)(g % kOthStages);
                        const uint32_t dph = (g / kDhStages) & 1u, oph = (g / kOthStages) & 1u;
                        if (!wait_bar(c, bar(base, B_DH_FULL + ds), dph, false) ||
                            !wait_bar(c, bar(base, B_OTH_FULL + os), oph, false) ||
                            (g > 0 && !wait_bar(c, bar(base, B_S_FREE), (g - 1) & 1u, false))) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const uint32_t dh = base + kOffDh + ds * kDhBytes + rank * kHalfBox;
                        const uint32_t ot = base + kOffOth + os * kOthBytes;
                        const uint32_t qs = base + kOffQs;
                        // own latent half: query columns from TMEM, own token rows of the PV tile
                        for (int k = 0; k < 16; ++k)
                            mma_ts(tmem + kColS, tmem + kColQ + 8u * k,
                                   smem_desc_sw128(dh + (k >> 2) * kDhBlock + (k & 3) * 32u, 16u, 1024u),
                                   idesc_qk, k > 0 ? 1u : 0u);
                        // RoPE
                        for (int k = 0; k < 4; ++k)
                            mma_ts(tmem + kColS, tmem + kColQRope + 8u * k,
                                   smem_desc_sw128(ot + 4 * kHalfBox + k * 32u, 16u, 1024u), idesc_qk, 1u);
                        // other latent half, first 128 columns: query from TMEM
                        for (int k = 0; k < 8; ++k)
                            mma_ts(tmem + kColS, tmem + kColQOther + 8u * k,
                                   smem_desc_sw128(ot + (k >> 2) * kHalfBox + (k & 3) * 32u, 16u, 1024u),
                                   idesc_qk, 1u);
                        // other latent half, last 128 columns: query from shared memory
                        for (int k = 0; k < 8; ++k)
                            mma_ss(tmem + kColS,
                                   smem_desc_sw128(qs + (k >> 2) * kQsBox + (k & 3) * 32u, 16u, 1024u),
                                   smem_desc_sw128(ot + (2 + (k >> 2)) * kHalfBox + (k & 3) * 32u, 16u, 1024u),
                                   idesc_qk, 1u);
                        mma_commit(bar(base, B_S_FULL));
                        mma_commit(bar(base, B_OTH_EMPTY + os));
                    }
                }
            }
            if (!ok) {
                // let issued MMAs drain before TMEM is released
                const long long t0 = (long long)clock64_now();
                while ((long long)clock64_now() - t0 < 20000000LL) {
                }
            }
        }
    } else if (warp == 6) {
        // ------------------------------------------------------------ PV issuer
        if (lane == 0) {
            constexpr uint32_t idesc_pv = idesc_bf16(128, 256, true);
            uint32_t g = 0;
            bool ok = true;
            for (int u = cl; u < units && ok; u += ncl) {
                for (int it = unit_begin[u]; it < unit_begin[u + 1] && ok; ++it) {
                    const WorkItem w = items[it];
                    const int ntiles = (w.t1 - w.t0 + kTileTokens - 1) / kTileTokens;
                    for (int j = 0; j < ntiles; ++j, ++g) {
                        // Per-slot barriers: a slot is only reused after both CTAs' PV of its
                        // previous tile, so no barrier here can run two phases ahead.
                        const int slot = (int)(g % kPSlots);
                        if (!wait_bar(c, bar(base, B_P_FULL + slot), (g / kPSlots) & 1u, false)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const int ds = (int)(g % kDhStages);
                        const uint32_t dh = base + kOffDh + ds * kDhBytes;
                        const uint32_t ps = base + kOffP + slot * kPSlotBytes;
                        for (int kk = 0; kk < 4; ++kk) {
                            const uint64_t ad = smem_desc_sw64(ps + (kk >> 1) * kPHalf + (kk & 1) * 32u, 512u);
                            const uint64_t bd = smem_desc_sw128(dh + kk * 2048u, kDhBlock, 1024u);
                            mma_ss(tmem + kColO, ad, bd, idesc_pv, (j == 0 && kk == 0) ? 0u : 1u);
                        }
                        mma_commit(bar(base, B_DH_EMPTY + ds));
                        mma_commit_multicast(bar(base, B_PFREE + slot), (uint16_t)3);
                        if (j == ntiles - 1) mma_commit(bar(base, B_O_FINAL));
                    }
                }
            }
            if (!ok) {
                const long long t0 = (long long)clock64_now();
                while ((long long)clock64_now() - t0 < 20000000LL) {
                }
            }
        }
    } else {
        // ------------------------------------------------------------ softmax + epilogue
        // Per tile: part A (scores -> own weights -> message to the peer), then part B
        // (merge with the peer's message -> PV may start).
        const int h = threadIdx.x;  // head row = TMEM lane
        const uint32_t trow = tmem + ((uint32_t)(warp * 32) << 16);
        const uint32_t peer_p = mapa(base + kOffP, peer);
        const float sc = a.scale_log2;  // > 0, checked on the host
        uint32_t g = 0, nitem = 0;
        bool ok = true;
        struct Pending {
            uint32_t g;
            int j, nvalid;
            float rown, lown;
        };
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
                // ---- query of this request: 448 columns into TMEM, 128 into shared memory
                {
                    const uint16_t *qn = a.q_nope + ((int64_t)b * a.H + h) * kDLatent;
                    const uint16_t *qr = a.q_rope + ((int64_t)b * a.H + h) * kDRope;
                    for (int cb = 0; cb < 7; ++cb) {
                        const uint16_t *src = cb < 4   ? qn + 256 * rank + 64 * cb
                                              : cb == 4 ? qr
                                                        : qn + 256 * peer + 64 * (cb - 5);
                        uint32_t v[32];
                        for (int q = 0; q < 8; ++q) {
                            uint4 x = make_uint4(0u, 0u, 0u, 0u);
                            if (h < a.H) x = reinterpret_cast<const uint4 *>(src)[q];
                            v[4 * q] = x.x;
                            v[4 * q + 1] = x.y;
                            v[4 * q + 2] = x.z;
                            v[4 * q + 3] = x.w;
                        }
                        tmem_st32(trow + kColQ + 32u * cb, v);
                    }
                    for (int bx = 0; bx < 2; ++bx) {
                        const uint4 *src = reinterpret_cast<const uint4 *>(qn + 256 * peer + 128 + 64 * bx);
                        uint8_t *row = gbase + kOffQs + bx * kQsBox + h * 128;
                        for (int q = 0; q < 8; ++q) {
                            uint4 x = make_uint4(0u, 0u, 0u, 0u);
                            if (h < a.H) x = src[q];
                            *reinterpret_cast<uint4 *>(row + ((q ^ (h & 7)) * 16)) = x;
                        }
                    }
                    fence_proxy_async_smem();
                    tmem_wait_st();
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(bar(base, B_Q_READY));
                }
                float m = -INFINITY, l = 0.f;
                Pending pend{0u, -1, 0, 0.f, 0.f};
                for (int j = 0; j < ntiles && ok; ++j) {
                    Pending cur{g, j, 0, 0.f, 0.f};
                    if (j < ntiles) {
                        // ================= part A of tile j
                        const int t = w.t0 + kTileTokens * j;
                        const int ds = (int)(g % kDhStages);
                        const uint32_t dph = (g / kDhStages) & 1u;
                        const int slot = (int)(g % kPSlots);
                        const uint32_t su = g / kPSlots;
                        if (!warp_wait(c, bar(base, B_S_FULL), g & 1u, false) ||
                            !warp_wait(c, bar(base, B_DH_FULL + ds), dph, false)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        float s[32];
                        {
                            uint32_t sr[32];
                            tmem_ld32(trow + kColS, sr);
                            tmem_wait_ld();
#pragma unroll
                            for (int i = 0; i < 32; ++i) s[i] = __uint_as_float(sr[i]);
                        }
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(bar(base, B_S_FREE));
                        const bool bad = misc[2 + ds] != 0u;
                        const int nvalid = bad ? 0 : min(kTileTokens, w.t1 - t);  // page rows attended
                        const int nown = max(0, min(32, nvalid - 32 * (int)rank));
                        if (nown < 32) {
#pragma unroll
                            for (int i = 0; i < 32; ++i)
                                if (i >= nown) s[i] = -INFINITY;
                        }
                        float mraw = s[0];
#pragma unroll
                        for (int i = 1; i < 32; ++i) mraw = fmaxf(mraw, s[i]);
                        const float mloc = mraw * sc;
                        // reference: the running maximum (known after part B of tile j-1 only
                        // for the tiles before it; any value works as long as both CTAs send
                        // the one they used)
                        const float mk = m;
                        const float rown = mloc > mk + kRescaleLog2 ? mloc : mk;
                        const float nr = rown == -INFINITY ? 0.f : -rown;
                        uint32_t pk[16];
                        float lown = 0.f;
#pragma unroll
                        for (int i = 0; i < 16; ++i) {
                            const float p0 = ex2_approx(fmaf(s[2 * i], sc, nr));
                            const float p1 = ex2_approx(fmaf(s[2 * i + 1], sc, nr));
                            lown += p0 + p1;
                            pk[i] = pack_bf16(p0, p1);
                        }
                        // slot reuse: both CTAs' PV of tile g-3 must be done
                        if (g >= (uint32_t)kPSlots &&
                            !warp_wait(c, bar(base, B_PFREE + slot), (su - 1u) & 1u, true)) {
                            ok = false;
                            break;
                        }
                        uint8_t *ps = gbase + kOffP + slot * kPSlotBytes;
                        const uint32_t poff = kOffP + slot * kPSlotBytes;
                        {
                            uint8_t *prow = ps + rank * kPHalf + h * 64;
#pragma unroll
                            for (int q = 0; q < 4; ++q)
                                *reinterpret_cast<uint4 *>(prow + ((q ^ ((h >> 1) & 3)) * 16)) =
                                    make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
                            float *rl = reinterpret_cast<float *>(ps + 2 * kPHalf + rank * kRlBytes);
                            rl[h] = rown;
                            rl[128 + h] = lown;
                        }
                        fence_proxy_async_smem();
                        __syncwarp();
                        const uint32_t rfull = bar(base, B_RFULL + slot);
                        if (threadIdx.x == 0) mbar_arrive_expect_tx(rfull, kMsgBytes);
                        if (lane == 0) {
                            const uint32_t rb = mapa(rfull, peer);
                            const uint32_t prows = poff + rank * kPHalf + warp * 32 * 64;
                            const uint32_t rls = poff + 2 * kPHalf + rank * kRlBytes + warp * 32 * 4;
                            bulk_copy_s2peer(peer_p - kOffP + prows, base + prows, 32 * 64, rb);
                            bulk_copy_s2peer(peer_p - kOffP + rls, base + rls, 32 * 4, rb);
                            bulk_copy_s2peer(peer_p - kOffP + rls + 512, base + rls + 512, 32 * 4, rb);
                            bulk_commit();
                        }
                        cur.nvalid = nvalid;
                        cur.rown = rown;
                        cur.lown = lown;
                        ++g;
                    }
                    pend = cur;
                    if (pend.j >= 0) {
                        // ================= part B of tile pend.j (merge, then PV may start)
                        const uint32_t gp = pend.g;
                        const int ds = (int)(gp % kDhStages);
                        const int slot = (int)(gp % kPSlots);
                        const uint32_t su = gp / kPSlots;
                        const uint32_t rfull = bar(base, B_RFULL + slot);
                        if (!warp_wait(c, rfull, su & 1u, true)) {
                            ok = false;
                            break;
                        }
                        uint8_t *ps = gbase + kOffP + slot * kPSlotBytes;
                        const float *rlp = reinterpret_cast<const float *>(ps + 2 * kPHalf + peer * kRlBytes);
                        const float rpeer = rlp[h], lpeer = rlp[128 + h];
                        const float r0 = rank == 0 ? pend.rown : rpeer, r1 = rank == 0 ? rpeer : pend.rown;
                        const float l0 = rank == 0 ? pend.lown : lpeer, l1 = rank == 0 ? lpeer : pend.lown;
                        const float mn = fmaxf(m, fmaxf(r0, r1));
                        float f0 = 1.f, f1 = 1.f, alpha = 1.f;
                        if (mn != -INFINITY) {
                            f0 = ex2_approx(r0 - mn);
                            f1 = ex2_approx(r1 - mn);
                            alpha = ex2_approx(m - mn);
                            l = l * alpha + l0 * f0 + l1 * f1;
                        }
                        const bool resc_o = pend.j > 0 && mn > m;
                        m = mn;
                        // a half whose reference lies below the new maximum is rescaled in
                        // place (this CTA's own rows only after the warp's bulk copies have
                        // read them)
                        const float fown = rank == 0 ? f0 : f1, fpeer = rank == 0 ? f1 : f0;
                        bool wrote = false;
                        if (__any_sync(0xffffffffu, fown < 1.f)) {
                            if (lane == 0) bulk_wait_read_all();
                            __syncwarp();
                            if (fown < 1.f) scale_row16(reinterpret_cast<uint4 *>(ps + rank * kPHalf + h * 64), fown);
                            wrote = true;
                        }
                        if (fpeer < 1.f) {
                            scale_row16(reinterpret_cast<uint4 *>(ps + peer * kPHalf + h * 64), fpeer);
                            wrote = true;
                        }
                        // cache rows this tile must not contribute (page tail, missing page):
                        // the PV operand must hold zeros there, not whatever the page holds
                        if (pend.nvalid < kTileTokens) {
                            const uint32_t dh = kOffDh + ds * kDhBytes;
                            const int nz = (kTileTokens - pend.nvalid) * 32;  // 16-B chunks in 4 blocks
                            for (int i = h; i < nz; i += 128) {
                                const int row = pend.nvalid + i / 32, ch = i % 32;
                                *reinterpret_cast<uint4 *>(gbase + dh + (ch / 8) * kDhBlock + row * 128 + (ch % 8) * 16) =
                                    make_uint4(0u, 0u, 0u, 0u);
                            }
                            wrote = true;
                        }
                        if (__any_sync(0xffffffffu, wrote)) fence_proxy_async_smem();
                        // O rescale: PV of the previous tile must have finished.  Its slot's
                        // barrier completes when both CTAs' PV of that tile are done and cannot
                        // complete again before this tile's PV, so its parity is unambiguous.
                        if (__any_sync(0xffffffffu, resc_o)) {
                            const uint32_t gq = gp - 1u;
                            if (!warp_wait(c, bar(base, B_PFREE + (int)(gq % kPSlots)), (gq / kPSlots) & 1u, true)) {
                                ok = false;
                                break;
                            }
                            tc_fence_after();
                            const float al = resc_o ? alpha : 1.f;
                            for (int cb = 0; cb < 256; cb += 32) {
                                uint32_t o[32];
                                tmem_ld32(trow + kColO + cb, o);
                                tmem_wait_ld();
#pragma unroll
                                for (int q = 0; q < 32; ++q) o[q] = __float_as_uint(__uint_as_float(o[q]) * al);
                                tmem_st32(trow + kColO + cb, o);
                            }
                            tmem_wait_st();
                        }
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(bar(base, B_P_FULL + slot));
                    }
                }
                if (!ok) break;
                // ---- epilogue: wait for the last PV of this item, normalise, store
                if (!warp_wait(c, bar(base, B_O_FINAL), nitem & 1u, false)) {
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
                ++nitem;
                tc_fence_before();
            }
        }
    }

    // ---------------------------------------------------------------- teardown
    if (warp < 4 && lane == 0) bulk_wait_read_all();
    tc_fence_before();
    __syncthreads();
    cluster_sync();  // the peer may still be copying into this CTA's shared memory
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
                             (int)kSmemBytes) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
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
    const cuuint32_t box[2] = {64, 32};
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
