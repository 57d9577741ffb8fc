// Tensor-core decode kernel for sm_103a (bf16 paged cache).
//
// One work unit = a cluster of two CTAs on two SMs.  Both CTAs walk the same work items
// (request b, token range) tile by tile; a tile is two 64-token pages.  CTA r owns
//   * the scores of page r of the tile — full 576-wide dot products for its 64 tokens, so
//     no partial score ever crosses between the SMs, and
//   * the output latent columns [256 r, 256 r + 256) of every head (its O half, 128 x 256
//     fp32 in TMEM; the full 128 x 512 accumulator does not fit one SM's TMEM).
// Per tile:
//   TMA (128-B swizzle, 64-row boxes)  own-half latent of both pages (PV operand; the own
//        page's copy is also the QK operand for those columns) and the other 320 columns
//        (other latent half + RoPE) of the own page (QK operand only, released once QK^T
//        has read it).  Page ids are read one tile ahead, off the loaders' critical path,
//        and each stage costs the loader one wait and one expect-tx.
//   QK^T  S[h, i] = q[h, :] . entry[own page row i, :]   tcgen05.mma M=128 heads, N=64,
//         K=576: 384 K from the query slice held in TMEM, 192 K from shared memory.
//   softmax (one thread per head): x = s * scale * log2(e); reference r = the running
//         maximum m, or the page's own maximum if that exceeds m by more than 8; own
//         weights p = 2^(x - r) in bf16 go to a shared-memory tile, followed by r and the
//         fp32 sum of p; each warp bulk-copies its 32 rows of that (4.25 KB) into the
//         peer's copy of the tile, completing on the peer's mbarrier (17 KB per tile).
//   merge: with both CTAs' (r, sum) both compute the same new maximum m', rescale a page
//         whose reference was below m' (2^(r - m')), the sum l and — when m' > m — O, so
//         both hold bitwise identical weights for all 128 tokens.
//   PV    O_r[h, :] += P[h, 0:128] . C[0:128, own latent half]   M=128, N=256, K=128,
//         A = the probability tile, B = the own-half cache tiles (MN-major); the peer's
//         page first, so that its buffer is handed back to the loader early.
//   epilogue: out = O / l, lse = (m + log2 l) ln 2, or a partial result for the merge.
//
// TMEM columns: O [0,256)  S [256,320)  query [320,512) (own latent half, RoPE, first 64
// columns of the other half; the other half's last 192 columns sit in shared memory).
// Warp roles: warps 0-3 softmax/epilogue (thread = head, warp w reads TMEM lanes
// 32w..32w+31), warp 4 loads the latent-half ring, warp 7 the other-columns ring (two
// warps, so that neither loader's waits hold up the other), warp 5 issues QK^T (and owns
// TMEM), warp 6 issues PV.
// Every wait is bounded: on timeout the kernel records MLA_ERR_TIMEOUT, stops issuing,
// and all roles fall through to a clean exit.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_fp16.h>

#include "common.cuh"
#include "launch.h"
#include "sm103_ptx.cuh"

namespace mla {
namespace {

using namespace ptx;

constexpr int kTile = 2 * kPageRows;             // tokens per tile
constexpr int kDhSlots = 3;                      // own-half latent of one page (until PV); see dh_slot
constexpr int kOthBoxes = 5;                     // other latent half (4 boxes) + RoPE, one stage
constexpr uint32_t kBox = 64 * 128;              // 64 rows x 64 bf16, 128-B swizzle
constexpr uint32_t kDhBytes = 4 * kBox;          // one page, 256 latent columns
constexpr uint32_t kQsBox = 128 * 128;           // 128 heads x 64 bf16
constexpr uint32_t kQsBytes = 3 * kQsBox;
constexpr uint32_t kPPage = 128 * 128;           // 128 heads x 64 tokens bf16, 128-B swizzle
constexpr uint32_t kRlBytes = 1024;              // r[128] and sum[128], fp32
constexpr uint32_t kPBytes = 2 * kPPage + 2 * kRlBytes;
constexpr uint32_t kMsgBytes = kPPage + kRlBytes;
constexpr int kThreads = 256;         // dense tiles
constexpr int kThreadsSparse = 384;   // sparse tiles: loader warps in pairs (see the loaders)
constexpr int kThreadsFp8 = 384;      // FP8 records: + raw-load and expansion warps
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColO = 0, kColS = 256, kColQ = 320;
constexpr uint32_t kColQRope = kColQ + 128, kColQOther = kColQ + 160;
constexpr float kRescaleLog2 = 8.0f;
// Sparse tiles: how many boxes of each stage (own page's latent half: 4, peer page's: 4, other
// columns: 5) copy their non-contiguous rows through the load/store path; the TMA gathers the
// rest.
constexpr int kSparseLsuOwn = 4, kSparseLsuPeer = 4, kSparseLsuOth = 5;

constexpr uint32_t kOffDh = 0;
constexpr uint32_t kOffOth = kOffDh + kDhSlots * kDhBytes;
constexpr uint32_t kOffQs = kOffOth + kOthBoxes * kBox;
constexpr uint32_t kOffP = kOffQs + kQsBytes;
constexpr uint32_t kOffBar = kOffP + kPBytes;
constexpr uint32_t kOffMisc = kOffBar + 8 * 32;
// FP8 records: per-row scales of the three latent-half slots and the other-columns stage
constexpr uint32_t kOffScale = (kOffMisc + 64 + 1023) / 1024 * 1024;
constexpr uint32_t kScaleBytes = 64 * 16;  // 64 rows x 4 fp32
constexpr uint32_t kSmemBytes = kOffScale + 4 * kScaleBytes + 1024;  // + slack for 1024-B alignment
static_assert(kSmemBytes <= 232448, "shared memory");

enum {
    B_DH_FULL = 0,                       // 2 per slot: own-page and peer-page loads
    B_DH_EMPTY = B_DH_FULL + 2 * kDhSlots,
    B_OTH_FULL = B_DH_EMPTY + kDhSlots,
    B_OTH_EMPTY,
    B_S_FULL,
    B_S_FREE,
    B_O_FINAL,  // the last PV of a work item (waited by the epilogue)
    B_Q_READY,
    B_RFULL,    // the peer's message for the current tile has landed
    B_PFREE,    // both CTAs' PV have finished reading the probability tile
    B_P_FULL,   // the probability tile holds the merged weights of its tile
    B_QLD,      // a round of query boxes has landed in the query area
    B_RAW,      // FP8: raw codes + scales of latent slot s (s < 3) or of the other-columns stage (3)
    B_STALL = B_RAW + 4,  // never completed: the injected stall of the timeout test waits on it
    B_QCP,      // dense / sparse: the query boxes copied into TMEM (tcgen05.cp) have been read
    B_QDONE,    // dense / sparse: every QK^T of the previous work item has completed
    B_COUNT
};
static_assert(B_COUNT <= 32, "barrier area");

struct Ctx {
    uint32_t base;
    int *status;
    volatile uint32_t *abort;
    long long wait_cycles;  // limit of one wait (DecodeArgs::wait_cycles)
};

__device__ __forceinline__ uint32_t bar(uint32_t base, int i) { return base + kOffBar + 8u * i; }

// Bounded wait by the calling thread.  False on timeout (recorded) or when another role
// has already given up.  The first test is inline; the polling loop is out of line, which
// keeps every role's code small in the instruction cache.
__device__ __noinline__ bool wait_bar_slow(const Ctx c, uint32_t b, uint32_t parity, bool cluster_scope) {
    const long long t0 = (long long)clock64_now();
    for (uint32_t i = 0;; ++i) {
        const bool ok = cluster_scope ? mbar_try_wait_cluster(b, parity) : mbar_try_wait(b, parity);
        if (ok) return true;
        if ((i & 63u) == 63u) {
            if (*c.abort) return false;
            if ((long long)clock64_now() - t0 > c.wait_cycles) {
                *c.abort = 1u;
                record_error(c.status, MLA_ERR_TIMEOUT);
                return false;
            }
        }
    }
}

__device__ __forceinline__ bool wait_bar(const Ctx &c, uint32_t b, uint32_t parity, bool cluster_scope) {
    const bool ok = cluster_scope ? mbar_try_wait_cluster(b, parity) : mbar_try_wait(b, parity);
    return ok || wait_bar_slow(c, b, parity, cluster_scope);
}

// All lanes of a warp wait; the outcome is made warp-uniform.
__device__ __forceinline__ bool warp_wait(const Ctx &c, uint32_t b, uint32_t parity,
                                          bool cluster_scope) {
    const bool ok = wait_bar(c, b, parity, cluster_scope);
    return __all_sync(0xffffffffu, ok);
}

// Gives TMA loads or MMAs already in flight a bounded time to finish before an aborting
// role leaves (shared memory and TMEM must outlive them).
__device__ __forceinline__ void drain_pause() {
    const long long t0 = (long long)clock64_now();
    while ((long long)clock64_now() - t0 < 20000000LL) {
    }
}

__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}
__device__ __forceinline__ uint32_t pack_f16(float lo, float hi) {
    __half2 v = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}
__device__ __forceinline__ float2 unpack_f16(uint32_t w) {
    return __half22float2(*reinterpret_cast<const __half2 *>(&w));
}
// The 16-bit operand type of the MMAs: bf16 for a bf16 cache (its values are the operands
// as stored), fp16 for FP8 records (code x scale keeps 3 more significand bits in fp16).
template <bool kF16>
__device__ __forceinline__ uint32_t pack_op(float lo, float hi) {
    if constexpr (kF16)
        return pack_f16(lo, hi);
    else
        return pack_bf16(lo, hi);
}
template <bool kF16>
__device__ __forceinline__ uint32_t scale_pair(uint32_t w, float f) {
    if constexpr (kF16) {
        const float2 v = unpack_f16(w);
        return pack_f16(v.x * f, v.y * f);
    } else {
        return pack_bf16(bf16lo(w) * f, bf16hi(w) * f);
    }
}
// Multiplies one 128-B row of 16-bit weights by f (the chunk order inside the row does not
// matter).
template <bool kF16>
__device__ __forceinline__ void scale_row(uint4 *prow, float f) {
    for (int q = 0; q < 8; ++q) {
        uint4 v = prow[q];
        v.x = scale_pair<kF16>(v.x, f);
        v.y = scale_pair<kF16>(v.y, f);
        v.z = scale_pair<kF16>(v.z, f);
        v.w = scale_pair<kF16>(v.w, f);
        prow[q] = v;
    }
}
// A bf16 pair as an fp16 pair (exact for |x| in the fp16 normal range); *amax collects
// the larger magnitude so that the caller can report values beyond the fp16 range.
__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t w, float *amax) {
    const float lo = bf16lo(w), hi = bf16hi(w);
    *amax = fmaxf(*amax, fmaxf(fabsf(lo), fabsf(hi)));
    return pack_f16(lo, hi);
}
// Largest magnitude an fp16 operand holds (beyond it the conversion gives infinity).
constexpr float kF16Max = 65504.0f;

// Page p (0 or 1) of the tile starting at token t of item w: its valid rows (0 when the page
// lies past the item's end) and its physical id (-1 when that id is out of range).
struct PageRef {
    int rows;
    int64_t id;
};
// The block-table entry is read with a volatile load: it is issued where page_of is called
// (callers call it ahead of a barrier wait) and not sunk to the first use of the id.
__device__ __forceinline__ int32_t ld_early(const int32_t *p) {
    int32_t v;
    asm volatile("ld.global.nc.b32 %0, [%1];" : "=r"(v) : "l"(p));
    return v;
}
__device__ __forceinline__ PageRef page_of(const DecodeArgs &a, const WorkItem &w, int t, int p) {
    const int t_p = t + kPageRows * p;
    PageRef r{0, -1};
    if (t_p >= w.t1) return r;
    r.rows = min(kPageRows, w.t1 - t_p);
    const int lp = t_p / kPageRows;
    const int64_t id = lp < a.max_pages ? (int64_t)ld_early(a.block_table + (int64_t)w.b * a.max_pages + lp) : -1;
    r.id = (id >= 0 && id < a.num_pages) ? id : -1;
    return r;
}

// Sparse tiles: row j of page p holds index slot t + 64 p + j of the item.  Lane l
// resolves slots l and l + 32: the cache row (page * 64 + row; row 0 for an invalid slot,
// which is never attended and is zeroed before PV) and whether the slot is attended
// (inside the item, index in [0, seq_len), page id in range).  Warp-collective.
struct SparseRows {
    int32_t row0, row1;
    uint32_t lo, hi;  // validity of slots 0-31 and 32-63
};
__device__ SparseRows sparse_rows(const DecodeArgs &a, const WorkItem &w, int t, int p, int lane, bool report) {
    // volatile loads: issued here (ahead of the caller's barrier wait), both slots' indices
    // and the length together, then the block-table entries
    int idxs[2] = {-1, -1};
#pragma unroll
    for (int k = 0; k < 2; ++k) {
        const int s = t + kPageRows * p + lane + 32 * k;
        if (s < w.t1) idxs[k] = ld_early(a.indices + (int64_t)w.b * a.topk + s);
    }
    const int L = max(0, ld_early(a.seq_lens + w.b));
    int32_t rows[2] = {0, 0};
    bool ok[2] = {false, false};
    for (int k = 0; k < 2; ++k) {
        const int s = t + kPageRows * p + lane + 32 * k;
        if (s >= w.t1) continue;
        const int idx = idxs[k];
        if (idx < 0) {
            if (idx < -1 && report) record_error(a.status, MLA_ERR_INDEX);
            continue;
        }
        const int lp = idx / kPageRows;
        const int64_t id = idx < L && lp < a.max_pages ? (int64_t)ld_early(a.block_table + (int64_t)w.b * a.max_pages + lp) : -1;
        if (id < 0 || id >= a.num_pages) {
            if (report) record_error(a.status, MLA_ERR_INDEX);
            continue;
        }
        rows[k] = (int32_t)(id * kPageRows + idx % kPageRows);
        ok[k] = true;
    }
    return SparseRows{rows[0], rows[1], __ballot_sync(0xffffffffu, ok[0]), __ballot_sync(0xffffffffu, ok[1])};
}

// Sparse tiles move a page's 64 rows in one of three ways.  When they are one whole cache
// page in order (a run of consecutive positions, as the local window of a top-k list gives),
// 64-row boxes of the page tensor map fetch them (~20 cycles of the SM's TMA unit per 8 KB).
// Otherwise either the TMA gathers them four rows at a time (tile::gather4: ~70 cycles of the
// TMA unit per 512 B, the limit of a TMA-only sparse tile) or the loading warp copies them in
// 16-B pieces through the load/store path (cp.async), which runs beside the TMA unit.
__device__ __forceinline__ bool rows_whole(const SparseRows &r, int lane) {
    const int32_t r00 = __shfl_sync(0xffffffffu, r.row0, 0);
    return r.lo == 0xffffffffu && r.hi == 0xffffffffu && (r00 & (kPageRows - 1)) == 0 &&
           __all_sync(0xffffffffu, r.row0 == r00 + lane && r.row1 == r00 + 32 + lane);
}
// Whole page: box i (columns x_of(i) .. + 63) by lane i.
template <typename XOf>
__device__ __forceinline__ void page_boxes(const SparseRows &r, int lane, uint32_t dst, const void *tmap_page, int nbox,
                                           XOf x_of, uint32_t bar) {
    const int32_t r00 = __shfl_sync(0xffffffffu, r.row0, 0);
    if (lane < nbox) tma_load_2d(dst + lane * kBox, tmap_page, x_of(lane), r00, bar);
}
// TMA gathers of boxes i0 .. nbox - 1: lanes 0-15 take groups of four rows, the two
// half-warps alternate boxes.
template <typename XOf>
__device__ __forceinline__ void gather_rows(const SparseRows &r, int lane, uint32_t dst, const void *tmap, int i0,
                                            int nbox, XOf x_of, uint32_t bar) {
    const int l = lane & 15;
    int32_t r4[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const int j = 4 * l + k;
        const int32_t a0 = __shfl_sync(0xffffffffu, r.row0, j & 31), a1 = __shfl_sync(0xffffffffu, r.row1, j & 31);
        r4[k] = j < 32 ? a0 : a1;
    }
    for (int i = i0 + (lane >> 4); i < nbox; i += 2)
        tma_gather4(dst + i * kBox + 512u * l, tmap, x_of(i), r4[0], r4[1], r4[2], r4[3], bar);
}
// Load/store path, rows 32 half .. 32 half + 31: lane l copies the 16-B piece l % 8 of row
// 4 k + l / 8 of every box, into its 128-B-swizzled place.  The caller waits for the copies
// (cp_async_wait_all) and fences them for the tensor cores before it signals the stage.
template <typename XOf>
__device__ __forceinline__ void copy_rows_lsu(const SparseRows &r, int lane, uint32_t dst,
                                              const unsigned char *cache, int nbox, XOf x_of, int half) {
    const int ch = lane & 7;
#pragma unroll 1
    for (int k = 8 * half; k < 8 * half + 8; ++k) {
        const int row = 4 * k + (lane >> 3);
        const int32_t R = __shfl_sync(0xffffffffu, k < 8 ? r.row0 : r.row1, row & 31);
        const unsigned char *src = cache + (int64_t)R * (kDEntry * 2) + ch * 16;
        const uint32_t d = dst + row * 128 + ((ch ^ (row & 7)) << 4);
#pragma unroll
        for (int i = 0; i < nbox; ++i) cp_async16(d + i * kBox, src + x_of(i) * 2);
    }
}
// Fills one stage of sparse rows (nbox boxes at dst), shared by a pair of warps (half 0 and
// 1), each of which arrives once on the stage's barrier `bar` (count 2).  A whole page comes
// in 64-row boxes, issued by half 0 with the bytes expected; otherwise boxes 0 .. nlsu - 1 are
// copied through the load/store path (each warp its 32 rows; the arrival follows once they
// have landed) and the rest gathered by the TMA (half 0), both at once.  Warp-collective.
template <typename XOf>
__device__ __forceinline__ void sparse_stage(const SparseRows &r, int lane, uint32_t dst, const void *tmap,
                                             const void *tmap_page, const unsigned char *cache, int nbox, XOf x_of,
                                             uint32_t bar, int nlsu, int half) {
    const bool whole = rows_whole(r, lane);
    if (whole || nlsu == 0) {
        if (half != 0) {
            if (lane == 0) mbar_arrive(bar);
            return;
        }
        if (lane == 0) mbar_arrive_expect_tx(bar, (uint32_t)nbox * kBox);
        __syncwarp();
        if (whole)
            page_boxes(r, lane, dst, tmap_page, nbox, x_of, bar);
        else
            gather_rows(r, lane, dst, tmap, 0, nbox, x_of, bar);
        return;
    }
    if (nlsu < nbox && half == 0) {
        if (lane == 0) mbar_expect_tx(bar, (uint32_t)(nbox - nlsu) * kBox);
        __syncwarp();
        gather_rows(r, lane, dst, tmap, nlsu, nbox, x_of, bar);
    }
    copy_rows_lsu(r, lane, dst, cache, nlsu, x_of, half);
    cp_async_wait_all();
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) mbar_arrive(bar);
}

// Which of page p's 64 rows attend (`valid`) and how many rows of the page lie inside the
// item (`cnt`; PV reads them in whole 16-row steps).  Warp-collective for sparse tiles.
struct PageMask {
    uint64_t valid;
    int cnt;
};
template <bool kSparse>
__device__ __forceinline__ PageMask page_mask(const DecodeArgs &a, const WorkItem &w, int t, int p, int lane) {
    PageMask m;
    m.cnt = max(0, min(kPageRows, w.t1 - (t + kPageRows * p)));
    if constexpr (kSparse) {
        const SparseRows r = sparse_rows(a, w, t, p, lane, false);
        m.valid = (uint64_t)r.lo | ((uint64_t)r.hi << 32);
    } else {
        const PageRef pg = page_of(a, w, t, p);
        m.valid = pg.id >= 0 && pg.rows > 0 ? (pg.rows >= 64 ? ~0ull : ((1ull << pg.rows) - 1ull)) : 0ull;
    }
    return m;
}

// Latent-half slots.  Tile g's own page (e = 0) sits in slot g % 3 and its peer page (e = 1)
// in slot (g + 2) % 3; the loader issues own(0), own(1), then peer(g), own(g + 2) for
// g = 0, 1, ...  PV of tile g hands back the peer page's slot first, and own(g + 2) — the
// page the scores need soonest — takes exactly that slot, ahead of peer(g + 1), which takes
// own(g)'s.  (Reading the own page first and loading peer(g + 1) first was measured 10 %
// slower per tile.)  Each slot alternates own and peer pages.  `fill` counts the slot's loads before
// this one (the phase of its empty barrier).  Own-page and peer-page loads complete on
// separate full barriers (`full`, phase `phase` = g / 3): the score issuer waits for own
// pages only, and with one barrier per slot a parity wait for the next own page could be
// satisfied by an older phase while the peer page between them is still loading.
// Sparse tiles load own and peer pages from two warps; there each slot has one of them as its
// only user (own pages alternate slots 0 and 1, peer pages use slot 2), so that each warp's
// parity waits on a slot follow its phases one by one.
struct DhSlot {
    int slot;
    uint32_t fill;
    int full;        // barrier index
    uint32_t phase;
};
template <bool kSplitSlots>
__device__ __forceinline__ DhSlot dh_slot(uint32_t g, int e) {
    if constexpr (kSplitSlots) {
        if (e == 0) return DhSlot{(int)(g & 1u), g >> 1, B_DH_FULL + 2 * (int)(g & 1u), g >> 1};
        return DhSlot{2, g, B_DH_FULL + 2 * 2 + 1, g};
    }
    const uint32_t q = g / 3u, r = g % 3u;
    const int slot = e == 0 ? (int)r : (int)((r + 2u) % 3u);
    const uint32_t fill = e == 0 ? 2u * q + (r == 2u ? 1u : 0u) : 2u * q + (r != 0u ? 1u : 0u);
    return DhSlot{slot, fill, B_DH_FULL + 2 * slot + e, q};
}

// Rare steps of the softmax warps, kept out of line: the per-tile loop then stays small
// enough for the instruction cache, which the loaders and MMA issuers share.
// O row of this thread (256 fp32 columns at taddr, warp-collective) times al.
__device__ __noinline__ void rescale_o_row(uint32_t taddr, float al) {
#pragma unroll 1
    for (int cb = 0; cb < 256; cb += 32) {
        uint32_t o[32];
        tmem_ld32(taddr + cb, o);
        tmem_wait_ld();
#pragma unroll
        for (int q = 0; q < 32; ++q) o[q] = __float_as_uint(__uint_as_float(o[q]) * al);
        tmem_st32(taddr + cb, o);
    }
    tmem_wait_st();
}
template <bool kF16>
__device__ __noinline__ void scale_row_ool(uint4 *prow, float f) {
    scale_row<kF16>(prow, f);
}
// Zeroes the rows of `zero` in a 64-row latent-half page (4 boxes); the 128 threads of the
// softmax warps share its 16-B chunks (thread h takes chunks h, h + 128, ...).
__device__ __noinline__ void zero_rows(uint8_t *dh, uint64_t zero, int h) {
    const int z1 = 64 - __clzll((long long)zero);  // rows below the last one to zero
    for (int i = h; i < z1 * 32; i += 128) {
        const int row = i / 32, ch = i % 32;
        if ((zero >> row) & 1ull)
            *reinterpret_cast<uint4 *>(dh + (ch / 8) * kBox + row * 128 + (ch % 8) * 16) = make_uint4(0u, 0u, 0u, 0u);
    }
}

// Epilogue of a work item (out of line): this thread's O row (TMEM columns at tcol) times inv,
// staged through its own 128-B row of stg so that each warp store covers whole lines; warp w
// writes back rows 32w .. 32w + 31 of the item's output (row 0 at obase).
__device__ __noinline__ void store_rows(uint32_t tcol, uint8_t *stg, float *obase, float inv, int h, int warp,
                                        int lane, int H) {
#pragma unroll 1
    for (int cb = 0; cb < 256; cb += 32) {
        uint32_t o[32];
        tmem_ld32(tcol + cb, o);
        tmem_wait_ld();
#pragma unroll
        for (int q = 0; q < 8; ++q)
            *reinterpret_cast<float4 *>(stg + h * 128 + ((q ^ (h & 7)) * 16)) =
                make_float4(__uint_as_float(o[4 * q]) * inv, __uint_as_float(o[4 * q + 1]) * inv,
                            __uint_as_float(o[4 * q + 2]) * inv, __uint_as_float(o[4 * q + 3]) * inv);
        __syncwarp();
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int row = warp * 32 + 4 * i + (lane >> 3), q = lane & 7;
            const float4 v = *reinterpret_cast<const float4 *>(stg + row * 128 + ((q ^ (row & 7)) * 16));
            if (row < H) *reinterpret_cast<float4 *>(obase + (int64_t)row * kDLatent + cb + 4 * q) = v;
        }
        __syncwarp();
    }
}

// Walks the tiles of this cluster's work in order: units cl, cl + ncl, ..., their items
// (those with tokens), and each item's 128-token tiles.
struct TileCursor {
    const int32_t *ub;
    const WorkItem *items;
    int units, ncl;
    int u, it;   // current unit and item; u >= units once every tile has been visited
    WorkItem w;  // items[it]
    int t;       // first token of the current tile
    __device__ void find() {
        while (u < units) {
            const int end = ub[u + 1];
            for (; it < end; ++it) {
                w = items[it];
                if (w.t1 > w.t0) {
                    t = w.t0;
                    return;
                }
            }
            u += ncl;
            if (u < units) it = ub[u];
        }
    }
    __device__ void begin(const int32_t *unit_begin, const WorkItem *its, int nunits, int cl, int n) {
        ub = unit_begin;
        items = its;
        units = nunits;
        ncl = n;
        u = cl;
        it = u < units ? ub[u] : 0;
        find();
    }
    __device__ bool done() const { return u >= units; }
    __device__ void next() {
        if (done()) return;
        t += kTile;
        if (t < w.t1) return;
        ++it;
        find();
    }
};

// Request of the first item with tokens after item `it` of unit `u`, in this cluster's
// order (units u, u + ncl, ...), or -1.
__device__ int next_request(const int32_t *ub, const WorkItem *items, int units, int ncl, int u, int it) {
    int nit = it + 1;
    while (u < units) {
        for (; nit < ub[u + 1]; ++nit) {
            const WorkItem w = items[nit];
            if (w.t1 > w.t0) return w.b;
        }
        u += ncl;
        if (u < units) nit = ub[u];
    }
    return -1;
}

// Two e4m3 codes (low byte first) times their block scale, as a packed fp16 pair: the code
// is widened exactly (e4m3 -> fp16 -> fp32), the product formed in fp32 and rounded once to
// fp16, the operand type of the FP8 path's MMAs.
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t two, float s) {
    const __half2_raw hr = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(two & 0xFFFFu), __NV_E4M3);
    const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&hr));
    return pack_f16(f.x * s, f.y * s);
}

// Expands 16 e4m3 codes (v) with block scale s into the 16-code chunk q (0..3) of row r of a
// bf16 box: box points at row r of a box of 64 columns stored as 128-B rows in the 128-B
// swizzle (16-B unit u of row r at u ^ (r % 8)); chunk q covers units 2q and 2q + 1.
__device__ __forceinline__ void expand_chunk(uint4 v, float s, uint8_t *box, int q, int r) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t o[8];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        o[2 * k] = e4m3x2_to_f16x2(w[k], s);
        o[2 * k + 1] = e4m3x2_to_f16x2(w[k] >> 16, s);
    }
    *reinterpret_cast<uint4 *>(box + (((2 * q) ^ (r & 7)) * 16)) = make_uint4(o[0], o[1], o[2], o[3]);
    *reinterpret_cast<uint4 *>(box + (((2 * q + 1) ^ (r & 7)) * 16)) = make_uint4(o[4], o[5], o[6], o[7]);
}

// FP8 records: the jobs of the latent-half ring (which 0: own(0), own(1), peer(0), then
// peer(g + 1), own(g + 2) for g = 0, 1, ...), of the other-columns stage (which 1: oth(g),
// one per tile), or all of them in the order they are consumed (which 2: oth(0), own(0),
// own(1), peer(0), then oth(g + 1), peer(g + 1), own(g + 2)).  f(kind, g, cursor): kind 0 own
// page, 1 peer page, 2 other columns.  Every job comes after the jobs whose consumers free its
// buffer: peer(g + 1) and own(g + 2) take the slots PV(g) frees, oth(g + 1) the stage QK(g)
// frees; and peer(g + 1), which PV(g + 1) waits for, goes before own(g + 2), which only
// QK(g + 2) needs.  One call site of f: the job bodies are large.
template <typename F>
__device__ bool fp8_jobs(const TileCursor &start, int which, F &&f) {
    TileCursor cur[3] = {start, start, start};  // next own, peer, other-columns job
    uint32_t gk[3] = {0u, 0u, 0u};
    for (int step = 0;; ++step) {
        int kind;
        if (which == 1) {
            kind = 2;
        } else if (which == 0) {
            kind = step < 3 ? (step < 2 ? 0 : 1) : ((step - 3) & 1) ? 0 : 1;
        } else {
            const int k = (step - 4) % 3;
            kind = step < 4 ? (step == 0 ? 2 : step < 3 ? 0 : 1) : k == 0 ? 2 : k == 1 ? 1 : 0;
        }
        if (cur[kind].done()) {
            const bool dh_done = cur[0].done() && cur[1].done();
            if (which == 0 ? dh_done : which == 1 ? true : dh_done && cur[2].done()) return true;
            continue;
        }
        if (!f(kind, gk[kind], cur[kind])) return false;
        ++gk[kind];
        cur[kind].next();
    }
}

// kMode 0: dense bf16 tiles (128 consecutive tokens, two pages, 64-row boxes).
// kMode 1: DSA sparse tiles (128 index slots gathered row by row, tile::gather4).
// kMode 2: dense FP8 records: raw e4m3 codes and scales are loaded by two extra warps (one
//          for the latent-half ring, one for the other-columns stage) and expanded to bf16
//          operand tiles by four warps; RoPE goes in directly.
// tmap: the cache (kMode 2: its bytes, 128-B boxes of codes; kMode 1: one-row boxes);
// tmap_sc: FP8 scales (16-B boxes) or, for kMode 1, the cache in 64-row boxes; tmap_rope:
// FP8 RoPE (bf16, 128-B swizzle); tmap_qn / tmap_qr:
// the queries (64 columns x 128 heads of one request, 128-B swizzle).
template <int kMode>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kMode == 2 ? kThreadsFp8 : kMode == 1 ? kThreadsSparse : kThreads, 1)
decode_sm103_kernel(const __grid_constant__ CUtensorMap tmap, const __grid_constant__ CUtensorMap tmap_sc,
                    const __grid_constant__ CUtensorMap tmap_rope, const __grid_constant__ CUtensorMap tmap_qn,
                    const __grid_constant__ CUtensorMap tmap_qr, DecodeArgs a) {
    constexpr bool kSparse = kMode == 1, kFp8 = kMode == 2;
    // arrivals that complete a latent / other-columns stage
    constexpr uint32_t kFullCount = kFp8 ? 4u : kSparse ? 2u : 1u;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *gbase = smem_raw + (base - raw);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank(), peer = rank ^ 1u;
    volatile uint32_t *misc = reinterpret_cast<volatile uint32_t *>(gbase + kOffMisc);
    // misc[0]: TMEM base address, misc[1]: abort flag
    Ctx c{base, a.status, misc + 1, a.wait_cycles};

    if (threadIdx.x == 0) {
        for (int s = 0; s < kDhSlots; ++s) {
            mbar_init(bar(base, B_DH_FULL + 2 * s), kFullCount);
            mbar_init(bar(base, B_DH_FULL + 2 * s + 1), kFullCount);
            mbar_init(bar(base, B_DH_EMPTY + s), 1);
        }
        for (int s = 0; s < 4; ++s) mbar_init(bar(base, B_RAW + s), 1);
        mbar_init(bar(base, B_OTH_FULL), kFullCount);
        mbar_init(bar(base, B_OTH_EMPTY), 1);
        mbar_init(bar(base, B_S_FULL), 1);
        mbar_init(bar(base, B_S_FREE), 4);
        mbar_init(bar(base, B_O_FINAL), 1);
        mbar_init(bar(base, B_Q_READY), 4);
        mbar_init(bar(base, B_RFULL), 1);  // + the message bytes
        mbar_init(bar(base, B_PFREE), 2);  // one commit from each CTA's PV
        mbar_init(bar(base, B_P_FULL), 4);
        mbar_init(bar(base, B_QLD), 1);  // + the boxes' bytes
        mbar_init(bar(base, B_STALL), 1);
        mbar_init(bar(base, B_QCP), 1);
        mbar_init(bar(base, B_QDONE), 1);
        misc[1] = 0u;
        fence_mbar_init();
    }
    if (warp == 5) {
        tmem_alloc(smem_u32(const_cast<uint32_t *>(misc)), kTmemCols);
        tmem_relinquish();
    }
    if (warp == 4 && lane == 0) {
        prefetch_tmap(&tmap);
        prefetch_tmap(&tmap_qn);
        prefetch_tmap(&tmap_qr);
        if (kFp8 || kSparse) prefetch_tmap(&tmap_sc);
        if (kFp8) prefetch_tmap(&tmap_rope);
    }
    tc_fence_before();
    cluster_sync();
    tc_fence_after();
    const uint32_t tmem = misc[0];
    // Everything above touches only this CTA's shared memory and TMEM, so it overlaps the
    // kernel before this one on the stream (the plan); the plan is read from here on.
    grid_dep_wait();
    if (!plan_matches(a)) {  // the same outcome in every CTA
        if (threadIdx.x == 0 && blockIdx.x == 0) record_error(a.status, MLA_ERR_WORKSPACE);
        if (warp == 5) tmem_dealloc(tmem, kTmemCols);
        return;
    }

    const PlanHeader *hd = reinterpret_cast<const PlanHeader *>(a.ws);
    const WsLayout L = ws_layout(hd->B, hd->H, hd->num_units);
    const int32_t *unit_begin = reinterpret_cast<const int32_t *>(a.ws + L.unit_begin);
    const WorkItem *items = reinterpret_cast<const WorkItem *>(a.ws + L.items);
    float *part_lse = reinterpret_cast<float *>(const_cast<unsigned char *>(a.ws) + L.part_lse);
    float *part_o = reinterpret_cast<float *>(const_cast<unsigned char *>(a.ws) + L.part_o);
    const int units = hd->num_units;
    const int cl = (int)cluster_id_x(), ncl = (int)nclusters_x();

    if (kFp8 && (warp == 4 || warp == 10 || warp == 7 || warp == 9)) {
        // ------------------------------------------------------------ FP8 expansion (4 warps)
        // Warps 4, 10, 7 and 9 (one per SM sub-partition) expand every job, in the order the
        // jobs are consumed.  Thread (r, p) expands part p (codes 128 p .. 128 p + 127) of row
        // r.  The codes of part p of row r arrive as one 128-B row of box 2p of the bf16
        // destination, the box that receives the first half of that part's output; the second
        // half goes to box 2p + 1 first, then the first half lands on the codes it came from,
        // read into registers beforehand.  No thread writes another thread's codes.
        const int eidx = warp == 4 ? 0 : warp == 10 ? 1 : warp == 7 ? 2 : 3;
        const int r = 32 * (eidx & 1) + lane, p = eidx >> 1;
        TileCursor start;
        start.begin(unit_begin, items, units, cl, ncl);
        const bool ok = fp8_jobs(start, 2, [&](int kind, uint32_t g, const TileCursor &t) -> bool {
            // a page that was not loaded (past the item's end, or an id out of range) is not
            // expanded; its stage only completes
            const PageRef pg = page_of(a, t.w, t.t, kind == 1 ? (int)peer : (int)rank);
            int raw_bar, half;
            uint32_t raw_phase, region, scale_off, full_bar;
            if (kind == 2) {
                raw_bar = B_RAW + 3;
                raw_phase = g;
                region = kOffOth;
                scale_off = kOffScale + 3 * kScaleBytes;
                half = (int)peer;
                full_bar = bar(base, B_OTH_FULL);
            } else {
                const DhSlot d = dh_slot<kSparse>(g, kind);
                raw_bar = B_RAW + d.slot;
                raw_phase = d.fill;
                region = kOffDh + d.slot * kDhBytes;
                scale_off = kOffScale + d.slot * kScaleBytes;
                half = (int)rank;
                full_bar = bar(base, d.full);
            }
            if (!warp_wait(c, bar(base, raw_bar), raw_phase & 1u, false)) return false;
            if (pg.rows > 0 && pg.id >= 0) {
                const float sc = reinterpret_cast<const float *>(gbase + scale_off + r * 16)[2 * half + p];
                // code x scale must stay inside the fp16 range of the operand (|x| <= 65504);
                // rows past the item's end may hold anything and are not checked
                if (r < pg.rows && !(fabsf(sc) * 448.f <= kF16Max)) record_error(a.status, MLA_ERR_RANGE);
                uint8_t *row = gbase + region + r * 128;                 // row r of box 0
                const uint8_t *codes = row + 2 * p * kBox;               // its 8 chunks of 16 codes
                uint8_t *first = row + 2 * p * kBox, *second = first + kBox;
                uint4 v[4];  // chunks (i + r) % 4, read before their box is overwritten
#pragma unroll
                for (int i = 0; i < 4; ++i) v[i] = *reinterpret_cast<const uint4 *>(codes + ((i + r) & 3) * 16);
                // chunks 4 + (i + r) % 4 -> second box (rotated: no bank conflicts on the stores)
                uint4 nxt = *reinterpret_cast<const uint4 *>(codes + (4 + (r & 3)) * 16);
#pragma unroll 1
                for (int i = 0; i < 4; ++i) {
                    const uint4 cur = nxt;
                    if (i < 3) nxt = *reinterpret_cast<const uint4 *>(codes + (4 + ((i + 1 + r) & 3)) * 16);
                    expand_chunk(cur, sc, second, (i + r) & 3, r);
                }
#pragma unroll
                for (int i = 0; i < 4; ++i) expand_chunk(v[i], sc, first, (i + r) & 3, r);
                fence_proxy_async_smem();
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(full_bar);
            return true;
        });
        if (!ok && lane == 0) drain_pause();
    } else if (kFp8 && (warp == 8 || warp == 11)) {
        // ------------------------------------------------------------ FP8 raw loads (one thread each:
        // warp 8 the latent-half ring, warp 11 the other-columns stage)
        if (lane == 0) {
            TileCursor start;
            start.begin(unit_begin, items, units, cl, ncl);
            const bool ok = fp8_jobs(start, warp == 8 ? 0 : 1, [&](int kind, uint32_t g, const TileCursor &t) -> bool {
                if (kind == 2) {
                    const PageRef pg = page_of(a, t.w, t.t, (int)rank);  // read before the wait
                    if (!wait_bar(c, bar(base, B_OTH_EMPTY), (g & 1u) ^ 1u, false)) return false;
                    const uint32_t rb = bar(base, B_RAW + 3), dst = base + kOffOth;
                    if (pg.rows > 0 && pg.id >= 0) {
                        const int32_t y = (int32_t)(pg.id * kPageRows);
                        mbar_arrive_expect_tx(rb, 16384 + kScaleBytes + kBox);
                        tma_load_2d(dst, &tmap, 256 * (int)peer, y, rb);  // other latent half, codes
                        tma_load_2d(dst + 2 * kBox, &tmap, 256 * (int)peer + 128, y, rb);
                        tma_load_2d(base + kOffScale + 3 * kScaleBytes, &tmap_sc, kDLatent, y, rb);
                        tma_load_2d(dst + 4 * kBox, &tmap_rope, (kDLatent + 16) / 2, y, rb);  // RoPE, bf16
                    } else {
                        mbar_arrive(rb);
                    }
                    return true;
                }
                const PageRef pg = page_of(a, t.w, t.t, kind == 0 ? (int)rank : (int)peer);
                const DhSlot d = dh_slot<kSparse>(g, kind);
                if (d.fill > 0 && !wait_bar(c, bar(base, B_DH_EMPTY + d.slot), (d.fill - 1u) & 1u, false))
                    return false;
                const uint32_t rb = bar(base, B_RAW + d.slot), dst = base + kOffDh + d.slot * kDhBytes;
                if (pg.rows > 0 && pg.id >= 0) {
                    const int32_t y = (int32_t)(pg.id * kPageRows);
                    mbar_arrive_expect_tx(rb, 16384 + kScaleBytes);
                    tma_load_2d(dst, &tmap, 256 * (int)rank, y, rb);  // own latent half, codes
                    tma_load_2d(dst + 2 * kBox, &tmap, 256 * (int)rank + 128, y, rb);
                    tma_load_2d(base + kOffScale + d.slot * kScaleBytes, &tmap_sc, kDLatent, y, rb);
                } else {
                    if (pg.rows > 0) record_error(a.status, MLA_ERR_INDEX);
                    mbar_arrive(rb);
                }
                return true;
            });
            if (!ok) drain_pause();
        }
    } else if (warp == 4 || warp == 7 || (kSparse && warp >= 8)) {
        // ------------------------------------------------------------ loaders (whole warps)
        TileCursor cur, nx;
        cur.begin(unit_begin, items, units, cl, ncl);
        nx = cur;
        nx.next();
        // Sparse tiles: a load/store-path copy holds its warp until it has landed, so each
        // kind of stage has its own pair of warps, which split the rows: own pages 4 and 9,
        // peer pages 8 and 10, other columns 7 and 11 (half 0 and 1).
        const int half = (warp == 9 || warp == 10 || warp == 11) ? 1 : 0;
        if (warp == 4 || (kSparse && warp >= 8 && warp <= 10)) {
            // own latent half of both pages, in the order own(0), own(1), peer(0), own(2),
            // peer(1), own(3), ...
            const int xown = 256 * (int)rank;
            // loads page (rank if e == 0, else peer) of tile g at cursor position t
            // (sparse: the rows r were resolved one load ahead)
            auto load = [&](const TileCursor &t, uint32_t g, int e, const SparseRows &r) -> bool {
                const int p = e == 0 ? (int)rank : (int)peer;
                const DhSlot d = dh_slot<kSparse>(g, e);
                const uint32_t fb = bar(base, d.full), dst = base + kOffDh + d.slot * kDhBytes;
                if constexpr (kSparse) {
                    if (d.fill > 0 && !warp_wait(c, bar(base, B_DH_EMPTY + d.slot), (d.fill - 1u) & 1u, false))
                        return false;
                    if (t.t + kPageRows * p < t.w.t1) {
                        sparse_stage(r, lane, dst, &tmap, &tmap_sc, a.cache, 4, [&](int i) { return xown + 64 * i; }, fb,
                                     e == 0 ? kSparseLsuOwn : kSparseLsuPeer, half);
                    } else if (lane == 0) {
                        mbar_arrive(fb);
                    }
                } else {
                    const PageRef pg = page_of(a, t.w, t.t, p);  // read before the wait
                    if (d.fill > 0 && !warp_wait(c, bar(base, B_DH_EMPTY + d.slot), (d.fill - 1u) & 1u, false))
                        return false;
                    if (lane == 0) {
                        if (pg.rows > 0 && pg.id >= 0) {
                            const int32_t y = (int32_t)(pg.id * kPageRows);
                            mbar_arrive_expect_tx(fb, kDhBytes);
                            for (int i = 0; i < 4; ++i) tma_load_2d(dst + i * kBox, &tmap, xown + 64 * i, y, fb);
                        } else {
                            if (pg.rows > 0) record_error(a.status, MLA_ERR_INDEX);
                            mbar_arrive(fb);
                        }
                    }
                }
                return true;
            };
            // the sequence of loads: own(0), own(1), then peer(g), own(g + 2) for g = 0, 1, ...
            TileCursor co = cur;  // next own page: tile go; cur: next peer page, tile gp
            uint32_t go = 0, gp = 0;
            if (kSparse) {
                if (warp == 4 || warp == 9)
                    cur.u = cur.units;  // own pages only
                else
                    co.u = co.units;  // peer pages only
            }
            int step = 0;
            struct Ld {
                int e;  // -1: none left
                uint32_t g;
                TileCursor t;
            };
            auto next_ld = [&]() {
                Ld x{-1, 0u, co};
                for (;; ++step) {
                    const int e = step < 2 ? 0 : ((step - 2) & 1) ? 0 : 1;
                    if (e == 0 && !co.done()) {
                        x = Ld{0, go++, co};
                        co.next();
                        ++step;
                        return x;
                    }
                    if (e == 1 && !cur.done()) {
                        x = Ld{1, gp++, cur};
                        cur.next();
                        ++step;
                        return x;
                    }
                    if (co.done() && cur.done()) return x;
                }
            };
            auto rows_of = [&](const Ld &x) {
                SparseRows r{0, 0, 0u, 0u};
                if constexpr (kSparse) {
                    if (x.e >= 0) r = sparse_rows(a, x.t.w, x.t.t, x.e == 0 ? (int)rank : (int)peer, lane, half == 0);
                }
                return r;
            };
            bool ok = true;
            Ld x = next_ld();
            SparseRows rx = rows_of(x);
            while (ok && x.e >= 0) {
                const Ld xn = next_ld();
                const SparseRows rn = rows_of(xn);  // issued before this load's wait
                ok = load(x.t, x.g, x.e, rx);
                x = xn;
                rx = rn;
            }
            if (!ok && lane == 0) drain_pause();
        } else {
            // other latent half + RoPE of the own page, one stage
            const int xoth = 256 * (int)peer;
            auto x_of = [&](int i) { return i < 4 ? xoth + 64 * i : kDLatent; };
            bool ok = true;
            // sparse: the rows of the next tile are resolved before this tile's wait
            SparseRows rnext{0, 0, 0u, 0u};
            if constexpr (kSparse) {
                if (!cur.done()) rnext = sparse_rows(a, cur.w, cur.t, (int)rank, lane, false);
            }
            for (uint32_t g = 0; !cur.done() && ok; ++g) {
                const uint32_t fb = bar(base, B_OTH_FULL), dst = base + kOffOth;
                if constexpr (kSparse) {
                    const SparseRows r = rnext;
                    if (!nx.done()) rnext = sparse_rows(a, nx.w, nx.t, (int)rank, lane, false);
                    if (!warp_wait(c, bar(base, B_OTH_EMPTY), (g & 1u) ^ 1u, false)) {
                        ok = false;
                        break;
                    }
                    if (cur.t + kPageRows * (int)rank < cur.w.t1) {
                        sparse_stage(r, lane, dst, &tmap, &tmap_sc, a.cache, kOthBoxes, x_of, fb, kSparseLsuOth, half);
                    } else if (lane == 0) {
                        mbar_arrive(fb);
                    }
                } else {
                    const PageRef pg = page_of(a, cur.w, cur.t, (int)rank);  // before the wait
                    if (!warp_wait(c, bar(base, B_OTH_EMPTY), (g & 1u) ^ 1u, false)) {
                        ok = false;
                        break;
                    }
                    if (lane == 0) {
                        if (pg.rows > 0 && pg.id >= 0) {
                            const int32_t y = (int32_t)(pg.id * kPageRows);
                            mbar_arrive_expect_tx(fb, kOthBoxes * kBox);
                            for (int i = 0; i < kOthBoxes; ++i) tma_load_2d(dst + i * kBox, &tmap, x_of(i), y, fb);
                        } else {
                            mbar_arrive(fb);
                        }
                    }
                }
                cur = nx;
                nx.next();
            }
            if (!ok && lane == 0) drain_pause();
        }
    } else if (warp == 5) {
        // ------------------------------------------------------------ QK^T issuer
        // The whole warp runs the loop (warp-uniform waits); one elected lane issues each
        // tcgen05 operation, and lane 0 the TMA loads.
        {
            // FP8 records: the latent columns in fp16, the RoPE columns (bf16 in the record and
            // in the query) in bf16; every MMA accumulates into the same fp32 scores
            constexpr uint32_t idesc_qk_rope = idesc_bf16(128, 64, false);
            constexpr uint32_t idesc_qk = kFp8 ? idesc_f16(128, 64, false) : idesc_qk_rope;
            uint32_t g = 0, nitem = 0;
            bool ok = true;
            // injected stall (test of the timeout path): a wait on a barrier nothing completes,
            // before any MMA is issued; it runs out after the wait limit and the CTA winds down
            if (a.stall_test && !warp_wait(c, bar(base, B_STALL), 0u, false)) ok = false;
            // Dense and sparse tiles: this thread loads each work item's query itself.  The TMA
            // brings three rounds of three 64-column x 128-head boxes (128-B swizzle; heads at or
            // past H read zeros) into the shared-memory query area; rounds 0 and 1 (own latent
            // half, RoPE, the other half's first 64 columns) go on into TMEM by tcgen05.cp, which
            // reads the swizzled boxes like an MMA operand and is ordered before the MMAs issued
            // after it; round 2 (the other half's last 192 columns) stays in shared memory as
            // an operand.  The next round reuses the area once the copies have read it
            // (tcgen05.commit).  The area and the TMEM columns are refilled only after the
            // previous item's last QK^T has completed (B_QDONE), and the softmax warps never
            // wait for any of it.  FP8 records convert the query to fp16 on the way in, which
            // the softmax warps do (B_Q_READY).
            uint32_t qld_phase = 0, qcp_phase = 0;
            auto load_query = [&](int bq) -> bool {
                const uint32_t qb = bar(base, B_QLD);
                for (int round = 0; round < 3; ++round) {
                    if (lane == 0) {
                        mbar_arrive_expect_tx(qb, 3 * kQsBox);
                        for (int i = 0; i < 3; ++i) {
                            const int blk = 3 * round + i;  // 0-3 own half, 4 RoPE, 5-8 other half
                            const uint32_t dst = base + kOffQs + i * kQsBox;
                            if (blk == 4)
                                tma_load_3d(dst, &tmap_qr, 0, 0, bq, qb);
                            else
                                tma_load_3d(dst, &tmap_qn,
                                            blk < 4 ? 256 * (int)rank + 64 * blk : 256 * (int)peer + 64 * (blk - 5), 0,
                                            bq, qb);
                        }
                    }
                    if (!warp_wait(c, qb, (qld_phase++) & 1u, false)) return false;
                    if (round == 2) break;
                    tc_fence_after();
                    for (int i = 0; i < 3; ++i)
                        for (int k = 0; k < 4; ++k)
                            tmem_cp_128x256b_warp(tmem + kColQ + 32u * (3 * round + i) + 8u * k,
                                                  smem_desc_sw128(base + kOffQs + i * kQsBox + k * 32u, 16u, 1024u));
                    mma_commit_warp(bar(base, B_QCP));
                    if (!warp_wait(c, bar(base, B_QCP), (qcp_phase++) & 1u, false)) return false;
                }
                tc_fence_after();
                return true;
            };
            for (int u = cl; u < units && ok; u += ncl) {
                for (int it = unit_begin[u]; it < unit_begin[u + 1] && ok; ++it) {
                    const WorkItem w = items[it];
                    if (w.t1 <= w.t0) continue;
                    if constexpr (kFp8) {
                        if (!warp_wait(c, bar(base, B_Q_READY), nitem & 1u, false)) {
                            ok = false;
                            break;
                        }
                    } else {
                        // the previous item's QK^T must be done with the query area and columns
                        if (nitem > 0 && !warp_wait(c, bar(base, B_QDONE), (nitem - 1) & 1u, false)) {
                            ok = false;
                            break;
                        }
                        if (!load_query(w.b)) {
                            ok = false;
                            break;
                        }
                        // the next item's query is loaded after this one: bring it into L2 now
                        const int bnext = next_request(unit_begin, items, units, ncl, u, it);
                        if (bnext >= 0 && lane == 0) {
                            prefetch_l2(a.q_nope + (int64_t)bnext * a.H * kDLatent, (uint32_t)(a.H * kDLatent * 2));
                            prefetch_l2(a.q_rope + (int64_t)bnext * a.H * kDRope, (uint32_t)(a.H * kDRope * 2));
                        }
                    }
                    ++nitem;
                    tc_fence_after();
                    for (int t = w.t0; t < w.t1 && ok; t += kTile, ++g) {
                        if (g > 0 && !warp_wait(c, bar(base, B_S_FREE), (g - 1) & 1u, false)) {
                            ok = false;
                            break;
                        }
                        const bool have = t + kPageRows * (int)rank < w.t1;  // own page exists
                        // other latent half and RoPE first: their stage goes back to the loader
                        // while the own-half rows may still wait for the previous tile's PV
                        if (!warp_wait(c, bar(base, B_OTH_FULL), g & 1u, false)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        for (int i = 0; i < kOthBoxes && have; ++i) {
                            const uint32_t ot = base + kOffOth + i * kBox;
                            for (int k = 0; k < 4; ++k) {
                                const uint64_t bd = smem_desc_sw128(ot + k * 32u, 16u, 1024u);
                                if (i == 0)
                                    mma_ts_warp(tmem + kColS, tmem + kColQOther + 8u * k, bd, idesc_qk, k > 0 ? 1u : 0u);
                                else if (i == 4)
                                    mma_ts_warp(tmem + kColS, tmem + kColQRope + 8u * k, bd, idesc_qk_rope, 1u);
                                else
                                    mma_ss_warp(tmem + kColS,
                                                smem_desc_sw128(base + kOffQs + (i - 1) * kQsBox + k * 32u, 16u, 1024u),
                                                bd, idesc_qk, 1u);
                            }
                        }
                        mma_commit_warp(bar(base, B_OTH_EMPTY));
                        const DhSlot dso = dh_slot<kSparse>(g, 0);
                        const int ds = dso.slot;
                        if (!warp_wait(c, bar(base, dso.full), dso.phase & 1u, false)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        if (have) {
                            const uint32_t dh = base + kOffDh + ds * kDhBytes;
                            for (int k = 0; k < 16; ++k)
                                mma_ts_warp(tmem + kColS, tmem + kColQ + 8u * k,
                                            smem_desc_sw128(dh + (k >> 2) * kBox + (k & 3) * 32u, 16u, 1024u), idesc_qk,
                                            1u);
                        }
                        mma_commit_warp(bar(base, B_S_FULL));
                    }
                    if (!kFp8 && ok) mma_commit_warp(bar(base, B_QDONE));  // this item's QK^T are issued
                }
            }
            if (!ok) drain_pause();
        }
    } else if (warp == 6) {
        // ------------------------------------------------------------ PV issuer
        // warp-wide like the QK^T issuer
        {
            constexpr uint32_t idesc_pv = kFp8 ? idesc_f16(128, 256, true) : idesc_bf16(128, 256, true);
            uint32_t g = 0;
            bool ok = true;
            for (int u = cl; u < units && ok; u += ncl) {
                for (int it = unit_begin[u]; it < unit_begin[u + 1] && ok; ++it) {
                    const WorkItem w = items[it];
                    bool first = true;
                    for (int t = w.t0; t < w.t1; t += kTile, ++g) {
                        // the probability tile is reused only after both CTAs' PV of the
                        // previous tile, so P_FULL never runs two phases ahead
                        if (!warp_wait(c, bar(base, B_P_FULL), g & 1u, false)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const int nvalid = min(kTile, w.t1 - t);
                        const uint32_t ps = base + kOffP;
                        for (int e = 1; e >= 0; --e) {  // peer page, then own page
                            const int p = e == 0 ? (int)rank : (int)peer;
                            const DhSlot d = dh_slot<kSparse>(g, e);
                            const int ds = d.slot;
                            const int ksteps = min(4, max(0, (nvalid - kPageRows * p + 15) / 16));
                            // wait even for a page that is absent (ksteps 0): the buffer is handed
                            // back below, and for FP8 records its expansion (a stage between the raw
                            // load and this barrier) must have passed first, or the raw loader could
                            // run two phases ahead of it
                            if (!warp_wait(c, bar(base, d.full), d.phase & 1u, false)) {
                                ok = false;
                                break;
                            }
                            tc_fence_after();
                            const uint32_t dh = base + kOffDh + ds * kDhBytes;
                            for (int kk = 0; kk < ksteps; ++kk) {
                                const uint64_t ad = smem_desc_sw128(ps + p * kPPage + kk * 32u, 16u, 1024u);
                                const uint64_t bd = smem_desc_sw128(dh + kk * 2048u, kBox, 1024u);
                                mma_ss_warp(tmem + kColO, ad, bd, idesc_pv, first ? 0u : 1u);
                                first = false;
                            }
                            mma_commit_warp(bar(base, B_DH_EMPTY + ds));
                        }
                        if (!ok) break;
                        mma_commit_multicast_warp(bar(base, B_PFREE), (uint16_t)3);
                        if (t + kTile >= w.t1) mma_commit_warp(bar(base, B_O_FINAL));
                    }
                }
            }
            if (!ok) drain_pause();
        }
    } else if (warp < 4) {
        // ------------------------------------------------------------ softmax + epilogue
        // Per tile: part A (scores -> own weights -> message to the peer), then part B
        // (merge with the peer's message -> PV may start).
        const int h = threadIdx.x;  // head row = TMEM lane
        const uint32_t trow = tmem + ((uint32_t)(warp * 32) << 16);
        const uint32_t peer_p = mapa(base + kOffP, peer);
        const float sc = a.scale_log2;  // > 0, checked on the host
        uint8_t *ps = gbase + kOffP;
        // Query of request bq: 384 columns into TMEM (own latent half, RoPE, the other
        // half's first 64), 192 into shared memory (the other half's last 192).  The TMA brings
        // them in three rounds of three 64-column boxes (128 heads, 128-B swizzle) through the
        // shared-memory query area: rounds 0 and 1 go on to TMEM, each thread moving its own
        // head's row; round 2 stays.  Heads at or beyond H lie outside the tensor: zeros.
        uint32_t qphase = 0;
        float qmax = 0.f;  // FP8 records: largest query magnitude converted to fp16
        // issues round `round` of request bq's query boxes (thread 0)
        auto q_round = [&](int bq, int round) {
            const uint32_t qb = bar(base, B_QLD);
            mbar_arrive_expect_tx(qb, 3 * kQsBox);
            for (int i = 0; i < 3; ++i) {
                // block 0-3: own half, 4: RoPE, 5: other half 0-63, 6-8: other half 64-255
                const int blk = 3 * round + i;
                const uint32_t dst = base + kOffQs + i * kQsBox;
                if (blk == 4)
                    tma_load_3d(dst, &tmap_qr, 0, 0, bq, qb);
                else
                    tma_load_3d(dst, &tmap_qn, blk < 4 ? 256 * (int)rank + 64 * blk : 256 * (int)peer + 64 * (blk - 5), 0,
                                bq, qb);
            }
        };
        // round0_issued: round 0 was issued already (as soon as the previous item's last
        // scores were read, so that its latency hides behind that tile's merge)
        // A warp whose wait fails still takes part in the named barriers of rounds 0 and 1
        // (bar.sync has no time limit, so every one of the 128 threads must arrive); it only
        // skips the work, and the load reports the failure at the end.
        auto load_q = [&](int bq, bool round0_issued) -> bool {
            const uint32_t qb = bar(base, B_QLD);
            bool okq = true;
            for (int round = 0; round < 3; ++round) {
                if (threadIdx.x == 0 && okq && !(round == 0 && round0_issued)) q_round(bq, round);
                if (okq) okq = warp_wait(c, qb, qphase & 1u, false);
                ++qphase;
                if (round == 2) break;
#pragma unroll 1
                for (int i = 0; i < 3 && okq; ++i) {
                    const uint8_t *row = gbase + kOffQs + i * kQsBox + h * 128;
                    uint32_t v[32];
#pragma unroll
                    for (int q = 0; q < 8; ++q) {
                        const uint4 x = *reinterpret_cast<const uint4 *>(row + ((q ^ (h & 7)) * 16));
                        v[4 * q] = x.x;
                        v[4 * q + 1] = x.y;
                        v[4 * q + 2] = x.z;
                        v[4 * q + 3] = x.w;
                    }
                    // FP8 records: the latent part of the query becomes fp16 like the latent
                    // operand it meets (block 4, the RoPE part, stays bf16)
                    if (kFp8 && 3 * round + i != 4) {
#pragma unroll
                        for (int q = 0; q < 32; ++q) v[q] = bf16x2_to_f16x2(v[q], &qmax);
                    }
                    tmem_st32(trow + kColQ + 32u * (3 * round + i), v);
                }
                named_bar_sync(1, 128);  // every head's rows are read before the next round lands
            }
            if (!okq) return false;
            if constexpr (kFp8) {
                // the query's last 192 latent columns stay in shared memory: each thread
                // converts its own head's rows in place (the conversion is per element, so the
                // swizzle of the 16-B units does not matter)
                for (int i = 0; i < 3; ++i) {
                    uint4 *row = reinterpret_cast<uint4 *>(gbase + kOffQs + i * kQsBox + h * 128);
#pragma unroll
                    for (int q = 0; q < 8; ++q) {
                        uint4 x = row[q];
                        x.x = bf16x2_to_f16x2(x.x, &qmax);
                        x.y = bf16x2_to_f16x2(x.y, &qmax);
                        x.z = bf16x2_to_f16x2(x.z, &qmax);
                        x.w = bf16x2_to_f16x2(x.w, &qmax);
                        row[q] = x;
                    }
                }
                fence_proxy_async_smem();
                if (qmax > kF16Max) record_error(a.status, MLA_ERR_RANGE);
                qmax = 0.f;
            }
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(base, B_Q_READY));
            return true;
        };
        uint32_t g = 0, nitem = 0;
        bool ok = true, q_ready = false;  // q_ready: the current item's query is in place
        for (int u = cl; u < units && ok; u += ncl) {
            for (int it = unit_begin[u]; it < unit_begin[u + 1] && ok; ++it) {
                const WorkItem w = items[it];
                const int b = w.b;
                float *orow;
                float *lrow;
                if (w.slot < 0) {
                    orow = a.out + ((int64_t)b * a.H + h) * kDLatent + rank * 256;
                    lrow = a.lse + (int64_t)b * a.H + h;
                } else {
                    orow = part_o + ((int64_t)w.slot * a.H + h) * kDLatent + rank * 256;
                    lrow = part_lse + (int64_t)w.slot * a.H + h;
                }
                if (w.t1 <= w.t0) {
                    if (h < a.H) {
                        for (int q = 0; q < 64; ++q)
                            reinterpret_cast<float4 *>(orow)[q] = make_float4(0.f, 0.f, 0.f, 0.f);
                        if (rank == 0) *lrow = -INFINITY;
                    }
                    continue;
                }
                // FP8 records: this warp group loads and converts the query (dense and sparse
                // tiles: the MMA issuer does, with tcgen05.cp)
                int bnext = -1;
                if constexpr (kFp8) {
                    if (!q_ready && !load_q(b, false)) {
                        ok = false;
                        break;
                    }
                    q_ready = false;
                    // the next item's query is loaded at the end of this one: bring it into L2 now
                    bnext = next_request(unit_begin, items, units, ncl, u, it);
                    if (bnext >= 0 && threadIdx.x == 0) {
                        prefetch_l2(a.q_nope + (int64_t)bnext * a.H * kDLatent, (uint32_t)(a.H * kDLatent * 2));
                        prefetch_l2(a.q_rope + (int64_t)bnext * a.H * kDRope, (uint32_t)(a.H * kDRope * 2));
                    }
                }
                float m = -INFINITY, l = 0.f;
                // which rows of each page attend (warp-collective), read one tile ahead
                PageMask nm0 = page_mask<kSparse>(a, w, w.t0, 0, lane), nm1 = page_mask<kSparse>(a, w, w.t0, 1, lane);
                for (int t = w.t0, j = 0; t < w.t1; t += kTile, ++j, ++g) {
                    // ================= part A: own page's scores -> weights -> message
                    const int nvalid = min(kTile, w.t1 - t);
                    const PageMask pm0 = nm0, pm1 = nm1;
                    if (t + kTile < w.t1) {
                        nm0 = page_mask<kSparse>(a, w, t + kTile, 0, lane);
                        nm1 = page_mask<kSparse>(a, w, t + kTile, 1, lane);
                    }
                    const uint64_t vown = rank == 0 ? pm0.valid : pm1.valid;
                    if (!warp_wait(c, bar(base, B_S_FULL), g & 1u, false)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    float s[64];
                    {
                        uint32_t sr[64];
                        tmem_ld32(trow + kColS, *reinterpret_cast<uint32_t(*)[32]>(&sr[0]));
                        tmem_ld32(trow + kColS + 32u, *reinterpret_cast<uint32_t(*)[32]>(&sr[32]));
                        tmem_wait_ld();
#pragma unroll
                        for (int i = 0; i < 64; ++i) s[i] = __uint_as_float(sr[i]);
                    }
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(bar(base, B_S_FREE));
                    // the item's last scores are read: its query area is free for the next query
                    if (kFp8 && t + kTile >= w.t1 && bnext >= 0 && threadIdx.x == 0) q_round(bnext, 0);
                    if (vown != ~0ull) {
#pragma unroll
                        for (int i = 0; i < 64; ++i)
                            if (!((vown >> i) & 1ull)) s[i] = -INFINITY;
                    }
                    float mraw = s[0];
#pragma unroll
                    for (int i = 1; i < 64; ++i) mraw = fmaxf(mraw, s[i]);
                    const float mloc = mraw * sc;
                    // reference: the running maximum; any value works as long as both CTAs
                    // use the one they send
                    const float rown = mloc > m + kRescaleLog2 ? mloc : m;
                    const float nr = rown == -INFINITY ? 0.f : -rown;
                    uint32_t pk[32];
                    float lown = 0.f;
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        const float p0 = ex2_approx(fmaf(s[2 * i], sc, nr));
                        const float p1 = ex2_approx(fmaf(s[2 * i + 1], sc, nr));
                        lown += p0 + p1;
                        pk[i] = pack_op<kFp8>(p0, p1);
                    }
                    // cache rows that PV reads but must not contribute (rows of the last
                    // 16-row step past the end, a page whose id was out of range, sparse slots
                    // that are padding or out of range) must hold zeros there, not whatever
                    // the loaded row holds; decided here, off the merge's path
                    uint64_t zmask[2];
#pragma unroll
                    for (int p = 0; p < 2; ++p) {
                        const PageMask pm = p == 0 ? pm0 : pm1;
                        const int z1 = min(kPageRows, (pm.cnt + 15) & ~15);
                        zmask[p] = ~pm.valid & (z1 >= 64 ? ~0ull : ((1ull << z1) - 1ull));
                    }
                    const bool need_zero = (zmask[0] | zmask[1]) != 0ull;  // the same in every lane
                    // the tile is reused: both CTAs' PV of the previous tile must be done
                    if (g > 0 && !warp_wait(c, bar(base, B_PFREE), (g - 1) & 1u, true)) {
                        ok = false;
                        break;
                    }
                    {
                        uint8_t *prow = ps + rank * kPPage + h * 128;
#pragma unroll
                        for (int q = 0; q < 8; ++q)
                            *reinterpret_cast<uint4 *>(prow + ((q ^ (h & 7)) * 16)) =
                                make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
                        float *rl = reinterpret_cast<float *>(ps + 2 * kPPage + rank * kRlBytes);
                        rl[h] = rown;
                        rl[128 + h] = lown;
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                    const uint32_t rfull = bar(base, B_RFULL);
                    if (threadIdx.x == 0) mbar_arrive_expect_tx(rfull, kMsgBytes);
                    if (lane == 0) {
                        const uint32_t rb = mapa(rfull, peer);
                        const uint32_t prows = kOffP + rank * kPPage + warp * 32 * 128;
                        const uint32_t rls = kOffP + 2 * kPPage + rank * kRlBytes + warp * 32 * 4;
                        bulk_copy_s2peer(peer_p - kOffP + prows, base + prows, 32 * 128, rb);
                        bulk_copy_s2peer(peer_p - kOffP + rls, base + rls, 32 * 4, rb);
                        bulk_copy_s2peer(peer_p - kOffP + rls + 512, base + rls + 512, 32 * 4, rb);
                        bulk_commit();
                    }
                    // ================= part B: merge with the peer's message
                    if (!warp_wait(c, rfull, g & 1u, true)) {
                        ok = false;
                        break;
                    }
                    const float *rlp = reinterpret_cast<const float *>(ps + 2 * kPPage + peer * kRlBytes);
                    const float rpeer = rlp[h], lpeer = rlp[128 + h];
                    const float r0 = rank == 0 ? rown : rpeer, r1 = rank == 0 ? rpeer : rown;
                    const float l0 = rank == 0 ? lown : lpeer, l1 = rank == 0 ? lpeer : lown;
                    const float mn = fmaxf(m, fmaxf(r0, r1));
                    float f0 = 1.f, f1 = 1.f, alpha = 1.f;
                    if (mn != -INFINITY) {
                        f0 = ex2_approx(r0 - mn);
                        f1 = ex2_approx(r1 - mn);
                        alpha = ex2_approx(m - mn);
                        l = l * alpha + l0 * f0 + l1 * f1;
                    }
                    const bool resc_o = j > 0 && mn > m;
                    m = mn;
                    // a page whose reference lies below the new maximum is rescaled in place
                    // (this CTA's own rows only after the warp's bulk copies have read them)
                    const float fown = rank == 0 ? f0 : f1, fpeer = rank == 0 ? f1 : f0;
                    bool wrote = false;
                    if (__any_sync(0xffffffffu, fown < 1.f)) {
                        if (lane == 0) bulk_wait_read_all();
                        __syncwarp();
                        if (fown < 1.f) scale_row_ool<kFp8>(reinterpret_cast<uint4 *>(ps + rank * kPPage + h * 128), fown);
                        wrote = true;
                    }
                    if (fpeer < 1.f) {
                        scale_row_ool<kFp8>(reinterpret_cast<uint4 *>(ps + peer * kPPage + h * 128), fpeer);
                        wrote = true;
                    }
                    // zero the rows decided in part A
                    for (int p = 0; p < 2 && need_zero; ++p) {
                        const uint64_t zero = zmask[p];
                        if (zero == 0ull) continue;
                        const DhSlot d = dh_slot<kSparse>(g, p == (int)rank ? 0 : 1);
                        const int ds = d.slot;
                        // wait for the slot's load (or its empty arrival) to land first
                        if (!warp_wait(c, bar(base, d.full), d.phase & 1u, false)) {
                            ok = false;
                            break;
                        }
                        zero_rows(gbase + kOffDh + ds * kDhBytes, zero, h);
                        wrote = true;
                    }
                    if (!ok) break;
                    if (__any_sync(0xffffffffu, wrote)) fence_proxy_async_smem();
                    // O rescale: the previous tile's PV is done (waited above before the
                    // probability tile was rewritten)
                    if (__any_sync(0xffffffffu, resc_o)) {
                        tc_fence_after();
                        rescale_o_row(trow + kColO, resc_o ? alpha : 1.f);
                    }
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(bar(base, B_P_FULL));
                }
                if (!ok) break;
                // ---- the next item's query: this item's QK^T is complete (its last S was
                // read), so the query columns are free; loading now lets the next item's
                // QK^T overlap this item's last PV and epilogue
                if (kFp8 && bnext >= 0) {
                    if (!load_q(bnext, true)) {
                        ok = false;
                        break;
                    }
                    q_ready = true;
                }
                // ---- epilogue: wait for the last PV of this item, normalise, store
                if (!warp_wait(c, bar(base, B_O_FINAL), nitem & 1u, false)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const float inv = l > 0.f ? 1.f / l : 0.f;
                // Each 32-column slice goes through this CTA's own probability rows (free
                // until the next tile's weights; the peer never writes them) so that every
                // warp store covers whole 128-B lines: thread h holds row h, but rows are
                // 2 KB apart in the output.  Warp w writes back its own rows 32w..32w+31.
                {
                    uint8_t *stg = ps + rank * kPPage;
                    float *obase = orow - (int64_t)h * kDLatent;  // row 0 of this item's output
                    if (lane == 0) bulk_wait_read_all();  // this warp's last message has left these rows
                    __syncwarp();
                    store_rows(trow + kColO, stg, obase, inv, h, warp, lane, a.H);
                }
                if (rank == 0 && h < a.H) *lrow = l > 0.f ? (m + log2f(l)) * kLn2 : -INFINITY;
                ++nitem;
                tc_fence_before();
            }
        }
    }

    // ---------------------------------------------------------------- teardown
    grid_dep_launch();  // the merge kernel may start launching
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

// Sets the shared-memory limit of the kernel variants once per device.
bool set_smem_attr() {
    static bool done[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return false;
    if (done[dev]) return true;
    if (cudaFuncSetAttribute(decode_sm103_kernel<0>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes) !=
            cudaSuccess ||
        cudaFuncSetAttribute(decode_sm103_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes) !=
            cudaSuccess ||
        cudaFuncSetAttribute(decode_sm103_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes) !=
            cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    done[dev] = true;
    return true;
}

// 2-D tensor map over the cache's rows (num_pages * 64 of `row_bytes` each).
bool make_tmap(CUtensorMap *m, const void *cache, int64_t num_pages, CUtensorMapDataType dtype, int elem_bytes,
               uint64_t row_bytes, uint32_t box_x, uint32_t box_y, CUtensorMapSwizzle swz) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)(row_bytes / elem_bytes), (cuuint64_t)num_pages * kPageRows};
    const cuuint64_t strides[1] = {(cuuint64_t)row_bytes};
    const cuuint32_t box[2] = {box_x, box_y};
    const cuuint32_t estr[2] = {1, 1};
    return enc(m, dtype, 2, const_cast<void *>(cache), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Queries [B][H][cols] bf16 as a 3-D tensor (cols, H, B); boxes of 64 columns x 128 heads of
// one request, 128-B swizzle.  Heads at or beyond H fall outside the tensor and read zeros.
bool make_tmap_q(CUtensorMap *m, const void *q, int cols, int H, int B) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return false;
    const cuuint64_t dims[3] = {(cuuint64_t)cols, (cuuint64_t)H, (cuuint64_t)B};
    const cuuint64_t strides[2] = {(cuuint64_t)cols * 2, (cuuint64_t)cols * 2 * H};
    const cuuint32_t box[3] = {64, 128, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(q), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

int sm103_max_units() {
    static int cached = -1;
    static int cached_dev = -1;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (cached >= 0 && cached_dev == dev) return cached;
    if (!set_smem_attr()) return 0;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2, 1, 1);
    cfg.blockDim = dim3(kThreadsFp8, 1, 1);
    cfg.dynamicSmemBytes = kSmemBytes;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeClusterDimension;
    attr.val.clusterDim.x = 2;
    attr.val.clusterDim.y = 1;
    attr.val.clusterDim.z = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, decode_sm103_kernel<2>, &cfg) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    cached = n;
    cached_dev = dev;
    return n;
}

// Launch with programmatic stream serialization: the grid may start while the plan kernel
// finishes (every CTA first waits for it in grid_dep_wait()).
template <typename K>
cudaError_t launch_pdl(K kernel, dim3 grid, int threads, cudaStream_t stream, const CUtensorMap &t0,
                       const CUtensorMap &t1, const CUtensorMap &t2, const CUtensorMap &t3, const CUtensorMap &t4,
                       const DecodeArgs &a) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(threads, 1, 1);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr.val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, t0, t1, t2, t3, t4, a);
}

cudaError_t launch_decode_sm103(const DecodeArgs &a, int num_clusters, cudaStream_t stream) {
    if (!set_smem_attr()) return cudaErrorInvalidValue;
    const dim3 grid(2 * num_clusters);
    CUtensorMap tm, tm_sc, tm_rope, tm_qn, tm_qr;
    if (!make_tmap_q(&tm_qn, a.q_nope, kDLatent, a.H, a.B) || !make_tmap_q(&tm_qr, a.q_rope, kDRope, a.H, a.B))
        return cudaErrorInvalidValue;
    if (a.kv_fp8) {
        // records of 656 B: codes as bytes (128-B boxes, a quarter of the latent of 64 rows), the 16-B
        // scale block, and the RoPE part as bf16 (element 264 = byte 528, 128-B swizzle)
        if (!make_tmap(&tm, a.cache, a.num_pages, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, kFp8RecordBytes, 128, kPageRows,
                       CU_TENSOR_MAP_SWIZZLE_NONE) ||
            !make_tmap(&tm_sc, a.cache, a.num_pages, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, kFp8RecordBytes, 16, kPageRows,
                       CU_TENSOR_MAP_SWIZZLE_NONE) ||
            !make_tmap(&tm_rope, a.cache, a.num_pages, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, kFp8RecordBytes, 64,
                       kPageRows, CU_TENSOR_MAP_SWIZZLE_128B))
            return cudaErrorInvalidValue;
        return launch_pdl(decode_sm103_kernel<2>, grid, kThreadsFp8, stream, tm, tm_sc, tm_rope, tm_qn, tm_qr, a);
    } else if (a.indices) {
        // one-row boxes for tile::gather4
        if (!make_tmap(&tm, a.cache, a.num_pages, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, (uint64_t)kDEntry * 2, 64, 1,
                       CU_TENSOR_MAP_SWIZZLE_128B))
            return cudaErrorInvalidValue;
        // and 64-row boxes for index runs that cover a whole page
        CUtensorMap tm_page;
        if (!make_tmap(&tm_page, a.cache, a.num_pages, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, (uint64_t)kDEntry * 2, 64,
                       kPageRows, CU_TENSOR_MAP_SWIZZLE_128B))
            return cudaErrorInvalidValue;
        return launch_pdl(decode_sm103_kernel<1>, grid, kThreadsSparse, stream, tm, tm_page, tm, tm_qn, tm_qr, a);
    } else {
        // 64-row boxes: one page
        if (!make_tmap(&tm, a.cache, a.num_pages, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, (uint64_t)kDEntry * 2, 64,
                       kPageRows, CU_TENSOR_MAP_SWIZZLE_128B))
            return cudaErrorInvalidValue;
        return launch_pdl(decode_sm103_kernel<0>, grid, kThreads, stream, tm, tm, tm, tm_qn, tm_qr, a);
    }
    return cudaGetLastError();
}

}  // namespace mla
