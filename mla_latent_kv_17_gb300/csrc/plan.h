// Split-KV work planner and workspace layout, shared by the device plan kernel and the
// host twin (mla_decode_plan_host).  The same function runs on both sides so the two
// produce byte-identical plans.
//
// A request's tokens are cut into 64-token tiles (one cache page each).  The persistent
// decode workers ("units", one per pair of SMs) each get an equal budget of tiles; the
// planner walks the requests in order and fills units one after another, so a request
// that straddles a unit boundary is cut into pieces (split-KV).  Each piece costs its
// tiles plus a fixed overhead (query load, epilogue), and no piece is made smaller than
// kMinPieceTiles unless it is the request's last.  Requests cut into several pieces write
// per-piece partial results (out_i normalised, lse_i), merged afterwards through their
// log-sum-exp ("Fused Reduction" of weight-absorbed decode, "MLA 最佳算子全景调研" §3).
#pragma once
#include <stddef.h>
#include <stdint.h>

#if defined(__CUDACC__)
#define MLA_HD __host__ __device__ __forceinline__
#else
#define MLA_HD inline
#endif

namespace mla {

constexpr int kDLatent = 512;
constexpr int kDRope = 64;
constexpr int kDEntry = 576;
constexpr int kPageRows = 64;
constexpr int kFp8RecordBytes = 656;
constexpr int kMaxHeads = 128;
constexpr int kTileTokens = 64;
constexpr int kSmsPerUnit = 2;
constexpr int kPieceOverheadTiles = 3;
constexpr int kMinPieceTiles = 4;
constexpr uint32_t kPlanMagic = 0x4D4C4150u;  // "MLAP"

struct PlanHeader {
    uint32_t magic;
    int32_t B, H, topk, num_units, num_items, max_items, max_partials;
    int32_t tiles_per_unit, num_partials, reserved[6];
};
static_assert(sizeof(PlanHeader) == 64, "plan header is 64 bytes");

// One unit of work: tokens [t0, t1) of request b (index slots for sparse decode).
// slot < 0: write out/lse directly; slot >= 0: write partial slot `slot`.
struct WorkItem {
    int32_t b, t0, t1, slot;
};

MLA_HD size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Byte offsets inside the workspace.  Everything up to `plan_end` is the plan proper.
struct WsLayout {
    size_t header, status, unit_begin, items, num_splits, split_base, plan_end;
    size_t part_lse, part_o, total;
    int max_items, max_partials, num_units;
};

MLA_HD WsLayout ws_layout(int B, int H, int num_units) {
    WsLayout L;
    L.num_units = num_units;
    L.max_items = B + num_units;
    L.max_partials = L.max_items;
    L.header = 0;
    L.status = 128;  // 4-byte device status word, outside the header
    size_t o = 256;
    L.unit_begin = o;
    o = align_up(o + sizeof(int32_t) * (size_t)(num_units + 1), 256);
    L.items = o;
    o = align_up(o + sizeof(WorkItem) * (size_t)L.max_items, 256);
    L.num_splits = o;
    o = align_up(o + sizeof(int32_t) * (size_t)B, 256);
    L.split_base = o;
    o = align_up(o + sizeof(int32_t) * (size_t)B, 256);
    L.plan_end = o;
    L.part_lse = o;
    o = align_up(o + sizeof(float) * (size_t)L.max_partials * H, 256);
    L.part_o = o;
    o = align_up(o + sizeof(float) * (size_t)L.max_partials * H * kDLatent, 256);
    L.total = o;
    return L;
}

MLA_HD int num_units_for(int num_sms) {
    int u = num_sms / kSmsPerUnit;
    return u < 1 ? 1 : u;
}

// Length (in tokens or index slots) that request b is planned over.
MLA_HD int32_t planned_len(const int32_t *seq_lens, int topk, int b) {
    if (topk > 0) return topk;
    int32_t L = seq_lens[b];
    return L < 0 ? 0 : L;
}

// Walks the requests with a per-unit budget of `per` cost units (tiles + a fixed overhead
// per piece), filling units in order.  With `emit`, writes the items, unit_begin and
// num_splits; always returns the cost that lands on the last unit (which takes whatever
// remains), so the caller can search for the smallest budget that does not overflow it.
MLA_HD long long walk_plan(const int32_t *seq_lens, int B, int topk, int num_units,
                           long long per, bool emit, int32_t *unit_begin, WorkItem *items,
                           int32_t *num_splits, int *n_items) {
    int n = 0;
    int u = 0;
    long long cap = per;
    if (emit)
        for (int i = 0; i <= num_units; ++i) unit_begin[i] = 0;
    for (int b = 0; b < B; ++b) {
        int32_t len = planned_len(seq_lens, topk, b);
        int32_t tiles = (len + kTileTokens - 1) / kTileTokens;
        if (emit) num_splits[b] = 0;
        if (tiles == 0) {
            if (emit) {
                items[n].b = b; items[n].t0 = 0; items[n].t1 = 0; items[n].slot = -1;
                num_splits[b] = 1;
            }
            ++n;
            continue;
        }
        int32_t t = 0;
        while (t < tiles) {
            long long avail = cap - kPieceOverheadTiles;
            int32_t rest = tiles - t;
            int32_t take;
            if (avail >= rest || u == num_units - 1) {
                take = rest;
            } else {
                take = avail < 0 ? 0 : (int32_t)avail;
                if (rest - take < kMinPieceTiles) take = rest - kMinPieceTiles;
                if (take < kMinPieceTiles) {
                    // too little room left here: continue in the next unit
                    if (emit) unit_begin[u + 1] = n;
                    ++u;
                    cap = per;
                    continue;
                }
            }
            if (emit) {
                items[n].b = b;
                items[n].t0 = t * kTileTokens;
                int32_t e = (t + take) * kTileTokens;
                items[n].t1 = e < len ? e : len;
                items[n].slot = -1;
                ++num_splits[b];
            }
            ++n;
            t += take;
            cap -= take + kPieceOverheadTiles;
            if (cap <= kPieceOverheadTiles && u < num_units - 1 && t < tiles) {
                if (emit) unit_begin[u + 1] = n;
                ++u;
                cap = per;
            }
        }
    }
    if (emit)
        for (int i = u + 1; i <= num_units; ++i) unit_begin[i] = n;
    *n_items = n;
    return u == num_units - 1 ? per - cap : 0;
}

// Builds the plan into `ws` (host or device memory laid out by ws_layout).  Sequential;
// on the device it runs on one thread.  The budget is the smallest one (binary search)
// for which the last unit is not overloaded.
MLA_HD void build_plan(const int32_t *seq_lens, int B, int H, int topk, int num_units,
                       unsigned char *ws) {
    WsLayout L = ws_layout(B, H, num_units);
    PlanHeader *hd = reinterpret_cast<PlanHeader *>(ws + L.header);
    int32_t *unit_begin = reinterpret_cast<int32_t *>(ws + L.unit_begin);
    WorkItem *items = reinterpret_cast<WorkItem *>(ws + L.items);
    int32_t *num_splits = reinterpret_cast<int32_t *>(ws + L.num_splits);
    int32_t *split_base = reinterpret_cast<int32_t *>(ws + L.split_base);

    long long total_cost = 0;
    for (int b = 0; b < B; ++b) {
        int32_t tiles = (planned_len(seq_lens, topk, b) + kTileTokens - 1) / kTileTokens;
        total_cost += tiles + (tiles > 0 ? kPieceOverheadTiles : 0);
    }
    long long lo = (total_cost + num_units - 1) / num_units;
    if (lo < kPieceOverheadTiles + kMinPieceTiles) lo = kPieceOverheadTiles + kMinPieceTiles;
    long long hi = total_cost + kPieceOverheadTiles + kMinPieceTiles;
    int n = 0;
    while (lo < hi) {
        long long mid = lo + (hi - lo) / 2;
        if (walk_plan(seq_lens, B, topk, num_units, mid, false, nullptr, nullptr, nullptr, &n) <= mid)
            hi = mid;
        else
            lo = mid + 1;
    }
    const long long per = lo;
    walk_plan(seq_lens, B, topk, num_units, per, true, unit_begin, items, num_splits, &n);
    // Partial slots for requests with more than one piece, in item order.
    for (int b = 0; b < B; ++b) split_base[b] = -1;
    int slots = 0;
    for (int i = 0; i < n; ++i) {
        int b = items[i].b;
        if (num_splits[b] > 1) {
            if (split_base[b] < 0) split_base[b] = slots;
            items[i].slot = slots++;
        }
    }
    hd->magic = kPlanMagic;
    hd->B = B;
    hd->H = H;
    hd->topk = topk;
    hd->num_units = num_units;
    hd->num_items = n;
    hd->max_items = L.max_items;
    hd->max_partials = L.max_partials;
    hd->tiles_per_unit = (int32_t)per;
    hd->num_partials = slots;
    for (int i = 0; i < 6; ++i) hd->reserved[i] = 0;
}

}  // namespace mla
