// Split-KV work planner and workspace layout, shared by the device plan kernel and the
// host twin (mla_decode_plan_host).  The same function runs on both sides so the two
// produce byte-identical plans.
//
// A request's tokens are cut into 128-token tiles (two cache pages; the tensor-core kernel
// works on one such tile per step, a page per SM of the pair).  The persistent decode
// workers ("units", one per pair of SMs) each get an equal budget of tiles; the
// planner walks the requests in order and fills units one after another, so a request
// that straddles a unit boundary is cut into pieces (split-KV).  Each piece costs its
// tiles plus a fixed overhead (query load, epilogue; piece_overhead), and no piece is made
// smaller than kMinPieceTiles unless it is the request's last.  Requests cut into several pieces write
// per-piece partial results (out_i normalised, lse_i), merged afterwards through their
// log-sum-exp ("Fused Reduction" of weight-absorbed decode, "MLA 最佳算子全景调研" §3).
#pragma once
#include <limits.h>
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
constexpr int kTileTokens = 128;
constexpr int kSmsPerUnit = 2;
constexpr int kMinPieceTiles = 2;
constexpr int kMergeCostTiles = 3;  // the split-KV merge's cost on the critical path, in tiles
constexpr uint32_t kPlanMagic = 0x4D4C4150u;  // "MLAP"

struct PlanHeader {
    uint32_t magic;
    int32_t B, H, topk, num_units, num_items, max_items, max_partials;
    int32_t tiles_per_unit, num_partials, num_split_reqs, piece_overhead, reserved[4];
};
static_assert(sizeof(PlanHeader) == 64, "plan header is 64 bytes");

// One unit of work: tokens [t0, t1) of request b (index slots for sparse decode).
// slot < 0: write out/lse directly; slot >= 0: write partial slot `slot`.
struct WorkItem {
    int32_t b, t0, t1, slot;
};

MLA_HD size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Byte offsets inside the workspace.  Everything up to `plan_end` is the plan proper;
// req_start and item_unit are planner scratch that the decode does not read; split_list
// holds the requests cut into several pieces, in order (num_split_reqs of them).
struct WsLayout {
    size_t header, status, unit_begin, items, num_splits, split_base, req_start, item_unit, split_list;
    size_t plan_end, part_lse, part_o, total;
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
    L.req_start = o;
    o = align_up(o + sizeof(int64_t) * (size_t)B, 256);
    L.item_unit = o;
    o = align_up(o + sizeof(int32_t) * (size_t)L.max_items, 256);
    L.split_list = o;
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

// Tiles request b is planned over (tokens, or index slots for sparse decode).
MLA_HD int32_t req_len(const int32_t *seq_lens, int topk, int b) {
    if (topk > 0) return topk;
    int32_t L = seq_lens[b];
    return L < 0 ? 0 : L;
}
MLA_HD int32_t req_tiles(const int32_t *seq_lens, int topk, int b) {
    return (req_len(seq_lens, topk, b) + kTileTokens - 1) / kTileTokens;
}
// What a piece costs beyond its tiles, in tiles: its query load, pipeline refill and
// epilogue.  Clock traces of the decode put an item at ~3 tiles of its own mode in both
// layouts; planned at 2 the bf16 cache runs fastest, and FP8 records (whose softmax warps
// also convert each item's query) at 3.
MLA_HD int piece_overhead(int fp8_records) { return fp8_records ? 3 : 2; }
MLA_HD int64_t req_cost(int32_t tiles, int ovh) { return tiles > 0 ? tiles + ovh : 0; }

// The budget axis: request b occupies cost positions [S_b, S_b + cost_b); its overhead
// comes first, so tile t sits at S_b + overhead + t.  Unit u owns positions
// [u * per, (u + 1) * per); the last unit also takes anything beyond.
MLA_HD int32_t unit_of(int64_t pos, int64_t per, int units) {
    // the same quotient in 32-bit arithmetic when it fits (always, for realistic batches): a
    // 64-bit division is a long instruction sequence on the GPU
    const int64_t u = (pos >= 0 && pos <= INT32_MAX && per <= INT32_MAX) ? (int64_t)((uint32_t)pos / (uint32_t)per)
                                                                          : pos / per;
    return u >= units ? units - 1 : (int32_t)u;
}

// How request b is cut into pieces.  Unit boundaries inside the request give runs of
// tiles that belong to one unit; a first or last run shorter than kMinPieceTiles is folded
// into its neighbour.  Cut k (1 <= k <= uf_last - uf) would start unit uf + k at tile
// (uf + k) * per - p0; cuts kfirst..klast are kept, so the request has
// klast - kfirst + 2 pieces.
struct ReqSplit {
    int64_t p0;
    int32_t uf, kfirst, klast, tiles, n;
};

MLA_HD ReqSplit req_split(int64_t S, int32_t tiles, int64_t per, int units, int ovh) {
    ReqSplit r;
    r.p0 = S + ovh;
    r.tiles = tiles;
    if (tiles <= 0) {
        r.uf = unit_of(S, per, units);
        r.kfirst = 1;
        r.klast = 0;
        r.n = 1;
        return r;
    }
    r.uf = unit_of(r.p0, per, units);
    const int32_t ul = unit_of(r.p0 + tiles - 1, per, units);
    r.kfirst = 1;
    r.klast = ul - r.uf;
    if (r.klast >= 1) {
        const int64_t first_len = (int64_t)(r.uf + 1) * per - r.p0;
        if (first_len < kMinPieceTiles) r.kfirst = 2;
        const int64_t last_len = tiles - ((int64_t)ul * per - r.p0);
        if (last_len < kMinPieceTiles && r.klast >= r.kfirst) r.klast -= 1;
    }
    r.n = r.klast - r.kfirst + 2;
    return r;
}

// Tile range [tb, te) and unit of piece i of a request.
MLA_HD void req_piece(const ReqSplit &r, int i, int64_t per, int units, int32_t *tb, int32_t *te,
                      int32_t *unit) {
    if (r.tiles <= 0) {
        *tb = 0;
        *te = 0;
        *unit = r.uf;
        return;
    }
    const int32_t k = r.kfirst + i;  // cut that ends piece i (if k <= klast)
    const int32_t b = i == 0 ? 0 : (int32_t)((int64_t)(r.uf + k - 1) * per - r.p0);
    const int32_t e = k <= r.klast ? (int32_t)((int64_t)(r.uf + k) * per - r.p0) : r.tiles;
    *tb = b;
    *te = e;
    *unit = unit_of(r.p0 + (b + e - 1) / 2, per, units);
}

// Per-unit budget: the total cost spread evenly, at least one minimal piece.  When every
// request costs the same (top-k lists: uniform_cost > 0, nreq of them), a budget of k whole
// requests per unit (k = ceil(nreq / units)) puts every request in one unit, with no partial
// results and no merge; it is taken whenever it exceeds the even budget by no more than the
// merge's cost (kMergeCostTiles).
MLA_HD int64_t plan_budget(int64_t total_cost, int units, int64_t uniform_cost, int64_t nreq, int ovh) {
    const int64_t num = total_cost + units - 1;
    int64_t per = num <= INT32_MAX ? (int64_t)((uint32_t)num / (uint32_t)units) : num / units;
    const int64_t lo = ovh + kMinPieceTiles;
    if (per < lo) per = lo;
    if (uniform_cost > 0 && nreq > 0) {
        const int64_t pack = (nreq + units - 1) / units * uniform_cost;
        if (pack <= per + kMergeCostTiles) return pack;
    }
    return per;
}

// Piece i of request b (len tokens, cut as r) as work item `item`; unit_copy, when given,
// receives the item's unit as well.
MLA_HD void emit_piece(unsigned char *ws, const WsLayout &L, int b, int32_t len, const ReqSplit &r, int i,
                       int64_t per, int units, int32_t item, int32_t slot0, int32_t *unit_copy) {
    WorkItem *items = reinterpret_cast<WorkItem *>(ws + L.items);
    int32_t *item_unit = reinterpret_cast<int32_t *>(ws + L.item_unit);
    int32_t tb, te, u;
    req_piece(r, i, per, units, &tb, &te, &u);
    WorkItem w;
    w.b = b;
    w.t0 = tb * kTileTokens;
    const int32_t e = te * kTileTokens;
    w.t1 = e < len ? e : len;
    w.slot = r.n > 1 ? slot0 + i : -1;
    items[item] = w;
    item_unit[item] = u;
    if (unit_copy) unit_copy[item] = u;
}

// Writes the pieces of request b (its item offset `off`, its first partial slot `slot0`
// or -1) into the workspace.
MLA_HD void emit_request(unsigned char *ws, const WsLayout &L, const int32_t *seq_lens, int topk,
                         int b, int64_t S, int64_t per, int units, int ovh, int32_t off, int32_t slot0,
                         int32_t *unit_copy = nullptr) {
    const int32_t len = req_len(seq_lens, topk, b);
    const int32_t tiles = (len + kTileTokens - 1) / kTileTokens;
    const ReqSplit r = req_split(S, tiles, per, units, ovh);
    for (int i = 0; i < r.n; ++i) emit_piece(ws, L, b, len, r, i, per, units, off + i, slot0, unit_copy);
}

MLA_HD void write_header(unsigned char *ws, const WsLayout &L, int B, int H, int topk, int units,
                         int n_items, int64_t per, int n_partials, int n_split_reqs, int ovh) {
    PlanHeader *hd = reinterpret_cast<PlanHeader *>(ws + L.header);
    hd->magic = kPlanMagic;
    hd->B = B;
    hd->H = H;
    hd->topk = topk;
    hd->num_units = units;
    hd->num_items = n_items;
    hd->max_items = L.max_items;
    hd->max_partials = L.max_partials;
    hd->tiles_per_unit = (int32_t)per;
    hd->num_partials = n_partials;
    hd->num_split_reqs = n_split_reqs;
    hd->piece_overhead = ovh;
    for (int i = 0; i < 4; ++i) hd->reserved[i] = 0;
}

// First item index whose unit is >= u (items are ordered by unit).
MLA_HD int32_t lower_bound_unit(const int32_t *item_unit, int32_t n, int32_t u) {
    int32_t lo = 0, hi = n;
    while (lo < hi) {
        int32_t mid = (lo + hi) / 2;
        if (item_unit[mid] < u)
            lo = mid + 1;
        else
            hi = mid;
    }
    return lo;
}

// Host planner: the same per-request functions in serial loops.  The device planner
// (plan kernel) computes the same prefix sums in parallel and writes identical bytes.
inline void build_plan_serial(const int32_t *seq_lens, int B, int H, int topk, int units, int ovh,
                              unsigned char *ws) {
    const WsLayout L = ws_layout(B, H, units);
    int32_t *num_splits = reinterpret_cast<int32_t *>(ws + L.num_splits);
    int32_t *split_base = reinterpret_cast<int32_t *>(ws + L.split_base);
    int64_t *req_start = reinterpret_cast<int64_t *>(ws + L.req_start);
    int32_t *unit_begin = reinterpret_cast<int32_t *>(ws + L.unit_begin);
    int32_t *item_unit = reinterpret_cast<int32_t *>(ws + L.item_unit);
    int32_t *split_list = reinterpret_cast<int32_t *>(ws + L.split_list);
    int64_t S = 0;
    for (int b = 0; b < B; ++b) {
        req_start[b] = S;
        S += req_cost(req_tiles(seq_lens, topk, b), ovh);
    }
    const int64_t per = plan_budget(S, units, topk > 0 ? req_cost(req_tiles(seq_lens, topk, 0), ovh) : 0, B, ovh);
    int32_t off = 0, slots = 0, nsr = 0;
    for (int b = 0; b < B; ++b) {
        const ReqSplit r = req_split(req_start[b], req_tiles(seq_lens, topk, b), per, units, ovh);
        num_splits[b] = r.n;
        split_base[b] = r.n > 1 ? slots : -1;
        emit_request(ws, L, seq_lens, topk, b, req_start[b], per, units, ovh, off, split_base[b]);
        off += r.n;
        if (r.n > 1) {
            slots += r.n;
            split_list[nsr++] = b;
        }
    }
    for (int u = 0; u <= units; ++u)
        unit_begin[u] = u == units ? off : lower_bound_unit(item_unit, off, u);
    write_header(ws, L, B, H, topk, units, off, per, slots, nsr, ovh);
}

}  // namespace mla
