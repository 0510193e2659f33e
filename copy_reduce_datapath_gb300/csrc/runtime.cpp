// Host runtime of libpurlin1: layouts, validation, the SNAC derivation of a
// work list from a layout pair, the per-context work-list cache and the launch
// of the persistent Atom kernel.
//
// "Purlin: Separating Orchestration from the Datapath of Collectives":
//   - abstract: collectives are specified as (input layout, output layout,
//     copy or reduction); SNAC derives coordination from that specification;
//   - Table 1 ("Derivability"): no explicit communication schedule is written
//     by hand -- here every work item, flag and ring slot comes from the
//     layout pair alone;
//   - Figure 6 caption: chunks are staged incrementally and the AllReduce
//     owner reduces its partition while the other ranks gather reduced chunks;
//   - Figure 10 caption: Purlin-ZS omits staging.
#include "purlin.h"
#include "snac.h"

#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cstring>
#include <map>
#include <memory>
#include <new>
#include <string>
#include <unordered_map>
#include <utility>
#include <vector>

using namespace purlin;

namespace {

constexpr uint64_t kDefaultTimeoutNs = 2000000000ull;
constexpr uint64_t kMinChunkBytes = 8 << 10;
constexpr uint64_t kMaxChunkBytes = 4 << 20;
constexpr uint64_t kTicketedChunkBytes = 256 << 10;
constexpr uint64_t kBulkAutoBytes = 64ull << 20;  // automatic bulk-ring datapath from this many bytes moved
constexpr int kItemsPerCta = 4;       // auto chunking aims at this many items per CTA
constexpr int kGuidedDiv = 4;         // guided chunking: each item moves remaining / (kGuidedDiv x grid) bytes
constexpr int kGuidedTailDiv = 16;    // ... down to a chunk of total / (kGuidedTailDiv x grid) bytes,
constexpr uint64_t kGuidedTailMin = 64 << 10;   // kept within [kGuidedTailMin, kGuidedTailMax]
constexpr uint64_t kGuidedTailMax = 256 << 10;
// ... and, counted in bytes moved (read plus written), no larger than the
// greater of these: so that an item of eight sources or destinations ends
// the list with about 128 KiB moved, not 576 KiB (on GB300 the last items of
// a ReduceScatterV of 128 MiB per rank took 29 us each on one CTA).
constexpr uint64_t kGuidedTailMovedMin = 256 << 10;
constexpr int kGuidedTailMovedDiv = 16;
// Up to this many bytes moved, guided items start at remaining / (2 x grid)
// instead of remaining / (kGuidedDiv x grid): fewer items, each paying the
// fixed cost of a work item once (measured on GB300 at 64-128 MiB per rank:
// AllGatherV 0.71 -> 0.75, ReduceScatterV 0.77 -> 0.84, AllToAllV 0.82 ->
// 0.85 of the roofline; from 256 MiB per rank the finer start wins).
constexpr uint64_t kGuidedCoarseMoved = 1536ull << 20;
constexpr uint64_t kGuidedRowsTailFloor = 128 << 10;  // see cut_guided_rows
constexpr uint64_t kOneItemBytes = 256 << 10;   // up to this many bytes per CTA: one item per CTA
// ... and for plans of one-to-one transfers (the AllToAll shape; measured: the
// AllToAllV of 16 MiB per rank, 431 KB per CTA, 63.3 us guided, 54.5 us with
// chunks of 512 KiB; at 64 MiB and more the guided chunks stay best)
constexpr uint64_t kOneItemBytesOneToOne = 512 << 10;
// ... up to 2 MiB when those transfers are not all 16-byte aligned (the
// AllToAllV, realigned by the spliced copy kernel; measured on GB300: 32 MiB
// per rank 0.76 -> 0.80 of the roofline, 64 MiB 0.86 -> 0.87, 128 MiB and
// more unchanged; the aligned AllToAll lost with it, 0.88 -> 0.81 at 32 MiB)
constexpr uint64_t kOneItemBytesOneToOneMisaligned = 2 << 20;
// ... and for the ReduceScatter shape between regions not all 16-byte aligned
// (the ReduceScatterV), whose realigning reduction runs best in one item per
// CTA (measured on GB300, Zipf lengths, R = 8 bf16, guided against one item
// per CTA: 128 MiB per rank 0.84 -> 0.92-0.94 of the roofline, 256 MiB
// 0.89 -> 0.94-0.97; with 2 MiB the 512 MiB point lost 0.953 -> 0.945)
constexpr uint64_t kOneItemBytesScatterMisaligned = 1 << 20;
constexpr uint64_t kChunkGrain = 256;           // automatic chunk sizes are multiples of this many bytes
constexpr uint64_t kBulkItemBytes = 512 << 10;  // bytes (read + written) of an automatic bulk-ring item
constexpr uint64_t kBulkChunkMin = 64 << 10;    // ... whose chunk stays within these
constexpr uint64_t kBulkChunkMax = 256 << 10;
// Inline-parameter plans (automatic): those whose every transfer reduces
// several sources into one destination (the ReduceScatter shape, faster in
// the inline kernel at every size measured, 1 KiB to 1 GiB), and others that
// move at most this many bytes (measured crossovers on GB300, R = 8 bf16:
// AllGather between 32 and 64 MiB per rank, 288 and 576 MiB moved; AllReduce
// near 16 MiB per rank, 256 MiB moved; beyond them the persistent kernel's
// bulk ring and pipelined items are faster).
constexpr uint64_t kInlineAutoMoved = 320ull << 20;
// Inline items over regions not all 16-byte aligned: at most this many body
// vectors, which the kernel's realigning loop moves: eight per thread for a
// copy (with four, an AllToAllV of 1 MiB per rank needed more than 152 items
// and ran 8.6 us on the persistent kernel; 4.9 us inline), two for a
// reduction (its loop holds one vector of 8 sources at a time; with four a
// ReduceScatterV of 4 MiB per rank ran 12.0 us against the persistent
// kernel's 10.5).
constexpr uint64_t kInlineMisalignedCopyVectors = 8 * kInlineThreads;
constexpr uint64_t kInlineMisalignedReduceVectors = 2 * kInlineThreads;
// A copy into one destination stores a vector once: twice the vectors.
constexpr uint64_t kInlineMisalignedOneDstVectors = 16 * kInlineThreads;

uint64_t misaligned_cap(bool reduction, size_t ndst)
{
    return reduction ? kInlineMisalignedReduceVectors : ndst == 1 ? kInlineMisalignedOneDstVectors
                                                                  : kInlineMisalignedCopyVectors;
}
// CTAs per SM of the SNAC kernels for aligned plans that copy, for aligned
// plans that only reduce, and for other plans.
struct Occupancy {
    int aligned = kCtasPerSmAligned;
    int aligned_reduce = kCtasPerSmAlignedReduce;
    int spliced = kCtasPerSmSpliced;
};
constexpr size_t kMaxCachedPlans = 1024;
constexpr uint32_t kMaxUsesPerLaunch = (1u << 24) - 2;

uint64_t elem_size(pl_dtype dt)
{
    switch (dt) {
    case PL_BF16:
    case PL_FP16:
        return 2;
    case PL_FP8:
        return 1;
    default:
        return 4;
    }
}

// PL_OK for a known op and dtype the datapath can run; one-byte elements are
// moved, never reduced.
pl_status check_op_dtype(pl_op op, pl_dtype dt)
{
    if ((op != PL_COPY && op != PL_SUM && op != PL_MAX) || dt < PL_BF16 || dt > PL_FP8)
        return PL_ERR_INVALID;
    if (dt == PL_FP8 && op != PL_COPY)
        return PL_ERR_UNSUPPORTED;
    return PL_OK;
}

}  // namespace

// ------------------------------------------------------------------ layouts

struct pl_layout {
    uint64_t id = 0;             // unique per created layout (layouts are immutable)
    int R = 0;
    std::vector<int> first;      // R + 1 prefix counts into parts
    std::vector<pl_part> parts;  // contiguous regions normalised to rows = 1
};

namespace {

bool mul_overflows(uint64_t a, uint64_t b) { return a != 0 && b > UINT64_MAX / a; }

// Last element index + 1 of a region.
uint64_t region_extent(const pl_part& p)
{
    if (p.len == 0)
        return p.offset;
    return p.offset + (p.rows - 1) * p.row_stride + p.len;
}

uint64_t region_count(const pl_part& p) { return p.rows * p.len; }

pl_status make_layout(pl_layout** out, int R, const std::vector<int>& counts, const std::vector<pl_part>& parts)
{
    if (!out || R < 1 || R > kMaxRanks || (int)counts.size() != R)
        return PL_ERR_INVALID;
    std::unique_ptr<pl_layout> L(new (std::nothrow) pl_layout);
    if (!L)
        return PL_ERR_NOMEM;
    static std::atomic<uint64_t> next_id{1};
    L->id = next_id.fetch_add(1);
    L->R = R;
    L->first.assign(R + 1, 0);
    size_t total = 0;
    for (int r = 0; r < R; ++r) {
        if (counts[r] < 0)
            return PL_ERR_INVALID;
        total += (size_t)counts[r];
        L->first[r + 1] = (int)total;
    }
    if (total != parts.size())
        return PL_ERR_INVALID;
    L->parts.reserve(total);
    for (pl_part p : parts) {
        if (p.rows == 0)
            return PL_ERR_INVALID;
        if (p.rows > 1 && p.row_stride < p.len)
            return PL_ERR_INVALID;
        if (mul_overflows(p.rows, p.len) || p.rows * p.len > (1ull << 56))
            return PL_ERR_INVALID;
        if (p.rows > 1 && (mul_overflows(p.rows - 1, p.row_stride) || (p.rows - 1) * p.row_stride > (1ull << 58)))
            return PL_ERR_INVALID;
        if (p.offset > (1ull << 58))
            return PL_ERR_INVALID;
        // A region whose rows touch end to end is contiguous: one row of rows*len.
        if (p.rows == 1 || p.row_stride == p.len) {
            p.len = p.rows * p.len;
            p.rows = 1;
            p.row_stride = p.len;
        }
        L->parts.push_back(p);
    }
    *out = L.release();
    return PL_OK;
}

}  // namespace

extern "C" {

PL_API int pl_abi_version(void) { return PL_ABI_VERSION; }

PL_API const char* pl_status_str(pl_status s)
{
    switch (s) {
    case PL_OK: return "ok";
    case PL_ERR_INVALID: return "invalid argument";
    case PL_ERR_LAYOUT: return "the layout pair does not name a valid collective for these buffers";
    case PL_ERR_ALIAS: return "an output overlaps another output or an input it may not alias";
    case PL_ERR_NOMEM: return "out of device memory, or scratch ring too small for the staged path";
    case PL_ERR_CUDA: return "a CUDA call failed";
    case PL_ERR_TIMEOUT: return "a bounded device wait expired";
    case PL_ERR_UNSUPPORTED: return "layout pair not supported by this datapath";
    default: return "unknown status";
    }
}

PL_API void pl_policy_default(pl_policy* pol)
{
    if (!pol)
        return;
    std::memset(pol, 0, sizeof *pol);
    pol->debug_drop_notify = -1;
}

PL_API pl_status pl_layout_create(pl_layout** layout, int R, const int* nparts, const pl_part* parts)
{
    if (!layout || !nparts || R < 1 || R > kMaxRanks)
        return PL_ERR_INVALID;
    std::vector<int> counts(nparts, nparts + R);
    size_t total = 0;
    for (int c : counts) {
        if (c < 0)
            return PL_ERR_INVALID;
        total += (size_t)c;
    }
    if (total && !parts)
        return PL_ERR_INVALID;
    std::vector<pl_part> v(parts, parts + total);
    return make_layout(layout, R, counts, v);
}

PL_API pl_status pl_layout_destroy(pl_layout* layout)
{
    delete layout;
    return PL_OK;
}

PL_API pl_status pl_layout_info(const pl_layout* layout, int* R, int* total_parts)
{
    if (!layout)
        return PL_ERR_INVALID;
    if (R)
        *R = layout->R;
    if (total_parts)
        *total_parts = (int)layout->parts.size();
    return PL_OK;
}

PL_API pl_status pl_layout_rank_owned(pl_layout** layout, int R, const uint64_t* lens)
{
    if (!lens || R < 1 || R > kMaxRanks)
        return PL_ERR_INVALID;
    std::vector<int> counts(R, 1);
    std::vector<pl_part> parts;
    for (int k = 0; k < R; ++k)
        parts.push_back(pl_part{(uint64_t)k, 0, lens[k], 1, lens[k]});
    return make_layout(layout, R, counts, parts);
}

PL_API pl_status pl_layout_partitioned(pl_layout** layout, int R, const uint64_t* lens)
{
    if (!lens || R < 1 || R > kMaxRanks)
        return PL_ERR_INVALID;
    std::vector<int> counts(R, R);
    std::vector<pl_part> parts;
    for (int r = 0; r < R; ++r) {
        uint64_t o = 0;
        for (int k = 0; k < R; ++k) {
            parts.push_back(pl_part{(uint64_t)k, o, lens[k], 1, lens[k]});
            o += lens[k];
        }
    }
    return make_layout(layout, R, counts, parts);
}

PL_API pl_status pl_layout_rank_owned_inplace(pl_layout** layout, int R, const uint64_t* lens)
{
    if (!lens || R < 1 || R > kMaxRanks)
        return PL_ERR_INVALID;
    std::vector<int> counts(R, 1);
    std::vector<pl_part> parts;
    uint64_t o = 0;
    for (int k = 0; k < R; ++k) {
        parts.push_back(pl_part{(uint64_t)k, o, lens[k], 1, lens[k]});
        o += lens[k];
    }
    return make_layout(layout, R, counts, parts);
}

PL_API pl_status pl_layout_alltoall_in(pl_layout** layout, int R, const uint64_t* m)
{
    if (!m || R < 1 || R > kMaxRanks)
        return PL_ERR_INVALID;
    std::vector<int> counts(R, R);
    std::vector<pl_part> parts;
    for (int r = 0; r < R; ++r) {
        uint64_t o = 0;
        for (int j = 0; j < R; ++j) {
            uint64_t n = m[(size_t)r * R + j];
            parts.push_back(pl_part{(uint64_t)r * R + j, o, n, 1, n});
            o += n;
        }
    }
    return make_layout(layout, R, counts, parts);
}

PL_API pl_status pl_layout_alltoall_out(pl_layout** layout, int R, const uint64_t* m)
{
    if (!m || R < 1 || R > kMaxRanks)
        return PL_ERR_INVALID;
    std::vector<int> counts(R, R);
    std::vector<pl_part> parts;
    for (int j = 0; j < R; ++j) {
        uint64_t o = 0;
        for (int r = 0; r < R; ++r) {
            uint64_t n = m[(size_t)r * R + j];
            parts.push_back(pl_part{(uint64_t)r * R + j, o, n, 1, n});
            o += n;
        }
    }
    return make_layout(layout, R, counts, parts);
}

PL_API pl_status pl_layout_ulysses_in(pl_layout** layout, int R, uint64_t S, uint64_t H, uint64_t D)
{
    if (R < 1 || R > kMaxRanks || H % (uint64_t)R)
        return PL_ERR_INVALID;
    uint64_t hs = H / (uint64_t)R;
    std::vector<int> counts(R, R);
    std::vector<pl_part> parts;
    for (int r = 0; r < R; ++r)
        for (int j = 0; j < R; ++j)
            parts.push_back(pl_part{(uint64_t)r * R + j, (uint64_t)j * hs * D, hs * D, S ? S : 1, H * D});
    if (S == 0)
        for (auto& p : parts)
            p.len = 0;
    return make_layout(layout, R, counts, parts);
}

PL_API pl_status pl_layout_ulysses_out(pl_layout** layout, int R, uint64_t S, uint64_t H, uint64_t D)
{
    if (R < 1 || R > kMaxRanks || H % (uint64_t)R)
        return PL_ERR_INVALID;
    uint64_t blk = S * (H / (uint64_t)R) * D;
    std::vector<int> counts(R, R);
    std::vector<pl_part> parts;
    for (int j = 0; j < R; ++j)
        for (int r = 0; r < R; ++r)
            parts.push_back(pl_part{(uint64_t)r * R + j, (uint64_t)r * blk, blk, 1, blk});
    return make_layout(layout, R, counts, parts);
}

}  // extern "C"

// --------------------------------------------------------------- derivation

namespace {

struct Region {
    int space;  // PL_SPACE_IN / PL_SPACE_OUT
    int rank;
    uint64_t offset, rows, cols, stride;
};

// All regions of one name: the transfer the name asks for.
struct Transfer {
    uint64_t name;
    std::vector<Region> srcs;  // rank order
    std::vector<Region> dsts;  // rank order
    uint64_t count;
};

struct Chunk {
    uint64_t row0, nrows, col0, ncols;
};

struct ResolvedPolicy {
    int path;       // PL_PATH_ZS / PL_PATH_STAGED
    int ar_form;    // PL_AR_FUSED / PL_AR_COMPOSED / PL_AR_NOTIFIED
    int datapath;   // PL_ATOM_VECTOR / PL_ATOM_BULK / PL_ATOM_INLINE
    bool datapath_auto;
    bool stages_auto;
    int ctas;       // 0 = auto
    int stages;
    uint64_t chunk_bytes;
    uint64_t timeout_ns;
    int64_t drop_notify;
};

pl_status resolve_policy(const pl_policy* p, ResolvedPolicy& rp)
{
    pl_policy d;
    pl_policy_default(&d);
    if (!p)
        p = &d;
    if (p->path < PL_PATH_AUTO || p->path > PL_PATH_STAGED)
        return PL_ERR_INVALID;
    if (p->allreduce_form < PL_AR_AUTO || p->allreduce_form > PL_AR_NOTIFIED)
        return PL_ERR_INVALID;
    if (p->datapath < PL_ATOM_AUTO || p->datapath > PL_ATOM_INLINE)
        return PL_ERR_INVALID;
    if (p->ctas < 0 || p->stages < 0 || p->stages > kBulkMaxStages)
        return PL_ERR_INVALID;
    rp.path = p->path == PL_PATH_AUTO ? PL_PATH_ZS : p->path;
    rp.ar_form = p->allreduce_form == PL_AR_AUTO ? PL_AR_FUSED : p->allreduce_form;
    rp.datapath = p->datapath == PL_ATOM_AUTO ? PL_ATOM_VECTOR : p->datapath;
    rp.datapath_auto = p->datapath == PL_ATOM_AUTO;
    rp.stages_auto = p->stages == 0;
    rp.ctas = p->ctas;
    rp.stages = p->stages ? p->stages : 4;
    // Work items address columns with 32-bit counts: keep chunks well below 2^32 elements.
    rp.chunk_bytes = p->chunk_bytes ? std::min<uint64_t>(std::max<uint64_t>(p->chunk_bytes, 256), 1ull << 30) : 0;
    rp.timeout_ns = p->poll_timeout_ns ? p->poll_timeout_ns : kDefaultTimeoutNs;
    rp.drop_notify = p->debug_drop_notify;
    return PL_OK;
}

struct HostPlan {
    int R = 0;
    pl_dtype dtype = PL_BF16;
    std::vector<Item> items;
    std::vector<Ref> refs;
    std::vector<Sync> syncs;
    uint32_t nflags = 0;
    int lag = 0;          // chunk rows between producers and their consumers in claim order
    int ops = 0;          // kOpsCopy | kOpsReduce, plus kOpsWide / kOpsMax
    int all_aligned = 0;  // every reference's byte offset and row stride is a multiple of 16
    int refs_per_item = 0;  // n > 0: every item has n references, item i's at [i * n, i * n + n)
    bool inline_form = false;  // one-row items that the inline-parameter kernel runs, one per CTA
    bool inline_any_alignment = false;  // ... over buffers at any alignment (small items)
    bool flagged_reduction = false;     // a list with flags that reduces: the two-CTA kernels
    pl_plan_stats stats{};
};

pl_status collect_transfers(const pl_layout& in, const pl_layout& out, pl_op op, int R,
                            std::vector<Transfer>& ts)
{
    std::unordered_map<uint64_t, std::vector<std::pair<int, int>>> by_name;
    for (int r = 0; r < R; ++r)
        for (int i = in.first[r]; i < in.first[r + 1]; ++i)
            by_name[in.parts[i].name].push_back({r, i});
    std::unordered_map<uint64_t, size_t> index;
    for (int r = 0; r < R; ++r) {
        for (int i = out.first[r]; i < out.first[r + 1]; ++i) {
            const pl_part& p = out.parts[i];
            auto it = index.find(p.name);
            if (it == index.end()) {
                index[p.name] = ts.size();
                Transfer t;
                t.name = p.name;
                t.count = region_count(p);
                ts.push_back(t);
                it = index.find(p.name);
            }
            Transfer& t = ts[it->second];
            if (region_count(p) != t.count)
                return PL_ERR_LAYOUT;
            t.dsts.push_back(Region{PL_SPACE_OUT, r, p.offset, p.rows, p.len, p.row_stride});
        }
    }
    for (Transfer& t : ts) {
        auto it = by_name.find(t.name);
        if (it == by_name.end())
            return PL_ERR_LAYOUT;
        const auto& srcs = it->second;
        if (op == PL_COPY) {
            if (srcs.size() != 1)
                return PL_ERR_LAYOUT;
        } else {
            if ((int)srcs.size() != R)
                return PL_ERR_LAYOUT;
            for (int r = 0; r < R; ++r)
                if (srcs[r].first != r)  // collected in rank order: one per rank means srcs[r] is rank r
                    return PL_ERR_LAYOUT;
        }
        for (auto [r, i] : srcs) {
            const pl_part& p = in.parts[i];
            if (region_count(p) != t.count)
                return PL_ERR_LAYOUT;
            t.srcs.push_back(Region{PL_SPACE_IN, r, p.offset, p.rows, p.len, p.row_stride});
        }
    }
    return PL_OK;
}

// Gives every region of a transfer the same row structure: strided regions
// keep theirs (they must agree on the row length), contiguous ones are cut
// into rows of that length.
pl_status normalise_rows(Transfer& t)
{
    uint64_t L = 0;
    auto visit = [&](const Region& g) -> bool {
        if (g.rows > 1) {
            if (L == 0)
                L = g.cols;
            else if (g.cols != L)
                return false;
        }
        return true;
    };
    for (auto& g : t.srcs)
        if (!visit(g))
            return PL_ERR_UNSUPPORTED;
    for (auto& g : t.dsts)
        if (!visit(g))
            return PL_ERR_UNSUPPORTED;
    auto fix = [&](Region& g) {
        if (L == 0 || t.count == 0) {
            g.rows = 1;
            g.cols = t.count;
            g.stride = t.count;
        } else if (g.rows == 1) {
            g.rows = t.count / L;
            g.cols = L;
            g.stride = L;
        }
    };
    for (auto& g : t.srcs)
        fix(g);
    for (auto& g : t.dsts)
        fix(g);
    return PL_OK;
}

// Chunks of a transfer.  One-row transfers are cut at element boundaries that
// keep the first destination 16-byte aligned after its first chunk; multi-row
// transfers are cut into row ranges, or row pieces when a row exceeds a chunk.
std::vector<Chunk> make_chunks(const Transfer& t, uint64_t chunk_elems, uint64_t vec_elems)
{
    std::vector<Chunk> out;
    if (t.count == 0)
        return out;
    const Region& d0 = t.dsts[0];
    auto cut_row = [&](uint64_t row, uint64_t cols, uint64_t dst_off) {
        uint64_t head = (vec_elems - dst_off % vec_elems) % vec_elems;
        uint64_t c0 = 0;
        while (c0 < cols) {
            uint64_t n = chunk_elems;
            if (c0 == 0)
                n += head;
            n = std::min(n, cols - c0);
            out.push_back(Chunk{row, 1, c0, n});
            c0 += n;
        }
    };
    if (d0.rows == 1) {
        cut_row(0, d0.cols, d0.offset);
    } else if (d0.cols >= chunk_elems) {
        for (uint64_t r = 0; r < d0.rows; ++r)
            cut_row(r, d0.cols, d0.offset + r * d0.stride);
    } else {
        uint64_t per = std::max<uint64_t>(1, chunk_elems / d0.cols);
        for (uint64_t r = 0; r < d0.rows; r += per)
            out.push_back(Chunk{r, std::min(per, d0.rows - r), 0, d0.cols});
    }
    return out;
}

// Where the next chunk of a transfer starts.
struct Cursor {
    uint64_t row = 0, col = 0;
};

// The next chunk of about `target` elements of transfer t from `cu` (the
// same cuts as make_chunks, with a size that may change from chunk to chunk).
Chunk next_chunk(const Transfer& t, Cursor& cu, uint64_t target, uint64_t vec_elems)
{
    const Region& d0 = t.dsts[0];
    const uint64_t cols = d0.cols;
    if (d0.rows > 1 && cu.col == 0 && cols <= target) {
        const uint64_t per = std::min<uint64_t>(std::max<uint64_t>(1, target / cols), d0.rows - cu.row);
        Chunk c{cu.row, per, 0, cols};
        cu.row += per;
        return c;
    }
    const uint64_t dst_off = d0.offset + cu.row * d0.stride;
    uint64_t n = target;
    if (cu.col == 0)
        n += (vec_elems - dst_off % vec_elems) % vec_elems;
    n = std::min(n, cols - cu.col);
    Chunk c{cu.row, 1, cu.col, n};
    cu.col += n;
    if (cu.col == cols) {
        cu.col = 0;
        ++cu.row;
    }
    return c;
}

class Builder {
public:
    Builder(HostPlan& hp, int R) : hp_(hp), R_(R) {}

    Ref region(const Region& g, const Chunk& c) const
    {
        Ref f{};
        f.buf = (uint32_t)(g.space == PL_SPACE_IN ? g.rank : R_ + g.rank);
        f.offset = g.offset + c.row0 * g.stride + c.col0;
        f.stride = g.stride;
        return f;
    }

    Ref slot(uint64_t s, uint64_t slot_elems, const Chunk& c) const
    {
        Ref f{};
        f.buf = (uint32_t)(2 * R_);
        f.offset = s * slot_elems;
        f.stride = c.ncols;
        return f;
    }

    struct Pending {
        std::vector<Ref> src, dst;
        std::vector<Sync> waits, posts;
    };

    void emit(const Pending& p, ItemKind kind, pl_op op, const Chunk& c)
    {
        Item it{};
        it.kind = kind;
        it.op = (uint8_t)(op != PL_COPY && p.src.size() > 1 ? (op == PL_MAX ? 2 : 1) : 0);
        it.nsrc = (uint16_t)p.src.size();
        it.ndst = (uint16_t)p.dst.size();
        it.rows = (uint32_t)c.nrows;
        it.cols = c.ncols;
        it.ref = (uint32_t)hp_.refs.size();
        hp_.refs.insert(hp_.refs.end(), p.src.begin(), p.src.end());
        hp_.refs.insert(hp_.refs.end(), p.dst.begin(), p.dst.end());
        it.sync = (uint32_t)hp_.syncs.size();
        it.nwait = (uint16_t)p.waits.size();
        it.npost = (uint16_t)p.posts.size();
        hp_.syncs.insert(hp_.syncs.end(), p.waits.begin(), p.waits.end());
        hp_.syncs.insert(hp_.syncs.end(), p.posts.begin(), p.posts.end());
        hp_.items.push_back(it);
    }

private:
    HostPlan& hp_;
    int R_;
};

Sync mk_sync(SyncType t, uint32_t flag, uint32_t use, uint32_t count = 0)
{
    Sync s{};
    s.type = t;
    s.flag = flag;
    s.use = use;
    s.count = count;
    return s;
}

// Checks that every wait of item j is satisfied by items with smaller
// indices, so that CTAs claiming items in index order always progress.
bool waits_precede(const HostPlan& hp)
{
    std::map<std::pair<uint32_t, uint32_t>, uint64_t> notified;            // (flag, use) -> item
    std::map<std::pair<uint32_t, uint32_t>, std::pair<uint64_t, uint32_t>> credits;  // -> (last item, n)
    std::map<std::pair<uint32_t, uint32_t>, uint32_t> credit_need;
    for (uint64_t j = 0; j < hp.items.size(); ++j) {
        const Item& it = hp.items[j];
        for (uint32_t k = it.nwait; k < (uint32_t)it.nwait + it.npost; ++k) {
            const Sync& s = hp.syncs[it.sync + k];
            auto key = std::make_pair(s.flag, s.use);
            if (s.type == kNotify)
                notified[key] = j;
            else if (s.type == kCredit) {
                auto& c = credits[key];
                c.first = j;
                c.second += 1;
                credit_need[key] = s.count;
            }
        }
    }
    for (uint64_t j = 0; j < hp.items.size(); ++j) {
        const Item& it = hp.items[j];
        for (uint32_t k = 0; k < it.nwait; ++k) {
            const Sync& s = hp.syncs[it.sync + k];
            auto key = std::make_pair(s.flag, s.use);
            if (s.type == kWaitFull) {
                auto f = notified.find(key);
                if (f == notified.end() || f->second >= j)
                    return false;
            } else {
                auto c = credits.find(key);
                if (c == credits.end() || c->second.first >= j || c->second.second != credit_need[key])
                    return false;
            }
        }
    }
    return true;
}

// Codesign policy for the datapath of the persistent kernel: large copy-only
// plans stream through the bulk-copy ring (one shared-memory read per chunk,
// one bulk store per destination) when their regions are 16-byte aligned, or
// when they write at least twice what they read (a broadcast, the
// AllGather(V) shape: misaligned sources are then realigned in shared memory
// between the bulk load and the bulk stores); everything else uses the
// vector datapath.  `hp.stats` holds the plan's bytes.
bool launch_bulk(const HostPlan& hp, const ResolvedPolicy& pol)
{
    if (pol.datapath == PL_ATOM_BULK)
        return true;
    const pl_plan_stats& ps = hp.stats;
    return pol.datapath_auto && hp.ops == kOpsCopy && (hp.all_aligned || ps.bytes_written >= 2 * ps.bytes_read) &&
           ps.bytes_read + ps.bytes_written >= kBulkAutoBytes;
}

// ---------------------------------------------------------------------------
// The derivation in three parts (Figure 1 caption: codesign policies tune the
// execution without changing the collective):
//   analyse        the layout pair -> its transfers and the facts about them;
//   choose_policy  those facts + the caller's policy -> chunk rule, chunk and
//                  slot sizes, grid, staged or zero-staging;
//   emit_items     transfers + policy -> work items, flags and ring slots in
//                  claim order (the SNAC steps of the abstract and Figure 6).
// ---------------------------------------------------------------------------

// What a layout pair asks for, before any policy.
struct PlanShape {
    std::vector<Transfer> ts;
    uint64_t S = 0;                   // element bytes
    uint64_t E = 0;                   // elements per 16-byte vector
    uint64_t total_bytes = 0;         // bytes of every transfer's region, counted once
    uint64_t moved = 0, rd = 0, wr = 0;  // zero-staging bytes read + written, read, written
    uint64_t fanout = 2;              // most references (sources + destinations) of one transfer
    bool copy_like = true;            // COPY, or every transfer has one source
    bool one_row = true;              // every region is one row
    bool all_aligned_regions = true;  // every region offset is a multiple of 16 bytes
    bool regions_aligned = true;      // ... and so is every multi-row region's row stride
    bool multi_dst_sum = false;       // a reduction with several destinations (the AllReduce shape)
    bool rs_shape = false;            // every transfer reduces several sources into one destination
    bool equal = true;                // one-row transfers of one size and fan-out
    bool one_to_one = true;           // every transfer has one source and one destination
};

pl_status analyse(const pl_layout& in, const pl_layout& out, pl_op op, pl_dtype dt, int R, PlanShape& sh)
{
    sh = PlanShape{};
    sh.S = elem_size(dt);
    sh.E = 16 / sh.S;
    pl_status st = collect_transfers(in, out, op, R, sh.ts);
    if (st != PL_OK)
        return st;
    const uint64_t S = sh.S;
    sh.rs_shape = op != PL_COPY;
    for (Transfer& t : sh.ts) {
        if ((st = normalise_rows(t)) != PL_OK)
            return st;
        sh.total_bytes += t.count * S;
        sh.copy_like &= op == PL_COPY || t.srcs.size() == 1;
        sh.moved += t.count * S * (t.srcs.size() + t.dsts.size());
        sh.rd += t.count * S * t.srcs.size();
        sh.wr += t.count * S * t.dsts.size();
        sh.fanout = std::max<uint64_t>(sh.fanout, t.srcs.size() + t.dsts.size());
        for (const auto* side : {&t.srcs, &t.dsts})
            for (const Region& g : *side) {
                sh.one_row &= g.rows == 1;
                sh.all_aligned_regions &= (g.offset * S) % 16 == 0;
                sh.regions_aligned &= (g.offset * S) % 16 == 0 && (g.rows == 1 || (g.stride * S) % 16 == 0);
            }
        sh.multi_dst_sum |= op != PL_COPY && t.srcs.size() > 1 && t.dsts.size() > 1;
        sh.rs_shape &= t.srcs.size() > 1 && t.dsts.size() == 1;
        sh.one_to_one &= t.srcs.size() == 1 && t.dsts.size() == 1;
    }
    for (const Transfer& t : sh.ts)
        sh.equal &= t.count == sh.ts[0].count && t.srcs.size() == sh.ts[0].srcs.size() &&
                    t.dsts.size() == sh.ts[0].dsts.size() && t.dsts[0].rows == 1;
    return PL_OK;
}

// How the transfers are cut into work items (the automatic rules apply to
// zero-staging lists whose items never wait on one another).
enum class ChunkRule {
    kFixed,   // equal chunks of chunk_elems (forced chunk size, staged and composed lists)
    kInline,  // each transfer's share of the inline kernel's items, one item per CTA
    kPerCta,  // small messages: each transfer's share of the grid, about one item per CTA
    kEqual,   // near-equal items, a few per CTA
    kGuided,  // guided self-scheduling: items shrink toward the end of the list
    kGuidedRows,  // guided sizes per chunk row, every transfer cut alike (lists with flags)
};

// The codesign policy of one plan.
struct PlanPolicy {
    bool staged = false;             // Stage -> Notify -> Consume through the scratch ring
    bool ticketed = false;           // items wait on flags: claimed in index order
    bool flagged_reduction = false;  // a list with flags that reduces: the two-CTA kernels
    bool composed = false;           // reductions with several destinations: the Figure 6 form
    bool vector_compose = false;     // ... zero-staging, at the grain of one vector (kCompose items, no flags)
    bool bulk = false;               // copy items of one-row regions go through the bulk ring
    int full_grid = 1;               // persistent grid for the plan's kernel class
    ChunkRule rule = ChunkRule::kFixed;
    uint64_t chunk_elems = 0;        // kFixed chunks (and the plan's reported chunk size)
    uint64_t slot_elems = 0;         // one chunk plus a vector of alignment head
    uint64_t slots_per_rank = 0;     // staged: slots in each rank's ring
    uint64_t grain = 0;              // automatic chunk sizes are multiples of this many elements
    std::vector<uint64_t> target;    // kInline / kPerCta / kEqual: elements per item of each transfer
};

// kInline: the inline-parameter form (the whole plan in the launch's
// parameters, one item per CTA, no metadata loads) for zero-staging one-row
// moves whose items and references fit the parameter block, every transfer's
// destinations at one offset mod 16 bytes.  Each transfer gets its share of
// kInlineMaxItems items by bytes moved, in multiples of the grain.  Regions
// not all 16-byte aligned: items of at most kInlineMisalignedCopyVectors
// (copies) or kInlineMisalignedReduceVectors (reductions) vectors (the
// kernel's fastest loop, for larger items, wants aligned references).
// Automatically: the ReduceScatter shape between aligned regions, or at most
// kInlineAutoMoved bytes moved.  Returns whether the plan takes the form, with
// the per-transfer item sizes in `target`.
bool inline_targets(const PlanShape& sh, pl_op op, uint64_t grain, std::vector<uint64_t>& target)
{
    const uint64_t S = sh.S, E = sh.E;
    bool fits = true;
    uint64_t nitems = 0, nptrs = 0;
    target.assign(sh.ts.size(), 0);
    for (size_t i = 0; fits && i < sh.ts.size(); ++i) {
        const Transfer& t = sh.ts[i];
        for (const auto* side : {&t.srcs, &t.dsts})
            for (const Region& g : *side)
                fits &= g.rows == 1;
        for (const Region& g : t.dsts)
            fits &= (g.offset * S) % 16 == (t.dsts[0].offset * S) % 16;
        fits &= t.dsts.size() <= (size_t)kMaxRanks && t.srcs.size() <= (size_t)kMaxRanks;
        if (!fits || t.count == 0)
            continue;
        const uint64_t nref = t.srcs.size() + t.dsts.size();
        const uint64_t share = std::max<uint64_t>(1, (uint64_t)kInlineMaxItems * (t.count * S * nref) / sh.moved);
        uint64_t tg = (t.count + share - 1) / share;
        tg = (tg + grain - 1) / grain * grain;
        if (!sh.regions_aligned)
            tg = std::min<uint64_t>(tg, misaligned_cap(op != PL_COPY && t.srcs.size() > 1, t.dsts.size()) * E);
        fits &= tg * t.dsts.size() <= (1ull << 31);  // the kernel's 32-bit (vector, destination) index
        target[i] = tg;
        const uint64_t n = (t.count + tg - 1) / tg;
        nitems += n;
        nptrs += n * nref;
    }
    return fits && nitems <= (uint64_t)kInlineMaxItems && nptrs <= (uint64_t)kInlineMaxPtrs;
}

// Per-transfer item sizes: each transfer cut into `share(i)` near-equal items
// in multiples of the grain, no smaller than `min_elems`.
template <class Share>
void share_targets(const PlanShape& sh, uint64_t grain, uint64_t min_elems, Share share, std::vector<uint64_t>& target)
{
    target.assign(sh.ts.size(), 0);
    for (size_t i = 0; i < sh.ts.size(); ++i) {
        if (sh.ts[i].count == 0)
            continue;
        const uint64_t n = share(sh.ts[i]);
        uint64_t tg = (sh.ts[i].count + n - 1) / n;
        target[i] = std::max(min_elems, (tg + grain - 1) / grain * grain);
    }
}

// The automatic chunk rule of a zero-staging list whose items never wait on
// one another.  A CTA moves its items one after another and each item starts
// with a memory round trip that nothing overlaps, so:
//  - small messages (at most kOneItemBytes per CTA; more for one-to-one
//    transfers and for misaligned ReduceScatters) get about one item per
//    CTA: each transfer is cut into its share of the grid;
//  - larger ones whose transfers all have one size and fan-out, and those
//    the bulk ring moves (aligned, or realigned in shared memory), are cut
//    into k near-equal items per CTA (k = kItemsPerCta, or enough to keep
//    chunks within the cap);
//  - the others are cut by guided self-scheduling: each next item moves about
//    remaining bytes / (kGuidedDiv x grid), so items shrink toward the end of
//    the list, and CTAs that claim them in order as they finish end within one
//    small item of each other, whatever the partition lengths.
// Sizes are multiples of kChunkGrain bytes, so chunks after the first of a
// row start as aligned as the row's aligned start.  (Strided transfers
// balance better guided: measured.)
void choose_auto_rule(const PlanShape& sh, pl_op op, const ResolvedPolicy& pol, PlanPolicy& pp)
{
    const uint64_t S = sh.S;
    const uint64_t grid = (uint64_t)pp.full_grid;
    const bool want_inline = pol.path == PL_PATH_ZS && pol.ctas == 0 && sh.moved > 0 && !pp.vector_compose &&
                             (pol.datapath == PL_ATOM_INLINE ||
                              (pol.datapath_auto && ((sh.rs_shape && sh.regions_aligned) || sh.moved <= kInlineAutoMoved)));
    if (want_inline && inline_targets(sh, op, pp.grain, pp.target)) {
        pp.rule = ChunkRule::kInline;
        return;
    }
    const uint64_t one_item = sh.one_to_one ? (sh.regions_aligned ? kOneItemBytesOneToOne : kOneItemBytesOneToOneMisaligned)
                              : sh.rs_shape && !sh.regions_aligned ? kOneItemBytesScatterMisaligned
                                                                   : kOneItemBytes;
    if (sh.total_bytes / grid <= one_item) {
        pp.rule = ChunkRule::kPerCta;
        const uint64_t min_elems = std::max(pp.grain, kMinChunkBytes / S / pp.grain * pp.grain);
        share_targets(sh, pp.grain, min_elems, [&](const Transfer& t) {
            return std::max<uint64_t>(1, grid * (t.count * S) / sh.total_bytes);
        }, pp.target);
        return;
    }
    if (sh.equal || pp.bulk) {
        // k items per CTA, each transfer cut into floor(its share of k x grid)
        // near-equal chunks: at most k items per CTA, none much larger than
        // total / (k x grid).  On the bulk ring an item moves about
        // kBulkItemBytes (measured on GB300: an AllGather at 1 GiB, one source
        // and eight destinations, best with 64 KiB chunks; the MoE AllToAll,
        // one and one, with 256 KiB; the Zipf AllGatherV, whose sources the
        // ring realigns, with 64 KiB chunks from 64 MiB per rank up: 0.81 ->
        // 0.87 of the roofline at 64 MiB, 0.82 -> 0.93 at 128 MiB, 0.94 ->
        // 0.98 at 1 GiB, against guided items).
        pp.rule = ChunkRule::kEqual;
        const uint64_t bulk_chunk = std::min(std::max(kBulkItemBytes / sh.fanout, kBulkChunkMin), kBulkChunkMax);
        const uint64_t cap = pp.bulk ? bulk_chunk : kMaxChunkBytes;
        const uint64_t per_cta = (sh.total_bytes + grid - 1) / grid;
        const uint64_t k = std::max<uint64_t>((per_cta + cap - 1) / cap, kItemsPerCta);
        const uint64_t items = k * grid;
        share_targets(sh, pp.grain, 0, [&](const Transfer& t) {
            return std::max<uint64_t>(1, (uint64_t)((double)items * (double)(t.count * S) / (double)sh.total_bytes));
        }, pp.target);
        return;
    }
    pp.rule = ChunkRule::kGuided;
}

pl_status choose_policy(const PlanShape& sh, pl_op op, int R, const ResolvedPolicy& pol, int num_sms,
                        Occupancy occ, uint64_t scratch_bytes, PlanPolicy& pp)
{
    const uint64_t S = sh.S, E = sh.E;
    pp = PlanPolicy{};
    // One-row copy plans the bulk ring will move: forced, or automatic for
    // plans moving at least kBulkAutoBytes whose regions are 16-byte aligned or
    // that write at least twice what they read (the rule of pl_collective).
    pp.bulk = (pol.datapath == PL_ATOM_BULK || pol.datapath_auto) && sh.copy_like && sh.one_row &&
              (pol.datapath == PL_ATOM_BULK ||
               (sh.moved >= kBulkAutoBytes && (sh.all_aligned_regions || sh.wr >= 2 * sh.rd)));
    pp.staged = pol.path == PL_PATH_STAGED;
    pp.composed = pol.ar_form == PL_AR_COMPOSED || pol.ar_form == PL_AR_NOTIFIED;
    // Figure 6 without flags, zero-staging (every name of a reduction has R
    // sources, so with several destinations every item reduces: the list
    // needs no copy path).
    pp.vector_compose = pol.ar_form == PL_AR_COMPOSED && !pp.staged && sh.multi_dst_sum;
    pp.ticketed = pp.staged || (sh.multi_dst_sum && pp.composed && !pp.vector_compose);
    // Lists with flags that reduce (staged, composed) run the two-CTA kernels
    // even when aligned: their waits leave the single CTA's warps idle
    // (measured at 1 GiB: staged AllReduce 7.0 -> 5.9 ms, staged ReduceScatter
    // 5.6 -> 4.9 ms, composed AllReduce 3.25 -> 3.18 ms; staged copies lose:
    // AllGather 2.5 -> 2.9 ms, so they keep one CTA).  Plans whose regions are
    // all 16-byte aligned run the aligned kernels, the others the spliced ones,
    // each with its own CTAs per SM.  (The bulk ring's shared memory holds one
    // CTA per SM, whatever the kernel.)
    pp.flagged_reduction = pp.ticketed && op != PL_COPY;
    // (every item of a reduction over R > 1 ranks reduces: the reduce-only kernels)
    const bool aligned_class = (sh.regions_aligned || pp.bulk) && !pp.flagged_reduction;
    const int per_sm = !aligned_class ? occ.spliced : op != PL_COPY && R > 1 ? occ.aligned_reduce : occ.aligned;
    pp.full_grid = std::max(1, num_sms) * std::max(1, per_sm);
    pp.grain = std::max<uint64_t>(E, kChunkGrain / S);

    uint64_t chunk_bytes = pol.chunk_bytes;
    if (chunk_bytes == 0) {
        chunk_bytes = sh.total_bytes / ((uint64_t)pp.full_grid * kItemsPerCta);
        chunk_bytes = std::min(std::max(chunk_bytes, kMinChunkBytes), kMaxChunkBytes);
    }
    chunk_bytes = std::max<uint64_t>(256, chunk_bytes / 256 * 256);
    // The staged path keeps chunks small, so that a ring of a given size holds
    // many rows of them (measured: the staged AllReduce does not gain from
    // larger chunks, the staged ReduceScatter loses).  The zero-staging
    // composed form takes the general rule (it gains from large chunks: at
    // 1 GiB, 256 KiB chunks ran at 0.68 of the roofline, 4 MiB at 0.79).
    if (pp.staged && pol.chunk_bytes == 0) {
        // The composed form re-stages every reduced chunk, one more item per
        // chunk, and gains from chunks twice as large (measured on GB300, the
        // staged composed AllReduce: 0.79 -> 0.83 of its own bytes at 128 MiB
        // per rank, 0.95 -> 0.99 at 1 GiB with 512 KiB chunks).
        const uint64_t f = pp.composed && sh.multi_dst_sum ? 2 : 1;
        chunk_bytes = std::min<uint64_t>(chunk_bytes * f, kTicketedChunkBytes * f);
        const uint64_t per_rank = scratch_bytes / (uint64_t)R;
        chunk_bytes = std::min(chunk_bytes, std::max<uint64_t>(256, per_rank / 4 / 256 * 256));
    }
    pp.chunk_elems = std::max<uint64_t>(E, chunk_bytes / S / E * E);
    // A slot holds one chunk; the first chunk of a row may carry up to one
    // vector more (the head that aligns the destination).
    pp.slot_elems = pp.chunk_elems + E;
    if (pp.staged) {
        // The ring of each rank holds at least 2 slots (a reducer re-stages
        // its result into its own ring while its inputs are still held).
        const uint64_t per_rank = scratch_bytes / (uint64_t)R;
        pp.slots_per_rank = per_rank / (pp.slot_elems * S);
        if (pp.slots_per_rank < 2)
            return PL_ERR_NOMEM;
        // A whole number of rows of one rank's stages, so that the stages a
        // rank makes in one row never wrap around its ring (they merge, below).
        std::vector<uint64_t> per_row(R, 0);
        for (const Transfer& t : sh.ts)
            for (const Region& g : t.srcs)
                ++per_row[g.rank];
        const uint64_t g = *std::max_element(per_row.begin(), per_row.end());
        if (g > 1 && pp.slots_per_rank >= 2 * g)
            pp.slots_per_rank = pp.slots_per_rank / g * g;
    }
    pp.rule = ChunkRule::kFixed;
    if (!pp.ticketed && pol.chunk_bytes == 0)
        choose_auto_rule(sh, op, pol, pp);
    else if (pp.ticketed && !pp.staged && pol.chunk_bytes == 0)
        pp.rule = ChunkRule::kGuidedRows;
    return PL_OK;
}

// The chunks of every transfer and the order in which they are emitted:
// (transfer, chunk) pairs, chunk c of every transfer before chunk c + 1,
// except under guided scheduling, which emits chunks as it cuts them.
struct Cuts {
    std::vector<std::vector<Chunk>> chunks;
    std::vector<std::pair<size_t, size_t>> order;
    size_t max_chunks = 0;
};

void cut_guided(const PlanShape& sh, const PlanPolicy& pp, Cuts& cu)
{
    const uint64_t S = sh.S, E = sh.E, grid = (uint64_t)pp.full_grid;
    auto round_grain = [&](uint64_t elems) { return std::max(pp.grain, elems / pp.grain * pp.grain); };
    std::vector<Cursor> cur(sh.ts.size());
    uint64_t rem_moved = 0;
    std::vector<uint64_t> rem(sh.ts.size()), w(sh.ts.size());
    for (size_t i = 0; i < sh.ts.size(); ++i) {
        rem[i] = sh.ts[i].count;
        w[i] = S * (sh.ts[i].srcs.size() + sh.ts[i].dsts.size());
        rem_moved += rem[i] * w[i];
    }
    const uint64_t tail_bytes =
        std::min(std::max(sh.total_bytes / (grid * kGuidedTailDiv), kGuidedTailMin), kGuidedTailMax);
    const uint64_t tail_moved = std::max(kGuidedTailMovedMin, sh.moved / (grid * kGuidedTailMovedDiv));
    const uint64_t div = sh.moved <= kGuidedCoarseMoved ? 2 : kGuidedDiv;
    const uint64_t max_elems = round_grain(kMaxChunkBytes / S);
    // transfers take turns
    for (size_t k = 0; rem_moved > 0; k = (k + 1) % sh.ts.size()) {
        if (rem[k] == 0)
            continue;
        const uint64_t min_elems = std::min(round_grain(tail_bytes / S), round_grain(tail_moved / w[k]));
        uint64_t target = rem_moved / (grid * div) / w[k];
        target = std::min(std::max(round_grain(target), min_elems), max_elems);
        const Chunk ch = next_chunk(sh.ts[k], cur[k], target, E);
        const uint64_t got = ch.nrows * ch.ncols;
        cu.chunks[k].push_back(ch);
        cu.order.push_back({k, cu.chunks[k].size() - 1});
        rem[k] -= got;
        rem_moved -= got * w[k];
    }
}

// kGuidedRows (the zero-staging composed AllReduce): chunk row c of every
// transfer has one size, the guided size of the row (the bytes all transfers
// still have to move / (kGuidedDiv x grid), within the guided tail and the
// chunk cap), so that rows keep their meaning for the lag between a row's
// producers and its consumers while the last rows are small: the grid ends
// within a small item of itself instead of a large one.  (Measured on GB300
// with equal chunks of total / (4 x grid): an AllReduce of 1 GiB per rank
// had its median CTA done 10% before its last.)
void cut_guided_rows(const PlanShape& sh, const PlanPolicy& pp, Cuts& cu)
{
    const uint64_t S = sh.S, E = sh.E, grid = (uint64_t)pp.full_grid;
    auto round_grain = [&](uint64_t elems) { return std::max(pp.grain, elems / pp.grain * pp.grain); };
    std::vector<Cursor> cur(sh.ts.size());
    std::vector<uint64_t> rem(sh.ts.size()), w(sh.ts.size());
    uint64_t rem_moved = 0;
    for (size_t i = 0; i < sh.ts.size(); ++i) {
        rem[i] = sh.ts[i].count;
        w[i] = S * (sh.ts[i].srcs.size() + sh.ts[i].dsts.size());
        rem_moved += rem[i] * w[i];
    }
    // The smallest rows: total / (kGuidedTailDiv x grid), from kMinChunkBytes (a
    // small message still gets several items per CTA) to kGuidedTailMax; and
    // at least total / (2 x grid) up to kGuidedRowsTailFloor, so that smaller
    // messages end in fewer, larger rows: each item of these lists waits on a
    // flag or posts one, and small items paid that cost too often (measured on
    // GB300, the notified AllReduce at 16 / 64 / 128 / 256 MiB / 1 GiB per
    // rank: 0.34 / 0.60 / 0.73 / 0.83 / 0.89 of the roofline with the plain
    // tail, 0.50 / 0.73 / 0.79 / 0.84 / 0.89 with this floor; a tail of
    // total / (2 x grid) up to 1 MiB cost the 1 GiB point 0.89 -> 0.86).
    const uint64_t tail_bytes =
        std::min(std::max({sh.total_bytes / (grid * kGuidedTailDiv),
                           std::min(sh.total_bytes / (grid * 2), kGuidedRowsTailFloor), kMinChunkBytes}),
                 kGuidedTailMax);
    const uint64_t min_elems = round_grain(tail_bytes / S);
    const uint64_t max_elems = round_grain(kMaxChunkBytes / S);
    while (rem_moved > 0) {
        const uint64_t row_moved = rem_moved;
        for (size_t i = 0; i < sh.ts.size(); ++i) {
            if (rem[i] == 0)
                continue;
            uint64_t target = row_moved / (grid * kGuidedDiv) / w[i];
            target = std::min(std::max(round_grain(target), min_elems), max_elems);
            const Chunk ch = next_chunk(sh.ts[i], cur[i], target, E);
            const uint64_t got = ch.nrows * ch.ncols;
            cu.chunks[i].push_back(ch);
            rem[i] -= got;
            rem_moved -= got * w[i];
        }
    }
}

// The last `m` chunks of one transfer (at most half of them) cut in two, in
// multiples of the grain: a list of equal items on the bulk ring then ends
// with about two grids of half-size items, so that the CTAs, which run at
// different rates, finish within half an item of each other instead of a
// whole one (measured on GB300, R = 8 bf16: AllGather 0.87 -> 0.89 of the
// roofline at 64 MiB per rank, 0.93 -> 0.95 at 128 MiB; AllToAll 0.94 ->
// 0.95 and 0.986 -> 0.996; MoE AllToAll 147 -> 145 us; cutting the last
// three grids, or into quarters, gained less).
void halve_last_chunks(std::vector<Chunk>& chunks, size_t m, uint64_t grain)
{
    m = std::min(m, chunks.size() / 2);
    std::vector<Chunk> tail(chunks.end() - (std::ptrdiff_t)m, chunks.end());
    chunks.resize(chunks.size() - m);
    for (const Chunk& c : tail) {
        if (c.nrows != 1) {
            chunks.push_back(c);
            continue;
        }
        const uint64_t half = std::max(grain, ((c.ncols + 1) / 2 + grain - 1) / grain * grain);
        for (uint64_t c0 = 0; c0 < c.ncols; c0 += half)
            chunks.push_back(Chunk{c.row0, 1, c.col0 + c0, std::min(half, c.ncols - c0)});
    }
}

Cuts cut_chunks(const PlanShape& sh, const PlanPolicy& pp)
{
    Cuts cu;
    cu.chunks.resize(sh.ts.size());
    if (pp.rule == ChunkRule::kGuided) {
        cut_guided(sh, pp, cu);
    } else if (pp.rule == ChunkRule::kGuidedRows) {
        cut_guided_rows(sh, pp, cu);
    } else {
        for (size_t i = 0; i < sh.ts.size(); ++i) {
            if (pp.rule == ChunkRule::kFixed) {
                cu.chunks[i] = make_chunks(sh.ts[i], pp.chunk_elems, sh.E);
                continue;
            }
            Cursor cur;
            for (uint64_t left = sh.ts[i].count; left > 0;) {
                const Chunk ch = next_chunk(sh.ts[i], cur, pp.target[i], sh.E);
                cu.chunks[i].push_back(ch);
                left -= ch.nrows * ch.ncols;
            }
            if (pp.rule == ChunkRule::kEqual && pp.bulk && sh.equal)
                halve_last_chunks(cu.chunks[i], (2 * (size_t)pp.full_grid + sh.ts.size() - 1) / sh.ts.size(),
                                  pp.grain);
        }
    }
    for (auto& cs : cu.chunks)
        cu.max_chunks = std::max(cu.max_chunks, cs.size());
    if (pp.rule != ChunkRule::kGuided)
        for (size_t c = 0; c < cu.max_chunks; ++c)
            for (size_t ti = 0; ti < sh.ts.size(); ++ti)
                if (c < cu.chunks[ti].size())
                    cu.order.push_back({ti, c});
    return cu;
}

// One item waiting to be emitted, with the chunk row and SNAC phase that
// place it in claim order.
struct Deferred {
    Builder::Pending p;
    ItemKind kind;
    pl_op op;
    Chunk ch;
};

// Items of the derivation, by chunk row and phase: 0 producers (zero-staging
// moves, stages, the owner's reduce of the zero-staging composed form),
// 1 consumers of staged chunks, 2 gathers of reduced chunks.  Without a lag
// items are emitted at once, in creation order (each transfer's producers,
// then its consumers).
class Emitter {
public:
    Emitter(HostPlan& hp, const PlanShape& sh, const PlanPolicy& pp, pl_op op, int R, int lag, size_t rows)
        : b(hp, R), sh_(sh), pp_(pp), op_(op), R_(R), lag_(lag), cursor_(R, 0)
    {
        for (auto& r : rows_)
            r.assign(rows, {});
        if (pp.staged)
            uses_.assign((size_t)R * pp.slots_per_rank, 0);
    }

    pl_status chunk(const Transfer& t, size_t row, const Chunk& ch)
    {
        if (!pp_.staged) {
            zero_staging(t, row, ch);
            return PL_OK;
        }
        tickets = true;
        return staged(t, row, ch);
    }

    void merge_stages();
    int resolve_lag(size_t max_chunks) const;
    void emit_in_lag_order(size_t max_chunks, int lag);

    Builder b;
    bool tickets = false;
    uint32_t next_flag = 0;
    uint64_t bytes_read = 0, bytes_written = 0;

private:
    void put(size_t row, int phase, Builder::Pending& pend, ItemKind kind, pl_op pop, const Chunk& ch)
    {
        if (lag_ == 0 || !pp_.ticketed)
            b.emit(pend, kind, pop, ch);
        else
            rows_[phase][row].push_back(Deferred{std::move(pend), kind, pop, ch});
    }

    // The slot of the next chunk `rank` stages, and which use of that slot it is.
    pl_status stage_slot(int rank, uint32_t& slot_out, uint32_t& use_out)
    {
        const uint64_t s = (uint64_t)rank * pp_.slots_per_rank + (cursor_[rank]++ % pp_.slots_per_rank);
        if (uses_[s] >= kMaxUsesPerLaunch)
            return PL_ERR_UNSUPPORTED;
        slot_out = (uint32_t)s;
        use_out = uses_[s]++;
        return PL_OK;
    }

    // The destination whose rank owns the transfer's partition (Figure 6: rank
    // k reduces partition k).
    static size_t owner_of(const Transfer& t)
    {
        for (size_t d = 0; d < t.dsts.size(); ++d)
            if ((uint64_t)t.dsts[d].rank == t.name)
                return d;
        return 0;
    }

    void zero_staging(const Transfer& t, size_t row, const Chunk& ch);
    pl_status staged(const Transfer& t, size_t row, const Chunk& ch);
    void staged_composed(const Transfer& t, size_t row, const Chunk& ch, const std::vector<uint32_t>& slot,
                         const std::vector<uint32_t>& use, uint32_t yslot, uint32_t yuse);

    const PlanShape& sh_;
    const PlanPolicy& pp_;
    pl_op op_;
    int R_;
    int lag_;
    std::vector<std::vector<Deferred>> rows_[3];
    std::vector<uint64_t> cursor_;  // staged: chunks each rank has staged so far
    std::vector<uint32_t> uses_;    // staged: uses of each slot so far
};

void Emitter::zero_staging(const Transfer& t, size_t row, const Chunk& ch)
{
    const uint64_t blk = ch.nrows * ch.ncols * sh_.S;
    const bool sum = op_ != PL_COPY && t.srcs.size() > 1;  // a reduction (sum or maximum)
    if (sum && t.dsts.size() > 1 && pp_.vector_compose) {
        // Figure 6 at the grain of one vector: one item reduces the chunk
        // into the owner's output (destination 0) and writes the others from
        // there; each vector's reread follows its store in the same thread.
        const size_t o = owner_of(t);
        Builder::Pending cm;
        for (auto& g : t.srcs)
            cm.src.push_back(b.region(g, ch));
        cm.dst.push_back(b.region(t.dsts[o], ch));
        for (size_t d = 0; d < t.dsts.size(); ++d)
            if (d != o)
                cm.dst.push_back(b.region(t.dsts[d], ch));
        put(row, 0, cm, kCompose, op_, ch);
        bytes_read += blk * (t.srcs.size() + 1);
        bytes_written += blk * t.dsts.size();
        return;
    }
    if (sum && t.dsts.size() > 1 && pp_.composed) {
        // Figure 6, zero-staging: the owner reduces the chunk into its output
        // and notifies; one item then reads the owner's chunk once and writes
        // it to every other rank (an AllGather item).
        tickets = true;
        const size_t o = owner_of(t);
        const uint32_t flag = next_flag++;
        Builder::Pending red;
        for (auto& g : t.srcs)
            red.src.push_back(b.region(g, ch));
        red.dst.push_back(b.region(t.dsts[o], ch));
        red.posts.push_back(mk_sync(kNotify, flag, 0));
        put(row, 0, red, kMove, op_, ch);
        bytes_read += blk * t.srcs.size();
        bytes_written += blk;
        Builder::Pending ag;
        ag.src.push_back(b.region(t.dsts[o], ch));
        for (size_t d = 0; d < t.dsts.size(); ++d)
            if (d != o)
                ag.dst.push_back(b.region(t.dsts[d], ch));
        ag.waits.push_back(mk_sync(kWaitFull, flag, 0));
        put(row, 2, ag, kConsume, PL_COPY, ch);
        bytes_read += blk;
        bytes_written += blk * (t.dsts.size() - 1);
        return;
    }
    // Zero-staging Consume: read the sources, write every destination.
    for (size_t d0 = 0; d0 < t.dsts.size(); d0 += kMaxRanks) {
        Builder::Pending mv;
        for (auto& g : t.srcs)
            mv.src.push_back(b.region(g, ch));
        const size_t d1 = std::min(t.dsts.size(), d0 + kMaxRanks);
        for (size_t d = d0; d < d1; ++d)
            mv.dst.push_back(b.region(t.dsts[d], ch));
        put(row, 0, mv, kMove, op_, ch);
        bytes_read += blk * t.srcs.size();
        bytes_written += blk * (d1 - d0);
    }
}

// Staged SNAC: every source rank stages its chunk into its ring and
// notifies; consumers wait, copy or reduce from the ring, and credit the slot
// so its producer may reuse it.
pl_status Emitter::staged(const Transfer& t, size_t row, const Chunk& ch)
{
    const uint64_t blk = ch.nrows * ch.ncols * sh_.S;
    const uint64_t se = pp_.slot_elems;
    const bool sum = op_ != PL_COPY && t.srcs.size() > 1;
    pl_status st;
    std::vector<uint32_t> slot(t.srcs.size()), use(t.srcs.size());
    for (size_t s = 0; s < t.srcs.size(); ++s) {
        if ((st = stage_slot(t.srcs[s].rank, slot[s], use[s])) != PL_OK)
            return st;
        Builder::Pending sg;
        sg.src.push_back(b.region(t.srcs[s], ch));
        sg.dst.push_back(b.slot(slot[s], se, ch));
        if (use[s] > 0)
            sg.waits.push_back(mk_sync(kWaitFree, slot[s], use[s] - 1));
        sg.posts.push_back(mk_sync(kNotify, slot[s], use[s]));
        put(row, 0, sg, kStage, PL_COPY, ch);
        bytes_read += blk;
        bytes_written += blk;
    }
    if (!sum) {
        // COPY: one consumer per destination rank, each reading the slot.
        const uint32_t n = (uint32_t)t.dsts.size();
        for (size_t d = 0; d < t.dsts.size(); ++d) {
            Builder::Pending cs;
            cs.src.push_back(b.slot(slot[0], se, ch));
            cs.dst.push_back(b.region(t.dsts[d], ch));
            cs.waits.push_back(mk_sync(kWaitFull, slot[0], use[0]));
            cs.posts.push_back(mk_sync(kCredit, slot[0], use[0], n));
            put(row, 1, cs, kConsume, PL_COPY, ch);
            bytes_read += blk;
            bytes_written += blk;
        }
        return PL_OK;
    }
    if (t.dsts.size() == 1 || !pp_.composed) {
        // SUM: one consumer reduces the R staged chunks into every destination.
        Builder::Pending cs;
        for (size_t s = 0; s < t.srcs.size(); ++s)
            cs.src.push_back(b.slot(slot[s], se, ch));
        for (auto& g : t.dsts)
            cs.dst.push_back(b.region(g, ch));
        for (size_t s = 0; s < t.srcs.size(); ++s) {
            cs.waits.push_back(mk_sync(kWaitFull, slot[s], use[s]));
            cs.posts.push_back(mk_sync(kCredit, slot[s], use[s], 1));
        }
        put(row, 1, cs, kConsume, op_, ch);
        bytes_read += blk * t.srcs.size();
        bytes_written += blk * t.dsts.size();
        return PL_OK;
    }
    // Figure 6: the owner reduces, writes its output and re-stages the reduced
    // chunk into its own ring; the other ranks gather it.
    const size_t o = owner_of(t);
    uint32_t yslot, yuse;
    if ((st = stage_slot(t.dsts[o].rank, yslot, yuse)) != PL_OK)
        return st;
    Builder::Pending red;
    for (size_t s = 0; s < t.srcs.size(); ++s)
        red.src.push_back(b.slot(slot[s], se, ch));
    red.dst.push_back(b.region(t.dsts[o], ch));
    red.dst.push_back(b.slot(yslot, se, ch));
    for (size_t s = 0; s < t.srcs.size(); ++s)
        red.waits.push_back(mk_sync(kWaitFull, slot[s], use[s]));
    if (yuse > 0)
        red.waits.push_back(mk_sync(kWaitFree, yslot, yuse - 1));
    for (size_t s = 0; s < t.srcs.size(); ++s)
        red.posts.push_back(mk_sync(kCredit, slot[s], use[s], 1));
    red.posts.push_back(mk_sync(kNotify, yslot, yuse));
    put(row, 1, red, kConsume, op_, ch);
    bytes_read += blk * t.srcs.size();
    bytes_written += 2 * blk;
    const uint32_t n = (uint32_t)t.dsts.size() - 1;
    for (size_t d = 0; d < t.dsts.size(); ++d) {
        if (d == o)
            continue;
        Builder::Pending ag;
        ag.src.push_back(b.slot(yslot, se, ch));
        ag.dst.push_back(b.region(t.dsts[d], ch));
        ag.waits.push_back(mk_sync(kWaitFull, yslot, yuse));
        ag.posts.push_back(mk_sync(kCredit, yslot, yuse, n));
        put(row, 2, ag, kConsume, PL_COPY, ch);
        bytes_read += blk;
        bytes_written += blk;
    }
    return PL_OK;
}

// Staged fused AllReduce (every transfer has as many destinations as
// sources): the stages one source rank makes in one chunk row (its chunk of
// each partition, equally spaced in its buffer, into consecutive slots of its
// ring) become one multi-row item, which moves as many bytes as a consume
// item: at R = 8 a row of 64 stage items and 8 consume items becomes 8 and 8
// (measured 7% faster).  Where consume items are lighter (ReduceScatter: 8
// sources, 1 destination) or re-stage (the composed form), merged stages
// measured 8-11% slower, so they stay one per chunk.
void Emitter::merge_stages()
{
    bool merge = pp_.staged && lag_ != 0 && !pp_.composed;
    for (const Transfer& t : sh_.ts)
        merge &= t.dsts.size() == t.srcs.size();
    if (!merge)
        return;
    for (auto& row : rows_[0]) {
        std::vector<Deferred> merged;
        merged.reserve(row.size());
        std::vector<bool> used(row.size(), false);
        for (size_t i = 0; i < row.size(); ++i) {
            if (used[i])
                continue;
            used[i] = true;
            Deferred d = std::move(row[i]);
            if (d.kind == kStage && d.ch.nrows == 1 && d.p.src.size() == 1 && d.p.dst.size() == 1) {
                const Ref s0 = d.p.src[0], d0 = d.p.dst[0];
                uint64_t ss = 0, ds = 0, n = 1;
                for (size_t j = i + 1; j < row.size(); ++j) {
                    if (used[j])
                        continue;
                    const Deferred& e = row[j];
                    if (e.kind != kStage || e.ch.nrows != 1 || e.ch.ncols != d.ch.ncols || e.p.src.size() != 1 ||
                        e.p.dst.size() != 1 || e.p.src[0].buf != s0.buf || e.p.dst[0].buf != d0.buf)
                        continue;
                    const Ref& se = e.p.src[0];
                    const Ref& de = e.p.dst[0];
                    if (se.offset <= s0.offset || de.offset <= d0.offset)
                        break;
                    const uint64_t sse = (se.offset - s0.offset) / n, dse = (de.offset - d0.offset) / n;
                    if (n == 1) {
                        ss = sse;
                        ds = dse;
                    }
                    if (sse != ss || dse != ds || ss * n != se.offset - s0.offset || ds * n != de.offset - d0.offset ||
                        ss < d.ch.ncols || ds < d.ch.ncols)
                        break;
                    used[j] = true;
                    ++n;
                    for (const Sync& w : e.p.waits)
                        d.p.waits.push_back(w);
                    for (const Sync& q : e.p.posts)
                        d.p.posts.push_back(q);
                }
                if (n > 1) {
                    d.p.src[0].stride = ss;
                    d.p.dst[0].stride = ds;
                    d.ch = Chunk{0, n, 0, d.ch.ncols};
                }
            }
            merged.push_back(std::move(d));
        }
        row = std::move(merged);
    }
}

// The lag in chunk rows between producers and their consumers.  The
// automatic lag (a negative `lag_`) puts about two grids of producers between
// a producer and its first consumer, so consumers are claimed once producers
// are done.  (Counting the consumers of a row too made the lag shorter and the
// composed AllReduce wait: 0.76 -> 0.49 of the roofline, measured.)
int Emitter::resolve_lag(size_t max_chunks) const
{
    if (lag_ >= 0 || max_chunks == 0)
        return lag_ < 0 ? 0 : lag_;
    const size_t per_row = std::max<size_t>(1, rows_[0][0].size());
    // CTAs hold claimed items ahead of the one they move, so about two grids
    // of items may be claimed but not yet finished
    return (int)std::min<size_t>(((size_t)2 * pp_.full_grid + per_row - 1) / per_row + 1, 64);
}

// Emit in claim order: producers of row t, their consumers L rows later,
// gathers of reduced chunks one more lag later (or L when nothing sits
// between).
void Emitter::emit_in_lag_order(size_t max_chunks, int lag)
{
    const size_t L = (size_t)lag;
    bool has_phase1 = false;
    for (auto& r : rows_[1])
        has_phase1 |= !r.empty();
    const size_t L2 = has_phase1 ? 2 * L : L;
    for (size_t t = 0; L > 0 && t < max_chunks + L2; ++t) {
        if (t < max_chunks)
            for (Deferred& d : rows_[0][t])
                b.emit(d.p, d.kind, d.op, d.ch);
        if (t >= L && t - L < max_chunks)
            for (Deferred& d : rows_[1][t - L])
                b.emit(d.p, d.kind, d.op, d.ch);
        if (t >= L2 && t - L2 < max_chunks)
            for (Deferred& d : rows_[2][t - L2])
                b.emit(d.p, d.kind, d.op, d.ch);
    }
}

// The plan's launch facts and statistics once its items exist: reference
// layout, alignment, the kernel's op mix, the claim rule and grid.
pl_status finalise_plan(HostPlan& hp, const PlanShape& sh, const PlanPolicy& pp, const ResolvedPolicy& pol,
                        pl_op op, pl_dtype dt, bool tickets)
{
    const uint64_t S = sh.S, E = sh.E;
    if (hp.items.size() >= (1ull << 31) || hp.refs.size() >= (1ull << 32) || hp.syncs.size() >= (1ull << 32))
        return PL_ERR_UNSUPPORTED;
    // Items with one reference count, laid out in order: a CTA that knows its
    // first item's index loads that item's references alongside its header.
    if (!hp.items.empty()) {
        const uint32_t n = (uint32_t)hp.items[0].nsrc + hp.items[0].ndst;
        bool uniform = n <= (uint32_t)kMaxRefsPerItem;
        for (size_t i = 0; uniform && i < hp.items.size(); ++i)
            uniform = (uint32_t)hp.items[i].nsrc + hp.items[i].ndst == n && hp.items[i].ref == (uint64_t)i * n;
        hp.refs_per_item = uniform ? (int)n : 0;
    }
    hp.all_aligned = 1;
    bool wide = true, compose = false;
    for (const Item& it : hp.items) {
        compose |= it.kind == kCompose;
        if (it.op)
            wide &= it.nsrc >= 8;
        if (it.nsrc > kMaxRanks || it.ndst > kMaxRanks || it.nsrc == 0 || it.ndst == 0)
            return PL_ERR_UNSUPPORTED;  // the kernel holds at most 64 sources and 64 destinations
        hp.ops |= it.op ? kOpsReduce : kOpsCopy;
        for (uint32_t k = it.ref; k < it.ref + it.nsrc + it.ndst; ++k) {
            const Ref& f = hp.refs[k];
            if ((f.offset * S) % 16 || (it.rows > 1 && (f.stride * S) % 16))
                hp.all_aligned = 0;
        }
    }
    // bf16 sums of 8+ sources stream best as 1 vector x 8 sources per step;
    // fp32 sums and fewer sources as 2 vectors x 4 sources (measured on GB300).
    // fp16 has bf16's vector shape and takes its rule.
    if (hp.ops == kOpsReduce && wide && op == PL_SUM && (dt == PL_BF16 || dt == PL_FP16))
        hp.ops |= kOpsWide;
    if (op == PL_MAX && (hp.ops & kOpsReduce))
        hp.ops |= kOpsMax;
    if (compose)
        hp.ops |= kOpsCompose;
    if (tickets && !waits_precede(hp))
        return PL_ERR_NOMEM;

    int ctas = pol.ctas ? pol.ctas : pp.full_grid;
    ctas = (int)std::min<uint64_t>((uint64_t)ctas, std::max<uint64_t>(1, hp.items.size()));
    ctas = std::max(1, ctas);
    // Claim rule: items are claimed in index order through the device ticket
    // when they wait on one another, and also whenever there are more items
    // than CTAs, so that a CTA that finishes early takes the next item
    // (dynamic balance; the guided sizes rely on it).  One item per CTA needs
    // no ticket.
    const bool claim_in_order = tickets || hp.items.size() > (size_t)ctas;
    if (hp.inline_form && (hp.items.size() > (size_t)kInlineMaxItems || hp.refs.size() > (size_t)kInlineMaxPtrs))
        hp.inline_form = false;  // (cannot happen: the inline cuts are the items)
    // Items within the misaligned vector counts run inline over buffers at any
    // alignment (a destination head of up to E - 1 elements goes first).
    hp.inline_any_alignment = hp.inline_form;
    for (const Item& it : hp.items)
        hp.inline_any_alignment &= it.cols <= misaligned_cap(it.op != 0, it.ndst) * E + E - 1;
    pl_plan_stats& s = hp.stats;
    s.items = hp.items.size();
    s.refs = hp.refs.size();
    s.syncs = hp.syncs.size();
    s.flags = hp.nflags;
    s.chunk_elems = pp.chunk_elems;
    s.slots = pp.slots_per_rank;
    s.slot_elems = pp.staged ? pp.slot_elems : 0;
    s.ctas = hp.inline_form ? (int)hp.items.size() : ctas;
    s.threads = hp.inline_form ? kInlineThreads
                               : snac_threads(hp.ops, hp.all_aligned && !hp.flagged_reduction);
    s.uses_tickets = hp.inline_form ? 0 : (claim_in_order ? 1 : 0);
    s.path = pol.path;
    s.datapath = hp.inline_form ? PL_ATOM_INLINE : launch_bulk(hp, pol) ? PL_ATOM_BULK : PL_ATOM_VECTOR;
    return PL_OK;
}

// Derives the work list of a layout pair with consumers emitted `lag` chunk
// rows behind the producers they wait for (so the CTAs that claim them in
// order rarely spin); lag < 0 picks the automatic lag.
pl_status derive_order(const pl_layout& in, const pl_layout& out, pl_op op, pl_dtype dt, int R,
                       const ResolvedPolicy& pol, int num_sms, Occupancy occ, uint64_t scratch_bytes, int lag,
                       HostPlan& hp)
{
    if (in.R != R || out.R != R)
        return PL_ERR_INVALID;
    hp = HostPlan{};
    hp.R = R;
    hp.dtype = dt;
    PlanShape sh;
    pl_status st = analyse(in, out, op, dt, R, sh);
    if (st != PL_OK)
        return st;
    PlanPolicy pp;
    if ((st = choose_policy(sh, op, R, pol, num_sms, occ, scratch_bytes, pp)) != PL_OK)
        return st;
    hp.flagged_reduction = pp.flagged_reduction;
    hp.inline_form = pp.rule == ChunkRule::kInline;
    const Cuts cu = cut_chunks(sh, pp);

    Emitter em(hp, sh, pp, op, R, lag, cu.max_chunks);
    for (const auto& oc : cu.order)
        if ((st = em.chunk(sh.ts[oc.first], oc.second, cu.chunks[oc.first][oc.second])) != PL_OK)
            return st;
    em.merge_stages();
    hp.lag = em.resolve_lag(cu.max_chunks);
    em.emit_in_lag_order(cu.max_chunks, hp.lag);
    hp.nflags = pp.staged ? (uint32_t)((uint64_t)R * pp.slots_per_rank) : em.next_flag;
    hp.stats.bytes_read = em.bytes_read;
    hp.stats.bytes_written = em.bytes_written;
    return finalise_plan(hp, sh, pp, pol, op, dt, em.tickets);
}

// The work list of a layout pair: the automatic lag is tried first; a lag the
// ring cannot hold (a slot would be reused before its consumers) or that
// breaks the claim-order rule falls back to smaller ones, down to none.
pl_status derive(const pl_layout& in, const pl_layout& out, pl_op op, pl_dtype dt, int R,
                 const ResolvedPolicy& pol, int num_sms, Occupancy occ, uint64_t scratch_bytes, HostPlan& hp)
{
    pl_status st = derive_order(in, out, op, dt, R, pol, num_sms, occ, scratch_bytes, -1, hp);
    if (st != PL_ERR_NOMEM)
        return st;
    for (int lag = hp.lag / 2; lag >= 0; lag = lag > 1 ? lag / 2 : lag - 1) {
        st = derive_order(in, out, op, dt, R, pol, num_sms, occ, scratch_bytes, lag, hp);
        if (st != PL_ERR_NOMEM)
            return st;
    }
    return st;
}

}  // namespace

// -------------------------------------------------------- plan introspection

struct pl_plan {
    HostPlan hp;
};

extern "C" {

PL_API pl_status pl_plan_create(pl_plan** plan, const pl_layout* in, const pl_layout* out, pl_op op,
                                pl_dtype dtype, int R, const pl_policy* policy, int num_sms,
                                uint64_t scratch_bytes)
{
    if (!plan || !in || !out || R < 1 || R > kMaxRanks || num_sms < 1)
        return PL_ERR_INVALID;
    pl_status vs = check_op_dtype(op, dtype);
    if (vs != PL_OK)
        return vs;
    ResolvedPolicy rp;
    pl_status st = resolve_policy(policy, rp);
    if (st != PL_OK)
        return st;
    std::unique_ptr<pl_plan> p(new (std::nothrow) pl_plan);
    if (!p)
        return PL_ERR_NOMEM;
    st = derive(*in, *out, op, dtype, R, rp, num_sms, Occupancy{}, scratch_bytes, p->hp);
    if (st != PL_OK)
        return st;
    *plan = p.release();
    return PL_OK;
}

PL_API pl_status pl_plan_destroy(pl_plan* plan)
{
    delete plan;
    return PL_OK;
}

PL_API pl_status pl_plan_get_stats(const pl_plan* plan, pl_plan_stats* stats)
{
    if (!plan || !stats)
        return PL_ERR_INVALID;
    *stats = plan->hp.stats;
    return PL_OK;
}

PL_API pl_status pl_plan_get_item(const pl_plan* plan, uint64_t i, pl_plan_item* item, pl_plan_ref* refs,
                                  int max_refs, pl_plan_sync* syncs, int max_syncs)
{
    if (!plan || !item || i >= plan->hp.items.size())
        return PL_ERR_INVALID;
    const HostPlan& hp = plan->hp;
    const Item& it = hp.items[i];
    item->kind = it.kind;
    item->op = it.op;
    item->nsrc = it.nsrc;
    item->ndst = it.ndst;
    item->nwait = it.nwait;
    item->npost = it.npost;
    item->rows = it.rows;
    item->cols = it.cols;
    int nref = it.nsrc + it.ndst;
    if (refs) {
        if (max_refs < nref)
            return PL_ERR_INVALID;
        for (int k = 0; k < nref; ++k) {
            const Ref& f = hp.refs[it.ref + k];
            int R = hp.R;
            pl_plan_ref& o = refs[k];
            if ((int)f.buf < R) {
                o.space = PL_SPACE_IN;
                o.index = (int)f.buf;
            } else if ((int)f.buf < 2 * R) {
                o.space = PL_SPACE_OUT;
                o.index = (int)f.buf - R;
            } else {
                o.space = PL_SPACE_SCRATCH;
                o.index = 0;
            }
            o.offset = f.offset;
            o.stride = f.stride;
        }
    }
    int nsync = it.nwait + it.npost;
    if (syncs) {
        if (max_syncs < nsync)
            return PL_ERR_INVALID;
        for (int k = 0; k < nsync; ++k) {
            const Sync& s = hp.syncs[it.sync + k];
            syncs[k].type = s.type;
            syncs[k].flag = s.flag;
            syncs[k].use = s.use;
            syncs[k].count = s.count;
        }
    }
    return PL_OK;
}

}  // extern "C"

// ------------------------------------------------------------------ context

namespace {

struct DevicePlan {
    HostPlan hp;  // host copy (stats, counts)
    void* mem = nullptr;
    const Item* items = nullptr;
    const Ref* refs = nullptr;
    const Sync* syncs = nullptr;
};

class DeviceGuard {
public:
    explicit DeviceGuard(int dev)
    {
        ok_ = cudaGetDevice(&prev_) == cudaSuccess;
        if (ok_ && prev_ != dev)
            ok_ = cudaSetDevice(dev) == cudaSuccess;
        dev_ = dev;
    }
    ~DeviceGuard()
    {
        if (prev_ != dev_)
            cudaSetDevice(prev_);
    }
    bool ok() const { return ok_; }

private:
    int prev_ = -1, dev_ = -1;
    bool ok_ = false;
};

}  // namespace

struct pl_ctx {
    int device = 0;
    int num_sms = 0;
    Occupancy occ;
    void* state_mem = nullptr;
    DeviceState st{};
    uint32_t flag_capacity = 0;
    char* scratch = nullptr;
    uint64_t scratch_bytes = 0;
    uint64_t launches = 0;
    int last_cuda_error = 0;
    std::unordered_map<std::string, std::unique_ptr<DevicePlan>> cache;
    std::map<std::pair<int, uint64_t>, pl_layout*> ar_layouts;
    // Host images of the inline kernel's parameter blocks (copied by each launch).
    InlineSmall inline_small{};
    std::unique_ptr<InlineLarge> inline_large;
};

namespace {

pl_status cuda_fail(pl_ctx* ctx, cudaError_t e)
{
    ctx->last_cuda_error = (int)e;
    cudaGetLastError();  // clear a sticky-free error so later calls see their own
    return e == cudaErrorMemoryAllocation ? PL_ERR_NOMEM : PL_ERR_CUDA;
}

// (Re)allocates the flag arrays so that at least n flags exist; all zero.
pl_status ensure_flags(pl_ctx* ctx, uint32_t n)
{
    if (n <= ctx->flag_capacity && ctx->state_mem)
        return PL_OK;
    uint32_t cap = std::max<uint32_t>(std::max<uint32_t>(n, 4096), ctx->flag_capacity * 2);
    size_t bytes = (size_t)cap * (8 + 8 + 4) + 64;
    void* mem = nullptr;
    if (ctx->state_mem) {
        cudaError_t e = cudaDeviceSynchronize();
        if (e != cudaSuccess)
            return cuda_fail(ctx, e);
    }
    cudaError_t e = cudaMalloc(&mem, bytes);
    if (e != cudaSuccess)
        return cuda_fail(ctx, e);
    e = cudaMemset(mem, 0, bytes);
    if (e != cudaSuccess) {
        cudaFree(mem);
        return cuda_fail(ctx, e);
    }
    if (ctx->state_mem)
        cudaFree(ctx->state_mem);
    ctx->state_mem = mem;
    ctx->flag_capacity = cap;
    char* p = (char*)mem;
    ctx->st.full = (unsigned long long*)p;
    ctx->st.done = (unsigned long long*)(p + (size_t)cap * 8);
    ctx->st.count = (unsigned int*)(p + (size_t)cap * 16);
    char* tail = p + (size_t)cap * 20;
    tail = (char*)(((uintptr_t)tail + 15) & ~(uintptr_t)15);
    ctx->st.ticket = (unsigned int*)tail;
    ctx->st.exited = (unsigned int*)(tail + 4);
    ctx->st.status = (int*)(tail + 8);
    ctx->st.abort = (int*)(tail + 12);
    ctx->st.epoch = (unsigned long long*)(tail + 16);
    return PL_OK;
}

// Layouts are immutable, so a plan is identified by the layouts' ids plus
// everything else that shapes the work list.
std::string plan_key(const pl_layout& in, const pl_layout& out, pl_op op, pl_dtype dt, int R,
                     const ResolvedPolicy& rp)
{
    uint64_t k[9] = {in.id, out.id, (uint64_t)op, (uint64_t)dt, (uint64_t)R, (uint64_t)rp.path,
                     (uint64_t)rp.ar_form,
                     ((uint64_t)rp.ctas << 32) | ((uint64_t)rp.datapath_auto << 8) | (uint64_t)rp.datapath,
                     rp.chunk_bytes};
    return std::string(reinterpret_cast<const char*>(k), sizeof k);
}

pl_status get_plan(pl_ctx* ctx, const pl_layout& in, const pl_layout& out, pl_op op, pl_dtype dt, int R,
                   const ResolvedPolicy& rp, DevicePlan*& dp)
{
    std::string key = plan_key(in, out, op, dt, R, rp);
    auto it = ctx->cache.find(key);
    if (it != ctx->cache.end()) {
        dp = it->second.get();
        return PL_OK;
    }
    std::unique_ptr<DevicePlan> p(new (std::nothrow) DevicePlan);
    if (!p)
        return PL_ERR_NOMEM;
    pl_status st = derive(in, out, op, dt, R, rp, ctx->num_sms, ctx->occ, ctx->scratch_bytes, p->hp);
    if (st != PL_OK)
        return st;
    size_t bi = p->hp.items.size() * sizeof(Item);
    size_t br = p->hp.refs.size() * sizeof(Ref);
    size_t bs = p->hp.syncs.size() * sizeof(Sync);
    size_t oi = 0, orr = (bi + 255) / 256 * 256, os = orr + (br + 255) / 256 * 256;
    size_t total = std::max<size_t>(256, os + bs);
    if (ctx->cache.size() >= kMaxCachedPlans) {
        cudaError_t e = cudaDeviceSynchronize();
        if (e != cudaSuccess)
            return cuda_fail(ctx, e);
        for (auto& kv : ctx->cache)
            cudaFree(kv.second->mem);
        ctx->cache.clear();
    }
    cudaError_t e = cudaMalloc(&p->mem, total);
    if (e != cudaSuccess)
        return cuda_fail(ctx, e);
    std::vector<char> host(total, 0);
    if (bi)
        std::memcpy(host.data() + oi, p->hp.items.data(), bi);
    if (br)
        std::memcpy(host.data() + orr, p->hp.refs.data(), br);
    if (bs)
        std::memcpy(host.data() + os, p->hp.syncs.data(), bs);
    e = cudaMemcpy(p->mem, host.data(), total, cudaMemcpyHostToDevice);
    if (e != cudaSuccess) {
        cudaFree(p->mem);
        return cuda_fail(ctx, e);
    }
    p->items = (const Item*)((char*)p->mem + oi);
    p->refs = (const Ref*)((char*)p->mem + orr);
    p->syncs = (const Sync*)((char*)p->mem + os);
    // The device copy holds everything the persistent kernel needs; keep host
    // vectors only for stats, and for the parameter block of an inline plan
    // (at most kInlineMaxItems items and kInlineMaxPtrs references).
    if (!p->hp.inline_form) {
        p->hp.items.clear();
        p->hp.items.shrink_to_fit();
        p->hp.refs.clear();
        p->hp.refs.shrink_to_fit();
    }
    p->hp.syncs.clear();
    p->hp.syncs.shrink_to_fit();
    dp = p.get();
    ctx->cache.emplace(std::move(key), std::move(p));
    return PL_OK;
}

struct Interval {
    uintptr_t lo, hi;
    bool is_out;
    int rank;
    const pl_part* part;
};

// Checks every part against its buffer, element alignment, and the alias
// rule: an output may only coincide exactly with one of its own sources.
pl_status check_buffers(const pl_layout& in, const pl_layout& out, pl_dtype dt, int R,
                        void* const* in_bufs, const uint64_t* in_counts,
                        void* const* out_bufs, const uint64_t* out_counts, bool* in_place = nullptr)
{
    if (in_place)
        *in_place = false;
    const uint64_t S = elem_size(dt);
    std::vector<Interval> iv;
    for (int side = 0; side < 2; ++side) {
        const pl_layout& L = side ? out : in;
        void* const* bufs = side ? out_bufs : in_bufs;
        const uint64_t* counts = side ? out_counts : in_counts;
        for (int r = 0; r < R; ++r) {
            if (counts[r] > 0 && !bufs[r])
                return PL_ERR_INVALID;
            if (bufs[r] && ((uintptr_t)bufs[r] % S))
                return PL_ERR_INVALID;
            for (int i = L.first[r]; i < L.first[r + 1]; ++i) {
                const pl_part& p = L.parts[i];
                if (region_count(p) == 0)
                    continue;
                if (region_extent(p) > counts[r])
                    return PL_ERR_LAYOUT;
                uintptr_t lo = (uintptr_t)bufs[r] + p.offset * S;
                uintptr_t hi = (uintptr_t)bufs[r] + region_extent(p) * S;
                iv.push_back(Interval{lo, hi, side == 1, r, &p});
            }
        }
    }
    std::sort(iv.begin(), iv.end(), [](const Interval& a, const Interval& b) { return a.lo < b.lo; });
    for (size_t i = 0; i < iv.size(); ++i) {
        for (size_t j = i + 1; j < iv.size() && iv[j].lo < iv[i].hi; ++j) {
            const Interval& a = iv[i];
            const Interval& b = iv[j];
            if (!a.is_out && !b.is_out)
                continue;  // inputs may overlap each other
            if (a.is_out && b.is_out)
                return PL_ERR_ALIAS;
            const Interval& o = a.is_out ? a : b;
            const Interval& n = a.is_out ? b : a;
            bool exact = o.lo == n.lo && o.hi == n.hi && o.part->name == n.part->name &&
                         o.part->rows == n.part->rows && o.part->len == n.part->len &&
                         (o.part->rows == 1 || o.part->row_stride == n.part->row_stride);
            if (!exact)
                return PL_ERR_ALIAS;
            if (in_place)
                *in_place = true;
        }
    }
    return PL_OK;
}

}  // namespace

extern "C" {

PL_API pl_status pl_ctx_create(pl_ctx** out, int device, uint64_t scratch_bytes)
{
    if (!out || device < 0)
        return PL_ERR_INVALID;
    *out = nullptr;
    int ndev = 0;
    if (cudaGetDeviceCount(&ndev) != cudaSuccess || device >= ndev) {
        cudaGetLastError();
        return PL_ERR_CUDA;
    }
    std::unique_ptr<pl_ctx> ctx(new (std::nothrow) pl_ctx);
    if (!ctx)
        return PL_ERR_NOMEM;
    ctx->inline_large.reset(new (std::nothrow) InlineLarge);
    if (!ctx->inline_large)
        return PL_ERR_NOMEM;
    ctx->device = device;
    DeviceGuard g(device);
    if (!g.ok())
        return cuda_fail(ctx.get(), cudaGetLastError());
    cudaError_t e = cudaDeviceGetAttribute(&ctx->num_sms, cudaDevAttrMultiProcessorCount, device);
    if (e != cudaSuccess)
        return cuda_fail(ctx.get(), e);
    const int occ_aligned = snac_ctas_per_sm(KernelClass::kAligned);
    const int occ_aligned_reduce = snac_ctas_per_sm(KernelClass::kAlignedReduce);
    const int occ_spliced = snac_ctas_per_sm(KernelClass::kSpliced);
    if (occ_aligned > 0)
        ctx->occ.aligned = std::min(occ_aligned, kCtasPerSmAligned);
    if (occ_aligned_reduce > 0)
        ctx->occ.aligned_reduce = std::min(occ_aligned_reduce, kCtasPerSmAlignedReduce);
    if (occ_spliced > 0)
        ctx->occ.spliced = std::min(occ_spliced, kCtasPerSmSpliced);
    pl_status st = ensure_flags(ctx.get(), 4096);
    if (st != PL_OK)
        return st;
    if (scratch_bytes) {
        e = cudaMalloc((void**)&ctx->scratch, scratch_bytes);
        if (e != cudaSuccess) {
            cudaFree(ctx->state_mem);
            return cuda_fail(ctx.get(), e);
        }
        ctx->scratch_bytes = scratch_bytes;
    }
    *out = ctx.release();
    return PL_OK;
}

PL_API pl_status pl_ctx_destroy(pl_ctx* ctx)
{
    if (!ctx)
        return PL_OK;
    {
        DeviceGuard g(ctx->device);
        cudaDeviceSynchronize();
        for (auto& kv : ctx->cache)
            cudaFree(kv.second->mem);
        if (ctx->state_mem)
            cudaFree(ctx->state_mem);
        if (ctx->scratch)
            cudaFree(ctx->scratch);
        for (auto& kv : ctx->ar_layouts)
            delete kv.second;
    }
    delete ctx;
    return PL_OK;
}

PL_API int pl_ctx_cuda_error(const pl_ctx* ctx) { return ctx ? ctx->last_cuda_error : 0; }

PL_API uint64_t pl_ctx_launches(const pl_ctx* ctx) { return ctx ? ctx->launches : 0; }

PL_API pl_status pl_ctx_status(pl_ctx* ctx, void* stream)
{
    if (!ctx)
        return PL_ERR_INVALID;
    DeviceGuard g(ctx->device);
    cudaStream_t s = (cudaStream_t)stream;
    cudaError_t e = cudaStreamSynchronize(s);
    if (e != cudaSuccess)
        return cuda_fail(ctx, e);
    int host[2] = {0, 0};
    e = cudaMemcpy(host, ctx->st.status, sizeof host, cudaMemcpyDeviceToHost);
    if (e != cudaSuccess)
        return cuda_fail(ctx, e);
    if (host[0] == 0)
        return PL_OK;
    // A wait gave up: flags may be half-updated.  Start the next launch clean.
    size_t bytes = (size_t)ctx->flag_capacity * 20 + 64;
    e = cudaMemset(ctx->state_mem, 0, bytes);
    if (e != cudaSuccess)
        return cuda_fail(ctx, e);
    return host[0];
}

PL_API pl_status pl_collective(pl_ctx* ctx, const pl_layout* in, const pl_layout* out, pl_op op, pl_dtype dt,
                               int R, void* const* in_bufs, const uint64_t* in_counts, void* const* out_bufs,
                               const uint64_t* out_counts, const pl_policy* policy, void* stream)
{
    if (!ctx || !in || !out || !in_bufs || !out_bufs || !in_counts || !out_counts)
        return PL_ERR_INVALID;
    if (R < 1 || R > kMaxRanks || in->R != R || out->R != R)
        return PL_ERR_INVALID;
    pl_status st = check_op_dtype(op, dt);
    if (st != PL_OK)
        return st;
    ResolvedPolicy rp;
    st = resolve_policy(policy, rp);
    if (st != PL_OK)
        return st;
    bool in_place = false;
    if ((st = check_buffers(*in, *out, dt, R, in_bufs, in_counts, out_bufs, out_counts, &in_place)) != PL_OK)
        return st;
    DeviceGuard g(ctx->device);
    if (!g.ok())
        return cuda_fail(ctx, cudaGetLastError());
    DevicePlan* dp = nullptr;
    if ((st = get_plan(ctx, *in, *out, op, dt, R, rp, dp)) != PL_OK)
        return st;
    const pl_plan_stats& ps = dp->hp.stats;
    if (ps.items == 0)
        return PL_OK;  // nothing to move
    if ((st = ensure_flags(ctx, dp->hp.nflags)) != PL_OK)
        return st;
    if (dp->hp.inline_form) {
        // The whole plan in the launch's parameters, each reference resolved
        // to its pointer.  Plans with items larger than a vector per thread
        // need 16-byte aligned buffers; small items take any alignment as long
        // as each item's destinations share their address mod 16.  Otherwise
        // the persistent kernel below runs the same items.
        bool aligned = true;
        for (int r = 0; r < R; ++r)
            aligned &= ((reinterpret_cast<uintptr_t>(in_bufs[r]) | reinterpret_cast<uintptr_t>(out_bufs[r])) & 15u) == 0;
        if (aligned || dp->hp.inline_any_alignment) {
            const int nitems = (int)dp->hp.items.size();
            const bool small = nitems <= kInlineSmallItems && dp->hp.refs.size() <= (size_t)kInlineSmallPtrs;
            InlineSmall* is = small ? &ctx->inline_small : nullptr;
            InlineLarge* il = small ? nullptr : ctx->inline_large.get();
            InlineItem* its = small ? is->it : il->it;
            char** ptrs = small ? is->ptr : il->ptr;
            const uint64_t S = elem_size(dt);
            // In place, a reduction item's destinations include its own
            // rank's source: each of its vectors is then read whole by one
            // thread before that thread writes it anywhere.
            for (int i = 0; i < nitems; ++i) {
                const Item& it = dp->hp.items[i];
                const bool whole = in_place && it.nsrc > 1 && it.ndst > 1;
                its[i] = InlineItem{it.nsrc, it.ndst, it.ref, (uint32_t)it.cols, whole ? kInlineVectorWhole : 0u};
            }
            // Zero-staging items reference inputs and outputs only; anything
            // else takes the persistent kernel.
            bool usable = true;
            for (size_t k = 0; usable && k < dp->hp.refs.size(); ++k) {
                const Ref& f = dp->hp.refs[k];
                usable = f.buf < 2u * (uint32_t)R;
                if (usable)
                    ptrs[k] = (f.buf < (uint32_t)R ? (char*)in_bufs[f.buf] : (char*)out_bufs[f.buf - R]) + f.offset * S;
            }
            // Per item: every pointer 16-byte aligned (the kernel's shortest
            // path), else the destinations must share their address mod 16.
            const bool all_aligned = aligned && dp->hp.all_aligned;  // aligned buffers, aligned offsets
            for (int i = 0; usable && i < nitems; ++i) {
                InlineItem& it = its[i];
                if (all_aligned) {
                    it.flags |= kInlineAligned;
                    continue;
                }
                uintptr_t any = 0;
                for (uint32_t k = 0; k < (uint32_t)it.nsrc + it.ndst; ++k)
                    any |= reinterpret_cast<uintptr_t>(ptrs[it.ref + k]);
                if ((any & 15u) == 0) {
                    it.flags |= kInlineAligned;
                    continue;
                }
                const uintptr_t c0 = reinterpret_cast<uintptr_t>(ptrs[it.ref + it.nsrc]) & 15u;
                for (uint32_t d = 1; d < it.ndst; ++d)
                    usable &= (reinterpret_cast<uintptr_t>(ptrs[it.ref + it.nsrc + d]) & 15u) == c0;
            }
            if (usable) {
                cudaError_t e = launch_inline(dt, (dp->hp.ops & kOpsMax) != 0, is, il, nitems, (cudaStream_t)stream);
                if (e != cudaSuccess)
                    return cuda_fail(ctx, e);
                ++ctx->launches;
                return PL_OK;
            }
        }
    }
    LaunchArgs a{};
    a.items = dp->items;
    a.refs = dp->refs;
    a.syncs = dp->syncs;
    a.nitems = (uint32_t)ps.items;
    a.use_tickets = ps.uses_tickets;
    a.dtype = dt;
    a.nbufs = 2 * R + 1;
    a.ops = dp->hp.ops;
    a.all_aligned = dp->hp.all_aligned && !dp->hp.flagged_reduction;
    a.refs_per_item = dp->hp.refs_per_item;
    a.no_spread = in_place && (dp->hp.ops & kOpsReduce) ? 1 : 0;
    a.static_head = ps.uses_tickets && ps.syncs == 0 ? 1 : 0;
    a.timeout_ns = rp.timeout_ns;
    a.drop_notify = rp.drop_notify;
    a.st = ctx->st;
    for (int r = 0; r < R; ++r) {
        a.bufs[r] = (char*)in_bufs[r];
        a.bufs[R + r] = (char*)out_bufs[r];
    }
    a.bufs[2 * R] = ctx->scratch;
    const bool bulk = launch_bulk(dp->hp, rp);
    int stages = rp.stages;
    if (bulk && rp.datapath_auto && rp.stages_auto)
        stages = kBulkMaxStages;
    // The bulk ring's shared memory holds one CTA per SM: a grid sized for the
    // two-CTA spliced kernels is trimmed to one CTA per SM (claims adapt).
    const int ctas = bulk && !a.all_aligned ? std::min(ps.ctas, ctx->num_sms) : ps.ctas;
    cudaError_t e = launch_snac(a, ctas, bulk, stages, (cudaStream_t)stream);
    if (e != cudaSuccess)
        return cuda_fail(ctx, e);
    ++ctx->launches;
    return PL_OK;
}

PL_API pl_status pl_allreduce_op(pl_ctx* ctx, pl_op op, pl_dtype dt, int R, uint64_t count, void* const* in_bufs,
                                 void* const* out_bufs, const pl_policy* policy, void* stream)
{
    if (!ctx || R < 1 || R > kMaxRanks || op == PL_COPY)
        return PL_ERR_INVALID;
    auto key = std::make_pair(R, count);
    auto it = ctx->ar_layouts.find(key);
    if (it == ctx->ar_layouts.end()) {
        std::vector<uint64_t> lens(R, count / (uint64_t)R);
        lens[R - 1] = count - (count / (uint64_t)R) * (uint64_t)(R - 1);
        pl_layout* L = nullptr;
        pl_status st = pl_layout_partitioned(&L, R, lens.data());
        if (st != PL_OK)
            return st;
        it = ctx->ar_layouts.emplace(key, L).first;
    }
    std::vector<uint64_t> counts(R, count);
    return pl_collective(ctx, it->second, it->second, op, dt, R, in_bufs, counts.data(), out_bufs,
                         counts.data(), policy, stream);
}

PL_API pl_status pl_allreduce(pl_ctx* ctx, pl_dtype dt, int R, uint64_t count, void* const* in_bufs,
                              void* const* out_bufs, const pl_policy* policy, void* stream)
{
    return pl_allreduce_op(ctx, PL_SUM, dt, R, count, in_bufs, out_bufs, policy, stream);
}

}  // extern "C"

// ------------------------------------------------ caller-memory work lists

namespace purlin {

int derive_staged_allreduce(int R, int dtype, uint64_t count, void* const* in_bufs, void* const* out_bufs,
                            int num_sms, uint64_t ring_bytes, uint64_t chunk_bytes, HostWorkList& out)
{
    if (R < 1 || R > kMaxRanks || !in_bufs || !out_bufs || (dtype != PL_BF16 && dtype != PL_FP32 && dtype != PL_FP16))
        return PL_ERR_INVALID;
    std::vector<uint64_t> lens(R, count / (uint64_t)R);
    lens[R - 1] = count - (count / (uint64_t)R) * (uint64_t)(R - 1);
    pl_layout* L = nullptr;
    pl_status st = pl_layout_partitioned(&L, R, lens.data());
    if (st != PL_OK)
        return st;
    std::unique_ptr<pl_layout> hold(L);
    std::vector<uint64_t> counts(R, count);
    if ((st = check_buffers(*L, *L, (pl_dtype)dtype, R, in_bufs, counts.data(), out_bufs, counts.data())) != PL_OK)
        return st;
    pl_policy pol;
    pl_policy_default(&pol);
    pol.path = PL_PATH_STAGED;
    pol.allreduce_form = PL_AR_FUSED;
    pol.chunk_bytes = chunk_bytes;
    ResolvedPolicy rp;
    if ((st = resolve_policy(&pol, rp)) != PL_OK)
        return st;
    HostPlan hp;
    if ((st = derive(*L, *L, PL_SUM, (pl_dtype)dtype, R, rp, num_sms, Occupancy{}, ring_bytes, hp)) != PL_OK)
        return st;
    out.items = std::move(hp.items);
    out.refs = std::move(hp.refs);
    out.syncs = std::move(hp.syncs);
    out.nflags = hp.nflags;
    out.ops = hp.ops;
    out.all_aligned = hp.all_aligned && !hp.flagged_reduction;
    out.refs_per_item = hp.refs_per_item;
    out.ctas = hp.stats.ctas;
    out.uses_tickets = hp.stats.uses_tickets;
    return PL_OK;
}

}  // namespace purlin
