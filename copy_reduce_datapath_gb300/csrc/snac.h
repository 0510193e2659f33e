// Internal layout of a SNAC work list as the device reads it, and the launch
// interface between the host runtime (runtime.cpp) and the Atom kernels
// (atom_impl.cuh and its per-dtype instantiations).  Not part of the public ABI.
#pragma once

#include <cstdint>
#include <vector>

#include <cuda_runtime.h>

namespace purlin {

constexpr int kMaxRanks = 64;
constexpr int kMaxRefsPerItem = 2 * kMaxRanks + 1;  // R sources + R destinations + one slot
constexpr int kThreads = 512;                        // threads per CTA of the kernels for aligned plans
constexpr int kThreadsSpliced = 512;                 // threads per CTA of the kernels for other plans
// ... and of those among them whose lists only copy: half the threads, each
// with twice the vectors in flight (16), and 128 registers, so nothing
// spills; the bulk ring's realignment and its barrier per piece also go
// faster with fewer threads.  Measured on GB300: AllGatherV 64 MiB 0.80 ->
// 0.84 of the roofline, AllToAllV 1 GiB 0.95 -> 0.98; the reductions lose
// with fewer threads (ReduceScatterV 128 MiB 0.84 -> 0.78), so they keep 512.
constexpr int kThreadsSplicedCopy = 256;
constexpr int kPrefetchThread = 32;  // the spliced kernels' first thread that prefetches the next item
static_assert(kThreads >= kMaxRefsPerItem && kThreadsSpliced >= kPrefetchThread + kMaxRefsPerItem &&
                  kThreadsSplicedCopy >= kPrefetchThread + kMaxRefsPerItem,
              "one thread per region reference of an item");
constexpr int kBulkMaxStages = 8;
// CTAs per SM the kernels are built for: those for plans proven 16-byte
// aligned keep 128 registers per thread; those for other plans (every body
// through the warp-spliced path) run two CTAs per SM at 64 registers, whose
// extra warps hide the splice and reduce arithmetic between memory waits.
constexpr int kCtasPerSmAligned = 1;
constexpr int kCtasPerSmSpliced = 2;
// The kernels for aligned plans whose lists only reduce run two CTAs of 256
// threads per SM at the same 128 registers: the same warps per SM in two
// independently scheduled halves (measured on GB300, R = 8 bf16: the fused
// AllReduce at 64 MiB 0.90 -> 0.93 of the roofline, at 128 MiB 0.946 ->
// 0.958, at 1 GiB 0.987 -> 0.985; the composed one 0.898 -> 0.920, 0.935 ->
// 0.947 and 0.972 -> 0.975).  Lists that copy keep one CTA of 512 (the bulk
// ring's shared memory holds one CTA per SM).
constexpr int kThreadsAlignedReduce = 256;
constexpr int kCtasPerSmAlignedReduce = 2;

enum ItemKind : uint8_t { kMove = 0, kStage = 1, kConsume = 2, kCompose = 3 };
enum SyncType : uint8_t { kWaitFull = 0, kWaitFree = 1, kNotify = 2, kCredit = 3 };

// Element types of a launch (the same codes as the public pl_dtype values).
constexpr int kDtBf16 = 0;
constexpr int kDtFp32 = 1;
constexpr int kDtFp16 = 2;
constexpr int kDtFp8 = 3;  // any one-byte element: copied, never reduced

// Which moves a work list contains: the kernel is instantiated per mix so that
// a copy-only or reduce-only list gets code without the other path.
constexpr int kOpsCopy = 1;
constexpr int kOpsReduce = 2;  // items with several sources reduce them
constexpr int kOpsWide = 4;    // every sum has at least 8 sources: one vector x 8 sources per step
constexpr int kOpsMax = 8;     // the reduction is the maximum, not the sum
// Every reduction with several destinations is a composed step (kCompose):
// destination 0 receives the reduced values, the others are written from it.
constexpr int kOpsCompose = 16;

// Threads per CTA, and CTAs per SM, of the kernel for an op mix and an
// alignment class.
constexpr int snac_threads(int ops, bool aligned)
{
    return aligned ? ((ops & kOpsCopy) ? kThreads : kThreadsAlignedReduce)
                   : (ops == kOpsCopy ? kThreadsSplicedCopy : kThreadsSpliced);
}
constexpr int snac_min_ctas(int ops, bool aligned)
{
    return aligned ? ((ops & kOpsCopy) ? kCtasPerSmAligned : kCtasPerSmAlignedReduce) : kCtasPerSmSpliced;
}

// One work item: move a rows x cols block from nsrc sources (copy if nsrc == 1,
// rank-ordered reduction otherwise) into ndst destinations (a kCompose item:
// into destination 0, then from destination 0 into the others).  Refs
// [ref, ref + nsrc) are sources, [ref + nsrc, ref + nsrc + ndst) destinations.
// Syncs [sync, sync + nwait) run before the move, [sync + nwait, + npost) after.
struct Item {
    uint8_t kind;
    uint8_t op;        // 0 copy, 1 sum, 2 maximum
    uint16_t nsrc;
    uint16_t ndst;
    uint16_t nwait;
    uint32_t ref;
    uint32_t sync;
    uint32_t rows;
    uint16_t npost;
    uint16_t pad;
    uint64_t cols;
};
static_assert(sizeof(Item) == 32, "Item is 32 bytes");

// A region reference: buffer slot `buf` of the launch's pointer table
// (inputs 0..R-1, outputs R..2R-1, scratch 2R), element offset of row 0 and
// element distance between rows.
struct Ref {
    uint32_t buf;
    uint32_t pad;
    uint64_t offset;
    uint64_t stride;
};
static_assert(sizeof(Ref) == 24, "Ref is 24 bytes");

struct Sync {
    uint8_t type;
    uint8_t pad[3];
    uint32_t flag;
    uint32_t use;
    uint32_t count;
};
static_assert(sizeof(Sync) == 16, "Sync is 16 bytes");

// Device-side SNAC state owned by a context.
struct DeviceState {
    unsigned long long* full;   // [nflags] notify tags
    unsigned long long* done;   // [nflags] slot-free tags
    unsigned int* count;        // [nflags] consumers seen for the current use
    unsigned int* ticket;       // next item to claim
    unsigned int* exited;       // CTAs that finished (the last one resets ticket/exited)
    int* status;                // 0 ok, else a pl_status
    int* abort;                 // set with status: every wait gives up at once
    unsigned long long* epoch;  // ticketed launches that ended; the tags of the next are
                                // (epoch << 24) | (use + 1), so they grow from launch to launch
                                // even when a captured CUDA graph repeats a launch's parameters
};

struct LaunchArgs {
    const Item* items;
    const Ref* refs;
    const Sync* syncs;
    uint32_t nitems;
    int32_t use_tickets;
    int32_t dtype;               // kDtBf16, kDtFp32, kDtFp16 or kDtFp8
    int32_t nbufs;
    int32_t ops;                 // kOpsCopy | kOpsReduce present in the list, plus kOpsWide / kOpsMax
    int32_t all_aligned;         // every reference's offset (and row stride) is a multiple of 16 bytes
    int32_t refs_per_item;       // n > 0: item i's references are refs[i * n .. i * n + n); 0: read the header
    int32_t no_spread;           // 1: every vector is read and written by one thread (a reduction in place)
    int32_t static_head;         // 1 (ticketed lists without flags): each CTA's first two items are static,
                                 // blockIdx.x and blockIdx.x + grid; the ticket hands out the rest from 2 x grid
    unsigned long long timeout_ns;
    long long drop_notify;       // item index whose notifies are skipped, or -1
    DeviceState st;
    char* bufs[kMaxRefsPerItem]; // inputs, outputs, scratch
};

// Launch of the persistent SNAC kernel (atom.cu).  `bulk` selects the
// cp.async.bulk shared-memory ring for copy items with `stages` stages.
cudaError_t launch_snac(const LaunchArgs& args, int ctas, bool bulk, int stages, cudaStream_t stream);

// The per-element-type launchers behind launch_snac (atom.cu, atom_fp16.cu,
// atom_fp32.cu, atom_fp8.cu).  `aligned`: every reference and buffer is
// 16-byte aligned, so the kernels without realigning bodies serve the plan.
cudaError_t launch_snac_bf16(const LaunchArgs& a, int ctas, bool bulk, bool aligned, int stages, cudaStream_t s);
cudaError_t launch_snac_fp16(const LaunchArgs& a, int ctas, bool bulk, bool aligned, int stages, cudaStream_t s);
cudaError_t launch_snac_fp32(const LaunchArgs& a, int ctas, bool bulk, bool aligned, int stages, cudaStream_t s);
cudaError_t launch_snac_fp8(const LaunchArgs& a, int ctas, bool bulk, bool aligned, int stages, cudaStream_t s);

// CTAs of the SNAC kernel that fit on one SM at once: for aligned plans whose
// lists copy (kAligned) or only reduce (kAlignedReduce), and for other plans.
enum class KernelClass { kAligned, kAlignedReduce, kSpliced };
int snac_ctas_per_sm(KernelClass k);

// ------------------------------------------------- inline-parameter launches
//
// A small plan whose items are one-row moves between 16-byte aligned regions
// travels whole in the kernel's parameters: one item per CTA, each reference
// a resolved pointer, so the kernel starts moving data without loading any
// metadata or waiting at a barrier.  Two sizes of parameter block: the small
// one costs less per launch (measured on GB300: 2.3 KB blocks launch about
// 0.2 us faster than 9-22 KB ones).
constexpr int kInlineThreads = 512;
constexpr int kInlineSmallItems = 16;
constexpr int kInlineSmallPtrs = 256;
constexpr int kInlineMaxItems = 152;
constexpr int kInlineMaxPtrs = 2432;

// One inline item: nsrc sources then ndst destinations at ptr[ref ..], count
// elements each (copied when nsrc == 1, else reduced in source order).
struct InlineItem {
    uint16_t nsrc;
    uint16_t ndst;
    uint32_t ref;
    uint32_t count;
    uint32_t flags;  // kInlineVectorWhole | kInlineAligned
};
// The item's destinations include one of its sources (a reduction in place):
// one thread reads each vector and writes it to every destination.
constexpr uint32_t kInlineVectorWhole = 1;
// Every pointer of the item is 16-byte aligned.
constexpr uint32_t kInlineAligned = 2;
static_assert(sizeof(InlineItem) == 16, "InlineItem is 16 bytes");

template <int NI, int NP>
struct InlineArgs {
    InlineItem it[NI];
    char* ptr[NP];
};
using InlineSmall = InlineArgs<kInlineSmallItems, kInlineSmallPtrs>;
using InlineLarge = InlineArgs<kInlineMaxItems, kInlineMaxPtrs>;
static_assert(sizeof(InlineLarge) <= 32764, "kernel parameter limit");

// Launch of an inline plan of `nitems` items (atom.cu): `small` selects the
// parameter block; `maxop` the maximum instead of the sum for reductions.
cudaError_t launch_inline(int dtype, bool maxop, const InlineSmall* small, const InlineLarge* large, int nitems,
                          cudaStream_t stream);
cudaError_t launch_inline_bf16(bool maxop, const InlineSmall* small, const InlineLarge* large, int nitems,
                               cudaStream_t s);
cudaError_t launch_inline_fp16(bool maxop, const InlineSmall* small, const InlineLarge* large, int nitems,
                               cudaStream_t s);
cudaError_t launch_inline_fp32(bool maxop, const InlineSmall* small, const InlineLarge* large, int nitems,
                               cudaStream_t s);
cudaError_t launch_inline_fp8(bool maxop, const InlineSmall* small, const InlineLarge* large, int nitems,
                              cudaStream_t s);

// Host-side work list of a staged AllReduce whose device state lives in
// caller-provided memory (runtime.cpp; used by the allocation-free entry point).
struct HostWorkList {
    std::vector<Item> items;
    std::vector<Ref> refs;
    std::vector<Sync> syncs;
    uint32_t nflags = 0;
    int ops = 0;
    int all_aligned = 0;
    int refs_per_item = 0;
    int ctas = 1;
    int uses_tickets = 0;
};

// Validates the buffers like pl_allreduce and derives the staged, fused
// AllReduce of `count` elements per rank over a ring of `ring_bytes` with
// chunks of `chunk_bytes`.  Host memory only; no CUDA call.
int derive_staged_allreduce(int R, int dtype, uint64_t count, void* const* in_bufs, void* const* out_bufs,
                            int num_sms, uint64_t ring_bytes, uint64_t chunk_bytes, HostWorkList& out);

}  // namespace purlin
