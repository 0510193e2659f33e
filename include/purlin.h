/*
 * libpurlin1 -- the C ABI of a GB300 (sm_103a) implementation of the data
 * path of Purlin collectives over R logical ranks held in one GPU's memory.
 *
 * Source: "Purlin: Separating Orchestration from the Datapath of Collectives".
 *   - Abstract: a collective is a naming of an input layout and an output
 *     layout plus a copy or a reduction; a shared orchestration protocol,
 *     Stage, Notify, And Consume (SNAC), is derived from that specification;
 *     a hardware-specific datapath ("Atom") provides copy and reduce.
 *   - Figure 4 caption: ReduceScatter, AllGather and AllToAll layouts.
 *   - Figure 6 caption: AllReduce composed as ReduceScatter then AllGather,
 *     chunk by chunk.
 *   - Table 2: the variable-length (V) forms; the Ulysses sequence <-> head
 *     re-partition.
 *   - Figure 10 / Figure 16 captions: a zero-staging variant (Purlin-ZS) for
 *     buffers the consumer can read directly, and a staged variant for
 *     ordinary buffers.
 *
 * Conventions for every call:
 *   - A "rank" is a logical rank: rank r owns one input buffer in_bufs[r] and
 *     one output buffer out_bufs[r], both device pointers on the context's
 *     GPU, owned by the caller and never freed by the library.
 *   - Offsets, lengths and buffer sizes are counted in ELEMENTS of the call's
 *     dtype, never bytes.  Every buffer pointer must be aligned to the element
 *     size; 16-byte alignment gives the fastest path.
 *   - `stream` is a cudaStream_t passed as void* (NULL = the legacy default
 *     stream).  Collective calls are asynchronous on that stream; the library
 *     launches exactly one kernel per call.
 *   - Host-side validation errors return before anything is launched.
 *   - A context is not thread-safe: calls on one context must be issued from
 *     one host thread, and their launches must be ordered (same stream, or
 *     streams ordered by events).  Launches of one context that overlap on the
 *     GPU would share its flag words and race.
 *   - The first call for a new (layout pair, op, dtype, policy) derives a work
 *     list and uploads it with a synchronous copy; later calls reuse it.  Make
 *     that first call before capturing a stream into a CUDA graph.  A captured
 *     call may be replayed any number of times: the SNAC flag tags of each
 *     launch come from a device counter that every launch with flags advances,
 *     not from the captured parameters.
 */
#ifndef PURLIN_H
#define PURLIN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define PL_API __attribute__((visibility("default")))
#else
#define PL_API
#endif

#define PL_ABI_VERSION 2

/* ------------------------------------------------------------ status codes */

typedef int32_t pl_status;
#define PL_OK               0
#define PL_ERR_INVALID      1 /* null pointer, R outside 1..64, unknown dtype/op/policy value, misaligned buffer */
#define PL_ERR_LAYOUT       2 /* a name without its sources, several sources for COPY, SUM without exactly one source
                                 per rank, unequal element counts, a part outside its buffer */
#define PL_ERR_ALIAS        3 /* an output overlaps another output, or an input other than by exactly aliasing one of
                                 its own sources */
#define PL_ERR_NOMEM        4 /* device allocation failed, or the scratch ring is too small for the staged path */
#define PL_ERR_CUDA         5 /* a CUDA call failed; pl_ctx_cuda_error() returns the cudaError_t value */
#define PL_ERR_TIMEOUT      6 /* a bounded device wait expired (reported by pl_ctx_status) */
#define PL_ERR_UNSUPPORTED  7 /* a valid request this datapath does not handle: two strided regions of one
                                 transfer with different row lengths, or a reduction of PL_FP8 elements */

typedef int32_t pl_op;
#define PL_COPY 0 /* every output region receives the unique input region of the same name */
#define PL_SUM  1 /* every output region receives the rank-ordered sum of the R input regions of its name */
#define PL_MAX  2 /* every output region receives the rank-ordered maximum of the R input regions of its name:
                     start from rank 0's element and take rank r's when it compares greater (so a NaN counts
                     only from rank 0, and of +0 and -0 the lower rank's is kept).  Not in the pages, whose
                     reductions are sums; it uses the same layouts and work lists. */

typedef int32_t pl_dtype;
#define PL_BF16 0 /* bfloat16 in and out; sums accumulate in fp32 and round once (nearest-even) */
#define PL_FP32 1 /* float32 in and out; sums accumulate in fp32 */
#define PL_FP16 2 /* IEEE binary16 in and out; sums accumulate in fp32 and round once (nearest-even) */
#define PL_FP8  3 /* any one-byte element (e4m3, e5m2, bytes): PL_COPY only; PL_SUM / PL_MAX give
                     PL_ERR_UNSUPPORTED.  Every layout offset and length is then a byte count. */

/* --------------------------------------------------------------- policies */

/* Codesign policy (Figure 1 caption: policies tune execution without changing
 * the collective).  Zero-initialise and set only what you want to force;
 * pl_policy_default() gives that.  A NULL policy pointer means all-auto. */
typedef struct pl_policy {
    int32_t path;            /* PL_PATH_AUTO / PL_PATH_ZS / PL_PATH_STAGED */
    int32_t allreduce_form;  /* PL_AR_AUTO / PL_AR_FUSED / PL_AR_COMPOSED / PL_AR_NOTIFIED (SUM or MAX with
                                several outputs per name) */
    int32_t datapath;        /* PL_ATOM_AUTO / PL_ATOM_VECTOR / PL_ATOM_BULK / PL_ATOM_INLINE */
    int32_t ctas;            /* CTAs in the persistent grid; 0 = sized from the GPU's SM count and occupancy */
    int32_t stages;          /* depth of the bulk-copy shared-memory ring, 1..8; 0 = auto */
    int32_t reserved0;
    uint64_t chunk_bytes;    /* bytes per work item (the SNAC chunk); 0 = auto from the message size */
    uint64_t poll_timeout_ns;/* limit of every device wait; 0 = 2 seconds */
    int64_t debug_drop_notify; /* test hook, -1 = off: the Notify of the work item with this index is skipped,
                                  so its consumers' bounded waits expire and pl_ctx_status reports a timeout */
} pl_policy;

#define PL_PATH_AUTO    0 /* zero-staging */
#define PL_PATH_ZS      1 /* Purlin-ZS: consumers read source buffers directly and write the output layout */
#define PL_PATH_STAGED  2 /* Stage into the context's scratch ring, Notify, Consume from the ring */

#define PL_AR_AUTO      0 /* fused */
#define PL_AR_FUSED     1 /* one work item reduces a chunk and writes it to every output of its name */
#define PL_AR_COMPOSED  2 /* Figure 6: the owner's reduce of its partition, then the gather of the reduced
                             values from the owner's output to every other output.  Zero-staging composes
                             at the grain of one 16-byte vector: the thread that stores a reduced vector
                             into the owner's output reads it back from there and writes it to the other
                             ranks, so program order takes the place of the Notify and the reread is served
                             by L2.  The staged path composes per chunk with flags (as PL_AR_NOTIFIED). */
#define PL_AR_NOTIFIED  3 /* Figure 6 per chunk: the owner's reduce item Notifies a flag; a separate gather
                             item waits for it, reads the owner's chunk and writes the other ranks */

#define PL_ATOM_AUTO    0 /* inline for plans that qualify (below) and either move at most 320 MiB or reduce
                             every name's sources into one destination (the ReduceScatter shape); else the bulk
                             ring (8 stages) for copy-only plans moving >= 64 MiB whose regions are 16-byte
                             aligned or that write at least twice what they read; vector otherwise */
#define PL_ATOM_VECTOR  1 /* 16-byte vector loads and stores by every thread */
#define PL_ATOM_BULK    2 /* cp.async.bulk through a shared-memory ring for COPY work items: aligned sources
                             directly; sources at a byte shift from their destinations realigned in shared
                             memory between the bulk load and the bulk stores (4 stages or more); other
                             items use the vector datapath */
#define PL_ATOM_INLINE  3 /* the whole work list in the kernel's launch parameters, one work item per CTA, every
                             reference resolved to its pointer: no metadata loads, no barriers.  For zero-staging
                             plans of one-row regions at 16-byte aligned offsets whose items (at most 152) and
                             references (at most 2432) fit the parameter block.  Buffers not 16-byte aligned at
                             launch, and plans that do not qualify, run the same work list on the vector (or bulk)
                             datapath; so do lists with flags and the zero-staging PL_AR_COMPOSED form. */

/* Fills *pol with the all-auto policy (debug_drop_notify = -1). */
PL_API void pl_policy_default(pl_policy* pol);

/* ---------------------------------------------------------------- layouts */

/* One named region of one rank's buffer: `rows` rows of `len` elements, row i
 * starting at element `offset + i * row_stride`.  rows = 1 is a contiguous
 * region (row_stride is then ignored).  Elements of a region are ordered row
 * by row; two regions of the same name correspond element by element in that
 * order.  Names are arbitrary 64-bit identifiers. */
typedef struct pl_part {
    uint64_t name;
    uint64_t offset;
    uint64_t len;
    uint64_t rows;
    uint64_t row_stride;
} pl_part;

typedef struct pl_layout pl_layout;

/* A layout: for each rank r < R, nparts[r] consecutive entries of `parts`.
 * The library copies what it needs; the caller keeps ownership of its arrays.
 * Errors: PL_ERR_INVALID (null pointers, R outside 1..64, rows = 0, a strided
 * region with row_stride < len, a negative count). */
PL_API pl_status pl_layout_create(pl_layout** layout, int R, const int* nparts, const pl_part* parts);
PL_API pl_status pl_layout_destroy(pl_layout* layout);
/* Rank count and number of parts of a layout (for checks by the caller). */
PL_API pl_status pl_layout_info(const pl_layout* layout, int* R, int* total_parts);

/* Layout builders for the collectives of the pages.  `lens` has R entries
 * (partition lengths; equal or variable); `lens_rxr` is R x R row-major
 * (row = source rank, column = destination rank).  Partition names: k for
 * partition k; r * R + j for AllToAll's (source r, destination j) pair. */

/* AllGather(V) input / ReduceScatter(V) output: rank k holds one region named
 * k, lens[k] long, at offset 0 (Figure 4: y_k at rank k). */
PL_API pl_status pl_layout_rank_owned(pl_layout** layout, int R, const uint64_t* lens);
/* AllGather(V) output, ReduceScatter(V) input, AllReduce input and output:
 * every rank holds regions 0..R-1 at prefix-sum offsets (Figure 4: all y_k in
 * rank order). */
PL_API pl_status pl_layout_partitioned(pl_layout** layout, int R, const uint64_t* lens);
/* In-place ReduceScatter(V) output: rank k holds region k at offset
 * lens[0] + ... + lens[k-1] of its own buffer, so the output buffers may be
 * the input buffers (zero-staging, output in place). */
PL_API pl_status pl_layout_rank_owned_inplace(pl_layout** layout, int R, const uint64_t* lens);
/* AllToAll(V) input: rank r holds regions r*R + j (j = 0..R-1) at prefix
 * offsets of row r of lens_rxr (Figure 4 bottom). */
PL_API pl_status pl_layout_alltoall_in(pl_layout** layout, int R, const uint64_t* lens_rxr);
/* AllToAll(V) output: rank j holds regions r*R + j (r = 0..R-1, source order)
 * at prefix offsets of column j of lens_rxr. */
PL_API pl_status pl_layout_alltoall_out(pl_layout** layout, int R, const uint64_t* lens_rxr);
/* Ulysses sequence -> head re-partition (Table 2), input: rank r holds a
 * [S, H, D] tensor; region r*R + j is heads [j*H/R, (j+1)*H/R): S rows of
 * (H/R)*D elements with row stride H*D.  H must be a multiple of R. */
PL_API pl_status pl_layout_ulysses_in(pl_layout** layout, int R, uint64_t S, uint64_t H, uint64_t D);
/* Ulysses output: rank j holds [R*S, H/R, D]; region r*R + j is the
 * contiguous block of S*(H/R)*D elements at offset r*S*(H/R)*D. */
PL_API pl_status pl_layout_ulysses_out(pl_layout** layout, int R, uint64_t S, uint64_t H, uint64_t D);

/* ---------------------------------------------------------------- context */

typedef struct pl_ctx pl_ctx;

/* Creates a context bound to CUDA device `device`.  The context owns the
 * device-side SNAC state (flag words, the status word, work-list copies) and a
 * scratch ring of `scratch_bytes` bytes for the staged path (0 = zero-staging
 * only).  The caller's current device is restored before returning.
 * Errors: PL_ERR_INVALID, PL_ERR_CUDA (no such device), PL_ERR_NOMEM. */
PL_API pl_status pl_ctx_create(pl_ctx** ctx, int device, uint64_t scratch_bytes);
/* Synchronises the context's device, then frees everything it owns. */
PL_API pl_status pl_ctx_destroy(pl_ctx* ctx);
/* Waits for `stream`, then reads and clears the device status word:
 * PL_OK, or PL_ERR_TIMEOUT when a bounded wait of an earlier launch expired
 * (the context's flag state is then reset so later calls start clean). */
PL_API pl_status pl_ctx_status(pl_ctx* ctx, void* stream);
/* The cudaError_t of the last failing CUDA call on this context (0 if none). */
PL_API int pl_ctx_cuda_error(const pl_ctx* ctx);
/* Number of kernels this context has launched since its creation. */
PL_API uint64_t pl_ctx_launches(const pl_ctx* ctx);

/* ------------------------------------------------------------ collectives */

/* Runs the collective named by (in_layout, out_layout, op) over R logical
 * ranks (abstract; Figure 4):
 *   COPY: every output region named p receives the unique input region named p;
 *   SUM:  every output region named p receives, element by element, the fp32
 *         sum over ranks 0..R-1 (in that order, starting from rank 0's value)
 *         of the input regions named p, one per rank, rounded once to dtype.
 * in_bufs[r] / out_bufs[r]: device buffers of rank r holding in_counts[r] /
 * out_counts[r] elements (a rank with count 0 may pass NULL).  Output
 * elements that no region names are left untouched.
 * An output region may coincide exactly with one of its own sources (same
 * address and shape), e.g. ReduceScatter in place; any other overlap between
 * an output and an input or another output is PL_ERR_ALIAS.
 * `policy` may be NULL (all auto).  Asynchronous on `stream`; exactly one
 * kernel launch.  Device-side waits that expire are reported by
 * pl_ctx_status(), not here. */
PL_API pl_status pl_collective(pl_ctx* ctx, const pl_layout* in_layout, const pl_layout* out_layout,
                               pl_op op, pl_dtype dtype, int R,
                               void* const* in_bufs, const uint64_t* in_counts,
                               void* const* out_bufs, const uint64_t* out_counts,
                               const pl_policy* policy, void* stream);

/* AllReduce of `count` elements per rank (Table 2, tensor-parallel row;
 * Figure 6): out_bufs[r][i] = rank-ordered sum over ranks of in_bufs[*][i]
 * for every r, by ReduceScatter then AllGather over R partitions (the first
 * R-1 of count/R elements, the last the rest).  policy->allreduce_form picks
 * the fused form (default) or a composed form of Figure 6 (PL_AR_COMPOSED,
 * PL_AR_NOTIFIED).
 * out_bufs may equal in_bufs (in place).  One kernel launch. */
PL_API pl_status pl_allreduce(pl_ctx* ctx, pl_dtype dtype, int R, uint64_t count,
                              void* const* in_bufs, void* const* out_bufs,
                              const pl_policy* policy, void* stream);

/* pl_allreduce with the reduction named: op = PL_SUM (the same call) or
 * PL_MAX (out_bufs[r][i] = rank-ordered maximum over ranks of in_bufs[*][i]).
 * PL_COPY returns PL_ERR_INVALID; PL_FP8 returns PL_ERR_UNSUPPORTED. */
PL_API pl_status pl_allreduce_op(pl_ctx* ctx, pl_op op, pl_dtype dtype, int R, uint64_t count,
                                 void* const* in_bufs, void* const* out_bufs,
                                 const pl_policy* policy, void* stream);

/* AllReduce that allocates no device memory.  The paper has no counterpart:
 * this entry point exists for callers that cannot call cudaMalloc -- a process
 * that reserves its device memory budget once at start-up and may not grow it,
 * a plug-in that does not own the process's device allocator, or code on a
 * latency path where an allocation (which can synchronise the device) is not
 * acceptable.  The result is the same as pl_allreduce with a staged policy:
 * out_bufs[r][i] = rank-ordered fp32 sum over ranks of in_bufs[*][i], rounded
 * once to dtype, for every r (out_bufs may equal in_bufs).  dtype is
 * PL_BF16, PL_FP16 or PL_FP32.
 *
 * No context: the flag words, the derived work list and the staging ring live
 * in one file-scope device array of 32 MiB that every GPU loading the library
 * holds until the process exits.  Limits: R <= 8 and count * element size
 * <= 256 MiB per rank; larger requests return PL_ERR_NOMEM before anything
 * runs.  Buffer errors return PL_ERR_INVALID / PL_ERR_ALIAS like pl_allreduce.
 *
 * The call works on the current CUDA device.  Its first call on a device also
 * looks up the array's device address there (cudaGetSymbolAddress); make that
 * first call before any stream capture.  Every call clears the array's flag
 * words on `stream` and launches one kernel there.  When its work list differs
 * from the one the array holds (the first call, or a new R, count or dtype),
 * it first copies the list into the array on `stream`, from a host image the
 * library keeps per device; that copy is from pageable host memory, so the
 * call waits for the work already queued on `stream` before it returns.  Calls issued in order on one stream are safe; calls whose work
 * overlaps on the GPU (other streams, other host threads) share the array and
 * race.  wait = 0 returns without waiting for the kernel and reports no device
 * error: the next call clears the status word, so a bounded wait that expired
 * in a wait = 0 call goes unreported.  wait != 0 also waits for `stream` and
 * returns the device status (PL_OK, or PL_ERR_TIMEOUT if a bounded wait
 * expired). */
PL_API pl_status pl_allreduce_noalloc(pl_dtype dtype, int R, uint64_t count, void* const* in_bufs,
                                      void* const* out_bufs, int wait, void* stream);

/* ----------------------------------------------------- plan introspection */

/* The SNAC work list derived from a layout pair (abstract: orchestration
 * derived from the specification, no hand-written schedule), for tests and
 * tools.  Host only: creating and reading a plan makes no CUDA call.
 * num_sms sizes the persistent grid as pl_collective would on such a GPU;
 * scratch_bytes is the ring that the staged path may use. */
typedef struct pl_plan pl_plan;

typedef struct pl_plan_stats {
    uint64_t items;        /* work items, in the order the device claims them */
    uint64_t refs;         /* region references (sources and destinations of items) */
    uint64_t syncs;        /* SNAC flag operations */
    uint64_t flags;        /* flag words the plan uses */
    uint64_t chunk_elems;  /* elements per chunk */
    uint64_t slots;        /* scratch ring slots per rank (staged path; 0 otherwise) */
    uint64_t slot_elems;   /* elements per slot */
    int32_t ctas;          /* persistent grid size (the inline form: one CTA per item) */
    int32_t threads;       /* threads per CTA */
    int32_t uses_tickets;  /* 1 = items are claimed in order through a device counter */
    int32_t path;          /* resolved PL_PATH_* */
    uint64_t bytes_read;   /* device bytes the plan reads per launch (algorithmic + staging) */
    uint64_t bytes_written;/* device bytes the plan writes per launch */
    int32_t datapath;      /* resolved PL_ATOM_VECTOR / PL_ATOM_BULK / PL_ATOM_INLINE (for 16-byte aligned buffers) */
    int32_t reserved0;
} pl_plan_stats;

/* Kinds of work items (SNAC steps). */
#define PL_ITEM_MOVE     0 /* zero-staging Consume: sources -> destinations */
#define PL_ITEM_STAGE    1 /* Stage: a source chunk -> a scratch slot, then Notify */
#define PL_ITEM_CONSUME  2 /* Consume: wait for notified chunks, copy or reduce them into destinations */
#define PL_ITEM_COMPOSE  3 /* zero-staging composed step (PL_AR_COMPOSED): reduce the sources into
                              destination 0, the partition's owner; then read the reduced values back
                              from destination 0 and write them to the other destinations */

/* Spaces a region reference points into. */
#define PL_SPACE_IN      0 /* in_bufs[index] */
#define PL_SPACE_OUT     1 /* out_bufs[index] */
#define PL_SPACE_SCRATCH 2 /* the context's scratch ring (index 0) */

/* SNAC flag operations. Tags are per launch: use u of a flag is tag u + 1. */
#define PL_SYNC_WAIT_FULL  0 /* wait until flag `flag` has been notified for use `use` (acquire) */
#define PL_SYNC_WAIT_FREE  1 /* wait until every consumer of use `use` of flag `flag` has finished (acquire) */
#define PL_SYNC_NOTIFY     2 /* mark use `use` of flag `flag` as filled (release) */
#define PL_SYNC_CREDIT     3 /* count one consumer of use `use`; the `count`-th frees the slot (release) */

typedef struct pl_plan_item {
    int32_t kind, op;
    int32_t nsrc, ndst;
    int32_t nwait, npost;
    uint64_t rows, cols;   /* every reference covers rows x cols elements */
} pl_plan_item;

typedef struct pl_plan_ref {
    int32_t space, index;
    uint64_t offset;       /* element offset of row 0 */
    uint64_t stride;       /* elements between rows */
} pl_plan_ref;

typedef struct pl_plan_sync {
    int32_t type;
    uint32_t flag, use, count;
} pl_plan_sync;

PL_API pl_status pl_plan_create(pl_plan** plan, const pl_layout* in_layout, const pl_layout* out_layout,
                                pl_op op, pl_dtype dtype, int R, const pl_policy* policy,
                                int num_sms, uint64_t scratch_bytes);
PL_API pl_status pl_plan_destroy(pl_plan* plan);
PL_API pl_status pl_plan_get_stats(const pl_plan* plan, pl_plan_stats* stats);
/* Item i, its references (sources first, then destinations) and its flag
 * operations (waits first, then notifies and credits). */
PL_API pl_status pl_plan_get_item(const pl_plan* plan, uint64_t i, pl_plan_item* item,
                                  pl_plan_ref* refs, int max_refs, pl_plan_sync* syncs, int max_syncs);

/* ------------------------------------------------------------------- misc */

PL_API const char* pl_status_str(pl_status status);
PL_API int pl_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* PURLIN_H */
