// The Atom datapath and the device side of SNAC for sm_103a.
//
// "Purlin: Separating Orchestration from the Datapath of Collectives":
//   - abstract: the Atom provides the two data-movement primitives of
//     collectives, copy and reduce; SNAC (Stage, Notify, And Consume) is the
//     orchestration above it;
//   - Table 1 ("Compatibility"): a datapath built on vectorised loads and
//     stores; Figure 11 caption: a pipelined copy with 1 to 8 stages.
//
// One persistent kernel executes a work list (see snac.h).  Every work item
// is "wait on flags -> move -> notify / credit flags", and the move is either
// a copy of one source into up to 64 destinations or a rank-ordered reduction
// (the fp32 sum, or the maximum) of up to 64 sources written to up to 64
// destinations.  The kernel is a template over the element type; atom.cu,
// atom_fp16.cu, atom_fp32.cu and atom_fp8.cu each instantiate one.  Items are
// claimed in index order (a device counter) whenever an item waits on another,
// so a waiting CTA only ever waits for items that were claimed before it and
// are therefore running: the grid makes progress without co-residency.  Every
// wait is bounded by a timeout on %globaltimer and an iteration cap; a wait
// that gives up records PL_ERR_TIMEOUT in the status word and raises an abort
// flag that makes every other wait give up too, so the kernel always returns.
#pragma once

#include "snac.h"

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>

namespace purlin {
namespace {

constexpr int kStatusTimeout = 6;  // PL_ERR_TIMEOUT
constexpr int kCopyUnroll = 8; // 16-byte vectors a thread keeps in flight in the copy bodies

// ------------------------------------------------------- memory-model helpers

__device__ __forceinline__ unsigned long long ld_acquire(const unsigned long long* p)
{
    unsigned long long v;
    asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void st_release(unsigned long long* p, unsigned long long v)
{
    asm volatile("st.release.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

__device__ __forceinline__ unsigned int atom_add_acq_rel(unsigned int* p, unsigned int v)
{
    unsigned int old;
    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
    return old;
}

__device__ __forceinline__ void st_relaxed_u32(unsigned int* p, unsigned int v)
{
    asm volatile("st.relaxed.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ int ld_relaxed_s32(const int* p)
{
    int v;
    asm volatile("ld.relaxed.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ unsigned long long global_ns()
{
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Streaming 16-byte load that is served from L2 (data may have been written
// by another CTA of this launch after a flag acquire).
__device__ __forceinline__ uint4 ld16(const char* p) { return __ldcg(reinterpret_cast<const uint4*>(p)); }
#if defined(PL_STORE_STREAMING)
// Developer build option: evict-first stores for outputs nobody rereads.
__device__ __forceinline__ void st16(char* p, uint4 v) { __stcs(reinterpret_cast<uint4*>(p), v); }
#else
__device__ __forceinline__ void st16(char* p, uint4 v) { *reinterpret_cast<uint4*>(p) = v; }
#endif

// ------------------------------------------------------------- bounded waits

__device__ void give_up(const LaunchArgs& a)
{
    atomicCAS(a.st.status, 0, kStatusTimeout);
    atomicExch(a.st.abort, 1);
}

// Waits until *flag >= target.  false: the wait expired or another wait did.
__device__ bool wait_at_least(const unsigned long long* flag, unsigned long long target, const LaunchArgs& a)
{
    const unsigned long long t0 = global_ns();
    // The cap bounds the loop even if %globaltimer stalled: every iteration
    // sleeps, and 2^26 iterations exceed any sensible timeout.
    const unsigned int cap = 1u << 26;
    for (unsigned int it = 0; it < cap; ++it) {
        if (ld_acquire(flag) >= target)
            return true;
        if ((it & 31) == 31) {
            if (ld_relaxed_s32(a.st.abort))
                return false;
            if (global_ns() - t0 > a.timeout_ns)
                break;
        }
        __nanosleep(it < 64 ? 32 : 256);
    }
    give_up(a);
    return false;
}

// The tag of use `use` of a flag in the launch of epoch `epoch`.
__device__ __forceinline__ unsigned long long tag(unsigned long long epoch, unsigned int use)
{
    return (epoch << 24) | (unsigned long long)(use + 1u);
}

// Warp 0 of the CTA: every wait of the item, one flag per lane (lanes take
// flags lane, lane + 32, ...), so an item's waits overlap instead of costing
// one round trip each.  Returns, in every lane, whether all waits passed.
__device__ bool run_waits(const LaunchArgs& a, const Item& it, int lane, unsigned long long epoch)
{
    bool ok = ld_relaxed_s32(a.st.abort) == 0;
    for (unsigned k = (unsigned)lane; ok && k < it.nwait; k += 32) {
        const Sync s = a.syncs[it.sync + k];
        const unsigned long long* f = s.type == kWaitFull ? a.st.full + s.flag : a.st.done + s.flag;
        ok = wait_at_least(f, tag(epoch, s.use), a);
    }
    return __all_sync(0xffffffffu, ok) != 0;
}

// Warp 0 of the CTA, after a barrier that follows the item's stores: the
// notifies and credits of the item, one flag per lane.  The CTA's writes are
// ordered before each posting lane's release by the barrier, and a release
// (st.release / atom.acq_rel at gpu scope) is cumulative, so a consumer whose
// acquire reads the tag sees them: no separate fence is needed.
__device__ void run_posts(const LaunchArgs& a, const Item& it, unsigned index, int lane, unsigned long long epoch)
{
    for (unsigned k = (unsigned)lane; k < it.npost; k += 32) {
        const Sync s = a.syncs[it.sync + it.nwait + k];
        if (s.type == kNotify) {
            if ((long long)index == a.drop_notify)
                continue;  // test hook: consumers of this item will time out
            st_release(a.st.full + s.flag, tag(epoch, s.use));
        } else if (s.type == kCredit) {
            unsigned old = atom_add_acq_rel(a.st.count + s.flag, 1u);
            if (old + 1u == s.count) {
                st_relaxed_u32(a.st.count + s.flag, 0u);
                st_release(a.st.done + s.flag, tag(epoch, s.use));
            }
        }
    }
}

// ------------------------------------------------- bulk-copy (TMA) primitives

constexpr unsigned kBulkPiece = 16384;  // bytes per ring stage
constexpr unsigned kBulkMin = 4096;     // smaller bodies use the vector path

__device__ __forceinline__ uint32_t smem_u32(const void* p)
{
    return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(unsigned long long* bar, unsigned count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(unsigned long long* bar, unsigned bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(unsigned long long* bar, unsigned parity)
{
    uint32_t ok;
    asm volatile("{\n\t.reg .pred p;\n\t"
                 "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
                 "selp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(ok)
                 : "r"(smem_u32(bar)), "r"(parity)
                 : "memory");
    return ok != 0;
}

// Global -> shared bulk copy that completes `bytes` transactions on `bar`.
__device__ __forceinline__ void bulk_g2s(void* smem, const void* g, unsigned bytes, unsigned long long* bar)
{
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     smem_u32(smem)),
                 "l"(g), "r"(bytes), "r"(smem_u32(bar))
                 : "memory");
}

// Shared -> global bulk copy in the current bulk group.
__device__ __forceinline__ void bulk_s2g(void* g, const void* smem, unsigned bytes)
{
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(g), "r"(smem_u32(smem)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read0() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read1() { asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
__device__ __forceinline__ void fence_proxy_async() { asm volatile("fence.proxy.async.global;" ::: "memory"); }
__device__ __forceinline__ void fence_proxy_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// At most n bulk groups of this thread still reading their shared memory
// (n >= 7 waits for at most 7).
__device__ __forceinline__ void bulk_wait_read_n(int n)
{
    switch (n) {
    case 0: asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); break;
    case 1: asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory"); break;
    case 2: asm volatile("cp.async.bulk.wait_group.read 2;" ::: "memory"); break;
    case 3: asm volatile("cp.async.bulk.wait_group.read 3;" ::: "memory"); break;
    case 4: asm volatile("cp.async.bulk.wait_group.read 4;" ::: "memory"); break;
    case 5: asm volatile("cp.async.bulk.wait_group.read 5;" ::: "memory"); break;
    case 6: asm volatile("cp.async.bulk.wait_group.read 6;" ::: "memory"); break;
    default: asm volatile("cp.async.bulk.wait_group.read 7;" ::: "memory"); break;
    }
}

__device__ __forceinline__ uint4 lds16(const char* p) { return *reinterpret_cast<const uint4*>(p); }
__device__ __forceinline__ void sts16(char* p, uint4 v) { *reinterpret_cast<uint4*>(p) = v; }

// Bounded wait for the phase `parity` of an mbarrier.
__device__ bool mbar_wait(unsigned long long* bar, unsigned parity, const LaunchArgs& a)
{
    const unsigned long long t0 = global_ns();
    for (unsigned it = 0; it < (1u << 26); ++it) {
        if (mbar_try_wait(bar, parity))
            return true;
        if ((it & 255) == 255 && global_ns() - t0 > a.timeout_ns)
            break;
    }
    give_up(a);
    return false;
}

// The CTA's bulk-copy ring: `stages` buffers of kBulkPiece bytes, one mbarrier
// each.  bulk_copy (thread 0 alone) tracks in `phase` the parity each stage's
// barrier will complete next.  bulk_shift_copy (every thread) uses the same
// buffers in pairs and its own barriers `sbar` with parities `sphase`, which
// every thread keeps identically.
//
// Pieces are numbered across the items of the CTA (`gcopy` for bulk_copy,
// `gshift` for bulk_shift_copy; each piece commits one bulk group of stores),
// so that the ring runs on from one item into the next: an item that posts no
// flags returns without waiting for its stores, which drain while the next
// item's first loads are in flight, and the next item reuses a buffer only
// once the stores that read it are done with it.  Switching between the two
// functions (`mode`) first waits until every store has read the ring.
struct BulkRing {
    char* buf;
    unsigned long long* bar;
    int stages;
    unsigned phase;
    unsigned long long* sbar;
    unsigned sphase;
    bool drain;       // the current item notifies or credits flags after its move
    int mode;         // 0 none, 1 bulk_copy, 2 bulk_shift_copy: the last user of the ring
    unsigned gcopy;   // thread 0: pieces bulk_copy has stored so far
    unsigned gshift;  // every thread: pieces bulk_shift_copy has stored so far
};

// End of a bulk move.  An item that posts flags waits until every store has
// landed and orders the async-proxy stores before the generic release that
// follows.  Any other item returns at once: nothing in the launch reads what
// it wrote, and the kernel waits for all stores before it exits.
__device__ __forceinline__ void bulk_finish(const BulkRing& bk)
{
    if (bk.drain) {
        bulk_wait_all();
        fence_proxy_async();
    }
}
constexpr int kShiftMaxDepth = kBulkMaxStages / 2;

// ------------------------------------------------------------- element math

// Element types, keyed by the launch's dtype code.  S is the element size in
// bytes; to_f / from_f widen to fp32 exactly and round back to nearest-even.
template <int DT> struct Elem;

template <> struct Elem<kDtBf16> {
    static constexpr int S = 2;
    static constexpr bool kReducible = true;
    static __device__ __forceinline__ float to_f(uint32_t h) { return __uint_as_float(h << 16); }
    static __device__ __forceinline__ uint32_t from_f(float f)
    {
        return (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(f));
    }
    static __device__ __forceinline__ uint32_t load(const char* p) { return __ldcg(reinterpret_cast<const unsigned short*>(p)); }
    static __device__ __forceinline__ void store(char* p, uint32_t v) { *reinterpret_cast<unsigned short*>(p) = (unsigned short)v; }
};

template <> struct Elem<kDtFp16> {
    static constexpr int S = 2;
    static constexpr bool kReducible = true;
    static __device__ __forceinline__ float to_f(uint32_t h) { return __half2float(__ushort_as_half((unsigned short)h)); }
    static __device__ __forceinline__ uint32_t from_f(float f) { return (uint32_t)__half_as_ushort(__float2half_rn(f)); }
    static __device__ __forceinline__ uint32_t load(const char* p) { return __ldcg(reinterpret_cast<const unsigned short*>(p)); }
    static __device__ __forceinline__ void store(char* p, uint32_t v) { *reinterpret_cast<unsigned short*>(p) = (unsigned short)v; }
};

template <> struct Elem<kDtFp32> {
    static constexpr int S = 4;
    static constexpr bool kReducible = true;
    static __device__ __forceinline__ float to_f(uint32_t w) { return __uint_as_float(w); }
    static __device__ __forceinline__ uint32_t from_f(float f) { return __float_as_uint(f); }
    static __device__ __forceinline__ uint32_t load(const char* p) { return __ldcg(reinterpret_cast<const unsigned int*>(p)); }
    static __device__ __forceinline__ void store(char* p, uint32_t v) { *reinterpret_cast<unsigned int*>(p) = v; }
};

// One-byte elements (an fp8 format, or any byte): moved, never reduced.
template <> struct Elem<kDtFp8> {
    static constexpr int S = 1;
    static constexpr bool kReducible = false;
    static __device__ __forceinline__ uint32_t load(const char* p) { return __ldcg(reinterpret_cast<const unsigned char*>(p)); }
    static __device__ __forceinline__ void store(char* p, uint32_t v) { *reinterpret_cast<unsigned char*>(p) = (unsigned char)v; }
};

// One step of the rank-ordered reduction: the fp32 sum, or the maximum that
// takes the next rank's value only when it is greater (a NaN never is, so a
// NaN survives only from rank 0, and of +0 and -0 the earlier rank's stays).
template <bool MAXOP>
__device__ __forceinline__ float combine(float acc, float x)
{
    if constexpr (MAXOP)
        return x > acc ? x : acc;
    else
        return __fadd_rn(acc, x);
}

// Two lanes of the sum at once: add.rn.f32x2 is two IEEE fp32 additions,
// each rounded to nearest even with subnormals kept, so the result is that of
// two __fadd_rn, in half the instructions.
__device__ __forceinline__ void add2_rn(float& a0, float& a1, float b0, float b1)
{
    asm("{\n\t.reg .b64 pa, pb;\n\t"
        "mov.b64 pa, {%0, %1};\n\t"
        "mov.b64 pb, {%2, %3};\n\t"
        "add.rn.f32x2 pa, pa, pb;\n\t"
        "mov.b64 {%0, %1}, pa;\n\t}"
        : "+f"(a0), "+f"(a1)
        : "f"(b0), "f"(b1));
}

// Accumulators of one 16-byte vector (8 two-byte or 4 four-byte lanes).  The
// maximum of widened values is exactly one of the inputs, so rounding it back
// reproduces that element.
template <int DT, bool MAXOP> struct Acc {
    using EL = Elem<DT>;
    static constexpr int S = EL::S;
    static constexpr int N = 16 / S;
    static_assert(EL::kReducible, "one-byte elements are never reduced");
    float v[N];
    static __device__ __forceinline__ float lane(const uint32_t (&w)[4], int i)
    {
        if constexpr (S == 2)
            return EL::to_f((i & 1) ? (w[i >> 1] >> 16) : (w[i >> 1] & 0xFFFFu));
        else
            return EL::to_f(w[i]);
    }
    __device__ __forceinline__ void set(uint4 x)
    {
        const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
        for (int i = 0; i < N; ++i)
            v[i] = lane(w, i);
    }
    __device__ __forceinline__ void add(uint4 x)
    {
        const uint32_t w[4] = {x.x, x.y, x.z, x.w};
        if constexpr (MAXOP) {
#pragma unroll
            for (int i = 0; i < N; ++i)
                v[i] = combine<true>(v[i], lane(w, i));
        } else {
#pragma unroll
            for (int i = 0; i < N; i += 2)
                add2_rn(v[i], v[i + 1], lane(w, i), lane(w, i + 1));
        }
    }
    __device__ __forceinline__ uint4 pack() const
    {
        uint32_t w[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            if constexpr (S == 2)
                w[i] = EL::from_f(v[2 * i]) | (EL::from_f(v[2 * i + 1]) << 16);
            else
                w[i] = EL::from_f(v[i]);
        }
        return make_uint4(w[0], w[1], w[2], w[3]);
    }
};

// The 16 bytes that start q bytes into the 32-byte pair (lo, hi), 0 <= q < 16.
// q is the same for every vector of a row (a warp-uniform branch): the word
// offset q / 4 picks the words, and four funnel shifts by (q mod 4) bytes
// join them.
__device__ __forceinline__ uint4 realign(uint4 lo, uint4 hi, int q)
{
    const unsigned sh = (unsigned)(q & 3) * 8u;
    switch (q >> 2) {
    case 0:
        return make_uint4(__funnelshift_r(lo.x, lo.y, sh), __funnelshift_r(lo.y, lo.z, sh),
                          __funnelshift_r(lo.z, lo.w, sh), __funnelshift_r(lo.w, hi.x, sh));
    case 1:
        return make_uint4(__funnelshift_r(lo.y, lo.z, sh), __funnelshift_r(lo.z, lo.w, sh),
                          __funnelshift_r(lo.w, hi.x, sh), __funnelshift_r(hi.x, hi.y, sh));
    case 2:
        return make_uint4(__funnelshift_r(lo.z, lo.w, sh), __funnelshift_r(lo.w, hi.x, sh),
                          __funnelshift_r(hi.x, hi.y, sh), __funnelshift_r(hi.y, hi.z, sh));
    default:
        return make_uint4(__funnelshift_r(lo.w, hi.x, sh), __funnelshift_r(hi.x, hi.y, sh),
                          __funnelshift_r(hi.y, hi.z, sh), __funnelshift_r(hi.z, hi.w, sh));
    }
}

// ------------------------------------------------------------ the datapath

// Per-item shared state: byte pointers of row 0 and byte strides between rows.
struct ItemShared {
    const char* src[kMaxRanks];
    char* dst[kMaxRanks];
    unsigned long long sstride[kMaxRanks];
    unsigned long long dstride[kMaxRanks];
};

// Row pointer of source s / destination d.
#define SRC_ROW(sh, s, row) ((sh).src[s] + (size_t)(row) * (sh).sstride[s])
#define DST_ROW(sh, d, row) ((sh).dst[d] + (size_t)(row) * (sh).dstride[d])

// Copy of nv 16-byte vectors from one source to every destination in `mask`,
// both 16-byte aligned at `body` (the kernels for aligned plans).  U vectors
// in flight per thread.
template <int U>
__device__ __forceinline__ void copy_body(const ItemShared& sh, unsigned long long mask, unsigned row, size_t body,
                                          unsigned nv, int tid, int nthr)
{
    const char* src = SRC_ROW(sh, 0, row) + body;
    const unsigned step = (unsigned)nthr * U;
    for (unsigned v0 = tid; v0 < nv; v0 += step) {
        uint4 x[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const unsigned v = v0 + u * nthr;
            if (v < nv)
                x[u] = ld16(src + (size_t)v * 16);
        }
#pragma unroll 1
        for (unsigned long long m = mask; m; m &= m - 1) {
            const int d = __ffsll((long long)m) - 1;
            char* dst = DST_ROW(sh, d, row) + body;
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const unsigned v = v0 + u * nthr;
                if (v < nv)
                    st16(dst + (size_t)v * 16, x[u]);
            }
        }
    }
}

// Rank-ordered reduction (fp32 sum or maximum) of nsrc aligned sources over
// nv vectors, rounded once, stored to every destination in `mask`: U vectors
// x G sources (U * G = 8 loads) in flight per thread.
template <int DT, bool MAXOP, int U>
__device__ __forceinline__ void sum_aligned(const ItemShared& sh, int nsrc, unsigned long long mask, unsigned row,
                                            size_t body, unsigned nv, int tid, int nthr)
{
    constexpr int G = 8 / U;
    const unsigned step = (unsigned)nthr * U;
    for (unsigned v0 = tid; v0 < nv; v0 += step) {
        Acc<DT, MAXOP> acc[U];
        for (int s0 = 0; s0 < nsrc; s0 += G) {
            uint4 x[U][G];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const unsigned v = v0 + u * nthr;
#pragma unroll
                for (int g = 0; g < G; ++g)
                    if (s0 + g < nsrc && v < nv)
                        x[u][g] = ld16(SRC_ROW(sh, s0 + g, row) + body + (size_t)v * 16);
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
#pragma unroll
                for (int g = 0; g < G; ++g) {
                    if (s0 + g < nsrc) {
                        if (s0 + g == 0)
                            acc[u].set(x[u][g]);
                        else
                            acc[u].add(x[u][g]);
                    }
                }
            }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const unsigned v = v0 + u * nthr;
            if (v < nv) {
                const uint4 out = acc[u].pack();
#pragma unroll 1
                for (unsigned long long m = mask; m; m &= m - 1) {
                    const int d = __ffsll((long long)m) - 1;
                    st16(DST_ROW(sh, d, row) + body + (size_t)v * 16, out);
                }
            }
        }
    }
}

// The same reduction when the sources sit at different byte shifts from the
// aligned destinations (rare): each source's 16 bytes are loaded as two
// aligned vectors and realigned, one source at a time.
template <int DT, bool MAXOP>
__device__ __forceinline__ void sum_mixed(const ItemShared& sh, int nsrc, unsigned long long mask, unsigned row,
                                          size_t body, unsigned nv, int tid, int nthr)
{
    for (unsigned v = tid; v < nv; v += nthr) {
        Acc<DT, MAXOP> acc;
        for (int s = 0; s < nsrc; ++s) {
            const char* p = SRC_ROW(sh, s, row) + body + (size_t)v * 16;
            const int q = (int)(reinterpret_cast<uintptr_t>(p) & 15u);
            const uint4 lo = ld16(p - q);
            const uint4 x = q ? realign(lo, ld16(p - q + 16), q) : lo;
            if (s == 0)
                acc.set(x);
            else
                acc.add(x);
        }
        const uint4 out = acc.pack();
#pragma unroll 1
        for (unsigned long long m = mask; m; m &= m - 1) {
            const int d = __ffsll((long long)m) - 1;
            st16(DST_ROW(sh, d, row) + body + (size_t)v * 16, out);
        }
    }
}

// Figure 6 at the grain of one vector (kCompose items, aligned plans): the
// rank-ordered reduction of nv vectors is stored to destination 0, the
// partition's owner; the same thread then reads each reduced vector back from
// the owner's output and writes it to the other destinations in `mask`.  A
// thread's load of an address it stored returns what it stored (program
// order), so no flag is needed between the reduce and the gather, and the
// reread is served by L2 (measured on GB300: DRAM reads of an AllReduce 8T,
// as with the fused form).  The reread of one step is issued with the source
// loads of the next, so its latency hides behind theirs.  U vectors x G
// sources in flight per thread, as in sum_aligned.
template <int DT, bool MAXOP, int U>
__device__ __forceinline__ void sum_compose(const ItemShared& sh, int nsrc, unsigned long long mask, unsigned row,
                                            size_t body, unsigned nv, int tid, int nthr)
{
    constexpr int G = 8 / U;
    const unsigned step = (unsigned)nthr * U;
    char* const own = DST_ROW(sh, 0, row) + body;
    const unsigned long long rest = mask & ~1ull;
    unsigned prev = ~0u;  // the first vector of this thread's previous step
    for (unsigned v0 = tid;; v0 += step) {
        const bool cur = v0 < nv;
        uint4 back[U];
        if (prev != ~0u) {
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const unsigned v = prev + u * nthr;
                if (v < nv)
                    back[u] = ld16(own + (size_t)v * 16);
            }
        }
        if (cur) {
            Acc<DT, MAXOP> acc[U];
            for (int s0 = 0; s0 < nsrc; s0 += G) {
                uint4 x[U][G];
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const unsigned v = v0 + u * nthr;
#pragma unroll
                    for (int g = 0; g < G; ++g)
                        if (s0 + g < nsrc && v < nv)
                            x[u][g] = ld16(SRC_ROW(sh, s0 + g, row) + body + (size_t)v * 16);
                }
#pragma unroll
                for (int u = 0; u < U; ++u) {
#pragma unroll
                    for (int g = 0; g < G; ++g) {
                        if (s0 + g < nsrc) {
                            if (s0 + g == 0)
                                acc[u].set(x[u][g]);
                            else
                                acc[u].add(x[u][g]);
                        }
                    }
                }
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const unsigned v = v0 + u * nthr;
                if (v < nv)
                    st16(own + (size_t)v * 16, acc[u].pack());
            }
        }
        if (prev != ~0u) {
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const unsigned v = prev + u * nthr;
                if (v < nv) {
#pragma unroll 1
                    for (unsigned long long m = rest; m; m &= m - 1) {
                        const int d = __ffsll((long long)m) - 1;
                        st16(DST_ROW(sh, d, row) + body + (size_t)v * 16, back[u]);
                    }
                }
            }
        }
        if (!cur)
            break;
        prev = v0;
    }
}

template <int DT, bool MAXOP, bool WIDE>
__device__ __forceinline__ void sum_body(const ItemShared& sh, int nsrc, unsigned long long mask, unsigned row,
                                         size_t body, unsigned nv, int tid, int nthr)
{
    // 8 loads in flight per thread either way: 1 vector x 8 sources when every
    // sum has 8 or more sources, else 2 vectors x 4 sources.
    sum_aligned<DT, MAXOP, WIDE ? 1 : 2>(sh, nsrc, mask, row, body, nv, tid, nthr);
}

// Thread 0: copies `nbytes` (a multiple of 16, both ends 16-byte aligned)
// from `src` to every destination in `mask` through the ring.  Loads run up
// to `stages` pieces ahead; a stage is refilled once the stores that read it
// have finished reading (stores of the previous items included: piece q of
// this item is global piece G + q, in stage (G + q) mod stages).
__device__ void bulk_copy(BulkRing& bk, const ItemShared& sh, unsigned long long mask, unsigned row, size_t body,
                          const char* src, unsigned nbytes, const LaunchArgs& a)
{
    const unsigned np = (nbytes + kBulkPiece - 1) / kBulkPiece;
    const unsigned st = (unsigned)bk.stages;
    fence_proxy_async();  // order earlier generic writes (after a flag acquire) before the async loads
    if (bk.mode != 1) {
        bulk_wait_read0();  // the ring was last used in pairs
        bk.mode = 1;
    }
    const unsigned G = bk.gcopy;
    unsigned issued = 0;
    auto load = [&](unsigned q) {
        const unsigned sidx = (G + q) % st;
        const unsigned bytes = min(kBulkPiece, nbytes - q * kBulkPiece);
        mbar_expect_tx(&bk.bar[sidx], bytes);
        bulk_g2s(bk.buf + (size_t)sidx * kBulkPiece, src + (size_t)q * kBulkPiece, bytes, &bk.bar[sidx]);
    };
    // The first loads reuse the stages of the previous item's last pieces:
    // piece q waits until global piece G + q - st has read its stage (G groups
    // committed, so at most st - 1 - q still reading).
    for (; issued < np && issued < st; ++issued) {
        if (G + issued >= st)
            bulk_wait_read_n((int)(st - 1 - issued));
        load(issued);
    }
    bool ok = true;
    unsigned p = 0;
    for (; p < np; ++p) {
        const unsigned sidx = (G + p) % st;
        if (st == 1 && p >= 1) {
            bulk_wait_read0();
            load(p);
            issued = p + 1;
        }
        ok = mbar_wait(&bk.bar[sidx], (bk.phase >> sidx) & 1u, a);
        if (!ok)
            break;
        bk.phase ^= 1u << sidx;
        const unsigned bytes = min(kBulkPiece, nbytes - p * kBulkPiece);
#pragma unroll 1
        for (unsigned long long m = mask; m; m &= m - 1) {
            const int d = __ffsll((long long)m) - 1;
            bulk_s2g(DST_ROW(sh, d, row) + body + (size_t)p * kBulkPiece, bk.buf + (size_t)sidx * kBulkPiece, bytes);
        }
        bulk_commit();
        if (st > 1 && p >= 1 && issued < np) {
            bulk_wait_read1();  // the stores of piece p-1 have read their stage
            load(issued);
            ++issued;
        }
    }
    if (!ok) {
        // A load never completed in time: wait (bounded) for every load still in
        // flight so no copy lands in shared memory after this CTA moves on.
        for (unsigned q = p; q < issued; ++q) {
            const unsigned sidx = (G + q) % st;
            if (mbar_wait(&bk.bar[sidx], (bk.phase >> sidx) & 1u, a))
                bk.phase ^= 1u << sidx;
        }
        bulk_wait_all();
    }
    bk.gcopy = G + p;
    bulk_finish(bk);
}

// Copy of nv output vectors from one source that sits q bytes (q != 0) past
// a 16-byte boundary to every destination in `mask` (16-byte aligned at
// `body`), through the shared-memory ring, by the whole CTA.  The ring's
// buffers pair up (depth = stages / 2 >= 2 pairs): piece p of 1023 output
// vectors is loaded (aligned source vectors p * 1023 .. p * 1023 + 1023, one
// more than it outputs) into the first buffer of pair p % depth by one bulk
// copy, realigned by every thread into the second buffer, and stored from
// there to each destination by one bulk copy.  Thread 0 keeps up to `depth`
// loads in flight; before the barrier of piece p it waits until the stores
// that last read the output buffer of piece p + 1 are done.  Every thread
// waits on the same barriers and takes the same branches (the barrier of each
// piece ANDs the waits' outcomes), so a load that never completes ends the
// copy for every thread at the same piece; thread 0 then waits, bounded, for
// the loads still in flight (the status word reports the timeout).
__device__ void bulk_shift_copy(BulkRing& bk, const ItemShared& sh, unsigned long long mask, unsigned row,
                                size_t body, const char* src_al, int q, unsigned nv, int tid, int nthr,
                                const LaunchArgs& a)
{
    constexpr unsigned kOut = kBulkPiece / 16 - 1;  // output vectors per piece
    const unsigned depth = (unsigned)bk.stages / 2;
    const unsigned np = (nv + kOut - 1) / kOut;
    // Piece p of this item is global piece G + p, in pair (G + p) mod depth:
    // the output buffer it realigns into was freed by the wait before the
    // barrier of the previous piece, of this item or of the last one.
    const unsigned G = bk.gshift;
    auto inb = [&](unsigned i) { return bk.buf + (size_t)(2 * i) * kBulkPiece; };
    auto outb = [&](unsigned i) { return bk.buf + (size_t)(2 * i + 1) * kBulkPiece; };
    auto nout_of = [&](unsigned p) { return min(kOut, nv - p * kOut); };
    auto load = [&](unsigned p) {
        const unsigned i = (G + p) % depth;
        const unsigned bytes = (nout_of(p) + 1u) * 16u;  // the last aligned vector still holds bytes of the row
        mbar_expect_tx(&bk.sbar[i], bytes);
        bulk_g2s(inb(i), src_al + (size_t)p * kOut * 16, bytes, &bk.sbar[i]);
    };
    unsigned issued = 0, waited = 0;  // thread 0's count of loads issued and of barrier waits passed
    if (tid == 0) {
        fence_proxy_async();  // earlier generic writes (after a flag acquire) before the async loads
        if (bk.mode != 2)
            bulk_wait_read0();  // the ring was last used as single stages
        // Input buffers are free: every thread realigned from them before a
        // barrier this thread has passed.
        for (; issued < np && issued < depth; ++issued)
            load(issued);
    }
    bk.mode = 2;
    bool all_ok = true;
    unsigned p = 0;
    for (; p < np; ++p) {
        const unsigned i = (G + p) % depth;
        const bool ok = mbar_wait(&bk.sbar[i], (bk.sphase >> i) & 1u, a);
        if (ok) {
            bk.sphase ^= 1u << i;
            ++waited;
            const char* in = inb(i);
            char* out = outb(i);
            const unsigned nout = nout_of(p);
            for (unsigned v = (unsigned)tid; v < nout; v += (unsigned)nthr)
                sts16(out + (size_t)v * 16, realign(lds16(in + (size_t)v * 16), lds16(in + (size_t)v * 16 + 16), q));
        }
        fence_proxy_async_smem();  // the realigned vectors before the bulk stores that read them
        if (tid == 0)
            bulk_wait_read_n((int)depth - 2);
        all_ok = __syncthreads_and(ok ? 1 : 0) != 0;
        if (!all_ok)
            break;
        if (tid == 0) {
            const unsigned nout = nout_of(p);
#pragma unroll 1
            for (unsigned long long m = mask; m; m &= m - 1) {
                const int d = __ffsll((long long)m) - 1;
                bulk_s2g(DST_ROW(sh, d, row) + body + (size_t)p * kOut * 16, outb(i), nout * 16u);
            }
            bulk_commit();
            if (issued < np) {
                fence_proxy_async_smem();  // every thread read this input buffer before the barrier
                load(issued);
                ++issued;
            }
        }
    }
    if (tid == 0) {
        // After a timeout, the loads still in flight land before the ring is reused.
        for (; !all_ok && waited < issued; ++waited) {
            const unsigned i = (G + waited) % depth;
            if (mbar_wait(&bk.sbar[i], (bk.sphase >> i) & 1u, a))
                bk.sphase ^= 1u << i;
        }
        if (!all_ok)
            bulk_wait_all();
        bulk_finish(bk);
    }
    bk.gshift = G + p;  // pieces whose stores were committed (every thread alike)
}

// Every source of the segment sits the same q bytes past a 16-byte boundary
// while the destinations are 16-byte aligned at `body`.  Each warp step loads
// consecutive aligned vectors of every source (one per lane) and reduces them
// lane by lane (sum or maximum); for q != 0 lanes 0..30 splice their result
// with the next lane's into one destination vector (31 outputs per 32 loaded
// vectors), for q == 0 all 32 lanes store their own.  One load per source per
// vector and at most one realignment per output.  For q != 0 aligned vector
// nv is the last one that holds bytes of the row; for q == 0, vector nv - 1.
// The kernels for plans not proven aligned move every vector body through
// here, aligned or not: one body instead of three keeps them within the
// register budget.
template <int DT, bool MAXOP, bool SUM, bool WIDE, int CU = 8>
__device__ __forceinline__ void shifted_body(const ItemShared& sh, int nsrc, unsigned long long mask, unsigned row,
                                             size_t body, unsigned nv, int q, int tid, int nthr)
{
    constexpr int U = SUM ? (WIDE ? 1 : 2) : CU;  // warp steps in flight per thread (a copy: CU)
    constexpr int G = SUM ? 8 / U : 1;           // sources in flight per step
    const int lane = tid & 31;
    const unsigned warp = (unsigned)tid >> 5;
    const unsigned per = q ? 31u : 32u;  // outputs per warp step
    const unsigned span = per * ((unsigned)nthr >> 5);
    const unsigned lim = q ? nv + 1u : nv;
    // A copy into one destination (the AllToAll(V) shape): its row pointer
    // once, not per vector.  (Not for reductions: the extra registers cost
    // their kernels more than the loads saved.)
    const bool one = !SUM && (mask & (mask - 1)) == 0;
    char* const d1 = SUM ? nullptr : DST_ROW(sh, __ffsll((long long)mask) - 1, row) + body;
    for (unsigned g0 = warp * per; g0 < nv; g0 += span * U) {
        uint4 r[U];
        if constexpr (!SUM) {
            const char* base = SRC_ROW(sh, 0, row) + body - q;
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const unsigned idx = g0 + u * span + lane;
                r[u] = idx < lim ? ld16(base + (size_t)idx * 16) : make_uint4(0, 0, 0, 0);
            }
        } else {
            Acc<DT, MAXOP> acc[U];
            for (int s0 = 0; s0 < nsrc; s0 += G) {
                uint4 x[U][G];
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const unsigned idx = g0 + u * span + lane;
#pragma unroll
                    for (int g = 0; g < G; ++g)
                        x[u][g] = (s0 + g < nsrc && idx < lim)
                                      ? ld16(SRC_ROW(sh, s0 + g, row) + body - q + (size_t)idx * 16)
                                      : make_uint4(0, 0, 0, 0);
                }
#pragma unroll
                for (int u = 0; u < U; ++u) {
#pragma unroll
                    for (int g = 0; g < G; ++g) {
                        if (s0 + g < nsrc) {
                            if (s0 + g == 0)
                                acc[u].set(x[u][g]);
                            else
                                acc[u].add(x[u][g]);
                        }
                    }
                }
            }
#pragma unroll
            for (int u = 0; u < U; ++u)
                r[u] = acc[u].pack();
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            uint4 v = r[u];
            if (q) {  // warp-uniform
                uint4 nb;
                nb.x = __shfl_down_sync(0xffffffffu, r[u].x, 1);
                nb.y = __shfl_down_sync(0xffffffffu, r[u].y, 1);
                nb.z = __shfl_down_sync(0xffffffffu, r[u].z, 1);
                nb.w = __shfl_down_sync(0xffffffffu, r[u].w, 1);
                v = realign(r[u], nb, q);
            }
            const unsigned out = g0 + u * span + lane;
            if ((unsigned)lane < per && out < nv) {
                if (!SUM && one) {
                    st16(d1 + (size_t)out * 16, v);
                } else {
#pragma unroll 1
                    for (unsigned long long m = mask; m; m &= m - 1) {
                        const int d = __ffsll((long long)m) - 1;
                        st16(DST_ROW(sh, d, row) + body + (size_t)out * 16, v);
                    }
                }
            }
        }
    }
}

// A multi-row block whose rows are whole 16-byte vectors at 16-byte aligned
// addresses in every source and destination: one flat index over
// rows x vectors-per-row spread over the whole CTA (no per-row heads, tails
// or realignment).  COMP (a kCompose item): each reduced vector is stored to
// destination 0, read back from there and written to the others.
template <int DT, bool MAXOP, bool SUM, int U, bool COMP = false>
__device__ __forceinline__ void flat2d_body(const ItemShared& sh, int nsrc, int ndst, unsigned rows, unsigned vpr,
                                            int tid, int nthr)
{
    const unsigned total = rows * vpr;
    if constexpr (!SUM) {
        for (unsigned v0 = tid; v0 < total; v0 += (unsigned)nthr * U) {
            uint4 x[U];
            unsigned rr[U], cc[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const unsigned v = v0 + u * nthr;
                rr[u] = v / vpr;
                cc[u] = v - rr[u] * vpr;
                if (v < total)
                    x[u] = ld16(SRC_ROW(sh, 0, rr[u]) + (size_t)cc[u] * 16);
            }
#pragma unroll 1
            for (int d = 0; d < ndst; ++d) {
#pragma unroll
                for (int u = 0; u < U; ++u)
                    if (v0 + u * nthr < total)
                        st16(DST_ROW(sh, d, rr[u]) + (size_t)cc[u] * 16, x[u]);
            }
        }
    } else {
        constexpr int G = 8;
        for (unsigned v = tid; v < total; v += nthr) {
            const unsigned rr = v / vpr;
            const unsigned cc = v - rr * vpr;
            Acc<DT, MAXOP> acc;
            for (int s0 = 0; s0 < nsrc; s0 += G) {
                uint4 x[G];
#pragma unroll
                for (int g = 0; g < G; ++g)
                    if (s0 + g < nsrc)
                        x[g] = ld16(SRC_ROW(sh, s0 + g, rr) + (size_t)cc * 16);
#pragma unroll
                for (int g = 0; g < G; ++g) {
                    if (s0 + g < nsrc) {
                        if (s0 + g == 0)
                            acc.set(x[g]);
                        else
                            acc.add(x[g]);
                    }
                }
            }
            uint4 out = acc.pack();
            int d = 0;
            if constexpr (COMP) {
                char* const own = DST_ROW(sh, 0, rr) + (size_t)cc * 16;
                st16(own, out);
                out = ld16(own);
                d = 1;
            }
#pragma unroll 1
            for (; d < ndst; ++d)
                st16(DST_ROW(sh, d, rr) + (size_t)cc * 16, out);
        }
    }
}

// One row segment of n elements, executed by `nthr` threads with index `tid`.
// Destinations in `mask` share the same address mod 16 (`dcls`); their
// stores are 16-byte aligned after a head of at most 16/S - 1 elements, and
// the rest up to the last whole vector goes through the vector bodies.
// COMP (kCompose items, aligned kernels): `mask` holds every destination,
// destination 0 first; each reduced value is stored to destination 0 and
// written to the others from there.
template <int DT, int OPS, bool BULK, bool ALIGN, bool COMP = false>
__device__ __forceinline__ void segment(const ItemShared& sh, int nsrc, unsigned long long mask, unsigned row,
                                        unsigned n, unsigned dcls, int tid, int nthr, BulkRing& bk,
                                        const LaunchArgs& a, bool proven)
{
    using EL = Elem<DT>;
    constexpr int S = EL::S;
    constexpr bool COPY = (OPS & kOpsCopy) != 0;
    constexpr bool REDUCE = (OPS & kOpsReduce) != 0 && EL::kReducible;
    constexpr bool MAXOP = (OPS & kOpsMax) != 0;
    constexpr int E = 16 / S;
    unsigned head = ((16u - dcls) & 15u) / S;
    if (head > n)
        head = n;
    unsigned nv = (n - head) / E;
    if (ALIGN && !proven) {
        // Kernels built for plans the host proved 16-byte aligned have no
        // realigning bodies; should a segment still be misaligned, it is moved
        // element by element below (correct, slower).  A composed item's
        // destinations then differ in alignment too: all of it element-wise.
        for (int s = 0; s < nsrc; ++s)
            if (((reinterpret_cast<uintptr_t>(SRC_ROW(sh, s, row)) + (size_t)head * S) & 15u) != 0)
                nv = 0;
        if (COMP)
            nv = 0;
    }
    const unsigned tail0 = head + nv * E;
    const unsigned ntail = n - tail0;

    // Scalar head and tail elements (and, see above, misaligned rows of aligned kernels).
    for (unsigned e = tid; e < head + ntail; e += nthr) {
        const unsigned i = e < head ? e : tail0 + (e - head);
        uint32_t v;
        if constexpr (REDUCE) {
            if (nsrc > 1) {
                // 8 source loads issued before any is folded, in rank order
                float acc = 0.f;
#pragma unroll 1
                for (int s0 = 0; s0 < nsrc; s0 += 8) {
                    uint32_t y[8];
#pragma unroll
                    for (int q = 0; q < 8; ++q)
                        y[q] = s0 + q < nsrc ? EL::load(SRC_ROW(sh, s0 + q, row) + (size_t)i * S) : 0u;
#pragma unroll
                    for (int q = 0; q < 8; ++q)
                        if (s0 + q < nsrc)
                            acc = s0 + q == 0 ? EL::to_f(y[q]) : combine<MAXOP>(acc, EL::to_f(y[q]));
                }
                v = EL::from_f(acc);
            } else {
                v = EL::load(SRC_ROW(sh, 0, row) + (size_t)i * S);
            }
        } else {
            v = EL::load(SRC_ROW(sh, 0, row) + (size_t)i * S);
        }
        unsigned long long rest = mask;
        if constexpr (COMP) {
            char* const own = DST_ROW(sh, 0, row) + (size_t)i * S;
            EL::store(own, v);
            v = EL::load(own);
            rest &= ~1ull;
        }
#pragma unroll 1
        for (unsigned long long m = rest; m; m &= m - 1) {
            const int d = __ffsll((long long)m) - 1;
            EL::store(DST_ROW(sh, d, row) + (size_t)i * S, v);
        }
    }
    if (nv == 0)
        return;

    const size_t body = (size_t)head * S;
    // Misalignment of every source relative to the aligned destinations (none
    // when the item's references are proven aligned).
    int q0 = 0;
    bool uniform = true;
    if (!proven) {
        q0 = (int)((reinterpret_cast<uintptr_t>(SRC_ROW(sh, 0, row)) + body) & 15u);
        for (int s = 1; s < nsrc; ++s)
            uniform &= (int)((reinterpret_cast<uintptr_t>(SRC_ROW(sh, s, row)) + body) & 15u) == q0;
    }
    const bool aligned = uniform && q0 == 0;
    if (ALIGN && proven && !a.no_spread && !COMP) {
        // A small item: one thread per (vector, destination), so the item's
        // stores issue at once instead of one destination after another (the
        // bodies below take any thread count).  Proven items come with the
        // destinations 0 .. nd-1 in one group.  Not for a reduction in place,
        // whose destinations include a source: there every vector is read
        // whole by one thread before that thread writes it.
        const unsigned nd = (unsigned)__popcll(mask);
        if (nd > 1 && nv * nd <= (unsigned)nthr) {
            const unsigned d = (unsigned)tid / nv;
            if (d >= nd)
                return;
            mask = 1ull << d;
            tid -= (int)(d * nv);
            nthr = (int)nv;
        }
    }
    if (COPY && (!REDUCE || nsrc == 1)) {
        if (BULK && aligned && nthr == (int)blockDim.x && nv * 16u >= kBulkMin) {
            if (tid == 0)
                bulk_copy(bk, sh, mask, row, body, SRC_ROW(sh, 0, row) + body, nv * 16u, a);
        } else if constexpr (ALIGN) {
            copy_body<kCopyUnroll>(sh, mask, row, body, nv, tid, nthr);
        } else if (BULK && nthr == (int)blockDim.x && bk.stages >= 4 && nv * 16u >= kBulkMin) {
            // a source misaligned against aligned destinations (q0 != 0 here)
            bulk_shift_copy(bk, sh, mask, row, body, SRC_ROW(sh, 0, row) + body - q0, q0, nv, tid, nthr, a);
        } else {
            // the copy-only kernels run half the threads with twice the vectors in flight
            shifted_body<DT, false, false, false, OPS == kOpsCopy ? 16 : 8>(sh, 1, mask, row, body, nv, q0, tid, nthr);
        }
    } else if constexpr (REDUCE) {
        constexpr bool WIDE = (OPS & kOpsWide) != 0;
        if constexpr (ALIGN && COMP)
            sum_compose<DT, MAXOP, WIDE ? 1 : 2>(sh, nsrc, mask, row, body, nv, tid, nthr);
        else if (ALIGN)
            sum_body<DT, MAXOP, WIDE>(sh, nsrc, mask, row, body, nv, tid, nthr);
        else if (uniform)
            shifted_body<DT, MAXOP, true, WIDE>(sh, nsrc, mask, row, body, nv, q0, tid, nthr);
        else
            sum_mixed<DT, MAXOP>(sh, nsrc, mask, row, body, nv, tid, nthr);
    }
}

// Moves one rows x cols block.  A one-row block is spread over the whole CTA;
// a multi-row block gives each warp whole rows.  Destinations are grouped by
// address mod 16; each group is one pass over the sources.  `proven`: every
// reference's row 0 and row stride are 16-byte aligned (checked per reference,
// in parallel, when the references were loaded), so all destinations form one
// group and no source needs realigning; the per-reference checks are skipped.
// COMP: a kCompose item in an aligned kernel (all destinations one group,
// destination 0 written first and read back for the others).
template <int DT, int OPS, bool BULK, bool ALIGN, bool COMP>
__device__ __forceinline__ void move_rows(const ItemShared& sh, int nsrc, int ndst, unsigned rows,
                                          unsigned long long cols, BulkRing& bk, const LaunchArgs& a, bool proven)
{
    constexpr int S = Elem<DT>::S;
    constexpr bool COPY = (OPS & kOpsCopy) != 0;
    constexpr bool REDUCE = (OPS & kOpsReduce) != 0 && Elem<DT>::kReducible;
    constexpr bool MAXOP = (OPS & kOpsMax) != 0;
    if (rows > 1 && ((cols * S) & 15u) == 0) {
        // Rows of whole vectors, every row start aligned in every reference?
        bool flat = true;
        for (int i = 0; !proven && i < nsrc; ++i)
            flat &= ((reinterpret_cast<uintptr_t>(sh.src[i]) | sh.sstride[i]) & 15u) == 0;
        for (int i = 0; !proven && i < ndst; ++i)
            flat &= ((reinterpret_cast<uintptr_t>(sh.dst[i]) | sh.dstride[i]) & 15u) == 0;
        if (flat) {
            const unsigned vpr = (unsigned)(cols * S / 16);
            if (COPY && (!REDUCE || nsrc == 1))
                flat2d_body<DT, false, false, kCopyUnroll>(sh, 1, ndst, rows, vpr, (int)threadIdx.x,
                                                          (int)blockDim.x);
            else if constexpr (REDUCE)
                flat2d_body<DT, MAXOP, true, 1, COMP>(sh, nsrc, ndst, rows, vpr, (int)threadIdx.x,
                                                      (int)blockDim.x);
            return;
        }
    }
    const bool one_row = rows == 1;
    const int tid = one_row ? (int)threadIdx.x : (int)(threadIdx.x & 31);
    const int nthr = one_row ? (int)blockDim.x : 32;
    const unsigned r0 = one_row ? 0u : threadIdx.x >> 5;
    const unsigned rstep = one_row ? 1u : blockDim.x >> 5;
    const unsigned long long all = ndst >= 64 ? ~0ull : ((1ull << ndst) - 1ull);
    for (unsigned r = r0; r < rows; r += rstep) {
        unsigned long long todo = all;
        while (todo) {
            unsigned cls = 0;
            unsigned long long group = todo;
            if (!proven && !COMP) {
                const int d0 = __ffsll((long long)todo) - 1;
                cls = (unsigned)(reinterpret_cast<uintptr_t>(DST_ROW(sh, d0, r)) & 15u);
                group = 0;
                for (unsigned long long m = todo; m; m &= m - 1) {
                    const int d = __ffsll((long long)m) - 1;
                    if ((unsigned)(reinterpret_cast<uintptr_t>(DST_ROW(sh, d, r)) & 15u) == cls)
                        group |= 1ull << d;
                }
            }
            todo &= ~group;
            segment<DT, OPS, BULK, ALIGN, COMP>(sh, nsrc, group, r, (unsigned)cols, cls, tid, nthr, bk, a, proven);
        }
    }
}

// Moves one work item (all threads of the CTA).  A kCompose item (Figure 6)
// runs at the grain of one vector in the aligned kernels (move_rows, COMP).
// The kernels for other plans compose it per item instead: the reduction
// into destination 0, a CTA barrier, which makes those stores visible to
// every thread of the CTA, and then a move whose one source is destination 0
// and whose destinations are the others (the item's shared image is
// rewritten for it: this item's last use of it).
template <int DT, int OPS, bool BULK, bool ALIGN>
__device__ __forceinline__ void move_item(ItemShared& sh, int nsrc, int ndst, unsigned rows,
                                          unsigned long long cols, BulkRing& bk, const LaunchArgs& a, bool proven)
{
    constexpr bool COMPOSE = (OPS & kOpsCompose) != 0;
    if constexpr (COMPOSE && !ALIGN) {
        // one inlined move for both steps (the register budget of these kernels)
        const bool two = nsrc > 1 && ndst > 1;
        for (int step = 0;; ++step) {
            move_rows<DT, OPS, BULK, ALIGN, false>(sh, step ? 1 : nsrc, two ? (step ? ndst - 1 : 1) : ndst, rows,
                                                   cols, bk, a, proven);
            if (!two || step)
                return;
            const int t = (int)threadIdx.x;
            char* d = nullptr;
            unsigned long long ds = 0;
            if (t + 1 < ndst) {
                d = sh.dst[t + 1];
                ds = sh.dstride[t + 1];
            }
            char* const own = sh.dst[0];
            const unsigned long long os = sh.dstride[0];
            __syncthreads();
            if (t + 1 < ndst) {
                sh.dst[t] = d;
                sh.dstride[t] = ds;
            }
            if (t == 0) {
                sh.src[0] = own;
                sh.sstride[0] = os;
            }
            __syncthreads();
        }
    } else {
        move_rows<DT, OPS, BULK, ALIGN, COMPOSE && ALIGN>(sh, nsrc, ndst, rows, cols, bk, a, proven);
    }
}

// ------------------------------------------------------------- the kernel

// Shared-memory image of one claimed work item: its header (16-byte aligned
// for the asynchronous copies that fill it) and its index.
struct __align__(16) Slot {
    Item item;
    unsigned index;
    unsigned pad[3];
};

// Thread 0: the next item index of this CTA (in index order through the
// device ticket when items wait on one another or outnumber the CTAs, else
// round-robin).  In lists without flags the item loops issue the claim of
// item k+3 while item k moves and read its result only in the next
// iteration, so the ticket's round trip (an atomic through L2, slow while the
// memory system is saturated) does not hold up thread 0, and with it the CTA,
// before a move.  Lists with flags claim item k+2 at the top of iteration k,
// so that a CTA holds fewer items that later ones may wait for.
// A list without flags (static_head) takes its first two items per CTA
// statically, so that a CTA starts without a ticket round trip; in-order
// claims only matter for later items (balance) and for lists whose items
// wait on one another (progress), which claim every item by ticket.
__device__ __forceinline__ unsigned claim(const LaunchArgs& a, unsigned k)
{
    if (!a.use_tickets || (a.static_head && k < 2))
        return blockIdx.x + k * gridDim.x;
    return atomicAdd(a.st.ticket, 1u) + (a.static_head ? 2u * gridDim.x : 0u);
}

// Asynchronous global -> shared copies (no registers held while in flight).
__device__ __forceinline__ void cp_async8(void* smem, const void* g)
{
    asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(smem_u32(smem)), "l"(g) : "memory");
}
__device__ __forceinline__ void cp_async16(void* smem, const void* g)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(smem)), "l"(g) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// Region pointer of reference `tid` of `it` into `sh`.  Returns true when its
// row 0 or its row stride is not a multiple of 16 bytes.
template <int DT>
__device__ __forceinline__ bool put_ref(const LaunchArgs& a, const Item& it, const Ref& f, ItemShared& sh, int tid)
{
    constexpr int S = Elem<DT>::S;
    char* base = a.bufs[f.buf] + f.offset * (unsigned long long)S;
    const unsigned long long stride = f.stride * (unsigned long long)S;
    if (tid < it.nsrc) {
        sh.src[tid] = base;
        sh.sstride[tid] = stride;
    } else {
        sh.dst[tid - it.nsrc] = base;
        sh.dstride[tid - it.nsrc] = stride;
    }
    return ((reinterpret_cast<uintptr_t>(base) | stride) & 15u) != 0;
}

// Work-item loop of the kernels for aligned plans.  While item k moves, the
// region references of item k+1 and the header of item k+2 are on their way
// into shared memory by asynchronous copies, so the move keeps every
// register.  Headers live in a ring of three slots (items k, k+1, k+2),
// region pointers in two ItemShared buffers (items k, k+1).
template <int DT, int OPS, bool BULK>
__device__ __forceinline__ void item_loop_async(const LaunchArgs& a, ItemShared* sh, Slot* slot, Ref* sref, int* s_ok,
                                                BulkRing& bk, int tid, bool bad, unsigned long long epoch,
                                                unsigned claimed)
{
    // `claimed` (thread 0, lists without flags): the index claimed for item
    // k+2, ~0u once a claim has returned the end of the list.
    for (unsigned k = 0;; ++k) {
        const int cur = (int)(k % 3u), nxt = (int)((k + 1u) % 3u), nn = (int)((k + 2u) % 3u);
        const int scur = (int)(k & 1u), snxt = scur ^ 1;
        const unsigned index = slot[cur].index;
        if (index >= a.nitems)
            break;
        const bool has_next = slot[nxt].index < a.nitems;
        if (has_next) {
            // This thread's reference of item k+1, and (thread 0) the header of
            // item k+2: slot[nn] last held item k-1, whose posts ended (warp 0
            // synchronised) before this iteration.
            const Item& nit = slot[nxt].item;
            if (tid < nit.nsrc + nit.ndst) {
                const char* g = reinterpret_cast<const char*>(a.refs + nit.ref + tid);
                char* d = reinterpret_cast<char*>(&sref[tid]);
                cp_async8(d, g);
                cp_async8(d + 8, g + 8);
                cp_async8(d + 16, g + 16);
            }
            if (tid == 0) {
                const unsigned i2 = a.static_head ? claimed : claim(a, k + 2);
                slot[nn].index = i2;
                claimed = ~0u;
                if (i2 < a.nitems) {
                    const char* g = reinterpret_cast<const char*>(a.items + i2);
                    char* d = reinterpret_cast<char*>(&slot[nn].item);
                    cp_async16(d, g);
                    cp_async16(d + 16, g + 16);
                    if (a.static_head)
                        claimed = claim(a, k + 3);  // read in the next iteration
                }
            }
        } else if (tid == 0) {
            slot[nn].index = ~0u;
        }
        cp_async_commit();
        if (tid < 32) {
            const bool ok = slot[cur].item.nwait ? run_waits(a, slot[cur].item, tid, epoch) : true;
            if (tid == 0)
                *s_ok = ok ? 1 : 0;
        }
        // `bad`: this thread's reference of item k is misaligned (put_ref)
        const bool proven = !__syncthreads_or(bad);
        const bool ok = *s_ok != 0;  // read by every thread before the next write (after the barrier below)
        if (ok) {
            const Item& it = slot[cur].item;
            bk.drain = it.npost != 0;
            move_item<DT, OPS, BULK, true>(sh[scur], it.nsrc, it.ndst, it.rows, it.cols, bk, a, proven);
        }
        cp_async_wait_all();
        __syncthreads();
        bad = false;
        if (has_next) {
            // sh[snxt] served item k-1, whose move ended before the previous barrier
            const Item& nit = slot[nxt].item;
            if (tid < nit.nsrc + nit.ndst)
                bad = put_ref<DT>(a, nit, sref[tid], sh[snxt], tid);
        }
        if (tid < 32) {
            if (ok && slot[cur].item.npost)
                run_posts(a, slot[cur].item, index, tid, epoch);
            __syncwarp();
        }
    }
}

// Work-item loop of the spliced kernels (plans not proven aligned).  The
// references of item k+1 and the header of item k+2 are loaded into
// registers while item k moves and stored after it; at two CTAs per SM
// these kernels ran 1-2% faster this way than with the asynchronous copies
// (which made the aligned kernels 1-3% faster).  Two header slots.  The
// loads and the claim are issued after the barrier that starts the move, by
// threads kPrefetchThread onwards: the move fills these kernels' 64
// registers, so a value held across it may be spilled, and a spill waits for
// its load (measured on GB300: 1.5-2 us per item when thread 0, which drives
// the bulk ring, issued them before the barrier).  After the barrier that
// wait overlaps the move's own first loads.
template <int DT, int OPS, bool BULK>
__device__ __forceinline__ void item_loop_regs(const LaunchArgs& a, ItemShared* sh, Slot* slot, int* s_ok,
                                               BulkRing& bk, int tid, bool bad, unsigned long long epoch,
                                               unsigned* s_claimed)
{
    const int rt = tid - kPrefetchThread;  // the reference of the next item this thread loads
    // `claimed` (thread kPrefetchThread, lists without flags): the index
    // claimed for item k+2, ~0u once a claim has returned the end of the list.
    unsigned claimed = tid == kPrefetchThread ? *s_claimed : ~0u;
    for (unsigned k = 0;; ++k) {
        const int cur = (int)(k & 1u), nxt = cur ^ 1;
        const unsigned index = slot[cur].index;
        if (index >= a.nitems)
            break;
        const Item it = slot[cur].item;
        const unsigned next_index = slot[nxt].index;
        if (tid < 32) {
            const bool ok = it.nwait ? run_waits(a, it, tid, epoch) : true;
            if (tid == 0)
                *s_ok = ok ? 1 : 0;
        }
        // `bad`: this thread's reference of item k is misaligned (put_ref)
        const bool proven = !__syncthreads_or(bad);
        const bool ok = *s_ok != 0;
        const Item nit = slot[nxt].item;
        const bool has_ref = next_index < a.nitems && rt >= 0 && rt < nit.nsrc + nit.ndst;
        Ref nref{};
        if (has_ref)
            nref = a.refs[nit.ref + rt];
        unsigned i2 = ~0u;
        Item h2{};
        if (tid == kPrefetchThread && next_index < a.nitems) {
            i2 = a.static_head ? claimed : claim(a, k + 2);
            claimed = ~0u;
            if (i2 < a.nitems) {
                h2 = a.items[i2];
                if (a.static_head)
                    claimed = claim(a, k + 3);  // read in the next iteration
            }
        }
        bk.drain = it.npost != 0;
        if (ok)
            move_item<DT, OPS, BULK, false>(sh[cur], it.nsrc, it.ndst, it.rows, it.cols, bk, a, proven);
        bad = false;
        if (has_ref)
            bad = put_ref<DT>(a, nit, nref, sh[nxt], rt);  // sh[nxt] served item k-1, done before the last barrier
        if (tid == kPrefetchThread) {
            // every thread read slot[cur] and slot[nxt] before the barrier above
            slot[cur].index = i2;
            slot[cur].item = h2;
        }
        __syncthreads();
        if (tid < 32 && ok && it.npost)
            run_posts(a, it, index, tid, epoch);
    }
}

// Work-item loop of the copy-only kernels (the spliced ones at 256 threads,
// the aligned ones at 512): nothing is held in registers across the move; the references of item k+1 and the
// header of item k+2 come into shared memory by asynchronous copies, and the
// headers stay in a ring of three slots that the loop reads in place.  The
// copies and the claim are issued by threads kPrefetchThread onwards after
// the barrier that starts the move, where any wait on them overlaps the
// move's own first loads; thread 0, which drives the bulk ring, starts at
// once.  (Measured on GB300: AllToAllV 1 GiB 0.95 -> 0.98 of the roofline
// against the register form below, and the aligned AllGather and AllToAll
// 1-2% faster than with the prefetch before the barrier; the reductions'
// kernels lost with this form: ReduceScatterV 1 GiB 0.99 -> 0.96, the aligned
// AllReduce at 128 MiB 0.95 -> 0.93.)
template <int DT, int OPS, bool BULK, bool ALIGN>
__device__ __forceinline__ void item_loop_copy(const LaunchArgs& a, ItemShared* sh, Slot* slot, Ref* sref,
                                                  int* s_ok, BulkRing& bk, int tid, bool bad,
                                                  unsigned long long epoch, const unsigned* s_claimed)
{
    const int rt = tid - kPrefetchThread;  // the reference of the next item this thread copies
    // `claimed` (thread kPrefetchThread, lists without flags): the index
    // claimed for item k+2, ~0u once a claim has returned the end of the list.
    unsigned claimed = tid == kPrefetchThread ? *s_claimed : ~0u;
    for (unsigned k = 0;; ++k) {
        const int cur = (int)(k % 3u), nxt = (int)((k + 1u) % 3u), nn = (int)((k + 2u) % 3u);
        const int scur = (int)(k & 1u), snxt = scur ^ 1;
        const unsigned index = slot[cur].index;
        if (index >= a.nitems)
            break;
        if (tid < 32) {
            const bool ok = slot[cur].item.nwait ? run_waits(a, slot[cur].item, tid, epoch) : true;
            if (tid == 0)
                *s_ok = ok ? 1 : 0;
        }
        // `bad`: this thread's reference of item k is misaligned (put_ref)
        const bool proven = !__syncthreads_or(bad);
        const bool ok = *s_ok != 0;  // read by every thread before the next write (after the barrier below)
        const bool has_next = slot[nxt].index < a.nitems;
        if (has_next) {
            // slot[nn] last held item k-1, whose posts ended before the barrier above
            const Item& nit = slot[nxt].item;
            if (rt >= 0 && rt < nit.nsrc + nit.ndst) {
                const char* g = reinterpret_cast<const char*>(a.refs + nit.ref + rt);
                char* d = reinterpret_cast<char*>(&sref[rt]);
                cp_async8(d, g);
                cp_async8(d + 8, g + 8);
                cp_async8(d + 16, g + 16);
            }
            if (tid == kPrefetchThread) {
                const unsigned i2 = a.static_head ? claimed : claim(a, k + 2);
                slot[nn].index = i2;
                claimed = ~0u;
                if (i2 < a.nitems) {
                    const char* g = reinterpret_cast<const char*>(a.items + i2);
                    char* d = reinterpret_cast<char*>(&slot[nn].item);
                    cp_async16(d, g);
                    cp_async16(d + 16, g + 16);
                    if (a.static_head)
                        claimed = claim(a, k + 3);  // read in the next iteration
                }
            }
        } else if (tid == kPrefetchThread) {
            slot[nn].index = ~0u;
        }
        cp_async_commit();
        bk.drain = slot[cur].item.npost != 0;
        if (ok) {
            const Item& it = slot[cur].item;
            move_item<DT, OPS, BULK, ALIGN>(sh[scur], it.nsrc, it.ndst, it.rows, it.cols, bk, a, proven);
        }
        cp_async_wait_all();
        bad = false;
        if (has_next) {
            // this thread's own copy of the reference; sh[snxt] served item k-1
            const Item& nit = slot[nxt].item;
            if (rt >= 0 && rt < nit.nsrc + nit.ndst)
                bad = put_ref<DT>(a, nit, sref[rt], sh[snxt], rt);
        }
        __syncthreads();
        if (tid < 32) {
            if (ok && slot[cur].item.npost)
                run_posts(a, slot[cur].item, index, tid, epoch);
            __syncwarp();
        }
    }
}

// The persistent SNAC kernel.  With tickets, a CTA holds at most four claimed
// items (the one it moves and the next three; three in lists with flags) and
// processes them in claim order; every wait of an item refers to items with smaller indices, held by
// running CTAs that process their own claims in increasing order, so the
// smallest unfinished item can always proceed and the grid progresses.  A CTA
// claims its next item only once its last claim returned an item of the list,
// so every CTA makes exactly one claim beyond the end of the list.
template <int DT, int OPS, bool BULK, bool ALIGN>
__global__ void __launch_bounds__(snac_threads(OPS, ALIGN), snac_min_ctas(OPS, ALIGN))
    snac_kernel(const __grid_constant__ LaunchArgs a, int stages)
{
    __shared__ ItemShared sh[2];
    __shared__ Slot slot[3];
    __shared__ __align__(16) Ref sref[kMaxRefsPerItem];
    __shared__ int s_ok;
    __shared__ unsigned long long s_epoch;
    __shared__ unsigned s_claimed;
    extern __shared__ __align__(128) char dyn[];
    BulkRing bk{dyn + 128, reinterpret_cast<unsigned long long*>(dyn), stages, 0u,
                reinterpret_cast<unsigned long long*>(dyn) + kBulkMaxStages, 0u, true};
    const int tid = (int)threadIdx.x;
    // With static claims the CTA's first item is blockIdx.x; when every item
    // has refs_per_item references in order, each thread loads its reference
    // of that item while thread 0 loads the header (one round trip less).
    const bool early =
        (!a.use_tickets || a.static_head) && a.refs_per_item > 0 && blockIdx.x < a.nitems && tid < a.refs_per_item;
    Ref r0{};
    if (early)
        r0 = a.refs[(size_t)blockIdx.x * (size_t)a.refs_per_item + (size_t)tid];
    unsigned claimed = ~0u;  // thread 0: the claim of item 2, carried into the item loop
    if (tid == 0) {
        if (BULK) {
            for (int i = 0; i < stages; ++i)
                mbar_init(&bk.bar[i], 1u);
            for (int i = 0; i < kShiftMaxDepth; ++i)
                mbar_init(&bk.sbar[i], 1u);
            asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        }
        // The epoch of this launch (lists with flags, all ticketed): the last
        // CTA out of the previous one advanced it.
        s_epoch = a.use_tickets && !a.static_head ? *reinterpret_cast<volatile const unsigned long long*>(a.st.epoch)
                                                  : 0ull;
        const unsigned i0 = claim(a, 0);
        const unsigned i1 = i0 < a.nitems ? claim(a, 1) : ~0u;
        claimed = a.static_head && i1 < a.nitems ? claim(a, 2) : ~0u;  // read in the loop's first iteration
        // both header loads in flight before either is stored
        Item h0{}, h1{};
        if (i0 < a.nitems)
            h0 = a.items[i0];
        if (i1 < a.nitems)
            h1 = a.items[i1];
        slot[0].index = i0;
        slot[1].index = i1;
        slot[0].item = h0;
        slot[1].item = h1;
    }
    __syncthreads();
    const unsigned long long epoch = s_epoch;
    bool bad = false;
    if (slot[0].index < a.nitems && tid < slot[0].item.nsrc + slot[0].item.ndst)
        bad = put_ref<DT>(a, slot[0].item, early ? r0 : a.refs[slot[0].item.ref + tid], sh[0], tid);
    // The loops' first barrier publishes sh[0] before item 0 moves.
    if constexpr (ALIGN && OPS != kOpsCopy) {
        item_loop_async<DT, OPS, BULK>(a, sh, slot, sref, &s_ok, bk, tid, bad, epoch, claimed);
    } else {
        if (tid == 0)
            s_claimed = claimed;  // (once per launch: the claim's round trip ends here)
        __syncthreads();
        if constexpr (OPS == kOpsCopy)
            item_loop_copy<DT, OPS, BULK, ALIGN>(a, sh, slot, sref, &s_ok, bk, tid, bad, epoch, &s_claimed);
        else
            item_loop_regs<DT, OPS, BULK>(a, sh, slot, &s_ok, bk, tid, bad, epoch, &s_claimed);
    }

    if (BULK && tid == 0)
        bulk_wait_all();  // the stores of items that did not drain have landed
    if (a.use_tickets && tid == 0) {
        __threadfence();
        if (atomicAdd(a.st.exited, 1u) == gridDim.x - 1) {
            // Last CTA out: every other CTA has taken its final ticket and read
            // this launch's epoch (at its start); the next launch's tags are
            // larger than every tag of this one.
            *a.st.ticket = 0u;
            *a.st.exited = 0u;
            if (!a.static_head)
                *a.st.epoch = epoch + 1ull;
            __threadfence();
        }
    }
}

// ------------------------------------------------------------- launches

template <int DT, int OPS, bool BULK, bool ALIGN>
cudaError_t launch_one(const LaunchArgs& args, int ctas, int stages, cudaStream_t stream)
{
    size_t dyn = BULK ? 128 + (size_t)stages * kBulkPiece : 0;
    if (BULK) {
        // The attribute belongs to the function in each device's context: one
        // bit per device (of the first 64) once it is set there.
        static std::atomic<unsigned long long> configured{0};
        int dev = 0;
        cudaError_t e = cudaGetDevice(&dev);
        if (e != cudaSuccess)
            return e;
        const unsigned long long bit = dev < 64 ? 1ull << dev : 0ull;
        if (!bit || !(configured.load(std::memory_order_acquire) & bit)) {
            e = cudaFuncSetAttribute(snac_kernel<DT, OPS, BULK, ALIGN>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)(128 + (size_t)kBulkMaxStages * kBulkPiece));
            if (e != cudaSuccess)
                return e;
            configured.fetch_or(bit, std::memory_order_acq_rel);
        }
    }
    constexpr int threads = snac_threads(OPS, ALIGN);
    snac_kernel<DT, OPS, BULK, ALIGN><<<ctas, threads, dyn, stream>>>(args, stages);
    return cudaGetLastError();
}

// One instantiation per mix of moves a work list can hold: copies only,
// reductions only (wide for 2-byte sums of 8+ sources), or both, each with
// the sum or the maximum; and reductions composed as in Figure 6 (kCompose
// items, every transfer reduced).  The bulk ring serves copy items only.
template <int DT, bool BULK, bool ALIGN>
cudaError_t launch_ops(const LaunchArgs& args, int ctas, int stages, cudaStream_t stream)
{
    if constexpr (!Elem<DT>::kReducible) {
        if (args.ops != kOpsCopy)
            return cudaErrorInvalidValue;
        return launch_one<DT, kOpsCopy, BULK, ALIGN>(args, ctas, stages, stream);
    } else {
        switch (args.ops) {
        case kOpsCopy:
            return launch_one<DT, kOpsCopy, BULK, ALIGN>(args, ctas, stages, stream);
        case kOpsReduce:
            return launch_one<DT, kOpsReduce, false, ALIGN>(args, ctas, stages, stream);
        case kOpsReduce | kOpsMax:
            return launch_one<DT, kOpsReduce | kOpsMax, false, ALIGN>(args, ctas, stages, stream);
        case kOpsCopy | kOpsReduce:
            return launch_one<DT, kOpsCopy | kOpsReduce, BULK, ALIGN>(args, ctas, stages, stream);
        case kOpsCopy | kOpsReduce | kOpsMax:
            return launch_one<DT, kOpsCopy | kOpsReduce | kOpsMax, BULK, ALIGN>(args, ctas, stages, stream);
        case kOpsReduce | kOpsWide:
            if constexpr (Elem<DT>::S == 2)
                return launch_one<DT, kOpsReduce | kOpsWide, false, ALIGN>(args, ctas, stages, stream);
            return cudaErrorInvalidValue;
        case kOpsReduce | kOpsCompose:
            return launch_one<DT, kOpsReduce | kOpsCompose, false, ALIGN>(args, ctas, stages, stream);
        case kOpsReduce | kOpsMax | kOpsCompose:
            return launch_one<DT, kOpsReduce | kOpsMax | kOpsCompose, false, ALIGN>(args, ctas, stages, stream);
        case kOpsReduce | kOpsWide | kOpsCompose:
            if constexpr (Elem<DT>::S == 2)
                return launch_one<DT, kOpsReduce | kOpsWide | kOpsCompose, false, ALIGN>(args, ctas, stages, stream);
            return cudaErrorInvalidValue;
        default:
            return cudaErrorInvalidValue;
        }
    }
}

// ------------------------------------------------- inline-parameter kernel

// The rank-ordered reduction (fp32 sum or maximum, rounded once) of the
// element at byte offset `off` of the ns sources p[0 ..]: 8 loads issued
// before any is folded.
template <int DT, bool MAXOP>
__device__ __forceinline__ uint32_t scalar_reduce(char* const* p, unsigned ns, size_t off)
{
    using EL = Elem<DT>;
    float acc = 0.f;
    for (unsigned s0 = 0; s0 < ns; s0 += 8) {
        uint32_t y[8];
#pragma unroll
        for (unsigned q = 0; q < 8; ++q)
            y[q] = s0 + q < ns ? EL::load(p[s0 + q] + off) : 0u;
#pragma unroll
        for (unsigned q = 0; q < 8; ++q)
            if (s0 + q < ns)
                acc = s0 + q == 0 ? EL::to_f(y[q]) : combine<MAXOP>(acc, EL::to_f(y[q]));
    }
    return EL::from_f(acc);
}

// The rank-ordered reduction (fp32 sum or maximum, rounded once) of the 16
// bytes at byte offset `off` of the ns sources p[0 ..], 8 sources in flight.
// ALIGNED: every source address is 16-byte aligned.  Otherwise a source at a
// byte shift q is read as the two aligned vectors around it (every load of
// the 8 sources is issued before any splice) and spliced; the aligned vector
// holding its last byte, which belongs to the region, is the second, so no
// load leaves the buffer.
template <int DT, bool MAXOP, bool ALIGNED>
__device__ __forceinline__ uint4 inline_reduce(char* const* p, unsigned ns, size_t off)
{
    Acc<DT, MAXOP> acc;
    for (unsigned s0 = 0; s0 < ns; s0 += 8) {
        uint4 lo[8], hi[8];
        int sh[8];
#pragma unroll
        for (unsigned q = 0; q < 8; ++q) {
            const char* a = s0 + q < ns ? p[s0 + q] + off : p[0] + off;
            sh[q] = ALIGNED ? 0 : (int)(reinterpret_cast<uintptr_t>(a) & 15u);
            lo[q] = s0 + q < ns ? ld16(a - sh[q]) : make_uint4(0, 0, 0, 0);
            hi[q] = !ALIGNED && s0 + q < ns && sh[q] ? ld16(a - sh[q] + 16) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (unsigned q = 0; q < 8; ++q) {
            if (s0 + q < ns) {
                const uint4 x = !ALIGNED && sh[q] ? realign(lo[q], hi[q], sh[q]) : lo[q];
                if (s0 + q == 0)
                    acc.set(x);
                else
                    acc.add(x);
            }
        }
    }
    return acc.pack();
}

// One item per CTA, read from the parameter block.
//  - An item whose every pointer is 16-byte aligned (kInlineAligned, from
//    the host) of at most one vector per thread: each vector is read by g
//    threads (g the CTA's threads per vector, at most the item's destination
//    count) and thread j of a vector writes destinations j, j + g, j + 2g,
//    ..., so the item's stores issue at once.  A larger one: one thread per
//    vector for every destination, U vectors in flight per thread (a copy:
//    U = 8; a reduction: 2 vectors x 8 sources per step), every source
//    vector read once.
//  - Another item: its destinations share their address mod 16 (the host
//    checks it; should they not, the whole item moves element by element).
//    The body between the destinations' first and last 16-byte boundaries
//    moves in vectors as above (g threads per vector, looping with g = 1 when
//    larger: copies 4 vectors in flight per thread, reductions 8 sources); a
//    source at another byte shift is read as the two aligned vectors around
//    each of its vectors and spliced.
//  - The elements before the body (the head) and after it (the tail) move one
//    (element, destination) pair per thread.
// Reductions combine the sources in rank order in fp32 (the sum or the
// maximum) and round once, exactly as the persistent kernel does.  With
// kInlineVectorWhole, g = 1: every vector is read whole by one thread before
// it writes any destination (one of which may be one of its sources).
template <int DT, bool MAXOP, int NI, int NP>
__global__ void __launch_bounds__(kInlineThreads, 1) snac_inline_kernel(const __grid_constant__ InlineArgs<NI, NP> a)
{
    using EL = Elem<DT>;
    constexpr int S = EL::S;
    constexpr unsigned E = 16 / S;
    const InlineItem it = a.it[blockIdx.x];
    char* const* p = a.ptr + it.ref;
    const unsigned ns = it.nsrc, nd = it.ndst, n = it.count, step = blockDim.x, tid = threadIdx.x;
    const bool whole = (it.flags & kInlineVectorWhole) != 0;
    const bool reduce = EL::kReducible && ns > 1;
    unsigned h = 0, nv = n / E;
    unsigned busy = step;  // threads the body's first round keeps busy
    if (it.flags & kInlineAligned) {
        if (nv > step) {
            if (!reduce) {
                constexpr int U = 8;
                for (unsigned v0 = tid; v0 < nv; v0 += U * step) {
                    uint4 x[U];
#pragma unroll
                    for (int u = 0; u < U; ++u)
                        if (v0 + u * step < nv)
                            x[u] = ld16(p[0] + (size_t)(v0 + u * step) * 16);
                    for (unsigned d = 0; d < nd; ++d) {
#pragma unroll
                        for (int u = 0; u < U; ++u)
                            if (v0 + u * step < nv)
                                st16(p[1 + d] + (size_t)(v0 + u * step) * 16, x[u]);
                    }
                }
            } else if constexpr (EL::kReducible) {
                constexpr int U = 2;
                for (unsigned v0 = tid; v0 < nv; v0 += U * step) {
                    Acc<DT, MAXOP> acc[U];
                    for (unsigned s0 = 0; s0 < ns; s0 += 8) {
                        uint4 x[U][8];
#pragma unroll
                        for (int u = 0; u < U; ++u) {
                            const unsigned v = v0 + u * step;
#pragma unroll
                            for (unsigned q = 0; q < 8; ++q)
                                x[u][q] = v < nv && s0 + q < ns ? ld16(p[s0 + q] + (size_t)v * 16) : make_uint4(0, 0, 0, 0);
                        }
#pragma unroll
                        for (int u = 0; u < U; ++u) {
#pragma unroll
                            for (unsigned q = 0; q < 8; ++q) {
                                if (s0 + q < ns) {
                                    if (s0 + q == 0)
                                        acc[u].set(x[u][q]);
                                    else
                                        acc[u].add(x[u][q]);
                                }
                            }
                        }
                    }
#pragma unroll
                    for (int u = 0; u < U; ++u) {
                        const unsigned v = v0 + u * step;
                        if (v < nv) {
                            const uint4 out = acc[u].pack();
                            for (unsigned d = 0; d < nd; ++d)
                                st16(p[ns + d] + (size_t)v * 16, out);
                        }
                    }
                }
            }
        } else if (nv > 0) {
            const unsigned g = whole ? 1u : max(1u, min(nd, step / nv));
            busy = nv * g;
            if (tid < nv * g) {
                const unsigned j = tid / nv, v = tid - j * nv;
                const size_t off = (size_t)v * 16;
                uint4 out;
                if constexpr (EL::kReducible)
                    out = reduce ? inline_reduce<DT, MAXOP, true>(p, ns, off) : ld16(p[0] + off);
                else
                    out = ld16(p[0] + off);
                for (unsigned d = j; d < nd; d += g)
                    st16(p[ns + d] + off, out);
            }
        }
    } else {
        const unsigned dcls = (unsigned)(reinterpret_cast<uintptr_t>(p[ns]) & 15u);
        bool congruent = true;
        for (unsigned d = 1; d < nd; ++d)
            congruent &= (unsigned)(reinterpret_cast<uintptr_t>(p[ns + d]) & 15u) == dcls;
        h = congruent ? min(n, ((16u - dcls) & 15u) / S) : n;
        nv = (n - h) / E;
        const size_t body = (size_t)h * S;
        const unsigned g = whole || nv > step ? 1u : max(1u, min(nd, step / max(nv, 1u)));
        const unsigned total = nv * g;
        busy = min(step, total);
        if (!reduce) {
            // one source at shift q: its aligned vectors, loaded before any splice
            constexpr int U = 4;
            const int q = (int)((reinterpret_cast<uintptr_t>(p[0]) + body) & 15u);
            const char* src = p[0] + body - q;
            for (unsigned k0 = tid; k0 < total; k0 += U * step) {
                uint4 lo[U], hi[U];
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const unsigned k = k0 + u * step;
                    const size_t at = (size_t)(k % nv) * 16;
                    lo[u] = k < total ? ld16(src + at) : make_uint4(0, 0, 0, 0);
                    hi[u] = k < total && q ? ld16(src + at + 16) : make_uint4(0, 0, 0, 0);
                }
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const unsigned k = k0 + u * step;
                    if (k < total) {
                        const uint4 x = q ? realign(lo[u], hi[u], q) : lo[u];
                        const size_t off = body + (size_t)(k % nv) * 16;
                        for (unsigned d = k / nv; d < nd; d += g)
                            st16(p[1 + d] + off, x);
                    }
                }
            }
        } else if constexpr (EL::kReducible) {
            for (unsigned k = tid; k < total; k += step) {
                const unsigned j = k / nv, v = k - j * nv;
                const size_t off = body + (size_t)v * 16;
                const uint4 out = inline_reduce<DT, MAXOP, false>(p, ns, off);
                for (unsigned d = j; d < nd; d += g)
                    st16(p[ns + d] + off, out);
            }
        }
    }
    // head [0, h) and tail [h + nv * E, n), one element each, first on the
    // threads the body left idle (so both are in flight at once)
    const unsigned t0 = h + nv * E, ne = h + (n - t0);
    if (ne == 0)
        return;
    const unsigned gt = whole ? 1u : max(1u, min(nd, step / ne));
    for (unsigned k = (tid + step - busy % step) % step; k < ne * gt; k += step) {
        const unsigned i = k % ne, e = i < h ? i : t0 + (i - h);
        uint32_t x;
        if constexpr (EL::kReducible) {
            x = reduce ? scalar_reduce<DT, MAXOP>(p, ns, (size_t)e * S) : EL::load(p[0] + (size_t)e * S);
        } else {
            x = EL::load(p[0] + (size_t)e * S);
        }
        for (unsigned d = k / ne; d < nd; d += gt)
            EL::store(p[ns + d] + (size_t)e * S, x);
    }
}

template <int DT, bool MAXOP>
cudaError_t launch_inline_op(const InlineSmall* small, const InlineLarge* large, int nitems, cudaStream_t stream)
{
    if (small)
        snac_inline_kernel<DT, MAXOP, kInlineSmallItems, kInlineSmallPtrs><<<nitems, kInlineThreads, 0, stream>>>(*small);
    else
        snac_inline_kernel<DT, MAXOP, kInlineMaxItems, kInlineMaxPtrs><<<nitems, kInlineThreads, 0, stream>>>(*large);
    return cudaGetLastError();
}

template <int DT>
cudaError_t launch_inline_dtype(bool maxop, const InlineSmall* small, const InlineLarge* large, int nitems,
                                cudaStream_t stream)
{
    if (nitems < 1 || (small ? nitems > kInlineSmallItems : (!large || nitems > kInlineMaxItems)))
        return cudaErrorInvalidValue;
    if constexpr (Elem<DT>::kReducible) {
        if (maxop)
            return launch_inline_op<DT, true>(small, large, nitems, stream);
    }
    return launch_inline_op<DT, false>(small, large, nitems, stream);
}

template <int DT>
cudaError_t launch_dtype(const LaunchArgs& args, int ctas, bool bulk, bool aligned, int stages, cudaStream_t stream)
{
    if (bulk)
        return aligned ? launch_ops<DT, true, true>(args, ctas, stages, stream)
                       : launch_ops<DT, true, false>(args, ctas, stages, stream);
    return aligned ? launch_ops<DT, false, true>(args, ctas, stages, stream)
                   : launch_ops<DT, false, false>(args, ctas, stages, stream);
}

}  // namespace
}  // namespace purlin
