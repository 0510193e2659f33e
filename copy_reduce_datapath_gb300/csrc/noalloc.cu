// pl_allreduce_noalloc: the staged SNAC AllReduce with every byte of its device
// state in one file-scope device array, for callers that must not allocate
// device memory.  Some callers cannot call cudaMalloc: a process that reserves
// its whole device memory budget at start-up and may not grow it, a plug-in
// that does not own the process's device allocator, or code on a latency path
// where an allocation (which may synchronise the device) is not acceptable.
// The context-based entry points allocate their flag words, work-list copies
// and staging ring on the device; this one uses the static array below
// instead and allocates nothing on the device.
#include "purlin.h"
#include "snac.h"

#include <cuda_runtime.h>

#include <cstring>
#include <mutex>
#include <vector>

using namespace purlin;

namespace {

// Layout of the static array (bytes):
//   [0, kStateBytes)                 flag words, counters, status word
//   [kListOffset, kRingOffset)       the derived work list
//   [kRingOffset, kScratchBytes)     the staging ring (R rings of slots)
constexpr size_t kScratchBytes = 32u << 20;
constexpr size_t kStateBytes = 64u << 10;
constexpr size_t kListOffset = kStateBytes;
constexpr size_t kRingOffset = 4u << 20;
constexpr size_t kListBytes = kRingOffset - kListOffset;
constexpr size_t kRingBytes = kScratchBytes - kRingOffset;
constexpr uint32_t kMaxFlags = 2048;                 // 20 bytes each, plus 16 bytes of counters
constexpr uint64_t kMaxBytesPerRank = 256ull << 20;  // the largest AllReduce this entry point accepts
constexpr int kMaxRanksNoAlloc = 8;                  // ranks whose work list fits the list region
constexpr uint64_t kChunkBytes = 256u << 10;
constexpr int kMaxDevices = 64;

static_assert((size_t)kMaxFlags * 20 + 64 <= kStateBytes, "flag words must fit the state region");

// Every GPU that loads the library holds this array until the process exits.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

// Host-side record of one device.  `list` is the host image of the work list
// the device's array last received.  Its storage is reserved once for the
// largest list and never moves or shrinks, so the copy that uploads it never
// reads freed memory; a call whose work list equals it uploads nothing.
struct DeviceSetup {
    std::mutex mu;         // serialises set-up and uploads of this device
    char* base = nullptr;  // device address of g_noalloc_scratch on this device
    int num_sms = 0;
    std::vector<unsigned char> list;
};
DeviceSetup g_setup[kMaxDevices];  // indexed by CUDA device ordinal (host side)

size_t align256(size_t n) { return (n + 255) / 256 * 256; }

// Once per device, with that device current and d.mu held: the device
// address of the static array (its name is only a host-side stand-in in host
// code) and the SM count that sizes the grid.
pl_status setup_device(int dev, DeviceSetup& d)
{
    if (d.base)
        return PL_OK;
    void* ptr = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
    if (e != cudaSuccess || !ptr) {
        cudaGetLastError();
        return PL_ERR_CUDA;
    }
    int sms = 0;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess || sms < 1) {
        cudaGetLastError();
        return PL_ERR_CUDA;
    }
    d.list.reserve(kListBytes);
    d.num_sms = sms;
    d.base = static_cast<char*>(ptr);
    return PL_OK;
}

}  // namespace

extern "C" PL_API pl_status pl_allreduce_noalloc(pl_dtype dtype, int R, uint64_t count, void* const* in_bufs,
                                                 void* const* out_bufs, int wait, void* stream)
{
    if (R < 1 || !in_bufs || !out_bufs || (dtype != PL_BF16 && dtype != PL_FP32 && dtype != PL_FP16))
        return PL_ERR_INVALID;
    if (R > kMaxRanksNoAlloc)
        return PL_ERR_NOMEM;  // the work list of more ranks may not fit the array
    const uint64_t esize = dtype == PL_FP32 ? 4 : 2;
    if (count > kMaxBytesPerRank / esize)
        return PL_ERR_NOMEM;  // beyond what the static array is sized for
    if (count == 0)
        return PL_OK;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return PL_ERR_CUDA;
    }
    if (dev < 0 || dev >= kMaxDevices)
        return PL_ERR_INVALID;
    DeviceSetup* d = &g_setup[dev];
    std::lock_guard<std::mutex> hold(d->mu);
    pl_status st = setup_device(dev, *d);
    if (st != PL_OK)
        return st;

    HostWorkList wl;
    st = derive_staged_allreduce(R, dtype, count, in_bufs, out_bufs, d->num_sms, kRingBytes, kChunkBytes, wl);
    if (st != PL_OK)
        return st;
    const size_t bi = wl.items.size() * sizeof(Item);
    const size_t br = wl.refs.size() * sizeof(Ref);
    const size_t bs = wl.syncs.size() * sizeof(Sync);
    const size_t oi = 0, orr = align256(bi), os = orr + align256(br);
    if (wl.nflags > kMaxFlags || os + bs > kListBytes || wl.items.empty())
        return PL_ERR_NOMEM;

    // The flag words and counters must start at zero: cleared on the caller's
    // stream.  The work list goes into the array by one copy on that stream,
    // from the device's host image, and only when it differs from the list the
    // array already holds (the same AllReduce called again uploads nothing).
    std::vector<unsigned char> host(os + bs, 0);
    std::memcpy(host.data() + oi, wl.items.data(), bi);
    std::memcpy(host.data() + orr, wl.refs.data(), br);
    std::memcpy(host.data() + os, wl.syncs.data(), bs);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    char* list = d->base + kListOffset;
    cudaError_t e = cudaMemsetAsync(d->base, 0, kStateBytes, s);
    if (e == cudaSuccess && host != d->list) {
        d->list.assign(host.begin(), host.end());  // within the reserved storage: no reallocation
        e = cudaMemcpyAsync(list, d->list.data(), d->list.size(), cudaMemcpyHostToDevice, s);
        if (e != cudaSuccess)
            d->list.clear();  // the array's list is unknown: upload again next time
    }
    if (e != cudaSuccess) {
        cudaGetLastError();
        return PL_ERR_CUDA;
    }

    LaunchArgs a{};
    a.items = reinterpret_cast<const Item*>(list + oi);
    a.refs = reinterpret_cast<const Ref*>(list + orr);
    a.syncs = reinterpret_cast<const Sync*>(list + os);
    a.nitems = (uint32_t)wl.items.size();
    a.use_tickets = wl.uses_tickets;
    a.dtype = dtype;
    a.nbufs = 2 * R + 1;
    a.ops = wl.ops;
    a.all_aligned = wl.all_aligned;
    a.refs_per_item = wl.refs_per_item;
    a.timeout_ns = 2000000000ull;
    a.drop_notify = -1;
    char* state = d->base;
    a.st.full = reinterpret_cast<unsigned long long*>(state);
    a.st.done = reinterpret_cast<unsigned long long*>(state + (size_t)kMaxFlags * 8);
    a.st.count = reinterpret_cast<unsigned int*>(state + (size_t)kMaxFlags * 16);
    char* tail = state + (size_t)kMaxFlags * 20;
    a.st.ticket = reinterpret_cast<unsigned int*>(tail);
    a.st.exited = reinterpret_cast<unsigned int*>(tail + 4);
    a.st.status = reinterpret_cast<int*>(tail + 8);
    a.st.abort = reinterpret_cast<int*>(tail + 12);
    a.st.epoch = reinterpret_cast<unsigned long long*>(tail + 16);  // zeroed above with the flags
    for (int r = 0; r < R; ++r) {
        a.bufs[r] = static_cast<char*>(in_bufs[r]);
        a.bufs[R + r] = static_cast<char*>(out_bufs[r]);
    }
    a.bufs[2 * R] = d->base + kRingOffset;
    e = launch_snac(a, wl.ctas, false, 4, s);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return PL_ERR_CUDA;
    }
    if (!wait)
        return PL_OK;
    e = cudaStreamSynchronize(s);
    int status = 0;
    if (e == cudaSuccess)
        e = cudaMemcpy(&status, a.st.status, sizeof status, cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return PL_ERR_CUDA;
    }
    return status;
}
