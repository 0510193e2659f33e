// Launches of the persistent SNAC kernel and of the inline-parameter kernel:
// each picks the element type's instantiation (this file holds the bf16 ones;
// atom_fp16.cu, atom_fp32.cu and atom_fp8.cu the others, compiled in
// parallel), and the persistent kernel whether the plan may use the kernels
// without realigning bodies.
#include "atom_impl.cuh"

namespace purlin {

cudaError_t launch_snac_bf16(const LaunchArgs& a, int ctas, bool bulk, bool aligned, int stages, cudaStream_t s)
{
    return launch_dtype<kDtBf16>(a, ctas, bulk, aligned, stages, s);
}

cudaError_t launch_inline_bf16(bool maxop, const InlineSmall* small, const InlineLarge* large, int nitems,
                               cudaStream_t s)
{
    return launch_inline_dtype<kDtBf16>(maxop, small, large, nitems, s);
}

cudaError_t launch_snac(const LaunchArgs& args, int ctas, bool bulk, int stages, cudaStream_t stream)
{
    if (stages < 1 || stages > kBulkMaxStages)
        stages = 4;
    // A plan whose every reference is 16-byte aligned, over 16-byte aligned
    // buffers, runs in the instantiation without realigning bodies.
    bool aligned = args.all_aligned != 0;
    for (int i = 0; aligned && i < args.nbufs; ++i)
        aligned = (reinterpret_cast<uintptr_t>(args.bufs[i]) & 15u) == 0;
    switch (args.dtype) {
    case kDtBf16:
        return launch_snac_bf16(args, ctas, bulk, aligned, stages, stream);
    case kDtFp32:
        return launch_snac_fp32(args, ctas, bulk, aligned, stages, stream);
    case kDtFp16:
        return launch_snac_fp16(args, ctas, bulk, aligned, stages, stream);
    case kDtFp8:
        return launch_snac_fp8(args, ctas, bulk, aligned, stages, stream);
    default:
        return cudaErrorInvalidValue;
    }
}

cudaError_t launch_inline(int dtype, bool maxop, const InlineSmall* small, const InlineLarge* large, int nitems,
                          cudaStream_t stream)
{
    switch (dtype) {
    case kDtBf16:
        return launch_inline_bf16(maxop, small, large, nitems, stream);
    case kDtFp32:
        return launch_inline_fp32(maxop, small, large, nitems, stream);
    case kDtFp16:
        return launch_inline_fp16(maxop, small, large, nitems, stream);
    case kDtFp8:
        return launch_inline_fp8(maxop, small, large, nitems, stream);
    default:
        return cudaErrorInvalidValue;
    }
}

int snac_ctas_per_sm(KernelClass k)
{
    int n = 0;
    constexpr int kMix = kOpsCopy | kOpsReduce, kWide = kOpsReduce | kOpsWide;
    const cudaError_t e =
        k == KernelClass::kAligned
            ? cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, snac_kernel<kDtBf16, kMix, false, true>,
                                                            snac_threads(kMix, true), 0)
        : k == KernelClass::kAlignedReduce
            ? cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, snac_kernel<kDtBf16, kWide, false, true>,
                                                            snac_threads(kWide, true), 0)
            : cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, snac_kernel<kDtBf16, kMix, false, false>,
                                                            snac_threads(kMix, false), 0);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    return n;
}

}  // namespace purlin
