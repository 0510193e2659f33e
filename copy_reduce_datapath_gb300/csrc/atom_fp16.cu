// The fp16 instantiations of the persistent SNAC kernel and of the inline-parameter
// kernel (see atom_impl.cuh).
#include "atom_impl.cuh"

namespace purlin {

cudaError_t launch_snac_fp16(const LaunchArgs& a, int ctas, bool bulk, bool aligned, int stages, cudaStream_t s)
{
    return launch_dtype<kDtFp16>(a, ctas, bulk, aligned, stages, s);
}

cudaError_t launch_inline_fp16(bool maxop, const InlineSmall* small, const InlineLarge* large, int nitems,
                               cudaStream_t s)
{
    return launch_inline_dtype<kDtFp16>(maxop, small, large, nitems, s);
}

}  // namespace purlin
