// The fp16 instantiation of the persistent SNAC kernel (see atom_impl.cuh).
#include "atom_impl.cuh"

namespace purlin {

cudaError_t launch_snac_fp16(const LaunchArgs& a, int ctas, bool bulk, bool aligned, int stages, cudaStream_t s)
{
    return launch_dtype<kDtFp16>(a, ctas, bulk, aligned, stages, s);
}

}  // namespace purlin
