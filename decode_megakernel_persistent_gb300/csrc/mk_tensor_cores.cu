// mk_tensor_cores.cu -- the batched megakernel instantiations: the widths with
// tensor-core geometry (MvShape::tc) on tensor-core pages, or a batch of two on
// CUDA-core pages (GEO_BCC).
#include "megakernel.cuh"

namespace ll {

const void *megakernel_tc_fn(bool flash, int geo) {
    if (geo == GEO_BCC)  // a batch of two on CUDA-core pages
        return flash ? reinterpret_cast<const void *>(decode_megakernel<true, true, GEO_BCC>)
                     : reinterpret_cast<const void *>(decode_megakernel<false, true, GEO_BCC>);
    return flash ? reinterpret_cast<const void *>(decode_megakernel<true, true>)
                 : reinterpret_cast<const void *>(decode_megakernel<false, true>);
}

}  // namespace ll
