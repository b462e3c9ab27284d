// mk_tensor_cores.cu -- the megakernel instantiations that take the widths with
// tensor-core geometry (MvShape::tc) on tensor-core pages.
#include "megakernel.cuh"

namespace ll {

const void *megakernel_tc_fn(bool flash) {
    return flash ? reinterpret_cast<const void *>(decode_megakernel<true, true>)
                 : reinterpret_cast<const void *>(decode_megakernel<false, true>);
}

}  // namespace ll
