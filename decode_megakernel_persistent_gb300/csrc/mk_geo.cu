// mk_geo.cu -- the per-warp attention megakernel carrying only one model
// family's matrix-vector geometries (see geo_has).
#include "megakernel.cuh"

namespace ll {

const void *megakernel_geo_fn(int geo) {
    return geo == GEO_2048 ? reinterpret_cast<const void *>(decode_megakernel<true, false, GEO_2048>)
                           : reinterpret_cast<const void *>(decode_megakernel<true, false, GEO_4096>);
}

}  // namespace ll
