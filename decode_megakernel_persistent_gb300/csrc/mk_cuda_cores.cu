// mk_cuda_cores.cu -- the megakernel instantiations whose matrix-vector
// products all run on CUDA cores, and the host side of every instantiation.
#include "megakernel.cuh"

namespace ll {

const void *megakernel_tc_fn(bool flash, int geo);  // mk_tensor_cores.cu
const void *megakernel_geo_fn(int geo);     // mk_geo.cu: per-warp attention, one geometry family

static const void *megakernel_fn(bool flash, bool tc, int geo) {
    if (tc) return megakernel_tc_fn(flash, geo);
    if (flash && geo != GEO_ALL) return megakernel_geo_fn(geo);
    return flash ? reinterpret_cast<const void *>(decode_megakernel<true, false>)
                 : reinterpret_cast<const void *>(decode_megakernel<false, false>);
}

int megakernel_smem_bytes() { return SMEM_BYTES; }

int megakernel_prepare(int smem_bytes) {
    for (int i = 0; i < 8; i++) {
        const void *fn = i < 4   ? megakernel_fn(i & 1, i & 2, GEO_ALL)
                         : i < 6 ? megakernel_fn(true, false, i == 4 ? GEO_2048 : GEO_4096)
                                 : megakernel_fn(i & 1, true, GEO_BCC);
        cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes);
        if (e != cudaSuccess) return LL_ERR_CUDA;
        int blocks = 0;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&blocks, fn, NTHREADS, smem_bytes);
        if (e != cudaSuccess) return LL_ERR_CUDA;
        if (blocks < 1) return LL_ERR_DEVICE;
    }
    return LL_OK;
}

int launch_megakernel(const KParams &p, void *stream, int smem_bytes) {
    void *args[] = {const_cast<KParams *>(&p)};
    const bool tc = p.geo == GEO_BCC || p.mv_h.tc || p.mv_q.tc || p.mv_i.tc;  // the batched kernels
    cudaError_t e = cudaLaunchCooperativeKernel(megakernel_fn(p.attn_flash != 0, tc, p.geo), dim3(p.nsm), dim3(NTHREADS),
                                                args, size_t(smem_bytes), static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? LL_OK : LL_ERR_CUDA;
}

}  // namespace ll
