// gemm_sm103.cu -- instantiates the tcgen05 GEMM kernel variants and launches them.
#include "gemm_kernel.cuh"
#include "internal.h"

namespace bwgemm {

namespace {

template <int CG, int BN, int STAGES>
cudaError_t launch_one(const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& c,
                       const GemmParams& p, int grid, cudaStream_t stream, bool pdl)
{
    using Cfg = KernelConfig<CG, BN, STAGES>;
    auto kernel = gemm_kernel<CG, BN, STAGES>;
    cudaError_t err =
        cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::kSmemBytes);
    if (err != cudaSuccess)
        return err;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(unsigned(grid), 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = Cfg::kSmemBytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    unsigned n = 0;
    if (CG == 2) {
        attr[n].id = cudaLaunchAttributeClusterDimension;
        attr[n].val.clusterDim.x = 2;
        attr[n].val.clusterDim.y = 1;
        attr[n].val.clusterDim.z = 1;
        ++n;
    }
    if (pdl) {
        attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[n].val.programmaticStreamSerializationAllowed = 1;
        ++n;
    }
    cfg.attrs = n ? attr : nullptr;
    cfg.numAttrs = n;
    return cudaLaunchKernelEx(&cfg, kernel, a, b, c, p);
}

template <int CG, int BN, int STAGES>
cudaError_t max_active_one(int* out)
{
    using Cfg = KernelConfig<CG, BN, STAGES>;
    auto kernel = gemm_kernel<CG, BN, STAGES>;
    cudaError_t err =
        cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::kSmemBytes);
    if (err != cudaSuccess)
        return err;
    if (CG == 1) {
        int per_sm = 0, dev = 0, sms = 0;
        err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, kThreads,
                                                            Cfg::kSmemBytes);
        if (err != cudaSuccess)
            return err;
        if ((err = cudaGetDevice(&dev)) != cudaSuccess)
            return err;
        if ((err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
            return err;
        *out = per_sm * sms;
        return cudaSuccess;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2, 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = Cfg::kSmemBytes;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaOccupancyMaxActiveClusters(out, kernel, &cfg);
}

}  // namespace

int find_variant(int cg, int bn)
{
    for (int i = 0; i < kNumVariants; ++i)
        if (kVariants[i].cg == cg && kVariants[i].bn == bn)
            return i;
    return -1;
}

int variant_smem_bytes(int idx)
{
    switch (idx) {
    case 0: return KernelConfig<1, 256, 4>::kSmemBytes;
    case 1: return KernelConfig<1, 128, 6>::kSmemBytes;
    case 2: return KernelConfig<2, 256, 6>::kSmemBytes;
    case 3: return KernelConfig<2, 128, 8>::kSmemBytes;
    default: return 0;
    }
}

cudaError_t launch_variant(int idx, const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& c,
                           const GemmParams& p, int grid, cudaStream_t stream, bool pdl)
{
    switch (idx) {
    case 0: return launch_one<1, 256, 4>(a, b, c, p, grid, stream, pdl);
    case 1: return launch_one<1, 128, 6>(a, b, c, p, grid, stream, pdl);
    case 2: return launch_one<2, 256, 6>(a, b, c, p, grid, stream, pdl);
    case 3: return launch_one<2, 128, 8>(a, b, c, p, grid, stream, pdl);
    default: return cudaErrorInvalidValue;
    }
}

cudaError_t variant_max_active(int idx, int* out)
{
    switch (idx) {
    case 0: return max_active_one<1, 256, 4>(out);
    case 1: return max_active_one<1, 128, 6>(out);
    case 2: return max_active_one<2, 256, 6>(out);
    case 3: return max_active_one<2, 128, 8>(out);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace bwgemm
