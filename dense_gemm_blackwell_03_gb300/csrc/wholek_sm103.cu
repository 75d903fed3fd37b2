// wholek_sm103.cu -- instantiates and launches the whole-K pair kernel for
// 129 to 256 rows of A (wholek_kernel.cuh) in clusters of two CTAs.
#include "internal.h"
#include "wholek_kernel.cuh"

namespace bwgemm {

namespace {

template <int BN>
cudaError_t launch_wk(const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& a3, const CUtensorMap& b3,
                      const CUtensorMap& c, const GemmParams& p, int grid, cudaStream_t stream, bool pdl)
{
    constexpr int KPS = wholek_kblocks(BN);
    constexpr int ST = wholek_stages(BN);
    using Cfg = WholeKConfig<BN, KPS, ST>;
    auto kernel = wholek_kernel<BN, KPS, ST>;
    if (grid % 2 != 0)
        return cudaErrorInvalidValue;
    cudaError_t err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::kSmemBytes);
    if (err != cudaSuccess)
        return err;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(unsigned(grid), 1, 1);
    cfg.blockDim = dim3(kWkThreads, 1, 1);
    cfg.dynamicSmemBytes = Cfg::kSmemBytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    unsigned n = 0;
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = 2;
    attr[n].val.clusterDim.y = 1;
    attr[n].val.clusterDim.z = 1;
    ++n;
    if (pdl) {
        attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[n].val.programmaticStreamSerializationAllowed = 1;
        ++n;
    }
    cfg.attrs = attr;
    cfg.numAttrs = n;
    return cudaLaunchKernelEx(&cfg, kernel, a, b, a3, b3, c, p);
}

}  // namespace

cudaError_t launch_wholek(int bn, const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& a3,
                          const CUtensorMap& b3, const CUtensorMap& c, const GemmParams& p, int grid,
                          cudaStream_t stream, bool pdl)
{
    static_assert(sizeof(kWholeKWidths) / sizeof(kWholeKWidths[0]) == 6, "one case per width below");
    switch (bn) {
    case 96: return launch_wk<96>(a, b, a3, b3, c, p, grid, stream, pdl);
    case 112: return launch_wk<112>(a, b, a3, b3, c, p, grid, stream, pdl);
    case 128: return launch_wk<128>(a, b, a3, b3, c, p, grid, stream, pdl);
    case 144: return launch_wk<144>(a, b, a3, b3, c, p, grid, stream, pdl);
    case 160: return launch_wk<160>(a, b, a3, b3, c, p, grid, stream, pdl);
    case 192: return launch_wk<192>(a, b, a3, b3, c, p, grid, stream, pdl);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace bwgemm
