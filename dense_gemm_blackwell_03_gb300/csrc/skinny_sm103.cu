// skinny_sm103.cu -- instantiates and launches the whole-K kernel for decode
// batches of at most 64 rows (skinny_kernel.cuh); the pair form in clusters
// of two CTAs.
#include "internal.h"
#include "skinny_kernel.cuh"

namespace bwgemm {

namespace {

template <int BN>
cudaError_t launch_sk(const CUtensorMap& w, const CUtensorMap& x, const CUtensorMap& w3, const CUtensorMap& x3,
                      const CUtensorMap& c, const GemmParams& p, int grid, cudaStream_t stream, bool pdl)
{
    constexpr int KPS = skinny_kblocks(BN);
    constexpr int ST = skinny_stages(BN);
    constexpr int CG = skinny_cg(BN);
    using Cfg = SkinnyConfig<BN, KPS, ST, CG>;
    auto kernel = skinny_kernel<BN, KPS, ST, CG>;
    if (grid % CG != 0)
        return cudaErrorInvalidValue;
    cudaError_t err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::kSmemBytes);
    if (err != cudaSuccess)
        return err;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(unsigned(grid), 1, 1);
    cfg.blockDim = dim3(kSkThreads, 1, 1);
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
    return cudaLaunchKernelEx(&cfg, kernel, w, x, w3, x3, c, p);
}

}  // namespace

cudaError_t launch_skinny(int bn, const CUtensorMap& w, const CUtensorMap& x, const CUtensorMap& w3,
                          const CUtensorMap& x3, const CUtensorMap& c, const GemmParams& p, int grid,
                          cudaStream_t stream, bool pdl)
{
    switch (bn) {
    case 16: return launch_sk<16>(w, x, w3, x3, c, p, grid, stream, pdl);
    case 32: return launch_sk<32>(w, x, w3, x3, c, p, grid, stream, pdl);
    case 64: return launch_sk<64>(w, x, w3, x3, c, p, grid, stream, pdl);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace bwgemm
