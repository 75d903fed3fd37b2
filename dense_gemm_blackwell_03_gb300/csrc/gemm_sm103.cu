// gemm_sm103.cu -- instantiates the tcgen05 GEMM kernel variants and launches them.
#include "gemm_kernel.cuh"
#include "internal.h"

namespace bwgemm {

namespace {

template <int CG, int BN, int STAGES, bool TR, int MC, int KS, bool RS>
cudaError_t launch_one(const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& c,
                       const CUtensorMap& a2, const CUtensorMap& b2, const CUtensorMap& c2,
                       const GemmParams& p, int grid, cudaStream_t stream, bool pdl)
{
    using Cfg = KernelConfig<CG, BN, STAGES, (KS > 1) || RS>;
    auto kernel = gemm_kernel<CG, BN, STAGES, TR, MC, KS, RS>;
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
    if (CG * MC * KS > 1) {
        attr[n].id = cudaLaunchAttributeClusterDimension;
        attr[n].val.clusterDim.x = CG * MC * KS;
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
    return cudaLaunchKernelEx(&cfg, kernel, a, b, c, a2, b2, c2, p);
}

template <int CG, int BN, int STAGES, bool TR, int MC, int KS, bool RS>
cudaError_t max_active_one(int* out)
{
    using Cfg = KernelConfig<CG, BN, STAGES, (KS > 1) || RS>;
    auto kernel = gemm_kernel<CG, BN, STAGES, TR, MC, KS, RS>;
    cudaError_t err =
        cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::kSmemBytes);
    if (err != cudaSuccess)
        return err;
    if (CG * MC * KS == 1) {
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
    cfg.gridDim = dim3(CG * MC * KS, 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = Cfg::kSmemBytes;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = CG * MC * KS;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaOccupancyMaxActiveClusters(out, kernel, &cfg);
}

struct VariantFns {
    cudaError_t (*launch)(const CUtensorMap&, const CUtensorMap&, const CUtensorMap&,
                          const CUtensorMap&, const CUtensorMap&, const CUtensorMap&, const GemmParams&,
                          int, cudaStream_t, bool);
    cudaError_t (*max_active)(int*);
    int smem_bytes;
};

#define BWGEMM_VARIANT_RS(CG, BN, ST, TR, MC, KS, RS)                                       \
    {&launch_one<CG, BN, ST, TR, MC, KS, RS>, &max_active_one<CG, BN, ST, TR, MC, KS, RS>, \
     KernelConfig<CG, BN, ST, (KS > 1) || RS>::kSmemBytes}
#define BWGEMM_VARIANT(CG, BN, ST, TR, MC, KS) BWGEMM_VARIANT_RS(CG, BN, ST, TR, MC, KS, false)

// same order as kVariants in internal.h
constexpr VariantFns kFns[] = {
    BWGEMM_VARIANT(1, 256, 4, false, 1, 1), BWGEMM_VARIANT(1, 128, 6, false, 1, 1),
    BWGEMM_VARIANT(2, 256, 6, false, 1, 1), BWGEMM_VARIANT(2, 128, 8, false, 1, 1),
    BWGEMM_VARIANT(2, 128, 8, true, 1, 1),  BWGEMM_VARIANT(2, 64, 9, true, 1, 1),
    BWGEMM_VARIANT(1, 128, 6, true, 1, 1),  BWGEMM_VARIANT(1, 64, 8, true, 1, 1),
    BWGEMM_VARIANT(2, 256, 6, false, 2, 1), BWGEMM_VARIANT(2, 128, 8, false, 2, 1),
    BWGEMM_VARIANT(2, 256, 7, false, 1, 2), BWGEMM_VARIANT(1, 64, 9, true, 1, 2),
    BWGEMM_VARIANT(2, 224, 6, false, 1, 1), BWGEMM_VARIANT(2, 224, 7, false, 1, 2),
    BWGEMM_VARIANT(2, 320, 5, false, 1, 1), BWGEMM_VARIANT(2, 320, 6, false, 1, 2),
    BWGEMM_VARIANT(2, 384, 4, false, 1, 1),
    BWGEMM_VARIANT_RS(2, 224, 7, false, 1, 1, true), BWGEMM_VARIANT_RS(2, 384, 5, false, 1, 1, true),
};
#undef BWGEMM_VARIANT
#undef BWGEMM_VARIANT_RS
static_assert(sizeof(kFns) / sizeof(kFns[0]) == kNumVariants, "variant tables out of step");

}  // namespace

int variant_smem_bytes(int idx) { return (idx >= 0 && idx < kNumVariants) ? kFns[idx].smem_bytes : 0; }

cudaError_t launch_variant(int idx, const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& c,
                           const CUtensorMap& a2, const CUtensorMap& b2, const CUtensorMap& c2,
                           const GemmParams& p, int grid, cudaStream_t stream, bool pdl)
{
    if (idx < 0 || idx >= kNumVariants)
        return cudaErrorInvalidValue;
    return kFns[idx].launch(a, b, c, a2, b2, c2, p, grid, stream, pdl);
}

cudaError_t variant_max_active(int idx, int* out)
{
    if (idx < 0 || idx >= kNumVariants)
        return cudaErrorInvalidValue;
    return kFns[idx].max_active(out);
}

}  // namespace bwgemm
