// probe.cu -- measures the dense rate of one SM's tensor pipe in FLOP per SM
// clock, so that a nominal peak (SMs x rate x clock) can be stated from a
// measurement rather than assumed.
//
// One CTA per SM issues a long run of tcgen05.mma (cta_group::1, M = 128,
// N = 256, K = 16, bf16 in, fp32 accumulation in TMEM) on operands that stay
// in shared memory, with no loads in the loop, and times the run from the
// first issue to the commit of the last MMA in SM cycles (clock64).  The
// operand values do not matter (zeros); the descriptors are the kernel's own
// (128B swizzle, K-major).  Every wait is bounded: a run that does not finish
// within the limit reports BWGEMM_ERR_TIMEOUT.
#include "gemm_kernel.cuh"
#include "internal.h"

#include <algorithm>
#include <vector>

namespace bwgemm {
namespace {

constexpr int kProbeThreads = 128;
constexpr int kProbeKBlocks = 1024;  // timed K blocks of four MMAs each
constexpr int kProbeWarmKBlocks = 64;
constexpr int kProbeN = 256;
constexpr int kProbeABytes = kRowsPerCta * kTileK * 2;  // 16 KiB
constexpr int kProbeBBytes = kProbeN * kTileK * 2;      // 32 KiB
// more than half of an SM's shared memory, so that one CTA runs per SM
constexpr int kProbeSmem = 120 * 1024;

__global__ void __launch_bounds__(kProbeThreads, 1)
    tensor_rate_probe(unsigned long long* cycles, uint32_t* status, long long limit_cycles)
{
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = ptx::smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* smem = smem_raw + (base - raw);
    const uint32_t sA = base;
    const uint32_t sB = base + kProbeABytes;
    const uint32_t bar = sB + kProbeBBytes;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kProbeABytes + kProbeBBytes + 8);
    const int warp = threadIdx.x >> 5;

    uint4* zero = reinterpret_cast<uint4*>(smem);
    for (int i = threadIdx.x; i < (kProbeABytes + kProbeBBytes) / 16; i += kProbeThreads)
        zero[i] = make_uint4(0u, 0u, 0u, 0u);
    if (warp == 0) {
        ptx::tmem_alloc<1>(ptx::smem_addr(tmem_slot), kProbeN);
        ptx::tmem_relinquish<1>();
    }
    if (threadIdx.x == 32) {
        ptx::mbar_init(bar, 1);
        ptx::fence_mbar_init();
    }
    ptx::fence_proxy_async_smem();  // the zeros, visible to the tensor pipe
    ptx::tc_fence_before_sync();
    __syncthreads();
    ptx::tc_fence_after_sync();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        const uint64_t a = make_sdesc_sw128(sA);
        const uint64_t b = make_sdesc_sw128(sB);
        const uint32_t idesc = make_idesc(0, kRowsPerCta, kProbeN);
        if (ptx::elect_one()) {
            bool ok = true;
            long long t0 = 0, t1 = 0;
            for (int run = 0; run < 2 && ok; ++run) {
                const int kblocks = run == 0 ? kProbeWarmKBlocks : kProbeKBlocks;
                t0 = clock64();
#pragma unroll 1
                for (int i = 0; i < kblocks; ++i) {
#pragma unroll
                    for (int kk = 0; kk < kTileK / kMmaK; ++kk)
                        ptx::mma_f16<1>(tmem, a + uint64_t(kk * 2), b + uint64_t(kk * 2), idesc,
                                        (i > 0 || kk > 0) ? 1u : 0u);
                }
                ptx::mma_commit(bar);
                while (!ptx::mbar_try_wait(bar, uint32_t(run))) {
                    if (clock64() - t0 > limit_cycles) {
                        atomicOr(status, 1u);
                        ok = false;
                        break;
                    }
                }
                t1 = clock64();
            }
            cycles[blockIdx.x] = ok ? (unsigned long long)(t1 - t0) : 0ull;
        }
        __syncwarp();
    }
    ptx::tc_fence_before_sync();
    __syncthreads();
    ptx::tc_fence_after_sync();
    if (warp == 0)
        ptx::tmem_dealloc<1>(tmem, kProbeN);
}

}  // namespace
}  // namespace bwgemm

using namespace bwgemm;

extern "C" bwgemm_status_t bwgemm_probe_tensor_rate(int device, double* flop_per_clock_per_sm, int32_t* sm_count)
{
    if (!flop_per_clock_per_sm || !sm_count)
        return BWGEMM_ERR_INVALID_ARG;
    int prev = 0;
    if (cudaGetDevice(&prev) != cudaSuccess)
        return BWGEMM_ERR_NO_DEVICE;
    if (cudaSetDevice(device) != cudaSuccess)
        return BWGEMM_ERR_NO_DEVICE;
    bwgemm_status_t st = BWGEMM_OK;
    int major = 0, minor = 0, sms = 0;
    cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, device);
    cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, device);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device);
    unsigned long long* d_cycles = nullptr;
    uint32_t* d_status = nullptr;
    std::vector<unsigned long long> h(size_t(sms > 0 ? sms : 1), 0ull);
    uint32_t h_status = 0;
    if (major != 10 || minor != 3 || sms <= 0) {
        st = BWGEMM_ERR_UNSUPPORTED;
    } else if (cudaMalloc(&d_cycles, size_t(sms) * sizeof(unsigned long long)) != cudaSuccess ||
               cudaMalloc(&d_status, sizeof(uint32_t)) != cudaSuccess ||
               cudaMemset(d_cycles, 0, size_t(sms) * sizeof(unsigned long long)) != cudaSuccess ||
               cudaMemset(d_status, 0, sizeof(uint32_t)) != cudaSuccess ||
               cudaFuncSetAttribute(tensor_rate_probe, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    kProbeSmem) != cudaSuccess) {
        st = BWGEMM_ERR_CUDA;
    } else {
        // about a second of cycles at the SM clock bounds each timed run
        tensor_rate_probe<<<sms, kProbeThreads, kProbeSmem>>>(d_cycles, d_status, 2000000000ll);
        if (cudaGetLastError() != cudaSuccess || cudaDeviceSynchronize() != cudaSuccess ||
            cudaMemcpy(h.data(), d_cycles, h.size() * sizeof(unsigned long long), cudaMemcpyDeviceToHost) !=
                cudaSuccess ||
            cudaMemcpy(&h_status, d_status, sizeof(uint32_t), cudaMemcpyDeviceToHost) != cudaSuccess)
            st = BWGEMM_ERR_CUDA;
        else if (h_status != 0)
            st = BWGEMM_ERR_TIMEOUT;
    }
    if (st == BWGEMM_OK) {
        std::sort(h.begin(), h.end());
        const double med = double(h[h.size() / 2]);
        const double flop = double(kProbeKBlocks) * (kTileK / kMmaK) * 2.0 * kRowsPerCta * kProbeN * kMmaK;
        if (med <= 0.0)
            st = BWGEMM_ERR_CUDA;
        else {
            *flop_per_clock_per_sm = flop / med;
            *sm_count = sms;
        }
    }
    if (d_cycles)
        cudaFree(d_cycles);
    if (d_status)
        cudaFree(d_status);
    cudaSetDevice(prev);
    return st;
}
