// ropekv_floor.cu -- libropekv_floor.so: a copy kernel launched exactly like
// libropekv's decode-sized launches (see include/ropekv_floor.h). It measures
// the floor of one dependent launch that moves the decode call's bytes in the
// decode call's grid; the fused RoPE + KV write never calls it.
#include <cuda_runtime.h>

#include <atomic>
#include <stdint.h>

#include "ropekv_floor.h"

namespace {

constexpr int kVecsPerThread = 4;  // a decode thread: two items of two 16-byte vectors

__device__ __forceinline__ void prefetch_l2(const void* p)
{
    asm volatile("prefetch.global.L2 [%0];" :: "l"(p));
}

__global__ void __launch_bounds__(256) floor_copy_kernel(const uint4* src, uint4* dst)
{
    const size_t base = (size_t)blockIdx.x * blockDim.x * kVecsPerThread + threadIdx.x;
#pragma unroll
    for (int k = 0; k < kVecsPerThread; ++k)
        prefetch_l2(src + base + (size_t)k * blockDim.x);
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    uint4 v[kVecsPerThread];
#pragma unroll
    for (int k = 0; k < kVecsPerThread; ++k)
        asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.u32 {%0,%1,%2,%3}, [%4], %5;"
                     : "=r"(v[k].x), "=r"(v[k].y), "=r"(v[k].z), "=r"(v[k].w)
                     : "l"(src + base + (size_t)k * blockDim.x), "l"(pol));
#pragma unroll
    for (int k = 0; k < kVecsPerThread; ++k)
        asm volatile("st.global.L2::cache_hint.v4.u32 [%0], {%1,%2,%3,%4}, %5;"
                     :: "l"(dst + base + (size_t)k * blockDim.x), "r"(v[k].x), "r"(v[k].y),
                        "r"(v[k].z), "r"(v[k].w), "l"(pol)
                     : "memory");
}

// The residency cap of libropekv's small launches: at most ceil(grid / SMs)
// CTAs per SM through unused dynamic shared memory (none above 8 per SM).
size_t cap_smem(unsigned grid, int* optin)
{
    int dev = 0, sms = 0, perSm = 0, reserved = 0;
    *optin = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&perSm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev) !=
            cudaSuccess ||
        cudaDeviceGetAttribute(optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) !=
            cudaSuccess ||
        cudaDeviceGetAttribute(&reserved, cudaDevAttrReservedSharedMemoryPerBlock, dev) !=
            cudaSuccess || sms <= 0) {
        return 0;  // launch uncapped
    }
    const unsigned per = (grid + (unsigned)sms - 1) / (unsigned)sms;
    if (per == 0 || per > 8)
        return 0;
    long long bytes = (long long)perSm / per - reserved;
    if (bytes > *optin)
        bytes = *optin;
    return bytes > 0 ? (size_t)(bytes & ~255LL) : 0;
}

}  // namespace

extern "C" int ropekv_floor_copy(const void* src, void* dst, int64_t bytes, int32_t threadsPerCta,
                                 int32_t cap, void* stream)
{
    if (!src || !dst)
        return -1;
    if ((reinterpret_cast<uintptr_t>(src) & 15u) || (reinterpret_cast<uintptr_t>(dst) & 15u))
        return -2;
    if (threadsPerCta < 32 || threadsPerCta > 256 || threadsPerCta % 32 != 0)
        return -6;
    const int64_t perCta = 16LL * kVecsPerThread * threadsPerCta;
    if (bytes <= 0 || bytes % perCta != 0 || bytes / perCta > 0x7FFFFFFFLL)
        return -6;
    const unsigned grid = (unsigned)(bytes / perCta);
    size_t smem = 0;
    if (cap) {
        int optin = 0;
        smem = cap_smem(grid, &optin);
        if (smem > 48 * 1024) {
            static std::atomic<unsigned long long> raised{0};
            int dev = 0;
            (void)cudaGetDevice(&dev);
            const unsigned long long bit = (dev >= 0 && dev < 64) ? 1ULL << dev : 0;
            if (!bit || !(raised.load(std::memory_order_relaxed) & bit)) {
                if (cudaFuncSetAttribute(floor_copy_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, optin) ==
                    cudaSuccess) {
                    raised.fetch_or(bit, std::memory_order_relaxed);
                } else {
                    smem = 0;  // launch uncapped
                }
            }
        }
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3((unsigned)threadsPerCta);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = (cudaStream_t)stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, floor_copy_kernel, static_cast<const uint4*>(src),
                              static_cast<uint4*>(dst)) == cudaSuccess
               ? 0
               : -10;
}
