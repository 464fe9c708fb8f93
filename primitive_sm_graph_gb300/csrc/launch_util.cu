// Per-device caches of the few attributes the launch planners need.  The
// caches are filled once per (device, kernel) and never change afterwards.
#include <cuda_runtime.h>

#include <cstdlib>
#include <mutex>
#include <unordered_map>

#include "launch_util.cuh"

namespace psg {

namespace {
constexpr int MAX_DEV = 64;
std::mutex g_mu;
int g_sms[MAX_DEV];
size_t g_l2[MAX_DEV];
std::unordered_map<uint64_t, int>& occ_cache()
{
    static std::unordered_map<uint64_t, int> m;
    return m;
}
std::unordered_map<uint64_t, cudaError_t>& smem_attr_cache()
{
    static std::unordered_map<uint64_t, cudaError_t> m;
    return m;
}
}  // namespace

int current_device()
{
    int d = 0;
    if (cudaGetDevice(&d) != cudaSuccess) d = 0;
    return d < 0 || d >= MAX_DEV ? 0 : d;
}

int num_sms()
{
    const int d = current_device();
    std::lock_guard<std::mutex> g(g_mu);
    if (g_sms[d] == 0) {
        int n = 0;
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, d);
        g_sms[d] = n > 0 ? n : 1;
    }
    return g_sms[d];
}

size_t l2_bytes()
{
    const int d = current_device();
    std::lock_guard<std::mutex> g(g_mu);
    if (g_l2[d] == 0) {
        int n = 0;
        cudaDeviceGetAttribute(&n, cudaDevAttrL2CacheSize, d);
        g_l2[d] = n > 0 ? (size_t)n : 1;
    }
    return g_l2[d];
}

int max_blocks_per_sm(const void* fn, int threads, size_t smem)
{
    const int d = current_device();
    const uint64_t key = ((uint64_t)(uintptr_t)fn * 1315423911ull) ^ ((uint64_t)d << 56) ^
                         ((uint64_t)threads << 40) ^ (uint64_t)smem;
    {
        std::lock_guard<std::mutex> g(g_mu);
        auto it = occ_cache().find(key);
        if (it != occ_cache().end()) return it->second;
    }
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, fn, threads, smem) != cudaSuccess) n = 1;
    if (n < 1) n = 1;
    std::lock_guard<std::mutex> g(g_mu);
    occ_cache()[key] = n;
    return n;
}

cudaError_t set_max_dynamic_smem(const void* fn, int bytes)
{
    const int d = current_device();
    const uint64_t key = ((uint64_t)(uintptr_t)fn * 2654435761ull) ^ ((uint64_t)d << 56) ^ (uint64_t)(uint32_t)bytes;
    std::lock_guard<std::mutex> g(g_mu);
    auto it = smem_attr_cache().find(key);
    if (it != smem_attr_cache().end()) return it->second;
    const cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    smem_attr_cache()[key] = e;
    return e;
}

bool pdl_enabled()
{
    static const bool on = std::getenv("PSG_NO_PDL") == nullptr;
    return on;
}

int kernel_regs(const void* fn)
{
    cudaFuncAttributes a;
    if (cudaFuncGetAttributes(&a, fn) != cudaSuccess) return -1;
    return a.numRegs;
}

}  // namespace psg
