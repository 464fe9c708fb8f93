// NVRTC front end and kernel cache of the runtime-specialised kernels.
#include "jit.h"

#include <nvrtc.h>

#include <cstdio>
#include <cstdlib>
#include <mutex>
#include <unordered_map>
#include <vector>

// kJitParams, kJitPrelude, kJitEw, kJitReduce: the hand-written sources under
// csrc/jit/, embedded as text by the build
#include "jit_sources.inc"

namespace psg {

namespace {

std::mutex g_mu;

std::unordered_map<std::string, cudaKernel_t>& cache()
{
    static std::unordered_map<std::string, cudaKernel_t> m;
    return m;
}

const char* const kOpts[] = {
    "--gpu-architecture=sm_103a", "-std=c++17", "--fmad=false", "--ftz=false",
    "--prec-div=true", "--prec-sqrt=true", "-lineinfo", "-default-device",
};

psg_status compile(const std::string& src, std::vector<char>* cubin, std::string* log)
{
    nvrtcProgram prog;
    if (nvrtcCreateProgram(&prog, src.c_str(), "psg_jit.cu", 0, nullptr, nullptr) != NVRTC_SUCCESS)
        return PSG_E_CUDA;
    // PSG_JIT_PTXAS_V=1 asks ptxas for its resource report (registers,
    // spills) in the program log
    std::vector<const char*> opts(kOpts, kOpts + sizeof(kOpts) / sizeof(kOpts[0]));
    if (std::getenv("PSG_JIT_PTXAS_V")) opts.push_back("--ptxas-options=-v");
    const nvrtcResult rc = nvrtcCompileProgram(prog, (int)opts.size(), opts.data());
    size_t ls = 0;
    nvrtcGetProgramLogSize(prog, &ls);
    if (log && ls > 1) {
        log->resize(ls);
        nvrtcGetProgramLog(prog, &(*log)[0]);
    }
    if (rc == NVRTC_SUCCESS && std::getenv("PSG_JIT_PTXAS_V") && log) std::fprintf(stderr, "%s\n", log->c_str());
    if (rc != NVRTC_SUCCESS) {
        if (std::getenv("PSG_JIT_VERBOSE") && log) std::fprintf(stderr, "%s\n%s\n", src.c_str(), log->c_str());
        nvrtcDestroyProgram(&prog);
        return PSG_E_CUDA;
    }
    if (cubin) {
        size_t n = 0;
        nvrtcGetCUBINSize(prog, &n);
        cubin->resize(n);
        nvrtcGetCUBIN(prog, cubin->data());
    }
    nvrtcDestroyProgram(&prog);
    return PSG_OK;
}

}  // namespace

// what NVRTC lacks for the tensor-core skeleton: the fixed-width integer
// types and the 128-byte tensor map the host encodes (an opaque blob)
const char* const kGemmPreamble =
    "typedef unsigned char uint8_t;\ntypedef unsigned short uint16_t;\ntypedef unsigned int uint32_t;\n"
    "typedef int int32_t;\ntypedef unsigned long long uint64_t;\ntypedef long long int64_t;\n"
    "typedef unsigned long long uintptr_t;\n"
    "struct __align__(64) CUtensorMap { unsigned long long opaque[16]; };\n";

std::string jit_source(JitSkeleton sk, const std::string& spec)
{
    std::string s;
    s.reserve(65536);
    s += kJitParams;
    s += "\n";
    s += kJitPrelude;
    if (sk == JIT_GEMM) {
        const size_t cut = spec.find('\x01');
        s += "\n";
        s += kGemmPreamble;
        s += kJitGemmParams;
        s += "\n";
        s += kJitTcDevice;
        s += "\n";
        s += kJitGemmBody;
        s += "\n// ---- operand tables ----\n";
        s += spec.substr(0, cut);
        s += "\n";
        s += kJitGemmEpi;
        s += "\n// ---- epilogue program and entry point ----\n";
        s += cut == std::string::npos ? std::string() : spec.substr(cut + 1);
        return s;
    }
    s += "\n// ---- program-specific part ----\n";
    s += spec;
    s += "\n// ---- kernel skeleton ----\n";
    s += sk == JIT_EW ? kJitEw : kJitReduce;
    return s;
}

psg_status jit_compile_only(const std::string& src, std::string* log)
{
    if (std::getenv("PSG_JIT_DUMP")) std::fprintf(stderr, "%s\n", src.c_str());
    return compile(src, nullptr, log);
}

psg_status jit_kernel(JitSkeleton sk, const std::string& spec, const char* name, cudaKernel_t* out)
{
    std::string key;
    key.reserve(spec.size() + 2);
    key += (char)('0' + (int)sk);
    key += spec;
    std::lock_guard<std::mutex> g(g_mu);
    auto it = cache().find(key);
    if (it != cache().end()) {
        *out = it->second;
        return PSG_OK;
    }
    const std::string src = jit_source(sk, spec);
    std::vector<char> cubin;
    std::string log;
    psg_status st = compile(src, &cubin, &log);
    if (st != PSG_OK) return st;
    cudaLibrary_t lib;
    if (cudaLibraryLoadData(&lib, cubin.data(), nullptr, nullptr, 0, nullptr, nullptr, 0) != cudaSuccess)
        return PSG_E_CUDA;
    cudaKernel_t k;
    if (cudaLibraryGetKernel(&k, lib, name) != cudaSuccess) return PSG_E_CUDA;
    cache().emplace(std::move(key), k);
    *out = k;
    return PSG_OK;
}

int jit_max_blocks_per_sm(cudaKernel_t k, int threads, size_t smem)
{
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, (const void*)k, threads, smem) != cudaSuccess) n = 1;
    return n < 1 ? 1 : n;
}

int jit_regs(cudaKernel_t k)
{
    cudaFuncAttributes a;
    if (cudaFuncGetAttributes(&a, (const void*)k) != cudaSuccess) return -1;
    return a.numRegs;
}

}  // namespace psg
