// attnres_jit.cu -- run-time compiled forward kernels (single- and
// multi-query) for one plan's exact shape.
//
// The forward templates (attnres_fwd_kernel.cuh, attnres_multi_fwd_kernel.cuh)
// take the source count, the
// rows per chunk, the softmax group rows and the ring depth either from its
// arguments (the precompiled instances) or as template constants.  With the
// constants the compiler unrolls a token's whole schedule (its groups, their
// chunk waits and the weighted-row loops): forward 0.474 against 0.488 ms on
// the long-sequence workload, 0.253 against 0.266 ms on the fused block read,
// 1.35 against 1.43 ms with 64 sources, bitwise equal outputs.  The pages'
// Triton kernels are specialised on the residual count the same way.  Here NVRTC compiles the header
// sources (embedded in this library when it is built) for the plan at hand,
// once per shape and device; the CUBIN is loaded through the driver API and
// launched on the caller's stream.  NVRTC and the driver library are opened
// with dlopen, and any failure (no NVRTC, a compile error, a load error)
// leaves the precompiled kernels in charge: the caller falls back on
// cudaErrorNotSupported.  ATTNRES_JIT=0 in the environment turns this path off.
#include <cuda.h>
#include <dlfcn.h>
#include <nvrtc.h>

#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <atomic>
#include <map>
#include <memory>
#include <mutex>
#include <string>
#include <tuple>
#include <vector>

#include "kernels.cuh"
#include "attnres_jit_sources.inc"  // generated at build time: kJitFiles[] = {name, text}

#ifndef ATTNRES_CUDA_LIBDIR
#define ATTNRES_CUDA_LIBDIR "/usr/local/cuda/lib64"
#endif

namespace attnres {
namespace {

// Headers the kernel sources include from the toolkit, reduced to what the
// device code needs (NVRTC declares the CUDA runtime types itself).
const char kIntTypes[] =
    "#pragma once\n"
    "typedef unsigned char uint8_t; typedef unsigned short uint16_t; typedef unsigned int uint32_t;\n"
    "typedef unsigned long long uint64_t; typedef signed char int8_t; typedef short int16_t;\n"
    "typedef int int32_t; typedef long long int64_t; typedef unsigned long size_t;\n"
    "typedef unsigned long uintptr_t; typedef long ptrdiff_t;\n";
const char kFloatLimits[] = "#pragma once\n#define FLT_MAX 3.402823466e+38F\n";
const char kEmpty[] = "#pragma once\n";

struct Api {
    bool ok = false;
    // NVRTC
    nvrtcResult (*createProgram)(nvrtcProgram*, const char*, const char*, int, const char* const*,
                                 const char* const*) = nullptr;
    nvrtcResult (*addNameExpression)(nvrtcProgram, const char*) = nullptr;
    nvrtcResult (*compileProgram)(nvrtcProgram, int, const char* const*) = nullptr;
    nvrtcResult (*getLoweredName)(nvrtcProgram, const char*, const char**) = nullptr;
    nvrtcResult (*getCUBINSize)(nvrtcProgram, size_t*) = nullptr;
    nvrtcResult (*getCUBIN)(nvrtcProgram, char*) = nullptr;
    nvrtcResult (*destroyProgram)(nvrtcProgram*) = nullptr;
    // driver
    CUresult (*moduleLoadData)(CUmodule*, const void*) = nullptr;
    CUresult (*moduleGetFunction)(CUfunction*, CUmodule, const char*) = nullptr;
    CUresult (*moduleGetGlobal)(CUdeviceptr*, size_t*, CUmodule, const char*) = nullptr;
    CUresult (*funcSetAttribute)(CUfunction, CUfunction_attribute, int) = nullptr;
    CUresult (*launchKernel)(CUfunction, unsigned, unsigned, unsigned, unsigned, unsigned, unsigned, unsigned,
                             CUstream, void**, void**) = nullptr;
    CUresult (*memcpyDtoH)(void*, CUdeviceptr, size_t) = nullptr;
    CUresult (*memcpyHtoD)(CUdeviceptr, const void*, size_t) = nullptr;
    CUresult (*occupancy)(int*, CUfunction, int, size_t) = nullptr;
};

template <typename F>
bool sym(void* lib, const char* name, F* out) {
    *out = reinterpret_cast<F>(dlsym(lib, name));
    return *out != nullptr;
}

const Api& api() {
    static Api a;
    static std::once_flag once;
    std::call_once(once, [] {
        void* nv = dlopen("libnvrtc.so.13", RTLD_NOW | RTLD_LOCAL);
        if (!nv) nv = dlopen(ATTNRES_CUDA_LIBDIR "/libnvrtc.so", RTLD_NOW | RTLD_LOCAL);
        void* cu = dlopen("libcuda.so.1", RTLD_NOW | RTLD_LOCAL);
        if (!nv || !cu) return;
        a.ok = sym(nv, "nvrtcCreateProgram", &a.createProgram) &&
               sym(nv, "nvrtcAddNameExpression", &a.addNameExpression) &&
               sym(nv, "nvrtcCompileProgram", &a.compileProgram) &&
               sym(nv, "nvrtcGetLoweredName", &a.getLoweredName) && sym(nv, "nvrtcGetCUBINSize", &a.getCUBINSize) &&
               sym(nv, "nvrtcGetCUBIN", &a.getCUBIN) && sym(nv, "nvrtcDestroyProgram", &a.destroyProgram) &&
               sym(cu, "cuModuleLoadData", &a.moduleLoadData) &&
               sym(cu, "cuModuleGetFunction", &a.moduleGetFunction) &&
               sym(cu, "cuModuleGetGlobal_v2", &a.moduleGetGlobal) &&
               sym(cu, "cuFuncSetAttribute", &a.funcSetAttribute) && sym(cu, "cuLaunchKernel", &a.launchKernel) &&
               sym(cu, "cuMemcpyDtoH_v2", &a.memcpyDtoH) && sym(cu, "cuMemcpyHtoD_v2", &a.memcpyHtoD) &&
               sym(cu, "cuOccupancyMaxActiveBlocksPerMultiprocessor", &a.occupancy);
    });
    return a;
}

// One compiled kernel: a plan shape on one device.  kind 0: the single-query
// forward <VPT, FULL, FUSED, NORM, S, G, GG, K>; kind 1: the multi-query
// forward <VPT, MB, SEL, MQ, S, G, GG, K>.
using Key = std::tuple<int, int, int, int, int, int, int, int, int, int>;  // device, kind, eight template values
struct Entry {
    bool ok = false;
    CUmodule mod = nullptr;
    CUfunction fn = nullptr;
    CUdeviceptr err = 0;  // the module's wait-failure word
};

// A launch shape checked against the device: `block` threads with `smem`
// bytes of dynamic shared memory, of which at least `ctas` CTAs fit on one SM
// (ok) or do not (rejected).
struct Fit {
    int block, smem, ctas;
    bool ok;
};

// One key's slot: compiled once (outside the cache lock, so launches of
// kernels already compiled never wait for a compile), then the launch shapes
// checked so far.
struct Slot {
    std::once_flag once;
    std::atomic<bool> compiled{false};
    Entry e;
    std::mutex mu;        // guards fits and smem_set
    std::vector<Fit> fits;
    int smem_set = 0;     // dynamic shared memory the function is set up for
};

std::mutex g_mu;  // guards the map only
std::map<Key, std::shared_ptr<Slot>> g_cache;

bool jit_enabled() {
    const char* e = std::getenv("ATTNRES_JIT");
    return !(e && e[0] == '0');
}

Entry compile(const Key& k) {
    Entry e;
    const Api& A = api();
    if (!A.ok) return e;
    const int kind = std::get<1>(k);
    const int t0 = std::get<2>(k), t1 = std::get<3>(k), t2 = std::get<4>(k), t3 = std::get<5>(k);
    const int S = std::get<6>(k), G = std::get<7>(k), GG = std::get<8>(k), K = std::get<9>(k);
    std::vector<const char*> bodies, names;
    for (const auto& f : kJitFiles) {
        names.push_back(f.name);
        bodies.push_back(f.text);
    }
    const char* sys_names[] = {"cstdint", "stdint.h", "cstddef", "stddef.h", "cfloat", "cuda_runtime.h"};
    const char* sys_bodies[] = {kIntTypes, kIntTypes, kIntTypes, kIntTypes, kFloatLimits, kEmpty};
    for (int i = 0; i < 6; ++i) {
        names.push_back(sys_names[i]);
        bodies.push_back(sys_bodies[i]);
    }
    const char* src = kind == 0 ? "#define ATTNRES_FWD_NS jit\n#include \"attnres_fwd_kernel.cuh\"\n"
                                : "#define ATTNRES_FWD_NS jit\n#include \"attnres_multi_fwd_kernel.cuh\"\n";
    char expr[192];
    if (kind == 0)
        std::snprintf(expr, sizeof expr, "attnres::jit::attnres_fwd_kernel<%d, %s, %s, %d, %d, %d, %d, %d>", t0,
                      t1 ? "true" : "false", t2 ? "true" : "false", t3, S, G, GG, K);
    else
        std::snprintf(expr, sizeof expr, "attnres::jit::attnres_multi_fwd_kernel<%d, %d, %s, %d, %d, %d, %d, %d>",
                      t0, t1, t2 ? "true" : "false", t3, S, G, GG, K);
    const char* err_expr = kind == 0 ? "&attnres::jit::g_fwd_error" : "&attnres::jit::g_multi_error";
    nvrtcProgram prog;
    if (A.createProgram(&prog, src, "attnres_fwd_jit.cu", static_cast<int>(bodies.size()), bodies.data(),
                        names.data()) != NVRTC_SUCCESS)
        return e;
    A.addNameExpression(prog, expr);
    A.addNameExpression(prog, err_expr);
#ifdef ATTNRES_DEBUG
    const char* opts[] = {"-arch=sm_103a", "-std=c++17", "-lineinfo", "-default-device", "-DATTNRES_DEBUG"};
#else
    const char* opts[] = {"-arch=sm_103a", "-std=c++17", "-lineinfo", "-default-device"};
#endif
    bool good = A.compileProgram(prog, static_cast<int>(sizeof opts / sizeof opts[0]), opts) == NVRTC_SUCCESS;
    std::string fn_name, err_name;
    std::vector<char> cubin;
    if (good) {
        const char* low = nullptr;
        good = A.getLoweredName(prog, expr, &low) == NVRTC_SUCCESS && low;
        if (good) fn_name = low;
        good = good && A.getLoweredName(prog, err_expr, &low) == NVRTC_SUCCESS && low;
        if (good) err_name = low;
        size_t n = 0;
        good = good && A.getCUBINSize(prog, &n) == NVRTC_SUCCESS && n > 0;
        if (good) {
            cubin.resize(n);
            good = A.getCUBIN(prog, cubin.data()) == NVRTC_SUCCESS;
        }
    }
    A.destroyProgram(&prog);
    if (!good) return e;
    cudaFree(nullptr);  // the runtime's primary context is current on this thread
    size_t bytes = 0;
    if (A.moduleLoadData(&e.mod, cubin.data()) != CUDA_SUCCESS) return e;
    if (A.moduleGetFunction(&e.fn, e.mod, fn_name.c_str()) != CUDA_SUCCESS) return e;
    if (A.moduleGetGlobal(&e.err, &bytes, e.mod, err_name.c_str()) != CUDA_SUCCESS || bytes != sizeof(unsigned))
        return e;
    e.ok = true;
    return e;
}


// Compile (once) and launch the kernel for key k with one struct argument.
// `ctas_per_sm` is what the plan counted on: a compiled kernel that fits
// fewer is not used.
cudaError_t launch_key(const Key& k, unsigned grid, unsigned block, int smem, int ctas_per_sm, const void* args,
                       cudaStream_t stream) {
    std::shared_ptr<Slot> slot;
    {
        std::lock_guard<std::mutex> lock(g_mu);
        auto& p = g_cache[k];
        if (!p) p = std::make_shared<Slot>();
        slot = p;
    }
    if (!slot->compiled.load(std::memory_order_acquire)) {
        // Compiling and loading a module are not stream work: during a
        // CUDA-graph capture they could invalidate it, so a shape first seen
        // there runs the precompiled kernel (and compiles later).
        cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
        if (cudaStreamIsCapturing(stream, &cap) != cudaSuccess || cap != cudaStreamCaptureStatusNone)
            return cudaErrorNotSupported;
        std::call_once(slot->once, [&] {
            slot->e = compile(k);
            slot->compiled.store(true, std::memory_order_release);
        });
    }
    const Entry& e = slot->e;
    if (!e.ok) return cudaErrorNotSupported;
    {
        // The launch shape must fit as many CTAs per SM as the plan counted
        // on.  A shape no larger (block, shared memory) and asking no more
        // CTAs than one already found to fit, fits; one no smaller than a
        // rejected shape is rejected; anything else is checked now.
        // Rejections are per shape: other launches of the key still use it.
        std::lock_guard<std::mutex> lock(slot->mu);
        int verdict = 0;  // 1 fits, -1 does not, 0 unknown
        for (const Fit& f : slot->fits) {
            if (f.ok && static_cast<int>(block) <= f.block && smem <= f.smem && ctas_per_sm <= f.ctas) verdict = 1;
            if (!f.ok && static_cast<int>(block) >= f.block && smem >= f.smem && ctas_per_sm >= f.ctas) verdict = -1;
            if (verdict) break;
        }
        if (verdict < 0) return cudaErrorNotSupported;
        if (verdict == 0) {
            if (smem > slot->smem_set) {
                if (api().funcSetAttribute(e.fn, CU_FUNC_ATTRIBUTE_MAX_DYNAMIC_SHARED_SIZE_BYTES, smem) != CUDA_SUCCESS)
                    return cudaErrorNotSupported;
                slot->smem_set = smem;
            }
            int fit = 0;
            const bool ok = api().occupancy(&fit, e.fn, static_cast<int>(block), static_cast<size_t>(smem)) ==
                                CUDA_SUCCESS &&
                            fit >= ctas_per_sm;
            slot->fits.push_back(Fit{static_cast<int>(block), smem, ok ? fit : ctas_per_sm, ok});
            if (!ok) return cudaErrorNotSupported;
        } else if (smem > slot->smem_set) {
            if (api().funcSetAttribute(e.fn, CU_FUNC_ATTRIBUTE_MAX_DYNAMIC_SHARED_SIZE_BYTES, smem) != CUDA_SUCCESS)
                return cudaErrorNotSupported;
            slot->smem_set = smem;
        }
    }
    void* params[] = {const_cast<void*>(args)};
    const CUresult r = api().launchKernel(e.fn, grid, 1, 1, block, 1, 1, static_cast<unsigned>(smem),
                                          reinterpret_cast<CUstream>(stream), params, nullptr);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorLaunchFailure;
}

int sm_count() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return 0;
    return n;
}

}  // namespace

cudaError_t jit_launch_fwd(const Plan& plan, const FwdArgs& a, cudaStream_t stream) {
    if (!jit_enabled()) return cudaErrorNotSupported;
    int dev = 0;
    const int sms = sm_count();
    if (cudaGetDevice(&dev) != cudaSuccess || sms == 0) return cudaErrorNotSupported;
    const int fused = a.delta ? 1 : 0;
    const int full = (!fused && (a.D / 8) == plan.vpt * 32 * plan.ncw) ? 1 : 0;
    const int norm = !a.out_norm ? 0 : (a.o_pre ? 2 : 1);
    const Key k{dev, 0, plan.vpt, full, fused, norm, a.S, a.rows, a.group, a.chunks};
    return launch_key(k, static_cast<unsigned>(plan.fgrid), static_cast<unsigned>((plan.ncw + 1) * 32),
                      static_cast<int>(plan.smem_fwd), (plan.fgrid + sms - 1) / sms, &a, stream);
}

cudaError_t jit_launch_multi_fwd(const MultiPlan& plan, const MultiFwdArgs& a, cudaStream_t stream) {
    if (!jit_enabled()) return cudaErrorNotSupported;
    int dev = 0;
    const int sms = sm_count();
    if (cudaGetDevice(&dev) != cudaSuccess || sms == 0) return cudaErrorNotSupported;
    const Key k{dev, 1, plan.vpt, plan.mb_f, a.ids ? 1 : 0, plan.mq, a.S, a.rows, a.group, a.chunks};
    return launch_key(k, static_cast<unsigned>(plan.fgrid), static_cast<unsigned>((plan.ncw + 1) * 32),
                      static_cast<int>(plan.smem_fwd), (plan.fgrid + sms - 1) / sms, &a, stream);
}

unsigned take_jit_error(int kind) {
    std::lock_guard<std::mutex> lock(g_mu);
    unsigned first = 0;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    for (auto& kv : g_cache) {
        if (!kv.second || !kv.second->compiled.load(std::memory_order_acquire)) continue;
        const Entry& e = kv.second->e;
        if (!e.mod || !e.err || std::get<0>(kv.first) != dev || std::get<1>(kv.first) != kind) continue;
        unsigned v = 0;
        if (api().memcpyDtoH(&v, e.err, sizeof v) != CUDA_SUCCESS) return 0xffffffffu;
        if (v) {
            const unsigned zero = 0;
            api().memcpyHtoD(e.err, &zero, sizeof zero);
            if (!first) first = v;
        }
    }
    return first;
}

int jit_fwd_kernels() {
    std::lock_guard<std::mutex> lock(g_mu);
    int n = 0;
    for (auto& kv : g_cache)
        n += (kv.second && kv.second->compiled.load(std::memory_order_acquire) && kv.second->e.ok) ? 1 : 0;
    return n;
}

}  // namespace attnres
