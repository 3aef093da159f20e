// common.cuh -- small device helpers shared by the library's kernels.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "moe.h"
#include "nvtx3/nvToolsExt.h"

namespace moe {

// An NVTX range named after a C-ABI entry point, for the duration of the call
// (host-side enqueue time; a profiler that attaches through NVTX shows the
// kernels each call launched inside it).  Without an attached tool the push
// and pop return at once.
struct NvtxRange {
    explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
    ~NvtxRange() { nvtxRangePop(); }
    NvtxRange(const NvtxRange&) = delete;
    NvtxRange& operator=(const NvtxRange&) = delete;
};

// Debug build that range-checks indices read from callers' buffers.
#ifdef MOE_CHECKED
constexpr bool kChecked = true;
#else
constexpr bool kChecked = false;
#endif

// Upper bound on any bounded device wait (nanoseconds of %globaltimer).
constexpr uint64_t kWaitTimeoutNs = 4000000000ull;  // 4 s

__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ unsigned lanemask_lt() {
    unsigned m;
    asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
    return m;
}

// Element traits: fp32 and bf16 storage, fp32 arithmetic.
template <typename T>
struct Elem;

template <>
struct Elem<float> {
    static constexpr int kPerVec = 4;  // elements per 16-byte vector
    __device__ __forceinline__ static void unpack(const uint4& v, float* f) {
        f[0] = __uint_as_float(v.x);
        f[1] = __uint_as_float(v.y);
        f[2] = __uint_as_float(v.z);
        f[3] = __uint_as_float(v.w);
    }
    __device__ __forceinline__ static uint4 pack(const float* f) {
        return make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]), __float_as_uint(f[2]),
                          __float_as_uint(f[3]));
    }
    __device__ __forceinline__ static float to_f(float v) { return v; }
    __device__ __forceinline__ static float from_f(float v) { return v; }
};

template <>
struct Elem<__nv_bfloat16> {
    static constexpr int kPerVec = 8;
    __device__ __forceinline__ static void unpack2(uint32_t w, float* f) {
        f[0] = __uint_as_float(w << 16);
        f[1] = __uint_as_float(w & 0xffff0000u);
    }
    __device__ __forceinline__ static void unpack(const uint4& v, float* f) {
        unpack2(v.x, f + 0);
        unpack2(v.y, f + 2);
        unpack2(v.z, f + 4);
        unpack2(v.w, f + 6);
    }
    __device__ __forceinline__ static uint32_t pack2(float a, float b) {
        __nv_bfloat162 h = __floats2bfloat162_rn(a, b);  // .x = a (low half)
        return *reinterpret_cast<uint32_t*>(&h);
    }
    __device__ __forceinline__ static uint4 pack(const float* f) {
        return make_uint4(pack2(f[0], f[1]), pack2(f[2], f[3]), pack2(f[4], f[5]),
                          pack2(f[6], f[7]));
    }
    __device__ __forceinline__ static float to_f(__nv_bfloat16 v) { return __bfloat162float(v); }
    __device__ __forceinline__ static __nv_bfloat16 from_f(float v) { return __float2bfloat16_rn(v); }
};

__device__ __forceinline__ uint4 ld_nc_v4(const void* p) {
    uint4 v;
    asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ uint4 ld_v4(const void* p) {
    return *reinterpret_cast<const uint4*>(p);
}

__device__ __forceinline__ void st_v4(void* p, const uint4& v) {
    *reinterpret_cast<uint4*>(p) = v;
}

// Streaming store (evict-first): output rows that are not re-read soon.
__device__ __forceinline__ void st_cs_v4(void* p, const uint4& v) {
    asm volatile("st.global.cs.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z),
                 "r"(v.w)
                 : "memory");
}

__device__ __forceinline__ uint64_t ld_relaxed_u64(const uint64_t* p) {
    uint64_t v;
    asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void st_relaxed_u64(uint64_t* p, uint64_t v) {
    asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

// Programmatic dependent launch.  A kernel launched with launch_pdl is
// pre-staged behind the kernel before it on the stream; pdl_wait blocks the
// calling thread until that kernel has completed and its memory writes are
// visible, so each kernel calls it before its first global read of the
// previous kernel's results (and before any global write).  No kernel here
// triggers its dependents early (griddepcontrol.launch_dependents): with early
// triggers the next kernel's CTAs became resident beside long-running ones and
// waited there, and whole-layer steps ran 2-5 % slower (Mixtral shape 8.17 ->
// 7.78 ms, DeepSeek shape 6.50 -> 6.37 ms without them), while the short
// kernels of small batches kept the launch-latency gain of the pre-staging.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// The fp32 expert activations: GELU in its erf form, 0.5 v (1 + erf(v / sqrt 2)),
// and SiLU, v / (1 + e^-v).
__device__ __forceinline__ float gelu_erf_f(float v) {
    return 0.5f * v * (1.f + erff(v * 0.70710678118654752440f));
}
__device__ __forceinline__ float silu_exact_f(float v) { return v / (1.f + expf(-v)); }

// Counts one kernel launch enqueued by this library (moe_launch_count).
void note_launch();
// Counts the launch just made with <<<...>>> if it was accepted; returns its error.
inline cudaError_t noted_launch() {
    cudaError_t e = cudaGetLastError();
    if (e == cudaSuccess) note_launch();
    return e;
}

// Launch with programmatic stream serialization (see pdl_wait).
template <typename K, typename... Args>
cudaError_t launch_pdl(K kernel, dim3 grid, unsigned block, size_t smem, cudaStream_t s,
                       Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(block);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, args...);
    if (e == cudaSuccess) note_launch();
    return e;
}

// Programmatic dependent launch of a kernel whose CTAs form thread-block
// clusters of `cluster` CTAs (the grid a multiple of it in every dimension).
template <typename K, typename... Args>
cudaError_t launch_pdl_cluster(K kernel, dim3 grid, unsigned block, size_t smem, cudaStream_t s,
                               dim3 cluster, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(block);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = cluster.x;
    attr[1].val.clusterDim.y = cluster.y;
    attr[1].val.clusterDim.z = cluster.z;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, args...);
    if (e == cudaSuccess) note_launch();
    return e;
}

// Thread-block clusters: this CTA's rank, a barrier over every thread of the
// cluster (release / acquire), and loads from another CTA's shared memory.
__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::
                     : "memory");
}
// Shared-memory address of the same variable in CTA `rank` of this cluster.
__device__ __forceinline__ uint32_t cluster_addr(const void* p, uint32_t rank) {
    uint32_t out;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;"
                 : "=r"(out)
                 : "r"(static_cast<uint32_t>(__cvta_generic_to_shared(p))), "r"(rank));
    return out;
}
__device__ __forceinline__ float ld_cluster_f32(uint32_t addr) {
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
    return v;
}

// Key order of the router's selection: larger key first, ties to the lower index.
__device__ __forceinline__ bool key_better(float a, int ia, float b, int ib) {
    return a > b || (a == b && ia < ib);
}

}  // namespace moe
