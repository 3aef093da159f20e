// balance.cu -- bias-based load balancing of the selection-only bias.
//
// Ultralytics glossary "Expert Parallelism", "Load Balancing and Capacity":
// DeepSeek-V3 lowers the selection bias of overloaded experts and raises it
// for idle ones after each step, which balances the load without an auxiliary
// loss.  Here an expert is overloaded when its load (assignments before drops)
// is above the even share T*k/E and underloaded when below it; the comparison
// is exact (count*E against T*k as integers) and the update is one fp32 add of
// -gamma or +gamma.  The step size gamma is the caller's.
#include "common.cuh"
#include "kernels.h"

namespace moe {
namespace {

__global__ void update_sel_bias_kernel(const int32_t* counts, float* bias, int E, int64_t even,
                                       float gamma) {
    const int e = blockIdx.x * blockDim.x + threadIdx.x;
    if (e >= E) return;
    const int64_t load = (int64_t)counts[e] * E;
    if (load > even)
        bias[e] = __fsub_rn(bias[e], gamma);
    else if (load < even)
        bias[e] = __fadd_rn(bias[e], gamma);
}

}  // namespace

cudaError_t launch_update_sel_bias(const int32_t* counts, float* bias, int E, int64_t T, int k,
                                   float gamma, cudaStream_t s) {
    update_sel_bias_kernel<<<(E + 255) / 256, 256, 0, s>>>(counts, bias, E, T * (int64_t)k, gamma);
    return noted_launch();
}

}  // namespace moe
