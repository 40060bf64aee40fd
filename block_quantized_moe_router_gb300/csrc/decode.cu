// decode.cu -- host entry of the fused few-token MoE block (the kernel is in decode_kernel.cuh;
// the one-token instantiations are compiled in decode_t1.cu).
#include "decode_kernel.cuh"

namespace moe {

cudaError_t launch_decode_fused(const FfnLaunch& L, const DecRoute& R, unsigned long long* bar,
                                int sms, cudaStream_t st) {
    if (L.T < 1 || L.T > kDecMaxT) return cudaErrorInvalidValue;
    if (L.T == 1) return launch_decode_fused_t1(L, R, bar, sms, st);
    return launch_decode_fused_ntok<kDecMaxT>(L, R, bar, sms, st);
}

// The barrier epoch one ahead of the arrival counter: no barrier of the next fused launch can
// complete, and every wait runs out its limit (a test aid for the bounded waits; nothing else
// launches it).
__global__ void barrier_skew_kernel(unsigned long long* bar) { atomicAdd(bar + 1, 1ull); }

cudaError_t launch_barrier_skew(unsigned long long* bar, cudaStream_t st) {
    if (!bar) return cudaErrorInvalidValue;
    barrier_skew_kernel<<<1, 1, 0, st>>>(bar);
    return cudaGetLastError();
}

}  // namespace moe
