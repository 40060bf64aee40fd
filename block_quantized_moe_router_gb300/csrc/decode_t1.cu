// decode_t1.cu -- the fused few-token MoE block instantiated for one token: activation chunks
// of 256 B per K-step instead of 2 KiB, so its stages are 3 KiB instead of 6.5 KiB.
#include "decode_kernel.cuh"

namespace moe {

cudaError_t launch_decode_fused_t1(const FfnLaunch& L, const DecRoute& R, unsigned long long* bar,
                                   int sms, cudaStream_t st) {
    return launch_decode_fused_ntok<1>(L, R, bar, sms, st);
}

}  // namespace moe
