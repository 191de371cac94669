// Key mask of the gathered key layout (vllm-omni PR #7641, follow-up review
// commit: after the K/V AllGather and the re-attach of the joint text keys,
// one merge owns the 2-D key mask). The gathered keys are S_img image keys
// and J joint keys, the joint segment first or last; a key is valid when its
// side has no mask or its mask byte is nonzero. Output bytes are 0/1.
//
// The mask is a few KB per batch row and is built once per forward, so the
// kernel is a plain grid-stride loop: one output byte per thread and step,
// both inputs read with one byte load each (L2 holds them).
#include <algorithm>

#include "internal.h"

namespace ctx {
namespace {

constexpr int kMaskThreads = 256;

__global__ void __launch_bounds__(kMaskThreads)
    merge_mask_kernel(const unsigned char *img, const unsigned char *jnt, long long B, long long S_img, long long J,
                      int front, unsigned char *out)
{
    const long long K = S_img + J;
    const long long n = B * K;
    const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
    for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < n; i += stride) {
        const long long b = i / K, pos = i - b * K;
        const long long j = front ? pos : pos - S_img;  // position inside the joint segment
        unsigned char valid;
        if (j >= 0 && j < J) {
            valid = jnt ? (jnt[b * J + j] != 0) : 1;
        } else {
            const long long s = front ? pos - J : pos;  // position inside the image segment
            valid = img ? (img[b * S_img + s] != 0) : 1;
        }
        out[i] = valid;
    }
}

}  // namespace

cudaError_t launch_merge_mask(const unsigned char *img, const unsigned char *jnt, int B, int S_img, int J, int front,
                              unsigned char *out, cudaStream_t stream)
{
    cudaError_t err = cudaSuccess;
    const int sms = sm_count(&err);
    if (err != cudaSuccess)
        return err;
    const long long n = static_cast<long long>(B) * (static_cast<long long>(S_img) + J);
    const long long blocks = std::min<long long>((n + kMaskThreads - 1) / kMaskThreads, 8LL * sms);
    merge_mask_kernel<<<static_cast<unsigned>(std::max<long long>(blocks, 1)), kMaskThreads, 0, stream>>>(
        img, jnt, B, S_img, J, front, out);
    return cudaGetLastError();
}

}  // namespace ctx
