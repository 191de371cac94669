// Packed varlen query metadata for one rank of the AllGather-KV group
// (vllm-omni PR #7641, packed query metadata): every global query document
// [cu[d], cu[d+1]) is intersected with the rank's span [lo, lo + len); the
// rank keeps one (possibly empty) entry per document, prefix-summed from 0,
// computed on the device so no host synchronisation is needed per layer.
// The single-document [real, pad] view narrows its query length to the
// rank's valid prefix. One block; documents in chunks of its size with a
// block-wide scan and a running carry.
#include <algorithm>

#include "internal.h"

namespace ctx {
namespace {

constexpr int kRemapThreads = 1024;

__global__ void __launch_bounds__(kRemapThreads) varlen_remap_kernel(const int *cu_g, int n_docs, long long lo,
                                                                      long long len, int *cu_l, const int *pad_in,
                                                                      int *pad_out)
{
    __shared__ int warp_sums[kRemapThreads / 32];
    __shared__ int carry;
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    const long long hi = lo + len;
    if (tid == 0) {
        carry = 0;
        cu_l[0] = 0;
        if (pad_in && pad_out) {
            const long long real = pad_in[0];
            const long long local = min(max(real - lo, 0LL), len);
            pad_out[0] = static_cast<int>(local);
            pad_out[1] = static_cast<int>(len - local);
        }
    }
    __syncthreads();
    for (int base = 0; base < n_docs; base += kRemapThreads) {
        const int d = base + tid;
        int v = 0;
        if (d < n_docs) {
            const long long a = max(static_cast<long long>(cu_g[d]), lo);
            const long long b = min(static_cast<long long>(cu_g[d + 1]), hi);
            v = static_cast<int>(max(b - a, 0LL));
        }
        // inclusive scan: inside the warp, then over warp totals
        for (int o = 1; o < 32; o <<= 1) {
            const int x = __shfl_up_sync(0xffffffffu, v, o);
            if (lane >= o)
                v += x;
        }
        if (lane == 31)
            warp_sums[wid] = v;
        __syncthreads();
        if (wid == 0) {
            int w = warp_sums[lane];
            for (int o = 1; o < 32; o <<= 1) {
                const int x = __shfl_up_sync(0xffffffffu, w, o);
                if (lane >= o)
                    w += x;
            }
            warp_sums[lane] = w;
        }
        __syncthreads();
        const int prefix = carry + (wid > 0 ? warp_sums[wid - 1] : 0);
        if (d < n_docs)
            cu_l[d + 1] = prefix + v;
        __syncthreads();
        if (tid == kRemapThreads - 1)
            carry = prefix + v;
        __syncthreads();
    }
}

}  // namespace

cudaError_t launch_varlen_remap(const int *cu_g, int n_docs, long long lo, long long len, int *cu_l,
                                const int *pad_in, int *pad_out, cudaStream_t stream)
{
    varlen_remap_kernel<<<1, kRemapThreads, 0, stream>>>(cu_g, n_docs, lo, len, cu_l, pad_in, pad_out);
    return cudaGetLastError();
}

}  // namespace ctx
