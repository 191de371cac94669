// Packed varlen query metadata for one rank of the AllGather-KV group
// (vllm-omni PR #7641, packed query metadata): every global query document
// [cu[d], cu[d+1]) is intersected with the rank's span [lo, lo + len); the
// rank keeps one (possibly empty) entry per document, prefix-summed from 0,
// computed on the device so no host synchronisation is needed per layer.
// The single-document [real, pad] view narrows its query length to the
// rank's valid prefix. One block; documents in chunks of its size with a
// block-wide scan and a running carry.
#include <algorithm>
#include <cmath>

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

// Plan of the balanced packed-varlen attention: the first split iteration of
// every document (key blocks x query-tile pairs x heads, counted exactly as
// the attention kernel's units), prefix-summed in 64 bits into prefix[0..n],
// so the kernel can hand every SM an equal share of iterations without the
// host knowing the document lengths. Query rows of documents without any key
// are written here (out = 0, lse = -inf): they hold no iteration.
__global__ void __launch_bounds__(kRemapThreads) varlen_plan_kernel(const int *cu_q, const int *cu_k, int n_docs,
                                                                     int Sq, int Sk, int H, int n_qpairs,
                                                                     long long *prefix, uint4 *out, float *lse,
                                                                     int dv)
{
    __shared__ long long warp_sums[kRemapThreads / 32];
    __shared__ long long carry;
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    if (tid == 0) {
        carry = 0;
        prefix[0] = 0;
    }
    __syncthreads();
    for (int base = 0; base < n_docs; base += kRemapThreads) {
        const int d = base + tid;
        long long v = 0;
        if (d < n_docs) {
            const int qs = min(max(cu_q[d], 0), Sq);
            const int q_len = min(max(cu_q[d + 1], qs), Sq) - qs;
            const int k0 = min(max(cu_k[d], 0), Sk);
            const int k_len = min(max(cu_k[d + 1], k0), Sk) - k0;
            const long long nqp = min((q_len + kAttnUnitRows - 1) / kAttnUnitRows, n_qpairs);
            v = static_cast<long long>(H) * nqp * ((k_len + kAttnKeyBlock - 1) / kAttnKeyBlock);
        }
        for (int o = 1; o < 32; o <<= 1) {
            const long long x = __shfl_up_sync(0xffffffffu, v, o);
            if (lane >= o)
                v += x;
        }
        if (lane == 31)
            warp_sums[wid] = v;
        __syncthreads();
        if (wid == 0) {
            long long w = warp_sums[lane];
            for (int o = 1; o < 32; o <<= 1) {
                const long long x = __shfl_up_sync(0xffffffffu, w, o);
                if (lane >= o)
                    w += x;
            }
            warp_sums[lane] = w;
        }
        __syncthreads();
        const long long pre = carry + (wid > 0 ? warp_sums[wid - 1] : 0);
        if (d < n_docs)
            prefix[d + 1] = pre + v;
        __syncthreads();
        if (tid == kRemapThreads - 1)
            carry = pre + v;
        __syncthreads();
    }
    // documents with query rows but no key: the rows the attention computes (the
    // first n_qpairs tile pairs) get out = 0, lse = -inf
    for (int d = 0; d < n_docs; ++d) {
        const int qs = min(max(cu_q[d], 0), Sq);
        const int qe = min(min(max(cu_q[d + 1], qs), Sq), qs + n_qpairs * kAttnUnitRows);
        const int k0 = min(max(cu_k[d], 0), Sk);
        const int k_len = min(max(cu_k[d + 1], k0), Sk) - k0;
        if (k_len > 0 || qe <= qs)
            continue;
        const long long n = static_cast<long long>(qe - qs) * H * dv;
        for (long long i = tid; i < n; i += kRemapThreads)
            out[static_cast<long long>(qs) * H * dv + i] = make_uint4(0u, 0u, 0u, 0u);
        if (lse)
            for (long long i = tid; i < static_cast<long long>(qe - qs) * H; i += kRemapThreads) {
                const long long h = i / (qe - qs), row = qs + i % (qe - qs);
                lse[h * Sq + row] = -INFINITY;
            }
    }
}

}  // namespace

cudaError_t launch_varlen_remap(const int *cu_g, int n_docs, long long lo, long long len, int *cu_l,
                                const int *pad_in, int *pad_out, cudaStream_t stream)
{
    varlen_remap_kernel<<<1, kRemapThreads, 0, stream>>>(cu_g, n_docs, lo, len, cu_l, pad_in, pad_out);
    return cudaGetLastError();
}

cudaError_t launch_varlen_plan(const int *cu_q, const int *cu_k, int n_docs, int Sq, int Sk, int H, int n_qpairs,
                               long long *prefix, void *out, float *lse, int D, cudaStream_t stream)
{
    varlen_plan_kernel<<<1, kRemapThreads, 0, stream>>>(cu_q, cu_k, n_docs, Sq, Sk, H, n_qpairs, prefix,
                                                        static_cast<uint4 *>(out), lse, D / 8);
    return cudaGetLastError();
}

}  // namespace ctx
