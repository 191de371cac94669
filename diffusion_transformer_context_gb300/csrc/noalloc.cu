// ctx_attn_lq_gkv_noalloc: the balanced attention schedule for callers that
// cannot allocate device memory.
//
// The balanced schedule needs a workspace (partial results of key-split
// units and their arrival counters). Most callers pass one to
// ctx_attn_lq_gkv. Some callers have no way to do that: a host framework
// that owns every device buffer and hands a plugin only its inputs and
// outputs, a plain C program that embeds this library without a device
// allocator of its own, or a latency-critical path that must not call
// cudaMalloc because it can synchronise the whole device. For them the
// workspace lives here instead, in one fixed-size array in device memory
// that every GPU loading the library holds until the process exits.
//
// Nothing is allocated on any call: the array exists once the module is
// loaded, and its device address is looked up once per device, on the first
// call made with that device current (so make that first call before any
// stream capture begins). All calls share the array and it keeps the last
// call's contents; the part that must start at zero (the arrival counters)
// is cleared after every call. Calls that can overlap on the GPU (different
// streams, or different host threads) race on the array: serialise them.
#include <cstdint>
#include <mutex>

#include "../../include/ctx.h"
#include "internal.h"

namespace {

// 44 MiB: the partial-result slots of a 160-SM grid at D = 128 (41.6 MB)
// plus arrival counters for up to 131072 work units.
constexpr long long kScratchBytes = 44LL << 20;

static __device__ __align__(256) unsigned char g_attn_scratch[kScratchBytes];

std::mutex g_mu;
void *g_scratch_addr[64] = {nullptr};

// Device address of g_attn_scratch on the current device. In host code the
// array's name only stands in for the symbol; the kernel must get this
// address instead.
cudaError_t scratch_address(void **out)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    if (dev < 0 || dev >= 64)
        return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> g(g_mu);
    if (!g_scratch_addr[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_attn_scratch);
        if (e != cudaSuccess)
            return e;
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return cudaSuccess;
}

}  // namespace

extern "C" ctx_status ctx_attn_lq_gkv_noalloc(const void *q, const void *k, const void *v,
                                              const unsigned char *key_mask, float scale, void *out, float *lse,
                                              int B, int Sq, int Sk, int H, int D, ctx_dtype dtype, void *stream)
{
    if (B <= 0 || Sq <= 0 || Sk <= 0 || H <= 0)
        return CTX_ERR_INVALID_ARG;
    if (D != 64 && D != 128)
        return CTX_ERR_UNSUPPORTED;
    const long long need = ctx_attn_lq_gkv_workspace_size(B, Sq, Sk, H, D);
    if (need < 0) {
        ctx::record_cuda_error(cudaErrorUnknown);
        return CTX_ERR_CUDA;
    }
    if (need > kScratchBytes)
        return CTX_ERR_UNSUPPORTED;  // more work units or SMs than the fixed scratch holds
    void *ws = nullptr;
    cudaError_t e = scratch_address(&ws);
    if (e != cudaSuccess) {
        ctx::record_cuda_error(e);
        return CTX_ERR_CUDA;
    }
    const ctx_status s = ctx_attn_lq_gkv(q, k, v, key_mask, scale, out, lse, ws, kScratchBytes, B, Sq, Sk, H, D,
                                         dtype, stream);
    if (s != CTX_OK)
        return s;
    // Arrival counters sit at the head of the workspace: clear them for the
    // next call even if this one ended early on the device.
    const long long n_units = static_cast<long long>((Sq + 255) / 256) * H * B;
    const long long counter_bytes = (n_units * 2 * 4 + 255) / 256 * 256;
    e = cudaMemsetAsync(ws, 0, static_cast<size_t>(counter_bytes), static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) {
        ctx::record_cuda_error(e);
        return CTX_ERR_CUDA;
    }
    return CTX_OK;
}
