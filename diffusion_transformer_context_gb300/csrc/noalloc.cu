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
// loaded. Its device address is looked up again by every call made outside a
// stream capture (a device reset reloads the module, possibly at another
// address); make the first call on each device before any stream capture.
// All calls share the array and it keeps the last call's contents; the part
// that must start at zero (the arrival counters) is cleared after every call.
// Calls that can overlap on the GPU (different streams, or different host
// threads) race on the array: serialise them.
#include <cstdint>

#include "../../include/ctx.h"
#include "internal.h"

namespace {

// 44 MiB: the partial-result slots of a 160-SM grid at D = 128 (42.6 MB)
// plus the arrived / written counters of up to 131072 work units (2 MiB).
constexpr long long kScratchBytes = 44LL << 20;

static __device__ __align__(256) unsigned char g_attn_scratch[kScratchBytes];

// Last looked-up device address of g_attn_scratch, per device. In host code
// the array's name only stands in for the symbol; the kernel must get this
// address instead.
void *g_scratch_addr[64] = {nullptr};

// B*Sq*H*D and B*Sk*H*D within 2^62 and at most INT_MAX work units: the sizes
// the attention entry point accepts.
bool sizes_ok(int B, int Sq, int Sk, int H, int D)
{
    const long long lim = 1LL << 62;
    long long nq = 1, nk = 1;
    for (long long x : {static_cast<long long>(B), static_cast<long long>(Sq), static_cast<long long>(H),
                        static_cast<long long>(D)}) {
        if (nq > lim / x)
            return false;
        nq *= x;
    }
    for (long long x : {static_cast<long long>(B), static_cast<long long>(Sk), static_cast<long long>(H),
                        static_cast<long long>(D)}) {
        if (nk > lim / x)
            return false;
        nk *= x;
    }
    return ctx::attention_units(B, Sq, H) <= 0x7fffffffLL;
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
    if (!sizes_ok(B, Sq, Sk, H, D))
        return CTX_ERR_INVALID_ARG;
    cudaError_t e = cudaSuccess;
    const long long need = ctx::attention_workspace_size(B, Sq, Sk, H, D, &e);
    if (e != cudaSuccess) {
        ctx::record_cuda_error(e);
        return CTX_ERR_CUDA;
    }
    if (need > kScratchBytes)
        return CTX_ERR_UNSUPPORTED;  // more work units or SMs than the fixed scratch holds
    void *ws = nullptr;
    e = ctx::device_symbol_address(reinterpret_cast<const void *>(&g_attn_scratch), g_scratch_addr,
                                   static_cast<cudaStream_t>(stream), &ws);
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
    e = cudaMemsetAsync(ws, 0, static_cast<size_t>(ctx::attention_counter_bytes(B, Sq, H)),
                        static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) {
        ctx::record_cuda_error(e);
        return CTX_ERR_CUDA;
    }
    return CTX_OK;
}
