// C ABI of libctx (declared in include/ctx.h): host-side validation, then one
// launch per call on the caller's stream. Nothing is allocated here; the only
// device state is one status word per device for bounded-wait timeouts.
#include <cmath>
#include <cstdint>
#include <mutex>

#include "../../include/ctx.h"
#include "internal.h"

namespace ctx {

__device__ int g_status_word;

namespace {
struct DeviceCache {
    std::mutex mu;
    int sms[64] = {0};
};
DeviceCache &cache()
{
    static DeviceCache c;
    return c;
}
}  // namespace

cudaError_t device_symbol_address(const void *symbol, void **slots, cudaStream_t stream, void **out)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    if (dev < 0 || dev >= 64)
        return cudaErrorInvalidDevice;
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    e = cudaStreamIsCapturing(stream, &cs);
    if (e != cudaSuccess)
        return e;
    DeviceCache &c = cache();
    std::lock_guard<std::mutex> g(c.mu);
    if (cs == cudaStreamCaptureStatusNone) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, symbol);
        if (e != cudaSuccess)
            return e;
        slots[dev] = p;
    } else if (!slots[dev]) {
        return cudaErrorStreamCaptureUnsupported;
    }
    *out = slots[dev];
    return cudaSuccess;
}

int *device_status_word(cudaStream_t stream, cudaError_t *err)
{
    static void *addr[64] = {nullptr};
    void *p = nullptr;
    *err = device_symbol_address(reinterpret_cast<const void *>(&g_status_word), addr, stream, &p);
    return *err == cudaSuccess ? static_cast<int *>(p) : nullptr;
}

int sm_count(cudaError_t *err)
{
    int dev = 0;
    *err = cudaGetDevice(&dev);
    if (*err != cudaSuccess)
        return 0;
    if (dev < 0 || dev >= 64) {
        *err = cudaErrorInvalidDevice;
        return 0;
    }
    DeviceCache &c = cache();
    std::lock_guard<std::mutex> g(c.mu);
    if (!c.sms[dev]) {
        *err = cudaDeviceGetAttribute(&c.sms[dev], cudaDevAttrMultiProcessorCount, dev);
        if (*err != cudaSuccess)
            return 0;
    }
    return c.sms[dev];
}

}  // namespace ctx

namespace {

thread_local int t_last_cuda_error = 0;

using ctx::RelayoutArgs;
using ctx::RelayoutMode;

struct Extent {
    uintptr_t lo, hi;  // [lo, hi)
};

Extent extent(const void *p, long long bytes)
{
    uintptr_t lo = reinterpret_cast<uintptr_t>(p);
    return Extent{lo, lo + static_cast<uintptr_t>(bytes)};
}

bool overlap(Extent a, Extent b)
{
    return a.lo < b.hi && b.lo < a.hi;
}

bool aligned16(const void *p)
{
    return (reinterpret_cast<uintptr_t>(p) & 15u) == 0;
}

bool valid_dtype(ctx_dtype d)
{
    return d == CTX_BF16 || d == CTX_FP16;
}

// Product of sizes, false on overflow past 2^62.
bool mul_ok(long long &acc, long long x)
{
    if (x <= 0)
        return false;
    if (acc > (1LL << 62) / x)
        return false;
    acc *= x;
    return true;
}

ctx_status cuda_fail(cudaError_t e)
{
    t_last_cuda_error = static_cast<int>(e);
    return CTX_ERR_CUDA;
}

// Device (or managed) memory check; runs after every host-only check.
ctx_status check_device_ptrs(std::initializer_list<const void *> ptrs)
{
    for (const void *p : ptrs) {
        if (!p)
            continue;
        cudaPointerAttributes attr;
        cudaError_t e = cudaPointerGetAttributes(&attr, p);
        if (e != cudaSuccess) {
            cudaGetLastError();
            return cuda_fail(e);
        }
        if (attr.type != cudaMemoryTypeDevice && attr.type != cudaMemoryTypeManaged)
            return CTX_ERR_INVALID_ARG;
    }
    return CTX_OK;
}

ctx_status run_relayout(RelayoutMode mode, const RelayoutArgs &a, void *stream)
{
    cudaError_t e = ctx::launch_relayout(mode, a, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? CTX_OK : cuda_fail(e);
}

}  // namespace

void ctx::record_cuda_error(cudaError_t e)
{
    t_last_cuda_error = static_cast<int>(e);
}

extern "C" {

int ctx_version(void)
{
    return 100;  // 0.1.0
}

const char *ctx_status_string(ctx_status s)
{
    switch (s) {
    case CTX_OK: return "CTX_OK";
    case CTX_ERR_INVALID_ARG: return "CTX_ERR_INVALID_ARG";
    case CTX_ERR_UNSUPPORTED: return "CTX_ERR_UNSUPPORTED";
    case CTX_ERR_MISALIGNED: return "CTX_ERR_MISALIGNED";
    case CTX_ERR_ALIASING: return "CTX_ERR_ALIASING";
    case CTX_ERR_CUDA: return "CTX_ERR_CUDA";
    case CTX_ERR_TIMEOUT: return "CTX_ERR_TIMEOUT";
    }
    return "CTX_ERR_UNKNOWN";
}

int ctx_last_cuda_error(void)
{
    return t_last_cuda_error;
}

ctx_status ctx_pack_qkv(const void *q, const void *k, const void *v, void *staging, int B, int S_l, int H, int D,
                        int U, ctx_dtype dtype, void *stream)
{
    if (!q || !k || !v || !staging || !valid_dtype(dtype))
        return CTX_ERR_INVALID_ARG;
    long long n = 1;
    if (!mul_ok(n, B) || !mul_ok(n, S_l) || !mul_ok(n, H) || !mul_ok(n, D) || U <= 0 || H % U != 0)
        return CTX_ERR_INVALID_ARG;
    if (D % 8 != 0 || !aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(staging))
        return CTX_ERR_MISALIGNED;
    const long long bytes = n * 2;
    const Extent st = extent(staging, 3 * bytes);
    if (overlap(st, extent(q, bytes)) || overlap(st, extent(k, bytes)) || overlap(st, extent(v, bytes)))
        return CTX_ERR_ALIASING;
    ctx_status s = check_device_ptrs({q, k, v, staging});
    if (s != CTX_OK)
        return s;
    RelayoutArgs a{};
    a.src0 = q;
    a.src1 = k;
    a.src2 = v;
    a.dst0 = staging;
    a.B = B;
    a.S_l = S_l;
    a.H = H;
    a.U = U;
    a.h_l = H / U;
    a.run_vec = static_cast<long long>(H / U) * D / 8;
    a.n_runs = 3LL * U * B * S_l;
    return run_relayout(RelayoutMode::PackQKV, a, stream);
}

ctx_status ctx_sim_all_to_all(const void *send, void *recv, int G, int U, long long chunk_bytes, void *stream)
{
    if (!send || !recv)
        return CTX_ERR_INVALID_ARG;
    long long n = 1;
    if (!mul_ok(n, G) || !mul_ok(n, U) || !mul_ok(n, U) || !mul_ok(n, chunk_bytes))
        return CTX_ERR_INVALID_ARG;
    if (chunk_bytes % 16 != 0 || !aligned16(send) || !aligned16(recv))
        return CTX_ERR_MISALIGNED;
    if (overlap(extent(send, n), extent(recv, n)))
        return CTX_ERR_ALIASING;
    ctx_status s = check_device_ptrs({send, recv});
    if (s != CTX_OK)
        return s;
    RelayoutArgs a{};
    a.src0 = send;
    a.dst0 = recv;
    a.U = U;
    a.G = G;
    a.run_vec = chunk_bytes / 16;
    a.n_runs = static_cast<long long>(G) * U * U;
    return run_relayout(RelayoutMode::AllToAll, a, stream);
}

ctx_status ctx_unpack_qkv(const void *recv, void *q, void *k, void *v, long long q_batch_stride_rows,
                          long long kv_batch_stride_rows, int B, int S_l, int h_l, int D, int U, ctx_dtype dtype,
                          void *stream)
{
    if (!recv || !q || !k || !v || !valid_dtype(dtype))
        return CTX_ERR_INVALID_ARG;
    long long n = 1;
    if (!mul_ok(n, B) || !mul_ok(n, S_l) || !mul_ok(n, h_l) || !mul_ok(n, D) || !mul_ok(n, U))
        return CTX_ERR_INVALID_ARG;
    const long long rows = static_cast<long long>(U) * S_l;
    if (q_batch_stride_rows < rows || kv_batch_stride_rows < rows)
        return CTX_ERR_INVALID_ARG;
    const long long row_bytes = static_cast<long long>(h_l) * D * 2;
    long long qspan = q_batch_stride_rows, kvspan = kv_batch_stride_rows;
    if (!mul_ok(qspan, B) || !mul_ok(qspan, row_bytes) || !mul_ok(kvspan, B) || !mul_ok(kvspan, row_bytes))
        return CTX_ERR_INVALID_ARG;
    if (D % 8 != 0 || !aligned16(recv) || !aligned16(q) || !aligned16(k) || !aligned16(v))
        return CTX_ERR_MISALIGNED;
    const long long q_bytes = ((static_cast<long long>(B) - 1) * q_batch_stride_rows + rows) * row_bytes;
    const long long kv_bytes = ((static_cast<long long>(B) - 1) * kv_batch_stride_rows + rows) * row_bytes;
    const Extent r = extent(recv, 3 * n * 2);
    const Extent eq = extent(q, q_bytes), ek = extent(k, kv_bytes), ev = extent(v, kv_bytes);
    if (overlap(r, eq) || overlap(r, ek) || overlap(r, ev) || overlap(eq, ek) || overlap(eq, ev) ||
        overlap(ek, ev))
        return CTX_ERR_ALIASING;
    ctx_status s = check_device_ptrs({recv, q, k, v});
    if (s != CTX_OK)
        return s;
    RelayoutArgs a{};
    a.src0 = recv;
    a.dst0 = q;
    a.dst1 = k;
    a.dst2 = v;
    a.B = B;
    a.S_l = S_l;
    a.h_l = h_l;
    a.U = U;
    a.q_batch_stride_rows = q_batch_stride_rows;
    a.kv_batch_stride_rows = kv_batch_stride_rows;
    a.run_vec = static_cast<long long>(h_l) * D / 8;
    a.n_runs = 3LL * U * B * S_l;
    return run_relayout(RelayoutMode::UnpackQKV, a, stream);
}

ctx_status ctx_pack_out(const void *o, void *send, long long o_batch_stride_rows, int B, int S_l, int h_l, int D,
                        int U, ctx_dtype dtype, void *stream)
{
    if (!o || !send || !valid_dtype(dtype))
        return CTX_ERR_INVALID_ARG;
    long long n = 1;
    if (!mul_ok(n, B) || !mul_ok(n, S_l) || !mul_ok(n, h_l) || !mul_ok(n, D) || !mul_ok(n, U))
        return CTX_ERR_INVALID_ARG;
    const long long rows = static_cast<long long>(U) * S_l;
    const long long row_bytes = static_cast<long long>(h_l) * D * 2;
    long long span = o_batch_stride_rows;
    if (o_batch_stride_rows < rows || !mul_ok(span, B) || !mul_ok(span, row_bytes))
        return CTX_ERR_INVALID_ARG;
    if (D % 8 != 0 || !aligned16(o) || !aligned16(send))
        return CTX_ERR_MISALIGNED;
    const long long o_bytes = ((static_cast<long long>(B) - 1) * o_batch_stride_rows + rows) * row_bytes;
    if (overlap(extent(o, o_bytes), extent(send, n * 2)))
        return CTX_ERR_ALIASING;
    ctx_status s = check_device_ptrs({o, send});
    if (s != CTX_OK)
        return s;
    RelayoutArgs a{};
    a.src0 = o;
    a.dst0 = send;
    a.B = B;
    a.S_l = S_l;
    a.h_l = h_l;
    a.U = U;
    a.q_batch_stride_rows = o_batch_stride_rows;
    a.run_vec = static_cast<long long>(h_l) * D / 8;
    a.n_runs = static_cast<long long>(U) * B * S_l;
    return run_relayout(RelayoutMode::PackOut, a, stream);
}

ctx_status ctx_unpack_out(const void *recv, void *y, int B, int S_l, int h_l, int D, int U, ctx_dtype dtype,
                          void *stream)
{
    if (!recv || !y || !valid_dtype(dtype))
        return CTX_ERR_INVALID_ARG;
    long long n = 1;
    if (!mul_ok(n, B) || !mul_ok(n, S_l) || !mul_ok(n, h_l) || !mul_ok(n, D) || !mul_ok(n, U))
        return CTX_ERR_INVALID_ARG;
    if (D % 8 != 0 || !aligned16(recv) || !aligned16(y))
        return CTX_ERR_MISALIGNED;
    if (overlap(extent(recv, n * 2), extent(y, n * 2)))
        return CTX_ERR_ALIASING;
    ctx_status s = check_device_ptrs({recv, y});
    if (s != CTX_OK)
        return s;
    RelayoutArgs a{};
    a.src0 = recv;
    a.dst0 = y;
    a.B = B;
    a.S_l = S_l;
    a.h_l = h_l;
    a.U = U;
    a.run_vec = static_cast<long long>(h_l) * D / 8;
    a.n_runs = static_cast<long long>(U) * B * S_l;
    return run_relayout(RelayoutMode::UnpackOut, a, stream);
}

ctx_status ctx_pack_qkv_ex(const void *q, const void *k, const void *v, void *staging, int B, int S_l, int H, int D,
                           int U, ctx_layout layout, ctx_dtype dtype, void *stream)
{
    if (!q || !k || !v || !staging || !valid_dtype(dtype) ||
        (layout != CTX_LAYOUT_TQKV && layout != CTX_LAYOUT_INTERLEAVED))
        return CTX_ERR_INVALID_ARG;
    long long n = 1;
    if (!mul_ok(n, B) || !mul_ok(n, S_l) || !mul_ok(n, H) || !mul_ok(n, D) || U <= 0)
        return CTX_ERR_INVALID_ARG;
    const long long h_l = (static_cast<long long>(H) + U - 1) / U;
    long long ns = static_cast<long long>(B) * S_l;
    if (!mul_ok(ns, h_l) || !mul_ok(ns, U) || !mul_ok(ns, 3) || !mul_ok(ns, D))
        return CTX_ERR_INVALID_ARG;
    if (D % 8 != 0 || !aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(staging))
        return CTX_ERR_MISALIGNED;
    const Extent st = extent(staging, ns * 2);
    if (overlap(st, extent(q, n * 2)) || overlap(st, extent(k, n * 2)) || overlap(st, extent(v, n * 2)))
        return CTX_ERR_ALIASING;
    ctx_status s = check_device_ptrs({q, k, v, staging});
    if (s != CTX_OK)
        return s;
    RelayoutArgs a{};
    a.src0 = q;
    a.src1 = k;
    a.src2 = v;
    a.dst0 = staging;
    a.B = B;
    a.S_l = S_l;
    a.H = U * h_l;
    a.H_real = H;
    a.U = U;
    a.h_l = h_l;
    if (layout == CTX_LAYOUT_TQKV) {
        a.run_vec = h_l * D / 8;
        a.n_runs = 3LL * U * B * S_l;
        return run_relayout(H % U == 0 ? RelayoutMode::PackQKV : RelayoutMode::PackQKVPad, a, stream);
    }
    a.run_vec = h_l * D / 8;
    a.head_vec = D / 8;
    a.n_runs = 3LL * U * B * S_l;
    return run_relayout(RelayoutMode::PackInter, a, stream);
}

ctx_status ctx_unpack_qkv_ex(const void *recv, void *q, void *k, void *v, long long q_batch_stride_rows,
                             long long kv_batch_stride_rows, int B, int S_l, int h_l, int D, int U, ctx_layout layout,
                             ctx_dtype dtype, void *stream)
{
    if (layout == CTX_LAYOUT_TQKV)
        return ctx_unpack_qkv(recv, q, k, v, q_batch_stride_rows, kv_batch_stride_rows, B, S_l, h_l, D, U, dtype,
                              stream);
    if (layout != CTX_LAYOUT_INTERLEAVED || !recv || !q || !k || !v || !valid_dtype(dtype))
        return CTX_ERR_INVALID_ARG;
    long long n = 1;
    if (!mul_ok(n, B) || !mul_ok(n, S_l) || !mul_ok(n, h_l) || !mul_ok(n, D) || !mul_ok(n, U))
        return CTX_ERR_INVALID_ARG;
    const long long rows = static_cast<long long>(U) * S_l;
    if (q_batch_stride_rows < rows || kv_batch_stride_rows < rows)
        return CTX_ERR_INVALID_ARG;
    const long long row_bytes = static_cast<long long>(h_l) * D * 2;
    long long qspan = q_batch_stride_rows, kvspan = kv_batch_stride_rows;
    if (!mul_ok(qspan, B) || !mul_ok(qspan, row_bytes) || !mul_ok(kvspan, B) || !mul_ok(kvspan, row_bytes))
        return CTX_ERR_INVALID_ARG;
    if (D % 8 != 0 || !aligned16(recv) || !aligned16(q) || !aligned16(k) || !aligned16(v))
        return CTX_ERR_MISALIGNED;
    const long long q_bytes = ((static_cast<long long>(B) - 1) * q_batch_stride_rows + rows) * row_bytes;
    const long long kv_bytes = ((static_cast<long long>(B) - 1) * kv_batch_stride_rows + rows) * row_bytes;
    const Extent r = extent(recv, 3 * n * 2);
    const Extent eq = extent(q, q_bytes), ek = extent(k, kv_bytes), ev = extent(v, kv_bytes);
    if (overlap(r, eq) || overlap(r, ek) || overlap(r, ev) || overlap(eq, ek) || overlap(eq, ev) ||
        overlap(ek, ev))
        return CTX_ERR_ALIASING;
    ctx_status s = check_device_ptrs({recv, q, k, v});
    if (s != CTX_OK)
        return s;
    RelayoutArgs a{};
    a.src0 = recv;
    a.dst0 = q;
    a.dst1 = k;
    a.dst2 = v;
    a.B = B;
    a.S_l = S_l;
    a.h_l = h_l;
    a.U = U;
    a.q_batch_stride_rows = q_batch_stride_rows;
    a.kv_batch_stride_rows = kv_batch_stride_rows;
    a.run_vec = static_cast<long long>(h_l) * D / 8;
    a.head_vec = D / 8;
    a.n_runs = 3LL * U * B * S_l;
    return run_relayout(RelayoutMode::UnpackInter, a, stream);
}

ctx_status ctx_unpack_out_ex(const void *recv, void *y, int B, int S_l, int h_l, int H, int D, int U, ctx_dtype dtype,
                             void *stream)
{
    if (!recv || !y || !valid_dtype(dtype))
        return CTX_ERR_INVALID_ARG;
    long long n = 1;
    if (!mul_ok(n, B) || !mul_ok(n, S_l) || !mul_ok(n, h_l) || !mul_ok(n, D) || !mul_ok(n, U) || H <= 0 ||
        static_cast<long long>(H) > static_cast<long long>(U) * h_l)
        return CTX_ERR_INVALID_ARG;
    if (H == U * h_l)
        return ctx_unpack_out(recv, y, B, S_l, h_l, D, U, dtype, stream);
    if (D % 8 != 0 || !aligned16(recv) || !aligned16(y))
        return CTX_ERR_MISALIGNED;
    const long long y_bytes = static_cast<long long>(B) * S_l * H * D * 2;
    if (overlap(extent(recv, n * 2), extent(y, y_bytes)))
        return CTX_ERR_ALIASING;
    ctx_status s = check_device_ptrs({recv, y});
    if (s != CTX_OK)
        return s;
    RelayoutArgs a{};
    a.src0 = recv;
    a.dst0 = y;
    a.B = B;
    a.S_l = S_l;
    a.h_l = h_l;
    a.H_real = H;
    a.U = U;
    a.run_vec = static_cast<long long>(h_l) * D / 8;
    a.n_runs = static_cast<long long>(U) * B * S_l;
    return run_relayout(RelayoutMode::UnpackOutPad, a, stream);
}

static ctx_status attn_common(const void *q, const void *k, const void *v, const unsigned char *key_mask,
                              float scale, void *out, float *lse, void *workspace, long long workspace_bytes, int B,
                              int Sq, int Sk, int H, int D, ctx_dtype dtype, void *stream, int blk_s, int blk_u,
                              int blk_b)
{
    if (!q || !k || !v || !out || !valid_dtype(dtype))
        return CTX_ERR_INVALID_ARG;
    long long nq = 1, nk = 1;
    if (!mul_ok(nq, B) || !mul_ok(nq, Sq) || !mul_ok(nq, H) || !mul_ok(nq, D))
        return CTX_ERR_INVALID_ARG;
    if (!mul_ok(nk, B) || !mul_ok(nk, Sk) || !mul_ok(nk, H) || !mul_ok(nk, D))
        return CTX_ERR_INVALID_ARG;
    if (ctx::attention_units(B, Sq, H) > 0x7fffffffLL)
        return CTX_ERR_INVALID_ARG;
    if (std::isnan(scale))
        scale = 1.0f / std::sqrt(static_cast<float>(D));
    if (!std::isfinite(scale) || !(scale > 0.f))
        return CTX_ERR_INVALID_ARG;
    if (workspace && workspace_bytes <= 0)
        return CTX_ERR_INVALID_ARG;
    if (D % 8 != 0 || !aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) ||
        (reinterpret_cast<uintptr_t>(lse) & 3u) != 0 || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
        return CTX_ERR_MISALIGNED;
    if (D != 64 && D != 128)
        return CTX_ERR_UNSUPPORTED;
    const Extent eo = extent(out, nq * 2);
    const Extent eq = extent(q, nq * 2), ek = extent(k, nk * 2), ev = extent(v, nk * 2);
    const Extent em = key_mask ? extent(key_mask, static_cast<long long>(B) * Sk) : Extent{0, 0};
    const Extent el = lse ? extent(lse, static_cast<long long>(B) * H * Sq * 4) : Extent{0, 0};
    const Extent ew = workspace ? extent(workspace, workspace_bytes) : Extent{0, 0};
    if (overlap(eo, eq) || overlap(eo, ek) || overlap(eo, ev) || overlap(eo, em))
        return CTX_ERR_ALIASING;
    if (overlap(el, eo) || overlap(el, eq) || overlap(el, ek) || overlap(el, ev) || overlap(el, em))
        return CTX_ERR_ALIASING;
    if (overlap(ew, eo) || overlap(ew, eq) || overlap(ew, ek) || overlap(ew, ev) || overlap(ew, em) ||
        overlap(ew, el))
        return CTX_ERR_ALIASING;
    ctx_status s = check_device_ptrs({q, k, v, out, lse, key_mask, workspace});
    if (s != CTX_OK)
        return s;
    if (workspace) {
        cudaError_t e = cudaSuccess;
        const long long need = ctx::attention_workspace_size(B, Sq, Sk, H, D, &e);
        if (e != cudaSuccess)
            return cuda_fail(e);
        if (workspace_bytes < need)
            return CTX_ERR_INVALID_ARG;
    }
    ctx::AttnArgs a{};
    a.q = q;
    a.k = k;
    a.v = v;
    a.mask = key_mask;
    a.out = out;
    a.lse = lse;
    a.B = B;
    a.Sq = Sq;
    a.Sk = Sk;
    a.H = H;
    a.D = D;
    a.bf16 = dtype == CTX_BF16;
    a.scale = scale;
    a.workspace = workspace;
    a.workspace_bytes = workspace_bytes;
    a.blk_s = blk_s;
    a.blk_u = blk_u;
    a.blk_b = blk_b;
    cudaError_t e = ctx::launch_attention(a, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? CTX_OK : cuda_fail(e);
}

ctx_status ctx_attn_lq_gkv(const void *q, const void *k, const void *v, const unsigned char *key_mask, float scale,
                           void *out, float *lse, void *workspace, long long workspace_bytes, int B, int Sq, int Sk,
                           int H, int D, ctx_dtype dtype, void *stream)
{
    return attn_common(q, k, v, key_mask, scale, out, lse, workspace, workspace_bytes, B, Sq, Sk, H, D, dtype, stream,
                       0, 0, 0);
}

ctx_status ctx_attn_lq_gkv_pack_out(const void *q, const void *k, const void *v, const unsigned char *key_mask,
                                    float scale, void *send, float *lse, void *workspace, long long workspace_bytes,
                                    int B, int Sq, int Sk, int H, int D, int U, int B_rank, int S_l, ctx_dtype dtype,
                                    void *stream)
{
    // the send layout must cover the output exactly: Sq = A*U*S_l rows, B = U'*B_rank with U' <= U
    if (U <= 0 || B_rank <= 0 || S_l <= 0 || Sq <= 0 || B <= 0 || Sq % (static_cast<long long>(U) * S_l) != 0 ||
        B % B_rank != 0 || B / B_rank > U)
        return CTX_ERR_INVALID_ARG;
    return attn_common(q, k, v, key_mask, scale, send, lse, workspace, workspace_bytes, B, Sq, Sk, H, D, dtype,
                       stream, S_l, U, B_rank);
}

long long ctx_attn_lq_gkv_workspace_size(int B, int Sq, int Sk, int H, int D)
{
    long long n = 1;
    if (!mul_ok(n, B) || !mul_ok(n, Sq) || !mul_ok(n, Sk) || !mul_ok(n, H) || (D != 64 && D != 128) ||
        ctx::attention_units(B, Sq, H) > 0x7fffffffLL)
        return -1;
    cudaError_t e = cudaSuccess;
    const long long bytes = ctx::attention_workspace_size(B, Sq, Sk, H, D, &e);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return -1;
    }
    return bytes;
}

ctx_status ctx_varlen_remap(const int *cu_seqlens_q, int n_docs, long long span_begin, long long span_len,
                            int *cu_seqlens_q_local, const int *packed_padding, int *packed_padding_local,
                            void *stream)
{
    if (!cu_seqlens_q || !cu_seqlens_q_local || n_docs <= 0 || span_begin < 0 || span_len < 0 ||
        span_begin + span_len > 0x7fffffffLL || ((packed_padding == nullptr) != (packed_padding_local == nullptr)))
        return CTX_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(cu_seqlens_q) & 3u) || (reinterpret_cast<uintptr_t>(cu_seqlens_q_local) & 3u) ||
        (reinterpret_cast<uintptr_t>(packed_padding) & 3u) || (reinterpret_cast<uintptr_t>(packed_padding_local) & 3u))
        return CTX_ERR_MISALIGNED;
    const long long cu_bytes = (static_cast<long long>(n_docs) + 1) * 4;
    const Extent eg = extent(cu_seqlens_q, cu_bytes), el = extent(cu_seqlens_q_local, cu_bytes);
    const Extent pi = packed_padding ? extent(packed_padding, 8) : Extent{0, 0};
    const Extent po = packed_padding_local ? extent(packed_padding_local, 8) : Extent{0, 0};
    if (overlap(eg, el) || overlap(po, eg) || overlap(po, el) || overlap(po, pi) || overlap(el, pi))
        return CTX_ERR_ALIASING;
    ctx_status s = check_device_ptrs({cu_seqlens_q, cu_seqlens_q_local, packed_padding, packed_padding_local});
    if (s != CTX_OK)
        return s;
    cudaError_t e = ctx::launch_varlen_remap(cu_seqlens_q, n_docs, span_begin, span_len, cu_seqlens_q_local,
                                             packed_padding, packed_padding_local, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? CTX_OK : cuda_fail(e);
}

ctx_status ctx_attn_varlen(const void *q, const void *k, const void *v, const int *cu_seqlens_q,
                           const int *cu_seqlens_k, int n_docs, int max_seqlen_q, const unsigned char *key_mask,
                           float scale, void *out, float *lse, void *workspace, long long workspace_bytes, int Sq,
                           int Sk, int H, int D, ctx_dtype dtype, void *stream)
{
    if (!q || !k || !v || !out || !cu_seqlens_q || !cu_seqlens_k || !valid_dtype(dtype) || n_docs <= 0 ||
        max_seqlen_q <= 0)
        return CTX_ERR_INVALID_ARG;
    long long nq = 1, nk = 1;
    if (!mul_ok(nq, Sq) || !mul_ok(nq, H) || !mul_ok(nq, D) || !mul_ok(nk, Sk) || !mul_ok(nk, H) || !mul_ok(nk, D))
        return CTX_ERR_INVALID_ARG;
    long long units = (static_cast<long long>(max_seqlen_q) + 255) / 256;
    if (!mul_ok(units, H) || !mul_ok(units, n_docs) || units > 0x7fffffffLL)
        return CTX_ERR_INVALID_ARG;
    if (std::isnan(scale))
        scale = 1.0f / std::sqrt(static_cast<float>(D));
    if (!std::isfinite(scale) || !(scale > 0.f))
        return CTX_ERR_INVALID_ARG;
    if (workspace && workspace_bytes <= 0)
        return CTX_ERR_INVALID_ARG;
    if (D % 8 != 0 || !aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) ||
        (reinterpret_cast<uintptr_t>(lse) & 3u) || (reinterpret_cast<uintptr_t>(cu_seqlens_q) & 3u) ||
        (reinterpret_cast<uintptr_t>(cu_seqlens_k) & 3u) || (reinterpret_cast<uintptr_t>(workspace) & 255u))
        return CTX_ERR_MISALIGNED;
    if (D != 64 && D != 128)
        return CTX_ERR_UNSUPPORTED;
    const Extent eo = extent(out, nq * 2);
    const Extent el = lse ? extent(lse, static_cast<long long>(H) * Sq * 4) : Extent{0, 0};
    const Extent ew = workspace ? extent(workspace, workspace_bytes) : Extent{0, 0};
    const Extent ins[] = {extent(q, nq * 2), extent(k, nk * 2), extent(v, nk * 2),
                          key_mask ? extent(key_mask, Sk) : Extent{0, 0},
                          extent(cu_seqlens_q, (static_cast<long long>(n_docs) + 1) * 4),
                          extent(cu_seqlens_k, (static_cast<long long>(n_docs) + 1) * 4)};
    for (const Extent &x : ins)
        if (overlap(eo, x) || overlap(el, x) || overlap(ew, x))
            return CTX_ERR_ALIASING;
    if (overlap(eo, el) || overlap(ew, eo) || overlap(ew, el))
        return CTX_ERR_ALIASING;
    ctx_status s = check_device_ptrs({q, k, v, out, lse, key_mask, cu_seqlens_q, cu_seqlens_k, workspace});
    if (s != CTX_OK)
        return s;
    if (workspace) {
        cudaError_t e = cudaSuccess;
        const long long need = ctx::varlen_workspace_size(n_docs, max_seqlen_q, H, D, &e);
        if (e != cudaSuccess)
            return cuda_fail(e);
        if (workspace_bytes < need)
            return CTX_ERR_INVALID_ARG;
    }
    ctx::AttnArgs a{};
    a.q = q;
    a.k = k;
    a.v = v;
    a.mask = key_mask;
    a.out = out;
    a.lse = lse;
    a.B = 1;
    a.Sq = Sq;
    a.Sk = Sk;
    a.H = H;
    a.D = D;
    a.bf16 = dtype == CTX_BF16;
    a.scale = scale;
    a.cu_q = cu_seqlens_q;
    a.cu_k = cu_seqlens_k;
    a.n_docs = n_docs;
    a.max_seqlen_q = max_seqlen_q;
    a.workspace = workspace;
    a.workspace_bytes = workspace_bytes;
    cudaError_t e = ctx::launch_attention(a, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? CTX_OK : cuda_fail(e);
}

long long ctx_attn_varlen_workspace_size(int n_docs, int max_seqlen_q, int H, int D)
{
    long long units = (static_cast<long long>(max_seqlen_q) + 255) / 256;
    if (n_docs <= 0 || max_seqlen_q <= 0 || !mul_ok(units, H) || !mul_ok(units, n_docs) ||
        units > 0x7fffffffLL || (D != 64 && D != 128))
        return -1;
    cudaError_t e = cudaSuccess;
    const long long bytes = ctx::varlen_workspace_size(n_docs, max_seqlen_q, H, D, &e);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return -1;
    }
    return bytes;
}

ctx_status ctx_merge_joint_attn_mask(const unsigned char *image_mask, int image_ndim, const long long *image_dims,
                                     const unsigned char *joint_mask, int joint_ndim, const long long *joint_dims,
                                     int B, int S_img, int J, int joint_front, unsigned char *key_mask, void *stream)
{
    if (!key_mask || B <= 0 || S_img < 0 || J < 0 || static_cast<long long>(S_img) + J <= 0 ||
        static_cast<long long>(S_img) + J > 0x7fffffffLL)
        return CTX_ERR_INVALID_ARG;
    // ranks, joint side first: a joint mask is only ever 2-D; a 4-D image
    // mask has no key-mask form (refused with or without a joint mask)
    if (joint_mask && (joint_ndim != 2 || !joint_dims))
        return CTX_ERR_INVALID_ARG;
    if (image_mask && !image_dims)
        return CTX_ERR_INVALID_ARG;
    if (image_mask && image_ndim == 4)
        return CTX_ERR_UNSUPPORTED;
    if (image_mask && image_ndim != 2)
        return CTX_ERR_INVALID_ARG;
    // a joint mask needs joint keys; each side must cover (B, its segment)
    if (joint_mask && J == 0)
        return CTX_ERR_INVALID_ARG;
    if (image_mask && (image_dims[0] != B || image_dims[1] != S_img))
        return CTX_ERR_INVALID_ARG;
    if (joint_mask && (joint_dims[0] != B || joint_dims[1] != J))
        return CTX_ERR_INVALID_ARG;
    const long long out_bytes = static_cast<long long>(B) * (static_cast<long long>(S_img) + J);
    const Extent eo = extent(key_mask, out_bytes);
    if ((image_mask && overlap(eo, extent(image_mask, static_cast<long long>(B) * S_img))) ||
        (joint_mask && overlap(eo, extent(joint_mask, static_cast<long long>(B) * J))))
        return CTX_ERR_ALIASING;
    ctx_status s = check_device_ptrs({image_mask, joint_mask, key_mask});
    if (s != CTX_OK)
        return s;
    cudaError_t e = ctx::launch_merge_mask(image_mask, joint_mask, B, S_img, J, joint_front ? 1 : 0, key_mask,
                                           static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? CTX_OK : cuda_fail(e);
}

ctx_status ctx_lse_merge(const void *o_parts, const float *lse_parts, int P, void *out, float *lse, int B, int Sq,
                         int H, int D, ctx_dtype dtype, void *stream)
{
    if (!o_parts || !lse_parts || !out || !valid_dtype(dtype))
        return CTX_ERR_INVALID_ARG;
    long long rows = 1;
    if (P <= 0 || !mul_ok(rows, B) || !mul_ok(rows, Sq) || !mul_ok(rows, H) || D <= 0)
        return CTX_ERR_INVALID_ARG;
    long long parts = rows;
    if (!mul_ok(parts, P) || !mul_ok(parts, D))
        return CTX_ERR_INVALID_ARG;
    if (D % 8 != 0 || !aligned16(o_parts) || !aligned16(out) || (reinterpret_cast<uintptr_t>(lse_parts) & 3u) ||
        (reinterpret_cast<uintptr_t>(lse) & 3u))
        return CTX_ERR_MISALIGNED;
    const Extent eo = extent(out, rows * D * 2), eop = extent(o_parts, parts * 2);
    const Extent elp = extent(lse_parts, rows * P * 4);
    const Extent el = lse ? extent(lse, rows * 4) : Extent{0, 0};
    if (overlap(eo, eop) || overlap(eo, elp) || overlap(el, eop) || overlap(el, elp) || overlap(el, eo))
        return CTX_ERR_ALIASING;
    ctx_status s = check_device_ptrs({o_parts, lse_parts, out, lse});
    if (s != CTX_OK)
        return s;
    ctx::LseMergeArgs a{};
    a.o_parts = o_parts;
    a.lse_parts = lse_parts;
    a.P = P;
    a.out = out;
    a.lse = lse;
    a.B = B;
    a.Sq = Sq;
    a.H = H;
    a.D = D;
    a.bf16 = dtype == CTX_BF16;
    cudaError_t e = ctx::launch_lse_merge(a, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? CTX_OK : cuda_fail(e);
}

ctx_status ctx_device_status(void *stream)
{
    cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess)
        return cuda_fail(e);
    int *word = ctx::device_status_word(static_cast<cudaStream_t>(stream), &e);
    if (e != cudaSuccess)
        return cuda_fail(e);
    int value = 0;
    e = cudaMemcpy(&value, word, sizeof(int), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess)
        return cuda_fail(e);
    if (value != 0) {
        const int zero = 0;
        e = cudaMemcpy(word, &zero, sizeof(int), cudaMemcpyHostToDevice);
        if (e != cudaSuccess)
            return cuda_fail(e);
    }
    return value == 0 ? CTX_OK : static_cast<ctx_status>(value);
}

ctx_status ctx_selftest_wait_timeout(long long limit_ns, void *stream)
{
    if (limit_ns < 1000 || limit_ns > 5000000000LL)
        return CTX_ERR_INVALID_ARG;
    cudaError_t e = ctx::launch_selftest_wait(static_cast<unsigned long long>(limit_ns),
                                              static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess)
        return cuda_fail(e);
    return ctx_device_status(stream);
}

}  // extern "C"
