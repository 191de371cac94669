// Log-sum-exp merge of attention results computed over disjoint key
// segments (the "merge" interface that consumes an LSE, ChituDiffusion Fast CP
// page; ring or segmented K/V): for every row (b, i, h)
//   lse = ln sum_p exp(lse_p),   out = sum_p exp(lse_p - lse) * o_p.
// HBM bound: a lane owns one 16-byte chunk (8 elements) of an output row,
// accumulates the P matching chunks in fp32 with weights from the row's P
// segment LSEs, and writes one rounded chunk. The weights take one
// exponential per segment: with m = max_p lse_p, e_p = exp(lse_p - m),
// l = sum_p e_p, the weight is e_p / l and lse = m + ln l (exp and log by
// the special-function unit's base-2 instructions).
#include <algorithm>
#include <cmath>
#include <cuda_fp16.h>
#include <mutex>

#include "internal.h"
#include "ptx.cuh"

namespace ctx {
namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.693147180559945309f;

template <bool BF16>
__device__ __forceinline__ void widen8(const uint4 &v, float *f)
{
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        if constexpr (BF16) {
            f[2 * i] = __uint_as_float(w[i] << 16);
            f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
        } else {
            f[2 * i] = __half2float(__ushort_as_half(static_cast<unsigned short>(w[i] & 0xffffu)));
            f[2 * i + 1] = __half2float(__ushort_as_half(static_cast<unsigned short>(w[i] >> 16)));
        }
    }
}

// DV = D/8 lanes own one row (a "lane group"); a warp holds 32/DV groups and
// every group merges kUnr rows per iteration. All PT segment LSEs and all PT
// 16-byte chunks of those rows are loaded before any of them is used, so a
// lane keeps PT*kUnr loads in flight and an iteration waits for one DRAM
// round trip. Row indices are decomposed once per row, in 32-bit arithmetic
// when every row index fits (I32); with 64 registers a thread, four blocks
// stay resident on an SM (three for four segments).
__host__ __device__ constexpr int merge_unroll(int pt) { return pt <= 2 ? 4 : 2; }
__host__ __device__ constexpr int merge_min_blocks(int pt) { return pt <= 3 ? 4 : 3; }

template <bool BF16, int DV, int PT, bool I32>
__global__ void __launch_bounds__(256, merge_min_blocks(PT)) lse_merge_kernel(const uint4 *__restrict__ o_parts,
                                                        const float *__restrict__ lse_parts, uint4 *out,
                                                        float *lse_out, long long rows, int Sq, int H)
{
    constexpr int kGroups = 32 / DV;
    constexpr int kUnr = merge_unroll(PT);
    const int lane = threadIdx.x & 31;
    const int grp = lane / DV, c = lane % DV;
    const long long warp = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const long long n_warps = (static_cast<long long>(gridDim.x) * blockDim.x) >> 5;
    for (long long r0 = warp * kGroups * kUnr; r0 < rows; r0 += n_warps * kGroups * kUnr) {
        long long r[kUnr], lrow[kUnr];
        float lv[kUnr][PT];
        uint4 ov[kUnr][PT];
#pragma unroll
        for (int u = 0; u < kUnr; ++u) {
            // rows are walked in output order r = (b*Sq + i)*H + h of [B, Sq, H, D], so a
            // warp's rows are one contiguous stretch of every part (the bulk of the bytes);
            // the LSE of a row sits at lrow = (b*H + h)*Sq + i of [B, H, Sq] (small, L2-resident)
            const long long l0 = r0 + static_cast<long long>(u) * kGroups + grp;
            const long long rr = l0 < rows ? l0 : rows - 1;  // clamp: loads stay in bounds
            if constexpr (I32) {
                const unsigned r32 = static_cast<unsigned>(rr), hu = static_cast<unsigned>(H);
                const unsigned bi = r32 / hu, h = r32 - bi * hu;
                const unsigned b = bi / static_cast<unsigned>(Sq), i = bi - b * static_cast<unsigned>(Sq);
                lrow[u] = static_cast<long long>((b * hu + h) * static_cast<unsigned>(Sq) + i);
            } else {
                const long long bi = rr / H, h = rr - bi * H;
                const long long b = bi / Sq, i = bi - b * Sq;
                lrow[u] = (b * H + h) * Sq + i;
            }
            r[u] = l0 < rows ? rr : rows;
#pragma unroll
            for (int p = 0; p < PT; ++p) {
                lv[u][p] = __ldg(lse_parts + p * rows + lrow[u]);
                ov[u][p] = __ldg(o_parts + (p * rows + rr) * DV + c);
            }
        }
#pragma unroll
        for (int u = 0; u < kUnr; ++u) {
            float m = lv[u][0];
#pragma unroll
            for (int p = 1; p < PT; ++p)
                m = fmaxf(m, lv[u][p]);
            float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
            float total = -INFINITY;
            if (m != -INFINITY) {
                // e_p = 2^((lse_p - m) log2 e): 0 for an empty segment (lse_p = -inf), 1 for the largest
                float e[PT], l = 0.f;
#pragma unroll
                for (int p = 0; p < PT; ++p) {
                    e[p] = ptx::ex2_approx((lv[u][p] - m) * kLog2e);
                    l += e[p];
                }
                const float inv = __frcp_rn(l);  // l >= 1
                total = m + kLn2 * ptx::lg2_approx(l);
#pragma unroll
                for (int p = 0; p < PT; ++p) {
                    const float w = e[p] * inv;
                    float f[8];
                    widen8<BF16>(ov[u][p], f);
#pragma unroll
                    for (int k = 0; k < 8; ++k)
                        acc[k] = fmaf(w, f[k], acc[k]);
                }
            }
            if (r[u] < rows) {
                out[r[u] * DV + c] = make_uint4(ptx::pack2<BF16>(acc[0], acc[1]), ptx::pack2<BF16>(acc[2], acc[3]),
                                                ptx::pack2<BF16>(acc[4], acc[5]), ptx::pack2<BF16>(acc[6], acc[7]));
                if (lse_out && c == 0)
                    lse_out[lrow[u]] = total;
            }
        }
    }
}

// Any D that is a multiple of 8: one thread per 16-byte chunk (same weights).
template <bool BF16>
__global__ void __launch_bounds__(256) lse_merge_generic(const uint4 *__restrict__ o_parts,
                                                         const float *__restrict__ lse_parts, int P, uint4 *out,
                                                         float *lse_out, long long rows, int Sq, int H, int dv)
{
    const long long n = rows * dv;
    for (long long t = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; t < n;
         t += static_cast<long long>(gridDim.x) * blockDim.x) {
        const long long r = t / dv;
        const int c = static_cast<int>(t - r * dv);
        const long long bi = r / H;
        const int h = static_cast<int>(r - bi * H);
        const long long b = bi / Sq, i = bi - b * Sq;
        const long long lrow = (b * H + h) * Sq + i;
        float m = -INFINITY;
        for (int p = 0; p < P; ++p)
            m = fmaxf(m, __ldg(lse_parts + p * rows + lrow));
        float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        float total = -INFINITY;
        if (m != -INFINITY) {
            float l = 0.f;
            for (int p = 0; p < P; ++p)
                l += ptx::ex2_approx((__ldg(lse_parts + p * rows + lrow) - m) * kLog2e);
            const float inv = __frcp_rn(l);
            total = m + kLn2 * ptx::lg2_approx(l);
            for (int p = 0; p < P; ++p) {
                const float lp = __ldg(lse_parts + p * rows + lrow);
                if (lp == -INFINITY)
                    continue;
                const float w = ptx::ex2_approx((lp - m) * kLog2e) * inv;
                float f[8];
                widen8<BF16>(__ldg(o_parts + (p * rows + r) * dv + c), f);
#pragma unroll
                for (int k = 0; k < 8; ++k)
                    acc[k] = fmaf(w, f[k], acc[k]);
            }
        }
        out[r * dv + c] = make_uint4(ptx::pack2<BF16>(acc[0], acc[1]), ptx::pack2<BF16>(acc[2], acc[3]),
                                     ptx::pack2<BF16>(acc[4], acc[5]), ptx::pack2<BF16>(acc[6], acc[7]));
        if (lse_out && c == 0)
            lse_out[lrow] = total;
    }
}

// Blocks of `kernel` (256 threads) that fit on one SM at once, cached per
// kernel and device: the grid is sized to what is resident together, so the
// grid-stride loop shares the rows evenly instead of running a partial last
// wave of blocks.
template <typename K>
int resident_blocks(K kernel, int dev)
{
    static int cache[64] = {0};
    static std::mutex mu;
    std::lock_guard<std::mutex> g(mu);
    if (dev >= 0 && dev < 64 && cache[dev] > 0)
        return cache[dev];
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, 256, 0) != cudaSuccess || n < 1)
        n = 1;
    if (dev >= 0 && dev < 64)
        cache[dev] = n;
    return n;
}

template <bool BF16>
cudaError_t launch_typed_merge(const LseMergeArgs &a, int sms, cudaStream_t stream)
{
    int dev = 0;
    cudaError_t derr = cudaGetDevice(&dev);
    if (derr != cudaSuccess)
        return derr;
    const long long rows = static_cast<long long>(a.B) * a.Sq * a.H;
    const int dv = a.D / 8;
    const uint4 *op = static_cast<const uint4 *>(a.o_parts);
    uint4 *out = static_cast<uint4 *>(a.out);
    auto grid_for = [&](long long rows_per_block, int per_sm) {
        const long long cap = static_cast<long long>(sms) * per_sm;
        return static_cast<unsigned>(std::max(1LL, std::min(cap, (rows + rows_per_block - 1) / rows_per_block)));
    };
    bool done = false;
    const bool i32 = rows <= 0x7fffffffLL;  // every row index, and (b*H + h)*Sq + i, fits in 32 bits
#define CTX_MERGE_CASE_I(DVV, PP, I)                                                                         \
    if (!done && dv == DVV && a.P == PP && i32 == I) {                                                      \
        lse_merge_kernel<BF16, DVV, PP, I><<<grid_for(8LL * (32 / DVV) * merge_unroll(PP),                   \
                                                       resident_blocks(lse_merge_kernel<BF16, DVV, PP, I>, dev)), \
                                             256, 0, stream>>>(                                               \
            op, a.lse_parts, out, a.lse, rows, a.Sq, a.H);                                                   \
        done = true;                                                                                         \
    }
#define CTX_MERGE_CASE(DVV, PP) CTX_MERGE_CASE_I(DVV, PP, true) CTX_MERGE_CASE_I(DVV, PP, false)
#define CTX_MERGE_DV(DVV) CTX_MERGE_CASE(DVV, 1) CTX_MERGE_CASE(DVV, 2) CTX_MERGE_CASE(DVV, 3) CTX_MERGE_CASE(DVV, 4)
    CTX_MERGE_DV(8)
    CTX_MERGE_DV(16)
#undef CTX_MERGE_DV
#undef CTX_MERGE_CASE
#undef CTX_MERGE_CASE_I
    if (!done)
        lse_merge_generic<BF16><<<grid_for(256 / std::max(1, dv), resident_blocks(lse_merge_generic<BF16>, dev)),
                                  256, 0, stream>>>(op, a.lse_parts, a.P, out,
                                                                                     a.lse, rows, a.Sq, a.H, dv);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_lse_merge(const LseMergeArgs &a, cudaStream_t stream)
{
    cudaError_t err = cudaSuccess;
    const int sms = sm_count(&err);
    if (err != cudaSuccess)
        return err;
    return a.bf16 ? launch_typed_merge<true>(a, sms, stream) : launch_typed_merge<false>(a, sms, stream);
}

}  // namespace ctx
