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
// every group merges kUnr rows per pass. All PT 16-byte chunks of those rows
// are loaded before any of them is used, so a lane keeps PT*kUnr loads in
// flight and a pass waits for one DRAM round trip. The pass's rows' weights
// are computed once per row by one lane each (its LSE loads, the row index
// decomposed in 32-bit arithmetic when every index fits, I32) and handed to
// the row's lanes by shuffle; the weighted sum runs as packed fp32 pairs.
// With 64 registers a thread, four blocks stay resident on an SM (three for
// four segments).
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
    constexpr int kRows = kGroups * kUnr;  // rows of one pass of the warp
    static_assert(kRows <= 32, "one lane per row computes the weights");
    for (long long r0 = warp * kRows; r0 < rows; r0 += n_warps * kRows) {
        // rows are walked in output order r = (b*Sq + i)*H + h of [B, Sq, H, D], so a
        // warp's rows are one contiguous stretch of every part (the bulk of the bytes)
        uint4 ov[kUnr][PT];
#pragma unroll
        for (int u = 0; u < kUnr; ++u) {
            const long long l0 = r0 + static_cast<long long>(u) * kGroups + grp;
            const long long rr = l0 < rows ? l0 : rows - 1;  // clamp: loads stay in bounds
#pragma unroll
            for (int p = 0; p < PT; ++p)
                ov[u][p] = __ldg(o_parts + (p * rows + rr) * DV + c);
        }
        // The weights of the pass's rows, once per row: lane j < kRows takes row
        // r0 + j (pass order u*kGroups + grp), whose LSE sits at
        // lrow = (b*H + h)*Sq + i of [B, H, Sq] (small, L2-resident). With
        // m = max_p lse_p, e_p = 2^((lse_p - m) log2 e) (0 for an empty segment,
        // 1 for the largest), l = sum_p e_p: w_p = e_p / l, lse = m + ln l.
        float w[PT];
#pragma unroll
        for (int p = 0; p < PT; ++p)
            w[p] = 0.f;
        if (lane < kRows) {
            const long long l0 = r0 + lane;
            const long long rr = l0 < rows ? l0 : rows - 1;
            long long lrow;
            if constexpr (I32) {
                const unsigned r32 = static_cast<unsigned>(rr), hu = static_cast<unsigned>(H);
                const unsigned bi = r32 / hu, h = r32 - bi * hu;
                const unsigned b = bi / static_cast<unsigned>(Sq), i = bi - b * static_cast<unsigned>(Sq);
                lrow = static_cast<long long>((b * hu + h) * static_cast<unsigned>(Sq) + i);
            } else {
                const long long bi = rr / H, h = rr - bi * H;
                const long long b = bi / Sq, i = bi - b * Sq;
                lrow = (b * H + h) * Sq + i;
            }
            float lv[PT];
#pragma unroll
            for (int p = 0; p < PT; ++p)
                lv[p] = __ldg(lse_parts + p * rows + lrow);
            float m = lv[0];
#pragma unroll
            for (int p = 1; p < PT; ++p)
                m = fmaxf(m, lv[p]);
            float total = -INFINITY;
            if (m != -INFINITY) {
                float e[PT], l = 0.f;
#pragma unroll
                for (int p = 0; p < PT; ++p) {
                    e[p] = ptx::ex2_approx((lv[p] - m) * kLog2e);
                    l += e[p];
                }
                const float inv = __frcp_rn(l);  // l >= 1
                total = m + kLn2 * ptx::lg2_approx(l);
#pragma unroll
                for (int p = 0; p < PT; ++p)
                    w[p] = e[p] * inv;
            }
            if (lse_out && l0 < rows)
                lse_out[lrow] = total;
        }
#pragma unroll
        for (int u = 0; u < kUnr; ++u) {
            const int src = u * kGroups + grp;  // the lane that holds this row's weights
            uint64_t acc[4] = {0, 0, 0, 0};     // (fp32, fp32) pairs of the lane's 8 columns
#pragma unroll
            for (int p = 0; p < PT; ++p) {
                const float wp = __shfl_sync(0xffffffffu, w[p], src);
                const uint64_t w2 = ptx::f2_pack(wp, wp);
                float f[8];
                widen8<BF16>(ov[u][p], f);
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    acc[k] = ptx::f2_fma(w2, ptx::f2_pack(f[2 * k], f[2 * k + 1]), acc[k]);
            }
            const long long l0 = r0 + static_cast<long long>(u) * kGroups + grp;
            if (l0 < rows)
                out[l0 * DV + c] =
                    make_uint4(ptx::pack2<BF16>(ptx::f2_lo(acc[0]), ptx::f2_hi(acc[0])),
                               ptx::pack2<BF16>(ptx::f2_lo(acc[1]), ptx::f2_hi(acc[1])),
                               ptx::pack2<BF16>(ptx::f2_lo(acc[2]), ptx::f2_hi(acc[2])),
                               ptx::pack2<BF16>(ptx::f2_lo(acc[3]), ptx::f2_hi(acc[3])));
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

// One block per 256 threads' share of the rows: every warp makes one pass
// (the grid-stride loops only matter beyond 2^31 - 1 blocks). Measured
// against a grid of the blocks resident at once, each looping over ten
// passes: 2 segments of the 480p output 6059 -> 6320 GB/s, 4 segments
// 6053 -> 6695, 2 segments of a Wan-14B-like rank 6276 -> 6746; the block
// scheduler fills an SM's slots as blocks finish, so no warp waits on a
// slow one of its block and the tail is a fraction of a pass.
template <bool BF16>
cudaError_t launch_typed_merge(const LseMergeArgs &a, cudaStream_t stream)
{
    const long long rows = static_cast<long long>(a.B) * a.Sq * a.H;
    const int dv = a.D / 8;
    const uint4 *op = static_cast<const uint4 *>(a.o_parts);
    uint4 *out = static_cast<uint4 *>(a.out);
    auto grid_for = [&](long long units, long long units_per_block) {
        const long long blocks = (units + units_per_block - 1) / units_per_block;
        return static_cast<unsigned>(std::max(1LL, std::min(0x7fffffffLL, blocks)));
    };
    bool done = false;
    const bool i32 = rows <= 0x7fffffffLL;  // every row index, and (b*H + h)*Sq + i, fits in 32 bits
#define CTX_MERGE_CASE_I(DVV, PP, I)                                                                         \
    if (!done && dv == DVV && a.P == PP && i32 == I) {                                                      \
        lse_merge_kernel<BF16, DVV, PP, I><<<grid_for(rows, 8LL * (32 / DVV) * merge_unroll(PP)), 256, 0,    \
                                             stream>>>(                                                       \
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
        lse_merge_generic<BF16><<<grid_for(rows * dv, 256), 256, 0, stream>>>(op, a.lse_parts, a.P, out, a.lse, rows,
                                                                               a.Sq, a.H, dv);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_lse_merge(const LseMergeArgs &a, cudaStream_t stream)
{
    return a.bf16 ? launch_typed_merge<true>(a, stream) : launch_typed_merge<false>(a, stream);
}

}  // namespace ctx
