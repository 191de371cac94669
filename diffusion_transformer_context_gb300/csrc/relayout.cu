// Ulysses layout steps: pack / unpack of Q,K,V, the reverse output exchange,
// and the simulated all_to_all_single between ranks on one GPU.
//
// All of them are permutations of "runs": h_l*D contiguous elements (one
// destination rank's heads of one row) that stay contiguous on both sides
// (sglang PR #33667, pack_qkv_destination_major: destination r gets heads
// [r*H/U, (r+1)*H/U) of every row). In the interleaved staging layout a run
// stays contiguous on the Q/K/V side and is cut into its heads on the staging
// side, where each head's D elements sit in a cell of 3*D (Q | K | V). The
// kernel is HBM bound: a warp moves one run (or one segment of a long run)
// with 16-byte vector loads that bypass L1 and 16-byte stores, each lane
// keeping up to 8 loads in flight before it stores, and the grid holds one
// warp per run or segment.
#include <algorithm>

#include "internal.h"

namespace ctx {
namespace {

__device__ __forceinline__ uint4 ld_stream(const uint4 *p)
{
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

// Source and destination of run `run` (in 16-byte vectors). rv = run length;
// a row of H heads is U runs long (H*D/8 = U*rv). `valid` is the number of
// vectors of the run that exist in the source (padded modes): the pack
// zero-fills the rest, the padded reverse exchange skips it. I is the type
// the run index is decomposed in: unsigned 32-bit whenever every run index
// fits (a 64-bit division is a long software sequence and a run takes up to
// five of them), else 64-bit; offsets are formed in 64-bit either way.
template <RelayoutMode M, typename I>
__device__ __forceinline__ void map_run(const RelayoutArgs &a, I run, const uint4 *&src, uint4 *&dst,
                                        long long &valid)
{
    const long long rv = a.run_vec;
    const I S_l = static_cast<I>(a.S_l), B = static_cast<I>(a.B), U = static_cast<I>(a.U);
    valid = rv;
    if constexpr (M == RelayoutMode::PackQKV) {
        // run = ((r*3 + t)*B + b)*S_l + s  (destination order)
        const I s = run % S_l, x = run / S_l;
        const I b = x % B, y = x / B;
        const I t = y % 3u, r = y / 3u;
        const uint4 *base = static_cast<const uint4 *>(t == 0 ? a.src0 : (t == 1 ? a.src1 : a.src2));
        src = base + ((static_cast<long long>(b) * a.S_l + s) * a.U + r) * rv;
        dst = static_cast<uint4 *>(a.dst0) + static_cast<long long>(run) * rv;
    } else if constexpr (M == RelayoutMode::PackQKVPad) {
        // as PackQKV over U*h_l padded heads; the source rows hold H_real heads
        const I s = run % S_l, x = run / S_l;
        const I b = x % B, y = x / B;
        const I t = y % 3u, r = y / 3u;
        const long long dv = rv / a.h_l;  // vectors per head
        const long long heads = min(max(a.H_real - static_cast<long long>(r) * a.h_l, 0LL), a.h_l);
        valid = heads * dv;
        const uint4 *base = static_cast<const uint4 *>(t == 0 ? a.src0 : (t == 1 ? a.src1 : a.src2));
        src = base + ((static_cast<long long>(b) * a.S_l + s) * a.H_real + static_cast<long long>(r) * a.h_l) * dv;
        dst = static_cast<uint4 *>(a.dst0) + static_cast<long long>(run) * rv;
    } else if constexpr (M == RelayoutMode::UnpackQKV) {
        // run = ((r*3 + t)*B + b)*S_l + s  (source order)
        const I s = run % S_l, x = run / S_l;
        const I b = x % B, y = x / B;
        const I t = y % 3u, r = y / 3u;
        uint4 *base = static_cast<uint4 *>(t == 0 ? a.dst0 : (t == 1 ? a.dst1 : a.dst2));
        const long long stride = t == 0 ? a.q_batch_stride_rows : a.kv_batch_stride_rows;
        src = static_cast<const uint4 *>(a.src0) + static_cast<long long>(run) * rv;
        dst = base + (static_cast<long long>(b) * stride + static_cast<long long>(r) * a.S_l + s) * rv;
    } else if constexpr (M == RelayoutMode::PackOut) {
        // run = (r*B + b)*S_l + s  (destination order)
        const I s = run % S_l, x = run / S_l;
        const I b = x % B, r = x / B;
        src = static_cast<const uint4 *>(a.src0) +
              (static_cast<long long>(b) * a.q_batch_stride_rows + static_cast<long long>(r) * a.S_l + s) * rv;
        dst = static_cast<uint4 *>(a.dst0) + static_cast<long long>(run) * rv;
    } else if constexpr (M == RelayoutMode::UnpackOut) {
        // run = (r*B + b)*S_l + s  (source order)
        const I s = run % S_l, x = run / S_l;
        const I b = x % B, r = x / B;
        src = static_cast<const uint4 *>(a.src0) + static_cast<long long>(run) * rv;
        dst = static_cast<uint4 *>(a.dst0) + ((static_cast<long long>(b) * a.S_l + s) * a.U + r) * rv;
    } else if constexpr (M == RelayoutMode::UnpackOutPad) {
        // as UnpackOut; destination rows hold H_real heads, pad heads are dropped
        const I s = run % S_l, x = run / S_l;
        const I b = x % B, r = x / B;
        const long long dv = rv / a.h_l;
        const long long heads = min(max(a.H_real - static_cast<long long>(r) * a.h_l, 0LL), a.h_l);
        valid = heads * dv;
        src = static_cast<const uint4 *>(a.src0) + static_cast<long long>(run) * rv;
        dst = static_cast<uint4 *>(a.dst0) +
              ((static_cast<long long>(b) * a.S_l + s) * a.H_real + static_cast<long long>(r) * a.h_l) * dv;
    } else if constexpr (M == RelayoutMode::PackInter) {
        // run = ((r*3 + t)*B + b)*S_l + s: part t (Q, K or V) of the h_l
        // heads destination r takes from row (b, s). The source side is
        // contiguous; on the staging side the run starts at t*dv of the
        // row's first cell and steps over the cells (kernel). Neighbouring
        // warps take neighbouring rows of one part, as in PackQKV (measured
        // 4 % faster with four ranks' packs in flight than the three parts
        // of one row side by side).
        const I s = run % S_l, x = run / S_l;
        const I b = x % B, y = x / B;
        const I t = y % 3u, r = y / 3u;
        const I row = (r * B + b) * S_l + s;
        const long long dv = a.head_vec;
        const long long heads = min(max(a.H_real - static_cast<long long>(r) * a.h_l, 0LL), a.h_l);
        valid = heads * dv;
        const uint4 *base = static_cast<const uint4 *>(t == 0 ? a.src0 : (t == 1 ? a.src1 : a.src2));
        src = base + ((static_cast<long long>(b) * a.S_l + s) * a.H_real + static_cast<long long>(r) * a.h_l) * dv;
        dst = static_cast<uint4 *>(a.dst0) + static_cast<long long>(row) * 3 * rv + static_cast<long long>(t) * dv;
    } else if constexpr (M == RelayoutMode::UnpackInter) {
        // run = ((r*B + b)*S_l + s)*3 + t  (source order), the reverse of PackInter
        const I t = run % 3u, row = run / 3u;
        const I s = row % S_l, x = row / S_l;
        const I b = x % B, r = x / B;
        uint4 *base = static_cast<uint4 *>(t == 0 ? a.dst0 : (t == 1 ? a.dst1 : a.dst2));
        const long long stride = t == 0 ? a.q_batch_stride_rows : a.kv_batch_stride_rows;
        src = static_cast<const uint4 *>(a.src0) + static_cast<long long>(row) * 3 * rv +
              static_cast<long long>(t) * a.head_vec;
        dst = base + (static_cast<long long>(b) * stride + static_cast<long long>(r) * a.S_l + s) * rv;
    } else {
        // AllToAll: run = (g*U + r)*U + j (source order) -> recv[g][j][r]
        const I j = run % U, x = run / U;
        const I r = x % U, g = x / U;
        src = static_cast<const uint4 *>(a.src0) + static_cast<long long>(run) * rv;
        dst = static_cast<uint4 *>(a.dst0) + ((static_cast<long long>(g) * a.U + j) * a.U + r) * rv;
    }
}

template <RelayoutMode M, int VPL, typename I>
__global__ void __launch_bounds__(256) relayout_kernel(RelayoutArgs a, long long n_items, int n_segs)
{
    constexpr long long kSegVec = 32LL * VPL;
    constexpr bool kInter = (M == RelayoutMode::PackInter || M == RelayoutMode::UnpackInter);
    constexpr bool kZeroFill = (M == RelayoutMode::PackQKVPad || M == RelayoutMode::PackInter);
    const int lane = threadIdx.x & 31;
    const long long warp = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const long long n_warps = (static_cast<long long>(gridDim.x) * blockDim.x) >> 5;
    // Interleaved modes: position c of a run is element c % dv of head c / dv,
    // which sits at c + 2*dv*(c / dv) on the staging side (cells of 3*dv). A
    // lane's positions step by 32, so the quotient and remainder are carried
    // from the lane's first position instead of divided per vector.
    I dv = 1, q32 = 0, r32 = 0, h_lane = 0, e_lane = 0;
    if constexpr (kInter) {
        dv = static_cast<I>(a.head_vec);
        q32 = static_cast<I>(32) / dv;
        r32 = static_cast<I>(32) - q32 * dv;
        h_lane = static_cast<I>(lane) / dv;
        e_lane = static_cast<I>(lane) - h_lane * dv;
    }
    for (long long item = warp; item < n_items; item += n_warps) {
        I run = static_cast<I>(item), seg = 0;
        if (n_segs > 1) {
            run = static_cast<I>(item) / static_cast<I>(n_segs);
            seg = static_cast<I>(item) - run * static_cast<I>(n_segs);
        }
        const uint4 *src;
        uint4 *dst;
        long long valid;
        map_run<M, I>(a, run, src, dst, valid);
        const long long base = static_cast<long long>(seg) * kSegVec;
        const long long lim = min(a.run_vec - base, kSegVec);
        const long long vlim = min(valid - base, kSegVec);
        uint4 buf[VPL];
        if constexpr (kInter) {
            // offsets from src / dst of the lane's positions on each side
            I soff[VPL], doff[VPL];
            I h = h_lane, e = e_lane;
            if (seg != 0) {
                const I c0 = static_cast<I>(base + lane);
                h = c0 / dv;
                e = c0 - h * dv;
            }
#pragma unroll
            for (int i = 0; i < VPL; ++i) {
                const I c = static_cast<I>(base + lane + 32 * i);
                soff[i] = M == RelayoutMode::UnpackInter ? c + 2 * dv * h : c;
                doff[i] = M == RelayoutMode::PackInter ? c + 2 * dv * h : c;
                e += r32;
                h += q32;
                if (e >= dv) {
                    e -= dv;
                    ++h;
                }
            }
#pragma unroll
            for (int i = 0; i < VPL; ++i) {
                const long long c = lane + 32 * i;
                if (c < vlim)
                    buf[i] = ld_stream(src + soff[i]);
                else
                    buf[i] = make_uint4(0u, 0u, 0u, 0u);
            }
#pragma unroll
            for (int i = 0; i < VPL; ++i) {
                const long long c = lane + 32 * i;
                if (c < vlim || (kZeroFill && c < lim))
                    dst[doff[i]] = buf[i];
            }
        } else {
#pragma unroll
            for (int i = 0; i < VPL; ++i) {
                const long long c = lane + 32 * i;
                if (c < vlim)
                    buf[i] = ld_stream(src + base + c);
                else
                    buf[i] = make_uint4(0u, 0u, 0u, 0u);
            }
#pragma unroll
            for (int i = 0; i < VPL; ++i) {
                const long long c = lane + 32 * i;
                if (c < vlim || (kZeroFill && c < lim))
                    dst[base + c] = buf[i];
            }
        }
    }
}

// One warp per item: the grid is every item's warp (8 per block), so each
// warp makes one pass and the block scheduler refills an SM as blocks finish
// (the loop over items only matters beyond 2^31 - 1 blocks). Measured against
// a grid of the blocks resident at once with the warps looping: neutral on
// the pack workload's 18.9 MB per-rank launches (-0.7 to +1.3 %), +0.3 to
// +0.9 % on the 480p unpacks, +1.6 to +4.3 % on the Wan-14B-like packs and
// unpacks (ranks' launches concurrent, both staging layouts).
template <RelayoutMode M, int VPL, typename I>
cudaError_t launch_vpl(const RelayoutArgs &a, cudaStream_t stream)
{
    const int n_segs = static_cast<int>((a.run_vec + 32LL * VPL - 1) / (32LL * VPL));
    const long long n_items = a.n_runs * n_segs;
    if (n_items == 0)
        return cudaSuccess;
    const long long want = (n_items + 7) / 8;  // 8 warps per block
    const unsigned grid = static_cast<unsigned>(std::min(want, 0x7fffffffLL));
    relayout_kernel<M, VPL, I><<<grid, 256, 0, stream>>>(a, n_items, n_segs);
    return cudaGetLastError();
}

template <RelayoutMode M, typename I>
cudaError_t launch_mode_i(const RelayoutArgs &a, cudaStream_t stream)
{
    const long long vpl = std::min(8LL, (a.run_vec + 31) / 32);
    switch (vpl) {
    case 1: return launch_vpl<M, 1, I>(a, stream);
    case 2: return launch_vpl<M, 2, I>(a, stream);
    case 3: return launch_vpl<M, 3, I>(a, stream);
    case 4: return launch_vpl<M, 4, I>(a, stream);
    case 5: return launch_vpl<M, 5, I>(a, stream);
    case 6: return launch_vpl<M, 6, I>(a, stream);
    case 7: return launch_vpl<M, 7, I>(a, stream);
    default: return launch_vpl<M, 8, I>(a, stream);
    }
}

template <RelayoutMode M>
cudaError_t launch_mode(const RelayoutArgs &a, cudaStream_t stream)
{
    // 32-bit decomposition when every item index (runs x segments, plus a
    // pass's stride over the grid) and every shape factor fits
    const long long n_segs = (a.run_vec + 255) / 256;  // upper bound over VPL
    const long long lim = 0xffffffffLL / 2;
    const bool i32 = a.n_runs * std::max(1LL, n_segs) <= lim && a.S_l <= lim && a.B <= lim && a.U <= lim &&
                     3 * a.run_vec <= lim;
    return i32 ? launch_mode_i<M, uint32_t>(a, stream) : launch_mode_i<M, long long>(a, stream);
}

}  // namespace

cudaError_t launch_relayout(RelayoutMode mode, const RelayoutArgs &a, cudaStream_t stream)
{
    switch (mode) {
    case RelayoutMode::PackQKV: return launch_mode<RelayoutMode::PackQKV>(a, stream);
    case RelayoutMode::UnpackQKV: return launch_mode<RelayoutMode::UnpackQKV>(a, stream);
    case RelayoutMode::PackOut: return launch_mode<RelayoutMode::PackOut>(a, stream);
    case RelayoutMode::UnpackOut: return launch_mode<RelayoutMode::UnpackOut>(a, stream);
    case RelayoutMode::AllToAll: return launch_mode<RelayoutMode::AllToAll>(a, stream);
    case RelayoutMode::PackQKVPad: return launch_mode<RelayoutMode::PackQKVPad>(a, stream);
    case RelayoutMode::UnpackOutPad: return launch_mode<RelayoutMode::UnpackOutPad>(a, stream);
    case RelayoutMode::PackInter: return launch_mode<RelayoutMode::PackInter>(a, stream);
    case RelayoutMode::UnpackInter: return launch_mode<RelayoutMode::UnpackInter>(a, stream);
    }
    return cudaErrorInvalidValue;
}

}  // namespace ctx
