// Local-Q / global-KV attention forward for sm_103a.
//
// What it computes (vllm-omni PR #7641, local-Q / global-KV attention after
// the K/V AllGather; ChituDiffusion "Fast CP": non-causal MHA): for every
// (b, h, query i), softmax over the valid keys of scale * q.k, applied to V,
// plus the natural-log LSE of the scores.
//
// How (GB300-first design):
//   * one CTA = two 128-row query tiles of one (b, h) sharing one K/V stream;
//   * warp 0 issues TMA loads: both Q tiles once, then K blocks of 128 keys
//     into a two-stage ring (128-byte swizzled tiles, mbarrier complete_tx
//     accounting), and warp 2 the V blocks into their own two-stage ring (in
//     the ticket-merge instantiation for short calls warp 0 loads V too);
//   * warp 1 allocates 512 TMEM columns and runs the MMA loop as a whole warp
//     (warp-uniform descriptors), one elected lane issuing every tcgen05.mma:
//     S_t = Q_t K^T (A and B from shared memory, K-major) into
//     TMEM columns [128t, 128t+128), and O_t += P_t V with P_t read from TMEM
//     (it overwrites S_t as 16-bit pairs) and V from shared memory (MN-major)
//     into columns [256 + Dt, 256 + D(t+1));
//   * warps 4-7 and 8-11 are the softmax of tile 0 and tile 1 (warps 2-3
//     hand registers over, and warp 2 then loads V: the first warpgroup runs
//     with 104 registers per thread, the softmax warpgroups with 200): each thread
//     owns one query row (its TMEM lane), reads its 128 scores with
//     tcgen05.ld, does the online softmax in the log2 domain with exp2, writes
//     P back with tcgen05.st and signals the MMA warp. The MMA warp issues
//     PV_0(j-1), S_0(j), PV_1(j-1), S_1(j), so the tensor core works on one
//     tile while the other tile's softmax runs;
//   * the first key block of a segment takes the block maximum and rescales
//     O only when a row maximum grows by more than 2^8 (a stale maximum keeps
//     every probability <= 2^8, exact after the final division), which the
//     public FlashAttention-4 write-up calls conditional rescaling; every
//     later block takes the exps against the running maximum directly and
//     keeps them when the block's probability sum is at most 2^15 (else the
//     block goes through the exact path, its scores still in TMEM);
//   * epilogue: O / l rounded to the input type, LSE = ln2 * (m + log2 l);
//   * schedules: one CTA per work unit, or (given a workspace) a persistent
//     grid of one CTA per SM that cuts units' key ranges between SMs and
//     merges the pieces by log-sum-exp; for packed varlen documents the
//     split iteration space is planned on the device (varlen.cu). Without a
//     workspace, where a last wave of 256-row units would leave SMs idle, a
//     unit is one 128-row tile whose key range the two tile slots share out
//     in halves (warp 2 then loads V), merged inside the CTA.
// Every wait is bounded (%globaltimer); on expiry the kernel records a
// timeout in the device status word, drains its own TMA loads and MMAs, frees
// TMEM and returns.
#include <algorithm>
#include <cmath>
#include <cudaTypedefs.h>
#include <mutex>

#include "internal.h"
#include "ptx.cuh"

namespace ctx {
namespace {

constexpr int kBM = 128;      // query rows per tile (= TMEM lanes)
constexpr int kBN = kAttnKeyBlock;  // keys per block (128)
constexpr int kTiles = 2;     // query tiles per CTA
constexpr int kStages = 2;    // depth of the K ring (two-tile units) and of the V ring
constexpr int kThreads = 384; // 12 warps: Q/K loads, MMA, V loads, one spare, 4 + 4 softmax
// Registers: the kernel is launched with kRegsLaunch per thread (the compiler's
// figure for 384 threads, checked on the host before the first launch); the
// first warpgroup (TMA, MMA) gives registers up to the two softmax warpgroups.
constexpr int kRegsLaunch = 168;
constexpr int kRegsControl = 104;
constexpr int kRegsSoftmax = 200;
static_assert(kRegsControl * 128 + kRegsSoftmax * 256 == kRegsLaunch * kThreads, "register split");
constexpr int kTmemCols = 512;
constexpr float kRescaleLog2 = 8.0f;
constexpr float kFastSumLimit = 32768.0f;  // 2^15: largest block sum accepted against a stale maximum
constexpr float kLn2 = 0.693147180559945309f;
static_assert(kTiles * kBM == kAttnUnitRows, "work unit rows");

struct Params {
    const unsigned char *mask;
    void *out;
    float *lse;
    int B, Sq, Sk, H;
    int n_qpairs;
    int n_kblocks;
    const int *cu_q;       // packed varlen: [n_docs + 1] local query boundaries (device), else NULL
    const int *cu_k;       // packed varlen: [n_docs + 1] key boundaries (device)
    int varlen;            // 1: units are (query-tile pair, head, document)
    int n_docs;            // packed varlen: documents
    const long long *var_prefix;  // packed varlen, balanced: [n_docs + 1] first key-block iteration of
                                  // every document (written on the device before the launch), else NULL
    int blk_s, blk_u, blk_b;  // > 0: out is the reverse exchange's send buffer (see out_row)
    int n_units;           // work units: (query-tile pair, head, batch or document)
    int grid;              // persistent CTAs
    int dp_waves;          // whole-unit waves: CTA c takes units c, c+grid, ...
    long long tail_iters;  // key blocks of the remaining units, split evenly over the grid
    float scale_log2;
    int *status;
    unsigned long long wait_limit_ns;
    int *counters;         // [n_units][kTiles][2] arrived / written pieces of split units (zero between calls)
    float2 *part_ml;       // [2*grid][kTiles*kBM] (m, l) of partial segments
    float4 *part_o;        // [2*grid][D/4][kTiles*kBM] unnormalised O of partial segments
};

// kHalves: units of one 128-row tile whose key range the two tile slots share
// out in halves (one Q tile in shared memory; the room of the other holds a
// third K stage, since the two slots draw two K blocks per step).
template <int D, bool kHalves = false>
struct Layout {
    static constexpr int kPanels = D / 64;          // 64-element (128-byte) swizzle panels
    static constexpr int kQBytes = kBM * D * 2;     // one Q tile
    static constexpr int kKVBytes = kBN * D * 2;    // one K or V block
    static constexpr int kQPanel = kBM * 128;       // bytes of one panel of a Q tile
    static constexpr int kKVPanel = kBN * 128;
    static constexpr int kQTiles = kHalves ? 1 : kTiles;
    static constexpr int kKStages = kHalves ? 3 : kStages;
    static constexpr int kVStages = kStages;
    static constexpr int kQOff = 0;
    static constexpr int kKOff = kQOff + kQTiles * kQBytes;
    static constexpr int kVOff = kKOff + kKStages * kKVBytes;
    static constexpr int kBarOff = kVOff + kVStages * kKVBytes;
    // q_full, q_empty, k_full[KS], k_empty[KS], v_full[VS], v_empty[VS],
    // s_full[T], p_full[T], o_full[T], o_empty[T], seg_done[T], merge_go[T], written_go[T], mma_done
    static constexpr int kNumBars = 2 + 2 * kKStages + 2 * kVStages + 7 * kTiles + 1;
    static constexpr int kMiscOff = kBarOff + kNumBars * 8;
    // per softmax warp: its 32 rows x 64 output columns, staged so that the
    // output rows leave as whole 128-byte lines
    static constexpr int kEpiWarpBytes = 32 * 128;
    static constexpr int kEpiOff = (kMiscOff + 32 + 127) / 128 * 128;
    static constexpr int kBytes = kEpiOff + 2 * 4 * kEpiWarpBytes;
    static constexpr int kAlloc = kBytes + 1024;    // room to align the base to 1024 B
    static_assert(kAlloc <= 227 * 1024, "shared memory per CTA");
};

// One contiguous run of key blocks [jb, je) of one work unit. first: the
// unit's first iteration in the split order; nb: the unit's key blocks.
struct Segment {
    int unit, jb, je, slot;
    bool full;
    long long first;
    int nb;
};

// Geometry of one work unit: kRows (256, or 128 in the halves mode) query
// rows [q0, min(q0 + kRows, q_end)) of head h and batch b, against keys
// [k0, k0 + k_len) in key blocks of 128.
// Packed varlen: the unit's document d gives q0 = cu_q[d] + 256*qp,
// q_end = cu_q[d+1], keys [cu_k[d], cu_k[d+1]) (vllm-omni PR #7641: local
// query boundaries, global key boundaries). nblk = 0 means nothing to compute.
struct Geom {
    int b, h, q0, q_end, k0, k_len, nblk;
};

template <int kRows = kTiles * kBM>
__device__ __forceinline__ void unit_geom(const Params &p, int unit, Geom &g)
{
    const int qp = unit % p.n_qpairs, bh = unit / p.n_qpairs;
    g.h = bh % p.H;
    const int x = bh / p.H;
    if (!p.varlen) {
        g.b = x;
        g.q0 = qp * kRows;
        g.q_end = p.Sq;
        g.k0 = 0;
        g.k_len = p.Sk;
    } else {
        // boundaries are clamped to the tensors, so malformed ones cannot
        // address memory outside q/out or k/v/mask
        g.b = 0;
        const int qs = min(max(__ldg(p.cu_q + x), 0), p.Sq);
        g.q0 = qs + qp * (kTiles * kBM);
        g.q_end = min(max(__ldg(p.cu_q + x + 1), qs), p.Sq);
        g.k0 = min(max(__ldg(p.cu_k + x), 0), p.Sk);
        g.k_len = min(max(__ldg(p.cu_k + x + 1), g.k0), p.Sk) - g.k0;
    }
    g.nblk = (g.q0 < g.q_end && g.k_len > 0) ? (g.k_len + kBN - 1) / kBN : 0;
}

// First element of output row (b, qrow, h). Plain layout: [B, Sq, H, D].
// Reverse-exchange layout (blk_s > 0, the send-side relayout of the output
// exchange fused into the epilogue): query row q = (a*blk_u + r)*blk_s + s
// of batch b = u*blk_b + b' goes to the send buffer of rank (a, u),
// destination r: [a][u][r][b'][s] — for one rank's call (a = u = 0) that is
// [U][B][S_l], the layout ctx_pack_out writes.
template <int D>
__device__ __forceinline__ uint4 *out_row(const Params &p, int b, int h, int qrow)
{
    size_t row;
    if (p.blk_s > 0) {
        const int qb = qrow / p.blk_s, s = qrow - qb * p.blk_s;
        const int a = qb / p.blk_u, r = qb - a * p.blk_u;
        const int u = b / p.blk_b, bb = b - u * p.blk_b;
        row = ((static_cast<size_t>(a) * p.blk_u + u) * p.blk_u + r) * p.blk_b * p.blk_s +
              static_cast<size_t>(bb) * p.blk_s + s;
    } else {
        row = static_cast<size_t>(b) * p.Sq + qrow;
    }
    return reinterpret_cast<uint4 *>(static_cast<uint16_t *>(p.out) + (row * p.H + h) * D);
}

// Output staging of one softmax warp (32 rows x 64 columns, 4 KB): row =
// lane, 16-byte chunk j of the row at j ^ (row & 7), so that both the row-wise
// writes and the line-wise reads hit 8 distinct bank groups per quarter warp.
// stage32: this thread's columns [32*qq, 32*qq + 32) of the half, times
// `scale`, rounded to the output type.
template <bool BF16>
__device__ __forceinline__ void stage32(uint4 *stg, int lane, int qq, const float *v, float scale)
{
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const int j = 4 * qq + k;
        stg[lane * 8 + (j ^ (lane & 7))] = make_uint4(ptx::pack2<BF16>(v[8 * k + 0] * scale, v[8 * k + 1] * scale),
                                                      ptx::pack2<BF16>(v[8 * k + 2] * scale, v[8 * k + 3] * scale),
                                                      ptx::pack2<BF16>(v[8 * k + 4] * scale, v[8 * k + 5] * scale),
                                                      ptx::pack2<BF16>(v[8 * k + 6] * scale, v[8 * k + 7] * scale));
    }
}

// The warp's staged half rows to global memory, four whole 128-byte row
// pieces per store instruction. orow: this lane's output row (0: the row does
// not exist); col16: the half's first 16-byte column. Warp-wide.
__device__ __forceinline__ void store_staged(const uint4 *stg, int lane, unsigned long long orow, int col16)
{
    __syncwarp();
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int r = 4 * i + (lane >> 3), cc = lane & 7;
        uint4 *const dst = reinterpret_cast<uint4 *>(__shfl_sync(0xffffffffu, orow, r));
        if (dst)
            dst[col16 + cc] = stg[r * 8 + (cc ^ (r & 7))];
    }
    __syncwarp();
}

// Segment `si` of CTA c, computed from its index alone (identical in every
// warp role, and no iterator state lives across the key-block loops): first
// the whole-unit waves (concurrent CTAs work on neighbouring units, so they
// share the same heads' K/V in L2), then an even share of the remaining
// units' key blocks, cut at unit boundaries (so every SM finishes at the same
// time; units cut between CTAs are merged by log-sum-exp).
__device__ __forceinline__ long long tail_start(const Params &p, long long total, int c)
{
    return static_cast<long long>(c) * total / p.grid;
}

// CTA whose tail range holds tail iteration `it`.
__device__ __forceinline__ int tail_cta_of(const Params &p, long long total, long long it)
{
    return static_cast<int>(((it + 1) * p.grid + total - 1) / total) - 1;
}

// Slot of CTA cc's piece of the unit whose first split iteration is `first`:
// the CTA's first segment when its range starts inside the unit, else its
// last one.
__device__ __forceinline__ int tail_slot(const Params &p, long long total, long long first, int cc)
{
    return (tail_start(p, total, cc) >= first) ? 2 * cc : 2 * cc + 1;
}

// Iterations shared by the split schedule: the tail of the dense schedule,
// or every key block of every document in the balanced varlen schedule.
__device__ __forceinline__ long long split_total(const Params &p)
{
    return p.var_prefix ? __ldg(p.var_prefix + p.n_docs) : p.tail_iters;
}

// Balanced packed varlen: the unit holding split iteration y (documents in
// order, then heads, then query-tile pairs, then key blocks; empty units hold
// no iteration), its first iteration and its key blocks. The per-document
// counts follow unit_geom exactly.
__device__ __forceinline__ void var_unit_at(const Params &p, long long y, int &unit, long long &ustart, int &nb)
{
    int lo = 0, hi = p.n_docs - 1;
    while (lo < hi) {  // the last document whose first iteration is <= y (skips empty ones)
        const int mid = (lo + hi + 1) >> 1;
        if (__ldg(p.var_prefix + mid) <= y)
            lo = mid;
        else
            hi = mid - 1;
    }
    const int d = lo;
    const int qs = min(max(__ldg(p.cu_q + d), 0), p.Sq);
    const int q_len = min(max(__ldg(p.cu_q + d + 1), qs), p.Sq) - qs;
    const int k0 = min(max(__ldg(p.cu_k + d), 0), p.Sk);
    const int k_len = min(max(__ldg(p.cu_k + d + 1), k0), p.Sk) - k0;
    nb = (k_len + kBN - 1) / kBN;
    const int nqp = min((q_len + kTiles * kBM - 1) / (kTiles * kBM), p.n_qpairs);
    const long long off = y - __ldg(p.var_prefix + d);
    const long long per_h = static_cast<long long>(nqp) * nb;
    const int h = static_cast<int>(off / per_h);
    const long long r = off - h * per_h;
    const int qp = static_cast<int>(r / nb), blk = static_cast<int>(r - static_cast<long long>(qp) * nb);
    unit = qp + p.n_qpairs * (h + p.H * d);
    ustart = y - blk;
}

__device__ __forceinline__ bool segment_at(const Params &p, int c, int si, Segment &s)
{
    if (p.var_prefix) {
        // balanced packed varlen: CTA c takes split iterations [x0, x1), cut at unit ends
        const long long total = split_total(p);
        const long long x0 = tail_start(p, total, c), x1 = tail_start(p, total, c + 1);
        long long y = x0, ustart = 0;
        int unit = 0, nb = 0;
        for (int j = 0;; ++j) {
            if (y >= x1)
                return false;
            var_unit_at(p, y, unit, ustart, nb);
            if (j == si)
                break;
            y = ustart + nb;
        }
        s.unit = unit;
        s.jb = static_cast<int>(y - ustart);
        s.je = static_cast<int>(min(static_cast<long long>(nb), x1 - ustart));
        s.full = (s.jb == 0 && s.je == nb);
        s.slot = (si == 0) ? 2 * c : 2 * c + 1;
        s.first = ustart;
        s.nb = nb;
        return true;
    }
    if (si < p.dp_waves) {
        s.unit = si * p.grid + c;
        s.jb = 0;
        if (p.varlen) {
            Geom g;
            unit_geom(p, s.unit, g);
            s.je = g.nblk;  // 0: an empty unit, skipped by every role
        } else {
            s.je = p.n_kblocks;
        }
        s.full = true;
        s.slot = -1;
        s.first = 0;
        s.nb = s.je;
        return true;
    }
    const long long nb = p.n_kblocks;
    const long long tb = static_cast<long long>(c) * p.tail_iters / p.grid;
    const long long te = static_cast<long long>(c + 1) * p.tail_iters / p.grid;
    const int k = si - p.dp_waves;
    const long long u0 = tb / nb;
    const long long start = (k == 0) ? tb : (u0 + k) * nb;
    if (start >= te)
        return false;
    const long long end = min(te, (u0 + k + 1) * nb);
    const long long u = start / nb;
    s.unit = p.dp_waves * p.grid + static_cast<int>(u);
    s.jb = static_cast<int>(start - u * nb);
    s.je = s.jb + static_cast<int>(end - start);
    s.full = (s.jb == 0 && s.je == p.n_kblocks);
    s.slot = (k == 0) ? 2 * c : 2 * c + 1;
    s.first = u * nb;
    s.nb = p.n_kblocks;
    return true;
}

// Hides the value of i from the optimiser, so a segment recomputed after a
// hot loop is not kept live in registers across it.
__device__ __forceinline__ int opaque(int i)
{
    asm volatile("" : "+r"(i));
    return i;
}

// Bounded wait on an mbarrier phase. honor_abort: give up as soon as another
// role has aborted. Returns false on abort or timeout.
__device__ __forceinline__ bool wait_bar(uint64_t *bar, uint32_t parity, volatile int *abort_flag,
                                         const Params &p, bool honor_abort = true)
{
    const uint32_t a = ptx::smem_u32(bar);
    if (ptx::mbar_try_wait(a, parity))
        return true;
    const uint64_t t0 = ptx::globaltimer();
    uint32_t spins = 0;
    while (true) {
        if (ptx::mbar_try_wait(a, parity))
            return true;
        if ((++spins & 31u) == 0) {
            if (honor_abort && *abort_flag)
                return false;
            if (ptx::globaltimer() - t0 > p.wait_limit_ns) {
                *abort_flag = 1;
                atomicExch(p.status, kStatusTimeout);
                return false;
            }
        }
    }
}

// Warp-uniform version for the softmax warps (tcgen05.ld/st are .sync.aligned).
__device__ __forceinline__ bool wait_bar_warp(uint64_t *bar, uint32_t parity, volatile int *abort_flag,
                                              const Params &p)
{
    const bool ok = wait_bar(bar, parity, abort_flag, p);
    return __all_sync(0xffffffffu, ok);
}

template <int D, bool BF16>
__device__ __forceinline__ void issue_qk(uint32_t tmem_s, uint32_t q_smem, uint32_t k_smem)
{
    using L = Layout<D>;
    constexpr uint32_t idesc = ptx::idesc_f16(kBM, kBN, BF16, false, false);
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t pnl = kk / 4, koff = (kk % 4) * 32;
        const uint64_t a = ptx::sdesc_sw128(q_smem + pnl * L::kQPanel + koff, 16, 1024);
        const uint64_t b = ptx::sdesc_sw128(k_smem + pnl * L::kKVPanel + koff, 16, 1024);
        ptx::mma_ss(tmem_s, a, b, idesc, kk > 0 ? 1u : 0u);
    }
}

template <int D, bool BF16>
__device__ __forceinline__ void issue_pv(uint32_t tmem_o, uint32_t tmem_p, uint32_t v_smem, bool accumulate)
{
    using L = Layout<D>;
    constexpr uint32_t idesc = ptx::idesc_f16(kBM, D, BF16, false, true);
#pragma unroll
    for (int kk = 0; kk < kBN / 16; ++kk) {
        // 16 keys = two 8-row groups of 128 B; the next 64 d-columns are one panel further
        const uint64_t b = ptx::sdesc_sw128(v_smem + kk * 16 * 128, L::kKVPanel, 1024);
        ptx::mma_ts(tmem_o, tmem_p + kk * 8, b, idesc, (accumulate || kk > 0) ? 1u : 0u);
    }
}

// Log-sum-exp merge of the pieces of a split unit (log2 domain): fold_ml
// takes the next piece's (m, l) into the running maximum M and sum lsum (a
// piece without a valid key, m = -inf, adds nothing); piece_weight is a
// piece's factor against the final M; add_piece accumulates a weighted
// piece. The ticket-first merge goes through these on both of its paths.
__device__ __forceinline__ void fold_ml(float &M, float &lsum, float2 ml)
{
    if (ml.x == -INFINITY)
        return;
    if (ml.x > M) {
        lsum = (M == -INFINITY) ? ml.y : fmaf(lsum, ptx::ex2_approx(M - ml.x), ml.y);
        M = ml.x;
    } else {
        lsum = fmaf(ptx::ex2_approx(ml.x - M), ml.y, lsum);
    }
}

__device__ __forceinline__ float piece_weight(float2 ml, float M)
{
    return (ml.x == -INFINITY) ? 0.f : ptx::ex2_approx(ml.x - M);
}

__device__ __forceinline__ float add_piece(float acc, float w, float v)
{
    return fmaf(w, v, acc);
}

// kTicketMerge: the merge protocol of units cut between CTAs (see the partial
// segment branch): a piece takes its arrival ticket as its last key block
// starts and the last one merges the others with its own O from TMEM
// (true), or every piece writes its partial and the last to have written
// merges them all from the workspace (false). The first shortens the end of
// a short call; the second is kept for long calls, where the kernel built
// without the ticket code runs its key-block loop faster.
template <int D, bool BF16, bool kTicketMerge, bool kHalves>
__global__ void __launch_bounds__(kThreads, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const Params p)
{
    static_assert(!(kTicketMerge && kHalves), "halves units are never split between CTAs");
    using L = Layout<D, kHalves>;
    constexpr int kUnitRows = kHalves ? kBM : kTiles * kBM;  // query rows of a work unit
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L::kBarOff);
    uint64_t *q_full = bars;
    uint64_t *q_empty = q_full + 1;
    uint64_t *k_full = q_empty + 1;
    uint64_t *k_empty = k_full + L::kKStages;
    uint64_t *v_full = k_empty + L::kKStages;
    uint64_t *v_empty = v_full + L::kVStages;
    uint64_t *s_full = v_empty + L::kVStages;
    uint64_t *p_full = s_full + kTiles;
    uint64_t *o_full = p_full + kTiles;
    uint64_t *o_empty = o_full + kTiles;
    uint64_t *seg_done = o_empty + kTiles;
    uint64_t *merge_go = seg_done + kTiles;
    uint64_t *written_go = merge_go + kTiles;
    uint64_t *mma_done = written_go + kTiles;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L::kMiscOff);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L::kMiscOff + 4);
    volatile int *merge_flag = reinterpret_cast<volatile int *>(smem + L::kMiscOff + 8);  // [kTiles]

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int cta = blockIdx.x;

    if (threadIdx.x == 0) {
        ptx::mbar_init(q_full, 1);
        ptx::mbar_init(q_empty, 1);
        for (int s = 0; s < L::kKStages; ++s) {
            ptx::mbar_init(k_full + s, 1);
            ptx::mbar_init(k_empty + s, 1);
        }
        for (int s = 0; s < L::kVStages; ++s) {
            ptx::mbar_init(v_full + s, 1);
            ptx::mbar_init(v_empty + s, 1);
        }
        for (int t = 0; t < kTiles; ++t) {
            ptx::mbar_init(s_full + t, 1);
            ptx::mbar_init(p_full + t, 128);
            ptx::mbar_init(o_full + t, 1);
            ptx::mbar_init(o_empty + t, 128);
            ptx::mbar_init(seg_done + t, 128);
            ptx::mbar_init(merge_go + t, 1);
            ptx::mbar_init(written_go + t, 1);
            merge_flag[t] = 0;
        }
        ptx::mbar_init(mma_done, 1);
        *abort_flag = 0;
        ptx::fence_mbar_init();
    }
    if (warp == 1) {
        ptx::tmem_alloc(tmem_slot, kTmemCols);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        ptx::setmaxnreg_dec<kRegsControl>();
        if (lane == 0) {
            ptx::tma_prefetch_desc(&tmQ);
            ptx::tma_prefetch_desc(&tmK);
            ptx::tma_prefetch_desc(&tmV);
            Segment sg;
            int kv = 0, act = 0;  // act: segments with work so far (phase of the per-segment barriers)
            int last_k[L::kKStages], last_v[L::kVStages];
            for (int s = 0; s < L::kKStages; ++s)
                last_k[s] = -1;
            for (int s = 0; s < L::kVStages; ++s)
                last_v[s] = -1;
            bool ok = true;
            for (int segi = 0; ok && segment_at(p, cta, segi, sg); ++segi) {
                if (sg.je == sg.jb)
                    continue;
                Geom ge;
                unit_geom<kUnitRows>(p, sg.unit, ge);
                const int h = ge.h, b = ge.b;
                if (act > 0 && !(ok = wait_bar(q_empty, (act - 1) & 1, abort_flag, p)))
                    break;
                ptx::mbar_arrive_expect_tx(q_full, L::kQTiles * L::kQBytes);
                for (int t = 0; t < L::kQTiles; ++t)
                    for (int pn = 0; pn < L::kPanels; ++pn)
                        ptx::tma_load_4d(&tmQ, q_full, smem + L::kQOff + t * L::kQBytes + pn * L::kQPanel, pn * 64,
                                         h, ge.q0 + t * kBM, b);
                ++act;
                if constexpr (kHalves) {
                    // Slot t takes key blocks [t*nh, t*nh + nh) of the unit's nb (the
                    // second slot one fewer when nb is odd), loaded in the order the MMA
                    // warp consumes them: block kv is step kv >> 1 of slot kv & 1 (only
                    // the last step can lack the second slot's block). This thread
                    // loads K; warp 2 loads V, so that a V stage waiting for its slot's
                    // previous PV never holds back the next K block.
                    const int nb = sg.je - sg.jb, nh = (nb + 1) / 2;
                    for (kv = 0; kv < nb; ++kv) {
                        const int j = sg.jb + (kv & 1) * nh + (kv >> 1);
                        const int sk = kv % L::kKStages, uk = kv / L::kKStages;
                        if (uk > 0 && !(ok = wait_bar(k_empty + sk, (uk - 1) & 1, abort_flag, p)))
                            break;
                        ptx::mbar_arrive_expect_tx(k_full + sk, L::kKVBytes);
                        for (int pn = 0; pn < L::kPanels; ++pn)
                            ptx::tma_load_4d(&tmK, k_full + sk, smem + L::kKOff + sk * L::kKVBytes + pn * L::kKVPanel,
                                             pn * 64, h, ge.k0 + j * kBN, b);
                        last_k[sk] = uk;
                    }
                } else {
                    for (int j = sg.jb; j < sg.je; ++j, ++kv) {
                        const int s = kv % kStages, u = kv / kStages;
                        if (u > 0 && !(ok = wait_bar(k_empty + s, (u - 1) & 1, abort_flag, p)))
                            break;
                        ptx::mbar_arrive_expect_tx(k_full + s, L::kKVBytes);
                        for (int pn = 0; pn < L::kPanels; ++pn)
                            ptx::tma_load_4d(&tmK, k_full + s, smem + L::kKOff + s * L::kKVBytes + pn * L::kKVPanel,
                                             pn * 64, h, ge.k0 + j * kBN, b);
                        last_k[s] = u;
                        if constexpr (kTicketMerge) {  // other instantiations: warp 2 loads V
                            if (u > 0 && !(ok = wait_bar(v_empty + s, (u - 1) & 1, abort_flag, p)))
                                break;
                            ptx::mbar_arrive_expect_tx(v_full + s, L::kKVBytes);
                            for (int pn = 0; pn < L::kPanels; ++pn)
                                ptx::tma_load_4d(&tmV, v_full + s,
                                                 smem + L::kVOff + s * L::kKVBytes + pn * L::kKVPanel, pn * 64, h,
                                                 ge.k0 + j * kBN, b);
                            last_v[s] = u;
                        }
                    }
                }
            }
            // Drain: every issued load has landed before the CTA can exit.
            if (act > 0)
                wait_bar(q_full, (act - 1) & 1, abort_flag, p, false);
            for (int s = 0; s < L::kKStages; ++s)
                if (last_k[s] >= 0)
                    wait_bar(k_full + s, last_k[s] & 1, abort_flag, p, false);
            for (int s = 0; s < L::kVStages; ++s)
                if (last_v[s] >= 0)
                    wait_bar(v_full + s, last_v[s] & 1, abort_flag, p, false);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issue
        ptx::setmaxnreg_dec<kRegsControl>();
        // The whole warp runs this loop (warp-uniform values, warp-wide waits);
        // one elected lane issues each MMA and commit.
        {
            const uint32_t qa0 = ptx::smem_u32(smem + L::kQOff);
            const uint32_t qa1 = qa0 + L::kQBytes;
            const uint32_t kbase = ptx::smem_u32(smem + L::kKOff);
            const uint32_t vbase = ptx::smem_u32(smem + L::kVOff);
            const uint32_t tS0 = tmem, tS1 = tmem + kBN;
            const uint32_t tO0 = tmem + 2 * kBN, tO1 = tmem + 2 * kBN + D;
            Segment sg;
            int kv = 0, g = 0, act = 0;
            bool ok = true;
            if constexpr (kHalves) {
                // One unit per CTA (one segment). Step i: slot 0's PV of block i-1 and
                // QK^T of block i, then slot 1's; every K and V block belongs to one slot.
                // Block kv is step i = kv >> 1 of slot t = kv & 1, whose V stage is t.
                if (segment_at(p, cta, 0, sg) && sg.je > sg.jb) {
                    const int nb = sg.je - sg.jb;
                    ok = wait_bar_warp(q_full, 0, abort_flag, p);
                    ptx::tc_fence_after();
                    for (kv = 0; ok && kv < nb; ++kv) {
                        const int i = kv >> 1, t = kv & 1;
                        const int sk = kv % L::kKStages, uk = kv / L::kKStages;
                        if (!(ok = wait_bar_warp(k_full + sk, uk & 1, abort_flag, p)))
                            break;
                        ptx::tc_fence_after();
                        const uint32_t tS = tmem + t * kBN;
                        if (i > 0) {  // this slot's PV of block i - 1 (V stage t, its use i - 1)
                            if (!(ok = wait_bar_warp(v_full + t, (i - 1) & 1, abort_flag, p) &&
                                       wait_bar_warp(p_full + t, (i - 1) & 1, abort_flag, p)))
                                break;
                            ptx::tc_fence_after();
                            issue_pv<D, BF16>(tmem + 2 * kBN + t * D, tS, vbase + t * L::kKVBytes, i > 1);
                            ptx::tc_commit(v_empty + t);
                        }
                        issue_qk<D, BF16>(tS, qa0, kbase + sk * L::kKVBytes);
                        ptx::tc_commit(s_full + t);
                        ptx::tc_commit(k_empty + sk);
                    }
                    if (ok)
                        ptx::tc_commit(q_empty);
                    for (int t = 0; ok && t < 2; ++t) {  // each slot's last PV
                        const int nt = t ? nb / 2 : (nb + 1) / 2;
                        if (nt == 0)
                            break;
                        if (!(ok = wait_bar_warp(v_full + t, (nt - 1) & 1, abort_flag, p) &&
                                   wait_bar_warp(p_full + t, (nt - 1) & 1, abort_flag, p)))
                            break;
                        ptx::tc_fence_after();
                        issue_pv<D, BF16>(tmem + 2 * kBN + t * D, tmem + t * kBN, vbase + t * L::kKVBytes, nt > 1);
                        ptx::tc_commit(o_full + t);
                        ptx::tc_commit(v_empty + t);
                    }
                }
            } else {
                for (int segi = 0; ok && segment_at(p, cta, segi, sg); ++segi) {
                    const int n = sg.je - sg.jb;
                    if (n == 0)
                        continue;
                    if (!(ok = wait_bar_warp(q_full, act & 1, abort_flag, p)))
                        break;
                    ptx::tc_fence_after();
                    for (int i = 0; i < n; ++i) {
                        const int cur = kv + i, s = cur % kStages, u = cur / kStages;
                        if (!(ok = wait_bar_warp(k_full + s, u & 1, abort_flag, p)))
                            break;
                        ptx::tc_fence_after();
                        const int prv = cur - 1, sp = (cur + kStages - 1) % kStages, up = prv / kStages;
                        if (i > 0) {
                            if (!(ok = wait_bar_warp(v_full + sp, up & 1, abort_flag, p)))
                                break;
                            if (!(ok = wait_bar_warp(p_full + 0, (g + i - 1) & 1, abort_flag, p)))
                                break;
                            if (i == 1 && act > 0 && !(ok = wait_bar_warp(o_empty + 0, (act - 1) & 1, abort_flag, p)))
                                break;
                            ptx::tc_fence_after();
                            issue_pv<D, BF16>(tO0, tS0, vbase + sp * L::kKVBytes, i > 1);
                        }
                        issue_qk<D, BF16>(tS0, qa0, kbase + s * L::kKVBytes);
                        ptx::tc_commit(s_full + 0);
                        if (i > 0) {
                            if (!(ok = wait_bar_warp(p_full + 1, (g + i - 1) & 1, abort_flag, p)))
                                break;
                            if (i == 1 && act > 0 && !(ok = wait_bar_warp(o_empty + 1, (act - 1) & 1, abort_flag, p)))
                                break;
                            ptx::tc_fence_after();
                            issue_pv<D, BF16>(tO1, tS1, vbase + sp * L::kKVBytes, i > 1);
                            ptx::tc_commit(v_empty + sp);
                        }
                        issue_qk<D, BF16>(tS1, qa1, kbase + s * L::kKVBytes);
                        ptx::tc_commit(s_full + 1);
                        ptx::tc_commit(k_empty + s);
                    }
                    if (!ok)
                        break;
                    ptx::tc_commit(q_empty);  // the segment's QK^T products are all issued
                    const int lst = kv + n - 1, sl = lst % kStages, ul = lst / kStages;
                    ok = wait_bar_warp(v_full + sl, ul & 1, abort_flag, p) &&
                         wait_bar_warp(p_full + 0, (g + n - 1) & 1, abort_flag, p) &&
                         (n > 1 || act == 0 || wait_bar_warp(o_empty + 0, (act - 1) & 1, abort_flag, p));
                    if (!ok)
                        break;
                    ptx::tc_fence_after();
                    issue_pv<D, BF16>(tO0, tS0, vbase + sl * L::kKVBytes, n > 1);
                    ptx::tc_commit(o_full + 0);
                    ok = wait_bar_warp(p_full + 1, (g + n - 1) & 1, abort_flag, p) &&
                         (n > 1 || act == 0 || wait_bar_warp(o_empty + 1, (act - 1) & 1, abort_flag, p));
                    if (!ok)
                        break;
                    ptx::tc_fence_after();
                    issue_pv<D, BF16>(tO1, tS1, vbase + sl * L::kKVBytes, n > 1);
                    ptx::tc_commit(o_full + 1);
                    ptx::tc_commit(v_empty + sl);
                    kv += n;
                    g += n;
                    ++act;
                }
            }
            // Every MMA issued above has retired before TMEM is released.
            ptx::tc_commit(mma_done);
            wait_bar(mma_done, 0, abort_flag, p, false);
            __syncwarp();
        }
    } else if (warp < 4) {
        ptx::setmaxnreg_dec<kRegsControl>();  // warps 2-3: registers only
        if constexpr (kHalves) {
            // ------------------------------------------------ V loads (halves units)
            // Block kv is step kv >> 1 of slot kv & 1; V stage t belongs to slot t
            // and is reused once that slot's PV of the previous step has retired.
            static_assert(L::kVStages == 2, "V stage t belongs to slot t");
            Segment sg;
            if (warp == 2 && lane == 0 && segment_at(p, cta, 0, sg) && sg.je > sg.jb) {
                ptx::tma_prefetch_desc(&tmV);
                Geom ge;
                unit_geom<kUnitRows>(p, sg.unit, ge);
                const int nb = sg.je - sg.jb, nh = (nb + 1) / 2;
                int last_v[2] = {-1, -1};
                for (int kv = 0; kv < nb; ++kv) {
                    const int sv = kv & 1, uv = kv >> 1;
                    if (uv > 0 && !wait_bar(v_empty + sv, (uv - 1) & 1, abort_flag, p))
                        break;
                    ptx::mbar_arrive_expect_tx(v_full + sv, L::kKVBytes);
                    for (int pn = 0; pn < L::kPanels; ++pn)
                        ptx::tma_load_4d(&tmV, v_full + sv, smem + L::kVOff + sv * L::kKVBytes + pn * L::kKVPanel,
                                         pn * 64, ge.h, ge.k0 + (sg.jb + sv * nh + uv) * kBN, ge.b);
                    last_v[sv] = uv;
                }
                // Drain: every issued load has landed before the CTA can exit.
                for (int s = 0; s < 2; ++s)
                    if (last_v[s] >= 0)
                        wait_bar(v_full + s, last_v[s] & 1, abort_flag, p, false);
            }
        } else if constexpr (!kTicketMerge) {
            // ------------------------------------------------ V loads (long calls)
            // Warp 0 loads Q and K; this thread loads V, so that a V stage waiting
            // for its PV never holds back the next K block (same-box A/B on GB300:
            // the batched Wan-like 480p call 1655 -> 1669-1671 TFLOP/s, one 480p rank
            // 1637-1641 -> 1647; the short calls of the ticket-merge instantiation
            // measured no better and keep V in the producer). Block kv of the load
            // order is the kv-th key block of the CTA's segments.
            if (warp == 2 && lane == 0) {
                ptx::tma_prefetch_desc(&tmV);
                int last_v[L::kVStages];
                for (int s = 0; s < L::kVStages; ++s)
                    last_v[s] = -1;
                Segment sg;
                int kv = 0;
                bool ok = true;
                for (int segi = 0; ok && segment_at(p, cta, segi, sg); ++segi) {
                    if (sg.je == sg.jb)
                        continue;
                    Geom ge;
                    unit_geom<kUnitRows>(p, sg.unit, ge);
                    for (int j = sg.jb; j < sg.je; ++j, ++kv) {
                        const int s = kv % L::kVStages, u = kv / L::kVStages;
                        if (u > 0 && !(ok = wait_bar(v_empty + s, (u - 1) & 1, abort_flag, p)))
                            break;
                        ptx::mbar_arrive_expect_tx(v_full + s, L::kKVBytes);
                        for (int pn = 0; pn < L::kPanels; ++pn)
                            ptx::tma_load_4d(&tmV, v_full + s, smem + L::kVOff + s * L::kKVBytes + pn * L::kKVPanel,
                                             pn * 64, ge.h, ge.k0 + j * kBN, ge.b);
                        last_v[s] = u;
                    }
                }
                // Drain: every issued load has landed before the CTA can exit.
                for (int s = 0; s < L::kVStages; ++s)
                    if (last_v[s] >= 0)
                        wait_bar(v_full + s, last_v[s] & 1, abort_flag, p, false);
            }
        }
    } else {
        // ------------------------------------------------------------ softmax
        ptx::setmaxnreg_inc<kRegsSoftmax>();
        const int t = (warp - 4) >> 2;  // query tile
        const int quad = warp & 3;      // TMEM lane quadrant this warp may access
        const int row = quad * 32 + lane;
        const int prow = kHalves ? row : t * kBM + row;  // row inside the unit's query rows
        const bool tile_leader = ((warp - 4) & 3) == 0 && lane == 0;
        const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
        const uint32_t tS = tmem + lane_off + t * kBN;
        const uint32_t tO = tmem + lane_off + 2 * kBN + t * D;
        const float c = p.scale_log2;
        int g = 0, segi = 0, act = 0;
        int ph = 0;  // phase parities of merge_go (bit 0), seg_done (bit 1) and written_go (bit 2)
        bool ok = true;
        for (; ok; ++segi) {
            const unsigned char *mrow;
            int n, jb, k_len;
            int tix = -1;    // ticket merge: the unit of a piece of a split unit, else -1
            int ticket = 0;  // ticket merge: this piece's arrival ticket
            {
                Segment sg;
                if (!segment_at(p, cta, segi, sg))
                    break;
                if constexpr (kTicketMerge)
                    tix = sg.full ? -1 : sg.unit;
                Geom ge;
                unit_geom<kUnitRows>(p, sg.unit, ge);
                // the key mask is indexed by the key's global position: batch row, then k0 + offset
                mrow = p.mask ? p.mask + static_cast<size_t>(ge.b) * p.Sk + ge.k0 : nullptr;
                n = sg.je - sg.jb;
                jb = sg.jb;
                if constexpr (kHalves) {
                    // this slot's half of the unit's key blocks: [jb + t*nh, ...)
                    const int nh = (n + 1) / 2;
                    jb += t * nh;
                    n = t ? n - nh : nh;
                    if (n == 0 && t == 1)
                        continue;  // nothing for the second slot (at most one key block)
                }
                k_len = ge.k_len;
                if (n == 0) {
                    // query rows with no key at all (a packed document without keys): O = 0, LSE = -inf
                    const int qrow = ge.q0 + prow;
                    if (ge.q0 < ge.q_end && qrow < ge.q_end) {
                        uint4 *orow = out_row<D>(p, ge.b, ge.h, qrow);
#pragma unroll
                        for (int k = 0; k < D / 8; ++k)
                            orow[k] = make_uint4(0u, 0u, 0u, 0u);
                        if (p.lse)
                            p.lse[(static_cast<size_t>(ge.b) * p.H + ge.h) * p.Sq + qrow] = -INFINITY;
                    }
                    continue;
                }
            }
            float m_run = -INFINITY, l_run = 0.f;
            for (int i = 0; i < n; ++i) {
                const int kb = (jb + i) * kBN;  // key offset inside the unit's key range
                // validity of the block's keys, one bit per key, identical in every lane
                uint32_t vb[4];
                if (mrow) {
#pragma unroll
                    for (int w = 0; w < 4; ++w) {
                        const int key = kb + w * 32 + lane;
                        const bool v = key < k_len && mrow[key] != 0;
                        vb[w] = __ballot_sync(0xffffffffu, v);
                    }
                } else {
                    const int vn = k_len - kb;
#pragma unroll
                    for (int w = 0; w < 4; ++w) {
                        const int nn = vn - 32 * w;
                        vb[w] = nn >= 32 ? 0xffffffffu : (nn <= 0 ? 0u : ((1u << nn) - 1u));
                    }
                }
                const bool all_valid = (vb[0] & vb[1] & vb[2] & vb[3]) == 0xffffffffu;
                if constexpr (kTicketMerge) {
                    // A piece of a split unit takes its arrival ticket as its last
                    // key block starts: the atomic's round trip overlaps the block,
                    // and the pieces still arrive in about the order they finish.
                    if (i == n - 1 && tix >= 0 && tile_leader)
                        ticket = atomicAdd(p.counters + (static_cast<size_t>(tix) * kTiles + t) * 2, 1);
                }

                if (!(ok = wait_bar_warp(s_full + t, (g + i) & 1, abort_flag, p)))
                    break;
                ptx::tc_fence_after();
                // After a segment's first block the exps are taken against the
                // running maximum without computing the block maximum first;
                // the block's probability sum shows whether that was safe.
                // Every p is at most the sum, so a sum <= 2^15 keeps every p
                // (and the 16-bit P) in range; a larger sum (a maximum that
                // grew by about 2^8 or more) sends the block through the exact
                // path below: block maximum, conditional rescale of O, exps.
                // S is still intact then: the fast path stores P only after
                // the check.
                bool fast = i > 0 && __all_sync(0xffffffffu, m_run != -INFINITY);
                float l_blk = 0.f;
                if (fast) {
                    const uint64_t c2 = ptx::f2_pack(c, c), nm2 = ptx::f2_pack(-m_run, -m_run);
                    uint64_t sum2[4] = {0, 0, 0, 0};
                    uint32_t pk[kBN / 2];
                    {
                        uint32_t sh[kBN];
                        static_assert(kBN == 128, "one 128-column TMEM load per block");
                        ptx::tmem_ld128(tS, sh);
                        ptx::tmem_ld_wait();
                        ptx::reg_fence128(sh);
                        if (!all_valid) {
#pragma unroll
                            for (int k = 0; k < kBN; ++k)
                                if (!((vb[k >> 5] >> (k & 31)) & 1u))
                                    sh[k] = __float_as_uint(-INFINITY);
                        }
#pragma unroll
                        for (int k = 0; k < kBN / 2; ++k) {
                            const uint64_t arg = ptx::f2_fma(
                                ptx::f2_pack(__uint_as_float(sh[2 * k]), __uint_as_float(sh[2 * k + 1])), c2, nm2);
                            const float p0 = ptx::ex2_approx(ptx::f2_lo(arg));
                            const float p1 = ptx::ex2_approx(ptx::f2_hi(arg));
                            sum2[k & 3] = ptx::f2_add(sum2[k & 3], ptx::f2_pack(p0, p1));
                            pk[k] = ptx::pack2<BF16>(p0, p1);
                        }
                    }
                    const uint64_t sum01 = ptx::f2_add(sum2[0], sum2[1]), sum23 = ptx::f2_add(sum2[2], sum2[3]);
                    const uint64_t tot = ptx::f2_add(sum01, sum23);
                    l_blk = ptx::f2_lo(tot) + ptx::f2_hi(tot);
                    if (__any_sync(0xffffffffu, !(l_blk <= kFastSumLimit))) {
                        fast = false;
                    } else {
                        ptx::tmem_st64(tS, pk);
                    }
                }
                if (!fast) {
                    float mx;
                    {
                        uint32_t sr[kBN];
                        ptx::tmem_ld32(tS + 0, sr + 0);
                        ptx::tmem_ld32(tS + 32, sr + 32);
                        ptx::tmem_ld32(tS + 64, sr + 64);
                        ptx::tmem_ld32(tS + 96, sr + 96);
                        ptx::tmem_ld_wait();
                        ptx::reg_fence32(sr + 0);
                        ptx::reg_fence32(sr + 32);
                        ptx::reg_fence32(sr + 64);
                        ptx::reg_fence32(sr + 96);
                        float s[kBN];
#pragma unroll
                        for (int k = 0; k < kBN; ++k)
                            s[k] = __uint_as_float(sr[k]);
                        if (!all_valid) {
#pragma unroll
                            for (int k = 0; k < kBN; ++k)
                                if (!((vb[k >> 5] >> (k & 31)) & 1u))
                                    s[k] = -INFINITY;
                        }
                        float acc[8];
#pragma unroll
                        for (int k = 0; k < 8; ++k)
                            acc[k] = s[k];
#pragma unroll
                        for (int k = 8; k < kBN; k += 16) {
#pragma unroll
                            for (int q = 0; q < 8; ++q)
                                acc[q] = ptx::max3(acc[q], s[k + q], s[k + 8 + q]);
                        }
                        mx = ptx::max3(ptx::max3(acc[0], acc[1], acc[2]), ptx::max3(acc[3], acc[4], acc[5]),
                                       fmaxf(acc[6], acc[7]));
                    }
                    const float m_new = fmaxf(m_run, mx * c);
                    if (i == 0) {
                        m_run = m_new;
                    } else {
                        const bool need = m_new > m_run + kRescaleLog2;
                        if (__any_sync(0xffffffffu, need)) {
                            const float alpha = need ? ptx::ex2_approx(m_run - m_new) : 1.0f;
                            if (need) {
                                l_run *= alpha;
                                m_run = m_new;
                            }
#pragma unroll 1
                            for (int c0 = 0; c0 < D / 16; ++c0) {
                                uint32_t o[16];
                                ptx::tmem_ld16(tO + c0 * 16, o);
                                ptx::tmem_ld_wait();
                                ptx::reg_fence16(o);
#pragma unroll
                                for (int k = 0; k < 16; ++k)
                                    o[k] = __float_as_uint(__uint_as_float(o[k]) * alpha);
                                ptx::tmem_st16(tO + c0 * 16, o);
                            }
                            ptx::tmem_st_wait();
                        }
                    }
                    const float neg_m = (m_run == -INFINITY) ? 0.f : -m_run;
                    const uint64_t c2 = ptx::f2_pack(c, c), nm2 = ptx::f2_pack(neg_m, neg_m);
                    uint64_t sum2[4] = {0, 0, 0, 0};
#pragma unroll
                    for (int half = 0; half < 2; ++half) {
                        uint32_t sh[64];
                        ptx::tmem_ld32(tS + 64 * half, sh);
                        ptx::tmem_ld32(tS + 64 * half + 32, sh + 32);
                        ptx::tmem_ld_wait();
                        ptx::reg_fence32(sh);
                        ptx::reg_fence32(sh + 32);
                        if (!all_valid) {
#pragma unroll
                            for (int k = 0; k < 64; ++k)
                                if (!((vb[2 * half + (k >> 5)] >> (k & 31)) & 1u))
                                    sh[k] = __float_as_uint(-INFINITY);
                        }
                        uint32_t pk[32];
#pragma unroll
                        for (int k = 0; k < 32; ++k) {
                            const uint64_t arg = ptx::f2_fma(
                                ptx::f2_pack(__uint_as_float(sh[2 * k]), __uint_as_float(sh[2 * k + 1])), c2, nm2);
                            const float p0 = ptx::ex2_approx(ptx::f2_lo(arg));
                            const float p1 = ptx::ex2_approx(ptx::f2_hi(arg));
                            sum2[k & 3] = ptx::f2_add(sum2[k & 3], ptx::f2_pack(p0, p1));
                            pk[k] = ptx::pack2<BF16>(p0, p1);
                        }
                        ptx::tmem_st32(tS + 32 * half, pk);
                    }
                    const uint64_t t01 = ptx::f2_add(sum2[0], sum2[1]), t23 = ptx::f2_add(sum2[2], sum2[3]);
                    const uint64_t tot = ptx::f2_add(t01, t23);
                    l_blk = ptx::f2_lo(tot) + ptx::f2_hi(tot);
                }
                l_run += l_blk;
                ptx::tmem_st_wait();
                ptx::tc_fence_before();
                ptx::mbar_arrive(p_full + t);
            }
            if (!ok)
                break;
            if (!(ok = wait_bar_warp(o_full + t, act & 1, abort_flag, p)))
                break;
            ptx::tc_fence_after();
            Segment sg;
            segment_at(p, cta, opaque(segi), sg);
            Geom ge;
            unit_geom<kUnitRows>(p, sg.unit, ge);
            const int h = ge.h, b = ge.b;
            const int qrow = ge.q0 + prow;
            const int q_end = ge.q_end;
            if constexpr (kHalves) {
                // The second slot hands its rows' (m, l) to the first through its unused
                // staging area; the first merges the two halves by log-sum-exp with
                // both O read from TMEM (the same lanes, the second half's columns).
                float2 *const ml_half = reinterpret_cast<float2 *>(reinterpret_cast<uint8_t *>(bars) +
                                                                   (L::kEpiOff - L::kBarOff) + 4 * L::kEpiWarpBytes);
                if (t == 1) {
                    ml_half[row] = make_float2(m_run, l_run);
                    ptx::mbar_arrive(seg_done + 1);
                } else {
                    const int nb = sg.je - sg.jb;
                    const bool has1 = nb - (nb + 1) / 2 > 0;
                    float2 ml1 = make_float2(-INFINITY, 0.f);
                    if (has1) {
                        if (!(ok = wait_bar_warp(seg_done + 1, 0, abort_flag, p) &&
                                   wait_bar_warp(o_full + 1, 0, abort_flag, p)))
                            break;
                        ptx::tc_fence_after();
                        ml1 = ml_half[row];
                    }
                    const float M = fmaxf(m_run, ml1.x);
                    const float w0 = m_run == -INFINITY ? 0.f : ptx::ex2_approx(m_run - M);
                    const float w1 = ml1.x == -INFINITY ? 0.f : ptx::ex2_approx(ml1.x - M);
                    const float lsum = fmaf(w1, ml1.y, w0 * l_run);
                    const float inv = lsum > 0.f ? 1.0f / lsum : 0.f;
                    const unsigned long long orow =
                        qrow < q_end ? reinterpret_cast<unsigned long long>(out_row<D>(p, b, h, qrow)) : 0ull;
                    uint4 *const stg = reinterpret_cast<uint4 *>(reinterpret_cast<uint8_t *>(bars) +
                                                                 (L::kEpiOff - L::kBarOff) + (warp - 4) * L::kEpiWarpBytes);
#pragma unroll
                    for (int hf = 0; hf < D / 64; ++hf) {
#pragma unroll
                        for (int qq = 0; qq < 2; ++qq) {
                            uint32_t o[32];
                            ptx::tmem_ld32(tO + hf * 64 + qq * 32, o);
                            ptx::tmem_ld_wait();
                            ptx::reg_fence32(o);
                            float of[32];
#pragma unroll
                            for (int k = 0; k < 32; ++k)
                                of[k] = w0 * __uint_as_float(o[k]);
                            if (has1) {
                                ptx::tmem_ld32(tO + D + hf * 64 + qq * 32, o);
                                ptx::tmem_ld_wait();
                                ptx::reg_fence32(o);
#pragma unroll
                                for (int k = 0; k < 32; ++k)
                                    of[k] = fmaf(w1, __uint_as_float(o[k]), of[k]);
                            }
                            stage32<BF16>(stg, lane, qq, of, inv);
                        }
                        store_staged(stg, lane, orow, hf * 8);
                    }
                    if (p.lse && qrow < q_end)
                        p.lse[(static_cast<size_t>(b) * p.H + h) * p.Sq + qrow] =
                            lsum > 0.f ? (M + log2f(lsum)) * kLn2 : -INFINITY;
                }
            } else if (sg.full) {
                const float inv = l_run > 0.f ? 1.0f / l_run : 0.f;
                const float lse_val = l_run > 0.f ? (m_run + log2f(l_run)) * kLn2 : -INFINITY;
                // Each thread converts its own row into the warp's staging
                // area; the warp then stores 4 rows x 128 bytes per
                // instruction instead of 32 scattered 16-byte pieces.
                const unsigned long long orow =
                    qrow < q_end ? reinterpret_cast<unsigned long long>(out_row<D>(p, b, h, qrow)) : 0ull;
                uint4 *const stg = reinterpret_cast<uint4 *>(reinterpret_cast<uint8_t *>(bars) +
                                                             (L::kEpiOff - L::kBarOff) + (warp - 4) * L::kEpiWarpBytes);
#pragma unroll
                for (int hf = 0; hf < D / 64; ++hf) {
#pragma unroll
                    for (int qq = 0; qq < 2; ++qq) {
                        uint32_t o[32];
                        ptx::tmem_ld32(tO + hf * 64 + qq * 32, o);
                        ptx::tmem_ld_wait();
                        ptx::reg_fence32(o);
                        if (hf == D / 64 - 1 && qq == 1) {
                            ptx::tc_fence_before();
                            ptx::mbar_arrive(o_empty + t);  // O is in registers: the next PV may start
                        }
                        float of[32];
#pragma unroll
                        for (int k = 0; k < 32; ++k)
                            of[k] = __uint_as_float(o[k]);
                        stage32<BF16>(stg, lane, qq, of, inv);
                    }
                    store_staged(stg, lane, orow, hf * 8);
                }
                if (p.lse && qrow < q_end)
                    p.lse[(static_cast<size_t>(b) * p.H + h) * p.Sq + qrow] = lse_val;
            } else if constexpr (kTicketMerge) {
                // Partial segment (the unit is cut between CTAs). The tile's leader
                // took an arrival ticket as the last key block started. Every piece but
                // the last to arrive writes its unnormalised O and (m, l) to this
                // CTA's slot and then counts itself written; the last piece waits
                // for the others' writes and merges them by log-sum-exp with its
                // own O, read straight from TMEM (it never writes or re-reads it).
                const long long total = split_total(p);
                const long long first = sg.first;  // the unit's first iteration in the split order
                const int c_lo = tail_cta_of(p, total, first), c_hi = tail_cta_of(p, total, first + sg.nb - 1);
                int *const arrive = p.counters + (static_cast<size_t>(sg.unit) * kTiles + t) * 2;
                int *const written = arrive + 1;
                if (tile_leader) {
                    merge_flag[t] = (ticket == c_hi - c_lo);
                    ptx::mbar_arrive(merge_go + t);
                }
                if (!(ok = wait_bar_warp(merge_go + t, ph & 1, abort_flag, p)))
                    break;
                ph ^= 1;
                if (!merge_flag[t]) {
                    float4 *po = p.part_o + static_cast<size_t>(sg.slot) * (D / 4) * (kTiles * kBM) + prow;
#pragma unroll
                    for (int c0 = 0; c0 < D / 32; ++c0) {
                        uint32_t o[32];
                        ptx::tmem_ld32(tO + c0 * 32, o);
                        ptx::tmem_ld_wait();
                        ptx::reg_fence32(o);
#pragma unroll
                        for (int k = 0; k < 8; ++k)
                            __stcg(po + static_cast<size_t>(c0 * 8 + k) * (kTiles * kBM),
                                   make_float4(__uint_as_float(o[4 * k]), __uint_as_float(o[4 * k + 1]),
                                               __uint_as_float(o[4 * k + 2]), __uint_as_float(o[4 * k + 3])));
                    }
                    __stcg(p.part_ml + static_cast<size_t>(sg.slot) * (kTiles * kBM) + prow,
                           make_float2(m_run, l_run));
                    ptx::tc_fence_before();
                    ptx::mbar_arrive(o_empty + t);
                    __threadfence();
                    ptx::mbar_arrive(seg_done + t);
                    if (tile_leader && wait_bar(seg_done + t, (ph >> 1) & 1, abort_flag, p)) {
                        __threadfence();
                        atomicAdd(written, 1);
                    }
                    ph ^= 2;
                } else {
                    // Wait (bounded) until the other pieces' partials are written; the
                    // leader then releases the tile's threads through written_go.
                    if (tile_leader) {
                        const uint64_t t0 = ptx::globaltimer();
                        while (!*abort_flag) {
                            if (*reinterpret_cast<volatile int *>(written) == c_hi - c_lo) {
                                __threadfence();
                                break;
                            }
                            if (ptx::globaltimer() - t0 > p.wait_limit_ns) {
                                *abort_flag = 1;
                                atomicExch(p.status, kStatusTimeout);
                                break;
                            }
                            __nanosleep(64);
                        }
                        ptx::mbar_arrive(written_go + t);
                    }
                    if (!(ok = wait_bar_warp(written_go + t, (ph >> 2) & 1, abort_flag, p)) || *abort_flag) {
                        ok = false;
                        break;
                    }
                    ph ^= 4;
                    // Every piece in the unit's order (this one's values from registers
                    // and TMEM, the others' from their slots), folded and weighted by
                    // the same two functions on either path: the same arithmetic
                    // whichever piece arrives last, so results are reproducible.
                    float M = -INFINITY, lsum = 0.f;
                    // rows leave through the warp's staging area as whole 128-byte lines
                    const unsigned long long orow =
                        qrow < q_end ? reinterpret_cast<unsigned long long>(out_row<D>(p, b, h, qrow)) : 0ull;
                    uint4 *const stg = reinterpret_cast<uint4 *>(
                        reinterpret_cast<uint8_t *>(bars) + (L::kEpiOff - L::kBarOff) + (warp - 4) * L::kEpiWarpBytes);
                    const float2 mine = make_float2(m_run, l_run);
                    if (c_hi - c_lo == 1) {
                        // Two pieces (the usual cut): the other piece's (m, l) and its
                        // first 64 columns are fetched together, and each next 64
                        // columns while the current ones are stored; this piece's O is
                        // combined as it leaves TMEM.
                        const bool own_lo = cta == c_lo;
                        const int sl = tail_slot(p, total, first, own_lo ? c_hi : c_lo);
                        const float2 mo = __ldcg(p.part_ml + static_cast<size_t>(sl) * (kTiles * kBM) + prow);
                        const float4 *src = p.part_o + static_cast<size_t>(sl) * (D / 4) * (kTiles * kBM) + prow;
                        float4 vo[16];
#pragma unroll
                        for (int k = 0; k < 16; ++k)
                            vo[k] = __ldcg(src + static_cast<size_t>(k) * (kTiles * kBM));
                        fold_ml(M, lsum, own_lo ? mine : mo);
                        fold_ml(M, lsum, own_lo ? mo : mine);
                        const float w_own = piece_weight(mine, M), w_oth = piece_weight(mo, M);
                        const float w_lo = own_lo ? w_own : w_oth, w_hi = own_lo ? w_oth : w_own;
                        const float inv = lsum > 0.f ? 1.0f / lsum : 0.f;
#pragma unroll
                        for (int hf = 0; hf < D / 64; ++hf) {
#pragma unroll
                            for (int qq = 0; qq < 2; ++qq) {
                                uint32_t r[32];
                                ptx::tmem_ld32(tO + hf * 64 + qq * 32, r);
                                ptx::tmem_ld_wait();
                                ptx::reg_fence32(r);
                                if (hf == D / 64 - 1 && qq == 1) {
                                    ptx::tc_fence_before();
                                    ptx::mbar_arrive(o_empty + t);  // O is in registers: the next PV may start
                                }
                                float of[32];
#pragma unroll
                                for (int k = 0; k < 8; ++k) {
                                    const float4 x = vo[qq * 8 + k];
                                    const float xs[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
                                    for (int j = 0; j < 4; ++j) {
                                        const float a = __uint_as_float(r[4 * k + j]);
                                        of[4 * k + j] = add_piece(add_piece(0.f, w_lo, own_lo ? a : xs[j]), w_hi,
                                                                  own_lo ? xs[j] : a);
                                    }
                                }
                                stage32<BF16>(stg, lane, qq, of, inv);
                            }
                            if (hf + 1 < D / 64) {
#pragma unroll
                                for (int k = 0; k < 16; ++k)
                                    vo[k] = __ldcg(src + static_cast<size_t>((hf + 1) * 16 + k) * (kTiles * kBM));
                            }
                            store_staged(stg, lane, orow, hf * 8);
                        }
                    } else {
#pragma unroll 4
                        for (int cc = c_lo; cc <= c_hi; ++cc)
                            fold_ml(M, lsum,
                                    cc == cta ? mine
                                              : __ldcg(p.part_ml + static_cast<size_t>(tail_slot(p, total, first, cc)) *
                                                                       (kTiles * kBM) + prow));
                        const float inv = lsum > 0.f ? 1.0f / lsum : 0.f;
#pragma unroll 1
                        for (int hf = 0; hf < D / 64; ++hf) {
                            // 64 columns at a time: a slot's 16 float4 in flight together
                            // (one L2 round trip per piece), this piece's from TMEM
                            float o[64];
#pragma unroll
                            for (int k = 0; k < 64; ++k)
                                o[k] = 0.f;
                            for (int cc = c_lo; cc <= c_hi; ++cc) {
                                float2 ml;
                                float4 v[16];
                                if (cc == cta) {
                                    ml = mine;
                                    uint32_t r[64];
                                    ptx::tmem_ld32(tO + hf * 64, r);
                                    ptx::tmem_ld32(tO + hf * 64 + 32, r + 32);
                                    ptx::tmem_ld_wait();
                                    ptx::reg_fence32(r);
                                    ptx::reg_fence32(r + 32);
                                    if (hf == D / 64 - 1) {
                                        ptx::tc_fence_before();
                                        ptx::mbar_arrive(o_empty + t);  // O is in registers: the next PV may start
                                    }
#pragma unroll
                                    for (int k = 0; k < 16; ++k)
                                        v[k] = make_float4(__uint_as_float(r[4 * k]), __uint_as_float(r[4 * k + 1]),
                                                           __uint_as_float(r[4 * k + 2]), __uint_as_float(r[4 * k + 3]));
                                } else {
                                    const int sl = tail_slot(p, total, first, cc);
                                    ml = __ldcg(p.part_ml + static_cast<size_t>(sl) * (kTiles * kBM) + prow);
                                    const float4 *src =
                                        p.part_o + (static_cast<size_t>(sl) * (D / 4) + hf * 16) * (kTiles * kBM) + prow;
#pragma unroll
                                    for (int k = 0; k < 16; ++k)
                                        v[k] = __ldcg(src + static_cast<size_t>(k) * (kTiles * kBM));
                                }
                                const float w = piece_weight(ml, M);
#pragma unroll
                                for (int k = 0; k < 16; ++k) {
                                    o[4 * k] = add_piece(o[4 * k], w, v[k].x);
                                    o[4 * k + 1] = add_piece(o[4 * k + 1], w, v[k].y);
                                    o[4 * k + 2] = add_piece(o[4 * k + 2], w, v[k].z);
                                    o[4 * k + 3] = add_piece(o[4 * k + 3], w, v[k].w);
                                }
                            }
                            stage32<BF16>(stg, lane, 0, o, inv);
                            stage32<BF16>(stg, lane, 1, o + 32, inv);
                            store_staged(stg, lane, orow, hf * 8);
                        }
                    }
                    if (p.lse && qrow < q_end)
                        p.lse[(static_cast<size_t>(b) * p.H + h) * p.Sq + qrow] =
                            lsum > 0.f ? (M + log2f(lsum)) * kLn2 : -INFINITY;
                    if (tile_leader) {
                        *arrive = 0;  // every piece has arrived and written: leave the
                        *written = 0; // workspace zeroed for the next call
                    }
                }
            } else {
                // Partial segment: unnormalised O and (m, l) go to this CTA's slot.
                float4 *po = p.part_o + static_cast<size_t>(sg.slot) * (D / 4) * (kTiles * kBM) + prow;
#pragma unroll
                for (int c0 = 0; c0 < D / 32; ++c0) {
                    uint32_t o[32];
                    ptx::tmem_ld32(tO + c0 * 32, o);
                    ptx::tmem_ld_wait();
                    ptx::reg_fence32(o);
#pragma unroll
                    for (int k = 0; k < 8; ++k)
                        __stcg(po + static_cast<size_t>(c0 * 8 + k) * (kTiles * kBM),
                               make_float4(__uint_as_float(o[4 * k]), __uint_as_float(o[4 * k + 1]),
                                           __uint_as_float(o[4 * k + 2]), __uint_as_float(o[4 * k + 3])));
                }
                __stcg(p.part_ml + static_cast<size_t>(sg.slot) * (kTiles * kBM) + prow, make_float2(m_run, l_run));
                ptx::tc_fence_before();
                ptx::mbar_arrive(o_empty + t);
                __threadfence();
                ptx::mbar_arrive(seg_done + t);
                const long long total = split_total(p);
                const long long first = sg.first;  // the unit's first iteration in the split order
                const int c_lo = tail_cta_of(p, total, first), c_hi = tail_cta_of(p, total, first + sg.nb - 1);
                if (tile_leader) {
                    int last = 0;
                    if (wait_bar(seg_done + t, (ph >> 1) & 1, abort_flag, p)) {
                        int *cnt = p.counters + (static_cast<size_t>(sg.unit) * kTiles + t) * 2;
                        const int old = atomicAdd(cnt, 1);
                        last = (old == c_hi - c_lo);
                        if (last)
                            *cnt = 0;  // leave the workspace zeroed for the next call
                        __threadfence();
                    }
                    merge_flag[t] = last;
                    ptx::mbar_arrive(merge_go + t);
                }
                if (!(ok = wait_bar_warp(merge_go + t, ph & 1, abort_flag, p)))
                    break;
                ph ^= 3;  // merge_go and seg_done each took one phase
                if (merge_flag[t]) {
                    // Last segment of this unit to finish: combine every segment by log-sum-exp.
                    // running maximum and sum of the pieces' (m, l) in one pass
                    float M = -INFINITY, lsum = 0.f;
#pragma unroll 4
                    for (int cc = c_lo; cc <= c_hi; ++cc) {
                        const int sl = tail_slot(p, total, first, cc);
                        const float2 ml = __ldcg(p.part_ml + static_cast<size_t>(sl) * (kTiles * kBM) + prow);
                        if (ml.x == -INFINITY)
                            continue;
                        if (ml.x > M) {
                            lsum = (M == -INFINITY ? 0.f : lsum * ptx::ex2_approx(M - ml.x)) + ml.y;
                            M = ml.x;
                        } else {
                            lsum += ptx::ex2_approx(ml.x - M) * ml.y;
                        }
                    }
                    const float inv = lsum > 0.f ? 1.0f / lsum : 0.f;
                    // rows leave through the warp's staging area as whole 128-byte lines
                    const unsigned long long orow =
                        qrow < q_end ? reinterpret_cast<unsigned long long>(out_row<D>(p, b, h, qrow)) : 0ull;
                    uint4 *const stg = reinterpret_cast<uint4 *>(
                        reinterpret_cast<uint8_t *>(bars) + (L::kEpiOff - L::kBarOff) + (warp - 4) * L::kEpiWarpBytes);
#pragma unroll 1
                    for (int hf = 0; hf < D / 64; ++hf) {
                        // 64 columns at a time: all 16 float4 of a piece are in flight
                        // together, one L2 round trip per piece
                        float o[64];
#pragma unroll
                        for (int k = 0; k < 64; ++k)
                            o[k] = 0.f;
                        for (int cc = c_lo; cc <= c_hi; ++cc) {
                            const int sl = tail_slot(p, total, first, cc);
                            const float2 ml = __ldcg(p.part_ml + static_cast<size_t>(sl) * (kTiles * kBM) + prow);
                            const float4 *src =
                                p.part_o + (static_cast<size_t>(sl) * (D / 4) + hf * 16) * (kTiles * kBM) + prow;
                            float4 v[16];
#pragma unroll
                            for (int k = 0; k < 16; ++k)
                                v[k] = __ldcg(src + static_cast<size_t>(k) * (kTiles * kBM));
                            const float w = (ml.x == -INFINITY) ? 0.f : ptx::ex2_approx(ml.x - M);
#pragma unroll
                            for (int k = 0; k < 16; ++k) {
                                o[4 * k] += w * v[k].x;
                                o[4 * k + 1] += w * v[k].y;
                                o[4 * k + 2] += w * v[k].z;
                                o[4 * k + 3] += w * v[k].w;
                            }
                        }
                        stage32<BF16>(stg, lane, 0, o, inv);
                        stage32<BF16>(stg, lane, 1, o + 32, inv);
                        store_staged(stg, lane, orow, hf * 8);
                    }
                    if (p.lse && qrow < q_end)
                        p.lse[(static_cast<size_t>(b) * p.H + h) * p.Sq + qrow] =
                            lsum > 0.f ? (M + log2f(lsum)) * kLn2 : -INFINITY;
                }
            }
            g += n;
            ++act;
        }
    }

    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, kTmemCols);
    }
}

// A single block waiting on an mbarrier that nothing arrives on: exercises the
// bounded-wait failure path (status word set, clean return).
__global__ void selftest_wait_kernel(int *status, unsigned long long limit_ns)
{
    __shared__ __align__(8) uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        ptx::mbar_init(&bar, 1);
        abort_flag = 0;
        ptx::fence_mbar_init();
    }
    __syncthreads();
    Params p{};
    p.status = status;
    p.wait_limit_ns = limit_ns;
    wait_bar(&bar, 0, &abort_flag, p);
}

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    });
    return fn;
}

// [B, S, H, D] 16-bit tensor viewed as 4-D (d, h, s, b), 64 x 1 x 128 x 1 boxes.
cudaError_t make_map(CUtensorMap *m, const void *base, int B, int S, int H, int D, bool bf16)
{
    auto enc = tensor_map_encoder();
    if (!enc)
        return cudaErrorNotSupported;
    cuuint64_t dims[4] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(H), static_cast<cuuint64_t>(S),
                          static_cast<cuuint64_t>(B)};
    cuuint64_t strides[3] = {static_cast<cuuint64_t>(D) * 2, static_cast<cuuint64_t>(H) * D * 2,
                             static_cast<cuuint64_t>(S) * H * D * 2};
    cuuint32_t box[4] = {64, 1, 128, 1};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    CUresult r = enc(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 4,
                     const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                     CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

struct Schedule {
    int n_units, n_kblocks, grid, dp_waves;
    long long tail_iters;
    bool ticket_merge;  // merge split units with the ticket-first protocol
    bool halves;        // units of one 128-row tile, key range shared out between the CTA's two slots
};

// Calls whose CTAs each run at most this many key blocks (about 250 us at the
// kernel's rate) take the ticket-first merge: the merge that ends them is a
// large share of their time. Measured on GB300, same box, outputs bitwise
// equal: one Qwen-like rank (21 key blocks per CTA) 757 -> 803 TFLOP/s, the
// batched Qwen-like layer (86) 1254 -> 1284; one Wan-like 480p rank (323)
// 1644 -> 1614 and the batched 480p call 1658 -> 1619 with it, so those keep
// the write-then-count merge.
constexpr long long kTicketMergeMaxBlocks = 160;

// Work split for one call. Without a workspace every CTA takes one whole unit
// (grid = units). With one, a persistent grid of one CTA per SM runs whole-unit
// waves and then shares the key blocks of the remaining units evenly. Every
// piece of a split unit costs a partial store and a share of a merge, and
// every segment a pipeline start-up, so: when the units left over after the
// whole waves give each CTA at least kMinTailBlocks key blocks, only they are
// split; otherwise the last whole wave joins them (longer pieces). Measured on
// GB300: one rank of the Wan-like 480p layer (192 units of 256 blocks) 1429 ->
// 1584 TFLOP/s with the first rule; the Qwen-like call (384 units of 34
// blocks) is faster with the second.
constexpr long long kMinTailBlocks = 32;

// Cost of one halves-mode key-block step against a two-tile step, in
// percent. Measured on GB300 without a workspace: one Wan-like 480p rank
// (Q 4095 x K/V 32760, 12 heads: 512 -> 384 steps) 1.45 -> 1.54 us per step,
// 1108 -> 1391 TFLOP/s; Q 9450 x K/V 75600, 10 heads (1773 -> 1480 steps)
// 1.44 -> 1.51 us, 1435 -> 1637 TFLOP/s.
constexpr long long kHalvesStepCost = 107;

Schedule plan(int B, int Sq, int Sk, int H, int sms, bool split)
{
    Schedule s{};
    // packed varlen: B counts documents and Sq is the longest document;
    // callers have checked that the unit count fits in an int
    s.n_units = static_cast<int>(attention_units(B, Sq, H));
    s.n_kblocks = (Sk + kBN - 1) / kBN;
    if (!split) {
        // Without a workspace no unit can be cut between CTAs. When the last
        // wave of 256-row units leaves many SMs idle, 128-row units whose two
        // halves of the key range run side by side in one CTA (merged inside
        // it) end sooner: the makespan in key-block steps, waves x blocks, is
        // compared, the halves steps counted kHalvesStepCost times (two K/V
        // streams per CTA instead of one shared).
        const long long n_h = (static_cast<long long>(Sq) + kBM - 1) / kBM * H * B;  // 128-row units
        const long long steps_t = (s.n_units + sms - 1) / sms * static_cast<long long>(s.n_kblocks);
        const long long steps_h = (n_h + sms - 1) / sms * ((s.n_kblocks + 1) / 2);
        if (s.n_kblocks >= 2 && n_h <= INT_MAX && steps_h * kHalvesStepCost < steps_t * 100) {
            s.halves = true;
            s.n_units = static_cast<int>(n_h);
        }
        s.grid = s.n_units;
        s.dp_waves = 1;
        s.tail_iters = 0;
        return s;
    }
    const long long total = static_cast<long long>(s.n_units) * s.n_kblocks;
    s.grid = static_cast<int>(std::min<long long>(sms, total));
    const int waves = s.n_units / s.grid, rem = s.n_units % s.grid;
    if (rem == 0 || static_cast<long long>(rem) * s.n_kblocks >= kMinTailBlocks * s.grid)
        s.dp_waves = waves;
    else
        s.dp_waves = std::max(0, waves - 1);
    s.tail_iters = static_cast<long long>(s.n_units - s.dp_waves * s.grid) * s.n_kblocks;
    const long long per_cta = static_cast<long long>(s.dp_waves) * s.n_kblocks + (s.tail_iters + s.grid - 1) / s.grid;
    s.ticket_merge = per_cta <= kTicketMergeMaxBlocks;
    return s;
}

// Packed varlen: one unit per (query-tile pair of the longest document, head,
// document). Without a split every unit gets a CTA; with one, a persistent grid
// of one CTA per SM shares every key block of every unit evenly (the totals are
// known only on the device; the plan kernel writes them).
Schedule plan_varlen(int n_docs, int max_seqlen_q, int H, int sms, bool split)
{
    Schedule s{};
    const int n_qpairs = (max_seqlen_q + kTiles * kBM - 1) / (kTiles * kBM);
    s.n_units = n_qpairs * H * n_docs;
    s.n_kblocks = 0;  // per document
    s.grid = split ? sms : s.n_units;
    s.dp_waves = split ? 0 : 1;
    s.tail_iters = 0;
    return s;
}

long long ws_prefix_bytes(int n_docs)
{
    return ((static_cast<long long>(n_docs) + 1) * 8 + 255) / 256 * 256;
}

long long ws_counter_bytes(const Schedule &s)
{
    return (static_cast<long long>(s.n_units) * kTiles * 2 * 4 + 255) / 256 * 256;
}

long long ws_ml_bytes(const Schedule &s)
{
    return 2LL * s.grid * kTiles * kBM * 8;
}

long long ws_bytes(const Schedule &s, int D)
{
    return ws_counter_bytes(s) + ws_ml_bytes(s) + 2LL * s.grid * (D / 4) * kTiles * kBM * 16;
}

// Once per device and kernel instantiation: refuse a build whose register
// count differs from kRegsLaunch (the warpgroups' register budgets add up to
// the launch's total only then; a larger split would never be granted), and
// raise the kernel's dynamic shared memory limit.
template <int D, bool BF16, bool TM, bool HV>
cudaError_t prepare_kernel()
{
    static bool attr_set[64] = {false};
    static std::mutex mu;
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess)
        return err;
    std::lock_guard<std::mutex> g(mu);
    if (dev < 64 && attr_set[dev])
        return cudaSuccess;
    cudaFuncAttributes fa{};
    err = cudaFuncGetAttributes(&fa, attn_fwd_kernel<D, BF16, TM, HV>);
    if (err != cudaSuccess)
        return err;
    if (fa.numRegs != kRegsLaunch || fa.maxThreadsPerBlock < kThreads)
        return cudaErrorInvalidDeviceFunction;
    err = cudaFuncSetAttribute(attn_fwd_kernel<D, BF16, TM, HV>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               Layout<D, HV>::kAlloc);
    if (err != cudaSuccess)
        return err;
    if (dev < 64)
        attr_set[dev] = true;
    return cudaSuccess;
}

template <int D, bool BF16>
cudaError_t launch_typed(const AttnArgs &a, cudaStream_t stream)
{
    using L = Layout<D>;
    cudaError_t err = cudaSuccess;
    const int sms = sm_count(&err);
    if (err != cudaSuccess)
        return err;
    const bool varlen = a.cu_q != nullptr;
    // varlen: units are (256 rows of the longest document, head, document); without a
    // workspace one CTA per unit, with one every SM takes an equal share of all key blocks
    const bool vsplit = varlen && a.workspace != nullptr;
    const Schedule sc = varlen ? plan_varlen(a.n_docs, a.max_seqlen_q, a.H, sms, vsplit)
                               : plan(a.B, a.Sq, a.Sk, a.H, sms, a.workspace != nullptr);
    if (a.workspace && a.workspace_bytes < ws_bytes(sc, D) + (vsplit ? ws_prefix_bytes(a.n_docs) : 0))
        return cudaErrorInvalidValue;
    CUtensorMap mq, mk, mv;
    if ((err = make_map(&mq, a.q, a.B, a.Sq, a.H, D, BF16)) != cudaSuccess)
        return err;
    if ((err = make_map(&mk, a.k, a.B, a.Sk, a.H, D, BF16)) != cudaSuccess)
        return err;
    if ((err = make_map(&mv, a.v, a.B, a.Sk, a.H, D, BF16)) != cudaSuccess)
        return err;
    Params p{};
    p.mask = a.mask;
    p.out = a.out;
    p.lse = a.lse;
    p.B = a.B;
    p.Sq = a.Sq;
    p.Sk = a.Sk;
    p.H = a.H;
    const int unit_rows = sc.halves ? kBM : kTiles * kBM;
    p.n_qpairs = ((varlen ? a.max_seqlen_q : a.Sq) + unit_rows - 1) / unit_rows;
    p.n_kblocks = sc.n_kblocks;
    p.cu_q = a.cu_q;
    p.cu_k = a.cu_k;
    p.varlen = varlen ? 1 : 0;
    p.blk_s = a.blk_s;
    p.blk_u = a.blk_u;
    p.blk_b = a.blk_b;
    p.n_units = sc.n_units;
    p.grid = sc.grid;
    p.dp_waves = sc.dp_waves;
    p.tail_iters = sc.tail_iters;
    p.scale_log2 = a.scale * 1.4426950408889634f;
    p.status = device_status_word(stream, &err);
    if (err != cudaSuccess)
        return err;
    p.wait_limit_ns = kDefaultWaitLimitNs;
    p.n_docs = varlen ? a.n_docs : 0;
    if (a.workspace) {
        uint8_t *ws = static_cast<uint8_t *>(a.workspace);
        p.counters = reinterpret_cast<int *>(ws);
        p.part_ml = reinterpret_cast<float2 *>(ws + ws_counter_bytes(sc));
        p.part_o = reinterpret_cast<float4 *>(ws + ws_counter_bytes(sc) + ws_ml_bytes(sc));
    }
    if (vsplit) {
        long long *prefix = reinterpret_cast<long long *>(static_cast<uint8_t *>(a.workspace) + ws_bytes(sc, D));
        if ((err = launch_varlen_plan(a.cu_q, a.cu_k, a.n_docs, a.Sq, a.Sk, a.H, p.n_qpairs, prefix, a.out, a.lse, D,
                                      stream)) != cudaSuccess)
            return err;
        p.var_prefix = prefix;
    }
    if (sc.halves) {
        if ((err = prepare_kernel<D, BF16, false, true>()) != cudaSuccess)
            return err;
        attn_fwd_kernel<D, BF16, false, true>
            <<<static_cast<unsigned>(sc.grid), kThreads, Layout<D, true>::kAlloc, stream>>>(mq, mk, mv, p);
    } else if (sc.ticket_merge) {
        if ((err = prepare_kernel<D, BF16, true, false>()) != cudaSuccess)
            return err;
        attn_fwd_kernel<D, BF16, true, false><<<static_cast<unsigned>(sc.grid), kThreads, L::kAlloc, stream>>>(mq, mk,
                                                                                                                mv, p);
    } else {
        if ((err = prepare_kernel<D, BF16, false, false>()) != cudaSuccess)
            return err;
        attn_fwd_kernel<D, BF16, false, false><<<static_cast<unsigned>(sc.grid), kThreads, L::kAlloc, stream>>>(mq, mk,
                                                                                                                 mv, p);
    }
    return cudaGetLastError();
}

}  // namespace

long long varlen_workspace_size(int n_docs, int max_seqlen_q, int H, int D, cudaError_t *err)
{
    const int sms = sm_count(err);
    if (*err != cudaSuccess)
        return -1;
    const Schedule sc = plan_varlen(n_docs, max_seqlen_q, H, sms, true);
    return ws_bytes(sc, D) + ws_prefix_bytes(n_docs);
}

long long attention_units(int B, int Sq, int H)
{
    return (static_cast<long long>(Sq) + kTiles * kBM - 1) / (kTiles * kBM) * H * B;
}

long long attention_counter_bytes(int B, int Sq, int H)
{
    return (attention_units(B, Sq, H) * kTiles * 2 * 4 + 255) / 256 * 256;
}

long long attention_workspace_size(int B, int Sq, int Sk, int H, int D, cudaError_t *err)
{
    const int sms = sm_count(err);
    if (*err != cudaSuccess)
        return -1;
    return ws_bytes(plan(B, Sq, Sk, H, sms, true), D);
}

cudaError_t launch_attention(const AttnArgs &a, cudaStream_t stream)
{
    if (a.D == 128)
        return a.bf16 ? launch_typed<128, true>(a, stream) : launch_typed<128, false>(a, stream);
    if (a.D == 64)
        return a.bf16 ? launch_typed<64, true>(a, stream) : launch_typed<64, false>(a, stream);
    return cudaErrorInvalidValue;
}

cudaError_t launch_selftest_wait(unsigned long long limit_ns, cudaStream_t stream)
{
    cudaError_t err = cudaSuccess;
    int *status = device_status_word(stream, &err);
    if (err != cudaSuccess)
        return err;
    selftest_wait_kernel<<<1, 32, 0, stream>>>(status, limit_ns);
    return cudaGetLastError();
}

}  // namespace ctx
