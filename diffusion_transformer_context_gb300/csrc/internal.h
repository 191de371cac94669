// Internal launcher interface between the C-ABI layer (api.cu) and the kernel
// translation units. Arguments reaching these functions are already validated.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace ctx {

// Device status codes written by kernels (same values as ctx_status).
constexpr int kStatusOk = 0;
constexpr int kStatusTimeout = 6;

// Bound for every device-side wait (nanoseconds of %globaltimer).
constexpr unsigned long long kDefaultWaitLimitNs = 2000000000ull;

// Attention work geometry shared by the kernel and the packed-varlen planner:
// a work unit is kAttnUnitRows query rows (two 128-row tiles) of one head,
// walked over its keys in blocks of kAttnKeyBlock.
constexpr int kAttnUnitRows = 256;
constexpr int kAttnKeyBlock = 128;

// Device address of a __device__ symbol on the current device. Outside a
// stream capture it is looked up on every call (a device reset reloads the
// module, possibly elsewhere) and remembered in slots[device]; while `stream`
// is capturing, the address of the last lookup on this device is used (none
// yet: cudaErrorStreamCaptureUnsupported), since a lookup may load the module.
cudaError_t device_symbol_address(const void *symbol, void **slots, cudaStream_t stream, void **out);

// Address of the current device's status word (see device_symbol_address).
int *device_status_word(cudaStream_t stream, cudaError_t *err);

// Number of SMs of the current device (cached per device).
int sm_count(cudaError_t *err);

enum class RelayoutMode : int {
    PackQKV = 0,
    UnpackQKV = 1,
    PackOut = 2,
    UnpackOut = 3,
    AllToAll = 4,
    PackQKVPad = 5,    // heads padded with zeros to U*h_l
    UnpackOutPad = 6,  // keeps the first H of the U*h_l heads
    PackInter = 7,     // interleaved staging [U][B][S_l][h_l][3][D] (cells of 3*D), heads padded
    UnpackInter = 8,   // interleaved staging back to Q', K', V'
};

// Every relayout step moves "runs": contiguous groups of 16-byte vectors that
// are contiguous in both source and destination. The mode maps a run index to
// its source and destination offsets.
struct RelayoutArgs {
    const void *src0;  // pack: q; otherwise the (only) source
    const void *src1;  // pack: k
    const void *src2;  // pack: v
    void *dst0;        // unpack: q'; otherwise the (only) destination
    void *dst1;        // unpack: k'
    void *dst2;        // unpack: v'
    long long n_runs;
    long long run_vec;  // 16-byte vectors per run
    // shape parameters (meaning depends on the mode)
    long long B, S_l, H, h_l, U, G;
    long long H_real;                // padded modes: heads that exist (< U*h_l)
    long long head_vec;              // interleaved modes: 16-byte vectors per head (D/8)
    long long q_batch_stride_rows;   // unpack: Q' batch stride; pack_out: O batch stride
    long long kv_batch_stride_rows;  // unpack: K'/V' batch stride
};

cudaError_t launch_relayout(RelayoutMode mode, const RelayoutArgs &a, cudaStream_t stream);

struct AttnArgs {
    const void *q, *k, *v;
    const unsigned char *mask;
    void *out;
    float *lse;
    int B, Sq, Sk, H, D;
    bool bf16;
    float scale;
    void *workspace;             // NULL: one CTA per work unit, no split
    long long workspace_bytes;
    const int *cu_q;             // packed varlen (B = 1): local query boundaries, NULL otherwise
    const int *cu_k;             // packed varlen: key boundaries
    int n_docs;
    int max_seqlen_q;
    int blk_s, blk_u, blk_b;     // > 0: write out in the reverse exchange's send layout
};

cudaError_t launch_attention(const AttnArgs &a, cudaStream_t stream);

// Bytes of workspace the balanced (split) schedule needs on the current device.
long long attention_workspace_size(int B, int Sq, int Sk, int H, int D, cudaError_t *err);

// Work units of a dense attention call (kAttnUnitRows query rows of one head
// and batch), in 64 bits; callers reject counts above INT_MAX.
long long attention_units(int B, int Sq, int H);

// Bytes at the head of the workspace that hold the arrival counters of the
// split units (zero between calls).
long long attention_counter_bytes(int B, int Sq, int H);

cudaError_t launch_selftest_wait(unsigned long long limit_ns, cudaStream_t stream);

struct LseMergeArgs {
    const void *o_parts;     // [P, B, Sq, H, D]
    const float *lse_parts;  // [P, B, H, Sq]
    int P;
    void *out;               // [B, Sq, H, D]
    float *lse;              // NULL or [B, H, Sq]
    int B, Sq, H, D;
    bool bf16;
};

cudaError_t launch_lse_merge(const LseMergeArgs &a, cudaStream_t stream);

cudaError_t launch_varlen_remap(const int *cu_g, int n_docs, long long lo, long long len, int *cu_l,
                                const int *pad_in, int *pad_out, cudaStream_t stream);

// Balanced packed varlen: per-document first split iteration into prefix[0..n_docs]
// and out = 0 / lse = -inf for query rows of documents without keys.
cudaError_t launch_varlen_plan(const int *cu_q, const int *cu_k, int n_docs, int Sq, int Sk, int H, int n_qpairs,
                               long long *prefix, void *out, float *lse, int D, cudaStream_t stream);

// Bytes of workspace the balanced packed-varlen attention needs on the current device.
long long varlen_workspace_size(int n_docs, int max_seqlen_q, int H, int D, cudaError_t *err);

// Key mask of the gathered layout: [B, S_img + J] bytes 0/1 from the optional
// image [B, S_img] and joint [B, J] masks (joint segment first when front).
cudaError_t launch_merge_mask(const unsigned char *img, const unsigned char *jnt, int B, int S_img, int J, int front,
                              unsigned char *out, cudaStream_t stream);

// Records a CUDA error for ctx_last_cuda_error() on the calling thread.
void record_cuda_error(cudaError_t e);

}  // namespace ctx
