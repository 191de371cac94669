/*
 * ctx.h — C ABI of libctx: the data-parallel hot path of context-parallel
 * diffusion-transformer attention on one GB300 (sm_103a).
 *
 * The path, in the order a rank runs it (vllm-omni PR #7641, "Compose Ulysses
 * with AllGather-KV as a 2D diffusion SP": Ulysses all-to-all in the U group,
 * K/V AllGather in the A group, local-Q / global-KV attention, reverse
 * Ulysses all-to-all):
 *
 *   ctx_pack_qkv     per-rank Q/K/V [B,S_l,H,D] -> destination-major staging
 *                    buffer [U,3,B,S_l,H/U,D] (sglang PR #33667,
 *                    pack_qkv_destination_major / _usp_input_all_to_all_qkv)
 *   ctx_sim_all_to_all   all_to_all_single chunk semantics between the
 *                    simulated ranks of one GPU (sglang PR #33667 unit test)
 *   ctx_unpack_qkv   received buffer -> [B,U*S_l,H/U,D] x3, written at a
 *                    caller-chosen row offset/stride so that K/V land in the
 *                    gathered global buffer (the AllGather placement)
 *   ctx_merge_joint_attn_mask   the key mask of the gathered layout from
 *                    the image and joint-text masks (missing side = valid)
 *   ctx_attn_lq_gkv  non-causal MHA of local queries against gathered keys,
 *                    optional per-key mask, scale, fp32 LSE
 *   ctx_pack_out / ctx_unpack_out   the reverse (output) exchange
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Every tensor pointer is a DEVICE pointer (cudaMalloc'd or managed memory);
 *    the library checks this and returns CTX_ERR_INVALID_ARG for host memory.
 *  - Tensors are dense, row-major, innermost dimension last, in the layouts
 *    written beside each argument. Element type is bf16 or fp16 (ctx_dtype);
 *    16-bit elements are moved bit for bit by the layout steps.
 *  - Every data pointer must be 16-byte aligned and D a multiple of 8 (rows a
 *    multiple of 16 bytes); otherwise CTX_ERR_MISALIGNED.
 *  - The caller owns every buffer, including the staging buffers; the library
 *    allocates nothing and keeps no state between calls.
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *    stream). Calls are asynchronous with respect to the host: CTX_OK means
 *    the work was validated and enqueued.
 *  - Arguments are validated on the host before anything is enqueued; a bad
 *    argument returns an error and enqueues nothing (fail closed: there is no
 *    fallback path).
 *  - Inputs and outputs of one call must occupy disjoint address ranges
 *    (CTX_ERR_ALIASING; the check is conservative: whole extents).
 *  - A failed launch returns CTX_ERR_CUDA; ctx_last_cuda_error() gives the
 *    cudaError_t of the last failure on the calling thread.
 *  - Device-side pipeline waits are bounded: a wait that runs out records
 *    CTX_ERR_TIMEOUT in a device status word and the kernel returns instead
 *    of hanging; ctx_device_status() reads and clears it.
 */
#ifndef CTX_H_
#define CTX_H_

#ifdef __cplusplus
extern "C" {
#endif

typedef enum ctx_status {
    CTX_OK = 0,
    CTX_ERR_INVALID_ARG = 1,  /* null pointer, non-positive size, bad shape, host pointer */
    CTX_ERR_UNSUPPORTED = 2,  /* valid request outside the supported set (e.g. D not 64/128) */
    CTX_ERR_MISALIGNED = 3,   /* pointer not 16-byte aligned or row not a multiple of 16 B */
    CTX_ERR_ALIASING = 4,     /* an output overlaps an input or another output */
    CTX_ERR_CUDA = 5,         /* a CUDA runtime / driver call failed */
    CTX_ERR_TIMEOUT = 6       /* a bounded device-side wait ran out */
} ctx_status;

typedef enum ctx_dtype { CTX_BF16 = 0, CTX_FP16 = 1 } ctx_dtype;

/* Staging layouts of the Ulysses exchange (destination-major either way). */
typedef enum ctx_layout {
    CTX_LAYOUT_TQKV = 0,        /* [U][3][B][S_l][h_l][D]: Q, K, V one after another */
    CTX_LAYOUT_INTERLEAVED = 1  /* [U][B][S_l][h_l][3*D]: Q|K|V per head (sglang PR #33667 excerpt) */
} ctx_layout;

/*
 * ctx_pack_qkv — Ulysses send-side relayout (sglang PR #33667, implementation
 * items 2-3 and the _usp_input_all_to_all_qkv excerpt: one kernel writes Q, K
 * and V destination-major into one staging buffer, replacing three
 * permute+contiguous copies).
 *
 *   staging[r][t][b][s][h][d] = X_t[b][s][r*h_l + h][d],  X_0,1,2 = q,k,v,
 *   h_l = H/U, r in [0,U)
 *
 * q, k, v  : [B, S_l, H, D] each, device, read only.
 * staging  : [U, 3, B, S_l, H/U, D], device, written in full. Chunk r (the
 *            r-th of U equal parts of the flat buffer) is what rank r must
 *            receive.
 * Errors   : INVALID_ARG if a size <= 0 or H % U != 0; MISALIGNED; ALIASING
 *            if staging overlaps q, k or v.
 */
ctx_status ctx_pack_qkv(const void *q, const void *k, const void *v, void *staging,
                        int B, int S_l, int H, int D, int U, ctx_dtype dtype,
                        void *stream);

/*
 * ctx_sim_all_to_all — all_to_all_single between simulated ranks on one GPU
 * (sglang PR #33667 unit test, _run_all_ranks: rank r's chunk j becomes rank
 * j's chunk r). It stands in for the NCCL collective of a multi-GPU
 * deployment: part of the single-GPU simulation, not of a rank's work.
 *
 * send : [G, U, U, chunk_bytes] bytes: group g, source rank r, chunk j.
 * recv : [G, U, U, chunk_bytes] bytes: group g, destination rank j, chunk r.
 *        recv[g][j][r] = send[g][r][j].
 * chunk_bytes must be a positive multiple of 16. Errors as above.
 */
ctx_status ctx_sim_all_to_all(const void *send, void *recv, int G, int U,
                              long long chunk_bytes, void *stream);

/*
 * ctx_unpack_qkv — Ulysses receive-side relayout (sglang PR #33667,
 * _usp_input_all_to_all_qkv excerpt: chunk r holds source rank r's rows,
 * which become rows [r*S_l, (r+1)*S_l) of the head-sharded sequence; batch
 * stays outermost).
 *
 *   X'_t[b][r*S_l + s][h][d] = recv[r][t][b][s][h][d]
 *
 * recv     : [U, 3, B, S_l, h_l, D], device, read only.
 * q        : output base; element (b, row, h, d) of Q' is at
 *            q + ((b*q_batch_stride_rows + row)*h_l + h)*D + d.
 * k, v     : output bases, same form with kv_batch_stride_rows.
 *            To place a rank's K/V straight into the gathered [B, Sk, h_l, D]
 *            buffer (the AllGather placement of vllm-omni PR #7641: A-group
 *            member a owns rows [a*S/A, (a+1)*S/A)), pass
 *            k = gathered_k + a*(U*S_l)*h_l*D and kv_batch_stride_rows = Sk.
 * q_batch_stride_rows, kv_batch_stride_rows : >= U*S_l.
 * Errors   : INVALID_ARG for bad sizes/strides; MISALIGNED; ALIASING if an
 *            output extent overlaps recv or another output.
 */
ctx_status ctx_unpack_qkv(const void *recv, void *q, void *k, void *v,
                          long long q_batch_stride_rows,
                          long long kv_batch_stride_rows, int B, int S_l,
                          int h_l, int D, int U, ctx_dtype dtype, void *stream);

/*
 * ctx_pack_qkv_ex — ctx_pack_qkv with uneven heads and a choice of layout.
 * Heads that do not divide by U are padded with zero heads to U*h_l,
 * h_l = ceil(H/U) (vllm-omni PR #7641, "advanced_uaa" head padding: 14 heads
 * at U=4 become 16, +14.3 % attention work); destination r gets padded heads
 * [r*h_l, (r+1)*h_l). layout selects CTX_LAYOUT_TQKV ([U,3,B,S_l,h_l,D], the
 * layout of ctx_pack_qkv) or CTX_LAYOUT_INTERLEAVED ([U,B,S_l,h_l,3D]).
 * q, k, v: [B, S_l, H, D]. Errors as ctx_pack_qkv (H % U is allowed).
 */
ctx_status ctx_pack_qkv_ex(const void *q, const void *k, const void *v,
                           void *staging, int B, int S_l, int H, int D, int U,
                           ctx_layout layout, ctx_dtype dtype, void *stream);

/*
 * ctx_unpack_qkv_ex — ctx_unpack_qkv for either staging layout; recv is
 * [U,3,B,S_l,h_l,D] (TQKV) or [U,B,S_l,h_l,3D] (INTERLEAVED). Outputs and
 * strides as ctx_unpack_qkv (h_l counts padded heads).
 */
ctx_status ctx_unpack_qkv_ex(const void *recv, void *q, void *k, void *v,
                             long long q_batch_stride_rows,
                             long long kv_batch_stride_rows, int B, int S_l,
                             int h_l, int D, int U, ctx_layout layout,
                             ctx_dtype dtype, void *stream);

/*
 * ctx_unpack_out_ex — ctx_unpack_out that drops padded heads: keeps the first
 * H of the U*h_l received heads (H <= U*h_l).
 *   y[b][s][r*h_l + h][d] = recv[r][b][s][h][d]   for r*h_l + h < H
 * recv : [U, B, S_l, h_l, D].   y : [B, S_l, H, D].
 */
ctx_status ctx_unpack_out_ex(const void *recv, void *y, int B, int S_l,
                             int h_l, int H, int D, int U, ctx_dtype dtype,
                             void *stream);

/*
 * ctx_merge_joint_attn_mask — the key mask of the gathered key layout
 * (vllm-omni PR #7641, follow-up review commit: after the K/V AllGather and
 * the re-attach of the joint text keys, one merge owns the 2-D key mask).
 * The gathered keys are S_img image keys and J joint keys, the joint segment
 * first (joint_front != 0) or last. For every batch row b and key position:
 *
 *   key_mask[b][p] = 1 if the key is valid, else 0; image key i is valid
 *   when image_mask is NULL or image_mask[b][i] != 0, joint key j when
 *   joint_mask is NULL or joint_mask[b][j] != 0 (a missing side is all valid).
 *
 * The result is the key_mask argument of ctx_attn_lq_gkv for the same keys.
 *
 * image_mask : NULL, or a byte mask (nonzero = attend) over the gathered
 *              global image keys whose shape is image_ndim sizes in the host
 *              array image_dims; it must be 2-D {B, S_img}.
 * joint_mask : NULL, or a byte mask of the joint keys, shape joint_ndim sizes
 *              in the host array joint_dims; it must be 2-D {B, J}. J is the
 *              length of the joint KEY tensor (a cached-K/V step without
 *              joint queries still has it).
 * key_mask   : [B, S_img + J] bytes, device, written in full (0/1). With
 *              both masks NULL every byte is 1, the same as passing no key
 *              mask to the attention.
 * Byte arrays have no alignment requirement. Checks, in this order (fail
 * closed, nothing enqueued): a joint mask that is not 2-D -> INVALID_ARG; a
 * 4-D image mask -> UNSUPPORTED (it has no key-mask form here, with or
 * without a joint mask); any other image rank but 2 -> INVALID_ARG; a joint
 * mask with J = 0 (no joint keys) -> INVALID_ARG; a mask whose dims are not
 * (B, its segment length) -> INVALID_ARG; key_mask overlapping an input ->
 * ALIASING; then the common checks.
 */
ctx_status ctx_merge_joint_attn_mask(const unsigned char *image_mask, int image_ndim,
                                     const long long *image_dims,
                                     const unsigned char *joint_mask, int joint_ndim,
                                     const long long *joint_dims, int B, int S_img,
                                     int J, int joint_front, unsigned char *key_mask,
                                     void *stream);

/*
 * ctx_attn_lq_gkv — local-Q / global-KV attention forward (vllm-omni PR
 * #7641: each rank attends its query slice against the gathered K/V as a
 * plain non-causal attention problem; ChituDiffusion "Fast CP" support
 * matrix: non-causal MHA, D=128). For every b, head h and query row i:
 *
 *   s_j = scale * <q[b,i,h,:], k[b,j,h,:]>   over keys j with key_mask[b,j] != 0
 *   out[b,i,h,:] = sum_j exp(s_j - m) v[b,j,h,:] / sum_j exp(s_j - m)
 *   lse[b,h,i]   = m + ln sum_j exp(s_j - m),   m = max_j s_j
 *
 * A row with no valid key gets out = 0 and lse = -inf.
 *
 * q        : [B, Sq, H, D], device.
 * k, v     : [B, Sk, H, D], device.
 * key_mask : NULL (all keys valid) or [B, Sk] bytes, nonzero = attend (the
 *            merged image + joint-text key mask; joint tokens may sit before
 *            or after the image keys).
 * scale    : softmax scale; NaN selects 1/sqrt(D). Otherwise finite and > 0.
 * out      : [B, Sq, H, D], device, same dtype as q.
 * lse      : NULL or [B, H, Sq] float32, device (natural log).
 * workspace, workspace_bytes :
 *            NULL / 0: no unit is split between CTAs. One CTA per (256 query
 *            rows, head, batch) unit, or, where that leaves a partial last
 *            wave on the SMs and it ends sooner, one CTA per (128 query rows,
 *            head, batch) unit whose two halves of the key range run side by
 *            side in the CTA and are merged inside it. Still slower than a
 *            workspace whenever the units do not fill the SMs evenly: on a
 *            152-SM GB300, one rank of a 480p video layer
 *            (Q [1,4095,12,128]) runs at about 0.85 of the balanced
 *            schedule's speed, and small calls (fewer units than SMs) leave
 *            SMs idle. Callers that can should pass a workspace (size from
 *            ctx_attn_lq_gkv_workspace_size; callers that cannot allocate
 *            have ctx_attn_lq_gkv_noalloc).
 *            Otherwise device memory of at least
 *            ctx_attn_lq_gkv_workspace_size(B, Sq, Sk, H, D) bytes, 256-byte
 *            aligned, filled with zeros before its first use: a persistent
 *            grid (one CTA per SM) runs whole-unit waves, then splits the key
 *            range of the leftover units evenly over all SMs and merges the
 *            pieces by log-sum-exp. A successful call leaves the workspace
 *            zeroed again; after CTX_ERR_TIMEOUT it must be re-zeroed. Calls
 *            that may run concurrently must not share a workspace.
 * D        : 64 or 128 (CTX_ERR_UNSUPPORTED otherwise).
 * Numerics : fp32 accumulation for QK^T, softmax and PV; the unnormalised
 *            probabilities exp(s_j - m') are taken against a running maximum
 *            m' (never more than 2^15, so they fit fp16) and rounded to the
 *            input dtype before the PV product; the final division by the
 *            row sum is exact up to fp32 rounding; out is rounded to nearest
 *            even. The two schedules agree up to that rounding of the
 *            probabilities (their running maxima differ where a key range
 *            is cut) and fp32 rounding of the merge.
 */
ctx_status ctx_attn_lq_gkv(const void *q, const void *k, const void *v,
                           const unsigned char *key_mask, float scale,
                           void *out, float *lse, void *workspace,
                           long long workspace_bytes, int B, int Sq, int Sk,
                           int H, int D, ctx_dtype dtype, void *stream);

/*
 * ctx_attn_lq_gkv_pack_out — ctx_attn_lq_gkv whose epilogue writes the output
 * directly in the send layout of the reverse Ulysses exchange (the output of
 * ctx_pack_out), saving one read and one write of O (the page's reverse
 * all-to-all after local-Q / global-KV attention; fusing it into the
 * epilogue is this library's choice).
 *
 * One rank: q is its local query [B_rank, U*S_l, h_l, D] (B = B_rank); send
 * is [U, B_rank, S_l, h_l, D]: send[r][b][s] = O[b][r*S_l + s].
 * Several ranks stacked as the simulation does (rank (a, u) holds query rows
 * [a*U*S_l, (a+1)*U*S_l) of batch block u, B = U'*B_rank, Sq = A*U*S_l):
 * send is [A][U'][U][B_rank][S_l][h_l][D], rank (a, u)'s send buffer at
 * [a][u]. lse keeps the plain [B, H, Sq] layout.
 * Errors: as ctx_attn_lq_gkv; INVALID_ARG unless Sq % (U*S_l) == 0,
 * B % B_rank == 0 and B / B_rank <= U.
 */
ctx_status ctx_attn_lq_gkv_pack_out(const void *q, const void *k, const void *v,
                                    const unsigned char *key_mask, float scale,
                                    void *send, float *lse, void *workspace,
                                    long long workspace_bytes, int B, int Sq,
                                    int Sk, int H, int D, int U, int B_rank,
                                    int S_l, ctx_dtype dtype, void *stream);

/*
 * ctx_attn_lq_gkv_workspace_size — bytes of workspace ctx_attn_lq_gkv needs
 * for its balanced schedule on the current device (it depends on the SM
 * count). Returns -1 for invalid sizes or when no device can be queried.
 */
long long ctx_attn_lq_gkv_workspace_size(int B, int Sq, int Sk, int H, int D);

/*
 * ctx_attn_lq_gkv_noalloc — ctx_attn_lq_gkv with the balanced schedule, for
 * callers that cannot allocate device memory (a host framework that owns
 * every buffer and passes only inputs and outputs, an embedding C program
 * with no device allocator, a path that must not let cudaMalloc synchronise
 * the device). The reference pages have no counterpart: it exists for this
 * library's callers.
 *
 * Same arguments, layouts and results as ctx_attn_lq_gkv, without the
 * workspace: the library keeps a fixed 44 MiB scratch array in device memory
 * (held by every GPU that loads the library until the process exits) and
 * allocates nothing on any call. The array's device address is looked up on
 * the current device by the calls made outside a stream capture (a device
 * reset can move it); make the first call on each device before any stream
 * capture. Calls share the array:
 * calls that can overlap on the GPU race and must be serialised by the
 * caller. The arrival counters are cleared after every call. Returns
 * CTX_ERR_INVALID_ARG for sizes ctx_attn_lq_gkv rejects, CTX_ERR_UNSUPPORTED
 * when the problem needs more scratch than 44 MiB (more than 131072 work
 * units of 256 query rows, or a grid of more than 160 SMs at D = 128).
 */
ctx_status ctx_attn_lq_gkv_noalloc(const void *q, const void *k, const void *v,
                                   const unsigned char *key_mask, float scale,
                                   void *out, float *lse, int B, int Sq, int Sk,
                                   int H, int D, ctx_dtype dtype, void *stream);

/*
 * ctx_pack_out — reverse Ulysses exchange, send side (sglang PR #33667,
 * _usp_output_all_to_all; vllm-omni PR #7641, reverse Ulysses all-to-all):
 * rows of the head-sharded output go back to the rank that owns them.
 *
 *   send[r][b][s][h][d] = o[b][r*S_l + s][h][d]
 *
 * o    : device; element (b, row, h, d) is at
 *        o + ((b*o_batch_stride_rows + row)*h_l + h)*D + d, row < U*S_l
 *        (a rank's rows inside a larger output buffer need no copy).
 * o_batch_stride_rows : >= U*S_l.
 * send : [U, B, S_l, h_l, D], device.
 */
ctx_status ctx_pack_out(const void *o, void *send, long long o_batch_stride_rows,
                        int B, int S_l, int h_l, int D, int U, ctx_dtype dtype,
                        void *stream);

/*
 * ctx_unpack_out — reverse Ulysses exchange, receive side: source rank r's
 * heads go back to heads [r*h_l, (r+1)*h_l) of the sequence-sharded output.
 *
 *   y[b][s][r*h_l + h][d] = recv[r][b][s][h][d]
 *
 * recv : [U, B, S_l, h_l, D], device.   y : [B, S_l, U*h_l, D], device.
 */
ctx_status ctx_unpack_out(const void *recv, void *y, int B, int S_l, int h_l,
                          int D, int U, ctx_dtype dtype, void *stream);

/*
 * ctx_lse_merge — combines attention results computed over P disjoint key
 * segments (ring / segmented K/V; the merge interface that consumes an LSE,
 * ChituDiffusion "Fast CP" page, Attention Planner notes). For every row:
 *
 *   lse[b,h,i]   = ln sum_p exp(lse_parts[p,b,h,i])
 *   out[b,i,h,:] = sum_p exp(lse_parts[p,b,h,i] - lse[b,h,i]) * o_parts[p,b,i,h,:]
 *
 * Segments with lse = -inf (no valid key) contribute nothing; a row whose
 * segments are all empty gets out = 0 and lse = -inf. The result equals
 * attention over all keys up to the rounding of the parts.
 *
 * o_parts   : [P, B, Sq, H, D] device, dtype (e.g. P outputs of ctx_attn_lq_gkv).
 * lse_parts : [P, B, H, Sq] float32 device (their LSEs).
 * out       : [B, Sq, H, D] device, dtype.   lse : NULL or [B, H, Sq] float32.
 * Arithmetic in fp32, out rounded to nearest even. D a multiple of 8.
 */
ctx_status ctx_lse_merge(const void *o_parts, const float *lse_parts, int P,
                         void *out, float *lse, int B, int Sq, int H, int D,
                         ctx_dtype dtype, void *stream);

/*
 * ctx_varlen_remap — packed varlen query metadata of one rank (vllm-omni PR
 * #7641, packed query metadata under AllGather-KV). Every global query
 * document [cu[d], cu[d+1]) is intersected with the rank's span
 * [span_begin, span_begin + span_len); the rank keeps exactly one (possibly
 * empty) entry per document, prefix-summed from 0, so its documents still
 * pair one to one with the global key boundaries (which stay unchanged).
 * Example from the page: documents [0,8,12] at A = 2 give [0,6,6] on rank 0
 * and [0,2,6] on rank 1. Computed on the device (no host synchronisation).
 *
 * cu_seqlens_q          : [n_docs + 1] int32 device, global query boundaries.
 * cu_seqlens_q_local    : [n_docs + 1] int32 device, written.
 * packed_padding        : NULL or [2] int32 device {real, pad} of a single
 *                         padded document; packed_padding_local (both or
 *                         neither) receives {local real, span_len - local
 *                         real}: the query length narrows to the rank's valid
 *                         prefix (the key length stays global).
 */
ctx_status ctx_varlen_remap(const int *cu_seqlens_q, int n_docs,
                            long long span_begin, long long span_len,
                            int *cu_seqlens_q_local, const int *packed_padding,
                            int *packed_padding_local, void *stream);

/*
 * ctx_attn_varlen — local-Q / global-KV attention over packed documents
 * (FlashAttention-varlen style metadata, vllm-omni PR #7641): query rows
 * [cu_seqlens_q[d], cu_seqlens_q[d+1]) attend keys
 * [cu_seqlens_k[d], cu_seqlens_k[d+1]) only; otherwise as ctx_attn_lq_gkv.
 * Query rows outside every document are not written; a document with query
 * rows but no keys gets out = 0 and lse = -inf.
 *
 * q            : [Sq, H, D] device (one packed sequence).
 * k, v         : [Sk, H, D] device.
 * cu_seqlens_q : [n_docs + 1] int32 device (local boundaries, e.g. from
 *                ctx_varlen_remap); cu_seqlens_k : [n_docs + 1] int32 device.
 *                Boundaries are clamped to [0, Sq] / [0, Sk] on the device.
 * max_seqlen_q : host int >= every document's query length (rows beyond it
 *                are not computed).
 * key_mask     : NULL or [Sk] bytes, nonzero = attend (global key index).
 * out          : [Sq, H, D]; lse : NULL or [H, Sq] float32.
 * workspace, workspace_bytes :
 *                NULL / 0: one CTA per (256 query rows, head, document) unit.
 *                Otherwise device memory of at least
 *                ctx_attn_varlen_workspace_size(n_docs, max_seqlen_q, H, D)
 *                bytes, 256-byte aligned, zero-filled before its first use: a
 *                small plan kernel counts every document's key blocks on the
 *                device, then a persistent grid (one CTA per SM) gives every SM
 *                an equal share of all key blocks, cutting units between SMs
 *                and merging the pieces by log-sum-exp (as ctx_attn_lq_gkv's
 *                balanced schedule). A successful call leaves the arrival
 *                counters zeroed; after CTX_ERR_TIMEOUT the workspace must be
 *                re-zeroed. Calls that may run concurrently must not share one.
 */
ctx_status ctx_attn_varlen(const void *q, const void *k, const void *v,
                           const int *cu_seqlens_q, const int *cu_seqlens_k,
                           int n_docs, int max_seqlen_q,
                           const unsigned char *key_mask, float scale,
                           void *out, float *lse, void *workspace,
                           long long workspace_bytes, int Sq, int Sk, int H,
                           int D, ctx_dtype dtype, void *stream);

/*
 * ctx_attn_varlen_workspace_size — bytes of workspace ctx_attn_varlen needs
 * for its balanced schedule on the current device (it depends on the SM
 * count, the number of documents and the longest document's query length).
 * Returns -1 for invalid sizes or when no device can be queried.
 */
long long ctx_attn_varlen_workspace_size(int n_docs, int max_seqlen_q, int H, int D);

/* Human-readable name of a status code (static storage, never NULL). */
const char *ctx_status_string(ctx_status status);

/*
 * ctx_device_status — synchronises `stream`, then reads and clears the
 * device status word of the current device. Returns CTX_OK, CTX_ERR_TIMEOUT
 * if a bounded device wait ran out since the last call, or CTX_ERR_CUDA if
 * the synchronisation failed.
 */
ctx_status ctx_device_status(void *stream);

/* cudaError_t of the last CTX_ERR_CUDA returned on the calling thread (0 if none). */
int ctx_last_cuda_error(void);

/*
 * ctx_selftest_wait_timeout — launches one block whose mbarrier wait can
 * never complete, bounded at `limit_ns` nanoseconds (1e3 .. 5e9), then
 * returns ctx_device_status(stream): CTX_ERR_TIMEOUT when the bounded wait
 * works as designed, with the context still usable. It tests the failure
 * path of the bounded waits without hanging or faulting a GPU.
 */
ctx_status ctx_selftest_wait_timeout(long long limit_ns, void *stream);

/* Library version as major*10000 + minor*100 + patch. */
int ctx_version(void);

#ifdef __cplusplus
}
#endif

#endif /* CTX_H_ */
