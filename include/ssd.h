/*
 * ssd.h -- C-ABI of the GB300 (sm_103a) Mamba-2 / SSD mixer core.
 *
 * Three operations, each one call on a CUDA stream:
 *   ssd_conv1d_rows  causal depthwise conv1d + SiLU over [conv state ; rows]
 *   ssd_chunk_scan   the chunked SSD scan over S prefill rows (optionally with
 *                    the conv fused in front), with carried conv/SSM state
 *   ssd_decode_step  K recurrent steps (tokens) for R rows at slot-indexed
 *                    states, updated in place
 * and ssd_chunk_scan_varlen (the scan over packed sequences of different
 * lengths with slot-indexed states) and ssd_gated_group_rmsnorm (the group
 * RMSNorm + SiLU(z) gate that follows the scan in the mixer).
 *
 * Sources (page title, section):
 *   TensorRT-Model-Connect PR #2207 "perf(nemotron_h): prefill single-GPU
 *     prompts in multi-token chunks", "Implementation": the chunk form
 *     (a_t = dt_t A, gamma_t = cumulative sum of a, gamma_S taken from the
 *     last cumulative-sum element, every exponent clamped at <= 0, 128-row
 *     chunks) and add_short_conv_rows (conv over previous state plus chunk).
 *   TensorSharp "docs/models/nemotron.md", 4.1 "Mamba2 SSM layer": the
 *     single-step recurrence dA = exp(softplus(dt + dt_bias) A),
 *     state = dA state + dt x B, y = state . C + D x; section 3 "Forward
 *     graph": conv, SiLU, scan, gate; section 6: parameter shapes; section
 *     10/11: conv state of convKernel-1 rows, per-slot state pools.
 *   vllm.cpp PR #1362 "NemotronH decodes on the single-step recurrent
 *     kernels": the x | B | C split of the conv output, the head -> group map
 *     g = h / (H / G), and the in-place state update at the state slot.
 *
 * Conventions shared by every call:
 *   - Every data pointer is DEVICE memory owned by the caller; the library
 *     keeps no pointer after the call returns and allocates nothing.  The only
 *     state the library holds is one device error word per GPU (see
 *     ssd_read_device_error) and the fixed scratch array behind
 *     ssd_chunk_scan_static_ws.
 *   - Arrays are dense, row-major, contiguous, in the layouts stated below.
 *     Data pointers must be 16-byte aligned and the row lengths a multiple of
 *     16 bytes (Cdim * sizeof(act) and H * P * sizeof(act)); otherwise the
 *     call returns SSD_ERR_INVALID_ARG.
 *   - Calls are asynchronous on `stream`.  All argument checks run on the host
 *     before anything is launched; on any error nothing is launched and no
 *     memory is touched.
 *   - A = the per-head decay rate, stored NEGATIVE (decay exp(dt A) <= 1).
 *   - dt = softplus(dt_raw + dt_bias) when SSD_DT_SOFTPLUS is set, else dt_raw
 *     (dt_bias ignored).  softplus has no threshold.
 *   - Conv: tap k = W-1 multiplies the newest row; the conv state holds the
 *     W-1 most recent raw (pre-conv) rows, oldest first, in the activation
 *     dtype.
 *   - The SSM state is always fp32, layout [.., H, P, N] (N fastest).
 *   - With SSD_HAS_Z, y is multiplied by silu(z) (the gate alone).  The
 *     mixer's gated group RMSNorm is ssd_chunk_scan_gated_norm (scan, gate
 *     and norm in one call), or the scan without SSD_HAS_Z followed by
 *     ssd_gated_group_rmsnorm.
 */
#ifndef SSD_GB300_SSD_H
#define SSD_GB300_SSD_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#if defined(__GNUC__)
#define SSD_API __attribute__((visibility("default")))
#else
#define SSD_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    SSD_OK = 0,
    SSD_ERR_INVALID_ARG = 1,  /* null/misaligned pointer, bad size, bad flag   */
    SSD_ERR_UNSUPPORTED = 2,  /* valid problem that no kernel here implements  */
    SSD_ERR_CUDA = 3,         /* a CUDA runtime call failed (launch, query)     */
    SSD_ERR_BAD_SLOT = 4,     /* device error word: a slot id out of range      */
    SSD_ERR_TIMEOUT = 5,      /* device error word: a bounded wait ran out      */
    SSD_ERR_DUPLICATE_SLOT = 6 /* device error word: a slot id given twice in one
                                  call (reported only with
                                  SSD_CHECK_DISTINCT_SLOTS on)                */
} ssd_status;

typedef enum { SSD_F32 = 0, SSD_BF16 = 1 } ssd_dtype; /* activation dtype */

enum {
    SSD_DT_SOFTPLUS = 1u,  /* dt = softplus(dt_raw + dt_bias)                    */
    SSD_HAS_Z = 2u,        /* multiply y by silu(z)                              */
    SSD_GATED_NORM = 4u    /* workspace query of ssd_chunk_scan_gated_norm       */
};

/*
 * Problem dimensions.  Cdim = nheads*headdim + 2*ngroups*dstate is the width
 * of the x | B | C stream.  nheads % ngroups == 0.  conv_width W in [1, 8].
 * chunk: rows per chunk of the chunk form; 0 selects 128.  The bf16 path runs
 * 128-row chunks only (other values -> SSD_ERR_UNSUPPORTED); the fp32 path
 * is exact in any chunking and ignores it.
 */
typedef struct {
    int batch, seqlen, nheads, headdim, dstate, ngroups, conv_width, chunk;
} ssd_dims;

/*
 * ssd_conv1d_rows -- causal depthwise conv1d with SiLU over S rows.
 * (TensorRT-Model-Connect #2207 "Implementation", add_short_conv_rows;
 *  TensorSharp nemotron.md section 3, Conv1dStep + SiLU.)
 *
 *   u = [conv_state_in ; xbc_in]   (W-1+S rows per sequence)
 *   xbc_out[b,t,c] = silu(conv_b[c] + sum_k conv_w[c,k] * u[b,t+k,c])
 *   conv_state_out[b] = the last W-1 rows of u
 *
 * xbc_in          [B,S,Cdim] act   raw rows
 * conv_w          [Cdim,W]   fp32
 * conv_b          [Cdim]     fp32, or NULL (no bias)
 * conv_state_in   [B,W-1,Cdim] act, or NULL (zeros: a fresh sequence)
 * xbc_out         [B,S,Cdim] act   (must not overlap xbc_in)
 * conv_state_out  [B,W-1,Cdim] act, or NULL (not written); may alias
 *                 conv_state_in exactly
 * Only batch, seqlen, conv_width and Cdim (from nheads, headdim, dstate,
 * ngroups) of `dims` are used.  S = 0 is valid (the state is copied).
 */
SSD_API ssd_status ssd_conv1d_rows(const ssd_dims* dims, ssd_dtype act,
                           const void* xbc_in, const float* conv_w, const float* conv_b,
                           const void* conv_state_in, void* xbc_out, void* conv_state_out,
                           cudaStream_t stream);

/*
 * ssd_chunk_scan -- the SSD scan over S prefill rows per sequence.
 * (TensorRT-Model-Connect #2207 "Implementation": chunk form, gamma_S from
 *  the last cumulative-sum element, exponents clamped <= 0; TensorSharp
 *  nemotron.md 4.1: the recurrence it equals.)
 *
 * For each sequence b and head h (group g = h / (H/G)), rows t = 0..S-1:
 *   dt_t = softplus(dt[b,t,h] + dt_bias[h])            (flag SSD_DT_SOFTPLUS)
 *   state = exp(dt_t A[h]) state + dt_t x_t B_t^T       state [P,N]
 *   y[b,t,h,:] = state C_t + D[h] x_t   (times silu(z) with SSD_HAS_Z)
 * computed in 128-row chunks on the tensor cores (bf16, P=64, N=128, W<=4,
 * any row count) or exactly row by row (fp32 and other shapes).
 *
 * xbc             [B,S,Cdim] act: raw rows when conv_w != NULL (the conv of
 *                 ssd_conv1d_rows runs first), else already post-conv rows.
 *                 Columns: x [H*P] | B [G*N] | C [G*N].
 * conv_w, conv_b  as in ssd_conv1d_rows (conv_b may be NULL); conv_w NULL
 *                 means no conv (conv_state_* must then be NULL).
 * conv_state_in   [B,W-1,Cdim] act or NULL (zeros)
 * conv_state_out  [B,W-1,Cdim] act or NULL; may alias conv_state_in
 * dt              [B,S,H]  fp32 (raw dt before the bias/softplus)
 * dt_bias         [H] fp32 or NULL (zero)
 * A               [H] fp32 (negative)
 * D               [H] fp32 or NULL (no skip term)
 * z               [B,S,H*P] act; required iff SSD_HAS_Z
 * ssm_state_in    [B,H,P,N] fp32 or NULL (zeros: a fresh request)
 * y               [B,S,H,P] act
 * ssm_state_out   [B,H,P,N] fp32; may alias ssm_state_in exactly
 * workspace       device scratch of at least ssd_chunk_scan_workspace_size()
 *                 bytes (may be NULL when that size is 0); contents on entry
 *                 are ignored, on exit undefined.  Two calls in flight at the
 *                 same time must not share one workspace.
 *
 * Calls chain: feeding ssm_state_out / conv_state_out of one call into the
 * next call as *_in continues the same sequences (any split of the rows).
 */
SSD_API ssd_status ssd_chunk_scan(const ssd_dims* dims, ssd_dtype act, unsigned flags,
                          const void* xbc, const float* conv_w, const float* conv_b,
                          const void* conv_state_in, void* conv_state_out,
                          const float* dt, const float* dt_bias, const float* A,
                          const float* D, const void* z, const float* ssm_state_in,
                          void* y, float* ssm_state_out,
                          void* workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * Scratch bytes ssd_chunk_scan needs for these dims, activation dtype and
 * whether the conv is fused (conv_fused != 0 <=> conv_w != NULL).  With
 * SSD_GATED_NORM in flags: the scratch of ssd_chunk_scan_gated_norm instead.
 * Writes the size to *bytes.  Returns SSD_ERR_INVALID_ARG for invalid dims.
 */
SSD_API ssd_status ssd_chunk_scan_workspace_size(const ssd_dims* dims, ssd_dtype act, unsigned flags,
                                         int conv_fused, size_t* bytes);

/*
 * ssd_chunk_scan_gated_norm -- the mixer's tail in one call: the scan of
 * ssd_chunk_scan, then the gated group RMSNorm of ssd_gated_group_rmsnorm
 * over its output.
 * (TensorSharp nemotron.md section 3, Mamba2 branch: out = SiLU(z) *
 *  GroupRMSNorm(y, ssm_norm.weight); section 4.1: y is normalised per group
 *  before the gate; section 6: one weight per channel of H*P.)
 *
 *   y_ssm  = ssd_chunk_scan's y without the gate
 *   y[r,c] = silu(z[r,c]) * y_ssm[r,c] / sqrt(mean_{c' in group} y_ssm[r,c']^2
 *            + eps) * norm_w[c]
 * with G = dims->ngroups groups of H*P/G contiguous channels (the scan's
 * groups; each a whole number of heads).
 *
 * Arguments as ssd_chunk_scan's, and
 *   flags     SSD_DT_SOFTPLUS; SSD_HAS_Z and SSD_GATED_NORM are implied
 *   z         [B,S,H*P] act, required (rows > 0)
 *   norm_w    [H*P] fp32, 16-byte aligned, required
 *   eps       finite, >= 0
 *   workspace at least ssd_chunk_scan_workspace_size(dims, act,
 *             flags | SSD_GATED_NORM, conv_fused) bytes
 * On the tensor-core path the scan's epilogue applies the gate and leaves
 * each row's sum of y_ssm^2 per head in the workspace (fp32, before y is
 * rounded); a second kernel scales y in place by the weight and the group's
 * inverse norm.  Elsewhere (fp32, other shapes, norm groups whose
 * head count is not a multiple of 4) the scan runs without the gate and
 * ssd_gated_group_rmsnorm follows it in place.  Group channel count as in
 * ssd_gated_group_rmsnorm, else SSD_ERR_UNSUPPORTED; errors as
 * ssd_chunk_scan's.
 */
SSD_API ssd_status ssd_chunk_scan_gated_norm(const ssd_dims* dims, ssd_dtype act, unsigned flags,
                                     const void* xbc, const float* conv_w, const float* conv_b,
                                     const void* conv_state_in, void* conv_state_out,
                                     const float* dt, const float* dt_bias, const float* A,
                                     const float* D, const void* z, const float* norm_w,
                                     float eps, const float* ssm_state_in, void* y,
                                     float* ssm_state_out, void* workspace,
                                     size_t workspace_bytes, cudaStream_t stream);

/*
 * ssd_chunk_scan_static_ws -- ssd_chunk_scan for callers that cannot
 * allocate device memory.  None of the cited pages has a counterpart: this is a library
 * convenience, not a step of the method.
 *
 * Who needs it: code that runs inside a host program which owns every device
 * allocation (a plugin loaded into another runtime with its own pool), and
 * serving loops that must not call cudaMalloc on their hot path (it can
 * synchronise the whole device).  Such callers cannot provide the scratch
 * ssd_chunk_scan asks for.  This entry point takes the same arguments minus
 * the workspace and uses, as scratch, a fixed array of
 * SSD_STATIC_SCRATCH_BYTES that the library's device image holds on every
 * GPU that loads it, until the process exits.  It allocates nothing.
 *
 * Results equal ssd_chunk_scan's with a caller workspace: the same kernels
 * run.  Limits and rules:
 *   - Problems whose ssd_chunk_scan_workspace_size() exceeds
 *     SSD_STATIC_SCRATCH_BYTES return SSD_ERR_UNSUPPORTED before anything is
 *     launched (for the bf16 tensor-core path with the conv fused that size
 *     is batch * seqlen * 2 * ngroups * dstate * 2 bytes, so with dstate 128
 *     batch * seqlen * ngroups may be at most 32768).  This size check runs
 *     first, before the pointer checks of ssd_chunk_scan: a problem that is
 *     too large gets SSD_ERR_UNSUPPORTED even if a pointer is also bad.
 *   - The array used is the one of the CURRENT device (cudaGetDevice), which
 *     must be the device `stream` belongs to.
 *   - Nothing in the array has to start at zero: every call writes the
 *     scratch rows it reads before reading them.  The array keeps the last
 *     call's contents, which mean nothing to the next call.
 *   - All calls on a GPU share the one array.  Calls that can overlap on that
 *     GPU (different streams without ordering between them, or different
 *     host threads) race on it and give wrong results; order them on one
 *     stream, or use ssd_chunk_scan with a workspace per stream.
 *   - The first call made on a device (with that device current) looks up the
 *     array's device address there (cudaGetSymbolAddress) and caches it; make
 *     that first call before any stream capture on that device.
 */
#define SSD_STATIC_SCRATCH_BYTES ((size_t)16 << 20) /* 16 MiB per GPU */
SSD_API ssd_status ssd_chunk_scan_static_ws(const ssd_dims* dims, ssd_dtype act, unsigned flags,
                                    const void* xbc, const float* conv_w, const float* conv_b,
                                    const void* conv_state_in, void* conv_state_out,
                                    const float* dt, const float* dt_bias, const float* A,
                                    const float* D, const void* z, const float* ssm_state_in,
                                    void* y, float* ssm_state_out, cudaStream_t stream);

/*
 * ssd_chunk_scan_varlen -- the scan over sequences of different lengths packed
 * row after row, each continuing from (or, when fresh, replacing) the states
 * at its slot of the state pools, updated in place.
 * (vllm.cpp #1362 summary: the prefill half of a mixed batch runs the chunk
 *  scan over packed rows, states at the state index, has_initial_state for
 *  fresh requests, in place, no gather/scatter copies; TensorSharp
 *  nemotron.md section 11: per-slot conv + SSM state pools.)
 *
 * dims->batch = nseq sequences, dims->seqlen = T rows in all.  Sequence i is
 * rows cu_seqlens[i] .. cu_seqlens[i+1]-1 (cu_seqlens[0] = 0, non-decreasing,
 * cu_seqlens[nseq] = T; empty sequences allowed), s = slot_ids[i]:
 *   states in  = ssm_pool[s], conv_pool[s]   if has_initial_state[i] != 0
 *                zeros                       otherwise (a fresh request)
 *   the rows of sequence i as one ssd_chunk_scan call from those states
 *   ssm_pool[s], conv_pool[s] = the final states                  (in place)
 * The decode rows of a mixed batch go to ssd_decode_step on the same pools.
 *
 * cu_seqlens, slot_ids       [nseq+1], [nseq] int32, DEVICE memory; slot ids
 *                            distinct (checked only with
 *                            SSD_CHECK_DISTINCT_SLOTS on; else duplicates race)
 * has_initial_state          [nseq] int32 DEVICE memory, or NULL (all 1)
 * xbc [T,Cdim], dt [T,H], z [T,H*P], y [T,H,P]: packed rows, as the
 *   [B,S,..] arrays of ssd_chunk_scan with B = 1, S = T
 * conv_w, conv_b             as in ssd_chunk_scan (conv_w NULL: post-conv
 *                            rows, conv_pool and conv_b must be NULL)
 * conv_pool                  [num_slots,W-1,Cdim] act (required iff conv_w)
 * ssm_pool                   [num_slots,H,P,N] fp32
 * workspace                  at least T*2*G*N*2 bytes when conv_w != NULL
 * A sequence whose rows leave [0, T) or whose slot is outside [0, num_slots)
 * sets the device error word to SSD_ERR_BAD_SLOT and writes nothing (neither
 * pool nor y); the other sequences are unaffected.  Runs on the tensor-core
 * path only: bf16, P=64, N=128, W<=4, chunk 128 (else SSD_ERR_UNSUPPORTED).
 */
SSD_API ssd_status ssd_chunk_scan_varlen(const ssd_dims* dims, ssd_dtype act, unsigned flags,
                                 const int32_t* cu_seqlens, const int32_t* slot_ids,
                                 const int32_t* has_initial_state, int num_slots,
                                 const void* xbc, const float* conv_w, const float* conv_b,
                                 void* conv_pool, const float* dt, const float* dt_bias,
                                 const float* A, const float* D, const void* z,
                                 float* ssm_pool, void* y, void* workspace,
                                 size_t workspace_bytes, cudaStream_t stream);

/*
 * ssd_decode_step -- K recurrent steps (K = 1 .. 16 tokens of each request)
 * for R rows at slot-indexed states, in place.
 * (TensorSharp nemotron.md 4.1 and section 11 "Batched / paged forward":
 *  per-slot conv + SSM state pool; vllm.cpp #1362: the update runs in place
 *  at the state slot, no gather/scatter copies.)
 *
 * dims->batch = R rows, dims->seqlen = K tokens per row (1 <= K <= 16; more
 * gives SSD_ERR_UNSUPPORTED).  For row i, s = slot_ids[i], tokens t = 0..K-1
 * in order (each exactly one step of the recurrence):
 *   if conv_w != NULL:  u = [conv_pool[s] ; xbc[i,t]],  x|B|C = silu(conv(u)),
 *                       conv_pool[s] = last W-1 rows of u        (in place)
 *   else                x|B|C = xbc[i,t]
 *   ssm_pool[s,h] = exp(dt A[h]) ssm_pool[s,h] + dt x_h B_g^T     (in place)
 *   y[i,t,h,:] = ssm_pool[s,h] C_g + D[h] x_h   (times silu(z) with SSD_HAS_Z)
 * The state is read once and written once per call however many tokens it
 * carries: K tokens in one call cost about one step's memory traffic, and
 * give the same values as K calls of one token.
 *
 * xbc        [R,K,Cdim] act (raw when conv_w != NULL)
 * conv_pool  [num_slots,W-1,Cdim] act; required iff conv_w != NULL
 * dt         [R,K,H] fp32;  dt_bias, A, D as in ssd_chunk_scan; z [R,K,H*P]
 * slot_ids   [R] int32, DEVICE memory.  Ids must be distinct (checked only
 *            with SSD_CHECK_DISTINCT_SLOTS on; else duplicate ids race).
 *            An id outside [0, num_slots) sets the device error word to
 *            SSD_ERR_BAD_SLOT and that row writes nothing (neither pool nor
 *            y); other rows are unaffected.
 * ssm_pool   [num_slots,H,P,N] fp32, updated in place
 * y          [R,K,H,P] act
 */
SSD_API ssd_status ssd_decode_step(const ssd_dims* dims, ssd_dtype act, unsigned flags,
                           const void* xbc, const float* conv_w, const float* conv_b,
                           void* conv_pool, const float* dt, const float* dt_bias,
                           const float* A, const float* D, const void* z,
                           const int32_t* slot_ids, int num_slots, float* ssm_pool, void* y,
                           cudaStream_t stream);

/*
 * ssd_gated_group_rmsnorm -- group RMSNorm of y, then the SiLU(z) gate.
 * (TensorSharp nemotron.md section 3, Mamba2 branch:
 *  out = SiLU(z) * GroupRMSNorm(y, ssm_norm.weight); section 4.1: the group
 *  norm normalises y per group before the gate multiplies; section 6:
 *  ssm_norm.weight, one weight per channel of dInner = H*P.)
 *
 * For each of the B*S rows and each of the G = dims->ngroups groups of
 * gs = H*P/G contiguous channels:
 *   out[r,c] = silu(z[r,c]) * y[r,c] / sqrt(mean_{c' in group} y[r,c']^2 + eps)
 *              * weight[c]
 *
 * y       [B,S,H*P] act: the scan output computed WITHOUT SSD_HAS_Z
 * z       [B,S,H*P] act
 * weight  [H*P] fp32
 * eps     finite, >= 0 (the pages give no value; 1e-5 is the usual one)
 * out     [B,S,H*P] act; may alias y exactly (in place), no other overlap
 * Only batch, seqlen, nheads, headdim and ngroups of `dims` are used.  gs must
 * be a multiple of 8 (bf16) or 4 (fp32) channels, else SSD_ERR_UNSUPPORTED.
 * Rows are independent; S = 0 launches nothing.
 */
SSD_API ssd_status ssd_gated_group_rmsnorm(const ssd_dims* dims, ssd_dtype act, const void* y,
                                           const void* z, const float* weight, float eps,
                                           void* out, cudaStream_t stream);

/*
 * Sequence-parallel state passing: the rows of one sequence split into
 * consecutive segments (one per GPU), each scanned with ssd_chunk_scan.
 * (TensorRT-Model-Connect #2207 "Implementation": the chunk form, where
 * gamma of a chunk is the cumulative sum of a = dt A, its last element
 * carries the state to the next chunk, h <- exp(min(gamma_S, 0)) h + the
 * chunk's own terms, and every exponent is clamped at <= 0 -- applied here
 * with a whole segment in the role of the chunk.)
 *
 * Segment k scanned from a zero state (ssm_state_in NULL) ends in its own
 * contribution h_k; its total decay is Gamma_k = ssd_segment_decay over its
 * rows.  With h_in_0 the sequence's initial state,
 *   h_in_{k+1} = exp(min(Gamma_k, 0)) h_in_k + h_k      (ssd_state_combine)
 * is the state at the start of segment k+1, and h_in_K the final state.
 * Rescanning segment k from h_in_k (its conv state: the last W-1 raw rows
 * before it) gives exactly the y of one call over all rows.  The exchange
 * of (Gamma_k, h_k) between GPUs is the caller's (an all-gather);
 * ssd_scan_gb300.seqpar drives the whole sequence with torch.distributed.
 */

/*
 * ssd_segment_decay -- gamma[b,h] = sum_{t<S} dt[b,t,h] * A[h], with
 * dt = softplus(dt_raw + dt_bias) under SSD_DT_SOFTPLUS (else dt_raw), the
 * per-row products in fp32 and their sum in fp64, stored as fp32.
 * Uses batch, seqlen and nheads of `dims`; flags: SSD_DT_SOFTPLUS only.
 * dt [B,S,H] fp32, dt_bias [H] or NULL, A [H], gamma [B,H] fp32 (written).
 * S = 0 gives gamma = 0.
 */
SSD_API ssd_status ssd_segment_decay(const ssd_dims* dims, unsigned flags, const float* dt,
                                     const float* dt_bias, const float* A, float* gamma,
                                     cudaStream_t stream);

/*
 * ssd_state_combine -- h_out = exp(min(gamma, 0)) * h_prev + h_seg for every
 * (sequence, head): gamma [B,H] fp32, h_prev / h_seg / h_out [B,H,P,N] fp32
 * (16-byte aligned; P*N a multiple of 4).  h_prev NULL means zeros; h_out may
 * alias h_prev or h_seg exactly.  Uses batch, nheads, headdim, dstate.
 */
SSD_API ssd_status ssd_state_combine(const ssd_dims* dims, const float* gamma,
                                     const float* h_prev, const float* h_seg, float* h_out,
                                     cudaStream_t stream);

/*
 * Kernel-launch counters, for observability (which path ran, how many
 * kernels a call launched).  Host-side, process-wide, monotonically
 * increasing; one counter per kernel kind below.  Copies min(n,
 * SSD_KERNEL_KINDS) counters into out[] and returns SSD_KERNEL_KINDS.
 */
enum {
    SSD_KERNEL_CONV_ROWS = 0,      /* conv1d + SiLU over rows               */
    SSD_KERNEL_CONV_STATE = 1,     /* conv state = last W-1 raw rows        */
    SSD_KERNEL_SCAN_SIMT = 2,      /* fp32-pipe scan (exact row order)      */
    SSD_KERNEL_SCAN_TC = 3,        /* tensor-core chunk scan (bf16)         */
    SSD_KERNEL_BC_CONV = 4,        /* conv of the B|C columns for the scan  */
    SSD_KERNEL_DECODE_STEP = 5,    /* slot-indexed decode step              */
    SSD_KERNEL_DECODE_CONV = 6,    /* conv-pool roll of the decode step     */
    SSD_KERNEL_GATED_NORM = 7,     /* group RMSNorm + SiLU(z) gate          */
    SSD_KERNEL_SEGMENT_DECAY = 8,  /* a segment's total decay               */
    SSD_KERNEL_STATE_COMBINE = 9,  /* state after two consecutive segments  */
    SSD_KERNEL_NORM_SCALE = 10,    /* fused gated norm: y times 1/rms       */
    SSD_KERNEL_KINDS = 11
};
SSD_API int ssd_launch_counts(uint64_t* out, int n);

/*
 * Debug checks (process-wide, off by default; they cost time on every call).
 * SSD_CHECK_DISTINCT_SLOTS: ssd_decode_step and ssd_chunk_scan_varlen check
 * on the device that no slot id appears twice in one call (the slot-id rule
 * of both entry points).  A row (decode) or sequence (varlen) whose slot id
 * already appeared at an earlier index sets SSD_ERR_DUPLICATE_SLOT in the
 * device error word and writes nothing (neither pool nor y); the earlier
 * occurrence runs normally, so the pools stay consistent.  Without the check
 * duplicate ids race.  Returns the flags that were set before.
 */
enum { SSD_CHECK_DISTINCT_SLOTS = 1u };
SSD_API unsigned ssd_set_debug_checks(unsigned flags);

/*
 * Bound, in nanoseconds, on each wait between the warps of the tensor-core
 * scan kernel (ssd_chunk_scan / ssd_chunk_scan_varlen / _static_ws on the
 * tensor-core path).  A wait that runs out ends the kernel early: the
 * outputs of that call are undefined and the device error word reports
 * SSD_ERR_TIMEOUT; the context stays usable (no trap).  Default 2 s, which
 * no healthy call comes near; 0 restores the default.  The kernel's final
 * waits for its own copies and tensor-core work in flight keep the 2 s bound
 * whatever this is.  Meant for failure-detection tests and watchdogs; it is
 * process-wide and read at each launch.  Returns the previous bound.
 */
SSD_API uint64_t ssd_set_wait_limit_ns(uint64_t ns);

/* Static text for a status code (never NULL). */
SSD_API const char* ssd_status_string(ssd_status status);

/*
 * Synchronises `stream`, then returns and clears the device error word of the
 * current device: SSD_OK, or SSD_ERR_BAD_SLOT, SSD_ERR_DUPLICATE_SLOT,
 * SSD_ERR_TIMEOUT (the first of these, in this order, among the kinds
 * recorded since the last read), or SSD_ERR_CUDA if a CUDA call failed.
 */
SSD_API ssd_status ssd_read_device_error(cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* SSD_GB300_SSD_H */
