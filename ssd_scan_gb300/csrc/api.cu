// api.cu -- the C-ABI of include/ssd.h: argument checks, dispatch, the
// per-device error word.  Every check runs before any launch; on error the
// call returns without touching device memory.
#include "../../include/ssd.h"
#include "internal.cuh"

#include <stdint.h>

#include <atomic>
#include <mutex>

namespace {

using namespace ssd;

// One error word per device (each device that loads the module has its own
// copy).  Kernels receive its address; ssd_read_device_error reads & clears.
__device__ unsigned g_ssd_error_word;

constexpr int kMaxDevices = 64;
unsigned* g_err_addr[kMaxDevices];  // host cache of each device's symbol address
std::mutex g_err_mutex;             // first calls on a device from several threads

// process-wide settings read at every launch (ssd_set_debug_checks,
// ssd_set_wait_limit_ns)
std::atomic<unsigned> g_debug_checks{0};
std::atomic<uint64_t> g_wait_ns{0};  // 0: the kernel's default

ssd_status error_word_address(unsigned** out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return SSD_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_err_mutex);
    if (g_err_addr[dev] == nullptr) {
        void* ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_ssd_error_word) != cudaSuccess) return SSD_ERR_CUDA;
        g_err_addr[dev] = static_cast<unsigned*>(ptr);
    }
    *out = g_err_addr[dev];
    return SSD_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

// Checks common to all calls.  Cdim is written on success.
ssd_status check_dims(const ssd_dims* d, ssd_dtype act, long long* cdim)
{
    if (d == nullptr) return SSD_ERR_INVALID_ARG;
    if (act != SSD_F32 && act != SSD_BF16) return SSD_ERR_INVALID_ARG;
    if (d->batch < 0 || d->seqlen < 0 || d->nheads <= 0 || d->headdim <= 0 || d->dstate <= 0 ||
        d->ngroups <= 0 || d->nheads % d->ngroups != 0 || d->conv_width < 1 ||
        d->conv_width > 8 || d->chunk < 0)
        return SSD_ERR_INVALID_ARG;
    const long long c = (long long)d->nheads * d->headdim + 2LL * d->ngroups * d->dstate;
    if (c > (1LL << 30)) return SSD_ERR_INVALID_ARG;
    const long long esize = act == SSD_BF16 ? 2 : 4;
    if ((c * esize) % 16 != 0) return SSD_ERR_INVALID_ARG;
    // every flat index used by the kernels fits in 63 bits
    const long long rows = (long long)d->batch * d->seqlen;
    if (rows > 0 && c > (1LL << 62) / rows) return SSD_ERR_INVALID_ARG;
    *cdim = c;
    return SSD_OK;
}

ssd_status from_cuda(cudaError_t e) { return e == cudaSuccess ? SSD_OK : SSD_ERR_CUDA; }

// The tensor-core chunk scan serves bf16 with P = 64, N = 128, W <= 4 and
// 128-row chunks; everything else runs on the row-exact fp32-pipe kernel.
// Calls of at most SSD_SHORT_CALL_ROWS rows per sequence would take the
// row-exact kernel even in bf16.  Measured (us per call, tensor cores / row
// kernel): 4 sequences x 128 heads, 1 row 26.7 / 24.6, 2 rows 26.7 / 26.7,
// 4 rows 26.6 / 32.8; 1 sequence, 1 row 12.4 / 16.5.  Calls of up to 128
// rows walk several units per CTA on the tensor cores, so none goes to the
// row kernel.
#ifndef SSD_SHORT_CALL_ROWS
#define SSD_SHORT_CALL_ROWS 0
#endif

bool use_tensor_cores(const ssd_dims* d, ssd_dtype act)
{
    const int chunk = d->chunk == 0 ? 128 : d->chunk;
    return act == SSD_BF16 && chunk == 128 && scan_tc_supports(d->headdim, d->dstate) &&
           d->conv_width <= 4 && d->seqlen > SSD_SHORT_CALL_ROWS;
}

// Scratch of the tensor-core path with the conv fused: the post-conv B|C
// columns of every row, [B, S, 2*G*N] bf16.
size_t tc_workspace_bytes(const ssd_dims* d)
{
    const size_t n = (size_t)d->batch * d->seqlen * 2 * d->ngroups * d->dstate * 2;
    return (n + 255) & ~(size_t)255;
}

// Scratch of the fused gated norm on the tensor-core path: each row's sum of
// y^2 per head, [B, H, S] fp32, after the B|C scratch.
size_t norm_ss_bytes(const ssd_dims* d)
{
    const size_t n = (size_t)d->batch * d->nheads * d->seqlen * 4;
    return (n + 255) & ~(size_t)255;
}

std::atomic<uint64_t> g_launches[SSD_KERNEL_KINDS];

// Records one launch of `kind` when it succeeded (kernels that a launcher
// skips for empty work are not launched and not counted).
ssd_status counted(cudaError_t e, int kind, bool launched = true)
{
    if (e == cudaSuccess && launched) g_launches[kind].fetch_add(1, std::memory_order_relaxed);
    return from_cuda(e);
}

}  // namespace

extern "C" {

unsigned ssd_set_debug_checks(unsigned flags)
{
    return g_debug_checks.exchange(flags & SSD_CHECK_DISTINCT_SLOTS);
}

uint64_t ssd_set_wait_limit_ns(uint64_t ns) { return g_wait_ns.exchange(ns); }

int ssd_launch_counts(uint64_t* out, int n)
{
    for (int i = 0; out != nullptr && i < n && i < SSD_KERNEL_KINDS; ++i)
        out[i] = g_launches[i].load(std::memory_order_relaxed);
    return SSD_KERNEL_KINDS;
}

const char* ssd_status_string(ssd_status s)
{
    switch (s) {
        case SSD_OK: return "ok";
        case SSD_ERR_INVALID_ARG: return "invalid argument";
        case SSD_ERR_UNSUPPORTED: return "unsupported problem shape or dtype";
        case SSD_ERR_CUDA: return "CUDA runtime error";
        case SSD_ERR_BAD_SLOT: return "slot id out of range (device)";
        case SSD_ERR_TIMEOUT: return "bounded device wait ran out (device)";
        case SSD_ERR_DUPLICATE_SLOT: return "slot id given twice in one call (device)";
    }
    return "unknown status";
}

ssd_status ssd_read_device_error(cudaStream_t stream)
{
    unsigned* addr = nullptr;
    if (error_word_address(&addr) != SSD_OK) return SSD_ERR_CUDA;
    if (cudaStreamSynchronize(stream) != cudaSuccess) return SSD_ERR_CUDA;
    unsigned v = 0;
    if (cudaMemcpy(&v, addr, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess) return SSD_ERR_CUDA;
    const unsigned zero = 0;
    if (cudaMemcpy(addr, &zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess)
        return SSD_ERR_CUDA;
    if (v & kErrBadSlot) return SSD_ERR_BAD_SLOT;
    if (v & kErrDupSlot) return SSD_ERR_DUPLICATE_SLOT;
    if (v & kErrTimeout) return SSD_ERR_TIMEOUT;
    return SSD_OK;
}

ssd_status ssd_conv1d_rows(const ssd_dims* dims, ssd_dtype act, const void* xbc_in,
                           const float* conv_w, const float* conv_b, const void* conv_state_in,
                           void* xbc_out, void* conv_state_out, cudaStream_t stream)
{
    long long cdim = 0;
    ssd_status s = check_dims(dims, act, &cdim);
    if (s != SSD_OK) return s;
    const bool any_rows = dims->batch > 0 && dims->seqlen > 0;
    if (conv_w == nullptr || !aligned4(conv_w) || (conv_b && !aligned4(conv_b)))
        return SSD_ERR_INVALID_ARG;
    if (any_rows && (xbc_in == nullptr || xbc_out == nullptr || !aligned16(xbc_in) ||
                     !aligned16(xbc_out) || xbc_in == xbc_out))
        return SSD_ERR_INVALID_ARG;
    if ((conv_state_in && !aligned16(conv_state_in)) ||
        (conv_state_out && !aligned16(conv_state_out)))
        return SSD_ERR_INVALID_ARG;
    if (dims->batch == 0) return SSD_OK;
    ConvParams p{dims->batch, dims->seqlen, (int)cdim, dims->conv_width,
                 xbc_in, conv_w, conv_b, conv_state_in, xbc_out, conv_state_out};
    const bool bf16 = act == SSD_BF16;
    s = counted(launch_conv1d_rows(p, bf16, stream), SSD_KERNEL_CONV_ROWS,
                dims->seqlen > 0);
    if (s != SSD_OK) return s;
    return counted(launch_conv_state(p, bf16, stream), SSD_KERNEL_CONV_STATE,
                   conv_state_out != nullptr && dims->conv_width > 1);
}

ssd_status ssd_chunk_scan_workspace_size(const ssd_dims* dims, ssd_dtype act, unsigned flags,
                                         int conv_fused, size_t* bytes)
{
    long long cdim = 0;
    if (bytes == nullptr) return SSD_ERR_INVALID_ARG;
    ssd_status s = check_dims(dims, act, &cdim);
    if (s != SSD_OK) return s;
    if (flags & ~(unsigned)(SSD_DT_SOFTPLUS | SSD_HAS_Z | SSD_GATED_NORM)) return SSD_ERR_INVALID_ARG;
    const bool tc = use_tensor_cores(dims, act);
    *bytes = (conv_fused && tc) ? tc_workspace_bytes(dims) : 0;
    if ((flags & SSD_GATED_NORM) && tc && norm_scale_supports(dims->nheads, dims->ngroups))
        *bytes += norm_ss_bytes(dims);
    return SSD_OK;
}

}  // extern "C"

namespace {

// ssd_chunk_scan, and with norm_w != NULL ssd_chunk_scan_gated_norm (the
// gate implied; flags then without SSD_HAS_Z and SSD_GATED_NORM).
ssd_status chunk_scan_impl(const ssd_dims* dims, ssd_dtype act, unsigned flags, const void* xbc,
                           const float* conv_w, const float* conv_b, const void* conv_state_in,
                           void* conv_state_out, const float* dt, const float* dt_bias,
                           const float* A, const float* D, const void* z,
                           const float* ssm_state_in, void* y, float* ssm_state_out,
                           void* workspace, size_t workspace_bytes, cudaStream_t stream,
                           const float* norm_w, float eps)
{
    long long cdim = 0;
    ssd_status s = check_dims(dims, act, &cdim);
    if (s != SSD_OK) return s;
    if (flags & ~(unsigned)(SSD_DT_SOFTPLUS | SSD_HAS_Z)) return SSD_ERR_INVALID_ARG;
    const bool norm = norm_w != nullptr;
    const bool rows = dims->batch > 0 && dims->seqlen > 0;
    const bool has_z = norm || (flags & SSD_HAS_Z) != 0;
    if (rows && (xbc == nullptr || dt == nullptr || y == nullptr || !aligned16(xbc) ||
                 !aligned16(y) || !aligned4(dt)))
        return SSD_ERR_INVALID_ARG;
    if (A == nullptr || !aligned4(A) || (dt_bias && !aligned4(dt_bias)) || (D && !aligned4(D)))
        return SSD_ERR_INVALID_ARG;
    if (has_z && rows && (z == nullptr || !aligned16(z))) return SSD_ERR_INVALID_ARG;
    if (ssm_state_out == nullptr || !aligned16(ssm_state_out) ||
        (ssm_state_in && !aligned16(ssm_state_in)))
        return SSD_ERR_INVALID_ARG;
    if (conv_w == nullptr && (conv_state_in || conv_state_out || conv_b))
        return SSD_ERR_INVALID_ARG;
    if (conv_w && !aligned4(conv_w)) return SSD_ERR_INVALID_ARG;
    if ((conv_state_in && !aligned16(conv_state_in)) ||
        (conv_state_out && !aligned16(conv_state_out)))
        return SSD_ERR_INVALID_ARG;
    if (norm) {
        if (!aligned16(norm_w) || !(eps >= 0.0f) || eps > 3.4e38f) return SSD_ERR_INVALID_ARG;
        const long long C = (long long)dims->nheads * dims->headdim;
        if (!gated_norm_supports((int)C, dims->ngroups, act == SSD_BF16)) return SSD_ERR_UNSUPPORTED;
    }
    size_t need = 0;
    s = ssd_chunk_scan_workspace_size(dims, act, flags | (norm ? (unsigned)SSD_GATED_NORM : 0u),
                                      conv_w != nullptr, &need);
    if (s != SSD_OK) return s;
    if (workspace_bytes < need || (need > 0 && (workspace == nullptr || !aligned16(workspace))))
        return SSD_ERR_INVALID_ARG;
    const int chunk = dims->chunk == 0 ? 128 : dims->chunk;
    if (act == SSD_BF16 && chunk != 128) return SSD_ERR_UNSUPPORTED;
    const bool tc = use_tensor_cores(dims, act);
    if (!tc && !scan_simt_supports(dims->headdim, dims->dstate)) return SSD_ERR_UNSUPPORTED;
    if (dims->batch == 0) return SSD_OK;
    if (norm && !(tc && norm_scale_supports(dims->nheads, dims->ngroups))) {
        // the row-exact kernels: the scan without the gate, then the norm in place
        s = chunk_scan_impl(dims, act, flags & ~(unsigned)SSD_HAS_Z, xbc, conv_w, conv_b,
                            conv_state_in, conv_state_out, dt, dt_bias, A, D, nullptr,
                            ssm_state_in, y, ssm_state_out, workspace, workspace_bytes, stream,
                            nullptr, 0.0f);
        if (s != SSD_OK) return s;
        return ssd_gated_group_rmsnorm(dims, act, y, z, norm_w, eps, y, stream);
    }

    unsigned* err = nullptr;
    s = error_word_address(&err);
    if (s != SSD_OK) return s;
    const bool bf16 = act == SSD_BF16;
    if (tc) {
        const int H = dims->nheads, P = dims->headdim, N = dims->dstate, G = dims->ngroups;
        // the scan kernel also writes the new conv state (each CTA its head's x
        // columns, one CTA per group its B|C columns)
        TcScanParams tp{dims->batch, dims->seqlen, H, G, dims->conv_width,
                        has_z ? flags | (unsigned)SSD_HAS_Z : flags,
                        conv_w != nullptr, xbc, xbc, (int)cdim, H * P, conv_w, conv_b,
                        conv_state_in, conv_w != nullptr ? conv_state_out : nullptr, dt, dt_bias,
                        A, D, has_z ? z : nullptr, ssm_state_in, y, ssm_state_out, err};
        tp.wait_ns = g_wait_ns.load(std::memory_order_relaxed);
        if (norm) {
            tp.norm_ss = reinterpret_cast<float*>(static_cast<char*>(workspace) +
                                                  (conv_w != nullptr ? tc_workspace_bytes(dims) : 0));
        }
        if (conv_w != nullptr) {
            // B|C columns: conv + SiLU once per group into the workspace
            ConvParams bp{dims->batch, dims->seqlen, (int)cdim, dims->conv_width, xbc, conv_w,
                          conv_b, conv_state_in, workspace, nullptr, H * P, 2 * G * N, 2 * G * N};
            s = counted(launch_conv1d_rows(bp, true, stream), SSD_KERNEL_BC_CONV);
            if (s != SSD_OK) return s;
            tp.bc = workspace;
            tp.bc_stride = 2 * G * N;
            tp.bc_col0 = 0;
        }
        s = counted(scan_units_supports(tp) ? launch_scan_units(tp, stream, conv_w != nullptr)
                                            : launch_scan_tc(tp, stream, conv_w != nullptr),
                    SSD_KERNEL_SCAN_TC);
        if (s == SSD_OK && norm) {
            NormScaleParams np{dims->batch, dims->seqlen, H, P, G, eps, tp.norm_ss, norm_w, y};
            s = counted(launch_norm_scale(np, stream), SSD_KERNEL_NORM_SCALE, dims->seqlen > 0);
        }
    } else {
        ScanParams p{dims->batch, dims->seqlen, dims->nheads, dims->headdim, dims->dstate,
                     dims->ngroups, dims->conv_width, flags, xbc, conv_w, conv_b, conv_state_in,
                     dt, dt_bias, A, D, has_z ? z : nullptr, ssm_state_in, y, ssm_state_out, err};
        s = counted(launch_scan_simt(p, bf16, stream), SSD_KERNEL_SCAN_SIMT);
    }
    if (s != SSD_OK) return s;
    if (conv_w != nullptr && conv_state_out != nullptr && !(tc && dims->seqlen > 0)) {
        ConvParams cp{dims->batch, dims->seqlen, (int)cdim, dims->conv_width,
                      xbc, conv_w, conv_b, conv_state_in, nullptr, conv_state_out};
        s = counted(launch_conv_state(cp, bf16, stream), SSD_KERNEL_CONV_STATE,
                    dims->conv_width > 1);
    }
    return s;
}

}  // namespace

extern "C" {

ssd_status ssd_chunk_scan(const ssd_dims* dims, ssd_dtype act, unsigned flags, const void* xbc,
                          const float* conv_w, const float* conv_b, const void* conv_state_in,
                          void* conv_state_out, const float* dt, const float* dt_bias,
                          const float* A, const float* D, const void* z,
                          const float* ssm_state_in, void* y, float* ssm_state_out,
                          void* workspace, size_t workspace_bytes, cudaStream_t stream)
{
    return chunk_scan_impl(dims, act, flags, xbc, conv_w, conv_b, conv_state_in, conv_state_out,
                           dt, dt_bias, A, D, z, ssm_state_in, y, ssm_state_out, workspace,
                           workspace_bytes, stream, nullptr, 0.0f);
}

ssd_status ssd_chunk_scan_gated_norm(const ssd_dims* dims, ssd_dtype act, unsigned flags,
                                     const void* xbc, const float* conv_w, const float* conv_b,
                                     const void* conv_state_in, void* conv_state_out,
                                     const float* dt, const float* dt_bias, const float* A,
                                     const float* D, const void* z, const float* norm_w,
                                     float eps, const float* ssm_state_in, void* y,
                                     float* ssm_state_out, void* workspace,
                                     size_t workspace_bytes, cudaStream_t stream)
{
    if (flags & ~(unsigned)(SSD_DT_SOFTPLUS | SSD_HAS_Z | SSD_GATED_NORM)) return SSD_ERR_INVALID_ARG;
    if (norm_w == nullptr) return SSD_ERR_INVALID_ARG;
    return chunk_scan_impl(dims, act, flags & (unsigned)SSD_DT_SOFTPLUS, xbc, conv_w, conv_b,
                           conv_state_in, conv_state_out, dt, dt_bias, A, D, z, ssm_state_in, y,
                           ssm_state_out, workspace, workspace_bytes, stream, norm_w, eps);
}

ssd_status ssd_decode_step(const ssd_dims* dims, ssd_dtype act, unsigned flags, const void* xbc,
                           const float* conv_w, const float* conv_b, void* conv_pool,
                           const float* dt, const float* dt_bias, const float* A,
                           const float* D, const void* z, const int32_t* slot_ids,
                           int num_slots, float* ssm_pool, void* y, cudaStream_t stream)
{
    long long cdim = 0;
    ssd_status s = check_dims(dims, act, &cdim);
    if (s != SSD_OK) return s;
    if (dims->seqlen < 1) return SSD_ERR_INVALID_ARG;
    if (dims->seqlen > kDecodeMaxTokens) return SSD_ERR_UNSUPPORTED;
    if (flags & ~(unsigned)(SSD_DT_SOFTPLUS | SSD_HAS_Z)) return SSD_ERR_INVALID_ARG;
    const bool rows = dims->batch > 0;
    const bool has_z = (flags & SSD_HAS_Z) != 0;
    if (num_slots < 0 || (rows && num_slots == 0)) return SSD_ERR_INVALID_ARG;
    if (rows && (xbc == nullptr || dt == nullptr || y == nullptr || slot_ids == nullptr ||
                 ssm_pool == nullptr || !aligned16(xbc) || !aligned16(y) || !aligned4(dt) ||
                 !aligned4(slot_ids) || !aligned16(ssm_pool)))
        return SSD_ERR_INVALID_ARG;
    if (A == nullptr || !aligned4(A) || (dt_bias && !aligned4(dt_bias)) || (D && !aligned4(D)))
        return SSD_ERR_INVALID_ARG;
    if (has_z && rows && (z == nullptr || !aligned16(z))) return SSD_ERR_INVALID_ARG;
    if (conv_w == nullptr && (conv_pool || conv_b)) return SSD_ERR_INVALID_ARG;
    if (conv_w && (!aligned4(conv_w) || conv_pool == nullptr || !aligned16(conv_pool)))
        return SSD_ERR_INVALID_ARG;
    if (!decode_supports(dims->nheads, dims->headdim, dims->dstate, dims->ngroups, dims->seqlen))
        return SSD_ERR_UNSUPPORTED;
    if (!rows) return SSD_OK;

    unsigned* err = nullptr;
    s = error_word_address(&err);
    if (s != SSD_OK) return s;
    const bool bf16 = act == SSD_BF16;
    DecodeParams p{dims->batch, dims->nheads, dims->headdim, dims->dstate, dims->ngroups,
                   dims->conv_width, flags, xbc, conv_w, conv_b, conv_pool, dt, dt_bias, A, D,
                   has_z ? z : nullptr, slot_ids, num_slots, ssm_pool, y, err};
    p.check_dups = (g_debug_checks.load(std::memory_order_relaxed) & SSD_CHECK_DISTINCT_SLOTS) != 0;
    p.K = dims->seqlen;
    s = counted(launch_decode_step(p, bf16, stream), SSD_KERNEL_DECODE_STEP);
    if (s != SSD_OK) return s;
    return counted(launch_decode_conv_roll(p, bf16, stream), SSD_KERNEL_DECODE_CONV,
                   conv_w != nullptr && dims->conv_width > 1);
}

ssd_status ssd_chunk_scan_varlen(const ssd_dims* dims, ssd_dtype act, unsigned flags,
                                 const int32_t* cu_seqlens, const int32_t* slot_ids,
                                 const int32_t* has_initial_state, int num_slots, const void* xbc,
                                 const float* conv_w, const float* conv_b, void* conv_pool,
                                 const float* dt, const float* dt_bias, const float* A,
                                 const float* D, const void* z, float* ssm_pool, void* y,
                                 void* workspace, size_t workspace_bytes, cudaStream_t stream)
{
    long long cdim = 0;
    ssd_status s = check_dims(dims, act, &cdim);
    if (s != SSD_OK) return s;
    if (flags & ~(unsigned)(SSD_DT_SOFTPLUS | SSD_HAS_Z)) return SSD_ERR_INVALID_ARG;
    const int nseq = dims->batch;
    const long long T = dims->seqlen;
    const bool has_z = (flags & SSD_HAS_Z) != 0;
    const int chunk = dims->chunk == 0 ? 128 : dims->chunk;
    if (act != SSD_BF16 || chunk != 128 || !scan_tc_supports(dims->headdim, dims->dstate) ||
        dims->conv_width > 4)
        return SSD_ERR_UNSUPPORTED;
    if (nseq == 0) return SSD_OK;
    if (cu_seqlens == nullptr || slot_ids == nullptr || !aligned4(cu_seqlens) ||
        !aligned4(slot_ids) || (has_initial_state && !aligned4(has_initial_state)) ||
        num_slots <= 0 || ssm_pool == nullptr || !aligned16(ssm_pool))
        return SSD_ERR_INVALID_ARG;
    if (A == nullptr || !aligned4(A) || (dt_bias && !aligned4(dt_bias)) || (D && !aligned4(D)))
        return SSD_ERR_INVALID_ARG;
    if (T > 0 && (xbc == nullptr || dt == nullptr || y == nullptr || !aligned16(xbc) ||
                  !aligned16(y) || !aligned4(dt) || (has_z && (z == nullptr || !aligned16(z)))))
        return SSD_ERR_INVALID_ARG;
    if (conv_w == nullptr && (conv_pool || conv_b)) return SSD_ERR_INVALID_ARG;
    if (conv_w && (!aligned4(conv_w) || (conv_b && !aligned4(conv_b)) || conv_pool == nullptr ||
                   !aligned16(conv_pool)))
        return SSD_ERR_INVALID_ARG;
    const int H = dims->nheads, P = dims->headdim, N = dims->dstate, G = dims->ngroups;
    const size_t need = conv_w ? (size_t)T * 2 * G * N * 2 : 0;  // post-conv B|C rows
    if (workspace_bytes < need || (need > 0 && (workspace == nullptr || !aligned16(workspace))))
        return SSD_ERR_INVALID_ARG;

    unsigned* err = nullptr;
    s = error_word_address(&err);
    if (s != SSD_OK) return s;
    TcScanParams tp{nseq, (int)T, H, G, dims->conv_width, flags, conv_w != nullptr, xbc, xbc,
                    (int)cdim, H * P, conv_w, conv_b, conv_pool, conv_pool, dt, dt_bias, A, D,
                    has_z ? z : nullptr, ssm_pool, y, ssm_pool, err};
    tp.cu_seqlens = cu_seqlens;
    tp.slot_ids = slot_ids;
    tp.has_init = has_initial_state;
    tp.num_slots = num_slots;
    tp.check_dups = (g_debug_checks.load(std::memory_order_relaxed) & SSD_CHECK_DISTINCT_SLOTS) != 0;
    tp.wait_ns = g_wait_ns.load(std::memory_order_relaxed);
    if (conv_w != nullptr) {
        ConvParams bp{1, (int)T, (int)cdim, dims->conv_width, xbc, conv_w, conv_b, conv_pool,
                      workspace, nullptr, H * P, 2 * G * N, 2 * G * N};
        bp.cu_seqlens = cu_seqlens;
        bp.slot_ids = slot_ids;
        bp.has_init = has_initial_state;
        bp.nseq = nseq;
        bp.num_slots = num_slots;
        s = counted(launch_conv1d_rows(bp, true, stream), SSD_KERNEL_BC_CONV, T > 0);
        if (s != SSD_OK) return s;
        tp.bc = workspace;
        tp.bc_stride = 2 * G * N;
        tp.bc_col0 = 0;
    }
    return counted(launch_scan_tc(tp, stream, conv_w != nullptr && T > 0), SSD_KERNEL_SCAN_TC);
}

ssd_status ssd_gated_group_rmsnorm(const ssd_dims* dims, ssd_dtype act, const void* y,
                                   const void* z, const float* weight, float eps, void* out,
                                   cudaStream_t stream)
{
    if (dims == nullptr || (act != SSD_F32 && act != SSD_BF16)) return SSD_ERR_INVALID_ARG;
    if (dims->batch < 0 || dims->seqlen < 0 || dims->nheads <= 0 || dims->headdim <= 0 ||
        dims->ngroups <= 0 || dims->nheads % dims->ngroups != 0)
        return SSD_ERR_INVALID_ARG;
    if (!(eps >= 0.0f) || eps > 3.4e38f) return SSD_ERR_INVALID_ARG;  // rejects NaN and inf
    const long long C = (long long)dims->nheads * dims->headdim;
    const long long rows = (long long)dims->batch * dims->seqlen;
    const bool bf16 = act == SSD_BF16;
    if (C > (1LL << 30)) return SSD_ERR_INVALID_ARG;
    if (!gated_norm_supports((int)C, dims->ngroups, bf16)) return SSD_ERR_UNSUPPORTED;
    if (weight == nullptr || !aligned16(weight)) return SSD_ERR_INVALID_ARG;
    if (rows > 0 && (y == nullptr || z == nullptr || out == nullptr || !aligned16(y) ||
                     !aligned16(z) || !aligned16(out)))
        return SSD_ERR_INVALID_ARG;
    if (rows == 0) return SSD_OK;
    // out may be y itself, but no other overlap with y or z
    const size_t bytes = (size_t)rows * C * (bf16 ? 2 : 4);
    auto overlaps = [&](const void* a, const void* b) {
        const char* pa = static_cast<const char*>(a);
        const char* pb = static_cast<const char*>(b);
        return pa < pb + bytes && pb < pa + bytes;
    };
    if ((out != y && overlaps(out, y)) || overlaps(out, z)) return SSD_ERR_INVALID_ARG;
    GatedNormParams p{rows, (int)C, dims->ngroups, eps, y, z, weight, out};
    return counted(launch_gated_norm(p, bf16, stream), SSD_KERNEL_GATED_NORM);
}

ssd_status ssd_segment_decay(const ssd_dims* dims, unsigned flags, const float* dt,
                             const float* dt_bias, const float* A, float* gamma,
                             cudaStream_t stream)
{
    if (dims == nullptr || dims->batch < 0 || dims->seqlen < 0 || dims->nheads <= 0)
        return SSD_ERR_INVALID_ARG;
    if (flags & ~(unsigned)SSD_DT_SOFTPLUS) return SSD_ERR_INVALID_ARG;
    if ((long long)dims->batch * dims->seqlen * dims->nheads > (1LL << 62)) return SSD_ERR_INVALID_ARG;
    if (A == nullptr || gamma == nullptr || !aligned4(A) || !aligned4(gamma) ||
        (dt_bias && !aligned4(dt_bias)))
        return SSD_ERR_INVALID_ARG;
    if (dims->batch > 0 && dims->seqlen > 0 && (dt == nullptr || !aligned4(dt)))
        return SSD_ERR_INVALID_ARG;
    if (dims->batch == 0) return SSD_OK;
    SegmentParams p{dims->batch, dims->seqlen, dims->nheads, flags, dt, dt_bias, A, gamma};
    return counted(launch_segment_decay(p, stream), SSD_KERNEL_SEGMENT_DECAY);
}

ssd_status ssd_state_combine(const ssd_dims* dims, const float* gamma, const float* h_prev,
                             const float* h_seg, float* h_out, cudaStream_t stream)
{
    if (dims == nullptr || dims->batch < 0 || dims->nheads <= 0 || dims->headdim <= 0 ||
        dims->dstate <= 0)
        return SSD_ERR_INVALID_ARG;
    const long long pn = (long long)dims->headdim * dims->dstate;
    if (pn % 4 != 0 || (long long)dims->batch * dims->nheads > (1LL << 30) || pn > (1LL << 30))
        return SSD_ERR_INVALID_ARG;
    if (gamma == nullptr || h_seg == nullptr || h_out == nullptr || !aligned4(gamma) ||
        !aligned16(h_seg) || !aligned16(h_out) || (h_prev && !aligned16(h_prev)))
        return SSD_ERR_INVALID_ARG;
    if (dims->batch == 0) return SSD_OK;
    CombineParams p{dims->batch * dims->nheads, pn, gamma, h_prev, h_seg, h_out};
    return counted(launch_state_combine(p, stream), SSD_KERNEL_STATE_COMBINE);
}

}  // extern "C"
