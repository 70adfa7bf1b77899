// internal.cuh -- launch parameters and helpers shared by the kernels of the
// GB300 SSD library.  Not part of the public ABI (see include/ssd.h).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace ssd {

// Bits of the per-device error word (first error kind wins in the report).
enum : unsigned { kErrBadSlot = 1u, kErrTimeout = 2u, kErrDupSlot = 4u };

enum : unsigned { kDtSoftplus = 1u, kHasZ = 2u };

struct ConvParams {
    int B, S, C, W;
    const void* x;        // [B,S,C] act, raw rows
    const float* w;       // [C,W]
    const float* bias;    // [C] or null
    const void* st_in;    // [B,W-1,C] act or null
    void* out;            // [B,S,out_stride] act: channels [col0, col0+ncols) of the conv
    void* st_out;         // [B,W-1,C] act or null
    int col0 = 0;         // first channel the rows kernel computes
    int ncols = -1;       // channels it computes (-1: all C)
    int out_stride = -1;  // output row length in elements (-1: C)
    // packed sequences (rows kernel only; null: B sequences of S rows): nseq
    // sequences over the S rows, sequence i = rows cu_seqlens[i] ..
    // cu_seqlens[i+1]-1, its conv state at slot slot_ids[i] of st_in (zeros
    // when has_init[i] == 0)
    const int* cu_seqlens = nullptr;
    const int* slot_ids = nullptr;
    const int* has_init = nullptr;
    int nseq = 0, num_slots = 0;
};

struct ScanParams {
    int B, S, H, P, N, G, W;
    unsigned flags;
    const void* xbc;            // [B,S,Cdim] act
    const float* conv_w;        // [Cdim,W] or null (xbc already post-conv)
    const float* conv_b;        // [Cdim] or null
    const void* conv_state_in;  // [B,W-1,Cdim] act or null
    const float* dt;            // [B,S,H]
    const float* dt_bias;       // [H] or null
    const float* A;             // [H]
    const float* D;             // [H] or null
    const void* z;              // [B,S,H*P] act or null
    const float* h0;            // [B,H,P,N] or null
    void* y;                    // [B,S,H,P] act
    float* hS;                  // [B,H,P,N]
    unsigned* err;              // device error word
};

// Tokens one decode call may carry per row (consecutive steps of a request).
constexpr int kDecodeMaxTokens = 16;

struct DecodeParams {
    int R, H, P, N, G, W;
    unsigned flags;
    const void* xbc;        // [R,Cdim] act
    const float* conv_w;    // [Cdim,W] or null
    const float* conv_b;    // [Cdim] or null
    void* conv_pool;        // [num_slots,W-1,Cdim] act or null
    const float* dt;        // [R,H]
    const float* dt_bias;   // [H] or null
    const float* A;         // [H]
    const float* D;         // [H] or null
    const void* z;          // [R,H*P] act or null
    const int32_t* slots;   // [R]
    int num_slots;
    float* pool;            // [num_slots,H,P,N]
    void* y;                // [R,H,P] act
    unsigned* err;
    int check_dups = 0;     // a row whose slot id appeared at an earlier row: report, skip
    int K = 1;              // tokens per row: xbc [R,K,Cdim], dt [R,K,H], z, y [R,K,..]
};

// Has slot id `s` already appeared among ids[0 .. i-1]?  (debug check)
__device__ __forceinline__ bool slot_seen_before(const int32_t* ids, int i, int s)
{
    for (int k = 0; k < i; ++k)
        if (ids[k] == s) return true;
    return false;
}

// ---- element conversions --------------------------------------------------
__device__ __forceinline__ float to_f32(float v) { return v; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 v) { return __bfloat162float(v); }
template <typename T> __device__ __forceinline__ T from_f32(float v);
template <> __device__ __forceinline__ float from_f32<float>(float v) { return v; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float v)
{
    return __float2bfloat16_rn(v);
}

// silu(v) = v * sigmoid(v), fp32, IEEE division.
__device__ __forceinline__ float silu_f32(float v) { return v / (1.0f + __expf(-v)); }

// softplus(v) = max(v,0) + log1p(exp(-|v|)), no threshold.
__device__ __forceinline__ float softplus_f32(float v)
{
    return fmaxf(v, 0.0f) + log1pf(__expf(-fabsf(v)));
}

// ---- launchers (each returns the cudaError_t of its launch) ----------------
cudaError_t launch_conv1d_rows(const ConvParams& p, bool bf16, cudaStream_t st);
cudaError_t launch_conv_state(const ConvParams& p, bool bf16, cudaStream_t st);
cudaError_t launch_scan_simt(const ScanParams& p, bool bf16, cudaStream_t st);
bool scan_simt_supports(int P, int N);
// Tensor-core chunk scan (bf16, P = 64, N = 128, 128-row chunks).
struct TcScanParams {
    int B, S, H, G, W;
    unsigned flags;
    bool conv;                   // x columns are raw: conv + SiLU in the kernel
    const void* xbc;             // [B,S,Cdim] bf16 (raw x when conv)
    const void* bc;              // post-conv B|C columns: rows of bc_stride elements
    int bc_stride, bc_col0;      // row length and first B column of `bc`
    const float* conv_w;         // [Cdim,W] (when conv)
    const float* conv_b;         // [Cdim] or null
    const void* conv_state_in;   // [B,W-1,Cdim] bf16 or null
    void* conv_state_out;        // [B,W-1,Cdim] bf16 or null (may alias conv_state_in)
    const float* dt;             // [B,S,H]
    const float* dt_bias;        // [H] or null
    const float* A;              // [H]
    const float* D;              // [H] or null
    const void* z;               // [B,S,H*64] bf16 or null
    const float* h0;             // [B,H,64,128] or null
    void* y;                     // [B,S,H,64] bf16
    float* hS;                   // [B,H,64,128]
    unsigned* err;
    // Packed sequences of different lengths (null: B sequences of S rows each).
    // Sequence i is rows cu_seqlens[i] .. cu_seqlens[i+1]-1 of the S rows of
    // every row array (B = number of sequences, batch 1 in the row arrays); its
    // states are slot slot_ids[i] of the pools h0 == hS and conv_state_in ==
    // conv_state_out, read as zeros when has_init[i] == 0.
    const int* cu_seqlens = nullptr;
    const int* slot_ids = nullptr;
    const int* has_init = nullptr;  // or null: every sequence continues its slot
    int num_slots = 0;
    int check_dups = 0;             // packed sequences: report and skip a repeated slot id
    unsigned long long wait_ns = 0; // bound on each wait between the kernel's warps
    // The gated group RMSNorm's epilogue share (fixed-length calls with z):
    // besides y silu(z), each row's sum of y^2 over the head's channels (y
    // before the gate) into norm_ss [B,H,S]; null: the plain gate.
    float* norm_ss = nullptr;
};
bool scan_tc_supports(int P, int N);
// Calls of at most 128 rows per sequence (fixed length, no fused norm): one CTA
// per SM walking several one-chunk (sequence, head) units.
bool scan_units_supports(const TcScanParams& p);
cudaError_t launch_scan_units(const TcScanParams& p, cudaStream_t st, bool after_prepass);
// after_prepass: the kernel just before it on `st` is the B|C conv writing p.bc;
// the scan is then launched to overlap that kernel's tail (programmatic
// dependent launch) and waits for it before its first read of p.bc.
cudaError_t launch_scan_tc(const TcScanParams& p, cudaStream_t st, bool after_prepass);

bool decode_supports(int H, int P, int N, int G, int K);
cudaError_t launch_decode_step(const DecodeParams& p, bool bf16, cudaStream_t st);

struct GatedNormParams {
    long long rows;   // B*S
    int C, G;         // channels per row (H*P), groups
    float eps;
    const void* y;    // [rows, C] act
    const void* z;    // [rows, C] act
    const float* w;   // [C]
    void* out;        // [rows, C] act, may alias y
};
// Sequence-parallel state passing (state_pass.cu).
struct SegmentParams {
    int B, S, H;
    unsigned flags;
    const float* dt;       // [B,S,H]
    const float* dt_bias;  // [H] or null
    const float* A;        // [H]
    float* gamma;          // [B,H]: sum over the rows of dt * A
};
struct CombineParams {
    int BH;                // sequences x heads
    long long PN;          // state elements per head (a multiple of 4)
    const float* gamma;    // [BH]
    const float* h_prev;   // [BH, PN] or null (zeros)
    const float* h_seg;    // [BH, PN]
    float* h_out;          // [BH, PN]; may alias h_prev or h_seg
};
cudaError_t launch_segment_decay(const SegmentParams& p, cudaStream_t st);
cudaError_t launch_state_combine(const CombineParams& p, cudaStream_t st);

// y[r, c] *= w[c] / sqrt(sum_{h in group(c)} ss[b, h, s] / gs + eps), in
// place: the second step of the gated group RMSNorm after a scan that applied
// the gate and left the per-head sums of squares (bf16 y).
struct NormScaleParams {
    int B, S, H, P, G;
    float eps;
    const float* ss;  // [B,H,S]
    const float* w;   // [H*P]
    void* y;          // [B,S,H,P] bf16, scaled in place
};
bool norm_scale_supports(int H, int G);
cudaError_t launch_norm_scale(const NormScaleParams& p, cudaStream_t st);

bool gated_norm_supports(int C, int G, bool bf16);
cudaError_t launch_gated_norm(const GatedNormParams& p, bool bf16, cudaStream_t st);
cudaError_t launch_decode_conv_roll(const DecodeParams& p, bool bf16, cudaStream_t st);

}  // namespace ssd
