// conv1d.cu -- causal depthwise conv1d + SiLU over [conv state ; rows].
//
// TensorRT-Model-Connect #2207 "Implementation" (add_short_conv_rows: the
// causal depthwise conv over the previous conv state plus the chunk) and
// TensorSharp nemotron.md section 3 (Conv1dStep then SiLU), section 6
// (ssm_conv1d.weight [xBCSize, convKernel], optional bias).
//
// HBM-bound: every raw element is read once and every output written once.
// One thread owns 16 bytes of channels (8 bf16 / 4 fp32) and walks a run of
// rows, keeping the last W-1 raw rows of its channels in registers, so a
// warp reads and writes 512 contiguous bytes per row.
#include "internal.cuh"
#include "sm100.cuh"

namespace ssd {
namespace {

constexpr int kRowsPerThread = 8;

// 16 bytes of channels: 8 bf16 or 4 fp32, kept packed in registers.
template <typename T> struct Vec16;
template <> struct Vec16<__nv_bfloat16> {
    static constexpr int n = 8;
    __device__ static uint4 load(const __nv_bfloat16* p)
    {
        return __ldg(reinterpret_cast<const uint4*>(p));
    }
    __device__ static void unpack(uint4 r, float* v)
    {
        const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&r);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float2 f = __bfloat1622float2(h[i]);
            v[2 * i] = f.x;
            v[2 * i + 1] = f.y;
        }
    }
    __device__ static void store(__nv_bfloat16* p, const float* v)
    {
        uint4 r;
        __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&r);
#pragma unroll
        for (int i = 0; i < 4; ++i) h[i] = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
        *reinterpret_cast<uint4*>(p) = r;
    }
    // bf16 outputs: silu through one tanh.approx (relative error ~2^-11,
    // below the bf16 rounding of the result)
    __device__ static float silu(float v)
    {
        float t;
        const float hv = 0.5f * v;
        asm("tanh.approx.f32 %0, %1;" : "=f"(t) : "f"(hv));
        return fmaf(hv, t, hv);
    }
};
template <> struct Vec16<float> {
    static constexpr int n = 4;
    __device__ static uint4 load(const float* p)
    {
        return __ldg(reinterpret_cast<const uint4*>(p));
    }
    __device__ static void unpack(uint4 r, float* v)
    {
        v[0] = __uint_as_float(r.x); v[1] = __uint_as_float(r.y);
        v[2] = __uint_as_float(r.z); v[3] = __uint_as_float(r.w);
    }
    __device__ static void store(float* p, const float* v)
    {
        *reinterpret_cast<float4*>(p) = make_float4(v[0], v[1], v[2], v[3]);
    }
    // fp32 outputs: exp + fast reciprocal division (a few ulp)
    __device__ static float silu(float v) { return __fdividef(v, 1.0f + __expf(-v)); }
};

template <typename T, int W>
__global__ void __launch_bounds__(128) conv1d_rows_kernel(ConvParams p)
{
    constexpr int V = Vec16<T>::n;
    constexpr int R = kRowsPerThread;
    const int nvec = p.ncols / V;
    // a scan launched to overlap this kernel may be scheduled now: it waits for
    // this grid to finish before it reads what this grid writes
    sm100::griddep_launch_dependents();
    const int cv = blockIdx.x * blockDim.x + threadIdx.x;
    if (cv >= nvec) return;
    const int b = blockIdx.z;
    const int t0 = blockIdx.y * R;
    const int nrows = min(R, p.S - t0);
    const int c0 = p.col0 + cv * V;        // absolute channel
    const int o0 = cv * V;                 // column in the output rows
    const T* __restrict__ x = static_cast<const T*>(p.x);
    const T* __restrict__ st = static_cast<const T*>(p.st_in);
    T* __restrict__ out = static_cast<T*>(p.out);

    // raw rows t0-(W-1) .. t0+R-1 of these channels, packed, all loads up front
    uint4 u[R + W - 1];
#pragma unroll
    for (int k = 0; k < W - 1; ++k) {
        const int r = t0 - (W - 1) + k;
        if (r >= 0) u[k] = Vec16<T>::load(x + ((size_t)b * p.S + r) * p.C + c0);
        else if (st) u[k] = Vec16<T>::load(st + ((size_t)b * (W - 1) + (r + W - 1)) * p.C + c0);
        else u[k] = make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int i = 0; i < R; ++i)
        u[W - 1 + i] = i < nrows ? Vec16<T>::load(x + ((size_t)b * p.S + t0 + i) * p.C + c0)
                                 : make_uint4(0, 0, 0, 0);
    // taps: the W floats of one channel are contiguous ([C, W] layout)
    float w[W][V], bias[V];
#pragma unroll
    for (int j = 0; j < V; ++j) {
        bias[j] = p.bias ? __ldg(p.bias + c0 + j) : 0.0f;
        const float* wc = p.w + (size_t)(c0 + j) * W;
        if (W == 4 && (reinterpret_cast<uintptr_t>(p.w) & 15) == 0) {
            const float4 q = __ldg(reinterpret_cast<const float4*>(wc));
            w[0][j] = q.x; w[1 % W][j] = q.y; w[2 % W][j] = q.z; w[3 % W][j] = q.w;
        } else {
#pragma unroll
            for (int k = 0; k < W; ++k) w[k][j] = __ldg(wc + k);
        }
    }
#pragma unroll
    for (int i = 0; i < R; ++i) {
        if (i >= nrows) break;
        float o[V];
#pragma unroll
        for (int j = 0; j < V; ++j) o[j] = bias[j];
#pragma unroll
        for (int k = 0; k < W; ++k) {
            float f[V];
            Vec16<T>::unpack(u[i + k], f);
#pragma unroll
            for (int j = 0; j < V; ++j) o[j] = fmaf(w[k][j], f[j], o[j]);
        }
#pragma unroll
        for (int j = 0; j < V; ++j) o[j] = Vec16<T>::silu(o[j]);
        Vec16<T>::store(out + ((size_t)b * p.S + t0 + i) * p.out_stride + o0, o);
    }
}

// Packed sequences: as conv1d_rows_kernel (8 rows per thread, the raw rows of
// the window and the taps in registers), with the sequence of each row found
// from cu_seqlens (a binary search for the first row, the last i with
// cu_seqlens[i] <= row, then a walk past sequence ends, skipping empty
// sequences).  A tap that reaches before its row's sequence start reads that
// sequence's conv state at its slot instead (zeros for a fresh sequence, or
// for a slot out of range, which the scan reports).  Rows run along grid.x.
template <typename T, int W>
__global__ void __launch_bounds__(128) conv1d_rows_varlen_kernel(ConvParams p)
{
    sm100::griddep_launch_dependents();
    constexpr int V = Vec16<T>::n;
    constexpr int R = kRowsPerThread;
    const int nvec = p.ncols / V;
    const int cv = blockIdx.y * blockDim.x + threadIdx.x;
    if (cv >= nvec) return;
    const long long t0 = (long long)blockIdx.x * R;
    const int nrows = (int)min((long long)R, (long long)p.S - t0);
    const int c0 = p.col0 + cv * V, o0 = cv * V;
    const T* __restrict__ x = static_cast<const T*>(p.x);
    const T* __restrict__ st = static_cast<const T*>(p.st_in);
    T* __restrict__ out = static_cast<T*>(p.out);

    // raw rows t0-(W-1) .. t0+R-1 (rows outside [0, S) read as zeros)
    uint4 u[R + W - 1];
#pragma unroll
    for (int k = 0; k < R + W - 1; ++k) {
        const long long r = t0 - (W - 1) + k;
        u[k] = (r >= 0 && r < p.S) ? Vec16<T>::load(x + r * p.C + c0) : make_uint4(0, 0, 0, 0);
    }
    float w[W][V], bias[V];
#pragma unroll
    for (int j = 0; j < V; ++j) {
        bias[j] = p.bias ? __ldg(p.bias + c0 + j) : 0.0f;
        const float* wc = p.w + (size_t)(c0 + j) * W;
        if (W == 4 && (reinterpret_cast<uintptr_t>(p.w) & 15) == 0) {
            const float4 q = __ldg(reinterpret_cast<const float4*>(wc));
            w[0][j] = q.x; w[1 % W][j] = q.y; w[2 % W][j] = q.z; w[3 % W][j] = q.w;
        } else {
#pragma unroll
            for (int k = 0; k < W; ++k) w[k][j] = __ldg(wc + k);
        }
    }
    // the sequence of row t0
    int lo = 0, hi = p.nseq;  // cu[lo] <= t0 < cu[hi]
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (p.cu_seqlens[mid] <= t0) lo = mid;
        else hi = mid;
    }
    int i = lo;
    long long s0 = p.cu_seqlens[i], s1 = p.cu_seqlens[i + 1];
#pragma unroll
    for (int rr = 0; rr < R; ++rr) {
        if (rr >= nrows) break;
        const long long r = t0 + rr;
        while (r >= s1 && i + 1 < p.nseq) {  // the next non-empty sequence
            ++i;
            s0 = s1;
            s1 = p.cu_seqlens[i + 1];
        }
        float o[V];
#pragma unroll
        for (int j = 0; j < V; ++j) o[j] = bias[j];
#pragma unroll
        for (int k = 0; k < W; ++k) {
            const long long src = r - (W - 1) + k;  // the row this tap reads
            uint4 raw = u[rr + k];
            if (src < s0) {  // before the sequence's first row: its conv state
                raw = make_uint4(0, 0, 0, 0);
                const int slot = p.slot_ids[i];
                const long long sr = (W - 1) + (src - s0);  // row of the state
                if (st != nullptr && (p.has_init == nullptr || p.has_init[i] != 0) && slot >= 0 &&
                    slot < p.num_slots && sr >= 0)
                    raw = Vec16<T>::load(st + ((size_t)slot * (W - 1) + sr) * p.C + c0);
            }
            float f[V];
            Vec16<T>::unpack(raw, f);
#pragma unroll
            for (int j = 0; j < V; ++j) o[j] = fmaf(w[k][j], f[j], o[j]);
        }
#pragma unroll
        for (int j = 0; j < V; ++j) o[j] = Vec16<T>::silu(o[j]);
        Vec16<T>::store(out + r * p.out_stride + o0, o);
    }
}

// conv_state_out[b, j, c] = u[b, S + j, c] with u = [state_in ; x].  One
// thread per (b, c) walks j upwards, so an in-place call (st_out == st_in)
// only ever overwrites rows it has already read.
template <typename T>
__global__ void conv_state_kernel(ConvParams p)
{
    const size_t idx = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (idx >= (size_t)p.B * p.C) return;
    const int b = (int)(idx / p.C), c = (int)(idx % p.C);
    const int nh = p.W - 1;
    const T* x = static_cast<const T*>(p.x);
    const T* st = static_cast<const T*>(p.st_in);
    T* so = static_cast<T*>(p.st_out);
    for (int j = 0; j < nh; ++j) {
        const int r = p.S + j;  // index into u
        T v;
        if (r < nh) v = st ? st[((size_t)b * nh + r) * p.C + c] : from_f32<T>(0.0f);
        else v = x[((size_t)b * p.S + (r - nh)) * p.C + c];
        so[((size_t)b * nh + j) * p.C + c] = v;
    }
}

template <typename T>
cudaError_t launch_rows_t(ConvParams p, cudaStream_t st)
{
    constexpr int V = Vec16<T>::n;
    if (p.ncols < 0) p.ncols = p.C;
    if (p.out_stride < 0) p.out_stride = p.ncols;
    if (p.ncols % V != 0 || p.col0 % V != 0 || p.out_stride % V != 0) return cudaErrorInvalidValue;
    const int nvec = p.ncols / V;
    dim3 block(128);
    if (p.cu_seqlens != nullptr) {  // packed sequences: rows along grid.x
        dim3 vgrid((unsigned)((p.S + kRowsPerThread - 1) / kRowsPerThread), (nvec + 127) / 128);
        switch (p.W) {
#define SSD_CONV_VCASE(w) \
    case w: conv1d_rows_varlen_kernel<T, w><<<vgrid, block, 0, st>>>(p); break;
            SSD_CONV_VCASE(1) SSD_CONV_VCASE(2) SSD_CONV_VCASE(3) SSD_CONV_VCASE(4)
            SSD_CONV_VCASE(5) SSD_CONV_VCASE(6) SSD_CONV_VCASE(7) SSD_CONV_VCASE(8)
#undef SSD_CONV_VCASE
            default: return cudaErrorInvalidValue;
        }
        return cudaGetLastError();
    }
    dim3 grid((nvec + 127) / 128, (p.S + kRowsPerThread - 1) / kRowsPerThread, p.B);
    switch (p.W) {
#define SSD_CONV_CASE(w) \
    case w: conv1d_rows_kernel<T, w><<<grid, block, 0, st>>>(p); break;
        SSD_CONV_CASE(1) SSD_CONV_CASE(2) SSD_CONV_CASE(3) SSD_CONV_CASE(4)
        SSD_CONV_CASE(5) SSD_CONV_CASE(6) SSD_CONV_CASE(7) SSD_CONV_CASE(8)
#undef SSD_CONV_CASE
        default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_conv1d_rows(const ConvParams& p, bool bf16, cudaStream_t st)
{
    if (p.B == 0 || p.S == 0 || p.C == 0) return cudaSuccess;
    return bf16 ? launch_rows_t<__nv_bfloat16>(p, st) : launch_rows_t<float>(p, st);
}

cudaError_t launch_conv_state(const ConvParams& p, bool bf16, cudaStream_t st)
{
    if (p.B == 0 || p.W <= 1 || p.C == 0 || p.st_out == nullptr) return cudaSuccess;
    const size_t n = (size_t)p.B * p.C;
    dim3 grid((unsigned)((n + 255) / 256));
    if (bf16) conv_state_kernel<__nv_bfloat16><<<grid, 256, 0, st>>>(p);
    else conv_state_kernel<float><<<grid, 256, 0, st>>>(p);
    return cudaGetLastError();
}

}  // namespace ssd
