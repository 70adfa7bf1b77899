// norm.cu -- group RMSNorm of the scan output y, then the SiLU(z) gate.
//
// TensorSharp nemotron.md section 3 (Mamba2 branch: out = SiLU(z) *
// GroupRMSNorm(y, ssm_norm.weight)), section 4.1 (the group norm normalises y
// per group, then the gate multiplies) and section 6 (ssm_norm.weight, one
// weight per channel of dInner = H*P).  For every row and each of the G groups
// of gs = H*P/G contiguous channels:
//   out[c] = silu(z[c]) * y[c] / sqrt(mean_{c' in group} y[c']^2 + eps) * w[c]
//
// HBM-bound (reads y, z; writes out): one warp per (row, group).  The first
// pass sums y^2 (16-byte vectors, fp32 accumulation, a warp reduction); the
// second reads y again (from L1: the warp just read it), z and w, and writes
// out.  Every lane writes only elements it has read, so out may alias y.
#include "internal.cuh"

namespace ssd {
namespace {

constexpr int kWarps = 8;  // (row, group) pairs per CTA

template <typename T> struct NormVec;
template <> struct NormVec<__nv_bfloat16> {
    static constexpr int n = 8;
    __device__ static void load(const void* p, float* v)
    {
        const uint4 r = __ldg(reinterpret_cast<const uint4*>(p));
        const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&r);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float2 f = __bfloat1622float2(h[i]);
            v[2 * i] = f.x;
            v[2 * i + 1] = f.y;
        }
    }
    __device__ static void store(void* p, const float* v)
    {
        uint4 r;
        __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&r);
#pragma unroll
        for (int i = 0; i < 4; ++i) h[i] = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
        *reinterpret_cast<uint4*>(p) = r;
    }
    // bf16 output: silu(v) = (v/2)(1 + tanh(v/2)) with the hardware tanh
    // (relative error ~2^-11, below the bf16 rounding of the result)
    __device__ static float silu(float v)
    {
        float t;
        const float hv = 0.5f * v;
        asm("tanh.approx.f32 %0, %1;" : "=f"(t) : "f"(hv));
        return fmaf(hv, t, hv);
    }
};
template <> struct NormVec<float> {
    static constexpr int n = 4;
    __device__ static void load(const void* p, float* v)
    {
        const float4 r = __ldg(reinterpret_cast<const float4*>(p));
        v[0] = r.x; v[1] = r.y; v[2] = r.z; v[3] = r.w;
    }
    __device__ static void store(void* p, const float* v)
    {
        *reinterpret_cast<float4*>(p) = make_float4(v[0], v[1], v[2], v[3]);
    }
    __device__ static float silu(float v) { return __fdividef(v, 1.0f + __expf(-v)); }
};

template <typename T>
__global__ void __launch_bounds__(kWarps * 32) gated_norm_kernel(GatedNormParams p)
{
    constexpr int V = NormVec<T>::n;
    const int lane = threadIdx.x & 31;
    const long long pair = (long long)blockIdx.x * kWarps + (threadIdx.x >> 5);
    if (pair >= p.rows * p.G) return;
    const long long row = pair / p.G;
    const int g = (int)(pair % p.G);
    const int gs = p.C / p.G;
    const size_t base = (size_t)row * p.C + (size_t)g * gs;  // first element of the group
    const T* y = static_cast<const T*>(p.y) + base;
    const T* z = static_cast<const T*>(p.z) + base;
    T* out = static_cast<T*>(p.out) + base;
    const float* w = p.w + (size_t)g * gs;

    float ss = 0.0f;
    for (int e = lane * V; e < gs; e += 32 * V) {
        float v[V];
        NormVec<T>::load(y + e, v);
#pragma unroll
        for (int i = 0; i < V; ++i) ss = fmaf(v[i], v[i], ss);
    }
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, d);
    const float r = rsqrtf(ss / (float)gs + p.eps);

    for (int e = lane * V; e < gs; e += 32 * V) {
        float v[V], zv[V], o[V];
        NormVec<T>::load(y + e, v);
        NormVec<T>::load(z + e, zv);
#pragma unroll
        for (int i = 0; i < V; i += 4) {
            const float4 wv = __ldg(reinterpret_cast<const float4*>(w + e + i));
            const float ws[4] = {wv.x, wv.y, wv.z, wv.w};
#pragma unroll
            for (int k = 0; k < 4; ++k) o[i + k] = NormVec<T>::silu(zv[i + k]) * (v[i + k] * r) * ws[k];
        }
        NormVec<T>::store(out + e, o);
    }
}

// One CTA per (row, group) when the group is a whole number of warps of
// vectors (gs = 32 V k, k <= 32): one vector of y and of z per thread, all
// loads in flight at once, a shared-memory reduction over the k warps.
template <typename T>
__global__ void __launch_bounds__(1024) gated_norm_block_kernel(GatedNormParams p)
{
    constexpr int V = NormVec<T>::n;
    __shared__ float part[32];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const long long row = blockIdx.x / p.G;
    const int g = (int)(blockIdx.x % p.G);
    const int gs = p.C / p.G;
    const size_t off = (size_t)row * p.C + (size_t)g * gs + (size_t)tid * V;
    float v[V], zv[V];
    NormVec<T>::load(static_cast<const T*>(p.y) + off, v);
    NormVec<T>::load(static_cast<const T*>(p.z) + off, zv);
    float ss = 0.0f;
#pragma unroll
    for (int i = 0; i < V; ++i) ss = fmaf(v[i], v[i], ss);
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, d);
    if (lane == 0) part[warp] = ss;
    __syncthreads();
    float tot = 0.0f;
    for (int i = 0; i < (int)(blockDim.x >> 5); ++i) tot += part[i];
    const float r = rsqrtf(tot / (float)gs + p.eps);
    const float* w = p.w + (size_t)g * gs + (size_t)tid * V;
    float o[V];
#pragma unroll
    for (int i = 0; i < V; i += 4) {
        const float4 wv = __ldg(reinterpret_cast<const float4*>(w + i));
        const float ws[4] = {wv.x, wv.y, wv.z, wv.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) o[i + k] = NormVec<T>::silu(zv[i + k]) * (v[i + k] * r) * ws[k];
    }
    NormVec<T>::store(static_cast<T*>(p.out) + off, o);
}

// The scale step of the gated group RMSNorm fused into the scan: the scan
// wrote y' = y silu(z) (bf16) and each row's sum of y^2 per head into ss.
// A group of the norm is H/G whole heads, so its mean square is the sum of
// those heads' partial sums over gs channels, and out = y' w / sqrt(ms + eps).
// kScaleRows rows per CTA; a thread owns the same 16-byte column vectors in
// each of them.  A warp's 32 vectors of one pass lie in one group, so each
// warp sums that group's partials itself (lane = head x row, shuffles) and
// needs no barrier.  Every load (y', the weights, the partial sums) is issued
// before the first wait, so their latencies overlap.
constexpr int kScaleRows = 2;
constexpr int kScaleThreads = 256;
constexpr int kScaleU = 1;  // column vectors per thread and row in one pass
constexpr int kScaleSs = kScaleRows > 1 ? kScaleRows / 2 : 1;  // partial-sum rows per lane

__global__ void __launch_bounds__(kScaleThreads) norm_scale_kernel(NormScaleParams p)
{
    const int tid = threadIdx.x, lane = tid & 31;
    const long long rows = (long long)p.B * p.S;
    const long long r0 = (long long)blockIdx.x * kScaleRows;
    const int nrows = (int)min((long long)kScaleRows, rows - r0);
    const int hg = p.H / p.G;
    const int vpr = p.H * p.P / 8;  // 16-byte vectors per row
    const int vpg = hg * p.P / 8;   // per group (a multiple of 32)
    const float inv_gs = 1.0f / (float)(hg * p.P);
    uint4* y = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.y) + (size_t)r0 * p.H * p.P);
    const float4* w4 = reinterpret_cast<const float4*>(p.w);
    // this lane's share of the partial sums: head k0 (+16, +32, ..) of rows
    // 2i + (lane >> 4); the two half-warps' sums meet in lanes 0 and 16
    const int k0 = lane & 15;
    const float* ssrow[kScaleSs];
#pragma unroll
    for (int i = 0; i < kScaleSs; ++i) {
        const int rl = 2 * i + (lane >> 4);
        const long long rr = r0 + rl;
        ssrow[i] = rl < nrows ? p.ss + (size_t)(rr / p.S) * p.H * p.S + rr % p.S : nullptr;
    }

    for (int cb = 0; cb < vpr; cb += kScaleU * kScaleThreads) {
        uint4 buf[kScaleRows][kScaleU];
        float4 wa[kScaleU], wb[kScaleU];
        float ssv[kScaleU][kScaleSs];
#pragma unroll
        for (int u = 0; u < kScaleU; ++u) {
            const int cv = cb + tid + u * kScaleThreads;
            if (cv < vpr) {
#pragma unroll
                for (int rl = 0; rl < kScaleRows; ++rl)
                    if (rl < nrows) buf[rl][u] = y[(size_t)rl * vpr + cv];
                wa[u] = __ldg(w4 + 2 * cv);
                wb[u] = __ldg(w4 + 2 * cv + 1);
            }
            const int cw = cb + (tid & ~31) + u * kScaleThreads;  // the warp's first vector
#pragma unroll
            for (int i = 0; i < kScaleSs; ++i) {
                float acc = 0.0f;
                if (cw < vpr && ssrow[i] != nullptr) {
                    const float* ss = ssrow[i] + (size_t)(cw / vpg) * hg * p.S;
                    for (int k = k0; k < hg; k += 16) acc += ss[(size_t)k * p.S];
                }
                ssv[u][i] = acc;
            }
        }
#pragma unroll
        for (int u = 0; u < kScaleU; ++u)
#pragma unroll
            for (int i = 0; i < kScaleSs; ++i)
#pragma unroll
                for (int d = 1; d < 16; d <<= 1) ssv[u][i] += __shfl_xor_sync(0xffffffffu, ssv[u][i], d);
#pragma unroll
        for (int u = 0; u < kScaleU; ++u) {
            const int cv = cb + tid + u * kScaleThreads;
#pragma unroll
            for (int rl = 0; rl < kScaleRows; ++rl) {
                const float f = rsqrtf(__shfl_sync(0xffffffffu, ssv[u][rl >> 1], 16 * (rl & 1)) * inv_gs + p.eps);
                if (cv >= vpr || rl >= nrows) continue;
                const float2 ff = make_float2(f, f);
                const float2 wf[4] = {__fmul2_rn(make_float2(wa[u].x, wa[u].y), ff),
                                      __fmul2_rn(make_float2(wa[u].z, wa[u].w), ff),
                                      __fmul2_rn(make_float2(wb[u].x, wb[u].y), ff),
                                      __fmul2_rn(make_float2(wb[u].z, wb[u].w), ff)};
                __nv_bfloat162* hv = reinterpret_cast<__nv_bfloat162*>(&buf[rl][u]);
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    hv[k] = __float22bfloat162_rn(__fmul2_rn(__bfloat1622float2(hv[k]), wf[k]));
                y[(size_t)rl * vpr + cv] = buf[rl][u];
            }
        }
    }
}

}  // namespace

bool norm_scale_supports(int H, int G)
{
    // a warp's 32 vectors in one group: a group of a multiple of 256 channels
    // (P = 64: a multiple of 4 heads)
    return G > 0 && H % G == 0 && (H / G) * 64 % 256 == 0;
}

cudaError_t launch_norm_scale(const NormScaleParams& p, cudaStream_t st)
{
    const long long rows = (long long)p.B * p.S;
    if (rows == 0) return cudaSuccess;
    const long long blocks = (rows + kScaleRows - 1) / kScaleRows;
    if (blocks > 0x7fffffffLL || p.P != 64 || !norm_scale_supports(p.H, p.G))
        return cudaErrorInvalidValue;
    norm_scale_kernel<<<(unsigned)blocks, kScaleThreads, 0, st>>>(p);
    return cudaGetLastError();
}

bool gated_norm_supports(int C, int G, bool bf16)
{
    if (G <= 0 || C % G != 0) return false;
    const int gs = C / G;
    return gs % (bf16 ? 8 : 4) == 0;
}

cudaError_t launch_gated_norm(const GatedNormParams& p, bool bf16, cudaStream_t st)
{
    if (p.rows == 0) return cudaSuccess;
    const long long pairs = p.rows * p.G;
    const int V = bf16 ? 8 : 4, gs = p.C / p.G;
    if (gs % (32 * V) == 0 && gs / V <= 1024 && pairs <= 0x7fffffffLL) {
        if (bf16) gated_norm_block_kernel<__nv_bfloat16><<<(unsigned)pairs, gs / V, 0, st>>>(p);
        else gated_norm_block_kernel<float><<<(unsigned)pairs, gs / V, 0, st>>>(p);
        return cudaGetLastError();
    }
    const dim3 grid((unsigned)((pairs + kWarps - 1) / kWarps));
    if (bf16) gated_norm_kernel<__nv_bfloat16><<<grid, kWarps * 32, 0, st>>>(p);
    else gated_norm_kernel<float><<<grid, kWarps * 32, 0, st>>>(p);
    return cudaGetLastError();
}

}  // namespace ssd
