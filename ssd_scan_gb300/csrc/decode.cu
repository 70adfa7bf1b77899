// decode.cu -- one recurrent step at slot-indexed states, in place.
//
// TensorSharp nemotron.md 4.1 (the single-step update dA = exp(dt A),
// state = dA state + dt x B^T, y = state . C + D x) and section 11 (per-slot
// conv + SSM state pool); vllm.cpp #1362 (the update runs at the state slot
// in place, with no gather/scatter copies of the states).
//
// The state read-modify-write is the whole cost: per (row, head) P*N fp32
// are read once and written once.  One CTA per (row i, group g): it conv's
// the x columns of the group's heads and the group's B and C columns once
// (the B|C conv is shared by the heads of the group), then its warps stream
// the state rows of those heads.  A lane owns 16 bytes (4 consecutive n) of
// a state row, so every warp access is a contiguous 512-byte run, loaded
// with streaming hints (the pool is touched once per step); each warp keeps
// several rows in flight.  y[p] is a warp shuffle reduction over n.
#include "internal.cuh"

namespace ssd {
namespace {

constexpr int kThreads = 512;
constexpr int kRowsInFlight = 4;  // state rows a warp keeps in flight

template <typename T>
__global__ void __launch_bounds__(kThreads) decode_step_kernel(DecodeParams p)
{
    extern __shared__ float sm[];  // x [hpg*P] | B [N] | C [N] | dt, dA [hpg]
    const int g = blockIdx.x, i = blockIdx.y;
    const int H = p.H, P = p.P, N = p.N, G = p.G;
    const int hpg = H / G;
    const int h0 = g * hpg;
    const int Cdim = H * P + 2 * G * N;
    const int XW = hpg * P;        // x columns of this group
    const int CH = XW + 2 * N;
    const int s = p.slots[i];
    if (s < 0 || s >= p.num_slots) {
        if (threadIdx.x == 0 && g == 0) atomicOr(p.err, kErrBadSlot);
        return;
    }
    if (p.check_dups && slot_seen_before(p.slots, i, s)) {  // the earlier row owns the slot
        if (threadIdx.x == 0 && g == 0) atomicOr(p.err, kErrDupSlot);
        return;
    }
    const T* xbc = static_cast<const T*>(p.xbc);
    const T* cpool = static_cast<const T*>(p.conv_pool);
    const int HW = p.W - 1;
    float* xs = sm;
    float* Bs = sm + XW;
    float* Cs = Bs + N;
    float* dts = Cs + N;
    float* dAs = dts + hpg;
    for (int c = threadIdx.x; c < CH; c += blockDim.x) {
        const int gc = c < XW ? h0 * P + c
                              : (c < XW + N ? H * P + g * N + (c - XW)
                                            : H * P + G * N + g * N + (c - XW - N));
        float v;
        if (p.conv_w) {
            v = p.conv_b ? p.conv_b[gc] : 0.0f;
            for (int k = 0; k < HW; ++k)
                v = fmaf(p.conv_w[(size_t)gc * p.W + k],
                         to_f32(cpool[((size_t)s * HW + k) * Cdim + gc]), v);
            v = fmaf(p.conv_w[(size_t)gc * p.W + HW], to_f32(xbc[(size_t)i * Cdim + gc]), v);
            v = v / (1.0f + expf(-v));
        } else {
            v = to_f32(xbc[(size_t)i * Cdim + gc]);
        }
        sm[c] = v;
    }
    for (int j = threadIdx.x; j < hpg; j += blockDim.x) {
        const int h = h0 + j;
        float dt = p.dt[(size_t)i * H + h];
        if (p.flags & kDtSoftplus) dt = softplus_f32(dt + (p.dt_bias ? p.dt_bias[h] : 0.0f));
        dts[j] = dt;
        dAs[j] = expf(dt * p.A[h]);
    }
    __syncthreads();

    const float4* B4 = reinterpret_cast<const float4*>(Bs);
    const float4* C4 = reinterpret_cast<const float4*>(Cs);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarp = blockDim.x >> 5;
    const int nv = N / 4;  // float4 per state row
    const T* zz = static_cast<const T*>(p.z);
    T* y = static_cast<T*>(p.y);
    const int nrows = hpg * P;  // state rows of this group, head-major
    float4* st0 = reinterpret_cast<float4*>(p.pool + ((size_t)s * H + h0) * (size_t)P * N);

    for (int r0 = warp * kRowsInFlight; r0 < nrows; r0 += nwarp * kRowsInFlight) {
        float acc[kRowsInFlight];
#pragma unroll
        for (int r = 0; r < kRowsInFlight; ++r) acc[r] = 0.0f;
        for (int v = lane; v < nv; v += 32) {
            float4 hv[kRowsInFlight];
#pragma unroll
            for (int r = 0; r < kRowsInFlight; ++r)
                if (r0 + r < nrows) hv[r] = __ldcs(st0 + (size_t)(r0 + r) * nv + v);
            const float4 bv = B4[v], cv = C4[v];
#pragma unroll
            for (int r = 0; r < kRowsInFlight; ++r) {
                if (r0 + r >= nrows) continue;
                const int j = (r0 + r) / P;  // head within the group
                const float dt = dts[j], dA = dAs[j];
                const float dx = dt * xs[r0 + r];
                float4 o;
                o.x = fmaf(dA, hv[r].x, dx * bv.x);
                o.y = fmaf(dA, hv[r].y, dx * bv.y);
                o.z = fmaf(dA, hv[r].z, dx * bv.z);
                o.w = fmaf(dA, hv[r].w, dx * bv.w);
                acc[r] = fmaf(o.x, cv.x, acc[r]);
                acc[r] = fmaf(o.y, cv.y, acc[r]);
                acc[r] = fmaf(o.z, cv.z, acc[r]);
                acc[r] = fmaf(o.w, cv.w, acc[r]);
                __stcs(st0 + (size_t)(r0 + r) * nv + v, o);
            }
        }
#pragma unroll
        for (int r = 0; r < kRowsInFlight; ++r) {
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) acc[r] += __shfl_xor_sync(0xffffffffu, acc[r], off);
        }
        if (lane < kRowsInFlight && r0 + lane < nrows) {
            float a = acc[0];
#pragma unroll
            for (int r = 1; r < kRowsInFlight; ++r) a = lane == r ? acc[r] : a;
            const int row = r0 + lane;       // j * P + pp
            const int h = h0 + row / P, pp = row % P;
            float yv = fmaf(p.D ? p.D[h] : 0.0f, xs[row], a);
            if (p.flags & kHasZ) {
                const float zv = to_f32(zz[(size_t)i * H * P + h * P + pp]);
                yv *= zv / (1.0f + expf(-zv));
            }
            y[((size_t)i * H + h) * P + pp] = from_f32<T>(yv);
        }
    }
}

// conv_pool[s] <- [conv_pool[s][1:], raw row i]  (one thread per (row, channel);
// it reads row k+1 before writing row k, so the shift is in place).
template <typename T>
__global__ void decode_conv_roll_kernel(DecodeParams p)
{
    const int Cdim = p.H * p.P + 2 * p.G * p.N;
    const int i = blockIdx.y;
    const int c = blockIdx.x * blockDim.x + threadIdx.x;
    if (c >= Cdim) return;
    const int s = p.slots[i];
    if (s < 0 || s >= p.num_slots) return;
    if (p.check_dups && slot_seen_before(p.slots, i, s)) return;
    const int HW = p.W - 1;
    T* cp = static_cast<T*>(p.conv_pool) + (size_t)s * HW * Cdim;
    for (int k = 0; k + 1 < HW; ++k) cp[(size_t)k * Cdim + c] = cp[(size_t)(k + 1) * Cdim + c];
    cp[(size_t)(HW - 1) * Cdim + c] = static_cast<const T*>(p.xbc)[(size_t)i * Cdim + c];
}

size_t decode_smem_bytes(const DecodeParams& p)
{
    const int hpg = p.H / p.G;
    return sizeof(float) * ((size_t)hpg * p.P + 2 * (size_t)p.N + 2 * (size_t)hpg);
}

}  // namespace

bool decode_supports(int H, int P, int N, int G)
{
    const size_t smem = sizeof(float) * ((size_t)(H / G) * P + 2 * (size_t)N + 2 * (size_t)(H / G));
    return N % 4 == 0 && P % 4 == 0 && smem <= 200 * 1024;
}

cudaError_t launch_decode_step(const DecodeParams& p, bool bf16, cudaStream_t st)
{
    if (p.R == 0) return cudaSuccess;
    dim3 grid(p.G, p.R);
    const size_t smem = decode_smem_bytes(p);
    if (bf16) {
        cudaError_t e = cudaFuncSetAttribute(decode_step_kernel<__nv_bfloat16>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        decode_step_kernel<__nv_bfloat16><<<grid, kThreads, smem, st>>>(p);
    } else {
        cudaError_t e = cudaFuncSetAttribute(decode_step_kernel<float>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        decode_step_kernel<float><<<grid, kThreads, smem, st>>>(p);
    }
    return cudaGetLastError();
}

cudaError_t launch_decode_conv_roll(const DecodeParams& p, bool bf16, cudaStream_t st)
{
    if (p.R == 0 || p.conv_w == nullptr || p.W <= 1) return cudaSuccess;
    const int Cdim = p.H * p.P + 2 * p.G * p.N;
    dim3 grid((Cdim + 255) / 256, p.R);
    if (bf16) decode_conv_roll_kernel<__nv_bfloat16><<<grid, 256, 0, st>>>(p);
    else decode_conv_roll_kernel<float><<<grid, 256, 0, st>>>(p);
    return cudaGetLastError();
}

}  // namespace ssd
