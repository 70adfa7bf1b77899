// decode.cu -- one recurrent step at slot-indexed states, in place.
//
// TensorSharp nemotron.md 4.1 (the single-step update dA = exp(dt A),
// state = dA state + dt x B^T, y = state . C + D x) and section 11 (per-slot
// conv + SSM state pool); vllm.cpp #1362 (the update runs at the state slot
// in place, with no gather/scatter copies of the states).
//
// The state read-modify-write is the whole cost: per (row, head) P*N fp32
// are read once and written once.  A row may carry K tokens (K consecutive
// steps of one request, e.g. several tokens of multi-token decoding): the
// state is then updated K times in registers between that one read and
// that one write.  One CTA per (row i, group g): it conv's
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

// One call steps every row K tokens (K = dims->seqlen, 1 <= K <= 16): the
// state is read once, updated K times in registers and written once.  KT is
// the compile-time bound on K (1, 2, 4, 8 or 16) and RF the state rows a warp
// keeps in flight; RF * KT (a power of two, at most 32) partial sums of y per
// lane are reduced over the warp together.
template <typename T, int KT, int RF, bool kZs>
__global__ void __launch_bounds__(kThreads) decode_step_kernel(DecodeParams p)
{
    // x [K][hpg*P] | B [K][N] | C [K][N] | dt, dA [K][hpg] | D [hpg] | silu(z) [K][hpg*P]
    // (the last with kZs, when it fits beside the rest: else z is read by the
    // lanes that write y)
    extern __shared__ float sm[];
    const int g = blockIdx.x, i = blockIdx.y;
    const int H = p.H, P = p.P, N = p.N, G = p.G, K = p.K;
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
    float* xs = sm;                 // [K][XW]
    float* Bs = xs + K * XW;        // [K][N]
    float* Cs = Bs + K * N;         // [K][N]
    float* dts = Cs + K * N;        // [K][hpg]
    float* dAs = dts + K * hpg;     // [K][hpg]
    float* Ds = dAs + K * hpg;      // [hpg]
    float* zs = Ds + hpg;           // [K][XW] (kZs)
    // conv + SiLU of the group's channels over u = [conv state ; the row's K
    // tokens]: output t reads u rows t .. t+W-1 (the first W-1 rows of u from
    // the slot's conv state, the rest from the row's raw tokens).  A thread per
    // (channel, token) output, so a row's K tokens spread over the CTA.
    for (int it = threadIdx.x; it < CH * K; it += blockDim.x) {
        const int c = it % CH, t = it / CH;
        const int gc = c < XW ? h0 * P + c
                              : (c < XW + N ? H * P + g * N + (c - XW)
                                            : H * P + G * N + g * N + (c - XW - N));
        float* dst = c < XW ? xs + c : (c < XW + N ? Bs + (c - XW) : Cs + (c - XW - N));
        const int ld = c < XW ? XW : N;  // row stride of dst
        float v;
        if (p.conv_w) {
            v = p.conv_b ? p.conv_b[gc] : 0.0f;
#pragma unroll 4
            for (int k = 0; k < p.W; ++k) {
                const int u = t + k;
                const float xv = u < HW ? to_f32(cpool[((size_t)s * HW + u) * Cdim + gc])
                                        : to_f32(xbc[((size_t)i * K + (u - HW)) * Cdim + gc]);
                v = fmaf(p.conv_w[(size_t)gc * p.W + k], xv, v);
            }
            v = v / (1.0f + expf(-v));
        } else {
            v = to_f32(xbc[((size_t)i * K + t) * Cdim + gc]);
        }
        dst[t * ld] = v;
    }
    for (int jt = threadIdx.x; jt < K * hpg; jt += blockDim.x) {
        const int t = jt / hpg, j = jt % hpg;
        const int h = h0 + j;
        float dt = p.dt[((size_t)i * K + t) * H + h];
        if (p.flags & kDtSoftplus) dt = softplus_f32(dt + (p.dt_bias ? p.dt_bias[h] : 0.0f));
        dts[jt] = dt;
        dAs[jt] = expf(dt * p.A[h]);
    }
    // the skip weights and the gate, so that no global load waits in the
    // state loop below
    for (int j = threadIdx.x; j < hpg; j += blockDim.x) Ds[j] = p.D ? p.D[h0 + j] : 0.0f;
    const T* zz = static_cast<const T*>(p.z);
    if (kZs && (p.flags & kHasZ)) {
        for (int e = threadIdx.x; e < K * XW; e += blockDim.x) {
            const int t = e / XW, c = e % XW;
            const float zv = to_f32(zz[((size_t)i * K + t) * H * P + h0 * P + c]);
            zs[e] = zv / (1.0f + expf(-zv));
        }
    }
    __syncthreads();

    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarp = blockDim.x >> 5;
    const int nv = N / 4;  // float4 per state row
    T* y = static_cast<T*>(p.y);
    const int nrows = hpg * P;  // state rows of this group, head-major
    float4* st0 = reinterpret_cast<float4*>(p.pool + ((size_t)s * H + h0) * (size_t)P * N);

    // RF consecutive state rows never cross a head (RF divides P): one head's
    // dt and decay per token for the whole group of rows
    for (int r0 = warp * RF; r0 < nrows; r0 += nwarp * RF) {
        const int j = r0 / P;  // head within the group
        float acc[RF * KT];
#pragma unroll
        for (int e = 0; e < RF * KT; ++e) acc[e] = 0.0f;
        for (int v = lane; v < nv; v += 32) {
            float4 hv[RF];
#pragma unroll
            for (int r = 0; r < RF; ++r) hv[r] = __ldcs(st0 + (size_t)(r0 + r) * nv + v);
#pragma unroll
            for (int t = 0; t < KT; ++t) {
                if (t >= K) break;
                const float4 bv = reinterpret_cast<const float4*>(Bs + t * N)[v];
                const float4 cv = reinterpret_cast<const float4*>(Cs + t * N)[v];
                const float dt = dts[t * hpg + j], dA = dAs[t * hpg + j];
#pragma unroll
                for (int r = 0; r < RF; ++r) {
                    const float dx = dt * xs[t * XW + r0 + r];
                    float4 o;
                    o.x = fmaf(dA, hv[r].x, dx * bv.x);
                    o.y = fmaf(dA, hv[r].y, dx * bv.y);
                    o.z = fmaf(dA, hv[r].z, dx * bv.z);
                    o.w = fmaf(dA, hv[r].w, dx * bv.w);
                    float a = acc[r * KT + t];
                    a = fmaf(o.x, cv.x, a);
                    a = fmaf(o.y, cv.y, a);
                    a = fmaf(o.z, cv.z, a);
                    a = fmaf(o.w, cv.w, a);
                    acc[r * KT + t] = a;
                    hv[r] = o;
                }
            }
#pragma unroll
            for (int r = 0; r < RF; ++r) __stcs(st0 + (size_t)(r0 + r) * nv + v, hv[r]);
        }
        // sum each of the RF*KT partial dot products over the 32 lanes at once:
        // each step halves the values a lane keeps and trades the other half
        // with its partner, so lane l ends with the total of value e(l)
        int e = 0;
        int n = RF * KT;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            if (n > 1) {
                const bool up = (lane & o) != 0;
                const int half = n / 2;
#pragma unroll
                for (int k = 0; k < RF * KT / 2; ++k) {
                    if (k < half) {
                        const float send = up ? acc[k] : acc[k + half];
                        const float keep = up ? acc[k + half] : acc[k];
                        acc[k] = keep + __shfl_xor_sync(0xffffffffu, send, o);
                    }
                }
                if (up) e += half;
                n = half;
            } else {
                acc[0] += __shfl_xor_sync(0xffffffffu, acc[0], o);
            }
        }
        // one lane per value: those whose bits below the last halving step are 0
        const int rr = e / KT, tt = e % KT;
        if ((lane & (32 / (RF * KT) - 1)) == 0 && tt < K) {
            const int row = r0 + rr;         // j * P + pp
            const int h = h0 + j, pp = row % P;
            float yv = fmaf(Ds[j], xs[tt * XW + row], acc[0]);
            if (p.flags & kHasZ) {
                if constexpr (kZs) {
                    yv *= zs[tt * XW + row];
                } else {
                    const float zv = to_f32(zz[((size_t)i * K + tt) * H * P + h * P + pp]);
                    yv *= zv / (1.0f + expf(-zv));
                }
            }
            y[(((size_t)i * K + tt) * H + h) * P + pp] = from_f32<T>(yv);
        }
    }
}

// conv_pool[s] <- the last W-1 rows of [conv_pool[s] ; the row's K raw tokens]
// (one thread per (row, channel); it reads row K + j before writing row j,
// which it never reads again, so the update is in place).
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
    const int HW = p.W - 1, K = p.K;
    T* cp = static_cast<T*>(p.conv_pool) + (size_t)s * HW * Cdim;
    const T* x = static_cast<const T*>(p.xbc) + (size_t)i * K * Cdim;
    for (int j = 0; j < HW; ++j) {
        const int u = K + j;  // row of [conv state ; tokens]
        cp[(size_t)j * Cdim + c] = u < HW ? cp[(size_t)u * Cdim + c] : x[(size_t)(u - HW) * Cdim + c];
    }
}

// Shared memory of a decode CTA, with or without the staged SiLU(z).
size_t decode_smem_bytes(int H, int P, int N, int G, int K, bool stage_z)
{
    const size_t hpg = (size_t)(H / G);
    const size_t zb = stage_z ? hpg * P : 0;
    return sizeof(float) * ((size_t)K * (hpg * P + 2 * (size_t)N + 2 * hpg + zb) + hpg);
}
constexpr size_t kDecodeSmemMax = 200 * 1024;

template <typename T, int KT, int RF, bool kZs>
cudaError_t launch_kz(const DecodeParams& p, cudaStream_t st)
{
    const size_t smem = decode_smem_bytes(p.H, p.P, p.N, p.G, p.K, kZs);
    cudaError_t e = cudaFuncSetAttribute(decode_step_kernel<T, KT, RF, kZs>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    decode_step_kernel<T, KT, RF, kZs><<<dim3(p.G, p.R), kThreads, smem, st>>>(p);
    return cudaGetLastError();
}

// SiLU(z) staged in shared memory when it fits there beside the tokens' x
// columns (every shape this library admits fits without it)
template <typename T, int KT, int RF>
cudaError_t launch_kt(const DecodeParams& p, cudaStream_t st)
{
    if ((p.flags & kHasZ) && decode_smem_bytes(p.H, p.P, p.N, p.G, p.K, true) <= kDecodeSmemMax)
        return launch_kz<T, KT, RF, true>(p, st);
    return launch_kz<T, KT, RF, false>(p, st);
}

template <typename T>
cudaError_t launch_t(const DecodeParams& p, cudaStream_t st)
{
    // rows in flight per warp, measured at 256 rows x 128 heads (ms per call,
    // 4 / 2 rows): K = 2: 0.393 / 0.470; K = 4: 0.713 / 0.621; K = 8: 0.999 / 0.878
    if (p.K <= 1) return launch_kt<T, 1, 4>(p, st);
    if (p.K <= 2) return launch_kt<T, 2, 4>(p, st);
    if (p.K <= 4) return launch_kt<T, 4, 2>(p, st);
    if (p.K <= 8) return launch_kt<T, 8, 2>(p, st);
    return launch_kt<T, 16, 2>(p, st);
}

}  // namespace

bool decode_supports(int H, int P, int N, int G, int K)
{
    return N % 4 == 0 && P % 4 == 0 && K >= 1 && K <= kDecodeMaxTokens &&
           decode_smem_bytes(H, P, N, G, K, false) <= kDecodeSmemMax;
}

cudaError_t launch_decode_step(const DecodeParams& p, bool bf16, cudaStream_t st)
{
    if (p.R == 0) return cudaSuccess;
    return bf16 ? launch_t<__nv_bfloat16>(p, st) : launch_t<float>(p, st);
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
