// scan_simt.cu -- the SSD scan on the fp32 pipes, exact row by row.
//
// TensorSharp nemotron.md 4.1 "Mamba2 SSM layer" (the recurrence
// state = exp(dt A) state + dt x B^T, y = state . C + D x) with the conv of
// section 3 in front.  This is the path for fp32 activations (tolerance 1e-4
// against the fp64 oracle) and for shapes the tensor-core path does not
// cover; it walks the rows of one (sequence, head) in order, so its result
// is the recurrence itself, in fp32.
//
// One CTA per (sequence b, head h).  The fp32 state [P,N] lives in
// registers: thread (p, q) holds state[p, j*NQ + q] for j < NPT, so the NQ
// threads of one p are adjacent lanes and y[p] is a shuffle reduction.  Rows
// are staged kRows at a time: the raw x_h | B_g | C_g columns of those rows
// (plus W-1 halo rows) go to shared memory, the conv + SiLU runs there, then
// the recurrence steps through the rows.
#include "internal.cuh"

namespace ssd {
namespace {

constexpr int kRows = 16;

struct SimtShape {
    int nq, npt, threads;
};

__host__ __device__ inline SimtShape simt_shape(int P, int N)
{
    // Aim for ~256 threads; NQ is a power of two dividing both N and 32.
    SimtShape s{1, N, P};
    int nq = 1;
    while (nq < 32 && N % (2 * nq) == 0 && (P * nq < 256 || N / nq > 32)) nq *= 2;
    s.nq = nq;
    s.npt = N / nq;
    s.threads = P * nq;
    return s;
}

template <typename T, int NPT>
__global__ void __launch_bounds__(1024) scan_simt_kernel(ScanParams p, int NQ)
{
    extern __shared__ float smem[];
    const int h = blockIdx.x, b = blockIdx.y;
    const int H = p.H, P = p.P, N = p.N, G = p.G;
    const int g = h / (H / G);
    const int CH = P + 2 * N;
    const int Cdim = H * P + 2 * G * N;
    const bool conv = p.conv_w != nullptr;
    const int HW = conv ? p.W - 1 : 0;  // halo rows
    const int nt = blockDim.x, tid = threadIdx.x;
    const int pp = tid / NQ, q = tid % NQ;
    // lanes present in this thread's warp (the last warp may be partial)
    const int wbase = tid & ~31;
    const unsigned lanes = nt - wbase >= 32 ? 0xffffffffu : ((1u << (nt - wbase)) - 1u);

    float* raw = smem;                          // [(kRows + HW) * CH]
    float* post = raw + (kRows + HW) * CH;      // [kRows * CH]
    float* halo = post + kRows * CH;            // [HW * CH]
    float* dts = halo + HW * CH;                // [kRows]
    float* dAs = dts + kRows;                   // [kRows]
    float* wsm = dAs + kRows;                   // conv taps [CH * W], then bias [CH]

    const T* xbc = static_cast<const T*>(p.xbc);
    const T* zz = static_cast<const T*>(p.z);
    T* y = static_cast<T*>(p.y);
    auto gch = [&](int c) -> int {
        return c < P ? h * P + c
                     : (c < P + N ? H * P + g * N + (c - P) : H * P + G * N + g * N + (c - P - N));
    };

    float st[NPT];
    const size_t sbase = (((size_t)b * H + h) * P + pp) * N;
#pragma unroll
    for (int j = 0; j < NPT; ++j) st[j] = p.h0 ? p.h0[sbase + j * NQ + q] : 0.0f;

    if (conv) {
        const T* cs = static_cast<const T*>(p.conv_state_in);
        for (int i = tid; i < HW * CH; i += nt) {
            const int r = i / CH, c = i % CH;
            halo[i] = cs ? to_f32(cs[((size_t)b * HW + r) * Cdim + gch(c)]) : 0.0f;
        }
        // the taps and bias of this head's columns, once (not per row and tap)
        for (int i = tid; i < CH * p.W; i += nt) wsm[i] = p.conv_w[(size_t)gch(i / p.W) * p.W + i % p.W];
        for (int c = tid; c < CH; c += nt) wsm[CH * p.W + c] = p.conv_b ? p.conv_b[gch(c)] : 0.0f;
    }
    // 16-byte row loads when every column segment (x | B | C) is a whole number
    // of vectors (segment starts are then vector aligned too)
    constexpr int VEC = 16 / (int)sizeof(T);
    const bool vec_rows = P % VEC == 0 && N % VEC == 0;
    const float Ah = p.A[h];
    const float bias = p.dt_bias ? p.dt_bias[h] : 0.0f;
    const float Dh = p.D ? p.D[h] : 0.0f;

    for (int t0 = 0; t0 < p.S; t0 += kRows) {
        const int rows = min(kRows, p.S - t0);
        __syncthreads();
        for (int i = tid; i < HW * CH; i += nt) raw[i] = halo[i];
        if (vec_rows) {
            const int vpr = CH / VEC;  // vectors per row
            for (int i = tid; i < rows * vpr; i += nt) {
                const int r = i / vpr, c = (i % vpr) * VEC;
                const uint4 v = __ldg(reinterpret_cast<const uint4*>(
                    xbc + ((size_t)b * p.S + t0 + r) * Cdim + gch(c)));
                const T* e = reinterpret_cast<const T*>(&v);
#pragma unroll
                for (int k = 0; k < VEC; ++k) raw[HW * CH + r * CH + c + k] = to_f32(e[k]);
            }
        } else {
            for (int i = tid; i < rows * CH; i += nt) {
                const int r = i / CH, c = i % CH;
                raw[HW * CH + i] = to_f32(xbc[((size_t)b * p.S + t0 + r) * Cdim + gch(c)]);
            }
        }
        for (int r = tid; r < rows; r += nt) {
            float v = p.dt[((size_t)b * p.S + t0 + r) * H + h];
            if (p.flags & kDtSoftplus) v = softplus_f32(v + bias);
            dts[r] = v;
            dAs[r] = expf(v * Ah);
        }
        __syncthreads();
        for (int i = tid; i < rows * CH; i += nt) {
            const int r = i / CH, c = i % CH;
            if (conv) {
                float v = wsm[CH * p.W + c];
                for (int k = 0; k < p.W; ++k) v = fmaf(wsm[c * p.W + k], raw[(r + k) * CH + c], v);
                post[i] = __fdividef(v, 1.0f + __expf(-v));  // silu
            } else {
                post[i] = raw[i];
            }
        }
        __syncthreads();
        for (int i = tid; i < HW * CH; i += nt) halo[i] = raw[rows * CH + i];

        for (int r = 0; r < rows; ++r) {
            const float* row = post + r * CH;
            const float xv = row[pp];
            const float dt = dts[r], dA = dAs[r];
            const float dtx = dt * xv;
            float acc = 0.0f;
#pragma unroll
            for (int j = 0; j < NPT; ++j) {
                const int n = j * NQ + q;
                st[j] = fmaf(dA, st[j], dtx * row[P + n]);
                acc = fmaf(st[j], row[P + N + n], acc);
            }
            for (int off = NQ / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(lanes, acc, off);
            if (q == 0) {
                const int t = t0 + r;
                float yv = fmaf(Dh, xv, acc);
                if (p.flags & kHasZ) {
                    const float zv = to_f32(zz[((size_t)b * p.S + t) * (H * P) + h * P + pp]);
                    yv *= zv / (1.0f + expf(-zv));
                }
                y[(((size_t)b * p.S + t) * H + h) * P + pp] = from_f32<T>(yv);
            }
        }
    }
#pragma unroll
    for (int j = 0; j < NPT; ++j) p.hS[sbase + j * NQ + q] = st[j];
}

template <typename T, int NPT>
cudaError_t launch_t(const ScanParams& p, const SimtShape& s, cudaStream_t st)
{
    const int CH = p.P + 2 * p.N;
    const int HW = p.conv_w ? p.W - 1 : 0;
    const size_t smem = sizeof(float) * ((size_t)(kRows + HW) * CH + (size_t)kRows * CH +
                                         (size_t)HW * CH + 2 * kRows +
                                         (p.conv_w ? (size_t)CH * (p.W + 1) : 0));
    auto kern = scan_simt_kernel<T, NPT>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    dim3 grid(p.H, p.B);
    kern<<<grid, s.threads, smem, st>>>(p, s.nq);
    return cudaGetLastError();
}

template <typename T>
cudaError_t launch_dispatch(const ScanParams& p, cudaStream_t st)
{
    const SimtShape s = simt_shape(p.P, p.N);
    switch (s.npt) {
        case 1: return launch_t<T, 1>(p, s, st);
        case 2: return launch_t<T, 2>(p, s, st);
        case 4: return launch_t<T, 4>(p, s, st);
        case 8: return launch_t<T, 8>(p, s, st);
        case 16: return launch_t<T, 16>(p, s, st);
        case 32: return launch_t<T, 32>(p, s, st);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

bool scan_simt_supports(int P, int N)
{
    const SimtShape s = simt_shape(P, N);
    if (s.threads > 1024) return false;
    if (s.npt != 1 && s.npt != 2 && s.npt != 4 && s.npt != 8 && s.npt != 16 && s.npt != 32)
        return false;
    if (s.npt * s.nq != N) return false;
    const size_t smem = sizeof(float) * ((size_t)(2 * kRows + 2 * 7) * (P + 2 * N) + 2 * kRows);
    return smem <= 227 * 1024;
}

cudaError_t launch_scan_simt(const ScanParams& p, bool bf16, cudaStream_t st)
{
    if (p.B == 0) return cudaSuccess;
    return bf16 ? launch_dispatch<__nv_bfloat16>(p, st) : launch_dispatch<float>(p, st);
}

}  // namespace ssd
