// state_pass.cu -- the two steps of sequence-parallel state passing.
//
// A sequence's rows split into consecutive segments (one per GPU); each
// segment is scanned from a zero state, giving its own contribution h_k to
// the state, and its total decay Gamma_k, the last element of the
// cumulative sum of a = dt A over its rows (TensorRT-Model-Connect #2207
// "Implementation": gamma_S is that last element, and a chunk carries the
// state as h <- exp(min(gamma_S, 0)) h + its own terms).  Chaining the
// segments in order, h <- exp(min(Gamma_k, 0)) h + h_k, gives each segment's
// initial state and the sequence's final state.
//
// segment_decay_kernel: Gamma[b, h] over S rows.  One CTA per (sequence, 32
// heads): thread (row group r, head lane) sums rows r, r + 32, ... of one
// head, each warp reading 32 consecutive heads of a row (128 contiguous
// bytes of dt); the 32 partial sums of a head are added in fp64, so the
// total keeps its precision at the ~1e6 decays of a stiff segment.
// state_combine_kernel: out = exp(min(Gamma, 0)) h_prev + h_seg, 16 bytes a
// thread (HBM-bound: two states read, one written).
#include "internal.cuh"

namespace ssd {
namespace {

constexpr int kRowGroups = 32;

__global__ void __launch_bounds__(1024) segment_decay_kernel(SegmentParams p)
{
    __shared__ double part[kRowGroups][33];
    const int b = blockIdx.y;
    const int hl = threadIdx.x & 31, rg = threadIdx.x >> 5;
    const int h = blockIdx.x * 32 + hl;
    double acc = 0.0;
    if (h < p.H) {
        const float Ah = p.A[h];
        const float bias = p.dt_bias ? p.dt_bias[h] : 0.0f;
        const bool sp = (p.flags & kDtSoftplus) != 0;
        const float* dt = p.dt + (size_t)b * p.S * p.H + h;
#pragma unroll 4
        for (int t = rg; t < p.S; t += kRowGroups) {
            float v = __ldg(dt + (size_t)t * p.H);
            if (sp) v = softplus_f32(v + bias);
            acc += (double)(v * Ah);
        }
    }
    part[rg][hl] = acc;
    __syncthreads();
    if (rg == 0 && h < p.H) {
        double s = 0.0;
        for (int k = 0; k < kRowGroups; ++k) s += part[k][hl];
        p.gamma[(size_t)b * p.H + h] = (float)s;
    }
}

__global__ void state_combine_kernel(CombineParams p)
{
    const size_t n4 = (size_t)p.BH * p.PN / 4;  // float4s in a state set
    const size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= n4) return;
    const size_t bh = (i * 4) / p.PN;
    const float g = p.gamma[bh];
    const float e = expf(fminf(g, 0.0f));
    const float4 s = reinterpret_cast<const float4*>(p.h_seg)[i];
    float4 o = s;
    if (p.h_prev) {
        const float4 a = reinterpret_cast<const float4*>(p.h_prev)[i];
        o.x = fmaf(e, a.x, s.x);
        o.y = fmaf(e, a.y, s.y);
        o.z = fmaf(e, a.z, s.z);
        o.w = fmaf(e, a.w, s.w);
    }
    reinterpret_cast<float4*>(p.h_out)[i] = o;
}

}  // namespace

cudaError_t launch_segment_decay(const SegmentParams& p, cudaStream_t st)
{
    if (p.B == 0) return cudaSuccess;
    dim3 grid((p.H + 31) / 32, p.B);
    segment_decay_kernel<<<grid, 32 * kRowGroups, 0, st>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_state_combine(const CombineParams& p, cudaStream_t st)
{
    const size_t n4 = (size_t)p.BH * p.PN / 4;
    if (n4 == 0) return cudaSuccess;
    state_combine_kernel<<<(unsigned)((n4 + 255) / 256), 256, 0, st>>>(p);
    return cudaGetLastError();
}

}  // namespace ssd
