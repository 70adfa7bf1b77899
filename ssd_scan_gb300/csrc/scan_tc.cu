// scan_tc.cu -- the chunked SSD scan on the 5th-generation tensor cores
// (tcgen05 + TMEM + TMA), bf16 activations, fp32 state, 128-row chunks.
//
// The chunk form of TensorRT-Model-Connect #2207 ("Implementation"): with
// a_t = dt_t A and gamma_t = sum_{i<=t} a_i inside a chunk,
//   y_t = sum_{s<=t} (C_t . B_s) exp(gamma_t - gamma_s) dt_s x_s
//         + exp(gamma_t) C_t h  +  D x_t
//   h  <- exp(gamma_Q) h + sum_s exp(gamma_Q - gamma_s) dt_s x_s B_s^T
// where gamma_Q is the last element of the cumulative sum (never a separate
// reduction) and every exponent is clamped at <= 0.  It equals the row
// recurrence of TensorSharp nemotron.md 4.1 up to rounding.
//
// One CTA walks all chunks of one (sequence b, head h); the fp32 state
// h [P=64, N=128] stays in registers (thread n owns column n) for the whole
// sequence.  Per chunk, four dense contractions run on the tensor cores, each
// 128 x {128,64} x 128, bf16 operands in shared memory, fp32 accumulators in
// TMEM:
//   G1  CB[t,s] = C_t . B_s                 A = C  (TMA tile)   B = B (TMA)
//   G3  Yo[t,p] = C_t . h[p,:]              A = C               B = bf16(h) rows [n][p]
//   G4  dH[n,p] = sum_s B[s,n] w_s x[s,p]   A = B^T (MN-major)  B = (w x) rows [s][p]
//   G2  Yd[t,p] = sum_s M[t,s] x[s,p]       A = M (masked, decayed CB)  B = x rows [s][p]
// Every operand the threads write is row-major with 16-byte stores; the
// operands whose K index runs along rows are read MN-major by the MMA.
// Two warpgroups (256 threads): the warps of each read one 32-lane quarter of
// TMEM (row t of the chunk for CB / Yd / Yo, state row n for dH) and the two
// warpgroups split the columns.  The threads compute dt and the cumulative
// sum (a double-float warp-shuffle scan), the x conv + SiLU from the raw TMA
// tile (4 rows x 8 channels per thread), the causal mask with its decays
// (blocks above the diagonal are written as zeros without a TMEM read; when
// the chunk's total decay is moderate the decay factors into exp(gamma_t) and
// exp(-gamma_s) dt_s, otherwise each entry takes its own clamped exponent),
// the state update and the epilogue y = Yd + exp(gamma_t) Yo, times silu(z);
// D x enters G2 through D on the diagonal of M.  Thread 0 issues the TMA
// loads and the MMAs.  B and C of a group are read by each of its heads'
// CTAs; they come from L2 after the first.
#include "internal.cuh"
#include "sm100.cuh"

#include <cudaTypedefs.h>

#include <mutex>

namespace ssd {
namespace {

using namespace sm100;

constexpr int Q = 128;   // rows per chunk
constexpr int P = 64;    // head dim
constexpr int N = 128;   // state dim
constexpr int kThreads = 256;  // two warpgroups; each owns one half of the columns
constexpr int kMaxW = 4;       // conv taps handled in the kernel (W-1 carried rows)
constexpr uint64_t kWaitNs = 2000000000ull;  // bound on any single wait: 2 s

// G1: A, B K-major.  G2, G3: A K-major, B MN-major (row tiles [k][p]).
// G4: A = B^T read MN-major from the B tile, B MN-major.
constexpr uint32_t kIdCB = idesc_bf16_f32(128, 128, false, false);
constexpr uint32_t kIdY = idesc_bf16_f32(128, 64, false, true);
constexpr uint32_t kIdState = idesc_bf16_f32(128, 64, true, true);

struct __align__(1024) TcSmem {
    __nv_bfloat16 C[2][Q * 64];    // C tile [t][n]: 2 panels of 64 n (TMA, SW128)
    __nv_bfloat16 B[2][Q * 64];    // B tile [s][n]
    __nv_bfloat16 Xr[Q * 64];      // x tile [t][p] (raw rows when the conv is fused)
    __nv_bfloat16 Z[Q * 64];       // z tile [t][p]
    __nv_bfloat16 XR[Q * 64];      // post-conv x rows [s][p] (SW128): G2's B
    __nv_bfloat16 XW[Q * 64];      // (w o x) rows [s][p]: G4's B
    __nv_bfloat16 M[2][Q * 64];    // masked decayed CB [t][s]: G2's A (K-major)
    __nv_bfloat16 Hs[N * 64];      // bf16 state rows [n][p]: G3's B
    __nv_bfloat16 carry[2][kMaxW - 1][P];  // raw x rows before the chunk, by parity
    float2 wconv[P / 2][kMaxW];    // taps of channel pairs (front-padded with zeros)
    float2 bconv[P / 2];
    float g2h[Q], g2l[Q];          // gamma * log2(e), double-float (hi, lo)
    float dts[Q];                  // dt_s
    float vfac[Q];                 // exp(-gamma_s) dt_s (factored mask only)
    float wrow[Q];                 // w_s = exp(min(gamma_Q - gamma_s, 0)) dt_s
    float wsum_hi[4], wsum_lo[4];
    uint64_t bar_ld, bar_z, bar_g1, bar_g34, bar_g2;
    uint32_t tmem_base;
};

constexpr size_t kSmemBytes = sizeof(TcSmem) + 1024;

// Below this total chunk decay (log2 units) the mask factors as
// exp(gamma_t) * exp(-gamma_s): every factor stays within fp32 (2^90 < 2^127).
constexpr float kFactorMinLog2 = -90.0f;

__device__ __forceinline__ float tanh_fast(float v)
{
    float t;
    asm("tanh.approx.f32 %0, %1;" : "=f"(t) : "f"(v));
    return t;
}

// silu(v) = v sigmoid(v) = 0.5 v (1 + tanh(v / 2)), two lanes at a time.
__device__ __forceinline__ float2 silu2(float2 v)
{
    const float2 hv = __fmul2_rn(v, make_float2(0.5f, 0.5f));
    return __ffma2_rn(hv, make_float2(tanh_fast(hv.x), tanh_fast(hv.y)), hv);
}

__device__ __forceinline__ float ex2_fast(float v)
{
    float r;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(v));
    return r;
}

// (hi, lo) += (bhi, blo), double-float (TwoSum then renormalise).
__device__ __forceinline__ void df_add(float& hi, float& lo, float bhi, float blo)
{
    const float s = hi + bhi;
    const float v = s - hi;
    float e = (hi - (s - v)) + (bhi - v);
    e += lo + blo;
    hi = s + e;
    lo = e - (hi - s);
}

__device__ __forceinline__ void unpack4x2(uint4 r, float2* f)
{
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&r);
#pragma unroll
    for (int i = 0; i < 4; ++i) f[i] = __bfloat1622float2(h[i]);
}

__device__ __forceinline__ uint32_t pack2(float2 a)
{
    __nv_bfloat162 h = __float22bfloat162_rn(a);
    return *reinterpret_cast<uint32_t*>(&h);
}

__device__ __forceinline__ uint4 pack4x2(const float2* f)
{
    return make_uint4(pack2(f[0]), pack2(f[1]), pack2(f[2]), pack2(f[3]));
}

// byte offset of 16-byte chunk j of row r in a SW128 tile of 64-element rows.
__device__ __forceinline__ uint32_t chunk_off(int r, int j)
{
    return (uint32_t)(r * 128 + (((j ^ r) & 7) << 4));
}

template <typename T>
__device__ __forceinline__ T& at(void* base, uint32_t off)
{
    return *reinterpret_cast<T*>(reinterpret_cast<uint8_t*>(base) + off);
}

__global__ void __launch_bounds__(kThreads, 1)
    scan_tc_kernel(const __grid_constant__ CUtensorMap map_x,
                   const __grid_constant__ CUtensorMap map_bc,
                   const __grid_constant__ CUtensorMap map_z, const TcScanParams p)
{
    extern __shared__ uint8_t smem_raw[];
    TcSmem& s = *reinterpret_cast<TcSmem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~uintptr_t(1023));
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int quarter = warp & 3;         // TMEM lane quarter of this warp
    const int half = warp >> 2;           // column half of this warpgroup
    const int row = 32 * quarter + lane;  // chunk row t (or state column n) of this thread
    const int h = blockIdx.x, b = blockIdx.y;
    const int H = p.H, G = p.G, W = p.W;
    const int g = h / (H / G);
    const int Cdim = H * P + 2 * G * N;
    const int nchunks = (p.S + Q - 1) / Q;
    const bool has_z = (p.flags & kHasZ) != 0;
    const bool softplus = (p.flags & kDtSoftplus) != 0;

    if (tid == 0) {
        mbar_init(&s.bar_ld, 1);
        mbar_init(&s.bar_z, 1);
        mbar_init(&s.bar_g1, 1);
        mbar_init(&s.bar_g34, 1);
        mbar_init(&s.bar_g2, 1);
        fence_mbar_init();
        prefetch_tmap(&map_x);
        prefetch_tmap(&map_bc);
        if (has_z) prefetch_tmap(&map_z);
    }
    if (warp == 0) {
        tmem_alloc(&s.tmem_base, 512);
        tmem_relinquish();
    }
    if (p.conv) {
        for (int i = tid; i < P / 2; i += kThreads) {
            float w4[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
            for (int e = 0; e < 2; ++e)
                for (int k = 0; k < W; ++k)
                    w4[e][kMaxW - W + k] = p.conv_w[(size_t)(h * P + 2 * i + e) * W + k];
            for (int k = 0; k < kMaxW; ++k) s.wconv[i][k] = make_float2(w4[0][k], w4[1][k]);
            s.bconv[i] = p.conv_b ? make_float2(p.conv_b[h * P + 2 * i], p.conv_b[h * P + 2 * i + 1])
                                  : make_float2(0.f, 0.f);
        }
        // raw rows -3..-1 before chunk 0: the last rows of the conv state (or zeros)
        const __nv_bfloat16* cs = static_cast<const __nv_bfloat16*>(p.conv_state_in);
        for (int i = tid; i < (kMaxW - 1) * P; i += kThreads) {
            const int j = i / P, pp = i % P;
            const int sr = (W - 1) + (j - (kMaxW - 1));
            __nv_bfloat16 v = __float2bfloat16_rn(0.0f);
            if (cs && sr >= 0) v = cs[((size_t)b * (W - 1) + sr) * Cdim + h * P + pp];
            s.carry[0][j][pp] = v;
        }
    }

    // The fp32 state: thread (n = row, half) owns h[32*half .. 32*half+31][n],
    // as 16 pairs of consecutive p.
    const int n = row;
    const int p0 = 32 * half;
    const size_t sbase = ((size_t)b * H + h) * P * N;
    float2 hreg[16];
#pragma unroll
    for (int i = 0; i < 16; ++i)
        hreg[i] = p.h0 ? make_float2(p.h0[sbase + (size_t)(p0 + 2 * i) * N + n],
                                     p.h0[sbase + (size_t)(p0 + 2 * i + 1) * N + n])
                       : make_float2(0.f, 0.f);
    // Hs row n holds bf16 h[0..63][n]; this thread writes its 4 chunks of 8 p
    auto store_h = [&]() {
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4)
            at<uint4>(s.Hs, chunk_off(n, 4 * half + q4)) = pack4x2(&hreg[4 * q4]);
    };
    store_h();

    // conv work split: thread (cj = channel group of 8, rb = block of 4 rows)
    const int cj = tid & 7, rb = tid >> 3;

    const float Ah = p.A[h];
    const float bias = p.dt_bias ? p.dt_bias[h] : 0.0f;
    const float Dh = p.D ? p.D[h] : 0.0f;
    float dt_next = (half == 0 && row < p.S) ? p.dt[((size_t)b * p.S + row) * H + h] : 0.0f;

    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    float2 wq[4][kMaxW], bq[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        bq[e] = make_float2(0.f, 0.f);
#pragma unroll
        for (int k = 0; k < kMaxW; ++k) wq[e][k] = make_float2(0.f, 0.f);
    }
    if (p.conv) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            bq[e] = s.bconv[4 * cj + e];
#pragma unroll
            for (int k = 0; k < kMaxW; ++k) wq[e][k] = s.wconv[4 * cj + e][k];
        }
    }
    const uint32_t tbase = s.tmem_base;
    const uint32_t lane_off = (uint32_t)(32 * quarter) << 16;
    const uint32_t t_cb = tbase, t_yd = tbase + 128, t_yo = tbase + 192, t_st = tbase + 256;

    const int xB = p.bc_col0 + g * N;          // first B column in the bc source
    const int xC = p.bc_col0 + G * N + g * N;  // first C column
    auto issue_main = [&](int c) {
        mbar_arrive_expect_tx(&s.bar_ld, 5 * Q * 64 * 2);
        tma_load_3d(s.C[0], &map_bc, &s.bar_ld, xC, c * Q, b);
        tma_load_3d(s.C[1], &map_bc, &s.bar_ld, xC + 64, c * Q, b);
        tma_load_3d(s.B[0], &map_bc, &s.bar_ld, xB, c * Q, b);
        tma_load_3d(s.B[1], &map_bc, &s.bar_ld, xB + 64, c * Q, b);
        tma_load_3d(s.Xr, &map_x, &s.bar_ld, h * P, c * Q, b);
    };
    auto issue_z = [&](int c) {
        mbar_arrive_expect_tx(&s.bar_z, Q * 64 * 2);
        tma_load_3d(s.Z, &map_z, &s.bar_z, h * P, c * Q, b);
    };
    if (tid == 0 && nchunks > 0) {
        issue_main(0);
        if (has_z) issue_z(0);
    }

    const uint32_t aC = smem_u32(s.C), aB = smem_u32(s.B), aXR = smem_u32(s.XR);
    const uint32_t aXW = smem_u32(s.XW), aM = smem_u32(s.M), aH = smem_u32(s.Hs);
    constexpr float kLog2e = 1.4426950408889634f;

    bool ok = true;
    for (int c = 0; c < nchunks; ++c) {
        const uint32_t par = c & 1;
        const int r0 = c * Q;
        const int rows = min(Q, p.S - r0);

        // ---- dt and the cumulative sum of a = dt A (double-float), warpgroup 0 ----
        float ghi = 0.0f, glo = 0.0f, dt = 0.0f;
        if (half == 0) {
            if (row < rows) dt = softplus ? softplus_f32(dt_next + bias) : dt_next;
            if (c + 1 < nchunks)
                dt_next = r0 + Q + row < p.S ? p.dt[((size_t)b * p.S + r0 + Q + row) * H + h] : 0.0f;
            ghi = dt * Ah;
#pragma unroll
            for (int d = 1; d < 32; d <<= 1) {
                const float ohi = __shfl_up_sync(0xffffffffu, ghi, d);
                const float olo = __shfl_up_sync(0xffffffffu, glo, d);
                if (lane >= d) df_add(ghi, glo, ohi, olo);
            }
            if (lane == 31) {
                s.wsum_hi[quarter] = ghi;
                s.wsum_lo[quarter] = glo;
            }
        }
        __syncthreads();
        if (half == 0) {
            for (int w2 = 0; w2 < quarter; ++w2) df_add(ghi, glo, s.wsum_hi[w2], s.wsum_lo[w2]);
            s.g2h[row] = ghi * kLog2e;
            s.g2l[row] = glo * kLog2e;
            s.dts[row] = dt;
        }

        // ---- this chunk's tiles; G1 = C B^T ---------------------------------------
        ok = ok && mbar_wait_ns(&s.bar_ld, par, kWaitNs);
        if (tid == 0 && ok) {
            tc_fence_after();
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const uint32_t off = (k >> 2) * (Q * 128) + (k & 3) * 32;
                mma_bf16_ss(t_cb, sdesc_sw128(aC + off, 16, 1024), sdesc_sw128(aB + off, 16, 1024),
                            kIdCB, k > 0);
            }
            mma_commit(&s.bar_g1);
        }
        __syncthreads();
        // gamma of this thread's row t and of the chunk's last row (log2 units)
        const float g2h_t = s.g2h[row], g2l_t = s.g2l[row];
        const float gLh = s.g2h[rows - 1], gLl = s.g2l[rows - 1];
        const float decay_t = ex2_fast(fminf(g2h_t + g2l_t, 0.0f));  // exp(min(gamma_t, 0))
        const float decay_S = ex2_fast(fminf(gLh + gLl, 0.0f));      // exp(min(gamma_Q, 0))
        // factored mask: a <= 0 everywhere (A <= 0) and gamma_Q not too negative
        const bool factored = Ah <= 0.0f && gLh + gLl >= kFactorMinLog2;
        if (half == 0) {
            const float dtt = s.dts[row];
            s.wrow[row] = row < rows ? ex2_fast(fminf((gLh - g2h_t) + (gLl - g2l_t), 0.0f)) * dtt
                                     : 0.0f;
            if (factored) s.vfac[row] = ex2_fast(-(g2h_t + g2l_t)) * dtt;
        }
        __syncthreads();

        // ---- x: conv + SiLU of 4 rows x 8 channels per thread -> x, w x rows ------
        {
            const int t0 = 4 * rb;
            float2 xo[4][4];  // [row][channel pair]
            if (p.conv) {
                float2 win[7][4];  // raw rows t0-3 .. t0+3
#pragma unroll
                for (int k = 0; k < 7; ++k) {
                    const int r = t0 - 3 + k;
                    const uint4 raw = r >= 0 ? at<const uint4>(s.Xr, chunk_off(r, cj))
                                             : *reinterpret_cast<const uint4*>(&s.carry[par][r + 3][8 * cj]);
                    unpack4x2(raw, win[k]);
                    if (r >= Q - (kMaxW - 1))  // rows Q-3..Q-1 carry into the next chunk
                        *reinterpret_cast<uint4*>(&s.carry[par ^ 1][r - (Q - 3)][8 * cj]) = raw;
                }
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const bool valid = t0 + i < rows;
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        float2 v = bq[e];
#pragma unroll
                        for (int k = 0; k < kMaxW; ++k) v = __ffma2_rn(wq[e][k], win[i + k][e], v);
                        xo[i][e] = valid ? silu2(v) : make_float2(0.f, 0.f);
                    }
                }
            } else {
#pragma unroll
                for (int i = 0; i < 4; ++i) unpack4x2(at<const uint4>(s.Xr, chunk_off(t0 + i, cj)), xo[i]);
            }
            const float4 w4 = *reinterpret_cast<const float4*>(&s.wrow[t0]);
            const float wr[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                float2 xw[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) xw[e] = __fmul2_rn(make_float2(wr[i], wr[i]), xo[i][e]);
                const uint32_t off = chunk_off(t0 + i, cj);
                at<uint4>(s.XR, off) = pack4x2(xo[i]);
                at<uint4>(s.XW, off) = pack4x2(xw);
            }
        }
        fence_proxy_async_smem();
        __syncthreads();
        if (tid == 0 && ok) {
            tc_fence_after();
#pragma unroll
            for (int k = 0; k < 8; ++k) {  // G3: Yo = C h^T  (K = n, 16 rows of Hs per step)
                const uint32_t offc = (k >> 2) * (Q * 128) + (k & 3) * 32;
                mma_bf16_ss(t_yo, sdesc_sw128(aC + offc, 16, 1024),
                            sdesc_sw128(aH + k * 2048, 8192, 1024), kIdY, k > 0);
            }
#pragma unroll
            for (int k = 0; k < 8; ++k) {  // G4: dH = B^T (w x)  (K = s)
                mma_bf16_ss(t_st, sdesc_sw128(aB + k * 2048, Q * 128, 1024),
                            sdesc_sw128(aXW + k * 2048, 8192, 1024), kIdState, k > 0);
            }
            mma_commit(&s.bar_g34);
        }

        // ---- causal mask with decays: M[t,s] = CB[t,s] exp(gamma_t - gamma_s) dt_s,
        //      plus D on the diagonal (so G2 also adds D x_t) -------------------------
        ok = ok && mbar_wait_ns(&s.bar_g1, par, kWaitNs);
        tc_fence_after();
        {
            const int t = row;
#pragma unroll
            for (int cb2 = 0; cb2 < 2; ++cb2) {
                const int cc = 2 * half + cb2;  // 32-column block of this thread
                __nv_bfloat16* mpanel = s.M[cc >> 1];
                if (cc > quarter) {  // strictly above the diagonal for the whole warp
#pragma unroll
                    for (int q4 = 0; q4 < 4; ++q4)
                        at<uint4>(mpanel, chunk_off(t, (cc & 1) * 4 + q4)) = make_uint4(0, 0, 0, 0);
                    continue;
                }
                float v[32];
                tmem_ld32(t_cb + lane_off + cc * 32, v);
                tmem_ld_wait();
                const bool diag = cc == quarter;
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4) {
                    const int sb = cc * 32 + q4 * 8;
                    float2 m[4];
                    if (factored) {
                        const float4 f0 = *reinterpret_cast<const float4*>(&s.vfac[sb]);
                        const float4 f1 = *reinterpret_cast<const float4*>(&s.vfac[sb + 4]);
                        const float2 uu = make_float2(decay_t, decay_t);
                        m[0] = __fmul2_rn(__fmul2_rn(make_float2(v[q4 * 8 + 0], v[q4 * 8 + 1]), make_float2(f0.x, f0.y)), uu);
                        m[1] = __fmul2_rn(__fmul2_rn(make_float2(v[q4 * 8 + 2], v[q4 * 8 + 3]), make_float2(f0.z, f0.w)), uu);
                        m[2] = __fmul2_rn(__fmul2_rn(make_float2(v[q4 * 8 + 4], v[q4 * 8 + 5]), make_float2(f1.x, f1.y)), uu);
                        m[3] = __fmul2_rn(__fmul2_rn(make_float2(v[q4 * 8 + 6], v[q4 * 8 + 7]), make_float2(f1.z, f1.w)), uu);
                    } else {
                        const float4 h0 = *reinterpret_cast<const float4*>(&s.g2h[sb]);
                        const float4 h1 = *reinterpret_cast<const float4*>(&s.g2h[sb + 4]);
                        const float4 l0 = *reinterpret_cast<const float4*>(&s.g2l[sb]);
                        const float4 l1 = *reinterpret_cast<const float4*>(&s.g2l[sb + 4]);
                        const float4 d0 = *reinterpret_cast<const float4*>(&s.dts[sb]);
                        const float4 d1 = *reinterpret_cast<const float4*>(&s.dts[sb + 4]);
                        const float gh[8] = {h0.x, h0.y, h0.z, h0.w, h1.x, h1.y, h1.z, h1.w};
                        const float gl[8] = {l0.x, l0.y, l0.z, l0.w, l1.x, l1.y, l1.z, l1.w};
                        const float ds[8] = {d0.x, d0.y, d0.z, d0.w, d1.x, d1.y, d1.z, d1.w};
                        float mm[8];
#pragma unroll
                        for (int e = 0; e < 8; ++e) {
                            const float ex = (g2h_t - gh[e]) + (g2l_t - gl[e]);
                            mm[e] = v[q4 * 8 + e] * ds[e] * ex2_fast(fminf(ex, 0.0f));
                        }
#pragma unroll
                        for (int e = 0; e < 4; ++e) m[e] = make_float2(mm[2 * e], mm[2 * e + 1]);
                    }
                    if (diag) {
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const int s0 = sb + 2 * e;
                            m[e].x = s0 < t ? m[e].x : (s0 == t ? m[e].x + Dh : 0.0f);
                            m[e].y = s0 + 1 < t ? m[e].y : (s0 + 1 == t ? m[e].y + Dh : 0.0f);
                        }
                    }
                    at<uint4>(mpanel, chunk_off(t, (cc & 1) * 4 + q4)) = pack4x2(m);
                }
            }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();
        if (tid == 0 && ok) {
            tc_fence_after();
#pragma unroll
            for (int k = 0; k < 8; ++k) {  // G2: Yd = M x  (K = s)
                const uint32_t offm = (k >> 2) * (Q * 128) + (k & 3) * 32;
                mma_bf16_ss(t_yd, sdesc_sw128(aM + offm, 16, 1024),
                            sdesc_sw128(aXR + k * 2048, 8192, 1024), kIdY, k > 0);
            }
            mma_commit(&s.bar_g2);
        }

        // ---- state: h <- exp(gamma_Q) h + dH; tiles of the next chunk --------------
        ok = ok && mbar_wait_ns(&s.bar_g34, par, kWaitNs);
        tc_fence_after();
        if (tid == 0 && ok && c + 1 < nchunks) issue_main(c + 1);
        {
            float v[32];
            tmem_ld32(t_st + lane_off + p0, v);
            tmem_ld_wait();
            const float2 dd = make_float2(decay_S, decay_S);
#pragma unroll
            for (int i = 0; i < 16; ++i)
                hreg[i] = __ffma2_rn(dd, hreg[i], make_float2(v[2 * i], v[2 * i + 1]));
            store_h();
        }

        // ---- epilogue: y = Yd + exp(gamma_t) Yo (Yd holds D x), gated -------------
        ok = ok && mbar_wait_ns(&s.bar_g2, par, kWaitNs);
        if (has_z) ok = ok && mbar_wait_ns(&s.bar_z, par, kWaitNs);
        tc_fence_after();
        {
            const int t = row;
            float yd[32], yo[32];
            tmem_ld32(t_yd + lane_off + p0, yd);
            tmem_ld32(t_yo + lane_off + p0, yo);
            tmem_ld_wait();
            uint4* yrow = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.y) +
                                                   (((size_t)b * p.S + r0 + t) * H + h) * P + p0);
            const float2 dec = make_float2(decay_t, decay_t);
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) {
                float2 out[4], zv[4];
                if (has_z) unpack4x2(at<const uint4>(s.Z, chunk_off(t, 4 * half + q4)), zv);
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int k = q4 * 8 + 2 * e;
                    float2 yv = __ffma2_rn(dec, make_float2(yo[k], yo[k + 1]),
                                           make_float2(yd[k], yd[k + 1]));
                    if (has_z) yv = __fmul2_rn(yv, silu2(zv[e]));
                    out[e] = yv;
                }
                if (t < rows) yrow[q4] = pack4x2(out);
            }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        if (__syncthreads_or(!ok)) ok = false;
        if (!ok) break;
        if (tid == 0 && has_z && c + 1 < nchunks) issue_z(c + 1);
    }

    if (ok) {
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            p.hS[sbase + (size_t)(p0 + 2 * i) * N + n] = hreg[i].x;
            p.hS[sbase + (size_t)(p0 + 2 * i + 1) * N + n] = hreg[i].y;
        }
    } else if (tid == 0) {
        atomicOr(p.err, kErrTimeout);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tbase, 512);
}

// ---- host side ------------------------------------------------------------------

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

bool encode_fn()
{
    std::call_once(g_encode_once, [] {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    });
    return g_encode != nullptr;
}

// 3-D map over rows of `cols` bf16: dims {cols, S, B}, box {64, 128, 1}, SW128.
bool make_map(CUtensorMap* m, const void* base, int cols, int S, int B)
{
    cuuint64_t dims[3] = {(cuuint64_t)cols, (cuuint64_t)S, (cuuint64_t)B};
    cuuint64_t strides[2] = {(cuuint64_t)cols * 2, (cuuint64_t)cols * 2 * (cuuint64_t)S};
    cuuint32_t box[3] = {64, (cuuint32_t)Q, 1};
    cuuint32_t es[3] = {1, 1, 1};
    return g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides,
                    box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool scan_tc_supports(int P_, int N_) { return P_ == P && N_ == N; }

cudaError_t launch_scan_tc(const TcScanParams& p, cudaStream_t st)
{
    if (p.B == 0 || p.S == 0) return cudaSuccess;
    if (p.W > kMaxW || !encode_fn()) return cudaErrorNotSupported;
    const int Cdim = p.H * P + 2 * p.G * N;
    CUtensorMap mx, mbc, mz;
    if (!make_map(&mx, p.xbc, Cdim, p.S, p.B)) return cudaErrorInvalidValue;
    if (!make_map(&mbc, p.bc, p.bc_stride, p.S, p.B)) return cudaErrorInvalidValue;
    if (p.z != nullptr) {
        if (!make_map(&mz, p.z, p.H * P, p.S, p.B)) return cudaErrorInvalidValue;
    } else {
        mz = mx;
    }
    cudaError_t e = cudaFuncSetAttribute(scan_tc_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)kSmemBytes);
    if (e != cudaSuccess) return e;
    dim3 grid(p.H, p.B);
    scan_tc_kernel<<<grid, kThreads, kSmemBytes, st>>>(mx, mbc, mz, p);
    return cudaGetLastError();
}

}  // namespace ssd
