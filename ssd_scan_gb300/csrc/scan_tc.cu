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
//   G3  Yo[t,p] = C_t . h[p,:]              A = C               B = bf16(h)
//   G4  dH[n,p] = sum_s B[s,n] w_s x[s,p]   A = B^T (MN-major)  B = (w x)^T
//   G2  Yd[t,p] = sum_s M[t,s] x[s,p]       A = M (masked, decayed CB)  B = x^T
// The 128 threads (one warpgroup) own one TMEM lane each: row t of the
// chunk for CB / Yd / Yo, state row n for dH.  They compute dt and the
// cumulative sum (a double-float warp-shuffle scan), the x conv + SiLU from
// the raw TMA tile, the causal mask with its decays, the state update and the
// epilogue y = Yd + exp(gamma_t) Yo + D x, times silu(z).  Thread 0 issues
// the TMA loads and the MMAs.  B and C of a group are read by each of its
// heads' CTAs; they come from L2 after the first.
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
constexpr int kThreads = 128;
constexpr int kMaxW = 4;  // conv taps handled in the kernel (W-1 carried rows)
constexpr uint64_t kWaitNs = 2000000000ull;  // bound on any single wait: 2 s

constexpr uint32_t kIdCB = idesc_bf16_f32(128, 128, false, false);
constexpr uint32_t kIdY = idesc_bf16_f32(128, 64, false, false);
constexpr uint32_t kIdState = idesc_bf16_f32(128, 64, true, false);

struct __align__(1024) TcSmem {
    __nv_bfloat16 C[2][Q * 64];    // C tile [t][n]: 2 panels of 64 n (TMA, SW128)
    __nv_bfloat16 B[2][Q * 64];    // B tile [s][n]
    __nv_bfloat16 Xr[Q * 64];      // x tile [t][p] (raw rows when the conv is fused)
    __nv_bfloat16 Z[Q * 64];       // z tile [t][p]
    __nv_bfloat16 XT[2][P * 64];   // x^T [p][s], 2 panels of 64 s (K-major SW128)
    __nv_bfloat16 XW[2][P * 64];   // (w o x)^T [p][s]
    __nv_bfloat16 M[2][Q * 64];    // masked decayed CB [t][s]
    __nv_bfloat16 Hs[2][P * 64];   // bf16 state [p][n], 2 panels of 64 n
    float carry[2][kMaxW - 1][P];  // raw x rows before the chunk, by chunk parity
    float wconv[P][kMaxW];
    float bconv[P];
    float gam_hi[Q], gam_lo[Q], dts[Q];
    float wsum_hi[4], wsum_lo[4];
    uint64_t bar_ld, bar_z, bar_g1, bar_g34, bar_g2;
    uint32_t tmem_base;
};

constexpr size_t kSmemBytes = sizeof(TcSmem) + 1024;

__device__ __forceinline__ float bf2f(__nv_bfloat16 v) { return __bfloat162float(v); }

// silu via one MUFU op: v * sigmoid(v) = 0.5 v (1 + tanh(v / 2)).
__device__ __forceinline__ float silu_fast(float v)
{
    float t;
    asm("tanh.approx.f32 %0, %1;" : "=f"(t) : "f"(0.5f * v));
    return 0.5f * v * (1.0f + t);
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

__device__ __forceinline__ void unpack8(uint4 r, float* f)
{
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&r);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 t = __bfloat1622float2(h[i]);
        f[2 * i] = t.x;
        f[2 * i + 1] = t.y;
    }
}

__device__ __forceinline__ uint4 pack8(const float* f)
{
    uint4 r;
    __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&r);
#pragma unroll
    for (int i = 0; i < 4; ++i) h[i] = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
    return r;
}

// 16-byte chunk j (8 elements) of row r of a SW128 tile of 64-element rows.
__device__ __forceinline__ const uint4* tile_chunk(const __nv_bfloat16* tile, int r, int j)
{
    return reinterpret_cast<const uint4*>(reinterpret_cast<const uint8_t*>(tile) + r * 128 +
                                          (((j ^ r) & 7) << 4));
}

// element (row, k) of a K-major operand stored as panels of 64 k.
__device__ __forceinline__ __nv_bfloat16* kmajor_elem(__nv_bfloat16 (*panels)[P * 64], int row,
                                                      int k)
{
    return reinterpret_cast<__nv_bfloat16*>(reinterpret_cast<uint8_t*>(panels[k >> 6]) +
                                            sw128_offset(row, k & 63));
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
        for (int i = tid; i < P * kMaxW; i += kThreads) {
            const int pp = i / kMaxW, k = i % kMaxW;
            s.wconv[pp][k] = k < W ? p.conv_w[(size_t)(h * P + pp) * W + k] : 0.0f;
        }
        for (int i = tid; i < P; i += kThreads) s.bconv[i] = p.conv_b ? p.conv_b[h * P + i] : 0.0f;
        // carry rows -3..-1 before chunk 0 come from the conv state (its last rows)
        const __nv_bfloat16* cs = static_cast<const __nv_bfloat16*>(p.conv_state_in);
        for (int i = tid; i < (kMaxW - 1) * P; i += kThreads) {
            const int j = i / P, pp = i % P;
            const int sr = (W - 1) + (j - (kMaxW - 1));  // state row holding raw row j-3
            float v = 0.0f;
            if (cs && sr >= 0) v = bf2f(cs[((size_t)b * (W - 1) + sr) * Cdim + h * P + pp]);
            s.carry[0][j][pp] = v;
        }
    }

    // the fp32 state, thread n owns h[:, n]
    const int n = tid;
    const size_t sbase = ((size_t)b * H + h) * P * N;
    float hreg[P];
#pragma unroll
    for (int pp = 0; pp < P; ++pp) hreg[pp] = p.h0 ? p.h0[sbase + (size_t)pp * N + n] : 0.0f;
#pragma unroll
    for (int pp = 0; pp < P; ++pp) *kmajor_elem(s.Hs, pp, n) = __float2bfloat16_rn(hreg[pp]);

    const float Ah = p.A[h];
    const float bias = p.dt_bias ? p.dt_bias[h] : 0.0f;
    const float Dh = p.D ? p.D[h] : 0.0f;
    float dt_next = tid < p.S ? p.dt[((size_t)b * p.S + tid) * H + h] : 0.0f;

    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = s.tmem_base;
    const uint32_t lane_off = (uint32_t)(32 * warp) << 16;
    const uint32_t t_cb = tbase, t_yd = tbase + 128, t_yo = tbase + 192, t_st = tbase + 256;

    const int xB = p.bc_col0 + g * N;            // first B column in the bc source
    const int xC = p.bc_col0 + G * N + g * N;    // first C column
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

    const uint32_t aC = smem_u32(s.C), aB = smem_u32(s.B), aXT = smem_u32(s.XT);
    const uint32_t aXW = smem_u32(s.XW), aM = smem_u32(s.M), aH = smem_u32(s.Hs);
    constexpr float kLog2e = 1.4426950408889634f;

    bool ok = true;
    for (int c = 0; c < nchunks; ++c) {
        const uint32_t par = c & 1;
        const int r0 = c * Q;
        const int rows = min(Q, p.S - r0);

        // ---- dt and the cumulative sum of a = dt A (double-float) --------------
        float dt = 0.0f;
        if (tid < rows) dt = softplus ? softplus_f32(dt_next + bias) : dt_next;
        if (c + 1 < nchunks)
            dt_next = r0 + Q + tid < p.S ? p.dt[((size_t)b * p.S + r0 + Q + tid) * H + h] : 0.0f;
        float ghi = dt * Ah, glo = 0.0f;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const float ohi = __shfl_up_sync(0xffffffffu, ghi, d);
            const float olo = __shfl_up_sync(0xffffffffu, glo, d);
            if (lane >= d) df_add(ghi, glo, ohi, olo);
        }
        if (lane == 31) {
            s.wsum_hi[warp] = ghi;
            s.wsum_lo[warp] = glo;
        }
        s.dts[tid] = dt;
        __syncthreads();
        for (int w2 = 0; w2 < warp; ++w2) df_add(ghi, glo, s.wsum_hi[w2], s.wsum_lo[w2]);
        s.gam_hi[tid] = ghi;
        s.gam_lo[tid] = glo;

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
        const float gShi = s.gam_hi[rows - 1], gSlo = s.gam_lo[rows - 1];
        const float decay_t = __expf(fminf(ghi + glo, 0.0f));
        const float w_t = tid < rows ? __expf(fminf((gShi - ghi) + (gSlo - glo), 0.0f)) * dt : 0.0f;
        const float decay_S = __expf(fminf(gShi + gSlo, 0.0f));

        // ---- x: conv + SiLU of the raw rows (or the post-conv tile) -> x^T, (w x)^T
        {
            const int t = tid;
#pragma unroll 2
            for (int j = 0; j < 8; ++j) {
                float xv[8];
                if (p.conv) {
                    float acc[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) acc[e] = s.bconv[8 * j + e];
                    for (int k = 0; k < W; ++k) {
                        const int r = t - (W - 1) + k;
                        float raw[8];
                        if (r >= 0) {
                            unpack8(*tile_chunk(s.Xr, r, j), raw);
                        } else {
#pragma unroll
                            for (int e = 0; e < 8; ++e) raw[e] = s.carry[par][kMaxW - 1 + r][8 * j + e];
                        }
#pragma unroll
                        for (int e = 0; e < 8; ++e) acc[e] = fmaf(s.wconv[8 * j + e][k], raw[e], acc[e]);
                    }
#pragma unroll
                    for (int e = 0; e < 8; ++e) xv[e] = t < rows ? silu_fast(acc[e]) : 0.0f;
                } else {
                    unpack8(*tile_chunk(s.Xr, t, j), xv);
                }
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    *kmajor_elem(s.XT, 8 * j + e, t) = __float2bfloat16_rn(xv[e]);
                    *kmajor_elem(s.XW, 8 * j + e, t) = __float2bfloat16_rn(w_t * xv[e]);
                }
            }
            if (p.conv && t >= Q - (kMaxW - 1)) {
                // raw rows Q-3..Q-1 carry into the next chunk
                for (int j = 0; j < 8; ++j) {
                    float raw[8];
                    unpack8(*tile_chunk(s.Xr, t, j), raw);
#pragma unroll
                    for (int e = 0; e < 8; ++e) s.carry[par ^ 1][t - (Q - (kMaxW - 1))][8 * j + e] = raw[e];
                }
            }
        }
        fence_proxy_async_smem();
        __syncthreads();
        if (tid == 0 && ok) {
            tc_fence_after();
#pragma unroll
            for (int k = 0; k < 8; ++k) {  // G3: Yo = C h^T
                const uint32_t offc = (k >> 2) * (Q * 128) + (k & 3) * 32;
                const uint32_t offh = (k >> 2) * (P * 128) + (k & 3) * 32;
                mma_bf16_ss(t_yo, sdesc_sw128(aC + offc, 16, 1024),
                            sdesc_sw128(aH + offh, 16, 1024), kIdY, k > 0);
            }
#pragma unroll
            for (int k = 0; k < 8; ++k) {  // G4: dH = B^T (w x)
                const uint32_t offx = (k >> 2) * (P * 128) + (k & 3) * 32;
                mma_bf16_ss(t_st, sdesc_sw128(aB + k * 2048, Q * 128, 1024),
                            sdesc_sw128(aXW + offx, 16, 1024), kIdState, k > 0);
            }
            mma_commit(&s.bar_g34);
        }

        // ---- causal mask with decays: M[t,s] = CB[t,s] exp(gamma_t - gamma_s) dt_s
        ok = ok && mbar_wait_ns(&s.bar_g1, par, kWaitNs);
        tc_fence_after();
        {
            const int t = tid;
#pragma unroll 1
            for (int cc = 0; cc < 4; ++cc) {
                float v[32];
                tmem_ld32(t_cb + lane_off + cc * 32, v);
                tmem_ld_wait();
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4) {
                    float m[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        const int sidx = cc * 32 + q4 * 8 + e;
                        float val = 0.0f;
                        if (sidx <= t) {
                            const float ex = (ghi - s.gam_hi[sidx]) + (glo - s.gam_lo[sidx]);
                            val = v[q4 * 8 + e] * exp2f(fminf(ex, 0.0f) * kLog2e) * s.dts[sidx];
                        }
                        m[e] = val;
                    }
                    const int k = cc * 32 + q4 * 8;  // first s of this 16-byte chunk
                    *reinterpret_cast<uint4*>(reinterpret_cast<uint8_t*>(s.M[k >> 6]) +
                                              sw128_offset(t, k & 63)) = pack8(m);
                }
            }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();
        if (tid == 0 && ok) {
            tc_fence_after();
#pragma unroll
            for (int k = 0; k < 8; ++k) {  // G2: Yd = M x
                const uint32_t offm = (k >> 2) * (Q * 128) + (k & 3) * 32;
                const uint32_t offx = (k >> 2) * (P * 128) + (k & 3) * 32;
                mma_bf16_ss(t_yd, sdesc_sw128(aM + offm, 16, 1024),
                            sdesc_sw128(aXT + offx, 16, 1024), kIdY, k > 0);
            }
            mma_commit(&s.bar_g2);
        }

        // ---- state: h <- exp(gamma_Q) h + dH; tiles of the next chunk --------------
        ok = ok && mbar_wait_ns(&s.bar_g34, par, kWaitNs);
        tc_fence_after();
        if (tid == 0 && ok && c + 1 < nchunks) issue_main(c + 1);
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            float v[32];
            tmem_ld32(t_st + lane_off + half * 32, v);
            tmem_ld_wait();
#pragma unroll
            for (int e = 0; e < 32; ++e) {
                const int pp = half * 32 + e;
                hreg[pp] = fmaf(decay_S, hreg[pp], v[e]);
                *kmajor_elem(s.Hs, pp, n) = __float2bfloat16_rn(hreg[pp]);
            }
        }

        // ---- epilogue: y = Yd + exp(gamma_t) Yo + D x, gated ------------------------
        ok = ok && mbar_wait_ns(&s.bar_g2, par, kWaitNs);
        if (has_z) ok = ok && mbar_wait_ns(&s.bar_z, par, kWaitNs);
        tc_fence_after();
        {
            const int t = tid;
            __nv_bfloat16* yrow = static_cast<__nv_bfloat16*>(p.y) +
                                  (((size_t)b * p.S + r0 + t) * H + h) * P;
#pragma unroll 1
            for (int half = 0; half < 2; ++half) {
                float yd[32], yo[32];
                tmem_ld32(t_yd + lane_off + half * 32, yd);
                tmem_ld32(t_yo + lane_off + half * 32, yo);
                tmem_ld_wait();
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4) {
                    const int j = half * 4 + q4;
                    float out[8], zv[8];
                    if (has_z) unpack8(*tile_chunk(s.Z, t, j), zv);
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        const int pp = 8 * j + e;
                        const float xv = bf2f(*kmajor_elem(s.XT, pp, t));
                        float yv = fmaf(decay_t, yo[q4 * 8 + e], yd[q4 * 8 + e]);
                        yv = fmaf(Dh, xv, yv);
                        if (has_z) yv *= silu_fast(zv[e]);
                        out[e] = yv;
                    }
                    if (t < rows) reinterpret_cast<uint4*>(yrow)[j] = pack8(out);
                }
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
        for (int pp = 0; pp < P; ++pp) p.hS[sbase + (size_t)pp * N + n] = hreg[pp];
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
