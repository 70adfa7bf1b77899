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
// h [P=64, N=128] stays in registers for the whole sequence.  Per chunk,
// four dense contractions run on the tensor cores (bf16 operands in shared
// memory, fp32 accumulators in TMEM):
//   G1  CB[t,s] = C_t . B_s                 A = C  (TMA tile)   B = B (TMA)
//   G3  Yo[t,p] = C_t . h[p,:]              A = C               B = bf16(h) rows [n][p]
//   G4  dH[n,p] = sum_s B[s,n] xw[s,p]      A = B^T (MN-major)  B = xw rows [s][p]
//   G2  Yd[t,p] = sum_s M[t,s] xv[s,p]      A = M (causal mask of CB)  B = xv rows [s][p]
// Two forms of the decay, chosen per chunk:
//   factored (a <= 0 and the chunk's total decay is moderate): with
//     u_t = exp(gamma_t) and v_s = exp(-gamma_s) dt_s,
//     M = mask(CB), xv = xw = v o x, y = u_t (Yd + Yo) + D x,
//     h <- exp(gamma_Q) (h + dH);  the mask is a plain select and convert.
//   exact (otherwise): M = mask(CB o exp(min(gamma_t - gamma_s, 0)) dt_s),
//     xv = x, xw = w o x with w_s = exp(min(gamma_Q - gamma_s, 0)) dt_s,
//     y = Yd + u_t Yo + D x,  h <- exp(gamma_Q) h + dH.
//
// The CTA is warp-specialised and software-pipelined over chunks, four
// warpgroups of 128 threads:
//   conv   x conv + SiLU of the raw TMA tile (4 rows x 8 channels per task)
//          into the x rows tile XR;
//   front  dt and the double-float cumulative sum of a; the scaled x tile XS
//          (v o x or w o x); the causal mask M from CB (blocks above the
//          diagonal are zero-filled without a TMEM read);
//   back   the state update and the epilogue y = a Yd + u Yo + D x, times
//          silu(z);
//   issuer one thread issues every TMA load and every MMA as soon as its
//          operands are ready.
// The conv and front run ahead on chunk c+1 while the back finishes chunk c;
// the accumulators the back reads (Yd, Yo, dH) are double-buffered in TMEM,
// and mbarriers carry every hand-off.  setmaxnreg moves registers from the
// issuing warpgroup to the others.  Every wait is bounded in time; a wait
// that runs out aborts the CTA and sets the device error word.
#include "internal.cuh"
#include "sm100.cuh"

#include <cudaTypedefs.h>

#include <cstddef>
#include <mutex>

namespace ssd {
namespace {

using namespace sm100;

constexpr int Q = 128;  // rows per chunk
constexpr int P = 64;   // head dim
constexpr int N = 128;  // state dim
constexpr int kWG = 128;                 // threads per warpgroup
constexpr int kThreads = 4 * kWG;        // conv, front, back, issuer
// Registers: launched at kLaunchRegs per thread (512 x 128 = 65,536, the
// whole pool); setmaxnreg then gives each warpgroup its share, adding up to
// the pool: 136 + 112 + 192 + 72 = 4 x 128.
constexpr uint32_t kLaunchRegs = 128;
constexpr uint32_t kConvRegs = 136, kFrontRegs = 112, kBackRegs = 192, kIssuerRegs = 72;
static_assert(kConvRegs + kFrontRegs + kBackRegs + kIssuerRegs == 4 * kLaunchRegs,
              "register split");
constexpr int kMaxW = 4;  // conv taps handled in the kernel (W-1 carried rows)
constexpr uint64_t kWaitNs = 2000000000ull;  // bound on any single wait: 2 s
constexpr uint32_t kBarConv = 1, kBarFront = 2;  // named barriers of two warpgroups

// G1: A, B K-major.  G2, G3: A K-major, B MN-major (row tiles [k][p]).
// G4: A = B^T read MN-major from the B tile, B MN-major.
constexpr uint32_t kIdCB = idesc_bf16_f32(128, 128, false, false);
constexpr uint32_t kIdY = idesc_bf16_f32(128, 64, false, true);
constexpr uint32_t kIdState = idesc_bf16_f32(128, 64, true, true);

// TMEM columns: CB, then Yd / Yo / dH, each double-buffered by chunk parity
constexpr uint32_t kColCB = 0, kColYd = 128, kColYo = 256, kColDH = 384;

// Below this total chunk decay (log2 units) the mask factors as
// exp(gamma_t) * exp(-gamma_s): every factor stays within fp32 (2^90 < 2^127).
constexpr float kFactorMinLog2 = -90.0f;

struct __align__(16) ChunkVals {  // per-chunk row values, written by the front
    float g2h[Q], g2l[Q];      // gamma * log2(e), double-float (hi, lo)
    float dts[Q];              // dt_s
    float vfac[Q];             // exp(-gamma_s) dt_s (factored mask only)
    float wrow[Q];             // w_s = exp(min(gamma_Q - gamma_s, 0)) dt_s
    float dec[Q];              // exp(min(gamma_t, 0))
    float decS;                // exp(min(gamma_Q, 0))
    int factored;              // which form of the decay this chunk uses
};

struct __align__(1024) TcSmem {
    __nv_bfloat16 C[2][Q * 64];     // C tile [t][n]: 2 panels of 64 n (TMA, SW128)
    __nv_bfloat16 B[2][Q * 64];     // B tile [s][n]
    __nv_bfloat16 Xr[2][Q * 64];    // raw (or post-conv) x tiles [t][p] by chunk parity
    __nv_bfloat16 XR[2][Q * 64];    // post-conv x rows [s][p] (SW128), by parity
    __nv_bfloat16 XS[2][Q * 64];    // scaled x rows: v o x (factored) or w o x (exact)
    __nv_bfloat16 M[2][Q * 64];     // masked CB [t][s]: G2's A (K-major)
    __nv_bfloat16 Hs[N * 64];       // bf16 state rows [n][p]: G3's B
    ChunkVals cv[2];
    alignas(16) __nv_bfloat16 carry[2][kMaxW - 1][P];  // raw x rows before the chunk, by parity
    alignas(16) float2 wconv[P / 2][kMaxW];  // taps of channel pairs (front-padded with zeros)
    float2 bconv[P / 2];
    float wsum_hi[4], wsum_lo[4];
    uint64_t tma_bc, tma_x[2], g1, g2[2], g3[2], g4[2];
    uint64_t xconv[2], xready[2], cvready[2], mready, hsready, epidone[2];
    uint32_t tmem_base;
    int abort;
};

constexpr size_t kSmemBytes = sizeof(TcSmem) + 1024;

// operand tiles start on 1024-byte swizzle atoms; vector-accessed members on
// their vector size
static_assert(offsetof(TcSmem, C) % 1024 == 0 && offsetof(TcSmem, B) % 1024 == 0, "tile");
static_assert(offsetof(TcSmem, Xr) % 1024 == 0 && offsetof(TcSmem, XR) % 1024 == 0, "tile");
static_assert(offsetof(TcSmem, XS) % 1024 == 0 && offsetof(TcSmem, M) % 1024 == 0, "tile");
static_assert(offsetof(TcSmem, Hs) % 1024 == 0, "tile");
static_assert(sizeof(ChunkVals) % 16 == 0 && offsetof(TcSmem, cv) % 16 == 0, "float4 rows");
static_assert(offsetof(ChunkVals, vfac) % 16 == 0 && offsetof(ChunkVals, wrow) % 16 == 0, "float4");
static_assert(offsetof(ChunkVals, g2l) % 16 == 0 && offsetof(ChunkVals, dts) % 16 == 0, "float4");
static_assert(offsetof(TcSmem, carry) % 16 == 0 && (P * 2) % 16 == 0, "uint4 carry rows");
static_assert(offsetof(TcSmem, wconv) % 8 == 0 && offsetof(TcSmem, bconv) % 8 == 0, "float2");
static_assert(offsetof(TcSmem, tma_bc) % 8 == 0, "mbarriers");
static_assert(kSmemBytes <= 232448, "shared memory per CTA");

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

// Bounded wait that also gives up as soon as another role has aborted.  After
// a few immediate polls it backs off with nanosleep so that waiting warps do
// not take issue slots from the warps doing the work.
__device__ __forceinline__ bool wait_or_abort(TcSmem& s, uint64_t* bar, uint32_t parity)
{
#pragma unroll 1
    for (int i = 0; i < 4; ++i)
        if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    uint32_t ns = 32;
    while (true) {
        __nanosleep(ns);
        if (mbar_try_wait(bar, parity)) return true;
        ns = ns < 256 ? ns * 2 : 256;
        if (*reinterpret_cast<volatile int*>(&s.abort)) return false;
        if (globaltimer_ns() - t0 > kWaitNs) {
            *reinterpret_cast<volatile int*>(&s.abort) = 1;
            return false;
        }
    }
}

__global__ void __launch_bounds__(kThreads, 1)
    scan_tc_kernel(const __grid_constant__ CUtensorMap map_x,
                   const __grid_constant__ CUtensorMap map_bc, const TcScanParams p)
{
    // Align to the 1024-byte swizzle atom with pointer arithmetic on the
    // shared array itself, so the compiler keeps every access in the shared
    // address space (LDS/STS rather than generic loads and stores).
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    TcSmem& s = *reinterpret_cast<TcSmem*>(smem_raw + ((1024u - (sm100::smem_u32(smem_raw) & 1023u)) & 1023u));
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int wg = warp >> 2;             // 0 conv, 1 front, 2 back, 3 issuer
    const int quarter = warp & 3;         // TMEM lane quarter of this warp
    const int h = blockIdx.x, b = blockIdx.y;
    const int H = p.H, G = p.G, W = p.W;
    const int g = h / (H / G);
    const int Cdim = H * P + 2 * G * N;
    const int nchunks = (p.S + Q - 1) / Q;
    const bool has_z = (p.flags & kHasZ) != 0;
    const bool softplus = (p.flags & kDtSoftplus) != 0;

    if (tid == 0) {
        mbar_init(&s.tma_bc, 1);
        mbar_init(&s.g1, 1);
        for (int i = 0; i < 2; ++i) {
            mbar_init(&s.tma_x[i], 1);
            mbar_init(&s.g2[i], 1);
            mbar_init(&s.g3[i], 1);
            mbar_init(&s.g4[i], 1);
            mbar_init(&s.xconv[i], kWG);
            mbar_init(&s.xready[i], kWG);
            mbar_init(&s.cvready[i], kWG);
            mbar_init(&s.epidone[i], kWG);
        }
        mbar_init(&s.mready, kWG);
        mbar_init(&s.hsready, kWG);
        s.abort = 0;
        fence_mbar_init();
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
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = s.tmem_base;
    const uint32_t lane_off = (uint32_t)(32 * quarter) << 16;
    const size_t sbase = ((size_t)b * H + h) * P * N;

    if (wg == 3) {
        // ===================== issuer: TMA + MMA (one thread) =====================
        regs_set<kIssuerRegs, kLaunchRegs>();
        if (warp == 12 && lane == 0 && nchunks > 0) {
            prefetch_tmap(&map_x);
            prefetch_tmap(&map_bc);
            const int xB = p.bc_col0 + g * N;          // first B column in the bc source
            const int xC = p.bc_col0 + G * N + g * N;  // first C column
            const uint32_t aC = smem_u32(s.C), aB = smem_u32(s.B);
            const uint32_t aM = smem_u32(s.M), aH = smem_u32(s.Hs);
            auto load_bc = [&](int c) {
                mbar_arrive_expect_tx(&s.tma_bc, 4 * Q * 64 * 2);
                tma_load_3d(s.C[0], &map_bc, &s.tma_bc, xC, c * Q, b);
                tma_load_3d(s.C[1], &map_bc, &s.tma_bc, xC + 64, c * Q, b);
                tma_load_3d(s.B[0], &map_bc, &s.tma_bc, xB, c * Q, b);
                tma_load_3d(s.B[1], &map_bc, &s.tma_bc, xB + 64, c * Q, b);
            };
            auto load_x = [&](int c) {
                mbar_arrive_expect_tx(&s.tma_x[c & 1], Q * 64 * 2);
                tma_load_3d(s.Xr[c & 1], &map_x, &s.tma_x[c & 1], h * P, c * Q, b);
            };
            load_bc(0);
            load_x(0);
            if (nchunks > 1) load_x(1);
            bool ok = true;
            for (int c = 0; c < nchunks && ok; ++c) {
                const uint32_t par = c & 1, bpar = (c >> 1) & 1;
                const int buf = c & 1;
                // G1(c): B, C landed; the front has read CB(c-1)
                ok = wait_or_abort(s, &s.tma_bc, par);
                if (ok && c > 0) ok = wait_or_abort(s, &s.mready, par ^ 1);
                if (!ok) break;
                tc_fence_after();
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    const uint32_t off = (k >> 2) * (Q * 128) + (k & 3) * 32;
                    mma_bf16_ss(tbase + kColCB, sdesc_sw128(aC + off, 16, 1024),
                                sdesc_sw128(aB + off, 16, 1024), kIdCB, k > 0);
                }
                mma_commit(&s.g1);
                // G4(c): scaled x written; dH[buf] free (the back finished chunk c-2)
                ok = wait_or_abort(s, &s.xready[buf], bpar);
                if (ok && c >= 2) ok = wait_or_abort(s, &s.epidone[buf], bpar ^ 1);
                if (!ok) break;
                tc_fence_after();
                const uint32_t aXS = smem_u32(s.XS[buf]);
#pragma unroll
                for (int k = 0; k < 8; ++k)
                    mma_bf16_ss(tbase + kColDH + 64 * buf, sdesc_sw128(aB + k * 2048, Q * 128, 1024),
                                sdesc_sw128(aXS + k * 2048, 8192, 1024), kIdState, k > 0);
                mma_commit(&s.g4[buf]);
                // raw x of chunk c+2 into Xr[buf] once the conv has read it
                if (c + 2 < nchunks) {
                    ok = wait_or_abort(s, &s.xconv[buf], bpar);
                    if (!ok) break;
                    load_x(c + 2);
                }
                // G3(c): the back wrote bf16 h of chunk c-1
                ok = wait_or_abort(s, &s.hsready, par);
                if (!ok) break;
                tc_fence_after();
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    const uint32_t offc = (k >> 2) * (Q * 128) + (k & 3) * 32;
                    mma_bf16_ss(tbase + kColYo + 64 * buf, sdesc_sw128(aC + offc, 16, 1024),
                                sdesc_sw128(aH + k * 2048, 8192, 1024), kIdY, k > 0);
                }
                mma_commit(&s.g3[buf]);
                // B, C of chunk c+1 once G1, G4, G3 of chunk c are done
                if (c + 1 < nchunks) {
                    ok = wait_or_abort(s, &s.g3[buf], bpar);
                    if (!ok) break;
                    load_bc(c + 1);
                }
                // G2(c): the front wrote M(c); x is XS (factored) or XR (exact)
                ok = wait_or_abort(s, &s.mready, par);
                if (!ok) break;
                tc_fence_after();
                const uint32_t aXV = smem_u32(s.cv[buf].factored ? s.XS[buf] : s.XR[buf]);
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    const uint32_t offm = (k >> 2) * (Q * 128) + (k & 3) * 32;
                    mma_bf16_ss(tbase + kColYd + 64 * buf, sdesc_sw128(aM + offm, 16, 1024),
                                sdesc_sw128(aXV + k * 2048, 8192, 1024), kIdY, k > 0);
                }
                mma_commit(&s.g2[buf]);
            }
            if (!ok) *reinterpret_cast<volatile int*>(&s.abort) = 1;
        }
    } else if (wg == 0) {
        // ===================== conv: x rows of each chunk =====================
        regs_set<kConvRegs, kLaunchRegs>();
        const int cj = tid & 7;  // channel group (8 channels)
        float2 wq[4][kMaxW], bq[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            bq[e] = p.conv ? s.bconv[4 * cj + e] : make_float2(0.f, 0.f);
#pragma unroll
            for (int k = 0; k < kMaxW; ++k)
                wq[e][k] = p.conv ? s.wconv[4 * cj + e][k] : make_float2(0.f, 0.f);
        }
        bool ok = true;
        for (int c = 0; c < nchunks; ++c) {
            const uint32_t bpar = (c >> 1) & 1;
            const int buf = c & 1;
            const int rows = min(Q, p.S - c * Q);
            // XR[buf] is free once the back finished chunk c-2
            if (c >= 2) ok = ok && wait_or_abort(s, &s.epidone[buf], bpar ^ 1);
            if (ok) ok = wait_or_abort(s, &s.tma_x[buf], bpar);
            // together: the carry rows of chunk c-1 are written; a common decision
            ok = !named_bar_or(kBarConv, kWG, !ok);
            if (!ok) break;
#pragma unroll 1
            for (int task = 0; task < 2; ++task) {
                const int t0 = 4 * ((tid >> 3) + 16 * task);
                float2 xo[4][4];  // [row][channel pair]
                if (p.conv) {
                    float2 win[7][4];  // raw rows t0-3 .. t0+3
#pragma unroll
                    for (int k = 0; k < 7; ++k) {
                        const int r = t0 - 3 + k;
                        const uint4 raw = r >= 0 ? at<const uint4>(s.Xr[buf], chunk_off(r, cj))
                                                 : *reinterpret_cast<const uint4*>(&s.carry[buf][r + 3][8 * cj]);
                        unpack4x2(raw, win[k]);
                        if (r >= Q - (kMaxW - 1))  // rows Q-3..Q-1 carry into the next chunk
                            *reinterpret_cast<uint4*>(&s.carry[buf ^ 1][r - (Q - 3)][8 * cj]) = raw;
                    }
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            float2 v = bq[e];
#pragma unroll
                            for (int k = 0; k < kMaxW; ++k) v = __ffma2_rn(wq[e][k], win[i + k][e], v);
                            xo[i][e] = t0 + i < rows ? silu2(v) : make_float2(0.f, 0.f);
                        }
                    }
                } else {
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        unpack4x2(at<const uint4>(s.Xr[buf], chunk_off(t0 + i, cj)), xo[i]);
                }
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    at<uint4>(s.XR[buf], chunk_off(t0 + i, cj)) = pack4x2(xo[i]);
            }
            fence_proxy_async_smem();  // XR is read by G2 in the exact form
            mbar_arrive(&s.xconv[buf]);
        }
        if (!ok) *reinterpret_cast<volatile int*>(&s.abort) = 1;
    } else if (wg == 1) {
        // ===================== front: gamma, scaled x, mask =====================
        regs_set<kFrontRegs, kLaunchRegs>();
        const int t = tid - kWG;  // chunk row of this thread
        const float Ah = p.A[h];
        const float bias = p.dt_bias ? p.dt_bias[h] : 0.0f;
        constexpr float kLog2e = 1.4426950408889634f;
        float dt_next = t < p.S ? p.dt[((size_t)b * p.S + t) * H + h] : 0.0f;
        bool ok = true;
        for (int c = 0; c < nchunks; ++c) {
            const uint32_t par = c & 1, bpar = (c >> 1) & 1;
            const int buf = c & 1;
            const int r0 = c * Q;
            const int rows = min(Q, p.S - r0);
            ChunkVals& cv = s.cv[buf];
            // ---- dt and the cumulative sum of a = dt A (double-float) ----
            float dt = 0.0f;
            if (t < rows) dt = softplus ? softplus_f32(dt_next + bias) : dt_next;
            if (c + 1 < nchunks)
                dt_next = r0 + Q + t < p.S ? p.dt[((size_t)b * p.S + r0 + Q + t) * H + h] : 0.0f;
            float ghi = dt * Ah, glo = 0.0f;
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
            // cv[buf] and XS[buf] are free once the back finished chunk c-2
            if (c >= 2) ok = ok && wait_or_abort(s, &s.epidone[buf], bpar ^ 1);
            ok = !named_bar_or(kBarFront, kWG, !ok);  // a common decision
            if (!ok) break;
            for (int w2 = 0; w2 < quarter; ++w2) df_add(ghi, glo, s.wsum_hi[w2], s.wsum_lo[w2]);
            const float g2h_t = ghi * kLog2e, g2l_t = glo * kLog2e;
            cv.g2h[t] = g2h_t;
            cv.g2l[t] = g2l_t;
            cv.dts[t] = dt;
            named_bar_sync(kBarFront, kWG);
            const float gLh = cv.g2h[rows - 1], gLl = cv.g2l[rows - 1];
            const bool factored = Ah <= 0.0f && gLh + gLl >= kFactorMinLog2;
            cv.dec[t] = ex2_fast(fminf(g2h_t + g2l_t, 0.0f));
            // the row's x scale: v_t = exp(-gamma_t) dt_t or w_t = exp(min(gamma_Q-gamma_t,0)) dt_t
            const float sc = factored ? ex2_fast(-(g2h_t + g2l_t)) * dt
                                      : (t < rows ? ex2_fast(fminf((gLh - g2h_t) + (gLl - g2l_t), 0.0f)) * dt : 0.0f);
            if (t == 0) {
                cv.decS = ex2_fast(fminf(gLh + gLl, 0.0f));
                cv.factored = factored;
            }
            mbar_arrive(&s.cvready[buf]);  // cv[buf] of chunk c is complete
            // ---- XS row t = sc * XR row t ----
            ok = wait_or_abort(s, &s.xconv[buf], bpar);
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                float2 xv[4];
                unpack4x2(at<const uint4>(s.XR[buf], chunk_off(t, j)), xv);
#pragma unroll
                for (int e = 0; e < 4; ++e) xv[e] = __fmul2_rn(make_float2(sc, sc), xv[e]);
                at<uint4>(s.XS[buf], chunk_off(t, j)) = pack4x2(xv);
            }
            fence_proxy_async_smem();
            mbar_arrive(&s.xready[buf]);

            // ---- causal mask (with the decays in the exact form) ----
            // M is free once G2(c-1) is done; CB(c) is ready once G1(c) is done
            if (ok && c >= 1) ok = wait_or_abort(s, &s.g2[buf ^ 1], ((c - 1) >> 1) & 1);
            if (ok) ok = wait_or_abort(s, &s.g1, par);
            ok = __all_sync(0xffffffffu, ok);  // warp-uniform: tcgen05.ld is .sync.aligned
            tc_fence_after();
#pragma unroll 1
            for (int cc = 0; cc < 4 && ok; ++cc) {  // 32-column blocks of s
                __nv_bfloat16* mpanel = s.M[cc >> 1];
                if (cc > quarter) {  // strictly above the diagonal for the whole warp
#pragma unroll
                    for (int q4 = 0; q4 < 4; ++q4)
                        at<uint4>(mpanel, chunk_off(t, (cc & 1) * 4 + q4)) = make_uint4(0, 0, 0, 0);
                    continue;
                }
#pragma unroll 1
                for (int hh = 0; hh < 2; ++hh) {  // 16 columns at a time
                    const int c0 = cc * 32 + 16 * hh;
                    float v[16];
                    tmem_ld16(tbase + kColCB + lane_off + c0, v);
                    tmem_ld_wait();
                    if (!factored) {
#pragma unroll
                        for (int q4 = 0; q4 < 4; ++q4) {
                            const int sb = c0 + 4 * q4;
                            const float4 gh = *reinterpret_cast<const float4*>(&cv.g2h[sb]);
                            const float4 gl = *reinterpret_cast<const float4*>(&cv.g2l[sb]);
                            const float4 ds = *reinterpret_cast<const float4*>(&cv.dts[sb]);
                            const float ghs[4] = {gh.x, gh.y, gh.z, gh.w}, gls[4] = {gl.x, gl.y, gl.z, gl.w};
                            const float dss[4] = {ds.x, ds.y, ds.z, ds.w};
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                const float ex = (g2h_t - ghs[e]) + (g2l_t - gls[e]);
                                v[4 * q4 + e] = v[4 * q4 + e] * dss[e] * ex2_fast(fminf(ex, 0.0f));
                            }
                        }
                    }
                    if (cc == quarter) {  // the diagonal block: keep s <= t
#pragma unroll
                        for (int e = 0; e < 16; ++e) v[e] = (c0 + e <= t) ? v[e] : 0.0f;
                    }
#pragma unroll
                    for (int q2 = 0; q2 < 2; ++q2) {
                        const float2 m[4] = {make_float2(v[8 * q2 + 0], v[8 * q2 + 1]),
                                             make_float2(v[8 * q2 + 2], v[8 * q2 + 3]),
                                             make_float2(v[8 * q2 + 4], v[8 * q2 + 5]),
                                             make_float2(v[8 * q2 + 6], v[8 * q2 + 7])};
                        at<uint4>(mpanel, chunk_off(t, (cc & 1) * 4 + 2 * hh + q2)) = pack4x2(m);
                    }
                }
            }
            fence_proxy_async_smem();
            tc_fence_before();
            mbar_arrive(&s.mready);
        }
        if (!ok) *reinterpret_cast<volatile int*>(&s.abort) = 1;
    } else {
        // ===================== back: state update, epilogue =====================
        regs_set<kBackRegs, kLaunchRegs>();
        const int t = tid - 2 * kWG;  // chunk row / state column of this thread
        const int n = t;
        float2 hreg[32];  // h[2i .. 2i+1][n]
#pragma unroll
        for (int i = 0; i < 32; ++i)
            hreg[i] = p.h0 ? make_float2(p.h0[sbase + (size_t)(2 * i) * N + n],
                                         p.h0[sbase + (size_t)(2 * i + 1) * N + n])
                           : make_float2(0.f, 0.f);
        auto store_h = [&]() {
#pragma unroll
            for (int q8 = 0; q8 < 8; ++q8) at<uint4>(s.Hs, chunk_off(n, q8)) = pack4x2(&hreg[4 * q8]);
        };
        store_h();
        fence_proxy_async_smem();
        mbar_arrive(&s.hsready);
        const __nv_bfloat16* zbase = static_cast<const __nv_bfloat16*>(p.z);
        const float Dh = p.D ? p.D[h] : 0.0f;
        bool ok = true;
        for (int c = 0; c < nchunks && ok; ++c) {
            const uint32_t bpar = (c >> 1) & 1;
            const int buf = c & 1;
            const int r0 = c * Q;
            const int rows = min(Q, p.S - r0);
            const ChunkVals& cv = s.cv[buf];
            // z of this row, early (used at the end)
            const uint4* zr = reinterpret_cast<const uint4*>(
                zbase + ((size_t)b * p.S + r0 + min(t, rows - 1)) * (H * P) + h * P);
            uint4 zq[8];
            if (has_z) {
#pragma unroll
                for (int q8 = 0; q8 < 8; ++q8) zq[q8] = __ldg(zr + q8);
            }
            // ---- state ----
            ok = wait_or_abort(s, &s.cvready[buf], bpar);     // cv of chunk c written
            if (ok) ok = wait_or_abort(s, &s.g4[buf], bpar);
            if (ok) ok = wait_or_abort(s, &s.g3[buf], bpar);  // G3(c) has read Hs
            ok = __all_sync(0xffffffffu, ok);  // warp-uniform: tcgen05.ld is .sync.aligned
            if (!ok) break;
            tc_fence_after();
            // h <- decS h + b dH, b = decS (factored: dH carries exp(-gamma_s)) or 1
            const bool factored = cv.factored != 0;
            const float2 dS = make_float2(cv.decS, cv.decS);
            const float2 bS = factored ? dS : make_float2(1.0f, 1.0f);
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                float v[32];
                tmem_ld32(tbase + kColDH + 64 * buf + lane_off + 32 * half, v);
                tmem_ld_wait();
#pragma unroll
                for (int i = 0; i < 16; ++i)
                    hreg[16 * half + i] = __ffma2_rn(dS, hreg[16 * half + i],
                                                     __fmul2_rn(bS, make_float2(v[2 * i], v[2 * i + 1])));
            }
            store_h();
            fence_proxy_async_smem();
            tc_fence_before();
            mbar_arrive(&s.hsready);
            // ---- epilogue ----
            ok = wait_or_abort(s, &s.g2[buf], bpar);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            tc_fence_after();
            // y = a Yd + u Yo + D x, a = u (factored) or 1
            const float dec = cv.dec[t];
            const float2 dd = make_float2(dec, dec);
            const float2 aa = factored ? dd : make_float2(1.0f, 1.0f);
            const float2 D2 = make_float2(Dh, Dh);
            uint4* yrow = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.y) +
                                                   (((size_t)b * p.S + r0 + t) * H + h) * P);
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) {  // 16 columns (2 chunks of 8 p) at a time
                float yd[16], yo[16];
                tmem_ld16(tbase + kColYd + 64 * buf + lane_off + 16 * q4, yd);
                tmem_ld16(tbase + kColYo + 64 * buf + lane_off + 16 * q4, yo);
                tmem_ld_wait();
#pragma unroll
                for (int j2 = 0; j2 < 2; ++j2) {
                    float2 out[4], zv[4], xv[4];
                    if (has_z) unpack4x2(zq[2 * q4 + j2], zv);
                    unpack4x2(at<const uint4>(s.XR[buf], chunk_off(t, 2 * q4 + j2)), xv);
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int k = j2 * 8 + 2 * e;
                        float2 yv = __ffma2_rn(dd, make_float2(yo[k], yo[k + 1]),
                                               __fmul2_rn(aa, make_float2(yd[k], yd[k + 1])));
                        yv = __ffma2_rn(D2, xv[e], yv);
                        if (has_z) yv = __fmul2_rn(yv, silu2(zv[e]));
                        out[e] = yv;
                    }
                    if (t < rows) yrow[2 * q4 + j2] = pack4x2(out);
                }
            }
            tc_fence_before();
            mbar_arrive(&s.epidone[buf]);
        }
        if (ok && !*reinterpret_cast<volatile int*>(&s.abort)) {
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                p.hS[sbase + (size_t)(2 * i) * N + n] = hreg[i].x;
                p.hS[sbase + (size_t)(2 * i + 1) * N + n] = hreg[i].y;
            }
        } else {
            *reinterpret_cast<volatile int*>(&s.abort) = 1;
        }
    }

    tc_fence_before();
    __syncthreads();
    if (tid == 0 && s.abort) atomicOr(p.err, kErrTimeout);
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tbase, 512);
    }
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
    CUtensorMap mx, mbc;
    if (!make_map(&mx, p.xbc, Cdim, p.S, p.B)) return cudaErrorInvalidValue;
    if (!make_map(&mbc, p.bc, p.bc_stride, p.S, p.B)) return cudaErrorInvalidValue;
    // The warpgroups' register split assumes the kernel was compiled to
    // exactly kLaunchRegs per thread; anything else is refused (a split that
    // does not add up would leave setmaxnreg waiting).
    cudaFuncAttributes fa;
    cudaError_t e = cudaFuncGetAttributes(&fa, scan_tc_kernel);
    if (e != cudaSuccess) return e;
    if (fa.numRegs != (int)kLaunchRegs) return cudaErrorNotSupported;
    e = cudaFuncSetAttribute(scan_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)kSmemBytes);
    if (e != cudaSuccess) return e;
    dim3 grid(p.H, p.B);
    scan_tc_kernel<<<grid, kThreads, kSmemBytes, st>>>(mx, mbc, p);
    return cudaGetLastError();
}

}  // namespace ssd
