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
// four dense contractions run on the tensor cores (bf16 operands, fp32
// accumulators in TMEM):
//   G1  CB[t,s] = C_t . B_s               A = C (smem, TMA)   B = B (smem, TMA)
//   G4  dH[n,p] = sum_s B[s,n] xs[s,p]    A = B^T (smem)      B = xs rows [s][p]
//   G3  Y[t,p]  = C_t . h[p,:]            A = C (smem)        B = bf16(h) rows [n][p]
//   G2  Y[t,p] += sum_s M[t,s] xv[s,p]    A = M (TMEM)        B = xv rows [s][p]
// Two forms of the decay, chosen per chunk:
//   factored (a <= 0 and the chunk's total decay is moderate): with
//     u_t = exp(gamma_t) and v_s = exp(-gamma_s) dt_s,
//     M = mask(CB), xv = xs = v o x, y = u_t Y + D x, h <- exp(gamma_Q) (h + dH):
//     G3 and G2 share one accumulator and the mask is a select and convert;
//   exact (otherwise): M = mask(CB o exp(min(gamma_t - gamma_s, 0)) dt_s),
//     xv = x, xs = w o x with w_s = exp(min(gamma_Q - gamma_s, 0)) dt_s,
//     G3 goes to its own accumulator Yo, y = Y + u_t Yo + D x,
//     h <- exp(gamma_Q) h + dH.
//
// The masked CB is written back into TMEM (bf16 pairs) and read from there
// by G2, so it never passes through shared memory: the tensor cores' operand
// reads and the threads' shared-memory traffic draw on one bandwidth, and for
// these small-N products it is the tighter limit.
//
// Warp roles (512 threads):
//   conv   (warps 0-3)  raw x rows straight from global memory (the next
//                       chunk's rows are in flight while the thread waits),
//                       conv + SiLU, written once as x rows (XR) and once
//                       scaled (XS);
//   mask   (warps 4-7)  CB -> M in TMEM, one row per thread;
//   back   (warps 8-11) the state update (one chunk ahead) and the epilogue
//                       y = ..., times silu(z);
//   issuer (warp 12)    one thread issues every TMA load and every MMA as soon
//                       as its inputs are ready and its output buffer is free;
//   gamma  (warp 13)    dt, the double-float cumulative sum of a and the
//                       per-row scales of each chunk, ahead of the others.
// Every hand-off is an mbarrier; buffers are double-buffered by chunk parity
// (x rows, scaled x rows, C tile, Y and dH accumulators, bf16 state rows,
// per-chunk values).  setmaxnreg gives each warpgroup its share of the
// register file.  Every wait is bounded in time; a wait that runs out aborts
// the CTA and sets the device error word.
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
constexpr int kThreads = 4 * kWG;        // conv, mask, back, issuer + gamma
// Registers: launched at kLaunchRegs per thread (512 x 128 = 65,536, the
// whole pool); setmaxnreg then gives each warpgroup its share, adding up to
// the pool: 136 + 112 + 192 + 72 = 4 x 128.
constexpr uint32_t kLaunchRegs = 128;
constexpr uint32_t kConvRegs = 136, kMaskRegs = 112, kBackRegs = 192, kIssuerRegs = 72;
static_assert(kConvRegs + kMaskRegs + kBackRegs + kIssuerRegs == 4 * kLaunchRegs,
              "register split");
constexpr int kMaxW = 4;  // conv taps handled in the kernel (W-1 carried rows)
constexpr int kRawRows = 16 + kMaxW - 1;     // raw rows a conv thread reads per chunk
constexpr uint64_t kWaitNs = 2000000000ull;  // bound on any single wait: 2 s

// G1: A, B K-major.  G2, G3: A K-major, B MN-major (row tiles [k][p]).
// G4: A = B^T read MN-major from the B tile, B MN-major.
constexpr uint32_t kIdCB = idesc_bf16_f32(128, 128, false, false);
constexpr uint32_t kIdY = idesc_bf16_f32(128, 64, false, true);
constexpr uint32_t kIdState = idesc_bf16_f32(128, 64, true, true);

// TMEM columns (512 allocated)
constexpr uint32_t kColCB = 0;    // CB fp32 [t][s]                    128
constexpr uint32_t kColM = 128;   // M bf16 pairs [t][s/2]              64
constexpr uint32_t kColY = 192;   // Y fp32 [t][p], by chunk parity  2 x 64
constexpr uint32_t kColDH = 320;  // dH fp32 [n][p], by chunk parity 2 x 64
constexpr uint32_t kColYo = 448;  // Yo fp32 [t][p] (exact chunks)      64

// Below this total chunk decay (log2 units) the mask factors as
// exp(gamma_t) * exp(-gamma_s): every factor stays within fp32 (2^90 < 2^127).
constexpr float kFactorMinLog2 = -90.0f;

struct __align__(16) ChunkVals {  // per-chunk row values, written by the gamma warp
    float g2h[Q], g2l[Q];      // gamma * log2(e), double-float (hi, lo)
    float dts[Q];              // dt_s (0 past the last row)
    float sc[Q];               // x scale of G4's operand: v_s (factored) or w_s (exact)
    float dec[Q];              // exp(min(gamma_t, 0))
    float decS;                // exp(min(gamma_Q, 0))
    int factored;              // which form of the decay this chunk uses
    int pad[2];
};

struct __align__(1024) TcSmem {
    __nv_bfloat16 C[2][2][Q * 64];  // C tiles [t][n] by chunk parity: 2 panels of 64 n (TMA, SW128)
    __nv_bfloat16 B[2][Q * 64];     // B tile [s][n]: 2 panels
    __nv_bfloat16 XR[2][Q * 64];    // post-conv x rows [s][p] (SW128), by parity
    __nv_bfloat16 XS[2][Q * 64];    // scaled x rows: v o x (factored) or w o x (exact)
    __nv_bfloat16 Hs[2][N * 64];    // bf16 state rows [n][p]: G3's B, by parity
    ChunkVals cv[2];
    alignas(16) float2 wconv[P / 2][kMaxW];  // taps of channel pairs (front-padded with zeros)
    float2 bconv[P / 2];
    uint64_t full_c[2], full_b;                       // TMA landed
    uint64_t g1, g4[2], g3[2], mfree, ydone[2], fin;  // MMA commits
    uint64_t cvready[2], xready[2], mready, hsready[2], epidone[2];
    uint32_t tmem_base;
    int abort;
};

constexpr size_t kSmemBytes = sizeof(TcSmem) + 1024;

// operand tiles start on 1024-byte swizzle atoms; vector-accessed members on
// their vector size
static_assert(offsetof(TcSmem, C) % 1024 == 0 && offsetof(TcSmem, B) % 1024 == 0, "tile");
static_assert(offsetof(TcSmem, XR) % 1024 == 0 && offsetof(TcSmem, XS) % 1024 == 0, "tile");
static_assert(offsetof(TcSmem, Hs) % 1024 == 0, "tile");
static_assert(sizeof(ChunkVals) % 16 == 0 && offsetof(TcSmem, cv) % 16 == 0, "float4 rows");
static_assert(offsetof(ChunkVals, g2l) % 16 == 0 && offsetof(ChunkVals, dts) % 16 == 0, "float4");
static_assert(offsetof(ChunkVals, sc) % 16 == 0 && offsetof(ChunkVals, dec) % 16 == 0, "float4");
static_assert(offsetof(TcSmem, wconv) % 16 == 0 && offsetof(TcSmem, bconv) % 8 == 0, "float2");
static_assert(offsetof(TcSmem, full_c) % 8 == 0, "mbarriers");
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

__device__ __forceinline__ float2 unpack2(uint32_t r)
{
    return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&r));
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

__device__ __forceinline__ uint2 ldg_u2(const __nv_bfloat16* p)
{
    return __ldg(reinterpret_cast<const uint2*>(p));
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

__device__ __forceinline__ bool aborted(TcSmem& s)
{
    return *reinterpret_cast<volatile int*>(&s.abort) != 0;
}

__device__ __forceinline__ void set_abort(TcSmem& s)
{
    *reinterpret_cast<volatile int*>(&s.abort) = 1;
}

// Bounded wait that also gives up as soon as another role has aborted.  The
// hinted try_wait suspends the thread until the phase completes (or about a
// microsecond passes), so a waiting warp takes no issue slots.
__device__ __forceinline__ bool wait_or_abort(TcSmem& s, uint64_t* bar, uint32_t parity)
{
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    while (true) {
        if (mbar_try_wait_hint(bar, parity, 1000)) return true;
        if (aborted(s)) return false;
        if (globaltimer_ns() - t0 > kWaitNs) {
            set_abort(s);
            return false;
        }
    }
}

__global__ void __launch_bounds__(kThreads, 1)
    scan_tc_kernel(const __grid_constant__ CUtensorMap map_bc, const TcScanParams p)
{
    // Align to the 1024-byte swizzle atom with pointer arithmetic on the
    // shared array itself, so the compiler keeps every access in the shared
    // address space (LDS/STS rather than generic loads and stores).
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    TcSmem& s = *reinterpret_cast<TcSmem*>(smem_raw + ((1024u - (sm100::smem_u32(smem_raw) & 1023u)) & 1023u));
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int wg = warp >> 2;             // 0 conv, 1 mask, 2 back, 3 issuer + gamma
    const int quarter = warp & 3;         // TMEM lane quarter of this warp
    const int h = blockIdx.x, b = blockIdx.y;
    const int H = p.H, G = p.G, W = p.W, S = p.S;
    const int g = h / (H / G);
    const int Cdim = H * P + 2 * G * N;
    const int nchunks = (S + Q - 1) / Q;
    const bool has_z = (p.flags & kHasZ) != 0;

    if (tid == 0) {
        mbar_init(&s.full_b, 1);
        mbar_init(&s.g1, 1);
        mbar_init(&s.mfree, 1);
        mbar_init(&s.fin, 1);
        mbar_init(&s.mready, kWG);
        for (int i = 0; i < 2; ++i) {
            mbar_init(&s.full_c[i], 1);
            mbar_init(&s.g4[i], 1);
            mbar_init(&s.g3[i], 1);
            mbar_init(&s.ydone[i], 1);
            mbar_init(&s.cvready[i], 32);
            mbar_init(&s.xready[i], kWG);
            mbar_init(&s.hsready[i], kWG);
            mbar_init(&s.epidone[i], kWG);
        }
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
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = s.tmem_base;
    const uint32_t lane_off = (uint32_t)(32 * quarter) << 16;
    const size_t sbase = ((size_t)b * H + h) * P * N;

    if (wg == 3) {
        regs_set<kIssuerRegs, kLaunchRegs>();
        if (warp == 12 && lane == 0 && nchunks > 0) {
            // ===================== issuer: TMA + MMA (one thread) =====================
            // Each op is issued once its inputs are ready and its output buffer is
            // free, in chunk order per op, with G1(c) before G3(c) before G2(c).
            // Every phase test below is exact: the previous phase of the barrier
            // it tests is known to be complete by then.
            prefetch_tmap(&map_bc);
            const int xB = p.bc_col0 + g * N;          // first B column in the bc source
            const int xC = p.bc_col0 + G * N + g * N;  // first C column
            const uint32_t aB = smem_u32(s.B);
            auto load_c = [&](int c) {
                uint64_t* bar = &s.full_c[c & 1];
                mbar_arrive_expect_tx(bar, 2 * Q * 64 * 2);
                tma_load_3d(s.C[c & 1][0], &map_bc, bar, xC, c * Q, b);
                tma_load_3d(s.C[c & 1][1], &map_bc, bar, xC + 64, c * Q, b);
            };
            auto load_b = [&](int c) {
                mbar_arrive_expect_tx(&s.full_b, 2 * Q * 64 * 2);
                tma_load_3d(s.B[0], &map_bc, &s.full_b, xB, c * Q, b);
                tma_load_3d(s.B[1], &map_bc, &s.full_b, xB + 64, c * Q, b);
            };
            int nC = 0, nB = 0;  // tiles whose load has been issued
            load_c(nC++);
            if (nchunks > 1) load_c(nC++);
            load_b(nB++);
            int i1 = 0, i4 = 0, i3 = 0, i2 = 0;  // next chunk of G1, G4, G3, G2
            uint64_t t_idle = 0;
            bool ok = true;
            while (i2 < nchunks || i4 < nchunks) {
                bool progress = false;
                // C tile k into buffer k & 1 once G3(k-2) (and so G1(k-2)) is done
                if (nC < nchunks && nC - 2 < i3 && mbar_test(&s.g3[nC & 1], ((nC - 2) >> 1) & 1)) {
                    load_c(nC++);
                    progress = true;
                }
                // B tile k once G4(k-1) (and so G1(k-1)) is done
                if (nB < nchunks && nB - 1 < i4 && mbar_test(&s.g4[(nB - 1) & 1], ((nB - 1) >> 1) & 1)) {
                    load_b(nB++);
                    progress = true;
                }
                // G1(c): C(c), B(c) landed; the mask warps have read CB(c-1)
                if (i1 < nC && i1 < nB && mbar_test(&s.full_c[i1 & 1], (i1 >> 1) & 1) &&
                    mbar_test(&s.full_b, i1 & 1) && (i1 == 0 || mbar_test(&s.mready, (i1 - 1) & 1))) {
                    tc_fence_after();
                    const uint32_t aC = smem_u32(s.C[i1 & 1]);
#pragma unroll
                    for (int k = 0; k < 8; ++k) {
                        const uint32_t off = (k >> 2) * (Q * 128) + (k & 3) * 32;
                        mma_bf16_ss(tbase + kColCB, sdesc_sw128(aC + off, 16, 1024),
                                    sdesc_sw128(aB + off, 16, 1024), kIdCB, k > 0);
                    }
                    mma_commit(&s.g1);
                    ++i1;
                    progress = true;
                }
                // G4(c): B(c) in place (G1(c) issued), xs(c) written, dH[c&1] read by state(c-2)
                if (i4 < i1 && mbar_test(&s.xready[i4 & 1], (i4 >> 1) & 1) &&
                    (i4 < 2 || mbar_test(&s.hsready[(i4 - 1) & 1], ((i4 - 1) >> 1) & 1))) {
                    tc_fence_after();
                    const uint32_t aXS = smem_u32(s.XS[i4 & 1]);
#pragma unroll
                    for (int k = 0; k < 8; ++k)
                        mma_bf16_ss(tbase + kColDH + 64 * (i4 & 1), sdesc_sw128(aB + k * 2048, Q * 128, 1024),
                                    sdesc_sw128(aXS + k * 2048, 8192, 1024), kIdState, k > 0);
                    mma_commit(&s.g4[i4 & 1]);
                    ++i4;
                    progress = true;
                }
                // G3(c): after G1(c) (so that "G3(c) done" also means "G1(c) done",
                // which frees the C buffer); bf16 h of chunk c-1 written; Y[c&1] free
                // (epilogue c-2); exact chunks also need Yo free (epilogue c-1)
                if (i3 < i1 && mbar_test(&s.cvready[i3 & 1], (i3 >> 1) & 1) &&
                    mbar_test(&s.hsready[i3 & 1], (i3 >> 1) & 1) &&
                    (i3 < 2 || mbar_test(&s.epidone[i3 & 1], ((i3 >> 1) & 1) ^ 1))) {
                    const bool fac = s.cv[i3 & 1].factored != 0;
                    if (fac || i3 == 0 || mbar_test(&s.epidone[(i3 - 1) & 1], ((i3 - 1) >> 1) & 1)) {
                        tc_fence_after();
                        const uint32_t aC = smem_u32(s.C[i3 & 1]);
                        const uint32_t aH = smem_u32(s.Hs[i3 & 1]);
                        const uint32_t dY = fac ? kColY + 64 * (i3 & 1) : kColYo;
#pragma unroll
                        for (int k = 0; k < 8; ++k) {
                            const uint32_t offc = (k >> 2) * (Q * 128) + (k & 3) * 32;
                            mma_bf16_ss(tbase + dY, sdesc_sw128(aC + offc, 16, 1024),
                                        sdesc_sw128(aH + k * 2048, 8192, 1024), kIdY, k > 0);
                        }
                        mma_commit(&s.g3[i3 & 1]);
                        ++i3;
                        progress = true;
                    }
                }
                // G2(c): M(c) in TMEM; x rows written; after G3(c) (same accumulator)
                if (i2 < i3 && mbar_test(&s.mready, i2 & 1) &&
                    mbar_test(&s.xready[i2 & 1], (i2 >> 1) & 1)) {
                    tc_fence_after();
                    const bool fac = s.cv[i2 & 1].factored != 0;
                    const uint32_t aXV = smem_u32(fac ? s.XS[i2 & 1] : s.XR[i2 & 1]);
#pragma unroll
                    for (int k = 0; k < 8; ++k)
                        mma_bf16_ts(tbase + kColY + 64 * (i2 & 1), tbase + kColM + 8 * k,
                                    sdesc_sw128(aXV + k * 2048, 8192, 1024), kIdY, fac || k > 0);
                    mma_commit(&s.mfree);
                    mma_commit(&s.ydone[i2 & 1]);
                    ++i2;
                    progress = true;
                }
                if (progress) {
                    t_idle = 0;
                } else {
                    if (aborted(s)) {
                        ok = false;
                        break;
                    }
                    const uint64_t now = globaltimer_ns();
                    if (t_idle == 0) {
                        t_idle = now;
                    } else if (now - t_idle > kWaitNs) {
                        ok = false;
                        break;
                    }
                    __nanosleep(32);
                }
            }
            if (!ok) set_abort(s);
            // Nothing of ours may be in flight when the CTA leaves: wait (bounded)
            // for the last MMAs and for tiles loaded but never consumed.
            mma_commit(&s.fin);
            const uint64_t t0 = globaltimer_ns();
            while (!mbar_test(&s.fin, 0) && globaltimer_ns() - t0 < kWaitNs) __nanosleep(64);
            for (int k = i1; k < nC; ++k)
                while (!mbar_test(&s.full_c[k & 1], (k >> 1) & 1) && globaltimer_ns() - t0 < kWaitNs)
                    __nanosleep(64);
            for (int k = i1; k < nB; ++k)
                while (!mbar_test(&s.full_b, k & 1) && globaltimer_ns() - t0 < kWaitNs) __nanosleep(64);
        } else if (warp == 13 && nchunks > 0) {
            // ===================== gamma: per-chunk row values (one warp) =====================
            // lane l owns rows 4l .. 4l+3 of every chunk
            const float Ah = p.A[h];
            const float bias = p.dt_bias ? p.dt_bias[h] : 0.0f;
            const bool softplus = (p.flags & kDtSoftplus) != 0;
            constexpr float kLog2e = 1.4426950408889634f;
            float dtn[4];
            auto load_dt = [&](int c) {
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int r = c * Q + 4 * lane + i;
                    dtn[i] = r < S ? p.dt[((size_t)b * S + r) * H + h] : 0.0f;
                }
            };
            load_dt(0);
            for (int c = 0; c < nchunks; ++c) {
                const int rows = min(Q, S - c * Q);
                ChunkVals& cv = s.cv[c & 1];
                float dt[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const float d = softplus ? softplus_f32(dtn[i] + bias) : dtn[i];
                    dt[i] = 4 * lane + i < rows ? d : 0.0f;
                }
                if (c + 1 < nchunks) load_dt(c + 1);
                // inclusive sums of a = dt A over this lane's rows, then across lanes
                float gh[4], gl[4];
                gh[0] = dt[0] * Ah;
                gl[0] = 0.0f;
#pragma unroll
                for (int i = 1; i < 4; ++i) {
                    gh[i] = gh[i - 1];
                    gl[i] = gl[i - 1];
                    df_add(gh[i], gl[i], dt[i] * Ah, 0.0f);
                }
                float th = gh[3], tl = gl[3];
#pragma unroll
                for (int d = 1; d < 32; d <<= 1) {
                    const float oh = __shfl_up_sync(0xffffffffu, th, d);
                    const float ol = __shfl_up_sync(0xffffffffu, tl, d);
                    if (lane >= d) df_add(th, tl, oh, ol);
                }
                float eh = __shfl_up_sync(0xffffffffu, th, 1);
                float el = __shfl_up_sync(0xffffffffu, tl, 1);
                if (lane == 0) eh = el = 0.0f;
#pragma unroll
                for (int i = 0; i < 4; ++i) df_add(gh[i], gl[i], eh, el);
                // gamma_Q: the last element of the cumulative sum (rows past the
                // end add a = 0, so row Q-1 holds it)
                const float gLh = __shfl_sync(0xffffffffu, th, 31) * kLog2e;
                const float gLl = __shfl_sync(0xffffffffu, tl, 31) * kLog2e;
                const bool factored = Ah <= 0.0f && gLh + gLl >= kFactorMinLog2;
                float o_h[4], o_l[4], o_sc[4], o_dec[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const float g2h = gh[i] * kLog2e, g2l = gl[i] * kLog2e;
                    o_h[i] = g2h;
                    o_l[i] = g2l;
                    o_dec[i] = ex2_fast(fminf(g2h + g2l, 0.0f));
                    o_sc[i] = factored ? ex2_fast(-(g2h + g2l)) * dt[i]
                                       : ex2_fast(fminf((gLh - g2h) + (gLl - g2l), 0.0f)) * dt[i];
                }
                // cv[c&1] is free once the epilogue of chunk c-2 is done
                const bool ok = c < 2 || wait_or_abort(s, &s.epidone[c & 1], ((c >> 1) & 1) ^ 1);
                if (!__all_sync(0xffffffffu, ok)) break;
                reinterpret_cast<float4*>(cv.g2h)[lane] = make_float4(o_h[0], o_h[1], o_h[2], o_h[3]);
                reinterpret_cast<float4*>(cv.g2l)[lane] = make_float4(o_l[0], o_l[1], o_l[2], o_l[3]);
                reinterpret_cast<float4*>(cv.dts)[lane] = make_float4(dt[0], dt[1], dt[2], dt[3]);
                reinterpret_cast<float4*>(cv.sc)[lane] = make_float4(o_sc[0], o_sc[1], o_sc[2], o_sc[3]);
                reinterpret_cast<float4*>(cv.dec)[lane] = make_float4(o_dec[0], o_dec[1], o_dec[2], o_dec[3]);
                if (lane == 0) {
                    cv.decS = ex2_fast(fminf(gLh + gLl, 0.0f));
                    cv.factored = factored;
                }
                mbar_arrive(&s.cvready[c & 1]);
            }
        }
    } else if (wg == 0) {
        // ===================== conv: x rows of each chunk =====================
        regs_set<kConvRegs, kLaunchRegs>();
        const int jq = lane & 15;                           // channels 4 jq .. 4 jq + 3
        const int rbase = 32 * quarter + 16 * (lane >> 4);  // 16 rows of each chunk
        float2 wq[kMaxW][2], bq[2];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            bq[e] = p.conv ? s.bconv[2 * jq + e] : make_float2(0.f, 0.f);
#pragma unroll
            for (int k = 0; k < kMaxW; ++k)
                wq[k][e] = p.conv ? s.wconv[2 * jq + e][k] : make_float2(0.f, 0.f);
        }
        const __nv_bfloat16* xb =
            static_cast<const __nv_bfloat16*>(p.xbc) + (size_t)b * S * Cdim + h * P + 4 * jq;
        const __nv_bfloat16* csb =
            p.conv_state_in
                ? static_cast<const __nv_bfloat16*>(p.conv_state_in) + (size_t)b * (W - 1) * Cdim + h * P + 4 * jq
                : nullptr;
        uint2 raw[kRawRows];  // raw rows rbase-3 .. rbase+15 of the chunk (4 channels each)
        auto load_raw = [&](int c) {
            const int g0 = c * Q + rbase - (kMaxW - 1);
#pragma unroll
            for (int i = 0; i < kRawRows; ++i) {
                const int gr = g0 + i;
                uint2 v = make_uint2(0u, 0u);
                if (gr >= 0) {
                    if (gr < S) v = ldg_u2(xb + (size_t)gr * Cdim);
                } else if (csb != nullptr && gr + W - 1 >= 0) {
                    v = ldg_u2(csb + (size_t)(gr + W - 1) * Cdim);
                }
                raw[i] = v;
            }
        };
        load_raw(0);
        const uint32_t coff = (uint32_t)((jq & 1) << 3);
        for (int c = 0; c < nchunks; ++c) {
            const int buf = c & 1;
            const int rows = min(Q, S - c * Q);
            bool ok = wait_or_abort(s, &s.cvready[buf], (c >> 1) & 1);
            // XR / XS [buf] are free once the epilogue of chunk c-2 is done
            if (ok && c >= 2) ok = wait_or_abort(s, &s.epidone[buf], ((c >> 1) & 1) ^ 1);
            if (!ok) break;
            const float* scv = s.cv[buf].sc;
            float2 win[kMaxW - 1][2];
#pragma unroll
            for (int k = 0; k < kMaxW - 1; ++k) {
                win[k][0] = unpack2(raw[k].x);
                win[k][1] = unpack2(raw[k].y);
            }
#pragma unroll
            for (int i4 = 0; i4 < 4; ++i4) {
                const float4 sc4 = *reinterpret_cast<const float4*>(&scv[rbase + 4 * i4]);
                const float scs[4] = {sc4.x, sc4.y, sc4.z, sc4.w};
#pragma unroll
                for (int ii = 0; ii < 4; ++ii) {
                    const int i = 4 * i4 + ii;
                    const int r = rbase + i;
                    const float2 u0 = unpack2(raw[i + kMaxW - 1].x), u1 = unpack2(raw[i + kMaxW - 1].y);
                    float2 x0, x1;
                    if (p.conv) {
                        float2 a0 = bq[0], a1 = bq[1];
#pragma unroll
                        for (int k = 0; k < kMaxW - 1; ++k) {
                            a0 = __ffma2_rn(wq[k][0], win[k][0], a0);
                            a1 = __ffma2_rn(wq[k][1], win[k][1], a1);
                        }
                        a0 = __ffma2_rn(wq[kMaxW - 1][0], u0, a0);
                        a1 = __ffma2_rn(wq[kMaxW - 1][1], u1, a1);
                        x0 = silu2(a0);
                        x1 = silu2(a1);
                    } else {
                        x0 = u0;
                        x1 = u1;
                    }
                    if (r >= rows) x0 = x1 = make_float2(0.f, 0.f);
                    const float2 sc2 = make_float2(scs[ii], scs[ii]);
                    const uint32_t off = chunk_off(r, jq >> 1) + coff;
                    at<uint2>(s.XR[buf], off) = make_uint2(pack2(x0), pack2(x1));
                    at<uint2>(s.XS[buf], off) =
                        make_uint2(pack2(__fmul2_rn(sc2, x0)), pack2(__fmul2_rn(sc2, x1)));
#pragma unroll
                    for (int k = 0; k < kMaxW - 2; ++k) {
                        win[k][0] = win[k + 1][0];
                        win[k][1] = win[k + 1][1];
                    }
                    win[kMaxW - 2][0] = u0;
                    win[kMaxW - 2][1] = u1;
                }
            }
            fence_proxy_async_smem();  // XR / XS are read by G4 / G2
            mbar_arrive(&s.xready[buf]);
            if (c + 1 < nchunks) load_raw(c + 1);
        }
    } else if (wg == 1) {
        // ===================== mask: CB -> M in TMEM =====================
        regs_set<kMaskRegs, kLaunchRegs>();
        const int t = tid - kWG;  // chunk row of this thread (its TMEM lane)
        // blocks of M strictly above the diagonal stay zero for the whole sequence
        {
            uint32_t zero[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) zero[i] = 0u;
            for (int cc = quarter + 1; cc < 4; ++cc) tmem_st16(tbase + lane_off + kColM + 16 * cc, zero);
            tmem_st_wait();
        }
        for (int c = 0; c < nchunks; ++c) {
            const int buf = c & 1;
            const ChunkVals& cv = s.cv[buf];
            bool ok = wait_or_abort(s, &s.cvready[buf], (c >> 1) & 1);
            if (ok) ok = wait_or_abort(s, &s.g1, c & 1);                     // CB(c)
            if (ok && c >= 1) ok = wait_or_abort(s, &s.mfree, (c - 1) & 1);  // G2(c-1) read M
            if (!__all_sync(0xffffffffu, ok)) {
                set_abort(s);
                break;
            }
            tc_fence_after();
            const bool factored = cv.factored != 0;
            const float g2h_t = cv.g2h[t], g2l_t = cv.g2l[t];
#pragma unroll 1
            for (int cc = 0; cc <= quarter; ++cc) {  // 32-column blocks of s
                float v[32];
                tmem_ld32(tbase + lane_off + kColCB + 32 * cc, v);
                tmem_ld_wait();
                if (!factored) {
#pragma unroll
                    for (int q4 = 0; q4 < 8; ++q4) {
                        const int sb = cc * 32 + 4 * q4;
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
                    for (int e = 0; e < 32; ++e) v[e] = (cc * 32 + e <= t) ? v[e] : 0.0f;
                }
                uint32_t m[16];
#pragma unroll
                for (int e = 0; e < 16; ++e) m[e] = pack2(make_float2(v[2 * e], v[2 * e + 1]));
                tmem_st16(tbase + lane_off + kColM + 16 * cc, m);
            }
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive(&s.mready);
        }
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
        auto store_h = [&](int slot) {
#pragma unroll
            for (int q8 = 0; q8 < 8; ++q8) at<uint4>(s.Hs[slot], chunk_off(n, q8)) = pack4x2(&hreg[4 * q8]);
        };
        // h of chunk -1 (the initial state) in slot 0
        store_h(0);
        fence_proxy_async_smem();
        mbar_arrive(&s.hsready[0]);
        const __nv_bfloat16* zbase = static_cast<const __nv_bfloat16*>(p.z);
        const float Dh = p.D ? p.D[h] : 0.0f;
        // state(c): h_c = decS h_{c-1} + b dH(c), stored to slot (c+1)&1
        auto state = [&](int c) -> bool {
            const int buf = c & 1;
            const ChunkVals& cv = s.cv[buf];
            bool ok = wait_or_abort(s, &s.cvready[buf], (c >> 1) & 1);
            if (ok) ok = wait_or_abort(s, &s.g4[buf], (c >> 1) & 1);
            // slot (c+1)&1 was last read by G3(c-1)
            if (ok && c >= 1) ok = wait_or_abort(s, &s.g3[(c - 1) & 1], ((c - 1) >> 1) & 1);
            if (!__all_sync(0xffffffffu, ok)) return false;
            tc_fence_after();
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
            store_h((c + 1) & 1);
            fence_proxy_async_smem();
            tc_fence_before();
            mbar_arrive(&s.hsready[(c + 1) & 1]);
            return true;
        };
        bool ok = nchunks == 0 || state(0);
        for (int c = 0; c < nchunks && ok; ++c) {
            const int buf = c & 1;
            const int r0 = c * Q;
            const int rows = min(Q, S - r0);
            // z of this row, early (used at the end)
            uint4 zq[8];
            if (has_z) {
                const uint4* zr = reinterpret_cast<const uint4*>(
                    zbase + ((size_t)b * S + r0 + min(t, rows - 1)) * (H * P) + h * P);
#pragma unroll
                for (int q8 = 0; q8 < 8; ++q8) zq[q8] = __ldg(zr + q8);
            }
            // the state runs one chunk ahead of the epilogue
            if (c + 1 < nchunks && !state(c + 1)) {
                ok = false;
                break;
            }
            // ---- epilogue(c) ----
            const ChunkVals& cv = s.cv[buf];
            ok = wait_or_abort(s, &s.ydone[buf], (c >> 1) & 1);
            if (!__all_sync(0xffffffffu, ok)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const bool factored = cv.factored != 0;
            // factored: y = u Y + D x;  exact: y = Y + u Yo + D x
            const float dec = cv.dec[t];
            const float2 dd = make_float2(dec, dec);
            const float2 D2 = make_float2(Dh, Dh);
            uint4* yrow = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.y) +
                                                   (((size_t)b * S + r0 + t) * H + h) * P);
#pragma unroll
            for (int half = 0; half < 2; ++half) {  // 32 columns (4 chunks of 8 p) at a time
                float yv[32];
                tmem_ld32(tbase + kColY + 64 * buf + lane_off + 32 * half, yv);
                if (!factored) {
                    float yo[32];
                    tmem_ld32(tbase + kColYo + lane_off + 32 * half, yo);
                    tmem_ld_wait();
#pragma unroll
                    for (int k = 0; k < 32; k += 2) {
                        const float2 r = __ffma2_rn(dd, make_float2(yo[k], yo[k + 1]),
                                                    make_float2(yv[k], yv[k + 1]));
                        yv[k] = r.x;
                        yv[k + 1] = r.y;
                    }
                } else {
                    tmem_ld_wait();
#pragma unroll
                    for (int k = 0; k < 32; k += 2) {
                        const float2 r = __fmul2_rn(dd, make_float2(yv[k], yv[k + 1]));
                        yv[k] = r.x;
                        yv[k + 1] = r.y;
                    }
                }
#pragma unroll
                for (int j4 = 0; j4 < 4; ++j4) {
                    const int j = 4 * half + j4;  // 16-byte chunk of the row (8 p)
                    float2 out[4], zv[4], xv[4];
                    if (has_z) unpack4x2(zq[j], zv);
                    unpack4x2(at<const uint4>(s.XR[buf], chunk_off(t, j)), xv);
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int k = j4 * 8 + 2 * e;
                        float2 v = __ffma2_rn(D2, xv[e], make_float2(yv[k], yv[k + 1]));
                        if (has_z) v = __fmul2_rn(v, silu2(zv[e]));
                        out[e] = v;
                    }
                    if (t < rows) yrow[j] = pack4x2(out);
                }
            }
            tc_fence_before();
            mbar_arrive(&s.epidone[buf]);
        }
        if (ok && !aborted(s)) {
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                p.hS[sbase + (size_t)(2 * i) * N + n] = hreg[i].x;
                p.hS[sbase + (size_t)(2 * i + 1) * N + n] = hreg[i].y;
            }
        } else {
            set_abort(s);
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
    CUtensorMap mbc;
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
    scan_tc_kernel<<<grid, kThreads, kSmemBytes, st>>>(mbc, p);
    return cudaGetLastError();
}

}  // namespace ssd
