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
//   factored (a <= 0, the chunk's total decay moderate, every dt > 0): with
//     u_t = exp(gamma_t) and v_s = exp(-gamma_s) dt_s (so u_t v_t = dt_t),
//     M = mask(CB) + diag(D / dt), xv = xs = v o x, y = u_t Y,
//     h <- exp(gamma_Q) (h + dH): G3 and G2 share one accumulator;
//   exact (otherwise): M = mask(CB o exp(min(gamma_t - gamma_s, 0)) dt_s) + diag(D),
//     xv = x, xs = w o x with w_s = exp(min(gamma_Q - gamma_s, 0)) dt_s,
//     G3 goes to its own accumulator Yo, y = Y + u_t Yo,
//     h <- exp(gamma_Q) h + dH.
//     Split blocks: when gamma never rises in the chunk (every a <= 0), the
//     decay of a 32-row block j of columns splits at its middle row m_j as
//     exp(gamma_t - gamma_m) exp(gamma_m - gamma_s).  The column factor
//     V_s = exp(gamma_m - gamma_s) dt_s scales the x rows G2 reads
//     (xv = V o x) and the mask keeps one factor per row, R_t =
//     exp(gamma_t - gamma_m): M = mask(CB R_t) with D R_t / dt_t on the
//     diagonal.  Below the diagonal R_t <= 1; inside block j both factors
//     stay within 2^60 when neither half of the block decays by more than
//     2^60, the condition for the split (else the block's columns keep the
//     per-element exponential and xv = x).
// The skip term D x_t rides on the diagonal of M.  The masked CB is written
// back into TMEM (bf16 pairs) and read from there by G2, so it never passes
// through shared memory.
//
// Threads (576): 16 compute warps, a control warp and a gamma warp.
//  - gamma warp: for up to four chunks ahead, dt (softplus + bias), the
//    double-float cumulative sum of a = dt A, the form of the chunk and the
//    per-row factors, into a ring of per-chunk value sets in shared memory.
//  - control warp (one thread): every TMA load (the C and B tiles of the next
//    chunk into the one C and B buffers once G4 of this chunk -- and so G1,
//    G3, issued before it -- is done; the raw x rows of the chunk after next,
//    with the 4 rows before them, double-buffered, once the conv of this chunk
//    is done; the z tile of the next chunk, double-buffered, once the mask of
//    this chunk is done) and every MMA, each as soon as its operands are ready
//    (mbarriers from the compute warps).
//  - compute warps, phase by phase on every chunk: mask (one 32x32 block of a
//    TMEM lane quarter per warp, warp % 4 = quarter), state update (16 state
//    columns per warp, h in fp32 registers, its bf16 copy into shared memory
//    for G3), conv of the next chunk (4 rows x 4 channels per thread: causal
//    taps over the raw rows of its TMA tiles, SiLU, the x and scaled-x
//    tiles), epilogue (16 columns of a lane quarter per warp: z from
//    its TMA tile, y written over it in place, each quarter's rows leaving
//    with one TMA store).  At the end they write the final state and the new
//    conv state.
// Per-thread global accesses that would scatter a warp over 32 rows (z, y)
// go through TMA tiles instead: the load/store unit would otherwise spend 32
// requests on every such instruction.  The raw x rows come by TMA too: per-
// thread loads of them a chunk ahead cost the compute warps ~0.5 us per chunk
// in issue and held 14 registers through every phase.  Every wait is bounded in time; a wait
// that runs out aborts the CTA (the other waits then fail fast) and sets the
// device error word.
#include "internal.cuh"
#include "sm100.cuh"

#include <cudaTypedefs.h>
#include <cuda_fp16.h>

#include <cstddef>
#include <cstring>
#include <mutex>

namespace ssd {
namespace {

using namespace sm100;

constexpr int Q = 128;  // rows per chunk
constexpr int P = 64;   // head dim
constexpr int N = 128;  // state dim
constexpr int kCompute = 512;              // compute threads (16 warps)
constexpr int kControlWarp = 16;           // TMA + MMA issue
constexpr int kGammaWarp = 17;             // per-chunk values
constexpr int kThreads = kCompute + 64;
constexpr int kCv = 4;                     // per-chunk value sets in flight
constexpr int kMaxW = 4;  // conv taps handled in the kernel (W-1 carried rows)
constexpr int kRaw = 4 + kMaxW - 1;          // raw rows a conv thread reads per chunk
constexpr uint64_t kWaitNs = 2000000000ull;  // default bound on a wait (the final drain's always)

// G1: A, B K-major.  G2, G3: A K-major, B MN-major (row tiles [k][p]).
// G4: A = B^T read MN-major from the B tile, B MN-major.
constexpr uint32_t kIdCB = idesc_bf16_f32(128, 128, false, false);
constexpr uint32_t kIdY = idesc_bf16_f32(128, 64, false, true);
constexpr uint32_t kIdState = idesc_bf16_f32(128, 64, true, true);

// TMEM columns (512 allocated)
constexpr uint32_t kColCB = 0;    // CB fp32 [t][s]                        128
constexpr uint32_t kColM = 128;   // M bf16 pairs [t][s/2]                  64
constexpr uint32_t kColY = 192;   // Y fp32 [t][p], by chunk parity     2 x 64
constexpr uint32_t kColYo = 320;  // Yo fp32 [t][p] (exact), by parity  2 x 64
constexpr uint32_t kColDH = 448;  // dH fp32 [n][p]                         64

// Below this total chunk decay (log2 units) the mask factors as
// exp(gamma_t) * exp(-gamma_s): every factor stays within fp32 (2^90 < 2^127).
constexpr float kFactorMinLog2 = -90.0f;
// Exact form: a column block splits at its middle row when neither half decays
// by more than this (log2 units): R_t and V_s / dt_s then stay within 2^60.
constexpr float kSplitMaxLog2 = 60.0f;

struct __align__(16) ChunkVals {  // per-chunk row values, written by the gamma warp
    float g2h[Q], g2l[Q];      // gamma * log2(e), double-float (hi, lo)
    float dts[Q];              // dt_s (0 past the last row)
    float sc[Q];               // x scale of G4's operand: v_s (factored) or w_s (exact)
    float vb[Q];               // scale of the x rows G2 reads in the exact form: V_s
                               // (split blocks) or 1
    float decS;                // exp(min(gamma_Q, 0))
    int factored;              // which form of the decay this chunk uses
    int split;                 // exact form: bit j set when column block j is split
    int pad;
};

struct __align__(1024) TcSmem {
    __nv_bfloat16 C[2][Q * 64];     // C tile [t][n]: 2 panels of 64 n (TMA, SW128); one chunk
    __nv_bfloat16 B[2][Q * 64];     // B tile [s][n]: 2 panels of 64 n (TMA, SW128); one chunk
    __nv_bfloat16 XS[2][Q * 64];    // scaled x rows [s][p] (SW128): v o x or w o x, by parity
    __nv_bfloat16 XR[2][Q * 64];    // x rows [s][p] (exact chunks), by parity
    __nv_bfloat16 XRAW[2][Q * 64];  // raw x rows [t][p] of a chunk (TMA, SW128), by parity
    __nv_bfloat16 Hs[N * 64];       // bf16 state rows [n][p] of the previous chunk: G3's B
    __nv_bfloat16 Zt[2][Q * 64];    // z rows [t][p] by chunk parity (TMA, SW128); y written
                                    // over them in place, stored by 32-row quarters
    __nv_bfloat16 XH[2][4 * 64];    // the 4 raw x rows before a chunk (TMA, unswizzled), by parity
    ChunkVals cv[kCv];              // ring of per-chunk values
    // taps by [tap][channel pair] (front-padded with zeros): a thread reads its two
    // pairs of a tap as one 16-byte vector, a half-warp a contiguous 256 bytes
    alignas(16) float2 wconv[kMaxW][P / 2];
    alignas(16) float2 bconv[P / 2];
    uint64_t full_c, full_b, full_z[2], full_x[2];  // TMA landed
    uint64_t g1, g3, g4, g2, fin;   // MMA commits
    uint64_t xready[2], mready, hsready;                 // compute -> control (xready by chunk parity)
    uint64_t cvready[kCv], epidone[kCv];                 // gamma warp <-> compute
    uint32_t tmem_base;
    int abort;
    // gated group RMSNorm share of the epilogue (the kNorm instantiation)
    float nsum[2][4][Q];  // by chunk parity, column group j, row: sum of y^2 over 16 channels
};

constexpr size_t kSmemBytes = sizeof(TcSmem) + 1024;

// operand tiles start on 1024-byte swizzle atoms; vector-accessed members on
// their vector size
static_assert(offsetof(TcSmem, C) % 1024 == 0 && offsetof(TcSmem, B) % 1024 == 0, "tile");
static_assert(offsetof(TcSmem, XS) % 1024 == 0 && offsetof(TcSmem, XR) % 1024 == 0, "tile");
static_assert(sizeof(((TcSmem*)nullptr)->XS[0]) % 1024 == 0, "tile");
static_assert(sizeof(((TcSmem*)nullptr)->XR[0]) % 1024 == 0, "tile");
static_assert(offsetof(TcSmem, Hs) % 1024 == 0 && offsetof(TcSmem, XRAW) % 1024 == 0, "tile");
static_assert(offsetof(TcSmem, XH) % 128 == 0 && sizeof(((TcSmem*)nullptr)->XH[0]) % 128 == 0, "tile");
static_assert(sizeof(ChunkVals) % 16 == 0 && offsetof(TcSmem, cv) % 16 == 0, "float4 rows");
static_assert(offsetof(ChunkVals, g2l) % 16 == 0 && offsetof(ChunkVals, dts) % 16 == 0, "float4");
static_assert(offsetof(ChunkVals, sc) % 16 == 0 && offsetof(ChunkVals, vb) % 16 == 0, "float4");
static_assert(offsetof(TcSmem, wconv) % 16 == 0 && offsetof(TcSmem, bconv) % 16 == 0, "float4");
static_assert(offsetof(TcSmem, Zt) % 1024 == 0, "tile");
static_assert(offsetof(TcSmem, full_c) % 8 == 0, "mbarriers");
static_assert(kSmemBytes <= 232448, "shared memory per CTA");


// silu(v) = v sigmoid(v) = 0.5 v (1 + tanh(v / 2)), two lanes at a time, with
// one half-precision tanh for both (one transcendental-unit operation instead
// of two; its absolute error, ~2^-10, is of the order of the fp32 approximate
// tanh's and below the bf16 rounding of every result).
__device__ __forceinline__ float2 silu2(float2 v)
{
    const float2 hv = __fmul2_rn(v, make_float2(0.5f, 0.5f));
    const __half2 hh = __float22half2_rn(hv);
    uint32_t th;
    asm("tanh.approx.f16x2 %0, %1;" : "=r"(th) : "r"(*reinterpret_cast<const uint32_t*>(&hh)));
    return __ffma2_rn(hv, __half22float2(*reinterpret_cast<const __half2*>(&th)), hv);
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

// (hi, lo) * log2(e) as a double-float: the product of hi with the fp32 part
// of log2(e), its exact rounding error by FMA (Dekker's product), plus the
// terms of lo and of log2(e)'s low part, renormalised.  A plain fp32 product
// hi * log2(e) would drop up to half an ulp of |gamma| (0.06 at |gamma| ~ 1e6),
// which exp2 turns into a relative error of several percent.
__device__ __forceinline__ void df_to_log2(float hi, float lo, float& rh, float& rl)
{
    constexpr float kL = 1.4426950408889634f;     // log2(e) rounded to fp32
    constexpr float kLlo = 1.925963e-8f;          // log2(e) - kL
    const float p = hi * kL;
    float e = fmaf(hi, kL, -p);
    e += fmaf(hi, kLlo, lo * kL);
    rh = p + e;
    rl = e - (rh - p);
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

template <typename SM>
__device__ __forceinline__ bool aborted(SM& s)
{
    return *reinterpret_cast<volatile int*>(&s.abort) != 0;
}

template <typename SM>
__device__ __forceinline__ void set_abort(SM& s)
{
    *reinterpret_cast<volatile int*>(&s.abort) = 1;
}

// Bounded wait that also gives up as soon as another thread has aborted.
// The hinted try_wait suspends the thread until the phase completes (or
// about a microsecond passes), so a waiting warp takes no issue slots.
template <typename SM>
__device__ __forceinline__ bool wait_or_abort(SM& s, uint64_t* bar, uint32_t parity,
                                              uint64_t limit_ns)
{
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    while (true) {
        if (mbar_try_wait_hint(bar, parity, 1000)) return true;
        if (aborted(s)) return false;
        if (globaltimer_ns() - t0 > limit_ns) {
            set_abort(s);
            return false;
        }
    }
}

template <bool kVarlen, bool kNorm>
__global__ void __launch_bounds__(kThreads, 1)
    scan_tc_kernel(const __grid_constant__ CUtensorMap map_bc, const __grid_constant__ CUtensorMap map_z,
                   const __grid_constant__ CUtensorMap map_y, const __grid_constant__ CUtensorMap map_x,
                   const __grid_constant__ CUtensorMap map_xh, const TcScanParams p)
{
    // Align to the 1024-byte swizzle atom with pointer arithmetic on the
    // shared array itself, so the compiler keeps every access in the shared
    // address space (LDS/STS rather than generic loads and stores).
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    TcSmem& s = *reinterpret_cast<TcSmem*>(smem_raw + ((1024u - (sm100::smem_u32(smem_raw) & 1023u)) & 1023u));
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int h = blockIdx.x, b = blockIdx.y;  // head, sequence
    const int H = p.H, G = p.G, W = p.W;
    // this CTA's sequence: its first row in the row arrays, its rows, its state
    // slot, and whether its states start from the slot or from zeros
    long long row0 = (long long)b * p.S;
    int S = p.S, slot = b;
    bool init = true;
    if constexpr (kVarlen) {
        row0 = p.cu_seqlens[b];
        const long long end = p.cu_seqlens[b + 1];
        slot = p.slot_ids[b];
        init = p.has_init == nullptr || p.has_init[b] != 0;
        // a bad row range or slot: report it and leave (every thread of the CTA
        // read the same values, so all of them leave here, before any setup)
        if (row0 < 0 || end < row0 || end > p.S || slot < 0 || slot >= p.num_slots) {
            if (threadIdx.x == 0) atomicOr(p.err, kErrBadSlot);
            return;
        }
        // debug check: an earlier sequence of this call owns the slot
        if (p.check_dups && slot_seen_before(p.slot_ids, b, slot)) {
            if (threadIdx.x == 0 && h == 0) atomicOr(p.err, kErrDupSlot);
            return;
        }
        S = (int)(end - row0);
    }
    const float* h0 = init ? p.h0 : nullptr;
    const void* cs_in = init ? p.conv_state_in : nullptr;
    // tile coordinates of chunk c: row and batch of the [cols, rows, batch] maps
    const int tz = kVarlen ? 0 : b;
    auto trow = [&](int c) { return kVarlen ? (int)(row0 + (long long)c * Q) : c * Q; };
    const int g = h / (H / G);
    const int Cdim = H * P + 2 * G * N;
    const int nchunks = (S + Q - 1) / Q;
    const bool has_z = (p.flags & kHasZ) != 0;
    const uint64_t wlim = p.wait_ns ? p.wait_ns : kWaitNs;  // pipeline waits

    // Work that needs nothing from the setup starts before its barrier: the
    // control thread's raw x tiles of the first two chunks (it initialises their
    // barriers itself) and the gamma warp's first dt rows.
    int loaded_x = 0;  // raw x tiles requested (control thread)
    auto load_x = [&](int c) {  // raw x tile of chunk c and the 4 rows before it
        const int kx = c & 1;
        mbar_arrive_expect_tx(&s.full_x[kx], Q * 64 * 2 + (c > 0 ? 4 * 64 * 2 : 0));
        tma_load_3d(s.XRAW[kx], &map_x, &s.full_x[kx], h * P, trow(c), tz);
        if (c > 0) tma_load_3d(s.XH[kx], &map_xh, &s.full_x[kx], h * P, trow(c) - 4, tz);
        loaded_x = c + 1;
    };
    if (warp == kControlWarp && lane == 0) {
        mbar_init(&s.full_x[0], 1);
        mbar_init(&s.full_x[1], 1);
        fence_mbar_init();
        if (nchunks > 0) {
            prefetch_tmap(&map_x);
            load_x(0);
            if (nchunks > 1) load_x(1);
        }
    }
    float dt0[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    if (warp == kGammaWarp) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int r = 4 * lane + i;
            if (r < S) dt0[i] = p.dt[((size_t)row0 + r) * H + h];
        }
    }
    if (tid == 0) {
        mbar_init(&s.full_c, 1);
        mbar_init(&s.full_z[0], 1);
        mbar_init(&s.full_z[1], 1);
        mbar_init(&s.full_b, 1);
        mbar_init(&s.g1, 1);
        mbar_init(&s.g3, 1);
        mbar_init(&s.g4, 1);
        mbar_init(&s.g2, 1);
        mbar_init(&s.fin, 1);
        mbar_init(&s.xready[0], kCompute);
        mbar_init(&s.xready[1], kCompute);
        mbar_init(&s.mready, kCompute);
        mbar_init(&s.hsready, kCompute);
        for (int i = 0; i < kCv; ++i) {
            mbar_init(&s.cvready[i], 32);
            mbar_init(&s.epidone[i], kCompute);
        }
        s.abort = 0;
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(&s.tmem_base, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = s.tmem_base;

    if (warp == kControlWarp) {
        // ===================== control: TMA + MMA (one thread) =====================
        // Order: G1(0), G3(0); per chunk c: G4(c), then (once G4(c) is done, so
        // are G1(c) and G3(c), issued before it) the C tile of chunk c+1 into the
        // one C buffer and the B tile of chunk c+2 into B[c&1]; G2(c), G1(c+1),
        // G3(c+1).  G3(c+1) needs only h of chunk c, so it runs while the compute
        // warps convolve chunk c+1; only G4 separates that conv from the next
        // state update.
        if (lane == 0 && nchunks > 0) {
            prefetch_tmap(&map_bc);
            // launched to overlap the B|C conv that writes the bc tiles (when there
            // is one): wait for it here, before the first tile load.  Every read of
            // the old conv state by that kernel is then done too, so the new conv
            // state written at the end (it may overwrite the old one in place) is
            // ordered after it: its writers wait on MMAs issued after this point.
            griddep_wait();
            const int xB = p.bc_col0 + g * N;          // first B column in the bc source
            const int xC = p.bc_col0 + G * N + g * N;  // first C column
            int loaded_c = 0, loaded_b = 0, loaded_z = 0;  // tiles requested so far
            auto load_c = [&](int c) {  // C tile of chunk c (the one buffer)
                mbar_arrive_expect_tx(&s.full_c, 2 * Q * 64 * 2);
                tma_load_3d(s.C[0], &map_bc, &s.full_c, xC, trow(c), tz);
                tma_load_3d(s.C[1], &map_bc, &s.full_c, xC + 64, trow(c), tz);
                loaded_c = c + 1;
            };
            auto load_b = [&](int c) {  // B tile of chunk c (the one buffer)
                mbar_arrive_expect_tx(&s.full_b, 2 * Q * 64 * 2);
                tma_load_3d(s.B[0], &map_bc, &s.full_b, xB, trow(c), tz);
                tma_load_3d(s.B[1], &map_bc, &s.full_b, xB + 64, trow(c), tz);
                loaded_b = c + 1;
            };
            // K step k of a K-major operand: (k>>2)*16 KB + (k&3)*32 B; of an MN-major
            // one: 2 KB (16 rows).  Descriptors count 16-byte units in their start
            // address field (no carry for shared addresses).
            auto kmaj = [](int k) { return (uint64_t)(((k >> 2) << 10) + ((k & 3) << 1)); };
            const uint64_t dHs = sdesc_sw128(smem_u32(s.Hs), 8192, 1024);
            const uint64_t dXS0 = sdesc_sw128(smem_u32(s.XS[0]), 8192, 1024);
            const uint64_t dXS1 = sdesc_sw128(smem_u32(s.XS[1]), 8192, 1024);
            const uint64_t dXR0 = sdesc_sw128(smem_u32(s.XR[0]), 8192, 1024);
            const uint64_t dXR1 = sdesc_sw128(smem_u32(s.XR[1]), 8192, 1024);
            const uint64_t dC = sdesc_sw128(smem_u32(s.C), 16, 1024);
            auto g1 = [&](int c) {
                const uint64_t dA = dC;
                const uint64_t dB = sdesc_sw128(smem_u32(s.B), 16, 1024);
#pragma unroll
                for (int k = 0; k < 8; ++k)
                    mma_bf16_ss(tbase + kColCB, dA + kmaj(k), dB + kmaj(k), kIdCB, k > 0);
                mma_commit(&s.g1);
            };
            // G3(c): h of chunk c-1 in the state tile; Y / Yo [c&1] read by the
            // epilogue of chunk c-2; the values of chunk c say which accumulator
            auto g3 = [&](int c) -> bool {
                bool r = wait_or_abort(s, &s.hsready, c & 1, wlim) &&
                         wait_or_abort(s, &s.cvready[c % kCv], (c / kCv) & 1, wlim);
                if (r && c >= 2) r = wait_or_abort(s, &s.epidone[(c - 2) % kCv], ((c - 2) / kCv) & 1, wlim);
                if (!r) return false;
                tc_fence_after();
                const uint32_t dY = (s.cv[c % kCv].factored ? kColY : kColYo) + 64 * (c & 1);
                const uint64_t dA = dC;
#pragma unroll
                for (int k = 0; k < 8; ++k)
                    mma_bf16_ss(tbase + dY, dA + kmaj(k), dHs + 128 * k, kIdY, k > 0);
                mma_commit(&s.g3);
                return true;
            };
            // z tile of chunk c into buffer c & 1
            auto load_z = [&](int c) {
                mbar_arrive_expect_tx(&s.full_z[c & 1], Q * 64 * 2);
                tma_load_3d(s.Zt[c & 1], &map_z, &s.full_z[c & 1], h * P, trow(c), tz);
                loaded_z = c + 1;
            };
            if (has_z) {
                prefetch_tmap(&map_z);
                load_z(0);
                if (nchunks > 1) load_z(1);
            }
            load_c(0);
            load_b(0);
            bool ok = wait_or_abort(s, &s.full_c, 0, wlim) && wait_or_abort(s, &s.full_b, 0, wlim);
            if (ok) {
                tc_fence_after();
                g1(0);
                ok = g3(0);
            }
            for (int c = 0; c < nchunks && ok; ++c) {
                const int kb = c & 1;
                // G4(c): x rows of chunk c in place; dH read by state(c-1)
                ok = wait_or_abort(s, &s.xready[c & 1], (c >> 1) & 1, wlim) && wait_or_abort(s, &s.hsready, c & 1, wlim);
                if (!ok) break;
                // the conv of chunk c is done with its raw tile: chunk c+2's goes there
                if (c + 2 < nchunks) load_x(c + 2);
                tc_fence_after();
                {
                    const uint64_t dA = sdesc_sw128(smem_u32(s.B), Q * 128, 1024);
#pragma unroll
                    for (int k = 0; k < 8; ++k)
                        mma_bf16_ss(tbase + kColDH, dA + 128 * k, (kb ? dXS1 : dXS0) + 128 * k, kIdState, k > 0);
                    mma_commit(&s.g4);
                }
                // tiles of chunk c+1: C (G1(c), G3(c) done) and B (G1(c), G4(c) done)
                if (c + 1 < nchunks) {
                    ok = wait_or_abort(s, &s.g4, c & 1, wlim);
                    if (!ok) break;
                    load_c(c + 1);
                    load_b(c + 1);
                }
                // z of chunk c once the epilogue of chunk c-1 is done (it comes before
                // the mask of chunk c, so this does not hold up G2(c))
                // G2(c): M(c) in TMEM (CB(c) consumed); onto G3(c) (factored) or fresh
                ok = wait_or_abort(s, &s.mready, c & 1, wlim);
                if (!ok) break;
                // z of chunk c+1 into the buffer of chunk c-1: its epilogue read the z
                // rows and its y store read the tile before these arrivals
                if (has_z && c >= 1 && c + 1 < nchunks) load_z(c + 1);
                tc_fence_after();
                {
                    const bool fac = s.cv[c % kCv].factored != 0;
                    const uint64_t dB = fac ? (kb ? dXS1 : dXS0) : (kb ? dXR1 : dXR0);
#pragma unroll
                    for (int k = 0; k < 8; ++k)
                        mma_bf16_ts(tbase + kColY + 64 * kb, tbase + kColM + 8 * k, dB + 128 * k, kIdY,
                                    fac || k > 0);
                    mma_commit(&s.g2);
                }
                if (c + 1 < nchunks) {
                    // G1(c+1): its tiles landed
                    ok = wait_or_abort(s, &s.full_c, (c + 1) & 1, wlim) &&
                         wait_or_abort(s, &s.full_b, (c + 1) & 1, wlim);
                    if (!ok) break;
                    tc_fence_after();
                    g1(c + 1);
                    ok = g3(c + 1);
                    if (!ok) break;
                }
            }
            if (!ok) set_abort(s);
            // nothing of ours may be in flight when the CTA leaves (bounded waits)
            mma_commit(&s.fin);
            const uint64_t t0 = globaltimer_ns();
            while (!mbar_test(&s.fin, 0) && globaltimer_ns() - t0 < kWaitNs) __nanosleep(64);
            if (loaded_c > 0) {
                const int k = loaded_c - 1;
                while (!mbar_test(&s.full_c, k & 1) && globaltimer_ns() - t0 < kWaitNs) __nanosleep(64);
            }
            if (loaded_b > 0) {
                const int k = loaded_b - 1;
                while (!mbar_test(&s.full_b, k & 1) && globaltimer_ns() - t0 < kWaitNs) __nanosleep(64);
            }
            for (int k = max(0, loaded_x - 2); k < loaded_x; ++k)  // the last load into each buffer
                while (!mbar_test(&s.full_x[k & 1], (k >> 1) & 1) && globaltimer_ns() - t0 < kWaitNs)
                    __nanosleep(64);
            for (int k = max(0, loaded_z - 2); k < loaded_z; ++k)  // the last load into each buffer
                while (!mbar_test(&s.full_z[k & 1], (k >> 1) & 1) && globaltimer_ns() - t0 < kWaitNs)
                    __nanosleep(64);
        }
    } else if (warp == kGammaWarp) {
        // ===================== gamma: per-chunk row values (one warp) =====================
        // lane l owns rows 4l .. 4l+3 of every chunk; runs up to kCv chunks ahead
        const float Ah = p.A[h];
        const float bias = p.dt_bias ? p.dt_bias[h] : 0.0f;
        const float Dabs = p.D ? fabsf(p.D[h]) : 0.0f;
        const bool softplus = (p.flags & kDtSoftplus) != 0;
        float dtn[4] = {dt0[0], dt0[1], dt0[2], dt0[3]};
        auto load_dt = [&](int c) {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int r = c * Q + 4 * lane + i;
                dtn[i] = r < S ? p.dt[((size_t)row0 + r) * H + h] : 0.0f;
            }
        };
        for (int c = 0; c < nchunks; ++c) {
            const int rows = min(Q, S - c * Q);
            ChunkVals& cv = s.cv[c % kCv];
            float dt[4];
            bool dt_ok = true;  // the factored form also needs D / dt finite on every row
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float d = softplus ? softplus_f32(dtn[i] + bias) : dtn[i];
                const bool valid = 4 * lane + i < rows;
                dt[i] = valid ? d : 0.0f;
                dt_ok = dt_ok && (!valid || (dt[i] > 0.0f && Dabs < dt[i] * 1e30f));
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
            // gamma in log2 units, per row; gamma_Q is the last element of the
            // cumulative sum as stored for row Q-1 (rows past the end add a = 0),
            // so its difference with that row is exactly 0
            float o_h[4], o_l[4], o_sc[4], o_vb[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) df_to_log2(gh[i], gl[i], o_h[i], o_l[i]);
            const float gLh = __shfl_sync(0xffffffffu, o_h[3], 31);
            const float gLl = __shfl_sync(0xffffffffu, o_l[3], 31);
            const bool factored = __all_sync(0xffffffffu, dt_ok) && Ah <= 0.0f && gLh + gLl >= kFactorMinLog2;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                o_sc[i] = factored ? ex2_fast(-(o_h[i] + o_l[i])) * dt[i]
                                   : ex2_fast(fminf((gLh - o_h[i]) + (gLl - o_l[i]), 0.0f)) * dt[i];
            }
            // exact form: the split of this lane's 32-row block (lanes 8j .. 8j+7
            // hold block j) from gamma at its first, middle and last rows, when
            // gamma never rises in the chunk and every row has dt > 0 with D / dt
            // bounded (the diagonal's D R_t / dt_t).  This warp runs close to the
            // chunk period, so factored chunks skip it.
            int split_bits = 0;
            if (!factored) {
                const int l0 = lane & ~7;
                const float gfh = __shfl_sync(0xffffffffu, o_h[0], l0), gfl = __shfl_sync(0xffffffffu, o_l[0], l0);
                const float gmh = __shfl_sync(0xffffffffu, o_h[0], l0 + 4), gml = __shfl_sync(0xffffffffu, o_l[0], l0 + 4);
                const float geh = __shfl_sync(0xffffffffu, o_h[3], l0 + 7), gel = __shfl_sync(0xffffffffu, o_l[3], l0 + 7);
                bool lane_ok = Ah <= 0.0f;
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    lane_ok = lane_ok && (4 * lane + i >= rows || (dt[i] > 0.0f && Dabs < dt[i] * 0x1p60f));
                lane_ok = lane_ok && (gfh - gmh) + (gfl - gml) <= kSplitMaxLog2 &&
                          (gmh - geh) + (gml - gel) <= kSplitMaxLog2;
                const bool mono = __all_sync(0xffffffffu, Ah <= 0.0f && dt[0] >= 0.0f && dt[1] >= 0.0f &&
                                                              dt[2] >= 0.0f && dt[3] >= 0.0f);
                const unsigned blk_ok = __ballot_sync(0xffffffffu, lane_ok);
                const bool split = mono && ((blk_ok >> l0) & 0xffu) == 0xffu;
#pragma unroll
                for (int k = 0; k < 4; ++k) split_bits |= (mono && ((blk_ok >> (8 * k)) & 0xffu) == 0xffu) << k;
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    o_vb[i] = split ? ex2_fast((gmh - o_h[i]) + (gml - o_l[i])) * dt[i] : 1.0f;
            }
            // cv[c % kCv] is free once the epilogue of chunk c-kCv is done
            const bool ok = c < kCv || wait_or_abort(s, &s.epidone[c % kCv], ((c / kCv) - 1) & 1, wlim);
            if (!__all_sync(0xffffffffu, ok)) break;
            reinterpret_cast<float4*>(cv.g2h)[lane] = make_float4(o_h[0], o_h[1], o_h[2], o_h[3]);
            reinterpret_cast<float4*>(cv.g2l)[lane] = make_float4(o_l[0], o_l[1], o_l[2], o_l[3]);
            reinterpret_cast<float4*>(cv.dts)[lane] = make_float4(dt[0], dt[1], dt[2], dt[3]);
            reinterpret_cast<float4*>(cv.sc)[lane] = make_float4(o_sc[0], o_sc[1], o_sc[2], o_sc[3]);
            if (!factored)  // (read only by exact chunks)
                reinterpret_cast<float4*>(cv.vb)[lane] = make_float4(o_vb[0], o_vb[1], o_vb[2], o_vb[3]);
            if (lane == 0) {
                cv.decS = ex2_fast(fminf(gLh + gLl, 0.0f));
                cv.factored = factored;
                cv.split = split_bits;
            }
            mbar_arrive(&s.cvready[c % kCv]);
        }
    } else {
        // ===================== compute warps =====================
        const int q = warp & 3;   // TMEM lane quarter: rows / state columns 32q .. 32q+31
        const int j = warp >> 2;  // column group of the quarter
        const int t = 32 * q + lane;  // chunk row (mask, epilogue) / state column n (state)
        const uint32_t lane_off = (uint32_t)(32 * q) << 16;
        const size_t sbase = ((size_t)slot * H + h) * P * N;
        const float Dh = p.D ? p.D[h] : 0.0f;
        bool ok = true;  // false after any failed wait: the thread then only walks the loop
        // conv taps by [tap][channel pair] and bias into shared memory (read by the
        // first conv, after the compute warps' barrier below)
        if (p.conv && tid < P / 2) {
            float w4[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
            for (int e = 0; e < 2; ++e)
                for (int k = 0; k < W; ++k)
                    w4[e][kMaxW - W + k] = p.conv_w[(size_t)(h * P + 2 * tid + e) * W + k];
            for (int k = 0; k < kMaxW; ++k) s.wconv[k][tid] = make_float2(w4[0][k], w4[1][k]);
            s.bconv[tid] = p.conv_b ? make_float2(p.conv_b[h * P + 2 * tid], p.conv_b[h * P + 2 * tid + 1])
                                    : make_float2(0.f, 0.f);
        }

        // -- conv share: rows 4 rq .. 4 rq + 3, channels 4 jq .. 4 jq + 3 --
        const int rq = tid >> 4, jq = tid & 15;
        const __nv_bfloat16* csb =
            cs_in ? static_cast<const __nv_bfloat16*>(cs_in) + (size_t)slot * (W - 1) * Cdim + h * P + 4 * jq
                  : nullptr;
        // the raw rows before chunk 0 (the conv state's x columns; rq == 0 only):
        // later chunks find theirs in the 4-row tile loaded with their own rows
        uint2 halo0[kMaxW - 1];
#pragma unroll
        for (int i = 0; i < kMaxW - 1; ++i) {
            const int gr = i - (kMaxW - 1);
            halo0[i] = make_uint2(0u, 0u);
            if (rq == 0 && csb != nullptr && gr + W - 1 >= 0) halo0[i] = ldg_u2(csb + (size_t)(gr + W - 1) * Cdim);
        }
        // conv(c): x rows and scaled x rows of chunk c (this thread's 4 x 4 share)
        auto conv = [&](int c) {
            const int rows = min(Q, S - c * Q);
            const ChunkVals& cv = s.cv[c % kCv];
            const bool need_x = cv.factored == 0;  // x rows feed G2 in the exact form
            const float4 sc4 = *reinterpret_cast<const float4*>(&cv.sc[4 * rq]);
            const float scs[4] = {sc4.x, sc4.y, sc4.z, sc4.w};
            // raw rows 4rq-3 .. 4rq+3: this chunk's tile, the 4-row tile before it
            // (later chunks) or the conv state (chunk 0)
            uint2 raw[kRaw];
#pragma unroll
            for (int i = 0; i < kRaw; ++i) {
                const int r = 4 * rq - (kMaxW - 1) + i;
                if (r >= 0)
                    raw[i] = at<uint2>(s.XRAW[c & 1], chunk_off(r, jq >> 1) + ((jq & 1) << 3));
                else if (c > 0)
                    raw[i] = at<uint2>(s.XH[c & 1], (uint32_t)((r + 4) * 128 + jq * 8));
                else
                    raw[i] = i < kMaxW - 1 ? halo0[i < kMaxW - 1 ? i : 0] : make_uint2(0u, 0u);
            }
            // out[i] = b + sum_k w[k] u[i+k] over raw rows i .. i+3, tap by tap (only
            // one tap's weights live at a time: registers are scarce with 18 warps)
            float2 acc[4][2];
            {
                const float4 bb = *reinterpret_cast<const float4*>(&s.bconv[2 * jq]);
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    acc[i][0] = make_float2(bb.x, bb.y);
                    acc[i][1] = make_float2(bb.z, bb.w);
                }
            }
            if (p.conv) {
#pragma unroll
                for (int k = 0; k < kMaxW; ++k) {
                    const float4 wk = *reinterpret_cast<const float4*>(&s.wconv[k][2 * jq]);
                    const float2 w0 = make_float2(wk.x, wk.y), w1 = make_float2(wk.z, wk.w);
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        acc[i][0] = __ffma2_rn(w0, unpack2(raw[i + k].x), acc[i][0]);
                        acc[i][1] = __ffma2_rn(w1, unpack2(raw[i + k].y), acc[i][1]);
                    }
                }
            }
            const uint32_t coff = (uint32_t)((jq & 1) << 3);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int r = 4 * rq + i;
                float2 x0, x1;
                if (p.conv) {
                    x0 = silu2(acc[i][0]);
                    x1 = silu2(acc[i][1]);
                } else {
                    x0 = unpack2(raw[kMaxW - 1 + i].x);
                    x1 = unpack2(raw[kMaxW - 1 + i].y);
                }
                if (r >= rows) x0 = x1 = make_float2(0.f, 0.f);
                const float2 sc2 = make_float2(scs[i], scs[i]);
                const uint32_t off = chunk_off(r, jq >> 1) + coff;
                if (need_x) {
                    const float vbi = cv.vb[4 * rq + i];
                    const float2 vb2 = make_float2(vbi, vbi);
                    at<uint2>(s.XR[c & 1], off) = make_uint2(pack2(__fmul2_rn(vb2, x0)), pack2(__fmul2_rn(vb2, x1)));
                }
                at<uint2>(s.XS[c & 1], off) = make_uint2(pack2(__fmul2_rn(sc2, x0)), pack2(__fmul2_rn(sc2, x1)));
            }
        };

        // -- state share: column n = t, p = 16 j .. 16 j + 15 --
        float2 hreg[8];  // h[16j + 2i .. +1][n]
#pragma unroll
        for (int i = 0; i < 8; ++i)
            hreg[i] = h0 ? make_float2(h0[sbase + (size_t)(16 * j + 2 * i) * N + t],
                                       h0[sbase + (size_t)(16 * j + 2 * i + 1) * N + t])
                           : make_float2(0.f, 0.f);
        auto store_h = [&]() {  // bf16 h[n][16j .. 16j+15]: 2 chunks of 16 bytes
            at<uint4>(s.Hs, chunk_off(t, 2 * j)) = pack4x2(&hreg[0]);
            at<uint4>(s.Hs, chunk_off(t, 2 * j + 1)) = pack4x2(&hreg[4]);
        };

        // prologue: h of chunk -1 in the state tile; M's blocks above the
        // diagonal (they stay zero); conv of chunk 0
        store_h();
        fence_proxy_async_smem();
        mbar_arrive(&s.hsready);
        if (j > q) {
            uint32_t zero[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) zero[i] = 0u;
            tmem_st16(tbase + lane_off + kColM + 16 * j, zero);
            tmem_st_wait();
        }
        named_bar_sync(5, kCompute);  // the conv weights
        if (nchunks > 0) {
            ok = wait_or_abort(s, &s.cvready[0], 0, wlim) && wait_or_abort(s, &s.full_x[0], 0, wlim);
            if (ok) conv(0);
            fence_proxy_async_smem();  // XR / XS are read by G4 / G2
            mbar_arrive(&s.xready[0]);
        }

        for (int c = 0; c < nchunks; ++c) {
            const int rows = min(Q, S - c * Q);
            const int kb = c & 1;
            const ChunkVals& cv = s.cv[c % kCv];

            // ---- mask(c): CB -> M in TMEM (this warp's 32-column block) ----
            const bool fac = cv.factored != 0;
            if (ok) ok = wait_or_abort(s, &s.g1, c & 1, wlim);
            if (__all_sync(0xffffffffu, ok)) {
                if (j <= q) {
                    tc_fence_after();
                    // exact form, a split column block: one factor per row, R_t =
                    // exp(gamma_t - gamma_m), m the block's middle row (the column
                    // factor is on the x rows)
                    const bool split = !fac && ((cv.split >> j) & 1);
                    const float dts_t = cv.dts[t];
                    float g2h_t = 0.0f, g2l_t = 0.0f, rt = 1.0f;
                    if (!fac) {  // (factored chunks read neither)
                        g2h_t = cv.g2h[t];
                        g2l_t = cv.g2l[t];
                        if (split)
                            rt = ex2_fast((g2h_t - cv.g2h[32 * j + 16]) + (g2l_t - cv.g2l[32 * j + 16]));
                    }
                    // the skip term on the diagonal, so that M_tt xv_t carries D x_t:
                    // D / dt_t (factored: y = u_t Y, u_t v_t = dt_t), D R_t / dt_t (split:
                    // xv_t = V_t x_t, R_t V_t = dt_t) or D; rows past the end get nothing
                    const float diag = (j == q && t < rows)
                                           ? (fac ? __fdividef(Dh, dts_t) : split ? __fdividef(Dh * rt, dts_t) : Dh)
                                           : 0.0f;
#pragma unroll 1
                    for (int hf = 0; hf < 2; ++hf) {  // 16 columns at a time
                        const int c0 = 32 * j + 16 * hf;
                        float v[16];
                        tmem_ld16(tbase + lane_off + kColCB + c0, v);
                        tmem_ld_wait();
                        if (split) {
#pragma unroll
                            for (int e = 0; e < 16; ++e) v[e] *= rt;
                        } else if (!fac) {
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
                        if (j == q) {  // the diagonal block: keep s <= t, add the skip term
#pragma unroll
                            for (int e = 0; e < 16; ++e)
                                v[e] = (c0 + e < t) ? v[e] : (c0 + e == t ? v[e] + diag : 0.0f);
                        }
                        uint32_t m[8];
#pragma unroll
                        for (int e = 0; e < 8; ++e) m[e] = pack2(make_float2(v[2 * e], v[2 * e + 1]));
                        tmem_st8(tbase + lane_off + kColM + 16 * j + 8 * hf, m);
                    }
                    tmem_st_wait();
                }
            } else {
                ok = false;
            }
            // the last y store of this quarter has read its tile before this
            // arrival: the control thread loads z of chunk c+1 into that buffer
            // only after it
            if (j == 0 && lane == 0 && c > 0) bulk_wait_read_all();
            tc_fence_before();
            mbar_arrive(&s.mready);

            // ---- state(c): h_c = decS h_{c-1} + b dH(c) ----
            if (ok) ok = wait_or_abort(s, &s.g4, c & 1, wlim) && wait_or_abort(s, &s.g3, c & 1, wlim);
            if (__all_sync(0xffffffffu, ok)) {
                tc_fence_after();
                const float2 dS = make_float2(cv.decS, cv.decS);
                const float2 bS = fac ? dS : make_float2(1.0f, 1.0f);
                float v[16];
                tmem_ld16(tbase + kColDH + lane_off + 16 * j, v);
                tmem_ld_wait();
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    hreg[i] = __ffma2_rn(dS, hreg[i], __fmul2_rn(bS, make_float2(v[2 * i], v[2 * i + 1])));
                store_h();
                fence_proxy_async_smem();
            } else {
                ok = false;
            }
            tc_fence_before();
            mbar_arrive(&s.hsready);

            // ---- conv(c+1): XS[(c+1)&1] and XR[(c+1)&1] were read by G4(c-1) and
            // G2(c-1), which this thread saw done in the epilogue of chunk c-1 ----
            if (c + 1 < nchunks) {
                if (ok)
                    ok = wait_or_abort(s, &s.cvready[(c + 1) % kCv], ((c + 1) / kCv) & 1, wlim) &&
                         wait_or_abort(s, &s.full_x[(c + 1) & 1], ((c + 1) >> 1) & 1, wlim);
                if (ok) conv(c + 1);
                fence_proxy_async_smem();  // XR / XS are read by G4 / G2
                mbar_arrive(&s.xready[(c + 1) & 1]);
            }

            // ---- epilogue(c): factored y = u Y; exact y = Y + u Yo; times silu(z).
            // z comes from its TMA tile and y is written over it in place; each
            // quarter's 32 rows leave with one TMA store (rows past the end are not
            // written).  The store of chunk c-2 from this buffer finished reading it
            // before its issuer's mask(c-1) arrival. ----
            // exp(min(gamma_t, 0)) from the chunk's values (ready since the conv
            // of chunk c), before the waits, so its shared-memory read is not held
            // behind them
            const float dec = ex2_fast(fminf(cv.g2h[t] + cv.g2l[t], 0.0f));
            if (ok) ok = wait_or_abort(s, &s.g2, c & 1, wlim);
            if (ok && has_z) ok = wait_or_abort(s, &s.full_z[kb], (c >> 1) & 1, wlim);
            if (__all_sync(0xffffffffu, ok)) {
                tc_fence_after();
                const float2 dd = make_float2(dec, dec);
                float2 ss2 = make_float2(0.0f, 0.0f);  // (kNorm) sum of y^2 over this thread's columns
#pragma unroll 1
                for (int hh = 0; hh < 2; ++hh) {  // 8 columns at a time
                    // z first: its shared-memory read overlaps the TMEM loads (the
                    // TMEM wait below orders every later memory access after it)
                    const uint32_t off = chunk_off(t, 2 * j + hh);  // row t, 8 columns (SW128)
                    uint4 zraw = make_uint4(0u, 0u, 0u, 0u);
                    if (has_z) zraw = at<uint4>(s.Zt[kb], off);
                    float yv[8];
                    tmem_ld8(tbase + kColY + 64 * kb + lane_off + 16 * j + 8 * hh, yv);
                    if (!fac) {
                        float yo[8];
                        tmem_ld8(tbase + kColYo + 64 * kb + lane_off + 16 * j + 8 * hh, yo);
                        tmem_ld_wait();
#pragma unroll
                        for (int k = 0; k < 8; k += 2) {
                            const float2 r = __ffma2_rn(dd, make_float2(yo[k], yo[k + 1]),
                                                        make_float2(yv[k], yv[k + 1]));
                            yv[k] = r.x;
                            yv[k + 1] = r.y;
                        }
                    } else {
                        tmem_ld_wait();
#pragma unroll
                        for (int k = 0; k < 8; k += 2) {
                            const float2 r = __fmul2_rn(dd, make_float2(yv[k], yv[k + 1]));
                            yv[k] = r.x;
                            yv[k + 1] = r.y;
                        }
                    }
                    float2 out[4], zv[4];
                    if (has_z) unpack4x2(zraw, zv);
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        float2 v = make_float2(yv[2 * e], yv[2 * e + 1]);
                        if constexpr (kNorm) ss2 = __ffma2_rn(v, v, ss2);  // the norm's sum of y^2
                        if (has_z) v = __fmul2_rn(v, silu2(zv[e]));
                        out[e] = v;
                    }
                    if (kVarlen && c * Q + 32 * q + 32 > S) {
                        // the sequence ends inside this quarter and the next sequence's
                        // rows follow it: this thread stores its own row, if it has one
                        if (t < rows)
                            *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.y) +
                                                      ((size_t)(row0 + c * Q + t) * H + h) * P +
                                                      16 * j + 8 * hh) = pack4x2(out);
                    } else {
                        at<uint4>(s.Zt[kb], off) = pack4x2(out);
                    }
                }
                if constexpr (kNorm) s.nsum[c & 1][j][t] = ss2.x + ss2.y;
            } else {
                ok = false;
            }
            fence_proxy_async_smem();   // the tile is read by the TMA store
            tc_fence_before();
            mbar_arrive(&s.epidone[c % kCv]);
            named_bar_sync(1 + q, 128);  // the quarter's four warps
            if constexpr (kNorm) {
                // the row's sum over the head's 64 channels, in a fixed order.  The
                // quarter's other warps write this parity's slots again at chunk
                // c + 2, after the quarter's barrier of chunk c + 1, which this
                // warp reaches only after these reads.
                if (j == 0 && ok && t < rows) {
                    const float ns = (s.nsum[c & 1][0][t] + s.nsum[c & 1][1][t]) +
                                     (s.nsum[c & 1][2][t] + s.nsum[c & 1][3][t]);
                    p.norm_ss[((size_t)b * H + h) * S + (size_t)c * Q + t] = ns;
                }
            }
            // a quarter with rows left (packed sequences: a whole quarter of them)
            if (j == 0 && lane == 0 && ok && (kVarlen ? c * Q + 32 * q + 32 <= S : c * Q + 32 * q < S)) {
                tma_store_3d(&map_y, reinterpret_cast<const char*>(s.Zt[kb]) + q * 32 * 128, h * P,
                             trow(c) + 32 * q, tz);
                bulk_commit();
            }
        }
        if (j == 0 && lane == 0) bulk_wait_read_all();  // the last y stores have read their tiles
        if (!ok) {
            set_abort(s);
        } else if (!aborted(s)) {
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                p.hS[sbase + (size_t)(16 * j + 2 * i) * N + t] = hreg[i].x;
                p.hS[sbase + (size_t)(16 * j + 2 * i + 1) * N + t] = hreg[i].y;
            }
        }
        // new conv state: rows S .. S+W-2 of [conv state ; x|B|C], for this head's x
        // columns and, from the first head of a group, the group's B and C columns.
        // Every read of the old state by this CTA (its x columns, chunk 0) and by the
        // B|C conv before it is long done; a thread reads its column's rows before
        // writing, in increasing order, so the state may be updated in place.
        const int hpg = H / G;
        const int ncol = P + (h % hpg == 0 ? 2 * N : 0);
        if (p.conv_state_out != nullptr && W > 1 && tid < ncol) {
            const int col = tid < P ? h * P + tid
                                    : (tid < P + N ? H * P + g * N + (tid - P) : H * P + G * N + g * N + (tid - P - N));
            const __nv_bfloat16* xs = static_cast<const __nv_bfloat16*>(p.xbc);
            const __nv_bfloat16* si = static_cast<const __nv_bfloat16*>(cs_in);
            __nv_bfloat16* so = static_cast<__nv_bfloat16*>(p.conv_state_out);
            const int nh = W - 1;
            const int L = nchunks - 1;  // the last chunk: its raw x tile and the 4 rows before it
            // every row read before any is written (one memory round trip)
            __nv_bfloat16 v[kMaxW - 1];
#pragma unroll
            for (int jj = 0; jj < kMaxW - 1; ++jj) {
                const int r = S + jj;  // row of [conv state ; rows]
                const int rr = r - nh;  // the same row of this call's rows
                v[jj] = __float2bfloat16_rn(0.0f);
                if (jj >= nh) {
                } else if (rr < 0) {
                    if (si) v[jj] = si[((size_t)slot * nh + r) * Cdim + col];
                } else if (tid < P && L >= 0 && (rr >= L * Q || L > 0)) {
                    // this head's x columns: from the raw tiles still in shared memory
                    v[jj] = rr >= L * Q
                                ? at<__nv_bfloat16>(s.XRAW[L & 1], chunk_off(rr - L * Q, tid >> 3) + (uint32_t)(tid & 7) * 2)
                                : at<__nv_bfloat16>(s.XH[L & 1], (uint32_t)((rr - L * Q + 4) * 128 + tid * 2));
                } else {
                    v[jj] = xs[((size_t)row0 + rr) * Cdim + col];
                }
            }
#pragma unroll
            for (int jj = 0; jj < kMaxW - 1; ++jj)
                if (jj < nh) so[((size_t)slot * nh + jj) * Cdim + col] = v[jj];
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

// ---- short calls: several one-chunk units per CTA --------------------------------
//
// A call of at most Q rows per sequence has one chunk per (sequence, head), and
// one CTA per unit spends more on its prologue (barriers, TMEM, the first
// tiles and row values) and its tail than on the chunk.  scan_units_kernel
// keeps one CTA per SM and walks the units blockIdx.x, blockIdx.x + gridDim.x,
// ... through the same chunk pipeline as scan_tc_kernel, each unit in the
// place of a chunk: its tiles, row values, conv taps and conv halo are
// requested while the unit before it is processed.  The state does not carry
// from unit to unit: the state update of unit c writes unit c's final state
// and puts unit c+1's initial state in the state tile (the arrival that G3 and
// G4 of unit c+1 wait for, as for the next chunk of one sequence).  The x
// columns of a unit's new conv state are written from the raw rows its conv
// reads.  Bit for bit the arithmetic of scan_tc_kernel.

constexpr int kUv = 2;  // per-unit value sets in flight

struct __align__(16) UnitVals {
    ChunkVals cv;                                   // the unit's row values
    alignas(16) float2 wconv[kMaxW][P / 2];         // its head's conv taps (front-padded)
    alignas(16) float2 bconv[P / 2];
    alignas(16) __nv_bfloat16 halo[kMaxW - 1][P];   // raw x rows -3 .. -1: its conv state
    float Dh;                                       // its head's D
    int pad[3];
};

struct __align__(1024) UnitSmem {
    __nv_bfloat16 C[2][Q * 64];
    __nv_bfloat16 B[2][Q * 64];
    __nv_bfloat16 XS[2][Q * 64];
    __nv_bfloat16 XR[2][Q * 64];
    __nv_bfloat16 XRAW[2][Q * 64];
    __nv_bfloat16 Hs[N * 64];
    __nv_bfloat16 Zt[2][Q * 64];
    UnitVals uv[kUv];
    uint64_t full_c, full_b, full_z[2], full_x[2];
    uint64_t g1, g3, g4, g2, fin;
    uint64_t xready, mready, hsready;
    uint64_t cvready[kUv], epidone[kUv];
    uint32_t tmem_base;
    int abort;
};

constexpr size_t kUnitSmemBytes = sizeof(UnitSmem) + 1024;
static_assert(offsetof(UnitSmem, B) % 1024 == 0 && offsetof(UnitSmem, XS) % 1024 == 0, "tile");
static_assert(offsetof(UnitSmem, XR) % 1024 == 0 && offsetof(UnitSmem, XRAW) % 1024 == 0, "tile");
static_assert(offsetof(UnitSmem, Hs) % 1024 == 0 && offsetof(UnitSmem, Zt) % 1024 == 0, "tile");
static_assert(sizeof(UnitVals) % 16 == 0 && offsetof(UnitSmem, uv) % 16 == 0, "float4 rows");
static_assert(offsetof(UnitVals, wconv) % 16 == 0 && offsetof(UnitVals, halo) % 16 == 0, "vectors");
static_assert(offsetof(UnitSmem, full_c) % 8 == 0, "mbarriers");
static_assert(kUnitSmemBytes <= 232448, "shared memory per CTA");

__global__ void __launch_bounds__(kThreads, 1)
    scan_units_kernel(const __grid_constant__ CUtensorMap map_bc, const __grid_constant__ CUtensorMap map_z,
                      const __grid_constant__ CUtensorMap map_y, const __grid_constant__ CUtensorMap map_x,
                      const TcScanParams p)
{
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    UnitSmem& s = *reinterpret_cast<UnitSmem*>(smem_raw + ((1024u - (sm100::smem_u32(smem_raw) & 1023u)) & 1023u));
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int H = p.H, G = p.G, W = p.W, S = p.S;  // S <= Q: one chunk per unit
    const int hpg = H / G;
    const int Cdim = H * P + 2 * G * N;
    // this CTA's units: c-th = (sequence, head) number blockIdx.x + c gridDim.x
    const int nu = (p.B * H - (int)blockIdx.x + (int)gridDim.x - 1) / (int)gridDim.x;
    auto unit_b = [&](int c) { return ((int)blockIdx.x + c * (int)gridDim.x) / H; };
    auto unit_h = [&](int c) { return ((int)blockIdx.x + c * (int)gridDim.x) % H; };
    const bool has_z = (p.flags & kHasZ) != 0;
    const uint64_t wlim = p.wait_ns ? p.wait_ns : kWaitNs;

    // the raw x tiles of the first two units before the setup barrier
    int loaded_x = 0;
    auto load_x = [&](int c) {
        const int kx = c & 1;
        mbar_arrive_expect_tx(&s.full_x[kx], Q * 64 * 2);
        tma_load_3d(s.XRAW[kx], &map_x, &s.full_x[kx], unit_h(c) * P, 0, unit_b(c));
        loaded_x = c + 1;
    };
    if (warp == kControlWarp && lane == 0) {
        mbar_init(&s.full_x[0], 1);
        mbar_init(&s.full_x[1], 1);
        fence_mbar_init();
        if (nu > 0) {
            prefetch_tmap(&map_x);
            load_x(0);
            if (nu > 1) load_x(1);
        }
    }
    if (tid == 0) {
        mbar_init(&s.full_c, 1);
        mbar_init(&s.full_z[0], 1);
        mbar_init(&s.full_z[1], 1);
        mbar_init(&s.full_b, 1);
        mbar_init(&s.g1, 1);
        mbar_init(&s.g3, 1);
        mbar_init(&s.g4, 1);
        mbar_init(&s.g2, 1);
        mbar_init(&s.fin, 1);
        mbar_init(&s.xready, kCompute);
        mbar_init(&s.mready, kCompute);
        mbar_init(&s.hsready, kCompute);
        for (int i = 0; i < kUv; ++i) {
            mbar_init(&s.cvready[i], 32);
            mbar_init(&s.epidone[i], kCompute);
        }
        s.abort = 0;
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(&s.tmem_base, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = s.tmem_base;

    if (warp == kControlWarp) {
        // ===================== control: TMA + MMA (one thread) =====================
        // scan_tc_kernel's order, unit c in the place of chunk c
        if (lane == 0 && nu > 0) {
            prefetch_tmap(&map_bc);
            griddep_wait();  // the B|C pre-pass (see scan_tc_kernel)
            int loaded_c = 0, loaded_b = 0, loaded_z = 0;
            auto load_c = [&](int c) {
                const int xC = p.bc_col0 + G * N + (unit_h(c) / hpg) * N;
                mbar_arrive_expect_tx(&s.full_c, 2 * Q * 64 * 2);
                tma_load_3d(s.C[0], &map_bc, &s.full_c, xC, 0, unit_b(c));
                tma_load_3d(s.C[1], &map_bc, &s.full_c, xC + 64, 0, unit_b(c));
                loaded_c = c + 1;
            };
            auto load_b = [&](int c) {
                const int xB = p.bc_col0 + (unit_h(c) / hpg) * N;
                mbar_arrive_expect_tx(&s.full_b, 2 * Q * 64 * 2);
                tma_load_3d(s.B[0], &map_bc, &s.full_b, xB, 0, unit_b(c));
                tma_load_3d(s.B[1], &map_bc, &s.full_b, xB + 64, 0, unit_b(c));
                loaded_b = c + 1;
            };
            auto kmaj = [](int k) { return (uint64_t)(((k >> 2) << 10) + ((k & 3) << 1)); };
            const uint64_t dHs = sdesc_sw128(smem_u32(s.Hs), 8192, 1024);
            const uint64_t dXS0 = sdesc_sw128(smem_u32(s.XS[0]), 8192, 1024);
            const uint64_t dXS1 = sdesc_sw128(smem_u32(s.XS[1]), 8192, 1024);
            const uint64_t dXR0 = sdesc_sw128(smem_u32(s.XR[0]), 8192, 1024);
            const uint64_t dXR1 = sdesc_sw128(smem_u32(s.XR[1]), 8192, 1024);
            const uint64_t dC = sdesc_sw128(smem_u32(s.C), 16, 1024);
            auto g1 = [&]() {
                const uint64_t dB = sdesc_sw128(smem_u32(s.B), 16, 1024);
#pragma unroll
                for (int k = 0; k < 8; ++k)
                    mma_bf16_ss(tbase + kColCB, dC + kmaj(k), dB + kmaj(k), kIdCB, k > 0);
                mma_commit(&s.g1);
            };
            // G3(c): unit c's initial state in the state tile; Y / Yo [c&1] read by
            // the epilogue of unit c-2
            auto g3 = [&](int c) -> bool {
                bool r = wait_or_abort(s, &s.hsready, c & 1, wlim) &&
                         wait_or_abort(s, &s.cvready[c % kUv], (c / kUv) & 1, wlim);
                if (r && c >= 2) r = wait_or_abort(s, &s.epidone[(c - 2) % kUv], ((c - 2) / kUv) & 1, wlim);
                if (!r) return false;
                tc_fence_after();
                const uint32_t dY = (s.uv[c % kUv].cv.factored ? kColY : kColYo) + 64 * (c & 1);
#pragma unroll
                for (int k = 0; k < 8; ++k)
                    mma_bf16_ss(tbase + dY, dC + kmaj(k), dHs + 128 * k, kIdY, k > 0);
                mma_commit(&s.g3);
                return true;
            };
            auto load_z = [&](int c) {
                mbar_arrive_expect_tx(&s.full_z[c & 1], Q * 64 * 2);
                tma_load_3d(s.Zt[c & 1], &map_z, &s.full_z[c & 1], unit_h(c) * P, 0, unit_b(c));
                loaded_z = c + 1;
            };
            if (has_z) {
                prefetch_tmap(&map_z);
                load_z(0);
                if (nu > 1) load_z(1);
            }
            load_c(0);
            load_b(0);
            bool ok = wait_or_abort(s, &s.full_c, 0, wlim) && wait_or_abort(s, &s.full_b, 0, wlim);
            if (ok) {
                tc_fence_after();
                g1();
                ok = g3(0);
            }
            for (int c = 0; c < nu && ok; ++c) {
                const int kb = c & 1;
                ok = wait_or_abort(s, &s.xready, c & 1, wlim) && wait_or_abort(s, &s.hsready, c & 1, wlim);
                if (!ok) break;
                if (c + 2 < nu) load_x(c + 2);
                tc_fence_after();
                {
                    const uint64_t dA = sdesc_sw128(smem_u32(s.B), Q * 128, 1024);
#pragma unroll
                    for (int k = 0; k < 8; ++k)
                        mma_bf16_ss(tbase + kColDH, dA + 128 * k, (kb ? dXS1 : dXS0) + 128 * k, kIdState, k > 0);
                    mma_commit(&s.g4);
                }
                if (c + 1 < nu) {
                    ok = wait_or_abort(s, &s.g4, c & 1, wlim);
                    if (!ok) break;
                    load_c(c + 1);
                    load_b(c + 1);
                }
                ok = wait_or_abort(s, &s.mready, c & 1, wlim);
                if (!ok) break;
                if (has_z && c >= 1 && c + 1 < nu) load_z(c + 1);
                tc_fence_after();
                {
                    const bool fac = s.uv[c % kUv].cv.factored != 0;
                    const uint64_t dB = fac ? (kb ? dXS1 : dXS0) : (kb ? dXR1 : dXR0);
#pragma unroll
                    for (int k = 0; k < 8; ++k)
                        mma_bf16_ts(tbase + kColY + 64 * kb, tbase + kColM + 8 * k, dB + 128 * k, kIdY,
                                    fac || k > 0);
                    mma_commit(&s.g2);
                }
                if (c + 1 < nu) {
                    ok = wait_or_abort(s, &s.full_c, (c + 1) & 1, wlim) &&
                         wait_or_abort(s, &s.full_b, (c + 1) & 1, wlim);
                    if (!ok) break;
                    tc_fence_after();
                    g1();
                    ok = g3(c + 1);
                    if (!ok) break;
                }
            }
            if (!ok) set_abort(s);
            mma_commit(&s.fin);
            const uint64_t t0 = globaltimer_ns();
            while (!mbar_test(&s.fin, 0) && globaltimer_ns() - t0 < kWaitNs) __nanosleep(64);
            if (loaded_c > 0) {
                const int k = loaded_c - 1;
                while (!mbar_test(&s.full_c, k & 1) && globaltimer_ns() - t0 < kWaitNs) __nanosleep(64);
            }
            if (loaded_b > 0) {
                const int k = loaded_b - 1;
                while (!mbar_test(&s.full_b, k & 1) && globaltimer_ns() - t0 < kWaitNs) __nanosleep(64);
            }
            for (int k = max(0, loaded_x - 2); k < loaded_x; ++k)
                while (!mbar_test(&s.full_x[k & 1], (k >> 1) & 1) && globaltimer_ns() - t0 < kWaitNs)
                    __nanosleep(64);
            for (int k = max(0, loaded_z - 2); k < loaded_z; ++k)
                while (!mbar_test(&s.full_z[k & 1], (k >> 1) & 1) && globaltimer_ns() - t0 < kWaitNs)
                    __nanosleep(64);
        } else if (lane == 0) {
            griddep_wait();
        }
    } else if (warp == kGammaWarp) {
        // ===================== gamma: per-unit values (one warp) =====================
        // scan_tc_kernel's per-chunk values, and the unit's head scalars, conv
        // taps (lane = channel pair) and conv halo; up to kUv units ahead
        const bool softplus = (p.flags & kDtSoftplus) != 0;
        const __nv_bfloat16* cs = static_cast<const __nv_bfloat16*>(p.conv_state_in);
        for (int c = 0; c < nu; ++c) {
            const int b = unit_b(c), h = unit_h(c);
            const float Ah = p.A[h];
            const float bias = p.dt_bias ? p.dt_bias[h] : 0.0f;
            const float Dh = p.D ? p.D[h] : 0.0f;
            const float Dabs = fabsf(Dh);
            float dtn[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int r = 4 * lane + i;
                dtn[i] = r < S ? p.dt[((size_t)b * S + r) * H + h] : 0.0f;
            }
            // taps front-padded to kMaxW (slot k holds tap k - (kMaxW - W)), indexed
            // statically so that they stay in registers
            float w4[2][kMaxW], b2[2];
#pragma unroll
            for (int e = 0; e < 2; ++e) {
#pragma unroll
                for (int k = 0; k < kMaxW; ++k) {
                    const int kk = k - (kMaxW - W);
                    w4[e][k] = p.conv && kk >= 0 ? p.conv_w[(size_t)(h * P + 2 * lane + e) * W + kk] : 0.0f;
                }
                b2[e] = p.conv && p.conv_b ? p.conv_b[h * P + 2 * lane + e] : 0.0f;
            }
            uint32_t hal[kMaxW - 1];  // two channels of each halo row
#pragma unroll
            for (int i = 0; i < kMaxW - 1; ++i) {
                const int sr = i - (kMaxW - 1) + W - 1;  // row of the conv state
                hal[i] = (cs != nullptr && sr >= 0)
                             ? *reinterpret_cast<const uint32_t*>(cs + ((size_t)b * (W - 1) + sr) * Cdim + h * P + 2 * lane)
                             : 0u;
            }
            const int rows = S;
            float dt[4];
            bool dt_ok = true;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float d = softplus ? softplus_f32(dtn[i] + bias) : dtn[i];
                const bool valid = 4 * lane + i < rows;
                dt[i] = valid ? d : 0.0f;
                dt_ok = dt_ok && (!valid || (dt[i] > 0.0f && Dabs < dt[i] * 1e30f));
            }
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
            float o_h[4], o_l[4], o_sc[4], o_vb[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) df_to_log2(gh[i], gl[i], o_h[i], o_l[i]);
            const float gLh = __shfl_sync(0xffffffffu, o_h[3], 31);
            const float gLl = __shfl_sync(0xffffffffu, o_l[3], 31);
            const bool factored = __all_sync(0xffffffffu, dt_ok) && Ah <= 0.0f && gLh + gLl >= kFactorMinLog2;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                o_sc[i] = factored ? ex2_fast(-(o_h[i] + o_l[i])) * dt[i]
                                   : ex2_fast(fminf((gLh - o_h[i]) + (gLl - o_l[i]), 0.0f)) * dt[i];
            }
            int split_bits = 0;
            if (!factored) {
                const int l0 = lane & ~7;
                const float gfh = __shfl_sync(0xffffffffu, o_h[0], l0), gfl = __shfl_sync(0xffffffffu, o_l[0], l0);
                const float gmh = __shfl_sync(0xffffffffu, o_h[0], l0 + 4), gml = __shfl_sync(0xffffffffu, o_l[0], l0 + 4);
                const float geh = __shfl_sync(0xffffffffu, o_h[3], l0 + 7), gel = __shfl_sync(0xffffffffu, o_l[3], l0 + 7);
                bool lane_ok = Ah <= 0.0f;
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    lane_ok = lane_ok && (4 * lane + i >= rows || (dt[i] > 0.0f && Dabs < dt[i] * 0x1p60f));
                lane_ok = lane_ok && (gfh - gmh) + (gfl - gml) <= kSplitMaxLog2 &&
                          (gmh - geh) + (gml - gel) <= kSplitMaxLog2;
                const bool mono = __all_sync(0xffffffffu, Ah <= 0.0f && dt[0] >= 0.0f && dt[1] >= 0.0f &&
                                                              dt[2] >= 0.0f && dt[3] >= 0.0f);
                const unsigned blk_ok = __ballot_sync(0xffffffffu, lane_ok);
                const bool split = mono && ((blk_ok >> l0) & 0xffu) == 0xffu;
#pragma unroll
                for (int k = 0; k < 4; ++k) split_bits |= (mono && ((blk_ok >> (8 * k)) & 0xffu) == 0xffu) << k;
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    o_vb[i] = split ? ex2_fast((gmh - o_h[i]) + (gml - o_l[i])) * dt[i] : 1.0f;
            }
            // the slot is free once the epilogue of unit c-kUv is done
            const bool ok = c < kUv || wait_or_abort(s, &s.epidone[c % kUv], ((c / kUv) - 1) & 1, wlim);
            if (!__all_sync(0xffffffffu, ok)) break;
            UnitVals& uv = s.uv[c % kUv];
            ChunkVals& cv = uv.cv;
            reinterpret_cast<float4*>(cv.g2h)[lane] = make_float4(o_h[0], o_h[1], o_h[2], o_h[3]);
            reinterpret_cast<float4*>(cv.g2l)[lane] = make_float4(o_l[0], o_l[1], o_l[2], o_l[3]);
            reinterpret_cast<float4*>(cv.dts)[lane] = make_float4(dt[0], dt[1], dt[2], dt[3]);
            reinterpret_cast<float4*>(cv.sc)[lane] = make_float4(o_sc[0], o_sc[1], o_sc[2], o_sc[3]);
            if (!factored)
                reinterpret_cast<float4*>(cv.vb)[lane] = make_float4(o_vb[0], o_vb[1], o_vb[2], o_vb[3]);
#pragma unroll
            for (int k = 0; k < kMaxW; ++k) uv.wconv[k][lane] = make_float2(w4[0][k], w4[1][k]);
            uv.bconv[lane] = make_float2(b2[0], b2[1]);
#pragma unroll
            for (int i = 0; i < kMaxW - 1; ++i) *reinterpret_cast<uint32_t*>(&uv.halo[i][2 * lane]) = hal[i];
            if (lane == 0) {
                cv.decS = ex2_fast(fminf(gLh + gLl, 0.0f));
                cv.factored = factored;
                cv.split = split_bits;
                uv.Dh = Dh;
            }
            mbar_arrive(&s.cvready[c % kUv]);
        }
    } else {
        // ===================== compute warps =====================
        const int q = warp & 3;
        const int j = warp >> 2;
        const int t = 32 * q + lane;
        const uint32_t lane_off = (uint32_t)(32 * q) << 16;
        bool ok = true;
        const int rq = tid >> 4, jq = tid & 15;
        auto state_base = [&](int c) { return ((size_t)unit_b(c) * H + unit_h(c)) * P * N; };
        // conv(c): unit c's x rows and scaled x rows (this thread's 4 x 4 share);
        // the thread holding rows S-3 .. S-1 also writes them as the x columns
        // of the unit's new conv state
        auto conv = [&](int c) {
            const int rows = S;
            const UnitVals& uv = s.uv[c % kUv];
            const ChunkVals& cv = uv.cv;
            const bool need_x = cv.factored == 0;
            const float4 sc4 = *reinterpret_cast<const float4*>(&cv.sc[4 * rq]);
            const float scs[4] = {sc4.x, sc4.y, sc4.z, sc4.w};
            uint2 raw[kRaw];
#pragma unroll
            for (int i = 0; i < kRaw; ++i) {
                const int r = 4 * rq - (kMaxW - 1) + i;
                if (r >= 0)
                    raw[i] = at<uint2>(s.XRAW[c & 1], chunk_off(r, jq >> 1) + ((jq & 1) << 3));
                else
                    raw[i] = *reinterpret_cast<const uint2*>(&uv.halo[i < kMaxW - 1 ? i : 0][4 * jq]);
            }
            if (p.conv_state_out != nullptr && W > 1 && rq == (S - 1) >> 2) {
                __nv_bfloat16* so = static_cast<__nv_bfloat16*>(p.conv_state_out) +
                                    (size_t)unit_b(c) * (W - 1) * Cdim + unit_h(c) * P + 4 * jq;
#pragma unroll
                for (int i = 0; i < kRaw; ++i) {
                    const int jj = 4 * rq - (kMaxW - 1) + i - (S - (W - 1));  // row of the new state
                    if (jj >= 0 && jj < W - 1) *reinterpret_cast<uint2*>(so + (size_t)jj * Cdim) = raw[i];
                }
            }
            float2 acc[4][2];
            {
                const float4 bb = *reinterpret_cast<const float4*>(&uv.bconv[2 * jq]);
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    acc[i][0] = make_float2(bb.x, bb.y);
                    acc[i][1] = make_float2(bb.z, bb.w);
                }
            }
            if (p.conv) {
#pragma unroll
                for (int k = 0; k < kMaxW; ++k) {
                    const float4 wk = *reinterpret_cast<const float4*>(&uv.wconv[k][2 * jq]);
                    const float2 w0 = make_float2(wk.x, wk.y), w1 = make_float2(wk.z, wk.w);
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        acc[i][0] = __ffma2_rn(w0, unpack2(raw[i + k].x), acc[i][0]);
                        acc[i][1] = __ffma2_rn(w1, unpack2(raw[i + k].y), acc[i][1]);
                    }
                }
            }
            const uint32_t coff = (uint32_t)((jq & 1) << 3);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int r = 4 * rq + i;
                float2 x0, x1;
                if (p.conv) {
                    x0 = silu2(acc[i][0]);
                    x1 = silu2(acc[i][1]);
                } else {
                    x0 = unpack2(raw[kMaxW - 1 + i].x);
                    x1 = unpack2(raw[kMaxW - 1 + i].y);
                }
                if (r >= rows) x0 = x1 = make_float2(0.f, 0.f);
                const float2 sc2 = make_float2(scs[i], scs[i]);
                const uint32_t off = chunk_off(r, jq >> 1) + coff;
                if (need_x) {
                    const float vbi = cv.vb[4 * rq + i];
                    const float2 vb2 = make_float2(vbi, vbi);
                    at<uint2>(s.XR[c & 1], off) = make_uint2(pack2(__fmul2_rn(vb2, x0)), pack2(__fmul2_rn(vb2, x1)));
                }
                at<uint2>(s.XS[c & 1], off) = make_uint2(pack2(__fmul2_rn(sc2, x0)), pack2(__fmul2_rn(sc2, x1)));
            }
        };

        // -- state share: column n = t, p = 16 j .. 16 j + 15 --
        float2 hreg[8];
        auto load_h = [&](int c) {  // unit c's initial state (zeros without one)
            const size_t sb = state_base(c);
#pragma unroll
            for (int i = 0; i < 8; ++i)
                hreg[i] = p.h0 ? make_float2(p.h0[sb + (size_t)(16 * j + 2 * i) * N + t],
                                             p.h0[sb + (size_t)(16 * j + 2 * i + 1) * N + t])
                               : make_float2(0.f, 0.f);
        };
        auto store_h = [&]() {
            at<uint4>(s.Hs, chunk_off(t, 2 * j)) = pack4x2(&hreg[0]);
            at<uint4>(s.Hs, chunk_off(t, 2 * j + 1)) = pack4x2(&hreg[4]);
        };

        if (nu > 0) load_h(0);
        store_h();
        fence_proxy_async_smem();
        mbar_arrive(&s.hsready);
        if (j > q) {
            uint32_t zero[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) zero[i] = 0u;
            tmem_st16(tbase + lane_off + kColM + 16 * j, zero);
            tmem_st_wait();
        }
        if (nu > 0) {
            ok = wait_or_abort(s, &s.cvready[0], 0, wlim) && wait_or_abort(s, &s.full_x[0], 0, wlim);
            if (ok) conv(0);
            fence_proxy_async_smem();
            mbar_arrive(&s.xready);
        }

        for (int c = 0; c < nu; ++c) {
            const int rows = S;
            const int kb = c & 1;
            const UnitVals& uv = s.uv[c % kUv];
            const ChunkVals& cv = uv.cv;
            const float Dh = uv.Dh;

            // ---- mask(c) ----
            const bool fac = cv.factored != 0;
            if (ok) ok = wait_or_abort(s, &s.g1, c & 1, wlim);
            if (__all_sync(0xffffffffu, ok)) {
                if (j <= q) {
                    tc_fence_after();
                    const bool split = !fac && ((cv.split >> j) & 1);
                    const float dts_t = cv.dts[t];
                    float g2h_t = 0.0f, g2l_t = 0.0f, rt = 1.0f;
                    if (!fac) {
                        g2h_t = cv.g2h[t];
                        g2l_t = cv.g2l[t];
                        if (split)
                            rt = ex2_fast((g2h_t - cv.g2h[32 * j + 16]) + (g2l_t - cv.g2l[32 * j + 16]));
                    }
                    const float diag = (j == q && t < rows)
                                           ? (fac ? __fdividef(Dh, dts_t) : split ? __fdividef(Dh * rt, dts_t) : Dh)
                                           : 0.0f;
#pragma unroll 1
                    for (int hf = 0; hf < 2; ++hf) {
                        const int c0 = 32 * j + 16 * hf;
                        float v[16];
                        tmem_ld16(tbase + lane_off + kColCB + c0, v);
                        tmem_ld_wait();
                        if (split) {
#pragma unroll
                            for (int e = 0; e < 16; ++e) v[e] *= rt;
                        } else if (!fac) {
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
                        if (j == q) {
#pragma unroll
                            for (int e = 0; e < 16; ++e)
                                v[e] = (c0 + e < t) ? v[e] : (c0 + e == t ? v[e] + diag : 0.0f);
                        }
                        uint32_t m[8];
#pragma unroll
                        for (int e = 0; e < 8; ++e) m[e] = pack2(make_float2(v[2 * e], v[2 * e + 1]));
                        tmem_st8(tbase + lane_off + kColM + 16 * j + 8 * hf, m);
                    }
                    tmem_st_wait();
                }
            } else {
                ok = false;
            }
            if (j == 0 && lane == 0 && c > 0) bulk_wait_read_all();
            tc_fence_before();
            mbar_arrive(&s.mready);

            // ---- state(c): unit c's final state h = decS h0 + b dH to memory; unit
            // c+1's initial state into the registers and the state tile ----
            if (ok) ok = wait_or_abort(s, &s.g4, c & 1, wlim) && wait_or_abort(s, &s.g3, c & 1, wlim);
            if (__all_sync(0xffffffffu, ok)) {
                tc_fence_after();
                const float2 dS = make_float2(cv.decS, cv.decS);
                const float2 bS = fac ? dS : make_float2(1.0f, 1.0f);
                float v[16];
                tmem_ld16(tbase + kColDH + lane_off + 16 * j, v);
                tmem_ld_wait();
                const size_t sb = state_base(c);
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const float2 hf = __ffma2_rn(dS, hreg[i], __fmul2_rn(bS, make_float2(v[2 * i], v[2 * i + 1])));
                    p.hS[sb + (size_t)(16 * j + 2 * i) * N + t] = hf.x;
                    p.hS[sb + (size_t)(16 * j + 2 * i + 1) * N + t] = hf.y;
                }
                if (c + 1 < nu) {
                    load_h(c + 1);
                    store_h();
                }
                fence_proxy_async_smem();
            } else {
                ok = false;
            }
            tc_fence_before();
            mbar_arrive(&s.hsready);

            // ---- conv(c+1) ----
            if (c + 1 < nu) {
                if (ok)
                    ok = wait_or_abort(s, &s.cvready[(c + 1) % kUv], ((c + 1) / kUv) & 1, wlim) &&
                         wait_or_abort(s, &s.full_x[(c + 1) & 1], ((c + 1) >> 1) & 1, wlim);
                if (ok) conv(c + 1);
                fence_proxy_async_smem();
                mbar_arrive(&s.xready);
            }

            // ---- epilogue(c) ----
            if (ok) ok = wait_or_abort(s, &s.g2, c & 1, wlim);
            if (ok && has_z) ok = wait_or_abort(s, &s.full_z[kb], (c >> 1) & 1, wlim);
            if (__all_sync(0xffffffffu, ok)) {
                tc_fence_after();
                const float dec = ex2_fast(fminf(cv.g2h[t] + cv.g2l[t], 0.0f));
                const float2 dd = make_float2(dec, dec);
#pragma unroll 1
                for (int hh = 0; hh < 2; ++hh) {
                    const uint32_t off = chunk_off(t, 2 * j + hh);  // z first, as in scan_tc_kernel
                    uint4 zraw = make_uint4(0u, 0u, 0u, 0u);
                    if (has_z) zraw = at<uint4>(s.Zt[kb], off);
                    float yv[8];
                    tmem_ld8(tbase + kColY + 64 * kb + lane_off + 16 * j + 8 * hh, yv);
                    if (!fac) {
                        float yo[8];
                        tmem_ld8(tbase + kColYo + 64 * kb + lane_off + 16 * j + 8 * hh, yo);
                        tmem_ld_wait();
#pragma unroll
                        for (int k = 0; k < 8; k += 2) {
                            const float2 r = __ffma2_rn(dd, make_float2(yo[k], yo[k + 1]),
                                                        make_float2(yv[k], yv[k + 1]));
                            yv[k] = r.x;
                            yv[k + 1] = r.y;
                        }
                    } else {
                        tmem_ld_wait();
#pragma unroll
                        for (int k = 0; k < 8; k += 2) {
                            const float2 r = __fmul2_rn(dd, make_float2(yv[k], yv[k + 1]));
                            yv[k] = r.x;
                            yv[k + 1] = r.y;
                        }
                    }
                    float2 out[4], zv[4];
                    if (has_z) unpack4x2(zraw, zv);
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        float2 v = make_float2(yv[2 * e], yv[2 * e + 1]);
                        if (has_z) v = __fmul2_rn(v, silu2(zv[e]));
                        out[e] = v;
                    }
                    at<uint4>(s.Zt[kb], off) = pack4x2(out);
                }
            } else {
                ok = false;
            }
            fence_proxy_async_smem();
            tc_fence_before();
            mbar_arrive(&s.epidone[c % kUv]);
            named_bar_sync(1 + q, 128);
            if (j == 0 && lane == 0 && ok && 32 * q < S) {
                tma_store_3d(&map_y, reinterpret_cast<const char*>(s.Zt[kb]) + q * 32 * 128, unit_h(c) * P,
                             32 * q, unit_b(c));
                bulk_commit();
            }
            // the B|C columns of the new conv state, from the first head of a group
            // (read from memory: these rows are not in shared memory)
            if (p.conv_state_out != nullptr && W > 1 && unit_h(c) % hpg == 0 && tid < 2 * N) {
                const int b = unit_b(c), g = unit_h(c) / hpg;
                const int col = tid < N ? H * P + g * N + tid : H * P + G * N + g * N + (tid - N);
                const __nv_bfloat16* xs = static_cast<const __nv_bfloat16*>(p.xbc);
                const __nv_bfloat16* si = static_cast<const __nv_bfloat16*>(p.conv_state_in);
                __nv_bfloat16* so = static_cast<__nv_bfloat16*>(p.conv_state_out);
                const int nh = W - 1;
                // every row read before any is written (one memory round trip; the
                // state may be updated in place)
                __nv_bfloat16 v[kMaxW - 1];
#pragma unroll
                for (int jj = 0; jj < kMaxW - 1; ++jj) {
                    const int r = S + jj;
                    v[jj] = __float2bfloat16_rn(0.0f);
                    if (jj < nh) {
                        if (r >= nh) v[jj] = xs[((size_t)b * S + (r - nh)) * Cdim + col];
                        else if (si) v[jj] = si[((size_t)b * nh + r) * Cdim + col];
                    }
                }
#pragma unroll
                for (int jj = 0; jj < kMaxW - 1; ++jj)
                    if (jj < nh) so[((size_t)b * nh + jj) * Cdim + col] = v[jj];
            }
        }
        if (j == 0 && lane == 0) bulk_wait_read_all();
        if (!ok) set_abort(s);
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

// 3-D map over rows of `cols` bf16: dims {cols, S, B}, box {64, box_rows, 1}, SW128
// (or unswizzled).
bool make_map(CUtensorMap* m, const void* base, int cols, int S, int B, int box_rows = Q,
              bool swizzle = true)
{
    cuuint64_t dims[3] = {(cuuint64_t)cols, (cuuint64_t)S, (cuuint64_t)B};
    cuuint64_t strides[2] = {(cuuint64_t)cols * 2, (cuuint64_t)cols * 2 * (cuuint64_t)S};
    cuuint32_t box[3] = {64, (cuuint32_t)box_rows, 1};
    cuuint32_t es[3] = {1, 1, 1};
    return g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides,
                    box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    swizzle ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool scan_tc_supports(int P_, int N_) { return P_ == P && N_ == N; }

bool scan_units_supports(const TcScanParams& p)
{
    return p.cu_seqlens == nullptr && p.norm_ss == nullptr && p.S >= 1 && p.S <= Q && p.W <= kMaxW;
}

cudaError_t launch_scan_units(const TcScanParams& p, cudaStream_t st, bool after_prepass)
{
    if (p.B == 0) return cudaSuccess;
    if (!scan_units_supports(p) || !encode_fn()) return cudaErrorNotSupported;
    const int Cdim = p.H * P + 2 * p.G * N;
    CUtensorMap mbc, mz, my, mx;
    if (!make_map(&mbc, p.bc, p.bc_stride, p.S, p.B) || !make_map(&my, p.y, p.H * P, p.S, p.B, 32) ||
        !make_map(&mx, p.xbc, Cdim, p.S, p.B))
        return cudaErrorInvalidValue;
    memset(&mz, 0, sizeof(mz));
    if ((p.flags & kHasZ) && !make_map(&mz, p.z, p.H * P, p.S, p.B)) return cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(scan_units_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)kUnitSmemBytes);
    if (e != cudaSuccess) return e;
    int dev = 0, nsm = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    const long long units = (long long)p.B * p.H;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(units < nsm ? units : nsm));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kUnitSmemBytes;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = after_prepass ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, scan_units_kernel, mbc, mz, my, mx, p);
}

cudaError_t launch_scan_tc(const TcScanParams& p, cudaStream_t st, bool after_prepass)
{
    const bool varlen = p.cu_seqlens != nullptr;
    // packed sequences still run with no rows at all: fresh ones get zero states
    if (p.B == 0 || (p.S == 0 && !varlen)) return cudaSuccess;
    if (p.W > kMaxW || !encode_fn()) return cudaErrorNotSupported;
    // row arrays as [cols, rows, batch]: packed sequences are one batch of all
    // rows; with no rows, any 16-byte aligned array stands in (no tile is read)
    const int mS = p.S > 0 ? p.S : 1, mB = varlen ? 1 : p.B;
    const void* stand_in = p.h0;
    CUtensorMap mbc, mz, my, mx, mxh;
    if (!make_map(&mbc, p.S > 0 ? p.bc : stand_in, p.bc_stride, mS, mB)) return cudaErrorInvalidValue;
    // raw x rows of a head (128-row tiles) and the 4 rows before a tile, [B, S, Cdim]
    const int Cdim = p.H * P + 2 * p.G * N;
    if (!make_map(&mx, p.S > 0 ? p.xbc : stand_in, Cdim, mS, mB) ||
        !make_map(&mxh, p.S > 0 ? p.xbc : stand_in, Cdim, mS, mB, 4, false))
        return cudaErrorInvalidValue;
    // z tiles in (128 rows), y leaves in 32-row quarters; both [B, S, H*P]
    memset(&mz, 0, sizeof(mz));
    if ((p.flags & kHasZ) && !make_map(&mz, p.S > 0 ? p.z : stand_in, p.H * P, mS, mB))
        return cudaErrorInvalidValue;
    if (!make_map(&my, p.S > 0 ? p.y : stand_in, p.H * P, mS, mB, 32)) return cudaErrorInvalidValue;
    if (p.norm_ss != nullptr && (varlen || !(p.flags & kHasZ))) return cudaErrorInvalidValue;
    auto kernel = varlen ? scan_tc_kernel<true, false>
                         : (p.norm_ss ? scan_tc_kernel<false, true> : scan_tc_kernel<false, false>);
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)kSmemBytes);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(p.H, p.B);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = after_prepass ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kernel, mbc, mz, my, mx, mxh, p);
}

}  // namespace ssd
