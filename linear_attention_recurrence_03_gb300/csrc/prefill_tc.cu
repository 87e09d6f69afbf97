// prefill_tc.cu -- chunked GDN prefill on the tcgen05 tensor cores: bf16 operands, fp32
// accumulation in tensor memory (TMEM), fp32 state master in registers.
//
// "GDN CTE Kernel API Reference": the gated delta rule in chunk-parallel form with an
// intra-chunk (I+A) inverse; q/k/v token-major, out head-major, state fp32 (Notes: the
// state is fp32 whatever the compute dtype). Specialisation: Dk = Dv = 128, bf16.
//
// Chunk algebra (derived from S_t = exp(g_t)(I - beta_t k_t k_t^T) S_{t-1} + beta_t k_t v_t^T,
// o_t = scale S_t^T q_t), chunk of C = 64 tokens, local index r, starting state S0:
//   gamma_r = sum_{i<=r} g_i, Gamma_r = exp(gamma_r), D[r,j] = exp(gamma_r - gamma_j) (j <= r)
//   A[r,j] = beta_r (k_r.k_j) D[r,j] (j < r)        T = (I + A)^-1
//   P[r,j] = (q_r.k_j) D[r,j]        (j <= r)
//   T_W = T diag(beta Gamma),  T_U = T diag(beta)
//   W = T_W K,  U~ = T_U V,  U = U~ - W S0,  U' = diag(exp(gamma_last - gamma)) U
//   O  = scale (diag(Gamma) (Q S0) + P U)
//   S1 = Gamma_last S0 + K^T U'
// D is formed without ratios of Gamma (which underflow): inside a 16-token block by
// exp(gamma_r - gamma_j), across blocks as exp(gamma_r - gamma_end) exp(gamma_end - gamma_j),
// both factors <= 1.
//
// Two kernels. Everything that does not depend on S0 (the Gram matrices, the decay
// masks, the (I+A)^-1 solve, T_U, P and W) is independent across chunks, so it runs
// first as a fully parallel grid ("prep", one CTA per (batch, value head, chunk)) that
// writes bf16 operand tiles (T_U, P, W, and for the two-slice carry K~ = diag(exp(
// gamma_last - gamma)) K) and the decay scalars per chunk to a workspace, the tiles
// already in the 128-byte swizzled layout the tensor cores read. The sequential part
// ("carry") then streams q, v and those tiles through a two-stage ring and keeps only the
// S0-dependent chain per chunk, in one of two forms:
//   carry_tc_kernel<64>: one CTA per (batch, value head, 64-column slice of the state;
//   the slices never communicate), state rows in TMEM lanes, used while two CTAs per
//   head fit the GPU (the Gamma scaling of the Q S0 rows is applied in its output step):
//          [T_U;-] V              -> U~                   (M128 N64  K64)
//          [W;Q] S0               -> W S0, Q S0           (M128 N64  K128)
//          [K~_1;P] U             -> P U                  (M128 N64  K64)
//          K~^T U                 -> state increment      (M128 N64  K64)
//   carry_t_kernel: one CTA per (batch, value head), the chain transposed (state columns
//   in TMEM lanes) so that U^T and S0^T enter the MMAs from TMEM; it loads q and k itself
//   and applies their row decays in its SIMT steps (U' = diag(exp(gamma_last - gamma)) U):
//          V^T T_U^T              -> U~^T                 (M128 N64  K64)
//          S0^T [W;Q]^T           -> (W S0)^T, (Q S0)^T   (M128 N128 K128, A in TMEM)
//          U'^T K                 -> dS^T                 (M128 N128 K64, A in TMEM)
//          U^T P^T                -> (P U)^T              (M128 N64  K64, A in TMEM)
//   prep   [Q;K] K^T              -> QK^T, KK^T           (M128 N64  K128)
//          [T_W;P] K              -> W                    (M128 N128 K64)
// Stacking two 64-row operands into one 128-row operand fills the M = 128 data path;
// the half of a result that is not needed is ignored.
//
// Every wait is bounded; on a timeout a kernel records a status bit, unwinds, waits for
// its own copies and MMAs, frees TMEM and returns.
#include <cudaTypedefs.h>

#include <algorithm>
#include <mutex>

#include "internal.h"
#include "sm100_ptx.cuh"

namespace gdn {

// Status bits set by kernels of this file when a bounded wait runs out.
__device__ uint32_t g_tc_status = 0;

uint32_t prefill_tc_take_status() {
    uint32_t bits = 0;
    if (cudaMemcpyFromSymbol(&bits, g_tc_status, sizeof(bits)) != cudaSuccess) return 0;
    if (bits != 0) {
        const uint32_t zero = 0;
        cudaMemcpyToSymbol(g_tc_status, &zero, sizeof(zero));
    }
    return bits;
}

#ifdef GDN_TRACE
// Profiling aid, compiled only with -DGDN_TRACE: per-chunk SM clock stamps of the
// pipeline events of carry CTA (0,0,0) and of the prep CTAs of head 0, batch 0, read
// back with gdn_trace_read().
constexpr int kTraceChunks = 64, kTraceEvents = 64;
__device__ unsigned long long g_trace[kTraceChunks][kTraceEvents];
#define TRACE(c, ev)                                                                    \
    do {                                                                                \
        if (blockIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0 && (c) < kTraceChunks) \
            g_trace[(c)][(ev)] = clock64();                                             \
    } while (0)
#define TRACE_PREP(ev)                                                        \
    do {                                                                      \
        if (blockIdx.y == 0 && blockIdx.z == 0 && blockIdx.x < kTraceChunks) \
            g_trace[blockIdx.x][(ev)] = clock64();                            \
    } while (0)
// a stamp taken into a register now (TCLK) and stored later (TPUT), away from MMA issue
#define TCLK(var) const unsigned long long var = clock64()
#define TPUT(c, ev, var)                                                                \
    do {                                                                                \
        if (blockIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0 && (c) < kTraceChunks) \
            g_trace[(c)][(ev)] = (var);                                                 \
    } while (0)
// Launch spans: per kernel (prep of segment j: slot 2j, its carry: 2j + 1, j < 4) the
// earliest CTA start and the latest CTA end (globaltimer ns), read back with
// gdn_trace_span_read().
__device__ unsigned long long g_span[8][2];
#define SPAN_BEGIN(slot)                                                                \
    do {                                                                                \
        if (threadIdx.x == 0 && (slot) < 8) atomicMin(&g_span[(slot)][0], ptx::globaltimer_ns()); \
    } while (0)
#define SPAN_END(slot)                                                                  \
    do {                                                                                \
        if (threadIdx.x == 0 && (slot) < 8) atomicMax(&g_span[(slot)][1], ptx::globaltimer_ns()); \
    } while (0)
#else
#define SPAN_BEGIN(slot) \
    do {                 \
    } while (0)
#define SPAN_END(slot) \
    do {               \
    } while (0)
#define TCLK(var) \
    do {          \
    } while (0)
#define TPUT(c, ev, var) \
    do {                 \
    } while (0)
#define TRACE(c, ev) \
    do {             \
    } while (0)
#define TRACE_PREP(ev) \
    do {               \
    } while (0)
#endif

namespace {
using namespace ptx;

constexpr int C = 64;    // chunk length
// Limit of every bounded wait. GDN_TEST_STALL (a test-only build, never the library's
// default) shortens it to 5 ms and has the carry kernels' producer skip the loads of the
// second chunk, so that a test can see the waits run out, the kernel unwind and the status
// word report it.
#ifdef GDN_TEST_STALL
constexpr uint64_t kWaitNs = 5000000ull;
#else
constexpr uint64_t kWaitNs = 2000000000ull;
#endif

// Overlapped schedule (the prep of the next segment of the sequence runs beside the carry
// of the current one): at most this many segments, of at least kMinSegmentChunks chunks.
// The prep of a segment on the SMs the carry leaves (88 of 152 for 64 carry CTAs) runs
// about 1.22x faster per chunk than the carry, so each segment can be that much longer
// than the one before, and the exposed prep of the first one shrinks as segments are
// added (45% of the chunks for two segments, 27% for three, 18% for four).
#ifndef GDN_OVERLAP_SEGMENTS
#define GDN_OVERLAP_SEGMENTS 2
#endif
#ifndef GDN_SEGMENT_GROWTH_PERMILLE
#define GDN_SEGMENT_GROWTH_PERMILLE 1220
#endif
constexpr int kOverlapSegments = GDN_OVERLAP_SEGMENTS;
// (Below two segments of this many chunks the boundary costs more than the prep it hides:
// S = 1024 on 16 heads ran 55 us as two segments of 8 chunks and 40 us as one; S = 2048
// 81 us as two of 16 and 66 us as one; from 64 chunks on two segments win.)
#ifndef GDN_MIN_SEGMENT_CHUNKS
#define GDN_MIN_SEGMENT_CHUNKS 24
#endif
constexpr int kMinSegmentChunks = GDN_MIN_SEGMENT_CHUNKS;
constexpr int kSegmentGrowthPermille = GDN_SEGMENT_GROWTH_PERMILLE;
// 1: a carry segment is launched as a programmatic dependent of the one before it, so its
// setup overlaps that one's last chunks (the state is read after griddepcontrol.wait).
#ifndef GDN_CARRY_PDL
#define GDN_CARRY_PDL 1
#endif
constexpr bool kCarryPdl = GDN_CARRY_PDL != 0;
constexpr int kMaxSegments = 8;
// Carry form while two CTAs per head fit the GPU: 1 = two 64-column state slices per head
// (carry_tc_kernel<64>), 0 = one transposed CTA per head (carry_t_kernel).
#ifndef GDN_CARRY_SPLIT
#define GDN_CARRY_SPLIT 1
#endif
constexpr bool kCarrySplit = GDN_CARRY_SPLIT != 0;

// ---- workspace: per (batch, value head, chunk) unit, bf16 tiles of 64 rows x 64 columns
// in the 128-byte swizzled layout, T_U | P | W[:, 0:64] | W[:, 64:128] | K~[:, 0:64] |
// K~[:, 64:128], then the carry's decay scalars, with K~ = diag(exp(gamma_last - gamma)) K.
// The K~ tiles are written only for the two-slice carry, whose chain reads them (its U
// step then writes one tile); the transposed carry reads k itself and applies the decays
// in its own steps. Both carries read q and apply diag(Gamma) to the rows of Q S0.
constexpr uint32_t WS_TU = 0, WS_P = 8192, WS_W = 16384, WS_KT = 32768, WS_CS = 49152;

struct CarryScalars {
    float kdec[C];  // exp(gamma_last - gamma_r)
    float Gam[C];   // exp(gamma_r)
    float Gl;       // exp(gamma_last)
    float pad[3];
};
constexpr uint32_t WS_UNIT = WS_CS + (uint32_t)sizeof(CarryScalars);
static_assert(sizeof(CarryScalars) % 16 == 0 && WS_UNIT % 16 == 0,
              "scalars and units are whole 16-byte rows");

// ---- prep kernel: shared memory map (offsets from a 1024-byte aligned base), sized
// for three CTAs per SM
//   block b (Dk columns 64b..64b+63): Q_b | K_b (8 KB each), stride 16 KB. Once the Gram
//   MMA has read Q, the Q_b slots hold the fp32 blocks of A (blocks 0-5 | 6-9), and once
//   the W MMA has read K and the solve is done, the bf16 W blocks (W_b in slot Q_b)
//   T_U, T_W, P (adjacent: [T_W; P] is one 128-row operand)
//   fp32 blocks of T, scalars, barriers
constexpr int PREP_THREADS = 288;  // warp 0: producer + MMA issuer; warps 1..8: prep
constexpr uint32_t PQ_STRIDE = 16384;
constexpr uint32_t PQ_Q = 0, PQ_K = 8192;
constexpr uint32_t P_TU = 32768, P_TW = 40960, P_P = 49152;
static_assert(P_P == P_TW + 8192, "[T_W; P] is one 128-row operand");
constexpr int BS = 20;  // row stride (floats) of a 16x16 fp32 block
constexpr uint32_t BLOCK_BYTES = 16 * BS * 4;
static_assert(6 * BLOCK_BYTES <= 8192 && 4 * BLOCK_BYTES <= 8192, "A blocks fit the Q slots");
constexpr uint32_t P_TB = 57344;                      // 10 lower blocks of T
constexpr uint32_t P_SCAL = P_TB + 10 * BLOCK_BYTES;

struct PrepScalars {
    float gam[C];     // gamma_r
    float beta[C];    // beta_r
    float ctab[C];    // exp(gamma_{end of r's 16-block} - gamma_r)
    float Gam[C];     // exp(gamma_r)
    float endgam[4];  // gamma at the end of each 16-block
};
constexpr uint32_t P_CS = P_SCAL + sizeof(PrepScalars);  // CarryScalars staging
constexpr uint32_t P_BAR = P_CS + sizeof(CarryScalars);
constexpr uint32_t P_MISC = P_BAR + 64;
constexpr uint32_t PREP_SMEM = P_MISC + 64 + 1024;  // + alignment slack
static_assert(P_BAR % 8 == 0 && P_CS % 16 == 0, "barrier and copy alignment");
static_assert(3 * (PREP_SMEM + 1024) <= 233472, "three prep CTAs per SM");

// prep TMEM columns (fp32, 128 lanes)
constexpr uint32_t PT_G = 0;  // Gram [QK^T; KK^T], 64 columns
constexpr uint32_t PT_W = 0;  // [W; -], 128 columns (the Gram matrices are read by then)
constexpr uint32_t PT_COLS = 128;

enum { PB_FULL = 0, PB_GRAM, PB_WDONE, PB_DRAIN, PB_COUNT };

// ---- carry kernel: one CTA per (NS-column slice of the state, value head, batch), NS = 64
// (CarryCfg<NS>; the transposed carry shares the stage layout with NS = 128). Shared
// memory map:
//   stage s (two stages, one chunk each), in two copy groups:
//     block b (Dk columns 64b..64b+63): W_b | Q_b | K~_b (8 KB each, stride 24 KB)
//       ([W_b; Q_b] is one 128-row operand), then P ([K~_1; P] one operand),
//     V slice (64 tokens x NS columns, in 64-column blocks), T_U ([T_U; -] one operand)
//     early group (read by U~ and [W; Q] S0, freed as soon as they complete): W, q, V,
//     T_U; late group (read by K~^T U, P U and the state update): K~, P and the scalars
//     (the transposed carry loads k into the K~ slots)
//   two U tiles (64 tokens x NS, by chunk parity), the bf16 state operand (128 x NS,
//   64-column blocks), per-stage scalars, barriers
// warp 0: producer; warp 1 (one thread): MMA issuer; warps 4..11: SIMT; warps 2 and 3
// only take part in the setup and the teardown
constexpr int CARRY_THREADS = 384;
constexpr uint32_t BLK_STRIDE = 24576;
constexpr uint32_t OFF_W = 0, OFF_Q = 8192, OFF_K = 16384;
constexpr uint32_t OFF_P = 49152, OFF_V = 57344;
static_assert(OFF_P == BLK_STRIDE + OFF_K + 8192, "[K~_1; P] is one 128-row operand");

template <int NS>
struct CarryCfg {
    static constexpr int NB = NS / 64;    // 64-column blocks of the slice
    static constexpr int CPT = NS / 2;    // state columns per SIMT thread
    static constexpr uint32_t OFF_TU = OFF_V + 8192u * NB;
    static constexpr uint32_t STAGE = OFF_TU + 8192u;
    static constexpr uint32_t U = 2 * STAGE;              // U tiles, NB blocks of 8 KB each
    static constexpr uint32_t UT = 8192u * NB;            // bytes of one U tile
    static constexpr uint32_t SM_S = U + 2 * UT;          // state operand, NB blocks of 16 KB
    static constexpr uint32_t SCAL = SM_S + 16384u * NB;
    static constexpr uint32_t BAR = SCAL + 2 * sizeof(CarryScalars);
    static constexpr uint32_t MISC = BAR + 128;
    static constexpr uint32_t SMEM = MISC + 64 + 1024;
    // TMEM (fp32 columns), two buffers of each kind by chunk parity:
    //   B[p]: U~ of the chunk (upper half), then, once U is formed, its state increment
    //   A[p]: [W S0; Q S0]
    //   C[p]: [-; P U]
    // The output of token r is scale (Gamma_r (Q S0)_r + (P U)_r).
    static constexpr uint32_t TMB = 0, TMA = 2 * NS, TMC = 4 * NS;
    static constexpr uint32_t TMCOLS = 6 * NS <= 256 ? 256 : 512;
    static_assert(BAR % 8 == 0 && SCAL % 16 == 0, "barrier and copy alignment");
    static_assert(NS != 64 || SMEM <= 232448, "shared memory budget");
};

// FULLE/EMPTYE: the early copy group of stage s; FULLL/EMPTYL: the late group
enum {
    B_FULLE0 = 0, B_FULLE1, B_FULLL0, B_FULLL1, B_EMPTYE0, B_EMPTYE1, B_EMPTYL0, B_EMPTYL1,
    B_ADONE, B_SDONE, B_CDONE, B_DRAIN, B_COUNT
};
static_assert(B_COUNT * 8 <= 128, "carry barrier block");

// status bits
constexpr uint32_t ST_PRODUCER = 1u, ST_MMA = 2u, ST_CARRY = 4u, ST_PREP = 8u;

// One launch pair processes chunks c0 .. c0 + nseg - 1 of every (batch, head); the
// workspace holds nseg units per head, indexed by the chunk's position in the launch.
struct TcArgs {
    const float* g;
    const float* beta;
    float scale;
    int B, Hk, Hv, S;
    int c0, nseg;
    float* state;
    int state_is_input;
    __nv_bfloat16* out;
    uint8_t* ws;
    // variable-length batch (NULL cu: the dense [B, H, S] layout): sequence n holds the
    // packed tokens cu[n] .. cu[n+1] - 1 of the [H, S] tensors and the chunks
    // cb[n] .. cb[n+1] - 1 of the grid, nseg = an upper bound of cb[N] chunks
    const int* cu;
    const int* cb;
    int N;
    // the prep writes K~ to the workspace (for the two-slice carry)
    int export_k;
    // the carry is a programmatic dependent of the prep that wrote its workspace: its
    // producer waits for that grid (griddepcontrol.wait) before the first copy
    int ws_wait;
};

__device__ __forceinline__ size_t ws_offset(int b, int h, int c, int Hv, int nch) {
    return ((size_t)(b * Hv + h) * (size_t)nch + (size_t)c) * WS_UNIT;
}

// Sequence n of a variable-length batch for chunk cl of the grid: cb[n] <= cl < cb[n+1]
// (binary search over the N + 1 chunk bases).
__device__ __forceinline__ int seq_of_chunk(const int* cb, int N, int cl) {
    int lo = 0, hi = N;  // invariant: cb[lo] <= cl < cb[hi]
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (cb[mid] <= cl) lo = mid; else hi = mid;
    }
    return lo;
}

__device__ __forceinline__ void bar_sync(uint32_t id, uint32_t n) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}

// Arrives at a named barrier without waiting for it to complete.
__device__ __forceinline__ void bar_arrive(uint32_t id, uint32_t n) {
    asm volatile("bar.arrive %0, %1;" ::"r"(id), "r"(n) : "memory");
}

// Named barrier that also ORs a predicate over the participating threads, so that a
// group decides to stop as one (every thread sees the same result).
__device__ __forceinline__ bool bar_any(uint32_t id, uint32_t n, bool v) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 q, %3, 0;\n\t"
        "bar.red.or.pred p, %1, %2, q;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(r)
        : "r"(id), "r"(n), "r"((uint32_t)v)
        : "memory");
    return r != 0;
}

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
    __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
                 "r"(d)
                 : "memory");
}

__device__ __forceinline__ void st_shared_b32(uint32_t addr, uint32_t v) {
    asm volatile("st.shared.b32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}

__device__ __forceinline__ void st_shared_b16(uint32_t addr, float x) {
    const __nv_bfloat16 h = __float2bfloat16_rn(x);
    asm volatile("st.shared.b16 [%0], %1;" ::"r"(addr),
                 "h"(*reinterpret_cast<const unsigned short*>(&h))
                 : "memory");
}

// Byte address of element (r, col) (bf16) in a 128-byte-swizzled tile of 64-wide rows.
__device__ __forceinline__ uint32_t sw128_elem(uint32_t tile, int r, int col) {
    return tile + (uint32_t)(r >> 3) * 1024u + (uint32_t)(r & 7) * 128u +
           ((uint32_t)(((col >> 3) ^ r) & 7) << 4) + (uint32_t)(col & 7) * 2u;
}

// Address of 16-byte chunk `ch` (logical) of row `r` in a 128-byte-swizzled tile.
__device__ __forceinline__ uint32_t sw128_chunk(uint32_t tile, int r, int ch) {
    return tile + (uint32_t)(r >> 3) * 1024u + (uint32_t)(r & 7) * 128u +
           ((uint32_t)((ch ^ r) & 7) << 4);
}

// Writes 32 bf16 values (16 packed pairs) into logical chunks ch0..ch0+3 of row r.
__device__ __forceinline__ void write_row32_packed(uint32_t tile, int r, int ch0,
                                                   const uint32_t* u) {
#pragma unroll
    for (int j = 0; j < 4; ++j)
        st_shared_v4(sw128_chunk(tile, r, ch0 + j), u[4 * j], u[4 * j + 1], u[4 * j + 2],
                     u[4 * j + 3]);
}

// Writes 32 fp32 values as bf16 into logical chunks ch0..ch0+3 of row r.
__device__ __forceinline__ void write_row32(uint32_t tile, int r, int ch0, const float* v) {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        st_shared_v4(sw128_chunk(tile, r, ch0 + j), pack_bf16(v[8 * j + 0], v[8 * j + 1]),
                     pack_bf16(v[8 * j + 2], v[8 * j + 3]), pack_bf16(v[8 * j + 4], v[8 * j + 5]),
                     pack_bf16(v[8 * j + 6], v[8 * j + 7]));
    }
}

__device__ __forceinline__ void record_failure(volatile int* abort_flag, uint32_t bit) {
    atomicOr(&g_tc_status, bit);
    *abort_flag = 1;
}

// Waits for the phase with the given parity, suspending between polls; gives up when
// another role has set the abort flag, or after kWaitNs (then records `bit`).
__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity,
                                              volatile int* abort_flag, uint32_t bit) {
    if (mbar_try_wait_sleep(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    while (true) {
        if (mbar_try_wait_sleep(bar, parity)) return true;
        if (*abort_flag) return false;
        if (globaltimer_ns() - t0 > kWaitNs) {
            record_failure(abort_flag, bit);
            return false;
        }
    }
}

// As wait_or_abort, for the short hand-offs of the carry chain: polls with try_wait
// without a suspend-time hint, which resumes the waiting thread sooner after the phase
// completes.
__device__ __forceinline__ bool wait_hot(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                         uint32_t bit) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if (*abort_flag) return false;
        if (globaltimer_ns() - t0 > kWaitNs) {
            record_failure(abort_flag, bit);
            return false;
        }
    }
}

// The waits of the two-slice carry's chain (SIMT warps on the MMA groups, the issuer on the
// late copy group) poll without a suspend hint: ~50 cycles sooner per hand-off.
__device__ __forceinline__ bool wait_chain(uint64_t* bar, uint32_t parity,
                                           volatile int* abort_flag, uint32_t bit) {
    return wait_hot(bar, parity, abort_flag, bit);
}

// Lower-triangular 16x16 block index of block (i, j), i >= j.
__host__ __device__ constexpr int bidx(int i, int j) { return i * (i + 1) / 2 + j; }

// ---------------------------------------------------------------- tf32 mma.sync helpers
// m16n8k8 fragments (thread g = lane/4, t = lane%4): A 16x8 row-major
// {(g,t), (g+8,t), (g,t+4), (g+8,t+4)}; B 8x8 {(t,g), (t+4,g)}; C/D 16x8
// {(g,2t), (g,2t+1), (g+8,2t), (g+8,2t+1)}.

__device__ __forceinline__ uint32_t to_tf32(float x) {
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
    return r;
}

__device__ __forceinline__ void mma_tf32(float (&d)[4], const uint32_t (&a)[4],
                                         const uint32_t (&b)[2]) {
    asm volatile(
        "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}

// d += Ablk (16x16) * Bblk[:, 8 nt .. 8 nt + 7]; both blocks hold values already rounded to
// tf32 (the off-diagonal blocks of A and the blocks of T are stored that way)
__device__ __forceinline__ void block_mma(float (&d)[4], const float* Ablk, const float* Bblk,
                                          int nt, int g, int t) {
#pragma unroll
    for (int ks = 0; ks < 2; ++ks) {
        uint32_t a[4], b[2];
        a[0] = __float_as_uint(Ablk[g * BS + ks * 8 + t]);
        a[1] = __float_as_uint(Ablk[(g + 8) * BS + ks * 8 + t]);
        a[2] = __float_as_uint(Ablk[g * BS + ks * 8 + t + 4]);
        a[3] = __float_as_uint(Ablk[(g + 8) * BS + ks * 8 + t + 4]);
        b[0] = __float_as_uint(Bblk[(ks * 8 + t) * BS + nt * 8 + g]);
        b[1] = __float_as_uint(Bblk[(ks * 8 + t + 4) * BS + nt * 8 + g]);
        mma_tf32(d, a, b);
    }
}

// C fragment of X (16x8) -> tf32 B fragments of X for the two k-steps of a 16-deep
// product, through warp shuffles: b[ks] = {X[8 ks + t][g], X[8 ks + t + 4][g]}.
__device__ __forceinline__ void c_to_b(const float (&x)[4], int g, int t, uint32_t (&b)[2][2]) {
    const int s0 = 4 * t + (g >> 1), s1 = s0 + 16;
    const float a0 = __shfl_sync(0xffffffffu, x[0], s0), a1 = __shfl_sync(0xffffffffu, x[1], s0);
    const float a2 = __shfl_sync(0xffffffffu, x[2], s0), a3 = __shfl_sync(0xffffffffu, x[3], s0);
    const float d0 = __shfl_sync(0xffffffffu, x[0], s1), d1 = __shfl_sync(0xffffffffu, x[1], s1);
    const float d2 = __shfl_sync(0xffffffffu, x[2], s1), d3 = __shfl_sync(0xffffffffu, x[3], s1);
    const bool odd = (g & 1) != 0;
    b[0][0] = to_tf32(odd ? a1 : a0);
    b[0][1] = to_tf32(odd ? d1 : d0);
    b[1][0] = to_tf32(odd ? a3 : a2);
    b[1][1] = to_tf32(odd ? d3 : d2);
}

// e += Tblk (16x16 block, tf32-rounded) * X, with X given as B fragments
__device__ __forceinline__ void block_mma_b(float (&e)[4], const float* Tblk,
                                            const uint32_t (&b)[2][2], int g, int t) {
#pragma unroll
    for (int ks = 0; ks < 2; ++ks) {
        uint32_t a[4];
        a[0] = __float_as_uint(Tblk[g * BS + ks * 8 + t]);
        a[1] = __float_as_uint(Tblk[(g + 8) * BS + ks * 8 + t]);
        a[2] = __float_as_uint(Tblk[g * BS + ks * 8 + t + 4]);
        a[3] = __float_as_uint(Tblk[(g + 8) * BS + ks * 8 + t + 4]);
        mma_tf32(e, a, b[ks]);
    }
}

// Stores T(i,j)[:, 8 nt .. 8 nt + 7] = -e (C fragment): the block (rounded to tf32: only
// the tf32 products read it) and the bf16 T_U / T_W entries (columns scaled by beta_j and
// beta_j Gamma_j, from the unrounded values).
__device__ __forceinline__ void block_store(const float (&e)[4], float* Tout, int i, int j, int nt,
                                            int g, int t, const float* beta, const float* Gam,
                                            uint32_t tu, uint32_t tw) {
    const int c0 = nt * 8 + 2 * t;  // column inside the block
    Tout[g * BS + c0] = __uint_as_float(to_tf32(-e[0]));
    Tout[g * BS + c0 + 1] = __uint_as_float(to_tf32(-e[1]));
    Tout[(g + 8) * BS + c0] = __uint_as_float(to_tf32(-e[2]));
    Tout[(g + 8) * BS + c0 + 1] = __uint_as_float(to_tf32(-e[3]));
    const int J = 16 * j + c0, R0 = 16 * i + g, R1 = R0 + 8;
    const float b0 = beta[J], b1 = beta[J + 1];
    const float w0 = b0 * Gam[J], w1 = b1 * Gam[J + 1];
    st_shared_b32(sw128_elem(tu, R0, J), pack_bf16(-e[0] * b0, -e[1] * b1));
    st_shared_b32(sw128_elem(tu, R1, J), pack_bf16(-e[2] * b0, -e[3] * b1));
    st_shared_b32(sw128_elem(tw, R0, J), pack_bf16(-e[0] * w0, -e[1] * w1));
    st_shared_b32(sw128_elem(tw, R1, J), pack_bf16(-e[2] * w0, -e[3] * w1));
}

// ---------------------------------------------------------------- MMA issue helpers

// The descriptors of a tile are built once; each k-step only adds its byte offset / 16
// to the start-address field (offsets stay inside the 14-bit field).
__device__ __forceinline__ uint64_t dadd(uint64_t d, uint32_t bytes) { return d + (bytes >> 4); }

// prep: [QK^T; KK^T] = [Q; K] K^T over Dk = 128 (two 64-column blocks)
__device__ __forceinline__ void issue_gram(uint32_t tmem, uint32_t sb) {
    constexpr uint32_t id = idesc_bf16(128, 64, false, false);
    const uint64_t a0 = smem_desc_sw128(sb + PQ_Q, 16, 1024);
    const uint64_t b0 = smem_desc_sw128(sb + PQ_K, 16, 1024);
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        const uint32_t off = (uint32_t)(k >> 2) * PQ_STRIDE + (uint32_t)(k & 3) * 32u;
        mma_bf16(tmem + PT_G, dadd(a0, off), dadd(b0, off), id, k > 0);
    }
}

// prep: [W; P K] = [T_W; P] K over the 64 tokens (K read N-major: Dk contiguous)
__device__ __forceinline__ void issue_w(uint32_t tmem, uint32_t sb) {
    constexpr uint32_t id = idesc_bf16(128, 128, false, true);
    const uint64_t aw = smem_desc_sw128(sb + P_TW, 16, 1024);
    const uint64_t bk = smem_desc_sw128(sb + PQ_K, PQ_STRIDE, 1024);
#pragma unroll
    for (int k = 0; k < 4; ++k) mma_bf16(tmem + PT_W, dadd(aw, k * 32), dadd(bk, k * 2048), id, k > 0);
}

// carry: [U~; -] = [T_U; -] V over the 64 tokens (V read N-major), into TMEM buffer `tb`
// (the lower half of the operand is whatever follows T_U; that half of the result is unused)
template <int NS>
__device__ __forceinline__ void issue_u(uint32_t tmem, uint32_t st, uint32_t tb) {
    constexpr uint32_t id = idesc_bf16(128, NS, false, true);
    const uint64_t au = smem_desc_sw128(st + CarryCfg<NS>::OFF_TU, 16, 1024);
    const uint64_t bv = smem_desc_sw128(st + OFF_V, 8192, 1024);
#pragma unroll
    for (int k = 0; k < 4; ++k) mma_bf16(tmem + tb, dadd(au, k * 32), dadd(bv, k * 2048), id, k > 0);
}

// carry: [W S0; Q S0] = [W; Q] S0 over Dk = 128, into the TMEM buffer `ta`
template <int NS>
__device__ __forceinline__ void issue_carry1(uint32_t tmem, uint32_t st, uint32_t s_tile,
                                             uint32_t ta) {
    constexpr uint32_t id = idesc_bf16(128, NS, false, true);
    const uint64_t a0 = smem_desc_sw128(st + OFF_W, 16, 1024);
    const uint64_t b0 = smem_desc_sw128(s_tile, 16384, 1024);
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        const uint32_t off = (uint32_t)(k >> 2) * BLK_STRIDE + (uint32_t)(k & 3) * 32u;
        mma_bf16(tmem + ta, dadd(a0, off), dadd(b0, k * 2048), id, k > 0);
    }
}

// carry: the state increment K~^T U over the tokens (K~ read M-major), into `tb`
template <int NS>
__device__ __forceinline__ void issue_carry3(uint32_t tmem, uint32_t st, uint32_t u_tile,
                                             uint32_t tb) {
    constexpr uint32_t id = idesc_bf16(128, NS, true, true);
    const uint64_t ak = smem_desc_sw128(st + OFF_K, BLK_STRIDE, 1024);
    const uint64_t bu2 = smem_desc_sw128(u_tile, 8192, 1024);
#pragma unroll
    for (int k = 0; k < 4; ++k)
        mma_bf16(tmem + tb, dadd(ak, k * 2048), dadd(bu2, k * 2048), id, k > 0);
}

// carry: [K~_1 U; P U] = [K~_1; P] U into the TMEM buffer `tc` (the upper half, over the
// K~ block that precedes P, is not used)
template <int NS>
__device__ __forceinline__ void issue_carry2(uint32_t tmem, uint32_t st, uint32_t u_tile,
                                             uint32_t tc) {
    constexpr uint32_t id = idesc_bf16(128, NS, false, true);
    const uint64_t ap = smem_desc_sw128(st + OFF_P - 8192, 16, 1024);
    const uint64_t bu = smem_desc_sw128(u_tile, 8192, 1024);
#pragma unroll
    for (int k = 0; k < 4; ++k)
        mma_bf16(tmem + tc, dadd(ap, k * 32), dadd(bu, k * 2048), id, k > 0);
}

// ---------------------------------------------------------------- the prep kernel

// One CTA per (chunk c, value head h, batch b). Warp 0 loads Q and K of the chunk (TMA),
// builds the decay tables from g and beta, and issues the two MMAs; warps 1..8 turn the
// Gram matrices into P and A, solve (I+A)^-1 in 16x16 blocks, write T_U, T_W and P as
// bf16 tiles, read W back from TMEM, and store T_U | P | W to the workspace.
__global__ void __launch_bounds__(PREP_THREADS, 3)
    prep_tc_kernel(const __grid_constant__ CUtensorMap mq, const __grid_constant__ CUtensorMap mk,
                   TcArgs a) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    // 1024-byte alignment by a byte offset from the shared array itself, so every
    // pointer derived from `sm` stays a shared-memory pointer.
    uint8_t* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const uint32_t sb = smem_u32(sm);
    uint64_t* bar = reinterpret_cast<uint64_t*>(sm + P_BAR);
    uint32_t* misc = reinterpret_cast<uint32_t*>(sm + P_MISC);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(misc + 1);
    PrepScalars& sc = *reinterpret_cast<PrepScalars*>(sm + P_SCAL);
    float* Tb = reinterpret_cast<float*>(sm + P_TB);
    // fp32 block (i, j) of A, in the Q slots
    auto Ablk = [&](int i, int j) -> float* {
        const int x = bidx(i, j);
        return reinterpret_cast<float*>(sm + (x < 6 ? PQ_Q : PQ_STRIDE + PQ_Q)) +
               (x < 6 ? x : x - 6) * 16 * BS;
    };

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int cl = blockIdx.x, h = blockIdx.y;
    const int kh = h / (a.Hv / a.Hk);  // value head h reads key head h // (Hv/Hk)
    const int S = a.S;
    const int nch = a.nseg;
    // the chunk: its first token `tc` and token bound `tend` in the [heads][S] tensors
    // (a variable-length batch packs its sequences along S; the grid then covers an upper
    // bound of their chunks and the surplus CTAs leave at once)
    int b = blockIdx.z, tc, tend;
    if (a.cu == nullptr) {
        tc = (a.c0 + cl) * C;
        tend = S;
    } else {
        if (cl >= a.cb[a.N]) return;
        const int n = seq_of_chunk(a.cb, a.N, cl);
        tc = a.cu[n] + (cl - a.cb[n]) * C;
        tend = a.cu[n + 1];
        b = 0;
    }

    const int zq = b * a.Hk + kh, zv = b * a.Hv + h;
    if (tid == 0) TRACE_PREP(29);
    SPAN_BEGIN(a.c0 == 0 ? 0 : 2);
    // g and beta of the chunk are loaded first and the copies of Q and K started at
    // once, so that their latency overlaps the setup (padding tokens -- past the end of
    // the sequence -- get g = beta = 0, an exact no-op)
    float x0 = 0.f, x1 = 0.f, be0 = 0.f, be1 = 0.f;
    if (warp == 0) {
        const float* gp = a.g + (size_t)zv * S;
        const float* bp = a.beta + (size_t)zv * S;
        const int t0 = tc + lane, t1 = t0 + 32;
        if (t0 < tend) x0 = gp[t0], be0 = bp[t0];
        if (t1 < tend) x1 = gp[t1], be1 = bp[t1];
    }
    if (tid == 0) {
        for (int i = 0; i < PB_COUNT; ++i) mbar_init(&bar[i], i == PB_FULL ? 2 : 1);
        *abort_flag = 0;
        fence_mbar_init();
        mbar_arrive_expect_tx(&bar[PB_FULL], 2 * 16384);
        for (int blk = 0; blk < 2; ++blk) {
            tma_load_3d(sm + blk * PQ_STRIDE + PQ_Q, &mq, &bar[PB_FULL], blk * 64, tc, zq);
            tma_load_3d(sm + blk * PQ_STRIDE + PQ_K, &mk, &bar[PB_FULL], blk * 64, tc, zq);
        }
        TRACE_PREP(20);
    }
    if (warp == 0) {
        tmem_alloc(misc, PT_COLS);
        tmem_relinquish();
    }
    // T_U / T_W blocks above the diagonal are never written: zero both tiles
    for (int i = tid; i < 2 * 8192 / 16; i += PREP_THREADS)
        st_shared_v4(sb + P_TU + 16 * i, 0u, 0u, 0u, 0u);
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = misc[0];
    // a carry launched as a programmatic dependent of this grid may start its setup once
    // every prep CTA has begun (it waits for the grid's end before reading the workspace)
    if (tid == 0) grid_dep_launch_dependents();

    if (warp == 0) {
        // -------------------------------------------- decay tables, MMA issue
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const float y0 = __shfl_up_sync(0xffffffffu, x0, off);
            const float y1 = __shfl_up_sync(0xffffffffu, x1, off);
            if (lane >= off) {
                x0 += y0;
                x1 += y1;
            }
        }
        x1 += __shfl_sync(0xffffffffu, x0, 31);
        const float gl = __shfl_sync(0xffffffffu, x1, 31);
        const float e0 = __shfl_sync(0xffffffffu, x0, lane | 15);
        const float e1 = __shfl_sync(0xffffffffu, x1, lane | 15);
        CarryScalars& cs = *reinterpret_cast<CarryScalars*>(sm + P_CS);
        cs.kdec[lane] = __expf(gl - x0);
        cs.kdec[lane + 32] = __expf(gl - x1);
        cs.Gam[lane] = __expf(x0);
        cs.Gam[lane + 32] = __expf(x1);
        if (lane == 31) cs.Gl = __expf(gl);
        sc.gam[lane] = x0;
        sc.gam[lane + 32] = x1;
        sc.beta[lane] = be0;
        sc.beta[lane + 32] = be1;
        sc.ctab[lane] = __expf(e0 - x0);
        sc.ctab[lane + 32] = __expf(e1 - x1);
        sc.Gam[lane] = __expf(x0);
        sc.Gam[lane + 32] = __expf(x1);
        if (lane == 15) {
            sc.endgam[0] = x0;
            sc.endgam[2] = x1;
        }
        if (lane == 31) {
            sc.endgam[1] = x0;
            sc.endgam[3] = x1;
        }
        fence_proxy_async_smem();  // the scalar staging is stored by a bulk copy
        __syncwarp();
        if (lane == 0) {
            mbar_arrive(&bar[PB_FULL]);  // the tables are written
            int issued = 0;
            if (wait_or_abort(&bar[PB_FULL], 0, abort_flag, ST_PREP)) {
                tc_fence_after();
                issue_gram(tmem, sb);
                tc_commit(&bar[PB_GRAM]);
                issued = 1;
                TRACE_PREP(21);
            } else {
                // the copies must land before the CTA exits
                mbar_wait_bounded(&bar[PB_FULL], 0, kWaitNs);
            }
            if (issued) {
                // no MMA may be in flight when TMEM is freed
                tc_commit(&bar[PB_DRAIN]);
                mbar_wait_bounded(&bar[PB_DRAIN], 0, kWaitNs);
            }
        }
    } else {
        // ------------------------------------------------------------ prep (256 threads)
        const int P = tid - 32;
        const int pw = P >> 5;  // prep warp 0..7
        const int wg = P >> 7;  // which 8 columns of each 16-block of the Gram matrices
        const int q = warp & 3;
        const int L = 32 * q + lane;
        const int g8 = lane >> 2, t4 = lane & 3;
        const uint32_t lane_off = (uint32_t)(32 * q) << 16;
        const uint32_t tu = sb + P_TU, tw = sb + P_TW;
        bool w_issued = false;  // thread P == 0 issued the W MMA

        // One warp polls the mbarriers; the others wait at the named barrier, which costs
        // no issue slots (the prep is bound by instruction issue, with three CTAs per SM).
        // The barrier then carries the phase's visibility to every prep thread.
        bool ok = true;
        if (pw == 0)
            ok = wait_or_abort(&bar[PB_FULL], 0, abort_flag, ST_PREP) &&
                 wait_or_abort(&bar[PB_GRAM], 0, abort_flag, ST_PREP);
        if (!bar_any(2, 256, !ok || *abort_flag)) {
            tc_fence_after();
            if (P == 0) TRACE_PREP(23);

            // ---- P (bf16 tile) and A (fp32 blocks) from the Gram matrices: thread (wg, L)
            // takes row L of [QK^T; KK^T], columns 16 bj + 8 wg .. + 7 of every 16-block bj.
            // A warp's rows fill the two row blocks bq, bq + 1, so blocks left of bq and
            // right of bq + 1 are uniform over the warp (one factor per block times the
            // column's table entry; zero); in the two blocks between, each lane selects left
            // of, on (the masked exp of a non-positive argument) or right of its diagonal.
            // The off-diagonal blocks of A feed only the tf32 products of the inverse's
            // doubling steps, so they are stored rounded to tf32.
            {
                const int r = L & 63, br = r >> 4, rl = r & 15;
                const int bq = (r >> 5) * 2;  // uniform over the warp
                const bool isP = L < 64;      // uniform over the warp
                const float gr = sc.gam[r];
                const float scl = isP ? 1.f : sc.beta[r];
                const int lim = isP ? rl : rl - 1;
                float gv[32];
                tmem_ld8x4(tmem + lane_off + PT_G + 8 * wg, gv);
                float dg[8];
                {
                    const float4* gp = reinterpret_cast<const float4*>(sc.gam + 16 * br + 8 * wg);
                    const float4 g0 = gp[0], g1 = gp[1];
                    const float gj[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
#pragma unroll
                    for (int e = 0; e < 8; ++e)
                        dg[e] = __expf(fminf(gr - gj[e], 0.f)) * ((8 * wg + e <= lim) ? scl : 0.f);
                }
#pragma unroll
                for (int bj = 0; bj < 4; ++bj) {
                    float* v = gv + 8 * bj;
                    if (bj > bq + 1) {  // right of the diagonal for the whole warp
                        if (isP)
                            st_shared_v4(sw128_chunk(sb + P_P, r, 2 * bj + wg), 0u, 0u, 0u, 0u);
                        continue;
                    }
                    const float4* cp = reinterpret_cast<const float4*>(sc.ctab + 16 * bj + 8 * wg);
                    const float4 c0 = cp[0], c1 = cp[1];
                    const float ct[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
                    if (bj < bq) {  // left of the diagonal for the whole warp
                        const float fb = __expf(gr - sc.endgam[bj]) * scl;
#pragma unroll
                        for (int e = 0; e < 8; ++e) v[e] *= fb * ct[e];
                    } else {
                        const float fb = (bj < br) ? __expf(gr - sc.endgam[bj]) * scl : 0.f;
#pragma unroll
                        for (int e = 0; e < 8; ++e)
                            v[e] *= (bj < br) ? fb * ct[e] : ((bj == br) ? dg[e] : 0.f);
                    }
                    if (isP) {
                        st_shared_v4(sw128_chunk(sb + P_P, r, 2 * bj + wg), pack_bf16(v[0], v[1]),
                                     pack_bf16(v[2], v[3]), pack_bf16(v[4], v[5]),
                                     pack_bf16(v[6], v[7]));
                    } else if (bj <= br) {
                        if (bj < br) {
#pragma unroll
                            for (int e = 0; e < 8; ++e) v[e] = __uint_as_float(to_tf32(v[e]));
                        }
                        float* dst = Ablk(br, bj) + rl * BS + 8 * wg;
                        *reinterpret_cast<float4*>(dst) = make_float4(v[0], v[1], v[2], v[3]);
                        *reinterpret_cast<float4*>(dst + 4) = make_float4(v[4], v[5], v[6], v[7]);
                    }
                }
            }
            tc_fence_before();  // the Gram columns are reused by the W MMA
            bar_sync(2, 256);
            if (P == 0) TRACE_PREP(24);

            // ---- T = (I + A)^-1 in 16x16 blocks
            // diagonal blocks (prep warps 0 and 1): forward substitution, one thread per
            // column of the block's inverse, its 16 entries in registers. The rows go in
            // lockstep, so the threads of a block read the same A entry (a broadcast);
            // the column's zeros above its diagonal keep the full sums exact.
            // Meanwhile warps 2..7 write K~ to the workspace (when it is exported).
            if (P < 64) {
                const int i = P >> 4, cc = P & 15;
                const float* Ad = Ablk(i, i);
                float x[16];
#pragma unroll
                for (int m = 0; m < 16; ++m) x[m] = (m == cc) ? 1.f : 0.f;
#pragma unroll
                for (int m = 1; m < 16; ++m) {
                    float s0 = 0.f, s1 = 0.f;
#pragma unroll
                    for (int n = 0; n < m; n += 2) {
                        s0 = fmaf(Ad[m * BS + n], x[n], s0);
                        if (n + 1 < m) s1 = fmaf(Ad[m * BS + n + 1], x[n + 1], s1);
                    }
                    if (m > cc) x[m] = -(s0 + s1);
                }
                float* Td = Tb + bidx(i, i) * 16 * BS;
#pragma unroll
                for (int m = 0; m < 16; ++m) Td[m * BS + cc] = __uint_as_float(to_tf32(x[m]));
            } else if (a.export_k) {
                // meanwhile K~ = diag(exp(gamma_last - gamma)) K goes straight to the
                // workspace: 16-byte chunk j of the two 64-column blocks, same swizzled
                // position, one packed bf16 product per pair (the row factor rounded to bf16)
                const CarryScalars& cs = *reinterpret_cast<const CarryScalars*>(sm + P_CS);
                uint8_t* wsk = a.ws + ws_offset(b, h, cl, a.Hv, nch) + WS_KT;
                for (int j = P - 64; j < 1024; j += 192) {
                    const int blk = j >> 9, off = (j & 511) * 16, row = (j & 511) >> 3;
                    const __nv_bfloat162 f2 = __float2bfloat162_rn(cs.kdec[row]);
                    const uint4 x = *reinterpret_cast<const uint4*>(sm + blk * PQ_STRIDE + PQ_K + off);
                    const uint32_t in[4] = {x.x, x.y, x.z, x.w};
                    uint32_t o[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const __nv_bfloat162 r =
                            __hmul2(*reinterpret_cast<const __nv_bfloat162*>(&in[e]), f2);
                        o[e] = *reinterpret_cast<const uint32_t*>(&r);
                    }
                    *reinterpret_cast<uint4*>(wsk + blk * 8192 + off) =
                        make_uint4(o[0], o[1], o[2], o[3]);
                }
            }
            bar_sync(2, 256);
            if (P == 0) TRACE_PREP(25);
            // off-diagonal blocks by doubling. Step 1: T(i,i-1) = -T(i,i) A(i,i-1) T(i-1,i-1)
            // for i = 1, 3; warp: (i, 8 columns)
            if (pw < 4) {
                const int i = (pw & 2) ? 3 : 1, j = i - 1, nt = pw & 1;
                float x[4] = {0.f, 0.f, 0.f, 0.f}, e[4] = {0.f, 0.f, 0.f, 0.f};
                block_mma(x, Ablk(i, j), Tb + bidx(j, j) * 16 * BS, nt, g8, t4);
                uint32_t bx[2][2];
                c_to_b(x, g8, t4, bx);
                block_mma_b(e, Tb + bidx(i, i) * 16 * BS, bx, g8, t4);
                block_store(e, Tb + bidx(i, j) * 16 * BS, i, j, nt, g8, t4, sc.beta, sc.Gam, tu,
                            tw);
            } else {
                // meanwhile the diagonal blocks go to the bf16 T_U / T_W tiles: thread = 8
                // columns (one 16-byte chunk) of one row of one block, columns scaled by
                // beta_J and beta_J Gamma_J (zeros above the diagonal come with the block)
                const int u = P - 128, i = u >> 5, m = (u >> 1) & 15, hh = u & 1;
                const float* src = Tb + bidx(i, i) * 16 * BS + m * BS + 8 * hh;
                const int J = 16 * i + 8 * hh;
                const float4 t0 = *reinterpret_cast<const float4*>(src);
                const float4 t1 = *reinterpret_cast<const float4*>(src + 4);
                const float4 b0 = *reinterpret_cast<const float4*>(sc.beta + J);
                const float4 b1 = *reinterpret_cast<const float4*>(sc.beta + J + 4);
                const float4 g0 = *reinterpret_cast<const float4*>(sc.Gam + J);
                const float4 g1 = *reinterpret_cast<const float4*>(sc.Gam + J + 4);
                const float tv[8] = {t0.x, t0.y, t0.z, t0.w, t1.x, t1.y, t1.z, t1.w};
                const float bv[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
                const float gv[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
                uint32_t ou[4], ow[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float u0 = tv[2 * e] * bv[2 * e], u1 = tv[2 * e + 1] * bv[2 * e + 1];
                    ou[e] = pack_bf16(u0, u1);
                    ow[e] = pack_bf16(u0 * gv[2 * e], u1 * gv[2 * e + 1]);
                }
                const int R = 16 * i + m;
                st_shared_v4(sw128_chunk(tu, R, J >> 3), ou[0], ou[1], ou[2], ou[3]);
                st_shared_v4(sw128_chunk(tw, R, J >> 3), ow[0], ow[1], ow[2], ow[3]);
            }
            bar_sync(2, 256);
            if (P == 0) TRACE_PREP(26);
            // Step 2: the lower-left 32x32 quadrant, T_BA = -T_BB (A_BA T_AA): with
            // X(l,j) = sum_{m=j..1} A(l,m) T(m,j), T(2,j) = -T(2,2) X(2,j) and
            // T(3,j) = -(T(3,2) X(2,j) + T(3,3) X(3,j)); warp: (i, j, 8 columns)
            {
                const int i = 2 + (pw >> 2), j = (pw >> 1) & 1, nt = pw & 1;
                float x2[4] = {0.f, 0.f, 0.f, 0.f}, x3[4] = {0.f, 0.f, 0.f, 0.f};
                float e[4] = {0.f, 0.f, 0.f, 0.f};
                for (int m = j; m < 2; ++m) {
                    block_mma(x2, Ablk(2, m), Tb + bidx(m, j) * 16 * BS, nt, g8,
                              t4);
                    if (i == 3)
                        block_mma(x3, Ablk(3, m), Tb + bidx(m, j) * 16 * BS, nt,
                                  g8, t4);
                }
                uint32_t bx[2][2];
                c_to_b(x2, g8, t4, bx);
                block_mma_b(e, Tb + bidx(i, 2) * 16 * BS, bx, g8, t4);
                if (i == 3) {
                    c_to_b(x3, g8, t4, bx);
                    block_mma_b(e, Tb + bidx(3, 3) * 16 * BS, bx, g8, t4);
                }
                block_store(e, Tb + bidx(i, j) * 16 * BS, i, j, nt, g8, t4, sc.beta, sc.Gam, tu,
                            tw);
            }
            fence_proxy_async_smem();  // T_U, T_W and P are read by the W MMA and copies
            bar_sync(2, 256);
            uint8_t* wsu = a.ws + ws_offset(b, h, cl, a.Hv, nch);
            if (P == 0) {
                TRACE_PREP(27);
                // [W; P K] = [T_W; P] K, issued here as soon as T_W is complete (the
                // Gram columns it overwrites were read before the mask barrier)
                tc_fence_after();
                issue_w(tmem, sb);
                tc_commit(&bar[PB_WDONE]);
                w_issued = true;
                TRACE_PREP(22);
                // T_U, P and the scalars are final: to the workspace now, under the W MMA
                bulk_s2g(wsu + WS_TU, sb + P_TU, 8192);
                bulk_s2g(wsu + WS_P, sb + P_P, 8192);
                bulk_s2g(wsu + WS_CS, sb + P_CS, sizeof(CarryScalars));
                bulk_commit();
            }
            // ---- W = T_W K from TMEM (rows 0..63: lanes 0..63) into the W staging tiles;
            // two warps per lane quadrant, one 64-column block each
            if (pw == 0) ok = wait_or_abort(&bar[PB_WDONE], 0, abort_flag, ST_PREP);
            if (P == 0) TRACE_PREP(54);
            if (!bar_any(2, 256, !ok || *abort_flag)) {
                tc_fence_after();
                if (q < 2) {
                    const int hc = (warp >= 5) ? 1 : 0;
#pragma unroll
                    for (int hh = 0; hh < 2; ++hh) {
                        float w[32];
                        tmem_ld32(tmem + lane_off + PT_W + 64 * hc + 32 * hh, w);
                        write_row32(sb + PQ_STRIDE * hc + PQ_Q, L, 4 * hh, w);
                    }
                }
                fence_proxy_async_smem();
                bar_sync(2, 256);
                if (P == 0) {
                    TRACE_PREP(28);
                    bulk_s2g(wsu + WS_W, sb + PQ_Q, 8192);
                    bulk_s2g(wsu + WS_W + 8192, sb + PQ_STRIDE + PQ_Q, 8192);
                    bulk_commit();
                }
            }
        }
        if (P == 0) {
            // the CTA may exit once the tiles are read out of shared memory: the carry, a
            // later kernel, sees the global writes completed
            bulk_wait_read_all();
            TRACE_PREP(53);
            // no MMA may be in flight when TMEM is freed
            if (w_issued && !mbar_wait_bounded(&bar[PB_WDONE], 0, kWaitNs))
                atomicOr(&g_tc_status, ST_PREP);
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, PT_COLS);
    }
    SPAN_END(a.c0 == 0 ? 0 : 2);
}

// ---------------------------------------------------------------- the carry kernel

// One CTA per (NS-column slice of the state, value head h, batch b), sequential over
// chunks. Warp 0 streams the chunk's q and v slice (TMA) and the prep's tiles and
// scalars (bulk copies) into a two-stage ring; warps 4..11 (two per TMEM lane quadrant,
// thread = state row L, NS/2 columns) keep the fp32 state in registers, form U (rows
// 0-63, the U warps 4, 5, 8, 9) while writing the previous chunk's output (rows 64-127, the
// output warps 6, 7, 10, 11), and update the state; one thread of warp 1 issues every MMA.
// MMA order per chunk c: [W; Q] S0, U~ of chunk c+1 if it has landed, then K~^T U, U~ of
// chunk c+1 if not issued yet, P U. (Every MMA comes from the one thread: the tensor pipe
// takes about one tcgen05.mma per 44 cycles whichever thread issues it, so a second issuer
// only puts the off-chain MMAs in front of the chain's.)

// The producer of a carry CTA (one thread): streams chunk c (token rows tbase + 64 c) into
// the two-stage ring, in the early (W, q, V, T_U) and late (K~ or k, P, scalars) copy
// groups: the prep's tiles and scalars from the head's workspace units (from `wsh`), the V
// slice (columns n0 .. n0 + NS - 1, tensor z = zv), q of the key head (tensor z = zq, both
// 64-column blocks) and either the prep's K~ (kt_ws, for the two-slice carry) or k of the
// key head (for the transposed carry, which also has chunk c + 2 prefetched into L2).
template <int NS>
__device__ __forceinline__ void carry_produce(uint8_t* sm, uint64_t* bar, CarryScalars* scal,
                                              const CUtensorMap* mqp, const CUtensorMap* mkp,
                                              const CUtensorMap* mvp, bool kt_ws, bool ws_wait,
                                              const uint8_t* wsh, int nch, int n0, int tbase,
                                              int zq, int zv, volatile int* abort_flag) {
    using Cfg = CarryCfg<NS>;
    if (ws_wait) grid_dep_wait();  // the prep before this grid wrote the workspace
    int lastE[2] = {-1, -1}, lastL[2] = {-1, -1};  // last chunk of each group in each stage
    for (int c = 0; c < nch; ++c) {
        const int s = c & 1;
#ifdef GDN_TEST_STALL
        if (c == 1) continue;  // test build: the second chunk is never loaded
#endif
        uint8_t* st = sm + s * Cfg::STAGE;
        const uint8_t* wsc = wsh + (size_t)c * WS_UNIT;
        const int t = tbase + c * C;
        // early group of chunk c: W, q, V, T_U
        if (c >= 2 && !wait_or_abort(&bar[B_EMPTYE0 + s], ((c >> 1) + 1) & 1, abort_flag,
                                     ST_PRODUCER))
            break;
        if (*abort_flag) break;
        TRACE(c, 19);
        uint64_t* fe = &bar[B_FULLE0 + s];
        mbar_arrive_expect_tx(fe, 4 * 8192 + Cfg::NB * 8192 + 8192);
        for (int blk = 0; blk < 2; ++blk) {
            uint8_t* sb = st + blk * BLK_STRIDE;
            bulk_g2s(sb + OFF_W, wsc + WS_W + blk * 8192, 8192, fe);
            tma_load_3d(sb + OFF_Q, mqp, fe, blk * 64, t, zq);
        }
        for (int blk = 0; blk < Cfg::NB; ++blk)
            tma_load_3d(st + OFF_V + blk * 8192, mvp, fe, n0 + blk * 64, t, zv);
        bulk_g2s(st + Cfg::OFF_TU, wsc + WS_TU, 8192, fe);
        lastE[s] = c;
        // late group of chunk c: K~ or k, P, scalars
        if (c >= 2 && !wait_or_abort(&bar[B_EMPTYL0 + s], ((c >> 1) + 1) & 1, abort_flag,
                                     ST_PRODUCER))
            break;
        uint64_t* fl = &bar[B_FULLL0 + s];
        TRACE(c, 18);
        mbar_arrive_expect_tx(fl, 3 * 8192 + (uint32_t)sizeof(CarryScalars));
        for (int blk = 0; blk < 2; ++blk) {
            uint8_t* dk = st + blk * BLK_STRIDE + OFF_K;
            if (kt_ws) bulk_g2s(dk, wsc + WS_KT + blk * 8192, 8192, fl);
            else tma_load_3d(dk, mkp, fl, blk * 64, t, zq);
        }
        bulk_g2s(st + OFF_P, wsc + WS_P, 8192, fl);
        bulk_g2s(&scal[s], wsc + WS_CS, sizeof(CarryScalars), fl);
        lastL[s] = c;
        // chunk c + 2 goes to L2 now, for the transposed carry, whose full waves are bound
        // by HBM bandwidth. The two-slice carry does without: the prefetches share the
        // SM's copy engine with the chunk loads its chain waits for (a traced chunk took
        // about 2.6K cycles without them, 2.9K with).
        if (!kt_ws && c + 2 < nch) {
            const int t2 = t + 2 * C;
            for (int blk = 0; blk < Cfg::NB; ++blk) tma_prefetch_l2_3d(mvp, n0 + blk * 64, t2, zv);
            for (int blk = 0; blk < 2; ++blk) {
                tma_prefetch_l2_3d(mqp, blk * 64, t2, zq);
                tma_prefetch_l2_3d(mkp, blk * 64, t2, zq);
            }
            bulk_prefetch_l2(wsc + 2 * WS_UNIT, WS_KT);
            bulk_prefetch_l2(wsc + 2 * WS_UNIT + WS_CS, sizeof(CarryScalars));
        }
    }
    // every load is issued (the last chunks are in flight): a dependent carry segment may
    // start its setup
    grid_dep_launch_dependents();
    // every copy issued lands before the CTA exits (also when a consumer gave up before
    // waiting for it); a group never issued is not waited for
    for (int s = 0; s < 2; ++s) {
        if (lastE[s] >= 0) mbar_wait_bounded(&bar[B_FULLE0 + s], (lastE[s] >> 1) & 1, kWaitNs);
        if (lastL[s] >= 0) mbar_wait_bounded(&bar[B_FULLL0 + s], (lastL[s] >> 1) & 1, kWaitNs);
    }
}


// The MMA issuer's warp. Warp 1 shares its SM sub-partition with the U warps 5 and 9,
// which wait while [W; Q] S0 is issued; the partitions of warps 2 and 3 hold the output
// warps, which are then writing the previous chunk.
constexpr int kIssuerWarp = 1;

template <int NS>
__global__ void __launch_bounds__(CARRY_THREADS, 1)
    carry_tc_kernel(const __grid_constant__ CUtensorMap mq, const __grid_constant__ CUtensorMap mk,
                    const __grid_constant__ CUtensorMap mv, TcArgs a) {
    using Cfg = CarryCfg<NS>;
    constexpr int CPT = Cfg::CPT, NP = CPT / 32;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const uint32_t sbase = smem_u32(sm);
    uint64_t* bar = reinterpret_cast<uint64_t*>(sm + Cfg::BAR);
    uint32_t* misc = reinterpret_cast<uint32_t*>(sm + Cfg::MISC);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(misc + 1);
    CarryScalars* scal = reinterpret_cast<CarryScalars*>(sm + Cfg::SCAL);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int n0 = blockIdx.x * NS, h = blockIdx.y;
    const int S = a.S;
    // The sequence of this CTA: its chunks (the workspace units u0 .. u0 + nch - 1 of
    // head row `wb`), first token `tbase`, token bound `tend`, state row `sb`. Dense
    // layout: batch b, chunks a.c0 .. a.c0 + a.nseg - 1. Variable-length batch: sequence
    // blockIdx.z, its packed tokens cu[n] .. cu[n+1] - 1.
    int wb, u0, nch, tbase, tend, sb;
    if (a.cu == nullptr) {
        wb = blockIdx.z, u0 = 0, nch = a.nseg, tbase = a.c0 * C, tend = S;
        sb = blockIdx.z * a.Hv + h;
    } else {
        const int n = blockIdx.z;
        wb = 0, u0 = a.cb[n], nch = a.cb[n + 1] - a.cb[n], tbase = a.cu[n], tend = a.cu[n + 1];
        sb = n * a.Hv + h;
    }
    if (nch == 0) {
        // an empty sequence: the state passes through (zero when none was supplied)
        grid_dep_wait();
        if (!a.state_is_input)
            for (int i = tid; i < 128 * NS; i += CARRY_THREADS)
                a.state[((size_t)sb * 128 + i / NS) * 128 + n0 + i % NS] = 0.f;
        return;
    }

    SPAN_BEGIN(a.c0 == 0 ? 1 : 3);
    if (tid == 0) {
        for (int i = 0; i < B_COUNT; ++i) mbar_init(&bar[i], 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(misc, Cfg::TMCOLS);
        tmem_relinquish();
    }
    if (tid == 32) prefetch_tensormap(&mv);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = misc[0];

    if (warp == 0) {
        // ------------------------------------------------- loads (one thread)
        if (lane == 0) {
            carry_produce<NS>(sm, bar, scal, &mq, &mk, &mv, true, a.ws_wait != 0,
                              a.ws + ws_offset(wb, h, u0, a.Hv, a.nseg), nch, n0, tbase,
                              wb * a.Hk + h / (a.Hv / a.Hk), wb * a.Hv + h, abort_flag);

        }
    } else if (warp == kIssuerWarp || warp >= 4) {
        // ----------------------------------------- carry (issuer warp, 4..11: 288 threads)
        const bool issuer = warp == kIssuerWarp;
        const bool leader = issuer && lane == 0;
        const int q = warp & 3, hc = issuer ? 0 : (warp - 4) >> 2;
        const int L = 32 * q + lane;
        const int col0 = CPT * hc;  // first state column of this thread within the slice
        const uint32_t lane_off = ((uint32_t)(32 * q) << 16) + (uint32_t)col0;
        const uint32_t s_base = sbase + Cfg::SM_S, u_tile = sbase + Cfg::U;
        float* gstate = a.state + ((size_t)sb * 128 + L) * 128 + n0 + col0;
        __nv_bfloat16* gout = a.out + (size_t)(wb * a.Hv + h) * S * 128 + n0 + col0;
        // 32-column piece p of this thread: tile block and 16-byte chunk within the block
        auto pblk = [&](int p) { return (uint32_t)((col0 + 32 * p) >> 6); };
        auto pch = [&](int p) { return ((col0 + 32 * p) & 63) >> 3; };

        // the fp32 state: row L, columns col0 .. col0 + CPT - 1 of the slice, in registers
        float Sr[CPT];
        if (!issuer) {
            grid_dep_wait();  // the carry of the segment before wrote this state
            if (a.state_is_input) {
#pragma unroll
                for (int j = 0; j < CPT; j += 4) {
                    const float4 x = *reinterpret_cast<const float4*>(gstate + j);
                    Sr[j] = x.x;
                    Sr[j + 1] = x.y;
                    Sr[j + 2] = x.z;
                    Sr[j + 3] = x.w;
                }
            } else {
#pragma unroll
                for (int j = 0; j < CPT; ++j) Sr[j] = 0.f;
            }
#pragma unroll
            for (int p = 0; p < NP; ++p) write_row32(s_base + 16384u * pblk(p), L, pch(p), Sr + 32 * p);
        }

        // out = scale (Gamma_r (Q S0)_r + (P U)_r) of chunk cc for token r = L - 64
        // (quadrants 2, 3), with gsc = scale Gamma_r
        auto write_out = [&](int cc, float gsc) {
            const int t = tbase + cc * C + (L - 64);
            const uint32_t ta = Cfg::TMA + (uint32_t)NS * (uint32_t)(cc & 1);
            const uint32_t tcb = Cfg::TMC + (uint32_t)NS * (uint32_t)(cc & 1);
#pragma unroll
            for (int p = 0; p < NP; ++p) {
                float o[32], pu[32];
                tmem_ld32x2(tmem + lane_off + ta + 32 * p, tmem + lane_off + tcb + 32 * p, o, pu);
                if (t < tend) {
                    uint4* dst = reinterpret_cast<uint4*>(gout + (size_t)t * 128 + 32 * p);
#pragma unroll
                    for (int j = 0; j < 32; ++j) o[j] = fmaf(gsc, o[j], a.scale * pu[j]);
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        uint4 w;
                        w.x = pack_bf16(o[8 * j + 0], o[8 * j + 1]);
                        w.y = pack_bf16(o[8 * j + 2], o[8 * j + 3]);
                        w.z = pack_bf16(o[8 * j + 4], o[8 * j + 5]);
                        w.w = pack_bf16(o[8 * j + 6], o[8 * j + 7]);
                        dst[j] = w;
                    }
                }
            }
        };

        int mmas = 0, done = 0;
        // SIMT warp -> issuer hand-offs, named barriers that also OR a failure flag over
        // their members (bar_any), so that every member learns at once that a wait ran out:
        //   BAR_S #c (issuer warp + 8 SIMT warps): the state tile of chunk c is written
        //            (#0: the initial state), the output of chunk c-2 is read out of TMEM
        //   BAR_U #c (issuer warp + the 4 U warps): U of chunk c is in its tile
        // Each member passes every barrier of every chunk in the same order until a BAR_S
        // reports a failure; then all of them stop there together. Every wait between the
        // barriers is bounded (and returns at once once the abort flag is set), so no
        // member can keep another waiting at a barrier.
        constexpr uint32_t BAR_S = 2, BAR_U = 3;
        auto handoff = [&]() {
            fence_proxy_async_smem();
            tc_fence_before();
        };
        bool ok = true, fail = false;
        // A failure seen by one lane (the issuing lane, or one lane's wait) becomes the whole
        // warp's before the next warp-collective instruction (tcgen05.ld, bar.red), so that
        // every lane of a warp always takes the same path to those.
        auto warp_fail = [&]() { fail = __any_sync(0xffffffffu, fail); };
        float gsc_prev = 0.f;  // output warps: scale Gamma_r of the previous chunk's row
        if (issuer) {
            bool u_next = false;  // U~(c+1) already issued
            bool stopped = false;
            if (leader) {
                if (wait_chain(&bar[B_FULLE0], 0, abort_flag, ST_MMA)) {
                    tc_fence_after();
                    issue_u<NS>(tmem, sbase, Cfg::TMB);
                    mmas = 1;
                } else {
                    fail = true;
                }
            }
            __syncwarp();
            for (int c = 0; c < nch; ++c) {
                const int s = c & 1;
                const uint32_t st = sbase + s * Cfg::STAGE;
                const uint32_t ta = Cfg::TMA + (uint32_t)NS * (uint32_t)s;
                const uint32_t tb = Cfg::TMB + (uint32_t)NS * (uint32_t)s;
                // MMA1 [W; Q] S0 once the state tile of chunk c is complete
                if (leader) TRACE(c, 52);
                if (bar_any(BAR_S, 288, fail)) {
                    stopped = true;
                    break;
                }
                if (leader) {
                    TRACE(c, 12);
                    tc_fence_after();
                    issue_carry1<NS>(tmem, st, s_base, ta);
                    TRACE(c, 6);
                    // ADONE also covers U~(c) and P U(c-1), issued earlier (U of chunk c may
                    // overwrite the U tile P U(c-2) read)
                    tc_commit(&bar[B_ADONE]);
                    tc_commit(&bar[B_EMPTYE0 + s]);  // the early group of chunk c is read
                    // U~(c+1) now if chunk c+1 has landed (it then runs while U is formed);
                    // its buffer was last read by the state update of chunk c-1
                    u_next = c + 1 < nch &&
                             mbar_test_wait(&bar[B_FULLE0 + (s ^ 1)], ((c + 1) >> 1) & 1);
                    if (u_next) {
                        issue_u<NS>(tmem, sbase + (s ^ 1) * Cfg::STAGE,
                                    Cfg::TMB + (uint32_t)NS * (uint32_t)(s ^ 1));
                        TRACE(c + 1, 5);
                    }
                }
                __syncwarp();
                // K~^T U once U of chunk c is formed, then P U
                if (bar_any(BAR_U, 160, fail)) fail = true;
                if (leader) TRACE(c, 7);
                if (leader && !fail) {
                    if (!wait_chain(&bar[B_FULLL0 + s], (c >> 1) & 1, abort_flag, ST_MMA)) {
                        fail = true;
                    } else {
                        TRACE(c, 14);
                        tc_fence_after();
                        const uint32_t ut = u_tile + Cfg::UT * (uint32_t)s;
                        issue_carry3<NS>(tmem, st, ut, tb);  // U~(c) is consumed
                        tc_commit(&bar[B_SDONE]);
                        TRACE(c, 9);
                        if (c + 1 < nch && !u_next) {
                            if (!wait_chain(&bar[B_FULLE0 + (s ^ 1)], ((c + 1) >> 1) & 1,
                                            abort_flag, ST_MMA))
                                fail = true;
                            else
                                issue_u<NS>(tmem, sbase + (s ^ 1) * Cfg::STAGE,
                                            Cfg::TMB + (uint32_t)NS * (uint32_t)(s ^ 1));
                            TRACE(c + 1, 5);
                        }
                        issue_carry2<NS>(tmem, st, ut, Cfg::TMC + (uint32_t)NS * (uint32_t)s);
                        tc_commit(&bar[B_CDONE]);
                        tc_commit(&bar[B_EMPTYL0 + s]);  // the late group of chunk c is read
                        TRACE(c, 4);
                        if (!fail) done = c + 1;
                    }
                }
                __syncwarp();
            }
            // the SIMT warps' last BAR_S (after the state update of the last chunk)
            if (!stopped) bar_any(BAR_S, 288, fail);
            ok = !fail;
        } else {
            // the initial state tile is written: BAR_S #0
            handoff();
            bool stop = bar_any(BAR_S, 288, false);
            for (int c = 0; c < nch && !stop; ++c) {
                const int s = c & 1;
                const uint32_t ta = Cfg::TMA + (uint32_t)NS * (uint32_t)s;
                const uint32_t tb = Cfg::TMB + (uint32_t)NS * (uint32_t)s;
                if (q >= 2) {
                    // the output of chunk c-1, once its P U is complete
                    if (c > 0) {
                        if (!wait_chain(&bar[B_CDONE], (c - 1) & 1, abort_flag, ST_CARRY)) fail = true;
                        warp_fail();
                        if (!fail) {
                            tc_fence_after();
                            write_out(c - 1, gsc_prev);
                        }
                    }
                    if (lane == 0 && warp == 6) TRACE(c, 17);
                } else {
                    if (!wait_chain(&bar[B_ADONE], c & 1, abort_flag, ST_CARRY)) fail = true;
                    warp_fail();
                    if (!fail) {
                        if (lane == 0) TRACE(c, 30 + (warp & 1) + ((warp >> 2) - 1) * 2);
                        tc_fence_after();
                        // U = U~ - W S0 for token L
                        const uint32_t ut = u_tile + Cfg::UT * (uint32_t)s;
#pragma unroll
                        for (int p = 0; p < NP; ++p) {
                            float ws[32], uv[32];
                            tmem_ld32x2(tmem + lane_off + ta + 32 * p,
                                        tmem + lane_off + tb + 32 * p, ws, uv);
                            uint32_t u[16];
#pragma unroll
                            for (int j = 0; j < 16; ++j)
                                u[j] = pack_bf16(uv[2 * j] - ws[2 * j],
                                                 uv[2 * j + 1] - ws[2 * j + 1]);
                            write_row32_packed(ut + 8192u * pblk(p), L, pch(p), u);
                        }
                        if (lane == 0) TRACE(c, 34 + (warp & 1) + ((warp >> 2) - 1) * 2);
                    }
                    handoff();
                    if (warp == 4 && lane == 0) TRACE(c, 48);
                    if (bar_any(BAR_U, 160, fail)) fail = true;
                    if (warp == 4 && lane == 0) TRACE(c, 49);
                }
                // S1 = Gamma_last S0 + K~^T U for state row L (the late group, with the
                // scalars, landed before K~^T U was issued and is reloaded only after P U)
                if (!fail && !(wait_chain(&bar[B_SDONE], c & 1, abort_flag, ST_CARRY) &&
                               wait_chain(&bar[B_FULLL0 + s], (c >> 1) & 1, abort_flag,
                                          ST_CARRY)))
                    fail = true;
                warp_fail();
                if (!fail) {
                    if (warp == 4 && lane == 0) TRACE(c, 15);
                    tc_fence_after();
                    const float Gl = scal[s].Gl;
                    if (q >= 2) gsc_prev = a.scale * scal[s].Gam[L - 64];
#pragma unroll
                    for (int p = 0; p < NP; ++p) {
                        float d[32];
                        tmem_ld32(tmem + lane_off + tb + 32 * p, d);
#pragma unroll
                        for (int j = 0; j < 32; ++j)
                            Sr[32 * p + j] = fmaf(Gl, Sr[32 * p + j], d[j]);
                        write_row32(s_base + 16384u * pblk(p), L, pch(p), Sr + 32 * p);
                    }
                    if (lane == 0) TRACE(c, 38 + warp - 4);
                }
                handoff();
                if (warp == 4 && lane == 0) TRACE(c, 50);
                stop = bar_any(BAR_S, 288, fail);
                if (warp == 4 && lane == 0) TRACE(c, 51);
                if (!fail) done = c + 1;
            }
            ok = !fail;
        }
        // every role of the carry group decides the epilogue together (lanes 1-31 of the
        // issuer warp only take part in this barrier)
        if ((leader || !issuer) && (!ok || done < nch) && !*abort_flag)
            record_failure(abort_flag, ST_CARRY);
        bar_sync(1, 288);
        ok = __all_sync(0xffffffffu, !*abort_flag);
        if (ok && !issuer && q >= 2) {
            // the output of the last chunk
            ok = __all_sync(0xffffffffu,
                            wait_chain(&bar[B_CDONE], (nch - 1) & 1, abort_flag, ST_CARRY));
            if (ok) {
                tc_fence_after();
                write_out(nch - 1, gsc_prev);
            }
        }
        if (ok && !issuer) {
#pragma unroll
            for (int j = 0; j < CPT; j += 4)
                *reinterpret_cast<float4*>(gstate + j) =
                    make_float4(Sr[j], Sr[j + 1], Sr[j + 2], Sr[j + 3]);
        }
        // no MMA of the carry may be in flight when TMEM is freed
        if (leader && mmas) {
            tc_commit(&bar[B_DRAIN]);
            mbar_wait_bounded(&bar[B_DRAIN], 0, kWaitNs);
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, Cfg::TMCOLS);
    }
    SPAN_END(a.c0 == 0 ? 1 : 3);
}

// ---------------------------------------------------------------- transposed carry

// carry_t_kernel: one CTA per (value head, sequence) over all 128 state columns, with the
// chunk recurrence written transposed, so that every operand the SIMT warps produce in a
// chunk stays in tensor memory and enters the next MMA as its A operand:
//   U~^T = V^T T_U^T,   [(W S0)^T | (Q S0)^T] = S0^T [W; Q]^T,   U^T = U~^T - (W S0)^T,
//   U'^T = U^T diag(exp(gamma_last - gamma)),   dS^T = U'^T K,
//   S1^T = Gamma_last S0^T + dS^T,   O^T = (Q S0)^T diag(Gamma) + U^T P^T.
// TMEM lanes are the value columns v of the state, so the U step and the state update
// run on all four SM sub-partitions, and no hand-off goes through shared memory.
// Warp 0: producer (carry_produce<128>, both 64-column V blocks); warp 1 (one thread):
// every MMA, in the order that keeps the tensor pipe free for the chain: dS^T(c), then
// U~(c+1) (runs during the state update), then [W; Q] S0 of chunk c+1 and U^T P^T(c)
// (both complete before the next U step rewrites U^T); warps 2..9: SIMT,
// warp (q = warp % 4, g = (warp - 2) / 4) owning lane v = 32 q + lane, fp32 state rows
// 64 g .. 64 g + 63 (registers) and tokens 32 g .. 32 g + 31 of U and of the output.
struct CarryT {
    static constexpr uint32_t STAGE = CarryCfg<128>::STAGE;
    static constexpr uint32_t SCAL = 2 * STAGE;
    static constexpr uint32_t BAR = SCAL + 2 * sizeof(CarryScalars);
    static constexpr uint32_t MISC = BAR + 128;
    static constexpr uint32_t SMEM = MISC + 64 + 1024;
    // TMEM (32-bit columns): per chunk parity p, from 192 p: U~^T (64) | (W S0)^T (64) |
    // O^T (64); once U is formed the state increment dS^T takes the first 128 columns.
    // Then the bf16 operands S0^T (128 x 128: 64 columns), U^T and U'^T (128 x 64: 32
    // columns each).
    static constexpr uint32_t UB = 0, WSC = 64, OQ = 128, PSTRIDE = 192;
    static constexpr uint32_t S0T = 384, UT = 448, UPT = 480, TMCOLS = 512;
    static_assert(SCAL % 16 == 0 && BAR % 8 == 0, "alignment");
    static_assert(SMEM <= 232448, "shared memory budget");
};
constexpr int CARRY_T_THREADS = 320;
// barriers 0..7 are the ring's (B_FULLE0 .. B_EMPTYL1)
enum { T_ADONE = B_EMPTYL1 + 1, T_SDONE, T_ODONE0, T_ODONE1, T_DRAIN, T_COUNT };
static_assert(T_COUNT * 8 <= 128, "barrier block");
static_assert(CarryT::OQ == CarryT::WSC + 64 && OFF_Q == OFF_W + 8192,
              "(W S0)^T and (Q S0)^T come from one 128-row operand into adjacent columns");

// U~^T = V^T T_U^T over the 64 tokens (V read M-major, T_U as K-major B), into `d`
__device__ __forceinline__ void issue_t_u(uint32_t tmem, uint32_t st, uint32_t d) {
    constexpr uint32_t id = idesc_bf16(128, 64, true, false);
    const uint64_t av = smem_desc_sw128(st + OFF_V, 8192, 1024);
    const uint64_t bt = smem_desc_sw128(st + CarryCfg<128>::OFF_TU, 16, 1024);
#pragma unroll
    for (int k = 0; k < 4; ++k) mma_bf16(tmem + d, dadd(av, k * 2048), dadd(bt, k * 32), id, k > 0);
}

// [(W S0)^T | (Q S0)^T] = S0^T [W; Q]^T over Dk = 128 ([W_b; Q_b] is one 128-row
// K-major operand per 64-column block), S0^T the A operand in TMEM; 128 columns at `d`
__device__ __forceinline__ void issue_t_s0(uint32_t tmem, uint32_t d, uint32_t st) {
    constexpr uint32_t id = idesc_bf16(128, 128, false, false);
    const uint64_t b0 = smem_desc_sw128(st + OFF_W, 16, 1024);
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        const uint32_t off = (uint32_t)(k >> 2) * BLK_STRIDE + (uint32_t)(k & 3) * 32u;
        mma_bf16_ts(tmem + d, tmem + CarryT::S0T + 8u * (uint32_t)k, dadd(b0, off), id, k > 0);
    }
}

// dS^T = U'^T K over the tokens (U'^T in TMEM at `ut`, K read N-major), 128 columns at `d`
__device__ __forceinline__ void issue_t_ds(uint32_t tmem, uint32_t d, uint32_t ut, uint32_t st) {
    constexpr uint32_t id = idesc_bf16(128, 128, false, true);
    const uint64_t bk = smem_desc_sw128(st + OFF_K, BLK_STRIDE, 1024);
#pragma unroll
    for (int k = 0; k < 4; ++k)
        mma_bf16_ts(tmem + d, tmem + ut + 8u * (uint32_t)k, dadd(bk, k * 2048), id, k > 0);
}

// O^T += U^T P^T (U^T at `ut`, P as K-major B), onto (Q S0)^T diag(Gamma) at `d`
__device__ __forceinline__ void issue_t_o(uint32_t tmem, uint32_t d, uint32_t ut, uint32_t st) {
    constexpr uint32_t id = idesc_bf16(128, 64, false, false);
    const uint64_t bp = smem_desc_sw128(st + OFF_P, 16, 1024);
#pragma unroll
    for (int k = 0; k < 4; ++k)
        mma_bf16_ts(tmem + d, tmem + ut + 8u * (uint32_t)k, dadd(bp, k * 32), id, 1);
}

__global__ void __launch_bounds__(CARRY_T_THREADS, 1)
    carry_t_kernel(const __grid_constant__ CUtensorMap mq, const __grid_constant__ CUtensorMap mk,
                   const __grid_constant__ CUtensorMap mv, TcArgs a) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const uint32_t sbase = smem_u32(sm);
    uint64_t* bar = reinterpret_cast<uint64_t*>(sm + CarryT::BAR);
    uint32_t* misc = reinterpret_cast<uint32_t*>(sm + CarryT::MISC);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(misc + 1);
    CarryScalars* scal = reinterpret_cast<CarryScalars*>(sm + CarryT::SCAL);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int h = blockIdx.y;
    const int S = a.S;
    // the sequence of this CTA, as in carry_tc_kernel
    int wb, u0, nch, tbase, tend, sb;
    if (a.cu == nullptr) {
        wb = blockIdx.z, u0 = 0, nch = a.nseg, tbase = a.c0 * C, tend = S;
        sb = blockIdx.z * a.Hv + h;
    } else {
        const int n = blockIdx.z;
        wb = 0, u0 = a.cb[n], nch = a.cb[n + 1] - a.cb[n], tbase = a.cu[n], tend = a.cu[n + 1];
        sb = n * a.Hv + h;
    }
    if (nch == 0) {
        grid_dep_wait();
        if (!a.state_is_input)
            for (int i = tid; i < 128 * 128; i += CARRY_T_THREADS)
                a.state[(size_t)sb * 128 * 128 + i] = 0.f;
        return;
    }
    const int zo = wb * a.Hv + h;  // head row of v and out

    if (tid == 0) {
        for (int i = 0; i < T_COUNT; ++i) mbar_init(&bar[i], 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(misc, CarryT::TMCOLS);
        tmem_relinquish();
    }
    if (tid == 32) {
        prefetch_tensormap(&mq);
        prefetch_tensormap(&mk);
        prefetch_tensormap(&mv);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = misc[0];

    if (warp == 0) {
        if (lane == 0) {
            carry_produce<128>(sm, bar, scal, &mq, &mk, &mv, false, a.ws_wait != 0,
                               a.ws + ws_offset(wb, h, u0, a.Hv, a.nseg), nch, 0, tbase,
                               wb * a.Hk + h / (a.Hv / a.Hk), zo, abort_flag);
        }
    } else {
        const bool issuer = warp == 1;
        const bool leader = issuer && lane == 0;
        const int q = warp & 3, g = (warp - 2) >> 2;
        const int v = 32 * q + lane;
        const uint32_t lo = (uint32_t)(32 * q) << 16;
        float* gst = a.state + ((size_t)sb * 128 + (size_t)(64 * g)) * 128 + v;
        __nv_bfloat16* gout = a.out + (size_t)zo * S * 128;

        float Sr[64];
        // the bf16 copy of this thread's state rows, as the A operand S0^T
        auto put_state = [&]() {
            uint32_t w[32];
#pragma unroll
            for (int j = 0; j < 32; ++j) w[j] = pack_bf16(Sr[2 * j], Sr[2 * j + 1]);
            tmem_st32u(tmem + lo + CarryT::S0T + 32u * (uint32_t)g, w);
            tmem_wait_st();
        };
        // out = scale O of chunk cc for tokens 32 g .. 32 g + 31 (below tend) of column v,
        // straight from the registers: for each token a warp writes 64 contiguous bytes
        auto store_out = [&](int cc) {
            const int t0 = tbase + cc * C + 32 * g;
            float o[32];
            tmem_ld32(tmem + lo + CarryT::PSTRIDE * (uint32_t)(cc & 1) + CarryT::OQ +
                          32u * (uint32_t)g,
                      o);
            unsigned short* dst = reinterpret_cast<unsigned short*>(gout) + (size_t)t0 * 128 + v;
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                const uint32_t w = pack_bf16(a.scale * o[2 * j], a.scale * o[2 * j + 1]);
                if (t0 + 2 * j < tend) dst[(size_t)(2 * j) * 128] = (unsigned short)(w & 0xffffu);
                if (t0 + 2 * j + 1 < tend) dst[(size_t)(2 * j + 1) * 128] = (unsigned short)(w >> 16);
            }
        };
        // U~ of chunk cc into its parity's columns; ADONE of chunk cc covers it
        auto issue_next_u = [&](int cc) -> bool {
            const int sc = cc & 1;
            if (!wait_or_abort(&bar[B_FULLE0 + sc], (cc >> 1) & 1, abort_flag, ST_MMA)) return false;
            tc_fence_after();
            issue_t_u(tmem, sbase + (uint32_t)sc * CarryT::STAGE,
                      CarryT::PSTRIDE * (uint32_t)sc + CarryT::UB);
            return true;
        };
        // [(W S0)^T | (Q S0)^T] of chunk cc from the state just published; its columns held
        // dS^T and O^T of chunk cc-2, both read by now
        auto issue_next_s0 = [&](int cc) {
            const int sc = cc & 1;
            TCLK(t12);
            tc_fence_after();
            issue_t_s0(tmem, CarryT::PSTRIDE * (uint32_t)sc + CarryT::WSC,
                       sbase + (uint32_t)sc * CarryT::STAGE);
            TCLK(t3);
            TPUT(cc, 12, t12);
            TPUT(cc, 3, t3);
        };

        // The chain hand-offs are named barriers of the SIMT warps and the issuer warp
        // (288 threads): barrier 3 when U^T is in TMEM (SIMT warps arrive, the issuer
        // waits), barrier 4 when the state is (a full barrier that also votes on stopping,
        // so the group leaves the loop as one). Every participant reaches both barriers in
        // every chunk: a failed wait only skips work.
        if (!issuer) {
            grid_dep_wait();  // the carry of the segment before wrote this state
            if (a.state_is_input) {
#pragma unroll
                for (int i = 0; i < 64; ++i) Sr[i] = gst[(size_t)i * 128];
            } else {
#pragma unroll
                for (int i = 0; i < 64; ++i) Sr[i] = 0.f;
            }
            put_state();
            tc_fence_before();
        }
        bool ok = true;
        int done = 0;
        if (leader) ok = issue_next_u(0);
        __syncwarp();
        bool stop = bar_any(4, 288, !ok || *abort_flag);
        if (leader && !stop) {
            issue_next_s0(0);
            tc_commit(&bar[T_ADONE]);
            tc_commit(&bar[B_EMPTYE0]);
        }
        for (int c = 0; !stop && c < nch; ++c) {
            const int s = c & 1;
            const uint32_t pb = CarryT::PSTRIDE * (uint32_t)s;
            const uint32_t st = sbase + (uint32_t)s * CarryT::STAGE;
            if (!issuer) {
                // the late group's scalars are read before barrier 4: it is reloaded only
                // after U^T P^T of the chunk, issued after that barrier
                ok = ok && wait_or_abort(&bar[B_FULLL0 + s], (c >> 1) & 1, abort_flag, ST_CARRY);
                const float Gl = ok ? scal[s].Gl : 0.f;
                // U^T = U~^T - (W S0)^T and U'^T = U^T diag(exp(gamma_last - gamma)) for
                // tokens 32 g .. 32 g + 31; ADONE(c) also covers U~(c) and U^T P^T of chunk
                // c-1, the last reader of U^T
                ok = ok && wait_hot(&bar[T_ADONE], c & 1, abort_flag, ST_CARRY);
                if (tid == 64) TRACE(c, 13);
                if (ok) {
                    tc_fence_after();
                    float ws[32], uv[32];
                    tmem_ld32x2(tmem + lo + pb + CarryT::WSC + 32u * (uint32_t)g,
                                tmem + lo + pb + CarryT::UB + 32u * (uint32_t)g, ws, uv);
                    const float4* kd4 = reinterpret_cast<const float4*>(scal[s].kdec + 32 * g);
                    uint32_t u[16], u2[16];
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        const float4 kd = kd4[j];
                        const float d0 = uv[4 * j] - ws[4 * j], d1 = uv[4 * j + 1] - ws[4 * j + 1];
                        const float d2 = uv[4 * j + 2] - ws[4 * j + 2];
                        const float d3 = uv[4 * j + 3] - ws[4 * j + 3];
                        u[2 * j] = pack_bf16(d0, d1);
                        u[2 * j + 1] = pack_bf16(d2, d3);
                        u2[2 * j] = pack_bf16(kd.x * d0, kd.y * d1);
                        u2[2 * j + 1] = pack_bf16(kd.z * d2, kd.w * d3);
                    }
                    tmem_st16u(tmem + lo + CarryT::UT + 16u * (uint32_t)g, u);
                    tmem_st16u(tmem + lo + CarryT::UPT + 16u * (uint32_t)g, u2);
                    tmem_wait_st();
                }
                if (lane == 0) TRACE(c, 20 + (warp - 2));
                tc_fence_before();
                __syncwarp();
                bar_arrive(3, 288);
                // while dS^T(c) runs: (Q S0)^T(c) diag(Gamma) in place, before U^T P^T(c)
                // accumulates onto it after barrier 4, and the output of chunk c-1
                if (ok) {
                    const uint32_t oq = tmem + lo + pb + CarryT::OQ + 32u * (uint32_t)g;
                    const float4* gm4 = reinterpret_cast<const float4*>(scal[s].Gam + 32 * g);
                    float o[32];
                    tmem_ld32(oq, o);
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        const float4 gm = gm4[j];
                        o[4 * j] *= gm.x;
                        o[4 * j + 1] *= gm.y;
                        o[4 * j + 2] *= gm.z;
                        o[4 * j + 3] *= gm.w;
                    }
                    tmem_st32(oq, o);
                    tmem_wait_st();
                }
                if (c > 0) {
                    ok = ok && wait_hot(&bar[T_ODONE0 + (s ^ 1)], ((c - 1) >> 1) & 1, abort_flag,
                                        ST_CARRY);
                    if (ok) {
                        tc_fence_after();
                        store_out(c - 1);
                    }
                }
                if (tid == 64) TRACE(c, 17);
                // S1^T = Gamma_last S0^T + dS^T for rows 64 g .. 64 g + 63 of column v
                ok = ok && wait_hot(&bar[T_SDONE], c & 1, abort_flag, ST_CARRY);
                if (tid == 64) TRACE(c, 15);
                if (ok) {
                    tc_fence_after();
                    float d0[32], d1[32];
                    tmem_ld32x2(tmem + lo + pb + 64u * (uint32_t)g,
                                tmem + lo + pb + 64u * (uint32_t)g + 32u, d0, d1);
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        Sr[j] = fmaf(Gl, Sr[j], d0[j]);
                        Sr[32 + j] = fmaf(Gl, Sr[32 + j], d1[j]);
                    }
                    put_state();
                }
                if (lane == 0) TRACE(c, 28 + (warp - 2));
                tc_fence_before();
                if (tid == 64) TRACE(c, 18);
                __syncwarp();
            } else {
                bar_sync(3, 288);
                if (leader) {
                    // dS^T(c) into [U~^T | (W S0)^T] of this parity (read by now), then
                    // U~(c+1) into the other parity, whose columns last held dS^T(c-1)
                    TCLK(t7);
                    TPUT(c, 7, t7);
                    ok = ok && wait_or_abort(&bar[B_FULLL0 + s], (c >> 1) & 1, abort_flag, ST_MMA);
                    if (ok) {
                        TCLK(t14);
                        tc_fence_after();
                        issue_t_ds(tmem, pb, CarryT::UPT, st);
                        tc_commit(&bar[T_SDONE]);
                        TCLK(t9);
                        TPUT(c, 14, t14);
                        TPUT(c, 9, t9);
                        if (c + 1 < nch) ok = issue_next_u(c + 1);
                        TCLK(t8);
                        TPUT(c, 8, t8);
                    }
                }
                __syncwarp();
            }
            stop = bar_any(4, 288, !ok || *abort_flag);
            if (stop) break;
            if (leader) {
                // [W; Q] S0 of chunk c+1, then O^T(c) += U^T P^T behind it in the pipe; the
                // next ADONE covers both, so the next U step finds U^T free
                if (c + 1 < nch) issue_next_s0(c + 1);
                TCLK(t4);
                issue_t_o(tmem, pb + CarryT::OQ, CarryT::UT, st);
                if (c + 1 < nch) {
                    tc_commit(&bar[T_ADONE]);
                    tc_commit(&bar[B_EMPTYE0 + (s ^ 1)]);  // W, Q, V, T_U of chunk c+1 are read
                }
                tc_commit(&bar[T_ODONE0 + s]);
                tc_commit(&bar[B_EMPTYL0 + s]);  // K, P, scalars of chunk c are read
                TPUT(c, 4, t4);
            }
            __syncwarp();
            done = c + 1;
        }
        // every role decides the epilogue together (lanes 1-31 of the issuer warp only
        // take part in this barrier)
        if ((leader || !issuer) && (!ok || done < nch) && !*abort_flag)
            record_failure(abort_flag, ST_CARRY);
        __syncwarp();
        bar_sync(1, 288);
        ok = !*abort_flag;
        if (!issuer) {
            // the output of the last chunk, then the state
            const int cl = nch - 1;
            if (ok) ok = wait_hot(&bar[T_ODONE0 + (cl & 1)], (cl >> 1) & 1, abort_flag, ST_CARRY);
            if (ok) {
                tc_fence_after();
                store_out(cl);
#pragma unroll
                for (int i = 0; i < 64; ++i) gst[(size_t)i * 128] = Sr[i];
            }
        }
        // no MMA may be in flight when TMEM is freed
        if (leader) {
            tc_commit(&bar[T_DRAIN]);
            mbar_wait_bounded(&bar[T_DRAIN], 0, kWaitNs);
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, CarryT::TMCOLS);
    }
}

// ---------------------------------------------------------------- variable-length batch

// One CTA: table[0..N] = chunk bases of the sequences cu[n] .. cu[n+1] - 1 in 64-token
// chunks (block-wide scan in tiles of 1024), table[N+1] = 1. A malformed cu (cu[0] != 0,
// a decreasing step or cu[N] > S) zeroes the table -- every sequence then counts as
// empty -- and sets the status bit instead.
__global__ void __launch_bounds__(1024) varlen_setup_kernel(const int* cu, int N, int S,
                                                            int* table) {
    __shared__ int wsum[32];
    __shared__ int carry, bad;
    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
    if (tid == 0) {
        carry = 0;
        bad = (cu[0] != 0 || cu[N] > S) ? 1 : 0;
        table[0] = 0;
    }
    __syncthreads();
    for (int base = 0; base < N; base += 1024) {
        const int n = base + tid;
        int x = 0;
        if (n < N) {
            const int len = cu[n + 1] - cu[n];
            if (len < 0) atomicOr(&bad, 1);
            x = len > 0 ? (len + C - 1) / C : 0;
        }
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, x, off);
            if (lane >= off) x += y;
        }
        if (lane == 31) wsum[w] = x;
        __syncthreads();
        if (w == 0) {
            int v = wsum[lane];
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, v, off);
                if (lane >= off) v += y;
            }
            wsum[lane] = v;
        }
        __syncthreads();
        const int incl = x + (w > 0 ? wsum[w - 1] : 0);
        if (n < N) table[n + 1] = carry + incl;
        __syncthreads();
        if (tid == 1023) carry += incl;
        __syncthreads();
    }
    if (bad) {
        for (int n = tid; n <= N + 1; n += 1024) table[n] = 0;
        if (tid == 0) atomicOr(&g_tc_status, kStatusBadSeqlens);
    } else if (tid == 0) {
        table[N + 1] = 1;
    }
}

// ---------------------------------------------------------------- host side

}  // namespace

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

namespace {

// 3-D bf16 map over [z][y][x] = [heads][S][128], box 64 x 64 x 1, 128-byte swizzle.
bool encode_3d(CUtensorMap* m, const void* base, int S, int heads) {
    auto fn = tensor_map_encoder();
    if (!fn) return false;
    cuuint64_t dims[3] = {128, (cuuint64_t)S, (cuuint64_t)heads};
    cuuint64_t strides[2] = {128 * 2, (cuuint64_t)S * 128 * 2};
    cuuint32_t box[3] = {64, 64, 1};
    cuuint32_t es[3] = {1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box,
              es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool prefill_tc_supported(const PrefillArgs& a, bool bf16) {
    return bf16 && a.Dk == 128 && a.Dv == 128 && a.S > 0;
}

size_t prefill_tc_workspace_bytes(int B, int Hv, int S) {
    const size_t nch = ((size_t)S + C - 1) / C;
    return (size_t)B * (size_t)Hv * nch * WS_UNIT;
}

size_t prefill_tc_unit_bytes() { return WS_UNIT; }

namespace {
size_t varlen_units_bytes(int N, int Hv, int S) {
    const size_t nmax = ((size_t)S + C - 1) / C + (size_t)N;
    return ((size_t)Hv * nmax * WS_UNIT + 255) / 256 * 256;
}
}  // namespace

size_t prefill_tc_varlen_workspace_bytes(int N, int Hv, int S) {
    return varlen_units_bytes(N, Hv, S) + varlen_table_ints(N) * sizeof(int);
}

cudaError_t launch_varlen_setup(const PrefillArgs& a, cudaStream_t stream) {
    varlen_setup_kernel<<<1, 1024, 0, stream>>>(a.cu_seqlens, a.N, a.S, a.table);
    return cudaGetLastError();
}

namespace {

// The two kernels of one segment of the sequence (chunks c0 .. c0 + nseg - 1), whose
// B Hv nseg workspace units start at `ws`.
struct SegmentLaunch {
    CUtensorMap mq, mk, mv;
    const PrefillArgs* a;
    int sms;

    TcArgs args(int c0, int nseg, uint8_t* ws, bool ws_wait = false) const {
        const int sin = (c0 > 0 || a->state_is_input) ? 1 : 0;
        return TcArgs{a->g,     a->beta, a->scale, a->B, a->Hk,  a->Hv,
                      a->S,     c0,      nseg,     a->state, sin,
                      static_cast<__nv_bfloat16*>(a->out), ws, a->cu_seqlens, a->table, a->N,
                      split() ? 1 : 0, ws_wait ? 1 : 0};
    }
    // sequences of the carry grid: the batch, or the variable-length batch's sequences
    int rows() const { return a->cu_seqlens ? a->N : a->B; }
    // A one-segment call's carry runs as a programmatic dependent of its prep (same stream)
    // when it is the two-slice carry: the B=2 Hk=4 Hv=8 S=1024 call took 37.5 us against
    // 39.6. The transposed carry (256 CTAs of the B=8 S=4096 call) and the overlapped
    // schedule's first carry measured slower that way (499 against 482 us; 235.5 against
    // 223.2 us for the layer call), so they follow their prep as plain stream successors.
    bool prep_pdl() const { return split(); }
    // two carry CTAs per head (64-column state slices) while that still fits the GPU in
    // one wave, else one transposed CTA per head
    bool split() const { return kCarrySplit && 2 * rows() * a->Hv <= sms; }

    cudaError_t prep(int c0, int nseg, uint8_t* ws, cudaStream_t st) const {
        prep_tc_kernel<<<dim3(nseg, a->Hv, a->B), PREP_THREADS, PREP_SMEM, st>>>(
            mq, mk, args(c0, nseg, ws));
        return cudaGetLastError();
    }
    // pdl: launched as a programmatic dependent of the previous kernel in `st`, which lets
    // its setup run before that one ends: the carry of the segment before (which wrote the
    // state), or with after_prep the prep that wrote its workspace (the producer then waits
    // for that grid before its first copy)
    cudaError_t carry(int c0, int nseg, uint8_t* ws, cudaStream_t st, bool pdl = false,
                      bool after_prep = false) const {
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cudaLaunchConfig_t cfg = {};
        cfg.stream = st;
        cfg.attrs = attr;
        cfg.numAttrs = (pdl || after_prep) ? 1 : 0;
        const TcArgs ta = args(c0, nseg, ws, after_prep);
        if (split()) {
            cfg.gridDim = dim3(2, a->Hv, rows());
            cfg.blockDim = dim3(CARRY_THREADS);
            cfg.dynamicSmemBytes = CarryCfg<64>::SMEM;
            return cudaLaunchKernelEx(&cfg, carry_tc_kernel<64>, mq, mk, mv, ta);
        }
        cfg.gridDim = dim3(1, a->Hv, rows());
        cfg.blockDim = dim3(CARRY_T_THREADS);
        cfg.dynamicSmemBytes = CarryT::SMEM;
        return cudaLaunchKernelEx(&cfg, carry_t_kernel, mq, mk, mv, ta);
    }
};

cudaError_t set_attributes() {
    static cudaError_t e = [] {
        cudaError_t r = cudaFuncSetAttribute(
            prep_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)PREP_SMEM);
        if (r == cudaSuccess)
            r = cudaFuncSetAttribute(carry_tc_kernel<64>,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)CarryCfg<64>::SMEM);
        if (r == cudaSuccess)
            r = cudaFuncSetAttribute(carry_t_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)CarryT::SMEM);

        return r;
    }();
    return e;
}

// Per-device streams and events of the overlapped schedule: the prep kernels run on a
// low-priority stream, the carry kernels on a high-priority one, both forked from and
// joined back to the caller's stream with events.
struct Overlap {
    std::mutex mu;
    bool ready = false;
    cudaStream_t prep = nullptr, carry = nullptr;
    cudaEvent_t fork = nullptr, prepped = nullptr, joined = nullptr;
};

Overlap* overlap_for(int dev) {
    constexpr int kMaxDevices = 64;
    static Overlap tab[kMaxDevices];
    return (dev >= 0 && dev < kMaxDevices) ? &tab[dev] : nullptr;
}

cudaError_t overlap_init(Overlap& o) {
    if (o.ready) return cudaSuccess;
    int least = 0, greatest = 0;
    cudaError_t e = cudaDeviceGetStreamPriorityRange(&least, &greatest);
    if (e == cudaSuccess) e = cudaStreamCreateWithPriority(&o.prep, cudaStreamNonBlocking, least);
    if (e == cudaSuccess)
        e = cudaStreamCreateWithPriority(&o.carry, cudaStreamNonBlocking, greatest);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&o.fork, cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&o.prepped, cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&o.joined, cudaEventDisableTiming);
    o.ready = e == cudaSuccess;
    return e;
}

cudaError_t prepare(SegmentLaunch& L, const PrefillArgs& a) {
    L.a = &a;
    if (!encode_3d(&L.mq, a.q, a.S, a.B * a.Hk) || !encode_3d(&L.mk, a.k, a.S, a.B * a.Hk) ||
        !encode_3d(&L.mv, a.v, a.S, a.B * a.Hv))
        return cudaErrorInvalidValue;
    cudaError_t e = set_attributes();
    if (e != cudaSuccess) return e;
    int dev = 0;
    e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&L.sms, cudaDevAttrMultiProcessorCount, dev);
    return e;
}

}  // namespace

int prefill_tc_schedule(int B, int Hv, int nch, int sms, int* sizes, int max_segments) {
    // The carry of a segment occupies B Hv or 2 B Hv SMs (one CTA each) for the whole
    // segment; the prep of the next segment runs meanwhile on the SMs left over. Without
    // enough of those, or with too few chunks, one segment.
    const int carry_sms = (kCarrySplit && 2 * B * Hv <= sms ? 2 : 1) * B * Hv;
    int g = std::min(std::min(kOverlapSegments, max_segments), nch / kMinSegmentChunks);
    if (carry_sms > sms || sms - carry_sms < sms / 4 || g < 2) g = 1;
    if (g == 1) {
        sizes[0] = nch;
        return 1;
    }
    // sizes s_k = s_1 r^k, sum nch: s_1 = nch (r - 1) / (r^g - 1)
    const double r = kSegmentGrowthPermille / 1000.0;
    double rg = 1.0;
    for (int k = 0; k < g; ++k) rg *= r;
    const double s1 = (double)nch * (r - 1.0) / (rg - 1.0);
    int used = 0;
    double x = s1;
    for (int k = 0; k < g; ++k, x *= r) {
        const int left = g - 1 - k;  // segments after this one
        int n = k == g - 1 ? nch - used : (int)(x + 0.5);
        n = std::max(kMinSegmentChunks, std::min(n, nch - used - left * kMinSegmentChunks));
        sizes[k] = n;
        used += n;
    }
    return g;
}

cudaError_t launch_prefill_tc(const PrefillArgs& a, int c0, int nseg, cudaStream_t stream,
                              int* launched) {
    *launched = 0;
    if (a.workspace == nullptr || nseg < 1 ||
        a.workspace_bytes < (size_t)a.B * (size_t)a.Hv * (size_t)nseg * WS_UNIT)
        return cudaErrorInvalidValue;
    SegmentLaunch L{};
    cudaError_t e = prepare(L, a);
    if (e != cudaSuccess) return e;
    uint8_t* ws = static_cast<uint8_t*>(a.workspace);
    e = L.prep(c0, nseg, ws, stream);
    if (e != cudaSuccess) return e;
    *launched = 1;
    e = L.carry(c0, nseg, ws, stream, false, L.prep_pdl());
    if (e == cudaSuccess) *launched = 2;
    return e;
}

cudaError_t launch_prefill_tc_varlen(const PrefillArgs& a, cudaStream_t stream, int* launched) {
    *launched = 0;
    if (a.workspace == nullptr || a.cu_seqlens == nullptr || a.B != 1 ||
        a.workspace_bytes < prefill_tc_varlen_workspace_bytes(a.N, a.Hv, a.S))
        return cudaErrorInvalidValue;
    PrefillArgs v = a;
    v.table = reinterpret_cast<int*>(static_cast<uint8_t*>(a.workspace) +
                                     varlen_units_bytes(a.N, a.Hv, a.S));
    SegmentLaunch L{};
    cudaError_t e = prepare(L, v);
    if (e != cudaSuccess) return e;
    e = launch_varlen_setup(v, stream);
    if (e != cudaSuccess) return e;
    *launched = 1;
    // the prep grid covers the chunk bound ceil(S/64) + N; CTAs past the last chunk leave
    const int nmax = (a.S + C - 1) / C + a.N;
    uint8_t* ws = static_cast<uint8_t*>(a.workspace);
    e = L.prep(0, nmax, ws, stream);
    if (e != cudaSuccess) return e;
    *launched = 2;
    e = L.carry(0, nmax, ws, stream, false, L.prep_pdl());
    if (e == cudaSuccess) *launched = 3;
    return e;
}

cudaError_t launch_prefill_tc_overlapped(const PrefillArgs& a, cudaStream_t stream,
                                         int* launched) {
    *launched = 0;
    const int nch = (a.S + C - 1) / C;
    if (a.workspace == nullptr || nch < 1 ||
        a.workspace_bytes < (size_t)a.B * (size_t)a.Hv * (size_t)nch * WS_UNIT)
        return cudaErrorInvalidValue;
    SegmentLaunch L{};
    cudaError_t e = prepare(L, a);
    if (e != cudaSuccess) return e;
    int dev = 0;
    cudaGetDevice(&dev);
    int sizes[kMaxSegments];
    const int g = prefill_tc_schedule(a.B, a.Hv, nch, L.sms, sizes, kMaxSegments);
    Overlap* o = overlap_for(dev);
    uint8_t* ws = static_cast<uint8_t*>(a.workspace);
    if (g == 1 || o == nullptr) {
        e = L.prep(0, nch, ws, stream);
        if (e != cudaSuccess) return e;
        *launched = 1;
        e = L.carry(0, nch, ws, stream, false, L.prep_pdl());
        if (e == cudaSuccess) *launched = 2;
        return e;
    }
    std::lock_guard<std::mutex> lock(o->mu);
    e = overlap_init(*o);
    if (e != cudaSuccess) return e;
    // fork: both helper streams start after the caller's earlier work
    e = cudaEventRecord(o->fork, stream);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(o->prep, o->fork, 0);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(o->carry, o->fork, 0);
    if (e != cudaSuccess) return e;
    // prep of segment j+1 overlaps the carry of segment j; each carry waits for its prep
    // (a wait takes the event's latest record at the time it is enqueued). The first
    // segment's prep runs on the carry stream, right before its carry (no event between
    // them: 223 us per layer call against 237 with this prep on the prep stream), and the
    // other preps start once it is done; the carries of the later segments are programmatic
    // dependents of the carry before them and wait for their prep's event.
    cudaError_t le = cudaSuccess;
    for (int j = 0, c0 = 0; j < g && le == cudaSuccess; c0 += sizes[j], ++j) {
        const int n = sizes[j];
        uint8_t* wsj = ws + (size_t)a.B * (size_t)a.Hv * (size_t)c0 * WS_UNIT;
        if (j == 0) {
            le = L.prep(c0, n, wsj, o->carry);
            if (le != cudaSuccess) break;
            ++*launched;
            le = cudaEventRecord(o->fork, o->carry);
            if (le == cudaSuccess) le = cudaStreamWaitEvent(o->prep, o->fork, 0);
            if (le == cudaSuccess) le = L.carry(c0, n, wsj, o->carry);
        } else {
            le = L.prep(c0, n, wsj, o->prep);
            if (le != cudaSuccess) break;
            ++*launched;
            le = cudaEventRecord(o->prepped, o->prep);
            if (le == cudaSuccess) le = cudaStreamWaitEvent(o->carry, o->prepped, 0);
            if (le == cudaSuccess) le = L.carry(c0, n, wsj, o->carry, kCarryPdl);
        }
        if (le == cudaSuccess) ++*launched;
    }
    // join, also after a failed launch, so that no work is left outside the caller's stream
    e = cudaEventRecord(o->joined, o->carry);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(stream, o->joined, 0);
    return le != cudaSuccess ? le : e;
}

}  // namespace gdn

#ifdef GDN_TRACE
extern "C" int gdn_trace_read(unsigned long long* dst) {
    return cudaMemcpyFromSymbol(dst, gdn::g_trace, sizeof(gdn::g_trace)) == cudaSuccess ? 0 : 1;
}
extern "C" int gdn_trace_span_reset() {
    unsigned long long init[8][2];
    for (int i = 0; i < 8; ++i) init[i][0] = ~0ull, init[i][1] = 0;
    return cudaMemcpyToSymbol(gdn::g_span, init, sizeof(init)) == cudaSuccess ? 0 : 1;
}
extern "C" int gdn_trace_span_read(unsigned long long* dst) {
    return cudaMemcpyFromSymbol(dst, gdn::g_span, sizeof(gdn::g_span)) == cudaSuccess ? 0 : 1;
}
#endif
