// prefill_tc.cu -- chunked GDN prefill on the tcgen05 tensor cores: bf16 operands,
// fp32 accumulation in tensor memory (TMEM), fp32 state master in registers.
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
// One CTA per (batch, value head, 64-column slice of the state); the state's columns
// evolve independently, so slices never communicate. Per chunk, on the tensor cores:
//   Gram   [Q;K] K^T               -> QK^T, KK^T          (M128 N64  K128)
//   WY     [T_W;P] K, [T_U;T_W] V   -> W, U~               (M128 N128 K64, M128 N64 K64)
//   carry  [W;Q] S0                 -> W S0, Q S0          (M128 N64  K128)
//          [T_W;P] U                -> P U                 (M128 N64  K64)
//          K^T U'                   -> state increment     (M128 N64  K64)
// Stacking two 64-row operands into one 128-row operand fills the M = 128 data path;
// the half of a result that is not needed is ignored.
//
// Warp roles (14 warps): 0 = TMA producer, which also computes the chunk's decay tables
// from g and beta; 1 = MMA issuer (one thread, carry MMAs first); 2-5 = carry (fp32
// state master, U, output, state update); 6-13 = prep (P and A from the Gram matrices,
// the (I+A)^-1 solve, the WY operands). The prep of chunk c+1 overlaps the carry of
// chunk c. The 16x16 block merges of the solve run on tf32 mma.sync.
//
// Every wait is bounded; on a timeout the kernel records a status bit, unwinds, waits
// for its own copies and MMAs, frees TMEM and returns.
#include <cudaTypedefs.h>

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
// pipeline events of CTA (0,0,0), read back with gdn_trace_read().
constexpr int kTraceChunks = 64, kTraceEvents = 48;
__device__ unsigned long long g_trace[kTraceChunks][kTraceEvents];
#define TRACE(c, ev)                                                                    \
    do {                                                                                \
        if (blockIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0 && (c) < kTraceChunks) \
            g_trace[(c)][(ev)] = clock64();                                             \
    } while (0)
#else
#define TRACE(c, ev) \
    do {             \
    } while (0)
#endif

namespace {
using namespace ptx;

constexpr int C = 64;           // chunk length
constexpr int NS = 64;          // state columns per CTA
constexpr int NTHREADS = 448;   // 14 warps
constexpr uint64_t kWaitNs = 2000000000ull;

// ---- shared memory map (offsets from a 1024-byte aligned base) ----
// stage s (two stages, one chunk each):
//   block b (b = 0,1 covers Dk columns 64b..64b+63): W | Q | K, 8 KB each (SW128, 64 rows)
//   V slice (64 tokens x 64 columns), T_U, T_W, P (64 x 64 each)
constexpr uint32_t BLK_STRIDE = 24576;
constexpr uint32_t OFF_W = 0, OFF_Q = 8192, OFF_K = 16384;
constexpr uint32_t OFF_V = 49152;
constexpr uint32_t OFF_TU = 57344, OFF_TW = 65536, OFF_P = 73728;
constexpr uint32_t STAGE_BYTES = 81920;
constexpr uint32_t OFF_U = 2 * STAGE_BYTES;   // U tile  (64 tokens x 64 columns)
constexpr uint32_t OFF_U2 = OFF_U + 8192;     // U' tile (decayed U)
constexpr uint32_t OFF_S = OFF_U2 + 8192;     // bf16 state operand (128 x 64)
constexpr uint32_t OFF_F32 = OFF_S + 16384;   // prep fp32 work area
constexpr int BS = 20;                        // row stride (floats) of a 16x16 block
constexpr uint32_t BLOCK_BYTES = 16 * BS * 4;
constexpr uint32_t OFF_AB = OFF_F32;                      // 10 lower blocks of A
constexpr uint32_t OFF_TB = OFF_AB + 10 * BLOCK_BYTES;    // 10 lower blocks of T
constexpr uint32_t OFF_XB = OFF_TB + 10 * BLOCK_BYTES;    // 16x8 scratch per prep warp
constexpr uint32_t OFF_SCAL = OFF_XB + 8 * 16 * 8 * 4;

struct StageScalars {
    float gam[C];    // gamma_r
    float beta[C];   // beta_r
    float ctab[C];   // exp(gamma_{end of r's 16-block} - gamma_r)
    float Gam[C];    // exp(gamma_r)
    float kdec[C];   // exp(gamma_last - gamma_r)
    float endgam[4]; // gamma at the end of each 16-block
    float Gl;        // exp(gamma_last)
    float pad[3];
};
constexpr uint32_t OFF_BAR = OFF_SCAL + 2 * sizeof(StageScalars);
constexpr uint32_t OFF_MISC = OFF_BAR + 128;
constexpr uint32_t SMEM_USED = OFF_MISC + 64;
constexpr uint32_t SMEM_BYTES = SMEM_USED + 1024;  // alignment slack
static_assert(OFF_BAR % 8 == 0, "barrier alignment");
static_assert(SMEM_BYTES <= 232448, "shared memory budget");

// TMEM columns (fp32, 128 lanes)
constexpr uint32_t TM_G = 0;     // Gram [QK^T; KK^T], 64 columns
constexpr uint32_t TM_W = 64;    // [W; -], 128 columns
constexpr uint32_t TM_U = 192;   // [U~; -], 64 columns
constexpr uint32_t TM_A = 256;   // [W S0; Q S0], 64 columns
constexpr uint32_t TM_S = 320;   // state increment, 64 columns
constexpr uint32_t TM_B = 384;   // [-; P U], 64 columns
constexpr uint32_t TM_COLS = 512;

// barrier indices
enum {
    B_FULL0 = 0, B_FULL1, B_EMPTY0, B_EMPTY1, B_GRAM, B_GFREE, B_PREP, B_WDONE,
    B_ADONE, B_CDONE, B_DRAIN, B_COUNT
};

// status bits
constexpr uint32_t ST_PRODUCER = 1u, ST_MMA = 2u, ST_CARRY = 4u, ST_PREP = 8u;

struct TcArgs {
    const float* g;
    const float* beta;
    float scale;
    int B, Hk, Hv, S;
    float* state;
    int state_is_input;
    __nv_bfloat16* out;
};

__device__ __forceinline__ void bar_sync(uint32_t id, uint32_t n) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
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

// Writes 16 fp32 values as bf16 into logical chunks ch0, ch0+1 of row r.
__device__ __forceinline__ void write_row16(uint32_t tile, int r, int ch0, const float* v) {
#pragma unroll
    for (int j = 0; j < 2; ++j) {
        st_shared_v4(sw128_chunk(tile, r, ch0 + j), pack_bf16(v[8 * j + 0], v[8 * j + 1]),
                     pack_bf16(v[8 * j + 2], v[8 * j + 3]), pack_bf16(v[8 * j + 4], v[8 * j + 5]),
                     pack_bf16(v[8 * j + 6], v[8 * j + 7]));
    }
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

// d += Ablk (16x16) * Bblk[:, 8 nt .. 8 nt + 7]
__device__ __forceinline__ void block_mma(float (&d)[4], const float* Ablk, const float* Bblk,
                                          int nt, int g, int t) {
#pragma unroll
    for (int ks = 0; ks < 2; ++ks) {
        uint32_t a[4], b[2];
        a[0] = to_tf32(Ablk[g * BS + ks * 8 + t]);
        a[1] = to_tf32(Ablk[(g + 8) * BS + ks * 8 + t]);
        a[2] = to_tf32(Ablk[g * BS + ks * 8 + t + 4]);
        a[3] = to_tf32(Ablk[(g + 8) * BS + ks * 8 + t + 4]);
        b[0] = to_tf32(Bblk[(ks * 8 + t) * BS + nt * 8 + g]);
        b[1] = to_tf32(Bblk[(ks * 8 + t + 4) * BS + nt * 8 + g]);
        mma_tf32(d, a, b);
    }
}

// Finishes T(i,j)[:, 8 nt ..] = -T(i,i) X for X held in x (C fragment): stores the fp32
// block and the bf16 T_U / T_W entries (columns scaled by beta_j and beta_j Gamma_j).
__device__ __forceinline__ void block_finish(const float (&x)[4], const float* Tii, float* Tout,
                                             float* xw, int i, int j, int nt, int g, int t,
                                             const float* beta, const float* Gam, uint32_t tu,
                                             uint32_t tw) {
    xw[g * 8 + 2 * t] = x[0];
    xw[g * 8 + 2 * t + 1] = x[1];
    xw[(g + 8) * 8 + 2 * t] = x[2];
    xw[(g + 8) * 8 + 2 * t + 1] = x[3];
    __syncwarp();
    float e[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int ks = 0; ks < 2; ++ks) {
        uint32_t a[4], b[2];
        a[0] = to_tf32(Tii[g * BS + ks * 8 + t]);
        a[1] = to_tf32(Tii[(g + 8) * BS + ks * 8 + t]);
        a[2] = to_tf32(Tii[g * BS + ks * 8 + t + 4]);
        a[3] = to_tf32(Tii[(g + 8) * BS + ks * 8 + t + 4]);
        b[0] = to_tf32(xw[(ks * 8 + t) * 8 + g]);
        b[1] = to_tf32(xw[(ks * 8 + t + 4) * 8 + g]);
        mma_tf32(e, a, b);
    }
    __syncwarp();
    const int c0 = nt * 8 + 2 * t;  // column inside the block
    Tout[g * BS + c0] = -e[0];
    Tout[g * BS + c0 + 1] = -e[1];
    Tout[(g + 8) * BS + c0] = -e[2];
    Tout[(g + 8) * BS + c0 + 1] = -e[3];
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

__device__ __forceinline__ void issue_gram(uint32_t tmem, uint32_t st) {
    constexpr uint32_t id = idesc_bf16(128, 64, false, false);
    const uint64_t a0 = smem_desc_sw128(st + OFF_Q, 16, 1024);
    const uint64_t b0 = smem_desc_sw128(st + OFF_K, 16, 1024);
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        const uint32_t off = (uint32_t)(k >> 2) * BLK_STRIDE + (uint32_t)(k & 3) * 32u;
        mma_bf16(tmem + TM_G, dadd(a0, off), dadd(b0, off), id, k > 0);
    }
}

__device__ __forceinline__ void issue_wy(uint32_t tmem, uint32_t st) {
    constexpr uint32_t idw = idesc_bf16(128, 128, false, true);
    const uint64_t aw = smem_desc_sw128(st + OFF_TW, 16, 1024);
    const uint64_t bk = smem_desc_sw128(st + OFF_K, BLK_STRIDE, 1024);
#pragma unroll
    for (int k = 0; k < 4; ++k) mma_bf16(tmem + TM_W, dadd(aw, k * 32), dadd(bk, k * 2048), idw, k > 0);
    constexpr uint32_t idu = idesc_bf16(128, 64, false, true);
    const uint64_t au = smem_desc_sw128(st + OFF_TU, 16, 1024);
    const uint64_t bv = smem_desc_sw128(st + OFF_V, 8192, 1024);
    const uint32_t du = tmem + TM_U;
#pragma unroll
    for (int k = 0; k < 4; ++k) mma_bf16(du, dadd(au, k * 32), dadd(bv, k * 2048), idu, k > 0);
}

__device__ __forceinline__ void issue_carry1(uint32_t tmem, uint32_t st, uint32_t s_tile) {
    constexpr uint32_t id = idesc_bf16(128, 64, false, true);
    const uint64_t a0 = smem_desc_sw128(st + OFF_W, 16, 1024);
    const uint64_t b0 = smem_desc_sw128(s_tile, 8192, 1024);
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        const uint32_t off = (uint32_t)(k >> 2) * BLK_STRIDE + (uint32_t)(k & 3) * 32u;
        mma_bf16(tmem + TM_A, dadd(a0, off), dadd(b0, k * 2048), id, k > 0);
    }
}

__device__ __forceinline__ void issue_carry23(uint32_t tmem, uint32_t st, uint32_t u_tile,
                                              uint32_t u2_tile) {
    constexpr uint32_t id2 = idesc_bf16(128, 64, false, true);
    const uint64_t aw = smem_desc_sw128(st + OFF_TW, 16, 1024);
    const uint64_t bu = smem_desc_sw128(u_tile, 8192, 1024);
#pragma unroll
    for (int k = 0; k < 4; ++k) mma_bf16(tmem + TM_B, dadd(aw, k * 32), dadd(bu, k * 2048), id2, k > 0);
    constexpr uint32_t id3 = idesc_bf16(128, 64, true, true);
    const uint64_t ak = smem_desc_sw128(st + OFF_K, BLK_STRIDE, 1024);
    const uint64_t bu2 = smem_desc_sw128(u2_tile, 8192, 1024);
#pragma unroll
    for (int k = 0; k < 4; ++k)
        mma_bf16(tmem + TM_S, dadd(ak, k * 2048), dadd(bu2, k * 2048), id3, k > 0);
}

// ---------------------------------------------------------------- the kernel

__global__ void __launch_bounds__(NTHREADS, 1)
    prefill_tc_kernel(const __grid_constant__ CUtensorMap mq, const __grid_constant__ CUtensorMap mk,
                      const __grid_constant__ CUtensorMap mv, TcArgs a) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    // 1024-byte alignment by a byte offset from the shared array itself, so every
    // pointer derived from `sm` stays a shared-memory pointer (an integer round trip
    // would turn the accesses into generic loads and stores).
    uint8_t* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const uint32_t sbase = smem_u32(sm);
    uint64_t* bar = reinterpret_cast<uint64_t*>(sm + OFF_BAR);
    uint32_t* misc = reinterpret_cast<uint32_t*>(sm + OFF_MISC);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(misc + 1);
    uint32_t* u_ctr = misc + 2;  // chunks whose U~ the carry has consumed
    StageScalars* scal = reinterpret_cast<StageScalars*>(sm + OFF_SCAL);
    float* Ab = reinterpret_cast<float*>(sm + OFF_AB);
    float* Tb = reinterpret_cast<float*>(sm + OFF_TB);
    float* Xb = reinterpret_cast<float*>(sm + OFF_XB);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int n0 = blockIdx.x * NS, h = blockIdx.y, b = blockIdx.z;
    const int kh = h / (a.Hv / a.Hk);  // value head h reads key head h // (Hv/Hk)
    const int S = a.S;
    const int nch = (S + C - 1) / C;

    if (tid == 0) {
        for (int i = 0; i < B_COUNT + 1; ++i)
            mbar_init(&bar[i], (i == B_FULL0 || i == B_FULL1) ? 2 : 1);
        *abort_flag = 0;
        *u_ctr = 0;
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(misc, TM_COLS);
        tmem_relinquish();
    }
    if (tid == 32) {
        prefetch_tensormap(&mq);
        prefetch_tensormap(&mk);
        prefetch_tensormap(&mv);
    }
    // T_U / T_W blocks above the diagonal are never written: zero both stages once
    for (int i = tid; i < 4 * 8192 / 16; i += NTHREADS) {
        const int tile = i >> 9, off = (i & 511) * 16;
        const uint32_t base =
            sbase + (uint32_t)(tile >> 1) * STAGE_BYTES + ((tile & 1) ? OFF_TW : OFF_TU);
        st_shared_v4(base + off, 0u, 0u, 0u, 0u);
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = misc[0];

    if (warp == 0) {
        // -------------------------------------------- TMA producer + decay tables (warp)
        const int zq = b * a.Hk + kh, zv = b * a.Hv + h;
        const float* gp = a.g + (size_t)zv * S;
        const float* bp = a.beta + (size_t)zv * S;
        int issued = 0;
        for (int c = 0; c < nch; ++c) {
            const int s = c & 1;
            int ok = 1;
            if (lane == 0) {
                if (c >= 2 &&
                    !mbar_wait_bounded(&bar[B_EMPTY0 + s], ((c >> 1) + 1) & 1, kWaitNs)) {
                    record_failure(abort_flag, ST_PRODUCER);
                    ok = 0;
                }
                if (*abort_flag) ok = 0;
            }
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) break;
            if (lane == 0) {
                uint8_t* st = sm + s * STAGE_BYTES;
                TRACE(c, 0);
                mbar_arrive_expect_tx(&bar[B_FULL0 + s], 2 * 16384 + 8192);
                for (int blk = 0; blk < 2; ++blk) {
                    tma_load_3d(st + blk * BLK_STRIDE + OFF_Q, &mq, &bar[B_FULL0 + s], blk * 64,
                                c * C, zq);
                    tma_load_3d(st + blk * BLK_STRIDE + OFF_K, &mk, &bar[B_FULL0 + s], blk * 64,
                                c * C, zq);
                }
                tma_load_3d(st + OFF_V, &mv, &bar[B_FULL0 + s], n0, c * C, zv);
            }
            issued = c + 1;
            // decay tables of chunk c (padding tokens: g = beta = 0, an exact no-op)
            StageScalars& sc = scal[s];
            const int t0 = c * C + lane, t1 = t0 + 32;
            float x0 = (t0 < S) ? gp[t0] : 0.f, x1 = (t1 < S) ? gp[t1] : 0.f;
            const float be0 = (t0 < S) ? bp[t0] : 0.f, be1 = (t1 < S) ? bp[t1] : 0.f;
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
            sc.gam[lane] = x0;
            sc.gam[lane + 32] = x1;
            sc.beta[lane] = be0;
            sc.beta[lane + 32] = be1;
            sc.ctab[lane] = __expf(e0 - x0);
            sc.ctab[lane + 32] = __expf(e1 - x1);
            sc.Gam[lane] = __expf(x0);
            sc.Gam[lane + 32] = __expf(x1);
            sc.kdec[lane] = __expf(gl - x0);
            sc.kdec[lane + 32] = __expf(gl - x1);
            if (lane == 15) {
                sc.endgam[0] = x0;
                sc.endgam[2] = x1;
            }
            if (lane == 31) {
                sc.endgam[1] = x0;
                sc.endgam[3] = x1;
                sc.Gl = __expf(gl);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&bar[B_FULL0 + s]);
        }
        if (lane == 0 && *abort_flag) {
            // let the copies already issued land before the CTA exits
            for (int c = (issued > 2 ? issued - 2 : 0); c < issued; ++c)
                mbar_wait_bounded(&bar[B_FULL0 + (c & 1)], (c >> 1) & 1, kWaitNs);
        }
    } else if (warp == 1) {
        // ------------------------------------------- MMA issuer for the prep (one thread)
        // Gram(c) once the chunk has landed and the prep has read Gram(c-1); WY(c) once
        // the prep has written T_U/T_W/P and the carry has consumed U~(c-1). The carry's
        // own MMAs are issued by the carry.
        if (lane == 0) {
            int g = 0, wu = 0;
            uint32_t idle = 0;
            uint64_t t_last = globaltimer_ns();
            while (wu < nch) {
                bool did = false;
                if (g < nch && (g == 0 || mbar_test_wait(&bar[B_GFREE], (g - 1) & 1)) &&
                    mbar_test_wait(&bar[B_FULL0 + (g & 1)], (g >> 1) & 1)) {
                    tc_fence_after();
                    issue_gram(tmem, sbase + (g & 1) * STAGE_BYTES);
                    tc_commit(&bar[B_GRAM]);
                    TRACE(g, 1);
                    ++g;
                    did = true;
                } else if (wu < g && ld_acquire_u32(u_ctr) >= (uint32_t)wu &&
                           mbar_test_wait(&bar[B_PREP], wu & 1)) {
                    tc_fence_after();
                    issue_wy(tmem, sbase + (wu & 1) * STAGE_BYTES);
                    tc_commit(&bar[B_WDONE]);
                    TRACE(wu, 2);
                    ++wu;
                    did = true;
                }
                if (did) {
                    idle = 0;
                } else if ((++idle & 255) == 0) {
                    // time and the abort flag are checked every 256 idle polls
                    const uint64_t now = globaltimer_ns();
                    if (idle == 256) t_last = now;
                    if (now - t_last > kWaitNs) {
                        record_failure(abort_flag, ST_MMA);
                        break;
                    }
                    if (*abort_flag) break;
                }
            }
            // no MMA of this thread may be in flight when TMEM is freed
            tc_commit(&bar[B_DRAIN]);
            mbar_wait_bounded(&bar[B_DRAIN], 0, kWaitNs);
        }
    } else if (warp < 6) {
        // ------------------------------------------------------------ carry (128 threads)
        // Issues its own MMAs (thread L = 0) so that the sequential chain carry ->
        // tensor core -> carry has no hand-off through another warp.
        const int q = warp & 3;
        const int L = 32 * q + lane;  // TMEM lane = state row (Dk index) = token for L < 64
        const uint32_t lane_off = (uint32_t)(32 * q) << 16;
        const uint32_t s_tile = sbase + OFF_S, u_tile = sbase + OFF_U, u2_tile = sbase + OFF_U2;
        float* gstate = a.state + ((size_t)(b * a.Hv + h) * 128 + L) * 128 + n0;
        __nv_bfloat16* gout = a.out + (size_t)(b * a.Hv + h) * S * 128 + n0;

        float Sm[NS];
        if (a.state_is_input) {
#pragma unroll
            for (int j = 0; j < NS; j += 4) {
                const float4 x = *reinterpret_cast<const float4*>(gstate + j);
                Sm[j] = x.x;
                Sm[j + 1] = x.y;
                Sm[j + 2] = x.z;
                Sm[j + 3] = x.w;
            }
        } else {
#pragma unroll
            for (int j = 0; j < NS; ++j) Sm[j] = 0.f;
        }
        write_row32(s_tile, L, 0, Sm);
        write_row32(s_tile, L, 4, Sm + 32);
        fence_proxy_async_smem();
        bar_sync(1, 128);

        for (int c = 0; c < nch; ++c) {
            const int s = c & 1;
            const uint32_t st = sbase + s * STAGE_BYTES;
            // W(c) = T_W K from TMEM into the W tile (bf16), then MMA1: [W; Q] S0
            bool ok = mbar_wait_bounded(&bar[B_WDONE], c & 1, kWaitNs);
            if (!ok) record_failure(abort_flag, ST_CARRY);
            if (bar_any(1, 128, !ok || *abort_flag)) break;
            if (L == 0) TRACE(c, 12);
            tc_fence_after();
            if (L < 64) {
#pragma unroll
                for (int qd = 0; qd < 4; ++qd) {
                    float w[32];
                    tmem_ld32(tmem + lane_off + TM_W + 32 * qd, w);
                    write_row32(st + (qd >> 1) * BLK_STRIDE + OFF_W, L, 4 * (qd & 1), w);
                }
            }
            fence_proxy_async_smem();
            tc_fence_before();
            bar_sync(1, 128);
            if (L == 0) {
                tc_fence_after();
                issue_carry1(tmem, st, s_tile);
                tc_commit(&bar[B_ADONE]);
                TRACE(c, 3);
            }
            ok = mbar_wait_bounded(&bar[B_ADONE], c & 1, kWaitNs);
            if (!ok) record_failure(abort_flag, ST_CARRY);
            if (bar_any(1, 128, !ok || *abort_flag)) break;
            if (L == 0) TRACE(c, 13);
            tc_fence_after();
            // per-chunk scalars are read now: the producer may rewrite this stage's tables
            // once the chunk's last MMAs complete
            const float Gl = scal[s].Gl;
            float gm = 0.f;
            if (L < 64) {
                // U = U~ - W S0 and U' = exp(gamma_last - gamma_L) U for token L
                const float kd = scal[s].kdec[L];
#pragma unroll
                for (int qq = 0; qq < 4; ++qq) {
                    float ws[16], ut[16];
                    tmem_ld16x2(tmem + lane_off + TM_A + 16 * qq, tmem + lane_off + TM_U + 16 * qq,
                                ws, ut);
#pragma unroll
                    for (int j = 0; j < 16; ++j) ut[j] -= ws[j];
                    write_row16(u_tile, L, 2 * qq, ut);
#pragma unroll
                    for (int j = 0; j < 16; ++j) ut[j] *= kd;
                    write_row16(u2_tile, L, 2 * qq, ut);
                }
            } else {
                gm = scal[s].Gam[L - 64];
            }
            fence_proxy_async_smem();
            tc_fence_before();
            bar_sync(1, 128);
            if (L == 0) {
                TRACE(c, 14);
                st_release_u32(u_ctr, (uint32_t)(c + 1));  // U~(c) consumed
                tc_fence_after();
                issue_carry23(tmem, st, u_tile, u2_tile);
                tc_commit(&bar[B_CDONE]);
                tc_commit(&bar[B_EMPTY0 + s]);
                TRACE(c, 4);
            }
            ok = mbar_wait_bounded(&bar[B_CDONE], c & 1, kWaitNs);
            if (!ok) record_failure(abort_flag, ST_CARRY);
            if (bar_any(1, 128, !ok || *abort_flag)) break;
            if (L == 0) TRACE(c, 15);
            tc_fence_after();
            if (L >= 64) {
                // O = scale (Gamma Q S0 + P U) for token L - 64
                const int t = c * C + (L - 64);
#pragma unroll
                for (int qq = 0; qq < 4; ++qq) {
                    float qs[16], pu[16];
                    tmem_ld16x2(tmem + lane_off + TM_A + 16 * qq, tmem + lane_off + TM_B + 16 * qq,
                                qs, pu);
                    if (t < S) {
                        uint4* dst = reinterpret_cast<uint4*>(gout + (size_t)t * 128 + 16 * qq);
#pragma unroll
                        for (int j = 0; j < 2; ++j) {
                            float o[8];
#pragma unroll
                            for (int e = 0; e < 8; ++e)
                                o[e] = a.scale * fmaf(gm, qs[8 * j + e], pu[8 * j + e]);
                            uint4 w;
                            w.x = pack_bf16(o[0], o[1]);
                            w.y = pack_bf16(o[2], o[3]);
                            w.z = pack_bf16(o[4], o[5]);
                            w.w = pack_bf16(o[6], o[7]);
                            dst[j] = w;
                        }
                    }
                }
            }
            // S1 = Gamma_last S0 + K^T U' for state row L
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                float d[32];
                tmem_ld32(tmem + lane_off + TM_S + 32 * hh, d);
#pragma unroll
                for (int j = 0; j < 32; ++j) Sm[32 * hh + j] = fmaf(Gl, Sm[32 * hh + j], d[j]);
                write_row32(s_tile, L, 4 * hh, Sm + 32 * hh);
            }
            fence_proxy_async_smem();
            tc_fence_before();
            bar_sync(1, 128);
            if (L == 0) TRACE(c, 16);
        }
        if (!*abort_flag) {
#pragma unroll
            for (int j = 0; j < NS; j += 4)
                *reinterpret_cast<float4*>(gstate + j) =
                    make_float4(Sm[j], Sm[j + 1], Sm[j + 2], Sm[j + 3]);
        }
        // no MMA of the carry may be in flight when TMEM is freed
        if (L == 0 && *abort_flag) {
            tc_commit(&bar[B_DRAIN + 1]);
            mbar_wait_bounded(&bar[B_DRAIN + 1], 0, kWaitNs);
        }
    } else {
        // ------------------------------------------------------------ prep (256 threads)
        const int P = tid - 192;
        const int pw = P >> 5;  // prep warp 0..7
        const int wg = P >> 7;  // column half of the Gram matrices
        const int q = warp & 3;
        const int L = 32 * q + lane;
        const int g8 = lane >> 2, t4 = lane & 3;
        const uint32_t lane_off = (uint32_t)(32 * q) << 16;
        float* xw = Xb + pw * 16 * 8;

        for (int c = 0; c < nch; ++c) {
            const int s = c & 1;
            const uint32_t st = sbase + s * STAGE_BYTES;
            const uint32_t tu = st + OFF_TU, tw = st + OFF_TW;
            const StageScalars& sc = scal[s];
            bool ok = mbar_wait_bounded(&bar[B_FULL0 + s], (c >> 1) & 1, kWaitNs) &&
                      mbar_wait_bounded(&bar[B_GRAM], c & 1, kWaitNs);
            if (!ok) record_failure(abort_flag, ST_PREP);
            if (bar_any(2, 256, !ok || *abort_flag)) break;
            if (P == 0) TRACE(c, 7);
            tc_fence_after();

            // ---- P (bf16 tile) and A (fp32 blocks) from the Gram matrices:
            // thread (wg, L) takes row L of [QK^T; KK^T], columns 32 wg .. 32 wg + 31
            {
                const int r = L & 63, br = r >> 4, rl = r & 15;
                const bool isP = L < 64;
                const float gr = sc.gam[r];
                const float scl = isP ? 1.f : sc.beta[r];
                float gv[32];
                tmem_ld32(tmem + lane_off + TM_G + 32 * wg, gv);
                if (P == 0) TRACE(c, 19);
                if (lane == 0) TRACE(c, 24 + pw);
#pragma unroll
                for (int bq = 0; bq < 2; ++bq) {
                    const int bj = 2 * wg + bq;
                    if (bj < br) {
                        const float f = __expf(gr - sc.endgam[bj]) * scl;
#pragma unroll
                        for (int jj = 0; jj < 16; ++jj)
                            gv[16 * bq + jj] *= f * sc.ctab[16 * bj + jj];
                    } else if (bj == br) {
                        // branch-free: exp of a non-positive argument, then the mask
                        const int lim = isP ? rl : rl - 1;
#pragma unroll
                        for (int jj = 0; jj < 16; ++jj) {
                            const float e = __expf(fminf(gr - sc.gam[16 * bj + jj], 0.f));
                            const float m = (jj <= lim) ? scl : 0.f;
                            gv[16 * bq + jj] *= e * m;
                        }
                    } else {
#pragma unroll
                        for (int jj = 0; jj < 16; ++jj) gv[16 * bq + jj] = 0.f;
                    }
                }
                if (isP) {
                    write_row32(st + OFF_P, r, 4 * wg, gv);
                } else {
#pragma unroll
                    for (int bq = 0; bq < 2; ++bq) {
                        const int bj = 2 * wg + bq;
                        if (bj <= br) {
                            float* dst = Ab + bidx(br, bj) * 16 * BS + rl * BS;
#pragma unroll
                            for (int jj = 0; jj < 16; jj += 4)
                                *reinterpret_cast<float4*>(dst + jj) =
                                    make_float4(gv[16 * bq + jj], gv[16 * bq + jj + 1],
                                                gv[16 * bq + jj + 2], gv[16 * bq + jj + 3]);
                        }
                    }
                }
            }
            if (lane == 0) TRACE(c, 32 + pw);
            tc_fence_before();
            bar_sync(2, 256);
            if (P == 0) {
                TRACE(c, 8);
                mbar_arrive(&bar[B_GFREE]);  // Gram(c) read: Gram(c+1) may overwrite it
            }

            // ---- T = (I + A)^-1 in 16x16 blocks
            // diagonal blocks: forward substitution, one column per thread
            if (P < 64) {
                const int i = P >> 4, cc = P & 15;
                const float* Ad = Ab + bidx(i, i) * 16 * BS;
                float xs[16], acc[16];
#pragma unroll
                for (int r = 0; r < 16; ++r) acc[r] = 0.f;
#pragma unroll
                for (int m = 0; m < 16; ++m) {
                    const float xm = (m < cc) ? 0.f : ((m == cc) ? 1.f : -acc[m]);
                    xs[m] = xm;
#pragma unroll
                    for (int r = m + 1; r < 16; ++r) acc[r] = fmaf(Ad[r * BS + m], xm, acc[r]);
                }
                float* Td = Tb + bidx(i, i) * 16 * BS;
                const int J = 16 * i + cc;
                const float bj = sc.beta[J], wj = bj * sc.Gam[J];
#pragma unroll
                for (int r = 0; r < 16; ++r) {
                    Td[r * BS + cc] = xs[r];
                    st_shared_b16(sw128_elem(tu, 16 * i + r, J), xs[r] * bj);
                    st_shared_b16(sw128_elem(tw, 16 * i + r, J), xs[r] * wj);
                }
            }
            bar_sync(2, 256);
            if (P == 0) TRACE(c, 9);
            // level 1: T(i,i-1) = -T(i,i) A(i,i-1) T(i-1,i-1), i = 1..3 (warp: block, 8 columns)
            if (pw < 6) {
                const int i = 1 + (pw >> 1), nt = pw & 1;
                float x[4] = {0.f, 0.f, 0.f, 0.f};
                block_mma(x, Ab + bidx(i, i - 1) * 16 * BS, Tb + bidx(i - 1, i - 1) * 16 * BS, nt,
                          g8, t4);
                block_finish(x, Tb + bidx(i, i) * 16 * BS, Tb + bidx(i, i - 1) * 16 * BS, xw, i,
                             i - 1, nt, g8, t4, sc.beta, sc.Gam, tu, tw);
            }
            bar_sync(2, 256);
            // level 2: T(j+2,j) = -T(j+2,j+2) (A(j+2,j) T(j,j) + A(j+2,j+1) T(j+1,j))
            if (pw < 4) {
                const int j = pw >> 1, i = j + 2, nt = pw & 1;
                float x[4] = {0.f, 0.f, 0.f, 0.f};
                block_mma(x, Ab + bidx(i, j) * 16 * BS, Tb + bidx(j, j) * 16 * BS, nt, g8, t4);
                block_mma(x, Ab + bidx(i, j + 1) * 16 * BS, Tb + bidx(j + 1, j) * 16 * BS, nt, g8,
                          t4);
                block_finish(x, Tb + bidx(i, i) * 16 * BS, Tb + bidx(i, j) * 16 * BS, xw, i, j, nt,
                             g8, t4, sc.beta, sc.Gam, tu, tw);
            }
            bar_sync(2, 256);
            // level 3: T(3,0) = -T(3,3) (A(3,0) T(0,0) + A(3,1) T(1,0) + A(3,2) T(2,0))
            if (pw < 2) {
                const int nt = pw;
                float x[4] = {0.f, 0.f, 0.f, 0.f};
                block_mma(x, Ab + bidx(3, 0) * 16 * BS, Tb + bidx(0, 0) * 16 * BS, nt, g8, t4);
                block_mma(x, Ab + bidx(3, 1) * 16 * BS, Tb + bidx(1, 0) * 16 * BS, nt, g8, t4);
                block_mma(x, Ab + bidx(3, 2) * 16 * BS, Tb + bidx(2, 0) * 16 * BS, nt, g8, t4);
                block_finish(x, Tb + bidx(3, 3) * 16 * BS, Tb + bidx(3, 0) * 16 * BS, xw, 3, 0, nt,
                             g8, t4, sc.beta, sc.Gam, tu, tw);
            }
            fence_proxy_async_smem();
            // the issuer must have taken prep_ready(c-1) (its WY has completed) before
            // prep_ready(c) is posted, so that barrier never runs two phases ahead
            ok = c == 0 || mbar_wait_bounded(&bar[B_WDONE], (c - 1) & 1, kWaitNs);
            if (!ok) record_failure(abort_flag, ST_PREP);
            if (bar_any(2, 256, !ok || *abort_flag)) break;
            if (P == 0) {
                TRACE(c, 10);
                mbar_arrive(&bar[B_PREP]);
            }

        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, TM_COLS);
    }
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
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

// 3-D bf16 map over [z][y][x] = [heads][S][128], box 64 x 64 x 1, 128-byte swizzle.
bool encode_3d(CUtensorMap* m, const void* base, int S, int heads) {
    auto fn = encode_fn();
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

cudaError_t launch_prefill_tc(const PrefillArgs& a, cudaStream_t stream, int* launched) {
    *launched = 0;
    CUtensorMap mq, mk, mv;
    if (!encode_3d(&mq, a.q, a.S, a.B * a.Hk) || !encode_3d(&mk, a.k, a.S, a.B * a.Hk) ||
        !encode_3d(&mv, a.v, a.S, a.B * a.Hv))
        return cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(prefill_tc_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM_BYTES);
    if (e != cudaSuccess) return e;
    TcArgs t{a.g, a.beta, a.scale, a.B, a.Hk, a.Hv, a.S, a.state, a.state_is_input,
             static_cast<__nv_bfloat16*>(a.out)};
    const dim3 grid(128 / NS, a.Hv, a.B);
    prefill_tc_kernel<<<grid, NTHREADS, SMEM_BYTES, stream>>>(mq, mk, mv, t);
    *launched = 1;
    return cudaGetLastError();
}

}  // namespace gdn

#ifdef GDN_TRACE
extern "C" int gdn_trace_read(unsigned long long* dst) {
    return cudaMemcpyFromSymbol(dst, gdn::g_trace, sizeof(gdn::g_trace)) == cudaSuccess ? 0 : 1;
}
#endif
