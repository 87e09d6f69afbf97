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
//   W = T_W K,  U~ = T_U V,  U = U~ - W S0
//   O  = scale (diag(Gamma) Q S0 + P U)
//   S1 = Gamma_last S0 + K~^T U,   K~ = diag(exp(gamma_last - gamma)) K
//
// One CTA per (batch, value head, 64-column slice of the state); the state's columns
// evolve independently, so slices never communicate. Per chunk, on the tensor cores:
//   Gram   [Q;K] K^T          -> QK^T and KK^T        (M128 N64  K128)
//   WY     [T_W;P] K, [T_U;T_W] V -> W and U~          (M128 N128 K64, M128 N64 K64)
//   carry  [W;GQ] S0          -> W S0 and Gamma Q S0   (M128 N64  K128)
//          [T_W;P] U (+=)     -> + P U                 (M128 N64  K64)
//          K~^T U             -> state increment       (M128 N64  K64)
// Stacking two 64-row operands into one 128-row operand fills the M = 128 data path;
// the half of the result that is not needed is ignored.
//
// Warp roles (14 warps): 0 = TMA producer, 1 = MMA issuer (one thread), 2-5 = carry
// (state master, U, output, state update), 6-13 = prep (decay tables, P and A from the
// Gram matrices, the (I+A)^-1 solve, WY operands). The prep of chunk c+1 overlaps the
// carry of chunk c. Every wait is bounded; on a timeout the kernel records a status bit,
// unwinds, waits for its own copies and MMAs, frees TMEM and returns.
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
constexpr uint32_t OFF_U = 2 * STAGE_BYTES;   // U tile (64 tokens x 64 columns)
constexpr uint32_t OFF_S = OFF_U + 8192;      // bf16 state operand (128 x 64)
constexpr uint32_t OFF_F32 = OFF_S + 16384;   // prep fp32 work area
constexpr int BS = 20;                        // row stride (floats) of a 16x16 block
constexpr uint32_t BLOCK_BYTES = 16 * BS * 4;
constexpr uint32_t OFF_AB = OFF_F32;                      // 10 lower blocks of A
constexpr uint32_t OFF_TB = OFF_AB + 10 * BLOCK_BYTES;    // 10 lower blocks of T
constexpr uint32_t OFF_XB = OFF_TB + 10 * BLOCK_BYTES;    // 3 scratch blocks
constexpr uint32_t OFF_SCAL = OFF_XB + 3 * BLOCK_BYTES;

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
constexpr uint32_t TM_U = 192;   // [U~; -], 64 columns x 2 buffers
constexpr uint32_t TM_A = 320;   // [W S0; Gamma Q S0 + P U], 64 columns
constexpr uint32_t TM_S = 384;   // state increment, 64 columns
constexpr uint32_t TM_COLS = 512;

// barrier indices
enum {
    B_FULL0 = 0, B_FULL1, B_EMPTY0, B_EMPTY1, B_GRAM, B_PREP, B_WDONE, B_WREADY,
    B_SREADY, B_ADONE, B_UREADY, B_CDONE, B_DRAIN, B_COUNT
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

__device__ __forceinline__ void ld_shared_v4(uint32_t addr, uint32_t& a, uint32_t& b, uint32_t& c,
                                             uint32_t& d) {
    asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(a), "=r"(b), "=r"(c), "=r"(d)
                 : "r"(addr)
                 : "memory");
}

// Address of 16-byte chunk `ch` (logical) of row `r` in a 128-byte-swizzled tile.
__device__ __forceinline__ uint32_t sw128_chunk(uint32_t tile, int r, int ch) {
    return tile + (uint32_t)(r >> 3) * 1024u + (uint32_t)(r & 7) * 128u +
           ((uint32_t)((ch ^ r) & 7) << 4);
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

__device__ __forceinline__ uint32_t scale_bf16x2(uint32_t v, float f) {
    __nv_bfloat162 h = *reinterpret_cast<__nv_bfloat162*>(&v);
    const float2 x = __bfloat1622float2(h);
    return pack_bf16(x.x * f, x.y * f);
}

// Multiplies one 16-byte chunk (8 bf16) in place by f.
__device__ __forceinline__ void scale_chunk(uint32_t addr, float f) {
    uint32_t a, b, c, d;
    ld_shared_v4(addr, a, b, c, d);
    st_shared_v4(addr, scale_bf16x2(a, f), scale_bf16x2(b, f), scale_bf16x2(c, f),
                 scale_bf16x2(d, f));
}

__device__ __forceinline__ void record_failure(volatile int* abort_flag, uint32_t bit) {
    atomicOr(&g_tc_status, bit);
    *abort_flag = 1;
}

// Lower-triangular 16x16 block index of block (i, j), i >= j.
__host__ __device__ constexpr int bidx(int i, int j) { return i * (i + 1) / 2 + j; }

// ---------------------------------------------------------------- MMA issue helpers

__device__ __forceinline__ void issue_gram(uint32_t tmem, uint32_t st) {
    constexpr uint32_t id = idesc_bf16(128, 64, false, false);
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        const uint32_t blk = st + (uint32_t)(k >> 2) * BLK_STRIDE + (uint32_t)(k & 3) * 32u;
        mma_bf16(tmem + TM_G, smem_desc_sw128(blk + OFF_Q, 16, 1024),
                 smem_desc_sw128(blk + OFF_K, 16, 1024), id, k > 0);
    }
}

__device__ __forceinline__ void issue_wy(uint32_t tmem, uint32_t st, int c) {
    constexpr uint32_t idw = idesc_bf16(128, 128, false, true);
#pragma unroll
    for (int k = 0; k < 4; ++k)
        mma_bf16(tmem + TM_W, smem_desc_sw128(st + OFF_TW + k * 32, 16, 1024),
                 smem_desc_sw128(st + OFF_K + k * 2048, BLK_STRIDE, 1024), idw, k > 0);
    constexpr uint32_t idu = idesc_bf16(128, 64, false, true);
#pragma unroll
    for (int k = 0; k < 4; ++k)
        mma_bf16(tmem + TM_U + 64u * (uint32_t)(c & 1),
                 smem_desc_sw128(st + OFF_TU + k * 32, 16, 1024),
                 smem_desc_sw128(st + OFF_V + k * 2048, 8192, 1024), idu, k > 0);
}

__device__ __forceinline__ void issue_carry1(uint32_t tmem, uint32_t st, uint32_t s_tile) {
    constexpr uint32_t id = idesc_bf16(128, 64, false, true);
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        const uint32_t blk = st + (uint32_t)(k >> 2) * BLK_STRIDE + (uint32_t)(k & 3) * 32u;
        mma_bf16(tmem + TM_A, smem_desc_sw128(blk + OFF_W, 16, 1024),
                 smem_desc_sw128(s_tile + k * 2048, 8192, 1024), id, k > 0);
    }
}

__device__ __forceinline__ void issue_carry23(uint32_t tmem, uint32_t st, uint32_t u_tile) {
    constexpr uint32_t id2 = idesc_bf16(128, 64, false, true);
#pragma unroll
    for (int k = 0; k < 4; ++k)
        mma_bf16(tmem + TM_A, smem_desc_sw128(st + OFF_TW + k * 32, 16, 1024),
                 smem_desc_sw128(u_tile + k * 2048, 8192, 1024), id2, 1);
    constexpr uint32_t id3 = idesc_bf16(128, 64, true, true);
#pragma unroll
    for (int k = 0; k < 4; ++k)
        mma_bf16(tmem + TM_S, smem_desc_sw128(st + OFF_K + k * 2048, BLK_STRIDE, 1024),
                 smem_desc_sw128(u_tile + k * 2048, 8192, 1024), id3, k > 0);
}

// ---------------------------------------------------------------- the kernel

__global__ void __launch_bounds__(NTHREADS, 1)
    prefill_tc_kernel(const __grid_constant__ CUtensorMap mq, const __grid_constant__ CUtensorMap mk,
                      const __grid_constant__ CUtensorMap mv, TcArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
    const uint32_t sbase = smem_u32(sm);
    uint64_t* bar = reinterpret_cast<uint64_t*>(sm + OFF_BAR);
    uint32_t* misc = reinterpret_cast<uint32_t*>(sm + OFF_MISC);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(misc + 1);
    float* scan_tot = reinterpret_cast<float*>(misc + 2);
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
        for (int i = 0; i < B_COUNT; ++i) mbar_init(&bar[i], 1);
        *abort_flag = 0;
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
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = misc[0];

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            const int zq = b * a.Hk + kh, zv = b * a.Hv + h;
            int issued = 0;
            for (int c = 0; c < nch; ++c) {
                const int s = c & 1;
                if (c >= 2 && !mbar_wait_bounded(&bar[B_EMPTY0 + s], ((c >> 1) + 1) & 1, kWaitNs)) {
                    record_failure(abort_flag, ST_PRODUCER);
                    break;
                }
                if (*abort_flag) break;
                uint8_t* st = sm + s * STAGE_BYTES;
                mbar_arrive_expect_tx(&bar[B_FULL0 + s], 2 * 16384 + 8192);
                for (int blk = 0; blk < 2; ++blk) {
                    tma_load_3d(st + blk * BLK_STRIDE + OFF_Q, &mq, &bar[B_FULL0 + s], blk * 64,
                                c * C, zq);
                    tma_load_3d(st + blk * BLK_STRIDE + OFF_K, &mk, &bar[B_FULL0 + s], blk * 64,
                                c * C, zq);
                }
                tma_load_3d(st + OFF_V, &mv, &bar[B_FULL0 + s], n0, c * C, zv);
                issued = c + 1;
            }
            if (*abort_flag) {
                // let the copies already issued land before the CTA exits
                for (int c = (issued > 2 ? issued - 2 : 0); c < issued; ++c)
                    mbar_wait_bounded(&bar[B_FULL0 + (c & 1)], (c >> 1) & 1, kWaitNs);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            int g = 0, wu = 0, m1 = 0, m23 = 0;
            uint64_t t_last = globaltimer_ns();
            const uint32_t u_tile = sbase + OFF_U, s_tile = sbase + OFF_S;
            while (m23 < nch) {
                bool did = false;
                if (m23 < m1 && mbar_try_wait(&bar[B_UREADY], m23 & 1)) {
                    tc_fence_after();
                    issue_carry23(tmem, sbase + (m23 & 1) * STAGE_BYTES, u_tile);
                    tc_commit(&bar[B_CDONE]);
                    tc_commit(&bar[B_EMPTY0 + (m23 & 1)]);
                    ++m23;
                    did = true;
                } else if (m1 == m23 && m1 < wu && mbar_try_wait(&bar[B_SREADY], m1 & 1) &&
                           mbar_try_wait(&bar[B_WREADY], m1 & 1)) {
                    tc_fence_after();
                    issue_carry1(tmem, sbase + (m1 & 1) * STAGE_BYTES, s_tile);
                    tc_commit(&bar[B_ADONE]);
                    ++m1;
                    did = true;
                } else if (g < nch && g == wu &&
                           mbar_try_wait(&bar[B_FULL0 + (g & 1)], (g >> 1) & 1)) {
                    tc_fence_after();
                    issue_gram(tmem, sbase + (g & 1) * STAGE_BYTES);
                    tc_commit(&bar[B_GRAM]);
                    ++g;
                    did = true;
                } else if (wu < g && m1 >= wu && m23 >= wu - 1 &&
                           mbar_try_wait(&bar[B_PREP], wu & 1)) {
                    tc_fence_after();
                    issue_wy(tmem, sbase + (wu & 1) * STAGE_BYTES, wu);
                    tc_commit(&bar[B_WDONE]);
                    ++wu;
                    did = true;
                }
                const uint64_t now = globaltimer_ns();
                if (did) {
                    t_last = now;
                } else if (now - t_last > kWaitNs) {
                    record_failure(abort_flag, ST_MMA);
                    break;
                }
                if (*abort_flag) break;
            }
            // no MMA may be in flight when TMEM is freed
            tc_commit(&bar[B_DRAIN]);
            mbar_wait_bounded(&bar[B_DRAIN], 0, kWaitNs);
        }
    } else if (warp < 6) {
        // ------------------------------------------------------------ carry (128 threads)
        const int q = warp & 3;
        const int L = 32 * q + lane;  // TMEM lane = state row (Dk index) = token for L < 64
        const uint32_t lane_off = (uint32_t)(32 * q) << 16;
        const uint32_t s_tile = sbase + OFF_S, u_tile = sbase + OFF_U;
        float* gstate = a.state + ((size_t)(b * a.Hv + h) * 128 + L) * 128 + n0;
        __nv_bfloat16* gout = a.out + (size_t)(b * a.Hv + h) * S * 128 + n0;

        float Sm[NS];
        if (a.state_is_input) {
#pragma unroll
            for (int j = 0; j < NS; j += 4) {
                const float4 x = *reinterpret_cast<const float4*>(gstate + j);
                Sm[j] = x.x; Sm[j + 1] = x.y; Sm[j + 2] = x.z; Sm[j + 3] = x.w;
            }
        } else {
#pragma unroll
            for (int j = 0; j < NS; ++j) Sm[j] = 0.f;
        }
        write_row32(s_tile, L, 0, Sm);
        write_row32(s_tile, L, 4, Sm + 32);
        fence_proxy_async_smem();
        bar_sync(1, 128);
        if (L == 0 && nch > 0) mbar_arrive(&bar[B_SREADY]);

        for (int c = 0; c < nch; ++c) {
            const int s = c & 1;
            bool ok = mbar_wait_bounded(&bar[B_ADONE], c & 1, kWaitNs);
            if (!ok) record_failure(abort_flag, ST_CARRY);
            if (bar_any(1, 128, !ok || *abort_flag)) break;
            tc_fence_after();
            const float Gl = scal[s].Gl;
            if (L < 64) {
                // U = U~ - W S0 for token L
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    float ws[32], ut[32];
                    tmem_ld32(tmem + lane_off + TM_A + 32 * hh, ws);
                    tmem_ld32(tmem + lane_off + TM_U + 64 * s + 32 * hh, ut);
#pragma unroll
                    for (int j = 0; j < 32; ++j) ut[j] -= ws[j];
                    write_row32(u_tile, L, 4 * hh, ut);
                }
            }
            fence_proxy_async_smem();
            tc_fence_before();
            bar_sync(1, 128);
            if (L == 0) mbar_arrive(&bar[B_UREADY]);

            ok = mbar_wait_bounded(&bar[B_CDONE], c & 1, kWaitNs);
            if (!ok) record_failure(abort_flag, ST_CARRY);
            if (bar_any(1, 128, !ok || *abort_flag)) break;
            tc_fence_after();
            if (L >= 64) {
                // O = scale (Gamma Q S0 + P U) for token L - 64
                const int t = c * C + (L - 64);
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    float o[32];
                    tmem_ld32(tmem + lane_off + TM_A + 32 * hh, o);
                    if (t < S) {
                        uint4* dst = reinterpret_cast<uint4*>(gout + (size_t)t * 128 + 32 * hh);
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            uint4 w;
                            w.x = pack_bf16(a.scale * o[8 * j + 0], a.scale * o[8 * j + 1]);
                            w.y = pack_bf16(a.scale * o[8 * j + 2], a.scale * o[8 * j + 3]);
                            w.z = pack_bf16(a.scale * o[8 * j + 4], a.scale * o[8 * j + 5]);
                            w.w = pack_bf16(a.scale * o[8 * j + 6], a.scale * o[8 * j + 7]);
                            dst[j] = w;
                        }
                    }
                }
            }
            // S1 = Gamma_last S0 + K~^T U for state row L
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
            if (L == 0 && c + 1 < nch) mbar_arrive(&bar[B_SREADY]);
        }
        if (!*abort_flag) {
#pragma unroll
            for (int j = 0; j < NS; j += 4)
                *reinterpret_cast<float4*>(gstate + j) = make_float4(Sm[j], Sm[j + 1], Sm[j + 2], Sm[j + 3]);
        }
    } else {
        // ------------------------------------------------------------ prep (256 threads)
        const int P = tid - 192;
        const int wg = P >> 7;
        const int q = warp & 3;
        const int L = 32 * q + lane;
        const uint32_t lane_off = (uint32_t)(32 * q) << 16;
        const float* gp = a.g + (size_t)(b * a.Hv + h) * S;
        const float* bp = a.beta + (size_t)(b * a.Hv + h) * S;

        for (int c = 0; c < nch; ++c) {
            const int s = c & 1;
            const uint32_t st = sbase + s * STAGE_BYTES;
            StageScalars& sc = scal[s];
            bool ok = mbar_wait_bounded(&bar[B_FULL0 + s], (c >> 1) & 1, kWaitNs);
            if (!ok) record_failure(abort_flag, ST_PREP);
            if (bar_any(2, 256, !ok || *abort_flag)) break;

            // ---- decay tables: inclusive cumsum of g over the chunk (padding: g = beta = 0)
            float x = 0.f;
            if (P < 64) {
                const int t = c * C + P;
                x = (t < S) ? gp[t] : 0.f;
                sc.beta[P] = (t < S) ? bp[t] : 0.f;
#pragma unroll
                for (int off = 1; off < 32; off <<= 1) {
                    const float y = __shfl_up_sync(0xffffffffu, x, off);
                    if (lane >= off) x += y;
                }
                if (P == 31) scan_tot[0] = x;
            }
            bar_sync(2, 256);
            if (P < 64) {
                if (P >= 32) x += scan_tot[0];
                sc.gam[P] = x;
            }
            bar_sync(2, 256);
            if (P < 64) {
                const float gr = sc.gam[P], gl = sc.gam[C - 1];
                sc.ctab[P] = __expf(sc.gam[P | 15] - gr);
                sc.Gam[P] = __expf(gr);
                sc.kdec[P] = __expf(gl - gr);
                if ((P & 15) == 15) sc.endgam[P >> 4] = gr;
                if (P == C - 1) sc.Gl = __expf(gl);
            }
            bar_sync(2, 256);

            // ---- Gram -> P (bf16 tile) and A (fp32 blocks); Q scaled by Gamma in place
            ok = mbar_wait_bounded(&bar[B_GRAM], c & 1, kWaitNs);
            if (!ok) record_failure(abort_flag, ST_PREP);
            if (bar_any(2, 256, !ok || *abort_flag)) break;
            tc_fence_after();
            if (wg == 0) {
                const int r = L & 63, br = r >> 4, rl = r & 15;
                const bool isP = L < 64;
                const float gr = sc.gam[r];
                float dd[16];
#pragma unroll
                for (int jj = 0; jj < 16; ++jj) dd[jj] = (jj <= rl) ? __expf(gr - sc.gam[16 * br + jj]) : 0.f;
                const float scl = isP ? 1.f : sc.beta[r];
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    float gv[32];
                    tmem_ld32(tmem + lane_off + TM_G + 32 * hh, gv);
#pragma unroll
                    for (int bq = 0; bq < 2; ++bq) {
                        const int bj = 2 * hh + bq;
                        const float f = __expf(gr - sc.endgam[bj]);
#pragma unroll
                        for (int jj = 0; jj < 16; ++jj) {
                            const int j = 16 * bj + jj;
                            float d;
                            if (bj < br) d = f * sc.ctab[j];
                            else if (bj == br) d = dd[jj];
                            else d = 0.f;
                            // P keeps the diagonal, A is strictly lower
                            if (!isP && bj == br && jj == rl) d = 0.f;
                            gv[16 * bq + jj] *= d * scl;
                        }
                    }
                    if (isP) {
                        write_row32(st + OFF_P, r, 4 * hh, gv);
                    } else {
#pragma unroll
                        for (int bq = 0; bq < 2; ++bq) {
                            const int bj = 2 * hh + bq;
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
            } else {
                const int Pq = P - 128;
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const int k = Pq + 128 * i;
                    const int blk = k >> 9, row = (k >> 3) & 63, ch = k & 7;
                    const uint32_t addr = st + blk * BLK_STRIDE + OFF_Q + (row >> 3) * 1024 +
                                          (row & 7) * 128 + ch * 16;
                    scale_chunk(addr, sc.Gam[row]);
                }
            }
            tc_fence_before();
            bar_sync(2, 256);

            // ---- T = (I + A)^-1 in 16x16 blocks
            {
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
#pragma unroll
                    for (int r = 0; r < 16; ++r) Td[r * BS + cc] = xs[r];
                }
                bar_sync(2, 256);
                const int r = P >> 4, cc = P & 15;
                // level 1: T(i,i-1) = -T(i,i) A(i,i-1) T(i-1,i-1), i = 1..3
#pragma unroll
                for (int i = 1; i < 4; ++i) {
                    const float* Ar = Ab + bidx(i, i - 1) * 16 * BS + r * BS;
                    const float* Tc = Tb + bidx(i - 1, i - 1) * 16 * BS + cc;
                    float acc = 0.f;
#pragma unroll
                    for (int m = 0; m < 16; ++m) acc = fmaf(Ar[m], Tc[m * BS], acc);
                    Xb[(i - 1) * 16 * BS + r * BS + cc] = acc;
                }
                bar_sync(2, 256);
#pragma unroll
                for (int i = 1; i < 4; ++i) {
                    const float* Tr = Tb + bidx(i, i) * 16 * BS + r * BS;
                    const float* Xc = Xb + (i - 1) * 16 * BS + cc;
                    float acc = 0.f;
#pragma unroll
                    for (int m = 0; m < 16; ++m) acc = fmaf(Tr[m], Xc[m * BS], acc);
                    Tb[bidx(i, i - 1) * 16 * BS + r * BS + cc] = -acc;
                }
                bar_sync(2, 256);
                // level 2: T(j+2,j) = -T(j+2,j+2) (A(j+2,j) T(j,j) + A(j+2,j+1) T(j+1,j)), j = 0,1
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    const int i = j + 2;
                    const float* A0 = Ab + bidx(i, j) * 16 * BS + r * BS;
                    const float* A1 = Ab + bidx(i, j + 1) * 16 * BS + r * BS;
                    const float* T0 = Tb + bidx(j, j) * 16 * BS + cc;
                    const float* T1 = Tb + bidx(j + 1, j) * 16 * BS + cc;
                    float acc = 0.f;
#pragma unroll
                    for (int m = 0; m < 16; ++m) {
                        acc = fmaf(A0[m], T0[m * BS], acc);
                        acc = fmaf(A1[m], T1[m * BS], acc);
                    }
                    Xb[j * 16 * BS + r * BS + cc] = acc;
                }
                bar_sync(2, 256);
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    const int i = j + 2;
                    const float* Tr = Tb + bidx(i, i) * 16 * BS + r * BS;
                    const float* Xc = Xb + j * 16 * BS + cc;
                    float acc = 0.f;
#pragma unroll
                    for (int m = 0; m < 16; ++m) acc = fmaf(Tr[m], Xc[m * BS], acc);
                    Tb[bidx(i, j) * 16 * BS + r * BS + cc] = -acc;
                }
                bar_sync(2, 256);
                // level 3: T(3,0) = -T(3,3) (A(3,0) T(0,0) + A(3,1) T(1,0) + A(3,2) T(2,0))
                {
                    const float* A0 = Ab + bidx(3, 0) * 16 * BS + r * BS;
                    const float* A1 = Ab + bidx(3, 1) * 16 * BS + r * BS;
                    const float* A2 = Ab + bidx(3, 2) * 16 * BS + r * BS;
                    const float* T0 = Tb + bidx(0, 0) * 16 * BS + cc;
                    const float* T1 = Tb + bidx(1, 0) * 16 * BS + cc;
                    const float* T2 = Tb + bidx(2, 0) * 16 * BS + cc;
                    float acc = 0.f;
#pragma unroll
                    for (int m = 0; m < 16; ++m) {
                        acc = fmaf(A0[m], T0[m * BS], acc);
                        acc = fmaf(A1[m], T1[m * BS], acc);
                        acc = fmaf(A2[m], T2[m * BS], acc);
                    }
                    Xb[r * BS + cc] = acc;
                }
                bar_sync(2, 256);
                {
                    const float* Tr = Tb + bidx(3, 3) * 16 * BS + r * BS;
                    const float* Xc = Xb + cc;
                    float acc = 0.f;
#pragma unroll
                    for (int m = 0; m < 16; ++m) acc = fmaf(Tr[m], Xc[m * BS], acc);
                    Tb[bidx(3, 0) * 16 * BS + r * BS + cc] = -acc;
                }
                bar_sync(2, 256);
            }

            // ---- T_U = T diag(beta), T_W = T diag(beta Gamma) as bf16 tiles
            {
                const int r = P >> 2, qq = P & 3, i = r >> 4, rl = r & 15;
                float tu[16], tw[16];
#pragma unroll
                for (int jj = 0; jj < 16; ++jj) {
                    const int j = 16 * qq + jj;
                    const float t = (qq <= i) ? Tb[bidx(i, qq) * 16 * BS + rl * BS + jj] : 0.f;
                    tu[jj] = t * sc.beta[j];
                    tw[jj] = tu[jj] * sc.Gam[j];
                }
#pragma unroll
                for (int k = 0; k < 2; ++k) {
                    const float* u8 = tu + 8 * k;
                    const float* w8 = tw + 8 * k;
                    st_shared_v4(sw128_chunk(st + OFF_TU, r, 2 * qq + k), pack_bf16(u8[0], u8[1]),
                                 pack_bf16(u8[2], u8[3]), pack_bf16(u8[4], u8[5]), pack_bf16(u8[6], u8[7]));
                    st_shared_v4(sw128_chunk(st + OFF_TW, r, 2 * qq + k), pack_bf16(w8[0], w8[1]),
                                 pack_bf16(w8[2], w8[3]), pack_bf16(w8[4], w8[5]), pack_bf16(w8[6], w8[7]));
                }
            }
            fence_proxy_async_smem();
            bar_sync(2, 256);
            if (P == 0) mbar_arrive(&bar[B_PREP]);

            // ---- W (bf16) from TMEM; K scaled in place by exp(gamma_last - gamma_r)
            ok = mbar_wait_bounded(&bar[B_WDONE], c & 1, kWaitNs);
            if (!ok) record_failure(abort_flag, ST_PREP);
            if (bar_any(2, 256, !ok || *abort_flag)) break;
            tc_fence_after();
            if (wg == 0) {
                if (L < 64) {
#pragma unroll
                    for (int qd = 0; qd < 4; ++qd) {
                        float w[32];
                        tmem_ld32(tmem + lane_off + TM_W + 32 * qd, w);
                        write_row32(st + (qd >> 1) * BLK_STRIDE + OFF_W, L, 4 * (qd & 1), w);
                    }
                }
            } else {
                const int Pq = P - 128;
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const int k = Pq + 128 * i;
                    const int blk = k >> 9, row = (k >> 3) & 63, ch = k & 7;
                    const uint32_t addr = st + blk * BLK_STRIDE + OFF_K + (row >> 3) * 1024 +
                                          (row & 7) * 128 + ch * 16;
                    scale_chunk(addr, sc.kdec[row]);
                }
            }
            fence_proxy_async_smem();
            tc_fence_before();
            bar_sync(2, 256);
            if (P == 0) mbar_arrive(&bar[B_WREADY]);
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
