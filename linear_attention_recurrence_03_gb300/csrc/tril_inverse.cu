// tril_inverse.cu -- T = (I + A)^-1 for a batch of strictly lower-triangular 64 x 64 fp32
// matrices A, the intra-chunk inverse of the chunked prefill, by either of two methods
// ("GDN CTE Kernel API Reference", :param algorithm: -- the inverse method is selectable):
//
//   substitution  forward substitution, one thread per column of T in fp32:
//                 T[r][j] = -sum_{m<r} A[r][m] T[m][j] (T[j][j] = 1, zero above).
//   neumann       X = -A is nilpotent (X^64 = 0), so (I + A)^-1 = sum_{n<64} X^n
//                 = (I + X)(I + X^2)(I + X^4) ... (I + X^32). With Y = X^(2^k) and P the
//                 product of the first k factors, one tensor-core product gives both
//                 Y^2 and Y P: six rounds from Y = X, P = I, on tcgen05 (kind::tf32,
//                 fp32 accumulation in tensor memory).
//
// Neither is the prep kernel's blocked solve; they exist to compare the two algorithms
// as such (work, parallelism, accuracy) on this GPU.
#include "internal.h"
#include "sm100_ptx.cuh"

namespace gdn {
namespace {

constexpr int CN = 64;      // matrix size
constexpr int LDS_ = 65;    // padded row stride (floats) of the substitution tiles

__global__ void __launch_bounds__(CN) tril_subst_kernel(const float* A, float* T) {
    __shared__ float As[CN][LDS_];
    __shared__ float Ts[CN][LDS_];
    const int j = threadIdx.x;
    const float* a = A + (size_t)blockIdx.x * CN * CN;
    for (int r = 0; r < CN; ++r) As[r][j] = a[r * CN + j];
    for (int r = 0; r < CN; ++r) Ts[r][j] = (r == j) ? 1.f : 0.f;
    __syncthreads();
    // rows in lockstep so every thread reads the same A[r][m] (a broadcast); column j has
    // zeros above its diagonal, so the full sums are exact
    for (int r = 1; r < CN; ++r) {
        float acc = 0.f;
        for (int m = 0; m < r; ++m) acc = fmaf(As[r][m], Ts[m][j], acc);
        if (r > j) Ts[r][j] = -acc;
    }
    float* t = T + (size_t)blockIdx.x * CN * CN;
    for (int r = 0; r < CN; ++r) t[r * CN + j] = Ts[r][j];
}

using namespace ptx;

// Status bit of a bounded wait that ran out (tril_take_status).
__device__ uint32_t g_tril_status = 0;
constexpr uint64_t kTrilWaitNs = 2000000000ull;

// The Neumann product, written transposed so that both factors of a round come out of one
// M = 128 product whose A operand is the previous round's result in tensor memory:
//   [Y^T; P^T] (128 x 64, TMEM)  x  Y^T (64 x 64, shared memory: Y row-major is Y^T as a
//   K-major B operand)  =  [(Y^2)^T; (Y P)^T].
// The next round's A is [(Y^2)^T; P^T + (Y P)^T]: the upper half is the accumulator as it
// stands, the lower half gets P^T added by the threads of lanes 64..127; the threads of
// lanes 0..63 write Y^2 row-major to shared memory as the next B. Two TMEM buffers of 64
// columns alternate between A and D. One CTA of 4 warps per matrix; warp w owns TMEM
// lanes 32w .. 32w + 31, thread = row m of the 128-row operand (a column of Y or of P).
constexpr int NEU_THREADS = 128;
constexpr uint32_t NEU_B_BYTES = 64 * 64 * 4;  // Y row-major, tf32, two 32-column k-blocks
// Dynamic shared memory: the B tile at a 1024-byte aligned offset (the 128-byte swizzle
// repeats every 1024 bytes), sized so that at most three CTAs (3 x 128 of the 512 TMEM
// columns) share an SM and no CTA waits in tcgen05.alloc.
constexpr uint32_t NEU_SMEM = 72 * 1024;
static_assert(NEU_B_BYTES + 1024 <= NEU_SMEM, "B tile and alignment slack");

__global__ void __launch_bounds__(NEU_THREADS) tril_neumann_tc_kernel(const float* A, float* T) {
    extern __shared__ __align__(1024) uint8_t neu_raw[];
    uint8_t* bsm = neu_raw + ((1024u - (smem_u32(neu_raw) & 1023u)) & 1023u);
    __shared__ uint64_t bar;
    __shared__ uint32_t tbase;
    __shared__ int failed;
    const int tid = threadIdx.x, warp = tid >> 5;
    const bool top = tid < 64;      // lanes 0..63: Y^T rows; 64..127: P^T rows
    const int m = tid & 63;         // column m of Y (top) or of P (bottom)
    const uint32_t lane_off = (uint32_t)(32 * warp) << 16;
    const uint32_t b_addr = smem_u32(bsm);
    const float* a = A + (size_t)blockIdx.x * 64 * 64;

    if (tid == 0) {
        mbar_init(&bar, 1);
        failed = 0;
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(&tbase, 128);
        tmem_relinquish();
    }
    // round 0 operands: A = [X^T; I], B = X row-major (X = -A)
    float x[64];
    if (top) {
#pragma unroll
        for (int r = 0; r < 64; ++r) x[r] = (r > m) ? -a[r * 64 + m] : 0.f;
#pragma unroll
        for (int r = 0; r < 64; ++r)
            *reinterpret_cast<float*>(bsm + sw128_offset32(r, m, 64)) = x[r];
    } else {
#pragma unroll
        for (int r = 0; r < 64; ++r) x[r] = (r == m) ? 1.f : 0.f;
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tm = tbase;
    {
        float h[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) h[j] = x[j];
        tmem_st32(tm + lane_off, h);
#pragma unroll
        for (int j = 0; j < 32; ++j) h[j] = x[32 + j];
        tmem_st32(tm + lane_off + 32, h);
        tmem_wait_st();
    }
    tc_fence_before();
    __syncthreads();

    constexpr uint32_t id = idesc_tf32(128, 64);
    const uint64_t bd = smem_desc_sw128(b_addr, 16, 1024);
    bool ok = true;
    for (int round = 0; round < 6 && ok; ++round) {
        const uint32_t ta = tm + 64u * (uint32_t)(round & 1);
        const uint32_t td = tm + 64u * (uint32_t)((round + 1) & 1);
        if (tid == 0) {
            tc_fence_after();
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const uint32_t off = (uint32_t)(k >> 2) * (64u * 128u) + (uint32_t)(k & 3) * 32u;
                mma_tf32_ts(td, ta + 8u * (uint32_t)k, bd + (off >> 4), id, k > 0);
            }
            tc_commit(&bar);
        }
        if (!mbar_wait_bounded(&bar, (uint32_t)(round & 1), kTrilWaitNs)) {
            atomicOr(&g_tril_status, 1u);
            failed = 1;
        }
        __syncthreads();
        ok = failed == 0;
        if (!ok) break;
        tc_fence_after();
        if (top) {
            if (round < 5) {
                // Y^2 row-major as the next B: this thread holds column m of Y^2
                float d[32];
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    tmem_ld32(td + lane_off + 32u * (uint32_t)hh, d);
#pragma unroll
                    for (int j = 0; j < 32; ++j)
                        *reinterpret_cast<float*>(bsm + sw128_offset32(32 * hh + j, m, 64)) = d[j];
                }
                fence_proxy_async_smem();
            }
        } else {
            // P^T += (Y P)^T in the D buffer, which becomes the next A
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                float d[32], p[32];
                tmem_ld32x2(td + lane_off + 32u * (uint32_t)hh, ta + lane_off + 32u * (uint32_t)hh,
                            d, p);
#pragma unroll
                for (int j = 0; j < 32; ++j) d[j] += p[j];
                tmem_st32(td + lane_off + 32u * (uint32_t)hh, d);
            }
            tmem_wait_st();
        }
        tc_fence_before();
        __syncthreads();
    }
    if (ok && !top) {
        // T = P: this thread holds column m of T (rows 0..63), in the last D buffer
        const uint32_t tf = tm + 64u * (uint32_t)(6 & 1);
        float* t = T + (size_t)blockIdx.x * 64 * 64;
        tc_fence_after();
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
            float d[32];
            tmem_ld32(tf + lane_off + 32u * (uint32_t)hh, d);
#pragma unroll
            for (int j = 0; j < 32; ++j) t[(32 * hh + j) * 64 + m] = d[j];
        }
    }
    if (!ok && tid == 0) mbar_wait_bounded(&bar, 0, kTrilWaitNs);  // nothing left in flight
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tm, 128);
    }
}

}  // namespace

cudaError_t launch_tril_inverse(const float* A, float* T, int n, int algorithm,
                                cudaStream_t stream) {
    if (n == 0) return cudaSuccess;
    if (algorithm == 0) {
        tril_subst_kernel<<<n, CN, 0, stream>>>(A, T);
    } else {
        static cudaError_t attr = cudaFuncSetAttribute(
            tril_neumann_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)NEU_SMEM);
        if (attr != cudaSuccess) return attr;
        tril_neumann_tc_kernel<<<n, NEU_THREADS, NEU_SMEM, stream>>>(A, T);
    }
    return cudaGetLastError();
}

uint32_t tril_take_status() {
    uint32_t bits = 0;
    if (cudaMemcpyFromSymbol(&bits, g_tril_status, sizeof(bits)) != cudaSuccess) return 0;
    if (bits != 0) {
        const uint32_t zero = 0;
        cudaMemcpyToSymbol(g_tril_status, &zero, sizeof(zero));
    }
    return bits;
}

}  // namespace gdn
