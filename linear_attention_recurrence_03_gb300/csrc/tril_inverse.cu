// tril_inverse.cu -- T = (I + A)^-1 for a batch of strictly lower-triangular 64 x 64 fp32
// matrices A, the intra-chunk inverse of the chunked prefill, by either of two methods
// ("GDN CTE Kernel API Reference", :param algorithm: -- the inverse method is selectable):
//
//   substitution  forward substitution, one thread per column of T in fp32:
//                 T[r][j] = -sum_{m<r} A[r][m] T[m][j] (T[j][j] = 1, zero above).
//   neumann       X = -A is nilpotent (X^64 = 0), so (I + A)^-1 = sum_{n<64} X^n. With
//                 Y = X^(2^k) and P = sum_{n<2^k} X^n, one product Y [Y | P] gives both
//                 X^(2^(k+1)) and the update P += Y P: six rounds from Y = X, P = I, all
//                 on the tensor cores (tf32 operands, fp32 accumulation).
//
// Neither is the prep kernel's blocked solve; they exist to compare the two algorithms
// as such (work, parallelism, accuracy) on this GPU.
#include "internal.h"

namespace gdn {
namespace {

constexpr int CN = 64;      // matrix size
constexpr int LDS_ = 65;    // padded row stride (floats) of the substitution tiles
constexpr int LDN = 68;     // padded row stride of the neumann tiles (fragment reads conflict-free)

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

__device__ __forceinline__ uint32_t tf32(float x) {
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
    return r;
}

__device__ __forceinline__ void mma_tf32_16x8x8(float (&d)[4], const uint32_t (&a)[4],
                                                uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// 4 warps, one matrix; warp w owns rows 16w .. 16w+15 of each product.
__global__ void __launch_bounds__(128) tril_neumann_kernel(const float* A, float* T) {
    __shared__ float Y[CN][LDN];
    __shared__ float P[CN][LDN];
    const int tid = threadIdx.x, w = tid >> 5, lane = tid & 31;
    const int g = lane >> 2, t = lane & 3;
    const float* a = A + (size_t)blockIdx.x * CN * CN;
    for (int i = tid; i < CN * CN; i += 128) {
        const int r = i / CN, c = i % CN;
        Y[r][c] = -a[i];
        P[r][c] = (r == c) ? 1.f : 0.f;
    }
    __syncthreads();
    const int r0 = 16 * w;
    for (int round = 0; round < 6; ++round) {
        const bool last = round == 5;  // X^64 = 0: the last round only updates P
        // A fragments of Y's rows r0 .. r0+15 for the eight k-steps
        uint32_t af[8][4];
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
            af[ks][0] = tf32(Y[r0 + g][8 * ks + t]);
            af[ks][1] = tf32(Y[r0 + g + 8][8 * ks + t]);
            af[ks][2] = tf32(Y[r0 + g][8 * ks + t + 4]);
            af[ks][3] = tf32(Y[r0 + g + 8][8 * ks + t + 4]);
        }
        // D = Y [Y | P]: column tiles 0-7 from Y, 8-15 from P
        float d[16][4];
#pragma unroll
        for (int nt = 0; nt < 16; ++nt) {
            d[nt][0] = d[nt][1] = d[nt][2] = d[nt][3] = 0.f;
            if (last && nt < 8) continue;
            const float(*B)[LDN] = nt < 8 ? Y : P;
            const int c = 8 * (nt & 7) + g;
#pragma unroll
            for (int ks = 0; ks < 8; ++ks)
                mma_tf32_16x8x8(d[nt], af[ks], tf32(B[8 * ks + t][c]), tf32(B[8 * ks + t + 4][c]));
        }
        __syncthreads();  // every warp has read Y and P
#pragma unroll
        for (int nt = 0; nt < 16; ++nt) {
            const int c = 8 * (nt & 7) + 2 * t;
            if (nt < 8) {
                if (!last) {
                    Y[r0 + g][c] = d[nt][0];
                    Y[r0 + g][c + 1] = d[nt][1];
                    Y[r0 + g + 8][c] = d[nt][2];
                    Y[r0 + g + 8][c + 1] = d[nt][3];
                }
            } else {
                P[r0 + g][c] += d[nt][0];
                P[r0 + g][c + 1] += d[nt][1];
                P[r0 + g + 8][c] += d[nt][2];
                P[r0 + g + 8][c + 1] += d[nt][3];
            }
        }
        __syncthreads();
    }
    float* out = T + (size_t)blockIdx.x * CN * CN;
    for (int i = tid; i < CN * CN; i += 128) out[i] = P[i / CN][i % CN];
}

}  // namespace

cudaError_t launch_tril_inverse(const float* A, float* T, int n, int algorithm,
                                cudaStream_t stream) {
    if (n == 0) return cudaSuccess;
    if (algorithm == 0)
        tril_subst_kernel<<<n, CN, 0, stream>>>(A, T);
    else
        tril_neumann_kernel<<<n, 128, 0, stream>>>(A, T);
    return cudaGetLastError();
}

}  // namespace gdn
