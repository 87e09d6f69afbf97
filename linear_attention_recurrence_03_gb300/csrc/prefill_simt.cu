// prefill_simt.cu -- chunked GDN prefill on the CUDA cores, computed in fp32.
//
// "GDN CTE Kernel API Reference": the recurrence in chunk-parallel form with an
// intra-chunk (I+A) inverse; the state is fp32 whatever the compute dtype (Notes).
// This kernel is the fp32 compute-dtype path and serves shapes the tensor-core kernel
// does not cover. All arithmetic is fp32 FFMA.
//
// Chunk algebra (derived from S_t = exp(g_t)(I - beta_t k_t k_t^T) S_{t-1} + beta_t k_t v_t^T,
// o_t = scale S_t^T q_t), for a chunk of C tokens, local index r, starting state S0:
//   gamma_r = sum_{i<=r} g_i,  Gamma_r = exp(gamma_r),  D[r,j] = exp(gamma_r - gamma_j)
//   A[r,j]  = beta_r (k_r . k_j) D[r,j]   (j < r),    T = (I + A)^-1
//   Y       = diag(beta) (V - diag(Gamma) K S0),       U = T Y
//   P[r,j]  = (q_r . k_j) D[r,j]          (j <= r)
//   O       = scale (diag(Gamma) Q S0 + P U)
//   S1      = Gamma_{C-1} S0 + sum_j exp(gamma_{C-1} - gamma_j) k_j u_j^T
// U = T Y is the same as U~ - W S0 with W = T diag(beta Gamma) K, U~ = T diag(beta) V.
// T itself is never formed: U solves (I + A) U = Y by forward substitution over the rows,
// U_r = Y_r - sum_{m<r} A[r,m] U_m, eight lanes per value column splitting each row's sum.
//
// A ragged last chunk is padded with tokens that have g = 0 and beta = 0: such a token
// leaves the state unchanged (alpha = 1, u = 0), so padding is exact.
//
// Grid: (ceil(Dv/32) value-column slices, Hv, B); the columns of S evolve
// independently (left-multiplication by (I - beta k k^T) never mixes them), so each
// CTA carries its own 32 columns of the state through the whole sequence in shared
// memory. A variable-length batch (B == 1, sequences packed along S by cu_seqlens) puts
// sequence n on grid row n; its chunks start at its first token.
#include "internal.h"

namespace gdn {
namespace {

constexpr int C = 64;      // chunk length
constexpr int NS = 32;     // state columns per CTA
constexpr int NT = 256;    // threads per CTA
constexpr int DKP = 132;    // row stride (floats) of the q/k tiles: 16-byte rows
constexpr int CP = C + 1;   // padded row stride of the C x C tiles
constexpr int NSP = NS + 4; // row stride of the 32-column tiles: 16-byte rows

struct Smem {
    float Q[C][DKP];    // q and k rows, zero from column Dk up to a multiple of 4
    float K[C][DKP];
    float Y[C][NSP];    // V slice, then Y = diag(beta)(V - diag(Gamma) K S0)
    float KS[C][NSP];
    float QS[C][NSP];
    float U[C][NSP];
    float S[kMaxHeadDim][NSP];
    float A[C][CP];
    float P[C][CP];
    float gam[C];
    float beta[C];
    float dec[C];       // exp(gamma_last - gamma_j)
    float Gam[C];       // exp(gamma_r)
};

__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }
__device__ __forceinline__ void store_as(float* p, float x) { *p = x; }
__device__ __forceinline__ void store_as(__nv_bfloat16* p, float x) { *p = __float2bfloat16_rn(x); }

template <typename Tin>
__global__ void __launch_bounds__(NT) prefill_simt_kernel(PrefillArgs a) {
    extern __shared__ float4 smem_raw[];
    Smem& s = *reinterpret_cast<Smem*>(smem_raw);
    const int tid = threadIdx.x;
    const int n0 = blockIdx.x * NS, h = blockIdx.y;
    const int Dk = a.Dk, Dv = a.Dv, S = a.S;
    const int Dk4 = (Dk + 3) & ~3;  // the q/k rows are read in groups of four
    const int nw = min(NS, Dv - n0);
    const int kh = h / (a.Hv / a.Hk);  // value head h reads key head h // (Hv/Hk)
    // this CTA's sequence: batch b (tensor row b, tokens 0 .. S-1), or packed sequence n
    // (tensor row 0, tokens cu[n] .. cu[n+1]-1; a malformed cu leaves every sequence empty)
    int b = blockIdx.z, t0 = 0, len = S, srow = blockIdx.z;
    if (a.cu_seqlens != nullptr) {
        const int n = blockIdx.z;
        const bool valid = a.table[a.N + 1] != 0;
        b = 0;
        t0 = valid ? a.cu_seqlens[n] : 0;
        len = valid ? a.cu_seqlens[n + 1] - t0 : 0;
    }

    const Tin* q = static_cast<const Tin*>(a.q) + ((size_t)b * a.Hk + kh) * (size_t)S * Dk +
                   (size_t)t0 * Dk;
    const Tin* k = static_cast<const Tin*>(a.k) + ((size_t)b * a.Hk + kh) * (size_t)S * Dk +
                   (size_t)t0 * Dk;
    const Tin* v = static_cast<const Tin*>(a.v) + ((size_t)b * a.Hv + h) * (size_t)S * Dv +
                   (size_t)t0 * Dv;
    const float* g = a.g + ((size_t)b * a.Hv + h) * (size_t)S + t0;
    const float* be = a.beta + ((size_t)b * a.Hv + h) * (size_t)S + t0;
    Tin* out = static_cast<Tin*>(a.out) + ((size_t)b * a.Hv + h) * (size_t)S * Dv +
               (size_t)t0 * Dv;
    float* st = a.state + ((size_t)srow * a.Hv + h) * (size_t)Dk * Dv;

    // Initial state: the supplied one, else zero with no load.
    for (int idx = tid; idx < kMaxHeadDim * NS; idx += NT) {
        const int i = idx / NS, n = idx % NS;
        s.S[i][n] = (a.state_is_input && i < Dk && n < nw) ? st[(size_t)i * Dv + n0 + n] : 0.f;
    }

    for (int c0 = 0; c0 < len; c0 += C) {
        const int L = min(C, len - c0);
        __syncthreads();
        for (int r = tid >> 6; r < C; r += NT >> 6) {
            for (int i = tid & 63; i < Dk4; i += 64) {
                const bool live = r < L && i < Dk;
                s.Q[r][i] = live ? to_f32(q[(size_t)(c0 + r) * Dk + i]) : 0.f;
                s.K[r][i] = live ? to_f32(k[(size_t)(c0 + r) * Dk + i]) : 0.f;
            }
        }
        for (int r = tid >> 5; r < C; r += NT >> 5) {
            const int n = tid & 31;
            s.Y[r][n] = (r < L && n < nw) ? to_f32(v[(size_t)(c0 + r) * Dv + n0 + n]) : 0.f;
        }
        if (tid < C) {
            s.gam[tid] = tid < L ? g[c0 + tid] : 0.f;
            s.beta[tid] = tid < L ? be[c0 + tid] : 0.f;
        }
        __syncthreads();
        // decay cumsum: two 32-wide warp scans joined by the first half's total
        if (tid < C) {
            float x = s.gam[tid];
            const int lane = tid & 31;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const float y = __shfl_up_sync(0xffffffffu, x, off);
                if (lane >= off) x += y;
            }
            s.gam[tid] = x;
        }
        __syncthreads();
        if (tid >= 32 && tid < C) s.gam[tid] += s.gam[31];
        __syncthreads();
        const float gl = s.gam[C - 1];
        if (tid < C) {
            s.dec[tid] = expf(gl - s.gam[tid]);
            s.Gam[tid] = expf(s.gam[tid]);
        }

        // A (strictly lower, beta and decay folded in) and P (lower incl. diagonal); every
        // dot product below runs as four interleaved partial sums
        {
            const int j = tid % C;
            for (int r = tid / C; r < C; r += NT / C) {
                float kk[4] = {0.f, 0.f, 0.f, 0.f}, qk[4] = {0.f, 0.f, 0.f, 0.f};
                if (j <= r) {
                    for (int i = 0; i < Dk4; i += 4) {
                        const float4 kj = *reinterpret_cast<const float4*>(&s.K[j][i]);
                        const float4 kr = *reinterpret_cast<const float4*>(&s.K[r][i]);
                        const float4 qr = *reinterpret_cast<const float4*>(&s.Q[r][i]);
                        kk[0] = fmaf(kr.x, kj.x, kk[0]);
                        kk[1] = fmaf(kr.y, kj.y, kk[1]);
                        kk[2] = fmaf(kr.z, kj.z, kk[2]);
                        kk[3] = fmaf(kr.w, kj.w, kk[3]);
                        qk[0] = fmaf(qr.x, kj.x, qk[0]);
                        qk[1] = fmaf(qr.y, kj.y, qk[1]);
                        qk[2] = fmaf(qr.z, kj.z, qk[2]);
                        qk[3] = fmaf(qr.w, kj.w, qk[3]);
                    }
                }
                const float kks = (kk[0] + kk[1]) + (kk[2] + kk[3]);
                const float qks = (qk[0] + qk[1]) + (qk[2] + qk[3]);
                const float d = (j <= r) ? expf(s.gam[r] - s.gam[j]) : 0.f;
                s.A[r][j] = (j < r) ? s.beta[r] * kks * d : 0.f;
                s.P[r][j] = qks * d;
            }
        }
        // K S0 and Q S0: thread = rows rb, rb + 32 and columns cb .. cb + 3, over four keys
        // at a time (16-byte loads of the q/k rows and of four state rows)
        {
            const int rb = tid >> 3, cb = 4 * (tid & 7);
            float ks[2][4] = {}, qs[2][4] = {};
            for (int i = 0; i < Dk4; i += 4) {
                float sv[4][4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float4 x = *reinterpret_cast<const float4*>(&s.S[i + e][cb]);
                    sv[e][0] = x.x, sv[e][1] = x.y, sv[e][2] = x.z, sv[e][3] = x.w;
                }
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    const int r = rb + 32 * hh;
                    const float4 kr = *reinterpret_cast<const float4*>(&s.K[r][i]);
                    const float4 qr = *reinterpret_cast<const float4*>(&s.Q[r][i]);
                    const float kv[4] = {kr.x, kr.y, kr.z, kr.w}, qv[4] = {qr.x, qr.y, qr.z, qr.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
#pragma unroll
                        for (int c = 0; c < 4; ++c) {
                            ks[hh][c] = fmaf(kv[e], sv[e][c], ks[hh][c]);
                            qs[hh][c] = fmaf(qv[e], sv[e][c], qs[hh][c]);
                        }
                    }
                }
            }
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    s.KS[rb + 32 * hh][cb + c] = ks[hh][c];
                    s.QS[rb + 32 * hh][cb + c] = qs[hh][c];
                }
            }
        }
        __syncthreads();
        // Y = diag(beta) (V - diag(Gamma) K S0)
        for (int idx = tid; idx < C * NS; idx += NT) {
            const int r = idx / NS, n = idx % NS;
            s.Y[r][n] = s.beta[r] * (s.Y[r][n] - s.Gam[r] * s.KS[r][n]);
        }
        __syncthreads();
        // U = (I + A)^-1 Y, row by row: warp w takes value columns 4w .. 4w + 3, lane
        // (column 4w + lane / 8, part lane % 8) the earlier rows part, part + 8, ...; three
        // shuffles join the parts. A padding row has A = 0 and Y = 0, hence U = 0.
        {
            const int lane = tid & 31;
            const int n = 4 * (tid >> 5) + (lane >> 3), part = lane & 7;
            for (int r = 0; r < C; ++r) {
                float acc = 0.f;
                for (int m = part; m < r; m += 8) acc = fmaf(s.A[r][m], s.U[m][n], acc);
                acc += __shfl_xor_sync(0xffffffffu, acc, 1);
                acc += __shfl_xor_sync(0xffffffffu, acc, 2);
                acc += __shfl_xor_sync(0xffffffffu, acc, 4);
                if (part == 0) s.U[r][n] = s.Y[r][n] - acc;
                __syncwarp();
            }
        }
        __syncthreads();
        // O = scale (diag(Gamma) Q S0 + P U), written for live rows and columns: thread =
        // rows rb, rb + 32 and columns cb .. cb + 3 (P is zero above the diagonal, so the
        // sum runs to the later row's diagonal for both)
        {
            const int rb = tid >> 3, cb = 4 * (tid & 7);
            float pu[2][4] = {};
            for (int j = 0; j <= rb + 32; ++j) {
                const float4 u = *reinterpret_cast<const float4*>(&s.U[j][cb]);
                const float uv[4] = {u.x, u.y, u.z, u.w};
                const float p0 = s.P[rb][j], p1 = s.P[rb + 32][j];
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    pu[0][c] = fmaf(p0, uv[c], pu[0][c]);
                    pu[1][c] = fmaf(p1, uv[c], pu[1][c]);
                }
            }
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                const int r = rb + 32 * hh;
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const int n = cb + c;
                    const float o = a.scale * fmaf(s.Gam[r], s.QS[r][n], pu[hh][c]);
                    if (r < L && n < nw) store_as(&out[(size_t)(c0 + r) * Dv + n0 + n], o);
                }
            }
        }
        // S1 = Gamma_last S0 + sum_j exp(gamma_last - gamma_j) k_j u_j^T: thread = state rows
        // ib + 32 m (m < 4) and columns cb .. cb + 3 (rows from Dk on stay zero)
        {
            const float Gl = expf(gl);
            const int ib = tid >> 3, cb = 4 * (tid & 7);
            float acc[4][4];
#pragma unroll
            for (int m = 0; m < 4; ++m) {
#pragma unroll
                for (int c = 0; c < 4; ++c) acc[m][c] = Gl * s.S[ib + 32 * m][cb + c];
            }
            for (int j = 0; j < C; ++j) {
                const float4 u = *reinterpret_cast<const float4*>(&s.U[j][cb]);
                const float uv[4] = {u.x, u.y, u.z, u.w};
                const float d = s.dec[j];
#pragma unroll
                for (int m = 0; m < 4; ++m) {
                    const int i = ib + 32 * m;
                    const float kd = i < Dk4 ? d * s.K[j][i] : 0.f;
#pragma unroll
                    for (int c = 0; c < 4; ++c) acc[m][c] = fmaf(kd, uv[c], acc[m][c]);
                }
            }
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                const int i = ib + 32 * m;
                if (i < Dk) {
#pragma unroll
                    for (int c = 0; c < 4; ++c) s.S[i][cb + c] = acc[m][c];
                }
            }
        }
    }
    __syncthreads();
    for (int idx = tid; idx < Dk * NS; idx += NT) {
        const int i = idx / NS, n = idx % NS;
        if (n < nw) st[(size_t)i * Dv + n0 + n] = s.S[i][n];
    }
}

}  // namespace

cudaError_t launch_prefill_simt(const PrefillArgs& a, bool bf16, cudaStream_t stream,
                                int* launched) {
    *launched = 0;
    const int rows = a.cu_seqlens ? a.N : a.B;
    if (rows == 0) return cudaSuccess;
    if (a.cu_seqlens) {
        const cudaError_t e = launch_varlen_setup(a, stream);
        if (e != cudaSuccess) return e;
        *launched = 1;
    }
    const dim3 grid((a.Dv + NS - 1) / NS, a.Hv, rows);
    const size_t smem = sizeof(Smem);
    cudaError_t e;
    if (bf16) {
        e = cudaFuncSetAttribute(prefill_simt_kernel<__nv_bfloat16>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        prefill_simt_kernel<__nv_bfloat16><<<grid, NT, smem, stream>>>(a);
    } else {
        e = cudaFuncSetAttribute(prefill_simt_kernel<float>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        prefill_simt_kernel<float><<<grid, NT, smem, stream>>>(a);
    }
    *launched += 1;
    return cudaGetLastError();
}

}  // namespace gdn
