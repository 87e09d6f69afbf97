// decode.cu -- fused single-token GDN decode step ("GDN TKG Kernel API Reference").
//
// Per row bh (h = bh mod num_v_heads, Dimensions):
//   q^ = q / sqrt(|q|^2 + eps), k^ likewise           (l2norm(q,k), Background)
//   beta = sigmoid(b); g = -exp(A_log[h]) softplus(a + dt_bias[h]); alpha = exp(g)
//   S' = alpha (I - beta k^ k^^T) S + beta k^ v^T        (state [K, V] fp32)
//   o  = S'^T q^ / sqrt(K)                              (Notes: exp(g) and 1/sqrt(K) inside)
//   out = bf16( o / sqrt(mean(o^2) + eps) * norm_weight * z sigmoid(z) )  (RMSNormGated)
//
// The step is bound by HBM: each row streams its 64 KB state in and out once. Both
// reductions are taken from the OLD state in the single read pass (derived):
//   x = S^T k^, y = S^T q^,  u = beta (v - alpha x),
//   S' = alpha S + k^ u^T,   S'^T q^ = alpha y + u (k^ . q^),
// so the state is loaded once into registers, and written once from them.
//
// One CTA of 8 warps per row. Warp w holds rows w, w+8, ..., lane l holds four state
// columns (4l..4l+3 as one 16-byte vector when V == 128, else l, l+32, l+64, l+96).
// Cross-warp sums go through shared memory in a fixed order, so results are bitwise
// reproducible and do not depend on the grid ("LNC1 is byte-identical", Notes).
//
// Multi-token form (T >= 2 consecutive steps of the same rows in one call; an extension,
// not on the pages): the state stays on chip across the T tokens, so its 2 x 64 KB of HBM
// traffic is paid once per call; token t's inputs sit at offset t * BH rows. The tokens
// are taken in blocks of eight in chunk form (derived from the same step):
// with gamma_t = g_1 + ... + g_t (from the block start), Gamma_t = exp(gamma_t) and
// D[t][i] = exp(gamma_t - gamma_i) (i <= t, never above 1),
//   X[t] = S0^T k^_t, Y[t] = S0^T q^_t            (one pass over the old state, all t)
//   u_t = beta_t (v_t - Gamma_t X[t]) - sum_{i<t} beta_t D[t][i] (k^_t . k^_i) u_i
//                                                 (a unit lower-triangular solve)
//   S_t^T q^_t = Gamma_t Y[t] + sum_{i<=t} D[t][i] (k^_i . q^_t) u_i
//   S_last = Gamma_last S0 + sum_t D[last][t] k^_t u_t^T   (one update pass)
// instead of one reduction, solve and update per token.
#include "internal.h"
#include "sm100_ptx.cuh"

namespace gdn {
namespace {

using namespace ptx;

constexpr int NT = 256;
constexpr int NWARP = NT / 32;
constexpr int ROWS = kMaxHeadDim / NWARP;  // 16 state rows per warp at most

// The single step stages one token's inputs (TG = 1; the loops over tokens below run once)
constexpr int TG = 1;
struct Smem {
    // inputs of the token: q^, k^ (normalised in place), v, z
    float qn[TG][kMaxHeadDim];
    float kn[TG][kMaxHeadDim];
    float v[TG][kMaxHeadDim];
    float z[TG][kMaxHeadDim];
    float u[kMaxHeadDim];
    float red[2][NWARP][kMaxHeadDim];
    float scal[TG][5];  // 0: k^.q^, 1: beta, 2: alpha, 3: 1/|q|, 4: 1/|k|
    float part[NWARP];
};

// Two fp32 FMAs in one instruction (fma.rn.f32x2): d.x = a.x b.x + c.x, d.y = a.y b.y + c.y,
// each rounded once, exactly as two fmaf would.
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
    unsigned long long d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;"
        : "=l"(d)
        : "l"(*reinterpret_cast<const unsigned long long*>(&a)),
          "l"(*reinterpret_cast<const unsigned long long*>(&b)),
          "l"(*reinterpret_cast<const unsigned long long*>(&c)));
    return *reinterpret_cast<const float2*>(&d);
}

// Two fp32 products in one instruction (mul.rn.f32x2), each rounded as a * b.
__device__ __forceinline__ float2 fmul2(float2 a, float2 b) {
    unsigned long long d;
    asm("mul.rn.f32x2 %0, %1, %2;"
        : "=l"(d)
        : "l"(*reinterpret_cast<const unsigned long long*>(&a)),
          "l"(*reinterpret_cast<const unsigned long long*>(&b)));
    return *reinterpret_cast<const float2*>(&d);
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) x += __shfl_xor_sync(0xffffffffu, x, off);
    return x;
}

__device__ __forceinline__ float softplus_f(float x) {
    return fmaxf(x, 0.f) + log1pf(expf(-fabsf(x)));
}
__device__ __forceinline__ float sigmoid_f(float x) { return 1.f / (1.f + expf(-x)); }

template <bool VEC4>
__device__ __forceinline__ int col_of(int lane, int c) {
    return VEC4 ? 4 * lane + c : lane + 32 * c;
}

template <bool VEC4>
__global__ void __launch_bounds__(NT, 2) decode_kernel(DecodeArgs a) {
    __shared__ Smem s;
    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
    const int bh = blockIdx.x, h = bh % a.H;
    const int K = a.K, V = a.V;
    const float* S0 = a.state_in + (size_t)bh * K * V;
    float* S1 = a.state_out + (size_t)bh * K * V;
    const size_t BH = (size_t)a.BH;

    // 0. the state of the row a later CTA on this SM will take (pf_rows = the CTAs resident
    // at once) goes to L2 now, so the reads keep streaming while this CTA computes
    if (tid == 0 && a.pf_rows > 0 && bh + a.pf_rows < a.BH && (K * V) % 4 == 0)
        asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(
                         S0 + (size_t)a.pf_rows * K * V),
                     "r"((uint32_t)(K * V) * 4u)
                     : "memory");

    // 1. issue the state loads first: 16 rows x 4 columns per thread
    float st[ROWS][4];
#pragma unroll
    for (int m = 0; m < ROWS; ++m) {
        const int i = w + NWARP * m;
        if (VEC4) {
            float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
            if (i < K) x = __ldcs(reinterpret_cast<const float4*>(S0 + (size_t)i * V) + lane);
            st[m][0] = x.x; st[m][1] = x.y; st[m][2] = x.z; st[m][3] = x.w;
        } else {
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const int j = col_of<false>(lane, c);
                st[m][c] = (i < K && j < V) ? __ldcs(S0 + (size_t)i * V + j) : 0.f;
            }
        }
    }

    // 2. the token's inputs, staged in shared memory and turned into q^, k^, k^.q^, beta and
    // alpha (none of it depends on the state); the step then needs two barriers
    for (int t0 = 0; t0 < a.T; t0 += TG) {
        const int nt = min(TG, a.T - t0);
        if (t0 > 0) __syncthreads();  // the previous group's inputs are read
        for (int e = tid; e < nt * kMaxHeadDim; e += NT) {
            const int t = e / kMaxHeadDim, i = e % kMaxHeadDim;
            const size_t row = (size_t)(t0 + t) * BH + (size_t)bh;
            s.qn[t][i] = i < K ? __bfloat162float(a.q[row * K + i]) : 0.f;
            s.kn[t][i] = i < K ? __bfloat162float(a.k[row * K + i]) : 0.f;
            s.v[t][i] = i < V ? __bfloat162float(a.v[row * V + i]) : 0.f;
            s.z[t][i] = i < V ? __bfloat162float(a.z[row * V + i]) : 0.f;
        }
        __syncthreads();
        // l2 norms: job j = 2 t + (0: q, 1: k) on warp j mod NWARP (each sum in
        // lane-strided order); beta and alpha of token t on lane 0 of warp (2 nt + t) mod
        // NWARP, so that one token's work spreads over three warps
        for (int j = w; j < 2 * nt; j += NWARP) {
            const int t = j >> 1;
            const float* x = (j & 1) ? s.kn[t] : s.qn[t];
            float acc = 0.f;
            for (int i = lane; i < kMaxHeadDim; i += 32) acc = fmaf(x[i], x[i], acc);
            acc = warp_sum(acc);
            if (lane == 0) s.scal[t][3 + (j & 1)] = 1.f / sqrtf(acc + kEpsL2);
        }
        if (lane == 0) {
            for (int t = 0; t < nt; ++t) {
                if ((2 * nt + t) % NWARP != w) continue;
                const size_t row = (size_t)(t0 + t) * BH + (size_t)bh;
                s.scal[t][1] = sigmoid_f(__bfloat162float(a.b[row]));
                const float gg = -expf(a.A_log[h]) *
                                 softplus_f(__bfloat162float(a.a[row]) + a.dt_bias[h]);
                s.scal[t][2] = expf(gg);
            }
        }
        __syncthreads();
        for (int e = tid; e < nt * kMaxHeadDim; e += NT) {
            const int t = e / kMaxHeadDim, i = e % kMaxHeadDim;
            s.qn[t][i] *= s.scal[t][3];
            s.kn[t][i] *= s.scal[t][4];
        }
        __syncthreads();
        // k^.q^ of token t on warp t (read after the first barrier of the token loop)
        if (w < nt) {
            float acc = 0.f;
            for (int i = lane; i < kMaxHeadDim; i += 32) acc = fmaf(s.kn[w][i], s.qn[w][i], acc);
            acc = warp_sum(acc);
            if (lane == 0) s.scal[w][0] = acc;
        }
        for (int t = 0; t < nt; ++t) {
            const size_t row = (size_t)(t0 + t) * BH + (size_t)bh;  // this token's row
            // 3. per-warp partial x = S^T k^ and y = S^T q^ over this warp's rows
            {
                // column pairs (0,1), (2,3) in paired FMAs: each lane as fmaf, same order
                float2 x01 = make_float2(0.f, 0.f), x23 = x01, y01 = x01, y23 = x01;
#pragma unroll
                for (int m = 0; m < ROWS; ++m) {
                    const int i = w + NWARP * m;
                    const float ki = s.kn[t][i], qi = s.qn[t][i];  // zero beyond K
                    const float2 kk = make_float2(ki, ki), qq = make_float2(qi, qi);
                    const float2 s01 = make_float2(st[m][0], st[m][1]);
                    const float2 s23 = make_float2(st[m][2], st[m][3]);
                    x01 = ffma2(kk, s01, x01);
                    x23 = ffma2(kk, s23, x23);
                    y01 = ffma2(qq, s01, y01);
                    y23 = ffma2(qq, s23, y23);
                }
                const float px[4] = {x01.x, x01.y, x23.x, x23.y};
                const float py[4] = {y01.x, y01.y, y23.x, y23.y};
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const int j = col_of<VEC4>(lane, c);
                    s.red[0][w][j] = px[c];
                    s.red[1][w][j] = py[c];
                }
            }
            __syncthreads();
            // 4. u = beta (v - alpha x); o = (alpha y + u (k^.q^)) / sqrt(K)
            const float kq = s.scal[t][0], beta = s.scal[t][1], alpha = s.scal[t][2];
            float o = 0.f;
            if (tid < kMaxHeadDim) {
                const int j = tid;
                float x = 0.f, y = 0.f;
#pragma unroll
                for (int ww = 0; ww < NWARP; ++ww) { x += s.red[0][ww][j]; y += s.red[1][ww][j]; }
                const float u = (j < V) ? beta * (s.v[t][j] - alpha * x) : 0.f;
                s.u[j] = u;
                o = (j < V) ? (alpha * y + u * kq) / sqrtf((float)K) : 0.f;
                const float sq = warp_sum(o * o);
                if (lane == 0) s.part[w] = sq;
            }
            __syncthreads();
            // 5. RMSNormGated epilogue (threads 0..V-1), bf16 out
            if (tid < V) {
                float ms = 0.f;
#pragma unroll
                for (int ww = 0; ww < kMaxHeadDim / 32; ++ww) ms += s.part[ww];
                ms /= (float)V;
                const float zj = s.z[t][tid];
                const float y =
                    o * (1.f / sqrtf(ms + kEpsRms)) * a.norm_weight[tid] * (zj * sigmoid_f(zj));
                a.out[row * V + tid] = __float2bfloat16_rn(y);
            }
            // 6. S' = alpha S + k^ u^T in registers (rows beyond K stay zero). The next
            // token's partials overwrite s.red only after this thread's reads of s.u and
            // s.part, and its u after the next barrier.
            {
                const float2 u01 = make_float2(s.u[col_of<VEC4>(lane, 0)], s.u[col_of<VEC4>(lane, 1)]);
                const float2 u23 = make_float2(s.u[col_of<VEC4>(lane, 2)], s.u[col_of<VEC4>(lane, 3)]);
                const float2 aa = make_float2(alpha, alpha);
#pragma unroll
                for (int m = 0; m < ROWS; ++m) {
                    const int i = w + NWARP * m;
                    const float ki = s.kn[t][i];  // zero beyond K
                    const float2 kk = make_float2(ki, ki);
                    // alpha S + (k_i u_j), each product rounded first, as fmaf(alpha, S, k u)
                    const float2 n01 =
                        ffma2(aa, make_float2(st[m][0], st[m][1]), fmul2(kk, u01));
                    const float2 n23 =
                        ffma2(aa, make_float2(st[m][2], st[m][3]), fmul2(kk, u23));
                    st[m][0] = n01.x;
                    st[m][1] = n01.y;
                    st[m][2] = n23.x;
                    st[m][3] = n23.y;
                }
            }
        }
    }
    // 7. the state, written once
#pragma unroll
    for (int m = 0; m < ROWS; ++m) {
        const int i = w + NWARP * m;
        if (i >= K) continue;
        if (VEC4) {
            __stcs(reinterpret_cast<float4*>(S1 + (size_t)i * V) + lane,
                   make_float4(st[m][0], st[m][1], st[m][2], st[m][3]));
        } else {
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const int j = col_of<false>(lane, c);
                if (j < V) __stcs(S1 + (size_t)i * V + j, st[m][c]);
            }
        }
    }
}


// ---------------------------------------------------------------- several tokens

// The chunk form (two or more tokens per call), in blocks of TB = 8 tokens (the last block
// padded with zero tokens: beta = g = 0 and zero q, k, v, which add exact zeros). The two
// passes over the state run on the tensor cores through mma.sync m16n8k8 (tf32 operands,
// fp32 accumulate). One CTA of eight warps per row. The state lives in registers for the
// whole call as S^T, laid out as the accumulator of the update product: warp w holds value
// columns j = 16 w .. 16 w + 15 (the product's 16 rows) over all 128 key rows i (16 tiles
// of 8). The same registers are the A operand of the reductions X^T = S^T K and
// Y^T = S^T Q when the key index is taken in the order (k-slot c <-> i = 8 s + 2 c,
// slot c + 4 <-> i = 8 s + 2 c + 1) within tile s, which the B operands follow, so no state
// element ever moves between threads, and the state is read and written once per call.
//
// Per block, with the header's notation (rows of K, Q, V: the block's tokens):
//   X^T = S0^T K_raw, Y^T = S0^T Q_raw                   (k, q as read: bf16 values)
//   R = diag(beta) (V - diag(Gamma / |k|) X)               (|k|, |q|: the l2 norms)
//   (I + A) U = R,  A[t][i] = beta_t D[t][i] (k^_t . k^_i)  (i < t)
//   O = (diag(Gamma / |q|) Y + P U) / sqrt(K),  P[t][i] = D[t][i] (k^_i . q^_t)  (i <= t)
//   S_last = Gamma_last S0 + K_raw^T diag(D[last][t] / |k_t|) U
// The 8 x 8 Gram products come from one warp's m16n8k8 products; the solve, O and U_d run
// in fp32 on every lane for its two value columns (the quad's four lanes hold the eight
// tokens of a column and share them by shuffles).
// Precision: k and q enter the products as their bf16 values (exact in tf32), the norms as
// scalars afterwards; the state and U_d enter as two tf32 terms (the leading 11 bits and
// the next 11: within 2^-21 relative of the fp32 value); the increment is added to the fp32
// state with fmaf.
constexpr int TB = 8;
constexpr int MT = 256;
constexpr int MW = MT / 32;
constexpr int KP = kMaxHeadDim + 8;  // row stride of the token-major q and k tiles
constexpr uint32_t kTf32Mask = 0xffffe000u;

struct MultiSmem {
    float qr[TB][KP];  // q of the block's tokens as read (bf16 values), token-major
    float kr[TB][KP];  // k likewise
    float v[TB][kMaxHeadDim];
    float z[TB][kMaxHeadDim];
    float KK[TB][TB];  // kr_t . kr_i
    float QK[TB][TB];  // qr_t . kr_i
    float A[TB][TB];   // beta_t D[t][i] (k^_t . k^_i), i < t
    float P[TB][TB];   // D[t][i] (k^_i . q^_t), i <= t
    float beta[TB], gam[TB], Gam[TB], dlast[TB], invq[TB], invk[TB];
    float braw[TB], araw[TB];  // b and a of the block's tokens as read
    float hconst[2];           // A_log and dt_bias of the row's head
    float part[MW][TB];        // per-warp sums of o_t^2
};

// the tf32 value of x's leading 11 significant bits, and of the next 11 of the remainder
// (x - hi is exact in fp32)
__device__ __forceinline__ uint32_t tf32_hi(float x) { return __float_as_uint(x) & kTf32Mask; }
__device__ __forceinline__ uint32_t tf32_lo(float x, uint32_t hi) {
    return __float_as_uint(x - __uint_as_float(hi)) & kTf32Mask;
}

// d += a b: one m16n8k8 product, tf32 operands (every operand is passed with its low 13 bits
// clear), fp32 accumulate. Fragments (g = lane / 4, c = lane % 4): a = A[g][c], A[g+8][c],
// A[g][c+4], A[g+8][c+4]; b = B[c][g], B[c+4][g]; d = D[g][2c], D[g][2c+1], D[g+8][2c],
// D[g+8][2c+1].
__device__ __forceinline__ void mma8(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                     uint32_t b1) {
    asm("mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// An accumulator fragment (rows g, g + 8; columns 2c, 2c + 1) as the A operand of a product
// over those columns, in the permuted k order (slot c <-> column 2c, slot c + 4 <-> 2c + 1),
// split into its two tf32 terms.
__device__ __forceinline__ void acc_as_a(const float (&d)[4], uint32_t (&hi)[4], uint32_t (&lo)[4]) {
    const float x[4] = {d[0], d[2], d[1], d[3]};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        hi[e] = tf32_hi(x[e]);
        lo[e] = tf32_lo(x[e], hi[e]);
    }
}

// Eight consecutive bf16 elements e0 .. e0 + 7 of a row of n as floats (zero beyond n): one
// 16-byte load when `vec` (the row is 16-byte aligned) and all eight are in the row.
__device__ __forceinline__ void load8(const __nv_bfloat16* row, int n, int e0, bool vec,
                                      float (&x)[8]) {
    if (vec && e0 + 8 <= n) {
        const uint4 w = __ldcs(reinterpret_cast<const uint4*>(row + e0));
        const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            x[2 * e] = __uint_as_float(u[e] << 16);
            x[2 * e + 1] = __uint_as_float(u[e] & 0xffff0000u);
        }
    } else {
#pragma unroll
        for (int e = 0; e < 8; ++e) x[e] = e0 + e < n ? __bfloat162float(row[e0 + e]) : 0.f;
    }
}

// Eight bf16 elements (16 bytes of shared memory) as floats.
__device__ __forceinline__ void bf16x8_to_float(const __nv_bfloat16* p, float (&x)[8]) {
    const uint4 w = *reinterpret_cast<const uint4*>(p);
    const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        x[2 * e] = __uint_as_float(u[e] << 16);
        x[2 * e + 1] = __uint_as_float(u[e] & 0xffff0000u);
    }
}

__device__ __forceinline__ void zero8(float (&x)[8]) {
#pragma unroll
    for (int e = 0; e < 8; ++e) x[e] = 0.f;
}

// Dynamic shared memory of the pipelined form (1024-byte aligned): the state of the CTA's
// next row as four tensor-copy boxes of 32 value columns x 128 key rows with the 128-byte
// swizzle (the 16-byte chunk c of key row i sits at chunk c ^ (i mod 8), so the fragment
// loads out of it hit 32 distinct banks), and the q, k, v, z rows of its next block of
// tokens (one box each). Both copies fill zeros outside K x V and beyond the last token.
struct MultiPipe {
    float S[4][kMaxHeadDim][32];
    __nv_bfloat16 in[4][TB][kMaxHeadDim];  // q, k, v, z
    uint64_t bar[2];                       // 0: the state landed, 1: the inputs landed
};
constexpr uint32_t kStateBytes = sizeof(float) * 4 * kMaxHeadDim * 32;
constexpr uint32_t kInputBytes = sizeof(__nv_bfloat16) * 4 * TB * kMaxHeadDim;
// Limit of the bounded waits. GDN_TEST_STALL (a test-only build, never the library's
// default) shortens it to 5 ms and has each pipelined CTA never copy in the inputs of its
// second block, so that a test can see the wait run out and the status word report it.
#ifdef GDN_TEST_STALL
constexpr uint64_t kDecodeWaitNs = 5000000ull;
#else
constexpr uint64_t kDecodeWaitNs = 2000000000ull;
#endif

// Status bit of a bounded wait of this file that ran out (decode_take_status).
__device__ uint32_t g_decode_status = 0;

#ifdef GDN_TRACE
// Profiling aid, compiled only with -DGDN_TRACE: SM clock stamps of the phases of the
// first four rows of the multi-token CTAs 0 and 1, per warp (gdn_decode_trace_read).
__device__ unsigned long long g_dtrace[2][4][16][8];
#define DTR(ev)                                                                        \
    do {                                                                               \
        if (blockIdx.x < 2 && rit < 4 && lane == 0) g_dtrace[blockIdx.x][rit][ev][w] = clock64(); \
    } while (0)
#else
#define DTR(ev) \
    do {        \
    } while (0)
#endif

// PIPE: persistent CTAs (two per SM), each taking rows blockIdx.x, blockIdx.x + gridDim.x,
// ...: the next row's state and the next block's inputs are copied into shared memory by
// the tensor-copy engine while the current block computes (maps ms: the state as
// [BH][K][V] fp32, mq .. mz: the inputs as [T][BH][K or V] bf16; needs K, V multiples of
// 8). Otherwise one CTA per row, the state read straight into registers (any K, V <= 128).
// FULL: K = V = 128.
template <bool PIPE, bool FULL>
__global__ void __launch_bounds__(MT, 2)
    decode_multi_kernel(const __grid_constant__ CUtensorMap ms,
                        const __grid_constant__ CUtensorMap mq,
                        const __grid_constant__ CUtensorMap mk,
                        const __grid_constant__ CUtensorMap mv,
                        const __grid_constant__ CUtensorMap mz, DecodeArgs a) {
    __shared__ __align__(16) MultiSmem s;
    extern __shared__ __align__(1024) uint8_t dsm_raw[];
    MultiPipe& pp = *reinterpret_cast<MultiPipe*>(
        dsm_raw + ((1024u - (smem_u32(dsm_raw) & 1023u)) & 1023u));
    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
    const int g = lane >> 2, c = lane & 3;
    const int K = FULL ? kMaxHeadDim : a.K, V = FULL ? kMaxHeadDim : a.V;
    const int j0 = 16 * w;  // this warp's value columns j0 .. j0 + 15
    const size_t BH = (size_t)a.BH;
    const int G = PIPE ? (int)gridDim.x : a.BH;  // row stride of this CTA's rows
    const float rsK = 1.f / sqrtf((float)K);
    // norm weights of this thread's two columns
    const float nw0 = j0 + g < V ? a.norm_weight[j0 + g] : 0.f;
    const float nw1 = j0 + g + 8 < V ? a.norm_weight[j0 + g + 8] : 0.f;
    const bool vec_qk = (K % 8) == 0;  // rows of q, k (v, z) start 16-byte aligned
    const bool vec_vz = (V % 8) == 0;

    // copies of the pipelined form (one thread each): the state of row r, and the inputs
    // of the block of row r starting at token t0
    auto issue_state = [&](int r) {
        mbar_arrive_expect_tx(&pp.bar[0], kStateBytes);
        for (int b = 0; b < 4; ++b) tma_load_3d(&pp.S[b][0][0], &ms, &pp.bar[0], 32 * b, 0, r);
    };
    auto issue_inputs = [&](int r, int t0) {
        mbar_arrive_expect_tx(&pp.bar[1], kInputBytes);
        tma_load_3d(&pp.in[0][0][0], &mq, &pp.bar[1], 0, r, t0);
        tma_load_3d(&pp.in[1][0][0], &mk, &pp.bar[1], 0, r, t0);
        tma_load_3d(&pp.in[2][0][0], &mv, &pp.bar[1], 0, r, t0);
        tma_load_3d(&pp.in[3][0][0], &mz, &pp.bar[1], 0, r, t0);
    };
    // raw b and a of token `lane` of the block (r, t0), and on lanes 8, 9 A_log and dt_bias
    // of the row's head (warp 1), loaded a block ahead and carried to the block's start
    float nb = 0.f, na = 0.f;
    auto load_gates = [&](int r, int t0) {
        nb = na = 0.f;
        if (lane < TB && t0 + lane < a.T) {
            const size_t row = (size_t)(t0 + lane) * BH + (size_t)r;
            nb = __bfloat162float(a.b[row]);
            na = __bfloat162float(a.a[row]);
        } else if (lane == TB || lane == TB + 1) {
            nb = (lane == TB ? a.A_log : a.dt_bias)[r % a.H];
        }
    };
    uint32_t ph_state = 0, ph_in = 0;
    bool state_pending = false, in_pending = false, failed = false;
    if (PIPE) {
        if (tid == 0) {
            mbar_init(&pp.bar[0], 1);
            mbar_init(&pp.bar[1], 1);
            fence_mbar_init();
        }
        __syncthreads();
        if (tid == 0) {
            issue_state(blockIdx.x);
            issue_inputs(blockIdx.x, 0);
        }
        if (w == 1) load_gates(blockIdx.x, 0);
        state_pending = in_pending = true;
    }

    int rit = 0;
    for (int r = blockIdx.x; r < a.BH && !failed; r += G, ++rit) {
        const int h = r % a.H;
        // the state as S^T fragments: st[s][e] = S[i][j] with i = 8 s + 2 c + (e & 1),
        // j = j0 + g + 8 (e >> 1) (zero outside K x V)
        float st[16][4];
        if (!PIPE) {
            const float* S0 = a.state_in + (size_t)r * K * V;
#pragma unroll
            for (int s8 = 0; s8 < 16; ++s8) {
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int i = 8 * s8 + 2 * c + (e & 1), j = j0 + g + 8 * (e >> 1);
                    st[s8][e] = (i < K && j < V) ? __ldcs(S0 + (size_t)i * V + j) : 0.f;
                }
            }
        }
        for (int t0 = 0; t0 < a.T; t0 += TB) {
            const int nt = min(TB, a.T - t0);  // real tokens of this block
            if (PIPE) {
                // this block's gates (read a block ahead) and copies; one barrier also
                // orders the previous block's reads of the tiles before they are rewritten
                DTR(0);
                if (w == 1 && lane < TB) {
                    s.braw[lane] = nb;
                    s.araw[lane] = na;
                }
                if (w == 1 && (lane == TB || lane == TB + 1)) s.hconst[lane - TB] = nb;
                bool ok = mbar_wait_bounded(&pp.bar[1], ph_in, kDecodeWaitNs);
                if (t0 == 0) ok = ok && mbar_wait_bounded(&pp.bar[0], ph_state, kDecodeWaitNs);
                if (!__syncthreads_and(ok)) {
                    failed = true;
                    break;
                }
                DTR(1);
                ph_in ^= 1;
                in_pending = false;
                if (t0 == 0) {
                    ph_state ^= 1;
                    state_pending = false;
                    // element (i, j) of box j / 32 at row i, chunk ((j % 32) / 4) ^ (i % 8);
                    // i % 8 = 2 c + (e & 1) for every tile
                    const float* box = &pp.S[w >> 1][0][0];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int e0 = e & 1, ch = (4 * (w & 1) + 2 * (e >> 1) + (g >> 2)) ^ (2 * c + e0);
                        const float* src = box + (2 * c + e0) * 32 + 4 * ch + (g & 3);
#pragma unroll
                        for (int s8 = 0; s8 < 16; ++s8) st[s8][e] = src[256 * s8];
                    }
                }
            } else if (t0 > 0) {
                __syncthreads();  // the previous block's tiles are read
            }
            // 1. inputs: 16 x 8 elements per input row, the 32 rows (q, k, v, z of 8
            // tokens) in two rounds; q and k with their squared norms (16 lanes per row)
            {
                const int rr = tid >> 4, p = tid & 15, t = rr & 7;
                const bool isk = rr >= 8;
                float x[8];
                if (PIPE) {
                    bf16x8_to_float(&pp.in[isk ? 1 : 0][t][8 * p], x);
                } else if (t < nt) {
                    const size_t row = (size_t)(t0 + t) * BH + (size_t)r;
                    load8((isk ? a.k : a.q) + row * K, K, 8 * p, vec_qk, x);
                } else {
                    zero8(x);
                }
                float ss = 0.f;
#pragma unroll
                for (int e = 0; e < 8; ++e) ss = fmaf(x[e], x[e], ss);
#pragma unroll
                for (int off = 8; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
                if (p == 0) (isk ? s.invk : s.invq)[t] = 1.f / sqrtf(ss + kEpsL2);
                float* dst = isk ? &s.kr[t][8 * p] : &s.qr[t][8 * p];
                *reinterpret_cast<float4*>(dst) = make_float4(x[0], x[1], x[2], x[3]);
                *reinterpret_cast<float4*>(dst + 4) = make_float4(x[4], x[5], x[6], x[7]);
            }
            {
                const int rr = (tid >> 4) + 16, p = tid & 15, t = rr & 7;
                const bool isz = rr >= 24;
                float x[8];
                if (PIPE) {
                    bf16x8_to_float(&pp.in[isz ? 3 : 2][t][8 * p], x);
                } else if (t < nt) {
                    const size_t row = (size_t)(t0 + t) * BH + (size_t)r;
                    load8((isz ? a.z : a.v) + row * V, V, 8 * p, vec_vz, x);
                } else {
                    zero8(x);
                }
                float* dst = isz ? &s.z[t][8 * p] : &s.v[t][8 * p];
                *reinterpret_cast<float4*>(dst) = make_float4(x[0], x[1], x[2], x[3]);
                *reinterpret_cast<float4*>(dst + 4) = make_float4(x[4], x[5], x[6], x[7]);
            }
            // gates of token t on lane t of warp 1, the decay prefix gamma_t over the block
            if (w == 1) {
                const int t = lane & 7;
                float bt = 0.f, gt = 0.f;
                if (lane < TB && t < nt) {
                    float braw, araw, alog, dtb;
                    if (PIPE) {
                        braw = s.braw[t];
                        araw = s.araw[t];
                        alog = s.hconst[0];
                        dtb = s.hconst[1];
                    } else {
                        const size_t row = (size_t)(t0 + t) * BH + (size_t)r;
                        braw = __bfloat162float(a.b[row]);
                        araw = __bfloat162float(a.a[row]);
                        alog = a.A_log[h];
                        dtb = a.dt_bias[h];
                    }
                    bt = sigmoid_f(braw);
                    gt = -expf(alog) * softplus_f(araw + dtb);
                }
                float gm = gt;
#pragma unroll
                for (int off = 1; off < TB; off <<= 1) {
                    const float y = __shfl_up_sync(0xffffffffu, gm, off);
                    if (t >= off) gm += y;
                }
                const float glast = __shfl_sync(0xffffffffu, gm, TB - 1);
                if (lane < TB) {
                    s.beta[t] = bt;
                    s.gam[t] = gm;
                    s.Gam[t] = expf(gm);
                    s.dlast[t] = expf(glast - gm);
                }
            }
            DTR(2);
            __syncthreads();
            DTR(3);
            if (PIPE) {
                // the staged state and inputs are read: the next copies go out now
                int nr = r, nt0 = t0 + TB;
                if (nt0 >= a.T) nr = r + G, nt0 = 0;
                if (t0 == 0 && r + G < a.BH) {
                    if (tid == 32) issue_state(r + G);
                    state_pending = true;
                }
                if (nr < a.BH) {
#ifdef GDN_TEST_STALL
                    const bool skip = r == (int)blockIdx.x && t0 == 0;  // the second block
#else
                    constexpr bool skip = false;
#endif
                    if (tid == 32 && !skip) issue_inputs(nr, nt0);
                    if (w == 1) load_gates(nr, nt0);
                    in_pending = true;
                }
            }
            // 2. warp 0: the Gram products [K_raw; Q_raw] K_raw^T (m16n8k8 over the keys, four
            // partial sums), then the coefficients A and P (zero outside their triangles)
            if (w == 0) {
                float d[4][4] = {};
#pragma unroll
                for (int s8 = 0; s8 < 16; ++s8) {
                    const float2 ka = *reinterpret_cast<const float2*>(&s.kr[g][8 * s8 + 2 * c]);
                    const float2 qa = *reinterpret_cast<const float2*>(&s.qr[g][8 * s8 + 2 * c]);
                    const uint32_t af[4] = {__float_as_uint(ka.x), __float_as_uint(qa.x),
                                            __float_as_uint(ka.y), __float_as_uint(qa.y)};
                    mma8(d[s8 & 3], af, __float_as_uint(ka.x), __float_as_uint(ka.y));
                }
#pragma unroll
                for (int e = 0; e < 4; ++e) d[0][e] = (d[0][e] + d[1][e]) + (d[2][e] + d[3][e]);
                s.KK[g][2 * c] = d[0][0];
                s.KK[g][2 * c + 1] = d[0][1];
                s.QK[g][2 * c] = d[0][2];
                s.QK[g][2 * c + 1] = d[0][3];
                __syncwarp();
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int t = lane >> 2, i = 2 * c + e;
                    const float D = i <= t ? expf(s.gam[t] - s.gam[i]) : 0.f;
                    s.A[t][i] = i < t ? s.beta[t] * D * (s.invk[t] * s.invk[i]) * s.KK[t][i] : 0.f;
                    s.P[t][i] = D * (s.invk[i] * s.invq[t]) * s.QK[t][i];
                }
            }

            DTR(4);
            // 3. X^T = S0^T K_raw and Y^T = S0^T Q_raw for this warp's 16 columns (x[e], y[e]:
            // column j0 + g + 8 (e >> 1), token 2c + (e & 1))
            float x[4] = {0.f, 0.f, 0.f, 0.f}, y[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int s8 = 0; s8 < 16; ++s8) {
                uint32_t ah[4], al[4];
                acc_as_a(st[s8], ah, al);
                const float2 kb = *reinterpret_cast<const float2*>(&s.kr[g][8 * s8 + 2 * c]);
                const float2 qb = *reinterpret_cast<const float2*>(&s.qr[g][8 * s8 + 2 * c]);
                const uint32_t k0 = __float_as_uint(kb.x), k1 = __float_as_uint(kb.y);
                const uint32_t q0 = __float_as_uint(qb.x), q1 = __float_as_uint(qb.y);
                mma8(x, al, k0, k1);
                mma8(y, al, q0, q1);
                mma8(x, ah, k0, k1);
                mma8(y, ah, q0, q1);
            }
            DTR(5);
            __syncthreads();  // A, P and the scalars are written
            DTR(6);

            // 4. R^T (r[e]: column j0 + g + 8 (e >> 1), token 2c + (e & 1)); each lane gathers
            // the eight tokens of its two columns from its quad and solves (I + A) U = R by
            // forward substitution in fp32 (u0: column j0 + g, u1: column j0 + g + 8), then
            // forms its own tokens' outputs o = Gamma / |q| Y + P U (before the 1 / sqrt(K))
            // and U_d = D[last][t] / |k_t| u_t for the state update
            float ud[4], o[4];
            {
                float r[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int t = 2 * c + (e & 1), j = j0 + g + 8 * (e >> 1);
                    r[e] = s.beta[t] * (s.v[t][j] - s.Gam[t] * (s.invk[t] * x[e]));
                }
                float u0[TB], u1[TB];
#pragma unroll
                for (int cc = 0; cc < 4; ++cc) {
                    const int src = (lane & ~3) | cc;
                    u0[2 * cc] = __shfl_sync(0xffffffffu, r[0], src);
                    u0[2 * cc + 1] = __shfl_sync(0xffffffffu, r[1], src);
                    u1[2 * cc] = __shfl_sync(0xffffffffu, r[2], src);
                    u1[2 * cc + 1] = __shfl_sync(0xffffffffu, r[3], src);
                }
#pragma unroll
                for (int t = 1; t < TB; ++t) {
#pragma unroll
                    for (int i = 0; i < t; ++i) {
                        const float at = s.A[t][i];
                        u0[t] = fmaf(-at, u0[i], u0[t]);
                        u1[t] = fmaf(-at, u1[i], u1[t]);
                    }
                }
#pragma unroll
                for (int e0 = 0; e0 < 2; ++e0) {
                    const int t = 2 * c + e0;
                    float o0 = 0.f, o1 = 0.f;
#pragma unroll
                    for (int i = 0; i < TB; ++i) {
                        const float pt = s.P[t][i];
                        o0 = fmaf(pt, u0[i], o0);
                        o1 = fmaf(pt, u1[i], o1);
                    }
                    const float gy = s.Gam[t] * s.invq[t];
                    o[e0] = fmaf(gy, y[e0], o0);
                    o[2 + e0] = fmaf(gy, y[2 + e0], o1);
                    // u_t of this lane's token t = 2c + e0 (selects, no dynamic register index)
                    float a0 = u0[e0], a1 = u1[e0];
#pragma unroll
                    for (int cc = 1; cc < 4; ++cc) {
                        if (c == cc) {
                            a0 = u0[2 * cc + e0];
                            a1 = u1[2 * cc + e0];
                        }
                    }
                    const float sc = s.dlast[t] * s.invk[t];
                    ud[e0] = sc * a0;
                    ud[2 + e0] = sc * a1;
                }
            }
            // 5. o / sqrt(K); RMSNormGated per token over the V columns (the columns beyond V
            // hold zeros)
#pragma unroll
            for (int e = 0; e < 4; ++e) o[e] *= rsK;
            {
                float s0 = fmaf(o[0], o[0], o[2] * o[2]), s1 = fmaf(o[1], o[1], o[3] * o[3]);
#pragma unroll
                for (int off = 4; off < 32; off <<= 1) {
                    s0 += __shfl_xor_sync(0xffffffffu, s0, off);
                    s1 += __shfl_xor_sync(0xffffffffu, s1, off);
                }
                if (g == 0) {
                    s.part[w][2 * c] = s0;
                    s.part[w][2 * c + 1] = s1;
                }
            }
            DTR(7);
            __syncthreads();
            DTR(8);
            {
                float m0 = 0.f, m1 = 0.f;
#pragma unroll
                for (int ww = 0; ww < MW; ++ww) {
                    m0 += s.part[ww][2 * c];
                    m1 += s.part[ww][2 * c + 1];
                }
                const float rstd[2] = {1.f / sqrtf(m0 / (float)V + kEpsRms),
                                       1.f / sqrtf(m1 / (float)V + kEpsRms)};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int t = 2 * c + (e & 1), j = j0 + g + 8 * (e >> 1);
                    if (t < nt && j < V) {
                        const float zj = s.z[t][j];
                        const float yv = o[e] * rstd[e & 1] * ((e >> 1) ? nw1 : nw0) *
                                         (zj * sigmoid_f(zj));
                        const size_t row = (size_t)(t0 + t) * BH + (size_t)r;
                        a.out[row * V + j] = __float2bfloat16_rn(yv);
                    }
                }
            }
            DTR(9);
            // 6. S^T <- Gamma_last S^T + U_d^T K_raw, tile by tile (B: k of tokens 2c, 2c + 1)
            {
                uint32_t uh[4], ul[4];
                acc_as_a(ud, uh, ul);
                const float Gl = s.Gam[TB - 1];
#pragma unroll
                for (int s8 = 0; s8 < 16; ++s8) {
                    const uint32_t b0 = __float_as_uint(s.kr[2 * c][8 * s8 + g]);
                    const uint32_t b1 = __float_as_uint(s.kr[2 * c + 1][8 * s8 + g]);
                    float d[4] = {0.f, 0.f, 0.f, 0.f};
                    mma8(d, ul, b0, b1);
                    mma8(d, uh, b0, b1);
#pragma unroll
                    for (int e = 0; e < 4; ++e) st[s8][e] = fmaf(Gl, st[s8][e], d[e]);
                }
            }
        }
        DTR(10);
        if (failed) break;
        // the state, written once
        float* S1 = a.state_out + (size_t)r * K * V;
#pragma unroll
        for (int s8 = 0; s8 < 16; ++s8) {
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int i = 8 * s8 + 2 * c + (e & 1), j = j0 + g + 8 * (e >> 1);
                if (i < K && j < V) __stcs(S1 + (size_t)i * V + j, st[s8][e]);
            }
        }
        DTR(11);
    }
    if (PIPE && failed && tid == 0) {
        // a copy gave up: the copies still in flight land before the CTA leaves
        atomicOr(&g_decode_status, 1u);
        if (state_pending) mbar_wait_bounded(&pp.bar[0], ph_state, kDecodeWaitNs);
        if (in_pending) mbar_wait_bounded(&pp.bar[1], ph_in, kDecodeWaitNs);
    }
}

// 3-D tensor map over [d2][d1][d0] (d0 contiguous) with a box of b0 x b1 x b2
bool encode_map(CUtensorMap* m, CUtensorMapDataType type, int esize, const void* base,
                uint64_t d0, uint64_t d1, uint64_t d2, uint32_t b0, uint32_t b1, uint32_t b2,
                CUtensorMapSwizzle swz) {
    auto fn = tensor_map_encoder();
    if (!fn) return false;
    cuuint64_t dims[3] = {d0, d1, d2};
    cuuint64_t strides[2] = {d0 * esize, d0 * d1 * esize};
    cuuint32_t box[3] = {b0, b1, b2};
    cuuint32_t es[3] = {1, 1, 1};
    return fn(m, type, 3, const_cast<void*>(base), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <bool PIPE, bool FULL>
cudaError_t launch_multi(const DecodeArgs& a, int sms, cudaStream_t stream) {
    CUtensorMap ms{}, mq{}, mk{}, mv{}, mz{};
    if constexpr (!PIPE) {
        decode_multi_kernel<false, FULL><<<a.BH, MT, 0, stream>>>(ms, mq, mk, mv, mz, a);
        return cudaGetLastError();
    }
    constexpr auto BF = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    const uint64_t T = (uint64_t)a.T, BH = (uint64_t)a.BH, K = (uint64_t)a.K, V = (uint64_t)a.V;
    if (!encode_map(&ms, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, a.state_in, V, K, BH, 32,
                    kMaxHeadDim, 1, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_map(&mq, BF, 2, a.q, K, BH, T, kMaxHeadDim, 1, TB, CU_TENSOR_MAP_SWIZZLE_NONE) ||
        !encode_map(&mk, BF, 2, a.k, K, BH, T, kMaxHeadDim, 1, TB, CU_TENSOR_MAP_SWIZZLE_NONE) ||
        !encode_map(&mv, BF, 2, a.v, V, BH, T, kMaxHeadDim, 1, TB, CU_TENSOR_MAP_SWIZZLE_NONE) ||
        !encode_map(&mz, BF, 2, a.z, V, BH, T, kMaxHeadDim, 1, TB, CU_TENSOR_MAP_SWIZZLE_NONE))
        return cudaErrorInvalidValue;
    constexpr int smem = (int)sizeof(MultiPipe) + 1024;  // + alignment slack
    static cudaError_t attr = cudaFuncSetAttribute(decode_multi_kernel<true, FULL>,
                                                   cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (attr != cudaSuccess) return attr;
    const int grid = min(a.BH, 2 * max(sms, 1));
    decode_multi_kernel<true, FULL><<<grid, MT, smem, stream>>>(ms, mq, mk, mv, mz, a);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_decode(const DecodeArgs& args, cudaStream_t stream) {
    if (args.BH == 0 || args.T == 0) return cudaSuccess;
    constexpr int kMaxDevices = 64;
    static int sms_of[kMaxDevices] = {};
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) == cudaSuccess && dev >= 0 && dev < kMaxDevices) {
        if (sms_of[dev] == 0) cudaDeviceGetAttribute(&sms_of[dev], cudaDevAttrMultiProcessorCount, dev);
        sms = sms_of[dev];
    }
    // Two or more tokens: the chunk form (blocks of eight), pipelined when K and V are
    // multiples of 8 (the tensor copies' 16-byte rows). Measured at BH = 8192 against
    // the single step's register loop run token after token: T = 2 0.213 against 0.212 ms,
    // T = 3 0.214 against 0.284, T = 4 0.214 against 0.318.
    if (args.T > 1) {
        if (args.K == kMaxHeadDim && args.V == kMaxHeadDim)
            return launch_multi<true, true>(args, sms, stream);
        if (args.K % 8 == 0 && args.V % 8 == 0) return launch_multi<true, false>(args, sms, stream);
        return launch_multi<false, false>(args, sms, stream);
    }
    // the single step: two CTAs per SM are resident (launch bounds), and the state of the
    // rows that far ahead is prefetched into L2
    DecodeArgs a = args;
    a.pf_rows = 2 * sms;
    if (a.V == kMaxHeadDim) decode_kernel<true><<<a.BH, NT, 0, stream>>>(a);
    else decode_kernel<false><<<a.BH, NT, 0, stream>>>(a);
    return cudaGetLastError();
}

uint32_t decode_take_status() {
    uint32_t bits = 0;
    if (cudaMemcpyFromSymbol(&bits, g_decode_status, sizeof(bits)) != cudaSuccess) return 0;
    if (bits != 0) {
        const uint32_t zero = 0;
        cudaMemcpyToSymbol(g_decode_status, &zero, sizeof(zero));
    }
    return bits;
}

}  // namespace gdn

#ifdef GDN_TRACE
extern "C" int gdn_decode_trace_read(unsigned long long* dst) {
    return cudaMemcpyFromSymbol(dst, gdn::g_dtrace, sizeof(gdn::g_dtrace)) == cudaSuccess ? 0 : 1;
}
#endif
