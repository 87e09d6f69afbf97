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
// Multi-token form (T consecutive steps of the same rows in one call; an extension, not
// on the pages): the state stays in registers across the T tokens, so its 2 x 64 KB of
// HBM traffic is paid once per call; token t's inputs sit at offset t * BH rows. Up to
// four tokens run one after another on the register state; more are taken in blocks of
// eight in chunk form (derived from the same step):
// with gamma_t = g_1 + ... + g_t (from the block start), Gamma_t = exp(gamma_t) and
// D[t][i] = exp(gamma_t - gamma_i) (i <= t, never above 1),
//   X[t] = S0^T k^_t, Y[t] = S0^T q^_t            (one pass over the old state, all t)
//   u_t = beta_t (v_t - Gamma_t X[t]) - sum_{i<t} beta_t D[t][i] (k^_t . k^_i) u_i
//                                                 (a unit lower-triangular solve)
//   S_t^T q^_t = Gamma_t Y[t] + sum_{i<=t} D[t][i] (k^_i . q^_t) u_i
//   S_last = Gamma_last S0 + sum_t D[last][t] k^_t u_t^T   (one update pass)
// instead of one reduction, solve and update per token.
#include "internal.h"

namespace gdn {
namespace {

constexpr int NT = 256;
constexpr int NWARP = NT / 32;
constexpr int ROWS = kMaxHeadDim / NWARP;  // 16 state rows per warp at most

// TG: tokens whose inputs are staged together (1 for a single step, NWARP otherwise)
template <int TG>
struct Smem {
    // inputs of up to TG tokens: q^, k^ (normalised in place), v, z
    float qn[TG][kMaxHeadDim];
    float kn[TG][kMaxHeadDim];
    float v[TG][kMaxHeadDim];
    float z[TG][kMaxHeadDim];
    float u[kMaxHeadDim];
    float red[2][NWARP][kMaxHeadDim];
    float scal[TG][5];  // 0: k^.q^, 1: beta, 2: alpha, 3: 1/|q|, 4: 1/|k|
    float part[NWARP];
};

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

template <bool VEC4, int TG>
__global__ void __launch_bounds__(NT, 2) decode_kernel(DecodeArgs a) {
    __shared__ Smem<TG> s;
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

    // 2. the inputs of TG tokens at a time, staged in shared memory and turned into q^, k^,
    // k^.q^, beta and alpha (none of it depends on the state); each token then needs two
    // barriers
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
                float px[4] = {0.f, 0.f, 0.f, 0.f}, py[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int m = 0; m < ROWS; ++m) {
                    const int i = w + NWARP * m;
                    const float ki = s.kn[t][i], qi = s.qn[t][i];  // zero beyond K
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        px[c] = fmaf(ki, st[m][c], px[c]);
                        py[c] = fmaf(qi, st[m][c], py[c]);
                    }
                }
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
#pragma unroll
            for (int m = 0; m < ROWS; ++m) {
                const int i = w + NWARP * m;
                const float ki = s.kn[t][i];  // zero beyond K
#pragma unroll
                for (int c = 0; c < 4; ++c)
                    st[m][c] = fmaf(alpha, st[m][c], ki * s.u[col_of<VEC4>(lane, c)]);
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

constexpr int TB = 8;   // tokens per block of the chunk form
constexpr int RG = 4;   // tokens per reduction group (partials held in registers)
constexpr int MROWS = kMaxHeadDim / NWARP;  // 16 contiguous state rows per warp

struct MultiSmem {
    float qn[TB][kMaxHeadDim];   // q^ (normalised in place); zero for padding tokens
    float kn[TB][kMaxHeadDim];   // k^
    float v[TB][kMaxHeadDim];
    float z[TB][kMaxHeadDim];
    float X[TB][kMaxHeadDim];    // S0^T k^_t, then u_t
    float Y[TB][kMaxHeadDim];    // S0^T q^_t, then the un-normalised o_t
    float red[2 * RG][NWARP][kMaxHeadDim];
    float A[TB][TB];             // beta_t D[t][i] (k^_t . k^_i), i < t
    float P[TB][TB];             // D[t][i] (k^_i . q^_t), i <= t
    float kk[TB][TB], kq[TB][TB];
    float gam[TB], Gam[TB], dlast[TB], beta[TB], g[TB], inv[2][TB];
    float ssq[TB][kMaxHeadDim / 32];
};

// NB tokens per block (the last block of a call may hold fewer real tokens, the rest
// padded with zero rows, which contribute exactly nothing). Warp w holds the
// contiguous state rows 16 w .. 16 w + 15, lane l four columns (as in the single step), so
// that a warp's slice of k^ or q^ is four 16-byte broadcast loads.
template <bool VEC4, int NB>
__global__ void __launch_bounds__(NT, 2) decode_multi_kernel(DecodeArgs a) {
    extern __shared__ __align__(16) uint8_t smraw[];
    MultiSmem& s = *reinterpret_cast<MultiSmem*>(smraw);
    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
    const int bh = blockIdx.x, h = bh % a.H;
    const int K = a.K, V = a.V;
    const float* S0 = a.state_in + (size_t)bh * K * V;
    float* S1 = a.state_out + (size_t)bh * K * V;
    const size_t BH = (size_t)a.BH;
    const float rsK = 1.f / sqrtf((float)K);
    const int r0w = MROWS * w;  // this warp's first state row

    // the state, loaded once: 16 rows x 4 columns per thread
    float st[MROWS][4];
#pragma unroll
    for (int m = 0; m < MROWS; ++m) {
        const int i = r0w + m;
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

    for (int t0 = 0; t0 < a.T; t0 += NB) {
        const int nt = min(NB, a.T - t0);  // real tokens of this block
        if (t0 > 0) __syncthreads();      // the previous block's inputs and u are read
        // 1. inputs of the block (padding tokens: zero rows, beta = 0, g = 0)
        for (int e = tid; e < NB * kMaxHeadDim; e += NT) {
            const int t = e / kMaxHeadDim, i = e % kMaxHeadDim;
            const size_t row = (size_t)(t0 + t) * BH + (size_t)bh;
            const bool real = t < nt;
            s.qn[t][i] = (real && i < K) ? __bfloat162float(a.q[row * K + i]) : 0.f;
            s.kn[t][i] = (real && i < K) ? __bfloat162float(a.k[row * K + i]) : 0.f;
            s.v[t][i] = (real && i < V) ? __bfloat162float(a.v[row * V + i]) : 0.f;
            s.z[t][i] = (real && i < V) ? __bfloat162float(a.z[row * V + i]) : 0.f;
        }
        if (tid < NB) {
            const size_t row = (size_t)(t0 + tid) * BH + (size_t)bh;
            const bool real = tid < nt;
            s.beta[tid] = real ? sigmoid_f(__bfloat162float(a.b[row])) : 0.f;
            s.g[tid] = real ? -expf(a.A_log[h]) *
                                  softplus_f(__bfloat162float(a.a[row]) + a.dt_bias[h])
                            : 0.f;
        }
        __syncthreads();
        // 2. the l2 norms (job j: token j / 2, q or k), the decay prefix (one thread)
        for (int j = w; j < 2 * NB; j += NWARP) {
            const float* x = (j & 1) ? s.kn[j >> 1] : s.qn[j >> 1];
            float acc = 0.f;
#pragma unroll
            for (int i = lane; i < kMaxHeadDim; i += 32) acc = fmaf(x[i], x[i], acc);
            acc = warp_sum(acc);
            if (lane == 0) s.inv[j & 1][j >> 1] = 1.f / sqrtf(acc + kEpsL2);
        }
        if (tid == NT - 1) {
            float gm = 0.f;
#pragma unroll
            for (int t = 0; t < NB; ++t) {
                gm += s.g[t];
                s.gam[t] = gm;
                s.Gam[t] = expf(gm);
            }
#pragma unroll
            for (int t = 0; t < NB; ++t) s.dlast[t] = expf(gm - s.gam[t]);
        }
        __syncthreads();
        for (int e = tid; e < NB * kMaxHeadDim; e += NT) {
            const int t = e / kMaxHeadDim, i = e % kMaxHeadDim;
            s.qn[t][i] *= s.inv[0][t];
            s.kn[t][i] *= s.inv[1][t];
        }
        __syncthreads();
        // 3. the small Gram products k^_t . k^_i and k^_i . q^_t (i <= t), one warp per job
        for (int j = w; j < NB * NB; j += NWARP) {
            const int t = j / NB, i = j % NB;
            if (i > t) continue;
            float akk = 0.f, akq = 0.f;
#pragma unroll
            for (int e = lane; e < kMaxHeadDim; e += 32) {
                akk = fmaf(s.kn[t][e], s.kn[i][e], akk);
                akq = fmaf(s.kn[i][e], s.qn[t][e], akq);
            }
            akk = warp_sum(akk);
            akq = warp_sum(akq);
            if (lane == 0) {
                s.kk[t][i] = akk;
                s.kq[t][i] = akq;
            }
        }
        // 4. X[t] = S0^T k^_t and Y[t] = S0^T q^_t from the registers, RG tokens at a time
#pragma unroll
        for (int r0 = 0; r0 < NB; r0 += RG) {
            constexpr int NR = NB < RG ? NB : RG;
            if (r0 > 0) __syncthreads();  // s.red of the previous group is read
            float px[NR][4], py[NR][4];
#pragma unroll
            for (int r = 0; r < NR; ++r)
#pragma unroll
                for (int c = 0; c < 4; ++c) px[r][c] = py[r][c] = 0.f;
#pragma unroll
            for (int m4 = 0; m4 < MROWS; m4 += 4) {
#pragma unroll
                for (int r = 0; r < NR; ++r) {
                    const float4 k4 = *reinterpret_cast<const float4*>(&s.kn[r0 + r][r0w + m4]);
                    const float4 q4 = *reinterpret_cast<const float4*>(&s.qn[r0 + r][r0w + m4]);
                    const float kv[4] = {k4.x, k4.y, k4.z, k4.w};
                    const float qv[4] = {q4.x, q4.y, q4.z, q4.w};
#pragma unroll
                    for (int mm = 0; mm < 4; ++mm)
#pragma unroll
                        for (int c = 0; c < 4; ++c) {
                            px[r][c] = fmaf(kv[mm], st[m4 + mm][c], px[r][c]);
                            py[r][c] = fmaf(qv[mm], st[m4 + mm][c], py[r][c]);
                        }
                }
            }
#pragma unroll
            for (int r = 0; r < NR; ++r) {
                if (VEC4) {  // this lane's four adjacent columns as one vector
                    *reinterpret_cast<float4*>(&s.red[2 * r][w][4 * lane]) =
                        make_float4(px[r][0], px[r][1], px[r][2], px[r][3]);
                    *reinterpret_cast<float4*>(&s.red[2 * r + 1][w][4 * lane]) =
                        make_float4(py[r][0], py[r][1], py[r][2], py[r][3]);
                } else {
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        const int j = col_of<false>(lane, c);
                        s.red[2 * r][w][j] = px[r][c];
                        s.red[2 * r + 1][w][j] = py[r][c];
                    }
                }
            }
            __syncthreads();
            // the sums over the warps, in a fixed order: thread (job, column)
#pragma unroll
            for (int e = tid; e < 2 * NR * kMaxHeadDim; e += NT) {
                const int jb = e / kMaxHeadDim, j = e % kMaxHeadDim;
                float acc = 0.f;
#pragma unroll
                for (int ww = 0; ww < NWARP; ++ww) acc += s.red[jb][ww][j];
                if (jb & 1) s.Y[r0 + (jb >> 1)][j] = acc;
                else s.X[r0 + (jb >> 1)][j] = acc;
            }
        }
        // the coefficients of the solve and of the outputs
        if (tid < NB * NB) {
            const int t = tid / NB, i = tid % NB;
            const float d = (i <= t) ? expf(s.gam[t] - s.gam[i]) : 0.f;
            s.A[t][i] = (i < t) ? s.beta[t] * d * s.kk[t][i] : 0.f;
            s.P[t][i] = (i <= t) ? d * s.kq[t][i] : 0.f;
        }
        __syncthreads();
        // 5. column j: the solve for u_t, then o_t (u into X, o into Y), and the partial
        // sums of o_t^2 per warp
        if (tid < kMaxHeadDim) {
            const int j = tid;
            float u[NB], o[NB];
#pragma unroll
            for (int t = 0; t < NB; ++t) {
                float r = (j < V) ? s.beta[t] * (s.v[t][j] - s.Gam[t] * s.X[t][j]) : 0.f;
#pragma unroll
                for (int i = 0; i < t; ++i) r = fmaf(-s.A[t][i], u[i], r);
                u[t] = r;
                float y = s.Gam[t] * s.Y[t][j];
#pragma unroll
                for (int i = 0; i <= t; ++i) y = fmaf(s.P[t][i], u[i], y);
                o[t] = (j < V) ? y * rsK : 0.f;
            }
#pragma unroll
            for (int t = 0; t < NB; ++t) {
                s.X[t][j] = u[t];
                s.Y[t][j] = o[t];
                const float sq = warp_sum(o[t] * o[t]);
                if (lane == 0) s.ssq[t][w] = sq;
            }
        }
        __syncthreads();
        // 6. RMSNormGated of each real token
        for (int e = tid; e < nt * kMaxHeadDim; e += NT) {
            const int t = e / kMaxHeadDim, j = e % kMaxHeadDim;
            if (j >= V) continue;
            float ms = 0.f;
#pragma unroll
            for (int ww = 0; ww < kMaxHeadDim / 32; ++ww) ms += s.ssq[t][ww];
            ms /= (float)V;
            const float zj = s.z[t][j];
            const float y = s.Y[t][j] * (1.f / sqrtf(ms + kEpsRms)) * a.norm_weight[j] *
                            (zj * sigmoid_f(zj));
            const size_t row = (size_t)(t0 + t) * BH + (size_t)bh;
            a.out[row * V + j] = __float2bfloat16_rn(y);
        }
        // 7. S_last = Gamma_last S0 + sum_t D[last][t] k^_t u_t^T in the registers, token
        // by token (a padding token adds exact zeros)
        const float Gl = s.Gam[NB - 1];
#pragma unroll
        for (int m = 0; m < MROWS; ++m)
#pragma unroll
            for (int c = 0; c < 4; ++c) st[m][c] *= Gl;
#pragma unroll
        for (int t = 0; t < NB; ++t) {
            float u4[4];
            if (VEC4) {
                const float4 x = *reinterpret_cast<const float4*>(&s.X[t][4 * lane]);
                u4[0] = x.x, u4[1] = x.y, u4[2] = x.z, u4[3] = x.w;
            } else {
#pragma unroll
                for (int c = 0; c < 4; ++c) u4[c] = s.X[t][col_of<false>(lane, c)];
            }
            const float dl = s.dlast[t];
#pragma unroll
            for (int c = 0; c < 4; ++c) u4[c] *= dl;
#pragma unroll
            for (int m4 = 0; m4 < MROWS; m4 += 4) {
                const float4 k4 = *reinterpret_cast<const float4*>(&s.kn[t][r0w + m4]);
                const float kv[4] = {k4.x, k4.y, k4.z, k4.w};
#pragma unroll
                for (int mm = 0; mm < 4; ++mm)
#pragma unroll
                    for (int c = 0; c < 4; ++c) st[m4 + mm][c] = fmaf(kv[mm], u4[c], st[m4 + mm][c]);
            }
        }
    }
    // the state, written once
#pragma unroll
    for (int m = 0; m < MROWS; ++m) {
        const int i = r0w + m;
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

// Launches the chunk form with NB tokens per block.
template <bool VEC4, int NB>
cudaError_t launch_multi(const DecodeArgs& a, cudaStream_t stream) {
    static cudaError_t attr = [] {
        // shared memory above the default 48 KB, and the largest carveout so that two CTAs
        // fit an SM
        cudaError_t e = cudaFuncSetAttribute(decode_multi_kernel<VEC4, NB>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)sizeof(MultiSmem));
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(decode_multi_kernel<VEC4, NB>,
                                     cudaFuncAttributePreferredSharedMemoryCarveout,
                                     (int)cudaSharedmemCarveoutMaxShared);
        return e;
    }();
    if (attr != cudaSuccess) return attr;
    decode_multi_kernel<VEC4, NB><<<a.BH, NT, sizeof(MultiSmem), stream>>>(a);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_decode(const DecodeArgs& args, cudaStream_t stream) {
    if (args.BH == 0 || args.T == 0) return cudaSuccess;
    // two CTAs per SM are resident (launch bounds): rows that far ahead are prefetched, in
    // the single step, where it was measured to help (the multi-token form, whose CTAs stay
    // T times as long, measured the same with and without it)
    constexpr int kMaxDevices = 64;
    static int sms_of[kMaxDevices] = {};
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) == cudaSuccess && dev >= 0 && dev < kMaxDevices) {
        if (sms_of[dev] == 0) cudaDeviceGetAttribute(&sms_of[dev], cudaDevAttrMultiProcessorCount, dev);
        sms = sms_of[dev];
    }
    DecodeArgs a = args;
    a.pf_rows = a.T == 1 ? 2 * sms : 0;
    // More than kPerTokenMaxT tokens: the chunk form (blocks of eight). Up to that, the
    // token loop, which measured faster there (T = 2: 0.212 against 0.242 ms, T = 4: 0.309
    // against 0.332 ms at BH = 8192; T = 8: 0.608 against 0.512 ms); a single step stages
    // one token's inputs (the smaller footprint keeps the streaming step at its bandwidth),
    // several tokens NWARP at a time.
    constexpr int kPerTokenMaxT = 4;
    if (a.T > kPerTokenMaxT)
        return a.V == kMaxHeadDim ? launch_multi<true, TB>(a, stream)
                                  : launch_multi<false, TB>(a, stream);
    if (a.V == kMaxHeadDim) {
        if (a.T == 1) decode_kernel<true, 1><<<a.BH, NT, 0, stream>>>(a);
        else decode_kernel<true, NWARP><<<a.BH, NT, 0, stream>>>(a);
    } else {
        if (a.T == 1) decode_kernel<false, 1><<<a.BH, NT, 0, stream>>>(a);
        else decode_kernel<false, NWARP><<<a.BH, NT, 0, stream>>>(a);
    }
    return cudaGetLastError();
}

}  // namespace gdn
