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

// The chunk form (more than four tokens per call), blocks of TB tokens. One CTA of
// MT = 512 threads per row; the 64 KB state sits in shared memory (one bulk copy, started
// first, so its latency overlaps the staging of the inputs, the norms and the small Gram
// products), which leaves the registers free for two CTAs per SM. k^ and q^ are stored
// token-minor ([row][token]), so that a thread's four tokens of a row are one 16-byte
// broadcast load in both passes over the state.
constexpr int TB = 8;
constexpr int MT = 512;
constexpr int MW = MT / 32;
constexpr uint64_t kDecodeWaitNs = 2000000000ull;

// Status bit of a bounded wait of this file that ran out (decode_take_status).
__device__ uint32_t g_decode_status = 0;

struct MultiSmem {
    float S[kMaxHeadDim * kMaxHeadDim];  // the state, row-major [K][V] (row stride 128)
    float kT[kMaxHeadDim][TB];           // k^ token-minor (zero rows for padding tokens)
    float qT[kMaxHeadDim][TB];           // q^ token-minor
    float v[TB][kMaxHeadDim];
    float z[TB][kMaxHeadDim];
    float X[TB][kMaxHeadDim];            // S0^T k^_t (partials summed), then u_t
    float Y[TB][kMaxHeadDim];            // S0^T q^_t, then the un-normalised o_t
    float red[2][2 * TB][kMaxHeadDim];   // the second row half's partial sums
    float A[TB][TB];                     // beta_t D[t][i] (k^_t . k^_i), i < t
    float P[TB][TB];                     // D[t][i] (k^_i . q^_t), i <= t
    float kk[TB][TB], kq[TB][TB];
    float gam[TB], Gam[TB], dlast[TB], beta[TB], g[TB], inv[2][TB];
    float ssq[TB][kMaxHeadDim / 32];
    unsigned long long bar;
    int failed;
};

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Waits (at most kDecodeWaitNs) for phase 0 of the mbarrier at `bar`; false if it ran out.
__device__ __forceinline__ bool wait_phase0(uint32_t bar) {
    const uint64_t t_start = globaltimer();
    while (true) {
        uint32_t ok;
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], 0;\n\t"
            "selp.u32 %0, 1, 0, p;\n\t}"
            : "=r"(ok)
            : "r"(bar)
            : "memory");
        if (ok) return true;
        if (globaltimer() - t_start > kDecodeWaitNs) return false;
    }
}

template <bool FULL>  // FULL: K = V = 128 (one bulk copy of the state)
__global__ void __launch_bounds__(MT, 2) decode_multi_kernel(DecodeArgs a) {
    extern __shared__ __align__(128) uint8_t smraw[];
    MultiSmem& s = *reinterpret_cast<MultiSmem*>(smraw);
    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
    const int bh = blockIdx.x, h = bh % a.H;
    const int K = a.K, V = a.V;
    const float* S0 = a.state_in + (size_t)bh * K * V;
    float* S1 = a.state_out + (size_t)bh * K * V;
    const size_t BH = (size_t)a.BH;
    const float rsK = 1.f / sqrtf((float)K);
    const uint32_t bar = smem_addr(&s.bar);

    // 0. the state: one bulk copy (K = V = 128), else plain loads with zero padding
    if (FULL) {
        if (tid == 0) {
            s.failed = 0;
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(bar) : "memory");
            asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
            asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar),
                         "r"(65536u)
                         : "memory");
            asm volatile(
                "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], "
                "%2, [%3];" ::"r"(smem_addr(s.S)),
                "l"(reinterpret_cast<uint64_t>(S0)), "r"(65536u), "r"(bar)
                : "memory");
        }
    } else {
        for (int e = tid; e < kMaxHeadDim * kMaxHeadDim; e += MT) {
            const int i = e / kMaxHeadDim, j = e % kMaxHeadDim;
            s.S[e] = (i < K && j < V) ? __ldcs(S0 + (size_t)i * V + j) : 0.f;
        }
        if (tid == 0) s.failed = 0;
    }

    for (int t0 = 0; t0 < a.T; t0 += TB) {
        const int nt = min(TB, a.T - t0);  // real tokens of this block
        const bool last = t0 + TB >= a.T;
        __syncthreads();  // (the mbarrier is initialised; the previous block is done)
        // 1. inputs of the block (padding tokens: zero rows, beta = 0, g = 0)
        for (int e = tid; e < TB * kMaxHeadDim; e += MT) {
            const int t = e / kMaxHeadDim, i = e % kMaxHeadDim;
            const size_t row = (size_t)(t0 + t) * BH + (size_t)bh;
            const bool real = t < nt;
            s.qT[i][t] = (real && i < K) ? __bfloat162float(a.q[row * K + i]) : 0.f;
            s.kT[i][t] = (real && i < K) ? __bfloat162float(a.k[row * K + i]) : 0.f;
            s.v[t][i] = (real && i < V) ? __bfloat162float(a.v[row * V + i]) : 0.f;
            s.z[t][i] = (real && i < V) ? __bfloat162float(a.z[row * V + i]) : 0.f;
        }
        if (tid < TB) {
            const size_t row = (size_t)(t0 + tid) * BH + (size_t)bh;
            const bool real = tid < nt;
            s.beta[tid] = real ? sigmoid_f(__bfloat162float(a.b[row])) : 0.f;
            s.g[tid] = real ? -expf(a.A_log[h]) *
                                  softplus_f(__bfloat162float(a.a[row]) + a.dt_bias[h])
                            : 0.f;
        }
        __syncthreads();
        // 2. the l2 norms (warp j: token j / 2, q or k), the decay prefix (one thread)
        if (w < 2 * TB) {
            const int t = w >> 1;
            float acc = 0.f;
#pragma unroll
            for (int i = lane; i < kMaxHeadDim; i += 32) {
                const float x = (w & 1) ? s.kT[i][t] : s.qT[i][t];
                acc = fmaf(x, x, acc);
            }
            acc = warp_sum(acc);
            if (lane == 0) s.inv[w & 1][t] = 1.f / sqrtf(acc + kEpsL2);
        }
        if (tid == MT - 1) {
            float gm = 0.f;
#pragma unroll
            for (int t = 0; t < TB; ++t) {
                gm += s.g[t];
                s.gam[t] = gm;
                s.Gam[t] = expf(gm);
            }
#pragma unroll
            for (int t = 0; t < TB; ++t) s.dlast[t] = expf(gm - s.gam[t]);
        }
        __syncthreads();
        for (int e = tid; e < TB * kMaxHeadDim; e += MT) {
            const int i = e / TB, t = e % TB;
            s.qT[i][t] *= s.inv[0][t];
            s.kT[i][t] *= s.inv[1][t];
        }
        __syncthreads();
        // 3. the small Gram products k^_t . k^_i and k^_i . q^_t (i <= t): four adjacent
        // threads per product, thread `part` taking rows part, part + 4, ... (so a warp's
        // loads fall in distinct banks), joined by two shuffles
        {
            const int part = tid & 3, pr = tid >> 2;  // pr: 0..127
            const int kind = pr >> 6, t = (pr >> 3) & 7, i = pr & 7;
            float acc = 0.f;
            if (i <= t) {
#pragma unroll 8
                for (int e = part; e < kMaxHeadDim; e += 4)
                    acc = fmaf(s.kT[e][i], kind ? s.qT[e][t] : s.kT[e][t], acc);
            }
            acc += __shfl_xor_sync(0xffffffffu, acc, 1);
            acc += __shfl_xor_sync(0xffffffffu, acc, 2);
            if (part == 0 && i <= t) {
                if (kind) s.kq[t][i] = acc;
                else s.kk[t][i] = acc;
            }
        }
        // the state has landed (first block); a copy that never lands is waited for once
        // more before the CTA leaves
        if (FULL && t0 == 0 && !wait_phase0(bar)) {
            atomicOr(&g_decode_status, 1u);
            s.failed = 1;
        }
        __syncthreads();
        if (s.failed) {
            if (tid == 0) wait_phase0(bar);
            return;
        }
        // 4. X[t] = S0^T k^_t and Y[t] = S0^T q^_t: thread (column j, tokens 4 th .. 4 th + 3,
        // rows 64 rh .. 64 rh + 63); the second row half adds its partials through red
        {
            const int j = tid & (kMaxHeadDim - 1), th = (tid >> 7) & 1, rh = tid >> 8;
            // token pairs in paired fp32 FMAs (each lane rounds as fmaf)
            float2 x01 = make_float2(0.f, 0.f), x23 = x01, y01 = x01, y23 = x01;
#pragma unroll 4
            for (int i = 64 * rh; i < 64 * rh + 64; ++i) {
                const float sv = s.S[i * kMaxHeadDim + j];
                const float2 ss = make_float2(sv, sv);
                const float4 k4 = *reinterpret_cast<const float4*>(&s.kT[i][4 * th]);
                const float4 q4 = *reinterpret_cast<const float4*>(&s.qT[i][4 * th]);
                x01 = ffma2(make_float2(k4.x, k4.y), ss, x01);
                x23 = ffma2(make_float2(k4.z, k4.w), ss, x23);
                y01 = ffma2(make_float2(q4.x, q4.y), ss, y01);
                y23 = ffma2(make_float2(q4.z, q4.w), ss, y23);
            }
            const float px[4] = {x01.x, x01.y, x23.x, x23.y};
            const float py[4] = {y01.x, y01.y, y23.x, y23.y};
            if (rh == 1) {
#pragma unroll
                for (int r = 0; r < 4; ++r) {
                    s.red[0][4 * th + r][j] = px[r];
                    s.red[1][4 * th + r][j] = py[r];
                }
            }
            __syncthreads();
            if (rh == 0) {
#pragma unroll
                for (int r = 0; r < 4; ++r) {
                    s.X[4 * th + r][j] = px[r] + s.red[0][4 * th + r][j];
                    s.Y[4 * th + r][j] = py[r] + s.red[1][4 * th + r][j];
                }
            }
        }
        // the coefficients of the solve and of the outputs
        if (tid >= MT - TB * TB) {
            const int e = tid - (MT - TB * TB), t = e / TB, i = e % TB;
            const float d = (i <= t) ? expf(s.gam[t] - s.gam[i]) : 0.f;
            s.A[t][i] = (i < t) ? s.beta[t] * d * s.kk[t][i] : 0.f;
            s.P[t][i] = (i <= t) ? d * s.kq[t][i] : 0.f;
        }
        __syncthreads();
        // 5. column j: the solve for u_t, then o_t (u into X, o into Y), and the partial
        // sums of o_t^2 per warp
        if (tid < kMaxHeadDim) {
            const int j = tid;
            float u[TB], o[TB];
#pragma unroll
            for (int t = 0; t < TB; ++t) {
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
            for (int t = 0; t < TB; ++t) {
                s.X[t][j] = u[t] * s.dlast[t];  // the update pass needs D[last][t] u_t
                s.Y[t][j] = o[t];
                const float sq = warp_sum(o[t] * o[t]);
                if (lane == 0) s.ssq[t][w] = sq;
            }
        }
        __syncthreads();
        // 6. RMSNormGated of each real token
        for (int e = tid; e < nt * kMaxHeadDim; e += MT) {
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
        // 7. S_last = Gamma_last S0 + sum_t D[last][t] k^_t u_t^T: thread (column j, rows
        // 32 rq .. 32 rq + 31); written to global memory after the last block, else back
        // to shared memory for the next one (a padding token adds exact zeros)
        {
            const int j = tid & (kMaxHeadDim - 1), rq = tid >> 7;
            const float Gl = s.Gam[TB - 1];
            // the token pairs (0,1), (2,3), (4,5), (6,7) in paired fp32 FMAs, the two halves
            // added at the end
            const float2 u01 = make_float2(s.X[0][j], s.X[1][j]);
            const float2 u23 = make_float2(s.X[2][j], s.X[3][j]);
            const float2 u45 = make_float2(s.X[4][j], s.X[5][j]);
            const float2 u67 = make_float2(s.X[6][j], s.X[7][j]);
#pragma unroll 4
            for (int i = 32 * rq; i < 32 * rq + 32; ++i) {
                const float4 k0 = *reinterpret_cast<const float4*>(&s.kT[i][0]);
                const float4 k1 = *reinterpret_cast<const float4*>(&s.kT[i][4]);
                float2 acc = make_float2(Gl * s.S[i * kMaxHeadDim + j], 0.f);
                acc = ffma2(make_float2(k0.x, k0.y), u01, acc);
                acc = ffma2(make_float2(k0.z, k0.w), u23, acc);
                acc = ffma2(make_float2(k1.x, k1.y), u45, acc);
                acc = ffma2(make_float2(k1.z, k1.w), u67, acc);
                const float x = acc.x + acc.y;
                if (last) {
                    if (i < K && j < V) __stcs(S1 + (size_t)i * V + j, x);
                } else {
                    s.S[i * kMaxHeadDim + j] = x;
                }
            }
        }
    }
}

template <bool FULL>
cudaError_t launch_multi(const DecodeArgs& a, cudaStream_t stream) {
    static cudaError_t attr = [] {
        // shared memory above the default 48 KB, and the largest carveout so that two CTAs
        // fit an SM
        cudaError_t e = cudaFuncSetAttribute(decode_multi_kernel<FULL>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)sizeof(MultiSmem));
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(decode_multi_kernel<FULL>,
                                     cudaFuncAttributePreferredSharedMemoryCarveout,
                                     (int)cudaSharedmemCarveoutMaxShared);
        return e;
    }();
    if (attr != cudaSuccess) return attr;
    decode_multi_kernel<FULL><<<a.BH, MT, sizeof(MultiSmem), stream>>>(a);
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
        return (a.K == kMaxHeadDim && a.V == kMaxHeadDim) ? launch_multi<true>(a, stream)
                                                          : launch_multi<false>(a, stream);
    if (a.V == kMaxHeadDim) {
        if (a.T == 1) decode_kernel<true, 1><<<a.BH, NT, 0, stream>>>(a);
        else decode_kernel<true, NWARP><<<a.BH, NT, 0, stream>>>(a);
    } else {
        if (a.T == 1) decode_kernel<false, 1><<<a.BH, NT, 0, stream>>>(a);
        else decode_kernel<false, NWARP><<<a.BH, NT, 0, stream>>>(a);
    }
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
