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
// HBM traffic is paid once per call; token t's inputs sit at offset t * BH rows.
#include "internal.h"

namespace gdn {
namespace {

constexpr int NT = 256;
constexpr int NWARP = NT / 32;
constexpr int ROWS = kMaxHeadDim / NWARP;  // 16 state rows per warp at most

struct Smem {
    float qn[kMaxHeadDim];
    float kn[kMaxHeadDim];
    float v[kMaxHeadDim];
    float z[kMaxHeadDim];
    float u[kMaxHeadDim];
    float red[2][NWARP][kMaxHeadDim];
    float scal[8];  // 0: 1/|q|, 1: 1/|k|, 2: k^.q^, 3: beta, 4: alpha, 5: 1/rms
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

template <bool VEC4>
__global__ void __launch_bounds__(NT, 2) decode_kernel(DecodeArgs a) {
    __shared__ Smem s;
    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
    const int bh = blockIdx.x, h = bh % a.H;
    const int K = a.K, V = a.V;
    const float* S0 = a.state_in + (size_t)bh * K * V;
    float* S1 = a.state_out + (size_t)bh * K * V;
    const size_t BH = (size_t)a.BH;

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

    // 2. small per-row inputs, token by token; thread i < 128 holds element i of the
    // next token's q, k, v, z (and thread 0 its b, a) in registers, loaded one token
    // ahead so that their latency hides behind the current token
    float nq = 0.f, nk = 0.f, nv = 0.f, nz = 0.f, nb = 0.f, na = 0.f;
    auto fetch = [&](int tok) {
        const size_t row = (size_t)tok * BH + (size_t)bh;
        if (tid < kMaxHeadDim) {
            nq = tid < K ? __bfloat162float(a.q[row * K + tid]) : 0.f;
            nk = tid < K ? __bfloat162float(a.k[row * K + tid]) : 0.f;
            nv = tid < V ? __bfloat162float(a.v[row * V + tid]) : 0.f;
            nz = tid < V ? __bfloat162float(a.z[row * V + tid]) : 0.f;
        }
        if (tid == 0) {
            nb = __bfloat162float(a.b[row]);
            na = __bfloat162float(a.a[row]);
        }
    };
    fetch(0);
    for (int tok = 0; tok < a.T; ++tok) {
    if (tok > 0) __syncthreads();  // the previous token's shared inputs are read
    const size_t row = (size_t)tok * BH + (size_t)bh;  // this token's input row
    if (tid < kMaxHeadDim) {
        s.qn[tid] = nq;
        s.kn[tid] = nk;
        s.v[tid] = nv;
        s.z[tid] = nz;
    }
    if (tid == 0) {
        s.scal[3] = sigmoid_f(nb);
        const float gg = -expf(a.A_log[h]) * softplus_f(na + a.dt_bias[h]);
        s.scal[4] = expf(gg);
    }
    if (tok + 1 < a.T) fetch(tok + 1);
    __syncthreads();
    // 3. l2 norms of q and k (warps 0 and 1), then normalise
    if (w < 2) {
        const float* x = (w == 0) ? s.qn : s.kn;
        float acc = 0.f;
        for (int i = lane; i < kMaxHeadDim; i += 32) acc = fmaf(x[i], x[i], acc);
        acc = warp_sum(acc);
        if (lane == 0) s.scal[w] = 1.f / sqrtf(acc + kEpsL2);
    }
    __syncthreads();
    for (int i = tid; i < kMaxHeadDim; i += NT) {
        s.qn[i] *= s.scal[0];
        s.kn[i] *= s.scal[1];
    }
    __syncthreads();
    if (w == 0) {
        float acc = 0.f;
        for (int i = lane; i < kMaxHeadDim; i += 32) acc = fmaf(s.kn[i], s.qn[i], acc);
        acc = warp_sum(acc);
        if (lane == 0) s.scal[2] = acc;
    }
    // 4. per-warp partial x = S^T k^ and y = S^T q^ over this warp's rows
    {
        float px[4] = {0.f, 0.f, 0.f, 0.f}, py[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int m = 0; m < ROWS; ++m) {
            const int i = w + NWARP * m;
            const float ki = s.kn[i], qi = s.qn[i];  // zero beyond K
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
    // 5. u = beta (v - alpha x); o = (alpha y + u (k^.q^)) / sqrt(K)
    const float beta = s.scal[3], alpha = s.scal[4];
    float o = 0.f;
    if (tid < kMaxHeadDim) {
        const int j = tid;
        float x = 0.f, y = 0.f;
#pragma unroll
        for (int ww = 0; ww < NWARP; ++ww) { x += s.red[0][ww][j]; y += s.red[1][ww][j]; }
        const float u = (j < V) ? beta * (s.v[j] - alpha * x) : 0.f;
        s.u[j] = u;
        o = (j < V) ? (alpha * y + u * s.scal[2]) / sqrtf((float)K) : 0.f;
        const float sq = warp_sum(o * o);
        if (lane == 0) s.part[w] = sq;
    }
    __syncthreads();
    // 6. RMSNormGated epilogue (threads 0..V-1), bf16 out
    if (tid < V) {
        float ms = 0.f;
#pragma unroll
        for (int ww = 0; ww < kMaxHeadDim / 32; ++ww) ms += s.part[ww];
        ms /= (float)V;
        const float zj = s.z[tid];
        const float y = o * (1.f / sqrtf(ms + kEpsRms)) * a.norm_weight[tid] * (zj * sigmoid_f(zj));
        a.out[row * V + tid] = __float2bfloat16_rn(y);
    }
    // 7. S' = alpha S + k^ u^T in registers (rows beyond K stay zero)
#pragma unroll
    for (int m = 0; m < ROWS; ++m) {
        const int i = w + NWARP * m;
        const float ki = s.kn[i];  // zero beyond K
#pragma unroll
        for (int c = 0; c < 4; ++c)
            st[m][c] = fmaf(alpha, st[m][c], ki * s.u[col_of<VEC4>(lane, c)]);
    }
    }  // tokens
    // 8. the state, written once
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

}  // namespace

cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t stream) {
    if (a.BH == 0 || a.T == 0) return cudaSuccess;
    if (a.V == kMaxHeadDim)
        decode_kernel<true><<<a.BH, NT, 0, stream>>>(a);
    else
        decode_kernel<false><<<a.BH, NT, 0, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace gdn
