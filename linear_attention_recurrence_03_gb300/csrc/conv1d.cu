// conv1d.cu -- one decode token through the depthwise causal convolution in front of the
// decode step ("GDN Block TKG Kernel API Reference": gdn_conv1d_decode -- conv + silu +
// slide-window state -- then the split of the conv output into q | k | v and the GQA
// repeat of q and k; conv_weight [conv_dim, K_win] fp32, conv_state [B, conv_dim, K_win]).
//
// Per batch b and channel c (the window oldest first; no bias -- the page lists none):
//   window' = (state[1], ..., state[K_win - 1], x)
//   y       = silu(sum_w weight[c][w] window'[w])        (fp32 arithmetic)
//   state'  = window'                                     (bf16, exact: a shift)
// Channel c < key_dim is q channel (head c / Dk, dim c % Dk), the next key_dim are k,
// the rest v (head (c - 2 key_dim) / Dv); q and k are written to every value head of
// their key head (value head h reads key head h / G), v to its own.
//
// HBM-bound: one thread per (b, c), consecutive channels in consecutive threads, so the
// window, weight and output accesses are coalesced.
#include "internal.h"

namespace gdn {
namespace {

constexpr int kConvThreads = 256;

// Writes y of channel c of batch b to its q / k rows (every value head of its key head)
// or to its v row.
__device__ __forceinline__ void put_channel(const Conv1dArgs& a, int b, int c, __nv_bfloat16 y) {
    const int kd = a.Hk * a.Dk, G = a.Hv / a.Hk;
    if (c < 2 * kd) {
        const int cc = c < kd ? c : c - kd;
        const int kh = cc / a.Dk, d = cc % a.Dk;
        __nv_bfloat16* dst = c < kd ? a.q : a.k;
        for (int g = 0; g < G; ++g)
            dst[((size_t)b * a.Hv + (size_t)kh * G + g) * a.Dk + d] = y;
    } else {
        const int cv = c - 2 * kd;
        a.v[((size_t)b * a.Hv + cv / a.Dv) * a.Dv + cv % a.Dv] = y;
    }
}

__device__ __forceinline__ __nv_bfloat16 silu_bf16(float s) {
    return __float2bfloat16_rn(s / (1.f + __expf(-s)));
}

// K_win = 4 (the usual width): the window is one 8-byte vector, the taps one float4.
__global__ void __launch_bounds__(kConvThreads) conv1d_decode_k4_kernel(Conv1dArgs a) {
    const int C = 2 * a.Hk * a.Dk + a.Hv * a.Dv;
    const long idx = (long)blockIdx.x * kConvThreads + threadIdx.x;
    if (idx >= (long)a.B * C) return;
    const int b = (int)(idx / C), c = (int)(idx % C);
    const uint2 sv = *reinterpret_cast<const uint2*>(a.state_in + (size_t)idx * 4);
    const float4 w = *reinterpret_cast<const float4*>(a.weight + (size_t)c * 4);
    const __nv_bfloat16 xn = a.x[idx];
    // window' = (s1, s2, s3, x): the upper bf16 of word 0, word 1, then x
    const __nv_bfloat162 s01 = *reinterpret_cast<const __nv_bfloat162*>(&sv.x);
    const __nv_bfloat162 s23 = *reinterpret_cast<const __nv_bfloat162*>(&sv.y);
    const float acc = fmaf(w.w, __bfloat162float(xn),
                           fmaf(w.z, __bfloat162float(s23.y),
                                fmaf(w.y, __bfloat162float(s23.x), w.x * __bfloat162float(s01.y))));
    __nv_bfloat162 n01, n23;
    n01.x = s01.y;
    n01.y = s23.x;
    n23.x = s23.y;
    n23.y = xn;
    uint2 ov;
    ov.x = *reinterpret_cast<const uint32_t*>(&n01);
    ov.y = *reinterpret_cast<const uint32_t*>(&n23);
    *reinterpret_cast<uint2*>(a.state_out + (size_t)idx * 4) = ov;
    put_channel(a, b, c, silu_bf16(acc));
}

// K_win = 4, head dims multiples of 4: four adjacent channels per thread (they never
// straddle a q / k / v head), so every access is a 16-, 32- or 64-byte vector.
__global__ void __launch_bounds__(kConvThreads) conv1d_decode_k4x4_kernel(Conv1dArgs a) {
    const int C = 2 * a.Hk * a.Dk + a.Hv * a.Dv, C4 = C / 4;
    const long idx = (long)blockIdx.x * kConvThreads + threadIdx.x;  // (b, channel quad)
    if (idx >= (long)a.B * C4) return;
    const int b = (int)(idx / C4), c = (int)(idx % C4) * 4;
    const size_t e0 = (size_t)b * C + c;  // first element (batch b, channel c)
    const uint4* sp = reinterpret_cast<const uint4*>(a.state_in + e0 * 4);
    const uint4 s0 = sp[0], s1 = sp[1];  // the four windows, 8 bf16 each half
    const float4* wp = reinterpret_cast<const float4*>(a.weight + (size_t)c * 4);
    const uint2 xv = *reinterpret_cast<const uint2*>(a.x + e0);
    const uint32_t sw[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
    const __nv_bfloat162 x01 = *reinterpret_cast<const __nv_bfloat162*>(&xv.x);
    const __nv_bfloat162 x23 = *reinterpret_cast<const __nv_bfloat162*>(&xv.y);
    const __nv_bfloat16 xs[4] = {x01.x, x01.y, x23.x, x23.y};
    uint32_t ow[8];
    __nv_bfloat16 y[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const float4 w = wp[j];
        const __nv_bfloat162 a01 = *reinterpret_cast<const __nv_bfloat162*>(&sw[2 * j]);
        const __nv_bfloat162 a23 = *reinterpret_cast<const __nv_bfloat162*>(&sw[2 * j + 1]);
        const float acc = fmaf(w.w, __bfloat162float(xs[j]),
                               fmaf(w.z, __bfloat162float(a23.y),
                                    fmaf(w.y, __bfloat162float(a23.x),
                                         w.x * __bfloat162float(a01.y))));
        __nv_bfloat162 n01, n23;
        n01.x = a01.y;
        n01.y = a23.x;
        n23.x = a23.y;
        n23.y = xs[j];
        ow[2 * j] = *reinterpret_cast<const uint32_t*>(&n01);
        ow[2 * j + 1] = *reinterpret_cast<const uint32_t*>(&n23);
        y[j] = silu_bf16(acc);
    }
    uint4* so = reinterpret_cast<uint4*>(a.state_out + e0 * 4);
    so[0] = make_uint4(ow[0], ow[1], ow[2], ow[3]);
    so[1] = make_uint4(ow[4], ow[5], ow[6], ow[7]);
    __nv_bfloat162 y01, y23;
    y01.x = y[0];
    y01.y = y[1];
    y23.x = y[2];
    y23.y = y[3];
    uint2 yv;
    yv.x = *reinterpret_cast<const uint32_t*>(&y01);
    yv.y = *reinterpret_cast<const uint32_t*>(&y23);
    const int kd = a.Hk * a.Dk, G = a.Hv / a.Hk;
    if (c < 2 * kd) {
        const int cc = c < kd ? c : c - kd;
        const int kh = cc / a.Dk, d = cc % a.Dk;
        __nv_bfloat16* dst = c < kd ? a.q : a.k;
        for (int g = 0; g < G; ++g)
            *reinterpret_cast<uint2*>(dst + ((size_t)b * a.Hv + (size_t)kh * G + g) * a.Dk + d) =
                yv;
    } else {
        const int cv = c - 2 * kd;
        *reinterpret_cast<uint2*>(a.v + ((size_t)b * a.Hv + cv / a.Dv) * a.Dv + cv % a.Dv) = yv;
    }
}

// Any width 1 <= K_win <= kMaxConvWidth.
__global__ void __launch_bounds__(kConvThreads) conv1d_decode_kernel(Conv1dArgs a) {
    const int C = 2 * a.Hk * a.Dk + a.Hv * a.Dv;
    const long idx = (long)blockIdx.x * kConvThreads + threadIdx.x;
    if (idx >= (long)a.B * C) return;
    const int b = (int)(idx / C), c = (int)(idx % C);
    const int K = a.K_win;
    const __nv_bfloat16* s = a.state_in + (size_t)idx * K;
    __nv_bfloat16* so = a.state_out + (size_t)idx * K;
    const float* w = a.weight + (size_t)c * K;
    __nv_bfloat16 win[kMaxConvWidth];
#pragma unroll
    for (int j = 0; j < kMaxConvWidth; ++j)
        if (j + 1 < K) win[j] = s[j + 1];
    win[K - 1] = a.x[idx];
    float acc = 0.f;
#pragma unroll
    for (int j = 0; j < kMaxConvWidth; ++j)
        if (j < K) acc = fmaf(w[j], __bfloat162float(win[j]), acc);
    // the whole window is read before any of it is written (state_out may be state_in)
#pragma unroll
    for (int j = 0; j < kMaxConvWidth; ++j)
        if (j < K) so[j] = win[j];
    put_channel(a, b, c, silu_bf16(acc));
}

}  // namespace

cudaError_t launch_conv1d_decode(const Conv1dArgs& a, cudaStream_t stream) {
    const long n = (long)a.B * (2 * a.Hk * a.Dk + a.Hv * a.Dv);
    if (n == 0) return cudaSuccess;
    const long blocks = (n + kConvThreads - 1) / kConvThreads;
    if (a.K_win == 4 && a.Dk % 4 == 0 && a.Dv % 4 == 0) {
        const long quads = (n / 4 + kConvThreads - 1) / kConvThreads;
        conv1d_decode_k4x4_kernel<<<(unsigned)quads, kConvThreads, 0, stream>>>(a);
    } else if (a.K_win == 4)
        conv1d_decode_k4_kernel<<<(unsigned)blocks, kConvThreads, 0, stream>>>(a);
    else
        conv1d_decode_kernel<<<(unsigned)blocks, kConvThreads, 0, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace gdn
