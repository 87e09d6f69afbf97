// gdn_api.cu -- the extern "C" entry points declared in include/gdn.h: argument
// validation, kernel selection and error reporting. No arithmetic of the method lives
// here; every step runs in the kernels.
#include <algorithm>
#include <atomic>
#include <cstdarg>
#include <cstdio>
#include <cstdint>
#include <mutex>
#include <string>

#include "gdn.h"
#include "internal.h"

namespace {

thread_local std::string g_last_error;
std::atomic<unsigned long long> g_launches{0};

// Scratch of gdn_prefill_noalloc, for callers that may not allocate device memory while
// they run: a file-scope device array of the library's own module (every device that loads
// the library holds it until the process exits), so the call itself allocates nothing.
constexpr size_t kStaticScratchBytes = size_t(128) << 20;
__device__ __align__(256) unsigned char g_prefill_scratch[kStaticScratchBytes];

// In host code `g_prefill_scratch` names a host-side stand-in, not device memory: the
// array's device address is looked up once per device (with that device current) and
// kept here; the kernels are given that address.
constexpr int kMaxScratchDevices = 64;
void* g_scratch_addr[kMaxScratchDevices];
cudaError_t g_scratch_err[kMaxScratchDevices];
std::once_flag g_scratch_once[kMaxScratchDevices];

// Device address of the scratch array on the current device (the set-up runs on the
// first call for each device).
cudaError_t scratch_address(void** addr) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxScratchDevices) return cudaErrorInvalidDevice;
    std::call_once(g_scratch_once[dev], [dev] {
        g_scratch_err[dev] = cudaGetSymbolAddress(&g_scratch_addr[dev], g_prefill_scratch);
    });
    *addr = g_scratch_addr[dev];
    return g_scratch_err[dev];
}

gdn_status fail(gdn_status st, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof(buf), fmt, ap);
    va_end(ap);
    g_last_error = buf;
    return st;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Sequences of one variable-length call (the carry grid's third dimension).
constexpr int kMaxSequences = 65535;

// Checks that p is non-NULL and 16-byte aligned (or NULL allowed when unused).
bool ptr_ok(const void* p, bool required) {
    if (p == nullptr) return !required;
    return aligned16(p);
}

gdn_status check_prefill_shape(int B, int Hk, int Hv, int S, int Dk, int Dv, gdn_dtype dt) {
    if (B < 1 || Hk < 1 || Hv < 1 || S < 0)
        return fail(GDN_EINVAL, "gdn_prefill: need B >= 1, Hk >= 1, Hv >= 1, S >= 0 "
                    "(got B=%d Hk=%d Hv=%d S=%d)", B, Hk, Hv, S);
    if (Hv % Hk != 0)
        return fail(GDN_EINVAL, "gdn_prefill: Hv (%d) must be a multiple of Hk (%d)", Hv, Hk);
    if (Dk < 1 || Dk > gdn::kMaxHeadDim || Dv < 1 || Dv > gdn::kMaxHeadDim)
        return fail(GDN_EINVAL, "gdn_prefill: need 1 <= Dk, Dv <= %d (got Dk=%d Dv=%d)",
                    gdn::kMaxHeadDim, Dk, Dv);
    if (dt != GDN_DTYPE_F32 && dt != GDN_DTYPE_BF16)
        return fail(GDN_EINVAL, "gdn_prefill: unknown dtype %d", (int)dt);
    return GDN_OK;
}

}  // namespace

extern "C" {

size_t gdn_prefill_workspace_bytes(int B, int Hk, int Hv, int S, int Dk, int Dv,
                                   gdn_dtype dtype) {
    if (check_prefill_shape(B, Hk, Hv, S, Dk, Dv, dtype) != GDN_OK) return (size_t)-1;
    gdn::PrefillArgs a{};
    a.B = B, a.Hk = Hk, a.Hv = Hv, a.S = S, a.Dk = Dk, a.Dv = Dv;
    return gdn::prefill_tc_supported(a, dtype == GDN_DTYPE_BF16)
               ? gdn::prefill_tc_workspace_bytes(B, Hv, S)
               : 0;
}

gdn_status gdn_prefill(const void* q, const void* k, const void* v, const float* g_log,
                       const float* beta, float scale, gdn_dtype dtype, int B, int Hk, int Hv,
                       int S, int Dk, int Dv, float* state, int state_is_input, void* out,
                       void* workspace, size_t workspace_bytes, void* stream) {
    gdn_status st = check_prefill_shape(B, Hk, Hv, S, Dk, Dv, dtype);
    if (st != GDN_OK) return st;
    const bool tok = S > 0;  // per-token tensors may be NULL only when S == 0
    if (!ptr_ok(q, tok) || !ptr_ok(k, tok) || !ptr_ok(v, tok) || !ptr_ok(g_log, tok) ||
        !ptr_ok(beta, tok) || !ptr_ok(out, tok) || !ptr_ok(state, true))
        return fail(GDN_EINVAL, "gdn_prefill: q, k, v, g_log, beta, out and state must be "
                    "non-NULL, 16-byte aligned device pointers");
    const size_t need = gdn_prefill_workspace_bytes(B, Hk, Hv, S, Dk, Dv, dtype);
    if (workspace_bytes < need || (need > 0 && !ptr_ok(workspace, true)))
        return fail(GDN_EINVAL, "gdn_prefill: workspace of %zu bytes needed, %zu given",
                    need, workspace_bytes);

    gdn::PrefillArgs a{q, k, v, g_log, beta, scale, B, Hk, Hv, S, Dk, Dv,
                       state, state_is_input ? 1 : 0, out, workspace, workspace_bytes};
    const cudaStream_t s = static_cast<cudaStream_t>(stream);
    int launched = 0;
    const bool bf16 = dtype == GDN_DTYPE_BF16;
    const cudaError_t e = gdn::prefill_tc_supported(a, bf16)
                              ? gdn::launch_prefill_tc_overlapped(a, s, &launched)
                              : gdn::launch_prefill_simt(a, bf16, s, &launched);
    g_launches += (unsigned long long)launched;
    if (e != cudaSuccess)
        return fail(GDN_ECUDA, "gdn_prefill: launch failed: %s", cudaGetErrorString(e));
    return GDN_OK;
}

size_t gdn_prefill_varlen_workspace_bytes(int N, int Hk, int Hv, int T, int Dk, int Dv,
                                          gdn_dtype dtype) {
    if (N < 0 || N > kMaxSequences || check_prefill_shape(1, Hk, Hv, T, Dk, Dv, dtype) != GDN_OK)
        return (size_t)-1;
    gdn::PrefillArgs a{};
    a.B = 1, a.Hk = Hk, a.Hv = Hv, a.S = T, a.Dk = Dk, a.Dv = Dv;
    if (gdn::prefill_tc_supported(a, dtype == GDN_DTYPE_BF16))
        return gdn::prefill_tc_varlen_workspace_bytes(N, Hv, T);
    return (gdn::varlen_table_ints(N) * sizeof(int) + 15) / 16 * 16;
}

gdn_status gdn_prefill_varlen(const void* q, const void* k, const void* v, const float* g_log,
                              const float* beta, float scale, gdn_dtype dtype,
                              const int* cu_seqlens, int N, int Hk, int Hv, int T, int Dk,
                              int Dv, float* state, int state_is_input, void* out,
                              void* workspace, size_t workspace_bytes, void* stream) {
    gdn_status st = check_prefill_shape(1, Hk, Hv, T, Dk, Dv, dtype);
    if (st != GDN_OK) return st;
    if (N < 0 || N > kMaxSequences)
        return fail(GDN_EINVAL, "gdn_prefill_varlen: need 0 <= N <= %d (got N=%d)",
                    kMaxSequences, N);
    if (N == 0) return GDN_OK;
    const bool tok = T > 0;
    if (!ptr_ok(q, tok) || !ptr_ok(k, tok) || !ptr_ok(v, tok) || !ptr_ok(g_log, tok) ||
        !ptr_ok(beta, tok) || !ptr_ok(out, tok) || !ptr_ok(state, true) ||
        !ptr_ok(cu_seqlens, true))
        return fail(GDN_EINVAL, "gdn_prefill_varlen: q, k, v, g_log, beta, out, state and "
                    "cu_seqlens must be non-NULL, 16-byte aligned device pointers");
    const size_t need = gdn_prefill_varlen_workspace_bytes(N, Hk, Hv, T, Dk, Dv, dtype);
    if (workspace_bytes < need || !ptr_ok(workspace, true))
        return fail(GDN_EINVAL, "gdn_prefill_varlen: workspace of %zu bytes needed, %zu given",
                    need, workspace_bytes);
    gdn::PrefillArgs a{q, k, v, g_log, beta, scale, 1, Hk, Hv, T, Dk, Dv,
                       state, state_is_input ? 1 : 0, out, workspace, workspace_bytes};
    a.cu_seqlens = cu_seqlens;
    a.N = N;
    a.table = static_cast<int*>(workspace);  // the fp32 path's table opens the workspace
    const cudaStream_t s = static_cast<cudaStream_t>(stream);
    int launched = 0;
    const bool bf16 = dtype == GDN_DTYPE_BF16;
    const cudaError_t e = gdn::prefill_tc_supported(a, bf16)
                              ? gdn::launch_prefill_tc_varlen(a, s, &launched)
                              : gdn::launch_prefill_simt(a, bf16, s, &launched);
    g_launches += (unsigned long long)launched;
    if (e != cudaSuccess)
        return fail(GDN_ECUDA, "gdn_prefill_varlen: launch failed: %s", cudaGetErrorString(e));
    return GDN_OK;
}

gdn_status gdn_prefill_noalloc(const void* q, const void* k, const void* v, const float* g_log,
                               const float* beta, float scale, gdn_dtype dtype, int B, int Hk,
                               int Hv, int S, int Dk, int Dv, float* state, int state_is_input,
                               void* out, void* stream) {
    const size_t need = gdn_prefill_workspace_bytes(B, Hk, Hv, S, Dk, Dv, dtype);
    if (need == (size_t)-1 || need == 0)  // a shape error, or a path without scratch
        return gdn_prefill(q, k, v, g_log, beta, scale, dtype, B, Hk, Hv, S, Dk, Dv, state,
                           state_is_input, out, nullptr, 0, stream);
    const bool tok = S > 0;
    if (!ptr_ok(q, tok) || !ptr_ok(k, tok) || !ptr_ok(v, tok) || !ptr_ok(g_log, tok) ||
        !ptr_ok(beta, tok) || !ptr_ok(out, tok) || !ptr_ok(state, true))
        return fail(GDN_EINVAL, "gdn_prefill_noalloc: q, k, v, g_log, beta, out and state must "
                    "be non-NULL, 16-byte aligned device pointers");
    // the sequence in segments of `seg` chunks, each using the whole static scratch; the
    // state carries over from one segment to the next
    const size_t units = kStaticScratchBytes / gdn::prefill_tc_unit_bytes();
    const size_t heads = (size_t)B * (size_t)Hv;
    if (heads > units)
        return fail(GDN_EUNSUPPORTED, "gdn_prefill_noalloc: B*Hv = %zu exceeds the %zu "
                    "(batch, head) pairs its static scratch holds", heads, units);
    void* scratch = nullptr;
    cudaError_t e = scratch_address(&scratch);
    if (e != cudaSuccess || scratch == nullptr)
        return fail(GDN_ECUDA, "gdn_prefill_noalloc: device address of the static scratch: %s",
                    cudaGetErrorString(e));
    const int nch = (S + 63) / 64;
    const int seg = (int)std::min<size_t>(units / heads, (size_t)nch);
    const cudaStream_t s = static_cast<cudaStream_t>(stream);
    for (int c0 = 0; c0 < nch; c0 += seg) {
        gdn::PrefillArgs a{q,     k,     v,  g_log, beta,  scale,
                           B,     Hk,    Hv, S,     Dk,    Dv,
                           state, (c0 == 0 && !state_is_input) ? 0 : 1,
                           out,   scratch, kStaticScratchBytes};
        int launched = 0;
        e = gdn::launch_prefill_tc(a, c0, std::min(seg, nch - c0), s, &launched);
        g_launches += (unsigned long long)launched;
        if (e != cudaSuccess)
            return fail(GDN_ECUDA, "gdn_prefill_noalloc: launch failed: %s",
                        cudaGetErrorString(e));
    }
    return GDN_OK;
}

}  // extern "C"

namespace {

// The decode step, T tokens in a row: validation, then one launch.
gdn_status decode_impl(const char* fn, const void* q, const void* k, const void* v,
                       const void* b, const void* a, const float* A_log, const float* dt_bias,
                       const void* z, const float* norm_weight, const float* state_in,
                       float* state_out, void* out, int T, int BH, int num_v_heads, int K,
                       int V, void* stream) {
    if (T < 0 || BH < 0 || num_v_heads < 1 || BH % num_v_heads != 0)
        return fail(GDN_EINVAL, "%s: need T >= 0, BH >= 0 and BH %% num_v_heads == 0 "
                    "(got T=%d BH=%d num_v_heads=%d)", fn, T, BH, num_v_heads);
    if (K < 1 || K > gdn::kMaxHeadDim || V < 1 || V > gdn::kMaxHeadDim)
        return fail(GDN_EINVAL, "%s: need 1 <= K, V <= %d (got K=%d V=%d)", fn,
                    gdn::kMaxHeadDim, K, V);
    const bool rows = BH > 0 && T > 0;
    if (!ptr_ok(q, rows) || !ptr_ok(k, rows) || !ptr_ok(v, rows) || !ptr_ok(b, rows) ||
        !ptr_ok(a, rows) || !ptr_ok(z, rows) || !ptr_ok(state_in, rows) ||
        !ptr_ok(state_out, rows) || !ptr_ok(out, rows) || !ptr_ok(A_log, true) ||
        !ptr_ok(dt_bias, true) || !ptr_ok(norm_weight, true))
        return fail(GDN_EINVAL, "%s: every pointer must be a non-NULL, 16-byte aligned "
                    "device pointer", fn);
    if (state_in != state_out && rows) {
        const uintptr_t i0 = reinterpret_cast<uintptr_t>(state_in);
        const uintptr_t o0 = reinterpret_cast<uintptr_t>(state_out);
        const uintptr_t n = (uintptr_t)BH * K * V * sizeof(float);
        if (i0 < o0 + n && o0 < i0 + n)
            return fail(GDN_EINVAL, "%s: state_out overlaps state_in without being equal "
                        "to it", fn);
    }
    gdn::DecodeArgs d{static_cast<const __nv_bfloat16*>(q), static_cast<const __nv_bfloat16*>(k),
                      static_cast<const __nv_bfloat16*>(v), static_cast<const __nv_bfloat16*>(b),
                      static_cast<const __nv_bfloat16*>(a), A_log, dt_bias,
                      static_cast<const __nv_bfloat16*>(z), norm_weight, state_in, state_out,
                      static_cast<__nv_bfloat16*>(out), BH, num_v_heads, K, V, T};
    const cudaError_t e = gdn::launch_decode(d, static_cast<cudaStream_t>(stream));
    if (rows) g_launches += 1;
    if (e != cudaSuccess)
        return fail(GDN_ECUDA, "%s: launch failed: %s", fn, cudaGetErrorString(e));
    return GDN_OK;
}

}  // namespace

extern "C" {

gdn_status gdn_decode_step(const void* q, const void* k, const void* v, const void* b,
                           const void* a, const float* A_log, const float* dt_bias,
                           const void* z, const float* norm_weight, const float* state_in,
                           float* state_out, void* out, int BH, int num_v_heads, int K, int V,
                           void* stream) {
    return decode_impl("gdn_decode_step", q, k, v, b, a, A_log, dt_bias, z, norm_weight,
                       state_in, state_out, out, 1, BH, num_v_heads, K, V, stream);
}

gdn_status gdn_decode_multi(const void* q, const void* k, const void* v, const void* b,
                            const void* a, const float* A_log, const float* dt_bias,
                            const void* z, const float* norm_weight, const float* state_in,
                            float* state_out, void* out, int T, int BH, int num_v_heads, int K,
                            int V, void* stream) {
    return decode_impl("gdn_decode_multi", q, k, v, b, a, A_log, dt_bias, z, norm_weight,
                       state_in, state_out, out, T, BH, num_v_heads, K, V, stream);
}

gdn_status gdn_conv1d_decode(const void* x, const float* conv_weight, const void* conv_state_in,
                             void* conv_state_out, void* q_out, void* k_out, void* v_out, int B,
                             int num_k_heads, int num_v_heads, int head_k_dim, int head_v_dim,
                             int K_win, void* stream) {
    if (B < 0 || num_k_heads < 1 || num_v_heads < 1 || num_v_heads % num_k_heads != 0)
        return fail(GDN_EINVAL, "gdn_conv1d_decode: need B >= 0 and num_v_heads a multiple of "
                    "num_k_heads (got B=%d num_k_heads=%d num_v_heads=%d)", B, num_k_heads,
                    num_v_heads);
    if (head_k_dim < 1 || head_k_dim > gdn::kMaxHeadDim || head_v_dim < 1 ||
        head_v_dim > gdn::kMaxHeadDim)
        return fail(GDN_EINVAL, "gdn_conv1d_decode: need 1 <= head_k_dim, head_v_dim <= %d",
                    gdn::kMaxHeadDim);
    if (K_win < 1 || K_win > gdn::kMaxConvWidth)
        return fail(GDN_EINVAL, "gdn_conv1d_decode: need 1 <= K_win <= %d (got %d)",
                    gdn::kMaxConvWidth, K_win);
    const bool rows = B > 0;
    if (!ptr_ok(x, rows) || !ptr_ok(conv_weight, true) || !ptr_ok(conv_state_in, rows) ||
        !ptr_ok(conv_state_out, rows) || !ptr_ok(q_out, rows) || !ptr_ok(k_out, rows) ||
        !ptr_ok(v_out, rows))
        return fail(GDN_EINVAL, "gdn_conv1d_decode: every pointer must be a non-NULL, "
                    "16-byte aligned device pointer");
    const size_t C = 2 * (size_t)num_k_heads * head_k_dim + (size_t)num_v_heads * head_v_dim;
    if (conv_state_in != conv_state_out && rows) {
        const uintptr_t i0 = reinterpret_cast<uintptr_t>(conv_state_in);
        const uintptr_t o0 = reinterpret_cast<uintptr_t>(conv_state_out);
        const uintptr_t n = (uintptr_t)B * C * K_win * 2;
        if (i0 < o0 + n && o0 < i0 + n)
            return fail(GDN_EINVAL, "gdn_conv1d_decode: conv_state_out overlaps conv_state_in "
                        "without being equal to it");
    }
    gdn::Conv1dArgs d{static_cast<const __nv_bfloat16*>(x), conv_weight,
                      static_cast<const __nv_bfloat16*>(conv_state_in),
                      static_cast<__nv_bfloat16*>(conv_state_out),
                      static_cast<__nv_bfloat16*>(q_out), static_cast<__nv_bfloat16*>(k_out),
                      static_cast<__nv_bfloat16*>(v_out), B, num_k_heads, num_v_heads,
                      head_k_dim, head_v_dim, K_win};
    const cudaError_t e = gdn::launch_conv1d_decode(d, static_cast<cudaStream_t>(stream));
    if (rows) g_launches += 1;
    if (e != cudaSuccess)
        return fail(GDN_ECUDA, "gdn_conv1d_decode: launch failed: %s", cudaGetErrorString(e));
    return GDN_OK;
}

gdn_status gdn_unit_lower_inverse(const float* A, float* T, int n, int C, int algorithm,
                                  void* stream) {
    if (n < 0 || n > (1 << 30) / (64 * 64))
        return fail(GDN_EINVAL, "gdn_unit_lower_inverse: need 0 <= n (got %d)", n);
    if (C != 64)
        return fail(GDN_EUNSUPPORTED, "gdn_unit_lower_inverse: only C = 64 (got %d)", C);
    if (algorithm != GDN_TRIL_SUBSTITUTION && algorithm != GDN_TRIL_NEUMANN)
        return fail(GDN_EINVAL, "gdn_unit_lower_inverse: unknown algorithm %d", algorithm);
    if (!ptr_ok(A, n > 0) || !ptr_ok(T, n > 0))
        return fail(GDN_EINVAL, "gdn_unit_lower_inverse: A and T must be non-NULL, 16-byte "
                    "aligned device pointers");
    if (A != T && n > 0) {
        const uintptr_t a0 = reinterpret_cast<uintptr_t>(A), t0 = reinterpret_cast<uintptr_t>(T);
        const uintptr_t bytes = (uintptr_t)n * 64 * 64 * sizeof(float);
        if (a0 < t0 + bytes && t0 < a0 + bytes)
            return fail(GDN_EINVAL, "gdn_unit_lower_inverse: T overlaps A without being "
                        "equal to it");
    }
    const cudaError_t e = gdn::launch_tril_inverse(A, T, n, algorithm,
                                                   static_cast<cudaStream_t>(stream));
    if (n > 0) g_launches += 1;
    if (e != cudaSuccess)
        return fail(GDN_ECUDA, "gdn_unit_lower_inverse: launch failed: %s",
                    cudaGetErrorString(e));
    return GDN_OK;
}

const char* gdn_last_error(void) { return g_last_error.c_str(); }

unsigned long long gdn_launch_count(void) { return g_launches.load(); }

gdn_status gdn_get_device_status(void* stream) {
    const cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess)
        return fail(GDN_ECUDA, "gdn_get_device_status: %s", cudaGetErrorString(e));
    const uint32_t bits =
        gdn::prefill_tc_take_status() | gdn::tril_take_status() | gdn::decode_take_status();
    if (bits & gdn::kStatusBadSeqlens)
        return fail(GDN_EINVAL, "gdn_prefill_varlen: cu_seqlens was not 0 = cu[0] <= ... <= "
                    "cu[N] <= T; every sequence was treated as empty");
    if (bits != 0)
        return fail(GDN_ETIMEOUT, "a kernel gave up a bounded wait (status bits 0x%x)", bits);
    return GDN_OK;
}

}  // extern "C"
