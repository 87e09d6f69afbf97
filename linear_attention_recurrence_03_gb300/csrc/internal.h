// internal.h -- declarations shared by the library's translation units (not part of
// the C ABI; see include/gdn.h for that).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cstddef>
#include <cstdint>

namespace gdn {

// Largest head dimension ("GDN CTE Kernel API Reference", Notes: Dk, Dv <= 128).
constexpr int kMaxHeadDim = 128;

// Unstated constants, read as the usual choices: l2norm eps and RMSNorm eps
// ("GDN TKG Kernel API Reference" names both operations but no eps).
constexpr float kEpsL2 = 1e-6f;
constexpr float kEpsRms = 1e-6f;

struct PrefillArgs {
    const void* q;      // [B, Hk, S, Dk]
    const void* k;      // [B, Hk, S, Dk]
    const void* v;      // [B, Hv, S, Dv]
    const float* g;     // [B, Hv, S]
    const float* beta;  // [B, Hv, S]
    float scale;
    int B, Hk, Hv, S, Dk, Dv;
    float* state;       // [B, Hv, Dk, Dv]
    int state_is_input;
    void* out;          // [B, Hv, S, Dv]
    void* workspace;
    size_t workspace_bytes;
    // Variable-length batch (cu_seqlens != NULL): B == 1, the N sequences are packed
    // along S (sequence n: tokens cu_seqlens[n] .. cu_seqlens[n+1] - 1), state is
    // [N, Hv, Dk, Dv]; `table` is device scratch of varlen_table_ints(N) ints that the
    // setup kernel fills (chunk bases, then a validity flag).
    const int* cu_seqlens = nullptr;
    int N = 0;
    int* table = nullptr;
};

// Ints of the variable-length batch's table: N + 1 chunk bases and a validity flag.
inline size_t varlen_table_ints(int N) { return (size_t)N + 2; }
// Fills the table from cu_seqlens (one CTA): chunk bases of 64-token chunks and the flag
// (0 when cu_seqlens is not 0 = cu[0] <= cu[1] <= ... <= cu[N] <= S; the status word
// then gets its input bit and every sequence is treated as empty).
cudaError_t launch_varlen_setup(const PrefillArgs& a, cudaStream_t stream);

struct DecodeArgs {
    const __nv_bfloat16* q;   // [T, BH, K]
    const __nv_bfloat16* k;   // [T, BH, K]
    const __nv_bfloat16* v;   // [T, BH, V]
    const __nv_bfloat16* b;   // [T, BH]
    const __nv_bfloat16* a;   // [T, BH]
    const float* A_log;       // [H]
    const float* dt_bias;     // [H]
    const __nv_bfloat16* z;   // [T, BH, V]
    const float* norm_weight; // [V]
    const float* state_in;    // [BH, K, V]
    float* state_out;         // [BH, K, V]
    __nv_bfloat16* out;       // [T, BH, V]
    int BH, H, K, V;
    int T;                    // consecutive tokens per call (1: the single decode step)
    int pf_rows = 0;          // set by the launcher: rows ahead whose state goes to L2
};

// SIMT fp32 chunked prefill (any Dk, Dv <= 128; q/k/v fp32 or bf16). *launched
// receives the number of kernels enqueued.
cudaError_t launch_prefill_simt(const PrefillArgs& a, bool bf16, cudaStream_t stream,
                                int* launched);

// tcgen05 chunked prefill (bf16, Dk = Dv = 128, S > 0): a parallel prep kernel writes
// up to 64.5 KB of operand tiles and scalars per (batch, value head, 64-token chunk) to
// the workspace, then a carry kernel runs the sequential part. *launched receives the
// kernels enqueued.
bool prefill_tc_supported(const PrefillArgs& a, bool bf16);
size_t prefill_tc_workspace_bytes(int B, int Hv, int S);
size_t prefill_tc_unit_bytes();
// Variable-length batch on the tensor cores: the workspace holds Hv * (ceil(S/64) + N)
// units, then the table.
size_t prefill_tc_varlen_workspace_bytes(int N, int Hv, int S);
cudaError_t launch_prefill_tc_varlen(const PrefillArgs& a, cudaStream_t stream, int* launched);
// Status bit of a malformed cu_seqlens (prefill_tc_take_status).
constexpr uint32_t kStatusBadSeqlens = 16u;
// Processes chunks c0 .. c0 + nseg - 1 of the sequence (64 tokens each) with a workspace of
// B * Hv * nseg units; the state carries over between consecutive calls.
cudaError_t launch_prefill_tc(const PrefillArgs& a, int c0, int nseg, cudaStream_t stream,
                              int* launched);
// The whole sequence with a workspace of B * Hv * ceil(S / 64) units, in the segments
// prefill_tc_schedule(...) gives when the carry leaves SMs free: the prep of segment j + 1
// (helper stream, low priority) then runs beside the carry of segment j (helper stream,
// high priority), forked from and joined back to `stream` by events.
cudaError_t launch_prefill_tc_overlapped(const PrefillArgs& a, cudaStream_t stream,
                                         int* launched);
// Segment sizes (chunks) of the overlapped schedule into sizes[0 .. n-1]; returns n (at
// most max_segments, 1 when the carry leaves too few SMs free or there are few chunks).
int prefill_tc_schedule(int B, int Hv, int nch, int sms, int* sizes, int max_segments);

// Depthwise causal conv1d decode token + silu + window shift, split into q | k | v with
// q and k repeated over the value heads.
constexpr int kMaxConvWidth = 16;
struct Conv1dArgs {
    const __nv_bfloat16* x;         // [B, conv_dim], conv_dim = 2 Hk Dk + Hv Dv
    const float* weight;            // [conv_dim, K_win]
    const __nv_bfloat16* state_in;  // [B, conv_dim, K_win]
    __nv_bfloat16* state_out;       // [B, conv_dim, K_win] (may equal state_in)
    __nv_bfloat16* q;               // [B * Hv, Dk]
    __nv_bfloat16* k;               // [B * Hv, Dk]
    __nv_bfloat16* v;               // [B * Hv, Dv]
    int B, Hk, Hv, Dk, Dv, K_win;
};
cudaError_t launch_conv1d_decode(const Conv1dArgs& a, cudaStream_t stream);

// (I + A)^-1 of n strictly lower-triangular 64 x 64 fp32 matrices: algorithm 0 forward
// substitution, 1 the Neumann product on the tcgen05 tensor cores (kind::tf32).
cudaError_t launch_tril_inverse(const float* A, float* T, int n, int algorithm,
                                cudaStream_t stream);

// Fused decode step, T tokens in a row (the state read and written once).
cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t stream);

// cuTensorMapEncodeTiled from the driver (nullptr when the driver has none).
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder();

// Device status word of each translation unit that has bounded waits: returns the
// bits set since the last call and clears them (the stream must be synchronised).
uint32_t prefill_tc_take_status();
uint32_t tril_take_status();
uint32_t decode_take_status();

}  // namespace gdn
