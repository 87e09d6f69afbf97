"""Python binding of the C ABI in include/gdn.h (ctypes over ``libgdn.so``).

Argument marshalling only: the functions check that tensors are CUDA, contiguous and of
the right dtype and shape, allocate outputs with torch when the caller passes none, and
call the library. Every step of the recurrence runs in the library's CUDA kernels; there
is no CPU path. If ``libgdn.so`` has not been built the first call raises.

Sources: "GDN CTE Kernel API Reference" (gdn_prefill) and "GDN TKG Kernel API
Reference" (gdn_decode_step), AWS Neuron NKI library.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libgdn.so")

GDN_OK, GDN_EINVAL, GDN_EUNSUPPORTED, GDN_ECUDA, GDN_ETIMEOUT = range(5)
GDN_DTYPE_F32, GDN_DTYPE_BF16 = 0, 1
GDN_TRIL_SUBSTITUTION, GDN_TRIL_NEUMANN = 0, 1
STATUS_NAMES = {0: "GDN_OK", 1: "GDN_EINVAL", 2: "GDN_EUNSUPPORTED", 3: "GDN_ECUDA",
                4: "GDN_ETIMEOUT"}

# Every symbol include/gdn.h declares.
EXPORTS = ("gdn_prefill_workspace_bytes", "gdn_prefill", "gdn_prefill_noalloc",
           "gdn_prefill_varlen_workspace_bytes", "gdn_prefill_varlen",
           "gdn_decode_step", "gdn_decode_multi", "gdn_conv1d_decode",
           "gdn_unit_lower_inverse", "gdn_last_error",
           "gdn_get_device_status", "gdn_launch_count")

_lock = threading.Lock()
_lib = None


class GDNError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {message}")
        self.status = status


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load ``libgdn.so`` and declare the C signatures. Raises if it is missing."""
    global _lib
    with _lock:
        if _lib is not None and path == LIB_PATH:
            return _lib
        if not os.path.exists(path):
            raise RuntimeError(f"{path} is missing: build the CUDA library first "
                               "(__graft_entry__.build() or python -m "
                               "linear_attention_recurrence_03_gb300.build)")
        lib = ctypes.CDLL(path)
        vp, i, f, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
        lib.gdn_prefill_workspace_bytes.argtypes = [i] * 7
        lib.gdn_prefill_workspace_bytes.restype = sz
        lib.gdn_prefill.argtypes = [vp, vp, vp, vp, vp, f, i, i, i, i, i, i, i, vp, i, vp,
                                    vp, sz, vp]
        lib.gdn_prefill.restype = i
        lib.gdn_prefill_noalloc.argtypes = [vp, vp, vp, vp, vp, f, i, i, i, i, i, i, i, vp, i,
                                            vp, vp]
        lib.gdn_prefill_noalloc.restype = i
        lib.gdn_prefill_varlen_workspace_bytes.argtypes = [i] * 7
        lib.gdn_prefill_varlen_workspace_bytes.restype = sz
        lib.gdn_prefill_varlen.argtypes = [vp, vp, vp, vp, vp, f, i, vp, i, i, i, i, i, i, vp,
                                           i, vp, vp, sz, vp]
        lib.gdn_prefill_varlen.restype = i
        lib.gdn_decode_step.argtypes = [vp] * 12 + [i] * 4 + [vp]
        lib.gdn_decode_step.restype = i
        lib.gdn_decode_multi.argtypes = [vp] * 12 + [i] * 5 + [vp]
        lib.gdn_decode_multi.restype = i
        lib.gdn_conv1d_decode.argtypes = [vp] * 7 + [i] * 6 + [vp]
        lib.gdn_conv1d_decode.restype = i
        lib.gdn_unit_lower_inverse.argtypes = [vp, vp, i, i, i, vp]
        lib.gdn_unit_lower_inverse.restype = i
        lib.gdn_last_error.argtypes = []
        lib.gdn_last_error.restype = ctypes.c_char_p
        lib.gdn_get_device_status.argtypes = [vp]
        lib.gdn_get_device_status.restype = i
        lib.gdn_launch_count.argtypes = []
        lib.gdn_launch_count.restype = ctypes.c_ulonglong
        if path == LIB_PATH:
            _lib = lib
        return lib


def _check(status: int):
    if status != GDN_OK:
        raise GDNError(status, gdn_last_error())


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, torch.cuda.Stream):
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))


def _need(t, name, dtype, shape, device):
    if t.device != device or not t.is_cuda:
        raise ValueError(f"{name} must be on {device}")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def gdn_last_error() -> str:
    return load_library().gdn_last_error().decode()


def gdn_launch_count() -> int:
    """Kernels the library has enqueued in this process so far."""
    return int(load_library().gdn_launch_count())


def gdn_get_device_status(stream=None) -> int:
    """Synchronise the stream and return the device status (GDN_OK or GDN_ETIMEOUT)."""
    return load_library().gdn_get_device_status(_stream(stream))


def gdn_prefill_workspace_bytes(B, Hk, Hv, S, Dk, Dv, dtype) -> int:
    dt = GDN_DTYPE_BF16 if dtype == torch.bfloat16 else GDN_DTYPE_F32
    n = load_library().gdn_prefill_workspace_bytes(B, Hk, Hv, S, Dk, Dv, dt)
    if n == ctypes.c_size_t(-1).value:
        raise ValueError("invalid prefill shape")
    return int(n)


def gdn_prefill(q, k, v, g_log, beta, scale, state=None, out=None, workspace=None,
                stream=None, state_is_input=None):
    """Chunked prefill. q,k [B,Hk,S,Dk], v [B,Hv,S,Dv] (fp32 or bf16, one dtype);
    g_log, beta [B,Hv,S] fp32. ``state`` [B,Hv,Dk,Dv] fp32, if given, is the initial
    state and is updated in place (with ``state_is_input=False`` it is only written: zero
    initial state, no load); if None a zero initial state is used and a new tensor
    returned. Returns (out [B,Hv,S,Dv], state)."""
    B, Hk, S, Dk = q.shape
    Hv, Dv = v.shape[1], v.shape[3]
    dev, dt = q.device, q.dtype
    if dt not in (torch.float32, torch.bfloat16):
        raise ValueError("q must be float32 or bfloat16")
    _need(q, "q", dt, (B, Hk, S, Dk), dev)
    _need(k, "k", dt, (B, Hk, S, Dk), dev)
    _need(v, "v", dt, (B, Hv, S, Dv), dev)
    _need(g_log, "g_log", torch.float32, (B, Hv, S), dev)
    _need(beta, "beta", torch.float32, (B, Hv, S), dev)
    if state_is_input is None:
        state_is_input = state is not None
    if state is None:
        if state_is_input:
            raise ValueError("state_is_input needs a state")
        state = torch.empty((B, Hv, Dk, Dv), dtype=torch.float32, device=dev)
    _need(state, "state", torch.float32, (B, Hv, Dk, Dv), dev)
    if out is None:
        out = torch.empty((B, Hv, S, Dv), dtype=dt, device=dev)
    _need(out, "out", dt, (B, Hv, S, Dv), dev)
    need = gdn_prefill_workspace_bytes(B, Hk, Hv, S, Dk, Dv, dt)
    if need and (workspace is None or workspace.numel() * workspace.element_size() < need):
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    wbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    code = GDN_DTYPE_BF16 if dt == torch.bfloat16 else GDN_DTYPE_F32
    _check(load_library().gdn_prefill(
        _ptr(q), _ptr(k), _ptr(v), _ptr(g_log), _ptr(beta), float(scale), code, B, Hk, Hv, S,
        Dk, Dv, _ptr(state), int(state_is_input), _ptr(out), _ptr(workspace), wbytes,
        _stream(stream)))
    return out, state


def gdn_prefill_noalloc(q, k, v, g_log, beta, scale, state=None, out=None, stream=None):
    """As gdn_prefill, through the entry point that uses the library's own static scratch
    instead of a workspace (calls must not run concurrently)."""
    B, Hk, S, Dk = q.shape
    Hv, Dv = v.shape[1], v.shape[3]
    dev, dt = q.device, q.dtype
    if dt not in (torch.float32, torch.bfloat16):
        raise ValueError("q must be float32 or bfloat16")
    _need(q, "q", dt, (B, Hk, S, Dk), dev)
    _need(k, "k", dt, (B, Hk, S, Dk), dev)
    _need(v, "v", dt, (B, Hv, S, Dv), dev)
    _need(g_log, "g_log", torch.float32, (B, Hv, S), dev)
    _need(beta, "beta", torch.float32, (B, Hv, S), dev)
    state_is_input = state is not None
    if state is None:
        state = torch.empty((B, Hv, Dk, Dv), dtype=torch.float32, device=dev)
    _need(state, "state", torch.float32, (B, Hv, Dk, Dv), dev)
    if out is None:
        out = torch.empty((B, Hv, S, Dv), dtype=dt, device=dev)
    _need(out, "out", dt, (B, Hv, S, Dv), dev)
    code = GDN_DTYPE_BF16 if dt == torch.bfloat16 else GDN_DTYPE_F32
    _check(load_library().gdn_prefill_noalloc(
        _ptr(q), _ptr(k), _ptr(v), _ptr(g_log), _ptr(beta), float(scale), code, B, Hk, Hv, S,
        Dk, Dv, _ptr(state), int(state_is_input), _ptr(out), _stream(stream)))
    return out, state


def gdn_decode_step(q, k, v, b, a, A_log, dt_bias, z, norm_weight, state_in, num_v_heads,
                    state_out=None, out=None, stream=None):
    """Fused decode step. q,k [BH,K], v,z [BH,V], b,a [BH] bf16; A_log, dt_bias
    [num_v_heads], norm_weight [V], state_in [BH,K,V] fp32. ``state_out`` may be
    ``state_in`` (in place); if None a new tensor is returned. Returns (out [BH,V] bf16,
    state_out)."""
    BH, K = q.shape
    V = v.shape[1]
    dev, bf = q.device, torch.bfloat16
    for t, n, sh in ((q, "q", (BH, K)), (k, "k", (BH, K)), (v, "v", (BH, V)), (z, "z", (BH, V)),
                     (b, "b", (BH,)), (a, "a", (BH,))):
        _need(t, n, bf, sh, dev)
    _need(A_log, "A_log", torch.float32, (num_v_heads,), dev)
    _need(dt_bias, "dt_bias", torch.float32, (num_v_heads,), dev)
    _need(norm_weight, "norm_weight", torch.float32, (V,), dev)
    _need(state_in, "state_in", torch.float32, (BH, K, V), dev)
    if state_out is None:
        state_out = torch.empty_like(state_in)
    _need(state_out, "state_out", torch.float32, (BH, K, V), dev)
    if out is None:
        out = torch.empty((BH, V), dtype=bf, device=dev)
    _need(out, "out", bf, (BH, V), dev)
    _check(load_library().gdn_decode_step(
        _ptr(q), _ptr(k), _ptr(v), _ptr(b), _ptr(a), _ptr(A_log), _ptr(dt_bias), _ptr(z),
        _ptr(norm_weight), _ptr(state_in), _ptr(state_out), _ptr(out), BH, num_v_heads, K, V,
        _stream(stream)))
    return out, state_out


def gdn_decode_multi(q, k, v, b, a, A_log, dt_bias, z, norm_weight, state_in, num_v_heads,
                     state_out=None, out=None, stream=None):
    """T consecutive fused decode tokens in one call. q,k [T,BH,K], v,z [T,BH,V], b,a
    [T,BH] bf16; the rest as gdn_decode_step. Returns (out [T,BH,V] bf16, state_out)."""
    T, BH, K = q.shape
    V = v.shape[2]
    dev, bf = q.device, torch.bfloat16
    for t, n, sh in ((q, "q", (T, BH, K)), (k, "k", (T, BH, K)), (v, "v", (T, BH, V)),
                     (z, "z", (T, BH, V)), (b, "b", (T, BH)), (a, "a", (T, BH))):
        _need(t, n, bf, sh, dev)
    _need(A_log, "A_log", torch.float32, (num_v_heads,), dev)
    _need(dt_bias, "dt_bias", torch.float32, (num_v_heads,), dev)
    _need(norm_weight, "norm_weight", torch.float32, (V,), dev)
    _need(state_in, "state_in", torch.float32, (BH, K, V), dev)
    if state_out is None:
        state_out = torch.empty_like(state_in)
    _need(state_out, "state_out", torch.float32, (BH, K, V), dev)
    if out is None:
        out = torch.empty((T, BH, V), dtype=bf, device=dev)
    _need(out, "out", bf, (T, BH, V), dev)
    _check(load_library().gdn_decode_multi(
        _ptr(q), _ptr(k), _ptr(v), _ptr(b), _ptr(a), _ptr(A_log), _ptr(dt_bias), _ptr(z),
        _ptr(norm_weight), _ptr(state_in), _ptr(state_out), _ptr(out), T, BH, num_v_heads, K,
        V, _stream(stream)))
    return out, state_out


def gdn_conv1d_decode(x, conv_weight, conv_state_in, num_k_heads, num_v_heads, head_k_dim,
                      head_v_dim, conv_state_out=None, stream=None):
    """One token through the depthwise causal conv + SiLU + window shift, split into
    q | k | v with q, k repeated over the value heads. x [B, conv_dim] bf16,
    conv_weight [conv_dim, K_win] fp32, conv_state_in [B, conv_dim, K_win] bf16.
    ``conv_state_out`` may be ``conv_state_in`` (in place). Returns (q, k, v,
    conv_state_out): q, k [B*num_v_heads, head_k_dim], v [B*num_v_heads, head_v_dim]."""
    B, C = x.shape
    K_win = conv_weight.shape[1]
    dev, bf = x.device, torch.bfloat16
    if C != 2 * num_k_heads * head_k_dim + num_v_heads * head_v_dim:
        raise ValueError("x: conv_dim must be 2 * num_k_heads * head_k_dim + "
                         "num_v_heads * head_v_dim")
    _need(x, "x", bf, (B, C), dev)
    _need(conv_weight, "conv_weight", torch.float32, (C, K_win), dev)
    _need(conv_state_in, "conv_state_in", bf, (B, C, K_win), dev)
    if conv_state_out is None:
        conv_state_out = torch.empty_like(conv_state_in)
    _need(conv_state_out, "conv_state_out", bf, (B, C, K_win), dev)
    q = torch.empty((B * num_v_heads, head_k_dim), dtype=bf, device=dev)
    k = torch.empty_like(q)
    v = torch.empty((B * num_v_heads, head_v_dim), dtype=bf, device=dev)
    _check(load_library().gdn_conv1d_decode(
        _ptr(x), _ptr(conv_weight), _ptr(conv_state_in), _ptr(conv_state_out), _ptr(q),
        _ptr(k), _ptr(v), B, num_k_heads, num_v_heads, head_k_dim, head_v_dim, K_win,
        _stream(stream)))
    return q, k, v, conv_state_out


def gdn_prefill_varlen_workspace_bytes(N, Hk, Hv, T, Dk, Dv, dtype) -> int:
    dt = GDN_DTYPE_BF16 if dtype == torch.bfloat16 else GDN_DTYPE_F32
    n = load_library().gdn_prefill_varlen_workspace_bytes(N, Hk, Hv, T, Dk, Dv, dt)
    if n == ctypes.c_size_t(-1).value:
        raise GDNError(GDN_EINVAL, "invalid shape")
    return n


def gdn_prefill_varlen(q, k, v, g_log, beta, scale, cu_seqlens, state=None, out=None,
                       workspace=None, stream=None):
    """Variable-length prefill: q,k [Hk,T,Dk], v [Hv,T,Dv], g_log, beta [Hv,T], cu_seqlens
    [N+1] int32 on the device (sequence n = tokens cu[n] .. cu[n+1]-1). ``state`` [N,Hv,Dk,Dv]
    fp32 is updated in place when given, else zero-initialised and returned. Returns
    (out [Hv,T,Dv], state)."""
    Hk, T, Dk = q.shape
    Hv, Dv = v.shape[0], v.shape[2]
    N = cu_seqlens.shape[0] - 1
    dev, dt = q.device, q.dtype
    code = GDN_DTYPE_BF16 if dt == torch.bfloat16 else GDN_DTYPE_F32
    _need(k, "k", dt, (Hk, T, Dk), dev)
    _need(v, "v", dt, (Hv, T, Dv), dev)
    _need(g_log, "g_log", torch.float32, (Hv, T), dev)
    _need(beta, "beta", torch.float32, (Hv, T), dev)
    _need(cu_seqlens, "cu_seqlens", torch.int32, (N + 1,), dev)
    state_is_input = state is not None
    if state is None:
        state = torch.empty((N, Hv, Dk, Dv), dtype=torch.float32, device=dev)
    _need(state, "state", torch.float32, (N, Hv, Dk, Dv), dev)
    if out is None:
        out = torch.empty((Hv, T, Dv), dtype=dt, device=dev)
    _need(out, "out", dt, (Hv, T, Dv), dev)
    need = gdn_prefill_varlen_workspace_bytes(N, Hk, Hv, T, Dk, Dv, dt)
    if workspace is None or workspace.numel() * workspace.element_size() < need:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=dev)
    _check(load_library().gdn_prefill_varlen(
        _ptr(q), _ptr(k), _ptr(v), _ptr(g_log), _ptr(beta), float(scale), code,
        _ptr(cu_seqlens), N, Hk, Hv, T, Dk, Dv, _ptr(state), int(state_is_input), _ptr(out),
        _ptr(workspace), workspace.numel() * workspace.element_size(), _stream(stream)))
    return out, state


def gdn_unit_lower_inverse(A, algorithm=GDN_TRIL_SUBSTITUTION, out=None, stream=None):
    """(I + A)^-1 for a batch of strictly lower-triangular 64x64 fp32 matrices A [n,64,64]
    (zero on and above the diagonal). ``algorithm``: GDN_TRIL_SUBSTITUTION or
    GDN_TRIL_NEUMANN. Returns T [n,64,64] fp32."""
    n, C, C2 = A.shape
    if C != C2:
        raise ValueError("A must be [n, C, C]")
    _need(A, "A", torch.float32, (n, C, C), A.device)
    if out is None:
        out = torch.empty_like(A)
    _need(out, "out", torch.float32, (n, C, C), A.device)
    _check(load_library().gdn_unit_lower_inverse(_ptr(A), _ptr(out), n, C, int(algorithm),
                                                 _stream(stream)))
    return out
