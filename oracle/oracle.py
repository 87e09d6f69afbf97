"""ctypes front end of the fp64 C oracle in ``gdn_oracle.c``.

TEST INFRASTRUCTURE: the tests, the smoke check and the benchmark's CPU baseline are
the only callers. Arguments are converted to contiguous float64 numpy arrays (bf16 and
fp32 convert to float64 exactly), so the oracle sees the very values a GPU run sees.

Sources: "GDN CTE Kernel API Reference" (prefill) and "GDN TKG Kernel API
Reference" (decode step), AWS Neuron NKI library. See ``gdn_oracle.c`` for the
recurrence, the derived chunk algebra and which readings are unpinned.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gdn_oracle.c")
_LIB_PATH = os.path.join(_HERE, "libgdn_oracle.so")
_lock = threading.Lock()
_lib = None

# Readings of constants the pages leave unstated (l2norm and RMSNorm eps).
EPS_L2 = 1e-6
EPS_RMS = 1e-6

_dp = ctypes.POINTER(ctypes.c_double)


def build(force: bool = False) -> str:
    """Compile ``gdn_oracle.c`` into ``libgdn_oracle.so`` with gcc (plain C11, -O2,
    no fast-math so IEEE fp64 semantics hold). Returns the library path."""
    stale = (not os.path.exists(_LIB_PATH)) or (
        os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC))
    if force or stale:
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
                        _SRC, "-o", tmp, "-lm"], check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _bind(path):
    lib = ctypes.CDLL(path)
    i, d = ctypes.c_int, ctypes.c_double
    lib.gdn_oracle_prefill.argtypes = [_dp] * 5 + [d] + [i] * 6 + [_dp, _dp, _dp, i]
    lib.gdn_oracle_prefill.restype = i
    lib.gdn_oracle_prefill_chunked.argtypes = [_dp] * 5 + [d] + [i] * 7 + [_dp, _dp, _dp, i]
    lib.gdn_oracle_prefill_chunked.restype = i
    lib.gdn_oracle_unit_lower_inverse.argtypes = [_dp, i, _dp]
    lib.gdn_oracle_unit_lower_inverse.restype = None
    lib.gdn_oracle_decode_step.argtypes = [_dp] * 10 + [i] * 4 + [d, d] + [_dp, _dp, i]
    lib.gdn_oracle_decode_step.restype = i
    lib.gdn_oracle_conv1d_decode.argtypes = [_dp] * 3 + [i] * 3 + [_dp, _dp]
    lib.gdn_oracle_conv1d_decode.restype = i
    return lib


def _f64(x) -> np.ndarray:
    """Any array-like (numpy, torch CPU tensor of any float dtype) -> C-contiguous f64."""
    if hasattr(x, "detach"):  # torch tensor: go through float64 on the CPU
        x = x.detach().to("cpu").double().numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(a: np.ndarray | None):
    return None if a is None else a.ctypes.data_as(_dp)


def _threads(n):
    return int(n) if n else max(1, os.cpu_count() or 1)


class Oracle:
    """The oracle's entry points bound to one compiled copy of ``gdn_oracle.c``."""

    def __init__(self, lib_path: str):
        self.lib = _bind(lib_path)

    def prefill(self, q, k, v, g_log, beta, scale, state0=None, nthreads=None):
        """Token-by-token recurrence. q,k [B,Hk,S,Dk]; v [B,Hv,S,Dv]; g_log, beta
        [B,Hv,S]; state0 [B,Hv,Dk,Dv] or None (zero). Returns (out [B,Hv,S,Dv],
        state [B,Hv,Dk,Dv])."""
        q, k, v, g, b = map(_f64, (q, k, v, g_log, beta))
        s0 = None if state0 is None else _f64(state0)
        B, Hk, S, Dk = q.shape
        Hv, Dv = v.shape[1], v.shape[3]
        out = np.empty((B, Hv, S, Dv))
        st = np.empty((B, Hv, Dk, Dv))
        rc = self.lib.gdn_oracle_prefill(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(b),
                                         float(scale), B, Hk, Hv, S, Dk, Dv, _ptr(s0),
                                         _ptr(out), _ptr(st), _threads(nthreads))
        if rc != 0:
            raise ValueError("oracle prefill: bad shapes")
        return out, st

    def prefill_chunked(self, q, k, v, g_log, beta, scale, chunk, state0=None,
                        nthreads=None):
        """Chunk-parallel (WY) form with chunk length ``chunk``; contract as prefill."""
        q, k, v, g, b = map(_f64, (q, k, v, g_log, beta))
        s0 = None if state0 is None else _f64(state0)
        B, Hk, S, Dk = q.shape
        Hv, Dv = v.shape[1], v.shape[3]
        out = np.empty((B, Hv, S, Dv))
        st = np.empty((B, Hv, Dk, Dv))
        rc = self.lib.gdn_oracle_prefill_chunked(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(b),
                                                 float(scale), B, Hk, Hv, S, Dk, Dv,
                                                 int(chunk), _ptr(s0), _ptr(out), _ptr(st),
                                                 _threads(nthreads))
        if rc != 0:
            raise ValueError("oracle prefill_chunked: bad shapes")
        return out, st

    def prefill_varlen(self, q, k, v, g_log, beta, scale, cu_seqlens, state0=None,
                       nthreads=None):
        """Variable-length batch: sequence n = tokens cu[n] .. cu[n+1]-1 of q,k [Hk,T,Dk],
        v [Hv,T,Dv], g_log, beta [Hv,T], each run through ``prefill`` from its own state
        (state0 [N,Hv,Dk,Dv] or None = zeros). Returns (out [Hv,T,Dv] -- zero past cu[N] --,
        state [N,Hv,Dk,Dv])."""
        q, k, v, g, b = map(_f64, (q, k, v, g_log, beta))
        cu = [int(x) for x in np.asarray(cu_seqlens).reshape(-1)]
        N = len(cu) - 1
        Hk, T, Dk = q.shape
        Hv, Dv = v.shape[0], v.shape[2]
        out = np.zeros((Hv, T, Dv))
        st = np.zeros((N, Hv, Dk, Dv)) if state0 is None else _f64(state0).copy()
        for n in range(N):
            t0, t1 = cu[n], cu[n + 1]
            if t1 <= t0:
                continue
            o, s1 = self.prefill(q[None, :, t0:t1], k[None, :, t0:t1], v[None, :, t0:t1],
                                 g[None, :, t0:t1], b[None, :, t0:t1], scale,
                                 st[n][None], nthreads)
            out[:, t0:t1] = o[0]
            st[n] = s1[0]
        return out, st

    def unit_lower_inverse(self, A):
        """(I + A)^-1 for strictly lower-triangular square A (forward substitution)."""
        A = _f64(A)
        n = A.shape[0]
        T = np.empty((n, n))
        self.lib.gdn_oracle_unit_lower_inverse(_ptr(A), n, _ptr(T))
        return T

    def decode_step(self, q, k, v, b, a, A_log, dt_bias, z, norm_weight, state_in,
                    num_v_heads, eps_l2=EPS_L2, eps_rms=EPS_RMS, nthreads=None):
        """Fused decode step. q,k [BH,K] raw; v,z [BH,V]; b,a [BH]; A_log, dt_bias [H];
        norm_weight [V]; state_in [BH,K,V]. Returns (out [BH,V] in fp64 -- the GPU
        rounds it to bf16 --, state_out [BH,K,V])."""
        q, k, v, b, a, Al, dtb, z, w, s0 = map(
            _f64, (q, k, v, b, a, A_log, dt_bias, z, norm_weight, state_in))
        BH, K = q.shape
        V = v.shape[1]
        out = np.empty((BH, V))
        st = np.empty((BH, K, V))
        rc = self.lib.gdn_oracle_decode_step(_ptr(q), _ptr(k), _ptr(v), _ptr(b), _ptr(a),
                                             _ptr(Al), _ptr(dtb), _ptr(z), _ptr(w), _ptr(s0),
                                             BH, int(num_v_heads), K, V, float(eps_l2),
                                             float(eps_rms), _ptr(out), _ptr(st),
                                             _threads(nthreads))
        if rc != 0:
            raise ValueError("oracle decode_step: bad shapes")
        return out, st


    def decode_multi(self, q, k, v, b, a, A_log, dt_bias, z, norm_weight, state_in,
                     num_v_heads, eps_l2=EPS_L2, eps_rms=EPS_RMS, nthreads=None):
        """T consecutive decode tokens: token t is decode_step applied to the state token
        t-1 left (the multi-token extension is defined as exactly that). q,k [T,BH,K];
        v,z [T,BH,V]; b,a [T,BH]; the rest as decode_step. Returns (out [T,BH,V] fp64,
        state_out [BH,K,V])."""
        q, k, v, b, a, z = map(_f64, (q, k, v, b, a, z))
        T = q.shape[0]
        st = _f64(state_in)
        outs = []
        for t in range(T):
            o, st = self.decode_step(q[t], k[t], v[t], b[t], a[t], A_log, dt_bias, z[t],
                                     norm_weight, st, num_v_heads, eps_l2, eps_rms, nthreads)
            outs.append(o)
        out = np.stack(outs) if outs else np.empty((0,) + v.shape[1:])
        return out, st


    def conv1d_decode(self, x, weight, state_in):
        """One token through the depthwise causal conv: x [B, C], weight [C, K_win],
        state_in [B, C, K_win] (oldest first). Returns (y = silu(conv) [B, C],
        state_out [B, C, K_win])."""
        x, w, s0 = map(_f64, (x, weight, state_in))
        B, C, K_win = s0.shape
        y = np.empty((B, C))
        st = np.empty((B, C, K_win))
        rc = self.lib.gdn_oracle_conv1d_decode(_ptr(x), _ptr(w), _ptr(s0), B, C, K_win,
                                               _ptr(y), _ptr(st))
        if rc != 0:
            raise ValueError("oracle conv1d_decode: bad shapes")
        return y, st

    def conv1d_split(self, y, num_k_heads, num_v_heads, head_k_dim, head_v_dim):
        """Split the conv output [B, conv_dim] into q | k | v and repeat q, k over the
        value heads (value head h reads key head h // (num_v_heads // num_k_heads)).
        Returns q, k [B * num_v_heads, head_k_dim] and v [B * num_v_heads, head_v_dim]."""
        y = _f64(y)
        B = y.shape[0]
        kd = num_k_heads * head_k_dim
        G = num_v_heads // num_k_heads
        q = y[:, :kd].reshape(B, num_k_heads, head_k_dim)
        k = y[:, kd:2 * kd].reshape(B, num_k_heads, head_k_dim)
        v = y[:, 2 * kd:].reshape(B * num_v_heads, head_v_dim)
        idx = np.arange(num_v_heads) // G
        return (q[:, idx].reshape(B * num_v_heads, head_k_dim),
                k[:, idx].reshape(B * num_v_heads, head_k_dim), v)


def default() -> Oracle:
    """The oracle built from ``gdn_oracle.c`` (compiled on first use)."""
    global _lib
    with _lock:
        if _lib is None:
            _lib = Oracle(build())
    return _lib


def prefill(*args, **kw):
    return default().prefill(*args, **kw)


def prefill_chunked(*args, **kw):
    return default().prefill_chunked(*args, **kw)


def unit_lower_inverse(A):
    return default().unit_lower_inverse(A)


def prefill_varlen(*args, **kw):
    return default().prefill_varlen(*args, **kw)


def decode_step(*args, **kw):
    return default().decode_step(*args, **kw)


def decode_multi(*args, **kw):
    return default().decode_multi(*args, **kw)


def conv1d_decode(*args, **kw):
    return default().conv1d_decode(*args, **kw)


def conv1d_split(*args, **kw):
    return default().conv1d_split(*args, **kw)
