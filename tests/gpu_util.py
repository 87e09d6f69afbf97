"""Helpers shared by the GPU parity tests: run the CUDA path through the binding and the
fp64 oracle on the same seeded inputs, on all heads or on a sample of them."""
import numpy as np
import torch

import oracle
import linear_attention_recurrence_03_gb300 as gdn
from linear_attention_recurrence_03_gb300 import build as lib_build

DEV = torch.device("cuda:0")
PREFILL_NAMES = ("q", "k", "v", "g_log", "beta")
DECODE_NAMES = ("q", "k", "v", "b", "a", "A_log", "dt_bias", "z", "norm_weight", "state")

# Tolerances (relative Frobenius error over the whole tensor).
TOL_F32 = dict(out=1e-4, state=1e-4)
TOL_BF16 = dict(out=2e-2, state=1e-2)


def ensure_built():
    lib_build.build()
    gdn.load_library()


def rel(x, ref) -> float:
    x = np.asarray(x, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    den = np.linalg.norm(ref.ravel())
    return float(np.linalg.norm((x - ref).ravel()) / (den if den > 0 else 1.0))


def to_np(t) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def gpu_prefill(x, state_in_place=True):
    """Runs gdn_prefill on cuda:0. Returns (out, final state) as CPU tensors."""
    args = [x[n].to(DEV) for n in PREFILL_NAMES]
    st = x["state"].to(DEV) if x["state"] is not None else None
    out, st = gdn.gdn_prefill(*args, x["scale"], state=st)
    torch.cuda.synchronize()
    return out.cpu(), st.cpu()


def oracle_prefill_heads(x, heads):
    """Oracle on selected (b, h) value heads only (each head is independent).
    Returns dicts {(b,h): (out [S,Dv], state [Dk,Dv])}."""
    B, Hk = x["q"].shape[:2]
    Hv = x["v"].shape[1]
    G = Hv // Hk
    res = {}
    for b, h in heads:
        sl = lambda t: t[b:b + 1, h:h + 1]  # noqa: E731
        s0 = None if x["state"] is None else sl(x["state"])
        o, s = oracle.prefill(x["q"][b:b + 1, h // G:h // G + 1], x["k"][b:b + 1, h // G:h // G + 1],
                              sl(x["v"]), sl(x["g_log"]), sl(x["beta"]), x["scale"], s0)
        res[(b, h)] = (o[0, 0], s[0, 0])
    return res


def oracle_prefill_all(x):
    s0 = x["state"]
    return oracle.prefill(*(x[n] for n in PREFILL_NAMES), x["scale"], s0)


def gpu_decode(x, in_place=False):
    args = [x[n].to(DEV) for n in DECODE_NAMES]
    st_out = args[-1] if in_place else None
    out, st = gdn.gdn_decode_step(*args, x["num_v_heads"], state_out=st_out)
    torch.cuda.synchronize()
    return out.cpu(), st.cpu()
