"""GPU parity of gdn_conv1d_decode (the conv1d decode token in front of the decode step,
"GDN Block TKG Kernel API Reference") against the fp64 oracle. The window shift is exact
(bf16 values moved); q, k, v = bf16(silu(conv)) are held to 1e-2 relative Frobenius
error (bf16 rounding of fp32 sums of K_win products)."""
import numpy as np
import pytest
import torch

from gpu_util import (DEV, TOL_BF16, ensure_built, rel, to_np)
import oracle
import linear_attention_recurrence_03_gb300 as gdn
from linear_attention_recurrence_03_gb300 import synthetic as syn

pytestmark = pytest.mark.gpu
TOL_CONV = 1e-2


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


def _run(w, x, in_place=False):
    xd, wd, sd = (x[n].to(DEV) for n in ("x", "conv_weight", "conv_state"))
    q, k, v, so = gdn.gdn_conv1d_decode(xd, wd, sd, w.num_k_heads, w.num_v_heads, w.head_k_dim,
                                        w.head_v_dim, conv_state_out=sd if in_place else None)
    torch.cuda.synchronize()
    return q.cpu(), k.cpu(), v.cpu(), so.cpu()


def _ref(w, x):
    y, st = oracle.conv1d_decode(x["x"], x["conv_weight"], x["conv_state"])
    q, k, v = oracle.conv1d_split(y, w.num_k_heads, w.num_v_heads, w.head_k_dim, w.head_v_dim)
    return q, k, v, st


@pytest.mark.parametrize("B,Hk,Hv,Dk,Dv,K", [(3, 2, 4, 16, 24, 4), (2, 2, 4, 6, 10, 4),
                                            (2, 1, 3, 128, 64, 3),
                                            (1, 4, 4, 8, 8, 1), (5, 2, 2, 32, 128, 16)])
def test_conv1d_matches_oracle(B, Hk, Hv, Dk, Dv, K):
    w = syn.Conv1dWorkload("t", B, Hk, Hv, Dk, Dv, K_win=K)
    x = syn.conv1d_inputs(w)
    q, k, v, so = _run(w, x)
    qr, kr, vr, sr = _ref(w, x)
    assert rel(to_np(q), qr) <= TOL_CONV and rel(to_np(k), kr) <= TOL_CONV
    assert rel(to_np(v), vr) <= TOL_CONV
    np.testing.assert_array_equal(to_np(so), sr)  # the shift is exact


def test_conv1d_in_place_and_full_size():
    """B = 256 tokens of a Qwen3.5-style layer's q|k|v channels (8192 channels, K_win = 4),
    window updated in place: every output against the oracle, equal to out-of-place."""
    w = syn.CONV1D_B256
    x = syn.conv1d_inputs(w)
    a = _run(w, x, in_place=False)
    b = _run(w, x, in_place=True)
    for t1, t2 in zip(a, b):
        assert torch.equal(t1, t2)
    qr, kr, vr, sr = _ref(w, x)
    assert rel(to_np(a[0]), qr) <= TOL_CONV and rel(to_np(a[1]), kr) <= TOL_CONV
    assert rel(to_np(a[2]), vr) <= TOL_CONV
    np.testing.assert_array_equal(to_np(a[3]), sr)


def test_conv1d_feeds_the_decode_step():
    """conv1d decode token -> decode step on the GPU, against the same two steps of the
    oracle (q, k, v from the oracle's conv, rounded to bf16 as the GPU hands them on)."""
    w = syn.Conv1dWorkload("t", B=4, num_k_heads=2, num_v_heads=4, head_k_dim=128,
                           head_v_dim=128)
    x = syn.conv1d_inputs(w)
    wd = syn.DecodeWorkload("t", B=4, num_k_heads=2, num_v_heads=4, K=128, V=128)
    d = syn.decode_inputs(wd, seed=3)
    q, k, v, _ = _run(w, x)
    args = [q, k, v] + [d[n] for n in ("b", "a", "A_log", "dt_bias", "z", "norm_weight",
                                       "state")]
    y, st = gdn.gdn_decode_step(*(t.to(DEV) for t in args), wd.num_v_heads)
    qr, kr, vr, _ = _ref(w, x)
    bf = lambda t: torch.from_numpy(t).to(torch.bfloat16)
    y_ref, s_ref = oracle.decode_step(bf(qr), bf(kr), bf(vr), d["b"], d["a"], d["A_log"],
                                      d["dt_bias"], d["z"], d["norm_weight"], d["state"],
                                      wd.num_v_heads)
    assert rel(to_np(y.cpu()), y_ref) <= TOL_BF16["out"]
    assert rel(to_np(st.cpu()), s_ref) <= TOL_BF16["state"]
