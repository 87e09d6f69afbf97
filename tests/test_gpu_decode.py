"""GPU parity of gdn_decode_step against the fp64 oracle ("GDN TKG Kernel API
Reference"). Tolerances: bf16 out 2e-2, fp32 state 1e-2 (relative Frobenius)."""
import numpy as np
import pytest
import torch

from gpu_util import (TOL_BF16, ensure_built, gpu_decode, oracle_decode_rows, rel, to_np)
import oracle
import linear_attention_recurrence_03_gb300 as gdn
from linear_attention_recurrence_03_gb300 import synthetic as syn
from gpu_util import DECODE_NAMES

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


def _all_rows(w, tol=TOL_BF16, in_place=False):
    x = syn.decode_inputs(w)
    y, st = gpu_decode(x, in_place=in_place)
    y_ref, s_ref = oracle.decode_step(*(x[n] for n in DECODE_NAMES), x["num_v_heads"])
    ey, es = rel(to_np(y), y_ref), rel(to_np(st), s_ref)
    assert ey <= tol["out"], f"out rel err {ey:.3e}"
    assert es <= tol["state"], f"state rel err {es:.3e}"
    return x, y, st


@pytest.mark.parametrize("K,V", [(128, 128), (64, 96), (100, 128), (128, 32), (8, 8)])
def test_decode_small(K, V):
    w = syn.DecodeWorkload("t", B=3, num_k_heads=2, num_v_heads=4, K=K, V=V)
    _all_rows(w)


def test_decode_in_place_matches_out_of_place():
    w = syn.DecodeWorkload("t", B=8, num_k_heads=4, num_v_heads=8, K=128, V=128)
    x = syn.decode_inputs(w)
    y1, s1 = gpu_decode(x, in_place=False)
    y2, s2 = gpu_decode(x, in_place=True)
    assert torch.equal(y1, y2) and torch.equal(s1, s2)


def test_decode_full_workload_sampled_rows():
    """BH = 8192 (B=256, 32 value heads), K = V = 128: the full launch, checked on 96
    sampled rows, and finite everywhere."""
    x = syn.decode_inputs(syn.DECODE_BH8192)
    y, st = gpu_decode(x, in_place=True)
    rng = np.random.default_rng(0)
    rows = np.sort(rng.choice(x["q"].shape[0], size=96, replace=False))
    rows[0], rows[-1] = 0, x["q"].shape[0] - 1
    y_ref, s_ref = oracle_decode_rows(x, rows)
    ey, es = rel(to_np(y[rows]), y_ref), rel(to_np(st[rows]), s_ref)
    assert ey <= TOL_BF16["out"], f"out rel err {ey:.3e}"
    assert es <= TOL_BF16["state"], f"state rel err {es:.3e}"
    assert torch.isfinite(y.float()).all() and torch.isfinite(st).all()


def test_decode_is_bitwise_reproducible():
    w = syn.DecodeWorkload("t", B=16, num_k_heads=16, num_v_heads=32, K=128, V=128)
    x = syn.decode_inputs(w)
    a = gpu_decode(x)
    b = gpu_decode(x)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


def test_decode_rows_are_independent():
    """Per-head independent recurrence (Notes): changing one row's inputs changes only
    that row's outputs."""
    w = syn.DecodeWorkload("t", B=4, num_k_heads=2, num_v_heads=4, K=128, V=128)
    x = syn.decode_inputs(w)
    y1, s1 = gpu_decode(x)
    x2 = dict(x, v=x["v"].clone())
    x2["v"][5] += 1.0
    y2, s2 = gpu_decode(x2)
    keep = [r for r in range(16) if r != 5]
    assert torch.equal(y1[keep], y2[keep]) and torch.equal(s1[keep], s2[keep])
    assert not torch.equal(s1[5], s2[5])


def test_decode_empty_batch():
    w = syn.DecodeWorkload("t", B=0, num_k_heads=2, num_v_heads=4, K=128, V=128)
    x = syn.decode_inputs(w)
    y, st = gpu_decode(x)
    assert y.shape == (0, 128) and st.shape == (0, 128, 128)
    assert gdn.gdn_get_device_status() == gdn.GDN_OK
