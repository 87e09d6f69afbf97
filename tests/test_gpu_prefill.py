"""GPU parity of gdn_prefill against the fp64 oracle, on seeded synthetic inputs.

Shapes and contract: "GDN CTE Kernel API Reference" (parameters, returns, Notes).
Tolerances (relative Frobenius error, whole tensor): fp32 compute dtype 1e-4 on out and
state; bf16 2e-2 on out and 1e-2 on state.
"""
import numpy as np
import pytest
import torch

from gpu_util import (DEV, TOL_BF16, TOL_F32, ensure_built, gpu_prefill, oracle_prefill_all,
                      oracle_prefill_heads, rel, to_np)
import linear_attention_recurrence_03_gb300 as gdn
from linear_attention_recurrence_03_gb300 import synthetic as syn

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


def _full_parity(w, tol, seed=None):
    x = syn.prefill_inputs(w, seed=seed)
    out, st = gpu_prefill(x)
    o_ref, s_ref = oracle_prefill_all(x)
    eo, es = rel(to_np(out), o_ref), rel(to_np(st), s_ref)
    assert eo <= tol["out"], f"out rel err {eo:.3e}"
    assert es <= tol["state"], f"state rel err {es:.3e}"
    return eo, es


def test_prefill_f32_small_workload():
    _full_parity(syn.PREFILL_F32_SMALL, TOL_F32)


@pytest.mark.parametrize("S", [0, 1, 63, 64, 65, 127, 200])
def test_prefill_f32_ragged_lengths(S):
    w = syn.shrink(syn.PREFILL_F32_SMALL, S=S, Hk=1, Hv=2, state_std=0.05)
    if S == 0:
        x = syn.prefill_inputs(w)
        out, st = gpu_prefill(x)
        assert out.shape[2] == 0
        assert torch.equal(st, x["state"])
        return
    _full_parity(w, TOL_F32)


@pytest.mark.parametrize("Dk,Dv", [(16, 16), (37, 100), (128, 128), (128, 64), (64, 128)])
def test_prefill_f32_head_dims(Dk, Dv):
    w = syn.shrink(syn.PREFILL_F32_SMALL, Dk=Dk, Dv=Dv, Hk=2, Hv=4, S=130, state_std=0.05,
                   scale=Dk ** -0.5)
    _full_parity(w, TOL_F32)


def test_prefill_zero_state_writes_state():
    """Omitted state: zero initial state, no load; the output buffer gets the final state
    whatever it held before."""
    w = syn.shrink(syn.PREFILL_F32_SMALL, S=96)
    x = syn.prefill_inputs(w)
    args = [x[n].to(DEV) for n in ("q", "k", "v", "g_log", "beta")]
    garbage = torch.full((1, 2, 64, 64), float("nan"), device=DEV)
    lib = gdn.load_library()
    import ctypes
    vp = ctypes.c_void_p
    out = torch.empty((1, 2, 96, 64), device=DEV)
    rc = lib.gdn_prefill(*(vp(t.data_ptr()) for t in args), x["scale"], gdn.GDN_DTYPE_F32, 1, 2,
                         2, 96, 64, 64, vp(garbage.data_ptr()), 0, vp(out.data_ptr()), None, 0,
                         vp(torch.cuda.current_stream().cuda_stream))
    assert rc == gdn.GDN_OK
    torch.cuda.synchronize()
    o_ref, s_ref = oracle_prefill_all(x)
    assert rel(to_np(garbage), s_ref) <= 1e-4
    assert rel(to_np(out), o_ref) <= 1e-4


def test_prefill_bf16_gqa_workload():
    """B=2, Hk=4, Hv=8, S=1024, D=128, supplied state, all heads compared."""
    _full_parity(syn.PREFILL_BF16_GQA2, TOL_BF16)


@pytest.mark.parametrize("S", [64, 100, 191, 256])
def test_prefill_bf16_small_cases(S):
    w = syn.shrink(syn.PREFILL_BF16_GQA2, B=1, Hk=2, Hv=4, S=S)
    _full_parity(w, TOL_BF16)


def test_prefill_bf16_other_head_dims():
    w = syn.shrink(syn.PREFILL_BF16_GQA2, B=1, Hk=1, Hv=2, S=160, Dk=64, Dv=96, scale=0.125)
    _full_parity(w, TOL_BF16)


def _sampled_parity(w, heads, tol):
    x = syn.prefill_inputs(w)
    out, st = gpu_prefill(x)
    ref = oracle_prefill_heads(x, heads)
    for (b, h), (o_ref, s_ref) in ref.items():
        eo, es = rel(to_np(out[b, h]), o_ref), rel(to_np(st[b, h]), s_ref)
        assert eo <= tol["out"], f"head {(b, h)} out rel err {eo:.3e}"
        assert es <= tol["state"], f"head {(b, h)} state rel err {es:.3e}"
    assert torch.isfinite(out.float()).all() and torch.isfinite(st).all()


def test_prefill_bf16_layer_workload_sampled_heads():
    """B=1, Hk=16, Hv=32, S=8192: the full launch, checked on three heads."""
    _sampled_parity(syn.PREFILL_BF16_LAYER, [(0, 0), (0, 17), (0, 31)], TOL_BF16)


def test_prefill_bf16_batched_workload_sampled_heads():
    """B=8, Hk=16, Hv=32, S=4096, state in place: the full launch, checked on three heads."""
    _sampled_parity(syn.PREFILL_BF16_BATCHED, [(0, 1), (3, 20), (7, 31)], TOL_BF16)


@pytest.mark.parametrize("S,state", [(187, 0.05), (128, None), (64 * 5, 0.05)])
def test_prefill_transposed_carry_full_parity(S, state):
    """B*Hv = 80 value heads: more than two carry CTAs per head fit, so the transposed
    one-CTA-per-head carry runs (state columns in TMEM lanes). Every head against the
    oracle, with a ragged tail, a zero start and a whole number of chunks; and the same
    bits on a second call."""
    w = syn.shrink(syn.PREFILL_BF16_GQA2, B=1, Hk=40, Hv=80, S=S, state_std=state)
    x = syn.prefill_inputs(w)
    out, st = gpu_prefill(x)
    o_ref, s_ref = oracle_prefill_all(x)
    assert rel(to_np(out), o_ref) <= TOL_BF16["out"]
    assert rel(to_np(st), s_ref) <= TOL_BF16["state"]
    o2, s2 = gpu_prefill(x)
    assert torch.equal(out, o2) and torch.equal(st, s2)


@pytest.mark.parametrize("w", [syn.PREFILL_F32_SMALL,
                               syn.shrink(syn.PREFILL_BF16_GQA2, S=256)], ids=["f32", "bf16"])
def test_prefill_is_bitwise_reproducible(w):
    x = syn.prefill_inputs(w)
    o1, s1 = gpu_prefill(x)
    o2, s2 = gpu_prefill(x)
    assert torch.equal(o1, o2) and torch.equal(s1, s2)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_prefill_split_and_carry_is_exact(dtype):
    """Prefill of [0,s) then of [s,S) from the carried state gives, at a chunk boundary,
    bit for bit the result of one prefill over [0,S)."""
    base = syn.PREFILL_F32_SMALL if dtype == "f32" else syn.PREFILL_BF16_GQA2
    w = syn.shrink(base, B=1, Hk=1, Hv=2, S=256, state_std=0.05)
    x = syn.prefill_inputs(w)
    out, st = gpu_prefill(x)
    s = 128
    first = dict(x, **{n: x[n][:, :, :s].contiguous() for n in ("q", "k", "v", "g_log", "beta")})
    second = dict(x, **{n: x[n][:, :, s:].contiguous() for n in ("q", "k", "v", "g_log", "beta")})
    o1, s1 = gpu_prefill(first)
    second["state"] = s1
    o2, s2 = gpu_prefill(second)
    assert torch.equal(torch.cat([o1, o2], dim=2), out)
    assert torch.equal(s2, st)


def test_device_status_clean_after_prefill():
    _full_parity(syn.shrink(syn.PREFILL_BF16_GQA2, B=1, S=128), TOL_BF16)
    assert gdn.gdn_get_device_status() == gdn.GDN_OK


def test_prefill_rejects_mixed_dtypes():
    w = syn.shrink(syn.PREFILL_BF16_GQA2, B=1, S=64)
    x = syn.prefill_inputs(w)
    args = [x[n].to(DEV) for n in ("q", "k", "v", "g_log", "beta")]
    args[2] = args[2].float()
    with pytest.raises(ValueError):
        gdn.gdn_prefill(*args, x["scale"])
    assert np.isfinite(x["scale"])


def test_prefill_noalloc_equals_prefill_one_segment():
    """The static-scratch entry point: same kernels, same result, bit for bit."""
    w = syn.shrink(syn.PREFILL_BF16_GQA2, S=200)
    x = syn.prefill_inputs(w)
    args = [x[n].to(DEV) for n in ("q", "k", "v", "g_log", "beta")]
    st0 = x["state"].to(DEV) if x["state"] is not None else None
    o1, s1 = gdn.gdn_prefill(*args, x["scale"], state=None if st0 is None else st0.clone())
    o2, s2 = gdn.gdn_prefill_noalloc(*args, x["scale"], state=None if st0 is None else st0.clone())
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(s1, s2)


def test_prefill_overlapped_segments_equal_one_pass():
    """Few heads and a long sequence: gdn_prefill runs the sequence as several segments,
    the prep of each beside the carry of the one before (two helper streams). The state
    crosses segments in fp32, so the result equals the one-segment run (the static
    scratch of gdn_prefill_noalloc holds this whole sequence) bit for bit, and matches the
    oracle on sampled heads."""
    w = syn.shrink(syn.PREFILL_BF16_GQA2, B=1, Hk=4, Hv=8, S=64 * 40 - 17, state_std=0.05)
    x = syn.prefill_inputs(w)
    args = [x[n].to(DEV) for n in ("q", "k", "v", "g_log", "beta")]
    st0 = x["state"].to(DEV)
    n0 = gdn.gdn_launch_count()
    o1, s1 = gdn.gdn_prefill(*args, x["scale"], state=st0.clone())
    assert gdn.gdn_launch_count() - n0 > 2  # more than one segment
    o2, s2 = gdn.gdn_prefill_noalloc(*args, x["scale"], state=st0.clone())
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(s1, s2)
    ref = oracle_prefill_heads(x, [(0, 0), (0, 5)])
    for (b, h), (o_ref, s_ref) in ref.items():
        assert rel(to_np(o1[b, h]), o_ref) <= TOL_BF16["out"]
        assert rel(to_np(s1[b, h]), s_ref) <= TOL_BF16["state"]


def test_prefill_noalloc_many_segments():
    """B*Hv = 1024 leaves room for one 64-token chunk per (batch, head) in the static
    scratch, so S = 320 runs as five segments with the state carried between them: the
    result equals gdn_prefill's bit for bit and matches the oracle on sampled heads."""
    w = syn.shrink(syn.PREFILL_BF16_GQA2, B=16, Hk=32, Hv=64, S=320, state_std=0.05)
    x = syn.prefill_inputs(w)
    args = [x[n].to(DEV) for n in ("q", "k", "v", "g_log", "beta")]
    st0 = x["state"].to(DEV)
    o1, s1 = gdn.gdn_prefill(*args, x["scale"], state=st0.clone())
    o2, s2 = gdn.gdn_prefill_noalloc(*args, x["scale"], state=st0.clone())
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(s1, s2)
    ref = oracle_prefill_heads(x, [(0, 0), (7, 33), (15, 63)])
    for (b, h), (o_ref, s_ref) in ref.items():
        assert rel(to_np(o2[b, h]), o_ref) <= TOL_BF16["out"]
        assert rel(to_np(s2[b, h]), s_ref) <= TOL_BF16["state"]
