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


def _whole_parity(w, tol):
    """Every head of the full launch against the oracle: relative Frobenius error of the
    whole out and state tensors, and the worst single head reported beside it."""
    x = syn.prefill_inputs(w)
    out, st = gpu_prefill(x)
    assert torch.isfinite(out.float()).all() and torch.isfinite(st).all()
    o_ref, s_ref = oracle_prefill_all(x)
    o, s = to_np(out), to_np(st)
    eo, es = rel(o, o_ref), rel(s, s_ref)
    B, Hv = o.shape[:2]
    worst_o = max(rel(o[b, h], o_ref[b, h]) for b in range(B) for h in range(Hv))
    worst_s = max(rel(s[b, h], s_ref[b, h]) for b in range(B) for h in range(Hv))
    print(f"{w.name}: out {eo:.3e} (worst head {worst_o:.3e}), "
          f"state {es:.3e} (worst head {worst_s:.3e})")
    assert eo <= tol["out"], f"out rel err {eo:.3e}"
    assert es <= tol["state"], f"state rel err {es:.3e}"


def test_prefill_bf16_layer_workload():
    """B=1, Hk=16, Hv=32, S=8192, zero start: all 32 heads, whole out and state."""
    _whole_parity(syn.PREFILL_BF16_LAYER, TOL_BF16)


def test_prefill_bf16_batched_workload():
    """B=8, Hk=16, Hv=32, S=4096, state updated in place: all 256 heads, whole out and
    state."""
    _whole_parity(syn.PREFILL_BF16_BATCHED, TOL_BF16)


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


def test_prefill_overlapped_segments_equal_one_pass():
    """Few heads and a long sequence: gdn_prefill runs the sequence as several segments,
    the prep of each beside the carry of the one before (two helper streams). The state
    crosses segments in fp32, so the result equals the one-segment run (the static
    scratch of gdn_prefill_noalloc holds this whole sequence) bit for bit, and matches the
    oracle on sampled heads."""
    w = syn.shrink(syn.PREFILL_BF16_GQA2, B=1, Hk=4, Hv=8, S=64 * 56 - 17, state_std=0.05)
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


# ---------------------------------------------------------------- edge cases of the method
# Through the tensor-core path (bf16, Dk = Dv = 128), with a ragged last chunk, for both
# state-carry forms: 2 value heads (two 64-column CTAs per head) and 80 (one CTA per
# head). Each case runs against the oracle at the bf16 tolerances and against its closed
# form ("GDN CTE Kernel API Reference": returns, :param recurrent_state:).
EDGE_SHAPES = {"two_slice": dict(B=1, Hk=1, Hv=2), "transposed": dict(B=1, Hk=40, Hv=80)}


def _edge_inputs(shape, S, g, beta, state_std=0.05, q_is_k=False, scale=None):
    w = syn.shrink(syn.PREFILL_BF16_GQA2, S=S, state_std=state_std, **EDGE_SHAPES[shape])
    if scale is not None:
        w = syn.shrink(w, scale=scale)
    x = syn.prefill_inputs(w, seed=11)
    gen = torch.Generator().manual_seed(12)
    shp = x["g_log"].shape
    x["g_log"] = g if torch.is_tensor(g) else torch.full(shp, float(g))
    if callable(beta):
        x["beta"] = beta(shp, gen)
    else:
        x["beta"] = torch.full(shp, float(beta))
    if q_is_k:
        x["q"] = x["k"].clone()
    return x


def _edge_parity(x):
    out, st = gpu_prefill(x)
    assert torch.isfinite(out.float()).all() and torch.isfinite(st).all()
    o_ref, s_ref = oracle_prefill_all(x)
    eo, es = rel(to_np(out), o_ref), rel(to_np(st), s_ref)
    assert eo <= TOL_BF16["out"], f"out rel err {eo:.3e}"
    assert es <= TOL_BF16["state"], f"state rel err {es:.3e}"
    return out, st, o_ref, s_ref


@pytest.mark.parametrize("shape", list(EDGE_SHAPES))
def test_edge_identity_beta0_g0(shape):
    """beta = 0 and g = 0: the state passes through unchanged and out = scale q S0."""
    x = _edge_inputs(shape, 250, 0.0, 0.0)
    out, st, _, _ = _edge_parity(x)
    assert torch.equal(st, x["state"])
    G = x["v"].shape[1] // x["q"].shape[1]
    qe = x["q"].double().repeat_interleave(G, dim=1)
    closed = x["scale"] * torch.einsum("bhsk,bhkv->bhsv", qe, x["state"].double())
    assert rel(to_np(out), closed.numpy()) <= TOL_BF16["out"]


@pytest.mark.parametrize("shape", list(EDGE_SHAPES))
def test_edge_exact_write_read(shape):
    """g = 0, beta = 1, q = k (unit rows), zero start, scale 1: each token reads back the
    value it just wrote, out = v (up to the bf16 rounding of the unit keys)."""
    x = _edge_inputs(shape, 200, 0.0, 1.0, state_std=None, q_is_k=True, scale=1.0)
    out, _, _, _ = _edge_parity(x)
    assert rel(to_np(out), to_np(x["v"])) <= TOL_BF16["out"]


@pytest.mark.parametrize("shape", list(EDGE_SHAPES))
def test_edge_fast_decay_underflows_within_a_chunk(shape):
    """g ~ U(-6, -3): exp(gamma) of a 64-token chunk falls far below the fp32 range
    within the chunk; the decay factors must be formed without ratios of it."""
    gen = torch.Generator().manual_seed(3)
    w_shape = syn.shrink(syn.PREFILL_BF16_GQA2, S=211, **EDGE_SHAPES[shape])
    g = torch.rand((w_shape.B, w_shape.Hv, w_shape.S), generator=gen) * 3.0 - 6.0
    x = _edge_inputs(shape, 211, g, lambda shp, gn: torch.rand(shp, generator=gn) * 0.9 + 0.05)
    _edge_parity(x)


@pytest.mark.parametrize("shape", list(EDGE_SHAPES))
def test_edge_reset(shape):
    """g <= -50 on every token: the history is forgotten at each step, S_t = beta_t k_t v_t^T
    and o_t = scale beta_t (k_t . q_t) v_t."""
    gen = torch.Generator().manual_seed(4)
    w_shape = syn.shrink(syn.PREFILL_BF16_GQA2, S=193, **EDGE_SHAPES[shape])
    g = -50.0 - torch.rand((w_shape.B, w_shape.Hv, w_shape.S), generator=gen) * 30.0
    x = _edge_inputs(shape, 193, g, lambda shp, gn: torch.rand(shp, generator=gn) * 0.9 + 0.05)
    out, st, _, _ = _edge_parity(x)
    G = x["v"].shape[1] // x["q"].shape[1]
    q = x["q"].double().repeat_interleave(G, dim=1)
    k = x["k"].double().repeat_interleave(G, dim=1)
    v, b = x["v"].double(), x["beta"].double()
    closed_o = x["scale"] * (b * (k * q).sum(-1))[..., None] * v
    closed_s = b[:, :, -1, None, None] * k[:, :, -1, :, None] * v[:, :, -1, None, :]
    assert rel(to_np(out), closed_o.numpy()) <= TOL_BF16["out"]
    assert rel(to_np(st), closed_s.numpy()) <= TOL_BF16["state"]
