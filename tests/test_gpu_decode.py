"""GPU parity of gdn_decode_step against the fp64 oracle ("GDN TKG Kernel API
Reference"). Tolerances: bf16 out 2e-2, fp32 state 1e-2 (relative Frobenius)."""
import pytest
import torch

from gpu_util import TOL_BF16, ensure_built, gpu_decode, rel, to_np
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


def test_decode_full_workload():
    """BH = 8192 (B=256, 32 value heads), K = V = 128, state updated in place: every row
    against the oracle (whole out and state), the worst head group reported beside it."""
    x = syn.decode_inputs(syn.DECODE_BH8192)
    y, st = gpu_decode(x, in_place=True)
    assert torch.isfinite(y.float()).all() and torch.isfinite(st).all()
    y_ref, s_ref = oracle.decode_step(*(x[n] for n in DECODE_NAMES), x["num_v_heads"])
    yn, sn = to_np(y), to_np(st)
    ey, es = rel(yn, y_ref), rel(sn, s_ref)
    H = x["num_v_heads"]
    worst = max(rel(sn[h::H], s_ref[h::H]) for h in range(H))
    print(f"decode BH=8192: out {ey:.3e}, state {es:.3e} (worst head {worst:.3e})")
    assert ey <= TOL_BF16["out"], f"out rel err {ey:.3e}"
    assert es <= TOL_BF16["state"], f"state rel err {es:.3e}"


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


# ---------------------------------------------------------------- multi-token decode
MULTI_NAMES = ("q", "k", "v", "b", "a", "A_log", "dt_bias", "z", "norm_weight", "state")


def _gpu_multi(x, in_place=False):
    args = [x[n].to("cuda") for n in MULTI_NAMES]
    out, st = gdn.gdn_decode_multi(*args, x["num_v_heads"],
                                   state_out=args[-1] if in_place else None)
    torch.cuda.synchronize()
    return out.cpu(), st.cpu()


@pytest.mark.parametrize("K,V,T", [(128, 128, 6), (64, 96, 3), (8, 8, 9), (128, 128, 2),
                                   (100, 128, 5), (128, 128, 16), (128, 32, 8)])
def test_decode_multi_matches_oracle(K, V, T):
    """T tokens in one call against T chained oracle steps (out per token, final state):
    the token loop (T <= 4) and the chunk form (blocks of eight, the last one padded)."""
    w = syn.DecodeWorkload("t", B=3, num_k_heads=2, num_v_heads=4, K=K, V=V)
    x = syn.decode_multi_inputs(w, T)
    y, st = _gpu_multi(x)
    y_ref, s_ref = oracle.decode_multi(*(x[n] for n in MULTI_NAMES), x["num_v_heads"])
    for t in range(T):
        assert rel(to_np(y[t]), y_ref[t]) <= TOL_BF16["out"], f"token {t}"
    assert rel(to_np(st), s_ref) <= TOL_BF16["state"]


@pytest.mark.parametrize("K,V,T", [(64, 96, 11), (128, 128, 9), (100, 128, 10), (8, 16, 3)])
def test_decode_multi_many_rows(K, V, T):
    """400 rows, more than two per SM: a CTA takes several rows in turn, with the next
    row's state and the next block's inputs copied in while it computes (K, V multiples
    of 8; K = 100 takes the one-row-per-CTA form). Two blocks of tokens where T > 8. Every
    row and token against the chained oracle; in place equals out of place bit for bit."""
    w = syn.DecodeWorkload("t", B=100, num_k_heads=2, num_v_heads=4, K=K, V=V)
    x = syn.decode_multi_inputs(w, T)
    y1, s1 = _gpu_multi(x)
    y2, s2 = _gpu_multi(x, in_place=True)
    assert torch.equal(y1, y2) and torch.equal(s1, s2)
    y_ref, s_ref = oracle.decode_multi(*(x[n] for n in MULTI_NAMES), x["num_v_heads"])
    for t in range(T):
        assert rel(to_np(y1[t]), y_ref[t]) <= TOL_BF16["out"], f"token {t}"
    assert rel(to_np(s1), s_ref) <= TOL_BF16["state"]


def test_decode_multi_one_token_is_the_step():
    """T = 1 is gdn_decode_step bit for bit; T = 0 leaves everything untouched."""
    w = syn.DecodeWorkload("t", B=4, num_k_heads=2, num_v_heads=8, K=128, V=128)
    x = syn.decode_multi_inputs(w, 1)
    y, st = _gpu_multi(x)
    one = {n: (x[n][0] if n in ("q", "k", "v", "b", "a", "z") else x[n]) for n in MULTI_NAMES}
    one["num_v_heads"] = x["num_v_heads"]
    y1, s1 = gpu_decode(one)
    assert torch.equal(y[0], y1) and torch.equal(st, s1)
    x0 = syn.decode_multi_inputs(w, 0)
    args = [x0[n].to("cuda") for n in MULTI_NAMES]
    state = args[-1].clone()
    q0 = torch.empty((0, w.BH, w.K), dtype=torch.bfloat16, device="cuda")
    v0 = torch.empty((0, w.BH, w.V), dtype=torch.bfloat16, device="cuda")
    r0 = torch.empty((0, w.BH), dtype=torch.bfloat16, device="cuda")
    out, st0 = gdn.gdn_decode_multi(q0, q0, v0, r0, r0, args[5], args[6], v0, args[8], state,
                                    x0["num_v_heads"], state_out=state)
    torch.cuda.synchronize()
    assert out.shape == (0, w.BH, w.V) and torch.equal(st0, args[-1])


@pytest.mark.parametrize("T", [4, 8])
def test_decode_multi_in_place_and_full_rows(T):
    """BH = 8192 (the decode workload's rows), state updated in place: every row against
    the chained oracle (whole out and state), finite everywhere, and equal to the
    out-of-place call."""
    x = syn.decode_multi_inputs(syn.DECODE_BH8192, T)
    y1, s1 = _gpu_multi(x, in_place=False)
    y2, s2 = _gpu_multi(x, in_place=True)
    assert torch.equal(y1, y2) and torch.equal(s1, s2)
    assert torch.isfinite(y1.float()).all() and torch.isfinite(s1).all()
    y_ref, s_ref = oracle.decode_multi(*(x[n] for n in MULTI_NAMES), x["num_v_heads"])
    assert rel(to_np(y1), y_ref) <= TOL_BF16["out"]
    assert rel(to_np(s1), s_ref) <= TOL_BF16["state"]
