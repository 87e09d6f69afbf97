"""GPU parity of gdn_prefill_varlen (sequences packed along the token axis by cu_seqlens)
against the fp64 oracle, run per sequence; and bit-for-bit against gdn_prefill on each
sequence alone (the chunks of a packed sequence start at its first token, as they do in
a call of its own). Tolerances as gdn_prefill: bf16 out 2e-2 / state 1e-2, fp32 1e-4."""
import numpy as np
import pytest
import torch

from gpu_util import DEV, TOL_BF16, TOL_F32, ensure_built, rel, to_np
import oracle
import linear_attention_recurrence_03_gb300 as gdn
from linear_attention_recurrence_03_gb300 import synthetic as syn

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


def _packed(base, lengths, Hk, Hv, D, seed=0, state=True):
    """Dense inputs of one batch row holding sum(lengths) tokens (the workload's
    distributions), the offsets and one state per sequence."""
    T = int(sum(lengths))
    w = syn.shrink(base, B=1, Hk=Hk, Hv=Hv, S=max(T, 1), Dk=D, Dv=D, state_std=None,
                   seed=seed)
    x = syn.prefill_inputs(w)
    x = {n: (t[0, :, :T] if n in ("q", "k", "v", "g_log", "beta") else t) for n, t in x.items()}
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    gen = torch.Generator().manual_seed(seed + 1)
    st = (torch.randn((len(lengths), Hv, D, D), generator=gen) * 0.05) if state else None
    return x, cu, st


def _gpu(x, cu, st):
    args = [x[n].to(DEV) for n in ("q", "k", "v", "g_log", "beta")]
    out, s = gdn.gdn_prefill_varlen(*args, x["scale"], torch.from_numpy(cu).to(DEV),
                                    state=None if st is None else st.to(DEV))
    torch.cuda.synchronize()
    assert gdn.gdn_get_device_status() == gdn.GDN_OK
    return out.cpu(), s.cpu()


LENGTHS = [0, 1, 63, 64, 65, 200, 130, 0, 7]


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_varlen_matches_oracle_and_single_calls(dtype):
    bf = dtype == "bf16"
    base = syn.PREFILL_BF16_GQA2 if bf else syn.PREFILL_F32_SMALL
    D = 128 if bf else 64
    x, cu, st = _packed(base, LENGTHS, Hk=2, Hv=4, D=D)
    out, s = _gpu(x, cu, st)
    o_ref, s_ref = oracle.prefill_varlen(x["q"], x["k"], x["v"], x["g_log"], x["beta"],
                                         x["scale"], cu, st)
    tol = TOL_BF16 if bf else TOL_F32
    assert rel(to_np(out), o_ref) <= tol["out"]
    assert rel(to_np(s), s_ref) <= tol["state"]
    # each sequence alone through gdn_prefill: the same bits
    for n, L in enumerate(LENGTHS):
        if L == 0:
            assert torch.equal(s[n], st[n])
            continue
        t0, t1 = int(cu[n]), int(cu[n + 1])
        one = [x[nm][None, :, t0:t1].contiguous().to(DEV)
               for nm in ("q", "k", "v", "g_log", "beta")]
        o1, s1 = gdn.gdn_prefill(*one, x["scale"], state=st[n][None].to(DEV).clone())
        torch.cuda.synchronize()
        assert torch.equal(out[:, t0:t1], o1[0].cpu()), f"sequence {n}"
        assert torch.equal(s[n], s1[0].cpu()), f"sequence {n}"


def test_varlen_zero_initial_states_and_empty_tail():
    """No states supplied (zero start, written for every sequence, empty ones included);
    cu[N] < T leaves the trailing tokens' output rows untouched."""
    lengths = [100, 0, 300]
    x, cu, _ = _packed(syn.PREFILL_BF16_GQA2, lengths + [37], Hk=1, Hv=2, D=128, state=False)
    cu = cu[:-1]  # the last 37 tokens belong to no sequence
    args = [x[n].to(DEV) for n in ("q", "k", "v", "g_log", "beta")]
    out = torch.full((2, 437, 128), 7.0, dtype=torch.bfloat16, device=DEV)
    o, s = gdn.gdn_prefill_varlen(*args, x["scale"], torch.from_numpy(cu).to(DEV), out=out)
    torch.cuda.synchronize()
    o_ref, s_ref = oracle.prefill_varlen(x["q"], x["k"], x["v"], x["g_log"], x["beta"],
                                         x["scale"], cu)
    assert rel(to_np(o[:, :400].cpu()), o_ref[:, :400]) <= TOL_BF16["out"]
    assert rel(to_np(s.cpu()), s_ref) <= TOL_BF16["state"]
    assert torch.equal(s[1].cpu(), torch.zeros(2, 128, 128))
    assert (o[:, 400:] == 7.0).all()


def test_varlen_malformed_offsets_are_reported():
    """A decreasing cu_seqlens is caught on the device: every sequence is treated as
    empty (supplied states unchanged) and the device status says GDN_EINVAL."""
    x, cu, st = _packed(syn.PREFILL_BF16_GQA2, [64, 64], Hk=1, Hv=2, D=128)
    bad = np.array([0, 100, 50], dtype=np.int32)
    args = [x[n].to(DEV) for n in ("q", "k", "v", "g_log", "beta")]
    s_dev = st.to(DEV)
    gdn.gdn_prefill_varlen(*args, x["scale"], torch.from_numpy(bad).to(DEV), state=s_dev)
    torch.cuda.synchronize()
    assert gdn.gdn_get_device_status() == gdn.GDN_EINVAL
    assert "cu_seqlens" in gdn.gdn_last_error()
    assert torch.equal(s_dev.cpu(), st)
    assert gdn.gdn_get_device_status() == gdn.GDN_OK  # reported once


def test_varlen_many_sequences_sampled():
    """64 sequences of 1..700 tokens (Hk = 16, Hv = 32, bf16): the carry grid holds
    2048 (sequence, head) rows, so the one-CTA-per-head carry runs; sampled sequences
    against the oracle."""
    rng = np.random.default_rng(5)
    lengths = rng.integers(1, 700, size=64).tolist()
    x, cu, st = _packed(syn.PREFILL_BF16_GQA2, lengths, Hk=16, Hv=32, D=128, seed=2)
    out, s = _gpu(x, cu, st)
    for n in (0, 17, 63):
        t0, t1 = int(cu[n]), int(cu[n + 1])
        o_ref, s_ref = oracle.prefill(x["q"][None, :, t0:t1], x["k"][None, :, t0:t1],
                                      x["v"][None, :, t0:t1], x["g_log"][None, :, t0:t1],
                                      x["beta"][None, :, t0:t1], x["scale"], st[n][None])
        assert rel(to_np(out[:, t0:t1]), o_ref[0]) <= TOL_BF16["out"]
        assert rel(to_np(s[n]), s_ref[0]) <= TOL_BF16["state"]
