"""gdn_prefill_noalloc, called through the C ABI, against gdn_prefill.

gdn_prefill_noalloc is the prefill for callers that cannot give the library device memory
while they run -- a plug-in inside a host runtime that owns the device memory and offers it
no allocator, or a latency-critical loop where an allocation (cudaMalloc can synchronise the
device) is not allowed. Instead of a caller workspace it uses a fixed 128 MiB array of the
library's own device memory, shared by every call and keeping the last call's contents.

These tests run its output against that of gdn_prefill (the entry point with a caller
workspace) on the same inputs, within the bf16 parity tolerance of the other tests (relative
Frobenius error: out 2e-2, state 1e-2) -- and, since both run the same kernels with the state
carried in fp32 across segments, bit for bit -- on calls in a row, so that a call that read
what the one before left in the array would show. This file runs last (its name sorts
last), and it builds and loads what it needs, so it also runs alone in a fresh process.
"""
import ctypes

import numpy as np
import pytest
import torch

from gpu_util import DEV, TOL_BF16, ensure_built, oracle_prefill_all, rel, to_np
import linear_attention_recurrence_03_gb300 as gdn
from linear_attention_recurrence_03_gb300 import synthetic as syn

pytestmark = pytest.mark.gpu

NAMES = ("q", "k", "v", "g_log", "beta")
VP = ctypes.c_void_p


@pytest.fixture(scope="module")
def lib():
    ensure_built()
    return gdn.load_library()


def _device_inputs(x):
    return {n: x[n].to(DEV) for n in NAMES}


def _shape(x):
    B, Hk, S, Dk = x["q"].shape
    return B, Hk, x["v"].shape[1], S, Dk, x["v"].shape[3]


def _run(lib, x, X, noalloc):
    """One call of either entry point through the C ABI on the device inputs X. Returns
    (out, final state) on the device."""
    B, Hk, Hv, S, Dk, Dv = _shape(x)
    sin = x["state"] is not None
    state = x["state"].to(DEV) if sin else torch.full((B, Hv, Dk, Dv), float("nan"),
                                                       device=DEV)
    out = torch.empty((B, Hv, S, Dv), dtype=torch.bfloat16, device=DEV)
    stream = VP(torch.cuda.current_stream().cuda_stream)
    args = [VP(X[n].data_ptr()) for n in NAMES] + [float(x["scale"]), gdn.GDN_DTYPE_BF16,
                                                   B, Hk, Hv, S, Dk, Dv,
                                                   VP(state.data_ptr()), int(sin),
                                                   VP(out.data_ptr())]
    if noalloc:
        rc = lib.gdn_prefill_noalloc(*args, stream)
    else:
        wsb = lib.gdn_prefill_workspace_bytes(B, Hk, Hv, S, Dk, Dv, gdn.GDN_DTYPE_BF16)
        ws = torch.empty(max(wsb, 16), dtype=torch.uint8, device=DEV)
        rc = lib.gdn_prefill(*args, VP(ws.data_ptr()), wsb, stream)
    assert rc == gdn.GDN_OK, lib.gdn_last_error().decode()
    torch.cuda.synchronize()
    return out, state


def _check_same(o1, s1, o2, s2):
    eo = rel(to_np(o2), to_np(o1))
    es = rel(to_np(s2), to_np(s1))
    assert eo <= TOL_BF16["out"], f"out rel diff {eo:.3e}"
    assert es <= TOL_BF16["state"], f"state rel diff {es:.3e}"
    assert torch.equal(o1, o2) and torch.equal(s1, s2), "not bit for bit"


def test_noalloc_equals_prefill_on_two_calls_in_a_row(lib):
    """Two different calls in a row (a supplied state, then a zero start with other inputs
    and a ragged tail): each equals gdn_prefill on its own inputs."""
    first = syn.prefill_inputs(syn.shrink(syn.PREFILL_BF16_GQA2, S=200))
    second = syn.prefill_inputs(syn.shrink(syn.PREFILL_BF16_GQA2, S=331, state_std=None),
                                seed=5)
    X1, X2 = _device_inputs(first), _device_inputs(second)
    a1 = _run(lib, first, X1, noalloc=True)
    a2 = _run(lib, second, X2, noalloc=True)
    _check_same(*_run(lib, first, X1, noalloc=False), *a1)
    _check_same(*_run(lib, second, X2, noalloc=False), *a2)
    assert gdn.gdn_get_device_status() == gdn.GDN_OK


def test_noalloc_segments_with_ragged_tail(lib):
    """B*Hv = 1300 leaves room for two chunks per (batch, head): S = 5*64 - 17 runs as
    segments of 2, 2 and 1 chunks, the last holding the ragged tail. With a zero start the
    later segments read back the state the earlier ones wrote. Both starts, two calls each,
    equal gdn_prefill and match the oracle over the whole tensor."""
    base = syn.shrink(syn.PREFILL_BF16_GQA2, B=5, Hk=130, Hv=260, S=5 * 64 - 17)
    for state_std in (None, 0.05):
        x = syn.prefill_inputs(syn.shrink(base, state_std=state_std))
        X = _device_inputs(x)
        r1 = _run(lib, x, X, noalloc=True)
        r2 = _run(lib, x, X, noalloc=True)
        ref = _run(lib, x, X, noalloc=False)
        _check_same(*ref, *r1)
        _check_same(*ref, *r2)
        o_ref, s_ref = oracle_prefill_all(x)
        assert rel(to_np(r1[0]), o_ref) <= TOL_BF16["out"]
        assert rel(to_np(r1[1]), s_ref) <= TOL_BF16["state"]


def test_noalloc_largest_head_count(lib):
    """B*Hv = 2701, the most (batch, head) pairs one chunk of which fits the scratch: the call
    is accepted and equals gdn_prefill; one more pair is refused."""
    x = syn.prefill_inputs(syn.shrink(syn.PREFILL_BF16_GQA2, B=1, Hk=1, Hv=2701, S=64))
    X = _device_inputs(x)
    _check_same(*_run(lib, x, X, noalloc=False), *_run(lib, x, X, noalloc=True))
    rc = lib.gdn_prefill_noalloc(VP(16), VP(16), VP(16), VP(16), VP(16), 1.0,
                                 gdn.GDN_DTYPE_BF16, 1, 1, 2702, 64, 128, 128, VP(16), 0,
                                 VP(16), None)
    assert rc == gdn.GDN_EUNSUPPORTED
    assert np.isfinite(x["scale"])
