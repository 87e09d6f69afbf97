"""A bounded wait of the tensor-core prefill runs out, and the library says so.

Every mbarrier wait in the tensor-core kernels has a time limit; when one runs out the
kernel records a status bit, the other roles leave their loops, the MMAs and copies already
issued complete, tensor memory is freed, and gdn_get_device_status() reports GDN_ETIMEOUT.
This test makes that happen without a fault: a copy of the library built with the test-only
define GDN_TEST_STALL (wait limit 5 ms; the carry kernel's producer never loads the second
64-token chunk) runs one tiny prefill (1 head, S = 128), whose consumers then wait for data
that never comes. The normal library is then called on the same GPU and must give a clean
status and parity with the oracle: the stalled kernel left no tensor memory allocated and
nothing waiting.
"""
import os

import pytest
import torch

from gpu_util import DEV, TOL_BF16, ensure_built, gpu_prefill, oracle_prefill_all, rel, to_np
import linear_attention_recurrence_03_gb300 as gdn
from linear_attention_recurrence_03_gb300 import build as lib_build
from linear_attention_recurrence_03_gb300 import synthetic as syn

pytestmark = pytest.mark.gpu


def _stall_library():
    path = os.path.join(lib_build.BUILD + "_gdn_test_stall", "libgdn_test_stall.so")
    lib_build.build(defines=("GDN_TEST_STALL",), lib_path=path)
    return gdn.load_library(path)


def test_bounded_wait_runs_out_then_library_recovers():
    ensure_built()
    stall = _stall_library()
    w = syn.shrink(syn.PREFILL_BF16_GQA2, B=1, Hk=1, Hv=1, S=128, state_std=None)
    x = syn.prefill_inputs(w)
    X = [x[n].to(DEV) for n in ("q", "k", "v", "g_log", "beta")]
    import ctypes
    vp = ctypes.c_void_p
    state = torch.empty((1, 1, 128, 128), dtype=torch.float32, device=DEV)
    out = torch.empty((1, 1, 128, 128), dtype=torch.bfloat16, device=DEV)
    wsb = stall.gdn_prefill_workspace_bytes(1, 1, 1, 128, 128, 128, gdn.GDN_DTYPE_BF16)
    ws = torch.empty(wsb, dtype=torch.uint8, device=DEV)
    stream = vp(torch.cuda.current_stream().cuda_stream)
    rc = stall.gdn_prefill(*(vp(t.data_ptr()) for t in X), float(x["scale"]),
                           gdn.GDN_DTYPE_BF16, 1, 1, 1, 128, 128, 128, vp(state.data_ptr()), 0,
                           vp(out.data_ptr()), vp(ws.data_ptr()), wsb, stream)
    assert rc == gdn.GDN_OK  # enqueued: the failure is found on the device
    assert stall.gdn_get_device_status(stream) == gdn.GDN_ETIMEOUT
    assert "bounded wait" in stall.gdn_last_error().decode()
    # the status word was read and cleared
    assert stall.gdn_get_device_status(stream) == gdn.GDN_OK
    # the normal library on the same GPU: clean status and parity
    o, s = gpu_prefill(x)
    assert gdn.gdn_get_device_status() == gdn.GDN_OK
    o_ref, s_ref = oracle_prefill_all(x)
    assert rel(to_np(o), o_ref) <= TOL_BF16["out"]
    assert rel(to_np(s), s_ref) <= TOL_BF16["state"]


def test_decode_multi_wait_runs_out_then_library_recovers():
    """The same for the multi-token decode: in the GDN_TEST_STALL build each pipelined CTA
    never copies in the inputs of its second block of eight tokens, so with T = 16 its
    bounded wait for them runs out (5 ms): the call reports GDN_ETIMEOUT, and the normal
    library then runs the same call with a clean status and parity with the chained
    oracle."""
    ensure_built()
    stall = _stall_library()
    import ctypes
    import oracle
    names = ("q", "k", "v", "b", "a", "A_log", "dt_bias", "z", "norm_weight", "state")
    w = syn.DecodeWorkload("t", B=1, num_k_heads=2, num_v_heads=4, K=128, V=128)
    x = syn.decode_multi_inputs(w, 16)
    d = [x[n].to(DEV) for n in names]
    vp = ctypes.c_void_p
    so = torch.empty_like(d[-1])
    out = torch.empty((16, w.BH, w.V), dtype=torch.bfloat16, device=DEV)
    stream = vp(torch.cuda.current_stream().cuda_stream)
    rc = stall.gdn_decode_multi(*(vp(t.data_ptr()) for t in d), vp(so.data_ptr()),
                                vp(out.data_ptr()), 16, w.BH, w.num_v_heads, 128, 128, stream)
    assert rc == gdn.GDN_OK  # enqueued: the failure is found on the device
    assert stall.gdn_get_device_status(stream) == gdn.GDN_ETIMEOUT
    assert "bounded wait" in stall.gdn_last_error().decode()
    assert stall.gdn_get_device_status(stream) == gdn.GDN_OK
    y, st = gdn.gdn_decode_multi(*d, w.num_v_heads)
    assert gdn.gdn_get_device_status() == gdn.GDN_OK
    y_ref, s_ref = oracle.decode_multi(*(x[n] for n in names), w.num_v_heads)
    for t in range(16):
        assert rel(to_np(y[t].cpu()), y_ref[t]) <= TOL_BF16["out"], f"token {t}"
    assert rel(to_np(st.cpu()), s_ref) <= TOL_BF16["state"]
