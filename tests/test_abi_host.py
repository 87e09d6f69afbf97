"""Host-side checks of the C ABI that need no GPU: the library loads, exports every
function include/gdn.h declares, and rejects invalid arguments before touching CUDA."""
import ctypes
import os
import re

import pytest

from conftest import ROOT

import linear_attention_recurrence_03_gb300 as gdn
from linear_attention_recurrence_03_gb300 import build as lib_build


@pytest.fixture(scope="module")
def lib():
    lib_build.build()
    return gdn.load_library()


def header_functions():
    src = open(os.path.join(ROOT, "include", "gdn.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(gdn_[a-z0-9_]+)\s*\(", src)))


def test_header_declares_the_binding_exports():
    assert header_functions() == sorted(gdn.EXPORTS)


def test_library_exports_every_declared_symbol(lib):
    for name in header_functions():
        assert hasattr(lib, name), name


def test_library_is_built_for_sm_103a_only(lib):
    flags = " ".join(lib_build.NVCC_FLAGS)
    assert "arch=compute_103a,code=sm_103a" in flags
    assert flags.count("-gencode") == 1


def _prefill(lib, **kw):
    args = dict(q=16, k=16, v=16, g=16, beta=16, scale=1.0, dtype=1, B=1, Hk=1, Hv=1, S=64,
                Dk=128, Dv=128, state=16, sin=0, out=16, ws=None, wsb=0, stream=None)
    args.update(kw)
    vp = ctypes.c_void_p
    return lib.gdn_prefill(vp(args["q"]), vp(args["k"]), vp(args["v"]), vp(args["g"]),
                           vp(args["beta"]), args["scale"], args["dtype"], args["B"],
                           args["Hk"], args["Hv"], args["S"], args["Dk"], args["Dv"],
                           vp(args["state"]), args["sin"], vp(args["out"]), args["ws"],
                           args["wsb"], args["stream"])


@pytest.mark.parametrize("kw,msg", [
    (dict(Hk=3, Hv=4), "multiple of Hk"),
    (dict(Dk=129), "Dk, Dv"),
    (dict(Dv=0), "Dk, Dv"),
    (dict(B=0), "B >= 1"),
    (dict(S=-1), "S >= 0"),
    (dict(dtype=7), "dtype"),
    (dict(q=None), "non-NULL"),
    (dict(state=8), "16-byte"),
])
def test_prefill_rejects_bad_arguments(lib, kw, msg):
    assert _prefill(lib, **kw) == gdn.GDN_EINVAL
    assert msg in lib.gdn_last_error().decode()


def test_workspace_query(lib):
    assert lib.gdn_prefill_workspace_bytes(1, 3, 4, 64, 128, 128, 1) == ctypes.c_size_t(-1).value
    # tensor-core path: 49680 bytes per (batch, value head, 64-token chunk), ragged tail
    # rounded up; the fp32 and other-head-dim paths need none
    assert lib.gdn_prefill_workspace_bytes(1, 16, 32, 8192, 128, 128, 1) == 32 * 128 * 49680
    assert lib.gdn_prefill_workspace_bytes(2, 1, 3, 65, 128, 128, 1) == 2 * 3 * 2 * 49680
    assert lib.gdn_prefill_workspace_bytes(1, 16, 32, 8192, 128, 128, 0) == 0
    assert lib.gdn_prefill_workspace_bytes(1, 16, 32, 8192, 64, 128, 1) == 0


def test_prefill_requires_its_workspace(lib):
    assert _prefill(lib) == gdn.GDN_EINVAL
    assert "workspace" in lib.gdn_last_error().decode()


@pytest.mark.parametrize("B,Hv", [(1, 4096), (1, 2702), (2, 1351), (8, 512)])
def test_noalloc_rejects_more_heads_than_its_scratch(lib, B, Hv):
    """The 128 MiB scratch holds 2701 units of 49680 bytes: B * Hv = 2702 and above are
    refused on the host, before any launch (the accepted 2701 runs in the GPU tests)."""
    assert (128 << 20) // 49680 == 2701
    vp = ctypes.c_void_p
    rc = lib.gdn_prefill_noalloc(vp(16), vp(16), vp(16), vp(16), vp(16), 1.0, 1, B, 1, Hv,
                                 64, 128, 128, vp(16), 0, vp(16), None)
    assert rc == gdn.GDN_EUNSUPPORTED
    assert "static scratch" in lib.gdn_last_error().decode()


@pytest.mark.parametrize("kw,msg", [
    (dict(BH=10, H=4), "BH % num_v_heads"),
    (dict(K=200), "K, V"),
    (dict(out=None), "non-NULL"),
    (dict(state_out=16 + 64), "overlaps"),
])
def test_decode_rejects_bad_arguments(lib, kw, msg):
    a = dict(q=16, k=16, v=16, b=16, a=16, A_log=16, dt_bias=16, z=16, w=16, state_in=16,
             state_out=1 << 40, out=16, BH=8, H=4, K=128, V=128)
    a.update(kw)
    vp = ctypes.c_void_p
    rc = lib.gdn_decode_step(*(vp(a[n]) for n in ("q", "k", "v", "b", "a", "A_log", "dt_bias",
                                                  "z", "w", "state_in", "state_out", "out")),
                             a["BH"], a["H"], a["K"], a["V"], None)
    assert rc == gdn.GDN_EINVAL
    assert msg in lib.gdn_last_error().decode()


@pytest.mark.parametrize("kw,msg", [
    (dict(T=-1), "T >= 0"),
    (dict(BH=10, H=4), "BH % num_v_heads"),
    (dict(V=0), "K, V"),
    (dict(z=None), "non-NULL"),
])
def test_decode_multi_rejects_bad_arguments(lib, kw, msg):
    a = dict(q=16, k=16, v=16, b=16, a=16, A_log=16, dt_bias=16, z=16, w=16, state_in=16,
             state_out=16, out=16, T=3, BH=8, H=4, K=128, V=128)
    a.update(kw)
    vp = ctypes.c_void_p
    rc = lib.gdn_decode_multi(*(vp(a[n]) for n in ("q", "k", "v", "b", "a", "A_log",
                                                   "dt_bias", "z", "w", "state_in",
                                                   "state_out", "out")),
                              a["T"], a["BH"], a["H"], a["K"], a["V"], None)
    assert rc == gdn.GDN_EINVAL
    assert msg in lib.gdn_last_error().decode()


@pytest.mark.parametrize("kw,msg", [
    (dict(Hk=3, Hv=4), "multiple of num_k_heads"),
    (dict(Dk=129), "head_k_dim"),
    (dict(K=0), "K_win"),
    (dict(K=17), "K_win"),
    (dict(x=None), "non-NULL"),
    (dict(q=24), "non-NULL"),
    (dict(so=16 + 64), "overlaps"),
])
def test_conv1d_rejects_bad_arguments(lib, kw, msg):
    a = dict(x=16, w=16, si=16, so=1 << 40, q=16, k=16, v=16, B=2, Hk=2, Hv=4, Dk=128,
             Dv=128, K=4)
    a.update(kw)
    vp = ctypes.c_void_p
    rc = lib.gdn_conv1d_decode(*(vp(a[n]) for n in ("x", "w", "si", "so", "q", "k", "v")),
                               a["B"], a["Hk"], a["Hv"], a["Dk"], a["Dv"], a["K"], None)
    assert rc == gdn.GDN_EINVAL
    assert msg in lib.gdn_last_error().decode()


def test_varlen_workspace_query(lib):
    # tensor-core path: Hv * (ceil(T/64) + N) units of 49680 bytes (to 256), then the
    # N + 2 ints of the chunk table; fp32 / other head dims: the table alone (to 16)
    units = 32 * (4096 // 64 + 5) * 49680
    assert lib.gdn_prefill_varlen_workspace_bytes(5, 16, 32, 4096, 128, 128, 1) == \
        (units + 255) // 256 * 256 + 4 * 7
    assert lib.gdn_prefill_varlen_workspace_bytes(5, 2, 2, 100, 64, 64, 0) == 32
    assert lib.gdn_prefill_varlen_workspace_bytes(-1, 2, 2, 100, 64, 64, 0) == \
        ctypes.c_size_t(-1).value


@pytest.mark.parametrize("N,ws,msg", [(-1, 1 << 20, "N <="), (70000, 1 << 20, "N <="),
                                      (3, 8, "workspace")])
def test_varlen_rejects_bad_arguments(lib, N, ws, msg):
    vp = ctypes.c_void_p
    rc = lib.gdn_prefill_varlen(vp(16), vp(16), vp(16), vp(16), vp(16), 1.0, 0, vp(16), N, 2, 2,
                                100, 64, 64, vp(16), 0, vp(16), vp(16), ws, None)
    assert rc == gdn.GDN_EINVAL
    assert msg in lib.gdn_last_error().decode()


@pytest.mark.parametrize("n,C,alg,code,msg", [(-1, 64, 0, gdn.GDN_EINVAL, "n"),
                                               (4, 32, 0, gdn.GDN_EUNSUPPORTED, "C = 64"),
                                               (4, 64, 2, gdn.GDN_EINVAL, "algorithm")])
def test_unit_lower_inverse_rejects_bad_arguments(lib, n, C, alg, code, msg):
    vp = ctypes.c_void_p
    assert lib.gdn_unit_lower_inverse(vp(16), vp(1 << 40), n, C, alg, None) == code
    assert msg in lib.gdn_last_error().decode()


def test_binding_fails_loudly_without_library(tmp_path):
    with pytest.raises(RuntimeError, match="missing"):
        gdn.load_library(str(tmp_path / "libgdn.so"))
