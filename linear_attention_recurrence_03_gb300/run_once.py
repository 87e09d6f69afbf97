"""Runs one workload a few times through the C ABI and exits: a small, deterministic
command for profilers (a fixed number of launches, no timing loop, no oracle).

    python -m linear_attention_recurrence_03_gb300.run_once decode --iters 2
    python -m linear_attention_recurrence_03_gb300.run_once prefill_layer --iters 2
    python -m linear_attention_recurrence_03_gb300.run_once prefill_batched --batch 3 --iters 2
    python -m linear_attention_recurrence_03_gb300.run_once decode_multi --tokens 8 --batch 64
    python -m linear_attention_recurrence_03_gb300.run_once tril --matrices 16384
"""
from __future__ import annotations

import argparse
import sys

import torch

from . import build as lib_build
from . import gdn
from . import synthetic as syn

PREFILL = {
    "prefill_small_f32": syn.PREFILL_F32_SMALL,
    "prefill_gqa": syn.PREFILL_BF16_GQA2,
    "prefill_layer": syn.PREFILL_BF16_LAYER,
    "prefill_batched": syn.PREFILL_BF16_BATCHED,
}


def main(argv=None) -> int:
    p = argparse.ArgumentParser()
    p.add_argument("workload", choices=sorted(PREFILL) + ["decode", "decode_multi", "tril"])
    p.add_argument("--iters", type=int, default=2)
    p.add_argument("--heads", type=int, default=0,
                   help="prefill: keep only this many value heads (0 = all)")
    p.add_argument("--batch", type=int, default=0,
                   help="decode: this many batch rows of 32 value heads (0 = all 256); "
                        "prefill: this many batch rows (0 = the workload's)")
    p.add_argument("--tokens", type=int, default=8, help="decode_multi: tokens per call")
    p.add_argument("--matrices", type=int, default=16384,
                   help="tril: 64 x 64 chunk matrices per call (16384: 256 MB in, 256 MB out)")
    p.add_argument("--algorithm", choices=["neumann", "substitution"], default="neumann")
    a = p.parse_args(argv)
    lib_build.build()
    dev = torch.device("cuda:0")
    if a.workload == "tril":
        # unit lower-triangular chunk matrices A[r, j] = beta_r (k_r . k_j) exp(gamma_r -
        # gamma_j), j < r, from unit keys (the prefill's intra-chunk matrices)
        gen = torch.Generator().manual_seed(0)
        n = a.matrices
        k = torch.randn((n, 64, 128), generator=gen)
        k = k / torch.linalg.vector_norm(k, dim=-1, keepdim=True)
        beta = torch.rand((n, 64), generator=gen) * 0.9 + 0.05
        gam = torch.cumsum(torch.rand((n, 64), generator=gen) * -0.295 - 0.005, dim=1)
        A = torch.tril(beta[:, :, None] * (k @ k.transpose(1, 2)) *
                       torch.exp(gam[:, :, None] - gam[:, None, :]), -1)
        Ad = A.to(dev)
        alg = gdn.GDN_TRIL_NEUMANN if a.algorithm == "neumann" else gdn.GDN_TRIL_SUBSTITUTION
        for _ in range(a.iters):
            gdn.gdn_unit_lower_inverse(Ad, alg)
    elif a.workload == "decode_multi":
        wd = syn.DECODE_BH8192
        if a.batch:
            wd = syn.DecodeWorkload(wd.name, a.batch, wd.num_k_heads, wd.num_v_heads, wd.K, wd.V)
        x = syn.decode_multi_inputs(wd, a.tokens)
        names = ("q", "k", "v", "b", "a", "A_log", "dt_bias", "z", "norm_weight", "state")
        d = [x[n].to(dev) for n in names]
        for _ in range(a.iters):
            gdn.gdn_decode_multi(*d, x["num_v_heads"], state_out=d[-1])
    elif a.workload == "decode":
        wd = syn.DECODE_BH8192
        if a.batch:
            wd = syn.DecodeWorkload(wd.name, a.batch, wd.num_k_heads, wd.num_v_heads, wd.K, wd.V)
        x = syn.decode_inputs(wd)
        names = ("q", "k", "v", "b", "a", "A_log", "dt_bias", "z", "norm_weight", "state")
        d = [x[n].to(dev) for n in names]
        for _ in range(a.iters):
            gdn.gdn_decode_step(*d, x["num_v_heads"], state_out=d[-1])
    else:
        w = PREFILL[a.workload]
        if a.heads:
            w = syn.shrink(w, Hv=a.heads, Hk=max(1, a.heads * w.Hk // w.Hv))
        if a.batch:
            w = syn.shrink(w, B=a.batch)
        x = syn.prefill_inputs(w)
        t = [x[n].to(dev) for n in ("q", "k", "v", "g_log", "beta")]
        st = None if x["state"] is None else x["state"].to(dev)
        for _ in range(a.iters):
            gdn.gdn_prefill(*t, x["scale"], state=st)
    torch.cuda.synchronize()
    return 0 if gdn.gdn_get_device_status() == gdn.GDN_OK else 1


if __name__ == "__main__":
    sys.exit(main())
