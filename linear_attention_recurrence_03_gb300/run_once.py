"""Runs one workload a few times through the C ABI and exits: a small, deterministic
command for profilers (a fixed number of launches, no timing loop, no oracle).

    python -m linear_attention_recurrence_03_gb300.run_once decode --iters 2
    python -m linear_attention_recurrence_03_gb300.run_once prefill_layer --iters 2
    python -m linear_attention_recurrence_03_gb300.run_once prefill_batched --batch 3 --iters 2
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
    p.add_argument("workload", choices=sorted(PREFILL) + ["decode"])
    p.add_argument("--iters", type=int, default=2)
    p.add_argument("--heads", type=int, default=0,
                   help="prefill: keep only this many value heads (0 = all)")
    p.add_argument("--batch", type=int, default=0,
                   help="decode: this many batch rows of 32 value heads (0 = all 256); "
                        "prefill: this many batch rows (0 = the workload's)")
    a = p.parse_args(argv)
    lib_build.build()
    dev = torch.device("cuda:0")
    if a.workload == "decode":
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
