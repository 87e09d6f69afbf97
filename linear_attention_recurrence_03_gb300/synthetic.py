"""Seeded synthetic inputs for the GDN prefill and decode-step workloads.

This module only draws random numbers and lays them out; it holds none of the
recurrence's arithmetic. Both the CUDA path (tests, benchmark) and the fp64 oracle are
fed from it, and it imports neither.

Shapes follow "GDN CTE Kernel API Reference" (q,k [B,Hk,S,Dk] token-major,
v [B,Hv,S,Dv], g_log and beta [B,Hv,S] fp32, optional fp32 state [B,Hv,Dk,Dv]) and
"GDN TKG Kernel API Reference" (q,k,v,z [BH,K|V], b,a [BH], A_log and dt_bias
[num_v_heads], norm_weight [V], state [BH,K,V], BH = batch * num_v_heads with heads
cycling fastest). Prefill q/k must arrive L2-normalised (CTE Notes); each row is drawn
N(0,1), divided by its norm in fp32, then cast to the compute dtype. Decode q/k arrive
raw (TKG parameters) and are drawn at the key-head count, then repeated so that value
head h reads key head h // (num_v_heads // num_k_heads).
"""
from __future__ import annotations

from dataclasses import dataclass, replace

import math

import torch


@dataclass(frozen=True)
class PrefillWorkload:
    name: str
    dtype: str            # compute dtype of q/k/v/out: "f32" or "bf16"
    B: int
    Hk: int
    Hv: int
    S: int
    Dk: int
    Dv: int
    g_lo: float           # g_log ~ U(g_lo, g_hi)
    g_hi: float
    beta_lo: float        # beta ~ U(beta_lo, beta_hi)
    beta_hi: float
    state_std: float | None  # None: no initial state supplied (zero, not loaded)
    scale: float
    seed: int = 0

    @property
    def tokens(self) -> int:
        return self.B * self.S


@dataclass(frozen=True)
class DecodeWorkload:
    name: str
    B: int
    num_k_heads: int
    num_v_heads: int
    K: int
    V: int
    state_std: float = 0.05
    seed: int = 0

    @property
    def BH(self) -> int:
        return self.B * self.num_v_heads


# The five workloads, named by what they are and their sizes.
PREFILL_F32_SMALL = PrefillWorkload(
    "prefill_f32_b1_h2_s128_d64", "f32", 1, 2, 2, 128, 64, 64,
    -0.5, -0.01, 0.05, 0.95, None, 1.0 / 8.0)
PREFILL_BF16_GQA2 = PrefillWorkload(
    "prefill_bf16_b2_hk4_hv8_s1024_d128", "bf16", 2, 4, 8, 1024, 128, 128,
    -0.3, -0.005, 0.05, 0.95, 0.05, 128 ** -0.5)
PREFILL_BF16_LAYER = PrefillWorkload(
    "prefill_bf16_layer_b1_hk16_hv32_s8192_d128", "bf16", 1, 16, 32, 8192, 128, 128,
    -0.3, -0.005, 0.05, 0.95, None, 128 ** -0.5)
PREFILL_BF16_BATCHED = PrefillWorkload(
    "prefill_bf16_batched_b8_hk16_hv32_s4096_d128", "bf16", 8, 16, 32, 4096, 128, 128,
    -1.0, -0.001, 0.01, 0.99, 0.05, 128 ** -0.5)
DECODE_BH8192 = DecodeWorkload("decode_bf16_b256_hv32_k128_v128", 256, 16, 32, 128, 128)

PREFILL_WORKLOADS = (PREFILL_F32_SMALL, PREFILL_BF16_GQA2, PREFILL_BF16_LAYER,
                     PREFILL_BF16_BATCHED)


@dataclass(frozen=True)
class VarlenWorkload:
    """A variable-length batch: N sequences packed along the token axis, lengths drawn
    uniformly from [len_lo, len_hi] (a mix of short and long prompts), the layer's heads
    and distributions otherwise."""
    name: str
    base: PrefillWorkload
    N: int
    len_lo: int
    len_hi: int
    seed: int = 0

    def lengths(self) -> list[int]:
        gen = torch.Generator().manual_seed(self.seed + 7)
        return torch.randint(self.len_lo, self.len_hi + 1, (self.N,), generator=gen).tolist()


PREFILL_BF16_VARLEN = VarlenWorkload("prefill_bf16_varlen_n16_len256to4096_hk16_hv32_d128",
                                     PREFILL_BF16_LAYER, N=16, len_lo=256, len_hi=4096)


def varlen_inputs(w: VarlenWorkload) -> dict:
    """CPU tensors of a packed batch ([H, T, D] q, k, v; [Hv, T] g_log, beta), drawn as
    prefill_inputs for one row of T = sum(lengths) tokens, then cu_seqlens (int32)."""
    lengths = w.lengths()
    T = int(sum(lengths))
    x = prefill_inputs(replace(w.base, B=1, S=T, state_std=None), seed=w.seed)
    out = {n: x[n][0] for n in ("q", "k", "v", "g_log", "beta")}
    cu = [0]
    for L in lengths:
        cu.append(cu[-1] + L)
    out["cu_seqlens"] = torch.tensor(cu, dtype=torch.int32)
    out["scale"] = x["scale"]
    return out


def shrink(w: PrefillWorkload, **kw) -> PrefillWorkload:
    """Same distributions, other sizes (for small parity cases)."""
    return replace(w, **kw)


def _torch_dtype(name: str) -> torch.dtype:
    return {"f32": torch.float32, "bf16": torch.bfloat16}[name]


def _uniform(gen, shape, lo, hi):
    return torch.rand(shape, generator=gen, dtype=torch.float32) * (hi - lo) + lo


def _unit_rows(gen, shape):
    x = torch.randn(shape, generator=gen, dtype=torch.float32)
    return x / torch.linalg.vector_norm(x, dim=-1, keepdim=True)


def prefill_inputs(w: PrefillWorkload, seed: int | None = None) -> dict:
    """CPU tensors for one prefill call, drawn in the order q, k, v, g_log, beta, state."""
    gen = torch.Generator().manual_seed(w.seed if seed is None else seed)
    dt = _torch_dtype(w.dtype)
    q = _unit_rows(gen, (w.B, w.Hk, w.S, w.Dk)).to(dt)
    k = _unit_rows(gen, (w.B, w.Hk, w.S, w.Dk)).to(dt)
    v = torch.randn((w.B, w.Hv, w.S, w.Dv), generator=gen, dtype=torch.float32).to(dt)
    g_log = _uniform(gen, (w.B, w.Hv, w.S), w.g_lo, w.g_hi)
    beta = _uniform(gen, (w.B, w.Hv, w.S), w.beta_lo, w.beta_hi)
    state = None
    if w.state_std is not None:
        state = torch.randn((w.B, w.Hv, w.Dk, w.Dv), generator=gen,
                            dtype=torch.float32) * w.state_std
    return dict(q=q, k=k, v=v, g_log=g_log, beta=beta, state=state, scale=w.scale)


def decode_inputs(w: DecodeWorkload, seed: int | None = None) -> dict:
    """CPU tensors for one decode step, drawn in the order q, k, v, z, b, a, A_log,
    dt_bias, norm_weight, state. Distributions: q,k,v,z,b,a ~ N(0,1) (bf16);
    A_log ~ U(-2,1); dt_bias ~ U(-1,1); norm_weight ~ U(0.5,1.5); state ~ N(0, std^2)."""
    gen = torch.Generator().manual_seed(w.seed if seed is None else seed)
    G = w.num_v_heads // w.num_k_heads
    bf = torch.bfloat16

    def heads_expanded(dim):
        x = torch.randn((w.B, w.num_k_heads, dim), generator=gen, dtype=torch.float32)
        return x.repeat_interleave(G, dim=1).reshape(w.BH, dim).to(bf)

    q = heads_expanded(w.K)
    k = heads_expanded(w.K)
    v = torch.randn((w.BH, w.V), generator=gen, dtype=torch.float32).to(bf)
    z = torch.randn((w.BH, w.V), generator=gen, dtype=torch.float32).to(bf)
    b = torch.randn((w.BH,), generator=gen, dtype=torch.float32).to(bf)
    a = torch.randn((w.BH,), generator=gen, dtype=torch.float32).to(bf)
    A_log = _uniform(gen, (w.num_v_heads,), -2.0, 1.0)
    dt_bias = _uniform(gen, (w.num_v_heads,), -1.0, 1.0)
    norm_weight = _uniform(gen, (w.V,), 0.5, 1.5)
    state = torch.randn((w.BH, w.K, w.V), generator=gen, dtype=torch.float32) * w.state_std
    return dict(q=q, k=k, v=v, z=z, b=b, a=a, A_log=A_log, dt_bias=dt_bias,
                norm_weight=norm_weight, state=state, num_v_heads=w.num_v_heads)


def decode_multi_inputs(w: DecodeWorkload, T: int, seed: int | None = None) -> dict:
    """CPU tensors for T consecutive decode tokens: per token, in token order, q, k, v,
    z, b, a drawn as in decode_inputs (stacked on a leading T axis), then A_log, dt_bias,
    norm_weight and the state once."""
    gen = torch.Generator().manual_seed(w.seed if seed is None else seed)
    G = w.num_v_heads // w.num_k_heads
    bf = torch.bfloat16
    per = {n: [] for n in ("q", "k", "v", "z", "b", "a")}
    for _ in range(T):
        for n in ("q", "k"):
            x = torch.randn((w.B, w.num_k_heads, w.K), generator=gen, dtype=torch.float32)
            per[n].append(x.repeat_interleave(G, dim=1).reshape(w.BH, w.K))
        for n in ("v", "z"):
            per[n].append(torch.randn((w.BH, w.V), generator=gen, dtype=torch.float32))
        for n in ("b", "a"):
            per[n].append(torch.randn((w.BH,), generator=gen, dtype=torch.float32))
    out = {n: torch.stack(xs).to(bf) if xs else torch.empty((0,), dtype=bf)
           for n, xs in per.items()}
    out["A_log"] = _uniform(gen, (w.num_v_heads,), -2.0, 1.0)
    out["dt_bias"] = _uniform(gen, (w.num_v_heads,), -1.0, 1.0)
    out["norm_weight"] = _uniform(gen, (w.V,), 0.5, 1.5)
    out["state"] = torch.randn((w.BH, w.K, w.V), generator=gen, dtype=torch.float32) * w.state_std
    out["num_v_heads"] = w.num_v_heads
    return out



@dataclass(frozen=True)
class Conv1dWorkload:
    """One conv1d decode token in front of the decode step (the q|k|v channels of a
    Qwen3.5-style GDN layer: conv_dim = 2 num_k_heads head_k_dim + num_v_heads head_v_dim)."""
    name: str
    B: int
    num_k_heads: int
    num_v_heads: int
    head_k_dim: int
    head_v_dim: int
    K_win: int = 4
    seed: int = 0

    @property
    def conv_dim(self) -> int:
        return 2 * self.num_k_heads * self.head_k_dim + self.num_v_heads * self.head_v_dim


CONV1D_B256 = Conv1dWorkload("conv1d_decode_b256_hk16_hv32_d128_k4", B=256, num_k_heads=16,
                             num_v_heads=32, head_k_dim=128, head_v_dim=128)


def conv1d_inputs(w: Conv1dWorkload, seed: int | None = None) -> dict:
    """CPU tensors drawn in the order x, conv_weight, conv_state: x ~ N(0,1) and the window
    ~ N(0,1) (bf16, earlier tokens of the same activations), conv_weight ~ U(-1/sqrt(K_win),
    1/sqrt(K_win)) fp32 (the usual random init of a depthwise conv)."""
    gen = torch.Generator().manual_seed(w.seed if seed is None else seed)
    x = torch.randn((w.B, w.conv_dim), generator=gen, dtype=torch.float32).to(torch.bfloat16)
    bound = 1.0 / math.sqrt(w.K_win)
    weight = _uniform(gen, (w.conv_dim, w.K_win), -bound, bound)
    state = torch.randn((w.B, w.conv_dim, w.K_win), generator=gen,
                        dtype=torch.float32).to(torch.bfloat16)
    return dict(x=x, conv_weight=weight, conv_state=state)
