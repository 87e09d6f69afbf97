"""The seeded input generator: shapes, dtypes, distributions and determinism."""
import torch

from linear_attention_recurrence_03_gb300 import synthetic as syn


def test_prefill_inputs_shapes_and_recipe():
    w = syn.shrink(syn.PREFILL_BF16_GQA2, S=128)
    x = syn.prefill_inputs(w)
    assert x["q"].shape == (2, 4, 128, 128) and x["q"].dtype == torch.bfloat16
    assert x["k"].shape == (2, 4, 128, 128) and x["v"].shape == (2, 8, 128, 128)
    assert x["g_log"].dtype == torch.float32 and x["g_log"].shape == (2, 8, 128)
    assert float(x["g_log"].min()) >= -0.3 and float(x["g_log"].max()) <= -0.005
    assert float(x["beta"].min()) >= 0.05 and float(x["beta"].max()) <= 0.95
    assert x["state"].shape == (2, 8, 128, 128)
    n = torch.linalg.vector_norm(x["q"].float(), dim=-1)
    assert torch.allclose(n, torch.ones_like(n), atol=1e-2)  # unit rows, then bf16
    x2 = syn.prefill_inputs(w)
    for key in ("q", "k", "v", "g_log", "beta", "state"):
        assert torch.equal(x[key], x2[key])
    assert not torch.equal(syn.prefill_inputs(w, seed=1)["q"], x["q"])


def test_zero_state_workloads_supply_none():
    x = syn.prefill_inputs(syn.PREFILL_F32_SMALL)
    assert x["state"] is None and x["q"].dtype == torch.float32
    assert x["scale"] == 1.0 / 8.0


def test_decode_inputs_gqa_expansion():
    w = syn.DecodeWorkload("t", B=3, num_k_heads=2, num_v_heads=4, K=16, V=8)
    x = syn.decode_inputs(w)
    assert x["q"].shape == (12, 16) and x["q"].dtype == torch.bfloat16
    q = x["q"].reshape(3, 4, 16)
    assert torch.equal(q[:, 0], q[:, 1]) and torch.equal(q[:, 2], q[:, 3])
    assert not torch.equal(q[:, 1], q[:, 2])
    assert x["state"].shape == (12, 16, 8) and x["state"].dtype == torch.float32
    assert x["A_log"].shape == (4,) and x["norm_weight"].shape == (8,)
    assert float(x["A_log"].min()) >= -2 and float(x["A_log"].max()) <= 1
