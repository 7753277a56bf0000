"""The seeded input recipes: shapes, dtypes, the outlier rows of the LayerNorm -> Dense workload,
and reproducibility.  CPU only, at reduced sizes."""

import torch

from workloads import WORKLOADS, make_inputs, random_tensor


def test_shapes_and_dtypes_follow_the_recipes():
    t = make_inputs("tiny_ln_mlp")
    assert t["x"].shape == (64, 128) and t["w1"].shape == (128, 512) and t["w2"].shape == (512, 128)
    assert t["x"].dtype == torch.float32 and t["act"] == "gelu" and t["eps"] == 1e-6
    g = make_inputs("llama_rms_mlp", M=16, H=64, F=48)
    assert g["w1"].shape == (64, 96) and g["w2"].shape == (48, 64)  # gated: W1 has 2F columns
    assert g["x"].dtype == torch.bfloat16 and "b1" not in g and g["zero_centered_gamma"]
    assert torch.count_nonzero(g["beta"]) == 0
    b = make_inputs("gpt_ln_mlp_bwd", M=32, H=64, F=80)
    assert b["dy"].shape == (32, 64) and b["w1"].shape == (64, 80)
    assert WORKLOADS["qkv_ln_dense"]["eps"] == 1e-5


def test_outlier_rows_scaled_by_eight():
    d = make_inputs("qkv_ln_dense", M=1000, H=512, N=64)
    x = d["x"].float()
    rms = x.pow(2).mean(dim=1).sqrt()
    outliers = torch.arange(0, 1000, 100)
    others = torch.tensor([r for r in range(1000) if r % 100])
    assert len(outliers) == 10  # 1% of the rows
    ratio = rms[outliers].mean() / rms[others].mean()
    assert 7.0 < float(ratio) < 9.0
    # at full size: rows 0, 100, ..., 16300
    assert len(range(0, WORKLOADS["qkv_ln_dense"]["M"], 100)) == 164


def test_same_seed_same_bytes_and_other_seeds_differ():
    a = make_inputs("gpt_ln_mlp", M=8, H=32, F=48, seed=3)
    b = make_inputs("gpt_ln_mlp", M=8, H=32, F=48, seed=3)
    c = make_inputs("gpt_ln_mlp", M=8, H=32, F=48, seed=4)
    for k in ("x", "w1", "w2", "b1", "b2", "gamma", "beta"):
        assert torch.equal(a[k], b[k]), k
    assert not torch.equal(a["x"], c["x"])
    r = random_tensor((64, 64), std=2.0, mean=1.0, seed=9, dtype="f32")
    assert abs(float(r.mean()) - 1.0) < 0.2 and abs(float(r.std()) - 2.0) < 0.2
