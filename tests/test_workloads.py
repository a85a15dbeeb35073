"""Seeded input generators: determinism, shapes and distribution recipes."""
import torch

from scaled_quantize_gemm_gb300 import workloads as wl


def test_same_seed_same_bits():
    a1, b1 = wl.w1_operands()
    a2, b2 = wl.w1_operands()
    assert torch.equal(a1, a2) and torch.equal(b1, b2)
    assert not torch.equal(a1, b1)


def test_w1_outliers():
    a, b = wl.w1_operands()
    assert a.shape == (256, 256) and a.dtype == torch.float32
    assert int((a.abs() == 30).sum()) == 4 and int((b.abs() == 30).sum()) == 4


def test_w2_drift_and_shapes():
    assert wl.w2_sigma(0) == 1.0 and wl.w2_sigma(19) == 8.0
    x = wl.linear_x(2, 0, 19, 2048, 768, std=wl.w2_sigma(19))
    assert x.dtype == torch.bfloat16 and x.shape == (2048, 768)
    assert 7.5 < float(x.float().std()) < 8.5
    w = wl.linear_w(2, 0, 2304, 768)
    assert 0.019 < float(w.float().std()) < 0.021
    dy = wl.linear_dy(2, 0, 0, 2048, 2304)
    assert 0.9e-3 < float(dy.float().std()) < 1.1e-3


def test_student_t_heavy_tail():
    x = wl.student_t3((512, 512), 123).float()
    # t(3) has variance 3 and far heavier tails than a normal
    assert 2.0 < float(x.var()) < 5.0
    assert float(x.abs().max()) > 15.0


def test_scaled_fraction_count():
    x = wl.with_scaled_fraction((256, 256), 1e-3, 100.0, 5, dtype=torch.float32)
    assert int((x.abs() > 20).sum()) >= 50   # 66 entries scaled by 100
