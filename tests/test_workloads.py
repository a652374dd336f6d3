"""The seeded input generator (paged_kv_cache_append_gb300/workloads.py), on
the CPU: the value-range knobs change V only, by the stated affine map, and
leave the default streams of every benchmark workload as they were."""

import numpy as np
import torch

from paged_kv_cache_append_gb300 import workloads as W


def _small(**kw):
    tables = np.arange(8, dtype=np.int32).reshape(2, 4)
    return W.Workload("t", "fp8_row", 2, 8, 2, 64, 256, 2, 8, tables,
                      table_rows=np.arange(2, dtype=np.int32), context=np.array([100, 37], np.int32),
                      scale=0.125, seed=42, outlier_p=0.05, outlier_mul=20.0, **kw)


def test_default_knobs_leave_the_streams_unchanged():
    a, b = _small(), _small(v_offset=0.0, v_mul=1.0)
    for layer in (0, 1):
        for x, y in zip(a.context_kv(layer, 1, 90) + a.step_kv(layer), b.context_kv(layer, 1, 90) + b.step_kv(layer)):
            assert torch.equal(x, y)


def test_power_of_two_multiplier_scales_v_exactly_and_nothing_else():
    base = _small()
    for k in (-14, -8, 10, 17):
        w = _small(v_mul=2.0 ** k)
        kb, vb = base.context_kv(0, 0, 120)
        kw_, vw = w.context_kv(0, 0, 120)
        assert torch.equal(kb, kw_)
        assert torch.equal(base.step_q(0), w.step_q(0))
        # bf16 rounding commutes with a power-of-two scale away from overflow
        # and the subnormal range
        assert torch.equal(vw.float(), vb.float() * 2.0 ** k)


def test_offset_is_added_before_the_multiplier():
    base, w = _small(), _small(v_offset=0.5, v_mul=4.0)
    _, vb = base.step_kv(1)
    _, vw = w.step_kv(1)
    # vw = bf16((x + 0.5) * 4) where vb = bf16(x): compare against the same
    # map applied to the float32 draw through bf16 once
    g = base._gen(1, 4, 0, "cpu")
    x = torch.randn(vb.shape, generator=g, dtype=torch.float32)
    u = torch.rand(vb.shape, generator=g)
    x = torch.where(u < base.outlier_p, x * base.outlier_mul, x)
    assert torch.equal(vb, x.to(torch.bfloat16))
    assert torch.equal(vw, ((x + 0.5) * 4.0).to(torch.bfloat16))
