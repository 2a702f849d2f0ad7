"""CPU checks of bench.py's host-side arithmetic: the FLOP count of the metric and the
L2-traffic model reported beside the roofline."""
import importlib.util
import math
import os

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    spec = importlib.util.spec_from_file_location("bench", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def test_mla_flops_count_every_product():
    b = _bench()
    n = 1000
    f_fwd, f_bwd = b.mla_flops(n)
    # forward: S = q kv^T over the 576-wide rows, O = P V over 512 channels, 64 heads
    assert f_fwd == 2 * 64 * n * (576 + 512)
    # backward: S and dP recomputed (576 + 512), dQ = dS kv (576), dKV = dS^T q (576) + P^T dO (512)
    assert f_bwd == 2 * 64 * n * (576 + 512 + 576 + 576 + 512)


def test_l2_model_bytes_and_times():
    b = _bench()
    n, tiles = 10_000_000, 80_000
    m = b.l2_model(n, tiles, fwd_ms=10.0, bwd_ms=20.0)
    red = 4 * 576 * n                       # one fp32 dkv row per valid slot
    gat_b = 2 * 2 * 576 * n + 2 * tiles * 128 * 64 * 2  # two bf16 row gathers + dS scratch out and back
    gat_f = 2 * 576 * n
    assert math.isclose(m["bwd"]["reduction_gb"], round(red / 1e9, 2))
    assert math.isclose(m["bwd"]["gather_gb"], round(gat_b / 1e9, 2))
    rr, rg = b.L2_RED_TBS * 1e12, b.L2_GATHER_TBS * 1e12  # the measured rates, bytes per second
    assert m["rates_tbs"] == {"reduction": b.L2_RED_TBS, "gather": b.L2_GATHER_TBS}
    t_b = (red / rr + gat_b / rg) * 1e3
    assert math.isclose(m["bwd"]["model_ms"], round(t_b, 3))
    assert math.isclose(m["bwd"]["frac"], round(t_b / 20.0, 4))
    assert math.isclose(m["fwd"]["model_ms"], round(gat_f / rg * 1e3, 3))
