"""Host logic of bench.py's clock record: samples outside the timed window and
rows of other GPUs are dropped; throttle reasons are read from the
nvidia-smi CSV columns."""
import importlib.util
import os
import time
from datetime import datetime

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    m = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(m)
    return m


def _row(ts, idx, uuid, sm, mx, hw="Not Active", cap="Not Active"):
    stamp = datetime.fromtimestamp(ts).strftime("%Y/%m/%d %H:%M:%S.%f")[:-3]
    return f"{stamp}, {idx}, {uuid}, {sm}, {mx}, 700.0, 0x0, {hw}, Not Active, Not Active, {cap}\n"


def _sampler(bench, rows, t0, t1, local=0, vis=None):
    old = os.environ.pop("CUDA_VISIBLE_DEVICES", None)
    if vis is not None:
        os.environ["CUDA_VISIBLE_DEVICES"] = vis
    try:
        c = bench.ClockSampler(local)
    finally:
        os.environ.pop("CUDA_VISIBLE_DEVICES", None)
        if old is not None:
            os.environ["CUDA_VISIBLE_DEVICES"] = old
    c.f.write("".join(rows))
    c.t0, c.t1 = t0, t1
    return c.summary()


def test_window_and_single_gpu():
    b = _bench()
    t = time.time()
    rows = [_row(t - 5, 0, "GPU-a", 1000, 2032),          # before the window
            _row(t + 0.1, 0, "GPU-a", 2032, 2032),
            _row(t + 0.2, 0, "GPU-a", 2010, 2032, cap="Active"),
            _row(t + 0.3, 0, "GPU-a", 2032, 2032),
            _row(t + 9, 0, "GPU-a", 300, 2032, hw="Active")]  # after it
    s = _sampler(b, rows, t, t + 1)
    assert s["samples"] == 3 and s["sm_mhz"] == 2032 and s["sm_max_mhz"] == 2032
    assert s["reasons"] == ["sw_power_cap"]


def test_picks_this_ranks_gpu():
    b = _bench()
    t = time.time()
    rows = []
    for j in range(3):
        rows += [_row(t + 0.1 * (j + 1), 0, "GPU-a", 1500, 2032, hw="Active"),
                 _row(t + 0.1 * (j + 1), 3, "GPU-d", 2032, 2032)]
    by_index = _sampler(b, rows, t, t + 1, local=1, vis="0,3")
    assert by_index["samples"] == 3 and by_index["sm_mhz"] == 2032 and by_index["reasons"] == []
    by_uuid = _sampler(b, rows, t, t + 1, local=0, vis="GPU-a")
    assert by_uuid["samples"] == 3 and by_uuid["reasons"] == ["hw_slowdown"]


def test_no_samples_reports_none():
    b = _bench()
    s = _sampler(b, [], time.time(), time.time() + 1)
    assert s["samples"] == 0 and s["sm_mhz"] is None
