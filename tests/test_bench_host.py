"""Host-side logic of bench.py that needs no GPU: the kernel-launch count it
claims, the clock-sample window, and the rule that a committed DRAM-traffic
record is used only while the kernel sources it was taken on are unchanged."""
import json
import os

import pytest

import bench
import workloads as W


@pytest.mark.parametrize("name,launches", [("prefill", 9), ("skewed", 9), ("reduced", 9), ("decode", 6),
                                           ("tiny", 6)])
def test_kernel_launches_per_forward(name, launches):
    # routing + permutation (two kernels when R > 1024, else one) + quantise
    # + FC1 and FC2 (a CTA-pair launch each when T > 64, plus a small-tile
    # launch each) + combine
    assert bench.kernel_launches(W.WORKLOADS[name]) == launches


def test_headline_config_is_shared_by_both_arms():
    a, b = bench.headline_config(1), bench.headline_config(1)
    assert a == b and a["global_batch"] == W.WORKLOADS["prefill"].T
    assert bench.headline_config(4)["global_batch"] == 4 * W.WORKLOADS["prefill"].T


class _Done:
    def terminate(self):
        pass

    def wait(self, timeout=None):
        return 0


def _sampler(tmp_path, lines, t0, t1):
    s = bench.ClockSampler(0)
    s.path = str(tmp_path / "clocks.csv")
    with open(s.path, "w") as f:
        f.write("\n".join(lines) + "\n")
    s.f = open(s.path, "a")
    s.proc = _Done()
    s.t0, s.t1 = t0, t1
    return s


def _line(stamp, mhz, reasons=()):
    names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
    flags = ["Active" if n in reasons else "Not Active" for n in names]
    return ", ".join([stamp, "0", str(mhz), "2070", "900.0", "0x0"] + flags)


def test_clock_samples_inside_the_timed_region_only(tmp_path):
    stamp = bench.ClockSampler._stamp
    t = [stamp(f"2026/12/02 10:00:0{i}.000") for i in range(6)]
    lines = [_line(f"2026/12/02 10:00:0{i}.000", mhz, r) for i, (mhz, r) in
             enumerate([(1000, ("hw_slowdown",)), (2070, ()), (2060, ("sw_power_cap",)), (2070, ()), (1200, ()),
                        (900, ("sw_thermal_slowdown",))])]
    out = _sampler(tmp_path, lines, t[1], t[3]).stop()
    assert out["samples"] == 3 and out["sm_mhz"] == 2070.0 and out["sm_max_mhz"] == 2070.0
    assert out["reasons"] == ["sw_power_cap"]          # the slowdowns outside the window are not counted


def test_clock_nearest_sample_when_none_inside(tmp_path):
    stamp = bench.ClockSampler._stamp
    lines = [_line("2026/12/02 10:00:00.000", 2000), _line("2026/12/02 10:00:05.000", 1500)]
    t0, t1 = stamp("2026/12/02 10:00:01.000"), stamp("2026/12/02 10:00:02.000")
    out = _sampler(tmp_path, lines, t0, t1).stop()
    assert out["samples"] == 1 and out["sm_mhz"] == 2000.0 and "nearest" in out["note"]


def _fake_root(tmp_path, sources):
    root = tmp_path / "root"
    csrc = root / "mxfp8_mxfp4_moe_gb300" / "csrc"
    csrc.mkdir(parents=True)
    for f in sources:
        (csrc / f).write_text(f"// {f}\n")
    (root / "profiles").mkdir()
    return root, csrc


@pytest.mark.parametrize("record,key,sha_fn,get_fn,sources", [
    ("fc1_dram_traffic.json", "fc1_kernel_sha256", "fc1_kernel_sha256", "fc1_traffic_record",
     bench.FC1_KERNEL_SOURCES),
    ("decode_fc1_dram_traffic.json", "decode_kernel_sha256", "decode_kernel_sha256", "decode_traffic_record",
     bench.DECODE_KERNEL_SOURCES),
])
def test_traffic_record_only_for_unchanged_sources(tmp_path, monkeypatch, record, key, sha_fn, get_fn, sources):
    root, csrc = _fake_root(tmp_path, sources)
    monkeypatch.setattr(bench, "ROOT", str(root))
    assert getattr(bench, get_fn)() is None                     # no record committed
    rec = {key: getattr(bench, sha_fn)(), "bytes": 123}
    (root / "profiles" / record).write_text(json.dumps(rec))
    assert getattr(bench, get_fn)() == rec                      # sources as captured
    (csrc / sources[-1]).write_text("// changed\n")
    assert getattr(bench, get_fn)() is None                     # a source changed since the capture


def test_committed_traffic_records_name_their_sources():
    for record, key in (("fc1_dram_traffic.json", "fc1_kernel_sha256"),
                        ("decode_fc1_dram_traffic.json", "decode_kernel_sha256")):
        rec = json.load(open(os.path.join(bench.ROOT, "profiles", record)))
        assert len(rec[key]) == 64 and "capture" in rec and "ncu" in rec["capture"]
