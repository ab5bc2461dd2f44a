"""Host-side logic of bench.py on CPU: ncu capture parsing into the machine-written
traffic records, the clock-window summary and the oracle's fixed sample."""
import json

import pytest

import bench


def test_ncu_kernel_key_normalises_template_arguments():
    fam, key = bench._ncu_kernel_key(
        "void fwd_kernel<128, 0, 0, 0, 0, 0>(CUtensorMap_st, CUtensorMap_st, CUtensorMap_st, "
        "FwdParams)")
    assert (fam, key) == ("fwd_kernel", "fwd_kernel<128,0,0,0,0,0>")
    fam, key = bench._ncu_kernel_key("void attn::bwd_kernel<64, (bool)1, (bool)0, true, "
                                     "false>(CUtensorMap)")
    assert key == "bwd_kernel<64,1,0,1,0>"
    assert bench._ncu_kernel_key("void stj_kernel<128, 0, 4>(CUtensorMap_st)")[1] == \
        "stj_kernel<128,0,4>"
    assert bench._ncu_kernel_key("void attn::nys_pool_kernel(attn::NysParams)")[0] == \
        "nys_pool_kernel"


def _csv(rows):
    head = ('"ID","Process ID","Process Name","Host Name","Kernel Name","Context","Stream",'
            '"Block Size","Grid Size","Device","CC","Section Name","Metric Name","Metric Unit",'
            '"Metric Value"')
    out = ["==PROF== preamble that is not CSV", head]
    for (lid, name, metric, unit, val) in rows:
        out.append('"%d","1","python","h","%s","1","7","(384, 1, 1)","(1024, 1, 1)","0",'
                   '"10.3","Command line profiler metrics","%s","%s","%s"'
                   % (lid, name, metric, unit, val))
    return "\n".join(out) + "\n"


def test_record_traffic_writes_json_that_the_bench_reads(tmp_path, monkeypatch):
    out = tmp_path / "dram_traffic.json"
    monkeypatch.setattr(bench, "TRAFFIC_JSON", str(out))
    fwd = "void fwd_kernel<128, 0, 0, 0, 0, 0>(CUtensorMap_st)"
    stj = "void stj_kernel<128, 0, 4>(CUtensorMap_st)"
    rows = []
    for lid, (rd, wr) in enumerate([(200.0, 45.0), (210.0, 45.0), (190.0, 45.0)]):
        rows += [(lid, fwd, "dram__bytes_read.sum", "Mbyte", "%.1f" % rd),
                 (lid, fwd, "dram__bytes_write.sum", "Mbyte", "%.1f" % wr),
                 (lid, fwd, "gpu__time_duration.sum", "usecond", "700")]
    rows += [(9, stj, "dram__bytes_read.sum", "Gbyte", "1.5"),
             (9, stj, "dram__bytes_write.sum", "byte", "1,000"),
             (9, stj, "gpu__time_duration.sum", "ns", "3,021,504")]  # ncu's short unit form
    csv_path = tmp_path / "cap.csv"
    csv_path.write_text(_csv(rows))
    bench.record_traffic(str(csv_path), "dense_b2_h16_n8192_d128", "ncu ...")
    data = json.loads(out.read_text())
    by_wl = {(r["family"], r["workload"]): r for r in data["rows"]}
    r = by_wl[("fwd_kernel", "dense_b2_h16_n8192_d128")]
    assert r["dram_bytes_per_launch"] == 245_000_000  # median of 245, 255, 235 MB
    assert r["launches"] == 3 and r["gpu_time_us_median_under_ncu"] == 700
    # a kernel only the Stieltjes row launches goes under that row's name
    assert by_wl[("stj_kernel", "stieltjes_b2_h16_n8192_d128_q4")][
        "dram_bytes_per_launch"] == 1_500_001_000
    assert by_wl[("stj_kernel", "stieltjes_b2_h16_n8192_d128_q4")][
        "gpu_time_us_median_under_ncu"] == 3021.5
    assert bench._recorded_traffic("fwd_kernel", "dense_b2_h16_n8192_d128") == 245e6
    assert bench._recorded_traffic("bwd_kernel", "dense_b2_h16_n8192_d128") is None
    # a record taken on other sources is ignored
    data["rows"][0]["source_hash"] = "0" * 16
    data["rows"][1]["source_hash"] = "0" * 16
    out.write_text(json.dumps(data))
    assert bench._recorded_traffic("fwd_kernel", "dense_b2_h16_n8192_d128") is None
    why = bench._traffic_or_why("stj_kernel", "stieltjes_b2_h16_n8192_d128_q4")
    assert why["traffic"] is None and "capture" in why["traffic_note"]
    # recording again replaces the row instead of adding a second one
    bench.record_traffic(str(csv_path), "dense_b2_h16_n8192_d128", "ncu ...")
    data = json.loads(out.read_text())
    assert sum(r["family"] == "fwd_kernel" for r in data["rows"]) == 1


def test_clock_summary_windows():
    c = bench.ClockSampler(0)
    c.samples = [(1.0, 1900.0, 2070.0, set()), (2.0, 2070.0, 2070.0, {"sw_power_cap"}),
                 (3.0, 2070.0, 2070.0, set()), (4.0, 1500.0, 2070.0, set())]
    whole = c.summary()
    assert whole["samples"] == 4 and whole["reasons"] == ["sw_power_cap"]
    w = c.summary(2.5, 3.5)
    assert w == {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": [], "samples": 1}
    assert c.summary(10.0, 11.0)["samples"] == 0


def test_workload_config_is_the_same_in_both_arms():
    a = bench.workload_config(bench.DEFAULT_WORKLOAD, 1)
    assert a == bench.workload_config(bench.DEFAULT_WORKLOAD, 1)
    assert a["l2"].startswith("no flush")
    assert bench.workload_config("dense_b1_h2_n256_d64", 1)["l2"].startswith("flushed")


def test_min_fwd_bytes_matches_the_configs_table():
    # B1 Hq2 N256 D64: 4 x 65,536 bytes of Q, K, V, O plus 2,048 of LSE
    assert bench.min_fwd_bytes(1, 2, 2, 256, 64) == 4 * 65536 + 2048
    # cfg 3: Q, O 8 MiB each, K, V 2 MiB each, LSE 128 KiB
    assert bench.min_fwd_bytes(1, 8, 2, 4096, 128) == 2 * 8 * 2**20 + 2 * 2 * 2**20 + 131072


@pytest.mark.parametrize("name", [c[0] for c in bench.BASELINE_CONFIGS])
def test_baseline_configs_are_well_formed(name):
    cfg = dict((c[0], c) for c in bench.BASELINE_CONFIGS)[name]
    B, Hq, Hkv, N, D, causal = cfg[1]
    assert Hq % Hkv == 0 and D in (64, 128) and cfg[2] in ("fwd", "fwd+bwd")


def test_clock_reader_parses_nvidia_smi_lines():
    import datetime
    c = bench.ClockSampler(0)

    class FakeProc:
        stdout = ["2026/12/02 10:41:00.500, 0, 2070, 2070, 900.10, 0x0000000000000004, "
                  "Not Active, Not Active, Not Active, Active\n",
                  "not a sample\n"]
    c.proc = FakeProc()
    c._read()
    assert len(c.samples) == 1
    when, sm, smax, active = c.samples[0]
    assert (sm, smax, active) == (2070.0, 2070.0, {"sw_power_cap"})
    assert when == datetime.datetime(2026, 12, 2, 10, 41, 0, 500000).timestamp()


def test_record_nystrom_traffic_sums_one_call_and_scales_the_streaming_passes(tmp_path,
                                                                               monkeypatch):
    out = tmp_path / "dram_traffic.json"
    monkeypatch.setattr(bench, "TRAFFIC_JSON", str(out))
    # (kernel, read MB, write MB): two calls, the second one's bytes 2 MB higher
    kernels = [("void nys_pool_kernel<128>(NysParams)", 100.0, 1.0),
               ("void nys_qt_kernel<128>(NysParams)", 2.0, 0.0),
               ("void nys_kv_kernel<128>(CUtensorMap_st, NysParams)", 200.0, 5.0),
               ("void nys_merge_kernel<128, 1>(NysParams)", 3.0, 0.0),
               ("void nys_lmy_kernel<128>(NysParams)", 4.0, 0.0),
               ("void nys_out_kernel<128>(CUtensorMap_st, NysParams)", 100.0, 100.0)]
    rows, lid = [], 0
    for extra in (0.0, 2.0):
        for name, rd, wr in kernels:
            rows += [(lid, name, "dram__bytes_read.sum", "Mbyte", "%.1f" % (rd + extra)),
                     (lid, name, "dram__bytes_write.sum", "Mbyte", "%.1f" % wr)]
            lid += 1
    csv_path = tmp_path / "nys.csv"
    csv_path.write_text(_csv(rows))
    bench.record_nystrom_traffic(str(csv_path), "nystrom_b4_h16_n131072_d128_m64", 8, "ncu ...")
    data = json.loads(out.read_text())
    (r,) = data["rows"]
    assert (r["family"], r["kernel"]) == ("nystrom_call", "nystrom_call")
    # medians: pool 102, qt 3, kv 206, merge 4, lmy 5, out 201 MB; streaming x 8
    assert r["per_kernel_bytes"]["nys_kv_kernel"] == 8 * 206_000_000
    assert r["per_kernel_bytes"]["nys_lmy_kernel"] == 5_000_000
    assert r["dram_bytes_per_launch"] == 8 * (102 + 206 + 201) * 10**6 + (3 + 4 + 5) * 10**6
    assert bench._recorded_traffic("nystrom_call", "nystrom_b4_h16_n131072_d128_m64") == \
        r["dram_bytes_per_launch"]
    # a capture without one of the six kernels is refused
    csv_path.write_text(_csv([x for x in rows if "lmy" not in x[1]]))
    with pytest.raises(SystemExit):
        bench.record_nystrom_traffic(str(csv_path), "nystrom_b4_h16_n131072_d128_m64", 8, "")
