"""The bench line's closing summary (CPU, no GPU): it names every protocol
and stays short enough to survive in the tail of a log that keeps only the
last few KB of output."""
import json

import bench


def _fake_line():
    sweep = []
    for op in ("ln", "rms"):
        for rows, d in ((32768, 8192), (8192, 768), (1024, 2048), (4096, 4096), (16384, 1024)):
            sweep.append({"op": op, "rows": rows, "d": d, "frac_of_measured_hbm": 0.7312345,
                          "kernel_over_copy_time": 1.0123,
                          "clean_l2": {"frac_of_measured_hbm": 0.8812345},
                          "back_to_back": {"frac_of_measured_hbm": 0.9012345}})
    small = [{"workload": f"rms_512x{d}_normal", "launch_latency_bound": False,
              "kernel_cold_us": 6.1234, "empty_cold_us": 4.1234,
              "bytes_at_measured_peak_us": 0.0123, "kernel_graph_us_per_launch": 1.6612,
              "empty_graph_us_per_launch": 0.8012}
             for d in (1, 31, 33, 127, 128, 4096, 8193)]
    small.insert(0, dict(small[0], workload="ln_512x128"))
    typed = [{"workload": f"ln_bfloat16_32768x8192_{i}", "frac_of_measured_hbm": 0.92345}
             for i in range(4)]
    bwd = [{"workload": f"ln_bwd_float32_16384x4096_{i}", "frac_of_measured_hbm": 0.90123}
           for i in range(6)]
    extra = {"sweep_cold_l2": sweep, "small_shapes_latency_bound": small,
             "storage_16bit_cold_l2": typed, "backward_cold_l2": bwd,
             "headline_stream_graph": {"frac_of_measured_hbm": 0.61234},
             "headline_cold_per_launch": {"frac_of_measured_hbm": 0.3461, "ms_mean": 0.0107}}
    return {"config": {"workload": "layernorm_fwd_fp32_4096x768"}, "ms_per_step": 0.0061234,
            "roofline": {"frac": 0.61234, "same_size_copy": {"kernel_over_copy_time": 0.98765}},
            "extra": extra}


def test_summary_is_short_and_names_its_protocols():
    s = bench.summary(_fake_line(), 6784.8)
    text = json.dumps(s)
    assert len(text) < 1500, len(text)
    assert set(s["protocols"]) == {"b2b", "cold", "clean"}
    assert s["headline"]["b2b_frac"] == 0.612
    assert s["shape_cols"] == ["b2b", "cold", "clean", "cold_over_copy"]
    assert s["shapes"]["ln_32768x8192"] == [0.901, 0.731, 0.881, 1.01]
    small = dict(zip(s["small_cols"], s["small"]["ln_512x128"]))
    assert small["latency_bound"] is False
    assert small["cold_bound_us"] == round(4.1234 + 0.0123 + 1.0, 2)


def test_both_arms_share_the_config():
    wl = bench.pick_workload("ln_4096x768")
    assert bench.headline_config(wl, 1) == bench.headline_config(wl, 1)
    assert "plan" not in bench.headline_config(wl, 1)
