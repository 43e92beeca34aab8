"""The pages' worked bandwidth figures, recomputed with the benchmark's own
accounting (CPU only).  The figures sit in tests/golden/pages_worked_numbers.txt,
each with the page and section that prints it (shivam2003.com, "A worked
bandwidth ceiling", "What a lane actually is" and "The arithmetic that forces
this"; agentlenshq.com, "Killing the 'Microsecond Losses'")."""
import os

import pytest

import bench
from synthetic import MODELS

HERE = os.path.dirname(os.path.abspath(__file__))


def _figures():
    out = {}
    with open(os.path.join(HERE, "golden", "pages_worked_numbers.txt")) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                name, value = line.split()
                out[name] = float(value)
    return out


FIG = _figures()


def test_every_figure_is_read():
    assert set(FIG) == {"params_2p3b_bytes_gb", "aggregate_bw_tbs", "measured_tok_s", "ceiling_fraction",
                        "lane_qkv_outputs", "launch_overhead_us_per_token", "launch_bound_tok_s",
                        "per_token_us_at_3000"}


def test_fp16_bytes_of_the_2p3b_decoder():
    # 2.3B parameters x 2 bytes; the ~2.3B workload's parameter count gives the same 4.6 GB
    assert 2.3e9 * 2 / 1e9 == pytest.approx(FIG["params_2p3b_bytes_gb"])
    assert MODELS["2.3b"].n_params() * 2 / 1e9 == pytest.approx(FIG["params_2p3b_bytes_gb"], abs=0.05)


def test_weight_only_ceiling_and_the_fraction_reached():
    bw = 8 * 4.3                                    # eight MI300X at ~4.3 TB/s each
    assert bw == pytest.approx(FIG["aggregate_bw_tbs"])
    bytes_tok = FIG["params_2p3b_bytes_gb"] * 1e9
    ceiling = bench.roofline_tok_s(bytes_tok, FIG["aggregate_bw_tbs"] * 1e3)
    assert ceiling == pytest.approx(7478, abs=1)    # 34.4 TB/s / 4.6 GB
    frac = bench.bandwidth_fraction(FIG["measured_tok_s"], bytes_tok, FIG["aggregate_bw_tbs"] * 1e3)
    assert frac == pytest.approx(FIG["ceiling_fraction"], abs=0.005)
    assert FIG["measured_tok_s"] / ceiling == pytest.approx(frac)


def test_launch_bound_rate_and_the_per_token_budget():
    # 1,125 us of launch overhead per token caps decode near 890 tokens/s
    assert bench.us_per_token(FIG["launch_bound_tok_s"]) == pytest.approx(FIG["launch_overhead_us_per_token"], rel=0.002)
    assert 1e6 / FIG["launch_overhead_us_per_token"] == pytest.approx(FIG["launch_bound_tok_s"], abs=1.5)
    # 3,000 tokens/s leaves 333 us per token
    assert bench.us_per_token(FIG["measured_tok_s"]) == pytest.approx(FIG["per_token_us_at_3000"], abs=0.5)


def test_lane_qkv_outputs():
    # one lane's fused QKV: 4 query heads, 2 key heads and 2 value heads of 96
    assert 4 * 96 + 2 * 96 + 2 * 96 == FIG["lane_qkv_outputs"]


def test_this_builds_ceiling_for_the_2p3b_workload():
    # the same accounting on this build's workload: 4.358 GB per step (weights + mean KV) at 8 TB/s
    from synthetic import WORKLOADS
    wl = WORKLOADS["2.3b"]
    mean_bytes = wl.decode_bytes(wl.prompt_len - 1, wl.decode_steps) / wl.decode_steps
    assert mean_bytes / 1e9 == pytest.approx(4.358, abs=0.002)
    assert bench.roofline_tok_s(mean_bytes, 8000) == pytest.approx(1836, abs=1)
