"""Host-side logic of bench.py (CPU only): the multi-rank timing reduction
over a 2-rank gloo group, seeds per rank, the clock-sample summary and the
recorded-traffic lookup."""
import os
import socket

import pytest
import torch.multiprocessing as mp

import bench


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, results):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        mx = bench.reduce_max(10.0 + rank)
        results[rank] = (mx, bench.rank_seed(0, rank))
    finally:
        dist.destroy_process_group()


def test_reduce_max_over_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        results = m.dict()
        port = _free_port()
        procs = [ctx.Process(target=_rank_main, args=(r, 2, port, results)) for r in range(2)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(120)
            assert p.exitcode == 0
        res = dict(results)
    assert res[0][0] == res[1][0] == 11.0          # both ranks see the max
    assert res[0][1] != res[1][1]                  # independent batches per rank


def test_reduce_max_without_a_group_is_identity():
    assert bench.reduce_max(3.5) == 3.5


def test_clock_summary_prefers_the_timed_window():
    c = bench.ClockSampler("GPU-abc")
    row = ["GPU-abc", "1965", "2070", "900.5", "0x0", "Not Active", "Not Active", "Not Active",
           "Active"]
    idle = ["GPU-abc", "600", "2070", "100.0", "0x0", "Not Active", "Not Active", "Not Active",
            "Not Active"]
    other = ["GPU-zzz", "100", "2070", "50", "0x0", "Active", "Active", "Active", "Active"]
    c.samples = [(1.0, idle), (2.0, row), (2.5, row), (2.6, other), (4.0, idle)]
    s = c.summary(1.5, 3.0)
    assert s["sm_mhz"] == 1965 and s["sm_max_mhz"] == 2070
    assert s["reasons"] == ["sw_power_cap"] and s["samples_in_timed_region"] == 2


def test_recorded_traffic_requires_matching_sources(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "PROFILES", str(tmp_path))
    d = bench.source_digest("tp_token_cta_kernel")
    assert d != bench.source_digest("beam_token_bulk_kernel")
    (tmp_path / "k.md").write_text(
        f"traffic: kernel=tp_token_cta_kernel workload=w bytes_per_launch=123 sources={d}\n"
        "traffic: kernel=tp_token_cta_kernel workload=v bytes_per_launch=9 sources=stale\n")
    assert bench.recorded_traffic("tp_token_cta_kernel", "w") == 123
    assert bench.recorded_traffic("tp_token_cta_kernel", "v") is None
    assert bench.recorded_traffic("other", "w") is None


def test_parse_args_defaults_and_warmup_floor():
    a = bench.parse_args([])
    assert a.gpus == 1 and a.workload == "roofline" and a.impl == "ours" and a.warmup >= 3
    assert bench.parse_args(["--warmup", "1"]).warmup == 3


def test_cold_mode_arguments():
    a = bench.parse_args(["--workload", "decode", "--tokens", "8", "--cold"])
    assert a.cold and not a.graph
    # twice the 129 MB L2 at least, so one write evicts every input
    assert bench.L2_FLUSH_BYTES >= 2 * 129 * 10 ** 6
    with pytest.raises(SystemExit):
        bench.parse_args(["--cold", "--graph"])


def test_bytes_per_token_matches_the_workload_formulas():
    import synth_inputs as si
    kind, case, _ = bench.workload_case("small", None, 0)
    assert bench.bytes_per_token(kind, case) == si.algorithmic_bytes_tp(1) == 73792
    beam = si.beam_case("b", 4, 8, 7168, 3, seed=1)
    assert bench.bytes_per_token("beam", beam) == 129056
    assert bench.bytes_per_token("beam_residual", beam) == si.algorithmic_bytes_beam_residual(
        1, 7168, 8, True)


def test_algorithmic_bytes_formula():
    import synth_inputs as si
    # K*H*2 + H*2 + K*4 + K*4 per token with FP32 weights
    assert si.algorithmic_bytes_tp(1) == 8 * 4096 * 2 + 4096 * 2 + 32 + 32 == 73792
    assert si.algorithmic_bytes_tp(32768) == 2418016256
    assert si.algorithmic_bytes_beam(8000, 7168, 8) == 8000 * 129056


def test_reference_arm_prints_one_json_line():
    # the reference arm (the oracle on the host cores) on the 16-token workload
    import json
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    p = subprocess.run([sys.executable, os.path.join(root, "bench.py"), "--impl", "reference",
                        "--workload", "small", "--steps", "3", "--warmup", "3"],
                       capture_output=True, text=True, timeout=300, cwd=root)
    assert p.returncode == 0, p.stderr
    lines = [l for l in p.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "tokens/s" and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["steps"] == 3 and d["warmup"] == 3
    # the config carries the GPU arm's keys with the same meaning: the whole
    # 16-token batch fits the time budget, so one step finalizes all of it
    assert d["config"]["global_batch"] == 16 and d["config"]["parallelism"] == "single GPU"
    assert set(d["config"]) == {"workload", "global_batch", "parallelism"}


def _fake_nvml(max_mhz=2070.0):
    n = bench.NvmlClock.__new__(bench.NvmlClock)
    n.error, n.max_mhz = None, max_mhz
    return n


def test_nvml_summary_decodes_the_reason_bits():
    n = _fake_nvml()
    s = n.summary([(1.0, 2070.0, 900.0, 0x0), (1.1, 1995.0, 1380.0, 0x4 | 0x1),
                   (1.2, 2070.0, 950.0, 0x0)])
    assert s["sm_mhz"] == 2070.0 and s["sm_max_mhz"] == 2070.0 and s["power_w_max"] == 1380.0
    assert s["reasons"] == ["sw_power_cap"] and s["samples"] == 3     # idle bit 0x1 not a reason
    s = n.summary([(1.0, 1200.0, 900.0, 0x8 | 0x40 | 0x20)])
    assert s["reasons"] == ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown"]


def test_clock_record_counts_samples_inside_the_timed_region():
    smi = {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": [], "samples": 1,
           "samples_in_timed_region": 0}
    rec = bench.clock_record(smi, _fake_nvml(), [(1.0, 2055.0, 800.0, 0), (1.001, 2070.0, 820.0, 0)])
    assert rec["samples_in_timed_region"] == 2 and rec["sm_mhz"] == 2062.5
    assert rec["samples"] == 3 and "NVML" in rec["source"]
    # without NVML the nvidia-smi record stands, and says so
    broken = _fake_nvml()
    broken.error = "NVML unavailable: test"
    rec = bench.clock_record(smi, broken, [])
    assert rec["samples_in_timed_region"] == 0 and "nvidia-smi" in rec["source"]


def test_nvml_poll_stops_when_the_region_ends():
    class Ev:
        def __init__(self):
            self.n = 0

        def query(self):
            self.n += 1
            return self.n > 3
    n = _fake_nvml()
    n.sample = lambda: (0.0, 2070.0, 500.0, 0)
    got = []
    n.poll(Ev(), got, interval_s=0.0)
    assert len(got) == 3


def test_input_copies_keep_each_launch_cold():
    # a launch of a few L2 sizes rotates among copies so that its rows were last
    # read at least 4 x L2 of traffic earlier; large launches and L2-sized
    # (decode) ones use their buffers as they are
    L2 = bench.L2_BYTES
    for b in (L2, 302186496, 2 * L2, 4 * L2 - 1):
        n = bench.input_copies(b)
        assert n > 1 and (n - 1) * b >= 4 * L2
    assert bench.input_copies(2418016256) == 1 and bench.input_copies(4 * L2) == 1
    assert bench.input_copies(73792) == 1 and bench.input_copies(L2 - 1) == 1


def test_same_layout_copy_keeps_a_padded_row_stride():
    import torch
    t = torch.arange(6 * 4160, dtype=torch.float32).view(6, 4160)[:, :4096]
    c = bench._same_layout_copy(torch, t)
    assert c.stride() == (4160, 1) and torch.equal(c, t) and c.data_ptr() != t.data_ptr()


def test_source_digest_ignores_comments_only():
    # a recorded traffic figure stays valid across comment edits, not code edits
    a = "int x = 1; // one\n/* a block\n   comment */ int y;\n"
    b = "int x = 1;\nint y;  // another comment\n"
    assert bench.code_only(a) == bench.code_only(b) == "int x = 1; int y;"
    assert bench.code_only("int x = 1;") != bench.code_only("int x = 2;")
