"""bench.py's reference arm on the CPU: `--impl reference` times the oracle on a
bounded sample of the balanced step and prints one JSON line with the keys the
benchmark contract names (the same metric, unit and direction as the GPU arm,
a cpu_baseline describing the run and an e2e object with no host copies).
Under torchrun only rank 0 prints; the others exit 0 without work."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def _run(env_extra=None):
    env = dict(os.environ)
    env.update(env_extra or {})
    p = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "0"],
                       capture_output=True, text=True, timeout=600, env=env, cwd=ROOT)
    return p


def test_reference_arm_json_line():
    import bench
    p = _run()
    assert p.returncode == 0, p.stderr[-2000:]
    lines = [l for l in p.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, p.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference"
    assert d["metric"] == bench.METRIC and d["unit"] == "TFLOP/s"
    assert d["higher_is_better"] is True and d["steps"] == 1 and d["warmup"] == 0
    assert d["value"] > 0 and d["ms_per_step"] > 0
    assert d["config"] == bench.bench_config(1)      # the GPU arm's config, every key
    assert d["config"]["workload"] == "deepseek_v3_moe_balanced"
    assert "extrapolated" in d["ms_per_step_basis"]
    om = d["oracle_measured"]
    assert om["seconds_per_step_sample"] > 0 and om["rows_per_gmm_per_sample"] >= 4
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"]
    assert isinstance(cb["sample"], str) and cb["sample"]
    e2e = d["e2e"]
    assert e2e["value"] == d["value"] and e2e["unit"] == d["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0


def test_reference_arm_other_ranks_do_no_work():
    p = _run({"RANK": "1", "WORLD_SIZE": "2", "LOCAL_RANK": "1",
              "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": "1"})
    assert p.returncode == 0, p.stderr[-2000:]
    assert not [l for l in p.stdout.splitlines() if l.startswith("{")]


def test_summarize_launches_groups_units_and_shares(tmp_path):
    """The launch-list summary behind the committed profiles: ncu's preamble
    lines are skipped, launches group by kernel name (template arguments kept,
    parameter list dropped), times in ns / us / ms all come out in us, and the
    shares add up to 1."""
    import bench
    hdr = ('"ID","Process ID","Process Name","Host Name","Kernel Name","Context","Stream",'
           '"Block Size","Grid Size","Device","CC","Section Name","Metric Name","Metric Unit",'
           '"Metric Value"')

    def row(i, name, unit, value):
        return (f'"{i}","1","python3","host","{name}","1","7","(896, 1, 1)","(152, 1, 1)","0",'
                f'"10.3","Command line profiler metrics","gpu__time_duration.sum","{unit}","{value}"')

    lines = ["==PROF== Connected to process 1", hdr,
             row(0, "void k::a<0>(int, float *)", "usecond", "300"),
             row(1, "void k::b(int)", "nsecond", "100,000"),
             row(2, "void k::a<0>(int, float *)", "msecond", "0.5"),
             row(3, "void k::a<1>(int, float *)", "usecond", "100")]
    p = tmp_path / "launches.csv"
    p.write_text("\n".join(lines) + "\n")
    table = bench.summarize_launches(str(p)).splitlines()
    assert table[0].startswith("| kernel | launches")
    body = [[c.strip() for c in l.strip("|").split("|")] for l in table[2:]]
    names = [b[0] for b in body]
    assert names == ["`void k::a<0>`", "`void k::b`", "`void k::a<1>`"]   # by total time
    a0 = body[0]
    assert a0[1] == "2" and float(a0[2]) == 800.0 and float(a0[3]) == 400.0
    assert float(body[1][2]) == 100.0 and float(body[2][2]) == 100.0
    assert abs(sum(float(b[4]) for b in body) - 1.0) < 2e-3


def test_traffic_is_null_unless_captured_on_the_current_sources(monkeypatch):
    """The roofline traffic figures are tied to a hash of the kernel sources
    they were measured on: a changed source gives null, not a stale number."""
    import bench
    t = dict(bench.TRAFFIC["wi_dlhs"])
    monkeypatch.setitem(bench.TRAFFIC, "wi_dlhs", dict(t, bytes=1.5e9,
                                                        sha1=bench.sources_sha1(t["sources"])))
    assert bench.traffic("wi_dlhs")[0] == 1.5e9
    monkeypatch.setitem(bench.TRAFFIC, "wi_dlhs", dict(t, bytes=1.5e9, sha1="0" * 40))
    b, why = bench.traffic("wi_dlhs")
    assert b is None and "changed" in why


def test_committed_traffic_figures_match_the_committed_sources():
    """Each traffic figure in bench.py was captured on the kernel sources as
    committed: a kernel change must come with a new capture."""
    import bench
    for kind in bench.TRAFFIC:
        b, why = bench.traffic(kind)
        assert b is not None, f"{kind}: {why}"
