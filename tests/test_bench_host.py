"""The benchmark's timing loop on CPU, with stand-ins for events, streams and the
clock sampler: the warm-up, the untimed run that keeps the GPU busy while clocks
are sampled, the timed region and the per-call latency pass each call the step
with call indices that only count up (so no timed call reuses the input copy or
the generator offset of the call before it), and the timed region holds exactly
`steps` calls."""
import ast
import os
import textwrap
import time
import types

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _timed_function(soak_s):
    src = open(os.path.join(ROOT, "bench.py")).read()
    tree = ast.parse(src)
    run_ours = next(n for n in tree.body if isinstance(n, ast.FunctionDef) and n.name == "run_ours")
    node = next(n for n in run_ours.body if isinstance(n, ast.FunctionDef) and n.name == "timed")
    code = textwrap.dedent(ast.get_source_segment(src, node))

    class Event:
        clock = 0.0

        def __init__(self, enable_timing=True):
            self.t = None

        def record(self, stream=None):
            Event.clock += 1.0
            self.t = Event.clock

        def elapsed_time(self, other):
            return other.t - self.t

    class Clocks:
        def __init__(self, idx):
            self.state = "new"

        def __enter__(self):
            self.state = "sampling"
            return self

        def __exit__(self, *exc):
            self.state = "stopped"

        def summary(self):
            return {"sm_mhz": 1.0, "state": self.state}

    cuda = types.SimpleNamespace(Event=Event, synchronize=lambda dev=None: None)
    ns = dict(torch=types.SimpleNamespace(cuda=cuda), time=time, SOAK_S=soak_s, Clocks=Clocks, local=0,
              smi_device_id=lambda local: "GPU-stand-in",
              dev=None, stream=None, barrier=lambda: None, slowest=lambda ms, dev: ms)
    exec(code, ns)
    return ns["timed"], Event


def test_timed_region_and_indices_with_clock_sampling():
    timed, Event = _timed_function(0.02)
    seen = []
    marks = []

    def step(i):
        seen.append(i)
        marks.append(Event.clock)

    t0 = time.perf_counter()
    total, per, clk = timed(step, 50, 5, clocks=True)
    assert time.perf_counter() - t0 >= 0.02          # the untimed run lasted the soak time
    assert seen == list(range(len(seen)))            # indices only count up
    soak = len(seen) - 5 - 2 * 50
    assert soak > 0 and soak % 64 == 0
    # The timed region: the 50 calls between its two events and nothing else.
    start_clock = marks[5 + soak]
    assert all(m == start_clock for m in marks[5 + soak:5 + soak + 50])
    assert total == 1.0 and len(per) == 50
    assert clk == {"sm_mhz": 1.0, "state": "stopped"}


def test_timed_without_clocks_has_no_untimed_run():
    timed, _ = _timed_function(5.0)
    seen = []
    total, per, clk = timed(seen.append, 20, 3)
    assert seen == list(range(3 + 2 * 20)) and clk is None and len(per) == 20


def test_reference_arm_prints_the_contract_line():
    """`bench.py --impl reference` (the CPU oracle, no GPU) prints one JSON line with
    the arm's metric, unit and config, the reference marks, and its own cpu_baseline
    and e2e figures."""
    import json
    import subprocess
    import sys
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "1", "--warmup", "0"],
                       cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [x for x in r.stdout.splitlines() if x.strip().startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    import bench
    assert d["impl"] == "reference" and d["metric"] == bench.METRIC and d["unit"] == "rows/s"
    assert d["n_gpus"] == 1 and d["steps"] == 1 and d["warmup"] == 0
    assert d["higher_is_better"] is True and d["scaling"] == "weak" and d["data"] == "synthetic"
    assert d["value"] > 0 and d["ms_per_step"] > 0 and d["vs_baseline"] is None
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"] and cb["sample"]
    e2e = d["e2e"]
    assert e2e["value"] == d["value"] and e2e["unit"] == d["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0
    assert d["config"]["batch"] == bench.B and d["config"]["vocab"] == bench.V
