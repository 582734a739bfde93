"""Host-side logic of bench.py (no GPU): the rotating input copies that stand in for an L2 flush, the note that
states what the timing saw, the lookup of committed ncu traffic, and the reference arm (the oracle on the host
cores), which needs no GPU at all."""
import json
import os
import subprocess
import sys

import pytest
import torch

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


class FakeCase(bench._Rotation):
    """Stand-in for a workload: one step 'touches' touch_bytes and records which copy it was handed."""

    def __init__(self, touch_bytes):
        self.dev = [torch.arange(8, dtype=torch.float32), torch.ones(4, dtype=torch.int32)]
        self.out = torch.zeros(3)
        self.lse = torch.zeros(2)
        self.touch_bytes = touch_bytes
        self.calls = []
        self._init_sets()

    def _call(self, dev, out, lse):
        self.calls.append((dev[0].data_ptr(), out.data_ptr(), lse.data_ptr()))


L2 = 129 * 10**6


@pytest.mark.parametrize("touch,steps,want", [
    (105 * 10**6, 200, 6),   # decode-sized step: 5 other steps cover 4x L2
    (2 * 10**9, 200, 2),     # one step already exceeds L2: two copies alternate
    (10**5, 200, 200),       # tiny step: capped at one copy per step
    (10**5, 1, 1),
])
def test_rotation_copy_count(touch, steps, want):
    c = FakeCase(touch)
    assert c.rotate_inputs(L2, max_copies=steps) == want
    assert len(c.sets) == want


def test_rotation_copies_are_distinct_and_equal():
    c = FakeCase(105 * 10**6)
    n = c.rotate_inputs(L2, max_copies=200)
    ptrs = {s[0][0].data_ptr() for s in c.sets}
    assert len(ptrs) == n  # every copy at its own address (L2 caches by address)
    for dev, out, lse in c.sets:
        assert torch.equal(dev[0], c.dev[0]) and torch.equal(dev[1], c.dev[1])
        assert out.shape == c.out.shape and lse.shape == c.lse.shape


def test_steps_cycle_through_every_copy_in_order():
    c = FakeCase(105 * 10**6)
    n = c.rotate_inputs(L2, max_copies=200)
    for _ in range(2 * n + 1):
        c.step()
    index = {s[0][0].data_ptr(): i for i, s in enumerate(c.sets)}
    order = [index[p[0]] for p in c.calls]
    assert order == [i % n for i in range(2 * n + 1)]
    # inputs and outputs of one step come from the same copy
    for p in c.calls:
        dev, out, lse = c.sets[index[p[0]]]
        assert (out.data_ptr(), lse.data_ptr()) == (p[1], p[2])


def test_l2_note_states_what_the_timing_saw():
    big = FakeCase(105 * 10**6)
    big.rotate_inputs(L2, max_copies=200)
    assert "inputs larger than L2" in bench.l2_note(big) and ">= 4x" in bench.l2_note(big)
    small = FakeCase(10**5)
    small.rotate_inputs(L2, max_copies=20)
    assert "may be L2-resident" in bench.l2_note(small)
    plain = FakeCase(10**5)  # never rotated (the host-only reference arm)
    assert "flushed" in bench.l2_note(plain)


def test_traffic_lookup_follows_the_kernel_source():
    # the committed decode summary matches the current source: its per-launch bytes are reported
    path = os.path.join(ROOT, "profiles", "decode_split_decode_gqa_traffic.txt")
    kv = dict(line.strip().split("=", 1) for line in open(path) if "=" in line and not line.startswith("#"))
    src = os.path.join(ROOT, "attention_attn_fwd_06_gb300", "csrc", kv["source"])
    if bench.code_digest(src) == kv["code_sha256_16"]:
        assert bench.read_traffic("decode_split", "decode_gqa") == float(kv["dram_bytes_per_launch"])
    assert bench.read_traffic("decode_split", "no_such_workload") is None


def test_code_digest_ignores_comments_but_not_code(tmp_path):
    a = tmp_path / "a.cu"
    a.write_text("int f(int x) {  // doubles\n  return 2 * x;\n}\n")
    b = tmp_path / "b.cu"
    b.write_text("int f(int x) {\n    return 2*x;  // the same code, other comments and spacing\n}\n")
    c = tmp_path / "c.cu"
    c.write_text("int f(int x) {\n  return 3 * x;\n}\n")
    assert bench.code_digest(str(a)) == bench.code_digest(str(b))
    assert bench.code_digest(str(a)) != bench.code_digest(str(c))


def _reference_run(extra_env=None, *args):
    env = dict(os.environ, **(extra_env or {}))
    cmd = [sys.executable, "bench.py", "--impl", "reference", "--workload", "tiny_causal", "--steps", "2",
           "--warmup", "1", "--ref-total", "2"] + list(args)
    return subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)


def test_reference_arm_prints_one_oracle_line():
    r = _reference_run()
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["metric"] == bench.METRIC
    assert line["value"] > 0 and line["unit"] == "TFLOP/s" and line["higher_is_better"] is True
    assert (line["steps"], line["warmup"], line["n_gpus"]) == (2, 1, 1)
    assert line["config"]["workload"] == "tiny_causal"
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == line["value"] and cb["sample"]
    assert line["e2e"] == {"value": line["value"], "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                           "d2h_bytes_per_step": 0}


def test_reference_arm_other_ranks_exit_without_work():
    r = _reference_run({"RANK": "1", "WORLD_SIZE": "2"})
    assert r.returncode == 0, r.stderr[-2000:]
    assert r.stdout.strip() == ""
