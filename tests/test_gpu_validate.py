"""CB_VALIDATE=1: the GPU calls copy their metadata back and refuse a bad
step on the host, before any launch, with cb_validate_step's message.

Run in a child process, since the setting is read once per process.
"""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r"""
import sys
sys.path.insert(0, {root!r})
import numpy as np, torch
import paged_attention_continuous_gb300 as cb
import workloads
from paged_attention_continuous_gb300.step import StepRunner
from tests.test_gpu_parity import _decode_scenario
from tests.sched_driver import c_from_config, scenario_to_config
sc = _decode_scenario([40, 50, 300], 8, 2, 128, "bf16")
s = c_from_config(scenario_to_config(sc))
for r in sc.running:
    s.add_running_request(r.req_id, r.prompt_len, r.output_len, r.num_cached)
st = s.schedule_step()
runner = StepRunner(num_blocks=sc.num_blocks, num_q_heads=8, num_kv_heads=2, head_dim=128,
                    dtype="bf16", max_reqs=sc.max_requests_per_batch,
                    max_tokens=sc.max_batch_tokens, max_blocks_per_seq=sc.max_blocks_per_seq)
T = st["num_tokens"]
q = torch.zeros(T, 8, 128, dtype=torch.bfloat16, device="cuda")
kv = torch.zeros(T, 2, 128, dtype=torch.bfloat16, device="cuda")
runner.run(runner.upload(st), q, kv, kv)          # a good step runs
torch.cuda.synchronize()
st["block_tables"][1, 2] = sc.num_blocks + 3      # inside row 1's sequence
try:
    runner.run(runner.upload(st), q, kv, kv)
    print("NOT REFUSED")
except cb.CBError as e:
    print("REFUSED", e)
st["block_tables"][1, 2] = 0
st["slot_mapping"][0] = sc.num_blocks * 16
try:
    runner.run(runner.upload(st), q, kv, kv)
    print("NOT REFUSED")
except cb.CBError as e:
    print("REFUSED", e)
assert runner.workspace.read_errors() == 0        # nothing reached the kernels
print("DONE")
"""


def test_validate_mode_refuses_bad_steps_before_launch():
    env = dict(os.environ, CB_VALIDATE="1")
    r = subprocess.run([sys.executable, "-c", CHILD.format(root=ROOT)], env=env, cwd=ROOT,
                       capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-3000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith(("REFUSED", "NOT", "DONE"))]
    assert lines[0].startswith("REFUSED") and "row 1: block_tables[2]" in lines[0], lines
    assert lines[1].startswith("REFUSED") and "slot_mapping[0]" in lines[1], lines
    assert lines[-1] == "DONE"
