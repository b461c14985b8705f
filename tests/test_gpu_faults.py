"""Failure detection without any GPU fault: errors are made on the host
(injected allocation failure, minimal buffers forcing the regrowth path, a
kernel wait given a flag value that nothing stores) and the library must
report them or recover with unchanged results."""
import os
import subprocess
import sys

import numpy as np
import pytest

from body_forces_morton_b300 import workloads as W

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r"""
import sys, json, numpy as np, torch
sys.path.insert(0, %r)
from body_forces_morton_b300 import native, workloads as W
g = W.generate(W.WORKLOADS[4], n=20000)
try:
    pl = native.Plan(20000, 4, 0.7, 16, "f32")
except native.FmmError as e:
    print(json.dumps({"create_error": str(e), "status": e.status})); sys.exit(0)
tp = torch.from_numpy(g["pos"]).cuda(); tm = torch.from_numpy(g["mass"]).cuda()
acc = torch.empty_like(tp)
pl.eval(tp, tm, acc)
st = pl.stats()
np.save(sys.argv[1], acc.cpu().numpy())
print(json.dumps({"retries": st["retries"]}))
""" % ROOT


def run_child(fault, out):
    env = dict(os.environ)
    if fault:
        env["BFM_FMM_FAULT"] = fault
    else:
        env.pop("BFM_FMM_FAULT", None)
    r = subprocess.run([sys.executable, "-c", CHILD, str(out)], env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr
    import json
    return json.loads(r.stdout.strip().splitlines()[-1])


def test_injected_allocation_failure_is_reported(tmp_path):
    res = run_child("alloc", tmp_path / "a.npy")
    assert res["status"] == 1 and "injected" in res["create_error"]


def test_minimal_buffers_regrow_to_the_same_result(tmp_path):
    normal = run_child(None, tmp_path / "n.npy")
    small = run_child("capacity", tmp_path / "s.npy")
    assert small["retries"] > 0
    assert np.array_equal(np.load(tmp_path / "n.npy"), np.load(tmp_path / "s.npy"))


SPIN_CHILD = r"""
import os, sys, json, time, numpy as np, torch
sys.path.insert(0, %r)
from body_forces_morton_b300 import native, workloads as W
g = W.generate(W.WORKLOADS[4], n=20000)
tp = torch.from_numpy(g["pos"]).cuda(); tm = torch.from_numpy(g["mass"]).cuda()
acc = torch.empty_like(tp)
res = {}
with native.Plan(20000, 4, 0.7, 16, "f32") as pl:  # created under BFM_FMM_FAULT=spin
    t0 = time.time()
    try:
        pl.eval(tp, tm, acc)
        res["error"] = None
    except native.FmmError as e:
        res["error"] = [e.status, str(e)]
    res["seconds"] = time.time() - t0
os.environ.pop("BFM_FMM_FAULT")
with native.Plan(20000, 4, 0.7, 16, "f32") as pl:
    pl.eval(tp, tm, acc)
np.save(sys.argv[1], acc.cpu().numpy())
print(json.dumps(res))
""" % ROOT


def test_expired_wait_is_reported_and_the_context_stays_usable(tmp_path):
    """Every L2L wait on a parent's flag is given a value that no pass stores:
    the waits run out their bound, the evaluation reports FMM_ERR_INTERNAL
    naming the spin limit, and a new plan in the same process still evaluates
    to the undisturbed result."""
    import json
    normal = run_child(None, tmp_path / "n.npy")
    assert normal["retries"] == 0
    env = dict(os.environ, BFM_FMM_FAULT="spin")
    r = subprocess.run([sys.executable, "-c", SPIN_CHILD, str(tmp_path / "s.npy")], env=env, capture_output=True,
                       text=True, timeout=600)
    assert r.returncode == 0, r.stderr
    res = json.loads(r.stdout.strip().splitlines()[-1])
    assert res["error"] is not None and res["error"][0] == 6 and "spin-limit" in res["error"][1], res
    assert np.array_equal(np.load(tmp_path / "n.npy"), np.load(tmp_path / "s.npy"))
