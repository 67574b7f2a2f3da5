"""Checkpoint / resume: inputs saved to disk and reloaded in a NEW process
give outputs whose chunk fingerprints are bitwise equal to the original
run's (the property the pages' bitwise-resume guarantee rests on)."""
import json
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

from bitwise_deterministic_moe_gb300 import api, synth
from tests import gpu_util
from tests.gpu_util import Problem

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r"""
import json, sys
import numpy as np, torch
sys.path.insert(0, sys.argv[1])
from bitwise_deterministic_moe_gb300 import api, synth
from tests.gpu_util import Problem
z = np.load(sys.argv[2])
cfg = synth.custom_config("resume", **json.loads(sys.argv[3]))
inp = synth.MoEInputs(cfg, z["ids"], z["X"], z["W"], z["G"], z["probs"])
p = Problem(cfg, inp)
out, dprob, slots = p.run_dprob()
res = {name: api.fingerprint_host(t) for name, t in (("out", out), ("dprob", dprob), ("slots", slots), ("src", p.src))}
assert api.read_status(p.ws) == 0
print(json.dumps(res))
"""


def test_resume_in_new_process_is_bitwise(tmp_path):
    gpu_util.ensure_built()
    shape = dict(T=3000, E=40, topk=5, K=256, N=512, routing="zipf", index=601)
    cfg = synth.custom_config("resume", **shape)
    inp = synth.make_inputs(cfg)
    p = Problem(cfg, inp)
    out, dprob, slots = p.run_dprob()
    ref = {name: api.fingerprint_host(t) for name, t in (("out", out), ("dprob", dprob), ("slots", slots),
                                                         ("src", p.src))}
    path = str(tmp_path / "inputs.npz")
    np.savez(path, ids=inp.topk_ids, X=inp.X, W=inp.W, G=inp.G, probs=inp.probs)
    r = subprocess.run([sys.executable, "-c", CHILD, ROOT, path, json.dumps(shape)],
                       capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    got = json.loads(r.stdout.strip().splitlines()[-1])
    for name in ref:
        assert [list(map(int, got[name][0])), int(got[name][1])] == [list(map(int, ref[name][0])), int(ref[name][1])], name
