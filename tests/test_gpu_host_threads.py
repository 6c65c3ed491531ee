"""Host threads whose FIRST calls into the library race (a fresh process, so nothing is
set up yet: the per-kernel shared-memory limits, the tensor-map encoder lookup, the side
streams): each thread runs its own layer on its own stream at the same moment, and the
results equal those of the same calls made one after the other.  The threads then exit
(their side streams are released) and new threads call again."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

SCRIPT = r'''
import sys, threading
import torch
sys.path.insert(0, sys.argv[1])
from expert_routed_ffn_router_gb300 import binding as B
from expert_routed_ffn_router_gb300 import synth

def problem(T, seed):
    w = synth.Workload("thr", T=T, H=256, E=16, K=4, I=128, Is=128, seed=seed, x_seed=seed + 1)
    d = synth.to_device({k: v for k, v in synth.host_inputs(w).items() if k != "K"}, "cuda:0")
    return w, d

torch.cuda.init()
probs = [problem(T, 100 + i) for i, T in enumerate((40, 300, 7, 2100))]
layers = [B.MoELayer(d, w.T, w.K) for (w, d) in probs]
torch.cuda.synchronize()
barrier = threading.Barrier(len(layers))
errors = []

def run(i):
    try:
        s = torch.cuda.Stream()
        with torch.cuda.stream(s):
            barrier.wait()
            layers[i].forward(probs[i][1]["X"])
        s.synchronize()
    except Exception as e:
        errors.append(repr(e))

def round_of_threads():
    th = [threading.Thread(target=run, args=(i,)) for i in range(len(layers))]
    for t in th: t.start()
    for t in th: t.join()

round_of_threads()                    # first calls of the process, all at once
assert not errors, errors
first = [(l.Y.clone(), l.topk_idx.clone(), l.counts.clone()) for l in layers]
assert all(l.status() == 0 for l in layers)
for i, l in enumerate(layers):        # the same calls one after the other
    l.forward(probs[i][1]["X"])
torch.cuda.synchronize()
for (Y, idx, c), l in zip(first, layers):
    assert torch.equal(idx, l.topk_idx) and torch.equal(c, l.counts)
    assert torch.equal(Y, l.Y)        # fixed summation orders: bitwise the same
round_of_threads()                    # new threads after the first ones exited
assert not errors, errors
torch.cuda.synchronize()
for (Y, idx, c), l in zip(first, layers):
    assert torch.equal(Y, l.Y)
print("threads ok")
'''


def test_first_calls_from_several_host_threads_race_safely():
    r = subprocess.run([sys.executable, "-c", SCRIPT, ROOT], capture_output=True, text=True,
                       timeout=600)
    assert r.returncode == 0 and "threads ok" in r.stdout, r.stdout + r.stderr
