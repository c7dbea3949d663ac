"""Failure reporting of the tcgen05 kernels without faulting the GPU.

Every pipeline wait in the tensor-core kernels is bounded.  With
SPRINT_TEST_STALL=1 (read once per process) the MMA role of each CTA first
waits on a barrier no one ever arrives on; with the limit set to 2 ms
(SPRINT_WAIT_CAP_NS) that wait expires, the CTA stops issuing work, waits
(with a separate one-second limit) for the copies and MMAs already issued,
frees its tensor memory and reports SPRINT_STATUS_TIMEOUT in the caller's
status word.  The CUDA context must stay usable afterwards.  Runs in a child
process so that the settings do not leak into other tests.
"""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r"""
import torch
from kv_cache_pruning_step_b300 import sprint as sp
dev = "cuda"
g = torch.Generator(device="cpu").manual_seed(5)
h = torch.randn(256, 256, generator=g).to(dev, torch.bfloat16)
W = (torch.randn(4096, 256, generator=g) / 16).to(dev, torch.bfloat16)
st = sp.new_status(dev)
sp.sprint_lmhead_confidence(h, W, None, status=st)
torch.cuda.synchronize()
lm = int(st.item())
S, NL, LB, Hq, Hkv, d, n = 1, 2, 32, 16, 4, 128, 1000
Q = torch.randn(S, NL, LB, Hq, d, generator=g).to(dev, torch.bfloat16)
K = torch.randn(NL * n * Hkv * d, generator=g).to(dev, torch.bfloat16)
V = torch.randn(NL * n * Hkv * d, generator=g).to(dev, torch.bfloat16)
Kb = torch.randn(S, NL, LB, Hkv, d, generator=g).to(dev, torch.bfloat16)
Vb = torch.randn(S, NL, LB, Hkv, d, generator=g).to(dev, torch.bfloat16)
off = torch.tensor([0, n], dtype=torch.int32, device=dev)
st2 = sp.new_status(dev)
sp.sprint_block_attn(Q, K, V, off, n, n, Kb, Vb, status=st2)
torch.cuda.synchronize()
at = int(st2.item())
x = (torch.ones(1000, device=dev) * 2).sum().item()   # context still usable
print("STATUS", lm, at, x)
"""


@pytest.mark.gpu
def test_wait_limit_reports_timeout_and_context_survives():
    env = dict(os.environ, SPRINT_WAIT_CAP_NS="2000000", SPRINT_TEST_STALL="1", PYTHONPATH=ROOT)
    r = subprocess.run([sys.executable, "-c", CHILD], env=env, cwd=ROOT, capture_output=True,
                       text=True, timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr
    line = [ln for ln in r.stdout.splitlines() if ln.startswith("STATUS")][-1]
    _, lm, at, x = line.split()
    from kv_cache_pruning_step_b300 import sprint as sp
    assert int(lm) & sp.STATUS_TIMEOUT, line
    assert int(at) & sp.STATUS_TIMEOUT, line
    assert float(x) == 2000.0
