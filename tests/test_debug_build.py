"""The debug build of the library (SPRINT_DEBUG_CHECKS): it compiles,
exports the same ABI, says it is the debug build, and on the GPU reports a
broken invariant in the status word where the release build, which trusts
that invariant, does not look.  No check traps or stops a kernel."""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _debug_library():
    from kv_cache_pruning_step_b300.build import build
    return build(debug=True)


def test_debug_build_compiles_and_exports_the_abi():
    path = _debug_library()
    assert path.endswith("libsprint_debug.so") and os.path.exists(path)
    code = ("from kv_cache_pruning_step_b300 import sprint as sp; "
            "import tests.test_abi_host as t; "
            "assert all(hasattr(sp.lib, n) for n in t.declared_functions()); "
            "print(sp.LIB_PATH, sp.sprint_debug_checks())")
    out = subprocess.run([sys.executable, "-c", code], cwd=ROOT, capture_output=True, text=True,
                         env=dict(os.environ, SPRINT_LIBRARY=path, PYTHONPATH=ROOT), timeout=300)
    assert out.returncode == 0, out.stderr
    lib, flag = out.stdout.split()
    assert lib == path and flag == "1"


def test_release_build_has_no_debug_checks():
    from kv_cache_pruning_step_b300 import sprint as sp
    assert sp.sprint_debug_checks() == 0


CHILD = r"""
import torch
from kv_cache_pruning_step_b300 import sprint as sp
dev = "cuda"
NL, Hkv, d, n = 2, 2, 64, 40
K = torch.randn(NL * n * Hkv * d, device=dev).to(torch.bfloat16)
V = torch.randn(NL * n * Hkv * d, device=dev).to(torch.bfloat16)
off = torch.tensor([0, n], dtype=torch.int32, device=dev)
kept_off = torch.tensor([0, 5], dtype=torch.int32, device=dev)
good = torch.tensor([1, 4, 9, 20, 39], dtype=torch.int32, device=dev)
bad = torch.tensor([1, 9, 4, 20, 39], dtype=torch.int32, device=dev)   # not ascending
out = []
for idx in (good, bad):
    st = sp.new_status(dev)
    Kp, Vp = sp.sprint_compact_kv(K, V, off, n, NL, Hkv, d, idx, kept_off, 5, status=st)
    torch.cuda.synchronize()
    out.append(int(st.item()))
# an unmasked position without a token: the caller's mask and tokens disagree
conf = torch.rand(1, 8, device=dev)
am = torch.arange(8, dtype=torch.int32, device=dev)[None]
mask = torch.ones(1, 8, dtype=torch.uint8, device=dev)
mask[0, 3] = 0
tokens = torch.full((1, 8), -1, dtype=torch.int32, device=dev)
m = torch.zeros(1, dtype=torch.int32, device=dev)
st = sp.new_status(dev)
sp.sprint_unmask(conf, am, mask, tokens, 0, 4, 0.9, m_out=m, status=st)
torch.cuda.synchronize()
out.append(int(st.item()))
print("STATUS", sp.sprint_debug_checks(), *out)
"""


@pytest.mark.gpu
def test_debug_checks_report_broken_invariants():
    path = _debug_library()
    from kv_cache_pruning_step_b300 import sprint as sp
    for lib, want in ((path, sp.STATUS_DEBUG_CHECK), (None, 0)):
        env = dict(os.environ, PYTHONPATH=ROOT)
        if lib:
            env["SPRINT_LIBRARY"] = lib
        else:
            env.pop("SPRINT_LIBRARY", None)
        r = subprocess.run([sys.executable, "-c", CHILD], env=env, cwd=ROOT, capture_output=True,
                           text=True, timeout=300)
        assert r.returncode == 0, r.stdout + r.stderr
        line = [ln for ln in r.stdout.splitlines() if ln.startswith("STATUS")][-1]
        _, flag, good, bad, unmask = line.split()
        assert int(flag) == (1 if lib else 0)
        assert int(good) == 0, line                  # ascending indices: nothing reported
        assert int(bad) == want, line                # only the debug build reports it
        assert int(unmask) == want, line
