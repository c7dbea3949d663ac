"""Host-side checks of the C ABI that need no GPU: the library loads, it
exports every function include/sprint.h declares, host helpers agree with
the oracle, and invalid arguments are rejected before any launch."""
import ctypes
import os
import re

import pytest

from oracle import sprint_oracle as orc

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    names = set()
    for fname in os.listdir(os.path.join(ROOT, "include")):
        if fname.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fname)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names |= set(re.findall(r"\b(sprint_\w+)\s*\(", text))
    return sorted(names)


@pytest.fixture(scope="module")
def sp():
    from kv_cache_pruning_step_b300 import sprint
    return sprint


def test_library_exports_every_declared_symbol(sp):
    names = declared_functions()
    assert len(names) >= 11
    for name in names:
        assert hasattr(sp.lib, name), name
        assert name in sp.SIGNATURES, f"binding lacks {name}"


def test_binding_names_match_header(sp):
    for name in declared_functions():
        assert callable(getattr(sp, name)), name


def test_version_and_strerror(sp):
    assert sp.sprint_version() == 100
    for code in (0, -1, -2, -3, -5, -77):
        assert isinstance(sp.sprint_strerror(code), str)


def test_keep_count_matches_oracle(sp):
    for n in (0, 1, 3, 7, 64, 100, 1024, 3072, 16384, 32768):
        for r in (0.0, 0.1, 0.25, 0.29, 0.5, 0.75, 0.8, 0.9, 0.95, 0.999, 1.0):
            assert sp.sprint_keep_count(n, r) == orc.keep_count(n, r), (n, r)
    assert sp.sprint_keep_count(-1, 0.5) == -1
    assert sp.sprint_keep_count(10, 1.5) == -1


def test_invalid_arguments_rejected_without_launch(sp):
    lib = sp.lib
    P = ctypes.c_void_p
    # negative sizes / bad dtype / null pointers: rejected on the host
    assert lib.sprint_lmhead_confidence(None, None, None, -1, 8, 8, 1, None, None, None,
                                        None, 0, None, None) == -1
    assert lib.sprint_lmhead_confidence(None, None, None, 4, 8, 8, 7, None, None, None,
                                        None, 0, None, None) == -1
    assert lib.sprint_lmhead_confidence(None, None, None, 4, 8, 8, 1, None, None, None,
                                        None, 0, None, None) == -1
    assert lib.sprint_score_prune(None, 1, None, 10, 1, 1, 8, 0, None, None, 0.5, 1.5, 1.0,
                                  None, None, None, None, 0, None, None) == -1
    assert lib.sprint_compact_kv(None, None, 1, None, 10, 1, 1, 8, 3, None, None, 4, None,
                                 None, None, None) == -1
    # attention: Hq not a multiple of Hkv; unsupported head dim
    assert lib.sprint_block_attn(None, None, None, None, 4, 4, None, None, 1, 1, 32, 3, 2, 64,
                                 0, None, None, 0, None, None) == -1
    assert lib.sprint_block_attn(None, None, None, None, 4, 4, None, None, 1, 1, 32, 4, 2, 96,
                                 0, None, None, 0, None, None) == -2
    # LB * group > 128 rows is not supported
    assert lib.sprint_block_attn(None, None, None, None, 4, 4, None, None, 1, 1, 64, 8, 2, 64,
                                 0, None, None, 0, None, None) == -2
    # keep pools: pool count out of range; null keep counts
    assert lib.sprint_score_prune_pools(None, 1, P(16), 8, 1, 1, 8, 1, P(16), P(16), 0, P(16),
                                        0.5, P(16), P(16), 4, None, P(16), 1 << 20, P(16),
                                        None) == -1
    assert lib.sprint_score_prune_pools(None, 1, P(16), 8, 1, 1, 8, 1, P(16), P(16), 257, P(16),
                                        0.5, P(16), P(16), 4, None, P(16), 1 << 20, P(16),
                                        None) == -1
    assert lib.sprint_score_prune_pools(P(16), 1, P(16), 8, 1, 1, 8, 1, P(16), P(16), 3, None,
                                        0.5, P(16), P(16), 4, None, P(16), 1 << 20, P(16),
                                        None) == -1
    assert sp.sprint_score_prune_pools_workspace_bytes(2, 100, 300) == 0
    assert sp.sprint_score_prune_pools_workspace_bytes(2, 100, 17) >= 2 * 100 * 4 + 2 * 17 * 32
    # indexed attention: no kept indices / more kept rows than prefix rows
    assert lib.sprint_block_attn_indexed(None, None, None, None, 8, None, None, 4, 4, None, None,
                                         1, 1, 32, 4, 2, 64, 1, None, None, 0, None, None) == -1
    assert lib.sprint_block_attn_indexed(P(16), P(16), P(16), P(16), 2, P(16), P(16), 4, 4,
                                         P(16), P(16), 1, 1, 32, 4, 2, 64, 1, P(16), P(16),
                                         1 << 30, P(16), None) == -1
    assert lib.sprint_block_attn_indexed(None, None, None, P(16), 8, P(16), None, 4, 4, None,
                                         None, 1, 1, 32, 4, 2, 96, 1, None, None, 0, None,
                                         None) == -2
    assert lib.sprint_unmask(None, None, None, None, None, 1, 0, 0, 4, 0.9, 0, None, None,
                             None) == -1
    assert lib.sprint_unmask(None, None, None, None, None, 1, 32, 0, 4, 0.9, 5, None, None,
                             None) == -1
    # empty work is a no-op
    assert lib.sprint_lmhead_confidence(None, None, None, 0, 8, 8, 1, None, None, None,
                                        None, 0, None, None) == 0
    assert lib.sprint_unmask(None, None, None, None, None, 0, 32, 0, 4, 0.9, 0, None, None,
                             None) == 0


def test_workspace_queries(sp):
    assert sp.sprint_lmhead_workspace_bytes(32, 2048, 157184, 1) >= 3 * 32 * 614 * 4
    assert sp.sprint_score_prune_workspace_bytes(1, 32768) >= 8 * 32768
    assert sp.sprint_block_attn_workspace_bytes(1, 8, 32, 16, 4, 128, 32768, 1) > 0
    assert sp.sprint_block_attn_workspace_bytes(1, 8, 32, 16, 3, 128, 32768, 1) == 0


def test_steps_args_struct_matches_header(sp, tmp_path):
    """The ctypes mirror of sprint_steps_args has the C layout (field
    offsets and size compiled from include/sprint.h with the host compiler)."""
    import shutil
    import subprocess
    if shutil.which("gcc") is None:
        pytest.skip("no host C compiler")
    names = [f[0] for f in sp.StepsArgs._fields_]
    src = ["#include <stdio.h>", "#include <stddef.h>", '#include "sprint.h"', "int main(void){"]
    src += [f'printf("%zu\\n", offsetof(sprint_steps_args, {n}));' for n in names]
    src += ['printf("%zu\\n", sizeof(sprint_steps_args)); return 0;}']
    c = tmp_path / "off.c"
    c.write_text("\n".join(src))
    exe = tmp_path / "off"
    subprocess.run(["gcc", "-I", os.path.join(ROOT, "include"), "-I", "/usr/local/cuda/include",
                    str(c), "-o", str(exe)], check=True)
    out = [int(x) for x in subprocess.run([str(exe)], capture_output=True, text=True,
                                          check=True).stdout.split()]
    assert out[:-1] == [getattr(sp.StepsArgs, n).offset for n in names]
    assert out[-1] == ctypes.sizeof(sp.StepsArgs)
