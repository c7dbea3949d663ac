"""The LM-head entry point that allocates nothing.

Some callers of this library cannot allocate device memory (a serving host
or plugin that owns all device memory through its own pool, or a loop that
must not call cudaMalloc); sprint_lmhead_confidence_noalloc serves them
from a fixed device array inside the library.  These tests call it through
the C ABI and check it against the allocating sprint_lmhead_confidence on
the same inputs, twice in a row, since the scratch array is reused between
calls.  The file is named to be collected last.
"""
import ctypes

import numpy as np
import pytest
import torch

from tests import gpu_cases as gc
from workload import generator

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _inputs(M, D, V, dtype, seed):
    g = generator(DEV, "noalloc", seed)
    h = torch.randn((M, D), generator=g, device=DEV).to(dtype)
    W = (torch.randn((V, D), generator=g, device=DEV) / 16).to(dtype)
    theta = 0.5 + 3.5 * torch.rand(M, generator=g, device=DEV)
    return h, W, theta


def _largest_rows_that_fit(D, V):
    """Most bf16 rows whose partials fit the library's scratch array."""
    from kv_cache_pruning_step_b300 import sprint as sp
    limit = 4 << 20
    M = 1
    while sp.lib.sprint_lmhead_workspace_bytes(M + 1, D, V, sp.BF16) <= limit:
        M += 1
    return M


@pytest.mark.parametrize("dtype,M,D,V", [(torch.bfloat16, 32, 2048, 157184),
                                         (torch.bfloat16, 300, 2048, 157184),
                                         (torch.bfloat16, "largest", 2048, 157184),
                                         (torch.float32, 40, 256, 1000)])
def test_noalloc_matches_allocating_entry_point_twice(dtype, M, D, V):
    """Block rows (one row tile), and 300 rows up to the largest call the
    array holds (row tiles in CTA pairs, partials filling the array)."""
    if M == "largest":
        M = _largest_rows_that_fit(D, V)
        assert M == 497
    from kv_cache_pruning_step_b300 import sprint as sp
    for seed in (1, 2):  # two calls in a row reuse the library's scratch array
        h, W, theta = _inputs(M, D, V, dtype, seed)
        c_ref, a_ref, l_ref = sp.sprint_lmhead_confidence(h, W, theta, want_logits=True)
        status = sp.new_status(DEV)
        c, a, lg = sp.sprint_lmhead_confidence_noalloc(h, W, theta, want_logits=True,
                                                       status=status)
        torch.cuda.synchronize()
        assert status.item() == 0
        err = (c.double() - c_ref.double()).abs().max().item()
        assert err <= gc.CONF_ATOL, err
        assert torch.equal(a, a_ref)
        gc.assert_close(gc.host(lg), gc.host(l_ref), dtype, "logits")


def test_noalloc_rejects_requests_beyond_its_array():
    from kv_cache_pruning_step_b300 import sprint as sp
    lib = sp.lib
    limit = sp.lib.sprint_lmhead_workspace_bytes(4096, 2048, 157184, sp.BF16)
    assert limit > (4 << 20)
    # too large: rejected on the host before any pointer is touched
    rc = lib.sprint_lmhead_confidence_noalloc(None, None, None, 4096, 2048, 157184, sp.BF16,
                                              None, None, None, None, None)
    assert rc == -6
    assert "scratch" in sp.sprint_strerror(rc)
    # one row past the largest call that fits is rejected the same way
    M = _largest_rows_that_fit(2048, 157184) + 1
    assert lib.sprint_lmhead_workspace_bytes(M, 2048, 157184, sp.BF16) > (4 << 20)
    rc = lib.sprint_lmhead_confidence_noalloc(None, None, None, M, 2048, 157184, sp.BF16,
                                              None, None, None, None, None)
    assert rc == -6
