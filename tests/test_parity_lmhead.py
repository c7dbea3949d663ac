"""GPU parity of sprint_lmhead_confidence against the oracle."""
import numpy as np
import pytest
import torch

from oracle import sprint_oracle as orc
from tests import gpu_cases as gc
from workload import (WORKLOADS, generator, lm_head_weight, prefix_inputs, step_inputs,
                      small_workload)

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def sp():
    from kv_cache_pruning_step_b300 import sprint
    return sprint


def draw(M, D, V, dtype, seed):
    g = generator(DEV, "lmhead-fuzz", seed)
    h = torch.randn((M, D), generator=g, device=DEV).to(dtype)
    W = (torch.randn((V, D), generator=g, device=DEV) / 16).to(dtype)
    theta = 0.5 + 3.5 * torch.rand(M, generator=g, device=DEV)
    return h, W, theta


def run(sp, h, W, theta, want_logits=True):
    status = sp.new_status(DEV)
    c, am, lg = sp.sprint_lmhead_confidence(h, W, theta, want_logits=want_logits, status=status)
    torch.cuda.synchronize()
    assert status.item() == 0
    return c, am, lg


def test_tiny_prefix_and_block_fp32(sp):
    w = WORKLOADS["tiny-256"]
    W = lm_head_weight(w, device=DEV)
    pre = prefix_inputs(w, device=DEV)
    x = step_inputs(w, 0, 0, 0, device=DEV)
    for h, th in ((pre["H"], pre["theta"]), (x["h"], x["theta"])):
        c, am, lg = run(sp, h, W, th)
        rows = np.arange(h.shape[0])
        z, _ = gc.check_confidence(c.cpu().numpy(), am.cpu().numpy(), h, W, th, rows, "tiny")
        gc.assert_close(gc.host(lg), z, torch.float32, "logits")


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("M,D,V", [(1, 8, 1), (37, 72, 255), (130, 256, 257), (300, 64, 1000),
                                   (129, 520, 513), (256, 128, 4096)])
def test_fuzz_shapes(sp, dtype, M, D, V):
    h, W, theta = draw(M, D, V, dtype, M * 7 + D + V)
    c, am, lg = run(sp, h, W, theta)
    z, _ = gc.check_confidence(c.cpu().numpy(), am.cpu().numpy(), h, W, theta, np.arange(M),
                               f"{M}x{D}x{V}")
    gc.assert_close(gc.host(lg), z, dtype, "logits")


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_closed_forms(sp, dtype):
    # h = 0: every logit 0, c = 1/V, argmax 0
    V, D = 777, 64
    h = torch.zeros((5, D), dtype=dtype, device=DEV)
    W = torch.randn((V, D), device=DEV).to(dtype)
    c, am, _ = run(sp, h, W, None, want_logits=False)
    assert torch.allclose(c, torch.full_like(c, 1.0 / V), rtol=1e-6, atol=0)
    assert (am == 0).all()
    # one dominant logit in the last column; ties resolve to the lowest index
    W = torch.zeros((V, D), dtype=dtype, device=DEV)
    W[V - 1, 0] = 8.0
    W[300, 1] = 2.0
    W[700, 1] = 2.0
    h = torch.zeros((3, D), dtype=dtype, device=DEV)
    h[0, 0] = 1.0
    h[1, 1] = 1.0
    h[2, 0] = 1.0
    theta = torch.tensor([1.0, 1.0, 4.0], device=DEV)
    c, am, _ = run(sp, h, W, theta, want_logits=False)
    assert am.tolist() == [V - 1, 300, V - 1]
    want0 = 1.0 / (1.0 + (V - 1) * np.exp(-8.0))
    want1 = 1.0 / (2.0 + (V - 2) * np.exp(-2.0))
    want2 = 1.0 / (1.0 + (V - 1) * np.exp(-2.0))
    np.testing.assert_allclose(c.cpu().numpy(), [want0, want1, want2], atol=1e-6)


def test_bad_temperature_reports_status(sp):
    h, W, theta = draw(4, 16, 40, torch.float32, 1)
    theta[2] = -1.0
    status = sp.new_status(DEV)
    sp.sprint_lmhead_confidence(h, W, theta, status=status)
    torch.cuda.synchronize()
    assert status.item() & sp.STATUS_BAD_TEMPERATURE


@pytest.fixture(scope="module")
def big_weight():
    return lm_head_weight(WORKLOADS["prefix-4k"], device=DEV)


def test_block_rows_full_vocab_bf16(sp, big_weight):
    w = WORKLOADS["prefix-4k"]
    x = step_inputs(w, 0, 0, 0, device=DEV)
    c, am, lg = run(sp, x["h"], big_weight, x["theta"])
    rows = np.arange(w.LB)
    z, nmis = gc.check_confidence(c.cpu().numpy(), am.cpu().numpy(), x["h"], big_weight,
                                  x["theta"], rows, "block rows")
    gc.assert_close(gc.host(lg), z, torch.bfloat16, "block logits")
    assert nmis <= 1


@pytest.mark.parametrize("M", [4096, 1000])
def test_prefix_rows_sampled_bf16(sp, big_weight, M):
    w = WORKLOADS["prefix-4k"]
    pre = prefix_inputs(w, device=DEV)
    H, theta = pre["H"][:M].contiguous(), pre["theta"][:M].contiguous()
    c, am, _ = run(sp, H, big_weight, theta, want_logits=False)
    rng = np.random.default_rng(M)
    rows = np.unique(np.concatenate([[0, M - 1, M // 2], rng.choice(M, 45, replace=False)]))
    _, nmis = gc.check_confidence(c.cpu().numpy()[rows], am.cpu().numpy()[rows], H, big_weight,
                                  theta, rows, "prefix rows")
    assert nmis <= 1
    # every confidence is a probability no smaller than 1/V
    cc = c.cpu().numpy()
    assert np.all(cc >= 1.0 / big_weight.shape[0] * (1 - 1e-5)) and np.all(cc <= 1.0 + 1e-6)


@pytest.mark.parametrize("M", [4096, 32, 700])
def test_confidence_without_argmax_bf16(sp, big_weight, M):
    """argmax_out = NULL (prefix scoring): the kernels skip the greedy token;
    the confidences are those of the call with it, bit for bit (the same
    maximum and sum per strip), and match the oracle."""
    w = WORKLOADS["prefix-4k"]
    pre = prefix_inputs(w, device=DEV)
    H, theta = pre["H"][:M].contiguous(), pre["theta"][:M].contiguous()
    c1, am1, _ = sp.sprint_lmhead_confidence(H, big_weight, theta)
    c0, am0, _ = sp.sprint_lmhead_confidence(H, big_weight, theta, want_argmax=False)
    torch.cuda.synchronize()
    assert am0 is None
    assert torch.equal(c0, c1)
    rows = np.unique(np.random.default_rng(M).choice(M, min(M, 40), replace=False))
    gc.check_confidence(c0.cpu().numpy()[rows], None, H, big_weight, theta, rows, "no argmax")


@pytest.mark.parametrize("M,V", [(20000, 2000), (40000, 30000), (20000, 40000)])
def test_tile_orders_bf16(sp, M, V):
    """h above the 32 MB band: (20000, 2000) keeps W in L2 in one band,
    (40000, 30000) keeps W in four bands, (20000, 40000) keeps h in three
    bands of 27 row units (6912 rows).  Each order must cover every output
    tile exactly once: sampled rows (among them both sides of a band edge)
    match the oracle, and every confidence is a probability of at least
    1/V."""
    D = 2048
    h, W, theta = draw(M, D, V, torch.bfloat16, M + V)
    c, am, _ = run(sp, h, W, theta, want_logits=False)
    rng = np.random.default_rng(V)
    edges = [0, M - 1, 6911, 6912, M // 2]
    rows = np.unique(np.concatenate([edges, rng.choice(M, 24, replace=False)]))
    rows = rows[rows < M]
    _, nmis = gc.check_confidence(c.cpu().numpy()[rows], am.cpu().numpy()[rows], h, W, theta,
                                  rows, f"order {M}x{V}")
    assert nmis <= 1
    cc = c.cpu().numpy()
    assert np.all(cc >= 1.0 / V * (1 - 1e-5)) and np.all(cc <= 1.0 + 1e-6)


def test_logit_error_is_within_the_argmax_excuse(sp):
    """The argmax excuse rests on the computed logits' error: at D = 2048
    (the model width) with temperatures down to 0.5 the fp32 logits stay
    within ARGMAX_EXCUSE / 4 of the fp64 oracle, so a greedy token can
    differ only on a near-tie of two logits."""
    g = generator(DEV, "logit-error", 2048)
    h = torch.randn((256, 2048), generator=g, device=DEV)
    W = torch.randn((8192, 2048), generator=g, device=DEV) / 16
    theta = 0.5 + 3.5 * torch.rand(256, generator=g, device=DEV)
    _, _, lg = run(sp, h, W, theta)
    _, _, z = orc.lm_confidence(h, W, theta, want_logits=True)
    err = np.abs(gc.host(lg).astype(np.float64) - z).max()
    assert err <= gc.ARGMAX_EXCUSE / 4, f"logit error {err:.3e}"
