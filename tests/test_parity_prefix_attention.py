"""GPU parity of sprint_prefix_attn (the prefix's own attention in a
block's first step) against the oracle's prefix_attention.

Element by element at small ragged shapes (empty and one-position
sequences, query and key tiles with ragged tails, GQA groups 1 to 4, head
dims 64 and 128); on sampled positions at the 4K-prefix workload shapes
(8 layers, 16 query / 4 KV heads, d = 128), every layer and head."""
import numpy as np
import pytest
import torch

from oracle import sprint_oracle as orc
from tests import gpu_cases as gc
from workload import WORKLOADS, generator, prefix_inputs, prefix_queries

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def sp():
    from kv_cache_pruning_step_b300 import sprint
    return sprint


def _scaled(shape, g):
    """z * exp(0.5 y), y per position (axis 1), as the workload draws keys."""
    z = torch.randn(shape, generator=g, device=DEV)
    y = torch.randn(shape[1], generator=g, device=DEV)
    return z * torch.exp(0.5 * y).view(1, -1, *([1] * (len(shape) - 2)))


def _draw(lens, NL, Hq, Hkv, d, seed):
    g = generator(DEV, "prefix-attn-fuzz", seed)
    seqs = []
    for n in lens:
        Q = torch.randn((NL, n, Hq, d), generator=g, device=DEV).to(torch.bfloat16)
        K = _scaled((NL, n, Hkv, d), g).to(torch.bfloat16)
        V = _scaled((NL, n, Hkv, d), g).to(torch.bfloat16)
        seqs.append((Q, K, V))
    off = [0]
    for n in lens:
        off.append(off[-1] + n)
    cat = [torch.cat([x[i].reshape(-1) for x in seqs]) for i in range(3)]
    return seqs, cat, off


def _run(sp, cat, off, NL, Hq, Hkv, d):
    Qc, Kc, Vc = cat
    off_d = torch.tensor(off, dtype=torch.int32, device=DEV)
    status = sp.new_status(DEV)
    Op = sp.sprint_prefix_attn(Qc, Kc, Vc, off_d, off[-1], NL, Hq, Hkv, d, status=status)
    torch.cuda.synchronize()
    assert status.item() == 0
    return Op


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("Hq,Hkv", [(2, 2), (4, 2), (8, 2)])
def test_ragged_sequences_elementwise(sp, d, Hq, Hkv):
    lens = [100, 0, 1, 129, 300, 256]
    NL = 2
    seqs, cat, off = _draw(lens, NL, Hq, Hkv, d, seed=d + 10 * Hq)
    Op = _run(sp, cat, off, NL, Hq, Hkv, d)
    for s, (Q, K, V) in enumerate(seqs):
        n = lens[s]
        got = Op[NL * off[s] * Hq * d:NL * off[s + 1] * Hq * d].view(NL, n, Hq, d)
        if n == 0:
            continue
        want = orc.prefix_attention(Q, K, V)
        gc.assert_close(gc.host(got), want, torch.bfloat16, f"seq {s} (n = {n})")


def test_identical_keys_give_the_mean_value(sp):
    """A closed form on the GPU: with every key equal, each query's output
    is the mean of the values (over a prefix of 3 key tiles plus a tail)."""
    NL, Hq, Hkv, d, n = 1, 4, 2, 128, 300
    g = generator(DEV, "prefix-attn-mean", 1)
    Q = torch.randn((NL, n, Hq, d), generator=g, device=DEV).to(torch.bfloat16)
    key = torch.randn(d, generator=g, device=DEV)
    K = key.expand(NL, n, Hkv, d).contiguous().to(torch.bfloat16)
    V = torch.randn((NL, n, Hkv, d), generator=g, device=DEV).to(torch.bfloat16)
    Op = _run(sp, [Q.reshape(-1), K.reshape(-1), V.reshape(-1)], [0, n], NL, Hq, Hkv, d)
    mean = V.double().mean(dim=1)                            # [NL, Hkv, d]
    want = mean[:, None, [h // (Hq // Hkv) for h in range(Hq)], :].expand(NL, n, Hq, d)
    gc.assert_close(gc.host(Op.view(NL, n, Hq, d)), want.cpu().numpy(), torch.bfloat16,
                    "identical keys")


def test_prefix_4k_sampled_positions(sp):
    w = WORKLOADS["prefix-4k"]
    pre = prefix_inputs(w, device=DEV)
    Qp = prefix_queries(w, device=DEV)
    n = Qp.shape[1]
    off = torch.tensor([0, n], dtype=torch.int32, device=DEV)
    status = sp.new_status(DEV)
    Op = sp.sprint_prefix_attn(Qp, pre["K"], pre["V"], off, n, w.NL, w.Hq, w.Hkv, w.d,
                               status=status)
    torch.cuda.synchronize()
    assert status.item() == 0
    rng = np.random.default_rng(4)
    rows = np.unique(np.concatenate([[0, 127, 128, n - 1], rng.choice(n, 28, replace=False)]))
    want = orc.prefix_attention(Qp, pre["K"], pre["V"], rows=rows)
    got = gc.host(Op)[:, rows]
    gc.assert_close(got, want, torch.bfloat16, "prefix-4k sampled rows")


def test_decoder_runs_the_prefix_attention_at_step_0(sp):
    """BlockDecoder(prefix_attn=True) fills O_prefix at step 0 (checked on
    sampled rows) and decodes the same block as without it: the output
    feeds nothing downstream."""
    from kv_cache_pruning_step_b300 import BlockDecoder
    from workload import lm_head_weight, small_workload, step_inputs
    w = small_workload("prefix-attn-dec", dtype="bf16", NL=2, Hq=8, Hkv=2, d=128, D=1024,
                       V=4096, T=4, seed=23, n=700, n_img=300)
    W = lm_head_weight(w, device=DEV)
    pre = prefix_inputs(w, device=DEV)
    pre["Qp"] = prefix_queries(w, device=DEV)
    steps = [step_inputs(w, 0, 0, t, device=DEV) for t in range(w.T)]
    mod = pre["modality"].cpu().numpy()
    counts = [(int((mod == 0).sum()), int((mod == 1).sum()))]

    def step_fn(t):
        x = steps[t]
        return {"Q": x["Q"][None].contiguous(), "Kb": x["Kb"][None].contiguous(),
                "Vb": x["Vb"][None].contiguous(), "h": x["h"], "theta": x["theta"]}

    out = []
    for pa in (True, False):
        dec = BlockDecoder(W, NL=w.NL, Hq=w.Hq, Hkv=w.Hkv, d=w.d, LB=w.LB, T=w.T, tau=w.tau,
                           r_text=w.r_text, r_img=w.r_img, modality_counts=counts,
                           prefix_attn=pa)
        res = dec.decode(pre, step_fn)
        torch.cuda.synchronize()
        assert dec.status.item() == 0
        out.append((res, dec))
    (ra, da), (rb, _) = out
    assert ra.steps == rb.steps and torch.equal(ra.tokens, rb.tokens)
    rows = [0, 1, 127, 128, 350, 699]
    want = orc.prefix_attention(pre["Qp"], pre["K"], pre["V"], rows=rows)
    got = gc.host(da.O_prefix.view(w.NL, 700, w.Hq, w.d))[:, rows]
    gc.assert_close(got, want, torch.bfloat16, "decoder O_prefix")


@pytest.mark.parametrize("pattern", ["ramp", "spikes"])
def test_row_maxima_moving_within_tiles(sp, pattern):
    """Prefix self-attention with keys whose scores climb through every key
    tile, or spike inside tiles, for every query (queries along one
    direction, keys scaled along it): the output must match the fp64 oracle
    whatever the order in which the row maxima appear."""
    NL, Hq, Hkv, d, n = 1, 2, 2, 128, 700
    g = generator(DEV, "prefix-attn-moving", 1)
    dirs = torch.randn((NL, 1, Hkv, d), generator=g, device=DEV)
    dirs = dirs / dirs.norm(dim=-1, keepdim=True)
    scale = torch.linspace(0.5, 1.5, n, device=DEV).view(1, n, 1, 1)
    Q = (dirs.repeat_interleave(Hq // Hkv, dim=2) * scale * 4.0).to(torch.bfloat16)
    i = torch.arange(n, device=DEV, dtype=torch.float32)
    if pattern == "ramp":
        a = 0.08 * i
    else:
        a = 0.3 * torch.randn(n, generator=g, device=DEV)
        for t0 in range(0, n, 128):
            for off, hgt in ((40, 6.0), (100, 12.0)):
                if t0 + off < n:
                    a[t0 + off] = hgt + t0 / 64.0
    K = (dirs * a.view(1, n, 1, 1) * (d ** 0.5)).to(torch.bfloat16)
    V = torch.randn((NL, n, Hkv, d), generator=g, device=DEV).to(torch.bfloat16)
    off = [0, n]
    Op = _run(sp, [Q.reshape(-1), K.reshape(-1), V.reshape(-1)], off, NL, Hq, Hkv, d)
    want = orc.prefix_attention(Q, K, V)
    got = gc.host(Op.view(NL, n, Hq, d))
    gc.assert_close(got, want, torch.bfloat16, pattern)
