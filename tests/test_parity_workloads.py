"""Whole-block decodes of the batched and the sequential workloads, checked
stage by stage against the oracle.

* batch-16x8k: 16 independent sequences of 8192 prefix positions with ragged
  image fractions, decoded together at unmask thresholds 0.7, 0.9 and 0.95;
* sequential-64-blocks: blocks 0 and 63 of a 64-block decode whose prefix
  grows from 2048 to 4064 positions (1024 image, then text).

Stage-wise: each stage is compared with the oracle given the GPU's own
inputs to that stage (prefix confidences on sampled rows; kept set from the
GPU's confidences; attention over the GPU's kept set; unmask decisions from
the GPU's block confidences), so errors do not compound.  The native step
driver and the call-per-step path must give the same tokens.
"""
import numpy as np
import pytest
import torch

from oracle import sprint_oracle as orc
from tests import gpu_cases as gc
from workload import WORKLOADS, lm_head_weight, prefix_inputs, step_inputs

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def sp():
    from kv_cache_pruning_step_b300 import sprint
    return sprint


_WEIGHTS = {}


def weights_of(name):
    """The workload's LM-head weight on the device and as an exact fp64 host
    copy for the oracle (made once per workload)."""
    if name not in _WEIGHTS:
        _WEIGHTS.clear()
        W = lm_head_weight(WORKLOADS[name], device=DEV)
        _WEIGHTS[name] = (W, gc.host(W).astype(np.float64))
    return _WEIGHTS[name]


def _decode_and_check(sp, w, weights, prefixes, step_sets, check_seqs, tau, indexed=False):
    W, W64 = weights
    from kv_cache_pruning_step_b300 import BlockDecoder
    S = len(prefixes)
    cat = gc.concat_prefixes(prefixes)
    counts = [(int((p["modality"] == 0).sum()), int((p["modality"] != 0).sum()))
              for p in prefixes]
    steps = []
    for t in range(w.T):
        xs = [step_sets[s][t] for s in range(S)]
        steps.append({k: (torch.stack([x[k] for x in xs]) if k in ("Q", "Kb", "Vb")
                          else torch.cat([x[k] for x in xs])).contiguous()
                      for k in ("Q", "Kb", "Vb", "h", "theta")})

    def make():
        return BlockDecoder(W, NL=w.NL, Hq=w.Hq, Hkv=w.Hkv, d=w.d, LB=w.LB, T=w.T, tau=tau,
                            r_text=w.r_text, r_img=w.r_img, alpha=w.alpha,
                            modality_counts=counts, indexed=indexed)

    native = make()
    r_native = native.decode(cat, lambda t: steps[t])
    seen = []

    def on_step(t, d):
        seen.append({"O": d.O.float().cpu(), "conf": d.conf_blk.cpu().numpy(),
                     "argmax": d.argmax_blk.cpu().numpy(), "acc": d.accepted.cpu().numpy()})

    dec = make()
    res = dec.decode(cat, lambda t: steps[t], on_step=on_step)
    torch.cuda.synchronize()
    assert native.status.item() == 0 and dec.status.item() == 0
    assert torch.equal(r_native.tokens, res.tokens) and r_native.steps == res.steps

    conf_prefix = dec.conf_prefix.cpu().numpy()
    kept = dec.kept_idx.cpu().numpy()
    off, koff = dec.prefix_off_host, dec.kept_off_host
    rng = np.random.default_rng(5)
    for s in check_seqs:
        p = prefixes[s]
        n = off[s + 1] - off[s]
        mod = p["modality"].cpu().numpy()
        # (a) prefix confidences on sampled rows
        rows = np.sort(rng.choice(n, size=min(24, n), replace=False))
        gc.check_confidence(conf_prefix[off[s]:off[s + 1]][rows], None,
                            p["H"], W64, p["theta"], rows, f"seq {s} prefix")
        # (b) kept set from the GPU's confidences
        score_o = orc.composite_score(orc.key_norm_importance(p["K"]),
                                      conf_prefix[off[s]:off[s + 1]], w.alpha)
        kept_s = kept[koff[s]:koff[s + 1]]
        gc.check_kept(kept_s, score_o, mod, w.r_text, w.r_img, f"seq {s}")
        # (c) attention of step 1 over the GPU's kept set, first and last layer
        if len(seen) > 1:
            x = step_sets[s][1]
            want = orc.block_attention(x["Q"], orc.compact(p["K"], kept_s),
                                       orc.compact(p["V"], kept_s), x["Kb"], x["Vb"],
                                       layers=[0, w.NL - 1])
            for layer in (0, w.NL - 1):
                gc.assert_close(seen[1]["O"][s, layer].numpy(), want[layer], w.torch_dtype,
                                f"seq {s} step 1 layer {layer}")
        # (d) block confidences of step 0, (e) every unmask decision
        rs = slice(s * w.LB, (s + 1) * w.LB)
        x0 = step_sets[s][0]
        gc.check_confidence(seen[0]["conf"][rs], seen[0]["argmax"][rs], x0["h"], W64,
                            x0["theta"], np.arange(w.LB), f"seq {s} step 0")
        mask = np.ones(w.LB, bool)
        tokens = np.full(w.LB, -1)
        for t, g in enumerate(seen):
            mask, tokens, acc = orc.unmask_step(g["conf"][rs], g["argmax"][rs], mask, tokens,
                                                t, w.T, tau)
            assert g["acc"][s].astype(bool).tolist() == acc.tolist(), f"seq {s} step {t}"
        assert res.tokens[s].cpu().numpy().tolist() == tokens.tolist()
        assert not mask.any()  # every block ends within T steps
    return res


@pytest.mark.parametrize("tau,indexed", [(0.7, False), (0.9, False), (0.93, False),
                                         (0.95, False), (0.9, True)])
def test_batch_16x8k_threshold_sweep(sp, tau, indexed):
    """tau sweep of the batched workload (0.93 is the paper's own setting);
    at 0.9 also with the later steps reading the kept rows through indices."""
    w = WORKLOADS["batch-16x8k"]
    prefixes = [prefix_inputs(w, seq=s, device=DEV) for s in range(w.S)]
    step_sets = [[step_inputs(w, s, 0, t, device=DEV) for t in range(w.T)] for s in range(w.S)]
    res = _decode_and_check(sp, w, weights_of(w.name), prefixes, step_sets, check_seqs=[0, 11],
                            tau=tau, indexed=indexed)
    assert res.steps <= w.T


@pytest.mark.parametrize("block", [0, 63])
def test_sequential_blocks(sp, block):
    w = WORKLOADS["sequential-64-blocks"]
    pre = prefix_inputs(w, seq=0, block=block, device=DEV)
    assert pre["modality"].numel() == 2048 + 32 * block
    # the cache grows by appending: block b's prefix starts with block 0's
    first = prefix_inputs(w, seq=0, block=0, device=DEV)
    assert torch.equal(pre["K"][:, :2048], first["K"])
    step_sets = [[step_inputs(w, 0, block, t, device=DEV) for t in range(w.T)]]
    _decode_and_check(sp, w, weights_of(w.name), [pre], step_sets, check_seqs=[0], tau=w.tau)


def test_sequential_prefix_confidence_cache_is_bit_exact(sp):
    """Block b+1's prefix is block b's plus the rows generated in between:
    reusing block b's prefix confidences and sending only the new rows
    through the LM head (together with the block's step-0 rows) gives
    bit-identical confidences, kept set and decoded tokens."""
    from kv_cache_pruning_step_b300 import BlockDecoder
    w = WORKLOADS["sequential-64-blocks"]
    W, _ = weights_of(w.name)

    def counts(p):
        m = p["modality"]
        return [(int((m == 0).sum()), int((m != 0).sum()))]

    def steps_of(block):
        xs = [step_inputs(w, 0, block, t, device=DEV) for t in range(w.T)]
        return lambda t: {"Q": xs[t]["Q"][None].contiguous(), "Kb": xs[t]["Kb"][None].contiguous(),
                          "Vb": xs[t]["Vb"][None].contiguous(), "h": xs[t]["h"],
                          "theta": xs[t]["theta"]}

    b = 20
    pre_a = prefix_inputs(w, seq=0, block=b, device=DEV)
    pre_b = prefix_inputs(w, seq=0, block=b + 1, device=DEV)
    n_a = pre_a["modality"].numel()

    def make(c):
        return BlockDecoder(W, NL=w.NL, Hq=w.Hq, Hkv=w.Hkv, d=w.d, LB=w.LB, T=w.T, tau=w.tau,
                            r_text=w.r_text, r_img=w.r_img, alpha=w.alpha, modality_counts=c)
    dec = make(counts(pre_a))
    dec.decode(pre_a, steps_of(b))
    dec.set_prefix(counts(pre_b))  # grows: old confidences are kept
    cached = dec.decode(pre_b, steps_of(b + 1), conf_from=n_a)
    fresh_dec = make(counts(pre_b))
    fresh = fresh_dec.decode(pre_b, steps_of(b + 1))
    torch.cuda.synchronize()
    assert dec.status.item() == 0 and fresh_dec.status.item() == 0
    assert torch.equal(dec.conf_prefix, fresh_dec.conf_prefix)
    assert torch.equal(dec.kept_idx, fresh_dec.kept_idx)
    assert cached.steps == fresh.steps and torch.equal(cached.tokens, fresh.tokens)
    # the cached decode ran step 0's block LM head within the prefix call
    assert cached.accepted_per_step == fresh.accepted_per_step


def test_sequential_blocks_enqueued_without_waiting(sp):
    """Consecutive blocks of one sequence enqueued with decode(wait=False)
    (set_prefix between them copies its tables without waiting for the GPU)
    decode exactly as the same blocks decoded one at a time."""
    from kv_cache_pruning_step_b300 import BlockDecoder
    w = WORKLOADS["sequential-64-blocks"]
    W, _ = weights_of(w.name)
    blocks = [30, 31, 32, 33]
    pres = [prefix_inputs(w, seq=0, block=b, device=DEV) for b in blocks]
    counts = [[(int((p["modality"] == 0).sum()), int((p["modality"] != 0).sum()))] for p in pres]
    xss = [[step_inputs(w, 0, b, t, device=DEV) for t in range(w.T)] for b in blocks]

    def steps_of(i):
        xs = xss[i]
        return lambda t: {"Q": xs[t]["Q"][None].contiguous(), "Kb": xs[t]["Kb"][None].contiguous(),
                          "Vb": xs[t]["Vb"][None].contiguous(), "h": xs[t]["h"],
                          "theta": xs[t]["theta"]}

    def make():
        return BlockDecoder(W, NL=w.NL, Hq=w.Hq, Hkv=w.Hkv, d=w.d, LB=w.LB, T=w.T, tau=w.tau,
                            r_text=w.r_text, r_img=w.r_img, alpha=w.alpha,
                            modality_counts=counts[-1])

    def run(wait):
        dec = make()
        out, pend, prev = [], [], 0
        for i in range(len(blocks)):
            dec.set_prefix(counts[i])
            r = dec.decode(pres[i], steps_of(i), conf_from=prev, wait=wait)
            # the live token buffer is the next block's: copy it on the stream
            out.append([r, dec.tokens.clone(), dec.conf_prefix.clone(), dec.kept_idx.clone()])
            prev = dec.total_rows
        res = [dec.finish(r) if not wait else r for r, *_ in out]
        torch.cuda.synchronize()
        assert dec.status.item() == 0
        return [(r.steps, r.accepted_per_step, tok, conf, kept)
                for r, (_, tok, conf, kept) in zip(res, out)]

    a, b = run(True), run(False)
    for i, (x, y) in enumerate(zip(a, b)):
        assert x[0] == y[0] and x[1] == y[1], f"block {blocks[i]}"
        for u, v in zip(x[2:], y[2:]):
            assert torch.equal(u, v), f"block {blocks[i]}"
