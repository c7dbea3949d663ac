"""GPU parity of sprint_unmask and of whole-block decoding against the oracle."""
import json
import os

import numpy as np
import pytest
import torch

from oracle import sprint_oracle as orc
from tests import gpu_cases as gc
from workload import WORKLOADS, lm_head_weight, prefix_inputs, small_workload, step_inputs

pytestmark = pytest.mark.gpu
DEV = "cuda"
GOLD = os.path.join(os.path.dirname(__file__), "golden")


@pytest.fixture(scope="module")
def sp():
    from kv_cache_pruning_step_b300 import sprint
    return sprint


def test_golden_cases(sp):
    cases = json.load(open(os.path.join(GOLD, "unmask_hand.json")))["cases"]
    for case in cases:
        mode = sp.UNMASK_FIXED if case["mode"] == "fixed" else sp.UNMASK_ADAPTIVE
        LB = len(case["conf"])
        conf = torch.tensor([case["conf"]], dtype=torch.float32, device=DEV)
        am = torch.arange(100, 100 + LB, dtype=torch.int32, device=DEV)[None]
        mask = torch.tensor([case["mask"]], dtype=torch.uint8, device=DEV)
        tokens = torch.full((1, LB), -1, dtype=torch.int32, device=DEV)
        m, acc = sp.sprint_unmask(conf, am, mask, tokens, case["t"], case["T"], case["tau"], mode)
        got = torch.nonzero(acc[0]).flatten().tolist()
        assert got == case["expected_accepted"], case
        assert m.item() == sum(case["mask"]) - len(got)
        for j in got:
            assert tokens[0, j].item() == 100 + j and mask[0, j].item() == 0


@pytest.mark.parametrize("mode", [0, 1])
@pytest.mark.parametrize("LB,T", [(32, 8), (32, 4), (7, 3), (1, 1), (100, 5), (1024, 9)])
def test_random_trajectories_match_oracle(sp, mode, LB, T):
    S = 6
    g = torch.Generator().manual_seed(LB * 31 + T)
    mask = torch.ones((S, LB), dtype=torch.uint8, device=DEV)
    tokens = torch.full((S, LB), -1, dtype=torch.int32, device=DEV)
    o_mask = [np.ones(LB, bool) for _ in range(S)]
    o_tok = [np.full(LB, -1) for _ in range(S)]
    for t in range(T):
        # coarse confidences: ties and values at tau are frequent
        conf = (torch.randint(0, 21, (S, LB), generator=g).float() / 20).to(DEV)
        am = torch.randint(0, 50000, (S, LB), generator=g, dtype=torch.int32).to(DEV)
        tau = [0.9, 0.95, 0.5, 1.0][t % 4]
        m, acc = sp.sprint_unmask(conf, am, mask, tokens, t, T, tau, mode)
        for s in range(S):
            o_mask[s], o_tok[s], o_acc = orc.unmask_step(conf[s].cpu().numpy(), am[s].cpu().numpy(),
                                                         o_mask[s], o_tok[s], t, T, tau, mode)
            assert acc[s].cpu().numpy().astype(bool).tolist() == o_acc.tolist()
            assert mask[s].cpu().numpy().astype(bool).tolist() == o_mask[s].tolist()
            assert tokens[s].cpu().numpy().tolist() == o_tok[s].tolist()
            assert m[s].item() == int(o_mask[s].sum())
    if mode == 0:
        assert int(mask.sum()) == 0  # terminates within T


def _check_block_stagewise(w, W, pre, steps, seen, ref, gpu_tokens, residual=False):
    """Compare every step of a GPU block decode stage by stage: the oracle's
    attention on the step's inputs (full prefix at step 0, the prefix pruned
    by the GPU's kept set afterwards); the oracle's confidences and greedy
    tokens on the step's LM-head input (h + the GPU's O with the residual
    chain); and the oracle's unmask rule applied to the GPU's own
    confidences, greedy tokens and mask state, which must give the GPU's
    decisions and state exactly.  The whole-block oracle trajectory is also
    followed while the decisions agree; the GPU may leave it only at a step
    where a confidence lies within CONF_ATOL of tau, and then the remaining
    steps are still compared stage by stage."""
    kept = seen[0]["kept"]
    Kp, Vp = orc.compact(pre["K"], kept), orc.compact(pre["V"], kept)
    mask = np.ones(w.LB, dtype=bool)
    tokens = np.full(w.LB, -1, dtype=np.int64)
    follows = True
    rows = np.arange(w.LB)
    for t, g in enumerate(seen):
        x = steps[t]
        Kt, Vt = (pre["K"], pre["V"]) if t == 0 else (Kp, Vp)
        O = orc.block_attention(x["Q"], Kt, Vt, x["Kb"], x["Vb"])
        gc.assert_close(g["O"], O, torch.float32, f"step {t} O")
        h = orc.residual_hidden(x["h"], g["O"]) if residual else gc.host(x["h"])
        gc.check_confidence(g["conf"], g["argmax"], h, W, x["theta"], rows, f"step {t}")
        mask, tokens, acc = orc.unmask_step(g["conf"], g["argmax"], mask, tokens, t, w.T, w.tau)
        assert acc.tolist() == g["acc"].astype(bool).tolist(), f"step {t}: unmask decisions"
        assert mask.tolist() == g["mask"].astype(bool).tolist(), f"step {t}: mask"
        assert tokens.tolist() == g["tokens"].astype(np.int64).tolist(), f"step {t}: tokens"
        if follows:
            r = ref["steps"][t]
            if r["accepted"].tolist() != acc.tolist():
                near = np.abs(r["conf"] - w.tau) <= gc.CONF_ATOL
                assert near.any(), f"step {t}: decisions leave the oracle's trajectory"
                follows = False
    assert not mask.any(), "the block must be unmasked within T steps"
    assert np.asarray(gpu_tokens).tolist() == tokens.tolist()
    if follows:
        assert len(seen) == len(ref["steps"])
        assert tokens.tolist() == ref["tokens"].tolist()
    return follows


@pytest.mark.parametrize("indexed", [False, True])
def test_tiny_block_end_to_end(sp, indexed):
    """Whole block on the fp32 tiny workload, every step compared (later
    steps over the compacted cache, or over the full cache through the kept
    indices)."""
    from kv_cache_pruning_step_b300 import BlockDecoder
    w = WORKLOADS["tiny-256"]
    W = lm_head_weight(w, device=DEV)
    pre = prefix_inputs(w, device=DEV)
    steps = [step_inputs(w, 0, 0, t, device=DEV) for t in range(w.T)]
    mod = pre["modality"].cpu().numpy()
    counts = [(int((mod == 0).sum()), int((mod == 1).sum()))]
    dec = BlockDecoder(W, NL=w.NL, Hq=w.Hq, Hkv=w.Hkv, d=w.d, LB=w.LB, T=w.T, tau=w.tau,
                       r_text=w.r_text, r_img=w.r_img, alpha=w.alpha, modality_counts=counts,
                       want_logits=True, indexed=indexed)
    seen = []

    def on_step(t, d):
        seen.append({"O": gc.host(d.O[0]), "conf": d.conf_blk.cpu().numpy(),
                     "argmax": d.argmax_blk.cpu().numpy(), "acc": d.accepted[0].cpu().numpy(),
                     "mask": d.mask[0].cpu().numpy(), "tokens": d.tokens[0].cpu().numpy(),
                     "kept": d.kept_idx.cpu().numpy(), "score": d.score.cpu().numpy(),
                     "conf_prefix": d.conf_prefix.cpu().numpy()})

    def step_fn(t):
        x = steps[t]
        return {"Q": x["Q"][None].contiguous(), "Kb": x["Kb"][None].contiguous(),
                "Vb": x["Vb"][None].contiguous(), "h": x["h"], "theta": x["theta"]}

    res = dec.decode({**pre, "modality": pre["modality"]}, step_fn, on_step=on_step)
    torch.cuda.synchronize()
    assert dec.status.item() == 0
    ref = orc.decode_block(pre, lambda t: steps[t], W, LB=w.LB, T=w.T, tau=w.tau,
                           r_text=w.r_text, r_img=w.r_img, alpha=w.alpha)
    # step-0 scoring: confidences, scores, kept set
    assert np.abs(seen[0]["conf_prefix"] - ref["prefix_conf"]).max() <= gc.CONF_ATOL
    assert np.abs(seen[0]["score"] - ref["score"]).max() <= gc.SCORE_EXCUSE
    gc.check_kept(seen[0]["kept"], ref["score"], mod, w.r_text, w.r_img, "tiny kept")
    assert res.steps == len(seen)
    _check_block_stagewise(w, W, pre, steps, seen, ref, res.tokens[0].cpu().numpy())


def _decoder_and_steps(name, tau=None, mode=0):
    from kv_cache_pruning_step_b300 import BlockDecoder
    w = WORKLOADS[name] if isinstance(name, str) else name
    W = lm_head_weight(w, device=DEV)
    pre = prefix_inputs(w, device=DEV)
    mod = pre["modality"].cpu().numpy()
    counts = [(int((mod == 0).sum()), int((mod == 1).sum()))]
    steps = []
    for t in range(w.T):
        x = step_inputs(w, 0, 0, t, device=DEV)
        steps.append({"Q": x["Q"][None].contiguous(), "Kb": x["Kb"][None].contiguous(),
                      "Vb": x["Vb"][None].contiguous(), "h": x["h"], "theta": x["theta"]})

    def make(indexed=False):
        return BlockDecoder(W, NL=w.NL, Hq=w.Hq, Hkv=w.Hkv, d=w.d, LB=w.LB, T=w.T,
                            tau=w.tau if tau is None else tau, r_text=w.r_text, r_img=w.r_img,
                            alpha=w.alpha, mode=mode, modality_counts=counts, indexed=indexed)
    return w, pre, steps, make


@pytest.mark.parametrize("name,mode", [("tiny-256", 0), ("tiny-256", 1), ("prefix-4k", 0)])
def test_native_step_driver_matches_stepwise(sp, name, mode):
    """sprint_decode_steps (all steps enqueued at once, gated on the device)
    gives the same trajectory as issuing the five calls step by step."""
    w, pre, steps, make = _decoder_and_steps(name, mode=mode)
    a, b = make(), make()
    a.timing, b.timing = {}, {}  # stage events recorded on both paths
    ra = a.decode(pre, lambda t: steps[t])
    rb = b.decode_stepwise(pre, lambda t: steps[t])
    torch.cuda.synchronize()
    for tm, n in ((a.timing, ra.steps), (b.timing, rb.steps)):
        assert len(tm["lmhead_block"]) == n and len(tm["unmask"]) == n
        assert len(tm["lmhead_prefix"]) == 1 and all(v > 0 for v in tm["lmhead_block"])
    assert a.status.item() == 0 and b.status.item() == 0
    assert ra.steps == rb.steps
    assert ra.accepted_per_step == rb.accepted_per_step
    assert torch.equal(ra.tokens, rb.tokens)
    assert torch.equal(a.O, b.O)
    assert torch.equal(a.conf_blk, b.conf_blk)


def test_native_step_driver_block_of_several_row_tiles(sp):
    """A block of 100 positions: the fused fold-and-unmask kernel (one
    cluster per sequence) loops over four tiles of 32 rows; the trajectory
    equals the stepwise one bit for bit."""
    w = small_workload("lb-fuzz", dtype="bf16", NL=2, Hq=2, Hkv=2, d=64, D=256, V=3000, LB=100,
                       T=5, n=300, n_img=100, seed=100)
    w, pre, steps, make = _decoder_and_steps(w)
    a, b = make(), make()
    ra = a.decode(pre, lambda t: steps[t])
    rb = b.decode_stepwise(pre, lambda t: steps[t])
    torch.cuda.synchronize()
    assert a.status.item() == 0 and b.status.item() == 0
    assert ra.steps == rb.steps and ra.accepted_per_step == rb.accepted_per_step
    assert sum(int(x[0]) for x in ra.accepted_per_step) == w.LB
    assert torch.equal(ra.tokens, rb.tokens)
    assert torch.equal(a.conf_blk, b.conf_blk)


def test_native_step_driver_4096_block_rows(sp):
    """128 sequences of 32 positions, 4096 block rows: above the fused
    kernel's row limit the driver runs the LM head's own combine and then
    the unmask kernel.  The trajectory equals the stepwise one bit for bit."""
    from kv_cache_pruning_step_b300 import BlockDecoder
    S = 128
    w = small_workload("rows-4096", dtype="bf16", NL=2, Hq=4, Hkv=2, d=64, D=256, V=3000, LB=32,
                       T=4, n=64, n_img=16, seed=3, S=S)
    W = lm_head_weight(w, device=DEV)
    prefixes = [prefix_inputs(w, seq=s, device=DEV) for s in range(S)]
    cat = gc.concat_prefixes(prefixes)
    counts = [(int((p["modality"] == 0).sum()), int((p["modality"] != 0).sum()))
              for p in prefixes]
    steps = []
    for t in range(w.T):
        xs = [step_inputs(w, s, 0, t, device=DEV) for s in range(S)]
        steps.append({k: (torch.stack([x[k] for x in xs]) if k in ("Q", "Kb", "Vb")
                          else torch.cat([x[k] for x in xs])).contiguous()
                      for k in ("Q", "Kb", "Vb", "h", "theta")})

    def make():
        return BlockDecoder(W, NL=w.NL, Hq=w.Hq, Hkv=w.Hkv, d=w.d, LB=w.LB, T=w.T, tau=w.tau,
                            r_text=w.r_text, r_img=w.r_img, alpha=w.alpha,
                            modality_counts=counts)
    a, b = make(), make()
    ra = a.decode(cat, lambda t: steps[t])
    rb = b.decode_stepwise(cat, lambda t: steps[t])
    torch.cuda.synchronize()
    assert a.status.item() == 0 and b.status.item() == 0
    assert ra.steps == rb.steps and ra.accepted_per_step == rb.accepted_per_step
    assert all(sum(int(x[s]) for x in ra.accepted_per_step) == w.LB for s in range(S))
    assert torch.equal(ra.tokens, rb.tokens)
    assert torch.equal(a.conf_blk, b.conf_blk)


def test_overlapped_key_norms_match_one_call(sp):
    """The default prefix pass (key norms on a side stream under the prefix
    LM head, then the selection on them) and one sprint_score_prune call
    after the LM head give the same scores, kept set and tokens."""
    from kv_cache_pruning_step_b300 import BlockDecoder
    w, pre, steps, _ = _decoder_and_steps("prefix-4k")
    W = lm_head_weight(w, device=DEV)
    mod = pre["modality"].cpu().numpy()
    counts = [(int((mod == 0).sum()), int((mod == 1).sum()))]
    res = []
    for overlap in (True, False):
        dec = BlockDecoder(W, NL=w.NL, Hq=w.Hq, Hkv=w.Hkv, d=w.d, LB=w.LB, T=w.T, tau=w.tau,
                           r_text=w.r_text, r_img=w.r_img, alpha=w.alpha,
                           modality_counts=counts, overlap_keynorm=overlap)
        r = dec.decode(pre, lambda t: steps[t])
        torch.cuda.synchronize()
        assert dec.status.item() == 0
        res.append((dec.score.clone(), dec.kept_idx.clone(), r.tokens.clone()))
    for a, b in zip(*res):
        assert torch.equal(a, b)


def test_native_step_driver_captured_in_a_cuda_graph(sp):
    """sprint_decode_steps captured into a CUDA graph from the caller's
    stream, the attention combines on the library's side stream included,
    and replayed: the same attention output, tokens and masked counts as
    the direct call."""
    w, pre, steps, make = _decoder_and_steps("prefix-4k")
    dec = make()
    r = dec.decode(pre, lambda t: steps[t])
    torch.cuda.synchronize()
    O_ref, tok_ref, m_ref = dec.O.clone(), r.tokens.clone(), dec.m_hist.clone()
    xs = steps
    args = dict(
        Q=[x["Q"] for x in xs], Kb=[x["Kb"] for x in xs], Vb=[x["Vb"] for x in xs],
        h=[x["h"] for x in xs], theta=[x.get("theta") for x in xs],
        Kf=pre["K"], Vf=pre["V"], prefix_off=dec.prefix_off, max_rows=dec.max_rows,
        total_rows=dec.total_rows, Kp=dec.Kp, Vp=dec.Vp, kept_off=dec.kept_off,
        max_kept=dec.max_kept, total_kept=dec.total_kept, W=dec.W, T=dec.T, tau=dec.tau,
        mode=dec.mode, O=dec.O, conf=dec.conf_blk, argmax=dec.argmax_blk, mask=dec.mask,
        tokens=dec.tokens, m_hist=dec.m_hist, ws_attn=dec.ws_attn, ws_lm=dec.ws_lm_blk,
        status=dec.status)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        sp.sprint_decode_steps(**args)
    dec.O.zero_()
    dec.tokens.fill_(-7)
    dec.m_hist.fill_(-7)
    g.replay()
    torch.cuda.synchronize()
    assert dec.status.item() == 0
    assert torch.equal(dec.O, O_ref)
    assert torch.equal(dec.tokens, tok_ref)
    assert torch.equal(dec.m_hist, m_ref)


def test_native_step_driver_skips_steps_after_the_block_is_done(sp):
    """tau below every confidence: step 0 accepts all LB positions, and the
    kernels of steps 1..T-1 return without touching any output."""
    w, pre, steps, make = _decoder_and_steps("tiny-256", tau=-1.0)
    a, b = make(), make()
    ra = a.decode(pre, lambda t: steps[t])
    rb = b.decode_stepwise(pre, lambda t: steps[t])
    torch.cuda.synchronize()
    assert ra.steps == rb.steps == 1
    assert ra.accepted_per_step == [[w.LB]]
    assert torch.equal(ra.tokens, rb.tokens)
    assert a.m_hist.cpu().tolist() == [[0]] * w.T
    # outputs still hold step 0's values: steps 1..T-1 did not run
    assert torch.equal(a.O, b.O) and torch.equal(a.conf_blk, b.conf_blk)


def test_pipelined_blocks_match_waiting_decode(sp):
    """decode(wait=False) lets the next block be enqueued before a block's
    step counts are read; results equal the waiting decode's."""
    w, pre, steps, make = _decoder_and_steps("tiny-256")
    a, b = make(), make()
    ref = a.decode(pre, lambda t: steps[t])
    ref_tokens = ref.tokens.clone()
    p1 = b.decode(pre, lambda t: steps[t], wait=False)
    t1 = p1.tokens.clone()  # stream-ordered copy before the next block
    p2 = b.decode(pre, lambda t: steps[t], wait=False)
    r1, r2 = b.finish(p1), b.finish(p2)
    torch.cuda.synchronize()
    assert r1.steps == r2.steps == ref.steps
    assert r1.accepted_per_step == r2.accepted_per_step == ref.accepted_per_step
    assert torch.equal(t1, ref_tokens) and torch.equal(b.tokens, ref_tokens)
    assert b.finish(p1) is r1  # finishing twice returns the same result


@pytest.mark.parametrize("name", ["tiny-256", "prefix-4k"])
def test_indexed_layout_matches_compacted(sp, name):
    """Later steps reading the kept rows through their indices give the same
    block, bit for bit, as the compacted cache: native driver and stepwise."""
    w, pre, steps, make = _decoder_and_steps(name)
    a, b, c = make(), make(indexed=True), make(indexed=True)
    ra = a.decode(pre, lambda t: steps[t])
    rb = b.decode(pre, lambda t: steps[t])
    outs = []
    rc = c.decode_stepwise(pre, lambda t: steps[t],
                           on_step=lambda t, d: outs.append(d.O.clone()))
    torch.cuda.synchronize()
    assert a.status.item() == b.status.item() == c.status.item() == 0
    assert b.Kp is None and b.Vp is None  # no compacted copy was made
    assert ra.steps == rb.steps == rc.steps
    assert ra.accepted_per_step == rb.accepted_per_step == rc.accepted_per_step
    assert torch.equal(ra.tokens, rb.tokens) and torch.equal(ra.tokens, rc.tokens)
    assert torch.equal(a.O, b.O) and torch.equal(a.O, outs[-1])
    assert torch.equal(a.conf_blk, b.conf_blk)


def test_tiny_block_residual_chain_end_to_end(sp):
    """Residual chain on the fp32 tiny workload: the LM head reads h + O of
    the last layer; every step's attention output, confidences and unmask
    decisions are compared with the oracle's chained decode."""
    from kv_cache_pruning_step_b300 import BlockDecoder
    w = WORKLOADS["tiny-256"]
    W = lm_head_weight(w, device=DEV)
    pre = prefix_inputs(w, device=DEV)
    steps = [step_inputs(w, 0, 0, t, device=DEV) for t in range(w.T)]
    mod = pre["modality"].cpu().numpy()
    counts = [(int((mod == 0).sum()), int((mod == 1).sum()))]
    dec = BlockDecoder(W, NL=w.NL, Hq=w.Hq, Hkv=w.Hkv, d=w.d, LB=w.LB, T=w.T, tau=w.tau,
                       r_text=w.r_text, r_img=w.r_img, alpha=w.alpha, modality_counts=counts,
                       residual=True)
    seen = []

    def on_step(t, d):
        seen.append({"O": gc.host(d.O[0]), "conf": d.conf_blk.cpu().numpy(),
                     "argmax": d.argmax_blk.cpu().numpy(), "acc": d.accepted[0].cpu().numpy(),
                     "mask": d.mask[0].cpu().numpy(), "tokens": d.tokens[0].cpu().numpy(),
                     "kept": d.kept_idx.cpu().numpy(), "h": gc.host(d.h_res)})

    def step_fn(t):
        x = steps[t]
        return {"Q": x["Q"][None].contiguous(), "Kb": x["Kb"][None].contiguous(),
                "Vb": x["Vb"][None].contiguous(), "h": x["h"], "theta": x["theta"]}

    res = dec.decode(pre, step_fn, on_step=on_step)
    torch.cuda.synchronize()
    assert dec.status.item() == 0
    ref = orc.decode_block(pre, lambda t: steps[t], W, LB=w.LB, T=w.T, tau=w.tau,
                           r_text=w.r_text, r_img=w.r_img, alpha=w.alpha, residual=True)
    assert res.steps == len(seen)
    for t, g in enumerate(seen):
        # h = h_in + O from the GPU's own O, and the chain changes the input
        want_h = orc.residual_hidden(steps[t]["h"], g["O"])
        np.testing.assert_allclose(g["h"], want_h, rtol=1e-6, atol=1e-6)
        assert np.abs(g["h"] - gc.host(steps[t]["h"])).max() > 1e-3
    _check_block_stagewise(w, W, pre, steps, seen, ref, res.tokens[0].cpu().numpy(),
                           residual=True)


@pytest.mark.parametrize("name", ["tiny-256", "prefix-4k"])
def test_residual_chain_native_matches_stepwise(sp, name):
    """The native driver's fused residual (in the attention's combine
    kernel) and the stepwise sprint_residual_hidden give the same block, bit
    for bit; the fused h equals h_in + O within one rounding of its type."""
    from kv_cache_pruning_step_b300 import BlockDecoder
    w, pre, steps, _ = _decoder_and_steps(name)
    W = lm_head_weight(w, device=DEV)
    mod = pre["modality"].cpu().numpy()
    counts = [(int((mod == 0).sum()), int((mod == 1).sum()))]

    def make():
        return BlockDecoder(W, NL=w.NL, Hq=w.Hq, Hkv=w.Hkv, d=w.d, LB=w.LB, T=w.T, tau=w.tau,
                            r_text=w.r_text, r_img=w.r_img, alpha=w.alpha,
                            modality_counts=counts, residual=True)
    a, b = make(), make()
    ra = a.decode(pre, lambda t: steps[t])
    rb = b.decode_stepwise(pre, lambda t: steps[t])
    torch.cuda.synchronize()
    assert a.status.item() == 0 and b.status.item() == 0
    assert ra.steps == rb.steps and ra.accepted_per_step == rb.accepted_per_step
    assert torch.equal(ra.tokens, rb.tokens)
    assert torch.equal(a.O, b.O) and torch.equal(a.h_res, b.h_res)
    assert torch.equal(a.conf_blk, b.conf_blk)
    last = ra.steps - 1
    want = orc.residual_hidden(steps[last]["h"], a.O[0])
    rtol = 1e-6 if w.dtype == "f32" else 2.0 ** -8
    np.testing.assert_allclose(gc.host(a.h_res), want, rtol=rtol, atol=1e-6)


def test_timing_of_selected_stages_only(sp):
    """timing_stages limits the recorded events (the native driver skips the
    others); the block decodes the same."""
    w, pre, steps, make = _decoder_and_steps("prefix-4k")
    a, b = make(), make()
    a.timing, a.timing_stages = {}, {"lmhead_block", "lmhead_prefix"}
    ra = a.decode(pre, lambda t: steps[t])
    rb = b.decode(pre, lambda t: steps[t])
    torch.cuda.synchronize()
    assert set(a.timing) == {"lmhead_block", "lmhead_prefix"}
    assert len(a.timing["lmhead_block"]) == ra.steps
    assert ra.steps == rb.steps and torch.equal(ra.tokens, rb.tokens)
