"""Block-decode driver of the SPRINT step: the host loop over denoising steps.

LLaDA2.0-Uni paper (arXiv 2604.20796), Inference section.  A block of LB
masked tokens is decoded in at most T steps.  Step 0 is the full forward
pass: the prefix rows' confidences are computed, every prefix position is
scored, the per-modality kept set is chosen and the pruned KV cache is
gathered; step 0 itself attends to the full prefix.  Every later step
attends to the pruned prefix.  Every step predicts the block's tokens and
unmasks a confidence-adaptive number of them.

The driver only sequences library calls and sizes buffers.  All buffers are
allocated once per decoder, so a decode call launches kernels and nothing
else.  decode() enqueues the prefix pass and then all T steps through the
library's native step driver (sprint_decode_steps): the GPU itself skips the
steps after the block is finished, and the host reads the per-step masked
counts once, after the block.  decode_stepwise() issues the five calls one
step at a time and reads the masked counts after every step (used when a
caller wants to look at each step's outputs).
"""
from __future__ import annotations

import contextlib
from dataclasses import dataclass

import torch

from . import sprint as sp


@dataclass
class BlockResult:
    steps: int                 # denoising steps executed (step 0 included)
    tokens: torch.Tensor       # [S][LB] int32 decoded tokens
    accepted_per_step: list    # per step: [S] accepted counts (host ints)


@dataclass
class PendingBlock:
    """A block enqueued by BlockDecoder.decode(wait=False)."""
    slot: int
    done: torch.cuda.Event     # recorded after the block's last work
    m_hist_host: torch.Tensor  # pinned [T][S] masked counts, valid after `done`
    step_events: list          # 6 * T timing events, or None
    stage_events: list         # (stage, start, end) of the prefix pass
    tokens: torch.Tensor       # live device token buffer of the decoder
    result: BlockResult = None
    step0_given: bool = False  # step 0's block LM head ran with the prefix rows


class BlockDecoder:
    """Buffers and call sequence for decoding blocks of S sequences.

    modality_counts[s] = (n_text, n_image) describes sequence s's prefix;
    set_prefix() re-targets the decoder to new counts (for a prefix that
    grows block by block) and decode(conf_from=...) reuses the confidences of
    prefix rows that did not change.

    indexed=True: no pruned copy of the cache is made; the steps after the
    first read the kept rows of the full cache through the kept indices
    (sprint_block_attn_indexed), with the same result.

    selection picks the keep pools (sprint_score_prune_pools for the last
    two): "modality" (the paper's: floor(r_text n) of the text and
    floor(r_img n) of the image positions), "per_image" (text at r_text and
    every image at r_img; pool_sizes[s] = [n_text, n_image_1, ...] and the
    prefix dict's "image" tensor gives each position's image number), or
    "global" (one pool, floor(r_global n) of all positions).

    prefix_argmax=True also stores the greedy token of every prefix row
    (self.argmax_prefix); scoring needs only the confidences, so by default
    the prefix LM head skips it.

    residual=True: each step's LM head reads h + O of the last layer (heads
    concatenated, Hq d = D) instead of h alone, so the attention output
    reaches the confidences; the native driver fuses the sum into the
    attention's combine kernel, the stepwise path calls
    sprint_residual_hidden.

    overlap_keynorm=True (default): the key norms of the scoring, which read
    every prefix key once (HBM-bound), run on a side stream while the prefix
    LM head (tensor-bound) computes the confidences, and the selection then
    runs on the key norms (sprint_key_norms + sprint_select_kept, the same
    bits as sprint_score_prune).  False: one sprint_score_prune call after
    the LM head.

    prefix_attn=True: step 0 also runs the prefix's own attention of the full
    forward pass (sprint_prefix_attn) on the prefix queries prefix["Qp"]
    ([NL][n][Hq][d] per sequence) into self.O_prefix.  The output feeds
    nothing downstream here (the backbone around it is not reproduced);
    the option puts that work into the timed step.
    """

    def __init__(self, W, *, NL, Hq, Hkv, d, LB, T, tau, r_text, r_img, alpha=0.5,
                 mode=sp.UNMASK_ADAPTIVE, modality_counts, want_logits=False, indexed=False,
                 selection="modality", r_global=0.5, pool_sizes=None, residual=False,
                 prefix_argmax=False, prefix_attn=False, overlap_keynorm=True):
        self.W = W
        self.dev = W.device
        self.dtype = W.dtype
        self.NL, self.Hq, self.Hkv, self.d = NL, Hq, Hkv, d
        self.LB, self.T, self.tau, self.mode = LB, T, tau, mode
        self.r_text, self.r_img, self.alpha = r_text, r_img, alpha
        self.indexed = bool(indexed)
        self.prefix_argmax = bool(prefix_argmax)
        if selection not in ("modality", "per_image", "global"):
            raise ValueError(f"unknown selection {selection!r}")
        self.selection, self.r_global = selection, r_global
        self.residual = bool(residual)
        self.prefix_attn = bool(prefix_attn)
        self.overlap_keynorm = bool(overlap_keynorm)
        if self.overlap_keynorm:
            self.side = torch.cuda.Stream(device=W.device)
            self._k_ready = torch.cuda.Event()
            self._u_ready = torch.cuda.Event()
        if self.residual and Hq * d != W.shape[1]:
            raise ValueError("the residual chain needs Hq * d == D")
        self.V, self.D = W.shape
        self.S = S = len(modality_counts)
        self.status = sp.new_status(self.dev)
        self._cap = {}  # capacity tensors of the prefix-sized buffers
        self.set_prefix(modality_counts, pool_sizes)
        dt = self._dt
        i32 = dict(dtype=torch.int32, device=self.dev)
        f32 = dict(dtype=torch.float32, device=self.dev)
        # per-step buffers
        self.O = torch.empty((S, NL, LB, Hq, d), dtype=self.dtype, device=self.dev)
        self.conf_blk = torch.empty(S * LB, **f32)
        self.argmax_blk = torch.empty(S * LB, **i32)
        self.logits = (torch.empty((S * LB, self.V), dtype=self.dtype, device=self.dev)
                       if want_logits else None)
        self.want_logits = want_logits
        self.ws_lm_blk = torch.empty(
            max(16, sp.sprint_lmhead_workspace_bytes(S * LB, self.D, self.V, dt)),
            dtype=torch.uint8, device=self.dev)
        self.h_res = (torch.empty((S * LB, self.D), dtype=self.dtype, device=self.dev)
                      if self.residual else None)
        self.mask = torch.empty((S, LB), dtype=torch.uint8, device=self.dev)
        self.tokens = torch.empty((S, LB), **i32)
        self.m_out = torch.empty(S, **i32)
        self.accepted = torch.empty((S, LB), dtype=torch.uint8, device=self.dev)
        self.m_host = torch.empty(S, dtype=torch.int32, pin_memory=True)
        self.m_hist = torch.empty((T, S), **i32)
        self.ev = torch.cuda.Event()
        # When a dict, every stage records (start, end) CUDA events on the
        # current stream; after the block the durations (ms) are appended to
        # timing[stage] (used by the benchmark).  timing_stages, when a set,
        # limits the events to those stages: an event between two kernels
        # keeps the second from launching before the first ends.
        self.timing = None
        self.timing_stages = None
        self._pending = []
        # Two slots for blocks decoded without waiting (decode(wait=False)).
        self._step_events = [None, None]
        self._m_hist_host = [torch.empty((T, S), dtype=torch.int32, pin_memory=True)
                             for _ in range(2)]
        self._done = [torch.cuda.Event(), torch.cuda.Event()]
        self._slots = [None, None]
        self._next_slot = 0

    def _buf(self, name, numel, dtype):
        """A contiguous view of `numel` elements of a buffer that only grows
        (a grown buffer keeps the old contents in its first elements, so the
        prefix confidences survive a longer prefix)."""
        t = self._cap.get(name)
        if t is None or t.numel() < numel:
            grown = torch.empty(max(int(numel), 1), dtype=dtype, device=self.dev)
            if t is not None:
                grown[:t.numel()].copy_(t)
            t = grown
            self._cap[name] = t
        return t[:numel]

    def _dev_ints(self, values):
        """An int32 device tensor of host ints, copied from pinned memory on
        the current stream without waiting for the GPU (a blocking copy
        from pageable memory would wait for every block still in flight)."""
        host = torch.tensor(values, dtype=torch.int32).pin_memory()
        return host.to(self.dev, non_blocking=True)

    def set_prefix(self, modality_counts, pool_sizes=None):
        """(Re)target the decoder to prefixes with these (n_text, n_image)
        counts per sequence (the number of sequences is fixed).  Buffers
        sized by the prefix grow when needed and are otherwise reused, so a
        prefix that grows block by block costs no reallocation once the
        largest has been seen."""
        if len(modality_counts) != self.S:
            raise ValueError("set_prefix keeps the number of sequences")
        S, NL, Hkv, d = self.S, self.NL, self.Hkv, self.d
        self.modality_counts = [tuple(c) for c in modality_counts]
        lens = [nt + ni for nt, ni in modality_counts]
        self.keep = None  # per-pool keep counts (pool selections)
        if self.selection == "modality":
            kept = [sp.sprint_keep_count(nt, self.r_text) + sp.sprint_keep_count(ni, self.r_img)
                    for nt, ni in modality_counts]
        else:
            if self.selection == "global":
                table = [[sp.sprint_keep_count(n, self.r_global)] for n in lens]
            else:
                if pool_sizes is None or len(pool_sizes) != S:
                    raise ValueError("per_image selection needs pool_sizes per sequence")
                if any(sum(ps) != n for ps, n in zip(pool_sizes, lens)):
                    raise ValueError("pool_sizes must add up to the prefix lengths")
                self.n_pools = max(len(ps) for ps in pool_sizes)
                table = [[sp.sprint_keep_count(int(c), self.r_text if p == 0 else self.r_img)
                          for p, c in enumerate(list(ps) + [0] * (self.n_pools - len(ps)))]
                         for ps in pool_sizes]
            self.n_pools = len(table[0])
            kept = [sum(row) for row in table]
            self.keep = self._dev_ints([c for row in table for c in row])
        self.prefix_off_host = [0]
        self.kept_off_host = [0]
        for n, k in zip(lens, kept):
            self.prefix_off_host.append(self.prefix_off_host[-1] + n)
            self.kept_off_host.append(self.kept_off_host[-1] + k)
        self.total_rows = self.prefix_off_host[-1]
        self.total_kept = self.kept_off_host[-1]
        self.max_rows = max(lens) if lens else 0
        self.max_kept = max(kept) if kept else 0
        self.prefix_off = self._dev_ints(self.prefix_off_host)
        self.kept_off = self._dev_ints(self.kept_off_host)
        dt = self._dt = sp.BF16 if self.dtype == torch.bfloat16 else sp.F32
        u8 = torch.uint8
        # step-0 prefix pass
        self.conf_prefix = self._buf("conf_prefix", self.total_rows, torch.float32)
        self.argmax_prefix = (self._buf("argmax_prefix", self.total_rows, torch.int32)
                              if self.prefix_argmax else None)
        self.ws_lm_prefix = self._buf(
            "ws_lm_prefix",
            max(16, sp.sprint_lmhead_workspace_bytes(self.total_rows, self.D, self.V, dt)), u8)
        self.kept_idx = self._buf("kept_idx", self.total_kept, torch.int32)
        self.score = self._buf("score", self.total_rows, torch.float32)
        self.u = self._buf("u", self.total_rows, torch.float32)
        ws_bytes = (sp.sprint_score_prune_workspace_bytes(S, self.total_rows)
                    if self.keep is None else
                    sp.sprint_score_prune_pools_workspace_bytes(S, self.total_rows, self.n_pools))
        self.ws_score = self._buf("ws_score", max(16, ws_bytes), u8)
        if self.selection == "global":
            self.zero_pool = self._buf("zero_pool", self.total_rows, u8)
            self.zero_pool.zero_()
        row = NL * Hkv * d
        if self.indexed:
            self.Kp = self.Vp = None
        else:
            self.Kp = self._buf("Kp", self.total_kept * row, self.dtype)
            self.Vp = self._buf("Vp", self.total_kept * row, self.dtype)
        self.ws_attn = self._buf(
            "ws_attn", max(16, sp.sprint_block_attn_workspace_bytes(
                S, NL, self.LB, self.Hq, Hkv, d, self.max_rows, dt)), u8)
        self.O_prefix = (self._buf("O_prefix", self.total_rows * NL * self.Hq * d, self.dtype)
                         if self.prefix_attn else None)

    def _timed(self, name):
        return self.timing is not None and (self.timing_stages is None
                                            or name in self.timing_stages)

    @contextlib.contextmanager
    def _stage(self, name):
        if not self._timed(name):
            yield
            return
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record()
        yield
        b.record()
        self._pending.append((name, a, b))

    def _flush_timing(self):
        """Durations of the stages recorded so far (their events are done)."""
        if self.timing is not None:
            for name, a, b in self._pending:
                self.timing.setdefault(name, []).append(a.elapsed_time(b))
        self._pending = []

    _STEP_STAGES = ("attn", "lmhead_block", "unmask")

    def _events_for_steps(self, slot):
        """6 * T timing events for the native step driver (one set per
        pending-block slot), created once; each is recorded once here so that
        its CUDA event exists.  Entries of stages not timed are None."""
        if self._step_events[slot] is None:
            evs = [torch.cuda.Event(enable_timing=True) for _ in range(6 * self.T)]
            for e in evs:
                e.record()
            self._step_events[slot] = evs
        evs = list(self._step_events[slot])
        for t in range(self.T):
            for k, name in enumerate(self._STEP_STAGES):
                full = "attn_full" if t == 0 else "attn_pruned"
                if not self._timed(full if name == "attn" else name):
                    evs[6 * t + 2 * k] = evs[6 * t + 2 * k + 1] = None
        return evs

    # -- the individual stages (each is one or two library calls) --------
    def prefix_pass(self, K, V, H, theta, modality, conf_from=0, image=None, step0=None,
                    Qp=None):
        """Step-0 scoring and pruning: confidences of every prefix row, the
        kept set, and the pruned cache (self.Kp / self.Vp; not made when the
        decoder reads the kept rows through their indices).

        conf_from > 0 (one sequence only): rows [0, conf_from) of H are the
        rows of the previous call's prefix, unchanged, whose confidences are
        still in self.conf_prefix; only rows [conf_from, n) go through the LM
        head.  A row's confidence depends on that row alone.  While the whole
        prefix stays below 4096 rows both ways of computing it use the same
        vocabulary strips and fold order, so the result is bit-identical;
        above that the full-prefix call folds wider strips and the two agree
        to rounding.

        step0 (with conf_from > 0): the block's step-0 inputs; the new prefix
        rows and the block's step-0 rows then go through one LM-head call
        (one pass over W instead of two), which fills self.conf_blk and
        self.argmax_blk for step 0 as well.  Returns True when it did."""
        r0 = int(conf_from)
        if r0:
            if self.S != 1 or not 0 < r0 <= self.total_rows:
                raise ValueError("conf_from needs one sequence and 0 < conf_from <= rows")
        if self.prefix_attn:
            if Qp is None:
                raise ValueError("prefix_attn needs the prefix queries prefix['Qp']")
            with self._stage("prefix_attn"):
                sp.sprint_prefix_attn(Qp, K, V, self.prefix_off, self.total_rows, self.NL,
                                      self.Hq, self.Hkv, self.d, Op=self.O_prefix,
                                      status=self.status)
        overlap = self.overlap_keynorm and self.total_rows > 0
        if overlap:
            self._k_ready.record()  # the prefix keys are ready on the current stream
        merged = False
        with self._stage("lmhead_prefix"):
            if r0 and step0 is not None and r0 < self.total_rows:
                merged = self._merged_lmhead(H, theta, r0, step0)
            if not merged and r0 < self.total_rows:
                sp.sprint_lmhead_confidence(
                    H[r0:], self.W, theta[r0:], conf=self.conf_prefix[r0:],
                    argmax=self.argmax_prefix[r0:] if self.prefix_argmax else None,
                    want_argmax=self.prefix_argmax, ws=self.ws_lm_prefix, status=self.status)
        if overlap:
            # launched after the LM head, so its CTAs find the GEMM's already
            # resident and fill the room beside them
            with torch.cuda.stream(self.side):
                self.side.wait_event(self._k_ready)
                with self._stage("keynorm"):
                    sp.sprint_key_norms(K, self.prefix_off, self.total_rows, self.NL,
                                        self.Hkv, self.d, u=self.u, status=self.status)
                self._u_ready.record(self.side)
            torch.cuda.current_stream().wait_event(self._u_ready)
        with self._stage("score_prune"):
            pool = None
            if self.keep is not None:
                pool = self.zero_pool if self.selection == "global" else image
                if pool is None:
                    raise ValueError("per_image selection needs the prefix's image numbers")
            if self.keep is None and overlap:
                sp.sprint_select_kept(self.u, self.prefix_off, self.total_rows,
                                      self.conf_prefix, modality, self.alpha, self.r_text,
                                      self.r_img, self.kept_off, self.total_kept,
                                      kept_idx=self.kept_idx, score=self.score,
                                      ws=self.ws_score, status=self.status)
            elif self.keep is None:
                sp.sprint_score_prune(K, self.prefix_off, self.total_rows, self.NL, self.Hkv,
                                      self.d, self.conf_prefix, modality, self.alpha,
                                      self.r_text, self.r_img, self.kept_off, self.total_kept,
                                      kept_idx=self.kept_idx, score=self.score,
                                      ws=self.ws_score, status=self.status)
            elif overlap:
                sp.sprint_select_kept_pools(self.u, self.prefix_off, self.total_rows,
                                            self.conf_prefix, pool, self.n_pools, self.keep,
                                            self.alpha, self.kept_off, self.total_kept,
                                            kept_idx=self.kept_idx, score=self.score,
                                            ws=self.ws_score, status=self.status)
            else:
                sp.sprint_score_prune_pools(K, self.prefix_off, self.total_rows, self.NL,
                                            self.Hkv, self.d, self.conf_prefix, pool,
                                            self.n_pools, self.keep, self.alpha, self.kept_off,
                                            self.total_kept, kept_idx=self.kept_idx,
                                            score=self.score, ws=self.ws_score,
                                            status=self.status)
        if self.indexed:
            return merged
        with self._stage("compact"):
            sp.sprint_compact_kv(K, V, self.prefix_off, self.total_rows, self.NL, self.Hkv,
                                 self.d, self.kept_idx, self.kept_off, self.total_kept,
                                 Kp=self.Kp, Vp=self.Vp, status=self.status)
        return merged

    def _merged_lmhead(self, H, theta, r0, step0):
        """One LM-head call over the new prefix rows [r0, n) and the block's
        step-0 rows, laid side by side (device copies); its outputs are
        copied back to the prefix and block buffers.  A row's result does
        not depend on the other rows of the call, so this equals the two
        separate calls bit for bit while both stay below 4096 rows."""
        if step0.get("theta") is None:
            return False
        n_new, M_blk = self.total_rows - r0, self.S * self.LB
        rows = n_new + M_blk
        if rows >= 4096 or self.total_rows >= 4096:  # keep both calls on the same strips
            return False
        dt = self._dt
        if sp.sprint_lmhead_workspace_bytes(rows, self.D, self.V, dt) > self.ws_lm_prefix.numel():
            return False
        hm = self._buf("h_merge", rows * self.D, self.dtype).view(rows, self.D)
        tm = self._buf("theta_merge", rows, torch.float32)
        cm = self._buf("conf_merge", rows, torch.float32)
        am = self._buf("argmax_merge", rows, torch.int32)
        hm[:n_new].copy_(H[r0:])
        hm[n_new:].copy_(step0["h"])
        tm[:n_new].copy_(theta[r0:])
        tm[n_new:].copy_(step0["theta"])
        sp.sprint_lmhead_confidence(hm, self.W, tm, conf=cm, argmax=am, ws=self.ws_lm_prefix,
                                    status=self.status)
        self.conf_prefix[r0:].copy_(cm[:n_new])
        if self.prefix_argmax:
            self.argmax_prefix[r0:].copy_(am[:n_new])
        self.conf_blk.copy_(cm[n_new:])
        self.argmax_blk.copy_(am[n_new:])
        return True

    def step(self, t, x, K, V):
        """One denoising step.  K, V: the full prefix cache; step 0 attends
        to all of it, later steps to the kept rows (the pruned copy, or K / V
        read through the kept indices)."""
        if t == 0:
            with self._stage("attn_full"):
                sp.sprint_block_attn(x["Q"], K, V, self.prefix_off, self.max_rows,
                                     self.total_rows, x["Kb"], x["Vb"], O=self.O,
                                     ws=self.ws_attn, status=self.status)
        elif self.indexed:
            with self._stage("attn_pruned"):
                sp.sprint_block_attn_indexed(x["Q"], K, V, self.prefix_off, self.total_rows,
                                             self.kept_idx, self.kept_off, self.max_kept,
                                             self.total_kept, x["Kb"], x["Vb"], O=self.O,
                                             ws=self.ws_attn, status=self.status)
        else:
            with self._stage("attn_pruned"):
                sp.sprint_block_attn(x["Q"], self.Kp, self.Vp, self.kept_off, self.max_kept,
                                     self.total_kept, x["Kb"], x["Vb"], O=self.O,
                                     ws=self.ws_attn, status=self.status)
        h = x["h"]
        if self.residual:
            with self._stage("residual"):
                h = sp.sprint_residual_hidden(x["h"], self.O, h_out=self.h_res)
        with self._stage("lmhead_block"):
            sp.sprint_lmhead_confidence(h, self.W, x["theta"], conf=self.conf_blk,
                                        argmax=self.argmax_blk, logits=self.logits,
                                        ws=self.ws_lm_blk, status=self.status)
        with self._stage("unmask"):
            sp.sprint_unmask(self.conf_blk, self.argmax_blk, self.mask, self.tokens, t, self.T,
                             self.tau, self.mode, m_out=self.m_out, accepted=self.accepted,
                             status=self.status)

    def masked_left(self):
        self.m_host.copy_(self.m_out, non_blocking=True)
        self.ev.record()
        self.ev.synchronize()
        return self.m_host.tolist()

    def decode(self, prefix, steps, on_step=None, wait=True, conf_from=0):
        """Decode one block.  prefix: dict K, V, H, theta, modality (device,
        sequences concatenated).  steps(t) -> dict Q, Kb, Vb, h, theta.
        With on_step (called after each step with (t, self)) the block is
        decoded step by step (decode_stepwise).

        wait=False returns a PendingBlock at once (nothing waits for the
        GPU); finish(pending) later returns its BlockResult.  Two blocks may
        be pending; `pending.tokens` is the live token buffer, which the
        next block overwrites, so copy it (on the stream) before that."""
        if on_step is not None:
            return self.decode_stepwise(prefix, steps, on_step, conf_from=conf_from)
        slot = self._next_slot
        self._next_slot ^= 1
        if self._slots[slot] is not None:  # at most two blocks in flight
            self.finish(self._slots[slot])
        xs = [steps(t) for t in range(self.T)]
        # With the prefix-confidence cache, step 0's block rows share the
        # prefix LM-head call (not with the residual chain: there step 0's
        # h depends on its attention).
        step0_given = self.prefix_pass(
            prefix["K"], prefix["V"], prefix["H"], prefix["theta"], prefix["modality"],
            conf_from=conf_from, image=prefix.get("image"),
            step0=xs[0] if conf_from and not self.residual and not self.want_logits else None,
            Qp=prefix.get("Qp"))
        events = self._events_for_steps(slot) if self.timing is not None else None
        sp.sprint_decode_steps(
            Q=[x["Q"] for x in xs], Kb=[x["Kb"] for x in xs], Vb=[x["Vb"] for x in xs],
            h=[x["h"] for x in xs], theta=[x.get("theta") for x in xs],
            Kf=prefix["K"], Vf=prefix["V"], prefix_off=self.prefix_off,
            max_rows=self.max_rows, total_rows=self.total_rows, Kp=self.Kp, Vp=self.Vp,
            kept_off=self.kept_off, max_kept=self.max_kept, total_kept=self.total_kept,
            W=self.W, T=self.T, tau=self.tau, mode=self.mode, O=self.O, conf=self.conf_blk,
            argmax=self.argmax_blk, mask=self.mask, tokens=self.tokens, m_hist=self.m_hist,
            ws_attn=self.ws_attn, ws_lm=self.ws_lm_blk, status=self.status,
            logits=self.logits, events=events,
            kept_idx=self.kept_idx if self.indexed else None, h_res=self.h_res,
            step0_given=step0_given)
        m_host = self._m_hist_host[slot]
        m_host.copy_(self.m_hist, non_blocking=True)
        done = self._done[slot]
        done.record()
        pending = PendingBlock(slot, done, m_host, events, self._pending, self.tokens,
                               step0_given=step0_given)
        self._pending = []
        self._slots[slot] = pending
        return self.finish(pending) if wait else pending

    def finish(self, pending) -> BlockResult:
        """Wait for a pending block and return its result (idempotent)."""
        if pending.result is not None:
            return pending.result
        pending.done.synchronize()
        hist = pending.m_hist_host.tolist()
        accepted, prev, n_steps = [], [self.LB] * self.S, 0
        timing = pending.stage_events
        for t in range(self.T):
            if t > 0 and not any(hist[t - 1]):
                break
            n_steps += 1
            accepted.append([p - q for p, q in zip(prev, hist[t])])
            prev = hist[t]
            if pending.step_events is not None:
                ev = pending.step_events
                for k, name in enumerate(("attn_full" if t == 0 else "attn_pruned",
                                          "lmhead_block", "unmask")):
                    if t == 0 and name == "lmhead_block" and pending.step0_given:
                        continue  # computed within the prefix LM-head stage
                    if ev[6 * t + 2 * k] is not None:
                        timing.append((name, ev[6 * t + 2 * k], ev[6 * t + 2 * k + 1]))
        if self.timing is not None:
            for name, a, b in timing:
                self.timing.setdefault(name, []).append(a.elapsed_time(b))
        pending.result = BlockResult(n_steps, pending.tokens, accepted)
        if self._slots[pending.slot] is pending:
            self._slots[pending.slot] = None
        return pending.result

    def decode_stepwise(self, prefix, steps, on_step=None, conf_from=0) -> BlockResult:
        """Decode one block one step at a time, reading the masked counts
        after every step (on_step(t, self) is called after each step)."""
        self.mask.fill_(1)
        self.tokens.fill_(-1)
        self.prefix_pass(prefix["K"], prefix["V"], prefix["H"], prefix["theta"],
                         prefix["modality"], conf_from=conf_from, image=prefix.get("image"),
                         Qp=prefix.get("Qp"))
        accepted = []
        prev = [self.LB] * self.S
        n_steps = 0
        for t in range(self.T):
            self.step(t, steps(t), prefix["K"], prefix["V"])
            n_steps += 1
            if on_step is not None:
                on_step(t, self)
            left = self.masked_left()
            accepted.append([p - q for p, q in zip(prev, left)])
            prev = left
            if not any(left):
                break
        self._flush_timing()
        return BlockResult(n_steps, self.tokens, accepted)
