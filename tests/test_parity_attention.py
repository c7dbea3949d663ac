"""GPU parity of sprint_block_attn against the oracle."""
import numpy as np
import pytest
import torch

from oracle import sprint_oracle as orc
from tests import gpu_cases as gc
from workload import WORKLOADS, prefix_inputs, step_inputs, small_workload

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def sp():
    from kv_cache_pruning_step_b300 import sprint
    return sprint


def run_attn(sp, w, prefixes, steps):
    cat = gc.concat_prefixes(prefixes)
    lens = [p["modality"].numel() for p in prefixes]
    Q = torch.stack([x["Q"] for x in steps]).contiguous()
    Kb = torch.stack([x["Kb"] for x in steps]).contiguous()
    Vb = torch.stack([x["Vb"] for x in steps]).contiguous()
    status = sp.new_status(DEV)
    O = sp.sprint_block_attn(Q, cat["K"], cat["V"], cat["off"], max(lens), sum(lens), Kb, Vb,
                             status=status)
    torch.cuda.synchronize()
    assert status.item() == 0
    return O


def check(w, prefixes, steps, O, layers=None, what=""):
    for s, (p, x) in enumerate(zip(prefixes, steps)):
        want = orc.block_attention(x["Q"], p["K"], p["V"], x["Kb"], x["Vb"], layers=layers)
        got = gc.host(O[s])
        sel = list(range(w.NL)) if layers is None else layers
        gc.assert_close(got[sel], want[sel], w.torch_dtype, f"{what} seq {s}")


def test_tiny_fp32_full_prefix(sp):
    w = WORKLOADS["tiny-256"]
    pre = prefix_inputs(w, device=DEV)
    x = step_inputs(w, 0, 0, 1, device=DEV)
    O = run_attn(sp, w, [pre], [x])
    check(w, [pre], [x], O, what="tiny")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("Hq,Hkv,d,LB", [(4, 2, 64, 32), (16, 4, 128, 32), (8, 8, 64, 16),
                                         (6, 2, 128, 7), (2, 1, 64, 1)])
def test_fuzz_ragged(sp, dtype, Hq, Hkv, d, LB):
    lens = [0, 1, 129, 700, 2051]
    prefixes, steps = [], []
    for s, n in enumerate(lens):
        w = small_workload(dtype=dtype, NL=2, Hq=Hq, Hkv=Hkv, d=d, LB=LB, n=n, n_img=n // 3,
                           seed=40 + s)
        prefixes.append(prefix_inputs(w, seq=s, device=DEV))
        steps.append(step_inputs(w, s, 0, 3, device=DEV))
    O = run_attn(sp, w, prefixes, steps)
    check(w, prefixes, steps, O, what=f"{dtype} {Hq}/{Hkv}/{d}/{LB}")


@pytest.mark.parametrize("d,LB,Hq,Hkv", [(128, 32, 16, 4), (64, 7, 6, 2)])
def test_output_buffer_with_bf16_alignment_only(sp, d, LB, Hq, Hkv):
    """O may start at any bf16 element: the combine then stores element by
    element, with the same bits as into a 16-byte aligned buffer."""
    w = small_workload(dtype="bf16", NL=2, Hq=Hq, Hkv=Hkv, d=d, LB=LB, n=900, n_img=300, seed=23)
    pre = prefix_inputs(w, device=DEV)
    x = step_inputs(w, 0, 0, 1, device=DEV)
    O = run_attn(sp, w, [pre], [x])
    cat = gc.concat_prefixes([pre])
    buf = torch.full((O.numel() + 1,), float("nan"), dtype=O.dtype, device=DEV)
    O1 = buf[1:].view(O.shape)
    assert O1.data_ptr() % 16 != 0
    status = sp.new_status(DEV)
    sp.sprint_block_attn(x["Q"][None].contiguous(), cat["K"], cat["V"], cat["off"], 900, 900,
                         x["Kb"][None].contiguous(), x["Vb"][None].contiguous(), O=O1,
                         status=status)
    torch.cuda.synchronize()
    assert status.item() == 0
    assert torch.equal(O1, O)
    assert torch.isnan(buf[0])


def test_identical_keys_average_values(sp):
    w = small_workload(dtype="f32", NL=1, Hq=4, Hkv=2, d=64, LB=8, n=50, n_img=0)
    pre = prefix_inputs(w, device=DEV)
    x = step_inputs(w, 0, 0, 0, device=DEV)
    pre["K"][:] = 0.25
    x["Kb"][:] = 0.25
    O = run_attn(sp, w, [pre], [x])
    vals = torch.cat([pre["V"][0], x["Vb"][0]], dim=0)  # [n+LB][Hkv][d]
    mean = vals.double().mean(dim=0)                      # [Hkv][d]
    for h in range(4):
        g = h * 2 // 4
        want = mean[g].expand(8, 64).cpu().numpy()
        gc.assert_close(gc.host(O[0, 0, :, h]), want, torch.float32, "mean of values")


@pytest.mark.parametrize("name", ["prefix-4k", "prefix-32k"])
def test_full_size_sampled_layers(sp, name):
    w = WORKLOADS[name]
    pre = prefix_inputs(w, device=DEV)
    x = step_inputs(w, 0, 0, 2, device=DEV)
    O = run_attn(sp, w, [pre], [x])
    check(w, [pre], [x], O, layers=[0, w.NL - 1], what=name)
    assert torch.isfinite(O.float()).all()


def test_batched_ragged_full_size(sp):
    w = WORKLOADS["batch-16x8k"]
    prefixes = [prefix_inputs(w, seq=s, device=DEV) for s in range(4)]
    # ragged: cut each prefix to a different length
    cuts = [8192, 5000, 1, 7777]
    for p, n in zip(prefixes, cuts):
        p["K"] = p["K"][:, :n].contiguous()
        p["V"] = p["V"][:, :n].contiguous()
        p["modality"] = p["modality"][:n]
    steps = [step_inputs(w, s, 0, 1, device=DEV) for s in range(4)]
    O = run_attn(sp, w, prefixes, steps)
    check(w, prefixes, steps, O, layers=[3], what="batch")


def test_full_retention_pruned_cache_equals_full_prefix_bitwise(sp):
    """r = 1 keeps every position: attention over the compacted cache must be
    bit-identical to attention over the full prefix (same kernel, same keys)."""
    w = WORKLOADS["prefix-4k"]
    pre = prefix_inputs(w, device=DEV)
    n = pre["modality"].numel()
    x = step_inputs(w, 0, 0, 1, device=DEV)
    off = torch.tensor([0, n], dtype=torch.int32, device=DEV)
    kept = torch.arange(n, dtype=torch.int32, device=DEV)
    status = sp.new_status(DEV)
    Kp, Vp = sp.sprint_compact_kv(pre["K"], pre["V"], off, n, w.NL, w.Hkv, w.d, kept, off, n,
                                  status=status)
    O_full = run_attn(sp, w, [pre], [x])
    O_pruned = sp.sprint_block_attn(x["Q"][None].contiguous(), Kp, Vp, off, n, n,
                                    x["Kb"][None].contiguous(), x["Vb"][None].contiguous(),
                                    status=status)
    torch.cuda.synchronize()
    assert status.item() == 0
    assert torch.equal(O_full, O_pruned)


def test_many_short_sequences_two_stage_ring(sp):
    """300 sequences of 0..200 prefix rows: the per-sequence tables take
    enough shared memory that the bf16 kernel runs a 2-stage K/V ring, and
    most segments are short (many pairs per CTA)."""
    rng = torch.Generator().manual_seed(11)
    lens = torch.randint(0, 201, (300,), generator=rng).tolist()
    prefixes, steps = [], []
    for s, n in enumerate(lens):
        w = small_workload(dtype="bf16", NL=1, Hq=8, Hkv=2, d=128, LB=16, n=n, n_img=n // 4,
                           seed=700 + s)
        prefixes.append(prefix_inputs(w, seq=s, device=DEV))
        steps.append(step_inputs(w, s, 0, 1, device=DEV))
    O = run_attn(sp, w, prefixes, steps)
    picks = [0, 1, 57, 150, 299] + [s for s, n in enumerate(lens) if n == 0][:2]
    check(w, [prefixes[s] for s in picks], [steps[s] for s in picks], O[picks],
          what="many sequences")


def _aligned_keys(Q, a, d):
    """Keys k_i = a_i * dir_g with dir_g = q_g sqrt(d) / (|q_g|^2 log2 e): a
    query equal to q_g scores key i at a_i in the kernel's log2 units."""
    q = Q[:, 0].float()                                     # [NL][Hkv][d] (one row per head)
    dirs = q * (d ** 0.5) / (q.pow(2).sum(-1, keepdim=True) * np.log2(np.e))
    return (a.view(1, -1, 1, 1) * dirs.unsqueeze(1))       # [NL][n][Hkv][d]


@pytest.mark.parametrize("pattern", ["ramp", "spikes", "descending"])
def test_row_maxima_moving_within_tiles(sp, pattern):
    """Scores that climb through a tile (the reference maximum moves in both
    key halves of most tiles), isolated spikes in the first and second half
    of tiles, and falling scores, for query rows that see them with either
    sign.  The output must match the fp64 oracle whatever the order in
    which the row maxima appear."""
    NL, Hq, Hkv, d, LB, n = 1, 2, 2, 128, 32, 1000
    w = small_workload(dtype="bf16", NL=NL, Hq=Hq, Hkv=Hkv, d=d, LB=LB, n=n, n_img=0, seed=77)
    pre = prefix_inputs(w, device=DEV)
    x = step_inputs(w, 0, 0, 1, device=DEV)
    g = torch.Generator(device=DEV).manual_seed(78)
    q = torch.randn((NL, 1, Hq, d), generator=g, device=DEV)
    sign = torch.ones(LB, device=DEV)
    sign[LB // 2:] = -1.0                                   # half the rows see -a
    x["Q"] = (q * sign.view(1, LB, 1, 1)).to(torch.bfloat16).contiguous()
    i = torch.arange(n, device=DEV, dtype=torch.float32)
    if pattern == "ramp":
        a = 0.6 * i                                         # +19 per 32-key chunk
    elif pattern == "spikes":
        a = 0.5 * torch.randn(n, generator=g, device=DEV)
        for t0 in range(0, n, 128):
            for off, hgt in ((40, 30.0), (70, 60.0), (100, 90.0)):
                if t0 + off < n:
                    a[t0 + off] = hgt + t0 / 10.0
    else:
        a = 40.0 - 0.04 * i
    pre["K"] = _aligned_keys(x["Q"].float(), a, d).to(torch.bfloat16).contiguous()
    x["Kb"] = (0.1 * torch.randn(x["Kb"].shape, generator=g, device=DEV)).to(torch.bfloat16)
    O = run_attn(sp, w, [pre], [x])
    check(w, [pre], [x], O, what=pattern)
