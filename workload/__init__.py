"""Seeded synthetic inputs for the SPRINT block-decode step.

This module is the only code that both the CUDA path and the CPU oracle see.
It draws tensors; it holds none of the method's arithmetic (no norms, no
softmax, no keep counts, no selection).  Every tensor is a pure function of
(workload seed, sequence, block, step, tensor name), so any block can be
regenerated in isolation.

Value distributions (the LLaDA2.0-Uni paper gives no activations, so these
stand in for a real backbone's):
  * prefix keys/values  K, V = z * exp(0.5 * y), z, y ~ N(0, 1); the
    log-normal scale exp(0.5*y) is drawn once per position and shared by all
    layers and KV heads, so a position's key norm is consistent across layers;
  * block keys/values   the same recipe, fresh per step;
  * queries Q and hidden states H, h ~ N(0, 1);
  * LM-head weight W ~ N(0, std = 1/16) (1/sqrt(256), every workload);
  * per-position logit temperature theta ~ U[0.5, 4].
bf16 workloads round once, at generation.

Modality layouts follow the image-token counts of the LLaDA2.0-Uni paper,
Stage 0 paragraph (about 256 tokens for a 256x256 image, about 1024 for a
512x512 one): image spans are runs of 1024 tokens, or of 256-token slots.
Tag 0 = text, 1 = image.  Each image of a layout also has a number (1, 2,
... in position order; 0 for text): a 1024-token span is one 512x512 image,
every 256-token image slot one 256x256 image.
"""
from __future__ import annotations

import hashlib
from dataclasses import dataclass, field

import torch

TEXT = 0
IMAGE = 1


@dataclass(frozen=True)
class Workload:
    """One SPRINT decode workload: model shapes, settings and prefix layout."""

    name: str
    dtype: str            # "f32" or "bf16" (storage; accumulation is fp32)
    NL: int               # attention layers
    Hq: int               # query heads
    Hkv: int              # KV heads (GQA)
    d: int                # head dim
    D: int                # hidden size
    V: int                # vocabulary
    LB: int               # block length (tokens decoded per block)
    T: int                # denoising steps per block
    tau: float            # unmask confidence threshold
    r_text: float         # keep ratio for text positions
    r_img: float          # keep ratio for image positions
    alpha: float          # blend weight of key-norm importance
    seed: int
    S: int = 1            # independent sequences decoded together
    blocks: int = 1       # blocks decoded one after another
    description: str = ""
    extra: dict = field(default_factory=dict, compare=False, hash=False)

    @property
    def torch_dtype(self) -> torch.dtype:
        return torch.float32 if self.dtype == "f32" else torch.bfloat16


def _spans(*pairs):
    out = []
    for count, tag in pairs:
        out += [tag] * count
    return out


WORKLOADS = {
    # 1 layer, fp32, 256-token prefix: 192 text then 64 image.
    "tiny-256": Workload(
        name="tiny-256", dtype="f32", NL=1, Hq=4, Hkv=2, d=64, D=256, V=1024,
        LB=32, T=4, tau=0.9, r_text=1.0, r_img=0.8, alpha=0.5, seed=1000,
        description="1 layer, fp32, prefix 192 text + 64 image"),
    # 8 layers, bf16, 4K prefix: 1024 text, then three 1024-token images.
    "prefix-4k": Workload(
        name="prefix-4k", dtype="bf16", NL=8, Hq=16, Hkv=4, d=128, D=2048,
        V=157184, LB=32, T=8, tau=0.9, r_text=1.0, r_img=0.8, alpha=0.5,
        seed=1001, description="8 layers, bf16, prefix 1024 text + 3 x 1024 image"),
    # 32K prefix: 16 x (1024 text, 1024 image), text first.
    "prefix-32k": Workload(
        name="prefix-32k", dtype="bf16", NL=8, Hq=16, Hkv=4, d=128, D=2048,
        V=157184, LB=32, T=8, tau=0.9, r_text=1.0, r_img=0.8, alpha=0.5,
        seed=1002, description="8 layers, bf16, prefix 16 x (1024 text + 1024 image)"),
    # 16 independent sequences of 8192, image fraction U[0, 0.9] in 256-slots.
    "batch-16x8k": Workload(
        name="batch-16x8k", dtype="bf16", NL=8, Hq=16, Hkv=4, d=128, D=2048,
        V=157184, LB=32, T=8, tau=0.9, r_text=1.0, r_img=0.8, alpha=0.5,
        seed=1003, S=16,
        description="16 sequences x 8192, image fraction U[0,0.9] in 256-token slots"),
    # 64 blocks decoded in order; prefix [1024 image][1024 text][32 b generated].
    "sequential-64-blocks": Workload(
        name="sequential-64-blocks", dtype="bf16", NL=8, Hq=16, Hkv=4, d=128,
        D=2048, V=157184, LB=32, T=8, tau=0.9, r_text=1.0, r_img=0.8,
        alpha=0.5, seed=1004, blocks=64,
        description="64 blocks of 32, prefix grows 2048 -> 4096"),
}


def small_workload(name="fuzz", *, dtype="f32", NL=2, Hq=4, Hkv=2, d=64, D=128,
                   V=300, LB=32, T=4, tau=0.9, r_text=1.0, r_img=0.8,
                   alpha=0.5, seed=7, S=1, n=96, n_img=32) -> Workload:
    """A workload of arbitrary (small) shapes for parity fuzzing; its prefix
    is n positions, the last n_img of them image."""
    return Workload(name=name, dtype=dtype, NL=NL, Hq=Hq, Hkv=Hkv, d=d, D=D, V=V,
                    LB=LB, T=T, tau=tau, r_text=r_text, r_img=r_img,
                    alpha=alpha, seed=seed, S=S, extra={"n": n, "n_img": n_img})


def _stream_seed(*key) -> int:
    """63-bit seed for the sub-stream named by ``key`` (stable across runs)."""
    h = hashlib.blake2b(repr(key).encode(), digest_size=8).digest()
    return int.from_bytes(h, "little") & ((1 << 63) - 1)


def generator(device, *key) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(_stream_seed(*key))
    return g


def prefix_layout(w: Workload, seq: int = 0, block: int = 0) -> torch.Tensor:
    """Modality tags (uint8, 0 text / 1 image) of one sequence's prefix."""
    if w.name == "tiny-256":
        tags = _spans((192, TEXT), (64, IMAGE))
    elif w.name == "prefix-4k":
        tags = _spans((1024, TEXT), (3 * 1024, IMAGE))
    elif w.name == "prefix-32k":
        tags = _spans(*[p for _ in range(16) for p in ((1024, TEXT), (1024, IMAGE))])
    elif w.name == "batch-16x8k":
        g = generator("cpu", w.seed, "layout", seq)
        f = 0.9 * torch.rand((), generator=g).item()
        n_img_slots = int(32 * f)
        perm = torch.randperm(32, generator=g)
        slot_tag = torch.zeros(32, dtype=torch.uint8)
        slot_tag[perm[:n_img_slots]] = IMAGE
        return slot_tag.repeat_interleave(256)
    elif w.name == "sequential-64-blocks":
        tags = _spans((1024, IMAGE), (1024, TEXT), (32 * block, TEXT))
    else:
        n = w.extra.get("n", 96)
        n_img = w.extra.get("n_img", n // 3)
        tags = _spans((n - n_img, TEXT), (n_img, IMAGE))
    return torch.tensor(tags, dtype=torch.uint8)


def image_layout(w: Workload, seq: int = 0, block: int = 0) -> torch.Tensor:
    """Image number of every prefix position (uint8): 0 for text, j for the
    j-th image of the layout in position order (an image is a 1024-token
    span, or a 256-token slot in the batched workload's layout)."""
    tags = prefix_layout(w, seq, block)
    ids = torch.zeros(tags.numel(), dtype=torch.uint8)
    span = {"batch-16x8k": 256, "prefix-4k": 1024, "prefix-32k": 1024,
            "sequential-64-blocks": 1024}.get(w.name)
    j, start, prev = 0, 0, TEXT
    for i, t in enumerate(tags.tolist()):
        if t == IMAGE:
            if prev != IMAGE:
                start = i
            if prev != IMAGE or (span is not None and (i - start) % span == 0):
                j += 1
            ids[i] = j
        prev = t
    return ids


def _scaled_normal(shape, pos_dim, g, device):
    """z * exp(0.5*y): z ~ N(0,1) per element, y ~ N(0,1) per position."""
    z = torch.randn(shape, generator=g, device=device)
    y = torch.randn(shape[pos_dim], generator=g, device=device)
    view = [1] * len(shape)
    view[pos_dim] = shape[pos_dim]
    return z * torch.exp(0.5 * y).view(view)


def prefix_inputs(w: Workload, seq: int = 0, block: int = 0, device="cpu",
                  n: int | None = None):
    """Prefix tensors of one sequence at one block's first step.

    Returns a dict with K, V [NL][n][Hkv][d], H [n][D], theta [n] (f32),
    modality [n] (uint8) and image [n] (uint8 image numbers, 0 for text).  For the sequential workload the cache grows by
    appending: block b sees the first 2048 + 32 b rows of one fixed cache.
    """
    modality = prefix_layout(w, seq, block)
    n = modality.numel() if n is None else n
    modality = modality[:n]
    image = image_layout(w, seq, block)[:n]
    full = n
    blk_key = block
    if w.name == "sequential-64-blocks":
        full = 2048 + 32 * w.blocks
        blk_key = 0
    g = generator(device, w.seed, "prefix", seq, blk_key)
    dt = w.torch_dtype
    K = _scaled_normal((w.NL, full, w.Hkv, w.d), 1, g, device)[:, :n].to(dt).contiguous()
    V = _scaled_normal((w.NL, full, w.Hkv, w.d), 1, g, device)[:, :n].to(dt).contiguous()
    H = torch.randn((full, w.D), generator=g, device=device)[:n].to(dt).contiguous()
    theta = (0.5 + 3.5 * torch.rand(full, generator=g, device=device))[:n].contiguous()
    return {"K": K, "V": V, "H": H, "theta": theta, "modality": modality.to(device),
            "image": image.to(device)}


def prefix_queries(w: Workload, seq: int = 0, block: int = 0, device="cpu",
                   n: int | None = None) -> torch.Tensor:
    """Queries of the prefix positions for the prefix's own attention in a
    block's first step: Qp [NL][n][Hq][d] ~ N(0, 1), in the storage type."""
    n = prefix_layout(w, seq, block).numel() if n is None else n
    g = generator(device, w.seed, "prefix-q", seq, block)
    return torch.randn((w.NL, n, w.Hq, w.d), generator=g, device=device).to(w.torch_dtype)


def step_inputs(w: Workload, seq: int, block: int, step: int, device="cpu"):
    """Per-step block tensors: Q [NL][LB][Hq][d], Kb, Vb [NL][LB][Hkv][d],
    h [LB][D] and theta [LB]."""
    g = generator(device, w.seed, "step", seq, block, step)
    dt = w.torch_dtype
    Q = torch.randn((w.NL, w.LB, w.Hq, w.d), generator=g, device=device).to(dt)
    Kb = _scaled_normal((w.NL, w.LB, w.Hkv, w.d), 1, g, device).to(dt)
    Vb = _scaled_normal((w.NL, w.LB, w.Hkv, w.d), 1, g, device).to(dt)
    h = torch.randn((w.LB, w.D), generator=g, device=device).to(dt)
    theta = 0.5 + 3.5 * torch.rand(w.LB, generator=g, device=device)
    return {"Q": Q, "Kb": Kb, "Vb": Vb, "h": h, "theta": theta}


def lm_head_weight(w: Workload, device="cpu") -> torch.Tensor:
    """LM-head weight W [V][D] ~ N(0, 1/16^2)."""
    g = generator(device, w.seed, "W")
    W = torch.empty((w.V, w.D), device=device)
    # Draw in row chunks to bound the fp32 temporary on large vocabularies.
    step = max(1, (1 << 26) // max(w.D, 1))
    for r0 in range(0, w.V, step):
        r1 = min(w.V, r0 + step)
        W[r0:r1] = torch.randn((r1 - r0, w.D), generator=g, device=device) / 16.0
    return W.to(w.torch_dtype)


def random_confidences(n: int, seed: int, device="cpu", low=0.0, high=1.0):
    """Stand-in per-position confidences in [low, high) for stage-wise tests."""
    g = generator(device, seed, "conf", n)
    return low + (high - low) * torch.rand(n, generator=g, device=device)
