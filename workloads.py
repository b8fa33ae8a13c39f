"""Seeded synthetic inputs and the workload table for the dense video-token
attention path and the AdaLN elementwise ops around it.

This module is shared by the tests, ``bench.py`` and ``__graft_entry__``.  It
holds no arithmetic of the method itself: it only sizes workloads from the
video geometry and draws seeded random tensors.  Both the CUDA path and the
oracle consume exactly the tensors drawn here.

Geometry follows "FreeVideo: a 66 GB video transformer on an 8 GB card",
section "What MiniMax H3 is, briefly": frames round up to 17n+5, which is
5n+2 latent frames; each latent frame at W x H holds (W/32) x (H/32) tokens
(16x VAE compression and a 1x2x2 patch), so 1344x768 gives 24 x 42 = 1,008
tokens per latent frame.  The same section fixes 56 heads of 128 (Q, K and V
7168 wide) and the hidden size 5,376.

Random recipe (stated once here, used everywhere):
  * every tensor gets its own ``torch.Generator('cpu')`` seeded
    ``1000 * base_seed + tensor_id`` (Q=0, K=1, V=2, x=3, a=4, shift=5,
    scale=6, gate=7), so the draws do not depend on the order of calls;
  * activations are ``torch.randn`` in float32, i.e. N(0, 1), then rounded
    to bfloat16 (round to nearest even);
  * AdaLN tables are N(0, 1) * 0.1 in float32 (standard deviation 0.1);
  * outlier channels (the half-resolution workload): 1% of K's 7,168
    columns, chosen by ``torch.randperm`` under seed 2, are scaled by 20 in
    float32 before the rounding to bfloat16;
  * sampled query rows per head h: ``randperm(N)`` under seed 5000 + h, the
    first k, plus rows 0, 1, N-1 and the first and last row of the last
    128-row tile.
"""
from __future__ import annotations

import dataclasses
import math

import torch

HEAD_DIM = 128          # D
NUM_HEADS = 56          # H
HIDDEN = 5376           # C, model width of the residual stream
TABLE_STEPS = 8         # rows of a per-step AdaLN table
ADALN_STEP = 3          # the step every workload reads
TILE = 128              # query/key tile edge of the attention kernel

TENSOR_IDS = {"q": 0, "k": 1, "v": 2, "x": 3, "a": 4, "shift": 5, "scale": 6, "gate": 7}


# --------------------------------------------------------------------------
# video geometry
# --------------------------------------------------------------------------
def latent_frames(frames: int) -> int:
    """Latent frames for a clip of ``frames`` video frames.

    Frames are rounded up to the next 17n+5; that clip holds 5n+2 latent
    frames (one 17-frame VAE chunk is 5 latent frames).
    """
    if frames < 1:
        raise ValueError("frames must be >= 1")
    n = max(0, -(-(frames - 5) // 17))
    return 5 * n + 2


def vae_chunk_latent_frames(chunks: int = 1) -> int:
    """Latent frames of ``chunks`` whole 17-frame VAE chunks (5 each)."""
    return 5 * chunks


def tokens_per_latent_frame(width: int, height: int) -> int:
    """Video tokens in one latent frame: (W/32) x (H/32)."""
    if width % 32 or height % 32:
        raise ValueError("width and height must be multiples of 32")
    return (width // 32) * (height // 32)


def video_tokens(width: int, height: int, frames: int) -> int:
    return latent_frames(frames) * tokens_per_latent_frame(width, height)


def attention_flops(n: int, heads: int = NUM_HEADS, d: int = HEAD_DIM) -> float:
    """Algorithmic FLOPs of one dense attention forward: 4 * N^2 * d * H."""
    return 4.0 * float(n) * float(n) * d * heads


def window_pairs(n: int, frame_tokens: int, chunk_frames: int = 5, window_chunks: int = 1) -> int:
    """(query, key) pairs the Video DeltaNet softmax window admits, for FLOP
    accounting: counted over latent-frame pairs, times frame_tokens^2."""
    frames = n // frame_tokens
    pairs = 0
    for f in range(frames):
        if f in (0, frames - 1):
            pairs += frames
            continue
        c = f // chunk_frames
        lo = max(0, (c - window_chunks) * chunk_frames)
        hi = min(frames, (c + window_chunks + 1) * chunk_frames)
        seen = set(range(lo, hi)) | {0, frames - 1}
        pairs += len(seen)
    return pairs * frame_tokens * frame_tokens


# --------------------------------------------------------------------------
# workload table
# --------------------------------------------------------------------------
@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    base_seed: int
    n: int                    # video tokens (attention sequence length)
    heads: int
    head_group: int
    outlier_k: bool = False   # 1% of K channels scaled x20
    rows_per_head: int = 0    # 0: check every row against the oracle
    modulate_rows: int = 0    # rows of x for the modulate op (0: none)
    gres_rows: int = 0        # rows of x / attn_out for the gated residual (0: none)

    @property
    def flops(self) -> float:
        return attention_flops(self.n, self.heads)


WORKLOADS = {
    # one latent frame at 1344x768, 4 heads; modulate on [1008, 5376]
    "tiny_1008": Workload("tiny_1008", 0, tokens_per_latent_frame(1344, 768), 4, 4,
                          modulate_rows=1008),
    # one 17-frame VAE chunk (5 latent frames) at 1344x768; gated residual on [5040, 5376]
    "clip17_5040": Workload("clip17_5040", 1, vae_chunk_latent_frames(1) * tokens_per_latent_frame(1344, 768), 56, 16,
                            gres_rows=5040),
    # half-resolution first pass of a 10 s clip, K with outlier channels
    "half_res_18144": Workload("half_res_18144", 2, video_tokens(672, 384, 243), 56, 16,
                               outlier_k=True, rows_per_head=256),
    # 10 s clip at 1344x768, head groups 16/16/16/8 (the headline workload)
    "clip10s_72576": Workload("clip10s_72576", 3, video_tokens(1344, 768, 243), 56, 16,
                              rows_per_head=256, modulate_rows=video_tokens(1344, 768, 243),
                              gres_rows=video_tokens(1344, 768, 243)),
    # 14.4 s clip at 1344x768, head group 8; modulate and gated residual at full size
    "clip14s_102816": Workload("clip14s_102816", 4, video_tokens(1344, 768, 345), 56, 8,
                               rows_per_head=128, modulate_rows=video_tokens(1344, 768, 345),
                               gres_rows=video_tokens(1344, 768, 345)),
}
HEADLINE = "clip10s_72576"


# --------------------------------------------------------------------------
# seeded generators
# --------------------------------------------------------------------------
def _gen(base_seed: int, tensor: str) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(1000 * base_seed + TENSOR_IDS[tensor])
    return g


def randn_bf16(shape, base_seed: int, tensor: str, chunk_rows: int = 8192) -> torch.Tensor:
    """N(0,1) float32 draws rounded to bfloat16, generated in row chunks so the
    float32 temporary stays small.  The values do not depend on chunk_rows."""
    g = _gen(base_seed, tensor)
    n = shape[0]
    row = math.prod(shape[1:]) if len(shape) > 1 else 1
    out = torch.empty(shape, dtype=torch.bfloat16)
    flat = out.view(n, row)
    for r0 in range(0, n, chunk_rows):
        r1 = min(n, r0 + chunk_rows)
        flat[r0:r1] = torch.randn((r1 - r0, row), generator=g, dtype=torch.float32).to(torch.bfloat16)
    return out


def outlier_channels(total_channels: int, frac: float = 0.01, seed: int = 2) -> torch.Tensor:
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    count = int(round(frac * total_channels))
    return torch.randperm(total_channels, generator=g)[:count].sort().values


def qkv(w: Workload):
    """Q, K, V as bfloat16 [N, H*128] (token-major; head h is columns
    [128h, 128h+128))."""
    width = w.heads * HEAD_DIM
    q = randn_bf16((w.n, width), w.base_seed, "q")
    v = randn_bf16((w.n, width), w.base_seed, "v")
    if not w.outlier_k:
        k = randn_bf16((w.n, width), w.base_seed, "k")
    else:
        g = _gen(w.base_seed, "k")
        cols = outlier_channels(width)
        mult = torch.ones(width, dtype=torch.float32)
        mult[cols] = 20.0
        k = torch.empty((w.n, width), dtype=torch.bfloat16)
        for r0 in range(0, w.n, 8192):
            r1 = min(w.n, r0 + 8192)
            k[r0:r1] = (torch.randn((r1 - r0, width), generator=g, dtype=torch.float32) * mult).to(torch.bfloat16)
    return q, k, v


def adaln_table(base_seed: int, tensor: str, steps: int = TABLE_STEPS, channels: int = HIDDEN) -> torch.Tensor:
    """One AdaLN vector for every step: float32 [steps, channels], N(0, 0.1^2)."""
    g = _gen(base_seed, tensor)
    return torch.randn((steps, channels), generator=g, dtype=torch.float32) * 0.1


def modulate_inputs(w: Workload, rows: int | None = None):
    rows = w.modulate_rows if rows is None else rows
    x = randn_bf16((rows, HIDDEN), w.base_seed, "x")
    return x, adaln_table(w.base_seed, "shift"), adaln_table(w.base_seed, "scale")


def gated_residual_inputs(w: Workload, rows: int | None = None):
    rows = w.gres_rows if rows is None else rows
    x = randn_bf16((rows, HIDDEN), w.base_seed, "x")
    a = randn_bf16((rows, HIDDEN), w.base_seed, "a")
    return x, a, adaln_table(w.base_seed, "gate")


def sampled_rows(n: int, head: int, k: int) -> torch.Tensor:
    """Query rows checked against the oracle for one head (sorted, unique)."""
    if k <= 0 or k >= n:
        return torch.arange(n)
    g = torch.Generator(device="cpu")
    g.manual_seed(5000 + head)
    pick = torch.randperm(n, generator=g)[:k]
    last_tile = ((n - 1) // TILE) * TILE
    extra = torch.tensor([0, min(1, n - 1), n - 1, last_tile, n - 1])
    return torch.unique(torch.cat([pick, extra]))
