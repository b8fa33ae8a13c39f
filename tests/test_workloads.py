"""Workload sizes against the numbers the pages print (tests/golden)."""
import json
import os

import numpy as np
import torch

import workloads as W

GOLDEN = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "page_numbers.json")))


def test_geometry_matches_pages():
    g = GOLDEN["geometry"]
    assert W.NUM_HEADS == g["heads"] and W.HEAD_DIM == g["head_dim"]
    assert W.NUM_HEADS * W.HEAD_DIM == g["qkv_width"]
    assert W.HIDDEN == g["hidden"]
    assert W.tokens_per_latent_frame(1344, 768) == g["tokens_per_latent_frame_1344x768"]
    assert (768 // 32, 1344 // 32) == tuple(g["latent_grid_1344x768"])
    assert W.vae_chunk_latent_frames(1) == g["vae_chunk"]["latent_frames"]
    for clip in g["clips"]:
        assert W.latent_frames(clip["frames"]) == clip["latent_frames"]
        if "tokens_1344x768" in clip:
            assert W.video_tokens(1344, 768, clip["frames"]) == clip["tokens_1344x768"]


def test_frame_rounding_rule():
    for f in GOLDEN["fixed_frame_counts"]["frames"]:
        assert (f - 5) % 17 == 0  # already of the form 17n+5: no rounding
        assert W.latent_frames(f) == 5 * ((f - 5) // 17) + 2
    # a frame count between two allowed lengths rounds up to the next 17n+5
    assert W.latent_frames(244) == W.latent_frames(260) == 77
    assert W.latent_frames(1) == 2 and W.latent_frames(5) == 2 and W.latent_frames(6) == 7


def test_activation_sizes_match_pages():
    s = GOLDEN["activation_sizes_bytes_at_102816_tokens"]
    n = 102816
    assert round(n * W.HIDDEN * 2 / 1e9, 2) == s["residual_stream_GB"]
    assert round(3 * n * W.NUM_HEADS * W.HEAD_DIM * 2 / 1e9, 2) == s["qkv_all_heads_GB"]
    assert round(n * n * 2 / 1e9, 1) == s["dense_scores_one_head_GB"]
    assert round(n * 4 * W.HEAD_DIM * 2 / 1e6) == s["four_head_slice_MB"]


def test_adaln_table_sizes_match_pages():
    a = GOLDEN["adaln_bytes_per_modality_timestep_per_layer"]
    assert a["modalities"] * a["vectors"] * a["channels"] == a["projection_rows"]
    assert a["channels"] == W.HIDDEN
    t = W.adaln_table(0, "shift")
    assert t.shape == (W.TABLE_STEPS, W.HIDDEN) and t.dtype == torch.float32


def test_workload_table():
    wl = W.WORKLOADS
    assert [w.n for w in wl.values()] == [1008, 5040, 18144, 72576, 102816]
    assert wl["clip10s_72576"].head_group == 16 and wl["clip14s_102816"].head_group == 8
    assert W.HEADLINE == "clip10s_72576"
    assert abs(wl["clip10s_72576"].flops / 1e12 - 151.0) < 0.1
    for w in wl.values():
        assert w.head_group in GOLDEN["head_groups"]["allowed"]


def test_generators_are_seeded_and_order_free():
    w = W.WORKLOADS["tiny_1008"]
    q1, k1, v1 = W.qkv(w)
    v2 = W.randn_bf16((w.n, w.heads * W.HEAD_DIM), w.base_seed, "v", chunk_rows=100)
    assert torch.equal(v1, v2)
    assert q1.dtype == torch.bfloat16 and q1.shape == (1008, 512)
    assert not torch.equal(q1, k1)
    # N(0, 1) draws
    assert abs(float(q1.float().mean())) < 0.01 and abs(float(q1.float().std()) - 1.0) < 0.01


def test_outlier_channels():
    w = W.WORKLOADS["half_res_18144"]
    cols = W.outlier_channels(w.heads * W.HEAD_DIM)
    assert len(cols) == 72 and len(set(cols.tolist())) == 72
    g = torch.Generator().manual_seed(1000 * w.base_seed + 1)
    k = W.randn_bf16((64, 7168), w.base_seed, "k")  # plain draw for comparison of scale only
    assert k.shape == (64, 7168)


def test_sampled_rows():
    r = W.sampled_rows(72576, 3, 256)
    assert len(r) >= 256 and r[0] == 0 and r[-1] == 72575
    assert 72576 - 1 - ((72576 - 1) % 128) in set(r.tolist())
    assert np.all(np.diff(r.numpy()) > 0)
    assert torch.equal(W.sampled_rows(100, 0, 0), torch.arange(100))
