"""GPU parity of the attention kernel against the fp64 oracle, through the C ABI."""
import math

import numpy as np
import pytest
import torch

import oracle
import video_diffusion_transformer_gb300 as fv
import workloads as W
from tests import parity as P

pytestmark = pytest.mark.gpu
SCALE = 1.0 / math.sqrt(128)


@pytest.fixture(scope="module", autouse=True)
def _lib(cuda_ok):
    from video_diffusion_transformer_gb300 import build
    build.build()
    fv.load_library()


def run(q, k, v, heads, head_group, scale=SCALE, want_lse=True):
    dev = torch.device("cuda")
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    lse = torch.full((heads, q.shape[0]), float("nan"), dtype=torch.float32, device=dev) if want_lse else None
    o = fv.attn_fwd(qd, kd, vd, head_group=head_group, scale=scale, lse=lse)
    fv.sync_status()
    return o, lse


def rand(n, heads, seed, mult=1.0):
    g = torch.Generator().manual_seed(seed)
    return [(torch.randn((n, heads * 128), generator=g) * mult).to(torch.bfloat16) for _ in range(3)]


@pytest.mark.parametrize("n", [1, 2, 3, 64, 127, 128, 129, 255, 256, 257, 383, 1000])
def test_small_and_ragged_lengths(n):
    heads = 3
    q, k, v = rand(n, heads, 100 + n)
    for hg in (1, 2, 3):
        o, lse = run(q, k, v, heads, hg)
        P.assert_attention_ok(P.attention_errors(q, k, v, o, heads, 0, SCALE, lse))


@pytest.mark.parametrize("name", ["tiny_1008", "clip17_5040"])
def test_workload_all_rows(name):
    w = W.WORKLOADS[name]
    q, k, v = W.qkv(w)
    o, lse = run(q, k, v, w.heads, w.head_group)
    err = P.attention_errors(q, k, v, o, w.heads, 0, SCALE, lse)
    print(name, err)
    P.assert_attention_ok(err)


@pytest.mark.parametrize("name", ["half_res_18144", "clip10s_72576", "clip14s_102816"])
def test_workload_sampled_rows(name):
    w = W.WORKLOADS[name]
    q, k, v = W.qkv(w)
    o, lse = run(q, k, v, w.heads, w.head_group)
    err = P.attention_errors(q, k, v, o, w.heads, w.rows_per_head, SCALE, lse)
    print(name, err)
    P.assert_attention_ok(err)


def test_maximum_head_count():
    """H = 256, the largest head count the ABI takes, at a ragged length: one
    launch of all heads, ragged groups of 7 and one head per launch give the
    same bits, and every head matches the oracle (sampled heads across the
    range, all rows)."""
    n, heads = 300, 256
    q, k, v = rand(n, heads, 256)
    outs = []
    for hg in (256, 7, 1):
        o, lse = run(q, k, v, heads, hg)
        outs.append((o, lse))
    for o, lse in outs[1:]:
        assert torch.equal(o, outs[0][0]) and torch.equal(lse, outs[0][1])
    o, lse = outs[0]
    err = P.attention_errors(q, k, v, o, heads, 0, SCALE, lse, head_list=[0, 1, 100, 127, 128, 200, 254, 255])
    P.assert_attention_ok(err)


@pytest.mark.parametrize("n", [100, 128, 129])
def test_many_short_units_per_cta(n):
    """256 heads of at most two K/V tiles in one launch: each CTA runs one
    (head, query block) unit after another with one or two K/V tiles each,
    so the ring of K/V slots, the P barriers and the thread that waits for
    the loads on the MMA thread's behalf cross unit boundaries every tile or
    two.  Every sampled head matches the oracle on all rows, and one head
    per launch gives the same bits."""
    heads = 256
    q, k, v = rand(n, heads, 400 + n)
    o, lse = run(q, k, v, heads, heads)
    o1, lse1 = run(q, k, v, heads, 1)
    assert torch.equal(o, o1) and torch.equal(lse, lse1)
    err = P.attention_errors(q, k, v, o, heads, 0, SCALE, lse, head_list=[0, 1, 151, 152, 153, 200, 255])
    P.assert_attention_ok(err)


def test_head_grouping_does_not_change_results():
    n, heads = 3000, 6
    q, k, v = rand(n, heads, 7)
    outs = [P.bf16_bits(run(q, k, v, heads, hg, want_lse=False)[0]) for hg in (6, 4, 1, 5)]
    for o in outs[1:]:
        assert np.array_equal(o, outs[0])


def test_deterministic():
    n, heads = 2000, 4
    q, k, v = rand(n, heads, 8)
    a = P.bf16_bits(run(q, k, v, heads, 4)[0])
    b = P.bf16_bits(run(q, k, v, heads, 2)[0])
    assert np.array_equal(a, b)


def test_constant_v_gives_that_vector():
    n, heads = 700, 2
    q, k, _ = rand(n, heads, 9)
    c = torch.randn((1, heads * 128), generator=torch.Generator().manual_seed(10)).to(torch.bfloat16)
    v = c.repeat(n, 1)
    o, _ = run(q, k, v, heads, 2)
    d = P.ulp_distance(P.bf16_bits(o), P.bf16_bits(v))
    assert d.max() <= 1


def test_permuting_keys_and_values():
    n, heads = 1500, 2
    q, k, v = rand(n, heads, 11)
    perm = torch.randperm(n, generator=torch.Generator().manual_seed(12))
    o1, l1 = run(q, k, v, heads, 2)
    o2, l2 = run(q, k[perm].contiguous(), v[perm].contiguous(), heads, 2)
    assert float((o1.float() - o2.float()).abs().max()) <= P.MAX_ABS
    assert float((l1 - l2).abs().max()) <= P.LSE_ABS


def test_scale_zero_gives_mean_of_v():
    n, heads = 513, 2
    q, k, v = rand(n, heads, 13)
    o, lse = run(q, k, v, heads, 2, scale=0.0)
    mean = v.double().mean(dim=0)
    assert float((o.double().cpu() - mean).abs().max()) <= 1e-2
    assert float((lse.cpu() - math.log(n)).abs().max()) <= 1e-4


def test_growing_scores_force_rescales():
    """Scores rise along the keys, so the running maximum grows in every tile
    and the output accumulator is rescaled again and again."""
    n, heads = 1400, 1
    u = torch.randn(128, generator=torch.Generator().manual_seed(14))
    u = u / u.norm()
    t = torch.linspace(-3.0, 9.0, n)
    q = (u * 16.0).repeat(n, 1).to(torch.bfloat16)
    k = (t[:, None] * u[None, :] * 6.0).to(torch.bfloat16)
    v = torch.randn((n, 128), generator=torch.Generator().manual_seed(15)).to(torch.bfloat16)
    o, lse = run(q, k, v, heads, 1)
    err = P.attention_errors(q, k, v, o, heads, 0, SCALE, lse)
    P.assert_attention_ok(err)


def test_large_magnitude_inputs():
    n, heads = 900, 2
    q, k, v = rand(n, heads, 16, mult=4.0)
    o, lse = run(q, k, v, heads, 2)
    err = P.attention_errors(q, k, v, o, heads, 0, SCALE, lse)
    assert err["max_abs"] <= 4 * P.MAX_ABS and err["rel_rms"] <= P.REL_RMS and err["lse_max_abs"] <= 4e-3, err


def test_sync_status_clean():
    fv.sync_status()
