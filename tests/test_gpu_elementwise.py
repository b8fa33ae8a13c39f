"""GPU parity of the AdaLN modulate and gated-residual kernels against the
fp64 oracle, through the C ABI."""
import numpy as np
import pytest
import torch

import oracle
import video_diffusion_transformer_gb300 as fv
import workloads as W
from tests import parity as P

pytestmark = pytest.mark.gpu
STEP = W.ADALN_STEP
EPS = 1e-6


@pytest.fixture(scope="module", autouse=True)
def _lib(cuda_ok):
    from video_diffusion_transformer_gb300 import build
    build.build()
    fv.load_library()


def check_modulate(x, shift, scale, rows, step=STEP, packed=None):
    dev = torch.device("cuda")
    xd = x.to(dev)
    if packed is None:
        sh_d, sc_d = shift.to(dev), scale.to(dev)
    else:  # strided views into one packed [steps, vectors, C] table
        sh_d, sc_d = packed
    y32 = fv.adaln_modulate(xd, sh_d, sc_d, step, eps=EPS, out_dtype=torch.float32)
    y16 = fv.adaln_modulate(xd, sh_d, sc_d, step, eps=EPS, out_dtype=torch.bfloat16)
    fv.sync_status()
    ref = oracle.modulate(x, shift[step].numpy(), scale[step].numpy(), EPS, rows=rows)
    got32 = y32.cpu().numpy()[rows].astype(np.float64)
    rel = np.abs(got32 - ref) / np.maximum(1.0, np.abs(ref))
    assert rel.max() <= P.MODULATE_REL, rel.max()
    # bf16 output: the bf16 rounding of a value within the float32 tolerance,
    # i.e. |y16 - y| <= half a bf16 step of y + 1e-5 * max(|y|, 1).  (Where y
    # is near zero by cancellation, that can be several bf16 steps of y.)
    got16 = y16.cpu()[rows].double().numpy()
    half_step = np.where(ref != 0, np.exp2(np.floor(np.log2(np.abs(ref) + 1e-300)) - 8), 0.0)
    bound = half_step + P.MODULATE_REL * np.maximum(1.0, np.abs(ref))
    assert np.all(np.abs(got16 - ref) <= bound), float(np.max(np.abs(got16 - ref) - bound))
    assert np.abs(got16 - ref).max() <= P.MAX_ABS and np.abs(got16 - ref).mean() <= P.MEAN_ABS


def test_modulate_tiny_all_rows():
    w = W.WORKLOADS["tiny_1008"]
    x, shift, scale = W.modulate_inputs(w)
    check_modulate(x, shift, scale, np.arange(w.n))


@pytest.mark.parametrize("name", ["clip10s_72576", "clip14s_102816"])
def test_modulate_full_size_sampled_rows(name):
    w = W.WORKLOADS[name]
    x, shift, scale = W.modulate_inputs(w)
    rows = np.unique(np.concatenate([np.arange(0, w.n, 97), [w.n - 1]]))
    check_modulate(x, shift, scale, rows)


def test_modulate_reads_strided_rows_of_a_packed_table():
    """Six vectors per step packed as [steps, 6, C] (shift, scale, gate for
    attention, then for the feed-forward); the call reads two strided views."""
    c, steps = W.HIDDEN, 8
    g = torch.Generator().manual_seed(5)
    packed = (torch.randn((steps, 6, c), generator=g) * 0.1).to(torch.float32)
    x = W.randn_bf16((300, c), 9, "x")
    dev = torch.device("cuda")
    pd = packed.to(dev)
    shift_view, scale_view = pd[:, 0, :], pd[:, 1, :]
    assert shift_view.stride(0) == 6 * c
    for step in (0, 5, 7):
        check_modulate(x, packed[:, 0, :].contiguous(), packed[:, 1, :].contiguous(), np.arange(300), step=step,
                       packed=(shift_view, scale_view))


@pytest.mark.parametrize("c", [8, 256, 1000, 2048, 4096, 5376, 8192])
def test_modulate_other_widths(c):
    x = W.randn_bf16((77, c), 3, "x")
    g = torch.Generator().manual_seed(c)
    shift = (torch.randn((4, c), generator=g) * 0.1).float()
    scale = (torch.randn((4, c), generator=g) * 0.1).float()
    check_modulate(x, shift, scale, np.arange(77), step=2)


def test_modulate_constant_row_gives_shift():
    c = W.HIDDEN
    x = torch.full((4, c), 1.5, dtype=torch.bfloat16)
    shift = W.adaln_table(0, "shift")
    scale = W.adaln_table(0, "scale")
    y = fv.adaln_modulate(x.cuda(), shift.cuda(), scale.cuda(), STEP, out_dtype=torch.float32).cpu()
    assert torch.equal(y, shift[STEP].expand(4, c))


def check_gres(x, a, gate, rows, step=STEP, in_place=False):
    dev = torch.device("cuda")
    xd, ad = x.to(dev), a.to(dev)
    out = fv.gated_residual(xd, ad, gate.to(dev), step, out=xd if in_place else None)
    fv.sync_status()
    _, ref_bits = oracle.gated_residual(x, a, gate[step].numpy(), rows=rows)
    d = P.ulp_distance(P.bf16_bits(out.cpu()[rows]), ref_bits)
    assert d.max() <= 1
    return int((d == 1).sum()), d.size


def test_gated_residual_all_rows():
    w = W.WORKLOADS["clip17_5040"]
    x, a, gate = W.gated_residual_inputs(w)
    ones, total = check_gres(x, a, gate, np.arange(w.n))
    print(f"gated residual: {ones} of {total} elements one bf16 step from the oracle")
    assert ones <= total * 1e-3


def test_gated_residual_in_place():
    w = W.WORKLOADS["clip17_5040"]
    x, a, gate = W.gated_residual_inputs(w, rows=1000)
    check_gres(x, a, gate, np.arange(1000), in_place=True)


@pytest.mark.parametrize("name", ["clip10s_72576", "clip14s_102816"])
def test_gated_residual_full_size_sampled_rows(name):
    w = W.WORKLOADS[name]
    x, a, gate = W.gated_residual_inputs(w)
    rows = np.unique(np.concatenate([np.arange(0, w.n, 61), [w.n - 1]]))
    check_gres(x, a, gate, rows)


@pytest.mark.parametrize("c", [8, 264, 2056, 6000])
def test_gated_residual_other_widths(c):
    x = W.randn_bf16((33, c), 4, "x")
    a = W.randn_bf16((33, c), 4, "a")
    gate = (torch.randn((2, c), generator=torch.Generator().manual_seed(c)) * 0.1).float()
    check_gres(x, a, gate, np.arange(33), step=1)


def test_zero_gate_is_identity():
    w = W.WORKLOADS["clip17_5040"]
    x, a, _ = W.gated_residual_inputs(w, rows=64)
    gate = torch.zeros((8, W.HIDDEN), dtype=torch.float32)
    out = fv.gated_residual(x.cuda(), a.cuda(), gate.cuda(), STEP).cpu()
    assert np.array_equal(P.bf16_bits(out), P.bf16_bits(x))


def test_off_ladder_step_is_rejected():
    x = torch.zeros((8, 64), dtype=torch.bfloat16, device="cuda")
    gate = torch.zeros((8, 64), dtype=torch.float32, device="cuda")
    with pytest.raises(fv.FvError) as e:
        fv.gated_residual(x, x.clone(), gate, 8)
    assert e.value.code == -4
    with pytest.raises(fv.FvError):
        fv.adaln_modulate(x, gate, gate, -1)


def packed_tags(n, gen_seed=3, runs=(300, 200)):
    """[text | audio | video] runs (tags 0, 1, 2), then a stretch of random tags."""
    t = torch.full((n,), 2, dtype=torch.uint8)
    t[:runs[0]] = 0
    t[runs[0]:runs[0] + runs[1]] = 1
    g = torch.Generator().manual_seed(gen_seed)
    tail = n // 3
    t[n - tail:] = torch.randint(0, 3, (tail,), generator=g).to(torch.uint8)
    return t


def test_modulate_tagged_rows():
    n, c, m, steps = 1500, W.HIDDEN, 3, 8
    x = W.randn_bf16((n, c), 11, "x")
    g = torch.Generator().manual_seed(12)
    shift = (torch.randn((steps * m, c), generator=g) * 0.1).float()
    scale = (torch.randn((steps * m, c), generator=g) * 0.1).float()
    tags = packed_tags(n)
    y = fv.adaln_modulate_tagged(x.cuda(), shift.cuda(), scale.cuda(), STEP, tags.cuda(), m, eps=EPS,
                                 out_dtype=torch.float32)
    fv.sync_status()
    y = y.cpu().numpy()
    for tag in range(m):
        rows = np.nonzero(tags.numpy() == tag)[0]
        ref = oracle.modulate(x, shift[STEP * m + tag].numpy(), scale[STEP * m + tag].numpy(), EPS, rows=rows)
        rel = np.abs(y[rows] - ref) / np.maximum(1.0, np.abs(ref))
        assert rel.max() <= P.MODULATE_REL, (tag, rel.max())


@pytest.mark.parametrize("c,m", [(5376, 5), (8192, 2)], ids=["five_modalities_5376", "two_modalities_8192"])
def test_modulate_tagged_rows_through_the_read_only_cache(c, m):
    """Tables too large to stage in shared memory (5 modalities at 5,376
    channels: 215 KB; any width above 5,376) take the kernel that reads each
    token's rows through the read-only cache.  Per tag group it must match the
    oracle, and bit for bit the untagged call with that group's table row
    (the same row code and the same float32 arithmetic)."""
    n, steps = 1200, 4
    step = 2
    x = W.randn_bf16((n, c), 21 + m, "x")
    g = torch.Generator().manual_seed(22 + m)
    shift = (torch.randn((steps * m, c), generator=g) * 0.1).float()
    scale = (torch.randn((steps * m, c), generator=g) * 0.1).float()
    gt = torch.Generator().manual_seed(23)
    tags = torch.randint(0, m, (n,), generator=gt).to(torch.uint8)
    tags[:100] = 0
    tags[100:150] = m - 1
    xd, shd, scd = x.cuda(), shift.cuda(), scale.cuda()
    y = fv.adaln_modulate_tagged(xd, shd, scd, step, tags.cuda(), m, eps=EPS, out_dtype=torch.float32)
    yb = fv.adaln_modulate_tagged(xd, shd, scd, step, tags.cuda(), m, eps=EPS)
    fv.sync_status()
    y, yb = y.cpu(), yb.cpu()
    for tag in range(m):
        rows = np.nonzero(tags.numpy() == tag)[0]
        row = step * m + tag
        ref = oracle.modulate(x, shift[row].numpy(), scale[row].numpy(), EPS, rows=rows)
        rel = np.abs(y.numpy()[rows] - ref) / np.maximum(1.0, np.abs(ref))
        assert rel.max() <= P.MODULATE_REL, (tag, rel.max())
        u = fv.adaln_modulate(xd, shd[row:row + 1], scd[row:row + 1], 0, eps=EPS, out_dtype=torch.float32)
        ub = fv.adaln_modulate(xd, shd[row:row + 1], scd[row:row + 1], 0, eps=EPS)
        fv.sync_status()
        assert torch.equal(y[rows], u.cpu()[rows]), tag
        assert torch.equal(yb[rows], ub.cpu()[rows]), tag


def test_gated_residual_tagged_rows():
    n, c, m, steps = 1500, W.HIDDEN, 3, 8
    x = W.randn_bf16((n, c), 13, "x")
    a = W.randn_bf16((n, c), 13, "a")
    gate = (torch.randn((steps * m, c), generator=torch.Generator().manual_seed(14)) * 0.1).float()
    tags = packed_tags(n, 5)
    out = fv.gated_residual_tagged(x.cuda(), a.cuda(), gate.cuda(), STEP, tags.cuda(), m).cpu()
    fv.sync_status()
    for tag in range(m):
        rows = np.nonzero(tags.numpy() == tag)[0]
        _, ref_bits = oracle.gated_residual(x, a, gate[STEP * m + tag].numpy(), rows=rows)
        assert P.ulp_distance(P.bf16_bits(out[rows]), ref_bits).max() <= 1


def test_single_modality_tags_equal_untagged_call():
    w = W.WORKLOADS["clip17_5040"]
    x, a, gate = W.gated_residual_inputs(w, rows=700)
    tags = torch.zeros(700, dtype=torch.uint8).cuda()
    o1 = fv.gated_residual_tagged(x.cuda(), a.cuda(), gate.cuda(), STEP, tags, 1)
    o2 = fv.gated_residual(x.cuda(), a.cuda(), gate.cuda(), STEP)
    xm, sh, sc = W.modulate_inputs(w, rows=700)
    y1 = fv.adaln_modulate_tagged(xm.cuda(), sh.cuda(), sc.cuda(), STEP, tags, 1, out_dtype=torch.float32)
    y2 = fv.adaln_modulate(xm.cuda(), sh.cuda(), sc.cuda(), STEP, out_dtype=torch.float32)
    fv.sync_status()
    assert torch.equal(o1, o2)
    # the staged tagged modulate runs the untagged kernel's row code
    assert torch.equal(y1, y2)


def test_out_of_range_tag_is_reported_and_context_survives():
    n, c = 64, 256
    x = torch.zeros((n, c), dtype=torch.bfloat16, device="cuda")
    gate = torch.zeros((2 * 3, c), dtype=torch.float32, device="cuda")
    tags = torch.full((n,), 3, dtype=torch.uint8, device="cuda")  # 3 modalities: tags 0..2
    fv.gated_residual_tagged(x, x.clone(), gate, 1, tags, 3)
    with pytest.raises(fv.FvError) as e:
        fv.sync_status()
    assert e.value.code == -8
    fv.sync_status()  # cleared
    tags.fill_(1)
    fv.gated_residual_tagged(x, x.clone(), gate, 1, tags, 3)
    fv.sync_status()
