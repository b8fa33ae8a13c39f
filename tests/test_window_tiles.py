"""The windowed attention's K/V tile lists, checked on the host against the
window rule itself ("FreeVideo: a 66 GB video transformer on an 8 GB card",
section "Where Video DeltaNet comes in": each query chunk of five latent frames
sees itself and its neighbours, every frame sees the first and the last latent
frame, and those two frames see everything).

The kernel visits, for each block of 256 query rows, only the K/V tiles of 128
keys that some row of the block may see, as up to three merged tile ranges
(csrc/attn_fwd.cu, window_kv_list, shared by the host's unit table and every
role of the kernel).  A small host program compiled from that source prints the
lists; here they are rebuilt frame by frame from the rule: a tile is visited
exactly when one of its keys lies in a frame that one of the block's rows
sees.  Any slip in the range arithmetic (a chunk edge off by one, a merge of
ranges that do not touch, a missed anchor) changes some list.  No GPU is
used: only the host side of the source is run."""
import os
import subprocess

import numpy as np
import pytest

from video_diffusion_transformer_gb300 import build as fvbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "video_diffusion_transformer_gb300", "csrc")
KV_ROWS, UNIT_ROWS = 128, 256

HARNESS = r'''
#include "attn_fwd.cu"
#include <cstdio>
namespace fv {
int64_t take_test_skip_load(int) { return -1; }   // the launch path is not used here
}
int main() {
    long long n;
    int t, c, w;
    while (std::scanf("%lld %d %d %d", &n, &t, &c, &w) == 4) {
        const int kv_tiles = (int)((n + 127) / 128), q_blocks = (int)((n + 255) / 256);
        for (int qb = 0; qb < q_blocks; ++qb) {
            const fv::KvList l = fv::window_kv_list((int)n, kv_tiles, t, c, w, qb);
            std::printf("%d", l.count);
            for (int i = 0; i < l.count; ++i) std::printf(" %d", l.tile(i));
            std::printf("\n");
        }
    }
    return 0;
}
'''


@pytest.fixture(scope="module")
def lister(tmp_path_factory):
    nvcc = fvbuild.nvcc()
    d = tmp_path_factory.mktemp("window_tiles")
    src, exe = d / "window_tiles_main.cu", d / "window_tiles_main"
    src.write_text(HARNESS)
    cmd = [nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O1", "-std=c++17", "--expt-relaxed-constexpr",
           "-I" + os.path.join(ROOT, "include"), "-I" + CSRC, "-o", str(exe), str(src)]
    try:
        res = subprocess.run(cmd, capture_output=True, text=True, timeout=600)
    except FileNotFoundError:
        pytest.skip("nvcc not available")
    assert res.returncode == 0, res.stdout + res.stderr

    def run(geos):
        text = "".join(f"{n} {t} {c} {w}\n" for n, t, c, w in geos)
        out = subprocess.run([str(exe)], input=text, capture_output=True, text=True, timeout=600, check=True)
        lines = out.stdout.split("\n")
        res, pos = [], 0
        for n, _, _, _ in geos:
            blocks = []
            for _ in range((n + UNIT_ROWS - 1) // UNIT_ROWS):
                v = [int(x) for x in lines[pos].split()]
                pos += 1
                assert v[0] == len(v) - 1
                blocks.append(np.array(v[1:], dtype=np.int64))
            res.append(blocks)
        return res

    return run


def tiles_by_rule(n, t, c, w, qb):
    """K/V tiles holding a key that some row of query block qb sees."""
    frames = n // t
    r0, r1 = qb * UNIT_ROWS, min(n, qb * UNIT_ROWS + UNIT_ROWS)
    g = np.arange(frames)
    seen = np.zeros(frames, dtype=bool)
    for f in range(r0 // t, (r1 - 1) // t + 1):
        if f == 0 or f == frames - 1:
            seen[:] = True
            break
        seen |= (g == 0) | (g == frames - 1) | (np.abs(g // c - f // c) <= w)
    kv_tiles = (n + KV_ROWS - 1) // KV_ROWS
    keys = np.zeros(kv_tiles * KV_ROWS, dtype=bool)
    keys[:n] = np.repeat(seen, t)
    return np.nonzero(keys.reshape(kv_tiles, KV_ROWS).any(axis=1))[0]


def check(lister, geos):
    for (n, t, c, w), blocks in zip(geos, lister(geos)):
        for qb, got in enumerate(blocks):
            ref = tiles_by_rule(n, t, c, w, qb)
            assert np.array_equal(got, ref), ((n, t, c, w), qb, got.tolist(), ref.tolist())


def test_model_geometries(lister):
    """10 s and 14 s clips and a single chunk at 1344x768 (1,008 tokens a
    latent frame, chunks of 5, one chunk either side); the 10 s clip at groups
    of 2 and at no neighbour."""
    check(lister, [(72 * 1008, 1008, 5, 1), (102 * 1008, 1008, 5, 1), (3 * 1008, 1008, 5, 1),
                   (72 * 1008, 1008, 2, 1), (72 * 1008, 1008, 5, 0)])


def test_edge_geometries(lister):
    """Frames shorter than a tile, one token a frame, a single frame, windows
    wider than the clip, chunks of one frame."""
    check(lister, [(1 * 1008, 1008, 5, 1), (2 * 64, 64, 5, 1), (400, 1, 3, 2), (37 * 17, 17, 1, 0),
                   (12 * 100, 100, 2, 6), (9 * 128, 128, 1, 0), (40 * 129, 129, 4, 1)])


def test_seeded_random_geometries(lister):
    rng = np.random.default_rng(2026)
    geos = []
    for _ in range(400):
        t = int(rng.choice([int(rng.integers(1, 64)), int(rng.integers(64, 400)), int(rng.integers(400, 1300))]))
        frames = int(rng.integers(1, max(2, min(90, 40000 // t))))
        geos.append((frames * t, t, int(rng.integers(1, 8)), int(rng.integers(0, 5))))
    check(lister, geos)
