"""The block-scaled GEMMs' static tile order, walked incrementally
(csrc/tile_walk.cuh), against the direct definition: position t is hot iff
floor((t+1)H/N) > floor(tH/N), then hot tile floor(tH/N), else cold tile
t - floor(tH/N); a list's tile j belongs to the largest group g with
start[g] <= j / MT.  Host code, compiled with g++."""
import os
import subprocess

import numpy as np
import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
HDR = os.path.join(HERE, "..", "deterministic_rl_gb300", "csrc")

PROG = r"""
#include <cstdio>
#include <vector>
#include "tile_walk.cuh"
int main() {
    int GG, MT, first, step;
    if (scanf("%d %d %d %d", &GG, &MT, &first, &step) != 4) return 1;
    std::vector<int> hs(GG + 1), cs(GG + 1);
    for (auto& v : hs) if (scanf("%d", &v) != 1) return 1;
    for (auto& v : cs) if (scanf("%d", &v) != 1) return 1;
    moe::TileOrder o{hs.data(), cs.data(), GG, MT, (uint32_t)(hs[GG] * MT),
                     (uint32_t)((hs[GG] + cs[GG]) * MT)};
    if (step > 0) {
        for (moe::TileWalk w = moe::tile_walk_begin(first, o); w.t >= 0; moe::tile_walk_next(w, step, o)) {
            const moe::TilePos p = moe::tile_walk_pos(w, o);
            printf("%d %d %d %d %d\n", w.t, p.g, p.m, p.nt, (int)p.hot);
        }
    } else {  // positions from stdin, increasing, -1 ends
        moe::TileWalk w = moe::tile_walk_begin(0, o);
        int t;
        while (scanf("%d", &t) == 1 && t >= 0) {
            moe::tile_walk_to(w, t, o);
            const moe::TilePos p = moe::tile_walk_pos(w, o);
            printf("%d %d %d %d %d\n", w.t, p.g, p.m, p.nt, (int)p.hot);
        }
    }
    return 0;
}
"""


@pytest.fixture(scope="module")
def walker(tmp_path_factory):
    d = tmp_path_factory.mktemp("walk")
    src = d / "walk.cpp"
    src.write_text(PROG)
    exe = d / "walk"
    subprocess.run(["g++", "-std=c++17", "-O1", "-I", HDR, str(src), "-o", str(exe)], check=True)
    return str(exe)


def expected(hs, cs, MT, first, step, positions=None):
    GG = len(hs) - 1
    H, N = hs[GG] * MT, (hs[GG] + cs[GG]) * MT

    def group(start, x):  # largest g in [0, GG) with start[g] <= x
        return int(np.searchsorted(np.asarray(start[:GG]), x, side="right")) - 1

    out = []
    for t in (range(first, N, step) if positions is None else positions):
        h0, h1 = t * H // N, (t + 1) * H // N
        if h1 > h0:
            j = h0
            g = group(hs, j // MT)
            ntg = hs[g + 1] - hs[g]
            l = j - hs[g] * MT
            out.append((t, g, l // ntg, l % ntg, 1))
        else:
            j = t - h0
            g = group(cs, j // MT)
            out.append((t, g, j - cs[g] * MT, 0, 0))
    return out


def order_from_counts(ntiles):
    hot = np.where(ntiles > 1, ntiles, 0)
    cold = np.where(ntiles == 1, 1, 0)
    hs = np.concatenate([[0], np.cumsum(hot)]).tolist()
    cs = np.concatenate([[0], np.cumsum(cold)]).tolist()
    return hs, cs


@pytest.mark.parametrize("seed", range(6))
def test_walk_matches_direct_order(walker, seed):
    rng = np.random.default_rng(seed)
    GG = int(rng.choice([1, 3, 17, 384]))
    MT = int(rng.choice([1, 8, 16, 28]))
    # token tiles per group: many empty, cold and hot groups
    ntiles = rng.choice([0, 0, 1, 1, 2, 3, 7], size=GG)
    if ntiles.sum() == 0:
        ntiles[0] = 1
    hs, cs = order_from_counts(ntiles)
    for step in (1, 3, 76):
        for first in sorted({0, step - 1, step // 2}):
            inp = f"{GG} {MT} {first} {step}\n" + " ".join(map(str, hs)) + "\n" + " ".join(map(str, cs)) + "\n"
            got = subprocess.run([walker], input=inp, capture_output=True, text=True, check=True).stdout
            got = [tuple(map(int, line.split())) for line in got.splitlines()]
            assert got == expected(hs, cs, MT, first, step), (GG, MT, first, step)


def test_walk_all_hot_all_cold_and_empty(walker):
    for ntiles in (np.array([2, 3, 4]), np.array([1, 1, 1, 1]), np.array([0, 0, 5, 0])):
        hs, cs = order_from_counts(ntiles)
        for step in (1, 2, 5):
            inp = f"{len(ntiles)} 4 0 {step}\n" + " ".join(map(str, hs)) + "\n" + " ".join(map(str, cs)) + "\n"
            got = subprocess.run([walker], input=inp, capture_output=True, text=True, check=True).stdout
            got = [tuple(map(int, line.split())) for line in got.splitlines()]
            assert got == expected(hs, cs, 4, 0, step)


@pytest.mark.parametrize("seed", range(4))
def test_walk_to_increasing_positions(walker, seed):
    """Tiles handed out by a counter: each reader sees increasing positions
    with arbitrary gaps (tile_walk_to)."""
    rng = np.random.default_rng(100 + seed)
    GG = int(rng.choice([5, 384]))
    MT = int(rng.choice([8, 28]))
    ntiles = rng.choice([0, 1, 1, 2, 4], size=GG)
    ntiles[0] = max(ntiles[0], 1)
    hs, cs = order_from_counts(ntiles)
    N = (hs[-1] + cs[-1]) * MT
    pos = np.sort(rng.choice(N, size=min(N, 200), replace=False)).tolist()
    inp = (f"{GG} {MT} 0 0\n" + " ".join(map(str, hs)) + "\n" + " ".join(map(str, cs)) + "\n"
           + " ".join(map(str, pos)) + " -1\n")
    got = subprocess.run([walker], input=inp, capture_output=True, text=True, check=True).stdout
    got = [tuple(map(int, line.split())) for line in got.splitlines()]
    assert got == expected(hs, cs, MT, 0, 1, positions=pos)
