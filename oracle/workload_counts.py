"""Counts of a benchmark workload measured by the oracle (TEST INFRASTRUCTURE).

Runs the float64 oracle on one view of a configuration (default: the outdoor scene, 1.6M
Gaussians, 1297x840, seeded) and writes profiles/workload_counts_<name>.md: duplicates D, (pixel,
Gaussian) pairs evaluated and blended, active (16x8 pixel block, Gaussian) and (tile, Gaussian)
pairs with the histogram, over the active blocks, of the lanes with a blending pixel (the backward
kernel's warp covers a 16x8 block with a column of four pixels per lane: the per-warp popcount of
DISTWAR's observations), and the algorithmic bytes of the backward raster:
    per tile, its list up to the largest contributor count x (4-byte index + 48-byte record),
    + per pixel 20 bytes (dL/dpixel, T_final, contributor count),
    + per Gaussian 48 bytes (the 2D gradient record written).
    pairs replayed by the backward: the sum over pixels of the contributor count (each pixel's list
    is replayed back to front from its last contributor).
The benchmark divides these by measured kernel times; nothing of the CUDA library is used here.

    python -m oracle.workload_counts [config]      (2 = outdoor, 4 = contention, ...)
"""
from __future__ import annotations

import json
import os
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import gs_scenes  # noqa: E402
import oracle  # noqa: E402

NAMES = {0: "tiny", 1: "object", 2: "outdoor", 3: "large", 4: "contention"}


def counts(cfg: int = 2) -> dict:
    s = gs_scenes.make_scene(cfg, views=1 if cfg == 3 else None)
    cam = s.cameras[0]
    t0 = time.perf_counter()
    out = oracle.view_step(s)
    dt = time.perf_counter() - t0
    st = out["bwd_stats"]
    nc = out["fwd"]["n_contrib"]
    ranges = out["ranges"]
    TX = cam.tiles_x
    ys, xs = np.mgrid[0:cam.height, 0:cam.width]
    tile = (ys // 16) * TX + xs // 16
    tmax = np.zeros(cam.n_tiles, np.int64)
    np.maximum.at(tmax, tile.ravel(), nc.ravel().astype(np.int64))
    tlen = (ranges[:, 1].astype(np.int64) - ranges[:, 0].astype(np.int64))
    listed = int(np.minimum(tlen, tmax).sum())
    P = cam.width * cam.height
    return {"workload": f"{NAMES[cfg]} {s.n} Gaussians {cam.width}x{cam.height} seed {cfg}", "n_gaussians": s.n,
            "pixels": P, "duplicates": int(len(out["vals"])), "pairs_evaluated": int(st["pairs_evaluated"]),
            "pairs_blended": int(st["pairs_blended"]), "warp_gauss_active": int(st["warp_gauss_active"]),
            "tile_gauss_active": int(st["tile_gauss_active"]), "lane_hist": [int(v) for v in st["lane_hist"]],
            "bwd_list_entries": listed, "bwd_bytes": listed * 52 + P * 20 + s.n * 48,
            "pairs_replayed_bwd": int(nc.astype(np.int64).sum()),
            "marginal_pixels": int(st["marginal_pixels"]), "oracle_seconds": dt, "threads": os.cpu_count()}


def main():
    cfg = int(sys.argv[1]) if len(sys.argv) > 1 else 2
    c = counts(cfg)
    path = os.path.join(ROOT, "profiles", f"workload_counts_{NAMES[cfg]}.md")
    hist = c["lane_hist"]
    active = max(1, sum(hist))
    with open(path, "w") as f:
        f.write(f"# Workload counts: {c['workload']}\n\n")
        f.write(f"Written by `python -m oracle.workload_counts {cfg}` (float64 oracle only). The benchmark's\n")
        f.write("roofline numerators use `pairs_replayed_bwd`, `pairs_blended` and `bwd_bytes`.\n\n")
        f.write(f"- duplicates D = {c['duplicates']:,}\n- pairs evaluated = {c['pairs_evaluated']:,}\n")
        f.write(f"- pairs blended = {c['pairs_blended']:,}\n")
        f.write(f"- pairs replayed by the backward (sum of contributor counts) = {c['pairs_replayed_bwd']:,}\n")
        f.write(f"- active (16x8 block, Gaussian) = {c['warp_gauss_active']:,}; "
                f"active (tile, Gaussian) = {c['tile_gauss_active']:,}\n")
        f.write("- lanes with a blending pixel per active (16x8 block, Gaussian), the warp's popcount: "
                f"all 32 in {hist[32] / active:.1%}, at least 28 in {sum(hist[28:]) / active:.1%}, "
                f"at most 4 in {sum(hist[1:5]) / active:.1%}; mean {sum(i * h for i, h in enumerate(hist)) / active:.1f}\n\n")
        f.write("| lanes | active blocks | share |\n|---|---|---|\n")
        for lo, hi in ((1, 4), (5, 8), (9, 12), (13, 16), (17, 20), (21, 24), (25, 27), (28, 31), (32, 32)):
            n = sum(hist[lo:hi + 1])
            f.write(f"| {lo}-{hi} | {n:,} | {n / active:.1%} |\n" if lo != hi else f"| {lo} | {n:,} | {n / active:.1%} |\n")
        f.write("\n```json\n" + json.dumps(c) + "\n```\n")
    print(path)


if __name__ == "__main__":
    main()
