"""Write float64 oracle outputs of full-size decodes to test fixtures.

    python tests/golden/make_decode_samples.py kl_zimage_512 [kl_zimage_1024 ...]

For each named workload this runs the oracle's dense decode (whole image, no
bands) on the workload's seeded latent and seeded weights, and writes
``decode_full_<workload>.npz`` (float64 results rounded once to float32):

* image decoders (output [B, 3, H, W]): ``out``, the complete output;
* video decoders (output [B, 3, T, H, W]): ``frames`` (frame indices: the
  first, the middle and the last frame) with ``frame_out`` [B, 3, len(frames),
  H, W], their complete outputs; and ``rows`` (every output row within three
  rows of a band boundary of the workload's band schedule, where the halo rows
  of every layer meet) with ``row_out`` [B, 3, T, len(rows), W], those rows in
  every frame.

Every file also holds ``shape`` (the whole output's shape) and ``l2norm`` (the
float64 L2 norm of the whole output).  Float32 storage moves a value by at most
2^-24 of itself, far below the bf16 bars the fixtures are checked against.

Only ``synth`` (seeded inputs) and ``oracle`` are used; nothing here touches the
CUDA library.  A full-size decode takes minutes to an hour of CPU time.
"""
from __future__ import annotations

import os
import sys
import time

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(os.path.dirname(HERE))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import synth  # noqa: E402
from oracle import decoder as odec  # noqa: E402

EDGE_ROWS = 3           # rows kept on each side of a band boundary (video decoders)


def boundary_rows(arch, latent_shape, n_bands, h_out):
    """Output rows within EDGE_ROWS of a band boundary of the band schedule."""
    f = h_out // latent_shape[-2]               # output rows per latent row
    rows, r0 = [], 0
    for r in odec.band_rows(latent_shape[-2], n_bands)[:-1]:
        r0 += r
        e = r0 * f
        rows.extend(y for y in range(e - EDGE_ROWS, e + EDGE_ROWS) if 0 <= y < h_out)
    return np.array(sorted(set(rows)), np.int64)


def fixture_arrays(y: np.ndarray, w) -> dict:
    arrays = dict(shape=np.array(y.shape, np.int64),
                  l2norm=np.array(float(np.linalg.norm(y.reshape(-1)))))
    if y.ndim == 4:
        arrays["out"] = y.astype(np.float32)
        return arrays
    t = y.shape[2]
    frames = np.array(sorted({0, t // 2, t - 1}), np.int64)
    rows = boundary_rows(w.arch, w.latent_shape, w.n_bands, y.shape[3])
    arrays["frames"] = frames
    arrays["frame_out"] = np.ascontiguousarray(y[:, :, frames]).astype(np.float32)
    arrays["rows"] = rows
    arrays["row_out"] = np.ascontiguousarray(y[:, :, :, rows]).astype(np.float32)
    return arrays


def main(names):
    for name in names:
        w = synth.WORKLOADS[name]
        W = synth.make_weights(w.arch, w.dtype)
        z = synth.make_latent(w.latent_shape, w.dtype)
        t0 = time.time()
        y = odec.decode(w.arch, W, z, None)
        dt = time.time() - t0
        arrays = fixture_arrays(y, w)
        arrays["note"] = np.array(
            f"float64 oracle dense decode of workload {name}: {w.description}; written by "
            f"tests/golden/make_decode_samples.py (oracle only); decode took {dt:.0f} s on "
            f"{os.cpu_count()} cores")
        path = os.path.join(HERE, f"decode_full_{name}.npz")
        np.savez_compressed(path, **arrays)
        print(f"{name}: decode {dt:.0f} s -> {path}", flush=True)


if __name__ == "__main__":
    main(sys.argv[1:] or ["kl_zimage_512"])
