"""Write sampled float64 oracle outputs of full-size decodes to text fixtures.

    python tests/golden/make_decode_samples.py kl_zimage_512 [kl_zimage_1024 ...]

For each named workload this runs the oracle's dense decode (whole image, no
bands) on the workload's seeded latent and seeded weights, and writes
``decode_samples_<workload>.txt``: a header with the output shape and the
output's L2 norm, then one line per sampled output element, ``flat_index value``.
The positions are drawn with a fixed seed: uniformly over the whole output, plus
extra positions on the two output rows on each side of every band boundary of the
workload's band schedule (where the halo rows of every layer meet).

Only ``synth`` (seeded inputs) and ``oracle`` are used; nothing here touches the
CUDA library.  A full-size decode takes minutes of CPU time per workload.
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

N_UNIFORM = 3000
N_PER_EDGE_ROW = 64
SEED = 20261202


def sample_positions(shape, arch, latent_shape, n_bands):
    """Flat indices: uniform samples plus samples on rows next to band boundaries."""
    rng = np.random.default_rng(SEED)
    total = int(np.prod(shape))
    idx = set(int(i) for i in rng.integers(0, total, N_UNIFORM))
    # output rows per latent row
    f = 2 ** sum(1 for u in arch.stage_upsample if u)
    rows = odec.band_rows(latent_shape[-2], n_bands)
    h_out, w_out = shape[-2], shape[-1]
    edges, r0 = [], 0
    for r in rows[:-1]:
        r0 += r
        edges.append(r0 * f)
    lead = shape[:-2]
    for e in edges:
        for y in (e - 2, e - 1, e, e + 1):
            if not 0 <= y < h_out:
                continue
            for _ in range(N_PER_EDGE_ROW):
                lead_idx = tuple(int(rng.integers(0, n)) for n in lead)
                x = int(rng.integers(0, w_out))
                idx.add(int(np.ravel_multi_index(lead_idx + (y, x), shape)))
    return np.array(sorted(idx), dtype=np.int64)


def main(names):
    for name in names:
        w = synth.WORKLOADS[name]
        W = synth.make_weights(w.arch, w.dtype)
        z = synth.make_latent(w.latent_shape, w.dtype)
        t0 = time.time()
        y = odec.decode(w.arch, W, z, None)
        dt = time.time() - t0
        pos = sample_positions(y.shape, w.arch, w.latent_shape, w.n_bands)
        flat = y.reshape(-1)
        path = os.path.join(HERE, f"decode_samples_{name}.txt")
        with open(path, "w") as fh:
            fh.write(f"# float64 oracle dense decode of workload {name}: {w.description}\n")
            fh.write("# written by tests/golden/make_decode_samples.py (oracle only); "
                     f"decode took {dt:.0f} s on {os.cpu_count()} cores\n")
            fh.write("shape " + " ".join(str(s) for s in y.shape) + "\n")
            fh.write(f"l2norm {float(np.linalg.norm(flat)):.12e}\n")
            fh.write(f"samples {len(pos)}\n")
            for i in pos:
                fh.write(f"{int(i)} {float(flat[i]):.9e}\n")
        print(f"{name}: {len(pos)} samples, decode {dt:.0f} s -> {path}", flush=True)


if __name__ == "__main__":
    main(sys.argv[1:] or ["kl_zimage_512"])
