"""Writes olmoe_rvq_codebooks.npy and olmoe_rvq_codebooks3.npy: the OLMoE-shaped layer's fp16 RVQ
codebook sets with two and with three stages (the first two stages of both are the same).

Calls only the oracle (and the seeded generators).  One codebook pair serves the
whole layer ("a single global codebook", Quantization as Cache Amplification,
section "Codec"): k-means (256 centroids, 25 Lloyd iterations or stable
assignments, lowest-index ties, empty clusters keep their centroid) on a seeded
pool of 2**17 8-dim vectors of the row-normalised rotated weights drawn evenly
from all 64 experts x 3 matrices; stage s is fit on what stages 1 .. s-1 leave.  The three-stage set
serves the frequency-conditioned layer, whose most popular experts use a third stage.

Run from the repository root:  python tests/golden/make_olmoe_rvq_codebooks.py
"""
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import synth  # noqa: E402
from oracle import rvq as R  # noqa: E402

POOL = 1 << 17


def main():
    cfg = synth.OLMOE_RVQ
    per = POOL // (cfg.E * 3)
    rng = np.random.default_rng(np.random.SeedSequence([cfg.seed, synth.TAG_KMEANS]))
    pool = []
    for e in range(cfg.E):
        for m in (synth.GATE, synth.UP, synth.DOWN):
            rows, cols = synth.rvq_matrix_shape(cfg, m)
            w = synth.rvq_weight(cfg.seed, e, m, rows, cols)
            so, si = synth.rvq_signs(cfg.seed, e, m, rows, cols)
            wr = R.rotate_weight(w, so, si)
            u = R.normalised_vectors(wr, R.row_scale_f16(wr), cfg.vec_dim)
            pool.append(u[np.sort(rng.choice(u.shape[0], size=per, replace=False))])
    pool = np.concatenate(pool)
    cb = R.fit_codebooks(pool, k=cfg.codebook_size, iters=25, seed=cfg.seed, stages=3)
    here = os.path.dirname(os.path.abspath(__file__))
    for name, c in (("olmoe_rvq_codebooks.npy", cb[:2]), ("olmoe_rvq_codebooks3.npy", cb)):
        out = os.path.join(here, name)
        np.save(out, c.astype(np.float16))
        print(f"wrote {out}: pool {pool.shape}, codebooks {c.shape}")


if __name__ == "__main__":
    main()
