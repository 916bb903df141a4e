"""CPU oracle for the fused decode-and-multiply path.  TEST INFRASTRUCTURE ONLY.

Plain, slow, obviously-correct float64 restatements of what the pages define:

* ``dictionary`` -- QMoE Algorithm 1 (dictionary generation) and the 64-bit
  entry format of QMoE Figure 4.
* ``codec``      -- the greedy longest-match encoder, the reference decoder and
  the effective-rate ledger.
* ``products``   -- dense float64 matrix-vector / skinny-matrix products.
* ``moe``        -- router, expert bucketing and the MoE feed-forward layer.
* ``rvq``        -- randomized Hadamard transform, k-means residual VQ and the
  transform-aware product.
* ``e8p``        -- the E8P structured lattice codebook (16-bit code words over a
  1 KiB base table), its brute-force nearest-codeword encoder and decoder.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  It shares no code with the CUDA path
(``decode_matvec_gb300``) and never imports it; both take their inputs from the
``synth`` generators.

Citations name the page and its section: [QMoE] is the paper-summary page
"QMoE: Practical Sub-1-Bit Compression of Trillion-Parameter Models";
[QCA] is "Quantization as Cache Amplification: Trillion-Parameter
Mixture-of-Experts Inference on a Commodity Laptop"; [M8.5] is
"M8.5 - Extreme Weight Compression and Representations".

Parity status: every function here is pinned by a ``-m "not gpu"`` test
against closed forms, brute force or values the pages print, except where a
function's docstring says "parity unpinned".
"""
