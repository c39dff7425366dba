"""CPU oracle for the OSCAR INT2 rotated paged KV cache (write + decode).

TEST INFRASTRUCTURE ONLY.  This package is a plain, slow, float64 NumPy
restatement of what the serving path computes, written from the OSCAR pages
("OSCAR: Offline Spectral Covariance-Aware Rotation for 2-bit KV Cache
Quantization": the arXiv abstract and the gist.science technical summaries).
It exists so the CUDA path can be checked against something independent.

Only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` may import it.  The product package
never imports it and shares no code with it; the two meet only through the
seeded generators in ``synthetic``.

Modules
-------
rotation   Sylvester Hadamard, bit-reversal permutation, the calibration
           covariances C_Q and C_S, the eigenbasis, R = U.H.P, clip thresholds.
quant      BF16 rounding, per-group asymmetric 2-bit min/max quantiser, the
           packed code layouts of K and V rows.
cache      the paged mixed-precision cache image: INT2 page pool + BF16
           sink/recent window; prefill/extend write, append-with-eviction.
attention  decode attention over the mixed cache (plain and fused forms) and
           textbook attention over an all-BF16 paged cache.

Pinning status: every function here is pinned by ``tests/test_oracle_pins.py``
(closed forms, brute force on tiny inputs, invariants).  Two things stay
"parity unpinned" because the pages print no numbers for them: the end-to-end
accuracy benefit of OSCAR's rotation (needs trained weights and datasets) and
the pages' own kernel outputs.
"""
from . import rotation, quant, cache, attention  # noqa: F401
