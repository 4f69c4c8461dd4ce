"""Plain CPU oracle for the packed 2-bit GEMV path.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and
the CPU-baseline leg of ``bench.py`` may import or run anything in this
package; the product path (``dequant_gemv_q2_gb300``) never does, and this
package never imports the product.  Both sides take their inputs from the
seeded generators in ``synth``.

Each format's module decodes the canonical representation into exact f64
weights, written the way the source pages state the format, and
``matvec`` forms ``y_ref[t][r] = sum_c w64[r][c] * x[t][c]`` in f64 together
with the per-output tolerance bound ``sum_c |w64[r][c] * x[t][c]|``.

Modules:
  bpdq     -- two bit-planes + per-(group, row) coefficients
              ("Qwen3-8B -- 2-bit BPDQ (packed)", section Format)
  trellis  -- bitshift trellis, L=16, T=4, V=2, table codebook
              ("Qwen3.8-27B on a 12 GB card", section "A trellis is a
              codebook you walk")
  leech    -- Leech-lattice blocks of 24 weights, Golay construction
              ("Unfolding the Leech Lattice", introduction and section 7)
  fp16     -- the dense fp16 control
  matvec   -- f64 reference product and the pass criterion
  rotate   -- the activation rotation x_rot = (H (x) Q)(S x) applied ahead
              of the GEMV ("Qwen3.8-27B on a 12 GB card", section "What
              the kernel does per token")

Parity status: every decode function is pinned by closed forms, special
cases or page-printed values in ``tests/test_oracle_*.py``.  The trellis
window orientation is pinned by the page's worked example; the choice of a
tail-biting window inside each 256-column segment and the reading of the
sign bit are readings of the pages, not page facts.
"""
