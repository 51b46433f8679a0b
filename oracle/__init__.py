"""Plain fp64 CPU oracle for the quantised-KV attention path.

TEST INFRASTRUCTURE ONLY.  Nothing in the product package imports, calls or
links this package; only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` use it.  It shares
no code with the CUDA path: it has its own quantiser, packer, window planner,
attention, k-means and PCA, each written from the method descriptions cited in
the module docstrings.

Sources (web pages on KV-cache quantisation for video generation):

* "Quantized Keys Steal Attention: Bias Correction for KV-Cache Compression in
  Video Diffusion" (arXiv 2605.26266), abstract: chunk-wise KV cache, INT2 keys
  with per-key step sizes, the Jensen bias and its second-order correction.
* "QuantWM: Temporally Consistent 2-Bit KV Cache Quantization for Video World
  Models", Innovations / Methodology: QSAC codebook keys and PSAC low-rank key
  compensation along the dominant query subspace.
* "WindowQuant" paper note (zenn.dev), sections 何が新しいのか, 技術的に面白い点 and
  実装者視点で気になった点: 32-token windows, FP16/INT4/INT2 by similarity,
  first window FP16, windows grouped by bit-width in memory.

The pages give no formulas; every equation here is an explicit reading, listed
with its justification in the repository's design notes.

Parity pins: every function is pinned by ``tests/test_oracle_*.py`` against
exact rational arithmetic, closed forms, brute force or library routines.
"""

from . import quant, layout, window, attention, codebook, psac  # noqa: F401
