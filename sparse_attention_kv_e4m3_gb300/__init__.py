"""CSA indexer for GB300: FP8 paged compressed-K scoring and top-k selection.

The compute lives in the C-ABI library `libcsa_index.so` (hand-written CUDA for
sm_103a, see include/csa_index.h). This package holds the thin Python binding
(`native`), its build step (`build`) and the seeded synthetic workloads
(`synth`). Importing the package does not load the library; the first call into
`native` does, and raises if it is missing.
"""
__all__ = ["native", "synth", "build"]
