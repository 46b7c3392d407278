"""CPU oracle for sorting-free top-k / top-p / min-p sampling.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path imports, links or runs
anything in this package; only the tests, ``__graft_entry__.smoke()`` and the
benchmark's ``cpu_baseline`` / ``--impl reference`` legs may.  It shares no code
with the CUDA library (``min_sampling_gb300``): no kernels, headers, helpers or
tables, and it imports nothing from it.

Sources (three web pages on one subject):
  [blog]      "Sorting-Free GPU Kernels for LLM Sampling" (FlashInfer blog, Chinese
              translation): sections Top-K / Top-P / Min-P, inverse transform
              sampling, rejection sampling, dual-pivot rejection sampling, the
              correctness proof (theorem and recurrence (star)), implementation
              details.
  [drill]     "F4: top-k / top-p without sorting" (GPU kernel drills hint page):
              sections 1-8 (worked row, bisection on count/mass, bisection on the
              fp32 bit pattern, pitfalls).
  [explainer] "FlashInfer sorting-free sampling" explainer: sections on the
              sampling pipeline (allowed set S and renormalised p~), Top-k, Top-p,
              Min-p, filter order, dual-pivot cases, numeric pitfalls, RNG
              ownership and the statistical test methodology.

Modules:
  filters      allowed sets, renormalised distributions, renorm / mask outputs (float64, sort-based)
  bruteforce   membership by counting, no sorting (small V)
  philox       Philox4x32-10 counter-based generator (Salmon et al., SC'11)
  dual_pivot   the dual-pivot rejection sampler as the pages state it; exact
               Markov-chain evaluation of its output law (small V)
  baseline     sort-based reference sampler used as the timed CPU baseline
  speculative  chain speculative-sampling verification (Leviathan et al. 2023; Chen et al. 2023)
"""
