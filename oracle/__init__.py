"""CPU oracle for the NVFP4 W4A4 small-M decode path and the ReSET sampler.

TEST INFRASTRUCTURE ONLY.  This package is a plain, slow, obviously correct
restatement of what the decode path computes, written from the ReSET pages:

* the NVFP4 format -- E2M1 4-bit elements, one E4M3 scale per 16-element
  block, one FP32 global scale per tensor (ReSET reading note, §2.1 and the
  §6.1 experimental setup);
* the small-M projection Y = dequant(Xq) . dequant(Wq)^T that the CUDA-core
  kernel computes (ReSET project page, "Core contribution -- the nvfp4r
  CUDA-core kernel");
* the ReSET step-aware temperature rule: token entropy, the online step-entropy
  estimate, the step-aware threshold and the two-temperature sample (ReSET
  reading note, §3.1, §3.2, §4.1-§4.3; project page, "Step-aware temperature
  scaling").

It shares no code with the CUDA library and imports nothing from it.  Only
``tests/``, ``__graft_entry__.smoke()`` and ``bench.py`` (its CPU-baseline and
reference legs) may import it; the product path never routes through it.

Precision: the quantize recipe is FP32 IEEE exactly as written (numpy float32
operations round once per operation, which is what the recipe specifies);
everything after dequantization is FP64.

Parity pins: every function here is pinned by tests under ``tests/`` marked
``not gpu`` (hand-worked encodings, exhaustive code enumeration, an independent
library's FP4/FP8 casts, closed-form entropies, brute force on tiny inputs).
Parity unpinned: none.
"""
