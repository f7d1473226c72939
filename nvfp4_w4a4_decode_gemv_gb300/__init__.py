"""NVFP4 W4A4 small-M decode path for GB300 (sm_103a).

The kernels live in libnvfp4_gb300.so (C ABI: include/nvfp4.h); this package
binds them (``api``), builds them (``build``) and generates the seeded
synthetic workloads used by the tests and the benchmark (``synth``).
Importing the package loads nothing; the first call into ``api`` loads the
library and raises if it has not been built.
"""
__version__ = "1.0.0"
