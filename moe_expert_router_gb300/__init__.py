"""GB300 (sm_103a) MegaMoE expert path at expert parallelism 1.

The compute lives in libmoe.so (CUDA kernels behind the C ABI of include/moe.h);
``binding`` is its ctypes binding, ``workloads`` the seeded input generator and
``build`` compiles the library in-tree.
"""
