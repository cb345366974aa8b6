"""TurboQuant hot path on one B300: packed bit-plane KV/DB compression and
scoring behind a small C ABI (``include/tq.h``).  The Python layer only
marshals arguments; every step runs in the CUDA kernels of ``libtq.so``."""
