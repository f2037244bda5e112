"""CPU oracle for the W4 + input-adaptive error-compensator linear.

Test infrastructure: only ``tests/``, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg import this package. The library never does, and
this package imports nothing from the library.

* ``spear_ref.c`` -- fp64 C implementation (OpenMP over output rows), loaded
  through ctypes by :mod:`oracle.ref`.
* ``brute.py`` -- pure-Python version for tiny shapes that materialises the
  per-token effective weight explicitly.
* ``rtn.py`` -- numpy RTN 4-bit quantiser (fp32 decisions, as the GPU kernel
  takes them) and the truncated-SVD initialisation of the compensator.
"""
