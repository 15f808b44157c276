"""Float64 CPU oracle for the SSD scan -- test infrastructure only.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The CUDA library never does, and this
package never imports the CUDA library.
"""
from .oracle import ssd_fwd_ref, ssd_bwd_ref, oracle_threads, mamba_fwd_ref, mamba_bwd_ref  # noqa: F401
