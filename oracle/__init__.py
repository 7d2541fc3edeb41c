"""fp64 CPU oracle of the SSD layer forward -- test infrastructure only.

Only tests/, ``__graft_entry__.smoke()`` and bench.py's CPU-baseline leg use
this package.  The CUDA library and its Python binding never import it.
"""
from .oracle import (brute_force, build, chunked_reference, linear_attention,
                     quadratic_form, rel_err, s6_brute_force, s6_scan, silu_gate, softplus,
                     ssd_bwd, ssd_scan, ssd_step)

__all__ = ["brute_force", "build", "chunked_reference", "linear_attention",
           "quadratic_form", "rel_err", "s6_brute_force", "s6_scan", "silu_gate", "softplus",
           "ssd_bwd", "ssd_scan", "ssd_step"]
