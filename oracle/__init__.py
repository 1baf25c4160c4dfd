"""Plain, slow CPU oracle for the mixture-of-experts layer.

TEST INFRASTRUCTURE ONLY.  This package is imported by ``tests/``, by
``__graft_entry__.smoke()`` and by the ``cpu_baseline`` / ``--impl reference``
legs of ``bench.py``; nothing in the product package may import it, and it
imports nothing from the product package.  It shares no kernels, helpers,
tables or constants with the CUDA path.

Everything is NumPy in float64.  Each function cites the passage of the
"Mixture-of-Kittens" pages (or the OCP Microscaling v1.0 format definition
that the MXFP8 configurations name) it follows.

Modules
-------
numerics : bfloat16 rounding, the OCP E4M3 code table, E4M3 encoding
           (brute force and sorted-table), MXFP8 block quantisation.
moe      : router top-k, device schedule (histogram, scan, stable
           permutation), expert SwiGLU FFNs, deterministic combine, shared
           expert, and the backward pass (chain rule, closed-form dlogits).

Parity pins (what ties this oracle to something other than itself) live in
``tests/test_oracle_*.py``; every public function here is pinned there.
"""
