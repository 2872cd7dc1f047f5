"""CPU oracle for the Mamba-2 SSD varlen forward prefill scan.

TEST INFRASTRUCTURE ONLY: imported by the tests, by the smoke check and by the
benchmark's CPU-baseline / reference leg, never by the product path.  It shares
no code with the CUDA path.

Three independent fp64 formulations live here, each written from the pages:

* ``recurrence.ssd_varlen_fwd`` -- THE oracle.  The per-token recurrence of the
  "Per-token recurrence" section of the Modular page "mamba2_ssd_scan",
  implemented in C (``ssd_oracle.c``) and called through ctypes.
* ``quadratic.ssd_varlen_fwd`` -- brute force: the materialised lower-triangular
  (C B^T o exp(segsum) o dt) matrix applied to X, with each segment sum added up
  term by term.  Used only to pin the oracle on small inputs.
* ``chunked.ssd_varlen_fwd`` -- the chunked SSD form described on the
  kernelindex page "Mamba chunk scan with segsum" (intra-chunk diagonal
  blocks, per-chunk states, inter-chunk state passing with exponential decay,
  off-diagonal contribution), in NumPy fp64 with a free chunk size.  Used to
  pin chunk-size invariance and as a per-stage reference.
"""
from . import recurrence, quadratic, chunked  # noqa: F401
