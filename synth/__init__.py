"""Seeded synthetic inputs for the fusion-group hot path.

This package only draws numbers and lays out workloads: shapes, value
distributions, leaf tables and the random node programs of the large group
workload.  It holds none of the method's arithmetic, so both the CPU oracle
and the CUDA path can take their inputs from it without sharing any code of
the computation they are compared on.

Two generators are used:

* ``host_*`` draws on the host with numpy's Philox4x32-10 bit generator (one
  independent stream per ``(seed, tensor_id)``), turned into uniforms with 53
  random bits and into normals with the Box-Muller transform in float64, then
  rounded once to float32 (and, for bf16 tensors, once more to bf16 by round
  to nearest even).  It is used for every workload the oracle evaluates whole.
* ``device_*`` draws on a CUDA device with torch's Philox-based generator,
  seeded the same way.  It is used for the full-size workloads, whose inputs
  would take minutes to draw on the host; parity at those sizes compares sampled
  outputs, whose inputs are copied back to the host for the oracle.
"""

from .generators import (  # noqa: F401
    host_normal,
    host_uniform,
    host_bf16_bits,
    device_normal,
    device_uniform,
    device_abs_normal,
)
from . import workloads  # noqa: F401
