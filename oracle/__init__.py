"""Plain, slow FP64 CPU oracle for the fused Clebsch-Gordan tensor-product convolution.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path may import this package:
only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` / ``--impl
reference`` legs of ``bench.py`` use it.  It shares no code, tables or constants
with the CUDA library under ``clebsch_gordan_tensor_racah_gb300/csrc``.

What it follows (pages of the method, by title and section):

* "An Efficient Sparse Kernel Generator for O(3)-Equivariant Deep Networks"
  (OpenEquivariance), Abstract and Figure 1: the CG tensor product contracts a
  block-sparse coefficient tensor with two dense vectors and is followed by a
  structured weight multiplication; Figure 4B: the same product embedded in a
  graph convolution that sums edge messages into the receiving node.
* "Sobek: Streaming Equivariant Tensor Product Convolutions", Abstract: the
  fully connected (uvw) multiplicity mixing with radial projection; the
  oracle forms each edge's weights W_e = sum_k R[e,k] M[k] explicitly, so the
  streaming reassociation of the CUDA path is checked against the plain
  definition.

The coefficients come from Racah's closed form, evaluated exactly with Python
integers and ``fractions.Fraction`` (``cg.py``).  Every function here is pinned by
``tests/test_oracle_*.py`` against textbook values, orthogonality, closed forms
for l <= 2, rotation/inversion equivariance, brute-force dense contraction and
finite differences.  Nothing is "parity unpinned" except the radial-basis
constants, which only shape an input distribution.
"""

from . import cg, irreps, conv, graph  # noqa: F401
