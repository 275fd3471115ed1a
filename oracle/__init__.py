"""CPU fp64 oracle for the channel-wise (UVU) Clebsch-Gordan tensor-product graph convolution.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path imports, links or runs this package:
only the test suite, the smoke check in ``__graft_entry__`` and the CPU-baseline leg of
``bench.py`` may use it.  It shares no code, table or helper with the CUDA library; the one
thing both sides consume is the seeded input generator
(``clebsch_gordan_tensor_receiver_gb300.workloads``), which holds none of the method's
arithmetic.

What the oracle computes follows the convolution described on the page "Receiver-streaming
convolutions for channel-wise UVU tensor products" (OpenEquivariance discussion #221, opening
post) and the CG tensor product + graph convolution of "An Efficient Sparse Kernel Generator for
O(3)-Equivariant Deep Networks" (abstract):

    out[r,u,p,m3] = sum_{e: recv(e)=r} w[e,p,u] sum_{m1,m2} C^p[m1,m2,m3] x[src(e),u,l1,m1] Y[e,l2,m2]

and its vector-Jacobian product with respect to x, Y and w.

Modules
-------
cg       complex CG from the Racah closed form (exact rational arithmetic under one square root),
         change to the real basis, canonical sign.
sh       real spherical harmonics, component-normalised, from an associated-Legendre recursion.
paths    irreps parsing, path enumeration and tensor layouts.
graph    receiver CSR and transposed (sender) CSR, by counting and a stable sort.
conv     forward and VJP as plain fp64 loops in C (``conv.c``), OpenMP over owners.
wigner   real Wigner-D matrices fitted from SH samples (used only by equivariance pins).
hvp      double backward (Hessian-vector product) through substituted forward / VJP calls.
tp       batched (non-convolution) tensor product and its VJP, per-sample or shared weights.
mix      per-path channel mixing that reduces a factorised UVW convolution to the UVU one.
radial   radial weights from edge lengths (Bessel basis, polynomial envelope, SiLU network), the
         convolution that uses them, and the reverse pass (edge-length and layer gradients,
         gradients of the last linear layer).

Parity status: every function here is pinned by ``tests/test_oracle_*.py`` against properties
that the mathematics fixes (orthogonality, completeness, closed forms for l <= 1, intertwining
under random rotations, finite differences, adjoint identities, a sparse-matrix special case and
a dense brute force).  The pages print no worked numerical example of this operation, so no
golden value comes from them; ``tests/golden/`` holds closed-form values derived by hand.
"""

from . import cg, sh, paths, graph, conv, wigner, hvp, tp, mix, radial  # noqa: F401
