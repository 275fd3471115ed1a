"""Seeded synthetic workloads for the UVU convolution: graphs, features, edge harmonics, weights.

This module draws inputs only.  It holds none of the convolution's arithmetic (no CG
coefficients, no path rules, no contraction); the callers pass the number of paths and the output
width they obtained from a plan.  Both the CUDA library's tests and benchmark and the CPU oracle
consume the same arrays produced here.

Workloads (graph topology from "Receiver-streaming convolutions for channel-wise UVU tensor
products", opening post, benchmark paragraph: 5,000 nodes, 280,000 edges, uniform degree 56,
receiver-sorted, graph construction untimed):

  0 tiny     N=100,   degree 8 uniform,  x 16x0e+16x1o,          SH lmax 2, lmax_out 2, fp32
  1 medium   N=5000,  degree 56 uniform, x 128x0e+128x1o,        SH lmax 3, lmax_out 3, fp32
  2 large    N=5000,  degree 56 uniform, x 128x0e+128x1o+128x2e, SH lmax 3, lmax_out 3, fp32
  3 wide     N=5000,  degree 56 uniform, x 256x0e+256x1o+256x2e, SH lmax 3, lmax_out 3, fp32
  4 fp64     20,000 atoms uniform in a periodic cube at 0.056 / A^3, all ordered pairs within
             5 A (minimum image), x 64x0e+64x1o+64x2e, SH lmax 3, lmax_out 3, fp64

Random streams: numpy PCG64; workload k uses SeedSequence(20260000 + k).spawn(6) for
(graph, x, vectors, w, d_out, spare).  Values: x ~ N(0,1); unit vectors = normalised N(0, I3)
(for workload 4, the normalised minimum-image bond vectors pos[src] - pos[recv]);
w ~ N(0,1)/sqrt(mean degree); d_out ~ N(0,1).  fp32 workloads draw fp32 normals directly.

Y is the component-normalised real SH of the unit vectors (sum_m Y_lm^2 = 2l+1, Y_1 = sqrt(3)
(y, z, x)), evaluated from the Cartesian polynomials below for lmax <= 3.  It is an input of
the convolution, not part of it.
"""

from __future__ import annotations

from dataclasses import dataclass, field
from math import sqrt

import numpy as np

SEED_BASE = 20260000


@dataclass(frozen=True)
class WorkloadSpec:
    key: int
    name: str
    n_nodes: int
    irreps_x: str
    irreps_sh: str
    lmax_out: int
    dtype: str  # "float32" | "float64"
    graph: str  # "uniform" | "periodic"
    degree: int = 0  # uniform graphs
    density: float = 0.0  # periodic graphs, atoms / A^3
    cutoff: float = 0.0  # periodic graphs, A
    w_scale_degree: float = 1.0
    extra: dict = field(default_factory=dict)

    @property
    def mul(self) -> int:
        return int(self.irreps_x.split("x")[0])

    @property
    def sh_lmax(self) -> int:
        return int(self.irreps_sh.split("+")[-1].split("x")[1][:-1])


SPECS = {
    0: WorkloadSpec(0, "tiny", 100, "16x0e+16x1o", "1x0e+1x1o+1x2e", 2, "float32",
                    "uniform", degree=8, w_scale_degree=8),
    1: WorkloadSpec(1, "mace_medium", 5000, "128x0e+128x1o", "1x0e+1x1o+1x2e+1x3o", 3,
                    "float32", "uniform", degree=56, w_scale_degree=56),
    2: WorkloadSpec(2, "mace_large", 5000, "128x0e+128x1o+128x2e", "1x0e+1x1o+1x2e+1x3o", 3,
                    "float32", "uniform", degree=56, w_scale_degree=56),
    3: WorkloadSpec(3, "wide", 5000, "256x0e+256x1o+256x2e", "1x0e+1x1o+1x2e+1x3o", 3,
                    "float32", "uniform", degree=56, w_scale_degree=56),
    4: WorkloadSpec(4, "irregular_fp64", 20000, "64x0e+64x1o+64x2e", "1x0e+1x1o+1x2e+1x3o", 3,
                    "float64", "periodic", density=0.056, cutoff=5.0, w_scale_degree=29),
}


def streams(key: int):
    ss = np.random.SeedSequence(SEED_BASE + key).spawn(6)
    names = ("graph", "x", "vectors", "w", "d_out", "spare")
    return {n: np.random.Generator(np.random.PCG64(s)) for n, s in zip(names, ss)}


# ----------------------------------------------------------------------------------- graphs

def uniform_graph(n_nodes: int, degree: int, rng: np.random.Generator):
    """Each receiver gets `degree` distinct senders != itself, ascending; receiver-sorted.

    Returns (recv[E], src[E]) as int32."""
    if degree > n_nodes - 1:
        raise ValueError("degree must be < n_nodes")
    src = np.empty((n_nodes, degree), dtype=np.int64)
    for r in range(n_nodes):
        s = rng.choice(n_nodes - 1, size=degree, replace=False)
        s = s + (s >= r)
        s.sort()
        src[r] = s
    recv = np.repeat(np.arange(n_nodes), degree)
    return recv.astype(np.int32), src.reshape(-1).astype(np.int32)


def random_degree_graph(n_nodes: int, degrees: np.ndarray, rng: np.random.Generator):
    """Receiver r gets degrees[r] senders drawn with replacement (self edges allowed) and
    sorted ascending; degree 0 gives an empty receiver.  Used for edge-case graphs."""
    degrees = np.asarray(degrees, dtype=np.int64)
    recv = np.repeat(np.arange(n_nodes), degrees)
    src = np.empty(recv.size, dtype=np.int64)
    pos = 0
    for r in range(n_nodes):
        d = int(degrees[r])
        s = np.sort(rng.integers(0, n_nodes, size=d))
        src[pos:pos + d] = s
        pos += d
    return recv.astype(np.int32), src.astype(np.int32)


def periodic_graph(n_atoms: int, density: float, cutoff: float, rng: np.random.Generator):
    """Atoms uniform in a periodic cube; all ordered pairs within `cutoff` (minimum image).

    Returns (recv[E], src[E], unit_vectors[E,3], box_length); edges sorted by receiver, then
    ascending sender.  The vector of edge e points from its receiver to its sender."""
    from scipy.spatial import cKDTree

    box = (n_atoms / density) ** (1.0 / 3.0)
    if box <= 2 * cutoff:
        raise ValueError("box too small for the minimum-image convention")
    pos = rng.random((n_atoms, 3)) * box
    tree = cKDTree(pos, boxsize=box)
    pairs = tree.query_pairs(r=cutoff, output_type="ndarray")
    a = np.concatenate([pairs[:, 0], pairs[:, 1]])
    b = np.concatenate([pairs[:, 1], pairs[:, 0]])
    order = np.lexsort((b, a))  # receiver a, then sender b
    recv, src = a[order], b[order]
    d = pos[src] - pos[recv]
    d -= box * np.round(d / box)
    vec = d / np.linalg.norm(d, axis=1, keepdims=True)
    return recv.astype(np.int32), src.astype(np.int32), vec, box


def unit_vectors(n: int, rng: np.random.Generator) -> np.ndarray:
    v = rng.standard_normal((n, 3))
    return v / np.linalg.norm(v, axis=1, keepdims=True)


# ----------------------------------------------------------------------- edge harmonics (input)

def sh_inputs(vec: np.ndarray, lmax: int) -> np.ndarray:
    """Component-normalised real SH of unit vectors, layout [n][(lmax+1)^2], fp64, lmax <= 3."""
    if lmax > 3:
        raise ValueError("input SH polynomials are written out for lmax <= 3")
    x, y, z = vec[:, 0], vec[:, 1], vec[:, 2]
    cols = [np.ones_like(x)]
    if lmax >= 1:
        s3 = sqrt(3.0)
        cols += [s3 * y, s3 * z, s3 * x]
    if lmax >= 2:
        s15 = sqrt(15.0)
        cols += [s15 * x * y, s15 * y * z, 0.5 * sqrt(5.0) * (3 * z * z - 1), s15 * x * z,
                 0.5 * s15 * (x * x - y * y)]
    if lmax >= 3:
        a = sqrt(35.0 / 8.0)
        b = sqrt(105.0)
        c = sqrt(21.0 / 8.0)
        cols += [a * (3 * x * x * y - y ** 3), b * x * y * z, c * y * (5 * z * z - 1),
                 0.5 * sqrt(7.0) * (5 * z ** 3 - 3 * z), c * x * (5 * z * z - 1),
                 0.5 * b * z * (x * x - y * y), a * (x ** 3 - 3 * x * y * y)]
    return np.stack(cols, axis=1)


# ------------------------------------------------------------------------------- workloads

@dataclass
class Workload:
    spec: WorkloadSpec
    recv: np.ndarray  # int32 [E], non-decreasing
    src: np.ndarray  # int32 [E]
    vectors: np.ndarray  # fp64 [E, 3]
    x: np.ndarray  # [N, U, D_x] in spec dtype
    Y: np.ndarray  # [E, D_Y] in spec dtype

    @property
    def n_nodes(self) -> int:
        return int(self.x.shape[0])

    @property
    def n_edges(self) -> int:
        return int(self.src.size)


def _normal(rng, shape, dtype):
    if dtype == np.float32:
        return rng.standard_normal(shape, dtype=np.float32)
    return rng.standard_normal(shape)


def dim_of(irreps: str) -> int:
    """Total width of an irreps string counted per channel (sum of 2l+1 over its terms)."""
    return sum(2 * int(t.split("x")[1][:-1]) + 1 for t in irreps.split("+"))


def make_workload(key_or_spec, n_nodes: int | None = None) -> Workload:
    spec = SPECS[key_or_spec] if isinstance(key_or_spec, int) else key_or_spec
    st = streams(spec.key)
    dtype = np.dtype(spec.dtype).type
    N = n_nodes or spec.n_nodes
    if spec.graph == "uniform":
        recv, src = uniform_graph(N, spec.degree, st["graph"])
        vec = unit_vectors(recv.size, st["vectors"])
    elif spec.graph == "periodic":
        recv, src, vec, _ = periodic_graph(N, spec.density, spec.cutoff, st["graph"])
    else:
        raise ValueError(spec.graph)
    U = spec.mul
    dx = dim_of(spec.irreps_x)
    x = _normal(st["x"], (N, U, dx), dtype)
    Y = sh_inputs(vec, spec.sh_lmax).astype(dtype)
    return Workload(spec, recv, src, vec, np.ascontiguousarray(x), np.ascontiguousarray(Y))


def make_weights(spec: WorkloadSpec, n_edges: int, n_paths: int) -> np.ndarray:
    """w[E][P][U] ~ N(0,1)/sqrt(mean degree)."""
    st = streams(spec.key)
    dtype = np.dtype(spec.dtype).type
    w = _normal(st["w"], (n_edges, n_paths, spec.mul), dtype)
    w *= dtype(1.0 / sqrt(spec.w_scale_degree))
    return w


def make_cotangent(spec: WorkloadSpec, n_nodes: int, dim_out: int) -> np.ndarray:
    """d_out[N][U][D_out] ~ N(0,1)."""
    st = streams(spec.key)
    dtype = np.dtype(spec.dtype).type
    return _normal(st["d_out"], (n_nodes, spec.mul, dim_out), dtype)


def custom_spec(key: int, n_nodes: int, irreps_x: str, irreps_sh: str, lmax_out: int,
                dtype: str = "float32", degree: int = 4) -> WorkloadSpec:
    """A small uniform-degree workload for tests (keys >= 100 keep their own seed streams)."""
    return WorkloadSpec(key, f"custom{key}", n_nodes, irreps_x, irreps_sh, lmax_out, dtype,
                        "uniform", degree=degree, w_scale_degree=max(degree, 1))


def tp_inputs(spec: WorkloadSpec, batch: int, n_paths: int, dim_out: int, shared: bool, seed: int = 0):
    """Inputs of the batched (non-convolution) tensor product on the irreps of `spec`:
    x [B][U][D_x] ~ N(0,1); y [B][D_Y] = SH of normalised N(0, I3) vectors; w ~ N(0,1), per sample
    [B][P][U] or shared [P][U]; d_out [B][U][D_out] ~ N(0,1).  Seeded by (spec key, seed)."""
    rng = np.random.default_rng(np.random.SeedSequence([SEED_BASE + spec.key, 7, seed]))
    dtype = np.dtype(spec.dtype).type
    x = _normal(rng, (batch, spec.mul, dim_of(spec.irreps_x)), dtype)
    y = sh_inputs(unit_vectors(batch, rng), spec.sh_lmax).astype(dtype)
    w = _normal(rng, (n_paths, spec.mul) if shared else (batch, n_paths, spec.mul), dtype)
    g = _normal(rng, (batch, spec.mul, dim_out), dtype)
    return np.ascontiguousarray(x), np.ascontiguousarray(y), np.ascontiguousarray(w), np.ascontiguousarray(g)


def radial_inputs(spec: WorkloadSpec, n_edges: int, n_paths: int, n_basis: int = 8, hidden=(64, 64, 64),
                  r_min: float = 0.75, r_cut: float = 5.0, seed: int = 0):
    """Inputs of the convolution with fused radial weights on the irreps of `spec`:
    edge lengths r [E] with density proportional to r^2 on [r_min, r_cut) (neighbours uniform in
    space around each atom, none closer than r_min), the radial network's layers
    W_i [H_(i-1)][H_i] ~ N(0, 1/H_(i-1)) with H_0 = n_basis, and its last layer
    W_last [H][P][U] ~ N(0, 1/H) / sqrt(mean degree).  Seeded by (spec key, seed)."""
    rng = np.random.default_rng(np.random.SeedSequence([SEED_BASE + spec.key, 11, seed]))
    dtype = np.dtype(spec.dtype).type
    a = (r_min / r_cut) ** 3
    r = r_cut * np.cbrt(rng.uniform(a, 1.0, size=n_edges))
    widths = [n_basis, *hidden]
    layers = [(rng.standard_normal((widths[i], widths[i + 1])) / sqrt(widths[i])).astype(dtype)
              for i in range(len(hidden))]
    H = widths[-1]
    w_last = rng.standard_normal((H, n_paths, spec.mul)) / sqrt(H) / sqrt(spec.w_scale_degree)
    return (np.ascontiguousarray(r.astype(dtype)), [np.ascontiguousarray(W) for W in layers],
            np.ascontiguousarray(w_last.astype(dtype)))
