"""Layout maps, sharded storage, resharding and unit tasks (oracle).

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__``).  Plain numpy, written
from the pages' index formulas; nothing here is shared with the GPU path.

Parity status: pinned.  ``tests/test_oracle_layouts.py`` checks bijection,
round trips, composition, the per-device memory formula of MP3D §3.1.1, the
y<->z exchange of MP3D §3.1.1 (last paragraph) and the worked example of
CMR §2 / Figure 2 (``tests/golden/cmr_figure2_unit_tasks.json``).

Storage convention (shared with the C ABI by specification, not by code):
a sharded tensor is one flat buffer holding every device's shard back to
back, in device order; each shard is dense and row-major.  A replicated
layout stores every replica.

Readings where the pages are silent:

* Virtual-device linear order: device (i, j, l) of the p x p x p cube is
  number (i*p + j)*p + l.  MP3D §2.3 names processors by (i, j, l) on the
  directions x, y, z but fixes no linear order.
* MP3D §3.1.1 prints the column range of the gathered weight block as
  ``lnp : np-1``; the plain reading is ``lnp : lnp+np-1`` (the same range as
  the shard formula just above it).
* Exchanging directions y and z (MP3D §3.1.1, last paragraph) means that the
  block a device (i, j, l) holds after the exchange is the block device
  (i, l, j) held before it; weights keep direction x.
* CMR §2 calls the slices of the first spec of Figure 2 "4x1" but then sends
  the slice [0, 1, 2, 3] of D = arange(16).reshape(4, 4) to devices 4 and 5
  only; the slices are therefore rows (1 x 4), i.e. a 4-way row split.
* Sizes that do not divide evenly are rejected (ValueError).
"""
from __future__ import annotations

from dataclasses import dataclass
from itertools import product

import numpy as np


def device_index(i: int, j: int, l: int, p: int) -> int:
    """Linear number of virtual device (i, j, l) (reading, see module doc)."""
    return (i * p + j) * p + l


def cube_devices(p: int):
    """All (i, j, l) of the p^3 cube in device order."""
    return [(i, j, l) for i in range(p) for j in range(p) for l in range(p)]


def _need(cond: bool, msg: str):
    if not cond:
        raise ValueError(msg)


# --------------------------------------------------------------------------
# Cube layouts, MP3D §3.1.1 (Load Balancing), Figure "3d2".
# m = M/p^2, n = N/p^2, k = K/p^2.  Ranges below are half-open; the paper's
# are inclusive (a : a+m-1).
# --------------------------------------------------------------------------

def _cube_a_block(R, C, p, i, j, l):
    # A_ijl = A[imp+jm : imp+jm+m-1, lnp : lnp+np-1]
    m, n = R // (p * p), C // (p * p)
    _need(R % (p * p) == 0 and C % p == 0, "CUBE_A needs R % p^2 == 0 and C % p == 0")
    np_ = C // p
    r0 = i * m * p + j * m
    c0 = l * np_
    return slice(r0, r0 + m), slice(c0, c0 + np_)


def _cube_b_block(R, C, p, i, j, l):
    # device (i, j, l) holds B_lji = B[lnp : lnp+np-1, jkp+ik : jkp+ik+k-1]
    _need(R % p == 0 and C % (p * p) == 0, "CUBE_B needs R % p == 0 and C % p^2 == 0")
    np_ = R // p
    k = C // (p * p)
    r0 = l * np_
    c0 = j * k * p + i * k
    return slice(r0, r0 + np_), slice(c0, c0 + k)


def _cube_c_block(R, C, p, i, j, l):
    # device (i, j, l) keeps C_ilj = C[imp+lm : imp+lm+m-1, jkp : jkp+kp-1]
    _need(R % (p * p) == 0 and C % p == 0, "CUBE_C needs R % p^2 == 0 and C % p == 0")
    m = R // (p * p)
    kp = C // p
    r0 = i * m * p + l * m
    c0 = j * kp
    return slice(r0, r0 + m), slice(c0, c0 + kp)


_CUBE_BLOCKS = {"A": _cube_a_block, "B": _cube_b_block, "C": _cube_c_block}


@dataclass(frozen=True)
class Cube:
    """A matrix laid out on the p^3 cube in the role ``role`` (A input,
    B weight, C output) of MP3D Algorithm 1.  ``swap`` = directions y and z
    exchanged (the next linear of a block, MP3D §3.1.1 / §3.2)."""
    role: str
    p: int
    swap: bool = False

    def slices(self, R: int, C: int):
        out = []
        f = _CUBE_BLOCKS[self.role]
        for (i, j, l) in cube_devices(self.p):
            jj, ll = (l, j) if self.swap else (j, l)
            out.append(f(R, C, self.p, i, jj, ll))
        return out


def CUBE_A(p):
    return Cube("A", p)


def CUBE_B(p):
    return Cube("B", p)


def CUBE_C(p):
    return Cube("C", p)


def CUBE_B_SWAP(p):
    return Cube("B", p, swap=True)


# --------------------------------------------------------------------------
# Diagonal vector layout, MP3D §3.1.1 (Figure "vector"): only devices with
# j = l hold b_ji = b[jnp+in : jnp+in+n-1], n = V/p^2.
# --------------------------------------------------------------------------

def vec_diag_slices(V: int, p: int):
    """{(i, j, l): slice of b} for the devices holding a piece (j == l)."""
    _need(V % (p * p) == 0, "VEC_DIAG needs V % p^2 == 0")
    n = V // (p * p)
    out = {}
    for (i, j, l) in cube_devices(p):
        if j == l:
            s = j * n * p + i * n
            out[(i, j, l)] = slice(s, s + n)
    return out


def vec_diag_gather_b(b: np.ndarray, p: int, j: int):
    """b_j, the vector a device with output column block j uses for C + b
    after the broadcast in z and the all-gather in x (MP3D §3.1.1)."""
    sl = vec_diag_slices(b.shape[0], p)
    parts = [b[sl[(i, j, j)]] for i in range(p)]
    return np.concatenate(parts)


# --------------------------------------------------------------------------
# Mesh sharding specs, CMR §2: a spec X0 X1 over a (m1, m2) mesh with
# X in {R, S0, S1, S01}; device (a, b) of the mesh is number a*m2 + b.
# --------------------------------------------------------------------------

@dataclass(frozen=True)
class MeshSpec:
    m1: int
    m2: int
    spec: tuple

    def _part(self, X, extent, a, b):
        if X == "R":
            return slice(0, extent)
        parts, idx = {"S0": (self.m1, a), "S1": (self.m2, b),
                      "S01": (self.m1 * self.m2, a * self.m2 + b)}[X]
        _need(extent % parts == 0, f"dimension {extent} not divisible by {parts}")
        w = extent // parts
        return slice(idx * w, idx * w + w)

    def slices(self, R: int, C: int):
        out = []
        for a, b in product(range(self.m1), range(self.m2)):
            out.append((self._part(self.spec[0], R, a, b),
                        self._part(self.spec[1], C, a, b)))
        return out


def ROW(s):
    """s-way row split (S^{01} R on a 1 x s mesh)."""
    return MeshSpec(1, s, ("S01", "R"))


def COL(s):
    """s-way column split (R S^{01})."""
    return MeshSpec(1, s, ("R", "S01"))


def BLOCK(a, b):
    """2-D block split S^0 S^1 on an a x b mesh."""
    return MeshSpec(a, b, ("S0", "S1"))


def REP(n):
    """n full replicas (R R)."""
    return MeshSpec(1, n, ("R", "R"))


# --------------------------------------------------------------------------
# Sharded storage and resharding.
# --------------------------------------------------------------------------

def to_sharded(G: np.ndarray, layout) -> np.ndarray:
    """Flat buffer holding every device's slice of G back to back."""
    R, C = G.shape
    return np.concatenate([G[rs, cs].ravel() for rs, cs in layout.slices(R, C)])


def from_sharded(buf: np.ndarray, layout, R: int, C: int) -> np.ndarray:
    """The global R x C matrix from a sharded buffer.  Where several devices
    hold the same element (replicas), the lowest-numbered device is read."""
    G = np.empty((R, C), dtype=buf.dtype)
    sls = layout.slices(R, C)
    offs = np.cumsum([0] + [(rs.stop - rs.start) * (cs.stop - cs.start) for rs, cs in sls])
    _need(offs[-1] == buf.size, "buffer size does not match the layout")
    for d in reversed(range(len(sls))):
        rs, cs = sls[d]
        G[rs, cs] = buf[offs[d]:offs[d + 1]].reshape(rs.stop - rs.start, cs.stop - cs.start)
    return G


def sharded_size(layout, R: int, C: int) -> int:
    return sum((rs.stop - rs.start) * (cs.stop - cs.start) for rs, cs in layout.slices(R, C))


def reshard(buf: np.ndarray, src, dst, R: int, C: int) -> np.ndarray:
    """Resharding: every destination element takes the bits of the same global
    element of the source (CMR §2, cross-mesh resharding).  Bits are copied
    as they are; dtype is preserved."""
    return to_sharded(from_sharded(buf, src, R, C), dst)


def unit_tasks(src, dst, R: int, C: int, src_offset: int = 0, dst_offset: int = 0):
    """CMR §2: one unit communication task per unique source data slice,
    sent to the destination devices whose slice overlaps it.  Returns a list
    of (rows, cols, source devices, destination devices) in first-holder
    order; source and destination devices are numbered from ``src_offset``
    and ``dst_offset`` (the two meshes are disjoint)."""
    tasks = []
    seen = {}
    for d, (rs, cs) in enumerate(src.slices(R, C)):
        key = (rs.start, rs.stop, cs.start, cs.stop)
        if key in seen:
            tasks[seen[key]][2].append(d + src_offset)
            continue
        dsts = []
        for e, (rd, cd) in enumerate(dst.slices(R, C)):
            if rd.start < rs.stop and rs.start < rd.stop and cd.start < cs.stop and cs.start < cd.stop:
                dsts.append(e + dst_offset)
        seen[key] = len(tasks)
        tasks.append((rs, cs, [d + src_offset], dsts))
    return tasks


def cube_memory_per_device(M: int, N: int, K: int, p: int) -> int:
    """MP3D §3.1.1: (M/p^2)(N/p) + (N/p)(K/p^2) + (M/p^2)(K/p) elements."""
    return (M // (p * p)) * (N // p) + (N // p) * (K // (p * p)) + (M // (p * p)) * (K // p)
