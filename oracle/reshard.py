"""CPU oracle for the M-to-N reshard over logical ranks.

TEST INFRASTRUCTURE ONLY (same rule as the rest of ``oracle/``).

Definition followed (the M2N part of the "NCCL M2N vs T-CCL" article on
lqnn.cn, §1.2-§1.4): a layout is a mesh of ranks (a shape, row-major rank
order, starting at a base rank) and one placement per mesh axis, either
``Shard(d)`` (tensor dimension d is cut into equal contiguous blocks along that
axis) or ``Replicate()``. With at most one sharded axis per layout (the
article's design constraint), the rank at mesh coordinates c holds the box
``[c_a * S_d / n_a, (c_a + 1) * S_d / n_a)`` along the sharded dimension d
(a the sharded axis, n_a its size) and the full extent along every other
dimension, stored contiguously in row-major order. ``reshard`` gives every
destination rank exactly the box its destination layout names, taken from the
source ranks' boxes.

The plain way: rebuild the global tensor from the source buffers (each element
taken from the first source rank, in mesh order, whose box holds it; source
replicas hold identical data by contract), then cut every destination box out
of it.
"""
from __future__ import annotations

import itertools

import numpy as np

REPLICATE = -1


def mesh_coords(dims, m):
    """Row-major coordinates of mesh rank m."""
    out = []
    for n in reversed(dims):
        out.append(m % n)
        m //= n
    return tuple(reversed(out))


def check_layout(dims, placements, shape):
    """The article's constraints: one placement per mesh axis, at most one
    sharded axis, a valid tensor dimension that the axis divides."""
    if len(placements) != len(dims):
        raise ValueError("one placement per mesh axis")
    sharded = [d for d in placements if d != REPLICATE]
    if len(sharded) > 1:
        raise ValueError("at most one sharded mesh axis per layout")
    for a, d in enumerate(placements):
        if d != REPLICATE and not (0 <= d < len(shape)):
            raise ValueError("sharded dimension out of range")


def local_box(shape, dims, placements, m):
    """[(lo, hi)] per tensor dimension held by mesh rank m."""
    check_layout(dims, placements, shape)
    box = [(0, s) for s in shape]
    coords = mesh_coords(dims, m)
    for a, d in enumerate(placements):
        if d == REPLICATE:
            continue
        n = dims[a]
        if shape[d] % n:
            raise ValueError("tensor dimension not divisible by the mesh axis")
        step = shape[d] // n
        box[d] = (coords[a] * step, (coords[a] + 1) * step)
    return box


def nranks(dims):
    out = 1
    for n in dims:
        out *= n
    return out


def reshard(src_bufs, src_dims, src_place, dst_dims, dst_place, shape):
    """Returns one array per destination mesh rank (row-major local blocks)."""
    dtype = src_bufs[0].dtype
    glob = np.zeros(shape, dtype=dtype)
    filled = np.zeros(shape, dtype=bool)
    for m in range(nranks(src_dims)):
        box = local_box(shape, src_dims, src_place, m)
        sl = tuple(slice(lo, hi) for lo, hi in box)
        local = np.asarray(src_bufs[m]).reshape([hi - lo for lo, hi in box])
        take = ~filled[sl]
        glob[sl][take] = local[take]
        filled[sl] = True
    if not filled.all():
        raise ValueError("the source layout does not cover the tensor")
    out = []
    for m in range(nranks(dst_dims)):
        box = local_box(shape, dst_dims, dst_place, m)
        out.append(np.ascontiguousarray(glob[tuple(slice(lo, hi) for lo, hi in box)]).ravel())
    return out


def element_owner_check(dst_bufs, dst_dims, dst_place, shape, value_of):
    """Independent element-by-element check (pure Python loops): every element
    of every destination block equals value_of(global coordinates)."""
    for m, buf in enumerate(dst_bufs):
        box = local_box(shape, dst_dims, dst_place, m)
        ext = [hi - lo for lo, hi in box]
        flat = np.asarray(buf).ravel()
        for i, local in enumerate(itertools.product(*[range(e) for e in ext])):
            g = tuple(lo + x for (lo, _), x in zip(box, local))
            if flat[i] != value_of(g):
                return False
    return True
