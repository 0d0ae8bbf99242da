"""The work partition of the decode-row kernels (csrc/simt.cuh, decode rows), checked on the
CPU for shapes and grids the GPU tests do not reach: the loops of decode_swiglu_kernel and
decode_apply_kernel, restated here over indices only, must read every 8-element slice of
every weight row once and write every output once.  (No arithmetic is modelled.)"""
import itertools

import numpy as np
import pytest

NW = 8  # warps per block (256 threads)


def swiglu_visits(d, f, grid, NB, NBATCH):
    """Count, per (column n, slice k/8), the loads the SwiGLU kernel issues."""
    seen = np.zeros((f, d // 8), dtype=np.int64)
    writes = np.zeros(f, dtype=np.int64)
    for block in range(grid):
        for n0 in range(block * NB, f, grid * NB):
            for warp, lane in itertools.product(range(NW), range(32)):
                for k0 in range((warp * 32 + lane) * 8, d, NW * 256 * NBATCH):
                    for j in range(NBATCH):
                        k = k0 + j * NW * 256
                        if k >= d:
                            break
                        for c in range(NB):
                            if n0 + c < f:
                                seen[n0 + c, k // 8] += 1
            for c in range(NB):  # the threads that finish the columns
                if n0 + c < f:
                    writes[n0 + c] += 1
    return seen, writes


def apply_visits(Bq, d, f, grid, NB, NBATCH):
    rows = Bq * d
    seen = np.zeros((rows, f // 8), dtype=np.int64)
    writes = np.zeros(rows, dtype=np.int64)
    groups = rows // NB
    for block in range(grid):
        for q in range(block, groups, grid):
            row0 = q * NB
            assert row0 // d == (row0 + NB - 1) // d, "a group spans two sequences"
            for warp, lane in itertools.product(range(NW), range(32)):
                for n0 in range((warp * 32 + lane) * 8, f, NW * 256 * NBATCH):
                    for j in range(NBATCH):
                        n = n0 + j * NW * 256
                        if n >= f:
                            break
                        for c in range(NB):
                            seen[row0 + c, n // 8] += 1
            for c in range(NB):
                writes[row0 + c] += 1
    return seen, writes


@pytest.mark.parametrize("d,f,grid", [(8, 8, 1), (64, 136, 3), (520, 264, 7), (2056, 8, 2), (264, 2056, 5)])
@pytest.mark.parametrize("NB,NBATCH", [(2, 2), (2, 1)])
def test_swiglu_rows_read_each_weight_slice_once(d, f, grid, NB, NBATCH):
    seen, writes = swiglu_visits(d, f, grid, NB, NBATCH)
    assert (seen == 1).all() and (writes == 1).all()


@pytest.mark.parametrize("Bq,d,f,grid", [(1, 8, 8, 1), (2, 64, 136, 3), (3, 136, 2056, 4), (1, 520, 264, 9)])
@pytest.mark.parametrize("NB,NBATCH", [(2, 2), (8, 1)])
def test_apply_rows_read_each_weight_slice_once(Bq, d, f, grid, NB, NBATCH):
    seen, writes = apply_visits(Bq, d, f, grid, NB, NBATCH)
    assert (seen == 1).all() and (writes == 1).all()
